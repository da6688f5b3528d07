"""Q8_0 weights on the GPU ("rvllm-metal", sections "What's basic about it" and "What's next":
the int8 weight stream): each kernel on awkward shapes, small models through every projection
kernel, and the batch-1 GPT-2-124M-shaped greedy workload at full size (GPU only)."""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import workloads as wl
from parity_util import LOGIT_TOL, check_ids, check_logits, oracle_teacher, record, run_gpu_teacher
from test_gpu_parity import LENGTHS, SMALL_GPT2, SMALL_LLAMA, STEPS, small_workload

pytestmark = pytest.mark.gpu

Q8_SHAPES = [(1, 33, 64), (3, 130, 768), (7, 64, 960), (16, 2304, 768), (32, 768, 3072), (64, 1000, 192),
             (127, 130, 64), (300, 576, 384), (1030, 200, 160)]


@pytest.mark.parametrize("variant", [1, 2], ids=["gemv", "simt"])
@pytest.mark.parametrize("M,N,K", Q8_SHAPES)
def test_q8_linear_matches_oracle(gpu_lib, variant, M, N, K):
    import torch
    r = np.random.default_rng(M * 7 + N + K)
    x = r.standard_normal((M, K), dtype=np.float32)
    q, d = wl.quantize_q8_0(r.standard_normal((N, K), dtype=np.float32) * np.float32(0.05))
    b = r.standard_normal(N, dtype=np.float32) * np.float32(0.1)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    gpu_lib.op_linear_q8(torch.from_numpy(x).cuda(), torch.from_numpy(q).cuda(), torch.from_numpy(d).cuda(),
                         torch.from_numpy(b).cuda(), y, variant)
    torch.cuda.synchronize()
    wf = oracle.dequant_q8_0(q, d)
    ref = oracle.OracleModel.linear(x.astype(np.float64), wf, b.astype(np.float64))
    got = y.cpu().numpy()
    scale = np.abs(x.astype(np.float64)) @ np.abs(wf).T + np.abs(b)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= 1e-6 + 4 * K * 2.0 ** -23 * scale), float(np.abs(got - ref).max())


Q8_MODELS = [replace(SMALL_GPT2, name="small-gpt2-q8", dtype=wl.DTYPE_Q8),
             replace(SMALL_LLAMA, name="small-llama-q8", dtype=wl.DTYPE_Q8)]


@pytest.mark.parametrize("variant", [0, 1, 2], ids=["auto", "gemv", "simt"])
@pytest.mark.parametrize("shape", Q8_MODELS, ids=[s.name for s in Q8_MODELS])
def test_small_q8_model_matches_oracle(gpu_lib, shape, variant):
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    model = oracle.OracleModel(w)
    run = WorkloadRun(small_workload(shape), host_weights=w, lengths=LENGTHS)
    stream = wl.draw_stream(run.B, STEPS, shape.vocab)
    ids, z = run_gpu_teacher(run, stream, variant=variant)
    assert run.dec.error_flags() == 0
    run.close()
    for b in range(run.B):
        ref = oracle_teacher(model, run.prompts[b], stream[:, b])
        check_logits(z[:, b], ref, shape.dtype, f"{shape.name} seq {b}")
        check_ids(ids[:, b], ref, f"{shape.name} seq {b}")


def test_gpt2_124m_q8_b1_greedy_stream(gpu_lib):
    """The batch-1 greedy workload (8 prompt ids, 16 greedy steps) with Q8_0 weights."""
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    W = wl.W_GPT2_Q8_B1
    w = wl.make_weights(W.model)
    model = oracle.OracleModel(w)
    run = WorkloadRun(W, host_weights=w)
    ids_ref, z_ref = oracle.greedy_generate(model, run.prompts[0], W.decode_steps)
    ids, z = run_gpu_teacher(run, ids_ref[:-1].reshape(-1, 1).astype(np.int32))
    err = check_logits(z[:, 0], z_ref, W.model.dtype, W.name)
    n = check_ids(ids[:, 0], z_ref, W.name)
    assert n >= 1
    record(W.name, err, LOGIT_TOL[W.model.dtype], n, rows=int(z_ref.shape[0]))
    assert run.dec.error_flags() == 0
    run.close()
