"""The one-kernel decode step (batches of at most 8 sequences) against the oracle and against
the step of one kernel a phase, and its grid barrier's bounded wait (GPU only)."""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import workloads as wl
from parity_util import LOGIT_TOL, check_ids, check_logits, oracle_teacher, record, run_gpu_teacher
from test_gpu_parity import SMALL, SMALL_GPT2, SMALL_LLAMA, STEPS
from test_gpu_variants import ALL_FEATURES

pytestmark = pytest.mark.gpu

# Eight sequences. The Llama shapes (n_ctx 512) hold contexts of 300 and 257 + STEPS keys, which
# the persistent kernel cuts into two 256-key attention items merged by the output projection;
# the GPT-2 shapes (n_ctx 128) stay within one item.
LENGTHS_GPT2 = np.array([5, 17, 70, 1, 33, 100, 9, 64], dtype=np.int32)
LENGTHS_LLAMA = np.array([5, 17, 70, 1, 33, 300, 9, 257], dtype=np.int32)
PK_LAUNCHES = 3   # step arguments, the persistent kernel, the argmax reduction


def _lengths(shape, B):
    return (LENGTHS_GPT2 if shape.arch == wl.ARCH_GPT2 else LENGTHS_LLAMA)[:B]


def _workload(shape, B, kv_dtype=wl.DTYPE_F32):
    return wl.Workload("pk", shape, batch=B, prompt_len=0, decode_steps=STEPS, mode="teacher", kv_dtype=kv_dtype)


def _run(shape, w, B, persistent, kv_dtype=wl.DTYPE_F32, stream=None):
    import torch
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    run = WorkloadRun(_workload(shape, B, kv_dtype), host_weights=w, lengths=_lengths(shape, B))
    assert run.dec.set_persistent(persistent), "the persistent step should apply to this model"
    if stream is None:
        stream = wl.draw_stream(B, STEPS, shape.vocab)
    ids, z = run_gpu_teacher(run, stream)
    torch.cuda.synchronize()
    launches = run.dec.last_launch_count()
    flags = run.dec.error_flags()
    prompts = run.prompts
    run.close()
    return ids, z, launches, flags, prompts, stream


@pytest.mark.parametrize("B", [1, 3, 8])
@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_persistent_step_matches_oracle(gpu_lib, shape, B):
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    ids, z, launches, flags, prompts, stream = _run(shape, w, B, True)
    assert flags == 0
    assert launches == PK_LAUNCHES, f"decode step took {launches} launches: not the persistent kernel"
    model = oracle.OracleModel(w)
    worst, n_ids = 0.0, 0
    for b in range(B):
        ref = oracle_teacher(model, prompts[b], stream[:, b])
        worst = max(worst, check_logits(z[:, b], ref, shape.dtype, f"{shape.name} B={B} seq {b}"))
        n_ids += check_ids(ids[:, b], ref, f"{shape.name} B={B} seq {b}")
    record(f"persistent {shape.name} B={B}", worst, LOGIT_TOL[shape.dtype], n_ids)


@pytest.mark.parametrize("shape", [SMALL_GPT2, SMALL_LLAMA], ids=["gpt2-f32", "llama-bf16"])
def test_persistent_step_agrees_with_per_phase_kernels(gpu_lib, shape):
    """Both paths on the same inputs: logits within the oracle bound of each other, the same
    greedy ids wherever the per-phase step's own margin is clear."""
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    ids_p, z_p, n_p, f_p, _, stream = _run(shape, w, 8, True)
    ids_g, z_g, n_g, f_g, _, _ = _run(shape, w, 8, False, stream=stream)
    assert f_p == 0 and f_g == 0
    assert n_p == PK_LAUNCHES and n_g >= 5 * shape.n_layers + 4
    err = float(np.abs(z_p.astype(np.float64) - z_g).max())
    assert err <= LOGIT_TOL[shape.dtype], err
    for s in range(z_g.shape[0]):
        for b in range(8):
            zz = z_g[s, b].astype(np.float64)
            if oracle.top2_margin(zz) > 2 * LOGIT_TOL[shape.dtype]:
                assert ids_p[s, b] == ids_g[s, b], (s, b)


def test_persistent_step_bf16_kv_and_model_variants(gpu_lib):
    """bf16 KV cache; sliding window (24, every second layer global), Q/K norm, attention biases
    and Llama 3 RoPE scaling, all inside the persistent kernel."""
    shape = replace(SMALL_LLAMA, name="small-llama-all", **ALL_FEATURES)
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    for kv in (wl.DTYPE_F32, wl.DTYPE_BF16):
        ids, z, launches, flags, prompts, stream = _run(shape, w, 8, True, kv_dtype=kv)
        assert flags == 0 and launches == PK_LAUNCHES
        model = oracle.OracleModel(w, kv_dtype=kv)
        for b in range(8):
            ref = oracle_teacher(model, prompts[b], stream[:, b])
            check_logits(z[:, b], ref, shape.dtype, f"all features kv={kv} seq {b}")
            check_ids(ids[:, b], ref, f"all features kv={kv} seq {b}")


def test_persistent_step_sampling_reads_its_logits(gpu_lib):
    """A sampled step after the persistent kernel: top_k = 1 gives the greedy ids."""
    import torch
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    shape = SMALL_LLAMA
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    run = WorkloadRun(_workload(shape, 4), host_weights=w, lengths=_lengths(shape, 4))
    assert run.dec.set_persistent(True)
    run.prefill()
    toks = torch.from_numpy(wl.draw_stream(4, 1, shape.vocab)[0]).cuda()
    zg = torch.empty((4, shape.vocab), dtype=torch.float32, device="cuda")
    greedy = torch.zeros(4, dtype=torch.int32, device="cuda")
    run.decode(toks, 0, logits=zg, next_ids=greedy)
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    z = torch.empty_like(zg)
    run.decode_sample(toks, 0, 0.8, 1, torch.rand(4, device="cuda"), logits=z, next_ids=ids)
    torch.cuda.synchronize()
    assert run.dec.error_flags() == 0
    assert torch.equal(z, zg) and torch.equal(ids, greedy)
    run.close()


def test_grid_barrier_timeout_sets_the_flag_and_the_context_stays_usable(gpu_lib):
    """One CTA withheld: the others' bounded barrier wait runs out (about a second), sets
    LLM_FLAG_WAIT_TIMEOUT, and every CTA leaves; the next steps equal a fresh run bit for bit."""
    import time
    import torch
    import transformer_decoder_forward_gb300 as L
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    shape = SMALL_GPT2
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    stream = wl.draw_stream(3, STEPS, shape.vocab)
    ref_ids, ref_z, _, _, _, _ = _run(shape, w, 3, True, stream=stream)
    run = WorkloadRun(_workload(shape, 3), host_weights=w, lengths=_lengths(shape, 3))
    assert run.dec.set_persistent(True)
    t0 = time.time()
    run.dec.selftest_grid_barrier()
    took = time.time() - t0
    assert run.dec.error_flags() & L.FLAG_WAIT_TIMEOUT
    assert 0.2 < took < 30.0, took
    ids, z = run_gpu_teacher(run, stream)
    torch.cuda.synchronize()
    assert run.dec.error_flags() == 0
    assert np.array_equal(ids, ref_ids) and np.array_equal(z, ref_z)
    run.close()
