"""CUDA path vs float64 oracle, element by element, through the C ABI (GPU only)."""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import workloads as wl
from parity_util import FLOOR_MULT, LOGIT_TOL, MARGIN, check_ids, check_logits, oracle_teacher, record, run_gpu_teacher

pytestmark = pytest.mark.gpu

# Small shapes: several 64-wide tiles, ragged tails (vocab 1000, lengths 5/17/70), 2 layers.
SMALL_GPT2 = wl.ModelShape("small-gpt2", wl.ARCH_GPT2, wl.DTYPE_F32, 2, 192, 3, 3, 64, 512, 1000, 128)
SMALL_GPT2_BF16 = replace(SMALL_GPT2, name="small-gpt2-bf16", dtype=wl.DTYPE_BF16)
SMALL_LLAMA = wl.ModelShape("small-llama", wl.ARCH_LLAMA, wl.DTYPE_BF16, 2, 384, 6, 2, 64, 320, 1024, 512)
SMALL_LLAMA_F32 = replace(SMALL_LLAMA, name="small-llama-f32", dtype=wl.DTYPE_F32)
SMALL = [SMALL_GPT2, SMALL_GPT2_BF16, SMALL_LLAMA, SMALL_LLAMA_F32]
LENGTHS = np.array([5, 17, 70], dtype=np.int32)
STEPS = 6


def small_workload(shape, contiguous=False, shuffle=True):
    return wl.Workload("small", shape, batch=len(LENGTHS), prompt_len=0, decode_steps=STEPS, mode="teacher",
                       contiguous_kv=contiguous, shuffle_tables=shuffle)


@pytest.fixture(scope="module")
def small_models():
    out = {}
    for s in SMALL:
        w = wl.make_weights(s, scale=2.0, perturb=True)
        out[s.name] = (w, oracle.OracleModel(w))
    return out


def _oracle_rows(model, run, stream):
    return [oracle_teacher(model, run.prompts[b], stream[:, b]) for b in range(run.B)]


@pytest.mark.parametrize("variant", [1, 2, 3, 4, 5], ids=["gemv", "simt", "tcgen05", "tcgen05-swap", "tcgen05-pair"])
@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_small_model_matches_oracle(gpu_lib, small_models, shape, variant):
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, model = small_models[shape.name]
    run = WorkloadRun(small_workload(shape), host_weights=w, lengths=LENGTHS)
    stream = wl.draw_stream(run.B, STEPS, shape.vocab)
    ids, z = run_gpu_teacher(run, stream, variant=variant)
    assert run.dec.error_flags() == 0
    ref = _oracle_rows(model, run, stream)
    for b in range(run.B):
        check_logits(z[:, b], ref[b], shape.dtype, f"{shape.name} seq {b}")
        check_ids(ids[:, b], ref[b], f"{shape.name} seq {b}")
    run.close()


@pytest.mark.parametrize("shape", [SMALL_GPT2, SMALL_LLAMA], ids=["small-gpt2", "small-llama"])
def test_many_sequences_split_decode_attention_matches_oracle(gpu_lib, small_models, shape):
    """17 sequences of 1..110 tokens: the decode attention cuts the longer ones into 64-token
    chunks (split kernel plus merge launch) next to sequences that fit one chunk; every sequence
    agrees with the oracle."""
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, model = small_models[shape.name]
    lengths = np.array([5, 17, 70, 33, 64, 65, 1, 100, 47, 16, 80, 2, 90, 31, 58, 110, 9], dtype=np.int32)
    W = wl.Workload("small-many", shape, batch=len(lengths), prompt_len=0, decode_steps=STEPS, mode="teacher")
    run = WorkloadRun(W, host_weights=w, lengths=lengths)
    stream = wl.draw_stream(run.B, STEPS, shape.vocab)
    ids, z = run_gpu_teacher(run, stream)
    assert run.dec.error_flags() == 0
    for b in range(run.B):
        ref = oracle_teacher(model, run.prompts[b], stream[:, b])
        check_logits(z[:, b], ref, shape.dtype, f"{shape.name} seq {b}")
        check_ids(ids[:, b], ref, f"{shape.name} seq {b}")
    run.close()


@pytest.mark.parametrize("variant", [0, 2, 5], ids=["auto", "simt", "tcgen05-pair"])
@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_small_model_bf16_kv_matches_oracle(gpu_lib, small_models, shape, variant):
    """A bf16 KV cache: every attention kernel (decode split-K, fp32-weight prefill tiles, tcgen05
    prefill) reads bf16 K/V, against the oracle that stores K and V rounded to bf16. The SM-pair
    projections write the bf16 K/V of the QKV epilogue (straight from tensor memory for GPT-2,
    through the staged tile with RoPE for the Llama variant)."""
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, _ = small_models[shape.name]
    model = oracle.OracleModel(w, kv_dtype=wl.DTYPE_BF16)
    run = WorkloadRun(replace(small_workload(shape), kv_dtype=wl.DTYPE_BF16), host_weights=w, lengths=LENGTHS)
    stream = wl.draw_stream(run.B, STEPS, shape.vocab)
    ids, z = run_gpu_teacher(run, stream, variant=variant)
    assert run.dec.error_flags() == 0
    run.close()
    for b in range(run.B):
        ref = oracle_teacher(model, run.prompts[b], stream[:, b])
        check_logits(z[:, b], ref, shape.dtype, f"{shape.name} bf16 KV seq {b}")
        check_ids(ids[:, b], ref, f"{shape.name} bf16 KV seq {b}")


# Prompts long enough that the prefill projections span several 128-row token tiles (the
# SM-pair GEMM above 256 rows, the one-SM kernel below): SwiGLU, RoPE and the KV writes of every
# tile, against the oracle, then a few decode steps reading those KV entries.
LONG_LENGTHS = {"small-gpt2": np.array([120, 100, 90], dtype=np.int32),
                "small-gpt2-bf16": np.array([120, 100, 90], dtype=np.int32),
                "small-llama": np.array([300, 17, 200], dtype=np.int32),
                "small-llama-f32": np.array([300, 17, 200], dtype=np.int32)}


@pytest.mark.parametrize("variant", [0, 3], ids=["auto", "tcgen05-one-sm"])
@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_long_prompt_prefill_matches_oracle(gpu_lib, small_models, shape, variant):
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, model = small_models[shape.name]
    lengths = LONG_LENGTHS[shape.name]
    run = WorkloadRun(small_workload(shape), host_weights=w, lengths=lengths)
    stream = wl.draw_stream(run.B, 3, shape.vocab)
    ids, z = run_gpu_teacher(run, stream, variant=variant)
    assert run.dec.error_flags() == 0
    for b in range(run.B):
        ref = oracle_teacher(model, run.prompts[b], stream[:, b])
        check_logits(z[:, b], ref, shape.dtype, f"{shape.name} long prompt seq {b}")
        check_ids(ids[:, b], ref, f"{shape.name} long prompt seq {b}")
    run.close()


def test_graph_replay_equals_eager_bitwise(gpu_lib, small_models):
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, _ = small_models[SMALL_LLAMA.name]
    stream = wl.draw_stream(len(LENGTHS), STEPS, SMALL_LLAMA.vocab)
    outs = []
    for graphs in (True, False):
        run = WorkloadRun(small_workload(SMALL_LLAMA), host_weights=w, lengths=LENGTHS)
        outs.append(run_gpu_teacher(run, stream, graphs=graphs))
        run.close()
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_profiled_step_equals_graph_step_bitwise(gpu_lib, small_models):
    """Per-launch timing (the step captured with an event node around every launch, replayed
    without programmatic launch) changes no result and times every kernel launch of the step."""
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, _ = small_models[SMALL_GPT2.name]
    stream = wl.draw_stream(len(LENGTHS), STEPS, SMALL_GPT2.vocab)
    outs = []
    for prof in (False, True):
        run = WorkloadRun(small_workload(SMALL_GPT2), host_weights=w, lengths=LENGTHS)
        run.dec.kernel_stats(reset=True)
        outs.append(run_gpu_teacher(run, stream, profiling=prof))
        stats = run.dec.kernel_stats(reset=True)
        per_step = run.dec.last_launch_count() - 1   # every launch but the step-arguments node
        run.close()
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])
    assert sum(n for n, _ in stats.values()) == STEPS * per_step
    assert all(t > 0.0 for _, t in stats.values()), stats


def test_programmatic_launch_does_not_change_results(gpu_lib, small_models):
    """Kernels launched with programmatic dependent launch (the default) and without it agree bitwise."""
    import subprocess
    import sys
    code = ("import sys, numpy as np; sys.path.insert(0, 'tests'); sys.path.insert(0, '.');"
            "import workloads as wl; from test_gpu_parity import *;"
            "from transformer_decoder_forward_gb300.runner import WorkloadRun;"
            "w = wl.make_weights(SMALL_LLAMA, scale=2.0, perturb=True);"
            "run = WorkloadRun(small_workload(SMALL_LLAMA), host_weights=w, lengths=LENGTHS);"
            "ids, z = run_gpu_teacher(run, wl.draw_stream(len(LENGTHS), STEPS, SMALL_LLAMA.vocab));"
            "np.save(sys.argv[1], z); np.save(sys.argv[1] + '.ids', ids)")
    import os
    import tempfile
    d = tempfile.mkdtemp()
    outs = []
    for flag in ("1", "0"):
        f = os.path.join(d, f"z{flag}.npy")
        env = dict(os.environ, LLM_PDL=flag)
        subprocess.run([sys.executable, "-c", code, f], check=True, env=env, cwd=os.path.dirname(os.path.dirname(__file__)) or ".")
        outs.append((np.load(f), np.load(f + ".ids.npy")))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_block_table_layout_does_not_change_results(gpu_lib, small_models):
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, _ = small_models[SMALL_GPT2.name]
    stream = wl.draw_stream(len(LENGTHS), STEPS, SMALL_GPT2.vocab)
    outs = []
    for contiguous, shuffle in ((False, True), (False, False), (True, False)):
        run = WorkloadRun(small_workload(SMALL_GPT2, contiguous, shuffle), host_weights=w, lengths=LENGTHS)
        outs.append(run_gpu_teacher(run, stream))
        run.close()
    for o in outs[1:]:
        np.testing.assert_array_equal(outs[0][0], o[0])
        np.testing.assert_array_equal(outs[0][1], o[1])


def test_sequence_result_independent_of_batch(gpu_lib, small_models):
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, _ = small_models[SMALL_LLAMA.name]
    stream = wl.draw_stream(len(LENGTHS), STEPS, SMALL_LLAMA.vocab)
    run = WorkloadRun(small_workload(SMALL_LLAMA), host_weights=w, lengths=LENGTHS)
    ids3, z3 = run_gpu_teacher(run, stream, variant=1)
    run.close()
    run1 = WorkloadRun(small_workload(SMALL_LLAMA), host_weights=w, lengths=LENGTHS, batch=1)
    ids1, z1 = run_gpu_teacher(run1, stream[:, :1], variant=1)
    run1.close()
    np.testing.assert_array_equal(ids1[:, 0], ids3[:, 0])
    np.testing.assert_array_equal(z1[:, 0], z3[:, 0])


def test_host_buffer_entry_point_matches_device_call(gpu_lib, small_models):
    import torch
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, _ = small_models[SMALL_LLAMA.name]
    stream = wl.draw_stream(len(LENGTHS), 2, SMALL_LLAMA.vocab)
    a = WorkloadRun(small_workload(SMALL_LLAMA), host_weights=w, lengths=LENGTHS)
    ids_dev, z_dev = run_gpu_teacher(a, stream)
    a.close()
    b = WorkloadRun(small_workload(SMALL_LLAMA), host_weights=w, lengths=LENGTHS)
    b.prefill()
    torch.cuda.synchronize()
    tables = np.ascontiguousarray(b.tables_np, dtype=np.int32)
    for s in range(2):
        ids = np.zeros(b.B, np.int32)
        z = np.zeros((b.B, SMALL_LLAMA.vocab), np.float32)
        pos = (b.lengths + s).astype(np.int32)
        b.dec.decode_step_host(np.ascontiguousarray(stream[s]), pos, tables, ids, z)
        np.testing.assert_array_equal(ids, ids_dev[s + 1])
        np.testing.assert_array_equal(z, z_dev[s + 1])
    b.close()


def test_device_error_flags_and_host_status(gpu_lib, small_models):
    import torch
    import transformer_decoder_forward_gb300 as L
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, _ = small_models[SMALL_GPT2.name]
    run = WorkloadRun(small_workload(SMALL_GPT2), host_weights=w, lengths=LENGTHS)
    run.prefill()
    assert run.dec.error_flags() == 0
    dev = "cuda"
    # token id out of range
    bad_tok = torch.tensor([5, SMALL_GPT2.vocab + 3, 1], dtype=torch.int32, device=dev)
    run.decode(bad_tok, 0)
    assert run.dec.error_flags() & L.FLAG_BAD_TOKEN
    # position beyond the learned position table and the block table
    pos = torch.tensor([5, 10_000, 70], dtype=torch.int32, device=dev)
    ok_tok = torch.tensor([1, 2, 3], dtype=torch.int32, device=dev)
    with torch.cuda.stream(run.stream):
        run.dec.decode_step(ok_tok, pos, run.tables, run.next_ids)
    assert run.dec.error_flags() & L.FLAG_BAD_POSITION
    # block id outside the pool
    bad_tables = run.tables.clone()
    bad_tables[1, :] = 1 << 20
    with torch.cuda.stream(run.stream):
        run.dec.decode_step(ok_tok, run.step_positions[0], bad_tables, run.next_ids)
    assert run.dec.error_flags() & L.FLAG_BAD_BLOCK
    assert run.dec.error_flags() == 0
    # host-side status codes: nothing is launched
    big = torch.zeros(run.B + 1, dtype=torch.int32, device=dev)
    with pytest.raises(L.LLMError) as e:
        run.dec.decode_step(big, big, run.tables, big)
    assert e.value.status == 2
    with pytest.raises(L.LLMError) as e:
        run.dec.prefill(run.tokens, [0, 1, 1], run.tables, run.next_ids)
    assert e.value.status == 1
    with pytest.raises(L.LLMError) as e:
        run.dec.prefill(run.tokens, [SMALL_GPT2.n_ctx + 1], run.tables, run.next_ids)
    assert e.value.status == 2
    # empty inputs (no sequence at all) are argument errors, refused before any launch
    empty = torch.zeros(0, dtype=torch.int32, device=dev)
    with pytest.raises(L.LLMError) as e:
        run.dec.decode_step(empty, empty, run.tables, empty)
    assert e.value.status == 1
    with pytest.raises(L.LLMError) as e:
        run.dec.prefill(empty, [], run.tables, run.next_ids)
    assert e.value.status == 1
    with pytest.raises(L.LLMError) as e:
        run.dec.step(empty, [], [], run.tables, run.next_ids)
    assert e.value.status == 1
    # and the handle still runs a valid step afterwards
    with torch.cuda.stream(run.stream):
        run.dec.decode_step(ok_tok, run.step_positions[0], run.tables, run.next_ids)
    torch.cuda.synchronize()
    assert run.dec.error_flags() == 0
    run.close()


@pytest.mark.parametrize("shape", [SMALL_GPT2, SMALL_LLAMA], ids=["small-gpt2", "small-llama"])
def test_context_filled_to_n_ctx_matches_oracle(gpu_lib, small_models, shape):
    """The largest context: a prompt of n_ctx - 1 tokens, then one decode step at position
    n_ctx - 1 (the last learned position of GPT-2, the last slot of the block table), with the
    last 16-token block ragged for the Llama shape's prompt."""
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, model = small_models[shape.name]
    lengths = np.array([shape.n_ctx - 1, 37], dtype=np.int32)
    W = wl.Workload("small-full", shape, batch=len(lengths), prompt_len=0, decode_steps=1, mode="teacher")
    run = WorkloadRun(W, host_weights=w, lengths=lengths)
    stream = wl.draw_stream(run.B, 1, shape.vocab)
    ids, z = run_gpu_teacher(run, stream)
    assert run.dec.error_flags() == 0
    for b in range(run.B):
        ref = oracle_teacher(model, run.prompts[b], stream[:, b])
        check_logits(z[:, b], ref, shape.dtype, f"{shape.name} full-context seq {b}")
        check_ids(ids[:, b], ref, f"{shape.name} full-context seq {b}")
    run.close()


def test_bounded_wait_gives_up_sets_flag_and_context_stays_usable(gpu_lib, small_models):
    """A device wait on a barrier that nothing completes gives up after its limit (about one
    second of SM clocks), sets the wait-timeout bit for the host, and later steps still run and
    match a fresh run bit for bit."""
    import time
    import transformer_decoder_forward_gb300 as L
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w, _ = small_models[SMALL_GPT2.name]
    stream = wl.draw_stream(len(LENGTHS), STEPS, SMALL_GPT2.vocab)
    ref = WorkloadRun(small_workload(SMALL_GPT2), host_weights=w, lengths=LENGTHS)
    want = run_gpu_teacher(ref, stream)
    ref.close()
    run = WorkloadRun(small_workload(SMALL_GPT2), host_weights=w, lengths=LENGTHS)
    assert run.dec.error_flags() == 0
    t0 = time.monotonic()
    run.dec.selftest_wait_timeout()
    assert run.dec.error_flags() == L.FLAG_WAIT_TIMEOUT
    assert 0.2 < time.monotonic() - t0 < 30.0
    got = run_gpu_teacher(run, stream)
    assert run.dec.error_flags() == 0
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])
    run.close()


# ------------------------------------------------------------------------------------------------
# the five workloads at their full sizes, in the launch configuration the bench uses
# ------------------------------------------------------------------------------------------------

def test_gpt2_124m_fp32_b1_greedy_stream(gpu_lib):
    """8 prompt ids, 16 greedy steps: the oracle's greedy stream is fed back (teacher forcing)."""
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    W = wl.W_GPT2_F32_B1
    w = wl.make_weights(W.model)
    model = oracle.OracleModel(w)
    run = WorkloadRun(W, host_weights=w)
    ids_ref, z_ref = oracle.greedy_generate(model, run.prompts[0], W.decode_steps)
    stream = ids_ref[:-1].reshape(-1, 1).astype(np.int32)
    ids, z = run_gpu_teacher(run, stream)
    err = check_logits(z[:, 0], z_ref, W.model.dtype, W.name)
    n = check_ids(ids[:, 0], z_ref, W.name)
    assert n >= 1
    record(W.name, err, LOGIT_TOL[W.model.dtype], n, rows=int(z_ref.shape[0]))
    assert run.dec.error_flags() == 0
    run.close()


@pytest.mark.parametrize("W", [wl.W_GPT2_F32_B32, wl.W_GPT2_F32_B32_X8], ids=["x1", "x8"])
def test_gpt2_124m_fp32_b32_teacher_forced(gpu_lib, W):
    """32 sequences x (128 prompt + 128 teacher-forced steps), contiguous KV; oracle on a sample."""
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w = wl.make_weights(W.model, scale=W.weight_scale)
    model = oracle.OracleModel(w)
    run = WorkloadRun(W, host_weights=w)
    stream = wl.draw_stream(run.B, W.decode_steps, W.model.vocab)
    rows = [0, 13, 31]
    ids, z = run_gpu_teacher(run, stream, rows=rows)
    assert run.dec.error_flags() == 0
    run.close()
    for i, b in enumerate(rows):
        ref = oracle_teacher(model, run.prompts[b], stream[:, b])
        tol, floor = LOGIT_TOL[W.model.dtype], None
        if W.weight_scale != 1.0:
            # the float32 floor of these very rows: a plain float32 evaluation against float64
            from fp32_eval import gpt2_forward_f32
            toks = np.concatenate([run.prompts[b], stream[:, b]])
            z32 = gpt2_forward_f32(w, toks)[len(run.prompts[b]) - 1:]
            floor = float(np.abs(z32 - ref).max())
            tol = max(tol, FLOOR_MULT * floor)
        what = f"{W.name} seq {b}"
        err = check_logits(z[:, i], ref, W.model.dtype, what, tol=tol)
        n = check_ids(ids[:, b], ref, what, margin=max(MARGIN, tol / 2))
        record(what, err, tol, n, rows=int(ref.shape[0]), float32_floor=floor)
    if W.weight_scale == 8.0:
        assert model.stats["max_gelu_arg"] > 15.0


def test_smollm2_360m_bf16_b64_decode(gpu_lib):
    """64 sequences of 64..2048 tokens in shuffled paged blocks, one decode step; oracle on 3."""
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    W = wl.W_SMOLLM2_B64
    w = wl.make_weights(W.model)
    model = oracle.OracleModel(w)
    run = WorkloadRun(W, host_weights=w)
    stream = wl.draw_stream(run.B, 1, W.model.vocab)
    lens = run.lengths
    rows = [int(np.argmin(lens)), int(np.argmax(lens)), 7]
    ids, z = run_gpu_teacher(run, stream, rows=rows)
    assert run.dec.error_flags() == 0
    for i, b in enumerate(rows):
        ref = oracle_teacher(model, run.prompts[b], stream[:, b])
        what = f"{W.name} seq {b} (ctx {int(lens[b]) + 1})"
        err = check_logits(z[:, i], ref, W.model.dtype, what)
        record(what, err, LOGIT_TOL[W.model.dtype], check_ids(ids[:, b], ref, what), rows=int(ref.shape[0]))
    run.close()


def test_gpt2_124m_bf16_prefill_16x1024(gpu_lib):
    import torch
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    W = wl.W_GPT2_BF16_PREFILL
    w = wl.make_weights(W.model)
    model = oracle.OracleModel(w)
    run = WorkloadRun(W, host_weights=w)
    logits = torch.empty((run.B, W.model.vocab), dtype=torch.float32, device="cuda")
    run.prefill(logits)
    torch.cuda.synchronize()
    assert run.dec.error_flags() == 0
    ids = run.next_ids.cpu().numpy()
    z = logits.cpu().numpy()
    for b in (0, 15):
        ref = oracle.forward_full(model, run.prompts[b], last_only=True)
        what = f"{W.name} seq {b}"
        err = check_logits(z[b:b + 1], ref, W.model.dtype, what)
        record(what, err, LOGIT_TOL[W.model.dtype], check_ids(ids[b:b + 1], ref, what), rows=1)
    run.close()


def test_gpt2_xl_bf16_b256_ctx1024(gpu_lib):
    """256 sequences: 960-token prompts in shuffled paged blocks, then 64 teacher-forced decode
    steps up to position 1023 (context 1024); the oracle recomputes two sampled sequences."""
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    W = wl.W_GPT2XL_B256
    w = wl.make_weights(W.model)
    run = WorkloadRun(W, host_weights=w)
    stream = wl.draw_stream(run.B, W.decode_steps, W.model.vocab)
    rows = [0, 255]
    ids, z = run_gpu_teacher(run, stream, rows=rows)
    assert run.dec.error_flags() == 0
    run.close()
    model = oracle.OracleModel(w)
    for i, b in enumerate(rows):
        ref = oracle_teacher(model, run.prompts[b], stream[:, b])
        what = f"{W.name} seq {b}"
        err = check_logits(z[:, i], ref, W.model.dtype, what)
        record(what, err, LOGIT_TOL[W.model.dtype], check_ids(ids[:, b], ref, what), rows=int(ref.shape[0]))
