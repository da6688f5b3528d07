"""Temperature / top-k sampling on the GPU against the oracle's definition (GPU only).

The sampled token is an integer that floating point decides: the running sum of p against
u * sum(p). Each check is taken where that decision has a margin larger than the arithmetic
can move it; the rows close to a boundary are counted, and most rows must be checked.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from parity_util import check_logits
from test_gpu_parity import SMALL_GPT2, SMALL_LLAMA, small_workload

pytestmark = pytest.mark.gpu

LENGTHS = np.array([5, 17, 70, 33, 1, 9, 64, 40] * 8, dtype=np.int32)     # 64 sequences


def _boundary_distance(z, T, k, u):
    """Smallest |running sum / sum - u| over the candidates' cut points (float64)."""
    z = np.asarray(z, dtype=np.float64)
    order = np.lexsort((np.arange(z.size), -z))[:k]
    p = np.exp((z[order] - z[order[0]]) / T)
    c = np.cumsum(p) / p.sum()
    return float(np.abs(c[:-1] - u).min()) if k > 1 else 1.0


def _setup(shape):
    import torch
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    run = WorkloadRun(small_workload(shape), host_weights=w, lengths=LENGTHS)
    run.prefill()
    torch.cuda.synchronize()
    return w, run


@pytest.mark.parametrize("shape", [SMALL_GPT2, SMALL_LLAMA], ids=["gpt2-f32", "llama-bf16"])
def test_sampled_step_matches_the_definition(gpu_lib, shape):
    import torch
    w, run = _setup(shape)
    model = oracle.OracleModel(w)
    B, V = run.B, shape.vocab
    toks = torch.from_numpy(wl.draw_stream(B, 1, V)[0]).cuda()
    rng = np.random.default_rng(9)
    refs = None
    checked_gpu = checked_oracle = total = 0
    for T, k in [(0.8, 5), (1.0, 40), (0.6, 64), (1.3, 2), (0.9, 1)]:
        u = rng.random(B).astype(np.float32)
        ud = torch.from_numpy(u).cuda()
        z = torch.empty((B, V), dtype=torch.float32, device="cuda")
        ids = torch.zeros(B, dtype=torch.int32, device="cuda")
        run.decode_sample(toks, 0, T, k, ud, logits=z, next_ids=ids)   # same position each time: the
        torch.cuda.synchronize()                                       # step rewrites the same K/V slot
        assert run.dec.error_flags() == 0
        zg, ig = z.cpu().numpy().astype(np.float64), ids.cpu().numpy()
        if refs is None:
            refs = np.stack([oracle.teacher_forced(model, run.prompts[b], [int(toks[b])])[-1] for b in range(B)])
        err = check_logits(zg, refs, shape.dtype, f"{shape.name} sampled step logits")
        for b in range(B):
            total += 1
            # the kernel's decision, from its own logits (float32 arithmetic vs float64: 1e-4)
            if _boundary_distance(zg[b], T, k, u[b]) > 1e-4:
                assert int(ig[b]) == oracle.sample_top_k(zg[b], T, k, u[b]), (T, k, b)
                checked_gpu += 1
            # the whole step against the oracle's logits: a logit error e moves the running
            # sums by at most about 2 e / T relative
            if _boundary_distance(refs[b], T, k, u[b]) > 4 * err / T + 1e-4:
                assert int(ig[b]) == oracle.sample_top_k(refs[b], T, k, u[b]), (T, k, b)
                checked_oracle += 1
    assert checked_gpu >= 0.95 * total and checked_oracle >= 0.8 * total, (checked_gpu, checked_oracle, total)
    run.close()


def test_sampling_limits_reduce_to_the_argmax(gpu_lib):
    """top_k = 1, temperature 0, or no uniforms (u = 0) give the greedy step's ids bit for bit;
    the sampled step replayed from its graph follows each call's new uniforms."""
    import torch
    shape = SMALL_LLAMA
    w, run = _setup(shape)
    B, V = run.B, shape.vocab
    toks = torch.from_numpy(wl.draw_stream(B, 1, V)[0]).cuda()
    zg = torch.empty((B, V), dtype=torch.float32, device="cuda")
    greedy = torch.zeros(B, dtype=torch.int32, device="cuda")
    run.decode(toks, 0, logits=zg, next_ids=greedy)
    ud = torch.rand(B, device="cuda")
    for T, k, uu in [(0.8, 1, ud), (0.0, 40, ud), (0.8, 40, None)]:
        ids = torch.zeros(B, dtype=torch.int32, device="cuda")
        z = torch.empty((B, V), dtype=torch.float32, device="cuda")
        run.decode_sample(toks, 0, T, k, uu, logits=z, next_ids=ids)
        torch.cuda.synchronize()
        assert torch.equal(z, zg)
        assert torch.equal(ids, greedy), (T, k, uu is None)
    # replays of the captured sampled step with new draws
    zz = zg.cpu().numpy().astype(np.float64)
    for seed in (1, 2, 3):
        u = np.random.default_rng(seed).random(B).astype(np.float32)
        ids = torch.zeros(B, dtype=torch.int32, device="cuda")
        run.decode_sample(toks, 0, 1.0, 64, torch.from_numpy(u).cuda(), next_ids=ids)
        torch.cuda.synchronize()
        got = ids.cpu().numpy()
        for b in range(B):
            if _boundary_distance(zz[b], 1.0, 64, u[b]) > 1e-4:
                assert int(got[b]) == oracle.sample_top_k(zz[b], 1.0, 64, u[b])
    run.close()


def test_sampling_ties_keep_the_lower_index_and_nan_wins(gpu_lib):
    """Two equal head rows as each sequence's top two logits: with top_k = 2 and T = 1 they
    share the probability half and half, the lower index first; a NaN logit wins as in the
    argmax and sets the flag."""
    import torch
    import transformer_decoder_forward_gb300 as L
    from test_gpu_argmax import BATCH_LENGTHS, PAIRS, _final_normed_hidden, _safe_prompts, _set_row
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    shape = SMALL_GPT2
    pairs = PAIRS[shape.name]
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    prompts = _safe_prompts(BATCH_LENGTHS, shape.vocab, [j for p in pairs for j in p] + [65])
    stream = np.array([3, 9, 44, 7], dtype=np.int32)
    m = oracle.OracleModel(w)
    X = np.stack([_final_normed_hidden(m, list(prompts[b]) + [int(stream[b])]) for b in range(4)])
    base = np.stack([oracle.teacher_forced(m, prompts[b], [int(stream[b])])[-1] for b in range(4)])
    E = np.diag(base.max(axis=1) + 8.0) @ np.linalg.pinv(X.T)
    for b, (j1, j2) in enumerate(pairs):
        _set_row(w, j1, E[b])
        _set_row(w, j2, E[b])

    def run_with(weights, u):
        run = WorkloadRun(small_workload(shape), host_weights=weights, lengths=BATCH_LENGTHS)
        run.prompts = prompts
        run.tokens = torch.from_numpy(np.concatenate(prompts).astype(np.int32)).cuda()
        run.prefill()
        ids = torch.zeros(4, dtype=torch.int32, device="cuda")
        run.decode_sample(torch.from_numpy(stream).cuda(), 0, 1.0, 2, torch.tensor(u, device="cuda"), next_ids=ids)
        torch.cuda.synchronize()
        out, flags = ids.cpu().numpy(), run.dec.error_flags()
        run.close()
        return out, flags

    lo, flags = run_with(w, [0.25] * 4)
    assert flags == 0 and lo.tolist() == [p[0] for p in pairs]
    hi, _ = run_with(w, [0.75] * 4)
    assert hi.tolist() == [p[1] for p in pairs]
    _set_row(w, 65, np.full(shape.d_model, np.nan, dtype=np.float32))
    nan_ids, flags = run_with(w, [0.5] * 4)
    assert flags & L.FLAG_NAN_LOGIT and np.all(nan_ids == 65)
