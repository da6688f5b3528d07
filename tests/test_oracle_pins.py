"""Pins of the float64 oracle to facts outside itself (closed forms, invariants, library
routines, brute force). CPU only."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import decoder as od
import workloads as wl

RTOL = 1e-12


def rng(seed=123):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------------------------------------
# GELU-tanh ("bare-metal-llm", section "The bug worth telling"; "batch_forge", GELU overflow fix)
# ------------------------------------------------------------------------------------------------

def test_gelu_closed_form_values_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50

    def exact(v):
        v = mpmath.mpf(v)
        return 0.5 * v * (1 + mpmath.tanh(mpmath.sqrt(2 / mpmath.pi) * (v + mpmath.mpf("0.044715") * v ** 3)))

    xs = np.array([1.0, -1.0, 3.0, 0.5, -2.25, 4.0, 1e-3])
    got = od.gelu_tanh(xs)
    for x, g in zip(xs, got):
        assert abs(g - float(exact(x))) <= 1e-15 * max(1.0, abs(g)), x


def test_gelu_printed_closed_form_values():
    # fp64 closed-form values of GPT-2's GELU-tanh
    assert od.gelu_tanh(np.array([1.0]))[0] == pytest.approx(0.8411919906082768, rel=1e-15)
    assert od.gelu_tanh(np.array([-1.0]))[0] == pytest.approx(-0.15880800939172330, rel=1e-14)
    assert od.gelu_tanh(np.array([3.0]))[0] == pytest.approx(2.996362607918227, rel=1e-15)


def test_gelu_matches_torch_tanh_gelu_below_clamp():
    x = np.linspace(-6.4, 6.4, 20001)        # |arg| < 15 on this range
    ref = F.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(od.gelu_tanh(x), ref, rtol=1e-14, atol=1e-15)


def test_gelu_within_textbook_bound_of_erf_gelu():
    from scipy.special import erf
    x = np.linspace(-12, 12, 400001)
    exact = 0.5 * x * (1 + erf(x / math.sqrt(2)))
    assert np.abs(od.gelu_tanh(x) - exact).max() < 5e-4


def test_gelu_saturates_without_nan():
    x = np.array([7.0, 10.0, 100.0, 1e3, 1e4])
    pos = od.gelu_tanh(x)
    neg = od.gelu_tanh(-x)
    assert np.all(np.isfinite(pos)) and np.all(np.isfinite(neg))
    np.testing.assert_allclose(pos, x, rtol=1e-12)
    assert np.all(np.abs(neg) <= 1e-12 * x)
    # the clamp is active exactly past |arg| = 15
    assert od.gelu_tanh_arg(np.array([6.5]))[0] < 15 < od.gelu_tanh_arg(np.array([7.0]))[0]


def test_gelu_clamp_is_what_keeps_float32_finite():
    """In float32, tanh written through exp(2u) overflows to inf/inf = NaN past |u| ~ 44
    (the failure the pages describe); the clamped argument never gets there."""
    x = np.float32(1e4)
    u = np.float32(od.GELU_C) * (x + np.float32(od.GELU_CUBIC) * x * x * x)

    def tanh_via_exp(v):
        with np.errstate(over="ignore", invalid="ignore"):
            e = np.exp(np.float32(2) * v)
            return (e - np.float32(1)) / (e + np.float32(1))

    assert np.isnan(tanh_via_exp(np.float32(u)))
    uc = np.clip(u, np.float32(-od.GELU_TANH_CLAMP), np.float32(od.GELU_TANH_CLAMP))
    t = tanh_via_exp(uc)
    assert np.isfinite(t) and t == np.float32(1.0)     # tanh(15) rounds to 1 in float32


# ------------------------------------------------------------------------------------------------
# softmax, norms, RoPE
# ------------------------------------------------------------------------------------------------

def test_softmax_rows_sum_to_one_and_shift_invariant():
    s = rng().normal(size=(64, 300)) * 10
    p = od.softmax(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-15 * 300)
    np.testing.assert_allclose(od.softmax(s + 123.25), p, rtol=1e-12, atol=1e-300)
    s2 = s.copy()
    s2[:, 200:] = -np.inf
    p2 = od.softmax(s2)
    assert np.all(p2[:, 200:] == 0.0)
    np.testing.assert_allclose(p2[:, :200], od.softmax(s[:, :200]), rtol=1e-12)


def test_layer_norm_matches_torch_and_invariants():
    r = rng()
    x = r.normal(size=(17, 768)) * 3 + 0.7
    g = r.normal(size=768)
    b = r.normal(size=768)
    ref = F.layer_norm(torch.from_numpy(x), (768,), torch.from_numpy(g), torch.from_numpy(b), eps=1e-5).numpy()
    np.testing.assert_allclose(od.layer_norm(x, g, b, 1e-5), ref, rtol=1e-12, atol=1e-12)
    y = od.layer_norm(x, np.ones(768), np.zeros(768), 1e-5)
    var = x.var(-1)
    np.testing.assert_allclose(y.mean(-1), 0.0, atol=1e-13)
    np.testing.assert_allclose(y.var(-1), var / (var + 1e-5), rtol=1e-12)


def test_rms_norm_matches_torch_and_invariants():
    r = rng(7)
    x = r.normal(size=(9, 960)) * 0.01       # small rows so eps matters
    g = r.normal(size=960)
    ref = F.rms_norm(torch.from_numpy(x), (960,), torch.from_numpy(g), eps=1e-5).numpy()
    np.testing.assert_allclose(od.rms_norm(x, g, 1e-5), ref, rtol=1e-12, atol=1e-15)
    y = od.rms_norm(x, np.ones(960), 1e-5)
    ms = (x * x).mean(-1)
    np.testing.assert_allclose(np.sqrt((y * y).mean(-1)), np.sqrt(ms / (ms + 1e-5)), rtol=1e-12)


def test_rope_invariants():
    r = rng(3)
    hd, theta = 64, 1e5
    x = r.normal(size=(5, 3, hd))
    pos = np.array([0, 1, 7, 100, 2047])
    y = od.rope(x, pos, theta)
    # pos 0 is the identity
    np.testing.assert_array_equal(y[0], x[0])
    # each (i, i + hd/2) pair keeps its norm
    n0 = x[..., :32] ** 2 + x[..., 32:] ** 2
    n1 = y[..., :32] ** 2 + y[..., 32:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-14)
    # pair 0 turns by exactly `pos` radians (its frequency is theta^0 = 1)
    z0 = x[:, :, 0] + 1j * x[:, :, 32]
    z1 = y[:, :, 0] + 1j * y[:, :, 32]
    np.testing.assert_allclose(z1, z0 * np.exp(1j * pos)[:, None], rtol=1e-13)
    # neighbouring pairs' frequencies differ by the factor theta^(2/hd): turn every pair
    # at pos = 1 and read the angles back from the complex ratio
    e = np.zeros((1, 1, hd))
    e[..., :32] = 1.0
    w = od.rope(e, np.array([1]), theta)[0, 0]
    ang = np.angle(w[:32] + 1j * w[32:])
    np.testing.assert_allclose(ang[1:] / ang[:-1], theta ** (-2.0 / hd), rtol=1e-12)


def test_rope_scores_depend_only_on_relative_position():
    r = rng(4)
    q = r.normal(size=(1, 1, 64))
    k = r.normal(size=(1, 1, 64))

    def score(m, n):
        return float((od.rope(q, np.array([m]), 1e5) * od.rope(k, np.array([n]), 1e5)).sum())

    for m, n in [(5, 2), (105, 102), (2003, 2000)]:
        assert score(m, n) == pytest.approx(score(3, 0), rel=1e-11)


# ------------------------------------------------------------------------------------------------
# attention
# ------------------------------------------------------------------------------------------------

def test_causal_attention_matches_torch_sdpa_with_gqa():
    r = rng(11)
    T, hq, hkv, hd = 13, 6, 2, 16
    q, k, v = r.normal(size=(T, hq, hd)), r.normal(size=(T, hkv, hd)), r.normal(size=(T, hkv, hd))
    got = od.causal_attention(q, k, v, np.arange(T)).reshape(T, hq, hd)
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    r = rng(12)
    hd = 8
    # one key: the output is that key's value
    v = r.normal(size=(1, 2, hd))
    out = od.causal_attention(r.normal(size=(1, 2, hd)), r.normal(size=(1, 2, hd)), v, np.array([0]))
    np.testing.assert_allclose(out.reshape(2, hd), v[0], rtol=1e-15)
    # equal keys: uniform weights, the output is the mean of the visible values
    T = 6
    k = np.tile(r.normal(size=(1, 1, hd)), (T, 1, 1))
    v = r.normal(size=(T, 1, hd))
    out = od.causal_attention(r.normal(size=(T, 1, hd)), k, v, np.arange(T))
    for t in range(T):
        np.testing.assert_allclose(out[t], v[: t + 1, 0].mean(0), rtol=1e-12)


def test_gqa_equals_mha_with_repeated_kv():
    r = rng(13)
    T, hq, hkv, hd = 7, 6, 3, 8
    q, k, v = r.normal(size=(T, hq, hd)), r.normal(size=(T, hkv, hd)), r.normal(size=(T, hkv, hd))
    rep = hq // hkv
    a = od.causal_attention(q, k, v, np.arange(T))
    b = od.causal_attention(q, np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1), np.arange(T))
    np.testing.assert_allclose(a, b, rtol=1e-15)


# ------------------------------------------------------------------------------------------------
# argmax rule ("rvllm-metal": argmax tested with ties and NaN)
# ------------------------------------------------------------------------------------------------

def test_argmax_rule_ties_and_nan():
    assert od.argmax_rule(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert od.argmax_rule(np.array([-np.inf, -np.inf])) == 0
    assert od.argmax_rule(np.array([1.0, np.nan, 5.0, np.nan])) == 1
    assert od.argmax_rule(np.array([np.inf, 1.0, np.inf])) == 0
    assert od.top2_margin(np.array([0.5, 2.0, 1.25])) == pytest.approx(0.75)
    z = rng().normal(size=1000)
    assert od.argmax_rule(z) == int(np.argmax(z))


# ------------------------------------------------------------------------------------------------
# whole model: brute force, cache == recompute, causality, reductions
# ------------------------------------------------------------------------------------------------

TINY = [
    wl.tiny_shape(wl.ARCH_GPT2),
    wl.tiny_shape(wl.ARCH_LLAMA, n_heads=4, n_kv_heads=2, head_dim=4, d_model=8, rope_theta=1e4),
    wl.tiny_shape(wl.ARCH_GPT2, n_layers=2, dtype=wl.DTYPE_BF16),
    wl.tiny_shape(wl.ARCH_LLAMA, n_layers=2, n_heads=2, n_kv_heads=1, dtype=wl.DTYPE_BF16),
]


@pytest.mark.parametrize("shape", TINY, ids=["gpt2", "llama-gqa", "gpt2-bf16-2l", "llama-bf16-2l"])
def test_brute_force_equals_vectorised_oracle(shape):
    w = wl.make_weights(shape, scale=20.0, perturb=True)   # large weights: non-trivial softmax / GELU
    tokens = [3, 10, 0, 7, 7, 1]
    brute = np.array(oracle.BruteModel(w).run(tokens))
    m = oracle.OracleModel(w)
    full = oracle.forward_full(m, tokens)
    np.testing.assert_allclose(full, brute, rtol=RTOL, atol=1e-12)
    seq = oracle.Sequence(m)
    step = np.stack([seq.step(t) for t in tokens])
    np.testing.assert_allclose(step, brute, rtol=RTOL, atol=1e-12)


SMALL = [
    wl.ModelShape("small-gpt2", wl.ARCH_GPT2, wl.DTYPE_F32, 2, 128, 2, 2, 64, 256, 97, 64),
    wl.ModelShape("small-llama", wl.ARCH_LLAMA, wl.DTYPE_BF16, 2, 192, 3, 1, 64, 160, 101, 64),
]


@pytest.mark.parametrize("shape", SMALL, ids=["gpt2", "llama"])
def test_cached_decode_equals_stateless_recompute(shape):
    w = wl.make_weights(shape, perturb=True)
    m = oracle.OracleModel(w)
    toks = wl.draw_prompts([21], shape.vocab)[0]
    full = oracle.forward_full(m, toks)
    # prefill 9 tokens, then one token at a time
    seq = oracle.Sequence(m)
    z = [seq.feed(toks[:9], all_logits=True)]
    for t in toks[9:]:
        z.append(seq.feed([t]))
    cached = np.concatenate(z)
    np.testing.assert_allclose(cached, full, rtol=RTOL, atol=1e-12)
    # a stateless recompute at step t gives the same last row
    for t in (9, 15, 20):
        np.testing.assert_allclose(oracle.forward_full(m, toks[: t + 1], last_only=True)[0], full[t],
                                   rtol=RTOL, atol=1e-12)


@pytest.mark.parametrize("shape", SMALL, ids=["gpt2", "llama"])
def test_causal_mask_future_tokens_do_not_change_past_logits(shape):
    m = oracle.OracleModel(wl.make_weights(shape, perturb=True))
    a = wl.draw_prompts([12], shape.vocab)[0]
    b = a.copy()
    b[7:] = (b[7:] + 5) % shape.vocab
    za, zb = oracle.forward_full(m, a), oracle.forward_full(m, b)
    np.testing.assert_array_equal(za[:7], zb[:7])
    assert np.abs(za[7:] - zb[7:]).max() > 0


def test_zero_weight_layer_is_identity_on_residual():
    shape = SMALL[0]
    w = wl.make_weights(shape, perturb=False)
    for l in range(shape.n_layers):
        w.w_o[l][:] = 0
        w.w_down[l][:] = 0
    m = oracle.OracleModel(w)
    h = np.random.default_rng(0).normal(size=(5, shape.d_model))
    out, _, _ = m.layer(0, h, np.arange(5), None, None)
    np.testing.assert_array_equal(out, h)


def test_magnitude_scaled_gpt2_drives_gelu_argument_past_clamp():
    """The x8 GPT-2 copy pushes the GELU tanh argument past 15 (so the clamp is exercised)."""
    from dataclasses import replace
    shape = replace(wl.GPT2_124M_F32, n_layers=1)
    m = oracle.OracleModel(wl.make_weights(shape, scale=8.0))
    seq = oracle.Sequence(m)
    z = seq.prefill(wl.draw_prompts([32], shape.vocab)[0])
    assert np.all(np.isfinite(z))
    assert m.stats["max_gelu_arg"] > 15.0


# ------------------------------------------------------------------------------------------------
# input generators (host logic shared by both sides)
# ------------------------------------------------------------------------------------------------

def test_bf16_rounding_matches_torch():
    x = np.concatenate([rng(5).normal(size=100000).astype(np.float32) * 0.02,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 65504.0, 1e-30], np.float32)])
    ours = wl.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(wl.bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_block_tables_are_a_partition_of_the_pool():
    lens = wl.draw_lengths(64, 64, 2048)
    assert lens.min() >= 64 and lens.max() <= 2048
    ctx = lens + 1
    tables, n = wl.make_block_tables(ctx, 129, shuffle=True)
    used = np.concatenate([tables[b, : wl.blocks_needed(c)] for b, c in enumerate(ctx)])
    assert sorted(used.tolist()) == list(range(n))
    assert np.all(tables[tables >= 0] < n)
    # shuffled: not the identity assignment
    ident, _ = wl.make_block_tables(ctx, 129, shuffle=False)
    assert not np.array_equal(tables, ident)


def test_weight_draws_are_reproducible_and_scaled():
    s = SMALL[0]
    a = wl.make_weights(s)
    b = wl.make_weights(s, scale=8.0)
    np.testing.assert_array_equal(a.w_qkv[1] * np.float32(8), b.w_qkv[1])
    assert abs(a.tok_emb.std() - 0.02) < 1e-3
    assert np.all(a.ln1_w[0] == 1) and np.all(a.b_o[0] == 0)


# ------------------------------------------------------------------------------------------------
# greedy generation ("bare-metal-llm", "What got built": prefill, then one token at a time, each
# new token the argmax of the previous step's logits)
# ------------------------------------------------------------------------------------------------

GREEDY = [
    (TINY[0], [3, 10, 0], 6),
    (TINY[1], [2, 8], 6),
    (SMALL[0], [2, 96, 17], 8),
    (SMALL[1], [2, 96, 17], 8),
]


@pytest.mark.parametrize("shape,prompt,steps", GREEDY, ids=["tiny-gpt2", "tiny-llama", "small-gpt2", "small-llama"])
def test_greedy_generate_is_the_argmax_chain_of_stateless_recomputes(shape, prompt, steps):
    """ids[i] is the argmax of the stateless recompute over prompt + ids[:i], and the logits the
    generator returns are that recompute's last row. Feeding back a wrong token (an older id, or
    the argmax of another row) changes the chain and fails here."""
    w = wl.make_weights(shape, scale=20.0 if shape.d_model <= 8 else 8.0, perturb=True)
    m = oracle.OracleModel(w)
    ids, zs = oracle.greedy_generate(m, prompt, steps)
    assert ids.shape == (steps + 1,) and zs.shape == (steps + 1, shape.vocab)
    assert len(set(ids.tolist())) > 1, "a constant stream would not tell which id was fed back"
    for i in range(steps + 1):
        ctx = list(prompt) + [int(t) for t in ids[:i]]
        z = oracle.forward_full(m, ctx, last_only=True)[0]
        np.testing.assert_allclose(zs[i], z, rtol=RTOL, atol=1e-12)
        assert int(ids[i]) == oracle.argmax_rule(z)
    if shape.d_model <= 8:
        # the scalar-loop model, fed the same chain, agrees row by row
        brute = np.array(oracle.BruteModel(w).run(list(prompt) + [int(t) for t in ids[:-1]]))
        np.testing.assert_allclose(zs, brute[len(prompt) - 1:], rtol=RTOL, atol=1e-12)
        assert [oracle.argmax_rule(z) for z in brute[len(prompt) - 1:]] == ids.tolist()


# ------------------------------------------------------------------------------------------------
# the float32 floor of the GPT-2 workloads (why the magnitude-scaled copy has a wider logit bound)
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("W", [wl.W_GPT2_F32_B32, wl.W_GPT2_F32_B32_X8], ids=["x1", "x8"])
def test_float32_floor_of_gpt2_workloads(W):
    """A plain float32 evaluation of the same definition (NumPy/BLAS, no GPU) against the float64
    oracle on one sequence of the batch-32 workload (its 128 prompt rows and 64 teacher-forced
    rows). On the x1 model it agrees to ~3e-6, far inside the 2e-3 bound. On the x8 copy (every
    weight x8) the logits are 8x larger and the model amplifies rounding: float32 itself misses
    float64 by more than 2e-3, so no float32 program can meet the literal fp32 bound there and
    the GPU test measures this floor and bounds the GPU by a small multiple of it."""
    from fp32_eval import gpt2_forward_f32
    w = wl.make_weights(W.model, scale=W.weight_scale)
    m = oracle.OracleModel(w)
    prompt = wl.draw_prompts(W.lengths(), W.model.vocab)[0]
    stream = wl.draw_stream(W.batch, W.decode_steps, W.model.vocab)[:64, 0]
    toks = np.concatenate([prompt, stream])
    gap = float(np.abs(gpt2_forward_f32(w, toks) - oracle.forward_full(m, toks)).max())
    if W.weight_scale == 1.0:
        assert gap < 2e-4, gap
    else:
        assert gap > 2e-3, gap
        assert gap < 2e-2, gap


# ------------------------------------------------------------------------------------------------
# bf16 KV cache ("rvllm-metal", section "What's basic about it": the F32 cache as a weakness)
# ------------------------------------------------------------------------------------------------

def test_round_bf16_matches_torch_and_bounds():
    x = np.concatenate([rng(21).normal(size=200000).astype(np.float32) * 3,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0, 1e-30], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = od.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(od.round_bf16(got), got)                 # idempotent
    assert np.all(np.abs(got - x) <= 2.0 ** -8 * np.abs(x))                # half an ulp of 8 significant bits


@pytest.mark.parametrize("shape", TINY[:2], ids=["gpt2", "llama-gqa"])
def test_bf16_kv_brute_force_equals_vectorised_oracle(shape):
    w = wl.make_weights(shape, scale=20.0, perturb=True)
    tokens = [3, 10, 0, 7, 7, 1]
    brute = np.array(oracle.BruteModel(w, kv_dtype=wl.DTYPE_BF16).run(tokens))
    m = oracle.OracleModel(w, kv_dtype=wl.DTYPE_BF16)
    np.testing.assert_allclose(oracle.forward_full(m, tokens), brute, rtol=RTOL, atol=1e-12)
    seq = oracle.Sequence(m)
    np.testing.assert_allclose(np.stack([seq.step(t) for t in tokens]), brute, rtol=RTOL, atol=1e-12)
    # the rounding is there: the fp32-cache model differs
    assert np.abs(np.array(oracle.BruteModel(w).run(tokens)) - brute).max() > 1e-6


# ------------------------------------------------------------------------------------------------
# temperature / top-k sampling ("batch_forge", component table: greedy, temperature, top-k)
# ------------------------------------------------------------------------------------------------

def test_sample_top_k_reduces_to_greedy():
    z = rng(31).normal(size=500)
    for u in (0.0, 0.3, 0.999):
        assert od.sample_top_k(z, 0.7, 1, u) == od.argmax_rule(z)      # k = 1
        assert od.sample_top_k(z, 0.0, 40, u) == od.argmax_rule(z)     # T = 0
        assert od.sample_top_k(z, 1e-6, 40, u) == od.argmax_rule(z)    # T -> 0
    assert od.sample_top_k(z, 0.9, 40, 0.0) == od.argmax_rule(z)       # u = 0: the top candidate
    zn = z.copy()
    zn[[7, 300]] = np.nan
    assert od.sample_top_k(zn, 0.9, 40, 0.5) == 7                      # NaN: the argmax rule


def test_sample_top_k_frequencies_are_the_truncated_softmax():
    """Over a uniform grid of u the chosen tokens' frequencies equal the temperature softmax
    restricted to the k largest logits (closed form, to 1/N)."""
    z = rng(32).normal(size=300) * 2
    T, k, N = 0.8, 12, 20000
    top = np.argsort(-z, kind="stable")[:k]
    p = np.exp((z[top] - z[top].max()) / T)
    p /= p.sum()
    counts = np.zeros(z.size)
    for u in (np.arange(N) + 0.5) / N:
        counts[od.sample_top_k(z, T, k, u)] += 1
    assert set(np.flatnonzero(counts)) <= set(top.tolist())
    np.testing.assert_allclose(counts[top] / N, p, atol=1.5 / N)
    # adding a constant to every logit changes nothing
    assert all(od.sample_top_k(z + 3.25, T, k, u) == od.sample_top_k(z, T, k, u) for u in (0.1, 0.5, 0.93))


def test_sample_top_k_tie_at_the_cut_keeps_the_lower_index():
    z = np.array([5.0, 1.0, 3.0, 3.0, 0.5, 3.0])
    # k = 2: candidates 0 and the lowest-index 3.0 (index 2); a u past token 0's share picks 2
    p0 = 1.0 / (1.0 + np.exp(-2.0))
    assert od.sample_top_k(z, 1.0, 2, p0 + 1e-6) == 2
    assert od.sample_top_k(z, 1.0, 2, p0 - 1e-6) == 0
    # k = 3: candidates 0, 2, 3; the last share belongs to index 3
    assert od.sample_top_k(z, 1.0, 3, 0.999999) == 3


# ------------------------------------------------------------------------------------------------
# model-feature variants ("rvllm-metal", section "What the kernels do", last paragraph: Llama 3
# RoPE scaling, Qwen2 attention biases, Qwen3 Q/K norm, Gemma's sliding window)
# ------------------------------------------------------------------------------------------------

LLAMA3_SCALING = (8.0, 1.0, 4.0, 8192)


def test_llama3_rope_scaling_regions():
    hd, theta = 128, 5e5
    f = theta ** (-(2.0 * np.arange(hd // 2)) / hd)
    g = od.llama3_scaled_inv_freq(f, *LLAMA3_SCALING)
    wl_ = 2 * np.pi / f
    hi_wl, lo_wl = 8192 / 4.0, 8192 / 1.0
    np.testing.assert_array_equal(g[wl_ < hi_wl], f[wl_ < hi_wl])                  # fast pairs kept
    np.testing.assert_allclose(g[wl_ > lo_wl], f[wl_ > lo_wl] / 8.0, rtol=1e-15)   # slow pairs / factor
    mid = (wl_ >= hi_wl) & (wl_ <= lo_wl)
    assert mid.any() and np.all(g[mid] <= f[mid]) and np.all(g[mid] >= f[mid] / 8.0)
    assert np.all(np.diff(g) < 0)                                                  # still ordered
    # the blend is continuous at both ends of the middle band
    for w_edge, want in ((hi_wl, 1.0), (lo_wl, 1.0 / 8.0)):
        fe = 2 * np.pi / w_edge
        got = od.llama3_scaled_inv_freq(np.array([fe * (1 - 1e-12), fe * (1 + 1e-12)]), *LLAMA3_SCALING)
        np.testing.assert_allclose(got / fe, want, rtol=1e-9)


def test_sliding_window_attention_special_cases_and_torch():
    r = rng(41)
    T, hq, hkv, hd = 11, 4, 2, 8
    q, k, v = r.normal(size=(T, hq, hd)), r.normal(size=(T, hkv, hd)), r.normal(size=(T, hkv, hd))
    pos = np.arange(T)
    full = od.causal_attention(q, k, v, pos)
    np.testing.assert_array_equal(od.causal_attention(q, k, v, pos, window=T), full)    # W >= T: plain causal
    one = od.causal_attention(q, k, v, pos, window=1).reshape(T, hq, hd)               # W = 1: itself only
    np.testing.assert_allclose(one, np.repeat(v, hq // hkv, axis=1), rtol=1e-15)
    W = 4
    i, j = np.arange(T)[:, None], np.arange(T)[None, :]
    allowed = torch.from_numpy((j <= i) & (j > i - W))
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=allowed).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(od.causal_attention(q, k, v, pos, window=W).reshape(T, hq, hd), ref,
                               rtol=1e-12, atol=1e-13)


VARIANTS = [
    wl.tiny_shape(wl.ARCH_LLAMA, n_heads=4, n_kv_heads=2, rope_theta=1e4, qk_norm=True, attn_bias=True,
                  rope_scaling=(4.0, 1.0, 4.0, 8), sliding_window=3),
    wl.tiny_shape(wl.ARCH_LLAMA, n_layers=2, n_heads=2, n_kv_heads=1, sliding_window=2, sliding_window_pattern=2,
                  dtype=wl.DTYPE_BF16),
    wl.tiny_shape(wl.ARCH_GPT2, sliding_window=3),
]


@pytest.mark.parametrize("shape", VARIANTS, ids=["llama-all-features", "llama-window-pattern", "gpt2-window"])
def test_feature_variants_brute_force_equals_vectorised_oracle(shape):
    w = wl.make_weights(shape, scale=20.0, perturb=True)
    tokens = [3, 10, 0, 7, 7, 1]
    brute = np.array(oracle.BruteModel(w).run(tokens))
    m = oracle.OracleModel(w)
    np.testing.assert_allclose(oracle.forward_full(m, tokens), brute, rtol=RTOL, atol=1e-12)
    seq = oracle.Sequence(m)
    np.testing.assert_allclose(np.stack([seq.step(t) for t in tokens]), brute, rtol=RTOL, atol=1e-12)
    # every feature changes the result (none is silently dropped)
    from dataclasses import replace
    for off in (dict(sliding_window=0), dict(qk_norm=False), dict(rope_scaling=None), dict(attn_bias=False)):
        key, val = next(iter(off.items()))
        if getattr(shape, key) == val:
            continue
        w2 = wl.make_weights(replace(shape, **off), scale=20.0, perturb=True)
        assert np.abs(oracle.forward_full(oracle.OracleModel(w2), tokens) - brute).max() > 1e-6, key


def test_qk_norm_gives_unit_rms_heads():
    r = rng(43)
    q = r.normal(size=(5, 3, 64)) * 0.1
    y = od.rms_norm(q, np.ones(64), 1e-5)
    ms = (q * q).mean(-1)
    np.testing.assert_allclose(np.sqrt((y * y).mean(-1)), np.sqrt(ms / (ms + 1e-5)), rtol=1e-12)


# ------------------------------------------------------------------------------------------------
# Q8_0 weights ("rvllm-metal", sections "What's basic about it" and "What's next")
# ------------------------------------------------------------------------------------------------

Q8_TINY = [wl.tiny_shape(wl.ARCH_GPT2, dtype=wl.DTYPE_Q8, d_model=64, d_ff=64, n_heads=2, head_dim=32),
           wl.tiny_shape(wl.ARCH_LLAMA, dtype=wl.DTYPE_Q8, d_model=64, d_ff=32, n_heads=2, n_kv_heads=1,
                         head_dim=32)]


@pytest.mark.parametrize("shape", Q8_TINY, ids=["gpt2-q8", "llama-q8"])
def test_q8_brute_force_equals_vectorised_oracle(shape):
    w = wl.make_weights(shape, scale=20.0, perturb=True)
    tokens = [3, 10, 0, 7]
    brute = np.array(oracle.BruteModel(w).run(tokens))
    m = oracle.OracleModel(w)
    np.testing.assert_allclose(oracle.forward_full(m, tokens), brute, rtol=RTOL, atol=1e-12)


def test_q8_dequant_is_block_scale_times_quant_and_close_to_the_draw():
    from dataclasses import replace
    sq = wl.tiny_shape(wl.ARCH_GPT2, dtype=wl.DTYPE_Q8, d_model=64, d_ff=64, n_heads=2, head_dim=32)
    wq = wl.make_weights(sq)
    wf = wl.make_weights(replace(sq, dtype=wl.DTYPE_F32))            # the same float32 draws
    deq = od.dequant_q8_0(wq.w_up[0], wq.w_up_scale[0])
    # value (r, j) = d[r, j // 32] * q[r, j], written out element by element
    r, j = 5, 45
    assert deq[r, j] == float(wq.w_up_scale[0][r, j // 32]) * float(wq.w_up[0][r, j])
    # within half a quantization step of the float32 draw, and the block maximum maps to +-127
    step = np.repeat(wq.w_up_scale[0].astype(np.float64), 32, axis=1)
    assert np.all(np.abs(deq - wf.w_up[0]) <= 0.5 * step * (1 + 1e-3) + 1e-12)
    assert np.abs(wq.w_up[0]).max() == 127
