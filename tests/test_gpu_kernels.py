"""Each projection kernel forced on awkward shapes, against the oracle's linear (GPU only)."""
import numpy as np
import pytest

import workloads as wl
from oracle import OracleModel

pytestmark = pytest.mark.gpu

SHAPES = [(1, 33, 8), (3, 130, 768), (7, 64, 960), (16, 2304, 768), (32, 768, 3072), (64, 1000, 192),
          (127, 130, 64), (128, 256, 1000), (300, 576, 384), (1030, 200, 136)]


def _inputs(M, N, K, bf16, seed):
    r = np.random.default_rng(seed)
    x = r.standard_normal((M, K), dtype=np.float32)
    w = (r.standard_normal((N, K), dtype=np.float32) * np.float32(0.05))
    b = r.standard_normal(N, dtype=np.float32) * np.float32(0.1)
    if bf16:
        w, b = (wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(a)) for a in (w, b))
    return x, w, b


def bf16_pair(x):
    """The library's activation storage for bf16 weights: row m = bf16 hi[0..K) then lo[0..K),
    hi = bf16(x), lo = bf16(x - hi). Returns (uint16 bits [M, 2K], the represented values hi + lo)."""
    hi_bits = wl.f32_to_bf16_bits(x)
    hi = wl.bf16_bits_to_f32(hi_bits)
    lo_bits = wl.f32_to_bf16_bits((x - hi).astype(np.float32))
    val = hi.astype(np.float64) + wl.bf16_bits_to_f32(lo_bits).astype(np.float64)
    return np.concatenate([hi_bits, lo_bits], axis=1), val


@pytest.mark.parametrize("variant", [1, 2, 3, 4, 5], ids=["gemv", "simt", "tcgen05", "tcgen05-swap", "tcgen05-pair"])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_kernel_matches_oracle(gpu_lib, variant, bf16, M, N, K):
    import torch
    if variant in (3, 5) and not bf16:
        pytest.skip("tcgen05 paths with activations on N are bf16 only")
    if variant == 1 and M > 64:
        pytest.skip("the weight-stream GEMV serves decode row counts")
    if variant == 4 and M > 256:
        pytest.skip("weights-on-M path serves at most 256 rows")
    x, w, b = _inputs(M, N, K, bf16, seed=M * 7 + N + K)
    dt = torch.bfloat16 if bf16 else torch.float32
    tw, tb = (torch.from_numpy(a).cuda().to(dt) for a in (w, b))
    if bf16:
        bits, xv = bf16_pair(x)
        tx = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        xv = x.astype(np.float64)
        tx = torch.from_numpy(x).cuda()
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    gpu_lib.op_linear(tx, tw, tb, y, variant)
    torch.cuda.synchronize()
    ref = OracleModel.linear(xv, w.astype(np.float64), b.astype(np.float64))
    got = y.cpu().numpy()
    # fp32 accumulation over K terms of size |x||w|: bound by K * 2^-23 * sum|x w| (+ margin).
    # The fp32 tensor-core path sums three tf32 products; the dropped low*low term and the
    # tf32 rounding of the low parts add about 2^-20 relative per product.
    scale = np.abs(xv) @ np.abs(w.astype(np.float64)).T + np.abs(b)
    tol = 1e-6 + 4 * K * 2.0 ** -23 * scale + (2.0 ** -19 * scale if (variant == 4 and not bf16) else 0)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= tol), float(np.abs(got - ref).max())


# ------------------------------------------------------------------------------------------------
# decode attention over a shuffled paged pool, against the oracle's causal attention
# ------------------------------------------------------------------------------------------------

def make_attention_case(B, H, Hkv, ctx_max, bf16, seed):
    """Random q and a shuffled paged K/V pool; returns host and device views."""
    import torch
    r = np.random.default_rng(seed)
    pos = r.integers(0, ctx_max, size=B).astype(np.int32)
    pos[0] = ctx_max - 1                                  # one row at the maximum context
    if B > 1:
        pos[1] = 0                                        # one row with a single key
    ctx = pos + 1
    mbps = wl.blocks_needed(int(ctx.max()))
    tables, nblk = wl.make_block_tables(ctx, mbps, shuffle=True, seed=seed)
    tables = np.where(tables < 0, 0, tables).astype(np.int32)
    k = r.standard_normal((nblk, Hkv, 16, 64), dtype=np.float32)
    v = r.standard_normal((nblk, Hkv, 16, 64), dtype=np.float32)
    q = r.standard_normal((B, H * 64), dtype=np.float32) * np.float32(0.5)
    if bf16:
        k, v = (wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(a)) for a in (k, v))
    dt = torch.bfloat16 if bf16 else torch.float32
    dev = dict(q=torch.from_numpy(q).cuda(), k=torch.from_numpy(k).cuda().to(dt), v=torch.from_numpy(v).cuda().to(dt),
               pos=torch.from_numpy(pos).cuda(), tables=torch.from_numpy(tables).cuda())
    return q, k, v, pos, tables, dev


def oracle_decode_attention(q, k, v, pos, tables, H, Hkv):
    from oracle import causal_attention
    out = []
    for b in range(len(pos)):
        t = np.arange(pos[b] + 1)
        blk = tables[b, t // 16]
        kk = k[blk, :, t % 16, :].astype(np.float64)     # [T, Hkv, 64]
        vv = v[blk, :, t % 16, :].astype(np.float64)
        qq = q[b].reshape(1, H, 64).astype(np.float64)
        out.append(causal_attention(qq, kk, vv, np.array([pos[b]]))[0])
    return np.stack(out)


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("B,H,Hkv,ctx", [(1, 12, 12, 1), (3, 12, 12, 200), (5, 15, 5, 2049), (4, 8, 1, 700),
                                         (64, 25, 25, 300), (80, 32, 16, 261)])
def test_decode_attention_matches_oracle(gpu_lib, bf16, B, H, Hkv, ctx):
    """Against the oracle on shuffled paged pools. The last two cases have enough (sequence, KV
    head) pairs for 1024-token chunks, where one or two query heads a KV head take the 8-warp,
    half-block instance (ctx 261: a ragged last half block)."""
    import torch
    q, k, v, pos, tables, d = make_attention_case(B, H, Hkv, ctx, bf16, seed=B + H + ctx)
    out = torch.full((B, H * 64), float("nan"), dtype=torch.float32, device="cuda")
    gpu_lib.op_attention_decode(d["q"], d["k"], d["v"], d["pos"], d["tables"], out, Hkv)
    torch.cuda.synchronize()
    ref = oracle_decode_attention(q, k, v, pos, tables, H, Hkv)
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=0, atol=2e-5)
