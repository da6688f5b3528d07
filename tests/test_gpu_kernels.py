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
        x, w, b = (wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(a)) for a in (x, w, b))
    return x, w, b


@pytest.mark.parametrize("variant", [1, 2, 3], ids=["gemv", "simt", "tcgen05"])
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_kernel_matches_oracle(gpu_lib, variant, bf16, M, N, K):
    import torch
    if variant == 3 and not bf16:
        pytest.skip("tcgen05 path is bf16 only")
    if variant == 1 and M > 64:
        pytest.skip("the weight-stream GEMV serves decode row counts")
    x, w, b = _inputs(M, N, K, bf16, seed=M * 7 + N + K)
    dt = torch.bfloat16 if bf16 else torch.float32
    tx, tw, tb = (torch.from_numpy(a).cuda().to(dt) for a in (x, w, b))
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    gpu_lib.op_linear(tx, tw, tb, y, variant)
    torch.cuda.synchronize()
    ref = OracleModel.linear(x.astype(np.float64), w.astype(np.float64), b.astype(np.float64))
    got = y.cpu().numpy()
    # fp32 accumulation over K terms of size |x||w|: bound by K * 2^-23 * sum|x w| (+ margin)
    scale = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T + np.abs(b)
    tol = 1e-6 + 4 * K * 2.0 ** -23 * scale
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= tol), float(np.abs(got - ref).max())
