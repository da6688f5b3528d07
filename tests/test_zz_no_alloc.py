"""The allocation-free decode-attention entry point, for callers that cannot allocate.

Some callers cannot call cudaMalloc (code running inside another component's stream
capture, or a process whose own allocator owns all of HBM).
llm_op_attention_decode_noalloc serves them with its scratch in a fixed device array.
This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test. It must pass alone in a fresh process and
after the other tests.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _case(B, H, Hkv, ctx, bf16, seed):
    from test_gpu_kernels import make_attention_case
    return make_attention_case(B, H, Hkv, ctx, bf16, seed)


def test_noalloc_matches_allocating_entry_point_on_two_calls_in_a_row(gpu_lib):
    import torch
    # two different calls back to back: the shared array keeps the first call's contents,
    # the second call must not depend on them
    for (B, H, Hkv, ctx, bf16, seed) in [(6, 15, 5, 1500, True, 11), (3, 12, 12, 300, False, 12)]:
        _, _, _, _, _, d = _case(B, H, Hkv, ctx, bf16, seed)
        ref = torch.full((B, H * 64), float("nan"), dtype=torch.float32, device="cuda")
        got = torch.full_like(ref, float("nan"))
        gpu_lib.op_attention_decode(d["q"], d["k"], d["v"], d["pos"], d["tables"], ref, Hkv)
        gpu_lib.op_attention_decode(d["q"], d["k"], d["v"], d["pos"], d["tables"], got, Hkv, noalloc=True)
        torch.cuda.synchronize()
        g, r = got.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(g))
        np.testing.assert_allclose(g, r, rtol=0, atol=2e-5)


def test_noalloc_rejects_sizes_beyond_its_array(gpu_lib):
    import torch
    lib = gpu_lib.load()
    q = torch.zeros((1024, 16 * 64), dtype=torch.float32, device="cuda")
    pool = torch.zeros((1, 1, 16, 64), dtype=torch.float32, device="cuda")
    pos = torch.zeros(1024, dtype=torch.int32, device="cuda")
    tables = torch.zeros((1024, 512), dtype=torch.int32, device="cuda")
    st = lib.llm_op_attention_decode_noalloc(0, 1024, 16, 16, q.data_ptr(), pool.data_ptr(), pool.data_ptr(), 1,
                                             pos.data_ptr(), tables.data_ptr(), 512, q.data_ptr(),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 2
    assert b"fixed array" in lib.llm_last_error()
