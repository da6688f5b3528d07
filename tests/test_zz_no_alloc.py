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


def _driver():
    """The CUDA driver API through ctypes (libcuda ships with the driver): stream capture and
    graph inspection without going through any allocator."""
    lib = ctypes.CDLL("libcuda.so.1")
    vp = ctypes.c_void_p
    lib.cuStreamBeginCapture_v2.argtypes = [vp, ctypes.c_int]
    lib.cuStreamEndCapture.argtypes = [vp, ctypes.POINTER(vp)]
    lib.cuGraphGetNodes.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_size_t)]
    lib.cuGraphNodeGetType.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    lib.cuGraphInstantiateWithFlags.argtypes = [ctypes.POINTER(vp), vp, ctypes.c_ulonglong]
    lib.cuGraphLaunch.argtypes = [vp, vp]
    lib.cuGraphExecDestroy.argtypes = [vp]
    lib.cuGraphDestroy.argtypes = [vp]
    return lib


CU_STREAM_CAPTURE_MODE_GLOBAL = 0
CU_GRAPH_NODE_TYPE_MEM_ALLOC, CU_GRAPH_NODE_TYPE_MEM_FREE = 10, 11


def test_noalloc_runs_inside_a_stream_capture(gpu_lib):
    """The caller this entry point exists for: one that captures a CUDA graph and cannot let the
    library allocate inside it. After one eager call per KV dtype (which resolves the array's
    address and the kernels' attributes), the call is captured in global capture mode (where an
    allocating call would fail), the graph holds no memory-allocation node, and its replay
    matches the allocating entry point."""
    import torch
    cu = _driver()
    for (B, H, Hkv, ctx, bf16, seed) in [(6, 15, 5, 1500, True, 21), (3, 12, 12, 300, False, 22)]:
        _, _, _, _, _, d = _case(B, H, Hkv, ctx, bf16, seed)
        ref = torch.full((B, H * 64), float("nan"), dtype=torch.float32, device="cuda")
        got = torch.full_like(ref, float("nan"))
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            gpu_lib.op_attention_decode(d["q"], d["k"], d["v"], d["pos"], d["tables"], ref, Hkv, stream=s)
            gpu_lib.op_attention_decode(d["q"], d["k"], d["v"], d["pos"], d["tables"], got, Hkv, stream=s,
                                        noalloc=True)   # eager warm-up of this dtype
        s.synchronize()
        got.fill_(float("nan"))
        torch.cuda.synchronize()
        h = ctypes.c_void_p(s.cuda_stream)
        assert cu.cuStreamBeginCapture_v2(h, CU_STREAM_CAPTURE_MODE_GLOBAL) == 0
        try:
            gpu_lib.op_attention_decode(d["q"], d["k"], d["v"], d["pos"], d["tables"], got, Hkv, stream=s,
                                        noalloc=True)
        finally:
            graph = ctypes.c_void_p()
            rc = cu.cuStreamEndCapture(h, ctypes.byref(graph))
        assert rc == 0
        n = ctypes.c_size_t(0)
        assert cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) == 0 and n.value >= 2
        nodes = (ctypes.c_void_p * n.value)()
        assert cu.cuGraphGetNodes(graph, nodes, ctypes.byref(n)) == 0
        types = []
        for i in range(n.value):
            t = ctypes.c_int(-1)
            assert cu.cuGraphNodeGetType(nodes[i], ctypes.byref(t)) == 0
            types.append(t.value)
        assert CU_GRAPH_NODE_TYPE_MEM_ALLOC not in types and CU_GRAPH_NODE_TYPE_MEM_FREE not in types, types
        exe = ctypes.c_void_p()
        assert cu.cuGraphInstantiateWithFlags(ctypes.byref(exe), graph, 0) == 0
        assert cu.cuGraphLaunch(exe, h) == 0
        s.synchronize()
        cu.cuGraphExecDestroy(exe)
        cu.cuGraphDestroy(graph)
        g, r = got.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(g))
        np.testing.assert_allclose(g, r, rtol=0, atol=2e-5)
