"""The C-ABI library loads, exports every function include/*.h declares, and rejects bad
arguments on the host. No GPU and no compute call."""
import ctypes
import glob
import os
import re

import pytest

import transformer_decoder_forward_gb300 as L
from transformer_decoder_forward_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(llm_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert "llm_create" in names and "llm_decode_step" in names and "llm_prefill" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(L.EXPORTS) <= set(names)


def gpt2_config(**kw):
    c = L.LLMConfig(arch=0, dtype=0, n_layers=2, d_model=128, n_heads=2, n_kv_heads=2, head_dim=64, d_ff=256,
                    vocab=100, n_ctx=64, norm_eps=1e-5, rope_theta=1e5, kv_block_size=16, num_kv_blocks=8,
                    max_batch=2, max_blocks_per_seq=4, max_prefill_tokens=64, contiguous_kv=0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def fake_weights(n_layers=2):
    arrs = []

    def arr():
        a = (ctypes.c_void_p * n_layers)(*([0x1000] * n_layers))
        arrs.append(a)
        return ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p))

    w = L.LLMWeights(tok_emb=0x1000, pos_emb=0x1000, lnf_w=0x1000, lnf_b=0x1000)
    for k in ("ln1_w", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_w", "ln2_b", "w_up", "b_up", "w_down", "b_down"):
        setattr(w, k, arr())
    return w, arrs


def create(lib, cfg, w):
    h = ctypes.c_void_p(123)
    st = lib.llm_create(ctypes.byref(cfg) if cfg is not None else None, ctypes.byref(w) if w is not None else None,
                        None, ctypes.byref(h))
    return st, h


def test_create_validates_arguments_before_touching_a_device(lib):
    w, _keep = fake_weights()
    st, h = create(lib, None, w)
    assert st == 1 and h.value is None
    assert create(lib, gpt2_config(head_dim=128), w)[0] == 4
    assert create(lib, gpt2_config(kv_block_size=32), w)[0] == 4
    assert create(lib, gpt2_config(n_heads=3, n_kv_heads=2), w)[0] == 1
    assert create(lib, gpt2_config(d_model=0), w)[0] == 1
    assert create(lib, gpt2_config(num_kv_blocks=0), w)[0] == 1
    assert create(lib, gpt2_config(arch=7), w)[0] == 1
    w.b_qkv = None
    assert create(lib, gpt2_config(), w)[0] == 1
    assert b"bias" in lib.llm_last_error()


def test_create_without_a_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    w, _keep = fake_weights()
    st, h = create(lib, gpt2_config(), w)
    assert st == 3 and h.value is None


def test_calls_on_a_null_handle_fail_cleanly(lib):
    assert lib.llm_decode_step(None, None, None, None, 1, None, None) == 1
    assert lib.llm_prefill(None, None, None, None, 1, None, None) == 1
    f = ctypes.c_uint32(0)
    assert lib.llm_get_error_flags(None, ctypes.byref(f)) == 1
    lib.llm_destroy(None)
    assert lib.llm_status_string(0) == b"ok"
    assert lib.llm_status_string(7) == b"device error flag set"


def test_control_calls_on_a_null_handle_fail_cleanly(lib):
    n = ctypes.c_int(0)
    assert lib.llm_selftest_wait_timeout(None) == 1
    assert lib.llm_set_profiling(None, 1) == 1
    assert lib.llm_set_graphs(None, 1) == 1
    assert lib.llm_set_linear_variant(None, 1) == 1
    assert lib.llm_last_launch_count(None, ctypes.byref(n)) == 1
    assert lib.llm_get_kernel_stats(None, None, 0, ctypes.byref(n), 0) == 1
    assert lib.llm_set_persistent(None, 1, ctypes.byref(n)) == 1
    assert lib.llm_selftest_grid_barrier(None) == 1


def test_op_linear_checks_arguments_on_the_host(lib):
    p = ctypes.c_void_p(256)   # never dereferenced: every call below fails its host checks
    F32, BF16 = 0, 1
    assert lib.llm_op_linear(F32, 0, 8, 8, p, p, None, p, 1, None) == 1       # size
    assert lib.llm_op_linear(F32, 4, 8, 8, None, p, None, p, 1, None) == 1    # NULL x
    assert lib.llm_op_linear(7, 4, 8, 8, p, p, None, p, 1, None) == 1         # dtype
    assert lib.llm_op_linear(F32, 4, 8, 8, p, p, None, p, 0, None) == 1       # variant
    assert lib.llm_op_linear(F32, 4, 8, 8, p, p, None, p, 3, None) == 4       # tcgen05 prefill GEMM is bf16 only
    assert lib.llm_op_linear(F32, 4, 8, 8, p, p, None, p, 5, None) == 4       # so is the SM-pair GEMM
    assert lib.llm_op_linear(BF16, 4, 8, 8, p, p, None, p, 6, None) == 1      # no variant 6
    assert lib.llm_op_linear(BF16, 4, 8, 12, p, p, None, p, 5, None) == 1     # K % 8
    assert lib.llm_op_linear(BF16, 4, 8, 12, p, p, None, p, 4, None) == 1     # K % 8
    assert lib.llm_op_linear(BF16, 300, 8, 16, p, p, None, p, 4, None) == 1   # weights-on-M path: M <= 256
    assert b"256" in lib.llm_last_error()


@pytest.mark.parametrize("entry", ["llm_op_attention_decode", "llm_op_attention_decode_noalloc"])
def test_op_attention_decode_checks_arguments_on_the_host(lib, entry):
    f = getattr(lib, entry)
    p = ctypes.c_void_p(256)
    #        kv_dtype, B, H, Hkv, q, k, v, blocks, pos, tables, mbps, out, stream
    assert f(0, 0, 12, 12, p, p, p, 8, p, p, 4, p, None) == 1        # B
    assert f(0, 2, 12, 12, None, p, p, 8, p, p, 4, p, None) == 1     # NULL q
    assert f(5, 2, 12, 12, p, p, p, 8, p, p, 4, p, None) == 1        # kv dtype
    assert f(0, 2, 12, 5, p, p, p, 8, p, p, 4, p, None) == 1         # H % Hkv
    assert f(0, 2, 18, 2, p, p, p, 8, p, p, 4, p, None) == 1         # more than 8 query heads a KV head
    if entry.endswith("noalloc"):                                    # scratch beyond the fixed array
        assert f(0, 256, 64, 8, p, p, p, 8, p, p, 4096, p, None) == 2
