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
