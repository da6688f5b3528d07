"""Python binding of libllm.so: the GB300 KV-cached decoder step.

Argument marshalling only. Every step of the forward pass runs in the CUDA
library; PyTorch provides device memory and streams. Loading fails loudly when
the library is missing or the device is not a GB300: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libllm.so")

LLM_OK = 0
STATUS = {0: "LLM_OK", 1: "LLM_ERR_INVALID_ARG", 2: "LLM_ERR_OUT_OF_RANGE", 3: "LLM_ERR_NO_DEVICE",
          4: "LLM_ERR_UNSUPPORTED", 5: "LLM_ERR_OOM", 6: "LLM_ERR_CUDA", 7: "LLM_ERR_DEVICE_FLAG"}
FLAG_BAD_TOKEN, FLAG_BAD_POSITION, FLAG_BAD_BLOCK, FLAG_NAN_LOGIT, FLAG_WAIT_TIMEOUT = 1, 2, 4, 8, 16

EXPORTS = ["llm_create", "llm_destroy", "llm_prefill", "llm_step", "llm_decode_step", "llm_decode_step_sample", "llm_decode_step_host",
           "llm_get_error_flags", "llm_selftest_wait_timeout", "llm_set_profiling", "llm_get_kernel_stats", "llm_last_launch_count",
           "llm_set_graphs", "llm_set_persistent", "llm_selftest_grid_barrier", "llm_set_linear_variant", "llm_op_linear", "llm_op_linear_q8", "llm_op_attention_decode",
           "llm_op_attention_decode_noalloc",
           "llm_status_string", "llm_last_error"]


class LLMError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class LLMConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("arch", "dtype", "n_layers", "d_model", "n_heads", "n_kv_heads",
                                             "head_dim", "d_ff", "vocab", "n_ctx")] + \
               [("norm_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)] + \
               [(n, ctypes.c_int) for n in ("kv_block_size", "num_kv_blocks", "max_batch", "max_blocks_per_seq",
                                             "max_prefill_tokens", "contiguous_kv", "kv_dtype", "sliding_window",
                                             "sliding_window_pattern", "qk_norm")] + \
               [(n, ctypes.c_float) for n in ("rope_scale_factor", "rope_low_freq_factor", "rope_high_freq_factor")] + \
               [("rope_original_max_pos", ctypes.c_int)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class LLMWeights(ctypes.Structure):
    _fields_ = [("tok_emb", ctypes.c_void_p), ("pos_emb", ctypes.c_void_p)] + \
               [(n, _PP) for n in ("ln1_w", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_w", "ln2_b",
                                   "w_up", "b_up", "w_down", "b_down")] + \
               [("lnf_w", ctypes.c_void_p), ("lnf_b", ctypes.c_void_p), ("q_norm_w", _PP), ("k_norm_w", _PP),
                ("tok_emb_scale", ctypes.c_void_p)] + \
               [(n, _PP) for n in ("w_qkv_scale", "w_o_scale", "w_up_scale", "w_down_scale")]


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libllm.so once. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m transformer_decoder_forward_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32p = ctypes.c_void_p, ctypes.c_void_p
    lib.llm_create.argtypes = [ctypes.POINTER(LLMConfig), ctypes.POINTER(LLMWeights), vp, ctypes.POINTER(vp)]
    lib.llm_destroy.argtypes = [vp]
    lib.llm_destroy.restype = None
    lib.llm_prefill.argtypes = [vp, i32p, ctypes.POINTER(ctypes.c_int32), i32p, ctypes.c_int, i32p, vp]
    lib.llm_step.argtypes = [vp, i32p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32), i32p,
                             ctypes.c_int, i32p, vp]
    lib.llm_decode_step.argtypes = [vp, i32p, i32p, i32p, ctypes.c_int, i32p, vp]
    lib.llm_decode_step_sample.argtypes = [vp, i32p, i32p, i32p, ctypes.c_int, ctypes.c_float, ctypes.c_int, vp,
                                           i32p, vp]
    lib.llm_decode_step_host.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp, vp]
    lib.llm_get_error_flags.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.llm_set_profiling.argtypes = [vp, ctypes.c_int]
    lib.llm_selftest_wait_timeout.argtypes = [vp]
    lib.llm_get_kernel_stats.argtypes = [vp, ctypes.POINTER(KernelStat), ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                         ctypes.c_int]
    lib.llm_last_launch_count.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    lib.llm_set_graphs.argtypes = [vp, ctypes.c_int]
    lib.llm_set_persistent.argtypes = [vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    lib.llm_selftest_grid_barrier.argtypes = [vp]
    lib.llm_set_linear_variant.argtypes = [vp, ctypes.c_int]
    lib.llm_op_linear.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, ctypes.c_int, vp]
    lib.llm_op_linear_q8.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, ctypes.c_int, vp]
    lib.llm_op_attention_decode.argtypes = [ctypes.c_int] * 4 + [vp, vp, vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, vp]
    lib.llm_op_attention_decode_noalloc.argtypes = lib.llm_op_attention_decode.argtypes
    lib.llm_status_string.argtypes = [ctypes.c_int]
    lib.llm_status_string.restype = ctypes.c_char_p
    lib.llm_last_error.argtypes = []
    lib.llm_last_error.restype = ctypes.c_char_p
    for name in ("llm_create", "llm_prefill", "llm_step", "llm_decode_step", "llm_decode_step_sample", "llm_decode_step_host", "llm_get_error_flags",
                 "llm_set_profiling", "llm_selftest_wait_timeout", "llm_get_kernel_stats", "llm_last_launch_count", "llm_set_graphs",
                 "llm_set_persistent", "llm_selftest_grid_barrier", "llm_set_linear_variant", "llm_op_linear",
                 "llm_op_linear_q8", "llm_op_attention_decode", "llm_op_attention_decode_noalloc"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != LLM_OK:
        raise LLMError(status, (_lib.llm_last_error() or b"").decode())


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def op_linear(x, w, bias, y, variant: int, stream=None) -> None:
    """y = x . w^T (+ bias) with one chosen projection kernel (tests / diagnostics).

    w [N, K] float32 or bfloat16, bias [N] (w's dtype) or None, y float32 [M, N]. x is the
    library's activation storage for w's dtype: float32 [M, K], or for bfloat16 weights a
    bfloat16 [M, 2K] tensor whose row holds hi[0..K) then lo[0..K) (x = hi + lo)."""
    import torch
    lib = load()
    dtype = 1 if w.dtype == torch.bfloat16 else 0
    N, K = w.shape
    M = x.shape[0]
    if x.dtype != w.dtype or x.shape[1] != (2 * K if dtype == 1 else K):
        raise ValueError("x must be float32 [M, K] for float32 weights, bfloat16 [M, 2K] for bfloat16 weights")
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(lib.llm_op_linear(dtype, M, N, K, _ptr(x), _ptr(w), _ptr(bias), _ptr(y), int(variant),
                             ctypes.c_void_p(s.cuda_stream)))


def op_linear_q8(x, wq, wscale, bias, y, variant: int, stream=None) -> None:
    """y = x . (wscale * wq)^T (+ bias) with Q8_0 weights: wq int8 [N, K], wscale float16 [N, K / 32],
    bias float32 [N] or None, x float32 [M, K], y float32 [M, N]; variant 1 (GEMV) or 2 (tiled GEMM)."""
    import torch
    lib = load()
    N, K = wq.shape
    M = x.shape[0]
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(lib.llm_op_linear_q8(M, N, K, _ptr(x), _ptr(wq), _ptr(wscale), _ptr(bias), _ptr(y), int(variant),
                                ctypes.c_void_p(s.cuda_stream)))


def op_attention_decode(q, k_pool, v_pool, positions, block_tables, out, n_kv_heads: int, stream=None,
                        noalloc: bool = False) -> None:
    """Paged decode attention of one layer (tests / diagnostics). See llm_op_attention_decode.

    noalloc=True calls llm_op_attention_decode_noalloc: the same kernels with their scratch in a
    fixed device array instead of memory allocated per call."""
    import torch
    lib = load()
    fn = lib.llm_op_attention_decode_noalloc if noalloc else lib.llm_op_attention_decode
    kv_dtype = 1 if k_pool.dtype == torch.bfloat16 else 0
    B, HD = q.shape
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(fn(kv_dtype, B, HD // 64, int(n_kv_heads), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                       k_pool.shape[0], _ptr(positions), _ptr(block_tables), block_tables.shape[1],
                                       _ptr(out), ctypes.c_void_p(s.cuda_stream)))


def upload_weights(w, device: str = "cuda"):
    """Copy a ``workloads.Weights`` host model to device tensors (fp32 or bf16). Returns a dict of tensors."""
    import torch

    def dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    out = {"tok_emb": dev(w.tok_emb), "pos_emb": dev(w.pos_emb), "lnf_w": dev(w.lnf_w), "lnf_b": dev(w.lnf_b)}
    for k in ("ln1_w", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_w", "ln2_b", "w_up", "b_up", "w_down", "b_down"):
        out[k] = [dev(a) for a in getattr(w, k)]
    for k in ("q_norm_w", "k_norm_w", "w_qkv_scale", "w_o_scale", "w_up_scale", "w_down_scale"):
        out[k] = None if getattr(w, k) is None else [dev(a) for a in getattr(w, k)]
    out["tok_emb_scale"] = dev(w.tok_emb_scale)
    return out


class Decoder:
    """One libllm handle over device-resident weights.

    ``shape`` is a ``workloads.ModelShape``; ``dev_w`` the dict from ``upload_weights``.
    All tensors passed to the step methods are CUDA tensors (int32 ids/positions/tables,
    float32 logits), except ``lengths`` of prefill, which is host data.
    """

    def __init__(self, shape, dev_w, *, max_batch: int, max_blocks_per_seq: int, num_kv_blocks: int = 0,
                 max_prefill_tokens: int = 4096, contiguous_kv: bool = False, kv_dtype: int = 0, stream=None):
        import torch
        self.lib = load()
        self.shape = shape
        self.dev_w = dev_w
        self.stream = stream if stream is not None else torch.cuda.Stream()
        c = LLMConfig(arch=shape.arch, dtype=shape.dtype, n_layers=shape.n_layers, d_model=shape.d_model,
                      n_heads=shape.n_heads, n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim,
                      d_ff=shape.d_ff, vocab=shape.vocab, n_ctx=shape.n_ctx, norm_eps=shape.norm_eps,
                      rope_theta=shape.rope_theta, kv_block_size=16, num_kv_blocks=num_kv_blocks,
                      max_batch=max_batch, max_blocks_per_seq=max_blocks_per_seq,
                      max_prefill_tokens=max_prefill_tokens, contiguous_kv=int(contiguous_kv),
                      kv_dtype=int(kv_dtype), sliding_window=int(shape.sliding_window),
                      sliding_window_pattern=int(shape.sliding_window_pattern), qk_norm=int(shape.qk_norm))
        if shape.rope_scaling is not None:
            c.rope_scale_factor, c.rope_low_freq_factor, c.rope_high_freq_factor = (float(x) for x in shape.rope_scaling[:3])
            c.rope_original_max_pos = int(shape.rope_scaling[3])
        self.config = c
        L = shape.n_layers
        self._arrays = []

        def arr(name):
            lst = dev_w.get(name)
            if lst is None or all(t is None for t in lst):
                return None
            a = (ctypes.c_void_p * L)(*[_ptr(t) for t in lst])
            self._arrays.append(a)
            return ctypes.cast(a, _PP)

        w = LLMWeights(tok_emb=_ptr(dev_w["tok_emb"]), pos_emb=_ptr(dev_w["pos_emb"]),
                       lnf_w=_ptr(dev_w["lnf_w"]), lnf_b=_ptr(dev_w["lnf_b"]),
                       tok_emb_scale=_ptr(dev_w.get("tok_emb_scale")))
        for k in ("ln1_w", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_w", "ln2_b", "w_up", "b_up", "w_down",
                  "b_down", "q_norm_w", "k_norm_w", "w_qkv_scale", "w_o_scale", "w_up_scale", "w_down_scale"):
            setattr(w, k, arr(k))
        handle = ctypes.c_void_p()
        torch.cuda.synchronize()
        _check(self.lib.llm_create(ctypes.byref(c), ctypes.byref(w), ctypes.c_void_p(self.stream.cuda_stream),
                                   ctypes.byref(handle)))
        self.handle = handle

    # ---- steps ---------------------------------------------------------------------------
    def prefill(self, tokens, lengths: Sequence[int], block_tables, next_ids, logits=None) -> None:
        lens = (ctypes.c_int32 * len(lengths))(*[int(x) for x in lengths])
        _check(self.lib.llm_prefill(self.handle, _ptr(tokens), lens, _ptr(block_tables), len(lengths),
                                    _ptr(next_ids), _ptr(logits)))

    def step(self, tokens, lengths: Sequence[int], starts: Sequence[int], block_tables, next_ids, logits=None) -> None:
        """Mixed pass: sequence b feeds lengths[b] tokens from position starts[b] (host lists)."""
        lens = (ctypes.c_int32 * len(lengths))(*[int(x) for x in lengths])
        sts = (ctypes.c_int32 * len(starts))(*[int(x) for x in starts])
        _check(self.lib.llm_step(self.handle, _ptr(tokens), lens, sts, _ptr(block_tables), len(lengths),
                                 _ptr(next_ids), _ptr(logits)))

    def decode_step(self, tokens, positions, block_tables, next_ids, logits=None) -> None:
        _check(self.lib.llm_decode_step(self.handle, _ptr(tokens), _ptr(positions), _ptr(block_tables),
                                        int(tokens.numel()), _ptr(next_ids), _ptr(logits)))

    def decode_step_sample(self, tokens, positions, block_tables, temperature: float, top_k: int, uniforms,
                           next_ids, logits=None) -> None:
        """A decode step that samples (temperature, top-k) with the caller's uniforms [B] (device)."""
        _check(self.lib.llm_decode_step_sample(self.handle, _ptr(tokens), _ptr(positions), _ptr(block_tables),
                                               int(tokens.numel()), float(temperature), int(top_k),
                                               _ptr(uniforms), _ptr(next_ids), _ptr(logits)))

    def decode_step_host(self, tokens: np.ndarray, positions: np.ndarray, block_tables: Optional[np.ndarray],
                         next_ids: np.ndarray, logits: Optional[np.ndarray] = None) -> None:
        """Host-buffer variant: numpy int32 inputs, numpy int32 / float32 outputs (synchronous)."""
        def p(a):
            return None if a is None else a.ctypes.data
        _check(self.lib.llm_decode_step_host(self.handle, p(tokens), p(positions), p(block_tables), len(tokens),
                                             p(next_ids), p(logits)))

    # ---- diagnostics ---------------------------------------------------------------------
    def error_flags(self) -> int:
        f = ctypes.c_uint32(0)
        st = self.lib.llm_get_error_flags(self.handle, ctypes.byref(f))
        if st not in (LLM_OK, 7):
            _check(st)
        return int(f.value)

    def selftest_wait_timeout(self) -> None:
        """Launch a kernel whose bounded wait runs out (about one second); the next
        error_flags() returns LLM_FLAG_WAIT_TIMEOUT."""
        _check(self.lib.llm_selftest_wait_timeout(self.handle))

    def set_profiling(self, on: bool) -> None:
        _check(self.lib.llm_set_profiling(self.handle, int(on)))

    def set_graphs(self, on: bool) -> None:
        _check(self.lib.llm_set_graphs(self.handle, int(on)))

    def set_persistent(self, on: bool) -> bool:
        """Decode steps of at most 8 sequences as one persistent kernel (default off: the
        per-phase graph measured faster); returns whether the model's shapes allow it here."""
        sup = ctypes.c_int(0)
        _check(self.lib.llm_set_persistent(self.handle, int(on), ctypes.byref(sup)))
        return bool(sup.value)

    def selftest_grid_barrier(self) -> None:
        """Run the persistent kernel with one CTA withheld: the grid barrier's bounded wait runs
        out (about one second); the next error_flags() returns LLM_FLAG_WAIT_TIMEOUT."""
        _check(self.lib.llm_selftest_grid_barrier(self.handle))

    def set_linear_variant(self, v: int) -> None:
        """0 auto, 1 CUDA-core GEMV, 2 CUDA-core tiled GEMM, 3 tcgen05 GEMM, 4 tcgen05 weights-on-M GEMM."""
        _check(self.lib.llm_set_linear_variant(self.handle, int(v)))

    def kernel_stats(self, reset: bool = True):
        buf = (KernelStat * 64)()
        n = ctypes.c_int(0)
        _check(self.lib.llm_get_kernel_stats(self.handle, buf, 64, ctypes.byref(n), int(reset)))
        return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(n.value)}

    def last_launch_count(self) -> int:
        n = ctypes.c_int(0)
        _check(self.lib.llm_last_launch_count(self.handle, ctypes.byref(n)))
        return n.value

    def close(self) -> None:
        if getattr(self, "handle", None):
            self.lib.llm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
