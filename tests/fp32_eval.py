"""A plain float32 evaluation of the GPT-2 variant's forward pass (test helper).

It computes the same definition as the float64 oracle, in NumPy float32 throughout (every
constant a float32, so nothing is promoted to float64), with the library's BLAS deciding the
summation order. It measures how far an accurate float32 program can be from the float64
oracle on a given model: the floor below which no float32 implementation, GPU or CPU, can be
asked to agree. It shares no code with the oracle or the CUDA library.
"""
from __future__ import annotations

import numpy as np

import workloads as wl

F = np.float32


def _w(w: wl.Weights, a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return wl.bf16_bits_to_f32(a)
    return np.ascontiguousarray(a, dtype=np.float32)


def _layer_norm(x, g, b, eps):
    mu = x.mean(axis=-1, keepdims=True, dtype=F)
    xc = x - mu
    var = (xc * xc).mean(axis=-1, keepdims=True, dtype=F)
    return xc / np.sqrt(var + F(eps)) * g + b


def _gelu(x):
    u = F(np.sqrt(2.0 / np.pi)) * (x + F(0.044715) * x * x * x)
    u = np.clip(u, F(-15.0), F(15.0))
    return F(0.5) * x * (F(1.0) + np.tanh(u))


def gpt2_forward_f32(w: wl.Weights, tokens) -> np.ndarray:
    """Logits [T, V] (float32) at positions 0..T-1, whole sequence at once."""
    s = w.shape
    assert s.arch == wl.ARCH_GPT2
    T = len(tokens)
    H, hd = s.n_heads, s.head_dim
    h = _w(w, w.tok_emb)[np.asarray(tokens)] + _w(w, w.pos_emb)[:T]
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    scale = F(1.0 / np.sqrt(hd))
    for l in range(s.n_layers):
        a = _layer_norm(h, _w(w, w.ln1_w[l]), _w(w, w.ln1_b[l]), s.norm_eps)
        qkv = a @ _w(w, w.w_qkv[l]).T + _w(w, w.b_qkv[l])
        q = qkv[:, : H * hd].reshape(T, H, hd)
        k = qkv[:, H * hd: 2 * H * hd].reshape(T, H, hd)
        v = qkv[:, 2 * H * hd:].reshape(T, H, hd)
        o = np.empty((T, H, hd), dtype=F)
        for hh in range(H):
            sc = (q[:, hh, :] @ k[:, hh, :].T) * scale
            sc = np.where(mask, F(-np.inf), sc)
            e = np.exp(sc - sc.max(axis=-1, keepdims=True))
            o[:, hh, :] = (e / e.sum(axis=-1, keepdims=True)) @ v[:, hh, :]
        h = h + o.reshape(T, H * hd) @ _w(w, w.w_o[l]).T + _w(w, w.b_o[l])
        m = _layer_norm(h, _w(w, w.ln2_w[l]), _w(w, w.ln2_b[l]), s.norm_eps)
        f = _gelu(m @ _w(w, w.w_up[l]).T + _w(w, w.b_up[l]))
        h = h + f @ _w(w, w.w_down[l]).T + _w(w, w.b_down[l])
        assert h.dtype == F
    z = _layer_norm(h, _w(w, w.lnf_w), _w(w, w.lnf_b), s.norm_eps) @ _w(w, w.tok_emb).T
    assert z.dtype == F
    return z
