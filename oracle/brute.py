"""Scalar-loop brute force of the decoder forward, for tiny models only.

TEST INFRASTRUCTURE (same rule as ``oracle.decoder``: tests, smoke and the bench
baseline only). It is written independently of ``oracle.decoder``: plain Python
floats and explicit loops, no NumPy matmul, so that a transposed operand, a
wrong head mapping or a dropped term in either implementation shows up as a
disagreement between the two. It follows the same per-layer sequence (GPT-2:
"bare-metal-llm", section "What got built"; Llama: "rvllm-metal", section
"What the kernels do") and the same readings of the open points.

Intended sizes: 1 layer, d = 8, 2 heads x 4, vocab 11, at most ~6 tokens.
"""
from __future__ import annotations

import math
import struct
from typing import List

from workloads import ARCH_GPT2, DTYPE_BF16, DTYPE_F32, DTYPE_Q8, Weights


def _f(a) -> List:
    """Tensor → nested Python lists of floats (exact widening of the stored values)."""
    return None if a is None else a.tolist()


def _bf16(v: float) -> float:
    """Nearest bfloat16 (ties to even) of v: float32 first, then the low 16 bits rounded away."""
    bits = struct.unpack("<I", struct.pack("<f", v))[0]
    lsb = (bits >> 16) & 1
    bits = ((bits + 0x7FFF + lsb) >> 16) << 16
    return struct.unpack("<f", struct.pack("<I", bits & 0xFFFFFFFF))[0]


def _q8(q, d):
    """Q8_0 rows: value j of a row is (scale of its 32-value block) * (int8 quant)."""
    out = []
    for r in range(len(q)):
        row = []
        for j in range(len(q[r])):
            row.append(float(d[r][j // 32]) * float(q[r][j]))
        out.append(row)
    return out


class BruteModel:
    def __init__(self, w: Weights, kv_dtype: int = DTYPE_F32):
        s = w.shape
        self.s = s
        self.kv_bf16 = kv_dtype == DTYPE_BF16
        q8 = s.dtype == DTYPE_Q8
        self.tok = _q8(w.tok_emb.tolist(), w.tok_emb_scale.tolist()) if q8 else _f(w.as_f64(w.tok_emb))
        self.pos = _f(w.as_f64(w.pos_emb))
        self.L = []
        for l in range(s.n_layers):
            self.L.append({k: _f(w.as_f64(getattr(w, k)[l])) for k in (
                "ln1_w", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_w", "ln2_b",
                "w_up", "b_up", "w_down", "b_down")})
            if q8:
                for k in ("w_qkv", "w_o", "w_up", "w_down"):
                    self.L[l][k] = _q8(getattr(w, k)[l].tolist(), getattr(w, k + "_scale")[l].tolist())
        self.lnf_w = _f(w.as_f64(w.lnf_w))
        self.lnf_b = _f(w.as_f64(w.lnf_b))
        if s.qk_norm:
            for l in range(s.n_layers):
                self.L[l]["q_norm_w"] = _f(w.as_f64(w.q_norm_w[l]))
                self.L[l]["k_norm_w"] = _f(w.as_f64(w.k_norm_w[l]))

    # ---- scalar helpers ------------------------------------------------------------------
    def _norm(self, x, g, b):
        n = len(x)
        eps = self.s.norm_eps
        if self.s.arch == ARCH_GPT2:
            mean = 0.0
            for v in x:
                mean += v
            mean /= n
            var = 0.0
            for v in x:
                var += (v - mean) * (v - mean)
            var /= n
            r = 1.0 / math.sqrt(var + eps)
            return [(x[i] - mean) * r * g[i] + (b[i] if b is not None else 0.0) for i in range(n)]
        ss = 0.0
        for v in x:
            ss += v * v
        r = 1.0 / math.sqrt(ss / n + eps)
        return [x[i] * r * g[i] for i in range(n)]

    @staticmethod
    def _matvec(w, x, b):
        out = []
        for r in range(len(w)):
            acc = 0.0
            row = w[r]
            for c in range(len(x)):
                acc += row[c] * x[c]
            if b is not None:
                acc += b[r]
            out.append(acc)
        return out

    @staticmethod
    def _gelu(x):
        u = math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)
        u = min(15.0, max(-15.0, u))
        return 0.5 * x * (1.0 + math.tanh(u))

    def _freq(self, i, hd):
        """Frequency of RoPE pair i, with Llama 3 scaling when the shape asks for it."""
        f = self.s.rope_theta ** (-2.0 * i / hd)
        if self.s.rope_scaling is None:
            return f
        factor, lo, hi, orig = self.s.rope_scaling
        wl = 2.0 * math.pi / f
        if wl < orig / hi:
            return f
        if wl > orig / lo:
            return f / factor
        sm = (orig / wl - lo) / (hi - lo)
        return (1.0 - sm) * f / factor + sm * f

    def _window(self, l):
        s = self.s
        if s.sliding_window <= 0 or (s.sliding_window_pattern > 0 and (l + 1) % s.sliding_window_pattern == 0):
            return 0
        return s.sliding_window

    def _head_rms(self, vec, g):
        ss = 0.0
        for x in vec:
            ss += x * x
        r = 1.0 / math.sqrt(ss / len(vec) + self.s.norm_eps)
        return [vec[i] * r * g[i] for i in range(len(vec))]

    def _rope(self, vec, pos):
        hd = len(vec)
        half = hd // 2
        out = list(vec)
        for i in range(half):
            ang = pos * self._freq(i, hd)
            c, sn = math.cos(ang), math.sin(ang)
            a, b = vec[i], vec[i + half]
            out[i] = a * c - b * sn
            out[i + half] = b * c + a * sn
        return out

    # ---- one token through the model with a per-layer list cache -------------------------
    def run(self, tokens):
        """Feed ``tokens`` one at a time from position 0; return logits after every token."""
        s = self.s
        hq, hkv, hd = s.n_heads, s.n_kv_heads, s.head_dim
        kc = [[] for _ in range(s.n_layers)]   # kc[l][pos][kv_head] -> list hd
        vc = [[] for _ in range(s.n_layers)]
        all_logits = []
        for t, tok in enumerate(tokens):
            h = list(self.tok[tok])
            if s.arch == ARCH_GPT2:
                h = [h[i] + self.pos[t][i] for i in range(s.d_model)]
            for l in range(s.n_layers):
                p = self.L[l]
                a = self._norm(h, p["ln1_w"], p["ln1_b"])
                qkv = self._matvec(p["w_qkv"], a, p["b_qkv"])
                q = [qkv[hh * hd:(hh + 1) * hd] for hh in range(hq)]
                k = [qkv[(hq + g) * hd:(hq + g + 1) * hd] for g in range(hkv)]
                v = [qkv[(hq + hkv + g) * hd:(hq + hkv + g + 1) * hd] for g in range(hkv)]
                if s.qk_norm:
                    q = [self._head_rms(x, p["q_norm_w"]) for x in q]
                    k = [self._head_rms(x, p["k_norm_w"]) for x in k]
                if s.arch != ARCH_GPT2:
                    q = [self._rope(x, t) for x in q]
                    k = [self._rope(x, t) for x in k]
                if self.kv_bf16:   # a bf16 KV cache stores rounded values
                    k = [[_bf16(x) for x in kk] for kk in k]
                    v = [[_bf16(x) for x in vv] for vv in v]
                kc[l].append(k)
                vc[l].append(v)
                o = []
                W = self._window(l)
                j0 = max(0, t - W + 1) if W > 0 else 0
                for hh in range(hq):
                    g = hh * hkv // hq
                    scores = []
                    for j in range(j0, t + 1):
                        dot = 0.0
                        for e in range(hd):
                            dot += q[hh][e] * kc[l][j][g][e]
                        scores.append(dot / math.sqrt(hd))
                    mx = max(scores)
                    ex = [math.exp(sc - mx) for sc in scores]
                    den = sum(ex)
                    for e in range(hd):
                        acc = 0.0
                        for j in range(j0, t + 1):
                            acc += ex[j - j0] / den * vc[l][j][g][e]
                        o.append(acc)
                proj = self._matvec(p["w_o"], o, p["b_o"])
                h = [h[i] + proj[i] for i in range(s.d_model)]
                m = self._norm(h, p["ln2_w"], p["ln2_b"])
                up = self._matvec(p["w_up"], m, p["b_up"])
                if s.arch == ARCH_GPT2:
                    f = [self._gelu(x) for x in up]
                else:
                    F = s.d_ff
                    f = [up[i] / (1.0 + math.exp(-up[i])) * up[F + i] for i in range(F)]
                down = self._matvec(p["w_down"], f, p["b_down"])
                h = [h[i] + down[i] for i in range(s.d_model)]
            hn = self._norm(h, self.lnf_w, self.lnf_b)
            logits = []
            for r in range(s.vocab):
                acc = 0.0
                for c in range(s.d_model):
                    acc += self.tok[r][c] * hn[c]
                logits.append(acc)
            all_logits.append(logits)
        return all_logits
