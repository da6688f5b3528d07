"""Float64 CPU oracle of the decoder-only transformer forward step.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import or run this module. The
product library never calls it and shares no code with it; both sides read the
same seeded inputs from ``workloads``.

What it computes is the plain definition of the model, written out in float64
NumPy with no blocking, fusion or reordering:

* GPT-2 variant ("bare-metal-llm", section "Picking the model" and "What got
  built"): learned position embeddings, LayerNorm, multi-head causal attention,
  GELU-tanh FFN, residual adds, final LayerNorm and a tied LM head (the
  "transposed variant for tied embeddings").
* Llama variant ("rvllm-metal", section "What the kernels do"): RMSNorm, Q/K/V
  projections, RoPE, grouped-query attention, output projection plus residual,
  RMSNorm, gate/up projections, silu(gate) * up, down projection plus residual;
  final norm, projection to the vocabulary and a greedy argmax.

Two modes, which must agree (a cached step is a full recompute with the old
keys and values kept; "bare-metal-llm", section "What got built", and the KV
cache remark in "batch_forge"):

* ``forward_full`` recomputes the whole sequence (stateless, O(T^2) per step);
* ``Sequence.prefill`` / ``Sequence.step`` keep per-layer K/V arrays.

Readings where the pages leave the step open:
GELU is GPT-2's tanh form with the tanh argument clamped to [-15, 15]
("batch_forge", GELU-overflow paragraph); LayerNorm uses the biased variance
with eps inside the square root; RMSNorm is x / sqrt(mean(x^2) + eps) * g; RoPE
pairs element i with element i + head_dim/2 and rotates by pos * theta^(-2i/hd);
query head h reads KV head h // (Hq / Hkv); scores are scaled by 1/sqrt(hd)
and masked with -inf; argmax ties go to the lowest index and NaN ranks above
every number (first NaN wins).
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np

from workloads import ARCH_GPT2, ARCH_LLAMA, DTYPE_BF16, DTYPE_F32, DTYPE_Q8, ModelShape, Weights

GELU_C = np.sqrt(2.0 / np.pi)
GELU_CUBIC = 0.044715
GELU_TANH_CLAMP = 15.0


# ----------------------------------------------------------------------------------------------
# elementwise / row operations
# ----------------------------------------------------------------------------------------------

def layer_norm(x: np.ndarray, g: np.ndarray, b: Optional[np.ndarray], eps: float) -> np.ndarray:
    """Row LayerNorm: (x - mean) / sqrt(var + eps) * g + b, biased variance over the last axis."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    y = (x - mu) / np.sqrt(var + eps) * g
    return y + b if b is not None else y


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """Row RMSNorm ("rvllm-metal", section "How a GPU runs your kernel": sum of squares of a row)."""
    ms = (x * x).mean(axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def gelu_tanh_arg(x: np.ndarray) -> np.ndarray:
    """The (unclamped) tanh argument of GELU-tanh: sqrt(2/pi) * (x + 0.044715 x^3)."""
    return GELU_C * (x + GELU_CUBIC * x * x * x)


def gelu_tanh(x: np.ndarray, stats: Optional[Dict[str, float]] = None) -> np.ndarray:
    """GELU-tanh with the tanh argument clamped to +-15 ("batch_forge", GELU overflow fix).

    tanh is saturated to +-1 well before |arg| = 15, so the clamp changes nothing
    in exact arithmetic beyond 1 - tanh(15) ~ 1.9e-13; it exists so that a float32
    implementation never forms exp(2 * arg) = inf.
    """
    u = gelu_tanh_arg(x)
    if stats is not None and u.size:
        stats["max_gelu_arg"] = max(stats.get("max_gelu_arg", 0.0), float(np.abs(u).max()))
    u = np.clip(u, -GELU_TANH_CLAMP, GELU_TANH_CLAMP)
    return 0.5 * x * (1.0 + np.tanh(u))


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x)."""
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def llama3_scaled_inv_freq(inv_freq: np.ndarray, factor: float, low_freq_factor: float, high_freq_factor: float,
                           original_max_position: int) -> np.ndarray:
    """Llama 3 RoPE scaling ("rvllm-metal", section "What the kernels do", last paragraph, names
    it; the rule is the one the Llama 3.1 release defines). A pair whose wavelength 2 pi / f is
    shorter than original_max_position / high_freq_factor keeps its frequency; one longer than
    original_max_position / low_freq_factor is slowed by `factor`; in between the two are
    mixed linearly in s = (original_max_position / wavelength - low_freq_factor) /
    (high_freq_factor - low_freq_factor): f' = (1 - s) f / factor + s f.
    """
    f = np.asarray(inv_freq, dtype=np.float64)
    wavelen = 2.0 * np.pi / f
    low_wl = original_max_position / low_freq_factor
    high_wl = original_max_position / high_freq_factor
    s = (original_max_position / wavelen - low_freq_factor) / (high_freq_factor - low_freq_factor)
    mid = (1.0 - s) * f / factor + s * f
    return np.where(wavelen < high_wl, f, np.where(wavelen > low_wl, f / factor, mid))


def rope(x: np.ndarray, pos: np.ndarray, theta: float, scaling=None) -> np.ndarray:
    """Rotate [T, H, hd] by position ("rvllm-metal", "What the kernels do": RoPE per pair).

    Element i of a head is paired with element i + hd/2 (half-split pairing);
    pair i turns by the angle pos * theta^(-2i/hd) (with Llama 3 scaling of those
    frequencies when ``scaling`` = (factor, low_freq_factor, high_freq_factor,
    original_max_position) is given).
    """
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / hd)
    if scaling is not None:
        inv_freq = llama3_scaled_inv_freq(inv_freq, *scaling)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]      # [T, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    """exp(s - max) / sum; entries equal to -inf get exactly 0."""
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=axis, keepdims=True)


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray, window: int = 0) -> np.ndarray:
    """Causal (grouped-query) attention.

    q [Tq, Hq, hd] at positions q_pos; k, v [Tk, Hkv, hd] hold positions 0..Tk-1.
    Query i of head h reads KV head h // (Hq/Hkv) over keys j <= q_pos[i] (and, with a
    sliding window W > 0, j > q_pos[i] - W: the W most recent positions, its own included;
    "rvllm-metal", section "What the kernels do", names Gemma's sliding window):
    softmax_j(q.k_j / sqrt(hd)) weighted sum of v_j. Returns [Tq, Hq * hd].
    """
    tq, hq, hd = q.shape
    tk, hkv, _ = k.shape
    group = hq // hkv
    scale = 1.0 / np.sqrt(hd)
    qp = np.asarray(q_pos)[:, None]
    mask = np.arange(tk)[None, :] > qp                                          # [Tq, Tk]
    if window > 0:
        mask = mask | (np.arange(tk)[None, :] <= qp - window)
    out = np.empty((tq, hq, hd), dtype=np.float64)
    for h in range(hq):
        g = h // group
        s = (q[:, h, :] @ k[:, g, :].T) * scale
        s = np.where(mask, -np.inf, s)
        out[:, h, :] = softmax(s) @ v[:, g, :]
    return out.reshape(tq, hq * hd)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value, ties to even (returned widened to float64).

    A bf16 KV cache stores each K and V element with the float32 exponent and the top 7
    explicit mantissa bits; the value is first taken to float32 (nearest), then its 16 low bits
    are rounded away to nearest, ties to the even result.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)) << np.uint64(16)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def argmax_rule(z: np.ndarray) -> int:
    """Greedy id: NaN ranks above every number (first NaN wins); ties go to the lowest index."""
    z = np.asarray(z)
    nan = np.isnan(z)
    if nan.any():
        return int(np.flatnonzero(nan)[0])
    return int(np.flatnonzero(z == z.max())[0])


def sample_top_k(z: np.ndarray, temperature: float, top_k: int, u: float) -> int:
    """Temperature / top-k sampling of one next token ("batch_forge", component table:
    sampling greedy, temperature, top-k), with the uniform draw u in [0, 1) given.

    The k largest logits are the candidates, ordered by value (ties: the lower index first,
    so a tie at the k-th place keeps the lower index); p_i = exp((z_i - z_top) / T) over them;
    the token is the first candidate whose running sum of p exceeds u * sum(p). top_k <= 1 or
    T <= 0 is greedy (the argmax rule). A NaN logit gives the argmax rule's first NaN.
    """
    z = np.asarray(z, dtype=np.float64)
    if np.isnan(z).any() or top_k <= 1 or temperature <= 0.0:
        return argmax_rule(z)
    k = min(int(top_k), z.size)
    order = np.lexsort((np.arange(z.size), -z))[:k]          # value descending, then index ascending
    p = np.exp((z[order] - z[order[0]]) / float(temperature))
    c = np.cumsum(p)
    i = int(np.searchsorted(c, float(u) * c[-1], side="right"))
    return int(order[min(i, k - 1)])


def top2_margin(z: np.ndarray) -> float:
    """top-1 minus top-2 logit (the near-tie test of "rvllm-metal", section "How I know it's correct")."""
    part = np.partition(np.asarray(z, dtype=np.float64), -2)
    return float(part[-1] - part[-2])


# ----------------------------------------------------------------------------------------------
# model
# ----------------------------------------------------------------------------------------------

def dequant_q8_0(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Q8_0 weights ("rvllm-metal", sections "What's basic about it" and "What's next": one
    byte a weight): each row is cut into blocks of 32; a block's value j is d_block * q_j, d an
    fp16 scale and q an int8."""
    q = np.asarray(q, dtype=np.float64)
    d = np.asarray(d, dtype=np.float64)
    return q * np.repeat(d, q.shape[1] // d.shape[1], axis=1)


class OracleModel:
    """A model's parameters widened to float64, plus the per-layer forward.

    ``kv_dtype`` is the element type of the KV cache the method stores: DTYPE_F32 keeps K and V
    as computed (float32 holds them to about 2^-24, below what the float64 oracle models);
    DTYPE_BF16 stores them rounded to bfloat16, which is part of what that mode computes, so
    the oracle rounds them the same way before any attention reads them.
    """

    def __init__(self, w: Weights, kv_dtype: int = DTYPE_F32):
        self.shape: ModelShape = w.shape
        self.kv_dtype = kv_dtype
        f = w.as_f64
        q8 = self.shape.dtype == DTYPE_Q8
        self.tok_emb = dequant_q8_0(w.tok_emb, w.tok_emb_scale) if q8 else f(w.tok_emb)
        self.pos_emb = f(w.pos_emb)
        self.layers = []
        for l in range(self.shape.n_layers):
            self.layers.append({k: f(getattr(w, k)[l]) for k in (
                "ln1_w", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_w", "ln2_b",
                "w_up", "b_up", "w_down", "b_down")})
            if q8:
                for k in ("w_qkv", "w_o", "w_up", "w_down"):
                    self.layers[l][k] = dequant_q8_0(getattr(w, k)[l], getattr(w, k + "_scale")[l])
        self.lnf_w = f(w.lnf_w)
        self.lnf_b = f(w.lnf_b)
        if self.shape.qk_norm:
            for l in range(self.shape.n_layers):
                self.layers[l]["q_norm_w"] = f(w.q_norm_w[l])
                self.layers[l]["k_norm_w"] = f(w.k_norm_w[l])
        self.stats: Dict[str, float] = {}

    def window(self, l: int) -> int:
        """Sliding window of layer l (0: full causal). With a pattern P > 0 every P-th layer
        (l + 1 a multiple of P) attends globally, as Gemma interleaves local and global layers."""
        s = self.shape
        if s.sliding_window <= 0:
            return 0
        if s.sliding_window_pattern > 0 and (l + 1) % s.sliding_window_pattern == 0:
            return 0
        return s.sliding_window

    # -- pieces ------------------------------------------------------------------------------
    def norm(self, x, g, b):
        if self.shape.arch == ARCH_GPT2:
            return layer_norm(x, g, b, self.shape.norm_eps)
        return rms_norm(x, g, self.shape.norm_eps)

    @staticmethod
    def linear(x, w, b):
        y = x @ w.T
        return y + b if b is not None else y

    def embed(self, tokens: np.ndarray, positions: np.ndarray) -> np.ndarray:
        h = self.tok_emb[np.asarray(tokens)]
        if self.shape.arch == ARCH_GPT2:
            h = h + self.pos_emb[np.asarray(positions)]
        return h

    def layer(self, l: int, h: np.ndarray, positions: np.ndarray,
              k_cache: Optional[np.ndarray], v_cache: Optional[np.ndarray]):
        """One block over new rows h [T, d] at ``positions``; the caches hold positions 0..P-1.

        Returns (h_out, k_all, v_all) where k_all/v_all include the new rows.
        """
        s = self.shape
        p = self.layers[l]
        hq, hkv, hd = s.n_heads, s.n_kv_heads, s.head_dim
        a = self.norm(h, p["ln1_w"], p["ln1_b"])
        qkv = self.linear(a, p["w_qkv"], p["b_qkv"])
        t = h.shape[0]
        q = qkv[:, : hq * hd].reshape(t, hq, hd)
        k = qkv[:, hq * hd: (hq + hkv) * hd].reshape(t, hkv, hd)
        v = qkv[:, (hq + hkv) * hd:].reshape(t, hkv, hd)
        if s.qk_norm:
            # Q/K norm ("rvllm-metal", "What the kernels do", names Qwen3's): RMSNorm of every
            # q and k head over its head_dim values, before RoPE
            q = rms_norm(q, p["q_norm_w"], s.norm_eps)
            k = rms_norm(k, p["k_norm_w"], s.norm_eps)
        if s.arch == ARCH_LLAMA:
            q = rope(q, positions, s.rope_theta, s.rope_scaling)
            k = rope(k, positions, s.rope_theta, s.rope_scaling)
        if self.kv_dtype == DTYPE_BF16:
            k, v = round_bf16(k), round_bf16(v)
        k_all = k if k_cache is None else np.concatenate([k_cache, k], axis=0)
        v_all = v if v_cache is None else np.concatenate([v_cache, v], axis=0)
        o = causal_attention(q, k_all, v_all, positions, self.window(l))
        h = h + self.linear(o, p["w_o"], p["b_o"])
        m = self.norm(h, p["ln2_w"], p["ln2_b"])
        up = self.linear(m, p["w_up"], p["b_up"])
        if s.arch == ARCH_GPT2:
            f = gelu_tanh(up, self.stats)
        else:
            f = silu(up[:, : s.d_ff]) * up[:, s.d_ff:]
        h = h + self.linear(f, p["w_down"], p["b_down"])
        return h, k_all, v_all

    def head(self, h: np.ndarray) -> np.ndarray:
        """Final norm then the tied LM head: logits = Norm_f(h) . tok_emb^T."""
        return self.norm(h, self.lnf_w, self.lnf_b) @ self.tok_emb.T


def forward_full(model: OracleModel, tokens, last_only: bool = False) -> np.ndarray:
    """Stateless forward over the whole sequence at positions 0..T-1 (the no-cache recompute).

    Returns logits [T, V] (or [1, V] for the last position when ``last_only``).
    """
    tokens = np.asarray(tokens)
    pos = np.arange(len(tokens))
    h = model.embed(tokens, pos)
    for l in range(model.shape.n_layers):
        h, _, _ = model.layer(l, h, pos, None, None)
    return model.head(h[-1:] if last_only else h)


class Sequence:
    """One sequence with its own KV cache (a logical cache: position j is row j)."""

    def __init__(self, model: OracleModel):
        self.model = model
        self.k: List[Optional[np.ndarray]] = [None] * model.shape.n_layers
        self.v: List[Optional[np.ndarray]] = [None] * model.shape.n_layers
        self.length = 0

    def feed(self, tokens, all_logits: bool = False) -> np.ndarray:
        """Append tokens at positions length.. and return logits of the last (or every) new row."""
        tokens = np.asarray(tokens).reshape(-1)
        pos = np.arange(self.length, self.length + len(tokens))
        if self.model.shape.arch == ARCH_GPT2 and pos[-1] >= self.model.shape.n_ctx:
            raise ValueError("position beyond the learned position table")
        h = self.model.embed(tokens, pos)
        for l in range(self.model.shape.n_layers):
            h, self.k[l], self.v[l] = self.model.layer(l, h, pos, self.k[l], self.v[l])
        self.length += len(tokens)
        return self.model.head(h if all_logits else h[-1:])

    def prefill(self, tokens) -> np.ndarray:
        return self.feed(tokens)[0]

    def step(self, token: int) -> np.ndarray:
        return self.feed([token])[0]


def greedy_generate(model: OracleModel, prompt, steps: int):
    """Prefill then ``steps`` greedy decode steps. Returns (ids [steps+1], logits [steps+1, V]).

    ids[0] is the argmax after the prompt, ids[i] the argmax after feeding ids[i-1].
    """
    seq = Sequence(model)
    z = seq.prefill(prompt)
    ids, zs = [argmax_rule(z)], [z]
    for _ in range(steps):
        z = seq.step(ids[-1])
        ids.append(argmax_rule(z))
        zs.append(z)
    return np.array(ids, dtype=np.int64), np.stack(zs)


def teacher_forced(model: OracleModel, prompt, stream) -> np.ndarray:
    """Prefill then feed ``stream`` one token at a time. Returns logits [1 + len(stream), V]."""
    seq = Sequence(model)
    zs = [seq.prefill(prompt)]
    for t in stream:
        zs.append(seq.step(int(t)))
    return np.stack(zs)
