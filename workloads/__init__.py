"""Seeded synthetic inputs for the KV-cached decoder step.

This module is shared by the float64 oracle and by the CUDA path's tests and
bench. It holds model shapes, workload shapes and seeded random draws only:
no part of the decoder's arithmetic lives here.

Seeds (numpy ``default_rng``, PCG64):
  0  weight matrices and embeddings, one draw per tensor in a fixed order
  1  prompt token ids, uniform over [0, vocab)
  2  context lengths
  3  block-table permutation of the paged KV pool
  4  teacher-forced decode streams
  5  optional perturbation of norm gains / biases (tests only); Q/K-norm gains and the
     Llama variant's attention biases are drawn after the final norm's

Weights are drawn as float32 N(0, 0.02) ("weights N(0,0.02) from seed, biases
0"); norm gains are 1 and biases 0 unless ``perturb`` asks for non-trivial
ones. bf16 models round each float32 draw to the nearest bf16 (ties to even)
and carry it as the uint16 bit pattern, so both sides read identical values.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, List, Optional

import numpy as np

ARCH_GPT2 = 0
ARCH_LLAMA = 1
DTYPE_F32 = 0
DTYPE_BF16 = 1
DTYPE_Q8 = 2       # matrices as Q8_0: int8 quants, one fp16 scale per 32-weight block
KV_BLOCK = 16
Q8_BLOCK = 32

SEED_WEIGHTS = 0
SEED_PROMPTS = 1
SEED_LENGTHS = 2
SEED_TABLES = 3
SEED_STREAM = 4
SEED_PERTURB = 5


@dataclass(frozen=True)
class ModelShape:
    name: str
    arch: int
    dtype: int
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    n_ctx: int
    norm_eps: float = 1e-5
    rope_theta: float = 1e5
    # model-feature variants (Llama variant; the window applies to either)
    sliding_window: int = 0          # W > 0: a query at position p sees keys p-W+1 .. p
    sliding_window_pattern: int = 0  # 0: every layer windowed; P > 0: every P-th layer (l+1 = P, 2P, ..) global
    qk_norm: bool = False            # RMSNorm (gain [head_dim] per layer) on each q and k head before RoPE
    rope_scaling: Optional[tuple] = None   # Llama-3 frequency scaling: (factor, low_freq_factor,
                                           # high_freq_factor, original_max_position)
    attn_bias: bool = False          # biases on the q, k, v projections (Llama variant)

    @property
    def qkv_dim(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def up_dim(self) -> int:
        # Llama fuses gate and up into one [2F, d] matrix (gate rows first).
        return 2 * self.d_ff if self.arch == ARCH_LLAMA else self.d_ff

    @property
    def elt_bytes(self) -> float:
        """Bytes a matrix weight takes: 4 (fp32), 2 (bf16), 1 + 2/32 (Q8_0 quant plus its share of a scale)."""
        return {DTYPE_F32: 4, DTYPE_BF16: 2, DTYPE_Q8: 1 + 2 / Q8_BLOCK}[self.dtype]

    def layer_params(self) -> int:
        d = self.d_model
        return self.qkv_dim * d + self.n_heads * self.head_dim * d + self.up_dim * d + self.d_ff * d


GPT2_124M_F32 = ModelShape("gpt2-124m", ARCH_GPT2, DTYPE_F32, 12, 768, 12, 12, 64, 3072, 50257, 1024)
GPT2_124M_BF16 = replace(GPT2_124M_F32, name="gpt2-124m-bf16", dtype=DTYPE_BF16)
SMOLLM2_360M = ModelShape("smollm2-360m", ARCH_LLAMA, DTYPE_BF16, 32, 960, 15, 5, 64, 2560, 49152, 8192)
GPT2_XL_BF16 = ModelShape("gpt2-xl", ARCH_GPT2, DTYPE_BF16, 48, 1600, 25, 25, 64, 6400, 50257, 1024)
GPT2_124M_Q8 = replace(GPT2_124M_F32, name="gpt2-124m-q8", dtype=DTYPE_Q8)


@dataclass(frozen=True)
class Workload:
    """One benchmark / parity workload (prompt lengths, batch, decode steps, KV layout)."""
    name: str
    model: ModelShape
    batch: int
    prompt_len: int            # fixed prompt length (0 when lengths are drawn)
    len_lo: int = 0            # drawn context lengths, inclusive range (seed 2)
    len_hi: int = 0
    decode_steps: int = 0
    mode: str = "greedy"       # "greedy" | "teacher" | "prefill"
    contiguous_kv: bool = False
    shuffle_tables: bool = True
    weight_scale: float = 1.0  # 8.0 for the magnitude-scaled GPT-2 copy
    kv_dtype: int = DTYPE_F32  # element type of the KV cache (DTYPE_BF16: rounded when written)

    def lengths(self) -> np.ndarray:
        if self.prompt_len:
            return np.full(self.batch, self.prompt_len, dtype=np.int32)
        return draw_lengths(self.batch, self.len_lo, self.len_hi)

    def max_ctx(self) -> int:
        return int(self.lengths().max()) + self.decode_steps


# The five workloads, named by what they are.
W_GPT2_F32_B1 = Workload("gpt2-124m-fp32-b1-greedy", GPT2_124M_F32, batch=1, prompt_len=8,
                         decode_steps=16, mode="greedy", shuffle_tables=False)
W_GPT2_F32_B32 = Workload("gpt2-124m-fp32-b32-teacher", GPT2_124M_F32, batch=32, prompt_len=128,
                          decode_steps=128, mode="teacher", contiguous_kv=True, shuffle_tables=False)
W_GPT2_F32_B32_X8 = replace(W_GPT2_F32_B32, name="gpt2-124m-fp32x8-b32-teacher", weight_scale=8.0)
W_SMOLLM2_B64 = Workload("smollm2-360m-bf16-b64-ctx64to2048", SMOLLM2_360M, batch=64, prompt_len=0,
                         len_lo=64, len_hi=2048, decode_steps=1, mode="teacher")
W_GPT2_BF16_PREFILL = Workload("gpt2-124m-bf16-prefill-16x1024", GPT2_124M_BF16, batch=16,
                               prompt_len=1024, mode="prefill")
W_GPT2XL_B256 = Workload("gpt2-xl-bf16-b256-ctx1024", GPT2_XL_BF16, batch=256, prompt_len=960,
                         decode_steps=64, mode="teacher")
# the batch-1 greedy workload with Q8_0 weights (the int8 weight stream)
W_GPT2_Q8_B1 = replace(W_GPT2_F32_B1, name="gpt2-124m-q8-b1-greedy", model=GPT2_124M_Q8)

WORKLOADS = {w.name: w for w in (W_GPT2_F32_B1, W_GPT2_F32_B32, W_GPT2_F32_B32_X8, W_SMOLLM2_B64,
                                 W_GPT2_BF16_PREFILL, W_GPT2XL_B256, W_GPT2_Q8_B1)}


# ----------------------------------------------------------------------------------------------
# bf16 bit patterns
# ----------------------------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); return uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    # keep NaN a NaN (never produced by the generators, but be safe)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, np.uint32(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------------------------

@dataclass
class Weights:
    """Host copy of a model's parameters.

    Matrices are row-major [out_features, in_features]; embeddings [rows, d].
    ``dtype`` DTYPE_F32 → float32 arrays; DTYPE_BF16 → uint16 bf16 bit patterns.
    Per-layer lists hold one entry per layer; absent tensors are None.
    """
    shape: ModelShape
    tok_emb: np.ndarray
    pos_emb: Optional[np.ndarray]
    ln1_w: List[np.ndarray]
    ln1_b: List[Optional[np.ndarray]]
    w_qkv: List[np.ndarray]
    b_qkv: List[Optional[np.ndarray]]
    w_o: List[np.ndarray]
    b_o: List[Optional[np.ndarray]]
    ln2_w: List[np.ndarray]
    ln2_b: List[Optional[np.ndarray]]
    w_up: List[np.ndarray]
    b_up: List[Optional[np.ndarray]]
    w_down: List[np.ndarray]
    b_down: List[Optional[np.ndarray]]
    lnf_w: np.ndarray
    lnf_b: Optional[np.ndarray]
    q_norm_w: Optional[List[np.ndarray]] = None   # [head_dim] per layer when shape.qk_norm
    k_norm_w: Optional[List[np.ndarray]] = None
    # Q8_0 models: the fp16 block scales [rows, K / 32] of each int8 matrix
    tok_emb_scale: Optional[np.ndarray] = None
    w_qkv_scale: Optional[List[np.ndarray]] = None
    w_o_scale: Optional[List[np.ndarray]] = None
    w_up_scale: Optional[List[np.ndarray]] = None
    w_down_scale: Optional[List[np.ndarray]] = None

    def as_f64(self, a: Optional[np.ndarray]) -> Optional[np.ndarray]:
        """Widen one stored tensor to float64 (bf16 patterns are decoded exactly; int8 quants are
        returned as their integer values, without their scales)."""
        if a is None:
            return None
        if a.dtype == np.uint16:
            return bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)


def _store(x: np.ndarray, dtype: int) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == DTYPE_BF16 else np.ascontiguousarray(x, dtype=np.float32)


def quantize_q8_0(x: np.ndarray):
    """Input preparation of a Q8_0 model: each row is cut into 32-value blocks, each block gets
    the fp16 scale d = max|x| / 127 and the int8 quants round(x / d). Returns (int8 [rows, K],
    float16 [rows, K / 32]); the model is exactly d * q."""
    rows, K = x.shape
    assert K % Q8_BLOCK == 0
    b = x.reshape(rows, K // Q8_BLOCK, Q8_BLOCK).astype(np.float32)
    d = (np.abs(b).max(axis=2) / np.float32(127)).astype(np.float16)
    df = d.astype(np.float32)[:, :, None]
    q = np.where(df > 0, np.rint(b / np.where(df > 0, df, 1)), 0)
    q = np.clip(q, -127, 127).astype(np.int8)
    return np.ascontiguousarray(q.reshape(rows, K)), np.ascontiguousarray(d)


def make_weights(shape: ModelShape, scale: float = 1.0, perturb: bool = False,
                 seed: int = SEED_WEIGHTS) -> Weights:
    """Draw a random-init model.

    Draw order on one generator (seed 0): tok_emb, pos_emb (GPT-2 only), then per
    layer w_qkv, w_o, w_up (gate rows then up rows for Llama), w_down. Each is
    float32 N(0, 0.02) times ``scale``. Norm gains are 1 and all biases 0, unless
    ``perturb`` is set: then gains are 1 + N(0, 0.1) and biases N(0, 0.05), drawn
    from a second generator (seed 5) so the matrices stay the same.
    """
    rng = np.random.default_rng(seed)
    prng = np.random.default_rng(SEED_PERTURB)
    s = np.float32(0.02 * scale)
    d, L = shape.d_model, shape.n_layers
    gpt2 = shape.arch == ARCH_GPT2

    q8 = shape.dtype == DTYPE_Q8
    vdt = DTYPE_F32 if q8 else shape.dtype      # Q8_0 models keep vectors and positions in fp32
    scales: Dict[str, list] = {k: [] for k in ("w_qkv_scale", "w_o_scale", "w_up_scale", "w_down_scale")}

    def mat(rows: int, cols: int, name: str = None):
        x = rng.standard_normal((rows, cols), dtype=np.float32) * s
        if not q8:
            return _store(x, shape.dtype)
        q, dsc = quantize_q8_0(x)
        if name:
            scales[name].append(dsc)
            return q
        return q, dsc

    def gain(n: int) -> np.ndarray:
        g = np.ones(n, np.float32)
        if perturb:
            g = g + prng.standard_normal(n, dtype=np.float32) * np.float32(0.1)
        return _store(g, vdt)

    def bias(n: int, present: bool = None) -> Optional[np.ndarray]:
        if not (gpt2 if present is None else present):
            return None
        b = np.zeros(n, np.float32)
        if perturb:
            b = prng.standard_normal(n, dtype=np.float32) * np.float32(0.05)
        return _store(b, vdt)

    tok = mat(shape.vocab, d)
    tok_scale = None
    if q8:
        tok, tok_scale = tok
    pos = (_store(rng.standard_normal((shape.n_ctx, d), dtype=np.float32) * s, vdt) if gpt2 else None)
    lists: Dict[str, list] = {k: [] for k in ("ln1_w", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_w",
                                              "ln2_b", "w_up", "b_up", "w_down", "b_down")}
    for _ in range(L):
        lists["w_qkv"].append(mat(shape.qkv_dim, d, "w_qkv_scale"))
        lists["w_o"].append(mat(d, shape.n_heads * shape.head_dim, "w_o_scale"))
        lists["w_up"].append(mat(shape.up_dim, d, "w_up_scale"))
        lists["w_down"].append(mat(d, shape.d_ff, "w_down_scale"))
    for _ in range(L):
        lists["ln1_w"].append(gain(d))
        lists["ln1_b"].append(bias(d))
        lists["b_qkv"].append(bias(shape.qkv_dim, gpt2 or shape.attn_bias))
        lists["b_o"].append(bias(d))
        lists["ln2_w"].append(gain(d))
        lists["ln2_b"].append(bias(d))
        lists["b_up"].append(bias(shape.up_dim))
        lists["b_down"].append(bias(d))
    lnf_w, lnf_b = gain(d), bias(d)
    qn = [gain(shape.head_dim) for _ in range(L)] if shape.qk_norm else None
    kn = [gain(shape.head_dim) for _ in range(L)] if shape.qk_norm else None
    extra = dict(tok_emb_scale=tok_scale, **scales) if q8 else {}
    return Weights(shape=shape, tok_emb=tok, pos_emb=pos, lnf_w=lnf_w, lnf_b=lnf_b, q_norm_w=qn, k_norm_w=kn, **lists,
                   **extra)


# ----------------------------------------------------------------------------------------------
# token streams, lengths, block tables
# ----------------------------------------------------------------------------------------------

def draw_prompts(lengths, vocab: int, seed: int = SEED_PROMPTS) -> List[np.ndarray]:
    """One int32 array per sequence, ids uniform over [0, vocab)."""
    rng = np.random.default_rng(seed)
    return [rng.integers(0, vocab, size=int(n), dtype=np.int64).astype(np.int32) for n in lengths]


def draw_lengths(batch: int, lo: int, hi: int, seed: int = SEED_LENGTHS) -> np.ndarray:
    """Context lengths uniform over [lo, hi] inclusive."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=batch, dtype=np.int64).astype(np.int32)


def draw_stream(batch: int, steps: int, vocab: int, seed: int = SEED_STREAM) -> np.ndarray:
    """Teacher-forced decode inputs [steps, batch], uniform over [0, vocab)."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, vocab, size=(steps, batch), dtype=np.int64).astype(np.int32)


def blocks_needed(ctx: int, block: int = KV_BLOCK) -> int:
    return (int(ctx) + block - 1) // block


def make_block_tables(ctx_per_seq, max_blocks_per_seq: int, shuffle: bool = True,
                      seed: int = SEED_TABLES, block: int = KV_BLOCK):
    """Assign physical KV blocks to sequences.

    ``ctx_per_seq[b]`` is the number of token slots sequence b will ever hold. The
    pool has exactly sum(ceil(ctx/block)) blocks; with ``shuffle`` the physical ids
    are a seeded permutation of the pool, otherwise sequence b gets consecutive ids.
    Unused table entries are -1. Returns (tables int32 [B, max_blocks_per_seq], n_blocks).
    """
    need = [blocks_needed(c, block) for c in ctx_per_seq]
    if max(need) > max_blocks_per_seq:
        raise ValueError("max_blocks_per_seq too small")
    total = int(sum(need))
    ids = np.arange(total, dtype=np.int64)
    if shuffle:
        ids = np.random.default_rng(seed).permutation(total)
    tables = np.full((len(need), max_blocks_per_seq), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(need):
        tables[b, :n] = ids[o:o + n]
        o += n
    return tables, total


def identity_tables(batch: int, max_blocks_per_seq: int) -> np.ndarray:
    """Sequence b owns blocks [b*max_blocks_per_seq, (b+1)*max_blocks_per_seq)."""
    return (np.arange(batch * max_blocks_per_seq, dtype=np.int32)
            .reshape(batch, max_blocks_per_seq))


def tiny_shape(arch: int, dtype: int = DTYPE_F32, **kw) -> ModelShape:
    """Small model shapes for oracle brute force and fast GPU parity runs."""
    base = dict(name="tiny", arch=arch, dtype=dtype, n_layers=1, d_model=8, n_heads=2,
                n_kv_heads=2, head_dim=4, d_ff=16, vocab=11, n_ctx=16)
    base.update(kw)
    return ModelShape(**base)
