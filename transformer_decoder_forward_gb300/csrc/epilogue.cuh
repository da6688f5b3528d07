// Output-tile epilogues shared by every projection kernel (CUDA-core GEMV, SIMT
// GEMM, tcgen05 GEMMs). The producer leaves an fp32 tile tile[m][c] in shared
// memory (row stride ldt) holding y = x . W^T for rows m0.. and tile columns
// c = 0..ncols-1, then every thread of the block calls run_epilogue().
//
// What each kind fuses ("rvllm-metal", section "What the kernels do"; "bare-metal-llm",
// section "What got built"):
//   RESID   residual add after the output / down projection;
//   GELU    GPT-2's GELU-tanh with the tanh argument clamped to +-15 ("batch_forge");
//   SWIGLU  silu(gate) * up;
//   QKV     bias, Q/K norm and RoPE on q and k (Llama), kv_write of k and v into the paged cache
//           (fp32 or bf16);
//   HEAD    tied-LM-head logits and a per-tile greedy argmax partial.
//
// Latency: the per-tile bias and the per-row KV slot are staged in shared memory
// once, and read-modify-write loads are issued in batches before their stores, so a
// thread never waits on one global round trip per element.
#pragma once
#include "common.cuh"

namespace llm {

constexpr int EPI_MAX_ROWS = 256;   // rows of one epilogue call (every projection tile fits)
constexpr int EPI_MAX_COLS = 128;   // tile columns of one epilogue call (two 64-column sub-tiles)

// Element n of a bias / gain vector of a model with weight type WT (fp32 for Q8_0 models).
template <typename WT>
__device__ __forceinline__ float bias_at(const void* b, int n) {
  using VT = typename VecT<WT>::type;
  return b ? to_f32(reinterpret_cast<const VT*>(b)[n]) : 0.0f;
}

// RoPE angle pos * inv_freq[d] reduced to about [-pi, pi] in fp32 without losing the
// position's precision. inv_freq is split on the host into hi (11 significant bits, so
// pos * hi is exact for pos < 2^13) + lo. The reduction is the Cody-Waite method (W. J. Cody
// and W. Waite, "Software Manual for the Elementary Functions", 1980): 2*pi is written as
// the sum of three floats whose leading parts have few significant bits, so each product
// k * part is exact for the quotients k that occur and the subtractions lose nothing.
__device__ __forceinline__ void rope_sincos(int pos, float2 f, float* s, float* c) {
  const float p = (float)pos;
  const float a_hi = p * f.x;                         // exact
  const float a_lo = p * f.y;
  const float k = rintf(a_hi * 0.15915494309189535f);   // 1 / (2 pi)
  float r = fmaf(-k, 6.28125f, a_hi);                 // 2 pi = 6.28125 + c2 + c3 (c2, c3 floats)
  r = fmaf(-k, 1.9353071693331003e-3f, r);
  r = fmaf(-k, 1.0253376273028358e-11f, r);
  r += a_lo;
  sincosf(r, s, c);
}

// tile: fp32 [.., ldt] in shared memory. Rows m0 .. m0+mrows-1 of the launch (mrows <=
// EPI_MAX_ROWS), tile columns 0..ncols-1 (ncols = 64 or 128, n0 a multiple of 64) map to
// output column n0 + c. SWIGLU: each 64-column sub-tile s holds 32 gate rows then the 32
// matching up rows, output columns n0 + 32 s .. n0 + 32 s + 31. HEAD: one argmax partial
// per 64-column sub-tile. N = output width. Every thread of the block must call it (it
// synchronises the block).
// WT: weight (and bias) type; activations are stored as ActOf<WT> (fp32 or a bf16 pair),
// the KV cache in fp32.
//
// run_epilogue = stage + apply. A kernel whose tile rows and columns are known before its
// accumulator is ready can call epi_stage early (with its own thread subset) and epi_apply
// once the tile is in shared memory, so the bias, position and KV-block loads overlap the
// contraction; a block-wide barrier must separate the two.

struct EpiStaging {
  float bias[EPI_MAX_COLS];
  int pos[EPI_MAX_ROWS];
  int blk[EPI_MAX_ROWS];
};
__device__ __forceinline__ EpiStaging& epi_staging() {
  __shared__ EpiStaging st;   // one per CTA
  return st;
}

// Stage the call's bias columns and (QKV) row positions / KV blocks; threads tid of nth.
template <typename WT>
__device__ void epi_stage(const Epilogue& e, int m0, int mrows, int n0, int ncols, int N, int tid, int nth) {
  EpiStaging& st = epi_staging();
  float* s_bias = st.bias;
  int* s_pos = st.pos;
  int* s_blk = st.blk;
  for (int t = tid; t < ncols; t += nth) {
    float b = 0.0f;
    if (e.bias) {
      if (e.kind == EPI_SWIGLU) {
        const int j = n0 + (t >> 6) * 32 + (t & 31);
        if (j < N) b = bias_at<WT>(e.bias, (t & 63) < 32 ? j : N + j);
      } else if (n0 + t < N) {
        b = bias_at<WT>(e.bias, n0 + t);
      }
    }
    s_bias[t] = b;
  }
  if (e.kind == EPI_QKV) {
    const StepArgs* a = e.args;
    const int H = e.n_heads;
    const bool kv_cols = n0 + ncols > H * HD;   // this tile holds k or v columns
    for (int m = tid; m < mrows; m += nth) {
      const int row = m0 + m;
      const int pos = a->positions[row];
      s_pos[m] = pos;
      if (kv_cols) {
        const int seq = a->row_seq ? a->row_seq[row] : row;
        s_blk[m] = kv_block(e.kv, a->block_tables, seq, pos, e.flags);
      }
    }
  }
}

// QKV: bias, Q/K norm (QKN) and RoPE on q and k, kv_write of k and v. unit = (row, head of the
// tile, g): dims 4g..4g+3 and 32+4g..32+4g+3 of the head, so a RoPE pair (d, d + 32) stays in
// one thread; N is a multiple of 64 (whole heads).
template <typename WT, bool QKN>
__device__ __forceinline__ void epi_qkv(const Epilogue& e, const float* tile, int ldt, int m0, int mrows, int n0,
                                        int ncols, int N, int tid, int nth, const float* s_bias, const int* s_pos,
                                        const int* s_blk) {
  const int H = e.n_heads, Hkv = e.kv.n_kv_heads;
  const int units_row = (ncols / HD) * 8;
  for (int i = tid; i < mrows * units_row; i += nth) {
    const int m = i / units_row, u = i - m * units_row;
    const int c = (u >> 3) * HD + (u & 7) * 4;   // tile column of dim d = 4g
    const int n = n0 + c;
    if (n >= N) continue;
    const int hh = n / HD, d = n - hh * HD;
    const int row = m0 + m;
    const int pos = s_pos[m];
    const bool is_q = hh < H, is_k = !is_q && hh < H + Hkv;
    float v0[4], v1[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      v0[t] = tile[m * ldt + c + t] + s_bias[c + t];
      v1[t] = tile[m * ldt + c + HD / 2 + t] + s_bias[c + HD / 2 + t];
    }
    if constexpr (QKN) {
      if (is_q || is_k) {
        // Q/K norm: RMSNorm of the head over its 64 values, before RoPE. The head's 8 units
        // are 8 consecutive i, so 8 consecutive lanes of one warp (every caller's thread index
        // is the hardware lane mod 32 and its thread count a multiple of 32), all of them here.
        float ss = 0.0f;
#pragma unroll
        for (int t = 0; t < 4; ++t) ss += v0[t] * v0[t] + v1[t] * v1[t];
        const unsigned gmask = 0xFFu << (threadIdx.x & 24);
        ss += __shfl_xor_sync(gmask, ss, 1);
        ss += __shfl_xor_sync(gmask, ss, 2);
        ss += __shfl_xor_sync(gmask, ss, 4);
        const float r = 1.0f / sqrtf(ss / HD + e.qk_eps);
        const void* gw = is_q ? e.qn_g : e.kn_g;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          v0[t] = v0[t] * r * bias_at<WT>(gw, d + t);
          v1[t] = v1[t] * r * bias_at<WT>(gw, d + HD / 2 + t);
        }
      }
    }
    if (e.rope && (is_q || is_k)) {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float sn, co;
        rope_sincos(pos, e.rope_tab[d + t], &sn, &co);
        const float r0 = v0[t] * co - v1[t] * sn;
        const float r1 = v1[t] * co + v0[t] * sn;
        v0[t] = r0;
        v1[t] = r1;
      }
    }
    float* dst;
    if (is_q) {
      dst = e.q_out + (size_t)row * H * HD + hh * HD;
    } else {
      const int pb = s_blk[m];
      if (pb < 0) continue;
      const int g = is_k ? hh - H : hh - H - Hkv;
      const size_t off = kv_offset(e.kv, pb, g, pos & (KVB - 1));
      if (e.kv.dtype == DT_BF16) {
        // a bf16 cache stores k and v rounded to nearest (ties to even)
        bf16* kd = reinterpret_cast<bf16*>(is_k ? e.kv.k : e.kv.v) + off;
        const __nv_bfloat162 a0 = __floats2bfloat162_rn(v0[0], v0[1]), a1 = __floats2bfloat162_rn(v0[2], v0[3]);
        const __nv_bfloat162 b0 = __floats2bfloat162_rn(v1[0], v1[1]), b1 = __floats2bfloat162_rn(v1[2], v1[3]);
        *reinterpret_cast<uint2*>(kd + d) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a0), *reinterpret_cast<const uint32_t*>(&a1));
        *reinterpret_cast<uint2*>(kd + d + HD / 2) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
        continue;
      }
      dst = reinterpret_cast<float*>(is_k ? e.kv.k : e.kv.v) + off;
    }
    *reinterpret_cast<float4*>(dst + d) = make_float4(v0[0], v0[1], v0[2], v0[3]);
    *reinterpret_cast<float4*>(dst + d + HD / 2) = make_float4(v1[0], v1[1], v1[2], v1[3]);
  }
}

// The QKV epilogue with Q/K norm, kept out of the projection kernels' inlined code.
template <typename WT>
__device__ __noinline__ void epi_qkv_norm(const Epilogue& e, const float* tile, int ldt, int m0, int mrows, int n0,
                                          int ncols, int N, int tid, int nth, const float* s_bias, const int* s_pos,
                                          const int* s_blk) {
  epi_qkv<WT, true>(e, tile, ldt, m0, mrows, n0, ncols, N, tid, nth, s_bias, s_pos, s_blk);
}

// The tile's outputs, from the staged values; threads tid of nth.
template <typename WT>
__device__ void epi_apply(const Epilogue& e, const float* tile, int ldt, int m0, int mrows, int n0, int ncols, int N,
                          int tid, int nth) {
  using AT = typename ActOf<WT>::type;
  EpiStaging& st = epi_staging();
  const float* s_bias = st.bias;
  const int* s_pos = st.pos;
  const int* s_blk = st.blk;
  // 4-wide path: 4 consecutive columns per thread step (vector loads and stores)
  const bool vec = (N % 4) == 0;
  switch (e.kind) {
    case EPI_STORE_F32:
    case EPI_STORE_ACT:
    case EPI_GELU: {
      const bool v4 = vec && (e.kind == EPI_STORE_F32 ? (e.ld_out % 4) == 0 : (e.ld_out % 8) == 0);
      if (v4) {
        const int c4n = ncols / 4;
        for (int i = tid; i < mrows * c4n; i += nth) {
          const int m = i / c4n, c = (i - m * c4n) * 4, n = n0 + c;
          if (n >= N) continue;
          float y[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            y[j] = tile[m * ldt + c + j] + s_bias[c + j];
            if (e.kind == EPI_GELU) y[j] = gelu_tanh_clamped(y[j]);
          }
          if (e.kind == EPI_STORE_F32)
            act_store4<float>(e.out, m0 + m, e.ld_out, n, y);
          else
            act_store4<AT>(e.out, m0 + m, e.ld_out, n, y);
        }
        break;
      }
      for (int i = tid; i < mrows * ncols; i += nth) {
        const int m = i / ncols, c = i - m * ncols, n = n0 + c;
        if (n >= N) continue;
        const float y = tile[m * ldt + c] + s_bias[c];
        if (e.kind == EPI_STORE_F32) reinterpret_cast<float*>(e.out)[(size_t)(m0 + m) * e.ld_out + n] = y;
        else act_store<AT>(e.out, m0 + m, e.ld_out, n, e.kind == EPI_STORE_ACT ? y : gelu_tanh_clamped(y));
      }
      break;
    }
    case EPI_RESID: {
      if (vec && (e.ld_resid % 4) == 0) {
        // residual read-modify-write, 16 bytes a step: a batch of loads, then the stores
        constexpr int RB = 4;
        const int c4n = ncols / 4, total = mrows * c4n;
        for (int i0 = 0; i0 < total; i0 += RB * nth) {
          float4 hv[RB];
          float4* ad[RB];
          bool ok[RB];
#pragma unroll
          for (int j = 0; j < RB; ++j) {
            const int i = i0 + j * nth + tid;
            const int m = i / c4n, c = (i - m * c4n) * 4;
            ok[j] = i < total && n0 + c < N;
            ad[j] = reinterpret_cast<float4*>(e.resid + (size_t)(m0 + m) * e.ld_resid + n0 + c);
            hv[j] = ok[j] ? *ad[j] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int j = 0; j < RB; ++j) {
            const int i = i0 + j * nth + tid;
            const int m = i / c4n, c = (i - m * c4n) * 4;
            if (!ok[j]) continue;
            const float* t = tile + m * ldt + c;
            *ad[j] = make_float4(hv[j].x + t[0] + s_bias[c], hv[j].y + t[1] + s_bias[c + 1],
                                 hv[j].z + t[2] + s_bias[c + 2], hv[j].w + t[3] + s_bias[c + 3]);
          }
        }
        break;
      }
      // residual read-modify-write: issue a batch of loads, then the stores
      constexpr int RB = 8;
      const int total = mrows * ncols;
      for (int i0 = 0; i0 < total; i0 += RB * nth) {
        float hv[RB];
        size_t ad[RB];
        bool ok[RB];
#pragma unroll
        for (int j = 0; j < RB; ++j) {
          const int i = i0 + j * nth + tid;
          const int m = i / ncols, c = i - m * ncols;
          ok[j] = i < total && n0 + c < N;
          ad[j] = (size_t)(m0 + m) * e.ld_resid + n0 + c;
          hv[j] = ok[j] ? e.resid[ad[j]] : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < RB; ++j) {
          const int i = i0 + j * nth + tid;
          const int m = i / ncols, c = i - m * ncols;
          if (ok[j]) e.resid[ad[j]] = hv[j] + tile[m * ldt + c] + s_bias[c];
        }
      }
      break;
    }
    case EPI_SWIGLU: {
      // sub-tile s, gate column c < 32: output column j = n0 + 32 s + c; N = d_ff
      const int nout = ncols / 2;
      if (vec && (e.ld_out % 8) == 0) {
        const int o4n = nout / 4;
        for (int i = tid; i < mrows * o4n; i += nth) {
          const int m = i / o4n, o = (i - m * o4n) * 4, c = (o >> 5) * 64 + (o & 31), j = n0 + o;
          if (j >= N) continue;
          float y[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float g = tile[m * ldt + c + t] + s_bias[c + t];
            const float u = tile[m * ldt + c + 32 + t] + s_bias[c + 32 + t];
            y[t] = silu_f(g) * u;
          }
          act_store4<AT>(e.out, m0 + m, e.ld_out, j, y);
        }
        break;
      }
      for (int i = tid; i < mrows * nout; i += nth) {
        const int m = i / nout, o = i - m * nout, c = (o >> 5) * 64 + (o & 31), j = n0 + o;
        if (j >= N) continue;
        const float g = tile[m * ldt + c] + s_bias[c];
        const float u = tile[m * ldt + c + 32] + s_bias[c + 32];
        act_store<AT>(e.out, m0 + m, e.ld_out, j, silu_f(g) * u);
      }
      break;
    }
    case EPI_QKV:
      // The Q/K-norm instance is a separate, non-inlined function: compiled into the loop, its
      // shuffles made every projection of the models without it about 0.4 us slower a launch.
      if (e.qn_g)
        epi_qkv_norm<WT>(e, tile, ldt, m0, mrows, n0, ncols, N, tid, nth, s_bias, s_pos, s_blk);
      else
        epi_qkv<WT, false>(e, tile, ldt, m0, mrows, n0, ncols, N, tid, nth, s_bias, s_pos, s_blk);
      break;
    case EPI_HEAD: {
      const StepArgs* a = e.args;
      float* logits = a->logits;
      if (logits) {
        for (int i = tid; i < mrows * ncols; i += nth) {
          const int m = i / ncols, c = i - m * ncols, n = n0 + c;
          if (n < N) logits[(size_t)(m0 + m) * e.vocab + n] = tile[m * ldt + c];
        }
      }
      // per-row argmax over each 64-column sub-tile: one warp per (row, sub-tile)
      const int warp = tid >> 5, lane = tid & 31, nwarps = nth >> 5;
      const int nsub = ncols / 64;
      const int B = a->B;
      for (int ms = warp; ms < mrows * nsub; ms += nwarps) {
        const int m = ms / nsub, sub = ms - m * nsub;
        const int tile_n = n0 / 64 + sub;
        float best = -INFINITY;
        int bi = 0x7fffffff;
        for (int c = sub * 64 + lane; c < sub * 64 + 64; c += 32) {
          const int n = n0 + c;
          if (n >= N) break;
          const float v = tile[m * ldt + c];
          if (argmax_better(v, n, best, bi)) { best = v; bi = n; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, best, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (argmax_better(ov, oi, best, bi)) { best = ov; bi = oi; }
        }
        if (lane == 0) {
          const size_t slot = (size_t)tile_n * B + (m0 + m);
          e.part_val[slot] = best;
          e.part_idx[slot] = bi;
        }
      }
      break;
    }
  }
}

// Every thread of the block: stage, then apply.
template <typename WT>
__device__ void run_epilogue(const Epilogue& e, const float* tile, int ldt, int m0, int mrows, int n0, int ncols,
                             int N) {
  __syncthreads();   // a previous call's readers are done with the staging arrays
  epi_stage<WT>(e, m0, mrows, n0, ncols, N, threadIdx.x, blockDim.x);
  __syncthreads();
  epi_apply<WT>(e, tile, ldt, m0, mrows, n0, ncols, N, threadIdx.x, blockDim.x);
}

}  // namespace llm
