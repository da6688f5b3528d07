// Output-tile epilogues shared by every projection kernel (CUDA-core GEMV, SIMT
// GEMM, tcgen05 GEMM). The producer leaves an fp32 tile tile[m][c] in shared
// memory (row stride ldt) holding y = x . W^T for rows m0.. and tile columns
// c = 0..ncols-1, then every thread of the block calls run_epilogue().
//
// What each kind fuses ("rvllm-metal", section "What the kernels do"; "bare-metal-llm",
// section "What got built"):
//   RESID   residual add after the output / down projection;
//   GELU    GPT-2's GELU-tanh with the tanh argument clamped to +-15 ("batch_forge");
//   SWIGLU  silu(gate) * up;
//   QKV     bias, RoPE on q and k (Llama), kv_write of k and v into the paged cache;
//   HEAD    tied-LM-head logits and a per-tile greedy argmax partial.
#pragma once
#include "common.cuh"

namespace llm {

template <typename WT>
__device__ __forceinline__ float bias_at(const void* b, int n) {
  return b ? to_f32(reinterpret_cast<const WT*>(b)[n]) : 0.0f;
}

template <typename AT>
__device__ __forceinline__ void store_act(void* out, size_t i, float v) {
  reinterpret_cast<AT*>(out)[i] = from_f32<AT>(v);
}

// Angle of RoPE pair d at position pos, reduced to [-pi, pi] in double precision
// so that large positions keep their accuracy in the float sincos.
__device__ __forceinline__ void rope_sincos(int pos, int d, float theta, float* s, float* c) {
  const double inv_freq = exp2(-(2.0 * d / HD) * log2((double)theta));
  double a = (double)pos * inv_freq;
  const double two_pi = 6.283185307179586476925;
  a -= two_pi * rint(a / two_pi);
  sincosf((float)a, s, c);
}

// tile: fp32 [.., ldt] in shared memory. Rows m0 .. m0+mrows-1 of the launch,
// tile columns 0..ncols-1 map to output column n0 + c (for SWIGLU: gate row n0 + c
// for c < 32 and up row F + n0 + c - 32; output column n0 + c). N = output width.
template <typename WT, typename AT>
__device__ void run_epilogue(const Epilogue& e, const float* tile, int ldt, int m0, int mrows, int n0, int ncols,
                             int N) {
  const int tid = threadIdx.x, nth = blockDim.x;
  switch (e.kind) {
    case EPI_STORE_F32:
    case EPI_STORE_ACT:
    case EPI_RESID:
    case EPI_GELU: {
      for (int i = tid; i < mrows * ncols; i += nth) {
        const int m = i / ncols, c = i - m * ncols, n = n0 + c;
        if (n >= N) continue;
        const float y = tile[m * ldt + c] + bias_at<WT>(e.bias, n);
        const size_t row = (size_t)(m0 + m);
        if (e.kind == EPI_STORE_F32) {
          reinterpret_cast<float*>(e.out)[row * e.ld_out + n] = y;
        } else if (e.kind == EPI_STORE_ACT) {
          store_act<AT>(e.out, row * e.ld_out + n, y);
        } else if (e.kind == EPI_RESID) {
          e.resid[row * e.ld_resid + n] += y;
        } else {
          store_act<AT>(e.out, row * e.ld_out + n, gelu_tanh_clamped(y));
        }
      }
      break;
    }
    case EPI_SWIGLU: {
      // output column j = n0 + c (c < 32); N = d_ff
      for (int i = tid; i < mrows * 32; i += nth) {
        const int m = i >> 5, c = i & 31, j = n0 + c;
        if (j >= N) continue;
        const float g = tile[m * ldt + c] + bias_at<WT>(e.bias, j);
        const float u = tile[m * ldt + 32 + c] + bias_at<WT>(e.bias, N + j);
        store_act<AT>(e.out, (size_t)(m0 + m) * e.ld_out + j, silu_f(g) * u);
      }
      break;
    }
    case EPI_QKV: {
      const StepArgs* a = e.args;
      const int H = e.n_heads, Hkv = e.kv.n_kv_heads;
      // one thread per (row, head-column-pair) when rotating, per element otherwise
      const int per_row = ncols;
      for (int i = tid; i < mrows * per_row; i += nth) {
        const int m = i / per_row, c = i - m * per_row, n = n0 + c;
        if (n >= N) continue;
        const int hh = n / HD, d = n - hh * HD;
        const int row = m0 + m;
        const int pos = a->positions[row];
        const bool is_q = hh < H, is_k = !is_q && hh < H + Hkv;
        float v0 = tile[m * ldt + c] + bias_at<WT>(e.bias, n);
        float v1 = 0.0f;
        if (e.rope && (is_q || is_k)) {
          if (d >= HD / 2) continue;                  // the partner thread writes this element
          v1 = tile[m * ldt + c + HD / 2] + bias_at<WT>(e.bias, n + HD / 2);
          float s, co;
          rope_sincos(pos, d, e.rope_theta, &s, &co);
          const float r0 = v0 * co - v1 * s;
          const float r1 = v1 * co + v0 * s;
          v0 = r0;
          v1 = r1;
        }
        if (is_q) {
          float* q = e.q_out + (size_t)row * H * HD + hh * HD;
          q[d] = v0;
          if (e.rope) q[d + HD / 2] = v1;
          continue;
        }
        const int seq = a->row_seq ? a->row_seq[row] : row;
        const int pb = kv_block(e.kv, a->block_tables, seq, pos, e.flags);
        if (pb < 0) continue;
        const int g = is_k ? hh - H : hh - H - Hkv;
        WT* dst = reinterpret_cast<WT*>(is_k ? e.kv.k : e.kv.v) + kv_offset(e.kv, pb, g, pos & (KVB - 1));
        dst[d] = from_f32<WT>(v0);
        if (e.rope && is_k) dst[d + HD / 2] = from_f32<WT>(v1);
      }
      break;
    }
    case EPI_HEAD: {
      const StepArgs* a = e.args;
      float* logits = a->logits;
      if (logits) {
        for (int i = tid; i < mrows * ncols; i += nth) {
          const int m = i / ncols, c = i - m * ncols, n = n0 + c;
          if (n < N) logits[(size_t)(m0 + m) * e.vocab + n] = tile[m * ldt + c];
        }
      }
      // per-row argmax over this tile's columns: one warp per row
      const int warp = tid >> 5, lane = tid & 31, nwarps = nth >> 5;
      const int tile_n = n0 / ncols;
      for (int m = warp; m < mrows; m += nwarps) {
        float best = -INFINITY;
        int bi = 0x7fffffff;
        for (int c = lane; c < ncols; c += 32) {
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
          const size_t slot = (size_t)tile_n * a->B + (m0 + m);
          e.part_val[slot] = best;
          e.part_idx[slot] = bi;
        }
      }
      break;
    }
  }
}

}  // namespace llm
