// Embedding gather, row norms, greedy-argmax reduction and the step-argument node.
#include <cuda_fp16.h>

#include <type_traits>

#include "misc.cuh"

namespace llm {

namespace {

constexpr int ROW_THREADS = 256;

// h[m] = tok_emb[token] (+ pos_emb[position] for GPT-2): "bare-metal-llm", section
// "What got built" (embedding lookup) and "Picking the model" (learned positions).
template <typename WT>
__global__ void __launch_bounds__(ROW_THREADS) k_embed(const EmbedParams p) {
  using ST = typename Elem<WT>::type;   // token-embedding element (int8 quants for Q8_0)
  using VT = typename VecT<WT>::type;   // learned positions (fp32 for Q8_0 models)
  const int m = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const StepArgs* a = p.args;
  int tok = a->tokens[m];
  const int pos = a->positions[m];
  if (tok < 0 || tok >= p.vocab) {
    if (threadIdx.x == 0) set_flag(p.flags, FLAG_BAD_TOKEN);
    tok = -1;
  }
  bool pos_ok = pos >= 0 && pos < p.n_ctx;
  if (!pos_ok && threadIdx.x == 0) set_flag(p.flags, FLAG_BAD_POSITION);
  const ST* te = reinterpret_cast<const ST*>(p.tok_emb) + (size_t)(tok < 0 ? 0 : tok) * p.d;
  const VT* pe = p.pos_emb ? reinterpret_cast<const VT*>(p.pos_emb) + (size_t)(pos_ok ? pos : 0) * p.d : nullptr;
  const __half* ts = std::is_same<WT, Q8>::value
                         ? reinterpret_cast<const __half*>(p.tok_scale) + (size_t)(tok < 0 ? 0 : tok) * (p.d / Q8_BLOCK)
                         : nullptr;
  for (int i = threadIdx.x; i < p.d; i += ROW_THREADS) {
    float v = 0.0f;
    if (tok >= 0) {
      if constexpr (std::is_same<WT, Q8>::value) v = (float)te[i] * __half2float(ts[i / Q8_BLOCK]);
      else v = to_f32(te[i]);
    }
    if (pe && pos_ok) v += to_f32(pe[i]);
    p.h[(size_t)m * p.d + i] = v;
  }
}

// LayerNorm ((x - mean) / sqrt(var + eps) * g + b, biased variance) or RMSNorm
// (x / sqrt(mean(x^2) + eps) * g): one warp per row, warp-shuffle reductions
// ("rvllm-metal", section "How a GPU runs your kernel": simd_sum, then no
// threadgroup round trip is needed when one simdgroup owns the row). The row is
// read with 16-byte loads; the variance pass re-reads it from L1.
constexpr int NORM_ROWS = 8;   // rows (warps) per CTA

// NORM_NV float4 per lane of the row are held in registers: d <= 128 NORM_NV. The gains and
// biases sit in shared memory, so the registers hold only the row and a prefill's norm keeps
// four CTAs (32 rows) an SM in flight instead of two.
template <typename WT, typename AT, int NORM_NV>
__global__ void __launch_bounds__(NORM_ROWS * 32) k_norm(const NormParams p) {
  __shared__ __align__(16) float s_g[NORM_NV * 128], s_b[NORM_NV * 128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * NORM_ROWS + warp;
  const int d4 = p.d >> 2;
  const WT* gw = reinterpret_cast<const WT*>(p.g);
  const WT* bw = reinterpret_cast<const WT*>(p.b);
  const int ld = std::is_same<AT, Split>::value ? 2 * p.d : p.d;
  // gains / biases: weights, so staged before waiting on the producer
  for (int i = threadIdx.x; i < p.d; i += NORM_ROWS * 32) {
    s_g[i] = to_f32(gw[i]);
    s_b[i] = bw ? to_f32(bw[i]) : 0.0f;
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (r >= p.rows) return;
  int src = r;
  if (p.use_last_row && p.args->last_row) src = p.args->last_row[r];
  float4 v[NORM_NV];
  float mean, scale;
  warp_row_stats<NORM_NV>(p.h + (size_t)src * p.d, p.d, p.layer_norm != 0, p.eps, v, mean, scale);
#pragma unroll
  for (int j = 0; j < NORM_NV; ++j) {
    const int i = lane + 32 * j;
    if (i >= d4) continue;
    const float xv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
    const float4 g4 = *reinterpret_cast<const float4*>(s_g + 4 * i);
    const float4 b4 = *reinterpret_cast<const float4*>(s_b + 4 * i);
    const float gv[4] = {g4.x, g4.y, g4.z, g4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
    float y[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) y[t] = norm_apply(xv[t], mean, scale, gv[t], bv[t]);
    act_store4<AT>(p.out, r, ld, 4 * i, y);
  }
}

// next_ids[b] = argmax over the per-tile partials of row b ("rvllm-metal", section
// "What the kernels do": a GPU argmax so one integer per sequence comes back).
__global__ void __launch_bounds__(ROW_THREADS) k_argmax_reduce(const ArgmaxParams p) {
  __shared__ float sv[ROW_THREADS / 32];
  __shared__ int si[ROW_THREADS / 32];
  const int b = blockIdx.x;
  pdl_wait();
  const StepArgs* a = p.args;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int t = threadIdx.x; t < p.n_tiles; t += ROW_THREADS) {
    const float v = p.part_val[(size_t)t * a->B + b];
    const int i = p.part_idx[(size_t)t * a->B + b];
    if (argmax_better(v, i, best, bi)) { best = v; bi = i; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (argmax_better(ov, oi, best, bi)) { best = ov; bi = oi; }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { sv[warp] = best; si[warp] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < ROW_THREADS / 32; ++w)
      if (argmax_better(sv[w], si[w], best, bi)) { best = sv[w]; bi = si[w]; }
    if (best != best) set_flag(p.flags, FLAG_NAN_LOGIT);
    a->next_ids[b] = bi;
  }
}

__global__ void k_set_args(StepArgs* dst, StepArgs v) { *dst = v; }

template <typename WT>
cudaError_t embed_t(const EmbedParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t c = make_launch_cfg(dim3(p.M), dim3(ROW_THREADS), 0, s, attr, pdl);
  return cudaLaunchKernelEx(&c, k_embed<WT>, p);
}
template <typename WT, typename AT>
cudaError_t norm_t(const NormParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t c = make_launch_cfg(dim3((p.rows + NORM_ROWS - 1) / NORM_ROWS), dim3(NORM_ROWS * 32), 0, s,
                                         attr, pdl);
  const int nv = (p.d + 127) / 128;   // registers sized for the row width
  if (nv <= 2) return cudaLaunchKernelEx(&c, k_norm<WT, AT, 2>, p);
  if (nv <= 4) return cudaLaunchKernelEx(&c, k_norm<WT, AT, 4>, p);
  if (nv <= 6) return cudaLaunchKernelEx(&c, k_norm<WT, AT, 6>, p);
  if (nv <= 8) return cudaLaunchKernelEx(&c, k_norm<WT, AT, 8>, p);
  if (nv <= 13) return cudaLaunchKernelEx(&c, k_norm<WT, AT, 13>, p);
  return cudaLaunchKernelEx(&c, k_norm<WT, AT, ROW_NV>, p);
}

}  // namespace

cudaLaunchConfig_t make_launch_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr,
                                   bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

cudaError_t launch_embed(const EmbedParams& p, int wdt, cudaStream_t s, bool pdl) {
  if (p.M <= 0) return cudaSuccess;
  if (wdt == DT_Q8) return (p.d % Q8_BLOCK == 0 && p.tok_scale) ? embed_t<Q8>(p, s, pdl) : cudaErrorInvalidValue;
  return wdt == DT_F32 ? embed_t<float>(p, s, pdl) : embed_t<bf16>(p, s, pdl);
}

cudaError_t launch_norm(const NormParams& p, int wdt, int adt, cudaStream_t s, bool pdl) {
  if (p.rows <= 0) return cudaSuccess;
  if (p.d % 8 != 0 || p.d > ROW_NV * 128) return cudaErrorInvalidValue;
  if (wdt == DT_F32 && adt == DT_F32) return norm_t<float, float>(p, s, pdl);
  if (wdt == DT_BF16 && adt == DT_SPLIT) return norm_t<bf16, Split>(p, s, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t launch_argmax(const ArgmaxParams& p, int B, cudaStream_t s, bool pdl) {
  if (B <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t c = make_launch_cfg(dim3(B), dim3(ROW_THREADS), 0, s, attr, pdl);
  return cudaLaunchKernelEx(&c, k_argmax_reduce, p);
}

cudaError_t launch_set_args(StepArgs* dst, const StepArgs& v, cudaStream_t s) {
  k_set_args<<<1, 1, 0, s>>>(dst, v);
  return cudaGetLastError();
}

const void* set_args_kernel() { return reinterpret_cast<const void*>(&k_set_args); }

// Self-test of the bounded wait every kernel uses: an mbarrier that nothing arrives at, so
// the wait gives up after its limit (about one second) and sets FLAG_WAIT_TIMEOUT.
__global__ void k_selftest_wait(unsigned* flags) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, flags);
}

cudaError_t launch_selftest_wait(unsigned* flags, cudaStream_t s) {
  k_selftest_wait<<<1, 32, 0, s>>>(flags);
  return cudaGetLastError();
}

}  // namespace llm
