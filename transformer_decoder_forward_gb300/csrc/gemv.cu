// Decode projection on CUDA cores: a weight stream for a handful of rows.
//
// Decode is memory bound: every step reads all weights once and does little
// arithmetic per byte ("rvllm-metal", section "The matmul pain story"). The
// pages' linear_small gives one simdgroup per output and re-reads the
// activations per output; here the activations of all M rows sit in shared
// memory and every weight element loaded (16-byte streaming loads, 8 lanes
// covering 128 contiguous bytes of a row) is used for all M rows.
//
// CTA = 256 threads = 8 warps; warp w owns tile columns 8w..8w+7; in a warp,
// lane = 4 row groups x 8 k-lanes and each thread holds 2 weight rows.
// Small matrices split K across CTAs (the pages' linear_mma_small splits K
// across simdgroups for the same reason: too few output tiles to fill the
// GPU); partial tiles go to a workspace and the last CTA to arrive for a tile
// sums them in split order (deterministic) and runs the epilogue.
#include <algorithm>

#include "epilogue.cuh"
#include "linear.cuh"

namespace llm {

namespace {

constexpr int GEMV_THREADS = 256;
constexpr int TL_LD = TILE_N + 1;   // padded row stride of the output tile in smem

template <typename WT, typename XT, typename AT, int MT>
__global__ void __launch_bounds__(GEMV_THREADS) k_gemv(const LinearParams p, int kc, int ks_total) {
  extern __shared__ __align__(16) float smem[];
  constexpr int VEC = Vec16<WT>::N;
  const int tile = blockIdx.x, ks = blockIdx.y, mbase = blockIdx.z * MT;
  const int mcount = min(MT, p.M - mbase);
  const int k0 = ks * kc;
  const int kcl = min(kc, p.K - k0);
  const int ldxs = kc + 4;
  float* xs = smem;                       // [MT][ldxs]
  float* tl = smem + MT * ldxs;           // [MT][TL_LD]
  const int F = p.N;                      // SWIGLU: output width = d_ff

  // Weights do not depend on earlier kernels: warm L2 with this CTA's rows before waiting.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 3, kl = lane & 7;
  const WT* W = reinterpret_cast<const WT*>(p.W);
  int wrow[2];
  bool rvalid[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int c = warp * 8 + g * 2 + r;   // tile column
    int row, outcol;
    if (p.swiglu) {
      outcol = tile * 32 + (c & 31);
      row = swiglu_row(tile * 32, c, F);
      rvalid[r] = outcol < F;
    } else {
      row = tile * TILE_N + c;
      rvalid[r] = row < p.N;
    }
    wrow[r] = rvalid[r] ? row : 0;
  }
  if (kl == 0) {
#pragma unroll
    for (int r = 0; r < 2; ++r)
      if (rvalid[r] && kcl > 0)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(W + (size_t)wrow[r] * p.K + k0));
  }
  pdl_wait();

  // Stage this CTA's slice of X (rows mbase.., columns k0..k0+kcl) as fp32.
  const XT* X = reinterpret_cast<const XT*>(p.X);
  for (int i = threadIdx.x; i < mcount * kcl; i += GEMV_THREADS) {
    const int m = i / kcl, k = i - m * kcl;
    xs[m * ldxs + k] = to_f32(X[(size_t)(mbase + m) * p.ldx + k0 + k]);
  }
  __syncthreads();

  float acc[2][MT];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = 0.0f;

  const bool vec_ok = (p.K % VEC) == 0;
  const int kvec_end = vec_ok ? (kcl / VEC) * VEC : 0;
  constexpr int U = MT <= 8 ? 4 : 2;
  constexpr int STRIDE = 8 * VEC;
  const WT* wp0 = W + (size_t)wrow[0] * p.K + k0;
  const WT* wp1 = W + (size_t)wrow[1] * p.K + k0;

  auto fma_chunk = [&](const uint4& w0, const uint4& w1, int k) {
    float f0[VEC], f1[VEC];
    Vec16<WT>::unpack(w0, f0);
    Vec16<WT>::unpack(w1, f1);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < mcount) {
        const float* xr = xs + m * ldxs + k;
#pragma unroll
        for (int j = 0; j < VEC; j += 4) {
          const float4 xv = *reinterpret_cast<const float4*>(xr + j);
          acc[0][m] = fmaf(f0[j], xv.x, acc[0][m]);
          acc[0][m] = fmaf(f0[j + 1], xv.y, acc[0][m]);
          acc[0][m] = fmaf(f0[j + 2], xv.z, acc[0][m]);
          acc[0][m] = fmaf(f0[j + 3], xv.w, acc[0][m]);
          acc[1][m] = fmaf(f1[j], xv.x, acc[1][m]);
          acc[1][m] = fmaf(f1[j + 1], xv.y, acc[1][m]);
          acc[1][m] = fmaf(f1[j + 2], xv.z, acc[1][m]);
          acc[1][m] = fmaf(f1[j + 3], xv.w, acc[1][m]);
        }
      }
    }
  };

  int k = kl * VEC;
  for (; k + (U - 1) * STRIDE + VEC <= kvec_end; k += U * STRIDE) {
    uint4 w0[U], w1[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      w0[u] = rvalid[0] ? ldg_stream16(wp0 + k + u * STRIDE) : make_uint4(0, 0, 0, 0);
      w1[u] = rvalid[1] ? ldg_stream16(wp1 + k + u * STRIDE) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) fma_chunk(w0[u], w1[u], k + u * STRIDE);
  }
  for (; k + VEC <= kvec_end; k += STRIDE) {
    const uint4 w0 = rvalid[0] ? ldg_stream16(wp0 + k) : make_uint4(0, 0, 0, 0);
    const uint4 w1 = rvalid[1] ? ldg_stream16(wp1 + k) : make_uint4(0, 0, 0, 0);
    fma_chunk(w0, w1, k);
  }
  // scalar tail (K not a multiple of the vector width)
  for (int kk = kvec_end + kl; kk < kcl; kk += 8) {
    const float a0 = rvalid[0] ? to_f32(wp0[kk]) : 0.0f;
    const float a1 = rvalid[1] ? to_f32(wp1[kk]) : 0.0f;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < mcount) {
        acc[0][m] = fmaf(a0, xs[m * ldxs + kk], acc[0][m]);
        acc[1][m] = fmaf(a1, xs[m * ldxs + kk], acc[1][m]);
      }
    }
  }

  // reduce over the 8 k-lanes
#pragma unroll
  for (int r = 0; r < 2; ++r) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float v = acc[r][m];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      if (kl == 0 && m < mcount) tl[m * TL_LD + warp * 8 + g * 2 + r] = v;
    }
  }
  __syncthreads();

  const int n0 = p.swiglu ? tile * 32 : tile * TILE_N;
  if (ks_total > 1) {
    const int ldp = gridDim.x * TILE_N;
    float* part = p.part + ((size_t)ks * p.M + mbase) * ldp + (size_t)tile * TILE_N;
    for (int i = threadIdx.x; i < mcount * TILE_N; i += GEMV_THREADS) {
      const int m = i / TILE_N, c = i - m * TILE_N;
      part[(size_t)m * ldp + c] = tl[m * TL_LD + c];
    }
    __threadfence();
    __syncthreads();
    __shared__ unsigned ticket;
    unsigned* ctr = p.counters + blockIdx.z * gridDim.x + tile;
    if (threadIdx.x == 0) ticket = atomicAdd(ctr, 1u);
    __syncthreads();
    if (ticket != (unsigned)ks_total - 1) return;
    __threadfence();
    const float* base = p.part + (size_t)mbase * ldp + (size_t)tile * TILE_N;
    for (int i = threadIdx.x; i < mcount * TILE_N; i += GEMV_THREADS) {
      const int m = i / TILE_N, c = i - m * TILE_N;
      float s = 0.0f;
      for (int j = 0; j < ks_total; ++j) s += __ldcg(base + ((size_t)j * p.M + m) * ldp + c);
      tl[m * TL_LD + c] = s;
    }
    if (threadIdx.x == 0) *ctr = 0u;
    __syncthreads();
  }
  pdl_trigger();
  run_epilogue<WT, AT>(p.epi, tl, TL_LD, mbase, mcount, n0, TILE_N, p.N);
}

template <typename WT, typename XT, typename AT, int MT>
cudaError_t launch_t(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
  constexpr int VEC = Vec16<WT>::N;
  const int tiles = linear_tiles(p);
  const int zch = (p.M + MT - 1) / MT;
  // Split K from the weight shape alone (never from M), so a row's arithmetic does not
  // depend on how many other rows share the launch: split until the tiles cover the GPU
  // twice (keeping >= 2 vector steps per lane) and at most KC_MAX columns per split.
  constexpr int KC_MAX = 512;
  const int step = 8 * VEC;
  int ks = 1;
  const int want = 2 * num_sms;
  while (tiles * ks < want && (p.K / (ks * 2)) >= 2 * step) ks *= 2;
  ks = std::max(ks, (p.K + KC_MAX - 1) / KC_MAX);
  int kc = (p.K + ks - 1) / ks;
  kc = ((kc + step - 1) / step) * step;
  ks = (p.K + kc - 1) / kc;
  auto smem_bytes = [&](int kcv) { return (size_t)(MT * (kcv + 4) + MT * TL_LD) * sizeof(float); };
  if (ks > 1) {
    const size_t need = (size_t)ks * p.M * tiles * TILE_N;
    if (need > p.part_elems || tiles * zch > p.counters_len) return cudaErrorInvalidValue;
  }
  const size_t smem = smem_bytes(kc);
  auto kern = k_gemv<WT, XT, AT, MT>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, ks, zch);
  cfg.blockDim = dim3(GEMV_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p, kc, ks);
}

template <typename WT, typename XT, typename AT>
cudaError_t launch_m(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
  if (p.M <= 1) return launch_t<WT, XT, AT, 1>(p, num_sms, s, pdl);
  if (p.M <= 2) return launch_t<WT, XT, AT, 2>(p, num_sms, s, pdl);
  if (p.M <= 4) return launch_t<WT, XT, AT, 4>(p, num_sms, s, pdl);
  if (p.M <= 8) return launch_t<WT, XT, AT, 8>(p, num_sms, s, pdl);
  if (p.M <= 16) return launch_t<WT, XT, AT, 16>(p, num_sms, s, pdl);
  return launch_t<WT, XT, AT, 32>(p, num_sms, s, pdl);
}

}  // namespace

cudaError_t launch_gemv(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
  if (p.M <= 0 || p.N <= 0 || p.K <= 0) return cudaSuccess;
  // weight dtype == activation dtype in this library: fp32 model -> fp32 activations,
  // bf16 model -> bf16 activations. X may also be fp32 for a bf16 model (tests).
  if (p.wdt == DT_F32) {
    if (p.xdt != DT_F32) return cudaErrorInvalidValue;
    return p.adt == DT_F32 ? launch_m<float, float, float>(p, num_sms, s, pdl)
                           : launch_m<float, float, bf16>(p, num_sms, s, pdl);
  }
  if (p.xdt == DT_BF16) {
    return p.adt == DT_BF16 ? launch_m<bf16, bf16, bf16>(p, num_sms, s, pdl)
                            : launch_m<bf16, bf16, float>(p, num_sms, s, pdl);
  }
  return p.adt == DT_BF16 ? launch_m<bf16, float, bf16>(p, num_sms, s, pdl)
                          : launch_m<bf16, float, float>(p, num_sms, s, pdl);
}

}  // namespace llm
