// Tiled projection on CUDA cores for many rows (prefill, fp32 models).
//
// The pages' linear_gemm: each threadgroup computes an output tile from slices
// of x and W staged in threadgroup memory ("rvllm-metal", section "The matmul
// pain story"). Here a 128 x 64 tile (64 = one head, so the shared epilogues
// see whole heads), K in steps of 16, 256 threads each holding an 8 x 4 block.
// This is the fp32 path, the Q8_0 path (quants dequantised as they are staged) and the
// reference path for bf16 weights (whose activations arrive as bf16 pairs); bf16 prefill uses
// the tcgen05 kernel.
#include <cuda_fp16.h>

#include <type_traits>

#include "epilogue.cuh"
#include "linear.cuh"

namespace llm {

namespace {

constexpr int BM = 128, BN = 64, BK = 16;
constexpr int SIMT_THREADS = 256;
constexpr int AS_LD = BM + 4, BS_LD = BN + 4, OT_LD = BN + 1;

template <typename WT>
__global__ void __launch_bounds__(SIMT_THREADS) k_gemm_simt(const LinearParams p) {
  using AT = typename ActOf<WT>::type;   // activation storage: fp32 or a bf16 pair
  using ST = typename Elem<WT>::type;     // stored weight element (int8 quants for Q8_0)
  constexpr bool IS_Q8 = std::is_same<WT, Q8>::value;
  __shared__ __align__(16) float smem[BM * OT_LD];   // reused: As/Bs during the loop, output tile after
  float* As = smem;                  // [BK][AS_LD]  (k-major, m contiguous)
  float* Bs = smem + BK * AS_LD;     // [BK][BS_LD]
  const int tid = threadIdx.x;
  const int tile = blockIdx.x, m0 = blockIdx.y * BM;
  const int F = p.N;
  const ST* W = reinterpret_cast<const ST*>(p.W);
  pdl_wait();

  // loader coordinates
  const int a_row = tid >> 1, a_k = (tid & 1) * 8;     // 128 rows x 16 k: 8 per thread
  const int b_col = tid >> 2, b_k = (tid & 3) * 4;     // 64 rows  x 16 k: 4 per thread
  int b_wrow;
  bool b_valid;
  if (p.swiglu) {
    b_valid = tile * 32 + (b_col & 31) < F;
    b_wrow = swiglu_row(tile * 32, b_col, F);
  } else {
    b_wrow = tile * BN + b_col;
    b_valid = b_wrow < p.N;
  }
  const bool a_valid = m0 + a_row < p.M;
  const ST* wb = W + (size_t)b_wrow * p.K;
  // Q8_0: this row's block scales (the value of quant k is scale[k / 32] * q[k])
  const __half* sb = IS_Q8 ? reinterpret_cast<const __half*>(p.Wscale) + (size_t)b_wrow * (p.K / Q8_BLOCK) : nullptr;

  const int ty = tid >> 4, tx = tid & 15;   // rows ty*8.., cols tx*4..
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int k0 = 0; k0 < p.K; k0 += BK) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = k0 + a_k + j;
      As[(a_k + j) * AS_LD + a_row] = (a_valid && k < p.K) ? act_load<AT>(p.X, m0 + a_row, p.ldx, k) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = k0 + b_k + j;
      float wv = 0.0f;
      if (b_valid && k < p.K) {
        if constexpr (IS_Q8) wv = (float)wb[k] * __half2float(sb[k / Q8_BLOCK]);
        else wv = to_f32(wb[k]);
      }
      Bs[(b_k + j) * BS_LD + b_col] = wv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(As + kk * AS_LD + ty * 8);
      const float4 a1 = *reinterpret_cast<const float4*>(As + kk * AS_LD + ty * 8 + 4);
      const float4 b = *reinterpret_cast<const float4*>(Bs + kk * BS_LD + tx * 4);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* ot = smem;   // [BM][OT_LD]
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) ot[(ty * 8 + i) * OT_LD + tx * 4 + j] = acc[i][j];
  __syncthreads();
  pdl_trigger();
  const int n0 = p.swiglu ? tile * 32 : tile * BN;
  run_epilogue<WT>(p.epi, ot, OT_LD, m0, min(BM, p.M - m0), n0, BN, p.N);
}

template <typename WT>
cudaError_t launch_t(const LinearParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(linear_tiles(p), (p.M + BM - 1) / BM);
  cfg.blockDim = dim3(SIMT_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_gemm_simt<WT>, p);
}

}  // namespace

cudaError_t launch_gemm_simt(const LinearParams& p, cudaStream_t s, bool pdl) {
  if (p.M <= 0 || p.N <= 0 || p.K <= 0) return cudaSuccess;
  if (p.wdt == DT_F32 && p.xdt == DT_F32 && p.adt == DT_F32) return launch_t<float>(p, s, pdl);
  if (p.wdt == DT_BF16 && p.xdt == DT_SPLIT && p.adt == DT_SPLIT) return launch_t<bf16>(p, s, pdl);
  if (p.wdt == DT_Q8 && p.xdt == DT_F32 && p.adt == DT_F32) {
    if (p.K % Q8_BLOCK != 0 || !p.Wscale) return cudaErrorInvalidValue;
    return launch_t<Q8>(p, s, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace llm
