// Projection kernels y = x . W^T with fused epilogues (declarations + parameters).
#pragma once
#include "common.cuh"

namespace llm {

// Tile columns per output tile: 64 = one head (keeps RoPE pairs and SwiGLU gate/up in one tile).
constexpr int TILE_N = 64;

struct LinearParams {
  const void* W;        // [rows][K] weight, dtype wdt (DT_Q8: the int8 quants)
  const void* Wscale;   // DT_Q8: [rows][K / 32] fp16 block scales; otherwise unused
  const void* X;        // [M][ldx] activations, dtype xdt
  int M, N, K, ldx;     // N: output columns of the epilogue (d_ff for SWIGLU)
  int wdt, xdt, adt;    // weight / input / activation-output dtypes
  int swiglu;           // 1: tile t reads gate rows t*32.. and up rows F + t*32..
  Epilogue epi;
  // Fused row norm (xnorm = 1): X is the fp32 residual stream h ([M][ldx], ldx = K) and the
  // kernel uses row m as Norm(h[m]) = (h[m] - mean) * rstd * g + b (LayerNorm), or
  // h[m] * rstd * g (RMSNorm), the statistics from warp_row_stats. Supported by the GEMV; the
  // others take the norm kernel's output instead.
  int xnorm;
  const void* norm_g;   // [K] gains, weight dtype
  const void* norm_b;   // [K] biases (LayerNorm) or nullptr
  float norm_eps;
  int norm_ln;          // 1: LayerNorm, 0: RMSNorm
};

inline int linear_tiles(const LinearParams& p) {
  return p.swiglu ? (p.N + 31) / 32 : (p.N + TILE_N - 1) / TILE_N;
}

// Variants. AUTO picks by M; the others force one kernel (tests sweep all of them).
//   LIN_GEMV     CUDA-core weight-stream GEMV (decode)
//   LIN_SIMT     CUDA-core tiled GEMM
//   LIN_TC       tcgen05 GEMM, activations on the MMA's M side (prefill, bf16)
//   LIN_TC_SWAP  tcgen05 GEMM, weights on the MMA's M side (decode, M <= 256; bf16, or fp32 as 3 x tf32)
//   LIN_TC_PAIR  tcgen05 GEMM on SM pairs (cta_group::2), 256 weight rows a tile (prefill, bf16)
enum : int { LIN_AUTO = 0, LIN_GEMV = 1, LIN_SIMT = 2, LIN_TC = 3, LIN_TC_SWAP = 4, LIN_TC_PAIR = 5 };

// Each returns cudaSuccess or the launch error; `name` receives the kernel family name.
cudaError_t launch_gemv(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl);
bool gemv_norm_supported(const LinearParams& p);
cudaError_t launch_gemm_simt(const LinearParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_gemm_tc(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl);
cudaError_t launch_gemm_tc2(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl);   // same support test
bool gemm_tc_supported(const LinearParams& p);
cudaError_t launch_gemm_tc_swap(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl);
bool gemm_tc_swap_supported(const LinearParams& p);

}  // namespace llm
