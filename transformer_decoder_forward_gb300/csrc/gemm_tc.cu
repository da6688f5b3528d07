// tcgen05 / TMEM tensor-core projection for many rows (prefill): bf16 weights,
// activations as bf16 (hi, lo) pairs, fp32 accumulation, fused epilogues.
//
// Prefill is arithmetic bound ("rvllm-metal", section "The matmul pain story":
// lots of rows, a tiled kernel staging slices of x and W). On sm_103a the tile
// is a 5th-generation tensor-core contraction:
//   - TMA (cp.async.bulk.tensor, 128-byte swizzle) stages 128 x 64 slices of
//     x_hi and x_lo (rows) and 128 x 64 slices of W into a 4-stage shared-memory
//     ring, each stage guarded by a "full" and an "empty" mbarrier;
//   - one elected thread issues tcgen05.mma (M = 128, N = 128, K = 16, bf16 in,
//     fp32 accumulate) for x_hi.W and x_lo.W into one 128 x 128 fp32 accumulator
//     in tensor memory, so the product carries the activations' full pair
//     accuracy; tcgen05.commit releases each stage once the MMAs that read it finish;
//   - after the last commit, four warps read the accumulator back with
//     tcgen05.ld (warp w owns TMEM lanes 32w..32w+31 = tile rows), stage it as
//     an fp32 tile in shared memory and run the shared epilogue per 64-column
//     sub-tile (bias, GELU / SwiGLU, RoPE + kv_write, residual add).
// Every wait is bounded (FLAG_WAIT_TIMEOUT) and the tensor memory is always freed.
#include "epilogue.cuh"
#include "linear.cuh"
#include "tcgen05.cuh"

namespace llm {

namespace {

constexpr int TC_BM = 128, TC_BN = 128, TC_BK = 64, TC_STAGES = 4;
constexpr int TC_THREADS = 128;
constexpr int A_STAGE = TC_BM * TC_BK * 2;   // bytes
constexpr int B_STAGE = TC_BN * TC_BK * 2;
constexpr int OT_LD = TC_BN + 1;
constexpr int STAGE = 2 * A_STAGE + B_STAGE;   // [x_hi][x_lo][W]
constexpr size_t TC_SMEM = 1024 + (size_t)TC_STAGES * STAGE + 256;

__global__ void __launch_bounds__(TC_THREADS, 1)
    k_gemm_tc(const LinearParams p, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAlo,
              const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto sA = [&](int s) { return base + (size_t)s * STAGE; };
  auto sAlo = [&](int s) { return base + (size_t)s * STAGE + A_STAGE; };
  auto sB = [&](int s) { return base + (size_t)s * STAGE + 2 * A_STAGE; };
  uint64_t* full = reinterpret_cast<uint64_t*>(base + TC_STAGES * STAGE);
  uint64_t* empty = full + TC_STAGES;
  uint64_t* done = empty + TC_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, tile_m = blockIdx.y;
  const int m0 = tile_m * TC_BM;
  const int kiters = (p.K + TC_BK - 1) / TC_BK;
  const int F = p.N;

  if (warp == 0) {
    tmem_alloc(tmem_slot, TC_BN);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  bool ok = true;
  if (warp == 0 && lane == 0) {
    // ---- TMA producer
    for (int i = 0; i < kiters; ++i) {
      const int s = i % TC_STAGES;
      if (i >= TC_STAGES && !mbar_wait(&empty[s], ((i / TC_STAGES) - 1) & 1, p.epi.flags)) break;
      mbar_arrive_expect_tx(&full[s], STAGE);
      const int kc = i * TC_BK;
      tma_load_2d(sA(s), &tmA, kc, m0, &full[s]);
      tma_load_2d(sAlo(s), &tmAlo, kc, m0, &full[s]);
      unsigned char* b = sB(s);
      if (p.swiglu) {
        // two 64-column sub-tiles, each 32 gate rows then the 32 matching up rows
        for (int sub = 0; sub < 2; ++sub) {
          const int j0 = (tile_n * 2 + sub) * 32;
          tma_load_2d(b + (sub * 64) * 128, &tmB, kc, j0, &full[s]);
          tma_load_2d(b + (sub * 64 + 32) * 128, &tmB, kc, F + j0, &full[s]);
        }
      } else {
        tma_load_2d(b, &tmB, kc, tile_n * TC_BN, &full[s]);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    constexpr uint32_t idesc = idesc_bf16(TC_BM, TC_BN);
    for (int i = 0; i < kiters; ++i) {
      const int s = i % TC_STAGES;
      if (!mbar_wait(&full[s], (i / TC_STAGES) & 1, p.epi.flags)) break;
      tc_fence_after();
      const uint64_t da = sw128_desc(sA(s)), dal = sw128_desc(sAlo(s));
      const uint64_t db = sw128_desc(sB(s));
#pragma unroll
      for (int kk = 0; kk < TC_BK / 16; ++kk) {   // 16 bf16 = 32 bytes per MMA step
        const uint64_t o = (uint64_t)(kk * 2);
        tc_mma(tmem, da + o, db + o, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        tc_mma(tmem, dal + o, db + o, idesc, 1u);
      }
      tc_commit(&empty[s]);
    }
    tc_commit(done);
  }
  // ---- epilogue: all four warps
  ok = mbar_wait(done, 0, p.epi.flags);
  if (!ok) ok = mbar_wait(done, 0, p.epi.flags);   // one more bounded wait for the MMAs in flight
  tc_fence_after();
  float* ot = reinterpret_cast<float*>(base);   // [128][OT_LD] over the drained pipeline buffers
  const int row = warp * 32 + lane;
  __syncwarp();   // lanes 0 of warps 0/1 come from the producer / MMA loops: reconverge for tcgen05.ld
  if (ok) {
#pragma unroll 1
    for (int c0 = 0; c0 < TC_BN; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) ot[row * OT_LD + c0 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TC_BN);
  }
  pdl_trigger();
  if (!ok) return;
  const int mrows = min(TC_BM, p.M - m0);
  run_epilogue<bf16>(p.epi, ot, OT_LD, m0, mrows, p.swiglu ? tile_n * 64 : tile_n * TC_BN, TC_BN, p.N);
}

}  // namespace

bool gemm_tc_supported(const LinearParams& p) {
  if (p.wdt != DT_BF16 || p.xdt != DT_SPLIT || p.adt != DT_SPLIT) return false;
  if (p.K % 8 != 0 || p.ldx % 16 != 0 || p.ldx < 2 * p.K) return false;
  if ((reinterpret_cast<uintptr_t>(p.W) | reinterpret_cast<uintptr_t>(p.X)) & 15) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_gemm_tc(const LinearParams& p, int /*num_sms*/, cudaStream_t s, bool pdl) {
  if (p.M <= 0 || p.N <= 0 || p.K <= 0) return cudaSuccess;
  if (!gemm_tc_supported(p)) return cudaErrorNotSupported;
  CUtensorMap ma, mal, mb;
  const int wrows = p.swiglu ? 2 * p.N : p.N;
  const bf16* xlo = reinterpret_cast<const bf16*>(p.X) + p.ldx / 2;
  if (!make_map(&ma, p.X, DT_BF16, p.M, p.K, p.ldx, TC_BM)) return cudaErrorInvalidValue;
  if (!make_map(&mal, xlo, DT_BF16, p.M, p.K, p.ldx, TC_BM)) return cudaErrorInvalidValue;
  if (!make_map(&mb, p.W, DT_BF16, wrows, p.K, p.K, p.swiglu ? 32 : TC_BN)) return cudaErrorInvalidValue;
  const int tiles_n = p.swiglu ? (p.N + 63) / 64 : (p.N + TC_BN - 1) / TC_BN;
  const int tiles_m = (p.M + TC_BM - 1) / TC_BM;
  auto kern = k_gemm_tc;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles_n, tiles_m);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = TC_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p, ma, mal, mb);
}

}  // namespace llm
