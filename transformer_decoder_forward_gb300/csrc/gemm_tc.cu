// tcgen05 / TMEM tensor-core projection for many rows (prefill): bf16 weights,
// activations as bf16 (hi, lo) pairs, fp32 accumulation, fused epilogues.
//
// Prefill is arithmetic bound ("rvllm-metal", section "The matmul pain story":
// lots of rows, a tiled kernel staging slices of x and W). On sm_103a the tile
// is a 5th-generation tensor-core contraction, run by a persistent kernel with
// one CTA per SM that walks the output tiles (128 rows x 128 weight rows) in
// turn, its warps specialised:
//   - warp 0, one lane: TMA producer. 128-byte-swizzled 128 x 64 slices of x_hi,
//     x_lo and W go into a 3-stage shared-memory ring, each stage guarded by a
//     "full" and an "empty" mbarrier; it runs ahead across tile boundaries.
//   - warp 1, one lane: issues tcgen05.mma with the weights on the M side and the
//     tokens on N: M = 128 weight rows, N = 256 = the tile's 128 rows of x_hi then
//     its 128 rows of x_lo (adjacent in the stage, so one B operand), K = 16, bf16
//     in, fp32 accumulate, into one of two 128 x 256 accumulators in tensor memory.
//     One MMA carries both halves of the activation pair, each operand byte is read
//     from shared memory once per MMA, and the stage costs 24 KB of shared-memory
//     traffic per 16 K rather than 28 KB with two 128 x 128 products: the kernel is
//     bound by shared-memory bandwidth. tcgen05.commit releases each stage once the
//     MMAs that read it finish, and marks the accumulator full after the tile's last.
//   - warps 2-17: read a full accumulator with tcgen05.ld (warp w owns TMEM lanes
//     32(w%4).. = weight rows, a quarter of the tokens), add the x_hi and x_lo
//     columns, hand the accumulator back to the MMA warp, stage the tile transposed
//     (tokens x weight rows, fp32) in shared memory and run the shared epilogue
//     (bias, GELU / SwiGLU, RoPE + kv_write, residual add) while the MMA warp
//     already fills the other accumulator with the next tile.
// Every wait is bounded (FLAG_WAIT_TIMEOUT) and the tensor memory is always freed.
#include <algorithm>

#include "epilogue.cuh"
#include "linear.cuh"
#include "tcgen05.cuh"

namespace llm {

namespace {

constexpr int TC_BM = 128, TC_BN = 128, TC_BK = 64, TC_STAGES = 3;
constexpr int TC_THREADS = 576;                 // producer warp, MMA warp, 16 epilogue warps
constexpr int TC_EPI_THREADS = 512;
constexpr int TC_EPI_WARPS = TC_EPI_THREADS / 32;
constexpr int A_STAGE = TC_BM * TC_BK * 2;      // bytes
constexpr int B_STAGE = TC_BN * TC_BK * 2;
constexpr int STAGE = 2 * A_STAGE + B_STAGE;    // [x_hi][x_lo][W]
constexpr int OT_LD = TC_BN + 1;                // epilogue tile row stride (floats): conflict-free row writes
constexpr size_t OT_BYTES = (size_t)TC_BM * OT_LD * 4;
constexpr int TC_ACC = 2;                       // accumulators in TMEM
constexpr int TC_ACC_COLS = 2 * TC_BM;          // x_hi tokens, then x_lo tokens
constexpr uint32_t TC_TMEM_COLS = TC_ACC * TC_ACC_COLS;   // all 512 columns
constexpr size_t TC_SMEM = 1024 + (size_t)TC_STAGES * STAGE + OT_BYTES + 256;

// Barrier among the epilogue warps only (named barrier 1), plain or with an AND of a
// predicate so that all of them take the same branch after it.
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"r"(TC_EPI_THREADS) : "memory"); }
__device__ __forceinline__ bool epi_bar_all(bool v) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.s32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((int)v), "r"(TC_EPI_THREADS)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    k_gemm_tc(const LinearParams p, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAlo,
              const __grid_constant__ CUtensorMap tmB, int tiles_m, int tiles_n) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto sA = [&](int s) { return base + (size_t)s * STAGE; };
  auto sAlo = [&](int s) { return base + (size_t)s * STAGE + A_STAGE; };
  auto sB = [&](int s) { return base + (size_t)s * STAGE + 2 * A_STAGE; };
  float* ot = reinterpret_cast<float*>(base + (size_t)TC_STAGES * STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)TC_STAGES * STAGE + OT_BYTES);
  uint64_t* empty = full + TC_STAGES;
  uint64_t* acc_full = empty + TC_STAGES;
  uint64_t* acc_empty = acc_full + TC_ACC;
  uint64_t* drain = acc_empty + TC_ACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kiters = (p.K + TC_BK - 1) / TC_BK;
  const int ntiles = tiles_m * tiles_n;
  const int F = p.N;
  unsigned* flags = p.epi.flags;

  if (warp == 0) {
    tmem_alloc(tmem_slot, TC_TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < TC_ACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], TC_EPI_WARPS);   // lane 0 of each epilogue warp
    }
    mbar_init(drain, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer: the stage ring runs across tiles
      pdl_wait();
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int tile_m = t / tiles_n, tile_n = t - tile_m * tiles_n;
        const int m0 = tile_m * TC_BM;
        for (int i = 0; i < kiters; ++i, ++it) {
          const int s = it % TC_STAGES;
          if (it >= TC_STAGES && !mbar_wait(&empty[s], ((it / TC_STAGES) - 1) & 1, flags)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], STAGE);
          const int kc = i * TC_BK;
          tma_load_2d(sA(s), &tmA, kc, m0, &full[s]);
          tma_load_2d(sAlo(s), &tmAlo, kc, m0, &full[s]);
          unsigned char* b = sB(s);
          if (p.swiglu) {
            // two 64-row sub-tiles, each 32 gate rows then the 32 matching up rows
            for (int sub = 0; sub < 2; ++sub) {
              const int j0 = (tile_n * 2 + sub) * 32;
              tma_load_2d(b + (sub * 64) * 128, &tmB, kc, j0, &full[s]);
              tma_load_2d(b + (sub * 64 + 32) * 128, &tmB, kc, F + j0, &full[s]);
            }
          } else {
            tma_load_2d(b, &tmB, kc, tile_n * TC_BN, &full[s]);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: accumulator (local tile count) % 2; A = W tile, B = [x_hi; x_lo]
      static_assert(TC_BN == 128 && 2 * TC_BM == 256, "M = 128 weight rows, N = 2 x 128 tokens");
      constexpr uint32_t idesc = idesc_bf16(TC_BN, 2 * TC_BM);
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++lt) {
        const int a = lt % TC_ACC;
        if (lt >= TC_ACC && !mbar_wait(&acc_empty[a], ((lt / TC_ACC) - 1) & 1, flags)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(a * TC_ACC_COLS);
        for (int i = 0; i < kiters; ++i, ++it) {
          const int s = it % TC_STAGES;
          if (!mbar_wait(&full[s], (it / TC_STAGES) & 1, flags)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dw = sw128_desc(sB(s));   // 128 weight rows
          const uint64_t dx = sw128_desc(sA(s));   // 256 rows: x_hi, then x_lo at +A_STAGE
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {   // 16 bf16 = 32 bytes per MMA step
            const uint64_t o = (uint64_t)(kk * 2);
            tc_mma(d, dw + o, dx + o, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&empty[s]);
        }
        if (ok) tc_commit(&acc_full[a]);
      }
      // every MMA issued so far has completed before the tensor memory is freed
      tc_commit(drain);
      mbar_wait(drain, 0, flags);
      pdl_trigger();
    }
    __syncwarp();
  } else {
    // ---- epilogue warps: four per TMEM lane quadrant, each reading a quarter of the tokens
    const int et = threadIdx.x - 64;   // 0..511
    const int q = warp & 3;            // TMEM lane quadrant = weight rows 32q..32q+31
    const int quarter = (warp - 2) >> 2;   // tokens 32 quarter .. 32 quarter + 31
    const int wrow = q * 32 + lane;
    pdl_wait();
    int lt = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
      const int tile_m = t / tiles_n, tile_n = t - tile_m * tiles_n;
      const int m0 = tile_m * TC_BM;
      const int mrows = min(TC_BM, p.M - m0);
      const int n0 = p.swiglu ? tile_n * 64 : tile_n * TC_BN;
      const int a = lt % TC_ACC;
      epi_stage<bf16>(p.epi, m0, mrows, n0, TC_BN, p.N, et, TC_EPI_THREADS);
      const bool ok = mbar_wait(&acc_full[a], (lt / TC_ACC) & 1, flags);
      if (!epi_bar_all(ok)) break;   // the epilogue warps leave together
      tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * TC_ACC_COLS);
      {
        const int c0 = quarter * 32;
        uint32_t rh[32], rl[32];
        tmem_ld32(ta + (uint32_t)c0, rh);             // x_hi . W
        tmem_ld32(ta + (uint32_t)(TC_BM + c0), rl);   // x_lo . W
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) ot[(c0 + j) * OT_LD + wrow] = __uint_as_float(rh[j]) + __uint_as_float(rl[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);   // the MMA warp may refill this accumulator
      epi_bar();                                   // tile and staging complete
      epi_apply<bf16>(p.epi, ot, OT_LD, m0, mrows, n0, TC_BN, p.N, et, TC_EPI_THREADS);
      epi_bar();                                   // tile and staging free for the next tile
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TC_TMEM_COLS);
  }
}

}  // namespace

bool gemm_tc_supported(const LinearParams& p) {
  if (p.wdt != DT_BF16 || p.xdt != DT_SPLIT || p.adt != DT_SPLIT) return false;
  if (p.K % 8 != 0 || p.ldx % 16 != 0 || p.ldx < 2 * p.K) return false;
  if ((reinterpret_cast<uintptr_t>(p.W) | reinterpret_cast<uintptr_t>(p.X)) & 15) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_gemm_tc(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
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
  static bool attr_set_dev[MAX_DEVICES] = {};
  bool& attr_set = attr_set_dev[current_device()];
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(std::min(tiles_m * tiles_n, num_sms));
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = TC_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_gemm_tc, p, ma, mal, mb, tiles_m, tiles_n);
}

}  // namespace llm
