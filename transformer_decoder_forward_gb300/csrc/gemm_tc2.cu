// tcgen05 projection for many rows (prefill) on SM pairs: bf16 weights, activations as bf16
// (hi, lo) pairs, fp32 accumulation, the same fused epilogues as the one-SM kernel.
//
// The one-SM kernel (gemm_tc.cu) reads 12 KB of operands from shared memory for every
// 128 x 256 x 16 MMA and its TMA loads write as many, which bounds it by shared-memory
// bandwidth. Here the two CTAs of a cluster run one MMA across both SMs' tensor cores
// (tcgen05 cta_group::2): M = 256 weight rows (128 in each CTA's shared memory), N = 256 =
// the tile's 128 tokens as x_hi (staged in the even CTA) then x_lo (the odd CTA), K = 16. Each
// SM then stages and reads 8 KB per MMA of the same size, and each CTA's tensor memory holds
// the accumulator of its own 128 weight rows with the columns ordered as in the one-SM kernel
// (x_hi tokens, then x_lo tokens), so the epilogue is unchanged.
//
// Roles, in both CTAs unless stated:
//   - warp 0, one lane: TMA producer. Loads this CTA's 128 weight rows and its half of the
//     activation pair into a 4-stage ring; the copies complete on the even CTA's "full"
//     barrier (whose producer expects both CTAs' bytes).
//   - warp 1, one lane, even CTA only: issues the pair MMAs into one of two accumulators;
//     each stage's commit is multicast to both CTAs' "empty" barriers, each tile's last to both
//     "accumulator full" barriers.
//   - warps 2-17: read the accumulator of this CTA's rows, hand it back by arriving on the even
//     CTA's "accumulator empty" barrier (which counts both CTAs' epilogue warps), and apply the
//     epilogue. The element-wise kinds (stores, GELU, residual add, and the QKV epilogue without
//     RoPE or Q/K norm) apply it straight from registers: a thread holds one output column (its
//     TMEM lane) for 32 tokens, so for every token a warp stores 32 consecutive columns. The
//     other kinds (SwiGLU pairs gate and up rows of different warps, RoPE pairs dims d and d + 32)
//     stage the tile transposed in shared memory and run the shared epilogue; without the staging
//     tile the element-wise instance keeps a 6-stage ring instead of 4.
// Every wait is bounded (FLAG_WAIT_TIMEOUT); a cluster barrier precedes the release of the
// tensor memory, so no CTA leaves while the pair's MMAs may still read its shared memory.
#include <algorithm>

#include "epilogue.cuh"
#include "linear.cuh"
#include "tcgen05.cuh"

namespace llm {

namespace {

constexpr int P_BM = 128;    // tokens per tile
constexpr int P_BN = 128;    // weight rows per CTA (256 per pair)
constexpr int P_BK = 64;
constexpr int P_THREADS = 576;   // producer warp, MMA warp, 16 epilogue warps
constexpr int P_EPI_THREADS = 512;
constexpr int P_EPI_WARPS = P_EPI_THREADS / 32;
constexpr int P_W_STAGE = P_BN * P_BK * 2;   // bytes
constexpr int P_X_STAGE = P_BM * P_BK * 2;
constexpr int P_STAGE = P_W_STAGE + P_X_STAGE;   // [W rows][x_hi or x_lo rows]
constexpr int P_OT_LD = P_BN + 1;
constexpr int P_ACC = 2;
constexpr int P_ACC_COLS = 2 * P_BM;   // x_hi tokens, then x_lo tokens
constexpr uint32_t P_TMEM_COLS = P_ACC * P_ACC_COLS;

// Ring depth and the transposed staging tile of the two instances.
template <bool DIRECT>
struct PairCfg {
  static constexpr int STAGES = DIRECT ? 6 : 4;
  static constexpr size_t OT_BYTES = DIRECT ? 0 : (size_t)P_BM * P_OT_LD * 4;
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * P_STAGE + OT_BYTES + 256;
  static_assert(SMEM <= 220 * 1024, "shared memory of one CTA, with the epilogue's static staging");
};

// The epilogue kinds that need no staging tile (see the file comment).
inline bool epi_direct_ok(const Epilogue& e) {
  return e.kind == EPI_STORE_F32 || e.kind == EPI_STORE_ACT || e.kind == EPI_GELU || e.kind == EPI_RESID ||
         (e.kind == EPI_QKV && !e.rope && e.qn_g == nullptr);
}

// Element-wise epilogue from registers: this thread's output column n0 + col (its TMEM lane) for
// tokens m0 + c0 + j, j < 32, with acc[j] = x_hi.W + x_lo.W. Same arithmetic, in the same order,
// as the staged path (epi_apply): (x_hi.W + x_lo.W) + bias.
__device__ __forceinline__ void epi_direct(const Epilogue& e, const float* acc, int m0, int mrows, int c0, int col,
                                           int n0, int N) {
  const int n = n0 + col;
  if (n >= N) return;
  const EpiStaging& st = epi_staging();
  const float b = st.bias[col];
  const int jn = min(32, mrows - c0);   // tokens of this thread's quarter inside the tile
  switch (e.kind) {
    case EPI_STORE_F32:
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < jn) reinterpret_cast<float*>(e.out)[(size_t)(m0 + c0 + j) * e.ld_out + n] = acc[j] + b;
      break;
    case EPI_STORE_ACT:
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < jn) act_store<Split>(e.out, m0 + c0 + j, e.ld_out, n, acc[j] + b);
      break;
    case EPI_GELU:
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < jn) act_store<Split>(e.out, m0 + c0 + j, e.ld_out, n, gelu_tanh_clamped(acc[j] + b));
      break;
    case EPI_RESID: {
#pragma unroll
      for (int h = 0; h < 32; h += 16) {   // 16 loads in flight, then their stores
        float hv[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) hv[j] = h + j < jn ? e.resid[(size_t)(m0 + c0 + h + j) * e.ld_resid + n] : 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (h + j < jn) e.resid[(size_t)(m0 + c0 + h + j) * e.ld_resid + n] = hv[j] + acc[h + j] + b;
      }
      break;
    }
    case EPI_QKV: {   // no RoPE, no Q/K norm: q to q_out, k and v to the row's KV slot
      const int H = e.n_heads, Hkv = e.kv.n_kv_heads;
      const int hh = n / HD, d = n - hh * HD;
      if (hh < H) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < jn) e.q_out[(size_t)(m0 + c0 + j) * H * HD + n] = acc[j] + b;
        break;
      }
      const bool is_k = hh < H + Hkv;
      const int g = is_k ? hh - H : hh - H - Hkv;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j >= jn) break;
        const int m = c0 + j;
        const int pb = st.blk[m];
        if (pb < 0) continue;
        const size_t off = kv_offset(e.kv, pb, g, st.pos[m] & (KVB - 1)) + d;
        const float y = acc[j] + b;
        if (e.kv.dtype == DT_BF16) reinterpret_cast<bf16*>(is_k ? e.kv.k : e.kv.v)[off] = __float2bfloat16_rn(y);
        else reinterpret_cast<float*>(is_k ? e.kv.k : e.kv.v)[off] = y;
      }
      break;
    }
    default:
      break;
  }
}

__device__ __forceinline__ void epi_bar2() { asm volatile("bar.sync 1, %0;" ::"r"(P_EPI_THREADS) : "memory"); }
__device__ __forceinline__ bool epi_bar2_all(bool v) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.s32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((int)v), "r"(P_EPI_THREADS)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

template <bool DIRECT>
__global__ void __launch_bounds__(P_THREADS, 1)
    k_gemm_tc2(const LinearParams p, const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXlo,
               const __grid_constant__ CUtensorMap tmW, int tiles_m, int tiles_n2) {
  constexpr int P_STAGES = PairCfg<DIRECT>::STAGES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto sW = [&](int s) { return base + (size_t)s * P_STAGE; };
  auto sX = [&](int s) { return base + (size_t)s * P_STAGE + P_W_STAGE; };
  float* ot = reinterpret_cast<float*>(base + (size_t)P_STAGES * P_STAGE);   // staged instance only
  uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)P_STAGES * P_STAGE + PairCfg<DIRECT>::OT_BYTES);
  uint64_t* empty = full + P_STAGES;
  uint64_t* acc_full = empty + P_STAGES;
  uint64_t* acc_empty = acc_full + P_ACC;
  uint64_t* drain = acc_empty + P_ACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int kiters = (p.K + P_BK - 1) / P_BK;
  const int ntiles = tiles_m * tiles_n2;
  const int F = p.N;
  unsigned* flags = p.epi.flags;

  if (warp == 0) {
    tmem_alloc_pair(tmem_slot, P_TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < P_ACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 2 * P_EPI_WARPS);   // lane 0 of every epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  cluster_arrive();   // both CTAs' barriers are initialised and the tensor memory allocated
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t full0 = cluster_addr(full, 0);             // the even CTA's "full" barriers
  const uint32_t acc_empty0 = cluster_addr(acc_empty, 0);   // and its "accumulator empty" barriers

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer (both CTAs): this CTA's weight rows and its half of the pair
      pdl_wait();
      const CUtensorMap* xmap = rank == 0 ? &tmX : &tmXlo;
      int it = 0;
      bool ok = true;
      for (int t = pair; t < ntiles && ok; t += npairs) {
        const int tile_m = t / tiles_n2, tile_n = (t - tile_m * tiles_n2) * 2 + (int)rank;
        const int m0 = tile_m * P_BM;
        for (int i = 0; i < kiters; ++i, ++it) {
          const int s = it % P_STAGES;
          if (it >= P_STAGES && !mbar_wait(&empty[s], ((it / P_STAGES) - 1) & 1, flags)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * P_STAGE);
          const uint32_t fb = full0 + (uint32_t)(s * 8);
          const int kc = i * P_BK;
          tma_load_2d_pair(sX(s), xmap, kc, m0, fb);
          unsigned char* w = sW(s);
          if (p.swiglu) {
            // two 64-row sub-tiles, each 32 gate rows then the 32 matching up rows
            for (int sub = 0; sub < 2; ++sub) {
              const int j0 = (tile_n * 2 + sub) * 32;
              tma_load_2d_pair(w + (sub * 64) * 128, &tmW, kc, j0, fb);
              tma_load_2d_pair(w + (sub * 64 + 32) * 128, &tmW, kc, F + j0, fb);
            }
          } else {
            tma_load_2d_pair(w, &tmW, kc, tile_n * P_BN, fb);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---- MMA issuer (even CTA): A = both CTAs' weight rows, B = [x_hi; x_lo]
      constexpr uint32_t idesc = idesc_bf16(2 * P_BN, 2 * P_BM);
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = pair; t < ntiles && ok; t += npairs, ++lt) {
        const int a = lt % P_ACC;
        if (lt >= P_ACC && !mbar_wait(&acc_empty[a], ((lt / P_ACC) - 1) & 1, flags)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(a * P_ACC_COLS);
        for (int i = 0; i < kiters; ++i, ++it) {
          const int s = it % P_STAGES;
          if (!mbar_wait(&full[s], (it / P_STAGES) & 1, flags)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dw = sw128_desc(sW(s));
          const uint64_t dx = sw128_desc(sX(s));
#pragma unroll
          for (int kk = 0; kk < P_BK / 16; ++kk) {   // 16 bf16 = 32 bytes per MMA step
            const uint64_t o = (uint64_t)(kk * 2);
            tc_mma_pair(d, dw + o, dx + o, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit_pair_mc(&empty[s], 0x3);
        }
        if (ok) tc_commit_pair_mc(&acc_full[a], 0x3);
      }
      // every MMA issued so far has completed before the pair's tensor memory is freed
      tc_commit_pair_mc(drain, 0x1);
      mbar_wait(drain, 0, flags);
      pdl_trigger();
    }
    __syncwarp();
  } else {
    // ---- epilogue warps: four per TMEM lane quadrant, each reading a quarter of the tokens
    const int et = threadIdx.x - 64;
    const int q = warp & 3;
    const int quarter = (warp - 2) >> 2;
    const int wrow = q * 32 + lane;
    pdl_wait();
    int lt = 0;
    for (int t = pair; t < ntiles; t += npairs, ++lt) {
      const int tile_m = t / tiles_n2, tile_n = (t - tile_m * tiles_n2) * 2 + (int)rank;
      const int m0 = tile_m * P_BM;
      const int mrows = min(P_BM, p.M - m0);
      const int n0 = p.swiglu ? tile_n * 64 : tile_n * P_BN;
      const int a = lt % P_ACC;
      epi_stage<bf16>(p.epi, m0, mrows, n0, P_BN, p.N, et, P_EPI_THREADS);
      const bool ok = mbar_wait(&acc_full[a], (lt / P_ACC) & 1, flags);
      if (!epi_bar2_all(ok)) break;   // the epilogue warps leave together
      tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * P_ACC_COLS);
      const int c0 = quarter * 32;
      float acc[32];
      {
        uint32_t rh[32], rl[32];
        tmem_ld32(ta + (uint32_t)c0, rh);             // x_hi . W
        tmem_ld32(ta + (uint32_t)(P_BM + c0), rl);    // x_lo . W
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = __uint_as_float(rh[j]) + __uint_as_float(rl[j]);
      }
      if constexpr (!DIRECT) {
#pragma unroll
        for (int j = 0; j < 32; ++j) ot[(c0 + j) * P_OT_LD + wrow] = acc[j];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + (uint32_t)(a * 8));   // the MMA may refill it
      if constexpr (DIRECT) {
        epi_direct(p.epi, acc, m0, mrows, c0, wrow, n0, p.N);
      } else {
        epi_bar2();
        epi_apply<bf16>(p.epi, ot, P_OT_LD, m0, mrows, n0, P_BN, p.N, et, P_EPI_THREADS);
      }
      epi_bar2();   // the staging arrays (and tile) are free for the next tile
    }
  }
  tc_fence_before();
  cluster_arrive();   // both CTAs are done with the pair's MMAs and tensor memory
  cluster_wait();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, P_TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_gemm_tc2(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
  if (p.M <= 0 || p.N <= 0 || p.K <= 0) return cudaSuccess;
  if (!gemm_tc_supported(p)) return cudaErrorNotSupported;
  CUtensorMap mx, mxl, mw;
  const int wrows = p.swiglu ? 2 * p.N : p.N;
  const bf16* xlo = reinterpret_cast<const bf16*>(p.X) + p.ldx / 2;
  if (!make_map(&mx, p.X, DT_BF16, p.M, p.K, p.ldx, P_BM)) return cudaErrorInvalidValue;
  if (!make_map(&mxl, xlo, DT_BF16, p.M, p.K, p.ldx, P_BM)) return cudaErrorInvalidValue;
  if (!make_map(&mw, p.W, DT_BF16, wrows, p.K, p.K, p.swiglu ? 32 : P_BN)) return cudaErrorInvalidValue;
  const int tiles_n = p.swiglu ? (p.N + 63) / 64 : (p.N + P_BN - 1) / P_BN;   // 128-weight-row tiles
  const int tiles_n2 = (tiles_n + 1) / 2;                                       // pair tiles
  const int tiles_m = (p.M + P_BM - 1) / P_BM;
  const int pairs = std::min(tiles_m * tiles_n2, num_sms / 2);
  if (pairs < 1) return cudaErrorInvalidValue;
  const bool direct = epi_direct_ok(p.epi);
  auto kern = direct ? k_gemm_tc2<true> : k_gemm_tc2<false>;
  const size_t smem = direct ? PairCfg<true>::SMEM : PairCfg<false>::SMEM;
  static bool attr_set_dev[MAX_DEVICES][2] = {};
  bool& attr_set = attr_set_dev[current_device()][direct ? 1 : 0];
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(P_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p, mx, mxl, mw, tiles_m, tiles_n2);
}

}  // namespace llm
