// Decode projection on tensor cores, weights on the MMA's M side ("swap-AB").
//
// A decode step multiplies a few rows of activations by every weight matrix, so it
// streams all weights once per step and is memory bound ("rvllm-metal", section
// "The matmul pain story"). The pages' answer is a simdgroup GEMV for 1-4 rows and
// a K-split small-tile kernel for 5-16 rows. On sm_103a this kernel puts 128 weight
// rows on the tcgen05 M side and the step's tokens on the N side (N = rows rounded
// up to 16, at most 256):
//   - warp 0, one lane: TMA producer. Before waiting on the previous kernel
//     (programmatic dependent launch) it already issues the weight tiles of the
//     first stages: weights never depend on earlier kernels.
//   - warp 1, one lane: issues tcgen05.mma into a 128 x N fp32 TMEM accumulator.
//   - bf16 weights: activations arrive as bf16 (hi, lo) pairs; a stage holds the
//     weight slice and both activation halves and the MMA sums W.X_hi + W.X_lo.
//   - warps 2-5: for fp32 models they split each staged tile into tf32 high and low
//     parts and release the TMA stage at once, so the weight stream runs ahead of the
//     conversion; the MMA sums W_hi.X_hi + W_hi.X_lo + W_lo.X_hi (three tf32
//     products, fp32-level accuracy). The weight parts go to tensor memory (each
//     thread owns one weight row, its TMEM lane) and the MMAs read A from there: read
//     three times from shared memory instead, the weight tile costs about 140 KB of
//     shared-memory traffic per 16 KB of weights.
//     After the last MMA they read the accumulator with tcgen05.ld and stage it
//     transposed (tokens x weight rows) for the shared epilogue.
// Small matrices split K across a thread-block cluster of up to 16 CTAs; partial tiles
// are summed in rank order through distributed shared memory. The split depends on the
// weight shape and the cluster occupancy of the kernel variant, never on the data. Every
// wait is bounded and TMEM is always freed.
#include <cooperative_groups.h>

#include <algorithm>
#include <type_traits>

#include "epilogue.cuh"
#include "linear.cuh"
#include "tcgen05.cuh"

namespace cg = cooperative_groups;

namespace llm {

namespace {

constexpr int SW_THREADS = 192;
constexpr int SW_ROWS = 128;                 // weight rows per tile (MMA M)
constexpr int SW_A_BYTES = SW_ROWS * 128;    // one 128-byte K slice of 128 weight rows
constexpr int SW_OT_LD = SW_ROWS + 4;        // output-tile row stride (floats): 16-byte rows
constexpr int SW_MAX_KS = 16;                // cluster size limit (non-portable; 8 is portable)
constexpr int SW_RED_GROUP = 8;              // peers whose tiles one reduction round reads

template <int NT, bool TF32>
struct SwapCfg {
  static constexpr int B_BYTES = NT * 128;                // one 128-byte K slice of NT activation rows
  static constexpr int RAW = SW_A_BYTES + (TF32 ? 1 : 2) * B_BYTES;   // TMA stage: [W][X] or [W][X_hi][X_lo]
  static constexpr int CONVB = 2 * B_BYTES;             // tf32: [X hi][X lo] (the weight parts sit in TMEM)
  // TMA stages: bf16 keeps up to 4 within ~100 KB (a second CTA fits on the SM); tf32 keeps
  // 4 raw stages for up to 32 tokens (about 97 KB, two CTAs an SM, so split-K clusters can
  // be twice as large), 6 for 64 (one CTA an SM), plus 2 converted buffers (1 for the widest).
  static constexpr int NRAW = TF32 ? (NT <= 32 ? 4 : (NT <= 64 ? 6 : (NT <= 128 ? 4 : 2)))
                                   : (4 * RAW <= 100 * 1024 ? 4 : (3 * RAW <= 100 * 1024 ? 3 : 2));
  static constexpr int NCONV = TF32 ? (NT <= 128 ? 2 : 1) : 0;
  static constexpr size_t PIPE = (size_t)NRAW * RAW + (size_t)NCONV * CONVB;
  static constexpr size_t OT = (size_t)NT * SW_OT_LD * 4;
  static constexpr size_t RED = (size_t)((NT + 1) / 2) * SW_OT_LD * 4;   // ks >= 2: a rank reduces <= NT/2 rows
  static constexpr size_t BODY = PIPE > OT + RED ? PIPE : OT + RED;
  static constexpr size_t SMEM = 1024 + BODY + 256;
  static constexpr int KE = TF32 ? 32 : 64;            // K elements per stage (128 bytes)
  // TMEM: the accumulator (NT columns), then for tf32 one A buffer per converted stage
  // (32 columns of W_hi, 32 of W_lo); allocations are powers of two
  static constexpr int A_COL0 = NT < 32 ? 32 : NT;
  static constexpr int COLS_USED = A_COL0 + (TF32 ? NCONV * 64 : 0);
  static constexpr int TMEM_COLS = COLS_USED <= 32 ? 32 : COLS_USED <= 64 ? 64 : COLS_USED <= 128 ? 128
                                 : COLS_USED <= 256 ? 256 : 512;
  static_assert(COLS_USED <= 512, "TMEM holds 512 columns");
  static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};

// tf32 high part: the fp32 value rounded to 10 mantissa bits (to nearest, ties away, by an
// integer add on the bit pattern) with its 13 low bits cleared, so it is exactly
// representable in tf32 and the tensor core uses it unchanged; the low part x - hi is exact
// in fp32 and at most 2^-11 |x|.
__device__ __forceinline__ float hi13(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}
__device__ __forceinline__ float4 tf32_hi(const float4& x) {
  return make_float4(hi13(x.x), hi13(x.y), hi13(x.z), hi13(x.w));
}

template <int NT, bool TF32>
__global__ void __launch_bounds__(SW_THREADS, 1)
    k_gemm_tc_swap(const LinearParams p, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXlo, int kcta,
                   int ks_total) {
  using C = SwapCfg<NT, TF32>;
  using WT = typename std::conditional<TF32, float, bf16>::type;   // weight type
  constexpr int NR = C::NRAW, NC = C::NCONV > 0 ? C::NCONV : 1;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::BODY);   // TMA -> consumer, per raw stage
  uint64_t* rfree = full + NR;                                      // consumer -> TMA, per raw stage
  uint64_t* conv = rfree + NR;                                      // tf32: converter -> MMA
  uint64_t* cfree = conv + NC;                                      // tf32: MMA -> converter
  uint64_t* done = cfree + NC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  auto raw_a = [&](int r) { return base + (size_t)r * C::RAW; };
  auto raw_b = [&](int r) { return base + (size_t)r * C::RAW + SW_A_BYTES; };
  auto cv = [&](int c) { return base + (size_t)NR * C::RAW + (size_t)c * C::CONVB; };   // [X hi][X lo]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, ks = blockIdx.y;
  const int k0 = ks * kcta;
  const int kend = min(p.K, k0 + kcta);
  const int kiters = (kend - k0 + C::KE - 1) / C::KE;
  const int F = p.N, M = p.M;
  unsigned* flags = p.epi.flags;

  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    for (int r = 0; r < NR; ++r) {
      mbar_init(&full[r], 1);
      mbar_init(&rfree[r], TF32 ? 4 : 1);
    }
    for (int c = 0; c < NC; ++c) {
      mbar_init(&conv[c], 4);
      mbar_init(&cfree[c], 1);
    }
    mbar_init(done, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer
    auto load_w = [&](int r, int kc) {
      unsigned char* a = raw_a(r);
      if (p.swiglu) {
        for (int sub = 0; sub < 2; ++sub) {
          const int j0 = (tile * 2 + sub) * 32;
          tma_load_2d(a + (sub * 64) * 128, &tmW, kc, j0, &full[r]);
          tma_load_2d(a + (sub * 64 + 32) * 128, &tmW, kc, F + j0, &full[r]);
        }
      } else {
        tma_load_2d(a, &tmW, kc, tile * SW_ROWS, &full[r]);
      }
    };
    const int pre = min(NR, kiters);
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&full[i], C::RAW);
      load_w(i, k0 + i * C::KE);
    }
    auto load_x = [&](int r, int kc) {
      tma_load_2d(raw_b(r), &tmX, kc, 0, &full[r]);
      if constexpr (!TF32) tma_load_2d(raw_b(r) + C::B_BYTES, &tmXlo, kc, 0, &full[r]);
    };
    pdl_wait();
    for (int i = 0; i < pre; ++i) load_x(i, k0 + i * C::KE);
    for (int i = pre; i < kiters; ++i) {
      const int r = i % NR;
      if (!mbar_wait(&rfree[r], ((i / NR) - 1) & 1, flags)) break;
      mbar_arrive_expect_tx(&full[r], C::RAW);
      load_w(r, k0 + i * C::KE);
      load_x(r, k0 + i * C::KE);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    pdl_wait();
    constexpr uint32_t idesc = TF32 ? idesc_tf32(SW_ROWS, NT) : idesc_bf16(SW_ROWS, NT);
    for (int i = 0; i < kiters; ++i) {
      if constexpr (TF32) {
        const int c = i % NC;
        if (!mbar_wait(&conv[c], (i / NC) & 1, flags)) break;
        tc_fence_after();
        const uint32_t ahi = tmem + (uint32_t)(C::A_COL0 + c * 64), alo = ahi + 32;
        const uint64_t db = sw128_desc(cv(c)), dbl = sw128_desc(cv(c) + C::B_BYTES);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {   // 8 K elements per MMA: 8 TMEM columns of A, 32 bytes of B
          const uint64_t o = (uint64_t)(kk * 2);
          const uint32_t ak = (uint32_t)(kk * 8);
          tc_mma_tf32_ts(tmem, ahi + ak, db + o, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          tc_mma_tf32_ts(tmem, ahi + ak, dbl + o, idesc, 1u);
          tc_mma_tf32_ts(tmem, alo + ak, db + o, idesc, 1u);
        }
        tc_commit(&cfree[c]);
      } else {
        const int r = i % NR;
        if (!mbar_wait(&full[r], (i / NR) & 1, flags)) break;
        tc_fence_after();
        const uint64_t da = sw128_desc(raw_a(r)), db = sw128_desc(raw_b(r));
        const uint64_t dbl = sw128_desc(raw_b(r) + C::B_BYTES);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t o = (uint64_t)(kk * 2);
          tc_mma(tmem, da + o, db + o, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          tc_mma(tmem, da + o, dbl + o, idesc, 1u);
        }
        tc_commit(&rfree[r]);
      }
    }
    tc_commit(done);
  } else if (warp >= 2) {
    pdl_wait();
    if constexpr (TF32) {
      // ---- tf32 split of raw stage r into buffer c, then r goes back to the producer.
      // Weights: thread = one row of the tile = its TMEM lane; the row's 32 values are read
      // from the 128-byte-swizzled tile (16-byte chunk j of row m sits at chunk j ^ (m mod 8),
      // so eight lanes cover all banks) and its high and low parts go to TMEM columns
      // [0, 32) and [32, 64) of A buffer c. Activations: split elementwise in shared memory
      // (the swizzled layout is kept), the MMA's B operand.
      const int t = threadIdx.x - 64;                 // 0..127
      const int row = (warp & 3) * 32 + lane;         // this warp's TMEM lane quadrant
      const uint32_t tq = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      constexpr int XV = C::B_BYTES / 16;             // float4 of the activation tile
      constexpr int XPER = (XV + 127) / 128;
      for (int i = 0; i < kiters; ++i) {
        const int r = i % NR, c = i % NC;
        if (!mbar_wait(&full[r], (i / NR) & 1, flags)) break;
        if (i >= NC) {
          if (!mbar_wait(&cfree[c], ((i / NC) - 1) & 1, flags)) break;
          tc_fence_after();   // the MMAs that read A buffer c are complete
        }
        const float4* wrow = reinterpret_cast<const float4*>(raw_a(r) + row * 128);
        const float4* xs = reinterpret_cast<const float4*>(raw_b(r));
        float4 wv[8], xv[XPER];
#pragma unroll
        for (int j = 0; j < 8; ++j) wv[j] = wrow[j ^ (row & 7)];
#pragma unroll
        for (int u = 0; u < XPER; ++u) xv[u] = (t + 128 * u < XV) ? xs[t + 128 * u] : make_float4(0.f, 0.f, 0.f, 0.f);
        const uint32_t ta = tq + (uint32_t)(C::A_COL0 + c * 64);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {   // 16 columns a store
          uint32_t whi[16], wlo[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 v = wv[hh * 4 + j];
            const float4 h = tf32_hi(v);
            whi[4 * j + 0] = __float_as_uint(h.x); wlo[4 * j + 0] = __float_as_uint(v.x - h.x);
            whi[4 * j + 1] = __float_as_uint(h.y); wlo[4 * j + 1] = __float_as_uint(v.y - h.y);
            whi[4 * j + 2] = __float_as_uint(h.z); wlo[4 * j + 2] = __float_as_uint(v.z - h.z);
            whi[4 * j + 3] = __float_as_uint(h.w); wlo[4 * j + 3] = __float_as_uint(v.w - h.w);
          }
          tmem_st16(ta + (uint32_t)(hh * 16), whi);
          tmem_st16(ta + (uint32_t)(32 + hh * 16), wlo);
        }
        float4* xh = reinterpret_cast<float4*>(cv(c));
        float4* xl = reinterpret_cast<float4*>(cv(c) + C::B_BYTES);
#pragma unroll
        for (int u = 0; u < XPER; ++u) {
          if (t + 128 * u >= XV) break;
          const float4 h = tf32_hi(xv[u]);
          xh[t + 128 * u] = h;
          xl[t + 128 * u] = make_float4(xv[u].x - h.x, xv[u].y - h.y, xv[u].z - h.z, xv[u].w - h.w);
        }
        tmem_st_wait();
        tc_fence_before();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&conv[c]);
          mbar_arrive(&rfree[r]);
        }
      }
    }
  }

  pdl_wait();   // every thread writes outputs in the epilogue: all of them pass the dependency wait
  // rows whose epilogue this CTA runs: all of them, or its rank's slice of the split-K sum
  int r0 = 0, r1 = M;
  if (ks_total > 1) {
    const int rank = (int)cg::this_cluster().block_rank();
    const int rp = (M + ks_total - 1) / ks_total;
    r0 = min(M, rank * rp);
    r1 = min(M, r0 + rp);
  }
  const int n0 = p.swiglu ? tile * 64 : tile * SW_ROWS;
  // ---- accumulator -> shared memory, transposed to [token][weight row]
  bool ok = true;
  float* ot = reinterpret_cast<float*>(base);
  if (warp >= 2) {
    // stage the epilogue's bias / positions / KV blocks while the MMAs run
    epi_stage<WT>(p.epi, r0, r1 - r0, n0, SW_ROWS, p.N, threadIdx.x - 64, SW_THREADS - 64);
    ok = mbar_wait(done, 0, flags);
    if (!ok) ok = mbar_wait(done, 0, flags);
    tc_fence_after();
    __syncwarp();
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;          // weight row inside the tile
    if (ok) {
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < NT; c0 += 64) {   // two 32-column loads in flight per wait
        uint32_t r[32], r2[32];
        tmem_ld32(ta + (uint32_t)c0, r);
        if (c0 + 32 < NT) tmem_ld32(ta + (uint32_t)(c0 + 32), r2);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c0 + j < NT) ot[(c0 + j) * SW_OT_LD + row] = __uint_as_float(r[j]);
        if (c0 + 32 < NT) {
#pragma unroll
          for (int j = 0; j < 32; ++j) ot[(c0 + 32 + j) * SW_OT_LD + row] = __uint_as_float(r2[j]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  pdl_trigger();
  ok = __syncthreads_and(warp < 2 ? 1 : (ok ? 1 : 0)) != 0;
  if (!ok) {
    if (ks_total > 1) {   // keep the cluster barriers matched
      cg::this_cluster().sync();
      cg::this_cluster().sync();
    }
    return;
  }

  // one epilogue over the tile's 128 columns (two 64-column sub-tiles), staged above
  if (ks_total == 1) {
    epi_apply<WT>(p.epi, ot, SW_OT_LD, 0, M, n0, SW_ROWS, p.N, threadIdx.x, SW_THREADS);
    return;
  }
  // ---- split-K: rank r sums rows [r*rp, (r+1)*rp) of all ranks' partial tiles, in rank order
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  float* red = ot + (size_t)NT * SW_OT_LD;
  constexpr int C4 = SW_ROWS / 4;   // 16-byte reads of the peers' tiles
  constexpr int RU = 2;              // row groups per thread per round: 2 x 8 reads in flight
  const int nwork = (r1 - r0) * C4;
  for (int i0 = threadIdx.x; i0 < nwork; i0 += RU * SW_THREADS) {
    float4 sum[RU];
#pragma unroll
    for (int u = 0; u < RU; ++u) sum[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    // peers in rank order, eight at a time; ranks past ks_total add exact zeros
    for (int j0 = 0; j0 < ks_total; j0 += SW_RED_GROUP) {
      float4 v[RU][SW_RED_GROUP];
#pragma unroll
      for (int jj = 0; jj < SW_RED_GROUP; ++jj) {
        const int j = j0 + jj;
        const float* src = cluster.map_shared_rank(ot, j < ks_total ? j : 0);
#pragma unroll
        for (int u = 0; u < RU; ++u) {
          const int i = i0 + u * SW_THREADS;
          const int m = r0 + i / C4, c = (i % C4) * 4;
          v[u][jj] = (i < nwork && j < ks_total) ? *reinterpret_cast<const float4*>(src + m * SW_OT_LD + c)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < RU; ++u) {
#pragma unroll
        for (int jj = 0; jj < SW_RED_GROUP; ++jj) {
          if (j0 + jj == 0) {
            sum[u] = v[u][jj];
          } else {
            sum[u].x += v[u][jj].x; sum[u].y += v[u][jj].y; sum[u].z += v[u][jj].z; sum[u].w += v[u][jj].w;
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      const int i = i0 + u * SW_THREADS;
      if (i >= nwork) break;
      const int m = r0 + i / C4, c = (i % C4) * 4;
      *reinterpret_cast<float4*>(red + (m - r0) * SW_OT_LD + c) = sum[u];
    }
  }
  // the peers may still read this CTA's tile: signal that this CTA is done reading theirs,
  // run the epilogue, and only wait for the peers before exiting
  cluster_arrive();
  __syncthreads();
  if (r1 > r0) epi_apply<WT>(p.epi, red, SW_OT_LD, r0, r1 - r0, n0, SW_ROWS, p.N, threadIdx.x, SW_THREADS);
  cluster_wait();
}

template <int NT, bool TF32>
cudaError_t launch_nt(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
  using C = SwapCfg<NT, TF32>;
  const int tiles = p.swiglu ? (p.N + 63) / 64 : (p.N + SW_ROWS - 1) / SW_ROWS;
  const int wrows = p.swiglu ? 2 * p.N : p.N;
  // K split from the weight shape only (never from M): the largest cluster size <= 8 whose
  // grid still runs as one wave (the cluster occupancy the driver reports for this kernel),
  // with at least two K stages per CTA. Sizes need not be powers of two.
  auto kern = k_gemm_tc_swap<NT, TF32>;
  static bool attr_set_dev[MAX_DEVICES] = {};
  bool& attr_set = attr_set_dev[current_device()];
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  static int capacity_dev[MAX_DEVICES][SW_MAX_KS + 1] = {};   // CTAs of one wave per cluster size
  int* capacity = capacity_dev[current_device()];
  auto wave = [&](int c) {
    if (!capacity[c]) {
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(1, c);
      q.blockDim = dim3(SW_THREADS);
      q.dynamicSmemBytes = C::SMEM;
      cudaLaunchAttribute a[1];
      a[0].id = cudaLaunchAttributeClusterDimension;
      a[0].val.clusterDim.x = 1;
      a[0].val.clusterDim.y = c;
      a[0].val.clusterDim.z = 1;
      q.attrs = a;
      q.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = c <= 8 ? num_sms / c : 0;   // a non-portable size the driver does not confirm is not used
      }
      capacity[c] = n * c;
    }
    return capacity[c];
  };
  // Candidate splits in whole K stages: r ranks of s = ceil(stages / r) stages each (the last
  // rank may hold fewer), kept when every rank but the last streams at least two stages and
  // the grid is one wave; the most ranks win. Any size is allowed: 6 ranks pack a 19-SM GPC
  // better than 8, and 12 or 16 shorten long K.
  const int stages = (p.K + C::KE - 1) / C::KE;
  int ks = 1, kst = stages;   // ranks, stages per rank
  for (int c = 2; c <= SW_MAX_KS; ++c) {
    const int spr = (stages + c - 1) / c;
    const int ranks = (stages + spr - 1) / spr;
    if (spr >= 2 && ranks > ks && tiles * ranks <= wave(ranks)) {
      ks = ranks;
      kst = spr;
    }
  }
  const int kcta = kst * C::KE;
  const int dt = TF32 ? DT_F32 : DT_BF16;
  CUtensorMap mw, mx, mxl;
  if (!make_map(&mw, p.W, dt, wrows, p.K, p.K, p.swiglu ? 32 : SW_ROWS)) return cudaErrorInvalidValue;
  if (!make_map(&mx, p.X, dt, p.M, p.K, p.ldx, NT)) return cudaErrorInvalidValue;
  if (TF32) {
    mxl = mx;   // unused
  } else if (!make_map(&mxl, reinterpret_cast<const bf16*>(p.X) + p.ldx / 2, dt, p.M, p.K, p.ldx, NT)) {
    return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, ks);
  cfg.blockDim = dim3(SW_THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (ks > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = ks;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, p, mw, mx, mxl, kcta, ks);
}

template <bool TF32>
cudaError_t launch_at(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
  if (p.M <= 16) return launch_nt<16, TF32>(p, num_sms, s, pdl);
  if (p.M <= 32) return launch_nt<32, TF32>(p, num_sms, s, pdl);
  if (p.M <= 64) return launch_nt<64, TF32>(p, num_sms, s, pdl);
  if (p.M <= 128) return launch_nt<128, TF32>(p, num_sms, s, pdl);
  return launch_nt<256, TF32>(p, num_sms, s, pdl);
}

}  // namespace

// fp32 weights with fp32 activations (three tf32 products) or bf16 weights with bf16-pair
// activations (two bf16 products).
bool gemm_tc_swap_supported(const LinearParams& p) {
  if (p.M <= 0 || p.M > 256 || p.xnorm) return false;
  const bool f32 = p.wdt == DT_F32 && p.xdt == DT_F32 && p.adt == DT_F32;
  const bool pair = p.wdt == DT_BF16 && p.xdt == DT_SPLIT && p.adt == DT_SPLIT;
  if (!f32 && !pair) return false;
  if (p.K % 8 != 0 || p.ldx % 8 != 0) return false;
  if (pair && (p.ldx % 16 != 0 || p.ldx < 2 * p.K)) return false;
  if ((reinterpret_cast<uintptr_t>(p.W) | reinterpret_cast<uintptr_t>(p.X)) & 15) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_gemm_tc_swap(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
  if (p.M <= 0 || p.N <= 0 || p.K <= 0) return cudaSuccess;
  if (!gemm_tc_swap_supported(p)) return cudaErrorNotSupported;
  return p.wdt == DT_F32 ? launch_at<true>(p, num_sms, s, pdl) : launch_at<false>(p, num_sms, s, pdl);
}

}  // namespace llm
