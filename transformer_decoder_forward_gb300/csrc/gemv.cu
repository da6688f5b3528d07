// Decode projection on CUDA cores: a weight stream for a handful of rows.
//
// Decode is memory bound: every step reads all weights once and does little
// arithmetic per byte ("rvllm-metal", section "The matmul pain story"). The
// pages' linear_small gives one simdgroup per output and re-reads the
// activations per output; here the activations of up to 32 rows sit in shared
// memory and every weight element loaded (16-byte streaming loads, 8 lanes
// covering 128 contiguous bytes of a row) is used for all of them.
//
// CTA = 256 threads = 8 warps and owns 64 output columns (one head: RoPE pairs,
// SwiGLU gate/up pairs and argmax tiles stay inside the CTA); warp w owns
// columns 8w..8w+7; in a warp, lane = 4 row groups x 8 k-lanes and each thread
// holds 2 weight rows.
//
// Small matrices split K across the CTAs of a thread-block cluster (the pages'
// linear_mma_small splits K across simdgroups because too few output tiles
// fill the GPU). Partials stay in shared memory; after a cluster barrier each
// CTA sums a slice of the rows over all ranks in rank order through
// distributed shared memory (deterministic, no global round trip) and runs the
// epilogue for that slice. The split depends on the weight shape only, so a
// row's arithmetic never depends on how many rows share the launch.
//
// Weights do not depend on earlier kernels: before waiting on its producer
// (programmatic dependent launch) a CTA already warms L2 with its weight slice
// and loads its first weight vectors into registers.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

#include "epilogue.cuh"
#include "linear.cuh"

namespace cg = cooperative_groups;

namespace llm {

namespace {

constexpr int GEMV_THREADS = 256;
constexpr int TL_LD = TILE_N + 1;   // padded row stride of the output tiles in smem
constexpr int GEMV_MT = 16;         // rows per CTA (larger M: more CTAs along grid.x)
// weight vectors per row in flight per thread and stage. One fp32 or bf16 row's accumulators
// leave registers free for four (qkv's and o's whole slice is then loaded before the dependency
// wait, the down projection's in three rounds instead of six: the batch-1 GPT-2 124M step 0.350 ->
// 0.318 ms). Two otherwise, so two CTAs an SM stay resident; for Q8_0 (16 weights a vector) three
// measured slower and four spill.
template <typename WT, int MT> constexpr int gemv_u() { return (MT == 1 && !std::is_same<WT, Q8>::value) ? 4 : 2; }

// 4 or 8 staged activations (fp32 in shared memory) into registers
template <int VEC>
__device__ __forceinline__ void lds_x(const float* p, float* f) {
#pragma unroll
  for (int i = 0; i < VEC; i += 4) {
    const float4 v = *reinterpret_cast<const float4*>(p + i);
    f[i] = v.x; f[i + 1] = v.y; f[i + 2] = v.z; f[i + 3] = v.w;
  }
}

__host__ __device__ constexpr size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Activations are staged in shared memory as fp32 (a bf16 pair is summed on the way in).
typedef float XT;
constexpr int XE = 4;   // staged x elements per 16 bytes

__host__ __device__ constexpr size_t gemv_smem(int MT, int kcta) {
  return align16((size_t)MT * (kcta + XE) * sizeof(XT)) + 2 * (size_t)MT * TL_LD * sizeof(float);
}

template <typename WT, int MT>
__global__ void __launch_bounds__(GEMV_THREADS) k_gemv(const LinearParams p, int kcta, int ks_total) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  using ST = typename Elem<WT>::type;   // stored weight element (int8 quants for Q8_0)
  using VT = typename VecT<WT>::type;   // norm gains / biases
  constexpr bool SPLIT_X = std::is_same<WT, bf16>::value;   // bf16 weights: x is a bf16 pair
  constexpr bool IS_Q8 = std::is_same<WT, Q8>::value;
  constexpr int VEC = Vec16<WT>::N;
  constexpr int STRIDE = 8 * VEC;
  constexpr int U = gemv_u<WT, MT>();
  // grid.x = row chunk (fastest, so the chunks sharing a weight slice run together), grid.y = K split,
  // grid.z = output tile
  const int tile = blockIdx.z, ks = blockIdx.y, mbase = blockIdx.x * MT;
  const int mcount = min(MT, p.M - mbase);
  const int k0 = ks * kcta;
  const int kcl = max(0, min(kcta, p.K - k0));
  const int ldxs = kcta + XE;
  XT* xs = reinterpret_cast<XT*>(smem_raw);                                          // [MT][ldxs]
  float* tl = reinterpret_cast<float*>(smem_raw + align16((size_t)MT * ldxs * sizeof(XT)));  // [MT][TL_LD]
  float* red = tl + MT * TL_LD;                                                      // [MT][TL_LD]
  const int F = p.N;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 3, kl = lane & 7;
  const ST* W = reinterpret_cast<const ST*>(p.W);
  const ST* wp[2];
  const __half* scl[2];   // Q8_0: the rows' block scales from k0
  bool rvalid[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int c = warp * 8 + g * 2 + r;   // tile column
    int row;
    if (p.swiglu) {
      row = swiglu_row(tile * 32, c, F);
      rvalid[r] = tile * 32 + (c & 31) < F;
    } else {
      row = tile * TILE_N + c;
      rvalid[r] = row < p.N;
    }
    wp[r] = W + (size_t)(rvalid[r] ? row : 0) * p.K + k0;
    scl[r] = IS_Q8 ? reinterpret_cast<const __half*>(p.Wscale) + (size_t)(rvalid[r] ? row : 0) * (p.K / Q8_BLOCK) +
                         k0 / Q8_BLOCK
                   : nullptr;
  }

  // ---- before the dependency wait: weights only
  const bool vec_ok = (p.K % VEC) == 0;
  const int kvec_end = vec_ok ? (kcl / VEC) * VEC : 0;
  if (threadIdx.x < TILE_N && kvec_end > 0 && ((p.K * sizeof(ST)) % 16) == 0) {
    const int c = threadIdx.x;
    const int row = p.swiglu ? swiglu_row(tile * 32, c, F) : tile * TILE_N + c;
    const bool ok = p.swiglu ? (tile * 32 + (c & 31) < F) : row < p.N;
    if (ok) bulk_prefetch_l2(W + (size_t)row * p.K + k0, (unsigned)(kvec_end * sizeof(ST)));
  }
  uint4 wa[U][2], wb[U][2];
  float da[U][2], db[U][2];   // Q8_0: the scale of each loaded 16-quant chunk's block
  auto load_w = [&](uint4 (&w)[U][2], float (&dd)[U][2], int kbase) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = kbase + u * STRIDE;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const bool in = rvalid[r] && kk < kvec_end;
        w[u][r] = in ? ldg_stream16(wp[r] + kk) : make_uint4(0, 0, 0, 0);
        if constexpr (IS_Q8) dd[u][r] = in ? __half2float(scl[r][kk / Q8_BLOCK]) : 0.0f;
      }
    }
  };
  load_w(wa, da, kl * VEC);
  // The epilogue's constants (the tile's bias, and for QKV the rows' positions and KV blocks)
  // depend on no kernel of the step either (the step arguments were written by its first node,
  // which has completed before any projection starts): staged before the wait, for the rows
  // this CTA's epilogue will handle.
  const int n0 = p.swiglu ? tile * 32 : tile * TILE_N;
  int er0 = 0, er1 = mcount;
  if (ks_total > 1) {
    const int rank = (int)cg::this_cluster().block_rank();
    const int rp = (mcount + ks_total - 1) / ks_total;
    er0 = min(mcount, rank * rp);
    er1 = min(mcount, er0 + rp);
  }
  if (er1 > er0) epi_stage<WT>(p.epi, mbase + er0, er1 - er0, n0, TILE_N, p.N, threadIdx.x, GEMV_THREADS);
  pdl_trigger();
  pdl_wait();

  // ---- stage this CTA's slice of X (rows mbase.., columns k0..k0+kcl) as fp32
  if (p.xnorm) {
    // X = Norm(h): each warp computes its rows' statistics over the whole row, then writes the
    // CTA's K slice of the normalised row (h is fp32, K % 4 == 0, K <= 2048)
    const float* hx = reinterpret_cast<const float*>(p.X);
    const VT* gw = reinterpret_cast<const VT*>(p.norm_g);
    const VT* bw = reinterpret_cast<const VT*>(p.norm_b);
    for (int m = warp; m < mcount; m += GEMV_THREADS / 32) {
      float4 v[ROW_NV];
      float mean, rstd;
      warp_row_stats(hx + (size_t)(mbase + m) * p.ldx, p.K, p.norm_ln != 0, p.norm_eps, v, mean, rstd);
      for (int k = lane; k < kcl; k += 32) {
        const float x = hx[(size_t)(mbase + m) * p.ldx + k0 + k];
        const float b = bw ? to_f32(bw[k0 + k]) : 0.0f;
        const float y = norm_apply(x, mean, rstd, to_f32(gw[k0 + k]), b);
        // bf16 weights: the value a stored activation pair would give back
        xs[(size_t)m * ldxs + k] = SPLIT_X ? pair_round(y) : y;
      }
    }
  } else if constexpr (SPLIT_X) {
    // row m: hi at [m*ldx + k], lo at [m*ldx + ldx/2 + k]
    const bf16* X = reinterpret_cast<const bf16*>(p.X);
    const int lo = p.ldx >> 1;
    const bool x_vec = ((lo % 4) == 0) && ((k0 % 4) == 0) && ((kcl % 4) == 0);
    if (x_vec) {
      const int chunks = kcl / 4;
      for (int i = threadIdx.x; i < mcount * chunks; i += GEMV_THREADS) {
        const int m = i / chunks, c = i - m * chunks;
        const bf16* r = X + (size_t)(mbase + m) * p.ldx + k0 + c * 4;
        const uint2 hi = *reinterpret_cast<const uint2*>(r);
        const uint2 lw = *reinterpret_cast<const uint2*>(r + lo);
        float4 v;
        v.x = __uint_as_float(hi.x << 16) + __uint_as_float(lw.x << 16);
        v.y = __uint_as_float(hi.x & 0xffff0000u) + __uint_as_float(lw.x & 0xffff0000u);
        v.z = __uint_as_float(hi.y << 16) + __uint_as_float(lw.y << 16);
        v.w = __uint_as_float(hi.y & 0xffff0000u) + __uint_as_float(lw.y & 0xffff0000u);
        *reinterpret_cast<float4*>(xs + (size_t)m * ldxs + c * 4) = v;
      }
    } else {
      for (int i = threadIdx.x; i < mcount * kcl; i += GEMV_THREADS) {
        const int m = i / kcl, k = i - m * kcl;
        xs[(size_t)m * ldxs + k] = act_load<Split>(X, mbase + m, p.ldx, k0 + k);
      }
    }
  } else {
    const float* X = reinterpret_cast<const float*>(p.X);
    const bool x_vec = ((p.ldx % XE) == 0) && ((k0 % XE) == 0) && ((kcl % XE) == 0);
    if (x_vec) {
      const int chunks = kcl / XE;
      for (int i = threadIdx.x; i < mcount * chunks; i += GEMV_THREADS) {
        const int m = i / chunks, c = i - m * chunks;
        cp_async16(xs + (size_t)m * ldxs + c * XE, X + (size_t)(mbase + m) * p.ldx + k0 + c * XE);
      }
      cp_async_commit();
      cp_async_wait_all();
    } else {
      for (int i = threadIdx.x; i < mcount * kcl; i += GEMV_THREADS) {
        const int m = i / kcl, k = i - m * kcl;
        xs[(size_t)m * ldxs + k] = X[(size_t)(mbase + m) * p.ldx + k0 + k];
      }
    }
  }
  __syncthreads();

  float acc[2][MT];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = 0.0f;

  auto fma_vec = [&](const uint4& w0, const uint4& w1, float d0, float d1, int k) {
    float f0[VEC], f1[VEC];
    Vec16<WT>::unpack(w0, f0);
    Vec16<WT>::unpack(w1, f1);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < mcount) {
        float xv[VEC];
        lds_x<VEC>(xs + (size_t)m * ldxs + k, xv);
        if constexpr (IS_Q8) {
          // the 16 quants share their block's scale: sum q * x, then scale once
          float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
          for (int j = 0; j < VEC; ++j) {
            s0 = fmaf(f0[j], xv[j], s0);
            s1 = fmaf(f1[j], xv[j], s1);
          }
          acc[0][m] = fmaf(d0, s0, acc[0][m]);
          acc[1][m] = fmaf(d1, s1, acc[1][m]);
        } else {
#pragma unroll
          for (int j = 0; j < VEC; ++j) {
            acc[0][m] = fmaf(f0[j], xv[j], acc[0][m]);
            acc[1][m] = fmaf(f1[j], xv[j], acc[1][m]);
          }
        }
      }
    }
  };

  for (int k = kl * VEC; k < kvec_end; k += U * STRIDE) {
    load_w(wb, db, k + U * STRIDE);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (k + u * STRIDE < kvec_end) fma_vec(wa[u][0], wa[u][1], da[u][0], da[u][1], k + u * STRIDE);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      wa[u][0] = wb[u][0];
      wa[u][1] = wb[u][1];
      da[u][0] = db[u][0];
      da[u][1] = db[u][1];
    }
  }
  // scalar tail (K not a multiple of the vector width; never for Q8_0, whose K is a multiple of 32)
  if constexpr (!IS_Q8) {
    for (int kk = kvec_end + kl; kk < kcl; kk += 8) {
      const float a0 = rvalid[0] ? to_f32(wp[0][kk]) : 0.0f;
      const float a1 = rvalid[1] ? to_f32(wp[1][kk]) : 0.0f;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < mcount) {
          const float x = xs[(size_t)m * ldxs + kk];
          acc[0][m] = fmaf(a0, x, acc[0][m]);
          acc[1][m] = fmaf(a1, x, acc[1][m]);
        }
      }
    }
  }

  // ---- reduce over the 8 k-lanes
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

  if (ks_total == 1) {
    __syncthreads();
    epi_apply<WT>(p.epi, tl, TL_LD, mbase, mcount, n0, TILE_N, p.N, threadIdx.x, GEMV_THREADS);
    return;
  }
  // ---- split-K reduction across the cluster through distributed shared memory
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int r0 = er0, r1 = er1;
  for (int i = threadIdx.x; i < (r1 - r0) * TILE_N; i += GEMV_THREADS) {
    const int m = r0 + i / TILE_N, c = i % TILE_N;
    float s = 0.0f;
#pragma unroll 8
    for (int j = 0; j < ks_total; ++j) s += cluster.map_shared_rank(tl, j)[m * TL_LD + c];
    red[(m - r0) * TL_LD + c] = s;
  }
  cluster.sync();   // every rank has finished reading the others' partials
  if (r1 > r0) epi_apply<WT>(p.epi, red, TL_LD, mbase + r0, r1 - r0, n0, TILE_N, p.N, threadIdx.x, GEMV_THREADS);
}

// K split (cluster size) from the weight shape only: enough CTAs to cover the SMs and an
// activation slice of at most 64 KB for a full row chunk.
template <typename WT>
void gemv_split(int tiles, int K, int num_sms, int* ks_out, int* kcta_out) {
  constexpr int STRIDE = 8 * Vec16<WT>::N;
  const int kmax = (64 * 1024) / (GEMV_MT * (int)sizeof(XT));
  int ks = 1;
  while (ks < 8 && (tiles * ks < num_sms || (K + ks - 1) / ks > kmax) && K / (ks * 2) >= STRIDE) ks *= 2;
  int kcta = (K + ks - 1) / ks;
  kcta = ((kcta + STRIDE - 1) / STRIDE) * STRIDE;
  *ks_out = (K + kcta - 1) / kcta;
  *kcta_out = kcta;
}

template <typename WT, int MT>
cudaError_t launch_t(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
  const int tiles = linear_tiles(p);
  const int zch = (p.M + MT - 1) / MT;
  int ks, kcta;
  gemv_split<WT>(tiles, p.K, num_sms, &ks, &kcta);
  const size_t smem = gemv_smem(MT, kcta);
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  auto kern = k_gemv<WT, MT>;
  static bool attr_set_dev[MAX_DEVICES] = {};
  bool& attr_set = attr_set_dev[current_device()];
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  if (tiles > 65535) return cudaErrorInvalidValue;
  cfg.gridDim = dim3(zch, ks, tiles);
  cfg.blockDim = dim3(GEMV_THREADS);
  cfg.dynamicSmemBytes = smem;
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
  return cudaLaunchKernelEx(&cfg, kern, p, kcta, ks);
}

template <typename WT>
cudaError_t launch_m(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
  if (p.M <= 1) return launch_t<WT, 1>(p, num_sms, s, pdl);
  if (p.M <= 2) return launch_t<WT, 2>(p, num_sms, s, pdl);
  if (p.M <= 4) return launch_t<WT, 4>(p, num_sms, s, pdl);
  if (p.M <= 8) return launch_t<WT, 8>(p, num_sms, s, pdl);
  return launch_t<WT, GEMV_MT>(p, num_sms, s, pdl);
}

}  // namespace

bool gemv_norm_supported(const LinearParams& p) {
  return p.M <= GEMV_MT && p.K % 4 == 0 && p.K <= ROW_NV * 128 && p.ldx % 4 == 0;
}

cudaError_t launch_gemv(const LinearParams& p, int num_sms, cudaStream_t s, bool pdl) {
  if (p.M <= 0 || p.N <= 0 || p.K <= 0) return cudaSuccess;
  if (p.wdt == DT_Q8 && (p.K % Q8_BLOCK != 0 || !p.Wscale)) return cudaErrorInvalidValue;
  if (p.xnorm) {
    if (!gemv_norm_supported(p) || p.xdt != DT_F32) return cudaErrorInvalidValue;
    if (p.wdt == DT_F32 && p.adt == DT_F32) return launch_m<float>(p, num_sms, s, pdl);
    if (p.wdt == DT_BF16 && p.adt == DT_SPLIT) return launch_m<bf16>(p, num_sms, s, pdl);
    if (p.wdt == DT_Q8 && p.adt == DT_F32) return launch_m<Q8>(p, num_sms, s, pdl);
    return cudaErrorInvalidValue;
  }
  if (p.wdt == DT_Q8 && p.xdt == DT_F32 && p.adt == DT_F32) return launch_m<Q8>(p, num_sms, s, pdl);
  if (p.wdt == DT_F32 && p.xdt == DT_F32 && p.adt == DT_F32) return launch_m<float>(p, num_sms, s, pdl);
  if (p.wdt == DT_BF16 && p.xdt == DT_SPLIT && p.adt == DT_SPLIT) return launch_m<bf16>(p, num_sms, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace llm
