// Causal attention reading K/V straight from the paged KV blocks.
//
// The pages run attention as five kernels (gather the paged context into a
// contiguous copy, scores, mask, softmax, probs @ V) and name a fused kernel
// that reads the blocks directly as the fix ("rvllm-metal", sections "What the
// kernels do" and "What's basic about it"). Both kernels here read each
// sequence's blocks in place through its block table (slot = table[pos / 16] * 16
// + pos mod 16) and never copy the context.
//
// Decode is split-K ("flash-decoding"): CTA (sequence b, KV head g, split s)
// scores the split's tokens for all query heads that share KV head g
// (grouped-query attention), keeps (max, sum of exp, unnormalised output), and a
// merge kernel rescales the splits to the common maximum. Prefill is a tiled
// online softmax: CTA (64 query rows, head) walks the causal key tiles.
//
// Scores are q.k / sqrt(64); masked keys get -inf so exp gives exactly 0.
#include "attention.cuh"

namespace llm {

namespace {

constexpr int AD_THREADS = 128;
constexpr int MAX_G = 8;
constexpr int MAX_SPLIT = 128;
constexpr float SM_SCALE = 0.125f;   // 1/sqrt(64)

// smem for one split: K and V blocks (split/16 blocks of 16 x 64 elements each), then a
// small fixed area. The whole split is in flight at once: one thread issues a TMA bulk
// copy per KV block (16 contiguous token rows of one head) onto a single mbarrier.
template <typename KT>
__host__ __device__ constexpr size_t attn_decode_smem(int split) {
  return 2 * (size_t)split * HD * sizeof(KT);
}

template <typename KT>
__global__ void __launch_bounds__(AD_THREADS) k_attn_decode_split(const AttnDecodeParams p) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ __align__(16) float qs[MAX_G][HD];
  __shared__ float sc[MAX_G][MAX_SPLIT];
  __shared__ __align__(16) float ored[AD_THREADS / 32][MAX_G][HD];
  __shared__ float red[AD_THREADS / 32][MAX_G];
  __shared__ float stat[2][MAX_G];
  __shared__ int blk_ok[MAX_SPLIT / KVB];
  __shared__ __align__(8) uint64_t bar;

  constexpr int EPL = 16 / sizeof(KT);    // elements per 16-byte load
  constexpr int LPT = HD / EPL;           // lanes per token row: 16 (fp32) or 8 (bf16)
  constexpr int TPW = 32 / LPT;           // token rows per warp load
  constexpr int NWARP = AD_THREADS / 32;
  constexpr unsigned BLK_BYTES = KVB * HD * sizeof(KT);

  const int Hkv = p.kv.n_kv_heads, H = p.n_heads, G = H / Hkv;
  const int b = blockIdx.x / Hkv, g = blockIdx.x - b * Hkv, sp = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  KT* Ks = reinterpret_cast<KT*>(dyn);
  KT* Vs = Ks + (size_t)p.split * HD;
  pdl_wait();   // the new token's K/V is written by the projection that precedes this kernel
  const StepArgs* a = p.args;
  const int pos = a->positions[b];
  const int ctx = pos + 1;
  const int t0 = sp * p.split;
  if (t0 >= ctx) return;
  const int nt = min(p.split, ctx - t0);
  const int nb = (nt + KVB - 1) / KVB;

  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) {
    const KT* kbase = reinterpret_cast<const KT*>(p.kv.k);
    const KT* vbase = reinterpret_cast<const KT*>(p.kv.v);
    int pbs[MAX_SPLIT / KVB];
    unsigned bytes = 0;
    for (int i = 0; i < nb; ++i) {
      pbs[i] = kv_block(p.kv, a->block_tables, b, t0 + i * KVB, p.flags);
      blk_ok[i] = pbs[i] >= 0;
      if (pbs[i] >= 0) bytes += 2 * BLK_BYTES;
    }
    mbar_arrive_expect_tx(&bar, bytes);
    for (int i = 0; i < nb; ++i) {
      if (pbs[i] < 0) continue;
      const size_t off = kv_offset(p.kv, pbs[i], g, 0);
      bulk_g2s(Ks + (size_t)i * KVB * HD, kbase + off, BLK_BYTES, &bar);
      bulk_g2s(Vs + (size_t)i * KVB * HD, vbase + off, BLK_BYTES, &bar);
    }
  }
  for (int i = tid; i < G * HD; i += AD_THREADS) {
    const int j = i / HD, d = i - j * HD;
    qs[j][d] = p.q[(size_t)b * H * HD + (size_t)(g * G + j) * HD + d] * SM_SCALE;
  }
  const bool ok = mbar_wait(&bar, 0, p.flags);
  __syncthreads();
  if (!ok) {
    // the copies may still be landing: give them one more bounded wait before leaving
    mbar_wait(&bar, 0, p.flags);
    return;
  }
  pdl_trigger();

  const int sub = lane / LPT, li = lane - sub * LPT;
  // ---- scores: LPT lanes per token row, 16-byte shared loads along the head dimension
  for (int tb = warp * TPW; tb < nt; tb += NWARP * TPW) {
    const int t = tb + sub;
    float kf[EPL];
    const bool valid = t < nt && blk_ok[t / KVB];
    if (valid) {
      Vec16<KT>::unpack(*reinterpret_cast<const uint4*>(Ks + (size_t)t * HD + li * EPL), kf);
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) kf[e] = 0.0f;
    }
    for (int j = 0; j < G; ++j) {
      float d = 0.0f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) d = fmaf(kf[e], qs[j][li * EPL + e], d);
#pragma unroll
      for (int o = LPT / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (li == 0 && t < nt) sc[j][t] = valid ? d : -INFINITY;
    }
  }
  __syncthreads();

  // ---- softmax statistics of this split
  for (int j = 0; j < G; ++j) {
    float m = -INFINITY;
    for (int t = tid; t < nt; t += AD_THREADS) m = fmaxf(m, sc[j][t]);
    m = warp_max(m);
    if (lane == 0) red[warp][j] = m;
  }
  __syncthreads();
  if (tid < G) {
    float m = red[0][tid];
    for (int w = 1; w < NWARP; ++w) m = fmaxf(m, red[w][tid]);
    stat[0][tid] = m;
  }
  __syncthreads();
  for (int j = 0; j < G; ++j) {
    const float m = stat[0][j];
    float l = 0.0f;
    for (int t = tid; t < nt; t += AD_THREADS) {
      const float e = m == -INFINITY ? 0.0f : expf(sc[j][t] - m);
      sc[j][t] = e;
      l += e;
    }
    l = warp_sum(l);
    if (lane == 0) red[warp][j] = l;
  }
  __syncthreads();
  if (tid < G) {
    float l = 0.0f;
    for (int w = 0; w < NWARP; ++w) l += red[w][tid];
    stat[1][tid] = l;
  }

  // ---- P . V: LPT lanes cover the head dimension, token groups stride the split
  constexpr int NTG = AD_THREADS / LPT;
  const int dg = tid % LPT, tg = tid / LPT;
  float acc[MAX_G][EPL];
#pragma unroll
  for (int j = 0; j < MAX_G; ++j)
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[j][e] = 0.0f;
  for (int t = tg; t < nt; t += NTG) {
    if (!blk_ok[t / KVB]) continue;
    float vf[EPL];
    Vec16<KT>::unpack(*reinterpret_cast<const uint4*>(Vs + (size_t)t * HD + dg * EPL), vf);
#pragma unroll
    for (int j = 0; j < MAX_G; ++j) {
      if (j < G) {
        const float pj = sc[j][t];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[j][e] = fmaf(pj, vf[e], acc[j][e]);
      }
    }
  }
  // reduce token groups inside the warp (lanes differing above the LPT bits), then across warps
#pragma unroll
  for (int j = 0; j < MAX_G; ++j) {
    if (j < G) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        float v = acc[j][e];
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        acc[j][e] = v;
      }
    }
  }
  if (lane < LPT) {
    for (int j = 0; j < G; ++j)
#pragma unroll
      for (int e = 0; e < EPL; ++e) ored[warp][j][dg * EPL + e] = acc[j][e];
  }
  __syncthreads();
  for (int i = tid; i < G * HD; i += AD_THREADS) {
    const int j = i / HD, d = i - j * HD;
    float o = 0.0f;
    for (int w = 0; w < NWARP; ++w) o += ored[w][j][d];
    const size_t hs = ((size_t)b * H + g * G + j) * p.max_splits + sp;
    p.part_o[hs * HD + d] = o;
    if (d == 0) {
      p.part_ml[hs * 2] = stat[0][j];
      p.part_ml[hs * 2 + 1] = stat[1][j];
    }
  }
}

template <typename AT>
__global__ void __launch_bounds__(HD) k_attn_decode_merge(const AttnDecodeParams p) {
  const int bh = blockIdx.x, b = bh / p.n_heads, d = threadIdx.x;
  pdl_wait();
  const int ctx = p.args->positions[b] + 1;
  const int ns = ctx <= 0 ? 0 : min(p.max_splits, (ctx + p.split - 1) / p.split);
  const float* ml = p.part_ml + (size_t)bh * p.max_splits * 2;
  const float* po = p.part_o + (size_t)bh * p.max_splits * HD;
  float m = -INFINITY;
  for (int s = 0; s < ns; ++s) m = fmaxf(m, ml[2 * s]);
  float l = 0.0f, o = 0.0f;
  for (int s = 0; s < ns; ++s) {
    const float w = m == -INFINITY ? 0.0f : expf(ml[2 * s] - m);
    l = fmaf(w, ml[2 * s + 1], l);
    o = fmaf(w, po[s * HD + d], o);
  }
  pdl_trigger();
  const float r = l > 0.0f ? o / l : 0.0f;
  reinterpret_cast<AT*>(p.out)[(size_t)bh * HD + d] = from_f32<AT>(r);
}

// ------------------------------------------------------------------------------------------------
// prefill: 64 query rows x 64 keys per tile, 256 threads, each 4 x 4 of S and of O
// ------------------------------------------------------------------------------------------------
constexpr int AP_THREADS = 256;
constexpr int AP_T = 64;
constexpr int AP_LD = AP_T + 4;

template <typename KT, typename AT>
__global__ void __launch_bounds__(AP_THREADS) k_attn_prefill(const AttnPrefillParams p) {
  extern __shared__ __align__(16) float sm[];
  float* Qt = sm;                  // [d][row]
  float* Kt = Qt + HD * AP_LD;     // [d][key]
  float* Vs = Kt + HD * AP_LD;     // [key][d]
  float* Pt = Vs + AP_T * AP_LD;   // [key][row]
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int4 it = p.items[blockIdx.x];
  const int seq = it.x, qp0 = it.y, row0 = it.z, len = it.w;
  const int h = blockIdx.y, H = p.n_heads, Hkv = p.kv.n_kv_heads, g = h / (H / Hkv);
  const int nq = min(AP_T, len - qp0);
  pdl_wait();
  const StepArgs* a = p.args;

  for (int i = tid; i < AP_T * HD; i += AP_THREADS) {
    const int r = i / HD, d = i - r * HD;
    Qt[d * AP_LD + r] = r < nq ? p.q[(size_t)(row0 + r) * H * HD + h * HD + d] * SM_SCALE : 0.0f;
  }
  float o[4][4], mrow[4], lrow[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    mrow[i] = -INFINITY;
    lrow[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) o[i][j] = 0.0f;
  }
  const KT* kbase = reinterpret_cast<const KT*>(p.kv.k);
  const KT* vbase = reinterpret_cast<const KT*>(p.kv.v);
  const int last_q = qp0 + nq - 1;
  const int n_kt = last_q / AP_T + 1;
  for (int kt = 0; kt < n_kt; ++kt) {
    __syncthreads();
    // load K (transposed) and V for keys kt*64 .. kt*64+63
    constexpr int EPL = 16 / sizeof(KT);
    for (int i = tid; i < AP_T * (HD / EPL); i += AP_THREADS) {
      const int key = i / (HD / EPL), d0 = (i - key * (HD / EPL)) * EPL;
      const int kp = kt * AP_T + key;
      float kf[EPL], vf[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) { kf[e] = 0.0f; vf[e] = 0.0f; }
      if (kp < len) {
        const int pb = kv_block(p.kv, a->block_tables, seq, kp, (d0 == 0) ? p.flags : nullptr);
        if (pb >= 0) {
          const size_t off = kv_offset(p.kv, pb, g, kp & (KVB - 1)) + d0;
          Vec16<KT>::unpack(ldg16(kbase + off), kf);
          Vec16<KT>::unpack(ldg16(vbase + off), vf);
        }
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        Kt[(d0 + e) * AP_LD + key] = kf[e];
        Vs[key * AP_LD + d0 + e] = vf[e];
      }
    }
    __syncthreads();
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s[i][j] = 0.0f;
#pragma unroll 8
    for (int d = 0; d < HD; ++d) {
      const float4 qv = *reinterpret_cast<const float4*>(Qt + d * AP_LD + ty * 4);
      const float4 kv = *reinterpret_cast<const float4*>(Kt + d * AP_LD + tx * 4);
      const float qa[4] = {qv.x, qv.y, qv.z, qv.w}, ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qa[i], ka[j], s[i][j]);
    }
    // causal mask, online softmax (rows spread over the 16 tx lanes of a half-warp)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qpos = qp0 + ty * 4 + i;
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int kp = kt * AP_T + tx * 4 + j;
        if (kp > qpos) s[i][j] = -INFINITY;
        tmax = fmaxf(tmax, s[i][j]);
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      const float mnew = fmaxf(mrow[i], tmax);
      const float alpha = expf(mrow[i] - mnew);   // mrow = -inf on the first tile -> 0
      float psum = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float e = expf(s[i][j] - mnew);
        s[i][j] = e;
        psum += e;
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      lrow[i] = lrow[i] * alpha + psum;
      mrow[i] = mnew;
#pragma unroll
      for (int j = 0; j < 4; ++j) o[i][j] *= alpha;
#pragma unroll
      for (int j = 0; j < 4; ++j) Pt[(tx * 4 + j) * AP_LD + ty * 4 + i] = s[i][j];
    }
    __syncthreads();
#pragma unroll 8
    for (int key = 0; key < AP_T; ++key) {
      const float4 pv = *reinterpret_cast<const float4*>(Pt + key * AP_LD + ty * 4);
      const float4 vv = *reinterpret_cast<const float4*>(Vs + key * AP_LD + tx * 4);
      const float pa[4] = {pv.x, pv.y, pv.z, pv.w}, va[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) o[i][j] = fmaf(pa[i], va[j], o[i][j]);
    }
  }
  pdl_trigger();
  AT* out = reinterpret_cast<AT*>(p.out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= nq) continue;
    const float inv = 1.0f / lrow[i];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      out[(size_t)(row0 + r) * H * HD + h * HD + tx * 4 + j] = from_f32<AT>(o[i][j] * inv);
  }
}

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr,
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

template <typename KT, typename AT>
cudaError_t decode_t(const AttnDecodeParams& p, cudaStream_t s, bool pdl) {
  const size_t smem = attn_decode_smem<KT>(p.split);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_decode_split<KT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)attn_decode_smem<KT>(MAX_SPLIT));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t c1 = make_cfg(dim3(p.B * p.kv.n_kv_heads, p.max_splits), dim3(AD_THREADS), smem, s, attr, pdl);
  cudaError_t e = cudaLaunchKernelEx(&c1, k_attn_decode_split<KT>, p);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr2[1];
  cudaLaunchConfig_t c2 = make_cfg(dim3(p.B * p.n_heads), dim3(HD), 0, s, attr2, pdl);
  return cudaLaunchKernelEx(&c2, k_attn_decode_merge<AT>, p);
}

template <typename KT, typename AT>
cudaError_t prefill_t(const AttnPrefillParams& p, cudaStream_t s, bool pdl) {
  const size_t smem = (size_t)(2 * HD * AP_LD + 2 * AP_T * AP_LD) * sizeof(float);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_prefill<KT, AT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t c = make_cfg(dim3(p.n_items, p.n_heads), dim3(AP_THREADS), smem, s, attr, pdl);
  return cudaLaunchKernelEx(&c, k_attn_prefill<KT, AT>, p);
}

}  // namespace

cudaError_t launch_attn_decode(const AttnDecodeParams& p, int kv_dtype, cudaStream_t s, bool pdl) {
  if (p.B <= 0) return cudaSuccess;
  if (p.n_heads / p.kv.n_kv_heads > MAX_G || p.split > MAX_SPLIT || (p.split % KVB) != 0)
    return cudaErrorInvalidValue;
  if (kv_dtype == DT_F32)
    return p.out_dtype == DT_F32 ? decode_t<float, float>(p, s, pdl) : decode_t<float, bf16>(p, s, pdl);
  return p.out_dtype == DT_F32 ? decode_t<bf16, float>(p, s, pdl) : decode_t<bf16, bf16>(p, s, pdl);
}

cudaError_t launch_attn_prefill(const AttnPrefillParams& p, int kv_dtype, cudaStream_t s, bool pdl) {
  if (p.n_items <= 0) return cudaSuccess;
  if (kv_dtype == DT_F32)
    return p.out_dtype == DT_F32 ? prefill_t<float, float>(p, s, pdl) : prefill_t<float, bf16>(p, s, pdl);
  return p.out_dtype == DT_F32 ? prefill_t<bf16, float>(p, s, pdl) : prefill_t<bf16, bf16>(p, s, pdl);
}

}  // namespace llm
