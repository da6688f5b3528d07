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
// merge kernel rescales the splits to the common maximum (no merge when every
// sequence fits one split). Prefill is a tiled
// online softmax: CTA (64 query rows, head) walks the causal key tiles.
//
// Scores are q.k / sqrt(64); masked keys get -inf so exp gives exactly 0.
#include <type_traits>

#include "attention.cuh"

namespace llm {

namespace {

constexpr int AD_WARPS = 4;
constexpr int MAX_G = 8;
constexpr int AD_MAX_BLOCKS_PER_WARP = 32;   // a split spans at most 4 * 32 blocks = 2048 tokens
constexpr float SM_SCALE = 0.125f;          // 1/sqrt(64)
constexpr float LOG2E = 1.4426950408889634f;

// Shared-memory ring of one warp: NST stages, each TOK tokens (a 16-token block, or half of
// one) of one KV head, K then V, filled by 1-D TMA bulk copies. NW warps a CTA.
template <typename KT, int NW = AD_WARPS, int TOK = KVB>
struct AttnRing {
  static constexpr int BLK = TOK * HD * (int)sizeof(KT);
  static constexpr int NST = sizeof(KT) == 4 ? 2 : 3;   // 64 KB (fp32) / 48 KB per CTA: three CTAs an SM
  static constexpr int WARP_BYTES = NST * 2 * BLK;
  static constexpr size_t SMEM = (size_t)NW * WARP_BYTES + (size_t)NW * NST * 8;
};

// Eight elements of one K or V row that lane dg (0..7) of a token row handles, as
// fp32: for fp32 rows dims 4dg..4dg+3 and 32+4dg..32+4dg+3 (two 16-byte reads that
// eight lanes take from distinct banks), for bf16 rows dims 8dg..8dg+7.
__device__ __forceinline__ int lane_dim(int dg, int e, bool f32) {
  return f32 ? (e < 4 ? 4 * dg + e : 32 + 4 * dg + (e - 4)) : 8 * dg + e;
}
template <typename KT> __device__ __forceinline__ void lds_row8(const KT* row, int dg, float* f);
template <> __device__ __forceinline__ void lds_row8<float>(const float* row, int dg, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(row + 4 * dg);
  const float4 c = *reinterpret_cast<const float4*>(row + 32 + 4 * dg);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
}
template <> __device__ __forceinline__ void lds_row8<bf16>(const bf16* row, int dg, float* f) {
  Vec16<bf16>::unpack(*reinterpret_cast<const uint4*>(row + 8 * dg), f);
}

// Decode attention, one CTA per (sequence b, KV head g, chunk of `split` tokens).
// The chunk's KV blocks are dealt to the NW warps in turn: 16-token blocks to 4 warps, or, for
// many long sequences with one or two query heads per KV head (the GPT-2 XL shape), 8-token half
// blocks to 8 warps (the same 64 KB ring a CTA, twice the warps streaming). Each warp runs its
// own pipeline: lane 0 streams the warp's blocks into a ring of shared-memory stages
// with 1-D TMA bulk copies (one mbarrier per stage), so several blocks per warp are
// in flight without holding them in registers, while the warp computes on the oldest
// stage and keeps an online softmax (running max, sum of exp, unnormalised output)
// for every query head of the group in registers. A token row is 8 lanes wide (8
// values a lane), four token rows per warp step; the lanes that score a token weight
// its value row, so no probability is broadcast. Scores are kept in log2 units (q is
// pre-scaled by log2(e)/sqrt(64)) so every exponential is one exp2. The warps'
// states are merged in shared memory at the end.
template <typename KT, typename AT, int GMAX, int NW = AD_WARPS, int TOK = KVB>
__global__ void __launch_bounds__(NW * 32) k_attn_decode_split(const AttnDecodeParams p) {
  using R = AttnRing<KT, NW, TOK>;
  constexpr int NST = R::NST, NTH = NW * 32;
  constexpr int TG = 4, IT = TOK / TG;        // 4 token rows per step, TOK / 4 steps per stage
  constexpr bool F32 = sizeof(KT) == 4;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float s_m[NW][GMAX], s_l[NW][GMAX];
  __shared__ __align__(16) float s_o[NW][GMAX][HD];

  const int Hkv = p.kv.n_kv_heads, H = p.n_heads, G = H / Hkv;
  const int b = blockIdx.x / Hkv, g = blockIdx.x - b * Hkv, sp = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int dg = lane & 7, tg = lane >> 3;
  unsigned char* ring = smem + (size_t)warp * R::WARP_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)NW * R::WARP_BYTES) + warp * NST;
  auto kst = [&](int s) { return reinterpret_cast<const KT*>(ring + (size_t)s * 2 * R::BLK); };
  auto vst = [&](int s) { return reinterpret_cast<const KT*>(ring + (size_t)s * 2 * R::BLK + R::BLK); };
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  __syncwarp();

  // Before the dependency wait this CTA reads only what no kernel of the step writes: the
  // step's positions and block tables, and every KV block except the one holding the new
  // token, which the projection that precedes this kernel writes. So the table lookups and
  // the first copies of older blocks overlap the end of that projection.
  const StepArgs* a = p.args;
  const int ctx = a->positions[b] + 1;
  // visible keys lo..ctx-1 (a sliding window starts at ctx - W); the span from the block that
  // holds lo is cut into ns = ceil(span / split) even chunks (16-token multiples). Every block
  // a warp reads then holds at least one visible key, so its score maximum is finite.
  const int lo = p.window > 0 ? max(0, ctx - p.window) : 0;
  const int tb = lo & ~(KVB - 1);
  const int span = ctx - tb;
  const int ns = ctx > 0 ? min(p.max_splits, (span + p.split - 1) / p.split) : 0;
  const int chunk = ns > 0 ? min(p.split, ((span + ns - 1) / ns + KVB - 1) / KVB * KVB) : 0;
  const int t0 = tb + sp * chunk;
  if (ns <= 0 || t0 >= ctx) {
    pdl_wait();
    return;
  }
  const int nt = min(chunk, ctx - t0);
  const int nblk = (nt + TOK - 1) / TOK;
  const int nj = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;   // this warp's stages: warp + NW*j
  // physical block of this warp's j-th stage, held by lane j
  int my_pb = -1;
  if (lane < nj) my_pb = kv_block(p.kv, a->block_tables, b, t0 + (warp + NW * lane) * TOK, p.flags);

  const KT* kbase = reinterpret_cast<const KT*>(p.kv.k);
  const KT* vbase = reinterpret_cast<const KT*>(p.kv.v);
  auto issue = [&](int j) {   // every lane calls; lane 0 fills stage j % NST with block j
    const int pb = __shfl_sync(0xffffffffu, my_pb, j);
    if (lane == 0) {
      uint64_t* bar = &bars[j % NST];
      if (pb >= 0) {
        // t0 is a multiple of 16: a half-block stage starts at slot 0 or 8 of its block
        const size_t off = kv_offset(p.kv, pb, g, ((warp + NW * j) * TOK) & (KVB - 1));
        mbar_arrive_expect_tx(bar, 2 * R::BLK);
        bulk_g2s(const_cast<KT*>(kst(j % NST)), kbase + off, R::BLK, bar);
        bulk_g2s(const_cast<KT*>(vst(j % NST)), vbase + off, R::BLK, bar);
      } else {
        mbar_arrive(bar);   // bad block (flagged): complete the phase without data
      }
    }
  };
  const int pre = min(NST, nj);
  const int new_blk = (ctx - 1 - t0) / TOK;   // chunk-relative stage of the new token
  int early = 0;                               // this warp's leading stages older than it
  while (early < pre && warp + NW * early < new_blk) ++early;
  for (int j = 0; j < early; ++j) issue(j);
  pdl_wait();   // q and the new token's K/V come from the preceding projection
  for (int j = early; j < pre; ++j) issue(j);

  float qf[GMAX][8], o[GMAX][8], m[GMAX], l[GMAX];
#pragma unroll
  for (int j = 0; j < GMAX; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      o[j][e] = 0.0f;
      qf[j][e] = j < G ? p.q[(size_t)b * H * HD + (size_t)(g * G + j) * HD + lane_dim(dg, e, F32)] * (SM_SCALE * LOG2E)
                       : 0.0f;
    }
  }

  bool ok = true;
  int j = 0;
  for (; j < nj; ++j) {
    const int s = j % NST;
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[s], (j / NST) & 1, p.flags)) != 0;
    if (!ok) break;
    const int pb = __shfl_sync(0xffffffffu, my_pb, j);
    if (pb >= 0) {
      const KT* K = kst(s);
      const KT* V = vst(s);
      const int tok0 = (warp + NW * j) * TOK;   // first token of the stage inside the chunk
      float sc[GMAX][IT];
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int t = it * TG + tg;
        float kf[8];
        lds_row8<KT>(K + t * HD, dg, kf);
        const bool valid = tok0 + t < nt && t0 + tok0 + t >= lo;
#pragma unroll
        for (int jj = 0; jj < GMAX; ++jj) {
          float d = 0.0f;
#pragma unroll
          for (int e = 0; e < 8; ++e) d = fmaf(kf[e], qf[jj][e], d);
          d += __shfl_xor_sync(0xffffffffu, d, 4);
          d += __shfl_xor_sync(0xffffffffu, d, 2);
          d += __shfl_xor_sync(0xffffffffu, d, 1);
          sc[jj][it] = valid ? d : -INFINITY;
        }
      }
#pragma unroll
      for (int jj = 0; jj < GMAX; ++jj) {
        if (jj >= G) continue;
        float mb = sc[jj][0];
#pragma unroll
        for (int it = 1; it < IT; ++it) mb = fmaxf(mb, sc[jj][it]);
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
        // mb is finite (every block holds a visible key) and the same in every lane; the
        // running state only needs rescaling when the maximum grows (alpha = 1 otherwise)
        if (mb > m[jj]) {
          const float alpha = exp2f(m[jj] - mb);   // m = -inf gives 0
          m[jj] = mb;
          l[jj] *= alpha;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[jj][e] *= alpha;
        }
      }
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        float vf[8];
        lds_row8<KT>(V + (it * TG + tg) * HD, dg, vf);
#pragma unroll
        for (int jj = 0; jj < GMAX; ++jj) {
          if (jj >= G) continue;
          const float pr = exp2f(sc[jj][it] - m[jj]);   // masked: exp2(-inf) = 0
          l[jj] += pr;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[jj][e] = fmaf(pr, vf[e], o[jj][e]);
        }
      }
    }
    __syncwarp();   // every lane is done with stage s
    if (j + NST < nj) {
      fence_async_smem();   // order the reads above before the bulk copy overwrites the stage
      issue(j + NST);
    }
  }
  if (!ok) {
    // a copy never arrived (flag set): wait, bounded, for this warp's copies still in flight
    for (int jj = j; jj < min(nj, j + NST); ++jj) mbar_wait(&bars[jj % NST], (jj / NST) & 1, p.flags);
  }

  // warp: sum l and o over the 4 token rows (m is warp-uniform)
#pragma unroll
  for (int jj = 0; jj < GMAX; ++jj) {
#pragma unroll
    for (int x = 8; x < 32; x <<= 1) {
      l[jj] += __shfl_xor_sync(0xffffffffu, l[jj], x);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[jj][e] += __shfl_xor_sync(0xffffffffu, o[jj][e], x);
    }
  }
  if (tg == 0) {
#pragma unroll
    for (int jj = 0; jj < GMAX; ++jj) {
      if (jj >= G) continue;
      if (dg == 0) {
        s_m[warp][jj] = ok ? m[jj] : -INFINITY;
        s_l[warp][jj] = ok ? l[jj] : 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) s_o[warp][jj][lane_dim(dg, e, F32)] = ok ? o[jj][e] : 0.0f;
    }
  }
  __syncthreads();
  pdl_trigger();
  // Combine the warps. With a single chunk per sequence (max_splits == 1) the result is
  // final; otherwise the chunk's (max, sum, output) goes to the partial buffer for the
  // merge kernel.
  const int ldo = (std::is_same<AT, Split>::value ? 2 : 1) * H * HD;
  for (int i = tid; i < G * HD; i += NTH) {
    const int jj = i / HD, d = i - jj * HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w][jj]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float c = s_m[w][jj] == -INFINITY ? 0.0f : exp2f(s_m[w][jj] - M);   // a warp without tokens: 0
      L = fmaf(c, s_l[w][jj], L);
      O = fmaf(c, s_o[w][jj][d], O);
    }
    if (p.max_splits == 1) {
      act_store<AT>(p.out, b, ldo, (g * G + jj) * HD + d, L > 0.0f ? O / L : 0.0f);
      continue;
    }
    const size_t hs = ((size_t)b * H + g * G + jj) * p.max_splits + sp;
    p.part_o[hs * HD + d] = O;
    if (d == 0) {
      p.part_ml[hs * 2] = M;
      p.part_ml[hs * 2 + 1] = L;
    }
  }
}

// Merge of a sequence's chunks (max_splits > 1): CTA = (sequence, query head), thread = dim.
// Rescales every chunk to the common maximum (log2 units) in chunk order.
template <typename AT>
__global__ void __launch_bounds__(HD) k_attn_decode_merge(const AttnDecodeParams p) {
  const int bh = blockIdx.x, b = bh / p.n_heads, d = threadIdx.x;
  pdl_wait();
  const int ctx = p.args->positions[b] + 1;
  const int tb = (p.window > 0 ? max(0, ctx - p.window) : 0) & ~(KVB - 1);   // as the split kernel
  const int ns = ctx <= 0 ? 0 : min(p.max_splits, (ctx - tb + p.split - 1) / p.split);
  const float* ml = p.part_ml + (size_t)bh * p.max_splits * 2;
  const float* po = p.part_o + (size_t)bh * p.max_splits * HD;
  constexpr int MS = 8;   // chunks per pass, all loads of a pass issued together
  float M = -INFINITY, L = 0.0f, O = 0.0f;
  for (int c0 = 0; c0 < ns; c0 += MS) {
    float mv[MS], lv[MS], ov[MS];
#pragma unroll
    for (int c = 0; c < MS; ++c) {
      const bool in = c0 + c < ns;
      mv[c] = in ? ml[2 * (c0 + c)] : -INFINITY;
      lv[c] = in ? ml[2 * (c0 + c) + 1] : 0.0f;
      ov[c] = in ? po[(size_t)(c0 + c) * HD + d] : 0.0f;
    }
    float Mn = M;
#pragma unroll
    for (int c = 0; c < MS; ++c) Mn = fmaxf(Mn, mv[c]);
    const float r = M == -INFINITY ? 0.0f : exp2f(M - Mn);
    L *= r;
    O *= r;
#pragma unroll
    for (int c = 0; c < MS; ++c) {
      const float w = mv[c] == -INFINITY ? 0.0f : exp2f(mv[c] - Mn);
      L = fmaf(w, lv[c], L);
      O = fmaf(w, ov[c], O);
    }
    M = Mn;
  }
  pdl_trigger();
  const int ldo = (std::is_same<AT, Split>::value ? 2 : 1) * p.n_heads * HD;
  act_store<AT>(p.out, b, ldo, (bh - b * p.n_heads) * HD + d, L > 0.0f ? O / L : 0.0f);
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
  const int W = p.window;
  const int kt0 = W > 0 ? max(0, qp0 - W + 1) / AP_T : 0;   // first tile any row's window reaches
  for (int kt = kt0; kt < n_kt; ++kt) {
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
        if (kp > qpos || (W > 0 && kp <= qpos - W)) s[i][j] = -INFINITY;
        tmax = fmaxf(tmax, s[i][j]);
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      const float mnew = fmaxf(mrow[i], tmax);
      // a row that has seen no visible key yet (its window starts later) keeps m = -inf; the
      // reference 0 then gives alpha = 0 and exp(-inf) = 0 instead of exp(-inf - -inf)
      const float mref = mnew == -INFINITY ? 0.0f : mnew;
      const float alpha = expf(mrow[i] - mref);   // mrow = -inf on the first tile -> 0
      float psum = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float e = expf(s[i][j] - mref);
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
  const int ld = (std::is_same<AT, Split>::value ? 2 : 1) * H * HD;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= nq) continue;
    const float inv = 1.0f / lrow[i];
    float y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) y[j] = o[i][j] * inv;
    act_store4<AT>(p.out, row0 + r, ld, h * HD + tx * 4, y);
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

}  // namespace

int attn_decode_split_for(int B, int n_kv_heads, int max_ctx, int num_sms) {
  if (const char* env = getenv("LLM_ATTN_SPLIT")) {
    const int v = atoi(env);
    if (v >= KVB && v % KVB == 0) return v;
  }
  // 512 tokens (1024 when the (sequence, KV head) pairs alone fill the GPU several times):
  // long streams per warp and few partials to merge, short enough that uneven context
  // lengths still balance; shorter while the grid would not give every SM two CTAs.
  const long long pairs = (long long)B * n_kv_heads;
  int split = pairs >= 8LL * num_sms ? 1024 : 512;
  while (split > 64 && pairs * ((max_ctx + split - 1) / split) < 2LL * num_sms) split /= 2;
  return split;
}

namespace {

// One split-kernel instance: set its shared-memory limit once per device, launch it and, when a
// sequence spans several chunks, the merge.
template <typename KT, typename AT, int GMAX, int NW, int TOK>
cudaError_t decode_launch(const AttnDecodeParams& p, cudaStream_t s, bool pdl) {
  using R = AttnRing<KT, NW, TOK>;
  auto kern = k_attn_decode_split<KT, AT, GMAX, NW, TOK>;
  static bool attr_set_dev[MAX_DEVICES] = {};
  bool& attr_set = attr_set_dev[current_device()];
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)R::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t c1 = make_cfg(dim3(p.B * p.kv.n_kv_heads, p.max_splits), dim3(NW * 32), R::SMEM, s, attr, pdl);
  cudaError_t e = cudaLaunchKernelEx(&c1, kern, p);
  if (e != cudaSuccess || p.max_splits == 1) return e;
  cudaLaunchAttribute attr2[1];
  cudaLaunchConfig_t c2 = make_cfg(dim3(p.B * p.n_heads), dim3(HD), 0, s, attr2, pdl);
  return cudaLaunchKernelEx(&c2, k_attn_decode_merge<AT>, p);
}

template <typename KT, typename AT>
cudaError_t decode_t(const AttnDecodeParams& p, cudaStream_t s, bool pdl) {
  const int G = p.n_heads / p.kv.n_kv_heads;
  // 1024-token chunks (the (sequence, KV head) pairs fill the GPU several times) with one or two
  // query heads a KV head: 8 warps on half blocks (GPT-2 XL batch 256: attention about 2% faster);
  // elsewhere the per-stage cost of half blocks outweighs the extra warps
  if (p.split >= 1024 && G <= 2)
    return G == 1 ? decode_launch<KT, AT, 1, 8, KVB / 2>(p, s, pdl) : decode_launch<KT, AT, 2, 8, KVB / 2>(p, s, pdl);
  return G == 1   ? decode_launch<KT, AT, 1, AD_WARPS, KVB>(p, s, pdl)
         : G == 2 ? decode_launch<KT, AT, 2, AD_WARPS, KVB>(p, s, pdl)
         : G == 3 ? decode_launch<KT, AT, 3, AD_WARPS, KVB>(p, s, pdl)
         : G == 4 ? decode_launch<KT, AT, 4, AD_WARPS, KVB>(p, s, pdl)
                  : decode_launch<KT, AT, 8, AD_WARPS, KVB>(p, s, pdl);
}

template <typename KT, typename AT>
cudaError_t prefill_t(const AttnPrefillParams& p, cudaStream_t s, bool pdl) {
  const size_t smem = (size_t)(2 * HD * AP_LD + 2 * AP_T * AP_LD) * sizeof(float);
  static bool attr_set_dev[MAX_DEVICES] = {};
  bool& attr_set = attr_set_dev[current_device()];
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
  if (p.n_heads / p.kv.n_kv_heads > MAX_G || p.split <= 0 || (p.split % KVB) != 0 ||
      p.split > AD_WARPS * AD_MAX_BLOCKS_PER_WARP * KVB)
    return cudaErrorInvalidValue;
  if (kv_dtype == DT_F32 && p.out_dtype == DT_F32) return decode_t<float, float>(p, s, pdl);
  if (kv_dtype == DT_F32 && p.out_dtype == DT_SPLIT) return decode_t<float, Split>(p, s, pdl);
  if (kv_dtype == DT_BF16 && p.out_dtype == DT_F32) return decode_t<bf16, float>(p, s, pdl);
  if (kv_dtype == DT_BF16 && p.out_dtype == DT_SPLIT) return decode_t<bf16, Split>(p, s, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_prefill(const AttnPrefillParams& p, int kv_dtype, cudaStream_t s, bool pdl) {
  if (p.n_items <= 0) return cudaSuccess;
  if (kv_dtype == DT_F32 && p.out_dtype == DT_F32) return prefill_t<float, float>(p, s, pdl);
  if (kv_dtype == DT_F32 && p.out_dtype == DT_SPLIT) return prefill_t<float, Split>(p, s, pdl);
  if (kv_dtype == DT_BF16 && p.out_dtype == DT_F32) return prefill_t<bf16, float>(p, s, pdl);
  if (kv_dtype == DT_BF16 && p.out_dtype == DT_SPLIT) return prefill_t<bf16, Split>(p, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace llm
