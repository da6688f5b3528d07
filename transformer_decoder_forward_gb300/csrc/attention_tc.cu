// Prefill attention on the tensor cores (tcgen05 / TMEM).
//
// Causal attention over the prompt, reading K and V from the paged fp32 cache in
// place ("rvllm-metal", sections "What the kernels do" and "What's basic about it":
// scores, -inf mask, softmax, probs @ V, without gathering the context into a
// contiguous copy). CTA = (128 query rows of one sequence, query head h); one thread
// per query row; two CTAs per SM overlap each other's loads. For each block of 64 keys:
//   1. the threads load the keys' K and V rows (fp32) from their paged blocks and
//      split every value v into bf16 hi = bf16(v), lo = bf16(v - hi), written straight
//      into the 128-byte-swizzled K-major layout the MMA reads (V transposed to
//      dims x keys);
//   2. one thread issues S = Q.K^T as hi.hi + hi.lo + lo.hi (tcgen05.mma, M = 128
//      queries, N = 64 keys, fp32 accumulate in TMEM), so the scores carry about
//      16 bits of the operands instead of bf16's 8;
//   3. each thread reads its score row from TMEM, applies the scale and the causal
//      mask, and updates an online softmax (running max and sum, log2 units); the
//      probabilities are split the same way into the A operand of P.V;
//   4. P.V (M = 128, N = 64, K = 64) goes to a second TMEM accumulator and each
//      thread folds it into its output row: o = o * exp2(m_old - m_new) + P.V.
// The output row is o / sum, stored as the activation dtype of the model.
// Every wait is bounded (FLAG_WAIT_TIMEOUT) and the tensor memory is always freed.
#include <type_traits>

#include "attention.cuh"
#include "tcgen05.cuh"

namespace llm {

namespace {

constexpr int PT_Q = 128;          // query rows per CTA (MMA M)
constexpr int PT_K = 64;           // keys per step
constexpr int PT_THREADS = 128;
constexpr int PT_TILE = 128 * 128;   // bytes of a 128-row x 64-bf16 swizzled tile
constexpr int PT_HALF = 64 * 128;    // bytes of a 64-row x 64-bf16 swizzled tile
// shared-memory layout (bytes from a 1024-aligned base): Q (128 queries x 64 dims),
// K (64 keys x 64 dims), V transposed (64 dims x 64 keys), P (128 queries x 64 keys)
constexpr int OFF_QHI = 0, OFF_QLO = OFF_QHI + PT_TILE;
constexpr int OFF_KHI = OFF_QLO + PT_TILE, OFF_KLO = OFF_KHI + PT_HALF;
constexpr int OFF_VHI = OFF_KLO + PT_HALF, OFF_VLO = OFF_VHI + PT_HALF;
constexpr int OFF_PHI = OFF_VLO + PT_HALF, OFF_PLO = OFF_PHI + PT_TILE;
constexpr int OFF_BAR = OFF_PLO + PT_TILE;
constexpr size_t PT_SMEM = 1024 + OFF_BAR + 64;
constexpr uint32_t PT_TMEM_COLS = 128;   // S: columns 0..63, P.V: 64..127
constexpr float SCALE_LOG2 = 0.125f * 1.4426950408889634f;   // log2(e) / sqrt(64)

// Byte offset of 16-byte chunk c (0..7) of row r in a K-major tile with 128-byte rows and
// the 128-byte swizzle (chunk index XOR row mod 8 within each 8-row, 1024-byte group).
__device__ __forceinline__ uint32_t sw_off(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// 8 fp32 -> 8 bf16 hi + 8 bf16 lo (hi = bf16(v), lo = bf16(v - hi)), each packed in 16 bytes.
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i] - __low2float(a), v[2 * i + 1] - __high2float(a));
    h[i] = *reinterpret_cast<const uint32_t*>(&a);
    l[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void load_row64(const float* src, float* v) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 x = *reinterpret_cast<const float4*>(src + 4 * i);
    v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
  }
}

template <typename AT>
__global__ void __launch_bounds__(PT_THREADS, 2) k_attn_prefill_tc(const AttnPrefillParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* barS = reinterpret_cast<uint64_t*>(base + OFF_BAR);
  uint64_t* barO = barS + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(barO + 1);

  const int r = threadIdx.x, warp = r >> 5;
  const int4 it = p.items[blockIdx.x];
  const int seq = it.x, qp0 = it.y, row0 = it.z, len = it.w;
  const int h = blockIdx.y, H = p.n_heads, Hkv = p.kv.n_kv_heads, g = h / (H / Hkv);
  const int nq = min(PT_Q, len - qp0);
  unsigned* flags = p.flags;

  if (warp == 0) {
    tmem_alloc(tmem_slot, PT_TMEM_COLS);
    tmem_relinquish();
  }
  if (r == 32) {
    mbar_init(barS, 1);
    mbar_init(barO, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_lane = (uint32_t)(warp * 32) << 16;   // this warp's TMEM lanes = its query rows
  pdl_wait();
  const StepArgs* a = p.args;

  // Q rows (unscaled) -> Q_hi / Q_lo
  {
    float v[64];
    if (r < nq) {
      load_row64(p.q + (size_t)(row0 + r) * H * HD + h * HD, v);
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] = 0.0f;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 hi, lo;
      split8(v + 8 * c, hi, lo);
      *reinterpret_cast<uint4*>(base + OFF_QHI + sw_off(r, c)) = hi;
      *reinterpret_cast<uint4*>(base + OFF_QLO + sw_off(r, c)) = lo;
    }
  }

  const int qpos = qp0 + min(r, nq - 1);        // rows beyond the item repeat the last query
  const int kend = min(len, qp0 + nq);          // keys 0..kend-1 are visible to some row
  const int nkb = (kend + PT_K - 1) / PT_K;
  const float* kpool = reinterpret_cast<const float*>(p.kv.k);
  const float* vpool = reinterpret_cast<const float*>(p.kv.v);
  constexpr uint32_t idS = idesc_bf16(PT_Q, PT_K);
  constexpr uint32_t idO = idesc_bf16(PT_Q, HD);
  float o[HD];
#pragma unroll
  for (int d = 0; d < HD; ++d) o[d] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;
  bool ok = true;

  for (int kb = 0; kb < nkb && ok; ++kb) {
    // ---- K and V of key kb*64 + (r mod 64): this thread converts dims 32h .. 32h + 31, h = r / 64
    {
      const int kr = r & 63, hf = r >> 6;
      const int t = kb * PT_K + kr;
      float v[32];
      int pb = -1;
      if (t < kend) pb = kv_block(p.kv, a->block_tables, seq, t, flags);
      const size_t off = (pb >= 0 ? kv_offset(p.kv, pb, g, t & (KVB - 1)) : 0) + hf * 32;
      auto load32 = [&](const float* src) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 x = pb >= 0 ? *reinterpret_cast<const float4*>(src + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
        }
      };
      load32(kpool + off);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 hi, lo;
        split8(v + 8 * c, hi, lo);
        *reinterpret_cast<uint4*>(base + OFF_KHI + sw_off(kr, 4 * hf + c)) = hi;
        *reinterpret_cast<uint4*>(base + OFF_KLO + sw_off(kr, 4 * hf + c)) = lo;
      }
      load32(vpool + off);
      // V transposed: B operand of P.V is dims (rows) x keys (K). Neighbouring keys 2j, 2j+1
      // (lanes kr, kr ^ 1) pair up so every store is one 32-bit word of two keys: the even
      // lane writes dims 0..15 of its half, the odd lane dims 16..31.
      const int odd = kr & 1, ck = kr >> 3, bk = (kr & 6) * 2;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float mine = odd ? v[16 + j] : v[j];
        const float other = __shfl_xor_sync(0xffffffffu, odd ? v[j] : v[16 + j], 1);
        const float ke = odd ? other : mine, ko = odd ? mine : other;   // keys 2j, 2j + 1
        const __nv_bfloat162 hi = __floats2bfloat162_rn(ke, ko);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(ke - __low2float(hi), ko - __high2float(hi));
        const int d = hf * 32 + odd * 16 + j;
        const uint32_t o2 = sw_off(d, ck) + bk;
        *reinterpret_cast<__nv_bfloat162*>(base + OFF_VHI + o2) = hi;
        *reinterpret_cast<__nv_bfloat162*>(base + OFF_VLO + o2) = lo;
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (r == 0) {
      const uint64_t dq = sw128_desc(base + OFF_QHI), dql = sw128_desc(base + OFF_QLO);
      const uint64_t dk = sw128_desc(base + OFF_KHI), dkl = sw128_desc(base + OFF_KLO);
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
        const uint64_t o2 = (uint64_t)(ks * 2);   // 32 bytes of K per MMA
        tc_mma(tmem, dq + o2, dk + o2, idS, ks > 0 ? 1u : 0u);
        tc_mma(tmem, dq + o2, dkl + o2, idS, 1u);
        tc_mma(tmem, dql + o2, dk + o2, idS, 1u);
      }
      tc_commit(barS);
    }
    ok = mbar_wait(barS, kb & 1, flags);
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    tc_fence_after();

    // ---- online softmax of this thread's score row (log2 units)
    float mb = -INFINITY;
#pragma unroll 1
    for (int c0 = 0; c0 < PT_K; c0 += 32) {
      uint32_t s[32];
      tmem_ld32(tmem + t_lane + (uint32_t)c0, s);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int t = kb * PT_K + c0 + j;
        if (t <= qpos && t < kend) mb = fmaxf(mb, __uint_as_float(s[j]) * SCALE_LOG2);
      }
    }
    const float m_new = fmaxf(m_run, mb);   // finite: key 0 <= qpos is in block 0
    const float alpha = exp2f(m_run - m_new);
    m_run = m_new;
    float lsum = 0.0f;
#pragma unroll 1
    for (int c0 = 0; c0 < PT_K; c0 += 32) {
      uint32_t s[32];
      tmem_ld32(tmem + t_lane + (uint32_t)c0, s);
      tmem_ld_wait();
      float pr[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int t = kb * PT_K + c0 + j;
        pr[j] = (t <= qpos && t < kend) ? exp2f(__uint_as_float(s[j]) * SCALE_LOG2 - m_new) : 0.0f;
        lsum += pr[j];
      }
      // P row r, keys c0..c0+31: chunks c0 / 8 ..
      unsigned char* phi = base + OFF_PHI;
      unsigned char* plo = base + OFF_PLO;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint4 hi, lo;
        split8(pr + 8 * cc, hi, lo);
        const int c = (c0 >> 3) + cc;
        *reinterpret_cast<uint4*>(phi + sw_off(r, c)) = hi;
        *reinterpret_cast<uint4*>(plo + sw_off(r, c)) = lo;
      }
    }
    l_run = l_run * alpha + lsum;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (r == 0) {
      const uint32_t dO = tmem + (uint32_t)PT_K;
#pragma unroll
      for (int ks = 0; ks < PT_K / 16; ++ks) {
        const uint64_t o2 = (uint64_t)(ks * 2);
        const uint64_t dp = sw128_desc(base + OFF_PHI) + o2;
        const uint64_t dpl = sw128_desc(base + OFF_PLO) + o2;
        const uint64_t dv = sw128_desc(base + OFF_VHI) + o2;
        const uint64_t dvl = sw128_desc(base + OFF_VLO) + o2;
        tc_mma(dO, dp, dv, idO, ks > 0 ? 1u : 0u);
        tc_mma(dO, dp, dvl, idO, 1u);
        tc_mma(dO, dpl, dv, idO, 1u);
      }
      tc_commit(barO);
    }
    ok = mbar_wait(barO, kb & 1, flags);
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    tc_fence_after();
    {
      uint32_t v0[32], v1[32];
      tmem_ld32(tmem + t_lane + (uint32_t)PT_K, v0);
      tmem_ld32(tmem + t_lane + (uint32_t)(PT_K + 32), v1);
      tmem_ld_wait();
#pragma unroll
      for (int d = 0; d < 32; ++d) {
        o[d] = fmaf(o[d], alpha, __uint_as_float(v0[d]));
        o[32 + d] = fmaf(o[32 + d], alpha, __uint_as_float(v1[d]));
      }
    }
    tc_fence_before();
    __syncthreads();   // every thread is done with this block's buffers and TMEM reads
    tc_fence_after();
  }
  pdl_trigger();
  if (ok && r < nq) {
    const float inv = 1.0f / l_run;
    const int ld = (std::is_same<AT, Split>::value ? 2 : 1) * H * HD;
#pragma unroll
    for (int d = 0; d < HD; d += 4) {
      float y[4] = {o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv};
      act_store4<AT>(p.out, row0 + r, ld, h * HD + d, y);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, PT_TMEM_COLS);
  }
}

template <typename AT>
cudaError_t prefill_tc_t(const AttnPrefillParams& p, cudaStream_t s, bool pdl) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(k_attn_prefill_tc<AT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PT_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_items, p.n_heads);
  cfg.blockDim = dim3(PT_THREADS);
  cfg.dynamicSmemBytes = PT_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_attn_prefill_tc<AT>, p);
}

}  // namespace

cudaError_t launch_attn_prefill_tc(const AttnPrefillParams& p, int kv_dtype, cudaStream_t s, bool pdl) {
  if (p.n_items <= 0) return cudaSuccess;
  if (kv_dtype != DT_F32 || p.n_heads % p.kv.n_kv_heads != 0) return cudaErrorInvalidValue;
  if (p.out_dtype == DT_F32) return prefill_tc_t<float>(p, s, pdl);
  if (p.out_dtype == DT_SPLIT) return prefill_tc_t<Split>(p, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace llm
