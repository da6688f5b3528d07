// Prefill attention on the tensor cores (tcgen05 / TMEM).
//
// Causal attention over the prompt, reading K and V from the paged cache (fp32 or bf16) in
// place ("rvllm-metal", sections "What the kernels do" and "What's basic about it":
// scores, -inf mask, softmax, probs @ V, without gathering the context into a
// contiguous copy). CTA = (128 query rows of one sequence, query head h); two threads
// per query row, each owning 32 of a block's 64 key columns in the softmax and 32 of the
// 64 output dims; two CTAs (16 warps) per SM. For each block of 64 keys:
//   1. the threads split the keys' K and V rows (fp32, loaded from their paged blocks
//      into registers during the previous block) into bf16 hi = bf16(v),
//      lo = bf16(v - hi), written straight into the 128-byte-swizzled K-major layout
//      the MMA reads (V transposed to dims x keys), then issue the loads of the next
//      block's rows, which land while steps 2-4 run;
//   2. one thread issues S = Q.K^T as hi.hi + hi.lo + lo.hi (tcgen05.mma, M = 128
//      queries, N = 64 keys, fp32 accumulate in TMEM), so the scores carry about
//      16 bits of the operands instead of bf16's 8;
//   3. each thread reads its half of the score row from TMEM, applies the scale and the
//      causal mask, and the two threads of a row agree on the row maximum through shared
//      memory; the online softmax (running max, partial sums, log2 units) proceeds and the
//      probabilities are split the same way into the A operand of P.V;
//   4. P.V (M = 128, N = 64, K = 64) goes to a second TMEM accumulator and each
//      thread folds its 32 dims into its output: o = o * exp2(m_old - m_new) + P.V.
// One thread per query row ran about 1,200 dependent instructions per block with only 8
// warps an SM to hide their latency; the kernel was issue-latency bound.
// The output row is o / sum, stored as the activation dtype of the model.
// Every wait is bounded (FLAG_WAIT_TIMEOUT) and the tensor memory is always freed.
#include <type_traits>

#include "attention.cuh"
#include "tcgen05.cuh"

namespace llm {

namespace {

constexpr int PT_Q = 128;          // query rows per CTA (MMA M)
constexpr int PT_K = 64;           // keys per step
constexpr int PT_THREADS = 256;    // two threads per query row
constexpr int PT_TILE = 128 * 128;   // bytes of a 128-row x 64-bf16 swizzled tile
constexpr int PT_HALF = 64 * 128;    // bytes of a 64-row x 64-bf16 swizzled tile
// shared-memory layout (bytes from a 1024-aligned base): Q (128 queries x 64 dims), two
// buffers of K (64 keys x 64 dims) and V transposed (64 dims x 64 keys), the halves' row
// maxima / sums, and the CTA's physical KV blocks
constexpr int OFF_QHI = 0, OFF_QLO = OFF_QHI + PT_TILE;
constexpr int OFF_KV = OFF_QLO + PT_TILE;
constexpr int KV_BUF = 4 * PT_HALF;                          // [K hi][K lo][V hi][V lo]
constexpr int KV_KHI = 0, KV_KLO = PT_HALF, KV_VHI = 2 * PT_HALF, KV_VLO = 3 * PT_HALF;
constexpr int OFF_RED = OFF_KV + 2 * KV_BUF;                 // [2][128] floats
constexpr int PT_MAX_LB = 256;                               // table entries staged (4096 keys)
constexpr int OFF_PB = OFF_RED + 2 * PT_Q * 4;               // [PT_MAX_LB] ints
constexpr int OFF_BAR = OFF_PB + PT_MAX_LB * 4;
constexpr size_t PT_SMEM = 1024 + OFF_BAR + 64;
// TMEM: S in columns 0..63 (fp32), overwritten in place by P as bf16 pairs (P_hi in
// columns 0..31, P_lo in 32..63, two keys a column) for the P.V MMA's A operand; P.V in 64..127
constexpr uint32_t PT_TMEM_COLS = 128;
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

// KT: element type of the KV pool. A bf16 pool holds exactly its bf16 values, so K and V need
// no lo half and S and P.V take two products each (Q_hi.K + Q_lo.K, P_hi.V + P_lo.V).
template <typename KT, typename AT>
__global__ void __launch_bounds__(PT_THREADS, 2) k_attn_prefill_tc(const AttnPrefillParams p) {
  constexpr bool KV16 = std::is_same<KT, bf16>::value;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* barS = reinterpret_cast<uint64_t*>(base + OFF_BAR);
  uint64_t* barO = barS + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(barO + 1);
  float* s_red = reinterpret_cast<float*>(base + OFF_RED);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = tid & (PT_Q - 1), half = tid >> 7;   // query row; key columns and dims 32 half ..
  const int4 it = p.items[blockIdx.x];
  const int seq = it.x, qp0 = it.y, row0 = it.z, len = it.w;
  const int h = blockIdx.y, H = p.n_heads, Hkv = p.kv.n_kv_heads, g = h / (H / Hkv);
  const int nq = min(PT_Q, len - qp0);
  unsigned* flags = p.flags;

  if (warp == 0) {
    tmem_alloc(tmem_slot, PT_TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(barS, 1);
    mbar_init(barO, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_lane = (uint32_t)((warp & 3) * 32) << 16;   // warp w reaches TMEM lanes 32(w%4).. = rows r
  pdl_wait();
  const StepArgs* a = p.args;

  // Q row r (unscaled), dims 32 half .. 32 half + 31 -> Q_hi / Q_lo chunks 4 half ..
  {
    float v[32];
    if (r < nq) {
      const float* src = p.q + (size_t)(row0 + r) * H * HD + h * HD + half * 32;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 x = *reinterpret_cast<const float4*>(src + 4 * i);
        v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 hi, lo;
      split8(v + 8 * c, hi, lo);
      *reinterpret_cast<uint4*>(base + OFF_QHI + sw_off(r, 4 * half + c)) = hi;
      *reinterpret_cast<uint4*>(base + OFF_QLO + sw_off(r, 4 * half + c)) = lo;
    }
  }

  const int qpos = qp0 + min(r, nq - 1);        // rows beyond the item repeat the last query
  const int kend = min(len, qp0 + nq);          // keys 0..kend-1 are visible to some row
  const int nkb = (kend + PT_K - 1) / PT_K;
  const int W = p.window;                       // sliding window: keys qpos-W+1 .. qpos
  const int kb0 = W > 0 ? max(0, qp0 - W + 1) / PT_K : 0;   // first 64-key block any row sees
  const int lb0 = kb0 * (PT_K / KVB);
  const KT* kpool = reinterpret_cast<const KT*>(p.kv.k);
  const KT* vpool = reinterpret_cast<const KT*>(p.kv.v);
  constexpr uint32_t idS = idesc_bf16(PT_Q, PT_K);
  constexpr uint32_t idO = idesc_bf16(PT_Q, HD);
  float o[32];
#pragma unroll
  for (int d = 0; d < 32; ++d) o[d] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;   // l_run: this thread's key columns only
  bool ok = true;

  // physical block of every 16-key block the CTA reads (-1: out of range, flagged), so the
  // loads below wait on no table lookup
  int* s_pb = reinterpret_cast<int*>(base + OFF_PB);
  const int nlb = (kend + KVB - 1) / KVB;
  for (int lb = lb0 + tid; lb < min(nlb, lb0 + PT_MAX_LB); lb += PT_THREADS)
    s_pb[lb - lb0] = kv_block(p.kv, a->block_tables, seq, lb * KVB, flags);
  __syncthreads();

  // K and V of key kb*64 + kr, kr = tid mod 64: this thread converts dims 16 q4 .. 16 q4 + 15,
  // q4 = tid / 64. kv holds a later block's values (K, then V), loaded ahead in registers
  // (fp32 pool: 32 floats; bf16 pool: K in kraw, V unpacked to floats for the transpose).
  const int kr = tid & 63, q4 = tid >> 6;
  float kv[32];
  uint4 kraw[2];
  auto prefetch = [&](int kb) {
    const int t = kb * PT_K + kr;
    int pb = -1;
    if (t < kend) pb = (t >> 4) - lb0 < PT_MAX_LB ? s_pb[(t >> 4) - lb0] : kv_block(p.kv, a->block_tables, seq, t, flags);
    const size_t off = (pb >= 0 ? kv_offset(p.kv, pb, g, t & (KVB - 1)) : 0) + q4 * 16;
    if constexpr (KV16) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        kraw[i] = pb >= 0 ? *reinterpret_cast<const uint4*>(kpool + off + 8 * i) : make_uint4(0, 0, 0, 0);
        const uint4 x = pb >= 0 ? *reinterpret_cast<const uint4*>(vpool + off + 8 * i) : make_uint4(0, 0, 0, 0);
        Vec16<bf16>::unpack(x, kv + 16 + 8 * i);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 x = pb >= 0 ? *reinterpret_cast<const float4*>(kpool + off + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
        kv[4 * i] = x.x; kv[4 * i + 1] = x.y; kv[4 * i + 2] = x.z; kv[4 * i + 3] = x.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 x = pb >= 0 ? *reinterpret_cast<const float4*>(vpool + off + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
        kv[16 + 4 * i] = x.x; kv[16 + 4 * i + 1] = x.y; kv[16 + 4 * i + 2] = x.z; kv[16 + 4 * i + 3] = x.w;
      }
    }
  };
  // split the values in kv into K / V-transposed buffer b
  auto store_kv = [&](int b) {
    unsigned char* kvb = base + OFF_KV + b * KV_BUF;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if constexpr (KV16) {
        *reinterpret_cast<uint4*>(kvb + KV_KHI + sw_off(kr, 2 * q4 + c)) = kraw[c];
      } else {
        uint4 hi, lo;
        split8(kv + 8 * c, hi, lo);
        *reinterpret_cast<uint4*>(kvb + KV_KHI + sw_off(kr, 2 * q4 + c)) = hi;
        *reinterpret_cast<uint4*>(kvb + KV_KLO + sw_off(kr, 2 * q4 + c)) = lo;
      }
    }
    // V transposed: B operand of P.V is dims (rows) x keys (K). Neighbouring keys 2j, 2j+1
    // (lanes kr, kr ^ 1) pair up so every store is one 32-bit word of two keys: the even
    // lane writes dims 0..7 of its 16, the odd lane dims 8..15.
    const float* v = kv + 16;
    const int odd = kr & 1, ck = kr >> 3, bk = (kr & 6) * 2;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float mine = odd ? v[8 + j] : v[j];
      const float other = __shfl_xor_sync(0xffffffffu, odd ? v[j] : v[8 + j], 1);
      const float ke = odd ? other : mine, ko = odd ? mine : other;   // keys 2j, 2j + 1
      const __nv_bfloat162 hi = __floats2bfloat162_rn(ke, ko);   // exact for a bf16 pool
      const int d = q4 * 16 + odd * 8 + j;
      const uint32_t o2 = sw_off(d, ck) + bk;
      *reinterpret_cast<__nv_bfloat162*>(kvb + KV_VHI + o2) = hi;
      if constexpr (!KV16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(ke - __low2float(hi), ko - __high2float(hi));
        *reinterpret_cast<__nv_bfloat162*>(kvb + KV_VLO + o2) = lo;
      }
    }
  };
  if (nkb > kb0) {
    prefetch(kb0);
    store_kv(0);
    if (nkb > kb0 + 1) prefetch(kb0 + 1);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();   // Q and block 0 in shared memory
  tc_fence_after();

  // Per block kb: the S MMA runs while the threads store block kb + 1 into the other buffer
  // and load block kb + 2; softmax; P to TMEM; the P.V MMA; fold into o.
  for (int kb = kb0; kb < nkb && ok; ++kb) {
    const int b = (kb - kb0) & 1;
    unsigned char* kvb = base + OFF_KV + b * KV_BUF;
    if (tid == 0) {   // S = Q.K^T (three products), over S / P's columns: P.V of kb - 1 has completed
      const uint64_t dq = sw128_desc(base + OFF_QHI), dql = sw128_desc(base + OFF_QLO);
      const uint64_t dk = sw128_desc(kvb + KV_KHI), dkl = sw128_desc(kvb + KV_KLO);
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
        const uint64_t o2 = (uint64_t)(ks * 2);   // 32 bytes of K per MMA
        tc_mma(tmem, dq + o2, dk + o2, idS, ks > 0 ? 1u : 0u);
        if constexpr (!KV16) tc_mma(tmem, dq + o2, dkl + o2, idS, 1u);
        tc_mma(tmem, dql + o2, dk + o2, idS, 1u);
      }
      tc_commit(barS);
    }
    if (kb + 1 < nkb) {
      store_kv(b ^ 1);   // buffer b ^ 1 was last read by the P.V MMA of kb - 1, complete
      if (kb + 2 < nkb) prefetch(kb + 2);
      fence_async_smem();
    }
    ok = mbar_wait(barS, (kb - kb0) & 1, flags);
    ok = __syncthreads_and(ok) != 0;   // also: block kb + 1 is in shared memory
    if (!ok) break;
    tc_fence_after();

    // ---- online softmax: this thread's 32 key columns of row r (log2 units)
    float sc[32];
    float mb = -INFINITY;
    {
      uint32_t sr[32];
      tmem_ld32(tmem + t_lane + (uint32_t)(32 * half), sr);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int t = kb * PT_K + 32 * half + j;
        sc[j] = (t <= qpos && t < kend && (W <= 0 || t > qpos - W)) ? __uint_as_float(sr[j]) * SCALE_LOG2 : -INFINITY;
        mb = fmaxf(mb, sc[j]);
      }
    }
    s_red[half * PT_Q + r] = mb;
    tc_fence_before();
    __syncthreads();   // both halves' maxima are visible, and every S column has been read
    tc_fence_after();
    const float m_new = fmaxf(m_run, fmaxf(mb, s_red[(half ^ 1) * PT_Q + r]));
    // -inf only for a row whose window has not started yet: the reference 0 keeps its state 0
    const float m_ref = m_new == -INFINITY ? 0.0f : m_new;
    const float alpha = exp2f(m_run - m_ref);
    m_run = m_new;
    float lsum = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      sc[j] = exp2f(sc[j] - m_ref);   // masked: exp2(-inf) = 0
      lsum += sc[j];
    }
    l_run = l_run * alpha + lsum;
    {   // P row r, keys 32 half .. + 31 as bf16 pairs: P_hi columns 16 half .., P_lo 32 + 16 half ..
      uint32_t ph[16], pl[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const __nv_bfloat162 hi = __floats2bfloat162_rn(sc[2 * i], sc[2 * i + 1]);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(sc[2 * i] - __low2float(hi), sc[2 * i + 1] - __high2float(hi));
        ph[i] = *reinterpret_cast<const uint32_t*>(&hi);
        pl[i] = *reinterpret_cast<const uint32_t*>(&lo);
      }
      tmem_st16(tmem + t_lane + (uint32_t)(16 * half), ph);
      tmem_st16(tmem + t_lane + (uint32_t)(32 + 16 * half), pl);
      tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();   // P complete in TMEM
    tc_fence_after();
    if (tid == 0) {   // P.V: A = P from TMEM (8 columns per 16 keys), B = V transposed
      const uint32_t dO = tmem + (uint32_t)PT_K;
      const uint64_t dv = sw128_desc(kvb + KV_VHI), dvl = sw128_desc(kvb + KV_VLO);
#pragma unroll
      for (int ks = 0; ks < PT_K / 16; ++ks) {
        const uint64_t o2 = (uint64_t)(ks * 2);
        const uint32_t ph = tmem + (uint32_t)(ks * 8), pl = tmem + (uint32_t)(32 + ks * 8);
        tc_mma_ts(dO, ph, dv + o2, idO, ks > 0 ? 1u : 0u);
        if constexpr (!KV16) tc_mma_ts(dO, ph, dvl + o2, idO, 1u);
        tc_mma_ts(dO, pl, dv + o2, idO, 1u);
      }
      tc_commit(barO);
    }
    ok = mbar_wait(barO, (kb - kb0) & 1, flags);
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    tc_fence_after();
    {
      uint32_t v0[32];
      tmem_ld32(tmem + t_lane + (uint32_t)(PT_K + 32 * half), v0);   // dims 32 half ..
      tmem_ld_wait();
#pragma unroll
      for (int d = 0; d < 32; ++d) o[d] = fmaf(o[d], alpha, __uint_as_float(v0[d]));
    }
    // the next S MMA writes only S / P's columns, which every thread is done with; the next
    // P.V MMA comes after two more barriers, so these P.V reads are complete by then
    tc_fence_before();
  }
  pdl_trigger();
  // the row's sum of exponentials: this thread's key columns plus its partner's
  __syncthreads();   // every thread is done with s_red
  s_red[half * PT_Q + r] = l_run;
  __syncthreads();
  if (ok && r < nq) {
    const float inv = 1.0f / (l_run + s_red[(half ^ 1) * PT_Q + r]);
    const int ld = (std::is_same<AT, Split>::value ? 2 : 1) * H * HD;
#pragma unroll
    for (int d = 0; d < 32; d += 4) {
      float y[4] = {o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv};
      act_store4<AT>(p.out, row0 + r, ld, h * HD + 32 * half + d, y);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, PT_TMEM_COLS);
  }
}

template <typename KT, typename AT>
cudaError_t prefill_tc_t(const AttnPrefillParams& p, cudaStream_t s, bool pdl) {
  static bool attr_set_dev[MAX_DEVICES] = {};
  bool& attr_set = attr_set_dev[current_device()];
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(k_attn_prefill_tc<KT, AT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PT_SMEM);
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
  return cudaLaunchKernelEx(&cfg, k_attn_prefill_tc<KT, AT>, p);
}

}  // namespace

cudaError_t launch_attn_prefill_tc(const AttnPrefillParams& p, int kv_dtype, cudaStream_t s, bool pdl) {
  if (p.n_items <= 0) return cudaSuccess;
  if (p.n_heads % p.kv.n_kv_heads != 0) return cudaErrorInvalidValue;
  if (kv_dtype == DT_F32 && p.out_dtype == DT_F32) return prefill_tc_t<float, float>(p, s, pdl);
  if (kv_dtype == DT_F32 && p.out_dtype == DT_SPLIT) return prefill_tc_t<float, Split>(p, s, pdl);
  if (kv_dtype == DT_BF16 && p.out_dtype == DT_F32) return prefill_tc_t<bf16, float>(p, s, pdl);
  if (kv_dtype == DT_BF16 && p.out_dtype == DT_SPLIT) return prefill_tc_t<bf16, Split>(p, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace llm
