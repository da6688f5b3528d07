// Prefill attention on the tensor cores, warp-specialised (tcgen05 / TMEM / bulk copies).
//
// Causal attention over the prompt reading K and V from the paged cache in place ("rvllm-metal",
// sections "What the kernels do" and "What's basic about it": scores, -inf mask, softmax,
// probs @ V, without gathering the context into a contiguous copy). CTA = one query head and
// two 128-row query tiles of one sequence (256 consecutive query positions); 64-key blocks.
// The roles run concurrently, joined by mbarriers:
//   loader (1 thread)     1-D bulk copies of the block's raw K and V rows (4 paged 16-token
//                         blocks each) into a three-stage raw ring;
//   converters (4 warps)  split each raw fp32 value into bf16 hi = bf16(v), lo = bf16(v - hi)
//                         and write K and V alike as [keys][dims] in 128-byte swizzled rows: K is
//                         S's K-major B operand, V P.V's MN-major B operand (a bf16 pool needs no
//                         lo half), three stages: S(j + 1) reads block j + 1 before P(j).V has
//                         released block j;
//   MMA (1 thread a tile) S_t = Q_t K^T as hi.hi + hi.lo + lo.hi into TMEM, with Q_t's hi and lo
//                         halves as the A operand in TMEM, and O_t += P_t V with P_t read from
//                         TMEM. S_t(j + 1) is issued as soon as the softmax has read S_t(j), so it
//                         runs while the softmax of block j does; P_t(j).V follows once P_t(j) is
//                         written;
//   softmax (8 warps a tile, two threads a query row, 32 key columns each)
//                         reads S from TMEM, masks, keeps the running maximum and sum (log2
//                         units), writes P as bf16 pairs into its own TMEM columns once the
//                         previous P.V has read them. O accumulates in TMEM;
//                         it is rescaled (read, multiplied, written back) only when a row's
//                         maximum grows by more than 2^8 over the reference the exponentials
//                         use, so most blocks touch O not at all.
// Every wait is bounded: one that gives up sets FLAG_WAIT_TIMEOUT and an abort word that makes
// every other role leave its loop; the MMA thread then drains the tensor pipe and the loader
// its copies before the TMEM is freed.
#include <type_traits>

#include "attention.cuh"
#include "tcgen05.cuh"

namespace llm {

namespace {

constexpr int Q2_T = 128;                 // query rows per tile (MMA M)
constexpr int Q2_K = 64;                  // keys per block
constexpr int Q2_CONV_WARPS = 4;
constexpr int Q2_SM_WARPS = 8;            // softmax warps per tile
constexpr int Q2_WARP_SM0 = 4, Q2_WARP_SM1 = 12, Q2_WARP_LOAD = 20, Q2_WARP_MMA = 21;   // MMA: warps 21, 22
constexpr int Q2_THREADS = 23 * 32;
constexpr float Q2_TAU = 8.0f;            // log2 units: rescale O when the max grows past 2^8
constexpr float Q2_SCALE_LOG2 = 0.125f * 1.4426950408889634f;   // log2(e) / sqrt(64), folded into Q

constexpr int Q2_HALF = 64 * 128;         // bytes of a 64-row x 64-bf16 swizzled tile
constexpr int Q2_NS = 3;                  // stages of the raw and of the converted K/V rings
constexpr int OFF_CV = 0;
constexpr int CV_STAGE = 4 * Q2_HALF;     // [K hi][K lo][V hi][V lo], rows = keys
constexpr int CV_KHI = 0, CV_KLO = Q2_HALF, CV_VHI = 2 * Q2_HALF, CV_VLO = 3 * Q2_HALF;
constexpr int OFF_RAW = OFF_CV + Q2_NS * CV_STAGE;
constexpr int RAW_STAGE = 2 * Q2_K * HD * 4;   // K rows then V rows (fp32 size; bf16 uses half)
constexpr int OFF_RED = OFF_RAW + Q2_NS * RAW_STAGE;
constexpr int Q2_MAX_LB = 512;                 // staged block-table entries (8192 keys)
constexpr int OFF_PB = OFF_RED + 2 * 2 * 2 * Q2_T * 4;   // [block parity][tile][half][row]
constexpr int OFF_BAR = OFF_PB + Q2_MAX_LB * 4;
constexpr int Q2_NBAR = 4 * Q2_NS + 12;
constexpr size_t Q2_SMEM = 1024 + OFF_BAR + Q2_NBAR * 8 + 16;
// tensor memory: tile t owns columns 256 t .. 256 t + 255: S (fp32, 64 keys), P (bf16 pairs: hi
// in 32 columns, lo in 32), O (fp32, 64 dims), Q (bf16 pairs: hi 32 columns, lo 32)
constexpr uint32_t Q2_TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_P = 64, TM_O = 128, TM_Q = 192;

__device__ __forceinline__ uint32_t sw_off2(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void split8b(const float* v, uint4& hi, uint4& lo) {
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

// Bounded wait that also leaves when another role gave up (abort word set).
__device__ __forceinline__ bool wait_ab(uint64_t* bar, unsigned parity, unsigned* flags, volatile int* abort_word) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (clock64() - t0 < WAIT_CYCLES) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_word) return false;
  }
  set_flag(flags, FLAG_WAIT_TIMEOUT);
  *abort_word = 1;
  return false;
}

__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// 2^x by the hardware approximation (PTX ex2.approx.ftz: relative error about 2^-22, 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename KT, typename AT>
__global__ void __launch_bounds__(Q2_THREADS, 1) k_attn_prefill_tc2(const AttnPrefillParams p) {
  constexpr bool KV16 = std::is_same<KT, bf16>::value;
  constexpr int BLKB = KVB * HD * (int)sizeof(KT);     // bytes of one 16-token block of one head
  constexpr int KREG = Q2_K * HD * (int)sizeof(KT);    // bytes of a raw stage's K rows
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + OFF_BAR);
  uint64_t* raw_full = bars + 0;
  uint64_t* raw_empty = raw_full + Q2_NS;
  uint64_t* kv_full = raw_empty + Q2_NS;
  uint64_t* kv_empty = kv_full + Q2_NS;
  uint64_t* q_full = kv_empty + Q2_NS;   // per tile, from here on
  uint64_t* s_full = q_full + 2;
  uint64_t* s_free = s_full + 2;         // the softmax has read S(j): S(j + 1) may overwrite it
  uint64_t* p_full = s_free + 2;
  uint64_t* pv_full = p_full + 2;
  uint64_t* done_bar = pv_full + 2;      // one per MMA thread
  volatile int* abort_word = reinterpret_cast<volatile int*>(bars + Q2_NBAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Q2_NBAR) + 1;
  float* red = reinterpret_cast<float*>(base + OFF_RED);
  int* s_pb = reinterpret_cast<int*>(base + OFF_PB);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int4 it = p.items[blockIdx.y];
  const int seq = it.x, qp0 = it.y, row0 = it.z, len = it.w;
  const int h = blockIdx.x, H = p.n_heads, Hkv = p.kv.n_kv_heads, g = h / (H / Hkv);
  unsigned* flags = p.flags;
  // tile t: query positions qp0 + 128 t + r, r < nq[t]; keys 0 .. kend[t] - 1 visible to some row
  int nq[2], kend[2], nkb[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    nq[t] = max(0, min(Q2_T, len - (qp0 + Q2_T * t)));
    kend[t] = nq[t] > 0 ? min(len, qp0 + Q2_T * t + nq[t]) : 0;
    nkb[t] = (kend[t] + Q2_K - 1) / Q2_K;
  }
  const int nkb_all = max(nkb[0], nkb[1]);
  const int kend_all = max(kend[0], kend[1]);

  if (warp == 0) {
    tmem_alloc(tmem_slot, Q2_TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int i = 0; i < Q2_NS; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], Q2_CONV_WARPS);
      mbar_init(&kv_full[i], Q2_CONV_WARPS);
      mbar_init(&kv_empty[i], 2);   // both tiles' MMA threads release a stage
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], Q2_SM_WARPS);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], Q2_SM_WARPS);
      mbar_init(&p_full[i], Q2_SM_WARPS);
      mbar_init(&pv_full[i], 1);
    }
    mbar_init(&done_bar[0], 1);
    mbar_init(&done_bar[1], 1);
    *abort_word = 0;
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  const StepArgs* a = p.args;

  // physical block of every 16-key block the CTA reads (-1: out of range, flagged)
  const int nlb = (kend_all + KVB - 1) / KVB;
  for (int lb = tid; lb < min(nlb, Q2_MAX_LB); lb += Q2_THREADS)
    s_pb[lb] = kv_block(p.kv, a->block_tables, seq, lb * KVB, flags);
  __syncthreads();
  auto pb_of = [&](int lb) {
    return lb < Q2_MAX_LB ? s_pb[lb] : kv_block(p.kv, a->block_tables, seq, lb * KVB, flags);
  };

  if (warp == Q2_WARP_LOAD) {
    // ---------------------------------------------------------------- loader
    if (lane == 0) {
      const KT* kpool = reinterpret_cast<const KT*>(p.kv.k);
      const KT* vpool = reinterpret_cast<const KT*>(p.kv.v);
      int last[Q2_NS] = {-1, -1, -1};
      for (int j = 0; j < nkb_all; ++j) {
        const int s = j % Q2_NS;
        if (j >= Q2_NS && !wait_ab(&raw_empty[s], ((j / Q2_NS) - 1) & 1, flags, abort_word)) break;
        unsigned char* raw = base + OFF_RAW + s * RAW_STAGE;
        int pbs[4];
        unsigned bytes = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int lb = 4 * j + i;
          pbs[i] = lb * KVB < kend_all ? pb_of(lb) : -1;
          if (pbs[i] >= 0) bytes += 2 * BLKB;
        }
        mbar_arrive_expect_tx(&raw_full[s], bytes);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (pbs[i] < 0) continue;
          const size_t off = kv_offset(p.kv, pbs[i], g, 0);
          bulk_g2s(raw + i * BLKB, kpool + off, BLKB, &raw_full[s]);
          bulk_g2s(raw + KREG + i * BLKB, vpool + off, BLKB, &raw_full[s]);
        }
        last[s] = j;
      }
      // copies still in flight must land before the CTA's shared memory goes away
      for (int s = 0; s < Q2_NS; ++s)
        if (last[s] >= 0) mbar_wait(&raw_full[s], (last[s] / Q2_NS) & 1, flags);
    }
  } else if (warp < Q2_CONV_WARPS) {
    // ---------------------------------------------------------------- converters
    // Thread ct converts key kr = ct mod 64 of the block, dims 32 dh .. 32 dh + 31 (dh = ct / 64),
    // one 16-byte chunk (4 fp32 / 8 bf16 values) at a time. Raw rows are 256 bytes apart, so the
    // lanes visit their chunks in an order rotated by kr / 2: the 8 lanes of a shared-memory
    // phase read 4 different chunk columns (two lanes, keys 2m and 2m + 1, share a chunk, which the
    // V transpose needs), instead of all reading the same one.
    const int ct = tid, kr = ct & 63, dh = ct >> 6;
    const int rot = kr >> 1;
    constexpr int EPC = 16 / (int)sizeof(KT);          // values of a 16-byte chunk
    constexpr int NCH = 32 / EPC;                       // chunks of the thread's 32 dims
    for (int j = 0; j < nkb_all; ++j) {
      const int s = j % Q2_NS;
      if (j >= Q2_NS && !__all_sync(0xffffffffu, wait_ab(&kv_empty[s], ((j / Q2_NS) - 1) & 1, flags, abort_word)))
        break;
      if (!__all_sync(0xffffffffu, wait_ab(&raw_full[s], (j / Q2_NS) & 1, flags, abort_word))) break;
      const unsigned char* raw = base + OFF_RAW + s * RAW_STAGE;
      unsigned char* cv = base + OFF_CV + s * CV_STAGE;
      const int t = j * Q2_K + kr;
      const bool valid = t < kend_all && pb_of(t >> 4) >= 0;   // else zeros: no stale value reaches P.V
      const KT* kraw = reinterpret_cast<const KT*>(raw) + kr * HD + 32 * dh;
      const KT* vraw = reinterpret_cast<const KT*>(raw + KREG) + kr * HD + 32 * dh;
      // All of a row's chunks are loaded first (independent shared-memory reads in flight
      // together), then converted and stored. K and V are stored alike, [keys][dims] in 128-byte
      // swizzled rows: K is S's K-major B operand, V P.V's MN-major B operand (N = dims
      // contiguous, K = keys along the rows), so V needs no transpose.
      uint4 xk[NCH];
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const KT* src = part ? vraw : kraw;
        const int hi_off = part ? CV_VHI : CV_KHI, lo_off = part ? CV_VLO : CV_KLO;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          const int c = (i + rot) & (NCH - 1);
          xk[i] = valid ? *reinterpret_cast<const uint4*>(src + EPC * c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          const int c = (i + rot) & (NCH - 1);
          const uint4 x = xk[i];
          if constexpr (KV16) {
            *reinterpret_cast<uint4*>(cv + hi_off + sw_off2(kr, 4 * dh + c)) = x;
          } else {
            const float v4[4] = {__uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z), __uint_as_float(x.w)};
            uint32_t h2[2], l2[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const __nv_bfloat162 hb = __floats2bfloat162_rn(v4[2 * q], v4[2 * q + 1]);
              const __nv_bfloat162 lb = __floats2bfloat162_rn(v4[2 * q] - __low2float(hb), v4[2 * q + 1] - __high2float(hb));
              h2[q] = *reinterpret_cast<const uint32_t*>(&hb);
              l2[q] = *reinterpret_cast<const uint32_t*>(&lb);
            }
            const uint32_t o = sw_off2(kr, 4 * dh + (c >> 1)) + (c & 1) * 8;   // 4 dims = 8 bytes of bf16
            *reinterpret_cast<uint2*>(cv + hi_off + o) = make_uint2(h2[0], h2[1]);
            *reinterpret_cast<uint2*>(cv + lo_off + o) = make_uint2(l2[0], l2[1]);
          }
        }
      }
      fence_async_smem();   // generic writes (and raw reads) before the tensor core / next copy
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&raw_empty[s]);
        mbar_arrive(&kv_full[s]);
      }
    }
  } else if (warp == Q2_WARP_MMA || warp == Q2_WARP_MMA + 1) {
    // ---------------------------------------------------------------- MMA issuers, one a tile
    // Issuing is the tile's critical resource (about 45 cycles a tcgen05.mma from one thread,
    // 48 MMAs a block for both tiles), so each tile has its own thread: S_t(j + 1) as soon as the
    // softmax has read S_t(j), P_t(j).V once P_t(j) is written. The tensor pipe runs a thread's
    // MMAs in order, so S_t(j + 2) completing means P_t(j).V has too. The two threads' MMAs touch
    // separate TMEM columns.
    if (lane == 0) {
      const int t = warp - Q2_WARP_MMA;
      constexpr uint32_t idS = idesc_bf16(Q2_T, Q2_K);
      constexpr uint32_t idO = idesc_bf16(Q2_T, HD) | (1u << 16);   // B (V) MN-major
      const uint32_t tt = tmem + (uint32_t)(256 * t);
      auto issue_S = [&](int j) {
        unsigned char* cv = base + OFF_CV + (j % Q2_NS) * CV_STAGE;
        const uint32_t qh = tt + TM_Q, ql = tt + TM_Q + 32;   // A: Q hi / lo, 8 columns a K step
        const uint64_t dk = sw128_desc(cv + CV_KHI), dkl = sw128_desc(cv + CV_KLO);
        const uint32_t d = tt + TM_S;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint64_t o2 = (uint64_t)(ks * 2);   // 32 bytes of K a step
          const uint32_t ak = (uint32_t)(ks * 8);
          tc_mma_ts(d, qh + ak, dk + o2, idS, ks > 0 ? 1u : 0u);
          if constexpr (!KV16) tc_mma_ts(d, qh + ak, dkl + o2, idS, 1u);
          tc_mma_ts(d, ql + ak, dk + o2, idS, 1u);
        }
        tc_commit(&s_full[t]);
      };
      auto issue_PV = [&](int j) {
        unsigned char* cv = base + OFF_CV + (j % Q2_NS) * CV_STAGE;
        const uint64_t dv = sw128_desc(cv + CV_VHI), dvl = sw128_desc(cv + CV_VLO);
        const uint32_t dO = tt + TM_O, sP = tt + TM_P;
#pragma unroll
        for (int ks = 0; ks < Q2_K / 16; ++ks) {
          const uint64_t o2 = (uint64_t)(ks * 128);   // 16 key rows of 128 bytes a step (MN-major B)
          const uint32_t ph = sP + (uint32_t)(ks * 8), pl = sP + (uint32_t)(32 + ks * 8);
          tc_mma_ts(dO, ph, dv + o2, idO, (j > 0 || ks > 0) ? 1u : 0u);
          if constexpr (!KV16) tc_mma_ts(dO, ph, dvl + o2, idO, 1u);
          tc_mma_ts(dO, pl, dv + o2, idO, 1u);
        }
        tc_commit(&pv_full[t]);
      };
      bool ok = wait_ab(&q_full[t], 0, flags, abort_word);
      int j = 0;
      if (ok && nkb[t] > 0) {
        ok = wait_ab(&kv_full[0], 0, flags, abort_word);
        if (ok) {
          tc_fence_after();
          issue_S(0);
        }
        for (; ok && j < nkb[t]; ++j) {
          if (j + 1 < nkb[t]) {
            const int s1 = (j + 1) % Q2_NS;
            if (!(ok = wait_ab(&s_free[t], j & 1, flags, abort_word))) break;
            if (!(ok = wait_ab(&kv_full[s1], ((j + 1) / Q2_NS) & 1, flags, abort_word))) break;
            tc_fence_after();
            issue_S(j + 1);
          }
          if (!(ok = wait_ab(&p_full[t], j & 1, flags, abort_word))) break;
          tc_fence_after();
          issue_PV(j);
          tc_commit(&kv_empty[j % Q2_NS]);   // this tile's reads of the stage are done when these complete
        }
      }
      // blocks only the other tile needs: release each stage in order, once it is filled (the
      // fill waited for this thread's earlier release of that stage)
      for (; ok && j < nkb_all; ++j) {
        if (!(ok = wait_ab(&kv_full[j % Q2_NS], (j / Q2_NS) & 1, flags, abort_word))) break;
        mbar_arrive(&kv_empty[j % Q2_NS]);
      }
      // every MMA issued completes before the tensor memory is freed
      tc_commit(&done_bar[t]);
      mbar_wait(&done_bar[t], 0, flags);
    }
  } else {
    // ---------------------------------------------------------------- softmax, tile t
    const int t = warp >= Q2_WARP_SM1 ? 1 : 0;
    const int gt = tid - 32 * (t ? Q2_WARP_SM1 : Q2_WARP_SM0);
    const int r = gt & (Q2_T - 1), half = gt >> 7;
    const uint32_t t_lane = (uint32_t)((warp & 3) * 32) << 16;
    const int nqt = nq[t];
    // Q rows of the tile (unscaled) -> hi / lo operands, dims 32 half .. 32 half + 31
    {
      float v[32];
      if (r < nqt) {
        // scaled into log2 units (log2(e) / sqrt(64)) before the split, so S needs no multiply
        const float* src = p.q + (size_t)(row0 + Q2_T * t + r) * H * HD + h * HD + half * 32;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 x = *reinterpret_cast<const float4*>(src + 4 * i);
          v[4 * i] = x.x * Q2_SCALE_LOG2; v[4 * i + 1] = x.y * Q2_SCALE_LOG2;
          v[4 * i + 2] = x.z * Q2_SCALE_LOG2; v[4 * i + 3] = x.w * Q2_SCALE_LOG2;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
      }
      // dims 32 half + 2i, 2i + 1 -> column 16 half + i of the hi and of the lo half (TMEM lane r)
      uint32_t qh[16], ql[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 hi, lo;
        split8b(v + 8 * c, hi, lo);
        qh[4 * c] = hi.x; qh[4 * c + 1] = hi.y; qh[4 * c + 2] = hi.z; qh[4 * c + 3] = hi.w;
        ql[4 * c] = lo.x; ql[4 * c + 1] = lo.y; ql[4 * c + 2] = lo.z; ql[4 * c + 3] = lo.w;
      }
      const uint32_t tq = tmem + t_lane + (uint32_t)(256 * t) + TM_Q + (uint32_t)(16 * half);
      tmem_st16(tq, qh);
      tmem_st16(tq + 32, ql);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[t]);
    }
    const int qpos = qp0 + Q2_T * t + min(r, max(nqt, 1) - 1);   // rows beyond the tile repeat its last
    float m_ref = -INFINITY, l_run = 0.0f;                        // l_run: this thread's 32 key columns
    bool ok = true;
    const uint32_t tS = tmem + t_lane + (uint32_t)(256 * t) + TM_S;
    const uint32_t tP = tmem + t_lane + (uint32_t)(256 * t) + TM_P;
    const uint32_t tO = tmem + t_lane + (uint32_t)(256 * t) + TM_O + (uint32_t)(32 * half);
    // the maxima exchange alternates between two buffers by block parity: S(j + 1) can complete
    // before the other half of a row has read block j's maximum, and a thread that runs ahead
    // then writes block j + 1's into the other buffer
    auto red_mine = [&](int j) { return red + ((j & 1) * 4 + 2 * t + half) * Q2_T; };
    auto red_other = [&](int j) { return red + ((j & 1) * 4 + 2 * t + (half ^ 1)) * Q2_T; };
    // Every warp of the group runs every iteration and every group barrier, also after a wait
    // gave up (ok false: the work is skipped), so no warp is left waiting at a named barrier.
    for (int j = 0; j < nkb[t]; ++j) {
      if (ok) ok = __all_sync(0xffffffffu, wait_ab(&s_full[t], j & 1, flags, abort_word));
      float sc[32];
      float mb = -INFINITY;
      if (ok) {
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld32(tS + (uint32_t)(32 * half), sr);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[t]);   // S(j + 1) may now overwrite S(j)
        // only blocks reaching past the tile's first query need the causal mask (warp-uniform)
        if (j * Q2_K + Q2_K - 1 <= qp0 + Q2_T * t) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            sc[c] = __uint_as_float(sr[c]);
            mb = fmaxf(mb, sc[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int key = j * Q2_K + 32 * half + c;
            sc[c] = key <= qpos ? __uint_as_float(sr[c]) : -INFINITY;
            mb = fmaxf(mb, sc[c]);
          }
        }
      }
      red_mine(j)[r] = mb;
      named_bar(1 + t, Q2_SM_WARPS * 32);   // both halves' maxima written; both have read S
      if (!ok) continue;
      const float m_blk = fmaxf(mb, red_other(j)[r]);
      // the exponentials use the reference m_ref; it moves (and O is rescaled) only when the
      // block's maximum passes it by more than 2^8, or on the first block (key 0 is visible to
      // every row). Both threads of a row decide alike; the TMEM accesses are warp-wide, so a
      // warp rescales when any of its rows needs it (alpha = 1 for the others)
      const bool grow = m_blk > m_ref + Q2_TAU;
      const float m_new = grow ? m_blk : m_ref;
      const float alpha = grow ? ex2(m_ref - m_new) : 1.0f;   // m_ref = -inf: 0
      l_run *= alpha;
      m_ref = m_new;
      float lsum = 0.0f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        sc[c] = ex2(sc[c] - m_ref);   // masked: exp2(-inf) = 0
        lsum += sc[c];
      }
      l_run += lsum;
      if (j > 0) {
        // P(j - 1).V has read the P columns and added into O before they are rewritten or O
        // is rescaled
        ok = __all_sync(0xffffffffu, wait_ab(&pv_full[t], (j - 1) & 1, flags, abort_word));
        if (!ok) continue;
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
          uint32_t ov[32];
          tmem_ld32(tO, ov);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
          tmem_st16(tO, ov);
          tmem_st16(tO + 16, ov + 16);
        }
      }
      uint32_t ph[16], pl[16];   // P row r, keys 32 half .. + 31 as bf16 pairs
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const __nv_bfloat162 hi = __floats2bfloat162_rn(sc[2 * i], sc[2 * i + 1]);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(sc[2 * i] - __low2float(hi), sc[2 * i + 1] - __high2float(hi));
        ph[i] = *reinterpret_cast<const uint32_t*>(&hi);
        pl[i] = *reinterpret_cast<const uint32_t*>(&lo);
      }
      // P_hi in columns 16 half .., P_lo in 32 + 16 half .. of the tile's P block
      tmem_st16(tP + (uint32_t)(16 * half), ph);
      tmem_st16(tP + (uint32_t)(32 + 16 * half), pl);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    if (nkb[t] > 0) {
      // the last P.V, then the row's sum over both halves
      if (ok) ok = __all_sync(0xffffffffu, wait_ab(&pv_full[t], (nkb[t] - 1) & 1, flags, abort_word));
      float o[32];
      if (ok) {
        tc_fence_after();
        uint32_t ov[32];
        tmem_ld32(tO, ov);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] = __uint_as_float(ov[c]);
      }
      named_bar(1 + t, Q2_SM_WARPS * 32);   // every thread is done with the maxima
      red_mine(0)[r] = l_run;
      named_bar(1 + t, Q2_SM_WARPS * 32);
      if (ok && !*abort_word && r < nqt) {
        const float inv = 1.0f / (l_run + red_other(0)[r]);
        const int ld = (std::is_same<AT, Split>::value ? 2 : 1) * H * HD;
#pragma unroll
        for (int d = 0; d < 32; d += 4) {
          float y[4] = {o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv};
          act_store4<AT>(p.out, row0 + Q2_T * t + r, ld, h * HD + 32 * half + d, y);
        }
      }
    }
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Q2_TMEM_COLS);
  }
}

template <typename KT, typename AT>
cudaError_t prefill_tc2_t(const AttnPrefillParams& p, cudaStream_t s, bool pdl) {
  static bool attr_set_dev[MAX_DEVICES] = {};
  bool& attr_set = attr_set_dev[current_device()];
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(k_attn_prefill_tc2<KT, AT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Q2_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_heads, p.n_items);   // heads fastest: the items (longest first) lead
  cfg.blockDim = dim3(Q2_THREADS);
  cfg.dynamicSmemBytes = Q2_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_attn_prefill_tc2<KT, AT>, p);
}

}  // namespace

cudaError_t launch_attn_prefill_tc2(const AttnPrefillParams& p, int kv_dtype, cudaStream_t s, bool pdl) {
  if (p.n_items <= 0) return cudaSuccess;
  if (p.n_heads % p.kv.n_kv_heads != 0 || p.window != 0 || p.n_items > 65535) return cudaErrorInvalidValue;
  if (kv_dtype == DT_F32 && p.out_dtype == DT_F32) return prefill_tc2_t<float, float>(p, s, pdl);
  if (kv_dtype == DT_F32 && p.out_dtype == DT_SPLIT) return prefill_tc2_t<float, Split>(p, s, pdl);
  if (kv_dtype == DT_BF16 && p.out_dtype == DT_F32) return prefill_tc2_t<bf16, float>(p, s, pdl);
  if (kv_dtype == DT_BF16 && p.out_dtype == DT_SPLIT) return prefill_tc2_t<bf16, Split>(p, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace llm
