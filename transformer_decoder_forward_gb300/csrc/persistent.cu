// A whole decode step of a few rows in one persistent kernel.
//
// A decode step issues a few dozen dependent kernels per layer, and with a handful of
// rows each of them is over in microseconds: the GPU waits between kernels more than it
// computes ("rvllm-metal", sections "What's basic about it": about 900 dispatches a step,
// and "What's next": fusing them). Here one cooperative launch of one CTA per SM walks
// every phase of the step, with a grid-wide barrier between dependent phases:
//
//   per layer: QKV projection (LayerNorm/RMSNorm of the residual stream folded into the
//              staging of its input, bias)
//              | attention (Q/K norm, RoPE, the new token's K/V into the paged cache, causal
//                or sliding-window softmax over the cached keys, grouped queries)
//              | output projection + residual
//              | FFN up projection (norm folded in) + GELU or SwiGLU
//              | FFN down projection + residual
//   then:      final norm, tied LM head, logits (when asked) and per-CTA argmax partials.
//
// Weights never depend on an earlier phase, so they stream independently of the barriers.
// Warp 8 of every CTA walks the CTA's share of every matrix of the step in the order the
// phases consume it and copies it into a ring of shared-memory stages with 1-D TMA bulk
// copies (one mbarrier per stage for "full", one for "empty"); while the compute warps wait
// at a barrier the ring already fills with the next phases' weights. Each CTA owns a
// contiguous range of output rows of each matrix (whole K, so no split-K reduction):
// the rows' outputs are complete in the CTA and the epilogues are element-wise (SwiGLU's
// gate row j and up row d_ff + j are copied into the same stage). Activations between
// phases live in small fp32 scratch arrays in global memory (L2), read with L1-bypassing
// loads; each CTA stages a phase's whole input in shared memory.
//
// Every wait is bounded: a stage wait or a grid barrier that runs past its limit (about a
// second of SM clocks) sets LLM_FLAG_WAIT_TIMEOUT and the abort word, every CTA leaves at
// its next barrier, and the weight streamer waits (bounded) for its copies in flight
// before its CTA exits. The launch is cooperative, so all CTAs are resident together.
//
// Measured on GB300 with global-timer stamps at every phase boundary (GPT-2 124M fp32, one
// sequence): a phase costs 3-5 us. The grid barrier takes about 2 us (arrival behind the
// slowest warp, then the release reaching every CTA), staging the input from L2 about 1 us and
// the matrix work 1.4-3 us on 8 warps an SM, whose load-FMA-shuffle chains leave most issue
// slots idle; the weights themselves arrive well ahead. The 61 dependent phases take 0.39 ms,
// against 0.37 ms for one kernel a phase with programmatic launch, and the 8-row instance is
// about twice as slow again, so the library takes this path only when asked to.
#include <cuda_fp16.h>

#include <climits>
#include <type_traits>

#include "epilogue.cuh"
#include "persistent.cuh"

namespace llm {

namespace {

constexpr int CW = PK_COMPUTE_WARPS;
constexpr int CT = CW * 32;
constexpr float SM_SCALE = 0.125f;   // 1/sqrt(64)
constexpr float LOG2E = 1.4426950408889634f;

// shared-memory layout: barriers and small state | the phase's constants (bias slice, norm
// gains and biases) | this CTA's slice of the residual stream | attention scratch | weight ring |
// staged input
constexpr int PK_HDR = 1024;
constexpr int PK_BIAS_OFF = PK_HDR;                                   // [2][PK_MAX_UNITS]
constexpr int PK_SH_OFF = PK_BIAS_OFF + 2 * PK_MAX_UNITS * 4;         // [PK_MAX_M][PK_MAX_UNITS]
constexpr int PK_G_OFF = PK_SH_OFF + PK_MAX_M * PK_MAX_UNITS * 4;     // [PK_MAX_D]
constexpr int PK_B_OFF = PK_G_OFF + PK_MAX_D * 4;                     // [PK_MAX_D]
constexpr int PK_ATT_OFF = PK_B_OFF + PK_MAX_D * 4;
constexpr int PK_GPASS = 4;   // query heads scored per pass over the keys
constexpr int PK_ATT_FLOATS = PK_MAX_G * HD + 2 * HD + 2 * CW * PK_GPASS + CW * PK_GPASS * HD;
constexpr int PK_RING_OFF = PK_ATT_OFF + ((PK_ATT_FLOATS * 4 + 127) / 128) * 128;

enum { PH_QKV = 0, PH_O = 1, PH_UP = 2, PH_DOWN = 3, PH_HEAD = 4 };

// the compute warps only (warp CW streams weights and never joins)
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(CT) : "memory"); }

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Stage release by a consumer warp. The stage's data was consumed (the dot products used every
// value loaded from it) before this, so no ordering is needed; a release arrive would also wait
// for the epilogue's global stores.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ unsigned ld_volatile(const unsigned* p) { return *reinterpret_cast<const volatile unsigned*>(p); }

// Bounded stage wait that also gives up when another CTA has aborted the step. sleep_ns > 0
// backs off between polls (the weight streamer, which runs far ahead, so that its polling does
// not take issue slots from the compute warps sharing its scheduler).
__device__ bool pk_wait(uint64_t* bar, unsigned parity, unsigned* abort, unsigned* flags, unsigned sleep_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  unsigned n = 0;
  while (true) {
    if (sleep_ns) __nanosleep(sleep_ns);
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 63) == 0) {
      if (abort && ld_volatile(abort) != 0u) return false;
      if (clock64() - t0 > WAIT_CYCLES) {
        set_flag(flags, FLAG_WAIT_TIMEOUT);
        if (abort) atomicExch(abort, 1u);
        return false;
      }
    }
  }
}

// Grid-wide barrier of the compute threads, split so that work which depends on no other CTA
// (staging the next phase's constants) overlaps the wait: pk_grid_arrive adds this CTA to the
// arrival counter (release); pk_grid_wait spins, bounded, until every CTA has arrived (acquire).
// A CTA that failed a stage wait does not arrive but raises the abort word instead.
__device__ void pk_grid_arrive(const PKParams& p, volatile int* s_fail) {
  cbar();
  if (threadIdx.x == 0) {
    if (*s_fail == 0) red_release_gpu_add(p.sync, 1u);
    else atomicExch(p.sync + 1, 1u);
  }
}
// Returns false (the same in every thread of the CTA) when the step is aborted.
__device__ bool pk_grid_wait(const PKParams& p, unsigned target, volatile int* s_fail, volatile int* s_ok) {
  if (threadIdx.x == 0) {
    bool ok = *s_fail == 0;
    if (ok) {
      const long long t0 = clock64();
      unsigned n = 0;
      while (ld_acquire_gpu(p.sync) < target) {
        if ((++n & 15) == 0) {
          if (ld_volatile(p.sync + 1) != 0u) { ok = false; break; }
          if (clock64() - t0 > WAIT_CYCLES) {
            set_flag(p.flags, FLAG_WAIT_TIMEOUT);
            atomicExch(p.sync + 1, 1u);
            ok = false;
            break;
          }
        }
      }
    }
    *s_ok = ok ? 1 : 0;
  }
  cbar();
  return *s_ok != 0;
}

// ---- the weight stream ---------------------------------------------------------------------
// One matrix phase as seen by this CTA: units [u0, u1) (a unit is one output row, or for
// SwiGLU the pair gate row j / up row rows2 + j), upc units per ring stage.
struct Mat {
  const unsigned char* w;   // [rows][K] values (Q8_0: int8 quants)
  const unsigned char* s;   // Q8_0: [rows][K/32] fp16 scales, else nullptr
  int K, rows2, u0, u1, upc, rb, sb;
};

template <typename WT>
__device__ __forceinline__ Mat pk_mat(const PKParams& p, const PKLayer& L, int ph) {
  using ST = typename Elem<WT>::type;
  constexpr bool Q8W = std::is_same<WT, Q8>::value;
  const void *w, *s;
  int K, units, rows2 = 0;
  switch (ph) {
    case PH_QKV: w = L.w_qkv; s = L.s_qkv; K = p.d; units = (p.H + 2 * p.Hkv) * HD; break;
    case PH_O: w = L.w_o; s = L.s_o; K = p.H * HD; units = p.d; break;
    case PH_UP: w = L.w_up; s = L.s_up; K = p.d; units = p.F; rows2 = p.gpt2 ? 0 : p.F; break;
    case PH_DOWN: w = L.w_down; s = L.s_down; K = p.F; units = p.d; break;
    default: w = p.tok_emb; s = p.tok_scale; K = p.d; units = p.vocab; break;
  }
  Mat m;
  m.w = static_cast<const unsigned char*>(w);
  m.s = static_cast<const unsigned char*>(s);
  m.K = K;
  m.rows2 = rows2;
  m.rb = K * (int)sizeof(ST);
  m.sb = Q8W ? K / Q8_BLOCK * 2 : 0;
  m.upc = PK_SLOT_BYTES / ((rows2 ? 2 : 1) * (m.rb + m.sb));
  m.u0 = (int)((long long)units * blockIdx.x / gridDim.x);
  m.u1 = (int)((long long)units * (blockIdx.x + 1) / gridDim.x);
  return m;
}

// Stage layout of a chunk of U units: [rows A: U rb][rows B: U rb][scales A: U sb][scales B: U sb].
template <typename WT>
__device__ void pk_produce(const PKParams& p, unsigned char* ring, uint64_t* full, uint64_t* empty) {
  unsigned* abort = p.sync + 1;
  const int ns = p.nslot;
  int seq = 0;   // chunks issued
  bool ok = true;
  for (int q = 0; q <= 4 * p.n_layers && ok; ++q) {
    const bool head = q == 4 * p.n_layers;
    const Mat m = pk_mat<WT>(p, p.layers[head ? 0 : q / 4], head ? PH_HEAD : q % 4);
    const int segs = m.rows2 ? 2 : 1;
    for (int ua = m.u0; ua < m.u1; ua += m.upc) {
      const int U = min(m.upc, m.u1 - ua);
      const int slot = seq % ns;
      if (seq >= ns && !pk_wait(&empty[slot], (unsigned)((seq / ns - 1) & 1), abort, p.flags, 256)) {
        ok = false;
        break;
      }
      fence_async_smem();   // the consumers' reads of the stage before the copy overwrites it
      unsigned char* dst = ring + (size_t)slot * PK_SLOT_BYTES;
      const unsigned wb = (unsigned)U * m.rb, sbb = (unsigned)U * m.sb;
      mbar_arrive_expect_tx(&full[slot], segs * (wb + sbb));
      bulk_g2s(dst, m.w + (size_t)ua * m.rb, wb, &full[slot]);
      if (m.rows2) bulk_g2s(dst + wb, m.w + (size_t)(m.rows2 + ua) * m.rb, wb, &full[slot]);
      if (m.sb) {
        bulk_g2s(dst + segs * wb, m.s + (size_t)ua * m.sb, sbb, &full[slot]);
        if (m.rows2) bulk_g2s(dst + segs * wb + sbb, m.s + (size_t)(m.rows2 + ua) * m.sb, sbb, &full[slot]);
      }
      ++seq;
    }
  }
  // the copies still in flight (at most the last issued chunk of each stage) must land
  // before the CTA may exit; normally the consumers have already seen them all
  for (int s = seq > ns ? seq - ns : 0; s < seq; ++s) mbar_wait(&full[s % ns], (unsigned)((s / ns) & 1), p.flags);
}

// ---- the compute warps --------------------------------------------------------------------
// The constants of matrix phase ph of layer l, into shared memory: the bias of this CTA's
// units (s_bias[0..], SwiGLU's up rows at s_bias[PK_MAX_UNITS..]) and, for the phases whose
// input is a norm of the residual stream, the norm's gains and biases as fp32. Weights only,
// which no CTA writes, so this runs while the CTA waits at a grid barrier; every load is
// issued before the first store.
template <typename WT>
__device__ void pk_stage(const PKParams& p, int l, int ph, float* s_bias, float* s_g, float* s_b, PKLayer* s_L) {
  const PKLayer& L = p.layers[ph == PH_HEAD ? 0 : l];
  if (ph == PH_QKV) {   // the layer's table entry, read by every phase of the layer
    static_assert(sizeof(PKLayer) % 4 == 0 && sizeof(PKLayer) <= 256, "layer entry");
    const int t = threadIdx.x;
    if (t < (int)(sizeof(PKLayer) / 4))
      reinterpret_cast<unsigned*>(s_L)[t] = reinterpret_cast<const unsigned*>(&L)[t];
  }
  const void *bias = nullptr, *g = nullptr, *b = nullptr;
  int units = 0, rows2 = 0;
  switch (ph) {
    case PH_QKV: bias = L.b_qkv; g = L.ln1_g; b = L.ln1_b; units = (p.H + 2 * p.Hkv) * HD; break;
    case PH_O: bias = L.b_o; units = p.d; break;
    case PH_UP: bias = L.b_up; g = L.ln2_g; b = L.ln2_b; units = p.F; rows2 = p.gpt2 ? 0 : p.F; break;
    case PH_DOWN: bias = L.b_down; units = p.d; break;
    default: g = p.lnf_g; b = p.lnf_b; break;
  }
  const int u0 = (int)((long long)units * blockIdx.x / gridDim.x);
  const int nu = (int)((long long)units * (blockIdx.x + 1) / gridDim.x) - u0;
  const int t = threadIdx.x;
  constexpr int NG = PK_MAX_D / CT;
  float gv[NG], bv[NG], bias_v = 0.0f;
  if (t < nu) bias_v = bias_at<WT>(bias, u0 + t);
  else if (rows2 && t >= PK_MAX_UNITS && t - PK_MAX_UNITS < nu) bias_v = bias_at<WT>(bias, rows2 + u0 + t - PK_MAX_UNITS);
#pragma unroll
  for (int j = 0; j < NG; ++j) {
    const int k = t + j * CT;
    gv[j] = (g && k < p.d) ? bias_at<WT>(g, k) : 0.0f;
    bv[j] = (g && k < p.d) ? bias_at<WT>(b, k) : 0.0f;
  }
  if (t < nu || (rows2 && t >= PK_MAX_UNITS && t - PK_MAX_UNITS < nu)) s_bias[t] = bias_v;
  if (g) {
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      const int k = t + j * CT;
      if (k < p.d) {
        s_g[k] = gv[j];
        s_b[k] = bv[j];
      }
    }
  }
}


// Two rows' dot products with the staged input rows: y0[m] = w0 . x[m], y1[m] = w1 . x[m]
// (all lanes get the sums). 16-byte weight vectors: 4 fp32, 8 bf16 or 16 Q8_0 quants (half
// a block, one scale).
template <typename WT, int MT>
__device__ __forceinline__ void pk_dot2(const unsigned char* r0, const unsigned char* s0, const unsigned char* r1,
                                        const unsigned char* s1, bool two, const float* xs, int K, int vb, int ve,
                                        int M, float (&y0)[MT], float (&y1)[MT]) {
  constexpr int VEC = Vec16<WT>::N;
  constexpr bool Q8W = std::is_same<WT, Q8>::value;
  constexpr int UN = 4;   // weight vectors in flight per lane and row: their loads issue together
  const int lane = threadIdx.x & 31;
  float a0[MT], a1[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) a0[m] = a1[m] = 0.0f;
  // 16-byte vectors vb..ve-1 of the rows (the whole row, or one warp's part of it)
  for (int v0 = vb + lane; v0 < ve; v0 += 32 * UN) {
    uint4 w0[UN], w1[UN];
    float d0[UN], d1[UN];
#pragma unroll
    for (int j = 0; j < UN; ++j) {
      const int v = v0 + 32 * j;
      const bool in = v < ve;
      w0[j] = in ? *reinterpret_cast<const uint4*>(r0 + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
      w1[j] = (in && two) ? *reinterpret_cast<const uint4*>(r1 + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
      d0[j] = d1[j] = 1.0f;
      if constexpr (Q8W) {
        d0[j] = in ? __half2float(reinterpret_cast<const __half*>(s0)[v * VEC / Q8_BLOCK]) : 0.0f;
        d1[j] = (in && two) ? __half2float(reinterpret_cast<const __half*>(s1)[v * VEC / Q8_BLOCK]) : 0.0f;
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < M) {
        float p0[UN], p1[UN];
#pragma unroll
        for (int j = 0; j < UN; ++j) {
          const int v = min(v0 + 32 * j, ve - 1);   // a lane past the end multiplies zero weights
          const float* xr = xs + (size_t)m * K + v * VEC;
          float f0[VEC], f1[VEC];
          Vec16<WT>::unpack(w0[j], f0);
          Vec16<WT>::unpack(w1[j], f1);
          float s0v = 0.0f, s1v = 0.0f;
#pragma unroll
          for (int e = 0; e < VEC; e += 4) {
            const float4 x = *reinterpret_cast<const float4*>(xr + e);
            s0v = fmaf(f0[e], x.x, s0v); s0v = fmaf(f0[e + 1], x.y, s0v);
            s0v = fmaf(f0[e + 2], x.z, s0v); s0v = fmaf(f0[e + 3], x.w, s0v);
            s1v = fmaf(f1[e], x.x, s1v); s1v = fmaf(f1[e + 1], x.y, s1v);
            s1v = fmaf(f1[e + 2], x.z, s1v); s1v = fmaf(f1[e + 3], x.w, s1v);
          }
          p0[j] = d0[j] * s0v;
          p1[j] = d1[j] * s1v;
        }
        a0[m] += (p0[0] + p0[1]) + (p0[2] + p0[3]);
        a1[m] += (p1[0] + p1[1]) + (p1[2] + p1[3]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    y0[m] = m < M ? warp_sum(a0[m]) : 0.0f;
    y1[m] = (m < M && two) ? warp_sum(a1[m]) : 0.0f;
  }
}

// One matrix phase: consume this CTA's chunks from the ring, write the element-wise epilogue.
// Lane m writes row m's outputs. A failed stage wait marks the CTA (s_fail) and skips the
// remaining work; the phase's grid barrier then aborts the step in every CTA.
template <typename WT, int MT>
__device__ void pk_matrix(const PKParams& p, const Mat& mt, int ph, const PKLayer& L, unsigned char* ring,
                          uint64_t* full, uint64_t* empty, int& seq, const float* xs, int M,
                          volatile int* s_fail, const float* s_bias, float* s_h, float* s_red2, int& nsplit,
                          float (&best)[MT], int (&bi)[MT]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const StepArgs* a = p.args;
  bool failed = *s_fail != 0;
  const int segs = mt.rows2 ? 2 : 1;
  const int upi = mt.rows2 ? 1 : 2;   // units per work item: two rows either way
  const int QN = (p.H + 2 * p.Hkv) * HD;
  float* logits = ph == PH_HEAD ? a->logits : nullptr;
  for (int ua = mt.u0; ua < mt.u1; ua += mt.upc, ++seq) {
    const int U = min(mt.upc, mt.u1 - ua);
    const int slot = seq % p.nslot;
    if (!failed) {
      failed = !__all_sync(0xffffffffu, pk_wait(&full[slot], (unsigned)((seq / p.nslot) & 1), p.sync + 1, p.flags));
      if (failed && lane == 0) *s_fail = 1;
    }
    const unsigned char* base = ring + (size_t)slot * PK_SLOT_BYTES;
    const size_t wb = (size_t)U * mt.rb;
    constexpr int VEC = Vec16<WT>::N;
    const int nv = mt.K / VEC;
    // Work items are row pairs (two one-row units, or one SwiGLU unit). With fewer pairs than
    // half the warps, S warps share a pair, each taking a part of K; the partial sums meet in
    // shared memory (double-buffered) and the pair's first warp adds them in warp order. Every
    // warp passes the chunk's barrier, also after a failed wait.
    const int npairs = (U + upi - 1) / upi;
    int S = 1;
    while (S < CW && 2 * S * npairs <= CW) S *= 2;
    const int pair = warp / S, part = warp - pair * S;
    auto run_pair = [&](int i, int vb, int ve, float (&y0)[MT], float (&y1)[MT]) -> bool {
      const bool two = mt.rows2 ? true : i + 1 < U;
      const unsigned char* r0 = base + (size_t)i * mt.rb;
      const unsigned char* s0 = base + segs * wb + (size_t)i * mt.sb;
      const unsigned char* r1 = mt.rows2 ? r0 + wb : r0 + mt.rb;
      const unsigned char* s1 = mt.rows2 ? s0 + (size_t)U * mt.sb : s0 + mt.sb;
      pk_dot2<WT, MT>(r0, s0, r1, s1, two, xs, mt.K, vb, ve, M, y0, y1);
      return two;
    };
    auto epilogue = [&](int i, bool two, const float (&y0)[MT], const float (&y1)[MT]) {
      const int u = ua + i;
      switch (ph) {
        case PH_QKV: {
          const float b0 = s_bias[u - mt.u0], b1 = two ? s_bias[u + 1 - mt.u0] : 0.0f;
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (m < M && lane == m) {
              p.qkv[(size_t)m * QN + u] = y0[m] + b0;
              if (two) p.qkv[(size_t)m * QN + u + 1] = y1[m] + b1;
            }
          break;
        }
        case PH_O:
        case PH_DOWN: {
          // the residual stream: this CTA owns units u0..u1 of it in every phase, so its copy in
          // shared memory is current; the global copy is what the other CTAs read
          const int i0 = u - mt.u0;
          const float b0 = s_bias[i0], b1 = two ? s_bias[i0 + 1] : 0.0f;
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (m < M && lane == m) {
              float* sh = s_h + m * PK_MAX_UNITS + i0;
              float* hr = p.h + (size_t)m * p.d + u;
              const float h0 = sh[0] + (y0[m] + b0);
              sh[0] = h0;
              hr[0] = h0;
              if (two) {
                const float h1 = sh[1] + (y1[m] + b1);
                sh[1] = h1;
                hr[1] = h1;
              }
            }
          break;
        }
        case PH_UP: {
          if (mt.rows2) {
            const float bg = s_bias[u - mt.u0], bu = s_bias[PK_MAX_UNITS + u - mt.u0];
#pragma unroll
            for (int m = 0; m < MT; ++m)
              if (m < M && lane == m) p.ff[(size_t)m * p.F + u] = silu_f(y0[m] + bg) * (y1[m] + bu);
          } else {
            const float b0 = s_bias[u - mt.u0], b1 = two ? s_bias[u + 1 - mt.u0] : 0.0f;
#pragma unroll
            for (int m = 0; m < MT; ++m)
              if (m < M && lane == m) {
                p.ff[(size_t)m * p.F + u] = gelu_tanh_clamped(y0[m] + b0);
                if (two) p.ff[(size_t)m * p.F + u + 1] = gelu_tanh_clamped(y1[m] + b1);
              }
          }
          break;
        }
        default: {   // PH_HEAD
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (m < M && lane == m) {
              if (logits) {
                logits[(size_t)m * p.vocab + u] = y0[m];
                if (two) logits[(size_t)m * p.vocab + u + 1] = y1[m];
              }
              if (argmax_better(y0[m], u, best[m], bi[m])) { best[m] = y0[m]; bi[m] = u; }
              if (two && argmax_better(y1[m], u + 1, best[m], bi[m])) { best[m] = y1[m]; bi[m] = u + 1; }
            }
          break;
        }
      }
    };
    if (S == 1) {
      if (!failed)
        for (int i = warp * upi; i < U; i += CW * upi) {
          float y0[MT], y1[MT];
          const bool two = run_pair(i, 0, nv, y0, y1);
          epilogue(i, two, y0, y1);
        }
    } else {
      float* red = s_red2 + (nsplit & 1) * (CW * 2 * PK_MAX_M);   // [CW][2][PK_MAX_M]
      ++nsplit;
      const int per = (nv + S - 1) / S;
      const int i = pair * upi;
      bool two = false;
      if (!failed && i < U) {
        float y0[MT], y1[MT];
        two = run_pair(i, min(nv, part * per), min(nv, (part + 1) * per), y0, y1);
        if (lane == 0) {
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            red[(warp * 2) * PK_MAX_M + m] = y0[m];
            red[(warp * 2 + 1) * PK_MAX_M + m] = y1[m];
          }
        }
      }
      cbar();
      if (!failed && i < U && part == 0) {
        float y0[MT], y1[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          y0[m] = y1[m] = 0.0f;
          for (int q = 0; q < S; ++q) {
            y0[m] += red[((warp + q) * 2) * PK_MAX_M + m];
            y1[m] += red[((warp + q) * 2 + 1) * PK_MAX_M + m];
          }
        }
        epilogue(i, two, y0, y1);
      }
    }
    if (failed) continue;
    __syncwarp();
    if (lane == 0) mbar_arrive_relaxed(&empty[slot]);
  }
}

// Layer 0: the embedding rows (token, plus the learned position for GPT-2) into xs; this CTA
// also stores its slice of them as the residual stream (global and shared copies). Loads are
// issued in batches before their stores.
template <typename WT>
__device__ void pk_embed(const PKParams& p, float* xs, int M, float* s_h) {
  using ST = typename Elem<WT>::type;
  using VT = typename VecT<WT>::type;
  const int d = p.d, n = M * d;
  const StepArgs* a = p.args;
  if (blockIdx.x == 0 && (int)threadIdx.x < M) {
    const int tok = a->tokens[threadIdx.x], pos = a->positions[threadIdx.x];
    if (tok < 0 || tok >= p.vocab) set_flag(p.flags, FLAG_BAD_TOKEN);
    if (pos < 0 || pos >= p.n_ctx) set_flag(p.flags, FLAG_BAD_POSITION);
  }
  const int h0 = (int)((long long)d * blockIdx.x / gridDim.x), h1 = (int)((long long)d * (blockIdx.x + 1) / gridDim.x);
  constexpr int NB = 8;
  for (int base = threadIdx.x; base < n; base += CT * NB) {
    float v[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int i = base + j * CT;
      v[j] = 0.0f;
      if (i < n) {
        const int m = i / d, k = i - m * d;
        const int tok = a->tokens[m], pos = a->positions[m];
        if (tok >= 0 && tok < p.vocab) {
          const size_t e = (size_t)tok * d + k;
          if constexpr (std::is_same<WT, Q8>::value)
            v[j] = (float)reinterpret_cast<const int8_t*>(p.tok_emb)[e] *
                   __half2float(reinterpret_cast<const __half*>(p.tok_scale)[e / Q8_BLOCK]);
          else
            v[j] = to_f32(reinterpret_cast<const ST*>(p.tok_emb)[e]);
        }
        if (p.pos_emb && pos >= 0 && pos < p.n_ctx) v[j] += to_f32(reinterpret_cast<const VT*>(p.pos_emb)[(size_t)pos * d + k]);
      }
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int i = base + j * CT;
      if (i < n) {
        const int m = i / d, k = i - m * d;
        xs[i] = v[j];
        if (k >= h0 && k < h1) {
          p.h[i] = v[j];
          s_h[m * PK_MAX_UNITS + k - h0] = v[j];
        }
      }
    }
  }
}

// xs[m][0..d) = Norm(h[m]) for m < M. The rows are copied into shared memory asynchronously
// (through L2: other CTAs wrote them); every thread then takes a slice of every row: the sums
// of x and of (x - mean)^2 are reduced over the warp, then over the warps in warp order, and
// the staged gains and biases are applied (LayerNorm for GPT-2, RMSNorm with zero biases
// otherwise). Layer 0 normalises the embedding instead. s_red: [CW][PK_MAX_M] scratch.
template <typename WT>
__device__ void pk_prep_norm(const PKParams& p, float* xs, int M, const float* s_g, const float* s_b, bool embed,
                             float* s_h, float* s_red, float* s_stat) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, d = p.d;
  if (embed) {
    pk_embed<WT>(p, xs, M, s_h);
  } else {
    for (int i = threadIdx.x; i < M * d / 4; i += CT) cp_async16(xs + 4 * i, p.h + 4 * i);
    cp_async_commit();
    cp_async_wait_all();
  }
  cbar();
  const int d4 = d / 4;
  // mean (LayerNorm only)
  if (p.gpt2) {
    for (int m = 0; m < M; ++m) {
      const float4* x4 = reinterpret_cast<const float4*>(xs + (size_t)m * d);
      float sum = 0.0f;
      for (int i = threadIdx.x; i < d4; i += CT) {
        const float4 v = x4[i];
        sum += (v.x + v.y) + (v.z + v.w);
      }
      sum = warp_sum(sum);
      if (lane == 0) s_red[warp * PK_MAX_M + m] = sum;
    }
    cbar();
    if ((int)threadIdx.x < M) {
      float sum = 0.0f;
      for (int w = 0; w < CW; ++w) sum += s_red[w * PK_MAX_M + threadIdx.x];
      s_stat[threadIdx.x] = sum / d;
    }
    cbar();
  }
  for (int m = 0; m < M; ++m) {
    const float mean = p.gpt2 ? s_stat[m] : 0.0f;
    const float4* x4 = reinterpret_cast<const float4*>(xs + (size_t)m * d);
    float sq = 0.0f;
    for (int i = threadIdx.x; i < d4; i += CT) {
      const float4 v = x4[i];
      const float a0 = v.x - mean, a1 = v.y - mean, a2 = v.z - mean, a3 = v.w - mean;
      sq += (a0 * a0 + a1 * a1) + (a2 * a2 + a3 * a3);
    }
    sq = warp_sum(sq);
    if (lane == 0) s_red[warp * PK_MAX_M + m] = sq;
  }
  cbar();
  if ((int)threadIdx.x < M) {
    float sq = 0.0f;
    for (int w = 0; w < CW; ++w) sq += s_red[w * PK_MAX_M + threadIdx.x];
    s_stat[PK_MAX_M + threadIdx.x] = 1.0f / sqrtf(sq / d + p.eps);
  }
  cbar();
  for (int i = threadIdx.x; i < M * d; i += CT) {
    const int m = i / d, k = i - m * d;
    const float mean = p.gpt2 ? s_stat[m] : 0.0f;
    xs[i] = norm_apply(xs[i], mean, s_stat[PK_MAX_M + m], s_g[k], s_b[k]);
  }
}

// Attention items of a row: the visible keys lo..pos cut into PK_ATT_CH-key chunks.
__device__ __forceinline__ int pk_nch(const PKParams& p, int window, int pos) {
  const int ctx = pos + 1;
  if (ctx <= 0) return 0;
  const int lo = window > 0 ? max(0, ctx - window) : 0;
  return min(p.max_ch, (ctx - lo + PK_ATT_CH - 1) / PK_ATT_CH);
}

// xs[m][h*64 + d] = the attention output: copied (rows whose context was one item) or the
// items merged to the common maximum (log2 units, in item order).
__device__ void pk_prep_att(const PKParams& p, float* xs, int M, int window) {
  const int HH = p.H * HD;
  for (int i = threadIdx.x; i < M * HH / 4; i += CT)
    if (pk_nch(p, window, p.args->positions[4 * i / HH]) == 1) cp_async16(xs + 4 * i, p.att + 4 * i);
  cp_async_commit();
  for (int i = threadIdx.x; i < M * HH; i += CT) {
    const int m = i / HH, hd = i - m * HH, hh = hd / HD, dd = hd - hh * HD;
    const int nch = pk_nch(p, window, p.args->positions[m]);
    if (nch == 1) continue;
    float x = 0.0f;
    if (nch > 1) {
      const size_t base = ((size_t)m * p.H + hh) * p.max_ch;
      float mx = -INFINITY;
      for (int c = 0; c < nch; ++c) mx = fmaxf(mx, __ldcg(p.part_ml + (base + c) * 2));
      float ls = 0.0f, os = 0.0f;
      for (int c = 0; c < nch; ++c) {
        const float mc = __ldcg(p.part_ml + (base + c) * 2);
        const float w = mc == -INFINITY ? 0.0f : exp2f(mc - mx);
        ls = fmaf(w, __ldcg(p.part_ml + (base + c) * 2 + 1), ls);
        os = fmaf(w, __ldcg(p.part_o + (base + c) * HD + dd), os);
      }
      x = ls > 0.0f ? os / ls : 0.0f;
    }
    xs[i] = x;
  }
  cp_async_wait_all();
}

__device__ void pk_prep_copy(float* xs, const float* src, int n) {
  for (int i = threadIdx.x; i < n / 4; i += CT) cp_async16(xs + 4 * i, src + 4 * i);
  cp_async_commit();
  cp_async_wait_all();
}

// Eight values of one K or V row for lane dg: dims 4dg..4dg+3 and 32+4dg..+3 (fp32 rows) or
// 8dg..8dg+7 (bf16 rows).
__device__ __forceinline__ int pk_dim(int dg, int e, bool f32) {
  return f32 ? (e < 4 ? 4 * dg + e : 32 + 4 * dg + (e - 4)) : 8 * dg + e;
}
template <typename KT> __device__ __forceinline__ void pk_row8(const KT* row, int dg, float* f);
template <> __device__ __forceinline__ void pk_row8<float>(const float* row, int dg, float* f) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(row + 4 * dg));
  const float4 c = __ldg(reinterpret_cast<const float4*>(row + 32 + 4 * dg));
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
}
template <> __device__ __forceinline__ void pk_row8<bf16>(const bf16* row, int dg, float* f) {
  Vec16<bf16>::unpack(ldg16(row + 8 * dg), f);
}

// The attention phase: work items (row m, KV head g, chunk c) dealt to the CTAs in turn.
// The item holding the new token writes its K/V into the cache (keys older than it were
// written by earlier steps and are read through the read-only path); the new key and value
// themselves come from shared memory. Eight lanes hold a key row, a warp scores four keys a
// step for every query head of the group; online softmax in log2 units per warp, warps
// merged in shared memory.
template <typename WT, typename KT>
__device__ void pk_attention(const PKParams& p, const PKLayer& L, float* sa, int M) {
  constexpr bool F32K = std::is_same<KT, float>::value;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, dg = lane & 7, tg = lane >> 3;
  const int H = p.H, Hkv = p.Hkv, Gq = H / Hkv, QN = (H + 2 * Hkv) * HD;
  float* sq = sa;                       // [PK_MAX_G][64] scaled queries
  float* snew = sq + PK_MAX_G * HD;     // [2][64] the new token's key and value
  float* s_m = snew + 2 * HD;           // [CW][PK_GPASS]
  float* s_l = s_m + CW * PK_GPASS;     // [CW][PK_GPASS]
  float* s_o = s_l + CW * PK_GPASS;     // [CW][PK_GPASS][64]
  const StepArgs* a = p.args;
  const KT* kb = reinterpret_cast<const KT*>(L.kv.k);
  const KT* vb = reinterpret_cast<const KT*>(L.kv.v);
  int total = 0;
  for (int m = 0; m < M; ++m) total += Hkv * pk_nch(p, L.window, a->positions[m]);
  for (int it = blockIdx.x; it < total; it += gridDim.x) {
    int m = 0, r = it, nch = 0;
    for (; m < M; ++m) {
      nch = pk_nch(p, L.window, a->positions[m]);
      if (r < Hkv * nch) break;
      r -= Hkv * nch;
    }
    const int g = r / nch, c = r - g * nch;
    const int pos = a->positions[m], ctx = pos + 1;
    const int lo = L.window > 0 ? max(0, ctx - L.window) : 0;
    const int t0 = lo + c * PK_ATT_CH, t1 = min(ctx, t0 + PK_ATT_CH);
    const bool has_new = t1 == ctx;

    // queries of the group, and the new token's key and value (Q/K norm, then RoPE)
    for (int job = warp; job < Gq + 2; job += CW) {
      if (job >= Gq && !has_new) continue;
      const int col = job < Gq ? (g * Gq + job) * HD : job == Gq ? (H + g) * HD : (H + Hkv + g) * HD;
      const float* src = p.qkv + (size_t)m * QN + col;
      float x0 = __ldcg(src + lane), x1 = __ldcg(src + lane + 32);
      if (job <= Gq) {
        if (L.qn_g) {
          const float ss = warp_sum(x0 * x0 + x1 * x1);
          const float rr = 1.0f / sqrtf(ss / HD + p.eps);
          const void* gw = job < Gq ? L.qn_g : L.kn_g;
          x0 = x0 * rr * bias_at<WT>(gw, lane);
          x1 = x1 * rr * bias_at<WT>(gw, lane + 32);
        }
        if (!p.gpt2) {
          float sn, co;
          rope_sincos(pos, p.rope_tab[lane], &sn, &co);
          const float r0 = x0 * co - x1 * sn, r1 = x1 * co + x0 * sn;
          x0 = r0;
          x1 = r1;
        }
      }
      if (job < Gq) {
        sq[job * HD + lane] = x0 * (SM_SCALE * LOG2E);
        sq[job * HD + lane + 32] = x1 * (SM_SCALE * LOG2E);
      } else {
        if constexpr (!F32K) {   // the cache holds them rounded; this step scores the rounded values too
          x0 = __bfloat162float(__float2bfloat16_rn(x0));
          x1 = __bfloat162float(__float2bfloat16_rn(x1));
        }
        snew[(job - Gq) * HD + lane] = x0;
        snew[(job - Gq) * HD + lane + 32] = x1;
        const int pb = kv_block(L.kv, a->block_tables, m, pos, p.flags);
        if (pb >= 0) {
          KT* dst = reinterpret_cast<KT*>(job == Gq ? L.kv.k : L.kv.v) + kv_offset(L.kv, pb, g, pos & (KVB - 1));
          dst[lane] = from_f32<KT>(x0);
          dst[lane + 32] = from_f32<KT>(x1);
        }
      }
    }
    cbar();

    // query heads in passes of up to PK_GPASS: registers hold each pass's running outputs,
    // the queries stay in shared memory (read per key step)
    for (int j0 = 0; j0 < Gq; j0 += PK_GPASS) {
      const int gn = min(PK_GPASS, Gq - j0);
      float mx[PK_GPASS], ls[PK_GPASS], o[PK_GPASS][8];
#pragma unroll
      for (int j = 0; j < PK_GPASS; ++j) {
        mx[j] = -INFINITY;
        ls[j] = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[j][e] = 0.0f;
      }
      auto fetch = [&](int t, float* kf, float* vf) -> bool {
        if (t >= t1) return false;
        if (t == pos) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            kf[e] = snew[pk_dim(dg, e, F32K)];
            vf[e] = snew[HD + pk_dim(dg, e, F32K)];
          }
          return true;
        }
        const int pb = kv_block(L.kv, a->block_tables, m, t, p.flags);
        if (pb < 0) return false;
        const size_t off = kv_offset(L.kv, pb, g, t & (KVB - 1));
        pk_row8<KT>(kb + off, dg, kf);
        pk_row8<KT>(vb + off, dg, vf);
        return true;
      };
      auto step = [&](const float* kf, const float* vf, bool have) {
#pragma unroll
        for (int j = 0; j < PK_GPASS; ++j) {
          if (j >= gn) continue;
          const float* qj = sq + (j0 + j) * HD;
          float dd = 0.0f;
#pragma unroll
          for (int e = 0; e < 8; ++e) dd = fmaf(kf[e], qj[pk_dim(dg, e, F32K)], dd);
          dd += __shfl_xor_sync(0xffffffffu, dd, 4);
          dd += __shfl_xor_sync(0xffffffffu, dd, 2);
          dd += __shfl_xor_sync(0xffffffffu, dd, 1);
          const float sc = have ? dd : -INFINITY;
          float mb = fmaxf(sc, __shfl_xor_sync(0xffffffffu, sc, 8));
          mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
          if (mb > mx[j]) {   // warp-uniform
            const float alpha = exp2f(mx[j] - mb);
            mx[j] = mb;
            ls[j] *= alpha;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[j][e] *= alpha;
          }
          const float pr = have ? exp2f(sc - mx[j]) : 0.0f;
          ls[j] += pr;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[j][e] = fmaf(pr, vf[e], o[j][e]);
        }
      };
      // two key steps' loads in flight before either is scored
      for (int t = t0 + warp * 4 + tg; t - tg < t1; t += 2 * CW * 4) {
        float ka[8], va[8], kc[8], vc[8];
        const bool ha = fetch(t, ka, va);
        const bool hc = fetch(t + CW * 4, kc, vc);
        if (!ha) {
#pragma unroll
          for (int e = 0; e < 8; ++e) ka[e] = va[e] = 0.0f;
        }
        if (!hc) {
#pragma unroll
          for (int e = 0; e < 8; ++e) kc[e] = vc[e] = 0.0f;
        }
        step(ka, va, ha);
        step(kc, vc, hc);
      }
      // merge: the four key rows of the warp, then the warps
#pragma unroll
      for (int j = 0; j < PK_GPASS; ++j) {
#pragma unroll
        for (int x = 8; x < 32; x <<= 1) {
          ls[j] += __shfl_xor_sync(0xffffffffu, ls[j], x);
#pragma unroll
          for (int e = 0; e < 8; ++e) o[j][e] += __shfl_xor_sync(0xffffffffu, o[j][e], x);
        }
      }
      if (tg == 0) {
#pragma unroll
        for (int j = 0; j < PK_GPASS; ++j) {
          if (j >= gn) continue;
          if (dg == 0) {
            s_m[warp * PK_GPASS + j] = mx[j];
            s_l[warp * PK_GPASS + j] = ls[j];
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) s_o[(warp * PK_GPASS + j) * HD + pk_dim(dg, e, F32K)] = o[j][e];
        }
      }
      cbar();
      for (int i = threadIdx.x; i < gn * HD; i += CT) {
        const int j = i / HD, dd = i - j * HD;
        float gm = -INFINITY;
#pragma unroll
        for (int w = 0; w < CW; ++w) gm = fmaxf(gm, s_m[w * PK_GPASS + j]);
        float gl = 0.0f, go = 0.0f;
#pragma unroll
        for (int w = 0; w < CW; ++w) {
          const float mw = s_m[w * PK_GPASS + j];
          const float cw = mw == -INFINITY ? 0.0f : exp2f(mw - gm);
          gl = fmaf(cw, s_l[w * PK_GPASS + j], gl);
          go = fmaf(cw, s_o[(w * PK_GPASS + j) * HD + dd], go);
        }
        const int hh = g * Gq + j0 + j;
        if (nch == 1) {
          p.att[(size_t)m * H * HD + hh * HD + dd] = gl > 0.0f ? go / gl : 0.0f;
        } else {
          const size_t hs = ((size_t)m * H + hh) * p.max_ch + c;
          p.part_o[hs * HD + dd] = go;
          if (dd == 0) {
            p.part_ml[hs * 2] = gm;
            p.part_ml[hs * 2 + 1] = gl;
          }
        }
      }
      cbar();   // s_m, s_l, s_o are reused by the next pass
    }
    cbar();   // the scratch is reused by the next item
  }
}

template <typename WT, int MT>
__global__ void __launch_bounds__(PK_THREADS, 1) k_decode_persistent(const PKParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + PK_MAX_SLOTS;
  volatile int* s_fail = reinterpret_cast<volatile int*>(smem + 128);
  volatile int* s_ok = s_fail + 1;
  float* s_best = reinterpret_cast<float*>(smem + 256);              // [CW][PK_MAX_M]
  float* s_red = s_best;                                              // norm partial sums (before the head combine)
  float* s_stat = reinterpret_cast<float*>(smem + 192);               // [2][PK_MAX_M]: mean, rstd
  int* s_bi = reinterpret_cast<int*>(smem + 256 + CW * PK_MAX_M * 4);  // [CW][PK_MAX_M]
  PKLayer* s_L = reinterpret_cast<PKLayer*>(smem + 768);          // the current layer's table entry
  float* s_bias = reinterpret_cast<float*>(smem + PK_BIAS_OFF);
  float* s_h = reinterpret_cast<float*>(smem + PK_SH_OFF);
  float* s_g = reinterpret_cast<float*>(smem + PK_G_OFF);
  float* s_b = reinterpret_cast<float*>(smem + PK_B_OFF);
  float* sa = reinterpret_cast<float*>(smem + PK_ATT_OFF);
  unsigned char* ring = smem + PK_RING_OFF;
  float* xs = reinterpret_cast<float*>(ring + (size_t)p.nslot * PK_SLOT_BYTES);
  if ((int)blockIdx.x == p.withhold) return;   // self-test: this CTA never arrives
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.nslot; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], CW);
    }
    *s_fail = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (warp == CW) {
    if (lane == 0) pk_produce<WT>(p, ring, full, empty);
    return;
  }
  if (p.withhold >= 0) {   // self-test: the first barrier runs out, the weight streamer drains
    pk_grid_arrive(p, s_fail);
    pk_grid_wait(p, gridDim.x, s_fail, s_ok);
    return;
  }

  const int M = p.args->M;
  int seq = 0, nsplit = 0;
  unsigned nbar = 0;
  const unsigned G = gridDim.x;
  float best[MT];
  int bi[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    best[m] = -INFINITY;
    bi[m] = INT_MAX;
  }
  // Each grid barrier: arrive, stage the next phase's constants, wait.
  bool ok = true;
  pk_stage<WT>(p, 0, PH_QKV, s_bias, s_g, s_b, s_L);
  cbar();
  for (int l = 0; l < p.n_layers; ++l) {
    const PKLayer& L = *s_L;
    pk_prep_norm<WT>(p, xs, M, s_g, s_b, l == 0, s_h, s_red, s_stat);
    cbar();
    pk_matrix<WT, MT>(p, pk_mat<WT>(p, L, PH_QKV), PH_QKV, L, ring, full, empty, seq, xs, M, s_fail, s_bias, s_h, sa, nsplit, best, bi);
    pk_grid_arrive(p, s_fail);
    if (!(ok = pk_grid_wait(p, ++nbar * G, s_fail, s_ok))) break;
    if (L.kv.dtype == DT_BF16) pk_attention<WT, bf16>(p, L, sa, M);
    else pk_attention<WT, float>(p, L, sa, M);
    pk_grid_arrive(p, s_fail);
    pk_stage<WT>(p, l, PH_O, s_bias, s_g, s_b, s_L);
    if (!(ok = pk_grid_wait(p, ++nbar * G, s_fail, s_ok))) break;
    pk_prep_att(p, xs, M, L.window);
    cbar();
    pk_matrix<WT, MT>(p, pk_mat<WT>(p, L, PH_O), PH_O, L, ring, full, empty, seq, xs, M, s_fail, s_bias, s_h, sa, nsplit, best, bi);
    pk_grid_arrive(p, s_fail);
    pk_stage<WT>(p, l, PH_UP, s_bias, s_g, s_b, s_L);
    if (!(ok = pk_grid_wait(p, ++nbar * G, s_fail, s_ok))) break;
    pk_prep_norm<WT>(p, xs, M, s_g, s_b, false, s_h, s_red, s_stat);
    cbar();
    pk_matrix<WT, MT>(p, pk_mat<WT>(p, L, PH_UP), PH_UP, L, ring, full, empty, seq, xs, M, s_fail, s_bias, s_h, sa, nsplit, best, bi);
    pk_grid_arrive(p, s_fail);
    pk_stage<WT>(p, l, PH_DOWN, s_bias, s_g, s_b, s_L);
    if (!(ok = pk_grid_wait(p, ++nbar * G, s_fail, s_ok))) break;
    pk_prep_copy(xs, p.ff, M * p.F);
    cbar();
    pk_matrix<WT, MT>(p, pk_mat<WT>(p, L, PH_DOWN), PH_DOWN, L, ring, full, empty, seq, xs, M, s_fail, s_bias, s_h, sa, nsplit, best,
                      bi);
    pk_grid_arrive(p, s_fail);
    if (l + 1 < p.n_layers) pk_stage<WT>(p, l + 1, PH_QKV, s_bias, s_g, s_b, s_L);
    else pk_stage<WT>(p, 0, PH_HEAD, s_bias, s_g, s_b, s_L);
    if (!(ok = pk_grid_wait(p, ++nbar * G, s_fail, s_ok))) break;
  }
  if (!ok) return;
  pk_prep_norm<WT>(p, xs, M, s_g, s_b, false, s_h, s_red, s_stat);
  cbar();
  pk_matrix<WT, MT>(p, pk_mat<WT>(p, *s_L, PH_HEAD), PH_HEAD, *s_L, ring, full, empty, seq, xs, M, s_fail, s_bias,
                    s_h, sa, nsplit, best, bi);
#pragma unroll
  for (int m = 0; m < MT; ++m)
    if (m < M && lane == m) {
      s_best[warp * PK_MAX_M + m] = best[m];
      s_bi[warp * PK_MAX_M + m] = bi[m];
    }
  cbar();
  if ((int)threadIdx.x < M) {
    const int m = threadIdx.x;
    float bv = s_best[m];
    int bx = s_bi[m];
    for (int w = 1; w < CW; ++w)
      if (argmax_better(s_best[w * PK_MAX_M + m], s_bi[w * PK_MAX_M + m], bv, bx)) {
        bv = s_best[w * PK_MAX_M + m];
        bx = s_bi[w * PK_MAX_M + m];
      }
    p.head_val[(size_t)blockIdx.x * p.args->B + m] = bv;
    p.head_idx[(size_t)blockIdx.x * p.args->B + m] = bx;
  }
}

template <typename WT, int MT>
cudaError_t set_smem(size_t smem) {
  static size_t set_dev[MAX_DEVICES] = {};
  size_t& cur = set_dev[current_device()];
  if (smem > cur) {
    const cudaError_t e = cudaFuncSetAttribute(k_decode_persistent<WT, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
    if (e != cudaSuccess) return e;
    cur = smem;
  }
  return cudaSuccess;
}

template <typename WT, int MT>
cudaError_t launch_t(const PKParams& p, int grid, cudaStream_t s) {
  const size_t smem = pk_smem_bytes(p.nslot, p.xs_floats);
  cudaError_t e = set_smem<WT, MT>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(PK_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_persistent<WT, MT>, p);
}

template <typename WT, int MT>
cudaError_t occupancy_t(size_t smem, int* n) {
  const cudaError_t e = set_smem<WT, MT>(smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, k_decode_persistent<WT, MT>, PK_THREADS, smem);
}

}  // namespace

size_t pk_smem_bytes(int nslot, int xs_floats) {
  return (size_t)PK_RING_OFF + (size_t)nslot * PK_SLOT_BYTES + (size_t)xs_floats * sizeof(float);
}

cudaError_t launch_decode_persistent(const PKParams& p, int wdt, int M, int grid, cudaStream_t s) {
  if (M < 1 || M > PK_MAX_M || p.nslot < 2 || p.nslot > PK_MAX_SLOTS || grid < 1) return cudaErrorInvalidValue;
  if (wdt == DT_F32) return M == 1 ? launch_t<float, 1>(p, grid, s) : launch_t<float, PK_MAX_M>(p, grid, s);
  if (wdt == DT_BF16) return M == 1 ? launch_t<bf16, 1>(p, grid, s) : launch_t<bf16, PK_MAX_M>(p, grid, s);
  if (wdt == DT_Q8) return M == 1 ? launch_t<Q8, 1>(p, grid, s) : launch_t<Q8, PK_MAX_M>(p, grid, s);
  return cudaErrorInvalidValue;
}

cudaError_t pk_blocks_per_sm(int wdt, int M, size_t smem, int* n) {
  if (wdt == DT_F32) return M == 1 ? occupancy_t<float, 1>(smem, n) : occupancy_t<float, PK_MAX_M>(smem, n);
  if (wdt == DT_BF16) return M == 1 ? occupancy_t<bf16, 1>(smem, n) : occupancy_t<bf16, PK_MAX_M>(smem, n);
  if (wdt == DT_Q8) return M == 1 ? occupancy_t<Q8, 1>(smem, n) : occupancy_t<Q8, PK_MAX_M>(smem, n);
  return cudaErrorInvalidValue;
}

}  // namespace llm
