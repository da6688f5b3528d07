// Shared device-side definitions of the decoder-step kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace llm {

// DT_SPLIT: activation storage of bf16-weight models (see Split below). DT_Q8: Q8_0 weights
// (int8 quants, one fp16 scale per 32-weight block; see Q8 below).
enum : int { DT_F32 = 0, DT_BF16 = 1, DT_SPLIT = 2, DT_Q8 = 3 };
enum : int { ARCH_GPT2 = 0, ARCH_LLAMA = 1 };
constexpr int HD = 64;          // head_dim (the only supported value)
constexpr int KVB = 16;         // tokens per KV block

// Launch state that belongs to a device (function attributes, occupancy answers) is cached
// per device, so one process may drive several GPUs.
constexpr int MAX_DEVICES = 64;
inline int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return 0;
  return d % MAX_DEVICES;
}

// Device error word bits (mirrors LLM_FLAG_* in include/llm.h).
constexpr unsigned FLAG_BAD_TOKEN = 0x01u;
constexpr unsigned FLAG_BAD_POSITION = 0x02u;
constexpr unsigned FLAG_BAD_BLOCK = 0x04u;
constexpr unsigned FLAG_NAN_LOGIT = 0x08u;
constexpr unsigned FLAG_WAIT_TIMEOUT = 0x10u;

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// Activations of bf16-weight models. A value v is kept as the bf16 pair hi = bf16(v),
// lo = bf16(v - hi), which holds v to about 2^-17 relative (bf16 alone: 2^-9). A row of n
// values is stored as its n hi values followed by its n lo values (row stride 2n bf16), so
// a tensor-core kernel reads the operand as two plain bf16 matrices and sums two products,
// and a CUDA-core kernel adds the halves. Only the weights are bf16; what the step
// computes between projections stays at fp32 accuracy.
struct Split {};
template <typename WT> struct ActOf { using type = float; };
template <> struct ActOf<bf16> { using type = Split; };

// Q8_0 weights ("rvllm-metal", sections "What's basic about it" and "What's next": one byte a
// weight): a matrix row is cut into blocks of 32 values, value j of a block is d * q_j with q an
// int8 quant and d the block's fp16 scale. The library keeps them as two planes: the quants
// [rows][K] int8 (16-byte vector loads) and the scales [rows][K / 32] fp16. Q8 is the tag type
// of such a matrix; its models keep vectors (gains, biases, learned positions) and activations
// in fp32.
struct Q8 {};
constexpr int Q8_BLOCK = 32;
template <> struct ActOf<Q8> { using type = float; };
// element type a matrix of weight type WT is stored in, and that of its model's vectors
template <typename WT> struct Elem { using type = WT; };
template <> struct Elem<Q8> { using type = int8_t; };
template <typename WT> struct VecT { using type = WT; };
template <> struct VecT<Q8> { using type = float; };

// Element n of row `row` of an activation matrix whose rows are `ld` storage elements apart
// (fp32: ld >= n_cols; Split: ld = 2 * n_cols, the lo half starting at ld / 2).
template <typename AT> __device__ __forceinline__ void act_store(void* base, size_t row, int ld, int n, float v);
template <> __device__ __forceinline__ void act_store<float>(void* base, size_t row, int ld, int n, float v) {
  reinterpret_cast<float*>(base)[row * ld + n] = v;
}
template <> __device__ __forceinline__ void act_store<Split>(void* base, size_t row, int ld, int n, float v) {
  bf16* r = reinterpret_cast<bf16*>(base) + row * ld;
  const bf16 hi = __float2bfloat16_rn(v);
  r[n] = hi;
  r[(ld >> 1) + n] = __float2bfloat16_rn(v - __bfloat162float(hi));
}
template <typename AT> __device__ __forceinline__ float act_load(const void* base, size_t row, int ld, int n);
template <> __device__ __forceinline__ float act_load<float>(const void* base, size_t row, int ld, int n) {
  return reinterpret_cast<const float*>(base)[row * ld + n];
}
template <> __device__ __forceinline__ float act_load<Split>(const void* base, size_t row, int ld, int n) {
  const bf16* r = reinterpret_cast<const bf16*>(base) + row * ld;
  return __bfloat162float(r[n]) + __bfloat162float(r[(ld >> 1) + n]);
}
// Four consecutive elements n..n+3 (n a multiple of 4, row start 16-byte aligned for fp32,
// 8-byte aligned for Split).
template <typename AT> __device__ __forceinline__ void act_store4(void* base, size_t row, int ld, int n, const float* v);
template <> __device__ __forceinline__ void act_store4<float>(void* base, size_t row, int ld, int n, const float* v) {
  *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + row * ld + n) = make_float4(v[0], v[1], v[2], v[3]);
}
template <> __device__ __forceinline__ void act_store4<Split>(void* base, size_t row, int ld, int n, const float* v) {
  bf16* r = reinterpret_cast<bf16*>(base) + row * ld;
  __nv_bfloat162 h[2], l[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    l[i] = __floats2bfloat162_rn(v[2 * i] - __low2float(h[i]), v[2 * i + 1] - __high2float(h[i]));
  }
  *reinterpret_cast<uint2*>(r + n) = *reinterpret_cast<const uint2*>(h);
  *reinterpret_cast<uint2*>(r + (ld >> 1) + n) = *reinterpret_cast<const uint2*>(l);
}

__device__ __forceinline__ void set_flag(unsigned* flags, unsigned bit) {
  if (flags) atomicOr(flags, bit);
}

// 16-byte global loads. Weights are read once per step: stream them past L1.
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ldg16(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Unpack 16 bytes into floats: 4 for fp32, 8 for bf16.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
};
template <> struct Vec16<Q8> {
  static constexpr int N = 16;
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int b = 0; b < 4; ++b) f[4 * i + b] = (float)(int8_t)((w[i] >> (8 * b)) & 0xffu);
  }
};
template <> struct Vec16<bf16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Row statistics of a LayerNorm / RMSNorm over one fp32 row x[0..d) by one warp (d a
// multiple of 4, d <= 2048): mean (0 for RMSNorm) and rstd = 1 / sqrt(var + eps), var the
// biased variance about the mean (RMSNorm: mean of squares). Every projection that
// normalises its own input and the stand-alone norm kernel use this one routine, so both
// give bit-identical normalised rows. The row is left in v (16 float4 a lane).
// NV: float4 per lane held (d <= 128 NV); any NV that covers d gives bit-identical results.
constexpr int ROW_NV = 16;
template <int NV = ROW_NV>
__device__ __forceinline__ void warp_row_stats(const float* x, int d, bool layer_norm, float eps, float4 (&v)[NV],
                                               float& mean, float& rstd) {
  const int lane = threadIdx.x & 31;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const int d4 = d >> 2;
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int i = lane + 32 * j;
    v[j] = i < d4 ? x4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    s += (v[j].x + v[j].y) + (v[j].z + v[j].w);
  }
  mean = layer_norm ? warp_sum(s) / d : 0.0f;
  float q = 0.0f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    if (lane + 32 * j < d4) {
      const float a = v[j].x - mean, b = v[j].y - mean, c = v[j].z - mean, e = v[j].w - mean;
      q += (a * a + b * b) + (c * c + e * e);
    }
  }
  rstd = 1.0f / sqrtf(warp_sum(q) / d + eps);
}

// One normalised element, with the arithmetic pinned (every kernel that normalises uses it,
// so fused and stand-alone norms agree bit for bit).
__device__ __forceinline__ float norm_apply(float x, float mean, float rstd, float g, float b) {
  return fmaf((x - mean) * rstd, g, b);
}
// v as a bf16 pair reads it back: bf16(v) + bf16(v - bf16(v)).
__device__ __forceinline__ float pair_round(float v) {
  const float hi = __bfloat162float(__float2bfloat16_rn(v));
  return hi + __bfloat162float(__float2bfloat16_rn(v - hi));
}

// Greedy-argmax order: NaN ranks above every number (lowest index among NaNs),
// otherwise larger value wins and ties go to the lower index.
__device__ __forceinline__ bool argmax_better(float a, int ia, float b, int ib) {
  const bool na = a != a, nb = b != b;
  if (na || nb) return na && (!nb || ia < ib);
  return a > b || (a == b && ia < ib);
}

// Programmatic dependent launch: wait for the producer grid / let the consumer start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- shared-memory addresses, mbarriers and asynchronous copies (inline PTX) ----------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make a freshly initialised mbarrier visible to the async (TMA) proxy; follow with __syncthreads().
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  // no suspend-time hint: a hint lets a failed poll sleep for the whole hint even when the
  // phase completes meanwhile, which put ~1 us on every pipeline hand-off
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: every spin in this library gives up after ~2^31 SM clock cycles (about
// one second), sets FLAG_WAIT_TIMEOUT and returns false.
constexpr long long WAIT_CYCLES = 1ll << 31;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, unsigned* flags) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (clock64() - t0 < WAIT_CYCLES)
    if (mbar_try_wait(bar, parity)) return true;
  set_flag(flags, FLAG_WAIT_TIMEOUT);
  return false;
}
// Split cluster barrier (every thread of every CTA of the cluster): arrive (release) now,
// wait (acquire) later, so work in between overlaps the other CTAs' arrival.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Order this thread's earlier generic-proxy shared-memory accesses before later async-proxy
// (TMA / tensor-core) accesses of the same shared memory.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// 1-D bulk copy global -> shared (TMA engine); completes `bytes` on the mbarrier.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// Warm L2 with [src, src + bytes) (16-byte aligned, multiple of 16) without touching shared memory.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// 16-byte Ampere-style async copy global -> shared (L2 only), grouped by commit/wait.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Per-call pointers that change from step to step. A graph replays with fixed
// kernel parameters, so kernels read these through one device-resident struct
// that the first node of the step rewrites.
struct StepArgs {
  const int* tokens;        // [M]
  const int* positions;     // [M] position of each row
  const int* row_seq;       // [M] sequence of each row, or nullptr (row m is sequence m)
  const int* block_tables;  // [B][mbps]
  int* next_ids;            // [B]
  float* logits;            // [B][V] or nullptr
  const int* last_row;      // [B] row of each sequence's last token, or nullptr (row b)
  int M;
  int B;
  // sampled decode steps: one uniform draw in [0, 1) per sequence, temperature and top-k
  const float* uniforms;    // [B] or nullptr
  float temperature;
  int top_k;
};

// Paged KV pool of one layer: [block][kv_head][16][64], fp32 (the default) or bf16.
struct KVLayer {
  void* k;
  void* v;
  int num_blocks;
  int n_kv_heads;
  int mbps;        // max blocks per sequence (block-table row length)
  int contiguous;  // sequence s owns blocks [s*mbps, (s+1)*mbps)
  int dtype;       // DT_F32 or DT_BF16: element type of k and v
};

// Physical block holding logical position `pos` of sequence `seq`, or -1 (and a flag).
__device__ __forceinline__ int kv_block(const KVLayer& kv, const int* tables, int seq, int pos, unsigned* flags) {
  const int lb = pos >> 4;
  if (pos < 0 || lb >= kv.mbps) { set_flag(flags, FLAG_BAD_POSITION); return -1; }
  const int pb = kv.contiguous ? seq * kv.mbps + lb : tables[(size_t)seq * kv.mbps + lb];
  if (pb < 0 || pb >= kv.num_blocks) { set_flag(flags, FLAG_BAD_BLOCK); return -1; }
  return pb;
}
__device__ __forceinline__ size_t kv_offset(const KVLayer& kv, int pb, int g, int slot) {
  return (((size_t)pb * kv.n_kv_heads + g) * KVB + slot) * HD;
}

// What a projection kernel does with its output tile.
enum : int {
  EPI_STORE_F32 = 0,  // out_f32[m][n] = y + b
  EPI_STORE_ACT = 1,  // out[m][n] = act(y + b) in the activation dtype
  EPI_RESID = 2,      // resid[m][n] += y + b              (fp32 residual stream)
  EPI_GELU = 3,       // out[m][n] = gelu_tanh_clamped(y + b) (activation dtype)
  EPI_SWIGLU = 4,     // out[m][j] = silu(gate_j) * up_j; tile columns = 32 gate rows + 32 up rows
  EPI_QKV = 5,        // q -> q_out (fp32, RoPE'd), k/v -> KV pool slot of the row
  EPI_HEAD = 6,       // logits (optional) + per-tile argmax partials
};

struct Epilogue {
  int kind;
  int act_dtype;        // DT_F32 / DT_SPLIT for `out`
  const void* bias;     // [N] in the weight dtype, or nullptr
  void* out;            // STORE / GELU / SWIGLU output
  int ld_out;
  float* resid;         // RESID
  int ld_resid;
  // QKV
  float* q_out;         // [M][H*64]
  KVLayer kv;
  int n_heads;
  int rope;             // 1: rotate q and k (Llama)
  float rope_theta;
  const float2* rope_tab;  // [HD/2] inverse frequency of pair d split as (hi, lo), hi with 11 significant bits
  const void* qn_g;     // Q/K norm: gains [HD] (weight dtype) of the q and k heads' RMSNorm, or nullptr
  const void* kn_g;
  float qk_eps;
  // HEAD
  float* part_val;      // [n_tiles][M]
  int* part_idx;
  int vocab;
  // shared
  const StepArgs* args;
  unsigned* flags;
};

// Row r of the SwiGLU tile: tile columns 0..31 are gate rows, 32..63 the matching up rows.
__device__ __forceinline__ int swiglu_row(int n0_half, int c, int d_ff) {
  return c < 32 ? n0_half + c : d_ff + n0_half + (c - 32);
}

// GELU-tanh with the tanh argument u clamped to [-15, 15]. 0.5 (1 + tanh(u)) equals the
// logistic function of 2u, so the value is x / (1 + e^(-2u)): one exponential and one
// division, and with the clamp the exponential stays below e^30 (finite).
__device__ __forceinline__ float gelu_tanh_clamped(float x) {
  const float kC = 0.7978845608028654f;   // sqrt(2/pi)
  float u = kC * (x + 0.044715f * x * x * x);
  u = fminf(15.0f, fmaxf(-15.0f, u));
  return __fdividef(x, 1.0f + __expf(-2.0f * u));
}
__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

}  // namespace llm
