// Temperature / top-k sampling of the next token from the LM head's logits.
//
// "batch_forge" (component table) samples greedily, with a temperature, or from the top-k.
// Here the head's epilogue has written each row's fp32 logits; one CTA per row then
//   1. returns the first NaN index (the argmax rule) when the row holds a NaN;
//   2. finds the k-th largest logit by a radix select over order-preserving 32-bit keys
//      (four 8-bit passes with a shared-memory histogram);
//   3. collects the k candidates: every logit above that value and, of those equal to it,
//      the lowest indices (an exclusive scan over contiguous index ranges keeps index order);
//   4. orders the candidates by value (ties: lower index first), forms
//      p_i = exp((z_i - z_top) / T) and their sum in that order in one thread, and returns
//      the first candidate whose running sum exceeds u * sum, u being the caller's uniform
//      draw for the row.
// top_k <= 1 or T <= 0 is greedy. No random numbers are drawn on the device.
#include <climits>

#include "misc.cuh"

namespace llm {

namespace {

constexpr int SM_THREADS = 512;
constexpr int SM_WARPS = SM_THREADS / 32;

// Ascending floats map to ascending unsigned keys (finite values and infinities).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(SM_THREADS) k_sample(const SampleParams p) {
  __shared__ unsigned hist[256];
  __shared__ unsigned s_warp[SM_WARPS];
  __shared__ uint32_t s_prefix;
  __shared__ unsigned s_kleft;
  __shared__ int s_nan, s_nc;
  __shared__ float c_val[SAMPLE_MAX_K], o_val[SAMPLE_MAX_K];
  __shared__ int c_idx[SAMPLE_MAX_K], o_idx[SAMPLE_MAX_K];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_trigger();
  const StepArgs* a = p.args;
  const int V = p.vocab;
  const float* z = a->logits + (size_t)b * V;
  const float T = a->temperature;
  int k = T > 0.0f ? a->top_k : 1;
  k = max(1, min(k, min(SAMPLE_MAX_K, V)));

  // 1. NaN: the first NaN index, as the argmax rule
  if (tid == 0) s_nan = INT_MAX;
  __syncthreads();
  for (int i = tid; i < V; i += SM_THREADS)
    if (z[i] != z[i]) atomicMin(&s_nan, i);
  __syncthreads();
  if (s_nan != INT_MAX) {
    if (tid == 0) {
      a->next_ids[b] = s_nan;
      set_flag(p.flags, FLAG_NAN_LOGIT);
    }
    return;
  }

  // 2. radix select: thr = key of the k-th largest logit, kleft = how many logits equal to it
  //    are among the k
  uint32_t prefix = 0, mask = 0;
  unsigned kleft = (unsigned)k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += SM_THREADS) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < V; i += SM_THREADS) {
      const uint32_t key = order_key(z[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      unsigned cum = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (cum + hist[d] >= kleft) break;
        cum += hist[d];
      }
      s_prefix = prefix | ((uint32_t)d << shift);
      s_kleft = kleft - cum;
    }
    __syncthreads();
    prefix = s_prefix;
    kleft = s_kleft;
    mask |= 0xFFu << shift;
  }
  const uint32_t thr = prefix;

  // 3. candidates: keys above thr, and the kleft lowest-index keys equal to thr. Thread t owns
  //    the contiguous indices [t * chunk, (t + 1) * chunk), so an exclusive scan of the per-
  //    thread counts of equal keys gives each its rank in index order.
  const int chunk = (V + SM_THREADS - 1) / SM_THREADS;
  const int i0 = min(V, tid * chunk), i1 = min(V, i0 + chunk);
  unsigned eq = 0;
  for (int i = i0; i < i1; ++i) eq += order_key(z[i]) == thr;
  unsigned incl = eq;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  if (tid == 0) s_nc = 0;
  __syncthreads();
  unsigned base = incl - eq;
  for (int w = 0; w < warp; ++w) base += s_warp[w];
  unsigned r = base;
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = order_key(z[i]);
    const bool take = key > thr || (key == thr && r++ < kleft);
    if (take) {
      const int slot = atomicAdd(&s_nc, 1);
      if (slot < SAMPLE_MAX_K) {
        c_val[slot] = z[i];
        c_idx[slot] = i;
      }
    }
  }
  __syncthreads();

  // 4. order the k candidates, then the inverse-CDF draw in one thread
  if (warp == 0) {
    const int nc = min(s_nc, k);
    for (int c = lane; c < nc; c += 32) {
      const float v = c_val[c];
      const int ix = c_idx[c];
      int rank = 0;
      for (int o = 0; o < nc; ++o) {
        const float w = c_val[o];
        rank += (w > v) || (w == v && c_idx[o] < ix);
      }
      o_val[rank] = v;
      o_idx[rank] = ix;
    }
    __syncwarp();
    if (lane == 0 && nc == 1) a->next_ids[b] = o_idx[0];   // greedy
    if (lane == 0 && nc > 1) {
      float u = a->uniforms ? a->uniforms[b] : 0.0f;
      u = fminf(fmaxf(u, 0.0f), 0.99999994f);
      const float zt = o_val[0];
      float sum = 0.0f;
      for (int j = 0; j < nc; ++j) {
        const float e = expf((o_val[j] - zt) / T);
        c_val[j] = e;
        sum += e;
      }
      const float target = u * sum;
      float cum = 0.0f;
      int pick = nc - 1;
      for (int j = 0; j < nc; ++j) {
        cum += c_val[j];
        if (cum > target) {
          pick = j;
          break;
        }
      }
      a->next_ids[b] = o_idx[pick];
    }
  }
}

}  // namespace

cudaError_t launch_sample(const SampleParams& p, int B, cudaStream_t s, bool pdl) {
  if (B <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t c = make_launch_cfg(dim3(B), dim3(SM_THREADS), 0, s, attr, pdl);
  return cudaLaunchKernelEx(&c, k_sample, p);
}

}  // namespace llm
