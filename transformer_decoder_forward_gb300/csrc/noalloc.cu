// Decode attention for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: code running inside a CUDA
// graph that is being captured elsewhere, allocators that forbid side allocations
// (a serving process that owns every byte of HBM through its own pool), or hosts
// where an allocation would synchronise the device at the wrong moment. For them
// llm_op_attention_decode_noalloc runs the same split-K decode attention as
// llm_op_attention_decode, but its scratch (the argument block and the per-split
// partial results) lives in the fixed array below instead of memory allocated per
// call. Every GPU that loads the library holds this array until the process exits.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "api_internal.h"
#include "attention.cuh"
#include "misc.cuh"

using namespace llm;

namespace {

// 4 MiB: a 256-byte argument block, then B * n_heads * splits * (64 + 2) floats of partials
// (splits = ceil(max_blocks_per_seq * 16 / split)). The split starts where the allocating entry
// point's does and doubles, up to the kernel's 2048-token limit, until the partials fit.
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(4) << 20;
constexpr size_t NOALLOC_ARGS_BYTES = 256;
constexpr int NOALLOC_MAX_SPLIT = 2048;   // a decode-attention chunk spans at most 2048 tokens

size_t noalloc_need(int B, int n_heads, int max_ctx, int split) {
  const size_t splits = (size_t)(max_ctx + split - 1) / split;
  return NOALLOC_ARGS_BYTES + (size_t)B * n_heads * splits * (HD + 2) * sizeof(float);
}
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, per device ordinal. In host code the symbol's name
// is a host-side stand-in, not a device address, so it is resolved once per device (with
// that device current) through cudaGetSymbolAddress and only that address is handed to
// kernels.
constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};

llm_status noalloc_scratch(int dev, unsigned char** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return llm_internal_fail(LLM_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    g_noalloc_ptr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_noalloc_ptr[dev]);
  return LLM_OK;
}

}  // namespace

extern "C" llm_status llm_op_attention_decode_noalloc(int kv_dtype, int B, int n_heads, int n_kv_heads,
                                                      const float* q, const void* k_pool, const void* v_pool,
                                                      int num_blocks, const int32_t* positions,
                                                      const int32_t* block_tables, int max_blocks_per_seq,
                                                      float* out, void* cuda_stream) {
  if (B <= 0 || n_heads <= 0 || n_kv_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
    return llm_internal_fail(LLM_ERR_INVALID_ARG, "sizes must be positive");
  if (!q || !k_pool || !v_pool || !positions || !block_tables || !out)
    return llm_internal_fail(LLM_ERR_INVALID_ARG, "NULL pointer argument");
  if (kv_dtype != LLM_DTYPE_F32 && kv_dtype != LLM_DTYPE_BF16)
    return llm_internal_fail(LLM_ERR_INVALID_ARG, "bad kv_dtype");
  if (n_heads % n_kv_heads != 0 || n_heads / n_kv_heads > 8)
    return llm_internal_fail(LLM_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads, at most 8 per KV head");
  const int max_ctx = max_blocks_per_seq * KVB;
  const size_t need_min = noalloc_need(B, n_heads, max_ctx, NOALLOC_MAX_SPLIT);
  if (need_min > NOALLOC_SCRATCH_BYTES)
    return llm_internal_fail(LLM_ERR_OUT_OF_RANGE,
                             "llm_op_attention_decode_noalloc: needs " + std::to_string(need_min) +
                                 " bytes of scratch at the largest split (2048 tokens), the fixed array holds " +
                                 std::to_string(NOALLOC_SCRATCH_BYTES) +
                                 " (B * n_heads * ceil(max_blocks_per_seq * 16 / 2048) * 264 + 256)");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return llm_internal_fail(LLM_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return llm_internal_fail(LLM_ERR_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
  // the allocating entry point's split, doubled until the partials fit the array
  int split = attn_decode_split_for(B, n_kv_heads, max_ctx, sms);
  while (noalloc_need(B, n_heads, max_ctx, split) > NOALLOC_SCRATCH_BYTES && split < NOALLOC_MAX_SPLIT)
    split = std::min(NOALLOC_MAX_SPLIT, split * 2);
  const int max_splits = (max_ctx + split - 1) / split;
  const size_t part_o = (size_t)B * n_heads * max_splits * HD;
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return llm_internal_fail(LLM_ERR_UNSUPPORTED, "device ordinal above 63");
  unsigned char* scratch = nullptr;
  llm_status st = noalloc_scratch(dev, &scratch);
  if (st != LLM_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  StepArgs* args = reinterpret_cast<StepArgs*>(scratch);
  StepArgs a{nullptr, positions, nullptr, block_tables, nullptr, nullptr, nullptr, B, B};
  AttnDecodeParams p{};
  p.q = q;
  p.kv.k = const_cast<void*>(k_pool);
  p.kv.v = const_cast<void*>(v_pool);
  p.kv.num_blocks = num_blocks;
  p.kv.n_kv_heads = n_kv_heads;
  p.kv.mbps = max_blocks_per_seq;
  p.kv.contiguous = 0;
  p.kv.dtype = kv_dtype == LLM_DTYPE_F32 ? DT_F32 : DT_BF16;
  p.args = args;
  p.B = B;
  p.n_heads = n_heads;
  p.split = split;
  p.max_splits = max_splits;
  p.part_o = reinterpret_cast<float*>(scratch + NOALLOC_ARGS_BYTES);
  p.part_ml = p.part_o + part_o;
  p.out = out;
  p.out_dtype = DT_F32;
  p.flags = nullptr;
  e = launch_set_args(args, a, s);
  if (e == cudaSuccess) e = launch_attn_decode(p, kv_dtype == LLM_DTYPE_F32 ? DT_F32 : DT_BF16, s, false);
  if (e != cudaSuccess)
    return llm_internal_fail(LLM_ERR_CUDA, std::string("llm_op_attention_decode_noalloc: ") + cudaGetErrorString(e));
  return LLM_OK;
}
