// Causal attention over the paged KV cache (declarations).
#pragma once
#include "common.cuh"

namespace llm {

// Decode: one query row per sequence, keys 0..positions[b].
struct AttnDecodeParams {
  const float* q;           // [B][H*64] fp32, RoPE already applied
  KVLayer kv;
  const StepArgs* args;     // positions, block tables
  int B;
  int n_heads;
  int split;                // tokens per split (multiple of 16)
  int max_splits;           // grid.y; 1: the split kernel writes `out` itself, no merge launch
  float* part_o;            // [B][H][max_splits][64]
  float* part_ml;           // [B][H][max_splits][2]  (running max in log2 units, sum of exp)
  void* out;                // [B][H*64] activations (DT_F32, or DT_SPLIT: row stride 2*H*64 bf16)
  int out_dtype;
  unsigned* flags;
  int window;               // sliding window W > 0: keys positions[b]-W+1 .. positions[b]; 0: all
};

// Prefill: packed rows; a work item is (sequence, first query position, row of that
// query, sequence length); keys of sequence s are positions 0..len-1 in the pool.
struct AttnPrefillParams {
  const float* q;           // [rows][H*64] fp32
  KVLayer kv;
  const StepArgs* args;     // block tables
  const int4* items;        // {seq, q_pos0, row0, len}
  int n_items;
  int n_heads;
  void* out;                // [rows][H*64] activations (DT_F32 or DT_SPLIT)
  int out_dtype;
  unsigned* flags;
  int window;               // sliding window W > 0: a query at p sees keys p-W+1 .. p; 0: all
};

// Tokens per decode split for a batch of B sequences of up to max_ctx keys (a multiple of
// 16; the environment variable LLM_ATTN_SPLIT overrides it).
int attn_decode_split_for(int B, int n_kv_heads, int max_ctx, int num_sms);

cudaError_t launch_attn_decode(const AttnDecodeParams& p, int kv_dtype, cudaStream_t s, bool pdl);
cudaError_t launch_attn_prefill(const AttnPrefillParams& p, int kv_dtype, cudaStream_t s, bool pdl);
// Tensor-core prefill attention: items of up to 128 query rows (any sliding window).
cudaError_t launch_attn_prefill_tc(const AttnPrefillParams& p, int kv_dtype, cudaStream_t s, bool pdl);
// Warp-specialised tensor-core prefill attention: items of up to 256 query rows (two 128-row
// tiles), no sliding window.
cudaError_t launch_attn_prefill_tc2(const AttnPrefillParams& p, int kv_dtype, cudaStream_t s, bool pdl);

}  // namespace llm
