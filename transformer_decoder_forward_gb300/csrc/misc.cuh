// Embedding, norm, argmax-reduce and step-argument kernels (declarations).
#pragma once
#include "common.cuh"

namespace llm {

struct EmbedParams {
  const void* tok_emb;     // [vocab][d]
  const void* tok_scale;   // Q8_0 token embedding: [vocab][d / 32] fp16 block scales, else nullptr
  const void* pos_emb;     // [n_ctx][d] or nullptr
  const StepArgs* args;    // tokens, positions
  float* h;                // [M][d]
  int M, d, vocab, n_ctx;
  unsigned* flags;
};

struct NormParams {
  const float* h;          // [.][d] fp32 residual stream
  const void* g;           // [d] weight dtype
  const void* b;           // [d] or nullptr
  void* out;               // [rows][d] activation dtype
  const StepArgs* args;    // for last_row
  int rows, d;
  int layer_norm;          // 1: LayerNorm, 0: RMSNorm
  int use_last_row;        // 1: row r reads h[args->last_row[r]] (when set)
  float eps;
};

struct ArgmaxParams {
  const float* part_val;   // [n_tiles][B]
  const int* part_idx;
  int n_tiles;
  const StepArgs* args;    // next_ids, B
  unsigned* flags;
};

// Temperature / top-k sampling of the next token (reads logits, uniforms, temperature and
// top_k from the step arguments).
constexpr int SAMPLE_MAX_K = 64;
struct SampleParams {
  const StepArgs* args;
  int vocab;
  unsigned* flags;
};

cudaLaunchConfig_t make_launch_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr,
                                   bool pdl);
cudaError_t launch_embed(const EmbedParams& p, int wdt, cudaStream_t s, bool pdl);
cudaError_t launch_norm(const NormParams& p, int wdt, int adt, cudaStream_t s, bool pdl);
cudaError_t launch_argmax(const ArgmaxParams& p, int B, cudaStream_t s, bool pdl);
cudaError_t launch_sample(const SampleParams& p, int B, cudaStream_t s, bool pdl);
cudaError_t launch_set_args(StepArgs* dst, const StepArgs& v, cudaStream_t s);
const void* set_args_kernel();
cudaError_t launch_selftest_wait(unsigned* flags, cudaStream_t s);

}  // namespace llm
