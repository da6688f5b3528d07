// One persistent kernel for a whole decode step of a few rows (decode batch <= PK_MAX_M).
#pragma once
#include "common.cuh"

namespace llm {

constexpr int PK_MAX_M = 8;            // rows (sequences) of one step
constexpr int PK_MAX_G = 8;            // query heads per KV head
constexpr int PK_COMPUTE_WARPS = 8;    // warps that compute; one more warp streams the weights
constexpr int PK_THREADS = (PK_COMPUTE_WARPS + 1) * 32;
constexpr int PK_SLOT_BYTES = 48 * 1024;   // one stage of the weight ring
constexpr int PK_MAX_SLOTS = 4;
constexpr int PK_ATT_CH = 256;         // keys of one attention work item
constexpr int PK_MAX_UNITS = 128;      // output rows (units) of one matrix a CTA may own
constexpr int PK_MAX_D = 2048;         // model width the staged norm vectors hold

// Weights and KV pool of one layer (device-resident table, one entry per layer).
struct PKLayer {
  const void *w_qkv, *s_qkv, *b_qkv;    // s_*: Q8_0 block scales, else nullptr
  const void *w_o, *s_o, *b_o;
  const void *w_up, *s_up, *b_up;
  const void *w_down, *s_down, *b_down;
  const void *ln1_g, *ln1_b, *ln2_g, *ln2_b;
  const void *qn_g, *kn_g;              // Q/K-norm gains, or nullptr
  KVLayer kv;
  int window;                           // sliding window (0: full causal)
};

struct PKParams {
  const PKLayer* layers;   // [n_layers] in device memory
  int n_layers, d, H, Hkv, F, vocab, n_ctx;
  int gpt2;                // 1: LayerNorm, GELU, learned positions; 0: RMSNorm, SwiGLU, RoPE
  float eps;
  const void *tok_emb, *tok_scale, *pos_emb, *lnf_g, *lnf_b;
  const float2* rope_tab;  // [HD/2] RoPE inverse frequencies split (hi, lo)
  const StepArgs* args;
  // scratch (fp32), written and read inside one launch
  float* h;                // [M][d] residual stream
  float* qkv;              // [M][(H + 2 Hkv) 64] projections plus bias
  float* att;              // [M][H 64] attention output of sequences whose context is one item
  float* ff;               // [M][F] FFN activation
  float* part_o;           // [M][H][max_ch][64] unnormalised outputs of attention items
  float* part_ml;          // [M][H][max_ch][2] their (max, sum) in log2 units
  int max_ch;
  float* head_val;         // [gridDim][B] argmax partials of the LM head
  int* head_idx;
  unsigned* sync;          // [0] grid arrival counter, [1] abort word; zeroed before every launch
  unsigned* flags;
  int withhold;            // >= 0: that CTA never arrives (bounded-barrier self-test); -1 normally
  int xs_floats;           // shared-memory activation capacity (floats)
  int nslot;               // stages of the weight ring
};

// Shared memory a launch needs for `nslot` ring stages and `xs_floats` staged activations.
size_t pk_smem_bytes(int nslot, int xs_floats);
// Launch (cooperative: the CTAs wait on one another, so all must be resident).
cudaError_t launch_decode_persistent(const PKParams& p, int wdt, int M, int grid, cudaStream_t s);
// CTAs of the kernel instance for (wdt, M) that fit on one SM with the given shared memory.
cudaError_t pk_blocks_per_sm(int wdt, int M, size_t smem, int* n);

}  // namespace llm
