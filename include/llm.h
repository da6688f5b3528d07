/*
 * llm.h — C ABI of the GB300 KV-cached decoder step (libllm.so).
 *
 * One library, one GPU. It computes the forward step of a decoder-only
 * transformer in two variants:
 *   - GPT-2: learned position embeddings, LayerNorm, multi-head causal attention,
 *     GELU-tanh FFN with the tanh argument clamped to +-15, tied LM head
 *     ("bare-metal-llm", sections "Picking the model", "What got built", "The bug
 *     worth telling"; "batch_forge", GELU overflow paragraph);
 *   - Llama: RMSNorm, RoPE, grouped-query attention, SwiGLU FFN, tied embeddings,
 *     no biases ("rvllm-metal", section "What the kernels do").
 * Prefill and batched single-token decode both end in a greedy argmax on the
 * GPU, so one int32 per sequence leaves the device ("rvllm-metal", "What the
 * kernels do", last paragraph). The KV cache is paged with 16-token blocks found
 * through a per-sequence block table ("rvllm-metal", "What the kernels do":
 * kv_write into the paged cache, division and modulo of the position).
 *
 * Precision: only the weights take config.dtype. The residual stream, the KV cache
 * (unless config.kv_dtype asks for bf16) and the logits are fp32 (the weights alone are half precision in "rvllm-metal",
 * section "The matmul pain story"; its KV cache is F32, section "What's basic about
 * it"); with bf16 weights the activations fed to a projection are kept as bf16
 * (hi, lo) pairs, about 2^-17 relative, so the tensor cores take two bf16 products
 * per step instead of rounding the activations to bf16. All arithmetic accumulates
 * in fp32.
 *
 * Conventions for every call:
 *   - Pointer arguments are DEVICE pointers unless the argument says HOST.
 *   - The caller owns weights, inputs and outputs; the library never frees them
 *     and keeps weight pointers (no copy) from llm_create to llm_destroy.
 *   - The handle owns its KV pool and workspace, allocated in llm_create.
 *   - Work is enqueued on the handle's stream and returns before it runs (except
 *     where a call says it synchronises). A handle must not be used from two
 *     host threads at once.
 *   - Every call checks its arguments on the host before any launch and returns
 *     a status; nothing is launched when the status is not LLM_OK. Errors that
 *     only the device can see (a token id, position or block id out of range,
 *     a NaN logit) set bits in the handle's device error word, skip the bad
 *     access and never trap; read them with llm_get_error_flags.
 *   - llm_last_error() gives a one-line message for the last non-OK status
 *     returned on the calling thread.
 */
#ifndef LLM_H
#define LLM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LLM_OK = 0,
  LLM_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size, inconsistent config */
  LLM_ERR_OUT_OF_RANGE = 2,  /* a size beyond what the handle was created for */
  LLM_ERR_NO_DEVICE = 3,     /* no CUDA device, or not a compute capability 10.3 device */
  LLM_ERR_UNSUPPORTED = 4,   /* a config the library does not implement (e.g. head_dim != 64) */
  LLM_ERR_OOM = 5,           /* device allocation failed in llm_create */
  LLM_ERR_CUDA = 6,          /* a CUDA runtime call failed */
  LLM_ERR_DEVICE_FLAG = 7    /* llm_get_error_flags found a device-side error bit set */
} llm_status;

enum { LLM_ARCH_GPT2 = 0, LLM_ARCH_LLAMA = 1 };
/* LLM_DTYPE_Q8: Q8_0 weights ("rvllm-metal", sections "What's basic about it" and "What's
 * next": one byte a weight): each matrix row is cut into blocks of 32 values, value j of a
 * block being d * q_j with q an int8 quant and d the block's fp16 scale. The library takes the
 * quants [rows][K] int8 and the scales [rows][K / 32] fp16 as two arrays (the *_scale fields of
 * llm_weights); vectors (gains, biases) and the learned positions of such a model are fp32. */
enum { LLM_DTYPE_F32 = 0, LLM_DTYPE_BF16 = 1, LLM_DTYPE_Q8 = 2 };

/* Bits of the device error word (llm_get_error_flags). */
#define LLM_FLAG_BAD_TOKEN     0x01u  /* token id outside [0, vocab) */
#define LLM_FLAG_BAD_POSITION  0x02u  /* position outside [0, n_ctx) or beyond the block table */
#define LLM_FLAG_BAD_BLOCK     0x04u  /* block-table entry outside [0, num_kv_blocks) */
#define LLM_FLAG_NAN_LOGIT     0x08u  /* a logit was NaN (argmax then returns the first NaN index) */
#define LLM_FLAG_WAIT_TIMEOUT  0x10u  /* a bounded device-side wait gave up */

typedef struct {
  int arch;               /* LLM_ARCH_GPT2 or LLM_ARCH_LLAMA */
  int dtype;              /* LLM_DTYPE_F32, LLM_DTYPE_BF16 or LLM_DTYPE_Q8: the weights' type */
  int n_layers;
  int d_model;
  int n_heads;            /* query heads */
  int n_kv_heads;         /* KV heads; n_heads % n_kv_heads == 0 (GPT-2: equal) */
  int head_dim;           /* must be 64 */
  int d_ff;               /* FFN width F */
  int vocab;
  int n_ctx;              /* GPT-2: rows of the position table; Llama: largest position + 1 */
  float norm_eps;         /* LayerNorm / RMSNorm epsilon, inside the square root */
  float rope_theta;       /* Llama only */
  int kv_block_size;      /* tokens per KV block; must be 16 */
  int num_kv_blocks;      /* physical blocks per layer in the pool (ignored when contiguous_kv) */
  int max_batch;          /* largest B of a decode step or prefill call */
  int max_blocks_per_seq; /* row length of a block table */
  int max_prefill_tokens; /* rows of one prefill chunk (workspace size); >= the longest prompt */
  int contiguous_kv;      /* 1: sequence b owns slots [b*max_blocks_per_seq*16, ...), tables ignored */
  int kv_dtype;           /* element type of the KV cache: LLM_DTYPE_F32 (0, the default) or
                             LLM_DTYPE_BF16, K and V rounded to nearest bf16 (ties to even) when
                             written; half the cache bytes ("rvllm-metal", section "What's basic
                             about it", names the F32 cache as a weakness) */
  /* Model-feature variants ("rvllm-metal", section "What the kernels do", last paragraph:
   * Llama 3 RoPE scaling, Qwen2 attention biases, Qwen3 Q/K norm, Gemma's sliding window).
   * All zero: none of them. Attention biases need no field: the Llama variant uses b_qkv
   * when the weights give it. */
  int sliding_window;         /* W > 0: a query at position p attends to p-W+1 .. p only */
  int sliding_window_pattern; /* 0: every layer windowed; P > 0: layers l with (l+1) % P == 0
                                 attend globally (Gemma's interleaving) */
  int qk_norm;                /* 1: RMSNorm (eps = norm_eps, gains q_norm_w / k_norm_w [head_dim]
                                 per layer) of every q and k head before RoPE (Llama variant) */
  float rope_scale_factor;    /* Llama 3 RoPE scaling when > 1: a pair with wavelength 2 pi / f
                                 above original / low_freq_factor turns at f / factor, below
                                 original / high_freq_factor at f, linearly mixed in between */
  float rope_low_freq_factor;
  float rope_high_freq_factor;
  int rope_original_max_pos;
} llm_config;

/*
 * Weights: DEVICE pointers, element type given by config.dtype (fp32, bf16, or for Q8_0
 * int8 matrices with fp16 block scales and fp32 vectors and positions), row-major. Per-layer fields are HOST arrays of n_layers device pointers; the
 * library copies those arrays. Absent tensors are NULL (all biases and ln*_b /
 * pos_emb for Llama). Shapes, d = d_model, H = n_heads, Hkv = n_kv_heads,
 * hd = head_dim, F = d_ff:
 *   tok_emb [vocab][d]            token embedding, also the tied LM head
 *   pos_emb [n_ctx][d]            GPT-2 learned positions
 *   ln1_w/ln1_b [d]               pre-attention norm gain / bias
 *   w_qkv [(H+2Hkv)*hd][d]        rows: all q heads, then k heads, then v heads
 *   b_qkv [(H+2Hkv)*hd]
 *   w_o   [d][H*hd],  b_o [d]
 *   ln2_w/ln2_b [d]
 *   w_up  GPT-2: [F][d]; Llama: [2F][d] with gate rows 0..F-1 then up rows F..2F-1
 *   b_up  [F] (GPT-2)
 *   w_down [d][F], b_down [d]
 *   lnf_w/lnf_b [d]               final norm
 *   q_norm_w/k_norm_w [head_dim]  Q/K-norm gains per layer (config.qk_norm), else NULL
 * The Llama variant has no biases except an optional b_qkv (attention biases).
 */
typedef struct {
  const void* tok_emb;
  const void* pos_emb;
  const void* const* ln1_w;
  const void* const* ln1_b;
  const void* const* w_qkv;
  const void* const* b_qkv;
  const void* const* w_o;
  const void* const* b_o;
  const void* const* ln2_w;
  const void* const* ln2_b;
  const void* const* w_up;
  const void* const* b_up;
  const void* const* w_down;
  const void* const* b_down;
  const void* lnf_w;
  const void* lnf_b;
  const void* const* q_norm_w;
  const void* const* k_norm_w;
  /* LLM_DTYPE_Q8 only (else NULL): fp16 block scales [rows][K / 32] of the int8 matrices */
  const void* tok_emb_scale;
  const void* const* w_qkv_scale;
  const void* const* w_o_scale;
  const void* const* w_up_scale;
  const void* const* w_down_scale;
} llm_weights;

typedef struct llm_handle llm_handle;

/* Set up one model on the current device: the session object of the pages' engines, which
 * keep the weights resident on the GPU and allocate the KV cache once ("rvllm-metal",
 * sections "What the kernels do": the paged cache that kv_write fills through a block
 * table, and "You record work, then you submit it": buffers the GPU reads without copies).
 * A device that cannot run the kernels is an error, never a silent fallback: "batch_forge"
 * (usage paragraph: an explicitly requested backend that is unavailable returns an error)
 * and "rvllm-metal", section "Things that were problematic" (a runtime that quietly gave up
 * made the GPU tests pass without running; a kernel that does not load is a hard failure).
 *
 * Validate the config, check the device (compute capability 10.3), copy the
 * per-layer pointer arrays, allocate the KV pool
 * (2 * n_layers * num_kv_blocks * n_kv_heads * 16 * head_dim values of kv_dtype,
 * laid out [layer][block][kv_head][16][head_dim], K and V in separate pools)
 * and the workspace. cuda_stream is a cudaStream_t (NULL = the legacy default
 * stream, which disables CUDA-graph replay). Errors: INVALID_ARG, UNSUPPORTED,
 * NO_DEVICE, OOM, CUDA. On error *out is NULL and nothing is leaked. */
llm_status llm_create(const llm_config* config, const llm_weights* weights, void* cuda_stream,
                      llm_handle** out);

/* The end of the lifetime llm_create starts (the pages describe set-up only; this is its
 * inverse): free the pool, workspace and cached graphs (synchronises the stream). The
 * caller's weights are untouched. NULL is a no-op. */
void llm_destroy(llm_handle* h);

/* Prompt prefill from position 0 ("rvllm-metal", sections "The matmul pain story"
 * and "Numbers": the whole prompt goes through at once).
 *   tokens        device int32 [sum(lengths)], the prompts packed back to back
 *   lengths       HOST int32 [B], each in [1, max_prefill_tokens] and, for GPT-2, <= n_ctx
 *   block_tables  device int32 [B][max_blocks_per_seq] physical block ids (ignored
 *                 when contiguous_kv); the first ceil(len/16) entries must be valid
 *   next_ids      device int32 [B]: argmax of the last position's logits
 *   logits        device float [B][vocab] last-position logits, or NULL
 * Writes K/V of every prompt position into the pool. Sequences are processed in
 * chunks of at most max_prefill_tokens rows. Errors: INVALID_ARG, OUT_OF_RANGE. */
llm_status llm_prefill(llm_handle* h, const int32_t* tokens, const int32_t* lengths, const int32_t* block_tables,
                       int B, int32_t* next_ids, float* logits);

/* One pass over sequences that each feed any number of new tokens: prefill and decode rows
 * mixed in one batch ("rvllm-metal", section "What's next": batched requests through one
 * forward pass; "What the kernels do": attention of the new tokens over the cached blocks).
 * Sequence b feeds lengths[b] tokens at positions starts[b] .. starts[b] + lengths[b] - 1,
 * writes their K/V into its blocks, attends over positions 0 .. starts[b] + lengths[b] - 1
 * (the earlier ones already in the cache), and gets the argmax after its last token. A decode
 * row is lengths[b] = 1 with starts[b] = its context length; a prompt is starts[b] = 0; a
 * prompt continued in chunks has starts[b] > 0.
 *   tokens        device int32 [sum(lengths)], packed by sequence in order
 *   lengths       HOST int32 [B], each in [1, max_prefill_tokens]
 *   starts        HOST int32 [B], each >= 0 (NULL: all 0), starts[b] + lengths[b] <= n_ctx
 *   block_tables  device int32 [B][max_blocks_per_seq] (row b for sequence b; ignored when
 *                 contiguous_kv); the first ceil((starts[b] + lengths[b]) / 16) entries valid
 *   next_ids      device int32 [B];  logits  device float [B][vocab] or NULL
 * Sequences are processed in chunks of at most max_prefill_tokens rows. When the batch opens
 * with one-token sequences, those rows take the split-K decode attention and the others the
 * tiled prefill attention, in the same pass. Errors: INVALID_ARG, OUT_OF_RANGE. */
llm_status llm_step(llm_handle* h, const int32_t* tokens, const int32_t* lengths, const int32_t* starts,
                    const int32_t* block_tables, int B, int32_t* next_ids, float* logits);

/* One batched decode step ("rvllm-metal", section "What the kernels do").
 *   tokens        device int32 [B], the token fed to each sequence
 *   positions     device int32 [B], its position = the sequence's context length before
 *                 this step; K/V are written at that slot and attention covers 0..positions[b]
 *   block_tables  device int32 [B][max_blocks_per_seq] (ignored when contiguous_kv)
 *   next_ids      device int32 [B]
 *   logits        device float [B][vocab], or NULL
 * The first call for a given B captures the step in a CUDA graph (when the
 * stream allows it); later calls replay it. Errors: INVALID_ARG, OUT_OF_RANGE. */
llm_status llm_decode_step(llm_handle* h, const int32_t* tokens, const int32_t* positions,
                           const int32_t* block_tables, int B, int32_t* next_ids, float* logits);

/* llm_decode_step that samples the next token instead of taking the argmax ("batch_forge",
 * component table: sampling greedy, temperature, top-k). Per sequence b the candidates are
 * the top_k largest logits (ties at the cut keep the lower index), ordered by value then
 * index; p_i = exp((z_i - z_top) / temperature); the token is the first candidate whose
 * running sum of p exceeds uniforms[b] * sum(p).
 *   temperature   >= 0; 0 is greedy
 *   top_k         1..64; 1 is greedy
 *   uniforms      device float [B], the caller's draws in [0, 1) (values outside are clamped),
 *                 or NULL for u = 0 (the most likely token); no random numbers are drawn here
 *   logits        device float [B][vocab] or NULL (the handle keeps its own copy then)
 * A NaN logit returns the first NaN index and sets LLM_FLAG_NAN_LOGIT, as the argmax does.
 * Other arguments, graph capture and errors as llm_decode_step (INVALID_ARG also for
 * temperature or top_k out of range). */
llm_status llm_decode_step_sample(llm_handle* h, const int32_t* tokens, const int32_t* positions,
                                  const int32_t* block_tables, int B, float temperature, int top_k,
                                  const float* uniforms, int32_t* next_ids, float* logits);

/* The same step from HOST buffers: copies tokens, positions and (unless NULL or
 * contiguous_kv) block_tables to the device, runs llm_decode_step, copies
 * next_ids (and logits when not NULL) back, and synchronises the stream before
 * returning. All five pointers are HOST memory (pinned or pageable). */
llm_status llm_decode_step_host(llm_handle* h, const int32_t* tokens, const int32_t* positions,
                                const int32_t* block_tables, int B, int32_t* next_ids, float* logits);

/* Errors the device sees ("rvllm-metal", section "Things that were problematic": a failure
 * that is swallowed instead of reported let every GPU test pass; "How I know it's correct":
 * argmax with NaN is a tested case). Kernels never trap: a token, position or block id out
 * of range, a NaN logit, or a bounded wait that gave up sets a bit of the handle's device
 * error word and the offending access is skipped.
 * Synchronise the stream, return the device error word in *flags and clear it.
 * Returns LLM_ERR_DEVICE_FLAG when any bit was set, LLM_OK otherwise. */
llm_status llm_get_error_flags(llm_handle* h, uint32_t* flags);

/* Self-test of the device-side bounded wait: launches, on the handle's stream, one
 * kernel that waits on a barrier nothing completes. The wait gives up after its limit
 * (about 2^31 SM clocks, one second) and sets LLM_FLAG_WAIT_TIMEOUT, which the next
 * llm_get_error_flags returns; the context stays usable. Asynchronous. */
llm_status llm_selftest_wait_timeout(llm_handle* h);

/* Per-kernel timing. While enabled, every launch is bracketed by CUDA events on the
 * handle's stream. A decode step is captured as a graph with an event record node
 * around each kernel and replayed once (programmatic launch off), so the events time
 * the kernels back to back on the device; prefill launches run eagerly. */
typedef struct {
  char name[48];
  int launches;
  double total_ms;
} llm_kernel_stat;

llm_status llm_set_profiling(llm_handle* h, int enable);
/* Synchronise, then fill up to max entries (one per kernel name) with the times
 * accumulated since profiling was enabled or last reset; *n gets the count. */
llm_status llm_get_kernel_stats(llm_handle* h, llm_kernel_stat* out, int max, int* n, int reset);
/* Kernel launches issued by the most recent llm_decode_step / llm_prefill call. */
llm_status llm_last_launch_count(llm_handle* h, int* n);
/* enable = 1 (default): decode steps are captured once per B and replayed as CUDA
 * graphs; 0: every launch is issued eagerly. Graphs need a non-default stream. */
llm_status llm_set_graphs(llm_handle* h, int enable);

/* One-kernel decode step ("rvllm-metal", sections "What's basic about it": a step is
 * about 900 dispatches and the GPU waits between kernels, and "What's next": fuse them).
 * enable = 1: a decode step of B <= 8 sequences runs as one cooperative persistent
 * kernel (one CTA per SM, grid-wide barriers between the dependent phases, every phase's
 * weights streamed ahead into shared memory) followed by the argmax or the sampling kernel;
 * other batch sizes, prefill and mixed steps keep one kernel a phase. 0 (default): every
 * decode step takes one kernel a phase, the faster path on GB300 as measured (GPT-2 124M
 * fp32 at batch 1: 0.386 against 0.371 ms a step; at batch 8 about twice as slow). The
 * environment variable LLM_PERSISTENT=1 sets the default to 1. *supported (may be NULL) receives 1
 * when the model's shapes allow the persistent step on this device (rows of 16-byte
 * vectors, Q8_0 rows a multiple of 256, at most 8 query heads per KV head, one CTA per SM
 * resident), else 0, in which case enable has no effect. Drops nothing: the cached
 * graphs are keyed by the path they hold. */
llm_status llm_set_persistent(llm_handle* h, int enable, int* supported);

/* Self-test of the persistent step's grid barrier: launches the persistent kernel with
 * one CTA that never arrives, so the other CTAs' bounded barrier wait gives up after its
 * limit (about one second), sets LLM_FLAG_WAIT_TIMEOUT and every CTA leaves (the weight
 * streamer waits for its copies in flight first). Synchronises the stream; the next
 * llm_get_error_flags returns the flag and the context stays usable. Computes nothing
 * and writes no output. Errors: UNSUPPORTED when the persistent step does not apply to
 * this model (see llm_set_persistent). */
llm_status llm_selftest_grid_barrier(llm_handle* h);

/* Projection kernel choice: 0 = by row count (default), 1 = CUDA-core weight-stream
 * GEMV, 2 = CUDA-core tiled GEMM, 3 = tcgen05 GEMM with the activation rows on the
 * MMA's M side (bf16 models; falls back to 2 where it does not apply), 4 = tcgen05
 * GEMM with the weight rows on the MMA's M side (at most 256 activation rows; bf16,
 * or fp32 as three tf32 products; falls back to 3 / 2), 5 = tcgen05 GEMM on SM pairs
 * (cta_group::2: 256 weight rows a tile split over the two CTAs of a cluster; bf16 models,
 * falls back to 2; the default for more than 256 rows, LLM_GEMM_PAIR=0 keeps 3). For tests that force every
 * kernel on every shape: a variant other than 0 also keeps decode steps off the persistent
 * kernel (llm_set_persistent). Drops cached graphs. Errors: INVALID_ARG for another value. */
llm_status llm_set_linear_variant(llm_handle* h, int variant);

/* Test and diagnostic entry point (no handle): one projection with a chosen kernel,
 *   y[m][n] = sum_k x[m][k] * w[n][k] (+ bias[n]),  m < M, n < N,
 * w DEVICE [N][K] row-major in `dtype` (LLM_DTYPE_F32 or LLM_DTYPE_BF16), bias DEVICE
 * [N] in `dtype` or NULL, y DEVICE float [M][N]. x DEVICE in the library's activation
 * storage for that dtype: fp32 [M][K] for LLM_DTYPE_F32; for LLM_DTYPE_BF16 a bf16
 * [M][2K] array whose row m holds hi[0..K) then lo[0..K), x[m][k] = hi[k] + lo[k]
 * (the library keeps the activations of bf16-weight models as such pairs).
 * variant: 1 CUDA-core GEMV, 2 CUDA-core tiled GEMM, 3 tcgen05 GEMM (bf16 only),
 * 4 tcgen05 GEMM with the weights on the MMA's M side (M <= 256; bf16, or fp32 as
 * three tf32 products), 5 tcgen05 GEMM on SM pairs (bf16 only). Variants 3, 4 and 5 need
 * K % 8 == 0. Enqueued on `cuda_stream`.
 * Errors: INVALID_ARG (bad sizes, NULL, K % 8 for variants 3/4/5, M > 256 for 4),
 * UNSUPPORTED (variant 3 or 5 with fp32), CUDA. */
llm_status llm_op_linear(int dtype, int M, int N, int K, const void* x, const void* w, const void* bias, float* y,
                         int variant, void* cuda_stream);

/* llm_op_linear for Q8_0 weights: y[m][n] = sum_k x[m][k] * (wscale[n][k / 32] * wq[n][k])
 * (+ bias[n]). wq DEVICE int8 [N][K], wscale DEVICE fp16 [N][K / 32], bias DEVICE float [N] or
 * NULL, x DEVICE float [M][K], y DEVICE float [M][N]. variant: 1 CUDA-core GEMV (the int8
 * weight stream, any M), 2 CUDA-core tiled GEMM. Errors: INVALID_ARG (sizes, NULL, K % 32,
 * variant), CUDA. */
llm_status llm_op_linear_q8(int M, int N, int K, const float* x, const void* wq, const void* wscale,
                            const float* bias, float* y, int variant, void* cuda_stream);

/* Test and diagnostic entry point (no handle): one layer of batched decode attention
 * over a paged KV pool, the split-K kernel pair of llm_decode_step ("rvllm-metal",
 * section "What the kernels do": scores, -inf mask, softmax, probs @ V, reading the
 * paged cache). Row b attends with its n_heads query heads (GQA: head h uses KV head
 * h / (n_heads / n_kv_heads)) over positions 0..positions[b]:
 *   q             DEVICE float [B][n_heads * 64] (already rotated for Llama)
 *   k_pool/v_pool DEVICE [num_blocks][n_kv_heads][16][64] in kv_dtype (LLM_DTYPE_*)
 *   positions     DEVICE int32 [B]
 *   block_tables  DEVICE int32 [B][max_blocks_per_seq], slot = table[pos / 16] * 16 + pos % 16
 *   out           DEVICE float [B][n_heads * 64]
 * Its split partials live in device scratch that this call allocates and frees
 * stream-ordered (cudaMallocAsync / cudaFreeAsync) on cuda_stream. Device-side range
 * errors (a position or block id out of range) are skipped, not reported.
 * Errors: INVALID_ARG (NULL, sizes, n_heads % n_kv_heads, more than 8 query heads per
 * KV head), OOM, CUDA. */
llm_status llm_op_attention_decode(int kv_dtype, int B, int n_heads, int n_kv_heads, const float* q,
                                   const void* k_pool, const void* v_pool, int num_blocks, const int32_t* positions,
                                   const int32_t* block_tables, int max_blocks_per_seq, float* out,
                                   void* cuda_stream);

/* llm_op_attention_decode for callers that cannot allocate device memory (code inside
 * someone else's stream capture, or a process whose allocator owns all of HBM). The
 * pages have no counterpart of this entry point. Same arguments, layouts and result as
 * llm_op_attention_decode, but no cudaMalloc / cudaFree / allocating call of any
 * library: the scratch (a 256-byte argument block plus B * n_heads * ceil(max_blocks_per_seq
 * * 16 / split) * 264 bytes of split partials) lives in one fixed 4 MiB __device__ array that
 * every GPU loading the library holds until the process exits. The split (tokens per chunk)
 * starts at llm_op_attention_decode's choice and doubles, up to 2048, until the partials fit.
 *   - The first call on a device resolves the array's device address (cudaGetSymbolAddress)
 *     for that device; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents: calls whose
 *     execution overlaps on the GPU (other streams, other threads) race on it.
 * Errors: as llm_op_attention_decode, plus OUT_OF_RANGE when the scratch needed at a split
 * of 2048 exceeds the array (nothing is launched), UNSUPPORTED for device ordinals above 63. */
llm_status llm_op_attention_decode_noalloc(int kv_dtype, int B, int n_heads, int n_kv_heads, const float* q,
                                           const void* k_pool, const void* v_pool, int num_blocks,
                                           const int32_t* positions, const int32_t* block_tables,
                                           int max_blocks_per_seq, float* out, void* cuda_stream);

const char* llm_status_string(llm_status s);
const char* llm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* LLM_H */
