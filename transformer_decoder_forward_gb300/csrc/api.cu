// C ABI of the decoder step: handle, workspace, step orchestration, CUDA graphs.
//
// A decode step is one CUDA graph: the pages record a whole forward pass into
// one command buffer and submit it once ("bare-metal-llm", section "What it
// taught me"; "rvllm-metal", section "You record work, then you submit it").
// Kernel parameters are fixed in a graph, so the per-call pointers (tokens,
// positions, block tables, outputs) travel through one device-resident
// StepArgs struct that the graph's first node rewrites; each replay only
// updates that node's parameters. Nothing is rebuilt per step on the host (the
// pages list per-step host-built tables as a weakness, "What's basic about it").
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "../../include/llm.h"
#include "api_internal.h"
#include "attention.cuh"
#include "linear.cuh"
#include "misc.cuh"
#include "persistent.cuh"

using namespace llm;

namespace {

thread_local std::string g_last_error;

llm_status fail(llm_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

#define CUDA_TRY(expr)                                                                          \
  do {                                                                                          \
    cudaError_t _e = (expr);                                                                    \
    if (_e != cudaSuccess)                                                                      \
      return fail(LLM_ERR_CUDA, std::string(#expr) + ": " + cudaGetErrorString(_e));           \
  } while (0)

struct LayerW {
  const void *ln1_w, *ln1_b, *w_qkv, *b_qkv, *w_o, *b_o, *ln2_w, *ln2_b, *w_up, *b_up, *w_down, *b_down;
  const void *q_norm_w, *k_norm_w;   // Q/K-norm gains, or nullptr
  const void *s_qkv, *s_o, *s_up, *s_down;   // Q8_0 block scales, or nullptr
};

struct GraphEntry {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphNode_t args_node = nullptr;
  int launches = 0;
};

struct ProfRec {
  std::string name;
  cudaEvent_t a, b;
};

struct Stat {
  int launches = 0;
  double ms = 0.0;
};

}  // namespace

llm_status llm_internal_fail(llm_status s, const std::string& msg) { return fail(s, msg); }

struct llm_handle {
  llm_config cfg{};
  int dev = 0, num_sms = 0;
  cudaStream_t stream = nullptr;
  int wdt = DT_F32;   // weights
  int adt = DT_F32;   // activations between kernels: DT_F32, or DT_SPLIT (bf16 pairs) for bf16 weights
  int act_mul = 1;    // row stride of an activation matrix in storage elements = act_mul * width
  const void *tok_emb = nullptr, *pos_emb = nullptr, *lnf_w = nullptr, *lnf_b = nullptr;
  const void* tok_scale = nullptr;   // Q8_0 block scales of tok_emb
  std::vector<LayerW> layers;
  // KV pool (fp32, or bf16 when cfg.kv_dtype asks for it)
  int kvdt = DT_F32;
  size_t kv_elt = 4;
  void* k_pool = nullptr;
  void* v_pool = nullptr;
  size_t layer_kv_elems = 0;
  int num_blocks = 0;
  // workspace
  int max_rows = 0;
  float* h = nullptr;
  void* xn = nullptr;
  float* q = nullptr;
  void* att = nullptr;
  void* ff = nullptr;
  int split = 64, max_splits = 1;
  float* attn_po = nullptr;
  float* attn_ml = nullptr;
  int head_tiles = 0;
  float* head_val = nullptr;
  int* head_idx = nullptr;
  unsigned* flags = nullptr;
  StepArgs* d_args = nullptr;
  int* d_row_pos = nullptr;
  int* d_row_seq = nullptr;
  int* d_last_row = nullptr;
  int4* d_items = nullptr;
  int max_items = 0;
  float2* d_rope = nullptr;   // RoPE inverse frequencies, split (hi, lo)
  // host-buffer entry point staging
  int* d_host_tokens = nullptr;
  int* d_host_pos = nullptr;
  int* d_host_tables = nullptr;
  int* d_host_ids = nullptr;
  float* d_host_logits = nullptr;
  float* d_samp_logits = nullptr;   // logits of a sampled step when the caller asks for none
  // execution options
  bool use_graphs = true;
  bool pdl = true;   // programmatic dependent launch between the step's kernels
  bool attn_tc2 = false;   // prefill attention: the warp-specialised kernel (256-row items)
  int lin_variant = LIN_AUTO;
  bool gemm_pair = true;   // prefill projections on SM pairs (LLM_GEMM_PAIR=0: one SM a tile)
  std::map<int, GraphEntry> graphs;
  // one-kernel decode step (decode batches of at most PK_MAX_M rows)
  bool pk_supported = false;   // shapes, alignment and residency allow it
  bool pk_multi = false;       // the instance for more than one row fits too
  bool pk_enabled = false;     // opt-in: measured slower than the per-phase graph (see llm.h)
  int pk_smem_max = 0;
  int pk_max_ch = 0;
  PKLayer* d_pk_layers = nullptr;
  float *pk_qkv = nullptr, *pk_att = nullptr, *pk_ff = nullptr, *pk_po = nullptr, *pk_ml = nullptr;
  float* pk_head_val = nullptr;
  int* pk_head_idx = nullptr;
  unsigned* pk_sync = nullptr;
  // profiling
  bool profiling = false;
  bool prof_capture = false;   // a profiled decode step is being captured
  std::vector<ProfRec> prof;
  std::vector<cudaEvent_t> event_pool;
  size_t event_next = 0;
  std::map<std::string, Stat> stats;
  int launch_counter = 0;
  int last_launches = 0;
  std::vector<void*> allocations;
};

namespace {

template <typename T>
llm_status dev_alloc(llm_handle* h, T** p, size_t count) {
  *p = nullptr;
  if (count == 0) count = 1;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(LLM_ERR_OOM, "cudaMalloc of " + std::to_string(count * sizeof(T)) + " bytes failed");
  }
  h->allocations.push_back(*p);
  e = cudaMemset(*p, 0, count * sizeof(T));
  if (e != cudaSuccess) return fail(LLM_ERR_CUDA, cudaGetErrorString(e));
  return LLM_OK;
}

void free_all(llm_handle* h) {
  for (auto& kv : h->graphs) {
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
    if (kv.second.graph) cudaGraphDestroy(kv.second.graph);
  }
  h->graphs.clear();
  for (auto ev : h->event_pool) cudaEventDestroy(ev);
  h->event_pool.clear();
  for (void* p : h->allocations) cudaFree(p);
  h->allocations.clear();
}

cudaEvent_t next_event(llm_handle* h) {
  if (h->event_next >= h->event_pool.size()) {
    cudaEvent_t e;
    cudaEventCreate(&e);
    h->event_pool.push_back(e);
  }
  return h->event_pool[h->event_next++];
}

// Every kernel launch goes through here: counts it and, when profiling, brackets it with events.
template <typename F>
llm_status run(llm_handle* h, const char* name, F&& f) {
  cudaEvent_t a = nullptr, b = nullptr;
  // inside a capture the records become event nodes of the graph
  const unsigned rec = h->prof_capture ? cudaEventRecordExternal : cudaEventRecordDefault;
  if (h->profiling) {
    a = next_event(h);
    b = next_event(h);
    cudaEventRecordWithFlags(a, h->stream, rec);
  }
  cudaError_t e = f();
  if (e != cudaSuccess) {
    cudaGetLastError();   // a failed launch must not be reported again by the next call
    return fail(LLM_ERR_CUDA, std::string(name) + ": " + cudaGetErrorString(e));
  }
  if (h->profiling) {
    cudaEventRecordWithFlags(b, h->stream, rec);
    h->prof.push_back({name, a, b});
  }
  h->launch_counter++;
  return LLM_OK;
}

#define RUN(name, expr)                              \
  do {                                               \
    llm_status _s = run(h, name, [&]() { return (expr); }); \
    if (_s != LLM_OK) return _s;                     \
  } while (0)

int pick_variant(const llm_handle* h, const LinearParams& p) {
  if (h->lin_variant != LIN_AUTO) return h->lin_variant;
  if (p.M <= 8) return LIN_GEMV;   // a few rows: the CUDA-core weight stream has the shortest path
  // 192..256 rows and at least 32 output tiles of 128 (GPT-2 XL's qkv, up and tied head at batch
  // 256): the activations-on-M kernel measured 9-54% faster than the weights-on-M one, which
  // stays better for the narrow o and down projections
  if (p.M >= 192 && p.N >= 32 * 128 && gemm_tc_supported(p)) return LIN_TC;
  if (p.M <= 256 && gemm_tc_swap_supported(p)) return LIN_TC_SWAP;
  if (p.M <= 64) return LIN_GEMV;
  // more than 256 rows (prefill): the SM-pair kernel halves the shared-memory bytes per MMA
  if (gemm_tc_supported(p)) return h->gemm_pair ? LIN_TC_PAIR : LIN_TC;
  return LIN_SIMT;
}

llm_status linear_v(llm_handle* h, const char* tag, const LinearParams& p, int v) {
  std::string name = std::string(v == LIN_GEMV      ? "gemv_"
                                 : v == LIN_TC      ? "gemm_tc_"
                                 : v == LIN_TC_PAIR ? "gemm_tc2_"
                                 : v == LIN_TC_SWAP ? "gemm_tcs_"
                                                    : "gemm_simt_") +
                     tag;
  if (v == LIN_GEMV) RUN(name.c_str(), launch_gemv(p, h->num_sms, h->stream, h->pdl));
  else if (v == LIN_TC) RUN(name.c_str(), launch_gemm_tc(p, h->num_sms, h->stream, h->pdl));
  else if (v == LIN_TC_PAIR) RUN(name.c_str(), launch_gemm_tc2(p, h->num_sms, h->stream, h->pdl));
  else if (v == LIN_TC_SWAP) RUN(name.c_str(), launch_gemm_tc_swap(p, h->num_sms, h->stream, h->pdl));
  else RUN(name.c_str(), launch_gemm_simt(p, h->stream, h->pdl));
  return LLM_OK;
}

llm_status linear(llm_handle* h, const char* tag, LinearParams p) {
  int v = pick_variant(h, p);
  if (v == LIN_TC_SWAP && !gemm_tc_swap_supported(p)) v = gemm_tc_supported(p) ? LIN_TC : LIN_SIMT;
  if ((v == LIN_TC || v == LIN_TC_PAIR) && !gemm_tc_supported(p)) v = LIN_SIMT;
  return linear_v(h, tag, p, v);
}

KVLayer kv_layer(const llm_handle* h, int l) {
  KVLayer kv;
  kv.k = static_cast<char*>(h->k_pool) + (size_t)l * h->layer_kv_elems * h->kv_elt;
  kv.v = static_cast<char*>(h->v_pool) + (size_t)l * h->layer_kv_elems * h->kv_elt;
  kv.dtype = h->kvdt;
  kv.num_blocks = h->num_blocks;
  kv.n_kv_heads = h->cfg.n_kv_heads;
  kv.mbps = h->cfg.max_blocks_per_seq;
  kv.contiguous = h->cfg.contiguous_kv;
  return kv;
}

// Sliding window of layer l (0: full causal attention).
int layer_window(const llm_handle* h, int l) {
  const llm_config& c = h->cfg;
  if (c.sliding_window <= 0) return 0;
  if (c.sliding_window_pattern > 0 && (l + 1) % c.sliding_window_pattern == 0) return 0;
  return c.sliding_window;
}

Epilogue base_epi(const llm_handle* h) {
  Epilogue e;
  memset(&e, 0, sizeof(e));
  e.act_dtype = h->adt;
  e.args = h->d_args;
  e.flags = h->flags;
  return e;
}

// y = Norm(h) . W^T. Where the chosen projection is the GEMV, it normalises its own input from
// the residual stream; otherwise the norm kernel writes xn (activation storage) first.
llm_status norm_linear(llm_handle* h, const char* tag, LinearParams p, const void* g, const void* b,
                       bool last_row) {
  const llm_config& c = h->cfg;
  const bool gpt2 = c.arch == LLM_ARCH_GPT2;
  if (!last_row) {
    LinearParams f = p;
    f.xnorm = 1;
    f.X = h->h;
    f.ldx = c.d_model;
    f.xdt = DT_F32;
    f.norm_g = g;
    f.norm_b = gpt2 ? b : nullptr;
    f.norm_eps = c.norm_eps;
    f.norm_ln = gpt2 ? 1 : 0;
    LinearParams plain = p;
    plain.X = h->xn;
    plain.ldx = h->act_mul * c.d_model;
    const int v = pick_variant(h, plain);
    if (v == LIN_GEMV && gemv_norm_supported(f)) return linear_v(h, tag, f, v);
  }
  NormParams np{h->h, g, gpt2 ? b : nullptr, h->xn, h->d_args, p.M, c.d_model, gpt2 ? 1 : 0, last_row ? 1 : 0,
                c.norm_eps};
  // Q8_0 models keep their gains and biases in fp32
  RUN("norm", launch_norm(np, h->wdt == DT_Q8 ? DT_F32 : h->wdt, h->adt, h->stream, h->pdl));
  p.X = h->xn;
  p.ldx = h->act_mul * c.d_model;
  return linear(h, tag, p);
}

// The kernels of one forward pass over M rows (decode: M = B, one row per
// sequence; prefill chunk: the packed prompt rows), reading d_args.
// items != 0 selects prefill attention over `n_items` work items.
// In a prefill pass, the first n_dec sequences (n_dec rows, one token each, rows 0..n_dec-1,
// block-table rows 0..n_dec-1) take the split-K decode attention and the items the rest.
// sample: the step ends in temperature / top-k sampling (StepArgs) instead of the argmax.
llm_status enqueue_forward(llm_handle* h, int M, int B, bool prefill, int n_items, int n_dec = 0,
                           bool sample = false) {
  const llm_config& c = h->cfg;
  const int d = c.d_model, H = c.n_heads, Hkv = c.n_kv_heads, F = c.d_ff;
  const bool gpt2 = c.arch == LLM_ARCH_GPT2;
  const int qkv_n = (H + 2 * Hkv) * HD;

  EmbedParams ep{h->tok_emb, h->tok_scale, gpt2 ? h->pos_emb : nullptr, h->d_args, h->h, M, d, c.vocab, c.n_ctx,
                 h->flags};
  RUN("embed", launch_embed(ep, h->wdt, h->stream, h->pdl));

  for (int l = 0; l < c.n_layers; ++l) {
    const LayerW& w = h->layers[l];
    LinearParams lp;
    memset(&lp, 0, sizeof(lp));
    lp.wdt = h->wdt; lp.xdt = h->adt; lp.adt = h->adt;
    lp.M = M;
    // norm + QKV + RoPE + kv_write
    lp.W = w.w_qkv; lp.Wscale = w.s_qkv; lp.N = qkv_n; lp.K = d; lp.swiglu = 0;
    lp.epi = base_epi(h);
    lp.epi.kind = EPI_QKV;
    lp.epi.bias = w.b_qkv;
    lp.epi.q_out = h->q;
    lp.epi.kv = kv_layer(h, l);
    lp.epi.n_heads = H;
    lp.epi.rope = gpt2 ? 0 : 1;
    lp.epi.rope_theta = c.rope_theta;
    lp.epi.rope_tab = h->d_rope;
    lp.epi.qn_g = w.q_norm_w;
    lp.epi.kn_g = w.k_norm_w;
    lp.epi.qk_eps = c.norm_eps;
    { llm_status s_ = norm_linear(h, "qkv", lp, w.ln1_w, w.ln1_b, false); if (s_ != LLM_OK) return s_; }

    // attention
    if (!prefill || n_dec > 0) {
      AttnDecodeParams ap;
      memset(&ap, 0, sizeof(ap));
      ap.q = h->q; ap.kv = kv_layer(h, l); ap.args = h->d_args; ap.B = prefill ? n_dec : B; ap.n_heads = H;
      ap.split = h->split; ap.max_splits = h->max_splits; ap.part_o = h->attn_po; ap.part_ml = h->attn_ml;
      ap.out = h->att; ap.out_dtype = h->adt; ap.flags = h->flags; ap.window = layer_window(h, l);
      RUN("attn_decode", launch_attn_decode(ap, h->kvdt, h->stream, h->pdl));
    }
    if (prefill && n_items > 0) {
      AttnPrefillParams ap;
      memset(&ap, 0, sizeof(ap));
      ap.q = h->q; ap.kv = kv_layer(h, l); ap.args = h->d_args; ap.items = h->d_items; ap.n_items = n_items;
      ap.n_heads = H; ap.out = h->att; ap.out_dtype = h->adt; ap.flags = h->flags; ap.window = layer_window(h, l);
      // bf16-weight models: tensor cores on bf16 (hi, lo) splits (about 16 bits of every
      // operand); fp32-weight models keep fp32 FMA so their attention stays at fp32 accuracy
      if (h->attn_tc2) RUN("attn_prefill", launch_attn_prefill_tc2(ap, h->kvdt, h->stream, h->pdl));
      else if (h->wdt == DT_BF16) RUN("attn_prefill", launch_attn_prefill_tc(ap, h->kvdt, h->stream, h->pdl));
      else RUN("attn_prefill", launch_attn_prefill(ap, h->kvdt, h->stream, h->pdl));
    }

    // out projection + residual
    lp.W = w.w_o; lp.Wscale = w.s_o; lp.X = h->att; lp.N = d; lp.K = H * HD; lp.ldx = h->act_mul * H * HD;
    lp.epi = base_epi(h);
    lp.epi.kind = EPI_RESID; lp.epi.bias = w.b_o; lp.epi.resid = h->h; lp.epi.ld_resid = d;
    { llm_status s_ = linear(h, "o", lp); if (s_ != LLM_OK) return s_; }

    // norm + FFN up (+gate) with the activation
    lp.W = w.w_up; lp.Wscale = w.s_up; lp.N = F; lp.K = d; lp.swiglu = gpt2 ? 0 : 1;
    lp.epi = base_epi(h);
    lp.epi.kind = gpt2 ? EPI_GELU : EPI_SWIGLU; lp.epi.bias = w.b_up; lp.epi.out = h->ff;
    lp.epi.ld_out = h->act_mul * F;
    { llm_status s_ = norm_linear(h, "up", lp, w.ln2_w, w.ln2_b, false); if (s_ != LLM_OK) return s_; }

    // FFN down + residual
    lp.W = w.w_down; lp.Wscale = w.s_down; lp.X = h->ff; lp.N = d; lp.K = F; lp.ldx = h->act_mul * F; lp.swiglu = 0;
    lp.epi = base_epi(h);
    lp.epi.kind = EPI_RESID; lp.epi.bias = w.b_down; lp.epi.resid = h->h; lp.epi.ld_resid = d;
    { llm_status s_ = linear(h, "down", lp); if (s_ != LLM_OK) return s_; }
  }

  // final norm on each sequence's last row, tied LM head + argmax partials, argmax reduce
  LinearParams hp;
  memset(&hp, 0, sizeof(hp));
  hp.wdt = h->wdt; hp.xdt = h->adt; hp.adt = h->adt;
  hp.W = h->tok_emb; hp.Wscale = h->tok_scale; hp.M = B; hp.N = c.vocab; hp.K = d;
  hp.epi = base_epi(h);
  hp.epi.kind = EPI_HEAD; hp.epi.part_val = h->head_val; hp.epi.part_idx = h->head_idx; hp.epi.vocab = c.vocab;
  { llm_status s_ = norm_linear(h, "head", hp, h->lnf_w, h->lnf_b, prefill); if (s_ != LLM_OK) return s_; }
  if (sample) {
    SampleParams sp{h->d_args, c.vocab, h->flags};
    RUN("sample", launch_sample(sp, B, h->stream, h->pdl));
    return LLM_OK;
  }
  ArgmaxParams amp{h->head_val, h->head_idx, h->head_tiles, h->d_args, h->flags};
  RUN("argmax", launch_argmax(amp, B, h->stream, h->pdl));
  return LLM_OK;
}

// ---- the one-kernel decode step -----------------------------------------------------------

// Ring stages and staged-input capacity of a persistent step of M rows; false when M rows'
// input does not leave room for two stages.
bool pk_plan(const llm_handle* h, int M, int* nslot, int* xs_floats) {
  const llm_config& c = h->cfg;
  const int kmax = std::max(c.d_model, std::max(c.n_heads * HD, c.d_ff));
  const size_t xsb = (size_t)M * kmax * sizeof(float);
  const size_t base = pk_smem_bytes(0, 0);
  if ((size_t)h->pk_smem_max < base + xsb) return false;
  const int ns = (int)std::min<size_t>(PK_MAX_SLOTS, ((size_t)h->pk_smem_max - base - xsb) / PK_SLOT_BYTES);
  if (ns < 2) return false;
  *nslot = ns;
  *xs_floats = M * kmax;
  return true;
}

bool pk_usable(const llm_handle* h, int B) {
  int ns, xs;
  // a forced projection kernel (tests that run every kernel on every shape) keeps one kernel a phase
  return h->pk_supported && h->pk_enabled && h->lin_variant == LIN_AUTO && B >= 1 &&
         B <= std::min(PK_MAX_M, h->cfg.max_batch) &&
         (B == 1 || h->pk_multi) && pk_plan(h, B, &ns, &xs);
}

PKParams pk_params(const llm_handle* h, int M) {
  const llm_config& c = h->cfg;
  const bool gpt2 = c.arch == LLM_ARCH_GPT2;
  PKParams p;
  memset(&p, 0, sizeof(p));
  p.layers = h->d_pk_layers;
  p.n_layers = c.n_layers; p.d = c.d_model; p.H = c.n_heads; p.Hkv = c.n_kv_heads; p.F = c.d_ff;
  p.vocab = c.vocab; p.n_ctx = c.n_ctx; p.gpt2 = gpt2 ? 1 : 0; p.eps = c.norm_eps;
  p.tok_emb = h->tok_emb; p.tok_scale = h->tok_scale; p.pos_emb = gpt2 ? h->pos_emb : nullptr;
  p.lnf_g = h->lnf_w; p.lnf_b = gpt2 ? h->lnf_b : nullptr;
  p.rope_tab = h->d_rope; p.args = h->d_args;
  p.h = h->h; p.qkv = h->pk_qkv; p.att = h->pk_att; p.ff = h->pk_ff; p.part_o = h->pk_po; p.part_ml = h->pk_ml;
  p.max_ch = h->pk_max_ch;
  p.head_val = h->pk_head_val; p.head_idx = h->pk_head_idx;
  p.sync = h->pk_sync; p.flags = h->flags; p.withhold = -1;
  pk_plan(h, M, &p.nslot, &p.xs_floats);
  return p;
}

// Shapes and pointers the persistent kernel handles, its scratch and its layer table. Any
// failure here only leaves the step on the graph of per-phase kernels.
void pk_setup(llm_handle* h) {
  const llm_config& c = h->cfg;
  h->pk_supported = h->pk_multi = false;
  int coop = 0, optin = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->dev) != cudaSuccess || !coop) {
    cudaGetLastError();
    return;
  }
  h->pk_smem_max = optin;
  const bool gpt2 = c.arch == LLM_ARCH_GPT2, q8 = h->wdt == DT_Q8;
  const int elt = h->wdt == DT_F32 ? 4 : h->wdt == DT_BF16 ? 2 : 1;
  const int H = c.n_heads, Hkv = c.n_kv_heads, d = c.d_model, F = c.d_ff;
  // rows are 16-byte vectors (Q8_0: scale rows too, K a multiple of 256)
  for (int K : {d, H * HD, F})
    if (K % 4 != 0 || (K * elt) % 16 != 0 || (q8 && K % 256 != 0)) return;
  if (d > PK_MAX_D || H / Hkv > PK_MAX_G) return;
  // every CTA's share of a matrix's rows fits the staged bias and residual slices
  for (int units : {(H + 2 * Hkv) * HD, d, F})
    if ((units + h->num_sms - 1) / h->num_sms > PK_MAX_UNITS) return;
  auto unit = [&](int K, int rows) { return (size_t)rows * ((size_t)K * elt + (q8 ? (size_t)K / 16 : 0)); };
  if (unit(d, gpt2 ? 1 : 2) > PK_SLOT_BYTES || unit(H * HD, 1) > PK_SLOT_BYTES || unit(F, 1) > PK_SLOT_BYTES) return;
  auto aligned = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!aligned(h->tok_emb) || !aligned(h->tok_scale)) return;
  for (const LayerW& w : h->layers)
    for (const void* p : {w.w_qkv, w.w_o, w.w_up, w.w_down, w.s_qkv, w.s_o, w.s_up, w.s_down})
      if (!aligned(p)) return;
  int ns, xs, nb = 0;
  if (!pk_plan(h, 1, &ns, &xs)) return;
  if (pk_blocks_per_sm(h->wdt, 1, pk_smem_bytes(ns, xs), &nb) != cudaSuccess || nb < 1) {
    cudaGetLastError();
    return;
  }
  const int MM = std::min(c.max_batch, PK_MAX_M);
  if (MM > 1 && pk_plan(h, MM, &ns, &xs)) {
    nb = 0;
    if (pk_blocks_per_sm(h->wdt, MM, pk_smem_bytes(ns, xs), &nb) == cudaSuccess && nb >= 1) h->pk_multi = true;
    cudaGetLastError();
  }
  h->pk_max_ch = (std::min(c.n_ctx, c.max_blocks_per_seq * KVB) + PK_ATT_CH - 1) / PK_ATT_CH;
  if (dev_alloc(h, &h->pk_qkv, (size_t)MM * (H + 2 * Hkv) * HD) != LLM_OK ||
      dev_alloc(h, &h->pk_att, (size_t)MM * H * HD) != LLM_OK || dev_alloc(h, &h->pk_ff, (size_t)MM * F) != LLM_OK ||
      dev_alloc(h, &h->pk_po, (size_t)MM * H * h->pk_max_ch * HD) != LLM_OK ||
      dev_alloc(h, &h->pk_ml, (size_t)MM * H * h->pk_max_ch * 2) != LLM_OK ||
      dev_alloc(h, &h->pk_head_val, (size_t)h->num_sms * MM) != LLM_OK ||
      dev_alloc(h, &h->pk_head_idx, (size_t)h->num_sms * MM) != LLM_OK || dev_alloc(h, &h->pk_sync, 2) != LLM_OK ||
      dev_alloc(h, &h->d_pk_layers, (size_t)c.n_layers) != LLM_OK)
    return;
  std::vector<PKLayer> tab(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerW& w = h->layers[l];
    PKLayer& t = tab[l];
    memset(&t, 0, sizeof(t));
    t.w_qkv = w.w_qkv; t.s_qkv = w.s_qkv; t.b_qkv = w.b_qkv;
    t.w_o = w.w_o; t.s_o = w.s_o; t.b_o = w.b_o;
    t.w_up = w.w_up; t.s_up = w.s_up; t.b_up = w.b_up;
    t.w_down = w.w_down; t.s_down = w.s_down; t.b_down = w.b_down;
    t.ln1_g = w.ln1_w; t.ln1_b = gpt2 ? w.ln1_b : nullptr;
    t.ln2_g = w.ln2_w; t.ln2_b = gpt2 ? w.ln2_b : nullptr;
    t.qn_g = w.q_norm_w; t.kn_g = w.k_norm_w;
    t.kv = kv_layer(h, l);
    t.window = layer_window(h, l);
  }
  if (cudaMemcpy(h->d_pk_layers, tab.data(), tab.size() * sizeof(PKLayer), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  h->pk_supported = true;
  if (const char* env = getenv("LLM_PERSISTENT")) h->pk_enabled = env[0] == '1';
}

// The step as one persistent kernel, then the argmax reduction (or the sampling kernel).
llm_status enqueue_persistent(llm_handle* h, int B, bool sample) {
  const PKParams p = pk_params(h, B);
  CUDA_TRY(cudaMemsetAsync(h->pk_sync, 0, 2 * sizeof(unsigned), h->stream));
  RUN("decode_persistent", launch_decode_persistent(p, h->wdt, B, h->num_sms, h->stream));
  if (sample) {
    SampleParams sp{h->d_args, h->cfg.vocab, h->flags};
    RUN("sample", launch_sample(sp, B, h->stream, h->pdl));
    return LLM_OK;
  }
  ArgmaxParams amp{h->pk_head_val, h->pk_head_idx, h->num_sms, h->d_args, h->flags};
  RUN("argmax", launch_argmax(amp, B, h->stream, h->pdl));
  return LLM_OK;
}

// A decode step's kernels: one persistent kernel where it applies, else one kernel a phase.
llm_status enqueue_decode(llm_handle* h, int B, bool sample) {
  if (pk_usable(h, B)) return enqueue_persistent(h, B, sample);
  return enqueue_forward(h, B, B, false, 0, 0, sample);
}

llm_status check_handle(llm_handle* h) {
  if (!h) return fail(LLM_ERR_INVALID_ARG, "handle is NULL");
  cudaError_t e = cudaSetDevice(h->dev);
  if (e != cudaSuccess) return fail(LLM_ERR_CUDA, cudaGetErrorString(e));
  return LLM_OK;
}

void begin_call(llm_handle* h) { h->launch_counter = 0; }
void end_call(llm_handle* h) { h->last_launches = h->launch_counter; }

bool stream_capturable(cudaStream_t s) { return s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread; }

// A decode step (greedy or sampled): eager, profiled or replayed from the graph cached for
// (B, sampled).
llm_status decode_step_impl(llm_handle* h, const StepArgs& a, bool sample) {
  const int B = a.B;
  llm_status st = LLM_OK;
  begin_call(h);
  if (h->profiling && stream_capturable(h->stream)) {
    // Per-launch timing. Launched one by one, a decode step's kernels are shorter than the
    // host's launch calls, so events around eager launches would time the host. The step is
    // captured with an event record node around every launch instead, and replayed once:
    // the events then time the kernels back to back on the device. Programmatic launch is
    // off in this mode, so each interval holds one kernel alone.
    const bool pdl = h->pdl;
    h->pdl = false;
    h->prof_capture = true;
    const size_t nprof = h->prof.size();
    cudaError_t e = cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal);
    llm_status fs = LLM_ERR_CUDA;
    cudaGraph_t g = nullptr;
    if (e == cudaSuccess) {
      e = launch_set_args(h->d_args, a, h->stream);
      h->launch_counter++;
      fs = e == cudaSuccess ? enqueue_decode(h, B, sample) : LLM_ERR_CUDA;
      const cudaError_t ee = cudaStreamEndCapture(h->stream, &g);
      if (e == cudaSuccess) e = ee;
    }
    h->pdl = pdl;
    h->prof_capture = false;
    cudaGraphExec_t x = nullptr;
    if (e == cudaSuccess && fs == LLM_OK) e = cudaGraphInstantiate(&x, g, 0);
    if (g) cudaGraphDestroy(g);
    if (e == cudaSuccess && fs == LLM_OK) e = cudaGraphLaunch(x, h->stream);
    if (x) cudaGraphExecDestroy(x);   // released once the replay completes
    end_call(h);
    if (fs != LLM_OK || e != cudaSuccess) {
      h->prof.resize(nprof);   // no records of a step that did not run
      if (fs != LLM_OK) return fs;
      cudaGetLastError();
      return fail(LLM_ERR_CUDA, std::string("profiled step: ") + cudaGetErrorString(e));
    }
    return LLM_OK;
  }
  if (!h->use_graphs || h->profiling) {
    CUDA_TRY(launch_set_args(h->d_args, a, h->stream));
    h->launch_counter++;
    st = enqueue_decode(h, B, sample);
    end_call(h);
    return st;
  }
  const bool pk = pk_usable(h, B);
  const int key = B | (sample ? (1 << 24) : 0) | (pk ? (1 << 25) : 0);
  auto it = h->graphs.find(key);
  if (it == h->graphs.end()) {
    GraphEntry ge;
    CUDA_TRY(cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal));
    cudaError_t e = launch_set_args(h->d_args, a, h->stream);
    h->launch_counter++;
    llm_status fs = e == cudaSuccess ? enqueue_decode(h, B, sample) : LLM_ERR_CUDA;
    cudaGraph_t g = nullptr;
    cudaError_t ee = cudaStreamEndCapture(h->stream, &g);
    if (pk && e == cudaSuccess && (fs != LLM_OK || ee != cudaSuccess)) {
      // the persistent kernel could not be captured: the step keeps one kernel a phase
      if (g) cudaGraphDestroy(g);
      cudaGetLastError();
      h->pk_supported = false;
      return decode_step_impl(h, a, sample);
    }
    if (e != cudaSuccess) return fail(LLM_ERR_CUDA, std::string("set_args: ") + cudaGetErrorString(e));
    if (fs != LLM_OK) { if (g) cudaGraphDestroy(g); return fs; }
    if (ee != cudaSuccess) return fail(LLM_ERR_CUDA, std::string("end capture: ") + cudaGetErrorString(ee));
    size_t nroots = 0;
    CUDA_TRY(cudaGraphGetRootNodes(g, nullptr, &nroots));
    std::vector<cudaGraphNode_t> roots(nroots);
    CUDA_TRY(cudaGraphGetRootNodes(g, roots.data(), &nroots));
    if (nroots != 1) { cudaGraphDestroy(g); return fail(LLM_ERR_CUDA, "captured step has more than one root"); }
    ge.graph = g;
    ge.args_node = roots[0];
    CUDA_TRY(cudaGraphInstantiate(&ge.exec, g, 0));
    ge.launches = h->launch_counter;
    it = h->graphs.emplace(key, ge).first;
  }
  cudaKernelNodeParams kp;
  memset(&kp, 0, sizeof(kp));
  StepArgs* dst = h->d_args;
  StepArgs av = a;
  void* params[2] = {&dst, &av};
  kp.func = const_cast<void*>(set_args_kernel());
  kp.gridDim = dim3(1);
  kp.blockDim = dim3(1);
  kp.kernelParams = params;
  CUDA_TRY(cudaGraphExecKernelNodeSetParams(it->second.exec, it->second.args_node, &kp));
  CUDA_TRY(cudaGraphLaunch(it->second.exec, h->stream));
  h->launch_counter = it->second.launches;
  end_call(h);
  return LLM_OK;
}

}  // namespace

extern "C" {

const char* llm_status_string(llm_status s) {
  switch (s) {
    case LLM_OK: return "ok";
    case LLM_ERR_INVALID_ARG: return "invalid argument";
    case LLM_ERR_OUT_OF_RANGE: return "out of range";
    case LLM_ERR_NO_DEVICE: return "no suitable CUDA device";
    case LLM_ERR_UNSUPPORTED: return "unsupported configuration";
    case LLM_ERR_OOM: return "out of device memory";
    case LLM_ERR_CUDA: return "CUDA error";
    case LLM_ERR_DEVICE_FLAG: return "device error flag set";
  }
  return "unknown status";
}

const char* llm_last_error(void) { return g_last_error.c_str(); }

llm_status llm_create(const llm_config* cfgp, const llm_weights* wp, void* cuda_stream, llm_handle** out) {
  if (!out) return fail(LLM_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cfgp || !wp) return fail(LLM_ERR_INVALID_ARG, "config or weights is NULL");
  const llm_config c = *cfgp;
  if (c.arch != LLM_ARCH_GPT2 && c.arch != LLM_ARCH_LLAMA) return fail(LLM_ERR_INVALID_ARG, "bad arch");
  if (c.dtype != LLM_DTYPE_F32 && c.dtype != LLM_DTYPE_BF16 && c.dtype != LLM_DTYPE_Q8)
    return fail(LLM_ERR_INVALID_ARG, "bad dtype");
  const bool q8 = c.dtype == LLM_DTYPE_Q8;
  if (q8 && (c.d_model % 32 != 0 || c.d_ff % 32 != 0))
    return fail(LLM_ERR_UNSUPPORTED, "Q8_0 weights need d_model and d_ff multiples of 32");
  if (q8 && (!wp->tok_emb_scale || !wp->w_qkv_scale || !wp->w_o_scale || !wp->w_up_scale || !wp->w_down_scale))
    return fail(LLM_ERR_INVALID_ARG, "Q8_0 weights need every block-scale array");
  if (c.n_layers <= 0 || c.d_model <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 || c.d_ff <= 0 || c.vocab <= 0 ||
      c.n_ctx <= 0 || c.max_batch <= 0 || c.max_blocks_per_seq <= 0 || c.max_prefill_tokens <= 0)
    return fail(LLM_ERR_INVALID_ARG, "sizes must be positive");
  if (c.head_dim != HD) return fail(LLM_ERR_UNSUPPORTED, "head_dim must be 64");
  if (c.kv_block_size != KVB) return fail(LLM_ERR_UNSUPPORTED, "kv_block_size must be 16");
  if (c.n_heads % c.n_kv_heads != 0) return fail(LLM_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads");
  if (c.n_heads / c.n_kv_heads > 8) return fail(LLM_ERR_UNSUPPORTED, "at most 8 query heads per KV head");
  if (c.d_model > 2048) return fail(LLM_ERR_UNSUPPORTED, "d_model above 2048");
  if (c.d_model % 8 != 0 || c.d_ff % 8 != 0) return fail(LLM_ERR_UNSUPPORTED, "d_model and d_ff must be multiples of 8");
  if (c.arch == LLM_ARCH_LLAMA && !(c.rope_theta > 0.0f)) return fail(LLM_ERR_INVALID_ARG, "rope_theta must be > 0");
  if (!c.contiguous_kv && c.num_kv_blocks <= 0) return fail(LLM_ERR_INVALID_ARG, "num_kv_blocks must be positive");
  if (c.kv_dtype != LLM_DTYPE_F32 && c.kv_dtype != LLM_DTYPE_BF16) return fail(LLM_ERR_INVALID_ARG, "bad kv_dtype");
  if (c.sliding_window < 0 || c.sliding_window_pattern < 0) return fail(LLM_ERR_INVALID_ARG, "negative sliding window");
  if (c.qk_norm && (!wp->q_norm_w || !wp->k_norm_w)) return fail(LLM_ERR_INVALID_ARG, "qk_norm needs q_norm_w and k_norm_w");
  if (c.rope_scale_factor > 1.0f &&
      !(c.rope_original_max_pos > 0 && c.rope_high_freq_factor > c.rope_low_freq_factor && c.rope_low_freq_factor > 0.0f))
    return fail(LLM_ERR_INVALID_ARG, "RoPE scaling needs original_max_pos > 0 and high_freq_factor > low_freq_factor > 0");
  const bool gpt2 = c.arch == LLM_ARCH_GPT2;
  if (!wp->tok_emb || (gpt2 && !wp->pos_emb) || !wp->lnf_w || (gpt2 && !wp->lnf_b))
    return fail(LLM_ERR_INVALID_ARG, "missing embedding or final-norm weights");
  if (!wp->ln1_w || !wp->w_qkv || !wp->w_o || !wp->ln2_w || !wp->w_up || !wp->w_down)
    return fail(LLM_ERR_INVALID_ARG, "missing per-layer weight arrays");
  if (gpt2 && (!wp->ln1_b || !wp->ln2_b || !wp->b_qkv || !wp->b_o || !wp->b_up || !wp->b_down))
    return fail(LLM_ERR_INVALID_ARG, "GPT-2 needs all bias arrays");

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    return fail(LLM_ERR_NO_DEVICE, "no CUDA device");
  }
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return fail(LLM_ERR_NO_DEVICE, "cannot query device");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(LLM_ERR_NO_DEVICE, "the library runs on compute capability 10.3 (GB300) only");

  llm_handle* h = new llm_handle();
  h->cfg = c;
  h->dev = dev;
  h->num_sms = prop.multiProcessorCount;
  h->stream = static_cast<cudaStream_t>(cuda_stream);
  // Only the weights take the model's dtype. Activations keep fp32 accuracy (bf16-weight
  // models store them as bf16 pairs for the tensor cores) and the KV cache is fp32.
  h->wdt = c.dtype == LLM_DTYPE_F32 ? DT_F32 : c.dtype == LLM_DTYPE_Q8 ? DT_Q8 : DT_BF16;
  h->adt = c.dtype == LLM_DTYPE_BF16 ? DT_SPLIT : DT_F32;
  h->tok_scale = q8 ? wp->tok_emb_scale : nullptr;
  h->act_mul = h->adt == DT_SPLIT ? 2 : 1;
  h->kvdt = c.kv_dtype == LLM_DTYPE_BF16 ? DT_BF16 : DT_F32;
  h->kv_elt = h->kvdt == DT_BF16 ? 2 : 4;
  h->tok_emb = wp->tok_emb;
  h->pos_emb = gpt2 ? wp->pos_emb : nullptr;
  h->lnf_w = wp->lnf_w;
  h->lnf_b = gpt2 ? wp->lnf_b : nullptr;
  h->layers.resize(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    LayerW& w = h->layers[l];
    w.ln1_w = wp->ln1_w[l]; w.ln1_b = wp->ln1_b ? wp->ln1_b[l] : nullptr;
    w.w_qkv = wp->w_qkv[l]; w.b_qkv = wp->b_qkv ? wp->b_qkv[l] : nullptr;
    w.w_o = wp->w_o[l]; w.b_o = wp->b_o ? wp->b_o[l] : nullptr;
    w.ln2_w = wp->ln2_w[l]; w.ln2_b = wp->ln2_b ? wp->ln2_b[l] : nullptr;
    w.w_up = wp->w_up[l]; w.b_up = wp->b_up ? wp->b_up[l] : nullptr;
    w.w_down = wp->w_down[l]; w.b_down = wp->b_down ? wp->b_down[l] : nullptr;
    w.s_qkv = q8 ? wp->w_qkv_scale[l] : nullptr;
    w.s_o = q8 ? wp->w_o_scale[l] : nullptr;
    w.s_up = q8 ? wp->w_up_scale[l] : nullptr;
    w.s_down = q8 ? wp->w_down_scale[l] : nullptr;
    if (q8 && (!w.s_qkv || !w.s_o || !w.s_up || !w.s_down)) {
      delete h;
      return fail(LLM_ERR_INVALID_ARG, "NULL Q8_0 scale array in layer " + std::to_string(l));
    }
    w.q_norm_w = c.qk_norm ? wp->q_norm_w[l] : nullptr;
    w.k_norm_w = c.qk_norm ? wp->k_norm_w[l] : nullptr;
    // the Llama variant has no biases but the optional attention (q, k, v) biases
    if (!gpt2) { w.ln1_b = w.b_o = w.ln2_b = w.b_up = w.b_down = nullptr; }
    if (c.qk_norm && (!w.q_norm_w || !w.k_norm_w)) {
      delete h;
      return fail(LLM_ERR_INVALID_ARG, "NULL Q/K-norm gain in layer " + std::to_string(l));
    }
    if (!w.ln1_w || !w.w_qkv || !w.w_o || !w.ln2_w || !w.w_up || !w.w_down ||
        (gpt2 && (!w.ln1_b || !w.b_qkv || !w.b_o || !w.ln2_b || !w.b_up || !w.b_down))) {
      delete h;
      return fail(LLM_ERR_INVALID_ARG, "NULL weight pointer in layer " + std::to_string(l));
    }
  }

  const int H = c.n_heads, Hkv = c.n_kv_heads, d = c.d_model, F = c.d_ff;
  h->num_blocks = c.contiguous_kv ? c.max_batch * c.max_blocks_per_seq : c.num_kv_blocks;
  h->layer_kv_elems = (size_t)h->num_blocks * Hkv * KVB * HD;
  h->max_rows = std::max(c.max_batch, c.max_prefill_tokens);
  const int max_ctx = std::min(c.n_ctx, c.max_blocks_per_seq * KVB);
  h->split = attn_decode_split_for(c.max_batch, c.n_kv_heads, max_ctx, h->num_sms);
  h->max_splits = std::max(1, (max_ctx + h->split - 1) / h->split);
  h->head_tiles = (c.vocab + TILE_N - 1) / TILE_N;
  h->max_items = c.max_prefill_tokens / 64 + c.max_batch + 1;
  const size_t act = 4;   // bytes per activation value: fp32, or a bf16 pair
  const size_t R = h->max_rows;
  llm_status st = LLM_OK;
#define ALLOC(ptr, T, n)                                                         \
  do {                                                                           \
    st = dev_alloc(h, reinterpret_cast<T**>(&(ptr)), (size_t)(n));               \
    if (st != LLM_OK) { free_all(h); delete h; return st; }                      \
  } while (0)
  ALLOC(h->k_pool, char, (size_t)c.n_layers * h->layer_kv_elems * h->kv_elt);
  ALLOC(h->v_pool, char, (size_t)c.n_layers * h->layer_kv_elems * h->kv_elt);
  ALLOC(h->h, float, R * d);
  ALLOC(h->xn, char, R * d * act);
  ALLOC(h->q, float, R * H * HD);
  ALLOC(h->att, char, R * H * HD * act);
  ALLOC(h->ff, char, R * F * act);
  ALLOC(h->attn_po, float, (size_t)c.max_batch * H * h->max_splits * HD);
  ALLOC(h->attn_ml, float, (size_t)c.max_batch * H * h->max_splits * 2);
  ALLOC(h->head_val, float, (size_t)h->head_tiles * R);
  ALLOC(h->head_idx, int, (size_t)h->head_tiles * R);
  ALLOC(h->flags, unsigned, 1);
  ALLOC(h->d_args, StepArgs, 1);
  ALLOC(h->d_row_pos, int, R);
  ALLOC(h->d_row_seq, int, R);
  ALLOC(h->d_last_row, int, c.max_batch);
  ALLOC(h->d_items, int4, h->max_items);
  ALLOC(h->d_host_tokens, int, c.max_batch);
  ALLOC(h->d_host_pos, int, c.max_batch);
  ALLOC(h->d_host_tables, int, (size_t)c.max_batch * c.max_blocks_per_seq);
  ALLOC(h->d_host_ids, int, c.max_batch);
  ALLOC(h->d_host_logits, float, (size_t)c.max_batch * c.vocab);
  ALLOC(h->d_samp_logits, float, (size_t)c.max_batch * c.vocab);
  ALLOC(h->d_rope, float2, HD / 2);
#undef ALLOC
  {
    // inverse frequency theta^(-2d/64) of RoPE pair d, split into hi (11 significant bits:
    // pos * hi is exact in fp32 for pos < 2^13) + lo, computed once here in double
    float2 tab[HD / 2];
    for (int d = 0; d < HD / 2; ++d) {
      double f = gpt2 ? 0.0 : pow((double)c.rope_theta, -2.0 * d / HD);
      if (!gpt2 && c.rope_scale_factor > 1.0f) {
        // Llama 3 frequency scaling: long wavelengths slowed by the factor, short ones kept,
        // a linear blend between the two bands
        const double pi = 3.14159265358979323846, orig = c.rope_original_max_pos;
        const double lo = c.rope_low_freq_factor, hi = c.rope_high_freq_factor, wl = 2.0 * pi / f;
        if (wl > orig / lo) {
          f = f / c.rope_scale_factor;
        } else if (wl >= orig / hi) {
          const double sm = (orig / wl - lo) / (hi - lo);
          f = (1.0 - sm) * f / c.rope_scale_factor + sm * f;
        }
      }
      float hi = (float)f;
      uint32_t bits;
      memcpy(&bits, &hi, 4);
      bits &= 0xFFFFE000u;   // keep 10 explicit mantissa bits (11 significant)
      memcpy(&hi, &bits, 4);
      tab[d] = make_float2(hi, (float)(f - (double)hi));
    }
    if (cudaMemcpy(h->d_rope, tab, sizeof(tab), cudaMemcpyHostToDevice) != cudaSuccess) {
      free_all(h);
      delete h;
      return fail(LLM_ERR_CUDA, "copy of the RoPE table failed");
    }
  }
  if (!stream_capturable(h->stream)) h->use_graphs = false;
  if (const char* env = getenv("LLM_NO_GRAPH")) h->use_graphs = h->use_graphs && env[0] != '1';
  if (const char* env = getenv("LLM_PDL")) h->pdl = env[0] != '0';
  // bf16-weight models without a sliding window take the warp-specialised prefill attention
  // (LLM_PREFILL_ATTN=1 keeps the earlier kernel, for comparisons)
  h->attn_tc2 = h->wdt == DT_BF16 && c.sliding_window == 0;
  if (const char* env = getenv("LLM_PREFILL_ATTN")) h->attn_tc2 = h->attn_tc2 && env[0] != '1';
  if (const char* env = getenv("LLM_GEMM_PAIR")) h->gemm_pair = env[0] != '0';
  pk_setup(h);
  *out = h;
  return LLM_OK;
}

void llm_destroy(llm_handle* h) {
  if (!h) return;
  cudaSetDevice(h->dev);
  cudaStreamSynchronize(h->stream);
  free_all(h);
  delete h;
}


llm_status llm_decode_step(llm_handle* h, const int32_t* tokens, const int32_t* positions, const int32_t* tables,
                           int B, int32_t* next_ids, float* logits) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  if (B <= 0) return fail(LLM_ERR_INVALID_ARG, "B must be positive");
  if (B > h->cfg.max_batch) return fail(LLM_ERR_OUT_OF_RANGE, "B exceeds max_batch");
  if (!tokens || !positions || !next_ids) return fail(LLM_ERR_INVALID_ARG, "NULL tokens/positions/next_ids");
  if (!tables && !h->cfg.contiguous_kv) return fail(LLM_ERR_INVALID_ARG, "NULL block_tables");
  StepArgs a{tokens, positions, nullptr, tables, next_ids, logits, nullptr, B, B, nullptr, 0.0f, 1};
  return decode_step_impl(h, a, false);
}

llm_status llm_decode_step_sample(llm_handle* h, const int32_t* tokens, const int32_t* positions,
                                  const int32_t* tables, int B, float temperature, int top_k, const float* uniforms,
                                  int32_t* next_ids, float* logits) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  if (B <= 0) return fail(LLM_ERR_INVALID_ARG, "B must be positive");
  if (B > h->cfg.max_batch) return fail(LLM_ERR_OUT_OF_RANGE, "B exceeds max_batch");
  if (!tokens || !positions || !next_ids) return fail(LLM_ERR_INVALID_ARG, "NULL tokens/positions/next_ids");
  if (!tables && !h->cfg.contiguous_kv) return fail(LLM_ERR_INVALID_ARG, "NULL block_tables");
  if (!(temperature >= 0.0f) || !std::isfinite(temperature)) return fail(LLM_ERR_INVALID_ARG, "temperature must be finite and >= 0");
  if (top_k < 1 || top_k > SAMPLE_MAX_K) return fail(LLM_ERR_INVALID_ARG, "top_k must be in 1..64");
  StepArgs a{tokens, positions, nullptr, tables, next_ids, logits ? logits : h->d_samp_logits, nullptr, B, B,
             uniforms, temperature, top_k};
  return decode_step_impl(h, a, true);
}

llm_status llm_step(llm_handle* h, const int32_t* tokens, const int32_t* lengths, const int32_t* starts,
                    const int32_t* tables, int B, int32_t* next_ids, float* logits) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  const llm_config& c = h->cfg;
  if (B <= 0) return fail(LLM_ERR_INVALID_ARG, "B must be positive");
  if (B > c.max_batch) return fail(LLM_ERR_OUT_OF_RANGE, "B exceeds max_batch");
  if (!tokens || !lengths || !next_ids) return fail(LLM_ERR_INVALID_ARG, "NULL tokens/lengths/next_ids");
  if (!tables && !c.contiguous_kv) return fail(LLM_ERR_INVALID_ARG, "NULL block_tables");
  for (int b = 0; b < B; ++b) {
    const int L = lengths[b], P = starts ? starts[b] : 0;
    if (L <= 0) return fail(LLM_ERR_INVALID_ARG, "length must be positive");
    if (P < 0) return fail(LLM_ERR_INVALID_ARG, "start position must be >= 0");
    if (L > c.max_prefill_tokens) return fail(LLM_ERR_OUT_OF_RANGE, "more tokens than max_prefill_tokens");
    if ((long long)P + L > c.n_ctx) return fail(LLM_ERR_OUT_OF_RANGE, "start + length beyond n_ctx");
    if ((P + L + KVB - 1) / KVB > c.max_blocks_per_seq)
      return fail(LLM_ERR_OUT_OF_RANGE, "sequence needs more blocks than max_blocks_per_seq");
  }
  begin_call(h);
  // query rows per prefill-attention CTA
  const int item_rows = h->attn_tc2 ? 256 : h->wdt == DT_BF16 ? 128 : 64;
  size_t tok_off = 0;
  int s0 = 0;
  while (s0 < B) {
    int s1 = s0, rows = 0;
    while (s1 < B && rows + lengths[s1] <= c.max_prefill_tokens) rows += lengths[s1++];
    const int nb = s1 - s0;
    // a leading run of one-token sequences in the first chunk (decode rows: row b is sequence b)
    // takes the split-K decode attention; every other sequence is cut into query tiles
    int n_dec = 0;
    if (s0 == 0)
      while (n_dec < nb && lengths[n_dec] == 1) ++n_dec;
    std::vector<int> row_pos(rows), row_seq(rows), last_row(nb);
    std::vector<int4> items;
    int r = 0;
    for (int b = s0; b < s1; ++b) {
      const int L = lengths[b], P = starts ? starts[b] : 0;
      for (int t = 0; t < L; ++t) { row_pos[r + t] = P + t; row_seq[r + t] = b; }
      if (b - s0 >= n_dec)
        for (int q0 = 0; q0 < L; q0 += item_rows) items.push_back(make_int4(b, P + q0, r + q0, P + L));
      r += L;
      last_row[b - s0] = r - 1;
    }
    if ((int)items.size() > h->max_items) { end_call(h); return fail(LLM_ERR_OUT_OF_RANGE, "too many attention tiles"); }
    // longest tiles (most keys) first, so the short ones fill the last wave
    std::stable_sort(items.begin(), items.end(), [&](const int4& x, const int4& y) {
      return std::min(x.w, x.y + item_rows) > std::min(y.w, y.y + item_rows);
    });
    CUDA_TRY(cudaMemcpyAsync(h->d_row_pos, row_pos.data(), rows * sizeof(int), cudaMemcpyHostToDevice, h->stream));
    CUDA_TRY(cudaMemcpyAsync(h->d_row_seq, row_seq.data(), rows * sizeof(int), cudaMemcpyHostToDevice, h->stream));
    CUDA_TRY(cudaMemcpyAsync(h->d_last_row, last_row.data(), nb * sizeof(int), cudaMemcpyHostToDevice, h->stream));
    if (!items.empty())
      CUDA_TRY(cudaMemcpyAsync(h->d_items, items.data(), items.size() * sizeof(int4), cudaMemcpyHostToDevice, h->stream));
    StepArgs a{tokens + tok_off, h->d_row_pos, h->d_row_seq, tables, next_ids + s0,
               logits ? logits + (size_t)s0 * c.vocab : nullptr, h->d_last_row, rows, nb};
    CUDA_TRY(launch_set_args(h->d_args, a, h->stream));
    h->launch_counter++;
    st = enqueue_forward(h, rows, nb, true, (int)items.size(), n_dec);
    if (st != LLM_OK) { end_call(h); return st; }
    tok_off += rows;
    s0 = s1;
  }
  end_call(h);
  return LLM_OK;
}

llm_status llm_prefill(llm_handle* h, const int32_t* tokens, const int32_t* lengths, const int32_t* tables, int B,
                       int32_t* next_ids, float* logits) {
  return llm_step(h, tokens, lengths, nullptr, tables, B, next_ids, logits);
}

llm_status llm_decode_step_host(llm_handle* h, const int32_t* tokens, const int32_t* positions,
                                const int32_t* tables, int B, int32_t* next_ids, float* logits) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  if (B <= 0) return fail(LLM_ERR_INVALID_ARG, "B must be positive");
  if (B > h->cfg.max_batch) return fail(LLM_ERR_OUT_OF_RANGE, "B exceeds max_batch");
  if (!tokens || !positions || !next_ids) return fail(LLM_ERR_INVALID_ARG, "NULL tokens/positions/next_ids");
  const bool need_tables = !h->cfg.contiguous_kv;
  if (need_tables && !tables) return fail(LLM_ERR_INVALID_ARG, "NULL block_tables");
  CUDA_TRY(cudaMemcpyAsync(h->d_host_tokens, tokens, B * sizeof(int), cudaMemcpyHostToDevice, h->stream));
  CUDA_TRY(cudaMemcpyAsync(h->d_host_pos, positions, B * sizeof(int), cudaMemcpyHostToDevice, h->stream));
  if (need_tables)
    CUDA_TRY(cudaMemcpyAsync(h->d_host_tables, tables, (size_t)B * h->cfg.max_blocks_per_seq * sizeof(int),
                             cudaMemcpyHostToDevice, h->stream));
  st = llm_decode_step(h, h->d_host_tokens, h->d_host_pos, need_tables ? h->d_host_tables : nullptr, B,
                       h->d_host_ids, logits ? h->d_host_logits : nullptr);
  if (st != LLM_OK) return st;
  CUDA_TRY(cudaMemcpyAsync(next_ids, h->d_host_ids, B * sizeof(int), cudaMemcpyDeviceToHost, h->stream));
  if (logits)
    CUDA_TRY(cudaMemcpyAsync(logits, h->d_host_logits, (size_t)B * h->cfg.vocab * sizeof(float),
                             cudaMemcpyDeviceToHost, h->stream));
  CUDA_TRY(cudaStreamSynchronize(h->stream));
  return LLM_OK;
}

llm_status llm_get_error_flags(llm_handle* h, uint32_t* flags) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  if (!flags) return fail(LLM_ERR_INVALID_ARG, "flags is NULL");
  CUDA_TRY(cudaStreamSynchronize(h->stream));
  unsigned v = 0;
  CUDA_TRY(cudaMemcpy(&v, h->flags, sizeof(v), cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemset(h->flags, 0, sizeof(unsigned)));
  *flags = v;
  return v ? fail(LLM_ERR_DEVICE_FLAG, "device error flags 0x" + std::to_string(v)) : LLM_OK;
}

llm_status llm_selftest_wait_timeout(llm_handle* h) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  CUDA_TRY(launch_selftest_wait(h->flags, h->stream));
  return LLM_OK;
}

llm_status llm_set_profiling(llm_handle* h, int enable) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  h->profiling = enable != 0;
  return LLM_OK;
}

llm_status llm_get_kernel_stats(llm_handle* h, llm_kernel_stat* out, int max, int* n, int reset) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  if (!n || (max > 0 && !out)) return fail(LLM_ERR_INVALID_ARG, "NULL output");
  CUDA_TRY(cudaStreamSynchronize(h->stream));
  for (auto& r : h->prof) {
    float ms = 0.0f;
    CUDA_TRY(cudaEventElapsedTime(&ms, r.a, r.b));
    Stat& s = h->stats[r.name];
    s.launches++;
    s.ms += ms;
  }
  h->prof.clear();
  h->event_next = 0;
  int i = 0;
  for (auto& kv : h->stats) {
    if (i >= max) break;
    memset(&out[i], 0, sizeof(out[i]));
    strncpy(out[i].name, kv.first.c_str(), sizeof(out[i].name) - 1);
    out[i].launches = kv.second.launches;
    out[i].total_ms = kv.second.ms;
    ++i;
  }
  *n = i;
  if (reset) h->stats.clear();
  return LLM_OK;
}

llm_status llm_last_launch_count(llm_handle* h, int* n) {
  if (!h || !n) return fail(LLM_ERR_INVALID_ARG, "NULL argument");
  *n = h->last_launches;
  return LLM_OK;
}

llm_status llm_set_graphs(llm_handle* h, int enable) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  h->use_graphs = enable != 0 && stream_capturable(h->stream);
  return LLM_OK;
}

llm_status llm_set_persistent(llm_handle* h, int enable, int* supported) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  h->pk_enabled = enable != 0;
  if (supported) *supported = h->pk_supported ? 1 : 0;
  return LLM_OK;
}

llm_status llm_selftest_grid_barrier(llm_handle* h) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  if (!h->pk_supported) return fail(LLM_ERR_UNSUPPORTED, "the persistent decode step does not apply to this model");
  PKParams p = pk_params(h, 1);
  p.withhold = 0;
  CUDA_TRY(cudaMemsetAsync(h->pk_sync, 0, 2 * sizeof(unsigned), h->stream));
  CUDA_TRY(launch_decode_persistent(p, h->wdt, 1, h->num_sms, h->stream));
  CUDA_TRY(cudaStreamSynchronize(h->stream));
  return LLM_OK;
}

llm_status llm_op_linear(int dtype, int M, int N, int K, const void* x, const void* w, const void* bias, float* y,
                         int variant, void* cuda_stream) {
  if (M <= 0 || N <= 0 || K <= 0) return fail(LLM_ERR_INVALID_ARG, "sizes must be positive");
  if (!x || !w || !y) return fail(LLM_ERR_INVALID_ARG, "NULL x, w or y");
  if (dtype != LLM_DTYPE_F32 && dtype != LLM_DTYPE_BF16) return fail(LLM_ERR_INVALID_ARG, "bad dtype");
  if (variant < LIN_GEMV || variant > LIN_TC_PAIR) return fail(LLM_ERR_INVALID_ARG, "variant must be 1..5");
  if ((variant == LIN_TC || variant == LIN_TC_PAIR) && dtype != LLM_DTYPE_BF16)
    return fail(LLM_ERR_UNSUPPORTED, "tcgen05 path is bf16 only");
  if ((variant == LIN_TC || variant == LIN_TC_SWAP || variant == LIN_TC_PAIR) && K % 8 != 0)
    return fail(LLM_ERR_INVALID_ARG, "tcgen05 paths need K % 8 == 0");
  if (variant == LIN_TC_SWAP && M > 256) return fail(LLM_ERR_INVALID_ARG, "weights-on-M tcgen05 path needs M <= 256");
  int dev = 0, nsm = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  LinearParams p;
  memset(&p, 0, sizeof(p));
  p.W = w; p.X = x; p.M = M; p.N = N; p.K = K;
  p.wdt = dtype == LLM_DTYPE_F32 ? DT_F32 : DT_BF16;
  p.xdt = p.adt = dtype == LLM_DTYPE_F32 ? DT_F32 : DT_SPLIT;
  p.ldx = dtype == LLM_DTYPE_F32 ? K : 2 * K;
  p.epi.kind = EPI_STORE_F32;
  p.epi.bias = bias;
  p.epi.out = y;
  p.epi.ld_out = N;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = variant == LIN_GEMV ? launch_gemv(p, nsm, s, false)
                  : variant == LIN_SIMT ? launch_gemm_simt(p, s, false)
                  : variant == LIN_TC   ? launch_gemm_tc(p, nsm, s, false)
                  : variant == LIN_TC_PAIR ? launch_gemm_tc2(p, nsm, s, false)
                                        : launch_gemm_tc_swap(p, nsm, s, false);
  if (e != cudaSuccess) return fail(LLM_ERR_CUDA, std::string("llm_op_linear: ") + cudaGetErrorString(e));
  return LLM_OK;
}

llm_status llm_op_linear_q8(int M, int N, int K, const float* x, const void* wq, const void* wscale,
                            const float* bias, float* y, int variant, void* cuda_stream) {
  if (M <= 0 || N <= 0 || K <= 0) return fail(LLM_ERR_INVALID_ARG, "sizes must be positive");
  if (!x || !wq || !wscale || !y) return fail(LLM_ERR_INVALID_ARG, "NULL x, wq, wscale or y");
  if (K % 32 != 0) return fail(LLM_ERR_INVALID_ARG, "Q8_0 needs K % 32 == 0");
  if (variant != LIN_GEMV && variant != LIN_SIMT) return fail(LLM_ERR_INVALID_ARG, "variant must be 1 or 2");
  int dev = 0, nsm = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  LinearParams p;
  memset(&p, 0, sizeof(p));
  p.W = wq; p.Wscale = wscale; p.X = x; p.M = M; p.N = N; p.K = K; p.ldx = K;
  p.wdt = DT_Q8; p.xdt = p.adt = DT_F32;
  p.epi.kind = EPI_STORE_F32;
  p.epi.bias = bias;
  p.epi.out = y;
  p.epi.ld_out = N;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = variant == LIN_GEMV ? launch_gemv(p, nsm, s, false) : launch_gemm_simt(p, s, false);
  if (e != cudaSuccess) return fail(LLM_ERR_CUDA, std::string("llm_op_linear_q8: ") + cudaGetErrorString(e));
  return LLM_OK;
}

llm_status llm_op_attention_decode(int kv_dtype, int B, int n_heads, int n_kv_heads, const float* q,
                                   const void* k_pool, const void* v_pool, int num_blocks, const int32_t* positions,
                                   const int32_t* block_tables, int max_blocks_per_seq, float* out,
                                   void* cuda_stream) {
  if (B <= 0 || n_heads <= 0 || n_kv_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
    return fail(LLM_ERR_INVALID_ARG, "sizes must be positive");
  if (!q || !k_pool || !v_pool || !positions || !block_tables || !out)
    return fail(LLM_ERR_INVALID_ARG, "NULL pointer argument");
  if (kv_dtype != LLM_DTYPE_F32 && kv_dtype != LLM_DTYPE_BF16) return fail(LLM_ERR_INVALID_ARG, "bad kv_dtype");
  if (n_heads % n_kv_heads != 0 || n_heads / n_kv_heads > 8)
    return fail(LLM_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads, at most 8 per KV head");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  int dev = 0, sms = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int split = attn_decode_split_for(B, n_kv_heads, max_blocks_per_seq * KVB, sms);
  const int max_splits = (max_blocks_per_seq * KVB + split - 1) / split;
  const size_t part_o = (size_t)B * n_heads * max_splits * HD, part_ml = (size_t)B * n_heads * max_splits * 2;
  char* scratch = nullptr;
  const size_t bytes = 256 + (part_o + part_ml) * sizeof(float);
  if (cudaMallocAsync(reinterpret_cast<void**>(&scratch), bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return fail(LLM_ERR_OOM, "cudaMallocAsync of the attention scratch failed");
  }
  StepArgs* args = reinterpret_cast<StepArgs*>(scratch);
  StepArgs a{nullptr, positions, nullptr, block_tables, nullptr, nullptr, nullptr, B, B};
  AttnDecodeParams p;
  memset(&p, 0, sizeof(p));
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
  p.part_o = reinterpret_cast<float*>(scratch + 256);
  p.part_ml = p.part_o + part_o;
  p.out = out;
  p.out_dtype = DT_F32;
  p.flags = nullptr;
  cudaError_t e = launch_set_args(args, a, s);
  if (e == cudaSuccess) e = launch_attn_decode(p, kv_dtype == LLM_DTYPE_F32 ? DT_F32 : DT_BF16, s, false);
  cudaError_t ef = cudaFreeAsync(scratch, s);
  if (e != cudaSuccess) return fail(LLM_ERR_CUDA, std::string("llm_op_attention_decode: ") + cudaGetErrorString(e));
  if (ef != cudaSuccess) return fail(LLM_ERR_CUDA, std::string("cudaFreeAsync: ") + cudaGetErrorString(ef));
  return LLM_OK;
}

llm_status llm_set_linear_variant(llm_handle* h, int variant) {
  llm_status st = check_handle(h);
  if (st != LLM_OK) return st;
  if (variant < LIN_AUTO || variant > LIN_TC_PAIR) return fail(LLM_ERR_INVALID_ARG, "variant must be 0..5");
  CUDA_TRY(cudaStreamSynchronize(h->stream));
  for (auto& kv : h->graphs) {
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
    if (kv.second.graph) cudaGraphDestroy(kv.second.graph);
  }
  h->graphs.clear();
  h->lin_variant = variant;
  return LLM_OK;
}

}  // extern "C"
