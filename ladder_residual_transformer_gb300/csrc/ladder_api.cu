// Host side of libladder.so: argument validation, workspace plan, the module
// schedule of the ladder residual, and the launch sequences of prefill and
// decode.  See include/ladder.h for the contract of every entry point.
#include "ladder.h"
#include "internal.cuh"

#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

using namespace ladder;

// ---------------------------------------------------------------------------
// Errors
// ---------------------------------------------------------------------------
static thread_local std::string g_last_error;

static int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

namespace ladder {
// Records `msg` as the last error of this thread and returns `code` (used by other translation units).
int set_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace ladder

#define CUDA_TRY(expr)                                                                          \
  do {                                                                                          \
    cudaError_t e_ = (expr);                                                                    \
    if (e_ != cudaSuccess) return fail(LADDER_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

// ---------------------------------------------------------------------------
// Workspace plan
// ---------------------------------------------------------------------------
namespace {

constexpr int kSplitLen = 128;      // keys per decode-attention split
constexpr int kArgmaxBlocks = 64;   // partial argmax blocks per sequence
// Largest decode projection (weight bytes) launched with programmatic dependent launch.
constexpr size_t kPdlMaxWeightBytes = (size_t)128 << 20;
constexpr size_t kPdlMaxMlpWeightBytes = (size_t)256 << 20;  // the MLP chain's limit at one or two rows
// Decode carveout rule (see ladder_model::gemv_carve): 8.4 MB (1.2B) off, 33.5 MB (8B) on.
constexpr size_t kCarveoutMinWeightBytes = (size_t)16 << 20;

// Split-K workspace of the batched decode projections (B > 2), one region per
// projection kind so that the two decode streams never share one.
enum SplitKKind { SK_QKV = 0, SK_OUT = 1, SK_GATEUP = 2, SK_DOWN = 3, SK_LMHEAD = 4, SK_KINDS = 5 };

struct Plan {
  size_t x[3], xn[2], ssq[3], q, ao, act, part_o, part_ml, am_v, am_i, rope_cos, rope_sin, meta, xlast, err, shard;
  size_t sk[SK_KINDS], sk_bytes[SK_KINDS];
  size_t total;
  int m_max, m_pad, nsplit_max;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

Plan make_plan(const ladder_config& c) {
  Plan p{};
  const size_t d = c.d_model, qd = (size_t)c.n_q_heads * c.head_dim, f = c.ffn_dim;
  p.m_max = c.max_prefill_tokens > c.max_batch ? c.max_prefill_tokens : c.max_batch;
  p.nsplit_max = (c.max_seq + kSplitLen - 1) / kSplitLen;
  p.m_pad = (p.m_max + 127) / 128 * 128;  // tensor-core operands are read in 128-row tiles
  const size_t M = p.m_max, Mp = p.m_pad, Bm = c.max_batch;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  for (int i = 0; i < 3; ++i) p.x[i] = take(M * d * 4);
  // Prefill GEMM A operands: a hi plane [Mp][K] and a lo plane [Mp][K] (the
  // 16-bit rounding remainders) right after it; decode reuses ao / act as fp32 rows.
  // The normalised-row operands x ⊙ g come in two slots (module c uses slot c % 2,
  // see ladder_prefill), and the per-chunk sums of squares of the stream states in
  // three (state j uses slot j % 3), [d / 128][Mp] fp32.
  for (int i = 0; i < 2; ++i) p.xn[i] = take(2 * Mp * d * 2);
  for (int i = 0; i < 3; ++i) p.ssq[i] = take(d / 128 * Mp * 4);
  p.q = take(std::max(Mp * qd * 2, Bm * qd * 4));
  p.ao = take(std::max(2 * Mp * qd * 2, Bm * qd * 4));
  p.act = take(std::max(2 * Mp * f * 2, Bm * f * 4));
  p.part_o = take(Bm * c.n_q_heads * (size_t)p.nsplit_max * c.head_dim * 4);
  p.part_ml = take(Bm * c.n_q_heads * (size_t)p.nsplit_max * 2 * 4);
  p.am_v = take(Bm * kArgmaxBlocks * 4);
  p.am_i = take(Bm * kArgmaxBlocks * 4);
  p.rope_cos = take((size_t)c.max_seq * (c.head_dim / 2) * 4);
  p.rope_sin = take((size_t)c.max_seq * (c.head_dim / 2) * 4);
  p.meta = take((2 * M + 3 * Bm) * 4);
  p.xlast = take(Bm * d * 4);
  p.err = take(256);
  p.shard = c.shard_k > 1 ? take(2 * Bm * c.shard_k * d * 4) : 0;  // double-buffered shard partials [B][k][d]
  if (c.max_batch > 2) {  // batched decode projections (3 rows and more) split K across CTAs
    const size_t kvd = (size_t)c.n_kv_heads * c.head_dim;
    const int nt[SK_KINDS] = {(int)((qd + 2 * kvd) / 2), (int)(d / 2), (int)f, (int)(d / 2), c.vocab / 2};
    const int kk[SK_KINDS] = {(int)d, (int)qd, (int)d, (int)f, (int)d};
    for (int i = 0; i < SK_KINDS; ++i) {
      p.sk_bytes[i] = gemv_splitk_bytes(nt[i], kk[i]);
      p.sk[i] = take(p.sk_bytes[i]);
    }
  }
  p.total = off;
  return p;
}

int validate_config(const ladder_config* c) {
  if (!c) return fail(LADDER_ERR_INVALID, "config is NULL");
  if (c->n_layers <= 0 || c->n_standard_layers < 0 || c->n_standard_layers > c->n_layers)
    return fail(LADDER_ERR_INVALID, "n_layers=%d n_standard_layers=%d out of range", c->n_layers, c->n_standard_layers);
  if (c->d_model <= 0 || c->d_model % 256)
    return fail(LADDER_ERR_INVALID, "d_model=%d must be a positive multiple of 256", c->d_model);
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(LADDER_ERR_UNSUPPORTED, "head_dim=%d: only 64 and 128 are supported", c->head_dim);
  if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->n_q_heads % c->n_kv_heads)
    return fail(LADDER_ERR_INVALID, "n_q_heads=%d must be a positive multiple of n_kv_heads=%d", c->n_q_heads, c->n_kv_heads);
  if (c->n_q_heads / c->n_kv_heads > 8)
    return fail(LADDER_ERR_UNSUPPORTED, "more than 8 query heads per KV head");
  if ((c->n_q_heads * c->head_dim) % 256)
    return fail(LADDER_ERR_INVALID, "n_q_heads*head_dim=%d must be a multiple of 256", c->n_q_heads * c->head_dim);
  if (c->ffn_dim <= 0 || c->ffn_dim % 256)
    return fail(LADDER_ERR_INVALID, "ffn_dim=%d must be a positive multiple of 256", c->ffn_dim);
  if (c->vocab <= 0 || c->vocab % 2) return fail(LADDER_ERR_INVALID, "vocab=%d must be positive and even", c->vocab);
  if (!(c->rope_theta > 1.0f) || !std::isfinite(c->rope_theta))
    return fail(LADDER_ERR_INVALID, "rope_theta must be finite and > 1");
  if (c->rope_scale_factor > 1.0f &&
      (!std::isfinite(c->rope_scale_factor) || !(c->rope_low_freq_factor > 0.0f) ||
       !(c->rope_high_freq_factor > c->rope_low_freq_factor) || !std::isfinite(c->rope_high_freq_factor) ||
       c->rope_original_max_pos <= 0))
    return fail(LADDER_ERR_INVALID, "rope scaling needs 0 < low_freq_factor < high_freq_factor and original_max_pos > 0");
  if (!(c->norm_eps > 0.0f) || !std::isfinite(c->norm_eps)) return fail(LADDER_ERR_INVALID, "norm_eps must be > 0");
  if (c->rope_interleaved != 1)
    return fail(LADDER_ERR_UNSUPPORTED, "only interleaved rotary pairs (rope_interleaved=1) are implemented");
  if (c->shard_k != 1 && c->shard_k != 2 && c->shard_k != 4 && c->shard_k != 8)
    return fail(LADDER_ERR_INVALID, "shard_k=%d must be 1, 2, 4 or 8", c->shard_k);
  if (c->shard_k > 1) {
    const int k = c->shard_k;
    if (c->n_q_heads % k || c->n_kv_heads % k)
      return fail(LADDER_ERR_INVALID, "shard_k=%d must divide n_q_heads and n_kv_heads", k);
    if ((c->n_q_heads * c->head_dim / k) % 256 || (c->ffn_dim / k) % 256 || c->ffn_dim % k)
      return fail(LADDER_ERR_UNSUPPORTED, "shard_k=%d: per-shard O and down depths must be multiples of 256", k);
    if ((size_t)(c->ffn_dim / k) * 4 > 64 * 1024)
      return fail(LADDER_ERR_UNSUPPORTED, "shard mode stages one shard's slice of a row: ffn_dim/shard_k <= 16384 required");
  }
  if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64)
    return fail(LADDER_ERR_INVALID, "page_size=%d must be 16, 32 or 64", c->page_size);
  if (c->max_batch <= 0 || c->max_batch > 64) return fail(LADDER_ERR_INVALID, "max_batch=%d must be in 1..64", c->max_batch);
  if (c->max_seq <= 0 || c->max_seq > (1 << 20)) return fail(LADDER_ERR_INVALID, "max_seq=%d out of range", c->max_seq);
  if (c->max_prefill_tokens <= 0) return fail(LADDER_ERR_INVALID, "max_prefill_tokens must be positive");
  if (c->tie_embeddings != 0 && c->tie_embeddings != 1) return fail(LADDER_ERR_INVALID, "tie_embeddings must be 0 or 1");
  if (c->strict_boundary != 0 && c->strict_boundary != 1) return fail(LADDER_ERR_INVALID, "strict_boundary must be 0 or 1");
  if (c->weight_dtype != LADDER_DTYPE_BF16 && c->weight_dtype != LADDER_DTYPE_F16)
    return fail(LADDER_ERR_INVALID, "weight_dtype=%d must be LADDER_DTYPE_BF16 or LADDER_DTYPE_F16", c->weight_dtype);
  return LADDER_OK;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

struct LayerW {
  const void *attn_norm, *wq, *wk, *wv, *wo, *mlp_norm, *w_gate, *w_up, *w_down;
};

// Tensor maps of one layer's weights for the prefill GEMMs.
struct LayerMaps {
  TmaOperand wq, wk, wv, wo, gate, up, down;
};

struct GraphEntry {
  int B;
  const int32_t* tok;
  float* logits;
  int32_t* next;
  const ladder_kv* kv;
  cudaGraphExec_t exec;
  int launches;
};

}  // namespace

struct ladder_model {
  ladder_config cfg;
  const void *embed, *final_norm, *lm_head;
  int wdt;  // weight dtype
  std::vector<LayerW> layers;
  std::vector<LayerMaps> maps;
  TmaOperand map_xn[2], map_ao, map_act;  // activation operands, m_pad rows
  CUtensorMap map_q;  // rotated queries [m_pad][n_q * hd], the prefill attention operand
  CUtensorMap map_x[3];   // stream buffers [m_max][d] fp32, epilogue blocks (prefill residual GEMMs)
  CUtensorMap map_act_st; // SwiGLU rows [m_pad][ffn], epilogue blocks (prefill gate/up GEMM)
  char* ws;
  Plan plan;
  int num_sms;
  // Decode projections ask, launch by launch, for the smallest shared-memory
  // carveout that holds their CTAs (the rest of the SM's unified memory is L1
  // for the weight loads in flight) when the model's smallest projection has
  // at least kCarveoutMinWeightBytes of weights; else the driver chooses.
  // Measured on the graph decode step (context 2048): 8B hybrid B = 1 2914 ->
  // 2828 us, shard mode (k = 8) 3221 -> 3176 us, 70B unchanged; 1.2B (8.4 MB O
  // projection) 587 -> 600 us with every launch, 617 us with only those of at
  // least 32 MB -- its short launches of the two ladder streams share SMs, which
  // launches of different carveouts cannot.
  bool gemv_carve = false;
  int residual_mode = LADDER_RESIDUAL_CONFIG;
  int flags = 0;
  // next-token rule: greedy when samp_t <= 0, else temperature / top-k sampling
  float samp_t = 0.f;
  int samp_k = 0;
  uint64_t samp_seed = 0;
  int launches = 0;
  std::vector<GraphEntry> graphs;
  std::vector<int32_t> meta_host;
  // Second stream of the decode schedule (the MLP chain of ladder layers; high priority) and the
  // events that order the two chains: one per stream buffer, recorded after the
  // kernel that writes it, plus one to fork the second stream from the caller's.
  cudaStream_t aux = nullptr;
  cudaEvent_t ev_slot[3] = {nullptr, nullptr, nullptr};
  cudaEvent_t ev_fork = nullptr;
  cudaEvent_t ev_part = nullptr;  // shard mode: partial sums of a module written
  // launch probe
  int probe_class = -1;
  int probe_count = 0;
  std::vector<cudaEvent_t> probe_events;  // start/stop pairs
  // launch timeline: an event pair per launch on its stream, and a reference event
  bool tl_on = false;
  int tl_count = 0;
  std::vector<cudaEvent_t> tl_events;  // start/stop pairs
  std::vector<int> tl_stream, tl_class;
  cudaEvent_t tl_ref = nullptr;
  bool capturing = false;

  float* X(int i) { return reinterpret_cast<float*>(ws + plan.x[i % 3]); }
  template <class T> T* at(size_t off) { return reinterpret_cast<T*>(ws + off); }
  int* err() { return at<int>(plan.err); }

  // Point a batched decode projection at its split-K region (no-op when the
  // model was created for at most 2 rows).
  void splitk(GemvParams& g, int kind) {
    if (!plan.sk_bytes[kind]) return;
    const GemvSplitK sk = gemv_splitk_shape(g.n_tasks, g.K);
    char* base = ws + plan.sk[kind];
    size_t off = align_up((size_t)sk.ksplit * sk.n_wtasks * 256 * 4, 256);
    g.sk_part = reinterpret_cast<float*>(base);
    g.sk_ss = reinterpret_cast<float*>(base + off);
    off += align_up((size_t)sk.n_groups * sk.ksplit * 16 * 4, 256);
    g.sk_count = reinterpret_cast<int*>(base + off);
  }

  // Index j of the stream state x_j that module k (1-based) reads.
  int input_index(int k) const {
    if (residual_mode == LADDER_RESIDUAL_PARALLEL) return (k & 1) ? k - 1 : k - 2;
    const int layer = (k - 1) / 2;
    const int nstd = residual_mode == LADDER_RESIDUAL_STANDARD ? cfg.n_layers : cfg.n_standard_layers;
    if (layer < nstd) return k - 1;
    if (cfg.strict_boundary) return k - 2 > 0 ? k - 2 : 0;
    const int b = 2 * nstd;
    return k - 2 > b ? k - 2 : b;
  }

  void drop_graphs() {
    for (auto& g : graphs) cudaGraphExecDestroy(g.exec);
    graphs.clear();
  }
  void drop_probe() {
    for (auto e : probe_events) cudaEventDestroy(e);
    probe_events.clear();
    probe_class = -1;
    probe_count = 0;
  }
  void drop_timeline() {
    for (auto e : tl_events)
      if (e) cudaEventDestroy(e);
    if (tl_ref) cudaEventDestroy(tl_ref);
    tl_events.clear();
    tl_stream.clear();
    tl_class.clear();
    tl_ref = nullptr;
    tl_on = false;
    tl_count = 0;
  }
  // Event pairs around one launch of `cls`: for the probe when it is armed for
  // this class, for the timeline when it is armed.
  struct Probe {
    int probe = -1, tl = -1;
  };
  Probe probe_start(int cls, cudaStream_t s) {
    Probe p;
    if (capturing) return p;
    if (cls == probe_class && 2 * (size_t)probe_count < probe_events.size()) {
      p.probe = probe_count;
      cudaEventRecord(probe_events[2 * probe_count], s);
    }
    if (tl_on && 2 * (size_t)tl_count < tl_events.size()) {
      p.tl = tl_count++;
      tl_stream[p.tl] = s == aux ? 1 : 0;
      tl_class[p.tl] = cls;
      cudaEventRecord(tl_events[2 * p.tl], s);
    }
    return p;
  }
  void probe_stop(Probe p, cudaStream_t s) {
    if (p.probe >= 0) {
      cudaEventRecord(probe_events[2 * p.probe + 1], s);
      ++probe_count;
    }
    if (p.tl >= 0) cudaEventRecord(tl_events[2 * p.tl + 1], s);
  }
};

struct ladder_kv {
  ladder_model* m;
  char* pool;  // 16-bit elements of the weight dtype
  int num_pages, max_pages;
  int32_t* block_table;
  int32_t* seq_lens;
  std::vector<int32_t> host_lens;
  std::vector<int32_t> host_table;
  std::vector<int32_t> pages_of;  // assigned pages per sequence
  std::vector<CUtensorMap> maps;   // per layer: the pool as a 3-D TMA map

  KvLayer layer(int l) const {
    KvLayer v;
    const ladder_config& c = m->cfg;
    const size_t page_elems = (size_t)2 * c.n_kv_heads * c.page_size * c.head_dim;
    v.base = pool + (size_t)l * num_pages * page_elems * 2;
    v.block_table = block_table;
    v.max_pages = max_pages;
    v.page_size = c.page_size;
    v.page_shift = __builtin_ctz((unsigned)c.page_size);
    v.n_kv = c.n_kv_heads;
    v.head_dim = c.head_dim;
    return v;
  }
  int capacity(int b) const {
    const int cap = pages_of[b] * m->cfg.page_size;
    return cap < m->cfg.max_seq ? cap : m->cfg.max_seq;
  }
};

// ---------------------------------------------------------------------------
// Entry points
// ---------------------------------------------------------------------------
extern "C" {

const char* ladder_last_error(void) { return g_last_error.c_str(); }

int ladder_query_sizes(const ladder_config* cfg, size_t* workspace_bytes, size_t* kv_page_bytes) {
  int rc = validate_config(cfg);
  if (rc) return rc;
  if (workspace_bytes) *workspace_bytes = make_plan(*cfg).total;
  if (kv_page_bytes)
    *kv_page_bytes = (size_t)cfg->n_layers * 2 * cfg->n_kv_heads * cfg->page_size * cfg->head_dim * 2;
  return LADDER_OK;
}

int ladder_create(const ladder_config* cfg, const ladder_weights* w, void* workspace, size_t workspace_bytes,
                  ladder_stream_t stream, ladder_model** out) {
  if (!out) return fail(LADDER_ERR_INVALID, "out is NULL");
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc) return rc;
  if (!w || !w->embed || !w->final_norm || (!cfg->tie_embeddings && !w->lm_head))
    return fail(LADDER_ERR_INVALID, "missing global weight pointer");
  if (!w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo || !w->mlp_norm || !w->w_gate || !w->w_up || !w->w_down)
    return fail(LADDER_ERR_INVALID, "missing per-layer weight array");
  Plan plan = make_plan(*cfg);
  if (!workspace) return fail(LADDER_ERR_INVALID, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(LADDER_ERR_INVALID, "workspace must be 256-byte aligned");
  if (workspace_bytes < plan.total)
    return fail(LADDER_ERR_CAPACITY, "workspace too small: %zu < %zu bytes", workspace_bytes, plan.total);

  auto* m = new ladder_model();
  m->cfg = *cfg;
  m->embed = w->embed;
  m->final_norm = w->final_norm;
  m->lm_head = cfg->tie_embeddings ? w->embed : w->lm_head;
  m->wdt = cfg->weight_dtype;
  const void* globals[3] = {m->embed, m->final_norm, m->lm_head};
  for (const void* p : globals)
    if (!aligned(p, 16)) { delete m; return fail(LADDER_ERR_INVALID, "weights must be 16-byte aligned"); }
  m->layers.resize(cfg->n_layers);
  for (int l = 0; l < cfg->n_layers; ++l) {
    LayerW& L = m->layers[l];
    L.attn_norm = w->attn_norm[l];
    L.wq = w->wq[l];
    L.wk = w->wk[l];
    L.wv = w->wv[l];
    L.wo = w->wo[l];
    L.mlp_norm = w->mlp_norm[l];
    L.w_gate = w->w_gate[l];
    L.w_up = w->w_up[l];
    L.w_down = w->w_down[l];
    const void* ps[9] = {L.attn_norm, L.wq, L.wk, L.wv, L.wo, L.mlp_norm, L.w_gate, L.w_up, L.w_down};
    for (const void* p : ps)
      if (!p || !aligned(p, 16)) { delete m; return fail(LADDER_ERR_INVALID, "layer %d: weight NULL or not 16-byte aligned", l); }
  }
  m->ws = static_cast<char*>(workspace);
  m->plan = plan;
  {
    const ladder_config& c = *cfg;
    const uint64_t d = c.d_model, qd = (uint64_t)c.n_q_heads * c.head_dim, kvd = (uint64_t)c.n_kv_heads * c.head_dim;
    const uint64_t f = c.ffn_dim, Mp = plan.m_pad;
    const int wdt = c.weight_dtype;
    bool ok = make_tma_operand(&m->map_xn[0], m->ws + plan.xn[0], Mp, d, wdt, true) &&
              make_tma_operand(&m->map_xn[1], m->ws + plan.xn[1], Mp, d, wdt, true) &&
              make_tma_operand(&m->map_ao, m->ws + plan.ao, Mp, qd, wdt, true) &&
              make_tma_operand(&m->map_act, m->ws + plan.act, Mp, f, wdt, true) &&
              make_tma_map(&m->map_q, m->ws + plan.q, Mp, qd, wdt) &&
              make_tma_map_epilogue(&m->map_x[0], m->ws + plan.x[0], plan.m_max, d, 4, wdt) &&
              make_tma_map_epilogue(&m->map_x[1], m->ws + plan.x[1], plan.m_max, d, 4, wdt) &&
              make_tma_map_epilogue(&m->map_x[2], m->ws + plan.x[2], plan.m_max, d, 4, wdt) &&
              make_tma_map_epilogue(&m->map_act_st, m->ws + plan.act, 2 * Mp, f, 2, wdt);
    m->maps.resize(c.n_layers);
    for (int l = 0; ok && l < c.n_layers; ++l) {
      const LayerW& L = m->layers[l];
      LayerMaps& T = m->maps[l];
      ok = make_tma_operand(&T.wq, L.wq, qd, d, wdt) && make_tma_operand(&T.wk, L.wk, kvd, d, wdt) &&
           make_tma_operand(&T.wv, L.wv, kvd, d, wdt) && make_tma_operand(&T.wo, L.wo, d, qd, wdt) &&
           make_tma_operand(&T.gate, L.w_gate, f, d, wdt) && make_tma_operand(&T.up, L.w_up, f, d, wdt) &&
           make_tma_operand(&T.down, L.w_down, d, f, wdt);
    }
    if (!ok) {
      delete m;
      return fail(LADDER_ERR_CUDA, "ladder_create: could not encode TMA tensor maps (driver entry point missing?)");
    }
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, dev);
  {
    const ladder_config& c = *cfg;
    const size_t d = c.d_model, qd = (size_t)c.n_q_heads * c.head_dim, kvd = (size_t)c.n_kv_heads * c.head_dim;
    const size_t f = c.ffn_dim;
    size_t smallest = d * (qd + 2 * kvd);  // elements of the QKV, O, gate/up and down weights
    if (qd * d < smallest) smallest = qd * d;
    if (2 * d * f < smallest) smallest = 2 * d * f;
    if (d * f < smallest) smallest = d * f;
    m->gemv_carve = smallest * 2 >= kCarveoutMinWeightBytes;
  }
  if (e == cudaSuccess) e = gemv_configure();
  if (e == cudaSuccess) e = gemm_tc_configure();
  if (e == cudaSuccess) e = attn_prefill_tcgen05_configure();
  if (e == cudaSuccess) e = attn_decode_tc_configure();
  // The second stream carries the longer chain (the MLP modules of ladder layers, or
  // the shard reduces), so its blocks are scheduled ahead of the caller's stream.
  int prio_least = 0, prio_greatest = 0;
  if (e == cudaSuccess) e = cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest);
  if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&m->aux, cudaStreamNonBlocking, prio_greatest);
  for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&m->ev_slot[i], cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_part, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaMemsetAsync(m->err(), 0, 256, stream);
  for (int i = 0; i < SK_KINDS && e == cudaSuccess; ++i)
    if (plan.sk_bytes[i]) e = cudaMemsetAsync(m->ws + plan.sk[i], 0, plan.sk_bytes[i], stream);
  if (e == cudaSuccess)
    e = launch_rope_tables(m->at<float>(plan.rope_cos), m->at<float>(plan.rope_sin), cfg->max_seq, cfg->head_dim,
                           cfg->rope_theta,
                           RopeScaling{cfg->rope_scale_factor, cfg->rope_low_freq_factor, cfg->rope_high_freq_factor,
                                       (double)cfg->rope_original_max_pos},
                           stream);
  if (e != cudaSuccess) {
    ladder_destroy(m);
    return fail(LADDER_ERR_CUDA, "ladder_create: %s", cudaGetErrorString(e));
  }
  *out = m;
  return LADDER_OK;
}

void ladder_destroy(ladder_model* m) {
  if (!m) return;
  m->drop_graphs();
  m->drop_probe();
  m->drop_timeline();
  for (auto& e : m->ev_slot)
    if (e) cudaEventDestroy(e);
  if (m->ev_fork) cudaEventDestroy(m->ev_fork);
  if (m->ev_part) cudaEventDestroy(m->ev_part);
  if (m->aux) cudaStreamDestroy(m->aux);
  delete m;
}

int ladder_set_mode(ladder_model* m, int residual_mode, int flags) {
  if (!m) return fail(LADDER_ERR_INVALID, "model is NULL");
  if (residual_mode != LADDER_RESIDUAL_CONFIG && residual_mode != LADDER_RESIDUAL_STANDARD &&
      residual_mode != LADDER_RESIDUAL_PARALLEL)
    return fail(LADDER_ERR_INVALID, "unknown residual mode %d", residual_mode);
  if (flags & ~(LADDER_FLAG_DECODE_GRAPH | LADDER_FLAG_NO_PDL | LADDER_FLAG_ALL_LOGITS | LADDER_FLAG_FAST_PREFILL))
    return fail(LADDER_ERR_INVALID, "unknown flags 0x%x", flags);
  if (residual_mode != m->residual_mode || flags != m->flags) m->drop_graphs();
  m->residual_mode = residual_mode;
  m->flags = flags;
  return LADDER_OK;
}

int ladder_set_sampling(ladder_model* m, float temperature, int32_t top_k, uint64_t seed) {
  if (!m) return fail(LADDER_ERR_INVALID, "model is NULL");
  if (temperature != temperature) return fail(LADDER_ERR_INVALID, "temperature is NaN");
  const float t = temperature > 0.f ? temperature : 0.f;
  if (t != m->samp_t || top_k != m->samp_k || seed != m->samp_seed) m->drop_graphs();
  m->samp_t = t;
  m->samp_k = top_k;
  m->samp_seed = seed;
  return LADDER_OK;
}

int ladder_kv_create(ladder_model* m, void* pool, int32_t num_pages, int32_t max_pages_per_seq,
                     int32_t* block_table, int32_t* seq_lens, ladder_kv** out) {
  if (!out) return fail(LADDER_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (!m || !pool || !block_table || !seq_lens) return fail(LADDER_ERR_INVALID, "NULL argument");
  if (!aligned(pool, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return fail(LADDER_ERR_INVALID, "pool must be 16-byte aligned");
  if (num_pages <= 0 || max_pages_per_seq <= 0) return fail(LADDER_ERR_INVALID, "num_pages and max_pages_per_seq must be positive");
  auto* kv = new ladder_kv();
  kv->m = m;
  kv->pool = static_cast<char*>(pool);
  kv->num_pages = num_pages;
  kv->max_pages = max_pages_per_seq;
  kv->block_table = block_table;
  kv->seq_lens = seq_lens;
  kv->host_lens.assign(m->cfg.max_batch, 0);
  kv->host_table.assign((size_t)m->cfg.max_batch * max_pages_per_seq, -1);
  kv->pages_of.assign(m->cfg.max_batch, 0);
  const ladder_config& c = m->cfg;
  kv->maps.resize(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    if (!make_kv_tma_map(&kv->maps[l], kv->layer(l).base, num_pages, c.n_kv_heads, c.page_size, c.head_dim,
                         m->wdt)) {
      delete kv;
      return fail(LADDER_ERR_CUDA, "ladder_kv_create: could not encode the KV pool tensor map");
    }
  }
  *out = kv;
  return LADDER_OK;
}

void ladder_kv_destroy(ladder_kv* kv) {
  if (!kv) return;
  // graphs captured against this handle must not be replayed for another one
  auto& gs = kv->m->graphs;
  for (size_t i = 0; i < gs.size();) {
    if (gs[i].kv == kv) {
      cudaGraphExecDestroy(gs[i].exec);
      gs.erase(gs.begin() + i);
    } else {
      ++i;
    }
  }
  delete kv;
}

int ladder_kv_set_pages(ladder_kv* kv, const int32_t* host_table, ladder_stream_t stream) {
  if (!kv || !host_table) return fail(LADDER_ERR_INVALID, "NULL argument");
  const int Bm = kv->m->cfg.max_batch, P = kv->max_pages;
  std::vector<char> used(kv->num_pages, 0);
  std::vector<int32_t> pages(Bm, 0);
  for (int b = 0; b < Bm; ++b) {
    bool ended = false;
    for (int i = 0; i < P; ++i) {
      const int32_t pg = host_table[(size_t)b * P + i];
      if (pg == -1) { ended = true; continue; }
      if (ended) return fail(LADDER_ERR_INVALID, "sequence %d: assigned pages must be a prefix of its row", b);
      if (pg < 0 || pg >= kv->num_pages) return fail(LADDER_ERR_INVALID, "sequence %d: page id %d out of range", b, pg);
      if (used[pg]) return fail(LADDER_ERR_INVALID, "page %d assigned twice", pg);
      used[pg] = 1;
      pages[b] = i + 1;
    }
    if (pages[b] * kv->m->cfg.page_size < kv->host_lens[b])
      return fail(LADDER_ERR_CAPACITY, "sequence %d: new pages hold fewer positions than its length", b);
  }
  cudaError_t e = cudaMemcpyAsync(kv->block_table, host_table, sizeof(int32_t) * (size_t)Bm * P,
                                  cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return fail(LADDER_ERR_CUDA, "block table copy: %s", cudaGetErrorString(e));
  // The copy from pageable memory is staged before cudaMemcpyAsync returns.
  kv->host_table.assign(host_table, host_table + (size_t)Bm * P);
  kv->pages_of = pages;
  return LADDER_OK;
}

int ladder_kv_reset(ladder_kv* kv, ladder_stream_t stream) {
  if (!kv) return fail(LADDER_ERR_INVALID, "kv is NULL");
  CUDA_TRY(cudaMemsetAsync(kv->seq_lens, 0, sizeof(int32_t) * kv->m->cfg.max_batch, stream));
  std::fill(kv->host_lens.begin(), kv->host_lens.end(), 0);
  return LADDER_OK;
}

int32_t ladder_kv_seq_len(const ladder_kv* kv, int32_t b) {
  if (!kv || b < 0 || b >= (int)kv->host_lens.size()) return -1;
  return kv->host_lens[b];
}

int32_t ladder_last_launch_count(const ladder_model* m) { return m ? m->launches : -1; }

int ladder_probe_begin(ladder_model* m, int kernel_class, int32_t max_launches) {
  if (!m) return fail(LADDER_ERR_INVALID, "model is NULL");
  if (kernel_class < LADDER_PROBE_QKV || kernel_class > LADDER_PROBE_REDUCE)
    return fail(LADDER_ERR_INVALID, "unknown kernel class %d", kernel_class);
  if (max_launches < 1 || max_launches > 65536) return fail(LADDER_ERR_INVALID, "max_launches out of range");
  if (m->flags & LADDER_FLAG_DECODE_GRAPH) return fail(LADDER_ERR_INVALID, "the probe times eager decode steps only");
  m->drop_probe();
  m->probe_events.resize(2 * (size_t)max_launches, nullptr);
  for (auto& e : m->probe_events) {
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) {
      e = nullptr;
      m->drop_probe();
      return fail(LADDER_ERR_CUDA, "cudaEventCreate: %s", cudaGetErrorString(err));
    }
  }
  m->probe_class = kernel_class;
  return LADDER_OK;
}

int ladder_timeline_begin(ladder_model* m, int32_t max_launches, ladder_stream_t stream) {
  if (!m) return fail(LADDER_ERR_INVALID, "model is NULL");
  if (max_launches < 1 || max_launches > 65536) return fail(LADDER_ERR_INVALID, "max_launches out of range");
  if (m->flags & LADDER_FLAG_DECODE_GRAPH) return fail(LADDER_ERR_INVALID, "the timeline records eager decode steps only");
  m->drop_timeline();
  m->tl_events.resize(2 * (size_t)max_launches, nullptr);
  m->tl_stream.assign(max_launches, 0);
  m->tl_class.assign(max_launches, 0);
  cudaError_t err = cudaEventCreate(&m->tl_ref);
  for (auto& e : m->tl_events)
    if (err == cudaSuccess) err = cudaEventCreate(&e);
  if (err == cudaSuccess) err = cudaEventRecord(m->tl_ref, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) {
    m->drop_timeline();
    return fail(LADDER_ERR_CUDA, "timeline events: %s", cudaGetErrorString(err));
  }
  m->tl_on = true;
  return LADDER_OK;
}

int ladder_timeline_end(ladder_model* m, int32_t capacity, int32_t* n, int32_t* streams, int32_t* classes,
                        float* start_ms, float* end_ms) {
  if (!m || !n || (capacity > 0 && (!streams || !classes || !start_ms || !end_ms)))
    return fail(LADDER_ERR_INVALID, "NULL argument");
  if (!m->tl_on) return fail(LADDER_ERR_INVALID, "the timeline is not armed");
  const int cnt = m->tl_count < capacity ? m->tl_count : capacity;
  for (int i = 0; i < cnt; ++i) {
    float t0 = 0.f, t1 = 0.f;
    cudaError_t e = cudaEventSynchronize(m->tl_events[2 * i + 1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t0, m->tl_ref, m->tl_events[2 * i]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t1, m->tl_ref, m->tl_events[2 * i + 1]);
    if (e != cudaSuccess) {
      m->drop_timeline();
      return fail(LADDER_ERR_CUDA, "timeline events: %s", cudaGetErrorString(e));
    }
    streams[i] = m->tl_stream[i];
    classes[i] = m->tl_class[i];
    start_ms[i] = t0;
    end_ms[i] = t1;
  }
  *n = cnt;
  m->drop_timeline();
  return LADDER_OK;
}

int ladder_probe_end(ladder_model* m, int32_t* launches, float* total_ms) {
  if (!m || !launches || !total_ms) return fail(LADDER_ERR_INVALID, "NULL argument");
  float total = 0.f;
  for (int i = 0; i < m->probe_count; ++i) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(m->probe_events[2 * i + 1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, m->probe_events[2 * i], m->probe_events[2 * i + 1]);
    if (e != cudaSuccess) {
      m->drop_probe();
      return fail(LADDER_ERR_CUDA, "probe events: %s", cudaGetErrorString(e));
    }
    total += ms;
  }
  *launches = m->probe_count;
  *total_ms = total;
  m->drop_probe();
  return LADDER_OK;
}

int ladder_get_device_error(ladder_model* m, ladder_stream_t stream, int32_t* code) {
  if (!m || !code) return fail(LADDER_ERR_INVALID, "NULL argument");
  int32_t v = 0;
  CUDA_TRY(cudaMemcpyAsync(&v, m->err(), sizeof(int32_t), cudaMemcpyDeviceToHost, stream));
  CUDA_TRY(cudaStreamSynchronize(stream));
  CUDA_TRY(cudaMemsetAsync(m->err(), 0, sizeof(int32_t), stream));
  *code = v;
  return LADDER_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Launch sequences
// ---------------------------------------------------------------------------
namespace {

#define LAUNCH(expr, n)                                                                          \
  do {                                                                                           \
    cudaError_t e_ = (expr);                                                                     \
    if (e_ != cudaSuccess) return fail(LADDER_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
    m->launches += (n);                                                                          \
  } while (0)


// One decode step for sequences 0..B-1.
//
// Schedule.  In a ladder layer the attention module k reads x_{k-2} and the MLP
// module k+1 reads x_{k-1}, so neither module's weight streaming waits for the
// module just before it; only their residual adds (x_k = x_{k-1} + h_k) join
// the two.  The attention chain runs on the caller's stream and the MLP chain of
// ladder layers on a second stream; each stream buffer has an event recorded by
// its writer, and a kernel that reads a buffer written on the other stream waits
// on that event.  Standard layers (and the STANDARD residual mode) keep every
// kernel on the caller's stream.  The three buffers hold x_k in buffer k mod 3;
// the write-after-read order on a reused buffer follows from these read
// dependencies (the module that overwrites x_{k-3} has already waited for a
// buffer written after every reader of x_{k-3}).
// Shard-mode decode step (shard_k > 1).  Every GEMV and attention kernel runs on
// the caller's stream; the per-module reduce of the k partial sums runs on the
// second stream.  A module's first kernel waits for the reduce that produced
// its input, which in a ladder layer is the reduce of the module two back, so
// the previous module's reduce overlaps this module's weight streaming; in a
// standard layer it is the previous module's reduce, which serialises them.
// The partial buffers alternate between modules; module k rewrites the buffer
// of module k-2 only after its first kernel has waited for a reduce at least
// as late as module k-2's.
int enqueue_decode_shard(ladder_model* m, ladder_kv* kv, const int32_t* tokens, int B, float* logits,
                         int32_t* next_tok, int nsplit, cudaStream_t s) {
  const ladder_config& c = m->cfg;
  const int d = c.d_model, qd = c.n_q_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim, f = c.ffn_dim;
  const int ksh = c.shard_k;
  const Plan& P = m->plan;
  float* q = m->at<float>(P.q);
  float* ao = m->at<float>(P.ao);
  float* act = m->at<float>(P.act);
  float* part = m->at<float>(P.shard);
  const size_t part_stride = (size_t)B * ksh * d;
  // Every kernel launches early here: the launch policy of enqueue_decode (early
  // launch only for short kernels behind short ones) made this schedule slower
  // (8B full ladder, k = 8: 3341 -> 3403 us per step); the reduces on the second
  // stream gain from it.
  const bool pdl = !(m->flags & LADDER_FLAG_NO_PDL);
  cudaStream_t rs = m->aux;
  int writer[3] = {0, 0, 0};  // 0: caller's stream (embed), 1: reduce stream
  auto use = [&](int buf) -> int {
    if (writer[buf % 3] == 1) CUDA_TRY(cudaStreamWaitEvent(s, m->ev_slot[buf % 3], 0));
    return LADDER_OK;
  };

  LAUNCH(launch_embed(tokens, B, m->embed, m->wdt, d, c.vocab, m->X(0), m->err(), s, pdl), 1);
  CUDA_TRY(cudaEventRecord(m->ev_slot[0], s));
  int rc;
  for (int k = 1; k <= 2 * c.n_layers; ++k) {
    const int l = (k - 1) / 2;
    const LayerW& L = m->layers[l];
    const int j = m->input_index(k);
    if ((rc = use(j))) return rc;
    float* pk = part + (size_t)(k & 1) * part_stride;
    GemvParams o{};
    o.carve = m->gemv_carve;
    if (k & 1) {  // attention module
      const KvLayer kvl = kv->layer(l);
      GemvParams g{};
      g.carve = m->gemv_carve;
      g.x = m->X(j); g.ldx = d; g.g = L.attn_norm; g.eps = c.norm_eps; g.B = B; g.K = d;
      g.w0 = L.wq; g.w1 = L.wk; g.w2 = L.wv; g.n_tasks = (qd + 2 * kvd) / 2;
      g.out = q; g.ldo = qd; g.nq_hd = qd; g.nkv_hd = kvd;
      g.rope_cos = m->at<float>(P.rope_cos); g.rope_sin = m->at<float>(P.rope_sin);
      g.pos = kv->seq_lens; g.kv = kvl; g.err = m->err();
      m->splitk(g, SK_QKV);
      auto pq = m->probe_start(LADDER_PROBE_QKV, s);
      LAUNCH(launch_gemv(g, GEMV_QKV, m->wdt, m->num_sms, s, pdl), gemv_launch_count(B, g.K, GEMV_QKV));
      m->probe_stop(pq, s);
      AttnDecodeParams a{};
      a.q = q; a.kv = kvl; a.seq_lens = kv->seq_lens; a.n_q = c.n_q_heads; a.split_len = kSplitLen;
      a.nsplit = nsplit; a.scale = 1.0f / sqrtf((float)c.head_dim);
      a.part_o = m->at<float>(P.part_o); a.part_ml = m->at<float>(P.part_ml); a.out = ao;
      auto pa = m->probe_start(LADDER_PROBE_ATTN, s);
      LAUNCH(launch_attn_decode_tc(&kv->maps[l], a, B, c.n_kv_heads, c.head_dim, m->wdt, m->err(), s, pdl, pdl), 2);
      m->probe_stop(pa, s);
      o.x = ao; o.ldx = qd; o.K = qd / ksh; o.kfull = qd; o.ldw = qd; o.w0 = L.wo;
    } else {  // MLP module
      GemvParams g{};
      g.carve = m->gemv_carve;
      g.x = m->X(j); g.ldx = d; g.g = L.mlp_norm; g.eps = c.norm_eps; g.B = B; g.K = d;
      g.w0 = L.w_gate; g.w1 = L.w_up; g.n_tasks = f; g.out = act; g.ldo = f; g.err = m->err();
      auto pe = m->probe_start(LADDER_PROBE_GATEUP, s);
      m->splitk(g, SK_GATEUP);
      LAUNCH(launch_gemv(g, GEMV_GATEUP, m->wdt, m->num_sms, s, pdl), gemv_launch_count(B, g.K, GEMV_GATEUP));
      m->probe_stop(pe, s);
      o.x = act; o.ldx = f; o.K = f / ksh; o.kfull = f; o.ldw = f; o.w0 = L.w_down;
    }
    // row-parallel partial sums: shard sh uses input block sh and writes part[b][sh][:]
    o.g = nullptr; o.B = B; o.shard_tasks = d / 2; o.n_tasks = ksh * (d / 2);
    o.out = pk; o.ldo = ksh * d; o.err = m->err();
    auto po = m->probe_start((k & 1) ? LADDER_PROBE_OUT : LADDER_PROBE_DOWN, s);
    LAUNCH(launch_gemv(o, GEMV_PARTIAL, m->wdt, m->num_sms, s, pdl), gemv_launch_count(B, o.kfull, GEMV_PARTIAL));
    m->probe_stop(po, s);
    CUDA_TRY(cudaEventRecord(m->ev_part, s));
    // the "all-reduce": x_k = x_{k-1} + sum of the partials, on the second stream
    CUDA_TRY(cudaStreamWaitEvent(rs, m->ev_part, 0));
    if (writer[(k - 1) % 3] == 0) CUDA_TRY(cudaStreamWaitEvent(rs, m->ev_slot[(k - 1) % 3], 0));
    auto pr = m->probe_start(LADDER_PROBE_REDUCE, rs);
    LAUNCH(launch_shard_reduce(pk, ksh, B, d, m->X(k - 1), m->X(k), rs, pdl), 1);
    m->probe_stop(pr, rs);
    CUDA_TRY(cudaEventRecord(m->ev_slot[k % 3], rs));
    writer[k % 3] = 1;
  }
  if ((rc = use(2 * c.n_layers))) return rc;
  GemvParams h{};
  h.carve = m->gemv_carve;
  h.x = m->X(2 * c.n_layers); h.ldx = d; h.g = m->final_norm; h.eps = c.norm_eps; h.B = B; h.K = d;
  h.w0 = m->lm_head; h.n_tasks = c.vocab / 2; h.out = logits; h.ldo = c.vocab; h.err = m->err();
  m->splitk(h, SK_LMHEAD);
  auto ph = m->probe_start(LADDER_PROBE_LMHEAD, s);
  LAUNCH(launch_gemv(h, GEMV_LOGITS, m->wdt, m->num_sms, s, pdl), gemv_launch_count(B, h.K, GEMV_LOGITS));
  m->probe_stop(ph, s);
  if (next_tok && m->samp_t > 0.f)  // the sampled token takes position seq_lens[b] + 1
    LAUNCH(launch_sample(logits, B, c.vocab, m->samp_t, m->samp_k, m->samp_seed, kv->seq_lens, 1, next_tok, s, pdl), 1);
  else if (next_tok)
    LAUNCH(launch_argmax(logits, B, c.vocab, m->at<float>(P.am_v), m->at<int>(P.am_i), kArgmaxBlocks, next_tok, s, pdl), 2);
  LAUNCH(launch_advance(kv->seq_lens, B, s, pdl), 1);
  return LADDER_OK;
}

int enqueue_decode(ladder_model* m, ladder_kv* kv, const int32_t* tokens, int B, float* logits,
                   int32_t* next_tok, int nsplit, cudaStream_t s) {
  if (m->cfg.shard_k > 1) return enqueue_decode_shard(m, kv, tokens, B, logits, next_tok, nsplit, s);
  const ladder_config& c = m->cfg;
  const int d = c.d_model, qd = c.n_q_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim, f = c.ffn_dim;
  const Plan& P = m->plan;
  float* q = m->at<float>(P.q);
  float* ao = m->at<float>(P.ao);
  float* act = m->at<float>(P.act);
  // layers below nstd run both modules on the caller's stream; above it the MLP
  // module (which does not read the attention module's output) runs on the second
  const int nstd = m->residual_mode == LADDER_RESIDUAL_STANDARD ? c.n_layers
                   : m->residual_mode == LADDER_RESIDUAL_PARALLEL ? 0
                                                                  : c.n_standard_layers;
  const bool pdl = !(m->flags & LADDER_FLAG_NO_PDL);
  // Programmatic dependent launch lets a kernel's blocks become resident while
  // the previous kernel of its stream finishes, which hides a short kernel's
  // ramp.  Behind a long kernel (a projection of more than kPdlMaxWeightBytes
  // of weights) those blocks would wait on SM slots that the other ladder
  // stream's kernels need, and a long kernel's own blocks would crowd the
  // other stream; so a kernel launches early only when it is short and so is
  // its predecessor.  The MLP chain (gate/up -> down, one chain across the
  // layers: the step's critical path) counts as short up to kPdlMaxMlpWeightBytes
  // at one or two rows: 8B hybrid B = 1 2828 -> 2763 us, 70B and 1.2B unchanged
  // (their MLP projections are above or below both limits); the attention
  // chain keeps the lower limit, since its early blocks hold SM slots the MLP
  // chain needs (the 70B's O projection, 134 MB, launched early: 20.72 ->
  // 21.67 ms).  Batched rows keep the lower limit for both (8B at 16 rows
  // within noise, 4960 vs 4998 us).
  bool long_prev[2] = {false, false};  // per stream: the last kernel was a long projection
  auto early = [&](int si, size_t weight_bytes, size_t lim = kPdlMaxWeightBytes) {
    return pdl && !long_prev[si] && weight_bytes <= lim;
  };
  auto ran = [&](int si, size_t weight_bytes, size_t lim = kPdlMaxWeightBytes) {
    long_prev[si] = weight_bytes > lim;
  };
  const size_t mlp_lim = B <= 2 ? kPdlMaxMlpWeightBytes : kPdlMaxWeightBytes;
  const size_t wb_qkv = (size_t)(qd + 2 * kvd) * d * 2, wb_o = (size_t)qd * d * 2;
  const size_t wb_gu = (size_t)2 * f * d * 2, wb_down = (size_t)f * d * 2, wb_lm = (size_t)c.vocab * d * 2;
  cudaStream_t streams[2] = {s, m->aux};
  int writer[3] = {0, 0, 0};  // stream index that last wrote each buffer
  bool forked = false;
  auto use = [&](int buf, int si) -> int {  // make stream si wait for the writer of x buffer `buf`
    const int b3 = buf % 3;
    if (writer[b3] == si) return LADDER_OK;
    if (si == 1 && !forked) {
      CUDA_TRY(cudaEventRecord(m->ev_fork, s));
      CUDA_TRY(cudaStreamWaitEvent(m->aux, m->ev_fork, 0));
      forked = true;
    }
    CUDA_TRY(cudaStreamWaitEvent(streams[si], m->ev_slot[b3], 0));
    return LADDER_OK;
  };
  auto wrote = [&](int buf, int si) -> int {
    writer[buf % 3] = si;
    CUDA_TRY(cudaEventRecord(m->ev_slot[buf % 3], streams[si]));
    return LADDER_OK;
  };
  int rc;

  LAUNCH(launch_embed(tokens, B, m->embed, m->wdt, d, c.vocab, m->X(0), m->err(), s, early(0, 0)), 1);
  ran(0, 0);
  if ((rc = wrote(0, 0))) return rc;
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerW& L = m->layers[l];
    const KvLayer kvl = kv->layer(l);
    const int mlp_stream = l < nstd ? 0 : 1;
    // attention module k = 2l + 1 (caller's stream)
    {
      const int k = 2 * l + 1;
      const int j = m->input_index(k);
      if ((rc = use(j, 0))) return rc;
      GemvParams g{};
      g.carve = m->gemv_carve;
      g.x = m->X(j); g.ldx = d; g.g = L.attn_norm; g.eps = c.norm_eps; g.B = B; g.K = d;
      g.w0 = L.wq; g.w1 = L.wk; g.w2 = L.wv; g.n_tasks = (qd + 2 * kvd) / 2;
      g.out = q; g.ldo = qd; g.nq_hd = qd; g.nkv_hd = kvd;
      g.rope_cos = m->at<float>(P.rope_cos); g.rope_sin = m->at<float>(P.rope_sin);
      g.pos = kv->seq_lens; g.kv = kvl;
      auto pe = m->probe_start(LADDER_PROBE_QKV, s);
      g.err = m->err();
      m->splitk(g, SK_QKV);
      LAUNCH(launch_gemv(g, GEMV_QKV, m->wdt, m->num_sms, s, early(0, wb_qkv)), gemv_launch_count(B, g.K, GEMV_QKV));
      ran(0, wb_qkv);
      m->probe_stop(pe, s);

      AttnDecodeParams a{};
      a.q = q; a.kv = kvl; a.seq_lens = kv->seq_lens; a.n_q = c.n_q_heads; a.split_len = kSplitLen;
      a.nsplit = nsplit; a.scale = 1.0f / sqrtf((float)c.head_dim);
      a.part_o = m->at<float>(P.part_o); a.part_ml = m->at<float>(P.part_ml); a.out = ao;
      pe = m->probe_start(LADDER_PROBE_ATTN, s);
      // the split kernel reads the K/V of every split (its size for the rule
      // above); the combine launches early only when the split kernel did
      const size_t kv_bytes = (size_t)B * nsplit * kSplitLen * kvd * 2 * 2;
      const bool attn_early = early(0, kv_bytes);
      LAUNCH(launch_attn_decode_tc(&kv->maps[l], a, B, c.n_kv_heads, c.head_dim, m->wdt, m->err(), s, attn_early,
                                   attn_early), 2);
      ran(0, kv_bytes);
      m->probe_stop(pe, s);

      if ((rc = use(k - 1, 0))) return rc;
      GemvParams o{};
      o.carve = m->gemv_carve;
      o.x = ao; o.ldx = qd; o.g = nullptr; o.B = B; o.K = qd; o.w0 = L.wo; o.n_tasks = d / 2;
      o.out = m->X(k); o.ldo = d; o.x_res = m->X(k - 1); o.ldr = d;
      pe = m->probe_start(LADDER_PROBE_OUT, s);
      o.err = m->err();
      m->splitk(o, SK_OUT);
      LAUNCH(launch_gemv(o, GEMV_RESID, m->wdt, m->num_sms, s, early(0, wb_o)), gemv_launch_count(B, o.K, GEMV_RESID));
      ran(0, wb_o);
      m->probe_stop(pe, s);
      if ((rc = wrote(k, 0))) return rc;
    }
    // MLP module k = 2l + 2 (second stream in ladder layers)
    {
      const int k = 2 * l + 2;
      const int j = m->input_index(k);
      cudaStream_t ms = streams[mlp_stream];
      if ((rc = use(j, mlp_stream))) return rc;
      GemvParams g{};
      g.carve = m->gemv_carve;
      g.x = m->X(j); g.ldx = d; g.g = L.mlp_norm; g.eps = c.norm_eps; g.B = B; g.K = d;
      g.w0 = L.w_gate; g.w1 = L.w_up; g.n_tasks = f; g.out = act; g.ldo = f;
      auto pe = m->probe_start(LADDER_PROBE_GATEUP, ms);
      g.err = m->err();
      m->splitk(g, SK_GATEUP);
      LAUNCH(launch_gemv(g, GEMV_GATEUP, m->wdt, m->num_sms, ms, early(mlp_stream, wb_gu, mlp_lim)), gemv_launch_count(B, g.K, GEMV_GATEUP));
      ran(mlp_stream, wb_gu, mlp_lim);
      m->probe_stop(pe, ms);

      if ((rc = use(k - 1, mlp_stream))) return rc;
      GemvParams o{};
      o.carve = m->gemv_carve;
      o.x = act; o.ldx = f; o.g = nullptr; o.B = B; o.K = f; o.w0 = L.w_down; o.n_tasks = d / 2;
      o.out = m->X(k); o.ldo = d; o.x_res = m->X(k - 1); o.ldr = d;
      pe = m->probe_start(LADDER_PROBE_DOWN, ms);
      o.err = m->err();
      m->splitk(o, SK_DOWN);
      LAUNCH(launch_gemv(o, GEMV_RESID, m->wdt, m->num_sms, ms, early(mlp_stream, wb_down, mlp_lim)), gemv_launch_count(B, o.K, GEMV_RESID));
      ran(mlp_stream, wb_down, mlp_lim);
      m->probe_stop(pe, ms);
      if ((rc = wrote(k, mlp_stream))) return rc;
    }
  }
  if ((rc = use(2 * c.n_layers, 0))) return rc;
  GemvParams h{};
  h.carve = m->gemv_carve;
  h.x = m->X(2 * c.n_layers); h.ldx = d; h.g = m->final_norm; h.eps = c.norm_eps; h.B = B; h.K = d;
  h.w0 = m->lm_head; h.n_tasks = c.vocab / 2; h.out = logits; h.ldo = c.vocab;
  auto pe = m->probe_start(LADDER_PROBE_LMHEAD, s);
  h.err = m->err();
  m->splitk(h, SK_LMHEAD);
  LAUNCH(launch_gemv(h, GEMV_LOGITS, m->wdt, m->num_sms, s, early(0, wb_lm)), gemv_launch_count(B, h.K, GEMV_LOGITS));
  ran(0, wb_lm);
  m->probe_stop(pe, s);
  if (next_tok && m->samp_t > 0.f)  // the sampled token takes position seq_lens[b] + 1
    LAUNCH(launch_sample(logits, B, c.vocab, m->samp_t, m->samp_k, m->samp_seed, kv->seq_lens, 1, next_tok, s, early(0, 0)), 1);
  else if (next_tok)
    LAUNCH(launch_argmax(logits, B, c.vocab, m->at<float>(P.am_v), m->at<int>(P.am_i), kArgmaxBlocks, next_tok, s, early(0, 0)), 2);
  LAUNCH(launch_advance(kv->seq_lens, B, s, pdl), 1);
  return LADDER_OK;
}

}  // namespace

extern "C" int ladder_decode_step(ladder_model* m, ladder_kv* kv, const int32_t* tokens, int32_t B,
                                  float* logits, int32_t* next_tok, ladder_stream_t stream) {
  if (!m || !kv || !tokens || !logits) return fail(LADDER_ERR_INVALID, "NULL argument");
  if (kv->m != m) return fail(LADDER_ERR_INVALID, "KV handle belongs to another model");
  if (B <= 0 || B > m->cfg.max_batch) return fail(LADDER_ERR_INVALID, "B=%d out of range 1..%d", B, m->cfg.max_batch);
  int max_ctx = 0;
  for (int b = 0; b < B; ++b) {
    if (kv->host_lens[b] + 1 > kv->capacity(b))
      return fail(LADDER_ERR_CAPACITY, "sequence %d: position %d exceeds its KV capacity %d", b, kv->host_lens[b], kv->capacity(b));
    if (kv->host_lens[b] + 1 > max_ctx) max_ctx = kv->host_lens[b] + 1;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool use_graph = (m->flags & LADDER_FLAG_DECODE_GRAPH) != 0;
  if (use_graph && s == nullptr) return fail(LADDER_ERR_INVALID, "graph mode needs a non-default stream");
  m->launches = 0;
  if (!use_graph) {
    const int nsplit = (max_ctx + kSplitLen - 1) / kSplitLen;
    int rc = enqueue_decode(m, kv, tokens, B, logits, next_tok, nsplit, s);
    if (rc) return rc;
  } else {
    GraphEntry* ge = nullptr;
    for (auto& g : m->graphs)
      if (g.B == B && g.tok == tokens && g.logits == logits && g.next == next_tok && g.kv == kv) ge = &g;
    if (!ge) {
      CUDA_TRY(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
      m->capturing = true;
      int rc = enqueue_decode(m, kv, tokens, B, logits, next_tok, m->plan.nsplit_max, s);
      m->capturing = false;
      cudaGraph_t graph = nullptr;
      cudaError_t e = cudaStreamEndCapture(s, &graph);
      if (rc) { if (graph) cudaGraphDestroy(graph); return rc; }
      if (e != cudaSuccess) return fail(LADDER_ERR_CUDA, "graph capture: %s", cudaGetErrorString(e));
      cudaGraphExec_t exec = nullptr;
      e = cudaGraphInstantiate(&exec, graph, 0);
      cudaGraphDestroy(graph);
      if (e != cudaSuccess) return fail(LADDER_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
      m->graphs.push_back(GraphEntry{B, tokens, logits, next_tok, kv, exec, m->launches});
      ge = &m->graphs.back();
    }
    CUDA_TRY(cudaGraphLaunch(ge->exec, s));
    m->launches = ge->launches;
  }
  for (int b = 0; b < B; ++b) kv->host_lens[b] += 1;
  return LADDER_OK;
}

extern "C" int ladder_prefill(ladder_model* m, ladder_kv* kv, const int32_t* tokens, const int32_t* host_lens,
                              int32_t B, float* logits, int32_t* next_tok, ladder_stream_t stream) {
  if (!m || !kv || !tokens || !host_lens || !logits) return fail(LADDER_ERR_INVALID, "NULL argument");
  if (kv->m != m) return fail(LADDER_ERR_INVALID, "KV handle belongs to another model");
  const ladder_config& c = m->cfg;
  if (B <= 0 || B > c.max_batch) return fail(LADDER_ERR_INVALID, "B=%d out of range 1..%d", B, c.max_batch);
  long long total = 0;
  for (int b = 0; b < B; ++b) {
    if (host_lens[b] <= 0) return fail(LADDER_ERR_INVALID, "sequence %d: length %d must be positive", b, host_lens[b]);
    if (kv->host_lens[b] != 0) return fail(LADDER_ERR_INVALID, "sequence %d is not empty: prefill starts from an empty cache", b);
    if (host_lens[b] > kv->capacity(b))
      return fail(LADDER_ERR_CAPACITY, "sequence %d: length %d exceeds its KV capacity %d", b, host_lens[b], kv->capacity(b));
    total += host_lens[b];
  }
  if (total > c.max_prefill_tokens)
    return fail(LADDER_ERR_CAPACITY, "%lld prompt tokens exceed max_prefill_tokens=%d", total, c.max_prefill_tokens);
  const bool all_rows = (m->flags & LADDER_FLAG_ALL_LOGITS) != 0;
  if (all_rows && next_tok && m->samp_t > 0.f)
    return fail(LADDER_ERR_UNSUPPORTED, "sampling is not available with LADDER_FLAG_ALL_LOGITS");
  const int M = (int)total;
  const int Bm = c.max_batch;
  const Plan& P = m->plan;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // Row metadata: row_b[M_max], row_pos[M_max], lens[Bm], last_row[Bm], start[Bm].
  std::vector<int32_t>& meta = m->meta_host;
  meta.assign(2 * (size_t)P.m_max + 3 * Bm, 0);
  int32_t* row_b = meta.data();
  int32_t* row_pos = row_b + P.m_max;
  int32_t* lens = row_pos + P.m_max;
  int32_t* last = lens + Bm;
  int32_t* start = last + Bm;
  int mm = 0, max_len = 0;
  for (int b = 0; b < B; ++b) {
    start[b] = mm;
    for (int t = 0; t < host_lens[b]; ++t, ++mm) {
      row_b[mm] = b;
      row_pos[mm] = t;
    }
    lens[b] = host_lens[b];
    last[b] = mm - 1;
    if (host_lens[b] > max_len) max_len = host_lens[b];
  }
  m->launches = 0;
  int32_t* dmeta = m->at<int32_t>(P.meta);
  CUDA_TRY(cudaMemcpyAsync(dmeta, meta.data(), meta.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  const int32_t* d_row_b = dmeta;
  const int32_t* d_row_pos = dmeta + P.m_max;
  const int32_t* d_lens = d_row_pos + P.m_max;
  const int32_t* d_last = d_lens + Bm;
  const int32_t* d_start = d_last + Bm;

  const int d = c.d_model, qd = c.n_q_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim, f = c.ffn_dim;
  const int wdt = m->wdt;
  void* qb = m->ws + P.q;     // rotated queries, weight dtype
  void* aob = m->ws + P.ao;   // attention output, weight dtype
  void* actb = m->ws + P.act; // SwiGLU output, weight dtype
  // Every prefill kernel waits for its predecessor before touching memory, so
  // each one is launched early and its prologue overlaps the previous tail.
  const bool pdl = !(m->flags & LADDER_FLAG_NO_PDL);
  // GEMM A operands as hi/lo pairs (the default) or rounded once (LADDER_FLAG_FAST_PREFILL).
  const bool wide = !(m->flags & LADDER_FLAG_FAST_PREFILL);
  const size_t Mp = P.m_pad;
  const size_t lo_ao = wide ? Mp * qd : 0;
  const int lo_act = wide ? (int)Mp : 0;
  const int n_mod = 2 * c.n_layers;

  // RMSNorm split between the writer of each stream state x_j (the embedding, or
  // a residual GEMM's epilogue) and the GEMMs of the modules that read it: the
  // writer leaves x_j ⊙ g_c for each reading module c (slot c % 2) and the
  // per-chunk sums of squares of x_j (slot j % 3); reading GEMM c scales its rows
  // by rsqrt(mean(x_j^2) + eps).  Module c reads x_{input_index(c)}, one or two
  // modules back, so at most two operands are pending at any time, and state j's
  // sums are read by module j + 2 at the latest, before state j + 3 is written.
  auto gain_of = [&](int k) -> const void* {
    const LayerW& L = m->layers[(k - 1) / 2];
    return (k & 1) ? L.attn_norm : L.mlp_norm;
  };
  auto norm_out = [&](int j) {
    NormOut o{};
    o.ld_ss = (int)Mp;
    o.u_lo = wide ? Mp * d : 0;
    int n = 0;
    for (int k = j + 1; k <= j + 2 && k <= n_mod; ++k)
      if (m->input_index(k) == j) {
        o.u[n] = m->ws + P.xn[k % 2];
        o.g[n] = gain_of(k);
        ++n;
      }
    if (n) o.ss = m->at<float>(P.ssq[j % 3]);
    return o;
  };
  auto reads_norm = [&](GemmParams& g, int k) {
    g.ss_in = m->at<float>(P.ssq[m->input_index(k) % 3]);
    g.nss = d / 128;
    g.ld_ss = (int)Mp;
    g.inv_k = 1.0f / (float)d;
    g.eps = c.norm_eps;
  };

  LAUNCH(launch_embed_norm(tokens, M, m->embed, wdt, d, c.vocab, m->X(0), norm_out(0), m->err(), s, pdl), 1);
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerMaps& T = m->maps[l];
    const KvLayer kvl = kv->layer(l);
    {
      const int k = 2 * l + 1;
      GemmParams g{};
      g.M = M; g.N = qd + 2 * kvd; g.K = d;
      g.out_h = qb; g.ldo = qd; g.nq_hd = qd; g.nkv_hd = kvd;
      g.rope_cos = m->at<float>(P.rope_cos); g.rope_sin = m->at<float>(P.rope_sin);
      g.row_b = d_row_b; g.row_pos = d_row_pos; g.kv = kvl;
      reads_norm(g, k);
      LAUNCH(launch_gemm_tc(&m->map_xn[k % 2], &T.wq, &T.wk, &T.wv, nullptr, nullptr, g, GEMM_QKV, wdt, m->num_sms,
                            m->err(), s, pdl, wide), 1);

      AttnPrefillParams a{};
      a.q = qb; a.kv = kvl; a.seq_start = d_start; a.seq_len = d_lens;
      a.n_q = c.n_q_heads; a.scale = 1.0f / sqrtf((float)c.head_dim); a.out = aob; a.lo_off = lo_ao;
      LAUNCH(launch_attn_prefill_tcgen05(&m->map_q, &kv->maps[l], a, c.head_dim, wdt, B, max_len, m->err(), s, pdl), 1);

      GemmParams o{};
      o.M = M; o.N = d; o.K = qd; o.out_f = m->X(k); o.ldo = d; o.x_res = m->X(k - 1);
      o.nout = norm_out(k);
      LAUNCH(launch_gemm_tc(&m->map_ao, &T.wo, nullptr, nullptr, &m->map_x[(k - 1) % 3], &m->map_x[k % 3], o,
                            GEMM_RESID, wdt, m->num_sms, m->err(), s, pdl, wide), 1);
    }
    {
      const int k = 2 * l + 2;
      GemmParams g{};
      g.M = M; g.N = f; g.K = d; g.out_h = actb; g.ldo = f; g.lo_row = lo_act;
      reads_norm(g, k);
      LAUNCH(launch_gemm_tc(&m->map_xn[k % 2], &T.gate, &T.up, nullptr, nullptr, &m->map_act_st, g, GEMM_GATEUP, wdt,
                            m->num_sms, m->err(), s, pdl, wide), 1);
      GemmParams o{};
      o.M = M; o.N = d; o.K = f; o.out_f = m->X(k); o.ldo = d; o.x_res = m->X(k - 1);
      o.nout = norm_out(k);
      LAUNCH(launch_gemm_tc(&m->map_act, &T.down, nullptr, nullptr, &m->map_x[(k - 1) % 3], &m->map_x[k % 3], o,
                            GEMM_RESID, wdt, m->num_sms, m->err(), s, pdl, wide), 1);
    }
  }
  GemvParams h{};
  h.carve = m->gemv_carve;
  h.ldx = d; h.g = m->final_norm; h.eps = c.norm_eps; h.K = d;
  h.w0 = m->lm_head; h.n_tasks = c.vocab / 2; h.ldo = c.vocab;
  h.err = m->err();
  m->splitk(h, SK_LMHEAD);
  if (all_rows) {
    // Every packed row, max_batch rows per launch (the row count the lm_head
    // projection's workspace is planned for); then each sequence's last row.
    for (int r0 = 0; r0 < M; r0 += Bm) {
      GemvParams hc = h;
      hc.x = m->X(2 * c.n_layers) + (size_t)r0 * d;
      hc.B = M - r0 < Bm ? M - r0 : Bm;
      hc.out = logits + (size_t)r0 * c.vocab;
      LAUNCH(launch_gemv(hc, GEMV_LOGITS, m->wdt, m->num_sms, s, pdl), gemv_launch_count(hc.B, hc.K, GEMV_LOGITS));
    }
    if (next_tok)
      for (int b = 0; b < B; ++b)
        LAUNCH(launch_argmax(logits + (size_t)last[b] * c.vocab, 1, c.vocab, m->at<float>(P.am_v), m->at<int>(P.am_i),
                             kArgmaxBlocks, next_tok + b, s, pdl), 2);
    LAUNCH(launch_set_lens(d_lens, B, kv->seq_lens, s, pdl), 1);
    for (int b = 0; b < B; ++b) kv->host_lens[b] = host_lens[b];
    return LADDER_OK;
  }
  float* xlast = m->at<float>(P.xlast);
  LAUNCH(launch_gather_rows(m->X(2 * c.n_layers), d, d_last, B, xlast, s, pdl), 1);
  h.x = xlast; h.B = B; h.out = logits;
  LAUNCH(launch_gemv(h, GEMV_LOGITS, m->wdt, m->num_sms, s, pdl), gemv_launch_count(B, h.K, GEMV_LOGITS));
  if (next_tok && m->samp_t > 0.f)  // the sampled token takes position T_b
    LAUNCH(launch_sample(logits, B, c.vocab, m->samp_t, m->samp_k, m->samp_seed, d_lens, 0, next_tok, s, pdl), 1);
  else if (next_tok)
    LAUNCH(launch_argmax(logits, B, c.vocab, m->at<float>(P.am_v), m->at<int>(P.am_i), kArgmaxBlocks, next_tok, s, pdl), 2);
  LAUNCH(launch_set_lens(d_lens, B, kv->seq_lens, s, pdl), 1);
  for (int b = 0; b < B; ++b) kv->host_lens[b] = host_lens[b];
  return LADDER_OK;
}

// ---------------------------------------------------------------------------
// Standalone sampler
// ---------------------------------------------------------------------------
int ladder_sample(const float* logits, int32_t B, int32_t V, float temperature, int32_t top_k, uint64_t seed,
                  const int32_t* positions, int32_t pos_offset, int32_t* out, ladder_stream_t stream) {
  if (!logits || !positions || !out) return fail(LADDER_ERR_INVALID, "ladder_sample: null pointer");
  if (B < 1 || V < 1) return fail(LADDER_ERR_INVALID, "ladder_sample: B=%d V=%d", B, V);
  if (!(temperature > 0.f)) return fail(LADDER_ERR_INVALID, "ladder_sample: temperature must be > 0");
  CUDA_TRY(launch_sample(logits, B, V, temperature, top_k, seed, positions, pos_offset, out,
                         reinterpret_cast<cudaStream_t>(stream), false));
  return LADDER_OK;
}

// ---------------------------------------------------------------------------
// Standalone decode attention
// ---------------------------------------------------------------------------
namespace {

int check_attention_shape(int32_t B, int32_t n_q, int32_t n_kv, int32_t hd, int32_t page_size, int32_t max_position) {
  if (B <= 0) return fail(LADDER_ERR_INVALID, "B=%d must be positive", B);
  if (hd != 64 && hd != 128) return fail(LADDER_ERR_UNSUPPORTED, "head_dim=%d: only 64 and 128 are supported", hd);
  if (n_q <= 0 || n_kv <= 0 || n_q % n_kv) return fail(LADDER_ERR_INVALID, "n_q_heads must be a multiple of n_kv_heads");
  if (n_q / n_kv > 8) return fail(LADDER_ERR_UNSUPPORTED, "more than 8 query heads per KV head");
  if (page_size != 16 && page_size != 32 && page_size != 64)
    return fail(LADDER_ERR_INVALID, "page_size=%d must be 16, 32 or 64", page_size);
  if (max_position < 0) return fail(LADDER_ERR_INVALID, "max_position must be >= 0");
  return LADDER_OK;
}

size_t attention_scratch(int32_t B, int32_t n_q, int32_t hd, int32_t max_position) {
  const size_t nsplit = ((size_t)max_position + 1 + kSplitLen - 1) / kSplitLen;
  const size_t po = align_up((size_t)B * n_q * nsplit * hd * 4, 256);
  return po + (size_t)B * n_q * nsplit * 2 * 4;
}

}  // namespace

extern "C" size_t ladder_attention_decode_scratch_bytes(int32_t B, int32_t n_q_heads, int32_t head_dim,
                                                        int32_t max_position) {
  if (B <= 0 || n_q_heads <= 0 || head_dim <= 0 || max_position < 0) return 0;
  return attention_scratch(B, n_q_heads, head_dim, max_position);
}

extern "C" int ladder_attention_decode(const float* q, const void* kv_layer, int32_t kv_dtype,
                                       const int32_t* block_table, int32_t max_pages_per_seq,
                                       const int32_t* positions, int32_t B, int32_t n_q_heads, int32_t n_kv_heads,
                                       int32_t head_dim, int32_t page_size, float scale, int32_t max_position,
                                       float* out, void* scratch, size_t scratch_bytes, ladder_stream_t stream) {
  if (!q || !kv_layer || !block_table || !positions || !out || !scratch) return fail(LADDER_ERR_INVALID, "NULL argument");
  if (kv_dtype != LADDER_DTYPE_BF16 && kv_dtype != LADDER_DTYPE_F16) return fail(LADDER_ERR_INVALID, "unknown kv_dtype %d", kv_dtype);
  int rc = check_attention_shape(B, n_q_heads, n_kv_heads, head_dim, page_size, max_position);
  if (rc) return rc;
  if (max_pages_per_seq <= 0 || (int64_t)max_pages_per_seq * page_size < (int64_t)max_position + 1)
    return fail(LADDER_ERR_CAPACITY, "max_pages_per_seq * page_size must cover max_position + 1");
  if (!aligned(q, 16) || !aligned(kv_layer, 16) || !aligned(out, 16) || !aligned(scratch, 16))
    return fail(LADDER_ERR_INVALID, "q, kv_layer, out and scratch must be 16-byte aligned");
  const size_t need = attention_scratch(B, n_q_heads, head_dim, max_position);
  if (scratch_bytes < need) return fail(LADDER_ERR_CAPACITY, "scratch too small: %zu < %zu bytes", scratch_bytes, need);
  AttnDecodeParams a{};
  a.q = q;
  a.kv.base = const_cast<void*>(kv_layer);
  a.kv.block_table = block_table;
  a.kv.max_pages = max_pages_per_seq;
  a.kv.page_size = page_size;
  a.kv.page_shift = __builtin_ctz((unsigned)page_size);
  a.kv.n_kv = n_kv_heads;
  a.kv.head_dim = head_dim;
  a.seq_lens = positions;
  a.n_q = n_q_heads;
  a.split_len = kSplitLen;
  a.nsplit = (max_position + 1 + kSplitLen - 1) / kSplitLen;
  a.scale = scale;
  a.part_o = static_cast<float*>(scratch);
  a.part_ml = reinterpret_cast<float*>(static_cast<char*>(scratch) +
                                       align_up((size_t)B * n_q_heads * a.nsplit * head_dim * 4, 256));
  a.out = out;
  cudaError_t e = launch_attn_decode(a, B, n_kv_heads, head_dim, kv_dtype, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(LADDER_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  return LADDER_OK;
}
