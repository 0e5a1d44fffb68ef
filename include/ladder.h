/*
 * ladder.h — C ABI of libladder.so: the forward pass of a Ladder Transformer
 * (prefill and single-token decode) on one GB300 (sm_103a).
 *
 * What it computes.  A decoder of n_layers layers, each an attention module
 * followed by a SwiGLU MLP module, numbered k = 1 .. 2*n_layers.  The residual
 * stream starts at x_0 = E[token] and every module adds its output to it:
 *     x_k = x_{k-1} + h_k( RMSNorm(x_in(k)) )
 * In a standard layer x_in(k) = x_{k-1}.  In a ladder layer the module reads
 * the stream from one module further back, x_in(k) = x_{k-2}, which is the
 * staggered residual x_{i+1} = h_{i+1}(x_{i-1}) + x_i of "Ladder Residual:
 * Parallelism-Aware Architecture for Accelerating Large Model Inference"
 * (ICML 2025 paper notes, sections 研究背景与动机 "core idea" and 方法详解 /
 * 关键设计 "staggered residual connection").  The hybrid model of the same
 * notes (关键设计, "hybrid ladder adaptation") keeps the lower
 * n_standard_layers standard.  Choices where the pages are silent:
 *   - x_{-1} := x_0 (the first two ladder modules read the embedding);
 *   - the first ladder module above a standard block reads x_b, b = 2 *
 *     n_standard_layers (strict_boundary = 1 reads x_{b-1});
 *   - module internals follow the Llama-3.1 base: pre-norm RMSNorm with eps
 *     inside the square root, no biases, grouped-query attention where query
 *     head h uses KV head h / (n_q_heads / n_kv_heads), rotary embedding on
 *     interleaved pairs (2j, 2j+1) with angle p * theta^(-2j/head_dim);
 *   - logits are those of each sequence's last position; the greedy token is
 *     the argmax with the lowest index on ties.
 *
 * Precision.  Weights, KV cache, queries and prefill tensor-core operands in
 * one 16-bit type (weight_dtype: bf16, or fp16 holding bf16-valued weights
 * exactly), rounded to nearest even; accumulation and residual stream fp32.
 *
 * Ownership.  The caller allocates every device buffer (weights, workspace, KV
 * pool, block table, sequence lengths, outputs) and passes raw device
 * pointers; the library never allocates device memory.  Weights are borrowed
 * and must outlive the model.  Handles are host objects owned by the library
 * and released by the matching *_destroy call.
 *
 * Streams.  Every device-side call is asynchronous on the stream given
 * (a cudaStream_t, 0 = legacy default stream).  Decode also uses a second
 * stream owned by the model (the MLP chain of ladder layers, or the shard
 * reduces), forked from and joined back into the given stream by events within
 * the call, so all of a call's work is ordered before later work on the given
 * stream.  A model and its KV handle must not be used from two streams
 * at once.
 *
 * Errors.  Every int-returning call returns LADDER_OK (0) or a negative code.
 * Arguments are validated on the host before anything is launched, so a call
 * that fails validation leaves device state untouched.  ladder_last_error()
 * returns a thread-local message for the last failure.  Device-side checks
 * (a token id >= vocab) never trap: the kernel records an error word that
 * ladder_get_device_error() reads back.
 */
#ifndef LADDER_H
#define LADDER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ladder_stream_t; /* same handle as cudaStream_t */
typedef struct ladder_model ladder_model;
typedef struct ladder_kv ladder_kv;

enum {
  LADDER_OK = 0,
  LADDER_ERR_INVALID = -1,     /* bad argument (null, out of range, misaligned) */
  LADDER_ERR_CUDA = -2,        /* a CUDA runtime call failed */
  LADDER_ERR_CAPACITY = -3,    /* workspace, batch, sequence or KV capacity exceeded */
  LADDER_ERR_UNSUPPORTED = -4  /* valid but not implemented (a shape or option) */
};

/* Residual schedule selected by ladder_set_mode. */
enum {
  LADDER_RESIDUAL_CONFIG = 0,   /* as configured: standard below n_standard_layers, ladder above */
  LADDER_RESIDUAL_STANDARD = 1, /* every layer standard (the baseline model, same weights) */
  LADDER_RESIDUAL_PARALLEL = 2  /* every layer a parallel block: the attention and the MLP of layer l
                                   both read x_{2l}, each through its own RMSNorm gain, and the stream
                                   accumulates both outputs (x_{2l+1} = x_{2l} + A, x_{2l+2} =
                                   x_{2l+1} + M).  This is the plain reading of the Parallel-70B
                                   comparison model in the notes' 70B latency table (section
                                   实验关键数据), which the pages do not spell out. */
};

/* Flags for ladder_set_mode. */
enum {
  LADDER_FLAG_DECODE_GRAPH = 1, /* capture each decode step shape in a CUDA graph and replay it */
  LADDER_FLAG_NO_PDL = 2,       /* launch prefill and decode kernels without programmatic dependent launch */
  LADDER_FLAG_ALL_LOGITS = 4,   /* prefill writes the logits of every position (a debugging aid) */
  LADDER_FLAG_FAST_PREFILL = 8  /* prefill GEMM activations rounded once to 16 bits (see below) */
};
/* Prefill precision.  Decode projections read the fp32 stream directly.  The
 * prefill projections are tensor-core GEMMs whose activation operand (the
 * normalised rows into QKV and gate/up, the attention output into W_o, the
 * SwiGLU output into W_down) is 16-bit.  By default each activation is held as
 * a hi/lo pair, hi = its 16-bit rounding and lo = the rounding of what is
 * left, and every GEMM multiplies both by the same weight tile: the
 * activations enter with about 22 significant bits (fp16 storage) and the
 * GEMMs do twice the tensor-core work.  LADDER_FLAG_FAST_PREFILL rounds them
 * once instead (11 significant bits, half the work).  Rounding the
 * activations once is within max-abs 3e-2 / relative L2 1e-2 of an fp32
 * forward pass on shallow models, but on deep random-init models the
 * rounding noise of 32 to 80 layers adds up to more than that. */

/* Model dimensions and capacities.  All int32 fields must be positive unless
 * stated.  Shape rules: d_model, n_q_heads*head_dim and ffn_dim multiples of
 * 256; head_dim 64 or 128; n_q_heads a multiple of n_kv_heads with at most 8
 * query heads per KV head; vocab even. */
typedef struct {
  int32_t n_layers;
  int32_t n_standard_layers;  /* 0 .. n_layers: lower layers with the standard residual */
  int32_t d_model;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t ffn_dim;
  int32_t vocab;
  float rope_theta;
  float norm_eps;
  int32_t tie_embeddings;     /* 1: lm_head is the embedding table */
  int32_t rope_interleaved;   /* must be 1 (pairs (2j, 2j+1)); weights laid out for half-split
                                 pairs (j, j + head_dim/2) need each head's W_q and W_k rows
                                 reordered first (new row 2j = row j, 2j+1 = row j + head_dim/2) */
  int32_t shard_k;            /* 1 = off; 2, 4 or 8 = shard mode (see below) */
  int32_t page_size;          /* KV positions per page: 16, 32 or 64 */
  int32_t max_batch;          /* sequences per call, <= 64 */
  int32_t max_seq;            /* positions per sequence */
  int32_t max_prefill_tokens; /* packed prompt tokens per prefill call */
  int32_t strict_boundary;    /* 0: first ladder module reads x_b; 1: reads x_{b-1} */
  int32_t weight_dtype;       /* storage of weights and prefill tensor-core operands:
                                 LADDER_DTYPE_BF16 or LADDER_DTYPE_F16 */
  /* Rotary frequency scaling (Llama-3.1 checkpoints; the official code's
   * apply_rope_scaling, named in the paper's codewithpapers record).  Off when
   * rope_scale_factor <= 1 (all four fields zero).  Otherwise, with f_j =
   * rope_theta^(-2j/head_dim), wavelength w = 2 pi / f_j and L =
   * rope_original_max_pos: f_j stays when w < L / rope_high_freq_factor, becomes
   * f_j / rope_scale_factor when w > L / rope_low_freq_factor, and in between
   * (1 - s) f_j / rope_scale_factor + s f_j with s = (L / w - low) / (high - low).
   * Requires 0 < rope_low_freq_factor < rope_high_freq_factor and L > 0. */
  float rope_scale_factor;
  float rope_low_freq_factor;
  float rope_high_freq_factor;
  int32_t rope_original_max_pos;
} ladder_config;

/* Shard mode (shard_k = k > 1) stands in, on one GPU, for the tensor-parallel
 * split of the Ladder Residual notes (关键设计: each module's output is an
 * all-reduce of per-device partial sums).  In decode, the column-parallel
 * projections (QKV, gate/up) are unchanged, and the row-parallel ones (O,
 * down) produce k partial sums, one per block of n_q_heads/k heads or
 * ffn_dim/k columns; a reduce kernel on a second stream adds them, in the
 * fixed order 0..k-1, to the residual.  A ladder module does not wait for the
 * previous module's reduce, so the reduce overlaps its GEMVs; a standard
 * module waits for it.  Requires n_q_heads, n_kv_heads divisible by k and
 * n_q_heads*head_dim/k, ffn_dim/k multiples of 256, ffn_dim/k at most 16384
 * (a decode GEMV of 2 rows: 8192; of 3 or 4 rows: 4096, else the decode step
 * returns LADDER_ERR_CUDA).  Prefill is unsharded (the
 * same function, up to fp32 reassociation). */

/* Storage types.  bf16-valued weights convert to fp16 exactly when
 * 2^-17 <= |w| <= 65504.  The KV cache, the prefill queries and the prefill
 * tensor-core operands (normalised activations, attention output, SwiGLU
 * output) use the same type as the weights; fp16 carries 3 more mantissa
 * bits than bf16. */
enum { LADDER_DTYPE_BF16 = 0, LADDER_DTYPE_F16 = 1 };

/* Weights: device pointers of the configured weight_dtype (bf16 or fp16),
 * row-major [out_features, in_features] unless stated, 16-byte aligned.  Per-layer fields are HOST arrays of n_layers device
 * pointers; the library copies the pointer values during ladder_create.
 *   embed [vocab, d_model]; final_norm [d_model]; lm_head [vocab, d_model]
 *   (ignored when tie_embeddings); attn_norm, mlp_norm [d_model];
 *   wq [n_q_heads*head_dim, d_model]; wk, wv [n_kv_heads*head_dim, d_model];
 *   wo [d_model, n_q_heads*head_dim]; w_gate, w_up [ffn_dim, d_model];
 *   w_down [d_model, ffn_dim]. */
typedef struct {
  const void* embed;
  const void* final_norm;
  const void* lm_head;
  const void* const* attn_norm;
  const void* const* wq;
  const void* const* wk;
  const void* const* wv;
  const void* const* wo;
  const void* const* mlp_norm;
  const void* const* w_gate;
  const void* const* w_up;
  const void* const* w_down;
} ladder_weights;

/* Sizes the caller must allocate: device workspace bytes for ladder_create and
 * bytes of one KV page (all layers: n_layers * 2 * n_kv_heads * page_size *
 * head_dim * 2).  Either output pointer may be NULL. */
int ladder_query_sizes(const ladder_config* cfg, size_t* workspace_bytes, size_t* kv_page_bytes);

/* Create a model over borrowed weights.  `workspace` is a device buffer of at
 * least the queried size, 256-byte aligned, owned by the caller and reserved
 * for this model until ladder_destroy.  Initialisation kernels (rotary tables)
 * run on `stream`. */
int ladder_create(const ladder_config* cfg, const ladder_weights* w, void* workspace,
                  size_t workspace_bytes, ladder_stream_t stream, ladder_model** out);
void ladder_destroy(ladder_model* m);

/* Residual schedule (LADDER_RESIDUAL_*) and flags (LADDER_FLAG_*). */
int ladder_set_mode(ladder_model* m, int residual_mode, int flags);

/* Next-token rule for the next_tok outputs of ladder_prefill and
 * ladder_decode_step.  temperature <= 0 (the default): greedy argmax, lowest
 * index on ties.  temperature > 0: temperature / top-k sampling, read from the
 * generation helpers the paper's codewithpapers record names
 * (logits_to_probs, multinomial_sample_one_no_sync, sample): the logits are
 * scaled by 1 / max(temperature, 1e-5), those below the top_k-th largest are
 * dropped (top_k <= 0 or >= vocab keeps all; logits equal to the top_k-th
 * largest stay), and the token is argmax_i p_i / q_i with q_i ~ Exp(1): a
 * sample of the softmax p of the kept logits (the "exponential race"), taken
 * as argmax_i l_i / T - ln(-ln u_i).  The uniforms are SplitMix64 counters keyed
 * by (seed, batch row, position of the sampled token): the same seed, batch
 * and positions reproduce the same tokens.  The logits outputs are unchanged.
 * Returns LADDER_ERR_INVALID for a NaN temperature. */
int ladder_set_sampling(ladder_model* m, float temperature, int32_t top_k, uint64_t seed);

/* Paged KV cache.  `pool` is a device buffer of num_pages * kv_page_bytes,
 * 16-byte aligned, laid out in the weight dtype [n_layers][num_pages][2 (K, V)][n_kv_heads]
 * [page_size][head_dim]; keys are stored after rotation.  `block_table` is a
 * device int32 [max_batch][max_pages_per_seq], `seq_lens` a device int32
 * [max_batch]; both are caller-owned and written only by the library.
 * Position p of sequence b lives in page block_table[b][p / page_size] at
 * offset p % page_size. */
int ladder_kv_create(ladder_model* m, void* pool, int32_t num_pages, int32_t max_pages_per_seq,
                     int32_t* block_table, int32_t* seq_lens, ladder_kv** out);
void ladder_kv_destroy(ladder_kv* kv);

/* Assign pages: host_table is a HOST int32 [max_batch][max_pages_per_seq];
 * entries are page ids in [0, num_pages) or -1 for "none".  Assigned pages of
 * a sequence must be a prefix of its row, and no page may be assigned twice.
 * Copies the table to the device block table on `stream`. */
int ladder_kv_set_pages(ladder_kv* kv, const int32_t* host_table, ladder_stream_t stream);

/* Set every sequence length to 0 (on the device, on `stream`, and in the
 * library's host copy). */
int ladder_kv_reset(ladder_kv* kv, ladder_stream_t stream);

/* Host copy of the current length of sequence b, or -1 if b is out of range. */
int32_t ladder_kv_seq_len(const ladder_kv* kv, int32_t b);

/* Prefill B sequences from empty caches.  `tokens` is a device int32 array of
 * the sum of host_lens packed sequence after sequence; `host_lens` a HOST int32
 * [B].  Writes every position's K/V into the cache, sets seq_lens[b] =
 * host_lens[b], and writes the last position's logits to `logits` (device fp32
 * [B, vocab]) and, if `next_tok` is not NULL, the greedy tokens (device int32
 * [B]) (or sampled ones, see ladder_set_sampling).  Fails with
 * LADDER_ERR_CAPACITY when a sequence exceeds its assigned pages or max_seq,
 * or the packed total exceeds max_prefill_tokens, and with LADDER_ERR_INVALID
 * when B is outside 1 .. max_batch or a length is not positive (an empty batch
 * or an empty prompt); every check runs before the first launch.
 * With LADDER_FLAG_ALL_LOGITS set, `logits` receives one row per packed token
 * instead ([sum of host_lens, vocab], in packing order: the lm_head runs over
 * max_batch rows per launch) and next_tok the greedy token of each sequence's
 * last row; sampling is not available in that mode (LADDER_ERR_UNSUPPORTED
 * when a temperature is set and next_tok is not NULL). */
int ladder_prefill(ladder_model* m, ladder_kv* kv, const int32_t* tokens, const int32_t* host_lens,
                   int32_t B, float* logits, int32_t* next_tok, ladder_stream_t stream);

/* One decode step for sequences 0 .. B-1: token tokens[b] (device int32 [B])
 * is placed at position seq_lens[b]; writes logits (device fp32 [B, vocab]),
 * the greedy tokens to next_tok (device int32 [B], may equal `tokens`, may be
 * NULL) and increments every seq_lens[b].  B outside 1 .. max_batch fails
 * with LADDER_ERR_INVALID, a full sequence with LADDER_ERR_CAPACITY, before
 * any launch.  With LADDER_FLAG_DECODE_GRAPH the step is captured once per
 * (B, pointer set) and replayed afterwards. */
int ladder_decode_step(ladder_model* m, ladder_kv* kv, const int32_t* tokens, int32_t B,
                       float* logits, int32_t* next_tok, ladder_stream_t stream);

/* Reads and clears the device error word (synchronises `stream`).  *code is 0
 * when no kernel reported a problem, else an OR of: 1 = a token id was outside
 * [0, vocab) (its row used a zero embedding); 2 = a pipeline wait ran out of
 * time and the kernel stopped early; 4 = a projection produced inf or NaN in a
 * 16-bit output (for example an activation beyond the range of fp16 storage):
 * the prefill GEMMs' 16-bit operands and cache writes, and the decode
 * projection's K/V cache write. */
int ladder_get_device_error(ladder_model* m, ladder_stream_t stream, int32_t* code);

/* Number of kernel launches the last prefill / decode call issued (a decode
 * step replayed from a graph reports the launches inside the graph). */
int32_t ladder_last_launch_count(const ladder_model* m);

/* Kernel classes that the launch probe can time. */
enum {
  LADDER_PROBE_QKV = 0,     /* decode: RMSNorm + QKV GEMV + RoPE + KV write */
  LADDER_PROBE_ATTN = 1,    /* decode: paged attention (split + combine) */
  LADDER_PROBE_OUT = 2,     /* decode: O-projection GEMV + residual */
  LADDER_PROBE_GATEUP = 3,  /* decode: RMSNorm + gate/up GEMV + SwiGLU */
  LADDER_PROBE_DOWN = 4,    /* decode: down-projection GEMV + residual */
  LADDER_PROBE_LMHEAD = 5,  /* decode: final RMSNorm + lm_head GEMV */
  LADDER_PROBE_REDUCE = 6   /* decode, shard mode: the reduce of a module's partial sums */
};

/* Start timing every launch of one kernel class in the following eager
 * (non-graph) decode steps: a CUDA event pair is recorded on the launching
 * stream around each launch, up to max_launches (1 .. 65536).  Fails while
 * LADDER_FLAG_DECODE_GRAPH is set. */
int ladder_probe_begin(ladder_model* m, int kernel_class, int32_t max_launches);

/* Stop timing: waits for the recorded events and returns how many launches
 * were timed and the sum of their durations in milliseconds. */
int ladder_probe_end(ladder_model* m, int32_t* launches, float* total_ms);

/* Launch timeline of eager decode steps (a tracing aid; the pages have no
 * counterpart).  ladder_timeline_begin arms it for up to max_launches launches
 * (1 .. 65536) and records a reference event on `stream`; every launch of a
 * probe class (LADDER_PROBE_*) in the following eager decode steps then records
 * an event before and after it on the stream it runs on.  ladder_timeline_end
 * waits for the events and writes, for the first min(recorded, capacity)
 * launches in issue order, the stream (0 = the caller's, 1 = the model's second
 * stream), the class, and the start and end in milliseconds after the
 * reference event; *n receives that count.  The event records sit between
 * kernels, so a launch cannot overlap the previous kernel of its own stream
 * (programmatic dependent launch is defeated); overlap between the two streams
 * is what the timeline shows.  Fails while LADDER_FLAG_DECODE_GRAPH is set. */
int ladder_timeline_begin(ladder_model* m, int32_t max_launches, ladder_stream_t stream);
int ladder_timeline_end(ladder_model* m, int32_t capacity, int32_t* n, int32_t* streams, int32_t* classes,
                        float* start_ms, float* end_ms);

/* Decode attention as a standalone operation: the split-context paged GQA
 * attention that ladder_decode_step runs in every layer.  For each sequence b
 * the query q[b] (device fp32 [B][n_q_heads*head_dim], already rotated) sits
 * at position positions[b] (device int32 [B]) and attends causally over the
 * cached positions 0 .. positions[b] of `kv_layer`, one layer of the pool:
 * [num_pages][2][n_kv_heads][page_size][head_dim] of kv_dtype
 * (LADDER_DTYPE_BF16 or LADDER_DTYPE_F16), addressed through
 * block_table (device int32 [B][max_pages_per_seq]).  Query head h reads KV
 * head h / (n_q_heads / n_kv_heads); scores are scaled by `scale`.  Writes
 * out (device fp32 [B][n_q_heads*head_dim]).  `scratch` is a caller-owned
 * device buffer of at least ladder_attention_decode_scratch_bytes(...) bytes,
 * 16-byte aligned, for the per-split partial results; every positions[b]
 * must be <= max_position (host int).  Same shape rules as the model
 * (head_dim 64 or 128, at most 8 query heads per KV head, page_size 16, 32
 * or 64). */
size_t ladder_attention_decode_scratch_bytes(int32_t B, int32_t n_q_heads, int32_t head_dim, int32_t max_position);
int ladder_attention_decode(const float* q, const void* kv_layer, int32_t kv_dtype, const int32_t* block_table,
                            int32_t max_pages_per_seq, const int32_t* positions, int32_t B, int32_t n_q_heads,
                            int32_t n_kv_heads, int32_t head_dim, int32_t page_size, float scale,
                            int32_t max_position, float* out, void* scratch, size_t scratch_bytes,
                            ladder_stream_t stream);

/* Decode attention that allocates nothing.  No counterpart on the pages: this
 * is a library convenience.  Same arguments and result as
 * ladder_attention_decode, minus the scratch buffer, for callers that cannot
 * allocate device memory (code running while a CUDA graph is being captured,
 * plugins whose host framework owns all device memory, loops that must not
 * stall on an allocation).  The partials live in a file-scope device array of
 * LADDER_STATIC_SCRATCH_BYTES bytes that every GPU running this code keeps
 * until the process exits.  Calls whose partials need more than that fail with
 * LADDER_ERR_CAPACITY (need = ladder_attention_decode_scratch_bytes(B,
 * n_q_heads, head_dim, max_position)).  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current
 * and keeps it for the life of the process; make that first call before any
 * stream capture.  A device reset (cudaDeviceReset) unloads the library's
 * device code and with it the array, so the kept address is no longer valid:
 * do not call this entry point on a device after resetting it in the same
 * process.  All calls share the one array: calls that can overlap on the GPU
 * (on different streams, or from different threads) race on it and must be
 * serialised by the caller. */
#define LADDER_STATIC_SCRATCH_BYTES (8u << 20)
int ladder_attention_decode_noalloc(const float* q, const void* kv_layer, int32_t kv_dtype,
                                    const int32_t* block_table, int32_t max_pages_per_seq,
                                    const int32_t* positions, int32_t B, int32_t n_q_heads, int32_t n_kv_heads,
                                    int32_t head_dim, int32_t page_size, float scale, int32_t max_position,
                                    float* out, ladder_stream_t stream);

/* Standalone sampler (the kernel behind ladder_set_sampling), for callers with
 * their own logits: logits is a device fp32 [B][V] row-major array, positions a
 * device int32 [B] array; row b draws with position positions[b] + pos_offset.
 * out is a device int32 [B] array.  temperature must be > 0 (greedy decoding
 * is the model's argmax).  Asynchronous on `stream`; allocates nothing. */
int ladder_sample(const float* logits, int32_t B, int32_t V, float temperature, int32_t top_k, uint64_t seed,
                  const int32_t* positions, int32_t pos_offset, int32_t* out, ladder_stream_t stream);

/* Thread-local message describing the last failed call on this thread. */
const char* ladder_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* LADDER_H */
