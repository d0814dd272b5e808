/* fq -- Qwen3 quantized single-token decode on GB300 (sm_103a): the C ABI.
 *
 * The calls follow the problem statement of the fucina Qwen3 pages:
 *   - "The qwen3 descriptor runner": the model as data (Descriptor) plus an interpreter
 *     (Model) that runs fused norm+QKV, half-rope QK-norm, grouped causal attention over
 *     a shared KvCache and a dense or softmax-top-k MoE FFN;
 *   - "14. Model families", section 14.1 (forward/decode surface: forwardStep contract,
 *     read-only Model, caller-owned logits, one context + cache per concurrent stream)
 *     and section 14.2 "Qwen3 -- dense and MoE" (Config fields and validation, load
 *     specifics, lockstep forwardStepBatch, KvCache).
 *
 * Conventions for every entry point:
 *   - Return an fq_status; on any contract error nothing is launched and no state
 *     changes.  fq_last_error() gives a thread-local message for the last failure.
 *   - "device" pointers are CUDA device addresses of the current device; "host"
 *     pointers are ordinary CPU memory.  The library never takes ownership of caller
 *     buffers and never retains a pointer past the call, except where stated.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All device work of
 *     a call is enqueued on it; calls return without synchronising unless stated.
 *   - A model is immutable after load.  Concurrent calls on one model are allowed with
 *     distinct caches and distinct streams (section 14.1: one context + one cache per
 *     concurrent stream); scratch memory is kept per stream.
 */
#ifndef FQ_H
#define FQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Error set of section 14.2 (InvalidConfig, InvalidSequenceLength, MismatchedKvCaches)
 * plus the cache's KvCacheOverflow (section 14.1 forwardStep contract) and the runtime
 * failures a GPU library adds. */
typedef enum fq_status {
    FQ_OK = 0,
    FQ_ERR_INVALID_CONFIG = 1,          /* descriptor rejected (section 14.2 validation) */
    FQ_ERR_INVALID_SEQUENCE_LENGTH = 2, /* pos0 != kv len, or an empty batch */
    FQ_ERR_KV_CACHE_OVERFLOW = 3,       /* len + new positions > capacity */
    FQ_ERR_MISMATCHED_KV_CACHES = 4,    /* duplicate caches, other model, other dtype */
    FQ_ERR_INVALID_ARGUMENT = 5,        /* null pointer, bad shape/dtype, token out of range */
    FQ_ERR_OUT_OF_MEMORY = 6,           /* device allocation failed */
    FQ_ERR_CUDA = 7,                    /* a CUDA runtime call failed (message has the text) */
    FQ_ERR_DEVICE_TIMEOUT = 8,          /* a bounded device wait gave up (fq_check_device) */
    FQ_ERR_UNSUPPORTED = 9              /* valid per the pages but not built here (e.g. head_dim != 128) */
} fq_status;

typedef enum fq_dtype {
    FQ_F32 = 0,
    FQ_BF16 = 1,
    FQ_Q8_0 = 8,   /* ggml Q8_0: 34-byte blocks = fp16 d + 32 int8, x = d*q           */
    FQ_Q4_K = 12   /* ggml Q4_K: 144-byte super-blocks of 256: fp16 d, fp16 dmin,
                      12 bytes of 6-bit scales/mins, 128 bytes of nibbles              */
} fq_dtype;

/* Section 14.2 Config.  moe_expert_top_p must be 1.0 (full top-k).  max_positions bounds
 * every cache capacity (0 selects 40960) and sizes the rotary table. */
typedef struct fq_desc_params {
    uint32_t vocab_size, hidden_size, intermediate_size, num_layers;
    uint32_t num_attention_heads, num_key_value_heads, head_dim;
    float rms_norm_eps, rope_theta;
    uint32_t num_experts;           /* 0 = dense */
    uint32_t num_experts_used;
    uint32_t moe_intermediate_size;
    int32_t norm_topk_prob;         /* renormalise the selected router weights */
    float moe_expert_top_p;
    uint32_t max_positions;
} fq_desc_params;

/* A validated descriptor (the pages' Descriptor: the model as data). */
typedef struct fq_desc {
    fq_desc_params p;
    uint32_t magic;                 /* set by fq_desc_init */
} fq_desc;

/* Section 14.2 validation: rejects zero dims or heads, num_attention_heads not divisible
 * by num_key_value_heads, odd head_dim, an inconsistent MoE trio (all three zero or all
 * set, num_experts_used <= num_experts), top_p != 1 -> FQ_ERR_INVALID_CONFIG.  Valid
 * configurations the kernels do not cover (head_dim != 128, hidden_size not a multiple of
 * 256, more than 256 experts or top-k above 8) -> FQ_ERR_UNSUPPORTED.  d: host, written. */
fq_status fq_desc_init(fq_desc* d, const fq_desc_params* p);

/* One packed host tensor, ggml row-major: `rows` rows of `cols` elements; for quantised
 * dtypes a row is cols/32*34 (Q8_0) or cols/256*144 (Q4_K) bytes.  data: host. */
typedef struct fq_tensor {
    fq_dtype dtype;
    uint64_t rows, cols;
    const void* data;
} fq_tensor;

/* Per-layer tensors (the GGUF blk.N.* set).  Dense layers fill w_gate/w_up/w_down; MoE
 * layers fill router (f32 [num_experts, hidden]) and the expert stacks gate_exps and
 * up_exps ([num_experts*moe_ffn, hidden], expert e's rows contiguous) and down_exps
 * ([num_experts*hidden, moe_ffn]).  Norm gains are f32. */
typedef struct fq_layer_src {
    fq_tensor attn_norm, wq, wk, wv, q_norm, k_norm, wo, ffn_norm;
    fq_tensor w_gate, w_up, w_down;
    fq_tensor router, gate_exps, up_exps, down_exps;
} fq_layer_src;

/* tok_embd [vocab, hidden], output_norm f32 [hidden], output [vocab, hidden]; a NULL
 * output.data means tied embeddings (section 14.2 load specifics).  A NULL tok_embd.data
 * (with a NULL output) loads a layer-only model that serves fq_layer_step alone; the
 * decode entry points reject it with FQ_ERR_INVALID_ARGUMENT.  layers: host array of
 * num_layers entries. */
typedef struct fq_weight_src {
    fq_tensor tok_embd, output_norm, output;
    const fq_layer_src* layers;
} fq_weight_src;

typedef struct fq_model fq_model;
typedef struct fq_kv fq_kv;

/* Load: copies every tensor to device memory the model owns (section 14.1: weights stay
 * in their GGUF dtype, no global dequantisation), fusing q/k/v into one QKV matrix and
 * gate/up into one gate_up matrix (section 14.1 fuseLinear), and repacking Q8_0 blocks into
 * 16-byte-aligned planes.  Dtypes: linears Q8_0 or Q4_K (one dtype for the attention and
 * FFN linears of every layer), embedding/output Q8_0 or Q4_K, norms and router f32.
 * Synchronises `stream` before returning; src is not retained.  *out: host, written.
 * Errors: INVALID_ARGUMENT (shape/dtype mismatch), OUT_OF_MEMORY, CUDA. */
fq_status fq_load_weights(const fq_desc* d, const fq_weight_src* src, void* stream, fq_model** out);
void fq_model_free(fq_model* m);

/* KvCache (section 14.2 initKvCache; uniform geometry layers x kv heads x head_dim x
 * capacity) in device memory owned by the cache, len = 0.  dtype FQ_F32, FQ_BF16 or FQ_Q8_0
 * (the runner page's q8_0 cache: half the bf16 bytes; decode scores it through the integer
 * q8 x q8 path, q quantised to Q8_0 blocks like a cached row).  Layout: [layer][kv_head]
 * [capacity][head_dim] values for K and again for V; Q8_0 stores int8 codes in that layout
 * and, after them, [layer][kv_head][capacity rounded up to even][head_dim / 32] fp16 block
 * scales.  New rows are quantised with ggml's Q8_0 rule (d = fp16(amax / 127), codes x / d
 * rounded half away from zero), the same as fq_quantize_q8_0. */
fq_status fq_kv_init(const fq_model* m, uint32_t capacity, fq_dtype kv_dtype, fq_kv** out);
void fq_kv_free(fq_kv* kv);
uint32_t fq_kv_len(const fq_kv* kv);
uint32_t fq_kv_capacity(const fq_kv* kv);

/* Bulk-write positions [pos, pos+n_pos) of one layer: k, v are device [n_pos][kv_heads]
 * [head_dim] in the cache dtype (Q8_0: ggml blocks, [n_pos][kv_heads][head_dim / 32] of 34
 * bytes each, any alignment).  pos must equal the cache's len (contiguous fill),
 * pos + n_pos <= capacity.  Does not change len; fq_kv_commit(kv, len) sets it once every
 * layer holds the positions (len <= capacity, len >= current len).  Errors:
 * INVALID_SEQUENCE_LENGTH (pos != len), KV_CACHE_OVERFLOW, INVALID_ARGUMENT. */
fq_status fq_kv_append(fq_kv* kv, uint32_t layer, uint32_t pos, uint32_t n_pos, const void* k, const void* v,
                       void* stream);
fq_status fq_kv_commit(fq_kv* kv, uint32_t len);
/* Rewind to a shorter length (the runner page's decoder contract lists rewind among the
 * cache capabilities): len <= current len, else INVALID_SEQUENCE_LENGTH.  Positions from
 * len on keep stale contents until later steps overwrite them.  Host-side only. */
fq_status fq_kv_rewind(fq_kv* kv, uint32_t len);
/* Copy positions [pos, pos+n_pos) of one layer out to device buffers in the cache dtype
 * (Q8_0: ggml blocks as fq_kv_append takes them). */
fq_status fq_kv_read(const fq_kv* kv, uint32_t layer, uint32_t pos, uint32_t n_pos, void* k, void* v,
                     void* stream);

/* One decoder layer for one token at absolute position pos == len (section 14.1
 * forwardStep, restricted to one block): x device f32 [hidden] is the residual stream,
 * updated in place; appends this layer's k/v at pos; does not advance len.  Errors:
 * INVALID_SEQUENCE_LENGTH, KV_CACHE_OVERFLOW, INVALID_ARGUMENT. */
fq_status fq_layer_step(const fq_model* m, uint32_t layer, fq_kv* kv, uint32_t pos, float* x, void* stream);

/* Section 14.1 forwardStep over len >= 1 tokens of one sequence: tokens (host, [len]) at
 * positions pos0..pos0+len-1, every row's K/V appended, len advanced by len, the last row's
 * logits written to `logits` (device f32 [vocab], caller-owned; NULL: append only).  A
 * prefill is one call on a fresh cache at pos0 == 0, and its logits equal forwardLastLogits
 * over the same ids.  Runs in passes of up to 32 rows: the dense projections of a pass read
 * every weight once for all its rows (tensor cores from 8 rows); each row attends causally
 * to the cache and the rows before it.  Errors (state unchanged): INVALID_SEQUENCE_LENGTH
 * (len == 0, pos0 != len), KV_CACHE_OVERFLOW (len + n > capacity), INVALID_ARGUMENT (a token
 * out of range, no embedding, or logits without an LM head), MISMATCHED_KV_CACHES (another
 * model's cache).  After a CUDA error the cache length covers the passes enqueued. */
fq_status fq_forward_step(const fq_model* m, fq_kv* kv, const int32_t* tokens, uint32_t len, uint32_t pos0,
                          float* logits, void* stream);

/* Section 14.1 forwardStep for one token: embedding row of `token`, every layer,
 * output norm, LM head -> logits device f32 [vocab] (caller-owned).  Contract: pos0 ==
 * len (else INVALID_SEQUENCE_LENGTH), len + 1 <= capacity (else KV_CACHE_OVERFLOW).
 * Advances len by one.  logits may be NULL (the step still appends K/V). */
fq_status fq_decode_step(const fq_model* m, fq_kv* kv, int32_t token, uint32_t pos0, float* logits,
                         void* stream);

/* Section 14.2 forwardStepBatch: one token per stream, stream s against caches[s] at its
 * own position (ragged); logits device f32 [n][vocab].  caches: host array of n distinct
 * caches of this model with one dtype (else MISMATCHED_KV_CACHES); tokens: host [n].
 * The dense trunk runs as one m=n pass over each weight; RoPE, KV append and attention
 * are per stream.  Every cache advances by one. */
fq_status fq_decode_step_batch(const fq_model* m, fq_kv* const* caches, uint32_t n, const int32_t* tokens,
                               float* logits, void* stream);

/* Section 14.1 forwardStepAllLogits, the verify pass of speculative decoding: the len
 * tokens (host [len], 1 <= len <= 64) of ONE sequence at positions pos0 .. pos0+len-1 in a
 * single pass, each attending causally to the cache and to the rows before it; logits of
 * every row -> device f32 [len][vocab] (caller-owned).  The same KV semantics as forwardStep:
 * pos0 == len (else INVALID_SEQUENCE_LENGTH, also for len outside 1..64), len + n <=
 * capacity (else KV_CACHE_OVERFLOW); advances len by len.  The dense trunk reads each weight
 * once for all rows (the tcgen05 GEMM from 8 rows on).  Equal, up to rounding, to len
 * consecutive fq_decode_step calls. */
fq_status fq_decode_step_all_logits(const fq_model* m, fq_kv* kv, const int32_t* tokens, uint32_t len, uint32_t pos0,
                                    float* logits, void* stream);

/* Greedy generation (section 14.1 generate, without the reset): n_steps decode steps on
 * the device, each feeding back the argmax (ties -> lowest id) of its own logits.
 * Stream s starts from first_tokens[s] (host [n]) at its cache len; tokens_out is device
 * int32 [n_steps][n] (the chosen ids); logits (device f32 [n][vocab] or NULL) holds the
 * last step's logits.  Caches advance by n_steps.  n = 1 is the single-stream loop. */
fq_status fq_decode_greedy(const fq_model* m, fq_kv* const* caches, uint32_t n, const int32_t* first_tokens,
                           uint32_t n_steps, int32_t* tokens_out, float* logits, void* stream);

/* ---- inspection (tests and tools; not the hot path) ---- */

/* Same as fq_decode_step_batch, also writing the residual stream after every layer to
 * layer_out (device f32 [layers][n][hidden]) and, for MoE models, the router choice to
 * route_idx (device int32 [layers][n][num_experts_used]) and route_w (device f32, same
 * shape) and the router logits before the softmax to route_logits (device f32
 * [layers][n][num_experts]); any of the four may be NULL. */
fq_status fq_decode_step_trace(const fq_model* m, fq_kv* const* caches, uint32_t n, const int32_t* tokens,
                               float* logits, float* layer_out, int32_t* route_idx, float* route_w,
                               float* route_logits, void* stream);

/* fq_layer_step that also copies the layer's intermediates out (device f32, any may be
 * NULL): qkv [(Hq + 2 Hkv) * head_dim] raw projections before QK-norm/rope (rows q | k | v),
 * attn [Hq * head_dim] attention output per q head, ffn [intermediate_size] SwiGLU
 * activations (dense models). */
fq_status fq_layer_step_trace(const fq_model* m, uint32_t layer, fq_kv* kv, uint32_t pos, float* x, float* qkv,
                              float* attn, float* ffn, void* stream);

/* Which weight to inspect with fq_dequant_rows. */
typedef enum fq_weight_id {
    FQ_W_TOK_EMBD = 0, FQ_W_OUTPUT = 1, FQ_W_Q = 2, FQ_W_K = 3, FQ_W_V = 4, FQ_W_O = 5,
    FQ_W_GATE = 6, FQ_W_UP = 7, FQ_W_DOWN = 8, FQ_W_GATE_EXPS = 9, FQ_W_UP_EXPS = 10, FQ_W_DOWN_EXPS = 11
} fq_weight_id;

/* Dequantise rows [row0, row0+n_rows) of one device-resident weight (as loaded, after
 * fusion and repacking) into out (device f32 [n_rows][cols]) with the same device
 * decoding the GEMV kernels use. */
fq_status fq_dequant_rows(const fq_model* m, uint32_t layer, fq_weight_id which, uint64_t row0, uint64_t n_rows,
                          float* out, void* stream);

/* ggml Q8_0 blocks (34 bytes per 32 values) of x[0, n) with the device quantiser a Q8_0
 * KvCache applies to q and to new k/v rows (runner page, "KV cache"): d = fp16(amax / 127)
 * rounded to nearest even, codes x / d rounded half away from zero and clamped to +-127, zero
 * when d is 0.  x: device f32, 16-byte aligned, n a multiple of 128; blocks: device, n / 32 * 34
 * bytes.  Errors: INVALID_ARGUMENT. */
fq_status fq_quantize_q8_0(const float* x, uint64_t n, void* blocks, void* stream);

/* y[b][r] = sum_k W[r][k] x[b][k] for b < n (n <= 64) over one device-resident weight, with
 * the launch configuration the decode step uses: x device f32 [n][cols], y device f32
 * [n][rows].  which: FQ_W_Q selects the whole fused QKV matrix (rows q | k | v),
 * FQ_W_GATE the fused gate_up matrix (rows interleaved gate_0, up_0, gate_1, ...),
 * FQ_W_O, FQ_W_DOWN, FQ_W_OUTPUT the others (layer ignored for FQ_W_OUTPUT). */
fq_status fq_gemv(const fq_model* m, uint32_t layer, fq_weight_id which, uint32_t n, const float* x, float* y,
                  void* stream);

/* fq_layer_step for callers that cannot allocate device memory at call time -- a host whose
 * allocator forbids allocations after start-up, code running while a CUDA graph is being
 * captured, an embedder that accounts for every device byte up front.  (The paper has no
 * counterpart; this is an interface of this library.)  Same arguments, contract, errors and
 * results as fq_layer_step, but it allocates nothing: all of the layer's scratch lives in one
 * 2 MiB array built into the library, which every GPU that loads the library holds until
 * the process exits.  A model + cache capacity whose layer scratch does not fit is rejected
 * with FQ_ERR_INVALID_ARGUMENT and a message giving the size (a 0.6B- or 8B-shaped dense layer
 * fits at any capacity up to 40960 positions).  The first call on a device looks up the
 * array's device address (once, with that device current), so make that first call before
 * any stream capture.  Every call shares the array: calls whose GPU work overlaps (other
 * streams, other threads) race and give wrong results; serialise them. */
fq_status fq_layer_step_noalloc(const fq_model* m, uint32_t layer, fq_kv* kv, uint32_t pos, float* x, void* stream);

/* Execution options of a model (no counterpart on the pages; they choose between equivalent
 * implementations of the same step).  Set them between steps, not while a step of the model
 * is in flight on another thread; a change drops the CUDA graphs captured so far.
 *   FQ_OPT_STEP_PATH          FQ_PATH_AUTO (default): a batch-1 step of a dense model with
 *                             a bf16 cache runs as one streamed persistent kernel (one
 *                             CTA per SM) whose producer warp copies the CTA's share of the
 *                             step's weights and cached K/V into shared memory ahead of the
 *                             activations; FQ_PATH_KERNELS: the
 *                             sequence of per-stage kernels (replayed from a CUDA graph).
 *   FQ_OPT_DEPENDENT_LAUNCH   0 (default) / 1: programmatic dependent launch between the
 *                             kernels of the sequence.
 *   FQ_OPT_GRAPHS             1 (default) / 0: capture the kernel sequence of a step once and
 *                             replay it, or launch the kernels directly every step.
 *   FQ_OPT_TENSOR_CORES       1 (default) / 0: tcgen05 GEMM for lockstep batches of 8 or more
 *                             rows, or the CUDA-core GEMV for every batch.
 * FQ_ERR_INVALID_ARGUMENT for an unknown option or value. */
typedef enum fq_option {
    FQ_OPT_STEP_PATH = 0, FQ_OPT_DEPENDENT_LAUNCH = 1, FQ_OPT_GRAPHS = 2, FQ_OPT_TENSOR_CORES = 3
} fq_option;
enum { FQ_PATH_AUTO = 0, FQ_PATH_KERNELS = 1 };
fq_status fq_set_option(fq_model* m, fq_option opt, int value);

/* *streamed = 1 when a step of n sequences with caches of kv_dtype runs as the streamed
 * persistent kernel under the model's current options, else 0.  Host-only. */
fq_status fq_step_path(const fq_model* m, uint32_t n, fq_dtype kv_dtype, int* streamed);

/* Number of kernels one step launches on `stream`: the kernel nodes of the CUDA graph most
 * recently replayed there by fq_decode_step / fq_decode_step_batch / fq_decode_greedy, or 1
 * when the step ran as the single streamed kernel (batch 1, dense model); 0 when nothing
 * has run there or the steps ran as direct launches.  Host-only; for accounting by
 * benchmarks. */
fq_status fq_step_kernels(const fq_model* m, void* stream, uint32_t* kernels);

/* Synchronise `stream` and report device-side failures recorded since the last check:
 * FQ_ERR_DEVICE_TIMEOUT when a kernel's bounded wait on its own copy pipeline or on another
 * CTA gave up (the kernel returned early; results of that step are invalid).  Clears the
 * record and, on a timeout, zeroes the arrival counters and tickets of every workspace of
 * the model (on each workspace's own stream), so that later steps start from a clean state. */
fq_status fq_check_device(const fq_model* m, void* stream);

/* Test hook for the failure path of the bounded device waits (no counterpart on the pages).
 * Launches the bulk-copy GEMV over the LM head with a producer that issues no copies, so
 * every consumer's bounded wait on its stage runs out (about a quarter second) with nothing
 * in flight; the kernel records the failure and returns without writing outputs.  The next
 * fq_check_device on `stream` reports FQ_ERR_DEVICE_TIMEOUT and re-arms the model's
 * workspaces, after which steps run normally.  FQ_ERR_UNSUPPORTED when the LM head is not
 * served by the bulk-copy GEMV (K % 256 != 0). */
fq_status fq_debug_wait_timeout(const fq_model* m, void* stream);

const char* fq_last_error(void);
const char* fq_status_str(fq_status s);

#ifdef __cplusplus
}
#endif
#endif
