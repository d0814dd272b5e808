/* Oracle for the Qwen3 single-token decode step -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU implementation in f64 of what the fucina Qwen3 pages define:
 *   - "The qwen3 descriptor runner" (block style .fused: fused norm+QKV, half-rope
 *     QK-norm, grouped causal attention over the KvCache, dense / softmax-top-k MoE FFN);
 *   - "14. Model families", section 14.1 (forwardStep / forwardLastLogits contract) and
 *     section 14.2 "Qwen3 -- dense and MoE" (Config, validation, forwardStepBatch,
 *     routerTopK with normalize_selected, tied embeddings).
 * Storage formats (ggml Q8_0 / Q4_K blocks, fp16 / bf16 / f32) are emulated exactly;
 * all arithmetic on values is f64.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline leg may
 * load this library.  It shares no code with the CUDA path.
 */
#ifndef FQ_ORACLE_H
#define FQ_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { OR_Q8_0 = 0, OR_Q4_K = 1, OR_F32 = 2 };
/* what a KvCache stores: f32 values, bf16 values, or ggml Q8_0 blocks of 32 along head_dim */
enum { OR_KV_F32 = 0, OR_KV_BF16 = 1, OR_KV_Q8_0 = 2 };

typedef struct or_dims {
    int vocab, hidden, ffn, layers, n_q, n_kv, head_dim;
    double eps, theta;
    int n_exp, n_used, moe_ffn, norm_topk;
    int wtype;    /* OR_Q8_0 or OR_Q4_K: every linear except the f32 router */
    int kv_type;  /* OR_KV_F32, OR_KV_BF16 or OR_KV_Q8_0 */
} or_dims;

typedef struct or_model or_model;
typedef struct or_cache or_cache;

/* threads used for independent output rows (OpenMP); returns the count in effect */
int or_set_threads(int n);

/* ---- storage codecs ---- */
double   or_fp16_to_f64(uint16_t h);
uint16_t or_f64_to_fp16(double v);
double   or_bf16_to_f64(uint16_t h);
uint16_t or_f64_to_bf16(double v);
float    or_f64_to_f32(double v);
void or_dequant_q8_0(const uint8_t* blocks, size_t n, float* out);
void or_quant_q8_0(const float* x, size_t n, uint8_t* blocks);
void or_q4k_scale_min(const uint8_t* s12, int j, int* sc, int* mn);
void or_q4k_pack_scale_min(const int* sc, const int* mn, uint8_t* s12);
void or_dequant_q4_k(const uint8_t* blocks, size_t n, float* out);
void or_quant_q4_k(const float* x, size_t n, uint8_t* blocks);

/* ---- building blocks ---- */
void or_rmsnorm(const double* x, int n, const float* g, double eps, double* y);
void or_rope(double* v, int d, int pos, double theta);
void or_attention(const double* q, const float* K, const float* V, int T, int d, size_t row_stride,
                  double* o);
/* The q8_0-cache form of the above ("integer q8 x q8 score path"): q is rounded to f32 and
 * quantised to Q8_0 blocks of 32 like a cached row, K and V hold dequantised Q8_0 rows.
 * Score t = (1/sqrt(d)) sum_b d_q[b] d_k[t][b] sum_i q_i k_i over the integer codes, which
 * equals the dot product of the dequantised rows; that form is evaluated in f64, where
 * every product of two dequantised values is exact. */
void or_attention_q8(const double* q, const float* K, const float* V, int T, int d, size_t row_stride,
                     double* o);
/* The values a cache of kv_type holds for a row x of n values (one head's k or v): f32 or
 * bf16 rounding of each value; for Q8_0 each value is rounded to f32 (the precision the
 * quantiser's decisions are taken in), then each block of 32 is quantised (or_quant_q8_0)
 * and dequantised.  n % 32 == 0 for Q8_0. */
void or_kv_round_row(int kv_type, const double* x, int n, float* out);
double or_silu(double z);
void or_router(const double* logits, int n_exp, int k, int norm, int* idx, double* w);
/* y[r] = sum_c W[r,c] x[c] over a packed [rows, cols] matrix (wtype OR_Q8_0/OR_Q4_K/OR_F32) */
void or_gemv(int wtype, const void* W, int rows, int cols, const double* x, double* y);

/* ---- model ---- */
int  or_validate(const or_dims* d);   /* 0 ok, 1 invalid config (section 14.2 validation) */
or_model* or_model_new(const or_dims* d);
void or_model_free(or_model* m);
void or_model_set_global(or_model* m, const void* tok_embd, const float* output_norm, const void* output);
void or_model_set_layer(or_model* m, int layer, const float* attn_norm, const void* wq, const void* wk,
                        const void* wv, const float* q_norm, const float* k_norm, const void* wo,
                        const float* ffn_norm, const void* w_gate, const void* w_up, const void* w_down,
                        const float* router, const void* gate_exps, const void* up_exps,
                        const void* down_exps);

or_cache* or_cache_new(const or_model* m, int capacity);
void or_cache_free(or_cache* c);
int  or_cache_len(const or_cache* c);
/* write n prior positions of one layer (values in the cache dtype, given as f32: bf16
 * caches round them again, Q8_0 caches quantise each row again, which is the identity for
 * dequantised Q8_0 rows); returns 0 or an error code */
int  or_cache_write(or_cache* c, int layer, int pos0, int n, const float* k, const float* v);
int  or_cache_set_len(or_cache* c, int len);
/* keep != 0: later layer steps on this cache attend over the k/v rows already written at the
 * step's position (or_cache_write) instead of storing their own; the step still computes q,
 * k and v.  A test uses it to continue from another implementation's rounded rows. */
int  or_cache_keep_current(or_cache* c, int keep);
/* read back [n][n_kv][head_dim] of one layer */
int  or_cache_read(const or_cache* c, int layer, int pos0, int n, float* k, float* v);

/* status codes mirror the C ABI's contract errors */
enum { OR_OK = 0, OR_INVALID_CONFIG = 1, OR_INVALID_SEQUENCE_LENGTH = 2, OR_KV_CACHE_OVERFLOW = 3,
       OR_MISMATCHED_KV_CACHES = 4, OR_INVALID_ARGUMENT = 5 };

/* One decoder layer for one token at absolute position pos (== cache len for this layer),
 * residual stream x (length hidden) updated in place.  Appends k/v at pos for this layer.
 * route_idx / route_w (may be NULL) receive the MoE selection. */
int or_layer_step(const or_model* m, int layer, or_cache* c, int pos, double* x, int* route_idx,
                  double* route_w);

/* or_layer_step that also writes the MoE router logits (n_exp values, before the softmax) to
 * route_logits (may be NULL). */
int or_layer_step_route(const or_model* m, int layer, or_cache* c, int pos, double* x, int* route_idx,
                        double* route_w, double* route_logits);

/* The attention block's projections for one token of layer `layer` at position pos, from the
 * already normalised input xn (length hidden): q [n_q][head_dim], k and v [n_kv][head_dim],
 * q and k after the per-head RMSNorm with q_norm / k_norm and then RoPE, v as projected. */
int or_qkv_project(const or_model* m, int layer, const double* xn, int pos, double* q, double* k, double* v);

/* forwardStep with one token at pos0 == cache len: embedding, all layers, output norm and
 * LM head into logits (vocab, may be NULL to skip the head).  layer_out (may be NULL)
 * receives the residual stream after every layer, [layers][hidden]; route (may be NULL)
 * the MoE indices [layers][n_used] and weights. Advances len by one. */
int or_decode_step(const or_model* m, or_cache* c, int token, int pos0, double* logits,
                   double* layer_out, int* route_idx, double* route_w);

/* forwardStepBatch: one token per stream, stream s against caches[s]; logits [n][vocab].
 * Validates the caches first (distinct, same model); all advance by one. */
int or_decode_step_batch(const or_model* m, or_cache* const* caches, int n, const int* tokens,
                         double* logits);

/* forwardLastLogits: cacheless causal forward over tokens[0..n), last row's logits */
int or_forward_last_logits(const or_model* m, const int* tokens, int n, double* logits);

/* index of the largest value, ties to the lowest index */
int or_argmax(const double* v, int n);

/* ---- sampling (runner page: --temp, --top-k, --top-p, --min-p, --repeat-penalty, --seed) ---- */
typedef struct or_sampling {
    double temp;            /* 0: greedy argmax */
    int top_k;              /* 0: off */
    double top_p;           /* 1: off */
    double min_p;           /* 0: off */
    double repeat_penalty;  /* 1: off */
} or_sampling;

/* The next token from one row of logits z[n]:
 *   1. repeat penalty over the distinct ids of history[n_hist]: z > 0 is divided by it,
 *      otherwise multiplied;
 *   2. temp == 0: argmax (ties to the lowest id);
 *   3. p = softmax(z / temp); candidates ordered by p descending, ties to the lower id;
 *   4. top_k > 0 keeps the first top_k; top_p < 1 keeps the shortest prefix whose mass
 *      reaches top_p of the kept mass; min_p > 0 drops p < min_p * (largest p); at least one
 *      candidate always stays;
 *   5. with Z the kept mass, the first candidate whose cumulative mass exceeds u * Z
 *      (u in [0, 1)). */
int or_sample(const double* z, int n, const or_sampling* s, const int* history, int n_hist, double u);

/* Counter-based uniform in [0, 1) on a 2^-24 grid (exact in f32): the top 24 bits of the
 * SplitMix64 output for state seed + (counter + 1) * 0x9E3779B97F4A7C15 (Steele, Lea and
 * Flood, "Fast splittable pseudorandom number generators", 2014). */
double or_uniform24(uint64_t seed, uint64_t counter);

#ifdef __cplusplus
}
#endif
#endif
