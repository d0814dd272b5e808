// Device data layouts and kernel launchers of the fq decode path.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#ifdef __CUDACC__
#define FQ_HD __host__ __device__
#else
#define FQ_HD
#endif

namespace fq {

constexpr int HEAD_DIM = 128;      // the only head_dim the kernels are built for
constexpr int MAX_TOPK = 8;
constexpr int MAX_EXPERTS = 256;

enum Fmt : int { FMT_F32 = 0, FMT_BF16 = 1, FMT_Q8_0 = 8, FMT_Q4_K = 12 };

// Tensor maps (TMA descriptors) of one weight's planes, built at load time; opaque bytes
// of CUtensorMap.  ok == 0 when the shape is not served by the bulk-copy GEMV.
struct TmaMaps {
    alignas(64) unsigned long long q[16];
    alignas(64) unsigned long long s[16];
    alignas(64) unsigned long long tcq[16];   // Q8_0 codes for the tensor-core GEMM
    int ok = 0;
    int tc_ok = 0;
};

// One device-resident weight matrix [N rows, K cols].
//   Q8_0: repacked into two 16-byte-aligned planes, q int8 [N][K] and s fp16 [N][K/32]
//         (the same bytes as the ggml blocks, split so that 16-byte loads line up);
//   Q4_K: ggml super-blocks as stored, [N][K/256 * 144] bytes (already 16-byte aligned);
//   F32 : plain row-major floats in q.
struct QMat {
    int fmt = FMT_F32;
    int N = 0, K = 0;
    const uint8_t* q = nullptr;
    const uint16_t* s = nullptr;
    const TmaMaps* tm = nullptr;   // host pointer (model-owned); never read on the device
    FQ_HD size_t row_bytes() const {
        return fmt == FMT_Q8_0 ? (size_t)K : fmt == FMT_Q4_K ? (size_t)K / 256 * 144 : (size_t)K * 4;
    }
    FQ_HD size_t bytes() const {   // algorithmic bytes of the whole matrix (ggml-equivalent size)
        return fmt == FMT_Q8_0 ? (size_t)N * K / 32 * 34 : (size_t)N * row_bytes();
    }
};

// Per-sequence state of one step, resident in the per-stream workspace.  Written by the
// set-up kernel before a step (or a chain of greedy steps); read by every kernel, so a
// captured graph is independent of the token, the positions and the cache pointers.
// What a KvCache stores per row: f32 or bf16 values, or Q8_0 (int8 codes and a plane of
// fp16 block scales).
enum KvType : int { KV_F32 = 0, KV_BF16 = 1, KV_Q8_0 = 2 };

struct SeqState {
    int32_t token;        // token consumed by this step's embedding
    int32_t pos;          // absolute position of the new token (== cache len)
    int32_t cap;          // cache capacity
    int32_t pad;
    void* k;              // cache planes, [layer][kv_head][cap][head_dim]
    void* v;
    void* ks;             // Q8_0 scale planes, [layer][kv_head][cap rounded up to even][4] fp16
    void* vs;
};

constexpr int MAX_SEQ = 64;

struct StepState {
    SeqState seq[MAX_SEQ];
    unsigned long long keys[MAX_SEQ];   // argmax keys of the current step
    int32_t step;                       // greedy step counter
    uint32_t lm_counter;                // CTAs of the LM head that finished
    int32_t* tokens_out;                // greedy output [n_steps][n] or null
    float* logits;                      // [n][vocab] or null
    int32_t greedy;                     // feed argmax back and advance positions
    int32_t n;
};

// GEMV / small-batch GEMM on CUDA cores:  y[b][r] (op)= sum_k W[r][k] * xin[b][k]
enum Epi : int { EPI_STORE = 0, EPI_ADD = 1, EPI_SWIGLU = 2, EPI_LOGITS = 3 };

struct GemvArgs {
    QMat W;
    int B = 1;                    // activation rows
    const float* x = nullptr;     // input [B][x_stride]
    int x_stride = 0;
    const float* norm_g = nullptr;// RMSNorm prologue gain (null: input used as is)
    float eps = 1e-6f;
    float* y = nullptr;           // output [B][y_stride]
    int y_stride = 0;
    int epi = EPI_STORE;          // SWIGLU: rows interleaved (2i gate, 2i+1 up) -> y[b][i]
    int ksplit = 1;               // warps of a row group splitting K (1, 2, 4, 8)
    StepState* st = nullptr;      // EPI_LOGITS: argmax keys and the greedy hand-off
    float* xn_out = nullptr;      // optional: CTA 0 stores the normalised input [B][K]
    int xn_stride = 0;
    // expert mode (MoE): blockIdx.y = active expert slot of `route`; W holds every expert's
    // rows_per_expert rows; activation rows are that expert's (token, slot) pairs
    const struct MoeRoute* route = nullptr;
    int moe_k = 0;
    int rows_per_expert = 0;
    int x_by_pair = 0;            // input row = token*moe_k + slot (else token)
    int max_experts = 0;          // grid.y
    uint32_t* err = nullptr;      // device error word: bit set when a bounded wait gave up
    int starve = 0;               // bulk-copy GEMV only: the producer issues no copies (the
                                  // consumers' bounded waits run out; used to test the timeout)
};

void launch_gemv(const GemvArgs& a, cudaStream_t s, bool pdl);
// one-time kernel attributes (large dynamic shared memory); call before any graph capture
void gemv_prepare();
// the bulk-copy fed variant; returns false when the shape is not covered (caller falls back)
bool launch_gemv_tma(const GemvArgs& a, cudaStream_t s, bool pdl);
void gemv_tma_prepare();
// build the tensor maps of W's planes for the bulk-copy GEMV and the tensor-core GEMM
// (false: the GEMV maps are not applicable; tc_ok tells about the GEMM's)
bool make_tma_maps(const QMat& W, TmaMaps* out);
// tensor map over f16 rows [rows][K], box 64 halves x box_rows, 128-byte swizzle
bool encode_f16_rows_sw128(void* map, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows);

// tcgen05 GEMM for lockstep batches of TC_MIN_BATCH..32 rows over Q8_0 weights: a prep
// kernel (RMSNorm + f16 hi/lo split into xh, 64 x K halves) and the GEMM
constexpr int TC_MIN_BATCH = 8;
void gemm_tc_prepare();
bool gemm_tc_applicable(const GemvArgs& a);
size_t gemm_tc_xh_elems(int K);
// part: split-K scratch of part_cap floats; tickets: TC_TICKETS zeroed counters
void launch_gemm_tc(const GemvArgs& a, void* xh, float* part, size_t part_cap, uint32_t* tickets, cudaStream_t s,
                    bool pdl_prep, bool pdl);
constexpr size_t TC_PART_FLOATS = (size_t)4 << 20;
constexpr int TC_TICKETS = 8192;

// Attention with fused QK-norm + rope + KV append (one query row per sequence).
struct AttnArgs {
    const float* qkv;             // [n][(Hq + 2 Hkv) * 128] raw projections
    int qkv_stride;
    const float* q_norm;          // [128]
    const float* k_norm;          // [128]
    const float2* rope;           // [max_pos][64] (cos, sin)
    float eps;
    int Hq, Hkv;
    int layer;
    int kv_type;                  // KvType of the caches
    int chunk;                    // positions per CTA (multiple of 32)
    int splits;                   // grid.x
    const StepState* st;
    float* part;                  // [n][Hq][splits][130] partial (m, l, o[128])
    uint32_t* counters;           // [n][Hq]: arrivals per (row, CTA group of query heads)
    float* out;                   // [n][Hq * 128]
    int n;
    uint32_t* err = nullptr;      // device error word (a staged copy that never landed)
    int append_only = 0;          // 1: only write the new k/v of each row, no attention
    int kv_store = 1;             // 0: the new k/v are already in the cache (kept, not stored)
};

void launch_attention(const AttnArgs& a, cudaStream_t s, bool pdl);
// one-time kernel attributes of the attention kernels; call before any graph capture
void attention_prepare();

// The whole batch-1 step of a dense model as one persistent kernel whose producer warps
// stream the step's weights and cached K/V ahead of the activations (stream_step.cu).
struct StreamLayer {
    QMat qkv, o, gate_up, down;
    const float *attn_norm, *ffn_norm, *q_norm, *k_norm;
};
// One CTA's share of one projection (every layer has the same shapes): rows [r0, r1), rows
// per ring item, and the K split of its tasks (kparts parts of `up` units of U per row).
struct ProjPlan {
    int r0, r1, rs, kparts, up, U;
};
enum { P_QKV = 0, P_O = 1, P_GU = 2, P_DN = 3, P_LM = 4, NPROJ = 5 };
struct StreamArgs {
    const StreamLayer* layers;    // device array [n_layers]
    int n_layers = 0, H = 0, F = 0, Hq = 0, Hkv = 0, V = 0;
    float eps = 1e-6f;
    QMat emb, out;
    const float* out_norm = nullptr;
    const float2* rope = nullptr;
    StepState* st = nullptr;
    // exchange words between CTAs (value bits | tag << 32): layer output, attention-block
    // output, raw QKV, attention partials [Hq][S][130], merged attention, SwiGLU activations
    unsigned long long *xf = nullptr, *xa = nullptr, *qkv = nullptr, *part = nullptr, *o = nullptr, *h = nullptr;
    float* logits = nullptr;      // LM-head output [V] or null
    float* trace_x = nullptr;     // optional: the residual stream after every layer [n_layers][H]
    int head = 0;                 // run the LM head
    int greedy = 0;               // argmax hand-off after the LM head
    uint32_t* ctl = nullptr;      // [0] finishing ticket (zero between launches), [1] launch sequence
    uint32_t* err = nullptr;
    int S = 0;                    // attention chunks per kv head
    int max_pos = 0;              // cache capacity the plan covers (positions)
    int score_cap = 0;            // attention scores per head the shared memory holds
    const ProjPlan* plan = nullptr;   // device [CTAs][NPROJ]
    // shared-memory plan (stream_plan)
    int nslot = 0, kmax = 0, lay_xs = 0, lay_xq = 0, lay_xr = 0, lay_red = 0, lay_bars = 0, smem_bytes = 0;
};
void stream_prepare();
int stream_ctas();
int stream_chunks(int Hkv);       // S for a model with Hkv kv heads
// fills the shared-memory plan and the per-CTA projection plans (host [CTAs][NPROJ]);
// false when the shapes do not fit
bool stream_plan(StreamArgs& a, const StreamLayer& l0, int fmt, int G, std::vector<ProjPlan>& plans);
bool launch_stream(const StreamArgs& a, int fmt, int G, cudaStream_t s);

// Embedding rows -> x [n][H]
void launch_embed(const QMat& emb, const StepState* st, int n, float* x, cudaStream_t s, bool pdl);

// Write the step state (tokens, positions, caches) before a step or a greedy chain.
struct SetupArgs {
    int n;
    int greedy;
    int32_t* tokens_out;
    float* logits;
    int32_t token[MAX_SEQ];
    int32_t pos[MAX_SEQ];
    int32_t cap[MAX_SEQ];
    void* k[MAX_SEQ];
    void* v[MAX_SEQ];
    void* ks[MAX_SEQ];
    void* vs[MAX_SEQ];
};
void launch_setup(StepState* st, const SetupArgs& a, cudaStream_t s);

// Q8_0 cache rows <-> ggml blocks: blocks [n_pos][Hkv][4][34 bytes]; codes / scales point at
// row 0 of kv head 0 of one layer, with per-head strides of cap and cap_s rows.
void launch_kv_q8_copy(int8_t* codes, uint16_t* scales, size_t cap, size_t cap_s, int Hkv, int pos, int n_pos,
                       uint8_t* blocks, bool to_cache, cudaStream_t s);
// ggml Q8_0 blocks of x[0, n) (n a multiple of 128) with the attention kernel's quantiser
void launch_quantize_q8_0(const float* x, size_t n, uint8_t* blocks, cudaStream_t s);

// LM-head finisher: decode argmax keys, hand the token to the next step.
void launch_lm_finish(StepState* st, int n, int vocab, cudaStream_t s, bool pdl);

// MoE: router logits + softmax top-k + grouping of (token, slot) pairs by expert.
struct MoeRoute {
    int32_t n_active;                     // distinct experts in use
    int32_t expert[256];                  // active expert ids, ascending
    int32_t start[257];                   // pair ranges per active expert
    int32_t pair_token[MAX_SEQ * 8];      // grouped pairs: token index
    int32_t pair_slot[MAX_SEQ * 8];       //                slot j of that token
    int32_t idx[MAX_SEQ * 8];             // [n][k] chosen experts
    float w[MAX_SEQ * 8];                 // [n][k] weights
};
// softmax top-k over router logits [n][E] and the grouping of pairs by expert (one CTA)
void launch_moe_route(const float* logits, int E, int k, int n, int norm_topk, MoeRoute* route, cudaStream_t s,
                      bool pdl);
// x[b] += sum_j w[b][j] * y[b*k + j]
void launch_moe_combine(float* x, const float* y, const MoeRoute* route, int n, int k, int H, cudaStream_t s,
                        bool pdl);

// Load-time helpers
// Source row r lands in destination row (r / group) * group_stride + (r % group) * step + off
// (fusing q/k/v, interleaving gate/up rows, stacking experts).
void launch_repack_q8_0(const uint8_t* ggml, int64_t rows, int64_t cols, uint8_t* q, uint16_t* sc, int64_t group,
                        int64_t group_stride, int64_t step, int64_t off, cudaStream_t s);
void launch_copy_rows(const uint8_t* src, int64_t rows, int64_t row_bytes, uint8_t* dst, int64_t group,
                      int64_t group_stride, int64_t step, int64_t off, cudaStream_t s);
void launch_rope_table(float2* tab, int max_pos, double theta, cudaStream_t s);
void launch_dequant(const QMat& W, int64_t row0, int64_t n_rows, float* out, cudaStream_t s);

}  // namespace fq
