// Host side of the fq C ABI: descriptor validation, weight upload and repacking, KV
// caches, per-stream workspaces, and the decode-step orchestration (a fixed kernel
// sequence per step, launched with programmatic dependent launch and captured once into
// a CUDA graph that replays for every step of the same shape).

#include <cuda_runtime.h>

#include <algorithm>
#include <deque>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "fq.h"
#include "kernels.h"

using namespace fq;

namespace {

thread_local std::string g_err;
constexpr uint32_t DESC_MAGIC = 0x51574633u;   // "QWF3"

fq_status fail(fq_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

#define CK(call)                                                                                       \
    do {                                                                                               \
        cudaError_t e_ = (call);                                                                       \
        if (e_ != cudaSuccess)                                                                         \
            return fail(e_ == cudaErrorMemoryAllocation ? FQ_ERR_OUT_OF_MEMORY : FQ_ERR_CUDA, "%s: %s", \
                        #call, cudaGetErrorString(e_));                                                \
    } while (0)

#define TRY(call)                  \
    do {                           \
        fq_status s_ = (call);     \
        if (s_ != FQ_OK) return s_; \
    } while (0)

}  // namespace

// ---------------------------------------------------------------- model and cache objects

struct LayerW {
    const float *attn_norm = nullptr, *ffn_norm = nullptr, *q_norm = nullptr, *k_norm = nullptr;
    QMat qkv, o, gate_up, down;            // dense FFN: gate_up rows interleaved (2i gate, 2i+1 up)
    QMat router, gate_up_exps, down_exps;  // MoE: expert e owns rows [e*2Fe, (e+1)*2Fe) / [e*H, (e+1)*H)
};

struct Workspace;

struct fq_model {
    fq_desc d;
    int device = 0;
    QMat tok_embd, output;
    const float* output_norm = nullptr;
    std::vector<LayerW> layers;
    float2* rope = nullptr;
    int max_pos = 0;
    uint32_t* err = nullptr;       // device error word (bounded waits that gave up)
    std::deque<TmaMaps> tmaps;     // tensor maps of the dense weights (stable addresses)
    StreamLayer* slayers = nullptr;    // device layer table of the streamed batch-1 step (null: not served)
    StreamArgs splan;                  // its shapes and shared-memory plan
    int sfmt = 0, sG = 0;
    // options (fq_set_option)
    int opt_path = FQ_PATH_AUTO;
    int opt_pdl = 0;
    int opt_graphs = 1;
    int opt_tc = 1;
    std::vector<void*> allocs;
    std::mutex ws_mu;
    std::map<cudaStream_t, Workspace*> ws;
    int qkv_rows() const { return (d.p.num_attention_heads + 2 * d.p.num_key_value_heads) * d.p.head_dim; }
    bool moe() const { return d.p.num_experts > 0; }
};

struct fq_kv {
    const fq_model* m = nullptr;
    uint32_t cap = 0, len = 0;
    int type = KV_BF16;            // KvType
    void* k = nullptr;             // [layer][kv head][cap][128] values or Q8_0 codes
    void* v = nullptr;
    void* ks = nullptr;            // Q8_0: [layer][kv head][cap_s()][4] fp16 scales, inside the k
    void* vs = nullptr;            //   and v allocations after the codes
    size_t elem() const { return type == KV_F32 ? 4 : type == KV_BF16 ? 2 : 1; }
    size_t cap_s() const { return (cap + 1) & ~1u; }   // even, so scale rows pair into 16 bytes
};

// Per-stream scratch and captured graphs (the pages' ExecContext: one per concurrent stream).
struct Workspace {
    int n_cap = 0;             // batch rows the buffers hold
    size_t part_cap = 0;       // floats in `part`
    StepState* st = nullptr;
    float *x = nullptr, *qkv = nullptr, *attn = nullptr, *h = nullptr, *part = nullptr, *logits = nullptr;
    float *xn = nullptr, *rlogits = nullptr, *he = nullptr, *ye = nullptr;
    void* xh = nullptr;        // f16 hi/lo activations for the tensor-core GEMM (batches >= 8)
    float* tc_part = nullptr;  // its split-K partial sums
    uint32_t* tc_tickets = nullptr;
    uint32_t* counters = nullptr;
    unsigned long long* sx = nullptr;   // streamed step: exchange words (see StreamArgs)
    uint32_t* sctl = nullptr;           //                finishing ticket + launch sequence
    MoeRoute* route = nullptr;
    std::vector<void*> allocs;
    struct Graph {
        int mode, n, chunk, splits, kv_type;
        float* logits;
        cudaGraphExec_t exec;
        uint32_t kernels;      // kernel nodes in the captured step
    };
    std::vector<Graph> graphs;
    uint32_t last_kernels = 0; // kernels of the step most recently replayed on this stream
    void drop_graphs() {
        for (auto& g : graphs) cudaGraphExecDestroy(g.exec);
        graphs.clear();
    }
    void release() {
        drop_graphs();
        for (void* p : allocs) cudaFree(p);
        allocs.clear();
    }
};

namespace {

template <class T>
fq_status dalloc(std::vector<void*>& owner, T** p, size_t count) {
    void* q = nullptr;
    if (count == 0) count = 1;
    cudaError_t e = cudaMalloc(&q, count * sizeof(T));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(FQ_ERR_OUT_OF_MEMORY, "cudaMalloc(%zu bytes): %s", count * sizeof(T), cudaGetErrorString(e));
    }
    owner.push_back(q);
    *p = (T*)q;
    return FQ_OK;
}

// attention split: chunks of 128 positions (one 32-position tile per warp) or a multiple,
// enough CTAs to cover the GPU at small batch, at most 4 tiles per warp for balance
void attn_split(int n, int Hkv, uint32_t cap_max, int& chunk, int& splits) {
    int target = std::max(1, 304 / std::max(1, n * Hkv));
    int m = (int)((cap_max + 128u * target - 1) / (128u * target));
    m = std::max(1, std::min(m, 4));
    chunk = 128 * m;
    splits = (int)((cap_max + chunk - 1) / chunk);
}

int choose_ksplit(const QMat& W, int R) {
    int units = W.K / (W.fmt == FMT_Q4_K ? 32 : W.fmt == FMT_Q8_0 ? 16 : 4);
    int ks = 1;
    while (ks < 8) {
        int rows_per_cta = (8 / ks) * R;
        int ctas = (W.N + rows_per_cta - 1) / rows_per_cta;
        if (ctas >= 256) break;
        if (units / (2 * ks) < 32) break;
        ks *= 2;
    }
    return ks;
}

int rows_per_warp(const QMat& W) { return W.fmt == FMT_Q4_K ? 2 : 4; }

// exchange words of the streamed step: xf, xa [H], qkv, part [Hq][S][130], o [Hq*128], h [F]
size_t stream_words(const fq_model* m) {
    const auto& p = m->d.p;
    return 2 * (size_t)p.hidden_size + (size_t)m->qkv_rows() +
           (size_t)p.num_attention_heads * m->splan.S * (HEAD_DIM + 2) + (size_t)p.num_attention_heads * HEAD_DIM +
           (size_t)p.intermediate_size;
}

fq_status ensure_ws(const fq_model* mc, cudaStream_t stream, int n, uint32_t cap_max, Workspace** out) {
    fq_model* m = const_cast<fq_model*>(mc);
    std::lock_guard<std::mutex> lk(m->ws_mu);
    Workspace*& w = m->ws[stream];
    if (!w) w = new Workspace();
    const auto& p = m->d.p;
    int chunk, splits;
    attn_split(n, p.num_key_value_heads, cap_max, chunk, splits);
    size_t part_need = (size_t)n * p.num_attention_heads * splits * (HEAD_DIM + 2);
    if (w->n_cap < n || w->part_cap < part_need) {
        int nn = std::max(n, w->n_cap);
        size_t pc = std::max(part_need, w->part_cap);
        // graphs hold the old pointers: wait for the stream, then rebuild everything
        cudaStreamSynchronize(stream);
        w->release();
        w->n_cap = 0;
        w->part_cap = 0;
        auto& A = w->allocs;
        const size_t H = p.hidden_size;
        TRY(dalloc(A, &w->st, 1));
        TRY(dalloc(A, &w->x, nn * H));
        TRY(dalloc(A, &w->qkv, (size_t)nn * m->qkv_rows()));
        TRY(dalloc(A, &w->attn, (size_t)nn * p.num_attention_heads * HEAD_DIM));
        TRY(dalloc(A, &w->h, (size_t)nn * std::max<size_t>(p.intermediate_size, 1)));
        TRY(dalloc(A, &w->part, pc));
        TRY(dalloc(A, &w->counters, (size_t)nn * p.num_attention_heads));   // one per (row, CTA head group) at most
        TRY(dalloc(A, &w->logits, (size_t)nn * p.vocab_size));
        CK(cudaMemsetAsync(w->counters, 0, sizeof(uint32_t) * nn * p.num_attention_heads, stream));
        if (m->slayers) {
            const size_t words = stream_words(m);
            TRY(dalloc(A, &w->sx, words));
            TRY(dalloc(A, &w->sctl, 4));
            CK(cudaMemsetAsync(w->sx, 0, sizeof(unsigned long long) * words, stream));
            CK(cudaMemsetAsync(w->sctl, 0, sizeof(uint32_t) * 4, stream));
        }
        if (nn >= TC_MIN_BATCH) {
            const int kmax = (int)std::max<size_t>({H, (size_t)p.num_attention_heads * HEAD_DIM,
                                                     (size_t)std::max<uint32_t>(p.intermediate_size, 1)});
            uint16_t* xh;
            TRY(dalloc(A, &xh, gemm_tc_xh_elems(kmax)));
            w->xh = xh;
            TRY(dalloc(A, &w->tc_part, TC_PART_FLOATS));
            TRY(dalloc(A, &w->tc_tickets, (size_t)TC_TICKETS));
            CK(cudaMemsetAsync(w->tc_tickets, 0, sizeof(uint32_t) * TC_TICKETS, stream));
        }
        CK(cudaMemsetAsync(w->st, 0, sizeof(StepState), stream));
        if (m->moe()) {
            size_t k = p.num_experts_used;
            TRY(dalloc(A, &w->xn, nn * H));
            TRY(dalloc(A, &w->rlogits, (size_t)nn * p.num_experts));
            TRY(dalloc(A, &w->he, nn * k * p.moe_intermediate_size));
            TRY(dalloc(A, &w->ye, nn * k * H));
            TRY(dalloc(A, &w->route, 1));
            CK(cudaMemsetAsync(w->route, 0, sizeof(MoeRoute), stream));
        }
        w->n_cap = nn;
        w->part_cap = pc;
    }
    *out = w;
    return FQ_OK;
}

// Zero the counters and tickets that the kernels of a step leave at zero when they finish
// normally (attention arrivals, tensor-core split-K tickets, the streamed step's ticket).
fq_status rearm_ws(const fq_model* m, Workspace* w, cudaStream_t s) {
    const auto& p = m->d.p;
    if (w->counters) CK(cudaMemsetAsync(w->counters, 0, sizeof(uint32_t) * w->n_cap * p.num_attention_heads, s));
    if (w->sctl) CK(cudaMemsetAsync(w->sctl, 0, sizeof(uint32_t), s));   // the ticket; the sequence may stay
    if (w->tc_tickets) CK(cudaMemsetAsync(w->tc_tickets, 0, sizeof(uint32_t) * TC_TICKETS, s));
    if (w->route) CK(cudaMemsetAsync(w->route, 0, sizeof(MoeRoute), s));
    return FQ_OK;
}

enum Mode { MODE_DECODE = 1, MODE_GREEDY = 2 };

struct Body {
    const fq_model* m;
    Workspace* w;
    int n;
    int chunk, splits;
    float* logits;          // LM-head output or null (no head)
    bool greedy;
    // trace (direct launches only)
    float* layer_out = nullptr;
    int32_t* route_idx = nullptr;
    float* route_w = nullptr;
    float* route_logits = nullptr;
    // rows are consecutive positions of one sequence (the all-logits step): every row's new
    // k/v is appended before any row attends
    bool block = false;
    // LM head on this row only (its logits go to `logits` as one row); -1: every row
    int head_row = -1;
};

// Batch 1 of a dense model with a bf16 cache runs as one streamed persistent kernel
// (stream_step.cu) unless the caller asked for the kernel sequence.
bool stream_eligible(const Body& b, int kv_type) {
    const fq_model* m = b.m;
    return m->slayers && m->opt_path != FQ_PATH_KERNELS && b.n == 1 && !b.route_idx && !b.route_logits && !b.block &&
           b.head_row < 0 && kv_type == KV_BF16;
}

// The kernels of one decode step, in order.  The first launch follows the set-up kernel
// with ordinary stream order; every later one uses programmatic dependent launch.
fq_status enqueue_step(const Body& b, cudaStream_t s, int kv_type, float* x_override, int layer_only) {
    const fq_model* m = b.m;
    Workspace* w = b.w;
    const auto& p = m->d.p;
    const int n = b.n, H = p.hidden_size, Hq = p.num_attention_heads, Hkv = p.num_key_value_heads;
    bool first = true;
    // Programmatic dependent launch is an option (off by default: measured on GB300 the
    // early-resident CTAs of the next kernel slowed the step down)
    const bool use_pdl = m->opt_pdl != 0;
    const bool no_tc = m->opt_tc == 0;
    auto pdl = [&]() { bool r = !first && use_pdl; first = false; return r; };
    // dense projection: tensor cores for lockstep batches, the GEMV kernels otherwise
    auto proj = [&](GemvArgs& g) {
        g.err = m->err;
        if (!no_tc && w->xh && gemm_tc_applicable(g)) {
            const bool p0 = pdl();
            launch_gemm_tc(g, w->xh, w->tc_part, TC_PART_FLOATS, w->tc_tickets, s, p0, use_pdl);
        } else {
            launch_gemv(g, s, pdl());
        }
    };
    float* x = x_override ? x_override : w->x;

    // batch 1 of a dense model: the whole step as one streamed persistent kernel
    if (layer_only < 0 && stream_eligible(b, kv_type)) {
        StreamArgs sa = m->splan;
        unsigned long long* q = w->sx;
        sa.xf = q; q += H;
        sa.xa = q; q += H;
        sa.qkv = q; q += m->qkv_rows();
        sa.part = q; q += (size_t)Hq * sa.S * (HEAD_DIM + 2);
        sa.o = q; q += (size_t)Hq * HEAD_DIM;
        sa.h = q;
        sa.st = w->st;
        sa.logits = b.logits;
        sa.trace_x = b.layer_out;
        sa.head = (b.logits || b.greedy) ? 1 : 0;
        sa.greedy = b.greedy ? 1 : 0;
        sa.ctl = w->sctl;
        sa.err = m->err;
        if (!launch_stream(sa, m->sfmt, m->sG, s)) {
            cudaGetLastError();
            return fail(FQ_ERR_CUDA, "streamed step launch refused");
        }
        CK(cudaGetLastError());
        return FQ_OK;
    }

    if (layer_only < 0) launch_embed(m->tok_embd, w->st, n, x, s, pdl());
    int L0 = layer_only < 0 ? 0 : layer_only, L1 = layer_only < 0 ? (int)p.num_layers : layer_only + 1;
    for (int L = L0; L < L1; ++L) {
        const LayerW& lw = m->layers[L];
        GemvArgs g;
        g.W = lw.qkv; g.B = n; g.x = x; g.x_stride = H; g.norm_g = lw.attn_norm; g.eps = p.rms_norm_eps;
        g.y = w->qkv; g.y_stride = m->qkv_rows(); g.epi = EPI_STORE;
        g.ksplit = choose_ksplit(g.W, rows_per_warp(g.W));
        proj(g);

        AttnArgs a;
        a.qkv = w->qkv; a.qkv_stride = m->qkv_rows(); a.q_norm = lw.q_norm; a.k_norm = lw.k_norm;
        a.rope = m->rope; a.eps = p.rms_norm_eps; a.Hq = Hq; a.Hkv = Hkv; a.layer = L; a.kv_type = kv_type;
        a.chunk = b.chunk; a.splits = b.splits; a.st = w->st; a.part = w->part; a.counters = w->counters;
        a.out = w->attn; a.n = n; a.err = m->err;
        if (b.block) {
            AttnArgs ap = a;
            ap.append_only = 1;
            launch_attention(ap, s, pdl());
            a.kv_store = 0;
        }
        launch_attention(a, s, pdl());

        GemvArgs o;
        o.W = lw.o; o.B = n; o.x = w->attn; o.x_stride = Hq * HEAD_DIM; o.y = x; o.y_stride = H; o.epi = EPI_ADD;
        o.ksplit = choose_ksplit(o.W, rows_per_warp(o.W));
        proj(o);

        if (!m->moe()) {
            GemvArgs gu;
            gu.W = lw.gate_up; gu.B = n; gu.x = x; gu.x_stride = H; gu.norm_g = lw.ffn_norm; gu.eps = p.rms_norm_eps;
            gu.y = w->h; gu.y_stride = p.intermediate_size; gu.epi = EPI_SWIGLU;
            gu.ksplit = choose_ksplit(gu.W, rows_per_warp(gu.W));
            proj(gu);

            GemvArgs dn;
            dn.W = lw.down; dn.B = n; dn.x = w->h; dn.x_stride = p.intermediate_size; dn.y = x; dn.y_stride = H;
            dn.epi = EPI_ADD; dn.ksplit = choose_ksplit(dn.W, rows_per_warp(dn.W));
            proj(dn);
        } else {
            const int E = p.num_experts, k = p.num_experts_used, Fe = p.moe_intermediate_size;
            GemvArgs r;
            r.W = lw.router; r.B = n; r.x = x; r.x_stride = H; r.norm_g = lw.ffn_norm; r.eps = p.rms_norm_eps;
            r.y = w->rlogits; r.y_stride = E; r.epi = EPI_STORE; r.xn_out = w->xn; r.xn_stride = H;
            r.ksplit = choose_ksplit(r.W, 4);
            r.err = m->err;
            launch_gemv(r, s, pdl());
            launch_moe_route(w->rlogits, E, k, n, p.norm_topk_prob, w->route, s, pdl());

            GemvArgs eg;
            eg.W = lw.gate_up_exps; eg.x = w->xn; eg.x_stride = H; eg.y = w->he; eg.y_stride = Fe;
            eg.epi = EPI_SWIGLU; eg.route = w->route; eg.moe_k = k; eg.rows_per_expert = 2 * Fe; eg.x_by_pair = 0;
            eg.max_experts = std::min(E, n * k);
            eg.ksplit = 1;
            eg.err = m->err;
            launch_gemv(eg, s, pdl());

            GemvArgs ed;
            ed.W = lw.down_exps; ed.x = w->he; ed.x_stride = Fe; ed.y = w->ye; ed.y_stride = H; ed.epi = EPI_STORE;
            ed.route = w->route; ed.moe_k = k; ed.rows_per_expert = H; ed.x_by_pair = 1;
            ed.max_experts = std::min(E, n * k);
            ed.ksplit = 2;
            ed.err = m->err;
            launch_gemv(ed, s, pdl());
            launch_moe_combine(x, w->ye, w->route, n, k, H, s, pdl());

            if (b.route_idx) {
                CK(cudaMemcpyAsync(b.route_idx + (size_t)L * n * k, w->route->idx, sizeof(int32_t) * n * k,
                                   cudaMemcpyDeviceToDevice, s));
                CK(cudaMemcpyAsync(b.route_w + (size_t)L * n * k, w->route->w, sizeof(float) * n * k,
                                   cudaMemcpyDeviceToDevice, s));
                first = true;
            }
            if (b.route_logits) {
                CK(cudaMemcpyAsync(b.route_logits + (size_t)L * n * E, w->rlogits, sizeof(float) * n * E,
                                   cudaMemcpyDeviceToDevice, s));
                first = true;
            }
        }
        if (b.layer_out) {
            CK(cudaMemcpyAsync(b.layer_out + (size_t)L * n * H, x, sizeof(float) * n * H, cudaMemcpyDeviceToDevice, s));
            first = true;
        }
    }
    if (b.logits) {
        GemvArgs lm;
        const bool one = b.head_row >= 0;
        lm.W = m->output; lm.B = one ? 1 : n; lm.x = one ? x + (size_t)b.head_row * H : x; lm.x_stride = H;
        lm.norm_g = m->output_norm; lm.eps = p.rms_norm_eps;
        lm.y = b.logits; lm.y_stride = p.vocab_size; lm.epi = b.greedy ? EPI_LOGITS : EPI_STORE; lm.st = w->st;
        lm.ksplit = choose_ksplit(lm.W, rows_per_warp(lm.W));
        proj(lm);
        if (b.greedy) launch_lm_finish(w->st, n, (int)p.vocab_size, s, pdl());
    }
    CK(cudaGetLastError());
    return FQ_OK;
}

// pos_step = 1: row b sits at position len + b (consecutive positions of one sequence)
fq_status setup_state(Workspace* w, fq_kv* const* caches, const int32_t* tokens, int n, bool greedy,
                      int32_t* tokens_out, float* logits, cudaStream_t s, int pos_step = 0) {
    SetupArgs a;
    memset(&a, 0, sizeof a);
    a.n = n;
    a.greedy = greedy ? 1 : 0;
    a.tokens_out = tokens_out;
    a.logits = logits;
    for (int b = 0; b < n; ++b) {
        a.token[b] = tokens ? tokens[b] : 0;
        a.pos[b] = (int32_t)caches[b]->len + b * pos_step;
        a.cap[b] = (int32_t)caches[b]->cap;
        a.k[b] = caches[b]->k;
        a.v[b] = caches[b]->v;
        a.ks[b] = caches[b]->ks;
        a.vs[b] = caches[b]->vs;
    }
    launch_setup(w->st, a, s);
    CK(cudaGetLastError());
    return FQ_OK;
}

// Run (capture once, replay) the step body for `reps` consecutive steps.
fq_status run_body(const Body& b, cudaStream_t s, int kv_type, int reps) {
    Workspace* w = b.w;
    const int mode = b.greedy ? MODE_GREEDY : MODE_DECODE;
    // one streamed kernel per step needs no graph
    if (!b.m->opt_graphs || b.layer_out || b.route_idx || b.route_logits || stream_eligible(b, kv_type)) {
        for (int r = 0; r < reps; ++r) TRY(enqueue_step(b, s, kv_type, nullptr, -1));
        w->last_kernels = stream_eligible(b, kv_type) ? 1u : 0u;
        return FQ_OK;
    }
    cudaGraphExec_t exec = nullptr;
    for (auto& g : w->graphs)
        if (g.mode == mode && g.n == b.n && g.chunk == b.chunk && g.splits == b.splits && g.kv_type == kv_type &&
            g.logits == b.logits) {
            exec = g.exec;
            w->last_kernels = g.kernels;
        }
    if (!exec) {
        cudaStream_t cs;
        CK(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
        cudaGraph_t graph;
        cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) {
            cudaStreamDestroy(cs);
            return fail(FQ_ERR_CUDA, "cudaStreamBeginCapture: %s", cudaGetErrorString(e));
        }
        fq_status st = enqueue_step(b, cs, kv_type, nullptr, -1);
        e = cudaStreamEndCapture(cs, &graph);
        cudaStreamDestroy(cs);
        if (st != FQ_OK) return st;
        if (e != cudaSuccess) return fail(FQ_ERR_CUDA, "cudaStreamEndCapture: %s", cudaGetErrorString(e));
        uint32_t kernels = 0;
        size_t n_nodes = 0;
        if (cudaGraphGetNodes(graph, nullptr, &n_nodes) == cudaSuccess && n_nodes) {
            std::vector<cudaGraphNode_t> nodes(n_nodes);
            if (cudaGraphGetNodes(graph, nodes.data(), &n_nodes) == cudaSuccess)
                for (auto nd : nodes) {
                    cudaGraphNodeType t;
                    if (cudaGraphNodeGetType(nd, &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++kernels;
                }
        }
        e = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return fail(FQ_ERR_CUDA, "cudaGraphInstantiate: %s", cudaGetErrorString(e));
        w->graphs.push_back({mode, b.n, b.chunk, b.splits, kv_type, b.logits, exec, kernels});
        w->last_kernels = kernels;
    }
    for (int r = 0; r < reps; ++r) CK(cudaGraphLaunch(exec, s));
    return FQ_OK;
}

fq_status check_caches(const fq_model* m, fq_kv* const* caches, uint32_t n, uint32_t steps) {
    if (!m || !caches) return fail(FQ_ERR_INVALID_ARGUMENT, "null model or caches");
    if (!m->tok_embd.q) return fail(FQ_ERR_INVALID_ARGUMENT, "layer-only model (loaded without tok_embd)");
    if (n == 0) return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "empty batch");
    if (n > (uint32_t)MAX_SEQ) return fail(FQ_ERR_INVALID_ARGUMENT, "batch %u exceeds %d", n, MAX_SEQ);
    for (uint32_t s = 0; s < n; ++s) {
        if (!caches[s]) return fail(FQ_ERR_INVALID_ARGUMENT, "cache %u is null", s);
        if (caches[s]->m != m) return fail(FQ_ERR_MISMATCHED_KV_CACHES, "cache %u belongs to another model", s);
        if (caches[s]->type != caches[0]->type) return fail(FQ_ERR_MISMATCHED_KV_CACHES, "cache dtypes differ");
        for (uint32_t t = 0; t < s; ++t)
            if (caches[t] == caches[s]) return fail(FQ_ERR_MISMATCHED_KV_CACHES, "cache %u repeated", s);
        if ((uint64_t)caches[s]->len + steps > caches[s]->cap)
            return fail(FQ_ERR_KV_CACHE_OVERFLOW, "cache %u: len %u + %u > capacity %u", s, caches[s]->len, steps,
                        caches[s]->cap);
    }
    return FQ_OK;
}

fq_status check_tokens(const fq_model* m, const int32_t* tokens, uint32_t n) {
    if (!tokens) return fail(FQ_ERR_INVALID_ARGUMENT, "null tokens");
    for (uint32_t i = 0; i < n; ++i)
        if (tokens[i] < 0 || (uint32_t)tokens[i] >= m->d.p.vocab_size)
            return fail(FQ_ERR_INVALID_ARGUMENT, "token %d out of range", tokens[i]);
    return FQ_OK;
}

uint32_t max_cap(fq_kv* const* caches, uint32_t n) {
    uint32_t c = 0;
    for (uint32_t i = 0; i < n; ++i) c = std::max(c, caches[i]->cap);
    return c;
}

// ---------------------------------------------------------------- loading

size_t packed_row_bytes(fq_dtype t, uint64_t cols) {
    switch (t) {
        case FQ_Q8_0: return cols / 32 * 34;
        case FQ_Q4_K: return cols / 256 * 144;
        case FQ_F32: return cols * 4;
        default: return 0;
    }
}

fq_status check_tensor(const fq_tensor& t, const char* name, uint64_t rows, uint64_t cols, bool quant) {
    if (!t.data) return fail(FQ_ERR_INVALID_ARGUMENT, "%s: missing data", name);
    if (t.rows != rows || t.cols != cols)
        return fail(FQ_ERR_INVALID_ARGUMENT, "%s: shape [%llu, %llu], expected [%llu, %llu]", name,
                    (unsigned long long)t.rows, (unsigned long long)t.cols, (unsigned long long)rows,
                    (unsigned long long)cols);
    if (quant) {
        if (t.dtype != FQ_Q8_0 && t.dtype != FQ_Q4_K) return fail(FQ_ERR_INVALID_ARGUMENT, "%s: dtype must be Q8_0 or Q4_K", name);
        if (t.dtype == FQ_Q4_K && cols % 256) return fail(FQ_ERR_INVALID_ARGUMENT, "%s: Q4_K needs cols %% 256 == 0", name);
        if (cols % 32) return fail(FQ_ERR_INVALID_ARGUMENT, "%s: cols %% 32 != 0", name);
    } else if (t.dtype != FQ_F32) {
        return fail(FQ_ERR_INVALID_ARGUMENT, "%s: dtype must be F32", name);
    }
    return FQ_OK;
}

struct Loader {
    fq_model* m;
    cudaStream_t s;
    uint8_t* staging = nullptr;
    size_t staging_cap = 0;

    fq_status stage(const fq_tensor& t, size_t bytes) {
        if (bytes > staging_cap) {
            CK(cudaStreamSynchronize(s));
            if (staging) cudaFree(staging);
            staging = nullptr;
            CK(cudaMalloc(&staging, bytes));
            staging_cap = bytes;
        }
        CK(cudaMemcpyAsync(staging, t.data, bytes, cudaMemcpyHostToDevice, s));
        return FQ_OK;
    }
    // allocate an empty matrix of `rows` x `cols` in format fmt
    fq_status alloc(QMat& q, int fmt, uint64_t rows, uint64_t cols) {
        q.fmt = fmt;
        q.N = (int)rows;
        q.K = (int)cols;
        uint8_t* qp;
        TRY(dalloc(m->allocs, &qp, q.row_bytes() * rows));
        q.q = qp;
        if (fmt == FMT_Q8_0) {
            uint16_t* sp;
            TRY(dalloc(m->allocs, &sp, rows * (cols / 32)));
            q.s = sp;
        }
        return FQ_OK;
    }
    // place the rows of t into q with the row mapping (group, group_stride, step, off)
    fq_status place(const fq_tensor& t, QMat& q, int64_t group, int64_t gstride, int64_t step, int64_t off) {
        size_t bytes = packed_row_bytes(t.dtype, t.cols) * t.rows;
        TRY(stage(t, bytes));
        if (q.fmt == FMT_Q8_0)
            launch_repack_q8_0(staging, (int64_t)t.rows, (int64_t)t.cols, const_cast<uint8_t*>(q.q),
                               const_cast<uint16_t*>(q.s), group, gstride, step, off, s);
        else
            launch_copy_rows(staging, (int64_t)t.rows, (int64_t)q.row_bytes(), const_cast<uint8_t*>(q.q), group,
                             gstride, step, off, s);
        CK(cudaGetLastError());
        return FQ_OK;
    }
    fq_status plain(const fq_tensor& t, QMat& q) {
        TRY(alloc(q, t.dtype, t.rows, t.cols));
        return place(t, q, (int64_t)t.rows, 0, 1, 0);
    }
    fq_status vec(const fq_tensor& t, const float** out, uint64_t n) {
        float* p;
        TRY(dalloc(m->allocs, &p, n));
        CK(cudaMemcpyAsync(p, t.data, n * 4, cudaMemcpyHostToDevice, s));
        *out = p;
        return FQ_OK;
    }
};

}  // namespace

// ==================================================================== C ABI

extern "C" {

const char* fq_last_error(void) { return g_err.c_str(); }

const char* fq_status_str(fq_status s) {
    switch (s) {
        case FQ_OK: return "ok";
        case FQ_ERR_INVALID_CONFIG: return "invalid config";
        case FQ_ERR_INVALID_SEQUENCE_LENGTH: return "invalid sequence length";
        case FQ_ERR_KV_CACHE_OVERFLOW: return "kv cache overflow";
        case FQ_ERR_MISMATCHED_KV_CACHES: return "mismatched kv caches";
        case FQ_ERR_INVALID_ARGUMENT: return "invalid argument";
        case FQ_ERR_OUT_OF_MEMORY: return "out of memory";
        case FQ_ERR_CUDA: return "cuda error";
        case FQ_ERR_DEVICE_TIMEOUT: return "device timeout";
        case FQ_ERR_UNSUPPORTED: return "unsupported";
    }
    return "unknown";
}

fq_status fq_desc_init(fq_desc* d, const fq_desc_params* p) {
    if (!d || !p) return fail(FQ_ERR_INVALID_ARGUMENT, "null descriptor");
    memset(d, 0, sizeof *d);
    // section 14.2 validation
    if (!p->vocab_size || !p->hidden_size || !p->num_layers || !p->head_dim)
        return fail(FQ_ERR_INVALID_CONFIG, "zero dimension");
    if (!p->num_attention_heads || !p->num_key_value_heads) return fail(FQ_ERR_INVALID_CONFIG, "zero heads");
    if (p->num_attention_heads % p->num_key_value_heads)
        return fail(FQ_ERR_INVALID_CONFIG, "num_attention_heads %u not divisible by num_key_value_heads %u",
                    p->num_attention_heads, p->num_key_value_heads);
    if (p->head_dim % 2) return fail(FQ_ERR_INVALID_CONFIG, "odd head_dim %u", p->head_dim);
    bool any = p->num_experts || p->num_experts_used || p->moe_intermediate_size;
    bool all = p->num_experts && p->num_experts_used && p->moe_intermediate_size;
    if (any && !all) return fail(FQ_ERR_INVALID_CONFIG, "inconsistent MoE fields");
    if (all && p->num_experts_used > p->num_experts) return fail(FQ_ERR_INVALID_CONFIG, "num_experts_used > num_experts");
    if (!all && !p->intermediate_size) return fail(FQ_ERR_INVALID_CONFIG, "zero intermediate_size");
    if (!(p->rms_norm_eps > 0.f) || !(p->rope_theta > 0.f)) return fail(FQ_ERR_INVALID_CONFIG, "eps/theta must be > 0");
    if (p->moe_expert_top_p != 1.0f) return fail(FQ_ERR_INVALID_CONFIG, "moe_expert_top_p must be 1.0 (full top-k)");
    // what the kernels are built for
    if (p->head_dim != HEAD_DIM) return fail(FQ_ERR_UNSUPPORTED, "head_dim %u (kernels take 128)", p->head_dim);
    if (p->hidden_size % 256) return fail(FQ_ERR_UNSUPPORTED, "hidden_size %% 256 != 0");
    int G = p->num_attention_heads / p->num_key_value_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return fail(FQ_ERR_UNSUPPORTED, "GQA group %d (1, 2, 4 or 8)", G);
    if (all && (p->num_experts > (uint32_t)MAX_EXPERTS || p->num_experts_used > (uint32_t)MAX_TOPK))
        return fail(FQ_ERR_UNSUPPORTED, "more than %d experts or top-k above %d", MAX_EXPERTS, MAX_TOPK);
    if (all && p->moe_intermediate_size % 32) return fail(FQ_ERR_UNSUPPORTED, "moe_intermediate_size %% 32 != 0");
    if (!all && p->intermediate_size % 32) return fail(FQ_ERR_UNSUPPORTED, "intermediate_size %% 32 != 0");
    d->p = *p;
    if (!d->p.max_positions) d->p.max_positions = 40960;
    d->magic = DESC_MAGIC;
    return FQ_OK;
}

fq_status fq_load_weights(const fq_desc* d, const fq_weight_src* src, void* stream, fq_model** out) {
    if (!d || !src || !out) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (d->magic != DESC_MAGIC) return fail(FQ_ERR_INVALID_ARGUMENT, "descriptor not initialised by fq_desc_init");
    if (!src->layers) return fail(FQ_ERR_INVALID_ARGUMENT, "null layers");
    *out = nullptr;
    const auto& p = d->p;
    const uint64_t H = p.hidden_size, D = p.head_dim, Hq = p.num_attention_heads, Hkv = p.num_key_value_heads;
    const bool moe = p.num_experts > 0;
    // ---- validate everything before allocating
    const bool has_embd = src->tok_embd.data != nullptr;   // layer-only models have none
    if (has_embd) TRY(check_tensor(src->tok_embd, "tok_embd", p.vocab_size, H, true));
    if (!has_embd && src->output.data)
        return fail(FQ_ERR_INVALID_ARGUMENT, "output without tok_embd");
    if (has_embd && check_tensor(src->output_norm, "output_norm", H, 1, false) != FQ_OK)
        TRY(check_tensor(src->output_norm, "output_norm", 1, H, false));
    if (src->output.data) TRY(check_tensor(src->output, "output", p.vocab_size, H, true));
    for (uint32_t L = 0; L < p.num_layers; ++L) {
        const fq_layer_src& l = src->layers[L];
        char nm[64];
        auto chk = [&](const fq_tensor& t, const char* what, uint64_t r, uint64_t c, bool q) {
            snprintf(nm, sizeof nm, "blk.%u.%s", L, what);
            return check_tensor(t, nm, r, c, q);
        };
        auto chkv = [&](const fq_tensor& t, const char* what, uint64_t n) {
            snprintf(nm, sizeof nm, "blk.%u.%s", L, what);
            if (check_tensor(t, nm, n, 1, false) == FQ_OK) return FQ_OK;
            return check_tensor(t, nm, 1, n, false);
        };
        TRY(chkv(l.attn_norm, "attn_norm", H));
        TRY(chkv(l.ffn_norm, "ffn_norm", H));
        TRY(chkv(l.q_norm, "attn_q_norm", D));
        TRY(chkv(l.k_norm, "attn_k_norm", D));
        TRY(chk(l.wq, "attn_q", Hq * D, H, true));
        TRY(chk(l.wk, "attn_k", Hkv * D, H, true));
        TRY(chk(l.wv, "attn_v", Hkv * D, H, true));
        TRY(chk(l.wo, "attn_output", H, Hq * D, true));
        if (l.wk.dtype != l.wq.dtype || l.wv.dtype != l.wq.dtype)
            return fail(FQ_ERR_INVALID_ARGUMENT, "blk.%u: q/k/v dtypes differ (cannot fuse)", L);
        if (!moe) {
            TRY(chk(l.w_gate, "ffn_gate", p.intermediate_size, H, true));
            TRY(chk(l.w_up, "ffn_up", p.intermediate_size, H, true));
            TRY(chk(l.w_down, "ffn_down", H, p.intermediate_size, true));
            if (l.w_up.dtype != l.w_gate.dtype) return fail(FQ_ERR_INVALID_ARGUMENT, "blk.%u: gate/up dtypes differ", L);
        } else {
            const uint64_t E = p.num_experts, Fe = p.moe_intermediate_size;
            TRY(chk(l.router, "ffn_gate_inp", E, H, false));
            TRY(chk(l.gate_exps, "ffn_gate_exps", E * Fe, H, true));
            TRY(chk(l.up_exps, "ffn_up_exps", E * Fe, H, true));
            TRY(chk(l.down_exps, "ffn_down_exps", E * H, Fe, true));
            if (l.up_exps.dtype != l.gate_exps.dtype)
                return fail(FQ_ERR_INVALID_ARGUMENT, "blk.%u: expert gate/up dtypes differ", L);
        }
    }
    int dev = 0;
    CK(cudaGetDevice(&dev));
    gemv_prepare();
    gemm_tc_prepare();
    attention_prepare();
    stream_prepare();
    CK(cudaGetLastError());
    fq_model* m = new fq_model();
    m->d = *d;
    m->device = dev;
    m->layers.resize(p.num_layers);
    cudaStream_t s = (cudaStream_t)stream;
    Loader ld{m, s};
    auto cleanup = [&](fq_status st) {
        cudaStreamSynchronize(s);
        if (ld.staging) cudaFree(ld.staging);
        if (st != FQ_OK) {
            for (void* q : m->allocs) cudaFree(q);
            delete m;
        }
        return st;
    };
    fq_status st = [&]() -> fq_status {
        if (has_embd) {
            TRY(ld.plain(src->tok_embd, m->tok_embd));
            TRY(ld.vec(src->output_norm, &m->output_norm, H));
            if (src->output.data) TRY(ld.plain(src->output, m->output));
            else m->output = m->tok_embd;   // tied embeddings
        }
        for (uint32_t L = 0; L < p.num_layers; ++L) {
            const fq_layer_src& l = src->layers[L];
            LayerW& w = m->layers[L];
            TRY(ld.vec(l.attn_norm, &w.attn_norm, H));
            TRY(ld.vec(l.ffn_norm, &w.ffn_norm, H));
            TRY(ld.vec(l.q_norm, &w.q_norm, D));
            TRY(ld.vec(l.k_norm, &w.k_norm, D));
            // q/k/v -> one QKV matrix (rows q | k | v)
            TRY(ld.alloc(w.qkv, l.wq.dtype, (Hq + 2 * Hkv) * D, H));
            TRY(ld.place(l.wq, w.qkv, (int64_t)(Hq * D), 0, 1, 0));
            TRY(ld.place(l.wk, w.qkv, (int64_t)(Hkv * D), 0, 1, (int64_t)(Hq * D)));
            TRY(ld.place(l.wv, w.qkv, (int64_t)(Hkv * D), 0, 1, (int64_t)((Hq + Hkv) * D)));
            TRY(ld.plain(l.wo, w.o));
            if (!moe) {
                const int64_t F = p.intermediate_size;
                // gate/up -> one gate_up matrix, rows interleaved so one warp owns both halves of h_i
                TRY(ld.alloc(w.gate_up, l.w_gate.dtype, 2 * F, H));
                TRY(ld.place(l.w_gate, w.gate_up, F, 0, 2, 0));
                TRY(ld.place(l.w_up, w.gate_up, F, 0, 2, 1));
                TRY(ld.plain(l.w_down, w.down));
            } else {
                const int64_t E = p.num_experts, Fe = p.moe_intermediate_size;
                TRY(ld.plain(l.router, w.router));
                TRY(ld.alloc(w.gate_up_exps, l.gate_exps.dtype, E * 2 * Fe, H));
                TRY(ld.place(l.gate_exps, w.gate_up_exps, Fe, 2 * Fe, 2, 0));
                TRY(ld.place(l.up_exps, w.gate_up_exps, Fe, 2 * Fe, 2, 1));
                TRY(ld.plain(l.down_exps, w.down_exps));
            }
        }
        uint32_t* errw;
        TRY(dalloc(m->allocs, &errw, 1));
        CK(cudaMemsetAsync(errw, 0, sizeof(uint32_t), s));
        m->err = errw;
        // tensor maps for the bulk-copy GEMV (expert stacks keep the register-fed path)
        auto attach = [&](QMat& q) {
            if (!q.q) return;
            m->tmaps.emplace_back();
            const bool gemv_ok = make_tma_maps(q, &m->tmaps.back());
            if (gemv_ok || m->tmaps.back().tc_ok) q.tm = &m->tmaps.back();
        };
        attach(m->tok_embd);
        if (m->output.q != m->tok_embd.q) attach(m->output);
        else m->output.tm = m->tok_embd.tm;
        for (auto& lw : m->layers) {
            attach(lw.qkv); attach(lw.o); attach(lw.gate_up); attach(lw.down); attach(lw.router);
        }
        // layer table of the streamed batch-1 step: a dense model whose projections and LM
        // head share one quantised format, with K % 256 == 0 (whole bulk-copy rows)
        {
            const int fmt = m->output.fmt;
            auto fits = [&](const QMat& q) { return q.q && q.fmt == fmt && q.K % 256 == 0; };
            const uint32_t G = p.num_attention_heads / p.num_key_value_heads;
            bool ok = !m->moe() && m->tok_embd.q && m->output.q && (fmt == FMT_Q8_0 || fmt == FMT_Q4_K) &&
                      m->output.K % 256 == 0 && (G == 1 || G == 2 || G == 4);
            std::vector<StreamLayer> sl(p.num_layers);
            for (uint32_t L = 0; L < p.num_layers && ok; ++L) {
                const LayerW& lw = m->layers[L];
                ok = fits(lw.qkv) && fits(lw.o) && fits(lw.gate_up) && fits(lw.down);
                sl[L] = StreamLayer{lw.qkv, lw.o, lw.gate_up, lw.down, lw.attn_norm, lw.ffn_norm, lw.q_norm, lw.k_norm};
            }
            StreamArgs& sp = m->splan;
            sp.n_layers = (int)p.num_layers;
            sp.H = (int)H;
            sp.F = (int)p.intermediate_size;
            sp.Hq = (int)Hq;
            sp.Hkv = (int)Hkv;
            sp.V = (int)p.vocab_size;
            sp.eps = p.rms_norm_eps;
            sp.emb = m->tok_embd;
            sp.out = m->output;
            sp.out_norm = m->output_norm;
            sp.head = 1;
            sp.S = stream_chunks((int)Hkv);
            sp.max_pos = (int)p.max_positions;
            std::vector<ProjPlan> plans;
            if (ok && stream_plan(sp, sl[0], fmt, (int)G, plans)) {
                StreamLayer* dsl;
                TRY(dalloc(m->allocs, &dsl, sl.size()));
                CK(cudaMemcpyAsync(dsl, sl.data(), sizeof(StreamLayer) * sl.size(), cudaMemcpyHostToDevice, s));
                ProjPlan* dpp;
                TRY(dalloc(m->allocs, &dpp, plans.size()));
                CK(cudaMemcpyAsync(dpp, plans.data(), sizeof(ProjPlan) * plans.size(), cudaMemcpyHostToDevice, s));
                m->slayers = dsl;
                sp.layers = dsl;
                sp.plan = dpp;
                m->sfmt = fmt;
                m->sG = (int)G;
            }
        }
        m->max_pos = (int)p.max_positions;
        float2* rope;
        TRY(dalloc(m->allocs, &rope, (size_t)m->max_pos * (HEAD_DIM / 2)));
        m->rope = rope;
        m->splan.rope = rope;
        launch_rope_table(rope, m->max_pos, (double)p.rope_theta, s);
        CK(cudaGetLastError());
        CK(cudaStreamSynchronize(s));
        return FQ_OK;
    }();
    st = cleanup(st);
    if (st == FQ_OK) *out = m;
    return st;
}

void fq_model_free(fq_model* m) {
    if (!m) return;
    for (auto& kv : m->ws) {
        cudaStreamSynchronize(kv.first);
        kv.second->release();
        delete kv.second;
    }
    for (void* p : m->allocs) cudaFree(p);
    delete m;
}

fq_status fq_kv_init(const fq_model* m, uint32_t capacity, fq_dtype kv_dtype, fq_kv** out) {
    if (!m || !out) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (capacity == 0) return fail(FQ_ERR_INVALID_ARGUMENT, "zero capacity");
    if (capacity > (uint32_t)m->max_pos)
        return fail(FQ_ERR_INVALID_ARGUMENT, "capacity %u exceeds max_positions %d", capacity, m->max_pos);
    if (kv_dtype != FQ_F32 && kv_dtype != FQ_BF16 && kv_dtype != FQ_Q8_0)
        return fail(FQ_ERR_INVALID_ARGUMENT, "kv dtype must be F32, BF16 or Q8_0");
    fq_kv* kv = new fq_kv();
    kv->m = m;
    kv->cap = capacity;
    kv->type = kv_dtype == FQ_F32 ? KV_F32 : kv_dtype == FQ_BF16 ? KV_BF16 : KV_Q8_0;
    const size_t heads = (size_t)m->d.p.num_layers * m->d.p.num_key_value_heads;
    const size_t vbytes = heads * capacity * HEAD_DIM * kv->elem();
    const size_t sbytes = kv->type == KV_Q8_0 ? heads * kv->cap_s() * (HEAD_DIM / 32) * 2 : 0;
    size_t bytes = vbytes + sbytes;
    cudaError_t e1 = cudaMalloc(&kv->k, bytes);
    cudaError_t e2 = e1 == cudaSuccess ? cudaMalloc(&kv->v, bytes) : e1;
    if (e1 != cudaSuccess || e2 != cudaSuccess) {
        cudaGetLastError();
        if (kv->k) cudaFree(kv->k);
        delete kv;
        return fail(FQ_ERR_OUT_OF_MEMORY, "kv cache of %zu bytes", 2 * bytes);
    }
    cudaMemset(kv->k, 0, bytes);
    cudaMemset(kv->v, 0, bytes);
    if (sbytes) {
        kv->ks = (char*)kv->k + vbytes;   // vbytes is a multiple of 128
        kv->vs = (char*)kv->v + vbytes;
    }
    *out = kv;
    return FQ_OK;
}

void fq_kv_free(fq_kv* kv) {
    if (!kv) return;
    cudaFree(kv->k);
    cudaFree(kv->v);
    delete kv;
}

uint32_t fq_kv_len(const fq_kv* kv) { return kv ? kv->len : 0; }
uint32_t fq_kv_capacity(const fq_kv* kv) { return kv ? kv->cap : 0; }

static fq_status kv_copy(const fq_kv* kv, uint32_t layer, uint32_t pos, uint32_t n_pos, void* k, void* v,
                         void* stream, bool to_cache) {
    const auto& p = kv->m->d.p;
    const size_t es = kv->elem(), row = HEAD_DIM * es, Hkv = p.num_key_value_heads;
    cudaStream_t s = (cudaStream_t)stream;
    if (kv->type == KV_Q8_0) {   // ggml blocks [n_pos][Hkv][4][34] <-> code and scale planes
        const size_t lc = (size_t)layer * Hkv * kv->cap * HEAD_DIM, ls = (size_t)layer * Hkv * kv->cap_s() * 4;
        launch_kv_q8_copy((int8_t*)kv->k + lc, (uint16_t*)kv->ks + ls, kv->cap, kv->cap_s(), (int)Hkv, (int)pos,
                          (int)n_pos, (uint8_t*)k, to_cache, s);
        launch_kv_q8_copy((int8_t*)kv->v + lc, (uint16_t*)kv->vs + ls, kv->cap, kv->cap_s(), (int)Hkv, (int)pos,
                          (int)n_pos, (uint8_t*)v, to_cache, s);
        CK(cudaGetLastError());
        return FQ_OK;
    }
    for (size_t h = 0; h < Hkv; ++h) {
        size_t coff = (((size_t)layer * Hkv + h) * kv->cap + pos) * row;
        char* ck = (char*)kv->k + coff;
        char* cv = (char*)kv->v + coff;
        char* uk = (char*)k + h * row;
        char* uv = (char*)v + h * row;
        if (to_cache) {
            CK(cudaMemcpy2DAsync(ck, row, uk, Hkv * row, row, n_pos, cudaMemcpyDeviceToDevice, s));
            CK(cudaMemcpy2DAsync(cv, row, uv, Hkv * row, row, n_pos, cudaMemcpyDeviceToDevice, s));
        } else {
            CK(cudaMemcpy2DAsync(uk, Hkv * row, ck, row, row, n_pos, cudaMemcpyDeviceToDevice, s));
            CK(cudaMemcpy2DAsync(uv, Hkv * row, cv, row, row, n_pos, cudaMemcpyDeviceToDevice, s));
        }
    }
    return FQ_OK;
}

fq_status fq_kv_append(fq_kv* kv, uint32_t layer, uint32_t pos, uint32_t n_pos, const void* k, const void* v,
                       void* stream) {
    if (!kv || !k || !v) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (layer >= kv->m->d.p.num_layers) return fail(FQ_ERR_INVALID_ARGUMENT, "layer %u out of range", layer);
    if (pos != kv->len) return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "append at %u but len is %u", pos, kv->len);
    if ((uint64_t)pos + n_pos > kv->cap) return fail(FQ_ERR_KV_CACHE_OVERFLOW, "%u + %u > capacity %u", pos, n_pos, kv->cap);
    if (n_pos == 0) return FQ_OK;
    return kv_copy(kv, layer, pos, n_pos, const_cast<void*>(k), const_cast<void*>(v), stream, true);
}

fq_status fq_kv_commit(fq_kv* kv, uint32_t len) {
    if (!kv) return fail(FQ_ERR_INVALID_ARGUMENT, "null cache");
    if (len > kv->cap) return fail(FQ_ERR_KV_CACHE_OVERFLOW, "len %u > capacity %u", len, kv->cap);
    if (len < kv->len) return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "len %u < current %u", len, kv->len);
    kv->len = len;
    return FQ_OK;
}

fq_status fq_kv_rewind(fq_kv* kv, uint32_t len) {
    if (!kv) return fail(FQ_ERR_INVALID_ARGUMENT, "null cache");
    if (len > kv->len) return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "rewind to %u beyond len %u", len, kv->len);
    kv->len = len;
    return FQ_OK;
}

fq_status fq_kv_read(const fq_kv* kv, uint32_t layer, uint32_t pos, uint32_t n_pos, void* k, void* v, void* stream) {
    if (!kv || !k || !v) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (layer >= kv->m->d.p.num_layers) return fail(FQ_ERR_INVALID_ARGUMENT, "layer %u out of range", layer);
    if ((uint64_t)pos + n_pos > kv->cap) return fail(FQ_ERR_INVALID_ARGUMENT, "range beyond capacity");
    if (n_pos == 0) return FQ_OK;
    return kv_copy(kv, layer, pos, n_pos, k, v, stream, false);
}

fq_status fq_layer_step(const fq_model* m, uint32_t layer, fq_kv* kv, uint32_t pos, float* x, void* stream) {
    if (!m || !kv || !x) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (layer >= m->d.p.num_layers) return fail(FQ_ERR_INVALID_ARGUMENT, "layer %u out of range", layer);
    if (kv->m != m) return fail(FQ_ERR_MISMATCHED_KV_CACHES, "cache belongs to another model");
    if (pos != kv->len) return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "pos %u != len %u", pos, kv->len);
    if ((uint64_t)pos + 1 > kv->cap) return fail(FQ_ERR_KV_CACHE_OVERFLOW, "len %u at capacity", kv->len);
    cudaStream_t s = (cudaStream_t)stream;
    Workspace* w;
    TRY(ensure_ws(m, s, 1, kv->cap, &w));
    fq_kv* caches[1] = {kv};
    TRY(setup_state(w, caches, nullptr, 1, false, nullptr, nullptr, s));
    Body b{m, w, 1, 0, 0, nullptr, false};
    attn_split(1, m->d.p.num_key_value_heads, kv->cap, b.chunk, b.splits);
    return enqueue_step(b, s, kv->type, x, (int)layer);
}

fq_status fq_decode_step_batch(const fq_model* m, fq_kv* const* caches, uint32_t n, const int32_t* tokens,
                               float* logits, void* stream) {
    TRY(check_caches(m, caches, n, 1));
    TRY(check_tokens(m, tokens, n));
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t cap = max_cap(caches, n);
    Workspace* w;
    TRY(ensure_ws(m, s, (int)n, cap, &w));
    TRY(setup_state(w, caches, tokens, (int)n, false, nullptr, logits, s));
    Body b{m, w, (int)n, 0, 0, logits, false};
    attn_split((int)n, m->d.p.num_key_value_heads, cap, b.chunk, b.splits);
    TRY(run_body(b, s, caches[0]->type, 1));
    for (uint32_t i = 0; i < n; ++i) caches[i]->len += 1;
    return FQ_OK;
}

// Rows of one sequence per pass of a multi-token forwardStep: the lockstep batch the
// tensor-core projections are built and tested for.
constexpr uint32_t FORWARD_ROWS = 32;

fq_status fq_forward_step(const fq_model* m, fq_kv* kv, const int32_t* tokens, uint32_t len, uint32_t pos0,
                          float* logits, void* stream) {
    if (!m || !kv) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (kv->m != m) return fail(FQ_ERR_MISMATCHED_KV_CACHES, "cache belongs to another model");
    if (!m->tok_embd.q) return fail(FQ_ERR_INVALID_ARGUMENT, "model has no embedding");
    if (logits && !m->output.q) return fail(FQ_ERR_INVALID_ARGUMENT, "model has no LM head");
    if (len == 0) return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "empty input");
    if (pos0 != kv->len) return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "pos0 %u != len %u", pos0, kv->len);
    if ((uint64_t)kv->len + len > kv->cap)
        return fail(FQ_ERR_KV_CACHE_OVERFLOW, "len %u + %u > capacity %u", kv->len, len, kv->cap);
    TRY(check_tokens(m, tokens, len));
    cudaStream_t s = (cudaStream_t)stream;
    std::vector<fq_kv*> rows(std::min(len, FORWARD_ROWS), kv);
    for (uint32_t off = 0; off < len; off += FORWARD_ROWS) {
        const uint32_t n = std::min(FORWARD_ROWS, len - off);
        const bool last = off + n == len;
        Workspace* w;
        TRY(ensure_ws(m, s, (int)n, kv->cap, &w));   // grows only; a shorter last pass may want more splits
        TRY(setup_state(w, rows.data(), tokens + off, (int)n, false, nullptr, nullptr, s, 1));
        Body b{m, w, (int)n, 0, 0, last ? logits : nullptr, false};
        b.block = true;
        b.head_row = (int)n - 1;
        attn_split((int)n, m->d.p.num_key_value_heads, kv->cap, b.chunk, b.splits);
        TRY(enqueue_step(b, s, kv->type, nullptr, -1));
        kv->len += n;   // the next pass's rows sit after this one's
    }
    return FQ_OK;
}

fq_status fq_decode_step_all_logits(const fq_model* m, fq_kv* kv, const int32_t* tokens, uint32_t len, uint32_t pos0,
                                    float* logits, void* stream) {
    if (!m || !kv || !logits) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (kv->m != m) return fail(FQ_ERR_MISMATCHED_KV_CACHES, "cache belongs to another model");
    if (!m->tok_embd.q || !m->output.q) return fail(FQ_ERR_INVALID_ARGUMENT, "model has no embedding or LM head");
    if (len == 0 || len > (uint32_t)MAX_SEQ)
        return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "len %u outside 1..%d", len, MAX_SEQ);
    if (pos0 != kv->len) return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "pos0 %u != len %u", pos0, kv->len);
    if ((uint64_t)kv->len + len > kv->cap)
        return fail(FQ_ERR_KV_CACHE_OVERFLOW, "len %u + %u > capacity %u", kv->len, len, kv->cap);
    TRY(check_tokens(m, tokens, len));
    cudaStream_t s = (cudaStream_t)stream;
    Workspace* w;
    TRY(ensure_ws(m, s, (int)len, kv->cap, &w));
    std::vector<fq_kv*> rows(len, kv);
    TRY(setup_state(w, rows.data(), tokens, (int)len, false, nullptr, logits, s, 1));
    Body b{m, w, (int)len, 0, 0, logits, false};
    b.block = true;
    attn_split((int)len, m->d.p.num_key_value_heads, kv->cap, b.chunk, b.splits);
    TRY(enqueue_step(b, s, kv->type, nullptr, -1));
    kv->len += len;
    return FQ_OK;
}

fq_status fq_decode_step(const fq_model* m, fq_kv* kv, int32_t token, uint32_t pos0, float* logits, void* stream) {
    if (!m || !kv) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (kv->m != m) return fail(FQ_ERR_MISMATCHED_KV_CACHES, "cache belongs to another model");
    if (pos0 != kv->len) return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "pos0 %u != len %u", pos0, kv->len);
    fq_kv* caches[1] = {kv};
    return fq_decode_step_batch(m, caches, 1, &token, logits, stream);
}

fq_status fq_decode_greedy(const fq_model* m, fq_kv* const* caches, uint32_t n, const int32_t* first_tokens,
                           uint32_t n_steps, int32_t* tokens_out, float* logits, void* stream) {
    TRY(check_caches(m, caches, n, n_steps));
    TRY(check_tokens(m, first_tokens, n));
    if (n_steps == 0) return FQ_OK;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t cap = max_cap(caches, n);
    Workspace* w;
    TRY(ensure_ws(m, s, (int)n, cap, &w));
    float* lg = logits ? logits : w->logits;
    TRY(setup_state(w, caches, first_tokens, (int)n, true, tokens_out, lg, s));
    Body b{m, w, (int)n, 0, 0, lg, true};
    attn_split((int)n, m->d.p.num_key_value_heads, cap, b.chunk, b.splits);
    TRY(run_body(b, s, caches[0]->type, (int)n_steps));
    for (uint32_t i = 0; i < n; ++i) caches[i]->len += n_steps;
    return FQ_OK;
}

fq_status fq_decode_step_trace(const fq_model* m, fq_kv* const* caches, uint32_t n, const int32_t* tokens,
                               float* logits, float* layer_out, int32_t* route_idx, float* route_w,
                               float* route_logits, void* stream) {
    TRY(check_caches(m, caches, n, 1));
    TRY(check_tokens(m, tokens, n));
    if ((route_idx || route_w || route_logits) && !m->moe())
        return fail(FQ_ERR_INVALID_ARGUMENT, "route trace on a dense model");
    if ((route_idx == nullptr) != (route_w == nullptr)) return fail(FQ_ERR_INVALID_ARGUMENT, "route_idx and route_w go together");
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t cap = max_cap(caches, n);
    Workspace* w;
    TRY(ensure_ws(m, s, (int)n, cap, &w));
    TRY(setup_state(w, caches, tokens, (int)n, false, nullptr, logits, s));
    Body b{m, w, (int)n, 0, 0, logits, false, layer_out, route_idx, route_w, route_logits};
    attn_split((int)n, m->d.p.num_key_value_heads, cap, b.chunk, b.splits);
    TRY(enqueue_step(b, s, caches[0]->type, nullptr, -1));
    for (uint32_t i = 0; i < n; ++i) caches[i]->len += 1;
    return FQ_OK;
}

fq_status fq_layer_step_trace(const fq_model* m, uint32_t layer, fq_kv* kv, uint32_t pos, float* x, float* qkv,
                              float* attn, float* ffn, void* stream) {
    TRY(fq_layer_step(m, layer, kv, pos, x, stream));
    cudaStream_t s = (cudaStream_t)stream;
    Workspace* w;
    TRY(ensure_ws(m, s, 1, kv->cap, &w));
    const auto& p = m->d.p;
    if (qkv) CK(cudaMemcpyAsync(qkv, w->qkv, sizeof(float) * m->qkv_rows(), cudaMemcpyDeviceToDevice, s));
    if (attn)
        CK(cudaMemcpyAsync(attn, w->attn, sizeof(float) * p.num_attention_heads * HEAD_DIM, cudaMemcpyDeviceToDevice, s));
    if (ffn && !m->moe()) CK(cudaMemcpyAsync(ffn, w->h, sizeof(float) * p.intermediate_size, cudaMemcpyDeviceToDevice, s));
    return FQ_OK;
}

fq_status fq_gemv(const fq_model* m, uint32_t layer, fq_weight_id which, uint32_t n, const float* x, float* y,
                  void* stream) {
    if (!m || !x || !y) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (n == 0 || n > (uint32_t)MAX_SEQ) return fail(FQ_ERR_INVALID_ARGUMENT, "n must be 1..%d", MAX_SEQ);
    if (which != FQ_W_OUTPUT && layer >= m->d.p.num_layers) return fail(FQ_ERR_INVALID_ARGUMENT, "layer out of range");
    QMat W;
    switch (which) {
        case FQ_W_Q: W = m->layers[layer].qkv; break;
        case FQ_W_O: W = m->layers[layer].o; break;
        case FQ_W_GATE: W = m->layers[layer].gate_up; break;
        case FQ_W_DOWN: W = m->layers[layer].down; break;
        case FQ_W_OUTPUT: W = m->output; break;
        default: return fail(FQ_ERR_INVALID_ARGUMENT, "fq_gemv takes FQ_W_Q, FQ_W_O, FQ_W_GATE, FQ_W_DOWN or FQ_W_OUTPUT");
    }
    if (!W.q) return fail(FQ_ERR_INVALID_ARGUMENT, "weight not present in this model");
    GemvArgs g;
    g.W = W; g.B = (int)n; g.x = x; g.x_stride = W.K; g.y = y; g.y_stride = W.N; g.epi = EPI_STORE;
    g.ksplit = choose_ksplit(W, rows_per_warp(W));
    g.err = m->err;
    cudaStream_t s = (cudaStream_t)stream;
    Workspace* w = nullptr;
    if (n >= (uint32_t)TC_MIN_BATCH) TRY(ensure_ws(m, s, (int)n, 1, &w));
    if (w && w->xh && gemm_tc_applicable(g) && m->opt_tc)
        launch_gemm_tc(g, w->xh, w->tc_part, TC_PART_FLOATS, w->tc_tickets, s, false, false);
    else launch_gemv(g, s, false);
    CK(cudaGetLastError());
    return FQ_OK;
}

fq_status fq_set_option(fq_model* m, fq_option opt, int value) {
    if (!m) return fail(FQ_ERR_INVALID_ARGUMENT, "null model");
    switch (opt) {
        case FQ_OPT_STEP_PATH:
            if (value != FQ_PATH_AUTO && value != FQ_PATH_KERNELS)
                return fail(FQ_ERR_INVALID_ARGUMENT, "step path %d (FQ_PATH_AUTO or FQ_PATH_KERNELS)", value);
            m->opt_path = value;
            break;
        case FQ_OPT_DEPENDENT_LAUNCH: m->opt_pdl = value != 0; break;
        case FQ_OPT_GRAPHS: m->opt_graphs = value != 0; break;
        case FQ_OPT_TENSOR_CORES: m->opt_tc = value != 0; break;
        default: return fail(FQ_ERR_INVALID_ARGUMENT, "unknown option %d", (int)opt);
    }
    // graphs captured under the old setting must not replay
    std::lock_guard<std::mutex> lk(m->ws_mu);
    for (auto& kv : m->ws) {
        cudaStreamSynchronize(kv.first);
        kv.second->drop_graphs();
    }
    return FQ_OK;
}

fq_status fq_step_path(const fq_model* m, uint32_t n, fq_dtype kv_dtype, int* streamed) {
    if (!m || !streamed) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    *streamed = m->slayers && m->opt_path != FQ_PATH_KERNELS && n == 1 && kv_dtype == FQ_BF16 ? 1 : 0;
    return FQ_OK;
}

fq_status fq_step_kernels(const fq_model* m, void* stream, uint32_t* kernels) {
    if (!m || !kernels) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    std::lock_guard<std::mutex> lk(const_cast<fq_model*>(m)->ws_mu);
    auto it = m->ws.find((cudaStream_t)stream);
    *kernels = it == m->ws.end() ? 0u : it->second->last_kernels;
    return FQ_OK;
}

fq_status fq_check_device(const fq_model* m, void* stream) {
    if (!m) return fail(FQ_ERR_INVALID_ARGUMENT, "null model");
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t host = 0;
    CK(cudaMemcpyAsync(&host, m->err, sizeof host, cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    if (host) {
        // A CTA that gave up left its arrival counters and tickets half counted; every
        // workspace of the model is re-armed on its own stream (after the work queued there)
        // so that the next step pairs its partial results correctly.
        fq_model* mm = const_cast<fq_model*>(m);
        std::lock_guard<std::mutex> lk(mm->ws_mu);
        for (auto& kv : mm->ws) TRY(rearm_ws(m, kv.second, kv.first));
        CK(cudaMemsetAsync(m->err, 0, sizeof(uint32_t), s));
        return fail(FQ_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up (code %u)", host);
    }
    return FQ_OK;
}

fq_status fq_debug_wait_timeout(const fq_model* m, void* stream) {
    if (!m) return fail(FQ_ERR_INVALID_ARGUMENT, "null model");
    if (!m->output.q || !m->output.tm || !m->output.tm->ok)
        return fail(FQ_ERR_UNSUPPORTED, "the model's LM head has no bulk-copy GEMV maps");
    cudaStream_t s = (cudaStream_t)stream;
    Workspace* w;
    TRY(ensure_ws(m, s, 1, 1, &w));
    GemvArgs g;
    g.W = m->output; g.B = 1; g.x = w->x; g.x_stride = m->output.K; g.y = w->logits; g.y_stride = m->output.N;
    g.epi = EPI_STORE; g.err = m->err; g.starve = 1;
    if (!launch_gemv_tma(g, s, false)) return fail(FQ_ERR_UNSUPPORTED, "bulk-copy GEMV not applicable");
    CK(cudaGetLastError());
    return FQ_OK;
}

fq_status fq_quantize_q8_0(const float* x, uint64_t n, void* blocks, void* stream) {
    if (!x || !blocks) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (n % 128) return fail(FQ_ERR_INVALID_ARGUMENT, "n = %llu is not a multiple of 128", (unsigned long long)n);
    if ((uintptr_t)x % 16) return fail(FQ_ERR_INVALID_ARGUMENT, "x is not 16-byte aligned");
    launch_quantize_q8_0(x, (size_t)n, (uint8_t*)blocks, (cudaStream_t)stream);
    CK(cudaGetLastError());
    return FQ_OK;
}

fq_status fq_dequant_rows(const fq_model* m, uint32_t layer, fq_weight_id which, uint64_t row0, uint64_t n_rows,
                          float* out, void* stream) {
    if (!m || !out) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    const auto& p = m->d.p;
    const bool global = which == FQ_W_TOK_EMBD || which == FQ_W_OUTPUT;
    if (!global && layer >= p.num_layers) return fail(FQ_ERR_INVALID_ARGUMENT, "layer out of range");
    const LayerW* lw = global ? nullptr : &m->layers[layer];
    const uint64_t D = p.head_dim, Hq = p.num_attention_heads, Hkv = p.num_key_value_heads;
    QMat W;
    uint64_t rows = 0, off = 0, step = 1, group = 0, gstride = 0;
    switch (which) {
        case FQ_W_TOK_EMBD: W = m->tok_embd; rows = W.N; if (!W.q) return fail(FQ_ERR_INVALID_ARGUMENT, "no tok_embd"); break;
        case FQ_W_OUTPUT: W = m->output; rows = W.N; if (!W.q) return fail(FQ_ERR_INVALID_ARGUMENT, "no output"); break;
        case FQ_W_Q: W = lw->qkv; rows = Hq * D; break;
        case FQ_W_K: W = lw->qkv; rows = Hkv * D; off = Hq * D; break;
        case FQ_W_V: W = lw->qkv; rows = Hkv * D; off = (Hq + Hkv) * D; break;
        case FQ_W_O: W = lw->o; rows = W.N; break;
        case FQ_W_GATE: case FQ_W_UP:
            if (m->moe()) return fail(FQ_ERR_INVALID_ARGUMENT, "dense FFN weight on a MoE model");
            W = lw->gate_up; rows = p.intermediate_size; step = 2; off = which == FQ_W_UP; break;
        case FQ_W_DOWN:
            if (m->moe()) return fail(FQ_ERR_INVALID_ARGUMENT, "dense FFN weight on a MoE model");
            W = lw->down; rows = W.N; break;
        case FQ_W_GATE_EXPS: case FQ_W_UP_EXPS:
            if (!m->moe()) return fail(FQ_ERR_INVALID_ARGUMENT, "expert weight on a dense model");
            W = lw->gate_up_exps; rows = (uint64_t)p.num_experts * p.moe_intermediate_size;
            group = p.moe_intermediate_size; gstride = 2 * group; step = 2; off = which == FQ_W_UP_EXPS; break;
        case FQ_W_DOWN_EXPS:
            if (!m->moe()) return fail(FQ_ERR_INVALID_ARGUMENT, "expert weight on a dense model");
            W = lw->down_exps; rows = W.N; break;
        default: return fail(FQ_ERR_INVALID_ARGUMENT, "unknown weight id");
    }
    if (row0 + n_rows > rows) return fail(FQ_ERR_INVALID_ARGUMENT, "rows beyond the weight");
    cudaStream_t s = (cudaStream_t)stream;
    for (uint64_t i = 0; i < n_rows;) {
        // contiguous runs in the device matrix
        uint64_t r = row0 + i;
        uint64_t dr = group ? (r / group) * gstride + (r % group) * step + off : r * step + off;
        uint64_t run = 1;
        if (step == 1)
            while (i + run < n_rows && (group == 0 || (r + run) / group == r / group)) ++run;
        launch_dequant(W, (int64_t)dr, (int64_t)run, out + i * W.K, s);
        i += run;
    }
    CK(cudaGetLastError());
    return FQ_OK;
}

}  // extern "C"

// ==================================================================== layer step without allocation
//
// For callers that cannot call cudaMalloc (or must not have a library do it for them):
// an allocator that forbids device allocations after start-up, a CUDA graph that is being
// captured, or a host that pre-plans every byte of device memory.  The one layer step below
// keeps all of its scratch -- the step state, the raw QKV projections, the attention
// output and split-K partials, the arrival counters, the FFN activations -- in one
// file-scope device array instead of the per-stream workspace.  Every GPU that loads this
// library holds the array until the process exits.

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 2u << 20;   // 2 MiB
__device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of the array on the current device.  In host code the symbol is only a
// host-side stand-in, so the address is looked up once per device (with that device
// current) and cached.
fq_status noalloc_base(int model_device, void** out) {
    int dev = 0;
    CK(cudaGetDevice(&dev));
    if (dev != model_device)
        return fail(FQ_ERR_INVALID_ARGUMENT,
                    "current device %d is not the model's device %d (the built-in scratch array is per device)", dev,
                    model_device);
    if (dev < 0 || dev >= 64) return fail(FQ_ERR_INVALID_ARGUMENT, "device %d beyond the scratch table", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(FQ_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return FQ_OK;
}

}  // namespace

extern "C" fq_status fq_layer_step_noalloc(const fq_model* m, uint32_t layer, fq_kv* kv, uint32_t pos, float* x,
                                           void* stream) {
    if (!m || !kv || !x) return fail(FQ_ERR_INVALID_ARGUMENT, "null argument");
    if (layer >= m->d.p.num_layers) return fail(FQ_ERR_INVALID_ARGUMENT, "layer %u out of range", layer);
    if (kv->m != m) return fail(FQ_ERR_MISMATCHED_KV_CACHES, "cache belongs to another model");
    if (pos != kv->len) return fail(FQ_ERR_INVALID_SEQUENCE_LENGTH, "pos %u != len %u", pos, kv->len);
    if ((uint64_t)pos + 1 > kv->cap) return fail(FQ_ERR_KV_CACHE_OVERFLOW, "len %u at capacity", kv->len);
    const auto& p = m->d.p;
    int chunk, splits;
    attn_split(1, p.num_key_value_heads, kv->cap, chunk, splits);

    // carve the array: every piece 256-byte aligned
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += (bytes + 255) & ~(size_t)255; return o; };
    const size_t o_st = take(sizeof(StepState));
    const size_t o_qkv = take(sizeof(float) * m->qkv_rows());
    const size_t o_attn = take(sizeof(float) * p.num_attention_heads * HEAD_DIM);
    const size_t o_part = take(sizeof(float) * p.num_attention_heads * splits * (HEAD_DIM + 2));
    const size_t o_ctr = take(sizeof(uint32_t) * p.num_attention_heads);
    size_t o_h = 0, o_xn = 0, o_rl = 0, o_he = 0, o_ye = 0, o_route = 0;
    if (!m->moe()) {
        o_h = take(sizeof(float) * p.intermediate_size);
    } else {
        o_xn = take(sizeof(float) * p.hidden_size);
        o_rl = take(sizeof(float) * p.num_experts);
        o_he = take(sizeof(float) * p.num_experts_used * p.moe_intermediate_size);
        o_ye = take(sizeof(float) * p.num_experts_used * p.hidden_size);
        o_route = take(sizeof(MoeRoute));
    }
    if (off > NOALLOC_SCRATCH_BYTES)
        return fail(FQ_ERR_INVALID_ARGUMENT,
                    "layer step needs %zu bytes of scratch for this model and cache capacity; the built-in "
                    "array holds %zu (use fq_layer_step)",
                    off, NOALLOC_SCRATCH_BYTES);
    void* base = nullptr;
    TRY(noalloc_base(m->device, &base));
    unsigned char* b = (unsigned char*)base;
    Workspace w;   // a view into the array; owns nothing
    w.n_cap = 1;
    w.st = (StepState*)(b + o_st);
    w.qkv = (float*)(b + o_qkv);
    w.attn = (float*)(b + o_attn);
    w.part = (float*)(b + o_part);
    w.counters = (uint32_t*)(b + o_ctr);
    if (!m->moe()) {
        w.h = (float*)(b + o_h);
    } else {
        w.xn = (float*)(b + o_xn);
        w.rlogits = (float*)(b + o_rl);
        w.he = (float*)(b + o_he);
        w.ye = (float*)(b + o_ye);
        w.route = (MoeRoute*)(b + o_route);
    }
    cudaStream_t s = (cudaStream_t)stream;
    // the arrival counters must start at zero; the array keeps whatever the last call left
    CK(cudaMemsetAsync(w.counters, 0, sizeof(uint32_t) * p.num_attention_heads, s));
    fq_kv* caches[1] = {kv};
    TRY(setup_state(&w, caches, nullptr, 1, false, nullptr, nullptr, s));
    Body body{m, &w, 1, chunk, splits, nullptr, false};
    return enqueue_step(body, s, kv->type, x, (int)layer);
}
