// The whole batch-1 decode step of a dense model as one persistent kernel (sm_103a).
//
// forwardStep (fucina "14. Model families", section 14.2) at batch 1 is a chain of small
// dependent stages: per layer the fused RMSNorm + QKV projection, attention over the cache,
// the O projection, RMSNorm + gate_up + SwiGLU and the down projection, then the final norm
// and the LM head.  Launched one kernel per stage, each stage pays a launch and a cold start
// that are longer than its own streaming time (a 0.6B layer is 16.5 MB of weights: 2.5 us at
// the copy peak).  Here one cooperative launch (one CTA per SM, all resident) runs every
// stage as a phase and separates the phases with a grid barrier:
//   * a phase's work is split over all CTAs (rows of a projection, (kv head, chunk) units of
//     the attention, two 128-thread attention groups per CTA);
//   * before a CTA waits at a barrier it asks L2 for the bytes it will stream three phases
//     later (its rows of that projection, or its attention units' cached K/V), so HBM keeps
//     streaming while the barriers and the dependent loads resolve;
//   * cross-CTA activations are read through L2 (ld.global.cg), never a stale L1 line;
//   * the LM head's argmax keys are folded per CTA and the last CTA to finish (atomic
//     ticket, no waiting) performs the greedy hand-off.
// The barrier is a counter plus a generation word; every wait is bounded by a clock budget
// and a CTA that gives up records the error and leaves, so a broken run reports instead of
// hanging.

#include "attn_unit.cuh"
#include "common.cuh"
#include "kernels.h"
#include "quant.cuh"

#include <algorithm>

namespace fq {

namespace {

constexpr int PT = 256;             // threads per CTA
constexpr int PW = PT / 32;         // warps per CTA
constexpr int AG = PT / 128;        // attention groups per CTA
constexpr long long BAR_BUDGET = 1ll << 29;

FQ_DEV uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier: bar[0] counts arrivals, bar[1] is the generation.  Returns false (and sets
// the error word) when this CTA gave up waiting.
FQ_DEV bool grid_sync(uint32_t* bar, uint32_t* err) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        ok = 1;
        const uint32_t gen = ld_acquire(&bar[1]);
        __threadfence();
        if (atomicAdd(&bar[0], 1u) == gridDim.x - 1) {
            bar[0] = 0u;
            __threadfence();
            atomicAdd(&bar[1], 1u);
        } else {
            const long long t0 = clock64();
            while (ld_acquire(&bar[1]) == gen)
                if (clock64() - t0 > BAR_BUDGET) {
                    atomicOr(err, 64u);
                    ok = 0;
                    break;
                }
        }
        __threadfence();
    }
    __syncthreads();
    return ok != 0;
}

FQ_DEV void named_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

FQ_DEV void row_range(int N, int c, int G, bool pairs, int& r0, int& r1) {
    if (pairs) {
        const long long P = N / 2;
        r0 = 2 * (int)(P * c / G);
        r1 = 2 * (int)(P * (c + 1) / G);
    } else {
        r0 = (int)((long long)N * c / G);
        r1 = (int)((long long)N * (c + 1) / G);
    }
}

// L2 prefetch of rows [r0, r1) of W (codes and, for Q8_0, scales), at most `cap` bytes of codes
FQ_DEV void prefetch_rows(const QMat& W, int r0, int r1, size_t cap) {
    if (r1 <= r0 || !W.q) return;
    const size_t rb = W.row_bytes();
    size_t bytes = (size_t)(r1 - r0) * rb;
    if (bytes > cap) bytes = cap;
    prefetch_l2_range(W.q + (size_t)r0 * rb, bytes & ~(size_t)15, threadIdx.x, PT);
    if (W.fmt == FMT_Q8_0) {
        const size_t sb = (size_t)W.K / 16;   // scale bytes per row
        size_t a = (size_t)r0 * sb, e = (size_t)r1 * sb;
        a = (a + 15) & ~(size_t)15;
        e &= ~(size_t)15;
        if (e > a) prefetch_l2_range(reinterpret_cast<const uint8_t*>(W.s) + a, e - a, threadIdx.x, PT);
    }
}

// L2 prefetch of the cached K/V rows the attention units of this CTA will read at `layer`
FQ_DEV void prefetch_kv(const AttnArgs& at, int layer, int kv_bytes) {
    const SeqState ss = at.st->seq[0];
    const int pos = ss.pos;
    const int n_units = at.Hkv * at.splits;
    for (int u = blockIdx.x * AG; u < n_units; u += gridDim.x * AG)
        for (int gi = 0; gi < AG && u + gi < n_units; ++gi) {
            const int g = (u + gi) / at.splits, s = (u + gi) % at.splits;
            const int t0 = s * at.chunk, tc = min(t0 + at.chunk, pos);
            if (tc <= t0) continue;
            const size_t off = (((size_t)layer * at.Hkv + g) * (size_t)ss.cap + t0) * HEAD_DIM * kv_bytes;
            const size_t n = (size_t)(tc - t0) * HEAD_DIM * kv_bytes;
            prefetch_l2_range(reinterpret_cast<const uint8_t*>(ss.k) + off, n, threadIdx.x, PT);
            prefetch_l2_range(reinterpret_cast<const uint8_t*>(ss.v) + off, n, threadIdx.x, PT);
        }
}

// Block sum over PT threads (red: >= PW floats of shared memory); every thread gets the sum.
FQ_DEV float block_sum_p(float v, float* red) {
    v = warp_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < PW; ++w) t += red[w];
    return t;
}

// Stage the activation vector (times the norm gain) into shared memory in the padded layout
// of FMT; returns 1/rms (1 without a norm).  src == null: the embedding row of `tok` from
// `emb`, which CTA 0 also writes to x_out.
template <int FMT>
FQ_DEV float stage_x(const float* src, int K, const float* gain, float eps, float* xs, float* xsum16, float* red,
                     const QMat* emb = nullptr, int64_t tok = 0, float* x_out = nullptr) {
    float ss = 0.f;
    for (int k = threadIdx.x * 4; k < K; k += PT * 4) {
        float4 v;
        if (src) {
            v = __ldcg(reinterpret_cast<const float4*>(src + k));
        } else {
            v.x = dequant_one(*emb, tok, k);
            v.y = dequant_one(*emb, tok, k + 1);
            v.z = dequant_one(*emb, tok, k + 2);
            v.w = dequant_one(*emb, tok, k + 3);
            if (x_out && blockIdx.x == 0) *reinterpret_cast<float4*>(x_out + k) = v;
        }
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        if (gain) {
            const float4 g = *reinterpret_cast<const float4*>(gain + k);
            v.x *= g.x; v.y *= g.y; v.z *= g.z; v.w *= g.w;
        }
        *reinterpret_cast<float4*>(xs + xpad<FMT>(k)) = v;
    }
    const float tot = block_sum_p(ss, red);
    if (FMT == FMT_Q4_K) {
        __syncthreads();
        for (int j = threadIdx.x; j < K / 16; j += PT) {
            const float4* p = reinterpret_cast<const float4*>(xs + xpad<FMT>(16 * j));
            float s = 0.f;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float4 v = p[t];
                s += v.x + v.y + v.z + v.w;
            }
            xsum16[j] = s;
        }
    }
    __syncthreads();
    return gain ? rsqrtf(tot / (float)K + eps) : 1.f;
}

struct Epi {
    int kind;                     // EPI_STORE / EPI_ADD / EPI_SWIGLU / EPI_LOGITS
    float* y;                     // output (LOGITS: may be null)
    float inv;                    // 1/rms of the staged input
    unsigned long long* best;     // shared: LOGITS argmax key of this CTA
};

template <int R>
FQ_DEV void finish_rows(const Epi& e, int row_base, int r1, float (&v)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] *= e.inv;
    if (e.kind == EPI_SWIGLU) {
#pragma unroll
        for (int r = 0; r + 1 < R; r += 2)
            if (row_base + r + 1 < r1) e.y[(row_base + r) >> 1] = silu(v[r]) * v[r + 1];
        return;
    }
    unsigned long long kb = 0ull;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int row = row_base + r;
        if (row >= r1) continue;
        if (e.kind == EPI_ADD) e.y[row] = __ldcg(&e.y[row]) + v[r];
        else if (e.y) e.y[row] = v[r];
        if (e.kind == EPI_LOGITS) {
            const unsigned long long k = argmax_key(v[r], (uint32_t)row);
            kb = k > kb ? k : kb;
        }
    }
    if (e.kind == EPI_LOGITS && kb) atomicMax(e.best, kb);
}

// Partial dot of one unit of one row with the staged activations, read from shared memory
// as they are consumed (the weights arrive from L2, so fewer loads need to be in flight than
// in the stand-alone GEMV and the registers go to rows instead).
template <int FMT>
FQ_DEV float dot_unit(const Raw& r, int u, const float* xs, const float* xsum16) {
    if constexpr (FMT == FMT_Q8_0) {
        const float4* p = reinterpret_cast<const float4*>(xs + xpad<FMT>(u * 16));
        const uint32_t w[4] = {r.q.x, r.q.y, r.q.z, r.q.w};
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float f[4];
            s8x4_to_f32(w[i], f);
            const float4 x = p[i];
            acc = fmaf(f[0], x.x, acc);
            acc = fmaf(f[1], x.y, acc);
            acc = fmaf(f[2], x.z, acc);
            acc = fmaf(f[3], x.w, acc);
        }
        return h2f(r.sc) * acc;
    } else {
        const int c = u & 3;
        const int e0 = (u >> 2) * 256 + 64 * c;
        const float4* plo = reinterpret_cast<const float4*>(xs + xpad<FMT>(e0));
        const float4* phi = reinterpret_cast<const float4*>(xs + xpad<FMT>(e0 + 32));
        const uint32_t w[8] = {r.q.x, r.q.y, r.q.z, r.q.w, r.q2.x, r.q2.y, r.q2.z, r.q2.w};
        // codes as 1 + q/128 (one byte permute each); sum q x recovered from the per-16 sums
        float slo = 0.f, shi = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lw = (w[i] & 0x0F0F0F0Fu) | 0x80808080u;
            const uint32_t hw = ((w[i] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;
            const float4 xl = plo[i], xh = phi[i];
            const float xla[4] = {xl.x, xl.y, xl.z, xl.w}, xha[4] = {xh.x, xh.y, xh.z, xh.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                slo = fmaf(__uint_as_float(__byte_perm(lw, 0x3F000000u, 0x7044u | (j << 8))), xla[j], slo);
                shi = fmaf(__uint_as_float(__byte_perm(hw, 0x3F000000u, 0x7044u | (j << 8))), xha[j], shi);
            }
        }
        const float d = h2f((unsigned short)(r.hdr.x & 0xFFFFu)), dmin = h2f((unsigned short)(r.hdr.x >> 16));
        const uint32_t W0 = r.hdr.y, W1 = r.hdr.z, W2 = r.hdr.w;
        uint32_t sc0, mn0, sc1, mn1;
        if (c < 2) {
            const uint32_t sh = 16u * c;
            sc0 = (W0 >> sh) & 63u; sc1 = (W0 >> (sh + 8)) & 63u;
            mn0 = (W1 >> sh) & 63u; mn1 = (W1 >> (sh + 8)) & 63u;
        } else {
            const uint32_t sh = 16u * (c - 2);
            const uint32_t a = W2 >> sh, b0 = W0 >> sh, b1 = W1 >> sh;
            sc0 = (a & 15u) | ((b0 >> 2) & 48u); sc1 = ((a >> 8) & 15u) | ((b0 >> 10) & 48u);
            mn0 = ((a >> 4) & 15u) | ((b1 >> 2) & 48u); mn1 = ((a >> 12) & 15u) | ((b1 >> 10) & 48u);
        }
        const float s_lo = xsum16[e0 >> 4] + xsum16[(e0 >> 4) + 1];
        const float s_hi = xsum16[(e0 >> 4) + 2] + xsum16[(e0 >> 4) + 3];
        return d * (float)sc0 * 128.f * (slo - s_lo) - dmin * (float)mn0 * s_lo + d * (float)sc1 * 128.f * (shi - s_hi) -
               dmin * (float)mn1 * s_hi;
    }
}

// Rows [r0, r1) of W times the staged activations.  Work items are (group of R rows, K part);
// the K parts of a group are added in shared memory.
template <int FMT>
FQ_DEV void gemv_rows(const QMat& W, int r0, int r1, const float* xs, const float* xsum16, const Epi& e, float* red) {
    constexpr int R = FMT == FMT_Q4_K ? 2 : 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_units = W.K / Unit<FMT>::ELEMS;
    const int nrows = r1 - r0;
    const int ngroups = nrows > 0 ? (nrows + R - 1) / R : 0;
    int ks = 1;
    while (ks < 8 && ngroups * ks * 2 <= PW && n_units / (ks * 2) >= 16) ks *= 2;
    const int items = ngroups * ks;
    const int upp = (n_units + ks - 1) / ks;
    for (int it = warp; it < items; it += PW) {
        const int grp = it / ks, kp = it % ks;
        const int row_base = r0 + grp * R;
        const int u_begin = kp * upp, u_end = min(n_units, u_begin + upp);
        float acc[R];
        bool row_ok[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            acc[r] = 0.f;
            row_ok[r] = row_base + r < r1;
        }
        for (int u = u_begin + lane; u < u_end; u += 32) {
            Raw q[R];
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (row_ok[r]) q[r] = load_unit<FMT>(W, row_base + r, u);
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (row_ok[r]) acc[r] += dot_unit<FMT>(q[r], u, xs, xsum16);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = warp_sum(acc[r]);
        if (ks == 1) {
            if (lane == 0) finish_rows<R>(e, row_base, r1, acc);
        } else if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) red[it * R + r] = acc[r];
        }
    }
    if (ks > 1) {
        __syncthreads();
        for (int grp = threadIdx.x; grp < ngroups; grp += PT) {
            float v[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                v[r] = 0.f;
                for (int kp = 0; kp < ks; ++kp) v[r] += red[(grp * ks + kp) * R + r];
            }
            finish_rows<R>(e, r0 + grp * R, r1, v);
        }
    }
}

// stage + rows for one projection phase, dispatched on the matrix format (not inlined: the
// phases get their registers allocated separately)
__device__ __noinline__ void proj_phase(const QMat& W, bool pairs, const float* src, int K, const float* gain, float eps, int kind,
                       float* y, float* smem, unsigned long long* best, const QMat* emb = nullptr, int64_t tok = 0,
                       float* x_out = nullptr) {
    int r0, r1;
    row_range(W.N, blockIdx.x, gridDim.x, pairs, r0, r1);
    float* red = smem;                       // [PW * 8]
    float* xs = smem + PW * 8;
    if (W.fmt == FMT_Q4_K) {
        float* xsum16 = xs + xpad_len<FMT_Q4_K>(K);
        const float inv = stage_x<FMT_Q4_K>(src, K, gain, eps, xs, xsum16, red, emb, tok, x_out);
        gemv_rows<FMT_Q4_K>(W, r0, r1, xs, xsum16, Epi{kind, y, inv, best}, red);
    } else {
        const float inv = stage_x<FMT_Q8_0>(src, K, gain, eps, xs, nullptr, red, emb, tok, x_out);
        gemv_rows<FMT_Q8_0>(W, r0, r1, xs, nullptr, Epi{kind, y, inv, best}, red);
    }
}

FQ_DEV void prefetch_proj(const QMat& W, bool pairs, size_t cap = ~(size_t)0) {
    int r0, r1;
    row_range(W.N, blockIdx.x, gridDim.x, pairs, r0, r1);
    prefetch_rows(W, r0, r1, cap);
}

template <int KVT, int G>
__device__ __noinline__ void attn_phase(const PersistArgs& a, const PersistLayer& lw, int L, float* smem) {
    AttnArgs at = a.at;
    at.layer = L;
    at.q_norm = lw.q_norm;
    at.k_norm = lw.k_norm;
    const int tid = threadIdx.x, grp = tid >> 7;
    AttnSmem<G>* sm = reinterpret_cast<AttnSmem<G>*>(smem) + grp;
    const int n_units = at.Hkv * at.splits;
    for (int u = blockIdx.x * AG + grp; u < n_units; u += gridDim.x * AG)
        attn_unit<KVT, G>(at, u % at.splits, u / at.splits, 0, tid & 127, *sm, [grp] { named_sync(1 + grp); });
}

template <int KVT, int G>
__global__ void __launch_bounds__(PT, 1) persist_kernel(const __grid_constant__ PersistArgs a) {
    extern __shared__ __align__(16) float smem[];
    __shared__ unsigned long long best;
    const int tid = threadIdx.x;
    const int kvb = KVT == 1 ? 2 : 4;
    const SeqState ss = a.at.st->seq[0];
    const int64_t tok = (ss.token >= 0 && ss.token < a.emb.N) ? ss.token : 0;
    if (tid == 0) best = 0ull;
    constexpr size_t LM_PREFETCH = 64 * 1024;   // per CTA: the LM head is far larger than L2

    // phases of layer 0 start cold
    prefetch_proj(a.layers[0].qkv, false);
    prefetch_kv(a.at, 0, kvb);
    prefetch_proj(a.layers[0].o, false);

    for (int L = 0; L < a.n_layers; ++L) {
        const PersistLayer& lw = a.layers[L];
        const bool last = L + 1 == a.n_layers;
        // ---- P1: RMSNorm + QKV (layer 0 reads the embedding row)
        proj_phase(lw.qkv, false, L == 0 ? nullptr : a.x, a.H, lw.attn_norm, a.eps, EPI_STORE, a.qkv, smem, &best,
                   &a.emb, tok, a.x);
        prefetch_proj(lw.gate_up, true);
        if (!grid_sync(a.bar, a.err)) return;

        // ---- P2: attention (QK-norm, RoPE, KV append, split-K, merge by the last unit)
        attn_phase<KVT, G>(a, lw, L, smem);
        prefetch_proj(lw.down, false);
        if (!grid_sync(a.bar, a.err)) return;

        // ---- P3: O projection + residual
        proj_phase(lw.o, false, a.attn, a.Hq * HEAD_DIM, nullptr, a.eps, EPI_ADD, a.x, smem, &best);
        if (!last) prefetch_proj(a.layers[L + 1].qkv, false);
        else if (a.logits) prefetch_proj(a.out, false, LM_PREFETCH);
        if (!grid_sync(a.bar, a.err)) return;

        // ---- P4: RMSNorm + gate_up + SwiGLU
        proj_phase(lw.gate_up, true, a.x, a.H, lw.ffn_norm, a.eps, EPI_SWIGLU, a.h, smem, &best);
        if (!last) prefetch_kv(a.at, L + 1, kvb);
        if (!grid_sync(a.bar, a.err)) return;

        // ---- P5: down + residual
        proj_phase(lw.down, false, a.h, a.F, nullptr, a.eps, EPI_ADD, a.x, smem, &best);
        if (!last) prefetch_proj(a.layers[L + 1].o, false);
        if (!grid_sync(a.bar, a.err)) return;
    }
    if (!a.logits) return;

    // ---- final RMSNorm + LM head (+ argmax keys for greedy decoding)
    proj_phase(a.out, false, a.x, a.H, a.out_norm, a.eps, a.greedy ? EPI_LOGITS : EPI_STORE, a.logits, smem, &best);
    if (!a.greedy) return;
    __syncthreads();
    if (tid == 0) {
        StepState* st = const_cast<StepState*>(a.at.st);
        if (best) atomicMax(&st->keys[0], best);
        __threadfence();
        if (atomicAdd(a.lm_ticket, 1u) == gridDim.x - 1) {
            // every CTA's key is in: hand the token to the next step
            *a.lm_ticket = 0u;
            __threadfence();
            const unsigned long long k = atomicExch(&st->keys[0], 0ull);
            const uint32_t idx = argmax_key_index(k);
            const int32_t t = idx < (uint32_t)a.V ? (int32_t)idx : 0;
            st->seq[0].token = t;
            st->seq[0].pos += 1;
            if (st->tokens_out) st->tokens_out[st->step] = t;
            st->step += 1;
        }
    }
}

int g_sms_p = 0;
size_t g_optin_p = 0;

template <int KVT, int G>
size_t smem_bytes(const PersistArgs& a) {
    const int kmax = std::max(std::max(a.H, a.F), a.Hq * HEAD_DIM);
    const size_t gemv = (size_t)(PW * 8 + xpad_len<FMT_Q8_0>(kmax) + kmax / 16) * sizeof(float) + 64;
    const size_t att = (size_t)AG * sizeof(AttnSmem<G>);
    return std::max(gemv, att);
}

template <int KVT, int G>
bool launch_kg(const PersistArgs& a, cudaStream_t s) {
    const size_t smem = smem_bytes<KVT, G>(a);
    if (smem > g_optin_p) return false;
    cudaFuncSetAttribute(persist_kernel<KVT, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, persist_kernel<KVT, G>, PT, smem);
    if (occ < 1) return false;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g_sms_p);
    cfg.blockDim = dim3(PT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, persist_kernel<KVT, G>, a) == cudaSuccess;
}

template <int KVT>
bool launch_k(const PersistArgs& a, cudaStream_t s) {
    switch (a.Hq / a.Hkv) {
        case 1: return launch_kg<KVT, 1>(a, s);
        case 2: return launch_kg<KVT, 2>(a, s);
        case 4: return launch_kg<KVT, 4>(a, s);
        case 8: return launch_kg<KVT, 8>(a, s);
        default: return false;
    }
}

}  // namespace

void persist_prepare() {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms_p, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    g_optin_p = (size_t)optin - 1024;   // static shared memory of the kernel
}

int persist_ctas() { return g_sms_p; }

bool launch_persist(const PersistArgs& a, cudaStream_t s) {
    if (g_sms_p == 0) return false;
    return a.at.kv_type == KV_BF16 ? launch_k<1>(a, s) : launch_k<0>(a, s);
}

}  // namespace fq
