// Grouped causal attention of one new query row per sequence against its KvCache, as a
// split-K flash-decode (sm_103a CUDA cores, cached rows staged by bulk copies).
//
// The fucina runner page lists, for the .fused block style, half-rope QK-norm and grouped
// causal attention over the shared KvCache; section 14.1 fixes that a step appends the new
// K/V at pos == len.  One CTA (256 threads) owns (sequence b, kv head g, chunk s of the
// positions); the G = n_q / n_kv query heads of the group share every K/V row it reads.
//   * Cached rows [t0, pos) of the chunk arrive in tiles of 64 (bf16; 32 for f32) positions
//     through a 3-slot ring of 1-D bulk copies (cp.async.bulk, completion on an mbarrier),
//     issued before anything else: they depend on earlier steps only.
//   * q heads: RMSNorm with the learned gain, rotate-half RoPE at the absolute position
//     (cos/sin table), scaled by log2(e)/sqrt(128) for a base-2 softmax.  The CTA whose
//     chunk holds pos does the same for k, rounds k and v to the cache dtype, writes them
//     at pos and uses the rounded values for that position itself.
//   * Scores: 8 lanes per position, each with 16 of the 128 dimensions (two 16-byte reads
//     that tile a 128-byte row segment: conflict-free), 3 shuffles to reduce.
//   * Online softmax per head (one warp per head) over each tile, then V accumulation with
//     threads over (pair of dimensions, one of 4 position groups).
//   * Partial (m, l, o) per chunk; the last CTA of a (sequence, kv head) to finish (atomic
//     ticket, no waiting) merges the chunks and writes the head outputs.
// The ring's waits are bounded: a copy that never lands sets the error word instead of
// hanging the kernel.

#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

#include <algorithm>

namespace fq {

namespace {

constexpr int A_THREADS = 256;
constexpr int A_WARPS = A_THREADS / 32;
constexpr int A_STAGES = 3;
constexpr float LOG2E_A = 1.4426950408889634f;

template <int KVT> struct KvT;
template <> struct KvT<0> { using T = float; static constexpr int TILE = 32; };
template <> struct KvT<1> { using T = uint16_t; static constexpr int TILE = 64; };

template <int KVT, int G>
struct ASmem {
    using T = typename KvT<KVT>::T;
    static constexpr int TILE = KvT<KVT>::TILE;
    static constexpr int ROW = HEAD_DIM * (int)sizeof(T);        // bytes per cached row
    static constexpr int SLOT = 2 * TILE * ROW;                   // K tile | V tile
    // ring first (16-byte aligned slots); the final reduction reuses it
    static constexpr int OFF_Q = A_STAGES * SLOT;                 // float q[G][128]
    static constexpr int OFF_S = OFF_Q + G * HEAD_DIM * 4;        // float s[G][TILE]
    static constexpr int OFF_KN = OFF_S + G * TILE * 4;           // float kn[128], vn[128]
    static constexpr int OFF_ML = OFF_KN + 2 * HEAD_DIM * 4;      // float m[G], l[G], corr[G]
    static constexpr int OFF_BAR = (OFF_ML + 3 * G * 4 + 15) & ~15;   // uint64 full[A_STAGES]
    static constexpr int OFF_MISC = OFF_BAR + A_STAGES * 8;       // int is_last; float hM[G], hL[G]
    static constexpr int BYTES = OFF_MISC + 16 + 2 * G * 4;
    static_assert(4 * G * HEAD_DIM * 4 <= A_STAGES * SLOT, "reduction must fit in the ring");
};

FQ_DEV float bf_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
FQ_DEV float bf_hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// normalise + rope one head held as 4 dims per lane (dims 4l..4l+3) by one warp
FQ_DEV void norm_rope4(float v[4], const float* gain, const float2* rope_row, float eps, int lane) {
    float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / (float)HEAD_DIM + eps);
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = v[j] * inv * gain[4 * lane + j];
    // rotate-half pairing (i, i + 64): lane l < 16 holds i = 4l+j, lane l + 16 holds i + 64
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float partner = __shfl_xor_sync(0xFFFFFFFFu, v[j], 16);
        const float2 cs = rope_row[(4 * lane + j) & 63];
        v[j] = lane < 16 ? v[j] * cs.x - partner * cs.y : partner * cs.y + v[j] * cs.x;
    }
}

template <int KVT, int G>
__global__ void __launch_bounds__(A_THREADS, 2) attn_kernel(const AttnArgs a) {
    using S = ASmem<KVT, G>;
    using T = typename S::T;
    constexpr int TILE = S::TILE;
    extern __shared__ __align__(128) uint8_t sm[];
    float* qs = reinterpret_cast<float*>(sm + S::OFF_Q);
    float* sc = reinterpret_cast<float*>(sm + S::OFF_S);
    float* kn = reinterpret_cast<float*>(sm + S::OFF_KN);
    float* vn = kn + HEAD_DIM;
    float* mh = reinterpret_cast<float*>(sm + S::OFF_ML);
    float* lh = mh + G;
    float* corr = lh + G;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + S::OFF_BAR);
    int* is_last = reinterpret_cast<int*>(sm + S::OFF_MISC);
    float* hM = reinterpret_cast<float*>(sm + S::OFF_MISC + 16);
    float* hL = hM + G;

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const SeqState ss = a.st->seq[b];
    const int pos = ss.pos, T_len = pos + 1;
    const int n_act = (T_len + a.chunk - 1) / a.chunk;
    if (s >= n_act) return;
    const int t0 = s * a.chunk, t1 = min(T_len, t0 + a.chunk);
    const int nt = (t1 - t0 + TILE - 1) / TILE;
    const size_t head_off = ((size_t)a.layer * a.Hkv + g) * (size_t)ss.cap * HEAD_DIM;
    const T* Kc = reinterpret_cast<const T*>(ss.k) + head_off;
    const T* Vc = reinterpret_cast<const T*>(ss.v) + head_off;

    // ---- cached rows (written by earlier steps) go out first
    auto issue = [&](int i) {
        const int tb = t0 + i * TILE;
        const int nr = max(0, min(tb + TILE, pos) - tb);   // cached rows of the tile (pos excluded)
        uint8_t* slot = sm + (size_t)(i % A_STAGES) * S::SLOT;
        mbar_arrive_expect_tx(&full[i % A_STAGES], (uint32_t)(2 * nr * S::ROW));
        if (nr > 0) {
            bulk_g2s(slot, Kc + (size_t)tb * HEAD_DIM, (uint32_t)(nr * S::ROW), &full[i % A_STAGES]);
            bulk_g2s(slot + TILE * S::ROW, Vc + (size_t)tb * HEAD_DIM, (uint32_t)(nr * S::ROW), &full[i % A_STAGES]);
        }
    };
    if (tid == 0) {
        for (int i = 0; i < A_STAGES; ++i) mbar_init(&full[i], 1);
        mbar_fence_init();
        for (int i = 0; i < min(nt, A_STAGES); ++i) issue(i);
    }
    pdl_trigger();
    pdl_wait();

    // ---- q heads of the group (and, in the chunk holding pos, the new k and v)
    const float* qkv = a.qkv + (size_t)b * a.qkv_stride;
    const float2* rope_row = a.rope + (size_t)pos * (HEAD_DIM / 2);
    const float qscale = LOG2E_A * rsqrtf((float)HEAD_DIM);
    const bool owns_new = (s == n_act - 1);
    for (int w = warp; w < G + (owns_new ? 2 : 0); w += A_WARPS) {
        if (w < G) {
            const int h = g * G + w;
            const float4 raw = __ldcg(reinterpret_cast<const float4*>(qkv + (size_t)h * HEAD_DIM + 4 * lane));
            float v[4] = {raw.x, raw.y, raw.z, raw.w};
            norm_rope4(v, a.q_norm, rope_row, a.eps, lane);
            *reinterpret_cast<float4*>(qs + w * HEAD_DIM + 4 * lane) =
                make_float4(v[0] * qscale, v[1] * qscale, v[2] * qscale, v[3] * qscale);
        } else {
            const bool isk = w == G;
            T* dst = const_cast<T*>(isk ? Kc : Vc) + (size_t)pos * HEAD_DIM;
            const float* src = qkv + (size_t)(a.Hq + (isk ? 0 : a.Hkv) + g) * HEAD_DIM;
            const float4 raw = __ldcg(reinterpret_cast<const float4*>(src + 4 * lane));
            float v[4] = {raw.x, raw.y, raw.z, raw.w};
            if (isk) norm_rope4(v, a.k_norm, rope_row, a.eps, lane);
            float* keep = isk ? kn : vn;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (KVT == 1) {
                    const __nv_bfloat16 hb = __float2bfloat16_rn(v[j]);
                    dst[4 * lane + j] = __bfloat16_as_ushort(hb);
                    keep[4 * lane + j] = __bfloat162float(hb);
                } else {
                    dst[4 * lane + j] = v[j];
                    keep[4 * lane + j] = v[j];
                }
            }
        }
    }
    if (tid < G) {
        mh[tid] = -INFINITY;
        lh[tid] = 0.f;
    }
    __syncthreads();

    // thread roles for V: dims 2dp, 2dp+1 over positions j = 4 jj + pg
    const int dp = tid & 63, pg = tid >> 6;
    float acc[G][2];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h][0] = acc[h][1] = 0.f;
    const int l8 = lane & 7, grp = lane >> 3;

    for (int i = 0; i < nt; ++i) {
        const int st = i % A_STAGES;
        if (!mbar_wait(&full[st], (uint32_t)(i / A_STAGES) & 1u) && lane == 0 && a.err) atomicOr(a.err, 128u);
        const uint8_t* Kt = sm + (size_t)st * S::SLOT;
        const uint8_t* Vt = Kt + TILE * S::ROW;
        const int tb = t0 + i * TILE;
        const int nv = min(TILE, t1 - tb);

        // ---- scores: position j = 32 r + 4 warp + grp (r < TILE / 32), lane l8 holds dims
        // 8 l8..8 l8+7 and 64 + 8 l8..
#pragma unroll 1
        for (int r = 0; r < TILE / 32; ++r) {
            const int j = 32 * r + 4 * warp + grp;
            const bool valid = j < nv;
            const bool fresh = tb + j == pos;
            float kf[16];
            if (fresh) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    kf[e] = kn[8 * l8 + e];
                    kf[8 + e] = kn[64 + 8 * l8 + e];
                }
            } else if (valid) {
                if constexpr (KVT == 1) {
                    const uint4 w0 = *reinterpret_cast<const uint4*>(Kt + j * S::ROW + 16 * l8);
                    const uint4 w1 = *reinterpret_cast<const uint4*>(Kt + j * S::ROW + 128 + 16 * l8);
                    const uint32_t u[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        kf[2 * e] = bf_lo_f(u[e]);
                        kf[2 * e + 1] = bf_hi_f(u[e]);
                    }
                } else {
                    const float4* p0 = reinterpret_cast<const float4*>(Kt + j * S::ROW + 32 * l8);
                    const float4* p1 = reinterpret_cast<const float4*>(Kt + j * S::ROW + 256 + 32 * l8);
                    const float4 x0 = p0[0], x1 = p0[1], x2 = p1[0], x3 = p1[1];
                    kf[0] = x0.x; kf[1] = x0.y; kf[2] = x0.z; kf[3] = x0.w;
                    kf[4] = x1.x; kf[5] = x1.y; kf[6] = x1.z; kf[7] = x1.w;
                    kf[8] = x2.x; kf[9] = x2.y; kf[10] = x2.z; kf[11] = x2.w;
                    kf[12] = x3.x; kf[13] = x3.y; kf[14] = x3.z; kf[15] = x3.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) kf[e] = 0.f;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float4* q0 = reinterpret_cast<const float4*>(qs + h * HEAD_DIM + 8 * l8);
                const float4* q1 = reinterpret_cast<const float4*>(qs + h * HEAD_DIM + 64 + 8 * l8);
                const float4 a0 = q0[0], a1 = q0[1], b0 = q1[0], b1 = q1[1];
                float d0 = a0.x * kf[0], d1 = a0.y * kf[1];
                d0 = fmaf(a0.z, kf[2], d0); d1 = fmaf(a0.w, kf[3], d1);
                d0 = fmaf(a1.x, kf[4], d0); d1 = fmaf(a1.y, kf[5], d1);
                d0 = fmaf(a1.z, kf[6], d0); d1 = fmaf(a1.w, kf[7], d1);
                d0 = fmaf(b0.x, kf[8], d0); d1 = fmaf(b0.y, kf[9], d1);
                d0 = fmaf(b0.z, kf[10], d0); d1 = fmaf(b0.w, kf[11], d1);
                d0 = fmaf(b1.x, kf[12], d0); d1 = fmaf(b1.y, kf[13], d1);
                d0 = fmaf(b1.z, kf[14], d0); d1 = fmaf(b1.w, kf[15], d1);
                float d = d0 + d1;
                d += __shfl_xor_sync(0xFFFFFFFFu, d, 1);
                d += __shfl_xor_sync(0xFFFFFFFFu, d, 2);
                d += __shfl_xor_sync(0xFFFFFFFFu, d, 4);
                if (l8 == 0) sc[h * TILE + j] = valid ? d : -INFINITY;
            }
        }
        __syncthreads();

        // ---- online softmax over the tile, one warp per head
        if (warp < G) {
            const int h = warp;
            float v[TILE / 32];
            float mt = -INFINITY;
#pragma unroll
            for (int r = 0; r < TILE / 32; ++r) {
                v[r] = sc[h * TILE + 32 * r + lane];
                mt = fmaxf(mt, v[r]);
            }
            mt = warp_max(mt);
            const float mold = mh[h];
            const float mnew = fmaxf(mold, mt);
            const float c = mnew == -INFINITY ? 1.f : exp2f(mold - mnew);
            float psum = 0.f;
#pragma unroll
            for (int r = 0; r < TILE / 32; ++r) {
                const float p = v[r] == -INFINITY ? 0.f : exp2f(v[r] - mnew);
                sc[h * TILE + 32 * r + lane] = p;
                psum += p;
            }
            psum = warp_sum(psum);
            if (lane == 0) {
                lh[h] = lh[h] * c + psum;
                mh[h] = mnew;
                corr[h] = c;
            }
        }
        __syncthreads();

        // ---- V: acc = corr * acc + sum_j p_j v_j
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float c = corr[h];
            acc[h][0] *= c;
            acc[h][1] *= c;
        }
#pragma unroll 4
        for (int jj = 0; jj < TILE / 4; ++jj) {
            const int j = 4 * jj + pg;
            if (j >= nv) break;
            float v0, v1;
            if (tb + j == pos) {
                v0 = vn[2 * dp];
                v1 = vn[2 * dp + 1];
            } else if constexpr (KVT == 1) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(Vt + j * S::ROW + 4 * dp);
                v0 = bf_lo_f(w);
                v1 = bf_hi_f(w);
            } else {
                const float2 w = *reinterpret_cast<const float2*>(Vt + j * S::ROW + 8 * dp);
                v0 = w.x;
                v1 = w.y;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float p = sc[h * TILE + j];
                acc[h][0] = fmaf(p, v0, acc[h][0]);
                acc[h][1] = fmaf(p, v1, acc[h][1]);
            }
        }
        __syncthreads();   // the slot and the probabilities are free again
        if (tid == 0 && i + A_STAGES < nt) issue(i + A_STAGES);
    }

    // ---- the 4 position groups into o[h][d] (the ring is free: all copies were consumed)
    float* red = reinterpret_cast<float*>(sm);   // [4][G][128]
#pragma unroll
    for (int h = 0; h < G; ++h)
        *reinterpret_cast<float2*>(red + ((size_t)pg * G + h) * HEAD_DIM + 2 * dp) = make_float2(acc[h][0], acc[h][1]);
    __syncthreads();
    float* outb = a.out + (size_t)b * a.Hq * HEAD_DIM;
    for (int i = tid; i < G * HEAD_DIM; i += A_THREADS) {
        const int h = i / HEAD_DIM, d = i % HEAD_DIM;
        const float O = red[(0 * G + h) * HEAD_DIM + d] + red[(1 * G + h) * HEAD_DIM + d] +
                        red[(2 * G + h) * HEAD_DIM + d] + red[(3 * G + h) * HEAD_DIM + d];
        const int hq = g * G + h;
        if (n_act == 1) {
            outb[(size_t)hq * HEAD_DIM + d] = O / lh[h];
        } else {
            float* p = a.part + (((size_t)b * a.Hq + hq) * a.splits + s) * (HEAD_DIM + 2);
            if (d == 0) {
                p[0] = mh[h];
                p[1] = lh[h];
            }
            p[2 + d] = O;
        }
    }
    if (n_act == 1) return;

    // ---- last CTA of this (sequence, kv head) merges the chunks (atomic ticket, no waiting)
    __syncthreads();
    if (tid == 0) {
        __threadfence();                        // release this CTA's partial (written above)
        uint32_t* ctr = a.counters + (size_t)b * a.Hkv + g;
        const uint32_t prev = atomicAdd(ctr, 1u);
        *is_last = (prev == (uint32_t)(n_act - 1));
        if (*is_last) *ctr = 0u;                // every chunk has arrived: re-arm for the next use
    }
    __syncthreads();
    if (!*is_last) return;
    __threadfence();
    // per-chunk weights exp2(m - M) / L in shared memory (the ring), then each thread sums
    // the chunks' o[d] for its (head, dimension) with independent loads
    float* wgt = red;                           // [G][n_act]
    const bool fits = (size_t)G * n_act * 4 <= (size_t)A_STAGES * S::SLOT;
    if (fits) {
        for (int i = tid; i < G * n_act; i += A_THREADS) {
            const int h = i / n_act, c = i % n_act;
            wgt[i] = __ldcg(a.part + (((size_t)b * a.Hq + g * G + h) * a.splits + c) * (HEAD_DIM + 2));
        }
        __syncthreads();
        if (tid < G) {
            float M = -INFINITY, L = 0.f;
            for (int c = 0; c < n_act; ++c) M = fmaxf(M, wgt[tid * n_act + c]);
            for (int c = 0; c < n_act; ++c) {
                const float* p = a.part + (((size_t)b * a.Hq + g * G + tid) * a.splits + c) * (HEAD_DIM + 2);
                L += __ldcg(p + 1) * exp2f(wgt[tid * n_act + c] - M);
            }
            hM[tid] = M;
            hL[tid] = 1.f / L;
        }
        __syncthreads();
        for (int i = tid; i < G * n_act; i += A_THREADS) wgt[i] = exp2f(wgt[i] - hM[i / n_act]) * hL[i / n_act];
        __syncthreads();
    }
    for (int i = tid; i < G * HEAD_DIM; i += A_THREADS) {
        const int h = i / HEAD_DIM, d = i % HEAD_DIM;
        const int hq = g * G + h;
        const float* base = a.part + ((size_t)b * a.Hq + hq) * a.splits * (HEAD_DIM + 2);
        float O = 0.f;
        if (fits) {
            for (int c0 = 0; c0 < n_act; c0 += 8) {
                float v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    v[j] = c0 + j < n_act ? __ldcg(base + (size_t)(c0 + j) * (HEAD_DIM + 2) + 2 + d) : 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (c0 + j < n_act) O = fmaf(wgt[h * n_act + c0 + j], v[j], O);
            }
        } else {                                // very long caches: plain loop
            float M = -INFINITY, L = 0.f;
            for (int c = 0; c < n_act; ++c) M = fmaxf(M, __ldcg(base + (size_t)c * (HEAD_DIM + 2)));
            for (int c = 0; c < n_act; ++c) {
                const float* p = base + (size_t)c * (HEAD_DIM + 2);
                const float w = exp2f(__ldcg(p) - M);
                L += __ldcg(p + 1) * w;
                O += __ldcg(p + 2 + d) * w;
            }
            O /= L;
        }
        outb[(size_t)hq * HEAD_DIM + d] = O;
    }
}

template <int KVT, int G>
void launch_t(const AttnArgs& a, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.splits, a.Hkv, a.n);
    cfg.blockDim = dim3(A_THREADS);
    cfg.dynamicSmemBytes = ASmem<KVT, G>::BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaLaunchKernelEx(&cfg, attn_kernel<KVT, G>, a);
}

template <int KVT>
void launch_kv(const AttnArgs& a, cudaStream_t s, bool pdl) {
    switch (a.Hq / a.Hkv) {
        case 1: launch_t<KVT, 1>(a, s, pdl); break;
        case 2: launch_t<KVT, 2>(a, s, pdl); break;
        case 4: launch_t<KVT, 4>(a, s, pdl); break;
        case 8: launch_t<KVT, 8>(a, s, pdl); break;
        default: break;   // rejected at descriptor validation
    }
}

template <int KVT, int G>
void prepare_t() {
    cudaFuncSetAttribute(attn_kernel<KVT, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, ASmem<KVT, G>::BYTES);
}

}  // namespace

void attention_prepare() {
    prepare_t<0, 1>(); prepare_t<0, 2>(); prepare_t<0, 4>(); prepare_t<0, 8>();
    prepare_t<1, 1>(); prepare_t<1, 2>(); prepare_t<1, 4>(); prepare_t<1, 8>();
}

void launch_attention(const AttnArgs& a, cudaStream_t s, bool pdl) {
    if (a.kv_bf16) launch_kv<1>(a, s, pdl);
    else launch_kv<0>(a, s, pdl);
}

}  // namespace fq
