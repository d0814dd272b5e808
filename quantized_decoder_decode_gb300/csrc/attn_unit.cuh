// Split-K attention unit shared by the stand-alone attention kernel and the persistent
// decode kernel: QK-norm, RoPE and the KV append of the new position fused in front of
// flash-decode over one chunk of cached positions, and the merge of the chunks by the last
// unit of a (sequence, kv head).  See attention.cu for the design.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace fq {

namespace {

constexpr int ATT_THREADS = 128;
constexpr int ATT_WARPS = 4;
constexpr float LOG2E = 1.4426950408889634f;

template <int KVT> struct KvElem;
template <> struct KvElem<0> { using T = float; };
template <> struct KvElem<1> { using T = uint16_t; };

// normalise + rope one head held as 4 dims per lane (dims 4l..4l+3) by one warp
FQ_DEV void norm_rope_head(float v[4], const float* gain, const float2* rope_row, float eps, int lane) {
    float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
    ss = warp_sum(ss);
    float inv = rsqrtf(ss / (float)HEAD_DIM + eps);
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = v[j] * inv * gain[4 * lane + j];
    // rotate-half pairing (i, i + 64): lane l < 16 holds i = 4l+j, lane l + 16 holds i + 64
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float partner = __shfl_xor_sync(0xFFFFFFFFu, v[j], 16);
        int i = (4 * lane + j) & 63;
        float2 cs = rope_row[i];
        v[j] = lane < 16 ? v[j] * cs.x - partner * cs.y : partner * cs.y + v[j] * cs.x;
    }
}

template <int KVT>
FQ_DEV void to_cache(float f, typename KvElem<KVT>::T* dst, float& rounded) {
    if constexpr (KVT == 1) {
        __nv_bfloat16 h = __float2bfloat16_rn(f);
        *dst = __bfloat16_as_ushort(h);
        rounded = __bfloat162float(h);
    } else {
        *dst = f;
        rounded = f;
    }
}

}  // namespace

// Shared memory of one attention unit (128 threads).
template <int G>
struct alignas(16) AttnSmem {
    float qs[G][HEAD_DIM];
    float kn[HEAD_DIM], vn[HEAD_DIM];
    float ps[ATT_WARPS][G][32];
    float mw[ATT_WARPS][G], lw[ATT_WARPS][G];
    float ow[ATT_WARPS][G][HEAD_DIM];
    float hM[G], hL[G];
    int is_last;
};

// One unit of the split-K attention: chunk s of the cached positions of (sequence b, kv
// head g), run by 128 threads (tid 0..127) that synchronise with sync().  The kernel below
// runs one unit per CTA; the persistent decode kernel runs several per CTA.
template <int KVT, int G, class Sync>
FQ_DEV void attn_unit(const AttnArgs& a, int s, int g, int b, int tid, AttnSmem<G>& sm, Sync sync) {
    using T = typename KvElem<KVT>::T;
    const int lane = tid & 31, warp = tid >> 5;
    const SeqState ss = a.st->seq[b];
    const int pos = ss.pos, T_len = pos + 1;
    const int n_act = (T_len + a.chunk - 1) / a.chunk;
    const int t0 = s * a.chunk, t1 = min(T_len, t0 + a.chunk);
    const size_t head_off = ((size_t)a.layer * a.Hkv + g) * (size_t)ss.cap * HEAD_DIM;
    const T* Kc = reinterpret_cast<const T*>(ss.k) + head_off;
    const T* Vc = reinterpret_cast<const T*>(ss.v) + head_off;
    if (s >= n_act) return;

    auto& qs = sm.qs;
    auto& kn = sm.kn;
    auto& vn = sm.vn;
    auto& ps = sm.ps;
    auto& mw = sm.mw;
    auto& lw = sm.lw;
    auto& ow = sm.ow;
    auto& hM = sm.hM;
    auto& hL = sm.hL;
    int& is_last = sm.is_last;

    const float* qkv = a.qkv + (size_t)b * a.qkv_stride;
    const float2* rope_row = a.rope + (size_t)pos * (HEAD_DIM / 2);
    const float qscale = LOG2E * rsqrtf((float)HEAD_DIM);

    // ---- the warp's first tile of K/V rows goes out before anything else: its latency is
    // then shared with the q prologue below.  Rows before pos were written by earlier steps.
    float m_run[G], l_run[G], acc[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[h][j] = 0.f;
    }
    constexpr int KW = KVT == 1 ? 16 : 32;      // 16-byte words per K row
    constexpr int VW = KVT == 1 ? 2 : 4;        // 32-bit words of one lane's 4 V dims
    constexpr int KPRE = KVT == 1 ? 16 : 1;     // K words held in registers across the prologue
    uint32_t vr[32][VW];
    uint4 kr[KPRE];
    auto issue = [&](int tb) {
        const int t = tb + lane;
        const int nvalid = min(32, t1 - tb);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int ti = tb + i;
            if (i < nvalid && ti != pos) {
                if constexpr (KVT == 1) {
                    uint2 w = ld_stream8(Vc + (size_t)ti * HEAD_DIM + 4 * lane);
                    vr[i][0] = w.x; vr[i][1] = w.y;
                } else {
                    uint4 w = ld_stream16(Vc + (size_t)ti * HEAD_DIM + 4 * lane);
                    vr[i][0] = w.x; vr[i][1] = w.y; vr[i][2] = w.z; vr[i][3] = w.w;
                }
            }
        }
        if constexpr (KVT == 1) {
            if (t < t1 && t != pos) {
                const char* krow = reinterpret_cast<const char*>(Kc + (size_t)t * HEAD_DIM);
#pragma unroll
                for (int c = 0; c < KPRE; ++c) kr[c] = ld_stream16(krow + 16 * c);
            } else {
#pragma unroll
                for (int c = 0; c < KPRE; ++c) kr[c] = make_uint4(0u, 0u, 0u, 0u);   // masked or fresh
            }
        }
    };
    int tb = t0 + warp * 32;
    if (tb < t1) issue(tb);

    // ---- q heads of the group: RMSNorm, rope, scale
    for (int hh = warp; hh < G; hh += ATT_WARPS) {
        int h = g * G + hh;
        float4 raw = __ldcg(reinterpret_cast<const float4*>(qkv + (size_t)h * HEAD_DIM + 4 * lane));
        float v[4] = {raw.x, raw.y, raw.z, raw.w};
        norm_rope_head(v, a.q_norm, rope_row, a.eps, lane);
#pragma unroll
        for (int j = 0; j < 4; ++j) qs[hh][4 * lane + j] = v[j] * qscale;
    }
    // ---- the chunk holding the new position appends k, v (rounded as stored)
    const bool owns_new = (s == n_act - 1);
    if (owns_new && warp < 2) {
        T* dst = const_cast<T*>(warp == 0 ? Kc : Vc) + (size_t)pos * HEAD_DIM;
        const float* src = qkv + (size_t)a.Hq * HEAD_DIM + (size_t)(warp == 0 ? 0 : a.Hkv) * HEAD_DIM +
                           (size_t)g * HEAD_DIM;
        float4 raw = __ldcg(reinterpret_cast<const float4*>(src + 4 * lane));
        float v[4] = {raw.x, raw.y, raw.z, raw.w};
        if (warp == 0) norm_rope_head(v, a.k_norm, rope_row, a.eps, lane);
        float* keep = warp == 0 ? kn : vn;
#pragma unroll
        for (int j = 0; j < 4; ++j) to_cache<KVT>(v[j], dst + 4 * lane + j, keep[4 * lane + j]);
    }
    sync();

    // ---- tiles of 32 positions, interleaved over warps; every K and V load of a tile is in
    // flight before its arithmetic starts
    for (bool first = true; tb < t1; tb += ATT_WARPS * 32, first = false) {
        if (!first) issue(tb);
        const int t = tb + lane;
        const bool valid = t < t1;
        const bool fresh = t == pos;            // the new position lives in shared memory
        const int nvalid = min(32, t1 - tb);
        float sc[G], sc2[G];                    // two partial sums per head (shorter chains)
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h] = sc2[h] = 0.f;
        // scores: one lane per position along its K row
        constexpr int KB = 16;                  // words per batch
#pragma unroll
        for (int c0 = 0; c0 < KW; c0 += KB) {
            uint4 kb[KB];
            if constexpr (KVT == 1) {
#pragma unroll
                for (int c = 0; c < KB; ++c) kb[c] = kr[c];
            } else {
                if (valid && !fresh) {
                    const char* krow = reinterpret_cast<const char*>(Kc + (size_t)t * HEAD_DIM);
#pragma unroll
                    for (int c = 0; c < KB; ++c) kb[c] = ld_stream16(krow + 16 * (c0 + c));
                } else {
#pragma unroll
                    for (int c = 0; c < KB; ++c) kb[c] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int c = 0; c < KB; ++c) {
                float kf[KVT == 1 ? 8 : 4];
                constexpr int EPW = KVT == 1 ? 8 : 4;   // elements per 16-byte word
                const int e0 = (c0 + c) * EPW;
                if (fresh) {
#pragma unroll
                    for (int e = 0; e < EPW; ++e) kf[e] = kn[e0 + e];
                } else if constexpr (KVT == 1) {
                    kf[0] = bf_lo(kb[c].x); kf[1] = bf_hi(kb[c].x); kf[2] = bf_lo(kb[c].y); kf[3] = bf_hi(kb[c].y);
                    kf[4] = bf_lo(kb[c].z); kf[5] = bf_hi(kb[c].z); kf[6] = bf_lo(kb[c].w); kf[7] = bf_hi(kb[c].w);
                } else {
                    kf[0] = __uint_as_float(kb[c].x); kf[1] = __uint_as_float(kb[c].y);
                    kf[2] = __uint_as_float(kb[c].z); kf[3] = __uint_as_float(kb[c].w);
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
#pragma unroll
                    for (int e = 0; e < EPW; e += 4) {
                        float4 q4 = *reinterpret_cast<const float4*>(&qs[h][e0 + e]);
                        float& acc_h = ((c + e / 4) & 1) ? sc2[h] : sc[h];
                        acc_h = fmaf(q4.x, kf[e], acc_h);
                        acc_h = fmaf(q4.y, kf[e + 1], acc_h);
                        acc_h = fmaf(q4.z, kf[e + 2], acc_h);
                        acc_h = fmaf(q4.w, kf[e + 3], acc_h);
                    }
                }
            }
        }
        // online softmax over the tile (base 2; q carries log2(e)/sqrt(D))
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h] += sc2[h];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float mt = warp_max(valid ? sc[h] : -INFINITY);
            float mnew = fmaxf(m_run[h], mt);
            float corr = exp2f(m_run[h] - mnew);
            float p = valid ? exp2f(sc[h] - mnew) : 0.f;
            l_run[h] = l_run[h] * corr + warp_sum(p);
            m_run[h] = mnew;
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[h][j] *= corr;
            ps[warp][h][lane] = p;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (i < nvalid) {
                float v4[4];
                if (tb + i == pos) {
                    float4 x = *reinterpret_cast<const float4*>(vn + 4 * lane);
                    v4[0] = x.x; v4[1] = x.y; v4[2] = x.z; v4[3] = x.w;
                } else if constexpr (KVT == 1) {
                    v4[0] = bf_lo(vr[i][0]); v4[1] = bf_hi(vr[i][0]); v4[2] = bf_lo(vr[i][1]); v4[3] = bf_hi(vr[i][1]);
                } else {
                    v4[0] = __uint_as_float(vr[i][0]); v4[1] = __uint_as_float(vr[i][1]);
                    v4[2] = __uint_as_float(vr[i][2]); v4[3] = __uint_as_float(vr[i][3]);
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float p = ps[warp][h][i];
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[h][j] = fmaf(p, v4[j], acc[h][j]);
                }
            }
        }
        __syncwarp();
    }

    // ---- merge the warps of the CTA
#pragma unroll
    for (int h = 0; h < G; ++h) {
        if (lane == 0) { mw[warp][h] = m_run[h]; lw[warp][h] = l_run[h]; }
        *reinterpret_cast<float4*>(&ow[warp][h][4 * lane]) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
    }
    sync();
    const int d = tid;   // one dimension per thread
    float* outb = a.out + (size_t)b * a.Hq * HEAD_DIM;
    for (int h = 0; h < G; ++h) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < ATT_WARPS; ++w) M = fmaxf(M, mw[w][h]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < ATT_WARPS; ++w) {
            float c = mw[w][h] == -INFINITY ? 0.f : exp2f(mw[w][h] - M);
            L += lw[w][h] * c;
            O += ow[w][h][d] * c;
        }
        const int hq = g * G + h;
        if (n_act == 1) {
            outb[(size_t)hq * HEAD_DIM + d] = O / L;
        } else {
            float* p = a.part + (((size_t)b * a.Hq + hq) * a.splits + s) * (HEAD_DIM + 2);
            if (d == 0) { p[0] = M; p[1] = L; }
            p[2 + d] = O;
        }
    }
    if (n_act == 1) return;

    // ---- last CTA of this (sequence, kv head) merges the chunks (atomic ticket, no waiting)
    sync();
    if (tid == 0) {
        __threadfence();                        // release this CTA's partial (written above)
        uint32_t* ctr = a.counters + (size_t)b * a.Hkv + g;
        uint32_t prev = atomicAdd(ctr, 1u);
        is_last = (prev == (uint32_t)(n_act - 1));
        if (is_last) *ctr = 0u;   // every chunk has arrived: re-arm for the next use
    }
    sync();
    if (!is_last) return;
    __threadfence();
    // (m, l) of every (head, chunk) into shared memory (reusing ow), then per-chunk weights
    // exp2(m - M) / L, then each thread d sums the chunks' o[d] with independent loads
    float* wm = &ow[0][0][0];                   // [G][n_act]
    float* wl = wm + G * n_act;
    const bool fits = 2 * G * n_act <= ATT_WARPS * G * HEAD_DIM;
    for (int h = 0; h < G; ++h) {
        const int hq = g * G + h;
        const float* base = a.part + ((size_t)b * a.Hq + hq) * a.splits * (HEAD_DIM + 2);
        if (!fits) {                            // very long caches: plain loop
            float M = -INFINITY;
            for (int c = 0; c < n_act; ++c) M = fmaxf(M, __ldcg(base + (size_t)c * (HEAD_DIM + 2)));
            float L = 0.f, O = 0.f;
            for (int c = 0; c < n_act; ++c) {
                const float* p = base + (size_t)c * (HEAD_DIM + 2);
                float w = exp2f(__ldcg(p) - M);
                L += __ldcg(p + 1) * w;
                O += __ldcg(p + 2 + d) * w;
            }
            outb[(size_t)hq * HEAD_DIM + d] = O / L;
        }
    }
    if (fits) {
        for (int i = tid; i < G * n_act; i += ATT_THREADS) {
            const int h = i / n_act, c = i % n_act;
            const float* p = a.part + (((size_t)b * a.Hq + g * G + h) * a.splits + c) * (HEAD_DIM + 2);
            wm[i] = __ldcg(p);
            wl[i] = __ldcg(p + 1);
        }
        sync();
        if (tid < G) {
            float M = -INFINITY, L = 0.f;
            for (int c = 0; c < n_act; ++c) M = fmaxf(M, wm[tid * n_act + c]);
            for (int c = 0; c < n_act; ++c) L += wl[tid * n_act + c] * exp2f(wm[tid * n_act + c] - M);
            hM[tid] = M;
            hL[tid] = 1.f / L;
        }
        sync();
        for (int i = tid; i < G * n_act; i += ATT_THREADS) wm[i] = exp2f(wm[i] - hM[i / n_act]) * hL[i / n_act];
        sync();
        for (int h = 0; h < G; ++h) {
            const int hq = g * G + h;
            const float* base = a.part + ((size_t)b * a.Hq + hq) * a.splits * (HEAD_DIM + 2) + 2 + d;
            float O = 0.f;
            for (int c0 = 0; c0 < n_act; c0 += 8) {
                float v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = c0 + j < n_act ? __ldcg(base + (size_t)(c0 + j) * (HEAD_DIM + 2)) : 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (c0 + j < n_act) O = fmaf(wm[h * n_act + c0 + j], v[j], O);
            }
            outb[(size_t)hq * HEAD_DIM + d] = O;
        }
    }
}

}  // namespace fq
