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
//   * Each warp owns 8 positions of every tile and keeps its own online-softmax state and
//     V accumulators (flash-decode with the warps as splits), so a tile needs no barrier but
//     the one that frees its ring slot.  Scores: 8 lanes per position, each with 16 of the
//     128 dimensions (two 16-byte reads that tile a 128-byte row segment: conflict-free),
//     q in registers, 3 shuffles to reduce.  V: lanes over dimensions (4 per lane).  The 8
//     warps merge at the end.  Groups of 8 query heads are split over two CTAs of 4 heads
//     (they read the same tiles, the second mostly from L2) so that every CTA fits the
//     registers of two CTAs per SM.
//   * Partial (m, l, o) per chunk; the last CTA of a (sequence, kv head) to finish (atomic
//     ticket, no waiting) merges the chunks and writes the head outputs.
// A q8_0 cache holds each row as 128 int8 codes plus four fp16 block scales (separate planes,
// both staged per tile).  Its scores take the integer q8 x q8 path the runner page names for
// that cache: q is quantised to Q8_0 blocks like a cached row, each lane forms 16-code
// integer dot products (dp4a) and scales them by d_q d_k; V rows are dequantised as they are
// accumulated.  The new k and v are quantised before they are stored and used.
// A step over several positions of one sequence (the all-logits step) runs the kernel twice:
// an append-only pass writes every row's new k/v, then the full pass reads them as cached rows
// (no store), so each row sees the rows before it.
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
template <> struct KvT<2> { using T = int8_t; static constexpr int TILE = 64; };   // Q8_0 codes

template <int KVT, int G>
struct ASmem {
    using T = typename KvT<KVT>::T;
    static constexpr int TILE = KvT<KVT>::TILE;
    static constexpr int ROW = HEAD_DIM * (int)sizeof(T);        // bytes per cached row
    static constexpr int SROW = KVT == 2 ? 8 : 0;                 // Q8_0: four fp16 block scales
    static constexpr int KPART = TILE * (ROW + SROW);             // codes/values, then scales
    static constexpr int SLOT = 2 * KPART;                        // K tile | V tile
    // ring first (16-byte aligned slots); the warps' final merge reuses it
    static constexpr int OFF_Q = A_STAGES * SLOT;                 // float4 q[G][4][8] (piece, lane group);
                                                                  // Q8_0: u32 codes[G][32], float d[G][4]
    static constexpr int OFF_KN = OFF_Q + G * HEAD_DIM * 4;       // float kn[128], vn[128]; Q8_0: kn =
                                                                  // u32 codes[32], float d[4]
    static constexpr int OFF_ML = OFF_KN + 2 * HEAD_DIM * 4;      // float mw[8][G], lw[8][G]
    static constexpr int OFF_P = (OFF_ML + 2 * A_WARPS * G * 4 + 15) & ~15;   // float pw[8][G][TILE/8 + 4]
    static constexpr int PSTRIDE = TILE / A_WARPS + 4;            // probabilities of a head, then its rescale
    static constexpr int OFF_BAR = (OFF_P + A_WARPS * G * PSTRIDE * 4 + 15) & ~15;   // uint64 full[A_STAGES]
    static constexpr int OFF_MISC = OFF_BAR + A_STAGES * 8;       // int is_last; float hM[G], hL[G]
    static constexpr int BYTES = OFF_MISC + 16 + 2 * G * 4;
    static_assert(A_WARPS * G * HEAD_DIM * 4 <= A_STAGES * SLOT, "warp merge must fit in the ring");
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

// G query heads per CTA (<= 4); hsplit CTAs share one kv head (G * hsplit = Hq / Hkv)
// Sum G per-head partials over the 8 lanes of a position group, transposing as it goes: the
// lane keeps half of its heads at each exchange, so after log2(G) exchanges it holds one
// head's value and the remaining exchanges are plain sums.  Returns the full sum for head
// *h of this lane (lanes l8 and l8 ^ (8 / G >> 1).. hold equal copies).
template <int G>
FQ_DEV float reduce8(const float (&d)[G], int l8, int& h) {
    if constexpr (G == 4) {
        const bool up = l8 & 4, up2 = l8 & 2;
        float k0 = up ? d[2] : d[0], k1 = up ? d[3] : d[1];
        const float s0 = up ? d[0] : d[2], s1 = up ? d[1] : d[3];
        k0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 4);
        k1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 4);
        float k = up2 ? k1 : k0;
        k += __shfl_xor_sync(0xFFFFFFFFu, up2 ? k0 : k1, 2);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 1);
        h = (up ? 2 : 0) + (up2 ? 1 : 0);
        return k;
    } else if constexpr (G == 2) {
        const bool up = l8 & 4;
        float k = up ? d[1] : d[0];
        k += __shfl_xor_sync(0xFFFFFFFFu, up ? d[0] : d[1], 4);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 2);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 1);
        h = up ? 1 : 0;
        return k;
    } else {
        float k = d[0];
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 4);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 2);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 1);
        h = 0;
        return k;
    }
}

template <int KVT, int G>
__global__ void __launch_bounds__(A_THREADS, 2) attn_kernel(const AttnArgs a, int hsplit) {
    using S = ASmem<KVT, G>;
    using T = typename S::T;
    constexpr int TILE = S::TILE;
    constexpr int PW = TILE / A_WARPS;                 // positions per warp per tile (8 or 4)
    extern __shared__ __align__(128) uint8_t sm[];
    float4* qp = reinterpret_cast<float4*>(sm + S::OFF_Q);   // [G][4 pieces][8 lane groups]
    float* kn = reinterpret_cast<float*>(sm + S::OFF_KN);
    float* vn = kn + HEAD_DIM;
    float* mw = reinterpret_cast<float*>(sm + S::OFF_ML);    // [8 warps][G]
    float* lw = mw + A_WARPS * G;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + S::OFF_BAR);
    int* is_last = reinterpret_cast<int*>(sm + S::OFF_MISC);
    float* hM = reinterpret_cast<float*>(sm + S::OFF_MISC + 16);
    float* hL = hM + G;

    const int s = blockIdx.x, g = blockIdx.y / hsplit, sub = blockIdx.y % hsplit, b = blockIdx.z;
    const int hq0 = (g * hsplit + sub) * G;            // first query head of this CTA
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const SeqState ss = a.st->seq[b];
    const int pos = ss.pos, T_len = pos + 1;
    const int n_act = (T_len + a.chunk - 1) / a.chunk;
    if (s >= n_act) return;
    const int t0 = s * a.chunk, t1 = min(T_len, t0 + a.chunk);
    const int nt = (t1 - t0 + TILE - 1) / TILE;
    const size_t head_row0 = (size_t)a.layer * a.Hkv + g;
    const size_t head_off = head_row0 * (size_t)ss.cap * HEAD_DIM;
    const T* Kc = reinterpret_cast<const T*>(ss.k) + head_off;
    const T* Vc = reinterpret_cast<const T*>(ss.v) + head_off;
    // Q8_0 scale planes [layer][kv head][cap rounded up to even][4] fp16 (16-byte aligned rows
    // pairs, so a tile's scales are one bulk copy)
    const size_t sc_off = head_row0 * (size_t)((ss.cap + 1) & ~1) * 4;
    const uint16_t* Ksc = reinterpret_cast<const uint16_t*>(ss.ks) + sc_off;
    const uint16_t* Vsc = reinterpret_cast<const uint16_t*>(ss.vs) + sc_off;

    // ---- cached rows (written by earlier steps) go out first
    auto issue = [&](int i) {
        const int tb = t0 + i * TILE;
        const int nr = max(0, min(tb + TILE, pos) - tb);   // cached rows of the tile (pos excluded)
        uint8_t* slot = sm + (size_t)(i % A_STAGES) * S::SLOT;
        // scales go in pairs of rows (16 bytes); an odd count ends at row pos, inside the plane
        const uint32_t sbytes = KVT == 2 ? (uint32_t)(((nr + 1) & ~1) * S::SROW) : 0u;
        mbar_arrive_expect_tx(&full[i % A_STAGES], (uint32_t)(2 * nr * S::ROW) + 2 * sbytes);
        if (nr > 0) {
            bulk_g2s(slot, Kc + (size_t)tb * HEAD_DIM, (uint32_t)(nr * S::ROW), &full[i % A_STAGES]);
            bulk_g2s(slot + S::KPART, Vc + (size_t)tb * HEAD_DIM, (uint32_t)(nr * S::ROW), &full[i % A_STAGES]);
            if constexpr (KVT == 2) {
                bulk_g2s(slot + TILE * S::ROW, Ksc + (size_t)tb * 4, sbytes, &full[i % A_STAGES]);
                bulk_g2s(slot + S::KPART + TILE * S::ROW, Vsc + (size_t)tb * 4, sbytes, &full[i % A_STAGES]);
            }
        }
    };
    // append-only pass (rows of one sequence in one step): just the new k/v of the chunk's owner
    const bool append_only = a.append_only != 0;
    if (append_only && s != n_act - 1) return;
    if (tid == 0 && !append_only) {
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
    const bool store = a.kv_store != 0 && sub == 0;   // the first CTA of the kv head stores, every one keeps
    for (int w = append_only ? G : warp; w < G + (owns_new ? 2 : 0); w += append_only ? 1 : A_WARPS) {
        if (append_only && w - G != warp) continue;     // warps 0 and 1: k and v
        if (w < G) {
            const int h = hq0 + w;
            const float4 raw = __ldcg(reinterpret_cast<const float4*>(qkv + (size_t)h * HEAD_DIM + 4 * lane));
            float v[4] = {raw.x, raw.y, raw.z, raw.w};
            norm_rope4(v, a.q_norm, rope_row, a.eps, lane);
            if constexpr (KVT == 2) {
                // q as Q8_0 blocks: codes of dims 4 lane..4 lane+3, block scale per 8 lanes
                unsigned short db;
                float d;
                const uint32_t code4 = q8_quant_lane4(v, db, d);
                reinterpret_cast<uint32_t*>(sm + S::OFF_Q)[w * 32 + lane] = code4;
                if ((lane & 7) == 0) reinterpret_cast<float*>(sm + S::OFF_Q + G * 128)[w * 4 + (lane >> 3)] = d;
            } else {
                // dims 4 lane..4 lane+3 = piece ((lane / 2) >= 8 ? 2 : 0) + (lane & 1) of lane group (lane / 2) % 8
                const int dim0 = 4 * lane, half = dim0 >= 64, grp8 = (dim0 % 64) / 8, piece = 2 * half + ((dim0 / 4) & 1);
                qp[(w * 4 + piece) * 8 + grp8] = make_float4(v[0] * qscale, v[1] * qscale, v[2] * qscale, v[3] * qscale);
            }
        } else {
            const bool isk = w == G;
            T* dst = const_cast<T*>(isk ? Kc : Vc) + (size_t)pos * HEAD_DIM;
            const float* src = qkv + (size_t)(a.Hq + (isk ? 0 : a.Hkv) + g) * HEAD_DIM;
            const float4 raw = __ldcg(reinterpret_cast<const float4*>(src + 4 * lane));
            float v[4] = {raw.x, raw.y, raw.z, raw.w};
            if (isk) norm_rope4(v, a.k_norm, rope_row, a.eps, lane);
            float* keep = isk ? kn : vn;
            if constexpr (KVT == 2) {
                unsigned short db;
                float d;
                const uint32_t code4 = q8_quant_lane4(v, db, d);
                if (store) {
                    reinterpret_cast<uint32_t*>(dst)[lane] = code4;
                    if ((lane & 7) == 0) const_cast<uint16_t*>(isk ? Ksc : Vsc)[(size_t)pos * 4 + (lane >> 3)] = db;
                }
                if (isk) {
                    reinterpret_cast<uint32_t*>(kn)[lane] = code4;
                    if ((lane & 7) == 0) kn[32 + (lane >> 3)] = d;
                } else {
                    float f[4];
                    s8x4_to_f32(code4, f);
#pragma unroll
                    for (int j = 0; j < 4; ++j) vn[4 * lane + j] = f[j] * d;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if constexpr (KVT == 1) {
                        const __nv_bfloat16 hb = __float2bfloat16_rn(v[j]);
                        if (store) dst[4 * lane + j] = __bfloat16_as_ushort(hb);
                        keep[4 * lane + j] = __bfloat162float(hb);
                    } else {
                        if (store) dst[4 * lane + j] = v[j];
                        keep[4 * lane + j] = v[j];
                    }
                }
            }
        }
    }
    if (append_only) return;
    __syncthreads();

    const int l8 = lane & 7, grp = lane >> 3;
    float4 qr[G][4];
    uint4 qw[G];           // Q8_0: codes of dims 16 l8..16 l8+15 and the scale of their block
    float qdl[G];
    if constexpr (KVT == 2) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            qw[h] = reinterpret_cast<const uint4*>(sm + S::OFF_Q)[h * 8 + l8];
            qdl[h] = reinterpret_cast<const float*>(sm + S::OFF_Q + G * 128)[h * 4 + (l8 >> 1)];
        }
    } else {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int pc = 0; pc < 4; ++pc) qr[h][pc] = qp[(h * 4 + pc) * 8 + l8];
    }
    // online softmax state of the lane's head (all lanes holding a head agree) and the V
    // accumulators of every head for dims 4 lane..4 lane+3
    float m_run[1] = {-INFINITY}, l_run[1] = {0.f}, acc[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = 0.f;
    int hl_own = 0;

    for (int i = 0; i < nt; ++i) {
        const int st = i % A_STAGES;
        if (!mbar_wait(&full[st], (uint32_t)(i / A_STAGES) & 1u) && lane == 0 && a.err) atomicOr(a.err, 128u);
        const uint8_t* Kt = sm + (size_t)st * S::SLOT;
        const uint8_t* Vt = Kt + S::KPART;
        const int tb = t0 + i * TILE;
        const int nv = min(TILE, t1 - tb);
        const int jw = warp * PW;                      // this warp's positions jw..jw+PW-1

        // ---- scores of the warp's positions: round r covers position jw + 4 r + grp; after the
        // reduction lane (grp, l8) holds the score of head hl for that position
        float sr[PW / 4];
        int hl = 0;
#pragma unroll
        for (int r = 0; r < PW / 4; ++r) {
            const int j = jw + 4 * r + grp;
            const bool valid = j < nv;
            if constexpr (KVT == 2) {
                // integer dot of 16 codes per lane, scaled by d_q d_k of their block
                uint4 kw = make_uint4(0u, 0u, 0u, 0u);
                float dk = 0.f;
                if (tb + j == pos) {
                    kw = reinterpret_cast<const uint4*>(kn)[l8];
                    dk = kn[32 + (l8 >> 1)];
                } else if (valid) {
                    kw = *reinterpret_cast<const uint4*>(Kt + j * S::ROW + 16 * l8);
                    dk = h2f(reinterpret_cast<const unsigned short*>(Kt + TILE * S::ROW)[j * 4 + (l8 >> 1)]);
                }
                float dd[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    int acc = __dp4a((int)kw.x, (int)qw[h].x, 0);
                    acc = __dp4a((int)kw.y, (int)qw[h].y, acc);
                    acc = __dp4a((int)kw.z, (int)qw[h].z, acc);
                    acc = __dp4a((int)kw.w, (int)qw[h].w, acc);
                    dd[h] = (float)acc * (qdl[h] * dk);
                }
                const float sc = reduce8<G>(dd, l8, hl) * qscale;
                hl_own = hl;
                sr[r] = valid ? sc : -INFINITY;
                continue;
            }
            float kf[16];
            if (tb + j == pos) {
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
            float dd[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float4* q4 = qr[h];
                float d0 = q4[0].x * kf[0], d1 = q4[0].y * kf[1];
                d0 = fmaf(q4[0].z, kf[2], d0); d1 = fmaf(q4[0].w, kf[3], d1);
                d0 = fmaf(q4[1].x, kf[4], d0); d1 = fmaf(q4[1].y, kf[5], d1);
                d0 = fmaf(q4[1].z, kf[6], d0); d1 = fmaf(q4[1].w, kf[7], d1);
                d0 = fmaf(q4[2].x, kf[8], d0); d1 = fmaf(q4[2].y, kf[9], d1);
                d0 = fmaf(q4[2].z, kf[10], d0); d1 = fmaf(q4[2].w, kf[11], d1);
                d0 = fmaf(q4[3].x, kf[12], d0); d1 = fmaf(q4[3].y, kf[13], d1);
                d0 = fmaf(q4[3].z, kf[14], d0); d1 = fmaf(q4[3].w, kf[15], d1);
                dd[h] = d0 + d1;
            }
            const float sc = reduce8<G>(dd, l8, hl);
            hl_own = hl;
            sr[r] = valid ? sc : -INFINITY;
        }

        // ---- online softmax of head hl over the warp's positions: the other 3 groups hold the
        // other positions of the same head (xor 8, 16)
        float mt = sr[0];
#pragma unroll
        for (int r = 1; r < PW / 4; ++r) mt = fmaxf(mt, sr[r]);
        mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 16));
        const float mold = m_run[0];              // lane-local state of head hl
        const float mnew = fmaxf(mold, mt);
        const float c = mnew == -INFINITY ? 1.f : exp2f(mold - mnew);
        float psum = 0.f;
        float pr[PW / 4];
#pragma unroll
        for (int r = 0; r < PW / 4; ++r) {
            pr[r] = sr[r] == -INFINITY ? 0.f : exp2f(sr[r] - mnew);
            psum += pr[r];
        }
        psum += __shfl_xor_sync(0xFFFFFFFFu, psum, 8);
        psum += __shfl_xor_sync(0xFFFFFFFFu, psum, 16);
        m_run[0] = mnew;
        l_run[0] = l_run[0] * c + psum;
        // probabilities [head][position] and the rescale of each head, per warp
        float* pw = reinterpret_cast<float*>(sm + S::OFF_P) + (size_t)warp * G * S::PSTRIDE;
        if ((l8 & (8 / G - 1)) == 0) {           // one writer per (group, head)
#pragma unroll
            for (int r = 0; r < PW / 4; ++r) pw[hl * S::PSTRIDE + 4 * r + grp] = pr[r];
            if (grp == 0) pw[hl * S::PSTRIDE + PW] = c;
        }
        __syncwarp();

        // ---- V: acc[h] = c_h acc[h] + sum_e p[h][e] v_e, lanes over dimensions
        if (__any_sync(0xFFFFFFFFu, mt != -INFINITY)) {
            float ph[G][PW];
#pragma unroll
            for (int h = 0; h < G; ++h) {
#pragma unroll
                for (int e = 0; e < PW; e += 4) {
                    const float4 t = *reinterpret_cast<const float4*>(pw + h * S::PSTRIDE + e);
                    ph[h][e] = t.x; ph[h][e + 1] = t.y; ph[h][e + 2] = t.z; ph[h][e + 3] = t.w;
                }
                const float ch = pw[h * S::PSTRIDE + PW];
#pragma unroll
                for (int d = 0; d < 4; ++d) acc[h][d] *= ch;
            }
#pragma unroll
            for (int e = 0; e < PW; ++e) {
                const int j = jw + e;
                if (j >= nv) break;
                float v4[4];
                if (tb + j == pos) {
                    const float4 x = *reinterpret_cast<const float4*>(vn + 4 * lane);
                    v4[0] = x.x; v4[1] = x.y; v4[2] = x.z; v4[3] = x.w;
                } else if constexpr (KVT == 2) {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(Vt + j * S::ROW + 4 * lane);
                    const float dv = h2f(reinterpret_cast<const unsigned short*>(Vt + TILE * S::ROW)[j * 4 + (lane >> 3)]);
                    s8x4_to_f32(w, v4);
#pragma unroll
                    for (int d = 0; d < 4; ++d) v4[d] *= dv;
                } else if constexpr (KVT == 1) {
                    const uint2 w = *reinterpret_cast<const uint2*>(Vt + j * S::ROW + 8 * lane);
                    v4[0] = bf_lo_f(w.x); v4[1] = bf_hi_f(w.x); v4[2] = bf_lo_f(w.y); v4[3] = bf_hi_f(w.y);
                } else {
                    const float4 x = *reinterpret_cast<const float4*>(Vt + j * S::ROW + 16 * lane);
                    v4[0] = x.x; v4[1] = x.y; v4[2] = x.z; v4[3] = x.w;
                }
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int d = 0; d < 4; ++d) acc[h][d] = fmaf(ph[h][e], v4[d], acc[h][d]);
            }
        } else {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float ch = pw[h * S::PSTRIDE + PW];
#pragma unroll
                for (int d = 0; d < 4; ++d) acc[h][d] *= ch;
            }
        }
        __syncwarp();
        __syncthreads();   // every warp is done with the slot
        if (tid == 0 && i + A_STAGES < nt) issue(i + A_STAGES);
    }

    // ---- merge the 8 warps (the ring is free: all copies were consumed)
    float* ow = reinterpret_cast<float*>(sm);   // [8][G][128]
    if ((l8 & (8 / G - 1)) == 0 && grp == 0) {   // one lane per head
        mw[warp * G + hl_own] = m_run[0];
        lw[warp * G + hl_own] = l_run[0];
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
        *reinterpret_cast<float4*>(ow + ((size_t)warp * G + h) * HEAD_DIM + 4 * lane) =
            make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
    __syncthreads();
    float* outb = a.out + (size_t)b * a.Hq * HEAD_DIM;
    for (int i = tid; i < G * HEAD_DIM; i += A_THREADS) {
        const int h = i / HEAD_DIM, d = i % HEAD_DIM;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < A_WARPS; ++w) M = fmaxf(M, mw[w * G + h]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < A_WARPS; ++w) {
            const float c = mw[w * G + h] == -INFINITY ? 0.f : exp2f(mw[w * G + h] - M);
            L += lw[w * G + h] * c;
            O += ow[((size_t)w * G + h) * HEAD_DIM + d] * c;
        }
        const int hq = hq0 + h;
        if (n_act == 1) {
            outb[(size_t)hq * HEAD_DIM + d] = O / L;
        } else {
            float* p = a.part + (((size_t)b * a.Hq + hq) * a.splits + s) * (HEAD_DIM + 2);
            if (d == 0) {
                p[0] = M;
                p[1] = L;
            }
            p[2 + d] = O;
        }
    }
    if (n_act == 1) return;

    // ---- last CTA of this (sequence, kv head) merges the chunks (atomic ticket, no waiting)
    __syncthreads();
    if (tid == 0) {
        __threadfence();                        // release this CTA's partial (written above)
        uint32_t* ctr = a.counters + (size_t)b * a.Hq + hq0;   // one counter per CTA group of heads
        const uint32_t prev = atomicAdd(ctr, 1u);
        *is_last = (prev == (uint32_t)(n_act - 1));
        if (*is_last) *ctr = 0u;                // every chunk has arrived: re-arm for the next use
    }
    __syncthreads();
    if (!*is_last) return;
    __threadfence();
    // per-chunk weights exp2(m - M) / L in shared memory (the ring), then each thread sums
    // the chunks' o[d] for its (head, dimension) with independent loads
    float* wgt = ow;                            // [G][n_act]
    const bool fits = (size_t)G * n_act * 4 <= (size_t)A_STAGES * S::SLOT;
    if (fits) {
        for (int i = tid; i < G * n_act; i += A_THREADS) {
            const int h = i / n_act, c = i % n_act;
            wgt[i] = __ldcg(a.part + (((size_t)b * a.Hq + hq0 + h) * a.splits + c) * (HEAD_DIM + 2));
        }
        __syncthreads();
        if (tid < G) {
            float M = -INFINITY, L = 0.f;
            for (int c = 0; c < n_act; ++c) M = fmaxf(M, wgt[tid * n_act + c]);
            for (int c = 0; c < n_act; ++c) {
                const float* p = a.part + (((size_t)b * a.Hq + hq0 + tid) * a.splits + c) * (HEAD_DIM + 2);
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
        const int hq = hq0 + h;
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
void launch_t(const AttnArgs& a, cudaStream_t s, bool pdl, int hsplit) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.splits, a.Hkv * hsplit, a.n);
    cfg.blockDim = dim3(A_THREADS);
    cfg.dynamicSmemBytes = ASmem<KVT, G>::BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaLaunchKernelEx(&cfg, attn_kernel<KVT, G>, a, hsplit);
}

template <int KVT>
void launch_kv(const AttnArgs& a, cudaStream_t s, bool pdl) {
    switch (a.Hq / a.Hkv) {
        case 1: launch_t<KVT, 1>(a, s, pdl, 1); break;
        case 2: launch_t<KVT, 2>(a, s, pdl, 1); break;
        case 4: launch_t<KVT, 4>(a, s, pdl, 1); break;
        case 8: launch_t<KVT, 4>(a, s, pdl, 2); break;
        default: break;   // rejected at descriptor validation
    }
}

template <int KVT, int G>
void prepare_t() {
    cudaFuncSetAttribute(attn_kernel<KVT, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, ASmem<KVT, G>::BYTES);
}

}  // namespace

void attention_prepare() {
    prepare_t<0, 1>(); prepare_t<0, 2>(); prepare_t<0, 4>();
    prepare_t<1, 1>(); prepare_t<1, 2>(); prepare_t<1, 4>();
    prepare_t<2, 1>(); prepare_t<2, 2>(); prepare_t<2, 4>();
}

void launch_attention(const AttnArgs& a, cudaStream_t s, bool pdl) {
    if (a.kv_type == KV_Q8_0) launch_kv<2>(a, s, pdl);
    else if (a.kv_type == KV_BF16) launch_kv<1>(a, s, pdl);
    else launch_kv<0>(a, s, pdl);
}

}  // namespace fq
