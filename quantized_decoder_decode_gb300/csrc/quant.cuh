// Decoding of the device-resident weight formats (ggml Q8_0 repacked into aligned planes,
// ggml Q4_K super-blocks as stored).  Shared by the GEMV kernels and the inspection /
// embedding kernels so that both read the bytes the same way.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace fq {

// byte i (0..15) of a 16-byte vector
FQ_DEV uint32_t byte_of(const uint4& v, int i) {
    uint32_t w = i < 4 ? v.x : i < 8 ? v.y : i < 12 ? v.z : v.w;
    return (w >> (8 * (i & 3))) & 0xFFu;
}

// Q4_K 6-bit (scale, min) of sub-block j; hdr = the block's first 16 bytes (d, dmin,
// then the 12 packed bytes s[0..11]).  j < 4: s[j] & 63, s[j+4] & 63.  j >= 4: low four
// bits from s[j+4] (scale in the low nibble, min in the high nibble), top two bits from
// bits 6-7 of s[j-4] (scale) and s[j] (min).
FQ_DEV void q4k_scale_min(const uint4& hdr, int j, uint32_t& sc, uint32_t& mn) {
    if (j < 4) {
        sc = byte_of(hdr, 4 + j) & 63u;
        mn = byte_of(hdr, 8 + j) & 63u;
    } else {
        uint32_t b = byte_of(hdr, 8 + j);
        sc = (b & 15u) | ((byte_of(hdr, j) >> 6) << 4);
        mn = (b >> 4) | ((byte_of(hdr, 4 + j) >> 6) << 4);
    }
}

// One weight as the f32 value it stands for (exact; for Q4_K (d sc) q - dmin mn with one
// rounding).  Used where single values are needed (embedding rows, inspection).
FQ_DEV float dequant_one(const QMat& W, int64_t row, int64_t k) {
    if (W.fmt == FMT_Q8_0) {
        int8_t q = (int8_t)W.q[row * W.K + k];
        return h2f(W.s[row * (W.K / 32) + k / 32]) * (float)q;
    }
    if (W.fmt == FMT_Q4_K) {
        const uint8_t* blk = W.q + row * (int64_t)(W.K / 256 * 144) + (k / 256) * 144;
        uint4 hdr = *reinterpret_cast<const uint4*>(blk);
        int e = (int)(k % 256), j = e / 32, c = j / 2, i = e % 32;
        uint32_t byte = blk[16 + 32 * c + i];
        uint32_t q = (j & 1) ? (byte >> 4) : (byte & 15u);
        uint32_t sc, mn;
        q4k_scale_min(hdr, j, sc, mn);
        float d = h2f((unsigned short)(hdr.x & 0xFFFFu)), dmin = h2f((unsigned short)(hdr.x >> 16));
        return fmaf(d * (float)sc, (float)q, -(dmin * (float)mn));
    }
    return reinterpret_cast<const float*>(W.q)[row * W.K + k];
}

// ---------------------------------------------------------------- GEMV units

// Q8_0 unit: 16 consecutive codes of one row (16 bytes) sharing one fp16 scale.
// Q4_K unit: one 32-byte nibble chunk c of a super-block = all 32 elements of sub-block 2c
// (low nibbles) and of sub-block 2c+1 (high nibbles), so a lane decodes one (scale, min)
// pair per 32 weights.
template <int FMT> struct Unit;
template <> struct Unit<FMT_Q8_0> { static constexpr int ELEMS = 16; };
template <> struct Unit<FMT_Q4_K> { static constexpr int ELEMS = 64; };
template <> struct Unit<FMT_F32> { static constexpr int ELEMS = 4; };

struct Raw {
    uint4 q;        // 16 bytes of codes (Q8_0; Q4_K first half of the chunk) or 4 floats (F32)
    uint4 q2;       // Q4_K: second 16 bytes of the chunk
    uint4 hdr;      // Q4_K: d, dmin, 12 scale bytes
    uint16_t sc;    // Q8_0 scale
};

template <int FMT>
FQ_DEV Raw load_unit(const QMat& W, int row, int u) {
    Raw r;
    if constexpr (FMT == FMT_Q8_0) {
        r.q = ld_stream16(W.q + (size_t)row * W.K + (size_t)u * 16);
        r.sc = ld_stream2(W.s + (size_t)row * (W.K / 32) + (u >> 1));
    } else if constexpr (FMT == FMT_Q4_K) {
        const uint8_t* blk = W.q + (size_t)row * ((size_t)W.K / 256 * 144) + (size_t)(u >> 2) * 144;
        const int c = u & 3;
        r.q = ld_stream16(blk + 16 + 32 * c);
        r.q2 = ld_stream16(blk + 32 + 32 * c);
        r.hdr = ld_stream16(blk);
    } else {
        r.q = ld_stream16((const float*)W.q + (size_t)row * W.K + (size_t)u * 4);
    }
    return r;
}

// Activations of one unit, loaded from shared memory once and shared by the warp's rows.
template <int FMT> struct XFrag { float v[Unit<FMT>::ELEMS]; };

// Staged activations carry 4 floats of padding after every 32 (Q8_0) or 64 (Q4_K) elements so
// that the 16-float runs read by the 8 lanes of one shared-memory phase start in distinct
// 16-byte bank groups (unpadded they all start at multiples of 256 or 64 bytes).
template <int FMT>
FQ_HD constexpr int xpad(int e) {
    return FMT == FMT_Q8_0 ? e + ((e >> 5) << 2) : FMT == FMT_Q4_K ? e + ((e >> 6) << 2) : e;
}
template <int FMT>
FQ_HD constexpr int xpad_len(int K) {
    return FMT == FMT_Q8_0 ? K + K / 8 : FMT == FMT_Q4_K ? K + K / 16 : K;
}

template <int FMT>
FQ_DEV void load_x(const float* xs, int u, XFrag<FMT>& f) {
    if constexpr (FMT == FMT_Q8_0) {
        const float4* p = reinterpret_cast<const float4*>(xs + xpad<FMT>(u * 16));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float4 t = p[i];
            f.v[4 * i] = t.x; f.v[4 * i + 1] = t.y; f.v[4 * i + 2] = t.z; f.v[4 * i + 3] = t.w;
        }
    } else if constexpr (FMT == FMT_Q4_K) {
        const int e0 = (u >> 2) * 256 + 64 * (u & 3);   // 32 low-nibble elements, then 32 high
        const float4* p = reinterpret_cast<const float4*>(xs + xpad<FMT>(e0));
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float4 t = p[i];
            f.v[4 * i] = t.x; f.v[4 * i + 1] = t.y; f.v[4 * i + 2] = t.z; f.v[4 * i + 3] = t.w;
        }
    } else {
        float4 t = reinterpret_cast<const float4*>(xs)[u];
        f.v[0] = t.x; f.v[1] = t.y; f.v[2] = t.z; f.v[3] = t.w;
    }
}

// Partial dot of one unit of one row with its activation fragment; xsum16: per-16 sums of
// the staged activations (Q4_K min terms).
template <int FMT>
FQ_DEV float dot_frag(const Raw& r, int u, const XFrag<FMT>& x, const float* xsum16) {
    if constexpr (FMT == FMT_Q8_0) {
        float f[16];
        s8x4_to_f32(r.q.x, f);
        s8x4_to_f32(r.q.y, f + 4);
        s8x4_to_f32(r.q.z, f + 8);
        s8x4_to_f32(r.q.w, f + 12);
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) acc = fmaf(f[i], x.v[i], acc);
        return h2f(r.sc) * acc;
    } else if constexpr (FMT == FMT_Q4_K) {
        const int c = u & 3;
        const int e0 = (u >> 2) * 256 + 64 * c;
        const uint32_t w[8] = {r.q.x, r.q.y, r.q.z, r.q.w, r.q2.x, r.q2.y, r.q2.z, r.q2.w};
        // each 4-bit code q becomes the float 1 + q/128 in one byte permute (byte 2 = 0x80 | q
        // under the exponent byte 0x3F); sum (1 + q/128) x = sum x + (sum q x) / 128, and the
        // per-16 sums of x recover sum q x below (about 4 of f32's 24 bits go to the cancellation)
        float slo = 0.f, shi = 0.f, slo2 = 0.f, shi2 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = (w[i] & 0x0F0F0F0Fu) | 0x80808080u;
            const uint32_t hi = ((w[i] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;
            float& al = (i & 1) ? slo2 : slo;
            float& ah = (i & 1) ? shi2 : shi;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                al = fmaf(__uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7044u | (j << 8))), x.v[4 * i + j], al);
                ah = fmaf(__uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7044u | (j << 8))), x.v[32 + 4 * i + j], ah);
            }
        }
        slo += slo2;
        shi += shi2;
        float d = h2f((unsigned short)(r.hdr.x & 0xFFFFu)), dmin = h2f((unsigned short)(r.hdr.x >> 16));
        // (scale, min) of sub-blocks 2c and 2c+1 straight from the three 32-bit scale words
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
        float d1 = d * (float)sc0, m1 = dmin * (float)mn0, d2 = d * (float)sc1, m2 = dmin * (float)mn1;
        // xsum16 holds per-16 sums; sub-blocks 2c and 2c+1 span two entries each
        const float s_lo = xsum16[e0 >> 4] + xsum16[(e0 >> 4) + 1];
        const float s_hi = xsum16[(e0 >> 4) + 2] + xsum16[(e0 >> 4) + 3];
        return d1 * 128.f * (slo - s_lo) - m1 * s_lo + d2 * 128.f * (shi - s_hi) - m2 * s_hi;
    } else {
        return __uint_as_float(r.q.x) * x.v[0] + __uint_as_float(r.q.y) * x.v[1] + __uint_as_float(r.q.z) * x.v[2] +
               __uint_as_float(r.q.w) * x.v[3];
    }
}

// One Q8_0 unit (16 codes, one scale) against up to NB activation rows: the codes become
// floats once and meet every row, read from shared memory as it is used.
template <int NB>
FQ_DEV void dot_q8_rows(const Raw& r, int u, const float* xs, int KP, int nb, float (&acc)[NB]) {
    float f[16];
    s8x4_to_f32(r.q.x, f);
    s8x4_to_f32(r.q.y, f + 4);
    s8x4_to_f32(r.q.z, f + 8);
    s8x4_to_f32(r.q.w, f + 12);
    const float d = h2f(r.sc);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        if (b >= nb) break;
        const float4* xp = reinterpret_cast<const float4*>(xs + (size_t)b * KP + xpad<FMT_Q8_0>(u * 16));
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 xv = xp[i];
            float& sa = (i & 1) ? s1 : s0;
            sa = fmaf(f[4 * i], xv.x, sa);
            sa = fmaf(f[4 * i + 1], xv.y, sa);
            sa = fmaf(f[4 * i + 2], xv.z, sa);
            sa = fmaf(f[4 * i + 3], xv.w, sa);
        }
        acc[b] = fmaf(d, s0 + s1, acc[b]);
    }
}

// One Q4_K unit against up to NB activation rows: each code becomes its float (1 + q/128, as
// in dot_frag) once and meets every row, read from shared memory as it is used.  xs: staged
// rows with stride KP; xsum16: their per-16 sums with stride K16; adds into acc[0..nb).
template <int NB>
FQ_DEV void dot_q4k_rows(const Raw& r, int u, const float* xs, int KP, const float* xsum16, int K16, int nb,
                         float (&acc)[NB]) {
    const int c = u & 3;
    const int e0 = (u >> 2) * 256 + 64 * c;
    const uint32_t w[8] = {r.q.x, r.q.y, r.q.z, r.q.w, r.q2.x, r.q2.y, r.q2.z, r.q2.w};
    float slo[NB], shi[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) slo[b] = shi[b] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = (w[i] & 0x0F0F0F0Fu) | 0x80808080u;
        const uint32_t hi = ((w[i] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;
        float fl[4], fh[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            fl[j] = __uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7044u | (j << 8)));
            fh[j] = __uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7044u | (j << 8)));
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b >= nb) break;
            const float4 xl = *reinterpret_cast<const float4*>(xs + (size_t)b * KP + xpad<FMT_Q4_K>(e0 + 4 * i));
            const float4 xh = *reinterpret_cast<const float4*>(xs + (size_t)b * KP + xpad<FMT_Q4_K>(e0 + 32 + 4 * i));
            slo[b] = fmaf(fl[0], xl.x, slo[b]); slo[b] = fmaf(fl[1], xl.y, slo[b]);
            slo[b] = fmaf(fl[2], xl.z, slo[b]); slo[b] = fmaf(fl[3], xl.w, slo[b]);
            shi[b] = fmaf(fh[0], xh.x, shi[b]); shi[b] = fmaf(fh[1], xh.y, shi[b]);
            shi[b] = fmaf(fh[2], xh.z, shi[b]); shi[b] = fmaf(fh[3], xh.w, shi[b]);
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
    const float d1 = d * (float)sc0 * 128.f, m1 = dmin * (float)mn0, d2 = d * (float)sc1 * 128.f,
                m2 = dmin * (float)mn1;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        if (b >= nb) break;
        const float* xq = xsum16 + (size_t)b * K16 + (e0 >> 4);
        const float s_lo = xq[0] + xq[1], s_hi = xq[2] + xq[3];
        acc[b] += d1 * (slo[b] - s_lo) - m1 * s_lo + d2 * (shi[b] - s_hi) - m2 * s_hi;
    }
}

}  // namespace fq
