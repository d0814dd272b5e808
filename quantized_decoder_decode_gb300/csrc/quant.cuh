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

}  // namespace fq
