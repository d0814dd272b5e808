// Oracle for the Qwen3 single-token decode step -- TEST INFRASTRUCTURE ONLY.
//
// Plain f64 CPU code written from the fucina Qwen3 pages ("The qwen3 descriptor runner";
// "14. Model families", sections 14.1 and 14.2) and the ggml block formats they name.
// Every value computation is the textbook definition, in f64, in the order the pages'
// block structure gives (pre-norm attention block, then pre-norm FFN block).  Storage
// types (fp16 scales, bf16/f32 cache, f32 dequantised weights) are emulated exactly.
// Output rows are independent, so loops over them may run on several OpenMP threads; no
// sum is split, blocked or reordered.
//
// Readings where the pages are silent (each also listed in the design notes):
//   * RMSNorm y = x / sqrt(mean(x^2) + eps) * g (gain multiplies directly);
//   * "half-rope over the full head dim" = rotate-half pairing (i, i + D/2), frequency
//     theta^(-2i/D), angle pos * freq, applied after the per-head q/k RMSNorm;
//   * attention scale 1/sqrt(D); q head h reads kv head h / (n_q / n_kv);
//   * the new token's k/v are rounded to the cache dtype before attention reads them;
//   * a q8_0 cache (runner page, "KV cache"; section 14.2 load specifics) holds each head's
//     k and v row as ggml Q8_0 blocks of 32 along head_dim, quantised from the f32 values
//     like weights; its scores use q quantised the same way (the integer q8 x q8 score
//     path), the 1/sqrt(D) scale applied to the score, and V dequantised;
//   * SwiGLU h = silu(gate) * up with silu(z) = z / (1 + e^-z);
//   * MoE: softmax over all router logits, top-k by value with ties to the lower expert
//     index, selected weights renormalised to sum 1 when norm_topk_prob is set;
//   * a missing output matrix means tied embeddings (section 14.2 load specifics).
//
// Parity with real GGUF files is unpinned (no files exist here); the codecs are pinned by
// round trips, hand-built blocks and library conversions in the tests.

#include "fq_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>
#include <vector>
#include <omp.h>

namespace {

// ---------------------------------------------------------------- number formats

// Round |v| to a binary format with p significant bits and minimum normal exponent emin,
// round-to-nearest-even, with gradual underflow.  Returns the rounded value as a double
// (infinite when the rounded magnitude exceeds max_finite).
double round_to_format(double v, int p, int emin, double max_finite) {
    if (v == 0 || std::isnan(v) || std::isinf(v)) return v;
    double a = std::fabs(v);
    int ex;
    std::frexp(a, &ex);          // a = m * 2^ex, m in [0.5, 1)
    int E = ex - 1;              // a in [2^E, 2^(E+1))
    if (E < emin) E = emin;      // subnormals share the 2^(emin-p+1) grid
    double ulp = std::ldexp(1.0, E - (p - 1));
    double q = a / ulp;          // exact: scaling by a power of two
    double fl = std::floor(q), rem = q - fl;
    if (rem > 0.5 || (rem == 0.5 && std::fmod(fl, 2.0) != 0.0)) fl += 1.0;
    double r = fl * ulp;
    if (r > max_finite) r = INFINITY;
    return v < 0 ? -r : r;
}

const double FP16_MAX = 65504.0;
const double BF16_MAX = std::ldexp(255.0, 120);   // (2 - 2^-7) * 2^127

uint16_t encode_fp16(double r) {   // r already representable
    uint16_t s = std::signbit(r) ? 0x8000 : 0;
    double a = std::fabs(r);
    if (std::isnan(r)) return 0x7E00;
    if (std::isinf(a)) return s | 0x7C00;
    if (a < std::ldexp(1.0, -14)) return s | (uint16_t)(a / std::ldexp(1.0, -24));
    int ex;
    std::frexp(a, &ex);
    int E = ex - 1;
    uint16_t mant = (uint16_t)(a / std::ldexp(1.0, E - 10) - 1024.0);
    return s | (uint16_t)((E + 15) << 10) | mant;
}

double decode_fp16(uint16_t h) {
    int e = (h >> 10) & 31, m = h & 1023;
    double s = (h & 0x8000) ? -1.0 : 1.0;
    if (e == 0) return s * std::ldexp((double)m, -24);
    if (e == 31) return m ? NAN : s * INFINITY;
    return s * std::ldexp((double)(1024 + m), e - 25);
}

double round_half_away(double v) { return v < 0 ? -std::floor(-v + 0.5) : std::floor(v + 0.5); }

// ---------------------------------------------------------------- ggml blocks
// Q8_0: 34 bytes per 32 weights = fp16 d (little endian) + 32 x int8 q; x_i = d * q_i.
const int Q8_BLK = 32, Q8_BYTES = 34;
// Q4_K: 144 bytes per 256 weights = fp16 d, fp16 dmin, 12 bytes of packed 6-bit
// (scale, min) pairs for eight 32-element sub-blocks, 128 bytes of 4-bit codes.
const int Q4K_BLK = 256, Q4K_BYTES = 144;

uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

void q4k_get(const uint8_t* s12, int j, int* sc, int* mn) {
    if (j < 4) {
        *sc = s12[j] & 63;
        *mn = s12[j + 4] & 63;
    } else {
        *sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);
        *mn = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
    }
}

size_t row_bytes(int wtype, int cols) {
    if (wtype == OR_Q8_0) return (size_t)cols / Q8_BLK * Q8_BYTES;
    if (wtype == OR_Q4_K) return (size_t)cols / Q4K_BLK * Q4K_BYTES;
    return (size_t)cols * 4;
}

// dequantise one packed row into f32 values (exact: every value is representable)
void dequant_row(int wtype, const uint8_t* row, int cols, float* out) {
    if (wtype == OR_Q8_0) {
        or_dequant_q8_0(row, (size_t)cols, out);
    } else if (wtype == OR_Q4_K) {
        or_dequant_q4_k(row, (size_t)cols, out);
    } else {
        std::memcpy(out, row, (size_t)cols * 4);
    }
}

double dot_row(int wtype, const uint8_t* row, int cols, const double* x, float* scratch) {
    dequant_row(wtype, row, cols, scratch);
    double acc = 0;
    for (int c = 0; c < cols; ++c) acc += (double)scratch[c] * x[c];
    return acc;
}

// serial y = W x (used inside position-parallel loops)
void gemv_serial(int wtype, const void* W, int rows, int cols, const double* x, double* y) {
    std::vector<float> buf(cols);
    const uint8_t* base = (const uint8_t*)W;
    size_t rb = row_bytes(wtype, cols);
    for (int r = 0; r < rows; ++r) y[r] = dot_row(wtype, base + rb * r, cols, x, buf.data());
}

void gemv_parallel(int wtype, const void* W, int rows, int cols, const double* x, double* y) {
    const uint8_t* base = (const uint8_t*)W;
    size_t rb = row_bytes(wtype, cols);
#pragma omp parallel if (rows >= 256)
    {
        std::vector<float> buf(cols);
#pragma omp for schedule(static)
        for (int r = 0; r < rows; ++r) y[r] = dot_row(wtype, base + rb * r, cols, x, buf.data());
    }
}

}  // namespace

// ==================================================================== C API

extern "C" {

int or_set_threads(int n) {
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
}

double or_fp16_to_f64(uint16_t h) { return decode_fp16(h); }
uint16_t or_f64_to_fp16(double v) { return encode_fp16(round_to_format(v, 11, -14, FP16_MAX)); }

double or_bf16_to_f64(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

uint16_t or_f64_to_bf16(double v) {
    if (std::isnan(v)) return 0x7FC0;
    float f = (float)round_to_format(v, 8, -126, BF16_MAX);   // exact in f32
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

float or_f64_to_f32(double v) {
    return (float)round_to_format(v, 24, -126, (double)3.4028234663852886e38);
}

void or_dequant_q8_0(const uint8_t* blocks, size_t n, float* out) {
    for (size_t b = 0; b < n / Q8_BLK; ++b) {
        const uint8_t* p = blocks + b * Q8_BYTES;
        double d = decode_fp16(rd16(p));
        for (int i = 0; i < Q8_BLK; ++i) out[b * Q8_BLK + i] = (float)(d * (double)(int8_t)p[2 + i]);
    }
}

// Reading of the Q8_0 quantiser: d = fp16(max|x| / 127), q = round-half-away(x / d)
// clamped to [-127, 127]; an all-zero block (d == 0) stores zeros.
void or_quant_q8_0(const float* x, size_t n, uint8_t* blocks) {
    for (size_t b = 0; b < n / Q8_BLK; ++b) {
        const float* xb = x + b * Q8_BLK;
        uint8_t* p = blocks + b * Q8_BYTES;
        double amax = 0;
        for (int i = 0; i < Q8_BLK; ++i) amax = std::max(amax, std::fabs((double)xb[i]));
        uint16_t dh = or_f64_to_fp16(amax / 127.0);
        double d = decode_fp16(dh);
        p[0] = (uint8_t)(dh & 0xFF);
        p[1] = (uint8_t)(dh >> 8);
        for (int i = 0; i < Q8_BLK; ++i) {
            double q = d == 0 ? 0 : std::min(127.0, std::max(-127.0, round_half_away((double)xb[i] / d)));
            p[2 + i] = (uint8_t)(int8_t)(int)q;
        }
    }
}

void or_q4k_scale_min(const uint8_t* s12, int j, int* sc, int* mn) { q4k_get(s12, j, sc, mn); }

void or_q4k_pack_scale_min(const int* sc, const int* mn, uint8_t* s12) {
    std::memset(s12, 0, 12);
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            s12[j] |= (uint8_t)(sc[j] & 63);
            s12[j + 4] |= (uint8_t)(mn[j] & 63);
        } else {
            s12[j + 4] |= (uint8_t)((sc[j] & 15) | ((mn[j] & 15) << 4));
            s12[j - 4] |= (uint8_t)(((sc[j] >> 4) & 3) << 6);
            s12[j] |= (uint8_t)(((mn[j] >> 4) & 3) << 6);
        }
    }
}

// x = (d * sc_j) * q - dmin * m_j, rounded once to f32 (both products are exact).
void or_dequant_q4_k(const uint8_t* blocks, size_t n, float* out) {
    for (size_t b = 0; b < n / Q4K_BLK; ++b) {
        const uint8_t* p = blocks + b * Q4K_BYTES;
        double d = decode_fp16(rd16(p)), dmin = decode_fp16(rd16(p + 2));
        const uint8_t* s12 = p + 4;
        const uint8_t* qs = p + 16;
        for (int j = 0; j < 8; ++j) {
            int sc, mn;
            q4k_get(s12, j, &sc, &mn);
            double step = d * sc, off = dmin * mn;
            for (int i = 0; i < 32; ++i) {
                uint8_t byte = qs[32 * (j / 2) + i];
                int q = (j & 1) ? (byte >> 4) : (byte & 15);
                out[b * Q4K_BLK + 32 * j + i] = (float)(step * q - off);
            }
        }
    }
}

// Reading of the Q4_K quantiser (a plain min/max fit): per sub-block lo = min(0, min x),
// s_j = (max x - lo) / 15, m_j = -lo; d = fp16(max s / 63), dmin = fp16(max m / 63);
// sc_j, mn_j = round(s_j / d), round(m_j / dmin) in [0, 63];
// q = round((x + dmin mn_j) / (d sc_j)) in [0, 15] (0 when d sc_j == 0).
void or_quant_q4_k(const float* x, size_t n, uint8_t* blocks) {
    for (size_t b = 0; b < n / Q4K_BLK; ++b) {
        const float* xb = x + b * Q4K_BLK;
        uint8_t* p = blocks + b * Q4K_BYTES;
        double s[8], m[8], smax = 0, mmax = 0;
        for (int j = 0; j < 8; ++j) {
            double lo = 0, hi = -INFINITY;
            for (int i = 0; i < 32; ++i) {
                lo = std::min(lo, (double)xb[32 * j + i]);
                hi = std::max(hi, (double)xb[32 * j + i]);
            }
            s[j] = (hi - lo) / 15.0;
            m[j] = -lo;
            smax = std::max(smax, s[j]);
            mmax = std::max(mmax, m[j]);
        }
        uint16_t dh = or_f64_to_fp16(smax / 63.0), mh = or_f64_to_fp16(mmax / 63.0);
        double d = decode_fp16(dh), dmin = decode_fp16(mh);
        int sc[8], mn[8];
        for (int j = 0; j < 8; ++j) {
            sc[j] = d == 0 ? 0 : (int)std::min(63.0, std::max(0.0, round_half_away(s[j] / d)));
            mn[j] = dmin == 0 ? 0 : (int)std::min(63.0, std::max(0.0, round_half_away(m[j] / dmin)));
        }
        p[0] = (uint8_t)(dh & 0xFF); p[1] = (uint8_t)(dh >> 8);
        p[2] = (uint8_t)(mh & 0xFF); p[3] = (uint8_t)(mh >> 8);
        or_q4k_pack_scale_min(sc, mn, p + 4);
        uint8_t* qs = p + 16;
        std::memset(qs, 0, 128);
        for (int j = 0; j < 8; ++j) {
            double step = d * sc[j], off = dmin * mn[j];
            for (int i = 0; i < 32; ++i) {
                int q = step == 0 ? 0
                        : (int)std::min(15.0, std::max(0.0, round_half_away(((double)xb[32 * j + i] + off) / step)));
                qs[32 * (j / 2) + i] |= (uint8_t)((j & 1) ? (q << 4) : q);
            }
        }
    }
}

// ---------------------------------------------------------------- building blocks

void or_rmsnorm(const double* x, int n, const float* g, double eps, double* y) {
    double ss = 0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / std::sqrt(ss / n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * inv * (double)g[i];
}

void or_rope(double* v, int d, int pos, double theta) {
    int half = d / 2;
    for (int i = 0; i < half; ++i) {
        double freq = std::pow(theta, -2.0 * i / d);
        double ang = (double)pos * freq;
        double c = std::cos(ang), s = std::sin(ang);
        double a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = a * s + b * c;
    }
}

// softmax(q . k_t / sqrt(d)) over t < T, then the weighted sum of v_t
void or_attention(const double* q, const float* K, const float* V, int T, int d, size_t row_stride,
                  double* o) {
    std::vector<double> s(T);
    double scale = 1.0 / std::sqrt((double)d), mx = -INFINITY;
    for (int t = 0; t < T; ++t) {
        double acc = 0;
        for (int i = 0; i < d; ++i) acc += q[i] * (double)K[t * row_stride + i];
        s[t] = acc * scale;
        mx = std::max(mx, s[t]);
    }
    double l = 0;
    for (int t = 0; t < T; ++t) { s[t] = std::exp(s[t] - mx); l += s[t]; }
    for (int i = 0; i < d; ++i) o[i] = 0;
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < d; ++i) o[i] += s[t] * (double)V[t * row_stride + i];
    for (int i = 0; i < d; ++i) o[i] /= l;
}

void or_kv_round_row(int kv_type, const double* x, int n, float* out) {
    if (kv_type == OR_KV_Q8_0) {
        std::vector<float> f(n);
        std::vector<uint8_t> blk((size_t)n / Q8_BLK * Q8_BYTES);
        for (int i = 0; i < n; ++i) f[i] = or_f64_to_f32(x[i]);
        or_quant_q8_0(f.data(), (size_t)n, blk.data());
        or_dequant_q8_0(blk.data(), (size_t)n, out);
    } else if (kv_type == OR_KV_BF16) {
        for (int i = 0; i < n; ++i) out[i] = (float)or_bf16_to_f64(or_f64_to_bf16(x[i]));
    } else {
        for (int i = 0; i < n; ++i) out[i] = or_f64_to_f32(x[i]);
    }
}

void or_attention_q8(const double* q, const float* K, const float* V, int T, int d, size_t row_stride,
                     double* o) {
    std::vector<float> qf(d);
    or_kv_round_row(OR_KV_Q8_0, q, d, qf.data());
    std::vector<double> qd(qf.begin(), qf.end());
    or_attention(qd.data(), K, V, T, d, row_stride, o);
}

double or_silu(double z) { return z / (1.0 + std::exp(-z)); }

void or_router(const double* logits, int n_exp, int k, int norm, int* idx, double* w) {
    double mx = -INFINITY;
    for (int e = 0; e < n_exp; ++e) mx = std::max(mx, logits[e]);
    std::vector<double> p(n_exp);
    double sum = 0;
    for (int e = 0; e < n_exp; ++e) { p[e] = std::exp(logits[e] - mx); sum += p[e]; }
    for (int e = 0; e < n_exp; ++e) p[e] /= sum;
    std::vector<int> order(n_exp);
    std::iota(order.begin(), order.end(), 0);
    // by probability descending, ties to the lower expert index
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return p[a] > p[b]; });
    double sel = 0;
    for (int j = 0; j < k; ++j) { idx[j] = order[j]; w[j] = p[order[j]]; sel += w[j]; }
    if (norm)
        for (int j = 0; j < k; ++j) w[j] /= sel;
}

void or_gemv(int wtype, const void* W, int rows, int cols, const double* x, double* y) {
    gemv_parallel(wtype, W, rows, cols, x, y);
}

int or_argmax(const double* v, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

}  // extern "C"

// ==================================================================== model

struct or_layer_w {
    const float *attn_norm = nullptr, *q_norm = nullptr, *k_norm = nullptr, *ffn_norm = nullptr;
    const float* router = nullptr;
    const void *wq = nullptr, *wk = nullptr, *wv = nullptr, *wo = nullptr;
    const void *w_gate = nullptr, *w_up = nullptr, *w_down = nullptr;
    const void *gate_exps = nullptr, *up_exps = nullptr, *down_exps = nullptr;
};

struct or_model {
    or_dims d;
    const void* tok_embd = nullptr;
    const float* output_norm = nullptr;
    const void* output = nullptr;
    std::vector<or_layer_w> layers;
};

struct or_cache {
    const or_model* m;
    int cap, len;
    int keep = 0;              // layer steps attend over the rows already at `len` instead of writing theirs
    std::vector<float> k, v;   // [layer][n_kv][cap][head_dim], values in the cache dtype
    size_t idx(int layer, int h, int pos) const {
        const or_dims& d = m->d;
        return (((size_t)layer * d.n_kv + h) * cap + pos) * d.head_dim;
    }
};

namespace {

// one head's row of n values as the cache stores it
void to_cache(const or_model* m, const double* x, int n, float* out) { or_kv_round_row(m->d.kv_type, x, n, out); }

void attend(const or_model* m, const double* q, const float* K, const float* V, int T, size_t row_stride,
            double* o) {
    if (m->d.kv_type == OR_KV_Q8_0) or_attention_q8(q, K, V, T, m->d.head_dim, row_stride, o);
    else or_attention(q, K, V, T, m->d.head_dim, row_stride, o);
}

// q/k/v for one token: xn -> per-head RMSNorm -> rope (section 14.2: per-head q/k RMSNorm,
// full RoPE; runner page: QK-norm + half-rope over the full head dim)
void qkv_project(const or_model* m, const or_layer_w& w, const double* xn, int pos, double* q,
                 double* k, double* v, bool serial) {
    const or_dims& d = m->d;
    auto gv = serial ? gemv_serial : gemv_parallel;
    gv(d.wtype, w.wq, d.n_q * d.head_dim, d.hidden, xn, q);
    gv(d.wtype, w.wk, d.n_kv * d.head_dim, d.hidden, xn, k);
    gv(d.wtype, w.wv, d.n_kv * d.head_dim, d.hidden, xn, v);
    std::vector<double> tmp(d.head_dim);
    for (int h = 0; h < d.n_q; ++h) {
        double* qh = q + (size_t)h * d.head_dim;
        or_rmsnorm(qh, d.head_dim, w.q_norm, d.eps, tmp.data());
        std::copy(tmp.begin(), tmp.end(), qh);
        or_rope(qh, d.head_dim, pos, d.theta);
    }
    for (int h = 0; h < d.n_kv; ++h) {
        double* kh = k + (size_t)h * d.head_dim;
        or_rmsnorm(kh, d.head_dim, w.k_norm, d.eps, tmp.data());
        std::copy(tmp.begin(), tmp.end(), kh);
        or_rope(kh, d.head_dim, pos, d.theta);
    }
}

// FFN block on one token (dense SwiGLU or routed mixture), returns the residual update
void ffn(const or_model* m, const or_layer_w& w, const double* x, double* dx, int* route_idx,
         double* route_w, bool serial, double* route_logits = nullptr) {
    const or_dims& d = m->d;
    auto gv = serial ? gemv_serial : gemv_parallel;
    std::vector<double> xn(d.hidden);
    or_rmsnorm(x, d.hidden, w.ffn_norm, d.eps, xn.data());
    if (d.n_exp == 0) {
        std::vector<double> g(d.ffn), u(d.ffn);
        gv(d.wtype, w.w_gate, d.ffn, d.hidden, xn.data(), g.data());
        gv(d.wtype, w.w_up, d.ffn, d.hidden, xn.data(), u.data());
        for (int i = 0; i < d.ffn; ++i) g[i] = or_silu(g[i]) * u[i];
        gv(d.wtype, w.w_down, d.hidden, d.ffn, g.data(), dx);
        return;
    }
    std::vector<double> r(d.n_exp);
    gv(OR_F32, w.router, d.n_exp, d.hidden, xn.data(), r.data());
    if (route_logits) std::copy(r.begin(), r.end(), route_logits);
    std::vector<int> idx(d.n_used);
    std::vector<double> wt(d.n_used);
    or_router(r.data(), d.n_exp, d.n_used, d.norm_topk, idx.data(), wt.data());
    if (route_idx) std::copy(idx.begin(), idx.end(), route_idx);
    if (route_w) std::copy(wt.begin(), wt.end(), route_w);
    int Fe = d.moe_ffn;
    size_t gu_rb = row_bytes(d.wtype, d.hidden), dn_rb = row_bytes(d.wtype, Fe);
    std::vector<double> g(Fe), u(Fe), y(d.hidden);
    for (int i = 0; i < d.hidden; ++i) dx[i] = 0;
    for (int j = 0; j < d.n_used; ++j) {
        int e = idx[j];
        gv(d.wtype, (const uint8_t*)w.gate_exps + gu_rb * Fe * e, Fe, d.hidden, xn.data(), g.data());
        gv(d.wtype, (const uint8_t*)w.up_exps + gu_rb * Fe * e, Fe, d.hidden, xn.data(), u.data());
        for (int i = 0; i < Fe; ++i) g[i] = or_silu(g[i]) * u[i];
        gv(d.wtype, (const uint8_t*)w.down_exps + dn_rb * d.hidden * e, d.hidden, Fe, g.data(), y.data());
        for (int i = 0; i < d.hidden; ++i) dx[i] += wt[j] * y[i];
    }
}

void lm_head(const or_model* m, const double* x, double* logits) {
    const or_dims& d = m->d;
    std::vector<double> xn(d.hidden);
    or_rmsnorm(x, d.hidden, m->output_norm, d.eps, xn.data());
    const void* W = m->output ? m->output : m->tok_embd;   // tied when output is absent
    gemv_parallel(d.wtype, W, d.vocab, d.hidden, xn.data(), logits);
}

void embed(const or_model* m, int token, double* x) {
    const or_dims& d = m->d;
    std::vector<float> row(d.hidden);
    dequant_row(d.wtype, (const uint8_t*)m->tok_embd + row_bytes(d.wtype, d.hidden) * token, d.hidden,
                row.data());
    for (int i = 0; i < d.hidden; ++i) x[i] = row[i];
}

}  // namespace

extern "C" {

// Section 14.2 validation: zero heads, non-divisible GQA grouping, odd head_dim and
// inconsistent MoE fields are InvalidConfig.
int or_validate(const or_dims* d) {
    if (!d) return OR_INVALID_ARGUMENT;
    if (d->hidden <= 0 || d->layers <= 0 || d->n_q <= 0 || d->n_kv <= 0 || d->head_dim <= 0) return OR_INVALID_CONFIG;
    if (d->n_q % d->n_kv != 0) return OR_INVALID_CONFIG;
    if (d->head_dim % 2 != 0) return OR_INVALID_CONFIG;
    if (d->kv_type < OR_KV_F32 || d->kv_type > OR_KV_Q8_0) return OR_INVALID_ARGUMENT;
    if (d->kv_type == OR_KV_Q8_0 && d->head_dim % 32 != 0) return OR_INVALID_CONFIG;   // whole blocks per row
    bool any = d->n_exp || d->n_used || d->moe_ffn, all = d->n_exp && d->n_used && d->moe_ffn;
    if (any && !all) return OR_INVALID_CONFIG;
    if (all && d->n_used > d->n_exp) return OR_INVALID_CONFIG;
    if (!all && d->ffn <= 0) return OR_INVALID_CONFIG;
    return OR_OK;
}

or_model* or_model_new(const or_dims* d) {
    if (or_validate(d) != OR_OK) return nullptr;
    auto* m = new or_model;
    m->d = *d;
    m->layers.resize(d->layers);
    return m;
}

void or_model_free(or_model* m) { delete m; }

void or_model_set_global(or_model* m, const void* tok_embd, const float* output_norm, const void* output) {
    m->tok_embd = tok_embd;
    m->output_norm = output_norm;
    m->output = output;
}

void or_model_set_layer(or_model* m, int layer, const float* attn_norm, const void* wq, const void* wk,
                        const void* wv, const float* q_norm, const float* k_norm, const void* wo,
                        const float* ffn_norm, const void* w_gate, const void* w_up, const void* w_down,
                        const float* router, const void* gate_exps, const void* up_exps,
                        const void* down_exps) {
    or_layer_w& w = m->layers[layer];
    w.attn_norm = attn_norm; w.wq = wq; w.wk = wk; w.wv = wv; w.q_norm = q_norm; w.k_norm = k_norm;
    w.wo = wo; w.ffn_norm = ffn_norm; w.w_gate = w_gate; w.w_up = w_up; w.w_down = w_down;
    w.router = router; w.gate_exps = gate_exps; w.up_exps = up_exps; w.down_exps = down_exps;
}

or_cache* or_cache_new(const or_model* m, int capacity) {
    if (!m || capacity <= 0) return nullptr;
    auto* c = new or_cache;
    c->m = m;
    c->cap = capacity;
    c->len = 0;
    size_t n = (size_t)m->d.layers * m->d.n_kv * capacity * m->d.head_dim;
    c->k.assign(n, 0.f);
    c->v.assign(n, 0.f);
    return c;
}

void or_cache_free(or_cache* c) { delete c; }
int or_cache_len(const or_cache* c) { return c->len; }

int or_cache_write(or_cache* c, int layer, int pos0, int n, const float* k, const float* v) {
    const or_dims& d = c->m->d;
    if (layer < 0 || layer >= d.layers || pos0 < 0 || n < 0 || pos0 + n > c->cap) return OR_INVALID_ARGUMENT;
    std::vector<double> kr(d.head_dim), vr(d.head_dim);
    for (int p = 0; p < n; ++p)
        for (int h = 0; h < d.n_kv; ++h) {
            size_t src = ((size_t)p * d.n_kv + h) * d.head_dim;
            for (int i = 0; i < d.head_dim; ++i) {
                kr[i] = k[src + i];
                vr[i] = v[src + i];
            }
            to_cache(c->m, kr.data(), d.head_dim, &c->k[c->idx(layer, h, pos0 + p)]);
            to_cache(c->m, vr.data(), d.head_dim, &c->v[c->idx(layer, h, pos0 + p)]);
        }
    return OR_OK;
}

int or_cache_keep_current(or_cache* c, int keep) {
    if (!c) return OR_INVALID_ARGUMENT;
    c->keep = keep != 0;
    return OR_OK;
}

int or_cache_set_len(or_cache* c, int len) {
    if (len < 0 || len > c->cap) return OR_INVALID_ARGUMENT;
    c->len = len;
    return OR_OK;
}

int or_cache_read(const or_cache* c, int layer, int pos0, int n, float* k, float* v) {
    const or_dims& d = c->m->d;
    if (layer < 0 || layer >= d.layers || pos0 < 0 || n < 0 || pos0 + n > c->cap) return OR_INVALID_ARGUMENT;
    for (int p = 0; p < n; ++p)
        for (int h = 0; h < d.n_kv; ++h)
            for (int i = 0; i < d.head_dim; ++i) {
                size_t dst = ((size_t)p * d.n_kv + h) * d.head_dim + i;
                k[dst] = c->k[c->idx(layer, h, pos0 + p) + i];
                v[dst] = c->v[c->idx(layer, h, pos0 + p) + i];
            }
    return OR_OK;
}

int or_qkv_project(const or_model* m, int layer, const double* xn, int pos, double* q, double* k, double* v) {
    const or_dims& d = m->d;
    if (layer < 0 || layer >= d.layers || !xn || !q || !k || !v || pos < 0) return OR_INVALID_ARGUMENT;
    qkv_project(m, m->layers[layer], xn, pos, q, k, v, true);
    return OR_OK;
}

int or_layer_step(const or_model* m, int layer, or_cache* c, int pos, double* x, int* route_idx,
                  double* route_w) {
    return or_layer_step_route(m, layer, c, pos, x, route_idx, route_w, nullptr);
}

int or_layer_step_route(const or_model* m, int layer, or_cache* c, int pos, double* x, int* route_idx,
                        double* route_w, double* route_logits) {
    const or_dims& d = m->d;
    if (layer < 0 || layer >= d.layers || !x) return OR_INVALID_ARGUMENT;
    if (c->m != m) return OR_MISMATCHED_KV_CACHES;
    if (pos != c->len) return OR_INVALID_SEQUENCE_LENGTH;
    if (pos + 1 > c->cap) return OR_KV_CACHE_OVERFLOW;
    const or_layer_w& w = m->layers[layer];
    int D = d.head_dim, qd = d.n_q * D, kvd = d.n_kv * D, group = d.n_q / d.n_kv;

    // attention block: fused norm + QKV, QK-norm + rope, append, grouped causal attention
    std::vector<double> xn(d.hidden), q(qd), k(kvd), v(kvd), o(qd), dx(d.hidden);
    or_rmsnorm(x, d.hidden, w.attn_norm, d.eps, xn.data());
    qkv_project(m, w, xn.data(), pos, q.data(), k.data(), v.data(), false);
    if (!c->keep)
        for (int h = 0; h < d.n_kv; ++h) {
            to_cache(m, &k[(size_t)h * D], D, &c->k[c->idx(layer, h, pos)]);
            to_cache(m, &v[(size_t)h * D], D, &c->v[c->idx(layer, h, pos)]);
        }
#pragma omp parallel for schedule(static)
    for (int h = 0; h < d.n_q; ++h) {   // heads are independent outputs
        int g = h / group;
        attend(m, &q[(size_t)h * D], &c->k[c->idx(layer, g, 0)], &c->v[c->idx(layer, g, 0)], pos + 1, D,
               &o[(size_t)h * D]);
    }
    gemv_parallel(d.wtype, w.wo, d.hidden, qd, o.data(), dx.data());
    for (int i = 0; i < d.hidden; ++i) x[i] += dx[i];

    // FFN block
    ffn(m, w, x, dx.data(), route_idx, route_w, false, route_logits);
    for (int i = 0; i < d.hidden; ++i) x[i] += dx[i];
    return OR_OK;
}

int or_decode_step(const or_model* m, or_cache* c, int token, int pos0, double* logits, double* layer_out,
                   int* route_idx, double* route_w) {
    const or_dims& d = m->d;
    if (c->m != m) return OR_MISMATCHED_KV_CACHES;
    if (pos0 != c->len) return OR_INVALID_SEQUENCE_LENGTH;
    if (c->len + 1 > c->cap) return OR_KV_CACHE_OVERFLOW;
    if (token < 0 || token >= d.vocab) return OR_INVALID_ARGUMENT;
    std::vector<double> x(d.hidden);
    embed(m, token, x.data());
    for (int L = 0; L < d.layers; ++L) {
        int rc = or_layer_step(m, L, c, pos0, x.data(), route_idx ? route_idx + (size_t)L * d.n_used : nullptr,
                               route_w ? route_w + (size_t)L * d.n_used : nullptr);
        if (rc) return rc;
        if (layer_out) std::copy(x.begin(), x.end(), layer_out + (size_t)L * d.hidden);
    }
    c->len = pos0 + 1;
    if (logits) lm_head(m, x.data(), logits);
    return OR_OK;
}

// Section 14.2 lockstep batch: sibling caches of this model, distinct pointers; row s is
// stream s's next-token distribution; every cache advances by one.
int or_decode_step_batch(const or_model* m, or_cache* const* caches, int n, const int* tokens, double* logits) {
    if (n <= 0) return OR_INVALID_SEQUENCE_LENGTH;
    for (int s = 0; s < n; ++s) {
        if (!caches[s] || caches[s]->m != m) return OR_MISMATCHED_KV_CACHES;
        for (int t = 0; t < s; ++t)
            if (caches[t] == caches[s]) return OR_MISMATCHED_KV_CACHES;
        if (caches[s]->len + 1 > caches[s]->cap) return OR_KV_CACHE_OVERFLOW;
        if (tokens[s] < 0 || tokens[s] >= m->d.vocab) return OR_INVALID_ARGUMENT;
    }
    for (int s = 0; s < n; ++s) {
        int rc = or_decode_step(m, caches[s], tokens[s], caches[s]->len,
                                logits ? logits + (size_t)s * m->d.vocab : nullptr, nullptr, nullptr, nullptr);
        if (rc) return rc;
    }
    return OR_OK;
}

// Section 14.1 forwardLastLogits: the whole sequence at once, layer by layer, with causal
// attention recomputed over all positions (k/v rounded to the cache dtype as a cache
// would hold them); no cache object is involved.
int or_forward_last_logits(const or_model* m, const int* tokens, int n, double* logits) {
    const or_dims& d = m->d;
    if (n <= 0) return OR_INVALID_SEQUENCE_LENGTH;
    for (int p = 0; p < n; ++p)
        if (tokens[p] < 0 || tokens[p] >= d.vocab) return OR_INVALID_ARGUMENT;
    int D = d.head_dim, qd = d.n_q * D, kvd = d.n_kv * D, group = d.n_q / d.n_kv;
    std::vector<double> X((size_t)n * d.hidden);
    for (int p = 0; p < n; ++p) embed(m, tokens[p], &X[(size_t)p * d.hidden]);
    std::vector<double> Q((size_t)n * qd);
    std::vector<float> K((size_t)n * kvd), V((size_t)n * kvd);   // [pos][n_kv][D]
    for (int L = 0; L < d.layers; ++L) {
        const or_layer_w& w = m->layers[L];
#pragma omp parallel for schedule(dynamic)
        for (int p = 0; p < n; ++p) {
            std::vector<double> xn(d.hidden), k(kvd), v(kvd);
            or_rmsnorm(&X[(size_t)p * d.hidden], d.hidden, w.attn_norm, d.eps, xn.data());
            qkv_project(m, w, xn.data(), p, &Q[(size_t)p * qd], k.data(), v.data(), true);
            for (int h = 0; h < d.n_kv; ++h) {
                to_cache(m, &k[(size_t)h * D], D, &K[(size_t)p * kvd + (size_t)h * D]);
                to_cache(m, &v[(size_t)h * D], D, &V[(size_t)p * kvd + (size_t)h * D]);
            }
        }
#pragma omp parallel for schedule(dynamic)
        for (int p = 0; p < n; ++p) {
            std::vector<double> o(qd), dx(d.hidden);
            for (int h = 0; h < d.n_q; ++h) {
                int g = h / group;
                attend(m, &Q[(size_t)p * qd + (size_t)h * D], &K[(size_t)g * D], &V[(size_t)g * D], p + 1,
                       (size_t)kvd, &o[(size_t)h * D]);
            }
            double* x = &X[(size_t)p * d.hidden];
            gemv_serial(d.wtype, w.wo, d.hidden, qd, o.data(), dx.data());
            for (int i = 0; i < d.hidden; ++i) x[i] += dx[i];
            ffn(m, w, x, dx.data(), nullptr, nullptr, true);
            for (int i = 0; i < d.hidden; ++i) x[i] += dx[i];
        }
    }
    lm_head(m, &X[(size_t)(n - 1) * d.hidden], logits);
    return OR_OK;
}

int or_sample(const double* z, int n, const or_sampling* s, const int* history, int n_hist, double u) {
    std::vector<double> v(z, z + n);
    if (s->repeat_penalty != 1.0) {
        std::vector<char> seen(n, 0);
        for (int i = 0; i < n_hist; ++i) {
            int t = history[i];
            if (t < 0 || t >= n || seen[t]) continue;
            seen[t] = 1;
            v[t] = v[t] > 0 ? v[t] / s->repeat_penalty : v[t] * s->repeat_penalty;
        }
    }
    if (s->temp == 0) return or_argmax(v.data(), n);
    double mx = -INFINITY;
    for (int i = 0; i < n; ++i) mx = std::max(mx, v[i] / s->temp);
    std::vector<double> p(n);
    double sum = 0;
    for (int i = 0; i < n; ++i) {
        p[i] = std::exp(v[i] / s->temp - mx);
        sum += p[i];
    }
    for (int i = 0; i < n; ++i) p[i] /= sum;
    std::vector<int> order(n);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return p[a] > p[b]; });   // ties: lower id first
    int keep = n;
    if (s->top_k > 0) keep = std::min(keep, s->top_k);
    if (s->top_p < 1.0) {
        double mass = 0, total = 0;
        for (int j = 0; j < keep; ++j) total += p[order[j]];
        int j = 0;
        while (j < keep) {
            mass += p[order[j]];
            ++j;
            if (mass >= s->top_p * total) break;
        }
        keep = j;
    }
    if (s->min_p > 0) {
        double cut = s->min_p * p[order[0]];
        int j = 1;
        while (j < keep && p[order[j]] >= cut) ++j;
        keep = j;
    }
    double Z = 0;
    for (int j = 0; j < keep; ++j) Z += p[order[j]];
    double target = u * Z, c = 0;
    for (int j = 0; j < keep; ++j) {
        c += p[order[j]];
        if (c > target) return order[j];
    }
    return order[keep - 1];
}

double or_uniform24(uint64_t seed, uint64_t counter) {
    uint64_t x = seed + (counter + 1) * 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    x ^= x >> 31;
    return (double)(x >> 40) * (1.0 / 16777216.0);
}

}  // extern "C"
