// Seeded synthetic input generator shared by the oracle harness and the GPU harness.
//
// This file produces INPUT DATA only: Gaussian weights packed into ggml Q8_0 / Q4_K
// blocks, norm gains, bf16/f32 KV-cache contents and token ids.  It holds none of the
// decode step's arithmetic (no dequantisation, no GEMV, no attention).  Both sides read
// the exact same bytes, so any disagreement downstream is in the decode path itself.
//
// Random numbers are counter based: element i of tensor `tid` under seed `seed` is a
// pure function of (seed, tid, i), computed with SplitMix64 (Steele, Lea, Flood,
// "Fast splittable pseudorandom number generators", OOPSLA 2014) and turned into normal
// deviates with the Box-Muller transform (Box & Muller, 1958).  Element 2j and 2j+1 of a
// stream are the cosine and sine outputs of the pair j.  Work is split over threads by
// index range, so the result does not depend on the thread count.
//
// Packing follows the ggml block formats the decode pages name (Q8_0: fp16 scale + 32
// int8; Q4_K: 256-element super-block with fp16 d/dmin, 12 bytes of 6-bit scales/mins and
// 128 bytes of nibbles).  The quantiser choices are the plain readings spelled out in the
// design notes: Q8_0 scale = fp16(max|x|/127), codes round-half-away; Q4_K uses a plain
// min/max fit per 32-element sub-block.
//
// Built with -ffp-contract=off so results are identical on x86-64 and aarch64 hosts.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

int g_threads = 0;

int thread_count() {
    if (g_threads > 0) return g_threads;
    unsigned h = std::thread::hardware_concurrency();
    return h == 0 ? 1 : (int)h;
}

template <class F>
void parallel_for(uint64_t n, uint64_t grain, F f) {
    int nt = thread_count();
    if (n <= grain || nt <= 1) { f(0, n); return; }
    uint64_t chunks = (n + grain - 1) / grain;
    int use = (int)std::min<uint64_t>(chunks, (uint64_t)nt);
    std::vector<std::thread> th;
    uint64_t per = (chunks + use - 1) / use * grain;
    for (int t = 0; t < use; ++t) {
        uint64_t b = (uint64_t)t * per, e = std::min(n, b + per);
        if (b >= e) break;
        th.emplace_back([=] { f(b, e); });
    }
    for (auto& x : th) x.join();
}

inline uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
    return splitmix64(splitmix64(seed) ^ (tid * 0xD1B54A32D192ED03ull));
}

// uniform in (0, 1] with 53 random bits
inline double u01(uint64_t key, uint64_t ctr) {
    uint64_t r = splitmix64(key + ctr * 0x9E3779B97F4A7C15ull);
    return (double)((r >> 11) + 1) * (1.0 / 9007199254740992.0);
}

inline double normal_at(uint64_t key, uint64_t i) {
    uint64_t pair = i >> 1;
    double u1 = u01(key, 2 * pair), u2 = u01(key, 2 * pair + 1);
    double r = std::sqrt(-2.0 * std::log(u1));
    double a = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? r * std::sin(a) : r * std::cos(a);
}

// IEEE binary16 from a double, round to nearest even (no double rounding via float).
uint16_t to_fp16(double v) {
    uint16_t sign = std::signbit(v) ? 0x8000 : 0;
    double a = std::fabs(v);
    if (std::isnan(v)) return 0x7E00;
    if (a >= 65520.0) return sign | 0x7C00;       // rounds to infinity
    if (a < std::ldexp(1.0, -25)) {                 // below half the smallest subnormal
        if (a == std::ldexp(1.0, -25)) return sign; // tie to even (zero)
        return sign;
    }
    int e;
    std::frexp(a, &e);                              // a = m * 2^e, m in [0.5, 1)
    int exp_unb = e - 1;                            // a in [2^exp_unb, 2^(exp_unb+1))
    if (exp_unb < -14) exp_unb = -14;               // subnormal range shares the 2^-24 grid
    double ulp = std::ldexp(1.0, exp_unb - 10);
    double q = a / ulp;                             // exact (power of two scaling)
    double fl = std::floor(q);
    double rem = q - fl;
    uint64_t m = (uint64_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (m & 1))) m += 1;
    // m counts ulps at exponent exp_unb; assemble bits
    if (exp_unb == -14 && m < 1024) return sign | (uint16_t)m;  // subnormal
    if (m == 2048) { m = 1024; exp_unb += 1; }
    if (exp_unb > 15) return sign | 0x7C00;
    return sign | (uint16_t)(((exp_unb + 15) << 10) | (m - 1024));
}

double fp16_value(uint16_t h) {
    int e = (h >> 10) & 31, m = h & 1023;
    double s = (h & 0x8000) ? -1.0 : 1.0;
    if (e == 0) return s * std::ldexp((double)m, -24);
    if (e == 31) return m ? NAN : s * INFINITY;
    return s * std::ldexp((double)(m + 1024), e - 25);
}

// bfloat16 from a float, round to nearest even
uint16_t to_bf16(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

inline double round_half_away(double v) { return v < 0 ? -std::floor(-v + 0.5) : std::floor(v + 0.5); }

void quant_q8_0_block(const float* x, uint8_t* out) {
    double amax = 0;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs((double)x[i]));
    uint16_t dh = to_fp16(amax / 127.0);
    double d = fp16_value(dh);
    out[0] = (uint8_t)(dh & 0xFF);
    out[1] = (uint8_t)(dh >> 8);
    for (int i = 0; i < 32; ++i) {
        int q = 0;
        if (d != 0) {
            double r = round_half_away((double)x[i] / d);
            q = (int)std::max(-127.0, std::min(127.0, r));
        }
        out[2 + i] = (uint8_t)(int8_t)q;
    }
}

void pack_scale_min(const int* sc, const int* mn, uint8_t* s12) {
    std::memset(s12, 0, 12);
    for (int j = 0; j < 4; ++j) {
        s12[j] = (uint8_t)(sc[j] & 63);
        s12[j + 4] = (uint8_t)(mn[j] & 63);
    }
    for (int j = 4; j < 8; ++j) {
        s12[j + 4] = (uint8_t)((sc[j] & 15) | ((mn[j] & 15) << 4));
        s12[j - 4] |= (uint8_t)((sc[j] >> 4) << 6);
        s12[j] |= (uint8_t)((mn[j] >> 4) << 6);
    }
}

void quant_q4_k_block(const float* x, uint8_t* out) {
    double s[8], m[8];
    for (int j = 0; j < 8; ++j) {
        double lo = 0, hi = -INFINITY;
        for (int i = 0; i < 32; ++i) {
            double v = x[32 * j + i];
            lo = std::min(lo, v);
            hi = std::max(hi, v);
        }
        s[j] = (hi - lo) / 15.0;
        m[j] = -lo;
    }
    double smax = 0, mmax = 0;
    for (int j = 0; j < 8; ++j) { smax = std::max(smax, s[j]); mmax = std::max(mmax, m[j]); }
    uint16_t dh = to_fp16(smax / 63.0), mh = to_fp16(mmax / 63.0);
    double d = fp16_value(dh), dmin = fp16_value(mh);
    int sc[8], mn[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = d == 0 ? 0 : (int)std::max(0.0, std::min(63.0, round_half_away(s[j] / d)));
        mn[j] = dmin == 0 ? 0 : (int)std::max(0.0, std::min(63.0, round_half_away(m[j] / dmin)));
    }
    out[0] = (uint8_t)(dh & 0xFF); out[1] = (uint8_t)(dh >> 8);
    out[2] = (uint8_t)(mh & 0xFF); out[3] = (uint8_t)(mh >> 8);
    pack_scale_min(sc, mn, out + 4);
    uint8_t* qs = out + 16;
    std::memset(qs, 0, 128);
    for (int j = 0; j < 8; ++j) {
        double step = d * sc[j], off = dmin * mn[j];
        for (int i = 0; i < 32; ++i) {
            int q = 0;
            if (step != 0) {
                double r = round_half_away(((double)x[32 * j + i] + off) / step);
                q = (int)std::max(0.0, std::min(15.0, r));
            }
            int chunk = j >> 1;
            if (j & 1) qs[32 * chunk + i] |= (uint8_t)(q << 4);
            else qs[32 * chunk + i] |= (uint8_t)q;
        }
    }
}

}  // namespace

extern "C" {

void synth_set_threads(int n) { g_threads = n; }

// out[i] = mean + std * N(0,1)[offset + i] of stream (seed, tid)
void synth_normal_f32(uint64_t seed, uint64_t tid, uint64_t offset, uint64_t n, double mean,
                      double stddev, float* out) {
    uint64_t key = stream_key(seed, tid);
    parallel_for(n, 1 << 16, [&](uint64_t b, uint64_t e) {
        for (uint64_t i = b; i < e; ++i) out[i] = (float)(mean + stddev * normal_at(key, offset + i));
    });
}

// bf16 bits of the f32 values synth_normal_f32 would produce
void synth_normal_bf16(uint64_t seed, uint64_t tid, uint64_t offset, uint64_t n, double mean,
                       double stddev, uint16_t* out) {
    uint64_t key = stream_key(seed, tid);
    parallel_for(n, 1 << 16, [&](uint64_t b, uint64_t e) {
        for (uint64_t i = b; i < e; ++i)
            out[i] = to_bf16((float)(mean + stddev * normal_at(key, offset + i)));
    });
}

// integers uniform in [lo, hi)
void synth_uniform_i32(uint64_t seed, uint64_t tid, uint64_t n, int64_t lo, int64_t hi, int32_t* out) {
    uint64_t key = stream_key(seed, tid);
    uint64_t span = (uint64_t)(hi - lo);
    for (uint64_t i = 0; i < n; ++i) {
        double u = u01(key, i) ;                    // (0, 1]
        uint64_t k = (uint64_t)((1.0 - u) * (double)span);
        if (k >= span) k = span - 1;
        out[i] = (int32_t)(lo + (int64_t)k);
    }
}

// rows x cols weights ~ N(0, std^2) (stream element r*cols + c), packed as ggml Q8_0 rows
void synth_q8_0(uint64_t seed, uint64_t tid, uint64_t rows, uint64_t cols, double stddev, uint8_t* out) {
    uint64_t key = stream_key(seed, tid);
    uint64_t nb = cols / 32;
    parallel_for(rows, 16, [&](uint64_t b, uint64_t e) {
        std::vector<float> x(cols);
        for (uint64_t r = b; r < e; ++r) {
            for (uint64_t c = 0; c < cols; ++c) x[c] = (float)(stddev * normal_at(key, r * cols + c));
            for (uint64_t k = 0; k < nb; ++k) quant_q8_0_block(&x[32 * k], out + (r * nb + k) * 34);
        }
    });
}

void synth_q4_k(uint64_t seed, uint64_t tid, uint64_t rows, uint64_t cols, double stddev, uint8_t* out) {
    uint64_t key = stream_key(seed, tid);
    uint64_t nb = cols / 256;
    parallel_for(rows, 16, [&](uint64_t b, uint64_t e) {
        std::vector<float> x(cols);
        for (uint64_t r = b; r < e; ++r) {
            for (uint64_t c = 0; c < cols; ++c) x[c] = (float)(stddev * normal_at(key, r * cols + c));
            for (uint64_t k = 0; k < nb; ++k) quant_q4_k_block(&x[256 * k], out + (r * nb + k) * 144);
        }
    });
}

// pack arbitrary f32 values (n a multiple of the block) -- used by tests to build
// inputs with chosen values
void synth_pack_q8_0(const float* x, uint64_t n, uint8_t* out) {
    for (uint64_t k = 0; k < n / 32; ++k) quant_q8_0_block(x + 32 * k, out + 34 * k);
}
void synth_pack_q4_k(const float* x, uint64_t n, uint8_t* out) {
    for (uint64_t k = 0; k < n / 256; ++k) quant_q4_k_block(x + 256 * k, out + 144 * k);
}

}  // extern "C"
