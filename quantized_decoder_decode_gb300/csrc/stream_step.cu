// The whole batch-1 decode step of a dense model as one persistent kernel that streams the
// step's bytes ahead of its dependency chain (sm_103a).
//
// forwardStep ("14. Model families", section 14.2) at batch 1 is bound by the bytes it must
// read: every weight of every layer, the LM head and the cached K/V rows (the fucina README,
// Performance: single-token decode is bound by the total weight bytes).  None of those bytes
// depends on the token being decoded -- only the activations do.  So each CTA (one per SM)
// runs two roles at once:
//   * a producer warp walks the CTA's fixed share of the whole step -- per layer its rows of
//     the QKV projection, its chunk of the cached K/V rows, its rows of the O, gate_up and
//     down projections, then its rows of the LM head -- and copies it into a ring of 16 KB
//     shared-memory slots with bulk asynchronous copies (cp.async.bulk + mbarrier), as fast
//     as slots free up.  It never waits for an activation, so HBM keeps streaming while the
//     consumers wait for the other CTAs;
//   * eleven consumer warps run the step's phases on what has landed.  Per layer:
//       QKV   RMSNorm(x) . W_qkv rows                        (x: the previous layer's output)
//       ATT   per-head QK-RMSNorm, half-rope, KV append, attention over the CTA's chunk of
//             one kv head's cached positions (split-K flash decode; partial m, l, o)
//       MERGE the chunks of a kv head merged, 8 dimensions per CTA
//       O     x_att = x + W_o . o
//       GU    h = silu(W_g . RMSNorm(x_att)) * (W_u . RMSNorm(x_att))  (gate/up rows paired)
//       DN    x_next = x_att + W_d . h
//     then the final RMSNorm + LM head with the greedy argmax.
// Activations cross CTAs as 64-bit exchange words (value bits | tag << 32) written with one
// store and read with one load: a reader polls the words it needs until every tag is the
// current (launch, layer) tag, so one L2 round trip carries both the data and its readiness
// -- no counters, fences or grid barriers.  A buffer is rewritten once per layer, and every
// reader of a buffer has finished with it before any CTA can write its next version (the
// layer's later phases depend on all of those readers), so one buffer per activation
// suffices.  Every wait is bounded; a CTA that gives up records the error word and leaves
// after its producer has waited for the copies it issued.

#include "common.cuh"
#include "kernels.h"
#include "quant.cuh"
#include "tma.cuh"

#include <algorithm>

namespace fq {

namespace {

constexpr int NW = 11;                // consumer warps (with the producer, 3 per SM sub-partition)
constexpr int NC = NW * 32;           // consumer threads
constexpr int NTH = NC + 32;          // + the producer warp
constexpr int SLOT = 16384;           // bytes per ring slot
constexpr int MAXSLOT = 16;
constexpr int TP = 64;                // cached positions per attention item (64 bf16 rows of K or of V: 16 KB)
constexpr int MSL = 16;               // merge slices per kv head (8 dimensions each)
constexpr int MAXS = 160;             // attention chunks per kv head at most
constexpr long long BUDGET = 1ll << 29;

// ---------------------------------------------------------------- exchange words

FQ_DEV void xw_store(unsigned long long* p, float v, uint32_t tag) {
    const unsigned long long w = ((unsigned long long)tag << 32) | (unsigned long long)__float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
FQ_DEV void xw_load2(const unsigned long long* p, unsigned long long& a, unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
FQ_DEV bool tag_ok(unsigned long long a, unsigned long long b, uint32_t tag) {
    return (uint32_t)(a >> 32) == tag && (uint32_t)(b >> 32) == tag;
}
FQ_DEV uint32_t ld_volatile(const uint32_t* p) { return *reinterpret_cast<const volatile uint32_t*>(p); }

// A launch-wide stop: a CTA that gives up writes `val` (its launch's sequence + 1) to `word`,
// and every wait of the same launch that sees it gives up too.  The next launch has another
// sequence, so a failed step does not stop later ones.
struct Stop {
    uint32_t* word;
    uint32_t val;
    FQ_DEV bool seen() const { return *reinterpret_cast<const volatile uint32_t*>(word) == val; }
    FQ_DEV void raise() const { atomicExch(word, val); }
};

// Shared state of one CTA besides the ring.
struct Ctl {
    int abort;                        // a wait gave up: every role leaves
    float inv;                        // 1/rms of the staged input
    unsigned long long best;          // LM head: this CTA's argmax key
    int last;                         // this CTA took the last finishing ticket
};

// Poll n exchange words (n even; src 16-byte aligned) until all carry `tag`, handing each
// pair to put(i, v_i, v_i+1, g_i, g_i+1) with the matching pair of `gain` (1 without one).
// Threads take pairs tid, tid + nthr, ... in batches of B; the gains of a batch are loaded
// with its first round, and every round re-issues the loads of the pairs that are not ready
// yet, so a batch costs one round trip after its last pair was written.
template <int B, class Put>
FQ_DEV bool xw_read(const unsigned long long* src, int n, uint32_t tag, int tid, int nthr, const Stop& stop,
                    const float* gain, Put put) {
    for (int base = 2 * tid; base < n; base += 2 * nthr * B) {
        unsigned long long a[B], b[B];
        float2 g[B];
        uint32_t pending = 0;
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int i = base + 2 * nthr * j;
            g[j] = make_float2(1.f, 1.f);
            if (i < n) {
                xw_load2(src + i, a[j], b[j]);
                if (gain) g[j] = *reinterpret_cast<const float2*>(gain + i);
                pending |= 1u << j;
            }
        }
        long long t0 = 0;
        int rounds = 0;
        while (true) {
#pragma unroll
            for (int j = 0; j < B; ++j)
                if ((pending >> j & 1u) && tag_ok(a[j], b[j], tag)) {
                    put(base + 2 * nthr * j, __uint_as_float((uint32_t)a[j]), __uint_as_float((uint32_t)b[j]), g[j]);
                    pending &= ~(1u << j);
                }
            if (!pending) break;
            if (rounds == 0) t0 = clock64();
            else if (clock64() - t0 > BUDGET) return false;
            if ((++rounds & 15) == 0 && stop.seen()) return false;
#pragma unroll
            for (int j = 0; j < B; ++j)
                if (pending >> j & 1u) xw_load2(src + base + 2 * nthr * j, a[j], b[j]);
        }
    }
    return true;
}

// Poll NP pairs of exchange words at p[0], p[1], ... (each 16-byte aligned) until all
// carry `tag`; every round re-issues the loads of the pairs not ready yet.
template <int NP>
FQ_DEV bool xw_read_pairs(const unsigned long long* const (&p)[NP], uint32_t tag, const Stop& stop,
                          float (&v)[2 * NP]) {
    unsigned long long a[NP], b[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) xw_load2(p[j], a[j], b[j]);
    uint32_t pending = (1u << NP) - 1u;
    long long t0 = 0;
    int rounds = 0;
    while (true) {
#pragma unroll
        for (int j = 0; j < NP; ++j)
            if ((pending >> j & 1u) && tag_ok(a[j], b[j], tag)) {
                v[2 * j] = __uint_as_float((uint32_t)a[j]);
                v[2 * j + 1] = __uint_as_float((uint32_t)b[j]);
                pending &= ~(1u << j);
            }
        if (!pending) return true;
        if (rounds == 0) t0 = clock64();
        else if (clock64() - t0 > BUDGET) return false;
        if ((++rounds & 15) == 0 && stop.seen()) return false;
#pragma unroll
        for (int j = 0; j < NP; ++j)
            if (pending >> j & 1u) xw_load2(p[j], a[j], b[j]);
    }
}

FQ_DEV void csync() { asm volatile("bar.sync 1, %0;" ::"r"(NC) : "memory"); }

inline int align_up(int v, int a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------- the step's schedule
// Producer and consumers derive the same item sequence from these functions.

FQ_HD inline void row_range(int N, bool pairs, int c, int G, int& r0, int& r1) {
    if (pairs) {
        const long long P = N / 2;
        r0 = 2 * (int)(P * c / G);
        r1 = 2 * (int)(P * (c + 1) / G);
    } else {
        r0 = (int)((long long)N * c / G);
        r1 = (int)((long long)N * (c + 1) / G);
    }
}

// bytes of one row in a slot: Q8_0 codes + fp16 scales, or Q4_K super-blocks
FQ_HD int slot_row_bytes(const QMat& W) { return W.fmt == FMT_Q8_0 ? W.K + W.K / 16 : W.K / 256 * 144; }
// rows per ring item: as many as a slot holds
FQ_HD int rows_per_item(const QMat& W) { return SLOT / slot_row_bytes(W); }

// How a phase's rows x K are cut into tasks (R rows x `up` units): the K split that gives the
// busiest warp the least work, with whole 32-lane passes; a split must save a tenth of that
// work to be taken, since it adds a barrier and the partial-sum epilogue.
struct Split {
    int kparts, up;
};
FQ_HD inline Split choose_split(int r0, int r1, int rs, int R, int U) {
    int groups = 0;
    for (int r = r0; r < r1; r += rs) groups += ((rs < r1 - r ? rs : r1 - r) + R - 1) / R;
    const int kmax = (U / 32 > 1 ? U / 32 : 1);
    Split best{1, U};
    long long best_cost = -1;
    for (int kp = 1; kp <= kmax; ++kp) {
        const int up = ((U + kp - 1) / kp + 31) / 32 * 32;
        const int kpe = (U + up - 1) / up;
        const long long cost = (long long)((groups * kpe + NW - 1) / NW) * up;
        if (best_cost < 0 || cost * 10 < best_cost * 9) {
            best_cost = cost;
            best = Split{kpe, up};
        }
    }
    return best;
}



// the attention unit of this CTA: kv head g, chunk c of S; positions [t0, t1) of T = pos + 1
struct AttnUnit {
    bool active;
    int g, c, t0, t1;
    int nt, e;        // ring tiles of cached rows [t0, e), e = min(t1, pos)
};
FQ_DEV AttnUnit attn_unit_of(int Hkv, int S, int pos) {
    AttnUnit u;
    u.active = (int)blockIdx.x < Hkv * S;
    u.g = blockIdx.x / S;
    u.c = blockIdx.x % S;
    const long long T = (long long)pos + 1;
    u.t0 = (int)(T * u.c / S);
    u.t1 = (int)(T * (u.c + 1) / S);
    if (!u.active) u.t0 = u.t1 = 0;
    u.e = min(u.t1, pos);
    u.nt = u.e > u.t0 ? (u.e - u.t0 + TP - 1) / TP : 0;   // K items, then as many V items
    return u;
}
// ---------------------------------------------------------------- producer

struct Ring {
    uint8_t* buf;
    uint64_t* full;
    uint64_t* empty;
    int nslot;
};

struct Producer {
    Ring r;
    volatile int* abort;
    uint32_t* err;
    Stop stop;
    uint32_t it = 0;
    int s = 0;              // it % nslot and the parity of it / nslot, kept as counters
    uint32_t par = 0;

    FQ_DEV bool wait_free() {
        const uint32_t ph = par ^ 1u;
        if (mbar_try_wait(&r.empty[s], ph)) return true;
        const long long t0 = clock64();
        while (!mbar_try_wait(&r.empty[s], ph)) {
            __nanosleep(128);   // the ring is full: back off instead of spinning on the barrier
            if (*abort) return false;
            if (clock64() - t0 > BUDGET) {
                atomicOr(err, 128u);
                stop.raise();
                *abort = 1;
                return false;
            }
        }
        return true;
    }
    // one item of up to two contiguous byte ranges (sizes multiples of 16) into the next slot
    FQ_DEV bool item(const void* a, uint32_t an, const void* b, uint32_t bn, uint32_t b_off) {
        if (!wait_free()) return false;
        uint8_t* dst = r.buf + (size_t)s * SLOT;
        mbar_arrive_expect_tx(&r.full[s], an + bn);
        if (an) bulk_g2s(dst, a, an, &r.full[s]);
        if (bn) bulk_g2s(dst + b_off, b, bn, &r.full[s]);
        ++it;
        if (++s == r.nslot) {
            s = 0;
            par ^= 1u;
        }
        return true;
    }
    FQ_DEV bool rows(const QMat& W, const ProjPlan& pp) {
        const int r0 = pp.r0, r1 = pp.r1, rs = pp.rs;
        for (int r = r0; r < r1; r += rs) {
            const int nr = min(rs, r1 - r);
            if (W.fmt == FMT_Q8_0) {
                if (!item(W.q + (size_t)r * W.K, (uint32_t)nr * W.K, reinterpret_cast<const uint8_t*>(W.s) + (size_t)r * (W.K / 16),
                          (uint32_t)nr * (W.K / 16), (uint32_t)nr * W.K))
                    return false;
            } else {
                const size_t rb = (size_t)W.K / 256 * 144;
                if (!item(W.q + (size_t)r * rb, (uint32_t)(nr * rb), nullptr, 0, 0)) return false;
            }
        }
        return true;
    }
    FQ_DEV bool kv(const StreamArgs& a, int layer, const SeqState& ss, const AttnUnit& u) {
        const int nt = u.nt;
        const int e = u.e;
        const size_t head = ((size_t)layer * a.Hkv + u.g) * (size_t)ss.cap * HEAD_DIM;
        const uint16_t* K = reinterpret_cast<const uint16_t*>(ss.k) + head;
        const uint16_t* V = reinterpret_cast<const uint16_t*>(ss.v) + head;
        for (int t = 0; t < 2 * nt; ++t) {   // the chunk's K rows, then its V rows
            const int tb = u.t0 + (t % nt) * TP, n = min(TP, e - tb);
            const uint16_t* src = (t < nt ? K : V) + (size_t)tb * HEAD_DIM;
            if (!item(src, (uint32_t)n * HEAD_DIM * 2, nullptr, 0, 0)) return false;
        }
        return true;
    }
    // wait until the copies of the last issued items have landed (the CTA must not leave
    // with copies in flight into its shared memory)
    FQ_DEV void drain() {
        const uint32_t n = min((uint32_t)r.nslot, it);
        for (uint32_t j = it - n; j < it; ++j) {
            const int s = j % r.nslot;
            if (!mbar_wait(&r.full[s], (j / r.nslot) & 1u)) atomicOr(err, 256u);
        }
    }
};

FQ_DEV void produce(const StreamArgs& a, Ring ring, volatile int* abort, Stop stop, const ProjPlan* pp,
                    const AttnUnit& u) {
    const SeqState ss = a.st->seq[0];
    Producer p{ring, abort, a.err, stop};
    // the consumers' phase order (one loop, so that each kind of copy exists once in the code)
    const int nq = 5 * a.n_layers + (a.head ? 1 : 0);
    for (int q = 0; q < nq; ++q) {
        const int L = q / 5, ph = q - 5 * L;
        const bool lm = L == a.n_layers;
        const StreamLayer& lw = a.layers[lm ? 0 : L];
        bool ok;
        if (ph == 1) {
            ok = p.kv(a, L, ss, u);
        } else {
            const int j = lm ? P_LM : ph == 0 ? P_QKV : ph == 2 ? P_O : ph == 3 ? P_GU : P_DN;
            const QMat& W = lm ? a.out : ph == 0 ? lw.qkv : ph == 2 ? lw.o : ph == 3 ? lw.gate_up : lw.down;
            ok = p.rows(W, pp[j]);
        }
        if (!ok) break;
    }
    p.drain();
}

// ---------------------------------------------------------------- consumers: projections

struct Cons {
    Ring ring;
    Ctl& ctl;
    uint32_t* err;
    Stop stop;
    uint32_t it = 0;           // items consumed so far (same sequence as the producer's)
    int s = 0;                 // it % nslot and the parity of it / nslot, kept as counters
    uint32_t par = 0;

    // this CTA gives up: record `code`, stop the launch, leave at the next barrier
    FQ_DEV void fail(uint32_t code) {
        atomicOr(err, code);
        stop.raise();
        ctl.abort = 1;
    }

    FQ_DEV bool wait_full(int lane) {
        if (mbar_try_wait(&ring.full[s], par)) return true;
        const long long t0 = clock64();
        while (!mbar_try_wait(&ring.full[s], par)) {
            if (ctl.abort) return false;
            if (clock64() - t0 > BUDGET) {
                fail(512u);
                return false;
            }
        }
        return true;
    }
    FQ_DEV const uint8_t* slot() const { return ring.buf + (size_t)s * SLOT; }
    FQ_DEV void release(int lane) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring.empty[s]);
        ++it;
        if (++s == ring.nslot) {
            s = 0;
            par ^= 1u;
        }
    }
};

// Butterfly sums of R values over the 32 lanes of a warp, transposing as it goes; the sum of
// value r ends in lane r * (32 / R).
template <int R>
FQ_DEV float reduce_rows(float (&v)[R], int lane) {
    if constexpr (R == 4) {
        const bool hi = lane & 16;
        float k0 = hi ? v[2] : v[0], k1 = hi ? v[3] : v[1];
        const float s0 = hi ? v[0] : v[2], s1 = hi ? v[1] : v[3];
        k0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 16);
        k1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 16);
        const bool h8 = lane & 8;
        float k = h8 ? k1 : k0;
        k += __shfl_xor_sync(0xFFFFFFFFu, h8 ? k0 : k1, 8);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 4);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 2);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 1);
        return k;
    } else {
        const bool hi = lane & 16;
        float k = hi ? v[1] : v[0];
        k += __shfl_xor_sync(0xFFFFFFFFu, hi ? v[0] : v[1], 16);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 8);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 4);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 2);
        k += __shfl_xor_sync(0xFFFFFFFFu, k, 1);
        return k;
    }
}

// ---------------------------------------------------------------- staged input of a projection
// The input vector of a projection (times its RMSNorm gain) is staged once per phase as
// 16-bit block fixed point: per block of 32 elements (the Q8_0 block, the Q4_K sub-block) a
// float scale s = max|x| / 32767 and integers v = round(x / s) in [-32767, 32767], stored as
// two byte planes hi = v >> 8 (signed) and lo = v & 255 (unsigned), v = 256 hi + lo.  A dot
// product with integer weight codes then runs on dp4a, exact in integers, and
// sum_k q_k x_k = s (256 sum q hi + sum q lo) up to the rounding of x, at most s / 2 per
// element (a relative 1.5e-5 of the block's largest value).
struct XStage {
    float* xs;        // [K] floats of the input (times the gain), before quantisation
    int8_t* hi;       // [K] high bytes, in the format's unit layout
    uint8_t* lo;      // [K] low bytes
    float* sc;        // [K / 32] block scales
    float* sum32;     // [K / 32] Q4_K: float sums of the input per sub-block (the min term)
};

// Byte index of element e in the unit layout: Q8_0 units (16 elements per lane) are plain
// runs; Q4_K units (64 elements per lane) are split into four 16-byte pieces stored
// piece-major, so that the lanes of a warp reading piece p of consecutive units hit
// consecutive 16-byte words.
template <int FMT>
FQ_DEV int xq_index(int e, int K) {
    if constexpr (FMT == FMT_Q8_0) return e;
    else return ((e & 63) >> 4) * (K >> 2) + (e >> 6) * 16 + (e & 15);
}

FQ_DEV int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
FQ_DEV int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
FQ_DEV int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
FQ_DEV int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Two independent fused multiply-adds in one instruction (the packed f32x2 form): each half is
// exactly fmaf(a, b, c) of that half.
FQ_DEV void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "mov.b64 d, {%0, %1};\n\t"
        "fma.rn.f32x2 d, a, b, d;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Two independent multiplies in one instruction (packed f32x2): (d0, d1) = (a0 b0, a1 b1).
FQ_DEV void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

template <int FMT> struct PCfg;
// rows per task R; elements per unit (one lane's share of a row per pass)
template <> struct PCfg<FMT_Q8_0> { static constexpr int R = 4, UE = 16; };
template <> struct PCfg<FMT_Q4_K> { static constexpr int R = 4, UE = 64; };

// R rows of an item (rows row0.. of its nr rows), units [ua, ub) of each row: lane takes units
// ua + lane, ua + lane + 32, ...  Returns per-row partial sums before the warp reduction.
// FULL: all R rows exist, and their work has no branches and interleaves; otherwise rows past
// the item's end are skipped one by one.
template <int FMT, bool FULL>
FQ_DEV void task_dot(const uint8_t* slot, int nr, int K, int row0, int ua, int ub, int lane, const XStage& x,
                     float (&acc)[PCfg<FMT>::R]) {
    constexpr int R = PCfg<FMT>::R;
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;
    if constexpr (FMT == FMT_Q8_0) {
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot + (size_t)nr * K);
        const int K32 = K >> 5;
        // (the unit loops stay rolled: unrolled by two, the larger code made the whole step
        // about 1 % slower, although a task alone ran faster)
#pragma unroll 1
        for (int u = ua + lane; u < ub; u += 32) {
            const uint4 h = *reinterpret_cast<const uint4*>(x.hi + 16 * u);
            const uint4 l = *reinterpret_cast<const uint4*>(x.lo + 16 * u);
            const float s = x.sc[u >> 1];
            auto dot = [&](int row, float& d, float& f) {   // one row's block: fp16 scale, integer sum
                const uint4 c = *reinterpret_cast<const uint4*>(slot + (size_t)row * K + 16 * u);
                d = h2f(sc[row * K32 + (u >> 1)]);
                int A = dp4a_ss(c.x, h.x, 0);
                A = dp4a_ss(c.y, h.y, A);
                A = dp4a_ss(c.z, h.z, A);
                A = dp4a_ss(c.w, h.w, A);
                int B = dp4a_su(c.x, l.x, 0);
                B = dp4a_su(c.y, l.y, B);
                B = dp4a_su(c.z, l.z, B);
                B = dp4a_su(c.w, l.w, B);
                f = (float)(A * 256 + B);
            };
            if constexpr (FULL) {
                // rows in pairs: d s and the accumulation as packed f32x2 (the same two
                // roundings per row as the scalar form)
#pragma unroll
                for (int r = 0; r < R; r += 2) {
                    float d0, f0, d1, f1;
                    dot(row0 + r, d0, f0);
                    dot(row0 + r + 1, d1, f1);
                    fmul2(d0, d1, d0, d1, s, s);
                    ffma2(acc[r], acc[r + 1], d0, d1, f0, f1);
                }
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int row = row0 + r;
                    if (row >= nr) break;
                    float d, f;
                    dot(row, d, f);
                    acc[r] = fmaf(d * s, f, acc[r]);
                }
            }
        }
    } else {
        const int rb = K / 256 * 144;
        const int P = K >> 2;   // bytes per piece plane
#pragma unroll 1
        for (int u = ua + lane; u < ub; u += 32) {   // 64-element unit: nibble chunk c of super-block u / 4
            const int c = u & 3;
            const int e0 = (u >> 2) * 256 + 64 * c;
            // pieces 0, 1: the low-nibble sub-block (elements e0 .. e0 + 31); 2, 3: the high one
            uint4 h[4], l[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                h[p] = *reinterpret_cast<const uint4*>(x.hi + p * P + 16 * u);
                l[p] = *reinterpret_cast<const uint4*>(x.lo + p * P + 16 * u);
            }
            // the high nibbles are used in place (16 x their value): 1/16 goes with their block scale
            const float s_lo = x.sc[e0 >> 5], s_hi = x.sc[(e0 >> 5) + 1] * 0.0625f;
            const float m_lo = x.sum32[e0 >> 5], m_hi = x.sum32[(e0 >> 5) + 1];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = row0 + r;
                if (!FULL && row >= nr) break;
                const uint8_t* blk = slot + (size_t)row * rb + (u >> 2) * 144;
                const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
                const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
                const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
                const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                int Alo = 0, Blo = 0, Ahi = 0, Bhi = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t qlo = w[i] & 0x0F0F0F0Fu, qhi = w[i] & 0xF0F0F0F0u;
                    const uint4& hl = h[i >> 2];
                    const uint4& ll = l[i >> 2];
                    const uint4& hh = h[2 + (i >> 2)];
                    const uint4& lh = l[2 + (i >> 2)];
                    const int k = i & 3;
                    Alo = dp4a_us(qlo, (&hl.x)[k], Alo);
                    Blo = dp4a_uu(qlo, (&ll.x)[k], Blo);
                    Ahi = dp4a_us(qhi, (&hh.x)[k], Ahi);
                    Bhi = dp4a_uu(qhi, (&lh.x)[k], Bhi);
                }
                const float d = h2f((unsigned short)(hdr.x & 0xFFFFu));
                const float dmin = h2f((unsigned short)(hdr.x >> 16));
                // 6-bit scale and min of sub-blocks 2c and 2c + 1 (the low pair, c < 2: byte j of
                // words 0 and 1; the high pair: low / high nibble of byte j - 4 of word 2, top
                // bits from bytes j - 4 of words 0 / 1), one form for both with selects, since c
                // differs between neighbouring lanes
                const uint32_t sh = 16u * (c & 1);
                const uint32_t a0 = hdr.w >> sh, b0 = hdr.y >> sh, b1 = hdr.z >> sh;
                const bool hp = c >= 2;
                const uint32_t X0 = hp ? a0 : b0, Y0 = hp ? b0 >> 2 : b0;
                const uint32_t X1 = hp ? a0 >> 4 : b1, Y1 = hp ? b1 >> 2 : b1;
                const uint32_t sc0 = (X0 & 15u) | (Y0 & 48u), sc1 = ((X0 >> 8) & 15u) | ((Y0 >> 8) & 48u);
                const uint32_t mn0 = (X1 & 15u) | (Y1 & 48u), mn1 = ((X1 >> 8) & 15u) | ((Y1 >> 8) & 48u);
                // both sub-blocks at once (packed pairs): d sc s (A 256 + B) - dmin mn m
                float t0, t1, u0, u1;
                fmul2(t0, t1, d, d, (float)sc0, (float)sc1);
                fmul2(t0, t1, t0, t1, s_lo, s_hi);
                fmul2(u0, u1, -dmin, -dmin, (float)mn0, (float)mn1);
                fmul2(u0, u1, u0, u1, m_lo, m_hi);
                ffma2(u0, u1, t0, t1, (float)(Alo * 256 + Blo), (float)(Ahi * 256 + Bhi));
                acc[r] += u0 + u1;
            }
        }
    }
}

// Rows [r0, r1) of W times the staged input: every item of the phase is waited for and
// released by every consumer warp in order; the phase's tasks (R rows of one item x one K
// part) go to the warps round-robin.  `direct` (one K part, and gate/up pairs never split
// between items): the task's warp finishes its rows at once, emit(row, y, y2) (y2: the up row
// after a gate row when `pairs`); otherwise partial sums land in red[row - r0][kpart].
// Returns false when a wait gave up.
template <int FMT, class Emit>
FQ_DEV bool proj_tasks(Cons& cs, const QMat& W, const ProjPlan& pp, const XStage& x, float* red, bool direct,
                       bool pairs, Emit&& emit) {
    constexpr int R = PCfg<FMT>::R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r0 = pp.r0, r1 = pp.r1, rs = pp.rs, U = pp.U;
    const int kparts = pp.kparts, up = pp.up;
    int first = warp;   // this warp's first task of the current item (tasks go round-robin)
    for (int r = r0; r < r1; r += rs) {
        const int nr = min(rs, r1 - r);
        const int ntask = (nr + R - 1) / R * kparts;
        if (!cs.wait_full(lane)) return 0;
        const uint8_t* slot = cs.slot();
        for (int t = first; t < ntask; t += NW) {
            const int g = t / kparts * R, kp = t - t / kparts * kparts;
            float acc[R];
            // (the branch-free form pays for Q8_0 rows; Q4_K's larger body runs slower interleaved)
            if (FMT == FMT_Q8_0 && g + R <= nr)
                task_dot<FMT, true>(slot, nr, W.K, g, kp * up, min(U, (kp + 1) * up), lane, x, acc);
            else task_dot<FMT, false>(slot, nr, W.K, g, kp * up, min(U, (kp + 1) * up), lane, x, acc);
            const float s = reduce_rows<R>(acc, lane);
            const int rr = lane / (32 / R);
            const bool owner = (lane & (32 / R - 1)) == 0 && g + rr < nr;
            if (direct) {
                const float s2 = __shfl_down_sync(0xFFFFFFFFu, s, 32 / R);   // the next row's sum
                if (owner && !(pairs && (rr & 1))) emit(r + g + rr, s, s2);
            } else if (owner) {
                red[(size_t)(r - r0 + g + rr) * kparts + kp] = s;
            }
        }
        first = ((first - ntask) % NW + NW) % NW;
        cs.release(lane);
    }
    return true;
}

// ---------------------------------------------------------------- consumers: attention

// q / k head held as 4 dims per lane (dims 4l..4l+3) by one warp: RMSNorm with the gain,
// then the rotate-half RoPE (pairs (i, i + 64): lane l < 16 holds i, lane l + 16 holds i + 64)
// (gain: the lane's 4 gains; rot: cos/sin of its 4 dims at the position, both loaded by the
// caller ahead of the values)
FQ_DEV void norm_rope4(float v[4], const float (&gain)[4], const float2 (&rot)[4], float eps, int lane) {
    float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / (float)HEAD_DIM + eps);
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = v[j] * inv * gain[j];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float partner = __shfl_xor_sync(0xFFFFFFFFu, v[j], 16);
        const float2 cs = rot[j];
        v[j] = lane < 16 ? v[j] * cs.x - partner * cs.y : partner * cs.y + v[j] * cs.x;
    }
}

// Shared memory of the attention phase (inside the staging area); the scores of the chunk's
// positions follow the struct, [G][score capacity].
template <int G>
struct alignas(16) AttSmem {
    // (the arrays read as float4 come first, at offsets that are multiples of 16)
    float qs[G][HEAD_DIM];            // normalised, rotated, scaled by log2(e)/sqrt(D)
    float ow[NW][G][HEAD_DIM];        // per-warp V sums for the cross-warp reduction
    float po[G * MAXS * 8];           // merge: 8 dimensions of the slice of every chunk
    uint16_t kv_new[2][HEAD_DIM];     // the new position's k and v as stored (bf16)
    float hm[G], hl[G];               // per head: max score, sum of exp2(score - max)
    float pm[G][MAXS], pl[G][MAXS];   //        and (m, l) of every chunk of the kv head
    float sc[1];                      // scores / weights [G][cap], cap = the plan's score capacity
};
static_assert(offsetof(AttSmem<1>, po) % 16 == 0 && offsetof(AttSmem<2>, po) % 16 == 0 &&
                  offsetof(AttSmem<4>, po) % 16 == 0 && offsetof(AttSmem<1>, ow) % 16 == 0,
              "float4 merge reads stay aligned");
static_assert(sizeof(float) * HEAD_DIM % 16 == 0, "vector-accessed attention arrays stay 16-byte aligned");
static_assert(NC % 32 == 0, "a warp stages whole blocks of 32 values");
static_assert(NW >= 6, "the prologue needs G + 2 warps");

// Scores of the K rows of groups first, first + NW, ... of an item of n rows (group g: rows
// 4g + (lane >> 3); 8 lanes per row, 16 dims each: 8i..8i+7 and 64+8i..64+8i+7); lane i == h
// of the row's group writes head h's score to sc[h][base + row].  The caller rotates `first`
// from item to item, so that the groups of the whole chunk go round the warps evenly.
template <int G>
FQ_DEV void att_scores(const float (&q)[G][16], const uint8_t* kb, int n, int base, float* sc, int cap, int first,
                       int lane) {
    const int j = lane >> 3, i = lane & 7;
    for (int grp = first; 4 * grp < n; grp += NW) {
        const int row = 4 * grp + j;
        const bool valid = row < n;
        float s[G];
#pragma unroll
        for (int h = 0; h < G; ++h) s[h] = 0.f;
        if (valid) {
            const uint4 a = *reinterpret_cast<const uint4*>(kb + (size_t)row * 256 + 16 * i);
            const uint4 b = *reinterpret_cast<const uint4*>(kb + (size_t)row * 256 + 128 + 16 * i);
            const float k[16] = {bf_lo(a.x), bf_hi(a.x), bf_lo(a.y), bf_hi(a.y), bf_lo(a.z), bf_hi(a.z),
                                 bf_lo(a.w), bf_hi(a.w), bf_lo(b.x), bf_hi(b.x), bf_lo(b.y), bf_hi(b.y),
                                 bf_lo(b.z), bf_hi(b.z), bf_lo(b.w), bf_hi(b.w)};
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float t0 = 0.f, t1 = 0.f;
#pragma unroll
                for (int e = 0; e < 16; e += 2) ffma2(t0, t1, q[h][e], q[h][e + 1], k[e], k[e + 1]);
                s[h] = t0 + t1;
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            s[h] += __shfl_xor_sync(0xFFFFFFFFu, s[h], 4);
            s[h] += __shfl_xor_sync(0xFFFFFFFFu, s[h], 2);
            s[h] += __shfl_xor_sync(0xFFFFFFFFu, s[h], 1);
            if (valid && i == h) sc[h * cap + base + row] = s[h];
        }
    }
}

// V rows first, first + NW, ... of an item of n rows weighted by p = sc[h][base + row]: lane
// takes dims 4 lane .. 4 lane + 3 of every head (`first` rotates from item to item).
template <int G>
FQ_DEV void att_values(float (&acc)[G][4], const uint8_t* vb, int n, int base, const float* sc, int cap, int first,
                       int lane) {
    for (int row = first; row < n; row += NW) {
        const uint2 v = *reinterpret_cast<const uint2*>(vb + (size_t)row * 256 + 8 * lane);
        const float vf[4] = {bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y)};
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float p = sc[h * cap + base + row];
            ffma2(acc[h][0], acc[h][1], p, p, vf[0], vf[1]);
            ffma2(acc[h][2], acc[h][3], p, p, vf[2], vf[3]);
        }
    }
}

// ---------------------------------------------------------------- consumers: phases

// Shared scratch of the consumers besides the staging area.
struct CtlX {
    float wsum[NW];
};

// Stage an input vector of K values (times `gain` when given; its raw values into xr when
// asked), then quantise it into the 16-bit block fixed point of XStage; returns 1/rms when a
// gain is given, else 1.  src == null: the embedding row of `tok` instead of exchange words.
template <int FMT, int XB>
FQ_DEV float stage(const StreamArgs& a, const unsigned long long* src, int K, uint32_t tag,
                                   const float* gain, bool keep_raw, const XStage& x, float* xr, Cons& cs, CtlX& cx,
                                   int64_t tok = 0) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    csync();
    float ss = 0.f;
    auto put = [&](int i, float v0, float v1, float2 g) {
        ss += v0 * v0 + v1 * v1;
        if (keep_raw) *reinterpret_cast<float2*>(xr + i) = make_float2(v0, v1);
        *reinterpret_cast<float2*>(x.xs + i) = make_float2(v0 * g.x, v1 * g.y);
    };
    if (src) {
        if (!xw_read<XB>(src, K, tag, tid, NC, cs.stop, gain, put)) {
            if (cs.stop.seen()) cs.ctl.abort = 1;   // another CTA gave up
            else cs.fail(1024u);
        }
    } else {
        for (int i = 2 * tid; i < K; i += 2 * NC)
            put(i, dequant_one(a.emb, tok, i), dequant_one(a.emb, tok, i + 1),
                gain ? *reinterpret_cast<const float2*>(gain + i) : make_float2(1.f, 1.f));
    }
    // Blocks of 32 values, quantised by the warp that staged them: a warp's threads take 64
    // consecutive values per round (2 NC values apart), so warp w holds blocks 2w, 2w + 1,
    // then 2w + NC / 16, ... and needs no CTA barrier before quantising them.  8 lanes per
    // block, 4 values per lane; lanes 16-31 take the warp's next pair of blocks.
    __syncwarp();
    const int nblk = K >> 5;
    constexpr int BSTRIDE = NC / 16;   // blocks between a warp's rounds
    for (int base = 2 * warp; base < nblk; base += 2 * BSTRIDE) {
        const int blk = base + (lane >> 4) * BSTRIDE + ((lane >> 3) & 1), j = lane & 7;
        const bool on = blk < nblk;
        const float4 v = on ? reinterpret_cast<const float4*>(x.xs)[blk * 8 + j] : make_float4(0.f, 0.f, 0.f, 0.f);
        float am = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        float sm = (v.x + v.y) + (v.z + v.w);
        am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
        am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 4));
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 1);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 2);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 4);
        if (!on) continue;
        const float inv = am > 0.f ? 32767.f / am : 0.f;
        const float e[4] = {v.x, v.y, v.z, v.w};
        uint32_t hw = 0, lw = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q = max(-32767, min(32767, __float2int_rn(e[k] * inv)));
            hw |= (uint32_t)(q >> 8 & 0xFF) << (8 * k);
            lw |= (uint32_t)(q & 0xFF) << (8 * k);
        }
        const int at = xq_index<FMT>(blk * 32 + 4 * j, K);
        *reinterpret_cast<uint32_t*>(x.hi + at) = hw;
        *reinterpret_cast<uint32_t*>(x.lo + at) = lw;
        if (j == 0) {
            x.sc[blk] = am / 32767.f;
            if (FMT == FMT_Q4_K) x.sum32[blk] = sm;
        }
    }
    ss = warp_sum(ss);
    if (lane == 0) cx.wsum[warp] = ss;
    csync();   // every block quantised, every warp's sum of squares in
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) tot += cx.wsum[w];
    return gain ? rsqrtf(tot / (float)K + a.eps) : 1.f;
}

FQ_DEV uint32_t tag_of(uint32_t seq, int layer) { return (seq << 8) | (uint32_t)(layer + 1); }

// Attention of this CTA's unit plus the merge of its kv head's chunks (8 dims per slice).
// A StreamLayer copied word by word (by one warp) into shared memory.
FQ_DEV void copy_layer(StreamLayer& dst, const StreamLayer& src, int lane) {
    static_assert(sizeof(StreamLayer) % 4 == 0, "copied as 32-bit words");
    constexpr int NWD = (int)(sizeof(StreamLayer) / 4);
    for (int i = lane; i < NWD; i += 32)
        reinterpret_cast<uint32_t*>(&dst)[i] = reinterpret_cast<const uint32_t*>(&src)[i];
}

// `next`: the next layer's table entry, copied into shared memory by the last warp while
// the others wait for q, k and v (null after the last layer).
template <int G>
FQ_DEV void attention_phase(const StreamArgs& a, const StreamLayer& lw, int layer, const SeqState& ss, uint32_t tag,
                            Cons& cs, AttSmem<G>& as, const AttnUnit& u, const StreamLayer* next, StreamLayer* next_dst) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = a.S;
    csync();
    if (next && warp == NW - 1) copy_layer(*next_dst, *next, lane);
    if (u.active && warp < G + 2) {
        // q heads of the group, then k and v of the kv head, from the QKV exchange words
        const int row = warp < G ? (u.g * G + warp) : warp == G ? (a.Hq + u.g) : (a.Hq + a.Hkv + u.g);
        // the gains and rotations of this lane's dims first: their loads overlap the wait
        float gn[4] = {1.f, 1.f, 1.f, 1.f};
        float2 rot[4] = {};
        if (warp <= G) {
            const float* g = warp < G ? lw.q_norm : lw.k_norm;
            const float2* rope_row = a.rope + (size_t)ss.pos * (HEAD_DIM / 2);
            const float4 g4 = *reinterpret_cast<const float4*>(g + 4 * lane);
            gn[0] = g4.x; gn[1] = g4.y; gn[2] = g4.z; gn[3] = g4.w;
#pragma unroll
            for (int j = 0; j < 4; ++j) rot[j] = rope_row[(4 * lane + j) & 63];
        }
        float v[4];
        const unsigned long long* src = a.qkv + (size_t)row * HEAD_DIM + 4 * lane;
        const unsigned long long* const pp[2] = {src, src + 2};
        if (!xw_read_pairs<2>(pp, tag, cs.stop, v)) {
            if (cs.stop.seen()) cs.ctl.abort = 1;
            else cs.fail(2048u);
        }
        if (warp < G) {
            norm_rope4(v, gn, rot, a.eps, lane);
            const float qscale = 1.4426950408889634f * rsqrtf((float)HEAD_DIM);
#pragma unroll
            for (int j = 0; j < 4; ++j) as.qs[warp][4 * lane + j] = v[j] * qscale;
        } else {
            if (warp == G) norm_rope4(v, gn, rot, a.eps, lane);
            const int which = warp - G;   // 0: k, 1: v
            uint16_t* dst = reinterpret_cast<uint16_t*>(warp == G ? ss.k : ss.v) +
                            (((size_t)layer * a.Hkv + u.g) * (size_t)ss.cap + ss.pos) * HEAD_DIM;
            const bool owner = u.c == S - 1;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
                as.kv_new[which][4 * lane + j] = b;
                if (owner) dst[4 * lane + j] = b;
            }
        }
    }
    csync();
    if (cs.ctl.abort || !u.active) {
        // an inactive CTA carries no attention items
        return;
    }
    const int nt = u.nt;
    const int n = u.e - u.t0 > 0 ? u.e - u.t0 : 0;          // cached positions of the chunk
    const bool owns_new = u.c == S - 1;
    const int cap = a.score_cap;
    float* sc = as.sc;
    // ---- pass 1: scores of every position (K items), the new position last
    {
        float q[G][16];
        const int i = lane & 7;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                q[h][e] = as.qs[h][8 * i + e];
                q[h][8 + e] = as.qs[h][64 + 8 * i + e];
            }
        for (int t = 0; t < nt; ++t) {
            if (!cs.wait_full(lane)) break;
            const int rot = (warp - (t * (TP / 4)) % NW + NW) % NW;   // this warp's first group of item t
            att_scores<G>(q, cs.slot(), min(TP, n - t * TP), t * TP, sc, cap, rot, lane);
            cs.release(lane);
        }
        if (owns_new && warp == 0)
            att_scores<G>(q, reinterpret_cast<const uint8_t*>(as.kv_new[0]), 1, n, sc, cap, 0, lane);
    }
    csync();
    if (cs.ctl.abort) return;
    // ---- softmax over the chunk: warp h takes head h (base 2; q carries log2(e)/sqrt(D))
    const int npos = n + (owns_new ? 1 : 0);
    for (int h = warp; h < G; h += NW) {
        float* sh = sc + h * cap;
        float m = -INFINITY;
        for (int t = lane; t < npos; t += 32) m = fmaxf(m, sh[t]);
        m = warp_max(m);
        float l = 0.f;
        for (int t = lane; t < npos; t += 32) {
            const float p = exp2f(sh[t] - m);
            sh[t] = p;
            l += p;
        }
        l = warp_sum(l);
        if (lane == 0) {
            as.hm[h] = npos ? m : -INFINITY;
            as.hl[h] = l;
        }
    }
    csync();
    // ---- pass 2: weighted V rows (V items), the new position last
    float acc[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int d = 0; d < 4; ++d) acc[h][d] = 0.f;
    for (int t = 0; t < nt; ++t) {
        if (!cs.wait_full(lane)) break;
        const int rot = (warp - (t * TP) % NW + NW) % NW;   // this warp's first row of item t
        att_values<G>(acc, cs.slot(), min(TP, n - t * TP), t * TP, sc, cap, rot, lane);
        cs.release(lane);
    }
    if (owns_new && warp == 0)
        att_values<G>(acc, reinterpret_cast<const uint8_t*>(as.kv_new[1]), 1, n, sc, cap, 0, lane);
#pragma unroll
    for (int h = 0; h < G; ++h)
        *reinterpret_cast<float4*>(&as.ow[warp][h][4 * lane]) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
    csync();
    if (cs.ctl.abort) return;
    for (int t = tid; t < G * HEAD_DIM; t += NC) {
        const int h = t / HEAD_DIM, d = t % HEAD_DIM;
        float O = 0.f;
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) O += as.ow[ww][h][d];
        unsigned long long* p = a.part + ((size_t)(u.g * G + h) * S + u.c) * (HEAD_DIM + 2);
        if (d == 0) {
            xw_store(p, as.hm[h], tag);
            xw_store(p + 1, as.hl[h], tag);
        }
        xw_store(p + 2 + d, O, tag);
    }
    // ---- merge: slice sl (dims 8 sl .. 8 sl + 7) of the group's heads, slices u.c, u.c + S, ...
    for (int sl = u.c; sl < MSL; sl += S) {
        csync();
        if (cs.ctl.abort) return;
        for (int t = tid; t < G * S; t += NC) {
            const int h = t / S, c = t % S;
            const unsigned long long* p = a.part + ((size_t)(u.g * G + h) * S + c) * (HEAD_DIM + 2);
            float v[10];
            const unsigned long long* o8 = p + 2 + 8 * sl;
            const unsigned long long* const pp[5] = {p, o8, o8 + 2, o8 + 4, o8 + 6};
            if (!xw_read_pairs<5>(pp, tag, cs.stop, v)) {
                if (cs.stop.seen()) cs.ctl.abort = 1;
                else cs.fail(4096u);
            }
            as.pm[h][c] = v[0];
            as.pl[h][c] = v[1];
            float* po = &as.po[(h * S + c) * 8];
#pragma unroll
            for (int k = 0; k < 8; ++k) po[k] = v[2 + k];
        }
        csync();
        if (cs.ctl.abort) return;
        // warp h merges head h: lanes take chunks c = lane, lane + 32, ...; the maximum, the
        // weight of every chunk and the 9 weighted sums are warp reductions
        if (warp < G) {
            const int h = warp;
            float M = -INFINITY;
            for (int c = lane; c < S; c += 32) M = fmaxf(M, as.pm[h][c]);
            M = warp_max(M);
            float Lsum = 0.f, O[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int c = lane; c < S; c += 32) {
                const float m = as.pm[h][c];
                if (m == -INFINITY) continue;
                const float wgt = exp2f(m - M);
                Lsum = fmaf(as.pl[h][c], wgt, Lsum);
                const float4 p0 = *reinterpret_cast<const float4*>(&as.po[(h * S + c) * 8]);
                const float4 p1 = *reinterpret_cast<const float4*>(&as.po[(h * S + c) * 8 + 4]);
                O[0] = fmaf(p0.x, wgt, O[0]); O[1] = fmaf(p0.y, wgt, O[1]);
                O[2] = fmaf(p0.z, wgt, O[2]); O[3] = fmaf(p0.w, wgt, O[3]);
                O[4] = fmaf(p1.x, wgt, O[4]); O[5] = fmaf(p1.y, wgt, O[5]);
                O[6] = fmaf(p1.z, wgt, O[6]); O[7] = fmaf(p1.w, wgt, O[7]);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                Lsum += __shfl_xor_sync(0xFFFFFFFFu, Lsum, off);
#pragma unroll
                for (int k = 0; k < 8; ++k) O[k] += __shfl_xor_sync(0xFFFFFFFFu, O[k], off);
            }
            if (lane < 8) {
                float o = O[0];
#pragma unroll
                for (int k = 1; k < 8; ++k) o = lane == k ? O[k] : o;
                xw_store(a.o + (size_t)(u.g * G + h) * HEAD_DIM + 8 * sl + lane, o / Lsum, tag);
            }
        }
    }
}

}  // namespace

// XB: exchange words a staging thread polls per batch (xw_read)
template <int FMT, int G, int XB>
__global__ void __launch_bounds__(NTH, 1) stream_step_kernel(const __grid_constant__ StreamArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ Ctl ctl;
    __shared__ CtlX cx;
    __shared__ ProjPlan pp[NPROJ];
    __shared__ AttnUnit au;
    __shared__ StreamLayer sl[2];   // this layer's and the next layer's table entries
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.lay_bars);
    Ring ring{smem, bars, bars + MAXSLOT, a.nslot};
    float* xs = reinterpret_cast<float*>(smem + a.lay_xs);
    XStage xq;
    xq.xs = xs;
    xq.hi = reinterpret_cast<int8_t*>(smem + a.lay_xq);
    xq.lo = reinterpret_cast<uint8_t*>(smem + a.lay_xq + a.kmax);
    xq.sc = reinterpret_cast<float*>(smem + a.lay_xq + 2 * a.kmax);
    xq.sum32 = xq.sc + a.kmax / 32;
    float* xr = reinterpret_cast<float*>(smem + a.lay_xr);
    float* red = reinterpret_cast<float*>(smem + a.lay_red);
    if (tid == 0) {
        for (int s = 0; s < a.nslot; ++s) {
            mbar_init(&ring.full[s], 1);
            mbar_init(&ring.empty[s], NW);
        }
        mbar_fence_init();
        ctl.abort = 0;
        ctl.best = 0ull;
        ctl.last = 0;
        au = attn_unit_of(a.Hkv, a.S, a.st->seq[0].pos);
    }
    if (tid < NPROJ) pp[tid] = a.plan[blockIdx.x * NPROJ + tid];
    if (warp == NW - 1) copy_layer(sl[0], a.layers[0], lane);
    __syncthreads();
    const uint32_t seq = ld_volatile(&a.ctl[1]) & 0xFFFFFFu;
    const Stop stop{a.ctl + 2, seq + 1u};
    if (warp == NW) {
        if (lane == 0) produce(a, ring, &ctl.abort, stop, pp, au);
        return;
    }

    const SeqState ss = a.st->seq[0];
    const int64_t tok = (ss.token >= 0 && ss.token < a.emb.N) ? ss.token : 0;
    Cons cs{ring, ctl, a.err, stop};
    AttSmem<G>& as = *reinterpret_cast<AttSmem<G>*>(xs);

    // The step as one loop over phases, so that every phase body exists once in the code:
    // q = 5 L + {0: RMSNorm + QKV, 1: attention, 2: O + residual, 3: RMSNorm + gate_up +
    // SwiGLU, 4: down + residual}; q = 5 n_layers: final RMSNorm + LM head.
    // A flag set by one warp is read only after a barrier that every warp passes, so that all
    // warps leave the loop at the same phase.
    const int nq = 5 * a.n_layers + (a.head ? 1 : 0);
    float inv = 1.f;
    for (int q = 0; q < nq; ++q) {
        const int L = q / 5, ph = q - 5 * L;
        const bool lm = L == a.n_layers;
        const StreamLayer& lw = sl[lm ? 0 : (L & 1)];   // the layer's table entry, in shared memory
        const uint32_t tag = tag_of(seq, L);
        if (ph == 1) {
            const bool more = L + 1 < a.n_layers;
            attention_phase<G>(a, lw, L, ss, tag, cs, as, au, more ? &a.layers[L + 1] : nullptr, &sl[(L + 1) & 1]);
            csync();
            if (ctl.abort) break;
            continue;
        }
        // ---- a projection phase: its matrix, input, gain and plan
        const int j = lm ? P_LM : ph == 0 ? P_QKV : ph == 2 ? P_O : ph == 3 ? P_GU : P_DN;
        const QMat& W = lm ? a.out : ph == 0 ? lw.qkv : ph == 2 ? lw.o : ph == 3 ? lw.gate_up : lw.down;
        const unsigned long long* src = lm ? a.xf : ph == 0 ? (L == 0 ? nullptr : a.xf) : ph == 2 ? a.o
                                                                                               : ph == 3 ? a.xa : a.h;
        const uint32_t tag_in = (lm || ph == 0) ? tag_of(seq, L - 1) : tag;
        const float* gain = lm ? a.out_norm : ph == 0 ? lw.attn_norm : ph == 3 ? lw.ffn_norm : nullptr;
        const bool keep_raw = ph == 0 || ph == 3;   // the residual for the next add
        const float inv_p = stage<FMT, XB>(a, src, W.K, tag_in, gain, keep_raw, xq, xr, cs, cx, tok);
        if (gain) inv = inv_p;
        if (ctl.abort) break;
        const ProjPlan& P = pp[j];
        const bool pairs = ph == 3 && !lm;   // gate/up rows come in pairs
        unsigned long long kb = 0ull;
        auto emit = [&](int r, float y, float y2) {
            if (lm) {
                y *= inv;
                if (a.logits) a.logits[r] = y;
                const unsigned long long key = argmax_key(y, (uint32_t)r);
                kb = key > kb ? key : kb;
            } else if (ph == 0) {
                xw_store(a.qkv + r, y * inv, tag);
            } else if (ph == 2) {
                xw_store(a.xa + r, xr[r] + y, tag);
            } else if (ph == 3) {
                xw_store(a.h + r / 2, silu(y * inv) * (y2 * inv), tag);
            } else {
                const float xn = xr[r] + y;
                xw_store(a.xf + r, xn, tag);
                if (a.trace_x) a.trace_x[(size_t)L * a.H + r] = xn;
            }
        };
        const bool direct = P.kparts == 1 && !(pairs && (P.rs & 1));
        if (!proj_tasks<FMT>(cs, W, P, xq, red, direct, pairs, emit)) ctl.abort = 1;
        const int kparts = P.kparts;
        if (!direct) {
            // ---- the epilogue over this CTA's rows after the partial sums
            csync();
            if (ctl.abort) break;
            const int step = pairs ? 2 : 1;
            for (int r = P.r0 + step * tid; r < P.r1; r += step * NC) {
                float y = 0.f, y2 = 0.f;
                for (int k = 0; k < kparts; ++k) y += red[(r - P.r0) * kparts + k];
                if (pairs)
                    for (int k = 0; k < kparts; ++k) y2 += red[(r + 1 - P.r0) * kparts + k];
                emit(r, y, y2);
            }
        }
        // direct: the rows were finished in the tasks; the next phase's first barrier
        // orders them before its writes to shared memory, and reads the flag after it
        if (lm && a.greedy) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, kb, o);
                kb = other > kb ? other : kb;
            }
            if (lane == 0 && kb) atomicMax(&ctl.best, kb);
        }
    }

    // ---- finishing ticket: the last CTA hands the greedy token on and advances the launch
    // sequence (every CTA takes it, also after a failure, so the sequence stays in step)
    csync();
    if (tid == 0) {
        StepState* st = a.st;
        if (a.greedy && ctl.best) atomicMax(&st->keys[0], ctl.best);
        __threadfence();
        const uint32_t t = atomicAdd(&a.ctl[0], 1u);
        if (t == gridDim.x - 1) {
            __threadfence();
            a.ctl[0] = 0u;
            if (a.greedy) {
                const unsigned long long k = atomicExch(&st->keys[0], 0ull);
                const uint32_t idx = argmax_key_index(k);
                const int32_t tk = idx < (uint32_t)a.V ? (int32_t)idx : 0;
                st->seq[0].token = tk;
                st->seq[0].pos += 1;
                if (st->tokens_out) st->tokens_out[st->step] = tk;
                st->step += 1;
            }
            __threadfence();
            atomicAdd(&a.ctl[1], 1u);
        }
    }
}

namespace {

int g_sms_s = 0;
int g_optin_s = 0;

template <int FMT, int G, int XB>
bool launch_fg(const StreamArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g_sms_s);
    cfg.blockDim = dim3(NTH);
    cfg.dynamicSmemBytes = a.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stream_step_kernel<FMT, G, XB>, a) == cudaSuccess;
}

template <int FMT, int G, int XB>
void prepare_one() {
    cudaFuncAttributes fa;
    cudaFuncGetAttributes(&fa, stream_step_kernel<FMT, G, XB>);
    cudaFuncSetAttribute(stream_step_kernel<FMT, G, XB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         g_optin_s - (int)fa.sharedSizeBytes);
}

template <int FMT, int G>
void prepare_fg() {
    prepare_one<FMT, G, 4>();
    prepare_one<FMT, G, 8>();
}

// Exchange words per staging batch: four while the largest staged input needs at most two
// batches of four per thread (the smaller kernel measured faster on the 0.6B step), else
// eight (fewer round trips: 1.855 against 1.819 ms on the 8B Q4_K step, whose down
// projection stages 12288 values).
template <int FMT, int G>
bool launch_fb(const StreamArgs& a, cudaStream_t s) {
    return a.kmax <= 16 * NC ? launch_fg<FMT, G, 4>(a, s) : launch_fg<FMT, G, 8>(a, s);
}

}  // namespace

void stream_prepare() {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms_s, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&g_optin_s, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    prepare_fg<FMT_Q8_0, 1>();
    prepare_fg<FMT_Q8_0, 2>();
    prepare_fg<FMT_Q8_0, 4>();
    prepare_fg<FMT_Q4_K, 1>();
    prepare_fg<FMT_Q4_K, 2>();
    prepare_fg<FMT_Q4_K, 4>();
}

int stream_ctas() { return g_sms_s; }

int stream_chunks(int Hkv) { return g_sms_s > 0 && Hkv > 0 ? g_sms_s / Hkv : 0; }

bool stream_plan(StreamArgs& a, const StreamLayer& l0, int fmt, int G, std::vector<ProjPlan>& plans) {
    if (g_sms_s == 0 || a.S < 1 || a.S > MAXS) return false;
    {
        const int R = fmt == FMT_Q8_0 ? PCfg<FMT_Q8_0>::R : PCfg<FMT_Q4_K>::R;
        const int UE = fmt == FMT_Q8_0 ? PCfg<FMT_Q8_0>::UE : PCfg<FMT_Q4_K>::UE;
        const QMat* mats[NPROJ] = {&l0.qkv, &l0.o, &l0.gate_up, &l0.down, &a.out};
        plans.assign((size_t)g_sms_s * NPROJ, ProjPlan{});
        for (int c = 0; c < g_sms_s; ++c)
            for (int j = 0; j < NPROJ; ++j) {
                const QMat& W = *mats[j];
                ProjPlan& q = plans[(size_t)c * NPROJ + j];
                row_range(W.N, j == P_GU, c, g_sms_s, q.r0, q.r1);
                q.rs = rows_per_item(W);
                if (q.rs < 1) return false;   // a row must fit one slot
                q.U = W.K / UE;
                const Split sp = choose_split(q.r0, q.r1, q.rs, R, q.U);
                q.kparts = sp.kparts;
                q.up = sp.up;
            }
    }
    const int kmax = std::max({a.H, a.F, a.Hq * HEAD_DIM});
    int red = 0;   // floats of per-(row, K part) partial sums: the largest share of a CTA
    for (const ProjPlan& q : plans)
        if (q.r1 > q.r0) red = std::max(red, (q.r1 - q.r0) * q.kparts);
    // scores of one chunk: its cached positions (at most ceil(max_pos / S)) and the new one
    a.score_cap = (a.max_pos + a.S - 1) / a.S + 2;
    size_t att = 0;
    switch (G) {
        case 1: att = sizeof(AttSmem<1>); break;
        case 2: att = sizeof(AttSmem<2>); break;
        case 4: att = sizeof(AttSmem<4>); break;
        default: return false;
    }
    att += (size_t)G * a.score_cap * sizeof(float);
    const int xs_bytes = std::max(kmax * 4, (int)att);               // float staging / attention scratch
    const int xq_bytes = 2 * kmax + 2 * (kmax / 32) * 4;              // hi, lo planes; block scales and sums
    const int fixed = align_up(xs_bytes, 16) + align_up(xq_bytes, 16) + align_up(a.H * 4, 16) +
                      align_up(red * 4, 16) + 2 * MAXSLOT * 8;
    const int avail = g_optin_s - 1024 - fixed;   // static shared memory of the kernel
    const int nslot = std::min(MAXSLOT, avail / SLOT);
    if (nslot < 4) return false;
    a.nslot = nslot;
    a.kmax = kmax;
    a.lay_xs = nslot * SLOT;
    a.lay_xq = a.lay_xs + align_up(xs_bytes, 16);
    a.lay_xr = a.lay_xq + align_up(xq_bytes, 16);
    a.lay_red = a.lay_xr + align_up(a.H * 4, 16);
    a.lay_bars = a.lay_red + align_up(red * 4, 16);
    a.smem_bytes = a.lay_bars + 2 * MAXSLOT * 8;
    return true;
}

bool launch_stream(const StreamArgs& a, int fmt, int G, cudaStream_t s) {
    if (g_sms_s == 0) return false;
    if (fmt == FMT_Q8_0) {
        switch (G) {
            case 1: return launch_fb<FMT_Q8_0, 1>(a, s);
            case 2: return launch_fb<FMT_Q8_0, 2>(a, s);
            case 4: return launch_fb<FMT_Q8_0, 4>(a, s);
        }
    } else if (fmt == FMT_Q4_K) {
        switch (G) {
            case 1: return launch_fb<FMT_Q4_K, 1>(a, s);
            case 2: return launch_fb<FMT_Q4_K, 2>(a, s);
            case 4: return launch_fb<FMT_Q4_K, 4>(a, s);
        }
    }
    return false;
}

}  // namespace fq
