// Lockstep batch decode GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Section 14.2 of the fucina pages: forwardStepBatch runs the dense trunk as one m = n pass
// so that every weight is read once for all streams.  With n = 8..32 rows the contraction
// y[b][r] = sum_k W[r][k] x[b][k] is dense enough for tensor cores, so it runs "swap-AB":
//   D[r, c] = sum_k A[r, k] B[c, k],  A = dequantised weight tile (M = 128 rows, f16),
//                                     B = activations, N = 2 * BP columns (f16).
// Nothing is rounded beyond f32 accuracy:
//   * activation row b is split into a high part hi = f16(x) (column b) and a low part
//     lo = f16(x - hi) (column BP + b), about 22 significant bits together;
//   * a Q8_0 weight d * q (int8 q, fp16 d) has at most 18 significant bits and is carried as
//     two f16 tiles, Wh = f16(q d) and Wl = q d - Wh (exact: one fused multiply-add in f16),
//   * D = Wh [hi lo] + Wl [hi lo] accumulates in f32 in tensor memory, y = D[:, b] + D[:, BP+b].
//
// Work split (stream-K): the (row tile, 64-element K chunk) iterations of the matrix are
// cut into one contiguous, equal range per CTA (one CTA per SM).  A tile whose chunks all
// fall to one CTA is finished in place; a tile split between CTAs is finished by the last of
// them to arrive (atomic ticket per tile and epilogue warp, no waiting), which adds the
// partial sums in CTA order, so results do not depend on timing.
//
// Roles in a CTA (448 threads):
//   warp 13     TMA producer: per chunk, the 128 x 64 code box (64-byte swizzle) and the
//               activation box (2BP x 64 halves, 128-byte swizzle = the MMA's K-major layout)
//               into a 6-slot ring;
//   warps 0-7   converters: thread (row, half) turns 32 codes into exact Wh / Wl halves and
//               writes them into the 128-byte swizzled A tiles (3-slot ring);
//   warp 12     one thread issues 2 x 4 tcgen05.mma (K = 16) per chunk into one of two
//               tensor-memory accumulators and commits the slots back;
//   warps 8-11  epilogue: tcgen05.ld of the accumulator (one row per thread), hi + lo, then
//               store / residual add / SwiGLU (gate, up rows adjacent) / logits + argmax.
// Every mbarrier wait is bounded; a stuck pipeline sets the error word and unwinds.

#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace fq {

namespace {

constexpr int TM = 128;                  // MMA M: weight rows per tile
constexpr int KCH = 64;                  // K elements per chunk: one 128-byte f16 swizzle atom
constexpr int RS = 6;                    // raw slots: codes + activations
constexpr int AS = 3;                    // converted weight slots: Wh + Wl
constexpr int CODE_BYTES = TM * KCH;     // 8 KB
constexpr int XB_BYTES = 64 * KCH * 2;   // 8 KB (N <= 64)
constexpr int RAW_BYTES = CODE_BYTES + XB_BYTES;
constexpr int A_TILE = TM * KCH * 2;     // 16 KB per f16 tile
constexpr int CONV_WARPS = 8, EPI_WARP0 = 8, MMA_WARP = 12, TMA_WARP = 13;
constexpr int TC_THREADS = 14 * 32;
constexpr uint32_t TMEM_COLS = 128;      // two accumulators of up to 64 columns
constexpr size_t TC_SMEM = (size_t)RS * RAW_BYTES + (size_t)AS * 2 * A_TILE + 1024 + 256;

struct TcArgs {
    alignas(64) unsigned long long mapq[16];   // codes [N][K] u8, box 64 x 128, 64-byte swizzle
    alignas(64) unsigned long long mapx[16];   // activations [2BP][K] f16, box 64 x 2BP, 128-byte swizzle
    QMat W;              // Q8_0 [N][K], K % 64 == 0
    int B;               // activation rows (<= BP)
    float* y;
    int y_stride;
    int epi;
    StepState* st;
    uint32_t* err;
    float* part;         // [grid][2][128][BP] partial sums of split tiles
    uint32_t* tickets;   // [4 * tiles] arrivals per (tile, epilogue warp), zero between uses
};

// iterations are (tile, chunk) pairs in tile-major order; total < 2^31 / G is checked on launch
FQ_DEV int iter_begin(int c, int total, int G) { return (int)((unsigned)(c * total) / (unsigned)G); }
// the CTA whose range holds iteration i
FQ_DEV int cta_of(int i, int total, int G) { return (int)((unsigned)((i + 1) * G + total - 1) / (unsigned)total) - 1; }

// (tile, chunk) of consecutive iterations without divisions in the loop
struct Cursor {
    int tile, chunk, nch;
    FQ_DEV Cursor(int it, int n) : tile(it / n), chunk(it % n), nch(n) {}
    FQ_DEV void next() {
        if (++chunk == nch) {
            chunk = 0;
            ++tile;
        }
    }
};

// two int8 codes (bytes 2p, 2p+1 of w, already offset by +128) -> exact f16 pair
FQ_DEV __half2 codes_to_h2(uint32_t w_biased, int p) {
    const uint32_t u = __byte_perm(w_biased, 0x64u, p == 0 ? 0x4140u : 0x4342u);   // 0x64XX: 1024 + q + 128
    return __hsub2(*reinterpret_cast<const __half2*>(&u), __floats2half2_rn(1152.f, 1152.f));
}

template <int BP>
__global__ void __launch_bounds__(TC_THREADS, 1) gemm_tc_kernel(const __grid_constant__ TcArgs a) {
    constexpr int NCOL = 2 * BP;         // MMA N
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* raw = smem;                                        // [RS][codes 8 KB | activations 8 KB]
    uint8_t* At = raw + (size_t)RS * RAW_BYTES;                 // [AS][Wh 16 KB | Wl 16 KB]
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(At + (size_t)AS * 2 * A_TILE);
    uint64_t* raw_empty = raw_full + RS;
    uint64_t* a_full = raw_empty + RS;
    uint64_t* a_empty = a_full + AS;
    uint64_t* acc_full = a_empty + AS;   // [2]
    uint64_t* acc_free = acc_full + 2;   // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_free + 2);
    __shared__ unsigned long long best[32];

    const QMat& W = a.W;
    const int N = W.N, K = W.K;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, c = blockIdx.x;
    const int nch = K / KCH, n_tiles = (N + TM - 1) / TM;
    const int total = n_tiles * nch;
    const int beg = iter_begin(c, total, G), end = iter_begin(c + 1, total, G);
    const int n_it = end - beg;

    if (tid == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], 1);
        }
        for (int s = 0; s < AS; ++s) {
            mbar_init(&a_full[s], CONV_WARPS);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_free[s], 4);
        }
        mbar_fence_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (tid < 32) best[tid] = 0ull;
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    pdl_trigger();
    pdl_wait();

    if (warp == TMA_WARP) {
        // ---------------- producer
        int issued = 0;
        Cursor cur(beg, nch);
        for (int i = 0; i < n_it; ++i, cur.next()) {
            const int tile = cur.tile, chunk = cur.chunk;
            const int s = i % RS;
            if (!mbar_wait(&raw_empty[s], ((uint32_t)(i / RS) & 1u) ^ 1u)) {
                if (a.err && lane == 0) atomicOr(a.err, 2u);
                break;
            }
            if (lane == 0) {
                uint8_t* slot = raw + (size_t)s * RAW_BYTES;
                mbar_arrive_expect_tx(&raw_full[s], (uint32_t)(CODE_BYTES + NCOL * KCH * 2));
                tma_load_2d(slot, a.mapq, chunk * KCH, tile * TM, &raw_full[s]);
                tma_load_2d(slot + CODE_BYTES, a.mapx, chunk * KCH, 0, &raw_full[s]);
            }
            __syncwarp();
            issued = i + 1;
        }
        // no copy may still be landing when the CTA exits (only possible after a timeout)
        for (int i = issued > RS ? issued - RS : 0; i < issued; ++i) mbar_wait(&raw_full[i % RS], (uint32_t)(i / RS) & 1u);
    } else if (warp < CONV_WARPS) {
        // ---------------- converters: thread (row rr, half h) owns K elements 32h..32h+31
        const int rr = (warp & 3) * 32 + lane, h = warp >> 2;
        // fp16 scale of (row, 32-element block) for iteration i, fetched four chunks ahead
        Cursor ahead(beg, nch);   // the iteration whose scale is fetched next
        int ia = 0;
        auto next_scale = [&]() -> uint32_t {
            uint32_t v = 0u;
            const int row = ahead.tile * TM + rr;
            if (ia < n_it && row < N) v = (uint32_t)__ldg(W.s + (size_t)row * (K / 32) + ahead.chunk * 2 + h);
            ++ia;
            ahead.next();
            return v;
        };
        // one chunk: wait for its codes and a free A slot, write Wh / Wl; false on a timeout
        auto convert = [&](int i, uint32_t sc) -> bool {
            const int s = i % RS, as = i % AS;
            if (!mbar_wait(&raw_full[s], (uint32_t)(i / RS) & 1u) ||
                !mbar_wait(&a_empty[as], ((uint32_t)(i / AS) & 1u) ^ 1u)) {
                if (a.err && lane == 0) atomicOr(a.err, 4u);
                return false;
            }
            // codes of row rr, logical 16-byte chunks 2h, 2h+1 (64-byte swizzle: chunk ^ bits 1-2 of the row)
            const uint8_t* crow = raw + (size_t)s * RAW_BYTES + rr * 64;
            const int sw = (rr >> 1) & 3;
            uint4 q[2];
            q[0] = *reinterpret_cast<const uint4*>(crow + (((2 * h) ^ sw) << 4));
            q[1] = *reinterpret_cast<const uint4*>(crow + (((2 * h + 1) ^ sw) << 4));
            const unsigned short dbits = (unsigned short)sc;
            const __half dh = *reinterpret_cast<const __half*>(&dbits);
            const __half2 d2 = __halves2half2(dh, dh);
            uint8_t* Ah = At + (size_t)as * 2 * A_TILE;
            uint8_t* Al = Ah + A_TILE;
#pragma unroll
            for (int j = 0; j < 4; ++j) {        // 16-byte output chunk 4h + j: K elements 32h + 8j ..
                const uint4 qv = q[j >> 1];
                const uint32_t w0 = ((j & 1) ? qv.z : qv.x) ^ 0x80808080u;
                const uint32_t w1 = ((j & 1) ? qv.w : qv.y) ^ 0x80808080u;
                __half2 qh[4] = {codes_to_h2(w0, 0), codes_to_h2(w0, 1), codes_to_h2(w1, 0), codes_to_h2(w1, 1)};
                __half2 hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    hi[e] = __hmul2(qh[e], d2);
                    lo[e] = __hfma2(qh[e], d2, __hneg2(hi[e]));
                }
                const uint32_t off = sw128_offset(rr, 4 * h + j);
                *reinterpret_cast<uint4*>(Ah + off) = *reinterpret_cast<const uint4*>(hi);
                *reinterpret_cast<uint4*>(Al + off) = *reinterpret_cast<const uint4*>(lo);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[as]);
            return true;
        };
        // four scale registers in a static rotation: each is refilled right after its use and
        // read again four chunks later, so a scale load's latency hides behind three chunks
        uint32_t sc0 = next_scale(), sc1 = next_scale(), sc2 = next_scale(), sc3 = next_scale();
        for (int i = 0; i < n_it; i += 4) {
            if (!convert(i, sc0)) break;
            sc0 = next_scale();
            if (i + 1 >= n_it || !convert(i + 1, sc1)) break;
            sc1 = next_scale();
            if (i + 2 >= n_it || !convert(i + 2, sc2)) break;
            sc2 = next_scale();
            if (i + 3 >= n_it || !convert(i + 3, sc3)) break;
            sc3 = next_scale();
        }
    } else if (warp == MMA_WARP) {
        // ---------------- MMA issue: one thread
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(TM, NCOL);
            int t = 0;   // segment (tile) counter
            int last = -1;   // last iteration whose MMAs were issued
            bool ok = true;
            int chunk0 = beg % nch;
            for (int i = 0; i < n_it && ok; chunk0 = 0) {
                const int len = min(nch - chunk0, n_it - i);
                const int slot = t & 1;
                if (!mbar_wait(&acc_free[slot], ((uint32_t)(t >> 1) & 1u) ^ 1u)) {
                    if (a.err) atomicOr(a.err, 8u);
                    break;
                }
                tc_fence_after();
                const uint32_t dacc = tbase + (uint32_t)(slot * 64);
                for (int j = 0; j < len; ++j, ++i) {
                    const int s = i % RS, as = i % AS;
                    if (!mbar_wait(&a_full[as], (uint32_t)(i / AS) & 1u) ||
                        !mbar_wait(&raw_full[s], (uint32_t)(i / RS) & 1u)) {
                        if (a.err) atomicOr(a.err, 16u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ah = smem_u32(At + (size_t)as * 2 * A_TILE);
                    const uint64_t dh = sdesc_sw128(ah), dl = sdesc_sw128(ah + A_TILE);
                    const uint64_t bd = sdesc_sw128(smem_u32(raw + (size_t)s * RAW_BYTES + CODE_BYTES));
#pragma unroll
                    for (int k = 0; k < KCH / 16; ++k)   // 32 bytes of K per MMA: start address + 2 (x16 B)
                        mma_f16(dacc, dh + 2 * k, bd + 2 * k, idesc, (j > 0 || k > 0) ? 1u : 0u);
#pragma unroll
                    for (int k = 0; k < KCH / 16; ++k) mma_f16(dacc, dl + 2 * k, bd + 2 * k, idesc, 1u);
                    mma_commit(&a_empty[as]);
                    mma_commit(&raw_empty[s]);
                    last = i;
                }
                if (ok) mma_commit(&acc_full[slot]);
                ++t;
            }
            // every issued MMA has finished before the accumulators are released
            if (last >= 0) mbar_wait(&raw_empty[last % RS], (uint32_t)(last / RS) & 1u);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: TMEM lanes 32q..32q+31 <-> tile rows
        const int q = warp - EPI_WARP0;
        const int rin = 32 * q + lane;
        int t = 0;
        int tile = beg / nch, chunk0 = beg % nch;
        for (int i = 0; i < n_it; ++t, ++tile, chunk0 = 0) {
            const int g0 = beg + i;
            const int len = min(nch - chunk0, n_it - i);
            i += len;
            const int slot = t & 1;
            if (!mbar_wait(&acc_full[slot], (uint32_t)(t >> 1) & 1u)) {
                if (a.err && lane == 0) atomicOr(a.err, 32u);
                break;
            }
            tc_fence_after();
            uint32_t v[NCOL];
#pragma unroll
            for (int c4 = 0; c4 < NCOL / 16; ++c4)
                tmem_ld16(tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)(slot * 64 + 16 * c4), v + 16 * c4);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_free[slot]);
            const int row = tile * TM + rin;
            const bool ok_row = row < N;
            float val[BP];
#pragma unroll
            for (int b = 0; b < BP; ++b) val[b] = __uint_as_float(v[b]) + __uint_as_float(v[BP + b]);
            const int tb = tile * nch;
            const int c_first = cta_of(tb, total, G), c_last = cta_of(tb + nch - 1, total, G);
            if (c_first != c_last) {
                // split tile: partial -> scratch; the last contributor adds them up in CTA order
                const int which = (g0 == beg) ? 0 : 1;
                float4* pp = reinterpret_cast<float4*>(a.part + (((size_t)c * 2 + which) * TM + rin) * BP);
#pragma unroll
                for (int b = 0; b < BP; b += 4) pp[b / 4] = make_float4(val[b], val[b + 1], val[b + 2], val[b + 3]);
                __threadfence();
                __syncwarp();
                uint32_t prev = 0u;
                if (lane == 0) {
                    prev = atomicAdd(&a.tickets[4 * tile + q], 1u);
                    if (prev == (uint32_t)(c_last - c_first)) a.tickets[4 * tile + q] = 0u;
                }
                prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
                if (prev != (uint32_t)(c_last - c_first)) continue;
                __threadfence();
#pragma unroll
                for (int b = 0; b < BP; ++b) val[b] = 0.f;
                for (int cc = c_first; cc <= c_last; ++cc) {
                    const int wh = (iter_begin(cc, total, G) >= tb) ? 0 : 1;   // cc starts inside this tile
                    const float4* src = reinterpret_cast<const float4*>(a.part + (((size_t)cc * 2 + wh) * TM + rin) * BP);
#pragma unroll
                    for (int b = 0; b < BP; b += 4) {
                        const float4 f = __ldcg(src + b / 4);
                        val[b] += f.x;
                        val[b + 1] += f.y;
                        val[b + 2] += f.z;
                        val[b + 3] += f.w;
                    }
                }
            }
            unsigned long long kb[BP];
#pragma unroll
            for (int b = 0; b < BP; ++b) {
                kb[b] = 0ull;
                if (a.epi == EPI_SWIGLU) {
                    const float up = __shfl_xor_sync(0xFFFFFFFFu, val[b], 1);
                    if (b < a.B && ok_row && (rin & 1) == 0 && row + 1 < N)
                        a.y[(size_t)b * a.y_stride + (row >> 1)] = silu(val[b]) * up;
                } else if (b < a.B && ok_row) {
                    float* yp = a.y + (size_t)b * a.y_stride + row;
                    if (a.epi == EPI_ADD) *yp += val[b];
                    else *yp = val[b];
                    if (a.epi == EPI_LOGITS) kb[b] = argmax_key(val[b], (uint32_t)row);
                }
            }
            if (a.epi == EPI_LOGITS) {
#pragma unroll
                for (int b = 0; b < BP; ++b) {
                    unsigned long long k = kb[b];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        unsigned long long ok2 = __shfl_xor_sync(0xFFFFFFFFu, k, o);
                        k = ok2 > k ? ok2 : k;
                    }
                    if (lane == 0 && b < a.B) atomicMax(&best[b], k);
                }
            }
        }
    }
    __syncthreads();
    if (a.epi == EPI_LOGITS && tid < a.B) atomicMax(&a.st->keys[tid], best[tid]);
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tbase, TMEM_COLS);
    }
}

// x (optionally RMSNorm-ed with gain g) -> f16 high / low rows for the MMA B operand;
// rows B..BP-1 are zero.  Grid (BP, K slices of XK elements): each CTA converts one slice of
// one row (the RMS of the whole row is recomputed per CTA, from L2).
constexpr int XK = 2048;
__global__ void __launch_bounds__(256) prep_xh_kernel(const float* x, int x_stride, int B, int BP, int K,
                                                      const float* g, float eps, __half* xh) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[32];
    const int b = blockIdx.x;
    const int k0 = blockIdx.y * XK, k1 = min(K, k0 + XK);
    __half* hi = xh + (size_t)b * K;
    __half* lo = xh + (size_t)(BP + b) * K;
    if (b >= B) {
        for (int k = k0 + 4 * threadIdx.x; k < k1; k += 4 * blockDim.x) {
            *reinterpret_cast<uint2*>(hi + k) = make_uint2(0u, 0u);
            *reinterpret_cast<uint2*>(lo + k) = make_uint2(0u, 0u);
        }
        return;
    }
    const float* xr = x + (size_t)b * x_stride;
    float inv = 1.f;
    if (g) {
        float ss = 0.f;
        for (int k = 4 * threadIdx.x; k < K; k += 4 * blockDim.x) {
            const float4 v = *reinterpret_cast<const float4*>(xr + k);
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = block_sum(ss, red);
        inv = rsqrtf(ss / (float)K + eps);
    }
    for (int k = k0 + 4 * threadIdx.x; k < k1; k += 4 * blockDim.x) {
        float4 v = *reinterpret_cast<const float4*>(xr + k);
        if (g) {
            const float4 gg = *reinterpret_cast<const float4*>(g + k);
            v.x = v.x * inv * gg.x; v.y = v.y * inv * gg.y; v.z = v.z * inv * gg.z; v.w = v.w * inv * gg.w;
        }
        const __half2 h01 = __floats2half2_rn(v.x, v.y), h23 = __floats2half2_rn(v.z, v.w);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        const __half2 l01 = __floats2half2_rn(v.x - f01.x, v.y - f01.y), l23 = __floats2half2_rn(v.z - f23.x, v.w - f23.y);
        *reinterpret_cast<uint2*>(hi + k) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
        *reinterpret_cast<uint2*>(lo + k) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
    }
}

int g_sms_tc = 0;

template <int BP>
void launch_bp(const TcArgs& t, cudaStream_t s, bool pdl) {
    const long long total = (long long)((t.W.N + TM - 1) / TM) * (t.W.K / KCH);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<long long>(total, g_sms_tc));   // total * grid < 2^31: see applicable
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = TC_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BP>, t);
}

}  // namespace

void gemm_tc_prepare() {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms_tc, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(gemm_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
    cudaFuncSetAttribute(gemm_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
    cudaFuncSetAttribute(gemm_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
}

bool gemm_tc_applicable(const GemvArgs& a) {
    return g_sms_tc > 0 && !a.route && a.W.fmt == FMT_Q8_0 && a.W.K % KCH == 0 && a.B >= TC_MIN_BATCH &&
           a.B <= 32 && !a.xn_out && a.W.tm && a.W.tm->tc_ok &&
           (size_t)4 * ((a.W.N + TM - 1) / TM) <= (size_t)TC_TICKETS &&
           (long long)((a.W.N + TM - 1) / TM) * (a.W.K / KCH) * (g_sms_tc + 1) < (1ll << 31);
}

size_t gemm_tc_xh_elems(int K) { return (size_t)64 * K; }

void launch_gemm_tc(const GemvArgs& a, void* xh_v, float* part, size_t part_cap, uint32_t* tickets, cudaStream_t s,
                    bool pdl_prep, bool pdl) {
    __half* xh = static_cast<__half*>(xh_v);
    const int BP = a.B <= 8 ? 8 : a.B <= 16 ? 16 : 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(BP, (a.W.K + XK - 1) / XK);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_prep ? 1 : 0;
    cudaLaunchKernelEx(&cfg, prep_xh_kernel, a.x, a.x_stride, a.B, BP, a.W.K, a.norm_g, a.eps, xh);
    TcArgs t;
    std::copy(a.W.tm->tcq, a.W.tm->tcq + 16, t.mapq);
    if (!encode_f16_rows_sw128(t.mapx, xh, (uint64_t)a.W.K, (uint64_t)(2 * BP), (uint32_t)(2 * BP))) {
        if (a.err) cudaMemsetAsync(a.err, 0xFF, sizeof(uint32_t), s);   // reported by fq_check_device
        return;
    }
    t.W = a.W;
    t.B = a.B;
    t.y = a.y;
    t.y_stride = a.y_stride;
    t.epi = a.epi;
    t.st = a.st;
    t.err = a.err;
    t.part = part;
    t.tickets = tickets;
    if ((size_t)g_sms_tc * 2 * TM * BP > part_cap) {
        if (a.err) cudaMemsetAsync(a.err, 0xFF, sizeof(uint32_t), s);
        return;
    }
    if (BP == 8) launch_bp<8>(t, s, pdl);
    else if (BP == 16) launch_bp<16>(t, s, pdl);
    else launch_bp<32>(t, s, pdl);
}

}  // namespace fq
