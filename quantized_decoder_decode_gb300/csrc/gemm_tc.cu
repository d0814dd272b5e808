// Lockstep batch decode GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Section 14.2 of the fucina pages: forwardStepBatch runs the dense trunk as one m = n pass
// so that every weight is read once for all streams.  With n = 8..32 rows the contraction
// y[b][r] = sum_k W[r][k] x[b][k] is dense enough for tensor cores, so it runs "swap-AB":
//   D[r, c] = sum_k A[r, k] B[c, k],  A = dequantised weight tile (M = 128 rows, f16),
//                                     B = activations, N = 2 * BP columns (f16),
// where activation row b is split into a high part hi = f16(x) (column b) and a low part
// lo = f16(x - hi) (column BP + b): hi + lo carries ~22 bits, so only the weights are
// rounded to f16 (relative 2^-12), and y = D[:, b] + D[:, BP + b] with f32 accumulation in
// tensor memory.
//
// Roles in a CTA (288 threads):
//   warps 0-3  converters: per stage of 64 K-elements, each thread streams one weight row's
//              64 Q8_0 codes + 2 scales from global memory, dequantises to exact products
//              d*q and rounds them once to f16 into the 128-byte-swizzled K-major layout,
//              and copies the stage's activation slice (prepared f16 hi/lo rows);
//   warp 8     one thread issues 4 tcgen05.mma (K = 16 each) per stage and commits the
//              stage back to the converters; after the tile's last stage it commits the
//              accumulator to the epilogue;
//   warps 4-7  epilogue: tcgen05.ld of the 128 x N accumulator (one row per thread), hi+lo,
//              then store / residual add / SwiGLU (gate, up rows adjacent) / logits+argmax.
// Work is split into (row tile, K slice) units so that narrow matrices still cover every
// SM: with several K slices each unit writes its partial sums to scratch and the last unit
// of a tile to finish (atomic ticket, no waiting) adds them up and applies the epilogue.
// Converter threads keep two chunks of codes in flight ahead of the one they decode.
// Every mbarrier wait is bounded; a stuck pipeline sets the error word and unwinds.

#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace fq {

namespace {

constexpr int TM = 128;                  // MMA M: weight rows per tile
constexpr int KCH = 64;                  // K elements per stage: one 128-byte f16 swizzle atom
constexpr int TSTAGES = 4;
constexpr int A_STAGE = TM * KCH * 2;    // 16 KB
constexpr int B_STAGE = 64 * KCH * 2;    // 8 KB (N <= 64)
constexpr int TC_THREADS = 9 * 32;
constexpr int CONV_WARPS = 4, EPI_WARP0 = 4, MMA_WARP = 8;
constexpr size_t TC_SMEM = (size_t)TSTAGES * (A_STAGE + B_STAGE) + 256;

struct TcArgs {
    QMat W;              // Q8_0 [N][K], K % 64 == 0
    const __half* xh;    // [2 * BP][K] f16: rows 0..BP-1 high parts, BP..2BP-1 low parts
    int B;               // activation rows (<= BP)
    float* y;
    int y_stride;
    int epi;
    StepState* st;
    uint32_t* err;
    int ks;              // K slices per tile (divides K / 64)
    float* part;         // [ks][B][N] partial sums (ks > 1)
    uint32_t* tickets;   // [4 * tiles] arrival counters per (tile, epilogue warp), zero between uses
};

template <int BP>
__global__ void __launch_bounds__(TC_THREADS, 2) gemm_tc_kernel(const TcArgs a) {
    constexpr int NCOL = 2 * BP;         // MMA N
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* As = smem;
    uint8_t* Bs = As + (size_t)TSTAGES * A_STAGE;
    uint64_t* full = reinterpret_cast<uint64_t*>(Bs + (size_t)TSTAGES * B_STAGE);
    uint64_t* freeb = full + TSTAGES;
    uint64_t* acc_full = freeb + TSTAGES;
    uint64_t* acc_free = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_free + 1);
    __shared__ unsigned long long best[32];

    const QMat& W = a.W;
    const int N = W.N, K = W.K;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_tiles = (N + TM - 1) / TM, n_chunks = K / KCH;
    const int KS = a.ks, cpk = n_chunks / KS;            // K slices per tile, chunks per slice
    const int n_units = n_tiles * KS;
    const int my_units = (int)blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (tid == 0) {
        for (int s = 0; s < TSTAGES; ++s) {
            mbar_init(&full[s], CONV_WARPS);
            mbar_init(&freeb[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_free, 4);
        mbar_fence_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(tmem_slot, 64);
        tmem_relinquish();
    }
    if (tid < 32) best[tid] = 0ull;
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    pdl_trigger();
    pdl_wait();

    if (warp < CONV_WARPS) {
        // ---------------- converters: one weight row per thread, two chunks of codes in flight
        const int r = tid;
        const int n_iters = my_units * cpk;
        struct Codes {
            uint4 c[4];
            uint32_t sc2;
        };
        auto fetch = [&](int it, Codes& cd) {
            const int unit = blockIdx.x + (it / cpk) * gridDim.x;
            const int tile = unit / KS, chunk = (unit % KS) * cpk + it % cpk;
            const int row = tile * TM + r;
            if (it < n_iters && row < N) {
                const uint8_t* src = W.q + (size_t)row * K + (size_t)chunk * KCH;
#pragma unroll
                for (int i = 0; i < 4; ++i) cd.c[i] = ld_stream16(src + 16 * i);
                cd.sc2 = ld_stream4(W.s + (size_t)row * (K / 32) + (size_t)chunk * 2);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) cd.c[i] = make_uint4(0u, 0u, 0u, 0u);
                cd.sc2 = 0u;
            }
        };
        Codes c0, c1, c2;
        fetch(0, c0);
        fetch(1, c1);
        for (int it = 0; it < n_iters; ++it) {
            fetch(it + 2, c2);
            const int unit = blockIdx.x + (it / cpk) * gridDim.x;
            const int chunk = (unit % KS) * cpk + it % cpk;
            const int stage = it % TSTAGES;
            const uint32_t ph = (uint32_t)(it / TSTAGES) & 1u;
            if (!mbar_wait(&freeb[stage], ph ^ 1u)) {
                if (a.err && lane == 0) atomicOr(a.err, 4u);
                break;
            }
            uint8_t* Ast = As + (size_t)stage * A_STAGE;
            const float d0 = h2f((unsigned short)(c0.sc2 & 0xFFFFu)), d1 = h2f((unsigned short)(c0.sc2 >> 16));
#pragma unroll
            for (int j = 0; j < 8; ++j) {          // 16-byte chunk j = K elements 8j..8j+7
                const uint4 w4 = c0.c[j >> 1];
                const uint32_t w0 = (j & 1) ? w4.z : w4.x, w1 = (j & 1) ? w4.w : w4.y;
                float f[8];
                s8x4_to_f32(w0, f);
                s8x4_to_f32(w1, f + 4);
                const float d = j < 4 ? d0 : d1;
                __half2 h[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(f[2 * e] * d, f[2 * e + 1] * d);
                *reinterpret_cast<uint4*>(Ast + sw128_offset(r, j)) = *reinterpret_cast<uint4*>(h);
            }
            uint8_t* Bst = Bs + (size_t)stage * B_STAGE;
            for (int q = r; q < NCOL * 8; q += CONV_WARPS * 32) {
                const int nrow = q >> 3, j = q & 7;
                const uint4 v = *reinterpret_cast<const uint4*>(a.xh + (size_t)nrow * K + (size_t)chunk * KCH + 8 * j);
                *reinterpret_cast<uint4*>(Bst + sw128_offset(nrow, j)) = v;
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[stage]);
            c0 = c1;
            c1 = c2;
        }
    } else if (warp == MMA_WARP) {
        // ---------------- MMA issue: one thread
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(TM, NCOL);
            int it = 0;
            bool ok = true;
            for (int t = 0; t < my_units && ok; ++t) {
                if (t > 0) {
                    if (!mbar_wait(acc_free, (uint32_t)(t - 1) & 1u)) {
                        if (a.err) atomicOr(a.err, 8u);
                        break;
                    }
                    tc_fence_after();
                }
                for (int chunk = 0; chunk < cpk; ++chunk, ++it) {
                    const int stage = it % TSTAGES;
                    const uint32_t ph = (uint32_t)(it / TSTAGES) & 1u;
                    if (!mbar_wait(&full[stage], ph)) {
                        if (a.err) atomicOr(a.err, 16u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_sw128(smem_u32(As + (size_t)stage * A_STAGE));
                    const uint64_t bd = sdesc_sw128(smem_u32(Bs + (size_t)stage * B_STAGE));
#pragma unroll
                    for (int k = 0; k < KCH / 16; ++k)   // 32 bytes of K per MMA: start address + 2 (x16 B)
                        mma_f16(tbase, ad + 2 * k, bd + 2 * k, idesc, (chunk > 0 || k > 0) ? 1u : 0u);
                    mma_commit(&freeb[stage]);
                }
                if (ok) mma_commit(acc_full);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: TMEM lanes 32q..32q+31 <-> tile rows
        const int q = warp - EPI_WARP0;
        const int rin = 32 * q + lane;
        for (int t = 0; t < my_units; ++t) {
            if (!mbar_wait(acc_full, (uint32_t)t & 1u)) {
                if (a.err && lane == 0) atomicOr(a.err, 32u);
                break;
            }
            tc_fence_after();
            uint32_t v[NCOL];
#pragma unroll
            for (int c4 = 0; c4 < NCOL / 16; ++c4) tmem_ld16(tbase + ((uint32_t)(32 * q) << 16) + 16 * c4, v + 16 * c4);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free);
            const int unit = blockIdx.x + t * gridDim.x;
            const int tile = unit / KS, ksl = unit % KS;
            const int row = tile * TM + rin;
            const bool ok_row = row < N;
            float val[BP];
#pragma unroll
            for (int b = 0; b < BP; ++b) val[b] = __uint_as_float(v[b]) + __uint_as_float(v[BP + b]);
            if (KS > 1) {
                // partial of this K slice -> scratch; the tile's last slice adds them up
                if (ok_row)
#pragma unroll
                    for (int b = 0; b < BP; ++b)
                        if (b < a.B) a.part[((size_t)ksl * a.B + b) * N + row] = val[b];
                // each epilogue warp owns 32 rows of the tile and its own ticket
                __threadfence();
                __syncwarp();
                uint32_t prev = 0u;
                if (lane == 0) {
                    prev = atomicAdd(&a.tickets[4 * tile + q], 1u);
                    if (prev == (uint32_t)(KS - 1)) a.tickets[4 * tile + q] = 0u;
                }
                prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
                if (prev != (uint32_t)(KS - 1)) continue;
                __threadfence();
#pragma unroll
                for (int b = 0; b < BP; ++b) {
                    float acc = 0.f;
                    if (b < a.B && ok_row)
                        for (int k2 = 0; k2 < KS; ++k2) acc += __ldcg(&a.part[((size_t)k2 * a.B + b) * N + row]);
                    val[b] = acc;
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
        tmem_dealloc(tbase, 64);
    }
}

// x (optionally RMSNorm-ed with gain g) -> f16 high / low rows for the MMA B operand;
// rows B..BP-1 are zero.  One CTA per padded row.
__global__ void __launch_bounds__(256) prep_xh_kernel(const float* x, int x_stride, int B, int BP, int K,
                                                      const float* g, float eps, __half* xh) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[32];
    const int b = blockIdx.x;
    __half* hi = xh + (size_t)b * K;
    __half* lo = xh + (size_t)(BP + b) * K;
    if (b >= B) {
        for (int k = threadIdx.x; k < K; k += blockDim.x) {
            hi[k] = __float2half_rn(0.f);
            lo[k] = __float2half_rn(0.f);
        }
        return;
    }
    const float* xr = x + (size_t)b * x_stride;
    float inv = 1.f;
    if (g) {
        float ss = 0.f;
        for (int k = threadIdx.x; k < K; k += blockDim.x) ss += xr[k] * xr[k];
        ss = block_sum(ss, red);
        inv = rsqrtf(ss / (float)K + eps);
    }
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const float v = g ? xr[k] * inv * g[k] : xr[k];
        const __half h = __float2half_rn(v);
        hi[k] = h;
        lo[k] = __float2half_rn(v - __half2float(h));
    }
}

int g_sms_tc = 0;

template <int BP>
void launch_bp(const TcArgs& t, cudaStream_t s, bool pdl) {
    const int tiles = (t.W.N + TM - 1) / TM;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(tiles * t.ks, 2 * g_sms_tc));
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
           a.B <= 32 && !a.xn_out;
}

size_t gemm_tc_xh_elems(int K) { return (size_t)64 * K; }

void launch_gemm_tc(const GemvArgs& a, void* xh_v, float* part, size_t part_cap, uint32_t* tickets, cudaStream_t s,
                    bool pdl_prep, bool pdl) {
    __half* xh = static_cast<__half*>(xh_v);
    const int BP = a.B <= 8 ? 8 : a.B <= 16 ? 16 : 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(BP);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_prep ? 1 : 0;
    cudaLaunchKernelEx(&cfg, prep_xh_kernel, a.x, a.x_stride, a.B, BP, a.W.K, a.norm_g, a.eps, xh);
    TcArgs t;
    t.W = a.W;
    t.xh = xh;
    t.B = a.B;
    t.y = a.y;
    t.y_stride = a.y_stride;
    t.epi = a.epi;
    t.st = a.st;
    t.err = a.err;
    // K slices: enough (row tile, K slice) units for two CTAs per SM, at least 4 chunks each
    const int tiles = (a.W.N + TM - 1) / TM, n_chunks = a.W.K / KCH;
    int ks = 1;
    while (tiles * ks < 2 * g_sms_tc && n_chunks % (2 * ks) == 0 && n_chunks / (2 * ks) >= 4 &&
           (size_t)(2 * ks) * a.B * a.W.N <= part_cap && 4 * tiles <= TC_TICKETS)
        ks *= 2;
    t.ks = ks;
    t.part = part;
    t.tickets = tickets;
    if (BP == 8) launch_bp<8>(t, s, pdl);
    else if (BP == 16) launch_bp<16>(t, s, pdl);
    else launch_bp<32>(t, s, pdl);
}

}  // namespace fq
