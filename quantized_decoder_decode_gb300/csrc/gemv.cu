// Dequantise-in-register GEMV for the decode step (CUDA cores, sm_103a).
//
// y[b][r] = sum_k W[r][k] * xin[b][k] for a handful of activation rows b, where W is a
// ggml Q8_0 or Q4_K matrix (fucina "14. Model families" 14.1: quantised weights stay
// resident in their GGUF dtype and run their own packed kernels).  Each weight byte is
// read once per step with 128-bit streaming loads; codes become exact floats in registers
// (byte-permute into the mantissa of 2^23) and meet the activations, which sit in shared
// memory, in f32 fused multiply-adds.  Warps reduce with shuffles.
//
// Fused around the contraction:
//   prologue  RMSNorm of the input rows (the runner page's "fused norm+QKV projection",
//             also used before gate_up and the LM head);
//   epilogues plain store (QKV), residual add (O and down projections), SwiGLU over
//             interleaved gate/up rows, and logits + argmax keys for greedy decoding.
//
// Q8_0 block sums use the factorisation sum_i (d q_i) x_i = d * sum_i q_i x_i.  Q4_K uses
// (d sc) q - dmin mn per 32-element sub-block, i.e. d sc * sum q x - dmin mn * sum x, with
// the activation sums per 16 elements computed once per CTA.

#include "common.cuh"
#include "kernels.h"
#include "quant.cuh"

#include <algorithm>
#include <cstdlib>

namespace fq {

namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;

// One CTA owns a tile of rows_per_cta = (8 / ksplit) * R rows at a time and walks the tiles
// with a CTA stride, so the input rows are staged (and their RMS computed) once per CTA.
// Warp w serves row group w / ksplit over K part w % ksplit; lanes stride over the units of
// that part, two units per iteration so that 2R independent 16-byte loads are in flight.
// An RMSNorm prologue stages x * g and applies 1/rms to the finished dot products
// (W (x/rms * g) = (W (x * g)) / rms), so no block reduction sits before the first load.
template <int FMT, int R, int NBG>
__global__ void __launch_bounds__(THREADS) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) float smem[];
    QMat W = a.W;
    const int K = W.K;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ksplit = a.ksplit;
    const int rows_per_cta = (WARPS / ksplit) * R;
    int B = a.B;
    const int32_t* ptok = nullptr;
    const int32_t* pslot = nullptr;

    if (a.route == nullptr) {
        // weights do not depend on earlier kernels: start streaming this CTA's first tile
        const int r0 = blockIdx.x * rows_per_cta;
        int nrows = min(rows_per_cta, W.N - r0);
        if (nrows > 0) {
            size_t rb = W.row_bytes();
            prefetch_l2_range(W.q + (size_t)r0 * rb, (size_t)nrows * rb, tid, THREADS);
            if (FMT == FMT_Q8_0 && ((size_t)r0 * (K / 32) * 2) % 16 == 0)
                prefetch_l2_range(W.s + (size_t)r0 * (K / 32), ((size_t)nrows * (K / 32) * 2) & ~(size_t)15, tid,
                                  THREADS);
        }
        pdl_trigger();
        pdl_wait();
    } else {
        // the expert and its tokens come from the route the previous kernel wrote
        pdl_trigger();
        pdl_wait();
        const MoeRoute* rt = a.route;
        const int ae = blockIdx.y;
        if (ae >= rt->n_active) return;
        const int e = rt->expert[ae], p0 = rt->start[ae];
        B = rt->start[ae + 1] - p0;
        ptok = rt->pair_token + p0;
        pslot = rt->pair_slot + p0;
        W.N = a.rows_per_expert;
        W.q += (size_t)e * a.rows_per_expert * W.row_bytes();
        if (W.s) W.s += (size_t)e * a.rows_per_expert * (K / 32);
    }
    auto in_row = [&](int b) -> const float* {
        size_t r = ptok ? (a.x_by_pair ? (size_t)ptok[b] * a.moe_k + pslot[b] : (size_t)ptok[b]) : (size_t)b;
        return a.x + r * a.x_stride;
    };
    auto out_row = [&](int b) -> float* {
        size_t r = ptok ? (size_t)ptok[b] * a.moe_k + pslot[b] : (size_t)b;
        return a.y + r * a.y_stride;
    };

    const int KP = xpad_len<FMT>(K);                                  // padded row length
    float* xs = smem;                                                 // [NBG][KP]
    float* xsum16 = smem + NBG * KP;                                  // [NBG][K/16] (Q4_K)
    float* red = xsum16 + (FMT == FMT_Q4_K ? NBG * (K / 16) : 0);     // [WARPS][R][NBG]
    float* ssw = red + WARPS * R * NBG;                               // [WARPS][NBG]
    __shared__ unsigned long long best[NBG];

    const int n_units = K / Unit<FMT>::ELEMS;
    const int rg = warp / ksplit, kp = warp % ksplit;
    const int upp = (n_units + ksplit - 1) / ksplit;
    const int u_begin = kp * upp, u_end = min(n_units, u_begin + upp);
    const int n_tiles = (W.N + rows_per_cta - 1) / rows_per_cta;

    // activation rows in groups of NBG: outside expert mode grid.y splits the groups
    const int g0 = a.route ? 0 : (int)blockIdx.y, gstep = a.route ? 1 : (int)gridDim.y;
    for (int b0 = g0 * NBG; b0 < B; b0 += NBG * gstep) {
        const int nb = min(NBG, B - b0);
        // ---- prologue: x (times the norm gain) into shared memory, partial sums of x^2
        for (int b = 0; b < nb; ++b) {
            const float* xin = in_row(b0 + b);
            float ss = 0.f;
            for (int k = tid * 4; k < K; k += THREADS * 4) {
                float4 v = *reinterpret_cast<const float4*>(xin + k);
                ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
                if (a.norm_g) {
                    float4 g = *reinterpret_cast<const float4*>(a.norm_g + k);
                    v.x *= g.x; v.y *= g.y; v.z *= g.z; v.w *= g.w;
                }
                *reinterpret_cast<float4*>(xs + b * KP + xpad<FMT>(k)) = v;
            }
            ss = warp_sum(ss);
            if (lane == 0) ssw[warp * NBG + b] = ss;
        }
        if (tid < NBG) best[tid] = 0ull;
        __syncthreads();
        float inv[NBG];
#pragma unroll
        for (int b = 0; b < NBG; ++b) {
            float t = 0.f;
            if (b < nb)
                for (int w = 0; w < WARPS; ++w) t += ssw[w * NBG + b];
            inv[b] = a.norm_g ? rsqrtf(t / (float)K + a.eps) : 1.f;
        }
        if (a.xn_out && blockIdx.x == 0) {
            for (int i = tid * 4; i < nb * K; i += THREADS * 4) {
                int b = i / K, k = i % K;
                float4 v = *reinterpret_cast<const float4*>(xs + b * KP + xpad<FMT>(k));
                float s = inv[0];
#pragma unroll
                for (int bb = 1; bb < NBG; ++bb)
                    if (bb == b) s = inv[bb];
                v.x *= s; v.y *= s; v.z *= s; v.w *= s;
                *reinterpret_cast<float4*>(a.xn_out + (size_t)(b0 + b) * a.xn_stride + k) = v;
            }
        }
        if (FMT == FMT_Q4_K) {
            for (int i = tid; i < nb * (K / 16); i += THREADS) {
                int b = i / (K / 16), j = i % (K / 16);
                const float4* p = reinterpret_cast<const float4*>(xs + b * KP + xpad<FMT>(16 * j));
                float s = 0.f;
#pragma unroll
                for (int t = 0; t < 4; ++t) { float4 v = p[t]; s += v.x + v.y + v.z + v.w; }
                xsum16[b * (K / 16) + j] = s;
            }
            __syncthreads();
        }

        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
            const int row_base = tile * rows_per_cta + rg * R;
            float acc[R][NBG];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int b = 0; b < NBG; ++b) acc[r][b] = 0.f;
            bool row_ok[R];
#pragma unroll
            for (int r = 0; r < R; ++r) row_ok[r] = row_base + r < W.N;

            int u = u_begin + lane;
            if constexpr (FMT == FMT_Q4_K && NBG > 1) {
                // several activation rows: each code is turned into a float once per weight row
                for (; u < u_end; u += 32) {
                    Raw rq[R];
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        if (row_ok[r]) rq[r] = load_unit<FMT>(W, row_base + r, u);
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        if (row_ok[r]) dot_q4k_rows<NBG>(rq[r], u, xs, KP, xsum16, K / 16, nb, acc[r]);
                }
            } else if constexpr (FMT == FMT_Q8_0 && NBG > 1) {
                // several activation rows: each unit's codes become floats once per weight row,
                // then meet every activation row (read from shared memory as they are used)
                for (; u < u_end; u += 32) {
                    Raw rq[R];
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        if (row_ok[r]) rq[r] = load_unit<FMT>(W, row_base + r, u);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (!row_ok[r]) continue;
                        float f[16];
                        s8x4_to_f32(rq[r].q.x, f);
                        s8x4_to_f32(rq[r].q.y, f + 4);
                        s8x4_to_f32(rq[r].q.z, f + 8);
                        s8x4_to_f32(rq[r].q.w, f + 12);
                        const float d = h2f(rq[r].sc);
#pragma unroll
                        for (int b = 0; b < NBG; ++b) {
                            if (b >= nb) break;
                            const float4* xp = reinterpret_cast<const float4*>(xs + b * KP + xpad<FMT>(u * 16));
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
                            acc[r][b] = fmaf(d, s0 + s1, acc[r][b]);
                        }
                    }
                }
            } else {
            for (; u + 32 < u_end; u += 64) {
                Raw r0[R], r1[R];
#pragma unroll
                for (int r = 0; r < R; ++r)
                    if (row_ok[r]) {
                        r0[r] = load_unit<FMT>(W, row_base + r, u);
                        r1[r] = load_unit<FMT>(W, row_base + r, u + 32);
                    }
#pragma unroll
                for (int b = 0; b < NBG; ++b) {
                    if (b < nb) {
                        XFrag<FMT> x0, x1;
                        load_x<FMT>(xs + b * KP, u, x0);
                        load_x<FMT>(xs + b * KP, u + 32, x1);
#pragma unroll
                        for (int r = 0; r < R; ++r)
                            if (row_ok[r])
                                acc[r][b] += dot_frag<FMT>(r0[r], u, x0, xsum16 + b * (K / 16)) +
                                             dot_frag<FMT>(r1[r], u + 32, x1, xsum16 + b * (K / 16));
                    }
                }
            }
            if (u < u_end) {
                Raw r0[R];
#pragma unroll
                for (int r = 0; r < R; ++r)
                    if (row_ok[r]) r0[r] = load_unit<FMT>(W, row_base + r, u);
#pragma unroll
                for (int b = 0; b < NBG; ++b) {
                    if (b < nb) {
                        XFrag<FMT> x0;
                        load_x<FMT>(xs + b * KP, u, x0);
#pragma unroll
                        for (int r = 0; r < R; ++r)
                            if (row_ok[r]) acc[r][b] += dot_frag<FMT>(r0[r], u, x0, xsum16 + b * (K / 16));
                    }
                }
            }
            }

            // ---- reduce: lanes, then the K parts of a row group
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int b = 0; b < NBG; ++b) acc[r][b] = warp_sum(acc[r][b]);
            if (ksplit > 1) {
                if (lane == 0)
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int b = 0; b < NBG; ++b) red[(warp * R + r) * NBG + b] = acc[r][b];
                __syncthreads();
                if (kp == 0 && lane == 0) {
                    for (int w = 1; w < ksplit; ++w)
#pragma unroll
                        for (int r = 0; r < R; ++r)
#pragma unroll
                            for (int b = 0; b < NBG; ++b) acc[r][b] += red[((warp + w) * R + r) * NBG + b];
                }
            }

            // ---- epilogue (one lane per row group)
            if (kp == 0 && lane == 0) {
#pragma unroll
                for (int b = 0; b < NBG; ++b) {
                    if (b >= nb) continue;
                    float* yrow = out_row(b0 + b);
#pragma unroll
                    for (int r = 0; r < R; ++r) acc[r][b] *= inv[b];
                    if (a.epi == EPI_SWIGLU) {
#pragma unroll
                        for (int r = 0; r + 1 < R; r += 2)
                            if (row_ok[r + 1]) yrow[(row_base + r) >> 1] = silu(acc[r][b]) * acc[r + 1][b];
                    } else {
                        unsigned long long kbest = 0ull;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            if (!row_ok[r]) continue;
                            int row = row_base + r;
                            if (a.epi == EPI_ADD) yrow[row] += acc[r][b];
                            else yrow[row] = acc[r][b];
                            if (a.epi == EPI_LOGITS) {
                                unsigned long long kk = argmax_key(acc[r][b], (uint32_t)row);
                                kbest = kk > kbest ? kk : kbest;
                            }
                        }
                        if (a.epi == EPI_LOGITS) atomicMax(&best[b], kbest);
                    }
                }
            }
            if (ksplit > 1) __syncthreads();   // red is reused by the next tile
        }
        __syncthreads();
        if (a.epi == EPI_LOGITS && tid < nb) atomicMax(&a.st->keys[b0 + tid], best[tid]);
        __syncthreads();
    }
}

int g_sms = 152;   // set by gemv_prepare

template <int FMT, int R, int NBG>
struct Occ {
    static int ctas_per_sm;   // resident CTAs per SM at the kernel's register / smem use
};
template <int FMT, int R, int NBG>
int Occ<FMT, R, NBG>::ctas_per_sm = 2;

template <int FMT, int R, int NBG>
void launch_t(const GemvArgs& a, cudaStream_t s, bool pdl) {
    const int rows_per_cta = (WARPS / a.ksplit) * R;
    const int rows = a.route ? a.rows_per_expert : a.W.N;
    const int tiles = (rows + rows_per_cta - 1) / rows_per_cta;
    // one wave of resident CTAs; larger matrices loop over tiles inside each CTA
    // one wave of resident CTAs over (row tiles, activation-row groups)
    const int groups = a.route ? a.max_experts : (a.B + NBG - 1) / NBG;
    const int per_group = std::max(1, Occ<FMT, R, NBG>::ctas_per_sm * g_sms / groups);
    // expert mode: up to eight waves of CTAs over the possible experts (measured best of 2, 4,
    // 8, 16 and one CTA per tile), each looping over row tiles of its expert, so that an
    // expert's token inputs are staged once per CTA rather than once per tile
    const int per_expert = std::max(1, 8 * Occ<FMT, R, NBG>::ctas_per_sm * g_sms / std::max(1, groups));
    dim3 grid(std::min(tiles, a.route ? per_expert : per_group), groups);
    size_t smem = (size_t)NBG * xpad_len<FMT>(a.W.K) * 4 + (FMT == FMT_Q4_K ? (size_t)NBG * (a.W.K / 16) * 4 : 0) +
                  (size_t)(WARPS * R * NBG + WARPS * NBG) * 4;
    auto kern = gemv_kernel<FMT, R, NBG>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaLaunchKernelEx(&cfg, kern, a);
}

template <int FMT, int R, int NBG>
void prepare_t(int optin) {
    cudaFuncAttributes fa;
    cudaFuncGetAttributes(&fa, gemv_kernel<FMT, R, NBG>);
    cudaFuncSetAttribute(gemv_kernel<FMT, R, NBG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         optin - (int)fa.sharedSizeBytes);
    int occ = 0;
    // typical stage: hidden 4096 in shared memory for each of NBG rows
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_kernel<FMT, R, NBG>, THREADS,
                                                  (size_t)NBG * 4096 * 4 + 2048);
    Occ<FMT, R, NBG>::ctas_per_sm = occ > 0 ? occ : 1;
}

}  // namespace

void gemv_prepare() {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    prepare_t<FMT_Q8_0, 4, 1>(optin);
    prepare_t<FMT_Q8_0, 4, 4>(optin);
    prepare_t<FMT_Q4_K, 2, 1>(optin);
    prepare_t<FMT_Q4_K, 2, 4>(optin);
    prepare_t<FMT_F32, 4, 1>(optin);
    prepare_t<FMT_F32, 4, 4>(optin);
    gemv_tma_prepare();
}

void launch_gemv(const GemvArgs& a, cudaStream_t s, bool pdl) {
    if (launch_gemv_tma(a, s, pdl)) return;
    // expert mode: an expert's tokens are only known on the device; the four-row variant reads
    // and converts each weight once for up to four of them
    const bool one = a.B == 1 && !(a.route && a.W.fmt == FMT_Q8_0);
    switch (a.W.fmt) {
        case FMT_Q8_0:
            if (one) launch_t<FMT_Q8_0, 4, 1>(a, s, pdl);
            else launch_t<FMT_Q8_0, 4, 4>(a, s, pdl);
            break;
        case FMT_Q4_K:
            if (one) launch_t<FMT_Q4_K, 2, 1>(a, s, pdl);
            else launch_t<FMT_Q4_K, 2, 4>(a, s, pdl);
            break;
        default:
            if (one) launch_t<FMT_F32, 4, 1>(a, s, pdl);
            else launch_t<FMT_F32, 4, 4>(a, s, pdl);
            break;
    }
}

}  // namespace fq
