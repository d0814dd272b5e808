// Weight-streaming GEMV fed by bulk asynchronous copies (TMA, sm_103a).
//
// Same contraction and fused prologue/epilogues as the register-fed GEMV (RMSNorm of the
// input rows; store, residual add, SwiGLU over interleaved gate/up rows, logits + argmax
// keys), but the weight bytes travel global -> shared memory through cp.async.bulk into a
// ring of STAGES buffers guarded by mbarriers:
//   * one producer warp walks this CTA's (row tile, K chunk) pairs and issues the copies of
//     the next free stage;
//   * eight consumer warps wait for a stage, decode codes to exact floats in registers,
//     multiply-accumulate against the activations staged in shared memory, release the
//     stage, and reduce + apply the epilogue at the end of each row tile.
// Each stage is one 2-D tensor-map copy of the codes (a box of rows x K-chunk) plus, for
// Q8_0, one of the scales; boxes that run past the last row or column are zero-filled.
// The producer starts before griddepcontrol.wait (weights never depend on an earlier
// kernel), so the first STAGES chunks are already landing while the previous kernel of
// the step finishes; only the consumers wait for the activations.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "quant.cuh"
#include "tma.cuh"

namespace fq {

namespace {

constexpr int CONSUMER_WARPS = 8;
constexpr int CONSUMERS = CONSUMER_WARPS * 32;
constexpr int THREADS_T = CONSUMERS + 32;   // + one producer warp
constexpr int STAGES = 4;

template <int FMT> struct TCfg;
// rows per warp R, rows per tile RT, K elements per chunk KC, unit passes per lane
template <> struct TCfg<FMT_Q8_0> { static constexpr int R = 4, RT = 32, KC = 512, UPL = 1; };
template <> struct TCfg<FMT_Q4_K> { static constexpr int R = 2, RT = 16, KC = 2048, UPL = 1; };
template <> struct TCfg<FMT_F32> { static constexpr int R = 4, RT = 32, KC = 128, UPL = 1; };

// elements per K chunk in the tensor maps' view of the planes
template <int FMT> struct TView;
template <> struct TView<FMT_Q8_0> { static constexpr int X = 128; };   // codes as u32
template <> struct TView<FMT_Q4_K> { static constexpr int X = 144; };   // blocks as u64
template <> struct TView<FMT_F32> { static constexpr int X = 128; };

template <int FMT>
FQ_HD constexpr int chunk_bytes(int kc) {   // bytes of kc elements of one row
    return FMT == FMT_Q8_0 ? kc : FMT == FMT_Q4_K ? kc / 256 * 144 : kc * 4;
}

template <int FMT, int NBG>
struct TLayout {
    static constexpr int QSTAGE = TCfg<FMT>::RT * chunk_bytes<FMT>(TCfg<FMT>::KC);
    static constexpr int SSTAGE = FMT == FMT_Q8_0 ? TCfg<FMT>::RT * (TCfg<FMT>::KC / 16) : 0;
    static size_t bytes(int K) {
        return (size_t)STAGES * (QSTAGE + SSTAGE) + (size_t)NBG * xpad_len<FMT>(K) * 4 +
               (FMT == FMT_Q4_K ? (size_t)NBG * (K / 16) * 4 : 0) + (size_t)CONSUMER_WARPS * NBG * 4 +
               2 * STAGES * 8 + 64;
    }
};

struct TmaParams {
    TmaMaps maps;
    GemvArgs a;
};

template <int FMT, int NBG>
__global__ void __launch_bounds__(THREADS_T, 2) gemv_tma_kernel(const __grid_constant__ TmaParams prm) {
    using C = TCfg<FMT>;
    using Lay = TLayout<FMT, NBG>;
    const GemvArgs& a = prm.a;
    extern __shared__ __align__(1024) uint8_t smem[];
    const QMat W = a.W;
    const int K = W.K, N = W.N;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    uint8_t* qbuf = smem;                                                    // [STAGES][RT][chunk bytes]
    uint8_t* sbuf = qbuf + (size_t)STAGES * Lay::QSTAGE;                     // [STAGES][RT][KC/16] (Q8_0)
    const int KP = xpad_len<FMT>(K);                                         // padded row length
    float* xs = reinterpret_cast<float*>(sbuf + (size_t)STAGES * Lay::SSTAGE);   // [NBG][KP]
    float* xsum16 = xs + (size_t)NBG * KP;                                   // [NBG][K/16] (Q4_K)
    float* ssw = xsum16 + (FMT == FMT_Q4_K ? (size_t)NBG * (K / 16) : 0);    // [CONSUMER_WARPS][NBG]
    uint64_t* full = reinterpret_cast<uint64_t*>(
        (reinterpret_cast<uintptr_t>(ssw + CONSUMER_WARPS * NBG) + 15) & ~(uintptr_t)15);
    uint64_t* empty = full + STAGES;
    __shared__ unsigned long long best[NBG];

    const int n_tiles = (N + C::RT - 1) / C::RT;
    const int n_chunks = (K + C::KC - 1) / C::KC;
    const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int n_iters = my_tiles * n_chunks;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CONSUMER_WARPS);
        }
        mbar_fence_init();
    }
    if (tid < NBG) best[tid] = 0ull;
    __syncthreads();
    pdl_trigger();

    if (warp == CONSUMER_WARPS) {
        // ---------------- producer: weights only, so no wait for the previous kernel
        constexpr uint32_t STAGE_BYTES = (uint32_t)(Lay::QSTAGE + Lay::SSTAGE);
        for (int it = 0; it < (a.starve ? 0 : n_iters); ++it) {
            const int stage = it % STAGES;
            const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
            if (!mbar_wait(&empty[stage], ph ^ 1u)) {
                if (a.err && lane == 0) atomicOr(a.err, 1u);
                break;
            }
            if (lane == 0) {
                const int tile = blockIdx.x + (it / n_chunks) * gridDim.x, chunk = it % n_chunks;
                mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                tma_load_2d(qbuf + (size_t)stage * Lay::QSTAGE, prm.maps.q, chunk * TView<FMT>::X, tile * C::RT,
                            &full[stage]);
                if (FMT == FMT_Q8_0)
                    tma_load_2d(sbuf + (size_t)stage * Lay::SSTAGE, prm.maps.s, chunk * (C::KC / 32), tile * C::RT,
                                &full[stage]);
            }
            __syncwarp();
        }
        pdl_wait();   // every thread of the grid waits before the grid may complete
        return;
    }

    // ---------------- consumers
    pdl_wait();
    for (int b = 0; b < a.B; ++b) {
        const float* xin = a.x + (size_t)b * a.x_stride;
        float ss = 0.f;
        for (int k = tid * 4; k < K; k += CONSUMERS * 4) {
            float4 v = *reinterpret_cast<const float4*>(xin + k);
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            if (a.norm_g) {
                float4 g = *reinterpret_cast<const float4*>(a.norm_g + k);
                v.x *= g.x; v.y *= g.y; v.z *= g.z; v.w *= g.w;
            }
            *reinterpret_cast<float4*>(xs + (size_t)b * KP + xpad<FMT>(k)) = v;
        }
        ss = warp_sum(ss);
        if (lane == 0) ssw[warp * NBG + b] = ss;
    }
    bar_sync_consumers(CONSUMERS);
    float inv[NBG];
#pragma unroll
    for (int b = 0; b < NBG; ++b) {
        float t = 0.f;
        if (b < a.B)
            for (int w = 0; w < CONSUMER_WARPS; ++w) t += ssw[w * NBG + b];
        inv[b] = a.norm_g ? rsqrtf(t / (float)K + a.eps) : 1.f;
    }
    if (a.xn_out && blockIdx.x == 0) {
        for (int i = tid * 4; i < a.B * K; i += CONSUMERS * 4) {
            const int b = i / K, k = i % K;
            float s = inv[0];
#pragma unroll
            for (int bb = 1; bb < NBG; ++bb)
                if (bb == b) s = inv[bb];
            float4 v = *reinterpret_cast<const float4*>(xs + (size_t)b * KP + xpad<FMT>(k));
            v.x *= s; v.y *= s; v.z *= s; v.w *= s;
            *reinterpret_cast<float4*>(a.xn_out + (size_t)b * a.xn_stride + k) = v;
        }
    }
    if (FMT == FMT_Q4_K) {
        for (int i = tid; i < a.B * (K / 16); i += CONSUMERS) {
            const int b = i / (K / 16), j = i % (K / 16);
            const float4* p = reinterpret_cast<const float4*>(xs + (size_t)b * KP + xpad<FMT>(16 * j));
            float s = 0.f;
#pragma unroll
            for (int t = 0; t < 4; ++t) { float4 v = p[t]; s += v.x + v.y + v.z + v.w; }
            xsum16[(size_t)b * (K / 16) + j] = s;
        }
        bar_sync_consumers(CONSUMERS);
    }

    constexpr int ELEMS = Unit<FMT>::ELEMS;
    constexpr int UNITS_PER_CHUNK = C::KC / ELEMS;
    int it = 0;
    bool ok = true;
    for (int t = 0; t < my_tiles && ok; ++t) {
        const int tile = blockIdx.x + t * gridDim.x;
        const int row_base = tile * C::RT + warp * C::R;
        float acc[C::R][NBG];
#pragma unroll
        for (int r = 0; r < C::R; ++r)
#pragma unroll
            for (int b = 0; b < NBG; ++b) acc[r][b] = 0.f;
        for (int chunk = 0; chunk < n_chunks; ++chunk, ++it) {
            const int stage = it % STAGES;
            const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
            if (!mbar_wait(&full[stage], ph)) {
                if (a.err && lane == 0) atomicOr(a.err, 2u);
                ok = false;
                break;
            }
            const int kc = min(C::KC, K - chunk * C::KC);
            const int units = kc / ELEMS;
            const uint8_t* qs = qbuf + (size_t)stage * Lay::QSTAGE;
            const uint16_t* sc = reinterpret_cast<const uint16_t*>(sbuf + (size_t)stage * Lay::SSTAGE);
#pragma unroll
            for (int j = 0; j < C::UPL; ++j) {
                const int ul = lane + 32 * j;
                if (ul < units) {
                    const int u = chunk * UNITS_PER_CHUNK + ul;
                    Raw raw[C::R];
#pragma unroll
                    for (int r = 0; r < C::R; ++r) {
                        const uint8_t* srow = qs + (size_t)(warp * C::R + r) * chunk_bytes<FMT>(C::KC);
                        if constexpr (FMT == FMT_Q8_0) {
                            raw[r].q = *reinterpret_cast<const uint4*>(srow + 16 * ul);
                            raw[r].sc = sc[(warp * C::R + r) * (C::KC / 32) + (ul >> 1)];
                        } else if constexpr (FMT == FMT_Q4_K) {
                            const uint8_t* blk = srow + (ul >> 2) * 144;
                            raw[r].q = *reinterpret_cast<const uint4*>(blk + 16 + 32 * (ul & 3));
                            raw[r].q2 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * (ul & 3));
                            raw[r].hdr = *reinterpret_cast<const uint4*>(blk);
                        } else {
                            raw[r].q = *reinterpret_cast<const uint4*>(srow + 16 * ul);
                        }
                    }
                    if constexpr (FMT == FMT_Q4_K && NBG > 1) {
                        // several activation rows: each code is turned into a float once
#pragma unroll
                        for (int r = 0; r < C::R; ++r) dot_q4k_rows<NBG>(raw[r], u, xs, KP, xsum16, K / 16, a.B, acc[r]);
                    } else if constexpr (FMT == FMT_Q8_0 && NBG > 1) {
#pragma unroll
                        for (int r = 0; r < C::R; ++r) dot_q8_rows<NBG>(raw[r], u, xs, KP, a.B, acc[r]);
                    } else {
#pragma unroll
                        for (int b = 0; b < NBG; ++b) {
                            if (b < a.B) {
                                XFrag<FMT> xf;
                                load_x<FMT>(xs + (size_t)b * KP, u, xf);
#pragma unroll
                                for (int r = 0; r < C::R; ++r)
                                    acc[r][b] += dot_frag<FMT>(raw[r], u, xf, xsum16 + (size_t)b * (K / 16));
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
        }
        if (!ok) break;
        // ---- reduce over lanes, epilogue by lane 0 (rows of this warp)
#pragma unroll
        for (int r = 0; r < C::R; ++r)
#pragma unroll
            for (int b = 0; b < NBG; ++b) acc[r][b] = warp_sum(acc[r][b]);
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < NBG; ++b) {
                if (b >= a.B) continue;
                float* yrow = a.y + (size_t)b * a.y_stride;
                if (a.epi == EPI_SWIGLU) {
#pragma unroll
                    for (int r = 0; r + 1 < C::R; r += 2)
                        if (row_base + r + 1 < N)
                            yrow[(row_base + r) >> 1] = silu(acc[r][b] * inv[b]) * (acc[r + 1][b] * inv[b]);
                } else {
                    unsigned long long kbest = 0ull;
#pragma unroll
                    for (int r = 0; r < C::R; ++r) {
                        const int row = row_base + r;
                        if (row >= N) continue;
                        const float v = acc[r][b] * inv[b];
                        if (a.epi == EPI_ADD) yrow[row] += v;
                        else yrow[row] = v;
                        if (a.epi == EPI_LOGITS) {
                            unsigned long long kk = argmax_key(v, (uint32_t)row);
                            kbest = kk > kbest ? kk : kbest;
                        }
                    }
                    if (a.epi == EPI_LOGITS) atomicMax(&best[b], kbest);
                }
            }
        }
    }
    if (a.epi == EPI_LOGITS) {
        bar_sync_consumers(CONSUMERS);
        if (tid < a.B) atomicMax(&a.st->keys[tid], best[tid]);
    }
}

int g_sms_t = 0;

template <int FMT, int NBG>
struct OccT {
    static int ctas_per_sm;
};
template <int FMT, int NBG>
int OccT<FMT, NBG>::ctas_per_sm = 1;

template <int FMT, int NBG>
bool launch_t(const GemvArgs& a, cudaStream_t s, bool pdl) {
    using C = TCfg<FMT>;
    const size_t smem = TLayout<FMT, NBG>::bytes(a.W.K);
    if (smem > 200 * 1024) return false;
    const int tiles = (a.W.N + C::RT - 1) / C::RT;
    // fewer row tiles than SMs (the 1024-row O and down projections of small models): the
    // register-fed kernel, which also splits K inside a CTA, keeps more SMs streaming
    if (tiles < g_sms_t && !a.starve) return false;
    TmaParams prm;
    prm.maps = *a.W.tm;
    prm.a = a;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(tiles, OccT<FMT, NBG>::ctas_per_sm * g_sms_t));
    cfg.blockDim = dim3(THREADS_T);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaLaunchKernelEx(&cfg, gemv_tma_kernel<FMT, NBG>, prm);
    return true;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool encode(void* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
            uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE) {
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(reinterpret_cast<CUtensorMap*>(map), dt, 2, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool load_encoder() {
    if (g_encode) return true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess || !fn)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

template <int FMT, int NBG>
void prepare_t(int optin) {
    cudaFuncAttributes fa;
    cudaFuncGetAttributes(&fa, gemv_tma_kernel<FMT, NBG>);
    cudaFuncSetAttribute(gemv_tma_kernel<FMT, NBG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         optin - (int)fa.sharedSizeBytes);
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_tma_kernel<FMT, NBG>, THREADS_T,
                                                  TLayout<FMT, NBG>::bytes(4096));
    OccT<FMT, NBG>::ctas_per_sm = occ > 0 ? occ : 1;
}

}  // namespace

void gemv_tma_prepare() {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&g_sms_t, cudaDevAttrMultiProcessorCount, dev);
    prepare_t<FMT_Q8_0, 1>(optin);
    prepare_t<FMT_Q8_0, 4>(optin);
    prepare_t<FMT_Q4_K, 1>(optin);
    prepare_t<FMT_Q4_K, 4>(optin);
    prepare_t<FMT_F32, 1>(optin);
    prepare_t<FMT_F32, 4>(optin);
}

bool make_tma_maps(const QMat& W, TmaMaps* out) {
    out->ok = 0;
    out->tc_ok = 0;
    if (!load_encoder()) return false;
    if (W.fmt == FMT_Q8_0 && W.K % 64 == 0 && W.N > 0)
        // tensor-core GEMM: 64 codes x 128 rows per box, 64-byte swizzle (conflict-free row reads)
        out->tc_ok = encode(out->tcq, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.q, (uint64_t)W.K, W.N, (uint64_t)W.K, 64, 128,
                            CU_TENSOR_MAP_SWIZZLE_64B)
                         ? 1
                         : 0;
    if (W.K % 256 != 0 || W.N <= 0) return false;
    const uint64_t rb = W.row_bytes();
    bool ok = false;
    if (W.fmt == FMT_Q8_0) {
        ok = encode(out->q, CU_TENSOR_MAP_DATA_TYPE_UINT32, W.q, (uint64_t)W.K / 4, W.N, rb, TView<FMT_Q8_0>::X,
                    TCfg<FMT_Q8_0>::RT) &&
             encode(out->s, CU_TENSOR_MAP_DATA_TYPE_UINT16, W.s, (uint64_t)W.K / 32, W.N, (uint64_t)W.K / 16,
                    TCfg<FMT_Q8_0>::KC / 32, TCfg<FMT_Q8_0>::RT);
    } else if (W.fmt == FMT_Q4_K) {
        ok = encode(out->q, CU_TENSOR_MAP_DATA_TYPE_UINT64, W.q, rb / 8, W.N, rb, TView<FMT_Q4_K>::X,
                    TCfg<FMT_Q4_K>::RT);
    } else if (W.fmt == FMT_F32) {
        ok = encode(out->q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, W.q, (uint64_t)W.K, W.N, rb, TView<FMT_F32>::X,
                    TCfg<FMT_F32>::RT);
    }
    out->ok = ok ? 1 : 0;
    return ok;
}

bool encode_f16_rows_sw128(void* map, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
    if (!load_encoder()) return false;
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, K, rows, K * 2, 64, box_rows,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

bool launch_gemv_tma(const GemvArgs& a, cudaStream_t s, bool pdl) {
    if (a.route || a.B > 4 || a.W.K % 256 != 0 || g_sms_t == 0 || !a.W.tm || !a.W.tm->ok) return false;
    const bool one = a.B == 1;
    switch (a.W.fmt) {
        case FMT_Q8_0: return one ? launch_t<FMT_Q8_0, 1>(a, s, pdl) : launch_t<FMT_Q8_0, 4>(a, s, pdl);
        case FMT_Q4_K: return one ? launch_t<FMT_Q4_K, 1>(a, s, pdl) : launch_t<FMT_Q4_K, 4>(a, s, pdl);
        case FMT_F32: return one ? launch_t<FMT_F32, 1>(a, s, pdl) : launch_t<FMT_F32, 4>(a, s, pdl);
        default: return false;
    }
}

}  // namespace fq
