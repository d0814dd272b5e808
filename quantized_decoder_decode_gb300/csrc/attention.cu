// Grouped causal attention of one new query row per sequence against its KvCache, as a
// split-K flash-decode (sm_103a CUDA cores).
//
// The fucina runner page lists, for the .fused block style, half-rope QK-norm and grouped
// causal attention over the shared KvCache; section 14.1 fixes that a step appends the
// new K/V at pos == len.  One CTA owns (sequence b, kv head g, chunk s of positions); the
// G = n_q / n_kv query heads of the group share every K/V row it streams.  Fused here:
//   * per-head RMSNorm of q and k with the learned gains, then rotate-half RoPE at the
//     absolute position (cos/sin table), q pre-scaled by log2(e)/sqrt(128);
//   * the CTA whose chunk holds the new position rounds k and v to the cache dtype,
//     writes them at pos and uses the rounded values itself;
//   * scores with one lane per position (16-byte loads along the row), online softmax
//     in base 2 per 32-position tile, V accumulation with lanes over dimensions;
//   * partial (m, l, o) per chunk; the last CTA of a (sequence, kv head) to finish
//     (atomic ticket, no waiting) merges the chunks and writes the head outputs.

#include "common.cuh"
#include "kernels.h"

#include "attn_unit.cuh"

namespace fq {

namespace {

template <int KVT, int G>
__global__ void __launch_bounds__(ATT_THREADS) attn_kernel(const AttnArgs a) {
    using T = typename KvType<KVT>::T;
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    {
        // cached rows [t0, min(t1, pos)) were written by earlier steps: warm L2 before waiting
        const SeqState ss = a.st->seq[b];
        const int pos = ss.pos, n_act = (pos + a.chunk) / a.chunk;
        const int t0 = s * a.chunk, tc = min(min(pos + 1, t0 + a.chunk), pos);
        if (s < n_act && tc > t0) {
            const size_t head_off = ((size_t)a.layer * a.Hkv + g) * (size_t)ss.cap * HEAD_DIM;
            const size_t rb = HEAD_DIM * sizeof(T);
            prefetch_l2_range(reinterpret_cast<const T*>(ss.k) + head_off + (size_t)t0 * HEAD_DIM,
                              (size_t)(tc - t0) * rb, threadIdx.x, ATT_THREADS);
            prefetch_l2_range(reinterpret_cast<const T*>(ss.v) + head_off + (size_t)t0 * HEAD_DIM,
                              (size_t)(tc - t0) * rb, threadIdx.x, ATT_THREADS);
        }
    }
    pdl_trigger();
    pdl_wait();
    __shared__ __align__(16) AttnSmem<G> sm;
    attn_unit<KVT, G>(a, s, g, b, threadIdx.x, sm, [] { __syncthreads(); });
}

template <int KVT, int G>
void launch_t(const AttnArgs& a, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.splits, a.Hkv, a.n);
    cfg.blockDim = dim3(ATT_THREADS);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaLaunchKernelEx(&cfg, attn_kernel<KVT, G>, a);
}

template <int KVT>
void launch_kv(const AttnArgs& a, cudaStream_t s, bool pdl) {
    switch (a.Hq / a.Hkv) {
        case 1: launch_t<KVT, 1>(a, s, pdl); break;
        case 2: launch_t<KVT, 2>(a, s, pdl); break;
        case 4: launch_t<KVT, 4>(a, s, pdl); break;
        case 8: launch_t<KVT, 8>(a, s, pdl); break;
        default: break;   // rejected at descriptor validation
    }
}

}  // namespace

void launch_attention(const AttnArgs& a, cudaStream_t s, bool pdl) {
    if (a.kv_bf16) launch_kv<1>(a, s, pdl);
    else launch_kv<0>(a, s, pdl);
}

}  // namespace fq
