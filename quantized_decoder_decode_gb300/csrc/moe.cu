// Mixture-of-experts pieces of the decode step (fucina section 14.2: the qwen3moe FFN
// routes with a softmax top-k -- routerTopK with normalize_selected = norm_topk_prob --
// and runs the router-weighted SwiGLU mixture; decode reads each selected expert once for
// all tokens that chose it).  The router logits and the expert contractions run in the
// GEMV kernel (F32 rows, then expert mode); this file holds the selection, the grouping
// of (token, slot) pairs by expert, and the weighted combine.

#include "common.cuh"
#include "kernels.h"

namespace fq {

namespace {

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, cudaStream_t s, bool pdl, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

// One warp per token: k rounds of (max logit, lowest index) over the unselected experts.
// Selecting on logits equals selecting on softmax probabilities (exp is increasing).
// Weights: exp(l_j - max) over the selected sum (norm_topk) or over all experts.
__global__ void __launch_bounds__(256) route_kernel(const float* logits, int E, int k, int n, int norm_topk,
                                                    MoeRoute* rt) {
    pdl_trigger();
    pdl_wait();
    __shared__ int sidx[MAX_SEQ * MAX_TOPK];
    __shared__ int cnt[MAX_EXPERTS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int b = warp; b < n; b += blockDim.x / 32) {
        const float* l = logits + (size_t)b * E;
        float v[MAX_EXPERTS / 32];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < MAX_EXPERTS / 32; ++i) {
            int e = lane + 32 * i;
            v[i] = e < E ? l[e] : -INFINITY;
            mx = fmaxf(mx, v[i]);
        }
        mx = warp_max(mx);
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < MAX_EXPERTS / 32; ++i) tot += (lane + 32 * i < E) ? expf(v[i] - mx) : 0.f;
        tot = warp_sum(tot);
        float selsum = 0.f;
        float wsel[MAX_TOPK];
        int isel[MAX_TOPK];
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int bi = 0x7FFFFFFF;
#pragma unroll
            for (int i = 0; i < MAX_EXPERTS / 32; ++i) {
                int e = lane + 32 * i;
                if (e < E && (v[i] > bv || (v[i] == bv && e < bi))) { bv = v[i]; bi = e; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
                int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if (bi >= E) bi = 0;   // only reachable with NaN logits; keeps every index in range
            isel[j] = bi;
            wsel[j] = expf(bv - mx);
            selsum += wsel[j];
#pragma unroll
            for (int i = 0; i < MAX_EXPERTS / 32; ++i)   // remove the winner from the candidates
                if (lane + 32 * i == bi) v[i] = -INFINITY;
        }
        if (lane == 0) {
            float den = norm_topk ? selsum : tot;
            for (int j = 0; j < k; ++j) {
                rt->idx[b * k + j] = isel[j];
                rt->w[b * k + j] = wsel[j] / den;
                sidx[b * k + j] = isel[j];
                atomicAdd(&cnt[isel[j]], 1);
            }
        }
    }
    __syncthreads();
    // active experts in ascending id order, with their pair ranges
    if (tid == 0) {
        int na = 0, off = 0;
        for (int e = 0; e < E; ++e) {
            if (cnt[e] == 0) continue;
            rt->expert[na] = e;
            rt->start[na] = off;
            off += cnt[e];
            ++na;
        }
        rt->start[na] = off;
        rt->n_active = na;
    }
    __syncthreads();
    // pairs of expert e in (token, slot) order; thread e scans the selections
    for (int e = tid; e < E; e += blockDim.x) {
        if (cnt[e] == 0) continue;
        int a = 0;
        for (int i = 0; i < E && rt->expert[i] != e; ++i) ++a;   // position of e among active
        int w = rt->start[a];
        for (int p = 0; p < n * k; ++p)
            if (sidx[p] == e) {
                rt->pair_token[w] = p / k;
                rt->pair_slot[w] = p % k;
                ++w;
            }
    }
}

__global__ void __launch_bounds__(256) combine_kernel(float* x, const float* y, const MoeRoute* rt, int k, int H) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    for (int i = threadIdx.x; i < H; i += blockDim.x) {
        float acc = 0.f;
        for (int j = 0; j < k; ++j) acc = fmaf(rt->w[b * k + j], y[((size_t)b * k + j) * H + i], acc);
        x[(size_t)b * H + i] += acc;
    }
}

}  // namespace

void launch_moe_route(const float* logits, int E, int k, int n, int norm_topk, MoeRoute* route, cudaStream_t s,
                      bool pdl) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3(1), dim3(256), s, pdl, attr);
    cudaLaunchKernelEx(&cfg, route_kernel, logits, E, k, n, norm_topk, route);
}

void launch_moe_combine(float* x, const float* y, const MoeRoute* route, int n, int k, int H, cudaStream_t s,
                        bool pdl) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3(n), dim3(256), s, pdl, attr);
    cudaLaunchKernelEx(&cfg, combine_kernel, x, y, route, k, H);
}

}  // namespace fq
