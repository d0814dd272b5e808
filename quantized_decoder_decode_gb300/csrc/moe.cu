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
// Weights: exp(l_j - max) over the selected sum (norm_topk) or over all experts.  The grouping
// of (token, slot) pairs by expert is built in shared memory: counts, an exclusive scan in
// expert order, then each pair's rank among the earlier pairs of its expert.
__global__ void __launch_bounds__(256) route_kernel(const float* logits, int E, int k, int n, int norm_topk,
                                                    MoeRoute* rt) {
    pdl_trigger();
    pdl_wait();
    __shared__ int sidx[MAX_SEQ * MAX_TOPK];
    __shared__ int cnt[MAX_EXPERTS];
    __shared__ int pos_of[MAX_EXPERTS];       // first grouped slot of expert e
    __shared__ int na_s;
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
    // active experts in ascending id order, with their pair ranges (warp 0: ballot scan)
    if (warp == 0) {
        int na = 0, off = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e < E ? cnt[e] : 0;
            const unsigned act = __ballot_sync(0xFFFFFFFFu, c > 0);
            int pre = c;   // inclusive scan of the counts over the lanes
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xFFFFFFFFu, pre, o);
                if (lane >= o) pre += t;
            }
            if (c > 0) {
                const int a = na + __popc(act & ((1u << lane) - 1u));
                rt->expert[a] = e;
                rt->start[a] = off + pre - c;
                pos_of[e] = off + pre - c;
            }
            na += __popc(act);
            off += __shfl_sync(0xFFFFFFFFu, pre, 31);
        }
        if (lane == 0) {
            rt->start[na] = off;
            rt->n_active = na;
            na_s = na;
        }
    }
    __syncthreads();
    // pair p goes to its expert's range after the earlier pairs of the same expert
    for (int p = tid; p < n * k; p += blockDim.x) {
        const int e = sidx[p];
        int rank = 0;
        for (int q = 0; q < p; ++q) rank += sidx[q] == e;
        const int w = pos_of[e] + rank;
        rt->pair_token[w] = p / k;
        rt->pair_slot[w] = p % k;
    }
}

// x[b][i] += sum_j w[b][j] y[b*k + j][i]; grid (n, column slices of 1024)
__global__ void __launch_bounds__(256) combine_kernel(float* x, const float* y, const MoeRoute* rt, int k, int H) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    const int i = blockIdx.y * 1024 + 4 * threadIdx.x;
    if (i >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const float wj = rt->w[b * k + j];
        const float4 v = *reinterpret_cast<const float4*>(y + ((size_t)b * k + j) * H + i);
        acc.x = fmaf(wj, v.x, acc.x);
        acc.y = fmaf(wj, v.y, acc.y);
        acc.z = fmaf(wj, v.z, acc.z);
        acc.w = fmaf(wj, v.w, acc.w);
    }
    float4* xp = reinterpret_cast<float4*>(x + (size_t)b * H + i);
    float4 xv = *xp;
    xv.x += acc.x; xv.y += acc.y; xv.z += acc.z; xv.w += acc.w;
    *xp = xv;
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
    cudaLaunchConfig_t cfg = make_cfg(dim3(n, (H + 1023) / 1024), dim3(256), s, pdl, attr);
    cudaLaunchKernelEx(&cfg, combine_kernel, x, y, route, k, H);
}

}  // namespace fq
