// Small kernels around the decode step: step set-up, embedding rows, the greedy argmax
// hand-off, and load-time work (Q8_0 repacking, the rotary table, inspection dequant).

#include "common.cuh"
#include "kernels.h"
#include "quant.cuh"

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

__global__ void setup_kernel(StepState* st, const SetupArgs a) {
    int b = threadIdx.x;
    if (b < a.n) {
        SeqState& q = st->seq[b];
        q.token = a.token[b];
        q.pos = a.pos[b];
        q.cap = a.cap[b];
        q.k = a.k[b];
        q.v = a.v[b];
        q.ks = a.ks[b];
        q.vs = a.vs[b];
        st->keys[b] = 0ull;
    }
    if (b == 0) {
        st->step = 0;
        st->lm_counter = 0;
        st->tokens_out = a.tokens_out;
        st->logits = a.logits;
        st->greedy = a.greedy;
        st->n = a.n;
    }
}

// x[b][:] = embedding row of seq b's token (section 14.2: token_embd, dequantised)
__global__ void __launch_bounds__(256) embed_kernel(const QMat emb, const StepState* st, float* x) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    int64_t row = st->seq[b].token;
    if (row < 0 || row >= emb.N) row = 0;   // ids are checked on the host; never read outside the table
    float* xb = x + (size_t)b * emb.K;
    for (int k = threadIdx.x; k < emb.K; k += blockDim.x) xb[k] = dequant_one(emb, row, k);
}

// After the LM head: decode the argmax keys; for greedy chains hand the token to the next
// step, record it and advance the positions.
__global__ void lm_finish_kernel(StepState* st, int n, int vocab) {
    pdl_trigger();
    pdl_wait();
    int b = threadIdx.x;
    if (b < n) {
        unsigned long long k = st->keys[b];
        uint32_t idx = argmax_key_index(k);
        int32_t tok = idx < (uint32_t)vocab ? (int32_t)idx : 0;
        st->keys[b] = 0ull;
        if (st->greedy) {
            st->seq[b].token = tok;
            st->seq[b].pos += 1;
            if (st->tokens_out) st->tokens_out[(size_t)st->step * n + b] = tok;
        }
    }
    __syncthreads();
    if (b == 0 && st->greedy) st->step += 1;
}

// ggml Q8_0 rows (34-byte blocks) -> aligned planes; source row r goes to destination
// row dst(r) = (r / group) * group_stride + (r % group) * step + off.
__global__ void repack_q8_0_kernel(const uint8_t* src, int64_t rows, int64_t cols, uint8_t* q, uint16_t* sc,
                                   int64_t group, int64_t group_stride, int64_t step, int64_t off) {
    const int64_t nb = cols / 32;
    const int64_t total = rows * nb;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = i / nb, blk = i % nb;
        int64_t dr = (r / group) * group_stride + (r % group) * step + off;
        const uint8_t* p = src + (r * nb + blk) * 34;
        sc[dr * nb + blk] = (uint16_t)(p[0] | (p[1] << 8));
        uint8_t* dq = q + dr * cols + blk * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j) dq[j] = p[2 + j];
    }
}

// row copy with the same destination mapping (Q4_K blocks and f32 rows keep their bytes)
__global__ void copy_rows_kernel(const uint8_t* src, int64_t rows, int64_t row_bytes, uint8_t* dst, int64_t group,
                                 int64_t group_stride, int64_t step, int64_t off) {
    const int64_t words = row_bytes / 16;
    const int64_t total = rows * words;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = i / words, w = i % words;
        int64_t dr = (r / group) * group_stride + (r % group) * step + off;
        reinterpret_cast<uint4*>(dst + dr * row_bytes)[w] = reinterpret_cast<const uint4*>(src + r * row_bytes)[w];
    }
}

// cos/sin of p * theta^(-2i/128) for i < 64, evaluated in double precision once at load
__global__ void rope_table_kernel(float2* tab, int max_pos, double theta) {
    int64_t total = (int64_t)max_pos * (HEAD_DIM / 2);
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
        int p = (int)(t / (HEAD_DIM / 2)), i = (int)(t % (HEAD_DIM / 2));
        double freq = pow(theta, -2.0 * i / (double)HEAD_DIM);
        double s, c;
        sincos((double)p * freq, &s, &c);
        tab[t] = make_float2((float)c, (float)s);
    }
}

__global__ void dequant_kernel(const QMat W, int64_t row0, int64_t n_rows, float* out) {
    int64_t total = n_rows * W.K;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x)
        out[t] = dequant_one(W, row0 + t / W.K, t % W.K);
}

// Q8_0 cache rows <-> ggml blocks, one thread per (position, kv head, block of 32)
__global__ void kv_q8_copy_kernel(int8_t* codes, uint16_t* scales, size_t cap, size_t cap_s, int Hkv, int pos,
                                  int n_pos, uint8_t* blocks, int to_cache) {
    const int64_t total = (int64_t)n_pos * Hkv * (HEAD_DIM / 32);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(i % (HEAD_DIM / 32));
        const int64_t ph = i / (HEAD_DIM / 32);
        const int h = (int)(ph % Hkv);
        const int64_t p = pos + ph / Hkv;
        uint8_t* blk = blocks + i * 34;
        int8_t* c = codes + ((size_t)h * cap + p) * HEAD_DIM + 32 * j;
        uint16_t* sc = scales + ((size_t)h * cap_s + p) * (HEAD_DIM / 32) + j;
        if (to_cache) {
            *sc = (uint16_t)(blk[0] | (blk[1] << 8));
            for (int k = 0; k < 32; ++k) c[k] = (int8_t)blk[2 + k];
        } else {
            const uint16_t d = *sc;
            blk[0] = (uint8_t)(d & 0xFFu);
            blk[1] = (uint8_t)(d >> 8);
            for (int k = 0; k < 32; ++k) blk[2 + k] = (uint8_t)c[k];
        }
    }
}

// ggml Q8_0 blocks of x, one warp per 128 values, with the quantiser the attention kernel
// applies to q and to the new k and v
__global__ void quantize_q8_0_kernel(const float* x, size_t n, uint8_t* blocks) {
    const size_t rows = n / 128;
    const int lane = threadIdx.x & 31;
    const size_t warps = ((size_t)gridDim.x * blockDim.x) >> 5;
    for (size_t r = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
        const float4 f = reinterpret_cast<const float4*>(x + r * 128)[lane];
        const float v[4] = {f.x, f.y, f.z, f.w};
        unsigned short db;
        float d;
        const uint32_t w = q8_quant_lane4(v, db, d);
        uint8_t* blk = blocks + (r * 4 + (lane >> 3)) * 34;
        if ((lane & 7) == 0) {
            blk[0] = (uint8_t)(db & 0xFFu);
            blk[1] = (uint8_t)(db >> 8);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) blk[2 + 4 * (lane & 7) + j] = (uint8_t)(w >> (8 * j));
    }
}

}  // namespace

void launch_kv_q8_copy(int8_t* codes, uint16_t* scales, size_t cap, size_t cap_s, int Hkv, int pos, int n_pos,
                       uint8_t* blocks, bool to_cache, cudaStream_t s) {
    const int64_t total = (int64_t)n_pos * Hkv * (HEAD_DIM / 32);
    const int grid = (int)std::min<int64_t>((total + 255) / 256, 4096);
    kv_q8_copy_kernel<<<grid, 256, 0, s>>>(codes, scales, cap, cap_s, Hkv, pos, n_pos, blocks, to_cache ? 1 : 0);
}

void launch_quantize_q8_0(const float* x, size_t n, uint8_t* blocks, cudaStream_t s) {
    const size_t warps = n / 128;
    const int grid = (int)std::min<size_t>((warps * 32 + 255) / 256, 1024);
    if (grid > 0) quantize_q8_0_kernel<<<grid, 256, 0, s>>>(x, n, blocks);
}

void launch_setup(StepState* st, const SetupArgs& a, cudaStream_t s) {
    setup_kernel<<<1, MAX_SEQ, 0, s>>>(st, a);
}

void launch_embed(const QMat& emb, const StepState* st, int n, float* x, cudaStream_t s, bool pdl) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3(n), dim3(256), s, pdl, attr);
    cudaLaunchKernelEx(&cfg, embed_kernel, emb, st, x);
}

void launch_lm_finish(StepState* st, int n, int vocab, cudaStream_t s, bool pdl) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3(1), dim3(MAX_SEQ), s, pdl, attr);
    cudaLaunchKernelEx(&cfg, lm_finish_kernel, st, n, vocab);
}

void launch_repack_q8_0(const uint8_t* src, int64_t rows, int64_t cols, uint8_t* q, uint16_t* sc, int64_t group,
                        int64_t group_stride, int64_t step, int64_t off, cudaStream_t s) {
    int64_t total = rows * (cols / 32);
    int grid = (int)std::min<int64_t>((total + 255) / 256, 4096);
    repack_q8_0_kernel<<<grid, 256, 0, s>>>(src, rows, cols, q, sc, group, group_stride, step, off);
}

void launch_copy_rows(const uint8_t* src, int64_t rows, int64_t row_bytes, uint8_t* dst, int64_t group,
                      int64_t group_stride, int64_t step, int64_t off, cudaStream_t s) {
    int64_t total = rows * (row_bytes / 16);
    int grid = (int)std::min<int64_t>((total + 255) / 256, 4096);
    copy_rows_kernel<<<grid, 256, 0, s>>>(src, rows, row_bytes, dst, group, group_stride, step, off);
}

void launch_rope_table(float2* tab, int max_pos, double theta, cudaStream_t s) {
    rope_table_kernel<<<1024, 256, 0, s>>>(tab, max_pos, theta);
}

void launch_dequant(const QMat& W, int64_t row0, int64_t n_rows, float* out, cudaStream_t s) {
    dequant_kernel<<<1024, 256, 0, s>>>(W, row0, n_rows, out);
}

}  // namespace fq
