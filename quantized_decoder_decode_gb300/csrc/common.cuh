// Device helpers shared by the fq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

#define FQ_DEV __device__ __forceinline__

namespace fq {

constexpr int WARP = 32;

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels are launched with programmatic stream serialisation: a kernel may start while
// its predecessor is still running.  Everything before pdl_wait() must only touch data
// that no earlier kernel of the step writes (weights, cache positions of earlier steps).
FQ_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
FQ_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Warm L2 with [p, p+bytes): p 16-byte aligned, bytes a multiple of 16.  A hint only.
FQ_DEV void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Split a prefetch of an arbitrary aligned range over the threads of a CTA.
FQ_DEV void prefetch_l2_range(const void* p, uint64_t bytes, int tid, int nthreads) {
    const uint32_t CH = 16384;
    const char* c = (const char*)p;
    uint64_t n = (bytes + CH - 1) / CH;
    for (uint64_t i = tid; i < n; i += nthreads) {
        uint64_t off = i * CH;
        uint64_t len = bytes - off < CH ? bytes - off : CH;
        len &= ~(uint64_t)15;
        if (len) prefetch_l2(c + off, (uint32_t)len);
    }
}

// ---------------------------------------------------------------- loads
// Streaming loads of data read exactly once per step (weights, cache): bypass L1.
FQ_DEV uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
FQ_DEV uint2 ld_stream8(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
FQ_DEV uint32_t ld_stream4(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
FQ_DEV unsigned short ld_stream2(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// ---------------------------------------------------------------- conversions
FQ_DEV float h2f(unsigned short h) { return __half2float(__ushort_as_half(h)); }
FQ_DEV float bf2f(unsigned short h) { return __uint_as_float((uint32_t)h << 16); }
FQ_DEV float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
FQ_DEV float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Four int8 codes of one 32-bit word to exact floats: bias each byte to unsigned, place it
// in the low mantissa bits of 2^23 (byte permute: selector nibble 0 picks source byte k of
// u, nibbles 1-2 pick zero bytes and nibble 3 the 0x4B exponent byte of the constant),
// subtract 2^23 + 128.
FQ_DEV void s8x4_to_f32(uint32_t w, float* f) {
    uint32_t u = w ^ 0x80808080u;
    const float bias = 8388736.0f;  // 2^23 + 128
    f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)) - bias;
    f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)) - bias;
    f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)) - bias;
    f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)) - bias;
}

// Four unsigned bytes (values 0..255) to exact floats.
FQ_DEV void u8x4_to_f32(uint32_t u, float* f) {
    const float bias = 8388608.0f;  // 2^23
    f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)) - bias;
    f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)) - bias;
    f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)) - bias;
    f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)) - bias;
}

// ggml Q8_0 quantisation of one value x of a block whose scale is d = fp16(amax / 127):
// the code is x / d rounded half away from zero, clamped to +-127 (0 when d is 0).  The
// quotient only picks a candidate n = trunc(|x| / d); the exact answer is n or n + 1, and
// |x| >= (n + 1/2) d decides it without rounding, because (n + 1/2) d has at most 20
// significant bits (n + 1/2 below 2^8 in halves, d an fp16 of 11 bits).
FQ_DEV int q8_code(float x, float d) {
    if (!(d > 0.f)) return 0;
    const float a = fabsf(x);
    int n = (int)fminf(__fdiv_rn(a, d), 255.f);
    if (a >= ((float)n + 0.5f) * d) ++n;
    n = n > 127 ? 127 : n;
    return x < 0.f ? -n : n;
}

// Q8_0 quantisation of a block of 32 values held 4 per lane by 8 consecutive lanes (lanes
// 8j..8j+7 of a warp, all of which call this): returns the lane's 4 codes as bytes of one
// word and sets the fp16 scale.  d = fp16(amax / 127), rounded to nearest even; the f32
// quotient cannot move amax / 127 across an fp16 rounding boundary (such a boundary lies
// more than half an f32 ulp away from any quotient of an f32 by 127 that is not on it).
FQ_DEV uint32_t q8_quant_lane4(const float v[4], unsigned short& d_bits, float& d) {
    float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 4));
    const __half dh = __float2half_rn(__fdiv_rn(am, 127.f));
    d = __half2float(dh);
    d_bits = __half_as_ushort(dh);
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) w |= ((uint32_t)q8_code(v[j], d) & 0xFFu) << (8 * j);
    return w;
}

// Order-preserving map of a float to u32 (larger float -> larger key).
FQ_DEV uint32_t float_order_key(float f) {
    uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// argmax key: value in the high word, and ~index in the low word so that equal values
// resolve to the lowest index under an unsigned max.
FQ_DEV unsigned long long argmax_key(float v, uint32_t idx) {
    return ((unsigned long long)float_order_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
FQ_DEV uint32_t argmax_key_index(unsigned long long k) { return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu); }

// ---------------------------------------------------------------- reductions
FQ_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
FQ_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Sum over all threads of a CTA (blockDim.x a multiple of 32, <= 1024); red: >= 32 floats.
FQ_DEV float block_sum(float v, float* red) {
    int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    float t = lane < nw ? red[lane] : 0.f;
    return warp_sum(t);
}

FQ_DEV float silu(float z) { return z / (1.0f + expf(-z)); }

}  // namespace fq
