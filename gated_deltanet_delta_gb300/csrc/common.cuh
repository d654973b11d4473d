// common.cuh -- small device helpers shared by the kernels of libgdn (bf16 widening and rounding,
// streaming loads and stores, warp reductions).  Nothing here is specific to one operation.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr unsigned kFullMask = 0xffffffffu;

// bfloat16 is the upper half of an IEEE float: widening is exact.
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

// Four packed bf16 (8 bytes, element 0 in the low half of .x) to a float4.
__device__ __forceinline__ float4 bf16x4_to_f32x4(uint2 p) {
    return make_float4(__uint_as_float(p.x << 16), __uint_as_float(p.x & 0xffff0000u),
                       __uint_as_float(p.y << 16), __uint_as_float(p.y & 0xffff0000u));
}

// Round a float to bfloat16, nearest-even (finite inputs; NaN stays NaN).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return uint16_t((u >> 16) | 0x40u);  // quiet NaN
    u += 0x7fffu + ((u >> 16) & 1u);
    return uint16_t(u >> 16);
}

// Two floats rounded to bf16 (nearest even, hardware conversion) packed as (lo, hi) halves.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Streaming 16-byte load / store: the state is touched once per call, so it is not kept in L1 and
// is marked evict-first in L2.
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, const float4& v) { __stcs(p, v); }

// Sum over aligned groups of W consecutive lanes (W a power of two <= 32).
template <int W>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) x += __shfl_xor_sync(kFullMask, x, o);
    return x;
}

__device__ __forceinline__ float dot4(const float4& a, const float4& b) {
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}

}  // namespace gdn
