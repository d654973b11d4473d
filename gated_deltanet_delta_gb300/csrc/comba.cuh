// comba.cuh -- the Comba decode-step kernel (one token, fp32 (K, V) state streamed once).
//
// What it computes: KBench specs/comba_decode_step.py, spec_md, for every (b, h) head with i over K
// and j over V (V contiguous):
//     S = exp(g) state;  u_j = beta (v_j - sum_i p_i S_ij);  S_new_ij = S_ij + k_i u_j;
//     o_j = sum_i (scale q_i) S_new_ij.
//
// GB300 mapping.  One CTA holds one head's whole K x V slab in registers (the resident-slab
// schedule the spec's perf_md asks for): thread (c, rg) owns column group c (4 adjacent columns,
// one float4) and the K/RG rows rg, rg+RG, ...  At a fixed row index a warp reads 32 consecutive
// float4, i.e. whole 512-byte rows when V = 128, so every load and store is a coalesced 16-byte
// access.  The reduction over K runs serially in registers per thread, then across the RG row
// groups through shared memory (one barrier for u, one for o).  p, k and scale*q are staged once
// per CTA as fp32.  The state is read once and written once.
#pragma once

#include "common.cuh"
#include "kernel_args.h"

namespace gdn {

template <int K, int V, int NT>
__global__ void __launch_bounds__(NT) comba_decode_kernel(const CombaArgs a) {
    constexpr int CG = V / 4;      // float4 column groups
    constexpr int RG = NT / CG;    // row groups
    constexpr int NR = K / RG;     // rows per thread
    static_assert(CG * 4 == V && RG * CG == NT && NR * RG == K, "tile split");

    __shared__ float ps[K], ks[K], qs[K];
    __shared__ float4 red_u[RG][CG];
    __shared__ float4 red_o[RG][CG];

    const size_t head = blockIdx.x;
    const int c = threadIdx.x % CG;
    const int rg = threadIdx.x / CG;
    const float4* src = reinterpret_cast<const float4*>(a.state + head * K * V);
    float4* dst = reinterpret_cast<float4*>(a.state_new + head * K * V);

    // 1. every state load of this thread first
    float4 s[NR];
#pragma unroll
    for (int m = 0; m < NR; ++m) s[m] = ld_stream(src + size_t(rg + RG * m) * CG + c);

    // 2. stage p, k, scale*q (fp32) and the head's scalars
    for (int i = threadIdx.x; i < K / 4; i += NT) {
        const float4 pp = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.p + head * K + 4 * i));
        const float4 kk = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.k + head * K + 4 * i));
        const float4 qq = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.q + head * K + 4 * i));
        ps[4 * i] = pp.x; ps[4 * i + 1] = pp.y; ps[4 * i + 2] = pp.z; ps[4 * i + 3] = pp.w;
        ks[4 * i] = kk.x; ks[4 * i + 1] = kk.y; ks[4 * i + 2] = kk.z; ks[4 * i + 3] = kk.w;
        qs[4 * i] = a.scale * qq.x; qs[4 * i + 1] = a.scale * qq.y;
        qs[4 * i + 2] = a.scale * qq.z; qs[4 * i + 3] = a.scale * qq.w;
    }
    const float gate = expf(a.g[head]);
    const float beta = bf16_to_f32(a.beta[head]);
    const float4 vv = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.v + head * V + 4 * c));
    __syncthreads();

    // 3. decay and this thread's part of S^T p
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < NR; ++m) {
        const float pi = ps[rg + RG * m];
        float4& x = s[m];
        x.x *= gate; x.y *= gate; x.z *= gate; x.w *= gate;
        r.x = fmaf(pi, x.x, r.x);
        r.y = fmaf(pi, x.y, r.y);
        r.z = fmaf(pi, x.z, r.z);
        r.w = fmaf(pi, x.w, r.w);
    }
    red_u[rg][c] = r;
    __syncthreads();
    r = red_u[0][c];
#pragma unroll
    for (int j = 1; j < RG; ++j) {
        const float4 t = red_u[j][c];
        r.x += t.x; r.y += t.y; r.z += t.z; r.w += t.w;
    }
    const float4 u = make_float4(beta * (vv.x - r.x), beta * (vv.y - r.y), beta * (vv.z - r.z),
                                 beta * (vv.w - r.w));

    // 4. rank-1 write with k, store, and this thread's part of the readout
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < NR; ++m) {
        const int i = rg + RG * m;
        const float ki = ks[i], qi = qs[i];
        float4& x = s[m];
        x.x = fmaf(ki, u.x, x.x);
        x.y = fmaf(ki, u.y, x.y);
        x.z = fmaf(ki, u.z, x.z);
        x.w = fmaf(ki, u.w, x.w);
        st_stream(dst + size_t(i) * CG + c, x);
        o.x = fmaf(qi, x.x, o.x);
        o.y = fmaf(qi, x.y, o.y);
        o.z = fmaf(qi, x.z, o.z);
        o.w = fmaf(qi, x.w, o.w);
    }
    red_o[rg][c] = o;
    __syncthreads();
    if (rg == 0) {
#pragma unroll
        for (int j = 1; j < RG; ++j) {
            const float4 t = red_o[j][c];
            o.x += t.x; o.y += t.y; o.z += t.z; o.w += t.w;
        }
        if (a.o_f32) {
            reinterpret_cast<float4*>(static_cast<float*>(a.o) + head * V)[c] = o;
        } else {
            uint2 pk;
            pk.x = uint32_t(f32_to_bf16_rne(o.x)) | (uint32_t(f32_to_bf16_rne(o.y)) << 16);
            pk.y = uint32_t(f32_to_bf16_rne(o.z)) | (uint32_t(f32_to_bf16_rne(o.w)) << 16);
            reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.o) + head * V)[c] = pk;
        }
    }
}

}  // namespace gdn
