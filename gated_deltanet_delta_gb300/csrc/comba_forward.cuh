// comba_forward.cuh -- the Comba recurrence over T tokens per head, the state slab held on chip.
#pragma once

#include "common.cuh"
#include "kernel_args.h"

namespace gdn {

// The Comba recurrence over T tokens of one head (KBench specs/comba_decode_step.py, spec_md: the
// decode step is the comba-forward task's recurrence for one token, and T steps reproduce that
// task).  The decode kernel's layout, with the slab held in registers across the tokens: the state
// is read once and written once per call.  Per token two barriers (the two reductions over K); the
// next token's p, k, q, v, g and beta are loaded into registers while the current one is computed
// and land in the other half of the double-buffered shared vectors before the second barrier.
template <int K, int V, int NT>
__global__ void __launch_bounds__(NT) comba_forward_kernel(const CombaFwdArgs a) {
    constexpr int CG = V / 4;      // float4 column groups
    constexpr int RG = NT / CG;    // row groups
    constexpr int NR = K / RG;     // rows per thread
    constexpr int KL = K / 4;      // threads that stage p, k and q (4 elements each)
    static_assert(CG * 4 == V && RG * CG == NT && NR * RG == K && KL <= NT, "tile split");

    __shared__ float4 ps[2][KL], ks[2][KL], qs[2][KL];
    __shared__ float4 red_u[2][RG][CG];
    __shared__ float4 red_o[2][RG][CG];

    const int head = blockIdx.x;  // b * H + h
    const int b = head / a.H, h = head - b * a.H;
    const int c = threadIdx.x % CG;
    const int rg = threadIdx.x / CG;
    const int T = a.T;
    float4* st = reinterpret_cast<float4*>(a.state + size_t(head) * K * V);
    auto tok = [&](int t) { return (size_t(b) * T + t) * a.H + h; };  // token t of this head

    // 1. every state load of this thread first
    float4 s[NR];
#pragma unroll
    for (int m = 0; m < NR; ++m) s[m] = ld_stream(st + size_t(rg + RG * m) * CG + c);

    // 2. token 0's vectors and scalars
    uint2 np = make_uint2(0u, 0u), nk = np, nq = np, nv = np;
    float ng = 0.f;
    uint16_t nb = 0;
    auto fetch = [&](int t) {  // token t's inputs into registers
        const size_t n = tok(t);
        if (threadIdx.x < KL) {
            np = *reinterpret_cast<const uint2*>(a.p + n * K + 4 * threadIdx.x);
            nk = *reinterpret_cast<const uint2*>(a.k + n * K + 4 * threadIdx.x);
            nq = *reinterpret_cast<const uint2*>(a.q + n * K + 4 * threadIdx.x);
        }
        nv = *reinterpret_cast<const uint2*>(a.v + n * V + 4 * c);
        ng = a.g[n];
        nb = a.beta[n];
    };
    auto stage = [&](int buf) {  // the fetched p, k, scale*q into shared buffer `buf`
        if (threadIdx.x < KL) {
            ps[buf][threadIdx.x] = bf16x4_to_f32x4(np);
            ks[buf][threadIdx.x] = bf16x4_to_f32x4(nk);
            const float4 qq = bf16x4_to_f32x4(nq);
            qs[buf][threadIdx.x] = make_float4(a.scale * qq.x, a.scale * qq.y, a.scale * qq.z, a.scale * qq.w);
        }
    };
    if (T > 0) {
        fetch(0);
        stage(0);
    }
    __syncthreads();
    const float* psf = reinterpret_cast<const float*>(ps);
    const float* ksf = reinterpret_cast<const float*>(ks);
    const float* qsf = reinterpret_cast<const float*>(qs);

    for (int t = 0; t < T; ++t) {
        const int bf = t & 1;
        const float gate = expf(ng);
        const float beta = bf16_to_f32(nb);
        const float4 vv = bf16x4_to_f32x4(nv);
        if (t + 1 < T) fetch(t + 1);

        // 3. decay and this thread's part of S^T p (packed f32x2 arithmetic on column pairs)
        const float2 g2 = make_float2(gate, gate);
        float2 r01 = make_float2(0.f, 0.f), r23 = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < NR; ++m) {
            const float pi = psf[bf * K + rg + RG * m];
            const float2 p2 = make_float2(pi, pi);
            float4& x = s[m];
            float2 x01 = __fmul2_rn(make_float2(x.x, x.y), g2);
            float2 x23 = __fmul2_rn(make_float2(x.z, x.w), g2);
            r01 = __ffma2_rn(p2, x01, r01);
            r23 = __ffma2_rn(p2, x23, r23);
            x = make_float4(x01.x, x01.y, x23.x, x23.y);
        }
        float4 r = make_float4(r01.x, r01.y, r23.x, r23.y);
        red_u[bf][rg][c] = r;
        __syncthreads();
        r = red_u[bf][0][c];
#pragma unroll
        for (int j = 1; j < RG; ++j) {
            const float4 y = red_u[bf][j][c];
            r.x += y.x; r.y += y.y; r.z += y.z; r.w += y.w;
        }
        const float4 u = make_float4(beta * (vv.x - r.x), beta * (vv.y - r.y), beta * (vv.z - r.z),
                                     beta * (vv.w - r.w));

        // 4. rank-1 write with k and this thread's part of the readout
        const float2 u01 = make_float2(u.x, u.y), u23 = make_float2(u.z, u.w);
        float2 o01 = make_float2(0.f, 0.f), o23 = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < NR; ++m) {
            const int i = rg + RG * m;
            const float ki = ksf[bf * K + i], qi = qsf[bf * K + i];
            const float2 k2 = make_float2(ki, ki), q2 = make_float2(qi, qi);
            float4& x = s[m];
            const float2 x01 = __ffma2_rn(k2, u01, make_float2(x.x, x.y));
            const float2 x23 = __ffma2_rn(k2, u23, make_float2(x.z, x.w));
            o01 = __ffma2_rn(q2, x01, o01);
            o23 = __ffma2_rn(q2, x23, o23);
            x = make_float4(x01.x, x01.y, x23.x, x23.y);
        }
        float4 o = make_float4(o01.x, o01.y, o23.x, o23.y);
        red_o[bf][rg][c] = o;
        if (t + 1 < T) stage(bf ^ 1);  // its last readers (token t - 1) passed this token's first barrier
        __syncthreads();
        if (rg == 0) {
#pragma unroll
            for (int j = 1; j < RG; ++j) {
                const float4 y = red_o[bf][j][c];
                o.x += y.x; o.y += y.y; o.z += y.z; o.w += y.w;
            }
            const size_t n = tok(t);
            if (a.o_f32) {
                reinterpret_cast<float4*>(static_cast<float*>(a.o) + n * V)[c] = o;
            } else {
                uint2 pk;
                pk.x = uint32_t(f32_to_bf16_rne(o.x)) | (uint32_t(f32_to_bf16_rne(o.y)) << 16);
                pk.y = uint32_t(f32_to_bf16_rne(o.z)) | (uint32_t(f32_to_bf16_rne(o.w)) << 16);
                reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.o) + n * V)[c] = pk;
            }
        }
    }

    // 5. the state after the last token
#pragma unroll
    for (int m = 0; m < NR; ++m) st_stream(st + size_t(rg + RG * m) * CG + c, s[m]);
}

}  // namespace gdn
