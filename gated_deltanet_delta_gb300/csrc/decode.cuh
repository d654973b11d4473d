// decode.cuh -- the GDN decode-step kernel (one token, fp32 state streamed once).
//
// What it computes: metaltile-std gated_delta.rs, module doc "Recurrence per step", for every
// (b, hv) head and state row r (Dv rows of Dk columns, Dk contiguous):
//     S'[r,:] = g S[r,:];  kv_r = S'[r,:] . k;  delta_r = (v_r - kv_r) beta;
//     S_new[r,:] = S'[r,:] + delta_r k;  y_r = scale * S_new[r,:] . q
// with key head hk = hv / (Hv / Hk) (the page's DISPATCH INVARIANTS).
//
// GB300 mapping.  The step is a stream of the fp32 state: 4 bytes in and 4 bytes out per element
// against ~6 flops, so HBM bandwidth is the only bound.  Each state row is split over TPR adjacent
// lanes; every lane owns NV float4 (16-byte) pieces of the row, TPR*16 bytes apart, so a warp's
// load instruction reads 32/TPR whole 128-byte segments.  A thread owns RPT rows and issues all of
// its RPT*NV 16-byte loads before any arithmetic (bytes in flight per SM = resident threads x
// RPT*NV*16).  kv and y are reduced with xor-shuffles inside the TPR-lane group; q and k are staged
// once per CTA in shared memory as fp32.  The state is never re-read: decay, update, store and the
// readout happen on the registers that the loads filled.
#pragma once

#include "common.cuh"
#include "kernel_args.h"

namespace gdn {

template <int DK, int TPR, int RPT, int NT>
__global__ void __launch_bounds__(NT) gdn_decode_kernel(const DecodeArgs a) {
    constexpr int NV = DK / (4 * TPR);  // float4 pieces per lane per row
    constexpr int RPP = NT / TPR;       // rows per pass of the CTA
    constexpr int ROWS = RPP * RPT;     // rows per CTA
    static_assert(NV * 4 * TPR == DK, "row split");
    static_assert(32 % TPR == 0, "a row group must not straddle warps");

    __shared__ float4 ks[DK / 4];
    __shared__ float4 qs[DK / 4];

    const int head = blockIdx.x / a.tiles;  // n = b * Hv + hv
    const int tile = blockIdx.x - head * a.tiles;
    const int hv = head % a.Hv;
    const int b = head / a.Hv;
    const int hk = hv / (a.Hv / a.Hk);
    const int lr = threadIdx.x % TPR;
    const int rw = threadIdx.x / TPR;

    const size_t head_off = size_t(head) * a.Dv * DK;
    const float4* src = reinterpret_cast<const float4*>(a.state_in + head_off);
    float4* dst = reinterpret_cast<float4*>(a.state_out + head_off);

    // 1. issue every state load of this thread first
    float4 s[RPT][NV];
    int row[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        row[r] = tile * ROWS + r * RPP + rw;
        const bool ok = row[r] < a.Dv;
#pragma unroll
        for (int m = 0; m < NV; ++m)
            s[r][m] = ok ? ld_stream(src + size_t(row[r]) * (DK / 4) + lr + TPR * m)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // 2. stage k and q of key head hk (bf16 -> fp32) and the per-row / per-head scalars
    const size_t qk_off = (size_t(b) * a.Hk + hk) * DK;
    for (int i = threadIdx.x; i < DK / 4; i += NT) {
        ks[i] = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.k + qk_off + 4 * i));
        qs[i] = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.q + qk_off + 4 * i));
    }
    const float gate = a.g[head];
    const float beta = bf16_to_f32(a.beta[head]);
    float vr[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r)
        vr[r] = row[r] < a.Dv ? bf16_to_f32(a.v[size_t(head) * a.Dv + row[r]]) : 0.f;
    __syncthreads();

    // 3. per row: decay + kv, delta, rank-1 update + store, readout
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        float kv = 0.f;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
            const float4 kk = ks[lr + TPR * m];
            float4& x = s[r][m];
            x.x *= gate;
            x.y *= gate;
            x.z *= gate;
            x.w *= gate;
            kv = fmaf(x.x, kk.x, kv);
            kv = fmaf(x.y, kk.y, kv);
            kv = fmaf(x.z, kk.z, kv);
            kv = fmaf(x.w, kk.w, kv);
        }
        kv = group_sum<TPR>(kv);
        const float delta = (vr[r] - kv) * beta;
        float acc = 0.f;
        const bool ok = row[r] < a.Dv;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
            const float4 kk = ks[lr + TPR * m];
            const float4 qq = qs[lr + TPR * m];
            float4& x = s[r][m];
            x.x = fmaf(delta, kk.x, x.x);
            x.y = fmaf(delta, kk.y, x.y);
            x.z = fmaf(delta, kk.z, x.z);
            x.w = fmaf(delta, kk.w, x.w);
            if (ok) st_stream(dst + size_t(row[r]) * (DK / 4) + lr + TPR * m, x);
            acc = fmaf(x.x, qq.x, acc);
            acc = fmaf(x.y, qq.y, acc);
            acc = fmaf(x.z, qq.z, acc);
            acc = fmaf(x.w, qq.w, acc);
        }
        acc = group_sum<TPR>(acc);
        if (ok && lr == 0) {
            const float yv = a.scale * acc;
            const size_t yi = size_t(head) * a.Dv + row[r];
            if (a.y_f32)
                static_cast<float*>(a.y)[yi] = yv;
            else
                static_cast<uint16_t*>(a.y)[yi] = f32_to_bf16_rne(yv);
        }
    }
}

// Rows covered by one CTA of a configuration.
template <int DK, int TPR, int RPT, int NT>
constexpr int decode_rows_per_cta() { return (NT / TPR) * RPT; }

}  // namespace gdn
