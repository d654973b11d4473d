// decode.cuh -- the GDN decode-step kernel (one token, fp32 state streamed once).
//
// What it computes: metaltile-std gated_delta.rs, module doc "Recurrence per step", for every
// (b, hv) head and state row r (Dv rows of Dk columns, Dk contiguous):
//     S'[r,:] = g S[r,:];  kv_r = S'[r,:] . k;  delta_r = (v_r - kv_r) beta;
//     S_new[r,:] = S'[r,:] + delta_r k;  y_r = scale * S_new[r,:] . q
// with key head hk = hv / (Hv / Hk) (the page's DISPATCH INVARIANTS).  In the pooled form the state
// of batch row b is slot slots[b] of a [pool, Hv, Dv, Dk] pool, updated in place.
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

    long long srow = b;  // the state row (pool slot) of batch row b
    if (a.slots) {
        srow = a.slots[b];
        if (srow < 0 || srow >= a.pool_size) {
            if (threadIdx.x == 0 && tile == 0 && hv == 0) atomicOr(a.status, 1);
            return;
        }
    }
    const size_t head_off = (size_t(srow) * a.Hv + hv) * a.Dv * DK;
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

// T consecutive decode steps ([gated_delta.rs] mt_gated_delta_chunk).  The single step's row split;
// the state rows stay in registers for all T tokens, held as c * R with one scalar c per head: the
// gate multiplies c instead of every element, the rank-1 update is R += k (delta / c), and c is
// folded back into R when |c| leaves [2^-40, 2^40] (uniform over the CTA: every thread sees the
// same gates).  Per token one pass over a thread's rows forms R k and R q (and the lane's share of
// k q), one reduction round inside the row group sums all of them, and
//     kv = c (R k),  delta = (v - kv) beta,  y = scale (c (R q) + delta (k q))
// -- the readout of the updated state, S_new q = g S q + delta (k q), regrouped -- before a second
// pass applies the update.  Arithmetic on column pairs with packed f32x2 FMAs.  Tokens are staged
// in blocks of TB: q and k of the key head (fp32), v of this CTA's rows, g and beta go to shared
// memory, then the block's tokens run with warp shuffles only, so a block costs two barriers.
constexpr float kMultiLo = 9.094947e-13f;  // 2^-40
constexpr float kMultiHi = 1.0995116e12f;  // 2^40
template <int DK, int TPR, int RPT, int NT, int TB>
__global__ void __launch_bounds__(NT) gdn_decode_multi_kernel(const DecodeMultiArgs a) {
    constexpr int NV = DK / (4 * TPR);
    constexpr int RPP = NT / TPR;
    constexpr int ROWS = RPP * RPT;
    __shared__ float4 ks[TB][DK / 4];
    __shared__ float4 qs[TB][DK / 4];
    __shared__ float vs[TB][ROWS];
    __shared__ float gs[TB], bs[TB];

    const int head = blockIdx.x / a.tiles;
    const int tile = blockIdx.x - head * a.tiles;
    const int hv = head % a.Hv;
    const int b = head / a.Hv;
    const int hk = hv / (a.Hv / a.Hk);
    const int lr = threadIdx.x % TPR;
    const int rw = threadIdx.x / TPR;
    const size_t head_off = size_t(head) * a.Dv * DK;
    const float4* src = reinterpret_cast<const float4*>(a.state_in + head_off);
    float4* dst = reinterpret_cast<float4*>(a.state_out + head_off);

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

    float c = 1.f;  // the state is c * s
    for (int t0 = 0; t0 < a.T; t0 += TB) {
        const int nb = a.T - t0 < TB ? a.T - t0 : TB;
        __syncthreads();  // the previous block's shared inputs are no longer read
        for (int i = threadIdx.x; i < nb * (DK / 4); i += NT) {
            const int tt = i / (DK / 4), cc = i - tt * (DK / 4);
            const size_t off = ((size_t(b) * a.T + t0 + tt) * a.Hk + hk) * DK + 4 * cc;
            ks[tt][cc] = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.k + off));
            qs[tt][cc] = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.q + off));
        }
        for (int i = threadIdx.x; i < nb * ROWS; i += NT) {
            const int tt = i / ROWS, r = i - tt * ROWS;
            const int rr = tile * ROWS + r;
            vs[tt][r] = rr < a.Dv ? bf16_to_f32(a.v[((size_t(b) * a.T + t0 + tt) * a.Hv + hv) * a.Dv + rr]) : 0.f;
        }
        if (threadIdx.x < nb) {
            const size_t gi = (size_t(b) * a.T + t0 + threadIdx.x) * a.Hv + hv;
            gs[threadIdx.x] = a.g[gi];
            bs[threadIdx.x] = bf16_to_f32(a.beta[gi]);
        }
        __syncthreads();
        for (int tt = 0; tt < nb; ++tt) {
            const float beta = bs[tt];
            c *= gs[tt];
            if (!(fabsf(c) >= kMultiLo && fabsf(c) <= kMultiHi)) {  // fold c into the rows
                const float2 c2 = make_float2(c, c);
#pragma unroll
                for (int r = 0; r < RPT; ++r)
#pragma unroll
                    for (int m = 0; m < NV; ++m) {
                        float4& x = s[r][m];
                        const float2 x01 = __fmul2_rn(make_float2(x.x, x.y), c2);
                        const float2 x23 = __fmul2_rn(make_float2(x.z, x.w), c2);
                        x = make_float4(x01.x, x01.y, x23.x, x23.y);
                    }
                c = 1.f;
            }
            // pass 1: R k, R q per row and this lane's share of k q
            float2 kq2 = make_float2(0.f, 0.f);
            float2 rk2[RPT], rq2[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) rk2[r] = rq2[r] = make_float2(0.f, 0.f);
#pragma unroll
            for (int m = 0; m < NV; ++m) {
                const float4 kk = ks[tt][lr + TPR * m];
                const float4 qq = qs[tt][lr + TPR * m];
                const float2 k01 = make_float2(kk.x, kk.y), k23 = make_float2(kk.z, kk.w);
                const float2 q01 = make_float2(qq.x, qq.y), q23 = make_float2(qq.z, qq.w);
                kq2 = __ffma2_rn(k01, q01, kq2);
                kq2 = __ffma2_rn(k23, q23, kq2);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const float2 x01 = make_float2(s[r][m].x, s[r][m].y), x23 = make_float2(s[r][m].z, s[r][m].w);
                    rk2[r] = __ffma2_rn(x01, k01, rk2[r]);
                    rk2[r] = __ffma2_rn(x23, k23, rk2[r]);
                    rq2[r] = __ffma2_rn(x01, q01, rq2[r]);
                    rq2[r] = __ffma2_rn(x23, q23, rq2[r]);
                }
            }
            float kq = kq2.x + kq2.y, rk[RPT], rq[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                rk[r] = rk2[r].x + rk2[r].y;
                rq[r] = rq2[r].x + rq2[r].y;
            }
#pragma unroll
            for (int o = TPR / 2; o > 0; o >>= 1) {
                kq += __shfl_xor_sync(kFullMask, kq, o);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    rk[r] += __shfl_xor_sync(kFullMask, rk[r], o);
                    rq[r] += __shfl_xor_sync(kFullMask, rq[r], o);
                }
            }
            // pass 2: delta, the readout, the rank-1 update (one reciprocal of c per token)
            const float ic = 1.f / c;
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const float delta = (vs[tt][r * RPP + rw] - c * rk[r]) * beta;
                const float yv = a.scale * fmaf(delta, kq, c * rq[r]);
                const float dc = delta * ic;
                const float2 d2 = make_float2(dc, dc);
#pragma unroll
                for (int m = 0; m < NV; ++m) {
                    const float4 kk = ks[tt][lr + TPR * m];
                    float4& x = s[r][m];
                    const float2 x01 = __ffma2_rn(make_float2(kk.x, kk.y), d2, make_float2(x.x, x.y));
                    const float2 x23 = __ffma2_rn(make_float2(kk.z, kk.w), d2, make_float2(x.z, x.w));
                    x = make_float4(x01.x, x01.y, x23.x, x23.y);
                }
                if (row[r] < a.Dv && lr == 0) {
                    const size_t yi = ((size_t(b) * a.T + t0 + tt) * a.Hv + hv) * a.Dv + row[r];
                    if (a.y_f32)
                        static_cast<float*>(a.y)[yi] = yv;
                    else
                        static_cast<uint16_t*>(a.y)[yi] = f32_to_bf16_rne(yv);
                }
            }
        }
    }
    const float2 c2 = make_float2(c, c);
#pragma unroll
    for (int r = 0; r < RPT; ++r)
        if (row[r] < a.Dv)
#pragma unroll
            for (int m = 0; m < NV; ++m) {
                const float4 x = s[r][m];
                const float2 x01 = __fmul2_rn(make_float2(x.x, x.y), c2);
                const float2 x23 = __fmul2_rn(make_float2(x.z, x.w), c2);
                st_stream(dst + size_t(row[r]) * (DK / 4) + lr + TPR * m, make_float4(x01.x, x01.y, x23.x, x23.y));
            }
}

// Rows covered by one CTA of a configuration.
template <int DK, int TPR, int RPT, int NT>
constexpr int decode_rows_per_cta() { return (NT / TPR) * RPT; }

}  // namespace gdn
