// window.cuh -- the fused decode-window kernel: conv + SiLU, L2 norm, gates, the delta-rule
// recurrence over ntok tokens and the gated RMSNorm output, with verify / commit / partial commit.
//
// What it computes: regolith baseline-kernels/gdn.metal, header comment and GdnArgs.  Per sequence
// n, value head h (key head hk = h % h_k) and token t:
//     conv: s = h0 w0 + h1 w1 + h2 w2 + x_t w3 (history oldest first); a = SiLU(s); history shifts
//     q^ = q / sqrt(|q|^2 + eps);  k^ = k / sqrt(|k|^2 + eps)
//     gate = exp(softplus(alpha + dt) ssm_a);  beta = sigmoid(beta_raw)
//     kv_j = sum_i S_ij k^_i;  delta_j = (v_j - gate kv_j) beta;  S_ij = gate S_ij + k^_i delta_j
//     o_j = (sum_i S_ij q^_i) / sqrt(128);  y_j = o_j rsqrt(mean_j o^2 + eps) gamma_j sigmoid(z_j)
// The state and the conv history are written after token commit_at (commit 1: the last token;
// 0x100|k: token k; 0: never).
//
// GB300 mapping.  A CTA of 128 threads owns one (n, h) head's 128 x 64 half of the state (columns
// 64*half ..): thread (c, rg) holds column group c (4 columns) of the 16 consecutive rows
// 16rg .. 16rg+15 in registers for the whole window, so the 64 KB head state is read from HBM once
// and written at most once; a warp's load covers two 256-byte row pieces.  The kernel is bound by
// instruction issue, not by memory, so the per-element work is cut to three packed f32x2 FMAs per
// two elements and token: the state is held as c * R with a per-head scalar c (the gate multiplies
// c, and R += k (rk delta / c) is the rank-1 update; c is folded back into R when it drops below
// 2^-40), and the L2 norms of q and k are applied to the reduced sums instead of every row.  The
// reductions over the rows (kv, o) run serially in registers, then over the two row groups of a
// warp with one shuffle, then over the four warps through shared memory.  The two halves of a head
// form a thread-block cluster of 2: the output RMSNorm needs sum_j o_j^2 over all 128 columns, so
// each half keeps its o_t and partial sums for every token in shared memory and the pair exchanges
// the partial sums once, through distributed shared memory, after the last token.  Each CTA
// convolves the 256 q/k channels of key head hk and its own 64 v channels (thread t: q channel t,
// k channel t, v channel t < 64), with histories and taps in registers, and prefetches the next
// token's inputs a token ahead.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernel_args.h"

namespace gdn {

__device__ __forceinline__ float silu_f32(float s) { return __fdividef(s, 1.0f + __expf(-s)); }
__device__ __forceinline__ float sigmoid_f32(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplus_f32(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

// The state of a head half is kept as c * R (c a per-head scalar, R in registers): the gate then
// scales c, not every element, and the rank-1 update becomes R += k (rk delta / c).  When c drops
// below kWinRenorm it is folded back into R.
constexpr float kWinRenorm = 9.094947e-13f;  // 2^-40

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kWinThreads, 4)
    gdn_window_kernel(const WindowArgs a) {
    namespace cg = cooperative_groups;
    constexpr int D = kWinD, CG = kWinHalf / 4, RG = kWinThreads / CG, NR = D / RG;
    static_assert(CG == 16 && RG == 8 && NR == 16, "window tile");

    // per-token buffers are double-buffered by token parity, so that a token needs two barriers:
    // one after the conv outputs are written, one after the kv partial sums are written
    __shared__ __align__(16) float qraw[2][D];
    __shared__ __align__(16) float kraw[2][D];
    __shared__ __align__(16) float vraw[2][kWinHalf];
    __shared__ float part_q[2][4], part_k[2][4], gb[2][2];
    __shared__ float4 red_kv[4][CG], red_o[2][4][CG];
    __shared__ float osm[kWinMaxTok][kWinHalf];
    __shared__ float ss[kWinMaxTok];

    cg::cluster_group cluster = cg::this_cluster();
    const int half = int(cluster.block_rank());
    const int unit = blockIdx.x >> 1;  // n * h_v + h
    const int h = unit % a.h_v;
    const int n = unit / a.h_v;
    const int hk = h % a.h_k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid % CG, rg = tid / CG;
    const int C = (2 * a.h_k + a.h_v) * D;
    const int ntok = a.ntok;

    // ---- the state half in registers: rows rg*16 .. rg*16+15, columns half*64 + 4c .. +3
    const size_t row_stride = size_t(a.h_v) * D;  // floats between consecutive rows i
    float* sbase = a.state + size_t(n) * D * row_stride + size_t(h) * D + half * kWinHalf + 4 * c;
    float2 R[NR][2];
#pragma unroll
    for (int m = 0; m < NR; ++m) {
        const float4 x = ld_stream(reinterpret_cast<const float4*>(sbase + size_t(rg * NR + m) * row_stride));
        R[m][0] = make_float2(x.x, x.y);
        R[m][1] = make_float2(x.z, x.w);
    }
    float cs = 1.0f;  // S = cs * R
    float rq_last = 0.f, cs_last = 0.f;  // the previous token's q norm and state scale

    // ---- this thread's conv channels: q and k of key head hk, and (tid < 64) one v channel
    const int ch_q = hk * D + tid;
    const int ch_k = (a.h_k + hk) * D + tid;
    const bool has_v = tid < kWinHalf;
    const int ch_v = (2 * a.h_k + h) * D + half * kWinHalf + (tid & (kWinHalf - 1));
    const float* hist_n = a.hist + size_t(n) * C * 3;
    float hq[3], hk3[3], hv[3];
#pragma unroll
    for (int e = 0; e < 3; ++e) {
        hq[e] = hist_n[size_t(ch_q) * 3 + e];
        hk3[e] = hist_n[size_t(ch_k) * 3 + e];
        hv[e] = has_v ? hist_n[size_t(ch_v) * 3 + e] : 0.f;
    }
    const float4 wq = *reinterpret_cast<const float4*>(a.conv_w + size_t(ch_q) * 4);
    const float4 wk = *reinterpret_cast<const float4*>(a.conv_w + size_t(ch_k) * 4);
    const float4 wv = has_v ? *reinterpret_cast<const float4*>(a.conv_w + size_t(ch_v) * 4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    // q/k history is owned by the head h == hk (half 0 writes q, half 1 writes k); v by every head
    const bool own_qk = h < a.h_k;
    const float dth = a.dt[h], ssm = a.ssm_a[h];

    const float* x_n = a.qkv + size_t(n) * ntok * C;
    float xq = x_n[ch_q], xk = x_n[ch_k], xv = has_v ? x_n[ch_v] : 0.f;

    // warp 0 finishes token u's readout (after the barrier that follows its partial sums): lanes
    // 0..15 sum the four warps' partials of 4 columns each, the warp sums o^2 for the RMSNorm
    auto finish_readout = [&](int u, float rq_u, float cs_u) {
        if (warp != 0) return;
        const int bu = u & 1;
        float e = 0.f;
        if (lane < CG) {
            const float4 r0 = red_o[bu][0][lane], r1 = red_o[bu][1][lane], r2 = red_o[bu][2][lane],
                         r3 = red_o[bu][3][lane];
            const float sc = cs_u * rq_u * 0.08838834764831845f;  // cs rq / sqrt(128)
            const float4 ot = make_float4(((r0.x + r1.x) + (r2.x + r3.x)) * sc,
                                          ((r0.y + r1.y) + (r2.y + r3.y)) * sc,
                                          ((r0.z + r1.z) + (r2.z + r3.z)) * sc,
                                          ((r0.w + r1.w) + (r2.w + r3.w)) * sc);
            reinterpret_cast<float4*>(osm[u])[lane] = ot;
            e = ot.x * ot.x + ot.y * ot.y + ot.z * ot.z + ot.w * ot.w;
        }
        e = group_sum<32>(e);
        if (lane == 0) ss[u] = e;
    };

    for (int t = 0; t < ntok; ++t) {
        // next token's conv inputs, ahead of this token's barriers
        float nq = 0.f, nk = 0.f, nv = 0.f;
        if (t + 1 < ntok) {
            const float* xn = x_n + size_t(t + 1) * C;
            nq = xn[ch_q];
            nk = xn[ch_k];
            nv = has_v ? xn[ch_v] : 0.f;
        }
        // conv + SiLU, history shift
        const float cq = silu_f32(fmaf(xq, wq.w, fmaf(hq[2], wq.z, fmaf(hq[1], wq.y, hq[0] * wq.x))));
        const float ck = silu_f32(fmaf(xk, wk.w, fmaf(hk3[2], wk.z, fmaf(hk3[1], wk.y, hk3[0] * wk.x))));
        const float cv = silu_f32(fmaf(xv, wv.w, fmaf(hv[2], wv.z, fmaf(hv[1], wv.y, hv[0] * wv.x))));
        hq[0] = hq[1]; hq[1] = hq[2]; hq[2] = xq;
        hk3[0] = hk3[1]; hk3[1] = hk3[2]; hk3[2] = xk;
        hv[0] = hv[1]; hv[1] = hv[2]; hv[2] = xv;
        if (t + 1 == a.commit_at) {
            float* ho = a.hist_out + size_t(n) * C * 3;
            if (own_qk) {
                const int ch = half == 0 ? ch_q : ch_k;
                const float* hh = half == 0 ? hq : hk3;
                ho[size_t(ch) * 3 + 0] = hh[0];
                ho[size_t(ch) * 3 + 1] = hh[1];
                ho[size_t(ch) * 3 + 2] = hh[2];
            }
            if (has_v) {
                ho[size_t(ch_v) * 3 + 0] = hv[0];
                ho[size_t(ch_v) * 3 + 1] = hv[1];
                ho[size_t(ch_v) * 3 + 2] = hv[2];
            }
        }
        xq = nq; xk = nk; xv = nv;

        // raw q, k, v to shared memory; sums of squares per warp; gate and beta on thread 0
        const int b = t & 1;
        qraw[b][tid] = cq;
        kraw[b][tid] = ck;
        if (has_v) vraw[b][tid] = cv;
        const float sq = group_sum<32>(cq * cq);
        const float sk = group_sum<32>(ck * ck);
        if (lane == 0) {
            part_q[b][warp] = sq;
            part_k[b][warp] = sk;
        }
        if (tid == 0) {
            const size_t gi = (size_t(n) * ntok + t) * a.h_v + h;
            gb[b][0] = expf(softplus_f32(a.alpha[gi] + dth) * ssm);
            gb[b][1] = sigmoid_f32(a.beta[gi]);
        }
        __syncthreads();
        if (t > 0) finish_readout(t - 1, rq_last, cs_last);

        const float rk = rsqrtf(((part_k[b][0] + part_k[b][1]) + (part_k[b][2] + part_k[b][3])) + a.eps);
        const float rq = rsqrtf(((part_q[b][0] + part_q[b][1]) + (part_q[b][2] + part_q[b][3])) + a.eps);
        const float gate = gb[b][0], beta = gb[b][1];
        const float4* k4 = reinterpret_cast<const float4*>(kraw[b] + rg * NR);
        const float4* q4 = reinterpret_cast<const float4*>(qraw[b] + rg * NR);

        // kv = cs rk sum_i R_ij k_i: this thread's 16 rows, the warp's two row groups, four warps
        float2 kva = make_float2(0.f, 0.f), kvb = make_float2(0.f, 0.f);
#pragma unroll
        for (int m4 = 0; m4 < NR / 4; ++m4) {
            const float4 kk = k4[m4];
            const float kr[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 k2 = make_float2(kr[u], kr[u]);
                kva = __ffma2_rn(R[m4 * 4 + u][0], k2, kva);
                kvb = __ffma2_rn(R[m4 * 4 + u][1], k2, kvb);
            }
        }
        float4 kv = make_float4(kva.x, kva.y, kvb.x, kvb.y);
        kv.x += __shfl_xor_sync(kFullMask, kv.x, 16);
        kv.y += __shfl_xor_sync(kFullMask, kv.y, 16);
        kv.z += __shfl_xor_sync(kFullMask, kv.z, 16);
        kv.w += __shfl_xor_sync(kFullMask, kv.w, 16);
        if (lane < 16) red_kv[warp][c] = kv;
        __syncthreads();
        {
            const float4 r0 = red_kv[0][c], r1 = red_kv[1][c], r2 = red_kv[2][c], r3 = red_kv[3][c];
            kv.x = (r0.x + r1.x) + (r2.x + r3.x);
            kv.y = (r0.y + r1.y) + (r2.y + r3.y);
            kv.z = (r0.z + r1.z) + (r2.z + r3.z);
            kv.w = (r0.w + r1.w) + (r2.w + r3.w);
        }
        const float4 vv = reinterpret_cast<const float4*>(vraw[b])[c];
        const float gk = gate * cs * rk;  // gate * kv_j = gk * (reduced sum)
        // delta_j = (v_j - gate kv_j) beta;  the update R += k (rk delta / cs'), cs' = gate cs
        float cn = gate * cs;
        if (cn < kWinRenorm) {  // uniform over the CTA: fold cs' into R
#pragma unroll
            for (int m = 0; m < NR; ++m) {
                const float2 c2 = make_float2(cn, cn);
                R[m][0] = __fmul2_rn(R[m][0], c2);
                R[m][1] = __fmul2_rn(R[m][1], c2);
            }
            cn = 1.0f;
        }
        const float ek = beta * rk / cn;
        const float2 ea = make_float2((vv.x - gk * kv.x) * ek, (vv.y - gk * kv.y) * ek);
        const float2 eb = make_float2((vv.z - gk * kv.z) * ek, (vv.w - gk * kv.w) * ek);
        cs = cn;
        rq_last = rq;
        cs_last = cs;

        // rank-1 update and the readout partial sum_i R_ij q_i
        float2 oa = make_float2(0.f, 0.f), ob = make_float2(0.f, 0.f);
#pragma unroll
        for (int m4 = 0; m4 < NR / 4; ++m4) {
            const float4 kk = k4[m4];
            const float4 qq = q4[m4];
            const float kr[4] = {kk.x, kk.y, kk.z, kk.w};
            const float qr[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int m = m4 * 4 + u;
                const float2 k2 = make_float2(kr[u], kr[u]);
                const float2 q2 = make_float2(qr[u], qr[u]);
                R[m][0] = __ffma2_rn(k2, ea, R[m][0]);
                R[m][1] = __ffma2_rn(k2, eb, R[m][1]);
                oa = __ffma2_rn(R[m][0], q2, oa);
                ob = __ffma2_rn(R[m][1], q2, ob);
            }
        }
        if (t + 1 == a.commit_at) {
#pragma unroll
            for (int m = 0; m < NR; ++m)
                st_stream(reinterpret_cast<float4*>(sbase + size_t(rg * NR + m) * row_stride),
                          make_float4(cs * R[m][0].x, cs * R[m][0].y, cs * R[m][1].x, cs * R[m][1].y));
        }
        float4 o = make_float4(oa.x, oa.y, ob.x, ob.y);
        o.x += __shfl_xor_sync(kFullMask, o.x, 16);
        o.y += __shfl_xor_sync(kFullMask, o.y, 16);
        o.z += __shfl_xor_sync(kFullMask, o.z, 16);
        o.w += __shfl_xor_sync(kFullMask, o.w, 16);
        if (lane < 16) red_o[b][warp][c] = o;
    }
    __syncthreads();
    finish_readout(ntok - 1, rq_last, cs_last);

    // the gated RMSNorm needs both halves' sums of o^2: exchange them once through the cluster
    cluster.sync();
    const float* peer_ss = cluster.map_shared_rank(ss, half ^ 1);
    for (int idx = tid; idx < ntok * kWinHalf; idx += kWinThreads) {
        const int t = idx / kWinHalf, j = idx % kWinHalf;
        const float tot = ss[t] + peer_ss[t];
        const float rs = rsqrtf(tot / float(D) + a.eps);
        const size_t yi = ((size_t(n) * ntok + t) * a.h_v + h) * D + half * kWinHalf + j;
        const int jj = half * kWinHalf + j;
        a.y[yi] = osm[t][j] * rs * a.gamma[jj] * sigmoid_f32(a.z[yi]);
    }
    cluster.sync();  // the peer has read this CTA's sums before it exits
}

}  // namespace gdn
