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
// GB300 mapping.  A CTA of 128 threads owns one (n, h) head: lane (column group cg, row block rb)
// of warp w holds the 4 columns 32w + 4cg .. of the 32 rows 32rb .. 32rb+31 in registers for the
// whole window, so the 64 KB head state is read from HBM once and written at most once.  Both
// reductions over the 128 rows (kv and o) are a register sum plus two xor-shuffles inside the warp,
// so a token needs one barrier (after the conv outputs are written; the per-token buffers are
// double-buffered by token parity).  The kernel is bound by instruction issue and latency, not
// memory, so the per-element work is three packed f32x2 FMAs per two elements and token, and the
// per-token scalar work (conv, norms, gates) is shared by 128 state elements per thread: the state
// is held as c * R with a per-head scalar c (the gate multiplies c; R += k (rk delta / c) is the
// rank-1 update; c is folded back into R when it drops below 2^-40), and the q/k norms are applied
// to reduced sums.  Each thread convolves q and k channel t of key head hk and v channel t of its
// value head, with histories and taps in registers, a token ahead of their use; the gated RMSNorm
// reads the head's outputs of every token from shared memory after the last token.
#pragma once

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

// Asynchronous 4-byte global -> shared copy (completes at cp_async_wait_all of the same thread).
__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__global__ void __launch_bounds__(kWinThreads, 2) gdn_window_kernel(const WindowArgs a) {
    constexpr int D = kWinD, NR = 32;  // rows per lane
    static_assert(kWinThreads == 128 && D == 128, "window tile");

    // per-token buffers, double-buffered by token parity: one barrier per token.  q and k of a
    // token by row block of 32, padded to a stride of 36 floats so that the four row blocks a warp
    // reads at once fall in different banks
    constexpr int RBS = 36;
    __shared__ __align__(16) float qraw[2][4 * RBS];
    __shared__ __align__(16) float kraw[2][4 * RBS];
    __shared__ __align__(16) float vraw[2][D];
    __shared__ float gates[kWinMaxTok][2];  // gate and beta of every token, computed up front
    __shared__ __align__(16) float osm[kWinMaxTok][D];
    __shared__ float ssw[kWinMaxTok][4];  // per-warp sums of o^2
    __shared__ float ss[kWinMaxTok];
    __shared__ float zs[kWinMaxTok * D];  // the epilogue's z and gamma, fetched up front
    __shared__ float gs[D];

    const int unit = blockIdx.x;  // n * h_v + h
    const int h = unit % a.h_v;
    const int n = unit / a.h_v;
    const int hk = h % a.h_k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = lane & 7;              // column group inside the warp
    const int rb = lane >> 3;             // block of 32 rows
    const int col = 32 * warp + 4 * cg;   // first of this lane's 4 columns
    const int C = (2 * a.h_k + a.h_v) * D;
    const int ntok = a.ntok;

    // ---- the state: rows 32rb .. 32rb+31, columns col .. col+3, held as cs * R
    const size_t row_stride = size_t(a.h_v) * D;
    float* sbase = a.state + size_t(n) * D * row_stride + size_t(h) * D + col;
    // packed along rows: R[p][j] = (S[2p][j], S[2p+1][j]) of this lane's rows and 4 columns, so that
    // the per-row k and q pairs come straight from float4 loads
    float2 R[NR / 2][4];
#pragma unroll
    for (int p = 0; p < NR / 2; ++p) {
        const float4 x = ld_stream(reinterpret_cast<const float4*>(sbase + size_t(rb * NR + 2 * p) * row_stride));
        const float4 y = ld_stream(reinterpret_cast<const float4*>(sbase + size_t(rb * NR + 2 * p + 1) * row_stride));
        R[p][0] = make_float2(x.x, y.x);
        R[p][1] = make_float2(x.y, y.y);
        R[p][2] = make_float2(x.z, y.z);
        R[p][3] = make_float2(x.w, y.w);
    }
    float cs = 1.0f;

    // ---- this thread's conv channels: q, k of key head hk and v of value head h, channel tid
    const int ch_q = hk * D + tid;
    const int ch_k = (a.h_k + hk) * D + tid;
    const int ch_v = (2 * a.h_k + h) * D + tid;
    const float* hist_n = a.hist + size_t(n) * C * 3;
    float hq[3], hk3[3], hv[3];
#pragma unroll
    for (int e = 0; e < 3; ++e) {
        hq[e] = hist_n[size_t(ch_q) * 3 + e];
        hk3[e] = hist_n[size_t(ch_k) * 3 + e];
        hv[e] = hist_n[size_t(ch_v) * 3 + e];
    }
    const float4 wq = *reinterpret_cast<const float4*>(a.conv_w + size_t(ch_q) * 4);
    const float4 wk = *reinterpret_cast<const float4*>(a.conv_w + size_t(ch_k) * 4);
    const float4 wv = *reinterpret_cast<const float4*>(a.conv_w + size_t(ch_v) * 4);
    const bool own_qk = h < a.h_k;  // the q/k history of key head hk is written by head h == hk
    const float dth = a.dt[h], ssm = a.ssm_a[h];
    const float* x_n = a.qkv + size_t(n) * ntok * C;
    float xq = x_n[ch_q], xk = x_n[ch_k], xv = x_n[ch_v];
    // every token's gate and beta (thread t), read after the first token's barrier
    if (tid < ntok) {
        const size_t gi = (size_t(n) * ntok + tid) * a.h_v + h;
        gates[tid][0] = expf(softplus_f32(a.alpha[gi] + dth) * ssm);
        gates[tid][1] = sigmoid_f32(a.beta[gi]);
    }
    // the epilogue's z (token i, column tid) and gamma, copied asynchronously now
#pragma unroll
    for (int i = 0; i < kWinMaxTok; ++i)
        if (i < ntok) cp_async4(&zs[i * D + tid], a.z + ((size_t(n) * ntok + i) * a.h_v + h) * D + tid);
    cp_async4(&gs[tid], a.gamma + tid);

    for (int t = 0; t < ntok; ++t) {
        const int b = t & 1;
        float nq = 0.f, nk = 0.f, nv = 0.f;
        if (t + 1 < ntok) {
            const float* xn = x_n + size_t(t + 1) * C;
            nq = xn[ch_q];
            nk = xn[ch_k];
            nv = xn[ch_v];
        }
        // conv + SiLU, history shift, committed history
        const float cq = silu_f32(fmaf(xq, wq.w, fmaf(hq[2], wq.z, fmaf(hq[1], wq.y, hq[0] * wq.x))));
        const float ck = silu_f32(fmaf(xk, wk.w, fmaf(hk3[2], wk.z, fmaf(hk3[1], wk.y, hk3[0] * wk.x))));
        const float cv = silu_f32(fmaf(xv, wv.w, fmaf(hv[2], wv.z, fmaf(hv[1], wv.y, hv[0] * wv.x))));
        hq[0] = hq[1]; hq[1] = hq[2]; hq[2] = xq;
        hk3[0] = hk3[1]; hk3[1] = hk3[2]; hk3[2] = xk;
        hv[0] = hv[1]; hv[1] = hv[2]; hv[2] = xv;
        if (t + 1 == a.commit_at) {
            float* ho = a.hist_out + size_t(n) * C * 3;
            if (own_qk) {
#pragma unroll
                for (int e = 0; e < 3; ++e) {
                    ho[size_t(ch_q) * 3 + e] = hq[e];
                    ho[size_t(ch_k) * 3 + e] = hk3[e];
                }
            }
#pragma unroll
            for (int e = 0; e < 3; ++e) ho[size_t(ch_v) * 3 + e] = hv[e];
        }
        xq = nq; xk = nk; xv = nv;
        qraw[b][(tid >> 5) * RBS + (tid & 31)] = cq;
        kraw[b][(tid >> 5) * RBS + (tid & 31)] = ck;
        vraw[b][tid] = cv;
        __syncthreads();

        // everything below is warp-local: the warp owns 32 whole columns
        const float gate = gates[t][0], beta = gates[t][1];
        const float4* k4 = reinterpret_cast<const float4*>(kraw[b] + rb * RBS);
        const float4* q4 = reinterpret_cast<const float4*>(qraw[b] + rb * RBS);

        // kv = cs rk sum_i R_ij k_i: 32 rows in registers (as 16 row pairs), then the 4 row blocks
        // by two shuffles; |k|^2 and |q|^2 (the L2 norms) ride along: each lane sums its row
        // block's 32 squares and the same two shuffles add the 4 blocks
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        float2 nk2 = make_float2(0.f, 0.f), nq2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int m4 = 0; m4 < NR / 4; ++m4) {
            const float4 kk = k4[m4];
            const float4 qq = q4[m4];
            const float2 k01 = make_float2(kk.x, kk.y), k23 = make_float2(kk.z, kk.w);
            const float2 q01 = make_float2(qq.x, qq.y), q23 = make_float2(qq.z, qq.w);
            nk2 = __ffma2_rn(k01, k01, __ffma2_rn(k23, k23, nk2));
            nq2 = __ffma2_rn(q01, q01, __ffma2_rn(q23, q23, nq2));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[j] = __ffma2_rn(R[2 * m4][j], k01, acc[j]);
                acc[j] = __ffma2_rn(R[2 * m4 + 1][j], k23, acc[j]);
            }
        }
        float kvs[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) kvs[j] = acc[j].x + acc[j].y;
        float ksq = nk2.x + nk2.y, qsq = nq2.x + nq2.y;
#pragma unroll
        for (int o = 8; o < 32; o <<= 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) kvs[j] += __shfl_xor_sync(kFullMask, kvs[j], o);
            ksq += __shfl_xor_sync(kFullMask, ksq, o);
            qsq += __shfl_xor_sync(kFullMask, qsq, o);
        }
        const float rk = rsqrtf(ksq + a.eps);
        const float rq = rsqrtf(qsq + a.eps);
        const float4 vv = *reinterpret_cast<const float4*>(vraw[b] + col);
        const float gk = gate * cs * rk;
        float cn = gate * cs;
        if (cn < kWinRenorm) {  // uniform over the CTA: fold cs' into R
#pragma unroll
            for (int p = 0; p < NR / 2; ++p)
#pragma unroll
                for (int j = 0; j < 4; ++j) R[p][j] = __fmul2_rn(R[p][j], make_float2(cn, cn));
            cn = 1.0f;
        }
        const float ek = beta * rk * __frcp_rn(cn);
        const float vj[4] = {vv.x, vv.y, vv.z, vv.w};
        float2 e2[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float e = (vj[j] - gk * kvs[j]) * ek;
            e2[j] = make_float2(e, e);
        }
        cs = cn;

        // rank-1 update and readout
        float2 oacc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int m4 = 0; m4 < NR / 4; ++m4) {
            const float4 kk = k4[m4];
            const float4 qq = q4[m4];
            const float2 k01 = make_float2(kk.x, kk.y), k23 = make_float2(kk.z, kk.w);
            const float2 q01 = make_float2(qq.x, qq.y), q23 = make_float2(qq.z, qq.w);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                R[2 * m4][j] = __ffma2_rn(k01, e2[j], R[2 * m4][j]);
                R[2 * m4 + 1][j] = __ffma2_rn(k23, e2[j], R[2 * m4 + 1][j]);
                oacc[j] = __ffma2_rn(R[2 * m4][j], q01, oacc[j]);
                oacc[j] = __ffma2_rn(R[2 * m4 + 1][j], q23, oacc[j]);
            }
        }
        if (t + 1 == a.commit_at) {
#pragma unroll
            for (int p = 0; p < NR / 2; ++p) {
                st_stream(reinterpret_cast<float4*>(sbase + size_t(rb * NR + 2 * p) * row_stride),
                          make_float4(cs * R[p][0].x, cs * R[p][1].x, cs * R[p][2].x, cs * R[p][3].x));
                st_stream(reinterpret_cast<float4*>(sbase + size_t(rb * NR + 2 * p + 1) * row_stride),
                          make_float4(cs * R[p][0].y, cs * R[p][1].y, cs * R[p][2].y, cs * R[p][3].y));
            }
        }
        float os[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) os[j] = oacc[j].x + oacc[j].y;
#pragma unroll
        for (int o = 8; o < 32; o <<= 1)
#pragma unroll
            for (int j = 0; j < 4; ++j) os[j] += __shfl_xor_sync(kFullMask, os[j], o);
        const float sc = cs * rq * 0.08838834764831845f;  // cs rq / sqrt(128)
        const float4 ot = make_float4(os[0] * sc, os[1] * sc, os[2] * sc, os[3] * sc);
        // lanes 0 .. 7 (row block 0) hold the warp's 32 outputs
        float e = rb == 0 ? ot.x * ot.x + ot.y * ot.y + ot.z * ot.z + ot.w * ot.w : 0.f;
        if (rb == 0) *reinterpret_cast<float4*>(&osm[t][col]) = ot;
        e += __shfl_xor_sync(kFullMask, e, 1);
        e += __shfl_xor_sync(kFullMask, e, 2);
        e += __shfl_xor_sync(kFullMask, e, 4);
        if (lane == 0) ssw[t][warp] = e;
    }
    cp_async_wait_all();  // this thread's z and gamma (read only by this thread)
    __syncthreads();
    if (tid < ntok) ss[tid] = (ssw[tid][0] + ssw[tid][1]) + (ssw[tid][2] + ssw[tid][3]);
    __syncthreads();
    // the gated RMSNorm over the head's 128 outputs of each token
#pragma unroll
    for (int i = 0; i < kWinMaxTok; ++i) {
        if (i < ntok) {
            const float rs = rsqrtf(ss[i] / float(D) + a.eps);
            const size_t yi = ((size_t(n) * ntok + i) * a.h_v + h) * D + tid;
            a.y[yi] = osm[i][tid] * rs * gs[tid] * sigmoid_f32(zs[i * D + tid]);
        }
    }
}

}  // namespace gdn
