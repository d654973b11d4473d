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
// of warp w holds the 4 columns 32w + 4cg .. of the 32 rows 32rb .. 32rb+31 in registers, so the
// 64 KB head state is read from HBM once and written at most once.  The window's tokens are not
// stepped one by one: their conv outputs, gates and Gram entries do not depend on the state, so the
// window runs as one chunk of the WY form (with k^_t = rk_t k_t, w_s = rk_s u_s, D_ts the product of
// the gates of tokens s+1 .. t and gamma_t that of tokens 0 .. t):
//     u_t = beta_t (v_t - rk_t (gamma_t S0^T k_t + sum_{s<t} D_ts (k_t . k_s) w_s))
//     o_t = rq_t / sqrt(128) (gamma_t S0^T q_t + sum_{s<=t} D_ts (q_t . k_s) w_s)
//     S after m tokens = gamma_{m-1} S0 + sum_{s<m} D_{m-1,s} k_s w_s^T
// -- the single steps regrouped (u_t is token t's delta, w_t = rk_t delta_t).  So the kernel is a
// conv prologue for every token, one pass over the slab forming S0^T k_t and S0^T q_t for all tokens
// (the reductions over the rows are register sums plus two xor-shuffles inside the warp), a
// per-column triangular solve (thread t owns column t, which its own warp holds), and, when the
// window commits, one pass applying the rank-m write: three CTA barriers per window.  The q and k
// L2 norms are scalars folded into the solve (|k_t|^2 and |q_t|^2 come with the Gram entries);
// every decay is the exponential of a sum of log gates over its own segment.  Each thread
// convolves q and k channel t of key head hk and v channel t of its value head for every token;
// the gated RMSNorm of each token's 128 outputs follows the last barrier.
#pragma once

#include "common.cuh"
#include "kernel_args.h"

namespace gdn {

__device__ __forceinline__ float silu_f32(float s) { return __fdividef(s, 1.0f + __expf(-s)); }
__device__ __forceinline__ float sigmoid_f32(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplus_f32(float x) { return x > 20.0f ? x : log1pf(expf(x)); }


// Asynchronous 4-byte global -> shared copy (completes at cp_async_wait_all of the same thread).
__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__global__ void __launch_bounds__(kWinThreads, 2) gdn_window_kernel(const WindowArgs a) {
    constexpr int D = kWinD, NR = 32, TK = kWinMaxTok;  // rows per lane, tokens per window at most
    static_assert(kWinThreads == 128 && D == 128 && TK == 8, "window tile");
    // conv outputs of q and k by token, channels by row block of 32 padded to a stride of 36 floats
    // so that the four row blocks a warp reads at once fall in different banks
    // (and by token at a stride of 148 floats, so that the Gram's eight keys fall in different banks)
    constexpr int RBS = 36, TSTR = 4 * RBS + 4;
    __shared__ __align__(16) float qc[TK][TSTR];
    __shared__ __align__(16) float kc[TK][TSTR];
    __shared__ __align__(16) float kvp[TK][D];  // S0^T k_t (raw k)
    __shared__ __align__(16) float qrp[TK][D];  // S0^T q_t (raw q)
    __shared__ __align__(16) float wsm[TK][D];  // w_t = rk_t delta_t
    __shared__ float kkd[TK][TK], qkd[TK][TK];  // D_ts (k_t . k_s), s < t; D_ts (q_t . k_s), s <= t
    __shared__ float kk2[TK], qq2[TK];          // |k_t|^2, |q_t|^2
    __shared__ float lg[TK], bet[TK], gam[TK], gtl[TK];  // log gate, beta, gamma_t, D_{m-1,t}
    __shared__ float ssw[TK][4];                // per-warp sums of o^2
    __shared__ float zs[TK * D];                // the epilogue's z and gamma, fetched up front
    __shared__ float gs[D];

    // The CTAs of one wave run in lock step (each streams its head's state, then computes with HBM
    // idle); the second CTA slot of each SM starts a little later in the first wave, and the slots
    // stay offset as later CTAs take their places, so one slot's state stream overlaps the other's
    // arithmetic.  A bounded delay on the clock: nothing is waited for.
    if (a.stagger_cycles > 0 && int(blockIdx.x) >= a.stagger_lo && int(blockIdx.x) < 2 * a.stagger_lo) {
        const long long t0 = clock64();
        while (clock64() - t0 < a.stagger_cycles) __nanosleep(256);
    }
    const int unit = blockIdx.x;  // n * h_v + h
    const int h = unit % a.h_v;
    const int n = unit / a.h_v;
    const int hk = h % a.h_k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = lane & 7;              // column group inside the warp
    const int rb = lane >> 3;             // block of 32 rows
    const int col = 32 * warp + 4 * cg;   // first of this lane's 4 columns
    const int C = (2 * a.h_k + a.h_v) * D;
    const int ntok = a.ntok, m = a.commit_at;

    // ---- the state: rows 32rb .. 32rb+31, columns col .. col+3, packed along rows:
    // R[p][j] = (S[32rb + 2p][col + j], S[32rb + 2p + 1][col + j])
    const size_t row_stride = size_t(a.h_v) * D;
    float* sbase = a.state + size_t(n) * D * row_stride + size_t(h) * D + col;
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

    // ---- conv + SiLU of this thread's channels (q, k of key head hk; v of value head h; channel
    // tid) for every token; the committed history; tokens past ntok read as zero
    const int ch_q = hk * D + tid;
    const int ch_k = (a.h_k + hk) * D + tid;
    const int ch_v = (2 * a.h_k + h) * D + tid;
    const float* hist_n = a.hist + size_t(n) * C * 3;
    const float* x_n = a.qkv + size_t(n) * ntok * C;
    // the sequence h0 h1 h2 x0 .. x_{ntok-1} of each channel
    float sq[TK + 3], sk[TK + 3], sv[TK + 3];
#pragma unroll
    for (int e = 0; e < 3; ++e) {
        sq[e] = hist_n[size_t(ch_q) * 3 + e];
        sk[e] = hist_n[size_t(ch_k) * 3 + e];
        sv[e] = hist_n[size_t(ch_v) * 3 + e];
    }
#pragma unroll
    for (int t = 0; t < TK; ++t) {
        const bool on = t < ntok;
        sq[t + 3] = on ? x_n[size_t(t) * C + ch_q] : 0.f;
        sk[t + 3] = on ? x_n[size_t(t) * C + ch_k] : 0.f;
        sv[t + 3] = on ? x_n[size_t(t) * C + ch_v] : 0.f;
    }
    const float4 wq = *reinterpret_cast<const float4*>(a.conv_w + size_t(ch_q) * 4);
    const float4 wk = *reinterpret_cast<const float4*>(a.conv_w + size_t(ch_k) * 4);
    const float4 wv = *reinterpret_cast<const float4*>(a.conv_w + size_t(ch_v) * 4);
    // the epilogue's z (token i, column tid) and gamma, copied asynchronously now
#pragma unroll
    for (int i = 0; i < TK; ++i)
        if (i < ntok) cp_async4(&zs[i * D + tid], a.z + ((size_t(n) * ntok + i) * a.h_v + h) * D + tid);
    cp_async4(&gs[tid], a.gamma + tid);

    float vt[TK];  // v conv outputs of column tid
    const int cidx = (tid >> 5) * RBS + (tid & 31);
#pragma unroll
    for (int t = 0; t < TK; ++t) {
        const bool on = t < ntok;
        const float cq = silu_f32(fmaf(sq[t + 3], wq.w, fmaf(sq[t + 2], wq.z, fmaf(sq[t + 1], wq.y, sq[t] * wq.x))));
        const float ck = silu_f32(fmaf(sk[t + 3], wk.w, fmaf(sk[t + 2], wk.z, fmaf(sk[t + 1], wk.y, sk[t] * wk.x))));
        const float cv = silu_f32(fmaf(sv[t + 3], wv.w, fmaf(sv[t + 2], wv.z, fmaf(sv[t + 1], wv.y, sv[t] * wv.x))));
        qc[t][cidx] = on ? cq : 0.f;
        kc[t][cidx] = on ? ck : 0.f;
        vt[t] = on ? cv : 0.f;
    }
    if (m > 0) {  // history after m tokens: elements m, m+1, m+2 of the sequence
        float* ho = a.hist_out + size_t(n) * C * 3;
#pragma unroll
        for (int e = 0; e < 3; ++e) {
            float hq = sq[e], hkv = sk[e], hv = sv[e];
#pragma unroll
            for (int r = 1; r <= TK; ++r)
                if (r == m) { hq = sq[r + e]; hkv = sk[r + e]; hv = sv[r + e]; }
            if (h < a.h_k) {  // the q/k history of key head hk is written by head h == hk
                ho[size_t(ch_q) * 3 + e] = hq;
                ho[size_t(ch_k) * 3 + e] = hkv;
            }
            ho[size_t(ch_v) * 3 + e] = hv;
        }
    }
    // the gates: log gate and beta of token lane, gamma_t, and the decay from t to token m-1
    if (warp == 0) {
        float l = 0.f, be = 0.f;
        if (lane < ntok) {
            const size_t gi = (size_t(n) * ntok + lane) * a.h_v + h;
            l = softplus_f32(a.alpha[gi] + a.dt[h]) * a.ssm_a[h];
            be = sigmoid_f32(a.beta[gi]);
        }
        float pre = l, suf = __shfl_down_sync(kFullMask, lane < m ? l : 0.f, 1);  // suf: sum over t < r < m
#pragma unroll
        for (int o = 1; o < TK; o <<= 1) {
            const float y = __shfl_up_sync(kFullMask, pre, o);
            if (lane >= o) pre += y;
            const float z = __shfl_down_sync(kFullMask, suf, o);
            if (lane + o < 32) suf += z;
        }
        if (lane < TK) {
            lg[lane] = l;
            bet[lane] = be;
            gam[lane] = expf(pre);
            gtl[lane] = lane < m ? expf(suf) : 0.f;
        }
    }
    __syncthreads();

    // ---- the Gram entries, one thread per entry of the 8 x 8 blocks K K^T and Q K^T (four
    // accumulators over the 128 channels); the thread of Q K^T's diagonal entry t also forms |q_t|^2
    {
        const int which = tid >> 6, t = (tid >> 3) & 7, s = tid & 7;
        const float* x = which ? qc[t] : kc[t];
        const float* y = kc[s];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), aq = acc;
#pragma unroll 8
        for (int c4 = 0; c4 < D / 4; ++c4) {
            const int off = (c4 >> 3) * RBS + 4 * (c4 & 7);
            const float4 xv = *reinterpret_cast<const float4*>(x + off);
            const float4 yv = *reinterpret_cast<const float4*>(y + off);
            acc.x = fmaf(xv.x, yv.x, acc.x); acc.y = fmaf(xv.y, yv.y, acc.y);
            acc.z = fmaf(xv.z, yv.z, acc.z); acc.w = fmaf(xv.w, yv.w, acc.w);
            aq.x = fmaf(xv.x, xv.x, aq.x); aq.y = fmaf(xv.y, xv.y, aq.y);
            aq.z = fmaf(xv.z, xv.z, aq.z); aq.w = fmaf(xv.w, xv.w, aq.w);
        }
        const float d = (acc.x + acc.y) + (acc.z + acc.w);
        float seg = 0.f;  // log gates of tokens s+1 .. t
        for (int r = s + 1; r <= t; ++r) seg += lg[r];
        if (which == 0) {
            if (s == t) kk2[t] = d;
            else if (s < t) kkd[t][s] = expf(seg) * d;
        } else if (s <= t) {
            qkd[t][s] = expf(seg) * d;
            if (s == t) qq2[t] = (aq.x + aq.y) + (aq.z + aq.w);
        }
    }

    // ---- S0^T k_t and S0^T q_t of this warp's 32 columns, a token pair at a time
    {
        const float4* k4 = reinterpret_cast<const float4*>(&kc[0][0] + rb * RBS);
        const float4* q4 = reinterpret_cast<const float4*>(&qc[0][0] + rb * RBS);
        constexpr int TS = TSTR / 4;  // float4 stride between tokens
#pragma unroll 1  // a rolled loop: the body is reused from the instruction cache
        for (int tp = 0; tp < TK / 2; ++tp) {
            if (2 * tp >= ntok) break;
            float2 ak[2][4], aq[2][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) ak[0][j] = ak[1][j] = aq[0][j] = aq[1][j] = make_float2(0.f, 0.f);
#pragma unroll
            for (int m4 = 0; m4 < NR / 4; ++m4) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float4 kk = k4[(2 * tp + u) * TS + m4];
                    const float4 qq = q4[(2 * tp + u) * TS + m4];
                    const float2 k01 = make_float2(kk.x, kk.y), k23 = make_float2(kk.z, kk.w);
                    const float2 q01 = make_float2(qq.x, qq.y), q23 = make_float2(qq.z, qq.w);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        ak[u][j] = __ffma2_rn(R[2 * m4][j], k01, ak[u][j]);
                        ak[u][j] = __ffma2_rn(R[2 * m4 + 1][j], k23, ak[u][j]);
                        aq[u][j] = __ffma2_rn(R[2 * m4][j], q01, aq[u][j]);
                        aq[u][j] = __ffma2_rn(R[2 * m4 + 1][j], q23, aq[u][j]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float kv[4], qr[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    kv[j] = ak[u][j].x + ak[u][j].y;
                    qr[j] = aq[u][j].x + aq[u][j].y;
                }
#pragma unroll
                for (int o = 8; o < 32; o <<= 1)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        kv[j] += __shfl_xor_sync(kFullMask, kv[j], o);
                        qr[j] += __shfl_xor_sync(kFullMask, qr[j], o);
                    }
                if (rb == 0) {
                    *reinterpret_cast<float4*>(&kvp[2 * tp + u][col]) = make_float4(kv[0], kv[1], kv[2], kv[3]);
                    *reinterpret_cast<float4*>(&qrp[2 * tp + u][col]) = make_float4(qr[0], qr[1], qr[2], qr[3]);
                }
            }
        }
    }
    __syncthreads();

    // ---- the triangular solve and the outputs of column tid (held by this thread's own warp)
    float ov[TK];
    {
        float w[TK];
#pragma unroll
        for (int t = 0; t < TK; ++t) {
            const float rk = rsqrtf(kk2[t] + a.eps);
            const float rq = rsqrtf(qq2[t] + a.eps) * 0.08838834764831845f;  // rq / sqrt(128)
            const float g = gam[t];
            float acc = g * kvp[t][tid];
#pragma unroll
            for (int s = 0; s < t; ++s) acc = fmaf(kkd[t][s], w[s], acc);
            w[t] = t < ntok ? rk * (bet[t] * (vt[t] - rk * acc)) : 0.f;  // tokens past ntok: no S0^T k_t
            float o = g * qrp[t][tid];
#pragma unroll
            for (int s = 0; s <= t; ++s) o = fmaf(qkd[t][s], w[s], o);
            ov[t] = o * rq;
            wsm[t][tid] = w[t];
        }
        // the sums of o^2 over this warp's 32 columns, per token
#pragma unroll
        for (int t = 0; t < TK; ++t) {
            float e = ov[t] * ov[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(kFullMask, e, o);
            if (lane == 0) ssw[t][warp] = e;
        }
    }
    __syncwarp();

    // ---- commit: S = gamma_{m-1} S0 + sum_{s<m} k_s (D_{m-1,s} w_s)^T, four tokens at a time
    if (m > 0) {
        const float gm = gam[m - 1];
        const float2 g2 = make_float2(gm, gm);
#pragma unroll
        for (int p = 0; p < NR / 2; ++p)
#pragma unroll
            for (int j = 0; j < 4; ++j) R[p][j] = __fmul2_rn(R[p][j], g2);
        const float4* k4 = reinterpret_cast<const float4*>(&kc[0][0] + rb * RBS);
        constexpr int TS = TSTR / 4;
#pragma unroll 1
        for (int hf = 0; hf < TK / 4; ++hf) {
            if (4 * hf >= m) break;
            float2 d2[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int s = 4 * hf + u;
                const float f = gtl[s];
                const float4 ww = s < m ? *reinterpret_cast<const float4*>(&wsm[s][col]) : make_float4(0.f, 0.f, 0.f, 0.f);
                d2[u][0] = make_float2(f * ww.x, f * ww.x);
                d2[u][1] = make_float2(f * ww.y, f * ww.y);
                d2[u][2] = make_float2(f * ww.z, f * ww.z);
                d2[u][3] = make_float2(f * ww.w, f * ww.w);
            }
#pragma unroll
            for (int m4 = 0; m4 < NR / 4; ++m4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 kk = k4[(4 * hf + u) * TS + m4];
                    const float2 k01 = make_float2(kk.x, kk.y), k23 = make_float2(kk.z, kk.w);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        R[2 * m4][j] = __ffma2_rn(k01, d2[u][j], R[2 * m4][j]);
                        R[2 * m4 + 1][j] = __ffma2_rn(k23, d2[u][j], R[2 * m4 + 1][j]);
                    }
                }
            }
        }
#pragma unroll
        for (int p = 0; p < NR / 2; ++p) {
            st_stream(reinterpret_cast<float4*>(sbase + size_t(rb * NR + 2 * p) * row_stride),
                      make_float4(R[p][0].x, R[p][1].x, R[p][2].x, R[p][3].x));
            st_stream(reinterpret_cast<float4*>(sbase + size_t(rb * NR + 2 * p + 1) * row_stride),
                      make_float4(R[p][0].y, R[p][1].y, R[p][2].y, R[p][3].y));
        }
    }

    cp_async_wait_all();  // this thread's z and gamma (read only by this thread)
    __syncthreads();
    // the gated RMSNorm over the head's 128 outputs of each token
#pragma unroll
    for (int i = 0; i < TK; ++i) {
        if (i < ntok) {
            const float ss = (ssw[i][0] + ssw[i][1]) + (ssw[i][2] + ssw[i][3]);
            const float rs = rsqrtf(ss / float(D) + a.eps);
            const size_t yi = ((size_t(n) * ntok + i) * a.h_v + h) * D + tid;
            a.y[yi] = ov[i] * rs * gs[tid] * sigmoid_f32(zs[i * D + tid]);
        }
    }
}

}  // namespace gdn
