// comba_forward.cuh -- the Comba recurrence over T tokens per head, the state slab held on chip.
#pragma once

#include "common.cuh"
#include "kernel_args.h"

namespace gdn {

// The Comba recurrence over T tokens of one head (KBench specs/comba_decode_step.py, spec_md: the
// decode step is the comba-forward task's recurrence for one token, and T steps reproduce that
// task), computed chunk by chunk (CH = 8 tokens) in the WY form, on CUDA cores, with the head's
// K x V slab in registers (read once, written once per call).  For a chunk with start state S0,
// gamma_t = exp(g_0 + ... + g_t) and D_ts = exp(g_{s+1} + ... + g_t):
//     u_t  = beta_t (v_t - gamma_t S0^T p_t) - sum_{s<t} beta_t D_ts (p_t . k_s) u_s
//     o_t  = gamma_t S0^T q_t + sum_{s<=t} D_ts (q_t . k_s) u_s          (q pre-scaled)
//     S    = gamma_L S0 + sum_s D_Ls k_s u_s^T
// -- the T single steps regrouped: u_t is the step's correction, the state before step t being
// gamma_t S0 + sum_{s<t} D_ts k_s u_s^T.  A chunk is one pass over the slab forming S0^T p_t and
// S0^T q_t for all its tokens, a reduction over K in shared memory, a small triangular solve per
// column (one warp), and one pass applying the chunk's writes.  Every decay is the exponential of a
// sum over its own segment (never a difference of running sums), so a gate of -inf zeroes exactly
// the terms whose segment crosses it.
//
// A thread holds 4 columns (column group c) of the rows rg + RG*m; rows m = 2j and 2j+1 form a pair,
// and the chunk's keys sit in shared memory as [row pair][token][2], so every packed f32x2 FMA of
// both passes takes a row pair of the state and a row pair of one key with no register shuffling.
template <int K, int V, int NT>
__global__ void __launch_bounds__(NT, 2) comba_forward_kernel(const CombaFwdArgs a) {
    constexpr int CG = V / 4;      // float4 column groups
    constexpr int RG = NT / CG;    // row groups
    constexpr int NR = K / RG;     // rows per thread
    constexpr int NP = NR / 2;     // row pairs per thread
    constexpr int CH = 8;          // tokens per chunk
    constexpr int TPE = NT / (2 * CH * CH);  // threads per Gram entry
    static_assert(CG * 4 == V && RG * CG == NT && NR * RG == K && NP * 2 == NR && RG >= CH, "tile split");
    static_assert(TPE == 2, "Gram split");

    extern __shared__ __align__(16) float4 dsm[];
    float* ps = reinterpret_cast<float*>(dsm);           // read keys    [K/2][CH][2]
    float* ks = ps + CH * K;                              // write keys   [K/2][CH][2]
    float* qs = ks + CH * K;                              // scale * q    [K/2][CH][2]
    float4* vs = reinterpret_cast<float4*>(qs + CH * K);  // [CH][CG] values, then the corrections u
    float4* red = vs + CH * CG;                           // [RG][CH][2][CG] partial S0^T p, S0^T q
    float4* tot = red + RG * CH * 2 * CG;                 // [CH][2][CG] their sums
    __shared__ float amat[CH][CH], qmat[CH][CH];          // beta_t D_ts (p_t.k_s), s<t; D_ts (q_t.k_s), s<=t
    __shared__ float glog[CH], bet[CH], gam[CH], gtail[CH];  // g_t, beta_t, gamma_t, D_{L-1,t}

    const int head = blockIdx.x;  // b * H + h
    const int b = head / a.H, h = head - b * a.H;
    const int c = threadIdx.x % CG;
    const int rg = threadIdx.x / CG;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T;
    float4* st = reinterpret_cast<float4*>(a.state + size_t(head) * K * V);
    auto tok = [&](int t) { return (size_t(b) * T + t) * a.H + h; };  // token t of this head
    // shared-memory offset of element i of token t's key
    auto koff = [](int i, int t) {
        const int m = i / RG, r = i - m * RG;
        return (((m >> 1) * RG + r) * CH + t) * 2 + (m & 1);
    };

    // the state, rows paired: s2[j][x] = (S[rg + RG*2j][4c+x], S[rg + RG*(2j+1)][4c+x])
    float2 s2[NP][4];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        const float4 r0 = ld_stream(st + size_t(rg + RG * (2 * j)) * CG + c);
        const float4 r1 = ld_stream(st + size_t(rg + RG * (2 * j + 1)) * CG + c);
        s2[j][0] = make_float2(r0.x, r1.x);
        s2[j][1] = make_float2(r0.y, r1.y);
        s2[j][2] = make_float2(r0.z, r1.z);
        s2[j][3] = make_float2(r0.w, r1.w);
    }

    for (int t0 = 0; t0 < T; t0 += CH) {
        const int n = T - t0 < CH ? T - t0 : CH;
        // ---- 1. the chunk's vectors (tokens past n: zero) and gates
        for (int e = threadIdx.x; e < CH * K / 4; e += NT) {
            const int t = e % CH, i4 = e / CH;
            float4 pp = make_float4(0.f, 0.f, 0.f, 0.f), kk = pp, qq = pp;
            if (t < n) {
                const size_t o = tok(t0 + t) * K + 4 * i4;
                pp = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.p + o));
                kk = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.k + o));
                qq = bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.q + o));
                qq = make_float4(a.scale * qq.x, a.scale * qq.y, a.scale * qq.z, a.scale * qq.w);
            }
            const int i = 4 * i4;
            ps[koff(i, t)] = pp.x; ps[koff(i + 1, t)] = pp.y; ps[koff(i + 2, t)] = pp.z; ps[koff(i + 3, t)] = pp.w;
            ks[koff(i, t)] = kk.x; ks[koff(i + 1, t)] = kk.y; ks[koff(i + 2, t)] = kk.z; ks[koff(i + 3, t)] = kk.w;
            qs[koff(i, t)] = qq.x; qs[koff(i + 1, t)] = qq.y; qs[koff(i + 2, t)] = qq.z; qs[koff(i + 3, t)] = qq.w;
        }
        for (int e = threadIdx.x; e < CH * CG; e += NT) {
            const int t = e / CG, cc = e - t * CG;
            vs[e] = t < n ? bf16x4_to_f32x4(*reinterpret_cast<const uint2*>(a.v + tok(t0 + t) * V + 4 * cc))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (warp == 0) {  // lanes past n (and past CH) carry g = 0, beta = 0
            float gl = 0.f, be = 0.f;
            if (lane < n) {
                gl = a.g[tok(t0 + lane)];
                be = bf16_to_f32(a.beta[tok(t0 + lane)]);
            }
            float pre = gl, suf = __shfl_down_sync(kFullMask, gl, 1);  // suf: the sum over r > t
#pragma unroll
            for (int o = 1; o < CH; o <<= 1) {
                const float y = __shfl_up_sync(kFullMask, pre, o);
                if (lane >= o) pre += y;
                const float z = __shfl_down_sync(kFullMask, suf, o);
                if (lane + o < 32) suf += z;
            }
            if (lane < CH) {
                glog[lane] = gl;
                bet[lane] = be;
                gam[lane] = expf(pre);
                gtail[lane] = expf(suf);
            }
        }
        __syncthreads();

        // ---- 2a. the Gram entries with their decays, two threads per entry (halves of the row pairs)
        {
            const int e = threadIdx.x / TPE, part = threadIdx.x % TPE;
            const int which = e / (CH * CH), t = (e / CH) % CH, s = e % CH;
            const float* x = which ? qs : ps;
            float d = 0.f;
            for (int sl = part; sl < K / 2; sl += TPE) {
                const float2 xv = *reinterpret_cast<const float2*>(x + (sl * CH + t) * 2);
                const float2 yv = *reinterpret_cast<const float2*>(ks + (sl * CH + s) * 2);
                d = fmaf(xv.x, yv.x, d);
                d = fmaf(xv.y, yv.y, d);
            }
            d += __shfl_xor_sync(kFullMask, d, 1);
            if (part == 0) {
                float seg = 0.f;  // g_{s+1} + ... + g_t
                for (int r = s + 1; r <= t; ++r) seg += glog[r];
                if (which == 0)
                    amat[t][s] = s < t ? bet[t] * expf(seg) * d : 0.f;
                else
                    qmat[t][s] = s <= t ? expf(seg) * d : 0.f;
            }
        }
        // ---- 2b. this thread's parts of S0^T p_t and S0^T q_t, a token pair at a time
#pragma unroll
        for (int tp = 0; tp < CH / 2; ++tp) {
            float2 ap[2][4], aq[2][4];
#pragma unroll
            for (int x = 0; x < 4; ++x) ap[0][x] = ap[1][x] = aq[0][x] = aq[1][x] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const int sl = j * RG + rg;
                const float4 pv = *reinterpret_cast<const float4*>(ps + (sl * CH + 2 * tp) * 2);
                const float4 qv = *reinterpret_cast<const float4*>(qs + (sl * CH + 2 * tp) * 2);
                const float2 p0 = make_float2(pv.x, pv.y), p1 = make_float2(pv.z, pv.w);
                const float2 q0 = make_float2(qv.x, qv.y), q1 = make_float2(qv.z, qv.w);
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    ap[0][x] = __ffma2_rn(p0, s2[j][x], ap[0][x]);
                    ap[1][x] = __ffma2_rn(p1, s2[j][x], ap[1][x]);
                    aq[0][x] = __ffma2_rn(q0, s2[j][x], aq[0][x]);
                    aq[1][x] = __ffma2_rn(q1, s2[j][x], aq[1][x]);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = 2 * tp + u;
                red[((rg * CH + t) * 2 + 0) * CG + c] = make_float4(ap[u][0].x + ap[u][0].y, ap[u][1].x + ap[u][1].y,
                                                                    ap[u][2].x + ap[u][2].y, ap[u][3].x + ap[u][3].y);
                red[((rg * CH + t) * 2 + 1) * CG + c] = make_float4(aq[u][0].x + aq[u][0].y, aq[u][1].x + aq[u][1].y,
                                                                    aq[u][2].x + aq[u][2].y, aq[u][3].x + aq[u][3].y);
            }
        }
        __syncthreads();
        // ---- 3. the sums over the row groups: row group t sums token t's parts
        if (rg < CH) {
            float4 sp = red[((0 * CH + rg) * 2 + 0) * CG + c], sq = red[((0 * CH + rg) * 2 + 1) * CG + c];
#pragma unroll
            for (int j = 1; j < RG; ++j) {
                const float4 yp = red[((j * CH + rg) * 2 + 0) * CG + c], yq = red[((j * CH + rg) * 2 + 1) * CG + c];
                sp.x += yp.x; sp.y += yp.y; sp.z += yp.z; sp.w += yp.w;
                sq.x += yq.x; sq.y += yq.y; sq.z += yq.z; sq.w += yq.w;
            }
            tot[(rg * 2 + 0) * CG + c] = sp;
            tot[(rg * 2 + 1) * CG + c] = sq;
        }
        __syncthreads();
        // ---- 4. the corrections u_t of this column group (first row group), in place of v_t
        if (rg == 0) {
            float4 u[CH];
#pragma unroll
            for (int t = 0; t < CH; ++t) {
                const float bt = bet[t], gm = gam[t];
                const float4 rp = tot[(t * 2 + 0) * CG + c], vv = vs[t * CG + c];
                float4 x = make_float4(bt * (vv.x - gm * rp.x), bt * (vv.y - gm * rp.y), bt * (vv.z - gm * rp.z),
                                       bt * (vv.w - gm * rp.w));
#pragma unroll
                for (int s = 0; s < t; ++s) {
                    const float f = amat[t][s];
                    x.x = fmaf(-f, u[s].x, x.x); x.y = fmaf(-f, u[s].y, x.y);
                    x.z = fmaf(-f, u[s].z, x.z); x.w = fmaf(-f, u[s].w, x.w);
                }
                u[t] = x;
                vs[t * CG + c] = x;
            }
        }
        __syncthreads();
        // ---- 5. the outputs: row group t forms o_t
        if (rg < n) {
            const int t = rg;
            const float gm = gam[t];
            const float4 rq = tot[(t * 2 + 1) * CG + c];
            float4 o = make_float4(gm * rq.x, gm * rq.y, gm * rq.z, gm * rq.w);
            for (int s = 0; s <= t; ++s) {
                const float f = qmat[t][s];
                const float4 us = vs[s * CG + c];
                o.x = fmaf(f, us.x, o.x); o.y = fmaf(f, us.y, o.y); o.z = fmaf(f, us.z, o.z); o.w = fmaf(f, us.w, o.w);
            }
            const size_t nn = tok(t0 + t);
            if (a.o_f32) {
                reinterpret_cast<float4*>(static_cast<float*>(a.o) + nn * V)[c] = o;
            } else {
                uint2 pkd;
                pkd.x = uint32_t(f32_to_bf16_rne(o.x)) | (uint32_t(f32_to_bf16_rne(o.y)) << 16);
                pkd.y = uint32_t(f32_to_bf16_rne(o.z)) | (uint32_t(f32_to_bf16_rne(o.w)) << 16);
                reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.o) + nn * V)[c] = pkd;
            }
        }
        // ---- 6. S = gamma_L S0 + sum_s k_s (D_Ls u_s)^T, four tokens at a time
        {
            const float gL = gam[CH - 1];
            const float2 g2 = make_float2(gL, gL);
#pragma unroll
            for (int j = 0; j < NP; ++j)
#pragma unroll
                for (int x = 0; x < 4; ++x) s2[j][x] = __fmul2_rn(s2[j][x], g2);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float2 d2[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int t = 4 * hf + u;
                    const float w = gtail[t];
                    const float4 us = vs[t * CG + c];
                    d2[u][0] = make_float2(w * us.x, w * us.x);
                    d2[u][1] = make_float2(w * us.y, w * us.y);
                    d2[u][2] = make_float2(w * us.z, w * us.z);
                    d2[u][3] = make_float2(w * us.w, w * us.w);
                }
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    const int sl = j * RG + rg;
                    const float4 k01 = *reinterpret_cast<const float4*>(ks + (sl * CH + 4 * hf) * 2);
                    const float4 k23 = *reinterpret_cast<const float4*>(ks + (sl * CH + 4 * hf + 2) * 2);
                    const float2 kp[4] = {make_float2(k01.x, k01.y), make_float2(k01.z, k01.w),
                                          make_float2(k23.x, k23.y), make_float2(k23.z, k23.w)};
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int x = 0; x < 4; ++x) s2[j][x] = __ffma2_rn(kp[u], d2[u][x], s2[j][x]);
                }
            }
        }
        __syncthreads();  // the chunk's shared vectors are no longer read
    }

    // the state after the last token
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        st_stream(st + size_t(rg + RG * (2 * j)) * CG + c,
                  make_float4(s2[j][0].x, s2[j][1].x, s2[j][2].x, s2[j][3].x));
        st_stream(st + size_t(rg + RG * (2 * j + 1)) * CG + c,
                  make_float4(s2[j][0].y, s2[j][1].y, s2[j][2].y, s2[j][3].y));
    }
}

// Dynamic shared memory of the kernel above.
template <int K, int V, int NT>
constexpr int comba_forward_smem() {
    constexpr int CG = V / 4, RG = NT / CG, CH = 8;
    return 3 * CH * K * 4 + (CH * CG + RG * CH * 2 * CG + CH * 2 * CG) * 16;
}

}  // namespace gdn
