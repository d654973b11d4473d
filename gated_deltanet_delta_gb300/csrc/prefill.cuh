// prefill.cuh -- the varlen chunkwise-WY prefill on tcgen05 tensor cores.
//
// What it computes: pymllm gdn_chunkwise, module doc "Algorithm (per chunk of C tokens with initial
// state S_0)", steps 1-3, over the sequences of gdn_extend_chunkwise (cu_seqlens, state_pool,
// cache_indices, gates derived from a, b, A_log, dt_bias).  Per (sequence, value head h, key head
// hk = h / (Hv/Hk)) and chunk of L <= 64 tokens, in the ratio form (every exponential is
// exp(G_t - G_s) with s <= t, G the in-chunk cumulative log-gate):
//     l_t = -exp(A_log) softplus(a_t + dt_bias);  G_t = sum_{r<=t} l_r;  beta_t = sigmoid(b_t)
//     k^ = k rk, q^ = scale q rq with rk = 1/sqrt(|k|^2 + eps), rq likewise
//     Lm_ts = beta_t k^_t.k^_s e^{G_t-G_s} (s < t);  T = (I + Lm)^-1           (fp32, CUDA cores)
//     W = T diag(beta gamma) K^,  U = T diag(beta) V                            (step 1, WY build)
//     Delta = U - W S0^T                                                        ("new values")
//     O = diag(gamma) Q^ S0^T + (Q^ K^^T o D) Delta                             (step 2)
//     S_new = gamma_L S0 + Delta^T diag(D_L) K^                                 (step 3)
// with D_ts = e^{G_t-G_s} for s <= t (0 above the diagonal), gamma_t = e^{G_t}, D_L = D_{L-1,.}.
// The page's w recursion is read untransposed and its "U^T K" as U K^T (the [V, K] state layout).
//
// GB300 mapping.  One CTA of 512 threads per (sequence, value head); threads i, i + 128, i + 256
// and i + 384 share TMEM lane i (each takes a quarter of the columns).  q, k and v rows arrive by
// TMA (cp.async.bulk.tensor, 64 tokens x 64 features per box) straight into the swizzled operand
// tiles; the next chunk's v and q are fetched as soon as their last MMA has read them, its k after
// the state update.  The fp32 state S (V x K = 128 x 128) lives in TMEM
// for the whole sequence and reaches HBM only at the start (gather from the pool slot) and at the
// end (scatter back).  Every contraction is a
// tcgen05.mma with M = 128 (the transposed forms keep V or the feature index on M):
//     G   = [K; Q] K^T              M=128 (64 k rows + 64 q rows), N=64,  K=128   bf16 (exact inputs)
//     W^T = K^T Tw^T,  U^T = V^T Tu^T   M=128, N=64, K=64   (Tw = T diag(beta gamma rk), Tu = T diag(beta))
//     Delta^T = U^T - S0 W^T,  P^T = S0 Q^T                M=128, N=64, K=128
//     (M Delta)^T = Delta^T M^T   (M = Q K^T o D rk_s)    M=128, N=64, K=64
//     S += Delta~^T K            (Delta~ = diag(D_L rk) Delta)   M=128, N=128, K=64
// Raw bf16 q, k, v tiles are exact MMA operands; all row scales (norms, gates, decays) are folded
// into the computed operand or applied in fp32 afterwards.  Computed operands are rounded to bf16,
// except T, Delta~ and both factors of M Delta, which are split into a bf16 high part and a bf16
// low part (x = hi + lo, two or three MMAs): with plain bf16 there the output and the carried state
// miss their tolerances.  The triangular inverse runs in fp32 on CUDA cores, blockwise (16 x 16
// diagonal blocks by column-parallel forward substitution, then the off-diagonal blocks).
// Chunks never straddle sequences; rows past a sequence's end are zero in the tiles and have
// beta = 0 and l = 0, so they change nothing and their outputs are not written.
#pragma once

#include "common.cuh"
#include "kernel_args.h"
#include "tcgen05.cuh"

namespace gdn {

namespace pf {
constexpr int C = 64;     // chunk size
constexpr int D = 128;    // K = V = 128
constexpr int NT = 512;   // threads per CTA: four per TMEM lane, each with a quarter of the columns
constexpr int LST = 68;   // row stride (floats) of the fp32 Lm and T matrices: rows are 16-byte aligned
constexpr int ZST = 36;   // row stride (floats) of the 32 x 32 scratch of the inverse
// dynamic shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;       // [K;Q] tile: two 64-feature halves of 16 KB, each 64 k rows + 64 q rows
constexpr uint32_t OFF_V = 32768;    // V tile: two halves of 8 KB (64 token rows)
constexpr uint32_t OFF_S = 49152;    // S0 bf16, K-major, 128 v rows, two halves of 16 KB
constexpr uint32_t OFF_W = 81920;    // W as MN-major B operand: 128 feature rows x 64 t
constexpr uint32_t OFF_T4 = 98304;   // Tw hi, Tw lo, Tu hi, Tu lo (8 KB each); later Delta~ hi, lo (16 KB each)
constexpr uint32_t OFF_DL = 131072;  // Delta^T hi, lo (16 KB each): 128 v rows x 64 s
constexpr uint32_t OFF_M = 163840;   // M hi, lo (8 KB each): 64 t rows x 64 s
constexpr uint32_t OFF_L = 180224;   // fp32 [64][LST] strictly lower Lm
constexpr uint32_t OFF_T = OFF_L + 64 * LST * 4;  // fp32 [64][LST] T = (I + Lm)^-1
constexpr uint32_t OFF_X = OFF_T + 64 * LST * 4;  // fp32 [32][ZST] scratch of the blockwise inverse
constexpr uint32_t SMEM_USED = OFF_X + 32 * ZST * 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
// TMEM columns (fp32, 128 lanes)
constexpr uint32_t TM_S = 0, TM_G = 128, TM_W = 192, TM_U = 256, TM_P = 320, TM_MD = 384;
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t kWaitLimit = 1u << 26;  // mbarrier polls before giving up (seconds of waiting)
}  // namespace pf

// Pack 8 floats to 8 bf16 (round to nearest even) in a uint4.
__device__ __forceinline__ uint4 pack_bf16x8(const float* x) {
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}
// Split 8 floats into bf16 high parts and bf16 low parts (x - hi, rounded).
__device__ __forceinline__ void split_bf16x8(const float* x, uint4& hi, uint4& lo) {
    hi = pack_bf16x8(x);
    const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w};
    float l[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        l[2 * i] = x[2 * i] - __uint_as_float(hw[i] << 16);
        l[2 * i + 1] = x[2 * i + 1] - __uint_as_float(hw[i] & 0xffff0000u);
    }
    lo = pack_bf16x8(l);
}
// A descriptor advanced by `bytes` (a multiple of 16): only the 14-bit start-address field changes,
// and addresses stay inside the 256 KB shared window, so a plain add cannot carry out of it.
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

__device__ __forceinline__ float bf16_sumsq8(const uint4& p) {
    const float4 a = bf16x4_to_f32x4(make_uint2(p.x, p.y));
    const float4 b = bf16x4_to_f32x4(make_uint2(p.z, p.w));
    return fmaf(a.x, a.x, fmaf(a.y, a.y, fmaf(a.z, a.z, fmaf(a.w, a.w,
           fmaf(b.x, b.x, fmaf(b.y, b.y, fmaf(b.z, b.z, b.w * b.w)))))));
}
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
    float a[16], b[16];
    tc::ld16(taddr, a);
    tc::ld16(taddr + 16, b);
    tc::wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = a[i];
        v[16 + i] = b[i];
    }
}

__global__ void __launch_bounds__(pf::NT, 1)
    gdn_prefill_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ PrefillMaps maps) {
    using namespace pf;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ float Gf[C], betas[C], rks[C], rqs[C], gams[C], dls[C];
    __shared__ float scan_total;
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(8) uint64_t mbar;     // MMA completion
    __shared__ __align__(8) uint64_t bar_vq;   // TMA of the v and q rows of a chunk
    __shared__ __align__(8) uint64_t bar_k;    // TMA of the k rows of a chunk

    const int n = blockIdx.x / a.Hv;
    const int h = blockIdx.x - n * a.Hv;
    const int hk = h / (a.Hv / a.Hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = tid & 127;   // the TMEM lane this thread reads and writes
    const int qt = tid >> 7;     // which quarter of the columns

    // ---- sequence bounds and pool slot (uniform over the CTA; bad ones are flagged and skipped)
    const long long bos = a.cu_seqlens[n], eos = a.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || eos > a.T) {
        if (tid == 0) atomicOr(a.status, 2);
        return;
    }
    const long long slot = a.cache_indices[n];
    if (slot < 0 || slot >= a.pool_size) {
        if (tid == 0) atomicOr(a.status, 1);
        return;
    }
    const long long Tn = eos - bos;
    if (Tn == 0) return;

    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = tc::smem_u32(sm);
    float* Ls = reinterpret_cast<float*>(sm + OFF_L);
    float* Ts = reinterpret_cast<float*>(sm + OFF_T);
    float* Xs = reinterpret_cast<float*>(sm + OFF_X);

    if (warp == 0) tc::tmem_alloc(&tmem_slot, TM_COLS);
    if (tid == 0) {
        tc::mbar_init(&mbar, 1);
        tc::mbar_init(&bar_vq, 1);
        tc::mbar_init(&bar_k, 1);
    }
    // T's blocks above the diagonal stay zero for the whole kernel
    for (int i = tid; i < C * LST; i += NT) Ts[i] = 0.f;
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = tmem_slot;
    const uint32_t trow = tm + (static_cast<uint32_t>((warp & 3) * 32) << 16);  // TMEM lane base
    uint32_t phase = 0, ph_vq = 0, ph_k = 0;
    bool timed_out = false;
    // operand descriptors at their tile bases (K-major: LBO unused; MN-major: LBO = half stride)
    const uint64_t dKQ = tc::sdesc(sb + OFF_KQ, 16, 1024);         // [K; Q] rows, K-major
    const uint64_t dKmn = tc::sdesc(sb + OFF_KQ, 16384, 1024);     // k rows read MN-major
    const uint64_t dVmn = tc::sdesc(sb + OFF_V, 8192, 1024);       // v rows read MN-major
    const uint64_t dS0 = tc::sdesc(sb + OFF_S, 16, 1024);          // S0, K-major
    const uint64_t dWmn = tc::sdesc(sb + OFF_W, 8192, 1024);       // W, MN-major
    const uint64_t dT4 = tc::sdesc(sb + OFF_T4, 16, 1024);         // Tw/Tu hi/lo, then Delta~ hi/lo
    const uint64_t dDL = tc::sdesc(sb + OFF_DL, 16, 1024);         // Delta hi/lo
    const uint64_t dM = tc::sdesc(sb + OFF_M, 16, 1024);           // M hi/lo

    // one thread polls the mbarrier for the MMAs committed so far; the barrier releases the rest
    // (a timeout on that thread stops every thread)
    auto mma_wait = [&]() -> bool {
        const bool ok = tid != 0 || tc::mbar_wait(&mbar, phase, kWaitLimit);
        phase ^= 1u;
        const bool all = __syncthreads_and(ok ? 1 : 0) != 0;
        tc::fence_after();
        return all;
    };
    auto publish = [&]() {
        tc::wait_st();
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };

    // ---- gather the state from its pool slot: row v, columns 32*qt .. -> TMEM and S0 (bf16)
    float* Sg = a.state_pool + (static_cast<size_t>(slot) * a.Hv + h) * D * D;
    {
        const float4* src = reinterpret_cast<const float4*>(Sg + static_cast<size_t>(row) * D + 32 * qt);
#pragma unroll
        for (int c16 = 0; c16 < 2; ++c16) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 f = src[c16 * 4 + j];
                v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
            }
            tc::st16(trow + TM_S + 32 * qt + c16 * 16, v);
            const int c8 = 4 * qt + 2 * c16;
            *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw_chunk(row, c8, 128)) = pack_bf16x8(v);
            *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw_chunk(row, c8 + 1, 128)) = pack_bf16x8(v + 8);
        }
    }

    const float a_mul = expf(a.A_log[h]);
    const float dtb = a.dt_bias[h];
    const size_t vo_stride = static_cast<size_t>(a.Hv) * D;  // elements between tokens of v, out

    // TMA of one chunk's rows (thread 0): v and q (both halves of each) on bar_vq, k on bar_k.  The
    // boxes land in the 128-byte swizzled operand layout; rows past T arrive as zeros.
    auto issue_vq = [&](long long c0n) {
        const int z = static_cast<int>(bos + c0n);
        tc::mbar_expect_tx(&bar_vq, 4 * 8192);
        tc::tma_load_3d(sb + OFF_KQ + 8192, &maps.q, 0, hk, z, &bar_vq);
        tc::tma_load_3d(sb + OFF_KQ + 16384 + 8192, &maps.q, 64, hk, z, &bar_vq);
        tc::tma_load_3d(sb + OFF_V, &maps.v, 0, h, z, &bar_vq);
        tc::tma_load_3d(sb + OFF_V + 8192, &maps.v, 64, h, z, &bar_vq);
    };
    auto issue_k = [&](long long c0n) {
        const int z = static_cast<int>(bos + c0n);
        tc::mbar_expect_tx(&bar_k, 2 * 8192);
        tc::tma_load_3d(sb + OFF_KQ, &maps.k, 0, hk, z, &bar_k);
        tc::tma_load_3d(sb + OFF_KQ + 16384, &maps.k, 64, hk, z, &bar_k);
    };
    uint16_t a_raw = 0, b_raw = 0;  // gate inputs of token tid (threads < 64)
    auto load_gates = [&](long long c0n) {
        if (tid < Tn - c0n && tid < C) {
            const size_t gi = static_cast<size_t>(bos + c0n + tid) * a.Hv + h;
            a_raw = a.a[gi];
            b_raw = a.b[gi];
        }
    };
    if (tid == 0) {
        issue_vq(0);
        issue_k(0);
    }
    load_gates(0);
    const int rp = tid >> 4, ch = tid & 15;  // norms: 16 threads per row, rows rp and rp + 32
    publish();

    for (long long c0 = 0; c0 < Tn && !timed_out; c0 += C) {
        const int L = static_cast<int>(Tn - c0 < C ? Tn - c0 : C);
        const long long tok0 = bos + c0;

        // ---- 1. wait for this chunk's rows, zero the rows past the sequence end, row norms
        {
            const bool ok = tc::mbar_wait(&bar_vq, ph_vq, kWaitLimit) && tc::mbar_wait(&bar_k, ph_k, kWaitLimit);
            ph_vq ^= 1u;
            ph_k ^= 1u;
            if (!__syncthreads_and(ok ? 1 : 0)) { timed_out = true; break; }
        }
        if (L < C) {
            for (int e = tid; e < (C - L) * 16; e += NT) {
                const int s = L + (e >> 4), c = e & 15;
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sm + OFF_KQ + tc::sw_chunk(s, c, 128)) = z;
                *reinterpret_cast<uint4*>(sm + OFF_KQ + tc::sw_chunk(64 + s, c, 128)) = z;
                *reinterpret_cast<uint4*>(sm + OFF_V + tc::sw_chunk(s, c, 64)) = z;
            }
            __syncthreads();
        }
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int s = p * 32 + rp;
            const uint4 kv4 = *reinterpret_cast<const uint4*>(sm + OFF_KQ + tc::sw_chunk(s, ch, 128));
            const uint4 qv4 = *reinterpret_cast<const uint4*>(sm + OFF_KQ + tc::sw_chunk(64 + s, ch, 128));
            float sk = bf16_sumsq8(kv4), sq = bf16_sumsq8(qv4);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                sk += __shfl_xor_sync(kFullMask, sk, o);
                sq += __shfl_xor_sync(kFullMask, sq, o);
            }
            if (ch == 0) {
                rks[s] = rsqrtf(sk + a.eps);
                rqs[s] = rsqrtf(sq + a.eps);
            }
        }
        publish();

        // ---- 2. G = [K; Q] K^T, committed alone; P^T = S0 Q^T is issued behind it and completes
        //         with the next commit group (it needs only this chunk's q rows and S0)
        if (tid == 0) {
            const uint32_t id = tc::idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t d = dadd(dKQ, (ks >> 2) * 16384 + (ks & 3) * 32);
                tc::mma_bf16(tm + TM_G, d, d, id, ks > 0);
            }
            tc::commit(&mbar);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                tc::mma_bf16(tm + TM_P, dadd(dS0, off), dadd(dKQ, 8192 + off), id, ks > 0);
            }
        }
        // ---- 3. gates and their in-chunk cumulative sum (while G is computed)
        if (tid < C) {
            const int t = tid;
            float ell = 0.f, be = 0.f;
            if (t < L) {
                const float x = bf16_to_f32(a_raw) + dtb;
                const float sp = x > 20.f ? x : log1pf(__expf(x));
                ell = -a_mul * sp;
                be = __frcp_rn(1.f + __expf(-bf16_to_f32(b_raw)));
            }
            float g = ell;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(kFullMask, g, o);
                if (lane >= o) g += y;
            }
            if (t == 31) scan_total = g;
            asm volatile("bar.sync 1, 64;" ::: "memory");
            if (t >= 32) g += scan_total;
            Gf[t] = g;
            betas[t] = be;
        }
        __syncthreads();
        if (tid < C) {
            gams[tid] = __expf(Gf[tid]);
            dls[tid] = tid < L ? __expf(Gf[L - 1] - Gf[tid]) : 0.f;
        }
        if (!mma_wait()) { timed_out = true; break; }

        // ---- 4. Lm (lanes t < 64, fp32) and M (lanes 64 + t, bf16 hi / lo) from G, 16 columns each
        {
            float g[16];
            tc::ld16(trow + TM_G + 16 * qt, g);
            tc::wait_ld();
            const int s0 = 16 * qt;
            if (row < C) {
                const int t = row;
                const float bt = betas[t] * rks[t];
                const float Gt = Gf[t];
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    float l4[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int s = s0 + 4 * i4 + u;
                        l4[u] = s < t ? bt * rks[s] * g[4 * i4 + u] * __expf(Gt - Gf[s]) : 0.f;
                    }
                    *reinterpret_cast<float4*>(Ls + t * LST + s0 + 4 * i4) = make_float4(l4[0], l4[1], l4[2], l4[3]);
                }
            } else {
                const int t = row - C;
                const float Gt = Gf[t];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float m8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int s = s0 + c * 8 + i;
                        m8[i] = s <= t ? rks[s] * g[c * 8 + i] * __expf(Gt - Gf[s]) : 0.f;
                    }
                    uint4 hi, lo;
                    split_bf16x8(m8, hi, lo);
                    *reinterpret_cast<uint4*>(sm + OFF_M + tc::sw_chunk(t, 2 * qt + c, 64)) = hi;
                    *reinterpret_cast<uint4*>(sm + OFF_M + 8192 + tc::sw_chunk(t, 2 * qt + c, 64)) = lo;
                }
            }
        }
        __syncthreads();

        // ---- 5. T = (I + Lm)^-1 (unit lower triangular, 64 x 64, fp32):
        //   A: the four 16 x 16 diagonal blocks by column-parallel forward substitution;
        //   B: T_{2p+1,2p} = -T_{2p+1,2p+1} Lm_{2p+1,2p} T_{2p,2p}   (32 x 32 diagonal blocks);
        //   C: T_{[32,64),[0,32)} = -T_br Lm_bl T_tl                 (the whole matrix).
        //   B and C give each thread one row and four consecutive columns (float4 operands).
        if (tid < C) {
            const int blk = tid >> 4, j = tid & 15;
            const float* Lb = Ls + (16 * blk) * LST + 16 * blk;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float acc0 = (i == j) ? 1.f : 0.f, acc1 = 0.f;
#pragma unroll
                for (int s2 = 0; s2 + 1 < i; s2 += 2) {
                    acc0 = fmaf(-Lb[i * LST + s2], x[s2], acc0);
                    acc1 = fmaf(-Lb[i * LST + s2 + 1], x[s2 + 1], acc1);
                }
                if (i & 1) acc0 = fmaf(-Lb[i * LST + i - 1], x[i - 1], acc0);
                x[i] = (i < j) ? 0.f : acc0 + acc1;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Ts[(16 * blk + i) * LST + 16 * blk + j] = x[i];
        }
        __syncthreads();
        float* Zs = Xs;
        const int pB = tid >> 6, rB = (tid >> 2) & 15, cB = 4 * (tid & 3);
        if (pB < 2) {  // X_p = Lm_{2p+1,2p} T_{2p,2p}
            const float* Lr = Ls + (32 * pB + 16 + rB) * LST + 32 * pB;
            const float* Tc = Ts + (32 * pB) * LST + 32 * pB + cB;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const float4 l = *reinterpret_cast<const float4*>(Lr + 4 * k4);
                const float lk[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 t4 = *reinterpret_cast<const float4*>(Tc + (4 * k4 + u) * LST);
                    acc.x = fmaf(lk[u], t4.x, acc.x); acc.y = fmaf(lk[u], t4.y, acc.y);
                    acc.z = fmaf(lk[u], t4.z, acc.z); acc.w = fmaf(lk[u], t4.w, acc.w);
                }
            }
            *reinterpret_cast<float4*>(Zs + (16 * pB + rB) * ZST + cB) = acc;
        }
        __syncthreads();
        if (pB < 2) {  // T_{2p+1,2p} = -T_{2p+1,2p+1} X_p
            const float* Tr = Ts + (32 * pB + 16 + rB) * LST + 32 * pB + 16;
            const float* Xc = Zs + (16 * pB) * ZST + cB;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const float4 tr = *reinterpret_cast<const float4*>(Tr + 4 * k4);
                const float tk[4] = {tr.x, tr.y, tr.z, tr.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 x4 = *reinterpret_cast<const float4*>(Xc + (4 * k4 + u) * ZST);
                    acc.x = fmaf(tk[u], x4.x, acc.x); acc.y = fmaf(tk[u], x4.y, acc.y);
                    acc.z = fmaf(tk[u], x4.z, acc.z); acc.w = fmaf(tk[u], x4.w, acc.w);
                }
            }
            *reinterpret_cast<float4*>(Ts + (32 * pB + 16 + rB) * LST + 32 * pB + cB) =
                make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();
        const int rC = (tid >> 3) & 31, cC = 4 * (tid & 7);
        if (tid < 256) {  // Z = Lm_bl T_tl
            const float* Lr = Ls + (32 + rC) * LST;
            const float* Tc = Ts + cC;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k4 = 0; k4 < 8; ++k4) {
                const float4 l = *reinterpret_cast<const float4*>(Lr + 4 * k4);
                const float lk[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 t4 = *reinterpret_cast<const float4*>(Tc + (4 * k4 + u) * LST);
                    acc.x = fmaf(lk[u], t4.x, acc.x); acc.y = fmaf(lk[u], t4.y, acc.y);
                    acc.z = fmaf(lk[u], t4.z, acc.z); acc.w = fmaf(lk[u], t4.w, acc.w);
                }
            }
            *reinterpret_cast<float4*>(Zs + rC * ZST + cC) = acc;
        }
        __syncthreads();
        if (tid < 256) {  // T_bl = -T_br Z
            const float* Tr = Ts + (32 + rC) * LST + 32;
            const float* Zc = Zs + cC;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k4 = 0; k4 < 8; ++k4) {
                const float4 tr = *reinterpret_cast<const float4*>(Tr + 4 * k4);
                const float tk[4] = {tr.x, tr.y, tr.z, tr.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 z4 = *reinterpret_cast<const float4*>(Zc + (4 * k4 + u) * ZST);
                    acc.x = fmaf(tk[u], z4.x, acc.x); acc.y = fmaf(tk[u], z4.y, acc.y);
                    acc.z = fmaf(tk[u], z4.z, acc.z); acc.w = fmaf(tk[u], z4.w, acc.w);
                }
            }
            *reinterpret_cast<float4*>(Ts + (32 + rC) * LST + cC) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();

        // ---- 6. Tw = T diag(beta gamma rk), Tu = T diag(beta) as bf16 hi / lo (rows t, K-major)
        {
            const int t = tid & (C - 1);
            const bool w_side = ((tid >> 6) & 1) == 0;
            const uint32_t base = OFF_T4 + (w_side ? 0u : 16384u);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int cc = 2 * qt + c;
                const float4 ta = *reinterpret_cast<const float4*>(Ts + t * LST + cc * 8);
                const float4 tb = *reinterpret_cast<const float4*>(Ts + t * LST + cc * 8 + 4);
                const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
                float x8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int s = cc * 8 + i;
                    const float w = w_side ? betas[s] * gams[s] * rks[s] : betas[s];
                    x8[i] = tv[i] * w;
                }
                uint4 hi, lo;
                split_bf16x8(x8, hi, lo);
                *reinterpret_cast<uint4*>(sm + base + tc::sw_chunk(t, cc, 64)) = hi;
                *reinterpret_cast<uint4*>(sm + base + 8192 + tc::sw_chunk(t, cc, 64)) = lo;
            }
        }
        publish();

        // ---- 7. W^T = K^T Tw^T and U^T = V^T Tu^T (A MN-major from the token tiles)
        if (tid == 0) {
            const uint32_t id = tc::idesc_bf16(128, 64, 1, 0, 0);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    tc::mma_bf16(tm + TM_W, dadd(dKmn, ks * 2048), dadd(dT4, part * 8192 + ks * 32), id,
                                 (part | ks) != 0);
                    tc::mma_bf16(tm + TM_U, dadd(dVmn, ks * 2048),
                                 dadd(dT4, 16384 + part * 8192 + ks * 32), id, (part | ks) != 0);
                }
            tc::commit(&mbar);
        }
        if (!mma_wait()) { timed_out = true; break; }
        if (c0 + C < Tn) {  // the V and Q tiles are free: fetch the next chunk's
            if (tid == 0) issue_vq(c0 + C);
            load_gates(c0 + C);
        }

        // ---- 8. W (bf16) as the MN-major B operand: lane f holds W[t][f], t = 16*qt ..
        {
            float w16[16];
            tc::ld16(trow + TM_W + 16 * qt, w16);
            tc::wait_ld();
#pragma unroll
            for (int c = 0; c < 2; ++c)
                *reinterpret_cast<uint4*>(sm + OFF_W + tc::sw_chunk(row, 2 * qt + c, 128)) =
                    pack_bf16x8(w16 + 8 * c);
        }
        publish();

        // ---- 9. Delta^T = U^T - S0 W^T (accumulated onto U^T, B negated)
        if (tid == 0) {
            const uint32_t idd = tc::idesc_bf16(128, 64, 0, 1, 1);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                tc::mma_bf16(tm + TM_U, dadd(dS0, (ks >> 2) * 16384 + (ks & 3) * 32), dadd(dWmn, ks * 2048),
                             idd, 1u);
            }
            tc::commit(&mbar);
        }
        if (!mma_wait()) { timed_out = true; break; }

        // ---- 10. Delta^T (hi / lo) and Delta~^T = Delta^T diag(D_L rk) (hi / lo), lane v, 16 s each;
        //          the state is scaled by gamma_L in TMEM before the update accumulates onto it
        {
            float d16[16], sa[16], sb16[16];
            tc::ld16(trow + TM_U + 16 * qt, d16);
            tc::ld16(trow + TM_S + 32 * qt, sa);
            tc::ld16(trow + TM_S + 32 * qt + 16, sb16);
            tc::wait_ld();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int cc = 2 * qt + c;
                uint4 hi, lo;
                split_bf16x8(d16 + 8 * c, hi, lo);
                *reinterpret_cast<uint4*>(sm + OFF_DL + tc::sw_chunk(row, cc, 128)) = hi;
                *reinterpret_cast<uint4*>(sm + OFF_DL + 16384 + tc::sw_chunk(row, cc, 128)) = lo;
                float x8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) x8[i] = d16[8 * c + i] * dls[8 * cc + i] * rks[8 * cc + i];
                split_bf16x8(x8, hi, lo);
                *reinterpret_cast<uint4*>(sm + OFF_T4 + tc::sw_chunk(row, cc, 128)) = hi;
                *reinterpret_cast<uint4*>(sm + OFF_T4 + 16384 + tc::sw_chunk(row, cc, 128)) = lo;
            }
            const float gL = gams[L - 1];
            float lo16[16], hi16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                lo16[i] = sa[i] * gL;
                hi16[i] = sb16[i] * gL;
            }
            tc::st16(trow + TM_S + 32 * qt, lo16);
            tc::st16(trow + TM_S + 32 * qt + 16, hi16);
        }
        publish();

        // ---- 11. (M Delta)^T = Delta^T M^T (three hi / lo products) and S += Delta~^T K
        if (tid == 0) {
            const uint32_t idm = tc::idesc_bf16(128, 64, 0, 0, 0);
            const uint32_t ids = tc::idesc_bf16(128, 128, 0, 1, 0);
#pragma unroll
            for (int pr = 0; pr < 3; ++pr) {
                const uint32_t pa = pr == 2 ? 16384u : 0u;  // Delta hi, hi, lo
                const uint32_t pb = pr == 1 ? 8192u : 0u;   // M hi, lo, hi
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tm + TM_MD, dadd(dDL, pa + ks * 32), dadd(dM, pb + ks * 32), idm,
                                 (pr | ks) != 0);
            }
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tm + TM_S, dadd(dT4, part * 16384 + ks * 32), dadd(dKmn, ks * 2048), ids, 1u);
            tc::commit(&mbar);
        }
        if (!mma_wait()) { timed_out = true; break; }
        if (tid == 0 && c0 + C < Tn) issue_k(c0 + C);  // the K tile is free

        // ---- 12. outputs o_t = gamma_t rq_t scale P_t + rq_t scale (M Delta)_t (lane v, 16 tokens);
        //          the new state to bf16 for the next chunk
        {
            float p16[16], m16[16];
            tc::ld16(trow + TM_P + 16 * qt, p16);
            tc::ld16(trow + TM_MD + 16 * qt, m16);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = 16 * qt + i;
                if (t < L) {
                    const float rq = rqs[t] * a.scale;
                    const float o = fmaf(p16[i], gams[t] * rq, m16[i] * rq);
                    a.out[static_cast<size_t>(tok0 + t) * vo_stride + h * D + row] =
                        static_cast<uint16_t>(pack_bf16x2(o, 0.f) & 0xffffu);
                }
            }
            if (c0 + C < Tn) {
                float s32[32];
                ld32(trow + TM_S + 32 * qt, s32);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw_chunk(row, 4 * qt + c, 128)) =
                        pack_bf16x8(s32 + 8 * c);
            }
        }
        publish();
    }

    if (timed_out) {
        if (tid == 0) atomicOr(a.status, 4);
    } else {
        // ---- scatter the final state back to its pool slot (row v, columns 32*qt ..)
        float4* dst = reinterpret_cast<float4*>(Sg + static_cast<size_t>(row) * D + 32 * qt);
        float s32[32];
        ld32(trow + TM_S + 32 * qt, s32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(s32[4 * i], s32[4 * i + 1], s32[4 * i + 2], s32[4 * i + 3]);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, TM_COLS);
}

}  // namespace gdn
