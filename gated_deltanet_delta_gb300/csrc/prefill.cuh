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
// GB300 mapping.  One CTA of 128 threads per (sequence, value head); thread i <-> TMEM lane i.  The
// fp32 state S (V x K = 128 x 128) lives in TMEM for the whole sequence and reaches HBM only at the
// start (gather from the pool slot) and at the end (scatter back).  Every contraction is a
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
constexpr int C = 64;    // chunk size
constexpr int D = 128;   // K = V = 128
constexpr int NT = 128;  // threads per CTA
// dynamic shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;       // [K;Q] tile: two 64-feature halves of 16 KB, each 64 k rows + 64 q rows
constexpr uint32_t OFF_V = 32768;    // V tile: two halves of 8 KB (64 token rows)
constexpr uint32_t OFF_S = 49152;    // S0 bf16, K-major, 128 v rows, two halves of 16 KB
constexpr uint32_t OFF_W = 81920;    // W as MN-major B operand: 128 feature rows x 64 t
constexpr uint32_t OFF_T4 = 98304;   // Tw hi, Tw lo, Tu hi, Tu lo (8 KB each); later Delta~ hi, lo (16 KB each)
constexpr uint32_t OFF_DL = 131072;  // Delta^T hi, lo (16 KB each): 128 v rows x 64 s
constexpr uint32_t OFF_M = 163840;   // M hi, lo (8 KB each): 64 t rows x 64 s
constexpr uint32_t OFF_L = 180224;   // fp32 [64][64] strictly lower Lm
constexpr uint32_t OFF_T = 196608;   // fp32 [64][64] T = (I + Lm)^-1
constexpr uint32_t OFF_X = 212992;   // fp32 [16][48] scratch of the blockwise inverse
constexpr uint32_t SMEM_USED = 216064;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
// TMEM columns (fp32, 128 lanes)
constexpr uint32_t TM_S = 0, TM_G = 128, TM_W = 192, TM_U = 256, TM_P = 320, TM_MD = 384;
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t kWaitLimit = 1u << 26;  // mbarrier polls before giving up (seconds of waiting)
}  // namespace pf

// Pack 8 floats to 8 bf16 (round to nearest even) in a uint4.
__device__ __forceinline__ uint4 pack_bf16x8(const float* x) {
    uint4 r;
    r.x = uint32_t(f32_to_bf16_rne(x[0])) | (uint32_t(f32_to_bf16_rne(x[1])) << 16);
    r.y = uint32_t(f32_to_bf16_rne(x[2])) | (uint32_t(f32_to_bf16_rne(x[3])) << 16);
    r.z = uint32_t(f32_to_bf16_rne(x[4])) | (uint32_t(f32_to_bf16_rne(x[5])) << 16);
    r.w = uint32_t(f32_to_bf16_rne(x[6])) | (uint32_t(f32_to_bf16_rne(x[7])) << 16);
    return r;
}
// Split 8 floats into bf16 high parts and bf16 low parts (x - hi, rounded).
__device__ __forceinline__ void split_bf16x8(const float* x, uint4& hi, uint4& lo) {
    float h[8], l[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        h[i] = bf16_to_f32(f32_to_bf16_rne(x[i]));
        l[i] = x[i] - h[i];
    }
    hi = pack_bf16x8(h);
    lo = pack_bf16x8(l);
}
__device__ __forceinline__ float bf16_sumsq8(const uint4& p) {
    const float4 a = bf16x4_to_f32x4(make_uint2(p.x, p.y));
    const float4 b = bf16x4_to_f32x4(make_uint2(p.z, p.w));
    return fmaf(a.x, a.x, fmaf(a.y, a.y, fmaf(a.z, a.z, fmaf(a.w, a.w,
           fmaf(b.x, b.x, fmaf(b.y, b.y, fmaf(b.z, b.z, b.w * b.w)))))));
}

__global__ void __launch_bounds__(pf::NT, 1) gdn_prefill_kernel(const PrefillArgs a) {
    using namespace pf;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ double Gd[C];
    __shared__ float betas[C], rks[C], rqs[C], gams[C], dls[C];
    __shared__ double scan_total;
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(8) uint64_t mbar;

    const int n = blockIdx.x / a.Hv;
    const int h = blockIdx.x - n * a.Hv;
    const int hk = h / (a.Hv / a.Hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

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
    if (tid == 0) tc::mbar_init(&mbar, 1);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = tmem_slot;
    const uint32_t lrow = static_cast<uint32_t>(warp * 32) << 16;  // this warp's TMEM lane base
    uint32_t phase = 0;
    bool timed_out = false;

    // wait for the MMAs committed so far; returns false (on every thread) after a timeout
    auto mma_wait = [&]() -> bool {
        const bool ok = tc::mbar_wait(&mbar, phase, kWaitLimit);
        phase ^= 1u;
        tc::fence_after();
        return __syncthreads_and(ok ? 1 : 0) != 0;
    };
    // make this thread's shared-memory and TMEM writes visible to the MMAs issued next
    auto publish = [&]() {
        tc::wait_st();
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };

    // ---- gather the state from its pool slot: row v = tid -> TMEM (fp32) and S0 tile (bf16)
    float* Sg = a.state_pool + (static_cast<size_t>(slot) * a.Hv + h) * D * D;
    {
        const float4* row = reinterpret_cast<const float4*>(Sg + static_cast<size_t>(tid) * D);
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 f = row[c16 * 4 + j];
                v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
            }
            tc::st16(tm + lrow + TM_S + c16 * 16, v);
            *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw_chunk(tid, 2 * c16, 128)) = pack_bf16x8(v);
            *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw_chunk(tid, 2 * c16 + 1, 128)) = pack_bf16x8(v + 8);
        }
    }
    publish();

    const float a_mul = expf(a.A_log[h]);
    const float dtb = a.dt_bias[h];
    const size_t qk_stride = static_cast<size_t>(a.Hk) * D;  // elements between tokens of q, k
    const size_t vo_stride = static_cast<size_t>(a.Hv) * D;  // elements between tokens of v, out

    for (long long c0 = 0; c0 < Tn && !timed_out; c0 += C) {
        const int L = static_cast<int>(Tn - c0 < C ? Tn - c0 : C);
        const long long tok0 = bos + c0;

        // ---- 1. k, q, v tiles (zero past the sequence end) and the row norms
        {
            const int rp = tid >> 4, ch = tid & 15;
            uint4 kr[8], qr[8], vr[8];
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const int s = p * 8 + rp;
                if (s < L) {
                    const size_t t = static_cast<size_t>(tok0 + s);
                    kr[p] = *reinterpret_cast<const uint4*>(a.k + t * qk_stride + hk * D + ch * 8);
                    qr[p] = *reinterpret_cast<const uint4*>(a.q + t * qk_stride + hk * D + ch * 8);
                    vr[p] = *reinterpret_cast<const uint4*>(a.v + t * vo_stride + h * D + ch * 8);
                } else {
                    kr[p] = qr[p] = vr[p] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const int s = p * 8 + rp;
                *reinterpret_cast<uint4*>(sm + OFF_KQ + tc::sw_chunk(s, ch, 128)) = kr[p];
                *reinterpret_cast<uint4*>(sm + OFF_KQ + tc::sw_chunk(64 + s, ch, 128)) = qr[p];
                *reinterpret_cast<uint4*>(sm + OFF_V + tc::sw_chunk(s, ch, 64)) = vr[p];
                float sk = bf16_sumsq8(kr[p]), sq = bf16_sumsq8(qr[p]);
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
        }
        // ---- 2. gates and their in-chunk cumulative sum (double, so that G_t - G_s is exact)
        if (tid < C) {
            const int t = tid;
            float ell = 0.f, be = 0.f;
            if (t < L) {
                const size_t gi = static_cast<size_t>(tok0 + t) * a.Hv + h;
                const float x = bf16_to_f32(a.a[gi]) + dtb;
                const float sp = x > 20.f ? x : log1pf(expf(x));
                ell = -a_mul * sp;
                be = 1.f / (1.f + expf(-bf16_to_f32(a.b[gi])));
            }
            double g = ell;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(kFullMask, g, o);
                if (lane >= o) g += y;
            }
            if (t == 31) scan_total = g;
            asm volatile("bar.sync 1, 64;" ::: "memory");
            if (t >= 32) g += scan_total;
            Gd[t] = g;
            betas[t] = be;
        }
        __syncthreads();
        if (tid < C) {
            gams[tid] = expf(static_cast<float>(Gd[tid]));
            dls[tid] = tid < L ? expf(static_cast<float>(Gd[L - 1] - Gd[tid])) : 0.f;
        }
        publish();

        // ---- 3. G = [K; Q] K^T
        if (tid == 0) {
            const uint32_t id = tc::idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                tc::mma_bf16(tm + TM_G, tc::sdesc(sb + OFF_KQ + off, 16, 1024),
                             tc::sdesc(sb + OFF_KQ + off, 16, 1024), id, ks > 0);
            }
            tc::commit(&mbar);
        }
        if (!mma_wait()) { timed_out = true; break; }

        // ---- 4. Lm (rows t < 64, fp32) and M (rows 64 + t, bf16 hi / lo) from G
        {
            float g[64];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v16[16];
                tc::ld16(tm + lrow + TM_G + j * 16, v16);
#pragma unroll
                for (int i = 0; i < 16; ++i) g[j * 16 + i] = v16[i];
            }
            tc::wait_ld();
            if (tid < C) {
                const int t = tid;
                const float bt = betas[t] * rks[t];
                const double Gt = Gd[t];
#pragma unroll
                for (int s = 0; s < C; ++s)
                    Ls[t * C + s] = s < t ? bt * rks[s] * g[s] * __expf(static_cast<float>(Gt - Gd[s])) : 0.f;
            } else {
                const int t = tid - C;
                const double Gt = Gd[t];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float m8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int s = c * 8 + i;
                        m8[i] = s <= t ? rks[s] * g[s] * __expf(static_cast<float>(Gt - Gd[s])) : 0.f;
                    }
                    uint4 hi, lo;
                    split_bf16x8(m8, hi, lo);
                    *reinterpret_cast<uint4*>(sm + OFF_M + tc::sw_chunk(t, c, 64)) = hi;
                    *reinterpret_cast<uint4*>(sm + OFF_M + 8192 + tc::sw_chunk(t, c, 64)) = lo;
                }
            }
            for (int i = tid; i < C * C; i += NT) Ts[i] = 0.f;
        }
        __syncthreads();

        // ---- 5. T = (I + Lm)^-1: 16 x 16 diagonal blocks, then the off-diagonal block rows
        if (tid < C) {
            const int blk = tid >> 4, j = tid & 15;
            const float* Lb = Ls + (16 * blk) * C + 16 * blk;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
                for (int s = 0; s < i; ++s) acc = fmaf(-Lb[i * C + s], x[s], acc);
                x[i] = (i < j) ? 0.f : acc;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Ts[(16 * blk + i) * C + 16 * blk + j] = x[i];
        }
        __syncthreads();
        for (int I = 1; I < 4; ++I) {
            const int W = 16 * I;  // columns to the left of block row I
            for (int e = tid; e < 16 * W; e += NT) {
                const int r = e / W, jc = e - r * W;
                float acc = 0.f;
                for (int k2 = jc & ~15; k2 < W; ++k2) acc = fmaf(Ls[(W + r) * C + k2], Ts[k2 * C + jc], acc);
                Xs[r * 48 + jc] = acc;
            }
            __syncthreads();
            for (int e = tid; e < 16 * W; e += NT) {
                const int r = e / W, jc = e - r * W;
                float acc = 0.f;
#pragma unroll
                for (int k2 = 0; k2 < 16; ++k2) acc = fmaf(Ts[(W + r) * C + W + k2], Xs[k2 * 48 + jc], acc);
                Ts[(W + r) * C + jc] = -acc;
            }
            __syncthreads();
        }

        // ---- 6. Tw = T diag(beta gamma rk), Tu = T diag(beta) as bf16 hi / lo (rows t, K-major)
        {
            const int t = tid & (C - 1);
            const bool w_side = tid < C;
            const uint32_t base = OFF_T4 + (w_side ? 0u : 16384u);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float x8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int s = c * 8 + i;
                    const float w = w_side ? betas[s] * gams[s] * rks[s] : betas[s];
                    x8[i] = Ts[t * C + s] * w;
                }
                uint4 hi, lo;
                split_bf16x8(x8, hi, lo);
                *reinterpret_cast<uint4*>(sm + base + tc::sw_chunk(t, c, 64)) = hi;
                *reinterpret_cast<uint4*>(sm + base + 8192 + tc::sw_chunk(t, c, 64)) = lo;
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
                    tc::mma_bf16(tm + TM_W, tc::sdesc(sb + OFF_KQ + ks * 2048, 16384, 1024),
                                 tc::sdesc(sb + OFF_T4 + part * 8192 + ks * 32, 16, 1024), id,
                                 (part | ks) != 0);
                    tc::mma_bf16(tm + TM_U, tc::sdesc(sb + OFF_V + ks * 2048, 8192, 1024),
                                 tc::sdesc(sb + OFF_T4 + 16384 + part * 8192 + ks * 32, 16, 1024), id,
                                 (part | ks) != 0);
                }
            tc::commit(&mbar);
        }
        if (!mma_wait()) { timed_out = true; break; }

        // ---- 8. W (bf16) as the MN-major B operand: row f = tid holds W[t][f] for t = 0..63
        {
            float w64[64];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v16[16];
                tc::ld16(tm + lrow + TM_W + j * 16, v16);
#pragma unroll
                for (int i = 0; i < 16; ++i) w64[j * 16 + i] = v16[i];
            }
            tc::wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(sm + OFF_W + tc::sw_chunk(tid, c, 128)) = pack_bf16x8(w64 + 8 * c);
        }
        publish();

        // ---- 9. Delta^T = U^T - S0 W^T (accumulated onto U^T, B negated) and P^T = S0 Q^T
        if (tid == 0) {
            const uint32_t idd = tc::idesc_bf16(128, 64, 0, 1, 1);
            const uint32_t idp = tc::idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t sa = tc::sdesc(sb + OFF_S + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                tc::mma_bf16(tm + TM_U, sa, tc::sdesc(sb + OFF_W + ks * 2048, 8192, 1024), idd, 1u);
                tc::mma_bf16(tm + TM_P, sa,
                             tc::sdesc(sb + OFF_KQ + 8192 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                             idp, ks > 0);
            }
            tc::commit(&mbar);
        }
        if (!mma_wait()) { timed_out = true; break; }

        // ---- 10. Delta^T (hi / lo) and Delta~^T = Delta^T diag(D_L rk) (hi / lo), row v = tid;
        //          the state is scaled by gamma_L in TMEM before the update accumulates onto it
        {
            float d64[64];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v16[16];
                tc::ld16(tm + lrow + TM_U + j * 16, v16);
#pragma unroll
                for (int i = 0; i < 16; ++i) d64[j * 16 + i] = v16[i];
            }
            tc::wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint4 hi, lo;
                split_bf16x8(d64 + 8 * c, hi, lo);
                *reinterpret_cast<uint4*>(sm + OFF_DL + tc::sw_chunk(tid, c, 128)) = hi;
                *reinterpret_cast<uint4*>(sm + OFF_DL + 16384 + tc::sw_chunk(tid, c, 128)) = lo;
                float x8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) x8[i] = d64[8 * c + i] * dls[8 * c + i] * rks[8 * c + i];
                split_bf16x8(x8, hi, lo);
                *reinterpret_cast<uint4*>(sm + OFF_T4 + tc::sw_chunk(tid, c, 128)) = hi;
                *reinterpret_cast<uint4*>(sm + OFF_T4 + 16384 + tc::sw_chunk(tid, c, 128)) = lo;
            }
            const float gL = gams[L - 1];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float v16[16];
                tc::ld16(tm + lrow + TM_S + j * 16, v16);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) v16[i] *= gL;
                tc::st16(tm + lrow + TM_S + j * 16, v16);
            }
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
                    tc::mma_bf16(tm + TM_MD, tc::sdesc(sb + OFF_DL + pa + ks * 32, 16, 1024),
                                 tc::sdesc(sb + OFF_M + pb + ks * 32, 16, 1024), idm, (pr | ks) != 0);
            }
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tm + TM_S, tc::sdesc(sb + OFF_T4 + part * 16384 + ks * 32, 16, 1024),
                                 tc::sdesc(sb + OFF_KQ + ks * 2048, 16384, 1024), ids, 1u);
            tc::commit(&mbar);
        }
        if (!mma_wait()) { timed_out = true; break; }

        // ---- 12. outputs o_t = gamma_t rq_t scale P_t + rq_t scale (M Delta)_t, column v = tid;
        //          the new state to bf16 for the next chunk
        {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float p16[16], m16[16];
                tc::ld16(tm + lrow + TM_P + j * 16, p16);
                tc::ld16(tm + lrow + TM_MD + j * 16, m16);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int t = j * 16 + i;
                    if (t < L) {
                        const float rq = rqs[t] * a.scale;
                        const float o = fmaf(p16[i], gams[t] * rq, m16[i] * rq);
                        a.out[static_cast<size_t>(tok0 + t) * vo_stride + h * D + tid] = f32_to_bf16_rne(o);
                    }
                }
            }
            if (c0 + C < Tn) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float v16[16];
                    tc::ld16(tm + lrow + TM_S + j * 16, v16);
                    tc::wait_ld();
                    *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw_chunk(tid, 2 * j, 128)) = pack_bf16x8(v16);
                    *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw_chunk(tid, 2 * j + 1, 128)) =
                        pack_bf16x8(v16 + 8);
                }
            }
        }
        publish();
    }

    if (timed_out) {
        if (tid == 0) atomicOr(a.status, 4);
    } else {
        // ---- scatter the final state back to its pool slot (row v = tid)
        float4* row = reinterpret_cast<float4*>(Sg + static_cast<size_t>(tid) * D);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float v16[16];
            tc::ld16(tm + lrow + TM_S + j * 16, v16);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 4; ++i)
                row[j * 4 + i] = make_float4(v16[4 * i], v16[4 * i + 1], v16[4 * i + 2], v16[4 * i + 3]);
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, TM_COLS);
}

}  // namespace gdn
