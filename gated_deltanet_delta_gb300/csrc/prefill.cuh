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
// GB300 mapping: three kernels on one stream.
//   gdn_prefill_offsets_kernel (one CTA): the first chunk of every sequence (a scan of the chunk
//     counts) and a table entry per chunk (first token, sequence, length).
//   gdn_prefill_prep_kernel (one CTA of 256 threads per (chunk, key head) and up to two of its value
//     heads, five per SM): all the work that does not depend on the carried state -- row norms,
//     gates, G = [K; Q] K^T (shared by the CTA's value heads) on the
//     tensor core, Lm, the triangular inverse, Tw = T diag(beta gamma rk) and Tu = T diag(beta),
//     M~ = diag(rq scale) M (all split into bf16 high and low parts) and Q~ = diag(gamma rq scale) Q
//     -- written as one chunk record (kPfRecordBytes, laid out as the sequential kernel's
//     shared-memory image).  This is the bulk of the CUDA-core work; here every chunk of every
//     sequence runs in parallel.
//   gdn_prefill_kernel (one CTA of 16 worker warps, a control warp and a producer warp per
//     (sequence, value head)): the chunk recurrence.  The fp32 state S (V x K = 128 x 128) lives in
//     TMEM for the whole sequence and reaches HBM only at the start (gather from the pool slot) and
//     at the end (scatter back).  The control lane issues the MMAs; the producer lane takes k and v
//     rows by TMA (cp.async.bulk.tensor, 64 tokens x 64 features per box) and the parts of the
//     chunk record by bulk copies, each as soon as its buffer is free; worker threads i, i + 128,
//     i + 256 and i + 384 share TMEM lane i (each takes a quarter of the columns).
// Every contraction is a tcgen05.mma with M = 128 (the transposed forms keep V or the feature index
// on M):
//     G   = [K; Q] K^T              M=128 (64 k rows + 64 q rows), N=64,  K=128   bf16 (exact inputs)
//     W^T = K^T Tw^T,  U^T = V^T Tu^T   M=128, N=64, K=64 (x2: hi, lo)
//     Delta^T = U^T - S0 W^T,  O^T = S0 Q~^T                M=128, N=64, K=128
//     O^T += Delta^T M~^T                                   M=128, N=64, K=64 (x3: hi/lo products)
//     S += Delta~^T K            (Delta~ = diag(D_L rk) Delta)   M=128, N=128, K=64 (x2)
// Raw bf16 k and v tiles are exact MMA operands; the row scales (norms, gates, decays) are folded
// into the computed operands or applied in fp32 afterwards.  Computed operands are rounded to bf16,
// except T, Delta~, both factors of M~ Delta and S0 in P~, which are split into a bf16 high part and
// a bf16 low part (x = hi + lo, two or three MMAs): with plain bf16 there the output and the carried
// state miss their tolerances.
// fp16 inputs (q, k, v, a, b and the output in IEEE binary16, the F16 instances): an MMA takes both
// operands in one type, so the products with raw tiles (G, W/U, the state update) run on fp16
// operands, with their computed partners (Tw, Tu, Delta~) split into fp16 high and low parts; the
// other products keep bf16.  fp16 high / low parts carry about 22 bits but only fp16's range: a
// partner entry beyond 65504 in magnitude (a key row of norm below |Delta| / 65504) overflows.  The triangular inverse runs in fp32 on CUDA cores, blockwise (16 x 16
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
constexpr uint32_t kWaitLimit = 1u << 26;  // mbarrier polls before giving up (seconds of waiting)
constexpr uint32_t kSleepWaitLimit = 1u << 22;  // the same for polls with a 1 us suspend hint

// chunk record (bytes): Tw hi, Tw lo, Tu hi, Tu lo | Q~ | M~ hi, M~ lo | vectors
constexpr uint32_t REC_T4 = 0, REC_QT = 32768, REC_M = 49152, REC_VEC = 65536, REC_BYTES = 66560;
constexpr uint32_t REC_VEC_BYTES = REC_BYTES - REC_VEC;
// vector offsets (floats) inside the record's vector block
constexpr int V_DL = 0, V_RK = 64, V_GL = 128;

// the chunk-preparation kernel: CTAs of 256 threads, five per SM; its dynamic shared memory (bytes
// from a 1024-aligned base) is the [K;Q] tile, reused once G, the norms and Q~ are done for the fp32
// Lm, which the blockwise inverse turns into T in place, and the inverse's scratch
constexpr int PNT = 256;
constexpr int PH = 2;          // value heads per preparation CTA (at most)
constexpr uint32_t P_KQ = 0;          // [K;Q] tile: two 16 KB feature halves, 64 k rows + 64 q rows
constexpr uint32_t P_L = 0;           // fp32 [64][LST]: Lm, then T = (I + Lm)^-1
constexpr uint32_t P_X = P_L + 64 * LST * 4;  // fp32 [32][ZST] scratch of the blockwise inverse; before
                                               // it, M~ hi / lo staged in the record's layout (16 KB)
constexpr uint32_t P_USED = P_X + 16384;
constexpr uint32_t P_SMEM = P_USED + 1024;
// Comba: the write keys' rows (the B operand of G = [P; Q] K^T) in a tile of their own
constexpr uint32_t P_K2 = (P_USED + 1023) / 1024 * 1024;
constexpr uint32_t P_SMEM_CB = P_K2 + 16384 + 1024;
constexpr uint32_t P_TM_G = 0, P_TM_COLS = 64;
static_assert(P_X + 32 * ZST * 4 <= P_USED && P_X % 16 == 0, "Lm, T, the M~ staging and the scratch fit");

// the sequential kernel's dynamic shared memory
constexpr uint32_t OFF_K = 0;          // two K tiles (chunks of even / odd index), 16 KB each: two
                                       // 64-feature halves of 8 KB, 64 token rows each
constexpr uint32_t OFF_V = 32768;      // V tile (two halves of 8 KB)
constexpr uint32_t OFF_S = 49152;      // S0 bf16, K-major, 128 v rows, two halves of 16 KB
constexpr uint32_t OFF_T4 = 81920;     // record part: Tw hi, Tw lo, Tu hi, Tu lo
constexpr uint32_t OFF_QT = 114688;    // record part: Q~
constexpr uint32_t OFF_M = 131072;     // record part: M~ hi, M~ lo
constexpr uint32_t OFF_VEC = 147456;   // record part: the vectors, two buffers of 1 KB
constexpr uint32_t OFF_DL = OFF_VEC + 2 * REC_VEC_BYTES;  // Delta^T hi, lo (16 KB each)
constexpr uint32_t OFF_DT = OFF_DL + 32768;      // Delta~^T hi, lo (16 KB each); before them, W as
                                                 // the MN-major B operand (128 feature rows x 64 t)
constexpr uint32_t SMEM_USED = OFF_DT + 32768;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
// TMEM columns (fp32, 128 lanes): the state, W, U and the outputs O = P~ + M~ Delta, the last two
// in a buffer per chunk parity; then the low bf16 parts of S0 (S - bf16(S), two per column, the
// even feature in the low half), the A operand of P~'s second product
constexpr uint32_t TM_S = 0, TM_W = 128, TM_U = 192, TM_O = 320, TM_SL = 448;
constexpr uint32_t TM_COLS = 512;
// the sequential kernel's threads: 16 worker warps (conversions, outputs), one control warp (lane 0
// issues every MMA) and one producer warp (lane 0 issues every TMA and bulk copy)
constexpr int NW = 16, NTS = 32 * (NW + 2);
// its mbarriers: MMA completions (tcgen05.commit), worker hand-offs (one arrival per worker warp)
// and copies
enum : int {
    B_A = 0,   // P~ and Delta of a chunk computed
    B_C,       // the state update of a chunk computed
    B_O,       // O = P~ + M~ Delta of a chunk computed
    B_WU,      // W and U of a chunk computed
    R_B,       // workers: Delta converted, state scaled
    R_S,       // workers: S0 (high parts in shared memory, low parts in TMEM) of the next chunk in place
    R_D,       // workers: W of the next chunk in place
    R_Z,       // workers: the tail of a short chunk zeroed
    B_K0, B_K1, B_V, B_R1, B_QT, B_RM, B_RV0, B_RV1,
    NBAR
};

static_assert(REC_BYTES == kPfRecordBytes && REC_VEC == kPfRecordVec, "chunk record layout");
static_assert(OFF_DL % 1024 == 0 && OFF_DT % 1024 == 0 && OFF_M % 1024 == 0 && OFF_QT % 1024 == 0 &&
                  OFF_T4 % 1024 == 0, "operand tiles 1024-aligned");
static_assert(OFF_T4 + REC_QT == OFF_QT && OFF_T4 + REC_M == OFF_M && OFF_T4 + REC_VEC == OFF_VEC,
              "record parts land at their tiles");
static_assert(5 * (P_SMEM + 4096) <= 228 * 1024, "five preparation CTAs per SM");
static_assert(SMEM_BYTES <= 227 * 1024, "sequential kernel shared memory");
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
// The input element type: bf16 (F16 = false) or IEEE binary16 (F16 = true).
template <bool F16>
__device__ __forceinline__ float in_to_f32(uint16_t h) {
    if constexpr (F16) return __half2float(__ushort_as_half(h));
    else return bf16_to_f32(h);
}
template <bool F16>
__device__ __forceinline__ float4 in4_to_f32x4(uint2 p) {
    if constexpr (F16) {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&p.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&p.y));
        return make_float4(a.x, a.y, b.x, b.y);
    } else {
        return bf16x4_to_f32x4(p);
    }
}
// One output element in the input type, round to nearest even.
template <bool F16>
__device__ __forceinline__ uint16_t f32_to_in(float x) {
    if constexpr (F16) return __half_as_ushort(__float2half_rn(x));
    else return static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xffffu);
}
// 2 floats to 2 elements of the input type (round to nearest even), the first in the low half.
template <bool F16>
__device__ __forceinline__ uint32_t pack_in_x2(float lo, float hi) {
    if constexpr (F16) {
        const __half2 h2 = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h2);
    } else {
        return pack_bf16x2(lo, hi);
    }
}
// 8 floats to 8 elements of the input type (round to nearest even) in a uint4.
template <bool F16>
__device__ __forceinline__ uint4 pack_in_x8(const float* x) {
    if constexpr (F16) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h2 = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        return pack_bf16x8(x);
    }
}
// Split 8 floats into high and low parts of the input type (the operands multiplied with raw tiles).
template <bool F16>
__device__ __forceinline__ void split_in_x8(const float* x, uint4& hi, uint4& lo) {
    if constexpr (F16) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h2 = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
            const float2 hf = __half22float2(h2);
            const __half2 l2 = __floats2half2_rn(x[2 * i] - hf.x, x[2 * i + 1] - hf.y);
            hw[i] = *reinterpret_cast<const uint32_t*>(&h2);
            lw[i] = *reinterpret_cast<const uint32_t*>(&l2);
        }
        hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    } else {
        split_bf16x8(x, hi, lo);
    }
}
// The instruction descriptor of an MMA whose operands are both of the input type.
template <bool F16>
__host__ __device__ constexpr uint32_t idesc_in(int M, int N, int a_mn, int b_mn, int b_neg) {
    return F16 ? (tc::idesc_bf16(M, N, a_mn, b_mn, b_neg) & ~((1u << 7) | (1u << 10)))
               : tc::idesc_bf16(M, N, a_mn, b_mn, b_neg);
}
// A descriptor advanced by `bytes` (a multiple of 16): only the 14-bit start-address field changes,
// and addresses stay inside the 256 KB shared window, so a plain add cannot carry out of it.
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

template <bool F16>
__device__ __forceinline__ float in_sumsq8(const uint4& p) {
    const float4 a = in4_to_f32x4<F16>(make_uint2(p.x, p.y));
    const float4 b = in4_to_f32x4<F16>(make_uint2(p.z, p.w));
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
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return p + ((1024u - (tc::smem_u32(p) & 1023u)) & 1023u);
}

// ------------------------------------------------------------------------------------------------
// The first chunk of every sequence, chunk_off[n] = sum over n' < n of ceil(len_n' / 64) (0 chunks
// for a sequence whose bounds are invalid: the sequential kernel flags it), and the chunk table:
// for chunk f of sequence n, (first token, n << 32 | length), for f < cap.  One CTA.
//
// Then the sequential kernel's schedule.  Its CTAs each run one chain (a sequence, a value head),
// one CTA per SM, so a call takes about max(longest chain, chunk-steps / SMs) chunk times.  When one
// sequence is much longer than the rest, its chain sets that time while most SMs idle.  The state
// recurrence is affine per chunk, S_{c+1} = S_c A_c + B_c (A_c = gamma_L I - W^T diag(D_L rk) K,
// B_c = U^T diag(D_L rk) K), and so are the chunk's outputs in its start state.  A sequence can
// therefore be cut after n1 chunks into a first part, run as usual, and a second part, run twice
// at the same time: from a zero state (outputs O', end state B') and, with v = 0, from the identity
// (outputs F, end state P = the product of the A_c).  With S_a the first part's end state, the true
// outputs of the second part are O' + S_a F and its end state is S_a P + B'; the fix-up kernel
// forms them.  The rule: take the longest sequences in turn (at most max_splits, each at least
// kPfMinSplitChunks chunks) and cut one in half when that lowers the estimate by at least 10 %
// (the second part's two chains add n2 chunk-steps per head; the fix-up is not counted).  The tasks
// list the split sequences' chains first (they are the longest), then the other sequences in order.
// With more than kPfOffThreads sequences nothing is split.
__global__ void __launch_bounds__(kPfOffThreads) gdn_prefill_offsets_kernel(const __grid_constant__ PrefillArgs a) {
    __shared__ long long warp_tot[kPfOffThreads / 32];
    __shared__ long long carry;
    __shared__ unsigned long long cand[kPfOffThreads / 32][kPfMaxSplits + 1];
    __shared__ int top_seq[kPfMaxSplits + 1];
    __shared__ long long top_cnt[kPfMaxSplits + 1];
    __shared__ int s_nsplit, s_seq[kPfMaxSplits], s_n1[kPfMaxSplits], s_base[kPfMaxSplits];
    // up to kPfOffThreads sequences (one tile): each sequence's first chunk, first token and length
    __shared__ long long s_off[kPfOffThreads + 1], s_bos[kPfOffThreads], s_len[kPfOffThreads];
    const int num_seqs = a.num_seqs;
    const bool one_tile = num_seqs <= kPfOffThreads;
    long long my_cnt = 0;  // one tile: this thread's sequence's chunks
    const long long T = a.T, cap = a.cap;
    long long* chunk_off = a.chunk_off;
    longlong2* chunk_tab = a.chunk_tab;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < num_seqs; base += kPfOffThreads) {
        const int i = base + tid;
        long long cnt = 0, bos = 0, len = 0;
        if (i < num_seqs) {
            bos = a.cu_seqlens[i];
            const long long eos = a.cu_seqlens[i + 1];
            if (bos >= 0 && eos >= bos && eos <= T) {
                len = eos - bos;
                cnt = (len + pf::C - 1) / pf::C;
            }
        }
        long long x = cnt;  // inclusive scan inside the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(kFullMask, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            long long w = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(kFullMask, w, o);
                if (lane >= o) w += y;
            }
            warp_tot[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const long long before = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - cnt;
        if (i < num_seqs) {
            chunk_off[i] = before;
            if (one_tile) {  // the table is filled in parallel below
                s_off[i] = before;
                s_bos[i] = bos;
                s_len[i] = len;
                my_cnt = cnt;
            } else {
                for (long long j = 0; j < cnt && before + j < cap; ++j) {
                    const long long L = len - j * pf::C < pf::C ? len - j * pf::C : pf::C;
                    chunk_tab[before + j] = make_longlong2(bos + j * pf::C, (static_cast<long long>(i) << 32) | L);
                }
            }
        }
        __syncthreads();
        if (tid == 0) carry += warp_tot[kPfOffThreads / 32 - 1];
        __syncthreads();
    }
    if (tid == 0) chunk_off[num_seqs] = carry;
    if (one_tile) {
        // chunk f belongs to the last sequence whose first chunk is <= f (empty sequences share
        // their successor's first chunk and come before it)
        const long long nch = carry < cap ? carry : cap;
        for (long long f = tid; f < nch; f += kPfOffThreads) {
            int lo = 0, hi = num_seqs - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_off[mid] <= f) lo = mid;
                else hi = mid - 1;
            }
            const long long j = f - s_off[lo], len = s_len[lo];
            const long long L = len - j * pf::C < pf::C ? len - j * pf::C : pf::C;
            chunk_tab[f] = make_longlong2(s_bos[lo] + j * pf::C, (static_cast<long long>(lo) << 32) | L);
        }
    }

    // ---- the schedule: the ms + 1 longest sequences (keys chunks << 16 | 0xffff - index, unique):
    //      each warp takes its own top ms + 1 by rounds of a warp maximum, then warp 0 merges the
    //      warps' sorted lists
    const int ms = (a.max_splits > 0 && num_seqs <= kPfOffThreads)
                       ? (a.max_splits < kPfMaxSplits ? a.max_splits : kPfMaxSplits) : 0;
    if (ms > 0) {
        // (sequences of fewer than kPfMinSplitChunks chunks are never split: key 0)
        unsigned long long key = 0;
        if (tid < num_seqs && my_cnt >= kPfMinSplitChunks)
            key = (static_cast<unsigned long long>(my_cnt) << 16) | static_cast<unsigned>(0xffff - tid);
        {
            int r = 0;
            if (__any_sync(kFullMask, key != 0)) {
                for (; r <= ms; ++r) {
                    unsigned long long m = key;
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) {
                        const unsigned long long y = __shfl_xor_sync(kFullMask, m, o);
                        m = y > m ? y : m;
                    }
                    if (m == 0) break;      // the rest of the warp's list is empty
                    if (key == m) key = 0;  // taken (keys are unique)
                    if (lane == 0) cand[warp][r] = m;
                }
            }
            if (lane == 0)
                for (; r <= ms; ++r) cand[warp][r] = 0;
        }
        __syncthreads();
        if (warp == 0) {
            int ptr = 0, r = 0;
            for (; r <= ms; ++r) {
                const unsigned long long mine = ptr <= ms ? cand[lane][ptr] : 0ull;
                unsigned long long m = mine;
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    const unsigned long long y = __shfl_xor_sync(kFullMask, m, o);
                    m = y > m ? y : m;
                }
                if (m == 0) break;
                if (mine == m) ++ptr;
                if (lane == 0) {
                    top_seq[r] = 0xffff - static_cast<int>(m & 0xffffu);
                    top_cnt[r] = static_cast<long long>(m >> 16);
                }
            }
            if (lane == 0)
                for (; r <= ms; ++r) {
                    top_seq[r] = -1;
                    top_cnt[r] = 0;
                }
        }
        __syncthreads();
    }
    if (tid == 0) {
        int ns = 0;
        long long nscr = 0;
        if (ms > 0) {
            const long long Hv = a.Hv, nsm = a.nsm > 0 ? a.nsm : 1;
            long long W = Hv * carry;  // chunk-steps
            long long longest_split = 0;
            for (int j = 0; j < ms; ++j) {
                const long long cj = top_cnt[j];
                if (top_seq[j] < 0 || cj < kPfMinSplitChunks) break;
                const long long next = top_seq[j + 1] >= 0 ? top_cnt[j + 1] : 0;
                const long long n1 = (cj + 1) / 2, n2 = cj - n1;
                if (nscr + n2 > a.cap2) break;
                const long long old_b = max(max(longest_split, cj), (W + nsm - 1) / nsm);
                const long long new_b = max(max(max(longest_split, n1), next), (W + Hv * n2 + nsm - 1) / nsm);
                if (10 * new_b > 9 * old_b) break;
                s_seq[ns] = top_seq[j];
                s_n1[ns] = static_cast<int>(n1);
                s_base[ns] = static_cast<int>(nscr);
                a.splits[ns] = make_int4(top_seq[j], static_cast<int>(n1), static_cast<int>(nscr), 0);
                nscr += n2;
                W += Hv * n2;
                longest_split = max(longest_split, n1);
                ++ns;
            }
        }
        s_nsplit = ns;
        a.plan->ntask = num_seqs + 2 * ns;
        a.plan->nsplit = ns;
        a.plan->nscr = nscr;
    }
    __syncthreads();
    const int ns = s_nsplit;
    for (int i = tid; i < num_seqs; i += kPfOffThreads) {
        int k = -1, below = 0;
        for (int j = 0; j < ns; ++j) {
            if (s_seq[j] == i) k = j;
            if (s_seq[j] < i) ++below;
        }
        if (k >= 0) {
            a.tasks[3 * k] = make_int4(i, kPfFirst, k, 0);
            a.tasks[3 * k + 1] = make_int4(i, kPfZero, k, 0);
            a.tasks[3 * k + 2] = make_int4(i, kPfOper, k, 0);
        } else {
            a.tasks[3 * ns + i - below] = make_int4(i, kPfWhole, 0, 0);
        }
    }
    for (int j = 0; j < ns; ++j) {  // the scratch chunks: the second parts' chunks (one tile)
        const int n = s_seq[j];
        const long long bos = s_bos[n], len = s_len[n];
        const long long n1 = s_n1[j], cnt = (len + pf::C - 1) / pf::C;
        for (long long c = n1 + tid; c < cnt; c += kPfOffThreads) {
            const long long L = len - c * pf::C < pf::C ? len - c * pf::C : pf::C;
            a.scr_tab[s_base[j] + c - n1] = make_longlong2(bos + c * pf::C, (static_cast<long long>(j) << 32) | L);
        }
    }
}

// ------------------------------------------------------------------------------------------------
// The state-independent part of one chunk for up to two value heads of one key head -> their chunk
// records.  The heads of a key head share the k and q rows, their norms and G = [K; Q] K^T, so a
// CTA loads and multiplies them once and repeats only the gate-dependent phases per head.  CTA
// b = (f * Hk + hk) * ngrp + g is chunk f (the table gives its first token and length), key head
// hk, value heads hk * R + 2g and, when R - 2g > 1, the next (R = Hv / Hk, ngrp = ceil(R / 2)).
// CTAs of 256 threads, five per SM: the latency-bound phases of one CTA (the inverse runs 64, 128
// and 256 threads wide) overlap with those of four others.  Every part of a record is written to
// the workspace directly.
// CB (Comba, read key p != write key k; inputs pre-normalised, gates given): the rows of G are
// [P; Q] K^T (Lm from P K^T, M~ from Q K^T), the norms are 1, the log decay and beta are read as
// they are; everything after G is the same.
template <bool F16, bool CB>
__global__ void __launch_bounds__(pf::PNT, 5)
    gdn_prefill_prep_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ PrefillMaps maps) {
    using namespace pf;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(16) float Gf[PH][C], betas[PH][C], gams[PH][C], wws[PH][C], wus[PH][C];
    __shared__ __align__(16) float rks[C], rqs[C];
    __shared__ float scan_total[PH];
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(8) uint64_t mbar;    // MMA completion
    __shared__ __align__(8) uint64_t bar_kq;  // TMA of the unit's k and q rows

    const long long total = a.chunk_off[a.num_seqs] < a.cap ? a.chunk_off[a.num_seqs] : a.cap;
    const int R = a.Hv / a.Hk, ngrp = (R + PH - 1) / PH;
    const long long u = blockIdx.x;
    if (u >= total * a.Hk * ngrp) return;
    const long long f = u / (static_cast<long long>(a.Hk) * ngrp);
    const int rem = static_cast<int>(u - f * a.Hk * ngrp);
    const int hk = rem / ngrp;
    const int h0 = hk * R + PH * (rem - hk * ngrp);  // first value head of this CTA
    const int nh = R - (h0 - hk * R) < PH ? R - (h0 - hk * R) : PH;
    const longlong2 entry = a.chunk_tab[f];
    const long long tok0 = entry.x;
    const int L = static_cast<int>(entry.y & 0xffffffffLL);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = tid & 127;   // the TMEM lane this thread reads
    const int hf = tid >> 7;     // which half of the 64 G columns
    uint8_t* sm = align1024(smem_raw);
    const uint32_t sb = tc::smem_u32(sm);
    float* Ls = reinterpret_cast<float*>(sm + P_L);
    float* Xs = reinterpret_cast<float*>(sm + P_X);
    // the record of value head h0 + j
    auto record = [&](int j) { return a.records + (f * a.Hv + h0 + j) * static_cast<long long>(REC_BYTES); };

    if (warp == 0) tc::tmem_alloc(&tmem_slot, P_TM_COLS);
    if (tid == 0) {
        tc::mbar_init(&mbar, 1);
        tc::mbar_init(&bar_kq, 1);
        const int z = static_cast<int>(tok0);
        tc::mbar_expect_tx(&bar_kq, (CB ? 6 : 4) * 8192);
        const CUtensorMap* top = CB ? &maps.p : &maps.k;  // the rows above Q in the tile
        tc::tma_load_3d(sb + P_KQ, top, 0, hk, z, &bar_kq);
        tc::tma_load_3d(sb + P_KQ + 16384, top, 64, hk, z, &bar_kq);
        tc::tma_load_3d(sb + P_KQ + 8192, &maps.q, 0, hk, z, &bar_kq);
        tc::tma_load_3d(sb + P_KQ + 16384 + 8192, &maps.q, 64, hk, z, &bar_kq);
        if constexpr (CB) {
            tc::tma_load_3d(sb + P_K2, &maps.k, 0, hk, z, &bar_kq);
            tc::tma_load_3d(sb + P_K2 + 8192, &maps.k, 64, hk, z, &bar_kq);
        }
    }
    // gate inputs: thread jg * 64 + t takes token t of value head h0 + jg
    const int jg = tid >> 6, tg = tid & (C - 1);
    uint16_t a_raw = 0, b_raw = 0;
    float a_mul = 0.f, dtb = 0.f, g_in = 0.f;
    if (jg < nh) {
        if (tg < L) {
            const size_t gi = static_cast<size_t>(tok0 + tg) * a.Hv + h0 + jg;
            if constexpr (CB) {
                g_in = a.g_log[gi];
                b_raw = a.beta_in[gi];
            } else {
                a_raw = a.a[gi];
                b_raw = a.b[gi];
            }
        }
        if constexpr (!CB) {
            a_mul = expf(a.A_log[h0 + jg]);
            dtb = a.dt_bias[h0 + jg];
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = tmem_slot;
    const uint32_t trow = tm + (static_cast<uint32_t>((warp & 3) * 32) << 16);  // TMEM lane base
    bool timed_out = false;

    do {
        // ---- 1. wait for the rows, zero the rows past the sequence end, row norms
        {
            const bool ok = tid != 0 || tc::mbar_wait(&bar_kq, 0, a.wait_polls);
            if (!__syncthreads_and(ok ? 1 : 0)) {  // give the copies one more bounded wait
                if (tid == 0) tc::mbar_wait(&bar_kq, 0, kWaitLimit);
                timed_out = true;
                break;
            }
        }
        if (L < C) {
            for (int e = tid; e < (C - L) * 16; e += PNT) {
                const int s = L + (e >> 4), c = e & 15;
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sm + P_KQ + tc::sw_chunk(s, c, 128)) = z;
                *reinterpret_cast<uint4*>(sm + P_KQ + tc::sw_chunk(64 + s, c, 128)) = z;
                if constexpr (CB) *reinterpret_cast<uint4*>(sm + P_K2 + tc::sw_chunk(s, c, 64)) = z;
            }
            __syncthreads();
        }
        if constexpr (CB) {  // the keys and queries come normalised
            if (tid < C) {
                rks[tid] = 1.f;
                rqs[tid] = 1.f;
            }
        } else {
            const int rp = tid >> 4, ch = tid & 15;  // 16 threads per row, rows rp + 16 p
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int s = p * 16 + rp;
                const uint4 kv4 = *reinterpret_cast<const uint4*>(sm + P_KQ + tc::sw_chunk(s, ch, 128));
                const uint4 qv4 = *reinterpret_cast<const uint4*>(sm + P_KQ + tc::sw_chunk(64 + s, ch, 128));
                float sk = in_sumsq8<F16>(kv4), sq = in_sumsq8<F16>(qv4);
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
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();

        // ---- 2. G = [K; Q] K^T (Comba: [P; Q] K^T, K in its own tile)
        if (tid == 0) {
            const uint64_t dKQ = tc::sdesc(sb + P_KQ, 16, 1024);
            const uint64_t dK2 = tc::sdesc(sb + P_K2, 16, 1024);
            const uint32_t id = idesc_in<F16>(128, 64, 0, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t d = dadd(dKQ, (ks >> 2) * 16384 + (ks & 3) * 32);
                const uint64_t bk = CB ? dadd(dK2, (ks >> 2) * 8192 + (ks & 3) * 32) : d;
                tc::mma_bf16(tm + P_TM_G, d, bk, id, ks > 0);
            }
            tc::commit(&mbar);
        }
        // ---- 3. gates and their in-chunk cumulative sum (while G is computed), every head at once:
        //         threads jg * 64 .. jg * 64 + 63 scan value head h0 + jg
        if (jg < nh) {
            const int t = tg;
            float ell = 0.f, be = 0.f;
            if (t < L) {
                if constexpr (CB) {
                    ell = g_in;
                    be = bf16_to_f32(b_raw);
                } else {
                    const float x = in_to_f32<F16>(a_raw) + dtb;
                    const float sp = x > 20.f ? x : log1pf(__expf(x));
                    ell = -a_mul * sp;
                    be = __frcp_rn(1.f + __expf(-in_to_f32<F16>(b_raw)));
                }
            }
            float g = ell;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(kFullMask, g, o);
                if (lane >= o) g += y;
            }
            if (t == 31) scan_total[jg] = g;
            if (jg == 0) asm volatile("bar.sync 1, 64;" ::: "memory");
            else asm volatile("bar.sync 2, 64;" ::: "memory");
            if (t >= 32) g += scan_total[jg];
            Gf[jg][t] = g;
            betas[jg][t] = be;
        }
        __syncthreads();
        if (jg < nh) {
            const int t = tg;
            float* vec = reinterpret_cast<float*>(record(jg) + REC_VEC);
            gams[jg][t] = __expf(Gf[jg][t]);
            wws[jg][t] = betas[jg][t] * gams[jg][t] * rks[t];
            wus[jg][t] = betas[jg][t];
            vec[V_DL + t] = t < L ? __expf(Gf[jg][L - 1] - Gf[jg][t]) : 0.f;
            vec[V_RK + t] = rks[t];
            if (t == 0) vec[V_GL] = __expf(Gf[jg][L - 1]);
        }
        {
            const bool ok = tid != 0 || tc::mbar_wait(&mbar, 0, a.wait_polls);
            if (!__syncthreads_and(ok ? 1 : 0)) {
                if (tid == 0) tc::mbar_wait(&mbar, 0, kWaitLimit);
                timed_out = true;
                break;
            }
            tc::fence_after();
        }

        // ---- 4. Q~ = diag(gamma_t rq_t scale) Q (bf16, rows t, K-major) from the q rows, to the
        //         record of every head (before Lm takes the tile's place)
        for (int e = tid; e < nh * C * 16; e += PNT) {
            const int j = e / (C * 16), t = (e >> 4) & (C - 1), cc = e & 15;
            uint8_t* rec = record(j);
            const uint4 q8 = *reinterpret_cast<const uint4*>(sm + P_KQ + tc::sw_chunk(64 + t, cc, 128));
            const float fq = gams[j][t] * (rqs[t] * a.scale);
            const float4 x0 = in4_to_f32x4<F16>(make_uint2(q8.x, q8.y));
            const float4 x1 = in4_to_f32x4<F16>(make_uint2(q8.z, q8.w));
            const float y[8] = {x0.x * fq, x0.y * fq, x0.z * fq, x0.w * fq, x1.x * fq, x1.y * fq, x1.z * fq, x1.w * fq};
            *reinterpret_cast<uint4*>(rec + REC_QT + tc::sw_chunk(t, cc, 64)) = pack_bf16x8(y);
        }
        __syncthreads();  // the [K;Q] tile is no longer needed: Lm takes its place

        // ---- 5 .. 7 per value head (Lm, T and the scratch reuse the same shared memory)
        for (int j = 0; j < nh; ++j) {
            const float* Gfj = Gf[j];
            const float* betasj = betas[j];
            const float* wwsj = wws[j];
            const float* wusj = wus[j];
            uint8_t* recj = record(j);
            // ---- 5. Lm (lanes t < 64, fp32, in place of the tile) and M~ = diag(rq_t scale) M (lanes
            //         64 + t, bf16 hi / lo, staged in shared memory in the record's layout) from G, 32
            //         columns per thread
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int s0 = 32 * hf + 16 * qq;
                // this warp's rows are t = (row & 32) .. + 31 (of Lm or of M~): columns s0 .. s0 + 15
                // all past them are zero in both (warps 4 and 6), so that block is only written
                if (s0 >= (row & 32) + 32) {
                    if (row < C) {
#pragma unroll
                        for (int i4 = 0; i4 < 4; ++i4)
                            *reinterpret_cast<float4*>(Ls + row * LST + s0 + 4 * i4) = make_float4(0.f, 0.f, 0.f, 0.f);
                    } else {
                        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            *reinterpret_cast<uint4*>(sm + P_X + tc::sw_chunk(row - C, s0 / 8 + c, 64)) = z;
                            *reinterpret_cast<uint4*>(sm + P_X + 8192 + tc::sw_chunk(row - C, s0 / 8 + c, 64)) = z;
                        }
                    }
                    continue;
                }
                float g[16];
                tc::ld16(trow + P_TM_G + s0, g);
                tc::wait_ld();
                if (row < C) {
                    const int t = row;
                    const float bt = betasj[t] * rks[t];
                    const float Gt = Gfj[t];
#pragma unroll
                    for (int i4 = 0; i4 < 4; ++i4) {
                        const float4 r4 = *reinterpret_cast<const float4*>(rks + s0 + 4 * i4);
                        const float4 G4 = *reinterpret_cast<const float4*>(Gfj + s0 + 4 * i4);
                        const float rr[4] = {r4.x, r4.y, r4.z, r4.w}, GG[4] = {G4.x, G4.y, G4.z, G4.w};
                        float l4[4];
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const int s = s0 + 4 * i4 + w;
                            l4[w] = s < t ? bt * rr[w] * g[4 * i4 + w] * __expf(Gt - GG[w]) : 0.f;
                        }
                        *reinterpret_cast<float4*>(Ls + t * LST + s0 + 4 * i4) = make_float4(l4[0], l4[1], l4[2], l4[3]);
                    }
                } else {
                    const int t = row - C;
                    const float Gt = Gfj[t];
                    const float rt = rqs[t] * a.scale;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const float4 ra = *reinterpret_cast<const float4*>(rks + s0 + 8 * c);
                        const float4 rb = *reinterpret_cast<const float4*>(rks + s0 + 8 * c + 4);
                        const float4 Ga = *reinterpret_cast<const float4*>(Gfj + s0 + 8 * c);
                        const float4 Gb = *reinterpret_cast<const float4*>(Gfj + s0 + 8 * c + 4);
                        const float rr[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
                        const float GG[8] = {Ga.x, Ga.y, Ga.z, Ga.w, Gb.x, Gb.y, Gb.z, Gb.w};
                        float m8[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int s = s0 + c * 8 + i;
                            m8[i] = s <= t ? rt * (rr[i] * g[c * 8 + i] * __expf(Gt - GG[i])) : 0.f;
                        }
                        uint4 mh, ml;
                        split_bf16x8(m8, mh, ml);
                        const int cc = s0 / 8 + c;
                        *reinterpret_cast<uint4*>(sm + P_X + tc::sw_chunk(t, cc, 64)) = mh;
                        *reinterpret_cast<uint4*>(sm + P_X + 8192 + tc::sw_chunk(t, cc, 64)) = ml;
                    }
                }
            }
            __syncthreads();

            // M~ to the record: consecutive threads write consecutive 16-byte chunks (the scratch of the
            // inverse takes its place after the next barrier)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = tid + PNT * k;
                *reinterpret_cast<uint4*>(recj + REC_M + 16 * e) = *reinterpret_cast<const uint4*>(sm + P_X + 16 * e);
            }

            // ---- 6. T = (I + Lm)^-1 (unit lower triangular, 64 x 64, fp32), in place of Lm:
            //   A: the four 16 x 16 diagonal blocks by column-parallel forward substitution (a block's
            //      16 threads share a warp: the warp reads its blocks of Lm before writing them over);
            //   B: T_{2p+1,2p} = -T_{2p+1,2p+1} Lm_{2p+1,2p} T_{2p,2p}   (32 x 32 diagonal blocks);
            //   C: T_{[32,64),[0,32)} = -T_br Lm_bl T_tl                 (the whole matrix).
            //   B and C read a block of Lm into the scratch product before its T overwrites it; each
            //   thread takes one row and four consecutive columns (float4 operands).  The blocks above
            //   the diagonal are zero from Lm.
            if (tid < C) {
                const int blk = tid >> 4, j = tid & 15;
                float* Lb = Ls + (16 * blk) * LST + 16 * blk;
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
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 16; ++i) Lb[i * LST + j] = x[i];
            }
            __syncthreads();
            float* Zs = Xs;
            // the 64 threads of product p: warp half hB = (tid >> 5) & 1
            const int pB = tid >> 6, hB = (tid >> 5) & 1, rB = (tid >> 2) & 15, cB = 4 * (tid & 3);
            if (pB < 2) {  // X_p = Lm_{2p+1,2p} T_{2p,2p} (lane & 15 = row, columns 8 hB + 4 (lane >> 4)
                           // .. + 3; T_{2p,2p} is lower triangular, so rows k >= 8 hB only)
                const int r1 = lane & 15, c1 = 8 * hB + 4 * (lane >> 4);
                const float* Lr = Ls + (32 * pB + 16 + r1) * LST + 32 * pB;
                const float* Tc = Ls + (32 * pB) * LST + 32 * pB + c1;
                float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    if (k4 < 2 * hB) continue;
                    const float4 l = *reinterpret_cast<const float4*>(Lr + 4 * k4);
                    const float lk[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float4 t4 = *reinterpret_cast<const float4*>(Tc + (4 * k4 + w) * LST);
                        const float2 l2 = make_float2(lk[w], lk[w]);
                        a01 = __ffma2_rn(l2, make_float2(t4.x, t4.y), a01);
                        a23 = __ffma2_rn(l2, make_float2(t4.z, t4.w), a23);
                    }
                }
                *reinterpret_cast<float4*>(Zs + (16 * pB + r1) * ZST + c1) = make_float4(a01.x, a01.y, a23.x, a23.y);
            }
            __syncthreads();
            if (pB < 2) {  // T_{2p+1,2p} = -T_{2p+1,2p+1} X_p, over Lm_{2p+1,2p} (rows 8 hB .. + 7;
                           // T_{2p+1,2p+1} is lower triangular, so k <= 8 hB + 7)
                const float* Tr = Ls + (32 * pB + 16 + rB) * LST + 32 * pB + 16;
                const float* Xc = Zs + (16 * pB) * ZST + cB;
                float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    if (k4 > 2 * hB + 1) break;
                    const float4 tr = *reinterpret_cast<const float4*>(Tr + 4 * k4);
                    const float tk[4] = {tr.x, tr.y, tr.z, tr.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float4 x4 = *reinterpret_cast<const float4*>(Xc + (4 * k4 + w) * ZST);
                        const float2 l2 = make_float2(tk[w], tk[w]);
                        a01 = __ffma2_rn(l2, make_float2(x4.x, x4.y), a01);
                        a23 = __ffma2_rn(l2, make_float2(x4.z, x4.w), a23);
                    }
                }
                *reinterpret_cast<float4*>(Ls + (32 * pB + 16 + rB) * LST + 32 * pB + cB) =
                    make_float4(-a01.x, -a01.y, -a23.x, -a23.y);
            }
            __syncthreads();
            {  // Z = Lm_bl T_tl (all 256 threads: lane = row, warp = group of four columns).  T_tl is
               // lower triangular, so column group 4 warp .. + 3 takes rows k >= 4 warp only
                const int r1 = lane, c1 = 4 * warp;
                const float* Lr = Ls + (32 + r1) * LST;
                const float* Tc = Ls + c1;
                float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) {
                    if (k4 < warp) continue;
                    const float4 l = *reinterpret_cast<const float4*>(Lr + 4 * k4);
                    const float lk[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float4 t4 = *reinterpret_cast<const float4*>(Tc + (4 * k4 + w) * LST);
                        const float2 l2 = make_float2(lk[w], lk[w]);
                        a01 = __ffma2_rn(l2, make_float2(t4.x, t4.y), a01);
                        a23 = __ffma2_rn(l2, make_float2(t4.z, t4.w), a23);
                    }
                }
                *reinterpret_cast<float4*>(Zs + r1 * ZST + c1) = make_float4(a01.x, a01.y, a23.x, a23.y);
            }
            __syncthreads();
            const int rC = (tid >> 3) & 31, cC = 4 * (tid & 7);
            {  // T_bl = -T_br Z, over Lm_bl (warp = rows 4 warp .. + 3; T_br is lower triangular, so
               // the products stop at k = 4 warp + 3)
                const float* Tr = Ls + (32 + rC) * LST + 32;
                const float* Zc = Zs + cC;
                float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) {
                    if (k4 > warp) break;
                    const float4 tr = *reinterpret_cast<const float4*>(Tr + 4 * k4);
                    const float tk[4] = {tr.x, tr.y, tr.z, tr.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float4 z4 = *reinterpret_cast<const float4*>(Zc + (4 * k4 + w) * ZST);
                        const float2 l2 = make_float2(tk[w], tk[w]);
                        a01 = __ffma2_rn(l2, make_float2(z4.x, z4.y), a01);
                        a23 = __ffma2_rn(l2, make_float2(z4.z, z4.w), a23);
                    }
                }
                *reinterpret_cast<float4*>(Ls + (32 + rC) * LST + cC) = make_float4(-a01.x, -a01.y, -a23.x, -a23.y);
            }
            __syncthreads();

            // ---- 7. Tw = T diag(beta gamma rk), Tu = T diag(beta) as hi / lo parts of the input type
            //         (rows t, K-major), to the record, in warp tiles of 8 rows x 4 16-byte chunks
            //         (lane: row 8 rb + (lane >> 2), chunk 4 ch + (lane & 3); a row's 4 chunks fill
            //         whole 32-byte sectors).  T is lower triangular, so on each side the 4 tiles with
            //         ch = 1 and rb < 4 are zero.  Warp w converts (side 0 and side 1, rb 4 + w / 2,
            //         ch w % 2) and (side w / 4, rb w % 4, ch 0), and stores the zero tile
            //         (side w / 4, rb w % 4, ch 1).
            {
                const int lr = lane >> 2, lc = lane & 3;
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const int side = k < 2 ? k : warp >> 2;
                    const int rb = k < 2 ? 4 + (warp >> 1) : warp & 3;
                    const int ch = k < 2 ? warp & 1 : 0;
                    const int t = 8 * rb + lr, cc = 4 * ch + lc;
                    uint8_t* base = recj + REC_T4 + (side == 0 ? 0u : 16384u);
                    const float* wsrc = side == 0 ? wwsj : wusj;
                    const float4 ta = *reinterpret_cast<const float4*>(Ls + t * LST + cc * 8);
                    const float4 tb = *reinterpret_cast<const float4*>(Ls + t * LST + cc * 8 + 4);
                    const float4 wa = *reinterpret_cast<const float4*>(wsrc + cc * 8);
                    const float4 wb = *reinterpret_cast<const float4*>(wsrc + cc * 8 + 4);
                    const float x8[8] = {ta.x * wa.x, ta.y * wa.y, ta.z * wa.z, ta.w * wa.w,
                                         tb.x * wb.x, tb.y * wb.y, tb.z * wb.z, tb.w * wb.w};
                    uint4 th, tl;
                    split_in_x8<F16>(x8, th, tl);
                    *reinterpret_cast<uint4*>(base + tc::sw_chunk(t, cc, 64)) = th;
                    *reinterpret_cast<uint4*>(base + 8192 + tc::sw_chunk(t, cc, 64)) = tl;
                }
                {  // this warp's zero tile: side warp >> 2, rb = warp & 3, ch = 1
                    const int t = 8 * (warp & 3) + lr, cc = 4 + lc;
                    uint8_t* base = recj + REC_T4 + ((warp >> 2) == 0 ? 0u : 16384u);
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(base + tc::sw_chunk(t, cc, 64)) = z;
                    *reinterpret_cast<uint4*>(base + 8192 + tc::sw_chunk(t, cc, 64)) = z;
                }
            }
            __syncthreads();  // this head's reads of Lm, T and the scratch are done
        }
    } while (false);

    if (timed_out && tid == 0) atomicOr(a.status, 4);
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, P_TM_COLS);
}

// ------------------------------------------------------------------------------------------------
// The chunk recurrence of one (sequence, value head), from its chunk records, warp-specialized.
// Per chunk c the state path is: P~ = S0 Q~^T and Delta = U - S0 W^T (tensor core) -> Delta to
// bf16 hi / lo and the state scaled by gamma_L (workers) -> S += Delta~^T K, then O = P~ + M~ Delta
// (tensor core) -> S and the next chunk's W to bf16 (workers) -> chunk c's outputs stored by the
// workers while chunk c + 1's P~ and Delta are computed.  W and U of chunk c + 1 are multiplied
// while the workers convert Delta (U and O alternate between two TMEM buffers).  The output scales
// are folded into Q~ and M~ by the preparation kernel, so an output is one TMEM read, an in-warp
// transpose and one 16-byte store per 8 columns.  The control lane issues each MMA batch as soon as
// the workers' hand-off arrives; the producer lane issues each copy as soon as its buffer's last
// reader is done.
// CB (Comba): W from the read keys' rows (one p tile), the state update from the write keys' rows
// (one k tile: the GDN path double-buffers k because W and the update share it), and the pool
// holds each head's state as [K][V].
template <bool F16, bool CB>
__global__ void __launch_bounds__(pf::NTS, 1)
    gdn_prefill_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ PrefillMaps maps) {
    using namespace pf;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(8) uint64_t bars[NBAR];
    __shared__ volatile int abort_flag;

    const int task = blockIdx.x / a.Hv;
    const int h = blockIdx.x - task * a.Hv;
    if (task >= a.plan->ntask) return;
    const int4 tk = a.tasks[task];
    const int n = tk.x, kind = tk.y, split = tk.z;
    const int hk = h / (a.Hv / a.Hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool control = warp == NW;
    const bool producer = warp == NW + 1;
    const int row = tid & 127;   // workers: the TMEM lane this thread reads and writes
    const int qt = tid >> 7;     // workers: which quarter of the columns

    // ---- sequence bounds, pool slot and records (uniform over the CTA; bad ones are flagged and skipped)
    long long bos = a.cu_seqlens[n];
    const long long eos = a.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || eos > a.T || a.chunk_off[n + 1] > a.cap) {
        if (tid == 0) atomicOr(a.status, 2);
        return;
    }
    const long long slot = a.cache_indices[n];
    if (slot < 0 || slot >= a.pool_size) {
        if (tid == 0) atomicOr(a.status, 1);
        return;
    }
    long long Tn = eos - bos;
    long long chunk0 = a.chunk_off[n];
    // a split sequence: the first part's n1 chunks, or the second part's chunks from a zero state
    // (outputs O'^T and end state to the scratch) or from the identity with v = 0 (outputs F as bf16
    // high / low tiles, end state P); sc = the second part's first scratch chunk
    long long sc = 0;
    float* Sdst = a.state_pool + (static_cast<size_t>(slot) * a.Hv + h) * D * D;  // end state
    if (kind != kPfWhole) {
        const int4 sp = a.splits[split];
        const long long n1 = sp.y;
        sc = sp.z;
        if (kind == kPfFirst) {
            Tn = n1 * C;
        } else {
            bos += n1 * C;
            Tn -= n1 * C;
            chunk0 += n1;
        }
        Sdst = a.scr_state + ((static_cast<size_t>(split) * 3 + (kind - 1)) * a.Hv + h) * D * D;
    }
    if (Tn == 0) return;
    const long long nch = (Tn + C - 1) / C;
    auto chunk_len = [&](long long c) -> int { return static_cast<int>(Tn - c * C < C ? Tn - c * C : C); };
    const bool short_last = chunk_len(nch - 1) < C;

    uint8_t* sm = align1024(smem_raw);
    const uint32_t sb = tc::smem_u32(sm);

    if (warp == 0) tc::tmem_alloc(&tmem_slot, TM_COLS);
    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) tc::mbar_init(&bars[i], (i == R_B || i == R_S || i == R_D || i == R_Z) ? NW : 1);
        abort_flag = 0;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = tmem_slot;
    const uint32_t trow = tm + (static_cast<uint32_t>((warp & 3) * 32) << 16);  // TMEM lane base

    // control: a bounded wait on phase `parity` of barrier i; on a timeout it raises the abort flag,
    // and it gives up once someone else has
    auto wait_bar = [&](int i, uint32_t parity) -> bool {
        if (tc::mbar_wait_or_abort(&bars[i], parity, a.wait_polls, &abort_flag)) return true;
        abort_flag = 1;
        return false;
    };
    // workers: the whole warp waits, converged, parked between polls
    auto warp_wait = [&](int i, uint32_t parity) -> bool {
        bool ok = tc::mbar_sleep_wait(&bars[i], parity, a.sleep_polls, 1000u, &abort_flag);
        ok = __all_sync(kFullMask, ok ? 1 : 0) != 0;
        if (!ok && lane == 0) abort_flag = 1;
        tc::fence_after();
        return ok;
    };
    // workers: hand this warp's shared-memory and TMEM writes to the tensor core
    auto warp_arrive = [&](int i) {
        tc::wait_st();
        tc::fence_proxy_async();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bars[i]);
    };
    // operand descriptors at their tile bases (K-major: LBO unused; MN-major: LBO = half stride)
    const uint64_t dQT = tc::sdesc(sb + OFF_QT, 16, 1024);         // Q~ rows, K-major
    const uint64_t dK0 = tc::sdesc(sb + OFF_K, 8192, 1024);        // k rows read MN-major (even chunks)
    const uint64_t dVmn = tc::sdesc(sb + OFF_V, 8192, 1024);       // v rows read MN-major
    const uint64_t dS0 = tc::sdesc(sb + OFF_S, 16, 1024);          // S0, K-major
    const uint64_t dWmn = tc::sdesc(sb + OFF_DT, 8192, 1024);      // W, MN-major
    const uint64_t dT4 = tc::sdesc(sb + OFF_T4, 16, 1024);         // Tw/Tu hi/lo
    const uint64_t dDL = tc::sdesc(sb + OFF_DL, 16, 1024);         // Delta hi/lo
    const uint64_t dDT = tc::sdesc(sb + OFF_DT, 16, 1024);         // Delta~ hi/lo
    const uint64_t dM = tc::sdesc(sb + OFF_M, 16, 1024);           // M~ hi/lo
    const size_t vo_stride = static_cast<size_t>(a.Hv) * D;       // elements between tokens of v, out
    float* Sg = a.state_pool + (static_cast<size_t>(slot) * a.Hv + h) * D * D;

    // ---- workers' pieces
    // zero the k and v rows of chunk c past the sequence end (before its W and U)
    // (Comba: the p and v rows, which W and U read; the k rows, which only the update reads and
    // which land a chunk later, are zeroed by zero_tail_k before the update)
    auto zero_tail = [&](long long c) {
        const int L = chunk_len(c);
        uint8_t* kt = sm + OFF_K + (CB ? 16384 : (c & 1) * 16384);
        for (int e = tid; e < (C - L) * 16; e += NW * 32) {
            const int s = L + (e >> 4), cc = e & 15;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(kt + tc::sw_chunk(s, cc, 64)) = z;
            *reinterpret_cast<uint4*>(sm + OFF_V + tc::sw_chunk(s, cc, 64)) = z;
        }
    };
    auto zero_tail_k = [&](long long c) {  // Comba
        const int L = chunk_len(c);
        for (int e = tid; e < (C - L) * 16; e += NW * 32) {
            const int s = L + (e >> 4), cc = e & 15;
            *reinterpret_cast<uint4*>(sm + OFF_K + tc::sw_chunk(s, cc, 64)) = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // workers: the tiles W and U read of chunk c have landed (before zero_tail)
    auto wait_tiles = [&](long long c) -> bool {
        if constexpr (CB)
            return warp_wait(B_K1, c & 1) && warp_wait(B_V, c & 1);
        else
            return warp_wait(B_K0 + static_cast<int>(c & 1), (c >> 1) & 1) && warp_wait(B_V, c & 1);
    };
    // W (W^T in TMEM) -> bf16 MN-major B operand: lane f holds W[t][f], t = 16*qt ..
    auto convert_w = [&]() {
        float w16[16];
        tc::ld16(trow + TM_W + 16 * qt, w16);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < 2; ++c)
            *reinterpret_cast<uint4*>(sm + OFF_DT + tc::sw_chunk(row, 2 * qt + c, 128)) = pack_bf16x8(w16 + 8 * c);
    };
    // S (TMEM) -> S0 for the next chunk's P~ and Delta: bf16 high parts (K-major, shared memory)
    // and, for P~ only, the bf16 low parts (TMEM, feature pairs packed per column)
    auto convert_s = [&]() {
        float s32[32], lo16[16];
        ld32(trow + TM_S + 32 * qt, s32);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint4 hi, lo;
            split_bf16x8(s32 + 8 * q4, hi, lo);
            *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw_chunk(row, 4 * qt + q4, 128)) = hi;
            lo16[4 * q4] = __uint_as_float(lo.x);
            lo16[4 * q4 + 1] = __uint_as_float(lo.y);
            lo16[4 * q4 + 2] = __uint_as_float(lo.z);
            lo16[4 * q4 + 3] = __uint_as_float(lo.w);
        }
        tc::st16(trow + TM_SL + 16 * qt, lo16);
    };
    // outputs of chunk c from O (TMEM), tokens 16*qt .. (lane v)
    // Lane v holds tokens 16*qt .. 16*qt+15 of its column; an 8 x 8 transpose inside each group of
    // 8 lanes (three xor-shuffle stages) gives lane 8b + j the columns 8b .. 8b+7 (of the warp's
    // 32) of token 8s + j, stored as one 16-byte vector per set s of 8 tokens.  The second part of
    // a split sequence writes its chunk's scratch row instead: O' in fp32 (rows t, 128 columns), or
    // F as bf16 high and low K-major tiles (rows t, 128 columns), the B operand image of the fix-up
    // kernel.
    auto outputs = [&](long long c) {
        const int L = chunk_len(c);
        float o16[16];
        tc::ld16(trow + TM_O + (c & 1) * 64 + 16 * qt, o16);
        tc::wait_ld();
        uint8_t* scr = a.scr_rows + ((sc + c) * a.Hv + h) * kPfScratchRowBytes;
        const int j8 = lane & 7;
        uint16_t* o = a.out + static_cast<size_t>(bos + c * C) * vo_stride + h * D + (row - j8);
#pragma unroll
        for (int set = 0; set < 2; ++set) {
            float r[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) r[i] = o16[8 * set + i];
#pragma unroll
            for (int k = 4; k >= 1; k >>= 1) {
                const bool up = (lane & k) != 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i & k) continue;
                    const float recv = __shfl_xor_sync(kFullMask, up ? r[i] : r[i | k], k);
                    if (up) r[i] = recv;
                    else r[i | k] = recv;
                }
            }
            const int t = 16 * qt + 8 * set + j8;
            if (kind == kPfZero) {
                float4* d = reinterpret_cast<float4*>(scr + (static_cast<size_t>(t) * D + row - j8) * 4);
                d[0] = make_float4(r[0], r[1], r[2], r[3]);
                d[1] = make_float4(r[4], r[5], r[6], r[7]);
            } else if (kind == kPfOper) {
                uint4 hi, lo;
                split_bf16x8(r, hi, lo);
                *reinterpret_cast<uint4*>(scr + 32768 + tc::sw_chunk(t, (row - j8) >> 3, 64)) = hi;
                *reinterpret_cast<uint4*>(scr + 49152 + tc::sw_chunk(t, (row - j8) >> 3, 64)) = lo;
            } else if (t < L) {
                *reinterpret_cast<uint4*>(o + static_cast<size_t>(t) * vo_stride) = pack_in_x8<F16>(r);
            }
        }
    };
    // Delta^T (hi / lo) and Delta~^T = Delta^T diag(D_L rk) (hi / lo), lane v, 16 s each (over W,
    // which Delta has read); the state is scaled by gamma_L in TMEM before the update accumulates.
    // When gamma_L is 0 in fp32 (the chunk's decay underflows) the scaled state is exactly 0: the
    // pass is skipped and the update overwrites the state instead (uniform over the CTA)
    auto convert_delta = [&](long long c) {
        const float* vec = reinterpret_cast<const float*>(sm + OFF_VEC + (c & 1) * REC_VEC_BYTES);
        const float gL = vec[V_GL];
        float d16[16], sa[16], sb16[16];
        tc::ld16(trow + TM_U + (c & 1) * 64 + 16 * qt, d16);
        if (gL != 0.f) {
            tc::ld16(trow + TM_S + 32 * qt, sa);
            tc::ld16(trow + TM_S + 32 * qt + 16, sb16);
        }
        tc::wait_ld();
#pragma unroll
        for (int cc2 = 0; cc2 < 2; ++cc2) {
            const int cc = 2 * qt + cc2;
            uint4 hi, lo;
            split_bf16x8(d16 + 8 * cc2, hi, lo);
            *reinterpret_cast<uint4*>(sm + OFF_DL + tc::sw_chunk(row, cc, 128)) = hi;
            *reinterpret_cast<uint4*>(sm + OFF_DL + 16384 + tc::sw_chunk(row, cc, 128)) = lo;
            const float4 dl0 = *reinterpret_cast<const float4*>(vec + V_DL + 8 * cc);
            const float4 dl1 = *reinterpret_cast<const float4*>(vec + V_DL + 8 * cc + 4);
            const float4 rk0 = *reinterpret_cast<const float4*>(vec + V_RK + 8 * cc);
            const float4 rk1 = *reinterpret_cast<const float4*>(vec + V_RK + 8 * cc + 4);
            const float dl[8] = {dl0.x, dl0.y, dl0.z, dl0.w, dl1.x, dl1.y, dl1.z, dl1.w};
            const float rk[8] = {rk0.x, rk0.y, rk0.z, rk0.w, rk1.x, rk1.y, rk1.z, rk1.w};
            float x8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x8[i] = d16[8 * cc2 + i] * dl[i] * rk[i];
            split_in_x8<F16>(x8, hi, lo);
            *reinterpret_cast<uint4*>(sm + OFF_DT + tc::sw_chunk(row, cc, 128)) = hi;
            *reinterpret_cast<uint4*>(sm + OFF_DT + 16384 + tc::sw_chunk(row, cc, 128)) = lo;
        }
        if (gL != 0.f) {
            float lo16[16], hi16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                lo16[i] = sa[i] * gL;
                hi16[i] = sb16[i] * gL;
            }
            tc::st16(trow + TM_S + 32 * qt, lo16);
            tc::st16(trow + TM_S + 32 * qt + 16, hi16);
        }
    };

    if (control) {
        if (lane == 0) {
            // barriers with an operation of this lane in flight, and the parity of its phase (for
            // the bounded drain after an abort)
            uint32_t inflight = 0, lastpar = 0;
            auto mark = [&](int i, uint32_t parity) {
                inflight |= 1u << i;
                lastpar = (lastpar & ~(1u << i)) | (parity << i);
            };
            // W^T = K^T Tw^T and U^T = V^T Tu^T of chunk c (A MN-major from the token tiles)
            auto issue_wu = [&](long long c) {
                const uint64_t dK = dadd(dK0, CB ? 16384u : static_cast<uint32_t>(c & 1) * 16384u);  // Comba: p
                const uint32_t tu = tm + TM_U + (c & 1) * 64;
                const uint32_t idw = idesc_in<F16>(128, 64, 1, 0, 0);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        tc::mma_bf16(tm + TM_W, dadd(dK, ks * 2048), dadd(dT4, part * 8192 + ks * 32), idw,
                                     (part | ks) != 0);
                        tc::mma_bf16(tu, dadd(dVmn, ks * 2048), dadd(dT4, 16384 + part * 8192 + ks * 32), idw,
                                     (part | ks) != 0);
                    }
                tc::commit(&bars[B_WU]);
                mark(B_WU, c & 1);
            };
            // the tiles of chunk c are in place for W and U (a short chunk: after the workers zeroed
            // its tail)
            auto wu_inputs = [&](long long c) -> bool {
                if (c == nch - 1 && short_last) return wait_bar(R_Z, 0) && wait_bar(B_R1, c & 1);
                const bool tile = CB ? wait_bar(B_K1, c & 1) : wait_bar(B_K0 + static_cast<int>(c & 1), (c >> 1) & 1);
                return tile && wait_bar(B_V, c & 1) && wait_bar(B_R1, c & 1);
            };
            auto wu_ready_now = [&](long long c) -> bool {
                const bool tile = CB ? tc::mbar_test(&bars[B_K1], c & 1)
                                     : tc::mbar_test(&bars[B_K0 + static_cast<int>(c & 1)], (c >> 1) & 1);
                return !(c == nch - 1 && short_last) && tile && tc::mbar_test(&bars[B_V], c & 1) &&
                       tc::mbar_test(&bars[B_R1], c & 1);
            };

            do {
                if (!wu_inputs(0)) break;
                tc::fence_after();
                issue_wu(0);
                for (long long c = 0; c < nch; ++c) {
                    const bool more = c + 1 < nch;
                    const uint32_t par = c & 1;
                    const uint64_t dK = dadd(dK0, CB ? 0u : static_cast<uint32_t>(c & 1) * 16384u);
                    // ---- A. P~^T = S0 Q~^T once S0 is in place, as S0's high parts (shared memory)
                    //      times Q~ plus its low parts (TMEM) times Q~; then, once W is in place,
                    //      Delta^T = U^T - S0 W^T (high parts; accumulated onto U^T, B negated)
                    if (!wait_bar(R_S, par) || !wait_bar(B_QT, par)) break;
                    tc::fence_after();
                    {
                        const uint32_t id = tc::idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_bf16(tm + TM_O + (c & 1) * 64, dadd(dS0, (ks >> 2) * 16384 + (ks & 3) * 32),
                                         dadd(dQT, (ks >> 2) * 8192 + (ks & 3) * 32), id, ks > 0);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_bf16_ts(tm + TM_O + (c & 1) * 64, tm + TM_SL + 8 * ks,
                                            dadd(dQT, (ks >> 2) * 8192 + (ks & 3) * 32), id, 1u);
                    }
                    if (!wait_bar(R_D, par)) break;
                    tc::fence_after();
                    {
                        const uint32_t idd = tc::idesc_bf16(128, 64, 0, 1, 1);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_bf16(tm + TM_U + (c & 1) * 64, dadd(dS0, (ks >> 2) * 16384 + (ks & 3) * 32),
                                         dadd(dWmn, ks * 2048), idd, 1u);
                        // Comba: with p != k the chunk transition is not a contraction and the
                        // rounding of S0 grows from chunk to chunk: its low parts (TMEM) too
                        if constexpr (CB) {
#pragma unroll
                            for (int ks = 0; ks < 8; ++ks)
                                tc::mma_bf16_ts(tm + TM_U + (c & 1) * 64, tm + TM_SL + 8 * ks, dadd(dWmn, ks * 2048),
                                                idd, 1u);
                        }
                        tc::commit(&bars[B_A]);
                        mark(B_A, par);
                    }
                    // W and U of the next chunk right behind, so that they run while the workers
                    // convert Delta (their TMEM buffers were last read before R_D), if the tiles are in
                    bool wu_done = !more;
                    if (more && wu_ready_now(c + 1)) {
                        issue_wu(c + 1);
                        wu_done = true;
                    }
                    // ---- C. S += Delta~^T K, which the workers wait for, then O^T = P~^T + Delta^T M~^T
                    //      (three hi / lo products), stored by the workers while they wait for Delta
                    if (!wait_bar(R_B, par) || !wait_bar(B_RM, par)) break;
                    if (CB && !wait_bar(B_K0, par)) break;  // Comba: the update's own k tile
                    if (!wu_done && wu_ready_now(c + 1)) {
                        tc::fence_after();
                        issue_wu(c + 1);
                        wu_done = true;
                    }
                    tc::fence_after();
                    {
                        const uint32_t idm = tc::idesc_bf16(128, 64, 0, 0, 0);
                        const uint32_t ids = idesc_in<F16>(128, 128, 0, 1, 0);
                        // gamma_L == 0: the decayed state is 0 and the update overwrites it
                        const float* vec = reinterpret_cast<const float*>(sm + OFF_VEC + (c & 1) * REC_VEC_BYTES);
                        const uint32_t keep = vec[V_GL] != 0.f ? 1u : 0u;
#pragma unroll
                        for (int part = 0; part < 2; ++part)
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                tc::mma_bf16(tm + TM_S, dadd(dDT, part * 16384 + ks * 32), dadd(dK, ks * 2048), ids,
                                             (part | ks) != 0 ? 1u : keep);
                        tc::commit(&bars[B_C]);
                        mark(B_C, par);
#pragma unroll
                        for (int pr = 0; pr < 3; ++pr) {
                            const uint32_t pa = pr == 2 ? 16384u : 0u;  // Delta hi, hi, lo
                            const uint32_t pb = pr == 1 ? 8192u : 0u;   // M~ hi, lo, hi
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                tc::mma_bf16(tm + TM_O + (c & 1) * 64, dadd(dDL, pa + ks * 32), dadd(dM, pb + ks * 32),
                                             idm, 1u);
                        }
                        tc::commit(&bars[B_O]);
                        mark(B_O, par);
                    }
                    if (!wu_done) {  // the tiles came late, or the next chunk is the short last one
                        if (!wu_inputs(c + 1)) break;
                        tc::fence_after();
                        issue_wu(c + 1);
                    }
                }
            } while (false);
            if (abort_flag) {  // give what is still in flight one more bounded wait
                for (int i = 0; i < NBAR; ++i)
                    if (inflight & (1u << i)) tc::mbar_wait(&bars[i], (lastpar >> i) & 1u, 1u << 20);
            }
        }
        __syncwarp();  // the control warp reconverges before the CTA barrier
    } else if (producer) {
        // ---- producer: every copy, issued as soon as its buffer's last reader is done
        if (lane == 0) {
            // barriers with an operation of this lane in flight, and the parity of its phase (for
            // the bounded drain after an abort)
            uint32_t inflight = 0, lastpar = 0;
            auto mark = [&](int i, uint32_t parity) {
                inflight |= 1u << i;
                lastpar = (lastpar & ~(1u << i)) | (parity << i);
            };
            // k or v rows from token z on by TMA (128-byte swizzled operand layout; rows past T arrive
            // as zeros)
            auto fetch_rows = [&](const CUtensorMap* map, int head, long long z64, uint32_t dst, int bar,
                                  uint32_t parity) {
                const int z = static_cast<int>(z64);
                tc::mbar_expect_tx(&bars[bar], 2 * 8192);
                tc::tma_load_3d(sb + dst, map, 0, head, z, &bars[bar]);
                tc::tma_load_3d(sb + dst + 8192, map, 64, head, z, &bars[bar]);
                mark(bar, parity);
            };
            // a part of chunk c's record by a bulk copy
            auto fetch_rec = [&](long long c, uint32_t from, uint32_t bytes, uint32_t dst, int bar, uint32_t parity) {
                const uint8_t* rec = a.records + ((chunk0 + c) * a.Hv + h) * static_cast<long long>(REC_BYTES);
                tc::mbar_expect_tx(&bars[bar], bytes);
                tc::bulk_load(sb + dst, rec + from, bytes, &bars[bar]);
                mark(bar, parity);
            };
            auto fetch_k = [&](long long c) {  // Comba: one k tile, for the update
                if constexpr (CB)
                    fetch_rows(&maps.k, hk, bos + c * C, OFF_K, B_K0, c & 1);
                else
                    fetch_rows(&maps.k, hk, bos + c * C, OFF_K + (c & 1) * 16384, B_K0 + static_cast<int>(c & 1),
                               (c >> 1) & 1);
            };
            auto fetch_p = [&](long long c) {  // Comba: one p tile, for W
                fetch_rows(&maps.p, hk, bos + c * C, OFF_K + 16384, B_K1, c & 1);
            };
            // v = 0 for the identity-start chain: a box wholly past the last token reads as zeros
            auto fetch_v = [&](long long c) {
                fetch_rows(&maps.v, h, kind == kPfOper ? a.T : bos + c * C, OFF_V, B_V, c & 1);
            };
            auto fetch_r1 = [&](long long c) { fetch_rec(c, REC_T4, REC_QT - REC_T4, OFF_T4, B_R1, c & 1); };
            auto fetch_qt = [&](long long c) { fetch_rec(c, REC_QT, REC_M - REC_QT, OFF_QT, B_QT, c & 1); };
            auto fetch_rm = [&](long long c) { fetch_rec(c, REC_M, REC_VEC - REC_M, OFF_M, B_RM, c & 1); };
            auto fetch_rv = [&](long long c) {
                fetch_rec(c, REC_VEC, REC_VEC_BYTES, OFF_VEC + (c & 1) * REC_VEC_BYTES, B_RV0 + static_cast<int>(c & 1),
                          (c >> 1) & 1);
            };
            fetch_k(0);
            if constexpr (CB) fetch_p(0);
            fetch_v(0);
            fetch_r1(0);
            fetch_qt(0);
            fetch_rm(0);
            fetch_rv(0);
            if (!CB && nch > 1) fetch_k(1);
            do {
                if (!wait_bar(B_WU, 0)) break;
                if (nch > 1) {  // U read the v tile, W and U the record part (and Comba's W the p tile)
                    fetch_v(1);
                    fetch_r1(1);
                    if constexpr (CB) fetch_p(1);
                }
                for (long long c = 0; c < nch; ++c) {
                    const bool more = c + 1 < nch;
                    const uint32_t par = c & 1;
                    if (!wait_bar(B_A, par)) break;  // P~, issued before Delta, read Q~
                    if (more) {
                        fetch_qt(c + 1);
                        fetch_rv(c + 1);  // its buffer's last reader, chunk c - 1's Delta conversion, is done
                        if (!wait_bar(B_WU, (c + 1) & 1)) break;
                        if (c + 2 < nch) {  // U read the v tile, W and U the record part (Comba: W the p tile)
                            fetch_v(c + 2);
                            fetch_r1(c + 2);
                            if constexpr (CB) fetch_p(c + 2);
                        }
                    }
                    if (!wait_bar(B_C, par)) break;
                    if (CB ? more : c + 2 < nch) fetch_k(CB ? c + 1 : c + 2);  // the update read this k tile
                    if (!wait_bar(B_O, par)) break;
                    if (more) fetch_rm(c + 1);         // M~ Delta read M~
                }
            } while (false);
            if (abort_flag) {  // give what is still in flight one more bounded wait
                for (int i = 0; i < NBAR; ++i)
                    if (inflight & (1u << i)) tc::mbar_wait(&bars[i], (lastpar >> i) & 1u, 1u << 20);
            }
        }
        __syncwarp();  // the producer warp reconverges before the CTA barrier
    } else {
        // ---- workers
        do {
            // gather the state from its pool slot (or the zero / identity start of a split
            // sequence's second part): row v, columns 32*qt .. -> TMEM and S0 (bf16 high parts in
            // shared memory, low parts in TMEM)
            {
                const float4* src = reinterpret_cast<const float4*>(Sg + static_cast<size_t>(row) * D + 32 * qt);
                float lo16[16];
#pragma unroll
                for (int c16 = 0; c16 < 2; ++c16) {
                    float v[16];
                    if (kind <= kPfFirst && CB) {  // Comba's pool holds [K][V]: lanes read consecutive v
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = Sg[static_cast<size_t>(32 * qt + 16 * c16 + j) * D + row];
                    } else if (kind <= kPfFirst) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float4 f = src[c16 * 4 + j];
                            v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
                        }
                    } else {  // zero state, or the identity
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            v[j] = (kind == kPfOper && row == 32 * qt + 16 * c16 + j) ? 1.f : 0.f;
                    }
                    tc::st16(trow + TM_S + 32 * qt + c16 * 16, v);
                    const int c8 = 4 * qt + 2 * c16;
#pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8) {
                        uint4 hi, lo;
                        split_bf16x8(v + 8 * h8, hi, lo);
                        *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw_chunk(row, c8 + h8, 128)) = hi;
                        lo16[8 * c16 + 4 * h8] = __uint_as_float(lo.x);
                        lo16[8 * c16 + 4 * h8 + 1] = __uint_as_float(lo.y);
                        lo16[8 * c16 + 4 * h8 + 2] = __uint_as_float(lo.z);
                        lo16[8 * c16 + 4 * h8 + 3] = __uint_as_float(lo.w);
                    }
                }
                tc::st16(trow + TM_SL + 16 * qt, lo16);
            }
            warp_arrive(R_S);  // S0 of chunk 0 in place
            if (nch == 1 && short_last) {
                if (!wait_tiles(0)) break;
                zero_tail(0);
                warp_arrive(R_Z);
            }
            if (!warp_wait(B_WU, 0)) break;
            convert_w();
            warp_arrive(R_D);  // W of chunk 0 in place
            bool ok = true;
            for (long long c = 0; c < nch && ok; ++c) {
                const bool more = c + 1 < nch;
                const uint32_t par = c & 1;
                if (!warp_wait(B_A, par) || !warp_wait(B_RV0 + static_cast<int>(c & 1), (c >> 1) & 1)) { ok = false; break; }
                convert_delta(c);
                if (CB && c == nch - 1 && short_last) {  // the update's k rows past the end
                    if (!warp_wait(B_K0, c & 1)) { ok = false; break; }
                    zero_tail_k(c);
                }
                warp_arrive(R_B);
                if (!warp_wait(B_C, par)) { ok = false; break; }
                if (more) {
                    convert_s();
                    warp_arrive(R_S);
                    const long long c1 = c + 1;
                    if (c1 == nch - 1 && short_last) {
                        if (!wait_tiles(c1)) {
                            ok = false;
                            break;
                        }
                        zero_tail(c1);
                        warp_arrive(R_Z);
                    }
                    if (!warp_wait(B_WU, c1 & 1)) { ok = false; break; }
                    convert_w();
                    warp_arrive(R_D);
                }
                // chunk c's outputs, while the next chunk's P~ and Delta are computed
                if (!warp_wait(B_O, par)) { ok = false; break; }
                outputs(c);
            }
            if (!ok) break;
        } while (false);
    }

    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (abort_flag) {
        if (tid == 0) atomicOr(a.status, 4);
    } else if (warp < NW) {
        // ---- workers: scatter the final state back to its pool slot (row v, columns 32*qt ..)
        float4* dst = reinterpret_cast<float4*>(Sdst + static_cast<size_t>(row) * D + 32 * qt);
        float s32[32];
        ld32(trow + TM_S + 32 * qt, s32);
        if (CB && kind == kPfWhole) {  // Comba's pool holds [K][V]
#pragma unroll
            for (int i = 0; i < 32; ++i) Sdst[static_cast<size_t>(32 * qt + i) * D + row] = s32[i];
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(s32[4 * i], s32[4 * i + 1], s32[4 * i + 2], s32[4 * i + 3]);
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, TM_COLS);
}

// ------------------------------------------------------------------------------------------------
// The fix-up of split sequences (the rule and the algebra are described at the offsets kernel).
// State jobs (the first max_splits CTAs of each head's column): for a split and a value head, the
// end state S_a P + B' written to the pool slot (two 128 x 64 x 128 products, P read MN-major).
// Chunk jobs: G consecutive scratch chunks of one split and value head, out[t] = O'[t] + S_a F[t]
// for the chunks' tokens, one 128 x 64 x 128 product per chunk with S_a and F as bf16 high + low
// parts (hi hi + hi lo + lo hi: about 16 bits, so the one rounding that counts is the output's).
// G is the smallest chunk count (at least 2) whose jobs, with the state jobs, fit one per CTA of
// a grid of one CTA per SM (each holds 226 KB of shared memory), which loops over the jobs if they
// do not fit.  A chunk job streams: its control lane keeps F three chunks ahead in a ring of four shared-memory
// buffers (bulk copies) and issues each chunk's products into one of two TMEM buffers as soon as
// that buffer has been read; eight output warps (TMEM lane = row v, two column halves) copy the
// product tile into shared memory as [t][v], then add O' (token-major, read one chunk ahead) and
// store the outputs row by row, coalesced, so the copies, the products and the stores of
// different chunks overlap.
namespace pf {
constexpr int FX_NW = 8;                       // output warps; the control warp is warp FX_NW
constexpr int FX_NT = 32 * (FX_NW + 1);
constexpr int FX_RING = 3;                     // F buffers
constexpr uint32_t FX_A = 0;                   // S_a hi, lo: 128 rows v x 128 columns, K-major, 32 KB each
constexpr uint32_t FX_B = 65536;               // ring of B buffers (hi, lo: 16 KB each)
constexpr uint32_t FX_O = FX_B + FX_RING * 32768;  // two O' buffers, fp32 [64 t][128 v]
constexpr uint32_t FX_USED = FX_O + 2 * 32768;
constexpr uint32_t FX_SMEM = FX_USED + 1024;   // + alignment slack
constexpr uint32_t FX_COLS = 128;              // two 64-column product buffers
}  // namespace pf

template <bool F16, bool CB>
__global__ void __launch_bounds__(pf::FX_NT, 1) gdn_prefill_fixup_kernel(const __grid_constant__ PrefillArgs a) {
    using namespace pf;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot;
    // F_FULL + s: F in ring buffer s; MMA_DONE + b: products in TMEM buffer b done; D_FREE + b:
    // TMEM buffer b read by the output warps; O_FULL + b: O' in buffer b; O_FREE + b: O' buffer b
    // read by the output warps
    enum { F_FULL = 0, MMA_DONE = FX_RING, D_FREE = FX_RING + 2, O_FULL = FX_RING + 4, O_FREE = FX_RING + 6,
           FX_NBAR = FX_RING + 8 };
    __shared__ __align__(8) uint64_t bars[FX_NBAR];
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = tid & 127, half = (tid >> 7) & 1;  // output warps
    const bool control = warp == FX_NW;
    const int nsplit = a.plan->nsplit;
    const long long nscr = a.plan->nscr;
    if (nsplit == 0) return;

    // jobs per value head: nsplit state jobs, then the chunk jobs of every split, G chunks each;
    // G is the smallest (at least 2) whose jobs fit one per CTA of the grid, else the longest part
    long long G = (nscr * a.Hv + gridDim.x - 1) / gridDim.x, longest = 0, J = 0;
    G = G < 2 ? 2 : G;
    for (int sp = 0; sp < nsplit; ++sp) {
        const long long n2 = (sp + 1 < nsplit ? a.splits[sp + 1].z : nscr) - a.splits[sp].z;
        longest = n2 > longest ? n2 : longest;
    }
    for (;; ++G) {
        J = nsplit;
        for (int sp = 0; sp < nsplit; ++sp)
            J += ((sp + 1 < nsplit ? a.splits[sp + 1].z : nscr) - a.splits[sp].z + G - 1) / G;
        if (J * a.Hv <= gridDim.x || G >= longest) break;
    }
    const long long total = J * a.Hv;
    if (static_cast<long long>(blockIdx.x) >= total) return;

    uint8_t* sm = align1024(smem_raw);
    const uint32_t sb = tc::smem_u32(sm);
    if (warp == 0) tc::tmem_alloc(&tmem_slot, FX_COLS);
    if (tid == 0) abort_flag = 0;
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = tmem_slot;
    int h = 0, split = -1;
    bool state_job = false;
    long long c0 = 0, c1 = 0;
    const uint32_t trow = tm + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint64_t dAh = tc::sdesc(sb + FX_A, 16, 1024), dAl = tc::sdesc(sb + FX_A + 32768, 16, 1024);
    const size_t DD = static_cast<size_t>(D) * D;
    auto state_of = [&](int which) -> const float* {
        return a.scr_state + (static_cast<size_t>(split) * 3 + which) * a.Hv * DD + static_cast<size_t>(h) * DD;
    };
    // output warps: 128 rows of fp32, nc columns from col0 per thread, to bf16 high / low 128-byte
    // swizzled tiles of 128 rows; the thread's first 16-byte chunk is c8_0
    auto convert_rows = [&](const float* src, int col0, int c8_0, uint32_t dst_hi, uint32_t dst_lo, int nc) {
        const float4* s4 = reinterpret_cast<const float4*>(src + static_cast<size_t>(row) * D + col0);
#pragma unroll 4
        for (int cc = 0; cc < nc / 8; ++cc) {
            const float4 x0 = s4[2 * cc], x1 = s4[2 * cc + 1];
            const float v8[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            uint4 hi, lo;
            split_bf16x8(v8, hi, lo);
            *reinterpret_cast<uint4*>(sm + dst_hi + tc::sw_chunk(row, c8_0 + cc, 128)) = hi;
            *reinterpret_cast<uint4*>(sm + dst_lo + tc::sw_chunk(row, c8_0 + cc, 128)) = lo;
        }
    };
    // control: TMEM buffer b = S_a times ring buffer s, as hi hi + hi lo + lo hi; B K-major (F: 64
    // rows t, 128 columns) or MN-major (P: 128 rows k', 64 columns, one swizzle span: no leading
    // offset), committed to MMA_DONE + b
    auto products = [&](int b, int s, bool b_mn) {
        const uint32_t base = sb + FX_B + 32768u * s;
        const uint64_t Bh = b_mn ? tc::sdesc(base, 16384, 1024) : tc::sdesc(base, 16, 1024);
        const uint64_t Bl = b_mn ? tc::sdesc(base + 16384, 16384, 1024) : tc::sdesc(base + 16384, 16, 1024);
        const uint32_t id = tc::idesc_bf16(128, 64, 0, b_mn ? 1 : 0, 0);
        const uint64_t A[3] = {dAh, dAh, dAl};
        const uint64_t B[3] = {Bh, Bl, Bh};
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t ao = (ks >> 2) * 16384 + (ks & 3) * 32;
                const uint32_t bo = b_mn ? ks * 2048 : (ks >> 2) * 8192 + (ks & 3) * 32;
                tc::mma_bf16(tm + 64 * b, dadd(A[p], ao), dadd(B[p], bo), id, (p | ks) != 0);
            }
        tc::commit(&bars[MMA_DONE + b]);
    };
    auto ctl_wait = [&](int i, uint32_t parity) -> bool {
        if (tc::mbar_wait_or_abort(&bars[i], parity, kWaitLimit, &abort_flag)) return true;
        abort_flag = 1;
        return false;
    };
    auto warp_wait = [&](int i, uint32_t parity) -> bool {
        bool ok = tc::mbar_sleep_wait(&bars[i], parity, kSleepWaitLimit, 1000u, &abort_flag);
        ok = __all_sync(kFullMask, ok ? 1 : 0) != 0;
        if (!ok && lane == 0) abort_flag = 1;
        tc::fence_after();
        return ok;
    };
    // output warps: TMEM buffer b, this thread's 32 columns; then hand the buffer back
    auto ld_d = [&](int b, float (&d)[32], bool release) {
        float x[16], y[16];
        tc::ld16(trow + 64 * b + 32 * half, x);
        tc::ld16(trow + 64 * b + 32 * half + 16, y);
        tc::wait_ld();
        if (release) {
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[D_FREE + b]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            d[i] = x[i];
            d[16 + i] = y[i];
        }
    };

    for (long long job = blockIdx.x; job < total && !abort_flag; job += gridDim.x) {
    h = static_cast<int>(job / J);
    {
        long long r = job - static_cast<long long>(h) * J;
        state_job = r < nsplit;
        split = -1;
        if (state_job) {
            split = static_cast<int>(r);
        } else {
            r -= nsplit;
            for (int sp = 0; sp < nsplit; ++sp) {
                const long long base = a.splits[sp].z;
                const long long top = sp + 1 < nsplit ? a.splits[sp + 1].z : nscr;
                const long long ng = (top - base + G - 1) / G;
                if (r < ng) {
                    split = sp;
                    c0 = base + r * G;
                    c1 = c0 + G < top ? c0 + G : top;
                    break;
                }
                r -= ng;
            }
        }
    }
    const long long slot = split < 0 ? -1 : a.cache_indices[a.splits[split].x];
    if (slot < 0 || slot >= a.pool_size) continue;  // the sequential kernel flagged and skipped it
    const int n = static_cast<int>(c1 - c0);
    // fresh barriers for every job (everything of the previous job has completed)
    if (tid == 0)
        for (int i = 0; i < FX_NBAR; ++i) {
            if (job != blockIdx.x)
                asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(&bars[i])) : "memory");
            tc::mbar_init(&bars[i], ((i >= D_FREE && i < O_FULL) || i >= O_FREE) ? FX_NW : 1);
        }
    __syncthreads();

    if (!control) convert_rows(state_of(0), 64 * half, 8 * half, FX_A, FX_A + 32768, 64);  // S_a -> A
    if (state_job) {
        // P's columns 64j .. 64j+63 -> MN-major B in ring buffer j (rows k', 64 columns; 32 per
        // thread), both products at once
        if (!control)
            for (int j = 0; j < 2; ++j)
                convert_rows(state_of(2), 64 * j + 32 * half, 4 * half, FX_B + 32768u * j, FX_B + 32768u * j + 16384, 32);
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        if (control) {
            if (lane == 0) {
                tc::fence_after();
                products(0, 0, true);
                products(1, 1, true);
            }
            __syncwarp();
        } else {
            float* Sdst = a.state_pool + (static_cast<size_t>(slot) * a.Hv + h) * DD;
            float4* Sdst4 = reinterpret_cast<float4*>(Sdst);
            const float4* Bz4 = reinterpret_cast<const float4*>(state_of(1));
            for (int j = 0; j < 2; ++j) {
                if (!warp_wait(MMA_DONE + j, 0)) break;
                float d[32];
                ld_d(j, d, false);
                const size_t o4 = (static_cast<size_t>(row) * D + 64 * j + 32 * half) / 4;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 b0 = Bz4[o4 + i];
                    const float4 r = make_float4(d[4 * i] + b0.x, d[4 * i + 1] + b0.y, d[4 * i + 2] + b0.z,
                                                 d[4 * i + 3] + b0.w);
                    if constexpr (CB) {  // Comba's pool holds [K][V]: column k of row v
                        const size_t k0 = 64 * j + 32 * half + 4 * i;
                        Sdst[(k0 + 0) * D + row] = r.x;
                        Sdst[(k0 + 1) * D + row] = r.y;
                        Sdst[(k0 + 2) * D + row] = r.z;
                        Sdst[(k0 + 3) * D + row] = r.w;
                    } else {
                        Sdst4[o4 + i] = r;
                    }
                }
            }
        }
    } else if (control) {
        // F of chunk c0 + i -> ring buffer i % FX_RING; O' of chunk c0 + i -> O' buffer i % 2
        auto fetch_f = [&](int i) {
            const int s = i % FX_RING;
            const uint8_t* src = a.scr_rows + ((c0 + i) * a.Hv + h) * kPfScratchRowBytes + 32768;
            tc::mbar_expect_tx(&bars[F_FULL + s], 32768);
            tc::bulk_load(sb + FX_B + 32768u * s, src, 32768, &bars[F_FULL + s]);
        };
        auto fetch_o = [&](int i) {
            const int s = i & 1;
            const uint8_t* src = a.scr_rows + ((c0 + i) * a.Hv + h) * kPfScratchRowBytes;
            tc::mbar_expect_tx(&bars[O_FULL + s], 32768);
            tc::bulk_load(sb + FX_O + 32768u * s, src, 32768, &bars[O_FULL + s]);
        };
        // barriers with a copy or a product of this lane in flight, and the parity of the last
        // phase issued on each (for the bounded drain after a give-up)
        uint32_t inflight = 0, lastpar = 0;
        auto mark = [&](int i, uint32_t parity) {
            inflight |= 1u << i;
            lastpar = (lastpar & ~(1u << i)) | (parity << i);
        };
        if (lane == 0) {
            for (int i = 0; i < n && i < FX_RING; ++i) {
                fetch_f(i);
                mark(F_FULL + i % FX_RING, (i / FX_RING) & 1);
            }
            for (int i = 0; i < n && i < 2; ++i) {
                fetch_o(i);
                mark(O_FULL + (i & 1), (i >> 1) & 1);
            }
        }
        __syncwarp();
        tc::fence_before();
        __syncthreads();  // A is in place
        if (lane == 0) {
            for (int i = 0; i < n; ++i) {
                const int s = i % FX_RING, b = i & 1;
                if (!ctl_wait(F_FULL + s, (i / FX_RING) & 1)) break;
                if (i >= 2 && !ctl_wait(D_FREE + b, ((i - 2) >> 1) & 1)) break;
                tc::fence_after();
                products(b, s, false);
                mark(MMA_DONE + b, (i >> 1) & 1);
                if (i >= 1) {
                    // the F buffer of chunk i - 1 once its products are done, and the O' buffer of
                    // chunk i - 1 once the output warps have read it
                    if (i - 1 + FX_RING < n) {
                        if (!ctl_wait(MMA_DONE + ((i - 1) & 1), ((i - 1) >> 1) & 1)) break;
                        fetch_f(i - 1 + FX_RING);
                        mark(F_FULL + (i - 1 + FX_RING) % FX_RING, ((i - 1 + FX_RING) / FX_RING) & 1);
                    }
                    if (i + 1 < n) {
                        if (!ctl_wait(O_FREE + ((i - 1) & 1), ((i - 1) >> 1) & 1)) break;
                        fetch_o(i + 1);
                        mark(O_FULL + ((i + 1) & 1), ((i + 1) >> 1) & 1);
                    }
                }
            }
            if (abort_flag) {  // one more bounded wait on the last phase of every barrier with a copy
                               // or a product in flight
                for (int i = 0; i < FX_NBAR; ++i)
                    if (inflight & (1u << i)) tc::mbar_wait(&bars[i], (lastpar >> i) & 1u, 1u << 20);
            }
        }
        __syncwarp();
    } else {
        tc::fence_proxy_async();  // A (generic-proxy writes) before the tensor core reads it
        tc::fence_before();
        __syncthreads();
        // every output warp runs every iteration (the named barrier needs all eight); after a
        // failed wait a warp only keeps the barrier count
        bool good = true;
        for (int i = 0; i < n; ++i) {
            const int b = i & 1;
            good = good && warp_wait(MMA_DONE + b, (i >> 1) & 1);
            float d[32];
            if (good) ld_d(b, d, true);
            good = good && warp_wait(O_FULL + b, (i >> 1) & 1);
            // the products added into O' (buffer b, [t][v]: lanes are consecutive v, no bank conflict)
            float* ob = reinterpret_cast<float*>(sm + FX_O + 32768u * b);
            if (good) {
#pragma unroll
                for (int k = 0; k < 32; ++k) ob[(32 * half + k) * D + row] += d[k];
            }
            asm volatile("bar.sync 1, %0;" ::"n"(32 * FX_NW) : "memory");
            if (!good) continue;
            // unit u = tid + 256 k (k < 8): token u >> 5, columns 4 (u & 31) .. + 3, stored coalesced
            const longlong2 e = a.scr_tab[c0 + i];
            const int L = static_cast<int>(e.y & 0xffffffffLL);
            uint16_t* o = a.out + static_cast<size_t>(e.x) * a.Hv * D + static_cast<size_t>(h) * D;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int u = tid + 256 * k, t = u >> 5, c4 = u & 31;
                const float4 p = *reinterpret_cast<const float4*>(ob + t * D + 4 * c4);
                if (t < L)
                    *reinterpret_cast<uint2*>(o + static_cast<size_t>(t) * a.Hv * D + 4 * c4) =
                        make_uint2(pack_in_x2<F16>(p.x, p.y), pack_in_x2<F16>(p.z, p.w));
            }
            tc::fence_proxy_async();  // the buffer is refilled by a bulk copy next
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[O_FREE + b]);
        }
    }
    tc::fence_before();
    __syncthreads();  // the job is done: its copies, products and TMEM reads have completed
    tc::fence_after();
    }
    if (abort_flag && tid == 0) atomicOr(a.status, 4);
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, FX_COLS);
}

}  // namespace gdn
