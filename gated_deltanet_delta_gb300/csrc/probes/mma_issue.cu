// mma_issue.cu -- a standalone probe of the tcgen05.mma issue cost on one SM (not part of libgdn).
//
// One CTA issues back-to-back tcgen05.mma.cta_group::1.kind::f16 instructions (bf16 operands,
// M = 128, K = 16 each, fp32 accumulate in TMEM, both operands K-major in shared memory, filled with
// zeros) from one thread, or split between one thread each of two warps (each into its own TMEM
// columns, with its own commit barrier), and reports with clock64 the cycles from the first issue
// to the last one and to the commit's arrival (second repetition of each case).  It uses only the
// library's tcgen05 wrappers.  Build and run on a GB300:
//     nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -I gated_deltanet_delta_gb300/csrc \
//          -o mma_issue gated_deltanet_delta_gb300/csrc/probes/mma_issue.cu && ./mma_issue
#include <cstdio>

#include <cuda_runtime.h>

#include "common.cuh"
#include "tcgen05.cuh"

using namespace gdn;

namespace {
constexpr int kThreads = 256;
constexpr uint32_t kSmem = 65536 + 1024;  // A (32 KB) and B (32 KB) tiles + alignment slack
__device__ unsigned long long g_cycles[4];  // per issuer: issue cycles, done cycles

// A descriptor advanced by `bytes` (16-byte units in the start-address field).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

template <int N, int NISSUE>
__global__ void __launch_bounds__(kThreads, 1) mma_issue_kernel(int nmma) {
    extern __shared__ __align__(1024) uint8_t raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(8) uint64_t done[2];
    uint8_t* sm = raw + ((1024 - (tc::smem_u32(raw) & 1023)) & 1023);
    const uint32_t sb = tc::smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 65536 / 4; i += kThreads) reinterpret_cast<uint32_t*>(sm)[i] = 0u;
    if (warp == 0) tc::tmem_alloc(&tmem_slot, 512);
    if (tid == 0) {
        tc::mbar_init(&done[0], 1);
        tc::mbar_init(&done[1], 1);
    }
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = tmem_slot;
    const uint64_t dA = tc::sdesc(sb, 16, 1024), dB = tc::sdesc(sb + 32768, 16, 1024);
    const uint32_t id = tc::idesc_bf16(128, N, 0, 0, 0);
    // issuer 0 is lane 0 of warp 0, issuer 1 lane 0 of warp 4 (columns 256 ..)
    const int me = warp == 0 ? 0 : (warp == 4 ? 1 : -1);
    for (int rep = 0; rep < 2; ++rep) {
        __syncthreads();
        if (lane == 0 && me >= 0 && me < NISSUE) {
            const long long t0 = clock64();
            const int per = nmma / NISSUE;
            for (int i = 0; i < per; ++i)
                tc::mma_bf16(tm + (NISSUE > 1 ? 256u * me : 0u), desc_add(dA, (i & 3) * 32), desc_add(dB, (i & 3) * 32),
                             id, i > 0);
            const long long t1 = clock64();
            tc::commit(&done[me]);
            tc::mbar_wait(&done[me], rep & 1, 1u << 26);  // bounded
            const long long t2 = clock64();
            if (rep == 1) {
                g_cycles[2 * me] = static_cast<unsigned long long>(t1 - t0);
                g_cycles[2 * me + 1] = static_cast<unsigned long long>(t2 - t0);
            }
        }
        __syncthreads();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tm, 512);
}

template <int N, int NISSUE>
bool run(int nmma) {
    if (cudaFuncSetAttribute(mma_issue_kernel<N, NISSUE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
        cudaSuccess)
        return false;
    const unsigned long long zero[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_cycles, zero, sizeof(zero)) != cudaSuccess) return false;
    mma_issue_kernel<N, NISSUE><<<1, kThreads, kSmem>>>(nmma);
    const cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        std::printf("error: %s\n", cudaGetErrorString(e));
        return false;
    }
    unsigned long long r[4];
    if (cudaMemcpyFromSymbol(r, g_cycles, sizeof(r)) != cudaSuccess) return false;
    const double per = nmma / NISSUE;
    std::printf("N=%3d issuers=%d mmas/issuer=%3d : issue %6llu cycles (%.1f per mma), done %6llu (%.1f per mma)",
                N, NISSUE, nmma / NISSUE, r[0], r[0] / per, r[1], r[1] / per);
    if (NISSUE > 1) std::printf(" | issuer 1: issue %llu, done %llu", r[2], r[3]);
    std::printf("\n");
    return true;
}
}  // namespace

int main() {
    const bool ok = run<16, 1>(32) && run<32, 1>(32) && run<64, 1>(32) && run<128, 1>(32) && run<256, 1>(32) &&
                    run<64, 1>(64) && run<64, 2>(64) && run<128, 2>(64) && run<256, 2>(64);
    return ok ? 0 : 1;
}
