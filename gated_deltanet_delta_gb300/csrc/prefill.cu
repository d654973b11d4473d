// prefill.cu -- launch of the chunkwise-WY prefill kernel (kernel in prefill.cuh).
#include <atomic>

#include "launch.h"
#include "prefill.cuh"

namespace gdn {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_smem_set[kMaxDevices];  // per device: dynamic shared memory limit raised
}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_smem_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(gdn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(pf::SMEM_BYTES));
        if (e != cudaSuccess) return e;
        g_smem_set[dev].store(1, std::memory_order_release);
    }
    const unsigned grid = static_cast<unsigned>(a.num_seqs) * static_cast<unsigned>(a.Hv);
    gdn_prefill_kernel<<<grid, pf::NT, pf::SMEM_BYTES, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
