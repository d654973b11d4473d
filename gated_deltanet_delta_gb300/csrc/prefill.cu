// prefill.cu -- launch of the chunkwise-WY prefill kernel (kernel in prefill.cuh): TMA descriptors of
// q, k, v and the per-device shared-memory limit.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "prefill.cuh"

namespace gdn {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_smem_set[kMaxDevices];  // per device: dynamic shared memory limit raised

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [T, H, 128] bf16, boxes of 64 features x 1 head x 64 tokens, 128-byte swizzle, zero fill past T.
bool encode_rows(CUtensorMap* map, const void* base, long long T, int H) {
    const auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[2] = {128 * 2, static_cast<cuuint64_t>(H) * 128 * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
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
    PrefillMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (a.T > 0) {  // with T = 0 every sequence is empty and the kernel never reads the maps
        if (!encode_rows(&maps.q, a.q, a.T, a.Hk) || !encode_rows(&maps.k, a.k, a.T, a.Hk) ||
            !encode_rows(&maps.v, a.v, a.T, a.Hv))
            return cudaErrorInvalidValue;
    }
    const unsigned grid = static_cast<unsigned>(a.num_seqs) * static_cast<unsigned>(a.Hv);
    gdn_prefill_kernel<<<grid, pf::NT, pf::SMEM_BYTES, stream>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace gdn
