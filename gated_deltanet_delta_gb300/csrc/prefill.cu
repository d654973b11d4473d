// prefill.cu -- launch of the chunkwise-WY prefill (kernels in prefill.cuh): the workspace layout, the
// TMA descriptors of q, k, v and the per-device shared-memory limits.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "prefill.cuh"

namespace gdn {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_smem_set[kMaxDevices];  // per device: dynamic shared memory limits raised

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

// [T, H, 128] bf16 or fp16, boxes of 64 features x 1 head x 64 tokens, 128-byte swizzle, zero fill
// past T.
bool encode_rows(CUtensorMap* map, const void* base, long long T, int H, bool f16) {
    const auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[2] = {128 * 2, static_cast<cuuint64_t>(H) * 128 * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

long long prefill_chunk_cap(long long T, int num_seqs) { return (T + pf::C - 1) / pf::C + num_seqs; }

size_t prefill_workspace_bytes(long long T, int num_seqs, int Hv) {
    if (num_seqs <= 0) return 0;
    const long long cap = prefill_chunk_cap(T, num_seqs);
    return prefill_header_bytes(num_seqs, cap) + static_cast<size_t>(cap) * Hv * static_cast<size_t>(kPfRecordBytes);
}

namespace {
template <bool F16>
cudaError_t set_smem_limits() {
    cudaError_t e = cudaFuncSetAttribute(gdn_prefill_kernel<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(pf::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gdn_prefill_prep_kernel<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(pf::P_SMEM));
}
}  // namespace

cudaError_t launch_prefill(const PrefillArgs& args, void* workspace, cudaStream_t stream, bool f16) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_smem_set[dev].load(std::memory_order_acquire)) {
        e = set_smem_limits<false>();
        if (e != cudaSuccess) return e;
        e = set_smem_limits<true>();
        if (e != cudaSuccess) return e;
        g_smem_set[dev].store(1, std::memory_order_release);
    }
    PrefillArgs a = args;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.cap = prefill_chunk_cap(a.T, a.num_seqs);
    a.chunk_off = reinterpret_cast<long long*>(ws);
    a.chunk_tab = reinterpret_cast<longlong2*>(ws + prefill_tab_offset(a.num_seqs));
    a.records = ws + prefill_header_bytes(a.num_seqs, a.cap);
    PrefillMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (a.T > 0) {  // with T = 0 every sequence is empty and no kernel reads the maps
        if (!encode_rows(&maps.q, a.q, a.T, a.Hk, f16) || !encode_rows(&maps.k, a.k, a.T, a.Hk, f16) ||
            !encode_rows(&maps.v, a.v, a.T, a.Hv, f16))
            return cudaErrorInvalidValue;
    }
    gdn_prefill_offsets_kernel<<<1, kPfOffThreads, 0, stream>>>(a.cu_seqlens, a.num_seqs, a.T, a.cap, a.chunk_off,
                                                                a.chunk_tab);
    if (a.T > 0) {  // one CTA per (chunk, key head, pair of value heads) of the capacity; the ones past
                    // the last chunk exit
        const int ngrp = (a.Hv / a.Hk + pf::PH - 1) / pf::PH;
        const unsigned pgrid = static_cast<unsigned>(a.cap) * static_cast<unsigned>(a.Hk) * static_cast<unsigned>(ngrp);
        if (f16) gdn_prefill_prep_kernel<true><<<pgrid, pf::PNT, pf::P_SMEM, stream>>>(a, maps);
        else gdn_prefill_prep_kernel<false><<<pgrid, pf::PNT, pf::P_SMEM, stream>>>(a, maps);
    }
    const unsigned grid = static_cast<unsigned>(a.num_seqs) * static_cast<unsigned>(a.Hv);
    if (f16) gdn_prefill_kernel<true><<<grid, pf::NTS, pf::SMEM_BYTES, stream>>>(a, maps);
    else gdn_prefill_kernel<false><<<grid, pf::NTS, pf::SMEM_BYTES, stream>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace gdn
