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

PrefillLayout prefill_layout(long long T, int num_seqs, int Hv) {
    PrefillLayout l;
    std::memset(&l, 0, sizeof(l));
    if (num_seqs <= 0) return l;
    auto up = [](size_t x, size_t m) { return (x + m - 1) / m * m; };
    l.cap = prefill_chunk_cap(T, num_seqs);
    l.cap2 = l.cap / 2;
    l.tab = up(static_cast<size_t>(num_seqs + 1) * 8, 16);
    l.plan = l.tab + static_cast<size_t>(l.cap) * 16;
    l.tasks = l.plan + 16;
    l.splits = l.tasks + static_cast<size_t>(num_seqs + 2 * kPfMaxSplits) * 16;
    l.scr_tab = l.splits + static_cast<size_t>(kPfMaxSplits) * 16;
    l.records = up(l.scr_tab + static_cast<size_t>(l.cap2) * 16, 1024);
    l.scr_state = l.records + static_cast<size_t>(l.cap) * Hv * static_cast<size_t>(kPfRecordBytes);
    l.bytes_min = l.scr_state;
    l.scr_rows = l.scr_state + static_cast<size_t>(kPfMaxSplits) * 3 * Hv * pf::D * pf::D * sizeof(float);
    l.bytes_full = l.scr_rows + static_cast<size_t>(l.cap2) * Hv * static_cast<size_t>(kPfScratchRowBytes);
    return l;
}

size_t prefill_workspace_bytes(long long T, int num_seqs, int Hv) { return prefill_layout(T, num_seqs, Hv).bytes_full; }

namespace {
std::atomic<int> g_nsm[kMaxDevices];  // per device: multiprocessor count (0: not read yet)

template <bool F16, bool CB>
cudaError_t set_smem_limits() {
    cudaError_t e = cudaFuncSetAttribute(gdn_prefill_kernel<F16, CB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(pf::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gdn_prefill_fixup_kernel<F16, CB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(pf::FX_SMEM));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gdn_prefill_prep_kernel<F16, CB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(CB ? pf::P_SMEM_CB : pf::P_SMEM));
}

// the three kernels of one variant
template <bool F16, bool CB>
void launch_variant(const PrefillArgs& a, const PrefillMaps& maps, bool split, cudaStream_t stream) {
    if (a.T > 0) {  // one CTA per (chunk, key head, pair of value heads) of the capacity; the ones past
                    // the last chunk exit
        const int ngrp = (a.Hv / a.Hk + pf::PH - 1) / pf::PH;
        const unsigned pgrid = static_cast<unsigned>(a.cap) * static_cast<unsigned>(a.Hk) * static_cast<unsigned>(ngrp);
        gdn_prefill_prep_kernel<F16, CB><<<pgrid, pf::PNT, CB ? pf::P_SMEM_CB : pf::P_SMEM, stream>>>(a, maps);
    }
    // one CTA per (task, value head); tasks past the schedule's count exit
    const unsigned grid = static_cast<unsigned>(a.num_seqs + 2 * a.max_splits) * static_cast<unsigned>(a.Hv);
    gdn_prefill_kernel<F16, CB><<<grid, pf::NTS, pf::SMEM_BYTES, stream>>>(a, maps);
    if (split && a.T > 0) {  // one CTA per SM, looping over the jobs (none when nothing was split)
        const unsigned fgrid = static_cast<unsigned>(a.nsm > 0 ? a.nsm : 1);
        gdn_prefill_fixup_kernel<F16, CB><<<fgrid, pf::FX_NT, pf::FX_SMEM, stream>>>(a);
    }
}
}  // namespace

cudaError_t launch_prefill(const PrefillArgs& args, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                           bool f16, bool comba) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_smem_set[dev].load(std::memory_order_acquire)) {
        e = set_smem_limits<false, false>();
        if (e != cudaSuccess) return e;
        e = set_smem_limits<true, false>();
        if (e != cudaSuccess) return e;
        e = set_smem_limits<false, true>();
        if (e != cudaSuccess) return e;
        int nsm = 0;
        e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_nsm[dev].store(nsm, std::memory_order_relaxed);
        g_smem_set[dev].store(1, std::memory_order_release);
    }
    PrefillArgs a = args;
    const PrefillLayout l = prefill_layout(a.T, a.num_seqs, a.Hv);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.cap = l.cap;
    a.cap2 = l.cap2;
    a.chunk_off = reinterpret_cast<long long*>(ws);
    a.chunk_tab = reinterpret_cast<longlong2*>(ws + l.tab);
    a.plan = reinterpret_cast<PfPlan*>(ws + l.plan);
    a.tasks = reinterpret_cast<int4*>(ws + l.tasks);
    a.splits = reinterpret_cast<int4*>(ws + l.splits);
    a.scr_tab = reinterpret_cast<longlong2*>(ws + l.scr_tab);
    a.records = ws + l.records;
    const bool split = prefill_splits(l, workspace_bytes, a.num_seqs);
    a.max_splits = split ? kPfMaxSplits : 0;
    a.scr_state = split ? reinterpret_cast<float*>(ws + l.scr_state) : nullptr;
    a.scr_rows = split ? ws + l.scr_rows : nullptr;
    a.nsm = g_nsm[dev].load(std::memory_order_relaxed);
    PrefillMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (a.T > 0) {  // with T = 0 every sequence is empty and no kernel reads the maps
        if (!encode_rows(&maps.q, a.q, a.T, a.Hk, f16) || !encode_rows(&maps.k, a.k, a.T, a.Hk, f16) ||
            !encode_rows(&maps.v, a.v, a.T, a.Hv, f16) || (comba && !encode_rows(&maps.p, a.p, a.T, a.Hk, false)))
            return cudaErrorInvalidValue;
    }
    gdn_prefill_offsets_kernel<<<1, kPfOffThreads, 0, stream>>>(a);
    if (comba) launch_variant<false, true>(a, maps, split, stream);
    else if (f16) launch_variant<true, false>(a, maps, split, stream);
    else launch_variant<false, false>(a, maps, split, stream);
    return cudaGetLastError();
}

}  // namespace gdn
