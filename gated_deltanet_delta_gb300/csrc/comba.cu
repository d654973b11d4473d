// comba.cu -- launch configurations of the Comba decode kernel (kernel in comba.cuh).
#include "comba.cuh"
#include "comba_forward.cuh"
#include "launch.h"

#include <atomic>

namespace gdn {

// One CTA of 256 threads per (b, h) head holds the head's K x V slab in registers.
void launch_comba(const CombaArgs& a, int heads, int K, int V, cudaStream_t stream) {
    const unsigned grid = unsigned(heads);
    if (K == 128 && V == 128)
        comba_decode_kernel<128, 128, 256><<<grid, 256, 0, stream>>>(a);
    else if (K == 64 && V == 128)
        comba_decode_kernel<64, 128, 256><<<grid, 256, 0, stream>>>(a);
    else if (K == 128 && V == 64)
        comba_decode_kernel<128, 64, 256><<<grid, 256, 0, stream>>>(a);
    else
        comba_decode_kernel<64, 64, 256><<<grid, 256, 0, stream>>>(a);
}

// The same tile for the T-token recurrence (chunked, see comba_forward.cuh), one CTA per head; the
// kernel's shared memory (the chunk's vectors and the reduction over K) exceeds the default 48 KB.
namespace {
std::atomic<int> g_fwd_attr[64];  // per device: dynamic shared-memory limits raised

template <int K, int V>
cudaError_t set_forward_limit() {
    return cudaFuncSetAttribute(comba_forward_kernel<K, V, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                comba_forward_smem<K, V, 256>());
}
template <int K, int V>
void run_forward(const CombaFwdArgs& a, int heads, cudaStream_t stream) {
    comba_forward_kernel<K, V, 256><<<unsigned(heads), 256, comba_forward_smem<K, V, 256>(), stream>>>(a);
}
}  // namespace

void launch_comba_forward(const CombaFwdArgs& a, int heads, int K, int V, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (!g_fwd_attr[dev].load(std::memory_order_acquire)) {
        if (set_forward_limit<128, 128>() != cudaSuccess || set_forward_limit<64, 128>() != cudaSuccess ||
            set_forward_limit<128, 64>() != cudaSuccess || set_forward_limit<64, 64>() != cudaSuccess)
            return;  // the launch below then fails and the caller reads the error
        g_fwd_attr[dev].store(1, std::memory_order_release);
    }
    if (K == 128 && V == 128)
        run_forward<128, 128>(a, heads, stream);
    else if (K == 64 && V == 128)
        run_forward<64, 128>(a, heads, stream);
    else if (K == 128 && V == 64)
        run_forward<128, 64>(a, heads, stream);
    else
        run_forward<64, 64>(a, heads, stream);
}

}  // namespace gdn
