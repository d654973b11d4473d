// comba.cu -- launch configurations of the Comba decode kernel (kernel in comba.cuh).
#include "comba.cuh"
#include "comba_forward.cuh"
#include "launch.h"

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

// The same tile for the T-token recurrence, one CTA per head.
void launch_comba_forward(const CombaFwdArgs& a, int heads, int K, int V, cudaStream_t stream) {
    const unsigned grid = unsigned(heads);
    if (K == 128 && V == 128)
        comba_forward_kernel<128, 128, 256><<<grid, 256, 0, stream>>>(a);
    else if (K == 64 && V == 128)
        comba_forward_kernel<64, 128, 256><<<grid, 256, 0, stream>>>(a);
    else if (K == 128 && V == 64)
        comba_forward_kernel<128, 64, 256><<<grid, 256, 0, stream>>>(a);
    else
        comba_forward_kernel<64, 64, 256><<<grid, 256, 0, stream>>>(a);
}

}  // namespace gdn
