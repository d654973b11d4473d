// window.cu -- launch of the fused decode-window kernel (kernel in window.cuh).
#include "window.cuh"
#include "launch.h"

namespace gdn {

// Two CTAs (a cluster, one per column half) per (sequence, value head).
void launch_window(const WindowArgs& a, int N, cudaStream_t stream) {
    const unsigned grid = 2u * unsigned(N) * unsigned(a.h_v);
    gdn_window_kernel<<<grid, kWinThreads, 0, stream>>>(a);
}

}  // namespace gdn
