// window.cu -- launch of the fused decode-window kernel (kernel in window.cuh).
#include "window.cuh"
#include "launch.h"

namespace gdn {

// One CTA per (sequence, value head); registers hold two per SM.
cudaError_t launch_window(const WindowArgs& a, int N, cudaStream_t stream) {
    const unsigned grid = unsigned(N) * unsigned(a.h_v);
    gdn_window_kernel<<<grid, kWinThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
