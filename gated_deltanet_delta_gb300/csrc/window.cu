// window.cu -- launch of the fused decode-window kernel (kernel in window.cuh).
#include <atomic>

#include "launch.h"
#include "window.cuh"

namespace gdn {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_win_nsm[kMaxDevices];  // per device: multiprocessor count (0: not read yet)
constexpr long long kWinStaggerCycles = 4000;  // about 2 us (4000, 8000, 12000 measured alike)
}  // namespace

// One CTA per (sequence, value head); registers hold two per SM.  When the heads make more than
// one wave, the second slot of each SM starts kWinStaggerCycles later (see the kernel).
cudaError_t launch_window(const WindowArgs& args, int N, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int nsm = g_win_nsm[dev].load();
    if (nsm == 0) {
        e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_win_nsm[dev].store(nsm);
    }
    WindowArgs a = args;
    const long long grid = static_cast<long long>(N) * a.h_v;
    a.stagger_lo = nsm;
    a.stagger_cycles = grid > 2LL * nsm ? kWinStaggerCycles : 0;
    gdn_window_kernel<<<static_cast<unsigned>(grid), kWinThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
