// launch.h -- internal launchers, one per operation, called by the C ABI (api.cu) after it has
// validated the arguments.  Each picks the kernel configuration for the shape and launches it on
// `stream`; the caller checks cudaGetLastError().
#pragma once

#include <cuda_runtime.h>

#include "kernel_args.h"

namespace gdn {

void launch_decode(DecodeArgs a, int B, int Dk, cudaStream_t stream);
void launch_decode_multi(DecodeMultiArgs a, int B, int Dk, cudaStream_t stream);
void launch_comba(const CombaArgs& a, int heads, int K, int V, cudaStream_t stream);
void launch_window(const WindowArgs& a, int N, cudaStream_t stream);
// Raises the kernel's shared-memory limit once per device, then launches; returns the launch error.
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

}  // namespace gdn
