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
void launch_comba_forward(const CombaFwdArgs& a, int heads, int K, int V, cudaStream_t stream);
cudaError_t launch_window(const WindowArgs& a, int N, cudaStream_t stream);
// Raises the kernel's shared-memory limit once per device, then launches; returns the launch error.
// The prefill workspace: the chunk offsets (8 bytes per sequence + 1, padded to 16 bytes) and the
// chunk table (16 bytes per chunk), together padded to 1 KB, then one kPfRecordBytes record per
// (chunk, value head), for up to cap = ceil(T / 64) + num_seqs chunks.
inline size_t prefill_tab_offset(int num_seqs) { return (static_cast<size_t>(num_seqs + 1) * 8 + 15) / 16 * 16; }
inline size_t prefill_header_bytes(int num_seqs, long long cap) {
    return (prefill_tab_offset(num_seqs) + static_cast<size_t>(cap) * 16 + 1023) / 1024 * 1024;
}
long long prefill_chunk_cap(long long T, int num_seqs);
size_t prefill_workspace_bytes(long long T, int num_seqs, int Hv);
// f16: q, k, v, a, b and out are IEEE binary16 (else bf16).
cudaError_t launch_prefill(const PrefillArgs& a, void* workspace, cudaStream_t stream, bool f16);

}  // namespace gdn
