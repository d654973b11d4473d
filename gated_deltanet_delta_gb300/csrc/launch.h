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
// The prefill workspace, in order: the chunk offsets (8 bytes per sequence + 1, padded to 16
// bytes), the chunk table (16 bytes per chunk), the schedule (PfPlan, the task list, the split list,
// the scratch chunk table), together padded to 1 KB; one kPfRecordBytes record per (chunk, value
// head), for up to cap = ceil(T / 64) + num_seqs chunks; then, only in a workspace large enough for
// it (split = true), the scratch of the split sequences: three 128 x 128 fp32 states per split and
// value head, and one kPfScratchRowBytes row per scratch chunk and value head, for up to
// cap2 = cap / 2 scratch chunks.
struct PrefillLayout {
    size_t tab, plan, tasks, splits, scr_tab, records, scr_state, scr_rows;
    size_t bytes_min, bytes_full;
    long long cap, cap2;
};
PrefillLayout prefill_layout(long long T, int num_seqs, int Hv);
// Whether a call with this workspace splits sequences (and so uses the scratch).
inline bool prefill_splits(const PrefillLayout& l, size_t workspace_bytes, int num_seqs) {
    return workspace_bytes >= l.bytes_full && num_seqs <= kPfOffThreads;
}
long long prefill_chunk_cap(long long T, int num_seqs);
size_t prefill_workspace_bytes(long long T, int num_seqs, int Hv);
// Raises the kernels' shared-memory limits once per device, then launches; returns the launch
// error.  Sequences are split only when workspace_bytes holds the scratch.
// f16: q, k, v, a, b and out are IEEE binary16 (else bf16).
// comba: the Comba variant (read keys p, given log decays and betas, [K][V] state pool; bf16).
cudaError_t launch_prefill(const PrefillArgs& a, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                           bool f16, bool comba = false);

}  // namespace gdn
