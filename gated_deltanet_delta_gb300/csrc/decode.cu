// decode.cu -- launch configurations of the GDN decode kernel (kernel in decode.cuh).
#include "decode.cuh"
#include "launch.h"

namespace gdn {

namespace {

template <int DK, int TPR, int RPT, int NT>
void run(DecodeArgs a, int B, cudaStream_t stream) {
    constexpr int rows = decode_rows_per_cta<DK, TPR, RPT, NT>();
    a.tiles = (a.Dv + rows - 1) / rows;
    const unsigned grid = unsigned(B) * unsigned(a.Hv) * unsigned(a.tiles);
    gdn_decode_kernel<DK, TPR, RPT, NT><<<grid, NT, 0, stream>>>(a);
}

template <int DK, int TPR, int RPT, int NT, int TB>
void run_multi(DecodeMultiArgs a, int B, cudaStream_t stream) {
    constexpr int rows = decode_rows_per_cta<DK, TPR, RPT, NT>();
    a.tiles = (a.Dv + rows - 1) / rows;
    const unsigned grid = unsigned(B) * unsigned(a.Hv) * unsigned(a.tiles);
    gdn_decode_multi_kernel<DK, TPR, RPT, NT, TB><<<grid, NT, 0, stream>>>(a);
}

}  // namespace

// Multi-token steps, 16 tokens staged per block.  Smaller CTAs than the single step, and for
// Dk = 128 / 256 half the lanes per row (8 float4 of a row per lane): the kernel is bound by
// instruction issue, and each token's reduction inside a row group then costs one shuffle level
// less per state element, while the CTA barriers of the token staging hold fewer warps.
// Dk = 256: 8 lanes per row, two rows per thread, 128 threads (32 rows per CTA).
// Dk = 128: 4 lanes per row, two rows per thread, 128 threads (64 rows per CTA).
// Dk = 64: 4 lanes per row (4 float4 each), two rows per thread, 64 threads (32 rows per CTA).
void launch_decode_multi(DecodeMultiArgs a, int B, int Dk, cudaStream_t stream) {
    if (Dk == 256)
        run_multi<256, 8, 2, 128, 16>(a, B, stream);
    else if (Dk == 128)
        run_multi<128, 4, 2, 128, 16>(a, B, stream);
    else
        run_multi<64, 4, 2, 64, 16>(a, B, stream);
}

// Dk = 256: a row is 64 float4 over 16 lanes (4 each); two rows per thread, 32 rows per CTA.
// Dk = 128: a row is 32 float4 over 8 lanes (4 each); two rows per thread, 64 rows per CTA.
// Dk = 64: a row is 16 float4 over 4 lanes (4 each); two rows per thread, 128 rows per CTA.
void launch_decode(DecodeArgs a, int B, int Dk, cudaStream_t stream) {
    if (Dk == 256)
        run<256, 16, 2, 256>(a, B, stream);
    else if (Dk == 128)
        run<128, 8, 2, 256>(a, B, stream);
    else
        run<64, 4, 2, 256>(a, B, stream);
}

}  // namespace gdn
