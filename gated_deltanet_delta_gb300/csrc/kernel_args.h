// kernel_args.h -- argument blocks of the kernels (passed by value) and the window's fixed sizes.
// Shared by the kernel headers and by the launchers; holds no device code.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gdn {

struct DecodeArgs {
    const float* state_in;
    float* state_out;
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const float* g;
    const uint16_t* beta;
    void* y;
    int y_f32;
    int Hk, Hv, Dv;
    int tiles;  // row tiles per head
    float scale;
    // pooled form: state_in == state_out is the pool [pool_size, Hv, Dv, Dk] and batch row b reads
    // and writes slot slots[b]; a slot outside [0, pool_size) sets bit 1 of *status and is skipped
    const int64_t* slots;  // null: state row b is batch row b
    int pool_size;
    int32_t* status;
};

struct DecodeMultiArgs {
    const float* state_in;
    float* state_out;
    const uint16_t* q;  // [B, T, Hk, Dk]
    const uint16_t* k;
    const uint16_t* v;  // [B, T, Hv, Dv]
    const float* g;     // [B, T, Hv]
    const uint16_t* beta;
    void* y;            // [B, T, Hv, Dv]
    int y_f32;
    int T, Hk, Hv, Dv;
    int tiles;
    float scale;
};

struct CombaArgs {
    const float* state;
    float* state_new;
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const uint16_t* p;
    const uint16_t* beta;
    const float* g;
    void* o;
    int o_f32;
    float scale;
};

// The Comba recurrence over T tokens per head: q, k, p [B, T, H, K], v [B, T, H, V], beta [B, T, H]
// (bf16), g [B, T, H] (fp32 log-decay), o [B, T, H, V]; state [B, H, K, V] fp32, updated in place.
struct CombaFwdArgs {
    float* state;
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const uint16_t* p;
    const uint16_t* beta;
    const float* g;
    void* o;
    int o_f32;
    int T, H;
    float scale;
};

struct WindowArgs {
    float* state;
    const float* hist;
    float* hist_out;
    const float* qkv;
    const float* alpha;
    const float* beta;
    const float* z;
    const float* conv_w;
    const float* dt;
    const float* ssm_a;
    const float* gamma;
    float* y;
    int h_k, h_v, ntok, commit_at;
    float eps;
};

struct PrefillArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const uint16_t* a;
    const uint16_t* b;
    const float* A_log;
    const float* dt_bias;
    float* state_pool;
    const int64_t* cache_indices;
    const int64_t* cu_seqlens;
    uint16_t* out;
    int32_t* status;
    long long* chunk_off;  // workspace: first chunk of every sequence, [num_seqs + 1]
    longlong2* chunk_tab;  // workspace: per chunk (first token, sequence << 32 | length), [cap]
    uint8_t* records;      // workspace: one record per (chunk, value head), kPfRecordBytes each
    long long T;
    long long cap;         // chunk capacity of the workspace
    int pool_size, num_seqs, Hk, Hv;
    float scale, eps;
};

// A prefill chunk record: everything a chunk contributes that does not depend on the state, laid
// out as the shared-memory image the sequential kernel uses (swizzled bf16 operand tiles):
//   [0, 32768)      Tw hi, Tw lo, Tu hi, Tu lo (64 x 64 each, rows t, K-major)
//   [32768, 49152)  Q~ = diag(gamma_t rq_t scale) Q (64 x 128, rows t, K-major)
//   [49152, 65536)  M~ = diag(rq_t scale) M, hi and lo (64 x 64 each, rows t, K-major)
//   [65536, 66560)  fp32 vectors: D_L [64], rk [64], gamma_L
constexpr long long kPfRecordBytes = 66560;
constexpr long long kPfRecordVec = 65536;

// TMA descriptors of the prefill's q [T, Hk, 128], k [T, Hk, 128] and v [T, Hv, 128] (bf16): boxes of
// 64 features x 1 head x 64 tokens with the 128-byte swizzle.
struct PrefillMaps {
    CUtensorMap q, k, v;
};

constexpr int kWinD = 128;       // head dim
constexpr int kWinThreads = 128;
constexpr int kWinMaxTok = 8;

}  // namespace gdn
