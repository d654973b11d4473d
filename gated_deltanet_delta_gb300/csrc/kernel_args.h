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
    // CTAs stagger_lo .. 2 stagger_lo - 1 (the second CTA slot of each SM in the first wave) start
    // stagger_cycles later; 0: no delay
    int stagger_lo;
    long long stagger_cycles;
};

// The sequential kernel's schedule.  A task is one chain of chunks, run for every value head: a
// whole sequence, or one of the three chains of a sequence split into a first and a second part
// (the first part from the pooled state; the second part once from a zero state and once from the
// identity with v = 0, the two combined with the first part's end state by the fix-up kernel).
constexpr int kPfOffThreads = 1024;      // the offsets kernel's CTA; more sequences: no split
constexpr int kPfMaxSplits = 8;
constexpr int kPfMinSplitChunks = 8;     // shorter sequences are never split
constexpr long long kPfScratchRowBytes = 65536;
enum PfTaskKind : int { kPfWhole = 0, kPfFirst = 1, kPfZero = 2, kPfOper = 3 };
struct PfPlan {
    int ntask, nsplit;
    long long nscr;  // scratch chunks in use
};

struct PrefillArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const uint16_t* a;
    const uint16_t* b;
    const float* A_log;
    const float* dt_bias;
    const uint16_t* p;        // Comba: read keys [T, H, K] (q, k, v as above; a, b, A_log, dt_bias unused)
    const float* g_log;       // Comba: log decay per token and head [T, H] (gate = exp(g_log))
    const uint16_t* beta_in;  // Comba: beta per token and head [T, H] (the value itself)
    float* state_pool;        // GDN: [pool, Hv, V, K]; Comba: [pool, H, K, V]
    const int64_t* cache_indices;
    const int64_t* cu_seqlens;
    uint16_t* out;
    int32_t* status;
    long long* chunk_off;  // workspace: first chunk of every sequence, [num_seqs + 1]
    longlong2* chunk_tab;  // workspace: per chunk (first token, sequence << 32 | length), [cap]
    uint8_t* records;      // workspace: one record per (chunk, value head), kPfRecordBytes each
    // the schedule of the sequential kernel (written by the offsets kernel) and the scratch of the
    // sequences it splits in two
    PfPlan* plan;
    int4* tasks;           // [num_seqs + 2 * max_splits]: (sequence, kind, split, 0)
    int4* splits;          // [kPfMaxSplits]: (sequence, chunks of the first part, first scratch chunk, 0)
    longlong2* scr_tab;    // per scratch chunk: (first token, split << 32 | length), [cap2]
    float* scr_state;      // [max_splits][3][Hv][128][128] fp32: S_a, B', P (see prefill.cuh)
    uint8_t* scr_rows;     // [cap2][Hv] kPfScratchRowBytes: O'^T (fp32) and F (bf16 hi, lo tiles)
    long long T;
    long long cap;         // chunk capacity of the workspace
    long long cap2;        // scratch chunk capacity (second parts of split sequences)
    int pool_size, num_seqs, Hk, Hv;
    int max_splits;        // 0: no sequence is split
    int nsm;               // multiprocessors of the device (the split rule's measure of width)
    float scale, eps;
    // polls of each device-side wait of the preparation and sequential kernels before it gives up
    // (sets GDN_STATUS_TIMEOUT and stops the CTA); the waits that drain copies and products still
    // in flight after such a give-up keep their own fixed limits
    uint32_t wait_polls;   // busy polls (control and producer lanes, the preparation kernel)
    uint32_t sleep_polls;  // polls with a 1 us suspend hint (worker warps)
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
    CUtensorMap p;  // Comba: the read keys [T, H, 128]
};

constexpr int kWinD = 128;       // head dim
constexpr int kWinThreads = 128;
constexpr int kWinMaxTok = 8;

}  // namespace gdn
