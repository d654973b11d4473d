// api.cu -- the C ABI of libgdn (declared in include/gdn.h): host-side validation, choice of kernel
// configuration, launch, and error reporting.  No device memory is allocated here.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "gdn.h"
#include "launch.h"

namespace {

thread_local char g_last_error[512] = "";

gdn_status fail(gdn_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// Two byte ranges overlap without being identical.
bool partial_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    if (pa == pb) return false;
    return pa < pb + nb && pb < pa + na;
}

bool any_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    return na > 0 && nb > 0 && pa < pb + nb && pb < pa + na;
}

gdn_status launched(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    g_last_error[0] = '\0';
    return GDN_OK;
}

#define REQUIRE(cond, status, ...)                    \
    do {                                              \
        if (!(cond)) return fail(status, __VA_ARGS__); \
    } while (0)

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported shape or option";
        case GDN_ERR_CUDA: return "CUDA error";
        case GDN_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

const char* gdn_last_error(void) { return g_last_error; }

// ------------------------------------------------------------------------------------------------
gdn_status gdn_decode_step(const float* state_in, float* state_out, const void* q, const void* k,
                           const void* v, const float* g, const void* beta, void* y,
                           gdn_dtype y_dtype, int B, int Hk, int Hv, int Dk, int Dv, float scale,
                           gdn_stream_t stream) {
    REQUIRE(B >= 0 && Hk >= 1 && Hv >= 1 && Dk >= 1 && Dv >= 1, GDN_ERR_INVALID_ARG,
            "gdn_decode_step: sizes must be B >= 0 and Hk, Hv, Dk, Dv >= 1 (got B=%d Hk=%d Hv=%d "
            "Dk=%d Dv=%d)", B, Hk, Hv, Dk, Dv);
    REQUIRE(Hv % Hk == 0, GDN_ERR_INVALID_ARG, "gdn_decode_step: Hv (%d) must be a multiple of Hk (%d)",
            Hv, Hk);
    REQUIRE(y_dtype == GDN_BF16 || y_dtype == GDN_F32, GDN_ERR_INVALID_ARG,
            "gdn_decode_step: y_dtype must be GDN_BF16 or GDN_F32");
    REQUIRE(Dk == 64 || Dk == 128 || Dk == 256, GDN_ERR_UNSUPPORTED,
            "gdn_decode_step: Dk must be 64, 128 or 256 (got %d)", Dk);
    if (B == 0) return GDN_OK;
    REQUIRE(state_in && state_out && q && k && v && g && beta && y, GDN_ERR_INVALID_ARG,
            "gdn_decode_step: null pointer");
    const size_t sbytes = size_t(B) * Hv * Dv * Dk * sizeof(float);
    REQUIRE(!partial_overlap(state_in, sbytes, state_out, sbytes), GDN_ERR_INVALID_ARG,
            "gdn_decode_step: state_out partially overlaps state_in");
    REQUIRE(aligned(state_in, 16) && aligned(state_out, 16), GDN_ERR_INVALID_ARG,
            "gdn_decode_step: state buffers must be 16-byte aligned");
    REQUIRE(aligned(q, 8) && aligned(k, 8), GDN_ERR_INVALID_ARG,
            "gdn_decode_step: q and k must be 8-byte aligned");
    REQUIRE(aligned(y, y_dtype == GDN_F32 ? 4 : 2) && aligned(v, 2) && aligned(beta, 2) && aligned(g, 4),
            GDN_ERR_INVALID_ARG, "gdn_decode_step: misaligned v, beta, g or y");
    const size_t yb = size_t(B) * Hv * Dv * (y_dtype == GDN_F32 ? 4 : 2);
    REQUIRE(!any_overlap(y, yb, state_out, sbytes), GDN_ERR_INVALID_ARG,
            "gdn_decode_step: y overlaps state_out");
    const long long heads = (long long)B * Hv;
    REQUIRE(heads * ((Dv + 31) / 32) < (1LL << 31), GDN_ERR_UNSUPPORTED, "gdn_decode_step: grid too large");

    gdn::DecodeArgs a;
    a.state_in = state_in;
    a.state_out = state_out;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.g = g;
    a.beta = static_cast<const uint16_t*>(beta);
    a.y = y;
    a.y_f32 = y_dtype == GDN_F32;
    a.Hk = Hk;
    a.Hv = Hv;
    a.Dv = Dv;
    a.scale = scale;
    a.tiles = 0;
    a.slots = nullptr;
    a.pool_size = 0;
    a.status = nullptr;
    gdn::launch_decode(a, B, Dk, static_cast<cudaStream_t>(stream));
    return launched("gdn_decode_step");
}

// ------------------------------------------------------------------------------------------------
gdn_status gdn_decode_multi(const float* state_in, float* state_out, const void* q, const void* k,
                            const void* v, const float* g, const void* beta, void* y,
                            gdn_dtype y_dtype, int B, int T, int Hk, int Hv, int Dk, int Dv,
                            float scale, gdn_stream_t stream) {
    REQUIRE(B >= 0 && T >= 0 && Hk >= 1 && Hv >= 1 && Dk >= 1 && Dv >= 1, GDN_ERR_INVALID_ARG,
            "gdn_decode_multi: sizes must be B, T >= 0 and Hk, Hv, Dk, Dv >= 1");
    REQUIRE(Hv % Hk == 0, GDN_ERR_INVALID_ARG, "gdn_decode_multi: Hv (%d) must be a multiple of Hk (%d)",
            Hv, Hk);
    REQUIRE(y_dtype == GDN_BF16 || y_dtype == GDN_F32, GDN_ERR_INVALID_ARG,
            "gdn_decode_multi: y_dtype must be GDN_BF16 or GDN_F32");
    REQUIRE(Dk == 64 || Dk == 128 || Dk == 256, GDN_ERR_UNSUPPORTED,
            "gdn_decode_multi: Dk must be 64, 128 or 256 (got %d)", Dk);
    if (B == 0 || T == 0) return GDN_OK;
    REQUIRE(state_in && state_out && q && k && v && g && beta && y, GDN_ERR_INVALID_ARG,
            "gdn_decode_multi: null pointer");
    const size_t sbytes = size_t(B) * Hv * Dv * Dk * sizeof(float);
    REQUIRE(!partial_overlap(state_in, sbytes, state_out, sbytes), GDN_ERR_INVALID_ARG,
            "gdn_decode_multi: state_out partially overlaps state_in");
    REQUIRE(aligned(state_in, 16) && aligned(state_out, 16) && aligned(q, 8) && aligned(k, 8),
            GDN_ERR_INVALID_ARG, "gdn_decode_multi: state must be 16-byte, q and k 8-byte aligned");
    REQUIRE(aligned(y, y_dtype == GDN_F32 ? 4 : 2) && aligned(v, 2) && aligned(beta, 2) && aligned(g, 4),
            GDN_ERR_INVALID_ARG, "gdn_decode_multi: misaligned v, beta, g or y");
    const size_t yb = size_t(B) * T * Hv * Dv * (y_dtype == GDN_F32 ? 4 : 2);
    REQUIRE(!any_overlap(y, yb, state_out, sbytes), GDN_ERR_INVALID_ARG, "gdn_decode_multi: y overlaps state_out");
    REQUIRE((long long)B * Hv * ((Dv + 31) / 32) < (1LL << 31), GDN_ERR_UNSUPPORTED,
            "gdn_decode_multi: grid too large");
    gdn::DecodeMultiArgs a;
    a.state_in = state_in;
    a.state_out = state_out;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.g = g;
    a.beta = static_cast<const uint16_t*>(beta);
    a.y = y;
    a.y_f32 = y_dtype == GDN_F32;
    a.T = T;
    a.Hk = Hk;
    a.Hv = Hv;
    a.Dv = Dv;
    a.tiles = 0;
    a.scale = scale;
    gdn::launch_decode_multi(a, B, Dk, static_cast<cudaStream_t>(stream));
    return launched("gdn_decode_multi");
}

// ------------------------------------------------------------------------------------------------
gdn_status gdn_decode_step_pooled(float* state_pool, int pool_size, const int64_t* cache_indices,
                                  const void* q, const void* k, const void* v, const float* g,
                                  const void* beta, void* y, gdn_dtype y_dtype, int B, int Hk, int Hv,
                                  int Dk, int Dv, float scale, int32_t* dev_status,
                                  gdn_stream_t stream) {
    REQUIRE(B >= 0 && pool_size >= 0 && Hk >= 1 && Hv >= 1 && Dk >= 1 && Dv >= 1, GDN_ERR_INVALID_ARG,
            "gdn_decode_step_pooled: sizes must be B, pool_size >= 0 and Hk, Hv, Dk, Dv >= 1");
    REQUIRE(Hv % Hk == 0, GDN_ERR_INVALID_ARG,
            "gdn_decode_step_pooled: Hv (%d) must be a multiple of Hk (%d)", Hv, Hk);
    REQUIRE(y_dtype == GDN_BF16 || y_dtype == GDN_F32, GDN_ERR_INVALID_ARG,
            "gdn_decode_step_pooled: y_dtype must be GDN_BF16 or GDN_F32");
    REQUIRE(Dk == 64 || Dk == 128 || Dk == 256, GDN_ERR_UNSUPPORTED,
            "gdn_decode_step_pooled: Dk must be 64, 128 or 256 (got %d)", Dk);
    if (B == 0) return GDN_OK;
    REQUIRE(state_pool && cache_indices && q && k && v && g && beta && y && dev_status,
            GDN_ERR_INVALID_ARG, "gdn_decode_step_pooled: null pointer");
    REQUIRE(aligned(state_pool, 16) && aligned(q, 8) && aligned(k, 8) && aligned(cache_indices, 8) &&
                aligned(dev_status, 4),
            GDN_ERR_INVALID_ARG, "gdn_decode_step_pooled: misaligned argument");
    REQUIRE(aligned(y, y_dtype == GDN_F32 ? 4 : 2) && aligned(v, 2) && aligned(beta, 2) && aligned(g, 4),
            GDN_ERR_INVALID_ARG, "gdn_decode_step_pooled: misaligned v, beta, g or y");
    const size_t pbytes = size_t(pool_size) * Hv * Dv * Dk * sizeof(float);
    const size_t yb = size_t(B) * Hv * Dv * (y_dtype == GDN_F32 ? 4 : 2);
    REQUIRE(!any_overlap(y, yb, state_pool, pbytes), GDN_ERR_INVALID_ARG,
            "gdn_decode_step_pooled: y overlaps state_pool");
    REQUIRE((long long)B * Hv * ((Dv + 31) / 32) < (1LL << 31), GDN_ERR_UNSUPPORTED,
            "gdn_decode_step_pooled: grid too large");
    gdn::DecodeArgs a;
    a.state_in = state_pool;
    a.state_out = state_pool;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.g = g;
    a.beta = static_cast<const uint16_t*>(beta);
    a.y = y;
    a.y_f32 = y_dtype == GDN_F32;
    a.Hk = Hk;
    a.Hv = Hv;
    a.Dv = Dv;
    a.scale = scale;
    a.tiles = 0;
    a.slots = cache_indices;
    a.pool_size = pool_size;
    a.status = dev_status;
    gdn::launch_decode(a, B, Dk, static_cast<cudaStream_t>(stream));
    return launched("gdn_decode_step_pooled");
}

// ------------------------------------------------------------------------------------------------
gdn_status comba_decode_step(const float* state, float* state_new, const void* q, const void* k,
                             const void* v, const void* p, const void* beta, const float* g,
                             void* o, gdn_dtype o_dtype, int B, int H, int K, int V, float scale,
                             gdn_stream_t stream) {
    REQUIRE(B >= 0 && H >= 1 && K >= 1 && V >= 1, GDN_ERR_INVALID_ARG,
            "comba_decode_step: sizes must be B >= 0 and H, K, V >= 1 (got B=%d H=%d K=%d V=%d)", B, H,
            K, V);
    REQUIRE(o_dtype == GDN_BF16 || o_dtype == GDN_F32, GDN_ERR_INVALID_ARG,
            "comba_decode_step: o_dtype must be GDN_BF16 or GDN_F32");
    REQUIRE((K == 64 || K == 128) && (V == 64 || V == 128), GDN_ERR_UNSUPPORTED,
            "comba_decode_step: K and V must each be 64 or 128 (got K=%d V=%d)", K, V);
    if (B == 0) return GDN_OK;
    REQUIRE(state && state_new && q && k && v && p && beta && g && o, GDN_ERR_INVALID_ARG,
            "comba_decode_step: null pointer");
    const size_t sbytes = size_t(B) * H * K * V * sizeof(float);
    REQUIRE(!partial_overlap(state, sbytes, state_new, sbytes), GDN_ERR_INVALID_ARG,
            "comba_decode_step: state_new partially overlaps state");
    REQUIRE(aligned(state, 16) && aligned(state_new, 16), GDN_ERR_INVALID_ARG,
            "comba_decode_step: state buffers must be 16-byte aligned");
    REQUIRE(aligned(q, 8) && aligned(k, 8) && aligned(p, 8) && aligned(v, 8), GDN_ERR_INVALID_ARG,
            "comba_decode_step: q, k, p and v must be 8-byte aligned");
    REQUIRE(aligned(o, o_dtype == GDN_F32 ? 16 : 8) && aligned(beta, 2) && aligned(g, 4),
            GDN_ERR_INVALID_ARG, "comba_decode_step: misaligned o, beta or g");
    const size_t ob = size_t(B) * H * V * (o_dtype == GDN_F32 ? 4 : 2);
    REQUIRE(!any_overlap(o, ob, state_new, sbytes), GDN_ERR_INVALID_ARG,
            "comba_decode_step: o overlaps state_new");
    REQUIRE((long long)B * H < (1LL << 31), GDN_ERR_UNSUPPORTED, "comba_decode_step: grid too large");

    gdn::CombaArgs a;
    a.state = state;
    a.state_new = state_new;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.p = static_cast<const uint16_t*>(p);
    a.beta = static_cast<const uint16_t*>(beta);
    a.g = g;
    a.o = o;
    a.o_f32 = o_dtype == GDN_F32;
    a.scale = scale;
    gdn::launch_comba(a, B * H, K, V, static_cast<cudaStream_t>(stream));
    return launched("comba_decode_step");
}

gdn_status comba_forward(float* state, const void* q, const void* k, const void* v, const void* p,
                         const void* beta, const float* g, void* o, gdn_dtype o_dtype, int B, int T, int H,
                         int K, int V, float scale, gdn_stream_t stream) {
    REQUIRE(B >= 0 && T >= 0 && H >= 1 && K >= 1 && V >= 1, GDN_ERR_INVALID_ARG,
            "comba_forward: sizes must be B, T >= 0 and H, K, V >= 1 (got B=%d T=%d H=%d K=%d V=%d)", B, T, H,
            K, V);
    REQUIRE(o_dtype == GDN_BF16 || o_dtype == GDN_F32, GDN_ERR_INVALID_ARG,
            "comba_forward: o_dtype must be GDN_BF16 or GDN_F32");
    REQUIRE((K == 64 || K == 128) && (V == 64 || V == 128), GDN_ERR_UNSUPPORTED,
            "comba_forward: K and V must each be 64 or 128 (got K=%d V=%d)", K, V);
    if (B == 0) return GDN_OK;
    REQUIRE(state, GDN_ERR_INVALID_ARG, "comba_forward: null state");
    REQUIRE(T == 0 || (q && k && v && p && beta && g && o), GDN_ERR_INVALID_ARG, "comba_forward: null pointer");
    REQUIRE(aligned(state, 16), GDN_ERR_INVALID_ARG, "comba_forward: state must be 16-byte aligned");
    REQUIRE(aligned(q, 8) && aligned(k, 8) && aligned(p, 8) && aligned(v, 8), GDN_ERR_INVALID_ARG,
            "comba_forward: q, k, p and v must be 8-byte aligned");
    REQUIRE(aligned(o, o_dtype == GDN_F32 ? 16 : 8) && aligned(beta, 2) && aligned(g, 4), GDN_ERR_INVALID_ARG,
            "comba_forward: misaligned o, beta or g");
    const size_t sbytes = size_t(B) * H * K * V * sizeof(float);
    const size_t ob = size_t(B) * T * H * V * (o_dtype == GDN_F32 ? 4 : 2);
    REQUIRE(!any_overlap(o, ob, state, sbytes), GDN_ERR_INVALID_ARG, "comba_forward: o overlaps state");
    REQUIRE((long long)B * H < (1LL << 31) && (long long)B * T * H * (K > V ? K : V) < (1LL << 62),
            GDN_ERR_UNSUPPORTED, "comba_forward: sizes too large");

    gdn::CombaFwdArgs a;
    a.state = state;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.p = static_cast<const uint16_t*>(p);
    a.beta = static_cast<const uint16_t*>(beta);
    a.g = g;
    a.o = o;
    a.o_f32 = o_dtype == GDN_F32;
    a.T = T;
    a.H = H;
    a.scale = scale;
    gdn::launch_comba_forward(a, B * H, K, V, static_cast<cudaStream_t>(stream));
    return launched("comba_forward");
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// The chunk sizes accepted: the page's two entry points default to 64 (the CUDA chunkwise one) and
// 128 (the fully batched torch one).  The chunked form computes the same function for every chunk
// size, up to rounding, so both run the same 64-token kernels.
static bool prefill_chunk_size_ok(int chunk_size) { return chunk_size == 64 || chunk_size == 128; }

extern "C" size_t gdn_prefill_workspace_size(int num_seqs, int64_t T, int Hk, int Hv, int K, int V,
                                             int chunk_size) {
    if (num_seqs <= 0 || T < 0 || Hk < 1 || Hv < 1 || Hv % Hk != 0 || K != 128 || V != 128 ||
        !prefill_chunk_size_ok(chunk_size) || T >= (1LL << 31) - 64)
        return 0;
    return gdn::prefill_workspace_bytes(T, num_seqs, Hv);
}

// gdn_prefill_chunked, gdn_prefill_chunked_f16 and comba_prefill_chunked: the same checks and
// launch, the token arrays (q, k, v, a, b, out) in bf16 or in IEEE binary16; for Comba (a, b, A_log,
// dt_bias unused) the read keys, log decays and betas of CombaIn instead.
struct CombaIn {
    const void* p;
    const void* beta;
    const float* g;
};
namespace {
// The prefill kernels' wait limit (gdn_prefill_set_wait_limit): 0 means the built-in limits.
std::atomic<uint32_t> g_prefill_wait_polls{0};
constexpr uint32_t kPrefillBusyPolls = 1u << 26;   // seconds of busy polling
constexpr uint32_t kPrefillSleepPolls = 1u << 22;  // polls with a 1 us suspend hint: seconds
}  // namespace

extern "C" void gdn_prefill_set_wait_limit(uint32_t polls) {
    g_prefill_wait_polls.store(polls, std::memory_order_relaxed);
}

static gdn_status prefill_entry(const char* fn, bool f16, const void* q, const void* k, const void* v,
                                const void* a, const void* b, const float* A_log, const float* dt_bias,
                                float* state_pool, int pool_size, const int64_t* cache_indices,
                                const int64_t* cu_seqlens, int num_seqs, int64_t T, int Hk, int Hv, int K,
                                int V, int chunk_size, float scale, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, gdn_stream_t stream,
                                const CombaIn* cb = nullptr) {
    REQUIRE(num_seqs >= 0 && T >= 0 && pool_size >= 0 && Hk >= 1 && Hv >= 1 && K >= 1 && V >= 1,
            GDN_ERR_INVALID_ARG, "%s: sizes must be num_seqs, T, pool_size >= 0 and Hk, Hv, K, V >= 1", fn);
    REQUIRE(Hv % Hk == 0, GDN_ERR_INVALID_ARG, "%s: Hv (%d) must be a multiple of Hk (%d)", fn, Hv, Hk);
    REQUIRE(K == 128 && V == 128, GDN_ERR_UNSUPPORTED, "%s: K and V must be 128 (got K=%d V=%d)", fn, K, V);
    REQUIRE(prefill_chunk_size_ok(chunk_size), GDN_ERR_UNSUPPORTED, "%s: chunk_size must be 64 or 128 (got %d)",
            fn, chunk_size);
    if (num_seqs == 0) return GDN_OK;
    REQUIRE(cache_indices && cu_seqlens && dev_status && state_pool && (cb || (A_log && dt_bias)),
            GDN_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (cb) {
        REQUIRE(T == 0 || (q && k && v && cb->p && cb->beta && cb->g && out), GDN_ERR_INVALID_ARG,
                "%s: null token pointer", fn);
        REQUIRE(aligned(cb->p, 16) && aligned(cb->beta, 2) && aligned(cb->g, 4), GDN_ERR_INVALID_ARG,
                "%s: misaligned argument (p 16 bytes, beta 2, g 4)", fn);
    } else {
        REQUIRE(T == 0 || (q && k && v && a && b && out), GDN_ERR_INVALID_ARG, "%s: null token pointer", fn);
        REQUIRE(aligned(a, 2) && aligned(b, 2) && aligned(A_log, 4) && aligned(dt_bias, 4), GDN_ERR_INVALID_ARG,
                "%s: misaligned argument", fn);
    }
    REQUIRE(aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(out, 16) && aligned(state_pool, 16),
            GDN_ERR_INVALID_ARG, "%s: q, k, v, out and state_pool must be 16-byte aligned", fn);
    REQUIRE(aligned(dev_status, 4) && aligned(cache_indices, 8) && aligned(cu_seqlens, 8),
            GDN_ERR_INVALID_ARG, "%s: misaligned argument", fn);
    const size_t obytes = size_t(T) * Hv * V * 2, pbytes = size_t(pool_size) * Hv * V * K * 4;
    REQUIRE(!any_overlap(out, obytes, state_pool, pbytes), GDN_ERR_INVALID_ARG, "%s: out overlaps state_pool",
            fn);
    REQUIRE((long long)(num_seqs + 2 * gdn::kPfMaxSplits) * Hv < (1LL << 31) && T < (1LL << 31) - 64 &&
                gdn::prefill_chunk_cap(T, num_seqs) * Hv < (1LL << 31),
            GDN_ERR_UNSUPPORTED, "%s: grid or token count too large", fn);
    const gdn::PrefillLayout lay = gdn::prefill_layout(T, num_seqs, Hv);
    REQUIRE(workspace && workspace_bytes >= lay.bytes_min, GDN_ERR_INVALID_ARG,
            "%s: workspace of %zu bytes given, %zu needed", fn, workspace ? workspace_bytes : 0, lay.bytes_min);
    REQUIRE(aligned(workspace, 256), GDN_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", fn);
    const size_t ws_used = gdn::prefill_splits(lay, workspace_bytes, num_seqs) ? lay.bytes_full : lay.bytes_min;
    REQUIRE(!any_overlap(workspace, ws_used, out, obytes) && !any_overlap(workspace, ws_used, state_pool, pbytes),
            GDN_ERR_INVALID_ARG, "%s: workspace overlaps out or state_pool", fn);

    gdn::PrefillArgs p;
    p.q = static_cast<const uint16_t*>(q);
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.a = static_cast<const uint16_t*>(a);
    p.b = static_cast<const uint16_t*>(b);
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.p = cb ? static_cast<const uint16_t*>(cb->p) : nullptr;
    p.g_log = cb ? cb->g : nullptr;
    p.beta_in = cb ? static_cast<const uint16_t*>(cb->beta) : nullptr;
    p.state_pool = state_pool;
    p.cache_indices = cache_indices;
    p.cu_seqlens = cu_seqlens;
    p.out = static_cast<uint16_t*>(out);
    p.status = dev_status;
    p.T = T;
    p.pool_size = pool_size;
    p.num_seqs = num_seqs;
    p.Hk = Hk;
    p.Hv = Hv;
    p.scale = scale;
    p.eps = 1e-6f;
    const uint32_t polls = g_prefill_wait_polls.load(std::memory_order_relaxed);
    p.wait_polls = polls ? polls : kPrefillBusyPolls;
    p.sleep_polls = polls ? polls : kPrefillSleepPolls;
    const cudaError_t e =
        gdn::launch_prefill(p, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), f16, cb != nullptr);
    if (e != cudaSuccess)
        return fail(GDN_ERR_CUDA, "%s: launch failed (TMA descriptors or kernel): %s", fn, cudaGetErrorString(e));
    g_last_error[0] = '\0';
    return GDN_OK;
}

extern "C" gdn_status gdn_prefill_chunked(const void* q, const void* k, const void* v, const void* a,
                                          const void* b, const float* A_log, const float* dt_bias,
                                          float* state_pool, int pool_size,
                                          const int64_t* cache_indices, const int64_t* cu_seqlens,
                                          int num_seqs, int64_t T, int Hk, int Hv, int K, int V,
                                          int chunk_size, float scale, void* out, void* workspace,
                                          size_t workspace_bytes, int32_t* dev_status,
                                          gdn_stream_t stream) {
    return prefill_entry("gdn_prefill_chunked", false, q, k, v, a, b, A_log, dt_bias, state_pool, pool_size,
                         cache_indices, cu_seqlens, num_seqs, T, Hk, Hv, K, V, chunk_size, scale, out,
                         workspace, workspace_bytes, dev_status, stream);
}

extern "C" gdn_status gdn_prefill_chunked_f16(const void* q, const void* k, const void* v, const void* a,
                                              const void* b, const float* A_log, const float* dt_bias,
                                              float* state_pool, int pool_size,
                                              const int64_t* cache_indices, const int64_t* cu_seqlens,
                                              int num_seqs, int64_t T, int Hk, int Hv, int K, int V,
                                              int chunk_size, float scale, void* out, void* workspace,
                                              size_t workspace_bytes, int32_t* dev_status,
                                              gdn_stream_t stream) {
    return prefill_entry("gdn_prefill_chunked_f16", true, q, k, v, a, b, A_log, dt_bias, state_pool, pool_size,
                         cache_indices, cu_seqlens, num_seqs, T, Hk, Hv, K, V, chunk_size, scale, out,
                         workspace, workspace_bytes, dev_status, stream);
}

extern "C" gdn_status comba_prefill_chunked(const void* q, const void* k, const void* v, const void* p,
                                            const void* beta, const float* g, float* state_pool, int pool_size,
                                            const int64_t* cache_indices, const int64_t* cu_seqlens,
                                            int num_seqs, int64_t T, int H, int K, int V, int chunk_size,
                                            float scale, void* out, void* workspace, size_t workspace_bytes,
                                            int32_t* dev_status, gdn_stream_t stream) {
    const CombaIn cb{p, beta, g};
    return prefill_entry("comba_prefill_chunked", false, q, k, v, nullptr, nullptr, nullptr, nullptr, state_pool,
                         pool_size, cache_indices, cu_seqlens, num_seqs, T, H, H, K, V, chunk_size, scale, out,
                         workspace, workspace_bytes, dev_status, stream, &cb);
}


// ------------------------------------------------------------------------------------------------
extern "C" gdn_status gdn_window_fused(float* state, const float* hist, float* hist_out,
                                       const float* qkv, const float* alpha, const float* beta,
                                       const float* z, const float* conv_w, const float* dt,
                                       const float* ssm_a, const float* gamma, float* y, int N,
                                       int h_k, int h_v, int ntok, unsigned commit, float eps,
                                       gdn_stream_t stream) {
    REQUIRE(N >= 0 && h_k >= 1 && h_v >= 1, GDN_ERR_INVALID_ARG,
            "gdn_window_fused: sizes must be N >= 0 and h_k, h_v >= 1 (got N=%d h_k=%d h_v=%d)", N, h_k,
            h_v);
    REQUIRE(ntok >= 1 && ntok <= gdn::kWinMaxTok, GDN_ERR_UNSUPPORTED,
            "gdn_window_fused: ntok must be in [1, %d] (got %d)", gdn::kWinMaxTok, ntok);
    REQUIRE(h_k <= h_v, GDN_ERR_UNSUPPORTED,
            "gdn_window_fused: h_k (%d) must not exceed h_v (%d)", h_k, h_v);
    int commit_at = -1;
    if (commit == 0u) commit_at = 0;
    else if (commit == 1u) commit_at = ntok;
    else if ((commit >> 8) == 1u && (commit & 0xffu) >= 1u && int(commit & 0xffu) <= ntok)
        commit_at = int(commit & 0xffu);
    REQUIRE(commit_at >= 0, GDN_ERR_INVALID_ARG,
            "gdn_window_fused: commit must be 0, 1 or 0x100|k with 1 <= k <= ntok (got 0x%x)", commit);
    if (N == 0) return GDN_OK;
    REQUIRE(state && hist && hist_out && qkv && alpha && beta && z && conv_w && dt && ssm_a && gamma &&
                y, GDN_ERR_INVALID_ARG, "gdn_window_fused: null pointer");
    const size_t C = size_t(2 * h_k + h_v) * gdn::kWinD;
    const size_t hbytes = size_t(N) * C * 3 * sizeof(float);
    REQUIRE(!any_overlap(hist, hbytes, hist_out, hbytes), GDN_ERR_INVALID_ARG,
            "gdn_window_fused: hist_out must not overlap hist (the q/k history is read by several heads)");
    const size_t sbytes = size_t(N) * gdn::kWinD * h_v * gdn::kWinD * sizeof(float);
    const size_t ybytes = size_t(N) * ntok * h_v * gdn::kWinD * sizeof(float);
    REQUIRE(!any_overlap(y, ybytes, state, sbytes) && !any_overlap(y, ybytes, hist_out, hbytes) &&
                !any_overlap(state, sbytes, hist_out, hbytes),
            GDN_ERR_INVALID_ARG, "gdn_window_fused: y, state and hist_out must not overlap");
    REQUIRE(aligned(state, 16) && aligned(conv_w, 16), GDN_ERR_INVALID_ARG,
            "gdn_window_fused: state and conv_w must be 16-byte aligned");
    REQUIRE(aligned(hist, 4) && aligned(hist_out, 4) && aligned(qkv, 4) && aligned(alpha, 4) &&
                aligned(beta, 4) && aligned(z, 4) && aligned(dt, 4) && aligned(ssm_a, 4) &&
                aligned(gamma, 4) && aligned(y, 4),
            GDN_ERR_INVALID_ARG, "gdn_window_fused: float arrays must be 4-byte aligned");
    REQUIRE(1LL * N * h_v < (1LL << 31), GDN_ERR_UNSUPPORTED, "gdn_window_fused: grid too large");

    gdn::WindowArgs a;
    a.state = state;
    a.hist = hist;
    a.hist_out = hist_out;
    a.qkv = qkv;
    a.alpha = alpha;
    a.beta = beta;
    a.z = z;
    a.conv_w = conv_w;
    a.dt = dt;
    a.ssm_a = ssm_a;
    a.gamma = gamma;
    a.y = y;
    a.h_k = h_k;
    a.h_v = h_v;
    a.ntok = ntok;
    a.commit_at = commit_at;
    a.eps = eps;
    const cudaError_t e = gdn::launch_window(a, N, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(GDN_ERR_CUDA, "gdn_window_fused: launch failed: %s", cudaGetErrorString(e));
    g_last_error[0] = '\0';
    return GDN_OK;
}

// ------------------------------------------------------------------------------------------------
// gdn_prefill_chunked_noalloc: the prefill for callers that cannot allocate device memory
// themselves (a host framework whose allocator owns all device memory, or code running where a
// cudaMalloc is not allowed).  Its workspace is a file-scope device array of fixed size, which
// every GPU that loads this library holds until the process exits.  Host code sees only a
// host-side stand-in for the array, so its device address is looked up once per device, with that
// device current, and handed to the kernels.
namespace {

constexpr size_t kNoallocScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) uint8_t g_prefill_scratch[kNoallocScratchBytes];

constexpr int kNoallocMaxDevices = 64;
void* g_scratch_ptr[kNoallocMaxDevices];    // the array's device address on each device
std::atomic<int> g_scratch_ready[kNoallocMaxDevices];
std::mutex g_scratch_mutex;

}  // namespace

extern "C" gdn_status gdn_prefill_chunked_noalloc(const void* q, const void* k, const void* v, const void* a,
                                                  const void* b, const float* A_log, const float* dt_bias,
                                                  float* state_pool, int pool_size,
                                                  const int64_t* cache_indices, const int64_t* cu_seqlens,
                                                  int num_seqs, int64_t T, int Hk, int Hv, int K, int V,
                                                  int chunk_size, float scale, void* out,
                                                  int32_t* dev_status, gdn_stream_t stream) {
    // the scratch must hold the records; long sequences are split only when it also holds the
    // split scratch
    const size_t full = gdn_prefill_workspace_size(num_seqs, T, Hk, Hv, K, V, chunk_size);
    const size_t need = full == 0 ? 0 : gdn::prefill_layout(T, num_seqs, Hv).bytes_min;
    REQUIRE(need <= kNoallocScratchBytes, GDN_ERR_UNSUPPORTED,
            "gdn_prefill_chunked_noalloc: these sizes need %zu bytes of workspace (%zu without splitting "
            "long sequences); the library's static scratch holds %zu (use gdn_prefill_chunked with a "
            "caller-owned workspace)",
            full, need, kNoallocScratchBytes);
    if (num_seqs == 0)  // nothing runs; the scratch is not needed
        return gdn_prefill_chunked(q, k, v, a, b, A_log, dt_bias, state_pool, pool_size, cache_indices,
                                   cu_seqlens, num_seqs, T, Hk, Hv, K, V, chunk_size, scale, out, nullptr, 0,
                                   dev_status, stream);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(GDN_ERR_CUDA, "gdn_prefill_chunked_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    REQUIRE(dev >= 0 && dev < kNoallocMaxDevices, GDN_ERR_UNSUPPORTED,
            "gdn_prefill_chunked_noalloc: device %d beyond the %d supported", dev, kNoallocMaxDevices);
    if (!g_scratch_ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        if (!g_scratch_ready[dev].load(std::memory_order_relaxed)) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_prefill_scratch);
            if (e != cudaSuccess || p == nullptr)
                return fail(GDN_ERR_CUDA, "gdn_prefill_chunked_noalloc: cudaGetSymbolAddress of the scratch: %s",
                            cudaGetErrorString(e));
            g_scratch_ptr[dev] = p;
            g_scratch_ready[dev].store(1, std::memory_order_release);
        }
    }
    return gdn_prefill_chunked(q, k, v, a, b, A_log, dt_bias, state_pool, pool_size, cache_indices, cu_seqlens,
                               num_seqs, T, Hk, Hv, K, V, chunk_size, scale, out, g_scratch_ptr[dev],
                               kNoallocScratchBytes, dev_status, stream);
}
