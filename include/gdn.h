/*
 * gdn.h -- C ABI of the GB300 gated delta-rule library (libgdn.so).
 *
 * Four operations of the gated delta-rule recurrence, each a set of hand-written CUDA kernels for
 * sm_103a:
 *   gdn_decode_step      one-token GDN step with key sharing (Hv value heads over Hk key heads)
 *   gdn_decode_step_pooled  the same on a pooled state indexed by cache_indices
 *   gdn_decode_multi     T consecutive decode steps with the state held on chip
 *   comba_decode_step    one-token Comba step (state read with key p, written with key k)
 *   comba_forward        the Comba recurrence over T tokens with the state held on chip
 *   gdn_prefill_chunked  varlen chunkwise-WY prefill over a pooled state, gates derived in-kernel
 *   gdn_prefill_chunked_f16  the same with IEEE binary16 token arrays
 *   gdn_prefill_chunked_noalloc  the same with the library's own fixed-size workspace
 *   comba_prefill_chunked  varlen chunkwise-WY prefill of the Comba recurrence over a pooled state
 *   gdn_window_fused     fused decode window: conv + SiLU, L2 norm, gates, recurrence over ntok
 *                        tokens, gated RMSNorm, with verify / commit / partial commit
 *
 * Conventions shared by every entry point
 *   - Every tensor argument is a DEVICE pointer to dense, contiguous, row-major memory in the layout
 *     given beside it.  "bf16" is IEEE bfloat16 (the upper half of a float32); "f16" is IEEE
 *     binary16; "f32" is IEEE float.
 *   - The caller owns every buffer, including the prefill workspace.  The library allocates no
 *     device memory and keeps no global state besides a per-device table of kernel attributes and
 *     the fixed 64 MiB device scratch array of gdn_prefill_chunked_noalloc.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *     Results are valid once the stream has been synchronised.
 *   - Arguments are validated on the host before anything is launched.  A rejected call returns
 *     GDN_ERR_INVALID_ARG or GDN_ERR_UNSUPPORTED and writes nothing.  A failed launch returns
 *     GDN_ERR_CUDA.  gdn_last_error() gives a human-readable reason for the last failure on the
 *     calling thread.
 *   - Sizes of zero are legal no-ops (nothing is launched; pointers may then be NULL).
 *
 * Sources (page title and section) of what each operation computes:
 *   [gated_delta.rs]  metaltile-std, src/ffai/gated_delta.rs: module doc "Recurrence per step",
 *                     "Layouts", "DISPATCH INVARIANTS".
 *   [comba spec]      KBench, specs/comba_decode_step.py: signature, spec_md, contract_md,
 *                     precision_md.
 *   [gdn_chunkwise]   pymllm, gdn_chunkwise: module doc "Algorithm (per chunk of C tokens)",
 *                     gdn_extend_chunkwise parameters.
 *   [gdn.metal]       regolith, baseline-kernels/gdn.metal: header comment and GdnArgs.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad layout or overlap */
    GDN_ERR_UNSUPPORTED = 2, /* a valid request outside the shapes the kernels are built for */
    GDN_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed (see gdn_last_error) */
    GDN_ERR_TIMEOUT = 4      /* reserved for bounded device-side waits that gave up */
} gdn_status;

typedef enum gdn_dtype { GDN_BF16 = 0, GDN_F32 = 1 } gdn_dtype;

/* A cudaStream_t, passed opaquely so that this header needs no CUDA header. */
typedef void* gdn_stream_t;

/* Bits of the device status word of gdn_prefill_chunked and gdn_decode_step_pooled. */
#define GDN_STATUS_BAD_CACHE_INDEX 1 /* a cache_indices entry outside [0, pool_size) */
#define GDN_STATUS_BAD_SEQLENS 2     /* cu_seqlens[n] < 0, decreasing, or beyond T */
#define GDN_STATUS_TIMEOUT 4         /* a bounded wait for the tensor core or a copy gave up */

/*
 * gdn_decode_step -- one GDN decode step for B sequences.  [gated_delta.rs] "Recurrence per step":
 *     S' = g S;  kv = S' k (sum over Dk);  delta = (v - kv) beta;  S_new = S' + delta (x) k;
 *     y = scale * S_new q (sum over Dk).
 * Value head hv reads key head hv / (Hv / Hk) ([gated_delta.rs] DISPATCH INVARIANTS).
 *
 *   state_in   f32  [B, Hv, Dv, Dk]  (Dk contiguous)      read
 *   state_out  f32  [B, Hv, Dv, Dk]                       written; may equal state_in (in place),
 *                                                         must not partially overlap it
 *   q, k       bf16 [B, Hk, Dk]                           k is used as given (no normalisation)
 *   v          bf16 [B, Hv, Dv]
 *   g          f32  [B, Hv]   linear forget gate (not its log)
 *   beta       bf16 [B, Hv]
 *   y          [B, Hv, Dv] of y_dtype (GDN_BF16: round to nearest even; GDN_F32)
 *   scale      readout scale (Dk^-0.5 is the usual choice; 1 reproduces the page exactly)
 * Supported: Dk in {64, 128, 256}, any Dv >= 1, Hk >= 1, Hv % Hk == 0.
 * All state arithmetic is f32; bf16 inputs are widened exactly.
 */
gdn_status gdn_decode_step(const float* state_in, float* state_out, const void* q, const void* k,
                           const void* v, const float* g, const void* beta, void* y,
                           gdn_dtype y_dtype, int B, int Hk, int Hv, int Dk, int Dv, float scale,
                           gdn_stream_t stream);

/*
 * gdn_decode_multi -- T consecutive GDN decode steps for B sequences in one call: the state stays
 * in registers across the tokens and crosses HBM once ([gated_delta.rs] mt_gated_delta_chunk:
 * the same recurrence as gdn_decode_step, wrapped in a loop over t).
 *
 *   state_in, state_out  f32 [B, Hv, Dv, Dk]   as gdn_decode_step (state_out after the T tokens)
 *   q, k       bf16 [B, T, Hk, Dk]
 *   v          bf16 [B, T, Hv, Dv]
 *   g          f32  [B, T, Hv]   linear gates
 *   beta       bf16 [B, T, Hv]
 *   y          [B, T, Hv, Dv] of y_dtype
 * Supported: as gdn_decode_step, any T >= 0 (T = 0 copies nothing and writes nothing).
 */
gdn_status gdn_decode_multi(const float* state_in, float* state_out, const void* q, const void* k,
                            const void* v, const float* g, const void* beta, void* y,
                            gdn_dtype y_dtype, int B, int T, int Hk, int Hv, int Dk, int Dv,
                            float scale, gdn_stream_t stream);

/*
 * gdn_decode_step_pooled -- the same decode step on a pooled state: batch row b reads and writes,
 * in place, slot cache_indices[b] of state_pool (the cache_indices / state_pool convention of
 * [gdn_chunkwise] gdn_extend_chunkwise, applied to one decode token).
 *
 *   state_pool     f32 [pool_size, Hv, Dv, Dk]   updated in place at the referenced slots only
 *   cache_indices  int64 [B]    distinct slots; duplicates give an undefined result
 *   q, k, v, g, beta, y, y_dtype, scale: as gdn_decode_step
 *   dev_status     device int32, zeroed by the caller; bit GDN_STATUS_BAD_CACHE_INDEX is set for a
 *                  slot outside [0, pool_size), whose batch row is then skipped (y not written)
 * Supported: as gdn_decode_step.
 */
gdn_status gdn_decode_step_pooled(float* state_pool, int pool_size, const int64_t* cache_indices,
                                  const void* q, const void* k, const void* v, const float* g,
                                  const void* beta, void* y, gdn_dtype y_dtype, int B, int Hk, int Hv,
                                  int Dk, int Dv, float scale, int32_t* dev_status,
                                  gdn_stream_t stream);

/*
 * comba_decode_step -- one Comba decode step for B sequences.  [comba spec] spec_md:
 *     S = exp(g) S;  u = beta (v - S^T p);  S_new = S + k u^T;  o = S_new^T (scale q).
 * The state is read with p and written with k.
 *
 *   state      f32  [B, H, K, V]  (V contiguous)          read
 *   state_new  f32  [B, H, K, V]                          written; may equal state (in place),
 *                                                         must not partially overlap it
 *   q, k, p    bf16 [B, H, K]
 *   v          bf16 [B, H, V]
 *   beta       bf16 [B, H]
 *   g          f32  [B, H]   log-decay (<= 0 in use; any finite value is accepted)
 *   o          [B, H, V] of o_dtype (GDN_BF16 or GDN_F32)
 *   scale      query scale ([comba spec]: K^-0.5 when the caller has no other value)
 * Supported: K in {64, 128} and V in {64, 128} (the shapes of the Comba spec's regime).
 */
gdn_status comba_decode_step(const float* state, float* state_new, const void* q, const void* k,
                             const void* v, const void* p, const void* beta, const float* g,
                             void* o, gdn_dtype o_dtype, int B, int H, int K, int V, float scale,
                             gdn_stream_t stream);

/*
 * comba_forward -- the Comba recurrence over T consecutive tokens of each of B sequences.
 * [comba spec] spec_md: the decode step is the comba-forward task's recurrence run for one token,
 * and running it T times reproduces that task.  Per (b, h) head and token t, the comba_decode_step
 * function on the state carried from token t - 1 (evaluated 8 tokens at a time in the equivalent
 * WY-regrouped form, so results match T single steps up to rounding order):
 *     S = exp(g_t) S;  u_j = beta_t (v_j - sum_i p_i S_ij);  S_ij += k_i u_j;
 *     o_t,j = sum_i (scale q_i) S_ij.
 *
 *   state      f32  [B, H, K, V]   V contiguous; the initial state, overwritten IN PLACE with the
 *                                  state after the last token (left as given when T = 0)
 *   q, k, p    bf16 [B, T, H, K]   k writes the state, p reads it
 *   v          bf16 [B, T, H, V]
 *   beta       bf16 [B, T, H]
 *   g          f32  [B, T, H]      log-decay (the gate is exp(g))
 *   o          [B, T, H, V] of o_dtype (GDN_BF16 round to nearest even, or GDN_F32); must not
 *              overlap state
 * Supported: K, V in {64, 128}.  The state is read once and written once per call; all arithmetic
 * is f32.
 */
gdn_status comba_forward(float* state, const void* q, const void* k, const void* v, const void* p,
                         const void* beta, const float* g, void* o, gdn_dtype o_dtype, int B, int T, int H,
                         int K, int V, float scale, gdn_stream_t stream);

/*
 * gdn_prefill_workspace_size -- bytes of device workspace gdn_prefill_chunked needs for these
 * sizes, with cap = ceil(T / 64) + num_seqs chunks and cap2 = floor(cap / 2):
 *   - a header padded to 1 KB: the first chunk of every sequence (8 bytes each, num_seqs + 1 of
 *     them, padded to 16 bytes), a 16-byte entry per chunk, and the schedule of the sequential
 *     kernel (16 bytes, 16 per task for num_seqs + 16 tasks, 16 per split for 8 splits, 16 per
 *     scratch chunk for cap2 of them);
 *   - one 66,560-byte record per (chunk, value head) (what a chunk contributes independently of
 *     the carried state: Tw, Tu and the output-scaled M split into bf16 high / low parts, the
 *     output-scaled q rows, and per-token scales);
 *   - the scratch of sequences split in two (a long sequence's second half runs next to its first
 *     half and is corrected afterwards): 3 x 65,536 bytes per split (at most 8) and value head,
 *     and 65,536 bytes per scratch chunk (cap2) and value head.
 * A workspace holding the header and the records but not the split scratch is also accepted;
 * then no sequence is split (same results up to rounding, slower when one sequence dominates).
 * Pure host function; returns 0 when num_seqs is 0 and for sizes gdn_prefill_chunked does not
 * support.
 */
size_t gdn_prefill_workspace_size(int num_seqs, int64_t T, int Hk, int Hv, int K, int V,
                                  int chunk_size);

/*
 * gdn_prefill_chunked -- varlen prefill of num_seqs sequences, chunkwise WY form.
 * [gdn_chunkwise] module doc, steps 1-3, and gdn_extend_chunkwise parameters.  Per sequence n
 * (tokens cu_seqlens[n] .. cu_seqlens[n+1]-1) and value head h (key head h / (Hv / Hk)):
 *     S <- state_pool[cache_indices[n], h];  per token t:
 *     log g_t = -exp(A_log[h]) softplus(a_t + dt_bias[h]) (softplus threshold 20);
 *     beta_t = sigmoid(b_t);  k^ = k / sqrt(|k|^2 + 1e-6);  q^ = scale q / sqrt(|q|^2 + 1e-6);
 *     S <- g_t S (I - beta_t k^ k^^T) + beta_t v_t k^^T;  out_t = S q^;
 *     state_pool[cache_indices[n], h] <- S.
 * computed chunk by chunk (64 tokens, chunks restart at each sequence start, the last one may be
 * short) with the WY representation; the inter-chunk carry is f32.  The chunked form gives the same
 * function for every chunk size up to rounding, so chunk_size selects nothing: the page's two
 * defaults, 64 and 128, are accepted and both run 64-token chunks.
 *
 *   q, k           bf16 [T, Hk, K]    not pre-normalised
 *   v              bf16 [T, Hv, V]
 *   a, b           bf16 [T, Hv]       raw gate inputs (before softplus / sigmoid)
 *   A_log, dt_bias f32  [Hv]
 *   state_pool     f32  [pool_size, Hv, V, K]  updated IN PLACE at the referenced slots only;
 *                                     other slots are not touched
 *   cache_indices  int64 [num_seqs]   distinct slots; duplicates give an undefined result
 *   cu_seqlens     int64 [num_seqs + 1]
 *   out            bf16 [T, Hv, V]    16-byte aligned; tokens of skipped sequences are not written
 *   workspace      device buffer of gdn_prefill_workspace_size(...) bytes (or at least its header
 *                  and records, see there; workspace_bytes tells which), 256-byte aligned,
 *                  overlapping neither out nor state_pool (NULL only when num_seqs is 0);
 *                  contents need not be initialised and are scratch after the call; calls that
 *                  share a workspace must not overlap on the GPU
 *   dev_status     device int32, zeroed by the caller; the kernels OR in GDN_STATUS_* bits for a
 *                  sequence they skip (slot out of range, malformed bounds)
 *   scale          query scale (K^-0.5 when the caller has no other value)
 * Supported: K = V = 128, chunk_size 64 or 128, Hv % Hk == 0.
 */
gdn_status gdn_prefill_chunked(const void* q, const void* k, const void* v, const void* a,
                               const void* b, const float* A_log, const float* dt_bias,
                               float* state_pool, int pool_size, const int64_t* cache_indices,
                               const int64_t* cu_seqlens, int num_seqs, int64_t T, int Hk, int Hv,
                               int K, int V, int chunk_size, float scale, void* out,
                               void* workspace, size_t workspace_bytes, int32_t* dev_status,
                               gdn_stream_t stream);

/*
 * gdn_prefill_chunked_f16 -- gdn_prefill_chunked with q, k, v, a, b and out in f16 instead of bf16
 * ([gdn_chunkwise] gdn_extend_chunkwise: q, k, v "bf16/fp16").  Same arguments, layouts, workspace
 * (gdn_prefill_workspace_size), checks and status bits; out is rounded to f16 (nearest even).
 * Inputs are widened exactly.  The products of raw k and v rows run on f16 operands; their
 * computed partners (the WY factors and the scaled Delta) are split into f16 high and low parts,
 * whose range is f16's: a key row of norm below |Delta| / 65504 (|Delta| the size of a value
 * correction) overflows them and gives non-finite outputs.  bf16 inputs have no such limit.
 */
gdn_status gdn_prefill_chunked_f16(const void* q, const void* k, const void* v, const void* a,
                                   const void* b, const float* A_log, const float* dt_bias,
                                   float* state_pool, int pool_size, const int64_t* cache_indices,
                                   const int64_t* cu_seqlens, int num_seqs, int64_t T, int Hk, int Hv,
                                   int K, int V, int chunk_size, float scale, void* out,
                                   void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                   gdn_stream_t stream);

/*
 * comba_prefill_chunked -- varlen prefill of the Comba recurrence ([comba spec] spec_md: the decode
 * step is the comba-forward recurrence for one token; here over every token of num_seqs sequences),
 * computed chunk by chunk with the same WY representation as gdn_prefill_chunked ([gdn_chunkwise]
 * steps 1-3), the read key p taking k's place where the state is read (the in-chunk triangular
 * system and W) and k kept where it is written.  Per sequence n and head h:
 *     S <- state_pool[cache_indices[n], h]  (K x V, V contiguous);  per token t:
 *     S <- exp(g_t) S;  u = beta_t (v_t - S^T p_t);  S <- S + k_t u^T;  out_t = S^T (scale q_t);
 *     state_pool[cache_indices[n], h] <- S.
 *   q, k, p        bf16 [T, H, K]     used as given (the spec passes them L2-normalised)
 *   v              bf16 [T, H, V]
 *   beta           bf16 [T, H]        the value itself
 *   g              f32  [T, H]        log decay (the gate is exp(g))
 *   state_pool     f32  [pool_size, H, K, V]  updated IN PLACE at the referenced slots only
 *   out            bf16 [T, H, V]     16-byte aligned
 *   q, k, p, v     16-byte aligned; beta 2-byte, g 4-byte aligned
 * cache_indices, cu_seqlens, workspace (gdn_prefill_workspace_size(num_seqs, T, H, H, K, V,
 * chunk_size)), dev_status, chunk_size and the checks are those of gdn_prefill_chunked.
 * Supported: K = V = 128, chunk_size 64 or 128.
 */
gdn_status comba_prefill_chunked(const void* q, const void* k, const void* v, const void* p,
                                 const void* beta, const float* g, float* state_pool, int pool_size,
                                 const int64_t* cache_indices, const int64_t* cu_seqlens, int num_seqs,
                                 int64_t T, int H, int K, int V, int chunk_size, float scale, void* out,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                 gdn_stream_t stream);

/*
 * gdn_prefill_chunked_noalloc -- gdn_prefill_chunked for callers that cannot allocate device memory
 * themselves, for instance code running under a host framework whose allocator owns all device
 * memory, or in a place where calling cudaMalloc is not allowed.  No page has a counterpart: this
 * is a deployment variant, not a different computation.  Same arguments, layouts and results as
 * gdn_prefill_chunked, without the workspace arguments.
 *
 * The workspace is a 64 MiB array of the library's own device memory (a static device variable,
 * which every GPU that loads the library holds until the process exits).  The call allocates and
 * frees nothing:
 *   - Sizes whose header and records (gdn_prefill_workspace_size without the split scratch)
 *     exceed 64 MiB are rejected with GDN_ERR_UNSUPPORTED before anything runs (use
 *     gdn_prefill_chunked then).  About 1,000 (chunk, value head) records fit: for instance
 *     T = 3,000 tokens over a few sequences with Hv = 16.  Long sequences are split only when the
 *     whole gdn_prefill_workspace_size(...) fits.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress, with
 *     that device current) and keeps it; make that first call before any stream capture.  The
 *     address kept is the one in the device's primary context (the CUDA runtime's default), so
 *     every call must run in that context: a caller that makes its own driver-API context on the
 *     same device current (cuCtxCreate, cuCtxPushCurrent) must not use this entry point.
 *   - Every call on a device shares the one array.  Nothing in it has to start at zero: each call
 *     writes everything it reads.  Calls whose kernels overlap on the GPU (different streams, no
 *     ordering between them) race on the array and give undefined results; order them on one stream.
 */
gdn_status gdn_prefill_chunked_noalloc(const void* q, const void* k, const void* v, const void* a,
                                       const void* b, const float* A_log, const float* dt_bias,
                                       float* state_pool, int pool_size,
                                       const int64_t* cache_indices, const int64_t* cu_seqlens,
                                       int num_seqs, int64_t T, int Hk, int Hv, int K, int V,
                                       int chunk_size, float scale, void* out, int32_t* dev_status,
                                       gdn_stream_t stream);

/*
 * gdn_window_fused -- fused decode window over ntok tokens for N independent sequences.
 * [gdn.metal] header comment, per token:
 *     conv: s = h0 w0 + h1 w1 + h2 w2 + x_t w3 (history oldest first), SiLU(s); history shifts;
 *     q, k: x / sqrt(sum x^2 + eps) (the page's rsqrt(sum/128 + eps/128) / sqrt(128));
 *     gate = exp(softplus(alpha + dt) ssm_a) (softplus threshold 20);  beta = sigmoid(beta_raw);
 *     kv_j = sum_i S[i][j] k_i;  delta_j = (v_j - gate kv_j) beta;  S[i][j] = gate S[i][j] + k_i delta_j;
 *     o_j = (sum_i S[i][j] q_i) / sqrt(128);  y_j = o_j rsqrt(mean(o^2) + eps) gamma_j sigmoid(z_j).
 * Value head h reads key head h % h_k.  Head dim is 128; C = (2 h_k + h_v) * 128 channels.  The
 * window is evaluated as one WY-regrouped chunk (the same function up to rounding order); a commit
 * after token k gives bit for bit what a k-token window gives.
 *
 *   state     f32 [N, 128, h_v, 128]  (key row i, head h, value column j)  read; written in place
 *                                     only when committing
 *   hist      f32 [N, C, 3]   conv history, oldest first                    read
 *   hist_out  f32 [N, C, 3]   committed history; must not overlap hist      written only when
 *                                                                           committing
 *   qkv       f32 [N, ntok, C]  q of key head hk at hk*128, k at (h_k+hk)*128, v of head h at
 *                                (2 h_k + h)*128
 *   alpha, beta  f32 [N, ntok, h_v]
 *   z, y      f32 [N, ntok, h_v, 128]
 *   conv_w    f32 [C, 4];  dt, ssm_a  f32 [h_v];  gamma  f32 [128]   shared by all sequences
 *   commit    0: verify (nothing but y written); 1: commit state and history after the last token;
 *             0x100 | k (1 <= k <= ntok): commit after token k (y still computed for all tokens)
 *   eps       1e-6 on the page
 * Supported: 1 <= ntok <= 8, h_k >= 1, h_v >= 1.
 */
gdn_status gdn_window_fused(float* state, const float* hist, float* hist_out, const float* qkv,
                            const float* alpha, const float* beta, const float* z,
                            const float* conv_w, const float* dt, const float* ssm_a,
                            const float* gamma, float* y, int N, int h_k, int h_v, int ntok,
                            unsigned commit, float eps, gdn_stream_t stream);

/*
 * gdn_prefill_set_wait_limit -- bound every device-side wait of the prefill kernels
 * (gdn_prefill_chunked, _f16, _noalloc and comba_prefill_chunked: the chunk preparation and the
 * chunk recurrence) to `polls` polls of its mbarrier instead of the built-in limits (seconds of
 * waiting).  No page has a counterpart: this is the knob of the failure path.  A wait that runs out
 * sets GDN_STATUS_TIMEOUT in the call's dev_status and its CTA stops after one more bounded wait
 * for the copies and products it has in flight, so the call returns with that status and partial
 * results (the state of a CTA that gave up is not written back; outputs may be partly written) and
 * the device stays usable.  A limit small enough to run out on a healthy GPU (say 1) is for tests
 * of that path; a caller may also use a tighter limit than the default as a watchdog.  0 restores
 * the built-in limits.  Process-wide; it applies to calls launched after it returns.
 */
void gdn_prefill_set_wait_limit(uint32_t polls);

/* Static description of a status code. */
const char* gdn_status_string(gdn_status status);

/* Detail of the last failure on the calling thread ("" if none). */
const char* gdn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
