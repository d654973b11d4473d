/*
 * gdn_oracle.h -- declarations of the plain CPU oracle for the gated delta-rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This header and gdn_oracle.c are used by the test-suite, by the smoke
 * check and by the CPU-baseline leg of the benchmark, and by nothing else.  The CUDA library
 * (gated_deltanet_delta_gb300/csrc) neither includes this header nor links this code, and this code
 * includes nothing from it.
 *
 * All arithmetic is IEEE double precision.  All arrays are dense, row-major and contiguous; every
 * floating-point input is given as double (bf16 and fp32 inputs are widened exactly by the caller).
 * Sources cited beside each function are the pages' titles and sections:
 *   [gated_delta.rs]   metaltile-std, src/ffai/gated_delta.rs (decode and multi-token Metal kernels)
 *   [gdn.metal]        regolith, baseline-kernels/gdn.metal (fused decode window)
 *   [comba spec]       KBench, specs/comba_decode_step.py (Comba decode-step task spec)
 *   [gdn_chunkwise]    pymllm, layers/attention/gdn_chunkwise (chunkwise WY prefill docs)
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes of the oracle (0 = ok). */
#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)

/* Bits of the per-call status word written by oracle_gdn_prefill (same meaning as the library's). */
#define ORACLE_STATUS_BAD_CACHE_INDEX 1
#define ORACLE_STATUS_BAD_SEQLENS 2

/* GDN decode step of one value head.  [gated_delta.rs] module doc "Recurrence per step".
 * S, S_new: [Dv][Dk] (Dk contiguous; may alias).  q, k: [Dk].  v, y: [Dv].  g: linear gate.
 * y[r] = scale * sum_c S_new[r][c] q[c]  (scale = 1 reproduces the page, which has no scale). */
void oracle_gdn_decode_head(int Dk, int Dv, const double* S, const double* q, const double* k,
                            const double* v, double g, double beta, double scale, double* S_new,
                            double* y);

/* GDN decode step of a batch.  [gated_delta.rs] module doc "Layouts":
 * state [B][Hv][Dv][Dk], q,k [B][Hk][Dk], v,y [B][Hv][Dv], g,beta [B][Hv];
 * value head hv reads key head hv / (Hv / Hk).  Returns ORACLE_EINVAL if Hv % Hk != 0. */
int oracle_gdn_decode(int B, int Hk, int Hv, int Dk, int Dv, const double* state, const double* q,
                      const double* k, const double* v, const double* g, const double* beta,
                      double scale, double* state_new, double* y);

/* Comba decode step of one head.  [comba spec] spec_md and reference_src.
 * S, S_new: [K][V] (V contiguous; may alias).  q, k, p: [K].  v, o: [V].  g_log: log-decay. */
void oracle_comba_decode_head(int K, int V, const double* S, const double* q, const double* k,
                              const double* v, const double* p, double beta, double g_log,
                              double scale, double* S_new, double* o);

/* Comba decode step of a batch: state [B][H][K][V], q,k,p [B][H][K], v,o [B][H][V], beta,g [B][H]. */
int oracle_comba_decode(int B, int H, int K, int V, const double* state, const double* q,
                        const double* k, const double* v, const double* p, const double* beta,
                        const double* g_log, double scale, double* state_new, double* o);

/* Comba forward over T tokens, [comba spec] spec_md ("running this step T times reproduces" the
 * comba-forward task): state [B][H][K][V] in, state_out [B][H][K][V] out (no aliasing);
 * q,k,p [B][T][H][K], v,o [B][T][H][V], beta,g_log [B][T][H]. */
int oracle_comba_forward(int B, int T, int H, int K, int V, const double* state, const double* q,
                         const double* k, const double* v, const double* p, const double* beta,
                         const double* g_log, double scale, double* state_out, double* o);

/* Sequential prefill of one (sequence, value head) unit: the recurrence that the chunkwise WY form
 * reproduces ([gdn_chunkwise] module doc), with the gates derived from the raw inputs
 * ([gdn_chunkwise] gdn_extend_chunkwise parameters a, b, A_log, dt_bias).
 * q, k point at the sequence's first token of [T][Hk][K]; v at [T][Hv][V]; a, b at [T][Hv];
 * out at [T][Hv][V].  S: [V][K] state of value head h (in/out).  Key head = h / (Hv / Hk). */
void oracle_gdn_prefill_unit(long T_n, int Hk, int Hv, int K, int V, int h, const double* q,
                             const double* k, const double* v, const double* a, const double* b,
                             double A_log_h, double dt_bias_h, double eps, double scale, double* S,
                             double* out);

/* Varlen prefill over a pooled state.  state_pool [pool][Hv][V][K] is updated in place; out is
 * [T][Hv][V].  A sequence whose slot is outside [0, pool) or whose bounds are malformed
 * (cu_seqlens decreasing or beyond T) is skipped and flagged in *status. */
int oracle_gdn_prefill(int num_seqs, const int64_t* cu_seqlens, const int64_t* cache_indices,
                       int pool_size, long T, int Hk, int Hv, int K, int V, const double* q,
                       const double* k, const double* v, const double* a, const double* b,
                       const double* A_log, const double* dt_bias, double eps, double scale,
                       double* state_pool, double* out, int32_t* status);

/* Fused decode window of one sequence.  [gdn.metal] header comment and GdnArgs.
 * D: head dim (128 on the page).  C = (2 h_k + h_v) D channels.
 * state [D][h_v][D] (key row i, head h, value column j); hist, hist_out [C][3] oldest first;
 * qkv [ntok][C]; alpha, beta [ntok][h_v]; z, y [ntok][h_v][D]; conv_w [C][4]; dt, ssm_a [h_v];
 * gamma [D].  commit: 0 verify, 1 commit after the last token, 0x100|k commit after token k.
 * Returns ORACLE_EINVAL for a commit code outside those forms. */
int oracle_gdn_window_seq(int D, int h_k, int h_v, int ntok, unsigned commit, double eps,
                          double* state, const double* hist, double* hist_out, const double* qkv,
                          const double* alpha, const double* beta, const double* z,
                          const double* conv_w, const double* dt, const double* ssm_a,
                          const double* gamma, double* y);

/* The same for N sequences, N outermost in every per-sequence array (weights are shared). */
int oracle_gdn_window(int N, int D, int h_k, int h_v, int ntok, unsigned commit, double eps,
                      double* state, const double* hist, double* hist_out, const double* qkv,
                      const double* alpha, const double* beta, const double* z,
                      const double* conv_w, const double* dt, const double* ssm_a,
                      const double* gamma, double* y);

#ifdef __cplusplus
}
#endif

#endif /* GDN_ORACLE_H */
