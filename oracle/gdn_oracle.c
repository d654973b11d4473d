/*
 * gdn_oracle.c -- plain, slow, obviously sequential CPU oracle for the gated delta-rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  It exists to say what the CUDA library must compute.  The tests, the
 * smoke check and the CPU-baseline leg of the benchmark load it; the product path never does.  It
 * shares no code, header, table or constant with the CUDA path.
 *
 * Rules followed throughout:
 *   - IEEE double precision, built with -ffp-contract=off (no fused multiply-add is introduced).
 *   - One head (one sequence) at a time, one token at a time, the steps in the order the pages give.
 *   - No blocking, fusion or reordering beyond what the definitions state.
 *
 * Sources (page title and section):
 *   [gated_delta.rs]  metaltile-std, src/ffai/gated_delta.rs: module doc "Recurrence per step",
 *                     "Layouts", "DISPATCH INVARIANTS" (GQA map hk = hv / (Hv / Hk)).
 *   [gdn.metal]       regolith, baseline-kernels/gdn.metal: header comment (conv, SiLU, L2 norm, gate,
 *                     recurrence, readout, gated RMSNorm), GdnArgs (commit codes, eps).
 *   [comba spec]      KBench, specs/comba_decode_step.py: spec_md (elementwise form), reference_src.
 *   [gdn_chunkwise]   pymllm, gdn_chunkwise: module doc (sequential recurrence reproduced by WY),
 *                     gdn_extend_chunkwise parameters (raw gate inputs, pool, cache_indices,
 *                     cu_seqlens).
 */
#include "gdn_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* softplus with the pages' threshold: x > 20 ? x : log(1 + e^x).  [gdn.metal] header comment. */
static double softplus_thr(double x) { return x > 20.0 ? x : log1p(exp(x)); }

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------------------------------------ */
/* GDN decode step.  [gated_delta.rs] module doc "Recurrence per step":                              */
/*   state_decayed = state * g;  kv_mem = sum_dk(state_decayed * k);  delta = (v - kv_mem) * beta;   */
/*   state_new = state_decayed + outer(delta, k);  y = sum_dk(state_new * q)   (times scale here).    */
/* ------------------------------------------------------------------------------------------------ */
void oracle_gdn_decode_head(int Dk, int Dv, const double* S, const double* q, const double* k,
                            const double* v, double g, double beta, double scale, double* S_new,
                            double* y) {
    for (int r = 0; r < Dv; ++r) {
        const double* row = S + (long)r * Dk;
        double* row_new = S_new + (long)r * Dk;
        /* kv_mem[r] = sum_c (g * S[r][c]) * k[c] */
        double kv = 0.0;
        for (int c = 0; c < Dk; ++c) kv += (g * row[c]) * k[c];
        double delta = (v[r] - kv) * beta;
        /* state_new[r][c] = g * S[r][c] + delta * k[c];  y[r] = scale * sum_c state_new[r][c] q[c] */
        double acc = 0.0;
        for (int c = 0; c < Dk; ++c) {
            double s = g * row[c] + delta * k[c];
            row_new[c] = s;
            acc += s * q[c];
        }
        y[r] = scale * acc;
    }
}

int oracle_gdn_decode(int B, int Hk, int Hv, int Dk, int Dv, const double* state, const double* q,
                      const double* k, const double* v, const double* g, const double* beta,
                      double scale, double* state_new, double* y) {
    if (B < 0 || Hk <= 0 || Hv <= 0 || Dk <= 0 || Dv <= 0 || Hv % Hk != 0) return ORACLE_EINVAL;
    const int group = Hv / Hk; /* value heads per key head */
    for (int b = 0; b < B; ++b) {
        for (int hv = 0; hv < Hv; ++hv) {
            const int hk = hv / group; /* [gated_delta.rs] DISPATCH INVARIANTS */
            const long n = (long)b * Hv + hv;
            const long qk = ((long)b * Hk + hk) * Dk;
            oracle_gdn_decode_head(Dk, Dv, state + n * Dv * Dk, q + qk, k + qk, v + n * Dv, g[n],
                                   beta[n], scale, state_new + n * Dv * Dk, y + n * Dv);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------------ */
/* Comba decode step.  [comba spec] spec_md, elementwise form (i indexes K, j indexes V):            */
/*   S[i,j] <- exp(g) state[i,j];  u[j] = beta (v[j] - sum_i p[i] S[i,j]);                          */
/*   S_new[i,j] = S[i,j] + k[i] u[j];  o[j] = sum_i (scale q[i]) S_new[i,j].                        */
/* ------------------------------------------------------------------------------------------------ */
void oracle_comba_decode_head(int K, int V, const double* S, const double* q, const double* k,
                              const double* v, const double* p, double beta, double g_log,
                              double scale, double* S_new, double* o) {
    const double gate = exp(g_log);
    double* u = (double*)malloc(sizeof(double) * (size_t)V);
    for (int j = 0; j < V; ++j) {
        double read = 0.0;
        for (int i = 0; i < K; ++i) read += p[i] * (gate * S[(long)i * V + j]);
        u[j] = beta * (v[j] - read);
    }
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
            S_new[(long)i * V + j] = gate * S[(long)i * V + j] + k[i] * u[j];
    for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int i = 0; i < K; ++i) acc += (scale * q[i]) * S_new[(long)i * V + j];
        o[j] = acc;
    }
    free(u);
}

int oracle_comba_decode(int B, int H, int K, int V, const double* state, const double* q,
                        const double* k, const double* v, const double* p, const double* beta,
                        const double* g_log, double scale, double* state_new, double* o) {
    if (B < 0 || H <= 0 || K <= 0 || V <= 0) return ORACLE_EINVAL;
    for (long n = 0; n < (long)B * H; ++n)
        oracle_comba_decode_head(K, V, state + n * K * V, q + n * K, k + n * K, v + n * V,
                                 p + n * K, beta[n], g_log[n], scale, state_new + n * K * V,
                                 o + n * V);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------------ */
/* Comba forward over T tokens.  [comba spec] spec_md: the decode step is the comba-forward task's   */
/* recurrence run for one token, and running the step T times reproduces that task; so each (b, h)  */
/* head carries its state through oracle_comba_decode_head once per token, in token order.           */
/* ------------------------------------------------------------------------------------------------ */
int oracle_comba_forward(int B, int T, int H, int K, int V, const double* state, const double* q,
                         const double* k, const double* v, const double* p, const double* beta,
                         const double* g_log, double scale, double* state_out, double* o) {
    if (B < 0 || T < 0 || H <= 0 || K <= 0 || V <= 0) return ORACLE_EINVAL;
    for (long b = 0; b < B; ++b)
        for (long h = 0; h < H; ++h) {
            double* S = state_out + (b * H + h) * K * V;
            memcpy(S, state + (b * H + h) * K * V, sizeof(double) * (size_t)K * (size_t)V);
            for (long t = 0; t < T; ++t) {
                const long n = (b * T + t) * H + h; /* token t of head (b, h) */
                oracle_comba_decode_head(K, V, S, q + n * K, k + n * K, v + n * V, p + n * K, beta[n],
                                         g_log[n], scale, S, o + n * V);
            }
        }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------------ */
/* Prefill: the sequential recurrence over the tokens of one sequence, one value head.               */
/* Per token ([gdn_chunkwise] gdn_extend_chunkwise parameters; gate form as in [gdn.metal] header):  */
/*   log g = -exp(A_log) softplus(a + dt_bias);  g = exp(log g);  beta = sigmoid(b);                 */
/*   k^ = k / sqrt(|k|^2 + eps);  q^ = scale q / sqrt(|q|^2 + eps);                                  */
/*   then the decode step above on the [V][K] state with (k^, q^, v, g, beta), scale folded in q^.   */
/* ------------------------------------------------------------------------------------------------ */
void oracle_gdn_prefill_unit(long T_n, int Hk, int Hv, int K, int V, int h, const double* q,
                             const double* k, const double* v, const double* a, const double* b,
                             double A_log_h, double dt_bias_h, double eps, double scale, double* S,
                             double* out) {
    const int hk = h / (Hv / Hk);
    double* kn = (double*)malloc(sizeof(double) * (size_t)K);
    double* qn = (double*)malloc(sizeof(double) * (size_t)K);
    for (long t = 0; t < T_n; ++t) {
        const double* qt = q + (t * Hk + hk) * (long)K;
        const double* kt = k + (t * Hk + hk) * (long)K;
        const double* vt = v + (t * Hv + h) * (long)V;
        const double log_g = -exp(A_log_h) * softplus_thr(a[t * Hv + h] + dt_bias_h);
        const double g = exp(log_g);
        const double beta = sigmoid(b[t * Hv + h]);
        double kk = 0.0, qq = 0.0;
        for (int c = 0; c < K; ++c) {
            kk += kt[c] * kt[c];
            qq += qt[c] * qt[c];
        }
        const double rk = 1.0 / sqrt(kk + eps), rq = 1.0 / sqrt(qq + eps);
        for (int c = 0; c < K; ++c) {
            kn[c] = kt[c] * rk;
            qn[c] = scale * (qt[c] * rq);
        }
        oracle_gdn_decode_head(K, V, S, qn, kn, vt, g, beta, 1.0, S, out + (t * Hv + h) * (long)V);
    }
    free(kn);
    free(qn);
}

int oracle_gdn_prefill(int num_seqs, const int64_t* cu_seqlens, const int64_t* cache_indices,
                       int pool_size, long T, int Hk, int Hv, int K, int V, const double* q,
                       const double* k, const double* v, const double* a, const double* b,
                       const double* A_log, const double* dt_bias, double eps, double scale,
                       double* state_pool, double* out, int32_t* status) {
    if (num_seqs < 0 || Hk <= 0 || Hv <= 0 || K <= 0 || V <= 0 || Hv % Hk != 0) return ORACLE_EINVAL;
    int32_t st = 0;
    for (int n = 0; n < num_seqs; ++n) {
        const int64_t bos = cu_seqlens[n], eos = cu_seqlens[n + 1];
        if (bos < 0 || eos < bos || eos > T) {
            st |= ORACLE_STATUS_BAD_SEQLENS;
            continue;
        }
        const int64_t slot = cache_indices[n];
        if (slot < 0 || slot >= pool_size) {
            st |= ORACLE_STATUS_BAD_CACHE_INDEX;
            continue;
        }
        for (int h = 0; h < Hv; ++h) {
            double* S = state_pool + ((slot * Hv + h) * (long)V) * K;
            oracle_gdn_prefill_unit(eos - bos, Hk, Hv, K, V, h, q + bos * Hk * (long)K,
                                    k + bos * Hk * (long)K, v + bos * Hv * (long)V, a + bos * Hv,
                                    b + bos * Hv, A_log[h], dt_bias[h], eps, scale, S,
                                    out + bos * Hv * (long)V);
        }
    }
    if (status) *status |= st;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------------ */
/* Fused decode window of one sequence.  [gdn.metal] header comment, in its order per token t:       */
/*   conv (4 taps over the 3-entry history, oldest first) -> SiLU on every q, k, v channel;          */
/*   q, k: L2 norm (x / sqrt(sum x^2 + eps), the page's two-rounding form in exact arithmetic);      */
/*   gate = exp(softplus(alpha + dt) * ssm_a);  beta = sigmoid(beta_raw);                            */
/*   kv_j = sum_i S[i][j] k_i;  delta_j = (v_j - gate kv_j) beta;  S[i][j] = gate S[i][j] + k_i d_j; */
/*   o_j = (sum_i S[i][j] q_i) / sqrt(D);  y_j = o_j / sqrt(mean(o^2) + eps) * gamma_j sigmoid(z_j). */
/* Value head h reads key head h % h_k.  Commit codes from GdnArgs.                                  */
/* ------------------------------------------------------------------------------------------------ */
static int commit_point(unsigned commit, int ntok) {
    if (commit == 0u) return 0;
    if (commit == 1u) return ntok;
    if ((commit >> 8) == 1u) {
        const int kk = (int)(commit & 0xFFu);
        if (kk >= 1 && kk <= ntok) return kk;
    }
    return -1;
}

int oracle_gdn_window_seq(int D, int h_k, int h_v, int ntok, unsigned commit, double eps,
                          double* state, const double* hist, double* hist_out, const double* qkv,
                          const double* alpha, const double* beta, const double* z,
                          const double* conv_w, const double* dt, const double* ssm_a,
                          const double* gamma, double* y) {
    if (D <= 0 || h_k <= 0 || h_v <= 0 || ntok < 1) return ORACLE_EINVAL;
    const int commit_at = commit_point(commit, ntok);
    if (commit_at < 0) return ORACLE_EINVAL;
    const long C = (long)(2 * h_k + h_v) * D;
    const long SD = (long)D * h_v * D;

    double* S = (double*)malloc(sizeof(double) * (size_t)SD);  /* working state, all heads */
    double* hs = (double*)malloc(sizeof(double) * (size_t)C * 3); /* working history */
    double* act = (double*)malloc(sizeof(double) * (size_t)C);    /* conv + SiLU output of token t */
    double* kn = (double*)malloc(sizeof(double) * (size_t)D);
    double* qn = (double*)malloc(sizeof(double) * (size_t)D);
    double* o = (double*)malloc(sizeof(double) * (size_t)D);
    memcpy(S, state, sizeof(double) * (size_t)SD);
    memcpy(hs, hist, sizeof(double) * (size_t)C * 3);

    for (int t = 0; t < ntok; ++t) {
        /* conv + SiLU, then shift the history by one token */
        for (long ch = 0; ch < C; ++ch) {
            const double x = qkv[(long)t * C + ch];
            const double vals[4] = {hs[ch * 3 + 0], hs[ch * 3 + 1], hs[ch * 3 + 2], x};
            double s = 0.0;
            for (int tap = 0; tap < 4; ++tap) s += vals[tap] * conv_w[ch * 4 + tap];
            act[ch] = s / (1.0 + exp(-s));
            hs[ch * 3 + 0] = hs[ch * 3 + 1];
            hs[ch * 3 + 1] = hs[ch * 3 + 2];
            hs[ch * 3 + 2] = x;
        }
        for (int h = 0; h < h_v; ++h) {
            const int hk = h % h_k;
            const double* qa = act + (long)hk * D;
            const double* ka = act + (long)h_k * D + (long)hk * D;
            const double* va = act + 2L * h_k * D + (long)h * D;
            double kk = 0.0, qq = 0.0;
            for (int i = 0; i < D; ++i) {
                kk += ka[i] * ka[i];
                qq += qa[i] * qa[i];
            }
            const double rk = 1.0 / sqrt(kk + eps), rq = 1.0 / sqrt(qq + eps);
            for (int i = 0; i < D; ++i) {
                kn[i] = ka[i] * rk;
                qn[i] = qa[i] * rq;
            }
            const double gate = exp(softplus_thr(alpha[(long)t * h_v + h] + dt[h]) * ssm_a[h]);
            const double be = sigmoid(beta[(long)t * h_v + h]);
            for (int j = 0; j < D; ++j) {
                double kv = 0.0;
                for (int i = 0; i < D; ++i) kv += S[((long)i * h_v + h) * D + j] * kn[i];
                const double delta = (va[j] - gate * kv) * be;
                double acc = 0.0;
                for (int i = 0; i < D; ++i) {
                    double* s = &S[((long)i * h_v + h) * D + j];
                    *s = gate * (*s) + kn[i] * delta;
                    acc += (*s) * qn[i];
                }
                o[j] = acc / sqrt((double)D);
            }
            double ms = 0.0;
            for (int j = 0; j < D; ++j) ms += o[j] * o[j];
            ms /= (double)D;
            const double rs = 1.0 / sqrt(ms + eps);
            for (int j = 0; j < D; ++j) {
                const long idx = ((long)t * h_v + h) * D + j;
                y[idx] = o[j] * rs * gamma[j] * sigmoid(z[idx]);
            }
        }
        if (t + 1 == commit_at) {
            memcpy(state, S, sizeof(double) * (size_t)SD);
            memcpy(hist_out, hs, sizeof(double) * (size_t)C * 3);
        }
    }
    free(S);
    free(hs);
    free(act);
    free(kn);
    free(qn);
    free(o);
    return ORACLE_OK;
}

int oracle_gdn_window(int N, int D, int h_k, int h_v, int ntok, unsigned commit, double eps,
                      double* state, const double* hist, double* hist_out, const double* qkv,
                      const double* alpha, const double* beta, const double* z,
                      const double* conv_w, const double* dt, const double* ssm_a,
                      const double* gamma, double* y) {
    if (N < 0) return ORACLE_EINVAL;
    const long C = (long)(2 * h_k + h_v) * D;
    const long SD = (long)D * h_v * D;
    for (int n = 0; n < N; ++n) {
        int rc = oracle_gdn_window_seq(D, h_k, h_v, ntok, commit, eps, state + n * SD,
                                       hist + n * C * 3, hist_out + n * C * 3, qkv + n * ntok * C,
                                       alpha + (long)n * ntok * h_v, beta + (long)n * ntok * h_v,
                                       z + (long)n * ntok * h_v * D, conv_w, dt, ssm_a, gamma,
                                       y + (long)n * ntok * h_v * D);
        if (rc != ORACLE_OK) return rc;
    }
    return ORACLE_OK;
}
