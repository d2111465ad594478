/*
 * fp64 CPU oracle for the context-parallel Gated DeltaNet forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may call this code.  It shares no source with the CUDA
 * library and is deliberately plain: every function is the defining formula
 * written out, in the order the source pages state it, with no blocking or
 * fusion.
 *
 * Sources (web pages):
 *   [FLA-CP]  flash-linear-attention, fla/ops/cp/context.py,
 *             get_cp_cu_seqlens, steps 1-5 (shard plan)
 *   [HP-CP]   hyper-parallel, linear_attention_context_parallel.py:
 *             _causal_conv1d_with_cp_halo (conv + SiLU with the previous
 *             shard's halo), _l2norm_torch, _prepare_gdn_chunks_for_summary /
 *             _run_prepared_gdn_chunks (the chunked gated delta rule, which is
 *             exact for the token recurrence below),
 *             _compute_gdn_state_summary_from_prepared (state_out =
 *             M @ state_in + S) and _merge_gdn_prefix_state_summaries_torch
 *             (the prefix merge over shards); the backward of the token
 *             recurrence (reverse mode, the state gradient flowing back the
 *             way _RecvInitialStateP2PFunction / _SendFinalStateP2PFunction
 *             send it).
 *
 * Layouts (all dense, row-major, fp64 unless stated):
 *   q, k [T, Hk, K]; v [T, Hv, V]; g, beta [T, Hv]; o [T, Hv, V]
 *   h0, h_final [N, Hv, K, V]; M [.., Hv, K, K]; summaries N [.., Hv, K, V]
 *   v-head h reads qk-head h / (Hv / Hk)   (repeat_interleave on the head dim)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Shard plan  [FLA-CP] get_cp_cu_seqlens                                    */
/* ------------------------------------------------------------------------ */

/* number of a[0..n) with a[i] <= x  (torch.searchsorted(a, x, side='right')) */
static int64_t ss_right(const int64_t *a, int64_t n, int64_t x) {
    int64_t c = 0;
    for (int64_t i = 0; i < n; ++i) c += (a[i] <= x);
    return c;
}
/* number of a[0..n) with a[i] < x   (torch.searchsorted(a, x, side='left')) */
static int64_t ss_left(const int64_t *a, int64_t n, int64_t x) {
    int64_t c = 0;
    for (int64_t i = 0; i < n; ++i) c += (a[i] < x);
    return c;
}

/*
 * Plan of shard `rank` of `world` for cu[0..n_seqs].  Writes the local
 * cu_seqlens (deduplicated) into local_cu (capacity n_seqs + 1) and returns
 * its length.  fields[0..8) = start_seq_idx, end_seq_idx, pre_num_ranks,
 * post_num_ranks, is_first_rank, is_last_rank, pre_num_conv_tokens, part_len.
 * Assumes cu is non-decreasing, cu[0] = 0 and total % world == 0.
 */
int64_t orc_plan_shard(const int64_t *cu, int64_t n_seqs, int64_t world, int64_t rank,
                       int64_t *local_cu, int64_t *fields, int64_t *local_seq) {
    /* step 2: total tokens and this rank's range */
    int64_t total = cu[n_seqs];
    int64_t part_len = total / world;
    int64_t rank_start = part_len * rank;
    int64_t rank_end = rank_start + part_len;
    /* step 3: first sequence whose end > rank_start; first whose start >= rank_end */
    int64_t start_seq_idx = ss_right(cu + 1, n_seqs, rank_start);
    int64_t end_seq_idx = ss_left(cu, n_seqs, rank_end);
    /* step 4: clamp the slice, shift to local coordinates, drop repeats */
    int64_t n_local = 0;
    for (int64_t i = start_seq_idx; i <= end_seq_idx; ++i) {
        int64_t c = cu[i];
        if (c < rank_start) c = rank_start;
        if (c > rank_end) c = rank_end;
        c -= rank_start;
        if (n_local == 0 || local_cu[n_local - 1] != c) local_cu[n_local++] = c;
    }
    /* step 5: first/last rank metadata */
    int64_t first_seq_global_start = cu[start_seq_idx];
    int64_t last_seq_global_end = cu[end_seq_idx];
    int64_t pre_conv = rank_start - first_seq_global_start;
    if (pre_conv < 0) pre_conv = 0;
    int64_t first_rank_of_first_seq = first_seq_global_start / part_len;
    int64_t last_rank_of_last_seq = (last_seq_global_end - 1) / part_len;
    fields[0] = start_seq_idx;
    fields[1] = end_seq_idx;
    fields[2] = rank - first_rank_of_first_seq;
    fields[3] = last_rank_of_last_seq - rank;
    fields[4] = (rank == first_rank_of_first_seq);
    fields[5] = (rank == last_rank_of_last_seq);
    fields[6] = pre_conv;
    fields[7] = part_len;
    /* the global sequence of each local segment: the one that holds the
       segment's first token (largest i with cu[i] <= that token) */
    for (int64_t j = 0; j + 1 < n_local; ++j)
        local_seq[j] = ss_right(cu + 1, n_seqs, rank_start + local_cu[j]);
    return n_local;
}

/* ------------------------------------------------------------------------ */
/* Causal depthwise conv1d + SiLU with a halo  [HP-CP] _causal_conv1d_with_cp_halo */
/* ------------------------------------------------------------------------ */

/*
 * y[t, c] = silu(bias[c] + sum_{j<Kc} w[c, j] * xin(t - (Kc-1) + j, c))
 * where xin(s, c) is x[s, c] when s lies in the same sequence as t, the halo
 * row for the first sequence's missing history (halo [Kc-1, C]; its last
 * row is the token immediately before cu[0]; only the last `halo_len` rows
 * are present), and 0 otherwise.  x has row stride ldx; y is [T, C].
 */
void orc_conv_silu(const double *x, int64_t ldx, int64_t T, int64_t C,
                   const double *w, const double *bias, int64_t Kc,
                   const int64_t *cu, int64_t n_seqs,
                   const double *halo, int64_t halo_len, double *y) {
    (void)T;
    for (int64_t n = 0; n < n_seqs; ++n) {
        int64_t s0 = cu[n], s1 = cu[n + 1];
#pragma omp parallel for schedule(static)
        for (int64_t t = s0; t < s1; ++t) {
            for (int64_t c = 0; c < C; ++c) {
                double acc = bias ? bias[c] : 0.0;
                for (int64_t j = 0; j < Kc; ++j) {
                    int64_t s = t - (Kc - 1) + j;
                    double xv = 0.0;
                    if (s >= s0) {
                        xv = x[s * ldx + c];
                    } else if (n == 0 && halo && s0 - s <= halo_len) {
                        xv = halo[(Kc - 1 - (s0 - s)) * C + c];
                    }
                    acc += w[c * Kc + j] * xv;
                }
                y[t * C + c] = acc / (1.0 + exp(-acc));   /* silu(a) = a * sigmoid(a) */
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Gated delta rule, token by token                                          */
/* ------------------------------------------------------------------------ */

/* x * rsqrt(sum(x^2) + 1e-6)  ([HP-CP] _l2norm_torch) */
static void l2norm(const double *x, double *out, int64_t K) {
    double ss = 0.0;
    for (int64_t i = 0; i < K; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss + 1e-6);
    for (int64_t i = 0; i < K; ++i) out[i] = x[i] * r;
}

/*
 * Per sequence n and v-head h, from S = h0[n, h] (or 0), for each token t:
 *   S <- exp(g_t) S                       (gate)
 *   u <- v_t - S^T k_t                    (delta-rule residual)
 *   S <- S + beta_t k_t u^T               (rank-1 write)
 *   o_t <- S^T (scale q_t)                (read with the updated state)
 * i.e. S_t = a_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T and
 * o_t = S_t^T q~_t, which the chunked WY/UT form of [HP-CP] computes exactly.
 * With l2norm != 0, q_t and k_t are first replaced by x * rsqrt(|x|^2 + 1e-6).
 * h_final[n, h] = S after the sequence's last token (h0 or 0 for an empty one).
 * o / h_final may be NULL.
 */
void orc_gdn_forward(const double *q, const double *k, const double *v,
                     const double *g, const double *beta, const double *h0,
                     const int64_t *cu, int64_t n_seqs, int64_t Hk, int64_t Hv,
                     int64_t K, int64_t V, double scale, int l2,
                     double *o, double *h_final) {
    int64_t G = Hv / Hk;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int64_t n = 0; n < n_seqs; ++n) {
        for (int64_t h = 0; h < Hv; ++h) {
            int64_t hk = h / G;
            double *S = (double *)malloc(sizeof(double) * K * V);
            double *u = (double *)malloc(sizeof(double) * V);
            double *kt = (double *)malloc(sizeof(double) * K);
            double *qt = (double *)malloc(sizeof(double) * K);
            if (h0) memcpy(S, h0 + ((n * Hv + h) * K) * V, sizeof(double) * K * V);
            else memset(S, 0, sizeof(double) * K * V);
            for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
                const double *kr = k + (t * Hk + hk) * K;
                const double *qr = q + (t * Hk + hk) * K;
                if (l2) { l2norm(kr, kt, K); l2norm(qr, qt, K); }
                else { memcpy(kt, kr, sizeof(double) * K); memcpy(qt, qr, sizeof(double) * K); }
                for (int64_t i = 0; i < K; ++i) qt[i] *= scale;
                double a = exp(g[t * Hv + h]);
                double b = beta[t * Hv + h];
                for (int64_t i = 0; i < K * V; ++i) S[i] *= a;
                const double *vr = v + (t * Hv + h) * V;
                for (int64_t j = 0; j < V; ++j) u[j] = vr[j];
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t j = 0; j < V; ++j) u[j] -= S[i * V + j] * kt[i];
                for (int64_t i = 0; i < K; ++i) {
                    double bk = b * kt[i];
                    for (int64_t j = 0; j < V; ++j) S[i * V + j] += bk * u[j];
                }
                if (o) {
                    double *orow = o + (t * Hv + h) * V;
                    for (int64_t j = 0; j < V; ++j) orow[j] = 0.0;
                    for (int64_t i = 0; i < K; ++i)
                        for (int64_t j = 0; j < V; ++j) orow[j] += S[i * V + j] * qt[i];
                }
            }
            if (h_final) memcpy(h_final + ((n * Hv + h) * K) * V, S, sizeof(double) * K * V);
            free(S); free(u); free(kt); free(qt);
        }
    }
}

/*
 * Affine summary of each segment [cu[n], cu[n+1]) and v-head h:
 *   state_out = M state_in + N     ([HP-CP] _compute_gdn_state_summary_from_prepared)
 * M = A_last ... A_first with A_t = exp(g_t) (I - beta_t k_t k_t^T)  [K, K]
 * N = the state reached from a zero state                           [K, V]
 * Each factor is applied as A_t X = exp(g_t) (X - beta_t k_t (k_t^T X)).
 */
void orc_gdn_summary(const double *k, const double *v, const double *g, const double *beta,
                     const int64_t *cu, int64_t n_seqs, int64_t Hk, int64_t Hv,
                     int64_t K, int64_t V, int l2, double *Mout, double *Nout) {
    int64_t G = Hv / Hk;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int64_t n = 0; n < n_seqs; ++n) {
        for (int64_t h = 0; h < Hv; ++h) {
            int64_t hk = h / G;
            double *M = Mout + ((n * Hv + h) * K) * K;
            double *Nn = Nout + ((n * Hv + h) * K) * V;
            double *kt = (double *)malloc(sizeof(double) * K);
            double *r = (double *)malloc(sizeof(double) * (K > V ? K : V));
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < K; ++j) M[i * K + j] = (i == j);
            memset(Nn, 0, sizeof(double) * K * V);
            for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
                const double *kr = k + (t * Hk + hk) * K;
                if (l2) l2norm(kr, kt, K);
                else memcpy(kt, kr, sizeof(double) * K);
                double a = exp(g[t * Hv + h]);
                double b = beta[t * Hv + h];
                const double *vr = v + (t * Hv + h) * V;
                /* M <- A_t M */
                for (int64_t j = 0; j < K; ++j) r[j] = 0.0;
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t j = 0; j < K; ++j) r[j] += kt[i] * M[i * K + j];
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t j = 0; j < K; ++j)
                        M[i * K + j] = a * (M[i * K + j] - b * kt[i] * r[j]);
                /* N <- A_t N + beta_t k_t v_t^T */
                for (int64_t j = 0; j < V; ++j) r[j] = 0.0;
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t j = 0; j < V; ++j) r[j] += kt[i] * Nn[i * V + j];
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t j = 0; j < V; ++j)
                        Nn[i * V + j] = a * (Nn[i * V + j] - b * kt[i] * r[j]) + b * kt[i] * vr[j];
            }
            free(kt); free(r);
        }
    }
}

/*
 * Prefix merge over P shards ([HP-CP] _merge_gdn_prefix_state_summaries_torch),
 * for every v-head: state(0) = S0 (or 0); state(r) = M[r-1] state(r-1) + N[r-1].
 * M [P, Hv, K, K], N [P, Hv, K, V], S_in [P, Hv, K, V] (state entering shard r).
 */
void orc_state_combine(const double *M, const double *N, const double *S0,
                       int64_t P, int64_t Hv, int64_t K, int64_t V, double *S_in) {
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < Hv; ++h) {
        double *cur = (double *)malloc(sizeof(double) * K * V);
        double *nxt = (double *)malloc(sizeof(double) * K * V);
        if (S0) memcpy(cur, S0 + h * K * V, sizeof(double) * K * V);
        else memset(cur, 0, sizeof(double) * K * V);
        for (int64_t r = 0; r < P; ++r) {
            memcpy(S_in + ((r * Hv + h) * K) * V, cur, sizeof(double) * K * V);
            if (r == P - 1) break;
            const double *Mr = M + ((r * Hv + h) * K) * K;
            const double *Nr = N + ((r * Hv + h) * K) * V;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int64_t m = 0; m < K; ++m) acc += Mr[i * K + m] * cur[m * V + j];
                    nxt[i * V + j] = acc + Nr[i * V + j];
                }
            double *tmp = cur; cur = nxt; nxt = tmp;
        }
        free(cur); free(nxt);
    }
}

/* ------------------------------------------------------------------------ */
/* The steps around the path in the wrappers' forward ([HP-CP])              */
/* ------------------------------------------------------------------------ */

/*
 * Gates from the raw projections, as the P2P / all-gather wrappers' forward
 * forms them before the delta rule:
 *   beta = sigmoid(b)
 *   g    = -exp(A_log[h]) * softplus(a + dt_bias[h]),  softplus(x) = log(1 + e^x)
 * a, b [T, Hv]; A_log, dt_bias [Hv]; g, beta [T, Hv].
 */
void orc_gates(const double *a, const double *b, const double *A_log, const double *dt_bias,
               int64_t T, int64_t Hv, double *g, double *beta) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < Hv; ++h) {
            const int64_t i = t * Hv + h;
            const double x = a[i] + dt_bias[h];
            const double sp = x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
            g[i] = -exp(A_log[h]) * sp;
            beta[i] = 1.0 / (1.0 + exp(-b[i]));
        }
}

/*
 * The gated RMS norm the wrappers apply to the attention output before the
 * output projection (base.norm(core_attn_out, z) on rows of head_v_dim):
 * for every row r of D values,
 *   y[r] = w * o[r] / sqrt(mean(o[r]^2) + eps) * silu(z[r]),  silu(x) = x / (1 + e^-x)
 * o, z, y [rows, D]; w [D].
 */
void orc_gated_rmsnorm(const double *o, const double *z, const double *w, double eps,
                       int64_t rows, int64_t D, double *y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int64_t d = 0; d < D; ++d) ss += o[r * D + d] * o[r * D + d];
        const double inv = 1.0 / sqrt(ss / (double)D + eps);
        for (int64_t d = 0; d < D; ++d) {
            const double zz = z[r * D + d];
            y[r * D + d] = w[d] * (o[r * D + d] * inv) * (zz / (1.0 + exp(-zz)));
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Backward of the token recurrence of orc_gdn_forward (reverse mode)        */
/* ------------------------------------------------------------------------ */

/*
 * Given the loss gradients dout [T, Hv, V] (w.r.t. o) and dh_final
 * [N, Hv, K, V] (w.r.t. the final states, or NULL), the gradients w.r.t.
 * q, k [T, Hk, K] (summed over the value heads that share a q/k head),
 * v [T, Hv, V], g, beta [T, Hv] and h0 [N, Hv, K, V].  Per token, with
 * a = e^g, P = a S_prev, u = v - P^T k, S = P + beta k u^T, o = S^T (scale q),
 * walked backwards with the state gradient dS:
 *   dq = scale S do;               dS += scale q do^T
 *   dbeta = k . (dS u);            dk = beta dS u;    du = beta dS^T k;  dv = du
 *   dP = dS - k du^T;              dk -= P du;        dg = <P, dP>;      dS_prev = a dP
 * (q, k here are the normalised vectors when l2 is set; their gradients are
 * carried back through x / sqrt(|x|^2 + 1e-6) at the end.)  The states before
 * each token are recomputed chunk by chunk (64 tokens) from states kept at
 * the chunk starts.
 */
static void l2norm_back(const double *x, const double *dxn, double *dx, int64_t K) {
    double ss = 0.0, xd = 0.0;
    for (int64_t i = 0; i < K; ++i) { ss += x[i] * x[i]; xd += x[i] * dxn[i]; }
    const double r = 1.0 / sqrt(ss + 1e-6);
    for (int64_t i = 0; i < K; ++i) dx[i] = r * dxn[i] - r * r * r * xd * x[i];
}

void orc_gdn_backward(const double *q, const double *k, const double *v,
                      const double *g, const double *beta, const double *h0,
                      const int64_t *cu, int64_t n_seqs, int64_t Hk, int64_t Hv,
                      int64_t K, int64_t V, double scale, int l2,
                      const double *dout, const double *dh_final,
                      double *dq, double *dk, double *dv, double *dg, double *dbeta, double *dh0) {
    const int64_t G = Hv / Hk, C = 64;
    const int64_t T = cu[n_seqs];
    memset(dq, 0, sizeof(double) * T * Hk * K);
    memset(dk, 0, sizeof(double) * T * Hk * K);
    /* a q/k head's gradient collects its G value heads: one task per (n, hk) */
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int64_t n = 0; n < n_seqs; ++n) {
        for (int64_t hk = 0; hk < Hk; ++hk) {
            const int64_t t0 = cu[n], L = cu[n + 1] - cu[n];
            const int64_t nch = (L + C - 1) / C;
            double *chk = (double *)malloc(sizeof(double) * K * V * (nch > 0 ? nch : 1));
            double *Sp = (double *)malloc(sizeof(double) * K * V * C);   /* states before each token of a chunk */
            double *S = (double *)malloc(sizeof(double) * K * V);
            double *dS = (double *)malloc(sizeof(double) * K * V);
            double *kn = (double *)malloc(sizeof(double) * K * (L > 0 ? L : 1));
            double *qn = (double *)malloc(sizeof(double) * K * (L > 0 ? L : 1));
            double *u = (double *)malloc(sizeof(double) * V);
            double *du = (double *)malloc(sizeof(double) * V);
            double *w1 = (double *)malloc(sizeof(double) * K);
            double *w2 = (double *)malloc(sizeof(double) * K);
            double *dqn = (double *)calloc((size_t)K * (L > 0 ? L : 1), sizeof(double));
            double *dkn = (double *)calloc((size_t)K * (L > 0 ? L : 1), sizeof(double));
            for (int64_t j = 0; j < L; ++j) {
                const double *kr = k + ((t0 + j) * Hk + hk) * K, *qr = q + ((t0 + j) * Hk + hk) * K;
                if (l2) { l2norm(kr, kn + j * K, K); l2norm(qr, qn + j * K, K); }
                else { memcpy(kn + j * K, kr, sizeof(double) * K); memcpy(qn + j * K, qr, sizeof(double) * K); }
            }
            for (int64_t h = hk * G; h < (hk + 1) * G; ++h) {
                /* forward: the state at every chunk start */
                if (h0) memcpy(S, h0 + ((n * Hv + h) * K) * V, sizeof(double) * K * V);
                else memset(S, 0, sizeof(double) * K * V);
                for (int64_t j = 0; j < L; ++j) {
                    if (j % C == 0) memcpy(chk + (j / C) * K * V, S, sizeof(double) * K * V);
                    const int64_t t = t0 + j;
                    const double a = exp(g[t * Hv + h]), b = beta[t * Hv + h];
                    const double *kt = kn + j * K, *vr = v + (t * Hv + h) * V;
                    for (int64_t i = 0; i < K * V; ++i) S[i] *= a;
                    for (int64_t c = 0; c < V; ++c) {
                        double s = vr[c];
                        for (int64_t i = 0; i < K; ++i) s -= S[i * V + c] * kt[i];
                        u[c] = s;
                    }
                    for (int64_t i = 0; i < K; ++i)
                        for (int64_t c = 0; c < V; ++c) S[i * V + c] += b * kt[i] * u[c];
                }
                /* backward, chunk by chunk from the last */
                if (dh_final) memcpy(dS, dh_final + ((n * Hv + h) * K) * V, sizeof(double) * K * V);
                else memset(dS, 0, sizeof(double) * K * V);
                for (int64_t ch = nch - 1; ch >= 0; --ch) {
                    const int64_t j0 = ch * C, j1 = (j0 + C < L) ? j0 + C : L;
                    memcpy(S, chk + ch * K * V, sizeof(double) * K * V);
                    for (int64_t j = j0; j < j1; ++j) {   /* recompute the states before each token */
                        memcpy(Sp + (j - j0) * K * V, S, sizeof(double) * K * V);
                        const int64_t t = t0 + j;
                        const double a = exp(g[t * Hv + h]), b = beta[t * Hv + h];
                        const double *kt = kn + j * K, *vr = v + (t * Hv + h) * V;
                        for (int64_t i = 0; i < K * V; ++i) S[i] *= a;
                        for (int64_t c = 0; c < V; ++c) {
                            double s = vr[c];
                            for (int64_t i = 0; i < K; ++i) s -= S[i * V + c] * kt[i];
                            u[c] = s;
                        }
                        for (int64_t i = 0; i < K; ++i)
                            for (int64_t c = 0; c < V; ++c) S[i * V + c] += b * kt[i] * u[c];
                    }
                    for (int64_t j = j1 - 1; j >= j0; --j) {
                        const int64_t t = t0 + j;
                        const double a = exp(g[t * Hv + h]), b = beta[t * Hv + h];
                        const double *kt = kn + j * K, *qt = qn + j * K, *vr = v + (t * Hv + h) * V;
                        const double *dor = dout + (t * Hv + h) * V;
                        const double *Sprev = Sp + (j - j0) * K * V;
                        /* u from P = a S_prev */
                        for (int64_t c = 0; c < V; ++c) {
                            double s = vr[c];
                            for (int64_t i = 0; i < K; ++i) s -= a * Sprev[i * V + c] * kt[i];
                            u[c] = s;
                        }
                        /* dq = scale S do with S = P + beta k u^T */
                        double udo = 0.0;
                        for (int64_t c = 0; c < V; ++c) udo += u[c] * dor[c];
                        for (int64_t i = 0; i < K; ++i) {
                            double s = 0.0;
                            for (int64_t c = 0; c < V; ++c) s += a * Sprev[i * V + c] * dor[c];
                            dqn[j * K + i] += scale * (s + b * kt[i] * udo);
                        }
                        /* the output's contribution to the state gradient */
                        for (int64_t i = 0; i < K; ++i)
                            for (int64_t c = 0; c < V; ++c) dS[i * V + c] += scale * qt[i] * dor[c];
                        /* through S = P + beta k u^T */
                        double db = 0.0;
                        for (int64_t i = 0; i < K; ++i) {
                            double s = 0.0;
                            for (int64_t c = 0; c < V; ++c) s += dS[i * V + c] * u[c];
                            w1[i] = s;                      /* dS u */
                            db += kt[i] * s;
                        }
                        for (int64_t c = 0; c < V; ++c) {
                            double s = 0.0;
                            for (int64_t i = 0; i < K; ++i) s += dS[i * V + c] * kt[i];
                            du[c] = b * s;                  /* beta dS^T k */
                        }
                        dbeta[t * Hv + h] = db;
                        for (int64_t c = 0; c < V; ++c) dv[(t * Hv + h) * V + c] = du[c];
                        /* through u = v - P^T k: dP = dS - k du^T, dk -= P du */
                        for (int64_t i = 0; i < K; ++i) {
                            double s = 0.0;
                            for (int64_t c = 0; c < V; ++c) s += a * Sprev[i * V + c] * du[c];
                            w2[i] = s;
                        }
                        for (int64_t i = 0; i < K; ++i) dkn[j * K + i] += b * w1[i] - w2[i];
                        for (int64_t i = 0; i < K; ++i)
                            for (int64_t c = 0; c < V; ++c) dS[i * V + c] -= kt[i] * du[c];
                        /* through P = a S_prev */
                        double pd = 0.0;
                        for (int64_t i = 0; i < K * V; ++i) pd += a * Sprev[i] * dS[i];
                        dg[t * Hv + h] = pd;
                        for (int64_t i = 0; i < K * V; ++i) dS[i] *= a;
                    }
                }
                if (dh0) memcpy(dh0 + ((n * Hv + h) * K) * V, dS, sizeof(double) * K * V);
            }
            /* q/k gradients of the stored (un-normalised) vectors */
            for (int64_t j = 0; j < L; ++j) {
                const int64_t t = t0 + j;
                double *dqo = dq + (t * Hk + hk) * K, *dko = dk + (t * Hk + hk) * K;
                if (l2) {
                    l2norm_back(q + (t * Hk + hk) * K, dqn + j * K, dqo, K);
                    l2norm_back(k + (t * Hk + hk) * K, dkn + j * K, dko, K);
                } else {
                    memcpy(dqo, dqn + j * K, sizeof(double) * K);
                    memcpy(dko, dkn + j * K, sizeof(double) * K);
                }
            }
            free(chk); free(Sp); free(S); free(dS); free(kn); free(qn); free(u); free(du);
            free(w1); free(w2); free(dqn); free(dkn);
        }
    }
}

int orc_max_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
