/*
 * kda_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU oracle for Kimi Delta Attention (KDA).  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load
 * it; the CUDA library never calls it and shares no code with it.
 *
 * What it computes is the explicit token-by-token recurrence that
 * "[kimi k3] add eager reference model with FSDP2" (torchtitan PR #4025,
 * Summary and the "Addresses the review feedback" note) keeps as the
 * numerical reference for the fused chunk_kda kernel:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * with the three in-kernel prologues that the same note and the
 * hyper-parallel "KDA context-parallel executors" page (`_run_local_kda`,
 * flags use_qk_l2norm_in_kernel / use_gate_in_kernel /
 * use_beta_sigmoid_in_kernel) switch on:
 *
 *   - q, k L2-normalised per head:   x / sqrt(|x|^2 + eps), eps = 1e-6
 *   - beta = sigmoid(beta_raw)
 *   - the lower-bounded ("safe") gate built from a_log [H], dt_bias [H*K]
 *     and a negative lower_bound (`_run_local_kda`, `_validate_projected_inputs`):
 *         g     = lower_bound * sigmoid(exp(a_log_h) * (g_raw + dt_bias_{h,c}))
 *         alpha = exp(g)
 *     The pages name these ingredients but never print the formula; this is
 *     the plainest reading that uses all three and keeps g in (lower_bound, 0).
 *   - the unbounded gate the same page keeps behind `safe_gate=False` (the
 *     torchtitan note compares kernel and recurrence under each of the two
 *     gate activations), gate kind 1:
 *         g     = -exp(a_log_h) * softplus(g_raw + dt_bias_{h,c})
 *     Also unprinted: the plainest form over the same ingredients that keeps
 *     g < 0 without a lower bound (a_log as a log-rate, dt_bias as the bias
 *     of a softplus step size).  lower_bound is then unused.
 *
 * Packed documents: nemo_automodel `kimi_k3.cp` ("segment_cu_seqlens",
 * "doc_ids_from_cu_seqlens"): every [cu[n], cu[n+1]) segment is its own
 * recurrence, started from initial_state[n] (or zero).
 *
 * Backward is reverse mode of the same loop, with the state checkpointed
 * every 64 tokens and recomputed inside each 64-token block.
 *
 * Layouts (token-first, as in `_validate_projected_inputs`):
 *   q, k [TT, Hk, K]; g_raw [TT, H, K]; v, out, dout [TT, H, V]; beta_raw [TT, H];
 *   a_log [H]; dt_bias [H*K]; states [N, H, K, V].   TT = B*T.
 * H counts value heads and Hk key heads.  The same page's shape checks
 * (`_validate_projected_inputs`) allow num_v_heads to be a multiple of
 * num_k_heads, with the gate, beta, a_log and dt_bias per value head; which
 * key head a value head reads is not printed.  Reading: value head h uses key
 * head h / (H / Hk), i.e. the key heads repeated in consecutive groups (the
 * usual grouped-head order).  dq and dk then sum over the value heads of a
 * group.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_EPS 1e-6
#define ORACLE_CKPT 64

static double sigm(double x) { return 1.0 / (1.0 + exp(-x)); }
/* log(1 + e^x), written so that neither branch overflows */
static double softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

#define ORACLE_GATE_LOWER_BOUNDED 0
#define ORACLE_GATE_SOFTPLUS 1

/* Segment boundaries: the caller's cu_seqlens, else B rows of T tokens. */
static int64_t seg_begin(const int32_t* cu, int T, int n) { return cu ? (int64_t)cu[n] : (int64_t)n * T; }
static int64_t seg_end(const int32_t* cu, int T, int n) { return cu ? (int64_t)cu[n + 1] : (int64_t)(n + 1) * T; }

/* ---- prologue --------------------------------------------------------- */

/* Gate, one element, of either kind (the readings stated in the header). */
double oracle_gate_value(double g_raw, double a_log, double dt_bias, double lower_bound, int gate)
{
    if (gate == ORACLE_GATE_SOFTPLUS) return -exp(a_log) * softplus(g_raw + dt_bias);
    double z = exp(a_log) * (g_raw + dt_bias);
    return lower_bound * sigm(z);
}

/* Prologue for one (segment, value head h): writes q_hat, k_hat [L,K], g [L,K],
 * beta [L] and the per-token inverse norms rq, rk [L].  q and k come from key
 * head h / (H / Hk). */
static void prologue(int64_t t0, int64_t L, int h, int H, int Hk, int K,
                     const double* q, const double* k, const double* g_raw, const double* beta_raw,
                     const double* a_log, const double* dt_bias, double lb, int gate,
                     double* qh, double* kh, double* g, double* beta, double* rq, double* rk)
{
    const int hk = h / (H / Hk);
    for (int64_t i = 0; i < L; ++i) {
        const int64_t row = (t0 + i) * H + h;
        const int64_t krow = (t0 + i) * Hk + hk;
        const double* qi = q + krow * K;
        const double* ki = k + krow * K;
        double sq = 0.0, sk = 0.0;
        for (int c = 0; c < K; ++c) { sq += qi[c] * qi[c]; sk += ki[c] * ki[c]; }
        rq[i] = 1.0 / sqrt(sq + ORACLE_EPS);
        rk[i] = 1.0 / sqrt(sk + ORACLE_EPS);
        for (int c = 0; c < K; ++c) {
            qh[i * K + c] = qi[c] * rq[i];
            kh[i * K + c] = ki[c] * rk[i];
            g[i * K + c] = oracle_gate_value(g_raw[row * K + c], a_log[h], dt_bias[h * K + c], lb, gate);
        }
        beta[i] = sigm(beta_raw[row]);
    }
}

/* ---- the recurrence ---------------------------------------------------- */

/* One token of the recurrence, in place on S [K,V]:
 *   P = Diag(exp(g)) S;  w = P^T k;  S = P + beta k (v - w)^T;  o = scale S^T q. */
static void step_fwd(int K, int V, double* S, const double* qh, const double* kh, const double* v,
                     const double* g, double beta, double scale, double* o, double* w)
{
    for (int c = 0; c < K; ++c) {
        const double a = exp(g[c]);
        for (int j = 0; j < V; ++j) S[c * V + j] *= a;
    }
    for (int j = 0; j < V; ++j) w[j] = 0.0;
    for (int c = 0; c < K; ++c)
        for (int j = 0; j < V; ++j) w[j] += S[c * V + j] * kh[c];
    for (int c = 0; c < K; ++c)
        for (int j = 0; j < V; ++j) S[c * V + j] += beta * kh[c] * (v[j] - w[j]);
    if (o) {
        for (int j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int c = 0; c < K; ++c) acc += S[c * V + j] * qh[c];
            o[j] = scale * acc;
        }
    }
}

/* Recurrence with the prologue bypassed (tests inject log-decay g and beta).
 * Single segment, single head.  qh, kh, g: [L,K]; v, out: [L,V]; beta: [L];
 * S0, ST: [K,V] (S0 may be NULL = zero state; ST may be NULL). */
int oracle_recurrence(int64_t L, int K, int V, const double* qh, const double* kh, const double* v,
                      const double* g, const double* beta, const double* S0, double scale,
                      double* out, double* ST)
{
    double* S = (double*)calloc((size_t)K * V, sizeof(double));
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!S || !w) { free(S); free(w); return 1; }
    if (S0) memcpy(S, S0, sizeof(double) * (size_t)K * V);
    for (int64_t t = 0; t < L; ++t)
        step_fwd(K, V, S, qh + t * K, kh + t * K, v + t * V, g + t * K, beta[t], scale,
                 out ? out + t * V : NULL, w);
    if (ST) memcpy(ST, S, sizeof(double) * (size_t)K * V);
    free(S); free(w);
    return 0;
}

/* ---- forward ------------------------------------------------------------ */

int oracle_kda_fwd(int B, int T, int H, int Hk, int K, int V, int num_seqs, const int32_t* cu_seqlens,
                   const double* q, const double* k, const double* v, const double* g_raw,
                   const double* beta_raw, const double* a_log, const double* dt_bias,
                   double scale, double lower_bound, int gate, const double* initial_state,
                   double* out, double* final_state, int nthreads)
{
    const int N = cu_seqlens ? num_seqs : B;
    const int pairs = N * H;
    int err = 0;
    (void)nthreads;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
#endif
    for (int p = 0; p < pairs; ++p) {
        const int n = p / H, h = p % H;
        const int64_t t0 = seg_begin(cu_seqlens, T, n), L = seg_end(cu_seqlens, T, n) - t0;
        double* qh = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * K);
        double* kh = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * K);
        double* g = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * K);
        double* beta = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double* rq = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double* rk = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double* S = (double*)calloc((size_t)K * V, sizeof(double));
        double* w = (double*)malloc(sizeof(double) * (size_t)V);
        double* vv = (double*)malloc(sizeof(double) * (size_t)V);
        double* o = (double*)malloc(sizeof(double) * (size_t)V);
        if (!qh || !kh || !g || !beta || !rq || !rk || !S || !w || !vv || !o) {
            err |= 1;
        } else {
            prologue(t0, L, h, H, Hk, K, q, k, g_raw, beta_raw, a_log, dt_bias, lower_bound, gate,
                     qh, kh, g, beta, rq, rk);
            if (initial_state)
                memcpy(S, initial_state + ((size_t)n * H + h) * K * V, sizeof(double) * (size_t)K * V);
            for (int64_t i = 0; i < L; ++i) {
                const int64_t row = (t0 + i) * H + h;
                for (int j = 0; j < V; ++j) vv[j] = v[row * V + j];
                step_fwd(K, V, S, qh + i * K, kh + i * K, vv, g + i * K, beta[i], scale, o, w);
                for (int j = 0; j < V; ++j) out[row * V + j] = o[j];
            }
            if (final_state)
                memcpy(final_state + ((size_t)n * H + h) * K * V, S, sizeof(double) * (size_t)K * V);
        }
        free(qh); free(kh); free(g); free(beta); free(rq); free(rk); free(S); free(w); free(vv); free(o);
    }
    return err;
}

/* ---- backward (reverse mode of the loop above) --------------------------- */

int oracle_kda_bwd(int B, int T, int H, int Hk, int K, int V, int num_seqs, const int32_t* cu_seqlens,
                   const double* q, const double* k, const double* v, const double* g_raw,
                   const double* beta_raw, const double* a_log, const double* dt_bias,
                   double scale, double lower_bound, int gate, const double* initial_state,
                   const double* dout, const double* dfinal_state,
                   double* dq, double* dk, double* dv, double* dg_raw, double* dbeta_raw,
                   double* da_log, double* ddt_bias, double* dinitial_state, int nthreads)
{
    const int N = cu_seqlens ? num_seqs : B;
    const int pairs = N * H;
    const int G = H / Hk;
    const size_t KV = (size_t)K * V;
    const int64_t TT = cu_seqlens ? (int64_t)cu_seqlens[num_seqs] : (int64_t)B * T;
    /* per-pair partial sums of the parameter gradients, reduced in a fixed order */
    double* pa = (double*)calloc((size_t)pairs, sizeof(double));
    double* pd = (double*)calloc((size_t)pairs * K, sizeof(double));
    /* with grouped heads, dq and dk per value head first ([TT, H, K]), summed over each group below */
    double* dqv = G > 1 ? (double*)calloc((size_t)TT * H * K, sizeof(double)) : dq;
    double* dkv = G > 1 ? (double*)calloc((size_t)TT * H * K, sizeof(double)) : dk;
    int err = 0;
    if (!pa || !pd || !dqv || !dkv) {
        free(pa); free(pd);
        if (G > 1) { free(dqv); free(dkv); }
        return 1;
    }
    (void)nthreads;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
#endif
    for (int p = 0; p < pairs; ++p) {
        const int n = p / H, h = p % H;
        const int64_t t0 = seg_begin(cu_seqlens, T, n), L = seg_end(cu_seqlens, T, n) - t0;
        const int64_t Lm = L > 0 ? L : 1;
        const int64_t ncp = (L + ORACLE_CKPT - 1) / ORACLE_CKPT;
        double* qh = (double*)malloc(sizeof(double) * (size_t)Lm * K);
        double* kh = (double*)malloc(sizeof(double) * (size_t)Lm * K);
        double* g = (double*)malloc(sizeof(double) * (size_t)Lm * K);
        double* beta = (double*)malloc(sizeof(double) * (size_t)Lm);
        double* rq = (double*)malloc(sizeof(double) * (size_t)Lm);
        double* rk = (double*)malloc(sizeof(double) * (size_t)Lm);
        double* dqh = (double*)calloc((size_t)Lm * K, sizeof(double));
        double* dkh = (double*)calloc((size_t)Lm * K, sizeof(double));
        double* dg = (double*)calloc((size_t)Lm * K, sizeof(double));
        double* dbeta = (double*)calloc((size_t)Lm, sizeof(double));
        double* ckpt = (double*)malloc(sizeof(double) * (size_t)(ncp > 0 ? ncp : 1) * KV);
        double* Sb = (double*)malloc(sizeof(double) * (size_t)(ORACLE_CKPT + 1) * KV);
        double* S = (double*)calloc(KV, sizeof(double));
        double* dS = (double*)calloc(KV, sizeof(double));
        double* P = (double*)malloc(sizeof(double) * KV);
        double* w = (double*)malloc(sizeof(double) * (size_t)V);
        double* e = (double*)malloc(sizeof(double) * (size_t)V);
        double* de = (double*)malloc(sizeof(double) * (size_t)V);
        double* vv = (double*)malloc(sizeof(double) * (size_t)V);
        if (!qh || !kh || !g || !beta || !rq || !rk || !dqh || !dkh || !dg || !dbeta || !ckpt || !Sb ||
            !S || !dS || !P || !w || !e || !de || !vv) {
            err |= 1;
            goto done;
        }
        prologue(t0, L, h, H, Hk, K, q, k, g_raw, beta_raw, a_log, dt_bias, lower_bound, gate,
                 qh, kh, g, beta, rq, rk);
        if (initial_state) memcpy(S, initial_state + ((size_t)n * H + h) * KV, sizeof(double) * KV);
        /* forward sweep: remember the state entering every 64-token block */
        for (int64_t i = 0; i < L; ++i) {
            if (i % ORACLE_CKPT == 0) memcpy(ckpt + (i / ORACLE_CKPT) * KV, S, sizeof(double) * KV);
            const int64_t row = (t0 + i) * H + h;
            for (int j = 0; j < V; ++j) vv[j] = v[row * V + j];
            step_fwd(K, V, S, qh + i * K, kh + i * K, vv, g + i * K, beta[i], scale, NULL, w);
        }
        if (dfinal_state) memcpy(dS, dfinal_state + ((size_t)n * H + h) * KV, sizeof(double) * KV);
        for (int64_t blk = ncp - 1; blk >= 0; --blk) {
            const int64_t b0 = blk * ORACLE_CKPT;
            const int64_t b1 = (b0 + ORACLE_CKPT < L) ? b0 + ORACLE_CKPT : L;
            /* Sb[i] = state before token b0+i; Sb[b1-b0] = state after the block */
            memcpy(Sb, ckpt + blk * KV, sizeof(double) * KV);
            for (int64_t i = b0; i < b1; ++i) {
                double* cur = Sb + (size_t)(i - b0 + 1) * KV;
                memcpy(cur, Sb + (size_t)(i - b0) * KV, sizeof(double) * KV);
                const int64_t row = (t0 + i) * H + h;
                for (int j = 0; j < V; ++j) vv[j] = v[row * V + j];
                step_fwd(K, V, cur, qh + i * K, kh + i * K, vv, g + i * K, beta[i], scale, NULL, w);
            }
            for (int64_t i = b1 - 1; i >= b0; --i) {
                const int64_t row = (t0 + i) * H + h;
                const double* Sprev = Sb + (size_t)(i - b0) * KV;
                const double* St = Sb + (size_t)(i - b0 + 1) * KV;
                const double* qi = qh + i * K;
                const double* ki = kh + i * K;
                const double* doi = dout + row * V;
                const double bt = beta[i];
                /* o = scale S_t^T q */
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j < V; ++j) {
                        acc += St[c * V + j] * doi[j];
                        dS[c * V + j] += scale * qi[c] * doi[j];
                    }
                    dqh[i * K + c] += scale * acc;
                }
                /* P = Diag(alpha) S_prev, w = P^T k, e = v - w */
                for (int c = 0; c < K; ++c) {
                    const double a = exp(g[i * K + c]);
                    for (int j = 0; j < V; ++j) P[c * V + j] = a * Sprev[c * V + j];
                }
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c) acc += P[c * V + j] * ki[c];
                    e[j] = v[row * V + j] - acc;
                }
                /* S_t = P + beta k e^T */
                double db = 0.0;
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j < V; ++j) acc += dS[c * V + j] * e[j];
                    db += ki[c] * acc;
                    dkh[i * K + c] += bt * acc;
                }
                dbeta[i] += db;
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c) acc += dS[c * V + j] * ki[c];
                    de[j] = bt * acc;
                    dv[row * V + j] = de[j];
                }
                /* e = v - w, w = P^T k: dP = dS - k de^T, dk -= P de */
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j < V; ++j) {
                        acc += P[c * V + j] * de[j];
                        dS[c * V + j] -= ki[c] * de[j]; /* dS now holds dP */
                    }
                    dkh[i * K + c] -= acc;
                }
                /* P = Diag(exp(g)) S_prev */
                for (int c = 0; c < K; ++c) {
                    const double a = exp(g[i * K + c]);
                    double acc = 0.0;
                    for (int j = 0; j < V; ++j) {
                        acc += dS[c * V + j] * Sprev[c * V + j];
                        dS[c * V + j] *= a;
                    }
                    dg[i * K + c] += a * acc;
                }
            }
        }
        if (dinitial_state) memcpy(dinitial_state + ((size_t)n * H + h) * KV, dS, sizeof(double) * KV);
        /* prologue backward */
        for (int64_t i = 0; i < L; ++i) {
            const int64_t row = (t0 + i) * H + h;
            /* x_hat = x r, r = (|x|^2 + eps)^-1/2  ->  dx = r (dy - y (y . dy)) */
            double sq = 0.0, sk = 0.0;
            for (int c = 0; c < K; ++c) {
                sq += qh[i * K + c] * dqh[i * K + c];
                sk += kh[i * K + c] * dkh[i * K + c];
            }
            for (int c = 0; c < K; ++c) {
                dqv[row * K + c] = rq[i] * (dqh[i * K + c] - qh[i * K + c] * sq);
                dkv[row * K + c] = rk[i] * (dkh[i * K + c] - kh[i * K + c] * sk);
            }
            dbeta_raw[row] = dbeta[i] * beta[i] * (1.0 - beta[i]);
            const double ea = exp(a_log[h]);
            for (int c = 0; c < K; ++c) {
                const double x = g_raw[row * K + c] + dt_bias[h * K + c];
                if (gate == ORACLE_GATE_SOFTPLUS) {
                    /* g = -e^a softplus(x):  dg/dx = -e^a sigmoid(x),  dg/da = g */
                    const double dx = -dg[i * K + c] * ea * sigm(x);
                    dg_raw[row * K + c] = dx;
                    pd[(size_t)p * K + c] += dx;
                    pa[p] += dg[i * K + c] * g[i * K + c];
                } else {
                    /* g = lb sigmoid(z), z = e^a x:  dg/dz = lb s (1 - s) */
                    const double z = ea * x;
                    const double s = sigm(z);
                    const double dz = dg[i * K + c] * lower_bound * s * (1.0 - s);
                    dg_raw[row * K + c] = dz * ea;
                    pd[(size_t)p * K + c] += dz * ea;
                    pa[p] += dz * z;
                }
            }
        }
    done:
        free(qh); free(kh); free(g); free(beta); free(rq); free(rk); free(dqh); free(dkh); free(dg);
        free(dbeta); free(ckpt); free(Sb); free(S); free(dS); free(P); free(w); free(e); free(de); free(vv);
    }
    for (int h = 0; h < H; ++h) {
        double a = 0.0;
        for (int c = 0; c < K; ++c) ddt_bias[h * K + c] = 0.0;
        for (int n = 0; n < N; ++n) {
            a += pa[n * H + h];
            for (int c = 0; c < K; ++c) ddt_bias[h * K + c] += pd[((size_t)n * H + h) * K + c];
        }
        da_log[h] = a;
    }
    if (G > 1) {
        /* key head hk collects the value heads hk*G .. hk*G + G-1, in that order */
        for (int64_t t = 0; t < TT; ++t)
            for (int hk = 0; hk < Hk; ++hk)
                for (int c = 0; c < K; ++c) {
                    double sq = 0.0, sk = 0.0;
                    for (int g2 = 0; g2 < G; ++g2) {
                        const int64_t vr = (t * H + hk * G + g2) * K + c;
                        sq += dqv[vr];
                        sk += dkv[vr];
                    }
                    dq[(t * Hk + hk) * K + c] = sq;
                    dk[(t * Hk + hk) * K + c] = sk;
                }
        free(dqv); free(dkv);
    }
    free(pa); free(pd);
    return err;
}

/* ---- the layer's q/k/v prologue: causal depthwise short convolution + SiLU ----
 *
 * hyper-parallel "KDA context-parallel executors" (`_run_causal_short_conv`,
 * `_local_short_conv`, `_validate_layer_short_conv`): each of q, k, v passes
 * through a depthwise Conv1d (groups = channels, stride 1, dilation 1, zero
 * padding kernel_size - 1 on the left, output cut to the input length) and
 * SiLU.  With packed documents every segment starts from zero history (the
 * same convention as the recurrence; the pages hand the conv kernel size to
 * FLA's per-document context for exactly these boundary tokens).
 *
 *   a[t, c] = bias[c] + sum_{i<W} weight[c, i] x[t - (W-1) + i, c]
 *   y[t, c] = a * sigmoid(a)
 * x [TT, C], weight [C, W], bias [C] or NULL. */
static int64_t seg_start_of(const int32_t* cu, int num_seqs, int T, int64_t t)
{
    if (!cu) return (t / T) * T;
    int lo = 0, hi = num_seqs - 1;           /* last n with cu[n] <= t */
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return cu[lo];
}

static double conv_pre(const double* x, const double* w, const double* b, int C, int W, int64_t s0, int64_t t,
                       int c)
{
    double a = b ? b[c] : 0.0;
    for (int i = 0; i < W; ++i) {
        const int64_t tau = t - (W - 1) + i;
        if (tau >= s0) a += w[c * W + i] * x[tau * C + c];
    }
    return a;
}

int oracle_short_conv_fwd(int64_t TT, int T, int C, int W, const int32_t* cu_seqlens, int num_seqs,
                          const double* x, const double* weight, const double* bias, double* y)
{
    for (int64_t t = 0; t < TT; ++t) {
        const int64_t s0 = seg_start_of(cu_seqlens, num_seqs, T, t);
        for (int c = 0; c < C; ++c) {
            const double a = conv_pre(x, weight, bias, C, W, s0, t, c);
            y[t * C + c] = a * sigm(a);
        }
    }
    return 0;
}

/* Reverse mode: da = dy * d silu(a)/da = dy * s (1 + a (1 - s)), s = sigmoid(a); then dx, dweight,
 * dbias by the chain rule through the sum above. */
int oracle_short_conv_bwd(int64_t TT, int T, int C, int W, const int32_t* cu_seqlens, int num_seqs,
                          const double* x, const double* weight, const double* bias, const double* dy,
                          double* dx, double* dweight, double* dbias)
{
    memset(dx, 0, sizeof(double) * (size_t)TT * C);
    memset(dweight, 0, sizeof(double) * (size_t)C * W);
    if (dbias) memset(dbias, 0, sizeof(double) * (size_t)C);
    for (int64_t t = 0; t < TT; ++t) {
        const int64_t s0 = seg_start_of(cu_seqlens, num_seqs, T, t);
        for (int c = 0; c < C; ++c) {
            const double a = conv_pre(x, weight, bias, C, W, s0, t, c);
            const double s = sigm(a);
            const double da = dy[t * C + c] * s * (1.0 + a * (1.0 - s));
            if (dbias) dbias[c] += da;
            for (int i = 0; i < W; ++i) {
                const int64_t tau = t - (W - 1) + i;
                if (tau < s0) continue;
                dx[tau * C + c] += weight[c * W + i] * da;
                dweight[c * W + i] += x[tau * C + c] * da;
            }
        }
    }
    return 0;
}

/* ---- the layer's output epilogue: gated RMS norm over each head's value vector ----
 *
 * hyper-parallel "KDA context-parallel executors" (`KimiDeltaAttentionUlyssesCP` forward, the
 * full-layer adapter) applies `o_norm(output, output_gate)` to the attention output before the
 * output projection, with `output_gate` from the layer's `g_proj` (or `g_b_proj(g_a_proj(.))`); the
 * torchtitan review describes the model's RMS norm as one reduced in fp32 with its own epsilon.
 * The pages print neither the norm's formula nor the gate's activation.  Reading: an RMS norm of
 * each head's V values with a per-channel weight, gated by the sigmoid of the output gate,
 *     y_v = o_v / sqrt(mean_u o_u^2 + eps) * w_v * sigmoid(gate_v),
 * eps given by the caller.  rows = B*T*H rows of V values each. */
int oracle_gated_norm_fwd(int64_t rows, int V, const double* o, const double* gate, const double* w, double eps,
                          double* y)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double* orow = o + r * V;
        double ss = 0.0;
        for (int v = 0; v < V; ++v) ss += orow[v] * orow[v];
        const double rn = 1.0 / sqrt(ss / V + eps);
        for (int v = 0; v < V; ++v) y[r * V + v] = orow[v] * rn * w[v] * sigm(gate[r * V + v]);
    }
    return 0;
}

/* Reverse mode.  With n = o rn and s = sigmoid(gate):  dgate = dy n w s (1 - s),
 * dw = sum_rows dy n s,  dn = dy w s,  do = rn (dn - n mean_u(dn_u n_u)). */
int oracle_gated_norm_bwd(int64_t rows, int V, const double* o, const double* gate, const double* w, double eps,
                          const double* dy, double* d_o, double* dgate, double* dw)
{
    for (int v = 0; v < V; ++v) dw[v] = 0.0;
    for (int64_t r = 0; r < rows; ++r) {
        const double* orow = o + r * V;
        double ss = 0.0;
        for (int v = 0; v < V; ++v) ss += orow[v] * orow[v];
        const double rn = 1.0 / sqrt(ss / V + eps);
        double dot = 0.0;
        for (int v = 0; v < V; ++v) {
            const double n = orow[v] * rn, s = sigm(gate[r * V + v]), g = dy[r * V + v];
            dot += g * w[v] * s * n;
        }
        for (int v = 0; v < V; ++v) {
            const double n = orow[v] * rn, s = sigm(gate[r * V + v]), g = dy[r * V + v];
            const double dn = g * w[v] * s;
            d_o[r * V + v] = rn * (dn - n * dot / V);
            dgate[r * V + v] = g * n * w[v] * s * (1.0 - s);
            dw[v] += g * n * s;
        }
    }
    return 0;
}
