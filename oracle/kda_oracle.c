/*
 * kda_oracle.c -- plain double-precision CPU oracle for the KDA layer step.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may build, load or call this file.  It shares no code,
 * header, table or helper with the CUDA library, and neither includes the
 * other.  It is deliberately slow and obvious: no blocking, fusion or
 * reordering beyond what the definitions below state.
 *
 * What it computes, per sequence and per head, token by token:
 *   a1  conv:  a depthwise causal convolution of width W over every raw q, k
 *       and v channel.  The last tap multiplies the current token, the other
 *       W-1 taps the previous raw inputs (kept per slot as the "conv tail",
 *       oldest first).  No bias.  SiLU follows on q, k and v: y = x*sigmoid(x).
 *   a2  L2:    q <- q / sqrt(sum_i q_i^2 + eps_l2), same for k; v untouched.
 *   a3  update: S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1}
 *                     + beta_t k_t v_t^T,            S is d_k x d_v
 *   a4  readout: o_t = S_t^T q_t   (the updated state, no 1/sqrt(d) scale)
 *   a5  gated norm: y_t = w_n * o_t / sqrt(mean_j o_tj^2 + eps_rms)
 *                        * sigmoid(g_t)
 *
 * Sources.  "vLLM Kimi K3 지원" (agentlenshq.com), section "Kimi K3 아키텍처 개요":
 * KDA is a linear-attention layer that keeps a fixed-size recurrent state.
 * Same page, section "Fused Kernels 및 메타데이터 최적화", KDA Decode bullet: the
 * decode step fuses the causal convolution, the recurrent update and the
 * RMSNorm; KDA Prefill bullet: prefill runs chunked (FlashKDA).  The pages do
 * not print the recurrence itself; a1..a5 above are the KDA (gated delta rule)
 * step this library is specified to compute.  Readings taken where the
 * specification is silent: SiLU on all of q, k, v; eps inside the square
 * roots; norm first, then the weight, then the sigmoid gate; alpha and beta
 * arrive as values in (0,1); the gate arrives as logits; a new sequence
 * starts from a zero state and a zero tail.
 *
 * The chunked entry (core_chunked) is the same recurrence re-associated over
 * chunks of C tokens (WY / UT form), written out in double with exact
 * per-element decay factors exp(G_r - G_s); it exists to pin the chunk algebra
 * that the GPU prefill uses, and must agree with the token loop to rounding.
 *
 * Layouts (row-major, double):
 *   raw q, k: [L][H][d_k]; raw v: [L][H][d_v]; alpha: [L][H][d_k];
 *   beta: [L][H]; gate: [L][H][d_v]; out: [L][H][d_v]
 *   conv channels: n_ch = H*(2*d_k + d_v), ordered q (h*d_k+i), then k
 *   (H*d_k + h*d_k+i), then v (2*H*d_k + h*d_v+j)
 *   conv_w: [n_ch][W]  (tap 0 = oldest input, tap W-1 = current token)
 *   tail:   [W-1][n_ch] (row 0 = oldest previous raw input)
 *   state:  [H][d_k][d_v]  (S[i][j], i = key channel, j = value channel)
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static double silu(double x) { return x * sigmoid(x); }

/* ---------------------------------------------------------------- a1 ---- */

/* Causal conv + SiLU for one channel over n tokens.  x(t) = x[t*xs].
 * tail[j*ts], j = 0..W-2, holds the previous raw inputs (oldest first) and is
 * advanced in place.  When hist is not NULL, the tail after token t is stored
 * at hist[t*hs + j*ts]. */
static void conv_silu_channel(int n, int W, const double *w, double *tail,
                              long ts, const double *x, long xs, double *y,
                              long ys, double *hist, long hs)
{
    for (int t = 0; t < n; ++t) {
        double acc = 0.0;
        for (int j = 0; j < W - 1; ++j)
            acc += w[j] * tail[j * ts];
        acc += w[W - 1] * x[t * xs];
        y[t * ys] = silu(acc);
        /* the window moves on: drop the oldest raw input, append this one */
        for (int j = 0; j < W - 2; ++j)
            tail[j * ts] = tail[(j + 1) * ts];
        tail[(W - 2) * ts] = x[t * xs];
        if (hist)
            for (int j = 0; j < W - 1; ++j)
                hist[t * hs + j * ts] = tail[j * ts];
    }
}

/* ---------------------------------------------------------------- a2 ---- */

static void l2norm(int d, double *x, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < d; ++i)
        ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < d; ++i)
        x[i] = x[i] * r;
}

/* ---------------------------------------------------------------- a5 ---- */

static void gated_rmsnorm(int dv, const double *o, const double *g,
                          const double *wn, double eps, double *y)
{
    double ms = 0.0;
    for (int j = 0; j < dv; ++j)
        ms += o[j] * o[j];
    ms = ms / dv;
    double r = 1.0 / sqrt(ms + eps);
    for (int j = 0; j < dv; ++j)
        y[j] = wn[j] * (o[j] * r) * sigmoid(g[j]);
}

/* ----------------------------------------------------------- a3 + a4 ---- */

/* Token loop for one head.  Row t of q/k/alpha is at q + t*qs etc.  M and u
 * are scratch of d_k*d_v and d_v doubles.  hist (may be NULL) receives S_t
 * after every token at hist + t*hs. */
static void core_recurrent(int n, int dk, int dv, const double *q, long qs,
                           const double *k, long ks, const double *v, long vs,
                           const double *alpha, long as, const double *beta,
                           long bs, double *S, double *o, long os,
                           double *hist, long hs, double *M, double *u)
{
    for (int t = 0; t < n; ++t) {
        const double *qt = q + t * qs, *kt = k + t * ks, *vt = v + t * vs;
        const double *at = alpha + t * as;
        const double bt = beta[t * bs];
        /* M = Diag(alpha_t) S_{t-1}: row i of S is scaled by alpha_t[i] */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                M[i * dv + j] = at[i] * S[i * dv + j];
        /* u = M^T k_t */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i)
                acc += kt[i] * M[i * dv + j];
            u[j] = acc;
        }
        /* S_t = M - beta k (M^T k)^T + beta k v^T = (I - beta k k^T) M + beta k v^T */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                S[i * dv + j] = M[i * dv + j] + bt * kt[i] * (vt[j] - u[j]);
        /* o_t = S_t^T q_t */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i)
                acc += qt[i] * S[i * dv + j];
            o[t * os + j] = acc;
        }
        if (hist)
            memcpy(hist + t * hs, S, sizeof(double) * dk * dv);
    }
}

/* Scratch needed by core_chunked for chunk size C. */
static long chunked_scratch(int C, int dk, int dv)
{
    return (long)C * dk /*G*/ + 2L * C * C /*A,T*/ + (long)C * dk /*W*/ +
           2L * C * dv /*Ut,U*/ + (long)dk * dv /*Snew*/;
}

/* The same recurrence over chunks of C tokens.  Within a chunk starting at
 * token c0 with n tokens, r and s index tokens 0..n-1 and
 *   G[r][i]  = sum_{s<=r} log alpha_{c0+s, i}         (cumulative log decay)
 *   A[r][s]  = beta_r sum_i k_r,i k_s,i exp(G_r,i - G_s,i)   for s < r
 *   T        = (I + A)^{-1}                                   (unit lower)
 *   W        = T diag(beta) Kt,   Kt[s][i] = exp(G_s,i) k_s,i
 *   Ut       = T diag(beta) V
 *   U        = Ut - W S                                       (new values)
 *   O[r]     = Qt[r] S + sum_{s<=r} P[r][s] U[s],
 *              Qt[r][i] = exp(G_r,i) q_r,i,
 *              P[r][s] = sum_i q_r,i k_s,i exp(G_r,i - G_s,i)
 *   S       <- Diag(exp(G_{n-1})) S + sum_s Kb[s] U[s]^T,
 *              Kb[s][i] = exp(G_{n-1},i - G_s,i) k_s,i
 * Requires alpha > 0. */
static void core_chunked(int L, int C, int dk, int dv, const double *q,
                         long qs, const double *k, long ks, const double *v,
                         long vs, const double *alpha, long as,
                         const double *beta, long bs, double *S, double *o,
                         long os, double *scratch)
{
    double *G = scratch;
    double *A = G + (long)C * dk;
    double *T = A + (long)C * C;
    double *Wm = T + (long)C * C;
    double *Ut = Wm + (long)C * dk;
    double *U = Ut + (long)C * dv;
    double *Sn = U + (long)C * dv;
    for (int c0 = 0; c0 < L; c0 += C) {
        const int n = (L - c0 < C) ? (L - c0) : C;
        const double *qc = q + c0 * qs, *kc = k + c0 * ks, *vc = v + c0 * vs;
        const double *ac = alpha + c0 * as, *bc = beta + c0 * bs;
        for (int i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int r = 0; r < n; ++r) {
                acc += log(ac[r * as + i]);
                G[r * dk + i] = acc;
            }
        }
        for (int r = 0; r < n; ++r)
            for (int s = 0; s < n; ++s) {
                double acc = 0.0;
                if (s < r)
                    for (int i = 0; i < dk; ++i)
                        acc += kc[r * ks + i] * kc[s * ks + i] *
                               exp(G[r * dk + i] - G[s * dk + i]);
                A[r * C + s] = bc[r * bs] * acc;
            }
        /* forward substitution: row r of T is e_r - sum_{s<r} A[r][s] T[s] */
        for (int r = 0; r < n; ++r)
            for (int c = 0; c < n; ++c) {
                double acc = (r == c) ? 1.0 : 0.0;
                for (int s = 0; s < r; ++s)
                    acc -= A[r * C + s] * T[s * C + c];
                T[r * C + c] = acc;
            }
        for (int r = 0; r < n; ++r) {
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int s = 0; s < n; ++s)
                    acc += T[r * C + s] * bc[s * bs] * exp(G[s * dk + i]) *
                           kc[s * ks + i];
                Wm[r * dk + i] = acc;
            }
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int s = 0; s < n; ++s)
                    acc += T[r * C + s] * bc[s * bs] * vc[s * vs + j];
                Ut[r * dv + j] = acc;
            }
        }
        for (int r = 0; r < n; ++r)
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i)
                    acc += Wm[r * dk + i] * S[i * dv + j];
                U[r * dv + j] = Ut[r * dv + j] - acc;
            }
        for (int r = 0; r < n; ++r)
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i)
                    acc += exp(G[r * dk + i]) * qc[r * qs + i] * S[i * dv + j];
                for (int s = 0; s <= r; ++s) {
                    double p = 0.0;
                    for (int i = 0; i < dk; ++i)
                        p += qc[r * qs + i] * kc[s * ks + i] *
                             exp(G[r * dk + i] - G[s * dk + i]);
                    acc += p * U[s * dv + j];
                }
                o[(c0 + r) * os + j] = acc;
            }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) {
                double acc = exp(G[(n - 1) * dk + i]) * S[i * dv + j];
                for (int s = 0; s < n; ++s)
                    acc += exp(G[(n - 1) * dk + i] - G[s * dk + i]) *
                           kc[s * ks + i] * U[s * dv + j];
                Sn[i * dv + j] = acc;
            }
        memcpy(S, Sn, sizeof(double) * dk * dv);
    }
}

/* ------------------------------------------------------- public entries -- */

static void set_threads(int n_threads)
{
#ifdef _OPENMP
    omp_set_num_threads(n_threads > 0 ? n_threads : omp_get_num_procs());
#else
    (void)n_threads;
#endif
}

int kdaref_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* a1 over all n_ch channels of x [L][n_ch]; y [L][n_ch]; tail advanced in
 * place; hist_tail (may be NULL) [L][W-1][n_ch]. */
void kdaref_conv_silu(int L, long n_ch, int W, const double *conv_w,
                      double *tail, const double *x, double *y,
                      double *hist_tail)
{
    for (long c = 0; c < n_ch; ++c)
        conv_silu_channel(L, W, conv_w + c * W, tail + c, n_ch, x + c, n_ch,
                          y + c, n_ch, hist_tail ? hist_tail + c : NULL,
                          (long)(W - 1) * n_ch);
}

/* a2 on n rows of length d, in place. */
void kdaref_l2norm_rows(long n, int d, double *x, double eps)
{
    for (long r = 0; r < n; ++r)
        l2norm(d, x + r * d, eps);
}

/* a5 on n rows of length dv. */
void kdaref_gated_rmsnorm_rows(long n, int dv, const double *o,
                               const double *g, const double *wn, double eps,
                               double *y)
{
    for (long r = 0; r < n; ++r)
        gated_rmsnorm(dv, o + r * dv, g + r * dv, wn, eps, y + r * dv);
}

/* a3 + a4 for one head on inputs that already went through a1 and a2.
 * q, k, alpha: [L][dk]; v: [L][dv]; beta: [L]; S: [dk][dv] in/out;
 * o: [L][dv]; hist (may be NULL, token loop only): [L][dk][dv].
 * chunk = 0 runs the token loop, chunk > 0 the chunked form.
 * Returns 0, or -1 on a bad argument or allocation failure. */
int kdaref_core(int L, int dk, int dv, int chunk, const double *q,
                const double *k, const double *v, const double *alpha,
                const double *beta, double *S, double *o, double *hist)
{
    if (L < 0 || dk <= 0 || dv <= 0 || chunk < 0 || (chunk > 0 && hist))
        return -1;
    if (chunk == 0) {
        double *M = malloc(sizeof(double) * ((long)dk * dv + dv));
        if (!M)
            return -1;
        core_recurrent(L, dk, dv, q, dk, k, dk, v, dv, alpha, dk, beta, 1, S,
                       o, dv, hist, (long)dk * dv, M, M + (long)dk * dv);
        free(M);
    } else {
        double *scr = malloc(sizeof(double) * chunked_scratch(chunk, dk, dv));
        if (!scr)
            return -1;
        core_chunked(L, chunk, dk, dv, q, dk, k, dk, v, dv, alpha, dk, beta, 1,
                     S, o, dv, scr);
        free(scr);
    }
    return 0;
}

/* The whole layer step a1..a5 for one sequence of L tokens, all heads.
 * state [H][dk][dv] and tail [W-1][n_ch] are read as the starting point and
 * overwritten with the end point.  out: [L][H][dv].  hist_state (may be
 * NULL, token loop only): [L][H][dk][dv], the state after every token;
 * hist_tail (may be NULL): [L][W-1][n_ch], the tail after every token.
 * Heads are independent and run in parallel on n_threads (0 = default).
 * Returns 0, or -1 on a bad argument or allocation failure. */
int kdaref_layer(int L, int H, int dk, int dv, int W, double eps_l2,
                 double eps_rms, int chunk, const double *q, const double *k,
                 const double *v, const double *alpha, const double *beta,
                 const double *gate, const double *conv_w,
                 const double *norm_w, double *state, double *tail,
                 double *out, double *hist_state, double *hist_tail,
                 int n_threads)
{
    if (L < 0 || H <= 0 || dk <= 0 || dv <= 0 || W < 2 || chunk < 0 ||
        (chunk > 0 && hist_state))
        return -1;
    const long n_ch = (long)H * (2 * dk + dv);
    const int blk = chunk > 0 ? chunk : 64;
    int failed = 0;
    set_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int h = 0; h < H; ++h) {
        const long cq = (long)h * dk, ck = (long)H * dk + (long)h * dk,
                   cv = 2L * H * dk + (long)h * dv;
        double *qc = malloc(sizeof(double) * blk * dk);
        double *kc = malloc(sizeof(double) * blk * dk);
        double *vc = malloc(sizeof(double) * blk * dv);
        double *oc = malloc(sizeof(double) * blk * dv);
        double *scr = malloc(sizeof(double) * (chunk > 0 ? chunked_scratch(
                                                   chunk, dk, dv)
                                                         : (long)dk * dv + dv));
        if (!qc || !kc || !vc || !oc || !scr) {
            failed = 1;
        } else {
            double *S = state + (long)h * dk * dv;
            for (int t0 = 0; t0 < L; t0 += blk) {
                const int n = (L - t0 < blk) ? (L - t0) : blk;
                double *ht = hist_tail ? hist_tail + (long)t0 * (W - 1) * n_ch
                                       : NULL;
                const long hts = (long)(W - 1) * n_ch;
                for (int i = 0; i < dk; ++i) {
                    conv_silu_channel(n, W, conv_w + (cq + i) * W,
                                      tail + cq + i, n_ch,
                                      q + (long)t0 * H * dk + (long)h * dk + i,
                                      (long)H * dk, qc + i, dk,
                                      ht ? ht + cq + i : NULL, hts);
                    conv_silu_channel(n, W, conv_w + (ck + i) * W,
                                      tail + ck + i, n_ch,
                                      k + (long)t0 * H * dk + (long)h * dk + i,
                                      (long)H * dk, kc + i, dk,
                                      ht ? ht + ck + i : NULL, hts);
                }
                for (int j = 0; j < dv; ++j)
                    conv_silu_channel(n, W, conv_w + (cv + j) * W,
                                      tail + cv + j, n_ch,
                                      v + (long)t0 * H * dv + (long)h * dv + j,
                                      (long)H * dv, vc + j, dv,
                                      ht ? ht + cv + j : NULL, hts);
                for (int t = 0; t < n; ++t) {
                    l2norm(dk, qc + t * dk, eps_l2);
                    l2norm(dk, kc + t * dk, eps_l2);
                }
                const double *al = alpha + (long)t0 * H * dk + (long)h * dk;
                const double *be = beta + (long)t0 * H + h;
                if (chunk > 0)
                    core_chunked(n, chunk, dk, dv, qc, dk, kc, dk, vc, dv, al,
                                 (long)H * dk, be, H, S, oc, dv, scr);
                else
                    core_recurrent(
                        n, dk, dv, qc, dk, kc, dk, vc, dv, al, (long)H * dk,
                        be, H, S, oc, dv,
                        hist_state ? hist_state + (long)t0 * H * dk * dv +
                                         (long)h * dk * dv
                                   : NULL,
                        (long)H * dk * dv, scr, scr + (long)dk * dv);
                for (int t = 0; t < n; ++t)
                    gated_rmsnorm(dv, oc + t * dv,
                                  gate + (long)(t0 + t) * H * dv +
                                      (long)h * dv,
                                  norm_w, eps_rms,
                                  out + (long)(t0 + t) * H * dv +
                                      (long)h * dv);
            }
        }
        free(qc);
        free(kc);
        free(vc);
        free(oc);
        free(scr);
    }
    return failed ? -1 : 0;
}
