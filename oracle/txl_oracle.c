/*
 * Plain fp64 CPU oracle for Transformer-XL relative-position attention.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark load this file.  It shares no code with the CUDA library and
 * the CUDA library never calls it.
 *
 * It follows "Transformer-XL: Attentive Language Models Beyond a Fixed-Length
 * Context" (Dai et al.):
 *   - §3.3, the re-parameterised score A^rel_{i,j} = (a) + (b) + (c) + (d):
 *       (a) q_i . k_j                 content-based addressing
 *       (b) q_i . W_kR R_{i-j}        content-dependent positional bias
 *       (c) u   . k_j                 global content bias
 *       (d) v   . W_kR R_{i-j}        global positional bias
 *   - §3.3, the N-layer summary: keys and values run over the extended context
 *     [SG(m) o h] (memory rows first), queries over the current segment only,
 *     and the scores go through a masked softmax and then multiply v.
 *   - §3.3: R is the sinusoid encoding matrix of Vaswani et al. (no learnable
 *     parameters), row p standing for a relative distance of p.
 *
 * Readings taken where the pages leave a step open (each is listed in the
 * design notes of the repository):
 *   - A is multiplied by `scale` (1/sqrt(d_head) in every workload) before the
 *     mask and the softmax.
 *   - query i (0-based, of L) sits at position M+i of the extended context; key
 *     j (0-based, of M+L) at position j.  The relative distance is M+i-j and the
 *     mask keeps key j iff that distance is >= 0 (Appendix B: B is zero to the
 *     right of its shifted diagonal).
 *   - the sinusoid interleaves sin and cos: R_p[2k] = sin(p w_k),
 *     R_p[2k+1] = cos(p w_k), w_k = 10000^(-2k/d).
 *
 * Everything is computed in fp64 with the four terms formed separately per
 * (i, j) pair and the relative vector looked up by distance for each pair (the
 * quadratic "naive way" of §3.3, not the Appendix B shortcut).
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double dotd(const double *x, const double *y, int n)
{
    double s = 0.0;
    for (int t = 0; t < n; ++t) s += x[t] * y[t];
    return s;
}

/* Sinusoid relative encoding table, indexed by distance: R[p][t] for
 * p in [0, n_dist), t in [0, d), d even.  Angles in long double, stored as
 * double. */
int txlo_sinusoid_table(double *R, int n_dist, int d)
{
    if (!R || n_dist < 0 || d <= 0 || (d & 1)) return -1;
    for (int p = 0; p < n_dist; ++p) {
        for (int k = 0; k < d / 2; ++k) {
            long double w = powl(10000.0L, -2.0L * (long double)k / (long double)d);
            long double a = (long double)p * w;
            R[(size_t)p * d + 2 * k] = (double)sinl(a);
            R[(size_t)p * d + 2 * k + 1] = (double)cosl(a);
        }
    }
    return 0;
}

/* The four score terms of one head, before scaling.  rel[delta][dh] holds
 * W_kR R_delta for delta in [0, M+L).  Outputs ta..td are [L][M+L]; a masked
 * pair (key after query) gets valid = 0 and zero terms. */
int txlo_score_terms(const double *q, const double *k, const double *rel,
                     const double *u, const double *vb, int M, int L, int dh,
                     double *ta, double *tb, double *tc, double *td, int *valid)
{
    if (M < 0 || L < 1 || dh < 1) return -1;
    const int K = M + L;
    for (int i = 0; i < L; ++i) {
        for (int j = 0; j < K; ++j) {
            const size_t o = (size_t)i * K + j;
            const int delta = M + i - j;
            if (delta < 0) {
                ta[o] = tb[o] = tc[o] = td[o] = 0.0;
                valid[o] = 0;
                continue;
            }
            const double *qi = q + (size_t)i * dh;
            const double *kj = k + (size_t)j * dh;
            const double *rd = rel + (size_t)delta * dh;
            ta[o] = dotd(qi, kj, dh);
            tb[o] = dotd(qi, rd, dh);
            tc[o] = dotd(u, kj, dh);
            td[o] = dotd(vb, rd, dh);
            valid[o] = 1;
        }
    }
    return 0;
}

/* One head: masked softmax over the extended context and the weighted sum of
 * the value rows.  A is caller scratch of K doubles. */
static void one_head(const double *q, const double *k, const double *v,
                     const double *rel, const double *u, const double *vb,
                     double *out, double *lse, int M, int L, int dh,
                     double scale, double *A)
{
    const int K = M + L;
    for (int i = 0; i < L; ++i) {
        const double *qi = q + (size_t)i * dh;
        double amax = -INFINITY;
        for (int j = 0; j < K; ++j) {
            const int delta = M + i - j;
            if (delta < 0) { A[j] = -INFINITY; continue; }
            const double *kj = k + (size_t)j * dh;
            const double *rd = rel + (size_t)delta * dh;
            const double a = dotd(qi, kj, dh);
            const double b = dotd(qi, rd, dh);
            const double c = dotd(u, kj, dh);
            const double d = dotd(vb, rd, dh);
            A[j] = scale * (a + b + c + d);
            if (A[j] > amax) amax = A[j];
        }
        double sum = 0.0;
        for (int j = 0; j < K; ++j) {
            const double p = (A[j] == -INFINITY) ? 0.0 : exp(A[j] - amax);
            A[j] = p;
            sum += p;
        }
        double *oi = out + (size_t)i * dh;
        for (int t = 0; t < dh; ++t) {
            double acc = 0.0;
            for (int j = 0; j < K; ++j) acc += A[j] * v[(size_t)j * dh + t];
            oi[t] = acc / sum;
        }
        if (lse) lse[i] = amax + log(sum);
    }
}

/* Relative-position attention for a batch of heads.
 *   q [B][H][L][dh], k and v [B][H][M+L][dh], rel [H][M+L][dh] by distance,
 *   u and vb [H][dh]; out [B][H][L][dh], lse [B][H][L] (natural log, may be NULL).
 * bh_list (may be NULL) restricts the work to n_bh flattened (b*H + h) pairs;
 * other outputs are left untouched.  nthreads <= 0 uses the OpenMP default. */
int txlo_relattn(const double *q, const double *k, const double *v,
                 const double *rel, const double *u, const double *vb,
                 double *out, double *lse, int B, int H, int M, int L, int dh,
                 double scale, const int *bh_list, int n_bh, int nthreads)
{
    if (B < 0 || H < 1 || M < 0 || L < 1 || dh < 1) return -1;
    const int K = M + L;
    const int n = bh_list ? n_bh : B * H;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double *A = (double *)malloc(sizeof(double) * (size_t)K);
        if (!A) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int s = 0; s < n; ++s) {
            if (!A) continue;
            const int bh = bh_list ? bh_list[s] : s;
            if (bh < 0 || bh >= B * H) continue;
            const int h = bh % H;
            one_head(q + (size_t)bh * L * dh, k + (size_t)bh * K * dh,
                     v + (size_t)bh * K * dh, rel + (size_t)h * K * dh,
                     u + (size_t)h * dh, vb + (size_t)h * dh,
                     out + (size_t)bh * L * dh, lse ? lse + (size_t)bh * L : NULL,
                     M, L, dh, scale, A);
        }
        free(A);
    }
    return bad ? -2 : 0;
}

/* Number of threads an OpenMP parallel region uses by default. */
int txlo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * Backward of the attention above for one segment (training backpropagates
 * within a segment, §3.2; the memory is SG(m), so no gradient leaves through
 * it, but its projected keys and values still receive one).
 *
 * With A_ij = scale (a + b + c + d) for a kept pair, P = softmax_j(A), O = P v
 * and dO the gradient of the output, the chain rule gives, per head:
 *   dv_j      = sum_i P_ij dO_i
 *   dP_ij     = dO_i . v_j
 *   dA_ij     = P_ij (dP_ij - sum_j' P_ij' dP_ij')
 *   g_ij      = scale dA_ij                      (gradient of a + b + c + d)
 *   dq_i      = sum_j g_ij (k_j + rel_{M+i-j})   (terms (a), (b))
 *   dk_j      = sum_i g_ij (q_i + u)             (terms (a), (c))
 *   du        = sum_ij g_ij k_j                  (term (c))
 *   dvb       = sum_ij g_ij rel_{M+i-j}          (term (d))
 *   drel_dlt  = sum_{i - j = dlt - M} g_ij (q_i + vb)   (terms (b), (d))
 * Masked pairs have P = 0 and contribute nothing.  rel, u, vb are shared by the
 * batch, so drel, du, dvb are sums over b as well.
 *
 * Shapes as txlo_relattn; dout [B][H][L][dh]; outputs dq [B][H][L][dh], dk, dv
 * [B][H][M+L][dh], drel [H][M+L][dh] (by distance), du, dvb [H][dh].  Heads
 * run in parallel; the batch loop inside a head is sequential, so the sums over
 * b need no synchronisation.
 * ------------------------------------------------------------------------- */
static void one_head_bwd(const double *q, const double *k, const double *v,
                         const double *rel, const double *u, const double *vb,
                         const double *dout, double *dq, double *dk, double *dv,
                         double *drel, double *du, double *dvb, int M, int L, int dh,
                         double scale, double *P, double *G)
{
    const int K = M + L;
    for (int i = 0; i < L; ++i) {
        const double *qi = q + (size_t)i * dh;
        const double *doi = dout + (size_t)i * dh;
        /* probabilities of row i */
        double amax = -INFINITY;
        for (int j = 0; j < K; ++j) {
            const int delta = M + i - j;
            if (delta < 0) { P[j] = -INFINITY; continue; }
            const double *kj = k + (size_t)j * dh;
            const double *rd = rel + (size_t)delta * dh;
            P[j] = scale * (dotd(qi, kj, dh) + dotd(qi, rd, dh) + dotd(u, kj, dh) +
                            dotd(vb, rd, dh));
            if (P[j] > amax) amax = P[j];
        }
        double sum = 0.0;
        for (int j = 0; j < K; ++j) {
            P[j] = (P[j] == -INFINITY) ? 0.0 : exp(P[j] - amax);
            sum += P[j];
        }
        for (int j = 0; j < K; ++j) P[j] /= sum;
        /* dP and its P-weighted row mean */
        double mean = 0.0;
        for (int j = 0; j < K; ++j) {
            G[j] = (P[j] == 0.0) ? 0.0 : dotd(doi, v + (size_t)j * dh, dh);
            mean += P[j] * G[j];
        }
        for (int j = 0; j < K; ++j) G[j] = scale * P[j] * (G[j] - mean);
        /* contributions of row i */
        double *dqi = dq + (size_t)i * dh;
        for (int j = 0; j < K; ++j) {
            const int delta = M + i - j;
            if (delta < 0) continue;
            const double *kj = k + (size_t)j * dh;
            const double *rd = rel + (size_t)delta * dh;
            double *dkj = dk + (size_t)j * dh, *dvj = dv + (size_t)j * dh;
            double *drd = drel + (size_t)delta * dh;
            for (int t = 0; t < dh; ++t) {
                dvj[t] += P[j] * doi[t];
                dqi[t] += G[j] * (kj[t] + rd[t]);
                dkj[t] += G[j] * (qi[t] + u[t]);
                du[t] += G[j] * kj[t];
                dvb[t] += G[j] * rd[t];
                drd[t] += G[j] * (qi[t] + vb[t]);
            }
        }
    }
}

int txlo_relattn_bwd(const double *q, const double *k, const double *v,
                     const double *rel, const double *u, const double *vb,
                     const double *dout, double *dq, double *dk, double *dv,
                     double *drel, double *du, double *dvb, int B, int H, int M, int L,
                     int dh, double scale, int nthreads)
{
    if (B < 0 || H < 1 || M < 0 || L < 1 || dh < 1) return -1;
    const int K = M + L;
    for (size_t x = 0; x < (size_t)B * H * L * dh; ++x) dq[x] = 0.0;
    for (size_t x = 0; x < (size_t)B * H * K * dh; ++x) dk[x] = dv[x] = 0.0;
    for (size_t x = 0; x < (size_t)H * K * dh; ++x) drel[x] = 0.0;
    for (size_t x = 0; x < (size_t)H * dh; ++x) du[x] = dvb[x] = 0.0;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double *P = (double *)malloc(sizeof(double) * 2 * (size_t)K);
        if (!P) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int h = 0; h < H; ++h) {
            if (!P) continue;
            for (int b = 0; b < B; ++b) {
                const size_t bh = (size_t)b * H + h;
                one_head_bwd(q + bh * L * dh, k + bh * K * dh, v + bh * K * dh,
                             rel + (size_t)h * K * dh, u + (size_t)h * dh, vb + (size_t)h * dh,
                             dout + bh * L * dh, dq + bh * L * dh, dk + bh * K * dh,
                             dv + bh * K * dh, drel + (size_t)h * K * dh, du + (size_t)h * dh,
                             dvb + (size_t)h * dh, M, L, dh, scale, P, P + K);
            }
        }
        free(P);
    }
    return bad ? -2 : 0;
}
