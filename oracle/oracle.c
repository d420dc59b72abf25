/*
 * Plain fp64 CPU oracle for fused candidate scoring.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it. It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes, per question b (source: PR #69 "cuda: add a fused
 * candidate-scoring kernel for CLM and Kev", the opening table of the two
 * models and the section "What is fused, precisely"):
 *
 *   t_k   = sum_d C[b,k,d] * q[b,d]                      (dot with the query)
 *   sim_k = t_k / ( max(|q_b|, eps) * max(|c_k|, eps) )  (cosine, CLM)
 *   sim_k = t_k                                          (plain dot, Kev)
 *   z_k   = scale * sim_k / temperature
 *   p_k   = exp(z_k - m) / sum_j exp(z_j - m),  m = max_k z_k
 *
 * Readings of points the page leaves open:
 *   - the CLM scale is passed already exponentiated (scale = exp(logit_scale));
 *   - the temperature divides the scaled similarity (the page names the
 *     temperature only among the rejected arguments of "Verified on hardware");
 *   - eps clamps each norm on its own, so a zero candidate gets sim = 0 and a
 *     zero query makes every sim 0 (uniform result);
 *   - subtracting the maximum is the standard exact rewrite of the softmax
 *     (the page's overflow case needs it); it changes nothing mathematically.
 *
 * Everything is accumulated in double, in index order, with no blocking,
 * reordering or fusion. Inputs are float32 (the values the GPU sees); the
 * outputs are double.
 */
#include <math.h>
#include <stddef.h>

/* Similarity logits z[b,k] for B questions. Q is [B,D], C is [B,K,D], z is
 * [B,K], all row-major and contiguous. Returns 0, or -1 for a bad size. */
int oracle_logits(const float *Q, const float *C, long B, long K, long D,
                  int normalize, double scale, double temperature, double eps,
                  double *z)
{
    if (B < 0 || K < 0 || D < 0) return -1;
    for (long b = 0; b < B; ++b) {
        const float *q = Q + (size_t)b * (size_t)D;
        double qq = 0.0;
        for (long d = 0; d < D; ++d) qq += (double)q[d] * (double)q[d];
        double qnorm = sqrt(qq);
        for (long k = 0; k < K; ++k) {
            const float *c = C + ((size_t)b * (size_t)K + (size_t)k) * (size_t)D;
            double t = 0.0;
            for (long d = 0; d < D; ++d) t += (double)c[d] * (double)q[d];
            double sim = t;
            if (normalize) {
                double cc = 0.0;
                for (long d = 0; d < D; ++d) cc += (double)c[d] * (double)c[d];
                double cnorm = sqrt(cc);
                double a = qnorm > eps ? qnorm : eps;
                double c_ = cnorm > eps ? cnorm : eps;
                sim = t / (a * c_);
            }
            z[(size_t)b * (size_t)K + (size_t)k] = scale * sim / temperature;
        }
    }
    return 0;
}

/* Softmax of each of the B rows of z[B,K] into p[B,K]. */
int oracle_softmax(const double *z, long B, long K, double *p)
{
    if (B < 0 || K < 0) return -1;
    for (long b = 0; b < B; ++b) {
        const double *zr = z + (size_t)b * (size_t)K;
        double *pr = p + (size_t)b * (size_t)K;
        if (K == 0) continue;
        double m = zr[0];
        for (long k = 1; k < K; ++k)
            if (zr[k] > m) m = zr[k];
        double s = 0.0;
        for (long k = 0; k < K; ++k) {
            pr[k] = exp(zr[k] - m);
            s += pr[k];
        }
        for (long k = 0; k < K; ++k) pr[k] = pr[k] / s;
    }
    return 0;
}

/* The whole readout: logits, then softmax, for B questions. z may be NULL,
 * in which case the logits go through the output buffer p itself. */
int oracle_score_batch(const float *Q, const float *C, long B, long K, long D,
                       int normalize, double scale, double temperature,
                       double eps, double *p)
{
    int rc = oracle_logits(Q, C, B, K, D, normalize, scale, temperature, eps, p);
    if (rc != 0) return rc;
    /* Row by row, the softmax reads z[b,:] fully before writing p[b,:]
     * except for the in-place exp, which reads z[b,k] before writing p[b,k]. */
    return oracle_softmax(p, B, K, p);
}

/* Projection of feature rows by a weight matrix (the caller-side heads of
 * PR #69's opening table: CLM's state_head / action_head, Kev's k() / q()):
 *   P[r][n] = sum_i H[r][i] * W[n][i]
 * H is [R][Din], W is [D][Din] (one output feature per row of W), P is
 * [R][D]; float inputs (the values the GPU sees), double accumulation in
 * index order. Returns 0, or -1 for a bad size. */
int oracle_project(const float *H, const float *W, long R, long Din, long D, double *P)
{
    if (R < 0 || Din < 0 || D < 0) return -1;
    for (long r = 0; r < R; ++r) {
        const float *h = H + (size_t)r * (size_t)Din;
        for (long n = 0; n < D; ++n) {
            const float *w = W + (size_t)n * (size_t)Din;
            double acc = 0.0;
            for (long i = 0; i < Din; ++i) acc += (double)h[i] * (double)w[i];
            P[(size_t)r * (size_t)D + (size_t)n] = acc;
        }
    }
    return 0;
}
