/*
 * EFLA oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, sequential fp64 implementation of the Error-Free Linear
 * Attention token mixer, used to check the CUDA path.  Only the tests, the
 * smoke entry and the CPU-baseline leg of the benchmark may load it; the
 * product path never does.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes, per (sequence, head), token by token:
 *
 *   lam_t   = ||k_t||^2
 *       ["Exact Flow Linear Attention" (gist.science), Metodologia 2:
 *        the rank-1 dynamics matrix A_t = k_t k_t^T has A_t^n = lam_t^{n-1} A_t]
 *   alpha_t = (1 - exp(-beta_t lam_t)) / lam_t, evaluated as
 *             -expm1(-beta_t lam_t) / lam_t; alpha_t = beta_t when lam_t == 0
 *       [same page, Metodologia 3; "Error-Free Linear Attention is a Free
 *        Lunch" (howistudyai), Step 1.  The lam -> 0 value is the limit of the
 *        formula, which the howistudyai page describes in Step 5 as small keys
 *        behaving like the delta rule.]
 *   S_t     = (I - alpha_t k_t k_t^T) S_{t-1} + alpha_t k_t v_t^T
 *       [gist.science, Metodologia 3; howistudyai, Step 2]
 *   o_t     = S_t^T q_t   (the state AFTER token t's update)
 *       [howistudyai, Step 3 and "Putting it all together (pipeline)"]
 *
 * With `euler` set, the gate is alpha_t = beta_t: the explicit-Euler (delta rule,
 * DeltaNet) step S_t = (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T that the
 * pages compare EFLA against [howistudyai, "Delta Rule (Linear Attention as
 * Online Learning)"; gist.science, "Enunciato del Problema"].
 *
 * The update is evaluated in the factored form
 *   x = S_{t-1}^T k_t;   S_t = S_{t-1} + alpha_t k_t (v_t - x)^T,
 * which is the same matrix as (I - alpha k k^T) S + alpha k v^T by
 * distributivity: (I - a k k^T) S + a k v^T = S - a k (k^T S) + a k v^T.
 * A literal d x d form of the same update is in oracle/literal.py and the
 * tests check that the two agree.
 *
 * Layouts (all row-major, fp64):
 *   q, k  [B, T, H, dk];  v [B, T, H, dv];  beta [B, T, H]
 *   S0, S_T [N, H, dk, dv]  (dv contiguous), S0 may be NULL (zeros)
 *   o     [B, T, H, dv]
 *   cu_seqlens [N+1] int64 or NULL.  When given, B must be 1 and sequence n
 *   covers tokens cu_seqlens[n] .. cu_seqlens[n+1]-1 of the packed T axis;
 *   sequences are independent and each starts from its own S0[n].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

double efla_oracle_alpha(double beta, double lam)
{
    if (lam > 0.0)
        return -expm1(-beta * lam) / lam;
    return beta;
}

/* One token of one head: updates S (dk x dv) in place and writes o (dv). */
static void oracle_token(const double *q, const double *k, const double *v, double beta,
                         double *S, double *o, int dk, int dv, double *x, int euler)
{
    double lam = 0.0;
    for (int i = 0; i < dk; ++i)
        lam += k[i] * k[i];
    const double a = euler ? beta : efla_oracle_alpha(beta, lam);

    for (int j = 0; j < dv; ++j)
        x[j] = 0.0;
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            x[j] += k[i] * S[(size_t)i * dv + j];

    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            S[(size_t)i * dv + j] += a * k[i] * (v[j] - x[j]);

    for (int j = 0; j < dv; ++j)
        o[j] = 0.0;
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            o[j] += q[i] * S[(size_t)i * dv + j];
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation failure. */
int efla_oracle_fwd_mode(const double *q, const double *k, const double *v, const double *beta,
                         const double *S0, const int64_t *cu_seqlens, double *o, double *S_T,
                         int B, int T, int H, int dk, int dv, int N, int nthreads, int euler)
{
    if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0 || N < 0)
        return -1;
    if (cu_seqlens) {
        if (B != 1)
            return -1;
        if (cu_seqlens[0] != 0 || cu_seqlens[N] != T)
            return -1;
        for (int n = 0; n < N; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n])
                return -1;
    } else if (N != B) {
        return -1;
    }
    const long units = (long)N * H;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (long u = 0; u < units; ++u) {
        const int n = (int)(u / H), h = (int)(u % H);
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        double *x = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!S || !x) {
            free(S);
            free(x);
            failed |= 1;
            continue;
        }
        const double *s0 = S0 ? S0 + ((size_t)n * H + h) * dk * dv : NULL;
        for (size_t e = 0; e < (size_t)dk * dv; ++e)
            S[e] = s0 ? s0[e] : 0.0;
        long t0, t1, b;
        if (cu_seqlens) {
            b = 0;
            t0 = cu_seqlens[n];
            t1 = cu_seqlens[n + 1];
        } else {
            b = n;
            t0 = 0;
            t1 = T;
        }
        for (long t = t0; t < t1; ++t) {
            const size_t row = ((size_t)b * T + t) * H + h;
            oracle_token(q + row * dk, k + row * dk, v + row * dv, beta[row], S, o + row * dv,
                         dk, dv, x, euler);
        }
        if (S_T)
            memcpy(S_T + ((size_t)n * H + h) * dk * dv, S, sizeof(double) * (size_t)dk * dv);
        free(S);
        free(x);
    }
    return failed ? -2 : 0;
}

int efla_oracle_fwd(const double *q, const double *k, const double *v, const double *beta,
                    const double *S0, const int64_t *cu_seqlens, double *o, double *S_T,
                    int B, int T, int H, int dk, int dv, int N, int nthreads)
{
    return efla_oracle_fwd_mode(q, k, v, beta, S0, cu_seqlens, o, S_T, B, T, H, dk, dv, N, nthreads, 0);
}

/* One decode step for B*H independent heads; S [B, H, dk, dv] updated in place. */
int efla_oracle_decode_mode(const double *q, const double *k, const double *v, const double *beta,
                            double *S, double *o, int B, int H, int dk, int dv, int nthreads, int euler)
{
    if (B < 0 || H <= 0 || dk <= 0 || dv <= 0)
        return -1;
    const long units = (long)B * H;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static) reduction(| : failed)
#endif
    for (long u = 0; u < units; ++u) {
        double *x = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!x) {
            failed |= 1;
            continue;
        }
        oracle_token(q + u * dk, k + u * dk, v + u * dv, beta[u], S + u * (size_t)dk * dv,
                     o + u * dv, dk, dv, x, euler);
        free(x);
    }
    return failed ? -2 : 0;
}

int efla_oracle_decode(const double *q, const double *k, const double *v, const double *beta,
                       double *S, double *o, int B, int H, int dk, int dv, int nthreads)
{
    return efla_oracle_decode_mode(q, k, v, beta, S, o, B, H, dk, dv, nthreads, 0);
}

/*
 * Gradients of the forward (reverse mode), for the backward pass.
 *
 * The pages give no backward formulas; this is the chain rule applied, step by
 * step in reverse token order, to the recurrence above.  For one token, with
 * S_{t-1} the state before it and S_t after it:
 *   o_t = S_t^T q_t          -> dq_t = S_t do_t;          dS_t += q_t do_t^T
 *   S_t = S_{t-1} + k u^T    -> du = dS_t^T k;            dk_t += dS_t u
 *   u = alpha (v - x)        -> dv_t = alpha du;          dalpha = du . (v - x);  dx = -alpha du
 *   x = S_{t-1}^T k          -> dk_t += S_{t-1} dx;       dS_{t-1} = dS_t + k dx^T
 *   alpha = f(beta, lam)     -> dbeta_t = dalpha df/dbeta; dk_t += 2 dalpha df/dlam k
 * starting from dS_T and ending with dS0 = dS_{t0-1}.  All states of the
 * sequence are kept from a forward sweep (plain; sized for test cases).
 *
 * The gate's derivatives, with z = beta lam and f = -expm1(-z)/lam:
 *   df/dbeta = exp(-z);   df/dlam = (beta exp(-z) - f) / lam = beta^2 g'(z),
 *   g(z) = (1 - e^{-z}) / z,  g'(z) = -1/2 + z/3 - z^2/8 + z^3/30 - z^4/144 + ...
 * (the series is used for |z| < 1e-3, where the difference form cancels);
 * at lam = 0: f = beta, df/dbeta = 1, df/dlam = -beta^2/2.  Delta rule: 1 and 0.
 */
void efla_oracle_gate_grad(double beta, double lam, int euler, double *dfdb, double *dfdl)
{
    if (euler) {
        *dfdb = 1.0;
        *dfdl = 0.0;
        return;
    }
    const double z = beta * lam;
    if (lam > 0.0 && fabs(z) >= 1e-3) {
        const double f = -expm1(-z) / lam;
        *dfdb = exp(-z);
        *dfdl = (beta * exp(-z) - f) / lam;
    } else {
        *dfdb = lam > 0.0 ? exp(-z) : 1.0;
        *dfdl = beta * beta * (-0.5 + z / 3.0 - z * z / 8.0 + z * z * z / 30.0 - z * z * z * z / 144.0);
    }
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation failure.
 * do_ [B,T,H,dv], dST [B,H,dk,dv] or NULL (zero); outputs dq, dk [B,T,H,dk],
 * dv [B,T,H,dv], dbeta [B,T,H], dS0 [B,H,dk,dv] (dS0 may be NULL). */
int efla_oracle_bwd_mode(const double *q, const double *k, const double *v, const double *beta,
                         const double *S0, const double *do_, const double *dST, double *dq, double *dk,
                         double *dv_out, double *dbeta, double *dS0, int B, int T, int H, int dkd, int dvd,
                         int nthreads, int euler)
{
    if (B < 0 || T < 0 || H <= 0 || dkd <= 0 || dvd <= 0)
        return -1;
    const long units = (long)B * H;
    const size_t mat = (size_t)dkd * dvd;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (long un = 0; un < units; ++un) {
        const int b = (int)(un / H), h = (int)(un % H);
        double *St = (double *)malloc(sizeof(double) * mat * ((size_t)T + 1));  /* states 0..T */
        double *xs = (double *)malloc(sizeof(double) * (size_t)dvd * (T > 0 ? T : 1));
        double *us = (double *)malloc(sizeof(double) * (size_t)dvd * (T > 0 ? T : 1));
        double *al = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
        double *lm = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
        double *G = (double *)malloc(sizeof(double) * mat);
        double *du = (double *)malloc(sizeof(double) * dvd), *dx = (double *)malloc(sizeof(double) * dvd);
        if (!St || !xs || !us || !al || !lm || !G || !du || !dx) {
            free(St); free(xs); free(us); free(al); free(lm); free(G); free(du); free(dx);
            failed |= 1;
            continue;
        }
        const double *s0 = S0 ? S0 + ((size_t)b * H + h) * mat : NULL;
        for (size_t e = 0; e < mat; ++e)
            St[e] = s0 ? s0[e] : 0.0;
        /* forward sweep, keeping every state */
        for (int t = 0; t < T; ++t) {
            const size_t row = ((size_t)b * T + t) * H + h;
            const double *kt = k + row * dkd, *vt = v + row * dvd;
            const double *Sp = St + (size_t)t * mat;
            double *Sn = St + (size_t)(t + 1) * mat;
            double lam = 0.0;
            for (int i = 0; i < dkd; ++i)
                lam += kt[i] * kt[i];
            const double a = euler ? beta[row] : efla_oracle_alpha(beta[row], lam);
            double *x = xs + (size_t)t * dvd, *u = us + (size_t)t * dvd;
            for (int j = 0; j < dvd; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dkd; ++i)
                    acc += kt[i] * Sp[(size_t)i * dvd + j];
                x[j] = acc;
                u[j] = a * (vt[j] - acc);
            }
            for (int i = 0; i < dkd; ++i)
                for (int j = 0; j < dvd; ++j)
                    Sn[(size_t)i * dvd + j] = Sp[(size_t)i * dvd + j] + kt[i] * u[j];
            al[t] = a;
            lm[t] = lam;
        }
        /* reverse sweep */
        const double *g0 = dST ? dST + ((size_t)b * H + h) * mat : NULL;
        for (size_t e = 0; e < mat; ++e)
            G[e] = g0 ? g0[e] : 0.0;
        for (int t = T - 1; t >= 0; --t) {
            const size_t row = ((size_t)b * T + t) * H + h;
            const double *qt = q + row * dkd, *kt = k + row * dkd, *vt = v + row * dvd, *dot = do_ + row * dvd;
            const double *Sp = St + (size_t)t * mat, *Sc = St + (size_t)(t + 1) * mat;
            const double *x = xs + (size_t)t * dvd, *u = us + (size_t)t * dvd;
            const double a = al[t];
            double *dqt = dq + row * dkd, *dkt = dk + row * dkd, *dvt = dv_out + row * dvd;
            /* o_t = S_t^T q_t */
            for (int i = 0; i < dkd; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dvd; ++j)
                    acc += Sc[(size_t)i * dvd + j] * dot[j];
                dqt[i] = acc;
            }
            for (int i = 0; i < dkd; ++i)
                for (int j = 0; j < dvd; ++j)
                    G[(size_t)i * dvd + j] += qt[i] * dot[j];
            /* S_t = S_{t-1} + k u^T */
            for (int j = 0; j < dvd; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dkd; ++i)
                    acc += G[(size_t)i * dvd + j] * kt[i];
                du[j] = acc;
            }
            for (int i = 0; i < dkd; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dvd; ++j)
                    acc += G[(size_t)i * dvd + j] * u[j];
                dkt[i] = acc;
            }
            /* u = alpha (v - x) */
            double da = 0.0;
            for (int j = 0; j < dvd; ++j) {
                dvt[j] = a * du[j];
                da += du[j] * (vt[j] - x[j]);
                dx[j] = -a * du[j];
            }
            /* x = S_{t-1}^T k */
            for (int i = 0; i < dkd; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dvd; ++j)
                    acc += Sp[(size_t)i * dvd + j] * dx[j];
                dkt[i] += acc;
            }
            for (int i = 0; i < dkd; ++i)
                for (int j = 0; j < dvd; ++j)
                    G[(size_t)i * dvd + j] += kt[i] * dx[j];
            /* alpha = f(beta, lam), lam = ||k||^2 */
            double dfdb, dfdl;
            efla_oracle_gate_grad(beta[row], lm[t], euler, &dfdb, &dfdl);
            dbeta[row] = da * dfdb;
            for (int i = 0; i < dkd; ++i)
                dkt[i] += 2.0 * da * dfdl * kt[i];
        }
        if (dS0)
            memcpy(dS0 + ((size_t)b * H + h) * mat, G, sizeof(double) * mat);
        free(St); free(xs); free(us); free(al); free(lm); free(G); free(du); free(dx);
    }
    return failed ? -2 : 0;
}

int efla_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
