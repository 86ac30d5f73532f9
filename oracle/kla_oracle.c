/*
 * kla_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, sequential fp64 CPU restatement of the Kaczmarz Linear
 * Attention (KLA) recurrence.  Only the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header or
 * constant with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes follows "KLA: Kaczmarz Linear Attention"
 * (gist.science/ko/paper/2605.08587), section "KLA update rule":
 *
 *   beta_t = eta_t / (||k_t||_2^2 + eps)
 *   S_t    = S~_{t-1} + beta_t k_t e_t^T,   e_t = v_t - S~_{t-1}^T k_t
 *
 * with the decayed previous state S~_{t-1} = a_t S_{t-1}, a_t = exp(g_t)
 * (the page's "decay gate", section "Implementation"; the exponential form of
 * the gate and the readout o_t = S_t^T q_t are the problem statement this
 * library is built to: one scalar log-decay g_t <= 0 and one relaxation gate
 * eta_t per (batch, token, head)).  The state has shape d_k x d_v (section
 * "Implementation": the GDN state shape is kept).
 *
 * Readings where the page is silent (each one is listed with its reason in
 * the design notes):
 *   - readout uses the state AFTER the token's update: o_t = S_t^T q_t;
 *   - no 1/sqrt(d_k) scaling of q and no extra normalisation of q or k;
 *   - eps is added to ||k_t||^2 inside the denominator.
 *
 * KLA_ORACLE_BETA_DIRECT takes beta_t = eta_t as given (eps unused): the
 * learned scalar coefficient of Gated DeltaNet that the same page's sections
 * "Problem statement" and "Methodology" name as what KLA replaces; with
 * g = 0 it is the ungated delta rule.  The library exposes this step size
 * as KLA_BETA_DIRECT.
 *
 * Test hook (never exported by the CUDA library): KLA_ORACLE_NO_ERASE drops
 * the erase term and uses unit write strength, S_t = a_t S_{t-1} + k_t v_t^T,
 * i.e. plain gated linear attention, so that a brute-force masked-attention
 * computation can pin the decay and readout parts of this loop.
 *
 * Layouts (row-major, contiguous):
 *   q, k  : [B, T, H, dk]      v, o : [B, T, H, dv]
 *   g, eta: [B, T, H]           h0, hT: [B, H, dk, dv]
 *   states (optional): [B, H, T, dk, dv], states[..., t, :, :] = S_t
 *
 * kla_oracle_backward is the reverse-mode derivative of the same loop: given
 * dL/do_t and dL/dS_T it returns dL/d{q,k,v,g,eta} and dL/dh0.  It first
 * runs the forward loop for one head and keeps every state S_t, then walks
 * t = T-1 .. 0 applying the chain rule to each operation of one step in
 * reverse order (readout, update, residual, decay, step size).  It is pinned
 * by central finite differences of kla_oracle_forward and by torch autograd.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread ... -lm
 * (no -ffast-math: every operation is IEEE fp64 in program order).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KLA_ORACLE_NO_ERASE 1
#define KLA_ORACLE_BETA_DIRECT 2

typedef struct {
    const double *q, *k, *v, *g, *eta, *h0;
    double eps;
    double *o, *hT, *states;
    int64_t B, T, H, dk, dv;
    int flags;
    int64_t next_unit; /* shared work counter over (b,h) units */
    pthread_mutex_t lock;
} job_t;

/* One (b,h) head: the plain sequential loop over t. */
static void run_head(job_t *J, int64_t b, int64_t h, double *S, double *x) {
    const int64_t T = J->T, H = J->H, dk = J->dk, dv = J->dv;
    /* S <- h0 (or zeros) */
    if (J->h0) {
        memcpy(S, J->h0 + (b * H + h) * dk * dv, sizeof(double) * dk * dv);
    } else {
        memset(S, 0, sizeof(double) * dk * dv);
    }
    for (int64_t t = 0; t < T; ++t) {
        const int64_t tok = (b * T + t) * H + h;
        const double *qt = J->q + tok * dk;
        const double *kt = J->k + tok * dk;
        const double *vt = J->v + tok * dv;
        const double a = exp(J->g[tok]);

        /* S~ = a * S  (decay gate) */
        for (int64_t i = 0; i < dk * dv; ++i) S[i] = a * S[i];

        if (J->flags & KLA_ORACLE_NO_ERASE) {
            /* plain gated linear attention: S = S~ + k v^T */
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += kt[i] * vt[j];
        } else {
            /* beta = eta / (||k||^2 + eps), or eta as given */
            double beta = J->eta[tok];
            if (!(J->flags & KLA_ORACLE_BETA_DIRECT)) {
                double kk = 0.0;
                for (int64_t i = 0; i < dk; ++i) kk += kt[i] * kt[i];
                beta = J->eta[tok] / (kk + J->eps);
            }
            /* e = v - S~^T k */
            for (int64_t j = 0; j < dv; ++j) x[j] = 0.0;
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j) x[j] += S[i * dv + j] * kt[i];
            for (int64_t j = 0; j < dv; ++j) x[j] = vt[j] - x[j];
            /* S = S~ + beta k e^T */
            for (int64_t i = 0; i < dk; ++i) {
                const double bk = beta * kt[i];
                for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += bk * x[j];
            }
        }
        /* o = S^T q */
        double *ot = J->o + tok * dv;
        for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) ot[j] += S[i * dv + j] * qt[i];
        if (J->states)
            memcpy(J->states + ((b * H + h) * T + t) * dk * dv, S, sizeof(double) * dk * dv);
    }
    if (J->hT) memcpy(J->hT + (b * H + h) * dk * dv, S, sizeof(double) * dk * dv);
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)(J->dk * J->dv));
    double *x = (double *)malloc(sizeof(double) * (size_t)J->dv);
    if (!S || !x) { free(S); free(x); return (void *)1; }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= J->B * J->H) break;
        run_head(J, u / J->H, u % J->H, S, x);
    }
    free(S);
    free(x);
    return NULL;
}

/*
 * Returns 0 on success, -1 on bad arguments, -2 on allocation or thread
 * failure.  nthreads <= 0 means one thread per (b,h) unit, capped at 64.
 */
int kla_oracle_forward(const double *q, const double *k, const double *v,
                       const double *g, const double *eta, double eps,
                       const double *h0, double *o, double *hT, double *states,
                       int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                       int flags, int nthreads) {
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0) return -1;
    if (!o || (T > 0 && (!q || !k || !v || !g || !eta))) return -1;
    job_t J;
    J.q = q; J.k = k; J.v = v; J.g = g; J.eta = eta; J.h0 = h0; J.eps = eps;
    J.o = o; J.hT = hT; J.states = states;
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv; J.flags = flags;
    J.next_unit = 0;
    pthread_mutex_init(&J.lock, NULL);
    int64_t units = B * H;
    int n = nthreads > 0 ? nthreads : (int)(units < 64 ? units : 64);
    if (n > units) n = (int)units;
    if (n < 1) n = 1;
    int rc = 0;
    if (n == 1) {
        if (worker(&J) != NULL) rc = -2;
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n);
        if (!th) { pthread_mutex_destroy(&J.lock); return -2; }
        int started = 0;
        for (int i = 0; i < n; ++i) {
            if (pthread_create(&th[i], NULL, worker, &J) != 0) { rc = -2; break; }
            ++started;
        }
        for (int i = 0; i < started; ++i) {
            void *ret = NULL;
            pthread_join(th[i], &ret);
            if (ret != NULL) rc = -2;
        }
        free(th);
    }
    pthread_mutex_destroy(&J.lock);
    return rc;
}


/* ------------------------------------------------------------------------ */
/* Reverse mode.                                                            */
/* ------------------------------------------------------------------------ */

typedef struct {
    const double *q, *k, *v, *g, *eta, *h0, *dout, *dhT;
    double eps;
    double *dq, *dk, *dv, *dg, *deta, *dh0;
    int64_t B, T, H, dk_, dv_;
    int flags;
    int64_t next_unit;
    pthread_mutex_t lock;
} bjob_t;

/* One (b,h) head.  Sall holds S_{-1} = h0, S_0, ..., S_{T-1}; dS and Sd are
 * dk x dv scratch; x, de are dv scratch. */
static void bwd_head(bjob_t *J, int64_t b, int64_t h, double *Sall, double *dS, double *Sd,
                     double *x, double *de) {
    const int64_t T = J->T, H = J->H, dk = J->dk_, dv = J->dv_, n = dk * dv;
    const int direct = (J->flags & KLA_ORACLE_BETA_DIRECT) != 0;

    /* forward, keeping every state */
    if (J->h0) memcpy(Sall, J->h0 + (b * H + h) * n, sizeof(double) * n);
    else memset(Sall, 0, sizeof(double) * n);
    for (int64_t t = 0; t < T; ++t) {
        const int64_t tok = (b * T + t) * H + h;
        const double *kt = J->k + tok * dk, *vt = J->v + tok * dv;
        const double a = exp(J->g[tok]);
        const double *Sp = Sall + t * n;
        double *S = Sall + (t + 1) * n;
        for (int64_t i = 0; i < n; ++i) S[i] = a * Sp[i];
        double beta = J->eta[tok];
        if (!direct) {
            double kk = 0.0;
            for (int64_t i = 0; i < dk; ++i) kk += kt[i] * kt[i];
            beta = J->eta[tok] / (kk + J->eps);
        }
        for (int64_t j = 0; j < dv; ++j) x[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) x[j] += S[i * dv + j] * kt[i];
        for (int64_t j = 0; j < dv; ++j) x[j] = vt[j] - x[j];
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += beta * kt[i] * x[j];
    }

    /* reverse: dS holds dL/dS_t while step t is undone */
    if (J->dhT) memcpy(dS, J->dhT + (b * H + h) * n, sizeof(double) * n);
    else memset(dS, 0, sizeof(double) * n);
    for (int64_t t = T - 1; t >= 0; --t) {
        const int64_t tok = (b * T + t) * H + h;
        const double *qt = J->q + tok * dk, *kt = J->k + tok * dk, *vt = J->v + tok * dv;
        const double *dot = J->dout + tok * dv;
        const double a = exp(J->g[tok]);
        const double *Sp = Sall + t * n;        /* S_{t-1} */
        const double *S = Sall + (t + 1) * n;   /* S_t */
        double kk = 0.0;
        for (int64_t i = 0; i < dk; ++i) kk += kt[i] * kt[i];
        const double beta = direct ? J->eta[tok] : J->eta[tok] / (kk + J->eps);

        /* readout o_t = S_t^T q_t: dS += q_t do_t^T, dq_t = S_t do_t */
        double *dqt = J->dq + tok * dk;
        for (int64_t i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
                dS[i * dv + j] += qt[i] * dot[j];
                acc += S[i * dv + j] * dot[j];
            }
            dqt[i] = acc;
        }
        /* recompute S~ = a S_{t-1} and e = v - S~^T k */
        for (int64_t i = 0; i < n; ++i) Sd[i] = a * Sp[i];
        for (int64_t j = 0; j < dv; ++j) x[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) x[j] += Sd[i * dv + j] * kt[i];
        for (int64_t j = 0; j < dv; ++j) x[j] = vt[j] - x[j];

        /* update S_t = S~ + beta k e^T */
        double dbeta = 0.0;
        for (int64_t j = 0; j < dv; ++j) de[j] = 0.0;
        double *dkt = J->dk + tok * dk;
        for (int64_t i = 0; i < dk; ++i) {
            double r = 0.0;                      /* (dS e)_i */
            for (int64_t j = 0; j < dv; ++j) {
                r += dS[i * dv + j] * x[j];
                de[j] += beta * kt[i] * dS[i * dv + j];
            }
            dbeta += kt[i] * r;
            dkt[i] = beta * r;
        }
        /* residual e = v - S~^T k: dv = de, dk -= S~ de, dS~ = dS - k de^T */
        double *dvt = J->dv + tok * dv;
        for (int64_t j = 0; j < dv; ++j) dvt[j] = de[j];
        for (int64_t i = 0; i < dk; ++i) {
            double r = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
                r += Sd[i * dv + j] * de[j];
                dS[i * dv + j] -= kt[i] * de[j];
            }
            dkt[i] -= r;
        }
        /* decay S~ = a S_{t-1}: dg = a <dS~, S_{t-1}>, dS_{t-1} = a dS~ */
        double da = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            da += dS[i] * Sp[i];
            dS[i] *= a;
        }
        J->dg[tok] = a * da;
        /* step size */
        if (direct) {
            J->deta[tok] = dbeta;
        } else {
            const double den = kk + J->eps;
            J->deta[tok] = dbeta / den;
            for (int64_t i = 0; i < dk; ++i) dkt[i] -= 2.0 * beta * dbeta / den * kt[i];
        }
    }
    if (J->dh0) memcpy(J->dh0 + (b * H + h) * n, dS, sizeof(double) * n);
}

static void *bwd_worker(void *arg) {
    bjob_t *J = (bjob_t *)arg;
    const size_t n = (size_t)(J->dk_ * J->dv_);
    double *Sall = (double *)malloc(sizeof(double) * n * (size_t)(J->T + 1));
    double *dS = (double *)malloc(sizeof(double) * n);
    double *Sd = (double *)malloc(sizeof(double) * n);
    double *x = (double *)malloc(sizeof(double) * (size_t)J->dv_);
    double *de = (double *)malloc(sizeof(double) * (size_t)J->dv_);
    void *rc = NULL;
    if (!Sall || !dS || !Sd || !x || !de) {
        rc = (void *)1;
    } else {
        for (;;) {
            pthread_mutex_lock(&J->lock);
            const int64_t u = J->next_unit++;
            pthread_mutex_unlock(&J->lock);
            if (u >= J->B * J->H) break;
            bwd_head(J, u / J->H, u % J->H, Sall, dS, Sd, x, de);
        }
    }
    free(Sall); free(dS); free(Sd); free(x); free(de);
    return rc;
}

/*
 * Gradients of kla_oracle_forward.  dout [B,T,H,dv]; dhT [B,H,dk,dv] or NULL
 * (zero); dh0 may be NULL.  Outputs have the layouts of their inputs.  The
 * no-erase test mode has no derivative here (-1).  Returns as
 * kla_oracle_forward.
 */
int kla_oracle_backward(const double *q, const double *k, const double *v,
                        const double *g, const double *eta, double eps,
                        const double *h0, const double *dout, const double *dhT,
                        double *dq, double *dk, double *dv, double *dg, double *deta,
                        double *dh0, int64_t B, int64_t T, int64_t H, int64_t dk_,
                        int64_t dv_, int flags, int nthreads) {
    if (B < 0 || T < 0 || H < 0 || dk_ <= 0 || dv_ <= 0) return -1;
    if (flags & KLA_ORACLE_NO_ERASE) return -1;
    if (T > 0 && (!q || !k || !v || !g || !eta || !dout || !dq || !dk || !dv || !dg || !deta))
        return -1;
    bjob_t J;
    J.q = q; J.k = k; J.v = v; J.g = g; J.eta = eta; J.h0 = h0; J.dout = dout; J.dhT = dhT;
    J.eps = eps;
    J.dq = dq; J.dk = dk; J.dv = dv; J.dg = dg; J.deta = deta; J.dh0 = dh0;
    J.B = B; J.T = T; J.H = H; J.dk_ = dk_; J.dv_ = dv_; J.flags = flags;
    J.next_unit = 0;
    pthread_mutex_init(&J.lock, NULL);
    int64_t units = B * H;
    int n = nthreads > 0 ? nthreads : (int)(units < 64 ? units : 64);
    if (n > units) n = (int)units;
    if (n < 1) n = 1;
    int rc = 0;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n);
    if (!th) { pthread_mutex_destroy(&J.lock); return -2; }
    int started = 0;
    for (int i = 0; i < n; ++i) {
        if (pthread_create(&th[i], NULL, bwd_worker, &J) != 0) { rc = -2; break; }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -2;
    }
    free(th);
    pthread_mutex_destroy(&J.lock);
    return rc;
}
