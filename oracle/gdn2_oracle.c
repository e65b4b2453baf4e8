/*
 * FP64 CPU oracle for the Gated DeltaNet-2 (GDN-2) prefill forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes (FlashInfer docs, "flashinfer.gdn2_prefill.
 * chunk_gated_delta_rule2", the recurrence in the op description), per
 * sequence n and value head hv, token by token, in double precision:
 *
 *     S      <- diag(exp(g_t)) S                      (decay, per key channel)
 *     u      =  w_t * v_t - (beta_t * k_t)^T S          (erase read of decayed S)
 *     S      <- S + k_t u^T                             (write)
 *     o_t    =  scale * q_t^T S                         (read after the write)
 *
 * S is K x V, initialised from initial_state[n, hs] (or zero); the final S
 * is returned.  Heads (FlashInfer docs' parameter list): H query heads, HK
 * key heads and HV value heads, where HK equals H or HV and H, HV are equal
 * or one a multiple of the other.  There is one state per state head hs <
 * HS = max(H, HV) (the docs' num_sab_heads: g, beta, w, the states and the
 * output are per state head).  State head hs reads query head
 * hs / (HS / H), key head hs / (HS / HK) and value head hs / (HS / HV)
 * (contiguous groups share a head; with HV = HS this is value head hv
 * reading key head hv / (HV / H)).  Missing gates take the
 * defaults the same parameter list gives: g = 0, beta = 1, w = 1.  With
 * use_qk_l2norm the rows of q and k are first divided by max(||x||_2, 1e-12)
 * (the docs' use_qk_l2norm_in_kernel; the epsilon follows the FlashGDN-2
 * quick start's torch.nn.functional.normalize).
 *
 * Inputs are double arrays, already converted exactly from the bf16/fp32
 * bytes the GPU sees.  Layouts (row-major, contiguous):
 *   q [T_tot, H, K]   k [T_tot, HK, K]   v [T_tot, HV, V]
 *   g, beta [T_tot, HS, K]   w [T_tot, HS, V]   h0 [N, HS, K, V]
 *   cu [N + 1] (int64)       o [T_tot, HS, V]   hT [N, HS, K, V]
 * Work is split over (n, hs) units with POSIX threads; each unit is
 * independent, so the thread count does not change any result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *g, *beta, *w, *h0;
    const int64_t *cu;
    int64_t T_tot;
    int N, H, HK, HV, HS, K, V, use_l2;
    double scale;
    const int32_t *units; /* pairs (n, hs); NULL = every unit */
    int n_units;
    double *o, *hT;
    int next; /* shared work counter */
    pthread_mutex_t lock;
    int err;
} job_t;

static void l2_normalise(const double *x, double *y, int n, int use_l2)
{
    double ss = 0.0, d;
    int i;
    if (!use_l2) {
        memcpy(y, x, (size_t)n * sizeof(double));
        return;
    }
    for (i = 0; i < n; i++) ss += x[i] * x[i];
    d = sqrt(ss);
    if (d < 1e-12) d = 1e-12;
    for (i = 0; i < n; i++) y[i] = x[i] / d;
}

/* One (n, hs) unit: the plain recurrence, token by token. */
static int run_unit(job_t *J, int n, int hs, double *S, double *qt, double *kt, double *u)
{
    const int K = J->K, V = J->V, H = J->H, HK = J->HK, HV = J->HV, HS = J->HS;
    /* head maps: contiguous groups of state heads share a q, k or v head */
    const int hq = hs / (HS / H);
    const int hk = hs / (HS / HK);
    const int hvv = hs / (HS / HV);
    const int64_t t0 = J->cu[n], t1 = J->cu[n + 1];
    int64_t t;
    int c, j;

    if (J->h0) memcpy(S, J->h0 + ((size_t)n * HS + hs) * K * V, (size_t)K * V * sizeof(double));
    else memset(S, 0, (size_t)K * V * sizeof(double));

    for (t = t0; t < t1; t++) {
        const double *g = J->g ? J->g + ((size_t)t * HS + hs) * K : NULL;
        const double *b = J->beta ? J->beta + ((size_t)t * HS + hs) * K : NULL;
        const double *w = J->w ? J->w + ((size_t)t * HS + hs) * V : NULL;
        const double *vv = J->v + ((size_t)t * HV + hvv) * V;
        double *o = J->o + ((size_t)t * HS + hs) * V;

        l2_normalise(J->q + ((size_t)t * H + hq) * K, qt, K, J->use_l2);
        l2_normalise(J->k + ((size_t)t * HK + hk) * K, kt, K, J->use_l2);

        /* decay: S <- diag(exp(g_t)) S */
        if (g) {
            for (c = 0; c < K; c++) {
                const double a = exp(g[c]);
                double *row = S + (size_t)c * V;
                for (j = 0; j < V; j++) row[j] *= a;
            }
        }
        /* erase read on the decayed state, then the gated write value */
        for (j = 0; j < V; j++) u[j] = 0.0;
        for (c = 0; c < K; c++) {
            const double bk = (b ? b[c] : 1.0) * kt[c];
            const double *row = S + (size_t)c * V;
            for (j = 0; j < V; j++) u[j] += bk * row[j];
        }
        for (j = 0; j < V; j++) u[j] = (w ? w[j] : 1.0) * vv[j] - u[j];
        /* write: S <- S + k_t u^T */
        for (c = 0; c < K; c++) {
            double *row = S + (size_t)c * V;
            for (j = 0; j < V; j++) row[j] += kt[c] * u[j];
        }
        /* output after the write: o_t = scale * q_t^T S */
        for (j = 0; j < V; j++) o[j] = 0.0;
        for (c = 0; c < K; c++) {
            const double *row = S + (size_t)c * V;
            for (j = 0; j < V; j++) o[j] += qt[c] * row[j];
        }
        for (j = 0; j < V; j++) o[j] *= J->scale;
    }
    memcpy(J->hT + ((size_t)n * HS + hs) * K * V, S, (size_t)K * V * sizeof(double));
    return 0;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const int total = J->units ? J->n_units : J->N * J->HS;
    double *S = (double *)malloc((size_t)J->K * J->V * sizeof(double));
    double *qt = (double *)malloc((size_t)J->K * sizeof(double));
    double *kt = (double *)malloc((size_t)J->K * sizeof(double));
    double *u = (double *)malloc((size_t)J->V * sizeof(double));
    if (!S || !qt || !kt || !u) {
        pthread_mutex_lock(&J->lock);
        J->err = 1;
        pthread_mutex_unlock(&J->lock);
        free(S); free(qt); free(kt); free(u);
        return NULL;
    }
    for (;;) {
        int i, n, hs;
        pthread_mutex_lock(&J->lock);
        i = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (i >= total) break;
        if (J->units) {
            n = J->units[2 * i];
            hs = J->units[2 * i + 1];
        } else {
            n = i / J->HS;
            hs = i % J->HS;
        }
        run_unit(J, n, hs, S, qt, kt, u);
    }
    free(S); free(qt); free(kt); free(u);
    return NULL;
}

/*
 * Returns 0 on success, -1 on a bad argument, -2 on allocation failure.
 * g, beta, w, h0 may be NULL (defaults above).  Only the rows of o that
 * belong to the requested units, and only their final states, are written.
 */
int gdn2_oracle_forward(const double *q, const double *k, const double *v,
                        const double *g, const double *beta, const double *w,
                        double scale, const double *h0, const int64_t *cu,
                        int64_t T_tot, int N, int H, int HK, int HV, int K, int V,
                        int use_qk_l2norm, const int32_t *units, int n_units,
                        double *o, double *hT, int n_threads)
{
    job_t J;
    pthread_t *th;
    int i, n;

    if (!q || !k || !v || !cu || !o || !hT) return -1;
    if (N < 0 || H <= 0 || HK <= 0 || HV <= 0 || K <= 0 || V <= 0) return -1;
    if (HK != H && HK != HV) return -1;
    if (HV % H != 0 && H % HV != 0) return -1;
    if (cu[0] != 0 || cu[N] != T_tot) return -1;
    for (n = 0; n < N; n++)
        if (cu[n + 1] < cu[n]) return -1;
    if (units) {
        for (i = 0; i < n_units; i++)
            if (units[2 * i] < 0 || units[2 * i] >= N || units[2 * i + 1] < 0 ||
                units[2 * i + 1] >= (H > HV ? H : HV))
                return -1;
    }
    if (scale <= 0.0) scale = 1.0 / sqrt((double)K);

    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.w = w; J.h0 = h0;
    J.cu = cu; J.T_tot = T_tot; J.N = N; J.H = H; J.HK = HK; J.HV = HV; J.HS = H > HV ? H : HV;
    J.K = K; J.V = V;
    J.use_l2 = use_qk_l2norm; J.scale = scale;
    J.units = units; J.n_units = n_units; J.o = o; J.hT = hT;
    pthread_mutex_init(&J.lock, NULL);

    if (n_threads < 1) n_threads = 1;
    th = (pthread_t *)malloc((size_t)n_threads * sizeof(pthread_t));
    if (!th) return -2;
    for (i = 0; i < n_threads; i++) pthread_create(&th[i], NULL, worker, &J);
    for (i = 0; i < n_threads; i++) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return J.err ? -2 : 0;
}
