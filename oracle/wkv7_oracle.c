/*
 * wkv7_oracle.c -- fp64 CPU oracle for the WKV-7 recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library,
 * its Python binding) links, loads or calls this file.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg use it.
 *
 * What it computes (Core AI model zoo, "Recurrent / linear-attention LLMs on
 * Core AI", section 1, the per-head WKV7 formula written with S = [K, V]):
 * for every sequence, head h and token t, in token order,
 *
 *     z   = kk^T S                        (projection of the OLD state)
 *     S   = diag(exp w) S - (kk .* a) z^T + k v^T
 *     o_t = S^T r                         (read-out of the NEW state)
 *
 * with S in R^{N x N}, rows indexed by the key channel i and columns by the
 * value channel j.  w is the log-decay, so the per-row decay is exp(w_i).
 * The same section's order "S = decay - delta; S += k v; o = r^T S" fixes
 * that both the decay and the delta term act on the old state and that the
 * read-out sees the state after the update.
 *
 * Readings taken where the pages are silent (also listed in the design
 * notes): kk is used exactly as passed (no normalisation inside), a is a
 * per-channel vector, there is no bonus term, S starts from the given
 * initial state or from zero, and is restarted at every sequence boundary.
 *
 * Arithmetic: every stored input (fp32, or bf16 widened exactly to fp32 by
 * the caller) is widened to double; all sums and products are in double;
 * exp is the C library's double exp.  There is no blocking, reordering or
 * chunking: it is the definition, one token at a time.
 *
 * Layout: token-major packed inputs [T_total, H, N]; sequence b owns tokens
 * cu_seqlens[b] .. cu_seqlens[b+1]-1.  States are [num_seqs, H, N, N] with the
 * value channel contiguous.
 *
 * Threads only split the independent (sequence, head) pairs; each pair is
 * still one sequential loop, so the result does not depend on the thread
 * count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* One (sequence, head) pair, tokens [t_begin, t_end). */
static void oracle_pair(int64_t t_begin, int64_t t_end, int H, int N, int h,
                        const float *r, const float *w, const float *k,
                        const float *v, const float *kk, const float *a,
                        const double *s0, double *S, double *z, double *o)
{
    int i, j;
    int64_t t;
    if (s0)
        memcpy(S, s0, sizeof(double) * (size_t)N * (size_t)N);
    else
        memset(S, 0, sizeof(double) * (size_t)N * (size_t)N);

    for (t = t_begin; t < t_end; ++t) {
        const size_t base = ((size_t)t * (size_t)H + (size_t)h) * (size_t)N;
        const float *rt = r + base, *wt = w + base, *kt = k + base;
        const float *vt = v + base, *kkt = kk + base, *at = a + base;
        double *ot = o + base;

        /* z_j = sum_i kk_i S[i][j], taken on the old state */
        for (j = 0; j < N; ++j) {
            double acc = 0.0;
            for (i = 0; i < N; ++i)
                acc += (double)kkt[i] * S[(size_t)i * N + j];
            z[j] = acc;
        }

        /* S[i][j] = exp(w_i) S[i][j] - (kk_i a_i) z_j + k_i v_j */
        for (i = 0; i < N; ++i) {
            const double decay = exp((double)wt[i]);
            const double c = (double)kkt[i] * (double)at[i];
            for (j = 0; j < N; ++j)
                S[(size_t)i * N + j] = decay * S[(size_t)i * N + j] - c * z[j] + (double)kt[i] * (double)vt[j];
        }

        /* o_j = sum_i r_i S[i][j], on the new state */
        for (j = 0; j < N; ++j) {
            double acc = 0.0;
            for (i = 0; i < N; ++i)
                acc += (double)rt[i] * S[(size_t)i * N + j];
            ot[j] = acc;
        }
    }
}

typedef struct {
    int num_seqs, H, N, nthreads, tid;
    const int64_t *cu;
    const float *r, *w, *k, *v, *kk, *a;
    const double *s0;
    double *o, *s_final;
    int failed;
} oracle_job;

static void *oracle_worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    const size_t NN = (size_t)job->N * (size_t)job->N;
    double *z = (double *)malloc(sizeof(double) * (size_t)job->N);
    const int64_t pairs = (int64_t)job->num_seqs * job->H;
    int64_t p;
    if (!z) {
        job->failed = 1;
        return NULL;
    }
    for (p = job->tid; p < pairs; p += job->nthreads) {
        const int b = (int)(p / job->H), h = (int)(p % job->H);
        const size_t slot = (size_t)b * job->H + h;
        oracle_pair(job->cu[b], job->cu[b + 1], job->H, job->N, h,
                    job->r, job->w, job->k, job->v, job->kk, job->a,
                    job->s0 ? job->s0 + slot * NN : NULL,
                    job->s_final + slot * NN, z, job->o);
    }
    free(z);
    return NULL;
}

/*
 * Run the recurrence over packed sequences.
 *   cu_seqlens : int64 [num_seqs + 1], cu[0] = 0, non-decreasing
 *   r,w,k,v,kk,a : float [T_total, H, N], T_total = cu[num_seqs]
 *   s0       : double [num_seqs, H, N, N] or NULL (zeros)
 *   o        : double [T_total, H, N]             (written)
 *   s_final  : double [num_seqs, H, N, N]         (written)
 *   nthreads : worker threads over (sequence, head) pairs (<= 0 means 1)
 * Returns 0 on success, -1 on a malformed argument, -2 if threads fail.
 */
int wkv7_oracle_run(int num_seqs, const int64_t *cu_seqlens, int H, int N,
                    const float *r, const float *w, const float *k,
                    const float *v, const float *kk, const float *a,
                    const double *s0, double *o, double *s_final, int nthreads)
{
    int b, t;
    oracle_job *jobs;
    pthread_t *threads;
    int rc = 0;

    if (num_seqs < 0 || H <= 0 || N <= 0 || !cu_seqlens || !o || !s_final)
        return -1;
    if (cu_seqlens[0] != 0)
        return -1;
    for (b = 0; b < num_seqs; ++b)
        if (cu_seqlens[b + 1] < cu_seqlens[b])
            return -1;
    if (cu_seqlens[num_seqs] > 0 && (!r || !w || !k || !v || !kk || !a))
        return -1;
    if (nthreads <= 0)
        nthreads = 1;
    if ((int64_t)nthreads > (int64_t)num_seqs * H)
        nthreads = (int)((int64_t)num_seqs * H);
    if (nthreads < 1)
        return 0;

    jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    threads = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !threads) {
        free(jobs);
        free(threads);
        return -2;
    }
    for (t = 0; t < nthreads; ++t) {
        oracle_job *j = &jobs[t];
        j->num_seqs = num_seqs; j->H = H; j->N = N;
        j->nthreads = nthreads; j->tid = t;
        j->cu = cu_seqlens;
        j->r = r; j->w = w; j->k = k; j->v = v; j->kk = kk; j->a = a;
        j->s0 = s0; j->o = o; j->s_final = s_final;
    }
    if (nthreads == 1) {
        oracle_worker(&jobs[0]);
    } else {
        int started = 0;
        for (t = 0; t < nthreads; ++t) {
            if (pthread_create(&threads[t], NULL, oracle_worker, &jobs[t]) != 0)
                break;
            ++started;
        }
        for (t = 0; t < started; ++t)
            pthread_join(threads[t], NULL);
        if (started != nthreads)
            rc = -2;
    }
    for (t = 0; t < nthreads; ++t)
        if (jobs[t].failed)
            rc = -2;
    free(jobs);
    free(threads);
    return rc;
}

/*
 * wkv7_oracle_tail -- the tail of the time-mix block that follows WKV, in
 * double, one (row, head) at a time.  The SwiftRWKV inference page names its
 * parts ("the tail of tmix (group norm, bonus, gate)", in "What the decode
 * path is made of" and in the fp32-stream prefill notes) and the RWKV-X page
 * lists the per-head bonus weight r_k ([n_head, head_size]).  Written out
 * (readings where the pages give no formula, also in the design notes: the
 * group is one head's N channels, the variance is the mean squared deviation,
 * eps is an argument, ln_w and ln_b are per channel of each head, the bonus
 * is added after the norm's affine part and the gate multiplies the sum):
 *
 *     mu  = (1/N) sum_j o_j ,   var = (1/N) sum_j (o_j - mu)^2
 *     y_j = ( (o_j - mu) / sqrt(var + eps) * ln_w_j + ln_b_j
 *             + (sum_i r_i k_i rk_i) v_j ) * g_j
 *
 *   n_rows          : rows (tokens of a packed prefill, or B for a decode step)
 *   o               : double [n_rows, H, N]   the WKV outputs
 *   r, k, v, g      : float  [n_rows, H, N]
 *   rk, ln_w, ln_b  : float  [H, N]           per-layer parameters
 *   eps             : the norm's epsilon (>= 0)
 *   y               : double [n_rows, H, N]   (written)
 * Returns 0, or -1 on a malformed argument.
 */
int wkv7_oracle_tail(int64_t n_rows, int H, int N, const double *o, const float *r, const float *k,
                     const float *v, const float *rk, const float *ln_w, const float *ln_b,
                     const float *g, double eps, double *y)
{
    int64_t row;
    int h, i, j;

    if (n_rows < 0 || H <= 0 || N <= 0 || eps < 0.0)
        return -1;
    if (n_rows > 0 && (!o || !r || !k || !v || !rk || !ln_w || !ln_b || !g || !y))
        return -1;
    for (row = 0; row < n_rows; ++row) {
        for (h = 0; h < H; ++h) {
            const size_t base = ((size_t)row * (size_t)H + (size_t)h) * (size_t)N;
            const size_t pbase = (size_t)h * (size_t)N;
            double mu = 0.0, var = 0.0, bonus = 0.0, inv;
            for (j = 0; j < N; ++j)
                mu += o[base + j];
            mu /= (double)N;
            for (j = 0; j < N; ++j)
                var += (o[base + j] - mu) * (o[base + j] - mu);
            var /= (double)N;
            inv = 1.0 / sqrt(var + eps);
            for (i = 0; i < N; ++i)
                bonus += (double)r[base + i] * (double)k[base + i] * (double)rk[pbase + i];
            for (j = 0; j < N; ++j) {
                const double normed = (o[base + j] - mu) * inv * (double)ln_w[pbase + j] + (double)ln_b[pbase + j];
                y[base + j] = (normed + bonus * (double)v[base + j]) * (double)g[base + j];
            }
        }
    }
    return 0;
}

/*
 * wkv7_oracle_backward -- the reverse-mode derivative of wkv7_oracle_run, in
 * double, one token at a time.
 *
 * It differentiates the same per-head recurrence (Core AI model zoo,
 * "Recurrent / linear-attention LLMs on Core AI", section 1) for the scalar
 * loss  L = sum_t do_t . o_t + sum dS_final .* S_final  and returns dL with
 * respect to every input.  Written as the chain rule taken backwards through
 * each token's three statements (no identities, no chunking), with
 * G = dL/dS for the state after the token being undone, c = kk .* a and
 * z = kk^T S_old from the forward pass:
 *
 *     G    += r do^T                              (the read-out o = S^T r)
 *     dr    = S_new do
 *     dv    = G^T k ,          dk = G v
 *     dw_i  = exp(w_i) sum_j G[i][j] S_old[i][j]
 *     dc    = -G z ,           u  = G^T c
 *     dkk   = -S_old u + a .* dc ,   da = kk .* dc
 *     G     = diag(exp w) G - kk u^T              (dL/dS_old)
 *
 * and dL/dS_initial is G after the first token.  The forward states of the
 * pair are kept (len + 1 matrices) so that S_old and S_new are exact.
 *
 *   cu_seqlens, r .. a, s0 : as for wkv7_oracle_run
 *   d_o      : double [T_total, H, N]             upstream gradient of o
 *   d_sfinal : double [num_seqs, H, N, N] or NULL upstream gradient of S_final
 *   dr, dw, dk, dv, dkk, da : double [T_total, H, N]  (written)
 *   d_s0     : double [num_seqs, H, N, N] or NULL    (written when given)
 * Returns 0, -1 on a malformed argument, -2 if memory or threads fail.
 */
typedef struct {
    int num_seqs, H, N, nthreads, tid;
    const int64_t *cu;
    const float *r, *w, *k, *v, *kk, *a;
    const double *s0, *d_o, *d_sf;
    double *dr, *dw, *dk, *dv, *dkk, *da, *d_s0;
    int failed;
} oracle_bwd_job;

static void oracle_pair_backward(const oracle_bwd_job *job, int b, int h, double *hist, double *zs,
                                 double *G, double *u, double *dc)
{
    const int H = job->H, N = job->N;
    const size_t NN = (size_t)N * (size_t)N;
    const size_t slot = (size_t)b * (size_t)H + (size_t)h;
    const int64_t t0 = job->cu[b], t1 = job->cu[b + 1];
    int64_t t;
    int i, j;

    /* forward: hist[s] is the state before local token s; hist[len] the final state */
    if (job->s0)
        memcpy(hist, job->s0 + slot * NN, sizeof(double) * NN);
    else
        memset(hist, 0, sizeof(double) * NN);
    for (t = t0; t < t1; ++t) {
        const size_t base = ((size_t)t * (size_t)H + (size_t)h) * (size_t)N;
        const double *S = hist + (size_t)(t - t0) * NN;
        double *Sn = hist + (size_t)(t - t0 + 1) * NN;
        double *z = zs + (size_t)(t - t0) * (size_t)N;
        for (j = 0; j < N; ++j) {
            double acc = 0.0;
            for (i = 0; i < N; ++i)
                acc += (double)job->kk[base + i] * S[(size_t)i * N + j];
            z[j] = acc;
        }
        for (i = 0; i < N; ++i) {
            const double decay = exp((double)job->w[base + i]);
            const double c = (double)job->kk[base + i] * (double)job->a[base + i];
            for (j = 0; j < N; ++j)
                Sn[(size_t)i * N + j] = decay * S[(size_t)i * N + j] - c * z[j]
                                        + (double)job->k[base + i] * (double)job->v[base + j];
        }
    }

    /* backward */
    if (job->d_sf)
        memcpy(G, job->d_sf + slot * NN, sizeof(double) * NN);
    else
        memset(G, 0, sizeof(double) * NN);
    for (t = t1 - 1; t >= t0; --t) {
        const size_t base = ((size_t)t * (size_t)H + (size_t)h) * (size_t)N;
        const double *S_old = hist + (size_t)(t - t0) * NN;
        const double *S_new = hist + (size_t)(t - t0 + 1) * NN;
        const double *z = zs + (size_t)(t - t0) * (size_t)N;
        const double *dot = job->d_o + base;

        for (i = 0; i < N; ++i)
            for (j = 0; j < N; ++j)
                G[(size_t)i * N + j] += (double)job->r[base + i] * dot[j];
        for (i = 0; i < N; ++i) {
            double acc_r = 0.0, acc_k = 0.0, acc_d = 0.0, acc_c = 0.0;
            for (j = 0; j < N; ++j) {
                acc_r += S_new[(size_t)i * N + j] * dot[j];
                acc_k += G[(size_t)i * N + j] * (double)job->v[base + j];
                acc_d += G[(size_t)i * N + j] * S_old[(size_t)i * N + j];
                acc_c += G[(size_t)i * N + j] * z[j];
            }
            job->dr[base + i] = acc_r;
            job->dk[base + i] = acc_k;
            job->dw[base + i] = exp((double)job->w[base + i]) * acc_d;
            dc[i] = -acc_c;
        }
        for (j = 0; j < N; ++j) {
            double acc_v = 0.0, acc_u = 0.0;
            for (i = 0; i < N; ++i) {
                acc_v += G[(size_t)i * N + j] * (double)job->k[base + i];
                acc_u += G[(size_t)i * N + j] * (double)job->kk[base + i] * (double)job->a[base + i];
            }
            job->dv[base + j] = acc_v;
            u[j] = acc_u;
        }
        for (i = 0; i < N; ++i) {
            double acc = 0.0;
            for (j = 0; j < N; ++j)
                acc += S_old[(size_t)i * N + j] * u[j];
            job->dkk[base + i] = -acc + (double)job->a[base + i] * dc[i];
            job->da[base + i] = (double)job->kk[base + i] * dc[i];
        }
        for (i = 0; i < N; ++i) {
            const double decay = exp((double)job->w[base + i]);
            for (j = 0; j < N; ++j)
                G[(size_t)i * N + j] = decay * G[(size_t)i * N + j] - (double)job->kk[base + i] * u[j];
        }
    }
    if (job->d_s0)
        memcpy(job->d_s0 + slot * NN, G, sizeof(double) * NN);
}

static void *oracle_bwd_worker(void *arg)
{
    oracle_bwd_job *job = (oracle_bwd_job *)arg;
    const size_t N = (size_t)job->N, NN = N * N;
    const int64_t pairs = (int64_t)job->num_seqs * job->H;
    int64_t p, max_len = 0;
    int b;
    double *hist, *zs, *G, *u, *dc;
    for (b = 0; b < job->num_seqs; ++b)
        if (job->cu[b + 1] - job->cu[b] > max_len)
            max_len = job->cu[b + 1] - job->cu[b];
    hist = (double *)malloc(sizeof(double) * NN * (size_t)(max_len + 1));
    zs = (double *)malloc(sizeof(double) * N * (size_t)(max_len + 1));
    G = (double *)malloc(sizeof(double) * NN);
    u = (double *)malloc(sizeof(double) * N);
    dc = (double *)malloc(sizeof(double) * N);
    if (!hist || !zs || !G || !u || !dc) {
        job->failed = 1;
    } else {
        for (p = job->tid; p < pairs; p += job->nthreads)
            oracle_pair_backward(job, (int)(p / job->H), (int)(p % job->H), hist, zs, G, u, dc);
    }
    free(hist);
    free(zs);
    free(G);
    free(u);
    free(dc);
    return NULL;
}

int wkv7_oracle_backward(int num_seqs, const int64_t *cu_seqlens, int H, int N,
                         const float *r, const float *w, const float *k,
                         const float *v, const float *kk, const float *a,
                         const double *s0, const double *d_o, const double *d_sfinal,
                         double *dr, double *dw, double *dk, double *dv, double *dkk, double *da,
                         double *d_s0, int nthreads)
{
    int b, t;
    oracle_bwd_job *jobs;
    pthread_t *threads;
    int rc = 0;

    if (num_seqs < 0 || H <= 0 || N <= 0 || !cu_seqlens)
        return -1;
    if (cu_seqlens[0] != 0)
        return -1;
    for (b = 0; b < num_seqs; ++b)
        if (cu_seqlens[b + 1] < cu_seqlens[b])
            return -1;
    if (cu_seqlens[num_seqs] > 0 &&
        (!r || !w || !k || !v || !kk || !a || !d_o || !dr || !dw || !dk || !dv || !dkk || !da))
        return -1;
    if (nthreads <= 0)
        nthreads = 1;
    if ((int64_t)nthreads > (int64_t)num_seqs * H)
        nthreads = (int)((int64_t)num_seqs * H);
    if (nthreads < 1)
        return 0;

    jobs = (oracle_bwd_job *)calloc((size_t)nthreads, sizeof(oracle_bwd_job));
    threads = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !threads) {
        free(jobs);
        free(threads);
        return -2;
    }
    for (t = 0; t < nthreads; ++t) {
        oracle_bwd_job *j = &jobs[t];
        j->num_seqs = num_seqs; j->H = H; j->N = N;
        j->nthreads = nthreads; j->tid = t;
        j->cu = cu_seqlens;
        j->r = r; j->w = w; j->k = k; j->v = v; j->kk = kk; j->a = a;
        j->s0 = s0; j->d_o = d_o; j->d_sf = d_sfinal;
        j->dr = dr; j->dw = dw; j->dk = dk; j->dv = dv; j->dkk = dkk; j->da = da; j->d_s0 = d_s0;
    }
    if (nthreads == 1) {
        oracle_bwd_worker(&jobs[0]);
    } else {
        int started = 0;
        for (t = 0; t < nthreads; ++t) {
            if (pthread_create(&threads[t], NULL, oracle_bwd_worker, &jobs[t]) != 0)
                break;
            ++started;
        }
        for (t = 0; t < started; ++t)
            pthread_join(threads[t], NULL);
        if (started != nthreads)
            rc = -2;
    }
    for (t = 0; t < nthreads; ++t)
        if (jobs[t].failed)
            rc = -2;
    free(jobs);
    free(threads);
    return rc;
}
