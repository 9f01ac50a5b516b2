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
