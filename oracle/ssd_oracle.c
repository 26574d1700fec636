/*
 * ssd_oracle.c -- plain, slow, fp64 CPU oracle for the Mamba-2 SSD layer forward
 * and, at the end of the file, its backward (gradients of a scalar loss).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA library is
 * checked against; it is used by the tests, by the smoke check and by the
 * timed CPU baseline of the benchmark, and by nothing else.  It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * calls it.
 *
 * What it computes (every function below, all arithmetic in fp64 on the exact
 * input values; bf16 inputs are widened exactly):
 *
 *   per head h (group g = h / (nheads/ngroups)), per headdim row p:
 *     s_{-1}[n] = init_state[b,h,p,n]            (0 when no init state)
 *     s_t[n]    = exp(dt_t*A_h) * s_{t-1}[n] + dt_t * x_t[p] * B_t[n]
 *     y_t[p]    = sum_n C_t[n] * s_t[n] + D_h * x_t[p]
 *     final_state[b,h,p,:] = s_{L-1}
 *
 * Sources:
 *   - "Mamba模型：线性复杂度序列建模的革命性突破" §2.2 and "Mamba 模型"
 *     §2.3.1 (discrete recurrent form h_t = Abar h_{t-1} + Bbar x_t, y = C h),
 *     with the discretisation fixed as Abar = exp(dt*A) (scalar A per head)
 *     and Bbar = dt*B (the simplified input scaling used by the SSD layer);
 *   - "深挖-Mamba", core concepts §1 (the observation equation keeps the
 *     feed-through term D x);
 *   - "Mamba 模型" §3.3 and "深挖-Mamba" §3 (B_t, C_t, dt_t vary per token);
 *   - "Mamba 模型" §4.1 (the semiseparable matrix form M, y = M x, used by
 *     oracle_ssd_quadratic);
 *   - "Mamba 模型" §3.4 (parallel associative scan, used by
 *     oracle_ssd_assoc_scan as an independent evaluation order).
 *
 * oracle_ssd_recurrence_pre adds the per-(token, head) pre-step of the scalar
 * inputs, from the same discretisation ("Mamba模型：线性复杂度序列建模的革命性突破"
 * §2.2 and "Mamba 模型" §2.3.1: zero-order hold Bbar = (dt A)^-1 (exp(dt A) - 1)
 * dt B; §3.2 of the first page: dt through a softplus):
 *     d_t   = dt_t + dt_bias[h]        (dt_bias may be NULL => 0)
 *     d_t   = log(1 + exp(d_t))        if ORACLE_PRE_SOFTPLUS
 *     s_t   = exp(d_t A) s_{t-1} + u_t x_t B_t
 *     u_t   = (exp(d_t A) - 1) / A     if ORACLE_PRE_ZOH (d_t when A = 0), else d_t
 *
 * Layouts (row-major, the same as the CUDA library's public ABI):
 *   x, y   [batch][seqlen][nheads][headdim]
 *   dt     [batch][seqlen][nheads]           fp32
 *   A, D   [nheads]                          fp32 (D may be NULL => 0)
 *   B, C   [batch][seqlen][ngroups][dstate]
 *   init   [batch][nheads][headdim][dstate]  fp32 (may be NULL => 0)
 * Outputs are fp64 and indexed by "row" r = (b*nheads + h)*headdim + p:
 *   y_rows     [nrows][seqlen]
 *   final_rows [nrows][dstate]
 * x, B and C are fp32 (in_dtype 0) or bf16 bit patterns (in_dtype 1).
 *
 * Return value: 0 on success, -1 on a bad argument, -2 when out of memory.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_IN_F32 0
#define ORACLE_IN_BF16 1
#define ORACLE_PRE_SOFTPLUS 1
#define ORACLE_PRE_ZOH 2

typedef struct {
    const void *x;
    const float *dt, *A;
    const void *B, *C;
    const float *D, *init;
    int in_dtype;
    long batch, seqlen, nheads, headdim, ngroups, dstate;
    const float *dt_bias;  /* pre-step (oracle_ssd_recurrence_pre only) */
    int pre_flags;
} oracle_problem;

/* Widen one stored input element to fp64 (exact for both fp32 and bf16). */
static double widen(const void *base, long i, int in_dtype)
{
    if (in_dtype == ORACLE_IN_F32)
        return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int check_problem(const oracle_problem *pr)
{
    if (!pr->x || !pr->dt || !pr->A || !pr->B || !pr->C)
        return -1;
    if (pr->batch <= 0 || pr->seqlen <= 0 || pr->nheads <= 0 || pr->headdim <= 0 ||
        pr->ngroups <= 0 || pr->dstate <= 0)
        return -1;
    if (pr->nheads % pr->ngroups != 0)
        return -1;
    if (pr->in_dtype != ORACLE_IN_F32 && pr->in_dtype != ORACLE_IN_BF16)
        return -1;
    return 0;
}

/* Decompose a row id into (batch, head, headdim index) and the head's group. */
static void row_coords(const oracle_problem *pr, long r, long *b, long *h, long *p, long *g)
{
    *p = r % pr->headdim;
    *h = (r / pr->headdim) % pr->nheads;
    *b = r / (pr->headdim * pr->nheads);
    *g = *h / (pr->nheads / pr->ngroups);
}

/* ------------------------------------------------------------------------ */
/* O1: the sequential recurrence, one row (b, h, p) at a time.              */
/* ------------------------------------------------------------------------ */

static void recurrence_row(const oracle_problem *pr, long r, double *s, double *y_row, double *final_row)
{
    long b, h, p, g;
    row_coords(pr, r, &b, &h, &p, &g);
    const long L = pr->seqlen, H = pr->nheads, P = pr->headdim, G = pr->ngroups, N = pr->dstate;
    const double A_h = (double)pr->A[h];
    const double D_h = pr->D ? (double)pr->D[h] : 0.0;

    for (long n = 0; n < N; ++n)
        s[n] = pr->init ? (double)pr->init[((b * H + h) * P + p) * N + n] : 0.0;

    for (long t = 0; t < L; ++t) {
        const double dt_t = (double)pr->dt[(b * L + t) * H + h];
        const double decay = exp(dt_t * A_h);
        const double x_t = widen(pr->x, ((b * L + t) * H + h) * P + p, pr->in_dtype);
        const long bc = ((b * L + t) * G + g) * N;
        double acc = 0.0;
        for (long n = 0; n < N; ++n) {
            s[n] = decay * s[n] + dt_t * x_t * widen(pr->B, bc + n, pr->in_dtype);
            acc += widen(pr->C, bc + n, pr->in_dtype) * s[n];
        }
        if (y_row)
            y_row[t] = acc + D_h * x_t;
    }
    if (final_row)
        for (long n = 0; n < N; ++n)
            final_row[n] = s[n];
}

/* The same recurrence with the pre-step of the scalar inputs (see the header). */
static void recurrence_row_pre(const oracle_problem *pr, long r, double *s, double *y_row, double *final_row)
{
    long b, h, p, g;
    row_coords(pr, r, &b, &h, &p, &g);
    const long L = pr->seqlen, H = pr->nheads, P = pr->headdim, G = pr->ngroups, N = pr->dstate;
    const double A_h = (double)pr->A[h];
    const double D_h = pr->D ? (double)pr->D[h] : 0.0;
    const double bias = pr->dt_bias ? (double)pr->dt_bias[h] : 0.0;

    for (long n = 0; n < N; ++n)
        s[n] = pr->init ? (double)pr->init[(((b * H + h) * P + p) * N) + n] : 0.0;

    for (long t = 0; t < L; ++t) {
        double d = (double)pr->dt[(b * L + t) * H + h] + bias;
        if (pr->pre_flags & ORACLE_PRE_SOFTPLUS)
            d = log(1.0 + exp(d));
        const double decay = exp(d * A_h);
        const double u = (pr->pre_flags & ORACLE_PRE_ZOH) ? (A_h != 0.0 ? (decay - 1.0) / A_h : d) : d;
        const double x_t = widen(pr->x, (b * L + t) * H * P + h * P + p, pr->in_dtype);
        const long bc = ((b * L + t) * G + g) * N;
        double acc = 0.0;
        for (long n = 0; n < N; ++n) {
            s[n] = decay * s[n] + u * x_t * widen(pr->B, bc + n, pr->in_dtype);
            acc += widen(pr->C, bc + n, pr->in_dtype) * s[n];
        }
        if (y_row)
            y_row[t] = D_h * x_t + acc;
    }
    if (final_row)
        for (long n = 0; n < N; ++n)
            final_row[n] = s[n];  /* the state after the last token */
}

typedef struct {
    const oracle_problem *pr;
    const long *rows;
    long nrows;
    double *y_rows, *final_rows;
    long next;      /* shared work counter, advanced atomically */
    int failed;
} recurrence_job;

static void *recurrence_worker(void *arg)
{
    recurrence_job *job = (recurrence_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)job->pr->dstate);
    if (!s) {
        __atomic_store_n(&job->failed, 1, __ATOMIC_RELAXED);
        return NULL;
    }
    for (;;) {
        long i = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (i >= job->nrows)
            break;
        long r = job->rows ? job->rows[i] : i;
        (job->pr->dt_bias || job->pr->pre_flags ? recurrence_row_pre : recurrence_row)(job->pr, r, s,
                       job->y_rows ? job->y_rows + i * job->pr->seqlen : NULL,
                       job->final_rows ? job->final_rows + i * job->pr->dstate : NULL);
    }
    free(s);
    return NULL;
}

/*
 * Sequential fp64 recurrence for the rows listed in `rows` (all rows, in
 * order, when rows == NULL), threaded over rows with `nthreads` workers.
 */
static int run_recurrence(const oracle_problem *prp, const long *rows, long nrows, double *y_rows,
                          double *final_rows, int nthreads);

int oracle_ssd_recurrence(const void *x, const float *dt, const float *A, const void *B, const void *C,
                          const float *D, const float *init_state, int in_dtype, long batch, long seqlen,
                          long nheads, long headdim, long ngroups, long dstate, const long *rows, long nrows,
                          double *y_rows, double *final_rows, int nthreads)
{
    oracle_problem pr = {x, dt, A, B, C, D, init_state, in_dtype, batch, seqlen, nheads, headdim, ngroups, dstate,
                         NULL, 0};
    return run_recurrence(&pr, rows, nrows, y_rows, final_rows, nthreads);
}

/* The recurrence with the pre-step of dt (flags ORACLE_PRE_SOFTPLUS, ORACLE_PRE_ZOH). */
int oracle_ssd_recurrence_pre(const void *x, const float *dt, const float *dt_bias, int pre_flags, const float *A,
                              const void *B, const void *C, const float *D, const float *init_state, int in_dtype,
                              long batch, long seqlen, long nheads, long headdim, long ngroups, long dstate,
                              const long *rows, long nrows, double *y_rows, double *final_rows, int nthreads)
{
    if (pre_flags & ~(ORACLE_PRE_SOFTPLUS | ORACLE_PRE_ZOH))
        return -1;
    oracle_problem pr = {x, dt, A, B, C, D, init_state, in_dtype, batch, seqlen, nheads, headdim, ngroups, dstate,
                         dt_bias, pre_flags};
    return run_recurrence(&pr, rows, nrows, y_rows, final_rows, nthreads);
}

static int run_recurrence(const oracle_problem *prp, const long *rows, long nrows, double *y_rows,
                          double *final_rows, int nthreads)
{
    const oracle_problem pr = *prp;
    const long batch = pr.batch, nheads = pr.nheads, headdim = pr.headdim;
    if (check_problem(&pr))
        return -1;
    const long total = batch * nheads * headdim;
    if (!rows)
        nrows = total;
    if (nrows < 0)
        return -1;
    if (rows)
        for (long i = 0; i < nrows; ++i)
            if (rows[i] < 0 || rows[i] >= total)
                return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 1024)
        nthreads = 1024;

    recurrence_job job = {&pr, rows, nrows, y_rows, final_rows, 0, 0};
    if (nthreads == 1) {
        recurrence_worker(&job);
    } else {
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        if (!tid)
            return -2;
        int started = 0;
        for (int i = 0; i < nthreads; ++i) {
            if (pthread_create(&tid[i], NULL, recurrence_worker, &job) != 0)
                break;
            ++started;
        }
        if (started == 0)
            recurrence_worker(&job);
        for (int i = 0; i < started; ++i)
            pthread_join(tid[i], NULL);
        free(tid);
    }
    return job.failed ? -2 : 0;
}

/* ------------------------------------------------------------------------ */
/* O2: the quadratic (semiseparable matrix) form, all rows, tiny inputs.     */
/* ------------------------------------------------------------------------ */

/*
 * y_i = sum_{j<=i} M_ij * dt_j * x_j + D x_i + exp(A * sum_{k=0..i} dt_k) * (C_i . h0)
 * with M_ij = (C_i . B_j) * exp(A * sum_{k=j+1..i} dt_k)        ("Mamba 模型" §4.1)
 * final[n] = sum_j exp(A * sum_{k=j+1..L-1} dt_k) dt_j x_j B_j[n]
 *            + exp(A * sum_{k=0..L-1} dt_k) h0[n]
 * Every decay exponent is summed afresh from dt for each (i, j): no running
 * state is carried from one token to the next.
 */
int oracle_ssd_quadratic(const void *x, const float *dt, const float *A, const void *B, const void *C,
                         const float *D, const float *init_state, int in_dtype, long batch, long seqlen,
                         long nheads, long headdim, long ngroups, long dstate, double *y_rows,
                         double *final_rows)
{
    oracle_problem pr = {x, dt, A, B, C, D, init_state, in_dtype, batch, seqlen, nheads, headdim, ngroups, dstate,
                         NULL, 0};
    if (check_problem(&pr))
        return -1;
    const long L = seqlen, H = nheads, P = headdim, G = ngroups, N = dstate;
    for (long b = 0; b < batch; ++b)
        for (long h = 0; h < H; ++h) {
            const long g = h / (H / G);
            const double A_h = (double)A[h];
            const double D_h = D ? (double)D[h] : 0.0;
            for (long p = 0; p < P; ++p) {
                const long r = (b * H + h) * P + p;
                for (long i = 0; i < L; ++i) {
                    const long ci = ((b * L + i) * G + g) * N;
                    double y = 0.0;
                    for (long j = 0; j <= i; ++j) {
                        const long bj = ((b * L + j) * G + g) * N;
                        double cb = 0.0;
                        for (long n = 0; n < N; ++n)
                            cb += widen(C, ci + n, in_dtype) * widen(B, bj + n, in_dtype);
                        double seg = 0.0;
                        for (long k = j + 1; k <= i; ++k)
                            seg += (double)dt[(b * L + k) * H + h];
                        const double dt_j = (double)dt[(b * L + j) * H + h];
                        const double x_j = widen(x, ((b * L + j) * H + h) * P + p, in_dtype);
                        y += cb * exp(A_h * seg) * dt_j * x_j;
                    }
                    if (init_state) {
                        double seg = 0.0;
                        for (long k = 0; k <= i; ++k)
                            seg += (double)dt[(b * L + k) * H + h];
                        double ch = 0.0;
                        for (long n = 0; n < N; ++n)
                            ch += widen(C, ci + n, in_dtype) * (double)init_state[r * N + n];
                        y += exp(A_h * seg) * ch;
                    }
                    y += D_h * widen(x, ((b * L + i) * H + h) * P + p, in_dtype);
                    if (y_rows)
                        y_rows[r * L + i] = y;
                }
                if (final_rows)
                    for (long n = 0; n < N; ++n) {
                        double f = 0.0;
                        for (long j = 0; j < L; ++j) {
                            double seg = 0.0;
                            for (long k = j + 1; k < L; ++k)
                                seg += (double)dt[(b * L + k) * H + h];
                            const double dt_j = (double)dt[(b * L + j) * H + h];
                            f += exp(A_h * seg) * dt_j * widen(x, ((b * L + j) * H + h) * P + p, in_dtype) *
                                 widen(B, ((b * L + j) * G + g) * N + n, in_dtype);
                        }
                        if (init_state) {
                            double seg = 0.0;
                            for (long k = 0; k < L; ++k)
                                seg += (double)dt[(b * L + k) * H + h];
                            f += exp(A_h * seg) * (double)init_state[r * N + n];
                        }
                        final_rows[r * N + n] = f;
                    }
            }
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O3: work-efficient (Blelloch) associative scan over (decay, input) pairs. */
/* ------------------------------------------------------------------------ */

/*
 * Element t is the affine map s -> a_t*s + u_t with a_t = exp(dt_t A),
 * u_t = dt_t x_t B_t.  Composition (first e1, then e2):
 *     (a1, u1) then (a2, u2) = (a1*a2, a2*u1 + u2)
 * which is associative ("Mamba 模型" §3.4).  The init state enters as a
 * leading element (0, h0).  An up-sweep/down-sweep over a power-of-two array
 * yields the exclusive prefix of every position; applying element t to it
 * gives s_t.  The order of the fp64 operations differs from O1's.
 */
int oracle_ssd_assoc_scan(const void *x, const float *dt, const float *A, const void *B, const void *C,
                          const float *D, const float *init_state, int in_dtype, long batch, long seqlen,
                          long nheads, long headdim, long ngroups, long dstate, double *y_rows,
                          double *final_rows)
{
    oracle_problem pr = {x, dt, A, B, C, D, init_state, in_dtype, batch, seqlen, nheads, headdim, ngroups, dstate,
                         NULL, 0};
    if (check_problem(&pr))
        return -1;
    const long L = seqlen, H = nheads, P = headdim, G = ngroups, N = dstate;
    long n_el = L + 1; /* the leading element carries the init state */
    long len = 1;
    while (len < n_el)
        len <<= 1;
    double *a = (double *)malloc(sizeof(double) * (size_t)len);
    double *u = (double *)malloc(sizeof(double) * (size_t)(len * N));
    double *tmp = (double *)malloc(sizeof(double) * (size_t)N);
    if (!a || !u || !tmp) {
        free(a);
        free(u);
        free(tmp);
        return -2;
    }
    for (long b = 0; b < batch; ++b)
        for (long h = 0; h < H; ++h) {
            const long g = h / (H / G);
            const double A_h = (double)A[h];
            const double D_h = D ? (double)D[h] : 0.0;
            for (long p = 0; p < P; ++p) {
                const long r = (b * H + h) * P + p;
                /* leaves: identity padding is (1, 0) */
                for (long i = 0; i < len; ++i) {
                    a[i] = 1.0;
                    for (long n = 0; n < N; ++n)
                        u[i * N + n] = 0.0;
                }
                a[0] = 0.0;
                for (long n = 0; n < N; ++n)
                    u[n] = init_state ? (double)init_state[r * N + n] : 0.0;
                for (long t = 0; t < L; ++t) {
                    const double dt_t = (double)dt[(b * L + t) * H + h];
                    const double x_t = widen(x, ((b * L + t) * H + h) * P + p, in_dtype);
                    a[t + 1] = exp(dt_t * A_h);
                    for (long n = 0; n < N; ++n)
                        u[(t + 1) * N + n] = dt_t * x_t * widen(B, ((b * L + t) * G + g) * N + n, in_dtype);
                }
                /* up-sweep: node i+2d-1 absorbs node i+d-1 (left then right) */
                for (long d = 1; d < len; d <<= 1)
                    for (long i = 0; i < len; i += 2 * d) {
                        const long lft = i + d - 1, rgt = i + 2 * d - 1;
                        for (long n = 0; n < N; ++n)
                            u[rgt * N + n] = a[rgt] * u[lft * N + n] + u[rgt * N + n];
                        a[rgt] = a[lft] * a[rgt];
                    }
                /* down-sweep: turns the tree into exclusive prefixes */
                a[len - 1] = 1.0;
                for (long n = 0; n < N; ++n)
                    u[(len - 1) * N + n] = 0.0;
                for (long d = len >> 1; d >= 1; d >>= 1)
                    for (long i = 0; i < len; i += 2 * d) {
                        const long lft = i + d - 1, rgt = i + 2 * d - 1;
                        /* new left = old right (prefix before this subtree);
                           new right = old right then old left */
                        const double a_l = a[lft], a_r = a[rgt];
                        for (long n = 0; n < N; ++n) {
                            tmp[n] = u[lft * N + n];
                            u[lft * N + n] = u[rgt * N + n];
                            u[rgt * N + n] = a_l * u[rgt * N + n] + tmp[n];
                        }
                        a[lft] = a_r;
                        a[rgt] = a_r * a_l;
                    }
                /* position t+1 holds the composition of elements 0..t; apply
                   element t+1 to get s_t.  Only the u part matters: the
                   exclusive prefix applied to the zero vector. */
                for (long t = 0; t < L; ++t) {
                    const double dt_t = (double)dt[(b * L + t) * H + h];
                    const double x_t = widen(x, ((b * L + t) * H + h) * P + p, in_dtype);
                    const double a_t = exp(dt_t * A_h);
                    const long ci = ((b * L + t) * G + g) * N;
                    double acc = 0.0;
                    for (long n = 0; n < N; ++n) {
                        const double s_t = a_t * u[(t + 1) * N + n] + dt_t * x_t * widen(B, ci + n, in_dtype);
                        acc += widen(C, ci + n, in_dtype) * s_t;
                        if (t == L - 1 && final_rows)
                            final_rows[r * N + n] = s_t;
                    }
                    if (y_rows)
                        y_rows[r * L + t] = acc + D_h * x_t;
                }
            }
        }
    free(a);
    free(u);
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward: gradients of a scalar loss through the recurrence.             */
/* ------------------------------------------------------------------------ */

/*
 * The loss is  sum_{b,t,h,p} dy[b,t,h,p] y[b,t,h,p] + sum dfinal * final_state
 * (dy and dfinal are the incoming gradients; dfinal may be NULL => 0), and the
 * gradients follow the recurrence above by the chain rule, in reverse time
 * ("Mamba 模型" §3.4: the backward pass recomputes the intermediate states
 * instead of reading stored ones; here each row's states are recomputed by a
 * forward sweep and kept for its reverse sweep).  Per row (b, h, p), with
 * a_t = exp(dt_t A_h) and lam_t = dLoss/ds_t (the whole vector over n):
 *     lam_{L-1} = dy_{L-1}[p] C_{L-1} + dfinal[b,h,p,:]
 *     lam_t     = dy_t[p] C_t + a_{t+1} lam_{t+1}
 *     dC_t[n]  += dy_t[p] s_t[n]
 *     dB_t[n]  += dt_t x_t[p] lam_t[n]
 *     dx_t[p]   = D_h dy_t[p] + dt_t (B_t . lam_t)
 *     ddt_t    += x_t[p] (B_t . lam_t) + A_h a_t (lam_t . s_{t-1})
 *     dA_h     += dt_t a_t (lam_t . s_{t-1})
 *     dD_h     += dy_t[p] x_t[p]
 *     dinit[b,h,p,:] = a_0 lam_0
 * (dB, dC sum over the heads of the group and over p; ddt over p; dA, dD over
 * b, t and p.)  dy is given in fp64 (the exact values the caller's dtype
 * holds).  Outputs are fp64, all with the layouts of the forward inputs:
 * dx [b][L][H][P], ddt [b][L][H], dA [H], dB, dC [b][L][G][N], dD [H],
 * dinit [b][H][P][N].  Work is threaded over (batch, group) pairs, each worker
 * owning every output element it writes.
 */
typedef struct {
    const oracle_problem *pr;
    const double *dy, *dfinal;
    double *dx, *ddt, *dB, *dC, *dinit;
    double *dA_part, *dD_part;  /* [batch * ngroups][nheads] partial sums */
    long next, npairs;
    int failed;
} backward_job;

static void backward_pair(backward_job *job, long bg, double *s_all, double *lam)
{
    const oracle_problem *pr = job->pr;
    const long L = pr->seqlen, H = pr->nheads, P = pr->headdim, G = pr->ngroups, N = pr->dstate;
    const long b = bg / G, g = bg % G, hpg = H / G;
    for (long h = g * hpg; h < (g + 1) * hpg; ++h) {
        const double A_h = (double)pr->A[h];
        const double D_h = pr->D ? (double)pr->D[h] : 0.0;
        for (long p = 0; p < P; ++p) {
            /* forward sweep: s_all[(t+1)*N + n] = s_t[n], s_all[n] = s_{-1}[n] */
            for (long n = 0; n < N; ++n)
                s_all[n] = pr->init ? (double)pr->init[((b * H + h) * P + p) * N + n] : 0.0;
            for (long t = 0; t < L; ++t) {
                const long ti = (b * L + t) * H + h; /* (b, t, h) */
                const double dt_t = (double)pr->dt[ti];
                const double a_t = exp(dt_t * A_h);
                const double x_t = widen(pr->x, ti * P + p, pr->in_dtype);
                const long bc = ((b * L + t) * G + g) * N;
                for (long n = 0; n < N; ++n)
                    s_all[(t + 1) * N + n] = a_t * s_all[t * N + n] + dt_t * x_t * widen(pr->B, bc + n, pr->in_dtype);
            }
            /* reverse sweep */
            for (long n = 0; n < N; ++n)
                lam[n] = job->dfinal ? job->dfinal[((b * H + h) * P + p) * N + n] : 0.0;
            for (long t = L - 1; t >= 0; --t) {
                const long ti = (b * L + t) * H + h;
                const double dt_t = (double)pr->dt[ti];
                const double a_t = exp(dt_t * A_h);
                const long xi = ti * P + p;
                const double x_t = widen(pr->x, xi, pr->in_dtype);
                const double dy_t = job->dy[xi];
                const long bc = ((b * L + t) * G + g) * N;
                double b_lam = 0.0, lam_sprev = 0.0;
                for (long n = 0; n < N; ++n) {
                    lam[n] += dy_t * widen(pr->C, bc + n, pr->in_dtype);  /* lam_t */
                    const double B_n = widen(pr->B, bc + n, pr->in_dtype);
                    job->dC[bc + n] += dy_t * s_all[(t + 1) * N + n];
                    job->dB[bc + n] += dt_t * x_t * lam[n];
                    b_lam += B_n * lam[n];
                    lam_sprev += lam[n] * s_all[t * N + n];
                }
                job->dx[xi] = D_h * dy_t + dt_t * b_lam;
                job->ddt[ti] += x_t * b_lam + A_h * a_t * lam_sprev;
                job->dA_part[bg * H + h] += dt_t * a_t * lam_sprev;
                job->dD_part[bg * H + h] += dy_t * x_t;
                for (long n = 0; n < N; ++n)
                    lam[n] *= a_t;  /* a_t lam_t: the part of lam_{t-1} carried back */
            }
            if (job->dinit)
                for (long n = 0; n < N; ++n)
                    job->dinit[((b * H + h) * P + p) * N + n] = lam[n];
        }
    }
}

static void *backward_worker(void *arg)
{
    backward_job *job = (backward_job *)arg;
    const long L = job->pr->seqlen, N = job->pr->dstate;
    double *s_all = (double *)malloc(sizeof(double) * (size_t)((L + 1) * N));
    double *lam = (double *)malloc(sizeof(double) * (size_t)N);
    if (!s_all || !lam) {
        __atomic_store_n(&job->failed, 1, __ATOMIC_RELAXED);
        free(s_all);
        free(lam);
        return NULL;
    }
    for (;;) {
        long i = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (i >= job->npairs)
            break;
        backward_pair(job, i, s_all, lam);
    }
    free(s_all);
    free(lam);
    return NULL;
}

int oracle_ssd_backward(const void *x, const float *dt, const float *A, const void *B, const void *C,
                        const float *D, const float *init_state, int in_dtype, long batch, long seqlen,
                        long nheads, long headdim, long ngroups, long dstate, const double *dy,
                        const double *dfinal, double *dx, double *ddt, double *dA, double *dB, double *dC,
                        double *dD, double *dinit, int nthreads)
{
    oracle_problem pr = {x, dt, A, B, C, D, init_state, in_dtype, batch, seqlen, nheads, headdim, ngroups, dstate,
                         NULL, 0};
    if (check_problem(&pr) || !dy || !dx || !ddt || !dA || !dB || !dC || !dD)
        return -1;
    const long npairs = batch * ngroups;
    memset(ddt, 0, sizeof(double) * (size_t)(batch * seqlen * nheads));
    memset(dB, 0, sizeof(double) * (size_t)(batch * seqlen * ngroups * dstate));
    memset(dC, 0, sizeof(double) * (size_t)(batch * seqlen * ngroups * dstate));
    double *dA_part = (double *)calloc((size_t)(npairs * nheads), sizeof(double));
    double *dD_part = (double *)calloc((size_t)(npairs * nheads), sizeof(double));
    if (!dA_part || !dD_part) {
        free(dA_part);
        free(dD_part);
        return -2;
    }
    backward_job job = {&pr, dy, dfinal, dx, ddt, dB, dC, dinit, dA_part, dD_part, 0, npairs, 0};
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > npairs)
        nthreads = (int)npairs;
    if (nthreads == 1) {
        backward_worker(&job);
    } else {
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        int started = 0;
        if (tid)
            for (int i = 0; i < nthreads; ++i) {
                if (pthread_create(&tid[i], NULL, backward_worker, &job) != 0)
                    break;
                ++started;
            }
        if (started == 0)
            backward_worker(&job);
        for (int i = 0; i < started; ++i)
            pthread_join(tid[i], NULL);
        free(tid);
    }
    /* the per-pair partial sums, added in a fixed order */
    for (long h = 0; h < nheads; ++h) {
        double a = 0.0, d = 0.0;
        for (long i = 0; i < npairs; ++i) {
            a += dA_part[i * nheads + h];
            d += dD_part[i * nheads + h];
        }
        dA[h] = a;
        dD[h] = d;
    }
    free(dA_part);
    free(dD_part);
    return job.failed ? -2 : 0;
}
