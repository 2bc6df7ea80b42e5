/*
 * w4a16_oracle.c -- float64 CPU reference for the fp16 x int4 group-quantized GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. The product library never links it and
 * shares no code, header, table or helper with it.
 *
 * What it computes (the plain definition; "Validation" section of the MatMulNBits
 * Marlin pull request, github.com/justinchuby/onnx-genai pull 960, which checks the
 * GPU kernel against "an f64 dequant->GEMM oracle"):
 *
 *   q[n,k]    = nibble k of row n of Bq; byte k/2, low nibble for even k
 *   zpv[n,j]  = nibble j of row n of the packed zero points (low nibble = even j),
 *               or 8 when no zero points are given (symmetric)
 *   W[n,k]    = (q[n,k] - zpv[n, k/group]) * scale[n, k/group]
 *   Y[m,n]    = sum_k A[m,k] * W[n,k]                (k ascending, float64)
 *   SwiGLU:     Y[m,n] = silu(Yg[m,n]) * Yu[m,n],  silu(x) = x / (1 + exp(-x))
 *
 * Activations and scales arrive already widened to float64 (a lossless
 * conversion from float16/float32 done by the Python wrapper); the nibbles arrive
 * as the original packed bytes, never as a repacked layout.
 *
 * Plain loops, no blocking or reordering. Columns are spread over POSIX threads;
 * each output is still one dot product over k in ascending order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

/* Nibble idx of a packed row: byte idx/2, low nibble first. */
static int packed_nibble(const uint8_t *row, int idx)
{
    uint8_t b = row[idx / 2];
    return (idx % 2 == 0) ? (b & 0x0F) : (b >> 4);
}

/* One dequantised weight row W[n, 0..K-1]. */
static void dequant_row(const uint8_t *bq, const double *scales, const uint8_t *zp,
                        int K, int group, int n, double *w)
{
    int G = K / group;
    const uint8_t *qrow = bq + (size_t)n * (size_t)(K / 2);
    const double *srow = scales + (size_t)n * (size_t)G;
    const uint8_t *zrow = zp ? zp + (size_t)n * (size_t)((G + 1) / 2) : NULL;
    for (int k = 0; k < K; ++k) {
        int j = k / group;
        int q = packed_nibble(qrow, k);
        int z = zrow ? packed_nibble(zrow, j) : 8;
        w[k] = (double)(q - z) * srow[j];
    }
}

static int check_shape(int M, int N, int K, int group)
{
    if (M < 0 || N < 0 || K <= 0 || group <= 0) return 1;
    if (K % 2 != 0 || K % group != 0) return 2;
    return 0;
}

int oracle_dequant(const uint8_t *bq, const double *scales, const uint8_t *zp,
                   int N, int K, int group, double *W)
{
    int rc = check_shape(0, N, K, group);
    if (rc) return rc;
    for (int n = 0; n < N; ++n)
        dequant_row(bq, scales, zp, K, group, n, W + (size_t)n * (size_t)K);
    return 0;
}

typedef struct {
    const double *A;
    int M, K, N, group;
    const uint8_t *bq[2];
    const double *scales[2];
    const uint8_t *zp[2];
    int swiglu;
    const int32_t *rows;
    int n_rows;
    const int32_t *cols;
    int n_cols;
    double *Y;
    int col_begin, col_end;
    int status;
} job_t;

static double dot_k(const double *a, const double *w, int K)
{
    double acc = 0.0;
    for (int k = 0; k < K; ++k) acc += a[k] * w[k];
    return acc;
}

static double silu(double x) { return x / (1.0 + exp(-x)); }

static void *run_job(void *arg)
{
    job_t *jb = (job_t *)arg;
    int K = jb->K;
    double *wg = (double *)malloc(sizeof(double) * (size_t)K);
    double *wu = jb->swiglu ? (double *)malloc(sizeof(double) * (size_t)K) : NULL;
    if (!wg || (jb->swiglu && !wu)) {
        free(wg);
        free(wu);
        jb->status = 3;
        return NULL;
    }
    for (int c = jb->col_begin; c < jb->col_end; ++c) {
        int n = jb->cols ? jb->cols[c] : c;
        dequant_row(jb->bq[0], jb->scales[0], jb->zp[0], K, jb->group, n, wg);
        if (jb->swiglu) dequant_row(jb->bq[1], jb->scales[1], jb->zp[1], K, jb->group, n, wu);
        for (int r = 0; r < jb->n_rows; ++r) {
            int m = jb->rows ? jb->rows[r] : r;
            const double *a = jb->A + (size_t)m * (size_t)K;
            double y = dot_k(a, wg, K);
            if (jb->swiglu) y = silu(y) * dot_k(a, wu, K);
            jb->Y[(size_t)r * (size_t)jb->n_cols + (size_t)c] = y;
        }
    }
    free(wg);
    free(wu);
    jb->status = 0;
    return NULL;
}

static int run_threads(job_t proto, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > proto.n_cols) nthreads = proto.n_cols > 0 ? proto.n_cols : 1;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return 3;
    }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].col_begin = (int)((long long)proto.n_cols * t / nthreads);
        jobs[t].col_end = (int)((long long)proto.n_cols * (t + 1) / nthreads);
        jobs[t].status = 4;
    }
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&tid[t], NULL, run_job, &jobs[t]) != 0) jobs[t].status = 5;
    run_job(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (jobs[t].status != 5) pthread_join(tid[t], NULL);
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status) rc = jobs[t].status;
    free(jobs);
    free(tid);
    return rc;
}

/*
 * Y[r][c] = sum_k A[rows[r], k] * W[cols[c], k].
 * rows == NULL selects all M rows (n_rows must equal M); cols == NULL selects all N.
 */
int oracle_gemm(const double *A, int M, int K,
                const uint8_t *bq, const double *scales, const uint8_t *zp,
                int N, int group,
                const int32_t *rows, int n_rows, const int32_t *cols, int n_cols,
                double *Y, int nthreads)
{
    int rc = check_shape(M, N, K, group);
    if (rc) return rc;
    job_t jb = {0};
    jb.A = A; jb.M = M; jb.K = K; jb.N = N; jb.group = group;
    jb.bq[0] = bq; jb.scales[0] = scales; jb.zp[0] = zp;
    jb.swiglu = 0;
    jb.rows = rows; jb.n_rows = n_rows; jb.cols = cols; jb.n_cols = n_cols;
    jb.Y = Y;
    return run_threads(jb, nthreads);
}

/* Y[r][c] = silu(A W_gate^T)[rows[r], cols[c]] * (A W_up^T)[rows[r], cols[c]]. */
int oracle_gemm_swiglu(const double *A, int M, int K,
                       const uint8_t *bq_gate, const double *s_gate, const uint8_t *zp_gate,
                       const uint8_t *bq_up, const double *s_up, const uint8_t *zp_up,
                       int N, int group,
                       const int32_t *rows, int n_rows, const int32_t *cols, int n_cols,
                       double *Y, int nthreads)
{
    int rc = check_shape(M, N, K, group);
    if (rc) return rc;
    job_t jb = {0};
    jb.A = A; jb.M = M; jb.K = K; jb.N = N; jb.group = group;
    jb.bq[0] = bq_gate; jb.scales[0] = s_gate; jb.zp[0] = zp_gate;
    jb.bq[1] = bq_up; jb.scales[1] = s_up; jb.zp[1] = zp_up;
    jb.swiglu = 1;
    jb.rows = rows; jb.n_rows = n_rows; jb.cols = cols; jb.n_cols = n_cols;
    jb.Y = Y;
    return run_threads(jb, nthreads);
}
