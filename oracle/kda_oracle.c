/*
 * fp64 token-by-token oracle for the Kimi Delta Attention (KDA) forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is built and called by the tests, by
 * the smoke check and by the benchmark's CPU-baseline leg.  The CUDA library
 * never links, includes or calls it, and it shares no code with the CUDA
 * kernels.
 *
 * What it computes (KDA as served by the FlashKDA library, page "FlashKDA:
 * High-performance KDA CUDA kernels for SM90+ GPUs"; that page names the fused
 * gate activation, beta sigmoid and q/k L2 norm under "Technical Features", the
 * [B,H,V,K] / [N,H,V,K] state layout and the cu_seqlens packing under "How does
 * FlashKDA's stateful/streaming (chunked) support work?", and the dtypes under
 * "How to seamlessly replace flash-linear-attention's chunk_kda").  The pages do
 * not print the recurrence; it is the standard KDA recurrence, per sequence and
 * per value head h, with state S (V x K), S[v][c]:
 *
 *   qhat = q / sqrt(sum q^2 + eps),  khat = k / sqrt(sum k^2 + eps),  eps=1e-6
 *   qt   = scale * qhat                      (only q carries the 1/sqrt(K) scale)
 *   beta = 1 / (1 + exp(-b))
 *   g_c  = -exp(A_log[h]) * softplus(graw_c),  softplus(x) = max(x,0)+log1p(exp(-|x|))
 *   S    = S Diag(exp g)                     (decay every column c)
 *   d    = S khat                            (V-vector)
 *   S    = S + beta (v - d) khat^T           (delta-rule write, S (I - beta k k^T) + beta v k^T)
 *   o    = S qt
 *
 * Every step is evaluated in double precision from the exact fp64 values of the
 * bf16 / fp32 inputs.  Sequences restart from their own initial state; value
 * head h reads query/key head h / (H_v / H_qk) (contiguous groups).
 *
 * The optional `mutation` argument plants one deliberate mistake; it exists
 * only so the tests can show that the pins catch each kind of mistake.  The
 * value 0 is the oracle.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KDA_ORACLE_EPS 1e-6

static double bf16_to_f64(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double softplus(double x) {
    return fmax(x, 0.0) + log1p(exp(-fabs(x)));
}

typedef struct {
    const uint16_t *q, *k, *v, *graw, *b;
    const float *A_log;
    double scale;
    const float *initial_state;
    double *final_state;
    const int32_t *cu_seqlens;
    int N, B, T, H_qk, H_v, K, V;
    double *out;
    int mutation;
    /* work distribution */
    int n_units;
    int next_unit;
    pthread_mutex_t lock;
} job_t;

/* One (sequence, value-head) chain, token by token. */
static void run_unit(job_t *J, int unit) {
    const int n = unit / J->H_v, h = unit % J->H_v;
    const int G = J->H_v / J->H_qk, hq = h / G;
    const int K = J->K, V = J->V;
    long bos, len;
    int bidx;
    if (J->cu_seqlens) {
        bos = J->cu_seqlens[n];
        len = (long)J->cu_seqlens[n + 1] - bos;
        bidx = 0;
    } else {
        bos = 0;
        len = J->T;
        bidx = n;
    }
    double *S = (double *)malloc(sizeof(double) * (size_t)V * K);
    double *qt = (double *)malloc(sizeof(double) * K);
    double *kh = (double *)malloc(sizeof(double) * K);
    double *dec = (double *)malloc(sizeof(double) * K);
    double *d = (double *)malloc(sizeof(double) * V);
    const size_t sbase = ((size_t)n * J->H_v + h) * (size_t)V * K;
    for (size_t i = 0; i < (size_t)V * K; ++i)
        S[i] = J->initial_state ? (double)J->initial_state[sbase + i] : 0.0;
    const double a = exp((double)J->A_log[h]);

    for (long t = 0; t < len; ++t) {
        const size_t tok = (size_t)bidx * J->T + (size_t)(bos + t);
        const uint16_t *qp = J->q + (tok * J->H_qk + hq) * K;
        const uint16_t *kp = J->k + (tok * J->H_qk + hq) * K;
        const uint16_t *vp = J->v + (tok * J->H_v + h) * V;
        const uint16_t *gp = J->graw + (tok * J->H_v + h) * K;
        const double bb = bf16_to_f64(J->b[tok * J->H_v + h]);

        double sq = 0.0, sk = 0.0;
        for (int c = 0; c < K; ++c) {
            double x = bf16_to_f64(qp[c]), y = bf16_to_f64(kp[c]);
            sq += x * x;
            sk += y * y;
        }
        double rq = 1.0 / sqrt(sq + KDA_ORACLE_EPS);
        double rk = 1.0 / sqrt(sk + KDA_ORACLE_EPS);
        if (J->mutation == 5) rk = 1.0;                 /* k not normalised */
        for (int c = 0; c < K; ++c) {
            qt[c] = J->scale * bf16_to_f64(qp[c]) * rq;
            kh[c] = bf16_to_f64(kp[c]) * rk;
            if (J->mutation == 6) kh[c] *= J->scale;     /* scale applied to k too */
        }
        double beta = 1.0 / (1.0 + exp(-bb));
        if (J->mutation == 7) beta = bb;                 /* no sigmoid */
        for (int c = 0; c < K; ++c) {
            double gc = -a * softplus(bf16_to_f64(gp[c]));
            if (J->mutation == 8) gc = -a * bf16_to_f64(gp[c]);   /* softplus dropped */
            dec[c] = exp(gc);
            if (J->mutation == 1) dec[c] = 1.0;          /* decay dropped */
        }
        if (J->mutation == 9) {                          /* channel index reversed in the decay */
            for (int c = 0; c < K / 2; ++c) {
                double tmp = dec[c];
                dec[c] = dec[K - 1 - c];
                dec[K - 1 - c] = tmp;
            }
        }
        for (int r = 0; r < V; ++r) {
            double *Sr = S + (size_t)r * K;
            double acc = 0.0;
            for (int c = 0; c < K; ++c) {
                Sr[c] *= dec[c];
                acc += Sr[c] * kh[c];
            }
            d[r] = acc;
        }
        if (J->mutation == 4) {                          /* state read transposed */
            for (int r = 0; r < V; ++r) {
                double acc = 0.0;
                for (int c = 0; c < K; ++c) acc += S[(size_t)c * K + r] * kh[c];
                d[r] = acc;
            }
        }
        double *op = J->out + (tok * J->H_v + h) * V;
        for (int r = 0; r < V; ++r) {
            double *Sr = S + (size_t)r * K;
            const double vr = bf16_to_f64(vp[r]);
            double delta = beta * (vr - d[r]);
            if (J->mutation == 2) delta = beta * (vr + d[r]);   /* wrong sign of the erase term */
            if (J->mutation == 3) {                              /* output read before the write */
                double acc0 = 0.0;
                for (int c = 0; c < K; ++c) acc0 += Sr[c] * qt[c];
                for (int c = 0; c < K; ++c) Sr[c] += delta * kh[c];
                op[r] = acc0;
                continue;
            }
            double acc = 0.0;
            for (int c = 0; c < K; ++c) {
                Sr[c] += delta * kh[c];
                acc += Sr[c] * qt[c];
            }
            op[r] = acc;
        }
    }
    if (J->final_state)
        memcpy(J->final_state + sbase, S, sizeof(double) * (size_t)V * K);
    free(S);
    free(qt);
    free(kh);
    free(dec);
    free(d);
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= J->n_units) break;
        run_unit(J, u);
    }
    return NULL;
}

/*
 * Forward over all sequences.  Layouts (row-major):
 *   q, k [B,T,H_qk,K] bf16 bits; v [B,T,H_v,V]; graw [B,T,H_v,K]; b [B,T,H_v];
 *   A_log [H_v] fp32; initial_state [Nseq,H_v,V,K] fp32 or NULL (zeros);
 *   final_state [Nseq,H_v,V,K] fp64 or NULL; out [B,T,H_v,V] fp64.
 * With cu_seqlens (int32 [N+1], host memory) B must be 1 and Nseq = N;
 * otherwise Nseq = B.  Returns 0, or -1 on bad arguments.
 */
int kda_oracle_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const uint16_t *graw, const uint16_t *b, const float *A_log,
                   float scale, const float *initial_state, double *final_state,
                   const int32_t *cu_seqlens, int N, int B, int T, int H_qk,
                   int H_v, int K, int V, double *out, int nthreads, int mutation) {
    if (B < 0 || T < 0 || H_qk <= 0 || H_v <= 0 || K <= 0 || V <= 0) return -1;
    if (H_v % H_qk != 0) return -1;
    if (cu_seqlens && B != 1) return -1;
    int nseq = cu_seqlens ? N : B;
    if (nseq < 0) return -1;
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.graw = graw; J.b = b; J.A_log = A_log;
    J.scale = (double)scale;
    J.initial_state = initial_state; J.final_state = final_state;
    J.cu_seqlens = cu_seqlens;
    J.N = N; J.B = B; J.T = T; J.H_qk = H_qk; J.H_v = H_v; J.K = K; J.V = V;
    J.out = out;
    J.mutation = mutation;
    J.n_units = nseq * H_v;
    J.next_unit = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > J.n_units) nthreads = J.n_units > 0 ? J.n_units : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &J);
    worker(&J);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return 0;
}
