/*
 * fp64 token-by-token oracle for lightning attention (linear attention with a
 * fixed per-head exponential decay).
 *
 * TEST INFRASTRUCTURE ONLY.  Built and called by the tests, the smoke check
 * and the benchmark's CPU-baseline leg; the CUDA library never links, includes
 * or calls it, and it shares no code with the CUDA kernels.
 *
 * What it computes.  The cuLA page ("cuLA benchmark results on GB200") times a
 * lightning-attention forward (fixed-length and varlen tables) and a
 * single-token `la_decode` with 64 heads of dimension 128, but prints no
 * formula.  The reading taken here is the standard lightning-attention
 * recurrence: per sequence and value head h, with state S (V x K), S[v][c],
 * a decay rate slope[h] >= 0 and lambda = exp(-slope[h]),
 *
 *   S_t = lambda S_{t-1} + v_t k_t^T          (decay first, then the write)
 *   o_t = scale * S_t q_t                     (read after the write)
 *
 * with no normalisation of q or k and no gate.  Value head h reads query/key
 * head h / (H_v / H_qk).  Every step is evaluated in double precision from the
 * exact values of the bf16 / fp32 inputs.
 *
 * The optional `mutation` argument plants one deliberate mistake so that the
 * tests can show the pins catch it; 0 is the oracle.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double la_bf16(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    const float *slope;
    double scale;
    const float *initial_state;
    double *final_state;
    const int32_t *cu_seqlens;
    int N, B, T, H_qk, H_v, K, V;
    double *out;
    int mutation;
    int n_units, next_unit;
    pthread_mutex_t lock;
} la_job_t;

static void la_unit(la_job_t *J, int unit) {
    const int n = unit / J->H_v, h = unit % J->H_v;
    const int G = J->H_v / J->H_qk;
    int hq = h / G;
    if (J->mutation == 6) hq = h % J->H_qk;                    /* heads grouped the wrong way */
    const int K = J->K, V = J->V;
    long bos = 0, len = J->T;
    int bidx = n;
    if (J->cu_seqlens) {
        bos = J->cu_seqlens[n];
        len = (long)J->cu_seqlens[n + 1] - bos;
        bidx = 0;
    }
    double *S = (double *)malloc(sizeof(double) * (size_t)V * K);
    const size_t sbase = ((size_t)n * J->H_v + h) * (size_t)V * K;
    for (size_t i = 0; i < (size_t)V * K; ++i)
        S[i] = J->initial_state ? (double)J->initial_state[sbase + i] : 0.0;
    int hs = h;
    if (J->mutation == 5) hs = (h + 1) % J->H_v;               /* another head's decay */
    const double lambda = exp(-(double)J->slope[hs]);
    const double scale = J->mutation == 4 ? 1.0 : J->scale;   /* 4: scale dropped */

    for (long t = 0; t < len; ++t) {
        const size_t tok = (size_t)bidx * J->T + (size_t)(bos + t);
        const uint16_t *qp = J->q + (tok * J->H_qk + hq) * K;
        const uint16_t *kp = J->k + (tok * J->H_qk + hq) * K;
        const uint16_t *vp = J->v + (tok * J->H_v + h) * V;
        double *op = J->out + (tok * J->H_v + h) * V;
        for (int r = 0; r < V; ++r) {
            double *Sr = S + (size_t)r * K;
            const double vr = la_bf16(vp[r]);
            double acc = 0.0;
            if (J->mutation == 2) {                             /* output read before the write */
                for (int c = 0; c < K; ++c) acc += lambda * Sr[c] * la_bf16(qp[c]);
                for (int c = 0; c < K; ++c) Sr[c] = lambda * Sr[c] + vr * la_bf16(kp[c]);
                op[r] = scale * acc;
                continue;
            }
            for (int c = 0; c < K; ++c) {
                const double w = J->mutation == 3 ? la_bf16(qp[c]) : la_bf16(kp[c]);   /* 3: q written */
                if (J->mutation == 1) Sr[c] = lambda * (Sr[c] + vr * w);          /* 1: write, then decay */
                else Sr[c] = lambda * Sr[c] + vr * w;
                acc += Sr[c] * la_bf16(qp[c]);
            }
            op[r] = scale * acc;
        }
    }
    if (J->final_state) memcpy(J->final_state + sbase, S, sizeof(double) * (size_t)V * K);
    free(S);
}

static void *la_worker(void *arg) {
    la_job_t *J = (la_job_t *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= J->n_units) break;
        la_unit(J, u);
    }
    return NULL;
}

/*
 * Forward over all sequences.  Layouts (row-major): q, k [B,T,H_qk,K] bf16
 * bits; v [B,T,H_v,V]; slope [H_v] fp32; initial_state [Nseq,H_v,V,K] fp32 or
 * NULL (zeros); final_state [Nseq,H_v,V,K] fp64 or NULL; out [B,T,H_v,V] fp64.
 * With cu_seqlens (int32 [N+1], host memory) B must be 1 and Nseq = N;
 * otherwise Nseq = B.  Returns 0, or -1 on bad arguments.
 */
int la_oracle_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *slope, float scale,
                  const float *initial_state, double *final_state, const int32_t *cu_seqlens, int N, int B,
                  int T, int H_qk, int H_v, int K, int V, double *out, int nthreads, int mutation) {
    if (B < 0 || T < 0 || H_qk <= 0 || H_v <= 0 || K <= 0 || V <= 0) return -1;
    if (H_v % H_qk != 0) return -1;
    if (cu_seqlens && B != 1) return -1;
    const int nseq = cu_seqlens ? N : B;
    if (nseq < 0) return -1;
    la_job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.slope = slope;
    J.scale = (double)scale;
    J.initial_state = initial_state; J.final_state = final_state;
    J.cu_seqlens = cu_seqlens;
    J.N = N; J.B = B; J.T = T; J.H_qk = H_qk; J.H_v = H_v; J.K = K; J.V = V;
    J.out = out;
    J.mutation = mutation;
    J.n_units = nseq * H_v;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > J.n_units) nthreads = J.n_units > 0 ? J.n_units : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, la_worker, &J);
    la_worker(&J);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return 0;
}
