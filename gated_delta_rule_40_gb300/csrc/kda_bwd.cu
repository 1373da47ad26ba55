// KDA backward in the chunk (UT / WY) form: gradients of the forward with respect to q, k,
// v, graw, b, A_log and the initial state, given the gradients of the outputs (do) and of
// the final states (dht).
//
// Per chunk of C = 64 rows (S_0 the state entering it; Gam the inclusive in-chunk prefix sum
// of g = -exp(A_log) softplus(graw), per channel; Gam_C its last row; Kh, Qt the normalised
// keys and scaled queries; beta = sigmoid(b)):
//   Kg = Kh e^Gam,  Qg = Qt e^Gam,  Kd = Kh e^(Gam_C - Gam)
//   A = strict_lower(diag(beta) Kh Kh^T with pair decays e^(Gam_r - Gam_j)),  T = (I + A)^-1
//   P = lower(Qt Kh^T with the same decays)
//   W = T diag(beta) Kg,  U = T diag(beta) V,  Delta = U - W S_0^T
//   O = Qg S_0^T + P Delta,   S_C = S_0 Diag(e^Gam_C) + Delta^T Kd
// and its backward, given dO and dS_C (the gradient of the state leaving the chunk):
//   dDelta = P^T dO + Kd dS_C^T        dKd = Delta dS_C     dQg = dO S_0     dW = -dDelta S_0
//   dS_0   = dS_C Diag(e^Gam_C) - (Kd dS_C^T)^T W + dO^T (Qg - P W)
//   dP = lower(dO Delta^T),  dT = dDelta (beta V)^T + dW (beta Kg)^T,  dA = strict_lower(-T^T dT T^T)
// then the products A, P, W, U and the decayed copies pass their gradients to Kh, Qt, V,
// beta and Gam (the pair products per 16-row sub-block pair, against the sub-block's
// reference point as the forward builds A and P), and dg_s = sum_{r >= s} dGam_r + dGam_C
// terms + the exclusive prefix sum of dKd * Kd (Kd_r depends on g_s for s > r only).
//
// Kernels (one "item" is a (chunk, value head) pair):
//   bwdc_prep_kernel     per item: the chunk's rows, A and P, T, W, U, Kd and N = Qg - P W
//                        (the operands of both state chains and of the gradient kernels)
//   bwdc_chain_kernel    per (sequence, value head, 64-row V block), chunks in order: the
//                        state entering every chunk (forward) or, chunks in reverse, the
//                        state gradient leaving every chunk (backward); dh0
//   bwdc_gradv_kernel    per (item, V half): the products that contract over the value
//                        dimension (Delta, dDelta, dKd, dQg, dW, dP, dT's V term), dv
//   bwdc_gradk_kernel    per item: dT, dA, the decayed pair products, dGam and dg
//   bwdc_jacobian_kernel per (query/key head, 64 tokens): the norms', gate's and sigmoid's
//                        Jacobians (dq and dk sum over the value heads of a group)
// Every product runs on the tensor cores (mma.sync m16n8k8, tf32 operands rounded to
// nearest, fp32 accumulation) from fp32 tiles in shared memory; the state chains keep the
// state in fp32 and apply the per-channel decay in fp32 outside the products.
#include "kda_common.cuh"
#include <cstring>

#include "kda_invert.cuh"
#include "kda_tma.cuh"

namespace kda {

cudaError_t launch_plan(const int32_t *cu, int N, int B, int T, SeqDesc *seqs, ChunkDesc *chunks, int *order,
                        int *hdr, long long max_chunks, cudaStream_t stream);
long long max_chunks_for(int N, int B, int T, bool varlen);
void timing_mark(const char *name, cudaStream_t s);

// ---------------------------------------------------------------- fp32 tiles
// A tile holds rows x W fp32 (W = 64 or 128) densely, with the 16-byte units of row r
// permuted: unit u sits at u ^ s(r), s(r) = 2 (r & 3) + ((r >> 2) & 1).  The two fragment
// shapes of mma.sync (eight rows x four consecutive columns, four rows x eight consecutive
// columns) then touch 32 distinct banks, and a tile moves between global and shared memory
// as one contiguous block.
template <int W>
__device__ __forceinline__ int toff(int r, int c) {
    return r * W + ((((c >> 2) ^ (((r & 3) << 1) | ((r >> 2) & 1)))) << 2) + (c & 3);
}

__device__ __forceinline__ int tswz(int r) { return ((r & 3) << 1) | ((r >> 2) & 1); }

// Four 8 x 8 b16 matrices from shared memory: lanes 8 i .. 8 i + 7 give the row addresses of
// matrix i; register i of lane l holds row l / 4, 32-bit column l % 4 of matrix i.  On an fp32
// tile, an 8 x 4 block of fp32 values is one such matrix, and lane l receives (l / 4, l % 4):
// the tf32 fragment element for (g, t).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// ---- fragment loaders: la(a, k) fills a[TM][4] (rows m0.. of A, columns k..k+7), lb(b, k)
// fills b[TN][2] (rows k..k+7 of B, columns n0..).  "K-contiguous" loaders read a tile whose
// rows are the fragment's M (or N) index and whose columns are K, with ldmatrix; RND adds the
// round-to-nearest step for values that are not tf32 numbers already.
template <int W, int TM, bool RND>
struct AKc {   // A (m, k) = tile[m][k], tile row stride W floats (unit-permuted) or AS (plain, W = 0)
    uint32_t base[TM];
    int sw[TM], hi;
    __device__ __forceinline__ AKc(const float *tile, int m0, int lane) {
        hi = lane >> 4;
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int r = m0 + 16 * i + (lane & 7) + ((lane >> 3) & 1) * 8;
            base[i] = smem_u32(tile) + (uint32_t)(r * (W ? W : AS) * 4);
            sw[i] = W ? tswz(r) : 0;
        }
    }
    __device__ __forceinline__ void operator()(uint32_t (&a)[TM][4], int k) const {
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            ldsm_x4(a[i], base[i] + ((((k >> 2) + hi) ^ sw[i]) << 4));
            if (RND)
#pragma unroll
                for (int e = 0; e < 4; ++e) a[i][e] += 0x1000u;
        }
    }
};
template <int W, int TN, bool RND>
struct BKc {   // B (k, n) = tile[n][k], TN even
    static_assert(TN % 2 == 0, "pairs of n8 tiles");
    uint32_t base[TN / 2];
    int sw[TN / 2], hi;
    __device__ __forceinline__ BKc(const float *tile, int n0, int lane) {
        hi = (lane >> 3) & 1;
#pragma unroll
        for (int q = 0; q < TN / 2; ++q) {
            const int r = n0 + 16 * q + (lane & 7) + (lane >> 4) * 8;
            base[q] = smem_u32(tile) + (uint32_t)(r * W * 4);
            sw[q] = tswz(r);
        }
    }
    __device__ __forceinline__ void operator()(uint32_t (&b)[TN][2], int k) const {
#pragma unroll
        for (int q = 0; q < TN / 2; ++q) {
            uint32_t r[4];
            ldsm_x4(r, base[q] + ((((k >> 2) + hi) ^ sw[q]) << 4));
            if (RND)
#pragma unroll
                for (int e = 0; e < 4; ++e) r[e] += 0x1000u;
            b[2 * q][0] = r[0];
            b[2 * q][1] = r[1];
            b[2 * q + 1][0] = r[2];
            b[2 * q + 1][1] = r[3];
        }
    }
};
// scalar loaders from value accessors f(m, k) / f(k, n); RND false when the values are tf32 numbers
template <int TM, bool RND, class F>
struct AFn {
    F f;
    int m0, g, t;
    __device__ __forceinline__ void operator()(uint32_t (&a)[TM][4], int k) const {
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int m = m0 + 16 * i + g;
            const float v[4] = {f(m, k + t), f(m + 8, k + t), f(m, k + t + 4), f(m + 8, k + t + 4)};
#pragma unroll
            for (int e = 0; e < 4; ++e) a[i][e] = RND ? tf32_rn_bits(v[e]) : __float_as_uint(v[e]);
        }
    }
};
template <int TN, bool RND, class F>
struct BFn {
    F f;
    int n0, g, t;
    __device__ __forceinline__ void operator()(uint32_t (&b)[TN][2], int k) const {
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int n = n0 + 8 * j + g;
            const float v0 = f(k + t, n), v1 = f(k + t + 4, n);
            b[j][0] = RND ? tf32_rn_bits(v0) : __float_as_uint(v0);
            b[j][1] = RND ? tf32_rn_bits(v1) : __float_as_uint(v1);
        }
    }
};
template <int TM, bool RND, class F>
__device__ __forceinline__ AFn<TM, RND, F> afn(F f, int m0, int g, int t) { return AFn<TM, RND, F>{f, m0, g, t}; }
template <int TN, bool RND, class F>
__device__ __forceinline__ BFn<TN, RND, F> bfn(F f, int n0, int g, int t) { return BFn<TN, RND, F>{f, n0, g, t}; }

// acc += A B over k in [k0, k1) with fragment loaders
template <int TM, int TN, class LA, class LB>
__device__ __forceinline__ void mma_frag(float (&acc)[TM][TN][4], int k0, int k1, const LA &la, const LB &lb) {
#pragma unroll 2
    for (int k = k0; k < k1; k += 8) {
        uint32_t a[TM][4], b[TN][2];
        la(a, k);
        lb(b, k);
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) mma_tf32(acc[i][j], a[i], b[j]);
    }
}

// fe(row, col, v[col], v[col + 1]) for every accumulator pair of the tile (col even)
template <int TM, int TN, class FE>
__device__ __forceinline__ void tile_out(const float (&acc)[TM][TN][4], int m0, int n0, int g, int t, FE fe) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int r = m0 + 16 * i + g, c = n0 + 8 * j + 2 * t;
            fe(r, c, acc[i][j][0], acc[i][j][1]);
            fe(r + 8, c, acc[i][j][2], acc[i][j][3]);
        }
}
template <int TM, int TN>
__device__ __forceinline__ void tile_zero(float (&acc)[TM][TN][4]) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
}
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(src_smem),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void st2(float *p, float a, float b) { *reinterpret_cast<float2 *>(p) = make_float2(a, b); }
__device__ __forceinline__ float ex2n(float x) { return ex2(x * LOG2E); }   // e^x

// ---------------------------------------------------------------- workspace records
// Per item, written by the prep kernel (fp32 tiles):
//   W, Kd, N = Qg - P W  [64 rows][128];  U as two [64 rows][64 v] halves;  P, T, KK [64][64]
//   (KK = the key products of A before the beta scaling);  D = e^Gam_C [128];  beta [64]
constexpr uint32_t BR_W = 0, BR_KD = 32768, BR_N = 65536, BR_U = 98304, BR_P = 131072, BR_T = 147456,
                   BR_KK = 163840, BR_D = 180224, BR_BETA = 180736, BR_BYTES = 181248;
constexpr uint32_t ST_BYTES = 65536;   // a state per item: [2 V blocks][64 v][128 k] fp32 tiles
// Per item, written by bwdc_gradv_kernel (sums over the 128 value columns):
//   dKd, dQg, dW [64][128];  dP (lower), dT's V term [64][64];  dbeta's V term [64];  colsum(S_0 dS_C) [128]
constexpr uint32_t CP_DKD = 0, CP_DQG = 32768, CP_DW = 65536, CP_DP = 98304, CP_DT = 114688, CP_DB = 131072,
                   CP_DGC = 131328, CP_BYTES = 131840;

struct BwdcParams {
    const uint16_t *q, *k, *v, *graw, *b, *dout;
    const float *A_log, *init, *dht;
    float scale;
    int H_qk, H_v, nseq;
    const SeqDesc *seqs;
    const ChunkDesc *chunks;
    const int *order;
    const int *hdr;
    unsigned char *rec;     // [item] BR_BYTES
    float *S0, *dSC;        // [item] ST_BYTES: state entering / state gradient leaving each chunk
    unsigned char *part;    // [item] CP_BYTES
    float *dqt, *dkh;       // [token][H_v][128]: gradients of Qt, Kh
    float *dgraw, *db;      // outputs [token][H_v][128], [token][H_v]
    float *dal;             // [item]: the item's share of dA_log
    float *dv, *dh0;
};


// The chunk's rows into shared memory: Kh = k / |k| and Qt = scale q / |q| (fp32 tiles),
// Gam (fp32 tile; rows past len repeat the last valid row, their g being 0), beta = sigmoid(b)
// (0 past len) and D = e^Gam_C.  All NT threads take part (sTot: NT floats of scratch);
// returns synchronised.
// L2 prefetch of one item's token rows, issued one item ahead so that the next item's row loads
// hit L2.  `mask` selects the tensors: RP_QKG (q and k of the item's q/k head, graw and b of its
// value head), RP_V (v), RP_DO (dO); two 128-byte lines per row of q, k, graw, v, dO and one for
// b.  The requests are spread over the CTA's threads.
enum { RP_QKG = 1, RP_V = 2, RP_DO = 4 };
template <int NT>
__device__ __forceinline__ void prefetch_rows_l2(const BwdcParams &p, const ChunkDesc &cd, int h, int hq, int mask,
                                                 int tid) {
    for (int u = tid; u < CH * 11; u += NT) {
        const int r = u / 11, w = u % 11;
        if (r >= cd.len) continue;
        const size_t tok = (size_t)cd.tok + r;
        const uint16_t *src = nullptr;
        if (w < 6) {
            if (!(mask & RP_QKG)) continue;
            src = w < 2 ? p.q + (tok * p.H_qk + hq) * KD : w < 4 ? p.k + (tok * p.H_qk + hq) * KD
                                                              : p.graw + (tok * p.H_v + h) * KD;
        } else if (w < 8) {
            if (!(mask & RP_V)) continue;
            src = p.v + (tok * p.H_v + h) * KD;
        } else if (w < 10) {
            if (!(mask & RP_DO)) continue;
            src = p.dout + (tok * p.H_v + h) * KD;
        } else {
            if (mask & RP_QKG) prefetch_line_l2(p.b + tok * p.H_v + h);
            continue;
        }
        prefetch_line_l2(src + 64 * (w & 1));
    }
}

// L2 prefetch of a contiguous global range (16-byte aligned, a multiple of 16 bytes) in bulk
// requests of at most 32 KiB, from one thread.
__device__ __forceinline__ void prefetch_range_l2(const void *src, uint32_t bytes) {
    const unsigned char *c = static_cast<const unsigned char *>(src);
    for (uint32_t o = 0; o < bytes; o += 32768u) prefetch_l2(c + o, bytes - o < 32768u ? bytes - o : 32768u);
}

template <int NT>
__device__ void bwdc_rows(const BwdcParams &p, int tok0, int len, int h, int hq, float a, float *sKh, float *sQt,
                          float *sG, float *sBeta, float *sD, float *sTot, int tid) {
    constexpr int NW = NT / 32, RPW = CH / NW;   // rows per warp
    const int warp = tid >> 5, lane = tid & 31;
    // the warp's rows: all loads first, then the arithmetic
    uint2 qw[RPW], kw[RPW], gw[RPW];
    float bv[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = warp + NW * i;
        qw[i] = kw[i] = gw[i] = make_uint2(0u, 0u);
        bv[i] = 0.f;
        if (r < len) {
            const size_t tok = (size_t)tok0 + r;
            const size_t qo = (tok * p.H_qk + hq) * KD + 4 * lane, vo = (tok * p.H_v + h) * KD + 4 * lane;
            qw[i] = *reinterpret_cast<const uint2 *>(p.q + qo);
            kw[i] = *reinterpret_cast<const uint2 *>(p.k + qo);
            gw[i] = *reinterpret_cast<const uint2 *>(p.graw + vo);
            bv[i] = bf16_to_f(p.b[tok * p.H_v + h]);
        }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = warp + NW * i;
        float4 kh = make_float4(0.f, 0.f, 0.f, 0.f), qt = kh, gg = kh;
        float beta = 0.f;
        if (r < len) {
            const float qv[4] = {bf16_lo(qw[i].x), bf16_hi(qw[i].x), bf16_lo(qw[i].y), bf16_hi(qw[i].y)};
            const float kv[4] = {bf16_lo(kw[i].x), bf16_hi(kw[i].x), bf16_lo(kw[i].y), bf16_hi(kw[i].y)};
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sq = fmaf(qv[e], qv[e], sq);
                sk = fmaf(kv[e], kv[e], sk);
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            const float rq = p.scale * rsqrtf(sq + L2_EPS), rk = rsqrtf(sk + L2_EPS);
            qt = make_float4(qv[0] * rq, qv[1] * rq, qv[2] * rq, qv[3] * rq);
            kh = make_float4(kv[0] * rk, kv[1] * rk, kv[2] * rk, kv[3] * rk);
            // g = -a softplus(graw), natural units
            const float na = -a * (1.0f / LOG2E);
            gg = make_float4(na * softplus_log2(bf16_lo(gw[i].x)), na * softplus_log2(bf16_hi(gw[i].x)),
                             na * softplus_log2(bf16_lo(gw[i].y)), na * softplus_log2(bf16_hi(gw[i].y)));
            beta = 1.0f / (1.0f + ex2(-bv[i] * LOG2E));
        }
        const int o = toff<KD>(r, 4 * lane);
        *reinterpret_cast<float4 *>(sKh + o) = kh;
        *reinterpret_cast<float4 *>(sQt + o) = qt;
        *reinterpret_cast<float4 *>(sG + o) = gg;
        if (lane == 0) sBeta[r] = beta;
    }
    __syncthreads();
    // prefix sums down each channel: NT / 128 threads per channel, each over a segment of rows,
    // then every segment adds the totals of the segments above it
    constexpr int SEG = NT / KD, SR = CH / SEG;
    const int c = tid & (KD - 1), seg = tid / KD;
    {
        float sacc = 0.f;
        for (int r = SR * seg; r < SR * (seg + 1); ++r) {
            const int o = toff<KD>(r, c);
            sacc += sG[o];
            sG[o] = sacc;
        }
        sTot[seg * KD + c] = sacc;
    }
    __syncthreads();
    if (seg > 0) {
        float base = 0.f;
        for (int s2 = 0; s2 < seg; ++s2) base += sTot[s2 * KD + c];
        float last = 0.f;
        for (int r = SR * seg; r < SR * (seg + 1); ++r) {
            const int o = toff<KD>(r, c);
            last = sG[o] + base;
            sG[o] = last;
        }
        if (seg == SEG - 1) sD[c] = ex2n(last);
    }
    __syncthreads();
}

// Decay factors of the sub-block pair (i, b), b <= i, for channel c: e^(Gam_r - Gam_j) =
// rowf(r) colf(j) for r in block i, j in block b.  Below the diagonal the reference point is
// Gam at the last row of block i - 1 (both factors <= 1); on it, the block's midpoint with
// both exponents clamped at 85 nats (exact unless a channel decays by more than 170 nats
// across the block).
struct PairRef {
    float ref;
    bool diag;
    __device__ __forceinline__ float rowf(float gam) const {
        return diag ? ex2n(fminf(gam - ref, 85.0f)) : ex2n(gam - ref);
    }
    __device__ __forceinline__ float colf(float gam) const {
        return diag ? ex2n(fminf(ref - gam, 85.0f)) : ex2n(ref - gam);
    }
};
__device__ __forceinline__ PairRef pair_ref(const float *sG, int i, int b, int c) {
    PairRef pr;
    pr.diag = (i == b);
    pr.ref = pr.diag ? 0.5f * (sG[toff<KD>(16 * i, c)] + sG[toff<KD>(16 * i + 15, c)]) : sG[toff<KD>(16 * i - 1, c)];
    return pr;
}
__device__ __forceinline__ void pair_of(int pr, int &i, int &b) {
    // (0,0) (1,0) (1,1) (2,0) (2,1) (2,2) (3,0) (3,1) (3,2) (3,3)
    i = pr < 1 ? 0 : pr < 3 ? 1 : pr < 6 ? 2 : 3;
    b = pr - (i * (i + 1)) / 2;
}

// =====================================================================
// Prep: per item the chunk's rows, KK (A before beta) and P by sub-block pairs, T, W, U, Kd,
// N; written to the item's record.  One item per CTA (16 warps) at a time.
// =====================================================================
constexpr int PN_THREADS = 512, PN_WARPS = 16;
constexpr uint32_t PS_KH = 0, PS_QT = 32768, PS_G = 65536, PS_W = 98304, PS_KK = 131072, PS_P = 147456,
                   PS_A = 163840, PS_T = 181248, PS_X = 198656, PS_MISC = 203264, PS_BYTES = 204288;
constexpr uint32_t PS_V = PS_QT;   // V (fp32 tile) once Qt is no longer read
static_assert(PS_T == PS_A + CH * AS * 4 && PS_X == PS_T + CH * AS * 4 && PS_MISC >= PS_X + 32 * XS * 4 &&
              PS_MISC >= PS_X + PN_THREADS * 4, "prep layout");

__global__ __launch_bounds__(PN_THREADS, 1) void bwdc_prep_kernel(const BwdcParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = aligned_smem<128>(smem_raw);
    if (p.hdr[1] == 0) return;
    float *sKh = reinterpret_cast<float *>(sm + PS_KH), *sQt = reinterpret_cast<float *>(sm + PS_QT);
    float *sG = reinterpret_cast<float *>(sm + PS_G), *sW = reinterpret_cast<float *>(sm + PS_W);
    float *sKK = reinterpret_cast<float *>(sm + PS_KK), *sP = reinterpret_cast<float *>(sm + PS_P);
    float *sA = reinterpret_cast<float *>(sm + PS_A), *sT = reinterpret_cast<float *>(sm + PS_T);
    float *sX = reinterpret_cast<float *>(sm + PS_X), *sV = reinterpret_cast<float *>(sm + PS_V);
    float *sBeta = reinterpret_cast<float *>(sm + PS_MISC), *sD = sBeta + 64;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const long long n_items = (long long)p.hdr[0] * p.H_v;
    const int group = p.H_v / p.H_qk;
    for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int h = (int)(item % p.H_v);
        const ChunkDesc cd = p.chunks[item / p.H_v];
        const int hq = h / group, len = cd.len;
        const float a = ex2n(p.A_log[h]);
        float *rec = reinterpret_cast<float *>(p.rec + (size_t)item * BR_BYTES);
        if (item + gridDim.x < n_items) {   // the next item's rows into L2
            const long long nx = item + gridDim.x;
            const int nh = (int)(nx % p.H_v);
            prefetch_rows_l2<PN_THREADS>(p, p.chunks[nx / p.H_v], nh, nh / group, RP_QKG | RP_V, tid);
        }
        __syncthreads();   // the previous item's reads of shared memory are done
        bwdc_rows<PN_THREADS>(p, cd.tok, len, h, hq, a, sKh, sQt, sG, sBeta, sD, sX, tid);

        // ---- KK and P per sub-block pair and 8-column half (20 units, one warp each):
        //      16 x 8, K = 128 channels
        for (int u = warp; u < 20; u += PN_WARPS) {
            int i, b;
            pair_of(u >> 1, i, b);
            const int jn = u & 1;
            float kk[4] = {0.f, 0.f, 0.f, 0.f}, pp[4] = {0.f, 0.f, 0.f, 0.f};
            const int r0 = 16 * i + g, j = 16 * b + 8 * jn + g;
#pragma unroll 4
            for (int k0 = 0; k0 < KD; k0 += 8) {
                const PairRef f0 = pair_ref(sG, i, b, k0 + t), f1 = pair_ref(sG, i, b, k0 + t + 4);
                const float e00 = f0.rowf(sG[toff<KD>(r0, k0 + t)]), e10 = f0.rowf(sG[toff<KD>(r0 + 8, k0 + t)]);
                const float e01 = f1.rowf(sG[toff<KD>(r0, k0 + t + 4)]), e11 = f1.rowf(sG[toff<KD>(r0 + 8, k0 + t + 4)]);
                uint32_t ak[4], aq[4], bb[2];
                ak[0] = tf32_rn_bits(sKh[toff<KD>(r0, k0 + t)] * e00);
                ak[1] = tf32_rn_bits(sKh[toff<KD>(r0 + 8, k0 + t)] * e10);
                ak[2] = tf32_rn_bits(sKh[toff<KD>(r0, k0 + t + 4)] * e01);
                ak[3] = tf32_rn_bits(sKh[toff<KD>(r0 + 8, k0 + t + 4)] * e11);
                aq[0] = tf32_rn_bits(sQt[toff<KD>(r0, k0 + t)] * e00);
                aq[1] = tf32_rn_bits(sQt[toff<KD>(r0 + 8, k0 + t)] * e10);
                aq[2] = tf32_rn_bits(sQt[toff<KD>(r0, k0 + t + 4)] * e01);
                aq[3] = tf32_rn_bits(sQt[toff<KD>(r0 + 8, k0 + t + 4)] * e11);
                bb[0] = tf32_rn_bits(sKh[toff<KD>(j, k0 + t)] * f0.colf(sG[toff<KD>(j, k0 + t)]));
                bb[1] = tf32_rn_bits(sKh[toff<KD>(j, k0 + t + 4)] * f1.colf(sG[toff<KD>(j, k0 + t + 4)]));
                mma_tf32(kk, ak, bb);
                mma_tf32(pp, aq, bb);
            }
            // masks by selection (above the diagonal the clamped factors may overflow)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = 16 * i + g + 8 * hh, c = 16 * b + 8 * jn + 2 * t;
                const float k0v = (i > b || c < r) ? kk[2 * hh] : 0.f;
                const float k1v = (i > b || c + 1 < r) ? kk[2 * hh + 1] : 0.f;
                const float p0v = (i > b || c <= r) ? pp[2 * hh] : 0.f;
                const float p1v = (i > b || c + 1 <= r) ? pp[2 * hh + 1] : 0.f;
                st2(sKK + toff<CH>(r, c), k0v, k1v);
                st2(sP + toff<CH>(r, c), tf32_rn(p0v), tf32_rn(p1v));   // P: a tensor-core operand only
            }
        }
        // the six blocks above the diagonal are zero
        for (int idx = tid; idx < 6 * 256; idx += PN_THREADS) {
            const int blk = idx >> 8, e = idx & 255;
            const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
            const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            const int o = toff<CH>(16 * bi + (e >> 4), 16 * bj + (e & 15));
            sKK[o] = 0.f;
            sP[o] = 0.f;
        }
        __syncthreads();
        // A = beta KK for the inversion; KK and P to the record
        for (int idx = tid; idx < CH * CH; idx += PN_THREADS) {
            const int r = idx >> 6, jj = idx & 63;
            sA[r * AS + jj] = sBeta[r] * sKK[toff<CH>(r, jj)];
        }
        for (int idx = tid; idx < CH * CH / 4; idx += PN_THREADS) {
            reinterpret_cast<float4 *>(rec + BR_KK / 4)[idx] = reinterpret_cast<const float4 *>(sKK)[idx];
            reinterpret_cast<float4 *>(rec + BR_P / 4)[idx] = reinterpret_cast<const float4 *>(sP)[idx];
        }
        __syncthreads();
        invert_unit_lower64<PN_THREADS>(sA, sT, sX, tid, warp, lane);
        for (int idx = tid; idx < CH * CH; idx += PN_THREADS) {
            const int r = idx >> 6, jj = idx & 63;
            rec[BR_T / 4 + toff<CH>(r, jj)] = tf32_rn(sT[r * AS + jj]);
        }
        if (tid < KD) rec[BR_D / 4 + tid] = sD[tid];
        if (tid < CH) rec[BR_BETA / 4 + tid] = sBeta[tid];
        // ---- W = T (beta Kg) -> shared (for N) and the record; Kd = Kh e^(Gam_C - Gam).  W, Kd, N,
        // P and T are tensor-core operands only wherever they are read: stored as tf32 numbers
        const int m0 = 16 * (warp >> 2), n0 = 32 * (warp & 3);   // this warp's 16 x 32 tile of 64 x 128
        {
            float acc[1][4][4];
            tile_zero(acc);
            mma_frag(acc, 0, CH, AKc<0, 1, true>(sT, m0, lane),
                     bfn<4, true>([&](int jj, int c) { return sBeta[jj] * sKh[toff<KD>(jj, c)] * ex2n(sG[toff<KD>(jj, c)]); },
                                  n0, g, t));
            tile_out<1, 4>(acc, m0, n0, g, t, [&](int r, int c, float v0, float v1) {
                st2(sW + toff<KD>(r, c), tf32_rn(v0), tf32_rn(v1));
                st2(rec + BR_W / 4 + toff<KD>(r, c), tf32_rn(v0), tf32_rn(v1));
            });
        }
        for (int idx = tid; idx < CH * KD / 4; idx += PN_THREADS) {
            const int r = idx >> 5, c = 4 * (idx & 31), o = toff<KD>(r, c);
            const float4 kh = *reinterpret_cast<const float4 *>(sKh + o), gm = *reinterpret_cast<const float4 *>(sG + o);
            const float4 gc = *reinterpret_cast<const float4 *>(sG + toff<KD>(CH - 1, c));
            *reinterpret_cast<float4 *>(rec + BR_KD / 4 + o) =
                make_float4(tf32_rn(kh.x * ex2n(gc.x - gm.x)), tf32_rn(kh.y * ex2n(gc.y - gm.y)),
                            tf32_rn(kh.z * ex2n(gc.z - gm.z)), tf32_rn(kh.w * ex2n(gc.w - gm.w)));
        }
        __syncthreads();
        // ---- N = Qt e^Gam - P W
        {
            float acc[1][4][4];
            tile_zero(acc);
            mma_frag(acc, 0, CH, AKc<CH, 1, false>(sP, m0, lane),
                     bfn<4, false>([&](int jj, int c) { return sW[toff<KD>(jj, c)]; }, n0, g, t));
            tile_out<1, 4>(acc, m0, n0, g, t, [&](int r, int c, float v0, float v1) {
                const int o = toff<KD>(r, c);
                st2(rec + BR_N / 4 + o, tf32_rn(sQt[o] * ex2n(sG[o]) - v0), tf32_rn(sQt[o + 1] * ex2n(sG[o + 1]) - v1));
            });
        }
        __syncthreads();
        // ---- V (fp32) over Qt, then U = T (beta V) as two 64-column halves
        for (int idx = tid; idx < CH * KD / 8; idx += PN_THREADS) {
            const int r = idx >> 4, c = 8 * (idx & 15);
            float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
            if (r < len) {
                const uint4 w = *reinterpret_cast<const uint4 *>(p.v + ((size_t)(cd.tok + r) * p.H_v + h) * KD + c);
                lo = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
                hi = make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
            }
            *reinterpret_cast<float4 *>(sV + toff<KD>(r, c)) = lo;
            *reinterpret_cast<float4 *>(sV + toff<KD>(r, c + 4)) = hi;
        }
        __syncthreads();
        {
            float acc[1][4][4];
            tile_zero(acc);
            mma_frag(acc, 0, CH, AKc<0, 1, true>(sT, m0, lane),
                     bfn<4, true>([&](int jj, int c) { return sBeta[jj] * sV[toff<KD>(jj, c)]; }, n0, g, t));
            tile_out<1, 4>(acc, m0, n0, g, t, [&](int r, int c, float v0, float v1) {
                st2(rec + BR_U / 4 + (c >> 6) * (CH * CH) + toff<CH>(r, c & 63), v0, v1);
            });
        }
    }
}

// =====================================================================
// State chains: one CTA per (sequence, value head, 64-row V block), the 64 x 128 state X in
// fp32 (a tile in shared memory).  Per chunk (forward: in order; backward: in reverse):
//   forward   E = X W^T,   Z = U^T - E,  X <- X Diag(D) + Z Kd              (X = S, stored as S_0)
//   backward  E = X Kd^T,  Z = -E,       X <- X Diag(D) + Z W + dO^T N      (X = dS, stored as dS_C)
// The item operands (32 KiB tiles W, Kd, N) stream through a ring of slots by bulk copies,
// issued one chunk ahead by thread 0 once the slots' previous contents are consumed; the
// per-chunk extras (D, and U's V block or the chunk's dO rows) through a double buffer.
// Every wait is bounded; a timeout records KDA_ERR_DEVICE_TIMEOUT and the CTA stops.
// =====================================================================
constexpr int CN_THREADS = 256, CN_WARPS = 8;
template <bool BWD>
struct ChainCfg {
    static constexpr int OPS = BWD ? 3 : 2;             // ring tiles per chunk
    static constexpr int SLOTS = BWD ? 5 : 4;
    // extras per chunk: backward: the chunk's dO block (64 rows x 64 bf16, a TMA box with the
    // 128-byte swizzle, 1024-byte aligned), then D; forward: D, then U's V block
    static constexpr uint32_t AUX_D = BWD ? 8192 : 0, AUX_M = BWD ? 0 : 512;
    static constexpr uint32_t AUX = BWD ? 9216 : 512 + CH * CH * 4;
    static constexpr uint32_t X = 0, Z = 32768, RING = 49152, AUXB = RING + SLOTS * 32768;
    // the backward's barriers sit in the unused tail of its second extras buffer
    static constexpr uint32_t BAR = BWD ? AUXB + AUX + 8704 : AUXB + 2 * AUX;
    static constexpr uint32_t BYTES = BWD ? AUXB + 2 * AUX : BAR + 8 * (SLOTS + 2);
};
static_assert(ChainCfg<true>::BAR + 8 * (ChainCfg<true>::SLOTS + 2) <= ChainCfg<true>::BYTES &&
              ChainCfg<true>::AUXB % 1024 == 0 && ChainCfg<true>::AUX % 1024 == 0, "chain layout");
static_assert(ChainCfg<true>::BYTES + 1024 <= 232448 && ChainCfg<false>::BYTES + 1024 <= 232448, "chain smem");

template <bool BWD>
__global__ __launch_bounds__(CN_THREADS, 1) void bwdc_chain_kernel(const __grid_constant__ CUtensorMap tdo,
                                                                     const BwdcParams p) {
    using Cfg = ChainCfg<BWD>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = aligned_smem<1024>(smem_raw);
    if (p.hdr[1] == 0) return;
    const int vb = blockIdx.x & 1;
    const int h = (blockIdx.x >> 1) % p.H_v;
    const int rank = (blockIdx.x >> 1) / p.H_v;
    if (rank >= p.nseq) return;
    const int seq = p.order[rank];
    const SeqDesc sd = p.seqs[seq];
    const int n = sd.nchunk;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    float *sX = reinterpret_cast<float *>(sm + Cfg::X), *sZ = reinterpret_cast<float *>(sm + Cfg::Z);
    const uint32_t sbase = smem_u32(sm), bar = sbase + Cfg::BAR;
    const size_t sh = ((size_t)seq * p.H_v + h) * KD * KD + (size_t)vb * CH * KD;   // rows of init / dht / dh0

    if (tid == 0) {
        for (int i = 0; i < Cfg::SLOTS + 2; ++i) mbar_init(bar + 8 * i, 1);
        mbar_fence_init();
    }
    // X from the initial state (forward) or the final state's gradient (backward)
    const float *x0 = BWD ? p.dht : p.init;
    for (int idx = tid; idx < CH * KD / 4; idx += CN_THREADS) {
        const int r = idx >> 5, c = 4 * (idx & 31);
        const float4 v = x0 ? *reinterpret_cast<const float4 *>(x0 + sh + (size_t)r * KD + c)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(sX + toff<KD>(r, c)) = v;
    }
    fence_async_smem();
    __syncthreads();

    auto chunk_of = [&](int s) { return BWD ? n - 1 - s : s; };
    auto item_of = [&](int s) { return ((size_t)sd.chunk0 + chunk_of(s)) * p.H_v + h; };
    auto issue = [&](int s) {   // thread 0: the ring tiles and extras of step s
        const unsigned char *rec = p.rec + item_of(s) * BR_BYTES;
        const uint32_t offs[3] = {BWD ? BR_KD : BR_W, BWD ? BR_W : BR_KD, BR_N};
        const uint32_t ab = bar + 8 * (Cfg::SLOTS + (s & 1)), aux = sbase + Cfg::AUXB + (s & 1) * Cfg::AUX;
#pragma unroll
        for (int op = 0; op < Cfg::OPS; ++op) {
            const int slot = (Cfg::OPS * s + op) % Cfg::SLOTS;
            mbar_expect_tx(bar + 8 * slot, 32768);
            bulk_g2s(sbase + Cfg::RING + slot * 32768, rec + offs[op], 32768, bar + 8 * slot);
        }
        if (BWD) {
            // the chunk's 64 dO rows, channels of this V block, in one tensor copy (rows past the
            // sequence are read but never used; past the tensor they are zero)
            mbar_expect_tx(ab, 512 + CH * CH * 2);
            bulk_g2s(aux + Cfg::AUX_D, rec + BR_D, 512, ab);
            tma_load_3d(aux, &tdo, vb * CH, h, sd.tok + chunk_of(s) * CH, ab);
        } else {
            mbar_expect_tx(ab, 512 + CH * CH * 4);
            bulk_g2s(aux, rec + BR_D, 512, ab);
            bulk_g2s(aux + Cfg::AUX_M, rec + BR_U + vb * (CH * CH * 4), CH * CH * 4, ab);
        }
    };
    if (tid == 0 && n > 0) issue(0);

    float *outbase = BWD ? p.dSC : p.S0;
    bool ok = true;
    for (int s = 0; s < n; ++s) {
        // all of step s's operands (bounded wait; the CTA decides together)
        bool mine = true;
#pragma unroll
        for (int op = 0; op < Cfg::OPS; ++op) {
            const int pos = Cfg::OPS * s + op;
            mine = mine && mbar_wait(bar + 8 * (pos % Cfg::SLOTS), (pos / Cfg::SLOTS) & 1);
        }
        mine = mine && mbar_wait(bar + 8 * (Cfg::SLOTS + (s & 1)), (s >> 1) & 1);
        if (!__syncthreads_and(mine)) {
            if (tid == 0) set_status(KDA_ERR_DEVICE_TIMEOUT);
            ok = false;
            break;
        }
        const float *op1 = reinterpret_cast<const float *>(sm + Cfg::RING + ((Cfg::OPS * s) % Cfg::SLOTS) * 32768);
        const float *op2 = reinterpret_cast<const float *>(sm + Cfg::RING + ((Cfg::OPS * s + 1) % Cfg::SLOTS) * 32768);
        const float *op3 = reinterpret_cast<const float *>(sm + Cfg::RING + ((Cfg::OPS * s + 2) % Cfg::SLOTS) * 32768);
        const unsigned char *aux = sm + Cfg::AUXB + (s & 1) * Cfg::AUX;
        const float *sD = reinterpret_cast<const float *>(aux + Cfg::AUX_D);
        const int c = chunk_of(s), len = min(CH, sd.len - c * CH);
        // the state entering this step, to the workspace
        if (tid == 0) {
            bulk_s2g(outbase + item_of(s) * (ST_BYTES / 4) + vb * (CH * KD), sbase + Cfg::X, 32768);
            bulk_commit();
        }
        // ---- E (64 v x 64 r) = X op1^T, then Z (a tensor-core operand only: stored as tf32 numbers)
        {
            static_assert(CN_WARPS == 8, "eight 16 x 32 tiles of E");
            const int m0 = 16 * (warp >> 1), n0 = 32 * (warp & 1);
            float acc[1][4][4];
            tile_zero(acc);
            mma_frag(acc, 0, KD, AKc<KD, 1, true>(sX, m0, lane), BKc<KD, 4, false>(op1, n0, lane));
            tile_out<1, 4>(acc, m0, n0, g, t, [&](int v, int r, float e0, float e1) {
                float z0 = -e0, z1 = -e1;
                if (!BWD) {
                    const float *u = reinterpret_cast<const float *>(aux + Cfg::AUX_M);   // U block [r][v]
                    z0 += u[toff<CH>(r, v)];
                    z1 += u[toff<CH>(r + 1, v)];
                }
                st2(sZ + toff<CH>(v, r), tf32_rn(z0), tf32_rn(z1));
            });
        }
        __syncthreads();   // Z complete; op1 consumed
        if (tid == 0 && s + 1 < n) issue(s + 1);
        // ---- X <- X Diag(D) + Z op2 (+ dO^T N)
        {
            const int m0 = 32 * (warp >> 2), n0 = 32 * (warp & 3);
            float acc[2][4][4];
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = m0 + 16 * i + g, cc = n0 + 8 * j + 2 * t;
                    const float d0 = sD[cc], d1 = sD[cc + 1];
                    acc[i][j][0] = sX[toff<KD>(r, cc)] * d0;
                    acc[i][j][1] = sX[toff<KD>(r, cc + 1)] * d1;
                    acc[i][j][2] = sX[toff<KD>(r + 8, cc)] * d0;
                    acc[i][j][3] = sX[toff<KD>(r + 8, cc + 1)] * d1;
                }
            mma_frag(acc, 0, CH, AKc<CH, 2, false>(sZ, m0, lane),
                     bfn<4, false>([&](int r, int cc) { return op2[toff<KD>(r, cc)]; }, n0, g, t));
            if (BWD) {
                // dO[r][v] in the TMA box: 128-byte rows, 16-byte unit u of row r at u ^ (r % 8)
                mma_frag(acc, 0, CH,
                         afn<2, false>(
                             [&](int v, int r) {
                                 const uint32_t off = (uint32_t)(r * 128 + ((((2 * v) >> 4) ^ (r & 7)) << 4) + ((2 * v) & 15));
                                 return r < len ? bf16_to_f(*reinterpret_cast<const uint16_t *>(aux + off)) : 0.f;
                             },
                             m0, g, t),
                         bfn<4, false>([&](int r, int cc) { return op3[toff<KD>(r, cc)]; }, n0, g, t));
            }
            if (tid == 0) bulk_wait_read_all();   // the store of X has read it
            __syncthreads();                      // every warp is done reading X, Z and the operands
            tile_out<2, 4>(acc, m0, n0, g, t, [&](int r, int cc, float v0, float v1) { st2(sX + toff<KD>(r, cc), v0, v1); });
        }
        fence_async_smem();
    }
    __syncthreads();
    if (BWD && ok) {
        for (int idx = tid; idx < CH * KD / 4; idx += CN_THREADS) {
            const int r = idx >> 5, cc = 4 * (idx & 31);
            *reinterpret_cast<float4 *>(p.dh0 + sh + (size_t)r * KD + cc) =
                *reinterpret_cast<const float4 *>(sX + toff<KD>(r, cc));
        }
    }
    if (tid == 0) bulk_wait_all();
    // a failed CTA may leave copies in flight: let them land before the CTA's memory goes away
    if (!ok && tid == 0)
        for (int i = 0; i < Cfg::SLOTS + 2; ++i) {
            mbar_wait(bar + 8 * i, 0, 1u << 14);
            mbar_wait(bar + 8 * i, 1, 1u << 14);
        }
}

// =====================================================================
// Gradients over the value dimension, per item (16 warps), the two 64-column halves of V in
// turn (S0_h, dS_h: rows of that half of the states):
//   Delta_h = U_h - W S0_h^T,  dDelta_h = P^T dO_h + Kd dS_h^T        (64 r x 64 v)
//   dKd += Delta_h dS_h,  dQg += dO_h S0_h,  dW += -dDelta_h S0_h      (64 r x 128 k, registers)
//   dP += dO_h Delta_h^T,  dT += dDelta_h (beta V_h)^T                 (64 x 64, registers)
//   dv_h = beta (T^T dDelta_h),  dbeta += rowsum(T^T dDelta_h * V_h),  dGam_C += colsum(S0_h * dS_h)
// then the sums to the item's record of value-side gradients.
// =====================================================================
constexpr int GN_THREADS = 512;
constexpr uint32_t GV_W = 0, GV_KD = 32768, GV_S0 = 65536, GV_DS = 98304, GV_U = 131072, GV_P = 147456,
                   GV_T = 163840, GV_DO = 180224, GV_V = 196608, GV_DDL = 212992, GV_MISC = 229376,
                   GV_BAR = GV_MISC + 768, GV_BYTES = GV_BAR + 16;
static_assert(GV_BYTES + 128 <= 232448, "gradv smem");

__global__ __launch_bounds__(GN_THREADS, 1) void bwdc_gradv_kernel(const BwdcParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = aligned_smem<128>(smem_raw);
    if (p.hdr[1] == 0) return;
    float *sW = reinterpret_cast<float *>(sm + GV_W), *sKd = reinterpret_cast<float *>(sm + GV_KD);
    float *sS0 = reinterpret_cast<float *>(sm + GV_S0), *sDS = reinterpret_cast<float *>(sm + GV_DS);
    float *sU = reinterpret_cast<float *>(sm + GV_U), *sP = reinterpret_cast<float *>(sm + GV_P);
    float *sT = reinterpret_cast<float *>(sm + GV_T), *sDO = reinterpret_cast<float *>(sm + GV_DO);
    float *sV = reinterpret_cast<float *>(sm + GV_V), *sDD = reinterpret_cast<float *>(sm + GV_DDL);
    float *sD = reinterpret_cast<float *>(sm + GV_MISC), *sBeta = sD + 128;
    const uint32_t sbase = smem_u32(sm), bar_item = sbase + GV_BAR, bar_half = bar_item + 8;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const long long n_items = (long long)p.hdr[0] * p.H_v;
    if (tid == 0) {
        mbar_init(bar_item, 1);
        mbar_init(bar_half, 1);
        mbar_fence_init();
    }
    __syncthreads();
    // fixed output tiles of this warp: 16 x 32 of the 64 x 128 products, 16 x 16 of the 64 x 64 ones
    const int m0 = 16 * (warp >> 2), bn0 = 32 * (warp & 3), sn0 = 16 * (warp & 3);
    uint32_t ph_item = 0, ph_half = 0;
    for (long long item = blockIdx.x; item < n_items; item += gridDim.x, ph_item ^= 1) {
        const int h = (int)(item % p.H_v);
        const ChunkDesc cd = p.chunks[item / p.H_v];
        const int len = cd.len;
        const unsigned char *rec = p.rec + (size_t)item * BR_BYTES;
        unsigned char *part = p.part + (size_t)item * CP_BYTES;
        float akd[1][4][4], aqg[1][4][4], aw[1][4][4], ap[1][2][4], at[1][2][4];
        tile_zero(akd);
        tile_zero(aqg);
        tile_zero(aw);
        tile_zero(ap);
        tile_zero(at);
        float dbr[2] = {0.f, 0.f}, gcs = 0.f;   // this thread's dbeta row sums and S0 dS column sum
        bool ok = true;
        for (int vh = 0; vh < 2; ++vh, ph_half ^= 1) {
            fence_async_smem();   // this thread's writes to shared memory before the bulk copies that reuse it
            __syncthreads();      // the previous half's (item's) reads of shared memory are done
            if (tid == 0) {
                if (vh == 0) {
                    mbar_expect_tx(bar_item, 2 * 32768 + 2 * 16384 + 768);
                    bulk_g2s(sbase + GV_W, rec + BR_W, 32768, bar_item);
                    bulk_g2s(sbase + GV_KD, rec + BR_KD, 32768, bar_item);
                    bulk_g2s(sbase + GV_P, rec + BR_P, 16384, bar_item);
                    bulk_g2s(sbase + GV_T, rec + BR_T, 16384, bar_item);
                    bulk_g2s(sbase + GV_MISC, rec + BR_D, 768, bar_item);   // D [128], beta [64]
                }
                mbar_expect_tx(bar_half, 2 * 32768 + 16384);
                bulk_g2s(sbase + GV_S0, p.S0 + item * (ST_BYTES / 4) + vh * (CH * KD), 32768, bar_half);
                bulk_g2s(sbase + GV_DS, p.dSC + item * (ST_BYTES / 4) + vh * (CH * KD), 32768, bar_half);
                bulk_g2s(sbase + GV_U, rec + BR_U + vh * 16384, 16384, bar_half);
            }
            // dO and V of this half (fp32 tiles, zero past len)
            for (int idx = tid; idx < 2 * CH * 8; idx += GN_THREADS) {
                const int which = idx >> 9, r = (idx >> 3) & 63, c = 8 * (idx & 7);
                float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
                if (r < len) {
                    const uint16_t *src = which ? p.v : p.dout;
                    const uint4 w =
                        *reinterpret_cast<const uint4 *>(src + ((size_t)(cd.tok + r) * p.H_v + h) * KD + vh * CH + c);
                    lo = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
                    hi = make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
                }
                float *dst = which ? sV : sDO;
                *reinterpret_cast<float4 *>(dst + toff<CH>(r, c)) = lo;
                *reinterpret_cast<float4 *>(dst + toff<CH>(r, c + 4)) = hi;
            }
            bool mine = (vh > 0 || mbar_wait(bar_item, ph_item)) && mbar_wait(bar_half, ph_half);
            if (!__syncthreads_and(mine)) {
                ok = false;
                break;
            }
            if (vh == 1 && item + gridDim.x < n_items) {
                // this item's copies have landed: the next item's tiles, states and rows into L2
                // while this half computes
                const long long nx = item + gridDim.x;
                const int nh = (int)(nx % p.H_v);
                prefetch_rows_l2<GN_THREADS>(p, p.chunks[nx / p.H_v], nh, 0, RP_V | RP_DO, tid);
                if (tid == 0) {
                    const unsigned char *nrec = p.rec + (size_t)nx * BR_BYTES;
                    prefetch_range_l2(nrec + BR_W, 2 * 32768);   // W, Kd
                    prefetch_range_l2(nrec + BR_U, 32768);       // U
                    prefetch_range_l2(nrec + BR_P, 2 * 16384);   // P, T
                    prefetch_range_l2(nrec + BR_D, 768);         // D, beta
                    prefetch_range_l2(p.S0 + nx * (ST_BYTES / 4), ST_BYTES);
                    prefetch_range_l2(p.dSC + nx * (ST_BYTES / 4), ST_BYTES);
                }
            }
            // ---- Delta (in place of U) and dDelta, both tensor-core operands only from here on
            // (stored as tf32 numbers); W, Kd, P, T arrive as tf32 numbers, S0, dS as fp32
            {
                float acc[1][2][4];
                tile_zero(acc);
                mma_frag(acc, 0, KD, AKc<KD, 1, false>(sW, m0, lane), BKc<KD, 2, true>(sS0, sn0, lane));
                float dd[1][2][4];
                tile_zero(dd);
                mma_frag(dd, 0, CH, afn<1, false>([&](int r, int j) { return sP[toff<CH>(j, r)]; }, m0, g, t),
                         bfn<2, false>([&](int j, int v) { return sDO[toff<CH>(j, v)]; }, sn0, g, t));
                mma_frag(dd, 0, KD, AKc<KD, 1, false>(sKd, m0, lane), BKc<KD, 2, true>(sDS, sn0, lane));
                tile_out<1, 2>(acc, m0, sn0, g, t, [&](int r, int v, float e0, float e1) {
                    const int o = toff<CH>(r, v);
                    st2(sU + o, tf32_rn(sU[o] - e0), tf32_rn(sU[o + 1] - e1));
                });
                tile_out<1, 2>(dd, m0, sn0, g, t,
                               [&](int r, int v, float v0, float v1) { st2(sDD + toff<CH>(r, v), tf32_rn(v0), tf32_rn(v1)); });
            }
            __syncthreads();
            // ---- the sums over this half's value columns
            {
                const auto lDelta = AKc<CH, 1, false>(sU, m0, lane), lDO = AKc<CH, 1, false>(sDO, m0, lane);
                const auto lDD = AKc<CH, 1, false>(sDD, m0, lane);
                mma_frag(akd, 0, CH, lDelta, bfn<4, true>([&](int v, int k) { return sDS[toff<KD>(v, k)]; }, bn0, g, t));
                const auto lS0 = bfn<4, true>([&](int v, int k) { return sS0[toff<KD>(v, k)]; }, bn0, g, t);
                mma_frag(aqg, 0, CH, lDO, lS0);
                mma_frag(aw, 0, CH, lDD, lS0);
                mma_frag(ap, 0, CH, lDO, BKc<CH, 2, false>(sU, sn0, lane));
                mma_frag(at, 0, CH, lDD, bfn<2, true>([&](int v, int j) { return sBeta[j] * sV[toff<CH>(j, v)]; }, sn0, g, t));
            }
            // dBV = T^T dDelta: dv and dbeta's V term
            {
                float acc[1][2][4];
                tile_zero(acc);
                mma_frag(acc, 0, CH, afn<1, false>([&](int r, int j) { return sT[toff<CH>(j, r)]; }, m0, g, t),
                         bfn<2, false>([&](int j, int v) { return sDD[toff<CH>(j, v)]; }, sn0, g, t));
                float rs[2] = {0.f, 0.f};
                tile_out<1, 2>(acc, m0, sn0, g, t, [&](int r, int v, float v0, float v1) {
                    const int o = toff<CH>(r, v);
                    rs[(r - m0) >> 3] += v0 * sV[o] + v1 * sV[o + 1];
                    if (r < len) {
                        const float be = sBeta[r];
                        st2(p.dv + ((size_t)(cd.tok + r) * p.H_v + h) * KD + vh * CH + v, be * v0, be * v1);
                    }
                });
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    rs[e] += __shfl_xor_sync(0xffffffffu, rs[e], 1);
                    rs[e] += __shfl_xor_sync(0xffffffffu, rs[e], 2);
                    dbr[e] += rs[e];
                }
            }
            // colsum(S0_h * dS_h) per channel (this thread: 16 of the half's rows)
            {
                const int c = tid & 127, v0 = 16 * (tid >> 7);
                for (int v = v0; v < v0 + 16; ++v) gcs = fmaf(sS0[toff<KD>(v, c)], sDS[toff<KD>(v, c)], gcs);
            }
        }
        if (!ok) {
            if (tid == 0) set_status(KDA_ERR_DEVICE_TIMEOUT);
            break;
        }
        float *pDKD = reinterpret_cast<float *>(part + CP_DKD), *pDQG = reinterpret_cast<float *>(part + CP_DQG);
        float *pDW = reinterpret_cast<float *>(part + CP_DW), *pDP = reinterpret_cast<float *>(part + CP_DP);
        float *pDT = reinterpret_cast<float *>(part + CP_DT);
        tile_out<1, 4>(akd, m0, bn0, g, t, [&](int r, int k, float v0, float v1) { st2(pDKD + toff<KD>(r, k), v0, v1); });
        tile_out<1, 4>(aqg, m0, bn0, g, t, [&](int r, int k, float v0, float v1) { st2(pDQG + toff<KD>(r, k), v0, v1); });
        // dW: a tensor-core operand only where it is read (stored as tf32 numbers)
        tile_out<1, 4>(aw, m0, bn0, g, t,
                       [&](int r, int k, float v0, float v1) { st2(pDW + toff<KD>(r, k), tf32_rn(-v0), tf32_rn(-v1)); });
        tile_out<1, 2>(ap, m0, sn0, g, t, [&](int r, int j, float v0, float v1) {
            st2(pDP + toff<CH>(r, j), j <= r ? v0 : 0.f, j + 1 <= r ? v1 : 0.f);
        });
        tile_out<1, 2>(at, m0, sn0, g, t, [&](int r, int j, float v0, float v1) { st2(pDT + toff<CH>(r, j), v0, v1); });
        // the partial row / column sums through the (now free) dO tile, added in a fixed order
        __syncthreads();
        float *sDB = sDO, *sGC = sDO + 4 * 64;   // [4 warps of a row block][64], [4 row segments][128]
        if (t == 0) {
            sDB[(warp & 3) * 64 + m0 + g] = dbr[0];
            sDB[(warp & 3) * 64 + m0 + g + 8] = dbr[1];
        }
        sGC[(tid >> 7) * 128 + (tid & 127)] = gcs;
        __syncthreads();
        if (tid < 64)
            reinterpret_cast<float *>(part + CP_DB)[tid] = (sDB[tid] + sDB[64 + tid]) + (sDB[128 + tid] + sDB[192 + tid]);
        else if (tid >= 128 && tid < 256) {
            const int c = tid - 128;
            reinterpret_cast<float *>(part + CP_DGC)[c] = (sGC[c] + sGC[128 + c]) + (sGC[256 + c] + sGC[384 + c]);
        }
    }
}

// =====================================================================
// Gradients over the keys, per item (16 warps): dT = dT_V + dW (beta Kg)^T,
// dA = strict_lower(-T^T dT T^T), dbeta, then (warp w owns channels 8 w .. 8 w + 7, its
// accumulators in registers) dBW = T^T dW, the decayed pair products of M = beta dA and dP's
// strict part, and
//   dKh = beta dBW e^Gam + (pair products) + diag(dP) Qt + dKd e^(Gam_C - Gam)
//   dQt = dQg e^Gam + (pair products) + diag(dP) Kh
//   dGam = beta dBW Kg + (pair products' Gam terms) + dQg Qg
// and dg per channel from dGam's suffix sums, dGam_C and the exclusive prefix sums of dKd Kd.
// =====================================================================
constexpr int KN_THREADS = 512, KN_WARPS = 16;
constexpr uint32_t GK_KH = 0, GK_QT = 32768, GK_G = 65536, GK_DW = 98304, GK_T = 131072, GK_KK = 147456,
                   GK_DT = 163840, GK_X = 180224, GK_DP = 196608, GK_MISC = 212992, GK_BAR = GK_MISC + 8192,
                   GK_BYTES = GK_BAR + 16;
static_assert(GK_BYTES + 128 <= 232448, "gradk smem");

__global__ __launch_bounds__(KN_THREADS, 1) void bwdc_gradk_kernel(const BwdcParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = aligned_smem<128>(smem_raw);
    if (p.hdr[1] == 0) return;
    float *sKh = reinterpret_cast<float *>(sm + GK_KH), *sQt = reinterpret_cast<float *>(sm + GK_QT);
    float *sG = reinterpret_cast<float *>(sm + GK_G), *sDW = reinterpret_cast<float *>(sm + GK_DW);
    float *sT = reinterpret_cast<float *>(sm + GK_T), *sKK = reinterpret_cast<float *>(sm + GK_KK);
    float *sDT = reinterpret_cast<float *>(sm + GK_DT), *sX = reinterpret_cast<float *>(sm + GK_X);
    float *sDP = reinterpret_cast<float *>(sm + GK_DP);
    // beta [64], D [128], dGam_C [128], dbeta's V term [64], then the dbeta row sums of the dA
    // products (four warps per row block) [4][64] and of the dBW products (one per warp) [16][64]
    float *sBeta = reinterpret_cast<float *>(sm + GK_MISC), *sD = sBeta + 64, *sDGC = sBeta + 192,
          *sDB = sBeta + 320, *sDBa = sBeta + 384, *sDBw = sBeta + 640;
    const uint32_t sbase = smem_u32(sm), bar = sbase + GK_BAR;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const long long n_items = (long long)p.hdr[0] * p.H_v;
    const int group = p.H_v / p.H_qk;
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    const int m0 = 16 * (warp >> 2), sn0 = 16 * (warp & 3);   // 16 x 16 tiles of the 64 x 64 products
    uint32_t phase = 0;
    for (long long item = blockIdx.x; item < n_items; item += gridDim.x, phase ^= 1) {
        const int h = (int)(item % p.H_v);
        const ChunkDesc cd = p.chunks[item / p.H_v];
        const int hq = h / group, len = cd.len;
        const float a = ex2n(p.A_log[h]);
        const unsigned char *rec = p.rec + (size_t)item * BR_BYTES;
        const unsigned char *pt = p.part + (size_t)item * CP_BYTES;
        fence_async_smem();   // this thread's writes to shared memory before the bulk copies that reuse it
        __syncthreads();
        if (tid == 0) {
            mbar_expect_tx(bar, 2 * 16384 + 32768 + 2 * 16384);
            bulk_g2s(sbase + GK_T, rec + BR_T, 16384, bar);
            bulk_g2s(sbase + GK_KK, rec + BR_KK, 16384, bar);
            bulk_g2s(sbase + GK_DW, pt + CP_DW, 32768, bar);
            bulk_g2s(sbase + GK_DT, pt + CP_DT, 16384, bar);
            bulk_g2s(sbase + GK_DP, pt + CP_DP, 16384, bar);
        }
        if (tid < 64) sDB[tid] = reinterpret_cast<const float *>(pt + CP_DB)[tid];
        bwdc_rows<KN_THREADS>(p, cd.tok, len, h, hq, a, sKh, sQt, sG, sBeta, sD, sX, tid);
        if (tid < 128) sDGC[tid] = reinterpret_cast<const float *>(pt + CP_DGC)[tid] * sD[tid];
        const bool mine = mbar_wait(bar, phase);
        if (!__syncthreads_and(mine)) {
            if (tid == 0) set_status(KDA_ERR_DEVICE_TIMEOUT);
            break;
        }
        // ---- dT += dW (beta Kg)^T  (dW, T arrive as tf32 numbers; dT, X and M, tensor-core
        // operands only, are stored as tf32 numbers)
        {
            float acc[1][2][4];
            tile_zero(acc);
            mma_frag(acc, 0, KD, AKc<KD, 1, false>(sDW, m0, lane),
                     bfn<2, true>([&](int k, int j) { return sBeta[j] * sKh[toff<KD>(j, k)] * ex2n(sG[toff<KD>(j, k)]); },
                                  sn0, g, t));
            tile_out<1, 2>(acc, m0, sn0, g, t, [&](int r, int j, float v0, float v1) {
                const int o = toff<CH>(r, j);
                st2(sDT + o, tf32_rn(sDT[o] + v0), tf32_rn(sDT[o + 1] + v1));
            });
        }
        __syncthreads();
        // ---- X = dT T^T
        {
            float acc[1][2][4];
            tile_zero(acc);
            mma_frag(acc, 0, CH, AKc<CH, 1, false>(sDT, m0, lane), BKc<CH, 2, false>(sT, sn0, lane));
            tile_out<1, 2>(acc, m0, sn0, g, t,
                           [&](int r, int i, float v0, float v1) { st2(sX + toff<CH>(r, i), tf32_rn(v0), tf32_rn(v1)); });
        }
        __syncthreads();
        // ---- dA = strict_lower(-T^T X); dbeta row sums of dA KK; M = beta dA over dT
        {
            float acc[1][2][4];
            tile_zero(acc);
            mma_frag(acc, 0, CH, afn<1, false>([&](int r, int j) { return sT[toff<CH>(j, r)]; }, m0, g, t),
                     bfn<2, false>([&](int j, int i) { return sX[toff<CH>(j, i)]; }, sn0, g, t));
            float rs[2] = {0.f, 0.f};
            tile_out<1, 2>(acc, m0, sn0, g, t, [&](int r, int i, float v0, float v1) {
                const int o = toff<CH>(r, i);
                const float d0 = i < r ? -v0 : 0.f, d1 = i + 1 < r ? -v1 : 0.f;
                rs[(r - m0) >> 3] += d0 * sKK[o] + d1 * sKK[o + 1];
                const float be = sBeta[r];
                st2(sDT + o, tf32_rn(be * d0), tf32_rn(be * d1));
            });
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                rs[e] += __shfl_xor_sync(0xffffffffu, rs[e], 1);
                rs[e] += __shfl_xor_sync(0xffffffffu, rs[e], 2);
            }
            if (t == 0) {
                sDBa[(warp & 3) * 64 + m0 + g] = rs[0];
                sDBa[(warp & 3) * 64 + m0 + g + 8] = rs[1];
            }
        }
        // ---- this warp's channels: dBW = T^T dW and the beta dBW terms
        const int cw = 8 * warp;
        float akh[4][1][4], aqt[4][1][4], agm[4][1][4];
        {
            float bw[4][1][4];
            tile_zero(bw);
            mma_frag(bw, 0, CH, afn<4, false>([&](int r, int j) { return sT[toff<CH>(j, r)]; }, 0, g, t),
                     bfn<1, false>([&](int j, int c) { return sDW[toff<KD>(j, c)]; }, cw, g, t));
            float rs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) rs[e] = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = 16 * i + g + 8 * (e >> 1), c = cw + 2 * t + (e & 1);
                    const int o = toff<KD>(r, c);
                    const float eg = ex2n(sG[o]), kh = sKh[o];
                    const float x = sBeta[r] * bw[i][0][e] * eg;
                    akh[i][0][e] = x;
                    agm[i][0][e] = x * kh;
                    aqt[i][0][e] = 0.f;
                    rs[2 * i + (e >> 1)] += bw[i][0][e] * kh * eg;
                }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                rs[e] += __shfl_xor_sync(0xffffffffu, rs[e], 1);
                rs[e] += __shfl_xor_sync(0xffffffffu, rs[e], 2);
            }
            if (t == 0)
#pragma unroll
                for (int e = 0; e < 8; ++e) sDBw[warp * 64 + 16 * (e >> 1) + g + 8 * (e & 1)] = rs[e];
        }
        __syncthreads();   // M complete
        // ---- decayed pair products on this warp's channels
#pragma unroll
        for (int pr = 0; pr < 10; ++pr) {
            const int i = pr < 1 ? 0 : pr < 3 ? 1 : pr < 6 ? 2 : 3;
            const int b = pr - (i * (i + 1)) / 2;
            const bool dg_ = (i == b);
            // references for the channels this lane touches: B operands (cw + g), accumulators
            // (cw + 2t, cw + 2t + 1)
            const PairRef fb = pair_ref(sG, i, b, cw + g);
            const PairRef fc[2] = {pair_ref(sG, i, b, cw + 2 * t), pair_ref(sG, i, b, cw + 2 * t + 1)};
            auto mval = [&](int r, int j) { return sDT[toff<CH>(r, j)]; };   // strictly lower, tf32 numbers
            auto pval = [&](int r, int j) { return (!dg_ || j < r) ? sDP[toff<CH>(r, j)] : 0.f; };
            // row side: MH = M_ib Hk, PH = dPs_ib Hk (rows of block i)
            float mh[4] = {0.f, 0.f, 0.f, 0.f}, ph[4] = {0.f, 0.f, 0.f, 0.f}, y[4] = {0.f, 0.f, 0.f, 0.f};
            const int c = cw + g;
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int r0 = 16 * i + g, j0 = 16 * b + 8 * ks + t;
                uint32_t am[4], ap[4], bh[2];
                am[0] = __float_as_uint(mval(r0, j0));
                am[1] = __float_as_uint(mval(r0 + 8, j0));
                am[2] = __float_as_uint(mval(r0, j0 + 4));
                am[3] = __float_as_uint(mval(r0 + 8, j0 + 4));
                ap[0] = tf32_rn_bits(pval(r0, j0));
                ap[1] = tf32_rn_bits(pval(r0 + 8, j0));
                ap[2] = tf32_rn_bits(pval(r0, j0 + 4));
                ap[3] = tf32_rn_bits(pval(r0 + 8, j0 + 4));
                bh[0] = tf32_rn_bits(sKh[toff<KD>(j0, c)] * fb.colf(sG[toff<KD>(j0, c)]));
                bh[1] = tf32_rn_bits(sKh[toff<KD>(j0 + 4, c)] * fb.colf(sG[toff<KD>(j0 + 4, c)]));
                mma_tf32(mh, am, bh);
                mma_tf32(ph, ap, bh);
            }
            // column side: y = M_ib^T Fk + dPs_ib^T Fq (rows of block b)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int j0 = 16 * b + g, r0 = 16 * i + 8 * ks + t;
                uint32_t am[4], ap[4], bk[2], bq[2];
                am[0] = __float_as_uint(mval(r0, j0));
                am[1] = __float_as_uint(mval(r0, j0 + 8));
                am[2] = __float_as_uint(mval(r0 + 4, j0));
                am[3] = __float_as_uint(mval(r0 + 4, j0 + 8));
                ap[0] = tf32_rn_bits(pval(r0, j0));
                ap[1] = tf32_rn_bits(pval(r0, j0 + 8));
                ap[2] = tf32_rn_bits(pval(r0 + 4, j0));
                ap[3] = tf32_rn_bits(pval(r0 + 4, j0 + 8));
                const int o0 = toff<KD>(r0, c), o1 = toff<KD>(r0 + 4, c);
                const float f0 = fb.rowf(sG[o0]), f1 = fb.rowf(sG[o1]);
                bk[0] = tf32_rn_bits(sKh[o0] * f0);
                bk[1] = tf32_rn_bits(sKh[o1] * f1);
                bq[0] = tf32_rn_bits(sQt[o0] * f0);
                bq[1] = tf32_rn_bits(sQt[o1] * f1);
                mma_tf32(y, am, bk);
                mma_tf32(y, ap, bq);
            }
            // accumulate: row side into rows of block i, column side into rows of block b
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int cc = cw + 2 * t + (e & 1);
                const PairRef &f = fc[e & 1];
                {
                    const int r = 16 * i + g + 8 * (e >> 1), o = toff<KD>(r, cc);
                    const float rf = f.rowf(sG[o]);
                    const float fk = tf32_rn(sKh[o] * rf), fq = tf32_rn(sQt[o] * rf);
                    akh[i][0][e] += rf * mh[e];
                    aqt[i][0][e] += rf * ph[e];
                    agm[i][0][e] += fk * mh[e] + fq * ph[e];
                }
                {
                    const int j = 16 * b + g + 8 * (e >> 1), o = toff<KD>(j, cc);
                    const float cf = f.colf(sG[o]);
                    const float hk = tf32_rn(sKh[o] * cf);
                    akh[b][0][e] += cf * y[e];
                    agm[b][0][e] -= hk * y[e];
                }
            }
        }
        // ---- the remaining terms, dqt / dkh out, dGam and dKd Kd over dW and Qt (since the
        // barrier after M, this warp alone reads or writes its channels' columns of those two tiles)
        __syncwarp();
        const float *pkd = reinterpret_cast<const float *>(pt + CP_DKD), *pqg = reinterpret_cast<const float *>(pt + CP_DQG);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = 16 * i + g + 8 * hh, c = cw + 2 * t, o = toff<KD>(r, c);
                const float2 dk2 = *reinterpret_cast<const float2 *>(pkd + o), dq2 = *reinterpret_cast<const float2 *>(pqg + o);
                const float dpd = sDP[toff<CH>(r, r)];
                const float dkd[2] = {dk2.x, dk2.y}, dqg[2] = {dq2.x, dq2.y};
                float okh[2], oqt[2], gam[2], kdk[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = 2 * hh + u;
                    const float gm = sG[o + u], gc = sG[toff<KD>(CH - 1, c + u)];
                    const float eg = ex2n(gm), ed = ex2n(gc - gm), qt = sQt[o + u], kh = sKh[o + u];
                    okh[u] = akh[i][0][e] + dpd * qt + dkd[u] * ed;
                    oqt[u] = aqt[i][0][e] + dqg[u] * eg + dpd * kh;
                    gam[u] = agm[i][0][e] + dqg[u] * qt * eg;
                    kdk[u] = dkd[u] * kh * ed;
                }
                st2(sDW + o, gam[0], gam[1]);
                st2(sQt + o, kdk[0], kdk[1]);
                if (r < len) {
                    const size_t go = ((size_t)(cd.tok + r) * p.H_v + h) * KD + c;
                    st2(p.dkh + go, okh[0], okh[1]);
                    st2(p.dqt + go, oqt[0], oqt[1]);
                }
            }
        __syncthreads();
        // ---- dg = suffix sums of dGam + dGam_C + exclusive prefix sums of dKd Kd (four threads
        // per channel over 16-row segments, the segment totals passed through shared memory), then
        // the gate's and the sigmoid's Jacobians: dgraw = dg (-a) sigmoid(graw), the item's share of
        // dA_log = sum dg g (g = -a softplus(graw)), db = dbeta beta (1 - beta)
        // this thread's 16 gate pre-activations, requested before the scans so that their latency
        // overlaps them
        float gr16[16];
        {
            const int c = tid & (KD - 1), r0 = 16 * (tid >> 7);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                gr16[i] = r0 + i < len ? bf16_to_f(p.graw[((size_t)(cd.tok + r0 + i) * p.H_v + h) * KD + c]) : 0.f;
        }
        {
            const int c = tid & (KD - 1), seg = tid >> 7, r0 = 16 * seg;
            float pre = 0.f;
            for (int r = r0; r < r0 + 16; ++r) {
                const int o = toff<KD>(r, c);
                const float x = sQt[o];
                sQt[o] = pre;
                pre += x;
            }
            float suf = 0.f;
            for (int r = r0 + 15; r >= r0; --r) {
                const int o = toff<KD>(r, c);
                suf += sDW[o];
                sDW[o] = suf;
            }
            sX[seg * KD + c] = pre;               // dKd Kd summed over the segment
            sX[4 * KD + seg * KD + c] = suf;      // dGam summed over the segment
        }
        __syncthreads();
        {
            const int c = tid & (KD - 1), seg = tid >> 7, r0 = 16 * seg;
            float add = sDGC[c];
            for (int s2 = 0; s2 < seg; ++s2) add += sX[s2 * KD + c];
            for (int s2 = seg + 1; s2 < 4; ++s2) add += sX[4 * KD + s2 * KD + c];
            float dal = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = r0 + i;
                if (r < len) {
                    const int o = toff<KD>(r, c);
                    const float dgv = sDW[o] + sQt[o] + add;
                    const float gr = gr16[i];
                    const float sp = softplus_log2(gr) * (1.0f / LOG2E);   // softplus (natural units)
                    const float sig = 1.0f / (1.0f + __expf(-gr));
                    p.dgraw[((size_t)(cd.tok + r) * p.H_v + h) * KD + c] = dgv * (-a) * sig;
                    dal = fmaf(dgv, -a * sp, dal);
                }
            }
            dal = warp_sum(dal);
            if (lane == 0) sX[8 * KD + warp] = dal;
        }
        if (tid < len) {
            float db = sDB[tid] + (sDBa[tid] + sDBa[64 + tid]) + (sDBa[128 + tid] + sDBa[192 + tid]);
#pragma unroll
            for (int w = 0; w < KN_WARPS; ++w) db += sDBw[w * 64 + tid];
            const float be = sBeta[tid];
            p.db[(size_t)(cd.tok + tid) * p.H_v + h] = db * be * (1.0f - be);
        }
        __syncthreads();
        if (tid == 0) {
            float dal = 0.f;
            for (int w = 0; w < KN_WARPS; ++w) dal += sX[8 * KD + w];
            p.dal[item] = dal;
        }
    }
}

// =====================================================================
// The norms' Jacobians, one warp per (query/key head, 16 tokens); lane = channels
// 4 lane .. 4 lane + 3:
//   dq = scale r_q (dqt_sum - r_q^2 q (q . dqt_sum)),  r_q = 1 / sqrt(|q|^2 + eps)   (dk alike, scale 1)
// with dqt_sum / dkh_sum the sums over the value heads of the group (the gate's and the
// sigmoid's Jacobians run at the end of bwdc_gradk_kernel).
// =====================================================================
constexpr int BP_WARPS = 8;
constexpr int BP_TOKENS = 16;   // tokens per warp

__global__ __launch_bounds__(BP_WARPS * 32, 2) void bwdc_jacobian_kernel(const BwdcParams p, float *dq, float *dk,
                                                                         long long tokens) {
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * BP_WARPS + (threadIdx.x >> 5);
    const long long n_ranges = (tokens + BP_TOKENS - 1) / BP_TOKENS;
    if (gw >= n_ranges * p.H_qk) return;
    const int hq = (int)(gw % p.H_qk);
    const long long t0 = (gw / p.H_qk) * BP_TOKENS, t1 = min(t0 + BP_TOKENS, tokens);
    const int group = p.H_v / p.H_qk;
    constexpr int U = 4;   // tokens in flight: their loads are issued before any of them is used
    for (long long tb = t0; tb < t1; tb += U) {
        uint2 qw[U], kw[U];
        float4 sq[U], sk[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long tok = tb + u;
            qw[u] = kw[u] = make_uint2(0u, 0u);
            sq[u] = sk[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (tok < t1) {
                const size_t qo = ((size_t)tok * p.H_qk + hq) * KD + 4 * lane;
                qw[u] = *reinterpret_cast<const uint2 *>(p.q + qo);
                kw[u] = *reinterpret_cast<const uint2 *>(p.k + qo);
                for (int g = 0; g < group; ++g) {
                    const size_t ho = ((size_t)tok * p.H_v + hq * group + g) * KD + 4 * lane;
                    const float4 x = *reinterpret_cast<const float4 *>(p.dqt + ho);
                    const float4 y = *reinterpret_cast<const float4 *>(p.dkh + ho);
                    sq[u].x += x.x; sq[u].y += x.y; sq[u].z += x.z; sq[u].w += x.w;
                    sk[u].x += y.x; sk[u].y += y.y; sk[u].z += y.z; sk[u].w += y.w;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long tok = tb + u;
            const float qv[4] = {bf16_lo(qw[u].x), bf16_hi(qw[u].x), bf16_lo(qw[u].y), bf16_hi(qw[u].y)};
            const float kv[4] = {bf16_lo(kw[u].x), bf16_hi(kw[u].x), bf16_lo(kw[u].y), bf16_hi(kw[u].y)};
            const float dqs[4] = {sq[u].x, sq[u].y, sq[u].z, sq[u].w}, dks[4] = {sk[u].x, sk[u].y, sk[u].z, sk[u].w};
            float nq = 0.f, nk = 0.f, qd = 0.f, kd = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                nq = fmaf(qv[i], qv[i], nq);
                nk = fmaf(kv[i], kv[i], nk);
                qd = fmaf(qv[i], dqs[i], qd);
                kd = fmaf(kv[i], dks[i], kd);
            }
            nq = warp_sum(nq);
            nk = warp_sum(nk);
            qd = warp_sum(qd);
            kd = warp_sum(kd);
            if (tok < t1) {
                const size_t qo = ((size_t)tok * p.H_qk + hq) * KD + 4 * lane;
                const float rq = rsqrtf(nq + L2_EPS), rk = rsqrtf(nk + L2_EPS);
                float4 oq, ok;
                oq.x = p.scale * rq * (dqs[0] - rq * rq * qv[0] * qd); oq.y = p.scale * rq * (dqs[1] - rq * rq * qv[1] * qd);
                oq.z = p.scale * rq * (dqs[2] - rq * rq * qv[2] * qd); oq.w = p.scale * rq * (dqs[3] - rq * rq * qv[3] * qd);
                ok.x = rk * (dks[0] - rk * rk * kv[0] * kd); ok.y = rk * (dks[1] - rk * rk * kv[1] * kd);
                ok.z = rk * (dks[2] - rk * rk * kv[2] * kd); ok.w = rk * (dks[3] - rk * rk * kv[3] * kd);
                *reinterpret_cast<float4 *>(dq + qo) = oq;
                *reinterpret_cast<float4 *>(dk + qo) = ok;
            }
        }
    }
}

// dA_log[h] = sum over the chunks of the items' shares dal[chunk][h], one CTA per head, in a
// fixed order (no atomics: the gradients are reproducible bit for bit).
__global__ __launch_bounds__(256) void bwdc_dalog_kernel(const BwdcParams p, float *dA_log) {
    __shared__ float red[256];
    if (p.hdr[1] == 0) return;
    const int h = blockIdx.x, tid = threadIdx.x;
    const long long n = p.hdr[0];
    float acc = 0.f;
    for (long long r = tid; r < n; r += 256) acc += p.dal[r * p.H_v + h];
    red[tid] = acc;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (tid < o) red[tid] += red[tid + o];
        __syncthreads();
    }
    if (tid == 0) dA_log[h] = red[0];
}

// ---------------------------------------------------------------- host side
namespace {
size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }
int sm_count() {
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    return nsm > 0 ? nsm : 1;
}
}  // namespace

size_t bwd_workspace_bytes(int N, int B, int T, int H_v, bool varlen, int /*grid*/) {
    const long long nseq = varlen ? N : B, nck = max_chunks_for(N, B, T, varlen), tokens = (long long)B * T;
    const size_t items = (size_t)(nck > 0 ? nck : 1) * H_v, tk = (size_t)(tokens > 0 ? tokens : 1) * H_v;
    size_t off = a256(256);
    off = a256(off + sizeof(SeqDesc) * (size_t)(nseq > 0 ? nseq : 1));
    off = a256(off + sizeof(ChunkDesc) * (size_t)(nck > 0 ? nck : 1));
    off = a256(off + sizeof(int) * (size_t)(nseq > 0 ? nseq : 1));
    off = a256(off + items * BR_BYTES);
    off = a256(off + items * ST_BYTES);
    off = a256(off + items * ST_BYTES);
    off = a256(off + items * CP_BYTES);
    off = a256(off + tk * KD * 4 * 2);   // dqt, dkh
    off = a256(off + items * 4);         // dA_log shares
    return off;
}

int bwd_grid(int, int) { return sm_count(); }

cudaError_t launch_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                       const uint16_t *b, const float *A_log, float scale, const float *init, const int32_t *cu, int N,
                       int B, int T, int H_qk, int H_v, const uint16_t *dout, const float *dht, float *dq, float *dk,
                       float *dv, float *dgraw, float *db, float *dA_log, float *dh0, void *ws_ptr, int grid,
                       cudaStream_t stream, int *launches) {
    const bool varlen = cu != nullptr;
    const int nseq = varlen ? N : B;
    const long long nck = max_chunks_for(N, B, T, varlen), tokens = (long long)B * T;
    const size_t items = (size_t)(nck > 0 ? nck : 1) * H_v, tk = (size_t)(tokens > 0 ? tokens : 1) * H_v;
    char *base = static_cast<char *>(ws_ptr);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = base + off;
        off = a256(off + bytes);
        return p;
    };
    int *hdr = reinterpret_cast<int *>(take(256));
    SeqDesc *seqs = reinterpret_cast<SeqDesc *>(take(sizeof(SeqDesc) * (size_t)(nseq > 0 ? nseq : 1)));
    ChunkDesc *chunks = reinterpret_cast<ChunkDesc *>(take(sizeof(ChunkDesc) * (size_t)(nck > 0 ? nck : 1)));
    int *order = reinterpret_cast<int *>(take(sizeof(int) * (size_t)(nseq > 0 ? nseq : 1)));
    BwdcParams bp;
    bp.rec = reinterpret_cast<unsigned char *>(take(items * BR_BYTES));
    bp.S0 = reinterpret_cast<float *>(take(items * ST_BYTES));
    bp.dSC = reinterpret_cast<float *>(take(items * ST_BYTES));
    bp.part = reinterpret_cast<unsigned char *>(take(items * CP_BYTES));
    float *t2 = reinterpret_cast<float *>(take(tk * KD * 4 * 2));
    bp.dqt = t2;
    bp.dkh = t2 + tk * KD;
    bp.dal = reinterpret_cast<float *>(take(items * 4));
    bp.dgraw = dgraw;
    bp.db = db;
    bp.q = q; bp.k = k; bp.v = v; bp.graw = graw; bp.b = b; bp.dout = dout;
    bp.A_log = A_log; bp.init = init; bp.dht = dht; bp.scale = scale;
    bp.H_qk = H_qk; bp.H_v = H_v; bp.nseq = nseq;
    bp.seqs = seqs; bp.chunks = chunks; bp.order = order; bp.hdr = hdr;
    bp.dv = dv; bp.dh0 = dh0;
    *launches = 0;
    cudaError_t e = launch_plan(cu, N, B, T, seqs, chunks, order, hdr, nck, stream);
    if (e != cudaSuccess) return e;
    ++*launches;
    if ((e = cudaMemsetAsync(dA_log, 0, sizeof(float) * H_v, stream)) != cudaSuccess) return e;
    timing_mark("plan_kernel", stream);
    const int nsm = grid > 0 ? grid : sm_count();
    auto smem_attr = [](auto kern, uint32_t bytes) {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(bytes + 128));
    };
    if (nck > 0) {
        const long long n_items = nck * H_v;
        const int g_items = (int)(n_items < nsm ? n_items : nsm);
        if ((e = smem_attr(bwdc_prep_kernel, PS_BYTES)) != cudaSuccess) return e;
        bwdc_prep_kernel<<<g_items, PN_THREADS, PS_BYTES + 128, stream>>>(bp);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        timing_mark("bwdc_prep_kernel", stream);
    }
    if (nseq > 0) {
        const unsigned chains = (unsigned)((long long)nseq * H_v * 2);
        if ((e = cudaFuncSetAttribute(bwdc_chain_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)(ChainCfg<false>::BYTES + 1024))) != cudaSuccess ||
            (e = cudaFuncSetAttribute(bwdc_chain_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)(ChainCfg<true>::BYTES + 1024))) != cudaSuccess)
            return e;
        // dO as [token][H_v][128] bf16, boxes of 64 channels x 64 rows (the reverse chain's extras)
        CUtensorMap tdo;
        memset(&tdo, 0, sizeof(tdo));
        if (tokens > 0 && (e = tma_map_rows_heads(&tdo, dout, tokens, H_v, CH, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
        bwdc_chain_kernel<false><<<chains, CN_THREADS, ChainCfg<false>::BYTES + 1024, stream>>>(tdo, bp);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        timing_mark("bwdc_chain_kernel<fwd>", stream);
        bwdc_chain_kernel<true><<<chains, CN_THREADS, ChainCfg<true>::BYTES + 1024, stream>>>(tdo, bp);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        timing_mark("bwdc_chain_kernel<bwd>", stream);
    }
    if (nck > 0) {
        const long long n_items = nck * H_v;
        const int g_items = (int)(n_items < nsm ? n_items : nsm);
        if ((e = smem_attr(bwdc_gradv_kernel, GV_BYTES)) != cudaSuccess) return e;
        if ((e = smem_attr(bwdc_gradk_kernel, GK_BYTES)) != cudaSuccess) return e;
        bwdc_gradv_kernel<<<g_items, GN_THREADS, GV_BYTES + 128, stream>>>(bp);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        timing_mark("bwdc_gradv_kernel", stream);
        bwdc_gradk_kernel<<<g_items, KN_THREADS, GK_BYTES + 128, stream>>>(bp);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        timing_mark("bwdc_gradk_kernel", stream);
    }
    if (tokens > 0) {
        const long long warps = ((tokens + BP_TOKENS - 1) / BP_TOKENS) * H_qk;
        bwdc_jacobian_kernel<<<(unsigned)((warps + BP_WARPS - 1) / BP_WARPS), BP_WARPS * 32, 0, stream>>>(
            bp, dq, dk, tokens);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        bwdc_dalog_kernel<<<H_v, 256, 0, stream>>>(bp, dA_log);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        timing_mark("bwdc_jacobian_kernel", stream);
    }
    return cudaSuccess;
}

}  // namespace kda
