// Chunked KDA forward: varlen plan, fused prologue + intra-chunk (UT/WY)
// kernel, and the inter-chunk state scan.
//
// Chunk algebra (chunk of C = 64 rows, state S_0 entering the chunk, per-channel
// log decay g, in-chunk inclusive prefix Gam_r = sum_{s<=r} g_s):
//   A[r,j] = beta_r sum_c kh[r,c] kh[j,c] exp(Gam[r,c]-Gam[j,c])   (j < r)
//   P[r,j] = sum_c qt[r,c] kh[j,c] exp(Gam[r,c]-Gam[j,c])          (j <= r)
//   T = (I + A)^{-1},  W = T diag(beta) (Kh*exp(Gam)),  U = T diag(beta) V
//   Delta = U - W S_0^T,  O = (Qt*exp(Gam)) S_0^T + P Delta
//   S_C = S_0 Diag(exp(Gam_C)) + Delta^T (Kh*exp(Gam_C - Gam))
// obtained by unrolling S_r = S_{r-1} D_r + delta_r kh_r^T with
// delta_r = beta_r (v_r - S_{r-1} D_r kh_r) inside the chunk.
//
// Numerical layout: Gam is kept in log2 units.  exp(Gam_r - Gam_j) is never
// formed as exp(Gam_r) exp(-Gam_j) across a chunk; 16-row sub-blocks below the
// diagonal use the reference m_i = Gam[16 i - 1] (both factors <= 1), diagonal
// sub-blocks use the per-channel midpoint of the block's first and last Gam
// with both exponents clamped at 85 nats.  Operand precision: the intra-chunk
// products and U, P, Kd, Delta are tf32 (fp32 accumulate); W and Qg are stored
// in bf16 and multiply a bf16 copy of the state; the state itself is fp32.
#include "kda_common.cuh"

namespace kda {

// =====================================================================
// Plan: sequence and chunk tables from cu_seqlens, longest sequence first.
// =====================================================================
constexpr int PLAN_THREADS = 1024;
constexpr int LPT_MAX_SEQ = 1024;

__global__ __launch_bounds__(PLAN_THREADS) void plan_kernel(const int32_t *__restrict__ cu, int N, int B, int T,
                                                            SeqDesc *__restrict__ seqs,
                                                            ChunkDesc *__restrict__ chunks,
                                                            int *__restrict__ order, int *__restrict__ hdr,
                                                            long long max_chunks) {
    __shared__ int s_bad;
    __shared__ int s_carry;
    __shared__ int s_scan[PLAN_THREADS];
    __shared__ int s_len[LPT_MAX_SEQ];
    const int tid = threadIdx.x;
    const int nseq = cu ? N : B;
    if (tid == 0) {
        s_bad = 0;
        s_carry = 0;
        if (cu && (cu[0] != 0 || cu[N] != T)) s_bad = 1;
    }
    __syncthreads();
    if (cu)
        for (int i = tid; i < N; i += PLAN_THREADS)
            if (cu[i + 1] < cu[i]) s_bad = 1;
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            hdr[0] = 0;
            hdr[1] = 0;
            set_status(KDA_ERR_BAD_SEQLENS);
        }
        return;
    }
    for (int base = 0; base < nseq; base += PLAN_THREADS) {
        const int i = base + tid;
        int len = 0, tok = 0;
        if (i < nseq) {
            tok = cu ? cu[i] : i * T;
            len = cu ? cu[i + 1] - cu[i] : T;
        }
        const int nc = (len + CH - 1) / CH;
        s_scan[tid] = nc;
        __syncthreads();
        for (int off = 1; off < PLAN_THREADS; off <<= 1) {
            const int x = tid >= off ? s_scan[tid - off] : 0;
            __syncthreads();
            s_scan[tid] += x;
            __syncthreads();
        }
        if (i < nseq) {
            SeqDesc sd;
            sd.tok = tok;
            sd.len = len;
            sd.chunk0 = s_carry + s_scan[tid] - nc;
            sd.nchunk = nc;
            seqs[i] = sd;
        }
        __syncthreads();
        if (tid == PLAN_THREADS - 1) s_carry += s_scan[PLAN_THREADS - 1];
        __syncthreads();
    }
    const int total = s_carry;
    if (total > max_chunks) {
        if (tid == 0) {
            hdr[0] = 0;
            hdr[1] = 0;
            set_status(KDA_ERR_BAD_SEQLENS);
        }
        return;
    }
    for (int i = tid; i < nseq; i += PLAN_THREADS) {
        const SeqDesc sd = seqs[i];
        for (int c = 0; c < sd.nchunk; ++c) {
            ChunkDesc cd;
            cd.seq = i;
            cd.tok = sd.tok + c * CH;
            cd.len = min(CH, sd.len - c * CH);
            cd.idx = c;
            chunks[sd.chunk0 + c] = cd;
        }
    }
    if (nseq <= LPT_MAX_SEQ) {
        for (int i = tid; i < nseq; i += PLAN_THREADS) s_len[i] = cu ? cu[i + 1] - cu[i] : T;
        __syncthreads();
        for (int i = tid; i < nseq; i += PLAN_THREADS) {
            const int li = s_len[i];
            int rank = 0;
            for (int j = 0; j < nseq; ++j) {
                const int lj = s_len[j];
                rank += (lj > li) || (lj == li && j < i);
            }
            order[rank] = i;
        }
    } else {
        for (int i = tid; i < nseq; i += PLAN_THREADS) order[i] = i;
    }
    if (tid == 0) {
        hdr[0] = total;
        hdr[1] = 1;
    }
}

// =====================================================================
// Intra-chunk kernel: one CTA per (chunk, value head).
// =====================================================================
constexpr int IN_THREADS = 256;
constexpr int SL = 32;            // channel slice
constexpr int OPS = SL + 4;       // operand row stride (floats): conflict-free fragments
constexpr int KGS = KD + 8;       // sKg row stride
constexpr int AS = CH + 4;        // sA / sT row stride
constexpr int GS = SL + 1;        // sG row stride

struct IntraSmem {
    uint16_t v[CH][KD];              // raw v rows (bf16), kept for U
    union {
        struct {
            uint16_t q[CH][KD];
            uint16_t k[CH][KD];
            uint16_t g[CH][KD];
        } raw;                       // live during the slice loop
        struct {
            float A[CH][AS];
            float T[CH][AS];
            float Z[3][SUB][SUB + 1];
        } inv;                       // live after the slice loop
    } u;
    float rq[CH], rk[CH], beta[CH], qk[CH];  // qk: qt . kh, the exact diagonal of P
    float G[CH][GS];                 // Gam slice (log2 units)
    float ref[5 + 4 + 3 + 4 + 4][SL];  // m0..m4, mu0..mu3, X(2,0) X(3,1) X(3,0), Eb0..3, Ea0..3
    float op[6][CH][OPS];            // FK FQ HK DRK DRQ DCK (tf32)
    float Kg[CH][KGS];               // kh * exp(Gam) (tf32), W operand
};

// Per (chunk, value head) record written by the intra-chunk kernel and read
// by the scan with bulk copies.  Every operand is stored as the exact shared
// memory image the scan's tcgen05.mma reads (K-major, 128-byte swizzle):
//   WQ  [Qg rows 0..63 ; W rows 64..127] x K=128, bf16          (32 KiB)
//   P   rows 0..63 x 64 (j), tf32                                (16 KiB)
//   KDT Kd^T: rows k = 0..127 x 64 (r), tf32                      (32 KiB)
//   U   [V block 0 | V block 1], each [64 r][64 v] fp32 row-major  (32 KiB)
//   GC  exp(Gam_C) per channel, fp32                              (512 B)
constexpr uint32_t REC_WQ = 0, REC_P = 32768, REC_KDT = 49152, REC_U = 81920, REC_GC = 114688;
constexpr uint32_t REC_BYTES = 115200;

struct IntraParams {
    const uint16_t *q, *k, *v, *graw, *b;
    const float *A_log;
    float scale;
    int H_qk, H_v;
    const ChunkDesc *chunks;
    const int *hdr;
    unsigned char *rec;   // [chunk][H_v] records of REC_BYTES
};

enum { OP_FK = 0, OP_FQ, OP_HK, OP_DRK, OP_DRQ, OP_DCK };
enum { R_M = 0, R_MU = 5, R_X = 9, R_EB = 12, R_EA = 16 };

// (block-row, block-col) pairs of the lower-triangular 4 x 4 sub-block grid
__constant__ int c_pair_i[10] = {0, 1, 1, 2, 2, 2, 3, 3, 3, 3};
__constant__ int c_pair_b[10] = {0, 0, 1, 0, 1, 2, 0, 1, 2, 3};

__global__ __launch_bounds__(IN_THREADS, 1) void intra_kernel(const IntraParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    IntraSmem &s = *reinterpret_cast<IntraSmem *>(smem_raw);
    const int chunk = blockIdx.x, h = blockIdx.y;
    if (p.hdr[1] == 0 || chunk >= p.hdr[0]) return;
    const ChunkDesc cd = p.chunks[chunk];
    const int hq = h / (p.H_v / p.H_qk);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;   // mma fragment coordinates
    const size_t ch = (size_t)chunk * p.H_v + h;
    unsigned char *rec = p.rec + ch * REC_BYTES;
    const int len = cd.len;

    // ---- 1. stage raw rows (cp.async 16 B), zero-fill the padded rows
    for (int idx = tid; idx < CH * (KD / 8); idx += IN_THREADS) {
        const int r = idx >> 4, c8 = (idx & 15) * 8;
        if (r < len) {
            const size_t tok = (size_t)cd.tok + r;
            cp_async16(&s.u.raw.q[r][c8], p.q + (tok * p.H_qk + hq) * KD + c8);
            cp_async16(&s.u.raw.k[r][c8], p.k + (tok * p.H_qk + hq) * KD + c8);
            cp_async16(&s.u.raw.g[r][c8], p.graw + (tok * p.H_v + h) * KD + c8);
            cp_async16(&s.v[r][c8], p.v + (tok * p.H_v + h) * KD + c8);
        } else {
            const uint4 z = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(&s.u.raw.q[r][c8]) = z;
            *reinterpret_cast<uint4 *>(&s.u.raw.k[r][c8]) = z;
            *reinterpret_cast<uint4 *>(&s.u.raw.g[r][c8]) = z;
            *reinterpret_cast<uint4 *>(&s.v[r][c8]) = z;
        }
    }
    cp_async_commit();
    if (tid < CH) {
        float be = 0.f;
        if (tid < len) {
            const float bb = bf16_to_f(p.b[((size_t)cd.tok + tid) * p.H_v + h]);
            be = 1.0f / (1.0f + ex2(-bb * LOG2E));
        }
        s.beta[tid] = be;
    }
    const float a_gate = ex2(p.A_log[h] * LOG2E);
    cp_async_wait<0>();
    __syncthreads();

    // ---- 2. row norms (warp w: rows 8w..8w+7)
    for (int rr = 0; rr < CH / 8; ++rr) {
        const int r = warp * 8 + rr;
        const uint2 qw = *reinterpret_cast<const uint2 *>(&s.u.raw.q[r][4 * lane]);
        const uint2 kw = *reinterpret_cast<const uint2 *>(&s.u.raw.k[r][4 * lane]);
        float a0 = bf16_lo(qw.x), a1 = bf16_hi(qw.x), a2 = bf16_lo(qw.y), a3 = bf16_hi(qw.y);
        float b0 = bf16_lo(kw.x), b1 = bf16_hi(kw.x), b2 = bf16_lo(kw.y), b3 = bf16_hi(kw.y);
        float sq = warp_sum(a0 * a0 + a1 * a1 + a2 * a2 + a3 * a3);
        float sk = warp_sum(b0 * b0 + b1 * b1 + b2 * b2 + b3 * b3);
        float sqk = warp_sum(a0 * b0 + a1 * b1 + a2 * b2 + a3 * b3);
        if (lane == 0) {
            const float rq = p.scale * rsqrtf(sq + L2_EPS), rk = rsqrtf(sk + L2_EPS);
            s.rq[r] = rq;
            s.rk[r] = rk;
            s.qk[r] = sqk * rq * rk;
        }
    }
    __syncthreads();

    // Accumulators: this warp's 5 of the 40 (pair, {A,P}, n8-half) tiles.
    float acc[5][4];
#pragma unroll
    for (int u = 0; u < 5; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[u][e] = 0.f;

    for (int sl = 0; sl < KD / SL; ++sl) {
        const int c0 = sl * SL;
        // ---- 3a. gate in log2 units
        for (int idx = tid; idx < CH * SL; idx += IN_THREADS) {
            const int r = idx / SL, c = idx % SL;
            float g2 = 0.f;
            if (r < len) g2 = -a_gate * softplus_log2(bf16_to_f(s.u.raw.g[r][c0 + c]));
            s.G[r][c] = g2;
        }
        __syncthreads();
        // ---- 3b. in-chunk inclusive prefix sum per channel
        {
            const int cc = warp * 4 + (lane >> 3), seg = lane & 7;
            float run = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                run += s.G[seg * 8 + j][cc];
                s.G[seg * 8 + j][cc] = run;
            }
            float incl = run;
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o, 8);
                if (seg >= o) incl += y;
            }
            const float excl = incl - run;
#pragma unroll
            for (int j = 0; j < 8; ++j) s.G[seg * 8 + j][cc] += excl;
        }
        __syncthreads();
        // ---- 3c. per-channel references
        if (tid < SL) {
            const int c = tid;
            float m[5];
            m[0] = 0.f;
            m[1] = s.G[15][c];
            m[2] = s.G[31][c];
            m[3] = s.G[47][c];
            m[4] = s.G[63][c];
#pragma unroll
            for (int i = 0; i < 5; ++i) s.ref[R_M + i][c] = m[i];
#pragma unroll
            for (int i = 0; i < 4; ++i) s.ref[R_MU + i][c] = 0.5f * (s.G[16 * i][c] + s.G[16 * i + 15][c]);
            s.ref[R_X + 0][c] = ex2(m[2] - m[1]);
            s.ref[R_X + 1][c] = ex2(m[3] - m[2]);
            s.ref[R_X + 2][c] = ex2(m[3] - m[1]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                s.ref[R_EB + i][c] = ex2(m[i]);
                s.ref[R_EA + i][c] = ex2(m[4] - m[i + 1]);
            }
            *reinterpret_cast<float *>(rec + REC_GC + 4 * (c0 + c)) = ex2(m[4]);
        }
        __syncthreads();
        // ---- 3d. gated operands
        for (int idx = tid; idx < CH * SL; idx += IN_THREADS) {
            const int r = idx / SL, c = idx % SL, bl = r >> 4;
            const float G = s.G[r][c];
            const float mb = s.ref[R_M + bl][c], mb1 = s.ref[R_M + bl + 1][c], mu = s.ref[R_MU + bl][c];
            const float f = ex2(G - mb);
            const float hh = ex2(mb1 - G);
            const float dr = ex2(fminf(G - mu, DIAG_CLAMP2));
            const float dc = ex2(fminf(mu - G, DIAG_CLAMP2));
            const float kh = bf16_to_f(s.u.raw.k[r][c0 + c]) * s.rk[r];
            const float qt = bf16_to_f(s.u.raw.q[r][c0 + c]) * s.rq[r];
            s.op[OP_FK][r][c] = to_tf32(kh * f);
            s.op[OP_FQ][r][c] = to_tf32(qt * f);
            s.op[OP_HK][r][c] = to_tf32(kh * hh);
            s.op[OP_DRK][r][c] = to_tf32(kh * dr);
            s.op[OP_DRQ][r][c] = to_tf32(qt * dr);
            s.op[OP_DCK][r][c] = to_tf32(kh * dc);
            const float eb = s.ref[R_EB + bl][c], ea = s.ref[R_EA + bl][c];
            s.Kg[r][c0 + c] = to_tf32(kh * f * eb);
            *reinterpret_cast<uint16_t *>(rec + REC_WQ + sw128_off(r, 2 * (c0 + c), 2 * CH)) = f_to_bf16(qt * f * eb);
            *reinterpret_cast<float *>(rec + REC_KDT + sw128_off(c0 + c, 4 * r, KD)) = to_tf32(kh * hh * ea);
        }
        __syncthreads();
        // ---- 3e. partial products over this slice's 32 channels
#pragma unroll
        for (int u = 0; u < 5; ++u) {
            const int tile = warp + 8 * u;          // 0..39
            const int pr = tile >> 2, mat = (tile >> 1) & 1, nt = tile & 1;
            const int bi = c_pair_i[pr], bj = c_pair_b[pr];
            const bool diag = (bi == bj);
            const float(*Aop)[OPS] = s.op[diag ? (mat ? OP_DRQ : OP_DRK) : (mat ? OP_FQ : OP_FK)];
            const float(*Bop)[OPS] = s.op[diag ? OP_DCK : OP_HK];
            // cross factor exp(m_i - m_{b+1}) for pairs two or three blocks apart
            const int xr = (bi == 2 && bj == 0) ? 0 : (bi == 3 && bj == 1) ? 1 : (bi == 3 && bj == 0) ? 2 : -1;
            const int ra = 16 * bi + gq, rb = 16 * bj + 8 * nt + gq;
#pragma unroll
            for (int ks = 0; ks < SL / 8; ++ks) {
                const int ca = 8 * ks + tq;
                float a0 = Aop[ra][ca], a1 = Aop[ra + 8][ca], a2 = Aop[ra][ca + 4], a3 = Aop[ra + 8][ca + 4];
                if (xr >= 0) {
                    const float x0 = s.ref[R_X + xr][ca], x1 = s.ref[R_X + xr][ca + 4];
                    a0 = to_tf32(a0 * x0);
                    a1 = to_tf32(a1 * x0);
                    a2 = to_tf32(a2 * x1);
                    a3 = to_tf32(a3 * x1);
                }
                const uint32_t af[4] = {__float_as_uint(a0), __float_as_uint(a1), __float_as_uint(a2),
                                        __float_as_uint(a3)};
                const uint32_t bf[2] = {__float_as_uint(Bop[rb][ca]), __float_as_uint(Bop[rb][ca + 4])};
                mma_tf32(acc[u], af, bf);
            }
        }
        __syncthreads();
    }

    // ---- 4. finalize A (to smem) and P (to global)
    for (int idx = tid; idx < CH * AS; idx += IN_THREADS) {
        (&s.u.inv.A[0][0])[idx] = 0.f;
        (&s.u.inv.T[0][0])[idx] = 0.f;
    }
    // zero P above the block diagonal
    for (int idx = tid; idx < 6 * SUB * SUB; idx += IN_THREADS) {
        const int blk = idx >> 8, e = idx & 255;
        const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        const int r = 16 * bi + (e >> 4), j = 16 * bj + (e & 15);
        *reinterpret_cast<float *>(rec + REC_P + sw128_off(r, 4 * j, CH)) = 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 5; ++u) {
        const int tile = warp + 8 * u;
        const int pr = tile >> 2, mat = (tile >> 1) & 1, nt = tile & 1;
        const int bi = c_pair_i[pr], bj = c_pair_b[pr];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = 16 * bi + gq + ((e & 2) ? 8 : 0);
            const int j = 16 * bj + 8 * nt + 2 * tq + (e & 1);
            float val = acc[u][e];
            if (mat == 0) {
                val = (j < r) ? val * s.beta[r] : 0.f;
                s.u.inv.A[r][j] = val;
            } else {
                // the decay factor of the j = r term is exactly 1 for any gate
                val = (j < r) ? val : (j == r ? s.qk[r] : 0.f);
                *reinterpret_cast<float *>(rec + REC_P + sw128_off(r, 4 * j, CH)) = to_tf32(val);
            }
        }
    }
    __syncthreads();

    // ---- 5. T = (I + A)^{-1}, blocked forward substitution
    if (tid < 64) {
        const int bi = tid >> 4, c = tid & 15, o = 16 * bi;
        float t[SUB];
#pragma unroll
        for (int r = 0; r < SUB; ++r) {
            float sacc = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < r; ++j) sacc = fmaf(-s.u.inv.A[o + r][o + j], t[j], sacc);
            t[r] = sacc;
        }
#pragma unroll
        for (int r = 0; r < SUB; ++r) s.u.inv.T[o + r][o + c] = t[r];
    }
    __syncthreads();
    // levels: distance 1 (three blocks), 2 (two blocks), 3 (one block)
    for (int dist = 1; dist <= 3; ++dist) {
        const int nblk = 4 - dist;
        // Z_ij = sum_{k=j}^{i-1} A_ik T_kj
        for (int idx = tid; idx < nblk * 256; idx += IN_THREADS) {
            const int bj = idx >> 8, e = idx & 255, bi = bj + dist;
            const int r = e >> 4, c = e & 15;
            float z = 0.f;
            for (int kk = 16 * bj; kk < 16 * bi; ++kk) z = fmaf(s.u.inv.A[16 * bi + r][kk], s.u.inv.T[kk][16 * bj + c], z);
            s.u.inv.Z[bj][r][c] = z;
        }
        __syncthreads();
        // T_ij = -T_ii Z_ij
        for (int idx = tid; idx < nblk * 256; idx += IN_THREADS) {
            const int bj = idx >> 8, e = idx & 255, bi = bj + dist;
            const int r = e >> 4, c = e & 15;
            float tv = 0.f;
            for (int kk = 0; kk <= r; ++kk) tv = fmaf(s.u.inv.T[16 * bi + r][16 * bi + kk], s.u.inv.Z[bj][kk][c], tv);
            s.u.inv.T[16 * bi + r][16 * bj + c] = -tv;
        }
        __syncthreads();
    }
    // T' = T diag(beta), tf32
    for (int idx = tid; idx < CH * CH; idx += IN_THREADS) {
        const int r = idx >> 6, j = idx & 63;
        s.u.inv.T[r][j] = to_tf32(s.u.inv.T[r][j] * s.beta[j]);
    }
    __syncthreads();

    // ---- 6. [W | U] = T' [Kg | V]   (64 x 256, K = 64, T' block lower triangular)
    {
        const int mi = warp & 3, nh = warp >> 2;
        float o[16][4];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
        const int ra = 16 * mi + gq;
        for (int ks = 0; ks < 2 * (mi + 1); ++ks) {
            const int ca = 8 * ks + tq;
            const uint32_t af[4] = {__float_as_uint(s.u.inv.T[ra][ca]), __float_as_uint(s.u.inv.T[ra + 8][ca]),
                                    __float_as_uint(s.u.inv.T[ra][ca + 4]),
                                    __float_as_uint(s.u.inv.T[ra + 8][ca + 4])};
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const int n = 8 * nt + gq;
                uint32_t bf[2];
                if (nh == 0) {
                    bf[0] = __float_as_uint(s.Kg[ca][n]);
                    bf[1] = __float_as_uint(s.Kg[ca + 4][n]);
                } else {
                    bf[0] = __float_as_uint(bf16_to_f(s.v[ca][n]));
                    bf[1] = __float_as_uint(bf16_to_f(s.v[ca + 4][n]));
                }
                mma_tf32(o[nt], af, bf);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int c = 8 * nt + 2 * tq;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int r = ra + 8 * hf;
                if (nh == 0) {
                    *reinterpret_cast<uint32_t *>(rec + REC_WQ + sw128_off(CH + r, 2 * c, 2 * CH)) =
                        pack_bf16x2(o[nt][2 * hf], o[nt][2 * hf + 1]);
                } else {
                    *reinterpret_cast<float2 *>(rec + REC_U + (c >> 6) * 16384 + (r * 64 + (c & 63)) * 4) =
                        make_float2(o[nt][2 * hf], o[nt][2 * hf + 1]);
                }
            }
        }
    }
}

// =====================================================================
// Inter-chunk scan on tcgen05: one CTA (4 warps) per (sequence, value head,
// 64-row V block).  The state block S^T (k = TMEM lane / thread, 64 v) lives in
// registers in fp32; per chunk:
//   MMA1 (bf16)  Y[128 x 64]  = [Qg; W] S^T            (A: WQ image, B: S in bf16)
//   Delta = U - Y[64..127]                              (threads 64..127, fp32 -> tf32)
//   MMA3 (tf32)  Z[128 x 64]  = Kd^T Delta               (state update, k x v)
//   MMA2 (tf32)  Y[0..63]    += P Delta                  (A = [P; 0], so rows 64.. untouched)
//   S = S * exp(Gam_C) + Z ;  O = Y[0..63] -> out (bf16)
// Thread 0 issues the MMAs and the bulk copies of the next chunk's record
// parts as soon as the buffer they overwrite has been consumed.  Every wait is
// bounded; on a timeout the CTA records KDA_ERR_DEVICE_TIMEOUT and stops.
// =====================================================================
constexpr int SC_THREADS = 128;
constexpr int VB = 64;   // state rows (v) per CTA

constexpr uint32_t SS_WQ = 0;          // 32 KiB  A of MMA1: 128 rows x 128 bf16
constexpr uint32_t SS_PP = 32768;      // 32 KiB  A of MMA2: 128 rows x 64 tf32, rows 64..127 zero
constexpr uint32_t SS_KDT = 65536;     // 32 KiB  A of MMA3: 128 rows x 64 tf32
constexpr uint32_t SS_SB = 98304;      // 16 KiB  B of MMA1: 64 rows (v) x 128 bf16 (k)
constexpr uint32_t SS_DT = 114688;     // 16 KiB  B of MMA2/3: 64 rows (v) x 64 tf32 (r)
constexpr uint32_t SS_U = 131072;      // 16 KiB  U block, fp32 [64 r][64 v]
constexpr uint32_t SS_GC = 147456;     // 512 B
constexpr uint32_t SS_BAR = 147968;    // 6 mbarriers
constexpr uint32_t SS_SLOT = 148032;   // TMEM address slot
constexpr uint32_t SS_FLAG = 148036;   // abort flag
constexpr uint32_t SS_BYTES = 148096 + 1024;   // + alignment slack

struct ScanParams {
    const unsigned char *rec;
    const SeqDesc *seqs;
    const int *order;
    const int *hdr;
    const float *init;
    float *fin;
    uint16_t *out;
    int H_v, nseq;
};

enum { BAR_WQ = 0, BAR_PK, BAR_U, BAR_MMA1, BAR_MMA3, BAR_MMA2 };

__global__ __launch_bounds__(SC_THREADS, 1) void scan_kernel(const ScanParams p) {
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled operand atoms
    unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    if (p.hdr[1] == 0) return;
    const int vb = blockIdx.x & 1;
    const int h = (blockIdx.x >> 1) % p.H_v;
    const int rank = (blockIdx.x >> 1) / p.H_v;
    if (rank >= p.nseq) return;
    const int seq = p.order[rank];
    const SeqDesc sd = p.seqs[seq];
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar = sbase + SS_BAR;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SS_FLAG);

    // zero rows 64..127 of the P operand (both K atoms); they are never rewritten
    for (int i = tid; i < 2 * 8192 / 16; i += SC_THREADS) {
        const int atom = i / 512, o = (i % 512) * 16;
        *reinterpret_cast<uint4 *>(sm + SS_PP + atom * 16384 + 8192 + o) = make_uint4(0, 0, 0, 0);
    }
    if (tid == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(bar + 8 * i, 1);
        mbar_fence_init();
        *abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(sbase + SS_SLOT, 128);
    // state block: thread k holds S[v][k] for the 64 v of this block
    float S[VB];
    const size_t st0 = (((size_t)seq * p.H_v + h) * KD + (size_t)vb * VB) * KD + tid;
#pragma unroll
    for (int v = 0; v < VB; ++v) S[v] = p.init ? p.init[st0 + (size_t)v * KD] : 0.f;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + SS_SLOT);
    const uint32_t tY = tmem, tZ = tmem + 64;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

    auto rec_of = [&](int c) { return p.rec + (((size_t)sd.chunk0 + c) * p.H_v + h) * REC_BYTES; };
    auto issue_wq = [&](int c) {
        mbar_expect_tx(bar + 8 * BAR_WQ, 32768);
        bulk_g2s(sbase + SS_WQ, rec_of(c) + REC_WQ, 32768, bar + 8 * BAR_WQ);
    };
    auto issue_pk = [&](int c) {
        const unsigned char *r = rec_of(c);
        mbar_expect_tx(bar + 8 * BAR_PK, 8192 * 2 + 32768);
        bulk_g2s(sbase + SS_PP, r + REC_P, 8192, bar + 8 * BAR_PK);
        bulk_g2s(sbase + SS_PP + 16384, r + REC_P + 8192, 8192, bar + 8 * BAR_PK);
        bulk_g2s(sbase + SS_KDT, r + REC_KDT, 32768, bar + 8 * BAR_PK);
    };
    auto issue_u = [&](int c) {
        const unsigned char *r = rec_of(c);
        mbar_expect_tx(bar + 8 * BAR_U, 16384 + 512);
        bulk_g2s(sbase + SS_U, r + REC_U + vb * 16384, 16384, bar + 8 * BAR_U);
        bulk_g2s(sbase + SS_GC, r + REC_GC, 512, bar + 8 * BAR_U);
    };
    // outstanding copy phases per barrier (for the bounded drain on abort)
    int pend_wq = 0, pend_pk = 0, pend_u = 0;
    if (tid == 0 && sd.nchunk > 0) {
        issue_wq(0);
        issue_pk(0);
        issue_u(0);
    }
    pend_wq = pend_pk = pend_u = (sd.nchunk > 0);

    const uint32_t id_b = idesc_bf16(128, VB), id_t = idesc_tf32(128, VB);
    int c = 0;
    for (; c < sd.nchunk; ++c) {
        const uint32_t ph = c & 1;
        const bool has_next = c + 1 < sd.nchunk;
        const int len = min(CH, sd.len - c * CH);
        const int tok0 = sd.tok + c * CH;
        // ---- S (bf16) -> SB:  element (v, k) of the B operand
#pragma unroll
        for (int v = 0; v < VB; ++v)
            *reinterpret_cast<uint16_t *>(sm + SS_SB + sw128_off(v, 2 * tid, VB)) = f_to_bf16(S[v]);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- MMA1
        if (tid == 0) {
            if (!mbar_wait(bar + 8 * BAR_WQ, ph)) {
                set_status(KDA_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            } else {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < KD / 16; ++ks) {
                    const int kb = ks * 32;
                    const uint64_t ad = umma_desc(sbase + SS_WQ + (kb >> 7) * 16384 + (kb & 127), 16, 1024);
                    const uint64_t bd = umma_desc(sbase + SS_SB + (kb >> 7) * 8192 + (kb & 127), 16, 1024);
                    umma_bf16(tY, ad, bd, id_b, ks > 0);
                }
                umma_commit(bar + 8 * BAR_MMA1);
            }
            pend_wq = 0;
        }
        __syncthreads();
        if (*abort_flag) break;
        const bool ok1 = mbar_wait(bar + 8 * BAR_MMA1, ph);
        const bool oku = mbar_wait(bar + 8 * BAR_U, ph);
        if (!ok1 || !oku) {
            set_status(KDA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
        tc_fence_after();
        if (tid == 0 && has_next && ok1) {
            issue_wq(c + 1);
            pend_wq = 1;
        }
        const float g = reinterpret_cast<const float *>(sm + SS_GC)[tid];
        // ---- Delta = U - W S^T (rows r = tid - 64), written as B operand (v, r)
        if (warp >= 2 && ok1 && oku) {
            const int r = tid - 64;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float y[32];
                tmem_ld32(tY + lane_off + half * 32, y);
                const float *urow = reinterpret_cast<const float *>(sm + SS_U) + r * 64 + half * 32;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int v = half * 32 + j;
                    *reinterpret_cast<float *>(sm + SS_DT + sw128_off(v, 4 * r, VB)) = to_tf32(urow[j] - y[j]);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (*abort_flag) break;
        if (tid == 0) {
            pend_u = 0;
            if (has_next) {
                issue_u(c + 1);
                pend_u = 1;
            }
            // ---- MMA3 (state update) then MMA2 (output correction)
            if (!mbar_wait(bar + 8 * BAR_PK, ph)) {
                set_status(KDA_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            } else {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < CH / 8; ++ks) {
                    const int kb = ks * 32;
                    const uint64_t ad = umma_desc(sbase + SS_KDT + (kb >> 7) * 16384 + (kb & 127), 16, 1024);
                    const uint64_t bd = umma_desc(sbase + SS_DT + (kb >> 7) * 8192 + (kb & 127), 16, 1024);
                    umma_tf32(tZ, ad, bd, id_t, ks > 0);
                }
                umma_commit(bar + 8 * BAR_MMA3);
#pragma unroll
                for (int ks = 0; ks < CH / 8; ++ks) {
                    const int kb = ks * 32;
                    const uint64_t ad = umma_desc(sbase + SS_PP + (kb >> 7) * 16384 + (kb & 127), 16, 1024);
                    const uint64_t bd = umma_desc(sbase + SS_DT + (kb >> 7) * 8192 + (kb & 127), 16, 1024);
                    umma_tf32(tY, ad, bd, id_t, 1);
                }
                umma_commit(bar + 8 * BAR_MMA2);
            }
            pend_pk = 0;
        }
        __syncthreads();
        if (*abort_flag) break;
        const bool ok3 = mbar_wait(bar + 8 * BAR_MMA3, ph);
        const bool ok2 = mbar_wait(bar + 8 * BAR_MMA2, ph);
        if (!ok3 || !ok2) {
            set_status(KDA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
        tc_fence_after();
        if (ok3 && ok2) {
            // ---- S = S * exp(Gam_C) + Z
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float z[32];
                tmem_ld32(tZ + lane_off + half * 32, z);
#pragma unroll
                for (int j = 0; j < 32; ++j) S[half * 32 + j] = fmaf(S[half * 32 + j], g, z[j]);
            }
            // ---- output rows r = tid (warps 0, 1)
            if (warp < 2) {
                const int r = tid;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float y[32];
                    tmem_ld32(tY + lane_off + half * 32, y);
                    if (r < len) {
                        uint16_t *dst = p.out + ((size_t)(tok0 + r) * p.H_v + h) * KD + vb * VB + half * 32;
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
                            uint4 w;
                            w.x = pack_bf16x2(y[j], y[j + 1]);
                            w.y = pack_bf16x2(y[j + 2], y[j + 3]);
                            w.z = pack_bf16x2(y[j + 4], y[j + 5]);
                            w.w = pack_bf16x2(y[j + 6], y[j + 7]);
                            *reinterpret_cast<uint4 *>(dst + j) = w;
                        }
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (*abort_flag) break;
        if (tid == 0 && has_next) {
            issue_pk(c + 1);
            pend_pk = 1;
        }
    }
    // ---- drain: on abort, wait (bounded) for copies still in flight
    if (tid == 0 && c < sd.nchunk) {
        // copies issued for chunk c (parity c & 1) or c + 1 (the other parity)
        for (uint32_t ph = 0; ph < 2; ++ph) {
            if (pend_wq) mbar_wait(bar + 8 * BAR_WQ, ph, 1u << 16);
            if (pend_pk) mbar_wait(bar + 8 * BAR_PK, ph, 1u << 16);
            if (pend_u) mbar_wait(bar + 8 * BAR_U, ph, 1u << 16);
            mbar_wait(bar + 8 * BAR_MMA1, ph, 1u << 16);
            mbar_wait(bar + 8 * BAR_MMA3, ph, 1u << 16);
            mbar_wait(bar + 8 * BAR_MMA2, ph, 1u << 16);
        }
    }
    if (p.fin && !*abort_flag) {
        float *dst = p.fin + st0;
#pragma unroll
        for (int v = 0; v < VB; ++v) dst[(size_t)v * KD] = S[v];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// =====================================================================
// Host-side launch of the three kernels.
// =====================================================================
struct FwdWorkspace {
    int *hdr;
    SeqDesc *seqs;
    ChunkDesc *chunks;
    int *order;
    unsigned char *rec;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

long long max_chunks_for(int N, int B, int T, bool varlen) {
    if (varlen) return (long long)T / CH + (long long)N + 1;
    return (long long)B * ((T + CH - 1) / CH);
}

size_t fwd_workspace_bytes(int N, int B, int T, int H_v, bool varlen, FwdWorkspace *ws, char *base) {
    const long long nseq = varlen ? N : B;
    const long long nck = max_chunks_for(N, B, T, varlen);
    const long long nch = nck * H_v;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align256(off + bytes);
        return base ? (void *)(base + o) : nullptr;
    };
    FwdWorkspace w;
    w.hdr = (int *)take(256);
    w.seqs = (SeqDesc *)take(sizeof(SeqDesc) * (size_t)(nseq > 0 ? nseq : 1));
    w.chunks = (ChunkDesc *)take(sizeof(ChunkDesc) * (size_t)(nck > 0 ? nck : 1));
    w.order = (int *)take(sizeof(int) * (size_t)(nseq > 0 ? nseq : 1));
    w.rec = (unsigned char *)take((size_t)nch * REC_BYTES);
    if (ws) *ws = w;
    return off;
}

cudaError_t launch_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                       const uint16_t *b, const float *A_log, float scale, const float *init, float *fin,
                       const int32_t *cu, int N, int B, int T, int H_qk, int H_v, uint16_t *out, void *ws_ptr,
                       cudaStream_t stream, int *launches) {
    const bool varlen = cu != nullptr;
    const int nseq = varlen ? N : B;
    FwdWorkspace ws;
    fwd_workspace_bytes(N, B, T, H_v, varlen, &ws, (char *)ws_ptr);
    const long long nck = max_chunks_for(N, B, T, varlen);
    *launches = 0;
    {
        cudaError_t e = cudaFuncSetAttribute(intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(IntraSmem));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SS_BYTES);
        if (e != cudaSuccess) return e;
    }
    plan_kernel<<<1, PLAN_THREADS, 0, stream>>>(cu, N, B, T, ws.seqs, ws.chunks, ws.order, ws.hdr, nck);
    ++*launches;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (nck > 0) {
        IntraParams ip;
        ip.q = q; ip.k = k; ip.v = v; ip.graw = graw; ip.b = b; ip.A_log = A_log; ip.scale = scale;
        ip.H_qk = H_qk; ip.H_v = H_v; ip.chunks = ws.chunks; ip.hdr = ws.hdr;
        ip.rec = ws.rec;
        intra_kernel<<<dim3((unsigned)nck, (unsigned)H_v), IN_THREADS, sizeof(IntraSmem), stream>>>(ip);
        ++*launches;
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (nseq > 0) {
        ScanParams sp;
        sp.rec = ws.rec;
        sp.seqs = ws.seqs; sp.order = ws.order; sp.hdr = ws.hdr;
        sp.init = init; sp.fin = fin; sp.out = out; sp.H_v = H_v; sp.nseq = nseq;
        const long long nblk = (long long)nseq * H_v * 2;
        scan_kernel<<<(unsigned)nblk, SC_THREADS, SS_BYTES, stream>>>(sp);
        ++*launches;
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kda
