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

// Per (chunk, value head) record written by the intra-chunk kernel and read
// by the scan with bulk copies.  The operands are stored as the exact shared
// memory images the scan's tcgen05.mma reads (K-major, 128-byte swizzle):
//   WQ  [Qg rows 0..63 ; W rows 64..127] x K=128, bf16          (32 KiB)
//   P   rows r = 0..63 x 64 (j), bf16                            (8 KiB)
//   KDT Kd^T: rows k = 0..127 x 64 (r), tf32                      (32 KiB)
//   U   [V block 0 | V block 1], each [64 v][68] fp32 (64 r + 4 pad)  (34 KiB)
//   GC  exp(Gam_C) per channel, fp32                              (512 B)
constexpr uint32_t REC_WQ = 0, REC_P = 32768, REC_KDT = 40960, REC_U = 73728, REC_GC = 108544;
constexpr uint32_t REC_U_BLOCK = 64 * 68 * 4;   // 17408 B per V block
constexpr uint32_t REC_BYTES = 109056;

// =====================================================================
// Intra-chunk kernel: persistent CTAs (16 warps), each looping over
// (chunk, value head) work items.
//
// Fuses the per-token pre-processing (L2 norms, beta sigmoid, gate
// activation, in-chunk prefix sum of the gate) with the UT/WY factorisation
// of the chunk and writes the chunk's record for the scan.
//
// Decay products exp(Gam_r - Gam_j) for the 64 x 64 matrices A and P are
// built from 16-row sub-blocks.  Row r of sub-block i carries the factor
// f_r = exp(Gam_r - m_i) (m_i = Gam at the end of sub-block i-1, so f <= 1);
// column j of sub-block b carries h_j = exp(m_{b+1} - Gam_j) (<= 1); a pair of
// sub-blocks i > b + 1 also needs the block decays between them,
// X = exp(m_i - m_{b+1}) = prod D, which is folded into per-pair versions of
// the column operand.  Diagonal sub-blocks use the per-channel midpoint mu of
// the block's first and last Gam (exponents clamped at 85 nats).  Per 32-channel
// slice, two tcgen05 MMAs (tf32, M = 128) accumulate
//   D_off [128 x 96] = [F_k ; F_q] . [H versions]^T     (all below-diagonal blocks)
//   D_diag[128 x 64] = [R_k ; R_q] . [C_k]^T            (the four diagonal blocks)
// into TMEM; rows 0..63 give A (times beta_r), rows 64..127 give P.  After the
// blocked inversion T = (I + A)^{-1}, one bf16 MMA chain gives
//   [W | U] = (T'_hi + T'_lo) [Kg | V],   T' = T diag(beta) split into two bf16 terms,
// with [Kg | V] an MN-major operand: V rows are copied straight from global
// memory and Kg (the gated key) is written in bf16.
// =====================================================================
constexpr int IN_THREADS = 512;
constexpr int SL = 32;                  // channels per slice (one 128-byte tf32 atom)
constexpr int RAWS = 136;               // raw row stride in bf16 (272 B)
constexpr int GAS = 132;                // Gam row stride (floats), all 128 channels
constexpr int AS = CH + 4;              // A / T row stride (floats)
constexpr int ZS = 20;                  // inversion scratch row stride (floats)

constexpr uint32_t IS_Q = 0;            // raw q, k, graw: [64][136] bf16 each
constexpr uint32_t IS_K = 17408;
constexpr uint32_t IS_G = 34816;
constexpr uint32_t IS_KV = 53248;       // B of the W/U MMA: [Kg | V] MN-major bf16, N = 256, K = 64 (32 KiB)
constexpr uint32_t IS_ROWS = 86016;     // 256 rows x 32 ch tf32: F_k, F_q, R_k, R_q
constexpr uint32_t IS_COLS = 118784;    // 160 rows x 32 ch tf32: C_k (64), H versions (96)
constexpr uint32_t IS_GA = 139264;      // Gam, fp32 [64][132] (log2 units)
constexpr uint32_t IS_TAB = 173056;     // per-channel tables [20][128] fp32
constexpr uint32_t IS_KDS = 183296;     // Kd^T slice staging, 2 x 4 KiB
constexpr uint32_t IS_RV = 191488;      // rq, rk, beta, qk [4][64] fp32
constexpr uint32_t IS_SEG = 192512;     // prefix-sum segment totals [4][128]
constexpr uint32_t IS_GCS = 194560;     // exp(Gam_C) staging [128]
constexpr uint32_t IS_BAR = 195072;     // 2 mbarriers
constexpr uint32_t IS_SLOT = 195096;    // TMEM address
constexpr uint32_t IS_BYTES = 195104 + 1024;
// aliases once the slices are done
constexpr uint32_t IS_A = 0;            // fp32 [64][68]
constexpr uint32_t IS_T = 17408;        // fp32 [64][68]
constexpr uint32_t IS_Z = 34816;        // fp32 [3][16][20]
constexpr uint32_t IS_TPH = IS_ROWS;    // A of the W/U MMA: T'_hi, 64 rows (r) x 64 (j) bf16 (8 KiB)
constexpr uint32_t IS_TPL = IS_ROWS + 8192;    // T'_lo
constexpr uint32_t IS_PI = IS_ROWS + 16384;    // P image staging (bf16, 8 KiB)
constexpr uint32_t IS_WS = IS_COLS;     // W half of the WQ image (2 x 8 KiB)
constexpr uint32_t IS_US = IS_GA;       // U image staging (2 x 64 x 68 fp32)

enum { TB_MU = 0, TB_M = 4, TB_EB = 9, TB_EA = 13, TB_D1 = 17, TB_D2 = 18, TB_D12 = 19 };
enum { RV_RQ = 0, RV_RK = 64, RV_BETA = 128, RV_QK = 192 };

struct IntraParams {
    const uint16_t *q, *k, *v, *graw, *b;
    const float *A_log;
    float scale;
    int H_qk, H_v;
    const ChunkDesc *chunks;
    const int *hdr;
    unsigned char *rec;   // [chunk][H_v] records of REC_BYTES
};

__device__ __forceinline__ void sts128(unsigned char *p, float a, float b, float c, float d) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(tf32_bits(a), tf32_bits(b), tf32_bits(c), tf32_bits(d));
}
// byte offset of element (n, kk) in an MN-major bf16 operand with 64-element
// atoms along N (stride 8 KiB) and 8-row K groups (stride 1 KiB)
__device__ __forceinline__ uint32_t mn_off_bf16(int n, int kk) {
    return (uint32_t)((n >> 6) * 8192 + (kk >> 3) * 1024 + (kk & 7) * 128 + ((((n & 63) >> 3) ^ (kk & 7)) << 4) +
                      ((n & 7) << 1));
}

// Four warps (wq = 0..3 of the group): Z (16 x 16) = sum over kk in [k0, k1) of X[r][kk] Y[kk][c];
// warp wq computes rows 4 wq .. 4 wq + 3, lane = (row, column pair).
__device__ __forceinline__ void quad_mm16(const float *X, int xs, const float *Y, int ys, int k0, int k1,
                                          float (&acc)[2], int wq, int lane) {
    const int r = 4 * wq + (lane >> 3), c = (lane & 7) * 2;
    for (int kb = k0; kb < k1; kb += 16) {   // k1 - k0 is a multiple of 16
#pragma unroll
        for (int kk = kb; kk < kb + 16; ++kk) {
            const float a = X[r * xs + kk];
            const float2 y = *reinterpret_cast<const float2 *>(Y + kk * ys + c);
            acc[0] = fmaf(a, y.x, acc[0]);
            acc[1] = fmaf(a, y.y, acc[1]);
        }
    }
}

__global__ __launch_bounds__(IN_THREADS, 1) void intra_kernel(const IntraParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    if (p.hdr[1] == 0) return;
    const long long n_items = (long long)p.hdr[0] * p.H_v;
    if ((long long)blockIdx.x >= n_items) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar_ap = sbase + IS_BAR, bar_wu = sbase + IS_BAR + 8;
    const uint64_t pol_ef = l2_evict_first_policy();
    float *rv = reinterpret_cast<float *>(sm + IS_RV);
    float *tab = reinterpret_cast<float *>(sm + IS_TAB);
    float *ga = reinterpret_cast<float *>(sm + IS_GA);
    float *sA = reinterpret_cast<float *>(sm + IS_A);
    float *sT = reinterpret_cast<float *>(sm + IS_T);
    float *sZ = reinterpret_cast<float *>(sm + IS_Z);
    if (tid == 0) {
        mbar_init(bar_ap, 1);
        mbar_init(bar_wu, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(sbase + IS_SLOT, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + IS_SLOT);
    const uint32_t t_off = tmem, t_diag = tmem + 96, t_wu = tmem;

    int it = 0;
    for (long long item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
        const int chunk = (int)(item / p.H_v), h = (int)(item % p.H_v);
        const ChunkDesc cd = p.chunks[chunk];
        const int hq = h / (p.H_v / p.H_qk);
        const size_t ch = (size_t)chunk * p.H_v + h;
        unsigned char *rec = p.rec + ch * REC_BYTES;
        const int len = cd.len;
        const float a_gate = ex2(p.A_log[h] * LOG2E);

        // ---- 0. the previous item's bulk stores must be done reading shared memory
        if (tid == 0) bulk_wait_read_all();
        __syncthreads();

        // beta's global load goes first so its latency overlaps the copies below
        float bb_raw = 0.f;
        if (tid < len) bb_raw = bf16_to_f(p.b[((size_t)cd.tok + tid) * p.H_v + h]);
        // ---- 1. stage raw q, k, graw rows and the V part of [Kg | V] (cp.async; V lands in
        //         the swizzled MN-major operand), zero-filling padded rows
        for (int idx = tid; idx < CH * (KD / 8); idx += IN_THREADS) {
            const int r = idx >> 4, c8 = (idx & 15) * 8;
            unsigned char *dq = sm + IS_Q + (r * RAWS + c8) * 2;
            unsigned char *dk = sm + IS_K + (r * RAWS + c8) * 2;
            unsigned char *dg = sm + IS_G + (r * RAWS + c8) * 2;
            unsigned char *dv = sm + IS_KV + mn_off_bf16(KD + c8, r);
            if (r < len) {
                const size_t tok = (size_t)cd.tok + r;
                cp_async16(dq, p.q + (tok * p.H_qk + hq) * KD + c8);
                cp_async16(dk, p.k + (tok * p.H_qk + hq) * KD + c8);
                cp_async16(dg, p.graw + (tok * p.H_v + h) * KD + c8);
                cp_async16(dv, p.v + (tok * p.H_v + h) * KD + c8);
            } else {
                const uint4 z = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(dq) = z;
                *reinterpret_cast<uint4 *>(dk) = z;
                *reinterpret_cast<uint4 *>(dg) = z;
                *reinterpret_cast<uint4 *>(dv) = z;
            }
        }
        cp_async_commit();
        // pull the next item's rows into L2 while this one is processed
        {
            const long long nitem = item + gridDim.x;
            if (nitem < n_items && tid < 4 * CH) {
                const int nchunk = (int)(nitem / p.H_v), nh = (int)(nitem % p.H_v);
                const ChunkDesc nd = p.chunks[nchunk];
                const int r = tid & 63, which = tid >> 6;
                if (r < nd.len) {
                    const size_t tok = (size_t)nd.tok + r;
                    const int nhq = nh / (p.H_v / p.H_qk);
                    const uint16_t *src = which == 0 ? p.q + (tok * p.H_qk + nhq) * KD
                                        : which == 1 ? p.k + (tok * p.H_qk + nhq) * KD
                                        : which == 2 ? p.graw + (tok * p.H_v + nh) * KD
                                                     : p.v + (tok * p.H_v + nh) * KD;
                    prefetch_l2(src, KD * 2);
                }
            }
        }
        cp_async_wait<0>();
        if (tid < CH) rv[RV_BETA + tid] = tid < len ? 1.0f / (1.0f + ex2(-bb_raw * LOG2E)) : 0.f;
        __syncthreads();

        // ---- 2. row norms: warp w, rows 4w..4w+3
        {
            float sq[4], sk[4], sqk[4];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int r = warp * 4 + rr;
                const uint2 qw = *reinterpret_cast<const uint2 *>(sm + IS_Q + (r * RAWS + 4 * lane) * 2);
                const uint2 kw = *reinterpret_cast<const uint2 *>(sm + IS_K + (r * RAWS + 4 * lane) * 2);
                const float a0 = bf16_lo(qw.x), a1 = bf16_hi(qw.x), a2 = bf16_lo(qw.y), a3 = bf16_hi(qw.y);
                const float b0 = bf16_lo(kw.x), b1 = bf16_hi(kw.x), b2 = bf16_lo(kw.y), b3 = bf16_hi(kw.y);
                sq[rr] = a0 * a0 + a1 * a1 + a2 * a2 + a3 * a3;
                sk[rr] = b0 * b0 + b1 * b1 + b2 * b2 + b3 * b3;
                sqk[rr] = a0 * b0 + a1 * b1 + a2 * b2 + a3 * b3;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    sq[rr] += __shfl_xor_sync(0xffffffffu, sq[rr], o);
                    sk[rr] += __shfl_xor_sync(0xffffffffu, sk[rr], o);
                    sqk[rr] += __shfl_xor_sync(0xffffffffu, sqk[rr], o);
                }
            if (lane < 4) {
                const int r = warp * 4 + lane;
                float a = sq[0], bq = sk[0], c = sqk[0];
#pragma unroll
                for (int rr = 1; rr < 4; ++rr)
                    if (lane == rr) {
                        a = sq[rr];
                        bq = sk[rr];
                        c = sqk[rr];
                    }
                const float rq = p.scale * rsqrtf(a + L2_EPS), rk = rsqrtf(bq + L2_EPS);
                rv[RV_RQ + r] = rq;
                rv[RV_RK + r] = rk;
                rv[RV_QK + r] = c * rq * rk;
            }
        }
        // ---- 3. gate (log2 units) and its in-chunk prefix sum for all 128 channels:
        //         thread = (channel c, 16-row segment)
        {
            const int c = tid & 127, sg = tid >> 7;
            float loc[16], run = 0.f;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const int r = sg * 16 + rr;
                float g2 = 0.f;
                if (r < len) {
                    const uint16_t gb = *reinterpret_cast<const uint16_t *>(sm + IS_G + (r * RAWS + c) * 2);
                    g2 = -a_gate * softplus_log2(bf16_to_f(gb));
                }
                run += g2;
                loc[rr] = run;
            }
            reinterpret_cast<float *>(sm + IS_SEG)[sg * 128 + c] = run;
            __syncthreads();
            float off = 0.f;
            for (int s2 = 0; s2 < sg; ++s2) off += reinterpret_cast<const float *>(sm + IS_SEG)[s2 * 128 + c];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) ga[(sg * 16 + rr) * GAS + c] = loc[rr] + off;
        }
        __syncthreads();
        // ---- 4. per-channel tables: four threads per channel (mu and m; exp(m_i); exp(m_4 - m_{i+1});
        //         block decays and exp(Gam_C))
        {
            const int c = tid & 127, part = tid >> 7;
            const float m1 = ga[15 * GAS + c], m2 = ga[31 * GAS + c], m3 = ga[47 * GAS + c], m4 = ga[63 * GAS + c];
            if (part == 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    tab[(TB_MU + i) * 128 + c] = 0.5f * (ga[(16 * i) * GAS + c] + ga[(16 * i + 15) * GAS + c]);
                tab[(TB_M + 0) * 128 + c] = 0.f;
                tab[(TB_M + 1) * 128 + c] = m1;
                tab[(TB_M + 2) * 128 + c] = m2;
                tab[(TB_M + 3) * 128 + c] = m3;
                tab[(TB_M + 4) * 128 + c] = m4;
            } else if (part == 1) {
                tab[(TB_EB + 0) * 128 + c] = 1.f;
                tab[(TB_EB + 1) * 128 + c] = ex2(m1);
                tab[(TB_EB + 2) * 128 + c] = ex2(m2);
                tab[(TB_EB + 3) * 128 + c] = ex2(m3);
            } else if (part == 2) {
                tab[(TB_EA + 0) * 128 + c] = ex2(m4 - m1);
                tab[(TB_EA + 1) * 128 + c] = ex2(m4 - m2);
                tab[(TB_EA + 2) * 128 + c] = ex2(m4 - m3);
                tab[(TB_EA + 3) * 128 + c] = 1.f;
            } else {
                tab[TB_D1 * 128 + c] = ex2(m2 - m1);
                tab[TB_D2 * 128 + c] = ex2(m3 - m2);
                tab[TB_D12 * 128 + c] = ex2(m3 - m1);
                reinterpret_cast<float *>(sm + IS_GCS)[c] = ex2(m4);
            }
        }
        __syncthreads();

        // ---- 5. channel slices: operands, then the A / P MMAs of the slice
        for (int sl = 0; sl < KD / SL; ++sl) {
            const int c0 = sl * SL;
            if (sl > 0) {
                // the previous slice's MMAs and Kd^T stores must be done with ROWS / COLS / KDS
                if (tid == 0) {
                    bulk_wait_read_all();
                    if (!mbar_wait(bar_ap, (sl - 1) & 1)) set_status(KDA_ERR_DEVICE_TIMEOUT);
                }
                __syncthreads();
                tc_fence_after();
            }
            {
                const int g4 = tid >> 6, r = tid & 63, bi = r >> 4, cl = 4 * g4, c = c0 + cl;
                const float4 G = *reinterpret_cast<const float4 *>(ga + r * GAS + c);
                const float4 MU = *reinterpret_cast<const float4 *>(tab + (TB_MU + bi) * 128 + c);
                const float4 M0 = *reinterpret_cast<const float4 *>(tab + (TB_M + bi) * 128 + c);
                const float4 M1 = *reinterpret_cast<const float4 *>(tab + (TB_M + bi + 1) * 128 + c);
                const float4 EB = *reinterpret_cast<const float4 *>(tab + (TB_EB + bi) * 128 + c);
                const float4 EA = *reinterpret_cast<const float4 *>(tab + (TB_EA + bi) * 128 + c);
                const uint2 qw = *reinterpret_cast<const uint2 *>(sm + IS_Q + (r * RAWS + c) * 2);
                const uint2 kw = *reinterpret_cast<const uint2 *>(sm + IS_K + (r * RAWS + c) * 2);
                const float rq = rv[RV_RQ + r], rk = rv[RV_RK + r];
                const float g[4] = {G.x, G.y, G.z, G.w}, mu[4] = {MU.x, MU.y, MU.z, MU.w};
                const float m0[4] = {M0.x, M0.y, M0.z, M0.w}, m1[4] = {M1.x, M1.y, M1.z, M1.w};
                const float eb[4] = {EB.x, EB.y, EB.z, EB.w}, ea[4] = {EA.x, EA.y, EA.z, EA.w};
                const float kh[4] = {bf16_lo(kw.x) * rk, bf16_hi(kw.x) * rk, bf16_lo(kw.y) * rk, bf16_hi(kw.y) * rk};
                const float qt[4] = {bf16_lo(qw.x) * rq, bf16_hi(qw.x) * rq, bf16_lo(qw.y) * rq, bf16_hi(qw.y) * rq};
                float fk[4], fq[4], dk[4], dq[4], ck[4], hk[4], kd[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float dr = ex2(fminf(g[e] - mu[e], DIAG_CLAMP2));
                    const float dc = ex2(fminf(mu[e] - g[e], DIAG_CLAMP2));
                    // block-relative factors (always <= 1, exact for any gate strength)
                    const float f = ex2(g[e] - m0[e]), hh = ex2(m1[e] - g[e]);
                    fk[e] = kh[e] * f;
                    fq[e] = qt[e] * f;
                    dk[e] = kh[e] * dr;
                    dq[e] = qt[e] * dr;
                    ck[e] = kh[e] * dc;
                    hk[e] = kh[e] * hh;
                    kd[e] = hk[e] * ea[e];
                }
                // Kg (bf16) into the MN-major [Kg | V] operand: element (k = c .. c + 3, j = r)
                *reinterpret_cast<uint2 *>(sm + IS_KV + mn_off_bf16(c, r)) =
                    make_uint2(pack_bf16x2(fk[0] * eb[0], fk[1] * eb[1]), pack_bf16x2(fk[2] * eb[2], fk[3] * eb[3]));
                // Kd^T slice staging: element (k, r)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kl = cl + e, k = c + e;
                    const uint32_t kds = (uint32_t)(r >> 5) * 4096 + (kl >> 3) * 1024 + (kl & 7) * 128 +
                                         (((((4 * r) & 127) >> 4) ^ (k & 7)) << 4) + ((4 * r) & 15);
                    *reinterpret_cast<uint32_t *>(sm + IS_KDS + kds) = tf32_bits(kd[e]);
                }
                const int kb = 16 * g4;
                sts128(sm + IS_ROWS + sw128_off(r, kb, 256), fk[0], fk[1], fk[2], fk[3]);
                sts128(sm + IS_ROWS + sw128_off(64 + r, kb, 256), fq[0], fq[1], fq[2], fq[3]);
                sts128(sm + IS_ROWS + sw128_off(128 + r, kb, 256), dk[0], dk[1], dk[2], dk[3]);
                sts128(sm + IS_ROWS + sw128_off(192 + r, kb, 256), dq[0], dq[1], dq[2], dq[3]);
                sts128(sm + IS_COLS + sw128_off(r, kb, 160), ck[0], ck[1], ck[2], ck[3]);
                const int rl = r & 15;
                if (bi == 0) {
                    const float4 D1 = *reinterpret_cast<const float4 *>(tab + TB_D1 * 128 + c);
                    const float4 D12 = *reinterpret_cast<const float4 *>(tab + TB_D12 * 128 + c);
                    sts128(sm + IS_COLS + sw128_off(64 + rl, kb, 160), hk[0], hk[1], hk[2], hk[3]);
                    sts128(sm + IS_COLS + sw128_off(80 + rl, kb, 160), hk[0] * D1.x, hk[1] * D1.y, hk[2] * D1.z,
                           hk[3] * D1.w);
                    sts128(sm + IS_COLS + sw128_off(112 + rl, kb, 160), hk[0] * D12.x, hk[1] * D12.y,
                           hk[2] * D12.z, hk[3] * D12.w);
                } else if (bi == 1) {
                    const float4 D2 = *reinterpret_cast<const float4 *>(tab + TB_D2 * 128 + c);
                    sts128(sm + IS_COLS + sw128_off(96 + rl, kb, 160), hk[0], hk[1], hk[2], hk[3]);
                    sts128(sm + IS_COLS + sw128_off(128 + rl, kb, 160), hk[0] * D2.x, hk[1] * D2.y, hk[2] * D2.z,
                           hk[3] * D2.w);
                } else if (bi == 2) {
                    sts128(sm + IS_COLS + sw128_off(144 + rl, kb, 160), hk[0], hk[1], hk[2], hk[3]);
                }
                // Qg (bf16) straight into the WQ image rows 0..63
                *reinterpret_cast<uint2 *>(rec + REC_WQ + sw128_off(r, 2 * c, 2 * CH)) =
                    make_uint2(pack_bf16x2(fq[0] * eb[0], fq[1] * eb[1]), pack_bf16x2(fq[2] * eb[2], fq[3] * eb[3]));
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                const uint32_t id_off = idesc_tf32(128, 96), id_diag = idesc_tf32(128, 64);
#pragma unroll
                for (int ks = 0; ks < SL / 8; ++ks) {
                    const uint32_t acc = (sl > 0 || ks > 0) ? 1u : 0u;
                    umma_tf32(t_off, umma_desc(sbase + IS_ROWS + ks * 32, 16, 1024),
                              umma_desc(sbase + IS_COLS + 8192 + ks * 32, 16, 1024), id_off, acc);
                    umma_tf32(t_diag, umma_desc(sbase + IS_ROWS + 16384 + ks * 32, 16, 1024),
                              umma_desc(sbase + IS_COLS + ks * 32, 16, 1024), id_diag, acc);
                }
                umma_commit(bar_ap);
                bulk_s2g_hint(rec + REC_KDT + c0 * 128, sbase + IS_KDS, 4096, pol_ef);
                bulk_s2g_hint(rec + REC_KDT + 16384 + c0 * 128, sbase + IS_KDS + 4096, 4096, pol_ef);
                bulk_commit();
            }
        }
        if (tid == 0 && !mbar_wait(bar_ap, (KD / SL - 1) & 1)) set_status(KDA_ERR_DEVICE_TIMEOUT);
        __syncthreads();
        tc_fence_after();

        // ---- 6. A (times beta) to smem, P image (bf16) to staging.  Warp w: TMEM lanes
        //         32 (w & 3) .. (K rows 0..63, Q rows 64..127), 16-column block cb = w >> 2.
        {
            const int q = warp & 3, cb = warp >> 2;
            const int l = q * 32 + lane, r = l & 63, bi = r >> 4, rl = r & 15, isq = l >> 6;
            const uint32_t lo = (uint32_t)(q * 32) << 16;
            const int bia = 2 * (q & 1), bib = bia + 1;
            // column offsets of the below-diagonal versions of row blocks 1, 2, 3 in D_off
            const int nsa = bia == 0 ? 0 : 16, nsb = bib == 1 ? 0 : 48;
            uint32_t va[16], vb2[16], vd[16];
            tmem_ld16_nowait(t_off + lo + nsa + 16 * (cb < 3 ? cb : 2), va);
            tmem_ld16_nowait(t_off + lo + nsb + 16 * (cb < 3 ? cb : 2), vb2);
            tmem_ld16_nowait(t_diag + lo + 16 * cb, vd);
            tmem_wait_ld();
            float o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float x = 0.f;
                if (cb < bi) x = __uint_as_float(bi == bia ? va[j] : vb2[j]);
                else if (cb == bi) x = (j < rl) ? __uint_as_float(vd[j]) : ((isq && j == rl) ? rv[RV_QK + r] : 0.f);
                o[j] = x;
            }
            if (!isq) {
                const float be = rv[RV_BETA + r];
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4 *>(sA + r * AS + 16 * cb + j) =
                        make_float4(o[j] * be, o[j + 1] * be, o[j + 2] * be, o[j + 3] * be);
            } else {
#pragma unroll
                for (int j = 0; j < 16; j += 8)
                    *reinterpret_cast<uint4 *>(sm + IS_PI + sw128_off(r, 2 * (16 * cb + j), CH)) =
                        make_uint4(pack_bf16x2(o[j], o[j + 1]), pack_bf16x2(o[j + 2], o[j + 3]),
                                   pack_bf16x2(o[j + 4], o[j + 5]), pack_bf16x2(o[j + 6], o[j + 7]));
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            bulk_s2g_hint(rec + REC_P, sbase + IS_PI, 8192, pol_ef);
            bulk_s2g_hint(rec + REC_GC, sbase + IS_GCS, 512, pol_ef);
            bulk_commit();
        }

        // ---- 7. T = (I + A)^{-1}: diagonal 16 x 16 blocks by forward substitution, then
        //         T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj, four warps per block, level by level.
        if (tid < 64) {
            const int bi = tid >> 4, c = tid & 15, o = 16 * bi;
            float t[SUB];
#pragma unroll
            for (int r = 0; r < SUB; ++r) {
                float sacc = (r == c) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < r; ++j) sacc = fmaf(-sA[(o + r) * AS + o + j], t[j], sacc);
                t[r] = sacc;
            }
#pragma unroll
            for (int r = 0; r < SUB; ++r) sT[(o + r) * AS + o + c] = t[r];
        } else {
            for (int idx = tid - 64; idx < 6 * 256; idx += IN_THREADS - 64) {
                const int blk = idx >> 8, e = idx & 255;
                const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
                const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                sT[(16 * bi + (e >> 4)) * AS + 16 * bj + (e & 15)] = 0.f;
            }
        }
        __syncthreads();
        for (int dist = 1; dist <= 3; ++dist) {
            const int nblk = 4 - dist, grp = warp >> 2, wq = warp & 3;
            const int r = 4 * wq + (lane >> 3), cc = (lane & 7) * 2;
            if (grp < nblk) {
                const int bj = grp, bi = bj + dist;
                float acc[2] = {0.f, 0.f};
                quad_mm16(sA + (16 * bi) * AS, AS, sT + 16 * bj, AS, 16 * bj, 16 * bi, acc, wq, lane);
                float *z = sZ + grp * 16 * ZS;
                *reinterpret_cast<float2 *>(z + r * ZS + cc) = make_float2(acc[0], acc[1]);
            }
            __syncthreads();
            if (grp < nblk) {
                const int bj = grp, bi = bj + dist;
                float t2[2] = {0.f, 0.f};
                // T_ii is lower triangular (zeros above its diagonal), so the full 16 terms are exact
                quad_mm16(sT + (16 * bi) * AS + 16 * bi, AS, sZ + grp * 16 * ZS, ZS, 0, 16, t2, wq, lane);
                *reinterpret_cast<float2 *>(sT + (16 * bi + r) * AS + 16 * bj + cc) = make_float2(-t2[0], -t2[1]);
            }
            __syncthreads();
        }
        // T' = T diag(beta), split into bf16 hi + lo, as the A operand (K-major, 64 r x 64 j)
        for (int idx = tid; idx < CH * (CH / 8); idx += IN_THREADS) {
            const int r = idx >> 3, j = (idx & 7) * 8;
            float x[8];
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = sT[r * AS + j + e] * rv[RV_BETA + j + e];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const uint32_t h2 = pack_bf16x2(x[e], x[e + 1]);
                hi[e >> 1] = h2;
                lo[e >> 1] = pack_bf16x2(x[e] - bf16_lo(h2), x[e + 1] - bf16_hi(h2));
            }
            *reinterpret_cast<uint4 *>(sm + IS_TPH + sw128_off(r, 2 * j, CH)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(sm + IS_TPL + sw128_off(r, 2 * j, CH)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 8. [W | U] = T'_hi [Kg | V] + T'_lo [Kg | V]   (M = 64, N = 256, K = 64, bf16)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(64, 256) | (1u << 16);   // B MN-major
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < CH / 16; ++ks)
                    umma_bf16(t_wu, umma_desc(sbase + (part ? IS_TPL : IS_TPH) + ks * 32, 16, 1024),
                              umma_desc(sbase + IS_KV + ks * 2048, 8192, 1024), id, (part > 0 || ks > 0) ? 1u : 0u);
            umma_commit(bar_wu);
            if (!mbar_wait(bar_wu, it & 1)) set_status(KDA_ERR_DEVICE_TIMEOUT);
        }
        __syncthreads();
        tc_fence_after();
        {
            // M = 64 layout: row r = 16 (w & 3) + lane for lane < 16; warp w >> 2 selects 64 columns
            const int q = warp & 3, cb = warp >> 2, r = q * 16 + lane;
            const uint32_t lo = (uint32_t)(q * 32) << 16;
            uint32_t x0[32], x1[32];
            tmem_ld32_nowait(t_wu + lo + 64 * cb, x0);
            tmem_ld32_nowait(t_wu + lo + 64 * cb + 32, x1);
            tmem_wait_ld();
            if (lane < 16) {
                if (cb < 2) {
                    // W[r][k], k = 64 cb .. : row 64 + r of the WQ image (bf16)
#pragma unroll
                    for (int j = 0; j < 64; j += 8) {
                        const uint32_t *xs = j < 32 ? x0 : x1;
                        const int jj = j & 31, k = 64 * cb + j;
                        const uint32_t off = (uint32_t)cb * 8192 + (r >> 3) * 1024 + (r & 7) * 128 +
                                             ((((2 * k) & 127) >> 4) ^ (r & 7)) * 16;
                        *reinterpret_cast<uint4 *>(sm + IS_WS + off) = make_uint4(
                            pack_bf16x2(__uint_as_float(xs[jj]), __uint_as_float(xs[jj + 1])),
                            pack_bf16x2(__uint_as_float(xs[jj + 2]), __uint_as_float(xs[jj + 3])),
                            pack_bf16x2(__uint_as_float(xs[jj + 4]), __uint_as_float(xs[jj + 5])),
                            pack_bf16x2(__uint_as_float(xs[jj + 6]), __uint_as_float(xs[jj + 7])));
                    }
                } else {
                    // U[r][v], v = 64 (cb - 2) .. : U image block cb - 2, row v, column r
                    float *us = reinterpret_cast<float *>(sm + IS_US) + (cb - 2) * (CH * 68) + r;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        us[j * 68] = __uint_as_float(x0[j]);
                        us[(32 + j) * 68] = __uint_as_float(x1[j]);
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            bulk_s2g_hint(rec + REC_WQ + 8192, sbase + IS_WS, 8192, pol_ef);
            bulk_s2g_hint(rec + REC_WQ + 16384 + 8192, sbase + IS_WS + 8192, 8192, pol_ef);
            bulk_s2g_hint(rec + REC_U, sbase + IS_US, 2 * CH * 68 * 4, pol_ef);
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// =====================================================================
// Inter-chunk scan on tcgen05: one CTA per (sequence, value head, 64-row V
// block): four epilogue warps and one issuer warp.
//
// Epilogue thread (k, half) keeps S[v][k] for the 32 v of its half of the
// block in fp32 registers (warps w and w + 4 share TMEM lane quarter w).  Per chunk, in transposed form:
//   MMA1 (bf16, M=64)   Y^T[v][m] = sum_k S[v][k] [Qg; W][m][k]      (A: S, MN-major; B: WQ image)
//   Delta^T[v][r] = U[r][v] - Y^T[v][64 + r]                         (threads v)
//   MMA3 (tf32, M=128)  Z[k][v]   = sum_r Kd^T[k][r] Delta^T[v][r]   (state update)
//   MMA2 (bf16, M=64)   Y^T[v][r] += sum_j Delta^T[v][j] P[r][j]     (output correction)
//   S = S * exp(Gam_C) + Z ;  O[r][v] = Y^T[v][r] -> out (bf16, via an smem transpose)
// The issuer warp waits for the epilogue's "S written" and "Delta written"
// mbarriers, issues the MMAs and the bulk copies of the chunk records (double
// buffered, fetched a chunk ahead, L2-prefetched two chunks ahead), so MMA
// issue never stalls the epilogue warps; the epilogue waits on the MMA commit
// barriers.  The two Y^T accumulators alternate so the output epilogue of chunk
// c overlaps MMA1 of chunk c + 1.  Every wait is bounded; a timeout records
// KDA_ERR_DEVICE_TIMEOUT and both roles stop.
// =====================================================================
constexpr int SC_EPI = 256;                // epilogue threads (warps 0..7)
constexpr int SC_THREADS = SC_EPI + 32;    // + issuer warp
constexpr int VB = 64;                     // state rows (v) per CTA

constexpr uint32_t SS_WQ = 0;          // 2 x 32 KiB  B of MMA1: 128 rows x 128 bf16 (K-major)
constexpr uint32_t SS_KDT = 65536;     // 2 x 32 KiB  A of MMA3: 128 rows x 64 tf32
constexpr uint32_t SS_P = 131072;      // 2 x 8 KiB   B of MMA2: 64 rows (r) x 64 bf16 (j)
constexpr uint32_t SS_SB = 147456;     // 16 KiB      A of MMA1: S, MN-major bf16 (64 v x 128 k)
constexpr uint32_t SS_DT = 163840;     // 16 KiB      Delta^T tf32: 64 rows (v) x 64 (r)   (B of MMA3)
constexpr uint32_t SS_DTB = 180224;    // 8 KiB       Delta^T bf16: 64 rows (v) x 64 (j)  (A of MMA2)
constexpr uint32_t SS_U = 188416;      // 17 KiB      U block, fp32 [64 v][68]
constexpr uint32_t SS_OS = 205824;     // 8 KiB       output transpose, bf16 [64 r][64 v]
constexpr uint32_t SS_GC = 214016;     // 512 B
constexpr uint32_t SS_BAR = 214528;    // mbarriers
constexpr uint32_t SS_SLOT = 214656;   // TMEM address slot
constexpr uint32_t SS_FLAG = 214660;   // abort flag
constexpr uint32_t SS_BYTES = 214720 + 1024;   // + alignment slack

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

enum { BAR_WQ0 = 0, BAR_WQ1, BAR_PK0, BAR_PK1, BAR_U, BAR_MMA1, BAR_MMA3, BAR_MMA2, BAR_SBR, BAR_DTR };

__global__ __launch_bounds__(SC_THREADS, 1) void scan_kernel(const ScanParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    if (p.hdr[1] == 0) return;
    const int vb = blockIdx.x & 1;
    const int h = (blockIdx.x >> 1) % p.H_v;
    const int rank = (blockIdx.x >> 1) / p.H_v;
    if (rank >= p.nseq) return;
    const int seq = p.order[rank];
    const SeqDesc sd = p.seqs[seq];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar = sbase + SS_BAR;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SS_FLAG);
    const int n = sd.nchunk;

    if (tid == 0) {
        for (int i = 0; i < BAR_SBR; ++i) mbar_init(bar + 8 * i, 1);
        mbar_init(bar + 8 * BAR_SBR, SC_EPI);
        mbar_init(bar + 8 * BAR_DTR, SC_EPI);
        mbar_fence_init();
        *abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(sbase + SS_SLOT, 512);
    // epilogue thread: channel k = tid & 127, v half = tid >> 7 (v = 32 half .. 32 half + 31)
    const int kme = tid & 127, vhalf = (tid >> 7) & 1;
    const size_t st0 = (((size_t)seq * p.H_v + h) * KD + (size_t)vb * VB + 32 * vhalf) * KD + kme;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + SS_SLOT);
    const uint32_t tZ = tmem + 256;   // 64 columns, lanes = k

    auto rec_of = [&](int c) { return p.rec + (((size_t)sd.chunk0 + c) * p.H_v + h) * REC_BYTES; };
    auto fail = [&]() {
        set_status(KDA_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == SC_EPI / 32) {
        // ------------------------------------------------------------ issuer
        if (lane == 0) {
            auto issue_wq = [&](int c) {
                const uint32_t b = bar + 8 * (BAR_WQ0 + (c & 1));
                mbar_expect_tx(b, 32768);
                bulk_g2s(sbase + SS_WQ + (c & 1) * 32768, rec_of(c) + REC_WQ, 32768, b);
            };
            auto issue_pk = [&](int c) {
                const unsigned char *r = rec_of(c);
                const uint32_t b = bar + 8 * (BAR_PK0 + (c & 1));
                mbar_expect_tx(b, 8192 + 32768);
                bulk_g2s(sbase + SS_P + (c & 1) * 8192, r + REC_P, 8192, b);
                bulk_g2s(sbase + SS_KDT + (c & 1) * 32768, r + REC_KDT, 32768, b);
            };
            auto issue_u = [&](int c) {
                const unsigned char *r = rec_of(c);
                mbar_expect_tx(bar + 8 * BAR_U, REC_U_BLOCK + 512);
                bulk_g2s(sbase + SS_U, r + REC_U + vb * REC_U_BLOCK, REC_U_BLOCK, bar + 8 * BAR_U);
                bulk_g2s(sbase + SS_GC, r + REC_GC, 512, bar + 8 * BAR_U);
            };
            const uint32_t id1 = idesc_bf16(64, 128) | (1u << 15);   // A (S) MN-major
            const uint32_t id2 = idesc_bf16(64, 64), id3 = idesc_tf32(128, VB);
            if (n > 0) {
                issue_wq(0);
                issue_pk(0);
                issue_u(0);
            }
            for (int c = 0; c < n && !*abort_flag; ++c) {
                const int b = c & 1;
                const uint32_t pp = (c >> 1) & 1;
                const uint32_t tY = tmem + b * 128;
                if (!mbar_wait(bar + 8 * BAR_SBR, c & 1) || !mbar_wait(bar + 8 * (BAR_WQ0 + b), pp)) { fail(); break; }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < KD / 16; ++ks) {
                    const int kb = ks * 32;
                    umma_bf16(tY, umma_desc(sbase + SS_SB + ks * 2048, 8192, 1024),
                              umma_desc(sbase + SS_WQ + b * 32768 + (kb >> 7) * 16384 + (kb & 127), 16, 1024), id1,
                              ks > 0);
                }
                umma_commit(bar + 8 * BAR_MMA1);
                if (c + 1 < n) {
                    // buffers (c + 1) & 1 were last read by the MMAs of chunk c - 1
                    if (c >= 1 && !mbar_wait(bar + 8 * BAR_MMA2, (c - 1) & 1)) { fail(); break; }
                    issue_wq(c + 1);
                    issue_pk(c + 1);
                }
                if (c + 2 < n) {
                    const unsigned char *r2 = rec_of(c + 2);
                    prefetch_l2(r2 + REC_WQ, 32768 + 8192 + 32768);
                    prefetch_l2(r2 + REC_U + vb * REC_U_BLOCK, REC_U_BLOCK);
                    prefetch_l2(r2 + REC_GC, 512);
                }
                if (!mbar_wait(bar + 8 * BAR_DTR, c & 1)) { fail(); break; }
                if (c + 1 < n) issue_u(c + 1);
                if (!mbar_wait(bar + 8 * (BAR_PK0 + b), pp)) { fail(); break; }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < CH / 8; ++ks) {
                    const int kb = ks * 32;
                    umma_tf32(tZ, umma_desc(sbase + SS_KDT + b * 32768 + (kb >> 7) * 16384 + (kb & 127), 16, 1024),
                              umma_desc(sbase + SS_DT + (kb >> 7) * 8192 + (kb & 127), 16, 1024), id3, ks > 0);
                }
                umma_commit(bar + 8 * BAR_MMA3);
#pragma unroll
                for (int ks = 0; ks < CH / 16; ++ks) {
                    umma_bf16(tY, umma_desc(sbase + SS_DTB + ks * 32, 16, 1024),
                              umma_desc(sbase + SS_P + b * 8192 + ks * 32, 16, 1024), id2, 1);
                }
                umma_commit(bar + 8 * BAR_MMA2);
            }
            // drain whatever is still in flight (bounded)
            for (int i = 0; i < BAR_SBR; ++i)
                for (uint32_t pp = 0; pp < 2; ++pp) mbar_wait(bar + 8 * i, pp, *abort_flag ? (1u << 14) : 0u);
        }
    } else {
        // ------------------------------------------------------------ epilogue (thread k = tid)
        constexpr int VH = VB / 2;
        float S[VH];
#pragma unroll
        for (int v = 0; v < VH; ++v) S[v] = p.init ? p.init[st0 + (size_t)v * KD] : 0.f;
        const int q = warp & 3;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int vme = q * 16 + lane;      // v owned in the M = 64 layout (lane < 16)
        const bool vact = lane < 16;
        auto emit_output = [&](int cc) {
            if (!mbar_wait(bar + 8 * BAR_MMA2, cc & 1)) fail();
            tc_fence_after();
            const uint32_t tY = tmem + (cc & 1) * 128;
            uint32_t y0[32];
            tmem_ld32_nowait(tY + lane_off + 32 * vhalf, y0);
            tmem_wait_ld();
            uint16_t *os = reinterpret_cast<uint16_t *>(sm + SS_OS);
            if (vact) {
#pragma unroll
                for (int j = 0; j < 32; ++j) os[(32 * vhalf + j) * VB + vme] = f_to_bf16(__uint_as_float(y0[j]));
            }
            named_bar(1, SC_EPI);
            const int len = min(CH, sd.len - cc * CH);
            const int tok0 = sd.tok + cc * CH;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int idx = i * SC_EPI + tid, r = idx >> 3, c8 = (idx & 7) * 8;
                if (r < len)
                    *reinterpret_cast<uint4 *>(p.out + ((size_t)(tok0 + r) * p.H_v + h) * KD + vb * VB + c8) =
                        *reinterpret_cast<const uint4 *>(os + r * VB + c8);
            }
            named_bar(1, SC_EPI);
        };
        int c = 0;
        for (; c < n; ++c) {
            if (*abort_flag) break;
            const int b = c & 1;
            const uint32_t tY = tmem + b * 128;
            // ---- S (bf16) -> SB: MN-major A operand, thread (k, half) writes half of row k of K-group k / 8
#pragma unroll
            for (int c4 = 0; c4 < VH / 8; ++c4) {
                const int c8 = 4 * vhalf + c4;
                uint4 w;
                w.x = pack_bf16x2(S[8 * c4 + 0], S[8 * c4 + 1]);
                w.y = pack_bf16x2(S[8 * c4 + 2], S[8 * c4 + 3]);
                w.z = pack_bf16x2(S[8 * c4 + 4], S[8 * c4 + 5]);
                w.w = pack_bf16x2(S[8 * c4 + 6], S[8 * c4 + 7]);
                *reinterpret_cast<uint4 *>(sm + SS_SB + (kme >> 3) * 1024 + (kme & 7) * 128 + ((c8 ^ (kme & 7)) << 4)) = w;
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar + 8 * BAR_SBR);
            // ---- Delta^T = U^T - (W S^T)^T, as tf32 (B of MMA3) and bf16 (A of MMA2)
            if (!mbar_wait(bar + 8 * BAR_MMA1, c & 1) || !mbar_wait(bar + 8 * BAR_U, c & 1)) fail();
            tc_fence_after();
            const float g = reinterpret_cast<const float *>(sm + SS_GC)[kme];
            {
                // this thread: v = vme, r = 32 vhalf .. 32 vhalf + 31
                uint32_t ys[32];
                tmem_ld32_nowait(tY + lane_off + 64 + 32 * vhalf, ys);
                tmem_wait_ld();
                if (vact) {
                    const float *urow = reinterpret_cast<const float *>(sm + SS_U) + vme * 68 + 32 * vhalf;
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 8) {
                        const int j = 32 * vhalf + jj;
                        const float4 ua = *reinterpret_cast<const float4 *>(urow + jj);
                        const float4 ub = *reinterpret_cast<const float4 *>(urow + jj + 4);
                        const float d0 = ua.x - __uint_as_float(ys[jj + 0]), d1 = ua.y - __uint_as_float(ys[jj + 1]);
                        const float d2 = ua.z - __uint_as_float(ys[jj + 2]), d3 = ua.w - __uint_as_float(ys[jj + 3]);
                        const float d4 = ub.x - __uint_as_float(ys[jj + 4]), d5 = ub.y - __uint_as_float(ys[jj + 5]);
                        const float d6 = ub.z - __uint_as_float(ys[jj + 6]), d7 = ub.w - __uint_as_float(ys[jj + 7]);
                        *reinterpret_cast<uint4 *>(sm + SS_DT + sw128_off(vme, 4 * j, VB)) =
                            make_uint4(tf32_bits(d0), tf32_bits(d1), tf32_bits(d2), tf32_bits(d3));
                        *reinterpret_cast<uint4 *>(sm + SS_DT + sw128_off(vme, 4 * j + 16, VB)) =
                            make_uint4(tf32_bits(d4), tf32_bits(d5), tf32_bits(d6), tf32_bits(d7));
                        *reinterpret_cast<uint4 *>(sm + SS_DTB + sw128_off(vme, 2 * j, VB)) =
                            make_uint4(pack_bf16x2(d0, d1), pack_bf16x2(d2, d3), pack_bf16x2(d4, d5),
                                       pack_bf16x2(d6, d7));
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar + 8 * BAR_DTR);
            // ---- previous chunk's output (overlaps MMA3 of this chunk)
            if (c > 0) emit_output(c - 1);
            // ---- S = S * exp(Gam_C) + Z   (lanes k of Z, columns v of this half)
            if (!mbar_wait(bar + 8 * BAR_MMA3, c & 1)) fail();
            tc_fence_after();
            {
                uint32_t z0[32];
                tmem_ld32_nowait(tZ + lane_off + 32 * vhalf, z0);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) S[j] = fmaf(S[j], g, __uint_as_float(z0[j]));
            }
            tc_fence_before();
        }
        if (!*abort_flag && n > 0) emit_output(n - 1);
        if (p.fin && !*abort_flag) {
            float *dst = p.fin + st0;
#pragma unroll
            for (int v = 0; v < VH; ++v) dst[(size_t)v * KD] = S[v];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
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

void timing_begin(cudaStream_t s);
void timing_mark(const char *name, cudaStream_t s);

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
                                             (int)IS_BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SS_BYTES);
        if (e != cudaSuccess) return e;
    }
    timing_begin(stream);
    plan_kernel<<<1, PLAN_THREADS, 0, stream>>>(cu, N, B, T, ws.seqs, ws.chunks, ws.order, ws.hdr, nck);
    ++*launches;
    timing_mark("plan_kernel", stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (nck > 0) {
        IntraParams ip;
        ip.q = q; ip.k = k; ip.v = v; ip.graw = graw; ip.b = b; ip.A_log = A_log; ip.scale = scale;
        ip.H_qk = H_qk; ip.H_v = H_v; ip.chunks = ws.chunks; ip.hdr = ws.hdr;
        ip.rec = ws.rec;
        int dev = 0, nsm = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        const long long items = nck * (long long)H_v;
        const unsigned grid = (unsigned)(items < nsm ? items : nsm);   // persistent: one CTA per SM
        intra_kernel<<<grid, IN_THREADS, IS_BYTES, stream>>>(ip);
        ++*launches;
        timing_mark("intra_kernel", stream);
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
        timing_mark("scan_kernel", stream);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kda
