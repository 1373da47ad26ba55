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
#include <type_traits>
#include <utility>

#include "kda_common.cuh"
#include "kda_invert.cuh"
#include "kda_tma.cuh"

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
    grid_dep_launch();
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
    if (!cu) {
        // B sequences of T tokens: the tables in closed form (no scan of chunk counts)
        const int nc = (int)(((long long)T + CH - 1) / CH);
        for (int i = tid; i < nseq; i += PLAN_THREADS) {
            SeqDesc sd;
            sd.tok = i * T;
            sd.len = T;
            sd.chunk0 = i * nc;
            sd.nchunk = nc;
            seqs[i] = sd;
        }
        if (tid == 0) s_carry = nseq * nc;
        __syncthreads();
    }
    for (int base = 0; cu && base < nseq; base += PLAN_THREADS) {
        const int i = base + tid;
        int len = 0, tok = 0;
        if (i < nseq) {
            tok = cu ? cu[i] : i * T;
            len = cu ? cu[i + 1] - cu[i] : T;
        }
        const int nc = (int)(((long long)len + CH - 1) / CH);
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
    if (!cu) {
        // B sequences of T tokens: chunk g is chunk g % nc of sequence g / nc (all threads)
        const int nc = (int)(((long long)T + CH - 1) / CH);
        for (int g = tid; g < total; g += PLAN_THREADS) {
            const int i = g / nc, c = g - i * nc;
            ChunkDesc cd;
            cd.seq = i;
            cd.tok = i * T + c * CH;
            cd.len = min(CH, T - c * CH);
            cd.idx = c;
            chunks[g] = cd;
        }
    } else {
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
    }
    if (!cu) {
        // equal lengths: the order is the identity
        for (int i = tid; i < nseq; i += PLAN_THREADS) order[i] = i;
    } else if (nseq <= LPT_MAX_SEQ) {
        for (int i = tid; i < nseq; i += PLAN_THREADS) s_len[i] = cu[i + 1] - cu[i];
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
//   RN  rq [64], rk [64], fp32                                     (512 B)
// The scalar-gate kernel leaves KDT and the Qg rows of WQ unwritten, stores f_r = rk_r
// exp(Gam_C - Gam_r) in the rk slot, rq_r exp(Gam_r) in entries 64..127 of GC and P times rq
// (its scan reads the raw key and query rows instead).
constexpr uint32_t REC_WQ = 0, REC_P = 32768, REC_KDT = 40960, REC_U = 73728, REC_GC = 108544, REC_RN = 109056;
constexpr uint32_t REC_U_BLOCK = 64 * 68 * 4;   // 17408 B per V block
constexpr uint32_t REC_BYTES = 109568;

// =====================================================================
// Intra-chunk kernel: persistent CTAs of 8 warps, two resident per SM, each
// looping over (chunk, value head) work items.  With two CTAs per SM the
// serial steps of one item (MMA round trips, the blocked inversion, barrier
// waits) overlap the elementwise work of the other.
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
// the block's first and last Gam (exponents clamped at 85 nats).  The 128
// channels are processed in four slices of 32; per slice the gate of the
// slice's channels is activated and prefix-summed inside each warp (4
// channels x 64 rows per warp), and two tcgen05 MMAs (tf32, M = 128) accumulate
//   D_off [128 x 96] = [F_k ; F_q] . [H versions]^T     (all below-diagonal blocks)
//   D_diag[128 x 64] = [R_k ; R_q] . [C_k]^T            (the four diagonal blocks)
// into TMEM; rows 0..63 give A (times beta_r), rows 64..127 give P.  After the
// blocked inversion T = (I + A)^{-1}, two bf16 MMA chains give
//   W = (T'_hi + T'_lo) Kg,  U = (T'_hi + T'_lo) V,   T' = T diag(beta) split into two bf16 terms,
// with Kg (the gated key, written in bf16 by the slices) and V as MN-major operands.
// =====================================================================
constexpr int IN_THREADS = 256;
constexpr int IN_CTAS_PER_SM = 2;
constexpr int SL = 32;                  // channels per slice (one 128-byte tf32 atom)
constexpr uint32_t RAW_T = 4096;        // one tensor of a raw slice: 64 rows x 32 bf16 (64-byte rows, 64-byte swizzle)
constexpr uint32_t RAW_SLICE = 3 * RAW_T;   // q, k, graw

constexpr uint32_t IS_KG = 0;                // B of the W MMA: Kg, MN-major bf16, N = 128 (k), K = 64 (j)
constexpr uint32_t IS_R1 = 16384;            // 52 KiB: slice operands; then A, T, scratch, P; then W, U staging
constexpr uint32_t IS_ROWS = IS_R1;          // 256 rows x 32 ch tf32: F_k, F_q, R_k, R_q
constexpr uint32_t IS_COLS = IS_R1 + 32768;  // 160 rows x 32 ch tf32: C_k (64), H versions (96)
constexpr uint32_t IS_R2 = 69632;            // raw q / k / graw slices (two buffers, TMA); then V
constexpr uint32_t IS_R3 = 94208;            // per-slice exchange of gate sums; then T'_hi, T'_lo
constexpr uint32_t IS_XW = IS_R3;            // per-warp gate totals [8 warps][32 ch] fp32
constexpr uint32_t IS_XG = IS_R3 + 1024;     // gate at each block's first row [4 blocks][32 ch] fp32
constexpr uint32_t IS_QGS = IS_R3 + 2048;    // Qg of two slices (one 64-channel atom, 8 KiB) for a bulk store
constexpr uint32_t IS_MISC = 110592;
constexpr uint32_t IS_RV = IS_MISC;          // rq, rk, beta, qk [4][64] fp32
constexpr uint32_t IS_GCS = IS_MISC + 1024;  // exp(Gam_C) [128]
constexpr uint32_t IS_BAR = IS_MISC + 1536;  // 5 mbarriers: A/P MMAs, W/U MMAs, raw buffer 0, raw buffer 1, V
constexpr uint32_t IS_SLOT = IS_MISC + 1576; // TMEM address
constexpr uint32_t IS_BYTES = IS_MISC + 1584 + 1024;   // + alignment slack
// aliases once the slices are done
constexpr uint32_t IS_A = IS_R1;             // fp32 [64][68]
constexpr uint32_t IS_T = IS_R1 + 17408;     // fp32 [64][68]
constexpr uint32_t IS_X = IS_R1 + 34816;     // fp32 [32][36] (or [2][16][20])
constexpr uint32_t IS_PI = IS_R1 + 39424;    // P image staging (bf16, 8 KiB)
constexpr uint32_t IS_V = IS_R2;             // B of the U MMA: V, MN-major bf16, N = 128 (v), K = 64 (j)
constexpr uint32_t IS_TWH = IS_A;            // A of the W MMA: T'_W = T diag(beta rk), hi / lo (A is dead by then)
constexpr uint32_t IS_TWL = IS_A + 8192;
constexpr uint32_t IS_TPH = IS_R3;           // A of the W/U MMAs: T'_hi, 64 rows (r) x 64 (j) bf16
constexpr uint32_t IS_TPL = IS_R3 + 8192;    // T'_lo
constexpr uint32_t IS_WS = IS_R1;            // W half of the WQ image (2 x 8 KiB)
constexpr uint32_t IS_US = IS_R1 + 16384;    // U image staging (2 x 64 x 68 fp32)
static_assert(IS_PI + 8192 <= IS_R2 && IS_US + 2 * CH * 68 * 4 <= IS_R2, "R1 aliases overflow");
static_assert(IS_XG + 512 <= IS_QGS && IS_QGS + 8192 <= IS_MISC && IS_QGS % 128 == 0, "Qg staging overflow");
static_assert(IS_R2 + 2 * RAW_SLICE <= IS_R3 && IS_XG + 512 <= IS_MISC && IS_TPL + 8192 <= IS_MISC,
              "R2 / R3 overflow");
static_assert(IS_R2 % 1024 == 0 && RAW_SLICE % 512 == 0 && RAW_T % 512 == 0, "TMA swizzle alignment");
static_assert(IN_CTAS_PER_SM * (IS_BYTES + 1024) <= 228 * 1024, "two CTAs per SM must fit");

enum { RV_RQ = 0, RV_RK = 64, RV_BETA = 128, RV_QK = 192 };

struct IntraParams {
    const uint16_t *q, *k, *v, *graw, *b;
    const float *A_log;
    float scale;
    int H_qk, H_v;        // head counts of the tensors (their strides)
    int h0, Hw;           // value-head window [h0, h0 + Hw) this launch processes
    const ChunkDesc *chunks;
    const int *hdr;
    unsigned char *rec;   // [chunk][Hw] records of REC_BYTES
};

// A / P operands are stored as fp32 bit patterns: the tf32 MMA uses their upper 19 bits
// (truncation), which the chunk-algebra error study shows costs nothing measurable here
__device__ __forceinline__ void sts128(unsigned char *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}
// byte offset of element (n, kk) in an MN-major bf16 operand with 64-element
// atoms along N (stride 8 KiB) and 8-row K groups (stride 1 KiB)
__device__ __forceinline__ uint32_t mn_off_bf16(int n, int kk) {
    return (uint32_t)((n >> 6) * 8192 + (kk >> 3) * 1024 + (kk & 7) * 128 + ((((n & 63) >> 3) ^ (kk & 7)) << 4) +
                      ((n & 7) << 1));
}
// Byte offset of the channel pair (2p, 2p + 1) of row r in a raw slice: 64-byte rows whose four
// 16-byte units are permuted by the TMA 64-byte swizzle (unit ^= (r / 2) % 4)
__device__ __forceinline__ uint32_t raw_pair_off(int r, int p) {
    return (uint32_t)(r * 64 + ((((p >> 2) ^ ((r >> 1) & 3))) << 4) + 4 * (p & 3));
}

__device__ __forceinline__ void stg_hint_b32(void *p, uint32_t v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;\n" ::"l"(p), "r"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void stg_hint_v4(void *p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;\n" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

__global__ __launch_bounds__(IN_THREADS, IN_CTAS_PER_SM) void intra_kernel(const __grid_constant__ CUtensorMap tq,
                                                                          const __grid_constant__ CUtensorMap tk,
                                                                          const __grid_constant__ CUtensorMap tg,
                                                                          const __grid_constant__ CUtensorMap tv,
                                                                          const IntraParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = aligned_smem<1024>(smem_raw);
    grid_dep_wait();     // the plan's tables
    grid_dep_launch();   // the scan's CTAs may be placed as this kernel's CTAs retire
    if (p.hdr[1] == 0) return;
    const long long n_items = (long long)p.hdr[0] * p.Hw;
    if ((long long)blockIdx.x >= n_items) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t sbase = smem_u32(sm);
    // mbarriers: A/P MMAs (two committers), W/U MMAs, raw buffers 0 and 1, V
    const uint32_t bar_ap = sbase + IS_BAR, bar_wu = bar_ap + 8, bar_raw = bar_ap + 16, bar_v = bar_ap + 32;
    const uint64_t pol_ef = l2_evict_first_policy();
    float *rv = reinterpret_cast<float *>(sm + IS_RV);
    float *gcs = reinterpret_cast<float *>(sm + IS_GCS);
    float *sA = reinterpret_cast<float *>(sm + IS_A);
    float *sT = reinterpret_cast<float *>(sm + IS_T);
    float *sX = reinterpret_cast<float *>(sm + IS_X);
    if (tid == 0) {
        mbar_init(bar_ap, 2);
        mbar_init(bar_wu, 1);
        mbar_init(bar_raw, 1);
        mbar_init(bar_raw + 8, 1);
        mbar_init(bar_v, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(sbase + IS_SLOT, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + IS_SLOT);
    const uint32_t t_off = tmem, t_diag = tmem + 96, t_w = tmem, t_u = tmem + 128;

    const int group = p.H_v / p.H_qk;
    // raw q / k / graw of slice s (32 channels) of item (d, hh) into buffer s % 2 (one thread issues;
    // rows past the tensor arrive as zeros, rows past the chunk's length are masked by the readers)
    auto issue_raw = [&](const ChunkDesc &d, int hh, int s) {
        const uint32_t dst = sbase + IS_R2 + (uint32_t)(s & 1) * RAW_SLICE, mb = bar_raw + 8 * (s & 1);
        mbar_expect_tx(mb, RAW_SLICE);
        tma_load_3d(dst, &tq, s * SL, hh / group, d.tok, mb);
        tma_load_3d(dst + RAW_T, &tk, s * SL, hh / group, d.tok, mb);
        tma_load_3d(dst + 2 * RAW_T, &tg, s * SL, hh, d.tok, mb);
    };

    // Thread mapping of the slice phase: channel pair cp = 2 (lane % 16) of the slice, 4-row segment
    // seg = 2 warp + lane / 16 (rows 4 seg .. 4 seg + 3), 16-row block blk = warp / 2.  The gate prefix
    // sum runs down the thread's own rows; segment and block sums are exchanged once per slice.
    const int pp = lane & 15, hs = lane >> 4, seg = 2 * warp + hs, blk = warp >> 1, r0 = 4 * seg, cp = 2 * pp;
    const bool wodd = (warp & 1) != 0;
    uint32_t roff[4];                 // raw-slice offsets of this thread's channel pair in its four rows
    uint32_t ooff[4];                 // tf32 operand-image offsets (row r0 + i, channels cp, cp + 1)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + i;
        roff[i] = raw_pair_off(r, pp);
        ooff[i] = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((pp >> 1) ^ (r & 7))) << 4) + 8 * (pp & 1));
    }
    // H versions (column operand times the block decay between the pair): rows 64 + 16 v + (r % 16) of COLS;
    // Kg / Qg (bf16, 64-channel atoms of 128-byte rows): element (row r, channel cp) of the slice's half-atom;
    // Kd^T (tf32, rows = channels, 128-byte rows of 32 columns): the 16-byte unit of rows r0 .. r0 + 3
    uint32_t hoo[4], kgo[4], kdo[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + i;
        hoo[i] = (ooff[i] & 1023u) + (uint32_t)(((r0 & 15) >> 3) * 1024);
        kgo[i] = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((pp >> 2) ^ (r & 7))) << 4) + 2 * (cp & 7));
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int k = cp + e;
        kdo[e] = (uint32_t)((k >> 3) * 1024 + (k & 7) * 128 + ((((seg & 7) ^ (k & 7))) << 4));
    }

    // The description of the next item (chunk, head, A_log) is fetched while the
    // current one is processed, and its first two raw slices are issued as soon as
    // the current item's W / U MMAs have released the raw buffers.
    // item = chunk * Hw + (head - h0) advances by gridDim.x: keep (chunk, head) incrementally
    const int step_c = (int)(gridDim.x / p.Hw), step_h = (int)(gridDim.x % p.Hw);
    long long item = blockIdx.x;
    int chunk_next = (int)(item / p.Hw), h_next = p.h0 + (int)(item % p.Hw);
    ChunkDesc cd_next = p.chunks[chunk_next];
    float alog_next = p.A_log[h_next];
    if (tid == 0) {
        issue_raw(cd_next, h_next, 0);
        issue_raw(cd_next, h_next, 1);
    }
    for (int it = 0; item < n_items; item += gridDim.x, ++it) {
        const int chunk = chunk_next, h = h_next;
        const ChunkDesc cd = cd_next;
        const float a_gate = ex2(alog_next * LOG2E);
        const size_t ch = (size_t)chunk * p.Hw + (h - p.h0);
        unsigned char *rec = p.rec + ch * REC_BYTES;
        const int len = cd.len;
        const long long nitem = item + gridDim.x;
        const bool has_next = nitem < n_items;
        if (has_next) {
            chunk_next += step_c;
            h_next += step_h;
            if (h_next >= p.h0 + p.Hw) {
                h_next -= p.Hw;
                ++chunk_next;
            }
            cd_next = p.chunks[chunk_next];
            alog_next = p.A_log[h_next];
        }

        // ---- 1. beta (global load); the previous item's bulk stores must be done reading shared
        //         memory (W/U staging, P, exp(Gam_C)) before this item's slices overwrite it
        float bb_raw = 0.f;
        if (tid < len) bb_raw = bf16_to_f(p.b[((size_t)cd.tok + tid) * p.H_v + h]);
        if (tid == 0) bulk_wait_read_all();
        if (tid < CH) rv[RV_BETA + tid] = tid < len ? 1.0f / (1.0f + ex2(-bb_raw * LOG2E)) : 0.f;

        // ---- 2. channel slices.  Per slice: gate of the thread's rows (softplus, prefix sum), exchange
        //         of segment sums, then every operand of the slice.  q and k enter the operands
        //         unnormalised: every product below is linear in a row's q or k, so the L2 norms
        //         (summed here over the slices) are applied afterwards: to A and P in their epilogue,
        //         to Kg through T' for W, and by the scan to Kd and Qg.
        const float na = -a_gate;
        const bool partial = len < CH;
        float nq[4] = {0.f, 0.f, 0.f, 0.f}, nk[4] = {0.f, 0.f, 0.f, 0.f}, nqk[4] = {0.f, 0.f, 0.f, 0.f};
        float *xw = reinterpret_cast<float *>(sm + IS_XW);
        float *xg = reinterpret_cast<float *>(sm + IS_XG);
#pragma unroll 1
        for (int sl = 0; sl < KD / SL; ++sl) {
            const int c0 = sl * SL;
            const unsigned char *rawb = sm + IS_R2 + (sl & 1) * RAW_SLICE;
            if (!mbar_wait(bar_raw + 8 * (sl & 1), (uint32_t)(sl >> 1) & 1)) set_status(KDA_ERR_DEVICE_TIMEOUT);
            // 2a. gate of rows r0 .. r0 + 3, channels c0 + cp, + 1 (log2 units), in-segment prefix sums
            uint32_t qw[4], kw[4];
            float2 G[4];
            {
                float sx = 0.f, sy = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    qw[i] = *reinterpret_cast<const uint32_t *>(rawb + roff[i]);
                    kw[i] = *reinterpret_cast<const uint32_t *>(rawb + RAW_T + roff[i]);
                    const uint32_t gw = *reinterpret_cast<const uint32_t *>(rawb + 2 * RAW_T + roff[i]);
                    float s0 = softplus_log2(bf16_lo(gw)), s1 = softplus_log2(bf16_hi(gw));
                    if (partial && r0 + i >= len) {   // rows past the chunk: no decay, q = k = 0
                        s0 = 0.f;
                        s1 = 0.f;
                        qw[i] = 0u;
                        kw[i] = 0u;
                    }
                    sx += s0;
                    sy += s1;
                    G[i] = make_float2(sx * na, sy * na);
                }
            }
            // 2b. segment sums -> per-warp sums and the block's first-row gate, exchanged through smem
            const float2 tseg = G[3];
            float2 tother;
            tother.x = __shfl_xor_sync(0xffffffffu, tseg.x, 16);
            tother.y = __shfl_xor_sync(0xffffffffu, tseg.y, 16);
            if (hs == 0) {
                *reinterpret_cast<float2 *>(xw + warp * SL + cp) = make_float2(tseg.x + tother.x, tseg.y + tother.y);
                if (!wodd) *reinterpret_cast<float2 *>(xg + blk * SL + cp) = G[0];
            }
            // the previous slice's MMAs must be done with ROWS / COLS before they are rewritten, and
            // from slice 2 on the bulk store of the first two slices' Qg (thread 64's) with its staging
            if (tid == 0 && sl > 0 && !mbar_wait(bar_ap, (uint32_t)(sl - 1) & 1)) set_status(KDA_ERR_DEVICE_TIMEOUT);
            if (tid == 64 && sl == 2) bulk_wait_read_all();
            __syncthreads();
            // block boundaries M_b = Gam at the end of block b - 1 (M_0 = 0, M_4 = Gam_C)
            float2 Mb, Mb1, Wlo;
            const float2 wt0 = *reinterpret_cast<const float2 *>(xw + 0 * SL + cp);
            const float2 wt1 = *reinterpret_cast<const float2 *>(xw + 1 * SL + cp);
            const float2 wt2 = *reinterpret_cast<const float2 *>(xw + 2 * SL + cp);
            const float2 wt3 = *reinterpret_cast<const float2 *>(xw + 3 * SL + cp);
            const float2 wt4 = *reinterpret_cast<const float2 *>(xw + 4 * SL + cp);
            const float2 wt5 = *reinterpret_cast<const float2 *>(xw + 5 * SL + cp);
            const float2 wt6 = *reinterpret_cast<const float2 *>(xw + 6 * SL + cp);
            const float2 wt7 = *reinterpret_cast<const float2 *>(xw + 7 * SL + cp);
            const float2 M1 = make_float2(wt0.x + wt1.x, wt0.y + wt1.y);
            const float2 M2 = make_float2(M1.x + (wt2.x + wt3.x), M1.y + (wt2.y + wt3.y));
            const float2 M3 = make_float2(M2.x + (wt4.x + wt5.x), M2.y + (wt4.y + wt5.y));
            const float2 M4 = make_float2(M3.x + (wt6.x + wt7.x), M3.y + (wt6.y + wt7.y));
            switch (blk) {
                case 0: Mb = make_float2(0.f, 0.f); Mb1 = M1; Wlo = wt0; break;
                case 1: Mb = M1; Mb1 = M2; Wlo = wt2; break;
                case 2: Mb = M2; Mb1 = M3; Wlo = wt4; break;
                default: Mb = M3; Mb1 = M4; Wlo = wt6; break;
            }
            const float2 gf = *reinterpret_cast<const float2 *>(xg + blk * SL + cp);
            // Gam - M_blk of row r0 + i is wlo + (pre + G[i]) (<= 0).  The block total is summed in the
            // same order, so that the block's last row has Gam - M_blk+1 = 0 exactly (its Kd factor is
            // exactly 1 however strong the gate).  The block's midpoint reference
            // mu = (Gam(first row) + M_blk+1) / 2 sits at hm above M_blk.
            const float2 wlo = make_float2(wodd ? Wlo.x : 0.f, wodd ? Wlo.y : 0.f);
            const float2 pre = make_float2(hs ? tother.x : 0.f, hs ? tother.y : 0.f);
            float2 tot;
            switch (blk) {
                case 0: tot = M1; break;
                case 1: tot = make_float2(wt2.x + wt3.x, wt2.y + wt3.y); break;
                case 2: tot = make_float2(wt4.x + wt5.x, wt4.y + wt5.y); break;
                default: tot = make_float2(wt6.x + wt7.x, wt6.y + wt7.y); break;
            }
            const float2 hm = make_float2(0.5f * (gf.x + tot.x), 0.5f * (gf.y + tot.y));
            const float2 eb = make_float2(ex2(Mb.x), ex2(Mb.y));                       // exp(M_blk)
            const float2 ea = make_float2(ex2(M4.x - Mb1.x), ex2(M4.y - Mb1.y));       // exp(Gam_C - M_blk+1)
            if (warp == 0 && hs == 0)
                *reinterpret_cast<float2 *>(gcs + c0 + cp) = make_float2(ex2(M4.x), ex2(M4.y));
            // block decays between sub-block pairs for the H versions of this block's rows
            float2 xa = make_float2(1.f, 1.f), xb = make_float2(1.f, 1.f);
            if (blk == 0) {
                xa = make_float2(ex2(M2.x - M1.x), ex2(M2.y - M1.y));   // pair (2, 0)
                xb = make_float2(ex2(M3.x - M1.x), ex2(M3.y - M1.y));   // pair (3, 0)
            } else if (blk == 1) {
                xa = make_float2(ex2(M3.x - M2.x), ex2(M3.y - M2.y));   // pair (3, 1)
            }
            // 2c. operands of rows r0 .. r0 + 3.  Offsets that depend on the slice: Kg / Qg images are
            // 64-channel atoms (the slice's half of an atom flips unit bit 2, byte offset 64), Kd^T
            // moves by 32 rows (4 KiB) per slice.
            const uint32_t x64 = 64u * (uint32_t)(sl & 1);
            unsigned char *const kgs = sm + IS_KG + 8192 * (sl >> 1);
            unsigned char *const qgs = sm + IS_QGS;
            unsigned char *const kds = rec + REC_KDT + (r0 >> 5) * 16384 + 4096 * sl;
            const float2 nhm = make_float2(-hm.x, -hm.y);
            auto operands = [&](auto blkc) {
                constexpr int BLK = decltype(blkc)::value;
                unsigned char *const rows = sm + IS_ROWS;
                unsigned char *const cols = sm + IS_COLS;
                float2 kdv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 x = __fadd2_rn(wlo, __fadd2_rn(pre, G[i]));
                    const float2 nx = make_float2(-x.x, -x.y);
                    const float2 kv = make_float2(bf16_lo(kw[i]), bf16_hi(kw[i]));
                    const float2 qv = make_float2(bf16_lo(qw[i]), bf16_hi(qw[i]));
                    // block-relative factors (always <= 1, exact for any gate strength) and the
                    // diagonal block's midpoint factors (exponents clamped at 85 nats)
                    const float2 ah = __fadd2_rn(tot, nx), ar = __fadd2_rn(x, nhm), ac = __fadd2_rn(hm, nx);
                    const float2 f = make_float2(ex2(x.x), ex2(x.y));
                    const float2 hf = make_float2(ex2(ah.x), ex2(ah.y));
                    const float2 dr = make_float2(ex2(fminf(ar.x, DIAG_CLAMP2)), ex2(fminf(ar.y, DIAG_CLAMP2)));
                    const float2 dc = make_float2(ex2(fminf(ac.x, DIAG_CLAMP2)), ex2(fminf(ac.y, DIAG_CLAMP2)));
                    const float2 fk = __fmul2_rn(kv, f), fq = __fmul2_rn(qv, f);
                    const float2 hk = __fmul2_rn(kv, hf);
                    *reinterpret_cast<float2 *>(rows + ooff[i]) = fk;
                    *reinterpret_cast<float2 *>(rows + 8192 + ooff[i]) = fq;
                    *reinterpret_cast<float2 *>(rows + 16384 + ooff[i]) = __fmul2_rn(kv, dr);
                    *reinterpret_cast<float2 *>(rows + 24576 + ooff[i]) = __fmul2_rn(qv, dr);
                    *reinterpret_cast<float2 *>(cols + ooff[i]) = __fmul2_rn(kv, dc);
                    // H versions: rows 64 + 16 v + r % 16 (v: pairs (1,0), (2,0), (2,1), (3,0), (3,1), (3,2))
                    if (BLK == 0) {
                        *reinterpret_cast<float2 *>(cols + 8 * 1024 + hoo[i]) = hk;
                        *reinterpret_cast<float2 *>(cols + 10 * 1024 + hoo[i]) = __fmul2_rn(hk, xa);
                        *reinterpret_cast<float2 *>(cols + 14 * 1024 + hoo[i]) = __fmul2_rn(hk, xb);
                    } else if (BLK == 1) {
                        *reinterpret_cast<float2 *>(cols + 12 * 1024 + hoo[i]) = hk;
                        *reinterpret_cast<float2 *>(cols + 16 * 1024 + hoo[i]) = __fmul2_rn(hk, xa);
                    } else if (BLK == 2) {
                        *reinterpret_cast<float2 *>(cols + 18 * 1024 + hoo[i]) = hk;
                    }
                    kdv[i] = __fmul2_rn(hk, ea);
                    // Kg (bf16) into the MN-major B operand of the W MMA (element (k = c0 + cp, j = r)),
                    // Qg (bf16) into the staging of rows 0..63 of one atom of the record's WQ image
                    const float2 kg = __fmul2_rn(fk, eb), qg = __fmul2_rn(fq, eb);
                    *reinterpret_cast<uint32_t *>(kgs + (kgo[i] ^ x64)) = pack_bf16x2(kg.x, kg.y);
                    *reinterpret_cast<uint32_t *>(qgs + (kgo[i] ^ x64)) = pack_bf16x2(qg.x, qg.y);
                    // partial row sums of q.q, k.k, q.k over this thread's two channels
                    nq[i] = fmaf(qv.x, qv.x, fmaf(qv.y, qv.y, nq[i]));
                    nk[i] = fmaf(kv.x, kv.x, fmaf(kv.y, kv.y, nk[i]));
                    nqk[i] = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, nqk[i]));
                }
                // Kd^T rows k = c0 + cp, c0 + cp + 1, columns r0 .. r0 + 3: one 16-byte unit each (tf32)
                stg_hint_v4(kds + kdo[0], make_uint4(tf32_rn_bits(kdv[0].x), tf32_rn_bits(kdv[1].x),
                                                     tf32_rn_bits(kdv[2].x), tf32_rn_bits(kdv[3].x)), pol_ef);
                stg_hint_v4(kds + kdo[1], make_uint4(tf32_rn_bits(kdv[0].y), tf32_rn_bits(kdv[1].y),
                                                     tf32_rn_bits(kdv[2].y), tf32_rn_bits(kdv[3].y)), pol_ef);
            };
            switch (blk) {
                case 0: operands(std::integral_constant<int, 0>{}); break;
                case 1: operands(std::integral_constant<int, 1>{}); break;
                case 2: operands(std::integral_constant<int, 2>{}); break;
                default: operands(std::integral_constant<int, 3>{}); break;
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            // the two accumulators are issued by lane 0 of warps 0 and 4 (each in k order), each
            // committing to the slice barrier, so neither warp carries the whole issue time
            if (tid == 0 || tid == 128) {
                tc_fence_after();
                const bool offd = tid == 0;
                const uint32_t id = offd ? idesc_tf32(128, 96) : idesc_tf32(128, 64);
                const uint32_t arow = sbase + IS_ROWS + (offd ? 0u : 16384u), bcol = sbase + IS_COLS + (offd ? 8192u : 0u);
#pragma unroll
                for (int ks = 0; ks < SL / 8; ++ks)
                    umma_tf32(offd ? t_off : t_diag, umma_desc(arow + ks * 32, 16, 1024), umma_desc(bcol + ks * 32, 16, 1024),
                              id, (sl > 0 || ks > 0) ? 1u : 0u);
                umma_commit(bar_ap);
            }
            if (tid == 64 && (sl & 1)) {
                // Qg of slices sl - 1 and sl: rows 0..63 of one 64-channel atom of the WQ image
                bulk_s2g_hint(rec + REC_WQ + 16384 * (sl >> 1), sbase + IS_QGS, 8192, pol_ef);
                bulk_commit();
            }
            if (tid == 32) {
                // raw buffer sl % 2 is free (every thread read it before the barrier): slice sl + 2,
                // or, after the last slice, V into the MN-major operand of the U MMA
                fence_async_smem();
                if (sl + 2 < KD / SL) {
                    issue_raw(cd, h, sl + 2);
                } else if (sl + 1 == KD / SL) {
                    mbar_expect_tx(bar_v, 2 * 8192);
                    tma_load_3d(sbase + IS_V, &tv, 0, h, cd.tok, bar_v);
                    tma_load_3d(sbase + IS_V + 8192, &tv, 64, h, cd.tok, bar_v);
                }
            }
        }
        // the last slice's MMAs (and so TMEM) complete before the epilogue
        if (tid == 0 && !mbar_wait(bar_ap, 1u)) set_status(KDA_ERR_DEVICE_TIMEOUT);
        // row norms: the 16 lanes of a half-warp hold the partial sums of the same four rows over
        // disjoint channel pairs; a reduce-scatter leaves the total of (row r0 + L / 4, quantity L % 4)
        // in lane L of the half.  rq = scale / |q|, rk = 1 / |k|; QK keeps the raw q.k (the P diagonal
        // is q.k rk; the column scaling of the epilogue supplies rk).
        {
            float v[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[4 * i] = nq[i];
                v[4 * i + 1] = nk[i];
                v[4 * i + 2] = nqk[i];
                v[4 * i + 3] = 0.f;
            }
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) {
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int j = 0; j < o; ++j) {
                    const float send = up ? v[j] : v[j + o];
                    const float keep = up ? v[j + o] : v[j];
                    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            const int L = lane & 15, row = r0 + (L >> 2), qty = L & 3;
            if (qty == 0) rv[RV_RQ + row] = p.scale * rsqrtf(v[0] + L2_EPS);
            else if (qty == 1) rv[RV_RK + row] = rsqrtf(v[0] + L2_EPS);
            else if (qty == 2) rv[RV_QK + row] = v[0];
        }
        __syncthreads();
        tc_fence_after();

        // ---- 3. A (times beta) to smem, P image (bf16) to staging.  Warp w: TMEM lanes
        //         32 (w & 3) .. (K rows 0..63, Q rows 64..127), 16-column blocks 2 (w >> 2) and 2 (w >> 2) + 1.
        {
            const int q = warp & 3, hf = warp >> 2;
            const int l = q * 32 + lane, r = l & 63, rl = r & 15, isq = l >> 6;
            const uint32_t lo = (uint32_t)(q * 32) << 16;
            const int bia = 2 * (q & 1), bib = bia + 1;
            // column offsets of the below-diagonal versions of row blocks 1, 2, 3 in D_off
            const int nsa = bia == 0 ? 0 : 16, nsb = bib == 1 ? 0 : 48;
            // A = beta_r rk_r rk_j (raw product); the P image holds P / rq_r = rk_j (raw product)
            const float be = rv[RV_BETA + r] * rv[RV_RK + r], qkd = rv[RV_QK + r];
            // Lanes 0..15 hold row block bia, lanes 16..31 row block bib = bia + 1 (half = lane >> 4).
            // A: the inversion reads only the blocks below the diagonal and the strict lower part of
            // the diagonal blocks, so A is stored unmasked.  P is the scan's exact lower-triangular
            // operand: masked diagonal blocks, zeros above.  Every case below is warp-uniform.
            const bool half = lane >= 16;
            // o = half ? (column block at cy) : (column block at cx), both read from TMEM
            auto load_pair = [&](uint32_t cx, uint32_t cy, float (&o)[16]) {
                uint32_t x[16], y[16];
                tmem_ld16_nowait(cx, x);
                tmem_ld16_nowait(cy, y);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) o[j] = __uint_as_float(half ? y[j] : x[j]);
            };
#pragma unroll 1
            for (int cbi = 0; cbi < 2; ++cbi) {
                const int cb = 2 * hf + cbi;
                const uint32_t ca = t_off + lo + nsa + 16 * cb, cbb = t_off + lo + nsb + 16 * cb, cd = t_diag + lo + 16 * cb;
                float o[16], ck[16];   // ck: column scales rk_j of this 16-column block
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(rv + RV_RK + 16 * cb + j);
                    ck[j] = t4.x;
                    ck[j + 1] = t4.y;
                    ck[j + 2] = t4.z;
                    ck[j + 3] = t4.w;
                }
                if (!isq) {
                    if (cb > bib) continue;
                    if (cb < bia) load_pair(ca, cbb, o);
                    else if (cb == bia) load_pair(cd, cbb, o);
                    else load_pair(cd, cd, o);
                    const float2 be2 = make_float2(be, be);
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float2 a0 = __fmul2_rn(__fmul2_rn(make_float2(o[j], o[j + 1]), be2), make_float2(ck[j], ck[j + 1]));
                        const float2 a1 = __fmul2_rn(__fmul2_rn(make_float2(o[j + 2], o[j + 3]), be2),
                                                     make_float2(ck[j + 2], ck[j + 3]));
                        *reinterpret_cast<float4 *>(sA + r * AS + 16 * cb + j) = make_float4(a0.x, a0.y, a1.x, a1.y);
                    }
                } else {
                    if (cb < bia) {
                        load_pair(ca, cbb, o);
                    } else if (cb <= bib) {
                        // lanes whose diagonal block this is keep j < rl and put q.k at j = rl; for
                        // cb == bia the other half holds its off-diagonal block, for cb == bib zeros
                        const bool diag = (cb == bia) != half;
                        load_pair(cd, cb == bia ? cbb : cd, o);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float dv = j < rl ? o[j] : (j == rl ? qkd : 0.f);
                            o[j] = diag ? dv : (cb == bia ? o[j] : 0.f);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] = 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float2 pj = __fmul2_rn(make_float2(o[j], o[j + 1]), make_float2(ck[j], ck[j + 1]));
                        o[j] = pj.x;
                        o[j + 1] = pj.y;
                    }
#pragma unroll
                    for (int j = 0; j < 16; j += 8)
                        *reinterpret_cast<uint4 *>(sm + IS_PI + sw128_off(r, 2 * (16 * cb + j), CH)) =
                            make_uint4(pack_bf16x2(o[j], o[j + 1]), pack_bf16x2(o[j + 2], o[j + 3]),
                                       pack_bf16x2(o[j + 4], o[j + 5]), pack_bf16x2(o[j + 6], o[j + 7]));
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        if (tid == 64) bulk_wait_read_all();   // the Qg staging is read before T' reuses R3
        __syncthreads();
        if (tid == 0) {
            bulk_s2g_hint(rec + REC_P, sbase + IS_PI, 8192, pol_ef);
            bulk_s2g_hint(rec + REC_GC, sbase + IS_GCS, 512, pol_ef);
            bulk_s2g_hint(rec + REC_RN, sbase + IS_RV, 512, pol_ef);   // rq[64], rk[64] for the scan
            bulk_commit();
        }

        // ---- 4. T = (I + A)^{-1} (blocked: diagonal 16 x 16 blocks by forward substitution, the
        //         off-diagonal blocks as split-tf32 products on mma.sync; synchronises the CTA)
        invert_unit_lower64<IN_THREADS>(sA, sT, sX, tid, warp, lane);
        // T' = T diag(beta) (for U) and T'_W = T diag(beta rk) (for W: Kg is unnormalised), each
        // split into bf16 hi + lo, as A operands (K-major, 64 r x 64 j)
        for (int idx = tid; idx < CH * (CH / 8); idx += IN_THREADS) {
            const int r = idx >> 3, j = (idx & 7) * 8;
            uint32_t hi[4], lo[4], hw[4], lw[4];
            // packed fp32 pairs: x = T beta, xw = x rk, and the hi / lo splits
            const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const float2 t2 = *reinterpret_cast<const float2 *>(sT + r * AS + j + e);
                const float2 b2 = *reinterpret_cast<const float2 *>(rv + RV_BETA + j + e);
                const float2 k2 = *reinterpret_cast<const float2 *>(rv + RV_RK + j + e);
                const float2 x2 = __fmul2_rn(t2, b2), xw2 = __fmul2_rn(x2, k2);
                const uint32_t h2 = pack_bf16x2(x2.x, x2.y);
                hi[e >> 1] = h2;
                const float2 l2 = __ffma2_rn(make_float2(bf16_lo(h2), bf16_hi(h2)), m1, x2);
                lo[e >> 1] = pack_bf16x2(l2.x, l2.y);
                const uint32_t w2 = pack_bf16x2(xw2.x, xw2.y);
                hw[e >> 1] = w2;
                const float2 lw2 = __ffma2_rn(make_float2(bf16_lo(w2), bf16_hi(w2)), m1, xw2);
                lw[e >> 1] = pack_bf16x2(lw2.x, lw2.y);
            }
            const uint32_t off = sw128_off(r, 2 * j, CH);
            *reinterpret_cast<uint4 *>(sm + IS_TPH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(sm + IS_TPL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<uint4 *>(sm + IS_TWH + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(sm + IS_TWL + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        // V arrives by TMA; rows past the chunk's length belong to the next sequence: zero them so
        // that they contribute exact zeros to U (their T' columns are zero) whatever they hold
        if (partial) {
            if (!mbar_wait(bar_v, (uint32_t)it & 1)) set_status(KDA_ERR_DEVICE_TIMEOUT);
            for (int idx = tid; idx < (CH - len) * 16; idx += IN_THREADS) {
                const int r = len + (idx >> 4), u = idx & 15;
                *reinterpret_cast<uint4 *>(sm + IS_V + (u >> 3) * 8192 + r * 128 + (u & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 5. W = (T'_W,hi + T'_W,lo) Kg   (M = 64 r, N = 128 k, K = 64 j, bf16; B MN-major) and
        //         U^T = V^T (T'_hi + T'_lo)^T   (M = 128 v, N = 64 r, K = 64 j; A = V MN-major, B = T'
        //         K-major), so that each TMEM lane v holds one row of the U image
        if (tid == 0) {
            if (!partial && !mbar_wait(bar_v, (uint32_t)it & 1)) set_status(KDA_ERR_DEVICE_TIMEOUT);
            tc_fence_after();
            const uint32_t id_w = idesc_bf16(64, 128) | (1u << 16);
            const uint32_t id_u = idesc_bf16(128, 64) | (1u << 15);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < CH / 16; ++ks) {
                    const uint64_t tp = umma_desc(sbase + (part ? IS_TPL : IS_TPH) + ks * 32, 16, 1024);
                    const uint64_t tw = umma_desc(sbase + (part ? IS_TWL : IS_TWH) + ks * 32, 16, 1024);
                    const uint32_t acc = (part > 0 || ks > 0) ? 1u : 0u;
                    umma_bf16(t_w, tw, umma_desc(sbase + IS_KG + ks * 2048, 8192, 1024), id_w, acc);
                    umma_bf16(t_u, umma_desc(sbase + IS_V + ks * 2048, 8192, 1024), tp, id_u, acc);
                }
            umma_commit(bar_wu);
            if (!mbar_wait(bar_wu, it & 1)) set_status(KDA_ERR_DEVICE_TIMEOUT);
            bulk_wait_read_all();   // the P image store is done reading before W / U staging reuses it
            // the raw buffers (V) are free: start the next item's first two slices
            if (has_next) {
                issue_raw(cd_next, h_next, 0);
                issue_raw(cd_next, h_next, 1);
            }
        }
        __syncthreads();
        tc_fence_after();
        {
            const int q = warp & 3;
            const uint32_t lo = (uint32_t)(q * 32) << 16;
            if (warp < 4) {
                // U^T: lane v = 32 q + lane holds U[r][v] for r = 0..63, i.e. row v of the U image
                const int v = q * 32 + lane;
                uint32_t x0[32], x1[32];
                tmem_ld32_nowait(t_u + lo, x0);
                tmem_ld32_nowait(t_u + lo + 32, x1);
                tmem_wait_ld();
                float *us = reinterpret_cast<float *>(sm + IS_US) + (v >> 6) * (CH * 68) + (v & 63) * 68;
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    *reinterpret_cast<float4 *>(us + j) = make_float4(__uint_as_float(x0[j]), __uint_as_float(x0[j + 1]),
                                                                      __uint_as_float(x0[j + 2]), __uint_as_float(x0[j + 3]));
                    *reinterpret_cast<float4 *>(us + 32 + j) = make_float4(__uint_as_float(x1[j]), __uint_as_float(x1[j + 1]),
                                                                           __uint_as_float(x1[j + 2]), __uint_as_float(x1[j + 3]));
                }
            } else {
                // W, M = 64 layout: row r = 16 q + lane for lane < 16
                const int r = q * 16 + lane;
#pragma unroll
                for (int rd = 0; rd < 2; ++rd) {
                    uint32_t x0[32], x1[32];
                    tmem_ld32_nowait(t_w + lo + 64 * rd, x0);
                    tmem_ld32_nowait(t_w + lo + 64 * rd + 32, x1);
                    tmem_wait_ld();
                    if (lane < 16) {
                        // W[r][k], k = 64 rd .. : row 64 + r of the WQ image (bf16)
#pragma unroll
                        for (int j = 0; j < 64; j += 8) {
                            const uint32_t *xs = j < 32 ? x0 : x1;
                            const int jj = j & 31, k = 64 * rd + j;
                            const uint32_t off = (uint32_t)rd * 8192 + (r >> 3) * 1024 + (r & 7) * 128 +
                                                 ((((2 * k) & 127) >> 4) ^ (r & 7)) * 16;
                            *reinterpret_cast<uint4 *>(sm + IS_WS + off) = make_uint4(
                                pack_bf16x2(__uint_as_float(xs[jj]), __uint_as_float(xs[jj + 1])),
                                pack_bf16x2(__uint_as_float(xs[jj + 2]), __uint_as_float(xs[jj + 3])),
                                pack_bf16x2(__uint_as_float(xs[jj + 4]), __uint_as_float(xs[jj + 5])),
                                pack_bf16x2(__uint_as_float(xs[jj + 6]), __uint_as_float(xs[jj + 7])));
                        }
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
    if (tid == 0 || tid == 64) bulk_wait_all();
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
constexpr uint32_t SS_GC = 214016;     // 1 KiB       exp(Gam_C) [128], then rq [64], rk [64] (record order)
constexpr uint32_t SS_RQ = 215040;     // 256 B       rq of the chunk whose output is emitted next
constexpr uint32_t SS_RQE = 215296;    // 256 B       scalar gate: rq exp(Gam_r) of that chunk
constexpr uint32_t SS_BAR = 215552;    // mbarriers
constexpr uint32_t SS_SLOT = 215680;   // TMEM address slot
constexpr uint32_t SS_FLAG = 215684;   // abort flag
constexpr uint32_t SS_BYTES = 215744 + 1024;   // + alignment slack

struct ScanParams {
    const unsigned char *rec;
    const SeqDesc *seqs;
    const int *order;
    const int *hdr;
    const float *init;
    float *fin;
    uint16_t *out;
    int H_qk, H_v, nseq;
    int h0, Hw;   // value-head window [h0, h0 + Hw); records are [chunk][Hw]
    int state_bf16;   // init / fin hold bf16 values (the recurrence itself stays fp32)
};

enum { BAR_WQ0 = 0, BAR_WQ1, BAR_PK0, BAR_PK1, BAR_U, BAR_MMA1, BAR_MMA3, BAR_MMA2, BAR_SBR, BAR_DTR };

// SG (scalar gate): the records carry neither Kd^T nor Qg, both row scalings of raw inputs.
//   Kd = diag(f) K, f_r = rk_r exp(Gam_C - Gam_r) (the record's rk slot): the state update reads
//     the chunk's key rows from the input (TMA map tk) and takes f on Delta instead,
//     Z = K^T (diag(f) Delta^T)^T, with K exact in bf16 and f Delta split into bf16 hi + lo.
//   Qg = diag(exp(Gam_r)) Q: MMA1's B operand takes the raw query rows (TMA map tq) in place of
//     Qg, and P Delta accumulates in its own TMEM columns (the record's P carries rq), so that
//     the output is O[r] = rq_r exp(Gam_r) (Q S^T)[r] + (P Delta)[r]; exp(Gam_C) is
//     channel-independent, so the record's exp(Gam_C) row keeps it in entries 0..63 and
//     rq_r exp(Gam_r) in 64..127.
// The general gate uses the record's Qg and tf32 Kd^T; tk and tq are unused.
template <bool SG>
__global__ __launch_bounds__(SC_THREADS, 1) void scan_kernel(const __grid_constant__ CUtensorMap tk,
                                                             const __grid_constant__ CUtensorMap tq,
                                                             const ScanParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = aligned_smem<1024>(smem_raw);
    grid_dep_wait();   // the chunk records of the intra-chunk kernel
    if (p.hdr[1] == 0) return;
    const int vb = blockIdx.x & 1;
    const int h = p.h0 + (blockIdx.x >> 1) % p.Hw;
    const int rank = (blockIdx.x >> 1) / p.Hw;
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
        // one arrival per epilogue warp (lane 0, after the warp's proxy fences and a warp sync)
        mbar_init(bar + 8 * BAR_SBR, SC_EPI / 32);
        mbar_init(bar + 8 * BAR_DTR, SC_EPI / 32);
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
    const uint32_t tP0 = tmem + 320;  // scalar gate: P Delta, two buffers of 64 columns

    auto rec_of = [&](int c) { return p.rec + (((size_t)sd.chunk0 + c) * p.Hw + (h - p.h0)) * REC_BYTES; };
    auto fail = [&]() {
        set_status(KDA_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == SC_EPI / 32) {
        // ------------------------------------------------------------ issuer
        if (lane == 0) {
            auto issue_wq = [&](int c) {
                const uint32_t b = bar + 8 * (BAR_WQ0 + (c & 1)), dst = sbase + SS_WQ + (c & 1) * 32768;
                mbar_expect_tx(b, 32768);
                if constexpr (SG) {
                    // [Q; W]: the raw query rows (one 64-channel box per K atom) and the record's W
                    const int hq = h / (p.H_v / p.H_qk), row = sd.tok + c * CH;
                    const unsigned char *r = rec_of(c);
                    tma_load_3d(dst, &tq, 0, hq, row, b);
                    tma_load_3d(dst + 16384, &tq, 64, hq, row, b);
                    bulk_g2s(dst + 8192, r + REC_WQ + 8192, 8192, b);
                    bulk_g2s(dst + 16384 + 8192, r + REC_WQ + 16384 + 8192, 8192, b);
                } else {
                    bulk_g2s(dst, rec_of(c) + REC_WQ, 32768, b);
                }
            };
            auto issue_pk = [&](int c) {
                const unsigned char *r = rec_of(c);
                const uint32_t b = bar + 8 * (BAR_PK0 + (c & 1));
                if constexpr (SG) {
                    // P and the chunk's raw key rows (two 64-channel boxes, 128-byte swizzle: the
                    // MN-major A operand of the state update, M = k)
                    const int hq = h / (p.H_v / p.H_qk), row = sd.tok + c * CH;
                    mbar_expect_tx(b, 8192 + 16384);
                    bulk_g2s(sbase + SS_P + (c & 1) * 8192, r + REC_P, 8192, b);
                    tma_load_3d(sbase + SS_KDT + (c & 1) * 32768, &tk, 0, hq, row, b);
                    tma_load_3d(sbase + SS_KDT + (c & 1) * 32768 + 8192, &tk, 64, hq, row, b);
                } else {
                    mbar_expect_tx(b, 8192 + 32768);
                    bulk_g2s(sbase + SS_P + (c & 1) * 8192, r + REC_P, 8192, b);
                    bulk_g2s(sbase + SS_KDT + (c & 1) * 32768, r + REC_KDT, 32768, b);
                }
            };
            auto issue_u = [&](int c) {
                const unsigned char *r = rec_of(c);
                mbar_expect_tx(bar + 8 * BAR_U, REC_U_BLOCK + 1024);
                bulk_g2s(sbase + SS_U, r + REC_U + vb * REC_U_BLOCK, REC_U_BLOCK, bar + 8 * BAR_U);
                bulk_g2s(sbase + SS_GC, r + REC_GC, 1024, bar + 8 * BAR_U);   // exp(Gam_C), rq, rk
            };
            const uint32_t id1 = idesc_bf16(64, 128) | (1u << 15);   // A (S) MN-major
            const uint32_t id2 = idesc_bf16(64, 64), id3 = idesc_tf32(128, VB);
            const uint32_t id3s = idesc_bf16(128, VB) | (1u << 15);   // A (raw K) MN-major
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
                    if constexpr (SG) {
                        prefetch_l2(r2 + REC_WQ + 8192, 8192);                // W, first K atom
                        prefetch_l2(r2 + REC_WQ + 16384 + 8192, 8192 + 8192);  // W, second atom; P
                        const int hq = h / (p.H_v / p.H_qk), row = sd.tok + (c + 2) * CH;
                        tma_prefetch_3d(&tk, 0, hq, row);
                        tma_prefetch_3d(&tk, 64, hq, row);
                        tma_prefetch_3d(&tq, 0, hq, row);
                        tma_prefetch_3d(&tq, 64, hq, row);
                    } else {
                        prefetch_l2(r2 + REC_WQ, 32768 + 8192 + 32768);
                    }
                    prefetch_l2(r2 + REC_U + vb * REC_U_BLOCK, REC_U_BLOCK);
                    prefetch_l2(r2 + REC_GC, 1024);
                }
                if (!mbar_wait(bar + 8 * BAR_DTR, c & 1)) { fail(); break; }
                if (!mbar_wait(bar + 8 * (BAR_PK0 + b), pp)) { fail(); break; }
                if constexpr (SG) {
                    const int lenc = min(CH, sd.len - c * CH);
                    if (lenc < CH) {
                        // key rows past the chunk's length belong to the next sequence: zero them, so
                        // that they contribute exact zeros whatever they hold (their f Delta rows are 0)
                        unsigned char *kt = sm + SS_KDT + b * 32768;
                        for (int i = lenc * 8; i < CH * 8; ++i) {
                            *reinterpret_cast<uint4 *>(kt + 16 * i) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4 *>(kt + 8192 + 16 * i) = make_uint4(0, 0, 0, 0);
                        }
                        fence_async_smem();
                    }
                    tc_fence_after();
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int ks = 0; ks < CH / 16; ++ks)
                            umma_bf16(tZ, umma_desc(sbase + SS_KDT + b * 32768 + ks * 2048, 8192, 1024),
                                      umma_desc(sbase + SS_DT + part * 8192 + ks * 32, 16, 1024), id3s,
                                      (part > 0 || ks > 0) ? 1u : 0u);
                } else {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < CH / 8; ++ks) {
                        const int kb = ks * 32;
                        umma_tf32(tZ, umma_desc(sbase + SS_KDT + b * 32768 + (kb >> 7) * 16384 + (kb & 127), 16, 1024),
                                  umma_desc(sbase + SS_DT + (kb >> 7) * 8192 + (kb & 127), 16, 1024), id3, ks > 0);
                    }
                }
                umma_commit(bar + 8 * BAR_MMA3);
                // P Delta onto Qg S^T (general gate) or into its own accumulator (scalar gate)
#pragma unroll
                for (int ks = 0; ks < CH / 16; ++ks) {
                    umma_bf16(SG ? tP0 + b * 64 : tY, umma_desc(sbase + SS_DTB + ks * 32, 16, 1024),
                              umma_desc(sbase + SS_P + b * 8192 + ks * 32, 16, 1024), id2, (SG && ks == 0) ? 0u : 1u);
                }
                umma_commit(bar + 8 * BAR_MMA2);
                // the U buffer is free once Delta of chunk c is written (after the MMAs: off the chain)
                if (c + 1 < n) issue_u(c + 1);
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
        for (int v = 0; v < VH; ++v)
            S[v] = !p.init ? 0.f
                 : p.state_bf16 ? bf16_to_f(reinterpret_cast<const uint16_t *>(p.init)[st0 + (size_t)v * KD])
                                : p.init[st0 + (size_t)v * KD];
        const int q = warp & 3;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int vme = q * 16 + lane;      // v owned in the M = 64 layout (lane < 16)
        const bool vact = lane < 16;
        auto emit_output = [&](int cc) {
            if (!mbar_spin(bar + 8 * BAR_MMA2, cc & 1)) fail();
            tc_fence_after();
            const uint32_t tY = tmem + (cc & 1) * 128;
            uint32_t y0[32];
            tmem_ld32_nowait(tY + lane_off + 32 * vhalf, y0);
            uint16_t *os = reinterpret_cast<uint16_t *>(sm + SS_OS);
            if constexpr (SG) {
                // O[r][v] = rq_r exp(Gam_r) (Q S^T)^T[v][r] + (P Delta)^T[v][r]  (the record's P carries rq)
                uint32_t y2[32];
                tmem_ld32_nowait(tP0 + (cc & 1) * 64 + lane_off + 32 * vhalf, y2);
                tmem_wait_ld();
                const float *rqe = reinterpret_cast<const float *>(sm + SS_RQE) + 32 * vhalf;
                if (vact) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 fe = *reinterpret_cast<const float4 *>(rqe + j);
                        const float fb[4] = {fe.x, fe.y, fe.z, fe.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            os[(32 * vhalf + j + i) * VB + vme] =
                                f_to_bf16(fmaf(__uint_as_float(y0[j + i]), fb[i], __uint_as_float(y2[j + i])));
                    }
                }
            } else {
                tmem_wait_ld();
                const float *rq = reinterpret_cast<const float *>(sm + SS_RQ) + 32 * vhalf;
                if (vact) {
                    // the record's Qg and P carry 1 / rq_r: O[r][v] = rq_r Y^T[v][r]
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 f = *reinterpret_cast<const float4 *>(rq + j);
                        os[(32 * vhalf + j) * VB + vme] = f_to_bf16(__uint_as_float(y0[j]) * f.x);
                        os[(32 * vhalf + j + 1) * VB + vme] = f_to_bf16(__uint_as_float(y0[j + 1]) * f.y);
                        os[(32 * vhalf + j + 2) * VB + vme] = f_to_bf16(__uint_as_float(y0[j + 2]) * f.z);
                        os[(32 * vhalf + j + 3) * VB + vme] = f_to_bf16(__uint_as_float(y0[j + 3]) * f.w);
                    }
                }
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
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + 8 * BAR_SBR);
            // ---- previous chunk's output, while MMA1 of this chunk runs
            if (c > 0) emit_output(c - 1);
            // ---- Delta^T = U^T - (W S^T)^T, as tf32 (B of MMA3) and bf16 (A of MMA2)
            if (!mbar_spin(bar + 8 * BAR_MMA1, c & 1) || !mbar_spin(bar + 8 * BAR_U, c & 1)) fail();
            tc_fence_after();
            const float g = reinterpret_cast<const float *>(sm + SS_GC)[SG ? 0 : kme];
            // keep this chunk's rq (and, scalar gate, rq exp(Gam_r)) for its output, emitted during
            // the next chunk (the record area is reloaded before that)
            if (tid < CH) {
                reinterpret_cast<float *>(sm + SS_RQ)[tid] = reinterpret_cast<const float *>(sm + SS_GC)[128 + tid];
                if (SG) reinterpret_cast<float *>(sm + SS_RQE)[tid] = reinterpret_cast<const float *>(sm + SS_GC)[64 + tid];
            }
            {
                // this thread: v = vme, r = 32 vhalf .. 32 vhalf + 31
                uint32_t ys[32];
                tmem_ld32_nowait(tY + lane_off + 64 + 32 * vhalf, ys);
                tmem_wait_ld();
                if (vact) {
                    const float *urow = reinterpret_cast<const float *>(sm + SS_U) + vme * 68 + 32 * vhalf;
                    // Kd in the record is unnormalised: the state update takes Delta_r rk_r (scalar gate:
                    // Delta_r f_r, the record's rk slot holding f_r = rk_r exp(Gam_C - Gam_r))
                    const float *rkr = reinterpret_cast<const float *>(sm + SS_GC) + 192 + 32 * vhalf;
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 8) {
                        const int j = 32 * vhalf + jj;
                        const float4 ua = *reinterpret_cast<const float4 *>(urow + jj);
                        const float4 ub = *reinterpret_cast<const float4 *>(urow + jj + 4);
                        // Delta = U - Y and its scaled copy, on packed fp32 pairs
                        const float2 m1 = make_float2(-1.f, -1.f);
                        const float2 p01 = __ffma2_rn(make_float2(__uint_as_float(ys[jj + 0]), __uint_as_float(ys[jj + 1])), m1,
                                                      make_float2(ua.x, ua.y));
                        const float2 p23 = __ffma2_rn(make_float2(__uint_as_float(ys[jj + 2]), __uint_as_float(ys[jj + 3])), m1,
                                                      make_float2(ua.z, ua.w));
                        const float2 p45 = __ffma2_rn(make_float2(__uint_as_float(ys[jj + 4]), __uint_as_float(ys[jj + 5])), m1,
                                                      make_float2(ub.x, ub.y));
                        const float2 p67 = __ffma2_rn(make_float2(__uint_as_float(ys[jj + 6]), __uint_as_float(ys[jj + 7])), m1,
                                                      make_float2(ub.z, ub.w));
                        const float d0 = p01.x, d1 = p01.y, d2 = p23.x, d3 = p23.y, d4 = p45.x, d5 = p45.y, d6 = p67.x,
                                    d7 = p67.y;
                        const float4 ka = *reinterpret_cast<const float4 *>(rkr + jj);
                        const float4 kb = *reinterpret_cast<const float4 *>(rkr + jj + 4);
                        const float2 e01 = __fmul2_rn(p01, make_float2(ka.x, ka.y)), e23 = __fmul2_rn(p23, make_float2(ka.z, ka.w));
                        const float2 e45 = __fmul2_rn(p45, make_float2(kb.x, kb.y)), e67 = __fmul2_rn(p67, make_float2(kb.z, kb.w));
                        if constexpr (SG) {
                            // f Delta as bf16 hi (SS_DT) + lo (SS_DT + 8 KiB): 64 rows (v) x 64 (r), K-major
                            const float e[8] = {e01.x, e01.y, e23.x, e23.y, e45.x, e45.y, e67.x, e67.y};
                            uint32_t hi[4], lo[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                hi[i] = pack_bf16x2(e[2 * i], e[2 * i + 1]);
                                lo[i] = pack_bf16x2(e[2 * i] - bf16_lo(hi[i]), e[2 * i + 1] - bf16_hi(hi[i]));
                            }
                            const uint32_t off = sw128_off(vme, 2 * j, VB);
                            *reinterpret_cast<uint4 *>(sm + SS_DT + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                            *reinterpret_cast<uint4 *>(sm + SS_DT + 8192 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        } else {
                            *reinterpret_cast<uint4 *>(sm + SS_DT + sw128_off(vme, 4 * j, VB)) =
                                make_uint4(tf32_rn_bits(e01.x), tf32_rn_bits(e01.y), tf32_rn_bits(e23.x), tf32_rn_bits(e23.y));
                            *reinterpret_cast<uint4 *>(sm + SS_DT + sw128_off(vme, 4 * j + 16, VB)) =
                                make_uint4(tf32_rn_bits(e45.x), tf32_rn_bits(e45.y), tf32_rn_bits(e67.x), tf32_rn_bits(e67.y));
                        }
                        *reinterpret_cast<uint4 *>(sm + SS_DTB + sw128_off(vme, 2 * j, VB)) =
                            make_uint4(pack_bf16x2(d0, d1), pack_bf16x2(d2, d3), pack_bf16x2(d4, d5),
                                       pack_bf16x2(d6, d7));
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + 8 * BAR_DTR);
            // ---- S = S * exp(Gam_C) + Z   (lanes k of Z, columns v of this half)
            if (!mbar_spin(bar + 8 * BAR_MMA3, c & 1)) fail();
            tc_fence_after();
            {
                uint32_t z0[32];
                tmem_ld32_nowait(tZ + lane_off + 32 * vhalf, z0);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float2 r = __ffma2_rn(make_float2(S[j], S[j + 1]), make_float2(g, g),
                                                make_float2(__uint_as_float(z0[j]), __uint_as_float(z0[j + 1])));
                    S[j] = r.x;
                    S[j + 1] = r.y;
                }
            }
            tc_fence_before();
        }
        if (!*abort_flag && n > 0) emit_output(n - 1);
        if (p.fin && !*abort_flag) {
            if (p.state_bf16) {
                uint16_t *dst = reinterpret_cast<uint16_t *>(p.fin) + st0;
#pragma unroll
                for (int v = 0; v < VH; ++v) dst[(size_t)v * KD] = f_to_bf16(S[v]);
            } else {
                float *dst = p.fin + st0;
#pragma unroll
                for (int v = 0; v < VH; ++v) dst[(size_t)v * KD] = S[v];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}


// W (M = 64 accumulator at t_w, 128 columns) to the W rows of the WQ image (bf16, two 8 KiB
// atoms at ws) and U^T (M = 128 accumulator at t_u, 64 columns, lane v) to the U image
// [v / 64][v % 64][68] fp32 at us.  Warps 0..3 take U, 4..7 take W.
__device__ __forceinline__ void store_wu(unsigned char *ws, unsigned char *us, uint32_t t_w, uint32_t t_u, int warp,
                                         int lane) {
    const int q = warp & 3;
    const uint32_t lo = (uint32_t)(q * 32) << 16;
    if (warp < 4) {
        const int v = q * 32 + lane;
        uint32_t x0[32], x1[32];
        tmem_ld32_nowait(t_u + lo, x0);
        tmem_ld32_nowait(t_u + lo + 32, x1);
        tmem_wait_ld();
        float *u = reinterpret_cast<float *>(us) + (v >> 6) * (CH * 68) + (v & 63) * 68;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            *reinterpret_cast<float4 *>(u + j) = make_float4(__uint_as_float(x0[j]), __uint_as_float(x0[j + 1]),
                                                             __uint_as_float(x0[j + 2]), __uint_as_float(x0[j + 3]));
            *reinterpret_cast<float4 *>(u + 32 + j) = make_float4(__uint_as_float(x1[j]), __uint_as_float(x1[j + 1]),
                                                                  __uint_as_float(x1[j + 2]), __uint_as_float(x1[j + 3]));
        }
    } else {
        const int r = q * 16 + lane;
#pragma unroll
        for (int rd = 0; rd < 2; ++rd) {
            uint32_t x0[32], x1[32];
            tmem_ld32_nowait(t_w + lo + 64 * rd, x0);
            tmem_ld32_nowait(t_w + lo + 64 * rd + 32, x1);
            tmem_wait_ld();
            if (lane < 16) {
#pragma unroll
                for (int j = 0; j < 64; j += 8) {
                    const uint32_t *xs = j < 32 ? x0 : x1;
                    const int jj = j & 31, k = 64 * rd + j;
                    const uint32_t off = (uint32_t)rd * 8192 + (r >> 3) * 1024 + (r & 7) * 128 +
                                         ((((2 * k) & 127) >> 4) ^ (r & 7)) * 16;
                    *reinterpret_cast<uint4 *>(ws + off) = make_uint4(
                        pack_bf16x2(__uint_as_float(xs[jj]), __uint_as_float(xs[jj + 1])),
                        pack_bf16x2(__uint_as_float(xs[jj + 2]), __uint_as_float(xs[jj + 3])),
                        pack_bf16x2(__uint_as_float(xs[jj + 4]), __uint_as_float(xs[jj + 5])),
                        pack_bf16x2(__uint_as_float(xs[jj + 6]), __uint_as_float(xs[jj + 7])));
                }
            }
        }
    }
}

// =====================================================================
// Intra-chunk kernel for a scalar gate (one decay per token and value head,
// graw [B, T, H_v]): the gated-delta-net special case.  The decay
// exp(Gam_r - Gam_j) is then the same for every channel, so
//   A[r,j] = beta_r rk_r rk_j exp(Gam_r - Gam_j) (k_r . k_j),   P[r,j] = rq_r rk_j exp(Gam_r - Gam_j) (q_r . k_j)
// come from one bf16 MMA of the raw inputs (exact products, fp32 accumulate)
// followed by a 64 x 64 decay mask, and W = T diag(beta rk exp(Gam)) K takes the
// staged raw K as its operand.  The record is the general kernel's without Kd^T and
// Qg, both row scalings of the raw inputs (Kd = diag(f) K with f_r = rk_r
// exp(Gam_C - Gam_r), Qg = diag(exp(Gam_r)) Q): it carries f in the rk slot,
// rq_r exp(Gam_r) in the upper half of the exp(Gam_C) row and P with its factor rq,
// and the scan's scalar-gate variant reads the key and query rows of the input itself.
// Persistent CTAs of 8 warps, two per SM, one (chunk, value head) item at a time.
// =====================================================================
constexpr uint32_t GD_QK = 0;               // [K rows 0..63; Q rows 64..127] K-major bf16 (2 x 16 KiB atoms);
                                            // after the A/P MMA: V (MN-major, 16 KiB) and K (MN-major, 16 KiB)
constexpr uint32_t GD_V = GD_QK, GD_KMN = GD_QK + 16384;
constexpr uint32_t GD_AT = 32768;           // A, T fp32 [64][68] and the inversion scratch; then U staging
constexpr uint32_t GD_A = GD_AT, GD_T = GD_AT + 17408, GD_X = GD_AT + 34816;
constexpr uint32_t GD_TP = 73728;           // T'_hi, T'_lo, T'_W hi, T'_W lo (4 x 8 KiB); the P image before them;
                                            // then W staging
constexpr uint32_t GD_PI = GD_TP, GD_TPH = GD_TP, GD_TPL = GD_TP + 8192, GD_TWH = GD_TP + 16384, GD_TWL = GD_TP + 24576;
constexpr uint32_t GD_MISC = 106496;
constexpr uint32_t GD_RV = GD_MISC;         // rq, rk, beta, raw q.k [4][64]
constexpr uint32_t GD_GAM = GD_MISC + 1024; // Gam [64] (log2 units)
constexpr uint32_t GD_EG = GD_MISC + 1280;  // exp(Gam) [64]
constexpr uint32_t GD_GCS = GD_MISC + 1536; // exp(Gam_C) [128] (the record's per-channel layout)
constexpr uint32_t GD_SCR = GD_MISC + 2048; // gate-scan carry
constexpr uint32_t GD_BAR = GD_MISC + 2112; // 2 mbarriers
constexpr uint32_t GD_SLOT = GD_MISC + 2128;
constexpr uint32_t GD_BYTES = GD_MISC + 2144 + 1024;
static_assert(GD_X + 32 * XS * 4 <= GD_TP && GD_TWL + 8192 <= GD_MISC, "scalar-gate layout overflow");
static_assert(IN_CTAS_PER_SM * (GD_BYTES + 1024) <= 228 * 1024, "two CTAs per SM must fit");

struct GdnParams {
    const uint16_t *q, *k, *v, *graw, *b;   // graw [B, T, H_v]
    const float *A_log;
    float scale;
    int H_qk, H_v;
    const ChunkDesc *chunks;
    const int *hdr;
    unsigned char *rec;                     // [chunk][H_v] records of REC_BYTES
};

__global__ __launch_bounds__(IN_THREADS, IN_CTAS_PER_SM) void intra_gdn_kernel(const GdnParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = aligned_smem<1024>(smem_raw);
    grid_dep_wait();
    grid_dep_launch();
    if (p.hdr[1] == 0) return;
    const long long n_items = (long long)p.hdr[0] * p.H_v;
    if ((long long)blockIdx.x >= n_items) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar_ap = sbase + GD_BAR, bar_wu = sbase + GD_BAR + 8;
    const uint64_t pol_ef = l2_evict_first_policy();
    float *rv = reinterpret_cast<float *>(sm + GD_RV);
    float *gam = reinterpret_cast<float *>(sm + GD_GAM);
    float *eg = reinterpret_cast<float *>(sm + GD_EG);
    float *gcs = reinterpret_cast<float *>(sm + GD_GCS);
    float *sA = reinterpret_cast<float *>(sm + GD_A);
    float *sT = reinterpret_cast<float *>(sm + GD_T);
    float *sX = reinterpret_cast<float *>(sm + GD_X);
    if (tid == 0) {
        mbar_init(bar_ap, 1);
        mbar_init(bar_wu, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(sbase + GD_SLOT, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + GD_SLOT);
    const uint32_t t_ap = tmem, t_w = tmem, t_u = tmem + 128;
    const size_t qk_stride = (size_t)p.H_qk * KD, gv_stride = (size_t)p.H_v * KD;
    const int group = p.H_v / p.H_qk;

    int it = 0;
    for (long long item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
        const int chunk = (int)(item / p.H_v), h = (int)(item % p.H_v), hq = h / group;
        const ChunkDesc cd = p.chunks[chunk];
        const int len = cd.len;
        unsigned char *rec = p.rec + ((size_t)chunk * p.H_v + h) * REC_BYTES;
        const uint16_t *qrow = p.q + ((size_t)cd.tok * p.H_qk + hq) * KD;   // row r at + r * qk_stride
        const uint16_t *krow = p.k + ((size_t)cd.tok * p.H_qk + hq) * KD;
        const uint16_t *vrow = p.v + ((size_t)cd.tok * p.H_v + h) * KD;     // row r at + r * gv_stride

        // ---- 1. raw K and Q rows into the [K; Q] operand (16-byte units, zero rows past len); the
        //         gate scalars and beta
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = tid + IN_THREADS * i, isq = idx >> 10, r = (idx >> 4) & 63, u = idx & 15;
            unsigned char *dst = sm + GD_QK + sw128_off(64 * isq + r, 16 * u, 2 * CH);
            if (r < len) cp_async16(dst, (isq ? qrow : krow) + r * qk_stride + 8 * u);
            else *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
        }
        cp_async_commit();
        float graw_r = 0.f, b_r = 0.f;
        if (tid < len) {
            const size_t row = ((size_t)cd.tok + tid) * p.H_v + h;
            graw_r = bf16_to_f(p.graw[row]);
            b_r = bf16_to_f(p.b[row]);
        }
        cp_async_wait<0>();
        // the previous item's bulk stores must be done reading shared memory (staging, P, tables)
        if (tid == 0) bulk_wait_read_all();
        __syncthreads();

        // ---- 2. row norms from the staged rows (thread: row, quarter of the channels); gate and
        //         its prefix sum over the chunk (warps 0, 1: one row per lane)
        {
            const int r = tid >> 2, part = tid & 3;
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int ub = 16 * (4 * part + u);
                const uint4 kw = *reinterpret_cast<const uint4 *>(sm + GD_QK + sw128_off(r, ub, 2 * CH));
                const uint4 qw = *reinterpret_cast<const uint4 *>(sm + GD_QK + sw128_off(64 + r, ub, 2 * CH));
                const uint32_t ka[4] = {kw.x, kw.y, kw.z, kw.w}, qa[4] = {qw.x, qw.y, qw.z, qw.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float k0 = bf16_lo(ka[e]), k1 = bf16_hi(ka[e]), q0 = bf16_lo(qa[e]), q1 = bf16_hi(qa[e]);
                    sq = fmaf(q0, q0, fmaf(q1, q1, sq));
                    sk = fmaf(k0, k0, fmaf(k1, k1, sk));
                }
            }
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            if (part == 0) {
                rv[RV_RQ + r] = p.scale * rsqrtf(sq + L2_EPS);
                rv[RV_RK + r] = rsqrtf(sk + L2_EPS);
            }
        }
        if (warp < 2) {
            const float a_gate = ex2(p.A_log[h] * LOG2E);
            float g2 = tid < len ? -a_gate * softplus_log2(graw_r) : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, g2, o);
                if (lane >= o) g2 += y;
            }
            if (tid == 31) reinterpret_cast<float *>(sm + GD_SCR)[0] = g2;
            named_bar(1, 64);
            if (warp == 1) g2 += reinterpret_cast<const float *>(sm + GD_SCR)[0];
            gam[tid] = g2;
            eg[tid] = ex2(g2);
            rv[RV_BETA + tid] = tid < len ? 1.0f / (1.0f + ex2(-b_r * LOG2E)) : 0.f;
            if (tid == CH - 1) reinterpret_cast<float *>(sm + GD_SCR)[1] = ex2(g2);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- 3. D[m][j] = [K; Q][m] . K[j]  (M = 128, N = 64, K = 128, bf16, raw inputs)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
            for (int ks = 0; ks < KD / 16; ++ks) {
                const uint32_t a = sbase + GD_QK + (ks >> 2) * 16384 + (ks & 3) * 32;
                umma_bf16(t_ap, umma_desc(a, 16, 1024), umma_desc(a, 16, 1024), id, ks > 0 ? 1u : 0u);
            }
            umma_commit(bar_ap);
        }
        // ---- 4. meanwhile, the scan's row factors (Qg and Kd are row scalings of the raw q and k,
        //         which the scan reads itself): the record's exp(Gam_C) row holds exp(Gam_C) in entries
        //         0..63 and rq_r exp(Gam_r) in 64..127; f_r = rk_r exp(Gam_C - Gam_r) (0 past len) goes
        //         to the slot of the raw q.k (unused here), stored in the record's rk slot
        if (tid < CH) gcs[tid] = reinterpret_cast<const float *>(sm + GD_SCR)[1];
        else if (tid < 2 * CH) gcs[tid] = rv[RV_RQ + tid - CH] * eg[tid - CH];
        if (tid < CH) rv[RV_QK + tid] = tid < len ? rv[RV_RK + tid] * ex2(gam[CH - 1] - gam[tid]) : 0.f;
        if (tid == 0 && !mbar_spin(bar_ap, it & 1)) set_status(KDA_ERR_DEVICE_TIMEOUT);
        __syncthreads();
        tc_fence_after();
        // the [K; Q] operand is free: V and K (MN-major) for the W / U MMAs
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = tid + IN_THREADS * i, isk = idx >> 10, r = (idx >> 4) & 63, c8 = (idx & 15) * 8;
            unsigned char *dst = sm + (isk ? GD_KMN : GD_V) + mn_off_bf16(c8, r);
            if (r < len) cp_async16(dst, (isk ? krow + r * qk_stride : vrow + r * gv_stride) + c8);
            else *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
        }
        cp_async_commit();

        // ---- 5. A and P from TMEM with the decay mask.  M = 128 layout: row m in lane m; warp w
        //         reads lanes 32 (w & 3) .. (rows of K for w & 3 < 2, of Q otherwise), columns 32 (w >> 2) ..
        {
            const int q = warp & 3, hf = warp >> 2, isq = q >> 1, r = 32 * (q & 1) + lane;
            const uint32_t lo = (uint32_t)(q * 32) << 16;
            uint32_t x[32];
            tmem_ld32_nowait(t_ap + lo + 32 * hf, x);
            tmem_wait_ld();
            const float gr = gam[r];
            // row scale: rq for P (the scan adds P Delta unscaled), beta rk for A
            const float rs = isq ? rv[RV_RQ + r] : rv[RV_BETA + r] * rv[RV_RK + r];
            float o[32];
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
                const int j = 32 * hf + jj;
                const float4 gj = *reinterpret_cast<const float4 *>(gam + j);
                const float4 kj = *reinterpret_cast<const float4 *>(rv + RV_RK + j);
                const float gv[4] = {gj.x, gj.y, gj.z, gj.w}, kv[4] = {kj.x, kj.y, kj.z, kj.w};
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    // packed fp32 pairs: D e^(Gam_r - Gam_j) rs rk_j for columns j + e, j + e + 1
                    const float2 v = __fmul2_rn(
                        __fmul2_rn(make_float2(__uint_as_float(x[jj + e]), __uint_as_float(x[jj + e + 1])),
                                   make_float2(ex2(gr - gv[e]), ex2(gr - gv[e + 1]))),
                        __fmul2_rn(make_float2(rs, rs), make_float2(kv[e], kv[e + 1])));
                    o[jj + e] = (isq ? (j + e <= r) : (j + e < r)) ? v.x : 0.f;
                    o[jj + e + 1] = (isq ? (j + e + 1 <= r) : (j + e + 1 < r)) ? v.y : 0.f;
                }
            }
            if (!isq) {
#pragma unroll
                for (int jj = 0; jj < 32; jj += 4)
                    *reinterpret_cast<float4 *>(sA + r * AS + 32 * hf + jj) = make_float4(o[jj], o[jj + 1], o[jj + 2], o[jj + 3]);
            } else {
#pragma unroll
                for (int jj = 0; jj < 32; jj += 8)
                    *reinterpret_cast<uint4 *>(sm + GD_PI + sw128_off(r, 2 * (32 * hf + jj), CH)) =
                        make_uint4(pack_bf16x2(o[jj], o[jj + 1]), pack_bf16x2(o[jj + 2], o[jj + 3]),
                                   pack_bf16x2(o[jj + 4], o[jj + 5]), pack_bf16x2(o[jj + 6], o[jj + 7]));
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            bulk_s2g_hint(rec + REC_P, sbase + GD_PI, 8192, pol_ef);
            bulk_s2g_hint(rec + REC_GC, sbase + GD_GCS, 512, pol_ef);
            bulk_s2g_hint(rec + REC_RN, sbase + GD_RV + 4 * RV_RQ, 256, pol_ef);         // rq
            bulk_s2g_hint(rec + REC_RN + 256, sbase + GD_RV + 4 * RV_QK, 256, pol_ef);   // f, in the rk slot
            bulk_commit();
        }

        // ---- 6. T = (I + A)^{-1}
        invert_unit_lower64<IN_THREADS>(sA, sT, sX, tid, warp, lane);
        // the P image store must be done reading before T' overwrites it
        if (tid == 0) bulk_wait_read_all();
        __syncthreads();
        // T' = T diag(beta) (for U) and T'_W = T diag(beta rk exp(Gam)) (for W on the raw K)
        for (int idx = tid; idx < CH * (CH / 8); idx += IN_THREADS) {
            const int r = idx >> 3, j = (idx & 7) * 8;
            uint32_t hi[4], lo[4], hw[4], lw[4];
            // packed fp32 pairs: x = T beta, xw = x rk exp(Gam), and the hi / lo splits
            const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const float2 x2 = __fmul2_rn(*reinterpret_cast<const float2 *>(sT + r * AS + j + e),
                                             *reinterpret_cast<const float2 *>(rv + RV_BETA + j + e));
                const float2 xw2 = __fmul2_rn(__fmul2_rn(x2, *reinterpret_cast<const float2 *>(rv + RV_RK + j + e)),
                                              *reinterpret_cast<const float2 *>(eg + j + e));
                const uint32_t h2 = pack_bf16x2(x2.x, x2.y);
                hi[e >> 1] = h2;
                const float2 l2 = __ffma2_rn(make_float2(bf16_lo(h2), bf16_hi(h2)), m1, x2);
                lo[e >> 1] = pack_bf16x2(l2.x, l2.y);
                const uint32_t w2 = pack_bf16x2(xw2.x, xw2.y);
                hw[e >> 1] = w2;
                const float2 lw2 = __ffma2_rn(make_float2(bf16_lo(w2), bf16_hi(w2)), m1, xw2);
                lw[e >> 1] = pack_bf16x2(lw2.x, lw2.y);
            }
            const uint32_t off = sw128_off(r, 2 * j, CH);
            *reinterpret_cast<uint4 *>(sm + GD_TPH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(sm + GD_TPL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<uint4 *>(sm + GD_TWH + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(sm + GD_TWL + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        cp_async_wait<0>();   // V and K (this thread's copies)
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- 7. W = T'_W K (M = 64, N = 128, B = K MN-major) and U^T = V T'^T (M = 128 over v, N = 64)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_w = idesc_bf16(64, 128) | (1u << 16);
            const uint32_t id_u = idesc_bf16(128, 64) | (1u << 15);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < CH / 16; ++ks) {
                    const uint64_t tp = umma_desc(sbase + (part ? GD_TPL : GD_TPH) + ks * 32, 16, 1024);
                    const uint64_t tw = umma_desc(sbase + (part ? GD_TWL : GD_TWH) + ks * 32, 16, 1024);
                    const uint32_t acc = (part > 0 || ks > 0) ? 1u : 0u;
                    umma_bf16(t_w, tw, umma_desc(sbase + GD_KMN + ks * 2048, 8192, 1024), id_w, acc);
                    umma_bf16(t_u, umma_desc(sbase + GD_V + ks * 2048, 8192, 1024), tp, id_u, acc);
                }
            umma_commit(bar_wu);
            if (!mbar_spin(bar_wu, it & 1)) set_status(KDA_ERR_DEVICE_TIMEOUT);
        }
        __syncthreads();
        tc_fence_after();
        store_wu(sm + GD_TP, sm + GD_AT, t_w, t_u, warp, lane);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            bulk_s2g_hint(rec + REC_WQ + 8192, sbase + GD_TP, 8192, pol_ef);
            bulk_s2g_hint(rec + REC_WQ + 16384 + 8192, sbase + GD_TP + 8192, 8192, pol_ef);
            bulk_s2g_hint(rec + REC_U, sbase + GD_AT, 2 * CH * 68 * 4, pol_ef);
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
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

// Launch with programmatic stream serialisation: the kernel may be scheduled while the previous
// kernel on the stream runs, and waits for it with grid_dep_wait() before touching its results.
template <typename... KArgs, typename... Args>
static cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                    Args &&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

void timing_begin(cudaStream_t s);
void timing_mark(const char *name, cudaStream_t s);

cudaError_t launch_plan(const int32_t *cu, int N, int B, int T, SeqDesc *seqs, ChunkDesc *chunks, int *order,
                        int *hdr, long long max_chunks, cudaStream_t stream) {
    plan_kernel<<<1, PLAN_THREADS, 0, stream>>>(cu, N, B, T, seqs, chunks, order, hdr, max_chunks);
    return cudaGetLastError();
}

long long max_chunks_for(int N, int B, int T, bool varlen) {
    if (varlen) return (long long)T / CH + (long long)N + 1;
    return (long long)B * (((long long)T + CH - 1) / CH);
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

// Forward for the value heads [h0, h0 + Hw) of the tensors (strides from H_qk, H_v); the
// workspace holds records for Hw heads.  With plan == false the chunk tables already in the
// workspace (from an earlier call on the same sequences) are reused.
static cudaError_t launch_fwd_impl(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                                   const uint16_t *b, const float *A_log, float scale, const float *init, float *fin,
                                   const int32_t *cu, int N, int B, int T, int H_qk, int H_v, int h0, int Hw,
                                   bool plan, uint16_t *out, void *ws_ptr, cudaStream_t stream, int *launches,
                                   bool state_bf16) {
    const bool varlen = cu != nullptr;
    const int nseq = varlen ? N : B;
    FwdWorkspace ws;
    fwd_workspace_bytes(N, B, T, Hw, varlen, &ws, (char *)ws_ptr);
    const long long nck = max_chunks_for(N, B, T, varlen);
    *launches = 0;
    {
        cudaError_t e = cudaFuncSetAttribute(intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)IS_BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(scan_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SS_BYTES);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaSuccess;
    timing_begin(stream);
    if (plan) {
        plan_kernel<<<1, PLAN_THREADS, 0, stream>>>(cu, N, B, T, ws.seqs, ws.chunks, ws.order, ws.hdr, nck);
        ++*launches;
        timing_mark("plan_kernel", stream);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const long long rows = (long long)B * T;
    if (nck > 0 && rows > 0) {
        // raw slices of q, k, graw: 32 channels x 64 rows (64-byte swizzle); V: 64 channels x 64 rows
        // (128-byte swizzle, the MN-major operand layout of the U MMA)
        CUtensorMap mq, mk, mg, mv;
        if ((e = tma_map_rows_heads(&mq, q, rows, H_qk, SL, CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess) return e;
        if ((e = tma_map_rows_heads(&mk, k, rows, H_qk, SL, CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess) return e;
        if ((e = tma_map_rows_heads(&mg, graw, rows, H_v, SL, CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess) return e;
        if ((e = tma_map_rows_heads(&mv, v, rows, H_v, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
        IntraParams ip;
        ip.q = q; ip.k = k; ip.v = v; ip.graw = graw; ip.b = b; ip.A_log = A_log; ip.scale = scale;
        ip.H_qk = H_qk; ip.H_v = H_v; ip.h0 = h0; ip.Hw = Hw; ip.chunks = ws.chunks; ip.hdr = ws.hdr;
        ip.rec = ws.rec;
        int dev = 0, nsm = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        const long long items = nck * (long long)Hw;
        const long long slots = (long long)nsm * IN_CTAS_PER_SM;   // persistent: two CTAs per SM
        const unsigned grid = (unsigned)(items < slots ? items : slots);
        if ((e = launch_dependent(intra_kernel, dim3(grid), dim3(IN_THREADS), IS_BYTES, stream, mq, mk, mg, mv, ip)) !=
            cudaSuccess)
            return e;
        ++*launches;
        timing_mark("intra_kernel", stream);
    }
    if (nseq > 0) {
        ScanParams sp;
        sp.rec = ws.rec;
        sp.seqs = ws.seqs; sp.order = ws.order; sp.hdr = ws.hdr;
        sp.init = init; sp.fin = fin; sp.out = out; sp.H_qk = H_qk; sp.H_v = H_v; sp.nseq = nseq; sp.h0 = h0;
        sp.Hw = Hw;
        sp.state_bf16 = state_bf16 ? 1 : 0;
        const long long nblk = (long long)nseq * Hw * 2;
        const CUtensorMap unused{};   // the general gate reads Kd^T and Qg from the records
        if ((e = launch_dependent(scan_kernel<false>, dim3((unsigned)nblk), dim3(SC_THREADS), SS_BYTES, stream, unused,
                                  unused, sp)) != cudaSuccess)
            return e;
        ++*launches;
        timing_mark("scan_kernel", stream);
    }
    return cudaSuccess;
}

// Forward with a scalar gate per token and value head (graw [B, T, H_v]): plan, the
// scalar-gate intra-chunk kernel, then the common scan.
cudaError_t launch_fwd_scalar_gate(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                                   const uint16_t *b, const float *A_log, float scale, const float *init,
                                   float *fin, const int32_t *cu, int N, int B, int T, int H_qk, int H_v,
                                   uint16_t *out, void *ws_ptr, cudaStream_t stream, int *launches) {
    const bool varlen = cu != nullptr;
    const int nseq = varlen ? N : B;
    FwdWorkspace ws;
    fwd_workspace_bytes(N, B, T, H_v, varlen, &ws, (char *)ws_ptr);
    const long long nck = max_chunks_for(N, B, T, varlen);
    *launches = 0;
    cudaError_t e = cudaFuncSetAttribute(intra_gdn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GD_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SS_BYTES);
    if (e != cudaSuccess) return e;
    timing_begin(stream);
    plan_kernel<<<1, PLAN_THREADS, 0, stream>>>(cu, N, B, T, ws.seqs, ws.chunks, ws.order, ws.hdr, nck);
    ++*launches;
    timing_mark("plan_kernel", stream);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (nck > 0) {
        GdnParams gp;
        gp.q = q; gp.k = k; gp.v = v; gp.graw = graw; gp.b = b; gp.A_log = A_log; gp.scale = scale;
        gp.H_qk = H_qk; gp.H_v = H_v; gp.chunks = ws.chunks; gp.hdr = ws.hdr; gp.rec = ws.rec;
        int dev = 0, nsm = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        const long long items = nck * (long long)H_v, slots = (long long)nsm * IN_CTAS_PER_SM;
        if ((e = launch_dependent(intra_gdn_kernel, dim3((unsigned)(items < slots ? items : slots)), dim3(IN_THREADS),
                                  GD_BYTES, stream, gp)) != cudaSuccess)
            return e;
        ++*launches;
        timing_mark("intra_gdn_kernel", stream);
    }
    if (nseq > 0) {
        ScanParams sp;
        sp.rec = ws.rec;
        sp.seqs = ws.seqs; sp.order = ws.order; sp.hdr = ws.hdr;
        sp.init = init; sp.fin = fin; sp.out = out; sp.H_qk = H_qk; sp.H_v = H_v; sp.nseq = nseq; sp.h0 = 0;
        sp.Hw = H_v;
        sp.state_bf16 = 0;
        // the raw key and query rows: 64 channels x 64 rows per box, 128-byte swizzle
        CUtensorMap mk{}, mq{};
        const long long rows = (long long)B * T;
        if (rows > 0 && ((e = tma_map_rows_heads(&mk, k, rows, H_qk, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess ||
                         (e = tma_map_rows_heads(&mq, q, rows, H_qk, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess))
            return e;
        if ((e = launch_dependent(scan_kernel<true>, dim3((unsigned)((long long)nseq * H_v * 2)), dim3(SC_THREADS),
                                  SS_BYTES, stream, mk, mq, sp)) != cudaSuccess)
            return e;
        ++*launches;
        timing_mark("scan_kernel", stream);
    }
    return cudaSuccess;
}

cudaError_t launch_fwd_heads(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                             const uint16_t *b, const float *A_log, float scale, const float *init, float *fin,
                             const int32_t *cu, int N, int B, int T, int H_qk, int H_v, int h0, int Hw, bool plan,
                             uint16_t *out, void *ws_ptr, cudaStream_t stream, int *launches) {
    return launch_fwd_impl(q, k, v, graw, b, A_log, scale, init, fin, cu, N, B, T, H_qk, H_v, h0, Hw, plan, out, ws_ptr,
                           stream, launches, false);
}

// The forward with the initial and final states stored as bf16.
cudaError_t launch_fwd_bf16_state(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                                  const uint16_t *b, const float *A_log, float scale, const uint16_t *init,
                                  uint16_t *fin, const int32_t *cu, int N, int B, int T, int H_qk, int H_v,
                                  uint16_t *out, void *ws_ptr, cudaStream_t stream, int *launches) {
    return launch_fwd_impl(q, k, v, graw, b, A_log, scale, reinterpret_cast<const float *>(init),
                           reinterpret_cast<float *>(fin), cu, N, B, T, H_qk, H_v, 0, H_v, true, out, ws_ptr, stream,
                           launches, true);
}

cudaError_t launch_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                       const uint16_t *b, const float *A_log, float scale, const float *init, float *fin,
                       const int32_t *cu, int N, int B, int T, int H_qk, int H_v, uint16_t *out, void *ws_ptr,
                       cudaStream_t stream, int *launches) {
    return launch_fwd_heads(q, k, v, graw, b, A_log, scale, init, fin, cu, N, B, T, H_qk, H_v, 0, H_v, true, out,
                            ws_ptr, stream, launches);
}

}  // namespace kda
