// KDA backward: gradients of the forward with respect to q, k, v, graw, b,
// A_log and the initial state, given the gradients of the outputs (do) and of
// the final states (dht).
//
// Per sequence and value head, token t (qt, kh normalised, e = exp(g), beta):
//   S' = S_{t-1} Diag(e),  d = S' kh,  delta = beta (v - d),  S_t = S' + delta kh^T,  o = S_t qt
// and, walking t backwards with dS = dL/dS_t (rows v of the state are
// independent in both directions; only the per-token parameter gradients sum
// over v):
//   dS   += do qt^T                     dqt  = S_t^T do
//   ddel  = dS kh                       dkh  = dS^T delta + S'^T dd,   dd = -beta ddel
//   dv    = beta ddel                   dbeta = ddel . (v - d)
//   dS'   = dS + dd kh^T                de    = colsum(S_{t-1} * dS')
//   dS_{t-1} = dS' Diag(e)
// then the prologue's Jacobians map dqt, dkh, de, dbeta to dq, dk, dgraw,
// dA_log, db (dq and dk sum over the value heads of a query/key group).
//
// bwd_recur_kernel: persistent CTAs of 8 warps, two per SM, one (sequence,
// value head, quarter of the state rows) item at a time: the 128 rows of a
// chain are independent, so four CTAs share a chain.  Warp w owns rows
// 4w .. 4w + 3 of the quarter, lane owns channels 4 lane .. 4 lane + 3, so S and
// dS live in registers (16 values each).  A first pass runs the recurrence and
// stores the state at every 16-token block start; the backward pass then takes
// the blocks in reverse: it recomputes the block's states from its checkpoint
// into a per-CTA scratch area (256 KiB; each thread reads back only what it
// wrote; the scratch of all resident CTAs stays within L2), then walks the
// block's tokens backwards.  The per-token vectors (qt,
// kh, e, v, do, beta) of a block are staged in shared memory; the sums over the
// quarter's rows of dqt, dkh, de and dbeta are reduced across warps through
// shared memory (one barrier per token, alternating areas) and written per
// (token, head, quarter) for bwd_prologue_kernel, which adds the quarters and the
// value heads of a group.  The per-row dot products of a warp's four rows use one
// four-value warp reduce-scatter.  This is the token recurrence on CUDA cores in
// fp32, a correct first form; its cost is O(T K V) per chain with no tensor-core
// use.
#include "kda_common.cuh"

namespace kda {

cudaError_t launch_plan(const int32_t *cu, int N, int B, int T, SeqDesc *seqs, ChunkDesc *chunks, int *order,
                        int *hdr, long long max_chunks, cudaStream_t stream);
long long max_chunks_for(int N, int B, int T, bool varlen);
void timing_mark(const char *name, cudaStream_t s);

constexpr int BW_WARPS = 8;
constexpr int BW_THREADS = BW_WARPS * 32;
constexpr int BW_PARTS = 4;                            // CTAs per chain
constexpr int BW_ROWS = KD / BW_PARTS / BW_WARPS;      // 4 state rows per warp
constexpr int BW_CT = 16;                              // tokens per block (checkpoint interval)
constexpr int BW_BPC = CH / BW_CT;                     // blocks per 64-token chunk
static_assert(CH % BW_CT == 0, "blocks tile a chunk");
constexpr uint32_t BW_VEC = BW_CT * KD * 4;            // one [BW_CT][128] fp32 table
constexpr uint32_t BW_QT = 0, BW_KH = BW_VEC, BW_E = 2 * BW_VEC, BW_V = 3 * BW_VEC, BW_DO = 4 * BW_VEC;
constexpr uint32_t BW_BETA = 5 * BW_VEC;            // [BW_CT]
constexpr uint32_t BW_RED = BW_BETA + 128;          // 2 x [8 warps][3][128] (alternating tokens)
constexpr uint32_t BW_REDB = BW_RED + 2 * BW_WARPS * 3 * KD * 4;   // 2 x [8]
constexpr uint32_t BW_BYTES = BW_REDB + 64;
static_assert(2 * (BW_BYTES + 128 + 1024) <= 228 * 1024, "two backward CTAs per SM");

struct BwdParams {
    const uint16_t *q, *k, *v, *graw, *b, *dout;
    const float *A_log, *init, *dht;
    float scale;
    int H_qk, H_v, nseq;
    const SeqDesc *seqs;
    const int *order;
    const int *hdr;
    float *ckpt;      // [BW_BPC chunk + block][H_v][V][K]
    float *scratch;   // [gridDim.x][BW_CT][32 rows][K]
    float *dqt, *dkh, *de, *dbeta;   // [token][H_v][part][128] (dbeta [token][H_v][part])
    float *dv, *dh0;                 // [token][H_v][V], [N][H_v][V][K]
};

// Per-token vectors of tokens tok0 .. tok0 + len - 1 into the shared tables; warp w takes tokens w, w + 8, ...
__device__ __forceinline__ void bwd_stage_chunk(const BwdParams &p, unsigned char *sm, int tok0, int len, int h,
                                                int hq, float a_gate, bool with_do, int warp, int lane) {
    float *sqt = reinterpret_cast<float *>(sm + BW_QT), *skh = reinterpret_cast<float *>(sm + BW_KH);
    float *se = reinterpret_cast<float *>(sm + BW_E), *sv = reinterpret_cast<float *>(sm + BW_V);
    float *sdo = reinterpret_cast<float *>(sm + BW_DO), *sbeta = reinterpret_cast<float *>(sm + BW_BETA);
    for (int r = warp; r < len; r += BW_WARPS) {
        const size_t tok = (size_t)tok0 + r;
        const size_t qo = (tok * p.H_qk + hq) * KD + 4 * lane, vo = (tok * p.H_v + h) * KD + 4 * lane;
        const uint2 qw = *reinterpret_cast<const uint2 *>(p.q + qo), kw = *reinterpret_cast<const uint2 *>(p.k + qo);
        const uint2 gw = *reinterpret_cast<const uint2 *>(p.graw + vo), vw = *reinterpret_cast<const uint2 *>(p.v + vo);
        const float qv[4] = {bf16_lo(qw.x), bf16_hi(qw.x), bf16_lo(qw.y), bf16_hi(qw.y)};
        const float kv[4] = {bf16_lo(kw.x), bf16_hi(kw.x), bf16_lo(kw.y), bf16_hi(kw.y)};
        const float gv[4] = {bf16_lo(gw.x), bf16_hi(gw.x), bf16_lo(gw.y), bf16_hi(gw.y)};
        const float vv[4] = {bf16_lo(vw.x), bf16_hi(vw.x), bf16_lo(vw.y), bf16_hi(vw.y)};
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sq = fmaf(qv[i], qv[i], sq);
            sk = fmaf(kv[i], kv[i], sk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float rq = p.scale * rsqrtf(sq + L2_EPS), rk = rsqrtf(sk + L2_EPS);
        float4 a, bq, c, d;
        a.x = qv[0] * rq; a.y = qv[1] * rq; a.z = qv[2] * rq; a.w = qv[3] * rq;
        bq.x = kv[0] * rk; bq.y = kv[1] * rk; bq.z = kv[2] * rk; bq.w = kv[3] * rk;
        c.x = ex2(-a_gate * softplus_log2(gv[0])); c.y = ex2(-a_gate * softplus_log2(gv[1]));
        c.z = ex2(-a_gate * softplus_log2(gv[2])); c.w = ex2(-a_gate * softplus_log2(gv[3]));
        d.x = vv[0]; d.y = vv[1]; d.z = vv[2]; d.w = vv[3];
        reinterpret_cast<float4 *>(sqt + r * KD)[lane] = a;
        reinterpret_cast<float4 *>(skh + r * KD)[lane] = bq;
        reinterpret_cast<float4 *>(se + r * KD)[lane] = c;
        reinterpret_cast<float4 *>(sv + r * KD)[lane] = d;
        if (with_do) {
            const uint2 ow = *reinterpret_cast<const uint2 *>(p.dout + vo);
            reinterpret_cast<float4 *>(sdo + r * KD)[lane] =
                make_float4(bf16_lo(ow.x), bf16_hi(ow.x), bf16_lo(ow.y), bf16_hi(ow.y));
        }
        if (lane == 0) {
            const float bb = bf16_to_f(p.b[tok * p.H_v + h]);
            sbeta[r] = 1.0f / (1.0f + ex2(-bb * LOG2E));
        }
    }
}

// Warp sums of four per-lane partials (one per state row), returned on every lane.  A
// reduce-scatter (xor 16 keeps two rows, xor 8 one, xor 4, 2, 1 finish it) leaves lane l with
// the sum of row 2 b4 + b3 (b = bits of l); four broadcasts return them: 10 shuffles instead
// of 20 for four butterflies.
__device__ __forceinline__ void warp_sum4(float (&a)[4], int lane) {
    const bool u16 = (lane & 16) != 0, u8 = (lane & 8) != 0;
    float b0 = u16 ? a[2] : a[0], b1 = u16 ? a[3] : a[1];
    const float s0 = u16 ? a[0] : a[2], s1 = u16 ? a[1] : a[3];
    b0 += __shfl_xor_sync(0xffffffffu, s0, 16);
    b1 += __shfl_xor_sync(0xffffffffu, s1, 16);
    float c = u8 ? b1 : b0;
    c += __shfl_xor_sync(0xffffffffu, u8 ? b0 : b1, 8);
    c += __shfl_xor_sync(0xffffffffu, c, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    a[0] = __shfl_sync(0xffffffffu, c, 0);
    a[1] = __shfl_sync(0xffffffffu, c, 8);
    a[2] = __shfl_sync(0xffffffffu, c, 16);
    a[3] = __shfl_sync(0xffffffffu, c, 24);
}
static_assert(BW_ROWS == 4, "warp_sum4 reduces four rows");

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

// One forward token on this thread's 4 rows x 4 channels: S <- S Diag(e) + beta (v - S Diag(e) kh) kh^T.
__device__ __forceinline__ void bwd_fwd_token(float4 (&S)[BW_ROWS], const float4 kh, const float4 e, float beta,
                                              const float *vrow, int r0, int lane) {
    float d[BW_ROWS];
#pragma unroll
    for (int i = 0; i < BW_ROWS; ++i) {
        S[i].x *= e.x; S[i].y *= e.y; S[i].z *= e.z; S[i].w *= e.w;
        d[i] = dot4(S[i], kh);
    }
    warp_sum4(d, lane);
#pragma unroll
    for (int i = 0; i < BW_ROWS; ++i) {
        const float del = beta * (vrow[r0 + i] - d[i]);
        S[i].x = fmaf(del, kh.x, S[i].x); S[i].y = fmaf(del, kh.y, S[i].y);
        S[i].z = fmaf(del, kh.z, S[i].z); S[i].w = fmaf(del, kh.w, S[i].w);
    }
}

__global__ __launch_bounds__(BW_THREADS, 2) void bwd_recur_kernel(const BwdParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = aligned_smem<128>(smem_raw);
    if (p.hdr[1] == 0) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float *sqt = reinterpret_cast<const float *>(sm + BW_QT), *skh = reinterpret_cast<const float *>(sm + BW_KH);
    const float *se = reinterpret_cast<const float *>(sm + BW_E), *sv = reinterpret_cast<const float *>(sm + BW_V);
    const float *sdo = reinterpret_cast<const float *>(sm + BW_DO), *sbeta = reinterpret_cast<const float *>(sm + BW_BETA);
    float *red = reinterpret_cast<float *>(sm + BW_RED), *redb = reinterpret_cast<float *>(sm + BW_REDB);
    float *scr = p.scratch + (size_t)blockIdx.x * BW_CT * (KD / BW_PARTS) * KD;
    const int n_items = p.nseq * p.H_v * BW_PARTS;
    const int group = p.H_v / p.H_qk;

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int part = item % BW_PARTS, h = (item / BW_PARTS) % p.H_v;
        const int seq = p.order[item / (BW_PARTS * p.H_v)], hq = h / group;
        const SeqDesc sd = p.seqs[seq];
        const int nblk = (sd.len + BW_CT - 1) / BW_CT;
        const float a_gate = ex2(p.A_log[h] * LOG2E);
        // rows of this thread in the full [V][K] matrix, and their offset within the quarter
        const int r0 = part * (KD / BW_PARTS) + warp * BW_ROWS, q0 = warp * BW_ROWS;
        const size_t sh = ((size_t)seq * p.H_v + h) * KD * KD;
        auto slice = [&](size_t base, int i) { return base + (size_t)(r0 + i) * KD + 4 * lane; };
        auto sslice = [&](int r, int i) { return ((size_t)r * (KD / BW_PARTS) + q0 + i) * KD + 4 * lane; };
        float4 S[BW_ROWS];
#pragma unroll
        for (int i = 0; i < BW_ROWS; ++i)
            S[i] = p.init ? *reinterpret_cast<const float4 *>(p.init + slice(sh, i)) : make_float4(0.f, 0.f, 0.f, 0.f);

        // ---- pass 1: the recurrence, storing the state at each block start
        for (int c = 0; c < nblk; ++c) {
            const int len = min(BW_CT, sd.len - c * BW_CT), tok0 = sd.tok + c * BW_CT;
            const size_t cb = ((size_t)(BW_BPC * sd.chunk0 + c) * p.H_v + h) * KD * KD;
#pragma unroll
            for (int i = 0; i < BW_ROWS; ++i) *reinterpret_cast<float4 *>(p.ckpt + slice(cb, i)) = S[i];
            __syncthreads();   // the previous block's tables are no longer read
            bwd_stage_chunk(p, sm, tok0, len, h, hq, a_gate, false, warp, lane);
            __syncthreads();
            for (int r = 0; r < len; ++r)
                bwd_fwd_token(S, reinterpret_cast<const float4 *>(skh + r * KD)[lane],
                              reinterpret_cast<const float4 *>(se + r * KD)[lane], sbeta[r], sv + r * KD, r0, lane);
        }

        // ---- pass 2: blocks in reverse
        float4 dS[BW_ROWS];
#pragma unroll
        for (int i = 0; i < BW_ROWS; ++i)
            dS[i] = p.dht ? *reinterpret_cast<const float4 *>(p.dht + slice(sh, i)) : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = nblk - 1; c >= 0; --c) {
            const int len = min(BW_CT, sd.len - c * BW_CT), tok0 = sd.tok + c * BW_CT;
            const size_t cb = ((size_t)(BW_BPC * sd.chunk0 + c) * p.H_v + h) * KD * KD;
            __syncthreads();
            bwd_stage_chunk(p, sm, tok0, len, h, hq, a_gate, true, warp, lane);
            __syncthreads();
            // recompute the block's states; scratch[r] = state before token r (this thread's slice)
#pragma unroll
            for (int i = 0; i < BW_ROWS; ++i) S[i] = *reinterpret_cast<const float4 *>(p.ckpt + slice(cb, i));
            for (int r = 0; r < len; ++r) {
#pragma unroll
                for (int i = 0; i < BW_ROWS; ++i) *reinterpret_cast<float4 *>(scr + sslice(r, i)) = S[i];
                if (r + 1 < len)
                    bwd_fwd_token(S, reinterpret_cast<const float4 *>(skh + r * KD)[lane],
                                  reinterpret_cast<const float4 *>(se + r * KD)[lane], sbeta[r], sv + r * KD, r0, lane);
            }
            // tokens backwards; the states of token r - 1 are loaded while token r is processed, and the
            // reduction areas alternate so one barrier per token suffices
            float4 spn[BW_ROWS];
#pragma unroll
            for (int i = 0; i < BW_ROWS; ++i) spn[i] = *reinterpret_cast<const float4 *>(scr + sslice(len - 1, i));
            for (int r = len - 1; r >= 0; --r) {
                const float4 kh = reinterpret_cast<const float4 *>(skh + r * KD)[lane];
                const float4 qt = reinterpret_cast<const float4 *>(sqt + r * KD)[lane];
                const float4 e = reinterpret_cast<const float4 *>(se + r * KD)[lane];
                const float beta = sbeta[r];
                float4 pq = make_float4(0.f, 0.f, 0.f, 0.f), pk = pq, pe = pq;
                float pb = 0.f;
                float4 sp[BW_ROWS];
#pragma unroll
                for (int i = 0; i < BW_ROWS; ++i) sp[i] = spn[i];
                if (r > 0) {
#pragma unroll
                    for (int i = 0; i < BW_ROWS; ++i) spn[i] = *reinterpret_cast<const float4 *>(scr + sslice(r - 1, i));
                }
                // S' = S_{t-1} Diag(e) and d = S' kh for the four rows
                float4 s1[BW_ROWS], g[BW_ROWS];
                float d[BW_ROWS], dd4[BW_ROWS], del[BW_ROWS];
#pragma unroll
                for (int i = 0; i < BW_ROWS; ++i) {
                    s1[i].x = sp[i].x * e.x; s1[i].y = sp[i].y * e.y; s1[i].z = sp[i].z * e.z; s1[i].w = sp[i].w * e.w;
                    d[i] = dot4(s1[i], kh);
                }
                warp_sum4(d, lane);
                // delta, S_t; dS += do qt^T; dqt += S_t^T do; ddel = dS kh
#pragma unroll
                for (int i = 0; i < BW_ROWS; ++i) {
                    const float dor = sdo[r * KD + r0 + i];
                    del[i] = beta * (sv[r * KD + r0 + i] - d[i]);
                    float4 st;
                    st.x = fmaf(del[i], kh.x, s1[i].x); st.y = fmaf(del[i], kh.y, s1[i].y);
                    st.z = fmaf(del[i], kh.z, s1[i].z); st.w = fmaf(del[i], kh.w, s1[i].w);
                    g[i] = dS[i];
                    g[i].x = fmaf(dor, qt.x, g[i].x); g[i].y = fmaf(dor, qt.y, g[i].y);
                    g[i].z = fmaf(dor, qt.z, g[i].z); g[i].w = fmaf(dor, qt.w, g[i].w);
                    pq.x = fmaf(st.x, dor, pq.x); pq.y = fmaf(st.y, dor, pq.y);
                    pq.z = fmaf(st.z, dor, pq.z); pq.w = fmaf(st.w, dor, pq.w);
                    dd4[i] = dot4(g[i], kh);
                }
                warp_sum4(dd4, lane);   // ddel per row
#pragma unroll
                for (int i = 0; i < BW_ROWS; ++i) {
                    const float ddel = dd4[i];
                    // dkh += dS^T delta ; dv ; dbeta
                    pk.x = fmaf(g[i].x, del[i], pk.x); pk.y = fmaf(g[i].y, del[i], pk.y);
                    pk.z = fmaf(g[i].z, del[i], pk.z); pk.w = fmaf(g[i].w, del[i], pk.w);
                    if (lane == 0) p.dv[((size_t)(tok0 + r) * p.H_v + h) * KD + r0 + i] = beta * ddel;
                    pb = fmaf(ddel, sv[r * KD + r0 + i] - d[i], pb);
                    // dd = -beta ddel ; dS' = dS + dd kh^T ; dkh += S'^T dd ; de += S_{t-1} * dS'
                    const float dd = -beta * ddel;
                    g[i].x = fmaf(dd, kh.x, g[i].x); g[i].y = fmaf(dd, kh.y, g[i].y);
                    g[i].z = fmaf(dd, kh.z, g[i].z); g[i].w = fmaf(dd, kh.w, g[i].w);
                    pk.x = fmaf(s1[i].x, dd, pk.x); pk.y = fmaf(s1[i].y, dd, pk.y);
                    pk.z = fmaf(s1[i].z, dd, pk.z); pk.w = fmaf(s1[i].w, dd, pk.w);
                    pe.x = fmaf(sp[i].x, g[i].x, pe.x); pe.y = fmaf(sp[i].y, g[i].y, pe.y);
                    pe.z = fmaf(sp[i].z, g[i].z, pe.z); pe.w = fmaf(sp[i].w, g[i].w, pe.w);
                    // dS_{t-1} = dS' Diag(e)
                    dS[i].x = g[i].x * e.x; dS[i].y = g[i].y * e.y; dS[i].z = g[i].z * e.z; dS[i].w = g[i].w * e.w;
                }
                // sums over the quarter's rows (8 warps)
                float *rd = red + (r & 1) * (BW_WARPS * 3 * KD), *rdb = redb + (r & 1) * BW_WARPS;
                reinterpret_cast<float4 *>(rd + (warp * 3 + 0) * KD)[lane] = pq;
                reinterpret_cast<float4 *>(rd + (warp * 3 + 1) * KD)[lane] = pk;
                reinterpret_cast<float4 *>(rd + (warp * 3 + 2) * KD)[lane] = pe;
                if (lane == 0) rdb[warp] = pb;
                __syncthreads();
                const size_t tp = ((size_t)(tok0 + r) * p.H_v + h) * BW_PARTS + part;
                for (int x = tid; x < 3 * KD; x += BW_THREADS) {
                    const int which = x / KD, ch = x % KD;
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < BW_WARPS; ++w) acc += rd[(w * 3 + which) * KD + ch];
                    float *dst = which == 0 ? p.dqt : which == 1 ? p.dkh : p.de;
                    dst[tp * KD + ch] = acc;
                }
                if (tid == 0) {
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < BW_WARPS; ++w) acc += rdb[w];
                    p.dbeta[tp] = acc;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < BW_ROWS; ++i) *reinterpret_cast<float4 *>(p.dh0 + slice(sh, i)) = dS[i];
    }
}

// The prologue's Jacobians, one warp per (query/key head, token range); lane = channels
// 4 lane .. 4 lane + 3:
//   dq = scale r_q dqt_sum - scale r_q^3 q (q . dqt_sum),  r_q = 1 / sqrt(|q|^2 + eps)   (dk alike, scale 1)
//   dgraw = de e (-a) sigmoid(graw),  dA_log += sum_c de e g,  db = dbeta beta (1 - beta)
// with dqt_sum / dkh_sum / de / dbeta the sums over the four row quarters (and, for dqt and dkh,
// over the value heads of the group).  dA_log is accumulated per warp and added once per head
// (per token and head when a group has more than 16 value heads).
constexpr int BP_WARPS = 8;
constexpr int BP_TOKENS = 64;   // tokens per warp

__global__ __launch_bounds__(BP_WARPS * 32) void bwd_prologue_kernel(const BwdParams p, float *dq, float *dk,
                                                                     float *dgraw, float *db, float *dA_log,
                                                                     long long tokens) {
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * BP_WARPS + (threadIdx.x >> 5);
    const long long n_ranges = (tokens + BP_TOKENS - 1) / BP_TOKENS;
    if (gw >= n_ranges * p.H_qk) return;
    const int hq = (int)(gw % p.H_qk);
    const long long t0 = (gw / p.H_qk) * BP_TOKENS, t1 = min(t0 + BP_TOKENS, tokens);
    const int group = p.H_v / p.H_qk;
    constexpr int MAXG = 16;
    float dal[MAXG];
#pragma unroll
    for (int g = 0; g < MAXG; ++g) dal[g] = 0.f;
    for (long long tok = t0; tok < t1; ++tok) {
        const size_t qo = ((size_t)tok * p.H_qk + hq) * KD + 4 * lane;
        const uint2 qw = *reinterpret_cast<const uint2 *>(p.q + qo), kw = *reinterpret_cast<const uint2 *>(p.k + qo);
        const float qv[4] = {bf16_lo(qw.x), bf16_hi(qw.x), bf16_lo(qw.y), bf16_hi(qw.y)};
        const float kv[4] = {bf16_lo(kw.x), bf16_hi(kw.x), bf16_lo(kw.y), bf16_hi(kw.y)};
        float sq[4] = {0.f, 0.f, 0.f, 0.f}, sk[4] = {0.f, 0.f, 0.f, 0.f};
        for (int g = 0; g < group; ++g)
#pragma unroll
            for (int pt = 0; pt < BW_PARTS; ++pt) {
                const size_t ho = (((size_t)tok * p.H_v + hq * group + g) * BW_PARTS + pt) * KD + 4 * lane;
                const float4 a = *reinterpret_cast<const float4 *>(p.dqt + ho);
                const float4 b = *reinterpret_cast<const float4 *>(p.dkh + ho);
                sq[0] += a.x; sq[1] += a.y; sq[2] += a.z; sq[3] += a.w;
                sk[0] += b.x; sk[1] += b.y; sk[2] += b.z; sk[3] += b.w;
            }
        float nq = 0.f, nk = 0.f, qd = 0.f, kd = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            nq = fmaf(qv[i], qv[i], nq);
            nk = fmaf(kv[i], kv[i], nk);
            qd = fmaf(qv[i], sq[i], qd);
            kd = fmaf(kv[i], sk[i], kd);
        }
        nq = warp_sum(nq);
        nk = warp_sum(nk);
        qd = warp_sum(qd);
        kd = warp_sum(kd);
        const float rq = rsqrtf(nq + L2_EPS), rk = rsqrtf(nk + L2_EPS);
        float4 oq, ok;
        oq.x = p.scale * rq * (sq[0] - rq * rq * qv[0] * qd); oq.y = p.scale * rq * (sq[1] - rq * rq * qv[1] * qd);
        oq.z = p.scale * rq * (sq[2] - rq * rq * qv[2] * qd); oq.w = p.scale * rq * (sq[3] - rq * rq * qv[3] * qd);
        ok.x = rk * (sk[0] - rk * rk * kv[0] * kd); ok.y = rk * (sk[1] - rk * rk * kv[1] * kd);
        ok.z = rk * (sk[2] - rk * rk * kv[2] * kd); ok.w = rk * (sk[3] - rk * rk * kv[3] * kd);
        *reinterpret_cast<float4 *>(dq + qo) = oq;
        *reinterpret_cast<float4 *>(dk + qo) = ok;
#pragma unroll 1
        for (int g = 0; g < group; ++g) {
            const int h = hq * group + g;
            const size_t vo = ((size_t)tok * p.H_v + h) * KD + 4 * lane;
            const float a = ex2(p.A_log[h] * LOG2E);
            const uint2 gw2 = *reinterpret_cast<const uint2 *>(p.graw + vo);
            const float gr[4] = {bf16_lo(gw2.x), bf16_hi(gw2.x), bf16_lo(gw2.y), bf16_hi(gw2.y)};
            float de[4] = {0.f, 0.f, 0.f, 0.f}, dbeta = 0.f;
#pragma unroll
            for (int pt = 0; pt < BW_PARTS; ++pt) {
                const float4 x = *reinterpret_cast<const float4 *>(p.de + (((size_t)tok * p.H_v + h) * BW_PARTS + pt) * KD + 4 * lane);
                de[0] += x.x; de[1] += x.y; de[2] += x.z; de[3] += x.w;
                dbeta += p.dbeta[((size_t)tok * p.H_v + h) * BW_PARTS + pt];
            }
            float out[4], acc = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float sp = softplus_log2(gr[i]) * (1.0f / LOG2E);   // softplus (natural units)
                const float gg = -a * sp, ee = __expf(gg);
                const float sig = 1.0f / (1.0f + __expf(-gr[i]));
                const float dg = de[i] * ee;
                out[i] = dg * (-a) * sig;
                acc = fmaf(dg, gg, acc);
            }
            *reinterpret_cast<float4 *>(dgraw + vo) = make_float4(out[0], out[1], out[2], out[3]);
            acc = warp_sum(acc);
            if (group <= MAXG) {
#pragma unroll
                for (int gg2 = 0; gg2 < MAXG; ++gg2)
                    if (gg2 == g) dal[gg2] += acc;
            } else if (lane == 0) {
                atomicAdd(&dA_log[h], acc);
            }
            if (lane == 0) {
                const float bb = bf16_to_f(p.b[(size_t)tok * p.H_v + h]);
                const float beta = 1.0f / (1.0f + __expf(-bb));
                db[(size_t)tok * p.H_v + h] = dbeta * beta * (1.0f - beta);
            }
        }
    }
    if (lane == 0 && group <= MAXG) {
#pragma unroll
        for (int g = 0; g < MAXG; ++g)
            if (g < group) atomicAdd(&dA_log[hq * group + g], dal[g]);
    }
}

// ---------------------------------------------------------------- host side
namespace {
size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }
}

size_t bwd_workspace_bytes(int N, int B, int T, int H_v, bool varlen, int grid) {
    const long long nseq = varlen ? N : B, nck = max_chunks_for(N, B, T, varlen), tokens = (long long)B * T;
    size_t off = a256(256);
    off = a256(off + sizeof(SeqDesc) * (size_t)(nseq > 0 ? nseq : 1));
    off = a256(off + sizeof(ChunkDesc) * (size_t)(nck > 0 ? nck : 1));
    off = a256(off + sizeof(int) * (size_t)(nseq > 0 ? nseq : 1));
    off = a256(off + (size_t)BW_BPC * (nck > 0 ? nck : 1) * H_v * KD * KD * 4);       // checkpoints
    off = a256(off + (size_t)grid * BW_CT * (KD / BW_PARTS) * KD * 4);          // scratch
    off = a256(off + (size_t)(tokens > 0 ? tokens : 1) * H_v * BW_PARTS * KD * 4 * 3);   // dqt, dkh, de
    off = a256(off + (size_t)(tokens > 0 ? tokens : 1) * H_v * BW_PARTS * 4);            // dbeta
    return off;
}

int bwd_grid(int nseq, int H_v) {
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const long long items = (long long)nseq * H_v * BW_PARTS, slots = 2LL * nsm;
    return (int)(items < slots ? (items > 0 ? items : 1) : slots);
}

cudaError_t launch_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                       const uint16_t *b, const float *A_log, float scale, const float *init, const int32_t *cu, int N,
                       int B, int T, int H_qk, int H_v, const uint16_t *dout, const float *dht, float *dq, float *dk,
                       float *dv, float *dgraw, float *db, float *dA_log, float *dh0, void *ws_ptr, int grid,
                       cudaStream_t stream, int *launches) {
    const bool varlen = cu != nullptr;
    const int nseq = varlen ? N : B;
    const long long nck = max_chunks_for(N, B, T, varlen), tokens = (long long)B * T;
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
    BwdParams bp;
    bp.ckpt = reinterpret_cast<float *>(take((size_t)BW_BPC * (nck > 0 ? nck : 1) * H_v * KD * KD * 4));
    bp.scratch = reinterpret_cast<float *>(take((size_t)grid * BW_CT * (KD / BW_PARTS) * KD * 4));
    const size_t tv = (size_t)(tokens > 0 ? tokens : 1) * H_v * BW_PARTS * KD;
    float *t3 = reinterpret_cast<float *>(take(tv * 4 * 3));
    bp.dqt = t3; bp.dkh = t3 + tv; bp.de = t3 + 2 * tv;
    bp.dbeta = reinterpret_cast<float *>(take((size_t)(tokens > 0 ? tokens : 1) * H_v * BW_PARTS * 4));
    bp.q = q; bp.k = k; bp.v = v; bp.graw = graw; bp.b = b; bp.dout = dout;
    bp.A_log = A_log; bp.init = init; bp.dht = dht; bp.scale = scale;
    bp.H_qk = H_qk; bp.H_v = H_v; bp.nseq = nseq; bp.seqs = seqs; bp.order = order; bp.hdr = hdr;
    bp.dv = dv; bp.dh0 = dh0;
    *launches = 0;
    cudaError_t e = launch_plan(cu, N, B, T, seqs, chunks, order, hdr, nck, stream);
    if (e != cudaSuccess) return e;
    ++*launches;
    if ((e = cudaMemsetAsync(dA_log, 0, sizeof(float) * H_v, stream)) != cudaSuccess) return e;
    timing_mark("plan_kernel", stream);
    if (nseq > 0) {
        if ((e = cudaFuncSetAttribute(bwd_recur_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)(BW_BYTES + 128))) != cudaSuccess)
            return e;
        bwd_recur_kernel<<<grid, BW_THREADS, BW_BYTES + 128, stream>>>(bp);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        timing_mark("bwd_recur_kernel", stream);
    }
    if (tokens > 0) {
        const long long warps = ((tokens + BP_TOKENS - 1) / BP_TOKENS) * H_qk;
        bwd_prologue_kernel<<<(unsigned)((warps + BP_WARPS - 1) / BP_WARPS), BP_WARPS * 32, 0, stream>>>(
            bp, dq, dk, dgraw, db, dA_log, tokens);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        timing_mark("bwd_prologue_kernel", stream);
    }
    return cudaSuccess;
}

}  // namespace kda
