// chunk_scan_tc.cu -- the chunked prefill (SSD form) on the tcgen05 tensor cores.
//
// Operations ("Hybrid SSM / Mamba models and non-KV state": mamba_chunk_scan_combined, whose
// within-chunk term is a masked matrix product on tensor cores and whose chunks are joined by a
// short scan over chunk states; a later chunk continues from the stored state; align-mode
// checkpoints; echobase "Mamba" notes: Y = (M (.) L) X with M_ij = C_i (prod_{k=j+1..i} Abar_k) Bbar_j):
//   per sub-chunk of up to 128 tokens and head h, with cum_t = sum_{k<=t} Delta_k A_h:
//     G     = C B^T                                         (tensor core, fp32 in TMEM)
//     M     = G (.) exp(cum_i - cum_j) (.) Delta_j, j <= i   (CUDA cores, bf16 into tensor memory)
//     Y     = M X + exp(cum_i) C h_prev^T + D x             (tensor core + epilogue)
//     h^T   = exp(cum_end) h^T + B^T (w (.) X),  w_j = exp(cum_end - cum_j) Delta_j   (tensor core)
//
// Design (GB300): one CTA per (sequence, head) walks its sequence in order, so the running
// state never leaves the SM: it lives in tensor memory in fp32 for the whole sequence (its bf16
// copy in shared memory feeds the next C h^T).  Per sub-chunk only C, B and X are read (TMA,
// 128-byte swizzle) and y is written: no per-chunk states travel through HBM.  The masked G is
// written as bf16 over the tensor-memory columns of G the mask has consumed and M X reads it
// from there (A operand in tensor memory), so the C tile is free as soon as C B^T and C h^T
// complete and the next sub-chunk's C is loaded while this one is still being masked.  The 256-token
// chunks of the checkpoint grid are processed as two 128-token halves (the MMA M of one CTA);
// the result is the same up to rounding.  Shared memory ~98 KB and 256 TMEM columns per CTA,
// so two CTAs share an SM and cover each other's waits; each CTA's eight warps split every
// row's work in two.  All waits are bounded.
#include <mutex>

#include "common.cuh"
#include "scan_tc.h"
#include "umma.cuh"

namespace ms {

using namespace umma;

namespace {

constexpr int SQ = 128;  // tokens per sub-chunk (MMA M)
constexpr int TP = 64;   // head_dim
constexpr int TN = 128;  // d_state
constexpr uint32_t BLK = 16384;  // one 128-row x 128-byte swizzled block
constexpr uint32_t kPolls = umma::kWaitPolls;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float kDiagSpan = 96.0f;  // largest base-2 exponent span of a diagonal block taken factored

// shared-memory map (from a 1024-aligned base)
constexpr uint32_t OFF_B = 0;          // B tile, rows j: [n 0..63 | n 64..127]
constexpr uint32_t OFF_C = 2 * BLK;    // C tile, rows i: [n 0..63 | n 64..127]
constexpr uint32_t OFF_X = 4 * BLK;    // X tile, rows j, p 0..63; then w * X
constexpr uint32_t OFF_H = 5 * BLK;    // h^T in bf16, rows n, p 0..63
constexpr uint32_t OFF_SMALL = 6 * BLK;
constexpr uint32_t SMEM_BYTES = OFF_SMALL + 4096 + 1024;  // + slack for the 1024-byte alignment

struct Small {
    uint64_t bar_c, bar_bx, bar_g, bar_yd, bar_s;
    uint32_t tmem;
    int pad;
    float cum2[SQ];   // cum * log2(e)
    float delta[SQ];
    float w[SQ];
    float ecol[SQ];   // column factors of the masked G below the diagonal blocks
    float ecold[SQ];  // column factors inside a diagonal block
    float warp_tot[4];
};
static_assert(sizeof(Small) <= 4096, "small area");

constexpr uint32_t ID_G = idesc_bf16(128, 128, false, false);   // C (K-major) x B (K-major)
constexpr uint32_t ID_YO = idesc_bf16(128, 64, false, true);    // C (K-major) x h^T (MN-major)
constexpr uint32_t ID_YD = idesc_bf16(128, 64, false, true);    // M (K-major) x X (MN-major)
constexpr uint32_t ID_S = idesc_bf16(128, 64, true, true);      // B^T (MN-major) x wX (MN-major)

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// The C tile of the sub-chunk starting at token t0 (completes on bar_c) ...
__device__ __forceinline__ void issue_c(unsigned char *sm, Small *sv, const CUtensorMap *mC, int g, int t0) {
    mbar_arrive_expect_tx(&sv->bar_c, 2 * BLK);
    tma_load_2d(sm + OFF_C, mC, g * TN, t0, &sv->bar_c);
    tma_load_2d(sm + OFF_C + BLK, mC, g * TN + 64, t0, &sv->bar_c);
}

// ... and its B and X tiles (complete on bar_bx).
__device__ __forceinline__ void issue_bx(unsigned char *sm, Small *sv, const CUtensorMap *mX, const CUtensorMap *mB,
                                         int h, int g, int t0) {
    mbar_arrive_expect_tx(&sv->bar_bx, 3 * BLK);
    tma_load_2d(sm + OFF_B, mB, g * TN, t0, &sv->bar_bx);
    tma_load_2d(sm + OFF_B + BLK, mB, g * TN + 64, t0, &sv->bar_bx);
    tma_load_2d(sm + OFF_X, mX, h * TP, t0, &sv->bar_bx);
}

// Tensor-memory column (relative to G) where the packed bf16 masked G of 32-column block jb goes:
// the two blocks a warp handles, hf and hf + 2, both land in block hf + 2's columns, which that
// same warp has already read.
__device__ __forceinline__ uint32_t m_col(int jb) { return 64u + 32u * (uint32_t)(jb & 1) + 16u * (uint32_t)(jb >> 1); }

// Writes the 64 p-values of h^T row n (fp32) as bf16 into the swizzled MN-major h tile.
__device__ __forceinline__ void store_hT_row(unsigned char *sm, int n, const float *v, int c0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u;
        u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        *reinterpret_cast<uint4 *>(sm + OFF_H + swz128_chunk(n, c0 / 8 + q)) = u;
    }
}

template <typename StateT>
__device__ __forceinline__ void write_state(StateT *dst, int n, const float *v, int c0) {
#pragma unroll
    for (int q = 0; q < 32; ++q) dst[(int64_t)(c0 + q) * TN + n] = from_f32<StateT>(v[q]);
}

}  // namespace

// Validates cu_seqlens and slot ids, and orders the sequences longest first (so the longest
// serial chains start first).  meta = [valid, pad x3, order[nseq]].
__global__ void __launch_bounds__(256) k_tc_meta(const ScanTcParams p) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    __shared__ int ok;
    const int tid = threadIdx.x;
    if (tid == 0) ok = p.cu[0] == 0 && p.cu[p.nseq] == p.T;
    __syncthreads();
    for (int s = tid; s < p.nseq; s += blockDim.x) {
        if (p.cu[s + 1] < p.cu[s]) ok = 0;
        const int32_t sl = p.slot[s];
        if (sl < -1 || sl >= p.num_slots) flag_error(p.err, MAMBA_ERR_SLOT_RANGE);
    }
    __syncthreads();
    if (!ok) {
        if (tid == 0) {
            flag_error(p.err, MAMBA_ERR_SEQLENS);
            p.meta[0] = 0;
        }
        return;
    }
    for (int s = tid; s < p.nseq; s += blockDim.x) {
        const int Ls = p.cu[s + 1] - p.cu[s];
        int r = 0;
        for (int s2 = 0; s2 < p.nseq; ++s2) {
            const int L2 = p.cu[s2 + 1] - p.cu[s2];
            r += (L2 > Ls) || (L2 == Ls && s2 < s);
        }
        p.meta[4 + r] = s;
    }
    if (tid == 0) p.meta[0] = 1;
}

// Threads: 8 warps.  Warp w works on TMEM lane quadrant q = w % 4 (rows 32q..32q+31 of every
// accumulator) and on half hf = w / 4 of the columns, so each row's work is split over two warps.
constexpr int kTcThreads = 256;

template <typename StateT>
__global__ void __launch_bounds__(kTcThreads, 2) k_ssd_tc(const ScanTcParams p, const __grid_constant__ CUtensorMap mX,
                                                          const __grid_constant__ CUtensorMap mB,
                                                          const __grid_constant__ CUtensorMap mC) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    extern __shared__ __align__(1024) unsigned char tc_smem[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(tc_smem) + 1023) &
                                                          ~static_cast<uintptr_t>(1023));
    Small *sv = reinterpret_cast<Small *>(sm + OFF_SMALL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, hf = warp >> 2;
    const int row = q * 32 + lane;  // TMEM lane of this thread: token row i, or state row n
    if (p.meta[0] == 0) return;  // bad cu_seqlens (flagged): nothing is done
    const int s = p.meta[4 + blockIdx.x / p.H];
    const int h = blockIdx.x % p.H;
    const int g = h / p.HG;
    const int t_begin = p.cu[s], len = p.cu[s + 1] - t_begin;
    const int32_t slot = p.slot[s];
    if (len <= 0 || slot < -1 || slot >= p.num_slots) return;  // empty, or bad slot (flagged)
    const bool has_init = slot >= 0 && p.has_init != nullptr && p.has_init[s] != 0;
    const float Ah = p.A[h], Dh = p.D ? p.D[h] : 0.0f, bias = p.dt_bias ? p.dt_bias[h] : 0.0f;
    StateT *pool = static_cast<StateT *>(p.ssm_pool);
    const int64_t head_off = (int64_t)h * TP * TN;

    if (tid == 0) {
        mbar_init(&sv->bar_c, 1);
        mbar_init(&sv->bar_bx, 1);
        mbar_init(&sv->bar_g, 1);
        mbar_init(&sv->bar_yd, 1);
        mbar_init(&sv->bar_s, 1);
        fence_mbar_init();
        tma_prefetch_desc(&mX);
        tma_prefetch_desc(&mB);
        tma_prefetch_desc(&mC);
    }
    if (warp == 0) {
        tmem_alloc(&sv->tmem, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = sv->tmem;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const uint32_t t_g = tm, t_yd = tm, t_yo = tm + 128, t_h = tm + 192;
    const int c0 = hf * 32;  // this warp's 32 of the 64 head_dim columns

    // the stored state seeds the scan (chunked prefill hand-off): h^T into TMEM and its bf16 copy
    if (has_init) {
        const StateT *src = pool + (int64_t)slot * p.ssm_stride + head_off;
        float v[32];
#pragma unroll
        for (int qq = 0; qq < 32; ++qq) v[qq] = to_f32(src[(int64_t)(c0 + qq) * TN + row]);
        tmem_st32(t_h + lane_base + c0, v);
        store_hT_row(sm, row, v, c0);
        fence_async_smem();
    }
    const int nsub = (len + SQ - 1) / SQ;
    // pending operations of thread 0 (bit 0: C tile, 1: G/Y_off, 2: Y_diag, 3: state, 4: B and X
    // tiles) and their parities
    uint32_t pending = 0, pend_par[5] = {0, 0, 0, 0, 0};
    if (tid == 0) {
        issue_c(sm, sv, &mC, g, t_begin);
        issue_bx(sm, sv, &mX, &mB, h, g, t_begin);
        pending |= 1u | 16u;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    bool h_valid = has_init;
    bool failed = false;
    uint32_t ph = 0;
    // dt of the sub-chunk about to run (prefetched one sub-chunk ahead; thread = token)
    float dt_next = tid < min(SQ, len) ? load_scalar(p.dt, (int64_t)(t_begin + tid) * p.H + h, p.dt_bf16) : 0.0f;
    for (int k = 0; k < nsub; ++k, ph ^= 1u) {
        const int t0 = t_begin + k * SQ, L = min(SQ, len - k * SQ);
        // this thread's 32 gate values of its token row, fetched now and used by the epilogue
        uint4 zrow[4];
        if (p.z && row < L) {
            const uint4 *zr = reinterpret_cast<const uint4 *>(static_cast<const bf16 *>(p.z) +
                                                              ((int64_t)(t0 + row) * p.H + h) * TP + c0);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) zrow[qq] = zr[qq];
        }
        // Delta and the within-sub-chunk cumulative sum of Delta*A (threads 0..127 = tokens)
        float dlt = 0.0f, run = 0.0f;
        if (tid < SQ) {
            if (tid < L) {
                const float sdt = dt_next + bias;
                dlt = p.dt_softplus ? softplus_f(sdt) : sdt;
            }
            const int Ln = min(SQ, len - (k + 1) * SQ);
            dt_next = (k + 1 < nsub && tid < Ln) ? load_scalar(p.dt, (int64_t)(t0 + SQ + tid) * p.H + h, p.dt_bf16)
                                                 : 0.0f;
            run = dlt * Ah;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, run, off);
                if (lane >= off) run += v;
            }
            if (lane == 31) sv->warp_tot[warp] = run;
        }
        __syncthreads();
        if (tid < SQ) {
            for (int w2 = 0; w2 < warp; ++w2) run += sv->warp_tot[w2];
            sv->cum2[tid] = run * LOG2E;
            sv->delta[tid] = dlt;
        }
        // G = C B^T and Y_off = C h_prev^T (every thread waits for the tiles itself: it reads X)
        int bad = (mbar_wait(&sv->bar_c, ph, kPolls) && mbar_wait(&sv->bar_bx, ph, kPolls)) ? 0 : 1;
        if (tid == 0) {
            if (!bad) {
                pending &= ~(1u | 16u);
                tc_fence_after();
                const uint32_t c = smem_u32(sm + OFF_C), b = smem_u32(sm + OFF_B), hh = smem_u32(sm + OFF_H);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(t_g, desc_kmajor(c, BLK, kk), desc_kmajor(b, BLK, kk), ID_G, kk > 0);
                if (h_valid) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(t_yo, desc_kmajor(c, BLK, kk), desc_mnmajor(hh, BLK, kk), ID_YO, kk > 0);
                }
                mma_commit(&sv->bar_g);
                pending |= 2u;
                pend_par[1] = ph;
            }
        }
        if (__syncthreads_or(bad)) {  // cum visible; a tile copy that gave up ends the CTA
            failed = true;
            break;
        }
        const float cend = sv->cum2[L - 1];
        if (tid < SQ) {
            // w_j = exp(cum_end - cum_j) Delta_j for the chunk state, and the column factor of the
            // masked G below the diagonal blocks: e_j = exp(cum_ref - cum_j) Delta_j with cum_ref the
            // cumulative sum at the LAST column of j's 32-column block.  For a row i past that block,
            // exp(cum_i - cum_j) = exp(cum_i - cum_ref) exp(cum_ref - cum_j) with both exponents <= 0
            // (cum is non-increasing: Delta >= 0, A <= 0), so neither factor can overflow whatever
            // the step size; a factor that underflows stands for a product below fp32's range.
            // Inside a diagonal block the same factoring with the block's FIRST column as the reference
            // (e_j = exp(cum_first - cum_j) Delta_j >= Delta_j, row factor <= 1) is used only when the
            // block spans at most 96 in base-2 exponent, so that both factors stay within 2^+-96;
            // a block with larger steps forms each decay from its own difference.
            const float cj = sv->cum2[tid];
            sv->w[tid] = tid < L ? exp2f(cend - cj) * dlt : 0.0f;
            sv->ecol[tid] = tid < L ? exp2f(sv->cum2[tid | 31] - cj) * dlt : 0.0f;
            sv->ecold[tid] = tid < L ? exp2f(fminf(sv->cum2[tid & ~31] - cj, kDiagSpan)) * dlt : 0.0f;
        }
        // this thread's 32 columns of its token row of X (for D x), read before the tile is scaled
        uint4 xrow[4];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq)
            xrow[qq] = *reinterpret_cast<const uint4 *>(sm + OFF_X + swz128_chunk(row, hf * 4 + qq));
        __syncthreads();  // ecol visible

        // M = G (.) exp(cum_i - cum_j) (.) Delta_j for j <= i, as packed bf16 into tensor memory
        // over G's columns.  Row i = this thread's lane; this warp forms column blocks jb = hf + 2
        // and then hf, and writes both into block hf + 2's columns (m_col), read just before.
        if (!mbar_wait(&sv->bar_g, ph, kPolls)) bad = 1;
        else if (tid == 0) pending &= ~2u;
        tc_fence_after();
        if (tid == 0 && !bad && k + 1 < nsub) {  // C B^T and C h^T are done with the C tile
            issue_c(sm, sv, &mC, g, t0 + SQ);
            pending |= 1u;
            pend_par[0] = ph ^ 1u;
        }
        {
            const float ci = sv->cum2[row];
#pragma unroll
            for (int bb = 1; bb >= 0; --bb) {
                const int jb = hf + 2 * bb;
                uint32_t pk[16];
                if (jb <= q) {  // warp-uniform: block jb can hold columns j <= i for these rows
                    float gv[32];
                    tmem_ld32(t_g + lane_base + jb * 32, gv);
                    if (jb < q) {  // every row is past the block: the factored form above
                        const float rf = row < L ? exp2f(ci - sv->cum2[jb * 32 + 31]) : 0.0f;
                        const float *ec = sv->ecol + jb * 32;
#pragma unroll
                        for (int qq = 0; qq < 32; qq += 2)
                            pk[qq / 2] = pack_bf16x2(gv[qq] * rf * ec[qq], gv[qq + 1] * rf * ec[qq + 1]);
                    } else if (sv->cum2[jb * 32] - sv->cum2[jb * 32 + 31] <= kDiagSpan) {
                        // diagonal block, j <= i, span within 2^96: factored at the block's first column
                        const float rf = row < L ? exp2f(ci - sv->cum2[jb * 32]) : 0.0f;
                        const float *ec = sv->ecold + jb * 32;
#pragma unroll
                        for (int qq = 0; qq < 32; qq += 2)
                            pk[qq / 2] = pack_bf16x2(qq <= lane ? gv[qq] * rf * ec[qq] : 0.0f,
                                                     qq + 1 <= lane ? gv[qq + 1] * rf * ec[qq + 1] : 0.0f);
                    } else {  // diagonal block with large steps: each decay from its own difference (<= 0)
                        const float *cc = sv->cum2 + jb * 32;
                        const float *dd = sv->delta + jb * 32;
                        const bool live = row < L;
#pragma unroll
                        for (int qq = 0; qq < 32; qq += 2) {
                            const float m0 = live && qq <= lane ? gv[qq] * exp2f(ci - cc[qq]) * dd[qq] : 0.0f;
                            const float m1 =
                                live && qq + 1 <= lane ? gv[qq + 1] * exp2f(ci - cc[qq + 1]) * dd[qq + 1] : 0.0f;
                            pk[qq / 2] = pack_bf16x2(m0, m1);
                        }
                    }
                } else {
#pragma unroll
                    for (int qq = 0; qq < 16; ++qq) pk[qq] = 0u;
                }
                tmem_st16(t_g + lane_base + m_col(jb), pk);
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // Y_diag = M X (A = M from tensor memory; into G's first 64 columns, which are consumed)
        if (tid == 0 && !bad) {
            const uint32_t x = smem_u32(sm + OFF_X);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ts(t_yd, t_g + m_col(kk >> 1) + 8u * (uint32_t)(kk & 1), desc_mnmajor(x, BLK, kk), ID_YD,
                            kk > 0);
            mma_commit(&sv->bar_yd);
            pending |= 4u;
            pend_par[2] = ph;
        }
        // h^T <- exp(cum_end) h^T (lane = state row n, this warp's 32 head_dim columns)
        if (h_valid) {
            const float decay = exp2f(cend);
            float v[32];
            tmem_ld32(t_h + lane_base + c0, v);
#pragma unroll
            for (int qq = 0; qq < 32; ++qq) v[qq] *= decay;
            tmem_st32(t_h + lane_base + c0, v);
        }
        if (!mbar_wait(&sv->bar_yd, ph, kPolls)) bad = 1;
        else if (tid == 0) pending &= ~4u;
        tc_fence_after();
        // w (.) X in place (the row of a 16-byte chunk is its byte offset / 128)
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const int cidx = tid + kTcThreads * qq;
            uint4 *ptr = reinterpret_cast<uint4 *>(sm + OFF_X + cidx * 16);
            const float wr = sv->w[cidx >> 3];
            uint4 u = *ptr;
            uint32_t *wd = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float lo = __uint_as_float(wd[e] << 16) * wr;
                const float hi = __uint_as_float(wd[e] & 0xffff0000u) * wr;
                wd[e] = pack_bf16x2(lo, hi);
            }
            *ptr = u;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // h^T += B^T (w X)
        if (tid == 0 && !bad) {
            const uint32_t b = smem_u32(sm + OFF_B), x = smem_u32(sm + OFF_X);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(t_h, desc_mnmajor(b, BLK, kk), desc_mnmajor(x, BLK, kk), ID_S, (h_valid || kk > 0) ? 1u : 0u);
            mma_commit(&sv->bar_s);
            pending |= 8u;
            pend_par[3] = ph;
        }
        // y = Y_diag + exp(cum_i) Y_off + D x, gated by SiLU(z) (lane = token row i, 32 columns)
        {
            const float ei = exp2f(sv->cum2[row]);
            float yd[32], yo[32];
            tmem_ld32(t_yd + lane_base + c0, yd);
            if (h_valid) {
                tmem_ld32(t_yo + lane_base + c0, yo);
            } else {
#pragma unroll
                for (int qq = 0; qq < 32; ++qq) yo[qq] = 0.0f;
            }
            if (row < L) {
                const bool gate = p.z != nullptr;
                bf16 *yr = static_cast<bf16 *>(p.y) + ((int64_t)(t0 + row) * p.H + h) * TP + c0;
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    const uint4 xv = xrow[q8];
                    const uint4 zv = gate ? zrow[q8] : make_uint4(0, 0, 0, 0);
                    const uint32_t *xw = reinterpret_cast<const uint32_t *>(&xv);
                    const uint32_t *zw = reinterpret_cast<const uint32_t *>(&zv);
                    uint4 out;
                    uint32_t *ow = reinterpret_cast<uint32_t *>(&out);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int qq = 8 * q8 + 2 * e;
                        float v0 = yd[qq] + ei * yo[qq] + Dh * __uint_as_float(xw[e] << 16);
                        float v1 = yd[qq + 1] + ei * yo[qq + 1] + Dh * __uint_as_float(xw[e] & 0xffff0000u);
                        if (gate) {
                            v0 *= silu_fast(__uint_as_float(zw[e] << 16));
                            v1 *= silu_fast(__uint_as_float(zw[e] & 0xffff0000u));
                        }
                        ow[e] = pack_bf16x2(v0, v1);
                    }
                    *reinterpret_cast<uint4 *>(yr + 8 * q8) = out;
                }
            }
        }
        // the state MMA must finish before the tiles are reloaded and the state is read
        if (!mbar_wait(&sv->bar_s, ph, kPolls)) bad = 1;
        tc_fence_after();
        h_valid = true;
        if (tid == 0 && !bad) {
            pending &= ~8u;
            if (k + 1 < nsub) {
                issue_bx(sm, sv, &mX, &mB, h, g, t0 + SQ);
                pending |= 16u;
                pend_par[4] = ph ^ 1u;
            }
        }
        // h^T -> bf16 copy for the next C h^T; checkpoints and the final state -> pool
        {
            const int done = k * SQ + L;
            StateT *dst = nullptr;
            StateT *dst2 = nullptr;
            if (p.ckpt_slots && p.ckpt_interval > 0 && done % p.ckpt_interval == 0) {
                const int m = done / p.ckpt_interval;
                if (m >= 1 && m <= p.max_ckpt) {
                    const int32_t cs = p.ckpt_slots[(int64_t)s * p.max_ckpt + m - 1];
                    if (cs >= p.num_slots || cs < -1) {
                        if (tid == 0 && h == 0) flag_error(p.err, MAMBA_ERR_SLOT_RANGE);
                    } else if (cs >= 0) {
                        dst = pool + (int64_t)cs * p.ssm_stride + head_off;
                    }
                }
            }
            if (k == nsub - 1 && slot >= 0) dst2 = pool + (int64_t)slot * p.ssm_stride + head_off;
            float v[32];
            tmem_ld32(t_h + lane_base + c0, v);
            if (k + 1 < nsub) store_hT_row(sm, row, v, c0);
            if (dst) write_state(dst, row, v, c0);
            if (dst2) write_state(dst2, row, v, c0);
        }
        fence_async_smem();
        tc_fence_before();
        if (__syncthreads_or(bad)) {  // an MMA wait that gave up anywhere in the CTA ends it here
            failed = true;
            break;
        }
        tc_fence_after();
    }
    if (failed) {
        // an operation did not complete in time: report it and let what this CTA still has in
        // flight finish (bounded) before the tensor memory is released
        if (tid == 0) {
            flag_error(p.err, MAMBA_ERR_TIMEOUT);
            if (pending & 1u) mbar_wait(&sv->bar_c, pend_par[0], kPolls);
            if (pending & 16u) mbar_wait(&sv->bar_bx, pend_par[4], kPolls);
            if (pending & 2u) mbar_wait(&sv->bar_g, pend_par[1], kPolls);
            if (pending & 4u) mbar_wait(&sv->bar_yd, pend_par[2], kPolls);
            if (pending & 8u) mbar_wait(&sv->bar_s, pend_par[3], kPolls);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// 2-D bf16 map over rows x cols (row pitch cols elements), 64 x 128 boxes, 128-byte swizzle,
// rows past the end read as zero.
static bool make_map(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, 128}, es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool scan_tc_eligible(const mamba_layer_desc *d, int chunk) {
    // an fp32 state pool asks for fp32 state arithmetic: its bf16 operand copies (M, w X, h) would
    // bound the written state at bf16 precision, so it takes the fp32 CUDA-core path instead
    return d->act_dtype == MAMBA_BF16 && d->state_dtype == MAMBA_BF16 && d->head_dim == TP && d->d_state == TN &&
           chunk > 0 && chunk % SQ == 0;
}

size_t scan_tc_workspace_bytes(int nseq) { return ((size_t)(4 + nseq) * sizeof(int32_t) + 255) / 256 * 256; }

int scan_tc_launch(const ScanTcParams &p, int state_bf16, cudaStream_t stream) {
    if (launch_pdl(k_tc_meta, dim3(1), dim3(256), 0, stream, p) != cudaSuccess) return MAMBA_ECUDA;
    if (p.T == 0) return launch_status();  // only empty sequences: nothing to compute or write
    CUtensorMap mX, mB, mC;
    if (!make_map(&mX, p.x, (uint64_t)p.H * TP, (uint64_t)p.T) ||
        !make_map(&mB, p.B, (uint64_t)p.G * TN, (uint64_t)p.T) ||
        !make_map(&mC, p.C, (uint64_t)p.G * TN, (uint64_t)p.T))
        return MAMBA_ECUDA;
    auto kern = state_bf16 ? k_ssd_tc<bf16> : k_ssd_tc<float>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES) != cudaSuccess)
        return MAMBA_ECUDA;
    if (launch_pdl(kern, dim3(p.nseq * p.H), dim3(kTcThreads), SMEM_BYTES, stream, p, mX, mB, mC) != cudaSuccess)
        return MAMBA_ECUDA;
    return launch_status();
}

}  // namespace ms
