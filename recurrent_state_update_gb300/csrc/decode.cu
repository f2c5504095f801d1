// decode.cu -- the batched decode step of the Mamba2 state update over a slot pool.
//
// Operations ("Hybrid SSM / Mamba models and non-KV state", state shapes and the decode call
// selective_state_update; echobase "Mamba" notes, block equations):
//   conv:   x|B|C = SiLU(causal depthwise conv1d over [conv state | new token])
//   step:   Delta = softplus(dt + dt_bias),  h <- exp(Delta*A) h + Delta * x B^T
//   out:    y = C.h + D*x,  y *= SiLU(z)
//
// Design (GB300): the state update is a pure HBM stream (about 1.25 flop per byte at bf16),
// so the kernel is built around moving each (slot, head) state tile of head_dim x d_state once
// in and once out with 16-byte coalesced accesses and evict-first cache hints, while the
// small per-group work (conv of x|B|C, Delta, exp) runs out of shared memory.
//
//  - One CTA per (row, group): the group's heads share one B and C, so the conv of the group's
//    B and C channels is done once and the CTA owns every conv-state column it writes (no two
//    CTAs touch one slot's conv channels).
//  - Within the CTA a head tile is split over TH threads: a row of d_state elements is VR
//    consecutive lanes, each holding one 16-byte vector per pass; each thread keeps its part
//    of the tile in fp32 registers across the (speculative) tokens.
//  - C.h is a row sum over VR lanes: a reduce-scatter of the per-pass partials (halving the
//    values exchanged at each shuffle step) leaves one row total per lane pair.
//  - The first head's state loads are issued before the conv phase so they are in flight
//    while the CTA convolves.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "umma.cuh"

namespace ms {

// ---------------------------------------------------------------------------------------
// tile geometry of one head's (head_dim x d_state) state
// ---------------------------------------------------------------------------------------

template <typename StateT, int P, int N>
struct Tile {
    static constexpr int VEC = Vec16<StateT>::n;  // elements per 16-byte vector
    static constexpr int VR = N / VEC;            // vectors (= lanes) per state row
    static constexpr int TV = P * N / VEC;        // vectors per head tile
    static constexpr int PR = TV / 128;
    static constexpr int PASSES = PR < 1 ? 1 : (PR > 8 ? 8 : PR);  // vectors per thread
    static constexpr int TH = TV / PASSES;        // threads per head tile
    static constexpr int RP = TH / VR;            // rows covered per pass
    static_assert(N % VEC == 0, "d_state must fill whole 16-byte vectors");
    static_assert(TV % PASSES == 0 && TH % 32 == 0 && TH <= 512, "tile must split into warps");
    static_assert(VR <= 32 && (VR & (VR - 1)) == 0, "a state row must sit inside one warp");
    static_assert(PASSES <= VR, "reduce-scatter needs at least as many lanes as partials");
};

// Reduce-scatter of CNT partials over the lanes that differ in bits OFF, OFF/2, ..., 1.
// Halving steps exchange half the values; once one value is left the rest are butterflies.
// On return v[0] is the full sum for partial index `idx`.
template <int CNT, int OFF>
struct ReduceScatter {
    static __device__ __forceinline__ void run(float *v, int lane, int &idx) {
        if constexpr (OFF == 0) {
            return;
        } else if constexpr (CNT > 1) {
            constexpr int HALF = CNT / 2;
            const bool upper = (lane & OFF) != 0;
#pragma unroll
            for (int k = 0; k < HALF; ++k) {
                const float send = upper ? v[k] : v[k + HALF];
                const float keep = upper ? v[k + HALF] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
            }
            if (upper) idx += HALF;
            ReduceScatter<HALF, OFF / 2>::run(v, lane, idx);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
            ReduceScatter<1, OFF / 2>::run(v, lane, idx);
        }
    }
};

// ---------------------------------------------------------------------------------------
// conv phase: block-cooperative conv1d + SiLU over a set of channel ranges
// ---------------------------------------------------------------------------------------

// Up to three contiguous global-channel ranges, numbered back to back as local channels.
struct ChanRanges {
    int lo[3];
    int len[3];
    int total;
};

__device__ __forceinline__ int local_to_global(const ChanRanges &r, int lc) {
    if (lc < r.len[0]) return r.lo[0] + lc;
    lc -= r.len[0];
    if (lc < r.len[1]) return r.lo[1] + lc;
    return r.lo[2] + (lc - r.len[1]);
}

// Stages the old conv state and the raw inputs in shared memory, writes SiLU(conv) of every
// (token, local channel) to xs[ntok][LC], and writes the shifted conv state back.
//   cstate: the slot's conv state (conv_dim x Wc, oldest column first), global memory.
//   u_row:  this row's raw inputs, (ntok x Cd).
template <typename ActT>
__device__ __forceinline__ void conv_phase(const ChanRanges &cr, ActT *cstate, int Wc, int W, int ntok,
                                           const ActT *u_row, int Cd, const float *__restrict__ w,
                                           const float *__restrict__ b, ActT *cs, float *uraw,
                                           float *xs) {
    const int tid = threadIdx.x, nthr = blockDim.x, LC = cr.total;
    int base = 0;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        const ActT *src = cstate + (int64_t)cr.lo[r] * Wc;
        for (int e = tid; e < cr.len[r] * Wc; e += nthr) cs[base * Wc + e] = src[e];
        base += cr.len[r];
    }
    for (int idx = tid; idx < ntok * LC; idx += nthr) {
        const int j = idx / LC, lc = idx - j * LC;
        uraw[idx] = to_f32(u_row[(int64_t)j * Cd + local_to_global(cr, lc)]);
    }
    __syncthreads();
    for (int idx = tid; idx < ntok * LC; idx += nthr) {
        const int j = idx / LC, lc = idx - j * LC;
        const int c = local_to_global(cr, lc);
        float v = b ? b[c] : 0.0f;
        for (int k = 0; k < W; ++k) {
            const int m = Wc + j - (W - 1) + k;  // index into [old state (Wc) | new tokens]
            const float val = m < Wc ? to_f32(cs[lc * Wc + m]) : uraw[(m - Wc) * LC + lc];
            v = fmaf(w[(int64_t)c * W + k], val, v);
        }
        xs[idx] = silu_f(v);
    }
    // new column k is input ntok + k of [old state | new tokens]
    base = 0;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        ActT *dst = cstate + (int64_t)cr.lo[r] * Wc;
        for (int e = tid; e < cr.len[r] * Wc; e += nthr) {
            const int lcl = e / Wc, k = e - lcl * Wc, m = ntok + k;
            dst[e] = m < Wc ? cs[(base + lcl) * Wc + m]
                            : from_f32<ActT>(uraw[(m - Wc) * LC + base + lcl]);
        }
        base += cr.len[r];
    }
}

// Element e of a register array of 16-byte vectors holding raw 16-bit (PW = 2) or 32-bit (PW = 1)
// values; e is a compile-time constant once the callers' loops are unrolled.
template <int PW, int K>
__device__ __forceinline__ uint32_t raw_at(const uint4 (&a)[K], int e) {
    const int wi = e / PW;
    const uint4 &q = a[wi / 4];
    const int c = wi % 4;
    const uint32_t w = c == 0 ? q.x : (c == 1 ? q.y : (c == 2 ? q.z : q.w));
    if (PW == 1) return w;
    return (e & 1) ? (w >> 16) : (w & 0xffffu);
}

template <int PW>
__device__ __forceinline__ float raw_f32(uint32_t r) {
    return PW == 1 ? __uint_as_float(r) : __uint_as_float(r << 16);
}

__device__ __forceinline__ void set_word(uint4 &q, int c, uint32_t w) {
    if (c == 0) q.x = w;
    else if (c == 1) q.y = w;
    else if (c == 2) q.z = w;
    else q.w = w;
}

// The new window of V channels after NTK tokens: the last WC entries of [old window (WC) | tokens],
// per channel, assembled from the raw values.
template <typename ActT, int NTK, int WC>
__device__ __forceinline__ void conv_new_window(const uint4 (&win)[WC], const uint4 (&tok)[NTK], uint4 (&nw)[WC]) {
    constexpr int V = Vec16<ActT>::n, PW = (int)(4 / sizeof(ActT));
    auto input = [&](int v, int m) -> uint32_t {
        return m < WC ? raw_at<PW>(win, v * WC + m) : raw_at<PW>(tok, (m - WC) * V + v);
    };
#pragma unroll
    for (int wi = 0; wi < WC * 4; ++wi) {  // 32-bit words of the new window
        uint32_t word;
        if (PW == 1) {
            const int e = wi, v = e / WC, k = e - v * WC;
            word = input(v, NTK + k);
        } else {
            const int e0 = 2 * wi, e1 = e0 + 1;
            const int v0 = e0 / WC, k0 = e0 - v0 * WC, v1 = e1 / WC, k1 = e1 - v1 * WC;
            word = input(v0, NTK + k0) | (input(v1, NTK + k1) << 16);
        }
        set_word(nw[wi / 4], wi % 4, word);
    }
}

// Conv phase of one 16-byte vector of channels (V channels, local channels lc0 .. lc0 + V - 1) for
// NTK tokens with a W-tap kernel and a window of WC >= W-1 columns: the vector's window is WC
// contiguous 16-byte loads (a slot keeps each channel's columns together), every load is issued
// before any arithmetic, and the new window is assembled from the raw values, so the conv state
// stays bit-exact.  With write_window false the new window is left for conv_window_shift.
// SiLU for the per-(row, group) kernel: the fast intrinsics for single-token launches (small
// batches: batch 1 and 8 took 6.0 / 9.1 us per layer with the accurate forms, 5.4 / 8.6 with these),
// the accurate forms for several tokens (there the fast forms measured slower: 0.312 against
// 0.3035 ms per draft + commit step).
template <int NTOK>
__device__ __forceinline__ float silu_tok(float v) {
    if constexpr (NTOK == 1) return silu_fast(v);
    else return silu_f(v);
}

template <typename ActT, int W, int NTK, int WC>
__device__ __forceinline__ void conv_phase_vec(const ChanRanges &cr, ActT *cstate, const ActT *u_row, int Cd,
                                               const float *__restrict__ w, const float *__restrict__ b,
                                               float *xs, int lc0, bool write_window) {
    static_assert(WC >= W - 1, "the window holds at least the W-1 inputs before a token");
    constexpr int V = Vec16<ActT>::n, PW = (int)(4 / sizeof(ActT));
    const int LC = cr.total;
    const int c0 = local_to_global(cr, lc0);
    uint4 *sp = reinterpret_cast<uint4 *>(cstate + (int64_t)c0 * WC);
    uint4 win[WC], tok[NTK];
#pragma unroll
    for (int k = 0; k < WC; ++k) win[k] = sp[k];
#pragma unroll
    for (int j = 0; j < NTK; ++j) tok[j] = *reinterpret_cast<const uint4 *>(u_row + (int64_t)j * Cd + c0);
    float wv[V * W];  // wv[v * W + k]: tap k of channel c0 + v
#pragma unroll
    for (int q = 0; q < V * W / 4; ++q) {
        const float4 t = reinterpret_cast<const float4 *>(w + (int64_t)c0 * W)[q];
        wv[4 * q] = t.x;
        wv[4 * q + 1] = t.y;
        wv[4 * q + 2] = t.z;
        wv[4 * q + 3] = t.w;
    }
    float bv[V];
#pragma unroll
    for (int v = 0; v < V; ++v) bv[v] = b ? b[c0 + v] : 0.0f;
    // input m of [old window (WC) | tokens (NTK)] for channel v
    auto input = [&](int v, int m) -> uint32_t {
        return m < WC ? raw_at<PW>(win, v * WC + m) : raw_at<PW>(tok, (m - WC) * V + v);
    };
#pragma unroll
    for (int j = 0; j < NTK; ++j) {
        float o[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float acc = bv[v];
#pragma unroll
            for (int k = 0; k < W; ++k) acc = fmaf(wv[v * W + k], raw_f32<PW>(input(v, WC + j - (W - 1) + k)), acc);
            o[v] = silu_tok<NTK>(acc);
        }
        float4 *dst = reinterpret_cast<float4 *>(xs + (size_t)j * LC + lc0);
#pragma unroll
        for (int q = 0; q < V / 4; ++q) dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    }
    if (write_window) {
        uint4 nw[WC];
        conv_new_window<ActT, NTK, WC>(win, tok, nw);
#pragma unroll
        for (int k = 0; k < WC; ++k) sp[k] = nw[k];
    }
}

// The window update of one channel vector whose conv_phase_vec left it unwritten: the old window
// is read again (no other CTA writes it) and shifted by the tokens.
template <typename ActT, int NTK, int WC>
__device__ __forceinline__ void conv_window_shift(const ChanRanges &cr, ActT *cstate, const ActT *u_row, int Cd,
                                                  int lc0) {
    const int c0 = local_to_global(cr, lc0);
    uint4 *sp = reinterpret_cast<uint4 *>(cstate + (int64_t)c0 * WC);
    uint4 win[WC], tok[NTK], nw[WC];
#pragma unroll
    for (int k = 0; k < WC; ++k) win[k] = sp[k];
#pragma unroll
    for (int j = 0; j < NTK; ++j) tok[j] = *reinterpret_cast<const uint4 *>(u_row + (int64_t)j * Cd + c0);
    conv_new_window<ActT, NTK, WC>(win, tok, nw);
#pragma unroll
    for (int k = 0; k < WC; ++k) sp[k] = nw[k];
}

// The compiled vectorised conv forms: a 4-tap kernel, 1..4 tokens, a window of W-1 columns or of
// W-1+ntok (speculative columns).
template <typename ActT, int NTK>
__device__ __forceinline__ void conv_vec_wc(bool wc_min, const ChanRanges &cr, ActT *cst, const ActT *u_row, int Cd,
                                            const float *w, const float *b, float *xs, int lc0, bool wr) {
    if (wc_min) conv_phase_vec<ActT, 4, NTK, 3>(cr, cst, u_row, Cd, w, b, xs, lc0, wr);
    else conv_phase_vec<ActT, 4, NTK, 3 + NTK>(cr, cst, u_row, Cd, w, b, xs, lc0, wr);
}
template <typename ActT, int NT>
__device__ __forceinline__ void conv_vec(int ntok, bool wc_min, const ChanRanges &cr, ActT *cst, const ActT *u_row,
                                         int Cd, const float *w, const float *b, float *xs, int lc0, bool wr) {
    if constexpr (NT == 1) {
        conv_vec_wc<ActT, 1>(wc_min, cr, cst, u_row, Cd, w, b, xs, lc0, wr);
    } else {
        switch (ntok) {
            case 1: conv_vec_wc<ActT, 1>(wc_min, cr, cst, u_row, Cd, w, b, xs, lc0, wr); break;
            case 2: conv_vec_wc<ActT, 2>(wc_min, cr, cst, u_row, Cd, w, b, xs, lc0, wr); break;
            case 3: conv_vec_wc<ActT, 3>(wc_min, cr, cst, u_row, Cd, w, b, xs, lc0, wr); break;
            default: conv_vec_wc<ActT, 4>(wc_min, cr, cst, u_row, Cd, w, b, xs, lc0, wr); break;
        }
    }
}
template <typename ActT, int NTK>
__device__ __forceinline__ void shift_wc(bool wc_min, const ChanRanges &cr, ActT *cst, const ActT *u_row, int Cd, int lc0) {
    if (wc_min) conv_window_shift<ActT, NTK, 3>(cr, cst, u_row, Cd, lc0);
    else conv_window_shift<ActT, NTK, 3 + NTK>(cr, cst, u_row, Cd, lc0);
}
template <typename ActT, int NT>
__device__ __forceinline__ void shift_vec(int ntok, bool wc_min, const ChanRanges &cr, ActT *cst, const ActT *u_row,
                                          int Cd, int lc0) {
    if constexpr (NT == 1) {
        shift_wc<ActT, 1>(wc_min, cr, cst, u_row, Cd, lc0);
    } else {
        switch (ntok) {
            case 1: shift_wc<ActT, 1>(wc_min, cr, cst, u_row, Cd, lc0); break;
            case 2: shift_wc<ActT, 2>(wc_min, cr, cst, u_row, Cd, lc0); break;
            case 3: shift_wc<ActT, 3>(wc_min, cr, cst, u_row, Cd, lc0); break;
            default: shift_wc<ActT, 4>(wc_min, cr, cst, u_row, Cd, lc0); break;
        }
    }
}

// All threads of all CTAs of the cluster (hardware barrier; the CTAs of a cluster are co-resident).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------------------
// fused decode kernel
// ---------------------------------------------------------------------------------------

struct DecodeArgs {
    void *ssm_pool;
    int64_t ssm_stride;
    int64_t num_slots;
    void *conv_pool;
    int64_t conv_stride;
    const float *conv_w, *conv_b;
    const int32_t *slot, *scratch;
    int32_t batch, ntok;
    const void *xbc, *dt;
    int dt_bf16;
    const float *A, *D, *dt_bias;
    int dt_softplus;
    const void *z;
    void *y;
    int32_t *err;
    int H, G, HG, W, Wc, Cd;
    int sps;  // state-tile stages per head slot
    int vec;  // 16-byte vectorised conv / output phases (see DecodeSmem)
    int ksplit;  // CTAs (one cluster) per (row, group), each taking HG / ksplit heads
};

// Bound on the polls of one mbarrier wait (a copy that never lands is reported, not waited on forever).
constexpr uint32_t kMaxPolls = umma::kWaitPolls;
constexpr int kFlagWords = 16;

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~(size_t)15; }

// Shared-memory map of k_decode (byte offsets): S tile stages, S + 1 mbarriers (the last one for
// the z rows), the flags, then the per-row areas.  The vectorised form (vec) keeps the conv window
// in registers and stages the row's z values; the general form stages the old conv state and the
// raw inputs instead.
struct DecodeSmem {
    size_t bars, flags, xs, uraw, dl, da, ys, dh, scr, cs, zs, total;
    __host__ __device__ DecodeSmem(int S, size_t tile, int ntok, int LC, int HG, int P, int Wc, size_t es, bool conv,
                                   bool vec) {
        bars = (size_t)S * tile;
        flags = align16(bars + 8 * (size_t)(S + 1));
        size_t o = flags + sizeof(int) * kFlagWords;
        xs = o;    o = align16(o + sizeof(float) * (size_t)ntok * LC);     // [ntok][LC] x | B | C after the conv
        uraw = o;  if (conv && !vec) o = align16(o + sizeof(float) * (size_t)ntok * LC);  // raw inputs
        dl = o;    o = align16(o + sizeof(float) * (size_t)ntok * HG);     // [ntok][HG] Delta
        da = o;    o = align16(o + sizeof(float) * (size_t)ntok * HG);     // [ntok][HG] exp(Delta*A)
        ys = o;    o = align16(o + sizeof(float) * (size_t)ntok * HG * P); // [ntok][HG*P] C.h
        dh = o;    o = align16(o + sizeof(float) * (size_t)HG);            // D of the group's heads
        scr = o;   o = align16(o + sizeof(int) * (size_t)ntok);            // the row's scratch slots
        cs = o;    if (conv && !vec) o = align16(o + es * (size_t)LC * Wc);  // old conv state
        zs = o;    if (vec) o = align16(o + es * (size_t)ntok * HG * P);   // [ntok][HG*P] z
        total = o;
    }
};

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    umma::mbar_arrive_expect_tx(bar, bytes);
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     umma::smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(umma::smem_u32(bar))
                 : "memory");
}

// Bulk copy without expect_tx (the caller posts the total once).
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     umma::smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(umma::smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <typename StateT, int P, int N>
__device__ __forceinline__ void store_tile(const float (&st)[Tile<StateT, P, N>::PASSES][Tile<StateT, P, N>::VEC],
                                           StateT *base, int th) {
    using TL = Tile<StateT, P, N>;
#pragma unroll
    for (int pass = 0; pass < TL::PASSES; ++pass)
        __stcs(reinterpret_cast<uint4 *>(base) + pass * TL::TH + th, pack16(st[pass]));
}

// One CTA per (row, group).  Head tiles of the group are staged into shared memory by bulk
// asynchronous copies: each head slot (TH threads) owns `sps` stages, so up to sps tiles per slot
// are in flight while the slot computes; the first copies are issued before the conv phase.
template <typename StateT, typename ActT, int P, int N, int NT>
__global__ void __launch_bounds__(512) k_decode(const DecodeArgs a) {
    using TL = Tile<StateT, P, N>;
    constexpr int VEC = TL::VEC, VR = TL::VR, TH = TL::TH, RP = TL::RP, PASSES = TL::PASSES;
    constexpr uint32_t TILE_BYTES = (uint32_t)(P * N * sizeof(StateT));
    // blockIdx.x = group * ksplit + rank: the ksplit CTAs of a (row, group) form one cluster and
    // split the group's heads
    const int ksplit = a.ksplit, g = blockIdx.x / ksplit, rank = blockIdx.x - g * ksplit, i = blockIdx.y;
    const int ntok = NT > 0 ? NT : a.ntok;
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31;

    pdl_wait();
    pdl_launch_dependents();
    const int32_t s = a.slot[i];
    if (s == -1) return;  // padding row
    bool bad = s < -1 || s >= a.num_slots;
    if (a.scratch)
        for (int j = 0; j < ntok; ++j) {
            const int32_t d = a.scratch[(int64_t)i * ntok + j];
            bad |= d < -1 || d >= a.num_slots;
        }
    if (bad) {
        if (tid == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
        return;
    }

    const int HG = a.HG / ksplit, LC = HG * P + 2 * N;  // this CTA's heads and local channels
    const int hg0 = g * a.HG + rank * HG;                // global index of its first head
    const bool conv = a.conv_pool != nullptr, vec = a.vec != 0;
    const int hs = tid / TH, th = tid - hs * TH, NHS = nthr / TH;
    const int S = a.sps * NHS;  // stages; head hl uses stage hl % S, which belongs to slot hl % NHS
    extern __shared__ __align__(128) unsigned char dec_smem[];
    const DecodeSmem L(S, TILE_BYTES, ntok, LC, HG, P, a.Wc, sizeof(ActT), conv, vec);
    unsigned char *stages = dec_smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(dec_smem + L.bars);
    uint64_t *zbar = full + S;  // the z rows (vectorised form)
    int *flags = reinterpret_cast<int *>(dec_smem + L.flags);  // [0, NHS): slot timed out; [NHS]: any
    float *xs = reinterpret_cast<float *>(dec_smem + L.xs);
    float *uraw = reinterpret_cast<float *>(dec_smem + L.uraw);
    float *dl = reinterpret_cast<float *>(dec_smem + L.dl);
    float *da = reinterpret_cast<float *>(dec_smem + L.da);
    float *ys = reinterpret_cast<float *>(dec_smem + L.ys);
    float *dh = reinterpret_cast<float *>(dec_smem + L.dh);
    int *scr = reinterpret_cast<int *>(dec_smem + L.scr);
    ActT *cs = reinterpret_cast<ActT *>(dec_smem + L.cs);
    ActT *zs = reinterpret_cast<ActT *>(dec_smem + L.zs);

    if (tid == 0) {
        for (int st = 0; st < S; ++st) umma::mbar_init(&full[st], 1);
        umma::mbar_init(zbar, 1);
        umma::fence_mbar_init();
    }
    if (tid < kFlagWords) flags[tid] = 0;
    if (tid < ntok) scr[tid] = a.scratch ? a.scratch[(int64_t)i * ntok + tid] : -1;
    __syncthreads();

    StateT *pool = static_cast<StateT *>(a.ssm_pool);
    StateT *grp = pool + (int64_t)s * a.ssm_stride + (int64_t)hg0 * P * N;
    if (th == 0)
        for (int k = 0; k < a.sps; ++k) {
            const int hl = hs + k * NHS;
            if (hl < HG) bulk_load(stages + (size_t)(hl % S) * TILE_BYTES, grp + (int64_t)hl * P * N, TILE_BYTES,
                                   &full[hl % S]);
        }
    const int HP = a.H * P, GN = a.G * N;
    const bool zvec = vec && a.z != nullptr;
    if (zvec && tid == 0) {
        // the row's z values of the group's heads, one contiguous run per token
        const uint32_t zb = (uint32_t)(HG * P * sizeof(ActT));
        umma::mbar_arrive_expect_tx(zbar, zb * (uint32_t)ntok);
        for (int j = 0; j < ntok; ++j)
            bulk_copy(zs + (size_t)j * HG * P,
                      static_cast<const ActT *>(a.z) + ((int64_t)i * ntok + j) * HP + (int64_t)hg0 * P, zb, zbar);
    }

    const ActT *u_row = static_cast<const ActT *>(a.xbc) + (int64_t)i * ntok * a.Cd;
    ChanRanges cr;
    cr.lo[0] = hg0 * P;       cr.len[0] = HG * P;
    cr.lo[1] = HP + g * N;    cr.len[1] = N;
    cr.lo[2] = HP + GN + g * N; cr.len[2] = N;
    cr.total = LC;
    // Delta, exp(Delta*A) and D of the group's heads, by threads first, first + stride, ...
    auto dt_phase = [&](int first, int stride) {
        for (int idx = first; idx < ntok * HG; idx += stride) {
            const int j = idx / HG, h = hg0 + (idx - j * HG);
            const float sdt = load_scalar(a.dt, ((int64_t)i * ntok + j) * a.H + h, a.dt_bf16) +
                              (a.dt_bias ? a.dt_bias[h] : 0.0f);
            const float delta = a.dt_softplus ? softplus_f(sdt) : sdt;
            dl[idx] = delta;
            da[idx] = expf(delta * a.A[h]);
        }
        for (int hh = first; hh < HG; hh += stride) dh[hh] = a.D ? a.D[hg0 + hh] : 0.0f;
    };
    if (vec) {
        // one thread per 16-byte vector of channels; the threads left over do the per-head work
        constexpr int VA = Vec16<ActT>::n;
        const int nv = LC / VA;
        if (conv) {
            ActT *cst = static_cast<ActT *>(a.conv_pool) + (int64_t)s * a.conv_stride;
            // split: the group's B and C windows are read by every CTA of the cluster and written by
            // its first CTA after the cluster barrier below
            for (int v = tid; v < nv; v += nthr) {
                const bool wr = ksplit == 1 || v * VA < HG * P;
                conv_vec<ActT, NT>(ntok, a.Wc == 3, cr, cst, u_row, a.Cd, a.conv_w, a.conv_b, xs, v * VA, wr);
            }
        } else {
            for (int v = tid; v < ntok * nv; v += nthr) {
                const int j = v / nv, lc0 = (v - j * nv) * VA;
                float f[VA];
                unpack16(*reinterpret_cast<const uint4 *>(u_row + (int64_t)j * a.Cd + local_to_global(cr, lc0)), f);
                float4 *dst = reinterpret_cast<float4 *>(xs + (size_t)j * LC + lc0);
#pragma unroll
                for (int q = 0; q < VA / 4; ++q) dst[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
            }
        }
        const int busy = conv ? nv : ntok * nv;
        if (busy < nthr) {
            if (tid >= busy) dt_phase(tid - busy, nthr - busy);
        } else {
            dt_phase(tid, nthr);
        }
    } else {
        if (conv) {
            conv_phase<ActT>(cr, static_cast<ActT *>(a.conv_pool) + (int64_t)s * a.conv_stride, a.Wc, a.W,
                             ntok, u_row, a.Cd, a.conv_w, a.conv_b, cs, uraw, xs);
        } else {
            for (int idx = tid; idx < ntok * LC; idx += nthr) {
                const int j = idx / LC, lc = idx - j * LC;
                xs[idx] = to_f32(u_row[(int64_t)j * a.Cd + local_to_global(cr, lc)]);
            }
        }
        dt_phase(tid, nthr);
    }
    if (ksplit > 1) {
        cluster_sync();  // every CTA of the cluster has read the old B and C windows
        if (conv && rank == 0) {
            constexpr int VA = Vec16<ActT>::n;
            ActT *cst = static_cast<ActT *>(a.conv_pool) + (int64_t)s * a.conv_stride;
            for (int v = HG * P / VA + tid; v < LC / VA; v += nthr)
                shift_vec<ActT, NT>(ntok, a.Wc == 3, cr, cst, u_row, a.Cd, v * VA);
        }
    }
    __syncthreads();

    const int rsub = th / VR, n0 = (th - rsub * VR) * VEC;
    int hl = hs;
    for (; hl < HG; hl += NHS) {  // slot-uniform: TH is a multiple of 32
        const int stg = hl % S;
        if (th == 0 && !umma::mbar_wait(&full[stg], (uint32_t)(hl / S) & 1u, kMaxPolls)) flags[hs] = 1;
        named_sync(1 + hs, TH);
        if (flags[hs]) break;
        const uint4 *tile = reinterpret_cast<const uint4 *>(stages + (size_t)stg * TILE_BYTES);
        float part[PASSES];
        if constexpr (NT == 1) {
            // single token: stream the tile through registers vector by vector
            const float dA = da[hl], dlt = dl[hl];
            float Bv[VEC], Cv[VEC];
#pragma unroll
            for (int e = 0; e < VEC; e += 4) {
                const float4 b4 = *reinterpret_cast<const float4 *>(xs + HG * P + n0 + e);
                const float4 c4 = *reinterpret_cast<const float4 *>(xs + HG * P + N + n0 + e);
                Bv[e] = b4.x; Bv[e + 1] = b4.y; Bv[e + 2] = b4.z; Bv[e + 3] = b4.w;
                Cv[e] = c4.x; Cv[e + 1] = c4.y; Cv[e + 2] = c4.z; Cv[e + 3] = c4.w;
            }
            StateT *dst = grp + (int64_t)hl * P * N;
            if (a.scratch) {
                const int32_t d = scr[0];
                dst = d >= 0 ? pool + (int64_t)d * a.ssm_stride + (int64_t)(hg0 + hl) * P * N : nullptr;
            }
#pragma unroll
            for (int pass = 0; pass < PASSES; ++pass) {
                float f[VEC];
                unpack16(tile[pass * TH + th], f);
                const float dtx = dlt * xs[hl * P + pass * RP + rsub];
                float acc = 0.0f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    f[e] = fmaf(dA, f[e], dtx * Bv[e]);
                    acc = fmaf(Cv[e], f[e], acc);
                }
                part[pass] = acc;
                if (dst) __stcs(reinterpret_cast<uint4 *>(dst) + pass * TH + th, pack16(f));
            }
            named_sync(1 + hs, TH);  // every thread of the slot has read the stage
            if (th == 0 && hl + S < HG)
                bulk_load(stages + (size_t)stg * TILE_BYTES, grp + (int64_t)(hl + S) * P * N, TILE_BYTES, &full[stg]);
            int idx = 0;
            ReduceScatter<PASSES, VR / 2>::run(part, lane, idx);
            if ((lane & (VR / PASSES - 1)) == 0) ys[hl * P + idx * RP + rsub] = part[0];
        } else {
            // several tokens: the tile stays in fp32 registers across them
            float st[PASSES][VEC];
#pragma unroll
            for (int pass = 0; pass < PASSES; ++pass) unpack16(tile[pass * TH + th], st[pass]);
            // the stage is refilled by an asynchronous bulk copy right after the barrier, while the
            // values just read are first used later: order the reads before that copy
            umma::fence_async_smem();
            named_sync(1 + hs, TH);
            if (th == 0 && hl + S < HG)
                bulk_load(stages + (size_t)stg * TILE_BYTES, grp + (int64_t)(hl + S) * P * N, TILE_BYTES, &full[stg]);
            for (int j = 0; j < ntok; ++j) {
                const float dA = da[j * HG + hl], dlt = dl[j * HG + hl];
                const float *xj = xs + j * LC;
                float Bv[VEC], Cv[VEC];
#pragma unroll
                for (int e = 0; e < VEC; e += 4) {
                    const float4 b4 = *reinterpret_cast<const float4 *>(xj + HG * P + n0 + e);
                    const float4 c4 = *reinterpret_cast<const float4 *>(xj + HG * P + N + n0 + e);
                    Bv[e] = b4.x; Bv[e + 1] = b4.y; Bv[e + 2] = b4.z; Bv[e + 3] = b4.w;
                    Cv[e] = c4.x; Cv[e + 1] = c4.y; Cv[e + 2] = c4.z; Cv[e + 3] = c4.w;
                }
#pragma unroll
                for (int pass = 0; pass < PASSES; ++pass) {
                    const float dtx = dlt * xj[hl * P + pass * RP + rsub];
                    float acc = 0.0f;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        st[pass][e] = fmaf(dA, st[pass][e], dtx * Bv[e]);
                        acc = fmaf(Cv[e], st[pass][e], acc);
                    }
                    part[pass] = acc;
                }
                int idx = 0;
                ReduceScatter<PASSES, VR / 2>::run(part, lane, idx);
                if ((lane & (VR / PASSES - 1)) == 0) ys[j * HG * P + hl * P + idx * RP + rsub] = part[0];
                if (a.scratch) {
                    const int32_t d = scr[j];
                    if (d >= 0)
                        store_tile<StateT, P, N>(st, pool + (int64_t)d * a.ssm_stride + (int64_t)(hg0 + hl) * P * N,
                                                 th);
                }
            }
            if (!a.scratch) store_tile<StateT, P, N>(st, grp + (int64_t)hl * P * N, th);
        }
    }
    if (hl < HG) {
        // a copy did not land in time: report it, let this slot's copies that are still in flight
        // finish (bounded), and skip the outputs of this row
        if (th == 0) {
            flag_error(a.err, MAMBA_ERR_TIMEOUT);
            flags[NHS] = 1;
            for (int h2 = hl + NHS; h2 < HG && h2 < hl + S; h2 += NHS)
                umma::mbar_wait(&full[h2 % S], (uint32_t)(h2 / S) & 1u, kMaxPolls);
        }
    }
    __syncthreads();
    if (flags[NHS]) {
        if (zvec && tid == 0) umma::mbar_wait(zbar, 0, kMaxPolls);  // the z copies still in flight (bounded)
        return;
    }

    // y = C.h + D*x, gated by SiLU(z)
    ActT *yr = static_cast<ActT *>(a.y);
    if (vec) {
        constexpr int VA = Vec16<ActT>::n;
        if (zvec) {
            if (tid == 0 && !umma::mbar_wait(zbar, 0, kMaxPolls)) {
                flag_error(a.err, MAMBA_ERR_TIMEOUT);
                flags[NHS] = 1;
            }
            __syncthreads();
            if (flags[NHS]) return;
        }
        const int nvy = HG * P / VA;
        for (int v = tid; v < ntok * nvy; v += nthr) {
            const int j = v / nvy, lc0 = (v - j * nvy) * VA;
            const float Dh = dh[lc0 / P];
            const float4 *x4 = reinterpret_cast<const float4 *>(xs + (size_t)j * LC + lc0);
            const float4 *y4 = reinterpret_cast<const float4 *>(ys + (size_t)j * HG * P + lc0);
            float zf[VA], o[VA];
            if (zvec) unpack16(*reinterpret_cast<const uint4 *>(zs + (size_t)j * HG * P + lc0), zf);
#pragma unroll
            for (int q = 0; q < VA / 4; ++q) {
                const float4 xv = x4[q], yv = y4[q];
                o[4 * q] = fmaf(Dh, xv.x, yv.x);
                o[4 * q + 1] = fmaf(Dh, xv.y, yv.y);
                o[4 * q + 2] = fmaf(Dh, xv.z, yv.z);
                o[4 * q + 3] = fmaf(Dh, xv.w, yv.w);
            }
            if (zvec) {
#pragma unroll
                for (int e = 0; e < VA; ++e) o[e] *= silu_tok<NT>(zf[e]);
            }
            *reinterpret_cast<uint4 *>(yr + ((int64_t)i * ntok + j) * HP + (int64_t)hg0 * P + lc0) = pack16(o);
        }
        return;
    }
    const ActT *zr = static_cast<const ActT *>(a.z);
    for (int idx = tid; idx < ntok * HG * P; idx += nthr) {
        const int j = idx / (HG * P), lc = idx - j * HG * P;
        const float xv = xs[j * LC + lc];
        float yv = fmaf(dh[lc / P], xv, ys[idx]);
        const int64_t o = ((int64_t)i * ntok + j) * HP + (int64_t)hg0 * P + lc;
        if (zr) yv *= silu_tok<NT>(to_f32(zr[o]));
        yr[o] = from_f32<ActT>(yv);
    }
}

// ---------------------------------------------------------------------------------------
// single-token decode as a persistent, warp-specialised stream
// ---------------------------------------------------------------------------------------
//
// Work item = (row, group).  Each CTA walks the items b, b + gridDim, ... with three roles:
//   producer warp:   bulk-copies the state tiles of its items, in order, into a ring of NS
//                    shared-memory stages, running ahead of the consumers by up to NS tiles
//                    (across item boundaries, so the copies never stop at an item's edge);
//   conv warps:      for the next item, the causal conv + SiLU of the group's x|B|C channels,
//                    the conv-state shift, Delta / exp(Delta*A) and the z gate values, into one
//                    of two per-item buffers;
//   consumer warps:  per tile, h <- exp(Delta*A) h + Delta x B^T, C.h, the state write-back, and
//                    after all of an item's heads, y = C.h + D x gated by SiLU(z).
// All waits are bounded: a wait that gives up sets the CTA's abort flag, every role stops, and
// the copies still in flight are drained (bounded) before the CTA exits.

constexpr int kStreamConsumers = 256;  // consumer threads (head slots of TH threads)
constexpr int kStreamConv = 128;       // conv threads
constexpr int kStreamThreads = kStreamConsumers + kStreamConv + 32;

struct StreamArgs {
    DecodeArgs d;
    int ns;  // tile stages
};

// Per-item buffer (byte offsets): xs[LC] | dl[HG] | da[HG] floats, the raw z row (ActT), ys[HG*P]
// floats; every part 16-byte aligned.
struct ItemLayout {
    size_t dl, da, zr, ys, bytes;
    __host__ __device__ ItemLayout(int LC, int HG, int P, size_t es) {
        dl = sizeof(float) * (size_t)LC;
        da = dl + sizeof(float) * (size_t)HG;
        zr = align16(da + sizeof(float) * (size_t)HG);
        ys = align16(zr + es * (size_t)HG * P);
        bytes = align16(ys + sizeof(float) * (size_t)HG * P);
    }
};

// Shared-memory map of the stream kernel (byte offsets).  The conv inputs of an item (old conv
// state, raw xBC, z row, dt slice) are double-buffered so the next item's copies overlap this one.
struct StreamSmem {
    size_t bars, flags, items, item_bytes, wsm, ga, gb, in0, in_bytes, cs, ur, zin, dts, total;
    __host__ __device__ StreamSmem(int ns, size_t tile, int LC, int HG, int P, int W, int Wc, size_t es, size_t dt_es) {
        bars = (size_t)ns * tile;                          // stages first (16-byte aligned tiles)
        flags = align16(bars + 8 * (size_t)(2 * ns + 8));  // full/empty, xs_full/empty, cons, conv, conv_in[2]
        items = flags + 16;                                // abort, issued
        item_bytes = ItemLayout(LC, HG, P, es).bytes;
        wsm = items + 2 * item_bytes;                      // conv taps of the cached group
        ga = align16(wsm + sizeof(float) * (size_t)LC * W);  // A of the cached group's heads
        gb = align16(ga + sizeof(float) * (size_t)HG);     // dt_bias of the cached group's heads
        in0 = align16(gb + sizeof(float) * (size_t)HG);
        cs = 0;                                            // offsets inside one input buffer:
        ur = align16(cs + es * (size_t)LC * Wc);           //   old conv state, raw xBC,
        zin = align16(ur + es * (size_t)LC);               //   z row,
        dts = align16(zin + es * (size_t)HG * P);          //   dt slice
        in_bytes = align16(dts + dt_es * (size_t)HG);
        total = in0 + 2 * in_bytes;
    }
};

__device__ __forceinline__ bool stream_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    for (uint32_t i = 0; i < kMaxPolls; ++i) {
        if (umma::mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 1023u && *abort) return false;
    }
    *abort = 1;
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(umma::smem_u32(bar)) : "memory");
}

// Bounded barrier among the members of one role: each member arrives, then waits for the phase.
// (No hardware named barrier is used inside the stream kernel, so a member that gives up can never
// leave the others blocked.)
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t &phase, volatile int *abort) {
    mbar_arrive(bar);
    const bool ok = stream_wait(bar, phase & 1u, abort);
    ++phase;
    return ok;
}

template <typename StateT, typename ActT, int P, int N>
__global__ void __launch_bounds__(kStreamThreads, 1) k_decode_stream(const StreamArgs sa) {
    using TL = Tile<StateT, P, N>;
    constexpr int VEC = TL::VEC, VR = TL::VR, TH = TL::TH, RP = TL::RP, PASSES = TL::PASSES;
    constexpr int NHS = kStreamConsumers / TH;
    constexpr uint32_t TILE_BYTES = (uint32_t)(P * N * sizeof(StateT));
    constexpr int ES = (int)sizeof(ActT);
    const DecodeArgs &a = sa.d;
    const int NS = sa.ns, HG = a.HG, LC = HG * P + 2 * N, G = a.G, Wk = a.W, Wc = a.Wc;
    const int HP = a.H * P, GN = a.G * N;
    const int tid = threadIdx.x;
    const int W = a.batch * G;
    const size_t DTES = a.dt_bf16 ? 2 : 4;
    const StreamSmem L(NS, TILE_BYTES, LC, HG, P, Wk, Wc, ES, DTES);

    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ __align__(128) unsigned char st_smem[];
    unsigned char *stages = st_smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(st_smem + L.bars);
    uint64_t *empty = full + NS;
    uint64_t *xs_full = empty + NS;    // [2]
    uint64_t *xs_empty = xs_full + 2;  // [2]
    uint64_t *cons_bar = xs_empty + 2;
    uint64_t *conv_bar = cons_bar + 1;
    uint64_t *conv_in = conv_bar + 1;  // [2]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(st_smem + L.flags);
    int *issued = reinterpret_cast<int *>(st_smem + L.flags) + 1;  // tiles issued by the producer
    const ItemLayout IL(LC, HG, P, ES);
    auto item = [&](int e) { return st_smem + L.items + (size_t)e * L.item_bytes; };
    float *wsm = reinterpret_cast<float *>(st_smem + L.wsm);
    float *gA = reinterpret_cast<float *>(st_smem + L.ga);
    float *gBias = reinterpret_cast<float *>(st_smem + L.gb);
    auto inbuf = [&](int b) { return st_smem + L.in0 + (size_t)b * L.in_bytes; };

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            umma::mbar_init(&full[s], 1);
            umma::mbar_init(&empty[s], TH);
        }
        for (int e = 0; e < 2; ++e) {
            umma::mbar_init(&xs_full[e], kStreamConv);
            umma::mbar_init(&xs_empty[e], kStreamConsumers);
        }
        umma::mbar_init(cons_bar, kStreamConsumers);
        umma::mbar_init(conv_bar, kStreamConv);
        umma::mbar_init(&conv_in[0], 1);
        umma::mbar_init(&conv_in[1], 1);
        umma::fence_mbar_init();
        *abort_flag = 0;
        *issued = 0;
    }
    __syncthreads();

    StateT *pool = static_cast<StateT *>(a.ssm_pool);
    // the slot of an item, or -1 when the item is skipped (padding row, or a slot outside the pool)
    auto item_slot = [&](int w) -> int32_t {
        const int32_t s = a.slot[w / G];
        return (s >= 0 && s < a.num_slots) ? s : -1;
    };

    if (tid >= kStreamConsumers + kStreamConv) {
        // ---------------- producer warp ----------------
        if (tid == kStreamConsumers + kStreamConv) {
            int t = 0;
            for (int w = blockIdx.x; w < W && !*abort_flag; w += gridDim.x) {
                const int32_t s = a.slot[w / G];
                if ((s < -1 || s >= a.num_slots) && w % G == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
                if (s < 0 || s >= a.num_slots) continue;
                const StateT *grp = pool + (int64_t)s * a.ssm_stride + (int64_t)(w % G) * HG * P * N;
                for (int hl = 0; hl < HG; ++hl, ++t) {
                    const int st = t % NS;
                    if (t >= NS && !stream_wait(&empty[st], (uint32_t)(t / NS - 1) & 1u, abort_flag)) break;
                    bulk_load(stages + (size_t)st * TILE_BYTES, grp + (int64_t)hl * P * N, TILE_BYTES, &full[st]);
                }
                *issued = t;
            }
            *issued = t;
        }
    } else if (tid >= kStreamConsumers) {
        // ---------------- conv warps ----------------
        // An item's conv inputs arrive by bulk copies into one of two input buffers: the next
        // item's copies are issued while this item is convolved.  The conv taps, A and dt_bias of
        // the item's group are cached and reloaded only when the group changes.
        const int ct = tid - kStreamConsumers;
        const size_t xseg = (size_t)HG * P, bseg = N;  // channels per segment: x | B | C
        auto next_valid = [&](int w) {
            while (w < W && item_slot(w) < 0) {
                if (ct == 0 && w % G == 0 && (a.slot[w / G] < -1 || a.slot[w / G] >= a.num_slots))
                    flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
                w += gridDim.x;
            }
            return w;
        };
        // issue the conv inputs of item w into input buffer b (and the group's parameters)
        auto issue_inputs = [&](int w, int b, bool params) {
            const int i = w / G, g = w % G;
            const int32_t s = item_slot(w);
            const int lo[3] = {g * HG * P, HP + g * N, HP + GN + g * N};
            const size_t len[3] = {xseg, bseg, bseg};
            unsigned char *ib = inbuf(b);
            uint32_t bytes = (uint32_t)((size_t)LC * Wc * ES + (size_t)LC * ES + (a.z ? (size_t)HG * P * ES : 0) +
                                        (size_t)HG * DTES);
            if (params) bytes += (uint32_t)(sizeof(float) * ((size_t)LC * Wk + HG + (a.dt_bias ? HG : 0)));
            umma::fence_async_smem();
            umma::mbar_arrive_expect_tx(&conv_in[b], bytes);
            const ActT *cstate = static_cast<const ActT *>(a.conv_pool) + (int64_t)s * a.conv_stride;
            const ActT *u_row = static_cast<const ActT *>(a.xbc) + (int64_t)i * a.Cd;
            size_t base = 0;
            for (int r = 0; r < 3; ++r) {
                bulk_copy(reinterpret_cast<ActT *>(ib + L.cs) + base * Wc, cstate + (int64_t)lo[r] * Wc,
                          (uint32_t)(len[r] * Wc * ES), &conv_in[b]);
                bulk_copy(reinterpret_cast<ActT *>(ib + L.ur) + base, u_row + lo[r], (uint32_t)(len[r] * ES), &conv_in[b]);
                if (params)
                    bulk_copy(wsm + base * Wk, a.conv_w + (int64_t)lo[r] * Wk, (uint32_t)(len[r] * Wk * sizeof(float)),
                              &conv_in[b]);
                base += len[r];
            }
            if (a.z)
                bulk_copy(ib + L.zin, static_cast<const ActT *>(a.z) + (int64_t)i * HP + (int64_t)g * HG * P,
                          (uint32_t)((size_t)HG * P * ES), &conv_in[b]);
            bulk_copy(ib + L.dts, static_cast<const unsigned char *>(a.dt) + ((int64_t)i * a.H + (int64_t)g * HG) * DTES,
                      (uint32_t)(HG * DTES), &conv_in[b]);
            if (params) {
                bulk_copy(gA, a.A + (int64_t)g * HG, (uint32_t)(HG * sizeof(float)), &conv_in[b]);
                if (a.dt_bias) bulk_copy(gBias, a.dt_bias + (int64_t)g * HG, (uint32_t)(HG * sizeof(float)), &conv_in[b]);
            }
        };
        uint32_t cph = 0, iph[2] = {0u, 0u}, issued_in[2] = {0u, 0u};
        int n = 0;
        int w = next_valid(blockIdx.x);
        if (ct == 0 && w < W) {
            issue_inputs(w, 0, true);
            ++issued_in[0];
        }
        while (w < W) {
            const int b = n & 1, e = n & 1;
            const int g = w % G, i = w / G;
            const int wn = next_valid(w + gridDim.x);
            const bool same_group = wn < W && wn % G == g;
            if (ct == 0 && same_group) {  // overlaps this item
                issue_inputs(wn, b ^ 1, false);
                ++issued_in[b ^ 1];
            }
            if (n >= 2 && !stream_wait(&xs_empty[e], (uint32_t)(n / 2 - 1) & 1u, abort_flag)) break;
            if (!stream_wait(&conv_in[b], iph[b] & 1u, abort_flag)) break;
            ++iph[b];
            const int32_t s = item_slot(w);
            const int lo[3] = {g * HG * P, HP + g * N, HP + GN + g * N};
            unsigned char *ib = inbuf(b), *it = item(e);
            const ActT *cs = reinterpret_cast<const ActT *>(ib + L.cs);
            const ActT *ur = reinterpret_cast<const ActT *>(ib + L.ur);
            float *xs = reinterpret_cast<float *>(it), *dl = reinterpret_cast<float *>(it + IL.dl),
                  *da = reinterpret_cast<float *>(it + IL.da);
            ActT *cstate = static_cast<ActT *>(a.conv_pool) + (int64_t)s * a.conv_stride;
            // conv + SiLU per channel; the channel's shifted window goes straight back to the pool
            for (int lc = ct; lc < LC; lc += kStreamConv) {
                const int r = lc < (int)xseg ? 0 : (lc < (int)(xseg + bseg) ? 1 : 2);
                const int c = lo[r] + lc - (r == 0 ? 0 : (r == 1 ? (int)xseg : (int)(xseg + bseg)));
                float v = a.conv_b ? a.conv_b[c] : 0.0f;
                const ActT *win = cs + lc * Wc;
                const ActT u = ur[lc];
                if (Wk == 4) {
                    const float4 w4 = *reinterpret_cast<const float4 *>(wsm + lc * 4);
                    v = fmaf(w4.x, to_f32(win[Wc - 3]), v);
                    v = fmaf(w4.y, to_f32(win[Wc - 2]), v);
                    v = fmaf(w4.z, to_f32(win[Wc - 1]), v);
                    v = fmaf(w4.w, to_f32(u), v);
                } else {
                    for (int k = 0; k < Wk; ++k) {
                        const int m = Wc - (Wk - 1) + k;
                        v = fmaf(wsm[lc * Wk + k], to_f32(m < Wc ? win[m] : u), v);
                    }
                }
                xs[lc] = silu_fast(v);
                ActT *nw = cstate + (int64_t)c * Wc;
                for (int k = 0; k + 1 < Wc; ++k) nw[k] = win[k + 1];
                nw[Wc - 1] = u;
            }
            if (a.z) {
                const uint4 *zsrc = reinterpret_cast<const uint4 *>(ib + L.zin);
                uint4 *zdst = reinterpret_cast<uint4 *>(it + IL.zr);
                for (int q = ct; q < (int)((size_t)HG * P * ES / 16); q += kStreamConv) zdst[q] = zsrc[q];
            }
            for (int hl = ct; hl < HG; hl += kStreamConv) {
                const float sdt = load_scalar(ib + L.dts, hl, a.dt_bf16) + (a.dt_bias ? gBias[hl] : 0.0f);
                const float delta = a.dt_softplus ? softplus_f(sdt) : sdt;
                dl[hl] = delta;
                da[hl] = expf(delta * gA[hl]);
            }
            mbar_arrive(&xs_full[e]);
            if (!group_sync(conv_bar, cph, abort_flag)) break;  // buffer b and the taps are no longer read
            if (ct == 0 && wn < W && !same_group) {
                issue_inputs(wn, b ^ 1, true);
                ++issued_in[b ^ 1];
            }
            (void)i;
            w = wn;
            ++n;
        }
        // after an abort, input copies this role issued may still be landing: wait for them (bounded)
        if (ct == 0)
            for (int b = 0; b < 2; ++b)
                if (issued_in[b] > iph[b]) umma::mbar_wait(&conv_in[b], iph[b] & 1u, kMaxPolls);
    } else {
        // ---------------- consumer warps ----------------
        const int hs = tid / TH, th = tid - hs * TH, lane = tid & 31;
        const int rsub = th / VR, n0 = (th - rsub * VR) * VEC;
        uint32_t bph = 0;
        int n = 0, t0 = 0;
        for (int w = blockIdx.x; w < W; w += gridDim.x) {
            const int32_t s = item_slot(w);
            if (s < 0) continue;
            const int e = n & 1;
            if (!stream_wait(&xs_full[e], (uint32_t)(n / 2) & 1u, abort_flag)) break;
            const int i = w / G, g = w % G;
            unsigned char *it = item(e);
            const float *xs = reinterpret_cast<const float *>(it), *dl = reinterpret_cast<const float *>(it + IL.dl),
                        *da = reinterpret_cast<const float *>(it + IL.da);
            const ActT *zraw = reinterpret_cast<const ActT *>(it + IL.zr);
            float *ys = reinterpret_cast<float *>(it + IL.ys);
            StateT *grp = pool + (int64_t)s * a.ssm_stride + (int64_t)g * HG * P * N;
            float Bv[VEC], Cv[VEC];
#pragma unroll
            for (int q = 0; q < VEC; q += 4) {
                const float4 b4 = *reinterpret_cast<const float4 *>(xs + HG * P + n0 + q);
                const float4 c4 = *reinterpret_cast<const float4 *>(xs + HG * P + N + n0 + q);
                Bv[q] = b4.x; Bv[q + 1] = b4.y; Bv[q + 2] = b4.z; Bv[q + 3] = b4.w;
                Cv[q] = c4.x; Cv[q + 1] = c4.y; Cv[q + 2] = c4.z; Cv[q + 3] = c4.w;
            }
            bool stop = false;
            for (int hl = hs; hl < HG; hl += NHS) {
                // stage st only ever holds this slot's tiles (the host sizes NS for that), so the
                // phase before t / NS is one this slot has already consumed
                const int t = t0 + hl, st = t % NS;
                if (!stream_wait(&full[st], (uint32_t)(t / NS) & 1u, abort_flag)) {
                    stop = true;
                    break;
                }
                const uint4 *tile = reinterpret_cast<const uint4 *>(stages + (size_t)st * TILE_BYTES);
                uint4 raw[PASSES];
#pragma unroll
                for (int pass = 0; pass < PASSES; ++pass) raw[pass] = tile[pass * TH + th];
                mbar_arrive(&empty[st]);  // the stage can be refilled
                const float dA = da[hl], dlt = dl[hl];
                StateT *dst = grp + (int64_t)hl * P * N;
                float part[PASSES];
#pragma unroll
                for (int pass = 0; pass < PASSES; ++pass) {
                    float f[VEC];
                    unpack16(raw[pass], f);
                    const float dtx = dlt * xs[hl * P + pass * RP + rsub];
                    float acc = 0.0f;
#pragma unroll
                    for (int q = 0; q < VEC; ++q) {
                        f[q] = fmaf(dA, f[q], dtx * Bv[q]);
                        acc = fmaf(Cv[q], f[q], acc);
                    }
                    part[pass] = acc;
                    __stcs(reinterpret_cast<uint4 *>(dst) + pass * TH + th, pack16(f));
                }
                int idx = 0;
                ReduceScatter<PASSES, VR / 2>::run(part, lane, idx);
                if ((lane & (VR / PASSES - 1)) == 0) ys[hl * P + idx * RP + rsub] = part[0];
            }
            if (stop) break;
            if (!group_sync(cons_bar, bph, abort_flag)) break;  // every head of the item is reduced
            ActT *yr = static_cast<ActT *>(a.y) + (int64_t)i * HP + (int64_t)g * HG * P;
            for (int q = tid; q < HG * P; q += kStreamConsumers) {
                const int h = g * HG + q / P;
                const float xv = xs[q];
                float yv = ys[q] + (a.D ? a.D[h] * xv : 0.0f);
                if (a.z) yv *= silu_fast(to_f32(zraw[q]));
                yr[q] = from_f32<ActT>(yv);
            }
            mbar_arrive(&xs_empty[e]);
            t0 += HG;
            ++n;
        }
    }
    __syncthreads();
    if (tid == 0 && *abort_flag) {
        // report, and let every copy this CTA issued land before its shared memory is released
        flag_error(a.err, MAMBA_ERR_TIMEOUT);
        const int ti = *issued;
        for (int t = ti - NS > 0 ? ti - NS : 0; t < ti; ++t) umma::mbar_wait(&full[t % NS], (uint32_t)(t / NS) & 1u, kMaxPolls);

    }
}

// ---------------------------------------------------------------------------------------
// standalone conv update
// ---------------------------------------------------------------------------------------

constexpr int CONV_CHANNELS = 256;

struct ConvArgs {
    void *conv_pool;
    int64_t conv_stride, num_slots;
    const int32_t *slot;
    int32_t ntok;
    const void *xbc_in;
    const float *w, *b;
    void *xbc_out;
    int32_t *err;
    int W, Wc, Cd;
};

// Single-token conv step for a window of exactly W-1 columns: one thread per 16-byte vector of
// channels (V = 8 bf16 or 4 fp32) and kConvRows batch rows, in small blocks so that a batch
// launches many of them.  The vector's taps (V x W fp32,
// contiguous) are loaded once as 16-byte vectors and reused for the rows; a slot keeps each
// channel's W-1 columns contiguous, so the vector's window is W-1 contiguous 16-byte loads.  All
// rows' loads are issued before any arithmetic; the new windows (shifted by one, the token
// appended) and the outputs are written back as 16-byte stores.
constexpr int kConvRows = 4;
constexpr int kConvThreads = 128;

template <typename ActT, int W>
__global__ void __launch_bounds__(kConvThreads) k_conv_step(const ConvArgs a, int batch) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int V = Vec16<ActT>::n;
    const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * V;
    if (c0 >= a.Cd) return;
    float wv[V * W];  // wv[v * W + k]: tap k of channel c0 + v
#pragma unroll
    for (int q = 0; q < V * W / 4; ++q) {
        const float4 t = reinterpret_cast<const float4 *>(a.w + (int64_t)c0 * W)[q];
        wv[4 * q] = t.x;
        wv[4 * q + 1] = t.y;
        wv[4 * q + 2] = t.z;
        wv[4 * q + 3] = t.w;
    }
    float bv[V];
#pragma unroll
    for (int v = 0; v < V; ++v) bv[v] = a.b ? a.b[c0 + v] : 0.0f;
    const int i0 = blockIdx.y * kConvRows;
    uint4 raw[kConvRows][W];  // [r][k < W-1]: the slot's window vectors, [r][W-1]: the token
    ActT *st[kConvRows];
#pragma unroll
    for (int r = 0; r < kConvRows; ++r) {
        st[r] = nullptr;
        const int i = i0 + r;
        if (i >= batch) continue;
        const int32_t s = a.slot[i];
        if (s == -1) continue;  // padding row
        if (s < -1 || s >= a.num_slots) {
            if (c0 == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
            continue;
        }
        st[r] = static_cast<ActT *>(a.conv_pool) + (int64_t)s * a.conv_stride + (int64_t)c0 * (W - 1);
#pragma unroll
        for (int k = 0; k < W - 1; ++k) raw[r][k] = reinterpret_cast<const uint4 *>(st[r])[k];
        raw[r][W - 1] = *reinterpret_cast<const uint4 *>(static_cast<const ActT *>(a.xbc_in) + (int64_t)i * a.Cd + c0);
    }
#pragma unroll
    for (int r = 0; r < kConvRows; ++r) {
        if (!st[r]) continue;
        // cur[v * (W-1) + c]: column c (oldest first) of channel c0 + v (the slot's channel-major
        // order); x[v]: the token
        float cur[V * (W - 1)], x[V];
#pragma unroll
        for (int k = 0; k < W - 1; ++k) {
            float f[V];
            unpack16(raw[r][k], f);
#pragma unroll
            for (int e = 0; e < V; ++e) cur[k * V + e] = f[e];
        }
        unpack16(raw[r][W - 1], x);
        float o[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float acc = fmaf(wv[v * W + W - 1], x[v], bv[v]);
#pragma unroll
            for (int c = 0; c < W - 1; ++c) acc = fmaf(wv[v * W + c], cur[v * (W - 1) + c], acc);
            o[v] = silu_fast(acc);
        }
        *reinterpret_cast<uint4 *>(static_cast<ActT *>(a.xbc_out) + (int64_t)(i0 + r) * a.Cd + c0) = pack16(o);
        // new window: every channel's columns shifted left by one, the token appended
        float nw[V * (W - 1)];
#pragma unroll
        for (int v = 0; v < V; ++v) {
#pragma unroll
            for (int c = 0; c + 1 < W - 1; ++c) nw[v * (W - 1) + c] = cur[v * (W - 1) + c + 1];
            nw[v * (W - 1) + W - 2] = x[v];
        }
#pragma unroll
        for (int k = 0; k < W - 1; ++k) {
            float f[V];
#pragma unroll
            for (int e = 0; e < V; ++e) f[e] = nw[k * V + e];
            reinterpret_cast<uint4 *>(st[r])[k] = pack16(f);
        }
    }
}

// Launches the single-token conv step when it applies (ntok 1, a window of W-1 columns, 16-byte
// aligned vectors); false when the general kernel must run instead.
template <typename ActT>
bool launch_conv_step(const ConvArgs &a, int batch, size_t ab, cudaStream_t st) {
    constexpr int V = Vec16<ActT>::n;
    if (a.ntok != 1 || a.Wc != a.W - 1 || a.Cd % V || !aligned16(a.conv_pool) || !aligned16(a.xbc_in) ||
        !aligned16(a.xbc_out) || !aligned16(a.w) || ((size_t)a.conv_stride * ab) % 16)
        return false;
    const dim3 grid((a.Cd / V + kConvThreads - 1) / kConvThreads, (batch + kConvRows - 1) / kConvRows);
    switch (a.W) {
        case 2: return launch_pdl(k_conv_step<ActT, 2>, grid, dim3(kConvThreads), 0, st, a, batch) == cudaSuccess;
        case 3: return launch_pdl(k_conv_step<ActT, 3>, grid, dim3(kConvThreads), 0, st, a, batch) == cudaSuccess;
        case 4: return launch_pdl(k_conv_step<ActT, 4>, grid, dim3(kConvThreads), 0, st, a, batch) == cudaSuccess;
        case 5: return launch_pdl(k_conv_step<ActT, 5>, grid, dim3(kConvThreads), 0, st, a, batch) == cudaSuccess;
        default: return false;
    }
}

template <typename ActT>
__global__ void __launch_bounds__(256) k_conv_update(const ConvArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    const int cb = blockIdx.x, i = blockIdx.y, ntok = a.ntok;
    const int32_t s = a.slot[i];
    if (s == -1) return;  // padding row
    if (s < -1 || s >= a.num_slots) {
        if (threadIdx.x == 0 && cb == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
        return;
    }
    ChanRanges cr;
    cr.lo[0] = cb * CONV_CHANNELS;
    cr.len[0] = min(CONV_CHANNELS, a.Cd - cr.lo[0]);
    cr.lo[1] = cr.lo[2] = 0;
    cr.len[1] = cr.len[2] = 0;
    cr.total = cr.len[0];
    const int LC = cr.total;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *xs = reinterpret_cast<float *>(smem_raw);
    float *uraw = xs + ntok * LC;
    ActT *cs = reinterpret_cast<ActT *>(uraw + ntok * LC);
    const ActT *u_row = static_cast<const ActT *>(a.xbc_in) + (int64_t)i * ntok * a.Cd;
    conv_phase<ActT>(cr, static_cast<ActT *>(a.conv_pool) + (int64_t)s * a.conv_stride, a.Wc, a.W, ntok,
                     u_row, a.Cd, a.w, a.b, cs, uraw, xs);
    ActT *out = static_cast<ActT *>(a.xbc_out) + (int64_t)i * ntok * a.Cd;
    for (int idx = threadIdx.x; idx < ntok * LC; idx += blockDim.x) {
        const int j = idx / LC, lc = idx - j * LC;
        out[(int64_t)j * a.Cd + cr.lo[0] + lc] = from_f32<ActT>(xs[idx]);
    }
}

// ---------------------------------------------------------------------------------------
// speculative commit
// ---------------------------------------------------------------------------------------

struct CommitArgs {
    void *ssm_pool;
    int64_t ssm_stride, num_slots;
    void *conv_pool;
    int64_t conv_stride;
    const int32_t *slot, *scratch, *accept;
    int32_t ntok;
    int32_t *err;
    int H, tile_vecs, Cd, Wc;
    int hpb;  // heads whose state tiles one block copies
};

// grid.x: H state-copy units (one head tile each) followed by conv units of CONV_CHANNELS
// channels; grid.y: batch rows.  Every unit of a row applies the same validity checks so a bad
// row is left entirely untouched.
template <typename ActT>
__global__ void __launch_bounds__(256) k_spec_commit(const CommitArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    const int unit = blockIdx.x, i = blockIdx.y, tid = threadIdx.x;
    const int32_t s = a.slot[i];
    if (s == -1) return;  // padding row
    if (s < -1) {
        if (unit == 0 && tid == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
        return;
    }
    const int32_t acc = a.accept[i];
    if (acc < 0 || acc > a.ntok) {
        if (unit == 0 && tid == 0) flag_error(a.err, MAMBA_ERR_ACCEPT_RANGE);
        return;
    }
    const int32_t src = acc >= 1 ? a.scratch[(int64_t)i * a.ntok + acc - 1] : 0;
    if (s >= a.num_slots || src < 0 || src >= a.num_slots) {
        if (unit == 0 && tid == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
        return;
    }
    const int ssm_units = (a.H + a.hpb - 1) / a.hpb;
    if (unit < ssm_units) {
        if (acc == 0) return;
        // the state tiles of heads [h0, h1): one contiguous run of the slot
        const int h0 = unit * a.hpb, h1 = min(a.H, h0 + a.hpb), nv = (h1 - h0) * a.tile_vecs;
        const int64_t off = (int64_t)h0 * a.tile_vecs * 16;
        const uint4 *from = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.ssm_pool) +
                                                            (int64_t)src * a.ssm_stride + off);
        uint4 *to = reinterpret_cast<uint4 *>(static_cast<char *>(a.ssm_pool) + (int64_t)s * a.ssm_stride + off);
        // every load of a batch is issued before its stores (source and destination may alias as far
        // as the compiler knows, so a plain copy loop would keep one load in flight per thread)
        constexpr int kBatch = 4;
        for (int v0 = tid; v0 < nv; v0 += blockDim.x * kBatch) {
            uint4 r[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int v = v0 + q * (int)blockDim.x;
                if (v < nv) r[q] = __ldcs(from + v);
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int v = v0 + q * (int)blockDim.x;
                if (v < nv) __stcs(to + v, r[q]);
            }
        }
        return;
    }
    if (!a.conv_pool) return;
    const int c0 = (unit - ssm_units) * CONV_CHANNELS;
    const int nc = min(CONV_CHANNELS, a.Cd - c0), Wc = a.Wc, shift = a.ntok - acc;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ActT *cs = reinterpret_cast<ActT *>(smem_raw);
    ActT *st = static_cast<ActT *>(a.conv_pool) + (int64_t)s * a.conv_stride + (int64_t)c0 * Wc;
    for (int e = tid; e < nc * Wc; e += blockDim.x) cs[e] = st[e];
    __syncthreads();
    for (int e = tid; e < nc * Wc; e += blockDim.x) {
        const int c = e / Wc, k = e - c * Wc;
        st[e] = k - shift >= 0 ? cs[c * Wc + k - shift] : from_f32<ActT>(0.0f);
    }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------

// Whether a cluster of the configuration's size can be resident, remembered per (device, kernel,
// cluster size, block, shared memory) so that small-batch calls do not repeat the occupancy query.
static bool cluster_fits(const void *kern, const cudaLaunchConfig_t &cfg) {
    struct Entry {
        int dev;
        const void *k;
        unsigned cx, bx;
        size_t smem;
        bool ok;
    };
    static Entry cache[32];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const unsigned cx = cfg.attrs[0].val.clusterDim.x, bx = cfg.blockDim.x;
    {
        std::lock_guard<std::mutex> g(mu);
        for (int e = 0; e < used; ++e)
            if (cache[e].dev == dev && cache[e].k == kern && cache[e].cx == cx && cache[e].bx == bx &&
                cache[e].smem == cfg.dynamicSmemBytes)
                return cache[e].ok;
    }
    int clusters = 0;
    const bool ok = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters >= 1;
    if (!ok) (void)cudaGetLastError();
    std::lock_guard<std::mutex> g(mu);
    if (used < 32) cache[used++] = {dev, kern, cx, bx, cfg.dynamicSmemBytes, ok};
    return ok;
}

// Raises a kernel's dynamic shared-memory limit on the current device to at least `smem` bytes;
// the attribute call is remembered per (device, kernel) so repeated launches skip it.
static bool smem_limit(const void *kern, size_t smem) {
    struct Entry {
        int dev;
        const void *k;
        size_t smem;
    };
    static Entry cache[64];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> g(mu);
    for (int e = 0; e < used; ++e)
        if (cache[e].dev == dev && cache[e].k == kern && cache[e].smem >= smem) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return false;
    for (int e = 0; e < used; ++e)
        if (cache[e].dev == dev && cache[e].k == kern) {
            cache[e].smem = smem;
            return true;
        }
    if (used < 64) cache[used++] = {dev, kern, smem};
    return true;
}

// SM count of the current device, read once per device (0 if it cannot be read).
static int device_sms() {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> count[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int n = count[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Persistent single-token launch, one CTA per SM, its ring depth chosen below.  Returns 1 when the
// layer's conv / xBC / z segments are not 16-byte aligned for bulk copies (the caller then uses
// the per-item kernel).
template <typename StateT, typename ActT, int P, int N>
static int launch_stream(const DecodeArgs &a, cudaStream_t stream) {
    const int LC = a.HG * P + 2 * N;
    const size_t es = sizeof(ActT), tile = (size_t)P * N * sizeof(StateT), dt_es = a.dt_bf16 ? 2 : 4;
    const size_t HP = (size_t)a.H * P, GN = (size_t)a.G * N, HGP = (size_t)a.HG * P;
    auto a16 = [](size_t v) { return v % 16 == 0; };
    auto p16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    const bool aligned = a.conv_pool && p16(a.conv_pool) && p16(a.xbc) && p16(a.conv_w) && (!a.z || p16(a.z)) &&
                         a16((size_t)a.conv_stride * es) && a16(HGP * a.Wc * es) && a16((size_t)N * a.Wc * es) &&
                         a16(HP * a.Wc * es) && a16(GN * a.Wc * es) && a16((size_t)a.Cd * es) && a16(HGP * es) &&
                         a16((size_t)N * es) && a16(HP * es) && a16(GN * es) && a16(HGP * a.W * 4) &&
                         a16((size_t)N * a.W * 4) && a16(HP * a.W * 4) && a16(GN * a.W * 4) && p16(a.dt) &&
                         p16(a.A) && (!a.dt_bias || p16(a.dt_bias)) && a16((size_t)a.HG * dt_es) &&
                         a16((size_t)a.H * dt_es) && a16((size_t)a.HG * 4);
    if (!aligned) return 1;
    // Stage ownership: tile t goes to stage t % ns and to head slot (t % HG) % NHS.  A stage must
    // always serve the same head slot (slot(t) == slot(t - ns)); otherwise a slot that runs ahead
    // could wait on a stage whose previous phase belongs to the other slot and is still pending,
    // and a parity wait cannot tell the two phases apart.  So ns is a multiple of NHS when NHS
    // divides HG, and a multiple of HG otherwise.
    //
    // Depth: at least two tiles in flight per head slot and 64 KB per CTA, or 128 KB when the
    // launch gives each CTA fewer than six items (its first copies are then a large share), no
    // more.  Measured on GB300 at the Nemotron shape, bf16 16 KB tiles, µs per launch at 4 / 6 / 8
    // stages: batch 40 (2.1 items a CTA) 38.6 / 37.2 / 36.2, batch 96 (5.1) 74.6 / 72.1 / 71.9,
    // batch 128 (6.7) 91.9 / 95.7 / 96.6, batch 256 (13.5) 178.2 / 179.6 / 182.1; fp32 32 KB tiles
    // at batch 256: 340 µs at 2 stages, 347 at 4.  One tile per slot starves the stream.
    const int sm_count = device_sms();
    if (sm_count <= 0) return MAMBA_ECUDA;
    const int W = a.batch * a.G;
    const int grid = W < sm_count ? W : sm_count;
    constexpr int NHS = kStreamConsumers / Tile<StateT, P, N>::TH;
    const int step = (a.HG % NHS == 0) ? NHS : a.HG;
    const size_t want = (W < 6 * grid ? 128 : 64) * (size_t)1024;
    int ns = step;
    while (ns < 2 * NHS || (size_t)ns * tile < want) ns += step;
    while (ns > step && (ns > 16 || StreamSmem(ns, tile, LC, a.HG, P, a.W, a.Wc, es, dt_es).total > 220 * 1024))
        ns -= step;
    if (ns < step || ns % step != 0) return 1;
    const size_t smem = StreamSmem(ns, tile, LC, a.HG, P, a.W, a.Wc, es, dt_es).total;
    if (smem > 227 * 1024) return 1;
    StreamArgs sa;
    sa.d = a;
    sa.ns = ns;
    auto kern = k_decode_stream<StateT, ActT, P, N>;
    if (!smem_limit(reinterpret_cast<const void *>(kern), smem)) return MAMBA_ECUDA;
    if (launch_pdl(kern, dim3(grid), dim3(kStreamThreads), smem, stream, sa) != cudaSuccess) return MAMBA_ECUDA;
    return launch_status();
}

template <typename StateT, typename ActT, int P, int N>
static int launch_decode_shape(const DecodeArgs &a0, int ntok, int P_, int N_, cudaStream_t stream) {
    using TL = Tile<StateT, P, N>;
    DecodeArgs a = a0;
    const bool conv = a.conv_pool != nullptr;
    const size_t tile = (size_t)P * N * sizeof(StateT), es = sizeof(ActT);
    // 16-byte vectorised conv and output phases: whole vectors of channels in every range, a
    // 4-tap conv whose window is W-1 or W-1+ntok columns, and 16-byte aligned rows
    constexpr int VA = Vec16<ActT>::n;
    const size_t HP = (size_t)a.H * P;
    bool vec = (a.HG * P) % VA == 0 && N % VA == 0 && aligned16(a.xbc) && ((size_t)a.Cd * es) % 16 == 0 &&
               aligned16(a.y) && (HP * es) % 16 == 0 && (!a.z || aligned16(a.z));
    if (conv)
        vec = vec && a.W == 4 && ntok >= 1 && ntok <= 4 && (a.Wc == a.W - 1 || a.Wc == a.W - 1 + ntok) &&
              aligned16(a.conv_pool) &&
              ((size_t)a.conv_stride * es) % 16 == 0 && aligned16(a.conv_w);
    a.vec = vec ? 1 : 0;
    // Small single-token batches: batch x groups CTAs would leave most SMs idle, so the heads of a
    // group are split over a cluster of up to 8 CTAs (a power of two dividing the heads per group,
    // at most enough for two CTAs per SM).
    //
    // Several tokens at batches that already fill the GPU: two CTAs per group (8 heads each at the
    // Nemotron shape) make the launch's last partial wave shorter.  Batch 128, 4 drafts on GB300:
    // 0.307 ms per draft + commit step against 0.312 unsplit and 0.344 with four CTAs per group.
    int ksplit = 1;
    const int sms = device_sms();
    if (vec && ntok > 1 && sms > 0 && (int64_t)a.batch * a.G >= 2 * sms && a.HG % 2 == 0 && ((a.HG / 2) * P) % VA == 0)
        ksplit = 2;
    if (vec && ntok == 1 && sms > 0 && (int64_t)a.batch * a.G < 2 * sms) {
        const int64_t want = (2 * (int64_t)sms + (int64_t)a.batch * a.G - 1) / ((int64_t)a.batch * a.G);
        while (ksplit * 2 <= 8 && ksplit * 2 <= want && a.HG % (ksplit * 2) == 0 && ((a.HG / (ksplit * 2)) * P) % VA == 0)
            ksplit *= 2;
    }
    for (;; ksplit = 1) {
    const int HGL = a.HG / ksplit, LC = HGL * P + 2 * N;
    int nhs = 256 / TL::TH;
    if (nhs < 1) nhs = 1;
    if (nhs > HGL) nhs = HGL;
    if (nhs > 8) nhs = 8;
    auto smem_for = [&](int k) { return DecodeSmem(k * nhs, tile, ntok, LC, HGL, P, a.Wc, es, conv, vec).total; };
    // Stages per head slot: one for several tokens (each tile stays in registers across the tokens
    // while the slot's next tile loads; batch 128, 4 drafts on GB300: 0.320 ms per draft + commit
    // step at one stage, 0.324 at two, 0.333 at three), two for the single-token launches here
    // (small batches: short launches, where the first copies are a large share).
    int sps = ntok > 1 ? 1 : 2;
    while (sps > 1 && smem_for(sps) > 227 * 1024) --sps;
    const size_t smem = smem_for(sps);
    if (smem > 227 * 1024) return MAMBA_EUNSUPPORTED;
    a.sps = sps;
    a.ksplit = ksplit;
    if constexpr (TL::TH <= kStreamConsumers && kStreamConsumers % TL::TH == 0) {
        if (ntok == 1 && a.scratch == nullptr && ksplit == 1) {
            const int rc = launch_stream<StateT, ActT, P, N>(a, stream);
            if (rc != 1) return rc;
        }
    }
    auto kern = ntok == 1 ? k_decode<StateT, ActT, P, N, 1> : k_decode<StateT, ActT, P, N, 0>;
    if (smem > 48 * 1024 && !smem_limit(reinterpret_cast<const void *>(kern), smem)) return MAMBA_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.G * ksplit, a.batch);
    cfg.blockDim = dim3(nhs * TL::TH);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ksplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (ksplit > 1 && !cluster_fits(reinterpret_cast<const void *>(kern), cfg)) continue;  // one CTA per (row, group)
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return MAMBA_ECUDA;
    return launch_status();
    }
}

// The compiled (head_dim, d_state) tiles.
#define MS_DECODE_SHAPES(X) X(16, 16) X(32, 64) X(64, 64) X(64, 128) X(128, 128)

static bool decode_shape_compiled(int P, int N) {
#define MS_SHAPE_CHECK(p, n) \
    if (P == p && N == n) return true;
    MS_DECODE_SHAPES(MS_SHAPE_CHECK)
#undef MS_SHAPE_CHECK
    return false;
}

template <typename StateT, typename ActT>
static int dispatch_decode_shape(const DecodeArgs &a, int ntok, int P, int N, cudaStream_t stream) {
#define MS_SHAPE_LAUNCH(p, n) \
    if (P == p && N == n) return launch_decode_shape<StateT, ActT, p, n>(a, ntok, P, N, stream);
    MS_DECODE_SHAPES(MS_SHAPE_LAUNCH)
#undef MS_SHAPE_LAUNCH
    return MAMBA_EUNSUPPORTED;
}

}  // namespace ms

using namespace ms;

extern "C" int mamba_decode_supported(const mamba_layer_desc *d) {
    int rc = check_desc(d);
    if (rc != MAMBA_OK) return rc;
    if (!decode_shape_compiled(d->head_dim, d->d_state)) return MAMBA_EUNSUPPORTED;
    if (d->conv_dtype != d->act_dtype) return MAMBA_EUNSUPPORTED;
    return MAMBA_OK;
}

extern "C" int mamba_state_update(const mamba_layer_desc *d, void *ssm_pool, int64_t ssm_slot_stride,
                                  int64_t num_slots, void *conv_pool, int64_t conv_slot_stride,
                                  const float *conv_w, const float *conv_b, const int32_t *slot_ids,
                                  const int32_t *scratch_slots, int32_t batch, int32_t ntok,
                                  const void *xbc, const void *dt, const float *A, const float *D,
                                  const float *dt_bias, int32_t dt_softplus, const void *z, void *y,
                                  int32_t *err_word, void *stream) {
    MS_TRACE("mamba_state_update");
    int rc = check_desc(d);
    if (rc != MAMBA_OK) return rc;
    if (batch < 0 || batch > 65535 || ntok < 1 || ntok > 8) return MAMBA_EINVAL;
    if (batch == 0) return MAMBA_OK;
    if (!ssm_pool || !slot_ids || !xbc || !dt || !A || !y) return MAMBA_EINVAL;
    const int H = d->nheads, P = d->head_dim, N = d->d_state, G = d->n_groups;
    const int Cd = mamba_conv_dim(d), Wc = d->conv_kernel - 1 + d->num_spec;
    if (num_slots <= 0 || ssm_slot_stride < (int64_t)H * P * N) return MAMBA_EINVAL;
    if (conv_pool && (!conv_w || conv_slot_stride < (int64_t)Cd * Wc)) return MAMBA_EINVAL;
    if ((rc = mamba_decode_supported(d)) != MAMBA_OK) return rc;
    const size_t sb = dtype_bytes(d->state_dtype);
    if (!aligned16(ssm_pool) || ((size_t)ssm_slot_stride * sb) % 16 != 0) return MAMBA_EALIGN;
    const size_t ab = dtype_bytes(d->act_dtype);
    if (((uintptr_t)xbc | (uintptr_t)y | (uintptr_t)z | (uintptr_t)conv_pool) % ab != 0) return MAMBA_EALIGN;

    DecodeArgs a;
    a.ssm_pool = ssm_pool; a.ssm_stride = ssm_slot_stride; a.num_slots = num_slots;
    a.conv_pool = conv_pool; a.conv_stride = conv_slot_stride; a.conv_w = conv_w; a.conv_b = conv_b;
    a.slot = slot_ids; a.scratch = scratch_slots; a.batch = batch; a.ntok = ntok;
    a.xbc = xbc; a.dt = dt; a.dt_bf16 = d->dt_dtype == MAMBA_BF16;
    a.A = A; a.D = D; a.dt_bias = dt_bias; a.dt_softplus = dt_softplus != 0;
    a.z = z; a.y = y; a.err = err_word;
    a.H = H; a.G = G; a.HG = H / G; a.W = d->conv_kernel; a.Wc = Wc; a.Cd = Cd;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool sbf = d->state_dtype == MAMBA_BF16, abf = d->act_dtype == MAMBA_BF16;
    if (sbf && abf) return dispatch_decode_shape<bf16, bf16>(a, ntok, P, N, st);
    if (sbf && !abf) return dispatch_decode_shape<bf16, float>(a, ntok, P, N, st);
    if (!sbf && abf) return dispatch_decode_shape<float, bf16>(a, ntok, P, N, st);
    return dispatch_decode_shape<float, float>(a, ntok, P, N, st);
}

extern "C" int mamba_conv_update(const mamba_layer_desc *d, void *conv_pool, int64_t conv_slot_stride,
                                 int64_t num_slots, const int32_t *slot_ids, int32_t batch, int32_t ntok,
                                 const void *xbc_in, const float *conv_w, const float *conv_b, void *xbc_out,
                                 int32_t *err_word, void *stream) {
    MS_TRACE("mamba_conv_update");
    int rc = check_desc(d);
    if (rc != MAMBA_OK) return rc;
    if (batch < 0 || batch > 65535 || ntok < 1 || ntok > 64) return MAMBA_EINVAL;
    if (batch == 0) return MAMBA_OK;
    if (!conv_pool || !slot_ids || !xbc_in || !conv_w || !xbc_out) return MAMBA_EINVAL;
    if (d->conv_dtype != d->act_dtype) return MAMBA_EUNSUPPORTED;
    const int Cd = mamba_conv_dim(d), Wc = d->conv_kernel - 1 + d->num_spec;
    if (num_slots <= 0 || conv_slot_stride < (int64_t)Cd * Wc) return MAMBA_EINVAL;
    const size_t ab = dtype_bytes(d->act_dtype);
    if (((uintptr_t)conv_pool | (uintptr_t)xbc_in | (uintptr_t)xbc_out) % ab != 0) return MAMBA_EALIGN;
    ConvArgs a;
    a.conv_pool = conv_pool; a.conv_stride = conv_slot_stride; a.num_slots = num_slots;
    a.slot = slot_ids; a.ntok = ntok; a.xbc_in = xbc_in; a.w = conv_w; a.b = conv_b;
    a.xbc_out = xbc_out; a.err = err_word; a.W = d->conv_kernel; a.Wc = Wc; a.Cd = Cd;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (d->act_dtype == MAMBA_BF16 ? launch_conv_step<bf16>(a, batch, ab, st) : launch_conv_step<float>(a, batch, ab, st))
        return launch_status();
    const size_t smem = sizeof(float) * 2 * (size_t)ntok * CONV_CHANNELS + ab * (size_t)CONV_CHANNELS * Wc;
    if (smem > 227 * 1024) return MAMBA_EUNSUPPORTED;
    const dim3 grid((Cd + CONV_CHANNELS - 1) / CONV_CHANNELS, batch), block(256);
    auto kern = d->act_dtype == MAMBA_BF16 ? k_conv_update<bf16> : k_conv_update<float>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MAMBA_ECUDA;
    if (launch_pdl(kern, grid, block, smem, st, a) != cudaSuccess) return MAMBA_ECUDA;
    return launch_status();
}

extern "C" int mamba1_conv_update(const mamba1_layer_desc *d, void *conv_pool, int64_t conv_slot_stride,
                                  int64_t num_slots, const int32_t *slot_ids, int32_t batch, int32_t ntok,
                                  const void *x_in, const float *conv_w, const float *conv_b, void *x_out,
                                  int32_t *err_word, void *stream) {
    MS_TRACE("mamba1_conv_update");
    if (!d || d->d_inner <= 0 || d->conv_kernel < 2 || d->conv_kernel > 8 || d->num_spec < 0 || d->num_spec > 32 ||
        !dtype_ok(d->act_dtype) || !dtype_ok(d->conv_dtype))
        return MAMBA_EINVAL;
    if (batch < 0 || batch > 65535 || ntok < 1 || ntok > 64) return MAMBA_EINVAL;
    if (batch == 0) return MAMBA_OK;
    if (!conv_pool || !slot_ids || !x_in || !conv_w || !x_out) return MAMBA_EINVAL;
    if (d->conv_dtype != d->act_dtype) return MAMBA_EUNSUPPORTED;
    const int Cd = d->d_inner, Wc = d->conv_kernel - 1 + d->num_spec;
    if (num_slots <= 0 || conv_slot_stride < (int64_t)Cd * Wc) return MAMBA_EINVAL;
    const size_t ab = dtype_bytes(d->act_dtype);
    if (((uintptr_t)conv_pool | (uintptr_t)x_in | (uintptr_t)x_out) % ab != 0) return MAMBA_EALIGN;
    ConvArgs a;
    a.conv_pool = conv_pool; a.conv_stride = conv_slot_stride; a.num_slots = num_slots;
    a.slot = slot_ids; a.ntok = ntok; a.xbc_in = x_in; a.w = conv_w; a.b = conv_b;
    a.xbc_out = x_out; a.err = err_word; a.W = d->conv_kernel; a.Wc = Wc; a.Cd = Cd;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (d->act_dtype == MAMBA_BF16 ? launch_conv_step<bf16>(a, batch, ab, st) : launch_conv_step<float>(a, batch, ab, st))
        return launch_status();
    const size_t smem = sizeof(float) * 2 * (size_t)ntok * CONV_CHANNELS + ab * (size_t)CONV_CHANNELS * Wc;
    if (smem > 227 * 1024) return MAMBA_EUNSUPPORTED;
    const dim3 grid((Cd + CONV_CHANNELS - 1) / CONV_CHANNELS, batch), block(256);
    auto kern = d->act_dtype == MAMBA_BF16 ? k_conv_update<bf16> : k_conv_update<float>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MAMBA_ECUDA;
    if (launch_pdl(kern, grid, block, smem, st, a) != cudaSuccess) return MAMBA_ECUDA;
    return launch_status();
}

extern "C" int mamba_spec_commit(const mamba_layer_desc *d, void *ssm_pool, int64_t ssm_slot_stride,
                                 int64_t num_slots, void *conv_pool, int64_t conv_slot_stride,
                                 const int32_t *slot_ids, const int32_t *scratch_slots,
                                 const int32_t *accept_len, int32_t batch, int32_t ntok, int32_t *err_word,
                                 void *stream) {
    MS_TRACE("mamba_spec_commit");
    int rc = check_desc(d);
    if (rc != MAMBA_OK) return rc;
    if (batch < 0 || batch > 65535 || ntok < 1) return MAMBA_EINVAL;
    if (batch == 0) return MAMBA_OK;
    if (!ssm_pool || !slot_ids || !scratch_slots || !accept_len) return MAMBA_EINVAL;
    const int H = d->nheads, P = d->head_dim, N = d->d_state;
    const int Cd = mamba_conv_dim(d), Wc = d->conv_kernel - 1 + d->num_spec;
    if (num_slots <= 0 || ssm_slot_stride < (int64_t)H * P * N) return MAMBA_EINVAL;
    if (conv_pool && (conv_slot_stride < (int64_t)Cd * Wc || ntok > d->num_spec)) return MAMBA_EINVAL;
    if (conv_pool && d->conv_dtype != d->act_dtype) return MAMBA_EUNSUPPORTED;
    const size_t sb = dtype_bytes(d->state_dtype);
    const int64_t tile_bytes = (int64_t)P * N * (int64_t)sb;
    if (!aligned16(ssm_pool) || ((size_t)ssm_slot_stride * sb) % 16 != 0 || tile_bytes % 16 != 0)
        return MAMBA_EALIGN;
    CommitArgs a;
    a.ssm_pool = ssm_pool; a.ssm_stride = ssm_slot_stride * (int64_t)sb; a.num_slots = num_slots;
    a.conv_pool = conv_pool; a.conv_stride = conv_slot_stride;
    a.slot = slot_ids; a.scratch = scratch_slots; a.accept = accept_len; a.ntok = ntok; a.err = err_word;
    a.H = H; a.tile_vecs = (int)(tile_bytes / 16); a.Cd = Cd; a.Wc = Wc;
    // four heads' tiles per block: the row's three dependent index loads are paid once per 64 KB
    // copied (batch 128, 4 drafts on GB300: draft + commit 0.3035 ms, against 0.3040 at two heads
    // and 0.3077 at one)
    a.hpb = 4;
    const int ssm_units = (H + a.hpb - 1) / a.hpb;
    const size_t ab = dtype_bytes(d->conv_dtype);
    const size_t smem = ab * (size_t)CONV_CHANNELS * Wc;
    const int conv_units = conv_pool ? (Cd + CONV_CHANNELS - 1) / CONV_CHANNELS : 0;
    const dim3 grid(ssm_units + conv_units, batch), block(256);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto kern = d->conv_dtype == MAMBA_BF16 ? k_spec_commit<bf16> : k_spec_commit<float>;
    if (launch_pdl(kern, grid, block, smem, st, a) != cudaSuccess) return MAMBA_ECUDA;
    return launch_status();
}
