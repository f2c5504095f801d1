// conv_varlen.cu -- the causal depthwise conv1d + SiLU in front of the chunked prefill, over a
// varlen batch of prompts, with each sequence's conv state read at its start and written back.
//
// Operation (echobase "Mamba" notes, the Mamba block: x = SiLU(Conv1d(x')); "Hybrid SSM / Mamba
// models and non-KV state": the conv state is one of the two per-request state objects, a
// window of the most recent inputs, and a later prefill chunk continues from what the earlier
// one stored): for sequence s with tokens [cu[s], cu[s+1]) and input stream
//     e_s(q) = conv state column Wc + q (q < 0; zeros when the sequence does not start from its
//              state), e_s(q) = xBC row cu[s] + q (q >= 0),
//     out[cu[s] + q, c] = SiLU(b_c + sum_k w[c, k] e_s(q - (W-1) + k)),
// split into x | B | C, and afterwards the slot's conv state holds e_s(L - Wc .. L - 1).
//
// Design (GB300): the conv is a streaming pass (read xBC once, write x, B, C once), so it is
// bound by HBM bandwidth.  A persistent kernel walks tiles of 16 tokens x 2 KB of channels (32
// tokens for W > 4), each CTA keeping one channel block and its taps in registers.  Warp 0
// bulk-copies a tile's rows, plus the W-1 rows before them, into one of two shared-memory stages
// a tile ahead (cp.async.bulk on an mbarrier); the threads convolve the resident tile into a
// shared output tile, which warp 0 writes back with bulk stores (cp.async.bulk shared -> global,
// one 2 KB row per lane).  Every input a token needs is in shared memory or, for the first W-1
// tokens of a sequence, in its stored window; a thread owns one 16-byte channel vector and 8
// tokens, the W-1 previous inputs in registers.  Two CTAs share an SM, so one CTA's copies
// overlap the other's arithmetic.  The state write-back is a second, tiny kernel: the first
// tokens of a sequence read the old window while other CTAs may be processing its last tokens, so
// the old window may only be overwritten once the conv kernel has finished (stream order
// guarantees it).
#include "common.cuh"
#include "umma.cuh"

namespace ms {

namespace {

constexpr int kVarThreads = 128;   // threads of the state write-back kernel
constexpr int kBulkVecs = 128;     // 16-byte channel vectors per tile row (2 KB)
constexpr uint32_t kVarPolls = umma::kWaitPolls;

struct VarlenArgs {
    const int32_t *cu;
    int nseq, T;
    const int32_t *slot;
    const uint8_t *init;
    void *conv_pool;
    int64_t conv_stride, num_slots;
    const void *xbc;
    const float *w, *b;
    void *x_out, *B_out, *C_out;
    int32_t *err;
    int Cd, HP, GN, Wc;
    int ncb;  // channel blocks of kBulkVecs vectors
};

// True when cu_seqlens is non-decreasing from 0 to T (every thread of the block gets the answer).
__device__ __forceinline__ bool seqlens_ok(const VarlenArgs &a) {
    int bad = 0;
    if (threadIdx.x == 0) bad = a.cu[0] != 0 || a.cu[a.nseq] != a.T;
    for (int s = threadIdx.x; s < a.nseq; s += blockDim.x) bad |= a.cu[s + 1] < a.cu[s];
    return !__syncthreads_or(bad);
}

// The last sequence s with cu[s] <= t (for t < T that is the non-empty sequence holding t).
__device__ __forceinline__ int seq_of(const int32_t *cu, int nseq, int t) {
    int lo = 0, hi = nseq;  // invariant: cu[lo] <= t, answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Tile geometry of the conv kernel for a conv width W: tokens per tile, input stages (loads run
// S-1 tiles ahead), output stages, and threads (16 warps while the taps and the window fit in 128
// registers a thread, else 8).
// SiLU(v) = v / (1 + exp(-v)) with exp(-v) = 2^(-v log2 e): one PTX approximate base-2
// exponential and one approximate reciprocal (about 2 ulp and 1 ulp); for v -> -inf the reciprocal
// of +inf gives 0, the limit.
__device__ __forceinline__ float silu_approx(float v) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(v * -1.4426950408889634f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return v * r;
}

// Tile geometry of the conv kernel for a conv width W: tokens per tile, input stages (loads run
// S-1 tiles ahead), output stages, threads, and CTAs per SM.  For W <= 4 two CTAs of 16-token
// tiles share an SM (about 110 KB of shared memory and at most 128 registers a thread each), so
// one CTA's copies overlap the other's convolution; wider windows need more registers and take a
// whole SM with 32-token tiles.
template <int W>
struct BulkGeom {
    static constexpr int TOKENS = W <= 4 ? 16 : 32;
    static constexpr int S = 2;
    static constexpr int SO = 1;
    static constexpr int THREADS = 256;
    static constexpr int MINB = W <= 4 ? 2 : 1;
    static constexpr int TOK = TOKENS / (THREADS / kBulkVecs);  // tokens per thread
    static constexpr int ROWS = TOKENS + W - 1;  // the tile's tokens and the W-1 before them
    static constexpr uint32_t ROW = kBulkVecs * 16;   // bytes of a tile row
    static constexpr uint32_t STAGE = (uint32_t)ROWS * ROW;
    static constexpr uint32_t OUT = (uint32_t)TOKENS * ROW;
    static constexpr uint32_t OFF_OUT = S * STAGE;
    static constexpr uint32_t OFF_BAR = OFF_OUT + SO * OUT;
    static constexpr uint32_t OFF_LIVE = OFF_BAR + 8 * S;
    static constexpr size_t SMEM = OFF_LIVE + 4 * SO * TOKENS;
    static_assert(TOKENS % (THREADS / kBulkVecs) == 0 && TOKENS <= 32, "tile rows per thread / per lane");
    static_assert(SMEM <= 227 * 1024, "conv tile too large");
};

// Persistent conv kernel.  CTA j owns channel block j % ncb (its taps stay in registers) and walks
// the token blocks j / ncb, j / ncb + gridDim.x / ncb, ...  Warp 0 bulk-copies each tile's rows,
// plus the W-1 rows before them, into a ring of S shared-memory stages, S-1 tiles ahead; the
// threads convolve the resident tile into one of SO shared output tiles (thread = channel vector
// x a share of the tokens, the W-1 previous inputs in registers), and warp 0 bulk-stores its rows
// (one row per lane, split at the x | B | C boundaries) while the next tiles are convolved.
template <typename ActT, int W>
__global__ void __launch_bounds__(BulkGeom<W>::THREADS, BulkGeom<W>::MINB) k_conv_varlen(const VarlenArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    using Geo = BulkGeom<W>;
    constexpr int kTokPerThread = Geo::TOK, kBulkTokens = Geo::TOKENS, S = Geo::S, SO = Geo::SO;
    constexpr int V = Vec16<ActT>::n;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Geo::OFF_BAR);
    int *rowlive = reinterpret_cast<int *>(smem + Geo::OFF_LIVE);
    if (!seqlens_ok(a)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(a.err, MAMBA_ERR_SEQLENS);
        return;
    }
    const int tid = threadIdx.x, lane = tid & 31;
    const int nvec = a.Cd / V;
    const int cb = blockIdx.x % a.ncb, tb_step = gridDim.x / a.ncb;
    const int ntb = (a.T + kBulkTokens - 1) / kBulkTokens;
    const int v0 = cb * kBulkVecs, nv = min(kBulkVecs, nvec - v0);
    if (tid == 0) {
        for (int k = 0; k < S; ++k) umma::mbar_init(&full[k], 1);
        umma::fence_mbar_init();
    }
    __syncthreads();

    // warp 0: copy the rows of token block tb into stage st (rows before 0 or from T on are not
    // copied and never read)
    auto issue = [&](int tb, int st) {
        const int t0 = tb * kBulkTokens;
        const int r0 = max(t0 - (W - 1), 0), r1 = min(t0 + kBulkTokens, a.T);
        if (lane == 0) umma::mbar_arrive_expect_tx(&full[st], (uint32_t)(r1 - r0) * (uint32_t)nv * 16u);
        __syncwarp();
        const unsigned char *u = static_cast<const unsigned char *>(a.xbc) + (size_t)v0 * 16;
        unsigned char *base = smem + st * Geo::STAGE;
        for (int r = r0 + lane; r < r1; r += 32)
            umma::bulk_g2s(base + (size_t)(r - t0 + W - 1) * Geo::ROW, u + (size_t)r * a.Cd * sizeof(ActT),
                           (uint32_t)nv * 16u, &full[st]);
    };
    const int tb0 = blockIdx.x / a.ncb;
    if (tid < 32) {
        for (int k = 0; k < S - 1; ++k)
            if (tb0 + k * tb_step < ntb) issue(tb0 + k * tb_step, k);
    }

    // this thread's channel vector and taps (fixed for the CTA)
    const int cv = tid % kBulkVecs, part = tid / kBulkVecs;
    const bool has_vec = cv < nv;
    const int c0 = (v0 + cv) * V;
    float wt[V][W], bv[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
#pragma unroll
        for (int k = 0; k < W; ++k) wt[v][k] = has_vec ? a.w[(int64_t)(c0 + v) * W + k] : 0.0f;
        bv[v] = has_vec && a.b ? a.b[c0 + v] : 0.0f;
    }
    // the sequence holding this thread's current token and what its window seed needs, kept in
    // registers across tiles (a thread's tokens only increase): advanced only at a boundary
    int s = -1, s_begin = 0, s_end = 0;
    bool live = true;
    const ActT *sp = nullptr;
    auto enter = [&](int t) {
        if (s < 0) {
            s = seq_of(a.cu, a.nseq, t);
        } else {
            while (a.cu[s + 1] <= t) ++s;  // empty sequences are skipped
        }
        s_begin = a.cu[s];
        s_end = a.cu[s + 1];
        const int32_t sl = a.slot ? a.slot[s] : -1;
        live = sl >= -1 && sl < a.num_slots;
        const bool has = a.conv_pool && sl >= 0 && live && a.init && a.init[s];
        sp = has ? static_cast<const ActT *>(a.conv_pool) + sl * a.conv_stride + (int64_t)c0 * a.Wc : nullptr;
    };
    bool failed = false;
    int i = 0;
    for (int tb = tb0; tb < ntb; tb += tb_step, ++i) {
        const int st = i % S, so = i % SO;
        ActT *outs = reinterpret_cast<ActT *>(smem + Geo::OFF_OUT + so * Geo::OUT) + (size_t)cv * V;
        int *live_row = rowlive + so * kBulkTokens;
        if (tid < 32) {
            if (tb + (S - 1) * tb_step < ntb) issue(tb + (S - 1) * tb_step, (i + S - 1) % S);
            umma::bulk_wait_read<SO - 1>();  // the stores of tile i - SO have read this output stage
        }
        const int t0 = tb * kBulkTokens;
        const int ta = t0 + part * kTokPerThread, tz = min(ta + kTokPerThread, a.T);
        if (has_vec && ta < tz && (s < 0 || ta >= s_end)) enter(ta);  // overlaps the copy wait
        const bool ok = umma::mbar_wait(&full[st], (uint32_t)(i / S) & 1u, kVarPolls);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        if (has_vec && ta < tz) {
            const ActT *rows = reinterpret_cast<const ActT *>(smem + st * Geo::STAGE) + (size_t)cv * V;
            // row of token t in the stage: t - t0 + W - 1
            auto row = [&](int t) { return rows + (size_t)(t - t0 + W - 1) * (kBulkVecs * V); };
            float win[W - 1][V];  // win[W-2]: the newest input before the current token
            // window of token t of the current sequence: inputs t-1..t-(W-1) from the tile when they
            // belong to it, else from the sequence's stored window (zeros without one)
            auto seed = [&](int t) {
#pragma unroll
                for (int k = 1; k < W; ++k) {
                    const int rel = t - k - s_begin;
                    if (rel >= 0) {
                        unpack16(*reinterpret_cast<const uint4 *>(row(t - k)), win[W - 1 - k]);
                    } else {
#pragma unroll
                        for (int v = 0; v < V; ++v)
                            win[W - 1 - k][v] = sp ? to_f32(sp[(int64_t)v * a.Wc + a.Wc + rel]) : 0.0f;
                    }
                }
            };
            // one token: convolve the window and input x, store, shift x into the window
            auto step = [&](int t, const float (&x)[V]) {
                float o[V];
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    float acc = fmaf(wt[v][W - 1], x[v], bv[v]);
#pragma unroll
                    for (int k = 0; k < W - 1; ++k) acc = fmaf(wt[v][k], win[k][v], acc);
                    o[v] = silu_approx(acc);
                }
#pragma unroll
                for (int k = 0; k + 1 < W - 1; ++k)
#pragma unroll
                    for (int v = 0; v < V; ++v) win[k][v] = win[k + 1][v];
#pragma unroll
                for (int v = 0; v < V; ++v) win[W - 2][v] = x[v];
                *reinterpret_cast<uint4 *>(outs + (size_t)(t - t0) * (kBulkVecs * V)) = pack16(o);
            };
            seed(ta);
            if (tz - ta == kTokPerThread && s_end >= tz) {
                // common case: all of this thread's tokens in one sequence, fully unrolled so the
                // tokens' independent work interleaves
                if (cv == 0) {
#pragma unroll
                    for (int j = 0; j < kTokPerThread; ++j) live_row[ta - t0 + j] = live;
                }
#pragma unroll
                for (int j = 0; j < kTokPerThread; ++j) {
                    float x[V];
                    unpack16(*reinterpret_cast<const uint4 *>(row(ta + j)), x);
                    step(ta + j, x);
                }
            } else {
                for (int t = ta; t < tz; ++t) {
                    if (t >= s_end) {  // first token of a later sequence
                        enter(t);
                        seed(t);
                    }
                    float x[V];
                    unpack16(*reinterpret_cast<const uint4 *>(row(t)), x);
                    step(t, x);
                    if (cv == 0) live_row[t - t0] = live;
                }
            }
        }
        umma::fence_async_smem();
        __syncthreads();  // output tile complete; the input stage is free for the copy a tile ahead
        if (tid < 32) {
            // lane r stores token row t0 + r, split at the x | B | C boundaries
            const int t = t0 + lane;
            if (lane < kBulkTokens && t < a.T && live_row[lane]) {
                const int cs = v0 * V, ce = cs + nv * V;
                const unsigned char *src = smem + Geo::OFF_OUT + so * Geo::OUT + (size_t)lane * Geo::ROW;
                const int bounds[4] = {0, a.HP, a.HP + a.GN, a.Cd};
                void *const bases[3] = {a.x_out, a.B_out, a.C_out};
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    const int lo = max(cs, bounds[r]), hi = min(ce, bounds[r + 1]);
                    if (lo < hi) {
                        const int pitch = bounds[r + 1] - bounds[r];
                        ActT *dst = static_cast<ActT *>(bases[r]) + (int64_t)t * pitch + (lo - bounds[r]);
                        umma::bulk_s2g(dst, src + (size_t)(lo - cs) * sizeof(ActT), (uint32_t)((hi - lo) * sizeof(ActT)));
                    }
                }
            }
            umma::bulk_commit();
        }
    }
    if (tid < 32) umma::bulk_wait_all();
    if (failed && tid < 32) {
        // a copy did not land in time: report it and let the copies still in flight finish (bounded)
        if (lane == 0) {
            flag_error(a.err, MAMBA_ERR_TIMEOUT);
            for (int k = 0; k < S; ++k) {
                const int tb = tb0 + (i + k) * tb_step;
                if (tb < ntb) umma::mbar_wait(&full[(i + k) % S], (uint32_t)((i + k) / S) & 1u, kVarPolls);
            }
        }
    }
}

// Conv state write-back, one thread per (sequence, channel): column i becomes e_s(L - Wc + i).
// Column i reads column i + L of the old window (only when L < Wc), which is not yet written.
template <typename ActT>
__global__ void __launch_bounds__(kVarThreads) k_conv_varlen_state(const VarlenArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    if (!seqlens_ok(a)) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) flag_error(a.err, MAMBA_ERR_SEQLENS);
        return;
    }
    const int s = blockIdx.y, c = blockIdx.x * kVarThreads + threadIdx.x;
    const int32_t sl = a.slot[s];
    if (sl < -1 || sl >= a.num_slots) {
        if (c == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
        return;
    }
    if (sl < 0 || c >= a.Cd) return;
    const int begin = a.cu[s], L = a.cu[s + 1] - begin, Wc = a.Wc;
    const bool has = a.init && a.init[s];
    ActT *st = static_cast<ActT *>(a.conv_pool) + sl * a.conv_stride + (int64_t)c * Wc;
    const ActT *u = static_cast<const ActT *>(a.xbc);
    for (int i = 0; i < Wc; ++i) {
        const int q = L - Wc + i;
        ActT v;
        if (q >= 0) v = u[(int64_t)(begin + q) * a.Cd + c];
        else v = has ? st[i + L] : from_f32<ActT>(0.0f);
        st[i] = v;
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

template <typename ActT, int W>
int launch_varlen(const VarlenArgs &a, cudaStream_t st) {
    using Geo = BulkGeom<W>;
    auto kern = k_conv_varlen<ActT, W>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Geo::SMEM) != cudaSuccess)
        return MAMBA_ECUDA;
    const int sms = sm_count();
    int occ = 0;
    if (sms <= 0 || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Geo::THREADS, Geo::SMEM) != cudaSuccess ||
        occ <= 0)
        return MAMBA_ECUDA;
    // a whole number of CTAs per channel block, no more than there are token blocks
    const int ntb = (a.T + Geo::TOKENS - 1) / Geo::TOKENS;
    const int per_cb = max(1, min(sms * occ / a.ncb, ntb));
    if (launch_pdl(kern, dim3(per_cb * a.ncb), dim3(Geo::THREADS), Geo::SMEM, st, a) != cudaSuccess) return MAMBA_ECUDA;
    return launch_status();
}

template <typename ActT>
int launch_varlen_w(const VarlenArgs &a, int W, cudaStream_t st) {
    switch (W) {
        case 2: return launch_varlen<ActT, 2>(a, st);
        case 3: return launch_varlen<ActT, 3>(a, st);
        case 4: return launch_varlen<ActT, 4>(a, st);
        case 5: return launch_varlen<ActT, 5>(a, st);
        case 6: return launch_varlen<ActT, 6>(a, st);
        case 7: return launch_varlen<ActT, 7>(a, st);
        default: return launch_varlen<ActT, 8>(a, st);
    }
}

}  // namespace

}  // namespace ms

using namespace ms;

extern "C" int mamba_conv_varlen(const mamba_layer_desc *d, void *conv_pool, int64_t conv_slot_stride,
                                 int64_t num_slots, const int32_t *cu_seqlens, int32_t nseq, int32_t total_tokens,
                                 const int32_t *slot_ids, const uint8_t *has_initial_state, const void *xbc,
                                 const float *conv_w, const float *conv_b, void *x_out, void *B_out, void *C_out,
                                 int32_t *err_word, void *stream) {
    MS_TRACE("mamba_conv_varlen");
    int rc = check_desc(d);
    if (rc != MAMBA_OK) return rc;
    if (nseq < 0 || total_tokens < 0) return MAMBA_EINVAL;
    if (nseq == 0) return total_tokens == 0 ? MAMBA_OK : MAMBA_EINVAL;
    if (!cu_seqlens || !conv_w || (total_tokens > 0 && (!xbc || !x_out || !B_out || !C_out)))
        return MAMBA_EINVAL;
    if (conv_pool && !slot_ids) return MAMBA_EINVAL;
    if (d->conv_dtype != d->act_dtype) return MAMBA_EUNSUPPORTED;
    const int Cd = mamba_conv_dim(d), Wc = d->conv_kernel - 1 + d->num_spec;
    const int HP = d->nheads * d->head_dim, GN = d->n_groups * d->d_state;
    if (conv_pool && (num_slots <= 0 || conv_slot_stride < (int64_t)Cd * Wc)) return MAMBA_EINVAL;
    const size_t ab = dtype_bytes(d->act_dtype);
    const int V = (int)(16 / ab);
    if (HP % V || GN % V) return MAMBA_EUNSUPPORTED;
    if (!aligned16(xbc) || !aligned16(x_out) || !aligned16(B_out) || !aligned16(C_out) ||
        (conv_pool && (uintptr_t)conv_pool % ab))
        return MAMBA_EALIGN;
    VarlenArgs a;
    a.cu = cu_seqlens; a.nseq = nseq; a.T = total_tokens; a.slot = conv_pool ? slot_ids : nullptr;
    a.init = has_initial_state; a.conv_pool = conv_pool; a.conv_stride = conv_slot_stride;
    a.num_slots = conv_pool ? num_slots : 1; a.xbc = xbc; a.w = conv_w; a.b = conv_b;
    a.x_out = x_out; a.B_out = B_out; a.C_out = C_out; a.err = err_word;
    a.Cd = Cd; a.HP = HP; a.GN = GN; a.Wc = Wc;
    a.ncb = (Cd / V + kBulkVecs - 1) / kBulkVecs;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (total_tokens > 0) {
        rc = d->act_dtype == MAMBA_BF16 ? launch_varlen_w<bf16>(a, d->conv_kernel, st)
                                        : launch_varlen_w<float>(a, d->conv_kernel, st);
        if (rc != MAMBA_OK) return rc;
    }
    if (conv_pool) {
        const dim3 grid((Cd + kVarThreads - 1) / kVarThreads, nseq);
        const cudaError_t e = d->act_dtype == MAMBA_BF16
                                  ? launch_pdl(k_conv_varlen_state<bf16>, grid, dim3(kVarThreads), 0, st, a)
                                  : launch_pdl(k_conv_varlen_state<float>, grid, dim3(kVarThreads), 0, st, a);
        rc = e != cudaSuccess ? MAMBA_ECUDA : launch_status();
    }
    return rc;
}
