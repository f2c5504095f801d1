// chunk_scan.cu -- varlen chunked prefill of the Mamba2 state update in the SSD form.
//
// Operations ("Hybrid SSM / Mamba models and non-KV state": mamba_chunk_scan_combined, whose
// within-chunk term is a masked matrix product and whose chunks are joined by a short scan over
// chunk states; a later chunk continues from the stored state; align-mode checkpoints; echobase
// "Mamba" notes:
// y_i = sum_{j<=i} C_i (prod_{k=j+1..i} Abar_k) Bbar_j x_j, Y = (M (.) L) X):
//   per chunk of Q tokens and head h, with cum_t = sum_{k<=t} Delta_k A_h inside the chunk:
//     G     = C B^T                                       (per group, Q x Q)
//     Y     = (G (.) exp(cum_i - cum_j) (.) Delta_j (.) [j<=i]) X + exp(cum_i) C h_prev^T + D X
//     S     = sum_j exp(cum_end - cum_j) Delta_j x_j B_j^T  (the chunk's own state)
//     h     = exp(cum_end) h_prev + S                     (state passing across chunks)
//
// This file is the portable CUDA-core form: six launches that communicate through a
// caller-provided workspace (chunk table, Delta and cum, G per group, per-chunk states).  It is
// the fp32 path (fp32 activations, any fp32 state pool), so the cumulative sums are kept in
// fp64: with large steps |cum| grows to hundreds within a chunk, and a decay exponent formed as
// the difference of two fp32 sums of that size would carry an absolute error of ~1e-4.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "scan_tc.h"

namespace ms {

// ---------------------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------------------

struct ScanLayout {
    int nchunks_max;
    size_t off_meta, off_dl, off_cum, off_cb, off_states, total;
};

static inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static ScanLayout scan_layout(int T, int nseq, int Q, int H, int G, int P, int N) {
    ScanLayout L;
    // every sequence adds at most one partial chunk
    L.nchunks_max = (T + Q - 1) / Q + nseq;
    size_t off = 0;
    L.off_meta = off;
    off = round_up(off + sizeof(int32_t) * (size_t)(4 + 4 * L.nchunks_max + 2 * nseq), 256);
    L.off_dl = off;
    off = round_up(off + sizeof(float) * (size_t)L.nchunks_max * H * Q, 256);
    L.off_cum = off;
    off = round_up(off + sizeof(double) * (size_t)L.nchunks_max * H * Q, 256);
    L.off_cb = off;
    off = round_up(off + sizeof(float) * (size_t)L.nchunks_max * G * Q * Q, 256);
    L.off_states = off;
    off = round_up(off + sizeof(float) * (size_t)L.nchunks_max * H * P * N, 256);
    L.total = off;
    return L;
}

// Chunk table inside the meta block: [count, pad x3 | seq[], start[], len[], kidx[] | first[], nch[]]
struct ChunkTable {
    int32_t *count, *seq, *start, *len, *kidx, *seq_first, *seq_nch;
    __host__ __device__ ChunkTable(int32_t *base, int nchunks_max, int nseq) {
        count = base;
        seq = base + 4;
        start = seq + nchunks_max;
        len = start + nchunks_max;
        kidx = len + nchunks_max;
        seq_first = kidx + nchunks_max;
        seq_nch = seq_first + nseq;
    }
};

struct ScanArgs {
    void *ssm_pool;
    int64_t ssm_stride, num_slots;
    const int32_t *cu, *slot;
    const uint8_t *has_init;
    const int32_t *ckpt_slots;
    int max_ckpt, ckpt_interval;
    int nseq, T, Q, H, G, HG, P, N;
    const void *x, *dt, *B, *C, *z;
    int dt_bf16, dt_softplus;
    const float *A, *D, *dt_bias;
    void *y;
    int32_t *err;
    int nchunks_max;
    int32_t *meta;
    float *dl;
    double *cum;
    float *cb, *states;
};

// ---------------------------------------------------------------------------------------
// 1. chunk table (one thread: the table is tiny)
// ---------------------------------------------------------------------------------------

__global__ void k_chunk_meta(const ScanArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    ChunkTable tb(a.meta, a.nchunks_max, a.nseq);
    bool ok = a.cu[0] == 0 && a.cu[a.nseq] == a.T;
    for (int s = 0; s < a.nseq && ok; ++s) ok = a.cu[s + 1] >= a.cu[s];
    if (!ok) {
        flag_error(a.err, MAMBA_ERR_SEQLENS);
        *tb.count = 0;
        for (int s = 0; s < a.nseq; ++s) tb.seq_first[s] = tb.seq_nch[s] = 0;
        return;
    }
    int n = 0;
    for (int s = 0; s < a.nseq; ++s) {
        const int32_t sl = a.slot[s];
        tb.seq_first[s] = n;
        if (sl < -1 || sl >= a.num_slots) {  // bad slot: the sequence is skipped entirely
            flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
            tb.seq_nch[s] = 0;
            continue;
        }
        const int L = a.cu[s + 1] - a.cu[s];
        const int nch = (L + a.Q - 1) / a.Q;
        for (int k = 0; k < nch && n < a.nchunks_max; ++k, ++n) {
            tb.seq[n] = s;
            tb.start[n] = a.cu[s] + k * a.Q;
            tb.len[n] = min(a.Q, L - k * a.Q);
            tb.kidx[n] = k;
        }
        tb.seq_nch[s] = n - tb.seq_first[s];
    }
    *tb.count = n;
}

// ---------------------------------------------------------------------------------------
// 2. Delta and the within-chunk cumulative sum of Delta*A, per (chunk, head)
// ---------------------------------------------------------------------------------------

__global__ void __launch_bounds__(1024) k_chunk_prep(const ScanArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    ChunkTable tb(a.meta, a.nchunks_max, a.nseq);
    const int c = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
    if (c >= *tb.count) return;
    extern __shared__ double sc[];
    const int len = tb.len[c];
    float delta = 0.0f;
    if (t < len) {
        const float s = load_scalar(a.dt, (int64_t)(tb.start[c] + t) * a.H + h, a.dt_bf16) +
                        (a.dt_bias ? a.dt_bias[h] : 0.0f);
        delta = a.dt_softplus ? softplus_f(s) : s;
    }
    sc[t] = t < len ? (double)delta * (double)a.A[h] : 0.0;
    __syncthreads();
    for (int off = 1; off < blockDim.x; off <<= 1) {  // inclusive scan
        const double v = t >= off ? sc[t - off] : 0.0;
        __syncthreads();
        sc[t] += v;
        __syncthreads();
    }
    const int64_t o = ((int64_t)c * a.H + h) * a.Q + t;
    a.dl[o] = delta;
    a.cum[o] = sc[t];
}

// ---------------------------------------------------------------------------------------
// 3. G = C B^T per (chunk, group): causal 64 x 64 tiles, 4 x 4 outputs per thread
// ---------------------------------------------------------------------------------------

template <typename ActT>
__global__ void __launch_bounds__(256) k_chunk_cb(const ScanArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    ChunkTable tb(a.meta, a.nchunks_max, a.nseq);
    const int c = blockIdx.x, g = blockIdx.y;
    const int ti = blockIdx.z / 4, tj = blockIdx.z % 4;  // 64-row tiles of a chunk of up to 256
    if (c >= *tb.count || tj > ti) return;
    const int len = tb.len[c], i0 = ti * 64, j0 = tj * 64;
    if (i0 >= len) return;
    __shared__ float Cs[64][33], Bs[64][33];
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    float acc[4][4] = {};
    const ActT *Cg = static_cast<const ActT *>(a.C);
    const ActT *Bg = static_cast<const ActT *>(a.B);
    for (int n0 = 0; n0 < a.N; n0 += 32) {
        for (int e = tid; e < 64 * 32; e += 256) {
            const int r = e / 32, k = e % 32;
            const int ti_ = i0 + r, tj_ = j0 + r;
            Cs[r][k] = ti_ < len ? to_f32(Cg[((int64_t)(tb.start[c] + ti_) * a.G + g) * a.N + n0 + k]) : 0.0f;
            Bs[r][k] = tj_ < len ? to_f32(Bg[((int64_t)(tb.start[c] + tj_) * a.G + g) * a.N + n0 + k]) : 0.0f;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < 32; ++k) {
            float cv[4], bv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                cv[u] = Cs[ty * 4 + u][k];
                bv[u] = Bs[tx * 4 + u][k];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(cv[u], bv[v], acc[u][v]);
        }
        __syncthreads();
    }
    float *out = a.cb + ((int64_t)c * a.G + g) * a.Q * a.Q;
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) out[(int64_t)(i0 + ty * 4 + u) * a.Q + j0 + tx * 4 + v] = acc[u][v];
}

// ---------------------------------------------------------------------------------------
// 4. the chunk's own state S = sum_j exp(cum_end - cum_j) Delta_j x_j B_j^T, per (chunk, head)
// ---------------------------------------------------------------------------------------

template <typename ActT>
__global__ void __launch_bounds__(256) k_chunk_state(const ScanArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    ChunkTable tb(a.meta, a.nchunks_max, a.nseq);
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= *tb.count) return;
    const int len = tb.len[c], g = h / a.HG, P = a.P, N = a.N;
    const double *cum = a.cum + ((int64_t)c * a.H + h) * a.Q;
    const float *dl = a.dl + ((int64_t)c * a.H + h) * a.Q;
    const double cum_end = cum[len - 1];
    extern __shared__ float sm[];
    float *Xs = sm;            // [32][P]  weighted x
    float *Bs = sm + 32 * P;   // [32][N]
    const ActT *xg = static_cast<const ActT *>(a.x);
    const ActT *Bg = static_cast<const ActT *>(a.B);
    const int tid = threadIdx.x;
    // thread owns column n = tid % N and rows p = tid / N + k * (256 / N), k < P / (256 / N)
    const int n = tid % N, p0 = tid / N, pstep = 256 / N, per = P / pstep;
    float acc[64];
#pragma unroll
    for (int k = 0; k < 64; ++k) acc[k] = 0.0f;
    for (int j0 = 0; j0 < len; j0 += 32) {
        for (int e = tid; e < 32 * P; e += 256) {
            const int r = e / P, p = e % P, j = j0 + r;
            float v = 0.0f;
            if (j < len)
                v = expf((float)(cum_end - cum[j])) * dl[j] *
                    to_f32(xg[((int64_t)(tb.start[c] + j) * a.H + h) * P + p]);
            Xs[e] = v;
        }
        for (int e = tid; e < 32 * N; e += 256) {
            const int r = e / N, nn = e % N, j = j0 + r;
            Bs[e] = j < len ? to_f32(Bg[((int64_t)(tb.start[c] + j) * a.G + g) * N + nn]) : 0.0f;
        }
        __syncthreads();
        for (int r = 0; r < 32; ++r) {
            const float bv = Bs[r * N + n];
            const float *xr = Xs + r * P + p0;
#pragma unroll
            for (int k = 0; k < 64; ++k)
                if (k < per) acc[k] = fmaf(xr[k * pstep], bv, acc[k]);
        }
        __syncthreads();
    }
    float *S = a.states + ((int64_t)c * a.H + h) * P * N;
#pragma unroll
    for (int k = 0; k < 64; ++k)
        if (k < per) S[(int64_t)(p0 + k * pstep) * N + n] = acc[k];
}

// ---------------------------------------------------------------------------------------
// 5. state passing over each sequence's chunks, per (sequence, head, element block).
//    states[c] is replaced by the state before chunk c; finals and checkpoints go to the pool.
// ---------------------------------------------------------------------------------------

template <typename StateT>
__global__ void __launch_bounds__(256) k_state_pass(const ScanArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    ChunkTable tb(a.meta, a.nchunks_max, a.nseq);
    const int s = blockIdx.x, h = blockIdx.y;
    const int64_t PN = (int64_t)a.P * a.N;
    const int64_t e = (int64_t)blockIdx.z * blockDim.x + threadIdx.x;
    if (e >= PN) return;
    const int32_t sl = a.slot[s];
    const int nch = tb.seq_nch[s], first = tb.seq_first[s];
    if (nch == 0) return;  // empty or skipped sequence
    StateT *pool = static_cast<StateT *>(a.ssm_pool);
    float hv = 0.0f;
    if (sl >= 0 && a.has_init && a.has_init[s]) hv = to_f32(pool[(int64_t)sl * a.ssm_stride + h * PN + e]);
    for (int k = 0; k < nch; ++k) {
        const int c = first + k;
        const int len = tb.len[c];
        float *S = a.states + ((int64_t)c * a.H + h) * PN + e;
        const float Sv = *S;
        *S = hv;  // state before chunk c
        const float decay = expf((float)a.cum[((int64_t)c * a.H + h) * a.Q + len - 1]);
        hv = fmaf(decay, hv, Sv);
        if (a.ckpt_slots && a.ckpt_interval > 0) {
            const int done = tb.kidx[c] * a.Q + len;
            if (done % a.ckpt_interval == 0) {
                const int m = done / a.ckpt_interval;
                if (m >= 1 && m <= a.max_ckpt) {
                    const int32_t cs = a.ckpt_slots[(int64_t)s * a.max_ckpt + m - 1];
                    if (cs >= a.num_slots || cs < -1) {
                        if (e == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
                    } else if (cs >= 0) {
                        pool[(int64_t)cs * a.ssm_stride + h * PN + e] = from_f32<StateT>(hv);
                    }
                }
            }
        }
    }
    if (sl >= 0) pool[(int64_t)sl * a.ssm_stride + h * PN + e] = from_f32<StateT>(hv);
}

// ---------------------------------------------------------------------------------------
// 6. outputs, per (chunk, head, 64-row tile): diagonal block + off-diagonal + D x, gate
// ---------------------------------------------------------------------------------------

template <typename ActT>
__global__ void __launch_bounds__(256) k_chunk_out(const ScanArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    ChunkTable tb(a.meta, a.nchunks_max, a.nseq);
    const int c = blockIdx.x, h = blockIdx.y, ti = blockIdx.z;
    if (c >= *tb.count) return;
    const int len = tb.len[c], i0 = ti * 64;
    if (i0 >= len) return;
    const int g = h / a.HG, P = a.P, N = a.N, Q = a.Q;
    const double *cum = a.cum + ((int64_t)c * a.H + h) * Q;
    const float *dl = a.dl + ((int64_t)c * a.H + h) * Q;
    const float *G = a.cb + ((int64_t)c * a.G + g) * Q * Q;
    const ActT *xg = static_cast<const ActT *>(a.x);
    const ActT *Cg = static_cast<const ActT *>(a.C);
    __shared__ float Ms[64][33];   // masked, decayed G tile (rows i, cols j)
    __shared__ float Xs[32][65];   // x_j tile (rows j, cols p), P <= 64
    __shared__ float Cs[64][33];   // C_i tile over 32 state columns
    __shared__ float Hs[64][33];   // h_prev tile [p][n]
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;  // 4 rows x 4 p per thread
    float acc[4][4] = {};
    const int start = tb.start[c];
    // diagonal block: j over [0, min(i0 + 64, len))
    const int jend = min(i0 + 64, len);
    for (int j0 = 0; j0 < jend; j0 += 32) {
        for (int e = tid; e < 64 * 32; e += 256) {
            const int r = e / 32, k = e % 32, i = i0 + r, j = j0 + k;
            float v = 0.0f;
            if (i < len && j < len && j <= i) v = G[(int64_t)i * Q + j] * expf((float)(cum[i] - cum[j])) * dl[j];
            Ms[r][k] = v;
        }
        for (int e = tid; e < 32 * 64; e += 256) {
            const int r = e / 64, p = e % 64, j = j0 + r;
            Xs[r][p] = (j < len && p < P) ? to_f32(xg[((int64_t)(start + j) * a.H + h) * P + p]) : 0.0f;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < 32; ++k) {
            float mv[4], xv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                mv[u] = Ms[ty * 4 + u][k];
                xv[u] = Xs[k][tx * 4 + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(mv[u], xv[v], acc[u][v]);
        }
        __syncthreads();
    }
    // off-diagonal: exp(cum_i) * C_i . h_prev[p, :]
    const float *hp = a.states + ((int64_t)c * a.H + h) * P * N;
    float off[4][4] = {};
    for (int n0 = 0; n0 < N; n0 += 32) {
        for (int e = tid; e < 64 * 32; e += 256) {
            const int r = e / 32, k = e % 32, i = i0 + r;
            Cs[r][k] = i < len ? to_f32(Cg[((int64_t)(start + i) * a.G + g) * N + n0 + k]) : 0.0f;
            Hs[r][k] = r < P ? hp[(int64_t)r * N + n0 + k] : 0.0f;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < 32; ++k) {
            float cv[4], hv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                cv[u] = Cs[ty * 4 + u][k];
                hv[u] = Hs[tx * 4 + u][k];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) off[u][v] = fmaf(cv[u], hv[v], off[u][v]);
        }
        __syncthreads();
    }
    const ActT *zg = static_cast<const ActT *>(a.z);
    ActT *yg = static_cast<ActT *>(a.y);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = i0 + ty * 4 + u;
        if (i >= len) continue;
        const float dec = expf((float)cum[i]);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int p = tx * 4 + v;
            if (p >= P) continue;
            const int64_t o = ((int64_t)(start + i) * a.H + h) * P + p;
            const float xv = to_f32(xg[o]);
            float yv = acc[u][v] + dec * off[u][v] + (a.D ? a.D[h] * xv : 0.0f);
            if (zg) yv *= silu_f(to_f32(zg[o]));
            yg[o] = from_f32<ActT>(yv);
        }
    }
}

template <typename ActT, typename StateT>
static int launch_scan(const ScanArgs &a, cudaStream_t st) {
    const size_t smem_state = sizeof(float) * 32 * (size_t)(a.P + a.N);
    const int64_t PN = (int64_t)a.P * a.N;
    if (launch_pdl(k_chunk_meta, dim3(1), dim3(32), 0, st, a) != cudaSuccess ||
        launch_pdl(k_chunk_prep, dim3(a.nchunks_max, a.H), dim3(a.Q), sizeof(double) * a.Q, st, a) != cudaSuccess ||
        launch_pdl(k_chunk_cb<ActT>, dim3(a.nchunks_max, a.G, 16), dim3(256), 0, st, a) != cudaSuccess ||
        launch_pdl(k_chunk_state<ActT>, dim3(a.nchunks_max, a.H), dim3(256), smem_state, st, a) != cudaSuccess ||
        launch_pdl(k_state_pass<StateT>, dim3(a.nseq, a.H, (unsigned)((PN + 255) / 256)), dim3(256), 0, st, a) !=
            cudaSuccess ||
        launch_pdl(k_chunk_out<ActT>, dim3(a.nchunks_max, a.H, (a.Q + 63) / 64), dim3(256), 0, st, a) != cudaSuccess)
        return MAMBA_ECUDA;
    return launch_status();
}

}  // namespace ms

using namespace ms;

static int scan_shape_ok(const mamba_layer_desc *d, int chunk) {
    // the portable kernels assume: chunk 256 (64-row tiles, one thread per token in the scan),
    // head_dim <= 64, d_state a power of two in 32..256 with (256 / d_state) | head_dim
    if (chunk != 256) return MAMBA_EUNSUPPORTED;
    if (d->head_dim > 64 || d->d_state % 32 || d->d_state > 256 || 256 % d->d_state ||
        d->head_dim % (256 / d->d_state))
        return MAMBA_EUNSUPPORTED;
    return MAMBA_OK;
}

// The tensor-core path (bf16 activations and state, head_dim 64, d_state 128): returns a status, or 1 when
// the layer is not eligible and the portable path must run.
static int try_scan_tc(const mamba_layer_desc *d, void *ssm_pool, int64_t ssm_slot_stride, int64_t num_slots,
                       const int32_t *cu_seqlens, int32_t nseq, int32_t total_tokens, const int32_t *slot_ids,
                       const uint8_t *has_initial_state, const int32_t *ckpt_slots, int32_t max_ckpt,
                       int32_t ckpt_interval, int32_t chunk, const void *x, const void *dt, const float *A,
                       const void *B, const void *C, const float *D, const float *dt_bias, int32_t dt_softplus,
                       const void *z, void *y, void *workspace, size_t workspace_bytes, int32_t *err_word,
                       cudaStream_t st) {
    if (!scan_tc_eligible(d, chunk)) return 1;
    if (workspace_bytes < scan_tc_workspace_bytes(nseq)) return MAMBA_ENOSPACE;
    if (!aligned16(workspace) || !aligned16(ssm_pool) || !aligned16(x) || !aligned16(B) || !aligned16(C) ||
        !aligned16(y) || (z && !aligned16(z)))
        return MAMBA_EALIGN;
    ScanTcParams p;
    p.ssm_pool = ssm_pool; p.ssm_stride = ssm_slot_stride; p.num_slots = num_slots;
    p.cu = cu_seqlens; p.slot = slot_ids; p.has_init = has_initial_state;
    p.ckpt_slots = ckpt_slots; p.max_ckpt = ckpt_slots ? max_ckpt : 0; p.ckpt_interval = ckpt_interval;
    p.nseq = nseq; p.T = total_tokens; p.H = d->nheads; p.G = d->n_groups; p.HG = d->nheads / d->n_groups;
    p.x = x; p.dt = dt; p.B = B; p.C = C; p.z = z; p.dt_bf16 = d->dt_dtype == MAMBA_BF16;
    p.dt_softplus = dt_softplus != 0; p.A = A; p.D = D; p.dt_bias = dt_bias; p.y = y; p.err = err_word;
    p.meta = static_cast<int32_t *>(workspace);
    return scan_tc_launch(p, d->state_dtype == MAMBA_BF16, st);
}

extern "C" size_t mamba_chunk_scan_workspace_bytes(const mamba_layer_desc *d, int32_t total_tokens, int32_t nseq,
                                                   int32_t chunk) {
    if (check_desc(d) != MAMBA_OK || total_tokens < 0 || nseq < 0 || chunk <= 0) return 0;
    if (scan_tc_eligible(d, chunk)) return scan_tc_workspace_bytes(nseq);
    return scan_layout(total_tokens, nseq, chunk, d->nheads, d->n_groups, d->head_dim, d->d_state).total;
}

extern "C" int mamba_chunk_scan(const mamba_layer_desc *d, void *ssm_pool, int64_t ssm_slot_stride,
                                int64_t num_slots, const int32_t *cu_seqlens, int32_t nseq, int32_t total_tokens,
                                const int32_t *slot_ids, const uint8_t *has_initial_state,
                                const int32_t *ckpt_slots, int32_t max_ckpt, int32_t ckpt_interval, int32_t chunk,
                                const void *x, const void *dt, const float *A, const void *B, const void *C,
                                const float *D, const float *dt_bias, int32_t dt_softplus, const void *z, void *y,
                                void *workspace, size_t workspace_bytes, int32_t *err_word, void *stream) {
    MS_TRACE("mamba_chunk_scan");
    int rc = check_desc(d);
    if (rc != MAMBA_OK) return rc;
    if (nseq < 0 || total_tokens < 0 || chunk <= 0) return MAMBA_EINVAL;
    if (nseq == 0) return MAMBA_OK;
    if (!ssm_pool || !cu_seqlens || !slot_ids || !A || !workspace) return MAMBA_EINVAL;
    if (total_tokens > 0 && (!x || !dt || !B || !C || !y)) return MAMBA_EINVAL;
    const int H = d->nheads, P = d->head_dim, N = d->d_state, G = d->n_groups;
    if (num_slots <= 0 || ssm_slot_stride < (int64_t)H * P * N) return MAMBA_EINVAL;
    if (ckpt_slots && (max_ckpt <= 0 || ckpt_interval <= 0 || ckpt_interval % chunk)) return MAMBA_EINVAL;
    rc = try_scan_tc(d, ssm_pool, ssm_slot_stride, num_slots, cu_seqlens, nseq, total_tokens, slot_ids,
                     has_initial_state, ckpt_slots, max_ckpt, ckpt_interval, chunk, x, dt, A, B, C, D, dt_bias,
                     dt_softplus, z, y, workspace, workspace_bytes, err_word, static_cast<cudaStream_t>(stream));
    if (rc != 1) return rc;
    if ((rc = scan_shape_ok(d, chunk)) != MAMBA_OK) return rc;
    const ScanLayout L = scan_layout(total_tokens, nseq, chunk, H, G, P, N);
    if (workspace_bytes < L.total) return MAMBA_ENOSPACE;
    if (!aligned16(workspace) || !aligned16(ssm_pool)) return MAMBA_EALIGN;
    ScanArgs a;
    a.ssm_pool = ssm_pool; a.ssm_stride = ssm_slot_stride; a.num_slots = num_slots;
    a.cu = cu_seqlens; a.slot = slot_ids; a.has_init = has_initial_state;
    a.ckpt_slots = ckpt_slots; a.max_ckpt = ckpt_slots ? max_ckpt : 0; a.ckpt_interval = ckpt_interval;
    a.nseq = nseq; a.T = total_tokens; a.Q = chunk; a.H = H; a.G = G; a.HG = H / G; a.P = P; a.N = N;
    a.x = x; a.dt = dt; a.B = B; a.C = C; a.z = z; a.dt_bf16 = d->dt_dtype == MAMBA_BF16;
    a.dt_softplus = dt_softplus != 0; a.A = A; a.D = D; a.dt_bias = dt_bias; a.y = y; a.err = err_word;
    a.nchunks_max = L.nchunks_max;
    char *ws = static_cast<char *>(workspace);
    a.meta = reinterpret_cast<int32_t *>(ws + L.off_meta);
    a.dl = reinterpret_cast<float *>(ws + L.off_dl);
    a.cum = reinterpret_cast<double *>(ws + L.off_cum);
    a.cb = reinterpret_cast<float *>(ws + L.off_cb);
    a.states = reinterpret_cast<float *>(ws + L.off_states);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool abf = d->act_dtype == MAMBA_BF16, sbf = d->state_dtype == MAMBA_BF16;
    if (abf && sbf) return launch_scan<bf16, bf16>(a, st);
    if (abf && !sbf) return launch_scan<bf16, float>(a, st);
    if (!abf && sbf) return launch_scan<float, bf16>(a, st);
    return launch_scan<float, float>(a, st);
}

// ---------------------------------------------------------------------------------------
// Allocation-free variant of mamba_chunk_scan.
//
// Some callers cannot hand this library a workspace: an engine that reserves all device
// memory for its own pool up front (a further cudaMalloc fails or forces a device-wide
// synchronisation that stalls every stream), or a latency-critical path that must not call
// cudaMalloc / cudaFree at all.  For them the scratch lives in one file-scope device array
// of fixed size.  Every GPU that loads this library holds that array until the process
// exits.  All calls share it: two calls that overlap on the GPU (different streams, or
// different host threads) race on it, so callers must order them.  Nothing in it needs to
// start at zero (each launch writes what it reads), so it is not cleared between calls.
// ---------------------------------------------------------------------------------------

#define MS_STATIC_SCAN_SCRATCH_BYTES (128ull << 20)

static __device__ __align__(256) unsigned char g_scan_scratch[MS_STATIC_SCAN_SCRATCH_BYTES];

// The driver's cuCtxGetCurrent, looked up once (no allocation).
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
static CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    });
    return fn;
}

// Device address of g_scan_scratch for the current device, looked up with that device current on
// the first call and again whenever the device's context has changed since (after a
// cudaDeviceReset the module, and with it the array, is loaded anew at another address).
static void *static_scratch_address(int *status) {
    constexpr int kMaxDevices = 64;
    static void *addr[kMaxDevices] = {};
    static CUcontext ctx_of[kMaxDevices] = {};
    static std::mutex mu;
    int dev = -1;
    *status = MAMBA_ECUDA;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (cudaSetDevice(dev) != cudaSuccess) return nullptr;  // same device: makes its primary context current
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || ctx_of[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scan_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev] = p;
        ctx_of[dev] = ctx;
    }
    *status = MAMBA_OK;
    return addr[dev];
}

extern "C" size_t mamba_chunk_scan_static_scratch_bytes(void) { return MS_STATIC_SCAN_SCRATCH_BYTES; }

extern "C" int mamba_chunk_scan_noalloc(const mamba_layer_desc *d, void *ssm_pool, int64_t ssm_slot_stride,
                                        int64_t num_slots, const int32_t *cu_seqlens, int32_t nseq,
                                        int32_t total_tokens, const int32_t *slot_ids,
                                        const uint8_t *has_initial_state, const int32_t *ckpt_slots,
                                        int32_t max_ckpt, int32_t ckpt_interval, int32_t chunk, const void *x,
                                        const void *dt, const float *A, const void *B, const void *C,
                                        const float *D, const float *dt_bias, int32_t dt_softplus, const void *z,
                                        void *y, int32_t *err_word, void *stream) {
    MS_TRACE("mamba_chunk_scan_noalloc");
    int rc = check_desc(d);
    if (rc != MAMBA_OK) return rc;
    if (nseq < 0 || total_tokens < 0 || chunk <= 0) return MAMBA_EINVAL;
    if (nseq == 0) return MAMBA_OK;
    if (!ssm_pool || !cu_seqlens || !slot_ids || !A) return MAMBA_EINVAL;
    if (total_tokens > 0 && (!x || !dt || !B || !C || !y)) return MAMBA_EINVAL;
    const int H = d->nheads, P = d->head_dim, N = d->d_state, G = d->n_groups;
    if (num_slots <= 0 || ssm_slot_stride < (int64_t)H * P * N) return MAMBA_EINVAL;
    if (ckpt_slots && (max_ckpt <= 0 || ckpt_interval <= 0 || ckpt_interval % chunk)) return MAMBA_EINVAL;
    if (scan_tc_eligible(d, chunk)) {
        if (scan_tc_workspace_bytes(nseq) > MS_STATIC_SCAN_SCRATCH_BYTES) return MAMBA_ENOSPACE;
        void *ws = static_scratch_address(&rc);
        if (rc != MAMBA_OK) return rc;
        return try_scan_tc(d, ssm_pool, ssm_slot_stride, num_slots, cu_seqlens, nseq, total_tokens, slot_ids,
                           has_initial_state, ckpt_slots, max_ckpt, ckpt_interval, chunk, x, dt, A, B, C, D,
                           dt_bias, dt_softplus, z, y, ws, MS_STATIC_SCAN_SCRATCH_BYTES, err_word,
                           static_cast<cudaStream_t>(stream));
    }
    if ((rc = scan_shape_ok(d, chunk)) != MAMBA_OK) return rc;
    const ScanLayout L = scan_layout(total_tokens, nseq, chunk, H, G, P, N);
    if (L.total > MS_STATIC_SCAN_SCRATCH_BYTES) return MAMBA_ENOSPACE;  // problem too large for the fixed scratch
    if (!aligned16(ssm_pool)) return MAMBA_EALIGN;
    void *workspace = static_scratch_address(&rc);
    if (rc != MAMBA_OK) return rc;
    ScanArgs a;
    a.ssm_pool = ssm_pool; a.ssm_stride = ssm_slot_stride; a.num_slots = num_slots;
    a.cu = cu_seqlens; a.slot = slot_ids; a.has_init = has_initial_state;
    a.ckpt_slots = ckpt_slots; a.max_ckpt = ckpt_slots ? max_ckpt : 0; a.ckpt_interval = ckpt_interval;
    a.nseq = nseq; a.T = total_tokens; a.Q = chunk; a.H = H; a.G = G; a.HG = H / G; a.P = P; a.N = N;
    a.x = x; a.dt = dt; a.B = B; a.C = C; a.z = z; a.dt_bf16 = d->dt_dtype == MAMBA_BF16;
    a.dt_softplus = dt_softplus != 0; a.A = A; a.D = D; a.dt_bias = dt_bias; a.y = y; a.err = err_word;
    a.nchunks_max = L.nchunks_max;
    char *ws = static_cast<char *>(workspace);
    a.meta = reinterpret_cast<int32_t *>(ws + L.off_meta);
    a.dl = reinterpret_cast<float *>(ws + L.off_dl);
    a.cum = reinterpret_cast<double *>(ws + L.off_cum);
    a.cb = reinterpret_cast<float *>(ws + L.off_cb);
    a.states = reinterpret_cast<float *>(ws + L.off_states);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool abf = d->act_dtype == MAMBA_BF16, sbf = d->state_dtype == MAMBA_BF16;
    if (abf && sbf) return launch_scan<bf16, bf16>(a, st);
    if (abf && !sbf) return launch_scan<bf16, float>(a, st);
    if (!abf && sbf) return launch_scan<float, bf16>(a, st);
    return launch_scan<float, float>(a, st);
}
