// mamba1.cu -- the batched single-token decode step of a Mamba1 (S6) layer over a slot pool.
//
// Operation (echobase "Mamba" notes, the Mamba block: Delta_t = Softplus(.), h_t = exp(Delta_t A)
// h_{t-1} + Delta_t B_t x_t, y_t = C_t h_t, y_hat = y (.) SiLU(z), with the classic D x_t skip;
// "Hybrid SSM / Mamba models and non-KV state": the Mamba1 recurrent state is (D, N)): every
// channel d has its own step Delta_d = softplus(dt_d + dt_bias_d) and its own row A[d, :], so
//     h[d, n] <- exp(Delta_d A[d, n]) h[d, n] + Delta_d B[n] x[d],
//     y[d] = sum_n C[n] h[d, n] + D[d] x[d],  y *= SiLU(z[d]).
//
// Design (GB300): HBM-bound like the Mamba2 step (one read and one write of the state per
// token), but the state of a channel is only N values (32 bytes at N = 16, bf16), so a thread owns
// one channel of a strided set of batch rows (the grid is one wave of blocks): its row of A is
// loaded once, and while one row's N state values are updated and C.h accumulated in registers,
// the next row's loads are in flight; a warp reads and writes 32 channels' state as one
// contiguous kilobyte.  The decay differs per element, so each element costs one exponential
// (exp2 of Delta A log2 e).  B and C of a row are read by every lane at once (a broadcast).
#include <algorithm>

#include "common.cuh"
#include "umma.cuh"

namespace ms {

namespace {

constexpr int kM1Threads = 256;  // channels per block
constexpr float kLog2e = 1.4426950408889634f;

struct M1Args {
    void *ssm;
    int64_t ssm_stride, num_slots;  // stride in elements
    const int32_t *slot;
    const void *x, *dt, *B, *C, *z;
    const float *A, *D, *dt_bias;
    void *y;
    int32_t *err;
    int Dn, batch, dt_bf16, dt_softplus;
};

// N consecutive state values <-> fp32, as 16-byte vectors.
template <typename StateT, int N>
__device__ __forceinline__ void load_row(const StateT *p, float (&h)[N]) {
    constexpr int V = Vec16<StateT>::n;
#pragma unroll
    for (int k = 0; k < N / V; ++k) {
        float f[V];
        unpack16(reinterpret_cast<const uint4 *>(p)[k], f);
#pragma unroll
        for (int e = 0; e < V; ++e) h[k * V + e] = f[e];
    }
}
template <typename StateT, int N>
__device__ __forceinline__ void store_row(StateT *p, const float (&h)[N]) {
    constexpr int V = Vec16<StateT>::n;
#pragma unroll
    for (int k = 0; k < N / V; ++k) {
        float f[V];
#pragma unroll
        for (int e = 0; e < V; ++e) f[e] = h[k * V + e];
        reinterpret_cast<uint4 *>(p)[k] = pack16(f);
    }
}

// 2^x by the PTX approximate base-2 exponential (about 2 ulp); the decay arguments Delta A log2 e
// are never positive, and very negative ones give 0, the limit.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Everything one row of one channel reads: its state, x, dt and z (slot < 0: nothing to do).
template <int N>
struct M1Row {
    float h[N];
    float x, dt, z;
    int32_t slot;
};

template <typename StateT, typename ActT, int N>
__device__ __forceinline__ void m1_load(const M1Args &a, int i, int d, M1Row<N> &r) {
    r.slot = -1;
    if (i >= a.batch) return;
    const int32_t s = a.slot[i];
    if (s == -1) return;  // padding row: nothing read or written
    if (s < -1 || s >= a.num_slots) {
        if (d == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
        return;
    }
    r.slot = s;
    const int64_t xi = (int64_t)i * a.Dn + d;
    load_row<StateT, N>(static_cast<const StateT *>(a.ssm) + s * a.ssm_stride + (int64_t)d * N, r.h);
    r.x = to_f32(static_cast<const ActT *>(a.x)[xi]);
    r.dt = load_scalar(a.dt, xi, a.dt_bf16);
    r.z = a.z ? to_f32(static_cast<const ActT *>(a.z)[xi]) : 0.0f;
}

// B and C of row i (act dtype) as fp32, with 16-byte loads (every lane reads the same row, a
// broadcast).
template <typename ActT, int N>
__device__ __forceinline__ void load_bc(const ActT *p, float (&f)[N]) {
    load_row<ActT, N>(p, f);
}

// Block (x, y): channels [256x, 256x + 256) of rows y, y + gridDim.y, ...  (the grid is one wave).
// A thread keeps its channel's row of A in registers and walks its rows, the next row's loads in
// flight while the current row is computed.
template <typename StateT, typename ActT, int N>
__global__ void __launch_bounds__(kM1Threads, N <= 16 ? 3 : 1) k_mamba1_update(const M1Args a) {
    pdl_wait();
    pdl_launch_dependents();
    const int d = blockIdx.x * kM1Threads + threadIdx.x;
    if (d >= a.Dn) return;
    float Ar[N];  // this channel's row of A, times log2(e)
#pragma unroll
    for (int k = 0; k < N / 4; ++k) {
        const float4 v = reinterpret_cast<const float4 *>(a.A + (int64_t)d * N)[k];
        Ar[4 * k] = v.x * kLog2e;
        Ar[4 * k + 1] = v.y * kLog2e;
        Ar[4 * k + 2] = v.z * kLog2e;
        Ar[4 * k + 3] = v.w * kLog2e;
    }
    const float Dd = a.D ? a.D[d] : 0.0f, bias = a.dt_bias ? a.dt_bias[d] : 0.0f;
    const int step = gridDim.y;
    M1Row<N> cur, nxt;
    m1_load<StateT, ActT, N>(a, blockIdx.y, d, cur);
    for (int i = blockIdx.y; i < a.batch; i += step) {
        m1_load<StateT, ActT, N>(a, i + step, d, nxt);
        if (cur.slot >= 0) {
            float bv[N], cv[N];
            load_bc<ActT, N>(static_cast<const ActT *>(a.B) + (int64_t)i * N, bv);
            load_bc<ActT, N>(static_cast<const ActT *>(a.C) + (int64_t)i * N, cv);
            const float sdt = cur.dt + bias;
            const float delta = a.dt_softplus ? softplus_f(sdt) : sdt;
            const float dx = delta * cur.x;
            float acc = 0.0f;
#pragma unroll
            for (int n = 0; n < N; ++n) {
                cur.h[n] = fmaf(ex2_approx(delta * Ar[n]), cur.h[n], dx * bv[n]);
                acc = fmaf(cv[n], cur.h[n], acc);
            }
            store_row<StateT, N>(static_cast<StateT *>(a.ssm) + cur.slot * a.ssm_stride + (int64_t)d * N, cur.h);
            float yv = acc + Dd * cur.x;
            if (a.z) yv *= silu_f(cur.z);
            static_cast<ActT *>(a.y)[(int64_t)i * a.Dn + d] = from_f32<ActT>(yv);
        }
        cur = nxt;
    }
}

// ---------------------------------------------------------------------------------------
// persistent bulk-copy stream (state rows of at most 64 bytes per channel)
// ---------------------------------------------------------------------------------------
//
// Work item = (batch row, block of kM1Threads channels).  A CTA owns one channel block (its
// channels' rows of A, D and dt_bias stay in registers) and walks the rows rb, rb + kpb, ...
// One producer thread bulk-copies each item's state rows (kM1Threads x N contiguous values in the
// slot), x, dt and z slices and the row's B and C into a ring of shared-memory stages, up to NS
// items ahead; 256 consumer threads (one channel each) update the state from the stage, write it
// back with evict-first 16-byte stores and write y.  Three CTAs share an SM.  Each stage has a
// full barrier (the copies' bytes) and an empty barrier (every consumer has used the stage).
// All waits are bounded.

constexpr int kM1StreamThreads = kM1Threads + 32;
constexpr uint32_t kM1Polls = umma::kWaitPolls;

__host__ __device__ inline uint32_t m1_al16(uint32_t v) { return (v + 15u) & ~15u; }

// Byte offsets inside one stage.
struct M1Stage {
    uint32_t x, dt, z, b, c, hdr, bytes;
    __host__ __device__ M1Stage(int N, uint32_t es_state, uint32_t es_act) {
        x = m1_al16(kM1Threads * N * es_state);
        dt = x + m1_al16(kM1Threads * es_act);
        z = dt + kM1Threads * 4;
        b = z + m1_al16(kM1Threads * es_act);
        c = b + m1_al16(N * es_act);
        hdr = c + m1_al16(N * es_act);
        bytes = (hdr + 16 + 127) & ~127u;
    }
};

struct M1StreamArgs {
    M1Args a;
    int ns, kpb, ncb;
};

template <typename ActT>
__device__ __forceinline__ float act_at(const unsigned char *p, int t) {
    return to_f32(reinterpret_cast<const ActT *>(p)[t]);
}

template <typename StateT, typename ActT, int N>
__global__ void __launch_bounds__(kM1StreamThreads, 3) k_mamba1_stream(const M1StreamArgs sa) {
    pdl_wait();
    pdl_launch_dependents();
    const M1Args &a = sa.a;
    const int NS = sa.ns, kpb = sa.kpb;
    const int cb = blockIdx.x % sa.ncb, rb = blockIdx.x / sa.ncb;
    const int tid = threadIdx.x;
    const int d0 = cb * kM1Threads, nch = min(kM1Threads, a.Dn - d0);
    const M1Stage L(N, sizeof(StateT), sizeof(ActT));
    extern __shared__ __align__(128) unsigned char m1_smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(m1_smem + (size_t)NS * L.bytes);
    uint64_t *empty = full + NS;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + NS);
    int *issued = const_cast<int *>(abort_flag) + 1;
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            umma::mbar_init(&full[s], 1);
            umma::mbar_init(&empty[s], kM1Threads);
        }
        umma::fence_mbar_init();
        *abort_flag = 0;
        *issued = 0;
    }
    __syncthreads();

    if (tid >= kM1Threads) {
        // ---------------- producer ----------------
        if (tid == kM1Threads) {
            const uint32_t es = sizeof(StateT), ea = sizeof(ActT), et = a.dt_bf16 ? 2u : 4u;
            const uint32_t hb = (uint32_t)nch * N * es, xb = (uint32_t)nch * ea, tb = (uint32_t)nch * et;
            const uint32_t bcb = (uint32_t)N * ea;
            int k = 0;
            for (int i = rb; i < a.batch; i += kpb, ++k) {
                const int st = k % NS;
                if (k >= NS) {
                    bool ok = false;
                    for (uint32_t it = 0; it < kM1Polls && !ok; ++it) {
                        ok = umma::mbar_try_wait(&empty[st], (uint32_t)(k / NS - 1) & 1u);
                        if (!ok && (it & 1023u) == 1023u && *abort_flag) break;
                    }
                    if (!ok) {
                        *abort_flag = 1;
                        break;
                    }
                }
                unsigned char *sp = m1_smem + (size_t)st * L.bytes;
                int32_t s = a.slot[i];
                if (s < -1 || s >= a.num_slots) {
                    if (cb == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
                    s = -1;
                }
                *reinterpret_cast<int32_t *>(sp + L.hdr) = s;
                if (s < 0) {
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(umma::smem_u32(&full[st])) : "memory");
                } else {
                    const int64_t xi = (int64_t)i * a.Dn + d0;
                    umma::mbar_arrive_expect_tx(&full[st], hb + xb + tb + (a.z ? xb : 0u) + 2 * bcb);
                    umma::bulk_g2s(sp, static_cast<const StateT *>(a.ssm) + s * a.ssm_stride + (int64_t)d0 * N, hb,
                                   &full[st]);
                    umma::bulk_g2s(sp + L.x, static_cast<const ActT *>(a.x) + xi, xb, &full[st]);
                    umma::bulk_g2s(sp + L.dt, static_cast<const unsigned char *>(a.dt) + xi * et, tb, &full[st]);
                    if (a.z) umma::bulk_g2s(sp + L.z, static_cast<const ActT *>(a.z) + xi, xb, &full[st]);
                    umma::bulk_g2s(sp + L.b, static_cast<const ActT *>(a.B) + (int64_t)i * N, bcb, &full[st]);
                    umma::bulk_g2s(sp + L.c, static_cast<const ActT *>(a.C) + (int64_t)i * N, bcb, &full[st]);
                }
                *issued = k + 1;
            }
        }
    } else {
        // ---------------- consumers (thread = channel d0 + tid) ----------------
        const int d = d0 + tid;
        const bool live = tid < nch;
        float Ar[N];
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            const float4 v = live ? reinterpret_cast<const float4 *>(a.A + (int64_t)d * N)[q] : make_float4(0, 0, 0, 0);
            Ar[4 * q] = v.x * kLog2e;
            Ar[4 * q + 1] = v.y * kLog2e;
            Ar[4 * q + 2] = v.z * kLog2e;
            Ar[4 * q + 3] = v.w * kLog2e;
        }
        const float Dd = (live && a.D) ? a.D[d] : 0.0f, bias = (live && a.dt_bias) ? a.dt_bias[d] : 0.0f;
        int k = 0;
        for (int i = rb; i < a.batch; i += kpb, ++k) {
            const int st = k % NS;
            bool ok = false;
            for (uint32_t it = 0; it < kM1Polls && !ok; ++it) {
                ok = umma::mbar_try_wait(&full[st], (uint32_t)(k / NS) & 1u);
                if (!ok && (it & 1023u) == 1023u && *abort_flag) break;
            }
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            const unsigned char *sp = m1_smem + (size_t)st * L.bytes;
            const int32_t s = *reinterpret_cast<const int32_t *>(sp + L.hdr);
            if (s >= 0 && live) {
                float h[N];
                load_row<StateT, N>(reinterpret_cast<const StateT *>(sp) + (size_t)tid * N, h);
                const float xv = act_at<ActT>(sp + L.x, tid);
                const float sdt = (a.dt_bf16 ? to_f32(reinterpret_cast<const bf16 *>(sp + L.dt)[tid])
                                             : reinterpret_cast<const float *>(sp + L.dt)[tid]) + bias;
                const float zv = a.z ? act_at<ActT>(sp + L.z, tid) : 0.0f;
                float bv[N], cv[N];
                load_row<ActT, N>(reinterpret_cast<const ActT *>(sp + L.b), bv);
                load_row<ActT, N>(reinterpret_cast<const ActT *>(sp + L.c), cv);
                const float delta = a.dt_softplus ? softplus_f(sdt) : sdt;
                const float dx = delta * xv;
                float acc = 0.0f;
#pragma unroll
                for (int n = 0; n < N; ++n) {
                    h[n] = fmaf(ex2_approx(delta * Ar[n]), h[n], dx * bv[n]);
                    acc = fmaf(cv[n], h[n], acc);
                }
                StateT *dst = static_cast<StateT *>(a.ssm) + s * a.ssm_stride + (int64_t)d * N;
                constexpr int V = Vec16<StateT>::n;
#pragma unroll
                for (int q = 0; q < N / V; ++q) {
                    float f[V];
#pragma unroll
                    for (int e = 0; e < V; ++e) f[e] = h[q * V + e];
                    __stcs(reinterpret_cast<uint4 *>(dst) + q, pack16(f));
                }
                float yv = acc + Dd * xv;
                if (a.z) yv *= silu_f(zv);
                static_cast<ActT *>(a.y)[(int64_t)i * a.Dn + d] = from_f32<ActT>(yv);
            }
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(umma::smem_u32(&empty[st])) : "memory");
        }
    }
    __syncthreads();
    if (tid == kM1Threads && *abort_flag) {
        // a wait gave up: report it and let the copies still in flight land (bounded)
        flag_error(a.err, MAMBA_ERR_TIMEOUT);
        const int n = *issued;
        for (int k = n > NS ? n - NS : 0; k < n; ++k) umma::mbar_wait(&full[k % NS], (uint32_t)(k / NS) & 1u, kM1Polls);
    }
}

int sm_count_m1() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

// The stream kernel when a channel's state row is at most 64 bytes and every slice it copies is
// 16-byte aligned; false when the strided kernel must run instead.
template <typename StateT, typename ActT, int N>
bool launch_m1_stream(const M1Args &a, int batch, cudaStream_t st) {
    constexpr size_t es = sizeof(StateT), ea = sizeof(ActT);
    if constexpr (N * es > 64) {
        return false;
    } else {
    const size_t et = a.dt_bf16 ? 2 : 4;
    auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(a.ssm) || !al(a.x) || !al(a.dt) || (a.z && !al(a.z)) || !al(a.B) || !al(a.C) ||
        ((size_t)a.Dn * ea) % 16 || ((size_t)a.Dn * et) % 16 || ((size_t)N * ea) % 16 || ((size_t)a.ssm_stride * es) % 16)
        return false;
    const M1Stage L(N, (uint32_t)es, (uint32_t)ea);
    const size_t tail = 16 * 8 * 2 + 16;  // barriers of up to 16 stages + flags
    // Three CTAs per SM with about 40 KB of stages each.  GB300, Mamba-2.8B-like shape, batch 256,
    // 64-layer conv + update step: 1.648 ms at 4 stages of 10.2 KB, 1.652 at 3, 1.661 at 6.  Two
    // CTAs per SM took 1.70 ms at their best depth (6 stages; 10 stages 1.79 ms).
    int ns = 2;
    while (ns < 16 && (size_t)(ns + 1) * L.bytes <= 42 * 1024) ++ns;
    while (ns > 2 && (size_t)ns * L.bytes + tail > 72 * 1024) --ns;
    const size_t smem = (size_t)ns * L.bytes + (size_t)ns * 16 + 16;
    const int sms = std::max(1, sm_count_m1());
    const int ncb = (a.Dn + kM1Threads - 1) / kM1Threads;
    const int kpb = std::min(batch, std::max(1, 3 * sms / ncb));
    auto kern = k_mamba1_stream<StateT, ActT, N>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return false;
    M1StreamArgs sa;
    sa.a = a; sa.ns = ns; sa.kpb = kpb; sa.ncb = ncb;
    return launch_pdl(kern, dim3(ncb * kpb), dim3(kM1StreamThreads), smem, st, sa) == cudaSuccess;
    }
}

template <typename StateT, typename ActT, int N>
void launch_m1n(const M1Args &a, int batch, cudaStream_t st) {
    if (launch_m1_stream<StateT, ActT, N>(a, batch, st)) return;
    // one wave: the blocks resident at once, split over the channel blocks; rows strided over the rest
    const int cb = (a.Dn + kM1Threads - 1) / kM1Threads;
    int occ = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_mamba1_update<StateT, ActT, N>, kM1Threads, 0);
    const int slots = std::max(1, sm_count_m1()) * std::max(1, occ);
    const int gy = std::min(batch, std::max(1, slots / cb));
    launch_pdl(k_mamba1_update<StateT, ActT, N>, dim3(cb, gy), dim3(kM1Threads), 0, st, a);
}

template <typename StateT, typename ActT>
int launch_m1(const M1Args &a, int N, int batch, cudaStream_t st) {
    switch (N) {
        case 8: launch_m1n<StateT, ActT, 8>(a, batch, st); break;
        case 16: launch_m1n<StateT, ActT, 16>(a, batch, st); break;
        case 32: launch_m1n<StateT, ActT, 32>(a, batch, st); break;
        case 64: launch_m1n<StateT, ActT, 64>(a, batch, st); break;
        default: return MAMBA_EUNSUPPORTED;
    }
    return launch_status();
}

}  // namespace

}  // namespace ms

using namespace ms;

extern "C" int mamba1_state_update(const mamba1_layer_desc *d, void *ssm_pool, int64_t ssm_slot_stride,
                                   int64_t num_slots, const int32_t *slot_ids, int32_t batch, const void *x,
                                   const void *dt, const float *A, const void *B, const void *C, const float *D,
                                   const float *dt_bias, int32_t dt_softplus, const void *z, void *y,
                                   int32_t *err_word, void *stream) {
    MS_TRACE("mamba1_state_update");
    if (!d || d->d_inner <= 0 || d->d_inner % 8 || !dtype_ok(d->state_dtype) || !dtype_ok(d->act_dtype) ||
        !dtype_ok(d->dt_dtype))
        return MAMBA_EINVAL;
    const int N = d->d_state;
    if (N != 8 && N != 16 && N != 32 && N != 64) return MAMBA_EUNSUPPORTED;
    if (batch < 0 || batch > 65535) return MAMBA_EINVAL;
    if (batch == 0) return MAMBA_OK;
    if (!ssm_pool || !slot_ids || !x || !dt || !A || !B || !C || !y || num_slots <= 0) return MAMBA_EINVAL;
    if (ssm_slot_stride < (int64_t)d->d_inner * N) return MAMBA_EINVAL;
    const size_t sb = dtype_bytes(d->state_dtype), ab = dtype_bytes(d->act_dtype), tb = dtype_bytes(d->dt_dtype);
    if (!aligned16(ssm_pool) || ((size_t)ssm_slot_stride * sb) % 16 || (uintptr_t)A % 16) return MAMBA_EALIGN;
    if (((uintptr_t)x | (uintptr_t)B | (uintptr_t)C | (uintptr_t)y | (uintptr_t)z) % ab || (uintptr_t)dt % tb)
        return MAMBA_EALIGN;
    M1Args a;
    a.ssm = ssm_pool; a.ssm_stride = ssm_slot_stride; a.num_slots = num_slots; a.slot = slot_ids;
    a.x = x; a.dt = dt; a.B = B; a.C = C; a.z = z; a.A = A; a.D = D; a.dt_bias = dt_bias; a.y = y; a.err = err_word;
    a.Dn = d->d_inner; a.batch = batch; a.dt_bf16 = d->dt_dtype == MAMBA_BF16; a.dt_softplus = dt_softplus;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool sbf = d->state_dtype == MAMBA_BF16, abf = d->act_dtype == MAMBA_BF16;
    if (sbf && abf) return launch_m1<bf16, bf16>(a, N, batch, st);
    if (sbf) return launch_m1<bf16, float>(a, N, batch, st);
    if (abf) return launch_m1<float, bf16>(a, N, batch, st);
    return launch_m1<float, float>(a, N, batch, st);
}
