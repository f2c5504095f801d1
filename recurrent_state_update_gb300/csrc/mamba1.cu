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

// Everything one row of one channel reads: its state, x, dt and z (slot < 0: nothing to do).
// 2^x by the PTX approximate base-2 exponential (about 2 ulp); the decay arguments Delta A log2 e
// are never positive, and very negative ones give 0, the limit.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

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
    if (s < 0) return;  // padding row: nothing read or written
    if (s >= a.num_slots) {
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

int sm_count_m1() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

template <typename StateT, typename ActT, int N>
void launch_m1n(const M1Args &a, int batch, cudaStream_t st) {
    // one wave: the blocks resident at once, split over the channel blocks; rows strided over the rest
    const int cb = (a.Dn + kM1Threads - 1) / kM1Threads;
    int occ = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_mamba1_update<StateT, ActT, N>, kM1Threads, 0);
    const int slots = std::max(1, sm_count_m1()) * std::max(1, occ);
    const int gy = std::min(batch, std::max(1, slots / cb));
    k_mamba1_update<StateT, ActT, N><<<dim3(cb, gy), kM1Threads, 0, st>>>(a);
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
