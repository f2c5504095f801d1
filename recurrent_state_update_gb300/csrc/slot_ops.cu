// slot_ops.cu -- whole-slot state operations of the prefix cache: a batched slot-to-slot copy
// (restore of a cached checkpoint into a fresh active slot, copy-on-write) and the int8
// checkpoint store (quantise a slot into a compact entry, dequantise an entry into a slot).
//
// Operations ("Hybrid SSM / Mamba models and non-KV state": on a prefix-cache hit the cached
// state is copied into a fresh slot rather than shared, because the recurrence updates its slot
// in place; the SGLang checkpoint store keeps cached temporal states in int8 with one symmetric
// scale per (head, k-channel), quantised once on store and dequantised once on a hit, and keeps
// the conv window at its native dtype).  The k-channel of the Mamba2 temporal state
// (H, head_dim, d_state) is the d_state index n, so a scale covers the head_dim values of one
// (head, n):  s = max_p |h[p, n]| / 127,  q = clamp(rint(h * (127 / max_p |h[p, n]|)), -127, 127),
// all in fp32 (the nearest code on the grid of step s).
//
// Design (GB300): all three are HBM streaming passes.  The copy moves 16-byte vectors, 16 KB
// per block, over the concatenation of a slot's SSM and conv bytes.  The store runs one warp
// per (row, head): the head's tile arrives in shared memory with one bulk async copy, and a
// thread per (8 adjacent d_state columns, half of the rows) finds the column maxima, combined
// with a shuffle; the load runs 128 threads per (row, head), one per (8 columns, share of the
// rows), each issuing all of its rows' code loads before converting any; 16-byte accesses,
// every row read or written as one contiguous run.
#include "common.cuh"
#include "umma.cuh"

namespace ms {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyBytes = kCopyThreads * 16 * 4;  // bytes one copy block moves
constexpr int kQThreads = 128;
constexpr int kStoreHeads = 1;           // heads quantised by one store block (more blocks in flight)
constexpr int kLoadRows = 8;             // rows per thread and pass of the load
constexpr uint32_t kQPolls = umma::kWaitPolls;  // bound on the wait for a staged tile

inline size_t align256(size_t b) { return (b + 255) / 256 * 256; }

struct EntryLayout {
    size_t q, scales, conv, total;  // section offsets and entry size in bytes
};

inline EntryLayout entry_layout(const mamba_layer_desc *d) {
    EntryLayout L;
    const size_t q = (size_t)d->nheads * d->head_dim * d->d_state;
    const size_t sc = (size_t)d->nheads * d->d_state * sizeof(float);
    const size_t cv = (size_t)mamba_conv_dim(d) * (d->conv_kernel - 1 + d->num_spec) * dtype_bytes(d->conv_dtype);
    L.q = 0;
    L.scales = align256(q);
    L.conv = L.scales + align256(sc);
    L.total = L.conv + align256(cv);
    return L;
}

struct CopyArgs {
    unsigned char *ssm;
    int64_t ssm_stride, num_slots;  // stride in bytes
    unsigned char *conv;
    int64_t conv_stride;  // bytes
    const int32_t *src, *dst;
    int64_t ssm_bytes, conv_bytes;
    int32_t *err;
};

// Block (b, i) copies bytes [b * kCopyBytes, ...) of slot src[i]'s SSM bytes followed by its conv
// bytes into slot dst[i].
__global__ void __launch_bounds__(kCopyThreads) k_slot_copy(const CopyArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    const int i = blockIdx.y;
    const int32_t s = a.src[i], d = a.dst[i];
    if (s < -1 || s >= a.num_slots || d < -1 || d >= a.num_slots) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
        return;
    }
    if (s < 0 || d < 0 || s == d) return;
    const int64_t base = (int64_t)blockIdx.x * kCopyBytes;
    const int64_t total = a.ssm_bytes + (a.conv ? a.conv_bytes : 0);
    uint4 v[4];
    int64_t off[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        off[k] = base + ((int64_t)k * kCopyThreads + threadIdx.x) * 16;
        if (off[k] < total) {
            const unsigned char *p = off[k] < a.ssm_bytes ? a.ssm + s * a.ssm_stride + off[k]
                                                          : a.conv + s * a.conv_stride + (off[k] - a.ssm_bytes);
            v[k] = __ldcs(reinterpret_cast<const uint4 *>(p));
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (off[k] < total) {
            unsigned char *p = off[k] < a.ssm_bytes ? a.ssm + d * a.ssm_stride + off[k]
                                                    : a.conv + d * a.conv_stride + (off[k] - a.ssm_bytes);
            *reinterpret_cast<uint4 *>(p) = v[k];
        }
    }
}

struct QArgs {
    unsigned char *ssm;  // pool base
    int64_t ssm_stride, num_slots;  // stride in bytes
    unsigned char *conv;
    int64_t conv_stride;  // bytes
    unsigned char *store;
    int64_t num_entries;
    EntryLayout lay;
    const int32_t *slots, *entries;
    int H, P, N;
    int64_t conv_bytes;
    int32_t *err;
};

// Eight consecutive state values <-> fp32 (one 16-byte vector of bf16, two of fp32).
__device__ __forceinline__ void load8(const bf16 *p, float (&f)[8]) { unpack16(*reinterpret_cast<const uint4 *>(p), f); }
__device__ __forceinline__ void load8(const float *p, float (&f)[8]) {
    const uint4 a = reinterpret_cast<const uint4 *>(p)[0], b = reinterpret_cast<const uint4 *>(p)[1];
    float lo[4], hi[4];
    unpack16(a, lo);
    unpack16(b, hi);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[k] = lo[k];
        f[4 + k] = hi[k];
    }
}
__device__ __forceinline__ void store8(bf16 *p, const float (&f)[8]) { *reinterpret_cast<uint4 *>(p) = pack16(f); }
__device__ __forceinline__ void store8(float *p, const float (&f)[8]) {
    const float lo[4] = {f[0], f[1], f[2], f[3]}, hi[4] = {f[4], f[5], f[6], f[7]};
    reinterpret_cast<uint4 *>(p)[0] = pack16(lo);
    reinterpret_cast<uint4 *>(p)[1] = pack16(hi);
}

// Copies conv bytes [chunk * 64 * blockDim.x, ...) between a slot and an entry (16-byte vectors).
__device__ __forceinline__ void copy_conv_chunk(const unsigned char *src, unsigned char *dst, int64_t bytes,
                                                int chunk) {
    for (int k = 0; k < 4; ++k) {
        const int64_t off = ((int64_t)chunk * 4 * blockDim.x + (int64_t)k * blockDim.x + threadIdx.x) * 16;
        if (off < bytes) *reinterpret_cast<uint4 *>(dst + off) = *reinterpret_cast<const uint4 *>(src + off);
    }
}

// Valid (slot, entry) pair of row i, else false (out-of-range ids are flagged once).
__device__ __forceinline__ bool pair_ok(const QArgs &a, int i, int32_t &sl, int32_t &en) {
    sl = a.slots[i];
    en = a.entries[i];
    if (sl < -1 || sl >= a.num_slots || en < -1 || en >= a.num_entries) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(a.err, MAMBA_ERR_SLOT_RANGE);
        return false;
    }
    return sl >= 0 && en >= 0;
}

// Row shares per column group in the store: the lanes of one warp, when the column groups of a
// row (a power of two) fill less than a warp; otherwise one.
__host__ __device__ inline int store_shares(int octs) {
    return (octs < 32 && (octs & (octs - 1)) == 0) ? 32 / octs : 1;
}

// Store: block (x, i); x < ceil(H / kStoreHeads) quantises a group of kStoreHeads heads of slot
// slots[i] into entry entries[i]; the blocks after them copy chunks of the conv window.  The
// group's state tiles (contiguous in the slot) arrive in shared memory with one bulk async copy;
// threads = (head, share of the rows, group of 8 d_state columns): pass 1 takes the column maxima
// of a share's rows and combines the shares with warp shuffles, pass 2 writes 8 codes per row.
template <typename StateT>
__global__ void __launch_bounds__(1024) k_ckpt_store_int8(const QArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    extern __shared__ __align__(128) unsigned char q_smem[];
    __shared__ uint64_t bar;
    int32_t sl, en;
    if (!pair_ok(a, blockIdx.y, sl, en)) return;
    unsigned char *entry = a.store + en * (int64_t)a.lay.total;
    const int hblocks = (a.H + kStoreHeads - 1) / kStoreHeads;
    if ((int)blockIdx.x >= hblocks) {
        if (a.conv)
            copy_conv_chunk(a.conv + sl * a.conv_stride, entry + a.lay.conv, a.conv_bytes, blockIdx.x - hblocks);
        return;
    }
    const int h0 = blockIdx.x * kStoreHeads, nh = min(kStoreHeads, a.H - h0);
    const int64_t tile = (int64_t)a.P * a.N;  // elements of one head
    const StateT *src = reinterpret_cast<const StateT *>(a.ssm + sl * a.ssm_stride) + h0 * tile;
    if (threadIdx.x == 0) {
        umma::mbar_init(&bar, 1);
        umma::fence_mbar_init();
        const uint32_t bytes = (uint32_t)(nh * tile * (int64_t)sizeof(StateT));
        umma::mbar_arrive_expect_tx(&bar, bytes);
        umma::bulk_g2s(q_smem, src, bytes, &bar);
    }
    __syncthreads();
    if (!umma::mbar_wait(&bar, 0, kQPolls)) {
        // the copy did not land in time: report it, give it one more bounded wait, and leave
        if (threadIdx.x == 0) {
            flag_error(a.err, MAMBA_ERR_TIMEOUT);
            umma::mbar_wait(&bar, 0, kQPolls);
        }
        return;
    }
    // thread = (head hl, row share sh, column group co), co fastest: a warp reads whole rows, and
    // the shares of one column group are lanes octs apart, combined with shuffles
    const int octs = a.N / 8, shares = store_shares(octs);
    const int hl = (int)threadIdx.x / (octs * shares), sh = ((int)threadIdx.x / octs) % shares;
    const int co = (int)threadIdx.x % octs;
    const int h = h0 + hl;
    const StateT *t = reinterpret_cast<const StateT *>(q_smem) + hl * tile + 8 * co;
    float m[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    if (hl < nh) {
#pragma unroll 4
        for (int p = sh; p < a.P; p += shares) {
            float v[8];
            load8(t + (int64_t)p * a.N, v);
#pragma unroll
            for (int k = 0; k < 8; ++k) m[k] = fmaxf(m[k], fabsf(v[k]));
        }
    }
    for (int off = octs; off < octs * shares; off <<= 1)  // all lanes of the warp take part
#pragma unroll
        for (int k = 0; k < 8; ++k) m[k] = fmaxf(m[k], __shfl_xor_sync(0xffffffffu, m[k], off));
    if (hl >= nh) return;
    float sc[8], rc[8];  // step amax / 127 and its reciprocal 127 / amax (0 for an all-zero column)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        sc[k] = m[k] / 127.0f;
        rc[k] = m[k] > 0.0f ? 127.0f / m[k] : 0.0f;
    }
    if (sh == 0) {
        float *scp = reinterpret_cast<float *>(entry + a.lay.scales) + (int64_t)h * a.N + 8 * co;
        reinterpret_cast<float4 *>(scp)[0] = make_float4(sc[0], sc[1], sc[2], sc[3]);
        reinterpret_cast<float4 *>(scp)[1] = make_float4(sc[4], sc[5], sc[6], sc[7]);
    }
    int8_t *q = reinterpret_cast<int8_t *>(entry + a.lay.q) + (int64_t)h * tile + 8 * co;
#pragma unroll 4
    for (int p = sh; p < a.P; p += shares) {
        float v[8];
        load8(t + (int64_t)p * a.N, v);
        // nearest code (round half to even, as rint), clamped to +-127, four codes packed per word
        int c[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) c[k] = max(-127, min(127, __float2int_rn(v[k] * rc[k])));
        const uint32_t w0 = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
        const uint32_t w1 = __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
        *reinterpret_cast<uint2 *>(q + (int64_t)p * a.N) = make_uint2(w0, w1);
    }
}

// Load: the inverse, state = q * s (fp32 product, then the pool dtype), into slot slots[i].
template <typename StateT>
__global__ void __launch_bounds__(kQThreads) k_ckpt_load_int8(const QArgs a) {
    pdl_wait();  // see pdl_wait: no global access before the previous grid is complete
    pdl_launch_dependents();
    int32_t sl, en;
    if (!pair_ok(a, blockIdx.y, sl, en)) return;
    const unsigned char *entry = a.store + en * (int64_t)a.lay.total;
    if ((int)blockIdx.x >= a.H) {
        if (a.conv) copy_conv_chunk(entry + a.lay.conv, a.conv + sl * a.conv_stride, a.conv_bytes, blockIdx.x - a.H);
        return;
    }
    const int h = blockIdx.x, octs = a.N / 8, shares = min(kQThreads / octs, a.P);
    const int co = threadIdx.x % octs, rs = threadIdx.x / octs;
    if (rs >= shares) return;
    const float4 *scp = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(entry + a.lay.scales) +
                                                         (int64_t)h * a.N + 8 * co);
    const float4 s0 = scp[0], s1 = scp[1];
    const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const int8_t *q = reinterpret_cast<const int8_t *>(entry + a.lay.q) + (int64_t)h * a.P * a.N + 8 * co;
    StateT *dst = reinterpret_cast<StateT *>(a.ssm + sl * a.ssm_stride) + (int64_t)h * a.P * a.N + 8 * co;
    // kLoadRows rows per pass, their codes loaded before any is converted
    for (int p0 = rs; p0 < a.P; p0 += shares * kLoadRows) {
        uint2 c[kLoadRows];
#pragma unroll
        for (int r = 0; r < kLoadRows; ++r) {
            const int p = p0 + r * shares;
            c[r] = p < a.P ? *reinterpret_cast<const uint2 *>(q + (int64_t)p * a.N) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int r = 0; r < kLoadRows; ++r) {
            const int p = p0 + r * shares;
            if (p >= a.P) break;
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t word = k < 4 ? c[r].x : c[r].y;
                const int code = (int)(int8_t)((word >> (8 * (k & 3))) & 0xffu);
                v[k] = (float)code * sc[k];
            }
            store8(dst + (int64_t)p * a.N, v);
        }
    }
}

// Host checks shared by store and load; fills the arguments.  MAMBA_OK or a negative status.
int q_args(const mamba_layer_desc *d, const void *ssm_pool, int64_t ssm_slot_stride, const void *conv_pool,
           int64_t conv_slot_stride, int64_t num_slots, const int32_t *slots, const int32_t *entries, int32_t n,
           const void *store, int64_t num_entries, int32_t *err, QArgs &a) {
    int rc = check_desc(d);
    if (rc != MAMBA_OK) return rc;
    if (n < 0 || n > 65535) return MAMBA_EINVAL;
    if (n == 0) return MAMBA_OK;
    if (!ssm_pool || !slots || !entries || !store || num_slots <= 0 || num_entries <= 0) return MAMBA_EINVAL;
    const int H = d->nheads, P = d->head_dim, N = d->d_state;
    if (N % 8 || N / 8 > kQThreads) return MAMBA_EUNSUPPORTED;
    if (ssm_slot_stride < (int64_t)H * P * N) return MAMBA_EINVAL;
    const size_t sb = dtype_bytes(d->state_dtype), cb = dtype_bytes(d->conv_dtype);
    const int64_t Cd = mamba_conv_dim(d), Wc = d->conv_kernel - 1 + d->num_spec;
    if (conv_pool && conv_slot_stride < Cd * Wc) return MAMBA_EINVAL;
    if (!aligned16(ssm_pool) || !aligned16(store) || (ssm_slot_stride * (int64_t)sb) % 16)
        return MAMBA_EALIGN;
    if (conv_pool && (!aligned16(conv_pool) || (conv_slot_stride * (int64_t)cb) % 16 || (Cd * Wc * (int64_t)cb) % 16))
        return MAMBA_EALIGN;
    a.ssm = static_cast<unsigned char *>(const_cast<void *>(ssm_pool));
    a.ssm_stride = ssm_slot_stride * (int64_t)sb;
    a.num_slots = num_slots;
    a.conv = static_cast<unsigned char *>(const_cast<void *>(conv_pool));
    a.conv_stride = conv_slot_stride * (int64_t)cb;
    a.store = static_cast<unsigned char *>(const_cast<void *>(store));
    a.num_entries = num_entries;
    a.lay = entry_layout(d);
    a.slots = slots;
    a.entries = entries;
    a.H = H;
    a.P = P;
    a.N = N;
    a.conv_bytes = Cd * Wc * (int64_t)cb;
    a.err = err;
    return MAMBA_OK;
}

}  // namespace

}  // namespace ms

using namespace ms;

extern "C" int mamba_slot_copy(const mamba_layer_desc *d, void *ssm_pool, int64_t ssm_slot_stride, int64_t num_slots,
                               void *conv_pool, int64_t conv_slot_stride, const int32_t *src_slots,
                               const int32_t *dst_slots, int32_t n, int32_t *err_word, void *stream) {
    MS_TRACE("mamba_slot_copy");
    int rc = check_desc(d);
    if (rc != MAMBA_OK) return rc;
    if (n < 0 || n > 65535) return MAMBA_EINVAL;
    if (n == 0) return MAMBA_OK;
    if (!ssm_pool || !src_slots || !dst_slots || num_slots <= 0) return MAMBA_EINVAL;
    const int64_t elems = (int64_t)d->nheads * d->head_dim * d->d_state;
    if (ssm_slot_stride < elems) return MAMBA_EINVAL;
    const size_t sb = dtype_bytes(d->state_dtype), cb = dtype_bytes(d->conv_dtype);
    const int64_t conv_elems = (int64_t)mamba_conv_dim(d) * (d->conv_kernel - 1 + d->num_spec);
    if (conv_pool && conv_slot_stride < conv_elems) return MAMBA_EINVAL;
    if (!aligned16(ssm_pool) || (ssm_slot_stride * (int64_t)sb) % 16 || (elems * (int64_t)sb) % 16) return MAMBA_EALIGN;
    if (conv_pool && (!aligned16(conv_pool) || (conv_slot_stride * (int64_t)cb) % 16 || (conv_elems * (int64_t)cb) % 16))
        return MAMBA_EALIGN;
    CopyArgs a;
    a.ssm = static_cast<unsigned char *>(ssm_pool);
    a.ssm_stride = ssm_slot_stride * (int64_t)sb;
    a.num_slots = num_slots;
    a.conv = static_cast<unsigned char *>(conv_pool);
    a.conv_stride = conv_slot_stride * (int64_t)cb;
    a.src = src_slots;
    a.dst = dst_slots;
    a.ssm_bytes = elems * (int64_t)sb;
    a.conv_bytes = conv_elems * (int64_t)cb;
    a.err = err_word;
    const int64_t total = a.ssm_bytes + (conv_pool ? a.conv_bytes : 0);
    const dim3 grid((unsigned)((total + kCopyBytes - 1) / kCopyBytes), n);
    if (launch_pdl(k_slot_copy, grid, dim3(kCopyThreads), 0, static_cast<cudaStream_t>(stream), a) != cudaSuccess)
        return MAMBA_ECUDA;
    return launch_status();
}

extern "C" size_t mamba_int8_entry_bytes(const mamba_layer_desc *d) {
    if (check_desc(d) != MAMBA_OK) return 0;
    return entry_layout(d).total;
}

extern "C" int mamba_ckpt_store_int8(const mamba_layer_desc *d, const void *ssm_pool, int64_t ssm_slot_stride,
                                     const void *conv_pool, int64_t conv_slot_stride, int64_t num_slots,
                                     const int32_t *src_slots, const int32_t *dst_entries, int32_t n, void *store,
                                     int64_t num_entries, int32_t *err_word, void *stream) {
    MS_TRACE("mamba_ckpt_store_int8");
    QArgs a;
    const int rc = q_args(d, ssm_pool, ssm_slot_stride, conv_pool, conv_slot_stride, num_slots, src_slots, dst_entries,
                          n, store, num_entries, err_word, a);
    if (rc != MAMBA_OK || n == 0) return rc;
    const size_t smem = (size_t)kStoreHeads * d->head_dim * d->d_state * dtype_bytes(d->state_dtype);
    const int octs = d->d_state / 8;
    int threads = kStoreHeads * octs * store_shares(octs);
    threads = (threads + 31) / 32 * 32;  // whole warps (the shuffles need every lane)
    if (smem > 200 * 1024 || threads > 1024) return MAMBA_EUNSUPPORTED;
    const int conv_blocks = conv_pool ? (int)((a.conv_bytes + 64 * threads - 1) / (64 * threads)) : 0;
    const dim3 grid((a.H + kStoreHeads - 1) / kStoreHeads + conv_blocks, n);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto kern = d->state_dtype == MAMBA_BF16 ? k_ckpt_store_int8<bf16> : k_ckpt_store_int8<float>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MAMBA_ECUDA;
    if (launch_pdl(kern, grid, dim3(threads), smem, st, a) != cudaSuccess) return MAMBA_ECUDA;
    return launch_status();
}

extern "C" int mamba_ckpt_load_int8(const mamba_layer_desc *d, void *ssm_pool, int64_t ssm_slot_stride,
                                    void *conv_pool, int64_t conv_slot_stride, int64_t num_slots,
                                    const int32_t *src_entries, const int32_t *dst_slots, int32_t n, const void *store,
                                    int64_t num_entries, int32_t *err_word, void *stream) {
    MS_TRACE("mamba_ckpt_load_int8");
    QArgs a;
    const int rc = q_args(d, ssm_pool, ssm_slot_stride, conv_pool, conv_slot_stride, num_slots, dst_slots, src_entries,
                          n, store, num_entries, err_word, a);
    if (rc != MAMBA_OK || n == 0) return rc;
    const int conv_blocks = conv_pool ? (int)((a.conv_bytes + 64 * kQThreads - 1) / (64 * kQThreads)) : 0;
    const dim3 grid(a.H + conv_blocks, n);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = d->state_dtype == MAMBA_BF16 ? launch_pdl(k_ckpt_load_int8<bf16>, grid, dim3(kQThreads), 0, st, a)
                                                       : launch_pdl(k_ckpt_load_int8<float>, grid, dim3(kQThreads), 0, st, a);
    if (e != cudaSuccess) return MAMBA_ECUDA;
    return launch_status();
}
