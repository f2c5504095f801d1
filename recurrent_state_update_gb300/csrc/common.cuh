// common.cuh -- dtype helpers, validation and launch plumbing shared by the CUDA sources of
// libmamba_state.so.  Nothing here is visible through the C ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdlib>

#include "mamba_state.h"

// NVTX ranges: every exported call that launches work opens a range named after the call for
// its host-side duration (argument checks and launches), so a timeline tool (Nsight Systems,
// or any NVTX injection library) shows which library call issued which kernels.  Built in by
// default; compile with -DMS_NVTX=0 to leave them out.  With no tool attached a range costs a
// call through a null-checked function pointer.
#ifndef MS_NVTX
#define MS_NVTX 1
#endif
#if MS_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace ms {

#if MS_NVTX
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
#define MS_TRACE(name) ::ms::NvtxRange ms_nvtx_range_(name)
#else
#define MS_TRACE(name) ((void)0)
#endif

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------------------------------
// scalar conversions: bf16 <-> fp32 (bf16 stores round to nearest even)
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// Unpack a 16-byte vector into fp32 values (8 bf16 or 4 fp32).
__device__ __forceinline__ void unpack16(const uint4 &r, float (&f)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}
__device__ __forceinline__ void unpack16(const uint4 &r, float (&f)[4]) {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
}

// Pack fp32 values into a 16-byte vector (bf16: round to nearest even).
__device__ __forceinline__ uint4 pack16(const float (&f)[8]) {
    uint4 r;
    uint32_t *w = reinterpret_cast<uint32_t *>(&r);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 v = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t *>(&v);
    }
    return r;
}
__device__ __forceinline__ uint4 pack16(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
}

// Elements per 16-byte vector.
template <typename T>
struct Vec16 {
    static constexpr int n = 16 / (int)sizeof(T);
};

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }

// SiLU with the fast exponential and divide intrinsics (a few ulp; for large negative v the
// divide by an infinite denominator gives 0, the limit).
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// softplus in fp32: log(1 + e^s), with the linear branch above 20 (the tail below the branch
// point differs from s by less than e^-20 relative).
__device__ __forceinline__ float softplus_f(float s) { return s > 20.0f ? s : log1pf(expf(s)); }

__device__ __forceinline__ float load_scalar(const void *p, int64_t idx, bool is_bf16) {
    return is_bf16 ? __bfloat162float(static_cast<const bf16 *>(p)[idx])
                   : static_cast<const float *>(p)[idx];
}

__device__ __forceinline__ void flag_error(int32_t *err, int32_t bit) {
    if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------------------

inline size_t dtype_bytes(int32_t dt) { return dt == MAMBA_BF16 ? 2 : (dt == MAMBA_F32 ? 4 : 0); }
inline bool dtype_ok(int32_t dt) { return dt == MAMBA_F32 || dt == MAMBA_BF16; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Basic structural checks on a layer descriptor; MAMBA_OK or MAMBA_EINVAL.
inline int check_desc(const mamba_layer_desc *d) {
    if (!d) return MAMBA_EINVAL;
    if (d->nheads <= 0 || d->head_dim <= 0 || d->d_state <= 0 || d->n_groups <= 0) return MAMBA_EINVAL;
    if (d->nheads % d->n_groups) return MAMBA_EINVAL;
    if (d->conv_kernel < 2 || d->conv_kernel > 8 || d->num_spec < 0 || d->num_spec > 32)
        return MAMBA_EINVAL;
    if (!dtype_ok(d->state_dtype) || !dtype_ok(d->conv_dtype) || !dtype_ok(d->act_dtype) ||
        !dtype_ok(d->dt_dtype))
        return MAMBA_EINVAL;
    return MAMBA_OK;
}

// Programmatic dependent launch.  The decode-path kernels are launched with the programmatic
// stream-serialization attribute, so the hardware may start their CTAs while the previous kernel
// in the stream is still finishing; each of them first executes pdl_wait(), which blocks until
// every prerequisite grid has completed and its memory is visible, before it touches global
// memory, so the result is the same as a plain launch: only the launch latency and the
// prologue overlap the previous kernel's tail.  pdl_wait() is a no-op in a kernel launched
// without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream be scheduled (it still waits for this one to complete).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// Whether launches request programmatic dependent launch: yes unless the environment variable
// MAMBA_PDL is "0" when the library first launches (read once per process).
inline bool pdl_enabled() {
    static const bool on = [] {
        const char *v = std::getenv("MAMBA_PDL");
        return !(v && v[0] == '0' && v[1] == 0);
    }();
    return on;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MAMBA_OK : MAMBA_ECUDA;
}

}  // namespace ms
