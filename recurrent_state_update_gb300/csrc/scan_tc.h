// scan_tc.h -- internal interface of the tensor-core chunked prefill (chunk_scan_tc.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mamba_state.h"

namespace ms {

struct ScanTcParams {
    void *ssm_pool;
    int64_t ssm_stride, num_slots;
    const int32_t *cu, *slot;
    const uint8_t *has_init;
    const int32_t *ckpt_slots;
    int max_ckpt, ckpt_interval;
    int nseq, T, H, G, HG;
    const void *x, *dt, *B, *C, *z;
    int dt_bf16, dt_softplus;
    const float *A, *D, *dt_bias;
    void *y;
    int32_t *err;
    int32_t *meta;  // workspace: [valid, pad x3, order[nseq]]
};

// True when the tensor-core path handles this layer and chunk (bf16 activations and state,
// head_dim 64, d_state 128, chunk a multiple of 128).
bool scan_tc_eligible(const mamba_layer_desc *d, int chunk);

// Workspace bytes of the tensor-core path.
size_t scan_tc_workspace_bytes(int nseq);

// Launches the tensor-core path; MAMBA_OK or a negative status.
int scan_tc_launch(const ScanTcParams &p, int state_bf16, cudaStream_t stream);

}  // namespace ms
