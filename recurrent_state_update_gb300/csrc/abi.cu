// abi.cu -- size helpers and status strings of the C ABI (host only).
#include "common.cuh"

using namespace ms;

extern "C" int32_t mamba_conv_dim(const mamba_layer_desc *d) {
    if (check_desc(d) != MAMBA_OK) return -1;
    return d->nheads * d->head_dim + 2 * d->n_groups * d->d_state;
}

extern "C" int64_t mamba_ssm_state_bytes(const mamba_layer_desc *d) {
    if (check_desc(d) != MAMBA_OK) return -1;
    return (int64_t)d->nheads * d->head_dim * d->d_state * (int64_t)dtype_bytes(d->state_dtype);
}

extern "C" int64_t mamba_conv_state_bytes(const mamba_layer_desc *d) {
    if (check_desc(d) != MAMBA_OK) return -1;
    return (int64_t)mamba_conv_dim(d) * (d->conv_kernel - 1 + d->num_spec) * (int64_t)dtype_bytes(d->conv_dtype);
}

extern "C" const char *mamba_status_string(int status) {
    switch (status) {
        case MAMBA_OK: return "MAMBA_OK";
        case MAMBA_EINVAL: return "MAMBA_EINVAL: invalid argument";
        case MAMBA_EUNSUPPORTED: return "MAMBA_EUNSUPPORTED: shape or dtype not compiled";
        case MAMBA_ECUDA: return "MAMBA_ECUDA: CUDA runtime error";
        case MAMBA_EALIGN: return "MAMBA_EALIGN: pointer or stride not aligned";
        case MAMBA_ENOSPACE: return "MAMBA_ENOSPACE: buffer too small";
        default: return "unknown mamba_status";
    }
}
