// abi.cu -- size helpers, status strings and the slot-id check of the C ABI (host only).
#include <vector>

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

// Host-side check of one call's slot ids: each id is -1 or inside the pool, and no id other
// than -1 is used twice by one call (the slot ids of live rows and their scratch slots).
extern "C" int mamba_check_slot_ids(const int32_t *slot_ids, int32_t batch, const int32_t *scratch_slots,
                                    int32_t ntok, int64_t num_slots, int64_t *first_bad) {
    if (first_bad) *first_bad = -1;
    if (batch < 0 || num_slots <= 0 || (batch > 0 && !slot_ids) || (scratch_slots && ntok <= 0)) return MAMBA_EINVAL;
    std::vector<uint8_t> used((size_t)num_slots, 0);
    auto take = [&](int32_t s, int64_t idx) {
        if (s == -1) return true;
        if (s < -1 || s >= num_slots || used[(size_t)s]) {
            if (first_bad) *first_bad = idx;
            return false;
        }
        used[(size_t)s] = 1;
        return true;
    };
    for (int32_t i = 0; i < batch; ++i)
        if (!take(slot_ids[i], i)) return MAMBA_EINVAL;
    if (scratch_slots)
        for (int32_t i = 0; i < batch; ++i) {
            if (slot_ids[i] == -1) continue;  // a padding row writes nothing, its scratch slots included
            for (int32_t j = 0; j < ntok; ++j)
                if (!take(scratch_slots[(int64_t)i * ntok + j], (int64_t)batch + (int64_t)i * ntok + j))
                    return MAMBA_EINVAL;
        }
    return MAMBA_OK;
}
