/*
 * mamba_state.h -- C ABI of libmamba_state.so: the Mamba2 recurrent-state update over a
 * slot-indexed state pool, on one NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (page title, section / equation):
 *  [P1] "Hybrid SSM / Mamba models and non-KV state" (mlinterviewnotes.com):
 *       - the Mamba2 state shapes: conv state (d_conv, W-1+num_spec) with
 *         d_conv = d_inner + 2*n_groups*d_state, temporal state (nheads, head_dim, d_state);
 *       - the slot pool: each state object is one tensor with a layer and a slot dimension,
 *         plus one extra slot used for padding; a request owns an integer slot id;
 *       - the decode call selective_state_update(ssm_state, x, dt, A, B, C, D, z, dt_bias,
 *         dt_softplus, state_batch_indices, out);
 *       - the prefill call mamba_chunk_scan_combined(x viewed (1, T, H, P), dt, A, ...) and the
 *         chunked-prefill state hand-off (has_initial_states);
 *       - align-mode checkpoints: states kept at multiples of the block size;
 *       - the block-table "none"/"align" columns 1 + num_speculative_blocks (speculative
 *         decode keeps 1 + num_spec state pages per request).
 *  [P4] echobase "Mamba" notes, the Mamba block equations:
 *         x = SiLU(Conv1d(x')),  Delta_t = Softplus(.),
 *         h_t = exp(Delta_t A) h_{t-1} + Delta_t B_t x_t,  y_t = C_t h_t,  y_hat = y (.) SiLU(z),
 *       the classic output y_t = C h_t + D x_t, and the SSD form Y = (M (.) L) X with
 *         M_ij = C_i (prod_{k=j+1..i} Abar_k) Bbar_j,  L the causal mask.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library allocates no
 *    memory.  Every tensor is dense row-major in the layout given beside it.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *    and never synchronise the host.
 *  - Errors the host can see (null required pointer, unsupported shape or dtype, a pointer
 *    not 16-byte aligned, a launch failure) return a negative mamba_status and launch
 *    nothing.  Errors that depend on device data (a slot id outside the pool, i.e. below -1
 *    or >= num_slots, an accept length out of range, bad cu_seqlens) are found in the kernel:
 *    the affected unit is left untouched and a MAMBA_ERR_* bit is OR-ed into *err_word (a
 *    device int32 the caller zeroes and reads; it may be NULL to ignore such errors).  A
 *    bounded wait that gives up (MAMBA_ERR_TIMEOUT) is the one exception: see that bit.
 *  - The method's domain is A <= 0 and steps Delta >= 0 (Delta = softplus(.) > 0 with
 *    dt_softplus): every decay factor exp(Delta*A) is then at most 1, for any step size.
 *  - Slot ids within one call must be distinct (also across slot_ids and scratch_slots);
 *    the result is undefined otherwise.  Slot id -1 marks a padding row: its state and its
 *    output rows are not touched.
 *  - Head h uses group g(h) = h / (nheads / n_groups).  xBC channels are ordered
 *    [x (nheads*head_dim) | B (n_groups*d_state) | C (n_groups*d_state)].
 */
#ifndef MAMBA_STATE_H
#define MAMBA_STATE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MAMBA_OK = 0,
    MAMBA_EINVAL = -1,       /* bad argument: null pointer, negative size, inconsistent shape */
    MAMBA_EUNSUPPORTED = -2, /* valid but not compiled: head_dim/d_state/dtype combination */
    MAMBA_ECUDA = -3,        /* a CUDA runtime call or kernel launch failed */
    MAMBA_EALIGN = -4,       /* a pointer or stride breaks the 16-byte alignment rule */
    MAMBA_ENOSPACE = -5      /* a caller-provided buffer is too small */
} mamba_status;

typedef enum { MAMBA_F32 = 0, MAMBA_BF16 = 1 } mamba_dtype;

/* Data-dependent error bits OR-ed into *err_word. */
#define MAMBA_ERR_SLOT_RANGE 0x1   /* a slot / scratch / checkpoint slot id below -1 or >= num_slots
                                      (-1 is padding / skip wherever a call allows it) */
#define MAMBA_ERR_ACCEPT_RANGE 0x2 /* an accept length outside [0, ntok] */
#define MAMBA_ERR_SEQLENS 0x4      /* cu_seqlens not non-decreasing from 0 to total_tokens */
#define MAMBA_ERR_TIMEOUT 0x8      /* an asynchronous copy or matrix operation did not complete within the
                                      kernel's bounded wait; that row / sequence is incomplete: its
                                      output is not written and its state may be partly advanced
                                      (some heads updated, others not), so restore it from a
                                      checkpoint or a copy before using it again */

/* One Mamba2 layer [P1 state shapes, P4 block equations]. */
typedef struct mamba_layer_desc {
    int32_t nheads;      /* H */
    int32_t head_dim;    /* P */
    int32_t d_state;     /* N */
    int32_t n_groups;    /* G; nheads % n_groups == 0 */
    int32_t conv_kernel; /* W, 2..8 */
    int32_t num_spec;    /* extra conv-state columns for speculative tokens, >= 0 */
    int32_t state_dtype; /* mamba_dtype of the SSM (temporal) state pool */
    int32_t conv_dtype;  /* mamba_dtype of the conv state pool; must equal act_dtype */
    int32_t act_dtype;   /* mamba_dtype of xBC, x, B, C, z and y */
    int32_t dt_dtype;    /* mamba_dtype of dt */
} mamba_layer_desc;

/* ---------------------------------------------------------------------------------------- */
/* sizes and status                                                                         */
/* ---------------------------------------------------------------------------------------- */

/* conv_dim = nheads*head_dim + 2*n_groups*d_state [P1 state shapes]; -1 on a bad desc. */
int32_t mamba_conv_dim(const mamba_layer_desc *desc);

/* Bytes of one slot of the SSM state, nheads*head_dim*d_state*sizeof(state_dtype)
 * [P1 temporal state]; -1 on a bad desc. */
int64_t mamba_ssm_state_bytes(const mamba_layer_desc *desc);

/* Bytes of one slot of the conv state, conv_dim*(conv_kernel-1+num_spec)*sizeof(conv_dtype)
 * [P1 conv state]; -1 on a bad desc. */
int64_t mamba_conv_state_bytes(const mamba_layer_desc *desc);

/* MAMBA_OK when the decode kernels are compiled for this desc, else MAMBA_EUNSUPPORTED or
 * MAMBA_EINVAL.  Compiled: (head_dim, d_state) in {(16,16), (32,64), (64,64), (64,128),
 * (128,128)}, state f32 or bf16, act bf16 or f32, dt f32 or bf16. */
int mamba_decode_supported(const mamba_layer_desc *desc);

/* Human-readable name of a mamba_status. */
const char *mamba_status_string(int status);

/*
 * mamba_check_slot_ids -- host-side check of one call's slot ids before they go to the device
 * [P1 slot pool: a request owns one slot id; a padding row uses a reserved id].  HOST pointers:
 *   slot_ids       (batch)       int32, -1 = padding row
 *   scratch_slots  (batch, ntok) int32 or NULL, -1 = no write for that token; the entries of a
 *                                padding row are ignored (the row writes nothing)
 * Every id must be -1 or in [0, num_slots), and no id other than -1 may appear twice among the
 * live rows' slot ids and scratch slots (the distinct-slot precondition of every call that
 * writes the pool).  Returns MAMBA_OK, or MAMBA_EINVAL with *first_bad (may be NULL) set to
 * the index of the first offending entry, scratch entry (i, j) counted as batch + i*ntok + j,
 * or -1 when the arguments themselves are invalid.  Uses host memory of num_slots bytes for
 * the duration of the call; touches no device memory.
 */
int mamba_check_slot_ids(const int32_t *slot_ids, int32_t batch, const int32_t *scratch_slots, int32_t ntok,
                         int64_t num_slots, int64_t *first_bad);

/*
 * mamba_selftest_wait_timeout -- diagnostic of this library's failure path (the pages have no
 * counterpart).  Every kernel here bounds each wait on its asynchronous copies and matrix
 * operations (2^18 mbarrier polls, about one second on GB300) and reports a wait that runs out as
 * MAMBA_ERR_TIMEOUT instead of hanging.  This call launches one small kernel that waits, with the same bounded wait, on a
 * barrier phase nothing completes: after about one second it gives up, ORs MAMBA_ERR_TIMEOUT
 * into *err_word (device int32, required) and stores the wait's duration in nanoseconds into
 * *elapsed_ns (device uint64, may be NULL).  It touches nothing else, and the CUDA context stays
 * usable.  Asynchronous on stream.
 */
int mamba_selftest_wait_timeout(int32_t *err_word, uint64_t *elapsed_ns, void *stream);

/* ---------------------------------------------------------------------------------------- */
/* decode                                                                                   */
/* ---------------------------------------------------------------------------------------- */

/*
 * mamba_conv_update -- causal depthwise conv1d + SiLU over ntok new tokens per request,
 * updating the conv state in place [P1: the conv state keeps the most recent W-1 inputs;
 * P4 x = SiLU(Conv1d(x'))].
 *
 *   conv_pool        (num_slots, ...) with slot s at conv_pool + s*conv_slot_stride elements;
 *                    a slot holds (conv_dim, Wc) with Wc = conv_kernel-1+num_spec, each
 *                    channel's Wc columns contiguous, oldest first.
 *   slot_ids         (batch) int32, -1 = padding (row skipped, xbc_out row not written).
 *   xbc_in           (batch, ntok, conv_dim) act_dtype, raw inputs.
 *   conv_w           (conv_dim, conv_kernel) fp32; the newest input meets conv_w[c, W-1].
 *   conv_b           (conv_dim) fp32 or NULL.
 *   xbc_out          (batch, ntok, conv_dim) act_dtype: SiLU(conv + bias).  May not alias xbc_in.
 * Token j's window is the last W-1 inputs before it followed by itself.  After the call the
 * slot holds the last Wc inputs (shifted left by ntok, new inputs appended).
 * Limits: 1 <= ntok <= 64, batch <= 65535.
 */
int mamba_conv_update(const mamba_layer_desc *desc, void *conv_pool, int64_t conv_slot_stride,
                      int64_t num_slots, const int32_t *slot_ids, int32_t batch, int32_t ntok,
                      const void *xbc_in, const float *conv_w, const float *conv_b, void *xbc_out,
                      int32_t *err_word, void *stream);

/*
 * mamba_state_update -- the batched decode step [P1 selective_state_update call; P4 block
 * equations]: for each row i with s = slot_ids[i] != -1, for tokens j = 0..ntok-1 in order,
 * for each head h (group g):
 *     Delta = softplus(dt[i,j,h] + dt_bias[h])   (dt + dt_bias when dt_softplus == 0)
 *     hst[p,n] <- exp(Delta*A[h]) * hst[p,n] + Delta * B[g,n] * x[h,p]
 *     y[i,j,h,p] = sum_n C[g,n] * hst[p,n] + D[h]*x[h,p];   y *= SiLU(z[i,j,h,p]) if z
 * where x | B | C are the xBC channels after the conv (when conv_pool != NULL the conv of
 * mamba_conv_update is fused in and the conv state is updated in place; when NULL, xbc is
 * taken as already convolved).
 *
 *   ssm_pool         slot s at ssm_pool + s*ssm_slot_stride elements: (nheads, head_dim,
 *                    d_state) state_dtype, d_state contiguous.  Read, updated in fp32, and
 *                    written back (bf16: round to nearest even).
 *   conv_pool        as in mamba_conv_update, or NULL.
 *   conv_w, conv_b   as in mamba_conv_update (conv_w required when conv_pool != NULL).
 *   slot_ids         (batch) int32, -1 = padding.
 *   scratch_slots    (batch, ntok) int32 or NULL.  When given (speculative decode), the state
 *                    after token j is written to slot scratch_slots[i, j] and slot_ids[i] is
 *                    NOT written; when NULL the state after the last token is written back to
 *                    slot_ids[i].
 *   xbc              (batch, ntok, conv_dim) act_dtype.
 *   dt               (batch, ntok, nheads) dt_dtype.
 *   A                (nheads) fp32, required.   D, dt_bias: (nheads) fp32 or NULL.
 *   z                (batch, ntok, nheads*head_dim) act_dtype or NULL (no gate).
 *   y                (batch, ntok, nheads*head_dim) act_dtype.
 * Limits: 1 <= ntok <= 8, batch <= 65535.
 * Alignment: ssm_pool and the SSM slot stride in bytes must be multiples of 16; the other
 * tensors must be aligned to their element size (MAMBA_EALIGN otherwise).
 */
int mamba_state_update(const mamba_layer_desc *desc, void *ssm_pool, int64_t ssm_slot_stride,
                       int64_t num_slots, void *conv_pool, int64_t conv_slot_stride,
                       const float *conv_w, const float *conv_b, const int32_t *slot_ids,
                       const int32_t *scratch_slots, int32_t batch, int32_t ntok, const void *xbc,
                       const void *dt, const float *A, const float *D, const float *dt_bias,
                       int32_t dt_softplus, const void *z, void *y, int32_t *err_word, void *stream);

/*
 * mamba_spec_commit -- after a speculative mamba_state_update of ntok draft tokens with
 * scratch slots, keep the first accept_len[i] tokens of row i [P1: 1 + num_speculative_blocks
 * state pages per request so a rejected suffix rolls back]:
 *   - accept a >= 1: the state in scratch_slots[i, a-1] is copied into slot_ids[i];
 *     a == 0 leaves slot_ids[i] unchanged;
 *   - conv_pool (may be NULL): the slot's conv state, which the speculative step left holding
 *     the last Wc inputs up to draft token ntok, is moved right by ntok - a columns so its
 *     last W-1 columns end at accepted token a; the ntok - a freed columns are zeroed.
 *     Requires ntok <= num_spec.
 * accept_len: (batch) int32 in [0, ntok]; out of range -> MAMBA_ERR_ACCEPT_RANGE, row skipped.
 */
int mamba_spec_commit(const mamba_layer_desc *desc, void *ssm_pool, int64_t ssm_slot_stride,
                      int64_t num_slots, void *conv_pool, int64_t conv_slot_stride,
                      const int32_t *slot_ids, const int32_t *scratch_slots,
                      const int32_t *accept_len, int32_t batch, int32_t ntok, int32_t *err_word,
                      void *stream);

/* ---------------------------------------------------------------------------------------- */
/* chunked prefill                                                                          */
/* ---------------------------------------------------------------------------------------- */

/*
 * mamba_conv_varlen -- the causal depthwise conv1d + SiLU that produces the scan's x, B and C
 * for a varlen prefill batch, continuing each sequence from its stored conv state and leaving
 * the conv state a later chunk or decode step continues from [P4 x = SiLU(Conv1d(x')); P1 the
 * conv state object, a window of the most recent inputs, carried across prefill chunks like the
 * temporal state (has_initial_states)].  For sequence s (tokens [cu_seqlens[s],
 * cu_seqlens[s+1]), length L) define its input stream
 *     e(q) = xbc[cu_seqlens[s] + q, c]                    for 0 <= q < L,
 *     e(q) = conv state column Wc + q of slot_ids[s]      for -Wc <= q < 0 when
 *            has_initial_state[s] != 0, else 0,
 * then  out[cu_seqlens[s] + q, c] = SiLU(conv_b[c] + sum_{k<W} conv_w[c, k] * e(q - (W-1) + k))
 * is split by channel into x_out (c < nheads*head_dim), B_out and C_out (the two blocks of
 * n_groups*d_state channels that follow), and afterwards the slot's conv state column i holds
 * e(L - Wc + i), i = 0..Wc-1 (Wc = conv_kernel-1+num_spec): the last Wc inputs of the stream.
 *
 *   conv_pool        as in mamba_conv_update, or NULL: then every sequence starts from zeros,
 *                    no conv state is read or written, and slot_ids / has_initial_state are
 *                    ignored.
 *   cu_seqlens       (nseq + 1) int32 as in mamba_chunk_scan (bad values: MAMBA_ERR_SEQLENS,
 *                    nothing written).
 *   slot_ids         (nseq) int32; -1: outputs computed from zeros, no state written; outside
 *                    [-1, num_slots): MAMBA_ERR_SLOT_RANGE and that sequence's outputs and
 *                    state are left untouched.
 *   has_initial_state (nseq) uint8 or NULL (all zero).
 *   xbc              (total_tokens, conv_dim) act_dtype raw inputs, 16-byte aligned.
 *   conv_w (conv_dim, conv_kernel) fp32;  conv_b (conv_dim) fp32 or NULL.
 *   x_out            (total_tokens, nheads*head_dim) act_dtype, 16-byte aligned.
 *   B_out, C_out     (total_tokens, n_groups*d_state) act_dtype, 16-byte aligned.
 * Requires nheads*head_dim and n_groups*d_state to be multiples of 16 bytes' worth of act_dtype
 * elements (MAMBA_EUNSUPPORTED otherwise).  Two kernels run in stream order: the conv, then the
 * state write-back.
 */
int mamba_conv_varlen(const mamba_layer_desc *desc, void *conv_pool, int64_t conv_slot_stride,
                      int64_t num_slots, const int32_t *cu_seqlens, int32_t nseq,
                      int32_t total_tokens, const int32_t *slot_ids,
                      const uint8_t *has_initial_state, const void *xbc, const float *conv_w,
                      const float *conv_b, void *x_out, void *B_out, void *C_out,
                      int32_t *err_word, void *stream);

/*
 * Bytes of device workspace mamba_chunk_scan needs for these sizes (0 on a bad argument).
 */
size_t mamba_chunk_scan_workspace_bytes(const mamba_layer_desc *desc, int32_t total_tokens,
                                        int32_t nseq, int32_t chunk);

/*
 * mamba_chunk_scan -- varlen chunked prefill in the SSD form [P1 mamba_chunk_scan_combined: the
 * within-chunk term as a masked matrix product on tensor cores, chunks joined by a short scan
 * over chunk states; P4 Y = (M (.) L) X].
 * Sequence s owns tokens [cu_seqlens[s], cu_seqlens[s+1]) of x; its tokens are split into
 * chunks of `chunk` tokens from its first token (the last chunk may be partial).  Per head:
 *     y_t = C_t . h_t + D*x_t  (then * SiLU(z_t) if z),  h_t = exp(Delta_t A) h_{t-1} + Delta_t x_t B_t^T
 * with h_{-1} = the state in slot_ids[s] when has_initial_state[s] != 0, else 0
 * [P1: a later prefill chunk continues from the stored state].  After the call slot_ids[s] holds the state after
 * the sequence's last token; when ckpt_slots is given, ckpt_slots[s, k-1] (k >= 1, -1 = skip)
 * receives the state after the first k*ckpt_interval tokens of the sequence [P1 align mode:
 * states cached at positions i * block_size].
 *
 *   ssm_pool, ssm_slot_stride, num_slots   as in mamba_state_update.
 *   cu_seqlens       (nseq + 1) int32, non-decreasing, cu_seqlens[0] = 0,
 *                    cu_seqlens[nseq] = total_tokens.
 *   slot_ids         (nseq) int32 (-1: the sequence's outputs are computed, no state written).
 *   has_initial_state (nseq) uint8 or NULL (all zero).
 *   ckpt_slots       (nseq, max_ckpt) int32 or NULL;  ckpt_interval must be a positive
 *                    multiple of chunk when given.
 *   chunk            tokens per chunk; 256 is compiled.
 *   x                (total_tokens, nheads, head_dim) act_dtype.
 *   dt               (total_tokens, nheads) dt_dtype.
 *   A (nheads) fp32;  D, dt_bias (nheads) fp32 or NULL.
 *   B, C             (total_tokens, n_groups, d_state) act_dtype.
 *   z                (total_tokens, nheads, head_dim) act_dtype or NULL.
 *   y                (total_tokens, nheads, head_dim) act_dtype.
 *   workspace        device buffer of at least mamba_chunk_scan_workspace_bytes(...) bytes,
 *                    16-byte aligned (MAMBA_ENOSPACE when workspace_bytes is smaller).
 * Paths: bf16 activations with a bf16 state pool at head_dim 64, d_state 128 and a chunk that
 * is a multiple of 128 run on the tensor cores (bf16 matrix operands, fp32 accumulation and
 * state).  Every other case, and any fp32 state pool, runs in fp32 on the CUDA cores, which
 * requires chunk 256, head_dim <= 64, and d_state a power of two in 32..256 with
 * 256 / d_state dividing head_dim (MAMBA_EUNSUPPORTED otherwise): an fp32 pool's states are
 * computed and written in fp32 throughout.
 */
int mamba_chunk_scan(const mamba_layer_desc *desc, void *ssm_pool, int64_t ssm_slot_stride,
                     int64_t num_slots, const int32_t *cu_seqlens, int32_t nseq,
                     int32_t total_tokens, const int32_t *slot_ids,
                     const uint8_t *has_initial_state, const int32_t *ckpt_slots,
                     int32_t max_ckpt, int32_t ckpt_interval, int32_t chunk, const void *x,
                     const void *dt, const float *A, const void *B, const void *C, const float *D,
                     const float *dt_bias, int32_t dt_softplus, const void *z, void *y,
                     void *workspace, size_t workspace_bytes, int32_t *err_word, void *stream);

/* ---------------------------------------------------------------------------------------- */
/* prefix-cache checkpoints: slot copy and the int8 checkpoint store                        */
/* ---------------------------------------------------------------------------------------- */

/*
 * mamba_slot_copy -- batched slot-to-slot copy of whole states [P1: on a prefix-cache hit the
 * cached state is copied into a fresh slot rather than shared (copy-on-write), since the
 * recurrence updates its slot in place].  For each i with src_slots[i] and dst_slots[i] both
 * != -1, the SSM state (and, when conv_pool is given, the conv state) of slot src_slots[i] is
 * copied bit for bit into slot dst_slots[i]; src == dst is a no-op.
 *   ssm_pool, conv_pool, strides, num_slots   as in mamba_state_update / mamba_conv_update.
 *   src_slots, dst_slots  (n) int32; an id outside [-1, num_slots): MAMBA_ERR_SLOT_RANGE and
 *                         that row is skipped.  dst ids must be distinct and no dst may be
 *                         another row's src.
 * Alignment: pools, slot strides and the per-slot state sizes in bytes multiples of 16.
 * Limits: n <= 65535.
 */
int mamba_slot_copy(const mamba_layer_desc *desc, void *ssm_pool, int64_t ssm_slot_stride,
                    int64_t num_slots, void *conv_pool, int64_t conv_slot_stride,
                    const int32_t *src_slots, const int32_t *dst_slots, int32_t n,
                    int32_t *err_word, void *stream);

/*
 * Bytes of one entry of the int8 checkpoint store (0 on a bad desc).  An entry holds, each
 * section starting on a 256-byte boundary: the codes q (nheads, head_dim, d_state) int8; the
 * scales (nheads, d_state) fp32; the conv window (conv_dim, conv_kernel-1+num_spec) in
 * conv_dtype.  At the Nemotron-H-8B shape an entry is about 1.1 MB against 2 MiB for a bf16 slot.
 */
size_t mamba_int8_entry_bytes(const mamba_layer_desc *desc);

/*
 * mamba_ckpt_store_int8 -- quantise cached states into the int8 store [P1: SGLang's checkpoint
 * store keeps cached temporal states in int8, symmetric per (head, k-channel), quantised once on
 * store; the conv window is kept at its native dtype].  The k-channel of the temporal state
 * (nheads, head_dim, d_state) is the d_state index n, so for each head h and n of slot
 * src_slots[i], in fp32:
 *     a = max_p |state[h, p, n]|,   s[h, n] = a / 127,
 *     q[h, p, n] = clamp(rint(state[h, p, n] * (127 / a)), -127, 127)   (0 where a == 0),
 * written to entry dst_entries[i] of `store` together with a copy of the slot's conv window
 * (when conv_pool is given).
 *   store        device buffer of num_entries * mamba_int8_entry_bytes(desc) bytes, 16-byte
 *                aligned; entry e starts at e * mamba_int8_entry_bytes(desc).
 *   src_slots, dst_entries  (n) int32, -1 = skip the row; out of range: MAMBA_ERR_SLOT_RANGE.
 * Requires d_state a multiple of 8, d_state <= 512 and 4 * head_dim * d_state state elements to
 * fit in 200 KB (MAMBA_EUNSUPPORTED otherwise); alignment as in
 * mamba_slot_copy.
 */
int mamba_ckpt_store_int8(const mamba_layer_desc *desc, const void *ssm_pool, int64_t ssm_slot_stride,
                          const void *conv_pool, int64_t conv_slot_stride, int64_t num_slots,
                          const int32_t *src_slots, const int32_t *dst_entries, int32_t n,
                          void *store, int64_t num_entries, int32_t *err_word, void *stream);

/*
 * mamba_ckpt_load_int8 -- dequantise entries into fresh active slots [P1: dequantised once into
 * a fresh active slot on a hit]: state[h, p, n] = q[h, p, n] * s[h, n] (fp32 product, stored in
 * state_dtype, bf16 round to nearest even), and the entry's conv window copied into the slot's
 * conv state (when conv_pool is given).
 *   src_entries, dst_slots  (n) int32, -1 = skip; out of range: MAMBA_ERR_SLOT_RANGE.
 * Other arguments and limits as in mamba_ckpt_store_int8.
 */
int mamba_ckpt_load_int8(const mamba_layer_desc *desc, void *ssm_pool, int64_t ssm_slot_stride,
                         void *conv_pool, int64_t conv_slot_stride, int64_t num_slots,
                         const int32_t *src_entries, const int32_t *dst_slots, int32_t n,
                         const void *store, int64_t num_entries, int32_t *err_word, void *stream);

/* ---------------------------------------------------------------------------------------- */
/* chunked prefill without a caller workspace                                               */
/* ---------------------------------------------------------------------------------------- */

/*
 * mamba_chunk_scan_noalloc -- the same operation, arguments and results as mamba_chunk_scan,
 * for callers that cannot provide a device workspace.  The pages have no counterpart: this
 * entry point exists for callers that must not allocate device memory, such as an engine whose
 * memory pool has already reserved the GPU (a further cudaMalloc fails, or synchronises the
 * whole device and stalls every stream) or a latency-critical path that may not call
 * cudaMalloc / cudaFree.  It allocates nothing and calls no allocating routine.
 *
 * Its scratch is one fixed array of mamba_chunk_scan_static_scratch_bytes() bytes (128 MiB)
 * compiled into the library: every GPU that loads the library holds that memory until the
 * process exits.  A call whose workspace would exceed it (mamba_chunk_scan_workspace_bytes
 * larger than that size) returns MAMBA_ENOSPACE and launches nothing.
 *
 * The first call on each device looks up that device's address of the array (with the device
 * current); make that first call before any stream capture.  All calls share the one array and
 * nothing in it carries over between calls, but two calls that run at the same time on the GPU
 * (on different streams or from different host threads) race on it: order them.
 */
int mamba_chunk_scan_noalloc(const mamba_layer_desc *desc, void *ssm_pool, int64_t ssm_slot_stride,
                             int64_t num_slots, const int32_t *cu_seqlens, int32_t nseq,
                             int32_t total_tokens, const int32_t *slot_ids,
                             const uint8_t *has_initial_state, const int32_t *ckpt_slots,
                             int32_t max_ckpt, int32_t ckpt_interval, int32_t chunk, const void *x,
                             const void *dt, const float *A, const void *B, const void *C,
                             const float *D, const float *dt_bias, int32_t dt_softplus, const void *z,
                             void *y, int32_t *err_word, void *stream);

/* Size in bytes of the fixed scratch mamba_chunk_scan_noalloc uses (no counterpart on the pages). */
size_t mamba_chunk_scan_static_scratch_bytes(void);

/* ---------------------------------------------------------------------------------------- */
/* Mamba1 (S6) layers                                                                        */
/* ---------------------------------------------------------------------------------------- */

/* One Mamba1 layer [P1: the Mamba1 conv state (D, W-1) and recurrent state (D, N); P4 the Mamba
 * block equations, with a step and a row of A per channel]. */
typedef struct mamba1_layer_desc {
    int32_t d_inner;     /* D, the channels; a multiple of 8 */
    int32_t d_state;     /* N: 8, 16, 32 or 64 */
    int32_t conv_kernel; /* W, 2..8 */
    int32_t num_spec;    /* extra conv-state columns, >= 0 */
    int32_t state_dtype; /* mamba_dtype of the (D, N) state pool */
    int32_t conv_dtype;  /* mamba_dtype of the conv state pool; must equal act_dtype */
    int32_t act_dtype;   /* mamba_dtype of x, B, C, z and y */
    int32_t dt_dtype;    /* mamba_dtype of dt */
} mamba1_layer_desc;

/*
 * mamba1_conv_update -- the causal depthwise conv1d + SiLU of a Mamba1 layer over ntok new tokens
 * per request (the D channels of x; B, C and the step are projected from its output outside this
 * library), with the conv state updated in place.  Same semantics, layouts and limits as
 * mamba_conv_update with conv_dim = d_inner.
 */
int mamba1_conv_update(const mamba1_layer_desc *desc, void *conv_pool, int64_t conv_slot_stride,
                       int64_t num_slots, const int32_t *slot_ids, int32_t batch, int32_t ntok,
                       const void *x_in, const float *conv_w, const float *conv_b, void *x_out,
                       int32_t *err_word, void *stream);

/*
 * mamba1_state_update -- the batched single-token decode step of a Mamba1 layer [P4: h_t =
 * exp(Delta_t A) h_{t-1} + Delta_t B_t x_t, y_t = C_t h_t (+ D x_t), y_hat = y (.) SiLU(z); P1 the
 * (D, N) state in a slot pool].  For each row i with s = slot_ids[i] != -1 and each channel d:
 *     Delta = softplus(dt[i, d] + dt_bias[d])   (dt + dt_bias when dt_softplus == 0)
 *     h[d, n] <- exp(Delta * A[d, n]) * h[d, n] + Delta * B[i, n] * x[i, d]
 *     y[i, d] = sum_n C[i, n] * h[d, n] + D[d] * x[i, d];   y *= SiLU(z[i, d]) if z
 *   ssm_pool    slot s at ssm_pool + s*ssm_slot_stride elements: (d_inner, d_state) state_dtype,
 *               d_state contiguous; read, updated in fp32 and written back (bf16: RNE).
 *   slot_ids    (batch) int32, -1 = padding (row skipped, y row not written).
 *   x           (batch, d_inner) act_dtype, the conv output.
 *   dt          (batch, d_inner) dt_dtype.
 *   A           (d_inner, d_state) fp32, required.   D, dt_bias: (d_inner) fp32 or NULL.
 *   B, C        (batch, d_state) act_dtype.
 *   z, y        (batch, d_inner) act_dtype (z may be NULL).
 * Alignment: ssm_pool and the slot stride in bytes multiples of 16, the other tensors aligned to
 * their element size.  Limits: batch <= 65535.
 */
int mamba1_state_update(const mamba1_layer_desc *desc, void *ssm_pool, int64_t ssm_slot_stride,
                        int64_t num_slots, const int32_t *slot_ids, int32_t batch, const void *x,
                        const void *dt, const float *A, const void *B, const void *C, const float *D,
                        const float *dt_bias, int32_t dt_softplus, const void *z, void *y,
                        int32_t *err_word, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_STATE_H */
