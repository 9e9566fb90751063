/*
 * sdpa_fwd.h -- C ABI of the sliding-window SDPA forward on GB300 (sm_103a):
 * O and the natural-log normaliser LSE that the backward (sdpa_bwd.h) takes as
 * inputs.
 *
 * What it computes (the forward whose gradients the cuDNN-frontend pages'
 * backward returns -- PR #2352 "Summary", PR #866 "Change"): for each q-head h
 * of sequence b and each query row i < Lq_b,
 *     s_ij = scale * q_i . k_j             over the keys j the mask admits
 *     LSE_i = log( sum_j exp(s_ij) + exp(sink_h) )   (sink term only with a sink)
 *     O_i  = sum_j exp(s_ij - LSE_i) v_j
 * with the mask of sdpa_bwd.h (modes, windows, anchor i + diag_b, lengths).
 * A row that admits no key gets O = 0 and LSE = -inf, or LSE = sink_h with a
 * sink. Rows of a slot past its sequence's length get O = 0 and LSE = -inf.
 * K and V are shared by the h_q / h_kv q-heads of a group (GQA, MQA).
 *
 * Precision: S and O accumulate in fp32 on the tensor cores, P is rounded to
 * the I/O dtype for the P V product (as the backward rounds P and dS); O is
 * written in the I/O dtype, LSE in fp32.
 *
 * Errors: host-side validation returns SDPA_ERR_INVALID_ARG / UNSUPPORTED with
 * a message (sdpa_bwd_last_error()); launch failures SDPA_ERR_CUDA. Every wait
 * inside the kernel is bounded; a wait that runs out sets a device status
 * word, shared by all forwards on the device, that sdpa_fwd_check_status()
 * returns (SDPA_ERR_TIMEOUT).
 */
#ifndef SDPA_FWD_H
#define SDPA_FWD_H

#include "sdpa_bwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Problem description: the fields mean what they mean in sdpa_bwd_params
 * (same layouts, strides in elements, 16-byte alignment, lengths, offsets).
 * O has Q's shape and layout; LSE is fp32 [b, h_q, s_q] (BSHD) or
 * [h_q, total_q] (THD), contiguous, as the backward reads it.
 */
typedef struct sdpa_fwd_params {
    int32_t dtype;          /* SDPA_BF16 | SDPA_F16 for Q, K, V, O */
    int32_t layout;         /* SDPA_BSHD | SDPA_THD */
    int32_t mask_mode;      /* SDPA_MASK_* */
    int32_t reserved0;
    int64_t b, h_q, h_kv, s_q, s_kv, total_q, total_kv, d;
    int64_t window_left, window_right;
    float scale;
    int32_t reserved1;
    const int32_t *seq_q_lens, *seq_kv_lens; /* device [b] or NULL */
    const int32_t *q_offsets, *kv_offsets;   /* device [b+1], THD only */
    const void *q, *k, *v;                   /* device inputs, dtype */
    const float *sink;                       /* device fp32 [h_q] or NULL */
    void *o;                                 /* device output, dtype */
    float *lse;                              /* device output, fp32 */
    int64_t q_stride[3], k_stride[3], v_stride[3], o_stride[3];
} sdpa_fwd_params;

/* Enqueues the forward on `stream` (a cudaStream_t; NULL = legacy default
 * stream). Owns no memory: every buffer is the caller's. */
sdpa_status_t sdpa_fwd(const sdpa_fwd_params *params, void *stream);

/* Synchronises `stream` and returns the forward's device status on the
 * current device (SDPA_OK or SDPA_ERR_TIMEOUT), then clears it.
 * The status word is one per device, shared by every sdpa_fwd call on it (the
 * forward takes no workspace): a timeout of any forward on the device is
 * reported by the next check, whichever stream it ran on, and forwards that
 * run concurrently on other streams while this call reads and clears the word
 * may have their status cleared with it. Check from one stream at a time, or
 * after synchronising the device, to attribute a status to one call. */
sdpa_status_t sdpa_fwd_check_status(void *stream);

/* sizeof(sdpa_fwd_params) as compiled into the library, for binding checks. */
size_t sdpa_fwd_params_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_FWD_H */
