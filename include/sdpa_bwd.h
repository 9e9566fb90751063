/*
 * sdpa_bwd.h -- C ABI of the GB300 (sm_103a) sliding-window scaled-dot-product
 * attention backward: dQ, dK, dV and (with attention sinks) dSink.
 *
 * The operation (cuDNN-frontend PR #866 "frost(sdpa): bound the SM80 backward
 * q-loop by the sliding window ... + window-aware deterministic relay",
 * "Change" section; PR #557 "frost(sdpa): GQA/MQA, padding mask, right-band
 * widening, and sink-token gradients for the SM120 f16 backward", "Summary"):
 *
 *   for batch b, q-head h, kv-head g = h / (h_q / h_kv), query row i < Lq_b:
 *     anchor(i) = i + diag_b,  diag_b = Lkv_b - Lq_b (bottom-right) else 0
 *     key j < Lkv_b is attended iff  anchor(i) - j <= window_left  (if >= 0)
 *                                and j - anchor(i) <= right        (if >= 0)
 *     where right = max(window_right, 0) for the causal modes and
 *     window_right (negative = unbounded) for SDPA_MASK_NONE;
 *     P_ij = exp(scale * q_i.k_j - LSE_i),  D_i = dO_i . O_i,
 *     dS_ij = P_ij (dO_i.v_j - D_i),
 *     dV_j = sum P_ij dO_i,  dK_j = scale sum dS_ij q_i,  dQ_i = scale sum dS_ij k_j,
 *     dSink_h = -sum_{b, i < Lq_b} exp(sink_h - LSE_i) D_i.
 *
 * Each kv-tile's sweep over q-tiles is clamped on both sides by the window
 * (work O(S*W) rather than O(S^2)); a kv-tile that no query reaches writes
 * dK = dV = 0.
 *
 * Conventions common to every entry point:
 *  - Ownership: the caller owns every buffer, including the workspace. The
 *    library allocates nothing and keeps no state between calls.
 *  - Asynchrony: the four compute calls enqueue kernels on `stream` and return
 *    without synchronising. They must be called in the order
 *      sdpa_bwd_preprocess, sdpa_bwd, sdpa_bwd_dq_convert, sdpa_bwd_gqa_reduce
 *    on one stream with the same params and workspace.
 *  - Errors: argument checks run on the host before anything is enqueued and
 *    return SDPA_ERR_INVALID_ARG / SDPA_ERR_UNSUPPORTED; sdpa_bwd_last_error()
 *    then names the offending argument. A failed launch returns SDPA_ERR_CUDA.
 *    Problems found on the device (a relay wait that ran out, sequence lengths
 *    that do not fit their slots) are recorded in a status word inside the
 *    workspace and reported by sdpa_bwd_check_status().
 *  - Pointers marked (device) must be device memory of the current device.
 */
#ifndef SDPA_BWD_H
#define SDPA_BWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SDPA_OK = 0,
    SDPA_ERR_INVALID_ARG = 1,  /* bad shape, pointer, stride or flag */
    SDPA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d not 64/128) */
    SDPA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    SDPA_ERR_TIMEOUT = 4,      /* a deterministic-relay wait ran out on the device */
    SDPA_ERR_BAD_LENGTHS = 5,  /* device-side: a sequence length exceeds its slot */
    SDPA_ERR_WORKSPACE = 6,    /* workspace NULL, misaligned or too small */
    SDPA_ERR_BOUNDS = 7        /* device-side, range-checked build only (compiled with
                                  -DSDPA_DEBUG_BOUNDS): a computed index fell outside its
                                  buffer; the access was skipped */
} sdpa_status_t;

enum { SDPA_BF16 = 0, SDPA_F16 = 1 };
enum { SDPA_BSHD = 0, SDPA_THD = 1 };
enum { SDPA_MASK_NONE = 0, SDPA_MASK_TOP_LEFT = 1, SDPA_MASK_BOTTOM_RIGHT = 2 };

/*
 * Problem description. All strides are in elements; the feature (d) stride
 * of every tensor is 1 and every other stride must be a multiple of 8
 * elements (16 bytes), with 16-byte aligned base pointers.
 *
 * Layouts
 *  SDPA_BSHD: Q, O, dO, dQ are [b, s_q, h_q, d]; K, V, dK, dV [b, s_kv, h_kv, d]
 *    (strides[0] = batch, [1] = sequence, [2] = head). seq_q_lens/seq_kv_lens
 *    (device int32 [b], optional) give the actual lengths (padding mask); NULL
 *    means every sequence is full (s_q / s_kv). LSE is fp32 [b, h_q, s_q],
 *    contiguous.
 *  SDPA_THD: tokens of all sequences packed: Q, O, dO, dQ are [total_q, h_q, d],
 *    K, V, dK, dV [total_kv, h_kv, d] (strides[0] ignored, [1] = token,
 *    [2] = head). q_offsets/kv_offsets (device int32 [b+1], required) are the
 *    first token of each sequence's slot, with offsets[0] = 0 and
 *    offsets[b] = total. Lengths (optional, device int32 [b]) may be shorter
 *    than the slots; tokens of a slot past its length are "gap" tokens. s_q and
 *    s_kv must be at least the longest slot (offsets difference). LSE is fp32
 *    [h_q, total_q], contiguous.
 *  Rows and tokens past a sequence's length receive dQ = 0 / dK = dV = 0; their
 *  input values are never read into a result.
 *
 * Semantics of the mask fields are those given at the top of this file.
 * LSE is the natural-log normaliser of the forward, including the sink
 * logit when a sink is used; a row that attended nothing has LSE = -inf.
 */
typedef struct sdpa_bwd_params {
    int32_t dtype;          /* SDPA_BF16 | SDPA_F16 for Q, K, V, O, dO, dQ, dK, dV */
    int32_t layout;         /* SDPA_BSHD | SDPA_THD */
    int32_t mask_mode;      /* SDPA_MASK_* */
    int32_t deterministic;  /* 0: dQ by unordered fp32 atomics; 1: bitwise
                               repeatable: per-visitor partial slots summed in
                               visitor order where a q-tile can have three or
                               more visitors and the slots fit 2 GiB of
                               workspace, else the ordered relay; 2: bitwise
                               repeatable, ordered relay only */
    int64_t b;              /* batch size (THD: number of sequences) */
    int64_t h_q, h_kv;      /* heads; h_q % h_kv == 0 (MHA, GQA, MQA) */
    int64_t s_q, s_kv;      /* BSHD: padded lengths; THD: longest slot */
    int64_t total_q, total_kv; /* THD: tokens in the packed tensors; BSHD: unused */
    int64_t d;              /* head dimension: 64 or 128 */
    int64_t window_left;    /* < 0: no left window */
    int64_t window_right;   /* right band; see the top of this file */
    float scale;            /* softmax scale applied to q.k (e.g. 1/sqrt(d)) */
    int32_t reserved0;
    const int32_t *seq_q_lens, *seq_kv_lens; /* device [b] or NULL */
    const int32_t *q_offsets, *kv_offsets;   /* device [b+1], THD only */
    const void *q, *k, *v, *o, *dout;        /* device, dtype */
    const float *lse;                        /* device fp32 (layout above) */
    const float *sink;                       /* device fp32 [h_q] or NULL */
    void *dq, *dk, *dv;                      /* device outputs, dtype */
    float *dsink;                            /* device fp32 [h_q]; set iff sink */
    int64_t q_stride[3], k_stride[3], v_stride[3], o_stride[3], do_stride[3];
    int64_t dq_stride[3], dk_stride[3], dv_stride[3];
} sdpa_bwd_params;

/*
 * Workspace size in bytes for `params` (0 on invalid params; see
 * sdpa_bwd_last_error). The workspace holds the fp32 dQ accumulator, D = rowsum
 * (dO*O), the relay counters, the dSink partials, the status word, at d = 64
 * the main kernel's table of decoded work items (152 bytes per (batch,
 * kv-head, kv-tile), rewritten by every sdpa_bwd call) and, in deterministic mode 1 when
 * a q-tile can have three or more visitors, up to 2 GiB of per-visitor partial
 * dQ tiles. It must be 256-byte aligned device memory; its contents need no
 * initialisation.
 */
size_t sdpa_bwd_workspace_bytes(const sdpa_bwd_params *params);

/*
 * Preprocess ("dot" kernel of PR #557's four-kernel split; delta of its dSink
 * formula): D[b,h,i] = sum_d dO*O in fp32 for every row; zeroes the per-q-tile
 * relay counters, the status word and (non-deterministic mode) the fp32 dQ
 * accumulator rows of q-tiles that three or more kv-tiles visit; writes the
 * dSink partials -exp(sink_h - LSE_i) * D_i summed over each block of
 * unpadded rows. O and dO are read by TMA in blocks of up to 16 q-heads x 16
 * rows (d = 64; 8 rows at d = 128; more rows with fewer heads).
 */
sdpa_status_t sdpa_bwd_preprocess(const sdpa_bwd_params *params, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * Main backward ("main" kernel; PR #866 clamp and relay): one work item per
 * (kv-tile, kv-head, batch); at d = 64 each CTA first decodes its items
 * (sequence lengths, clamped q-tile range) into the workspace's item table,
 * which its roles then read. For each q-head of the kv-head's group and each
 * q-tile in the clamped range [q_lo, q_hi) (swept from the top down) it
 * recomputes P and dS and accumulates dV, dK in tensor memory, so the GQA/MQA
 * group sum (PR #557) happens in place, in head order; stores dK, dV.
 * dQ = scale * dS K of a q-tile is combined over the contiguous kv-tiles that
 * visit it, [kv_first, kv_first + n) with kv_first = max((q_row0 + diag - W)
 * // tile_kv, 0): a lone visitor stores dQ directly; with two visitors, or in
 * deterministic mode without slots, the tile passes along the relay (turn
 * t - kv_first) through the fp32 accumulator and the last turn stores dQ; in
 * deterministic mode with slots (three or more visitors), each visitor stores
 * its fp32 partial in its own slot (turn) and sdpa_bwd_dq_convert sums them in
 * visitor order; otherwise the visitors add with fp32 atomics and
 * sdpa_bwd_dq_convert stores dQ.
 */
sdpa_status_t sdpa_bwd(const sdpa_bwd_params *params, void *workspace, size_t workspace_bytes,
                       void *stream);

/*
 * dQ convert ("cvt" kernel): dQ = dtype(fp32 accumulator) on the q-tiles that
 * took unordered atomics, dQ = dtype(sum of the visitors' partial slots, in
 * visitor order) on the q-tiles that used slots, dQ = 0 on rows no kv-tile
 * visits (padding, gap tokens, rows outside every window), and dsink[h] =
 * fixed-order sum of the dSink partials (when a sink is used).
 */
sdpa_status_t sdpa_bwd_dq_convert(const sdpa_bwd_params *params, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * GQA reduction ("reduce" step, PR #557 GQA/MQA): dK[., g] and dV[., g] are
 * sums over the q-heads of group g. sdpa_bwd already forms these sums in
 * tensor memory (in head order), so this call only validates its arguments and
 * enqueues nothing; it is kept so that the four-call sequence is the same for
 * every head layout.
 */
sdpa_status_t sdpa_bwd_gqa_reduce(const sdpa_bwd_params *params, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * Synchronises `stream` and returns the device status word of the last
 * backward run on `workspace`: SDPA_OK, SDPA_ERR_TIMEOUT (a device wait gave
 * up -- a dQ relay turn, the partial of a dQ pair split between two CTAs, or a
 * hand-off inside the main kernel, named by sdpa_bwd_last_error(); the
 * gradients are then incomplete), SDPA_ERR_BAD_LENGTHS, SDPA_ERR_BOUNDS (a
 * range-checked build found an index outside its buffer), or
 * SDPA_ERR_UNSUPPORTED (the
 * device placed the main kernel's dynamic shared memory off a 1024-byte
 * boundary, which its swizzled tiles need; it then computed nothing).
 */
sdpa_status_t sdpa_bwd_check_status(const void *workspace, void *stream);

/*
 * Whole backward without a caller-provided workspace. The pages have no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory: a plug-in whose host application owns all device memory and
 * lends none, a latency-critical path that must not pay for cudaMalloc's
 * implicit synchronisation, or a deployment that forbids allocation once it
 * has started.
 *
 * It enqueues the same four stages as sdpa_bwd_preprocess, sdpa_bwd,
 * sdpa_bwd_dq_convert and sdpa_bwd_gqa_reduce on `stream`, with their scratch
 * in a fixed array of SDPA_BWD_NO_ALLOC_MAX_BYTES inside this library (static
 * device memory that every GPU loading the library keeps until the process
 * exits). It calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Size limit: a problem whose sdpa_bwd_workspace_bytes() exceeds
 *    SDPA_BWD_NO_ALLOC_MAX_BYTES is rejected with SDPA_ERR_WORKSPACE before
 *    anything is enqueued; use the workspace entry points for it. In
 *    deterministic mode 1 the per-visitor dQ slots are dropped first (the call
 *    runs as mode 2, the relay: also bitwise repeatable) when that makes the
 *    problem fit.
 *  - Set-up: every call looks up the array's device address on the current
 *    device (cudaGetSymbolAddress: no allocation). The first call on a device
 *    may load the library's device code there, so make it before any stream
 *    capture.
 *  - Sharing: every call on a device uses the same array and leaves its
 *    contents behind; each call re-zeroes what must start at zero. Calls whose
 *    work overlaps on the GPU (other streams, other threads) race on the array
 *    and must be serialised by the caller.
 *  - Device-side status (a wait that ran out, lengths longer than their
 *    slots) lands at the start of the array: sdpa_bwd_no_alloc_check_status()
 *    reads it. Host-side errors are returned as for the other calls.
 */
#define SDPA_BWD_NO_ALLOC_MAX_BYTES ((size_t)32 << 20)
sdpa_status_t sdpa_bwd_no_alloc(const sdpa_bwd_params *params, void *stream);

/*
 * Device status of the last sdpa_bwd_no_alloc run on the current device, as
 * sdpa_bwd_check_status() reports it for a workspace: synchronises `stream`
 * (the stream that run was enqueued on) and reads the status word at the start
 * of the fixed scratch. Like the array itself, the word is shared by every call
 * on the device. Allocates nothing. The pages have no counterpart to this call.
 */
sdpa_status_t sdpa_bwd_no_alloc_check_status(void *stream);

/* Message of the last host-side error on the calling thread ("" if none). */
const char *sdpa_bwd_last_error(void);

/*
 * Test hook for the device-side failure handling; not for production use.
 * Every wait inside the backward kernels is bounded (2 s by default): a wait
 * that runs out records SDPA_ERR_TIMEOUT in the workspace's status word, the
 * kernel stops issuing work, lets the copies and contractions already in
 * flight finish, frees its tensor memory and returns, and
 * sdpa_bwd_check_status() reports it (the gradients are then incomplete).
 * This call changes, for the calling thread's later sdpa_bwd() calls:
 *   wait_limit_ns  the bound of every device wait (<= 0: the default);
 *   flags          bit 0: each dQ relay turn waits for a counter value no
 *                  visitor writes; bit 1: the second visitor of a dQ pair split
 *                  between two CTAs waits for a flag no visitor sets (both
 *                  waits then run out); 0: normal operation.
 * Returns SDPA_ERR_INVALID_ARG for undefined flag bits. Call it with (0, 0) to
 * restore normal operation.
 */
sdpa_status_t sdpa_bwd_test_hook(int64_t wait_limit_ns, int32_t flags);

/* sizeof(sdpa_bwd_params) as compiled into the library, for binding checks. */
size_t sdpa_bwd_params_bytes(void);

/* Main-kernel tile sizes (rows of a kv-tile and of a q-tile). */
int32_t sdpa_bwd_tile_kv(void);
int32_t sdpa_bwd_tile_q(void);

/*
 * Number of GPU kernels that sdpa_bwd_preprocess, sdpa_bwd,
 * sdpa_bwd_dq_convert and sdpa_bwd_gqa_reduce launch, together, for `params`
 * (sdpa_bwd_no_alloc launches the same ones); -1 if the shape is invalid. No
 * device work: the counts follow the host-side decisions those calls make
 * (empty problems launch nothing; dq_convert is skipped when the main kernel
 * has written every dQ row; gqa_reduce never launches).
 */
int32_t sdpa_bwd_kernel_launches(const sdpa_bwd_params *params);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_BWD_H */
