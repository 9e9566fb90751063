// sdpa_internal.h -- argument blocks shared by the host launcher (api.cu) and
// the kernels (aux_kernels.cu, main_kernel.cu). Plain structs passed by value
// as kernel parameters.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace swa {

constexpr int kTileKV = 128;      // kv rows per CTA work item (MMA M of dK/dV side)
constexpr int kTileQ = 128;       // q rows per inner-loop step
// Preprocess block: up to 16 q-heads x `rows` token rows, the most that one
// 256-thread CTA covers with one (row, head) unit (d = 64) or half a unit
// (d = 128) per thread; rows is a power of two that divides 128.
struct PreTile {
    int heads, rows;
};
inline __host__ __device__ PreTile pre_tile(int64_t h_q, int64_t d)
{
    const int heads = h_q < 16 ? static_cast<int>(h_q) : 16;
    const int units = 256 / static_cast<int>(d / 64);
    int rows = 1;
    while (rows * 2 * heads <= units && rows < 128) rows *= 2;
    return PreTile{heads, rows};
}
// Bytes of one decoded main-kernel work item (the kernel checks its record
// type against this).
constexpr size_t kItemBytes = 152;
constexpr int kStatusUnsupported = 2;  // same codes as sdpa_status_t
constexpr int kStatusTimeout = 4;
constexpr int kStatusBadLengths = 5;
constexpr int kStatusBounds = 7;     // range-checked build: an access fell outside its buffer
// Second status word: which global-memory wait of the main kernel ran out
// first (0: none, or an mbarrier hand-off inside a CTA).
constexpr int kWhereRelay = 200;   // a relay turn
constexpr int kWherePair = 201;    // the partial of a strip-mode pair split between two CTAs

// Workspace layout (byte offsets from the workspace base, 256-B aligned).
struct WsLayout {
    size_t status;      // int32 status, int32 where (which global-memory wait ran out)
    size_t dq_acc;      // fp32 [rows_q][h_q][d]
    size_t stats;       // fp32 per-row statistics, [b][h_q][n_q_tiles][2][128]: per q-tile
                        // 128 x -LSE * log2(e), then 128 x -D
    size_t sems;        // int32 [b][h_q][n_q_tiles]
    size_t dsink_part;  // fp32 [h_q][n_row_blocks]
    // deterministic mode, q-tiles with three or more visitors: one fp32 partial
    // dQ tile per visitor, [b][h_q][n_q_tiles][n_slots][128][d] (0: relay only)
    size_t dq_part;
    int64_t n_slots;
    // d = 64: the main kernel's decoded work items, one kItemBytes record per
    // (sequence, kv-head, kv-tile), written and read by that launch only
    size_t items;
    size_t total;
    int64_t n_sems;
    int64_t n_row_blocks;
};

// Elements reachable from each base pointer, for the range-checked build
// (-DSDPA_DEBUG_BOUNDS): every raw global access checks its index against
// these, records kStatusBounds and skips the access if it falls outside.
// Unused (and the checks compiled out) otherwise.
struct Extents {
    int64_t q, k, v, o, dout, dq, dk, dv;   // 16-bit elements
    int64_t lse, stats, dq_acc, dq_part, dsink_part, sink;   // fp32 elements
    int64_t sems;                           // int32 counters
};

// Sequence geometry common to all kernels.
struct Geometry {
    int32_t layout;     // 0 BSHD, 1 THD
    int32_t mask_mode;  // 0 none, 1 top-left, 2 bottom-right
    int64_t b, h_q, h_kv, s_q, s_kv, d;
    int64_t rows_q, rows_kv;   // BSHD: b*s; THD: total tokens
    int64_t window_left;       // < 0 unbounded
    int64_t right;             // effective right bound, < 0 unbounded
    const int32_t* seq_q_lens;
    const int32_t* seq_kv_lens;
    const int32_t* q_offsets;
    const int32_t* kv_offsets;
    Extents ext;
};

struct PreArgs {
    // TMA descriptors of O and dO (BSHD 4-D (d, h, s, b), THD 3-D (d, h, t)),
    // boxes of d x pre_heads x pre_rows, no swizzle
    CUtensorMap tm_o, tm_do;
    int32_t pre_heads, pre_rows;
    Geometry g;
    const void* o;
    const void* dout;
    const float* lse;
    const float* sink;
    int64_t o_stride[3], do_stride[3];
    float* dq_acc;       // zeroed here on q-tiles that take unordered atomics
    int32_t deterministic;
    // Per q-tile of a (sequence, q-head): 128 x -LSE * log2(e) (-inf where a row
    // attends nothing or lies past the length), then 128 x -D (0 there). Negated
    // and split so that the main kernel forms each pair of exponent arguments
    // with one packed fp32x2 FMA and each pair of (dP - D) with one packed add.
    float* stats;
    int64_t stats_row;   // rows per (sequence, q-head): n_q_tiles * 128 (2 floats each)
    int32_t* status;     // status + where (2 ints)
    int32_t* sems;
    int64_t n_sems;
    float* dsink_part;
    int64_t n_row_blocks;
    uint32_t ring_bytes;  // shared-memory ring of O/dO stages (set by the launcher)
};

struct MainArgs {
    // TMA descriptors of Q, K, V, dO: BSHD 4-D (d, h, s, b), THD 3-D (d, h, t);
    // 64 x 1 x 128 boxes with the 128-byte swizzle.
    CUtensorMap tm_q, tm_k, tm_v, tm_do;
    // Output descriptors for TMA stores from staged tiles: dQ, dK, dV (I/O
    // dtype, 64 x 1 x 128 boxes) and the fp32 dQ accumulator (32 x 1 x 128
    // boxes), all with the 128-byte swizzle.
    CUtensorMap tm_dq, tm_dk, tm_dv, tm_acc;
    // the per-visitor partial dQ tiles (fp32, 3-D (d, 1, rows), 32 x 1 x 128
    // boxes, 128-byte swizzle); used when n_slots > 0
    CUtensorMap tm_part;
    Geometry g;
    const void *q, *k, *v, *dout;
    const float* stats;       // per q-tile -LSE * log2(e) and -D runs (see PreArgs)
    int64_t stats_row;
    float* dq_acc;            // fp32 partial sums of q-tiles with several visitors
    void* dq;                 // dQ output (I/O dtype), written by each q-tile's last visitor
    int64_t dq_stride[3];
    void *dk, *dv;            // dK, dV (I/O dtype), summed over each kv-head's group
    int32_t* status;
    int32_t* sems;
    int64_t q_stride[3], k_stride[3], v_stride[3], do_stride[3], dk_stride[3], dv_stride[3];
    int64_t n_kv_tiles;       // tiles per sequence slot (grid x)
    int64_t n_q_tiles;        // relay counters per (b, h)
    float scale;
    float scale_log2;         // scale * log2(e)
    int32_t deterministic;
    int64_t n_slots;          // per-visitor partial dQ slots (deterministic mode), 0: relay
    int64_t timeout_ns;
    // d = 64: n_items = b * h_kv * n_kv_tiles records of kItemBytes (8-byte
    // aligned); each CTA decodes its own items into it once, before its roles
    // start, when use_items is set (the launcher sets it when a CTA has few
    // items; with many, the roles decode in place)
    void* items;
    int32_t use_items;
    // Strip mode (non-zero when no q-tile can have more than two visiting
    // kv-tiles, d = 64): each CTA walks a contiguous run of work items
    // numbered kv-tile fastest and sweeps each item's q-tiles from the bottom
    // up, so that the two visitors of a q-tile are consecutive steps of one CTA
    // except where the run ends. The main kernel's launcher sets it to the
    // number of consecutive kv-heads whose items share one set of runs.
    int32_t strip;
    // Test hook (zero in normal use): bit 0 makes every relay turn wait for a
    // counter value no visitor writes, bit 1 makes the second arrival of a
    // pair split between two CTAs wait for a flag no visitor sets; with a short
    // timeout_ns both give up and report SDPA_ERR_TIMEOUT.
    int32_t test_flags;
};

struct CvtArgs {
    Geometry g;
    const float* dq_acc;  // converted here on q-tiles that took unordered atomics
    const float* dq_part; // per-visitor partials, summed here in visitor order
    int64_t n_slots;      // 0: no partial slots
    int64_t n_q_tiles;
    int32_t deterministic;
    void* dq;
    int64_t dq_stride[3];
    const float* dsink_part;
    int64_t n_row_blocks;
    float* dsink;
    int32_t* status;      // device status word (range-checked build)
    int32_t head_chunk;   // q-heads per unit (set by the launcher)
};

// The forward pass (O and LSE): one work item per (q-tile, q-head, sequence).
struct FwdArgs {
    // TMA descriptors of Q, K, V (loads) and O (stores): 64 x 1 x 128 boxes,
    // 128-byte swizzle; BSHD 4-D (d, h, s, b), THD 3-D (d, h, t).
    CUtensorMap tm_q, tm_k, tm_v, tm_o;
    Geometry g;
    void* o;                  // O (I/O dtype)
    float* lse;               // LSE, natural log, fp32 (backward's layout)
    const float* sink;        // [h_q] or null
    int64_t o_stride[3];
    int64_t n_q_tiles;        // q-tiles per sequence slot
    float scale_log2;         // scale * log2(e)
    int32_t* status;          // device status word (timeouts)
    int64_t timeout_ns;
};

// Launchers (defined next to their kernels). Return the launch error.
cudaError_t launch_preprocess(const PreArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_dq_convert(const CvtArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_main(const MainArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_fwd(const FwdArgs& a, int dtype, cudaStream_t s);

}  // namespace swa
