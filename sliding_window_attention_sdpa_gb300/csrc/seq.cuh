// seq.cuh -- per-sequence geometry on the device: where a sequence's rows
// live (BSHD batch slot or THD token slot), its actual lengths, and the
// bottom-right diagonal shift. Lengths larger than the slot are clamped to it
// and reported through the status word.
#pragma once

#include "sdpa_internal.h"

namespace swa {

struct SeqInfo {
    int64_t q_row0, kv_row0;   // first row of the slot in the packed row space
    int64_t slot_q, slot_kv;   // rows in the slot
    int64_t len_q, len_kv;     // actual lengths (<= slot)
    int64_t diag;              // anchor(i) = i + diag
    bool bad;                  // a length exceeded its slot (clamped)
};

__device__ __forceinline__ SeqInfo seq_info(const Geometry& g, int64_t bi)
{
    SeqInfo s;
    if (g.layout == 1) {
        s.q_row0 = g.q_offsets[bi];
        s.kv_row0 = g.kv_offsets[bi];
        s.slot_q = g.q_offsets[bi + 1] - s.q_row0;
        s.slot_kv = g.kv_offsets[bi + 1] - s.kv_row0;
    } else {
        s.q_row0 = bi * g.s_q;
        s.kv_row0 = bi * g.s_kv;
        s.slot_q = g.s_q;
        s.slot_kv = g.s_kv;
    }
    s.len_q = g.seq_q_lens ? g.seq_q_lens[bi] : s.slot_q;
    s.len_kv = g.seq_kv_lens ? g.seq_kv_lens[bi] : s.slot_kv;
    s.bad = s.len_q < 0 || s.len_kv < 0 || s.len_q > s.slot_q || s.len_kv > s.slot_kv ||
            s.slot_q < 0 || s.slot_kv < 0 || s.slot_q > g.s_q || s.slot_kv > g.s_kv;
    s.len_q = s.len_q < 0 ? 0 : (s.len_q > s.slot_q ? s.slot_q : s.len_q);
    s.len_kv = s.len_kv < 0 ? 0 : (s.len_kv > s.slot_kv ? s.slot_kv : s.len_kv);
    s.diag = g.mask_mode == 2 ? s.len_kv - s.len_q : 0;
    return s;
}

// Sequence holding packed q row `row` (THD: largest bi with offsets[bi] <= row).
__device__ __forceinline__ int64_t q_row_seq(const Geometry& g, int64_t row)
{
    if (g.layout != 1) return row / g.s_q;
    int64_t lo = 0, hi = g.b;
    while (hi - lo > 1) {
        const int64_t mid = (lo + hi) >> 1;
        if (g.q_offsets[mid] <= row) lo = mid; else hi = mid;
    }
    return lo;
}

// Element offset of (packed row, head) for a tensor with strides
// (batch, sequence/token, head); BSHD rows are split back into (bi, i).
__device__ __forceinline__ int64_t elem_offset(const Geometry& g, const int64_t* st, int64_t row,
                                               int64_t seq_len_max, int64_t head)
{
    if (g.layout == 1) return row * st[1] + head * st[2];
    const int64_t bi = row / seq_len_max, i = row - bi * seq_len_max;
    return bi * st[0] + i * st[1] + head * st[2];
}

// Index of the per-row statistic (LSE, D) of q-head h at packed q row `row`.
__device__ __forceinline__ int64_t stat_offset(const Geometry& g, int64_t row, int64_t h)
{
    if (g.layout == 1) return h * g.rows_q + row;
    const int64_t bi = row / g.s_q, i = row - bi * g.s_q;
    return (bi * g.h_q + h) * g.s_q + i;
}

__device__ __forceinline__ void set_status(int32_t* status, int code)
{
    atomicCAS(status, 0, code);
}

// Range-checked build (-DSDPA_DEBUG_BOUNDS): true if elements [p, p + count)
// lie inside [base, base + extent); otherwise records kStatusBounds and
// returns false so that the caller skips the access. Always true otherwise.
template <typename T>
__device__ __forceinline__ bool in_bounds(int32_t* status, const T* p, const void* base, int64_t extent,
                                          int64_t count)
{
#ifdef SDPA_DEBUG_BOUNDS
    const int64_t off = p - static_cast<const T*>(base);
    if (off < 0 || off + count > extent) {
        set_status(status, kStatusBounds);
        return false;
    }
#else
    (void)status; (void)p; (void)base; (void)extent; (void)count;
#endif
    return true;
}

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }

__host__ __device__ __forceinline__ int64_t fdiv(int64_t a, int64_t b)
{
    int64_t q = a / b;
    if ((a % b != 0) && ((a < 0) != (b < 0))) --q;
    return q;
}

// q-tile range [lo, hi) swept by kv-tile t of a sequence: lo is the first
// q-tile holding a row that reaches the tile's first key (right bound), hi the
// clamp ceil((kv_end + W - diag) / tile_q) with kv_end the tile's last key + 1
// (cuDNN-frontend PR #866, "Change"). Host-callable: the launcher uses it to
// tell whether the dQ convert kernel has anything to do.
__host__ __device__ __forceinline__ void q_tile_range(const Geometry& g, const SeqInfo& s, int64_t t,
                                             int64_t& lo, int64_t& hi)
{
    const int64_t kv_base = t * kTileKV;
    const int64_t n_q = (s.len_q + kTileQ - 1) / kTileQ;
    lo = 0;
    hi = n_q;
    if (kv_base >= s.len_kv || n_q == 0) {
        hi = 0;
        return;
    }
    const int64_t kv_end = imin64(kv_base + kTileKV, s.len_kv);
    if (g.right >= 0) {
        const int64_t first = kv_base - g.right - s.diag;
        lo = first > 0 ? first / kTileQ : 0;
    }
    if (g.window_left >= 0) {
        const int64_t c = fdiv(kv_end + g.window_left - s.diag + kTileQ - 1, kTileQ);
        if (c < hi) hi = c;
    }
    if (hi < lo) hi = lo;
}

// The kv-tiles that sweep q-tile j: the contiguous run [first, first + count)
// (both bounds of q_tile_range are non-decreasing in t). `first` is the relay's
// kv_first = max((q_row0 + diag - W) // tile_kv, 0) (PR #866, "Change"), or 0
// without a left window.
__host__ __device__ __forceinline__ void q_tile_visitors(const Geometry& g, const SeqInfo& s, int64_t j,
                                                int64_t& first, int64_t& count)
{
    const int64_t n_kv = (s.len_kv + kTileKV - 1) / kTileKV;
    first = 0;
    count = 0;
    if (n_kv == 0 || j * kTileQ >= s.len_q) return;
    if (g.window_left >= 0) first = imax64(fdiv(j * kTileQ + s.diag - g.window_left, kTileKV), 0);
    int64_t last = n_kv - 1;
    if (g.right >= 0) last = imin64(last, fdiv((j + 1) * kTileQ + g.right + s.diag - 1, kTileKV));
    if (last < first) return;
    int64_t lo, hi;
    q_tile_range(g, s, first, lo, hi);
    if (!(lo <= j && j < hi)) return;
    count = last - first + 1;
}

}  // namespace swa
