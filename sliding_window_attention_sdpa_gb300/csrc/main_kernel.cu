// main_kernel.cu -- fused sliding-window SDPA backward on sm_103a tensor cores.
//
// Work item = (kv-tile t, kv-head g, sequence b). A persistent CTA (one per SM)
// walks its items; for each it keeps the kv-tile's K and V in shared memory and,
// for every q-head of g's group in turn, sweeps the q-tiles in the
// window-clamped range [q_lo, q_hi) (cuDNN-frontend PR #866, "Change": no query
// with anchor > kv_base + tile_kv - 1 + W reaches the tile) from the top down,
// issuing the five contractions as tcgen05.mma with fp32 accumulators in tensor
// memory (TMEM). dK and dV accumulate over the whole group in TMEM (the GQA
// reduction of PR #557, in head order) and are stored once per item:
//
//   S^T  = K Q^T     [kv x q]  cols   0..127
//   dP^T = V dO^T    [kv x q]  cols 128..255
//   dV  += P^T dO    [kv x d]  cols 256..      (d = 64: P^T read from TMEM)
//   dK  += dS^T Q    [kv x d]  cols 256+d..
//   dQ   = dS K      [q x d]   cols 384.. (d = 64) or aliasing S^T (d = 128)
//   P^T (16-bit)     [kv x q]  cols 448..511 (d = 64; two q per column)
//
// Warp roles (512 threads):
//   warp 0      TMA producer: K, V per item; Q, dO per q-tile into a ring of
//               kStages stages (128-byte swizzle, zero fill past the tensor),
//               each with the q-tile's per-row (LSE log2, D) pairs (1 KB bulk copy)
//   warp 1      MMA issuer (lane 0 of the converged warp) and TMEM owner. At
//               d = 64 it issues the next q-tile's S^T/dP^T ahead of this
//               q-tile's dV/dK/dQ, so the softmax of one q-tile overlaps the
//               gradient contractions of the previous one (dS^T double-buffered)
//   warps 2-3   idle
//   warps 4-11  softmax: two warps per TMEM sub-partition, each thread one kv
//               row (TMEM lane) and one 64-column half of the q-tile; recomputes
//               P = exp2(S*scale*log2e - LSE*log2e) and dS = P (dP - D) with the
//               mask, skipping 16-column chunks the window masks for the whole
//               warp; writes P^T / dS^T as swizzled 16-bit tiles; at the end of
//               an item one half writes dV, the other dK, through a staged tile
//   warps 12-15 dQ: one thread per q row reads dQ from TMEM into a staged fp32
//               tile, from which the group writes whole rows: converted, stored
//               as the first partial sum, or added to the accumulator (vector
//               atomics, or in order along the relay)
// Hand-offs are mbarriers; every wait is bounded (status word on timeout).
//
// Shared-memory operand layout: rows of 64 16-bit elements (128 B), 8-row
// atoms of 1024 B, 16-byte chunk c of row r at chunk position c ^ (r % 8)
// (the TMA 128-byte swizzle); 64-column blocks of a 128-row tile 16 KB apart.
// One buffer serves as a K-major operand or, through another descriptor, as an
// MN-major one.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>
#include <vector>

#include "ptx.cuh"
#include "sdpa_internal.h"
#include "seq.cuh"

namespace swa {

namespace {

constexpr int kThreads = 512;
// The item table is used when a CTA has at most this many items.
constexpr int64_t kItemTableMaxPerCta = 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBlock16K = 128 * 128;  // one 64-column block of a 128-row tile
constexpr float kLog2e = 1.4426950408889634f;

// warp roles
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpSoft0 = 4, kWarpDq0 = 12;
constexpr int kSoftThreads = 256;
constexpr int kBarDq = 1, kBarSoft = 2;  // named barriers of the two 128-thread groups

template <int HD>
struct Cfg {
    static constexpr int kStages = HD == 64 ? 2 : 1;    // Q/dO/LSE/D ring
    static constexpr int kKvStages = HD == 64 ? 2 : 1;  // K/V ring (per work item)
    // d = 64: the next q-tile's S^T/dP^T contractions are issued ahead of this
    // q-tile's gradient contractions, so that the softmax runs while the tensor
    // core works; dS^T is double-buffered for it. Both rings must hold two
    // entries, or the look-ahead would wait on a buffer it has yet to release.
    static constexpr bool kAhead = HD == 64;
    static constexpr int kDsBufs = kAhead ? 2 : 1;
    static_assert(!kAhead || (kStages >= 2 && kKvStages >= 2), "look-ahead needs two ring entries");
    static constexpr uint32_t kTile = 128 * HD * 2;
    // shared memory offsets (from a 1024-aligned base)
    static constexpr uint32_t kK = 0;                           // kKvStages tiles
    static constexpr uint32_t kV = kK + kKvStages * kTile;      // kKvStages tiles
    static constexpr uint32_t kQ = kV + kKvStages * kTile;      // kStages tiles
    static constexpr uint32_t kDO = kQ + kStages * kTile;       // kStages tiles
    // P^T is kept in TMEM (the A operand of dV). At d = 128 a 32 KB region at kP
    // holds half of the dK/dV epilogue's staging (the dS^T buffer the other)
    // and, during the dQ warps' turn, half of a stored dQ partial.
    static constexpr uint32_t kP = kDO + kStages * kTile;
    static constexpr uint32_t kDS = kP + (HD == 64 ? 0 : 32768); // kDsBufs x dS^T [128 kv x 128 q]
    // dQ staging: 128 rows x 64 fp32 (two 16 KB blocks of 32 columns; the whole
    // row at d = 64, half of it at d = 128), or the whole 16-bit dQ tile
    static constexpr int kDqCols = 64;
    static constexpr uint32_t kDqStage = kDS + kDsBufs * 32768;
    static constexpr uint32_t kStat = kDqStage + 128 * kDqCols * 4;  // kStages x (128 -LSE log2, 128 -D)
    static constexpr uint32_t kBars = kStat + kStages * 1024;   // mbarriers
    static constexpr uint32_t kMisc = kBars + 256;              // tmem slot, flags, deferred epilogue
    static constexpr uint32_t kBytes = kMisc + 128;
    static_assert(kBytes <= 232448, "shared memory above the 227 KB a CTA may opt into");
    // The dK/dV epilogue stages two 128 x HD 16-bit tiles (2 x 16 KB at d = 64,
    // 2 x 32 KB at d = 128) in the item's K/V ring entry (d = 64) or in the
    // region at kP and the dS^T buffer (d = 128), all idle once the work item's
    // contractions are done.
    static_assert(HD == 64 ? 2 * 128 * HD * 2 <= 32768 : (kDS == kP + 32768 && 2 * 128 * HD * 2 <= 65536),
                  "epilogue staging does not fit");
    // TMEM columns
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + HD;
    static constexpr uint32_t kColDQ = HD == 64 ? 384 : 0;
    // P^T's TMEM column for 16-bit chunk sc (q columns 16 sc .. 16 sc + 15, two
    // to a column): at d = 64 its own columns 448-511; at d = 128 over the dP^T
    // columns already read by the warp that writes it (the half of the q-tile
    // at column 64 h goes to dP^T's columns 128 + 64 h ..., which hold its
    // chunks 4 h, 4 h + 1 and are read before chunk 4 h + 2 is written)
    static constexpr uint32_t kColP = 448;
    static __host__ __device__ constexpr uint32_t p_col(int sc)
    {
        return HD == 64 ? kColP + 8u * sc : 128u + 64u * (sc >> 2) + 8u * (sc & 3);
    }
    static constexpr bool kDqAliasesS = HD != 64;
    // d = 64: the dQ warps write each item's dK/dV, staged in the item's own
    // K/V ring entry (idle once its last contractions are done), and hand the
    // entry back to the producer when their stores have read it. The softmax
    // group then runs its q-tiles back to back across items. At d = 128 the
    // softmax group writes them, staged in the region at kP and its dS^T buffer.
    static constexpr bool kEpiDq = HD == 64;
    static_assert(!(kAhead && kDqAliasesS), "look-ahead overwrites S^T while dQ would alias it");
};

// mbarrier indices
enum Bar : int {
    kSFull = 0, kPFull, kPEmpty, kDqFull, kDqEmpty, kAccFull, kAccEmpty,
    kQFull0, kQFull1, kQEmpty0, kQEmpty1, kKvFull0, kKvFull1, kKvEmpty0, kKvEmpty1, kDqLoad, kDrain,
    kDqLoad1,   // d = 128: the second half of a stored dQ partial (kDqLoad: the first)
    kNumBars
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    uint32_t r;
    if constexpr (BF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t swz(int r, int chunk)
{
    return static_cast<uint32_t>((chunk >> 3) * kBlock16K + (r >> 3) * 1024 + (r & 7) * 128 +
                                 (((chunk & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Shared -> global tensor copies (bulk-group completion): a plain store, or an
// element-wise add into global memory performed at L2 (fp32 maps only here).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2, int c3)
{
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void tma_add_4d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2, int c3)
{
    asm volatile("cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

__device__ __forceinline__ void tma_add_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2)
{
    asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// One 128-row box of a [., h, d] tensor map at column c0 of head h: BSHD maps
// are 4-D (d, h, s, b), THD maps 3-D (d, h, t); `row` is s (BSHD) or t (THD).
__device__ __forceinline__ void tma_put(bool add, bool thd, const CUtensorMap* map, uint32_t src, int c0, int h,
                                        int row, int b)
{
    if (add) {
        if (thd) tma_add_3d(map, src, c0, h, row);
        else tma_add_4d(map, src, c0, h, row, b);
    } else {
        if (thd) tma_store_3d(map, src, c0, h, row);
        else tma_store_4d(map, src, c0, h, row, b);
    }
}

// Byte offset of 16-byte chunk c of row r in a staged tile of 128-byte rows:
// blocks of 128 rows x 128 B (8 chunks), chunk c & 7 at position (c & 7) ^ (r % 8)
// -- the layout a TMA 128-byte-swizzle box of 128 rows reads from shared memory.
__device__ __forceinline__ uint32_t stg_off(int r, int c)
{
    return static_cast<uint32_t>((c >> 3) * kBlock16K + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// One 128-row box of a head-strided tensor map at column c0 (see tma_put).
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, uint32_t bar, bool thd, int c0,
                                        int head, int row, int batch)
{
    if (thd) tma_load_3d(dst, map, bar, c0, head, row);
    else tma_load_4d(dst, map, bar, c0, head, row, batch);
}

// Starts moving one box of a tensor map (coordinates as for tma_box) into L2.
// Nothing completes or is waited for: later loads of those rows find them in L2.
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap* map, bool thd, int c0, int head, int row, int batch)
{
    if (thd)
        asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                         reinterpret_cast<uint64_t>(map)),
                     "r"(c0), "r"(head), "r"(row)
                     : "memory");
    else
        asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                         reinterpret_cast<uint64_t>(map)),
                     "r"(c0), "r"(head), "r"(row), "r"(batch)
                     : "memory");
}

// Loads rows [row, row + 128) of one head of a [., HD] tensor into a swizzled tile
// (HD/64 boxes of 64 columns). BSHD maps are 4-D (d, h, s, b); THD maps 3-D (d, h, t).
template <int HD>
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                         bool thd, int head, int row, int batch)
{
#pragma unroll
    for (int cb = 0; cb < HD / 64; ++cb) {
        if (thd) tma_load_3d(dst + cb * kBlock16K, map, bar, cb * 64, head, row);
        else tma_load_4d(dst + cb * kBlock16K, map, bar, cb * 64, head, row, batch);
    }
}

// Starts moving the 128-byte line holding `p` into this SM's L1.
__device__ __forceinline__ void prefetch_l1(const void* p)
{
    asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

__device__ __forceinline__ void named_bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Barrier over `count` threads (named barrier `id`) returning the AND of `v`.
__device__ __forceinline__ bool bar_and(int id, int count, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Barrier over `count` threads (named barrier `id`) returning the OR of `v`.
__device__ __forceinline__ bool bar_or(int id, int count, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Optional timeline trace (build with -DSDPA_BWD_TRACE): SM clock stamps of each
// role's hand-offs for the first kTraceCtas CTAs and kTraceTiles q-tiles, written
// to the workspace at byte offset kTraceOffset (the caller sizes the workspace
// for it). Off by default; it records and changes nothing else.
constexpr int kTraceCtas = 8, kTraceTiles = 64, kTraceSlots = 24;
constexpr size_t kTraceOffset = size_t(256) << 20;
#ifdef SDPA_BWD_TRACE
#define SWA_TRACE(slot, tile)                                                                    \
    do {                                                                                         \
        if (blockIdx.x < kTraceCtas && (tile) < kTraceTiles)                                     \
            reinterpret_cast<uint64_t*>(reinterpret_cast<char*>(a.status) + kTraceOffset)       \
                [(blockIdx.x * kTraceTiles + (tile)) * kTraceSlots + (slot)] = clock64();         \
    } while (0)
#else
#define SWA_TRACE(slot, tile) do { } while (0)
#endif

struct Item {
    int64_t t, bi, gk;
    int64_t h0, group;   // q-heads [h0, h0 + group) share kv-head gk
    SeqInfo s;
    int64_t kv_base, q_lo, q_hi;
    int64_t nq, steps;   // q-tiles per head, steps = group * nq
    bool has_work;       // at least one q-tile to sweep
    bool in_slot;        // the kv-tile has rows inside the sequence's slot
    // strip mode: tmem_pair() of the first and the last step (the only steps
    // that can pair when a q-tile has at most two visitors), set by with_pairs
    uint8_t tp_first, tp_last;
    // Steps run q-head h0 .. h0 + group - 1, each over its q-tiles from q_hi - 1
    // down to q_lo, or (strip mode, UP) from q_lo up to q_hi - 1. With QMAJOR
    // (strip mode at d = 64) they run q-tile by q-tile instead, each over every
    // q-head of the group, so that the q-tile this item shares with the next
    // one (its Q and dO rows, and the partial dQ the pair passes on) comes back
    // to the CTA after one q-tile's steps, not a whole item's. (At d = 128 that
    // order bunches the steps that add a partial, whose dQ turn holds S^T's
    // columns, and was slower.) Counters rather than divisions (there is no
    // 64-bit divider, and these sit on every role's hand-off path).
    template <bool UP>
    __device__ __forceinline__ int64_t first_j() const { return UP ? q_lo : q_hi - 1; }
    template <bool UP, bool QMAJOR = false>
    __device__ __forceinline__ void advance(int64_t& j, int64_t& hh) const
    {
        if constexpr (UP && QMAJOR) {
            if (hh == h0 + group - 1) {
                hh = h0;
                ++j;
            } else {
                ++hh;
            }
        } else if constexpr (UP) {
            if (j == q_hi - 1) {
                j = q_lo;
                ++hh;
            } else {
                ++j;
            }
        } else if (j == q_lo) {
            j = q_hi - 1;
            ++hh;
        } else {
            --j;
        }
    }
};

static_assert(sizeof(Item) == kItemBytes, "the host sizes the item table with kItemBytes");

// One work item's dK/dV store, as the softmax group runs it (d = 64 defers it
// to after the next item's first q-tile, keeping it in shared memory).
struct Epi {
    int64_t kv_base, kv_row0, len_kv, slot_kv, bi, gk;
    uint32_t acc_par;   // parity of the item's acc-full phase
    int32_t buf;        // dS^T buffer to stage in (d = 64)
    int32_t have;       // TMEM holds the item's dK/dV (else the rows are zero)
    int32_t last;       // the item's last step (trace index)
};

// Per-launch constants of the item numbering (32-bit: the host keeps the item
// count below 2^31).
struct ItemCounts {
    uint32_t h_kv, n_kv_tiles, group, b;
};

// The work items a CTA walks: begin, begin + stride, ... below end.
//  - Round-robin (STRIP false): items numbered head-fastest, CTA c takes
//    c, c + grid, ... The CTAs running at one time then cover all kv-heads of
//    a few kv-tiles; in the [row][head][d] tensors one head is a narrow column
//    of every row, so numbering them kv-tile fastest under this walk (all CTAs
//    on one head) concentrates their loads and stores on a few memory
//    partitions. The previous kv-tile of the same head (the dQ relay partner)
//    is item - h_kv, which runs in the same wave.
//  - Strip mode: items numbered (kv-head, sequence, kv-tile), kv-tile
//    fastest. Groups of G consecutive kv-heads (G chosen by the launcher so
//    that the grid fills the SMs: 16 kv-heads on 152 SMs take G = 2, 19 runs
//    per group) share R contiguous runs of their items, equal in items, or
//    (sequences of different lengths) in kv-tiles that hold keys; CTA c walks
//    group c % (h_kv / G) over run c / (h_kv / G). The two kv-tiles visiting
//    a q-tile are then consecutive items of one CTA except where a run ends.
//    A run may cross from one kv-head or sequence into the next: no q-tile
//    has visitors on both sides of such a boundary (a sequence's first
//    kv-tile is the first visitor of each of its q-tiles), so no pair is
//    formed across it. The CTAs on one run index read the same token rows of
//    every group at about the same time, as the round-robin walk does.
struct Walk {
    int64_t begin, end, stride;
};

// The round-robin walk's item order, set by the host when it knows every item's
// steps (BSHD, no length arrays): items go out longest first, each to the CTA
// with the fewest steps so far, and each CTA takes its own in ascending number,
// so that a relay partner (the kv-tile before, a lower number) is never behind
// the item that waits for it. Without one (NoOrder, the kernel instance
// whose parameter it is), CTA c takes c, c + grid, ...
constexpr int kOrderMaxItems = 4096, kOrderMaxCtas = 256;
struct ItemOrder {
    uint16_t off[kOrderMaxCtas + 1];      // CTA c takes item[off[c]] .. item[off[c + 1] - 1]
    uint16_t item[kOrderMaxItems];
};
struct NoOrder {};

// Strip mode with sequences of different lengths (packed, or length arrays):
// the offset, inside a group's items, of run boundary `run` of `runs`, placed
// so that each run holds an equal share of the kv-tiles that hold keys
// (ceil(len_kv / 128) per sequence and kv-head). Items past a sequence's keys
// (slot padding, dK/dV zero-fill only) go with the run before them. With
// equal shares of items instead, a run over long sequences held all their
// work and one over short ones little. -1 if no sequence holds keys.
__device__ __forceinline__ int64_t work_boundary(const Geometry& g, int64_t n_kv_tiles, int64_t group_heads,
                                                 int64_t run, int64_t runs)
{
    auto tiles = [&](int64_t bi) -> int64_t {
        const int64_t t = (seq_info(g, bi).len_kv + kTileKV - 1) / kTileKV;
        return t < n_kv_tiles ? t : n_kv_tiles;
    };
    int64_t per_head = 0;
    for (int64_t bi = 0; bi < g.b; ++bi) per_head += tiles(bi);
    if (per_head == 0) return -1;
    const int64_t total = per_head * group_heads;
    if (run <= 0) return 0;
    if (run >= runs) return group_heads * g.b * n_kv_tiles;
    const int64_t target = total * run / runs;   // working tiles before the boundary
    const int64_t head = target / per_head;
    int64_t rem = target - head * per_head;
    for (int64_t bi = 0; bi < g.b; ++bi) {
        const int64_t t = tiles(bi);
        if (rem < t) return (head * g.b + bi) * n_kv_tiles + rem;
        rem -= t;
    }
    return (head + 1) * g.b * n_kv_tiles;   // not reached
}

template <bool STRIP>
__device__ __forceinline__ Walk item_walk(const Geometry& g, int64_t n_items, int64_t n_kv_tiles, int64_t group_heads)
{
    if constexpr (STRIP) {
        // groups of group_heads consecutive kv-heads share R runs: CTA c walks
        // group c % (h_kv / group_heads) over the (c / ...)-th run of its items
        const int64_t n_groups = g.h_kv / group_heads;
        const int64_t runs = gridDim.x / n_groups, grp = blockIdx.x % n_groups, run = blockIdx.x / n_groups;
        const int64_t per_group = n_items / g.h_kv * group_heads;
        if ((g.layout == 1 || g.seq_kv_lens != nullptr) && g.b <= 256) {
            const int64_t lo = work_boundary(g, n_kv_tiles, group_heads, run, runs);
            if (lo >= 0)
                return Walk{grp * per_group + lo, grp * per_group + work_boundary(g, n_kv_tiles, group_heads,
                                                                                  run + 1, runs), 1};
        }
        return Walk{grp * per_group + per_group * run / runs, grp * per_group + per_group * (run + 1) / runs, 1};
    }
    return Walk{static_cast<int64_t>(blockIdx.x), n_items, static_cast<int64_t>(gridDim.x)};
}

template <bool STRIP>
__device__ __forceinline__ Item decode(const MainArgs& a, const ItemCounts& n, int64_t item)
{
    const Geometry& g = a.g;
    Item it;
    const uint32_t u = static_cast<uint32_t>(item);
    if constexpr (STRIP) {
        const uint32_t rest = u / n.n_kv_tiles, gq = rest / n.b;
        it.t = u - rest * n.n_kv_tiles;
        it.bi = rest - gq * n.b;
        it.gk = gq;
    } else {
        const uint32_t rest = u / n.h_kv, bq = rest / n.n_kv_tiles;
        it.gk = u - rest * n.h_kv;
        it.t = rest - bq * n.n_kv_tiles;
        it.bi = bq;
    }
    it.group = n.group;
    it.h0 = it.gk * it.group;
    it.s = seq_info(g, it.bi);
    it.kv_base = it.t * kTileKV;
    q_tile_range(g, it.s, it.t, it.q_lo, it.q_hi);
    it.nq = it.q_hi - it.q_lo;
    it.steps = it.nq > 0 ? it.nq * it.group : 0;
    it.in_slot = it.kv_base < it.s.slot_kv;
    it.has_work = it.nq > 0 && it.in_slot;
    return it;
}

// Strip mode with one q-head per kv-head: a q-tile visited by kv-tiles t and
// t + 1 that are consecutive items of this CTA is the last step of t and the
// first of t + 1, so the second dQ contraction accumulates onto the first in
// tensor memory and only the sum is read. Returns 1 for the first of such a
// pair (its dQ is not read), 2 for the second (it reads the sum), else 0.
template <bool STRIP>
__device__ __forceinline__ int tmem_pair(const Geometry& g, const Item& it, int64_t j, int64_t item, const Walk& wk)
{
    if constexpr (!STRIP) {
        return 0;
    } else {
        if (it.group != 1) return 0;
        int64_t first, nvis;
        q_tile_visitors(g, it.s, j, first, nvis);
        if (nvis != 2) return 0;
        const int turn = static_cast<int>(it.t - first);
        const bool local = turn == 0 ? item + 1 < wk.end : item > wk.begin;
        return local ? 1 + turn : 0;
    }
}

// An item with its first and last steps' tmem_pair() filled in (once per
// item, instead of the visitor arithmetic at every step of the MMA warp).
template <bool STRIP>
__device__ __forceinline__ Item with_pairs(const Geometry& g, Item it, int64_t item, const Walk& wk)
{
    it.tp_first = it.tp_last = 0;
    if (STRIP && it.has_work && it.group == 1) {
        it.tp_first = static_cast<uint8_t>(tmem_pair<STRIP>(g, it, it.template first_j<STRIP>(), item, wk));
        it.tp_last = static_cast<uint8_t>(tmem_pair<STRIP>(g, it, STRIP ? it.q_hi - 1 : it.q_lo, item, wk));
    }
    return it;
}

// Zeroes rows [nvalid, 128) of a swizzled tile (whole 128-byte rows, so the
// swizzle does not matter); run by one warp, then made visible to the tensor
// core. Used where rows past a sequence end hold data of another sequence
// or padding (TMA fills only past the tensor's extent).
template <int HD>
__device__ __forceinline__ void zero_tail(uint8_t* tile, int64_t nvalid, int lane)
{
    const int first = nvalid < 0 ? 0 : static_cast<int>(nvalid);
    if (first >= 128) return;
#pragma unroll
    for (int cb = 0; cb < HD / 64; ++cb) {
        uint4* p = reinterpret_cast<uint4*>(tile + cb * kBlock16K + first * 128);
        const int n16 = (128 - first) * 8;
        for (int k = lane; k < n16; k += 32) p[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    __syncwarp();
}

}  // namespace

__device__ __forceinline__ int64_t ord_off(const ItemOrder& o, unsigned c) { return o.off[c]; }
__device__ __forceinline__ int64_t ord_off(const NoOrder&, unsigned) { return 0; }
__device__ __forceinline__ int64_t ord_item(const ItemOrder& o, int64_t i) { return o.item[i]; }
__device__ __forceinline__ int64_t ord_item(const NoOrder&, int64_t i) { return i; }

// A global-memory wait (relay turn, split pair) that ran out: marks the CTA
// aborted and records the status and which wait it was (out of line: cold).
__device__ __noinline__ bool gave_up(int32_t* status, volatile uint32_t* abort_flag, int where)
{
    *abort_flag = 1;
    set_status(status, kStatusTimeout);
    set_status(status + 1, where);
    return false;
}

template <int HD, bool BF16, bool STRIP, bool ORDER>
__global__ void __launch_bounds__(kThreads, 1)
    sdpa_bwd_main_kernel(const __grid_constant__ MainArgs a,
                         const __grid_constant__ std::conditional_t<ORDER, ItemOrder, NoOrder> ord)
{
    static_assert(!(STRIP && ORDER), "the strip walk sets its own order");
    using C = Cfg<HD>;
    // The 128-byte-swizzled operand tiles need a 1024-byte aligned base; the
    // dynamic shared memory is declared so, and checked rather than padded
    // (the layout leaves no room for the padding at d = 64).
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        grid_dep_wait();   // the preprocess zeroes the status word
        if (threadIdx.x == 0) set_status(a.status, kStatusUnsupported);
        return;
    }
    uint8_t* sm = smem_raw;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bars = sbase + C::kBars;
    auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::kMisc);  // [0] tmem base, [1] abort flag

    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint64_t tmo = static_cast<uint64_t>(a.timeout_ns);
    const int64_t n_items = g.b * g.h_kv * a.n_kv_tiles;
    const bool thd = g.layout == 1;
    const ItemCounts cnt{static_cast<uint32_t>(g.h_kv), static_cast<uint32_t>(a.n_kv_tiles),
                         static_cast<uint32_t>(g.h_q / g.h_kv), static_cast<uint32_t>(g.b)};
    const Walk wk = ORDER ? Walk{ord_off(ord, blockIdx.x), ord_off(ord, blockIdx.x + 1), 1}
                          : item_walk<STRIP>(g, n_items, a.n_kv_tiles, a.strip > 0 ? a.strip : 1);
    // item number at walk position i (the same unless the host set an order)
    auto item_no = [&](int64_t i) -> int64_t { return ord_item(ord, i); };

    if (tid == 0) {
        misc[1] = 0;
        for (int s = 0; s < C::kKvStages; ++s) {
            mbar_init(bar(kKvFull0 + s), 1);
            mbar_init(bar(kKvEmpty0 + s), 1);
        }
        mbar_init(bar(kSFull), 1);
        mbar_init(bar(kPFull), kSoftThreads);
        mbar_init(bar(kPEmpty), 1);
        mbar_init(bar(kDqFull), 1);
        mbar_init(bar(kDqEmpty), 128);
        mbar_init(bar(kAccFull), 1);
        mbar_init(bar(kAccEmpty), C::kEpiDq ? 128 : kSoftThreads);
        mbar_init(bar(kDqLoad), 1);
        mbar_init(bar(kDqLoad1), 1);
        mbar_init(bar(kDrain), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(kQFull0 + s), 1);
            mbar_init(bar(kQEmpty0 + s), 1);
        }
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(sbase + C::kMisc, kTmemCols);
        tmem_relinquish();
    }
    // d = 64 with few items per CTA (the launcher sets use_items): every item
    // of this CTA is decoded once, by all threads in parallel, into the item
    // table, and the roles read their items from it. Decoding in each role at
    // each item boundary ran as cold code on the critical path (about 1 K
    // cycles per item on the softmax warps), and an item has only a few q-tile
    // steps there. With many items per CTA, and at d = 128 (no look-ahead,
    // more registers live), the roles decode in place: there the table was
    // slower.
    Item* items = static_cast<Item*>(a.items);
    const bool use_items = C::kAhead && a.use_items != 0;
    // Strip mode pairs a q-tile's two dQ contractions in tensor memory only
    // where dQ has columns of its own (d = 64); at d = 128 it aliases S^T,
    // which the next step overwrites, so the pair goes through the
    // accumulator rows instead.
    constexpr bool kTmemPairs = STRIP && !C::kDqAliasesS;
    constexpr bool kQMajor = STRIP && !C::kDqAliasesS;   // the step order within an item (Item::advance)
    if (use_items)
        for (int64_t item = wk.begin + static_cast<int64_t>(tid) * wk.stride; item < wk.end;
             item += static_cast<int64_t>(kThreads) * wk.stride)
            items[item] = with_pairs<kTmemPairs>(g, decode<STRIP>(a, cnt, item_no(item)), item, wk);
    auto item_at = [&](int64_t i) -> Item { return use_items ? items[i] : decode<STRIP>(a, cnt, item_no(i)); };
    tc_fence_before();
    __syncthreads();   // also publishes the item table to the CTA
    tc_fence_after();
    // Everything above reads only the caller's inputs; from here on the roles
    // read the preprocess's statistics, counters and status word. With
    // programmatic stream serialization the prologue above overlapped the
    // preprocess's last blocks and this launch's own latency.
    grid_dep_wait();
    grid_dep_launch();
    const uint32_t tmem = misc[0];
    volatile uint32_t* abort_flag = misc + 1;

    // A wait that gives up marks the CTA aborted; later waits of every role
    // return at once so that the kernel drains and frees TMEM.
    auto wait = [&](int b, uint32_t parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait(bar(b), parity, tmo)) return true;
        *abort_flag = 1;
        set_status(a.status, kStatusTimeout);
        return false;
    };
    auto wait_warp = [&](int b, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait(b, parity));
    };
    auto wait_group = [&](int id, int count, int b, uint32_t parity) -> bool {
        return bar_and(id, count, wait(b, parity));
    };

    // Register split at d = 64 (the launch gives each thread 128 registers, the
    // whole register file). With 128 each the dQ role spilled, and the dQ warps
    // (dQ, and each item's dK/dV epilogue) pace the MMA warp through DqEmpty
    // and AccEmpty. The producer, MMA and idle warps give 16 each to the dQ
    // warps: x + 128 + 128 + y = 512 per lane of the four warpgroups, x = 112,
    // y = 144. Main kernel: headline 93 -> 90 us, W512 621 -> 592 us,
    // non-square W8000 506 -> 474 us. At d = 128 the same split made the
    // b12 h48/6 S16484 case 5% slower, so that kernel keeps 128 everywhere.
    if (warp == kWarpTma) {
        if constexpr (C::kAhead) asm volatile("setmaxnreg.dec.sync.aligned.u32 112;");
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kv_it = 0, q_it = 0;
            for (int64_t item = wk.begin; item < wk.end; item += wk.stride) {
                const Item it = item_at(item);
                if (use_items) {
                    // The next two items' records toward this SM's L1, ahead of
                    // the roles' reads (every role reaches them after this warp).
                    for (int64_t nx = item + wk.stride; nx < wk.end && nx <= item + 2 * wk.stride; nx += wk.stride) {
                        const char* rec = reinterpret_cast<const char*>(items + nx);
                        prefetch_l1(rec);
                        prefetch_l1(rec + kItemBytes / 2);
                        prefetch_l1(rec + kItemBytes - 1);
                    }
                }
                if (!it.has_work) continue;
                const int ks = kv_it % C::kKvStages;
                if (!wait(kKvEmpty0 + ks, ((kv_it / C::kKvStages) & 1) ^ 1)) break;
                ++kv_it;
                const int kvrow = static_cast<int>((thd ? it.s.kv_row0 : 0) + it.kv_base);
                mbar_arrive_expect_tx(bar(kKvFull0 + ks), 2 * C::kTile);
                tma_tile<HD>(sbase + C::kK + ks * C::kTile, &a.tm_k, bar(kKvFull0 + ks), thd,
                             (int)it.gk, kvrow, (int)it.bi);
                tma_tile<HD>(sbase + C::kV + ks * C::kTile, &a.tm_v, bar(kKvFull0 + ks), thd,
                             (int)it.gk, kvrow, (int)it.bi);
                bool ok = true;
                for (int64_t k = 0, j = it.first_j<STRIP>(), hh = it.h0; k < it.steps; ++k, ++q_it, it.template advance<STRIP, kQMajor>(j, hh)) {
                    const int st = q_it % C::kStages;
                    if (!wait(kQEmpty0 + st, ((q_it / C::kStages) & 1) ^ 1)) { ok = false; break; }
                    SWA_TRACE(12, q_it);
                    const int qrow = static_cast<int>((thd ? it.s.q_row0 : 0) + j * kTileQ);
                    mbar_arrive_expect_tx(bar(kQFull0 + st), 2 * C::kTile + 1024);
                    tma_tile<HD>(sbase + C::kQ + st * C::kTile, &a.tm_q, bar(kQFull0 + st), thd,
                                 (int)hh, qrow, (int)it.bi);
                    tma_tile<HD>(sbase + C::kDO + st * C::kTile, &a.tm_do, bar(kQFull0 + st), thd,
                                 (int)hh, qrow, (int)it.bi);
                    const float* srow = a.stats + 2 * ((static_cast<int64_t>(it.bi) * g.h_q + hh) * a.stats_row +
                                                       static_cast<int64_t>(j) * kTileQ);
                    if (in_bounds(a.status, srow, a.stats, g.ext.stats, 2 * kTileQ))
                        bulk_load(sbase + C::kStat + st * 1024, srow, 1024, bar(kQFull0 + st));
                    SWA_TRACE(13, q_it);
                }
                if (!ok) break;
            }
            // After a wait gave up, loads may still be on their way into this
            // CTA's shared memory: wait (bounded) for the last one issued on each
            // ring entry before the CTA can exit (at most one is outstanding per
            // entry; one that the consumer saw complete returns at once).
            for (uint32_t i = kv_it > C::kKvStages ? kv_it - C::kKvStages : 0; i < kv_it; ++i)
                mbar_wait(bar(kKvFull0 + i % C::kKvStages), (i / C::kKvStages) & 1, tmo);
            for (uint32_t i = q_it > C::kStages ? q_it - C::kStages : 0; i < q_it; ++i)
                mbar_wait(bar(kQFull0 + i % C::kStages), (i / C::kStages) & 1, tmo);
        }
    } else if (warp == kWarpMma) {
        if constexpr (C::kAhead) asm volatile("setmaxnreg.dec.sync.aligned.u32 112;");
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t kIdQK = idesc_f16(BF16, 128, 128, false, false);
        constexpr uint32_t kIdPV = idesc_f16(BF16, 128, HD, false, true);
        constexpr uint32_t kIdDQ = idesc_f16(BF16, 128, HD, true, true);
        const uint32_t tm_s = tmem + C::kColS, tm_dp = tmem + C::kColDP;
        const uint32_t tm_dv = tmem + C::kColDV, tm_dk = tmem + C::kColDK, tm_dq = tmem + C::kColDQ;
        uint32_t kv_it = 0, q_it = 0, p_it = 0, dq_it = 0, acc_it = 0;
        // The q-tile step whose gradient contractions (dV, dK, dQ) are not yet
        // issued: they need the softmax's P^T / dS^T of that step.
        struct Pending {
            bool valid, first, last;  // first / last step of its work item
            int st, ks;               // Q/dO and K/V ring entries
            uint32_t q_it;            // step index (selects the dS^T buffer)
            int tpair;                // tmem_pair() of the step
        };
        Pending pend{false, false, false, 0, 0, 0u, 0};
        // Operand descriptors of ring entry 0 and dS^T buffer 0; other entries
        // are a byte offset away (sdesc_at). K-major (16, 1024) for S^T, dP^T
        // and the dK A operand; MN-major (16 KB, 1024) for the B operands of
        // dV, dK and the operands of dQ.
        const uint64_t dK0 = sdesc_sw128(sbase + C::kK, 16, 1024), dV0 = sdesc_sw128(sbase + C::kV, 16, 1024);
        const uint64_t dQ0 = sdesc_sw128(sbase + C::kQ, 16, 1024), dDO0 = sdesc_sw128(sbase + C::kDO, 16, 1024);
        const uint64_t dDOmn0 = sdesc_sw128(sbase + C::kDO, kBlock16K, 1024);
        const uint64_t dQmn0 = sdesc_sw128(sbase + C::kQ, kBlock16K, 1024);
        const uint64_t dKmn0 = sdesc_sw128(sbase + C::kK, kBlock16K, 1024);
        const uint64_t dDSk0 = sdesc_sw128(sbase + C::kDS, 16, 1024);
        const uint64_t dDSmn0 = sdesc_sw128(sbase + C::kDS, kBlock16K, 1024);
        // dV += P^T dO, dK += dS^T Q, dQ = dS K for step `p` (softmax done).
        auto issue_grads = [&](const Pending& p) -> bool {
            if (p.first && !wait_warp(kAccEmpty, (acc_it & 1) ^ 1)) return false;
            const uint32_t kv_off = p.ks * C::kTile, q_off = p.st * C::kTile;
            const uint32_t ds_off = (p.q_it % C::kDsBufs) * 32768u;
            {
                SWA_TRACE(3, p.q_it);
                tc_fence_after();
                const uint32_t acc = p.first ? 0u : 1u;
                // K-major (16, 1024) and MN-major (16 KB, 1024) descriptors of the
                // operand tiles; each contraction step adds its byte offset
                const uint64_t dDOmn = sdesc_at(dDOmn0, q_off), dQmn = sdesc_at(dQmn0, q_off);
                const uint64_t dDSk = sdesc_at(dDSk0, ds_off);
                // contraction step k: P^T columns 8 k (from chunk 4's column on for
                // the second half), dO rows 16 k (2 KB)
                umma_f16_ts_x4(tm_dv, tmem + C::p_col(0), 8, dDOmn, 2048 >> 4, kIdPV, acc);
                umma_f16_ts_x4(tm_dv, tmem + C::p_col(4), 8, sdesc_at(dDOmn, 4 * 2048), 2048 >> 4, kIdPV, 1);
                // P^T is free (and, with everything issued before, the dS^T
                // buffer of the step before this one)
                if constexpr (C::kAhead) umma_commit(bar(kPEmpty));
                {
                    // dS^T columns 16 k (32 bytes, then the next 16 KB block), Q rows 16 k
                    umma_f16_ss_x4(tm_dk, dDSk, 32 >> 4, dQmn, 2048 >> 4, kIdPV, acc);
                    umma_f16_ss_x4(tm_dk, sdesc_at(dDSk, kBlock16K), 32 >> 4, sdesc_at(dQmn, 4 * 2048), 2048 >> 4,
                                   kIdPV, 1);
                }
                // Q and dO have been read (dQ below reads only dS and K): the
                // stage goes back to the producer
                umma_commit(bar(kQEmpty0 + p.st));
            }
            __syncwarp();
            // dQ overwrites the TMEM columns the dQ warps read for the last step;
            // waiting only here lets dV and dK run meanwhile. The second step of
            // a tensor-memory pair adds onto the first's (unread) dQ instead.
            const bool dq_onto = p.tpair == 2;
            if (!dq_onto) {
                if (!C::kDqAliasesS && !wait_warp(kDqEmpty, (dq_it & 1) ^ 1)) return false;
                ++dq_it;
            }
            {
                tc_fence_after();
                const uint64_t dKmn = sdesc_at(dKmn0, kv_off), dDSmn = sdesc_at(dDSmn0, ds_off);
                {
                    // dS rows and K rows 16 k (2 KB each)
                    umma_f16_ss_x4(tm_dq, dDSmn, 2048 >> 4, dKmn, 2048 >> 4, kIdDQ, dq_onto);
                    umma_f16_ss_x4(tm_dq, sdesc_at(dDSmn, 4 * 2048), 2048 >> 4, sdesc_at(dKmn, 4 * 2048), 2048 >> 4,
                                   kIdDQ, 1);
                }
                if (p.tpair != 1) umma_commit(bar(kDqFull));
                SWA_TRACE(4, p.q_it);
                if (p.last) {
                    // after dQ: the epilogue stages dK/dV in this step's dS^T
                    // buffer (d = 128) or in this item's K/V entry (d = 64, whose
                    // epilogue releases the entry)
                    umma_commit(bar(kAccFull));
                    if constexpr (!C::kEpiDq) umma_commit(bar(kKvEmpty0 + p.ks));
                }
            }
            __syncwarp();
            if (p.last) ++acc_it;
            return true;
        };
        bool ok = true;
        for (int64_t item = wk.begin; item < wk.end && ok; item += wk.stride) {
            const Item it = use_items ? items[item] : with_pairs<kTmemPairs>(g, item_at(item), item, wk);
            if (!it.has_work) continue;
            const int ks = kv_it % C::kKvStages;
            if (!(ok = wait_warp(kKvFull0 + ks, (kv_it / C::kKvStages) & 1))) break;
            ++kv_it;
            if (it.kv_base + kTileKV > it.s.len_kv)
                zero_tail<HD>(sm + C::kK + ks * C::kTile, it.s.len_kv - it.kv_base, lane);
            for (int64_t k = 0, j = it.first_j<STRIP>(), hh = it.h0; k < it.steps; ++k, ++q_it, it.template advance<STRIP, kQMajor>(j, hh)) {
                const int st = q_it % C::kStages;
                if (!(ok = wait_warp(kQFull0 + st, (q_it / C::kStages) & 1))) break;
                if (lane == 0) SWA_TRACE(0, q_it);
                const int64_t q0 = j * kTileQ;
                if (q0 + kTileQ > it.s.len_q) {
                    zero_tail<HD>(sm + C::kQ + st * C::kTile, it.s.len_q - q0, lane);
                    zero_tail<HD>(sm + C::kDO + st * C::kTile, it.s.len_q - q0, lane);
                }
                // this step's bookkeeping and operand descriptors, ahead of the
                // wait for the softmax
                const int tp = it.steps <= 2 ? (k == 0 ? it.tp_first : it.tp_last) : tmem_pair<kTmemPairs>(g, it, j, item, wk);
                const Pending cur{true, k == 0, k + 1 == it.steps, st, ks, q_it, tp};
                const uint64_t dK = sdesc_at(dK0, ks * C::kTile), dQ = sdesc_at(dQ0, st * C::kTile);
                const uint64_t dV = sdesc_at(dV0, ks * C::kTile), dDO = sdesc_at(dDO0, st * C::kTile);
                if (C::kAhead && pend.valid) {
                    // P^T, dS^T of the pending step are written and the softmax
                    // is done with S^T, dP^T
                    if (!(ok = wait_warp(kPFull, p_it & 1))) break;
                    if (lane == 0) SWA_TRACE(2, pend.q_it);
                    ++p_it;
                }
                // S^T and dP^T overwrite TMEM that the previous dQ may alias
                if (C::kDqAliasesS && !(ok = wait_warp(kDqEmpty, (dq_it & 1) ^ 1))) break;
                {
                    tc_fence_after();
                    // contraction step k: 32 bytes into the rows of K, Q, V, dO (then,
                    // at d = 128, the same in the second 64-column block)
                    umma_f16_ss_x4(tm_s, dK, 32 >> 4, dQ, 32 >> 4, kIdQK, 0);
                    if constexpr (HD == 128)
                        umma_f16_ss_x4(tm_s, sdesc_at(dK, kBlock16K), 32 >> 4, sdesc_at(dQ, kBlock16K), 32 >> 4,
                                       kIdQK, 1);
                    umma_f16_ss_x4(tm_dp, dV, 32 >> 4, dDO, 32 >> 4, kIdQK, 0);
                    if constexpr (HD == 128)
                        umma_f16_ss_x4(tm_dp, sdesc_at(dV, kBlock16K), 32 >> 4, sdesc_at(dDO, kBlock16K), 32 >> 4,
                                       kIdQK, 1);
                    umma_commit(bar(kSFull));
                    SWA_TRACE(1, q_it);
                }
                __syncwarp();
                if constexpr (C::kAhead) {
                    if (pend.valid && !(ok = issue_grads(pend))) break;
                    pend = cur;
                } else {
                    if (!(ok = wait_warp(kPFull, p_it & 1))) break;
                    if (lane == 0) SWA_TRACE(2, q_it);
                    ++p_it;
                    if (!(ok = issue_grads(cur))) break;
                }
            }
        }
        if (ok && pend.valid) {
            ok = wait_warp(kPFull, p_it & 1);
            ++p_it;
            if (ok) issue_grads(pend);
        }
        // every contraction issued has finished before TMEM is freed (after a
        // wait gave up some may still be running)
        umma_commit(bar(kDrain));
        mbar_wait(bar(kDrain), 0, tmo);
    } else if (warp < kWarpSoft0) {
        if constexpr (C::kAhead) asm volatile("setmaxnreg.dec.sync.aligned.u32 112;");
        // warps 2-3: no role
    } else if (warp < kWarpDq0) {
        // ------------------------------------------------------------ softmax + dK/dV epilogue
        const int r = (warp & 3) * 32 + lane;        // kv row within the tile = TMEM lane
        const int half = (warp - kWarpSoft0) >> 2;   // q columns [64 half, 64 half + 64)
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint32_t q_it = 0, s_it = 0, acc_it = 0;
        // dS^T buffer that an epilogue's TMA store may still be reading (-1: none);
        // the thread that issued it waits before the buffer is written again
        int store_buf = -1;
        auto release_buf = [&](int buf) {
            if (store_buf == buf) {
                if (r == 0) bulk_wait_read0();
                store_buf = -1;
            }
        };
        bool ok = true;
        Epi* epi_slot = reinterpret_cast<Epi*>(sm + C::kMisc + 16);
        bool epi_pending = false;   // an item's dK/dV store waits in epi_slot
        // Epilogue of one item: half 0 writes the tile's dV, half 1 its dK
        // (scaled). Each thread converts its kv row from TMEM into a staged
        // 16-bit tile (128-byte-swizzle layout), which one thread stores with TMA;
        // a tile ending past its sequence's slot (THD) is stored row-wise instead.
        // Rows past the sequence's length are zero; rows past its slot (or past
        // s_kv, where the BSHD maps end) are not written.
        auto run_epi = [&](const Epi e) {
            constexpr int kCpr = HD / 8;   // 16-byte chunks per row
            const int64_t kj = e.kv_base + r;
            bool have = e.have != 0;
            if (have) {
                release_buf(e.buf);   // ordered by the barrier below
                ok = wait_group(kBarSoft, kSoftThreads, kAccFull, e.acc_par);
                have = ok;
                if (lane == 0 && (warp == kWarpSoft0 || warp == kWarpSoft0 + 4))
                    SWA_TRACE(warp == kWarpSoft0 ? 16 : 17, e.last);
                if (ok) tc_fence_after();
            }
            const uint32_t stg_base = (C::kAhead ? C::kDS + e.buf * 32768u : C::kP) + half * (128 * HD * 2);
            uint8_t* stg = sm + stg_base;
            const bool use_tma = !thd || e.kv_base + kTileKV <= e.slot_kv;
            const int64_t* sst = half == 0 ? a.dv_stride : a.dk_stride;
            uint16_t* base = static_cast<uint16_t*>(half == 0 ? a.dv : a.dk);
            if (have) {
                const uint32_t col = tmem + (half == 0 ? C::kColDV : C::kColDK);
                const float mul = half == 0 ? 1.f : a.scale;
                const bool live = kj < e.len_kv;
#pragma unroll 1
                for (int blk = 0; blk < HD / 32; ++blk) {
                    uint32_t v[32];
                    tmem_ld32(col + lane_off + blk * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float f[8];
#pragma unroll
                        for (int x = 0; x < 8; ++x) f[x] = live ? __uint_as_float(v[8 * c + x]) * mul : 0.f;
                        *reinterpret_cast<uint4*>(stg + stg_off(r, blk * 4 + c)) =
                            make_uint4(pack2<BF16>(f[0], f[1]), pack2<BF16>(f[2], f[3]),
                                       pack2<BF16>(f[4], f[5]), pack2<BF16>(f[6], f[7]));
                    }
                }
                tc_fence_before();
                mbar_arrive(bar(kAccEmpty));
                if (use_tma) fence_proxy_async_smem();
                named_bar_sync(kBarSoft, kSoftThreads);
                if (use_tma) {
                    if (r == 0) {
                        const int kvrow = static_cast<int>((thd ? e.kv_row0 : 0) + e.kv_base);
#pragma unroll
                        for (int cb = 0; cb < HD / 64; ++cb)
                            tma_put(false, thd, half == 0 ? &a.tm_dv : &a.tm_dk, sbase + stg_base + cb * kBlock16K,
                                    cb * 64, static_cast<int>(e.gk), kvrow, static_cast<int>(e.bi));
                        bulk_commit();
                    }
                    store_buf = e.buf;
                    if (lane == 0 && (warp == kWarpSoft0 || warp == kWarpSoft0 + 4))
                        SWA_TRACE(warp == kWarpSoft0 ? 18 : 19, e.last);
                    return;
                }
            }
            // row-wise: HD/8 threads per row
            const int c = r % kCpr;
#pragma unroll 1
            for (int pass = 0; pass < kCpr; ++pass) {
                const int row = pass * (128 / kCpr) + r / kCpr;
                const int64_t kr = e.kv_base + row;
                if (kr >= e.slot_kv) break;   // rows ascend with the pass
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (have) w = *reinterpret_cast<const uint4*>(stg + stg_off(row, c));
                uint16_t* dst = base + (thd ? (e.kv_row0 + kr) * sst[1] : e.bi * sst[0] + kr * sst[1]) +
                                e.gk * sst[2] + c * 8;
                if (in_bounds(a.status, dst, base, half == 0 ? g.ext.dv : g.ext.dk, 8))
                    *reinterpret_cast<uint4*>(dst) = w;
            }
        };
        // The next item's record is read right after this one's last P^T
        // hand-off, so that the load overlaps the epilogue bookkeeping.
        auto decode_at = [&](int64_t i) -> Item { return item_at(i < wk.end ? i : wk.begin); };
        Item it = item_at(wk.begin), nxt;
        bool have_nxt = false;
        for (int64_t item = wk.begin; item < wk.end;
             item += wk.stride, it = have_nxt ? nxt : decode_at(item), have_nxt = false) {
            const int64_t kj = it.kv_base + r;
            if (r == 0 && half == 0 && it.s.bad && it.t == 0 && it.gk == 0)
                set_status(a.status, kStatusBadLengths);
            if (it.has_work && ok) {
                int64_t i_lo = 0, i_hi = it.s.len_q - 1;
                if (g.right >= 0) i_lo = imax(i_lo, kj - g.right - it.s.diag);
                if (g.window_left >= 0) i_hi = imin(i_hi, kj + g.window_left - it.s.diag);
                if (kj >= it.s.len_kv) i_hi = -1;
                for (int64_t k = 0, j = it.first_j<STRIP>(), hh = it.h0; k < it.steps; ++k, ++q_it, it.template advance<STRIP, kQMajor>(j, hh)) {
                    const int st = q_it % C::kStages;
                    if (lane == 0 && warp == kWarpSoft0) SWA_TRACE(20, q_it);
                    if constexpr (!C::kEpiDq)
                        release_buf(static_cast<int>(q_it % C::kDsBufs));   // ordered by the barrier below
                    if (lane == 0 && warp == kWarpSoft0) SWA_TRACE(21, q_it);
                    // this q-tile's (LSE, D) pairs and S^T, dP^T: one group barrier
                    if (!(ok = bar_and(kBarSoft, kSoftThreads,
                                       wait(kQFull0 + st, (q_it / C::kStages) & 1) && wait(kSFull, s_it & 1))))
                        break;
                    if (lane == 0 && (warp == kWarpSoft0 || warp == kWarpSoft0 + 4))
                        SWA_TRACE(warp == kWarpSoft0 ? 5 : 7, q_it);
                    ++s_it;
                    tc_fence_after();
                    // the q-tile's statistics: 128 x -LSE * log2(e), then 128 x -D
                    const float* nls = reinterpret_cast<const float*>(sm + C::kStat + st * 1024);
                    const float* nds = nls + kTileQ;
                    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
                    const int64_t q0 = j * kTileQ;
                    const int c_lo = static_cast<int>(imax(i_lo - q0, 0));
                    const int c_hi = static_cast<int>(imin(i_hi - q0, 127));
                    uint8_t* ds_buf = sm + C::kDS + (q_it % C::kDsBufs) * 32768u;
#pragma unroll 1
                    for (int sc = 4 * half; sc < 4 * half + 4; ++sc) {
                        const int c0 = sc * 16;
                        // warp-uniform class of this 16-column chunk
                        const bool none = __all_sync(0xffffffffu, c_hi < c0 || c_lo > c0 + 15);
                        const bool full = __all_sync(0xffffffffu, c_lo <= c0 && c_hi >= c0 + 15);
                        uint32_t pk[8], dk[8];
                        if (none) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) pk[e] = dk[e] = 0u;
                        } else {
                            uint32_t sv[16], dpv[16];
                            tmem_ld16(tmem + C::kColS + lane_off + c0, sv);
                            tmem_ld16(tmem + C::kColDP + lane_off + c0, dpv);
                            tmem_ld_wait();
                            // Column pairs in packed fp32x2 arithmetic: x = s * scale * log2(e)
                            // - LSE * log2(e), P = 2^x, dS = P (dP - D).
                            if (full) {
#pragma unroll
                                for (int e = 0; e < 16; e += 2) {
                                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                                                sc2, *reinterpret_cast<const float2*>(nls + c0 + e));
                                    const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
                                    const float2 t = __fadd2_rn(make_float2(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])),
                                                                *reinterpret_cast<const float2*>(nds + c0 + e));
                                    const float2 d = __fmul2_rn(make_float2(p0, p1), t);
                                    pk[e >> 1] = pack2<BF16>(p0, p1);
                                    dk[e >> 1] = pack2<BF16>(d.x, d.y);
                                }
                            } else {
                                // masked columns: x = -inf gives P = 0; dS is selected to 0
                                // (dP may be NaN there: padding rows need not be finite)
#pragma unroll
                                for (int e = 0; e < 16; e += 2) {
                                    const int c = c0 + e;
                                    const bool att0 = c >= c_lo && c <= c_hi, att1 = c + 1 >= c_lo && c + 1 <= c_hi;
                                    float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                                          sc2, *reinterpret_cast<const float2*>(nls + c));
                                    x.x = att0 ? x.x : -INFINITY;
                                    x.y = att1 ? x.y : -INFINITY;
                                    const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
                                    const float2 t = __fadd2_rn(make_float2(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])),
                                                                *reinterpret_cast<const float2*>(nds + c));
                                    const float2 d = __fmul2_rn(make_float2(p0, p1), t);
                                    pk[e >> 1] = pack2<BF16>(p0, p1);
                                    dk[e >> 1] = pack2<BF16>(att0 ? d.x : 0.f, att1 ? d.y : 0.f);
                                }
                            }
                        }
                        if constexpr (C::kAhead) {
                            // Before the first write: the gradient contractions of
                            // the previous step have read P^T, and (issued after all
                            // those of the step before it) this dS^T buffer.
                            if (sc == 4 * half && q_it > 0) {
                                if (!(ok = wait_group(kBarSoft, kSoftThreads, kPEmpty, (q_it - 1) & 1))) break;
                                tc_fence_after();
                            }
                        }
                        tmem_st8(tmem + C::p_col(sc) + lane_off, pk);
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            const uint32_t off = swz(r, sc * 2 + m);
                            *reinterpret_cast<uint4*>(ds_buf + off) =
                                make_uint4(dk[4 * m], dk[4 * m + 1], dk[4 * m + 2], dk[4 * m + 3]);
                        }
                    }
                    if (!ok) break;
                    tmem_st_wait();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(kPFull));
                    if (lane == 0 && (warp == kWarpSoft0 || warp == kWarpSoft0 + 4))
                        SWA_TRACE(warp == kWarpSoft0 ? 6 : 8, q_it);
                    if constexpr (!C::kEpiDq) {
                        if (epi_pending) {
                            // the previous item's dK/dV store, deferred to here
                            epi_pending = false;
                            run_epi(*epi_slot);
                        }
                    }
                }
                nxt = decode_at(item + wk.stride);
                have_nxt = true;
            }
            if (C::kEpiDq || !it.in_slot) continue;   // d = 64: the dQ warps write dK/dV
            const Epi e{it.kv_base, it.s.kv_row0, it.s.len_kv, it.s.slot_kv, it.bi, it.gk, acc_it & 1,
                        static_cast<int32_t>((q_it + C::kDsBufs - 1) % C::kDsBufs),
                        static_cast<int32_t>(it.has_work && ok), static_cast<int32_t>(q_it - 1)};
            if (it.has_work) ++acc_it;
            if (C::kAhead && e.have) {
                // run after the next item's first q-tile, when these gradients
                // are long done (the next item's first gradient contractions
                // wait for it)
                if (r == 0 && half == 0) *epi_slot = e;
                epi_pending = true;
            } else {
                run_epi(e);
            }
        }
        if (!C::kEpiDq && epi_pending) {
            named_bar_sync(kBarSoft, kSoftThreads);   // epi_slot's write is visible
            run_epi(*epi_slot);
        }
        tmem_st_wait();   // a step left early may have P^T stores in flight
    } else {
        if constexpr (C::kAhead) asm volatile("setmaxnreg.inc.sync.aligned.u32 144;");
        // ------------------------------------------------------------ dQ
        // Visitors of a q-tile are the contiguous kv-tiles [first, first + n).
        //  - n == 1: the lone visitor converts its dQ rows and stores them.
        //  - deterministic mode, or n == 2: the tile is passed along the relay
        //    (turn = t - first; wait until the counter equals the turn): the
        //    first stores fp32 rows into the accumulator, middle turns add,
        //    the last adds the accumulator to its registers, converts and
        //    stores dQ. Sums run in kv-tile order: bitwise repeatable.
        //  - otherwise (n >= 3): unordered vector atomics into the accumulator,
        //    which the preprocess zeroed for these tiles; the dQ convert
        //    kernel converts them.
        // Each thread reads its q row (a TMEM lane) and scales it; 32 columns at
        // a time go through a staged fp32 tile (16-byte chunk c of row r at
        // chunk c ^ (r % 8)), from which 8 threads per row apply them to global
        // memory, so that each warp access covers whole rows.
        const int r = tid - kWarpDq0 * 32;  // q row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint8_t* stg = sm + C::kDqStage;
        const uint32_t stg_s = sbase + C::kDqStage;
        uint32_t dq_it = 0, ld_it = 0, ld1_it = 0;
        bool ok = true;
        // d = 64 dK/dV epilogue state: K/V ring entry an issued store may still
        // be reading (-1: none), and the counters of items with work (their
        // K/V entry and accumulator phase, as the producer and MMA count them)
        int kv_pend = -1;
        uint32_t ekv_it = 0, eacc_it = 0;
        // The entry goes back to the producer once thread 0's stores have read
        // it. Called before every wait of this group (a later item's loads may
        // need the entry) and before the next staging.
        auto kv_release = [&]() {
            if constexpr (C::kEpiDq) {
                if (kv_pend >= 0) {
                    if (r == 0) {
                        bulk_wait_read0();
                        mbar_arrive(bar(kKvEmpty0 + kv_pend));
                    }
                    kv_pend = -1;
                }
            }
        };
        // One item's dK (scaled) and dV, d = 64: each thread converts its kv row
        // (a TMEM lane) of both accumulators into the item's K/V ring entry (V
        // entry: dV, K entry: dK; 128-byte-swizzle tiles), thread 0 stores both
        // with TMA, and the entry is released later (kv_release). A tile ending
        // past its sequence's slot (THD) is written row-wise from the staging.
        // Rows past the sequence's length are zero; rows past its slot (or past
        // s_kv, where the BSHD maps end) are not written. ks < 0: the item has no
        // work (nothing staged; its rows in the slot get zeros).
        auto run_epi_dq = [&](const Item& it, int ks, uint32_t acc_par) {
            constexpr int kCpr = HD / 8;   // 16-byte chunks per row
            kv_release();
            bool have = ks >= 0 && ok;
            if (have) {
                ok = wait_group(kBarDq, 128, kAccFull, acc_par);
                have = ok;
                if (r == 0) SWA_TRACE(16, eacc_it);
                if (ok) tc_fence_after();
            }
            const bool use_tma = !thd || it.kv_base + kTileKV <= it.s.slot_kv;
            if (have) {
                const bool live = it.kv_base + r < it.s.len_kv;
#pragma unroll 1
                for (int ts = 0; ts < 2; ++ts) {
                    uint8_t* stg = sm + (ts == 0 ? C::kV : C::kK) + ks * C::kTile;
                    const uint32_t col = tmem + (ts == 0 ? C::kColDV : C::kColDK) + lane_off;
                    const float mul = ts == 0 ? 1.f : a.scale;
                    uint32_t v0[32], v1[32];
                    tmem_ld32(col, v0);
                    tmem_ld32(col + 32, v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        float f[8];
#pragma unroll
                        for (int x = 0; x < 8; ++x)
                            f[x] = live ? __uint_as_float(c < 4 ? v0[8 * c + x] : v1[8 * (c - 4) + x]) * mul : 0.f;
                        *reinterpret_cast<uint4*>(stg + stg_off(r, c)) =
                            make_uint4(pack2<BF16>(f[0], f[1]), pack2<BF16>(f[2], f[3]),
                                       pack2<BF16>(f[4], f[5]), pack2<BF16>(f[6], f[7]));
                    }
                }
                tc_fence_before();
                mbar_arrive(bar(kAccEmpty));
                if (use_tma) fence_proxy_async_smem();
                named_bar_sync(kBarDq, 128);
                if (use_tma) {
                    if (r == 0) {
                        const int kvrow = static_cast<int>((thd ? it.s.kv_row0 : 0) + it.kv_base);
                        tma_put(false, thd, &a.tm_dv, sbase + C::kV + ks * C::kTile, 0, static_cast<int>(it.gk),
                                kvrow, static_cast<int>(it.bi));
                        tma_put(false, thd, &a.tm_dk, sbase + C::kK + ks * C::kTile, 0, static_cast<int>(it.gk),
                                kvrow, static_cast<int>(it.bi));
                        bulk_commit();
                        SWA_TRACE(18, eacc_it);
                    }
                    kv_pend = ks;
                    return;
                }
            }
            // row-wise: HD/8 threads per row, dV then dK
            const int c = r % kCpr;
#pragma unroll 1
            for (int ts = 0; ts < 2; ++ts) {
                const uint8_t* stg = sm + (ts == 0 ? C::kV : C::kK) + (ks < 0 ? 0 : ks) * C::kTile;
                const int64_t* sst = ts == 0 ? a.dv_stride : a.dk_stride;
                uint16_t* base = static_cast<uint16_t*>(ts == 0 ? a.dv : a.dk);
#pragma unroll 1
                for (int pass = 0; pass < kCpr; ++pass) {
                    const int row = pass * (128 / kCpr) + r / kCpr;
                    const int64_t kr = it.kv_base + row;
                    if (kr >= it.s.slot_kv) break;   // rows ascend with the pass
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (have) w = *reinterpret_cast<const uint4*>(stg + stg_off(row, c));
                    uint16_t* dst = base + (thd ? (it.s.kv_row0 + kr) * sst[1] : it.bi * sst[0] + kr * sst[1]) +
                                    it.gk * sst[2] + c * 8;
                    if (in_bounds(a.status, dst, base, ts == 0 ? g.ext.dv : g.ext.dk, 8))
                        *reinterpret_cast<uint4*>(dst) = w;
                }
            }
            if (ks >= 0) {
                // the staging has been read: the entry goes back at once
                named_bar_sync(kBarDq, 128);
                if (r == 0) mbar_arrive(bar(kKvEmpty0 + ks));
            }
        };
        for (int64_t item = wk.begin; item < wk.end && ok; item += wk.stride) {
            const Item it = item_at(item);
            if (!it.has_work) {
                if (C::kEpiDq && it.in_slot) run_epi_dq(it, -1, 0u);
                continue;
            }
            const int eks = static_cast<int>(ekv_it % C::kKvStages);
            const uint32_t epar = eacc_it & 1;
            for (int64_t k = 0, j = it.first_j<STRIP>(), hh = it.h0; k < it.steps; ++k, it.template advance<STRIP, kQMajor>(j, hh)) {
                // this visit's bookkeeping first, while the dQ contraction runs
                // (after the wait it delayed the TMEM read by ~1 K cycles)
                int64_t first, nvis;
                q_tile_visitors(g, it.s, j, first, nvis);
                const int turn = static_cast<int>(it.t - first);
                int32_t* sem = a.sems + (it.bi * g.h_q + hh) * a.n_q_tiles + j;
                if (!in_bounds(a.status, sem, a.sems, g.ext.sems, 1)) sem = a.sems;
                // TMA writes whole 128-row boxes: the tile must lie inside the
                // sequence's slot (always so for BSHD, whose maps end at s_q)
                const bool use_tma = !thd || (j + 1) * kTileQ <= it.s.slot_q;
                // Strip mode (at most two visitors, kv-tiles t and t + 1 of one
                // head): the two are consecutive items of this CTA unless its run
                // ends between them ("local"), and combine with no waiting. At
                // d = 64 with one q-head per kv-head their dQ contractions add up
                // in tensor memory; otherwise the first stores its fp32 partial in
                // the accumulator rows and the second loads it back. A pair split
                // between two CTAs goes by arrival order: the first to arrive
                // stores its partial and flags it, the second adds it to its own.
                // A sum of two rounded partials does not depend on their order,
                // so this stays bitwise repeatable.
                const bool local = STRIP && nvis == 2 && (turn == 0 ? item + 1 < wk.end : item > wk.begin);
                // d = 64, one q-head per kv-head: the pair's dQ adds up in tensor
                // memory (tmem_pair); the first step reads nothing, the second the sum
                const int tpair = kTmemPairs && local && it.group == 1 ? 1 + turn : 0;
                if (tpair == 1) continue;
                const bool pair = STRIP && nvis == 2 && !local;
                const bool single = nvis <= 1 || tpair == 2;   // no partial to combine
                // two visitors, or deterministic mode where no per-visitor slots
                // apply (fewer than three visitors, or none allotted): hand the
                // tile along in turn order
                const bool relay = !STRIP && (nvis == 2 || (a.deterministic && (nvis < 3 || a.n_slots == 0)));
                // deterministic mode otherwise: each visitor stores its own fp32
                // partial (slot = turn), which the convert kernel sums in visitor
                // order
                const bool slots = !STRIP && a.deterministic && !relay;
                bool conv_now = single || (relay && turn == nvis - 1) || (local && turn == 1);
                const bool lpair = local && !tpair;   // a local pair through the accumulator rows
                // accumulator write: a store for the first relay turn (and for
                // every strip-mode partial), else an add
                const bool add = !STRIP && !(relay && turn == 0);
                const int qrow = static_cast<int>((thd ? it.s.q_row0 : 0) + j * kTileQ);
                const int tb = static_cast<int>(it.bi), th = static_cast<int>(hh);
                kv_release();
                if (STRIP && C::kDqAliasesS && r == 0) {
                    // Strip mode at d = 128: the second visitor of a pair inside this
                    // CTA's run reads the partial that the first stored one item
                    // earlier, by then often out of L2, while its dQ columns (and so
                    // the next S^T) wait. Move it back for the next step (of this
                    // item, or the next item's first) while this one runs.
                    int64_t j2 = j, h2 = hh;
                    Item nx = it;
                    bool have = true;
                    if (k + 1 < it.steps) {
                        it.template advance<STRIP, kQMajor>(j2, h2);
                    } else if (item + wk.stride < wk.end) {
                        nx = item_at(item + wk.stride);
                        j2 = nx.first_j<STRIP>();
                        h2 = nx.h0;
                        have = nx.has_work;
                    } else {
                        have = false;
                    }
                    if (have) {
                        int64_t f2, n2;
                        q_tile_visitors(g, nx.s, j2, f2, n2);
                        if (n2 == 2 && nx.t - f2 == 1 && (!thd || (j2 + 1) * kTileQ <= nx.s.slot_q)) {
                            const int row2 = static_cast<int>((thd ? nx.s.q_row0 : 0) + j2 * kTileQ);
#pragma unroll
                            for (int c = 0; c < HD; c += 32)
                                tma_prefetch_l2(&a.tm_acc, thd, c, static_cast<int>(h2), row2, static_cast<int>(nx.bi));
                        }
                    }
                }
                if (r == 0) bulk_wait_read0();   // the staging is free again
                // Second step of a pair inside this CTA's run: the partial was stored
                // an item ago, so it (at d = 128 its first half) comes into the
                // staging while the dQ contraction runs
                const bool pre0 = lpair && turn == 1 && use_tma && (!C::kDqAliasesS || k + 1 < it.steps);
                const uint32_t pre_ld = ld_it;
                if (pre0) {
                    if (r == 0) {
                        bulk_wait0();   // this thread stored the partial
                        fence_proxy_async_global();
                        mbar_arrive_expect_tx(bar(kDqLoad), 2 * kBlock16K);
                        tma_box(stg_s, &a.tm_acc, bar(kDqLoad), thd, 0, th, qrow, tb);
                        tma_box(stg_s + kBlock16K, &a.tm_acc, bar(kDqLoad), thd, 32, th, qrow, tb);
                    }
                    ++ld_it;
                }
                if (!(ok = wait_group(kBarDq, 128, kDqFull, dq_it & 1))) break;
                if (r == 0) SWA_TRACE(9, dq_it);
                ++dq_it;
                tc_fence_after();
                // Waits for this visit's turn (relay) in thread 0; true in all 128
                // threads if the turn came (or none was needed) and nothing aborted.
                bool early = false;   // pair: this visitor arrived first
                auto wait_turn = [&]() -> bool {
                    bool mine = true;
                    if (pair && r == 0) {
                        // each arrival adds 1; the first adds 4 once its partial
                        // is in place, which the second waits for
                        early = atom_add_acq_rel_gpu(sem, 1) == 0;
                        if (!early) {
                            const uint64_t t0 = globaltimer_ns();
                            const int flag = (a.test_flags & 2) ? 1024 : 4;
                            while (!(ld_acquire_gpu(sem) & flag)) {
                                if (*abort_flag || globaltimer_ns() - t0 > tmo) {
                                    mine = gave_up(a.status, abort_flag, kWherePair);
                                    break;
                                }
                            }
                            fence_proxy_async_global();
                        }
                    }
                    if (relay && turn > 0 && r == 0) {
                        const uint64_t t0 = globaltimer_ns();
                        for (;;) {
                            if (ld_acquire_gpu(sem) == turn + ((a.test_flags & 1) << 30)) break;
                            if (*abort_flag || globaltimer_ns() - t0 > tmo) {
                                mine = gave_up(a.status, abort_flag, kWhereRelay);
                                break;
                            }
                        }
                        // later async-proxy writes follow the acquired ones
                        fence_proxy_async_global();
                    }
                    const bool go_on = bar_and(kBarDq, 128, mine && *abort_flag == 0);
                    if (pair) {
                        early = bar_or(kBarDq, 128, early);   // thread 0's arrival, to the group
                        conv_now = !early;
                    }
                    return go_on;
                };
                // Converts 32 dQ values of this row (columns [32 ch, 32 ch + 32)),
                // adding the earlier visitors' partial sum unless alone, into the
                // staged 16-bit tile.
                auto stage_out = [&](int ch, const uint32_t (&v)[32]) {
                    float f[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]) * a.scale;
                    if (!single) {
                        // rows past the sequence's length hold zeros and take none
                        // (their load reads the last row instead, a valid address)
                        const int64_t qi = j * kTileQ + r;
                        const bool row_ok = qi < it.s.len_q;
                        const float* accr =
                            a.dq_acc + ((it.s.q_row0 + (row_ok ? qi : it.s.len_q - 1)) * g.h_q + hh) * HD + ch * 32;
                        const float m = row_ok ? 1.f : 0.f;
                        const bool acc_ok = in_bounds(a.status, accr, a.dq_acc, g.ext.dq_acc, 32);
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            const float4 o = acc_ok ? ld_cg_f4(accr + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                            f[e] += m * o.x; f[e + 1] += m * o.y; f[e + 2] += m * o.z; f[e + 3] += m * o.w;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        *reinterpret_cast<uint4*>(stg + stg_off(r, ch * 4 + i)) =
                            make_uint4(pack2<BF16>(f[8 * i], f[8 * i + 1]), pack2<BF16>(f[8 * i + 2], f[8 * i + 3]),
                                       pack2<BF16>(f[8 * i + 4], f[8 * i + 5]),
                                       pack2<BF16>(f[8 * i + 6], f[8 * i + 7]));
                };
                // Stages 32 fp32 values of this row as chunks [8 blk, 8 blk + 8).
                auto stage_acc = [&](int blk, const uint32_t (&v)[32]) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<float4*>(stg + stg_off(r, blk * 8 + i)) =
                            make_float4(__uint_as_float(v[4 * i]) * a.scale, __uint_as_float(v[4 * i + 1]) * a.scale,
                                        __uint_as_float(v[4 * i + 2]) * a.scale,
                                        __uint_as_float(v[4 * i + 3]) * a.scale);
                };
                // Writes the staged fp32 columns [col0, col0 + 64) of the tile
                // from thread 0 with two TMA boxes: into the accumulator, or as
                // this visitor's own partial (a store into its slot).
                auto put_acc = [&](int col0) {
                    fence_proxy_async_smem();
                    named_bar_sync(kBarDq, 128);
                    if (r == 0) {
                        // a slot: a plain store at the slot's rows of the 3-D partials map
                        const CUtensorMap* map = slots ? &a.tm_part : &a.tm_acc;
                        // the slot's first row (n_slots covers every possible visitor)
                        const int row = slots ? static_cast<int>((((it.bi * g.h_q + hh) * a.n_q_tiles + j) *
                                                                      a.n_slots + turn) * kTileQ)
                                              : qrow;
                        const int hd = slots ? 0 : th;
                        tma_put(add && !slots, thd || slots, map, stg_s, col0, hd, row, tb);
                        tma_put(add && !slots, thd || slots, map, stg_s + kBlock16K, col0 + 32, hd, row, tb);
                        bulk_commit();
                    }
                };
                // Row-wise fallback for a tile that ends past its sequence's slot
                // (THD): applies staged fp32 columns [col0, col0 + 64) with 16
                // threads per row -- converted (plus the earlier visitors' sum
                // unless alone), stored as the first partial, or added to it.
                // Partial sums are loaded 8 rows at a time before any store.
                auto apply = [&](int col0) {
                    named_bar_sync(kBarDq, 128);
                    const int c = r & 15, col = col0 + c * 4;
                    const int64_t qi0 = j * kTileQ + (r >> 4);   // pass p: row (r >> 4) + 8 p
                    const int64_t nrows = it.s.len_q - qi0;     // passes with 8 p < nrows run
                    float* acc0 = a.dq_acc + ((it.s.q_row0 + qi0) * g.h_q + hh) * HD + col;
                    const int64_t acc_step = 8 * g.h_q * HD;
                    // last row of the sequence, a valid address for every pass's load
                    float* acc_last = a.dq_acc + ((it.s.q_row0 + it.s.len_q - 1) * g.h_q + hh) * HD + col;
#pragma unroll
                    for (int p0 = 0; p0 < 16; p0 += 8) {
                        float4 v[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            v[u] = *reinterpret_cast<const float4*>(stg + stg_off((p0 + u) * 8 + (r >> 4), c));
                        if (conv_now && !single) {
                            float4 o[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const float* pl = (p0 + u) * 8 < nrows ? acc0 + (p0 + u) * acc_step : acc_last;
                                o[u] = in_bounds(a.status, pl, a.dq_acc, g.ext.dq_acc, 4) ? ld_cg_f4(pl)
                                                                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                v[u].x += o[u].x; v[u].y += o[u].y; v[u].z += o[u].z; v[u].w += o[u].w;
                            }
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            if ((p0 + u) * 8 >= nrows) break;
                            float* accp = acc0 + (p0 + u) * acc_step;
                            if (conv_now) {
                                const int64_t qi = qi0 + (p0 + u) * 8, prow = it.s.q_row0 + qi;
                                uint16_t* dqp = static_cast<uint16_t*>(a.dq) +
                                                (thd ? prow * a.dq_stride[1]
                                                     : it.bi * a.dq_stride[0] + qi * a.dq_stride[1]) +
                                                hh * a.dq_stride[2] + col;
                                if (in_bounds(a.status, dqp, a.dq, g.ext.dq, 4))
                                    *reinterpret_cast<uint2*>(dqp) =
                                        make_uint2(pack2<BF16>(v[u].x, v[u].y), pack2<BF16>(v[u].z, v[u].w));
                            } else if (!in_bounds(a.status, accp, a.dq_acc, g.ext.dq_acc, 4)) {
                            } else if (!add) {
                                *reinterpret_cast<float4*>(accp) = v[u];
                            } else {
                                red_add_v4(accp, v[u].x, v[u].y, v[u].z, v[u].w);
                            }
                        }
                    }
                };
                bool go;
                if constexpr (HD == 64) {
                    // read the whole row and free TMEM before any wait
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tmem + C::kColDQ + lane_off, v0);
                    tmem_ld32(tmem + C::kColDQ + lane_off + 32, v1);
                    tmem_ld_wait();
                    tc_fence_before();
                    mbar_arrive(bar(kDqEmpty));
                    if (r == 0) SWA_TRACE(10, dq_it - 1);
                    go = wait_turn();
                    if (r == 0) SWA_TRACE(15, dq_it - 1);
                    if (go) {
                        if (conv_now && use_tma && !single) {
                            // the earlier visitors' partial sum: one TMA load of the
                            // fp32 tile into the staging (issued above for a pair
                            // inside the run); each thread then adds its row and
                            // writes it back converted, in place
                            uint32_t ldi = pre_ld;
                            if (!pre0) {
                                ldi = ld_it++;
                                if (r == 0) {
                                    mbar_arrive_expect_tx(bar(kDqLoad), 2 * kBlock16K);
                                    tma_box(stg_s, &a.tm_acc, bar(kDqLoad), thd, 0, th, qrow, tb);
                                    tma_box(stg_s + kBlock16K, &a.tm_acc, bar(kDqLoad), thd, 32, th, qrow, tb);
                                }
                            }
                            const bool got = wait_group(kBarDq, 128, kDqLoad, ldi & 1);
                            if (got) {
                                // 16-bit chunk i (columns 8i..8i+7) from fp32 chunks 2i,
                                // 2i+1; it lands where fp32 chunk i was, already used
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const float4 x0 = *reinterpret_cast<const float4*>(stg + stg_off(r, 2 * i));
                                    const float4 x1 = *reinterpret_cast<const float4*>(stg + stg_off(r, 2 * i + 1));
                                    const uint32_t* v = i < 4 ? v0 + 8 * i : v1 + 8 * (i - 4);
                                    if constexpr (STRIP) {
                                        // own partial rounded, then one add: a two-term
                                        // sum that does not depend on which came first
                                        auto sum = [&](int e, float x) {
                                            return __fadd_rn(__fmul_rn(__uint_as_float(v[e]), a.scale), x);
                                        };
                                        *reinterpret_cast<uint4*>(stg + stg_off(r, i)) = make_uint4(
                                            pack2<BF16>(sum(0, x0.x), sum(1, x0.y)), pack2<BF16>(sum(2, x0.z), sum(3, x0.w)),
                                            pack2<BF16>(sum(4, x1.x), sum(5, x1.y)), pack2<BF16>(sum(6, x1.z), sum(7, x1.w)));
                                        continue;
                                    }
                                    *reinterpret_cast<uint4*>(stg + stg_off(r, i)) = make_uint4(
                                        pack2<BF16>(fmaf(__uint_as_float(v[0]), a.scale, x0.x),
                                                    fmaf(__uint_as_float(v[1]), a.scale, x0.y)),
                                        pack2<BF16>(fmaf(__uint_as_float(v[2]), a.scale, x0.z),
                                                    fmaf(__uint_as_float(v[3]), a.scale, x0.w)),
                                        pack2<BF16>(fmaf(__uint_as_float(v[4]), a.scale, x1.x),
                                                    fmaf(__uint_as_float(v[5]), a.scale, x1.y)),
                                        pack2<BF16>(fmaf(__uint_as_float(v[6]), a.scale, x1.z),
                                                    fmaf(__uint_as_float(v[7]), a.scale, x1.w)));
                                }
                            }
                            fence_proxy_async_smem();
                            named_bar_sync(kBarDq, 128);
                            if (r == 0 && got) {
                                tma_put(false, thd, &a.tm_dq, stg_s, 0, th, qrow, tb);
                                bulk_commit();
                            }
                        } else if (conv_now && use_tma) {
                            stage_out(0, v0);
                            stage_out(1, v1);
                            fence_proxy_async_smem();
                            named_bar_sync(kBarDq, 128);
                            if (r == 0) {
                                tma_put(false, thd, &a.tm_dq, stg_s, 0, th, qrow, tb);
                                bulk_commit();
                            }
                        } else {
                            stage_acc(0, v0);
                            stage_acc(1, v1);
                            // a slot is a whole 128-row tile of the workspace
                            if (use_tma || slots) put_acc(0);
                            else apply(0);
                        }
                    }
                } else {
                    go = wait_turn();
                    if (r == 0) SWA_TRACE(15, dq_it - 1);
                    // A partial sum to add comes by TMA for whole tiles (first
                    // branch); tiles that end past a THD slot take the row-wise
                    // path, which loads it eight rows at a time (read per row, its
                    // latency would hold the dQ columns of TMEM, aliasing S^T, four
                    // times over).
                    if (conv_now && use_tma && go && !single && k + 1 < it.steps) {
                        // Adds the stored partial and converts, a 64-column half at a
                        // time: the fp32 partial comes by TMA (half 0 into the staging,
                        // half 1 into the epilogue's region at kP, idle apart from an
                        // item's last step, which this path leaves out), this visit's
                        // dQ from TMEM, and each half of the 16-bit tile goes out from
                        // the staging.
                        uint32_t ld0 = pre_ld;
                        if (!pre0) {
                            ld0 = ld_it++;
                            if (r == 0) {
                                if (lpair) {
                                    bulk_wait0();   // this thread stored the partial
                                    fence_proxy_async_global();
                                }
                                mbar_arrive_expect_tx(bar(kDqLoad), 2 * kBlock16K);
                                tma_box(stg_s, &a.tm_acc, bar(kDqLoad), thd, 0, th, qrow, tb);
                                tma_box(stg_s + kBlock16K, &a.tm_acc, bar(kDqLoad), thd, 32, th, qrow, tb);
                            }
                        }
                        const uint32_t ld1 = ld1_it++;
                        if (r == 0) {
                            mbar_arrive_expect_tx(bar(kDqLoad1), 2 * kBlock16K);
                            tma_box(sbase + C::kP, &a.tm_acc, bar(kDqLoad1), thd, 64, th, qrow, tb);
                            tma_box(sbase + C::kP + kBlock16K, &a.tm_acc, bar(kDqLoad1), thd, 96, th, qrow, tb);
                        }
#pragma unroll 1
                        for (int hf = 0; hf < 2; ++hf) {
                            uint32_t v0[32], v1[32];
                            tmem_ld32(tmem + C::kColDQ + lane_off + 64 * hf, v0);
                            tmem_ld32(tmem + C::kColDQ + lane_off + 64 * hf + 32, v1);
                            tmem_ld_wait();
                            const bool got = hf == 0 ? wait_group(kBarDq, 128, kDqLoad, ld0 & 1)
                                                     : wait_group(kBarDq, 128, kDqLoad1, ld1 & 1);
                            const uint8_t* src = hf == 0 ? stg : sm + C::kP;
                            if (got) {
                                // 16-bit chunk i of the half (columns 8i..8i+7) from fp32
                                // chunks 2i, 2i+1; written to staging chunk 8 hf + i
                                // (half 0 in place, over fp32 chunks already read)
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const float4 x0 = *reinterpret_cast<const float4*>(src + stg_off(r, 2 * i));
                                    const float4 x1 = *reinterpret_cast<const float4*>(src + stg_off(r, 2 * i + 1));
                                    const uint32_t* v = i < 4 ? v0 + 8 * i : v1 + 8 * (i - 4);
                                    // strip mode: own partial rounded, then one add (a
                                    // two-term sum that does not depend on which came
                                    // first); the relay adds in turn order
                                    auto sum = [&](int e, float x) {
                                        return STRIP ? __fadd_rn(__fmul_rn(__uint_as_float(v[e]), a.scale), x)
                                                     : fmaf(__uint_as_float(v[e]), a.scale, x);
                                    };
                                    *reinterpret_cast<uint4*>(stg + stg_off(r, 8 * hf + i)) = make_uint4(
                                        pack2<BF16>(sum(0, x0.x), sum(1, x0.y)), pack2<BF16>(sum(2, x0.z), sum(3, x0.w)),
                                        pack2<BF16>(sum(4, x1.x), sum(5, x1.y)), pack2<BF16>(sum(6, x1.z), sum(7, x1.w)));
                                }
                            }
                            if (hf == 1) {
                                // TMEM and the region at kP have been read
                                tc_fence_before();
                                mbar_arrive(bar(kDqEmpty));
                            }
                            fence_proxy_async_smem();
                            named_bar_sync(kBarDq, 128);
                            if (r == 0 && got) {
                                tma_put(false, thd, &a.tm_dq, stg_s + hf * kBlock16K, 64 * hf, th, qrow, tb);
                                bulk_commit();
                            }
                        }
                    } else if (conv_now && use_tma && single) {
#pragma unroll 1
                        for (int ch = 0; ch < HD / 32; ++ch) {
                            uint32_t v[32];
                            tmem_ld32(tmem + C::kColDQ + lane_off + ch * 32, v);
                            tmem_ld_wait();
                            if (go) stage_out(ch, v);
                        }
                        tc_fence_before();
                        mbar_arrive(bar(kDqEmpty));
                        fence_proxy_async_smem();
                        named_bar_sync(kBarDq, 128);
                        if (r == 0 && go) {
                            tma_put(false, thd, &a.tm_dq, stg_s, 0, th, qrow, tb);
                            tma_put(false, thd, &a.tm_dq, stg_s + kBlock16K, 64, th, qrow, tb);
                            bulk_commit();
                        }
                    } else {
#pragma unroll 1
                        for (int rd = 0; rd < HD / 64; ++rd) {
                            if (rd > 0) {
                                // the previous half has left the staging
                                if (r == 0) bulk_wait_read0();
                                named_bar_sync(kBarDq, 128);
                            }
                            uint32_t v[32];
                            tmem_ld32(tmem + C::kColDQ + lane_off + rd * 64, v);
                            tmem_ld_wait();
                            stage_acc(0, v);
                            tmem_ld32(tmem + C::kColDQ + lane_off + rd * 64 + 32, v);
                            tmem_ld_wait();
                            stage_acc(1, v);
                            if ((use_tma || slots) && !conv_now) {
                                fence_proxy_async_smem();
                                named_bar_sync(kBarDq, 128);
                                if (r == 0 && go) {
                                    const CUtensorMap* map = slots ? &a.tm_part : &a.tm_acc;
                                    const int row = slots ? static_cast<int>((((it.bi * g.h_q + hh) * a.n_q_tiles +
                                                                                j) * a.n_slots + turn) * kTileQ)
                                                          : qrow;
                                    const int hd = slots ? 0 : th;
                                    tma_put(add && !slots, thd || slots, map, stg_s, rd * 64, hd, row, tb);
                                    tma_put(add && !slots, thd || slots, map, stg_s + kBlock16K, rd * 64 + 32, hd,
                                            row, tb);
                                    bulk_commit();
                                }
                            } else if (go) {
                                if (lpair && rd == 0 && r == 0) {
                                    // this thread stored the partial in an earlier step
                                    bulk_wait0();
                                    fence_proxy_async_global();
                                }
                                apply(rd * 64);
                            } else {
                                named_bar_sync(kBarDq, 128);
                            }
                        }
                        tc_fence_before();
                        mbar_arrive(bar(kDqEmpty));
                    }
                }
                if (r == 0) SWA_TRACE(11, dq_it - 1);
                if (pair && early && go) {
                    // the partial is in place: complete its copies, then flag it (+4)
                    if (use_tma) {
                        if (r == 0) {
                            bulk_wait0();
                            fence_proxy_async_global();
                            red_add_release_gpu(sem, 4);
                        }
                    } else {
                        named_bar_sync(kBarDq, 128);
                        if (r == 0) {
                            __threadfence();
                            red_add_release_gpu(sem, 4);
                        }
                    }
                    continue;
                }
                if (!relay || turn + 1 >= nvis) continue;
                // publish this turn's partial sum to the next visitor
                if (use_tma) {
                    // thread 0 issued every copy of the tile: complete them first
                    if (r == 0) {
                        bulk_wait0();
                        fence_proxy_async_global();
                        st_release_gpu(sem, turn + 1);
                    }
                } else {
                    // the group's stores are ordered before one release
                    named_bar_sync(kBarDq, 128);
                    if (r == 0) st_release_gpu(sem, turn + 1);
                }
            }
            if constexpr (C::kEpiDq) {
                if (ok) run_epi_dq(it, eks, epar);
            }
            ++ekv_it;
            ++eacc_it;
        }
        // a partner tile whose load a given-up wait did not see complete
        if (r == 0 && ld_it > 0) mbar_wait(bar(kDqLoad), (ld_it - 1) & 1, tmo);
        if (r == 0 && ld1_it > 0) mbar_wait(bar(kDqLoad1), (ld1_it - 1) & 1, tmo);
    }

    bulk_wait0();   // copies issued from this CTA's shared memory are complete
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// The round-robin walk's order (ItemOrder) for BSHD problems without length
// arrays: every item of kv-tile t takes the same steps, (q-tiles it sweeps) x
// (q-heads per kv-head), plus one for its dK/dV store. False (plain round
// robin) when the host cannot tell the steps or the table does not hold them.
static bool balanced_order(const MainArgs& a, int64_t items, int64_t grid, ItemOrder& o)
{
    const Geometry& g = a.g;
    if (g.layout != 0 || g.seq_q_lens || g.seq_kv_lens || items > kOrderMaxItems || grid > kOrderMaxCtas ||
        grid < 2)
        return false;
    SeqInfo sq{};
    sq.slot_q = sq.len_q = g.s_q;
    sq.slot_kv = sq.len_kv = g.s_kv;
    sq.diag = g.mask_mode == 2 ? g.s_kv - g.s_q : 0;
    const int64_t group = g.h_q / g.h_kv;
    std::vector<int64_t> steps(a.n_kv_tiles);
    for (int64_t t = 0; t < a.n_kv_tiles; ++t) {
        int64_t lo, hi;
        q_tile_range(g, sq, t, lo, hi);
        steps[t] = (hi > lo ? hi - lo : 0) * group + 1;
    }
    // items numbered head fastest: kv-tile (i / h_kv) mod n_kv_tiles
    auto work = [&](int64_t i) { return steps[(i / g.h_kv) % a.n_kv_tiles]; };
    std::vector<int32_t> by_work(items);
    for (int64_t i = 0; i < items; ++i) by_work[i] = static_cast<int32_t>(i);
    std::stable_sort(by_work.begin(), by_work.end(), [&](int32_t x, int32_t y) { return work(x) > work(y); });
    // longest first to the least-loaded CTA (ties: the lower CTA)
    std::vector<std::pair<int64_t, int32_t>> heap;
    for (int32_t c = 0; c < grid; ++c) heap.push_back({0, c});
    auto later = [](const std::pair<int64_t, int32_t>& x, const std::pair<int64_t, int32_t>& y) { return x > y; };
    std::vector<int32_t> cta_of(items);
    for (int32_t i : by_work) {
        std::pop_heap(heap.begin(), heap.end(), later);
        cta_of[i] = heap.back().second;
        heap.back().first += work(i);
        std::push_heap(heap.begin(), heap.end(), later);
    }
    // each CTA's items in ascending number
    std::vector<int32_t> count(grid + 1, 0);
    for (int64_t i = 0; i < items; ++i) ++count[cta_of[i] + 1];
    for (int64_t c = 0; c < grid; ++c) count[c + 1] += count[c];
    for (int64_t c = 0; c <= grid; ++c) o.off[c] = static_cast<uint16_t>(count[c]);
    std::vector<int32_t> fill(count.begin(), count.end() - 1);
    for (int64_t i = 0; i < items; ++i) o.item[fill[cta_of[i]]++] = static_cast<uint16_t>(i);
    return true;
}

template <int HD, bool BF16, bool STRIP>
static cudaError_t launch_typed(const MainArgs& a, cudaStream_t s)
{
    const uint32_t bytes = Cfg<HD>::kBytes;
    cudaError_t e;
    const int64_t items = a.g.b * a.g.h_kv * a.n_kv_tiles;
    if (items == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int64_t grid = items < sms ? items : sms;
    int64_t group_heads = 1;
    if constexpr (STRIP) {
        // R runs per group of G kv-heads, at least one item each. The
        // smallest G that fills the most SMs (G = 1 for the lockstep of every
        // head; the host falls back to the round-robin walk when there are
        // more kv-heads than SMs).
        const int64_t per_head = items / a.g.h_kv;
        int64_t best = 0;
        for (int64_t G = 1; G <= a.g.h_kv && G <= 8; ++G) {   // e.g. 6 kv-heads: G = 3, 2 x 76 runs
            if (a.g.h_kv % G) continue;
            int64_t runs = sms * G / a.g.h_kv;
            if (runs > per_head * G) runs = per_head * G;
            if (runs * (a.g.h_kv / G) > best) {
                best = runs * (a.g.h_kv / G);
                group_heads = G;
            }
        }
        grid = best;
    }
    MainArgs b = a;
    if constexpr (STRIP) b.strip = static_cast<int32_t>(group_heads);
    b.use_items = items <= kItemTableMaxPerCta * grid;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    // Strip instance: programmatic stream serialization, so that this grid's
    // prologue overlaps the preprocess's last blocks and the launch latency
    // (b2 h16 S8192 step 0.113 -> 0.110 ms, S2048 0.047 -> 0.044 ms). The
    // round-robin instance launches plainly: with it the non-square W8000
    // step ran 0.59 ms against 0.535 ms, though no kernel of it ran longer.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = STRIP ? 1 : 0;
    static_assert(kOrderMaxItems <= 65536, "item numbers are 16-bit");
    // the balanced order, built per launch on the host and passed by value
    // with it (its own kernel instance, so that launches without one carry no
    // order parameter)
    static thread_local ItemOrder ord;
    if (!STRIP && balanced_order(b, items, grid, ord)) {
        auto kern = sdpa_bwd_main_kernel<HD, BF16, false, true>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
            return e;
        if ((e = cudaLaunchKernelEx(&cfg, kern, b, ord)) != cudaSuccess) return e;
    } else {
        auto kern = sdpa_bwd_main_kernel<HD, BF16, STRIP, false>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
            return e;
        if ((e = cudaLaunchKernelEx(&cfg, kern, b, NoOrder{})) != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_main(const MainArgs& a, int dtype, cudaStream_t s)
{
    if (a.g.d == 64) {
        if (a.strip) return dtype == 0 ? launch_typed<64, true, true>(a, s) : launch_typed<64, false, true>(a, s);
        return dtype == 0 ? launch_typed<64, true, false>(a, s) : launch_typed<64, false, false>(a, s);
    }
    if (a.strip) return dtype == 0 ? launch_typed<128, true, true>(a, s) : launch_typed<128, false, true>(a, s);
    return dtype == 0 ? launch_typed<128, true, false>(a, s) : launch_typed<128, false, false>(a, s);
}

}  // namespace swa
