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
//               kStages stages (128-byte swizzle, zero fill past the tensor)
//   warp 1      MMA issuer (one thread) and TMEM owner
//   warps 2-3   idle (the q-tile's per-row (LSE log2, D) pairs arrive with the
//               producer's Q/dO loads as one 1 KB bulk copy)
//   warps 4-11  softmax: two warps per TMEM sub-partition, each thread one kv
//               row (TMEM lane) and one 64-column half of the q-tile; recomputes
//               P = exp2(S*scale*log2e - LSE*log2e) and dS = P (dP - D) with the
//               mask, skipping 32-column chunks the window masks for the whole
//               warp; writes P^T / dS^T as swizzled 16-bit tiles; at the end of
//               an item one half stores dV, the other dK (or fp32 GQA partials)
//   warps 12-15 dQ: one thread per q row reads dQ from TMEM and adds it to the
//               fp32 accumulator (vector atomics, or the ordered relay)
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

#include "ptx.cuh"
#include "sdpa_internal.h"
#include "seq.cuh"

namespace swa {

namespace {

constexpr int kThreads = 512;
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
    static constexpr uint32_t kTile = 128 * HD * 2;
    // shared memory offsets (from a 1024-aligned base)
    static constexpr uint32_t kK = 0;                           // kKvStages tiles
    static constexpr uint32_t kV = kK + kKvStages * kTile;      // kKvStages tiles
    static constexpr uint32_t kQ = kV + kKvStages * kTile;      // kStages tiles
    static constexpr uint32_t kDO = kQ + kStages * kTile;       // kStages tiles
    static constexpr bool kPInTmem = HD == 64;                  // P^T kept in TMEM
    static constexpr uint32_t kP = kDO + kStages * kTile;       // P^T  [128 kv x 128 q] (d = 128)
    static constexpr uint32_t kDS = kP + (kPInTmem ? 0 : 32768); // dS^T [128 kv x 128 q]
    static constexpr uint32_t kStat = kDS + 32768;              // kStages x 128 float2
    static constexpr uint32_t kBars = kStat + kStages * 1024;   // mbarriers
    static constexpr uint32_t kMisc = kBars + 256;              // tmem slot, flags
    static constexpr uint32_t kBytes = kMisc + 64;
    static constexpr uint32_t kAlloc = kBytes + 1024;
    // TMEM columns
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + HD;
    static constexpr uint32_t kColDQ = HD == 64 ? 384 : 0;
    static constexpr uint32_t kColP = 448;                      // d = 64 only
    static constexpr bool kDqAliasesS = HD != 64;
};

// mbarrier indices
enum Bar : int {
    kSFull = 0, kPFull, kDqFull, kDqEmpty, kAccFull, kAccEmpty,
    kQFull0, kQFull1, kQEmpty0, kQEmpty1, kKvFull0, kKvFull1, kKvEmpty0, kKvEmpty1, kNumBars
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

// Optional timeline trace (build with -DSDPA_BWD_TRACE): SM clock stamps of each
// role's hand-offs for the first kTraceCtas CTAs and kTraceTiles q-tiles, written
// to the workspace at byte offset kTraceOffset (the caller sizes the workspace
// for it). Off by default; it records and changes nothing else.
constexpr int kTraceCtas = 8, kTraceTiles = 64, kTraceSlots = 16;
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
    // step k: q-head h0 + k / nq, q-tile q_hi - 1 - k % nq
    __device__ __forceinline__ int64_t head(int64_t k) const { return h0 + k / nq; }
    __device__ __forceinline__ int64_t qtile(int64_t k) const { return q_hi - 1 - k % nq; }
};

__device__ __forceinline__ Item decode(const MainArgs& a, int64_t item)
{
    const Geometry& g = a.g;
    Item it;
    it.t = item % a.n_kv_tiles;
    it.gk = (item / a.n_kv_tiles) % g.h_kv;
    it.bi = item / (a.n_kv_tiles * g.h_kv);
    it.group = g.h_q / g.h_kv;
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

template <int HD, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) sdpa_bwd_main_kernel(const __grid_constant__ MainArgs a)
{
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
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

    if (tid == 0) {
        misc[1] = 0;
        for (int s = 0; s < C::kKvStages; ++s) {
            mbar_init(bar(kKvFull0 + s), 1);
            mbar_init(bar(kKvEmpty0 + s), 1);
        }
        mbar_init(bar(kSFull), 1);
        mbar_init(bar(kPFull), kSoftThreads);
        mbar_init(bar(kDqFull), 1);
        mbar_init(bar(kDqEmpty), 128);
        mbar_init(bar(kAccFull), 1);
        mbar_init(bar(kAccEmpty), kSoftThreads);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
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

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kv_it = 0, q_it = 0;
            for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
                const Item it = decode(a, item);
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
                for (int64_t k = 0; k < it.steps; ++k, ++q_it) {
                    const int64_t j = it.qtile(k), hh = it.head(k);
                    const int st = q_it % C::kStages;
                    if (!wait(kQEmpty0 + st, ((q_it / C::kStages) & 1) ^ 1)) { ok = false; break; }
                    SWA_TRACE(12, q_it);
                    const int qrow = static_cast<int>((thd ? it.s.q_row0 : 0) + j * kTileQ);
                    mbar_arrive_expect_tx(bar(kQFull0 + st), 2 * C::kTile + 1024);
                    tma_tile<HD>(sbase + C::kQ + st * C::kTile, &a.tm_q, bar(kQFull0 + st), thd,
                                 (int)hh, qrow, (int)it.bi);
                    tma_tile<HD>(sbase + C::kDO + st * C::kTile, &a.tm_do, bar(kQFull0 + st), thd,
                                 (int)hh, qrow, (int)it.bi);
                    bulk_load(sbase + C::kStat + st * 1024,
                              a.stats + (static_cast<int64_t>(it.bi) * g.h_q + hh) * a.stats_row +
                                  static_cast<int64_t>(j) * kTileQ,
                              1024, bar(kQFull0 + st));
                    SWA_TRACE(13, q_it);
                }
                if (!ok) break;
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t kIdQK = idesc_f16(BF16, 128, 128, false, false);
        constexpr uint32_t kIdPV = idesc_f16(BF16, 128, HD, false, true);
        constexpr uint32_t kIdDQ = idesc_f16(BF16, 128, HD, true, true);
        const uint32_t tm_s = tmem + C::kColS, tm_dp = tmem + C::kColDP;
        const uint32_t tm_dv = tmem + C::kColDV, tm_dk = tmem + C::kColDK, tm_dq = tmem + C::kColDQ;
        uint32_t kv_it = 0, q_it = 0, p_it = 0, dq_it = 0, acc_it = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const Item it = decode(a, item);
            if (!it.has_work) continue;
            const int ks = kv_it % C::kKvStages;
            if (!(ok = wait_warp(kKvFull0 + ks, (kv_it / C::kKvStages) & 1))) break;
            ++kv_it;
            const uint32_t sK = sbase + C::kK + ks * C::kTile, sV = sbase + C::kV + ks * C::kTile;
            if (it.kv_base + kTileKV > it.s.len_kv)
                zero_tail<HD>(sm + C::kK + ks * C::kTile, it.s.len_kv - it.kv_base, lane);
            for (int64_t k = 0; k < it.steps; ++k, ++q_it) {
                const int64_t j = it.qtile(k);
                const int st = q_it % C::kStages;
                if (!(ok = wait_warp(kQFull0 + st, (q_it / C::kStages) & 1))) break;
                if (lane == 0) SWA_TRACE(0, q_it);
                const int64_t q0 = j * kTileQ;
                if (q0 + kTileQ > it.s.len_q) {
                    zero_tail<HD>(sm + C::kQ + st * C::kTile, it.s.len_q - q0, lane);
                    zero_tail<HD>(sm + C::kDO + st * C::kTile, it.s.len_q - q0, lane);
                }
                // S^T and dP^T overwrite TMEM that the previous dQ may alias
                if (C::kDqAliasesS && !(ok = wait_warp(kDqEmpty, (dq_it & 1) ^ 1))) break;
                const uint32_t sQ = sbase + C::kQ + st * C::kTile, sDO = sbase + C::kDO + st * C::kTile;
                if (lane == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < HD / 16; ++k) {
                        const uint32_t koff = (k >> 2) * kBlock16K + (k & 3) * 32;
                        umma_f16_ss(tm_s, sdesc_sw128(sK + koff, 16, 1024),
                                    sdesc_sw128(sQ + koff, 16, 1024), kIdQK, k > 0);
                    }
#pragma unroll
                    for (int k = 0; k < HD / 16; ++k) {
                        const uint32_t koff = (k >> 2) * kBlock16K + (k & 3) * 32;
                        umma_f16_ss(tm_dp, sdesc_sw128(sV + koff, 16, 1024),
                                    sdesc_sw128(sDO + koff, 16, 1024), kIdQK, k > 0);
                    }
                    umma_commit(bar(kSFull));
                    SWA_TRACE(1, q_it);
                }
                __syncwarp();
                // P^T, dS^T ready in shared memory (softmax done with S^T, dP^T)
                if (!(ok = wait_warp(kPFull, p_it & 1))) break;
                if (lane == 0) SWA_TRACE(2, q_it);
                ++p_it;
                if (!C::kDqAliasesS && !(ok = wait_warp(kDqEmpty, (dq_it & 1) ^ 1))) break;
                if (k == 0 && !(ok = wait_warp(kAccEmpty, (acc_it & 1) ^ 1))) break;
                ++dq_it;
                if (lane == 0) {
                    SWA_TRACE(3, q_it);
                    tc_fence_after();
                    const uint32_t acc = k > 0 ? 1u : 0u;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint64_t bdesc = sdesc_sw128(sDO + k * 2048, kBlock16K, 1024);
                        if constexpr (C::kPInTmem) {
                            umma_f16_ts(tm_dv, tmem + C::kColP + k * 8, bdesc, kIdPV, acc | (k > 0));
                        } else {
                            const uint32_t aoff = (k >> 2) * kBlock16K + (k & 3) * 32;
                            umma_f16_ss(tm_dv, sdesc_sw128(sbase + C::kP + aoff, 16, 1024), bdesc, kIdPV,
                                        acc | (k > 0));
                        }
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t aoff = (k >> 2) * kBlock16K + (k & 3) * 32;
                        umma_f16_ss(tm_dk, sdesc_sw128(sbase + C::kDS + aoff, 16, 1024),
                                    sdesc_sw128(sQ + k * 2048, kBlock16K, 1024), kIdPV, acc | (k > 0));
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        umma_f16_ss(tm_dq, sdesc_sw128(sbase + C::kDS + k * 2048, kBlock16K, 1024),
                                    sdesc_sw128(sK + k * 2048, kBlock16K, 1024), kIdDQ, k > 0);
                    umma_commit(bar(kDqFull));
                    umma_commit(bar(kQEmpty0 + st));
                    SWA_TRACE(4, q_it);
                    if (k + 1 == it.steps) {
                        umma_commit(bar(kAccFull));
                        umma_commit(bar(kKvEmpty0 + ks));
                    }
                }
                __syncwarp();
            }
            if (!ok) break;
            ++acc_it;
        }
    } else if (warp < kWarpSoft0) {
        // warps 2-3: no role
    } else if (warp < kWarpDq0) {
        // ------------------------------------------------------------ softmax + dK/dV epilogue
        const int r = (warp & 3) * 32 + lane;        // kv row within the tile = TMEM lane
        const int half = (warp - kWarpSoft0) >> 2;   // q columns [64 half, 64 half + 64)
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint32_t q_it = 0, s_it = 0, acc_it = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
            const Item it = decode(a, item);
            const int64_t kj = it.kv_base + r;
            if (r == 0 && half == 0 && it.s.bad && it.t == 0 && it.gk == 0)
                set_status(a.status, kStatusBadLengths);
            if (it.has_work && ok) {
                int64_t i_lo = 0, i_hi = it.s.len_q - 1;
                if (g.right >= 0) i_lo = imax(i_lo, kj - g.right - it.s.diag);
                if (g.window_left >= 0) i_hi = imin(i_hi, kj + g.window_left - it.s.diag);
                if (kj >= it.s.len_kv) i_hi = -1;
                for (int64_t k = 0; k < it.steps; ++k, ++q_it) {
                    const int64_t j = it.qtile(k);
                    const int st = q_it % C::kStages;
                    if (!(ok = wait_group(kBarSoft, kSoftThreads, kQFull0 + st, (q_it / C::kStages) & 1))) break;
                    if (!(ok = wait_group(kBarSoft, kSoftThreads, kSFull, s_it & 1))) break;
                    if (lane == 0 && (warp == kWarpSoft0 || warp == kWarpSoft0 + 4))
                        SWA_TRACE(warp == kWarpSoft0 ? 5 : 7, q_it);
                    ++s_it;
                    tc_fence_after();
                    const float2* stv = reinterpret_cast<const float2*>(sm + C::kStat + st * 1024);
                    const int64_t q0 = j * kTileQ;
                    const int c_lo = static_cast<int>(imax(i_lo - q0, 0));
                    const int c_hi = static_cast<int>(imin(i_hi - q0, 127));
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
                            if (full) {
#pragma unroll
                                for (int e = 0; e < 16; e += 2) {
                                    const float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), a.scale_log2, -stv[c0 + e].x));
                                    const float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), a.scale_log2, -stv[c0 + e + 1].x));
                                    pk[e >> 1] = pack2<BF16>(p0, p1);
                                    dk[e >> 1] = pack2<BF16>(p0 * (__uint_as_float(dpv[e]) - stv[c0 + e].y),
                                                             p1 * (__uint_as_float(dpv[e + 1]) - stv[c0 + e + 1].y));
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 16; e += 2) {
                                    float p2[2], d2[2];
#pragma unroll
                                    for (int u = 0; u < 2; ++u) {
                                        const int c = c0 + e + u;
                                        const bool att = c >= c_lo && c <= c_hi;
                                        const float p = att ? ex2_approx(fmaf(__uint_as_float(sv[e + u]),
                                                                             a.scale_log2, -stv[c].x))
                                                            : 0.f;
                                        p2[u] = p;
                                        d2[u] = att ? p * (__uint_as_float(dpv[e + u]) - stv[c].y) : 0.f;
                                    }
                                    pk[e >> 1] = pack2<BF16>(p2[0], p2[1]);
                                    dk[e >> 1] = pack2<BF16>(d2[0], d2[1]);
                                }
                            }
                        }
                        if constexpr (C::kPInTmem) {
                            tmem_st8(tmem + C::kColP + lane_off + sc * 8, pk);
                        }
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            const uint32_t off = swz(r, sc * 2 + m);
                            if constexpr (!C::kPInTmem)
                                *reinterpret_cast<uint4*>(sm + C::kP + off) =
                                    make_uint4(pk[4 * m], pk[4 * m + 1], pk[4 * m + 2], pk[4 * m + 3]);
                            *reinterpret_cast<uint4*>(sm + C::kDS + off) =
                                make_uint4(dk[4 * m], dk[4 * m + 1], dk[4 * m + 2], dk[4 * m + 3]);
                        }
                    }
                    if constexpr (C::kPInTmem) tmem_st_wait();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(kPFull));
                    if (lane == 0 && (warp == kWarpSoft0 || warp == kWarpSoft0 + 4))
                        SWA_TRACE(warp == kWarpSoft0 ? 6 : 8, q_it);
                }
                if (ok) ok = wait_group(kBarSoft, kSoftThreads, kAccFull, acc_it & 1);
                ++acc_it;
                if (ok) tc_fence_after();
            }
            // epilogue: half 0 stores this kv row's dV, half 1 its dK (scaled)
            if (!it.in_slot) continue;
            const bool live = it.has_work && ok && kj < it.s.len_kv;
            const bool row_in_slot = kj < it.s.slot_kv;
            const int64_t prow = it.s.kv_row0 + kj;
            const int which = half;
            {
                const uint32_t col = tmem + (which == 0 ? C::kColDV : C::kColDK);
                const float mul = which == 0 ? 1.f : a.scale;
#pragma unroll 1
                for (int ch = 0; ch < HD / 16; ++ch) {
                    uint32_t v[16];
                    if (it.has_work && ok) {
                        tmem_ld16(col + lane_off + ch * 16, v);
                        tmem_ld_wait();
                    }
                    float f[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) f[e] = live ? __uint_as_float(v[e]) * mul : 0.f;
                    if (!row_in_slot) continue;
                    {
                        const int64_t* sst = which == 0 ? a.dv_stride : a.dk_stride;
                        uint16_t* base = static_cast<uint16_t*>(which == 0 ? a.dv : a.dk);
                        uint16_t* dst = base + (thd ? prow * sst[1] : it.bi * sst[0] + kj * sst[1]) +
                                        it.gk * sst[2] + ch * 16;
#pragma unroll
                        for (int e = 0; e < 16; e += 8)
                            *reinterpret_cast<uint4*>(dst + e) =
                                make_uint4(pack2<BF16>(f[e], f[e + 1]), pack2<BF16>(f[e + 2], f[e + 3]),
                                           pack2<BF16>(f[e + 4], f[e + 5]), pack2<BF16>(f[e + 6], f[e + 7]));
                    }
                }
            }
            if (it.has_work && ok) {
                tc_fence_before();
                mbar_arrive(bar(kAccEmpty));
            }
        }
    } else {
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
        const int r = tid - kWarpDq0 * 32;  // q row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint32_t dq_it = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const Item it = decode(a, item);
            if (!it.has_work) continue;
            for (int64_t k = 0; k < it.steps; ++k) {
                const int64_t j = it.qtile(k), hh = it.head(k);
                if (!(ok = wait_group(kBarDq, 128, kDqFull, dq_it & 1))) break;
                if (r == 0) SWA_TRACE(9, dq_it);
                ++dq_it;
                tc_fence_after();
                const int64_t qi = j * kTileQ + r;
                const bool row_ok = qi < it.s.len_q;
                const int64_t prow = it.s.q_row0 + qi;
                int64_t first, nvis;
                q_tile_visitors(g, it.s, j, first, nvis);
                const int turn = static_cast<int>(it.t - first);
                const bool single = nvis <= 1;
                int32_t* sem = a.sems + (it.bi * g.h_q + hh) * a.n_q_tiles + j;
                float* acc = a.dq_acc + (prow * g.h_q + hh) * HD;
                uint16_t* dqp = static_cast<uint16_t*>(a.dq) +
                                (thd ? prow * a.dq_stride[1] : it.bi * a.dq_stride[0] + qi * a.dq_stride[1]) +
                                hh * a.dq_stride[2];
                // two visitors, or deterministic mode: hand the tile along in turn order
                const bool relay = a.deterministic || nvis == 2;
                const bool accumulate = !single && !relay;
                const bool conv_now = single || (relay && turn == nvis - 1);
                // Waits for this visit's turn (relay) or for the first visitor's store.
                auto wait_turn = [&]() -> bool {
                    if (!relay || turn == 0) return true;
                    if (r == 0) {
                        const uint64_t t0 = globaltimer_ns();
                        for (;;) {
                            if (ld_acquire_gpu(sem) == turn) break;
                            if (*abort_flag || globaltimer_ns() - t0 > tmo) {
                                set_status(a.status, kStatusTimeout);
                                *abort_flag = 1;
                                break;
                            }
                        }
                    }
                    named_bar_sync(kBarDq, 128);
                    return *abort_flag == 0;
                };
                // Writes 32 dQ values of this row: converted (plus the partial sum
                // of the earlier visitors unless alone), stored as the first
                // partial, or added to it.
                auto emit = [&](int col, float (&f)[32]) {
                    if (conv_now) {
                        if (!single) {
#pragma unroll
                            for (int e = 0; e < 32; e += 4) {
                                const float4 o = ld_cg_f4(acc + col + e);
                                f[e] += o.x; f[e + 1] += o.y; f[e + 2] += o.z; f[e + 3] += o.w;
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 32; e += 8)
                            *reinterpret_cast<uint4*>(dqp + col + e) =
                                make_uint4(pack2<BF16>(f[e], f[e + 1]), pack2<BF16>(f[e + 2], f[e + 3]),
                                           pack2<BF16>(f[e + 4], f[e + 5]), pack2<BF16>(f[e + 6], f[e + 7]));
                    } else if (turn == 0 && !accumulate) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(acc + col + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; e += 4) red_add_v4(acc + col + e, f[e], f[e + 1], f[e + 2], f[e + 3]);
                    }
                };
                bool turn_ok = true;
                if constexpr (HD == 64) {
                    // the whole row fits in registers: free TMEM before any wait
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tmem + C::kColDQ + lane_off, v0);
                    tmem_ld32(tmem + C::kColDQ + lane_off + 32, v1);
                    tmem_ld_wait();
                    tc_fence_before();
                    mbar_arrive(bar(kDqEmpty));
                    if (r == 0) SWA_TRACE(10, dq_it - 1);
                    float f0[32], f1[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        f0[e] = __uint_as_float(v0[e]) * a.scale;
                        f1[e] = __uint_as_float(v1[e]) * a.scale;
                    }
                    turn_ok = wait_turn();
                    if (row_ok && turn_ok) {
                        emit(0, f0);
                        emit(32, f1);
                    }
                } else {
                    turn_ok = wait_turn();
#pragma unroll 1
                    for (int ch = 0; ch < HD / 32; ++ch) {
                        uint32_t v[32];
                        tmem_ld32(tmem + C::kColDQ + lane_off + ch * 32, v);
                        tmem_ld_wait();
                        float f[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]) * a.scale;
                        if (row_ok && turn_ok) emit(ch * 32, f);
                    }
                    tc_fence_before();
                    mbar_arrive(bar(kDqEmpty));
                }
                if (r == 0) SWA_TRACE(11, dq_it - 1);
                if (!relay) continue;
                // publish: the group's writes are ordered before one release
                named_bar_sync(kBarDq, 128);
                if (r == 0 && turn + 1 < nvis) st_release_gpu(sem, turn + 1);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int HD, bool BF16>
static cudaError_t launch_typed(const MainArgs& a, cudaStream_t s)
{
    auto kern = sdpa_bwd_main_kernel<HD, BF16>;
    const uint32_t bytes = Cfg<HD>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    const int64_t items = a.g.b * a.g.h_kv * a.n_kv_tiles;
    if (items == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t grid = items < sms ? items : sms;
    kern<<<static_cast<unsigned>(grid), kThreads, bytes, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_main(const MainArgs& a, int dtype, cudaStream_t s)
{
    if (a.g.d == 64) return dtype == 0 ? launch_typed<64, true>(a, s) : launch_typed<64, false>(a, s);
    return dtype == 0 ? launch_typed<128, true>(a, s) : launch_typed<128, false>(a, s);
}

}  // namespace swa
