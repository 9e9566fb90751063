// fwd_kernel.cu -- sliding-window SDPA forward (O, LSE) on sm_103a tensor cores.
//
// Work item = (q-tile j, q-head h, sequence b), numbered head-fastest. A
// persistent CTA (one per SM) walks its items; for each it loads the q-tile
// once and sweeps the kv-tiles that the mask admits for any of the tile's rows,
// keeping per row a running maximum m and sum l of the exponentials (the
// online softmax, in the log2 domain):
//
//   S   = Q K^T    [q x kv]  TMEM columns 0..127 / 128..255 (two buffers)
//   O  += P V      [q x d]   TMEM columns 256..
//
// Warp roles (256 threads):
//   warp 0      TMA producer: Q per item; K, V per kv-tile into a 2-stage ring
//   warp 1      MMA issuer (lane 0 of the converged warp) and TMEM owner;
//               S of kv-tile t + 1 is issued before P V of kv-tile t, so the
//               softmax of one kv-tile overlaps the tensor core's work on the
//               next
//   warps 2-3   idle
//   warps 4-7   softmax and epilogue, one q row (TMEM lane) per thread, the
//               whole 128-column S row in registers: m' = max(m, max_j s_j),
//               p_j = exp2(s_j - m'), l = l * exp2(m - m') + sum_j p_j; once the
//               previous P V is done it rescales its O row by exp2(m - m') and
//               writes P (16-bit) to shared memory; at the end O / l (with the
//               sink's term in l) is staged and stored by TMA, LSE written.
// Hand-offs are mbarriers; every wait is bounded (status word on timeout).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sdpa_internal.h"
#include "seq.cuh"

namespace swa {

namespace {

constexpr int kFThreads = 256;
constexpr int kFWarpSoft0 = 4;
constexpr int kFBarSoft = 1;   // named barrier of the 128 softmax threads
constexpr uint32_t kFBlock = 128 * 128;  // one 64-column block of a 128-row 16-bit tile
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int HD>
struct FCfg {
    static constexpr uint32_t kTile = 128 * HD * 2;
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kTile;        // 2 stages
    static constexpr uint32_t kV = kK + 2 * kTile;    // 2 stages
    static constexpr uint32_t kP = kV + 2 * kTile;    // P [128 q x 128 kv], then the O staging
    static constexpr uint32_t kBars = kP + 32768;
    static constexpr uint32_t kMisc = kBars + 256;    // tmem slot, abort flag
    static constexpr uint32_t kBytes = kMisc + 64;
    static_assert(kBytes <= 232448, "shared memory above the 227 KB a CTA may opt into");
    static_assert(128 * HD * 2 <= 32768, "O staging must fit the P buffer");
    static constexpr uint32_t kColS = 0;              // + 128 * buffer
    static constexpr uint32_t kColO = 256;
};

enum FBar : int {
    fQFull = 0, fQEmpty, fKvFull0, fKvFull1, fKvEmpty0, fKvEmpty1, fSFull0, fSFull1, fSFree0, fSFree1,
    fPFull, fPvDone, fOEmpty, fNumBars
};

template <bool BF16>
__device__ __forceinline__ uint32_t fpack2(float lo, float hi)
{
    uint32_t r;
    if constexpr (BF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 16-byte chunk c of row r of a swizzled 128-row tile of 128-byte rows (blocks
// of 64 16-bit columns 16 KB apart; the TMA 128-byte swizzle).
__device__ __forceinline__ uint32_t fswz(int r, int c)
{
    return static_cast<uint32_t>((c >> 3) * kFBlock + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void ftma_load(uint32_t dst, const CUtensorMap* map, uint32_t bar, bool thd, int c0,
                                          int head, int row, int batch)
{
    if (thd)
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(head), "r"(row)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(head), "r"(row), "r"(batch)
            : "memory");
}

__device__ __forceinline__ void ftma_store(uint32_t src, const CUtensorMap* map, bool thd, int c0, int head,
                                           int row, int batch)
{
    if (thd)
        asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                         reinterpret_cast<uint64_t>(map)),
                     "r"(src), "r"(c0), "r"(head), "r"(row)
                     : "memory");
    else
        asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                         reinterpret_cast<uint64_t>(map)),
                     "r"(src), "r"(c0), "r"(head), "r"(row), "r"(batch)
                     : "memory");
}

// Rows [row, row + 128) of one head, HD columns, as HD/64 swizzled boxes.
template <int HD>
__device__ __forceinline__ void ftma_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar, bool thd, int head,
                                          int row, int batch)
{
#pragma unroll
    for (int cb = 0; cb < HD / 64; ++cb) ftma_load(dst + cb * kFBlock, map, bar, thd, cb * 64, head, row, batch);
}

// Zeroes rows [nvalid, 128) of a swizzled tile (whole rows); one warp.
template <int HD>
__device__ __forceinline__ void fzero_tail(uint8_t* tile, int64_t nvalid, int lane)
{
    const int first = nvalid < 0 ? 0 : static_cast<int>(nvalid);
    if (first >= 128) return;
#pragma unroll
    for (int cb = 0; cb < HD / 64; ++cb) {
        uint4* p = reinterpret_cast<uint4*>(tile + cb * kFBlock + first * 128);
        const int n16 = (128 - first) * 8;
        for (int k = lane; k < n16; k += 32) p[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    __syncwarp();
}

__device__ __forceinline__ bool fbar_and(int id, int count, bool v)
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

struct FItem {
    int64_t j, h, g, bi;
    SeqInfo s;
    int64_t q0;           // first row of the q-tile within the sequence
    int64_t kv_lo, kv_hi; // kv-tiles [kv_lo, kv_hi] hold every admitted key
    bool rows;            // the q-tile has rows inside the slot (to write)
    bool keys;            // some row of it admits some key
};

struct FCounts {
    uint32_t h_q, n_q_tiles, group;
};

// Keys [k_lo, k_hi] that query row i (anchor i + diag) admits; empty if k_lo > k_hi.
__device__ __forceinline__ void row_keys(const Geometry& g, const SeqInfo& s, int64_t i, int64_t& k_lo,
                                         int64_t& k_hi)
{
    if (i >= s.len_q || s.len_kv == 0) {
        k_lo = 1;
        k_hi = 0;
        return;
    }
    const int64_t anchor = i + s.diag;
    k_lo = g.window_left >= 0 ? imax64(anchor - g.window_left, 0) : 0;
    k_hi = g.right >= 0 ? imin64(anchor + g.right, s.len_kv - 1) : s.len_kv - 1;
}

__device__ __forceinline__ FItem fdecode(const FwdArgs& a, const FCounts& n, int64_t item)
{
    const Geometry& g = a.g;
    FItem it;
    // head-fastest: the CTAs running together read every head of a few q-tiles
    const uint32_t u = static_cast<uint32_t>(item);
    const uint32_t rest = u / n.h_q, bq = rest / n.n_q_tiles;
    it.h = u - rest * n.h_q;
    it.j = rest - bq * n.n_q_tiles;
    it.bi = bq;
    it.g = it.h / n.group;
    it.s = seq_info(g, it.bi);
    it.q0 = it.j * kTileQ;
    it.rows = it.q0 < it.s.slot_q;
    it.keys = false;
    it.kv_lo = 0;
    it.kv_hi = -1;
    if (it.q0 < it.s.len_q) {
        // the admitted key range grows with the row: first and last rows bound it
        int64_t lo0, hi0, lo1, hi1;
        row_keys(g, it.s, it.q0, lo0, hi0);
        row_keys(g, it.s, imin64(it.q0 + kTileQ, it.s.len_q) - 1, lo1, hi1);
        const int64_t lo = lo0, hi = hi1;
        if (lo <= hi && hi >= 0) {
            it.keys = true;
            it.kv_lo = lo / kTileKV;
            it.kv_hi = hi / kTileKV;
        }
    }
    return it;
}

}  // namespace

template <int HD, bool BF16>
__global__ void __launch_bounds__(kFThreads, 1) sdpa_fwd_kernel(const __grid_constant__ FwdArgs a)
{
    using C = FCfg<HD>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) set_status(a.status, kStatusUnsupported);
        return;
    }
    uint8_t* sm = smem_raw;
    const uint32_t sbase = smem_u32(sm);
    auto bar = [&](int i) -> uint32_t { return sbase + C::kBars + 8u * i; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::kMisc);  // [0] tmem base, [1] abort flag

    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint64_t tmo = static_cast<uint64_t>(a.timeout_ns);
    const int64_t n_items = g.b * g.h_q * a.n_q_tiles;
    const bool thd = g.layout == 1;
    const FCounts cnt{static_cast<uint32_t>(g.h_q), static_cast<uint32_t>(a.n_q_tiles),
                      static_cast<uint32_t>(g.h_q / g.h_kv)};

    if (tid == 0) {
        misc[1] = 0;
        mbar_init(bar(fQFull), 1);
        mbar_init(bar(fQEmpty), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(fKvFull0 + s), 1);
            mbar_init(bar(fKvEmpty0 + s), 1);
            mbar_init(bar(fSFull0 + s), 1);
            mbar_init(bar(fSFree0 + s), 128);
        }
        mbar_init(bar(fPFull), 128);
        mbar_init(bar(fPvDone), 1);
        mbar_init(bar(fOEmpty), 128);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + C::kMisc, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    volatile uint32_t* abort_flag = misc + 1;

    auto wait = [&](int b, uint32_t parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait(bar(b), parity, tmo)) return true;
        *abort_flag = 1;
        set_status(a.status, kStatusTimeout);
        return false;
    };
    auto wait_warp = [&](int b, uint32_t parity) -> bool { return __all_sync(0xffffffffu, wait(b, parity)); };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kv_it = 0, q_it = 0;
            bool ok = true;
            for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                const FItem it = fdecode(a, cnt, item);
                if (!it.keys) continue;
                if (!(ok = wait(fQEmpty, (q_it & 1) ^ 1))) break;
                ++q_it;
                mbar_arrive_expect_tx(bar(fQFull), C::kTile);
                ftma_tile<HD>(sbase + C::kQ, &a.tm_q, bar(fQFull), thd, static_cast<int>(it.h),
                              static_cast<int>((thd ? it.s.q_row0 : 0) + it.q0), static_cast<int>(it.bi));
                for (int64_t t = it.kv_lo; t <= it.kv_hi; ++t, ++kv_it) {
                    const int st = kv_it & 1;
                    if (!(ok = wait(fKvEmpty0 + st, ((kv_it >> 1) & 1) ^ 1))) break;
                    const int row = static_cast<int>((thd ? it.s.kv_row0 : 0) + t * kTileKV);
                    mbar_arrive_expect_tx(bar(fKvFull0 + st), 2 * C::kTile);
                    ftma_tile<HD>(sbase + C::kK + st * C::kTile, &a.tm_k, bar(fKvFull0 + st), thd,
                                  static_cast<int>(it.g), row, static_cast<int>(it.bi));
                    ftma_tile<HD>(sbase + C::kV + st * C::kTile, &a.tm_v, bar(fKvFull0 + st), thd,
                                  static_cast<int>(it.g), row, static_cast<int>(it.bi));
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t kIdS = idesc_f16(BF16, 128, 128, false, false);
        constexpr uint32_t kIdPV = idesc_f16(BF16, 128, HD, false, true);
        const uint32_t tm_o = tmem + C::kColO;
        uint32_t kv_it = 0, q_it = 0, s_it = 0, p_it = 0, o_it = 0;
        struct Pend {
            bool valid, first;
            int st;
        };
        // O += P V for the kv-tile in ring stage pd.st (softmax done with it)
        auto issue_pv = [&](const Pend& pd) -> bool {
            if (!wait_warp(fPFull, p_it & 1)) return false;
            ++p_it;
            // the first P V of an item overwrites O: the epilogue has read it
            if (pd.first) {
                if (!wait_warp(fOEmpty, (o_it & 1) ^ 1)) return false;
                ++o_it;
            }
            {
                tc_fence_after();
                const uint64_t dP = sdesc_sw128(sbase + C::kP, 16, 1024);
                const uint64_t dV = sdesc_sw128(sbase + C::kV + pd.st * C::kTile, kFBlock, 1024);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t aoff = (k >> 2) * kFBlock + (k & 3) * 32;
                    umma_f16_ss(tm_o, sdesc_at(dP, aoff), sdesc_at(dV, k * 2048), kIdPV,
                                (pd.first && k == 0) ? 0u : 1u);
                }
                umma_commit(bar(fPvDone));
                umma_commit(bar(fKvEmpty0 + pd.st));
            }
            __syncwarp();
            return true;
        };
        bool ok = true;
        for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const FItem it = fdecode(a, cnt, item);
            if (!it.keys) continue;
            if (!(ok = wait_warp(fQFull, q_it & 1))) break;
            ++q_it;
            Pend pend{false, false, 0};
            for (int64_t t = it.kv_lo; t <= it.kv_hi && ok; ++t, ++kv_it, ++s_it) {
                const int st = kv_it & 1;
                if (!(ok = wait_warp(fKvFull0 + st, (kv_it >> 1) & 1))) break;
                // keys past the sequence's length are masked out of P, but their
                // V rows meet P's zeros in the product: make them zero too
                if (t * kTileKV + kTileKV > it.s.len_kv)
                    fzero_tail<HD>(sm + C::kV + st * C::kTile, it.s.len_kv - t * kTileKV, lane);
                const int sb = s_it & 1;
                if (!(ok = wait_warp(fSFree0 + sb, ((s_it >> 1) & 1) ^ 1))) break;
                {
                    tc_fence_after();
                    const uint64_t dQ = sdesc_sw128(sbase + C::kQ, 16, 1024);
                    const uint64_t dK = sdesc_sw128(sbase + C::kK + st * C::kTile, 16, 1024);
#pragma unroll
                    for (int k = 0; k < HD / 16; ++k) {
                        const uint32_t koff = (k >> 2) * kFBlock + (k & 3) * 32;
                        umma_f16_ss(tmem + C::kColS + sb * 128, sdesc_at(dQ, koff), sdesc_at(dK, koff), kIdS, k > 0);
                    }
                    umma_commit(bar(fSFull0 + sb));
                    if (t == it.kv_hi) umma_commit(bar(fQEmpty));
                }
                __syncwarp();
                if (pend.valid && !(ok = issue_pv(pend))) break;
                pend = Pend{true, t == it.kv_lo, st};
            }
            if (ok && pend.valid) ok = issue_pv(pend);
        }
    } else if (warp >= kFWarpSoft0) {
        // ------------------------------------------------------------ softmax + epilogue
        const int r = tid - kFWarpSoft0 * 32;   // q row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint8_t* sP = sm + C::kP;
        uint32_t s_it = 0, gt = 0;
        bool ok = true;
        // every decision the 128 threads take is the same in all of them, so
        // that they meet the same named barriers
        auto wait_group = [&](int b, uint32_t parity) -> bool { return fbar_and(kFBarSoft, 128, wait(b, parity)); };
        for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
            const FItem it = fdecode(a, cnt, item);
            if (!it.rows) continue;
            const int64_t i = it.q0 + r;
            const bool valid = i < it.s.len_q;
            const bool in_slot = i < it.s.slot_q;
            int64_t k_lo, k_hi;
            row_keys(g, it.s, i, k_lo, k_hi);
            float m = -INFINITY, l = 0.f;
            bool have = it.keys && ok;
            if (have) {
                for (int64_t t = it.kv_lo; t <= it.kv_hi; ++t, ++s_it, ++gt) {
                    const int sb = s_it & 1;
                    if (!(ok = wait_group(fSFull0 + sb, (s_it >> 1) & 1))) break;
                    tc_fence_after();
                    float sv[128];
#pragma unroll
                    for (int cb = 0; cb < 4; ++cb) {
                        uint32_t v[32];
                        tmem_ld32(tmem + C::kColS + sb * 128 + lane_off + cb * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) sv[cb * 32 + e] = __uint_as_float(v[e]);
                    }
                    tc_fence_before();
                    mbar_arrive(bar(fSFree0 + sb));
                    const int64_t c_lo64 = k_lo - t * kTileKV, c_hi64 = k_hi - t * kTileKV;
                    const int c_lo = static_cast<int>(imax64(c_lo64, 0));
                    const int c_hi = static_cast<int>(imin64(c_hi64, 127));
                    float mt = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= c_lo && c <= c_hi) mt = fmaxf(mt, sv[c]);
                    const float m_new = fmaxf(m, mt * a.scale_log2);
                    const float alpha = m_new == m ? 1.f : ex2_approx(m - m_new);
                    float sum = 0.f;
                    uint32_t pk[64];
#pragma unroll
                    for (int c = 0; c < 128; c += 2) {
                        const float p0 = (c >= c_lo && c <= c_hi) ? ex2_approx(fmaf(sv[c], a.scale_log2, -m_new)) : 0.f;
                        const float p1 =
                            (c + 1 >= c_lo && c + 1 <= c_hi) ? ex2_approx(fmaf(sv[c + 1], a.scale_log2, -m_new)) : 0.f;
                        sum += p0 + p1;
                        pk[c >> 1] = fpack2<BF16>(p0, p1);
                    }
                    l = l * alpha + sum;
                    m = m_new;
                    if (t > it.kv_lo) {
                        // the previous P V is done: O is stable and P is free
                        if (!(ok = wait_group(fPvDone, (gt - 1) & 1))) break;
                        tc_fence_after();
                        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                            for (int cb = 0; cb < HD / 32; ++cb) {
                                uint32_t v[32];
                                tmem_ld32(tmem + C::kColO + lane_off + cb * 32, v);
                                tmem_ld_wait();
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    uint32_t w[8];
#pragma unroll
                                    for (int e = 0; e < 8; ++e)
                                        w[e] = __float_as_uint(__uint_as_float(v[8 * q + e]) * alpha);
                                    tmem_st8(tmem + C::kColO + lane_off + cb * 32 + 8 * q, w);
                                }
                            }
                            tmem_st_wait();
                        }
                    } else {
                        // P's buffer held the previous item's O staging: its
                        // store has read it before anyone writes P
                        if (r == 0) bulk_wait_read0();
                        asm volatile("bar.sync %0, %1;" ::"r"(kFBarSoft), "r"(128) : "memory");
                    }
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc)
                        *reinterpret_cast<uint4*>(sP + fswz(r, cc)) =
                            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(fPFull));
                }
                have = ok;
                // the last P V is done: O is final (P's buffer is free)
                if (have) {
                    have = ok = wait_group(fPvDone, (gt - 1) & 1);
                    tc_fence_after();
                }
            }
            // Normaliser with the sink's term; LSE in natural log.
            float m_fin = m, l_tot = l;
            if (a.sink != nullptr && valid && in_bounds(a.status, a.sink + it.h, a.sink, g.ext.sink, 1)) {
                const float sl = a.sink[it.h] * kLog2e;
                if (m == -INFINITY) {
                    m_fin = sl;
                    l_tot = 1.f;
                } else {
                    const float mx = fmaxf(m, sl);
                    l_tot = l * ex2_approx(m - mx) + ex2_approx(sl - mx);
                    m_fin = mx;
                }
            }
            const float o_mul = (valid && have && l_tot > 0.f) ? ex2_approx(m - m_fin) / l_tot : 0.f;
            const float lse = (valid && m_fin != -INFINITY) ? (m_fin + __log2f(l_tot)) * kLn2 : -INFINITY;
            if (in_slot) {
                const int64_t so = thd ? it.h * g.rows_q + it.s.q_row0 + i : (it.bi * g.h_q + it.h) * g.s_q + i;
                if (in_bounds(a.status, a.lse + so, a.lse, g.ext.lse, 1)) a.lse[so] = lse;
            }
            // O row: staged in the TMA layout (P's buffer), stored by TMA, or
            // row-wise for a THD tile that ends past its slot
            const bool use_tma = !thd || it.q0 + kTileQ <= it.s.slot_q;
            uint8_t* stg = sP;
            if (have) {
#pragma unroll 1
                for (int cb = 0; cb < HD / 32; ++cb) {
                    uint32_t v[32];
                    tmem_ld32(tmem + C::kColO + lane_off + cb * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(stg + fswz(r, cb * 4 + q)) = make_uint4(
                            fpack2<BF16>(__uint_as_float(v[8 * q]) * o_mul, __uint_as_float(v[8 * q + 1]) * o_mul),
                            fpack2<BF16>(__uint_as_float(v[8 * q + 2]) * o_mul, __uint_as_float(v[8 * q + 3]) * o_mul),
                            fpack2<BF16>(__uint_as_float(v[8 * q + 4]) * o_mul, __uint_as_float(v[8 * q + 5]) * o_mul),
                            fpack2<BF16>(__uint_as_float(v[8 * q + 6]) * o_mul, __uint_as_float(v[8 * q + 7]) * o_mul));
                }
                tc_fence_before();
                mbar_arrive(bar(fOEmpty));
            } else {
                // no key for any row (or an abort): O = 0; the staging may hold
                // the previous item's O until its store has read it
                if (r == 0) bulk_wait_read0();
                asm volatile("bar.sync %0, %1;" ::"r"(kFBarSoft), "r"(128) : "memory");
#pragma unroll
                for (int cc = 0; cc < HD / 8; ++cc) *reinterpret_cast<uint4*>(stg + fswz(r, cc)) = make_uint4(0u, 0u, 0u, 0u);
            }
            if (use_tma) fence_proxy_async_smem();
            asm volatile("bar.sync %0, %1;" ::"r"(kFBarSoft), "r"(128) : "memory");
            if (use_tma) {
                if (r == 0) {
                    const int qrow = static_cast<int>((thd ? it.s.q_row0 : 0) + it.q0);
#pragma unroll
                    for (int cb = 0; cb < HD / 64; ++cb)
                        ftma_store(sbase + C::kP + cb * kFBlock, &a.tm_o, thd, cb * 64, static_cast<int>(it.h), qrow,
                                   static_cast<int>(it.bi));
                    bulk_commit();
                }
            } else if (in_slot) {
                uint16_t* dst = static_cast<uint16_t*>(a.o) + (it.s.q_row0 + i) * a.o_stride[1] + it.h * a.o_stride[2];
                if (in_bounds(a.status, dst, a.o, g.ext.o, HD)) {
#pragma unroll
                    for (int cc = 0; cc < HD / 8; ++cc)
                        *reinterpret_cast<uint4*>(dst + cc * 8) = *reinterpret_cast<const uint4*>(stg + fswz(r, cc));
                }
            }
        }
    }

    bulk_wait0();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ----------------------------------------------------------------------------
// d = 64: two q-tiles in flight.
//
// Two slots, each with its own Q tile, S (TMEM columns 128 s ..), O (TMEM
// columns 256 + 64 s ..), double-buffered P and softmax warpgroup, share the
// producer, the MMA warp and the 2-stage K/V ring. The CTA's n-th work item
// goes to slot n % 2, and the producer and the MMA warp walk the two slots'
// kv steps alternately: the MMA warp issues S of one slot before P V of the
// other, so the tensor core works for one group while the other runs its
// softmax, and every SM sub-partition has two softmax warps to interleave.
// 384 threads: warp 0 producer, warp 1 MMA issuer, warps 2-3 idle, warps 4-7
// slot 0, warps 8-11 slot 1. At 168 registers a thread, a softmax thread reads
// its S row in 32-column chunks, twice (row maximum, then exponentials);
// chunks the mask excludes for the whole warp are skipped.
namespace {

constexpr int kPThreads = 384;
constexpr int kPWarpSoft0 = 4;

struct PCfg {
    static constexpr uint32_t kTile = 128 * 64 * 2;   // one 128-row tile of 64 16-bit features
    static constexpr uint32_t kQ = 0;                  // 2 slots
    static constexpr uint32_t kK = kQ + 2 * kTile;     // 2 stages
    static constexpr uint32_t kV = kK + 2 * kTile;     // 2 stages
    static constexpr uint32_t kP = kV + 2 * kTile;     // [slot][buffer] P [128 q x 128 kv]; buffer 0 stages O
    static constexpr uint32_t kBars = kP + 4 * 32768;
    static constexpr uint32_t kMisc = kBars + 256;     // tmem slot, abort flag
    static constexpr uint32_t kBytes = kMisc + 64;
    static_assert(kBytes <= 232448, "shared memory above the 227 KB a CTA may opt into");
};

// mbarriers: per-slot ones at index + slot
enum PBar : int {
    pQFull = 0, pQEmpty = 2, pSFull = 4, pSFree = 6, pPFull = 8, pPvDone = 10, pOEmpty = 12,
    pKvFull0 = 14, pKvFull1, pKvEmpty0, pKvEmpty1, pNumBars
};
static_assert(pNumBars * 8 <= 256, "mbarrier area");

// A slot's walk over its work items that have keys: the n-th item of the CTA
// goes to slot n % 2.
struct SlotWalk {
    int64_t n;   // local index of the next item to decode
    FItem it;    // current item
    int64_t t;   // current kv-tile
    bool live;   // a step is pending
};

__device__ __forceinline__ void slot_next(const FwdArgs& a, const FCounts& cnt, int64_t n_items, SlotWalk& w)
{
    for (;;) {
        const int64_t item = blockIdx.x + w.n * static_cast<int64_t>(gridDim.x);
        if (item >= n_items) {
            w.live = false;
            return;
        }
        w.it = fdecode(a, cnt, item);
        w.n += 2;
        if (w.it.keys) {
            w.t = w.it.kv_lo;
            w.live = true;
            return;
        }
    }
}

// The next step of the alternating walk: slot `cur` unless it is done.
__device__ __forceinline__ int pick_slot(const SlotWalk (&w)[2], int cur)
{
    if (w[cur].live) return cur;
    if (w[cur ^ 1].live) return cur ^ 1;
    return -1;
}

__device__ __forceinline__ void slot_advance(const FwdArgs& a, const FCounts& cnt, int64_t n_items, SlotWalk& w)
{
    if (w.t == w.it.kv_hi) slot_next(a, cnt, n_items, w);
    else ++w.t;
}

}  // namespace

template <bool BF16>
__global__ void __launch_bounds__(kPThreads, 1) sdpa_fwd_pp_kernel(const __grid_constant__ FwdArgs a)
{
    using C = PCfg;
    constexpr int HD = 64;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) set_status(a.status, kStatusUnsupported);
        return;
    }
    uint8_t* sm = smem_raw;
    const uint32_t sbase = smem_u32(sm);
    auto bar = [&](int i) -> uint32_t { return sbase + C::kBars + 8u * i; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::kMisc);  // [0] tmem base, [1] abort flag

    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint64_t tmo = static_cast<uint64_t>(a.timeout_ns);
    const int64_t n_items = g.b * g.h_q * a.n_q_tiles;
    const bool thd = g.layout == 1;
    const FCounts cnt{static_cast<uint32_t>(g.h_q), static_cast<uint32_t>(a.n_q_tiles),
                      static_cast<uint32_t>(g.h_q / g.h_kv)};

    if (tid == 0) {
        misc[1] = 0;
        for (int sl = 0; sl < 2; ++sl) {
            mbar_init(bar(pQFull + sl), 1);
            mbar_init(bar(pQEmpty + sl), 1);
            mbar_init(bar(pSFull + sl), 1);
            mbar_init(bar(pSFree + sl), 128);
            mbar_init(bar(pPFull + sl), 128);
            mbar_init(bar(pPvDone + sl), 1);
            mbar_init(bar(pOEmpty + sl), 128);
            mbar_init(bar(pKvFull0 + sl), 1);
            mbar_init(bar(pKvEmpty0 + sl), 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + C::kMisc, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    volatile uint32_t* abort_flag = misc + 1;

    auto wait = [&](int b, uint32_t parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait(bar(b), parity, tmo)) return true;
        *abort_flag = 1;
        set_status(a.status, kStatusTimeout);
        return false;
    };
    auto wait_warp = [&](int b, uint32_t parity) -> bool { return __all_sync(0xffffffffu, wait(b, parity)); };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            SlotWalk w[2];
            w[0].n = 0;
            w[1].n = 1;
            slot_next(a, cnt, n_items, w[0]);
            slot_next(a, cnt, n_items, w[1]);
            uint32_t kv_it = 0, q_cnt[2] = {0u, 0u};
            for (int cur = 0;;) {
                const int sl = pick_slot(w, cur);
                if (sl < 0) break;
                const FItem& it = w[sl].it;
                const int64_t t = w[sl].t;
                if (t == it.kv_lo) {
                    if (!wait(pQEmpty + sl, (q_cnt[sl] & 1) ^ 1)) break;
                    ++q_cnt[sl];
                    mbar_arrive_expect_tx(bar(pQFull + sl), C::kTile);
                    ftma_tile<HD>(sbase + C::kQ + sl * C::kTile, &a.tm_q, bar(pQFull + sl), thd,
                                  static_cast<int>(it.h), static_cast<int>((thd ? it.s.q_row0 : 0) + it.q0),
                                  static_cast<int>(it.bi));
                }
                const int st = kv_it & 1;
                if (!wait(pKvEmpty0 + st, ((kv_it >> 1) & 1) ^ 1)) break;
                ++kv_it;
                const int row = static_cast<int>((thd ? it.s.kv_row0 : 0) + t * kTileKV);
                mbar_arrive_expect_tx(bar(pKvFull0 + st), 2 * C::kTile);
                ftma_tile<HD>(sbase + C::kK + st * C::kTile, &a.tm_k, bar(pKvFull0 + st), thd, static_cast<int>(it.g),
                              row, static_cast<int>(it.bi));
                ftma_tile<HD>(sbase + C::kV + st * C::kTile, &a.tm_v, bar(pKvFull0 + st), thd, static_cast<int>(it.g),
                              row, static_cast<int>(it.bi));
                slot_advance(a, cnt, n_items, w[sl]);
                cur = sl ^ 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t kIdS = idesc_f16(BF16, 128, 128, false, false);
        constexpr uint32_t kIdPV = idesc_f16(BF16, 128, HD, false, true);
        SlotWalk w[2];
        w[0].n = 0;
        w[1].n = 1;
        slot_next(a, cnt, n_items, w[0]);
        slot_next(a, cnt, n_items, w[1]);
        uint32_t kv_it = 0, q_cnt[2] = {0u, 0u}, s_cnt[2] = {0u, 0u}, p_cnt[2] = {0u, 0u}, o_cnt[2] = {0u, 0u};
        struct Pend {
            bool valid, first;
            int sl, st;
        };
        // O += P V for a step whose softmax has written P
        auto issue_pv = [&](const Pend& pd) -> bool {
            if (!wait_warp(pPFull + pd.sl, p_cnt[pd.sl] & 1)) return false;
            const uint32_t pbuf = p_cnt[pd.sl] & 1;
            ++p_cnt[pd.sl];
            // the first P V of an item overwrites O: the epilogue has read it
            if (pd.first) {
                if (!wait_warp(pOEmpty + pd.sl, (o_cnt[pd.sl] & 1) ^ 1)) return false;
                ++o_cnt[pd.sl];
            }
            tc_fence_after();
            const uint64_t dP = sdesc_sw128(sbase + C::kP + (pd.sl * 2 + pbuf) * 32768u, 16, 1024);
            const uint64_t dV = sdesc_sw128(sbase + C::kV + pd.st * C::kTile, kFBlock, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t aoff = (k >> 2) * kFBlock + (k & 3) * 32;
                umma_f16_ss(tmem + 256 + pd.sl * HD, sdesc_at(dP, aoff), sdesc_at(dV, k * 2048), kIdPV,
                            (pd.first && k == 0) ? 0u : 1u);
            }
            umma_commit(bar(pPvDone + pd.sl));
            umma_commit(bar(pKvEmpty0 + pd.st));
            __syncwarp();
            return true;
        };
        Pend pend{false, false, 0, 0};
        bool ok = true;
        for (int cur = 0; ok;) {
            const int sl = pick_slot(w, cur);
            if (sl < 0) break;
            const FItem& it = w[sl].it;
            const int64_t t = w[sl].t;
            if (t == it.kv_lo) {
                if (!(ok = wait_warp(pQFull + sl, q_cnt[sl] & 1))) break;
                ++q_cnt[sl];
            }
            const int st = kv_it & 1;
            if (!(ok = wait_warp(pKvFull0 + st, (kv_it >> 1) & 1))) break;
            ++kv_it;
            // keys past the sequence's length are masked out of P, but their V
            // rows meet P's zeros in the product: make them zero too
            if (t * kTileKV + kTileKV > it.s.len_kv)
                fzero_tail<HD>(sm + C::kV + st * C::kTile, it.s.len_kv - t * kTileKV, lane);
            if (!(ok = wait_warp(pSFree + sl, (s_cnt[sl] & 1) ^ 1))) break;
            ++s_cnt[sl];
            tc_fence_after();
            const uint64_t dQ = sdesc_sw128(sbase + C::kQ + sl * C::kTile, 16, 1024);
            const uint64_t dK = sdesc_sw128(sbase + C::kK + st * C::kTile, 16, 1024);
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint32_t koff = (k >> 2) * kFBlock + (k & 3) * 32;
                umma_f16_ss(tmem + sl * 128, sdesc_at(dQ, koff), sdesc_at(dK, koff), kIdS, k > 0);
            }
            umma_commit(bar(pSFull + sl));
            if (t == it.kv_hi) umma_commit(bar(pQEmpty + sl));
            __syncwarp();
            if (pend.valid && !(ok = issue_pv(pend))) break;
            pend = Pend{true, t == it.kv_lo, sl, st};
            slot_advance(a, cnt, n_items, w[sl]);
            cur = sl ^ 1;
        }
        if (ok && pend.valid) issue_pv(pend);
    } else if (warp >= kPWarpSoft0) {
        // ------------------------------------------------------------ softmax + epilogue
        const int sl = (warp - kPWarpSoft0) >> 2;          // slot
        const int gbar = 1 + sl;                           // the group's named barrier
        const int r = tid - (kPWarpSoft0 + 4 * sl) * 32;   // q row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tm_s = tmem + sl * 128 + lane_off, tm_o = tmem + 256 + sl * HD + lane_off;
        uint8_t* sP = sm + C::kP + sl * 2 * 32768u;        // this slot's two P buffers; buffer 0 stages O
        uint32_t s_it = 0, gt = 0;
        bool ok = true;
        auto wait_group = [&](int b, uint32_t parity) -> bool { return fbar_and(gbar, 128, wait(b, parity)); };
        for (int64_t n = sl;; n += 2) {
            const int64_t item = blockIdx.x + n * static_cast<int64_t>(gridDim.x);
            if (item >= n_items) break;
            const FItem it = fdecode(a, cnt, item);
            if (!it.rows) continue;
            const int64_t i = it.q0 + r;
            const bool valid = i < it.s.len_q;
            const bool in_slot = i < it.s.slot_q;
            int64_t k_lo, k_hi;
            row_keys(g, it.s, i, k_lo, k_hi);
            float m = -INFINITY, l = 0.f;
            bool have = it.keys && ok;
            if (have) {
                // the previous item's O store has read the staging (P buffer 0)
                if (r == 0) bulk_wait_read0();
                asm volatile("bar.sync %0, %1;" ::"r"(gbar), "r"(128) : "memory");
                for (int64_t t = it.kv_lo; t <= it.kv_hi; ++t, ++s_it, ++gt) {
                    if (!(ok = wait_group(pSFull + sl, s_it & 1))) break;
                    tc_fence_after();
                    const int64_t c_lo64 = k_lo - t * kTileKV, c_hi64 = k_hi - t * kTileKV;
                    const int c_lo = static_cast<int>(imax64(imin64(c_lo64, 128), -1));
                    const int c_hi = static_cast<int>(imin64(imax64(c_hi64, -1), 127));
                    // pass 1: row maximum over the admitted columns
                    float mt = -INFINITY;
#pragma unroll 1
                    for (int cb = 0; cb < 4; ++cb) {
                        const int c0 = cb * 32;
                        if (__all_sync(0xffffffffu, c_hi < c0 || c_lo > c0 + 31)) continue;
                        uint32_t v[32];
                        tmem_ld32(tm_s + c0, v);
                        tmem_ld_wait();
                        float x[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) x[q] = -INFINITY;
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int c = c0 + e;
                            if (c >= c_lo && c <= c_hi) x[e & 7] = fmaxf(x[e & 7], __uint_as_float(v[e]));
                        }
                        mt = fmaxf(mt, fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                                             fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7]))));
                    }
                    const float m_new = fmaxf(m, mt * a.scale_log2);
                    const float alpha = m_new == m ? 1.f : ex2_approx(m - m_new);
                    // pass 2: P = exp2(s * scale * log2 e - m), 16-bit, into this
                    // step's P buffer (the P V two steps back has read it)
                    uint8_t* pb = sP + (gt & 1) * 32768u;
                    float sum = 0.f;
#pragma unroll 1
                    for (int cb = 0; cb < 4; ++cb) {
                        const int c0 = cb * 32;
                        uint32_t pk[16];
                        if (__all_sync(0xffffffffu, c_hi < c0 || c_lo > c0 + 31)) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) pk[e] = 0u;
                        } else {
                            uint32_t v[32];
                            tmem_ld32(tm_s + c0, v);
                            tmem_ld_wait();
                            float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const int c = c0 + e;
                                const float p0 = (c >= c_lo && c <= c_hi)
                                                     ? ex2_approx(fmaf(__uint_as_float(v[e]), a.scale_log2, -m_new))
                                                     : 0.f;
                                const float p1 = (c + 1 >= c_lo && c + 1 <= c_hi)
                                                     ? ex2_approx(fmaf(__uint_as_float(v[e + 1]), a.scale_log2, -m_new))
                                                     : 0.f;
                                ps[(e >> 1) & 3] += p0 + p1;
                                pk[e >> 1] = fpack2<BF16>(p0, p1);
                            }
                            sum += (ps[0] + ps[1]) + (ps[2] + ps[3]);
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4*>(pb + fswz(r, cb * 4 + q)) =
                                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                    }
                    // S has been read: the next S of this slot may overwrite it
                    tc_fence_before();
                    mbar_arrive(bar(pSFree + sl));
                    l = l * alpha + sum;
                    m = m_new;
                    if (t > it.kv_lo) {
                        // the previous P V is done: O is stable for the rescale
                        if (!(ok = wait_group(pPvDone + sl, (gt - 1) & 1))) break;
                        tc_fence_after();
                        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                            for (int cb = 0; cb < HD / 32; ++cb) {
                                uint32_t v[32];
                                tmem_ld32(tm_o + cb * 32, v);
                                tmem_ld_wait();
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    uint32_t w8[8];
#pragma unroll
                                    for (int e = 0; e < 8; ++e)
                                        w8[e] = __float_as_uint(__uint_as_float(v[8 * q + e]) * alpha);
                                    tmem_st8(tm_o + cb * 32 + 8 * q, w8);
                                }
                            }
                            tmem_st_wait();
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(pPFull + sl));
                }
                have = ok;
                // the last P V is done: O is final
                if (have) {
                    have = ok = wait_group(pPvDone + sl, (gt - 1) & 1);
                    tc_fence_after();
                }
            }
            // Normaliser with the sink's term; LSE in natural log.
            float m_fin = m, l_tot = l;
            if (a.sink != nullptr && valid && in_bounds(a.status, a.sink + it.h, a.sink, g.ext.sink, 1)) {
                const float sk = a.sink[it.h] * kLog2e;
                if (m == -INFINITY) {
                    m_fin = sk;
                    l_tot = 1.f;
                } else {
                    const float mx = fmaxf(m, sk);
                    l_tot = l * ex2_approx(m - mx) + ex2_approx(sk - mx);
                    m_fin = mx;
                }
            }
            const float o_mul = (valid && have && l_tot > 0.f) ? ex2_approx(m - m_fin) / l_tot : 0.f;
            const float lse = (valid && m_fin != -INFINITY) ? (m_fin + __log2f(l_tot)) * kLn2 : -INFINITY;
            if (in_slot) {
                const int64_t so = thd ? it.h * g.rows_q + it.s.q_row0 + i : (it.bi * g.h_q + it.h) * g.s_q + i;
                if (in_bounds(a.status, a.lse + so, a.lse, g.ext.lse, 1)) a.lse[so] = lse;
            }
            // O row: staged in the TMA layout (P buffer 0), stored by TMA, or
            // row-wise for a THD tile that ends past its slot
            const bool use_tma = !thd || it.q0 + kTileQ <= it.s.slot_q;
            uint8_t* stg = sP;
            if (have) {
#pragma unroll 1
                for (int cb = 0; cb < HD / 32; ++cb) {
                    uint32_t v[32];
                    tmem_ld32(tm_o + cb * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(stg + fswz(r, cb * 4 + q)) = make_uint4(
                            fpack2<BF16>(__uint_as_float(v[8 * q]) * o_mul, __uint_as_float(v[8 * q + 1]) * o_mul),
                            fpack2<BF16>(__uint_as_float(v[8 * q + 2]) * o_mul, __uint_as_float(v[8 * q + 3]) * o_mul),
                            fpack2<BF16>(__uint_as_float(v[8 * q + 4]) * o_mul, __uint_as_float(v[8 * q + 5]) * o_mul),
                            fpack2<BF16>(__uint_as_float(v[8 * q + 6]) * o_mul, __uint_as_float(v[8 * q + 7]) * o_mul));
                }
                tc_fence_before();
                mbar_arrive(bar(pOEmpty + sl));
            } else {
                // no key for any row (or an abort): O = 0; the staging may hold
                // the previous item's O until its store has read it
                if (r == 0) bulk_wait_read0();
                asm volatile("bar.sync %0, %1;" ::"r"(gbar), "r"(128) : "memory");
#pragma unroll
                for (int cc = 0; cc < HD / 8; ++cc)
                    *reinterpret_cast<uint4*>(stg + fswz(r, cc)) = make_uint4(0u, 0u, 0u, 0u);
            }
            if (use_tma) fence_proxy_async_smem();
            asm volatile("bar.sync %0, %1;" ::"r"(gbar), "r"(128) : "memory");
            if (use_tma) {
                if (r == 0) {
                    ftma_store(sbase + C::kP + sl * 2 * 32768u, &a.tm_o, thd, 0, static_cast<int>(it.h),
                               static_cast<int>((thd ? it.s.q_row0 : 0) + it.q0), static_cast<int>(it.bi));
                    bulk_commit();
                }
            } else if (in_slot) {
                uint16_t* dst = static_cast<uint16_t*>(a.o) + (it.s.q_row0 + i) * a.o_stride[1] + it.h * a.o_stride[2];
                if (in_bounds(a.status, dst, a.o, g.ext.o, HD)) {
#pragma unroll
                    for (int cc = 0; cc < HD / 8; ++cc)
                        *reinterpret_cast<uint4*>(dst + cc * 8) = *reinterpret_cast<const uint4*>(stg + fswz(r, cc));
                }
            }
        }
    }

    bulk_wait0();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int HD, bool BF16>
static cudaError_t launch_fwd_typed(const FwdArgs& a, cudaStream_t s)
{
    auto kern = sdpa_fwd_kernel<HD, BF16>;
    const uint32_t bytes = FCfg<HD>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    const int64_t items = a.g.b * a.g.h_q * a.n_q_tiles;
    if (items == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t grid = items < sms ? items : sms;
    kern<<<static_cast<unsigned>(grid), kFThreads, bytes, s>>>(a);
    return cudaGetLastError();
}

template <bool BF16>
static cudaError_t launch_fwd_pp(const FwdArgs& a, cudaStream_t s)
{
    auto kern = sdpa_fwd_pp_kernel<BF16>;
    const uint32_t bytes = PCfg::kBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    const int64_t items = a.g.b * a.g.h_q * a.n_q_tiles;
    if (items == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // two items in flight per CTA
    const int64_t want = (items + 1) / 2;
    const int64_t grid = want < sms ? want : sms;
    kern<<<static_cast<unsigned>(grid), kPThreads, bytes, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdArgs& a, int dtype, cudaStream_t s)
{
    if (a.g.d == 64) return dtype == 0 ? launch_fwd_pp<true>(a, s) : launch_fwd_pp<false>(a, s);
    return dtype == 0 ? launch_fwd_typed<128, true>(a, s) : launch_fwd_typed<128, false>(a, s);
}

}  // namespace swa
