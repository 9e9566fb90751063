// aux_kernels.cu -- the two HBM-bound kernels around the main backward:
//  * preprocess ("dot"): D = rowsum(dO * O) in fp32, zero the relay / visit
//    counters and the status word, dSink partials;
//  * dq_convert ("cvt"): the main kernel already stored dQ (converted by each
//    q-tile's last visitor); this writes dQ = 0 on the rows no kv-tile visits
//    (padding, gap tokens, rows outside every window), converts the q-tiles
//    that took unordered atomics, sums (in visitor order) and converts those
//    whose visitors stored per-visitor partials (deterministic mode), and
//    finishes dSink.
// Both move 16-byte vectors per thread with consecutive threads on
// consecutive 16-byte pieces of a row, so every warp access is coalesced.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sdpa_internal.h"
#include "seq.cuh"

namespace swa {

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            float2 t = __half22float2(h);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
}

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

template <bool BF16>
__device__ __forceinline__ uint4 pack8(const float (&f)[8])
{
    return make_uint4(pack2<BF16>(f[0], f[1]), pack2<BF16>(f[2], f[3]), pack2<BF16>(f[4], f[5]),
                      pack2<BF16>(f[6], f[7]));
}

// ---------------------------------------------------------------- preprocess
// Persistent CTAs (one per SM) walk blocks of pre_rows token rows x pre_heads
// q-heads (block = (sequence, row block, head chunk), head chunk fastest). The
// TMA engine stages each block's O and dO boxes in a 3-stage shared-memory
// ring; each thread then reduces one (row, head) unit of HD features (d = 64)
// or half of one (d = 128) from shared memory. The per-element work of the
// register path (address arithmetic per 16 bytes, cross-thread reductions)
// made it issue-bound at about half the HBM bandwidth. Every row of every
// q-tile is covered: rows past the length get the statistics that make P = 0.
// Bytes of the ring (stages of an O box and a dO box): 192 KB with one CTA
// per SM, 64 KB with three. Three CTAs of two stages each keep as many bytes in
// flight as one CTA of six, and one CTA's wait-reduce-reissue turn overlaps the
// others' (THD b16 h64: 201 us against 258; b2 h16 S8192: 16.6 against
// 18.9 us). Small problems (fewer than four blocks per CTA at three per SM)
// keep one CTA per SM.
constexpr uint32_t kPreRingOne = 196608, kPreRingThree = 65536;
constexpr int kPreMaxStages = 8;

__device__ __forceinline__ void pre_tma_load(uint32_t dst, const CUtensorMap* map, uint32_t bar, bool thd,
                                             int head, int row, int batch)
{
    if (thd)
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(head), "r"(row)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(head), "r"(row), "r"(batch)
            : "memory");
}

template <int HD, bool BF16>
__global__ void __launch_bounds__(256, 3) preprocess_kernel(const __grid_constant__ PreArgs a)
{
    constexpr int TPU = HD / 64;   // threads per (row, head) unit, 128 B each
    extern __shared__ __align__(1024) uint8_t smem[];
    // [stage][O box | dO box], dSink row terms [2][256] fp32, mbarriers
    const uint32_t ring = a.ring_bytes;
    float* red = reinterpret_cast<float*>(smem + ring);
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 127u) {   // TMA destinations need 128-byte alignment
        if (threadIdx.x == 0) set_status(a.status, kStatusUnsupported);
        return;
    }
    const uint32_t bars = sbase + ring + 2 * 256 * 4;
    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    const bool thd = g.layout == 1;
    const bool with_sink = a.sink != nullptr;
    const int hc_n = a.pre_heads, rows_n = a.pre_rows;
    const int units = hc_n * rows_n;
    const uint32_t box_bytes = static_cast<uint32_t>(units) * HD * 2;
    // block counts fit 32 bits (the host checks): no 64-bit divisions here
    const uint32_t nrb = static_cast<uint32_t>(a.stats_row / rows_n);   // row blocks per sequence
    const uint32_t nhc = static_cast<uint32_t>((g.h_q + hc_n - 1) / hc_n);   // head chunks
    const uint32_t n_items = static_cast<uint32_t>(g.b) * nrb * nhc;
    // as many ring stages as boxes of this size fit
    const uint32_t stage_bytes = 2 * box_bytes;
    const int n_stages = static_cast<int>(min(ring / stage_bytes, static_cast<uint32_t>(kPreMaxStages)));

    // relay / visit counters, ticket and status: zeroed by the whole grid
    {
        const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
        const int64_t id = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid;
        for (int64_t k = id; k < a.n_sems; k += nthr) a.sems[k] = 0;
        if (id == 0) {
            a.status[0] = 0;
            a.status[1] = 0;
        }
    }
    if (tid == 0) {
        for (int st = 0; st < n_stages; ++st) mbar_init(bars + 8u * st, 1);
        fence_mbar_init();
    }
    __syncthreads();

    struct Blk {
        uint32_t bi, rb, hc;
    };
    auto coords = [&](uint32_t item) -> Blk {
        const uint32_t rest = item / nhc;
        return Blk{rest / nrb, rest % nrb, item - rest * nhc};
    };
    // thread 0: stage the O and dO boxes of `item` into ring entry `st`
    auto issue = [&](uint32_t item, int st) {
        const Blk b = coords(item);
        const int64_t row0 = thd ? g.q_offsets[b.bi] : 0;
        const int row = static_cast<int>(row0 + b.rb * rows_n);
        const uint32_t bar = bars + 8u * st;
        mbar_arrive_expect_tx(bar, 2 * box_bytes);
        const uint32_t dst = sbase + st * stage_bytes;
        pre_tma_load(dst, &a.tm_o, bar, thd, static_cast<int>(b.hc * hc_n), row, static_cast<int>(b.bi));
        pre_tma_load(dst + box_bytes, &a.tm_do, bar, thd, static_cast<int>(b.hc * hc_n), row, static_cast<int>(b.bi));
    };
    if (tid == 0)
        for (int st = 0; st < n_stages; ++st) {
            const uint32_t item = blockIdx.x + st * gridDim.x;
            if (item < n_items) issue(item, st);
        }
    // the main kernel may start its prologue (it waits for this grid before
    // reading anything written here)
    grid_dep_launch();

    const int u = tid / TPU, half = tid % TPU;
    const int r = u / hc_n, hl = u - r * hc_n;   // this thread's unit in every block
    const bool in_box = u < units;
    int j = 0;
    int st = 0;
    uint32_t phase = 0;
    for (uint32_t item = blockIdx.x; item < n_items; item += gridDim.x, ++j) {
        const Blk b = coords(item);
        const SeqInfo s = seq_info(g, b.bi);
        const int64_t h = static_cast<int64_t>(b.hc) * hc_n + hl;
        const int64_t i = static_cast<int64_t>(b.rb) * rows_n + r;
        const bool unit = in_box && h < g.h_q;       // a (row, head) of the slot's row space
        const bool valid = unit && i < s.len_q;
        // the row's LSE, loaded before the wait for the box
        float lse = -INFINITY;
        if (valid && half == 0)
        {
            const float* pl = a.lse + (thd ? h * g.rows_q + s.q_row0 + i : (b.bi * g.h_q + h) * g.s_q + i);
            if (in_bounds(a.status, pl, a.lse, g.ext.lse, 1)) lse = __ldg(pl);
        }
        // q-tiles with three or more visitors take unordered atomics (unless
        // deterministic): their accumulator rows start at zero
        bool zero_acc = false;
        if (!a.deterministic && b.rb * rows_n < s.len_q) {
            int64_t first, n;
            q_tile_visitors(g, s, (b.rb * rows_n) / kTileQ, first, n);
            zero_acc = n >= 3;
        }
        const bool got = __syncthreads_and(mbar_wait(bars + 8u * st, phase, 2000000000ull));
        if (!got) {
            if (tid == 0) set_status(a.status, kStatusTimeout);
            return;
        }
        float part = 0.f;
        if (in_box) {
            const uint8_t* po = smem + st * stage_bytes + u * (HD * 2) + half * 128;
            const uint8_t* pd = po + box_bytes;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                // rotated chunk order: the 8 threads sharing a 128-byte line
                // read different banks
                const int c = (k + tid) & 7;
                float fo[8], fd[8];
                unpack8<BF16>(*reinterpret_cast<const uint4*>(po + c * 16), fo);
                unpack8<BF16>(*reinterpret_cast<const uint4*>(pd + c * 16), fd);
#pragma unroll
                for (int e = 0; e < 8; ++e) part = fmaf(fo[e], fd[e], part);
            }
        }
        if constexpr (TPU == 2) part += __shfl_xor_sync(0xffffffffu, part, 1);
        if (zero_acc && valid) {
            float* zf = a.dq_acc + ((s.q_row0 + i) * g.h_q + h) * HD + half * 64;
            float4* z = reinterpret_cast<float4*>(zf);
            if (in_bounds(a.status, zf, a.dq_acc, g.ext.dq_acc, 64)) {
#pragma unroll
                for (int k = 0; k < 16; ++k) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (unit && half == 0) {
            // per-row statistics for the main kernel, one slot for every row of
            // every q-tile: -LSE * log2(e) and -D in the tile's two 128-float
            // runs; rows past the length or that attend nothing get (-inf, 0)
            // so that P = 0 there
            float nl2 = -INFINITY, ds = 0.f;
            if (valid && lse != -INFINITY) {
                nl2 = -(lse * 1.4426950408889634f);
                if (with_sink && in_bounds(a.status, a.sink + h, a.sink, g.ext.sink, 1))
                    ds = -expf(a.sink[h] - lse) * part;
            }
            float* srow = a.stats + 2 * ((b.bi * g.h_q + h) * a.stats_row + (i & ~int64_t(kTileQ - 1))) + (i & (kTileQ - 1));
            if (in_bounds(a.status, srow, a.stats, g.ext.stats, kTileQ + 1)) {
                srow[0] = nl2;
                srow[kTileQ] = valid ? -part : 0.f;
            }
            if (with_sink) red[(j & 1) * 256 + hl * rows_n + r] = ds;
        }
        __syncthreads();   // ring entry st is read; dSink terms are written
        if (tid == 0) {
            const uint32_t next = item + n_stages * gridDim.x;
            if (next < n_items) issue(next, st);
        }
        if (with_sink && tid < hc_n && b.hc * hc_n + tid < g.h_q) {
            // this block's dSink partial of a head: its rows summed in order
            float t = 0.f;
            for (int k = 0; k < rows_n; ++k) t += red[(j & 1) * 256 + tid * rows_n + k];
            float* pd = a.dsink_part + (b.hc * hc_n + tid) * a.n_row_blocks + static_cast<int64_t>(b.bi) * nrb + b.rb;
            if (in_bounds(a.status, pd, a.dsink_part, g.ext.dsink_part, 1)) *pd = t;
        }
        if (++st == n_stages) {
            st = 0;
            phase ^= 1u;
        }
    }
}

// ---------------------------------------------------------------- convert
// The main kernel already stored dQ for every q-tile some kv-tile visits (its
// last visitor converts). This writes dQ = 0 on the other rows of a slot:
// rows past the sequence's length and q-tiles no kv-tile visits; converts the
// q-tiles whose visitors added with unordered atomics, and sums (in visitor
// order) and converts those whose visitors stored per-visitor partials. It
// also finishes dSink in a fixed order.
// Persistent: CTA c walks the units c, c + grid, ... of (sequence, q-tile,
// chunk of head_chunk q-heads), chunk fastest. A unit reads its sequence's
// lengths and visitor run once and then moves all of its (row, head) pieces
// as one flat, coalesced range ([row][head][d] rows hold every head side by
// side), four 32-byte loads in flight per thread.
template <int HD, bool BF16>
__global__ void __launch_bounds__(256) dq_convert_kernel(const CvtArgs a)
{
    constexpr int TPR = HD / 8;         // threads per (row, head): 8 values each
    constexpr int kBatch = 4;
    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    grid_dep_wait();   // the main kernel's dQ, partials and the dSink partials
    if (a.dsink != nullptr) {
        // fixed-order finish, one CTA per head: thread t sums partials t,
        // t + 256, ... in order (eight loads in flight at a time), then a fixed
        // butterfly in each warp and the eight warp sums in warp order; bitwise
        // repeatable for a given problem
        __shared__ float wsum[8];
        const int lane = tid & 31, wid = tid >> 5;
        for (int64_t hh = blockIdx.x; hh < g.h_q; hh += gridDim.x) {
            const float* src = a.dsink_part + hh * a.n_row_blocks;
            float t = 0.f;
#pragma unroll 1
            for (int64_t k0 = tid; k0 < a.n_row_blocks; k0 += 8 * 256) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int64_t k = k0 + q * 256;
                    v[q] = (k < a.n_row_blocks && in_bounds(a.status, src + k, a.dsink_part, g.ext.dsink_part, 1))
                               ? src[k] : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) t += v[q];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
            if (lane == 0) wsum[wid] = t;
            __syncthreads();
            if (tid == 0) {
                float s = 0.f;
                for (int w = 0; w < 8; ++w) s += wsum[w];
                a.dsink[hh] = s;
            }
            __syncthreads();
        }
    }
    const bool thd = g.layout == 1;
    uint16_t* dq = static_cast<uint16_t*>(a.dq);
    const uint32_t hq = static_cast<uint32_t>(g.h_q), nx = static_cast<uint32_t>(a.n_q_tiles);
    const uint32_t hc = static_cast<uint32_t>(a.head_chunk);
    const uint32_t nhc = (hq + hc - 1) / hc;
    const uint32_t n_units = nhc * nx * static_cast<uint32_t>(g.b);
    for (uint32_t u = blockIdx.x; u < n_units; u += gridDim.x) {
        const uint32_t rest = u / nhc, bq = rest / nx;
        const uint32_t h0 = (u - rest * nhc) * hc, j = rest - bq * nx;
        const uint32_t nh = min(hc, hq - h0);
        const int64_t bi = bq;
        const SeqInfo s = seq_info(g, bi);
        const int64_t t0 = static_cast<int64_t>(j) * kTileQ;
        const int64_t t1 = imin(t0 + kTileQ, s.slot_q);
        if (t0 >= t1) continue;
        int64_t z0 = t0;  // first row to zero
        bool accumulated = false, from_slots = false;
        int64_t n_vis = 0;
        if (t0 < s.len_q) {
            int64_t first;
            q_tile_visitors(g, s, j, first, n_vis);
            if (n_vis > 0) z0 = s.len_q;
            accumulated = n_vis >= 3 && !a.deterministic;
            from_slots = n_vis >= 3 && a.deterministic && a.n_slots > 0;
        }
        const int64_t e1 = imin(t1, s.len_q);
        const uint32_t per_row = nh * TPR;   // pieces of one row
        // piece k of rows [r0, ...): row r0 + k / per_row, head h0 + (k / TPR) % nh, column block k % TPR
        auto dst_of = [&](int64_t i, uint32_t h, uint32_t c) {
            return dq + (thd ? (s.q_row0 + i) * a.dq_stride[1] : bi * a.dq_stride[0] + i * a.dq_stride[1]) +
                   static_cast<int64_t>(h) * a.dq_stride[2] + c * 8;
        };
        if (accumulated) {
            // rows whose dQ was summed with unordered atomics
            const uint32_t n = static_cast<uint32_t>(e1 - t0) * per_row;
#pragma unroll 1
            for (uint32_t k0 = tid; k0 < n; k0 += kBatch * 256) {
                float4 x[kBatch], y[kBatch];
#pragma unroll
                for (int q = 0; q < kBatch; ++q) {
                    const uint32_t k = k0 + q * 256;
                    x[q] = y[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                    const uint32_t r = k / per_row, rem = k - r * per_row;
                    const float* pf = a.dq_acc + ((s.q_row0 + t0 + r) * g.h_q + h0) * HD + rem * 8;
                    if (k < n && in_bounds(a.status, pf, a.dq_acc, g.ext.dq_acc, 8)) {
                        const float4* src = reinterpret_cast<const float4*>(pf);
                        x[q] = src[0];
                        y[q] = src[1];
                    }
                }
#pragma unroll
                for (int q = 0; q < kBatch; ++q) {
                    const uint32_t k = k0 + q * 256;
                    if (k >= n) break;
                    const uint32_t r = k / per_row, rem = k - r * per_row, hl = rem / TPR;
                    uint16_t* dst = dst_of(t0 + r, h0 + hl, rem - hl * TPR);
                    const float f[8] = {x[q].x, x[q].y, x[q].z, x[q].w, y[q].x, y[q].y, y[q].z, y[q].w};
                    if (in_bounds(a.status, dst, a.dq, g.ext.dq, 8))
                        *reinterpret_cast<uint4*>(dst) = pack8<BF16>(f);
                }
            }
        }
        if (from_slots) {
            // deterministic mode: the visitors' partials, summed in visitor order
            const int64_t nv = imin(n_vis, a.n_slots);
            const uint32_t n = static_cast<uint32_t>(e1 - t0) * per_row;
#pragma unroll 1
            for (uint32_t k = tid; k < n; k += 256) {
                const uint32_t r = k / per_row, rem = k - r * per_row, hl = rem / TPR, c = rem - hl * TPR;
                const float* src = a.dq_part +
                                   (((bi * g.h_q + h0 + hl) * a.n_q_tiles + j) * a.n_slots * kTileQ + r) * HD + c * 8;
                float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                // eight visitors' loads in flight, then their sums in visitor order
#pragma unroll 1
                for (int64_t v0 = 0; v0 < nv; v0 += 8) {
                    float4 xv[8], yv[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        xv[q] = yv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                        const float* pv = src + (v0 + q) * kTileQ * HD;
                        if (v0 + q < nv && in_bounds(a.status, pv, a.dq_part, g.ext.dq_part, 8)) {
                            xv[q] = reinterpret_cast<const float4*>(pv)[0];
                            yv[q] = reinterpret_cast<const float4*>(pv)[1];
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (v0 + q >= nv) break;
                        f[0] += xv[q].x; f[1] += xv[q].y; f[2] += xv[q].z; f[3] += xv[q].w;
                        f[4] += yv[q].x; f[5] += yv[q].y; f[6] += yv[q].z; f[7] += yv[q].w;
                    }
                }
                uint16_t* dst = dst_of(t0 + r, h0 + hl, c);
                if (in_bounds(a.status, dst, a.dq, g.ext.dq, 8))
                    *reinterpret_cast<uint4*>(dst) = pack8<BF16>(f);
            }
        }
        if (z0 >= t1) continue;
        const uint32_t n = static_cast<uint32_t>(t1 - z0) * per_row;
#pragma unroll 1
        for (uint32_t k = tid; k < n; k += 256) {
            const uint32_t r = k / per_row, rem = k - r * per_row, hl = rem / TPR;
            uint16_t* dst = dst_of(z0 + r, h0 + hl, rem - hl * TPR);
            if (in_bounds(a.status, dst, a.dq, g.ext.dq, 8)) *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// ---------------------------------------------------------------- launchers

#define SWA_DISPATCH(KERNEL, ARGS, GRID, STREAM)                                   \
    do {                                                                           \
        if (a.g.d == 64 && dtype == 0) KERNEL<64, true><<<GRID, 256, 0, STREAM>>>(ARGS);   \
        else if (a.g.d == 64) KERNEL<64, false><<<GRID, 256, 0, STREAM>>>(ARGS);           \
        else if (dtype == 0) KERNEL<128, true><<<GRID, 256, 0, STREAM>>>(ARGS);            \
        else KERNEL<128, false><<<GRID, 256, 0, STREAM>>>(ARGS);                           \
    } while (0)

cudaError_t launch_preprocess(const PreArgs& a_in, int dtype, cudaStream_t s)
{
    PreArgs a = a_in;
    if (a.stats_row == 0 || a.g.b == 0 || a.g.h_q == 0) return cudaSuccess;
    const int64_t items = a.g.b * (a.stats_row / a.pre_rows) * ((a.g.h_q + a.pre_heads - 1) / a.pre_heads);
    if (items >= (int64_t(1) << 31)) return cudaErrorInvalidValue;   // blocks are counted in 32 bits
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const bool three = items >= int64_t(4) * 3 * sms;
    a.ring_bytes = three ? kPreRingThree : kPreRingOne;
    const int64_t cap = three ? int64_t(3) * sms : sms;
    const unsigned grid = static_cast<unsigned>(items < cap ? items : cap);
    const size_t smem = a.ring_bytes + 2 * 256 * 4 + 8 * kPreMaxStages;
#define SWA_PRE(HD, BF)                                                                                   \
    do {                                                                                                  \
        if ((e = cudaFuncSetAttribute(preprocess_kernel<HD, BF>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                      static_cast<int>(smem))) != cudaSuccess)                            \
            return e;                                                                                     \
        preprocess_kernel<HD, BF><<<grid, 256, smem, s>>>(a);                                             \
    } while (0)
    if (a.g.d == 64 && dtype == 0) SWA_PRE(64, true);
    else if (a.g.d == 64) SWA_PRE(64, false);
    else if (dtype == 0) SWA_PRE(128, true);
    else SWA_PRE(128, false);
#undef SWA_PRE
    return cudaGetLastError();
}

cudaError_t launch_dq_convert(const CvtArgs& a_in, int dtype, cudaStream_t s)
{
    CvtArgs a = a_in;
    const int64_t n_bj = a.n_q_tiles * a.g.b;
    if (n_bj == 0 || a.g.h_q == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // heads per unit: as many as keep at least two units per SM
    int64_t hc = a.g.h_q * n_bj / (2 * static_cast<int64_t>(sms));
    hc = hc < 1 ? 1 : (hc > a.g.h_q ? a.g.h_q : hc);
    a.head_chunk = static_cast<int32_t>(hc);
    const int64_t units = n_bj * ((a.g.h_q + hc - 1) / hc);
    if (units >= (int64_t(1) << 31) || 128 * a.g.h_q * (a.g.d / 8) >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;   // units and pieces are counted in 32 bits
    // eight 256-thread CTAs fit on an SM
    const int64_t cap = int64_t(8) * sms;
    const unsigned grid = static_cast<unsigned>(units < cap ? units : cap);
    // launched with programmatic stream serialization: it waits for the main
    // kernel in griddepcontrol.wait instead of in the launch queue
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.g.d == 64) e = dtype == 0 ? cudaLaunchKernelEx(&cfg, dq_convert_kernel<64, true>, a)
                                    : cudaLaunchKernelEx(&cfg, dq_convert_kernel<64, false>, a);
    else e = dtype == 0 ? cudaLaunchKernelEx(&cfg, dq_convert_kernel<128, true>, a)
                        : cudaLaunchKernelEx(&cfg, dq_convert_kernel<128, false>, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace swa
