// main_kernel.cu -- fused sliding-window SDPA backward on sm_103a tensor cores.
//
// One CTA per work item (kv-tile t, q-head h, sequence b). The kv-tile's K and
// V rows stay in shared memory; the CTA sweeps the q-tiles in the window-clamped
// range [q_lo, q_hi) (cuDNN-frontend PR #866, "Change": no query with
// anchor > kv_base + tile_kv - 1 + W reaches the tile), and for each q-tile
// issues the five contractions as tcgen05.mma with fp32 accumulators in tensor
// memory (TMEM):
//
//   S^T  = K Q^T          [kv x q]   TMEM cols   0..127
//   dP^T = V dO^T         [kv x q]   TMEM cols 128..255
//   dV  += P^T dO         [kv x d]   TMEM cols 256..256+d
//   dK  += dS^T Q         [kv x d]   TMEM cols 256+d..256+2d
//   dQ   = dS K           [q x d]    TMEM cols   0..d (reuses S^T once read)
//
// Between them the 128 threads (one per TMEM lane = kv row) recompute
// P = exp(S*scale - LSE) and dS = P (dP - D) in registers, apply the mask
// (top-left / bottom-right causal with left window, window-only, right band,
// padding) and write P^T and dS^T to shared memory as 16-bit operands. dQ rows
// are added to the fp32 accumulator with vector atomics, or in deterministic
// mode through the ordered relay whose turn is t - kv_first(q-tile).
//
// Shared-memory operands use the 128-byte swizzled layout: rows of 64 16-bit
// elements (128 B), 8-row atoms of 1024 B, 16-byte chunk c of row r stored at
// chunk position c ^ (r % 8); 64-column blocks of a 128-row tile are 16 KB apart.
// The same buffer serves as a K-major operand (contraction along the row) or
// an MN-major one (contraction across rows) through different descriptors.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sdpa_internal.h"
#include "seq.cuh"

namespace swa {

namespace {

constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256;
constexpr uint32_t kBlock16K = 128 * 128;  // one 64-column block of a 128-row tile

template <int HD>
struct Smem {
    static constexpr uint32_t kTile = 128 * HD * 2;
    static constexpr uint32_t kK = 0;
    static constexpr uint32_t kV = kK + kTile;
    static constexpr uint32_t kQ = kV + kTile;
    static constexpr uint32_t kDO = kQ + kTile;
    static constexpr uint32_t kP = kDO + kTile;     // P^T  [128 kv x 128 q]
    static constexpr uint32_t kDS = kP + 32768;     // dS^T [128 kv x 128 q]
    static constexpr uint32_t kLse = kDS + 32768;   // 128 fp32 (log2 domain)
    static constexpr uint32_t kDelta = kLse + 512;  // 128 fp32
    static constexpr uint32_t kBar = kDelta + 512;  // mbarrier (8 B)
    static constexpr uint32_t kMisc = kBar + 16;    // tmem slot, item, flags
    static constexpr uint32_t kBytes = kMisc + 64;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-B alignment
};

__device__ __forceinline__ uint32_t swz(int r, int chunk)
{
    // byte offset of 16-byte chunk `chunk` (0..HD/8-1) of row r in a 128-row tile
    return static_cast<uint32_t>((chunk >> 3) * kBlock16K + (r >> 3) * 1024 + (r & 7) * 128 +
                                 (((chunk & 7) ^ (r & 7)) << 4));
}

// Copies rows [0, 128) of a row-strided [., HD] 16-bit matrix into a swizzled
// tile; rows at or past `nvalid` are zero.
template <int HD>
__device__ __forceinline__ void load_tile(uint8_t* dst, const uint16_t* src, int64_t row_stride,
                                          int64_t nvalid, int tid)
{
    constexpr int CPR = HD / 8;
#pragma unroll 4
    for (int idx = tid; idx < 128 * CPR; idx += kThreads) {
        const int r = idx / CPR, c = idx % CPR;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < nvalid) v = ld_nc_v4(src + r * row_stride + c * 8);
        *reinterpret_cast<uint4*>(dst + swz(r, c)) = v;
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

// q-tile range [lo, hi) of kv rows [kv_base, kv_end) of one sequence: lo is
// the first q-tile holding a row that reaches key kv_base (right bound), hi
// the clamp ceil((kv_end + W - diag) / tile_q) (left window).
__device__ __forceinline__ void q_range(const Geometry& g, const SeqInfo& s, int64_t kv_base,
                                        int64_t kv_end, int64_t& lo, int64_t& hi)
{
    const int64_t n_q = (s.len_q + kTileQ - 1) / kTileQ;
    lo = 0;
    hi = n_q;
    if (kv_base >= s.len_kv || n_q == 0) {
        hi = 0;
        return;
    }
    if (g.right >= 0) {
        const int64_t first = kv_base - g.right - s.diag;
        lo = first > 0 ? first / kTileQ : 0;
    }
    if (g.window_left >= 0) {
        const int64_t c = floor_div(kv_end + g.window_left - s.diag + kTileQ - 1, kTileQ);
        if (c < hi) hi = c;
    }
    if (hi < lo) hi = lo;
}

}  // namespace

template <int HD, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) sdpa_bwd_main_kernel(const __grid_constant__ MainArgs a)
{
    using L = Smem<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(sm);
    float* sLse = reinterpret_cast<float*>(sm + L::kLse);
    float* sDelta = reinterpret_cast<float*>(sm + L::kDelta);
    const uint32_t bar = sbase + L::kBar;
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + L::kMisc);  // [0] tmem, [1] item, [2] flag

    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;

    if (tid == 0) {
        misc[1] = a.deterministic ? static_cast<uint32_t>(atomicAdd(&a.status[1], 1)) : blockIdx.x;
        misc[2] = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(sbase + L::kMisc, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const int64_t item = misc[1];

    const int64_t t = item % a.n_kv_tiles;
    const int64_t h = (item / a.n_kv_tiles) % g.h_q;
    const int64_t bi = item / (a.n_kv_tiles * g.h_q);
    const int64_t gk = h / (g.h_q / g.h_kv);
    const SeqInfo s = seq_info(g, bi);
    if (s.bad && t == 0 && h == 0 && tid == 0) set_status(a.status, kStatusBadLengths);

    const int64_t kv_base = t * kTileKV;
    const int64_t kv_end = imin(kv_base + kTileKV, s.len_kv);
    int64_t q_lo, q_hi;
    q_range(g, s, kv_base, kv_end, q_lo, q_hi);
    const bool has_work = q_hi > q_lo && kv_base < s.slot_kv;

    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tm_s = tmem + kColS, tm_dp = tmem + kColDP;
    const uint32_t tm_dv = tmem + kColDV, tm_dk = tmem + kColDV + HD, tm_dq = tmem + kColS;
    constexpr uint32_t kIdQK = idesc_f16(BF16, 128, 128, false, false);
    constexpr uint32_t kIdPV = idesc_f16(BF16, 128, HD, false, true);
    constexpr uint32_t kIdDQ = idesc_f16(BF16, 128, HD, true, true);

    const uint16_t* qp = static_cast<const uint16_t*>(a.q);
    const uint16_t* kp = static_cast<const uint16_t*>(a.k);
    const uint16_t* vp = static_cast<const uint16_t*>(a.v);
    const uint16_t* dop = static_cast<const uint16_t*>(a.dout);
    // element offsets of row 0 of the sequence's slot for the head in use
    auto seq_base = [&](const int64_t* st, int64_t row0_packed, int64_t head) -> int64_t {
        return (g.layout == 1 ? row0_packed * st[1] : bi * st[0]) + head * st[2];
    };
    const int64_t kbase = seq_base(a.k_stride, s.kv_row0, gk);
    const int64_t vbase = seq_base(a.v_stride, s.kv_row0, gk);
    const int64_t qbase = seq_base(a.q_stride, s.q_row0, h);
    const int64_t dobase = seq_base(a.do_stride, s.q_row0, h);

    // this thread's kv row and the q rows it attends: [i_lo, i_hi]
    const int64_t kj = kv_base + tid;
    int64_t i_lo = 0, i_hi = s.len_q - 1;
    if (g.right >= 0) i_lo = imax(i_lo, kj - g.right - s.diag);
    if (g.window_left >= 0) i_hi = imin(i_hi, kj + g.window_left - s.diag);
    if (kj >= s.len_kv) i_hi = -1;

    uint32_t phase = 0;
    bool ok = true;

    if (has_work) {
        load_tile<HD>(sm + L::kK, kp + kbase + kv_base * a.k_stride[1], a.k_stride[1],
                      s.len_kv - kv_base, tid);
        load_tile<HD>(sm + L::kV, vp + vbase + kv_base * a.v_stride[1], a.v_stride[1],
                      s.len_kv - kv_base, tid);
    }

#pragma unroll 1
    for (int64_t j = q_lo; j < q_hi && ok; ++j) {
        const int64_t q0 = j * kTileQ;
        // ---- stage Q, dO, LSE, D of q-tile j
        load_tile<HD>(sm + L::kQ, qp + qbase + q0 * a.q_stride[1], a.q_stride[1], s.len_q - q0, tid);
        load_tile<HD>(sm + L::kDO, dop + dobase + q0 * a.do_stride[1], a.do_stride[1],
                      s.len_q - q0, tid);
        {
            const int64_t qi = q0 + tid;
            float lse = INFINITY, dlt = 0.f;
            if (qi < s.len_q) {
                const int64_t st = stat_offset(g, s.q_row0 + qi, h);
                lse = a.lse[st];
                dlt = a.delta[st];
                if (lse == -INFINITY) lse = INFINITY;  // row attends nothing: P = 0
            }
            sLse[tid] = lse * 1.4426950408889634f;
            sDelta[tid] = dlt;
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- S^T = K Q^T, dP^T = V dO^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint32_t koff = (k >> 2) * kBlock16K + (k & 3) * 32;
                umma_f16_ss(tm_s, sdesc_sw128(sbase + L::kK + koff, 16, 1024),
                            sdesc_sw128(sbase + L::kQ + koff, 16, 1024), kIdQK, k > 0);
            }
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint32_t koff = (k >> 2) * kBlock16K + (k & 3) * 32;
                umma_f16_ss(tm_dp, sdesc_sw128(sbase + L::kV + koff, 16, 1024),
                            sdesc_sw128(sbase + L::kDO + koff, 16, 1024), kIdQK, k > 0);
            }
            umma_commit(bar);
        }
        ok = __syncthreads_and(mbar_wait(bar, phase, a.timeout_ns));
        phase ^= 1;
        if (!ok) break;
        tc_fence_after();

        // ---- P^T, dS^T rows of this thread's kv row
        {
            const int64_t c_lo = imax(i_lo - q0, 0);
            const int64_t c_hi = imin(i_hi - q0, 127);
            uint8_t* prow = sm + L::kP;
            uint8_t* dsrow = sm + L::kDS;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t sv[32], dpv[32];
                tmem_ld32(tm_s + lane_off + ch * 32, sv);
                tmem_ld32(tm_dp + lane_off + ch * 32, dpv);
                tmem_ld_wait();
                uint32_t pk[16], dk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float p2[2], d2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int c = ch * 32 + e + u;
                        const bool att = c >= c_lo && c <= c_hi;
                        const float sc = __uint_as_float(sv[e + u]);
                        const float dp = __uint_as_float(dpv[e + u]);
                        const float p = att ? ex2_approx(fmaf(sc, a.scale_log2, -sLse[c])) : 0.f;
                        p2[u] = p;
                        d2[u] = att ? p * (dp - sDelta[c]) : 0.f;
                    }
                    pk[e >> 1] = pack2<BF16>(p2[0], p2[1]);
                    dk[e >> 1] = pack2<BF16>(d2[0], d2[1]);
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t off = swz(tid, ch * 4 + m);
                    *reinterpret_cast<uint4*>(prow + off) =
                        make_uint4(pk[4 * m], pk[4 * m + 1], pk[4 * m + 2], pk[4 * m + 3]);
                    *reinterpret_cast<uint4*>(dsrow + off) =
                        make_uint4(dk[4 * m], dk[4 * m + 1], dk[4 * m + 2], dk[4 * m + 3]);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- dV += P^T dO, dK += dS^T Q, dQ = dS K
        if (tid == 0) {
            tc_fence_after();
            const uint32_t acc = j > q_lo ? 1u : 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t aoff = (k >> 2) * kBlock16K + (k & 3) * 32;
                umma_f16_ss(tm_dv, sdesc_sw128(sbase + L::kP + aoff, 16, 1024),
                            sdesc_sw128(sbase + L::kDO + k * 2048, kBlock16K, 1024), kIdPV,
                            acc | (k > 0));
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t aoff = (k >> 2) * kBlock16K + (k & 3) * 32;
                umma_f16_ss(tm_dk, sdesc_sw128(sbase + L::kDS + aoff, 16, 1024),
                            sdesc_sw128(sbase + L::kQ + k * 2048, kBlock16K, 1024), kIdPV,
                            acc | (k > 0));
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                umma_f16_ss(tm_dq, sdesc_sw128(sbase + L::kDS + k * 2048, kBlock16K, 1024),
                            sdesc_sw128(sbase + L::kK + k * 2048, kBlock16K, 1024), kIdDQ, k > 0);
            }
            umma_commit(bar);
        }
        ok = __syncthreads_and(mbar_wait(bar, phase, a.timeout_ns));
        phase ^= 1;
        if (!ok) break;
        tc_fence_after();

        // ---- dQ rows (this thread: q row q0 + tid) into the fp32 accumulator
        {
            const int64_t qi = q0 + tid;
            const bool row_ok = qi < s.len_q;
            float* dst = a.dq_acc + ((s.q_row0 + qi) * g.h_q + h) * HD;
            bool turn_ok = true;
            int* sem = nullptr;
            int turn = 0;
            if (a.deterministic) {
                const int64_t first = g.window_left >= 0
                                          ? imax(floor_div(q0 + s.diag - g.window_left, kTileKV), 0)
                                          : 0;
                turn = static_cast<int>(t - first);
                sem = a.sems + (bi * g.h_q + h) * a.n_q_tiles + j;
                if (tid == 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(sem) != turn) {
                        if (globaltimer_ns() - t0 > static_cast<uint64_t>(a.timeout_ns)) {
                            set_status(a.status, kStatusTimeout);
                            misc[2] = 1;
                            break;
                        }
                    }
                }
                __syncthreads();
                turn_ok = misc[2] == 0;
            }
#pragma unroll 1
            for (int ch = 0; ch < HD / 32; ++ch) {
                uint32_t v[32];
                tmem_ld32(tm_dq + lane_off + ch * 32, v);
                tmem_ld_wait();
                if (row_ok && turn_ok) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        red_add_v4(dst + ch * 32 + e, __uint_as_float(v[e]) * a.scale,
                                   __uint_as_float(v[e + 1]) * a.scale,
                                   __uint_as_float(v[e + 2]) * a.scale,
                                   __uint_as_float(v[e + 3]) * a.scale);
                }
            }
            if (a.deterministic) {
                __threadfence();
                __syncthreads();
                if (tid == 0) st_release_gpu(sem, turn + 1);
            }
        }
        tc_fence_before();
        __syncthreads();
    }

    // ---- epilogue: dV, dK (scaled) rows of this thread's kv row
    if (kv_base < s.slot_kv) {
        const bool row_in_slot = kj < s.slot_kv;
        const bool live = has_work && ok && kj < s.len_kv;
        const int64_t prow = s.kv_row0 + kj;  // packed kv row
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
            const uint32_t col = which == 0 ? tm_dv : tm_dk;
            const float mul = which == 0 ? 1.f : a.scale;
#pragma unroll 1
            for (int ch = 0; ch < HD / 32; ++ch) {
                uint32_t v[32];
                if (has_work && ok) {
                    tmem_ld32(col + lane_off + ch * 32, v);
                    tmem_ld_wait();
                }
                float f[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) f[e] = live ? __uint_as_float(v[e]) * mul : 0.f;
                if (!row_in_slot) continue;
                if (a.dk_ws != nullptr) {
                    float* dst = (which == 0 ? a.dv_ws : a.dk_ws) + (prow * g.h_q + h) * HD + ch * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(dst + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
                } else {
                    const int64_t* st = which == 0 ? a.dv_stride : a.dk_stride;
                    uint16_t* base = static_cast<uint16_t*>(which == 0 ? a.dv : a.dk);
                    uint16_t* dst = base + (g.layout == 1 ? prow * st[1] : bi * st[0] + kj * st[1]) +
                                    gk * st[2] + ch * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
                        *reinterpret_cast<uint4*>(dst + e) =
                            make_uint4(pack2<BF16>(f[e], f[e + 1]), pack2<BF16>(f[e + 2], f[e + 3]),
                                       pack2<BF16>(f[e + 4], f[e + 5]), pack2<BF16>(f[e + 6], f[e + 7]));
                }
            }
        }
    }
    if (!ok && tid == 0) set_status(a.status, kStatusTimeout);

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int HD, bool BF16>
static cudaError_t launch_typed(const MainArgs& a, cudaStream_t s)
{
    auto kern = sdpa_bwd_main_kernel<HD, BF16>;
    const uint32_t bytes = Smem<HD>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    const int64_t items = a.g.b * a.g.h_q * a.n_kv_tiles;
    if (items == 0) return cudaSuccess;
    kern<<<static_cast<unsigned>(items), kThreads, bytes, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_main(const MainArgs& a, int dtype, cudaStream_t s)
{
    if (a.g.d == 64) return dtype == 0 ? launch_typed<64, true>(a, s) : launch_typed<64, false>(a, s);
    return dtype == 0 ? launch_typed<128, true>(a, s) : launch_typed<128, false>(a, s);
}

}  // namespace swa
