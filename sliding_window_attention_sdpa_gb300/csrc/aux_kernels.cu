// aux_kernels.cu -- the two HBM-bound kernels around the main backward:
//  * preprocess ("dot"): D = rowsum(dO * O) in fp32, zero the relay / visit
//    counters and the status word, dSink partials;
//  * dq_convert ("cvt"): the main kernel already stored dQ (converted by each
//    q-tile's last visitor); this writes dQ = 0 on the rows no kv-tile visits
//    (padding, gap tokens, rows outside every window), converts the q-tiles
//    that took unordered atomics, and finishes dSink.
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
// grid (ceil(s_q / 128), h_q, b): one q-tile (kPreRows = 128 rows) of one
// sequence's slot for one q-head, covering every row of every q-tile (rows
// past the length included); each thread has four rows' loads in flight.
// Each row of HD features is read by HD/8 consecutive threads (16 B each).
template <int HD, bool BF16>
__global__ void __launch_bounds__(256) preprocess_kernel(const PreArgs a)
{
    constexpr int TPR = HD / 8;          // threads per row
    constexpr int RPP = 256 / TPR;       // rows per pass
    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    const int c = tid % TPR;
    const int64_t h = blockIdx.y, bi = blockIdx.z;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kPreRows;
    const bool with_sink = a.sink != nullptr;

    // relay / visit counters, ticket and status: zeroed by the whole grid
    {
        const int64_t nthr = static_cast<int64_t>(gridDim.x) * gridDim.y * gridDim.z * blockDim.x;
        const int64_t id = ((static_cast<int64_t>(blockIdx.z) * gridDim.y + blockIdx.y) * gridDim.x +
                            blockIdx.x) * blockDim.x + tid;
        for (int64_t k = id; k < a.n_sems; k += nthr) a.sems[k] = 0;
        if (id == 0) {
            a.status[0] = 0;
            a.status[1] = 0;
        }
    }
    const SeqInfo s = seq_info(g, bi);
    const int64_t blk = bi * gridDim.x + blockIdx.x;  // dSink partial slot
    const float sink = with_sink ? a.sink[h] : 0.f;
    // q-tiles with three or more visitors take unordered atomics (unless
    // deterministic): their accumulator rows start at zero
    bool zero_acc = false;
    if (!a.deterministic && i0 < s.len_q) {
        int64_t first, n;
        q_tile_visitors(g, s, i0 / kTileQ, first, n);
        zero_acc = n >= 3;
    }
    const uint16_t* o = static_cast<const uint16_t*>(a.o);
    const uint16_t* dout = static_cast<const uint16_t*>(a.dout);
    const bool thd = g.layout == 1;
    float dsink_acc = 0.f;

#pragma unroll 4
    for (int r = tid / TPR; r < kPreRows; r += RPP) {
        const int64_t i = i0 + r;
        const bool valid = i < s.len_q;
        float part = 0.f;
        if (valid) {
            const int64_t oo = (thd ? (s.q_row0 + i) * a.o_stride[1] : bi * a.o_stride[0] + i * a.o_stride[1]) +
                               h * a.o_stride[2] + c * 8;
            const int64_t od = (thd ? (s.q_row0 + i) * a.do_stride[1] : bi * a.do_stride[0] + i * a.do_stride[1]) +
                               h * a.do_stride[2] + c * 8;
            float fo[8], fd[8];
            unpack8<BF16>(ld_nc_v4(o + oo), fo);
            unpack8<BF16>(ld_nc_v4(dout + od), fd);
#pragma unroll
            for (int e = 0; e < 8; ++e) part = fmaf(fo[e], fd[e], part);
        }
        if (zero_acc && valid) {
            float4* z = reinterpret_cast<float4*>(a.dq_acc + ((s.q_row0 + i) * g.h_q + h) * HD + c * 8);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (c == 0) {
            // per-row statistics for the main kernel, one slot for every row of
            // every q-tile: (LSE * log2(e), D); rows past the length or that
            // attend nothing get (+inf, 0) so that P = 0 there
            float l2 = INFINITY;
            if (valid) {
                const int64_t so = thd ? h * g.rows_q + s.q_row0 + i : (bi * g.h_q + h) * g.s_q + i;
                const float lse = a.lse[so];
                if (lse != -INFINITY) {
                    l2 = lse * 1.4426950408889634f;
                    if (with_sink) dsink_acc -= expf(sink - lse) * part;
                }
            }
            a.stats[(bi * g.h_q + h) * a.stats_row + i] = make_float2(l2, valid ? part : 0.f);
        }
    }

    if (with_sink) {
        __shared__ float red[8];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dsink_acc += __shfl_xor_sync(0xffffffffu, dsink_acc, off);
        if ((tid & 31) == 0) red[tid >> 5] = dsink_acc;
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < 8; ++w) t += red[w];
            a.dsink_part[h * a.n_row_blocks + blk] = t;
        }
    }
}

// ---------------------------------------------------------------- convert
// The main kernel already stored dQ for every q-tile some kv-tile visits (its
// last visitor converts). This writes dQ = 0 on the other rows of a slot:
// rows past the sequence's length and q-tiles no kv-tile visits. grid
// (ceil(s_q / 128), h_q, b). It also finishes dSink in a fixed order.
template <int HD, bool BF16>
__global__ void __launch_bounds__(256) dq_convert_kernel(const CvtArgs a)
{
    constexpr int TPR = HD / 8;
    constexpr int RPP = 256 / TPR;
    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    const int c = tid % TPR;
    const int64_t j = blockIdx.x, h = blockIdx.y, bi = blockIdx.z;
    if (a.dsink != nullptr && j == 0 && h == 0 && bi == 0) {
        // fixed-order finish: bitwise repeatable
        for (int64_t hh = tid; hh < g.h_q; hh += blockDim.x) {
            float t = 0.f;
            for (int64_t k = 0; k < a.n_row_blocks; ++k) t += a.dsink_part[hh * a.n_row_blocks + k];
            a.dsink[hh] = t;
        }
    }
    const SeqInfo s = seq_info(g, bi);
    const int64_t t0 = j * kTileQ;
    const int64_t t1 = imin(t0 + kTileQ, s.slot_q);
    if (t0 >= t1) return;
    int64_t z0 = t0;  // first row to zero
    bool accumulated = false;
    if (t0 < s.len_q) {
        int64_t first, n;
        q_tile_visitors(g, s, j, first, n);
        if (n > 0) z0 = s.len_q;
        accumulated = n >= 3 && !a.deterministic;
    }
    const bool thd = g.layout == 1;
    uint16_t* dq = static_cast<uint16_t*>(a.dq);
    if (accumulated) {
        // rows whose dQ was summed with unordered atomics: convert them
        const int64_t e1 = imin(t1, s.len_q);
#pragma unroll 1
        for (int64_t i = t0 + tid / TPR; i < e1; i += RPP) {
            const float4* src = reinterpret_cast<const float4*>(a.dq_acc + ((s.q_row0 + i) * g.h_q + h) * HD + c * 8);
            const float4 x = src[0], y = src[1];
            const float f[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
            uint16_t* dst = dq + (thd ? (s.q_row0 + i) * a.dq_stride[1] : bi * a.dq_stride[0] + i * a.dq_stride[1]) +
                            h * a.dq_stride[2] + c * 8;
            *reinterpret_cast<uint4*>(dst) = pack8<BF16>(f);
        }
    }
    if (z0 >= t1) return;
#pragma unroll 1
    for (int64_t i = z0 + tid / TPR; i < t1; i += RPP) {
        uint16_t* dst = dq + (thd ? (s.q_row0 + i) * a.dq_stride[1] : bi * a.dq_stride[0] + i * a.dq_stride[1]) +
                        h * a.dq_stride[2] + c * 8;
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
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

cudaError_t launch_preprocess(const PreArgs& a, int dtype, cudaStream_t s)
{
    const int64_t nx = a.stats_row / kPreRows;  // every row of every q-tile
    if (nx == 0 || a.g.b == 0 || a.g.h_q == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>(nx), static_cast<unsigned>(a.g.h_q), static_cast<unsigned>(a.g.b));
    SWA_DISPATCH(preprocess_kernel, a, grid, s);
    return cudaGetLastError();
}

cudaError_t launch_dq_convert(const CvtArgs& a, int dtype, cudaStream_t s)
{
    const int64_t nx = (a.g.s_q + kTileQ - 1) / kTileQ;
    if (nx == 0 || a.g.b == 0 || a.g.h_q == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>(nx), static_cast<unsigned>(a.g.h_q), static_cast<unsigned>(a.g.b));
    SWA_DISPATCH(dq_convert_kernel, a, grid, s);
    return cudaGetLastError();
}

}  // namespace swa
