// aux_kernels.cu -- the three HBM-bound kernels around the main backward:
//  * preprocess ("dot"): D = rowsum(dO * O) in fp32, zero the fp32 dQ
//    accumulator / relay counters / status, dSink partials;
//  * dq_convert ("cvt"): fp32 dQ accumulator -> I/O dtype, dSink finish;
//  * gqa_reduce ("reduce"): per-q-head fp32 dK/dV partials summed over each
//    kv-head's group in head order -> I/O dtype.
// All three move 16-byte vectors per thread with consecutive threads on
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
// grid (n_row_blocks, h_q), 256 threads. Each row of HD features is read by
// HD/8 consecutive threads (16 B each).
template <int HD, bool BF16>
__global__ void __launch_bounds__(256) preprocess_kernel(const PreArgs a)
{
    constexpr int TPR = HD / 8;          // threads per row
    constexpr int RPP = 256 / TPR;       // rows per pass
    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    const int c = tid % TPR;
    const int64_t h = blockIdx.y;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kPreRows;
    const bool with_sink = a.sink != nullptr;
    const float sink = with_sink ? a.sink[h] : 0.f;
    float dsink_acc = 0.f;

    // relay counters, ticket and status: zeroed by the whole grid
    {
        const int64_t nthr = static_cast<int64_t>(gridDim.x) * gridDim.y * blockDim.x;
        const int64_t id = (static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x) * blockDim.x + tid;
        for (int64_t k = id; k < a.n_sems; k += nthr) a.sems[k] = 0;
        if (id == 0) {
            a.status[0] = 0;
            a.status[1] = 0;
        }
    }

#pragma unroll 1
    for (int r = tid / TPR; r < kPreRows; r += RPP) {
        const int64_t row = row0 + r;
        const bool in_range = row < g.rows_q;
        float part = 0.f;
        bool valid = false;
        int64_t stat = 0;
        if (in_range) {
            const int64_t bi = q_row_seq(g, row);
            const SeqInfo s = seq_info(g, bi);
            valid = (row - s.q_row0) < s.len_q;
            stat = stat_offset(g, row, h);
            if (valid) {
                const int64_t oo = elem_offset(g, a.o_stride, row, g.s_q, h) + c * 8;
                const int64_t od = elem_offset(g, a.do_stride, row, g.s_q, h) + c * 8;
                float fo[8], fd[8];
                unpack8<BF16>(ld_nc_v4(static_cast<const uint16_t*>(a.o) + oo), fo);
                unpack8<BF16>(ld_nc_v4(static_cast<const uint16_t*>(a.dout) + od), fd);
#pragma unroll
                for (int e = 0; e < 8; ++e) part = fmaf(fo[e], fd[e], part);
            }
            float4* acc = reinterpret_cast<float4*>(a.dq_acc + (row * g.h_q + h) * HD + c * 8);
            acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (in_range && c == 0) {
            a.delta[stat] = valid ? part : 0.f;
            if (with_sink && valid) {
                const float lse = a.lse[stat];
                if (lse != -INFINITY) dsink_acc -= expf(sink - lse) * part;
            }
        }
    }

    if (with_sink) {
        __shared__ float red[8];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dsink_acc += __shfl_xor_sync(0xffffffffu, dsink_acc, off);
        if ((tid & 31) == 0) red[tid >> 5] = dsink_acc;
        __syncthreads();
        if (tid == 0) {
            float s = 0.f;
            for (int w = 0; w < 8; ++w) s += red[w];
            a.dsink_part[h * a.n_row_blocks + blockIdx.x] = s;
        }
    }
}

// ---------------------------------------------------------------- convert
template <int HD, bool BF16>
__global__ void __launch_bounds__(256) dq_convert_kernel(const CvtArgs a)
{
    constexpr int TPR = HD / 8;
    constexpr int RPP = 256 / TPR;
    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    const int c = tid % TPR;
    const int64_t h = blockIdx.y;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kPreRows;
#pragma unroll 1
    for (int r = tid / TPR; r < kPreRows; r += RPP) {
        const int64_t row = row0 + r;
        if (row >= g.rows_q) break;
        const float4* src = reinterpret_cast<const float4*>(a.dq_acc + (row * g.h_q + h) * HD + c * 8);
        const float4 x = src[0], y = src[1];
        const float f[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
        uint16_t* dst = static_cast<uint16_t*>(a.dq) + elem_offset(g, a.dq_stride, row, g.s_q, h) + c * 8;
        *reinterpret_cast<uint4*>(dst) = pack8<BF16>(f);
    }
    if (a.dsink != nullptr && blockIdx.x == 0 && blockIdx.y == 0) {
        // fixed-order finish: bitwise repeatable
        for (int64_t hh = tid; hh < g.h_q; hh += blockDim.x) {
            float s = 0.f;
            for (int64_t k = 0; k < a.n_row_blocks; ++k) s += a.dsink_part[hh * a.n_row_blocks + k];
            a.dsink[hh] = s;
        }
    }
}

// ---------------------------------------------------------------- GQA reduce
template <int HD, bool BF16>
__global__ void __launch_bounds__(256) gqa_reduce_kernel(const ReduceArgs a)
{
    constexpr int TPR = HD / 8;
    constexpr int RPP = 256 / TPR;
    const Geometry& g = a.g;
    const int tid = threadIdx.x;
    const int c = tid % TPR;
    const int64_t gk = blockIdx.y;
    const int64_t group = g.h_q / g.h_kv;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kPreRows;
#pragma unroll 1
    for (int r = tid / TPR; r < kPreRows; r += RPP) {
        const int64_t row = row0 + r;
        if (row >= g.rows_kv) break;
        float sk[8] = {0, 0, 0, 0, 0, 0, 0, 0}, sv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int64_t hh = gk * group; hh < (gk + 1) * group; ++hh) {
            const int64_t o = (row * g.h_q + hh) * HD + c * 8;
            const float4* pk = reinterpret_cast<const float4*>(a.dk_ws + o);
            const float4* pv = reinterpret_cast<const float4*>(a.dv_ws + o);
            const float4 k0 = pk[0], k1 = pk[1], v0 = pv[0], v1 = pv[1];
            sk[0] += k0.x; sk[1] += k0.y; sk[2] += k0.z; sk[3] += k0.w;
            sk[4] += k1.x; sk[5] += k1.y; sk[6] += k1.z; sk[7] += k1.w;
            sv[0] += v0.x; sv[1] += v0.y; sv[2] += v0.z; sv[3] += v0.w;
            sv[4] += v1.x; sv[5] += v1.y; sv[6] += v1.z; sv[7] += v1.w;
        }
        uint16_t* dk = static_cast<uint16_t*>(a.dk) + elem_offset(g, a.dk_stride, row, g.s_kv, gk) + c * 8;
        uint16_t* dv = static_cast<uint16_t*>(a.dv) + elem_offset(g, a.dv_stride, row, g.s_kv, gk) + c * 8;
        *reinterpret_cast<uint4*>(dk) = pack8<BF16>(sk);
        *reinterpret_cast<uint4*>(dv) = pack8<BF16>(sv);
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
    if (a.n_row_blocks == 0 || a.g.h_q == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>(a.n_row_blocks), static_cast<unsigned>(a.g.h_q));
    SWA_DISPATCH(preprocess_kernel, a, grid, s);
    return cudaGetLastError();
}

cudaError_t launch_dq_convert(const CvtArgs& a, int dtype, cudaStream_t s)
{
    if (a.n_row_blocks == 0 || a.g.h_q == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>(a.n_row_blocks), static_cast<unsigned>(a.g.h_q));
    SWA_DISPATCH(dq_convert_kernel, a, grid, s);
    return cudaGetLastError();
}

cudaError_t launch_gqa_reduce(const ReduceArgs& a, int dtype, cudaStream_t s)
{
    const int64_t blocks = (a.g.rows_kv + kPreRows - 1) / kPreRows;
    if (blocks == 0 || a.g.h_kv == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(a.g.h_kv));
    SWA_DISPATCH(gqa_reduce_kernel, a, grid, s);
    return cudaGetLastError();
}

}  // namespace swa
