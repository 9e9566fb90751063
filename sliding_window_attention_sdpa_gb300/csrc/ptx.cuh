// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers, the tcgen05
// tensor-core instructions with tensor-memory (TMEM) accumulators, shared
// memory matrix descriptors, TMA bulk-tensor loads and a few scalar helpers.
// Every wait in this file is bounded by a wall-clock limit so that a kernel
// never spins forever; callers turn a timeout into a status code.
#pragma once

#include <cstdint>

namespace swa {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; false after
// `limit_ns` nanoseconds without completion.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Contiguous global -> shared copy by the TMA engine, completing on `bar` (both
// addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------- proxies

// Makes generic-proxy shared-memory writes visible to the async proxy
// (tensor cores, TMA) before a barrier that orders them.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- bulk groups

// Closes the group of bulk copies (shared -> global) issued so far by this thread.
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// The copies committed so far have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// The copies committed so far are complete (their global writes performed).
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders the async proxy's global writes (completed bulk copies) before the
// generic-proxy operations that follow, such as a release that publishes them.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The MMA issue helpers below are called by a whole, converged warp with the
// same operands in every lane; lane 0 alone issues (a predicate inside the
// instruction sequence, not a branch around it). Issued from inside an
// `if (lane == 0)` branch, each tcgen05.mma took about 100 SM cycles to issue,
// more than a 128 x 128 x 16 contraction takes to run; issued this way, about 40.
// tcgen05.commit tracks the issuing thread's MMAs, so commits go through the
// same lane.

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (fp16/bf16 in, fp32 acc).
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
        "mov.u32 l, %%laneid;\n\t"
        "setp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]: A (M x K, 16-bit) lives in tensor memory,
// lane = row, each 32-bit column holding two consecutive K elements (low half
// first).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
        "mov.u32 l, %%laneid;\n\t"
        "setp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Programmatic dependent launch. launch_dependents lets the next kernel of
// the stream (launched with programmatic stream serialization) start its
// prologue before this one ends; wait, in that next kernel, blocks until the
// previous kernel has completed and its memory is visible. Without the launch
// attribute both are no-ops in effect: the kernel starts after its
// predecessor anyway.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Four contractions in one sequence, D (+)= A_k B_k for k = 0..3, lane 0
// issuing: descriptor k is the first plus k * step (units of 16 bytes in the
// start-address field, which never carries), or for an A operand in tensor
// memory the first column plus k * step. The first contraction accumulates if
// `accumulate` is non-zero, the other three always. One predicate setup for
// the four, and 32-bit steps instead of 64-bit descriptor arithmetic between
// them: the issuing warp shares its SM sub-partition with the softmax warps,
// so its instruction count per step sets how soon the next step's
// contractions start.
__device__ __forceinline__ void umma_f16_ss_x4(uint32_t d_tmem, uint64_t a_desc, uint32_t a_step, uint64_t b_desc,
                                               uint32_t b_step, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e, t;\n\t.reg .b32 l;\n\t.reg .b64 a, b, as, bs;\n\t"
        "mov.u32 l, %%laneid;\n\t"
        "setp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.eq.u32 t, l, l;\n\t"
        "cvt.u64.u32 as, %2;\n\t"
        "cvt.u64.u32 bs, %4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %3, %5, p;\n\t"
        "add.s64 a, %1, as;\n\t"
        "add.s64 b, %3, bs;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, t;\n\t"
        "add.s64 a, a, as;\n\t"
        "add.s64 b, b, bs;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, t;\n\t"
        "add.s64 a, a, as;\n\t"
        "add.s64 b, b, bs;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, t;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "r"(a_step), "l"(b_desc), "r"(b_step), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_f16_ts_x4(uint32_t d_tmem, uint32_t a_tmem, uint32_t a_step, uint64_t b_desc,
                                               uint32_t b_step, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e, t;\n\t.reg .b32 l, a;\n\t.reg .b64 b, bs;\n\t"
        "mov.u32 l, %%laneid;\n\t"
        "setp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.eq.u32 t, l, l;\n\t"
        "cvt.u64.u32 bs, %4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %3, %5, p;\n\t"
        "add.u32 a, %1, %2;\n\t"
        "add.s64 b, %3, bs;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %5, t;\n\t"
        "add.u32 a, a, %2;\n\t"
        "add.s64 b, b, bs;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %5, t;\n\t"
        "add.u32 a, a, %2;\n\t"
        "add.s64 b, b, bs;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %5, t;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(a_step), "l"(b_desc), "r"(b_step), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Each thread of the warp writes 8 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by lane 0 has
// completed (called by the whole warp, like the MMA helpers).
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\t"
        "mov.u32 l, %%laneid;\n\t"
        "setp.eq.u32 e, l, 0;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
//  K-major: rows of 64 16-bit elements (128 B), 8-row groups `sbo` bytes apart
//           (lbo unused);
//  MN-major: 64 MN-elements per 128-B row, one row per K index, 8-row K groups
//           `sbo` bytes apart, 64-element MN blocks `lbo` bytes apart.
// Bits: [0,14) start>>4, [16,30) lbo>>4, [32,46) sbo>>4, [46,49) = 0b001,
// [49,52) base offset (0: atoms are 1024-B aligned), [61,64) swizzle (2 = 128 B).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// The descriptor of saddr + off, from that of saddr: the start field holds
// addresses up to 256 KB, so adding off >> 4 never carries out of it.
__device__ __forceinline__ uint64_t sdesc_at(uint64_t desc, uint32_t off)
{
    return desc + (off >> 4);
}

// Instruction descriptor of tcgen05.mma kind::f16 with fp32 accumulation.
// Bits: [4,6) D format (1 = f32), [7,10) A format, [10,13) B format
// (0 = f16, 1 = bf16), 15 A MN-major, 16 B MN-major, [17,23) N>>3, [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int m, int n, bool a_mn, bool b_mn)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// ---------------------------------------------------------------- scalar

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

__device__ __forceinline__ float4 ld_cg_f4(const float* p)
{
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_add_release_gpu(int* p, int v)
{
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_release_gpu(int* p, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int64_t imin(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t imax(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ int64_t floor_div(int64_t a, int64_t b)
{
    int64_t q = a / b;
    if ((a % b != 0) && ((a < 0) != (b < 0))) --q;
    return q;
}

}  // namespace swa
