// api.cu -- the C ABI declared in include/sdpa_bwd.h: host-side argument
// checks, the workspace layout, and the launches of the four kernels on the
// caller's stream. Nothing here allocates or synchronises (except
// sdpa_bwd_check_status, which reads the device status word).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sdpa_bwd.h"
#include "../../include/sdpa_fwd.h"
#include "sdpa_internal.h"
#include "seq.cuh"

namespace {

thread_local std::string g_last_error;

// sdpa_bwd_test_hook's settings for this thread's next sdpa_bwd calls.
constexpr int64_t kWaitLimitNs = 2000000000LL;
thread_local int64_t g_test_wait_ns = 0;
thread_local int32_t g_test_flags = 0;

sdpa_status_t fail(sdpa_status_t code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side validation that needs no device access.
sdpa_status_t check_shape(const sdpa_bwd_params* p)
{
    if (p == nullptr) return fail(SDPA_ERR_INVALID_ARG, "params is NULL");
    if (p->dtype != SDPA_BF16 && p->dtype != SDPA_F16)
        return fail(SDPA_ERR_INVALID_ARG, "dtype: expected SDPA_BF16 or SDPA_F16, got %d", p->dtype);
    if (p->layout != SDPA_BSHD && p->layout != SDPA_THD)
        return fail(SDPA_ERR_INVALID_ARG, "layout: expected SDPA_BSHD or SDPA_THD, got %d", p->layout);
    if (p->mask_mode < SDPA_MASK_NONE || p->mask_mode > SDPA_MASK_BOTTOM_RIGHT)
        return fail(SDPA_ERR_INVALID_ARG, "mask_mode: unknown value %d", p->mask_mode);
    if (p->deterministic < 0 || p->deterministic > 2)
        return fail(SDPA_ERR_INVALID_ARG, "deterministic: expected 0, 1 or 2, got %d", p->deterministic);
    if (p->b < 0 || p->h_q <= 0 || p->h_kv <= 0 || p->s_q < 0 || p->s_kv < 0)
        return fail(SDPA_ERR_INVALID_ARG,
                    "shape: b=%lld h_q=%lld h_kv=%lld s_q=%lld s_kv=%lld (need b,s >= 0, h > 0)",
                    (long long)p->b, (long long)p->h_q, (long long)p->h_kv, (long long)p->s_q,
                    (long long)p->s_kv);
    if (p->h_q % p->h_kv != 0)
        return fail(SDPA_ERR_INVALID_ARG, "h_q=%lld is not a multiple of h_kv=%lld",
                    (long long)p->h_q, (long long)p->h_kv);
    if (p->d != 64 && p->d != 128)
        return fail(SDPA_ERR_UNSUPPORTED, "d=%lld: only head dimensions 64 and 128 are implemented",
                    (long long)p->d);
    if (p->window_left < -1 || p->window_right < -1)
        return fail(SDPA_ERR_INVALID_ARG, "window_left=%lld window_right=%lld: must be >= -1",
                    (long long)p->window_left, (long long)p->window_right);
    if (!(p->scale > 0.f) || p->scale != p->scale)
        return fail(SDPA_ERR_INVALID_ARG, "scale must be a positive finite number");
    if (p->layout == SDPA_THD) {
        if (p->q_offsets == nullptr || p->kv_offsets == nullptr)
            return fail(SDPA_ERR_INVALID_ARG, "THD layout needs q_offsets and kv_offsets");
        if (p->total_q < 0 || p->total_kv < 0)
            return fail(SDPA_ERR_INVALID_ARG, "THD layout: total_q/total_kv must be >= 0");
    }
    if ((p->sink == nullptr) != (p->dsink == nullptr))
        return fail(SDPA_ERR_INVALID_ARG, "sink and dsink must both be set or both be NULL");
    // the main kernel numbers its work items (b x h_kv x kv-tiles) in 32 bits
    const int64_t n_items = p->b * p->h_kv * ((p->s_kv + swa::kTileKV - 1) / swa::kTileKV);
    if (n_items >= (int64_t(1) << 31))
        return fail(SDPA_ERR_UNSUPPORTED, "%lld work items (b x h_kv x ceil(s_kv/128)): at most 2^31 - 1",
                    (long long)n_items);
    return SDPA_OK;
}

sdpa_status_t check_strides(const char* name, const int64_t* st, bool thd)
{
    for (int i = thd ? 1 : 0; i < 3; ++i)
        if (st[i] < 0 || st[i] % 8 != 0)
            return fail(SDPA_ERR_INVALID_ARG,
                        "%s_stride[%d]=%lld: strides must be non-negative multiples of 8 elements",
                        name, i, (long long)st[i]);
    return SDPA_OK;
}

sdpa_status_t check_device_ptr(const char* name, const void* ptr, bool required, int device)
{
    if (ptr == nullptr) {
        if (required) return fail(SDPA_ERR_INVALID_ARG, "%s is NULL", name);
        return SDPA_OK;
    }
    if (!aligned16(ptr))
        return fail(SDPA_ERR_INVALID_ARG, "%s=%p is not 16-byte aligned", name, ptr);
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SDPA_ERR_INVALID_ARG, "%s=%p: not a CUDA pointer (%s)", name, ptr,
                    cudaGetErrorString(e));
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return fail(SDPA_ERR_INVALID_ARG, "%s=%p is not device memory (memory type %d)", name, ptr,
                    (int)attr.type);
    if (attr.device != device)
        return fail(SDPA_ERR_INVALID_ARG, "%s=%p lives on device %d, current device is %d", name, ptr,
                    attr.device, device);
    return SDPA_OK;
}

int64_t rows_q(const sdpa_bwd_params* p) { return p->layout == SDPA_THD ? p->total_q : p->b * p->s_q; }
int64_t rows_kv(const sdpa_bwd_params* p) { return p->layout == SDPA_THD ? p->total_kv : p->b * p->s_kv; }

// Most kv-tiles that can visit one q-tile. The clamped q-tile ranges of
// consecutive kv-tiles shift by one q-tile, so a q-tile has at most as many
// visitors as a range is wide: 1 + ceil(W_left / 128) + ceil(W_right / 128),
// plus one when the bottom-right diagonal shift is not a multiple of 128 or is
// not known on the host (length arrays, packed sequences); every kv-tile when
// the window is unbounded on either side.
int64_t max_visitors(const sdpa_bwd_params* p)
{
    const int64_t nkv = (p->s_kv + swa::kTileKV - 1) / swa::kTileKV;
    const int64_t right = p->mask_mode == SDPA_MASK_NONE ? p->window_right
                                                          : (p->window_right > 0 ? p->window_right : 0);
    if (p->window_left < 0 || right < 0) return nkv;
    int64_t v = 1 + (p->window_left + swa::kTileQ - 1) / swa::kTileQ + (right + swa::kTileQ - 1) / swa::kTileQ;
    if (p->mask_mode == SDPA_MASK_BOTTOM_RIGHT) {
        const bool known = p->layout == SDPA_BSHD && p->seq_q_lens == nullptr && p->seq_kv_lens == nullptr;
        if (!known || (p->s_kv - p->s_q) % swa::kTileKV != 0) ++v;
    }
    return v < nkv ? v : nkv;
}

// Strip mode of the main kernel (at most two visitors per q-tile): the two
// visitors of a q-tile combine dQ inside one CTA, or by arrival order between
// two, without the relay or per-visitor slots.
bool strip_mode(const sdpa_bwd_params* p) { return max_visitors(p) <= 2; }

// Most workspace the per-visitor dQ slots may take; beyond it deterministic
// mode keeps the relay.
constexpr size_t kSlotCapBytes = size_t(2) << 30;

swa::WsLayout layout_of(const sdpa_bwd_params* p)
{
    swa::WsLayout w{};
    const int64_t rq = rows_q(p);
    const int64_t nqt = (p->s_q + swa::kTileQ - 1) / swa::kTileQ;
    w.n_sems = p->b * p->h_q * nqt;
    w.n_row_blocks = p->b * ((p->s_q + swa::kTileQ - 1) / swa::kTileQ) * (swa::kTileQ / swa::pre_tile(p->h_q, p->d).rows);
    size_t off = 0;
    w.status = off;
    off = align256(off + 16);
    w.dq_acc = off;
    off = align256(off + static_cast<size_t>(rq) * p->h_q * p->d * 4);
    w.stats = off;
    off = align256(off + static_cast<size_t>(p->b) * p->h_q * nqt * swa::kTileQ * 8);
    w.sems = off;
    off = align256(off + static_cast<size_t>(w.n_sems) * 4);
    w.dsink_part = off;
    if (p->sink != nullptr) off = align256(off + static_cast<size_t>(p->h_q) * w.n_row_blocks * 4);
    // the main kernel's table of decoded work items (d = 64)
    w.items = off;
    if (p->d == 64)
        off = align256(off + static_cast<size_t>(p->b) * p->h_kv * ((p->s_kv + swa::kTileKV - 1) / swa::kTileKV) *
                                 swa::kItemBytes);
    // Deterministic mode (1): q-tiles that three or more kv-tiles visit keep one
    // fp32 partial per visitor, summed in visitor order by the convert kernel,
    // instead of passing one tile along the relay, when the slots fit the cap.
    w.dq_part = off;
    w.n_slots = 0;
    if (p->deterministic == 1 && !strip_mode(p)) {
        const int64_t bound = max_visitors(p);
        const size_t bytes = static_cast<size_t>(p->b) * p->h_q * nqt * bound * swa::kTileQ * p->d * 4;
        if (bound >= 3 && bytes <= kSlotCapBytes) {
            w.n_slots = bound;
            off = align256(off + bytes);
        }
    }
    w.total = off;
    return w;
}

swa::Geometry geometry_of(const sdpa_bwd_params* p)
{
    swa::Geometry g{};
    g.layout = p->layout;
    g.mask_mode = p->mask_mode;
    g.b = p->b;
    g.h_q = p->h_q;
    g.h_kv = p->h_kv;
    g.s_q = p->s_q;
    g.s_kv = p->s_kv;
    g.d = p->d;
    g.rows_q = rows_q(p);
    g.rows_kv = rows_kv(p);
    g.window_left = p->window_left;
    if (p->mask_mode == SDPA_MASK_NONE) g.right = p->window_right;
    else g.right = p->window_right > 0 ? p->window_right : 0;
    g.seq_q_lens = p->seq_q_lens;
    g.seq_kv_lens = p->seq_kv_lens;
    g.q_offsets = p->q_offsets;
    g.kv_offsets = p->kv_offsets;
    return g;
}

// Elements reachable from a strided [b][s][h][d] (BSHD) or [t][h][d] (THD)
// tensor's base pointer.
int64_t tensor_extent(bool thd, const int64_t* st, int64_t b, int64_t s, int64_t h, int64_t d, int64_t total)
{
    if (thd) return total > 0 && h > 0 ? (total - 1) * st[1] + (h - 1) * st[2] + d : 0;
    return b > 0 && s > 0 && h > 0 ? (b - 1) * st[0] + (s - 1) * st[1] + (h - 1) * st[2] + d : 0;
}

// Buffer extents for the range-checked build (the workspace sections from
// `w`; null for the forward, which has none).
swa::Extents extents_of(const sdpa_bwd_params* p, const swa::WsLayout* w)
{
    const bool thd = p->layout == SDPA_THD;
    const int64_t nqt = (p->s_q + swa::kTileQ - 1) / swa::kTileQ;
    swa::Extents e{};
    e.q = tensor_extent(thd, p->q_stride, p->b, p->s_q, p->h_q, p->d, p->total_q);
    e.o = tensor_extent(thd, p->o_stride, p->b, p->s_q, p->h_q, p->d, p->total_q);
    e.dout = tensor_extent(thd, p->do_stride, p->b, p->s_q, p->h_q, p->d, p->total_q);
    e.dq = tensor_extent(thd, p->dq_stride, p->b, p->s_q, p->h_q, p->d, p->total_q);
    e.k = tensor_extent(thd, p->k_stride, p->b, p->s_kv, p->h_kv, p->d, p->total_kv);
    e.v = tensor_extent(thd, p->v_stride, p->b, p->s_kv, p->h_kv, p->d, p->total_kv);
    e.dk = tensor_extent(thd, p->dk_stride, p->b, p->s_kv, p->h_kv, p->d, p->total_kv);
    e.dv = tensor_extent(thd, p->dv_stride, p->b, p->s_kv, p->h_kv, p->d, p->total_kv);
    e.lse = thd ? p->h_q * p->total_q : p->b * p->h_q * p->s_q;
    e.sink = p->sink ? p->h_q : 0;
    if (w != nullptr) {
        e.stats = p->b * p->h_q * nqt * swa::kTileQ * 2;
        e.dq_acc = rows_q(p) * p->h_q * p->d;
        e.dq_part = p->b * p->h_q * nqt * w->n_slots * swa::kTileQ * p->d;
        e.dsink_part = p->sink ? p->h_q * w->n_row_blocks : 0;
        e.sems = w->n_sems;
    }
    return e;
}

// Full check before a launch: shapes, strides, pointers and workspace.
sdpa_status_t check_all(const sdpa_bwd_params* p, const void* ws, size_t ws_bytes)
{
    sdpa_status_t st = check_shape(p);
    if (st != SDPA_OK) return st;
    const bool thd = p->layout == SDPA_THD;
    const struct { const char* n; const int64_t* s; } strides[] = {
        {"q", p->q_stride},   {"k", p->k_stride},   {"v", p->v_stride},   {"o", p->o_stride},
        {"dout", p->do_stride}, {"dq", p->dq_stride}, {"dk", p->dk_stride}, {"dv", p->dv_stride}};
    for (const auto& s : strides)
        if ((st = check_strides(s.n, s.s, thd)) != SDPA_OK) return st;
    const swa::WsLayout w = layout_of(p);
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return fail(SDPA_ERR_WORKSPACE, "workspace=%p must be non-NULL and 256-byte aligned", ws);
    if (ws_bytes < w.total)
        return fail(SDPA_ERR_WORKSPACE, "workspace_bytes=%zu, need %zu", ws_bytes, w.total);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return fail(SDPA_ERR_CUDA, "no CUDA device available");
    }
    const bool empty_q = rows_q(p) == 0, empty_kv = rows_kv(p) == 0;
    const struct { const char* n; const void* ptr; bool req; } ptrs[] = {
        {"q", p->q, !empty_q},       {"k", p->k, !empty_kv},     {"v", p->v, !empty_kv},
        {"o", p->o, !empty_q},       {"dout", p->dout, !empty_q}, {"lse", p->lse, !empty_q},
        {"dq", p->dq, !empty_q},     {"dk", p->dk, !empty_kv},   {"dv", p->dv, !empty_kv},
        {"sink", p->sink, false},    {"dsink", p->dsink, false},
        {"seq_q_lens", p->seq_q_lens, false}, {"seq_kv_lens", p->seq_kv_lens, false},
        {"q_offsets", p->q_offsets, thd}, {"kv_offsets", p->kv_offsets, thd},
        {"workspace", ws, true}};
    for (const auto& q : ptrs)
        if ((st = check_device_ptr(q.n, q.ptr, q.req, dev)) != SDPA_OK) return st;
    return SDPA_OK;
}

sdpa_status_t cuda_status(cudaError_t e, const char* what)
{
    if (e == cudaSuccess) return SDPA_OK;
    return fail(SDPA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// TMA descriptor of one head-strided tensor (strides in elements): boxes of
// `box_d` x 1 x 128 (x 1) elements with the 128-byte swizzle (box_d elements
// span 128 bytes), zero fill outside the tensor. BSHD maps are 4-D (d, h, s, b),
// THD maps 3-D (d, h, t). Sizes of 1 get a harmless non-zero stride.
sdpa_status_t make_map(CUtensorMap* m, const char* name, const void* base, CUtensorMapDataType dt,
                       int64_t esize, uint32_t box_d, bool thd, int64_t d, int64_t h, int64_t rows,
                       int64_t b, const int64_t* st)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(d * esize);
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h),
                          static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(b)};
    cuuint64_t hs = h > 1 ? static_cast<cuuint64_t>(st[2] * esize) : row_bytes;
    cuuint64_t ss = rows > 1 ? static_cast<cuuint64_t>(st[1] * esize) : hs * h;
    cuuint64_t bs = b > 1 ? static_cast<cuuint64_t>(st[0] * esize) : ss * (rows > 0 ? rows : 1);
    cuuint64_t strides[3] = {hs, ss, bs};
    cuuint32_t box[4] = {box_d, 1, 128, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const cuuint32_t rank = thd ? 3 : 4;
    CUresult r = fn(m, dt, rank, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(SDPA_ERR_UNSUPPORTED,
                    "%s: TMA descriptor rejected (error %d) for strides (%lld, %lld, %lld)", name,
                    (int)r, (long long)st[0], (long long)st[1], (long long)st[2]);
    return SDPA_OK;
}

// Descriptor of a 16-bit tensor read in whole-row boxes of d x box_h heads x
// box_rows rows, unswizzled (the preprocess's O and dO).
sdpa_status_t make_box_map(CUtensorMap* m, const char* name, const void* base, int dtype, bool thd, int64_t d,
                           int64_t h, int64_t rows, int64_t b, const int64_t* st, uint32_t box_h, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return fail(SDPA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const CUtensorMapDataType dt =
        dtype == SDPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int64_t esize = 2;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h),
                          static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(b)};
    cuuint64_t hs = h > 1 ? static_cast<cuuint64_t>(st[2] * esize) : static_cast<cuuint64_t>(d * esize);
    cuuint64_t ss = rows > 1 ? static_cast<cuuint64_t>(st[1] * esize) : hs * h;
    cuuint64_t bs = b > 1 ? static_cast<cuuint64_t>(st[0] * esize) : ss * (rows > 0 ? rows : 1);
    cuuint64_t strides[3] = {hs, ss, bs};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(d), box_h, box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, dt, thd ? 3 : 4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(SDPA_ERR_UNSUPPORTED, "%s: TMA descriptor rejected (error %d) for strides (%lld, %lld, %lld)",
                    name, (int)r, (long long)st[0], (long long)st[1], (long long)st[2]);
    return SDPA_OK;
}

// Descriptor of a 16-bit I/O tensor (64-element boxes).
sdpa_status_t make_map(CUtensorMap* m, const char* name, const void* base, int dtype, bool thd,
                       int64_t d, int64_t h, int64_t rows, int64_t b, const int64_t* st)
{
    const CUtensorMapDataType dt =
        dtype == SDPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return make_map(m, name, base, dt, 2, 64, thd, d, h, rows, b, st);
}

// The dQ convert kernel zero-fills rows past a sequence's length and q-tiles
// no kv-tile visits, converts q-tiles whose visitors added with unordered
// atomics (three or more, not deterministic) and finishes dSink. For a BSHD
// problem without length arrays every sequence has the same q-tiles, so the
// launcher can tell on the host that none of this applies and skip the launch.
bool convert_has_work(const sdpa_bwd_params* p, const swa::Geometry& g)
{
    if (p->dsink != nullptr || p->layout != SDPA_BSHD || p->seq_q_lens != nullptr ||
        p->seq_kv_lens != nullptr)
        return true;
    const bool slots = layout_of(p).n_slots > 0;
    swa::SeqInfo s{};
    s.slot_q = s.len_q = p->s_q;
    s.slot_kv = s.len_kv = p->s_kv;
    s.diag = p->mask_mode == SDPA_MASK_BOTTOM_RIGHT ? p->s_kv - p->s_q : 0;
    const int64_t nqt = (p->s_q + swa::kTileQ - 1) / swa::kTileQ;
    for (int64_t j = 0; j < nqt; ++j) {
        int64_t first, n;
        swa::q_tile_visitors(g, s, j, first, n);
        if (n == 0 || (n >= 3 && (!p->deterministic || slots))) return true;
    }
    return false;
}

template <typename T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

void copy3(int64_t* dst, const int64_t* src) { memcpy(dst, src, 3 * sizeof(int64_t)); }

}  // namespace

extern "C" {

size_t sdpa_bwd_workspace_bytes(const sdpa_bwd_params* p)
{
    if (check_shape(p) != SDPA_OK) return 0;
    g_last_error.clear();
    return layout_of(p).total;
}

sdpa_status_t sdpa_bwd_preprocess(const sdpa_bwd_params* p, void* ws, size_t ws_bytes, void* stream)
{
    sdpa_status_t st = check_all(p, ws, ws_bytes);
    if (st != SDPA_OK) return st;
    const swa::WsLayout w = layout_of(p);
    swa::PreArgs a{};
    a.g = geometry_of(p);
    a.g.ext = extents_of(p, &w);
    a.o = p->o;
    a.dout = p->dout;
    a.lse = p->lse;
    a.sink = p->sink;
    copy3(a.o_stride, p->o_stride);
    copy3(a.do_stride, p->do_stride);
    a.dq_acc = at<float>(ws, w.dq_acc);
    a.deterministic = p->deterministic;
    a.stats = at<float>(ws, w.stats);
    a.stats_row = ((p->s_q + swa::kTileQ - 1) / swa::kTileQ) * swa::kTileQ;
    a.status = at<int32_t>(ws, w.status);
    a.sems = at<int32_t>(ws, w.sems);
    a.n_sems = w.n_sems;
    a.dsink_part = p->sink ? at<float>(ws, w.dsink_part) : nullptr;
    a.n_row_blocks = w.n_row_blocks;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (a.n_row_blocks == 0) {
        // nothing to reduce: still reset the status words and the dSink output
        st = cuda_status(cudaMemsetAsync(a.status, 0, 8, s), "preprocess memset");
        if (st == SDPA_OK && p->dsink)
            st = cuda_status(cudaMemsetAsync(p->dsink, 0, p->h_q * sizeof(float), s), "dsink memset");
        return st;
    }
    const swa::PreTile pt = swa::pre_tile(p->h_q, p->d);
    a.pre_heads = pt.heads;
    a.pre_rows = pt.rows;
    const bool thd = p->layout == SDPA_THD;
    const int64_t rq = thd ? p->total_q : p->s_q;
    if ((st = make_box_map(&a.tm_o, "o", p->o, p->dtype, thd, p->d, p->h_q, rq, p->b, p->o_stride, pt.heads,
                           pt.rows)) != SDPA_OK ||
        (st = make_box_map(&a.tm_do, "dout", p->dout, p->dtype, thd, p->d, p->h_q, rq, p->b, p->do_stride, pt.heads,
                           pt.rows)) != SDPA_OK)
        return st;
    return cuda_status(swa::launch_preprocess(a, p->dtype, s), "preprocess launch");
}

sdpa_status_t sdpa_bwd(const sdpa_bwd_params* p, void* ws, size_t ws_bytes, void* stream)
{
    sdpa_status_t st = check_all(p, ws, ws_bytes);
    if (st != SDPA_OK) return st;
    const swa::WsLayout w = layout_of(p);
    swa::MainArgs a{};
    a.g = geometry_of(p);
    a.g.ext = extents_of(p, &w);
    a.q = p->q;
    a.k = p->k;
    a.v = p->v;
    a.dout = p->dout;
    a.stats = at<float>(ws, w.stats);
    a.stats_row = ((p->s_q + swa::kTileQ - 1) / swa::kTileQ) * swa::kTileQ;
    a.dq_acc = at<float>(ws, w.dq_acc);
    a.dq = p->dq;
    copy3(a.dq_stride, p->dq_stride);
    a.dk = p->dk;
    a.dv = p->dv;
    a.status = at<int32_t>(ws, w.status);
    a.sems = at<int32_t>(ws, w.sems);
    copy3(a.q_stride, p->q_stride);
    copy3(a.k_stride, p->k_stride);
    copy3(a.v_stride, p->v_stride);
    copy3(a.do_stride, p->do_stride);
    copy3(a.dk_stride, p->dk_stride);
    copy3(a.dv_stride, p->dv_stride);
    a.n_kv_tiles = (p->s_kv + swa::kTileKV - 1) / swa::kTileKV;
    a.n_q_tiles = (p->s_q + swa::kTileQ - 1) / swa::kTileQ;
    a.scale = p->scale;
    a.scale_log2 = p->scale * 1.4426950408889634f;
    a.deterministic = p->deterministic;
    a.timeout_ns = g_test_wait_ns > 0 ? g_test_wait_ns : kWaitLimitNs;
    a.test_flags = g_test_flags;
    if (p->b * p->h_q * a.n_kv_tiles == 0) return SDPA_OK;
    const bool thd = p->layout == SDPA_THD;
    const int64_t rq = thd ? p->total_q : p->s_q, rk = thd ? p->total_kv : p->s_kv;
    if (rk == 0) return SDPA_OK;  // no keys: dK, dV are empty and dQ stays zero
    // With no q rows the main kernel only writes dK = dV = 0; Q and dO then get
    // placeholder descriptors over K that are never used.
    const int64_t rq_map = rq > 0 ? rq : 1, rk_map = rk;
    const void* qptr = rq > 0 ? p->q : p->k;
    const void* doptr = rq > 0 ? p->dout : p->k;
    const int64_t* qst = rq > 0 ? p->q_stride : p->k_stride;
    const int64_t* dost = rq > 0 ? p->do_stride : p->k_stride;
    const int64_t hq_map = rq > 0 ? p->h_q : p->h_kv;
    if ((st = make_map(&a.tm_q, "q", qptr, p->dtype, thd, p->d, hq_map, rq_map, p->b, qst)) != SDPA_OK ||
        (st = make_map(&a.tm_do, "dout", doptr, p->dtype, thd, p->d, hq_map, rq_map, p->b, dost)) != SDPA_OK ||
        (st = make_map(&a.tm_k, "k", p->k, p->dtype, thd, p->d, p->h_kv, rk_map, p->b, p->k_stride)) != SDPA_OK ||
        (st = make_map(&a.tm_v, "v", p->v, p->dtype, thd, p->d, p->h_kv, rk_map, p->b, p->v_stride)) != SDPA_OK ||
        (st = make_map(&a.tm_dk, "dk", p->dk, p->dtype, thd, p->d, p->h_kv, rk_map, p->b, p->dk_stride)) != SDPA_OK ||
        (st = make_map(&a.tm_dv, "dv", p->dv, p->dtype, thd, p->d, p->h_kv, rk_map, p->b, p->dv_stride)) != SDPA_OK)
        return st;
    // dQ and its fp32 accumulator ([rows][h_q][d], packed). With no q rows they
    // are placeholders over K, never used.
    const int64_t acc_st[3] = {p->s_q * p->h_q * p->d, p->h_q * p->d, p->d};
    if (rq > 0) {
        if ((st = make_map(&a.tm_dq, "dq", p->dq, p->dtype, thd, p->d, p->h_q, rq, p->b, p->dq_stride)) != SDPA_OK ||
            (st = make_map(&a.tm_acc, "dq accumulator", a.dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 32, thd,
                           p->d, p->h_q, rq, p->b, acc_st)) != SDPA_OK)
            return st;
    } else {
        a.tm_dq = a.tm_k;
        a.tm_acc = a.tm_k;
    }
    // per-visitor partial dQ tiles: rows of d fp32 values, one 128-row tile
    // per (sequence, q-head, q-tile, visitor)
    a.n_slots = rq > 0 ? w.n_slots : 0;
    if (a.n_slots > 0) {
        const int64_t rows = p->b * p->h_q * a.n_q_tiles * a.n_slots * swa::kTileQ;
        const int64_t part_st[3] = {rows * p->d, p->d, p->d};
        if ((st = make_map(&a.tm_part, "dq partials", at<float>(ws, w.dq_part), CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                           4, 32, true, p->d, 1, rows, 1, part_st)) != SDPA_OK)
            return st;
    } else {
        a.tm_part = a.tm_k;
    }
    a.items = at<uint8_t>(ws, w.items);
    a.strip = strip_mode(p) ? 1 : 0;
    return cuda_status(swa::launch_main(a, p->dtype, static_cast<cudaStream_t>(stream)), "main launch");
}

sdpa_status_t sdpa_bwd_dq_convert(const sdpa_bwd_params* p, void* ws, size_t ws_bytes, void* stream)
{
    sdpa_status_t st = check_all(p, ws, ws_bytes);
    if (st != SDPA_OK) return st;
    const swa::WsLayout w = layout_of(p);
    swa::CvtArgs a{};
    a.g = geometry_of(p);
    a.g.ext = extents_of(p, &w);
    a.status = at<int32_t>(ws, w.status);
    a.dq_acc = at<float>(ws, w.dq_acc);
    a.dq_part = at<float>(ws, w.dq_part);
    a.n_slots = w.n_slots;
    a.n_q_tiles = (p->s_q + swa::kTileQ - 1) / swa::kTileQ;
    a.deterministic = p->deterministic;
    a.dq = p->dq;
    copy3(a.dq_stride, p->dq_stride);
    a.dsink_part = p->sink ? at<float>(ws, w.dsink_part) : nullptr;
    a.n_row_blocks = w.n_row_blocks;
    a.dsink = p->dsink;
    if (a.n_row_blocks == 0) return SDPA_OK;
    if (!convert_has_work(p, a.g)) return SDPA_OK;
    return cuda_status(swa::launch_dq_convert(a, p->dtype, static_cast<cudaStream_t>(stream)),
                       "dq_convert launch");
}

sdpa_status_t sdpa_bwd_gqa_reduce(const sdpa_bwd_params* p, void* ws, size_t ws_bytes, void* stream)
{
    // The group sum of dK/dV happens inside sdpa_bwd (TMEM accumulation over
    // the group's q-heads, in head order); this call only checks its arguments
    // so that the four-call sequence stays the same for every head layout.
    (void)stream;
    return check_all(p, ws, ws_bytes);
}

sdpa_status_t sdpa_bwd_check_status(const void* ws, void* stream)
{
    if (ws == nullptr) return fail(SDPA_ERR_WORKSPACE, "workspace is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t host[2] = {0, 0};
    sdpa_status_t st = cuda_status(cudaStreamSynchronize(s), "stream synchronize");
    if (st != SDPA_OK) return st;
    st = cuda_status(cudaMemcpy(host, ws, sizeof(host), cudaMemcpyDeviceToHost), "status read");
    if (st != SDPA_OK) return st;
    if (host[0] == SDPA_ERR_TIMEOUT)
        return fail(SDPA_ERR_TIMEOUT, "a device wait ran out (%s)",
                    host[1] == swa::kWhereRelay  ? "a dQ relay turn"
                    : host[1] == swa::kWherePair ? "the partial of a dQ pair split between two CTAs"
                                                 : "a hand-off inside the main kernel");
    if (host[0] == SDPA_ERR_BAD_LENGTHS)
        return fail(SDPA_ERR_BAD_LENGTHS, "a sequence length exceeds its slot (or s_q/s_kv)");
    if (host[0] == SDPA_ERR_BOUNDS)
        return fail(SDPA_ERR_BOUNDS, "a device index fell outside its buffer (range-checked build); the access was skipped");
    if (host[0] == SDPA_ERR_UNSUPPORTED)
        return fail(SDPA_ERR_UNSUPPORTED, "the device gave the main kernel shared memory not 1024-byte aligned");
    if (host[0] != 0) return fail(SDPA_ERR_CUDA, "unknown device status %d", host[0]);
    return SDPA_OK;
}

const char* sdpa_bwd_last_error(void) { return g_last_error.c_str(); }

sdpa_status_t sdpa_bwd_test_hook(int64_t wait_limit_ns, int32_t flags)
{
    if (flags & ~3) return fail(SDPA_ERR_INVALID_ARG, "test hook flags=%d: only bits 0 and 1 are defined", flags);
    g_test_wait_ns = wait_limit_ns > 0 ? wait_limit_ns : 0;
    g_test_flags = flags;
    g_last_error.clear();
    return SDPA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward without a caller-provided workspace, for callers that cannot
// allocate device memory (see sdpa_bwd_no_alloc in the header). Its scratch is
// this fixed array; host code never uses the array's name as an address (on
// the host it is only a stand-in): the device address comes from
// cudaGetSymbolAddress, looked up on every call with the caller's device
// current (cheap, allocates nothing, and never stale after a device reset).
namespace {

static __device__ __align__(256) unsigned char g_no_alloc_scratch[SDPA_BWD_NO_ALLOC_MAX_BYTES];

sdpa_status_t no_alloc_scratch(void** out)
{
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return fail(SDPA_ERR_CUDA, "sdpa_bwd_no_alloc: cannot resolve the scratch array on the current device (%s)",
                    cudaGetErrorString(e));
    }
    *out = p;
    return SDPA_OK;
}

}  // namespace

extern "C" {

sdpa_status_t sdpa_bwd_no_alloc(const sdpa_bwd_params* params, void* stream)
{
    sdpa_status_t st = check_shape(params);
    if (st != SDPA_OK) return st;
    // deterministic mode 1 whose per-visitor dQ slots do not fit the scratch
    // uses the relay (mode 2): the same bitwise-repeatable sums, no slots
    sdpa_bwd_params local = *params;
    size_t need = layout_of(&local).total;
    if (need > SDPA_BWD_NO_ALLOC_MAX_BYTES && local.deterministic == 1) {
        local.deterministic = 2;
        need = layout_of(&local).total;
    }
    const sdpa_bwd_params* p = &local;
    if (need > SDPA_BWD_NO_ALLOC_MAX_BYTES)
        return fail(SDPA_ERR_WORKSPACE,
                    "sdpa_bwd_no_alloc: this problem needs %zu bytes of scratch, more than the fixed "
                    "%zu bytes this entry point owns; call the workspace entry points instead",
                    need, static_cast<size_t>(SDPA_BWD_NO_ALLOC_MAX_BYTES));
    void* ws = nullptr;
    if ((st = no_alloc_scratch(&ws)) != SDPA_OK) return st;
    const size_t n = SDPA_BWD_NO_ALLOC_MAX_BYTES;
    if ((st = sdpa_bwd_preprocess(p, ws, n, stream)) != SDPA_OK) return st;
    if ((st = sdpa_bwd(p, ws, n, stream)) != SDPA_OK) return st;
    if ((st = sdpa_bwd_dq_convert(p, ws, n, stream)) != SDPA_OK) return st;
    return sdpa_bwd_gqa_reduce(p, ws, n, stream);
}

sdpa_status_t sdpa_bwd_no_alloc_check_status(void* stream)
{
    void* ws = nullptr;
    const sdpa_status_t st = no_alloc_scratch(&ws);
    if (st != SDPA_OK) return st;
    return sdpa_bwd_check_status(ws, stream);
}

size_t sdpa_bwd_params_bytes(void) { return sizeof(sdpa_bwd_params); }

int32_t sdpa_bwd_tile_kv(void) { return swa::kTileKV; }
int32_t sdpa_bwd_tile_q(void) { return swa::kTileQ; }

int32_t sdpa_bwd_kernel_launches(const sdpa_bwd_params* p)
{
    if (check_shape(p) != SDPA_OK) return -1;
    g_last_error.clear();
    const swa::WsLayout w = layout_of(p);
    const int64_t n_kv_tiles = (p->s_kv + swa::kTileKV - 1) / swa::kTileKV;
    const int64_t stats_row = ((p->s_q + swa::kTileQ - 1) / swa::kTileQ) * swa::kTileQ;
    int32_t n = 0;
    // the preprocess: a memset instead when there are no rows
    if (w.n_row_blocks > 0 && stats_row > 0 && p->b > 0 && p->h_q > 0) ++n;
    // the main kernel: nothing without work items or keys
    if (p->b * p->h_q * n_kv_tiles != 0 && rows_kv(p) != 0 && p->b * p->h_kv * n_kv_tiles > 0) ++n;
    // the dQ convert
    if (w.n_row_blocks > 0 && p->s_q > 0 && p->b > 0 && p->h_q > 0 && convert_has_work(p, geometry_of(p))) ++n;
    return n;
}

}  // extern "C"

// ---------------------------------------------------------------- forward

namespace {

// The forward's device status word (timeouts), one per device; as for the
// allocation-free scratch above, host code takes its device address from
// cudaGetSymbolAddress on every call. Every forward on a device shares it.
static __device__ int32_t g_fwd_status;

sdpa_status_t fwd_status_word(int32_t** out)
{
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fwd_status);
    if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return fail(SDPA_ERR_CUDA, "sdpa_fwd: cannot resolve the status word on the current device (%s)",
                    cudaGetErrorString(e));
    }
    *out = static_cast<int32_t*>(p);
    return SDPA_OK;
}

// The fields the two passes share, in the backward's parameter block, so that
// the forward uses the same validation and geometry.
sdpa_bwd_params fwd_view(const sdpa_fwd_params* f)
{
    sdpa_bwd_params p{};
    p.dtype = f->dtype;
    p.layout = f->layout;
    p.mask_mode = f->mask_mode;
    p.deterministic = 0;
    p.b = f->b;
    p.h_q = f->h_q;
    p.h_kv = f->h_kv;
    p.s_q = f->s_q;
    p.s_kv = f->s_kv;
    p.total_q = f->total_q;
    p.total_kv = f->total_kv;
    p.d = f->d;
    p.window_left = f->window_left;
    p.window_right = f->window_right;
    p.scale = f->scale;
    p.seq_q_lens = f->seq_q_lens;
    p.seq_kv_lens = f->seq_kv_lens;
    p.q_offsets = f->q_offsets;
    p.kv_offsets = f->kv_offsets;
    p.q = f->q;
    p.k = f->k;
    p.v = f->v;
    p.o = f->o;
    p.lse = f->lse;
    p.sink = f->sink;
    p.dsink = const_cast<float*>(f->sink);  // the pairing check has no forward meaning
    copy3(p.q_stride, f->q_stride);
    copy3(p.k_stride, f->k_stride);
    copy3(p.v_stride, f->v_stride);
    copy3(p.o_stride, f->o_stride);
    return p;
}

}  // namespace

extern "C" {

sdpa_status_t sdpa_fwd(const sdpa_fwd_params* f, void* stream)
{
    if (f == nullptr) return fail(SDPA_ERR_INVALID_ARG, "params is NULL");
    const sdpa_bwd_params p = fwd_view(f);
    sdpa_status_t st = check_shape(&p);
    if (st != SDPA_OK) return st;
    const bool thd = p.layout == SDPA_THD;
    const struct { const char* n; const int64_t* s; } strides[] = {
        {"q", p.q_stride}, {"k", p.k_stride}, {"v", p.v_stride}, {"o", p.o_stride}};
    for (const auto& x : strides)
        if ((st = check_strides(x.n, x.s, thd)) != SDPA_OK) return st;
    const int64_t n_q_tiles = (p.s_q + swa::kTileQ - 1) / swa::kTileQ;
    if (p.b * p.h_q * n_q_tiles >= (int64_t(1) << 31))
        return fail(SDPA_ERR_UNSUPPORTED, "%lld forward work items (b x h_q x ceil(s_q/128)): at most 2^31 - 1",
                    (long long)(p.b * p.h_q * n_q_tiles));
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return fail(SDPA_ERR_CUDA, "no CUDA device available");
    }
    const int64_t rq = rows_q(&p), rk = rows_kv(&p);
    const struct { const char* n; const void* ptr; bool req; } ptrs[] = {
        {"q", p.q, rq > 0},   {"k", p.k, rk > 0},   {"v", p.v, rk > 0},  {"o", p.o, rq > 0},
        {"lse", p.lse, rq > 0}, {"sink", p.sink, false}, {"seq_q_lens", p.seq_q_lens, false},
        {"seq_kv_lens", p.seq_kv_lens, false}, {"q_offsets", p.q_offsets, thd}, {"kv_offsets", p.kv_offsets, thd}};
    for (const auto& x : ptrs)
        if ((st = check_device_ptr(x.n, x.ptr, x.req, dev)) != SDPA_OK) return st;
    if (rq == 0 || p.b == 0) return SDPA_OK;  // no row to write
    swa::FwdArgs a{};
    if ((st = fwd_status_word(&a.status)) != SDPA_OK) return st;
    a.g = geometry_of(&p);
    a.g.ext = extents_of(&p, nullptr);
    a.o = f->o;
    a.lse = f->lse;
    a.sink = f->sink;
    copy3(a.o_stride, f->o_stride);
    a.n_q_tiles = n_q_tiles;
    a.scale_log2 = f->scale * 1.4426950408889634f;
    a.timeout_ns = kWaitLimitNs;
    // the maps' row extent is one sequence slot (BSHD: s, where a 4-D map
    // clips boxes that overhang it) or the packed tokens (THD)
    const int64_t rq_map = thd ? p.total_q : p.s_q, rk_map = thd ? p.total_kv : p.s_kv;
    if ((st = make_map(&a.tm_q, "q", p.q, p.dtype, thd, p.d, p.h_q, rq_map, p.b, p.q_stride)) != SDPA_OK ||
        (st = make_map(&a.tm_o, "o", p.o, p.dtype, thd, p.d, p.h_q, rq_map, p.b, p.o_stride)) != SDPA_OK)
        return st;
    if (rk > 0) {
        if ((st = make_map(&a.tm_k, "k", p.k, p.dtype, thd, p.d, p.h_kv, rk_map, p.b, p.k_stride)) != SDPA_OK ||
            (st = make_map(&a.tm_v, "v", p.v, p.dtype, thd, p.d, p.h_kv, rk_map, p.b, p.v_stride)) != SDPA_OK)
            return st;
    } else {
        // no keys anywhere: no row admits one and K, V are never loaded
        a.tm_k = a.tm_q;
        a.tm_v = a.tm_q;
    }
    return cuda_status(swa::launch_fwd(a, p.dtype, static_cast<cudaStream_t>(stream)), "forward launch");
}

sdpa_status_t sdpa_fwd_check_status(void* stream)
{
    int32_t* word = nullptr;
    sdpa_status_t st = fwd_status_word(&word);
    if (st != SDPA_OK) return st;
    if ((st = cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream synchronize")) != SDPA_OK)
        return st;
    int32_t host = 0;
    if ((st = cuda_status(cudaMemcpy(&host, word, sizeof(host), cudaMemcpyDeviceToHost), "status read")) != SDPA_OK)
        return st;
    if (host == 0) return SDPA_OK;
    if ((st = cuda_status(cudaMemset(word, 0, sizeof(int32_t)), "status reset")) != SDPA_OK) return st;
    if (host == SDPA_ERR_TIMEOUT) return fail(SDPA_ERR_TIMEOUT, "a forward wait ran out on the device");
    if (host == SDPA_ERR_BOUNDS)
        return fail(SDPA_ERR_BOUNDS, "a forward index fell outside its buffer (range-checked build)");
    if (host == SDPA_ERR_UNSUPPORTED)
        return fail(SDPA_ERR_UNSUPPORTED, "the device gave the forward kernel shared memory not 1024-byte aligned");
    return fail(SDPA_ERR_CUDA, "unknown forward device status %d", host);
}

size_t sdpa_fwd_params_bytes(void) { return sizeof(sdpa_fwd_params); }

}  // extern "C"
