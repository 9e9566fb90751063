"""GB300 (sm_103a) sliding-window SDPA backward.

Thin Python binding over the C ABI of ``include/sdpa_bwd.h`` (ctypes; argument
marshalling only -- every step of the backward runs in the CUDA library). The
functions ``sdpa_bwd_workspace_bytes``, ``sdpa_bwd_preprocess``, ``sdpa_bwd``,
``sdpa_bwd_dq_convert``, ``sdpa_bwd_gqa_reduce`` and ``sdpa_bwd_check_status``
mirror the C entry points one to one; ``backward()`` is the convenience call a
PyTorch user makes (it allocates outputs and the workspace with torch and runs
the four kernels on the current stream).

If the compiled library is missing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import _build

SDPA_OK, SDPA_ERR_INVALID_ARG, SDPA_ERR_UNSUPPORTED, SDPA_ERR_CUDA = 0, 1, 2, 3
SDPA_ERR_TIMEOUT, SDPA_ERR_BAD_LENGTHS, SDPA_ERR_WORKSPACE, SDPA_ERR_BOUNDS = 4, 5, 6, 7
SDPA_BF16, SDPA_F16 = 0, 1
SDPA_BSHD, SDPA_THD = 0, 1
SDPA_MASK_NONE, SDPA_MASK_TOP_LEFT, SDPA_MASK_BOTTOM_RIGHT = 0, 1, 2

ENTRY_POINTS = ("sdpa_bwd_workspace_bytes", "sdpa_bwd_preprocess", "sdpa_bwd",
                "sdpa_bwd_dq_convert", "sdpa_bwd_gqa_reduce", "sdpa_bwd_check_status",
                "sdpa_bwd_last_error", "sdpa_bwd_params_bytes", "sdpa_bwd_tile_kv",
                "sdpa_bwd_tile_q", "sdpa_bwd_no_alloc", "sdpa_bwd_kernel_launches",
                "sdpa_fwd", "sdpa_fwd_check_status", "sdpa_fwd_params_bytes",
                "sdpa_bwd_test_hook", "sdpa_bwd_no_alloc_check_status")

_i64x3 = ctypes.c_int64 * 3


class SdpaBwdParams(ctypes.Structure):
    """Mirror of ``sdpa_bwd_params`` (field order and types as in the header)."""
    _fields_ = [
        ("dtype", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("mask_mode", ctypes.c_int32), ("deterministic", ctypes.c_int32),
        ("b", ctypes.c_int64), ("h_q", ctypes.c_int64), ("h_kv", ctypes.c_int64),
        ("s_q", ctypes.c_int64), ("s_kv", ctypes.c_int64),
        ("total_q", ctypes.c_int64), ("total_kv", ctypes.c_int64),
        ("d", ctypes.c_int64), ("window_left", ctypes.c_int64),
        ("window_right", ctypes.c_int64),
        ("scale", ctypes.c_float), ("reserved0", ctypes.c_int32),
        ("seq_q_lens", ctypes.c_void_p), ("seq_kv_lens", ctypes.c_void_p),
        ("q_offsets", ctypes.c_void_p), ("kv_offsets", ctypes.c_void_p),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("dout", ctypes.c_void_p),
        ("lse", ctypes.c_void_p), ("sink", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("dsink", ctypes.c_void_p),
        ("q_stride", _i64x3), ("k_stride", _i64x3), ("v_stride", _i64x3),
        ("o_stride", _i64x3), ("do_stride", _i64x3),
        ("dq_stride", _i64x3), ("dk_stride", _i64x3), ("dv_stride", _i64x3),
    ]


class SdpaFwdParams(ctypes.Structure):
    """Mirror of ``sdpa_fwd_params`` (field order and types as in the header)."""
    _fields_ = [
        ("dtype", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("mask_mode", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("b", ctypes.c_int64), ("h_q", ctypes.c_int64), ("h_kv", ctypes.c_int64),
        ("s_q", ctypes.c_int64), ("s_kv", ctypes.c_int64),
        ("total_q", ctypes.c_int64), ("total_kv", ctypes.c_int64), ("d", ctypes.c_int64),
        ("window_left", ctypes.c_int64), ("window_right", ctypes.c_int64),
        ("scale", ctypes.c_float), ("reserved1", ctypes.c_int32),
        ("seq_q_lens", ctypes.c_void_p), ("seq_kv_lens", ctypes.c_void_p),
        ("q_offsets", ctypes.c_void_p), ("kv_offsets", ctypes.c_void_p),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("sink", ctypes.c_void_p), ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("q_stride", _i64x3), ("k_stride", _i64x3), ("v_stride", _i64x3), ("o_stride", _i64x3),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    """The in-tree library, or the one SWA_SDPA_LIB names (e.g. the
    range-checked build, libswa_sdpa_bwd_dbg.so)."""
    return os.environ.get("SWA_SDPA_LIB") or _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load the compiled library (raises if it is missing and not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"CUDA library {path} is not built; run __graft_entry__.build() or "
                    "python -m sliding_window_attention_sdpa_gb300._build")
            _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(SdpaBwdParams)
        vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        lib.sdpa_bwd_workspace_bytes.argtypes = [P]
        lib.sdpa_bwd_workspace_bytes.restype = sz
        for name in ("sdpa_bwd_preprocess", "sdpa_bwd", "sdpa_bwd_dq_convert",
                     "sdpa_bwd_gqa_reduce"):
            f = getattr(lib, name)
            f.argtypes = [P, vp, sz, vp]
            f.restype = st
        lib.sdpa_bwd_no_alloc.argtypes = [P, vp]
        lib.sdpa_bwd_no_alloc.restype = st
        lib.sdpa_bwd_check_status.argtypes = [vp, vp]
        lib.sdpa_bwd_check_status.restype = st
        lib.sdpa_bwd_last_error.argtypes = []
        lib.sdpa_bwd_last_error.restype = ctypes.c_char_p
        lib.sdpa_bwd_params_bytes.restype = sz
        lib.sdpa_bwd_tile_kv.restype = ctypes.c_int32
        lib.sdpa_bwd_tile_q.restype = ctypes.c_int32
        lib.sdpa_bwd_kernel_launches.argtypes = [P]
        lib.sdpa_bwd_kernel_launches.restype = ctypes.c_int32
        lib.sdpa_bwd_test_hook.argtypes = [ctypes.c_int64, ctypes.c_int32]
        lib.sdpa_bwd_test_hook.restype = st
        lib.sdpa_bwd_no_alloc_check_status.argtypes = [vp]
        lib.sdpa_bwd_no_alloc_check_status.restype = st
        lib.sdpa_fwd.argtypes = [ctypes.POINTER(SdpaFwdParams), vp]
        lib.sdpa_fwd.restype = st
        lib.sdpa_fwd_check_status.argtypes = [vp]
        lib.sdpa_fwd_check_status.restype = st
        lib.sdpa_fwd_params_bytes.restype = sz
        _lib = lib
        return lib


class SdpaError(RuntimeError):
    def __init__(self, code: int, where: str, message: str):
        super().__init__(f"{where} failed with status {code}: {message}")
        self.code = code


def last_error() -> str:
    return load().sdpa_bwd_last_error().decode()


def _check(code: int, where: str) -> int:
    if code != SDPA_OK:
        raise SdpaError(code, where, last_error())
    return code


# ----------------------------------------------------- one-to-one C entry points

def sdpa_bwd_workspace_bytes(params: SdpaBwdParams) -> int:
    return int(load().sdpa_bwd_workspace_bytes(ctypes.byref(params)))


def sdpa_bwd_kernel_launches(params: SdpaBwdParams) -> int:
    return int(load().sdpa_bwd_kernel_launches(ctypes.byref(params)))


def sdpa_bwd_preprocess(params, workspace: int, workspace_bytes: int, stream: int) -> int:
    return load().sdpa_bwd_preprocess(ctypes.byref(params), workspace, workspace_bytes, stream)


def sdpa_bwd(params, workspace: int, workspace_bytes: int, stream: int) -> int:
    return load().sdpa_bwd(ctypes.byref(params), workspace, workspace_bytes, stream)


def sdpa_bwd_dq_convert(params, workspace: int, workspace_bytes: int, stream: int) -> int:
    return load().sdpa_bwd_dq_convert(ctypes.byref(params), workspace, workspace_bytes, stream)


def sdpa_bwd_gqa_reduce(params, workspace: int, workspace_bytes: int, stream: int) -> int:
    return load().sdpa_bwd_gqa_reduce(ctypes.byref(params), workspace, workspace_bytes, stream)


def sdpa_bwd_check_status(workspace: int, stream: int) -> int:
    return load().sdpa_bwd_check_status(workspace, stream)


# Largest scratch (bytes) sdpa_bwd_no_alloc can serve; see include/sdpa_bwd.h.
SDPA_BWD_NO_ALLOC_MAX_BYTES = 32 << 20


def sdpa_bwd_no_alloc_check_status(stream: int) -> int:
    """Device status of the last sdpa_bwd_no_alloc run on this device."""
    return load().sdpa_bwd_no_alloc_check_status(stream)


def sdpa_bwd_test_hook(wait_limit_ns: int, flags: int) -> int:
    """Test-only: device wait limit and unreachable-wait flags for this
    thread's later sdpa_bwd calls (see the C header); (0, 0) restores them."""
    return load().sdpa_bwd_test_hook(int(wait_limit_ns), int(flags))


def sdpa_bwd_no_alloc(params, stream: int) -> int:
    """Whole backward with the library's own fixed scratch: for callers that
    cannot allocate device memory (no workspace argument, no allocation)."""
    return load().sdpa_bwd_no_alloc(ctypes.byref(params), stream)


# ------------------------------------------------------------- torch helpers

def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _strides(t, layout: int):
    if t is None:
        return (0, 0, 0)
    if t.numel() == 0:  # no element is ever addressed: report packed strides
        s = [1] * t.dim()
        for i in range(t.dim() - 2, -1, -1):
            s[i] = s[i + 1] * max(t.shape[i + 1], 1)
        return (0, s[0], s[1]) if layout == SDPA_THD else (s[0], s[1], s[2])
    s = t.stride()
    if t.stride(-1) != 1:
        raise ValueError("the feature dimension must be contiguous (stride 1)")
    if layout == SDPA_THD:   # [T, H, D]
        return (0, s[0], s[1])
    return (s[0], s[1], s[2])  # [B, S, H, D]


def make_params(q, k, v, o, dout, lse, dq, dk, dv, *, scale: float,
                mask_mode: int = SDPA_MASK_TOP_LEFT, window_left: int = -1,
                window_right: int = -1, deterministic: int = 0,
                seq_q_lens=None, seq_kv_lens=None, q_offsets=None, kv_offsets=None,
                max_seqlen_q: Optional[int] = None, max_seqlen_kv: Optional[int] = None,
                sink=None, dsink=None) -> SdpaBwdParams:
    """Fill an SdpaBwdParams from torch tensors (BSHD if q is 4-D, THD if 3-D)."""
    import torch
    thd = q.dim() == 3
    layout = SDPA_THD if thd else SDPA_BSHD
    if q.dtype == torch.bfloat16:
        dtype = SDPA_BF16
    elif q.dtype == torch.float16:
        dtype = SDPA_F16
    else:
        raise ValueError(f"unsupported dtype {q.dtype}")
    p = SdpaBwdParams()
    p.dtype, p.layout, p.mask_mode = dtype, layout, mask_mode
    # False/0: unordered atomics; True/1: bitwise repeatable (per-visitor
    # slots where they apply, else the relay); 2: bitwise repeatable, relay only
    p.deterministic = int(deterministic) if deterministic in (0, 1, 2) else 1
    if thd:
        if q_offsets is None or kv_offsets is None:
            raise ValueError("THD layout needs q_offsets and kv_offsets")
        p.b = q_offsets.numel() - 1
        p.total_q, p.total_kv = q.shape[0], k.shape[0]
        p.h_q, p.h_kv, p.d = q.shape[1], k.shape[1], q.shape[2]
        if max_seqlen_q is None or max_seqlen_kv is None:
            raise ValueError("THD layout needs max_seqlen_q / max_seqlen_kv (longest slot)")
        p.s_q, p.s_kv = max_seqlen_q, max_seqlen_kv
    else:
        p.b, p.s_q, p.h_q, p.d = q.shape
        p.s_kv, p.h_kv = k.shape[1], k.shape[2]
    p.window_left, p.window_right = window_left, window_right
    p.scale = scale
    p.seq_q_lens, p.seq_kv_lens = _ptr(seq_q_lens), _ptr(seq_kv_lens)
    p.q_offsets, p.kv_offsets = _ptr(q_offsets), _ptr(kv_offsets)
    p.q, p.k, p.v, p.o, p.dout = map(_ptr, (q, k, v, o, dout))
    p.lse, p.sink = _ptr(lse), _ptr(sink)
    p.dq, p.dk, p.dv, p.dsink = map(_ptr, (dq, dk, dv, dsink))
    p.q_stride = _i64x3(*_strides(q, layout))
    p.k_stride = _i64x3(*_strides(k, layout))
    p.v_stride = _i64x3(*_strides(v, layout))
    p.o_stride = _i64x3(*_strides(o, layout))
    p.do_stride = _i64x3(*_strides(dout, layout))
    p.dq_stride = _i64x3(*_strides(dq, layout))
    p.dk_stride = _i64x3(*_strides(dk, layout))
    p.dv_stride = _i64x3(*_strides(dv, layout))
    return p


def run(params: SdpaBwdParams, workspace, stream: Optional[int] = None) -> None:
    """Enqueue the four kernels of the backward on `stream` (torch's current
    stream by default). `workspace` is a uint8 CUDA tensor of at least
    sdpa_bwd_workspace_bytes(params) bytes."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    ws, nb = workspace.data_ptr(), workspace.numel()
    _check(sdpa_bwd_preprocess(params, ws, nb, stream), "sdpa_bwd_preprocess")
    _check(sdpa_bwd(params, ws, nb, stream), "sdpa_bwd")
    _check(sdpa_bwd_dq_convert(params, ws, nb, stream), "sdpa_bwd_dq_convert")
    _check(sdpa_bwd_gqa_reduce(params, ws, nb, stream), "sdpa_bwd_gqa_reduce")


def alloc_workspace(params: SdpaBwdParams, device):
    import torch
    n = sdpa_bwd_workspace_bytes(params)
    if n == 0:
        raise SdpaError(SDPA_ERR_INVALID_ARG, "sdpa_bwd_workspace_bytes", last_error())
    return torch.empty(n, dtype=torch.uint8, device=device)


def backward(q, k, v, o, dout, lse, *, scale: float, mask_mode: int = SDPA_MASK_TOP_LEFT,
             window_left: int = -1, window_right: int = -1, deterministic: int = 0,
             seq_q_lens=None, seq_kv_lens=None, q_offsets=None, kv_offsets=None,
             max_seqlen_q=None, max_seqlen_kv=None, sink=None, workspace=None,
             check_status: bool = False):
    """dQ, dK, dV (and dSink when `sink` is given) of sliding-window SDPA.

    Tensors live on one CUDA device: BSHD q/o/dout [b, s_q, h_q, d], k/v
    [b, s_kv, h_kv, d], lse fp32 [b, h_q, s_q]; or THD q [total_q, h_q, d],
    k/v [total_kv, h_kv, d], lse [h_q, total_q] with int32 offsets.
    Returns (dq, dk, dv, dsink_or_None).
    """
    import torch
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dsink = torch.empty(q.shape[-2], dtype=torch.float32, device=q.device) if sink is not None else None
    p = make_params(q, k, v, o, dout, lse, dq, dk, dv, scale=scale, mask_mode=mask_mode,
                    window_left=window_left, window_right=window_right,
                    deterministic=deterministic, seq_q_lens=seq_q_lens, seq_kv_lens=seq_kv_lens,
                    q_offsets=q_offsets, kv_offsets=kv_offsets, max_seqlen_q=max_seqlen_q,
                    max_seqlen_kv=max_seqlen_kv, sink=sink, dsink=dsink)
    if workspace is None:
        workspace = alloc_workspace(p, q.device)
    run(p, workspace)
    if check_status:
        _check(sdpa_bwd_check_status(workspace.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream),
               "sdpa_bwd_check_status")
    return dq, dk, dv, dsink


def sdpa_fwd(params: SdpaFwdParams, stream) -> int:
    return load().sdpa_fwd(ctypes.byref(params), stream)


def sdpa_fwd_check_status(stream) -> int:
    return load().sdpa_fwd_check_status(stream)


def make_fwd_params(q, k, v, o, lse, *, scale: float, mask_mode: int = SDPA_MASK_TOP_LEFT,
                    window_left: int = -1, window_right: int = -1, seq_q_lens=None,
                    seq_kv_lens=None, q_offsets=None, kv_offsets=None,
                    max_seqlen_q: Optional[int] = None, max_seqlen_kv: Optional[int] = None,
                    sink=None) -> SdpaFwdParams:
    """Fill an SdpaFwdParams from torch tensors (BSHD if q is 4-D, THD if 3-D)."""
    import torch
    thd = q.dim() == 3
    layout = SDPA_THD if thd else SDPA_BSHD
    if q.dtype == torch.bfloat16:
        dtype = SDPA_BF16
    elif q.dtype == torch.float16:
        dtype = SDPA_F16
    else:
        raise ValueError(f"unsupported dtype {q.dtype}")
    p = SdpaFwdParams()
    p.dtype, p.layout, p.mask_mode = dtype, layout, mask_mode
    if thd:
        if q_offsets is None or kv_offsets is None:
            raise ValueError("THD layout needs q_offsets and kv_offsets")
        if max_seqlen_q is None or max_seqlen_kv is None:
            raise ValueError("THD layout needs max_seqlen_q / max_seqlen_kv (longest slot)")
        p.b = q_offsets.numel() - 1
        p.total_q, p.total_kv = q.shape[0], k.shape[0]
        p.h_q, p.h_kv, p.d = q.shape[1], k.shape[1], q.shape[2]
        p.s_q, p.s_kv = max_seqlen_q, max_seqlen_kv
    else:
        p.b, p.s_q, p.h_q, p.d = q.shape
        p.s_kv, p.h_kv = k.shape[1], k.shape[2]
    p.window_left, p.window_right = window_left, window_right
    p.scale = scale
    p.seq_q_lens, p.seq_kv_lens = _ptr(seq_q_lens), _ptr(seq_kv_lens)
    p.q_offsets, p.kv_offsets = _ptr(q_offsets), _ptr(kv_offsets)
    p.q, p.k, p.v, p.sink, p.o, p.lse = map(_ptr, (q, k, v, sink, o, lse))
    p.q_stride = _i64x3(*_strides(q, layout))
    p.k_stride = _i64x3(*_strides(k, layout))
    p.v_stride = _i64x3(*_strides(v, layout))
    p.o_stride = _i64x3(*_strides(o, layout))
    return p


def forward(q, k, v, *, scale: float, mask_mode: int = SDPA_MASK_TOP_LEFT, window_left: int = -1,
            window_right: int = -1, seq_q_lens=None, seq_kv_lens=None, q_offsets=None,
            kv_offsets=None, max_seqlen_q=None, max_seqlen_kv=None, sink=None,
            check_status: bool = False):
    """O and LSE of sliding-window SDPA (the inputs `backward` takes).

    Layouts as in `backward`; returns (o, lse) with o like q and lse fp32
    [b, h_q, s_q] (BSHD) or [h_q, total_q] (THD).
    """
    import torch
    o = torch.empty_like(q)
    if q.dim() == 3:
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    else:
        lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=q.device)
    p = make_fwd_params(q, k, v, o, lse, scale=scale, mask_mode=mask_mode, window_left=window_left,
                        window_right=window_right, seq_q_lens=seq_q_lens, seq_kv_lens=seq_kv_lens,
                        q_offsets=q_offsets, kv_offsets=kv_offsets, max_seqlen_q=max_seqlen_q,
                        max_seqlen_kv=max_seqlen_kv, sink=sink)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    _check(sdpa_fwd(p, stream), "sdpa_fwd")
    if check_status:
        _check(sdpa_fwd_check_status(stream), "sdpa_fwd_check_status")
    return o, lse
