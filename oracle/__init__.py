"""fp64 CPU oracle for the sliding-window SDPA forward and backward.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. It shares no code with
the CUDA path: the arithmetic lives in ``swa_oracle.c`` (plain C, fp64), and
this module only builds it with gcc and marshals numpy arrays through ctypes.

The definition it follows, and the readings taken where the pages leave a step
open, are written at the top of ``swa_oracle.c``. Sources: the cuDNN-frontend
pull requests "frost(sdpa): bound the SM80 backward q-loop by the sliding
window ... + window-aware deterministic relay" (#866, "Change" section) and
"frost(sdpa): GQA/MQA, padding mask, right-band widening, and sink-token
gradients for the SM120 f16 backward" (#557, "Summary" section).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swa_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libswa_oracle.so")
_lock = threading.Lock()
_lib = None

BSHD, THD = 0, 1
MASK_NONE, MASK_TOP_LEFT, MASK_BOTTOM_RIGHT = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile swa_oracle.c into a shared library (no CUDA involved).

    -ffp-contract=off keeps gcc from fusing multiply-adds, so the oracle gives
    the same bits on x86-64 and AArch64.
    """
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
             _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("layout", ctypes.c_int32),
        ("mask_mode", ctypes.c_int32),
        ("b", ctypes.c_int64), ("h_q", ctypes.c_int64), ("h_kv", ctypes.c_int64),
        ("s_q", ctypes.c_int64), ("s_kv", ctypes.c_int64), ("d", ctypes.c_int64),
        ("window_left", ctypes.c_int64),
        ("window_right", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("seq_q_lens", ctypes.c_void_p),
        ("seq_kv_lens", ctypes.c_void_p),
        ("q_offsets", ctypes.c_void_p),
        ("kv_offsets", ctypes.c_void_p),
        ("has_sink", ctypes.c_int32),
        ("nthreads", ctypes.c_int32),
        ("unit_mask", ctypes.c_void_p),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Problem)
            dp = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.swa_attended.argtypes = [P, i64, i64, i64]
            lib.swa_attended.restype = ctypes.c_int
            lib.swa_len_q.argtypes = [P, i64]
            lib.swa_len_q.restype = i64
            lib.swa_len_kv.argtypes = [P, i64]
            lib.swa_len_kv.restype = i64
            lib.swa_diag.argtypes = [P, i64]
            lib.swa_diag.restype = i64
            lib.swa_forward.argtypes = [P, dp, dp, dp, dp, dp, dp, ctypes.c_int]
            lib.swa_forward.restype = None
            lib.swa_backward.argtypes = [P] + [dp] * 12 + [ctypes.c_int]
            lib.swa_backward.restype = None
            lib.swa_tile_q_range.argtypes = [P, i64, i64, i64, i64,
                                             ctypes.POINTER(i64), ctypes.POINTER(i64)]
            lib.swa_tile_q_range.restype = None
            lib.swa_kv_first.argtypes = [P, i64, i64, i64, i64]
            lib.swa_kv_first.restype = i64
            _lib = lib
    return _lib


@dataclass
class Problem:
    """Shape and mask of one attention problem (see swa_oracle.c for layouts).

    window_left / window_right < 0 mean "unbounded" (a causal mode treats a
    negative right bound as 0). For THD, q_offsets / kv_offsets are the token
    offsets of each sequence ([b+1]); lens may be shorter than the slots.
    """
    b: int
    h_q: int
    h_kv: int
    s_q: int
    s_kv: int
    d: int
    scale: float
    mask_mode: int = MASK_TOP_LEFT
    window_left: int = -1
    window_right: int = -1
    layout: int = BSHD
    seq_q_lens: Optional[np.ndarray] = None
    seq_kv_lens: Optional[np.ndarray] = None
    q_offsets: Optional[np.ndarray] = None
    kv_offsets: Optional[np.ndarray] = None
    has_sink: bool = False
    nthreads: int = field(default_factory=lambda: os.cpu_count() or 1)
    unit_mask: Optional[np.ndarray] = None

    def _c(self):
        keep = []

        def ptr(a, dt):
            if a is None:
                return None
            a = np.ascontiguousarray(a, dtype=dt)
            keep.append(a)
            return a.ctypes.data

        cp = _Problem(
            self.layout, self.mask_mode, self.b, self.h_q, self.h_kv, self.s_q, self.s_kv, self.d,
            self.window_left, self.window_right, float(self.scale),
            ptr(self.seq_q_lens, np.int32), ptr(self.seq_kv_lens, np.int32),
            ptr(self.q_offsets, np.int64), ptr(self.kv_offsets, np.int64),
            int(self.has_sink), int(self.nthreads), ptr(self.unit_mask, np.uint8))
        return cp, keep

    # shapes of the dense tensors in this layout
    def q_shape(self):
        if self.layout == THD:
            return (int(self.q_offsets[-1]), self.h_q, self.d)
        return (self.b, self.s_q, self.h_q, self.d)

    def kv_shape(self):
        if self.layout == THD:
            return (int(self.kv_offsets[-1]), self.h_kv, self.d)
        return (self.b, self.s_kv, self.h_kv, self.d)

    def stat_shape(self):
        if self.layout == THD:
            return (self.h_q, int(self.q_offsets[-1]))
        return (self.b, self.h_q, self.s_q)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def attended(p: Problem, bi: int, i: int, j: int) -> bool:
    cp, keep = p._c()
    return bool(_load().swa_attended(ctypes.byref(cp), bi, i, j))


def len_q(p: Problem, bi: int) -> int:
    cp, keep = p._c()
    return int(_load().swa_len_q(ctypes.byref(cp), bi))


def len_kv(p: Problem, bi: int) -> int:
    cp, keep = p._c()
    return int(_load().swa_len_kv(ctypes.byref(cp), bi))


def forward(p: Problem, q, k, v, sink=None, dense: bool = False, fill_lse: float = -np.inf):
    """O and LSE in fp64. Padded rows and rows of unselected units keep
    O = 0 and LSE = fill_lse."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    o = np.zeros(p.q_shape(), np.float64)
    lse = np.full(p.stat_shape(), fill_lse, np.float64)
    s = _f64(sink) if (p.has_sink and sink is not None) else None
    cp, keep = p._c()
    _load().swa_forward(ctypes.byref(cp), q.ctypes.data, k.ctypes.data, v.ctypes.data,
                        None if s is None else s.ctypes.data, o.ctypes.data, lse.ctypes.data,
                        int(dense))
    return o, lse


def backward(p: Problem, q, k, v, o, dout, lse, sink=None, dense: bool = False):
    """dQ, dK, dV, D (delta) and dSink in fp64 from the given O and LSE.

    Padded rows (and rows outside the selected units) are returned as 0.
    dSink is None without a sink.
    """
    q, k, v, o, dout, lse = map(_f64, (q, k, v, o, dout, lse))
    dq = np.zeros(p.q_shape(), np.float64)
    dk = np.zeros(p.kv_shape(), np.float64)
    dv = np.zeros(p.kv_shape(), np.float64)
    delta = np.zeros(p.stat_shape(), np.float64)
    dsink = np.zeros(p.h_q, np.float64) if p.has_sink else None
    s = _f64(sink) if p.has_sink else None
    cp, keep = p._c()
    _load().swa_backward(ctypes.byref(cp), q.ctypes.data, k.ctypes.data, v.ctypes.data,
                         o.ctypes.data, dout.ctypes.data, lse.ctypes.data,
                         None if s is None else s.ctypes.data,
                         dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, delta.ctypes.data,
                         None if dsink is None else dsink.ctypes.data, int(dense))
    return dq, dk, dv, delta, dsink


def tile_q_range(p: Problem, bi: int, t: int, tile_q: int, tile_kv: int):
    cp, keep = p._c()
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    _load().swa_tile_q_range(ctypes.byref(cp), bi, t, tile_q, tile_kv,
                             ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def kv_first(p: Problem, bi: int, j: int, tile_q: int, tile_kv: int) -> int:
    cp, keep = p._c()
    return int(_load().swa_kv_first(ctypes.byref(cp), bi, j, tile_q, tile_kv))


def attended_pairs(p: Problem) -> int:
    """Number of attended (q, k) pairs per head, summed over sequences
    (brute force over the predicate; small problems only)."""
    n = 0
    for bi in range(p.b):
        for i in range(len_q(p, bi)):
            for j in range(len_kv(p, bi)):
                n += attended(p, bi, i, j)
    return n
