"""Test-side glue: builds one seeded problem, runs the fp64 oracle on it and
the CUDA path through the C ABI, and compares them element by element.

Inputs come from sliding_window_attention_sdpa_gb300.inputs (shared with the
bench); the oracle sees exactly the tensors the GPU sees: Q, K, V, dO in the
I/O dtype, O = the oracle forward rounded to the I/O dtype, LSE rounded to
fp32. Tolerances are those of the method's target (relative Frobenius error /
max-abs error): bf16 1e-2 / 5e-2, f16 5e-3 / 2e-2.

Full-size workloads are checked on sampled units: a unit is one (sequence,
kv-head) pair with all q-heads of its group. The oracle runs each unit as a
problem of its own (b = 1, h_kv = 1), which the oracle's pins show equal to the
same rows of the whole problem (GQA, padding and THD invariants); rows of the
other units get filler inputs (O = 0, LSE = 10) and are not compared.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

import oracle
from sliding_window_attention_sdpa_gb300 import inputs

TOL = {"bf16": (1e-2, 5e-2), "f16": (5e-3, 2e-2)}
MODES = {"none": oracle.MASK_NONE, "tl": oracle.MASK_TOP_LEFT, "br": oracle.MASK_BOTTOM_RIGHT}


@dataclass
class Case:
    name: str
    b: int
    h_q: int
    h_kv: int
    s_q: int
    s_kv: int
    d: int
    mask: str = "tl"
    wl: int = -1
    wr: int = -1
    dtype: str = "bf16"
    layout: str = "bshd"
    lens_q: Optional[List[int]] = None      # BSHD padding mask
    lens_kv: Optional[List[int]] = None
    thd_lens: Optional[List[int]] = None    # THD: q and kv lengths (equal)
    slot_align: int = 1
    sink: bool = False
    det: bool = False
    seed: int = 0
    gen_device: str = "cpu"

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d)


@dataclass
class Built:
    case: Case
    dev: dict       # device tensors (q, k, v, o, do, lse, sink)
    kwargs: dict    # keyword arguments of swa.backward
    checks: list    # (label, selector(outputs) -> tensor, expected numpy) triples
    dsink_heads: Optional[np.ndarray]
    dsink_want: Optional[np.ndarray]
    ref_o: Optional[np.ndarray] = None    # oracle forward (fp64), whole-problem builds
    ref_lse: Optional[np.ndarray] = None
    # sampled builds: (label, o selector, expected o, lse selector, expected lse)
    fwd_checks: list = field(default_factory=list)


def _f64(x):
    return x.double().cpu().numpy()


def build(case: Case, device="cuda", units=None) -> Built:
    thd = case.layout == "thd"
    G = case.h_q // case.h_kv
    io = inputs.DTYPES[case.dtype]
    if thd:
        lens = np.asarray(case.thd_lens, np.int32)
        offs = inputs.thd_offsets(lens, case.slot_align)
        total = int(offs[-1])
        nb = len(lens)
        q_shape, kv_shape = (total, case.h_q, case.d), (total, case.h_kv, case.d)
        slot_max = int(np.diff(offs).max()) if nb else 0
    else:
        nb = case.b
        q_shape = (case.b, case.s_q, case.h_q, case.d)
        kv_shape = (case.b, case.s_kv, case.h_kv, case.d)
    t = inputs.make_tensors(q_shape, kv_shape, case.h_q, case.dtype, case.seed, case.sink,
                            device=case.gen_device)
    sink_np = None if t.sink is None else _f64(t.sink)
    checks = []
    fwd_checks = []
    dsink_heads, dsink_want = None, None
    ref_o, ref_lse = None, None

    def problem(**kw):
        base = dict(d=case.d, scale=case.scale, mask_mode=MODES[case.mask],
                    window_left=case.wl, window_right=case.wr, has_sink=case.sink)
        base.update(kw)
        return oracle.Problem(**base)

    if units is None:
        # the whole problem in one oracle call
        if thd:
            prob = problem(b=nb, h_q=case.h_q, h_kv=case.h_kv, s_q=slot_max, s_kv=slot_max,
                           layout=oracle.THD, seq_q_lens=lens, seq_kv_lens=lens,
                           q_offsets=offs, kv_offsets=offs)
        else:
            prob = problem(b=case.b, h_q=case.h_q, h_kv=case.h_kv, s_q=case.s_q, s_kv=case.s_kv,
                           seq_q_lens=None if case.lens_q is None else np.asarray(case.lens_q, np.int32),
                           seq_kv_lens=None if case.lens_kv is None else np.asarray(case.lens_kv, np.int32))
        q, k, v, do = _f64(t.q), _f64(t.k), _f64(t.v), _f64(t.do)
        o, lse = oracle.forward(prob, q, k, v, sink_np)
        ref_o, ref_lse = o, lse
        o_io = torch.from_numpy(o).to(io)
        lse32 = torch.from_numpy(lse).float()
        dq, dk, dv, _, dsink = oracle.backward(prob, q, k, v, _f64(o_io), do,
                                               lse32.double().numpy(), sink_np)
        checks = [("dq", lambda out: out[0], dq), ("dk", lambda out: out[1], dk),
                  ("dv", lambda out: out[2], dv)]
        if case.sink:
            dsink_heads, dsink_want = np.arange(case.h_q), dsink
        o_dev, lse_dev = o_io.to(device), lse32.to(device)
    else:
        # filler for the rows no unit covers, then each unit on its own
        o_dev = torch.zeros(q_shape, dtype=io, device=device)
        lse_dev = torch.full((case.h_q, total) if thd else (case.b, case.h_q, case.s_q), 10.0,
                             dtype=torch.float32, device=device)
        ds_acc = np.zeros(case.h_q)
        ds_seen = np.zeros((nb, case.h_kv), bool)
        for bi, g in units:
            hs = slice(g * G, (g + 1) * G)
            ds_seen[bi, g] = True
            if thd:
                a, e = int(offs[bi]), int(offs[bi + 1])
                rows = slice(a, e)
                sub = lambda x, hh: x[rows, hh][None]
                lq = lkv = np.asarray([lens[bi]], np.int32)
                s_q = s_kv = e - a
            else:
                sub = lambda x, hh: x[bi:bi + 1, :, hh]
                lq = None if case.lens_q is None else np.asarray([case.lens_q[bi]], np.int32)
                lkv = None if case.lens_kv is None else np.asarray([case.lens_kv[bi]], np.int32)
                s_q, s_kv = case.s_q, case.s_kv
            prob = problem(b=1, h_q=G, h_kv=1, s_q=s_q, s_kv=s_kv, seq_q_lens=lq, seq_kv_lens=lkv)
            gs = slice(g, g + 1)
            q, do = _f64(sub(t.q, hs)), _f64(sub(t.do, hs))
            k, v = _f64(sub(t.k, gs)), _f64(sub(t.v, gs))
            snk = None if sink_np is None else sink_np[hs]
            o, lse = oracle.forward(prob, q, k, v, snk)
            o_io = torch.from_numpy(o).to(io)
            lse32 = torch.from_numpy(lse).float()
            dq, dk, dv, _, dsink = oracle.backward(prob, q, k, v, _f64(o_io), do,
                                                   lse32.double().numpy(), snk)
            if thd:
                o_dev[rows, hs] = o_io[0].to(device)
                lse_dev[hs, rows] = lse32[0].to(device)
                fwd_checks.append((f"[{bi},{g}]", lambda o_, r=rows, h=hs: o_[r, h], o[0],
                                   lambda l_, r=rows, h=hs: l_[h, r], lse[0]))
                checks += [
                    (f"dq[{bi},{g}]", lambda out, r=rows, h=hs: out[0][r, h], dq[0]),
                    (f"dk[{bi},{g}]", lambda out, r=rows, h=gs: out[1][r, h], dk[0]),
                    (f"dv[{bi},{g}]", lambda out, r=rows, h=gs: out[2][r, h], dv[0])]
            else:
                o_dev[bi, :, hs] = o_io[0].to(device)
                lse_dev[bi, hs] = lse32[0].to(device)
                fwd_checks.append((f"[{bi},{g}]", lambda o_, b_=bi, h=hs: o_[b_, :, h], o[0],
                                   lambda l_, b_=bi, h=hs: l_[b_, h], lse[0]))
                checks += [
                    (f"dq[{bi},{g}]", lambda out, b_=bi, h=hs: out[0][b_, :, h], dq[0]),
                    (f"dk[{bi},{g}]", lambda out, b_=bi, h=gs: out[1][b_, :, h], dk[0]),
                    (f"dv[{bi},{g}]", lambda out, b_=bi, h=gs: out[2][b_, :, h], dv[0])]
            if case.sink:
                ds_acc[hs] += dsink
        if case.sink:
            full = [g for g in range(case.h_kv) if ds_seen[:, g].all()]
            if full:
                dsink_heads = np.concatenate([np.arange(g * G, (g + 1) * G) for g in full])
                dsink_want = ds_acc[dsink_heads]

    to = lambda x: None if x is None else x.to(device)
    dev = dict(q=to(t.q), k=to(t.k), v=to(t.v), o=o_dev, do=to(t.do), lse=lse_dev,
               sink=to(t.sink))
    kw = dict(scale=case.scale, mask_mode=MODES[case.mask], window_left=case.wl,
              window_right=case.wr, deterministic=case.det, sink=dev["sink"])
    if thd:
        offs32 = torch.from_numpy(offs.astype(np.int32)).to(device)
        lens32 = torch.from_numpy(lens).to(device)
        kw.update(q_offsets=offs32, kv_offsets=offs32, seq_q_lens=lens32, seq_kv_lens=lens32,
                  max_seqlen_q=slot_max, max_seqlen_kv=slot_max)
    else:
        if case.lens_q is not None:
            kw["seq_q_lens"] = torch.tensor(case.lens_q, dtype=torch.int32, device=device)
        if case.lens_kv is not None:
            kw["seq_kv_lens"] = torch.tensor(case.lens_kv, dtype=torch.int32, device=device)
    return Built(case, dev, kw, checks, dsink_heads, dsink_want, ref_o, ref_lse, fwd_checks)


def run_gpu(bt: Built, **over):
    import sliding_window_attention_sdpa_gb300 as swa
    d = bt.dev
    kw = dict(bt.kwargs)
    kw.update(over)
    out = swa.backward(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"], check_status=True, **kw)
    torch.cuda.synchronize()
    return out


def compare(name, got, want, dtype):
    """Relative Frobenius and max-abs error of `got` against `want`; asserts the
    tolerance of `dtype` and returns (rel, maxabs)."""
    rel_tol, abs_tol = TOL[dtype]
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{name}: shape {got.shape} vs {want.shape}"
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = got - want
    nrm = np.linalg.norm(want)
    rel = float(np.linalg.norm(err) / nrm) if nrm > 0 else 0.0
    mx = float(np.abs(err).max()) if err.size else 0.0
    assert mx <= abs_tol, f"{name}: max-abs error {mx:.3e} > {abs_tol}"
    if nrm > 1e-3:
        assert rel <= rel_tol, f"{name}: relative error {rel:.3e} > {rel_tol}"
    return rel, mx


def check_all(bt: Built, out):
    c = bt.case
    res = {}
    for label, sel, want in bt.checks:
        res[label] = compare(f"{c.name} {label}", sel(out), want, c.dtype)
    if bt.dsink_heads is not None and out[3] is not None:
        res["dsink"] = compare(f"{c.name} dsink", out[3][torch.as_tensor(bt.dsink_heads)],
                               bt.dsink_want, c.dtype)
    return res
