"""The allocation-free entry point, sdpa_bwd_no_alloc.

It serves callers that cannot allocate device memory (a plug-in whose host
application owns all device memory, a latency-critical path that must avoid
cudaMalloc's synchronisation, a deployment that forbids allocation after
start-up): it runs the whole backward with a fixed scratch array inside the
library instead of a caller-provided workspace. These tests check, through the
C ABI, that two calls in a row give the same gradients as the workspace entry
points (within the bf16 tolerance of the other parity tests) and as the fp64
oracle, that deterministic mode still gives bitwise-repeatable gradients when
its per-visitor slots do not fit the scratch, that the device status of a run
can be read back without a workspace, and that a problem too large for the
fixed scratch is refused on the host.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import math

import numpy as np
import pytest
import torch

import sliding_window_attention_sdpa_gb300 as swa
from swa_cases import Case, build, check_all, compare


def test_oversized_problem_is_refused_on_the_host():
    swa._build.build()
    p = swa.SdpaBwdParams()
    p.dtype, p.layout, p.mask_mode = swa.SDPA_BF16, swa.SDPA_BSHD, swa.SDPA_MASK_TOP_LEFT
    p.b, p.h_q, p.h_kv, p.s_q, p.s_kv, p.d = 2, 16, 16, 8192, 8192, 64
    p.window_left, p.window_right, p.scale = 128, -1, 0.125
    need = swa.sdpa_bwd_workspace_bytes(p)
    assert need > swa.SDPA_BWD_NO_ALLOC_MAX_BYTES
    assert swa.sdpa_bwd_no_alloc(p, None) == swa.SDPA_ERR_WORKSPACE
    msg = swa.last_error()
    assert str(need) in msg and str(swa.SDPA_BWD_NO_ALLOC_MAX_BYTES) in msg


def test_deterministic_slots_give_way_to_the_relay():
    """A deterministic problem whose per-visitor dQ slots do not fit the fixed
    scratch, but whose relay-only workspace does, passes the size check (it
    runs in relay-only mode); only a later step can refuse it here (no device
    or no real tensors)."""
    swa._build.build()
    p = swa.SdpaBwdParams()
    p.dtype, p.layout, p.mask_mode = swa.SDPA_BF16, swa.SDPA_BSHD, swa.SDPA_MASK_TOP_LEFT
    p.b, p.h_q, p.h_kv, p.s_q, p.s_kv, p.d = 1, 4, 4, 4096, 4096, 64
    p.window_left, p.window_right, p.scale = 1024, -1, 0.125
    p.deterministic = 1
    assert swa.sdpa_bwd_workspace_bytes(p) > swa.SDPA_BWD_NO_ALLOC_MAX_BYTES
    p.deterministic = 2
    assert swa.sdpa_bwd_workspace_bytes(p) <= swa.SDPA_BWD_NO_ALLOC_MAX_BYTES
    p.deterministic = 1
    assert swa.sdpa_bwd_no_alloc(p, None) != swa.SDPA_ERR_WORKSPACE


@pytest.mark.gpu
def test_no_alloc_matches_workspace_entry_points_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    swa.load()
    # GQA + sink + padding so that every part of the scratch is in use
    case = Case("no_alloc_gqa_sink", 2, 4, 2, 300, 300, 64, "tl", 64, lens_q=[300, 211],
                lens_kv=[300, 211], sink=True, seed=31)
    bt = build(case)
    d = bt.dev
    ref = swa.backward(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"], check_status=True,
                       **bt.kwargs)
    torch.cuda.synchronize()
    want = [t.double().cpu().numpy() for t in ref]

    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = (torch.full_like(d[n], float("nan")) for n in ("q", "k", "v"))
        dsink = torch.full((case.h_q,), float("nan"), dtype=torch.float32, device=d["q"].device)
        kw = dict(bt.kwargs)
        sink = kw.pop("sink")
        p = swa.make_params(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"], dq, dk, dv,
                            sink=sink, dsink=dsink, **kw)
        assert swa.sdpa_bwd_workspace_bytes(p) <= swa.SDPA_BWD_NO_ALLOC_MAX_BYTES
        rc = swa.sdpa_bwd_no_alloc(p, stream)
        assert rc == swa.SDPA_OK, swa.last_error()
        torch.cuda.synchronize()
        for name, got, w in zip(("dq", "dk", "dv", "dsink"), (dq, dk, dv, dsink), want):
            compare(f"call {call} {name}", got, w, case.dtype)
        # and the oracle's gradients, element by element
        check_all(bt, (dq, dk, dv, dsink))
        assert swa.sdpa_bwd_no_alloc_check_status(stream) == swa.SDPA_OK, swa.last_error()


def _no_alloc(d, kw, stream, **over):
    """One sdpa_bwd_no_alloc call into fresh NaN-filled outputs."""
    kw = dict(kw)
    kw.update(over)
    kw.pop("sink", None)
    dq, dk, dv = (torch.full_like(d[n], float("nan")) for n in ("q", "k", "v"))
    p = swa.make_params(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"], dq, dk, dv, **kw)
    rc = swa.sdpa_bwd_no_alloc(p, stream)
    assert rc == swa.SDPA_OK, swa.last_error()
    torch.cuda.synchronize()
    return dq, dk, dv, p


@pytest.mark.gpu
def test_no_alloc_deterministic_without_slots_is_bitwise_repeatable():
    """Deterministic mode 1 whose per-visitor dQ slots exceed the fixed scratch
    runs as mode 2 (the relay): two calls give the same bits, the bits of the
    workspace entry points in mode 2, and the oracle's gradients."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    swa.load()
    case = Case("no_alloc_det_w1024", 1, 4, 4, 4096, 4096, 64, "tl", 1024, det=True, seed=32)
    bt = build(case)
    d = bt.dev
    stream = torch.cuda.current_stream().cuda_stream
    runs = []
    for _ in range(2):
        dq, dk, dv, p = _no_alloc(d, bt.kwargs, stream, deterministic=1)
        runs.append((dq, dk, dv))
    p.deterministic = 1
    assert swa.sdpa_bwd_workspace_bytes(p) > swa.SDPA_BWD_NO_ALLOC_MAX_BYTES
    p.deterministic = 2
    assert swa.sdpa_bwd_workspace_bytes(p) <= swa.SDPA_BWD_NO_ALLOC_MAX_BYTES
    ref = swa.backward(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"], check_status=True,
                       **dict(bt.kwargs, deterministic=2))
    torch.cuda.synchronize()
    for a, b, r in zip(runs[0], runs[1], ref[:3]):
        assert torch.equal(a, b) and torch.equal(a, r)
    check_all(bt, (*runs[0], None))
    assert swa.sdpa_bwd_no_alloc_check_status(stream) == swa.SDPA_OK, swa.last_error()


@pytest.mark.gpu
def test_no_alloc_status_reports_lengths_longer_than_the_slot():
    """A sequence length above s_q is clamped on the device (no access past the
    slot) and reported through sdpa_bwd_no_alloc_check_status; the next valid
    call reports SDPA_OK again."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    swa.load()
    case = Case("no_alloc_bad_len", 2, 2, 2, 256, 256, 64, "tl", 64, lens_q=[256, 200],
                lens_kv=[256, 200], seed=33)
    bt = build(case)
    d = bt.dev
    stream = torch.cuda.current_stream().cuda_stream
    bad = torch.tensor([256 + 5, 200], dtype=torch.int32, device=d["q"].device)
    _no_alloc(d, bt.kwargs, stream, seq_q_lens=bad)
    assert swa.sdpa_bwd_no_alloc_check_status(stream) == swa.SDPA_ERR_BAD_LENGTHS
    assert "length" in swa.last_error()
    dq, dk, dv, _ = _no_alloc(d, bt.kwargs, stream)
    assert swa.sdpa_bwd_no_alloc_check_status(stream) == swa.SDPA_OK, swa.last_error()
    check_all(bt, (dq, dk, dv, None))
