"""Parity of the CUDA forward (O, LSE) with the fp64 oracle's forward, element
by element, on the same seeded inputs (the cases of the backward's parity
tests: masks, windows, GQA, sinks, padding, THD, d = 128, f16). O is compared
with the I/O dtype's tolerance; LSE must be -inf exactly where the oracle's is
and within 2e-3 elsewhere (fp32 logits from 16-bit inputs, fp32 sums)."""
import numpy as np
import pytest
import torch

from swa_cases import Case, build, compare
from test_gpu_parity import FULL, SMALL

pytestmark = pytest.mark.gpu

FWD_CASES = SMALL + [
    # an empty sequence and rows past every window in one batch
    Case("fwd_thd_empty_and_tiny", 0, 4, 2, 0, 0, 64, "tl", 32, layout="thd",
         thd_lens=[0, 5, 300, 129], slot_align=1, seed=40),
    Case("fwd_none_w0", 1, 2, 2, 260, 260, 128, "none", 0, seed=41),
]


def run_forward(bt, **over):
    import sliding_window_attention_sdpa_gb300 as swa
    d, kw = bt.dev, dict(bt.kwargs)
    kw.pop("deterministic", None)
    kw.update(over)
    o, lse = swa.forward(d["q"], d["k"], d["v"], check_status=True, **kw)
    torch.cuda.synchronize()
    return o, lse


def check_forward(bt, o, lse):
    c = bt.case
    compare(f"{c.name} o", o, bt.ref_o, c.dtype)
    got = lse.double().cpu().numpy()
    want = bt.ref_lse
    assert got.shape == want.shape, f"{c.name} lse shape {got.shape} vs {want.shape}"
    inf_w, inf_g = np.isneginf(want), np.isneginf(got)
    assert np.array_equal(inf_w, inf_g), f"{c.name}: -inf rows differ ({inf_w.sum()} vs {inf_g.sum()})"
    assert np.all(np.isfinite(got[~inf_g])), f"{c.name}: non-finite LSE"
    err = np.abs(got[~inf_w] - want[~inf_w])
    assert err.size == 0 or err.max() <= 2e-3, f"{c.name}: LSE max error {err.max():.3e}"


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: c.name)
def test_forward_parity(case):
    bt = build(case)
    o, lse = run_forward(bt)
    check_forward(bt, o, lse)


def test_forward_feeds_backward():
    """The forward's O and LSE, given to the backward, give the gradients the
    oracle gets from its own O and LSE."""
    import sliding_window_attention_sdpa_gb300 as swa
    from swa_cases import check_all
    case = Case("fwd_bwd_chain_gqa_sink", 2, 4, 2, 333, 333, 64, "br", 100, sink=True, seed=42)
    bt = build(case)
    o, lse = run_forward(bt)
    check_forward(bt, o, lse)
    d = bt.dev
    out = swa.backward(d["q"], d["k"], d["v"], o, d["do"], lse, check_status=True, **bt.kwargs)
    torch.cuda.synchronize()
    check_all(bt, out)


def test_forward_is_repeatable():
    bt = build(Case("fwd_repeat", 1, 2, 2, 700, 700, 64, "tl", 200, seed=43))
    o1, l1 = run_forward(bt)
    o2, l2 = run_forward(bt)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# the forward has no deterministic mode: one case per input set
FWD_FULL = [(c, u) for c, u in FULL if not c.det]


@pytest.mark.parametrize("case,units", FWD_FULL, ids=lambda x: x.name if isinstance(x, Case) else "")
def test_forward_full_size_sampled(case, units):
    """The benchmark's full-size workloads in the launch configuration the
    benchmark times (every CTA walks several items per slot): the forward of
    the whole problem, compared on the oracle's sampled (sequence, kv-head)
    units."""
    import sliding_window_attention_sdpa_gb300 as swa
    bt = build(case, units=units)
    d, kw = bt.dev, dict(bt.kwargs)
    kw.pop("deterministic", None)
    o, lse = swa.forward(d["q"], d["k"], d["v"], check_status=True, **kw)
    torch.cuda.synchronize()
    assert bt.fwd_checks
    for label, osel, o_want, lsel, l_want in bt.fwd_checks:
        compare(f"{case.name} o{label}", osel(o), o_want, case.dtype)
        got = lsel(lse).double().cpu().numpy()
        inf_w, inf_g = np.isneginf(l_want), np.isneginf(got)
        assert np.array_equal(inf_w, inf_g), f"{case.name} lse{label}: -inf rows differ"
        err = np.abs(got[~inf_w] - l_want[~inf_w])
        assert err.size == 0 or err.max() <= 2e-3, f"{case.name} lse{label}: max error {err.max():.3e}"
    del bt, o, lse
    torch.cuda.empty_cache()
