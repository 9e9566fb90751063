"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test ties the oracle to something independent of its own code: a closed
form worked out by hand, a library routine (torch's CPU scaled-dot-product
attention in float64 and its autograd), central finite differences of the
oracle's own forward (which checks the backward formulas), statements printed
on the pages, or structural invariants (GQA = repeated MHA, THD = separate
runs, padding = truncation). Sources: cuDNN-frontend PR #866 "frost(sdpa):
bound the SM80 backward q-loop by the sliding window ..." ("Change" section)
and PR #557 "frost(sdpa): GQA/MQA, padding mask, right-band widening, and
sink-token gradients ..." ("Summary" section).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import BSHD, MASK_BOTTOM_RIGHT, MASK_NONE, MASK_TOP_LEFT, THD, Problem


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def data(p, seed, sink=False):
    q = rnd(p.q_shape(), seed)
    k = rnd(p.kv_shape(), seed + 1)
    v = rnd(p.kv_shape(), seed + 2)
    do = rnd(p.q_shape(), seed + 3)
    s = rnd((p.h_q,), seed + 4) if sink else None
    return q, k, v, do, s


def full_backward(p, q, k, v, do, s, dense=False):
    o, lse = oracle.forward(p, q, k, v, s, dense=dense)
    return (o, lse) + oracle.backward(p, q, k, v, o, do, lse, s, dense=dense)


# ---------------------------------------------------------------- closed forms

def test_hand_worked_two_token_example():
    """S=2, d=1, scale=1, causal: q=[1,2], k=[0,1], v=[3,5], dO=[1,1].
    Row 0 sees key 0 only; row 1 sees both with P = [a, c], a = 1/(1+e^2).
    By hand: O1 = 3a+5c, dS10 = -2ac, dS11 = 2ac, so dQ1 = 2ac, dK = [-4ac, 4ac],
    dV = [1+a, c], LSE = [0, log(1+e^2)]."""
    p = Problem(b=1, h_q=1, h_kv=1, s_q=2, s_kv=2, d=1, scale=1.0, window_left=1)
    q = np.array([1.0, 2.0]).reshape(1, 2, 1, 1)
    k = np.array([0.0, 1.0]).reshape(1, 2, 1, 1)
    v = np.array([3.0, 5.0]).reshape(1, 2, 1, 1)
    do = np.ones_like(q)
    o, lse, dq, dk, dv, delta, _ = full_backward(p, q, k, v, do, None)
    a = 1.0 / (1.0 + math.e ** 2)
    c = 1.0 - a
    np.testing.assert_allclose(o.ravel(), [3.0, 3 * a + 5 * c], rtol=1e-14)
    np.testing.assert_allclose(lse.ravel(), [0.0, math.log(1 + math.e ** 2)], rtol=1e-14)
    np.testing.assert_allclose(dq.ravel(), [0.0, 2 * a * c], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dk.ravel(), [-4 * a * c, 4 * a * c], rtol=1e-13)
    np.testing.assert_allclose(dv.ravel(), [1 + a, c], rtol=1e-14)
    np.testing.assert_allclose(delta.ravel(), o.ravel(), rtol=1e-15)


def test_window_zero_is_identity_attention():
    """W=0 under top-left causal: every row attends only its own key, so
    P = I, O = V, dV = dO and dQ = dK = 0 exactly."""
    p = Problem(b=2, h_q=2, h_kv=2, s_q=9, s_kv=9, d=5, scale=0.37, window_left=0)
    q, k, v, do, _ = data(p, 1)
    o, lse, dq, dk, dv, delta, _ = full_backward(p, q, k, v, do, None)
    assert np.array_equal(o, v)
    assert np.array_equal(dv, do)
    assert not dq.any() and not dk.any()


def _torch_sdpa(q, k, v, do, causal, scale):
    """Library reference: torch SDPA (fp64, CPU) and its autograd, BSHD in."""
    tq, tk, tv = (torch.tensor(x).permute(0, 2, 1, 3).requires_grad_(True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                           scale=scale)
    out.backward(torch.tensor(do).permute(0, 2, 1, 3))
    back = lambda t: t.detach().permute(0, 2, 1, 3).numpy()
    return back(out), back(tq.grad), back(tk.grad), back(tv.grad)


@pytest.mark.parametrize("mode,window,causal", [
    (MASK_TOP_LEFT, -1, True), (MASK_TOP_LEFT, 40, True), (MASK_BOTTOM_RIGHT, 17, True),
    (MASK_NONE, -1, False), (MASK_NONE, 33, False)])
def test_wide_window_matches_library_sdpa(mode, window, causal):
    """A window at least as long as the sequence leaves plain (causal or full)
    softmax attention, which torch computes independently."""
    p = Problem(b=2, h_q=3, h_kv=3, s_q=17, s_kv=17, d=8, scale=0.3, mask_mode=mode,
                window_left=window)
    q, k, v, do, _ = data(p, 2)
    o, lse, dq, dk, dv, _, _ = full_backward(p, q, k, v, do, None)
    to, tdq, tdk, tdv = _torch_sdpa(q, k, v, do, causal, 0.3)
    for a, b in ((o, to), (dq, tdq), (dk, tdk), (dv, tdv)):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_sink_at_minus_infinity_is_no_sink():
    """A sink logit of -1e30 carries zero probability: bitwise the no-sink result."""
    p = Problem(b=1, h_q=2, h_kv=1, s_q=11, s_kv=11, d=4, scale=0.5, window_left=3)
    q, k, v, do, _ = data(p, 3)
    ps = Problem(**{**p.__dict__, "has_sink": True})
    a = full_backward(p, q, k, v, do, None)
    b = full_backward(ps, q, k, v, do, np.full(2, -1e30))
    for x, y in zip(a[:6], b[:6]):
        assert np.array_equal(x, y)
    assert np.array_equal(b[6], np.zeros(2))


@pytest.mark.parametrize("sink", [False, True])
def test_shift_invariance_of_dk(sink):
    """Softmax is invariant to adding a constant to a row's logits, so
    sum_j dS_ij = 0 without a sink and sum_k dK_k = 0 per (batch, kv-head).
    With a sink, sum_j dS_ij = P_sink,i * D_i, which gives
    sum_k dK_k = scale * sum_i P_sink,i D_i q_i and dSink = -sum_i P_sink,i D_i."""
    p = Problem(b=2, h_q=2, h_kv=2, s_q=13, s_kv=13, d=6, scale=0.4, window_left=4,
                has_sink=sink)
    q, k, v, do, s = data(p, 4, sink)
    o, lse, dq, dk, dv, delta, dsink = full_backward(p, q, k, v, do, s)
    tot = dk.sum(axis=1)  # [b, h_kv, d]
    if not sink:
        assert np.abs(tot).max() < 1e-12
    else:
        psink = np.exp(s[None, :, None] - lse)  # [b, h, s_q]
        want = 0.4 * np.einsum("bhi,bhi,bihd->bhd", psink, delta, q)
        np.testing.assert_allclose(tot, want, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dsink, -(psink * delta).sum(axis=(0, 2)), rtol=1e-12)


# ------------------------------------------------------- statements of the pages

def test_window_edge_from_relay_first_visitor():
    """PR #866 names the relay's first visitor of a q-tile whose first row is
    q_row0: kv_first = (q_row0 + diag - W) // tile_kv. So the row with anchor a
    reaches key a - W (inclusive edge), and the clamp says no row with anchor
    beyond key + W attends that key."""
    for mode in (MASK_TOP_LEFT, MASK_BOTTOM_RIGHT, MASK_NONE):
        p = Problem(b=1, h_q=1, h_kv=1, s_q=40, s_kv=64, d=1, scale=1.0, mask_mode=mode,
                    window_left=7)
        diag = 24 if mode == MASK_BOTTOM_RIGHT else 0
        for i in range(40):
            a = i + diag
            if 0 <= a - 7 < 64:
                assert oracle.attended(p, 0, i, a - 7)
            if 0 <= a - 8 < 64:
                assert not oracle.attended(p, 0, i, a - 8)


def test_causal_and_right_band():
    """Causal modes admit no key right of the anchor unless the right band
    (PR #557 "Right-band widening") widens it; the window-only mode has no
    right bound."""
    base = dict(b=1, h_q=1, h_kv=1, s_q=20, s_kv=20, d=1, scale=1.0, window_left=3)
    tl = Problem(**base, mask_mode=MASK_TOP_LEFT)
    wide = Problem(**base, mask_mode=MASK_TOP_LEFT, window_right=2)
    none = Problem(**base, mask_mode=MASK_NONE)
    for i in range(20):
        assert oracle.attended(tl, 0, i, i)
        assert not oracle.attended(tl, 0, i, i + 1)
        assert oracle.attended(wide, 0, i, min(i + 2, 19))
        assert not oracle.attended(wide, 0, i, i + 3)
        assert oracle.attended(none, 0, i, 19)


def test_dsink_matches_finite_difference_and_pages_formula():
    """dsink[h] = -sum_{b,q} exp(sink[h] - LSE[b,h,q]) * delta[b,h,q] (PR #557),
    over unpadded rows, equals the numerical derivative of sum(dO * O)."""
    lens = np.array([9, 5], np.int32)
    p = Problem(b=2, h_q=2, h_kv=1, s_q=9, s_kv=9, d=4, scale=0.6, window_left=2,
                has_sink=True, seq_q_lens=lens, seq_kv_lens=lens)
    q, k, v, do, s = data(p, 5, True)
    o, lse, dq, dk, dv, delta, dsink = full_backward(p, q, k, v, do, s)
    want = np.zeros(2)
    for bi in range(2):
        for h in range(2):
            for i in range(lens[bi]):
                want[h] -= math.exp(s[h] - lse[bi, h, i]) * delta[bi, h, i]
    np.testing.assert_allclose(dsink, want, rtol=1e-13)
    for h in range(2):
        e = np.zeros(2)
        e[h] = 1e-6
        lp = (do * oracle.forward(p, q, k, v, s + e)[0]).sum()
        lm = (do * oracle.forward(p, q, k, v, s - e)[0]).sum()
        assert abs((lp - lm) / 2e-6 - dsink[h]) < 1e-7 * max(1.0, abs(dsink[h]))


# --------------------------------------------------------- finite differences

FD_CASES = {
    "tl_w0": dict(mask_mode=MASK_TOP_LEFT, window_left=0),
    "tl_w1": dict(mask_mode=MASK_TOP_LEFT, window_left=1),
    "tl_w3_gqa": dict(mask_mode=MASK_TOP_LEFT, window_left=3, h_q=4, h_kv=2),
    "tl_nowin_mqa": dict(mask_mode=MASK_TOP_LEFT, window_left=-1, h_q=4, h_kv=1),
    "br_w3_kv_longer": dict(mask_mode=MASK_BOTTOM_RIGHT, window_left=3, s_kv=15),
    "br_w2_q_longer_sink": dict(mask_mode=MASK_BOTTOM_RIGHT, window_left=2, s_q=14, s_kv=9,
                                has_sink=True),
    "none_w3": dict(mask_mode=MASK_NONE, window_left=3),
    "none_w3_r2": dict(mask_mode=MASK_NONE, window_left=3, window_right=2),
    "tl_w2_right1_sink": dict(mask_mode=MASK_TOP_LEFT, window_left=2, window_right=1,
                              has_sink=True),
    "pad_br_w4": dict(mask_mode=MASK_BOTTOM_RIGHT, window_left=4,
                      seq_q_lens=np.array([10, 6], np.int32),
                      seq_kv_lens=np.array([12, 9], np.int32), s_q=10, s_kv=12),
}


def _numgrad(f, x, idx, eps=1e-6):
    x0 = x[idx]
    x[idx] = x0 + eps
    fp = f()
    x[idx] = x0 - eps
    fm = f()
    x[idx] = x0
    return (fp - fm) / (2 * eps)


@pytest.mark.parametrize("name", sorted(FD_CASES))
def test_backward_matches_finite_differences(name):
    """Central differences of L = sum(dO * O(Q, K, V, sink)) in fp64."""
    kw = dict(b=2, h_q=2, h_kv=2, s_q=12, s_kv=12, d=4, scale=0.45)
    kw.update(FD_CASES[name])
    p = Problem(**kw)
    q, k, v, do, s = data(p, 11, p.has_sink)
    o, lse, dq, dk, dv, delta, dsink = full_backward(p, q, k, v, do, s)
    loss = lambda: float((do * oracle.forward(p, q, k, v, s)[0]).sum())
    rng = np.random.default_rng(0)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        scale = max(1.0, np.abs(g).max())
        for _ in range(40):
            idx = tuple(rng.integers(0, n) for n in x.shape)
            assert abs(_numgrad(loss, x, idx) - g[idx]) < 1e-7 * scale, (name, idx)
    if p.has_sink:
        for h in range(p.h_q):
            assert abs(_numgrad(loss, s, (h,)) - dsink[h]) < 1e-7 * max(1.0, abs(dsink[h]))


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("mode", [MASK_TOP_LEFT, MASK_BOTTOM_RIGHT, MASK_NONE])
def test_window_sweep_equals_dense_sweep_bitwise(mode):
    """The window-bounded sweep (the method's reachable keys) adds the same
    terms in the same order as the full masked sweep: results are bitwise equal."""
    p = Problem(b=2, h_q=4, h_kv=2, s_q=37, s_kv=45, d=8, scale=0.3, mask_mode=mode,
                window_left=6, has_sink=True)
    q, k, v, do, s = data(p, 12, True)
    a = full_backward(p, q, k, v, do, s, dense=True)
    b = full_backward(p, q, k, v, do, s, dense=False)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_keys_outside_every_window_get_zero_gradient():
    """Bottom-right with Lkv > Lq: keys left of Lkv - Lq - W are attended by no
    row, so their dK and dV are exactly zero; the others are not."""
    p = Problem(b=1, h_q=2, h_kv=2, s_q=8, s_kv=30, d=4, scale=0.5,
                mask_mode=MASK_BOTTOM_RIGHT, window_left=5)
    q, k, v, do, _ = data(p, 13)
    o, lse, dq, dk, dv, _, _ = full_backward(p, q, k, v, do, None)
    dead = 30 - 8 - 5
    assert not dk[:, :dead].any() and not dv[:, :dead].any()
    assert np.abs(dv[:, dead:]).min(axis=-1).min() > 0


def test_gqa_equals_repeated_mha():
    """PR #557 GQA: H_q a multiple of H_kv. Equal to MHA with K/V repeated over
    the group and dK/dV summed over the group."""
    g = Problem(b=2, h_q=6, h_kv=2, s_q=14, s_kv=14, d=4, scale=0.5, window_left=3,
                has_sink=True)
    m = Problem(**{**g.__dict__, "h_kv": 6})
    q, k, v, do, s = data(g, 14, True)
    kr, vr = np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2)
    og, lg, dqg, dkg, dvg, _, dsg = full_backward(g, q, k, v, do, s)
    om, lm, dqm, dkm, dvm, _, dsm = full_backward(m, q, kr, vr, do, s)
    np.testing.assert_allclose(og, om, rtol=1e-14)
    np.testing.assert_allclose(dqg, dqm, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dkg, dkm.reshape(2, 14, 2, 3, 4).sum(3), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dvg, dvm.reshape(2, 14, 2, 3, 4).sum(3), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dsg, dsm, rtol=1e-13)


def test_padding_equals_truncated_runs():
    """PR #557 padding mask: a padded batch equals per-batch runs on the
    sequences cut to their actual lengths; padded rows get zero gradients."""
    lq, lkv = np.array([7, 11], np.int32), np.array([9, 4], np.int32)
    p = Problem(b=2, h_q=2, h_kv=1, s_q=11, s_kv=9, d=4, scale=0.5,
                mask_mode=MASK_BOTTOM_RIGHT, window_left=3, has_sink=True,
                seq_q_lens=lq, seq_kv_lens=lkv)
    q, k, v, do, s = data(p, 15, True)
    o, lse, dq, dk, dv, _, dsink = full_backward(p, q, k, v, do, s)
    ds_sum = np.zeros(2)
    for bi in range(2):
        a, c = lq[bi], lkv[bi]
        pb = Problem(b=1, h_q=2, h_kv=1, s_q=int(a), s_kv=int(c), d=4, scale=0.5,
                     mask_mode=MASK_BOTTOM_RIGHT, window_left=3, has_sink=True)
        r = full_backward(pb, q[bi:bi + 1, :a], k[bi:bi + 1, :c], v[bi:bi + 1, :c],
                          do[bi:bi + 1, :a], s)
        np.testing.assert_array_equal(o[bi:bi + 1, :a], r[0])
        np.testing.assert_array_equal(dq[bi:bi + 1, :a], r[2])
        np.testing.assert_array_equal(dk[bi:bi + 1, :c], r[3])
        np.testing.assert_array_equal(dv[bi:bi + 1, :c], r[4])
        assert not dq[bi, a:].any() and not dk[bi, c:].any() and not dv[bi, c:].any()
        ds_sum += r[6]
    np.testing.assert_allclose(dsink, ds_sum, rtol=1e-14)


def test_thd_equals_separate_sequences():
    """THD packing (PR #866: in-sequence indices, per-sequence bound): equal to
    one b=1 run per sequence; gap tokens between slots get zero gradients."""
    lens = np.array([5, 12, 1, 9], np.int32)
    offs = np.array([0, 8, 24, 32, 41], np.int64)
    p = Problem(b=4, h_q=4, h_kv=2, s_q=12, s_kv=12, d=4, scale=0.5, window_left=3,
                layout=THD, seq_q_lens=lens, seq_kv_lens=lens, q_offsets=offs,
                kv_offsets=offs, has_sink=True)
    q, k, v, do, s = data(p, 16, True)
    o, lse, dq, dk, dv, delta, dsink = full_backward(p, q, k, v, do, s)
    live = np.zeros(41, bool)
    ds_sum = np.zeros(4)
    for bi in range(4):
        a, n = offs[bi], lens[bi]
        live[a:a + n] = True
        pb = Problem(b=1, h_q=4, h_kv=2, s_q=int(n), s_kv=int(n), d=4, scale=0.5,
                     window_left=3, has_sink=True)
        sl = lambda x: x[None, a:a + n]
        r = full_backward(pb, sl(q), sl(k), sl(v), sl(do), s)
        np.testing.assert_array_equal(o[a:a + n], r[0][0])
        np.testing.assert_array_equal(lse[:, a:a + n], r[1][0])
        np.testing.assert_array_equal(dq[a:a + n], r[2][0])
        np.testing.assert_array_equal(dk[a:a + n], r[3][0])
        np.testing.assert_array_equal(dv[a:a + n], r[4][0])
        ds_sum += r[6]
    assert not dq[~live].any() and not dk[~live].any() and not dv[~live].any()
    np.testing.assert_allclose(dsink, ds_sum, rtol=1e-14)


def test_bottom_right_equals_front_padded_top_left():
    """Bottom-right alignment with Lq < Lkv places the last query on the last
    key: the same as top-left causal on Lkv queries keeping the last Lq rows."""
    br = Problem(b=1, h_q=2, h_kv=2, s_q=6, s_kv=15, d=4, scale=0.5,
                 mask_mode=MASK_BOTTOM_RIGHT, window_left=4)
    tl = Problem(**{**br.__dict__, "mask_mode": MASK_TOP_LEFT, "s_q": 15})
    q, k, v, _, _ = data(tl, 17)
    o_tl, lse_tl = oracle.forward(tl, q, k, v)
    o_br, lse_br = oracle.forward(br, q[:, 9:], k, v)
    np.testing.assert_array_equal(o_br, o_tl[:, 9:])
    np.testing.assert_array_equal(lse_br, lse_tl[:, :, 9:])


def test_rows_with_nothing_attended():
    """Bottom-right with Lq > Lkv: the first Lq - Lkv rows have a negative
    anchor and reach no key; without a sink they get LSE = -inf, O = 0, dQ = 0."""
    p = Problem(b=1, h_q=1, h_kv=1, s_q=10, s_kv=4, d=3, scale=0.5,
                mask_mode=MASK_BOTTOM_RIGHT, window_left=2)
    q, k, v, do, _ = data(p, 18)
    o, lse, dq, dk, dv, _, _ = full_backward(p, q, k, v, do, None)
    assert np.all(np.isneginf(lse[0, 0, :6])) and np.all(np.isfinite(lse[0, 0, 6:]))
    assert not o[0, :6].any() and not dq[0, :6].any()
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def test_bottom_right_longer_queries_equals_top_left_on_last_rows():
    """Bottom-right with Lq > Lkv puts query i at anchor i - (Lq - Lkv): the
    last Lkv rows are top-left causal on an Lkv x Lkv problem (same window),
    and the first Lq - Lkv rows reach no key, so they leave dK and dV alone."""
    br = Problem(b=1, h_q=2, h_kv=1, s_q=11, s_kv=5, d=4, scale=0.5,
                 mask_mode=MASK_BOTTOM_RIGHT, window_left=2)
    tl = Problem(**{**br.__dict__, "mask_mode": MASK_TOP_LEFT, "s_q": 5})
    q, k, v, do, _ = data(br, 19)
    o, lse, dq, dk, dv, _, _ = full_backward(br, q, k, v, do, None)
    o2, lse2, dq2, dk2, dv2, _, _ = full_backward(tl, q[:, 6:], k, v, do[:, 6:], None)
    np.testing.assert_array_equal(o[:, 6:], o2)
    np.testing.assert_array_equal(dq[:, 6:], dq2)
    np.testing.assert_array_equal(dk, dk2)
    np.testing.assert_array_equal(dv, dv2)
    assert not dq[:, :6].any() and np.all(np.isneginf(lse[:, :, :6]))


# ------------------------------------------------ integer identities (tiling)

def _geometries():
    for mode in (MASK_TOP_LEFT, MASK_BOTTOM_RIGHT, MASK_NONE):
        for (lq, lkv) in ((24, 24), (13, 29), (29, 13), (1, 7), (0, 5), (17, 0)):
            for wl in (-1, 0, 1, 3, 9, 40):
                for wr in (-1, 0, 2):
                    yield mode, lq, lkv, wl, wr


@pytest.mark.parametrize("tq,tk", [(4, 4), (4, 8), (8, 4), (3, 5)])
def test_clamped_q_range_covers_every_attended_pair(tq, tk):
    """PR #866 clamp: kv-tile t sweeps q-tiles [q_lo, q_hi) with
    q_hi = ceil((kv_base + tile_kv + W - diag) / tile_q). Brute force: every
    attended pair lies in its kv-tile's range; an empty range attends nothing;
    each q-tile's visitors are contiguous and start at kv_first."""
    for mode, lq, lkv, wl, wr in _geometries():
        lens_q, lens_kv = np.array([lq], np.int32), np.array([lkv], np.int32)
        p = Problem(b=1, h_q=1, h_kv=1, s_q=max(lq, 1), s_kv=max(lkv, 1), d=1, scale=1.0,
                    mask_mode=mode, window_left=wl, window_right=wr,
                    seq_q_lens=lens_q, seq_kv_lens=lens_kv)
        n_kv = -(-lkv // tk)
        n_q = -(-lq // tq)
        ranges = [oracle.tile_q_range(p, 0, t, tq, tk) for t in range(n_kv)]
        for i in range(lq):
            for j in range(lkv):
                if oracle.attended(p, 0, i, j):
                    lo, hi = ranges[j // tk]
                    assert lo <= i // tq < hi, (mode, lq, lkv, wl, wr, i, j)
        for jt in range(n_q):
            visitors = [t for t in range(n_kv) if ranges[t][0] <= jt < ranges[t][1]]
            if visitors:
                assert visitors == list(range(visitors[0], visitors[-1] + 1))
                assert visitors[0] == oracle.kv_first(p, 0, jt, tq, tk), \
                    (mode, lq, lkv, wl, wr, jt)
