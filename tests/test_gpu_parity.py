"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on seeded
inputs: element by element at sizes the oracle finishes in seconds (several
tiles, ragged tails), and on sampled (batch, kv-head) units at the full sizes
of the benchmark workloads. Covers every mask mode, window edge cases, GQA/MQA,
BSHD padding, THD packing with gaps and empty sequences, sinks, f16/bf16,
d = 64/128 and the deterministic relay (bitwise repeatable)."""
import math

import numpy as np
import pytest
import torch

from swa_cases import Case, build, check_all, compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sliding_window_attention_sdpa_gb300 as swa
    swa.load()


SMALL = [
    Case("tiny_b1_h2_d64_s256_tl_w32", 1, 2, 2, 256, 256, 64, "tl", 32),
    Case("tiny_b1_h2_d64_s256_tl_w32_det", 1, 2, 2, 256, 256, 64, "tl", 32, det=True),
    Case("tl_w128_ragged_s700", 2, 4, 4, 700, 700, 64, "tl", 128, seed=1),
    Case("tl_no_window_s300", 1, 2, 2, 300, 300, 64, "tl", -1, seed=2),
    Case("tl_w0_s200", 1, 2, 2, 200, 200, 64, "tl", 0, seed=3),
    Case("tl_w1_s200_f16", 1, 2, 2, 200, 200, 64, "tl", 1, dtype="f16", seed=4),
    Case("br_w96_gqa8x2_d128_s1000", 2, 8, 2, 1000, 1000, 128, "br", 96, seed=5),
    Case("br_w96_gqa8x2_d128_s1000_f16", 2, 8, 2, 1000, 1000, 128, "br", 96, dtype="f16", seed=6),
    Case("br_nonsquare_q128_kv1100_w800", 2, 8, 2, 128, 1100, 64, "br", 800, seed=7),
    Case("none_w200_s600", 1, 4, 4, 600, 600, 64, "none", 200, seed=8),
    Case("none_w100_r30_s500_d128", 1, 2, 2, 500, 500, 128, "none", 100, 30, seed=9),
    Case("tl_w50_r5_s400", 1, 2, 2, 400, 400, 64, "tl", 50, 5, seed=10),
    Case("mqa_h4x1_tl_w64_s500", 2, 4, 1, 500, 500, 64, "tl", 64, seed=11),
    Case("pad_br_w64_sink_gqa4x2", 2, 4, 2, 517, 517, 64, "br", 64, lens_q=[300, 517],
         lens_kv=[450, 200], sink=True, seed=12),
    Case("thd_gqa8x2_f16_tl_w128_sink_det", 0, 8, 2, 0, 0, 64, "tl", 128, dtype="f16",
         layout="thd", thd_lens=[130, 1, 0, 700, 257], slot_align=128, sink=True, det=True,
         seed=13),
    Case("thd_d128_none_w300", 0, 4, 4, 0, 0, 128, "none", 300, layout="thd",
         thd_lens=[390, 64, 1000], slot_align=8, seed=14),
    Case("br_q_longer_than_kv_lens", 2, 2, 2, 400, 400, 64, "br", 40, lens_q=[400, 300],
         lens_kv=[150, 400], seed=15),
    # bottom-right with more queries than keys and no length arrays: the first
    # s_q - s_kv rows reach no key (their LSE is -inf)
    Case("br_q_longer_than_kv_bshd_gqa4x2", 2, 4, 2, 700, 300, 64, "br", 100, seed=19),
    Case("br_causal_q_longer_than_kv_bshd_d128", 1, 2, 2, 520, 130, 128, "br", -1, seed=20),
    # window-only with more queries than keys: rows past Lkv + W reach no key
    Case("none_w50_q600_kv300", 1, 2, 2, 600, 300, 64, "none", 50, seed=16),
    # many visitors per q-tile (unordered atomics path) with GQA and a sink
    Case("tl_w700_gqa4x2_sink_s900", 1, 4, 2, 900, 900, 64, "tl", 700, sink=True, seed=17),
    Case("tl_w700_gqa4x2_sink_s900_det", 1, 4, 2, 900, 900, 64, "tl", 700, sink=True, det=True,
         seed=17),
    Case("none_w300_d128_f16", 1, 2, 2, 700, 700, 128, "none", 300, dtype="f16", seed=18),
    # deterministic with three or more visitors: per-visitor dQ slots, at d = 128
    # and with THD tiles that end inside a slot
    Case("br_w300_gqa4x2_d128_det_slots", 1, 4, 2, 700, 700, 128, "br", 300, det=True, seed=24),
    Case("thd_none_w300_det_slots", 0, 4, 2, 0, 0, 64, "none", 300, layout="thd",
         thd_lens=[390, 64, 1000], slot_align=8, det=True, seed=23),
    Case("br_nonsquare_q128_kv1100_w800_det_slots", 2, 8, 2, 128, 1100, 64, "br", 800, det=True,
         seed=25),
    # strip mode (at most two visitors per q-tile) with THD tiles that end past
    # their slot (row-wise dQ paths): GQA pairs through the accumulator rows, and
    # 40 one-head sequences over more items than SMs (pairs inside a CTA's run
    # adding in tensor memory, pairs split between CTAs)
    Case("thd_strip_gqa4x2_w100_rowwise", 0, 4, 2, 0, 0, 64, "tl", 100, layout="thd",
         thd_lens=[390, 64, 1000, 129], slot_align=8, seed=26),
    Case("thd_strip_mha_40seq_w128_rowwise_det", 0, 1, 1, 0, 0, 64, "tl", 128, layout="thd",
         thd_lens=[300 + (37 * i) % 300 for i in range(40)], slot_align=8, det=True, seed=27),
    # strip mode with 16 kv-heads: pairs of kv-heads share 19 runs, so runs
    # cross from one kv-head's items into the next (MHA pairs in tensor
    # memory, and GQA pairs through the accumulator rows)
    Case("strip_headpair_b1_h16_s2560_w128_det", 1, 16, 16, 2560, 2560, 64, "tl", 128, det=True, seed=28),
    Case("strip_headpair_gqa32x16_s1280_w128", 1, 32, 16, 1280, 1280, 64, "tl", 128, seed=29),
    # strip mode at d = 128, where dQ shares its tensor-memory columns with
    # S^T: every pair goes through the accumulator rows (one head per kv-head,
    # deterministic; THD tiles that end past their slot, and 40 one-head
    # sequences whose pairs are split between CTAs)
    Case("strip_d128_mha_b2_h4_s1300_w128_det", 2, 4, 4, 1300, 1300, 128, "tl", 128, det=True, seed=30),
    Case("thd_strip_d128_gqa4x2_w100_rowwise", 0, 4, 2, 0, 0, 128, "tl", 100, layout="thd",
         thd_lens=[390, 64, 1000, 129], slot_align=8, seed=31),
    Case("thd_strip_d128_mha_40seq_w128_rowwise_det", 0, 1, 1, 0, 0, 128, "tl", 128, layout="thd",
         thd_lens=[300 + (37 * i) % 300 for i in range(40)], slot_align=8, det=True, seed=32),
    # strip runs split by kv-tiles that hold keys, with empty sequences first
    # and in between, and more runs (76 per kv-head) than such kv-tiles (18)
    Case("thd_strip_runs_by_work_leading_empty_det", 0, 4, 2, 0, 0, 64, "tl", 128, layout="thd",
         thd_lens=[0, 0, 700, 0, 64, 1300, 0], slot_align=8, det=True, seed=33),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c.name)
def test_small_parity(case):
    bt = build(case)
    out = run_gpu(bt)
    check_all(bt, out)


def test_deterministic_is_bitwise_repeatable_and_matches_nondet():
    case = Case("det_tl_w128_s1000_gqa", 2, 8, 4, 1000, 1000, 64, "tl", 128, sink=True,
                det=True, seed=20)
    bt = build(case)
    runs = [run_gpu(bt) for _ in range(3)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    check_all(bt, runs[0])
    nd = run_gpu(bt, deterministic=False)
    for name, a, b in zip(("dq", "dk", "dv", "dsink"), runs[0], nd):
        compare(name, a, b.double().cpu().numpy(), "bf16")


def test_deterministic_slots_and_relay():
    """Deterministic mode with three or more visitors per q-tile: mode 1 keeps
    one fp32 partial per visitor and the convert kernel sums them in visitor
    order; mode 2 passes the tile along the relay. Both match the oracle and
    are bitwise repeatable; they add the same partials in the same order, up
    to the relay's fused last add (a last-bit difference before rounding)."""
    case = Case("det_none_w300_r100_gqa4x2_sink", 2, 4, 2, 900, 900, 64, "none", 300, 100,
                sink=True, det=True, seed=22)
    bt = build(case)
    slots = [run_gpu(bt, deterministic=1) for _ in range(2)]
    relay = [run_gpu(bt, deterministic=2) for _ in range(2)]
    for runs in (slots, relay):
        for a, b in zip(runs[0], runs[1]):
            assert torch.equal(a, b)
        check_all(bt, runs[0])
    for name, a, b in zip(("dq", "dk", "dv", "dsink"), slots[0], relay[0]):
        compare(name, a, b.double().cpu().numpy(), "bf16")
    # dK, dV and dSink do not depend on the dQ scheme
    for a, b in zip(slots[0][1:], relay[0][1:]):
        assert torch.equal(a, b)


def test_padding_values_never_leak():
    """NaN in every padded row of Q, K, V, O, dO and LSE: results in the valid
    region are unchanged and padded rows get zero gradients."""
    case = Case("pad_nan", 2, 4, 4, 300, 300, 64, "br", 50, lens_q=[200, 300],
                lens_kv=[260, 120], seed=21)
    bt = build(case)
    d = bt.dev
    for bi, (lq, lk) in enumerate(zip(case.lens_q, case.lens_kv)):
        for name in ("q", "o", "do"):
            d[name][bi, lq:] = float("nan")
        d["lse"][bi, :, lq:] = float("nan")
        for name in ("k", "v"):
            d[name][bi, lk:] = float("nan")
    dq, dk, dv, _ = run_gpu(bt)
    check_all(bt, (dq, dk, dv, None))
    for bi, (lq, lk) in enumerate(zip(case.lens_q, case.lens_kv)):
        assert not dq[bi, lq:].any() and not dk[bi, lk:].any() and not dv[bi, lk:].any()


def test_strided_inputs():
    """Q, K, V sliced out of one packed [b, s, 3, h, d] tensor (non-contiguous)."""
    case = Case("strided", 1, 4, 4, 333, 333, 64, "tl", 70, seed=22)
    bt = build(case)
    d = bt.dev
    packed = torch.stack([d["q"], d["k"], d["v"]], dim=2)  # [b, s, 3, h, d]
    q, k, v = packed[:, :, 0], packed[:, :, 1], packed[:, :, 2]
    assert not q.is_contiguous()
    import sliding_window_attention_sdpa_gb300 as swa
    out = swa.backward(q, k, v, d["o"], d["do"], d["lse"], check_status=True, **bt.kwargs)
    check_all(bt, out)


def test_empty_problem():
    """A batch whose sequences are all empty runs and writes nothing."""
    case = Case("thd_empty", 0, 2, 2, 0, 0, 64, "tl", 16, layout="thd", thd_lens=[0, 0],
                slot_align=8, seed=23)
    bt = build(case)
    out = run_gpu(bt)
    assert out[0].numel() == 0


# ---- full-size workloads of the benchmark, sampled units

FULL = [
    (Case("gptoss_b2_h16_d64_w128_s8192", 2, 16, 16, 8192, 8192, 64, "tl", 128, seed=1001,
          gen_device="cuda"), [(0, 3), (1, 15)]),
    (Case("gptoss_b2_h16_d64_w128_s8192_det", 2, 16, 16, 8192, 8192, 64, "tl", 128, det=True,
          seed=1001, gen_device="cuda"), [(1, 0)]),
    (Case("gqa_b12_h48x6_d128_s16484_br_w96", 12, 48, 6, 16484, 16484, 128, "br", 96,
          seed=1002, gen_device="cuda"), [(11, 5)]),
    (Case("nonsquare_b12_h40x8_d64_q128_kv8960_br_w8000", 12, 40, 8, 128, 8960, 64, "br", 8000,
          seed=1003, gen_device="cuda"), [(0, 0), (7, 3)]),
    (Case("winonly_b4_h16_d64_s4096_w512", 4, 16, 16, 4096, 4096, 64, "none", 512, seed=1004,
          gen_device="cuda"), [(2, 9)]),
    (Case("gqa_b24_h28x4_d128_s128_br_w8000_f16", 24, 28, 4, 128, 128, 128, "br", 8000,
          dtype="f16", seed=1006, gen_device="cuda"), [(bi, g) for bi in range(24) for g in range(4)]),
    # the gpt_oss shape at the other lengths the pages sweep (S = 2k, 32k), and
    # the b12 h48/6 d128 shape in f16
    (Case("gptoss_b2_h16_d64_w128_s2048", 2, 16, 16, 2048, 2048, 64, "tl", 128, seed=1007,
          gen_device="cuda"), [(0, 5), (1, 11)]),
    (Case("gptoss_b2_h16_d64_w128_s32768", 2, 16, 16, 32768, 32768, 64, "tl", 128, seed=1008,
          gen_device="cuda"), [(1, 7)]),
    (Case("gqa_b12_h48x6_d128_s16484_br_w96_f16", 12, 48, 6, 16484, 16484, 128, "br", 96,
          dtype="f16", seed=1009, gen_device="cuda"), [(3, 2)]),
]


@pytest.mark.parametrize("case,units", FULL, ids=lambda x: x.name if isinstance(x, Case) else "")
def test_full_size_sampled(case, units):
    bt = build(case, units=units)
    out = run_gpu(bt)
    check_all(bt, out)
    for t in out[:3]:
        assert torch.isfinite(t).all()
    del bt, out
    torch.cuda.empty_cache()


def test_thd_varlen_sinks_det_full_size():
    from sliding_window_attention_sdpa_gb300 import inputs
    lens = inputs.thd_lengths(16, 128, 8192, seed=1005).tolist()
    case = Case("thd16_h64x8_d64_f16_tl_w128_sink_det", 0, 64, 8, 0, 0, 64, "tl", 128,
                dtype="f16", layout="thd", thd_lens=lens, slot_align=128, sink=True, det=True,
                seed=1005, gen_device="cuda")
    units = [(bi, g) for bi in range(16) for g in (2,)]
    bt = build(case, units=units)
    out = run_gpu(bt)
    check_all(bt, out)


def _three_runs_bitwise(bt):
    runs = [run_gpu(bt) for _ in range(3)]
    for r in runs[1:]:
        for name, a, b in zip(("dq", "dk", "dv", "dsink"), runs[0], r):
            if a is not None:
                assert torch.equal(a, b), f"{bt.case.name}: {name} differs between runs"
    return runs[0]


def test_full_size_deterministic_is_bitwise_repeatable():
    """Deterministic mode at the gpt_oss headline size (b2 h16 d64 S8192 W128):
    three backward passes give the same bits (cuDNN-frontend PR #866,
    "Tests": bitwise repeatable across three passes), and a sampled unit
    matches the oracle."""
    case = Case("gptoss_b2_h16_d64_w128_s8192_det3", 2, 16, 16, 8192, 8192, 64, "tl", 128,
                det=True, seed=1010, gen_device="cuda")
    bt = build(case, units=[(0, 9)])
    out = _three_runs_bitwise(bt)
    check_all(bt, out)
    del bt, out
    torch.cuda.empty_cache()


def test_thd_varlen_sinks_det_full_size_bitwise_repeatable():
    """The packed variable-length workload (16 sequences of U[128, 8192] tokens,
    h 64/8, f16, sinks, deterministic): three passes give the same bits,
    dSink included."""
    from sliding_window_attention_sdpa_gb300 import inputs
    lens = inputs.thd_lengths(16, 128, 8192, seed=1005).tolist()
    case = Case("thd16_h64x8_d64_f16_tl_w128_sink_det3", 0, 64, 8, 0, 0, 64, "tl", 128,
                dtype="f16", layout="thd", thd_lens=lens, slot_align=128, sink=True, det=True,
                seed=1011, gen_device="cuda")
    bt = build(case, units=[(bi, 5) for bi in range(16)])
    out = _three_runs_bitwise(bt)
    check_all(bt, out)
    del bt, out
    torch.cuda.empty_cache()


def test_full_size_d128_deterministic_is_bitwise_repeatable():
    """Deterministic mode at b12 h48/6 d128 S16484 bottom-right W96 (strip
    mode at d = 128: pairs through the accumulator rows, the partial loaded by
    TMA): three passes give the same bits, and a sampled unit matches the
    oracle."""
    case = Case("gqa_b12_h48x6_d128_s16484_br_w96_det3", 12, 48, 6, 16484, 16484, 128, "br", 96,
                det=True, seed=1012, gen_device="cuda")
    bt = build(case, units=[(5, 4)])
    out = _three_runs_bitwise(bt)
    check_all(bt, out)
    del bt, out
    torch.cuda.empty_cache()
