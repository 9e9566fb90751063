"""Bounded device waits: a wait that runs out is reported, not hung on.

Every wait inside the backward kernels has a time limit. These tests use the
library's test hook to shorten the limit to a few milliseconds and to make one
kind of wait unreachable (a counter value or flag that no visitor ever writes):
  - the dQ relay of deterministic mode (cuDNN-frontend PR #866: a wrong first
    visitor "would hang the relay"; here each later turn waits for a turn that
    never comes);
  - the pair protocol of the strip-mode kernel, where the second visitor of a
    q-tile split between two CTAs waits for the first one's partial.
The backward must then report SDPA_ERR_TIMEOUT through sdpa_bwd_check_status
(naming the wait), leave the device usable, and the next call without the
hook must match the oracle."""
import pytest
import torch

import sliding_window_attention_sdpa_gb300 as swa
from swa_cases import Case, build, check_all, run_gpu


def test_hook_rejects_unknown_flags():
    swa._build.build()
    assert swa.sdpa_bwd_test_hook(0, 4) == swa.SDPA_ERR_INVALID_ARG
    assert "flags" in swa.last_error()
    assert swa.sdpa_bwd_test_hook(0, 0) == swa.SDPA_OK


def _times_out_then_recovers(case, flags, words, **over):
    bt = build(case)
    assert swa.sdpa_bwd_test_hook(2_000_000, flags) == swa.SDPA_OK
    try:
        with pytest.raises(swa.SdpaError) as err:
            run_gpu(bt, **over)
    finally:
        swa.sdpa_bwd_test_hook(0, 0)
    assert err.value.code == swa.SDPA_ERR_TIMEOUT, str(err.value)
    assert words in str(err.value), str(err.value)
    # the context is still usable and the same call now gives the oracle's gradients
    out = run_gpu(bt, **over)
    check_all(bt, out)


@pytest.mark.gpu
def test_relay_wait_runs_out_and_is_reported():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    swa.load()
    # W = 200: up to three kv-tiles visit a q-tile; deterministic mode 2 passes
    # every shared q-tile along the relay
    case = Case("relay_timeout_w200", 1, 2, 2, 700, 700, 64, "tl", 200, det=True, seed=50)
    _times_out_then_recovers(case, 1, "relay turn", deterministic=2)


@pytest.mark.gpu
def test_split_pair_wait_runs_out_and_is_reported():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    swa.load()
    # W = 128 (strip mode), one head: 16 kv-tiles over 16 CTAs, so every q-tile
    # with two visitors is split between two CTAs
    case = Case("pair_timeout_w128", 1, 1, 1, 2048, 2048, 64, "tl", 128, seed=51)
    _times_out_then_recovers(case, 2, "split between two CTAs")
