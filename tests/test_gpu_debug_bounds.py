"""The range-checked build (-DSDPA_DEBUG_BOUNDS): every raw global-memory
index of the kernels (row-wise stores at tile tails, THD offsets, workspace
sections, statistics, partial slots) is checked against its buffer's extent,
and an out-of-range one is reported as SDPA_ERR_BOUNDS and skipped instead of
accessed. (Tensor-map copies are bounded by the hardware.) This stands in for
a memory checker: the parity cases below -- every mask mode, GQA/MQA,
padding, THD slots with gaps and ragged tails, sinks, d = 64/128, the
deterministic modes -- must run clean under it."""
import os
import subprocess
import sys

import pytest
import torch

from sliding_window_attention_sdpa_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_parity_cases_run_clean_in_the_range_checked_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _build.build(debug_bounds=True)
    assert lib.endswith("_dbg.so") and os.path.exists(lib)
    env = dict(os.environ, SWA_SDPA_LIB=lib)
    # the parity tests call sdpa_bwd_check_status after every backward (and
    # the forward's check after every forward): any recorded out-of-range
    # index fails them with SDPA_ERR_BOUNDS
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_parity.py"),
                        os.path.join(ROOT, "tests", "test_gpu_forward.py"),
                        "-k", "small or padding or strided or empty or forward_parity or repeatable_and"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert " passed" in r.stdout
