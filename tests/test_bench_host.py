"""Host-side logic of bench.py, on CPU: the closed-form attended-pair count
(checked against the oracle's mask predicate by brute force), and the
multi-rank timing reduction with two gloo ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle


@pytest.mark.parametrize("mask,sq,skv,w", [
    ("tl", 40, 40, 7), ("tl", 40, 40, -1), ("tl", 33, 50, 0), ("br", 20, 45, 9),
    ("br", 45, 20, 5), ("none", 37, 37, 6), ("none", 30, 30, -1)])
def test_attended_pairs_closed_form(mask, sq, skv, w):
    mode = {"tl": oracle.MASK_TOP_LEFT, "br": oracle.MASK_BOTTOM_RIGHT, "none": oracle.MASK_NONE}
    p = oracle.Problem(b=1, h_q=1, h_kv=1, s_q=sq, s_kv=skv, d=1, scale=1.0, mask_mode=mode[mask],
                       window_left=w)
    assert bench.attended_pairs(sq, skv, mask, w) == oracle.attended_pairs(p)


def test_headline_flops():
    # b2 h16 d64 W128 S8192: 1,048,512 attended pairs per head (21.47 GFLOP)
    assert bench.attended_pairs(8192, 8192, "tl", 128) == 1048512


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    step_ms = [2.0, 3.0][rank]
    e2e_ms = [7.0, 5.0][rank]
    vals = bench.max_over_ranks([step_ms, e2e_ms], dist, torch.device("cpu"))
    value, t = bench.aggregate([vals[0]], [1e12 * world])
    out[rank] = (vals[0], vals[1], value)
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        step, e2e, value = res[rank]
        assert step == 3.0 and e2e == 7.0
        # 2 ranks x 1 TFLOP over the slowest rank's 3 ms
        assert abs(value - 2.0 / 3e-3) < 1e-9


def test_other_workloads_are_known_shapes():
    """Every shape timed after the default workload is one of the benchmark
    set's workloads, none twice, and the default appears only in its
    deterministic mode (its non-deterministic figures are the line's own)."""
    names = [(n, det) for n, det in bench.OTHER_WORKLOADS]
    assert len(set(names)) == len(names)
    for n, det in names:
        assert n in bench.WORKLOADS or n in bench.THD_WORKLOADS
        assert n != bench.DEFAULT or det
        # spec() resolves each (THD lengths included) without a device
        sp = bench.spec(n)
        assert bench.workload_flops(sp) > 0
