"""Benchmark of the GB300 sliding-window SDPA backward.

Default workload: gpt_oss-style sliding-window attention backward, b=2, h=16,
d=64, S=8192, top-left causal with a 128-key left window, bf16, non-deterministic
dQ (the configuration the cuDNN-frontend pages time on A100 at 0.980 ms).

A step is one whole backward: preprocess, main, dq_convert, gqa_reduce (a
no-op for MHA) -- every kernel of the path. The L2 cache is flushed between
timed steps, outside the per-step CUDA events: a 512 MB write, then a 512 MB
read of another buffer, so that none of the step's data is cached and no
dirty line of the flush is left for the step's first kernel to write back
(the cold, clean state in which ncu times kernels).

  value      attended TFLOP/s (10*d FLOPs per attended (q, k) pair per head)
             with inputs resident in HBM, summed over ranks / max-over-ranks time
  e2e        the same metric through the public API from pinned host buffers,
             host->device copies of Q, K, V, O, dO, LSE and the device->host
             read of dQ, dK, dV inside every timed step (consecutive steps'
             copies and compute overlap on three streams); link_gbs holds the
             same copies timed alone, one direction at a time
  roofline   the main kernel: algorithmic bytes per launch / its mean duration
             (CUDA events on the launching stream) against measured HBM peak
  cpu_baseline  the fp64 CPU oracle on the same workload (host cores)
  other_workloads  (one GPU, default workload) the benchmark set's other
             shapes, each timed the same way after the headline's figures:
             whole step and main kernel, CUDA events, L2 flushed

--impl reference times that oracle as the reference arm (no GPU work).
Multi-GPU (torchrun): every rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from sliding_window_attention_sdpa_gb300 import inputs  # noqa: E402

WORKLOADS = {
    # name: (b, h_q, h_kv, s_q, s_kv, d, mask, window_left, dtype)
    "tiny_b1_h2_d64_s256_tl_w32": (1, 2, 2, 256, 256, 64, "tl", 32, "bf16"),
    "gptoss_b2_h16_d64_w128_s2048": (2, 16, 16, 2048, 2048, 64, "tl", 128, "bf16"),
    "gptoss_b2_h16_d64_w128_s4096": (2, 16, 16, 4096, 4096, 64, "tl", 128, "bf16"),
    "gptoss_b2_h16_d64_w128_s8192": (2, 16, 16, 8192, 8192, 64, "tl", 128, "bf16"),
    "gptoss_b2_h16_d64_w128_s32768": (2, 16, 16, 32768, 32768, 64, "tl", 128, "bf16"),
    "gqa_b12_h48x6_d128_s16484_br_w96": (12, 48, 6, 16484, 16484, 128, "br", 96, "bf16"),
    "gqa_b24_h28x4_d128_s128_br_w8000": (24, 28, 4, 128, 128, 128, "br", 8000, "f16"),
    # one sequence of the shape above: small enough for a full ncu capture of
    # the d = 128 main kernel (~1.3 GB on the device)
    "gqa_b1_h48x6_d128_s16484_br_w96": (1, 48, 6, 16484, 16484, 128, "br", 96, "bf16"),
    "nonsquare_b12_h40x8_d64_q128_kv8960_br_w8000": (12, 40, 8, 128, 8960, 64, "br", 8000, "bf16"),
    "winonly_b4_h16_d64_s4096_w512": (4, 16, 16, 4096, 4096, 64, "none", 512, "bf16"),
}
# Packed variable-length (THD) workloads: n sequences with lengths drawn
# uniformly from [lo, hi], each in a slot padded to a multiple of `align`
# tokens (the gap tokens hold N(0, 1) values, never read into a result).
THD_WORKLOADS = {
    "thd16_h64x8_d64_f16_w128_sink_det": dict(n=16, lo=128, hi=8192, h_q=64, h_kv=8, d=64, mask="tl",
                                             w=128, dtype="f16", sink=True, det=True, seed=1005, align=128),
}
DEFAULT = "gptoss_b2_h16_d64_w128_s8192"
# The benchmark set's other shapes (workload, deterministic), timed after the
# default workload's figures by a one-GPU run of the default workload.
OTHER_WORKLOADS = (
    ("gptoss_b2_h16_d64_w128_s8192", True),
    ("gptoss_b2_h16_d64_w128_s2048", False),
    ("gptoss_b2_h16_d64_w128_s4096", False),
    ("gptoss_b2_h16_d64_w128_s32768", False),
    ("gqa_b12_h48x6_d128_s16484_br_w96", False),
    ("gqa_b12_h48x6_d128_s16484_br_w96", True),
    ("gqa_b24_h28x4_d128_s128_br_w8000", False),
    ("nonsquare_b12_h40x8_d64_q128_kv8960_br_w8000", False),
    ("nonsquare_b12_h40x8_d64_q128_kv8960_br_w8000", True),
    ("winonly_b4_h16_d64_s4096_w512", False),
    ("winonly_b4_h16_d64_s4096_w512", True),
    ("thd16_h64x8_d64_f16_w128_sink_det", True),
)
MODE = {"none": 0, "tl": 1, "br": 2}
L2_FLUSH_BYTES = 512 << 20


class L2Flush:
    """Evicts everything from the 129 MB L2: writes one buffer larger than it,
    then reads another (the read evicts the written lines, which are written
    back here rather than inside the next timed region)."""

    def __init__(self, device):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.fill_(1.0)
        self.r.sum()


def attended_pairs(s_q: int, s_kv: int, mask: str, w: int) -> int:
    """Attended (q, k) pairs per head in closed form: each row i reaches keys
    j with anchor - w <= j (left window, if any) and j <= anchor (causal modes)."""
    diag = s_kv - s_q if mask == "br" else 0
    i = np.arange(s_q, dtype=np.int64)
    anchor = i + diag
    hi = np.minimum(anchor, s_kv - 1) if mask in ("tl", "br") else np.full(s_q, s_kv - 1)
    lo = np.maximum(anchor - w, 0) if w >= 0 else np.zeros(s_q, np.int64)
    return int(np.clip(hi - lo + 1, 0, None).sum())


def algorithmic_bytes(rows_q, rows_kv, h_q, h_kv, d):
    """Main kernel, inputs read once and outputs written once: per q-row per
    q-head Q, dO (2*2d B), LSE, D (8 B) and the fp32 dQ accumulation (4d B);
    per kv-row per kv-head K, V (2*2d B) and dK, dV (2*2d B; the GQA group sum
    is formed in tensor memory, so dK, dV are written once per kv-head)."""
    return rows_q * h_q * (2 * 2 * d + 8 + 4 * d) + rows_kv * h_kv * 4 * 2 * d


def spec(name: str) -> dict:
    """Shape of a workload: BSHD (b, s_q, s_kv) or THD (sequence lengths and
    slot offsets), heads, head dim, mask, window, dtype, sink, deterministic."""
    if name in THD_WORKLOADS:
        w = dict(THD_WORKLOADS[name])
        lens = inputs.thd_lengths(w["n"], w["lo"], w["hi"], seed=w["seed"])
        offs = inputs.thd_offsets(lens, w["align"])
        slot = int(np.diff(offs).max())
        w.update(layout="thd", b=w["n"], lens=lens, offs=offs, total=int(offs[-1]), s_q=slot, s_kv=slot)
        return w
    b, hq, hkv, sq, skv, d, mask, wl, dt = WORKLOADS[name]
    return dict(layout="bshd", b=b, h_q=hq, h_kv=hkv, s_q=sq, s_kv=skv, d=d, mask=mask, w=wl, dtype=dt,
                sink=False, det=False, lens=None, offs=None, total=None, seed=1002)


def workload_flops(sp: dict) -> int:
    """10 d FLOPs per attended (q, k) pair and q-head."""
    if sp["layout"] == "thd":
        pairs = sum(attended_pairs(int(L), int(L), sp["mask"], sp["w"]) for L in sp["lens"])
        return 10 * sp["d"] * pairs * sp["h_q"]
    return 10 * sp["d"] * attended_pairs(sp["s_q"], sp["s_kv"], sp["mask"], sp["w"]) * sp["b"] * sp["h_q"]


def workload_rows(sp: dict):
    """Token rows that carry data: (q rows, kv rows)."""
    if sp["layout"] == "thd":
        n = int(np.sum(sp["lens"]))
        return n, n
    return sp["b"] * sp["s_q"], sp["b"] * sp["s_kv"]


class Problem:
    """Device tensors, outputs, workspace and C-ABI params of one workload."""

    def __init__(self, name: str, device, seed: int, deterministic: bool = False):
        import sliding_window_attention_sdpa_gb300 as swa
        self.swa = swa
        sp = self.sp = spec(name)
        b, hq, hkv, sq, skv, d = sp["b"], sp["h_q"], sp["h_kv"], sp["s_q"], sp["s_kv"], sp["d"]
        mask, w, dt = sp["mask"], sp["w"], sp["dtype"]
        self.name, self.b, self.h_q, self.h_kv, self.s_q, self.s_kv, self.d = name, b, hq, hkv, sq, skv, d
        self.mask, self.w, self.dtype = mask, w, dt
        self.deterministic = bool(deterministic or sp["det"])
        self.scale = 1.0 / math.sqrt(d)
        thd = sp["layout"] == "thd"
        if thd:
            seed = sp["seed"]
            qs, kvs = (sp["total"], hq, d), (sp["total"], hkv, d)
            lse_shape = (hq, sp["total"])
        else:
            qs, kvs = (b, sq, hq, d), (b, skv, hkv, d)
            lse_shape = (b, hq, sq)
        t = inputs.make_tensors(qs, kvs, hq, dt, seed, sp["sink"], device=device)
        self.q, self.k, self.v, self.do, self.sink = t.q, t.k, t.v, t.do, t.sink
        # O and LSE with the magnitudes of a real forward over ~(w+1) keys of
        # N(0,1) logits: O ~ N(0, 1/n), LSE = log(n) + 1/2.
        n = (w + 1) if w >= 0 else skv
        n = min(n, skv)
        self.o = (inputs.randn(qs, seed * 16 + 6, torch.float32, device) / math.sqrt(n)).to(inputs.DTYPES[dt])
        self.lse = torch.full(lse_shape, math.log(n) + 0.5, dtype=torch.float32, device=device)
        self.dq = torch.empty_like(self.q)
        self.dk = torch.empty_like(self.k)
        self.dv = torch.empty_like(self.v)
        self.dsink = torch.empty(hq, dtype=torch.float32, device=device) if sp["sink"] else None
        # keyword arguments of the binding's backward()/make_params() besides the tensors
        self.kw = dict(scale=self.scale, mask_mode=MODE[mask], window_left=w)
        if thd:
            offs = torch.from_numpy(sp["offs"].astype(np.int32)).to(device)
            lens = torch.from_numpy(sp["lens"].astype(np.int32)).to(device)
            self.kw.update(q_offsets=offs, kv_offsets=offs, seq_q_lens=lens, seq_kv_lens=lens,
                           max_seqlen_q=sq, max_seqlen_kv=skv)
        self.params = swa.make_params(self.q, self.k, self.v, self.o, self.do, self.lse, self.dq,
                                      self.dk, self.dv, deterministic=self.deterministic,
                                      sink=self.sink, dsink=self.dsink, **self.kw)
        self.ws = swa.alloc_workspace(self.params, device)
        # the forward on the same inputs (its own outputs)
        self.fo = torch.empty_like(self.q)
        self.flse = torch.empty_like(self.lse)
        self.fparams = swa.make_fwd_params(self.q, self.k, self.v, self.fo, self.flse, sink=self.sink, **self.kw)
        rows_q, rows_kv = workload_rows(sp)
        self.flops = workload_flops(sp)
        self.fwd_flops = self.flops * 4 // 10
        # Q, K, V read once, O and LSE written once
        self.fwd_bytes = rows_q * hq * (2 * 2 * d + 4) + rows_kv * hkv * 2 * 2 * d
        self.main_bytes = algorithmic_bytes(rows_q, rows_kv, hq, hkv, d)

    def step(self, stream: int, ev=None):
        """The whole backward; `ev` = (before_main, after_main) events."""
        swa, p = self.swa, self.params
        ws, nb = self.ws.data_ptr(), self.ws.numel()
        swa._check(swa.sdpa_bwd_preprocess(p, ws, nb, stream), "preprocess")
        if ev is not None:
            ev[0].record()
        swa._check(swa.sdpa_bwd(p, ws, nb, stream), "sdpa_bwd")
        if ev is not None:
            ev[1].record()
        swa._check(swa.sdpa_bwd_dq_convert(p, ws, nb, stream), "dq_convert")
        swa._check(swa.sdpa_bwd_gqa_reduce(p, ws, nb, stream), "gqa_reduce")

    def launches_per_step(self) -> int:
        return self.swa.sdpa_bwd_kernel_launches(self.params)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms while the GPU
    runs the warm-up, the timed steps and the end-to-end leg."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_dir: str | None = None, tag: str = ""):
        import tempfile
        self.gpu = gpu_index
        self.proc = None
        # the raw samples; the JSON line carries their summary
        self.path = os.path.join(log_dir or tempfile.gettempdir(), f"clocks_rank{gpu_index}{tag}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one main-kernel
# launch from an ncu capture (profiles/sdpa_bwd_main_kernel_*.md), valid only
# for the kernel source it was taken on (sha256 of the main kernel's sources,
# first 16 hex digits); any other source reports null.
MAIN_TRAFFIC = {
    "gptoss_b2_h16_d64_w128_s8192": {"kernel": "2b44da694746a8eb", "bytes": 283117056},
}
KERNEL_SOURCES = ("main_kernel.cu", "ptx.cuh", "seq.cuh", "sdpa_internal.h")
# The same for one forward launch (profiles/sdpa_fwd_kernel_*.md).
FWD_TRAFFIC = {
    "gptoss_b2_h16_d64_w128_s8192": {"kernel": "1a167d12b75e8039", "bytes": 114572544},
}
FWD_SOURCES = ("fwd_kernel.cu", "ptx.cuh", "seq.cuh", "sdpa_internal.h")


def main_kernel_digest(sources=KERNEL_SOURCES) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sliding_window_attention_sdpa_gb300", "csrc")
    for f in sources:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(name: str, table=MAIN_TRAFFIC, sources=KERNEL_SOURCES):
    t = table.get(name)
    if t is None or t["kernel"] != main_kernel_digest(sources):
        return None
    return t["bytes"]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            j = json.load(f)
        return j["hbm_gbs"], j["bf16_tflops"], "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def time_device(prob: Problem, steps: int, warmup: int):
    """Per-step device time (ms) of the whole backward and of the main kernel.

    The whole step is timed with events before and after it only; events
    recorded between its kernels cost ~3.5 us a step. The main kernel is
    timed in a second loop of the same steps, with events around it.
    """
    stream = torch.cuda.current_stream()
    sid = stream.cuda_stream
    flush = L2Flush(prob.q.device)
    for _ in range(warmup):
        prob.step(sid)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record()
        prob.step(sid)
        b.record()
    torch.cuda.synchronize()
    total = [a.elapsed_time(b) for a, b in ev]
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e in ev:
        flush()
        prob.step(sid, e)
    torch.cuda.synchronize()
    main = [a.elapsed_time(b) for a, b in ev]
    return total, main


def time_other_workloads(device, steps: int, warmup: int, peak_gbs: float, peak_tf: float):
    """Whole-step and main-kernel device times of OTHER_WORKLOADS, one shape
    at a time (its tensors freed before the next). A shape that fails to run
    is reported with its error instead of stopping the benchmark."""
    out = []
    for name, det in OTHER_WORKLOADS:
        rec = {"workload": name, "deterministic": det}
        try:
            prob = Problem(name, device, seed=1000 + 2, deterministic=det)
            total, main = time_device(prob, steps, warmup)
            status = prob.swa.sdpa_bwd_check_status(prob.ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
            step_ms, main_ms = statistics.median(total), statistics.median(main)
            rec.update(step_ms=step_ms, main_kernel_ms=main_ms,
                       step_tflops=prob.flops / (step_ms * 1e-3) / 1e12,
                       main_kernel_tflops=prob.flops / (main_ms * 1e-3) / 1e12,
                       tensor_peak_frac=prob.flops / (main_ms * 1e-3) / 1e12 / peak_tf,
                       hbm_frac=prob.main_bytes / (main_ms * 1e-3) / 1e9 / peak_gbs,
                       device_status=int(status))
            del prob
        except Exception as e:  # noqa: BLE001 - reported in the line, not fatal
            rec["error"] = f"{type(e).__name__}: {e}"[:300]
        torch.cuda.empty_cache()
        out.append(rec)
    return out


def time_forward(prob: Problem, steps: int, warmup: int):
    """Per-call device time (ms) of the forward, L2 flushed before each call."""
    swa = prob.swa
    sid = torch.cuda.current_stream().cuda_stream
    flush = L2Flush(prob.q.device)
    for _ in range(warmup):
        swa._check(swa.sdpa_fwd(prob.fparams, sid), "sdpa_fwd")
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record()
        swa._check(swa.sdpa_fwd(prob.fparams, sid), "sdpa_fwd")
        b.record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_e2e(prob: Problem, steps: int, warmup: int):
    """Same backward through the public API from pinned host buffers.

    Every step copies its inputs (Q, K, V, O, dO, LSE) host -> device, runs
    `backward()` and copies dQ, dK, dV device -> host, all inside the timed
    region. The three stages of consecutive steps overlap on three streams,
    as a training loop would feed its batches: the copy of step k + 1's inputs
    and the read of step k - 1's results run while step k computes. Device
    input buffers alternate between two sets. Returns (ms per step, host ->
    device bytes per step, device -> host bytes per step, link rates): the
    link rates are the same copies timed alone after the timed region, each
    direction on its own (GB/s), which bound the pipelined step from below.
    """
    import sliding_window_attention_sdpa_gb300 as swa
    names = (prob.q, prob.k, prob.v, prob.o, prob.do, prob.lse) + ((prob.sink,) if prob.sink is not None else ())
    outs = (prob.dq, prob.dk, prob.dv) + ((prob.dsink,) if prob.dsink is not None else ())
    host_in = [t.cpu().pin_memory() for t in names]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    dev_in = [[torch.empty_like(t) for t in names] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    kw = dict(prob.kw, workspace=prob.ws, deterministic=prob.deterministic)
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    for e in done:
        e.record(s_run)

    def one(k):
        buf = k % 2
        s_in.wait_event(done[buf])           # step k - 2 has read this input set
        with torch.cuda.stream(s_in):
            for d, h in zip(dev_in[buf], host_in):
                d.copy_(h, non_blocking=True)
        copied[buf].record(s_in)
        s_run.wait_event(copied[buf])
        with torch.cuda.stream(s_run):
            ins = dev_in[buf]
            res = swa.backward(*ins[:6], sink=ins[6] if len(ins) > 6 else None, **kw)
            res = tuple(x for x in res if x is not None)
        done[buf].record(s_run)
        s_out.wait_event(done[buf])
        with torch.cuda.stream(s_out):
            for h, d in zip(host_out, res):
                d.record_stream(s_out)
                h.copy_(d, non_blocking=True)

    for k in range(warmup):
        one(k)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for k in range(steps):
        one(warmup + k)
    b.record(s_out)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps

    def alone(stream, pairs, nbytes, reps=5):
        out = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            with torch.cuda.stream(stream):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1))
        return nbytes / (sorted(out)[reps // 2] * 1e-3) / 1e9

    link = {"h2d_gbs": alone(s_in, list(zip(dev_in[0], host_in)), h2d),
            "d2h_gbs": alone(s_out, list(zip(host_out, outs)), d2h)}
    return ms, h2d, d2h, link


def cpu_oracle_step(name: str, nthreads: int, units=None):
    """One fp64 oracle backward (window-bounded sweep) of the workload on the
    host cores; returns (seconds, fraction of the workload's FLOPs run).
    `units` limits the run to the first (sequence, kv-head) units."""
    import oracle
    sp = spec(name)
    b, hq, hkv, d = sp["b"], sp["h_q"], sp["h_kv"], sp["d"]
    f64 = lambda x: x.double().numpy()
    n = min((sp["w"] + 1) if sp["w"] >= 0 else sp["s_kv"], sp["s_kv"])
    kw = dict(b=b, h_q=hq, h_kv=hkv, s_q=sp["s_q"], s_kv=sp["s_kv"], d=d, scale=1 / math.sqrt(d),
              mask_mode=MODE[sp["mask"]], window_left=sp["w"], nthreads=nthreads, has_sink=sp["sink"])
    if sp["layout"] == "thd":
        qs, kvs, lse_shape = (sp["total"], hq, d), (sp["total"], hkv, d), (hq, sp["total"])
        kw.update(layout=oracle.THD, seq_q_lens=sp["lens"], seq_kv_lens=sp["lens"],
                  q_offsets=sp["offs"], kv_offsets=sp["offs"])
    else:
        qs, kvs, lse_shape = (b, sp["s_q"], hq, d), (b, sp["s_kv"], hkv, d), (b, hq, sp["s_q"])
    t = inputs.make_tensors(qs, kvs, hq, sp["dtype"], 7, sp["sink"])
    o = (inputs.randn(qs, 7 * 16 + 6) / math.sqrt(n)).to(inputs.DTYPES[sp["dtype"]])
    lse = np.full(lse_shape, math.log(n) + 0.5)
    p = oracle.Problem(**kw)
    frac = 1.0
    if units is not None and units < b * hkv:
        m = np.zeros(b * hkv, np.uint8)
        m[:units] = 1
        p.unit_mask = m
        if sp["layout"] == "thd":
            # units are (sequence, kv-head), sequence-major: FLOPs of the sampled ones
            pairs = [attended_pairs(int(L), int(L), sp["mask"], sp["w"]) for L in sp["lens"]]
            done = sum(pairs[u // hkv] for u in range(units))
            frac = done / (sum(pairs) * hkv)
        else:
            frac = units / (b * hkv)
    args = (f64(t.q), f64(t.k), f64(t.v), f64(o), f64(t.do), lse)
    sink = f64(t.sink) if t.sink is not None else None
    t0 = time.perf_counter()
    oracle.backward(p, *args, sink)
    return time.perf_counter() - t0, frac


def cpu_units_for_budget(name: str, budget_s: float, nthreads: int):
    """Units (sequence, kv-head) that fit about `budget_s` seconds of oracle time."""
    sp = spec(name)
    total = sp["b"] * sp["h_kv"]
    probe = max(1, min(total, nthreads))
    t, frac = cpu_oracle_step(name, nthreads, probe)
    per_unit_wave = t  # one wave of `probe` units in parallel
    waves = max(1, int(budget_s / max(per_unit_wave, 1e-3)))
    return min(total, probe * waves)


# Single-thread oracle figures the CPU baseline reports beside the all-core
# one: the tiny case whole, and the gpt_oss shape at S = 2048 on one
# (batch, head) unit of its 32.
SINGLE_THREAD = {"tiny_b1_h2_d64_s256_tl_w32": None, "gptoss_b2_h16_d64_w128_s2048": 1}


def single_thread_figures():
    out = {}
    for name, units in SINGLE_THREAD.items():
        sec, frac = cpu_oracle_step(name, 1, units)
        flops = workload_flops(spec(name)) * frac
        out[name] = {"value": flops / sec / 1e9, "unit": "GFLOP/s", "cores": 1,
                     "sample": "whole workload" if units is None else f"{units} (batch, kv-head) unit"}
    return out


def reference_arm(args, rank, world):
    """The oracle as the reference arm: K timed steps of the workload's
    backward (bounded sample) on the host cores."""
    if rank != 0:
        return
    name = args.workload
    cores = os.cpu_count() or 1
    units = cpu_units_for_budget(name, 20.0 / max(args.steps + args.warmup, 1), cores)
    for _ in range(args.warmup):
        cpu_oracle_step(name, cores, units)
    times = []
    frac = 1.0
    for _ in range(args.steps):
        t, frac = cpu_oracle_step(name, cores, units)
        times.append(t)
    sp = spec(name)
    flops = workload_flops(sp) * frac
    b, hkv = sp["b"], sp["h_kv"]
    sec = statistics.mean(times)
    val = flops / sec / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3 / frac, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(name),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{units} of {b * hkv} (batch, kv-head) units per step, "
                                   "time scaled to the whole workload"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "SWA bwd attended TFLOP/s (b2 h16 d64 W128 S8k bf16)"


def workload_config(name):
    sp = spec(name)
    c = {"workload": name, "global_batch": sp["b"], "seq_len": sp["s_q"], "seq_len_kv": sp["s_kv"],
         "heads_q": sp["h_q"], "heads_kv": sp["h_kv"], "head_dim": sp["d"],
         "mask": {"tl": "top_left_causal", "br": "bottom_right_causal", "none": "window_only"}[sp["mask"]],
         "window_left": sp["w"], "dtype": sp["dtype"],
         "l2": "flushed between timed steps (512 MB write, then 512 MB read of another buffer)",
         "parallelism": "replicas"}
    if sp["layout"] == "thd":
        c.update(layout="thd", sequences=sp["b"], tokens=int(np.sum(sp["lens"])), slot_tokens=sp["total"],
                 lengths=f"uniform [{THD_WORKLOADS[name]['lo']}, {THD_WORKLOADS[name]['hi']}] (seed "
                         f"{THD_WORKLOADS[name]['seed']}), slots padded to {THD_WORKLOADS[name]['align']}",
                 sinks=sp["sink"])
    return c


def aggregate(per_rank_ms, per_rank_flops):
    """Whole-job throughput: all ranks' FLOPs over the slowest rank's time."""
    t = max(per_rank_ms)
    return sum(per_rank_flops) / (t * 1e-3) / 1e12, t


def max_over_ranks(values, dist, device):
    """Element-wise max of a list of floats over all ranks (identity without
    a process group)."""
    if dist is None:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS) + sorted(THD_WORKLOADS))
    ap.add_argument("--deterministic", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the benchmark set's other shapes after the default workload")
    ap.add_argument("--clock-log-dir", default=None,
                    help="folder for the raw nvidia-smi clock samples (default: the temp folder)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import sliding_window_attention_sdpa_gb300 as swa
    swa.load()

    prob = Problem(args.workload, dev, seed=1000 + 2, deterministic=args.deterministic)
    peak_gbs, peak_tf, peak_kind = measured_peaks()

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local, args.clock_log_dir) as clk:
        total, main_ms = time_device(prob, args.steps, args.warmup)
        torch.cuda.synchronize()
        e2e_ms, h2d, d2h, link = time_e2e(prob, max(3, args.steps), 2)
        fwd_ms = time_forward(prob, args.steps, args.warmup)
    step_ms = sum(total) / len(total)
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    fwd_status = swa.sdpa_fwd_check_status(torch.cuda.current_stream().cuda_stream)
    main_avg = sum(main_ms) / len(main_ms)
    status = swa.sdpa_bwd_check_status(prob.ws.data_ptr(), torch.cuda.current_stream().cuda_stream)

    step_max, e2e_max = max_over_ranks([step_ms, e2e_ms], dist, dev)
    value, _ = aggregate([step_max], [prob.flops * world])
    e2e_val, _ = aggregate([e2e_max], [prob.flops * world])

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    achieved = prob.main_bytes / (main_avg * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": prob.dtype, "data": "synthetic",
        "config": workload_config(args.workload),
        "main_kernel_ms": main_avg,
        "main_kernel_tflops": prob.flops / (main_avg * 1e-3) / 1e12,
        "tensor_peak_frac": prob.flops / (main_avg * 1e-3) / 1e12 / peak_tf,
        "deterministic": prob.deterministic,
        "device_status": int(status),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak_gbs, "unit": "GB/s",
                     "frac": achieved / peak_gbs, "traffic": measured_traffic(args.workload),
                     "kernel": "sdpa_bwd_main_kernel", "peak_kind": peak_kind,
                     "algorithmic_bytes": prob.main_bytes},
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "ms_per_step": e2e_max,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "overlap": "step k+1's host->device copy and step k-1's device->host read run "
                           "during step k (three streams)",
                # the step's copies timed alone, one direction at a time
                "link_gbs": {k: round(v, 1) for k, v in link.items()}},
        "gpu_launches": prob.launches_per_step() * args.steps,
        "clocks": clk.summary(),
        # the forward (O, LSE) on the same workload, timed after the backward's
        # region; 4 d FLOPs per attended pair and head
        "forward": {"ms": fwd_avg, "tflops": prob.fwd_flops / (fwd_avg * 1e-3) / 1e12,
                    "kernel": "sdpa_fwd_kernel", "algorithmic_bytes": prob.fwd_bytes,
                    "hbm_frac": prob.fwd_bytes / (fwd_avg * 1e-3) / 1e9 / peak_gbs,
                    "tensor_peak_frac": prob.fwd_flops / (fwd_avg * 1e-3) / 1e12 / peak_tf,
                    "traffic": measured_traffic(args.workload, FWD_TRAFFIC, FWD_SOURCES),
                    "device_status": int(fwd_status)},
    }
    flops = prob.flops
    if world == 1 and args.workload == DEFAULT and not args.no_other_workloads:
        del prob   # the other shapes get the device memory to themselves
        torch.cuda.empty_cache()
        with ClockSampler(local, args.clock_log_dir, tag="_other") as clk_other:
            others = time_other_workloads(dev, min(args.steps, 10), 3, peak_gbs, peak_tf)
        line["other_workloads"] = {
            "steps": min(args.steps, 10), "warmup": 3, "stat": "median",
            "l2": "flushed between timed steps, as for the default workload",
            "clocks": clk_other.summary(), "results": others}
    if not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        name = args.workload
        units = cpu_units_for_budget(name, 15.0, cores)
        sec, frac = cpu_oracle_step(name, cores, units)
        cpu_val = flops * frac / sec / 1e12
        sp = spec(name)
        line["cpu_baseline"] = {"value": cpu_val, "unit": "TFLOP/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"{units} of {sp['b'] * sp['h_kv']} (sequence, kv-head) units, "
                                          "fp64 window-bounded backward",
                                "single_thread": single_thread_figures()}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
