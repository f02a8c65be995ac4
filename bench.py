"""Benchmark of the relation-aware attention forward hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one forward pass over one batch of the named workload (default: the long
key-only causal case, B=4 H=16 n=4096 d=128 k=64 bf16, the largest configuration): a single
kernel launch through the C ABI. Inputs are seeded and synthetic (workloads.py) and
resident in HBM; to keep L2 from serving them, the timed steps rotate over enough input
sets to exceed 4x L2, and exactly --steps launches are replayed from one CUDA graph (the
short workloads are a few microseconds long, so host launch overhead would otherwise
dominate). The other forward configurations (--also) are timed the same way in the same
run and reported as compact lines under "workloads".

Printed (rank 0, one JSON line): the whole-job TFLOP/s over the timed steps; the per-launch
kernel time measured with CUDA events on the launching stream (mean, p10, p90, and for the
HBM-bound workloads a single launch after an L2 flush) and its roofline fraction;
an end-to-end number through the same C ABI with host (pinned) buffers and the
host<->device copies inside the timed region; the fp64 CPU oracle timed on a bounded
sample of the same workload; SM clocks sampled while the timed region runs.

Under torchrun (N > 1) each rank runs the same per-GPU workload on its own GPU (the path
shards over independent (batch, head) units, so there is no collective on the data path;
only the timing reduction uses the process group): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("fused rel-attn fwd TFLOP/s (bf16) and % of GB300 tensor/HBM roofline vs CPU oracle")
# the largest single-GPU configuration (the compute-bound one); the other forward
# configurations are measured in the same run as compact lines under "workloads"
DEFAULT_WORKLOAD = "long_keyonly"
ALSO_WORKLOADS = "base_encoder,big_decoder,t5_bias"
# fp32 FMA peak of the SIMT units: 152 SMs x 128 lanes x 2 flop x 2.07 GHz (max SM clock)
FP32_SIMT_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------- accounting
def pairs_per_sequence(w, kv_len_b: int) -> int:
    """Unmasked (i, j) pairs of one (b, h)."""
    n = w.n
    kv = n if kv_len_b is None else max(0, min(int(kv_len_b), n))
    if not w.causal:
        return n * kv
    # row i keeps j <= min(i, kv - 1)
    return sum(min(i + 1, kv) for i in range(n))


def algorithmic_flops(w, kv_len) -> float:
    """4*d per unmasked pair (Q.K^T and P.V) + 2*d*n per reachable table row and term.
    Decode step: one query row per (b, h) over its cache_len keys. Gradients: 2.5 times the
    forward's count (Q.K^T, dP = dZ.V^T, dQ, dK, dV against Q.K^T and P.V; the same ratio
    for the table terms)."""
    if w.kind == "bwd":
        return 2.5 * algorithmic_flops(w.replace(kind="shaw"), kv_len)
    if w.kind == "txl":  # (q + u).k_j, (q + v).r_ij and p v_j: 3 x 2 d per unmasked pair
        kvs = [None] * w.B if kv_len is None else [int(x) for x in kv_len]
        return 6.0 * w.d * sum(pairs_per_sequence(w, kvs[b]) for b in range(w.B)) * w.H
    if w.kind == "decode":
        terms = int(w.key_term) + int(w.value_term)
        rows = sum(min(int(x), w.n) for x in kv_len) * w.H
        live = sum(1 for x in kv_len if int(x) > 0) * w.H
        return 4.0 * w.d * rows + 2.0 * w.d * (w.clip_k + 1) * terms * live
    kvs = [None] * w.B if kv_len is None else [int(x) for x in kv_len]
    pairs = sum(pairs_per_sequence(w, kvs[b]) for b in range(w.B)) * w.H
    flops = 4.0 * w.d * pairs
    if w.kind in ("shaw", "labeled"):
        reach = (w.num_labels if w.kind == "labeled" else
                 (w.clip_k + 1) if w.causal else (2 * w.clip_k + 1))
        terms = int(w.key_term) + int(w.value_term)
        flops += 2.0 * w.d * w.n * reach * terms * w.B * w.H
    return flops


def algorithmic_bytes(w, kv_len) -> float:
    """Q and O in full, K and V rows below kv_len, the tables once (bf16 / fp32 elements).
    Decode step: q and out rows, the cached K and V rows below cache_len, table rows 0..k."""
    es = 2 if w.dtype == "bf16" else 4
    if w.kind == "bwd":  # reads q, k, v, dout and the tables; writes fp32 dq, dk, dv, dtables
        Ht = 1 if w.shared_tables else w.H
        tab = Ht * (2 * w.clip_k + 1) * w.d * (int(w.key_term) + int(w.value_term))
        return float(4 * w.B * w.H * w.n * w.d * es + 3 * w.B * w.H * w.n * w.d * 4 +
                     tab * (es + 4))
    if w.kind == "decode":
        rows = sum(min(int(x), w.n) for x in kv_len) * w.H
        Ht = 1 if w.shared_tables else w.H
        tabs = Ht * (w.clip_k + 1) * w.d * (int(w.key_term) + int(w.value_term))
        return float(es * (2 * w.B * w.H * w.d + 2 * rows * w.d + tabs) + 4 * w.B)
    BHnd = w.B * w.H * w.n * w.d
    kvs = [w.n] * w.B if kv_len is None else [min(int(x), w.n) for x in kv_len]
    kv_rows = sum(kvs) * w.H
    byt = es * (2 * BHnd + 2 * kv_rows * w.d)
    Ht = 1 if w.shared_tables else w.H
    if w.kind == "shaw":
        byt += es * Ht * (2 * w.clip_k + 1) * w.d * (int(w.key_term) + int(w.value_term))
    elif w.kind == "t5":
        byt += 4 * w.num_buckets * w.H
    elif w.kind == "alibi":  # the slopes
        byt += 4 * w.H
    elif w.kind == "txl":  # the projected offset encodings and the two bias vectors
        byt += es * Ht * (2 * w.n - 1 + 2) * w.d
    elif w.kind == "labeled":  # the tables and the uint8 label matrices
        byt += es * Ht * w.num_labels * w.d * (int(w.key_term) + int(w.value_term))
        byt += (w.B if w.labels_per_sequence else 1) * w.n * w.n
    else:  # "offset": the clipped per-offset table
        byt += 4 * Ht * (2 * w.clip_k + 1)
    return float(byt)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, \
            "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# the sources each measured kernel is built from (argument structs in relattn_internal.h
# and the host entry points do not change the kernels' code)
KERNEL_SOURCES = {
    "fused": ["device_common.cuh", "relattn_tc_d128.cu", "relattn_tc_d64.cu",
              "relattn_tc_kernel.cuh", "relattn_tc_launch.cuh", "sm103_ptx.cuh"],
    "decode": ["relattn_decode.cu"],
    "bwd": ["relattn_bwd.cu"],
    "bwd_tc": ["relattn_bwd_tc.cu", "relattn_tc_kernel.cuh", "relattn_tc_launch.cuh", "sm103_ptx.cuh"],
    "labeled": ["relattn_labeled_tc.cuh", "relattn_labeled_tc.cu", "relattn_tc_kernel.cuh",
                "sm103_ptx.cuh"],
    "txl": ["relattn_txl.cu"],
    "txl_tc": ["relattn_txl_tc.cu", "relattn_tc_kernel.cuh", "relattn_tc_launch.cuh", "sm103_ptx.cuh"],
    "short": ["relattn_short.cuh", "relattn_short.cu", "relattn_tc_kernel.cuh",
              "relattn_tc_launch.cuh", "sm103_ptx.cuh"],
}


def bwd_on_tensor_cores(w) -> bool:
    """The library routes bf16 gradients with d = 64 / 128 and at most 128 staged table rows
    to its tensor-core kernels (the others run on the SIMT kernels)."""
    rows = w.clip_k + 1 if w.causal else 2 * w.clip_k + 1
    return w.kind == "bwd" and w.dtype == "bf16" and w.d in (64, 128) and rows <= 128


def txl_on_tensor_cores(w) -> bool:
    """bf16 Transformer-XL with d = 64 / 128 runs on the tensor-core kernel."""
    return w.kind == "txl" and w.dtype == "bf16" and w.d in (64, 128)


def simt_roof(w) -> bool:
    """Workloads whose kernels run on the SIMT units (roof: the derived fp32 FMA rate)."""
    return ((w.kind == "txl" and not txl_on_tensor_cores(w)) or
            (w.kind == "bwd" and not bwd_on_tensor_cores(w)) or
            (w.kind == "labeled" and w.dtype != "bf16"))


def kernel_family(w) -> str:
    fam = {"decode": "decode", "bwd": "bwd", "labeled": "labeled", "txl": "txl"}.get(w.kind, "fused")
    if fam == "bwd" and bwd_on_tensor_cores(w):
        fam = "bwd_tc"
    if fam == "txl" and txl_on_tensor_cores(w):
        fam = "txl_tc"
    if fam == "fused" and w.kind == "shaw" and w.dtype == "bf16" and w.d == 64 and w.n <= 256:
        rows = (w.clip_k + 1 if w.causal else 2 * w.clip_k + 1) if (w.key_term or w.value_term) else 1
        if rows <= 64:  # the library routes these to the short-sequence kernel
            fam = "short"
    return fam


def kernel_source_hash(family: str = "fused") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "relative_position_representations_gb300", "csrc")
    for name in KERNEL_SOURCES[family]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, family: str = "fused"):
    """DRAM bytes per launch from the committed ncu summary, if it matches this source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 3 and not line.startswith("#") and parts[0] == workload:
                    if parts[1] == kernel_source_hash(family):
                        return float(parts[2])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU is busy."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        mhz, max_mhz, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if ts < t0 or ts > t1:
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                max_mhz = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": max_mhz, "reasons": sorted(reasons),
                    "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max_mhz,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ----------------------------------------------------------------------- CPU oracle
def workload_by_name(name):
    from relative_position_representations_gb300 import workloads as wl
    if name in wl.DECODE_WORKLOADS:
        return wl.DECODE_WORKLOADS[name]
    if name in wl.BWD_WORKLOADS:
        return wl.BWD_WORKLOADS[name]
    if name in wl.BIAS_WORKLOADS:
        return wl.BIAS_WORKLOADS[name]
    if name in wl.LABELED_WORKLOADS:
        return wl.LABELED_WORKLOADS[name]
    if name in wl.TXL_WORKLOADS:
        return wl.TXL_WORKLOADS[name]
    return wl.WORKLOADS[name]


def draw(w, seed):
    from relative_position_representations_gb300 import workloads as wl
    if w.kind == "decode":
        return wl.draw_decode_inputs(w, seed)
    if w.kind == "bwd":
        return wl.draw_bwd_inputs(w, seed)
    return wl.draw_inputs(w, seed)


def oracle_bwd_batches(w, x, batches):
    """The gradient oracle on the sequences in `batches` (all heads), one at a time."""
    from oracle import backward
    from relative_position_representations_gb300 import workloads as wl
    out = []
    for b in batches:
        sl = lambda t: None if t is None else t[b:b + 1].double().numpy()
        tab = lambda t: None if t is None else t.double().numpy()
        kv = None if x["kv_len"] is None else x["kv_len"][b:b + 1].numpy()
        out.append(backward.relattn_bwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), tab(x["aK"]),
                                        tab(x["aV"]), sl(x["dout"]), w.clip_k, w.causal,
                                        w.softmax_scale, kv_len=kv,
                                        table_head_stride=wl.table_head_stride(w)))
    return out


def oracle_txl_batches(w, x, batches):
    """The Transformer-XL oracle on the sequences in `batches` (all heads), one at a time."""
    import numpy as np
    from oracle import txl
    f = lambda t: t.double().numpy()
    rel, u, vb = f(x["rel"]), f(x["u"]), f(x["vb"])
    if rel.shape[0] == 1 and w.H > 1:
        rel, u, vb = (np.repeat(t, w.H, axis=0) for t in (rel, u, vb))
    out = []
    for b in batches:
        sl = lambda t: t[b:b + 1].double().numpy()
        kv = None if x["kv_len"] is None else x["kv_len"][b:b + 1].numpy()
        out.append(txl.txl_fwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), rel, u, vb, w.causal,
                               w.softmax_scale, kv_len=kv))
    return out


def key_lengths(w, x):
    key = "cache_len" if w.kind == "decode" else "kv_len"
    return None if x.get(key) is None else x[key].tolist()


def oracle_decode_rows(w, x, batches, nthreads):
    """The oracle for the decode step of the sequences in `batches` (all heads): row
    t = cache_len - 1 of the causal forward, one sequence at a time."""
    import numpy as np
    import oracle
    from relative_position_representations_gb300 import workloads as wl
    out = []
    for b in batches:
        L = min(int(x["cache_len"][b]), w.n)
        if L == 0:
            continue
        qf = np.zeros((1, w.H, L, w.d))
        qf[0, :, L - 1] = x["q"][b].double().numpy()
        sl = lambda t: None if t is None else t[b:b + 1, :, :L].double().numpy()
        tab = lambda t: None if t is None else t.double().numpy()
        rows = [h * L + L - 1 for h in range(w.H)]
        out.append(oracle.relattn_fwd(qf, sl(x["k"]), sl(x["v"]), tab(x["aK"]), tab(x["aV"]),
                                      w.clip_k, True, w.softmax_scale,
                                      table_head_stride=wl.table_head_stride(w), rows=rows,
                                      nthreads=nthreads))
    return out


def host_arrays(x):
    """The inputs as numpy arrays (floating point in fp64), converted once."""
    import numpy as np
    import torch
    out = {}
    for k, t in x.items():
        if isinstance(t, torch.Tensor):
            t = t.double().numpy() if t.is_floating_point() else t.numpy()
            t = np.ascontiguousarray(t)
        out[k] = t
    return out


def oracle_rows_call(w, x, rows, nthreads):
    import numpy as np
    import oracle

    def np_(t):
        if t is None or isinstance(t, np.ndarray):
            return t
        return t.float().numpy()

    def raw(t):  # integer / fp32 side inputs
        return t if isinstance(t, np.ndarray) else t.numpy()

    if w.kind == "decode":  # rows are sequence indices
        return oracle_decode_rows(w, x, rows, nthreads)
    if w.kind == "bwd":  # rows are sequence indices
        return oracle_bwd_batches(w, x, rows)
    if w.kind == "txl":  # rows are sequence indices
        return oracle_txl_batches(w, x, rows)

    kv = None if x.get("kv_len") is None else raw(x["kv_len"])
    if w.kind == "t5":
        return oracle.t5bias_fwd(np_(x["q"]), np_(x["k"]), np_(x["v"]), raw(x["bias"]),
                                 w.num_buckets, w.max_distance, w.bidirectional, w.causal,
                                 w.softmax_scale, kv_len=kv, rows=rows, nthreads=nthreads)
    if w.kind == "alibi":
        return oracle.alibi_fwd(np_(x["q"]), np_(x["k"]), np_(x["v"]), raw(x["slopes"]),
                                w.causal, w.softmax_scale, kv_len=kv, rows=rows,
                                nthreads=nthreads)
    if w.kind == "offset":
        return oracle.offset_table_fwd(np_(x["q"]), np_(x["k"]), np_(x["v"]), raw(x["table"]),
                                       w.clip_k, w.causal, w.softmax_scale, kv_len=kv,
                                       rows=rows, nthreads=nthreads)
    if w.kind == "labeled":
        from relative_position_representations_gb300 import workloads as wl
        return oracle.labeled_fwd(np_(x["q"]), np_(x["k"]), np_(x["v"]), np_(x["aK"]),
                                  np_(x["aV"]), raw(x["labels"]), w.causal, w.softmax_scale,
                                  kv_len=kv, table_head_stride=wl.table_head_stride(w),
                                  rows=rows, nthreads=nthreads)
    from relative_position_representations_gb300 import workloads as wl
    return oracle.relattn_fwd(np_(x["q"]), np_(x["k"]), np_(x["v"]), np_(x["aK"]), np_(x["aV"]),
                              w.clip_k, w.causal, w.softmax_scale, kv_len=kv,
                              table_head_stride=wl.table_head_stride(w), rows=rows,
                              nthreads=nthreads)


def row_flops(w, kv_len, rows):
    """Algorithmic FLOPs of a set of flat row ids (same accounting as algorithmic_flops);
    for the decode step the ids are sequences (all heads)."""
    if w.kind in ("decode", "bwd", "txl"):
        return algorithmic_flops(w.replace(B=len(rows)),
                                 None if kv_len is None else [kv_len[int(b)] for b in rows])
    total = 0.0
    reach = 0
    if w.kind == "shaw":
        reach = ((w.clip_k + 1) if w.causal else (2 * w.clip_k + 1)) * (
            int(w.key_term) + int(w.value_term))
    elif w.kind == "labeled":
        reach = w.num_labels * (int(w.key_term) + int(w.value_term))
    for r in rows:
        bh, i = divmod(int(r), w.n)
        b = bh // w.H
        kv = w.n if kv_len is None else min(int(kv_len[b]), w.n)
        keys = min(i + 1, kv) if w.causal else kv
        total += 4.0 * w.d * keys + 2.0 * w.d * reach
    return total


def time_oracle(w, x, budget_s: float, seed: int = 1, nthreads=None):
    """Run the oracle on random rows of the workload for about budget_s seconds."""
    import numpy as np
    import oracle
    nthreads = nthreads or oracle.default_threads()
    rng = np.random.default_rng(seed)
    total_rows = w.B if w.kind in ("decode", "bwd", "txl") else w.B * w.H * w.n
    kv = key_lengths(w, x)
    # calibrate on a small batch of rows
    count = min(total_rows, max(nthreads * 4, 64))
    while True:
        rows = rng.choice(total_rows, size=count, replace=False)
        t0 = time.perf_counter()
        oracle_rows_call(w, x, rows, nthreads)
        dt = time.perf_counter() - t0
        if dt >= 0.5 or count >= total_rows:
            break
        count = min(total_rows, count * 4)
    target = min(total_rows, max(count, int(count * budget_s / max(dt, 1e-6))))
    rows = rng.choice(total_rows, size=target, replace=False)
    fl1 = row_flops(w, kv, rows)
    passes, fl, t0 = 0, 0.0, time.perf_counter()
    while True:  # whole passes over the sample until the budget is used
        oracle_rows_call(w, x, rows, nthreads)
        passes += 1
        fl += fl1
        dt = time.perf_counter() - t0
        if dt >= budget_s or target < total_rows:
            break
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": "%d of %d %s (random, seed %d) x %d pass(es), fp64 %s, "
                      "%.1f s" % (target, total_rows,
                                  "sequences (all heads)" if w.kind in ("decode", "bwd", "txl")
                                  else "query rows",
                                  seed, passes,
                                  "numpy gradient oracle" if w.kind == "bwd" else
                                  "numpy Transformer-XL oracle" if w.kind == "txl" else "C loop",
                                  dt)}, fl, dt


# ----------------------------------------------------------------------- GPU arm
def gpu_call(rp, w, g, out, stream):
    from relative_position_representations_gb300 import workloads as wl
    if w.kind == "bwd":
        if "ws" not in g:  # the caller's workspace (made once)
            import torch
            nb = rp.relattn_bwd_workspace_size(w.B, w.H, w.n, w.d, w.clip_k)
            g["ws"] = torch.empty(max(nb, 4), dtype=torch.uint8, device=g["q"].device)
        return rp.relattn_bwd(g["q"], g["k"], g["v"], g["dout"], aK=g["aK"], aV=g["aV"],
                              clip_k=w.clip_k, causal=w.causal, scale=w.softmax_scale,
                              kv_len=g["kv_len"], table_head_stride=wl.table_head_stride(w),
                              workspace=g["ws"], stream=stream)
    if w.kind == "decode":
        if "ws" not in g:  # the caller's scratch for the split over the caches (made once)
            import torch
            nb = rp.relattn_decode_workspace_size(w.B, w.H, w.n, w.d)
            g["ws"] = (None if NO_DECODE_WORKSPACE else
                       torch.empty(max(nb, 16), dtype=torch.uint8, device=g["q"].device))
        return rp.relattn_decode_fwd(g["q"], g["k"], g["v"], g["cache_len"], aK=g["aK"],
                                     aV=g["aV"], clip_k=w.clip_k, scale=w.softmax_scale, out=out,
                                     table_head_stride=wl.table_head_stride(w), workspace=g["ws"],
                                     stream=stream)
    if w.kind == "t5":
        return rp.relattn_t5bias_fwd(g["q"], g["k"], g["v"], g["bias"], w.num_buckets,
                                     w.max_distance, w.bidirectional, w.causal, w.softmax_scale,
                                     kv_len=g.get("kv_len"), out=out, stream=stream)
    if w.kind == "alibi":
        return rp.relattn_alibi_fwd(g["q"], g["k"], g["v"], g["slopes"], w.causal,
                                    w.softmax_scale, kv_len=g["kv_len"], out=out, stream=stream)
    if w.kind == "txl":
        return rp.relattn_txl_fwd(g["q"], g["k"], g["v"], g["rel"], g["u"], g["vb"],
                                  causal=w.causal, scale=w.softmax_scale, kv_len=g["kv_len"],
                                  out=out, stream=stream)
    if w.kind == "labeled":
        return rp.relattn_labeled_fwd(g["q"], g["k"], g["v"], g["labels"], aK=g["aK"], aV=g["aV"],
                                      causal=w.causal, scale=w.softmax_scale, kv_len=g["kv_len"],
                                      out=out, table_head_stride=wl.table_head_stride(w),
                                      stream=stream)
    if w.kind == "offset":
        return rp.relattn_offset_bias_fwd(g["q"], g["k"], g["v"], g["table"], w.clip_k,
                                          w.causal, w.softmax_scale, kv_len=g["kv_len"],
                                          out=out, stream=stream)
    return rp.relattn_fwd(g["q"], g["k"], g["v"], g["aK"], g["aV"], w.clip_k, w.causal,
                          w.softmax_scale, kv_len=g["kv_len"], out=out,
                          table_head_stride=wl.table_head_stride(w), stream=stream)


NO_DECODE_WORKSPACE = False  # --no-decode-workspace: the decode step gets no scratch


def launches_per_step(rp, w) -> int:
    """Kernels one step launches: the fused kernel, or the decode pieces and their combine."""
    if (w.kind == "decode" and not NO_DECODE_WORKSPACE and
            rp.relattn_decode_workspace_size(w.B, w.H, w.n, w.d) > 0):
        return 2
    if w.kind == "bwd":  # the table memsets and the dq memset are not kernels of ours
        rows = w.clip_k + 1 if w.causal else 2 * w.clip_k + 1
        if (bwd_on_tensor_cores(w) and w.d == 64 and w.n <= 128 and
                (rows <= 48 or not (w.key_term or w.value_term))):
            return 1  # the one-tile kernel
        return 3 if (w.key_term or w.value_term) else 2
    return 1


def make_event(external: bool):
    import torch
    if external:
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return None
    return torch.cuda.Event(enable_timing=True)


def workload_config(w, world: int, l2_note: str) -> dict:
    """The JSON `config` of both arms: the workload by name and shape."""
    return {"workload": w.name, "B": w.B, "H": w.H, "n": w.n, "d": w.d,
            "kind": w.kind,
            "clip_k": w.clip_k if w.kind in ("shaw", "decode", "bwd", "offset") else None,
            "causal": w.causal,
            "terms": ("t5 bias" if w.kind == "t5" else
                      "Transformer-XL (q+u).k + (q+v).r over every offset" if w.kind == "txl" else
                      "alibi bias (slopes 2^(-%g(h+1)/H))" % w.alibi_max_bias
                      if w.kind == "alibi" else
                      "per-offset scalar bias, radius %d" % w.clip_k if w.kind == "offset" else
                      "%s with %d labels (uint8 label matrix %s)" % (
                          "+".join(t for t, on in (("aK", w.key_term), ("aV", w.value_term)) if on),
                          w.num_labels, "per sequence" if w.labels_per_sequence else "shared")
                      if w.kind == "labeled" else
                      "+".join(t for t, on in (("aK", w.key_term), ("aV", w.value_term))
                               if on) or "none"),
            ("cache_len" if w.kind == "decode" else "kv_len"):
                "U{%d..%d} per sequence" % w.kv_len_range if w.kv_len_range else None,
            "parallelism": "dp%d (independent shards, no collective)" % world,
            "l2": l2_note}


def whole_job(elapsed_ms: float, work: float, world: int, device) -> tuple:
    """Whole-job timing over ranks: the slowest rank's time and the work of all ranks.

    Each rank processes its own independent shard (weak scaling), so the job ends when the
    slowest rank ends. No data moves between ranks; only these two scalars are reduced."""
    if world <= 1:
        return float(elapsed_ms), float(work)
    import torch
    import torch.distributed as dist
    tt = torch.tensor([elapsed_ms], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    ww = torch.tensor([work], device=device, dtype=torch.float64)
    dist.all_reduce(ww, op=dist.ReduceOp.SUM)
    return float(tt.item()), float(ww.item())


def input_sets(w, x, dev):
    """Enough resident copies of the inputs (distinct buffers, same values) that a pass over
    them exceeds 4x L2, so the timed reads come from HBM."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    in_bytes = sum(t.numel() * t.element_size() for t in x.values() if t is not None)
    n_sets = max(1, min(64, math.ceil(4 * l2 / max(in_bytes, 1))))
    sets = []
    for s in range(n_sets):
        g = {kk: (vv.to(dev) if vv is not None else None) for kk, vv in x.items()}
        if s > 0:
            g = {kk: (vv.clone() if vv is not None else None) for kk, vv in g.items()}
        sets.append((g, torch.empty_like(g["q"])))
    note = ("inputs larger than L2: %d rotating input sets of %.1f MB (%.0f MB > 4 x %.0f MB "
            "L2), replayed from a CUDA graph" % (n_sets, in_bytes / 1e6, n_sets * in_bytes / 1e6,
                                                 l2 / 1e6))
    return sets, l2, note


def percentile(xs, q):
    ys = sorted(xs)
    if not ys:
        return None
    k = (len(ys) - 1) * q
    lo, hi = int(math.floor(k)), int(math.ceil(k))
    return ys[lo] + (ys[hi] - ys[lo]) * (k - lo)


class DeviceTimer:
    """One CUDA graph of exactly `steps` launches over the rotating input sets, with an
    external CUDA event recorded on the launching stream before each launch and after the
    last, so that one replay gives the timed region and every launch's duration."""

    def __init__(self, rp, w, sets, stream, steps, warmup):
        import torch
        self.stream = stream
        self.steps = steps
        with torch.cuda.stream(stream):  # warm-up, also sets the kernel attributes
            for i in range(max(warmup, 1)):
                g, o = sets[i % len(sets)]
                gpu_call(rp, w, g, o, stream)
        stream.synchronize()
        probe = make_event(True)
        self.use_events = probe is not None
        self.evs = [make_event(True) for _ in range(steps + 1)] if self.use_events else []
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            for s in range(steps):
                if self.use_events:
                    self.evs[s].record(stream)
                g, o = sets[s % len(sets)]
                gpu_call(rp, w, g, o, stream)
            if self.use_events:
                self.evs[steps].record(stream)
        with torch.cuda.stream(stream):
            self.graph.replay()  # untimed replay
        stream.synchronize()

    def replay(self):
        import torch
        with torch.cuda.stream(self.stream):
            self.graph.replay()

    def timed(self):
        """(elapsed ms of one replay, per-launch ms list)."""
        import torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            self.graph.replay()
            e1.record(self.stream)
        torch.cuda.synchronize()
        per = ([self.evs[s].elapsed_time(self.evs[s + 1]) for s in range(self.steps)]
               if self.use_events else [])
        return e0.elapsed_time(e1), per


def l2_flushed_launch_ms(rp, w, g, o, dev, stream, reps=20):
    """Single launches, each after a write of a buffer twice the L2 size (torch fill, not
    timed): CUDA events on the launching stream around the kernel alone; the median."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1, dtype=torch.float32, device=dev)
    ts = []
    with torch.cuda.stream(stream):
        for r in range(reps + 2):
            flush.fill_(float(r))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gpu_call(rp, w, g, o, stream)
            e1.record(stream)
            stream.synchronize()
            if r >= 2:
                ts.append(e0.elapsed_time(e1))
    del flush
    return statistics.median(ts)


def roofline(w, flops, byts, kern_ms, peaks, peak_src):
    """Bound, achieved and fraction of the dominant roof for one launch of kern_ms."""
    alu = simt_roof(w)
    compute_peak = FP32_SIMT_TFLOPS if alu else peaks["bf16_tflops"]
    t_roof_compute = flops / (compute_peak * 1e12)
    t_roof_mem = byts / (peaks["hbm_gbs"] * 1e9)
    if alu and t_roof_compute > t_roof_mem:
        achieved = flops / (kern_ms * 1e-3) / 1e12
        return {"bound": "alu", "achieved": round(achieved, 2), "peak": FP32_SIMT_TFLOPS,
                "unit": "TFLOP/s", "frac": round(achieved / FP32_SIMT_TFLOPS, 4),
                "peak_source": "derived: 152 SMs x 128 fp32 FMA/clk x 2 flop x 2.07 GHz"}
    if t_roof_mem >= t_roof_compute:
        achieved = byts / (kern_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": peak_src + " (STREAM-style copy)"}
    achieved = flops / (kern_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
            "peak_source": peak_src + " (cuBLAS bf16 burst)"}


def measure_also(rp, name, args, dev, stream, peaks, peak_src):
    """A compact device-timed line for another workload: the same graph timing (--steps
    launches over rotating input sets), roofline and profiled traffic; no e2e, no oracle."""
    import torch
    w = workload_by_name(name)
    x = draw(w, seed=args.seed)
    kv_len = key_lengths(w, x)
    flops, byts = algorithmic_flops(w, kv_len), algorithmic_bytes(w, kv_len)
    sets, _, note = input_sets(w, x, dev)
    tm = DeviceTimer(rp, w, sets, stream, args.steps, args.warmup)
    elapsed_ms, per = tm.timed()
    status = rp.relattn_get_device_error(stream)
    if status != 0:
        raise RuntimeError("device status word set while timing %s: %s"
                           % (name, rp.relattn_status_string(status)))
    kern_ms = statistics.mean(per) if per else elapsed_ms / args.steps
    roof = roofline(w, flops, byts, kern_ms, peaks, peak_src)
    roof["traffic"] = profiled_traffic(w.name, kernel_family(w))
    roof["kernel_ms"] = round(kern_ms, 5)
    if per:
        roof["kernel_ms_p10"] = round(percentile(per, 0.1), 5)
        roof["kernel_ms_p90"] = round(percentile(per, 0.9), 5)
    if roof["bound"] == "hbm":
        roof["kernel_ms_l2_flushed"] = round(
            l2_flushed_launch_ms(rp, w, sets[0][0], sets[0][1], dev, stream), 5)
    line = {"workload": name, "value": round(flops * args.steps / (elapsed_ms * 1e-3) / 1e12, 3),
            "unit": "TFLOP/s", "steps": args.steps, "ms_per_step": round(elapsed_ms / args.steps, 6),
            "config": workload_config(w, 1, note), "roofline": roof,
            "gpu_launches": args.steps * launches_per_step(rp, w)}
    del tm, sets
    torch.cuda.synchronize()
    return line


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import relative_position_representations_gb300 as rp

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = workload_by_name(args.workload)
    x = draw(w, seed=args.seed + rank)
    kv_len = key_lengths(w, x)
    flops = algorithmic_flops(w, kv_len)
    byts = algorithmic_bytes(w, kv_len)
    sets, l2, l2_note = input_sets(w, x, dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    steps = args.steps
    tm = DeviceTimer(rp, w, sets, stream, steps, args.warmup)

    # clocks sampled around and during the timed region, with the same launches running
    sampler = ClockSampler(local_rank)
    soak = 0.0 if args.no_clocks else 0.6

    def soak_for(sec):
        until = time.time() + sec
        while time.time() < until:
            tm.replay()
            stream.synchronize()

    if soak:
        sampler.start()
        soak_for(soak)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start_wall = time.time()
    elapsed_ms, kernel_ms = tm.timed()
    t_end_wall = time.time()
    if world > 1:
        dist.barrier()
    if soak:
        soak_for(soak)
    sampler.stop()
    # a bounded device wait that ran out voids the timing (and the outputs)
    status = rp.relattn_get_device_error(stream)
    if status != 0:
        raise RuntimeError("device status word set during the timed region: %s"
                           % rp.relattn_status_string(status))
    clocks = sampler.summary(t_start_wall - soak, t_end_wall + soak) if soak else None
    if kernel_ms and any(m > 0 for m in kernel_ms):
        kern_ms = statistics.mean(kernel_ms)
        kern_src = ("cuda events on the launching stream between the %d launches of the timed "
                    "graph replay" % len(kernel_ms))
    else:
        kern_ms = elapsed_ms / steps
        kern_src = "timed-region elapsed / steps (events in graphs unavailable)"

    # whole-job reduction over ranks (max time, summed work)
    t_max, total_flops = whole_job(elapsed_ms, flops * steps, world, dev)
    value = total_flops / (t_max * 1e-3) / 1e12

    peaks, peak_src = read_peaks()
    roof = roofline(w, flops, byts, kern_ms, peaks, peak_src)
    roof["traffic"] = profiled_traffic(w.name, kernel_family(w))
    roof["kernel_ms"] = round(kern_ms, 5)
    if kernel_ms:
        roof["kernel_ms_p10"] = round(percentile(kernel_ms, 0.1), 5)
        roof["kernel_ms_p90"] = round(percentile(kernel_ms, 0.9), 5)
    if roof["bound"] == "hbm" and w.kind not in ("decode",):
        roof["kernel_ms_l2_flushed"] = round(
            l2_flushed_launch_ms(rp, w, sets[0][0], sets[0][1], dev, stream), 5)
    roof["kernel_time_source"] = kern_src
    roof["algorithmic_flops"] = flops
    roof["algorithmic_bytes"] = byts
    del tm, sets
    torch.cuda.synchronize()

    # end to end through the C ABI with pinned host buffers
    e2e = None if args.no_e2e else measure_e2e(rp, w, x, dev, stream, flops, args)

    # the other forward configurations, device-timed the same way (rank 0, one GPU)
    also = []
    if rank == 0 and world == 1 and args.also:
        for name in [a for a in args.also.split(",") if a and a != w.name]:
            also.append(measure_also(rp, name, args, dev, stream, peaks, peak_src))

    alu = simt_roof(w)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, _, _ = time_oracle(w, x, args.cpu_budget)
        cpu["model"] = host_cpu_model()
        # the small configurations also get a 1-thread figure
        if w.name in ("tiny_fp32", "base_encoder", "big_decoder"):
            one, _, _ = time_oracle(w, x, min(args.cpu_budget, 4.0), nthreads=1)
            cpu["single_thread"] = {"value": one["value"], "sample": one["sample"]}

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(t_max / steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # the arithmetic type: the tensor-core kernels multiply bf16, the SIMT kernels fp32
        "dtype": "bf16" if (w.dtype == "bf16" and not alu) else "f32", "data": "synthetic",
        "config": workload_config(w, world, l2_note),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": steps * launches_per_step(rp, w),
        "clocks": clocks,
    }
    if also:
        line["workloads"] = also
    return line


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def measure_e2e(rp, w, x, dev, stream, flops, args):
    """Same step through the C ABI with pinned host inputs: H2D copies, launch, D2H copy,
    every step, run as a two-slot pipeline the way an input pipeline feeds a device: the next
    step's inputs copy in on copy streams (one per input tensor, so the copies of one step
    run side by side) while this step computes on `stream`, and each step's result copies out
    on another stream. Per step the copies and the launch are those of a serial loop; they
    overlap across steps, with events ordering each buffer's reuse.
    Decode step: the key/value caches and the tables are resident state (copied once, before
    timing); each step copies the new queries and the cache lengths."""
    import torch
    per_step = ("q", "cache_len") if w.kind == "decode" else tuple(x.keys())
    host = {k: (v.pin_memory() if v is not None else None) for k, v in x.items()}
    slots = []
    for _ in range(2):
        g = {k: (torch.empty_like(v, device=dev) if v is not None else None) for k, v in x.items()}
        for k, v in host.items():
            if v is not None and k not in per_step:
                g[k].copy_(v)
        slots.append({"g": g, "out": torch.empty_like(g["q"]), "res": None, "back": None,
                      "h2d": torch.cuda.Event(), "done": torch.cuda.Event(), "d2h": torch.cuda.Event()})
    h2d = sum(v.numel() * v.element_size() for k, v in host.items()
              if v is not None and k in per_step)
    in_keys = [k for k, v in host.items() if v is not None and k in per_step]
    cp_in = {k: torch.cuda.Stream(device=dev) for k in in_keys}
    for sl in slots:
        sl["h2d"] = {k: torch.cuda.Event() for k in in_keys}
    cp_out = torch.cuda.Stream(device=dev)
    t0_stream = torch.cuda.Stream(device=dev)  # marks the start of the timed region
    issued = [0]

    def step():
        sl = slots[issued[0] % 2]
        first_use = issued[0] < 2
        issued[0] += 1
        for k in in_keys:  # inputs: once the slot's previous kernel has read them
            cs = cp_in[k]
            with torch.cuda.stream(cs):
                if not first_use:
                    cs.wait_event(sl["done"])
                sl["g"][k].copy_(host[k], non_blocking=True)
                sl["h2d"][k].record(cs)
        with torch.cuda.stream(stream):  # the step, once its inputs are in and the slot's last
            for k in in_keys:  # results are out
                stream.wait_event(sl["h2d"][k])
            if not first_use:
                stream.wait_event(sl["d2h"])
            res = gpu_call(rp, w, sl["g"], sl["out"], stream)
            res = [t for t in res if t is not None] if isinstance(res, tuple) else [res]
            sl["done"].record(stream)
        sl["res"] = res  # keeps the result tensors alive until their copy out has run
        if sl["back"] is None:
            sl["back"] = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in res]
        with torch.cuda.stream(cp_out):
            cp_out.wait_event(sl["done"])
            for hb, t in zip(sl["back"], res):
                hb.copy_(t, non_blocking=True)
            sl["d2h"].record(cp_out)

    for _ in range(4):
        step()
    torch.cuda.synchronize(dev)
    d2h = sum(t.numel() * t.element_size() for t in slots[0]["back"])
    n = max(5, min(200, args.steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(t0_stream)
    for cs in cp_in.values():
        cs.wait_stream(t0_stream)
    for _ in range(n):
        step()
    cp_out.wait_event(slots[(issued[0] - 1) % 2]["d2h"])
    e1.record(cp_out)
    torch.cuda.synchronize(dev)
    status = rp.relattn_get_device_error(stream)
    if status != 0:
        raise RuntimeError("device status word set during the end-to-end run: %s"
                           % rp.relattn_status_string(status))
    ms = e0.elapsed_time(e1) / n
    return {"value": round(flops / (ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 5), "steps": n,
            "pipeline": "two slots: H2D of the next step on copy streams (one per input "
                        "tensor), the step on the compute stream, D2H of its result on another"}


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, on bounded samples of the workload: the
    inputs are converted to the oracle's fp64 arrays once, the sample size is calibrated once,
    and every step then runs the oracle on a fresh random sample of that many rows, so the
    whole run stays within about ref_budget seconds whatever --steps is."""
    import numpy as np
    import oracle
    w = workload_by_name(args.workload)
    x = draw(w, seed=args.seed)
    if w.kind not in ("decode", "bwd", "txl"):
        x = host_arrays(x)
    nthreads = oracle.default_threads()
    per_step = max(0.02, args.ref_budget / max(1, args.steps + args.warmup))
    total_rows = w.B if w.kind in ("decode", "bwd", "txl") else w.B * w.H * w.n
    kv = key_lengths(w, x)
    rng = np.random.default_rng(args.seed + 1)
    count = min(total_rows, max(nthreads, 16))
    while True:  # calibration: grow the sample until one call takes a measurable time
        t0 = time.perf_counter()
        oracle_rows_call(w, x, rng.choice(total_rows, size=count, replace=False), nthreads)
        dt = time.perf_counter() - t0
        if dt >= 0.2 or count >= total_rows:
            break
        count = min(total_rows, count * 4)
    size = int(min(total_rows, max(1, count * per_step / max(dt, 1e-6))))
    for _ in range(args.warmup):
        oracle_rows_call(w, x, rng.choice(total_rows, size=size, replace=False), nthreads)
    tot_fl, tot_dt = 0.0, 0.0
    for _ in range(args.steps):
        rows = rng.choice(total_rows, size=size, replace=False)
        t0 = time.perf_counter()
        oracle_rows_call(w, x, rows, nthreads)
        tot_dt += time.perf_counter() - t0
        tot_fl += row_flops(w, kv, rows)
    value = tot_fl / tot_dt / 1e12
    unit_name = "sequences (all heads)" if w.kind in ("decode", "bwd", "txl") else "query rows"
    cpu = {"value": round(value, 6), "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
           "sample": "each step: %d of %d %s (random, seed %d), fp64 oracle, %.3f s per step"
                     % (size, total_rows, unit_name, args.seed + 1, tot_dt / max(1, args.steps))}
    return {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": workload_config(w, world, "host memory (the oracle runs on the CPU cores)"),
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-decode-workspace", action="store_true",
                    help="decode workloads: call without a workspace (one CTA per cache)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="total seconds of oracle work for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true", help="skip clock sampling and its soak")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--also", default=ALSO_WORKLOADS,
                    help="comma-separated workloads also device-timed in the same run ('' = none)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    global NO_DECODE_WORKSPACE
    NO_DECODE_WORKSPACE = args.no_decode_workspace

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line = run_ours(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
