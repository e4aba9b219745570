#!/usr/bin/env python
"""Benchmark: masked multi-head attention forward TFLOPS on GB300.

Default workload: long causal self-attention, bf16, B=4 h=16 n=m=8192 d_k=64
(the workload the throughput target is stated on).  One step = one attn_fwd
call over the whole batch (every step of the hot path runs in that one
kernel launch).  Inputs: 3 x 64 MiB + 64 MiB output = 268 MB, larger than the
126 MB L2, so consecutive steps cannot serve each other from L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own full
batch (independent (batch, head) work, no collective on the data path) and
the time is the max over ranks: weak scaling.

Besides the contract's keys, the line carries (unless --kernel-only):
other_workloads (the four short configurations), backward, decode, window
(d_k = 64), head_widths (the encoder shape at d_k 16, 32, 64, 128), wide_heads
(d_k = 128 on the long sequences: causal, unmasked, windows 256 and 1024), mha
(projections + attention) and cpu_baseline.  roofline.traffic is the DRAM bytes
of one launch from the committed ncu capture, reported while roofline.source_hash
(the flash kernel's sources) matches it.  parity holds the check of the buffers
that were timed against the fp64 oracle the cpu_baseline leg runs anyway: the
sampled rows of the main workload in the output of its last timed step, and
workloads 1-4 element by element in the outputs of their timed launches (1e-2
absolute for bf16, 1e-4 for fp32); a miss ends the run with an error.

--impl reference times the fp64 CPU oracle on the host cores instead, on a
bounded sample of query rows of the same workload per step (the pages have no
GPU implementation to compare against).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import DECODE, draw_dout, draw_mha, WORKLOADS, draw  # noqa: E402

METRIC = "masked MHA fwd TFLOPS on 1 GB300 (and % of bf16 tensor peak / HBM GB/s)"
UNIT = "TFLOPS"


def nominal_flops(w) -> float:
    """4 * B * h * m * n * d_k, halved for a causal mask (the headline formula)."""
    f = 4.0 * w.B * w.h * w.m * w.n * w.d
    return f / 2 if w.causal else f


def allowed_pairs(w, lengths) -> float:
    """Number of (query, key) pairs the mask allows, summed over batch and heads."""
    total = 0.0
    for b in range(w.B):
        L = w.n if not w.padded else max(0, min(int(lengths[b]), w.n))
        if w.causal:
            # keys j <= i and j < L, for i in [0, m)
            total += sum(min(i + 1, L) for i in range(w.m))
        else:
            total += w.m * L
    return total * w.h


def useful_flops(w, lengths) -> float:
    """4 * d_k per allowed pair (2 d_k for Q K^T, 2 d_k for P V)."""
    return 4.0 * w.d * allowed_pairs(w, lengths)


def algorithmic_bytes(w, lengths) -> float:
    """Q and O once, K and V once up to the allowed length per (batch)."""
    esz = 2 if w.dtype == "bf16" else 4
    kv_rows = 0
    for b in range(w.B):
        L = w.n if not w.padded else max(0, min(int(lengths[b]), w.n))
        kv_rows += L
    return esz * w.d * (2 * w.B * w.h * w.m + 2 * w.h * kv_rows)


def row_pairs(w, lengths, rows) -> float:
    """Allowed (query, key) pairs of the given linear output rows ((b*h + head)*m + i)."""
    rows = np.asarray(rows, dtype=np.int64)
    i = rows % w.m
    b = (rows // w.m) // w.h
    L = np.clip(np.asarray(lengths, dtype=np.int64)[b], 0, w.n) if w.padded else np.full(rows.shape, w.n)
    return float((np.minimum(i + 1, L) if w.causal else L).sum())


# DRAM bytes (read + write) of one flash-kernel launch on the default workload,
# from one ncu capture of that launch (dram__bytes_read.sum + dram__bytes_write.sum), keyed by a hash of
# the sources the kernel is compiled from: any later change to them reports null.
MEASURED_TRAFFIC = {"3664032251713a35": 201701632 + 48632064}
FLASH_SOURCES = ("attn_flash.cu", "softmax_tile.cuh", "ptx.cuh")


def flash_source_hash():
    import hashlib
    h = hashlib.sha256()
    for name in FLASH_SOURCES:
        h.update(open(os.path.join(ROOT, "transformer_scaled_dot_masked_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic():
    return MEASURED_TRAFFIC.get(flash_source_hash())


def workload_config(w):
    """The workload part of the JSON line's config, the same on both arms."""
    return {"workload": w.description, "B": w.B, "h": w.h, "m": w.m, "n": w.n, "d_k": w.d,
            "mask": "causal" if w.causal else ("key_padding" if w.padded else "none")}


def load_sustained_peak():
    """The bf16 dense rate measured over seconds under the power cap (None if absent)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return None


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for _, _, flags in rows for k, f in enumerate(flags) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def to_device(x, dtype, torch, device):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def max_over_ranks(ms, dist, device):
    """The slowest rank's time: every rank must be done for the job to be done."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank, world, ms):
    """Aggregate throughput: the work of all ranks over the slowest rank's time."""
    return flops_per_rank * world / (ms * 1e-3) / 1e12


def time_launches(fn, steps, torch, stream):
    """Average device time of `steps` calls of fn on `stream`, CUDA events on that stream."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / steps


SHORT_REPLAYS = 10  # graph replays per short workload; the figure is their median


def short_workloads(torch, attn, device, peak_hbm):
    """Per-launch time of the memory-bound workloads (and the fp32 one) with
    input sets rotated so their total exceeds twice the L2 size; launches are
    captured in a CUDA graph so the figure is device time, not launch latency.
    Also returns, by workload name, the output the timed launches wrote into the
    first input set's buffer (float64 on the host), for the parity check."""
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    res, outputs = {}, {}
    for cfg in (1, 2, 3, 4):
        w = WORKLOADS[cfg]
        inp = draw(w)
        esz = 2 if w.dtype == "bf16" else 4
        set_bytes = esz * w.d * (2 * w.B * w.h * w.m + 2 * w.B * w.h * w.n)
        copies = max(1, min(64, int(np.ceil(2 * l2 / set_bytes))))
        sets = []
        for _ in range(copies):
            q, k, v = (to_device(x, w.dtype, torch, device) for x in (inp.q, inp.k, inp.v))
            lens = torch.from_numpy(inp.key_lengths).to(device)
            sets.append((q, k, v, lens, torch.empty_like(q)))
        kern = attn.select_kernel(w.B, w.h, w.m, w.n, w.d, 0 if w.dtype == "bf16" else 1, w.mask)
        stream = torch.cuda.Stream(device)
        with torch.cuda.stream(stream):
            for s in sets:
                attn.attn_fwd(s[0], s[1], s[2], s[3], w.mask, w.scale, out=s[4], stream=stream)
            stream.synchronize()
            reps = max(1, 200 // copies)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    for s in sets:
                        attn.attn_fwd(s[0], s[1], s[2], s[3], w.mask, w.scale, out=s[4], stream=stream)
            g.replay()
            stream.synchronize()
            times = []
            for _ in range(SHORT_REPLAYS):
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record(stream)
                g.replay()
                t1.record(stream)
                t1.synchronize()
                times.append(t0.elapsed_time(t1) / (reps * copies))
        ms = statistics.median(times)
        outputs[w.name] = sets[0][4].double().cpu().numpy()
        nb = algorithmic_bytes(w, inp.key_lengths)
        res[w.name] = {
            "kernel": attn._native.KERNEL_NAMES[kern], "us_per_launch": ms * 1e3,
            "tflops_nominal": nominal_flops(w) / (ms * 1e-3) / 1e12,
            "tflops_useful": useful_flops(w, inp.key_lengths) / (ms * 1e-3) / 1e12,
            "hbm_gbs_algorithmic": nb / (ms * 1e-3) / 1e9,
            "hbm_frac": nb / (ms * 1e-3) / 1e9 / peak_hbm,
            "input_sets": copies, "launches_timed": reps * copies * SHORT_REPLAYS,
        }
        del sets, g
        torch.cuda.empty_cache()
    return res, outputs


def backward_workload(torch, attn, device, peak_tf, steps=20):
    """The backward of workload 5 (B4 h16 n=m=8192 causal): attn_bwd from the output and
    log-sum-exp of attn_fwd_lse, inputs resident; per call three kernels (row pass,
    tensor-core pass, dQ conversion).  Useful work: 10*d_k FLOPs per allowed pair
    (S recomputed, dP, dV, dK, dQ)."""
    w = WORKLOADS[5]
    inp = draw(w)
    q, k, v = (to_device(x, w.dtype, torch, device) for x in (inp.q, inp.k, inp.v))
    do = to_device(draw_dout(w), w.dtype, torch, device)
    lens = torch.from_numpy(inp.key_lengths).to(device)
    stream = torch.cuda.current_stream(device)
    out, lse = attn.attn_fwd_lse(q, k, v, lens, w.mask, w.scale, stream=stream)
    ws = torch.empty(attn.bwd_workspace_size(w.B, w.h, w.m, w.n, w.d), dtype=torch.uint8, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def bwd():
        attn.attn_bwd(q, k, v, out, do, lse, lens, w.mask, w.scale, dq, dk, dv, ws, stream=stream)

    def fwd():
        attn.attn_fwd_lse(q, k, v, lens, w.mask, w.scale, out=out, lse=lse, stream=stream)

    for _ in range(3):
        bwd()
    torch.cuda.synchronize()
    ms_b = time_launches(bwd, steps, torch, stream)
    ms_f = time_launches(fwd, steps, torch, stream)
    st, info = attn.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} (info {info}) after the backward loop")
    flops_b = 2.5 * useful_flops(w, inp.key_lengths)
    return {"workload": w.description, "entry_point": "attn_bwd (after attn_fwd_lse)",
            "us_per_call": ms_b * 1e3, "tflops_useful": flops_b / (ms_b * 1e-3) / 1e12,
            "frac_of_peak": flops_b / (ms_b * 1e-3) / 1e12 / peak_tf,
            "forward_with_lse_us": ms_f * 1e3,
            "training_pass_tflops": 3.5 * useful_flops(w, inp.key_lengths) / ((ms_b + ms_f) * 1e-3) / 1e12,
            "calls_timed": steps, "algorithmic": "10*d_k FLOPs per allowed (query, key) pair"}


def mha_workload(torch, attn, device, peak_tf, steps=50):
    """Multi-head self-attention with its projections for the big model's width (d_model
    1024, h = 16, d_k = 64): B32 sentences of 256 positions with key padding (lengths in
    [128, 256]), through attn_mha_fwd (three input projections, attention, output
    projection).  Useful work: 2*B*L*d_model*h*64 FLOPs per projection (four of them)
    plus 4*d_k per allowed (query, key) pair."""
    B, h, L, dm = 32, 16, 256, 1024
    xq, _, wq, wk, wv, wo = draw_mha(B, h, L, L, dm, seed=1007, self_attention=True)
    lens_np = np.random.default_rng(1008).integers(128, 257, size=B).astype(np.int32)
    dev = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)
    x, Wq, Wk, Wv, Wo = dev(xq), dev(wq), dev(wk), dev(wv), dev(wo)
    lens = torch.from_numpy(lens_np).to(device)
    out = torch.empty_like(x)
    ws = torch.empty(attn.mha_workspace_size(B, h, L, L, dm), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        attn.attn_mha_fwd(x, x, Wq, Wk, Wv, Wo, h, lens, attn.MASK_KEY_PADDING, 0.125, out=out, workspace=ws,
                          stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ms = time_launches(step, steps, torch, stream)
    st, info = attn.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} (info {info}) after the multi-head loop")
    proj = 4 * 2.0 * B * L * dm * h * 64
    att = 4 * 64 * float(np.clip(lens_np, 0, L).sum()) * L * h
    return {"workload": f"multi-head self-attention with projections, bf16, B={B} L={L} d_model={dm} h={h}, "
                        "key padding with lengths in [128,256]",
            "entry_point": "attn_mha_fwd", "us_per_call": ms * 1e3,
            "tflops_useful": (proj + att) / (ms * 1e-3) / 1e12,
            "frac_of_peak": (proj + att) / (ms * 1e-3) / 1e12 / peak_tf, "calls_timed": steps,
            "algorithmic": "4 projections of 2*B*L*d_model*h*64 FLOPs + 4*d_k per allowed pair"}


def head_width_workloads(torch, attn, device, steps=50):
    """The model variants that trade heads for head width at h * d_k = 512 (h=4 d_k=128,
    h=16 d_k=32, h=32 d_k=16) on the encoder workload's shape (B64, n=m=100, key padding),
    next to the base h=8 d_k=64.  All run on tensor cores: widths 16 and 32 zero-padded
    on the d_k = 64 kernels, width 128 on its own kernel."""
    base = WORKLOADS[2]
    res = {}
    for h, d in ((8, 64), (4, 128), (16, 32), (32, 16)):
        w = base.with_(h=h, d=d, scale=d ** -0.5, name=f"encoder_h{h}_d{d}")
        inp = draw(w)
        q, k, v = (to_device(x, w.dtype, torch, device) for x in (inp.q, inp.k, inp.v))
        lens = torch.from_numpy(inp.key_lengths).to(device)
        out = torch.empty_like(q)
        stream = torch.cuda.current_stream(device)

        def step():
            attn.attn_fwd(q, k, v, lens, w.mask, w.scale, out=out, stream=stream)

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        ms = time_launches(step, steps, torch, stream)
        kern = attn.select_kernel(w.B, w.h, w.m, w.n, w.d, 0, w.mask)
        res[w.name] = {"kernel": attn._native.KERNEL_NAMES[kern], "us_per_launch": ms * 1e3,
                       "tflops_useful": useful_flops(w, inp.key_lengths) / (ms * 1e-3) / 1e12}
    return res


def wide_workload(torch, attn, device, peak_tf, steps=50, extra=True):
    """Heads of width 128 on the long causal sequences: workload 5 with h=8, d_k=128
    (B4 n=m=8192, the same d_model of 1024), inputs 268 MB in all (> L2).  Useful work:
    4*d_k FLOPs per allowed (query, key) pair.  With `extra`, the same kernel also on
    the unmasked B4 h8 n=4096 case and on restricted attention with windows 256 and
    1024 over the n=8192 inputs (through attn_fwd_window)."""
    w = WORKLOADS[5].with_(h=8, d=128, scale=128 ** -0.5, name="long_causal_h8_d128")
    inp = draw(w)
    q, k, v = (to_device(x, w.dtype, torch, device) for x in (inp.q, inp.k, inp.v))
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(device)

    def timed(step, what):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        ms = time_launches(step, steps, torch, stream)
        st, info = attn.device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} (info {info}) after the wide-head loop ({what})")
        return ms

    ms = timed(lambda: attn.attn_fwd(q, k, v, None, w.mask, w.scale, out=out, stream=stream), "causal")
    flops = useful_flops(w, inp.key_lengths)
    kern = attn.select_kernel(w.B, w.h, w.m, w.n, w.d, 0, w.mask)
    res = {"workload": f"causal self-attention, bf16, B={w.B} h={w.h} n=m={w.n} d_k={w.d}",
           "entry_point": "attn_fwd", "kernel": attn._native.KERNEL_NAMES[kern], "us_per_call": ms * 1e3,
           "tflops_useful": flops / (ms * 1e-3) / 1e12, "frac_of_peak": flops / (ms * 1e-3) / 1e12 / peak_tf,
           "calls_timed": steps, "algorithmic": "4*d_k FLOPs per allowed (query, key) pair"}
    if not extra:
        return res
    half = w.n // 2
    qh, kh, vh = (x[:, :, :half].contiguous() for x in (q, k, v))
    oh = torch.empty_like(qh)
    ms = timed(lambda: attn.attn_fwd(qh, kh, vh, None, attn.MASK_NONE, w.scale, out=oh, stream=stream), "no mask")
    fl = 4.0 * w.d * w.B * w.h * half * half
    res["no_mask_n4096"] = {"us_per_call": ms * 1e3, "tflops_useful": fl / (ms * 1e-3) / 1e12,
                            "frac_of_peak": fl / (ms * 1e-3) / 1e12 / peak_tf}
    i = np.arange(w.n)
    for win in (256, 1024):
        ms = timed(lambda: attn.attn_fwd_window(q, k, v, None, attn.MASK_WINDOW, win, w.scale, out=out,
                                                stream=stream), f"window {win}")
        pairs = float((np.minimum(i + win, w.n - 1) - np.maximum(i - win, 0) + 1).sum()) * w.B * w.h
        fl = 4.0 * w.d * pairs
        res[f"window_{win}"] = {"us_per_call": ms * 1e3, "tflops_useful": fl / (ms * 1e-3) / 1e12,
                                "frac_of_peak": fl / (ms * 1e-3) / 1e12 / peak_tf}
    return res


def window_workload(torch, attn, device, peak_tf, steps=50, window=256):
    """Restricted self-attention on the long sequences of workload 5 without the causal
    mask: B4 h16 n=m=8192, keys with |i - j| <= 256 (513-position neighbourhoods), through
    attn_fwd_window.  Useful work: 4*d_k FLOPs per allowed (query, key) pair."""
    w = WORKLOADS[5]
    inp = draw(w)
    q, k, v = (to_device(x, w.dtype, torch, device) for x in (inp.q, inp.k, inp.v))
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(device)

    def step():
        attn.attn_fwd_window(q, k, v, None, attn.MASK_WINDOW, window, w.scale, out=out, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ms = time_launches(step, steps, torch, stream)
    st, info = attn.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} (info {info}) after the window loop")
    i = np.arange(w.n)
    pairs = float((np.minimum(i + window, w.n - 1) - np.maximum(i - window, 0) + 1).sum()) * w.B * w.h
    flops = 4 * w.d * pairs
    return {"workload": f"restricted self-attention, bf16, B={w.B} h={w.h} n=m={w.n} d_k={w.d}, window {window}",
            "entry_point": "attn_fwd_window", "us_per_call": ms * 1e3,
            "tflops_useful": flops / (ms * 1e-3) / 1e12, "frac_of_peak": flops / (ms * 1e-3) / 1e12 / peak_tf,
            "calls_timed": steps, "algorithmic": "4*d_k FLOPs per allowed (query, key) pair"}


def decode_workload(torch, attn, device, peak_hbm, steps=50):
    """One incremental-decoding step (workloads.DECODE: B64 h16, one new row each, K/V
    caches of capacity 4096 holding 1024..4096 rows) through attn_decode, caches
    resident (1.07 GB > L2, so no flush).  Algorithmic bytes: every live cached K and
    V row once, plus Q and O."""
    w = DECODE
    inp = draw(w)
    q, k, v = (to_device(x, w.dtype, torch, device) for x in (inp.q, inp.k, inp.v))
    lens = torch.from_numpy(inp.key_lengths).to(device)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(device)
    ws_bytes = attn.decode_workspace_size(w.B, w.h, w.m, w.n)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=device)

    def step():
        attn.attn_decode(q, k, v, lens, w.scale, out=out, workspace=ws, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ms = time_launches(step, steps, torch, stream)
    st, info = attn.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} (info {info}) after the decode loop")
    live = float(np.clip(inp.key_lengths, 0, w.n).sum()) * w.h
    nbytes = live * w.d * 2 * 2 + 2 * w.B * w.h * w.m * w.d * 2 + 4 * w.B
    return {"workload": w.description, "entry_point": "attn_decode (split-KV, CUDA cores)",
            "us_per_call": ms * 1e3, "hbm_gbs_algorithmic": nbytes / (ms * 1e-3) / 1e9,
            "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peak_hbm, "calls_timed": steps,
            "algorithmic": "each live cached K and V row once, plus Q and O (bf16)"}


def parity_tol(w):
    """The bar of the parity tests: 1e-2 absolute for bf16 outputs, 1e-4 for fp32."""
    return 1e-2 if w.dtype == "bf16" else 1e-4


def cpu_oracle_sample(w, inp, target_s, seed=3):
    """Time the fp64 oracle on random query rows of w for about target_s seconds."""
    import oracle
    orc = oracle.load()
    qd, kd, vd = orc.widen(inp.q), orc.widen(inp.k), orc.widen(inp.v)
    rng = np.random.default_rng(seed)
    total_rows = w.B * w.h * w.m

    probe = rng.integers(0, total_rows, size=16)
    t0 = time.perf_counter()
    orc.attn_rows(qd, kd, vd, inp.key_lengths, w.mask, w.scale, probe, widened=True)
    dt = max(time.perf_counter() - t0, 1e-6)
    count = int(np.clip(16 * target_s / dt, 16, total_rows))
    rows = rng.integers(0, total_rows, size=count)
    t0 = time.perf_counter()
    ref = orc.attn_rows(qd, kd, vd, inp.key_lengths, w.mask, w.scale, rows, widened=True)
    el = time.perf_counter() - t0
    flops = 4.0 * w.d * row_pairs(w, inp.key_lengths, rows)
    return {"value": flops / el / 1e12, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"{count} random query rows of {w.description} ({el:.1f} s, fp64, "
                      f"{flops / 1e9:.1f} GFLOP useful)", "seconds": el}, (rows, ref)


def cpu_per_config(all_cores_c5, timed_outputs, parity):
    """The oracle on workloads 1-4 in full, on one core and on all of them, and on
    workload 5's row sample on all cores: useful TFLOPS and seconds per run.  The
    full outputs also check, element by element, the outputs the GPU wrote in the
    timed launches of workloads 1-4 (timed_outputs, by workload name), into parity."""
    import oracle
    orc = oracle.load()
    cores = orc.num_threads()
    res = {"nproc": os.cpu_count(), "threads_all": cores}
    for cfg in (1, 2, 3, 4):
        w = WORKLOADS[cfg]
        inp = draw(w)
        flops = useful_flops(w, inp.key_lengths)
        entry = {}
        for label, threads in (("one_core", 1), ("all_cores", cores)):
            orc.set_num_threads(threads)
            t0 = time.perf_counter()
            ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
            el = time.perf_counter() - t0
            entry[label] = {"tflops_useful": flops / el / 1e12, "seconds": el, "threads": threads}
        res[w.name] = entry
        if w.name in timed_outputs:
            err = float(np.abs(timed_outputs[w.name] - ref).max())
            parity[w.name] = {"elements": int(ref.size), "max_abs_err": err, "tol": parity_tol(w),
                              "ok": err <= parity_tol(w)}
    # workload 5 (5.5e11 useful FLOP, minutes on one core): one core on a random row sample
    w = WORKLOADS[5]
    inp = draw(w)
    orc.set_num_threads(1)
    one, _ = cpu_oracle_sample(w, inp, 3.0, seed=4)
    orc.set_num_threads(cores)
    res[w.name] = {"all_cores": all_cores_c5,
                   "one_core": {"tflops_useful": one["value"], "seconds": one["seconds"], "threads": 1,
                                "sample": one["sample"]}}
    return res


def run_reference(args, w):
    """--impl reference: the fp64 CPU oracle, one bounded row sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    inp = draw(w)
    orc = oracle.load()
    qd, kd, vd = orc.widen(inp.q), orc.widen(inp.k), orc.widen(inp.v)
    rng = np.random.default_rng(11)
    total_rows = w.B * w.h * w.m
    # size each step so the whole run stays within about two minutes
    probe = rng.integers(0, total_rows, size=8)
    t0 = time.perf_counter()
    orc.attn_rows(qd, kd, vd, inp.key_lengths, w.mask, w.scale, probe, widened=True)
    per_row = max((time.perf_counter() - t0) / 8, 1e-6)
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows_per_step = int(np.clip(budget / per_row, 1, 4096))
    for _ in range(args.warmup):
        orc.attn_rows(qd, kd, vd, inp.key_lengths, w.mask, w.scale,
                      rng.integers(0, total_rows, size=rows_per_step), widened=True)
    flops = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        rows = rng.integers(0, total_rows, size=rows_per_step)
        orc.attn_rows(qd, kd, vd, inp.key_lengths, w.mask, w.scale, rows, widened=True)
        flops += 4.0 * w.d * row_pairs(w, inp.key_lengths, rows)
    el = time.perf_counter() - t0
    value = flops / el / 1e12
    sample = f"{rows_per_step} random query rows per step of {w.description}"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=5, choices=sorted(WORKLOADS))
    ap.add_argument("--kernel-only", action="store_true",
                    help="time only the main kernel loop (for profiler runs)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-workspace", action="store_true",
                    help="call attn_fwd (static tile schedule) instead of attn_fwd_ws")
    args = ap.parse_args()
    w = WORKLOADS[args.workload]

    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    import transformer_scaled_dot_masked_gb300 as attn

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    inp = draw(w)  # every rank processes a full batch of its own (weak scaling)
    q, k, v = (to_device(x, w.dtype, torch, device) for x in (inp.q, inp.k, inp.v))
    lens = torch.from_numpy(inp.key_lengths).to(device)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(device)
    kern = attn.select_kernel(w.B, w.h, w.m, w.n, w.d, 0 if w.dtype == "bf16" else 1, w.mask)
    ws = None if args.no_workspace else attn.make_workspace(device)

    def step():
        attn.attn_fwd(q, k, v, lens, w.mask, w.scale, out=out, stream=stream, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        ms = time_launches(step, args.steps, torch, stream)
    torch.cuda.synchronize()
    if dist:
        ms = max_over_ranks(ms, dist, device)
        dist.barrier()
    st, info = attn.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} (info {info}) after the timed loop")

    peak_tf, peak_hbm, peak_src = load_peaks()
    flops_nom = nominal_flops(w)
    value = whole_job_tflops(flops_nom, world, ms)
    flops_use = useful_flops(w, inp.key_lengths)
    achieved = flops_use / (ms * 1e-3) / 1e12
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {**workload_config(w),
                   "kernel": attn._native.KERNEL_NAMES[kern],
                   "entry_point": "attn_fwd" if ws is None else "attn_fwd_ws (dynamic tile schedule)",
                   "l2": "inputs+output 268 MB > L2, no flush between steps",
                   "parallelism": f"replicas x{world} ((batch, head) work is independent)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf,
                     "traffic": measured_traffic() if args.workload == 5 else None,
                     "source_hash": flash_source_hash(),
                     "peak_source": f"{peak_src} bf16 dense burst",
                     "peak_sustained": load_sustained_peak(),
                     "frac_sustained": (achieved / load_sustained_peak()) if load_sustained_peak() else None,
                     "algorithmic": "4*d_k FLOPs per allowed (query, key) pair per launch"},
        "gpu_launches": args.steps,
    }
    result["clocks"] = clk.summary()

    if not args.kernel_only:
        # end to end through the public API on host buffers: attn_fwd_host copies the pinned
        # inputs in, runs the kernels and copies the output back (chunk by chunk, overlapped)
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        hl = lens.cpu().pin_memory()
        ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hws = torch.empty(attn.host_workspace_size(w.B, w.h, w.m, w.n, w.d), dtype=torch.uint8, device=device)

        def e2e_step():
            attn.attn_fwd_host(hq, hk, hv, hl, w.mask, w.scale, out=ho, workspace=hws, stream=stream)

        e2e_steps = max(3, min(args.steps, 50))
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        ems = time_launches(e2e_step, e2e_steps, torch, stream)
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hl))
        result["e2e"] = {"value": flops_nom * world / (ems * 1e-3) / 1e12, "unit": UNIT,
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": ho.numel() * ho.element_size(),
                         "ms_per_step": ems, "steps": e2e_steps,
                         "entry_point": "attn_fwd_host (host buffers; copies in, kernels and copies out overlapped)"}
        result["gpu_launches"] = args.steps  # e2e launches are outside the device-timed region
        result["other_workloads"], timed_outputs = short_workloads(torch, attn, device, peak_hbm)
        result["backward"] = backward_workload(torch, attn, device, peak_tf)
        result["decode"] = decode_workload(torch, attn, device, peak_hbm)
        result["window"] = window_workload(torch, attn, device, peak_tf)
        result["head_widths"] = head_width_workloads(torch, attn, device)
        result["wide_heads"] = wide_workload(torch, attn, device, peak_tf)
        result["mha"] = mha_workload(torch, attn, device, peak_tf)
        if rank == 0:
            cb, (rows, ref) = cpu_oracle_sample(w, inp, args.cpu_seconds)
            seconds = cb.pop("seconds", None)
            # parity on the buffers that were timed: the oracle rows of the sample against
            # the same rows of the output the last timed step wrote, and workloads 1-4 in
            # full against their timed outputs
            got = out.reshape(-1, w.d)[torch.from_numpy(rows).to(device)].double().cpu().numpy()
            err = float(np.abs(got - ref).max())
            parity = {w.name: {"elements": int(ref.size), "rows": int(rows.size), "max_abs_err": err,
                               "tol": parity_tol(w), "ok": err <= parity_tol(w)}}
            cb["per_config"] = cpu_per_config({"tflops_useful": cb["value"], "seconds": seconds,
                                               "threads": cb["cores"], "sample": cb["sample"]},
                                              timed_outputs, parity)
            result["cpu_baseline"] = cb
            result["parity"] = parity
            bad = [k for k, v in parity.items() if not v["ok"]]
            if bad:
                print(json.dumps(result))
                raise RuntimeError(f"timed outputs differ from the oracle beyond the tolerance: {bad}")

    if rank == 0:
        print(json.dumps(result))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
