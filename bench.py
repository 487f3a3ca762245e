#!/usr/bin/env python
"""Benchmark of the Gated DeltaNet recurrence library on GB300.

One step = one gdn_forward call over the decode workload (D_k = D_v = 128,
n_k_heads = 16, n_v_heads = 32, n_tokens = 1, n_seqs = 64, f32; seeded
synthetic inputs), updating the state in place.  Prints ONE JSON line.

Timing: W untimed warm-up steps, then exactly K steps replayed from CUDA
graphs of C-ABI calls, bracketed by a barrier and a device synchronize, timed
with CUDA events on the launching stream; the maximum over ranks is taken.
Steps rotate over 4 independent input/state sets, so about 1.1 GB is touched
between two uses of the same buffer (more than 8x the L2).

Also reported: the end-to-end number through the public API from pinned host
buffers (copies inside the timed region), the HBM roofline of the kernel, the
CPU oracle as a baseline, SM clocks sampled during the timed region, and
quick timings of the other workloads (wide-GQA decode, capture, prefill).

``--impl reference`` times the double-precision CPU oracle on the same
workload and metric instead (a bounded sample of heads per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN decode us/call + state HBM GB/s (% of 8 TB/s); prefill tokens/s"
WORKLOAD_TEXT = ("decode: D_k=D_v=128, n_k_heads=16, n_v_heads=32, n_tokens=1, n_seqs=64, f32, "
                 "in-place state update")
N_SETS = 4
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
SM_COUNT = 152
FP32_LANES_PER_SM = 128


# ---------------------------------------------------------------- helpers

def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "sm_max_mhz": 2070.0}, "fallback"


def kernel_traffic(kernel: str, n_tokens: int | None = None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (the record's "source" and every file in its
    "deps", each matching its sha256); else None.  A record taken on a shorter
    prefill (its "n_tokens") is scaled to ``n_tokens`` by the tokens
    processed (the kernels' traffic grows in proportion); a record with
    several kernels (one call launching both passes) is summed."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)[kernel]
    except Exception:
        return None
    # every file the kernel is built from, each with the hash it was profiled at
    pairs = [(t["source"], t["source_sha256"])] + list(t.get("deps", {}).items())
    for rel, want in pairs:
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != want:
                    return None
        except OSError:
            return None
    b = t["dram_bytes_per_launch"]
    if isinstance(b, dict):
        b = sum(b.values())
    if n_tokens is not None and t.get("n_tokens"):
        b = int(round(b * n_tokens / t["n_tokens"]))
    return b


# ---------------------------------------------------------------- prefill rooflines

def chunked_mma_flops(w, two_pass: bool, split: bool = False, bf16_in: bool = False) -> int:
    """Tensor-core flops the chunked prefill issues per call (2 per MAC of
    every tcgen05 product, full 64-token chunks even for a ragged last one;
    with split-bf16 operands every product runs as three bf16 MMAs, so three
    times the TF32 form's count; with bf16 activations (one-pass form) the
    products of exact inputs leave out their zero lo terms: the Gram one
    product, V^T T''^T, X = S K^T and S Q^T two each, the rest three; in the
    two-pass form the Gram one, [X | Z] and the state update two, the rest
    three).
    Per (seq, value head, chunk) the one-pass form runs the Gram [K;Q]K^T
    (M 128, N 64, K 128), V^T T''^T, X = S K^T, X(-T')^T, S Q'^T, U^T P'^T
    (each M 128, N 64; K 64, 128, 64, 128, 64) and S += U^T K'^T (M 128,
    N 128, K 64).  The two-pass form runs the Gram once per (seq, key head,
    chunk) in its chunk pass, and per (seq, value head, chunk) [X | Z] =
    S [K; Q]^T (M 128, N 128, K 128), U^T = W T''^T and U^T P'^T (M 128, N 64,
    K 64) and S += U~^T K^T (M 128, N 128, K 64)."""
    terms = 3 if split else 1
    nch = -(-w.n_tokens // 64)
    mm = lambda m, n, k: 2 * m * n * k  # noqa: E731
    gram = mm(128, 64, 128)
    if bf16_in and two_pass:
        per_head = 2 * mm(128, 128, 128) + 3 * mm(128, 64, 64) + 3 * mm(128, 64, 64) + 2 * mm(128, 128, 64)
        return nch * w.n_seqs * (w.n_v_heads * per_head + w.n_k_heads * gram)
    if bf16_in and not two_pass:
        per_head = gram + 2 * mm(128, 64, 64) + 2 * mm(128, 64, 128) + 3 * mm(128, 64, 64) \
            + 2 * mm(128, 64, 128) + 3 * mm(128, 64, 64) + 3 * mm(128, 128, 64)
        return nch * w.n_seqs * w.n_v_heads * per_head
    if two_pass:
        per_head = mm(128, 128, 128) + 2 * mm(128, 64, 64) + mm(128, 128, 64)
        return terms * nch * w.n_seqs * (w.n_v_heads * per_head + w.n_k_heads * gram)
    per_head = gram + mm(128, 64, 64) + mm(128, 64, 128) + mm(128, 64, 64) + mm(128, 64, 128) \
        + mm(128, 64, 64) + mm(128, 128, 64)
    return terms * nch * w.n_seqs * w.n_v_heads * per_head


def scan_executed_flops(w) -> int:
    """Flops the FP32 scan executes per call: with the state kept as c * S~
    (lazy decay) every state cell takes 3 FMAs per token (S~ k, the rank-1
    update, S~ q) = 6 flops; the decay multiply of the method's 7 is folded
    into per-token scalars."""
    return 6 * w.d_k * w.d_v * w.n_v_heads * w.n_seqs * w.n_tokens


def prefill_roofline(kind: str, w, seconds: float, peaks: dict, peak_kind: str, clk: dict | None,
                     act: str = "f32") -> dict:
    """Compute roofline of one prefill call.  ``kind``: "scan" (FP32 CUDA
    cores), "chunked" (one-pass) or "chunked_two_pass" (tensor cores,
    split-bf16 operands), each chunked kind with "_tf32" for TF32 operands."""
    mhz = (clk or {}).get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    mhz_src = "median SM clock sampled in the timed region" if (clk or {}).get("sm_mhz") \
        else "maximum SM clock (no clock samples)"
    hbm = float(peaks["hbm_gbs"])
    bytes_ = w.algorithmic_bytes(act)
    out = {"unit": "TFLOP/s"}
    if kind == "scan":
        peak = SM_COUNT * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
        ex = scan_executed_flops(w)
        out.update(bound="alu", achieved=round(ex / seconds / 1e12, 2), peak=round(peak, 1),
                   peak_kind=f"derived: {SM_COUNT} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 flop "
                             f"(FMA) x {mhz:.0f} MHz ({mhz_src})",
                   flops_per_call=ex, flops_counted="executed: 3 FMAs per state cell per token")
        traffic_key = "scan" + ("_bf16" if act == "bf16" else "")
    else:
        tf32 = kind.endswith("_tf32")
        two = kind.startswith("chunked_two_pass")
        src = "bf16_tflops, MEASURED_PEAKS.json" if peak_kind == "measured" else "recipe fallback"
        ex = chunked_mma_flops(w, two, split=not tf32, bf16_in=act == "bf16")
        if tf32:
            peak = float(peaks["bf16_tflops"]) * 0.5
            out.update(peak_kind=f"of {peak_kind}: bf16 dense tensor peak ({src}) x 1/2, the nominal "
                                 "tf32:bf16 rate ratio",
                       flops_counted="tcgen05 kind::tf32 MMA flops issued per call")
        else:
            peak = float(peaks["bf16_tflops"])
            out.update(peak_kind=f"of {peak_kind}: bf16 dense tensor peak ({src})",
                       flops_counted="tcgen05 kind::f16 (bf16) MMA flops issued per call: three per "
                                     "product of split operands")
        out.update(bound="tensor", achieved=round(ex / seconds / 1e12, 2), peak=round(peak, 1),
                   flops_per_call=ex)
        traffic_key = ("chunked_split" if two else "chunked") + ("_tf32" if tf32 else "") + \
            ("_bf16" if act == "bf16" else "")
    out["frac"] = round(out["achieved"] / out["peak"], 3)
    out["hbm_achieved_GB_s"] = round(bytes_ / seconds / 1e9, 1)
    out["hbm_frac"] = round(bytes_ / seconds / 1e9 / hbm, 3)
    out["algorithmic_bytes"] = bytes_
    out["traffic"] = kernel_traffic(traffic_key, w.n_tokens)
    out["scope"] = "one C-ABI call (both passes for the two-pass form)"
    return out


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local: int, interval_ms: int = 100):
        self.index = self.smi_id(local)
        self.interval_ms = int(interval_ms)
        self.proc = None
        self.file = None

    @staticmethod
    def smi_id(local: int) -> str:
        """nvidia-smi ignores CUDA_VISIBLE_DEVICES, so name the GPU by UUID."""
        try:
            import torch
            u = str(torch.cuda.get_device_properties(local).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return str(local)

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 8:
                continue
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
            except ValueError:
                continue
            for n, v in zip(names, r[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (each rank's elapsed time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: float, elapsed_s: float, world: int, device=None):
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    t = max_over_ranks(elapsed_s, world, device)
    return per_rank_units * world / t, t


# ---------------------------------------------------------------- our arm

def make_sets(torch, w, n_sets, device, capture=False, act="f32"):
    from serving_gdn_decode_gb300.workloads import make_inputs
    sets = []
    adt = torch.bfloat16 if act == "bf16" else torch.float32
    for i in range(n_sets):
        x = make_inputs(w, seed=i, act=act)
        d = {k: torch.from_numpy(v).to(device) for k, v in x.items()}
        for k in ("q", "k", "v"):
            d[k] = d[k].to(adt)
        d["output"] = torch.empty(w.v_elems, dtype=adt, device=device)
        d["state"] = d.pop("state_in")  # updated in place
        if capture:
            d["capture"] = torch.empty(w.capture_elems, dtype=torch.float32, device=device)
        sets.append(d)
    return sets


def call(nat, d, params, capture):
    if "ws" in d:
        nat.gdn_forward_ws(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"], d["output"],
                           d["state"], params, d["ws"])
    elif capture:
        nat.gdn_forward_capture(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"], d["output"],
                                d["state"], params, d["capture"])
    else:
        nat.gdn_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"], d["output"],
                        d["state"], params)


def time_graphed(torch, nat, sets, params, steps, warmup, capture=False, world=1, clocks=None):
    """Exactly `steps` calls (rotating over `sets`) from CUDA graphs; returns
    (elapsed seconds on the device, max over ranks)."""
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(warmup):
            call(nat, sets[i % len(sets)], params, capture)
    torch.cuda.synchronize()
    chunk = max(1, min(steps, 64 * len(sets)))
    graphs = []

    def graph_of(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                call(nat, sets[i % len(sets)], params, capture)
        return g

    full, rest = divmod(steps, chunk)
    g_full = graph_of(chunk) if full else None
    g_rest = graph_of(rest) if rest else None
    if g_full is not None:
        graphs += [g_full] * full
    if g_rest is not None:
        graphs.append(g_rest)
    # one untimed replay of each graph (first replay uploads the graph)
    with torch.cuda.stream(stream):
        for g in {id(x): x for x in graphs}.values():
            g.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if clocks is not None:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for g in graphs:
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks is not None else None
    return start.elapsed_time(end) / 1e3, clk


def time_e2e(torch, nat, w, params, steps, device):
    """End to end through the public API from pinned host memory, two ways.

    zero_copy (the reported e2e): every step is one gdn_forward_host call on
    pinned host buffers -- the kernel reads all inputs from host memory and
    writes output and state back to host memory over the CPU-GPU link.
    copy_engines: HostPipeline -- per step, copies of all inputs to device
    buffers, gdn_forward, copies of output and state back, overlapped over 4
    groups of sequences.  Both move the same bytes across the link per step.
    """
    from serving_gdn_decode_gb300.workloads import make_inputs
    x = make_inputs(w, seed=100)
    host = {k: torch.from_numpy(v).pin_memory() for k, v in x.items()}
    out_h = torch.empty(w.v_elems, dtype=torch.float32).pin_memory()
    st_h = torch.empty(w.state_elems, dtype=torch.float32).pin_memory()
    pipe = nat.HostPipeline(params, groups=4, device=device)

    def zero_copy():
        nat.gdn_forward_host(host["q"], host["k"], host["v"], host["g"], host["beta"],
                             host["state_in"], out_h, st_h, params, device=device)

    def copy_engines():
        pipe(host["q"], host["k"], host["v"], host["g"], host["beta"], host["state_in"], out_h,
             st_h)

    res = {}
    for name, step in (("zero_copy", zero_copy), ("copy_engines", copy_engines)):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(steps):
            step()
        end.record()
        torch.cuda.synchronize()
        res[name] = start.elapsed_time(end) / 1e3 / steps
    return res, pipe.h2d_bytes(), pipe.d2h_bytes()


def extras(torch, nat, peaks, peak_kind, device):
    peak_gbs = float(peaks["hbm_gbs"])
    from serving_gdn_decode_gb300.params import PATH_CHUNKED_TF32, PATH_SCAN
    from serving_gdn_decode_gb300.workloads import WORKLOADS
    res = {}

    def hbm_case(key, w, params, capture, n_sets, steps, act="f32"):
        sets = make_sets(torch, w, n_sets, device, capture, act=act)
        t, _ = time_graphed(torch, nat, sets, params, steps, 5, capture)
        us = t / steps * 1e6
        gbs = w.algorithmic_bytes(act) / (t / steps) / 1e9
        res[key] = {"path": nat.gdn_path_name(params, capture), "us_per_call": round(us, 2),
                    "GB_s": round(gbs, 1), "hbm_frac": round(gbs / peak_gbs, 3)}
        del sets
        torch.cuda.empty_cache()

    wg = WORKLOADS["decode_wide_gqa"]
    hbm_case("decode_wide_gqa_mod", wg, wg.params(), False, 3, 60)
    hbm_case("decode_wide_gqa_div", wg, wg.params(khead_div=True), False, 3, 60)
    wc = WORKLOADS["spec_capture"]
    hbm_case("spec_capture_s32", wc, wc.params(), True, 4, 200)
    wc64 = wc.with_(n_seqs=64)
    hbm_case("spec_capture_s64", wc64, wc64.params(), True, 3, 120)
    # bf16 activations (q, k, v, output), f32 state
    wd = WORKLOADS["decode"]
    hbm_case("decode_bf16", wd, wd.params(), False, 4, 400, act="bf16")
    hbm_case("spec_capture_s32_bf16", wc, wc.params(), True, 4, 200, act="bf16")
    # other head sizes, each with the decode workload's 134 MB of state per call
    for key, dk, dv, ns in (("decode_dk64", 64, 64, 256), ("decode_dk32", 32, 32, 1024),
                            ("decode_dk128_dv64", 128, 64, 128)):
        wx = wd.with_(d_k=dk, d_v=dv, n_seqs=ns)
        hbm_case(key, wx, wx.params(), False, 4, 400)

    # speculative-decode rollback commit: gathers one captured state per sequence
    import numpy as np
    sets = make_sets(torch, wc, 3, device, capture=True)
    for d in sets:
        d["idx"] = torch.from_numpy(
            np.random.default_rng(1).integers(0, wc.n_tokens, wc.n_seqs).astype(np.int32)).to(device)
    stream = torch.cuda.Stream()
    steps = 300
    with torch.cuda.stream(stream):
        for i in range(10):
            d = sets[i % 3]
            nat.gdn_commit_capture(d["capture"], d["idx"], d["state"], wc.params())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps):
                d = sets[i % 3]
                nat.gdn_commit_capture(d["capture"], d["idx"], d["state"], wc.params())
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / steps
    nbytes = 2 * wc.state_elems * 4 + wc.n_seqs * 4
    res["commit_capture_s32"] = {"us_per_call": round(t * 1e6, 2), "GB_s": round(nbytes / t / 1e9, 1),
                                 "hbm_frac": round(nbytes / t / 1e9 / peak_gbs, 3)}
    del sets, g
    torch.cuda.empty_cache()

    # 32 linear-attention layers of single-token decode: one launch per layer
    # vs one gdn_forward_layers launch for all of them
    for S in (1, 8):
        res[f"decode_32_layers_s{S}"] = layers_case(torch, nat, WORKLOADS["decode"].with_(n_seqs=S),
                                                    32, peak_gbs, device)

    # long prefill: each form timed over about 0.3 s so the clock sampler sees
    # the load; inputs (1.1 GB) are larger than L2
    wp = WORKLOADS["long_prefill"]
    for key, params, act, kind, steps in (
            ("long_prefill_auto", wp.params(), "f32", None, 300),
            ("long_prefill_auto_ws", wp.params(), "ws", None, 400),
            ("long_prefill_scan", wp.params(path=PATH_SCAN), "f32", "scan", 100),
            ("long_prefill_chunked_tf32", wp.params(path=PATH_CHUNKED_TF32), "f32", "chunked_tf32", 300),
            ("long_prefill_chunked_two_pass_tf32", wp.params(path=PATH_CHUNKED_TF32), "ws",
             "chunked_two_pass_tf32", 500),
            ("long_prefill_auto_bf16", wp.params(), "bf16", None, 300),
            ("long_prefill_auto_ws_bf16", wp.params(), "ws_bf16", None, 400),
            ("long_prefill_scan_bf16", wp.params(path=PATH_SCAN), "bf16", "scan", 100)):
        ws = act.startswith("ws")
        act = {"ws": "f32", "ws_bf16": "bf16"}.get(act, act)
        sets = make_sets(torch, wp, 1, device, act=act)
        if ws:
            sets[0]["ws"] = torch.empty(nat.gdn_workspace_size(params), dtype=torch.uint8,
                                        device=device)
        path = nat.gdn_path_name(params)
        if kind is None:
            kind = "scan" if path.startswith("scan") else "chunked_two_pass" if ws else "chunked"
        clocks = ClockSampler(device.index or 0, interval_ms=50)
        t, clk = time_graphed(torch, nat, sets, params, steps, 3, clocks=clocks)
        s = t / steps
        res[key] = {"path": path + (" (two-pass, gdn_forward_ws)" if ws else ""),
                    "ms_per_call": round(s * 1e3, 3),
                    "tokens_per_s": round(wp.n_tokens * wp.n_seqs / s, 1),
                    "head_tokens_per_s": round(wp.n_tokens * wp.n_seqs * wp.n_v_heads / s, 1),
                    "method_tflops_equiv": round(wp.flops() / s / 1e12, 2),
                    "method_tflops_note": "7 flops per state cell per token of the sequential "
                                          "recurrence / time: an equivalent rate, not work done",
                    "roofline": prefill_roofline(kind, wp, s, peaks, peak_kind, clk,
                                                 act="bf16" if act == "bf16" else "f32"),
                    "clocks": clk}
        del sets
        torch.cuda.empty_cache()
    return res


def layers_case(torch, nat, w, n_layers, peak_gbs, device):
    params = w.params()
    n_sets = max(2, int(np.ceil(4 * 130e6 / (w.algorithmic_bytes() * n_layers))))
    sets = []
    for i in range(n_sets):
        layers = []
        for l in range(n_layers):
            x = make_small_inputs(w, 1000 * i + l)
            d = {k: torch.from_numpy(v).to(device) for k, v in x.items()}
            d["output"] = torch.empty(w.v_elems, dtype=torch.float32, device=device)
            d["state_out"] = d["state_in"]
            layers.append(d)
        sets.append(layers)
    stream = torch.cuda.Stream()

    def per_layer(layers):
        for d in layers:
            nat.gdn_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state_in"], d["output"],
                            d["state_out"], params)

    def batched(layers):
        nat.gdn_forward_layers(layers, params)

    out = {}
    for name, fn in (("per_layer_launches", per_layer), ("one_launch", batched)):
        with torch.cuda.stream(stream):
            for layers in sets:
                fn(layers)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for layers in sets:
                    fn(layers)
            g.replay()
        torch.cuda.synchronize()
        reps = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / (reps * n_sets)   # one forward = all layers of one set
        gbs = w.algorithmic_bytes() * n_layers / t / 1e9
        out[name] = {"us_per_forward": round(t * 1e6, 2), "GB_s": round(gbs, 1),
                     "hbm_frac": round(gbs / peak_gbs, 3)}
    del sets
    torch.cuda.empty_cache()
    return out


def make_small_inputs(w, seed):
    from serving_gdn_decode_gb300.workloads import make_inputs
    return make_inputs(w, seed)


def cpu_baseline(w, budget_s=2.0):
    """The oracle as it stands, on all host cores, over whole decode calls."""
    import oracle
    from serving_gdn_decode_gb300.workloads import make_inputs
    x = make_inputs(w, seed=0)
    p = w.params()
    cores = oracle.default_threads()
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.forward(p, **x, n_threads=cores)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    per = el / n
    return {"value": round(w.algorithmic_bytes() / per / 1e9, 3), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{n} whole decode call(s) of the oracle (all {w.heads} heads), "
                      f"{per * 1e3:.1f} ms each"}


def run_ours(args):
    import torch

    from serving_gdn_decode_gb300 import _native as nat
    from serving_gdn_decode_gb300 import build as native_build
    from serving_gdn_decode_gb300.workloads import WORKLOADS

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    native_build.build()
    nat.lib()
    peaks, peak_kind = load_peaks()
    peak_gbs = float(peaks["hbm_gbs"])

    w = WORKLOADS["decode"]
    params = w.params()
    kernel = nat.gdn_path_name(params)
    sets = make_sets(torch, w, N_SETS, device)
    clocks = ClockSampler(local)
    elapsed, clk = time_graphed(torch, nat, sets, params, args.steps, args.warmup, world=world,
                                clocks=clocks)
    bytes_per_call = w.algorithmic_bytes()
    value_bps, t_max = aggregate(bytes_per_call * args.steps, elapsed, world, device)
    per_call_s = elapsed / args.steps
    achieved = bytes_per_call / per_call_s / 1e9
    del sets
    torch.cuda.empty_cache()

    e2e_t, h2d, d2h = time_e2e(torch, nat, w, params, min(args.steps, 30), device)
    e2e_s = e2e_t["zero_copy"]
    e2e_val, _ = aggregate(bytes_per_call, e2e_s, world, device)

    line = {
        "metric": METRIC,
        "value": round(value_bps / 1e9, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max / args.steps * 1e3, 5),
        "us_per_call": round(per_call_s * 1e6, 2),
        "hbm_frac_of_8TBs": round(achieved / 8000.0, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded: q,k ~N(0,1) L2-normalised, v ~N(0,1), g ~U[0,0.5), "
                "beta ~U[0,1), state ~N(0,0.1))",
        "config": {"workload": WORKLOAD_TEXT, "kernel": kernel,
                   "l2": f"{N_SETS} rotating input/state sets, "
                         f"{N_SETS * bytes_per_call / 1e9:.2f} GB touched between reuses",
                   "timing": "CUDA graphs of C-ABI calls, CUDA events on the launching stream",
                   "parallelism": f"replicas: each of {world} rank(s) runs the whole workload"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak_gbs,
                     "unit": "GB/s", "frac": round(achieved / peak_gbs, 3),
                     "peak_kind": f"of {peak_kind} ({'hbm_gbs, MEASURED_PEAKS.json' if peak_kind == 'measured' else 'recipe fallback'})",
                     "bytes_per_launch": bytes_per_call,
                     "traffic": kernel_traffic(kernel)},
        "e2e": {"value": round(e2e_val / 1e9, 2), "unit": "GB/s",
                "us_per_call": round(e2e_s * 1e6, 1), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "gdn_forward_host (zero-copy): per step one C-ABI call on pinned host "
                       "buffers; the kernel reads every input from host memory and writes output "
                       "and state to host memory over the CPU-GPU link",
                "copy_engines": {"value": round(bytes_per_call / e2e_t["copy_engines"] / 1e9, 2),
                                 "us_per_call": round(e2e_t["copy_engines"] * 1e6, 1),
                                 "how": "HostPipeline: copies of all inputs in and of output and "
                                        "state out around gdn_forward, overlapped over 4 groups "
                                        "of sequences"}},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if not args.no_extras and rank == 0:
        line["other_workloads"] = extras(torch, nat, peaks, peak_kind, device)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from serving_gdn_decode_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS["decode"]
    x = make_inputs(w, seed=0)
    p = w.params()
    cores = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.forward_heads(p, **x, heads=np.arange(w.heads, dtype=np.uint32), n_threads=cores)
    t_full = time.perf_counter() - t0
    budget = 90.0 / max(1, args.steps + args.warmup)
    n_heads = int(max(1, min(w.heads, w.heads * budget / max(t_full, 1e-6))))
    heads = [np.arange(i * n_heads, (i + 1) * n_heads) % w.heads for i in range(4)]
    for i in range(args.warmup):
        oracle.forward_heads(p, **x, heads=heads[i % 4], n_threads=cores)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.forward_heads(p, **x, heads=heads[i % 4], n_threads=cores)
    el = time.perf_counter() - t0
    bytes_per_step = w.algorithmic_bytes() * n_heads / w.heads
    value = bytes_per_step * args.steps / el / 1e9
    sample = (f"{n_heads} of {w.heads} (seq, value-head) pairs of the decode workload per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT, "kernel": "CPU oracle (double precision)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
