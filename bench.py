#!/usr/bin/env python
"""Benchmark of ReplaySSM ring spec-verify for one Gated DeltaNet layer.

Metric: verified tokens/s per GDN layer, and the verify kernel's achieved HBM
GB/s against the measured roofline, on one GB300.

Workload (default): the Qwen3-Next-shaped layer (H=16 q/k heads, HV=32 v-heads,
K=V=128, bf16 I/O, fp32 checkpoint, draft window T=4, ring L=64) at B=128 rows
scattered in a 512-slot pool.  State is built by the library itself: 16 prefix
rounds (64 tokens, all accepted) from a zero checkpoint, then 48 rounds with
accept_len ~ U{1..4} so that the slots' ring fill levels spread out.  All inputs
are seeded synthetic tensors (the pages measure on served models and datasets,
which are not available here).

A step is one decode round of the layer: verify (output of the whole draft
window, ring side channel) -> commit(accept_len) -> fold (exact, only slots whose
is_flush is set; cursors move after).  Steps are captured in CUDA graphs and
timed with CUDA events; timing events inside the graph bracket every tenth
verify (an event node between kernels costs the step a few microseconds), so
the verify kernel's own duration is measured in the timed region.  The
checkpoint working set (B x 32 x 64 KiB = 256 MiB at B=128) exceeds L2.

--impl reference times the fp64 CPU oracle (the reference arm: the oracle
itself on the host cores) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tokens/s per GDN layer and achieved HBM GB/s vs roofline, 1×GB300"
UNIT = "tokens/s"


# ----------------------------------------------------------------- accounting

def verify_bytes_per_unit(W: np.ndarray, K: int, V: int, T: int, G: int, e: int,
                          per_key: bool) -> np.ndarray:
    """Algorithmic HBM bytes one verify must move per (row, v-head) unit with W
    committed-but-unfolded ring records: checkpoint read, history records,
    window inputs, outputs and the ring write of the window."""
    gbytes = 4 * K if per_key else 4
    rec = V * e + K * e / G + gbytes + 4                  # rawv + rawk share + g + beta
    win_in = 2 * K * e / G + V * e + (K * e if per_key else e) + e   # q, k share, v, a, b
    return V * K * 4 + W * rec + T * win_in + T * V * e + T * rec


def verify_d_bytes_per_unit(W: np.ndarray, K: int, V: int, T: int, G: int, e: int) -> np.ndarray:
    """Algorithmic HBM bytes of one derived-d verify per (row, v-head) unit:
    checkpoint read, history records (fp32 d, raw k share, g, beta), window
    inputs, outputs, the window's raw records and its fp32 d written."""
    hist = V * 4 + K * e / G + 8
    win_in = 2 * K * e / G + V * e + 2 * e
    rec = V * e + K * e / G + 8
    return V * K * 4 + W * hist + T * win_in + T * V * e + T * (rec + V * 4)


def mirror_cursors(wp, base, acc_rows, T, L):
    """Host copy of the cursor arithmetic (commit then fold), used only to know
    each verify's ring fill W for byte accounting.  Returns W per step [steps, B]."""
    wp = wp.astype(np.int64).copy()
    out = []
    for acc in acc_rows:
        out.append(wp.copy())
        wp = wp + acc
        flush = wp + 2 * T > L
        wp[flush] = 0
    return np.array(out)


def kernel_source_hash(path_name: str = "tc") -> str:
    """Hash of the sources of one verify path (its kernel file and the headers
    it includes), which keys the committed ncu traffic record."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_spec_gb300", "csrc")
    src = {"tc_kda": "verify_kda.cu"}.get(path_name, f"verify_{path_name}.cu")
    for name in (src, "common.cuh", "ptx_sm100.cuh"):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


# Arithmetic of each path (the JSON line's "dtype" is the arithmetic type; bf16 is
# only the type of the inputs and outputs).
ARITH = {
    "tc": "fp32; the Gram and the checkpoint product on tensor cores with tf32 operands "
          "and fp32 accumulation",
    "generic": "fp32 on CUDA cores",
    "tc_kda": "fp32; the per-channel-decayed key products off the diagonal blocks and the "
              "checkpoint product on tensor cores with tf32 operands and fp32 accumulation; "
              "the diagonal blocks and the solve on CUDA cores",
    "chunk": "fp32; the chunk's Gram (bf16 operands), the state products and the update (tf32 "
             "operands, the update split into high and low parts) on tensor cores with fp32 "
             "accumulation; the triangular solve on CUDA cores",
}
# tf32 dense tensor peak as a fraction of the bf16 one (nominal 1.1 / 2.25 PFLOP/s)
TF32_OVER_BF16 = 1.1 / 2.25


def profiled_traffic(path_name: str, B: int, T: int, algorithmic_bytes: float):
    """DRAM bytes per verify launch from the committed ncu record, if it was
    taken on the current verify source and the same window; else None.  The
    record holds DRAM bytes over algorithmic bytes of the profiled launches;
    that ratio times this run's algorithmic bytes is the per-launch figure
    (traffic grows with the units and the ring fill as the bytes do)."""
    f = os.path.join(ROOT, "profiles", f"verify_{path_name}_traffic.json")
    if not os.path.exists(f):
        return None
    try:
        rec = json.load(open(f))
    except Exception:
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash(path_name) or rec.get("T") != T:
        return None
    ratio = rec.get("dram_over_algorithmic")
    if ratio is None:
        return None
    return round(float(ratio) * algorithmic_bytes)


def measured_peaks():
    f = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(f):
        return json.load(open(f)), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (stamped on arrival) of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return None
        rows = [s for t, s in self.samples if t0 <= t <= t1]
        if not rows:  # short region: take the nearest samples around it
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))
            rows = [s for _, s in near[:3]]
        if not rows:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": num(rows[0][1]),
                "power_w_max": max(num(r[2]) for r in rows), "samples": len(rows),
                "reasons": reasons}


# ----------------------------------------------------------------- our arm

class Workload:
    def __init__(self, B: int, T: int | None = None, kda: bool = False):
        """The Qwen3-Next-shaped layer at B rows; T = 1 is plain decode (a window
        of one token through the same calls, checkpoint, ring and cursors); kda:
        one gate per key channel (the KDA variant) on the same shape."""
        from gated_delta_rule_spec_gb300 import inputs as gen
        c = gen.WORKLOADS["C2"]
        T = c.T if T is None else T
        self.kda = kda
        self.name = f"qwen3next-{'kda' if kda else 'gdn'}-{'decode' if T == 1 else 'verify'}-b{B}" + (
            f"-t{T}" if T not in (1, c.T) else "")
        self.B, self.H, self.HV, self.K, self.V, self.T, self.L = B, c.H, c.HV, c.K, c.V, T, c.L
        self.num_slots = max(c.num_slots, B)
        self.G = self.HV // self.H
        self.e = 2

    def config(self, extra=None):
        d = {"workload": self.name, "model_layer": "Qwen3-Next-shaped GDN layer",
             "B": self.B, "H": self.H, "HV": self.HV, "K": self.K, "V": self.V, "T": self.T,
             "L": self.L, "num_slots": self.num_slots, "io_dtype": "bf16",
             "state_dtype": "fp32", "step": "verify+commit+fold",
             "l2": "inputs larger than L2 (checkpoint working set "
                   f"{self.B * self.HV * self.V * self.K * 4 >> 20} MiB per step)",
             "parallelism": "replicas"}
        if extra:
            d.update(extra)
        return d


def build_state(wl: Workload, seed: int, device, random_rounds: int = 48, dring=None):
    """Layer state built by the library's own rounds from a zero checkpoint:
    16 full-accept rounds, then random_rounds with accept_len ~ U{1..T}.  During
    the random rounds each row first sits out a random number of rounds (accept
    0), drawn from [0, one fold cycle] (a cycle is about (L - 2T) / E[accept_len]
    rounds), so that the rows' ring fill levels and fold times spread out as in
    a serving batch instead of moving in lockstep.  With a d ring the rounds
    verify through gdn_spec_verify_d, which fills it."""
    import torch
    from gated_delta_rule_spec_gb300 import binding
    from gated_delta_rule_spec_gb300 import inputs as gen

    rng = gen.rng_for(seed, "bench", wl.B)
    layer = binding.SpecLayer(wl.H, wl.HV, wl.K, wl.V, wl.T, wl.L, wl.num_slots, per_key_gate=wl.kda,
                              device=device)
    cur = binding.SpecCursors(wl.num_slots, device=device)
    A_log, dt_bias = gen.layer_params(rng, wl.HV, wl.K, wl.kda)
    A_log = torch.from_numpy(A_log).to(device)
    dt_bias = torch.from_numpy(dt_bias).to(device)
    slots = torch.from_numpy(gen.scattered_slots(rng, wl.num_slots, wl.B)).to(device)

    def dev_window():
        w = gen.window_inputs(rng, wl.B, wl.T, wl.H, wl.HV, wl.K, wl.V, gen.BF16, wl.kda)
        return {n: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
                for n, x in w.items()}

    binding.reset(cur, slots)
    full = torch.full((wl.B,), wl.T, dtype=torch.int32, device=device)
    cycle = (wl.L - 2 * wl.T) * 2 // (wl.T + 1) + 2
    pause = rng.integers(0, max(1, cycle), size=wl.B)
    for r in range(16 + random_rounds):
        w = dev_window()
        if dring is None:
            binding.verify(layer, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt_bias)
        else:
            binding.verify_d(layer, dring, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log,
                             dt_bias)
        if r < 16:
            acc = full
        else:
            a_np = gen.accept_lens(rng, wl.B, wl.T)
            a_np[pause > r - 16] = 0
            acc = torch.from_numpy(a_np).to(device)
        binding.commit(cur, wl.T, wl.L, slots, acc)
        binding.fold(layer, cur, slots)
    torch.cuda.synchronize()
    return rng, layer, cur, A_log, dt_bias, slots, dev_window


def run_ours(args, rank: int, world: int) -> dict | None:
    import torch
    import torch.distributed as dist
    from gated_delta_rule_spec_gb300 import binding
    from gated_delta_rule_spec_gb300 import inputs as gen

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    binding.load()
    wl = Workload(args.batch, args.window, args.kda)
    rng, layer, cur, A_log, dt_bias, slots, dev_window = build_state(wl, 1000 + rank, device,
                                                                     args.setup_rounds)
    path = binding.verify_path(layer)

    NI = 16
    R = max(1, min(args.steps, 200))
    inputs = [dev_window() for _ in range(NI)]
    acc_np = np.stack([gen.accept_lens(rng, wl.B, wl.T) for _ in range(R)])
    acc_dev = torch.from_numpy(acc_np).to(device)
    # events bracket every EV_EVERY-th verify of the timed graph: an event node
    # between kernels costs the step several microseconds, so sample
    EV_EVERY = 10 if R >= 20 else 1
    ev_steps = list(range(0, R, EV_EVERY))
    try:
        ev = {i: (torch.cuda.Event(enable_timing=True, external=True),
                  torch.cuda.Event(enable_timing=True, external=True)) for i in ev_steps}
    except TypeError:  # torch without external events: time verify in its own graph below
        ev = None

    def step(i, timed_events=True):
        w = inputs[i % NI]
        timed = timed_events and ev is not None and i in ev
        if timed:
            ev[i][0].record()
        binding.verify(layer, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt_bias,
                       out=outs[i % NI])
        if timed:
            ev[i][1].record()
        binding.commit(cur, wl.T, wl.L, slots, acc_dev[i % R])
        binding.fold(layer, cur, slots)

    outs = [torch.empty(wl.B, wl.T, wl.HV, wl.V, dtype=torch.bfloat16, device=device)
            for _ in range(NI)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graphs = {}
    with torch.cuda.stream(side):
        for name, n in (("warm", args.warmup), ("chunk", R), ("rem", args.steps % R)):
            if n == 0:
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    step(i, timed_events=(name == "chunk"))
            graphs[name] = g
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    # the capture ran nothing; cursors are as build_state left them
    if "warm" in graphs:
        graphs["warm"].replay()
    torch.cuda.synchronize()
    wp0 = cur.write_pos[slots.long()].cpu().numpy()

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_start.record()
    for _ in range(args.steps // R):
        graphs["chunk"].replay()
    if "rem" in graphs:
        graphs["rem"].replay()
    t_end.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        dist.barrier()
    ms = t_start.elapsed_time(t_end)
    # per-verify durations sampled inside the timed region (every EV_EVERY-th step
    # of the last chunk replay): a cross-check of the verify-only graph below
    verify_ms_in_step = []
    if args.steps // R > 0 and ev is not None:
        try:
            verify_ms_in_step = [ev[i][0].elapsed_time(ev[i][1]) for i in ev_steps]
        except RuntimeError:
            verify_ms_in_step = []
    clocks = sampler.summary(wall0, wall1) if sampler else None
    if sampler:
        sampler.stop()
    status = binding.read_status(cur)
    # the verify kernel on its own: median over 10 replays of a graph of 20
    # back-to-back verify calls on the state the timed steps left (inputs rotate
    # over 16 windows; the 256 MiB checkpoint working set is larger than L2)
    W_now = cur.write_pos[slots.long()].cpu().numpy().astype(np.int64)
    verify_graph_ms, verify_graph_all = verify_only_times(binding, layer, cur, slots, inputs, outs,
                                                          A_log, dt_bias, n=20, reps=10)
    graph_bytes = float(verify_bytes_per_unit(W_now, wl.K, wl.V, wl.T, wl.G, wl.e, wl.kda).sum()
                        * wl.HV)
    status |= binding.read_status(cur)

    # byte accounting for the verifies of the last chunk replay
    acc_seq = np.array([acc_np[i % R] for i in range(args.warmup)]
                       + [acc_np[i % R] for i in range(R)] * (args.steps // R)
                       + [acc_np[i % R] for i in range(args.steps % R)])
    # W per step from the cursors read before the timed region (after warm-up)
    W_all = mirror_cursors(wp0, None, acc_seq[args.warmup:], wl.T, wl.L)
    last = slice((args.steps // R - 1) * R, (args.steps // R) * R)
    W_last = W_all[last] if args.steps // R > 0 else W_all
    if args.steps // R > 0 and ev is not None:   # the verifies the events bracketed
        W_last = W_last[ev_steps]
    bytes_in_step = float(np.mean([
        verify_bytes_per_unit(Wr, wl.K, wl.V, wl.T, wl.G, wl.e, wl.kda).sum() * wl.HV
        for Wr in W_last]))
    mean_W = float(W_now.mean())
    # committed tokens of the timed steps (sum of accept_len over rows)
    committed = float(acc_seq[args.warmup:].sum()) * world

    # e2e through the binding with host buffers: every step copies its inputs
    # (q, k, v, a, b and accept_len, packed in one pinned buffer) to the device
    # and its output back.  The transfers overlap the previous and next steps'
    # kernels as in a serving loop: H2D one step ahead on a copy stream, D2H on
    # another, device buffers doubled, events ordering every reuse.
    names = ["q", "k", "v", "a", "b"]
    shapes = {n: inputs[0][n].shape for n in names}
    dtypes = {n: inputs[0][n].dtype for n in names}
    offs, off = {}, 0
    for n in names:
        offs[n] = off
        off += (inputs[0][n].numel() * inputs[0][n].element_size() + 255) // 256 * 256
    offs["acc"] = off
    flat_bytes = off + wl.B * 4

    def views(flat):
        vw = {n: flat[offs[n]:offs[n] + inputs[0][n].numel() * inputs[0][n].element_size()]
              .view(dtypes[n]).view(shapes[n]) for n in names}
        vw["acc"] = flat[offs["acc"]:offs["acc"] + wl.B * 4].view(torch.int32)
        return vw

    host_flat = [torch.empty(flat_bytes, dtype=torch.uint8).pin_memory() for _ in range(4)]
    for i in range(4):
        hv_ = views(host_flat[i])
        for n in names:
            hv_[n].copy_(inputs[i][n].cpu())
        hv_["acc"].copy_(torch.from_numpy(acc_np[i % R]))
    dev_flat = [torch.empty(flat_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
    dev_v = [views(f) for f in dev_flat]
    dev_out = [torch.empty(wl.B, wl.T, wl.HV, wl.V, dtype=torch.bfloat16, device=device) for _ in range(2)]
    host_out = [torch.empty(wl.B, wl.T, wl.HV, wl.V, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = flat_bytes
    d2h = host_out[0].numel() * host_out[0].element_size()
    K_e2e = max(3, min(args.steps, 200))
    comp = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]   # a step's inputs consumed
    ev_out = [torch.cuda.Event() for _ in range(2)]    # a step's output written
    ev_read = [torch.cuda.Event() for _ in range(2)]   # a step's output copied out

    def upload(i):
        buf = i % 2
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(ev_free[buf])
            dev_flat[buf].copy_(host_flat[i % 4], non_blocking=True)
            ev_in[buf].record(h2d_s)

    def run_e2e(n_steps):
        upload(0)
        for i in range(n_steps):
            if i + 1 < n_steps:
                upload(i + 1)
            buf = i % 2
            d = dev_v[buf]
            comp.wait_event(ev_in[buf])
            comp.wait_event(ev_read[buf])
            binding.verify(layer, cur, slots, d["q"], d["k"], d["v"], d["a"], d["b"], A_log, dt_bias,
                           out=dev_out[buf])
            binding.commit(cur, wl.T, wl.L, slots, d["acc"])
            ev_free[buf].record(comp)
            binding.fold(layer, cur, slots)
            ev_out[buf].record(comp)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_out[buf])
                host_out[buf].copy_(dev_out[buf], non_blocking=True)
                ev_read[buf].record(d2h_s)
        comp.wait_stream(d2h_s)

    run_e2e(3)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    run_e2e(K_e2e)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    if world > 1:
        ms, e2e_ms = reduce_max([ms, e2e_ms], device)
    if rank != 0:
        return None

    tokens = world * wl.B * wl.T * args.steps
    value = tokens / (ms / 1e3)
    peaks, peak_kind = measured_peaks()
    v_ms = verify_graph_ms
    achieved = graph_bytes / (v_ms / 1e3) / 1e9
    v_step_ms = float(np.mean(verify_ms_in_step)) if verify_ms_in_step else None
    traffic = profiled_traffic(path, wl.B, wl.T, graph_bytes)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; Qwen3-Next-shaped GDN layer, random weights)",
        "config": wl.config({"verify_kernel": path, "arith": ARITH[path],
                             "mean_ring_fill_W": round(mean_W, 2)}),
        "us_per_round": round(ms / args.steps * 1e3, 2),
        "committed_tokens_per_s": round(committed / (ms / 1e3), 1),
        "e2e": {"value": round(world * wl.B * wl.T * K_e2e / (e2e_ms / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "steps": K_e2e,
                "api": "python binding -> C ABI, host pinned buffers; transfers overlap the "
                       "neighbouring steps' kernels (copy streams, double buffers)"},
        "gpu_launches": 4 * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": round(graph_bytes),
                     "kernel": f"verify ({path})", "peak_kind": peak_kind,
                     "verify_us": round(v_ms * 1e3, 2),
                     "verify_timing": "median of 10 replays of a CUDA graph of 20 back-to-back "
                                      "verify calls, after the timed steps",
                     "verify_us_replays": [round(x * 1e3, 2) for x in verify_graph_all],
                     "verify_us_in_step": (round(v_step_ms * 1e3, 2) if v_step_ms else None),
                     "algorithmic_bytes_per_launch_in_step": round(bytes_in_step)},
        "verify_tokens_per_s": round(wl.B * wl.T / (v_ms / 1e3), 1),
        "device_status": status,
        "clocks": clocks,
    }
    return line


def run_verify_only(args) -> dict:
    """Profiling aid: the bench's state, then --steps plain verify calls (no
    commit, so every call sees the same ring fill) and nothing else; prints the
    algorithmic bytes of one call, so that DRAM counters taken on these launches
    can be set against them."""
    import torch
    from gated_delta_rule_spec_gb300 import binding

    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    binding.load()
    wl = Workload(args.batch, args.window, args.kda)
    rng, layer, cur, A_log, dt_bias, slots, dev_window = build_state(wl, 1000, device,
                                                                     args.setup_rounds)
    inputs = [dev_window() for _ in range(4)]
    out = torch.empty(wl.B, wl.T, wl.HV, wl.V, dtype=torch.bfloat16, device=device)
    W = cur.write_pos[slots.long()].cpu().numpy().astype(np.int64)
    for i in range(args.steps):
        w = inputs[i % 4]
        binding.verify(layer, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt_bias,
                       out=out)
    torch.cuda.synchronize()
    byts = float(verify_bytes_per_unit(W, wl.K, wl.V, wl.T, wl.G, wl.e, wl.kda).sum() * wl.HV)
    return {"mode": "verify-only", "workload": wl.name, "verify_kernel": binding.verify_path(layer),
            "calls": args.steps, "setup_verify_calls": 16 + args.setup_rounds,
            "algorithmic_bytes_per_launch": round(byts), "mean_ring_fill_W": round(float(W.mean()), 2),
            "device_status": binding.read_status(cur)}


def reduce_max(values, device="cpu"):
    """Max over ranks of each value (the job time is the slowest rank's)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def verify_only_times(binding, layer, cur, slots, inputs, outs, A_log, dt_bias, n=20, reps=10):
    """Per-call time (ms) of a graph of n back-to-back verify calls: (median over
    reps replays, every replay's value)."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(n):
                w = inputs[i % len(inputs)]
                binding.verify(layer, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log,
                               dt_bias, out=outs[i % len(outs)])
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / n)
    return statistics.median(times), times


def cpu_baseline(B: int, seconds: float = 10.0, T: int | None = None, kda: bool = False,
                 single_thread_seconds: float = 4.0) -> dict:
    """The fp64 oracle, as it stands, on the host cores: verify of a sample of
    the workload's rows (all heads), ring fill W ~ U[0, L-2T] as in the sweep;
    then the same on one thread."""
    import oracle
    from gated_delta_rule_spec_gb300 import inputs as gen

    c = gen.WORKLOADS["C2"]
    if T is not None and T != c.T:
        c = dataclasses.replace(c, T=T)
    rows = min(B, 16)
    rng = gen.rng_for(7, "cpu-baseline", rows)
    d = oracle.Dims(H=c.H, HV=c.HV, K=c.K, V=c.V, T=c.T, L=c.L, num_slots=rows, per_key_gate=kda)
    ring = gen.garbage_ring(rng, rows, c.H, c.HV, c.L, c.K, c.V, gen.BF16, kda)
    ly = oracle.Layer(d, checkpoint=rng.standard_normal((rows, c.HV, c.V, c.K)) * 0.1,
                      rawv=gen.to_f64(ring["rawv"]), rawk=gen.to_f64(ring["rawk"]),
                      ring_g=-np.abs(ring["g"].astype(np.float64)),
                      ring_beta=np.abs(ring["beta"].astype(np.float64)) % 1.0)
    wp, base, flag = gen.random_cursors(rng, rows, c.L, c.T)
    cur = oracle.Cursors(rows, wp, base, flag)
    A_log, dt = gen.layer_params(rng, c.HV, c.K, kda)
    w = {n: gen.to_f64(x) for n, x in
         gen.window_inputs(rng, rows, c.T, c.H, c.HV, c.K, c.V, gen.BF16, kda).items()}
    cores = os.cpu_count() or 1
    slot_idx = np.arange(rows, dtype=np.int32)

    def timed(nthreads, secs, rows_used):
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle.verify(d, ly, cur, slot_idx[:rows_used], w["q"][:rows_used], w["k"][:rows_used],
                          w["v"][:rows_used], w["a"][:rows_used], w["b"][:rows_used], A_log, dt,
                          nthreads=nthreads)
            reps += 1
            el = time.perf_counter() - t0
            if el >= secs or reps >= 10000:
                return reps, el

    reps, el = timed(cores, seconds, rows)
    reps1, el1 = timed(1, single_thread_seconds, 1)
    return {"value": round(rows * c.T * reps / el, 2), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{rows} rows x {c.HV} v-heads of the B={B} workload, fp64 verify, "
                      f"{reps} repetitions in {el:.1f} s, W ~ U[0, {c.L - 2 * c.T}]",
            "single_thread": {"value": round(c.T * reps1 / el1, 2), "unit": UNIT, "cores": 1,
                              "sample": f"1 row x {c.HV} v-heads, {reps1} repetitions in "
                                        f"{el1:.1f} s"}}


# ----------------------------------------------------------------- snapshot comparison

def snapshot_bytes_per_unit(K: int, V: int, T: int, G: int, e: int) -> float:
    """Algorithmic bytes per (row, v-head) of one snapshot step: the state read,
    T full states written, the window's q, k (shared by G v-heads), v, a, b
    read, the outputs written, and the commit's copy of one state."""
    return V * K * 4 + T * V * K * 4 + T * (2 * K * e / G + V * e + 2 * e) + T * V * e + 2 * V * K * 4


def run_snapshot(args, rank: int, world: int) -> dict | None:
    """The per-draft snapshot design (comparison variant) on the bench's
    workload: a step is snapshot verify (T full states stored) + commit (the
    accepted state copied back), captured in CUDA graphs."""
    import torch
    from gated_delta_rule_spec_gb300 import binding
    from gated_delta_rule_spec_gb300 import inputs as gen

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    binding.load()
    wl = Workload(args.batch, args.window)
    rng = gen.rng_for(4000 + rank, "snapshot", wl.B)
    layer = binding.SpecLayer(wl.H, wl.HV, wl.K, wl.V, wl.T, wl.L, wl.num_slots, device=device)
    layer.checkpoint.normal_(0.0, 0.1)
    cur = binding.SpecCursors(wl.num_slots, device=device)
    A_log, dt_bias = (torch.from_numpy(x).to(device) for x in gen.layer_params(rng, wl.HV, wl.K, False))
    slots = torch.from_numpy(gen.scattered_slots(rng, wl.num_slots, wl.B)).to(device)
    NI = 8
    inputs = [{n: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device) for n, x in
               gen.window_inputs(rng, wl.B, wl.T, wl.H, wl.HV, wl.K, wl.V, gen.BF16).items()}
              for _ in range(NI)]
    accs = [torch.from_numpy(gen.accept_lens(rng, wl.B, wl.T)).to(device) for _ in range(NI)]
    out = torch.empty(wl.B, wl.T, wl.HV, wl.V, dtype=torch.bfloat16, device=device)
    snap = torch.empty(wl.B, wl.T, wl.HV, wl.V, wl.K, dtype=torch.float32, device=device)

    def step(i):
        w = inputs[i % NI]
        binding.snapshot_verify(layer, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log,
                                dt_bias, out=out, snap=snap)
        binding.snapshot_commit(layer, cur, slots, accs[i % NI], snap)

    for i in range(args.warmup):
        step(i)
    R = max(1, min(args.steps, 50))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(R):
                step(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    reps = max(1, (args.steps + R - 1) // R)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    ms = e0.elapsed_time(e1)
    clocks = sampler.summary(wall0, wall1) if sampler else None
    if sampler:
        sampler.stop()
    status = binding.read_status(cur)
    if world > 1:
        ms, = reduce_max([ms], device)
    if rank != 0:
        return None
    steps = reps * R
    t_step = ms / 1e3 / steps
    peaks, peak_kind = measured_peaks()
    byts = snapshot_bytes_per_unit(wl.K, wl.V, wl.T, wl.G, wl.e) * wl.B * wl.HV
    achieved = byts / t_step / 1e9
    return {
        "metric": METRIC, "variant": "snapshot (comparison: per-draft full states, no ring)",
        "value": round(world * wl.B * wl.T / t_step, 1), "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms / steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; Qwen3-Next-shaped GDN layer, random weights)",
        "config": wl.config({"workload": wl.name.replace("-verify-", "-snapshot-verify-"),
                             "arith": ARITH["generic"],
                             "step": "snapshot verify + snapshot commit",
                             "snapshot_bytes": int(snap.numel() * 4)}),
        "gpu_launches": 2 * steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                     "algorithmic_bytes_per_step": round(byts), "kernel": "snapshot verify + commit",
                     "peak_kind": peak_kind},
        # per (row, v-head, draft position): one full fp32 state; the ring path
        # writes one raw record instead (V e + K e / G + 8 bytes)
        "state_bytes_written_per_head_step": wl.V * wl.K * 4,
        "ring_bytes_written_per_head_step": int(wl.V * wl.e + wl.K * wl.e / wl.G + 8),
        "device_status": status,
        "clocks": clocks,
    }

# ----------------------------------------------------------------- derived-d comparison

def run_derived_d(args, rank: int, world: int) -> dict | None:
    """The derived-d ring (comparison variant: the ring also caches each token's
    corrected delta, so verify solves only the window's system; with --window 1
    the no-inverse decode): a step is gdn_spec_verify_d -> commit -> fold,
    captured in CUDA graphs; the verify kernel is timed on its own as the
    median of 10 replays of a graph of 20 calls."""
    import torch
    from gated_delta_rule_spec_gb300 import binding
    from gated_delta_rule_spec_gb300 import inputs as gen

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    binding.load()
    wl = Workload(args.batch, args.window)
    name = wl.name.replace("-gdn-", "-gdn-derived-d-")
    layer0 = binding.SpecLayer(wl.H, wl.HV, wl.K, wl.V, wl.T, wl.L, wl.num_slots, device=device)
    dring = layer0.new_dring()
    del layer0
    rng, layer, cur, A_log, dt_bias, slots, dev_window = build_state(wl, 2000 + rank, device,
                                                                     args.setup_rounds, dring=dring)
    NI = 16
    R = max(1, min(args.steps, 200))
    inputs = [dev_window() for _ in range(NI)]
    outs = [torch.empty(wl.B, wl.T, wl.HV, wl.V, dtype=torch.bfloat16, device=device) for _ in range(NI)]
    acc_dev = torch.from_numpy(np.stack([gen.accept_lens(rng, wl.B, wl.T) for _ in range(R)])).to(device)

    def vd(i):
        w = inputs[i % NI]
        binding.verify_d(layer, dring, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt_bias,
                         out=outs[i % NI])

    def step(i):
        vd(i)
        binding.commit(cur, wl.T, wl.L, slots, acc_dev[i % R])
        binding.fold(layer, cur, slots)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graphs = {}
    with torch.cuda.stream(side):
        for gname, n in (("warm", args.warmup), ("chunk", R), ("rem", args.steps % R)):
            if n == 0:
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    step(i)
            graphs[gname] = g
        gv = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gv, stream=side):
            for i in range(20):
                vd(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    if "warm" in graphs:
        graphs["warm"].replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    e0.record()
    for _ in range(args.steps // R):
        graphs["chunk"].replay()
    if "rem" in graphs:
        graphs["rem"].replay()
    e1.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    ms = e0.elapsed_time(e1)
    clocks = sampler.summary(wall0, wall1) if sampler else None
    if sampler:
        sampler.stop()
    W_now = cur.write_pos[slots.long()].cpu().numpy().astype(np.int64)
    times = []
    for _ in range(10):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record()
        gv.replay()
        b_.record()
        torch.cuda.synchronize()
        times.append(a_.elapsed_time(b_) / 20)
    v_ms = statistics.median(times)
    status = binding.read_status(cur)
    if world > 1:
        ms, = reduce_max([ms], device)
    if rank != 0:
        return None
    byts = float(verify_d_bytes_per_unit(W_now, wl.K, wl.V, wl.T, wl.G, wl.e).sum() * wl.HV)
    peaks, peak_kind = measured_peaks()
    achieved = byts / (v_ms / 1e3) / 1e9
    return {
        "metric": METRIC, "variant": "derived-d (comparison: the ring also caches each token's corrected delta)",
        "value": round(world * wl.B * wl.T * args.steps / (ms / 1e3), 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; Qwen3-Next-shaped GDN layer, random weights)",
        "config": wl.config({"workload": name, "arith": ARITH["tc"],
                             "step": "verify_d + commit + fold", "mean_ring_fill_W": round(float(W_now.mean()), 2),
                             "d_ring_bytes": int(dring.numel() * 4)}),
        "gpu_launches": 4 * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                     "algorithmic_bytes_per_launch": round(byts), "kernel": "verify_d",
                     "peak_kind": peak_kind, "verify_us": round(v_ms * 1e3, 2),
                     "verify_timing": "median of 10 replays of a CUDA graph of 20 verify_d calls",
                     "verify_us_replays": [round(x * 1e3, 2) for x in times]},
        "verify_tokens_per_s": round(wl.B * wl.T / (v_ms / 1e3), 1),
        "device_status": status,
        "clocks": clocks,
    }


# ----------------------------------------------------------------- prefill

PREFILL_METRIC = "prefilled tokens/s per GDN layer, 1\u00d7GB300"


def _prefill_flops(B: int, N: int, wl: "Workload") -> float:
    """Algorithmic flops of one prefill call: per token and v-head the delta
    (S k, 2VK), the rank-1 update (2VK) and the output (S q, 2VK)."""
    return 6.0 * wl.V * wl.K * B * N * wl.HV


def _prefill_chunk_flops(B: int, N: int, wl: "Workload", C: int = 64) -> float:
    """Algorithmic tensor flops of one chunk-parallel prefill call: per (row,
    v-head) and chunk of n tokens the Gram [K; Q] K^T (2 K 2n n), the state
    products S [K; Q]^T (2 V K 2n), the intra-chunk outputs D W^T (2 V n n)
    and the state update D K (2 V K n).  The high/low split of the update is
    not counted."""
    total = 0.0
    for c0 in range(0, N, C):
        n = min(C, N - c0)
        total += 2.0 * wl.K * 2 * n * n + 2.0 * wl.V * wl.K * 2 * n + 2.0 * wl.V * n * n + 2.0 * wl.V * wl.K * n
    return total * B * wl.HV


def run_prefill(args, rank: int, world: int) -> dict | None:
    """gdn_spec_prefill of B prompts of N tokens (from a zero state) on the
    Qwen3-Next-shaped layer, timed in CUDA graphs, plus an end-to-end leg
    (pinned host prompts in, outputs out, every call)."""
    import torch
    from gated_delta_rule_spec_gb300 import binding
    from gated_delta_rule_spec_gb300 import inputs as gen

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    binding.load()
    wl = Workload(args.batch)
    B, N = wl.B, args.prefill
    rng = gen.rng_for(3000 + rank, "prefill", B)
    layer = binding.SpecLayer(wl.H, wl.HV, wl.K, wl.V, wl.T, wl.L, wl.num_slots, device=device)
    cur = binding.SpecCursors(wl.num_slots, device=device)
    A_log, dt_bias = (torch.from_numpy(x).to(device) for x in gen.layer_params(rng, wl.HV, wl.K, False))
    slots = torch.from_numpy(gen.scattered_slots(rng, wl.num_slots, B)).to(device)
    host = gen.window_inputs(rng, B, N, wl.H, wl.HV, wl.K, wl.V, gen.BF16)
    w = {n: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device) for n, x in host.items()}
    out = torch.empty(B, N, wl.HV, wl.V, dtype=torch.bfloat16, device=device)

    def call(ins, o):
        binding.prefill(layer, cur, slots, ins["q"], ins["k"], ins["v"], ins["a"], ins["b"], A_log,
                        dt_bias, out=o, from_zero=True)

    for _ in range(args.warmup):
        call(w, out)
    R = max(1, min(args.steps, 10))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for _ in range(R):
                call(w, out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    reps = max(1, (args.steps + R - 1) // R)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    ms = e0.elapsed_time(e1)
    clocks = sampler.summary(wall0, wall1) if sampler else None
    if sampler:
        sampler.stop()
    calls = reps * R

    # end to end: prompts from pinned host memory in, outputs out, every call
    hin = {n: t.cpu().pin_memory() for n, t in w.items()}
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    din = {n: torch.empty_like(t) for n, t in w.items()}
    K_e2e = max(3, min(args.steps, 20))

    def e2e_call():
        for n in din:
            din[n].copy_(hin[n], non_blocking=True)
        call(din, out)
        hout.copy_(out, non_blocking=True)

    e2e_call()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(K_e2e):
        e2e_call()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if world > 1:
        ms, e2e_ms = reduce_max([ms, e2e_ms], device)
    if rank != 0:
        return None
    t_call = ms / 1e3 / calls
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    peaks, peak_src = measured_peaks()
    path = binding.prefill_path(layer)
    if path == "chunk":
        peak = float(peaks["bf16_tflops"]) * TF32_OVER_BF16
        roofline = {"bound": "tensor", "achieved": round(_prefill_chunk_flops(B, N, wl) / t_call / 1e12, 2),
                    "peak": round(peak, 2), "unit": "TFLOP/s", "traffic": None,
                    "kernel": "prefill_tc_kernel (chunk-parallel)",
                    "peak_kind": f"{peak_src} bf16 dense x nominal tf32/bf16 ratio (1.1/2.25)"}
    else:
        sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
        peak = sms * 128 * 2 * sm_mhz * 1e6 / 1e12    # fp32 FMA lanes x 2 flops x clock, TFLOP/s
        roofline = {"bound": "alu", "achieved": round(_prefill_flops(B, N, wl) / t_call / 1e12, 2),
                    "peak": round(peak, 2), "unit": "TFLOP/s", "traffic": None,
                    "kernel": "prefill_kernel (sequential)",
                    "peak_kind": "derived: SMs x 128 fp32 lanes x 2 x max SM clock"}
    roofline["frac"] = round(roofline["achieved"] / roofline["peak"], 4)
    roofline["us_per_call"] = round(t_call * 1e6, 2)
    h2d = sum(t.numel() * t.element_size() for t in hin.values())
    return {
        "metric": PREFILL_METRIC, "value": round(world * B * N / t_call, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": calls, "warmup": args.warmup, "ms_per_step": round(ms / calls, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; Qwen3-Next-shaped GDN layer, random weights)",
        "config": {"workload": f"qwen3next-gdn-prefill-b{B}-n{N}", "B": B, "N": N, "H": wl.H,
                   "HV": wl.HV, "K": wl.K, "V": wl.V, "io_dtype": "bf16", "state_dtype": "fp32",
                   "arith": ARITH["chunk" if path == "chunk" else "generic"], "path": path,
                   "step": "prefill from a zero state (outputs, checkpoint, cursor reset)",
                   "parallelism": "replicas"},
        "e2e": {"value": round(world * B * N * K_e2e / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(hout.numel() * hout.element_size()), "steps": K_e2e,
                "api": "python binding -> C ABI, host pinned buffers"},
        "gpu_launches": 2 * calls,
        "roofline": roofline,
        "clocks": clocks,
    }


def prefill_cpu(B: int, N: int, seconds: float = 10.0) -> dict:
    """The fp64 oracle's prefill, as it stands, on the host cores, on a sample
    of the workload (2 rows, all v-heads, the first 32 tokens of each prompt)."""
    import oracle
    from gated_delta_rule_spec_gb300 import inputs as gen

    c = gen.WORKLOADS["C2"]
    rows, n = min(B, 2), min(N, 32)
    rng = gen.rng_for(9, "prefill-cpu", rows)
    d = oracle.Dims(H=c.H, HV=c.HV, K=c.K, V=c.V, T=c.T, L=c.L, num_slots=rows)
    ly = oracle.Layer(d)
    w = {x: gen.to_f64(y) for x, y in
         gen.window_inputs(rng, rows, n, c.H, c.HV, c.K, c.V, gen.BF16).items()}
    A_log, dt = (x.astype(np.float64) for x in gen.layer_params(rng, c.HV, c.K, False))
    cores = os.cpu_count() or 1
    slots = np.arange(rows, dtype=np.int32)
    reps, t0 = 0, time.perf_counter()
    while True:
        cur = oracle.Cursors(rows)
        oracle.prefill(d, ly, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt,
                       from_zero=True, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 1000:
            break
    return {"value": round(rows * n * reps / el, 2), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{rows} prompts x {n} tokens x {c.HV} v-heads of the B={B}, N={N} workload, "
                      f"fp64 prefill, {reps} repetitions in {el:.1f} s"}

# ----------------------------------------------------------------- reference arm

def run_reference(args, rank: int, world: int) -> dict | None:
    """fp64 oracle steps (verify -> commit -> fold; with --variant snapshot,
    snapshot verify -> snapshot commit) on a bounded sample of the workload's
    rows, timed on the host cores."""
    if rank != 0:
        return None
    import oracle
    from gated_delta_rule_spec_gb300 import inputs as gen

    wl = Workload(args.batch, args.window, args.kda)
    c = dataclasses.replace(gen.WORKLOADS["C2"], T=wl.T)
    rows = 2
    rng = gen.rng_for(11, "reference-arm", rows)
    d = oracle.Dims(H=c.H, HV=c.HV, K=c.K, V=c.V, T=c.T, L=c.L, num_slots=rows, per_key_gate=wl.kda)
    ring = gen.garbage_ring(rng, rows, c.H, c.HV, c.L, c.K, c.V, gen.BF16, wl.kda)
    ly = oracle.Layer(d, checkpoint=rng.standard_normal((rows, c.HV, c.V, c.K)) * 0.1,
                      rawv=gen.to_f64(ring["rawv"]), rawk=gen.to_f64(ring["rawk"]),
                      ring_g=-np.abs(ring["g"].astype(np.float64)),
                      ring_beta=np.abs(ring["beta"].astype(np.float64)) % 1.0)
    wp, base, flag = gen.random_cursors(rng, rows, c.L, c.T)
    cur = oracle.Cursors(rows, wp, base, flag)
    A_log, dt = gen.layer_params(rng, c.HV, c.K, wl.kda)
    slot_idx = np.arange(rows, dtype=np.int32)
    cores = os.cpu_count() or 1
    wins = [{n: gen.to_f64(x) for n, x in
             gen.window_inputs(rng, rows, c.T, c.H, c.HV, c.K, c.V, gen.BF16, wl.kda).items()}
            for _ in range(4)]
    accs = [gen.accept_lens(rng, rows, c.T) for _ in range(4)]

    snapshot = args.variant == "snapshot"

    def step(i):
        w = wins[i % 4]
        if snapshot:
            _, snap, _ = oracle.snapshot_verify(d, ly, slot_idx, w["q"], w["k"], w["v"], w["a"],
                                                w["b"], A_log, dt)
            oracle.snapshot_commit(d, ly, slot_idx, accs[i % 4], snap)
            return
        if args.variant == "derived-d":   # the same outputs, plus the window's d
            oracle.verify_d(d, ly, cur, slot_idx, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt,
                            nthreads=cores)
        else:
            oracle.verify(d, ly, cur, slot_idx, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt,
                          nthreads=cores)
        oracle.commit(d, cur, slot_idx, accs[i % 4])
        oracle.fold(d, ly, cur, slot_idx, nthreads=cores)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t0
    value = rows * c.T * args.steps / el
    what = "snapshot verify + snapshot commit" if snapshot else "verify + commit + fold"
    sample = (f"{rows} rows x {c.HV} v-heads of the B={args.batch} workload per step "
              f"({what}, fp64), {args.steps} steps")
    extra = {"sample_rows_per_step": rows}
    if snapshot:
        extra.update(workload=wl.name.replace("-verify-", "-snapshot-verify-"), step=what)
    if args.variant == "derived-d":
        extra.update(workload=wl.name.replace("-gdn-", "-gdn-derived-d-"),
                     step="verify_d + commit + fold")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": wl.config(extra),
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--batch", type=int, default=128)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--window", type=int, default=None,
                    help="draft window T (default: the workload's 4; 1 = plain decode)")
    ap.add_argument("--kda", action="store_true",
                    help="the KDA variant (one gate per key channel) on the same shape")
    ap.add_argument("--variant", choices=("ring", "snapshot", "derived-d"), default="ring",
                    help="snapshot: the per-draft state design the ring replaces; derived-d: the "
                         "ring also caches each token's corrected delta (comparisons)")
    ap.add_argument("--prefill", type=int, default=0, metavar="N",
                    help="measure gdn_spec_prefill of --batch prompts of N tokens instead")
    ap.add_argument("--verify-only", action="store_true",
                    help="profiling aid: build the state, run --steps plain verify calls, print "
                         "their algorithmic bytes")
    ap.add_argument("--setup-rounds", type=int, default=48,
                    help="random rounds of the state build (fewer: a short run to profile)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if args.impl == "reference":
            backend = "gloo"
        dist.init_process_group(backend)
    if args.verify_only:
        print(json.dumps(run_verify_only(args)), flush=True)
        return
    if args.prefill and args.impl == "reference":
        line = None
        if rank == 0:   # the oracle's prefill on the host cores, a bounded sample
            cb = prefill_cpu(args.batch, args.prefill, seconds=5.0)
            line = {"impl": "reference", "metric": PREFILL_METRIC, "value": cb["value"],
                    "unit": cb["unit"], "n_gpus": world, "steps": 1, "warmup": args.warmup,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "dtype": "f64", "data": "synthetic",
                    "config": {"workload": f"qwen3next-gdn-prefill-b{args.batch}-n{args.prefill}"},
                    "cpu_baseline": cb,
                    "e2e": {"value": cb["value"], "unit": cb["unit"], "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
    elif args.variant == "snapshot" and args.impl != "reference":
        line = run_snapshot(args, rank, world)
    elif args.variant == "derived-d" and args.impl != "reference":
        line = run_derived_d(args, rank, world)
    elif args.prefill:
        line = run_prefill(args, rank, world)
        if line is not None and world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = prefill_cpu(args.batch, args.prefill)
    elif args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world)
        if line is not None and world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.batch, T=args.window, kda=args.kda)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
