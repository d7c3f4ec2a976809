"""Benchmark of the LoGRA sketching hot path on GB300.

One step = one optimizer step of the 7B-class decoder projection set (hidden
3584, 28 layers × {q, k, v, o, gate, up, down}): 8 micro-batches of 16384
tokens accumulated into all 196 sketches, predicted KL over 64 responses ×
1024 tokens × vocab 151936 (bf16), the step size on the device, and the rank-r
merge of every weight.  Inputs are synthetic and seeded (see synthetic.py), all
resident in HBM (≈140 GB, far larger than L2, so no flush is needed between
steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--rank 64|256]
                    [--impl ours|reference] [--workload qwen7b|qwen1.5b]

`--workload qwen1.5b` runs the 1.5B-class set instead (hidden 1536, 4
micro-batches of 8192 tokens, r ∈ {4, 16, 64, 256}), with the same KL.

Prints one JSON line (rank 0).  `value` is tokens/s of the whole step; the
per-phase numbers, the roofline of the dominant kernel (sketch accumulation),
the end-to-end figure through pinned host buffers and the fp64 oracle's CPU
baseline are extra keys.  On the 7B set the same run also times the step at
the workload's other rank, r = 256, with the signs rebuilt on chip, and
reports its phases under `phases_r256`.  Under torchrun each rank runs its own 8 micro-batches
(weak scaling), the sketches are summed across ranks (the O(d·r) exchange of
data-parallel accumulation) and every rank applies the same merge.
"""

from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synthetic  # noqa: E402

WORKLOAD = "qwen7b"
KL_WORKLOAD = "qwen"
ETA = 2e-4          # αη = α·η with α ≤ α_max = 1, so αη ≤ 2e-4 as in the merge of the 7B workload
ALPHA_MAX = 1.0
TEMPERATURE = 1.0

# DRAM traffic per sketch pass (one micro-batch over the 196 matrices): the
# DRAM read + write of one ncu capture of a decoder layer's grouped launch
# (its seven matrices: projection, contraction and split reduce) times the 28
# layers, which all have the same shapes.  Keyed by the sha256 of the kernel
# source it was captured on (sketch.cu and the common.cuh it includes), and
# reported only while that source is unchanged.
TRAFFIC = {
    # one layer at r = 64: 3053.0 MB of DRAM traffic for 2978.2 MB algorithmic (1.025x)
    ("qwen7b", "sketch", 64): (85_485_094_912, "16870d1b56119bd4"),
    # one layer at r = 256: 3181.4 MB for 3054.5 MB algorithmic (1.042x)
    ("qwen7b", "sketch", 256): (89_079_201_792, "16870d1b56119bd4"),
}


def _src_sha(*names: str) -> str:
    """sha256[:16] of the named csrc files, concatenated in order."""
    h = hashlib.sha256()
    for name in names:
        h.update(open(os.path.join(ROOT, "rank_gradient_sketching_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.index = str(device)
        try:
            p = torch.cuda.get_device_properties(device)
            self.index = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        except (AttributeError, RuntimeError):
            pass
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[0]))
                smax = float(f[1])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def layer_set():
    w = synthetic.WORKLOADS[WORKLOAD]
    return [(layer, name, d, k, sid, w["seeds"][layer]) for layer, mats in enumerate(w["layers"])
            for (name, d, k, sid) in mats]


def sketch_bytes_per_token(mats) -> int:
    return sum(2 * (d + k) for (_, _, d, k, _, _) in mats)


# --------------------------------------------------------------------- ours

SET_NAME = {"qwen7b": "7B", "qwen1.5b": "1.5B"}


def metric() -> str:
    return f"sketch-accum tokens/s ({SET_NAME[WORKLOAD]} projection set; step also holds predicted KL and merge)"


def workload_config(args, rows, tokens_step):
    """The `config` of the bench line, shared by both arms."""
    w = synthetic.WORKLOADS[WORKLOAD]
    kw = synthetic.KL_WORKLOADS[KL_WORKLOAD]
    return {"workload": f"{WORKLOAD} projection set, 28 layers x 7 matrices, r={args.rank}, {args.microbatches} "
                        f"micro-batches x {w['tokens']} tokens per rank, predicted KL {rows}x{kw['vocab']} bf16 "
                        f"(eps={kw['eps'][0]}), merge of every weight"
                        + (", input X shared by q/k/v and by gate/up" if args.share_x else ", each matrix with its own X"),
            "global_batch": tokens_step, "seq_len": 1024, "rank": args.rank,
            "inputs": "one seeded (X, dY) pair per matrix, resident in HBM and fed to every micro-batch of the step "
                      "(the micro-batches re-read the same 83 GB, far larger than L2, so each pass streams from HBM)"}


class StepRunner:
    """One optimizer step of the projection set at rank r over resident
    inputs: the sketch of every micro-batch into all sketches, the predicted
    KL, the step size on the device, the merge of every weight.  The work is
    spread over worker streams (one workspace each); CUDA events on the
    launch stream bracket each phase."""

    def __init__(self, args, lg, dp, dev, stream, mats, inputs, units, weights, kl, r, cache, world):
        self.args, self.lg, self.dp, self.dev, self.stream = args, lg, dp, dev, stream
        self.mats, self.inputs, self.units, self.weights = mats, inputs, units, weights
        self.cur, self.prop, self.kl_ws, self.q_buf, self.ae_buf, self.deltas, self.rows = kl
        self.r, self.world = r, world
        w = synthetic.WORKLOADS[WORKLOAD]
        self.T, self.MB = w["tokens"], args.microbatches
        T = self.T
        self.s_flat = torch.zeros(sum(d * r for (_, _, d, _, _, _) in mats), dtype=torch.float32, device=dev)
        self.sketches, off = [], 0
        for (_, _, d, _, _, _) in mats:
            self.sketches.append(self.s_flat[off:off + d * r].view(d, r))
            off += d * r

        def unit_ws_bytes(u):
            k = mats[u[0]][3]
            if len(u) == 1:
                return lg.logra_sketch_workspace_bytes(T, mats[u[0]][2], k, r)
            return lg.logra_sketch_shared_x_workspace_bytes(T, k, [mats[j][2] for j in u], r)

        ws_bytes = max(unit_ws_bytes(u) for u in units)
        # Round-robin over the streams in issue order, so that at any moment the
        # streams work on neighbouring units of different sizes.  When a layer
        # holds a multiple of the stream count of units (4 with --share-x on 4
        # streams), plain round-robin would pin each unit type to one stream for
        # the whole pass; the order is then rotated by one stream per layer.
        per_layer = len(units) // len(w["layers"])
        rotate = per_layer % args.streams == 0
        self.unit_stream = [(n + (n // per_layer if rotate else 0)) % args.streams for n in range(len(units))]
        self.mat_stream = [j % args.streams for j in range(len(mats))]
        self.streams = [torch.cuda.Stream(dev) for _ in range(args.streams)]
        self.wss = [torch.empty(ws_bytes, dtype=torch.uint8, device=dev) for _ in range(args.streams)]
        # Projection basis: fixed (one seed per layer for the whole run),
        # refreshed (a new seed every step), or refreshed Gaussian.  The sketch and
        # merge kernels either rebuild the ±1 tiles on chip from the seed, or read
        # a cached bf16 operand Ã (r×k per weight) by TMA: always for the Gaussian
        # basis, and for the signs when the projection cache is on.  A fixed basis
        # is cached once at setup; a refreshed one is regenerated every step.
        cache = cache or args.projection == "gaussian"
        self.op_kind = lg.LOGRA_PROJ_GAUSS_BF16 if args.projection == "gaussian" else lg.LOGRA_PROJ_SIGN_BF16
        self.gauss_ops = ([torch.empty((r, mats[j][3]), dtype=torch.bfloat16, device=dev) for j in range(len(mats))]
                          if cache else None)
        self.step_seeds = [m[5] for m in mats]
        if self.gauss_ops is not None and args.projection == "fixed":
            for j, m in enumerate(mats):
                lg.logra_regen_projection(m[5], m[4], r, m[3], self.op_kind, out=self.gauss_ops[j])
        # momentum on the sketch: M ← β·M + S once per step, merged as U = M
        self.m_flat = torch.zeros_like(self.s_flat) if args.momentum is not None else None
        self.m_views, off = [], 0
        for (_, _, d, _, _, _) in mats:
            if self.m_flat is not None:
                self.m_views.append(self.m_flat[off:off + d * r].view(d, r))
            off += d * r
        self.merge_mode = args.merge
        if self.merge_mode == "auto":
            # small weights (the 1.5B set) leave each per-weight launch's start
            # and end idle, and one launch over all of them fills the GPU
            # (measured 69 -> 88 % of HBM at r = 16); large weights (the 7B set)
            # already fill it on eight streams, where the plan lookup at each
            # CTA's start costs more than the launch tails (88 -> 83 %).
            mean_elems = sum(d * k for (_, _, d, k, _, _) in mats) / len(mats)
            self.merge_mode = "group" if mean_elems < 2**24 else "per-weight"
        self.merge_plan = None
        if self.merge_mode == "group":
            self.plan_merge()
        # The sketch of a micro-batch: one call per matrix (or unit) over the
        # worker streams, or with --sketch group one launch per phase over all
        # matrices on the launch stream.  The plan holds the inputs' and the
        # sketches' addresses, which every micro-batch reuses; like the merge
        # plan it is rebuilt when the seeds change.
        self.sketch_plan = None
        if args.sketch == "group":
            self.plan_sketch()
        # kernels of ours per step: projection + contraction (+ the split reduce)
        # per matrix and micro-batch, the two KL kernels, the step size, the merges
        sketch_launches = len(units) + sum(1 + (lg.logra_sketch_splits(T, d, k, r) > 1)
                                           for (_, _, d, k, _, _) in mats)
        if args.sketch == "group":
            # one projection, one contraction and (when a matrix splits T) one reduce launch
            sketch_launches = 2 + any(lg.logra_sketch_splits(T, d, k, r) > 1 for (_, _, d, k, _, _) in mats)
        self.launches_per_step = (self.MB * sketch_launches + 2 + 1
                                  + (1 if self.merge_mode == "group" else len(mats))
                                  + (len(mats) if self.gauss_ops is not None and args.projection != "fixed" else 0)
                                  + (1 if self.m_flat is not None else 0))
        self.ev = {}

    # ---- work on the worker streams
    def record(self, name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        self.ev.setdefault(name, []).append(e)

    def fan_out(self, work, idx=None, unit_order=False):
        """Runs work(j, stream, workspace) for every matrix j (or unit j, or
        those in idx) over the worker streams, ordered after everything
        already queued on the launch stream, and makes the launch stream wait
        for all of it."""
        fork = torch.cuda.Event()
        fork.record(self.stream)
        for st in self.streams:
            st.wait_event(fork)
        smap = self.unit_stream if unit_order else self.mat_stream
        n = len(self.units) if unit_order else len(self.mats)
        for j in (range(n) if idx is None else idx):
            work(j, self.streams[smap[j]], self.wss[smap[j]])
        for st in self.streams:
            join = torch.cuda.Event()
            join.record(st)
            self.stream.wait_event(join)

    def sketch_one(self, j, st, wsj):
        lg, r = self.lg, self.r
        (X, dY), S, (layer, name, d, k, sid, seed) = self.inputs[j], self.sketches[j], self.mats[j]
        if self.gauss_ops is not None:
            lg.logra_sketch_accumulate_proj(X, dY, S, self.gauss_ops[j], r, wsj, stream=st)
        else:
            lg.logra_sketch_accumulate(X, dY, S, self.step_seeds[j], sid, r, wsj, stream=st)

    def regen_one(self, j, st, wsj):
        (layer, name, d, k, sid, seed) = self.mats[j]
        self.lg.logra_regen_projection(self.step_seeds[j], sid, self.r, k, self.op_kind, out=self.gauss_ops[j],
                                       stream=st)

    def sketch_unit(self, n, st, wsj):
        lg, r, u = self.lg, self.r, self.units[n]
        if len(u) == 1:
            self.sketch_one(u[0], st, wsj)
        elif self.gauss_ops is not None:
            X = self.inputs[u[0]][0]
            lg.logra_sketch_accumulate_shared_x_proj(
                X, [(self.inputs[j][1], self.sketches[j], self.gauss_ops[j]) for j in u], r, wsj, stream=st)
        else:
            X = self.inputs[u[0]][0]
            lg.logra_sketch_accumulate_shared_x(
                X, [(self.inputs[j][1], self.sketches[j], self.step_seeds[j], self.mats[j][4]) for j in u], r, wsj,
                stream=st)

    def merge_one(self, j, st, wsj):
        lg, r = self.lg, self.r
        W, S, (layer, name, d, k, sid, seed) = self.weights[j], self.sketches[j], self.mats[j]
        U = self.m_views[j] if self.m_flat is not None else S
        if self.gauss_ops is not None:
            lg.logra_merge_update_proj(W, U, self.gauss_ops[j], r, 0.0, alpha_eta_dev=self.ae_buf, stream=st)
        else:
            lg.logra_merge_update(W, U, self.step_seeds[j], sid, r, 0.0, alpha_eta_dev=self.ae_buf, stream=st)

    # The merge of all weights is one launch over a plan (tensor maps and
    # descriptors of every weight, copied to the device on the launch stream),
    # or one launch per weight over the worker streams.  The plan holds the
    # seeds: with refreshed signs built on chip it is rebuilt every step, while
    # cached operands are regenerated in place and keep it valid.
    def plan_merge(self):
        tg = []
        for j, (layer, name, d, k, sid, seed) in enumerate(self.mats):
            U = self.m_views[j] if self.m_flat is not None else self.sketches[j]
            tg.append((self.weights[j], U, self.gauss_ops[j]) if self.gauss_ops is not None
                      else (self.weights[j], U, self.step_seeds[j], sid))
        self.merge_plan = self.lg.logra_merge_group_plan(tg, self.r, stream=self.stream)

    def plan_sketch(self):
        tg = []
        for j, (layer, name, d, k, sid, seed) in enumerate(self.mats):
            X, dY = self.inputs[j]
            tg.append((X, dY, self.sketches[j], self.gauss_ops[j]) if self.gauss_ops is not None
                      else (X, dY, self.sketches[j], self.step_seeds[j], sid))
        self.sketch_plan = self.lg.logra_sketch_group_plan(tg, self.r, stream=self.stream, reuse=self.sketch_plan)

    def do_sketch(self):
        if self.sketch_plan is not None:
            self.lg.logra_sketch_accumulate_group(self.sketch_plan, stream=self.stream)
        else:
            self.fan_out(self.sketch_unit, unit_order=True)

    def do_merge(self):
        if self.merge_mode == "group":
            self.lg.logra_merge_update_group(self.merge_plan, 0.0, alpha_eta_dev=self.ae_buf, stream=self.stream)
        else:
            self.fan_out(self.merge_one)

    def step(self, i, timed):
        lg, args = self.lg, self.args
        if args.projection != "fixed":
            self.step_seeds[:] = [lg.logra_refreshed_seed(m[5], i) for m in self.mats]
            if self.merge_mode == "group" and self.gauss_ops is None:
                self.plan_merge()
            if self.sketch_plan is not None and self.gauss_ops is None:
                self.plan_sketch()
        if self.gauss_ops is not None and args.projection != "fixed":
            if timed:
                self.record("pj0")
            self.fan_out(self.regen_one)
            if timed:
                self.record("pj1")
        if self.m_flat is None:
            self.s_flat.zero_()  # (with momentum the momentum call clears S)
        for mb in range(self.MB):
            if timed:
                self.record("sk0")
            self.do_sketch()
            if timed:
                self.record("sk1")
        if self.world > 1:
            self.dp.allreduce_sketch(self.s_flat)
        if timed:
            self.record("kl0")
        lg.logra_predicted_kl(self.cur, self.prop, TEMPERATURE, q_out=self.q_buf, workspace=self.kl_ws)
        if self.world > 1:
            self.dp.global_q(self.q_buf, self.rows)
        lg.logra_step_size_device(self.q_buf, self.deltas[i % len(self.deltas)], ALPHA_MAX, ETA, self.ae_buf)
        if timed:
            self.record("kl1")
        if self.m_flat is not None:
            if timed:
                self.record("mo0")
            lg.logra_sketch_momentum(self.m_flat.view(-1, self.r), self.s_flat.view(-1, self.r), args.momentum,
                                     clear_s=True)
            if timed:
                self.record("mo1")
        if timed:
            self.record("mg0")
        self.do_merge()
        if timed:
            self.record("mg1")

    def measure(self, steps, warmup, local_rank, clocks=True):
        """Warm-up, then `steps` timed steps bracketed by a barrier and a
        synchronize; returns ms per step (max over ranks) and the clocks."""
        lg = self.lg
        for i in range(warmup):
            self.step(i, False)
        torch.cuda.synchronize()
        if lg.logra_device_error() != 0:
            raise RuntimeError("a kernel recorded a device error during warm-up")
        self.ev = {}
        if self.world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        with ClockSampler(local_rank) if clocks else contextlib.nullcontext() as clk:
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            start.record(self.stream)
            for i in range(steps):
                self.step(warmup + i, True)
            end.record(self.stream)
            torch.cuda.synchronize()
        if self.world > 1:
            torch.distributed.barrier()
        ms_total = start.elapsed_time(end)
        if self.world > 1:
            t = torch.tensor([ms_total], device=self.dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            ms_total = float(t.item())
        if lg.logra_device_error() != 0:
            raise RuntimeError("a kernel recorded a device error in the timed region")
        return ms_total / steps, (clk.summary() if clocks else None)

    def phases(self):
        """Per-phase times, bandwidths and roofline fractions of the timed steps."""
        ev, mats, units, T, r = self.ev, self.mats, self.units, self.T, self.r
        kw = synthetic.KL_WORKLOADS[KL_WORKLOAD]
        sk_ms = [a.elapsed_time(b) for a, b in zip(ev["sk0"], ev["sk1"])]
        kl_ms = [a.elapsed_time(b) for a, b in zip(ev["kl0"], ev["kl1"])]
        mg_ms = [a.elapsed_time(b) for a, b in zip(ev["mg0"], ev["mg1"])]
        hbm, bf16, bf16_sus, peak_kind = _peaks()
        # algorithmic bytes of one sketch pass: each input X read once per unit, each dY once, S read + written
        sk_bytes = (sum(2 * T * mats[u[0]][3] for u in units)
                    + sum(2 * T * d + 8 * d * r for (_, _, d, k, _, _) in mats))
        sk_flops = sum(2 * T * r * (d + k) for (_, _, d, k, _, _) in mats)
        sk_avg = statistics.mean(sk_ms)
        sk_gbs = sk_bytes / (sk_avg / 1e3) / 1e9
        sk_tfs = sk_flops / (sk_avg / 1e3) / 1e12
        kl_bytes = 2 * self.rows * kw["vocab"] * 2
        kl_gbs = kl_bytes / (statistics.mean(kl_ms) / 1e3) / 1e9
        mg_bytes = sum(4 * d * k + 4 * d * r for (_, _, d, k, _, _) in mats)
        mg_gbs = mg_bytes / (statistics.mean(mg_ms) / 1e3) / 1e9
        # the binding roofline of the sketch: HBM at r ≤ 64; above, the larger
        # of the HBM time and the tensor time of the algorithmic FLOPs at the
        # sustained bf16 rate (the two are about equal at r = 256)
        t_hbm = sk_bytes / (hbm * 1e9)
        t_tc = sk_flops / (bf16_sus * 1e12)
        bound = "hbm" if r <= 64 or t_hbm >= t_tc else "tensor"
        ph = {
            "sketch_accum": {"tokens_per_s": round(T * self.world / (sk_avg / 1e3), 1), "GB_per_s": round(sk_gbs, 1),
                             "hbm_frac": round(sk_gbs / hbm, 4), "TFLOP_per_s": round(sk_tfs, 1),
                             "tensor_frac_sustained": round(sk_tfs / bf16_sus, 4),
                             "binding": bound,
                             "binding_frac": round((t_hbm if bound == "hbm" else t_tc) / (sk_avg / 1e3), 4),
                             "ms_per_microbatch": round(sk_avg, 4)},
            "predicted_kl": {"GB_per_s": round(kl_gbs, 1), "hbm_frac": round(kl_gbs / hbm, 4),
                             "ms": round(statistics.mean(kl_ms), 4), "bytes": kl_bytes},
            "merge": {"GB_per_s": round(mg_gbs, 1), "hbm_frac": round(mg_gbs / hbm, 4),
                      "ms": round(statistics.mean(mg_ms), 4), "bytes": mg_bytes},
        }
        if self.gauss_ops is not None and self.args.projection != "fixed":
            pj_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(ev["pj0"], ev["pj1"]))
            ph["projection_regen"] = {"ms": round(pj_ms, 4), "bytes_written": sum(2 * r * k for (_, _, _, k, _, _) in mats)}
        if self.m_flat is not None:
            mo_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(ev["mo0"], ev["mo1"]))
            mo_bytes = 16 * self.s_flat.numel()  # read M and S, write M and S (cleared)
            ph["momentum"] = {"ms": round(mo_ms, 4), "GB_per_s": round(mo_bytes / mo_ms / 1e6, 1), "bytes": mo_bytes}
        return ph, {"sk_bytes": sk_bytes, "sk_flops": sk_flops, "sk_avg": sk_avg, "sk_gbs": sk_gbs,
                    "sk_tfs": sk_tfs, "kl_bytes": kl_bytes, "mg_bytes": mg_bytes, "bound": bound,
                    "peaks": (hbm, bf16, bf16_sus, peak_kind)}

    def projection_desc(self):
        r, args = self.r, self.args
        return {"fixed": "fixed Rademacher", "refreshed": "refreshed Rademacher",
                "gaussian": "refreshed Gaussian"}[args.projection] + (
            f", cached bf16 operand in HBM ({sum(2 * r * m[3] for m in self.mats) / 1e6:.0f} MB)"
            if self.gauss_ops is not None else ", signs rebuilt on chip")

    def free(self):
        self.s_flat = self.sketches = self.wss = self.gauss_ops = self.m_flat = self.m_views = None
        self.merge_plan = self.sketch_plan = None


def run_ours(args, rank, world, local_rank):
    import rank_gradient_sketching_gb300 as lg
    from rank_gradient_sketching_gb300 import dp

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synthetic.WORKLOADS[WORKLOAD]
    kw = synthetic.KL_WORKLOADS[KL_WORKLOAD]
    T, MB, r = w["tokens"], args.microbatches, args.rank
    mats = layer_set()
    stream = torch.cuda.current_stream(dev)

    # ---- resident inputs (shared by every rank measured below)
    t_setup = time.time()
    inputs, weights = [], []
    # Work units: one matrix each, or with --share-x the groups that read one
    # input in a decoder layer (q/k/v and gate/up), sketched by one call.
    units = []
    for (layer, name, d, k, sid, seed) in mats:
        j = len(inputs)
        X, dY = synthetic.microbatch(WORKLOAD, layer, name, rank, T, d, k, dev)
        # a group stacks (r rounded up to 16) rows per weight, at most 512 in one call
        fits = len(units) and (len(units[-1]) + 1) * ((r + 15) // 16 * 16) <= 512
        if args.share_x and name in ("k", "v", "up") and fits:
            X = inputs[j - 1][0]  # the previous matrix of the group already holds the shared input
            units[-1].append(j)
        else:
            units.append([j])
        inputs.append((X, dY))
        weights.append(synthetic.weight(WORKLOAD, layer, name, d, k, dev))
    rows = kw["rows"] // world if world > 1 else kw["rows"]
    cur, prop = synthetic.kl_logits(KL_WORKLOAD, kw["eps"][0], rows=rows, device=dev)
    kl_ws = torch.empty(lg.logra_kl_workspace_bytes(rows), dtype=torch.uint8, device=dev)
    q_buf = torch.zeros((), dtype=torch.float64, device=dev)
    ae_buf = torch.zeros((), dtype=torch.float32, device=dev)
    deltas = lg.delta_schedule(kw["delta"][0], kw["delta"][1], kw["steps"])
    kl = (cur, prop, kl_ws, q_buf, ae_buf, deltas, rows)
    cache = args.cache_projection == "on"
    run = StepRunner(args, lg, dp, dev, stream, mats, inputs, units, weights, kl, r, cache, world)
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup

    ms_step, clocks = run.measure(args.steps, args.warmup, local_rank)
    tokens_step = T * MB * world
    value = tokens_step / (ms_step / 1e3)
    phases, m = run.phases()
    hbm, bf16, bf16_sus, peak_kind = m["peaks"]
    sha = _src_sha("sketch.cu", "common.cuh")  # the sketch kernels and the helpers they include
    traffic = TRAFFIC.get((WORKLOAD, "sketch", r))
    traffic_val = traffic[0] if traffic and traffic[1] == sha else None
    if m["bound"] == "hbm":
        roof = {"bound": "hbm", "achieved": round(m["sk_gbs"], 1), "peak": hbm, "unit": "GB/s",
                "frac": round(m["sk_gbs"] / hbm, 4), "traffic": traffic_val}
    else:
        roof = {"bound": "tensor", "achieved": round(m["sk_tfs"], 1), "peak": bf16_sus, "unit": "TFLOP/s",
                "frac": round(m["sk_tfs"] / bf16_sus, 4), "traffic": traffic_val}
    roof.update({"kernel": "sketch accumulation (projection + contraction + split reduce), one micro-batch over "
                           "196 matrices",
                 "algorithmic_bytes": m["sk_bytes"], "algorithmic_flops": m["sk_flops"],
                 "launch_ms": round(m["sk_avg"], 4),
                 "peak_source": f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback",
                 "hbm_frac": round(m["sk_gbs"] / hbm, 4),
                 "tensor_frac_sustained": round(m["sk_tfs"] / bf16_sus, 4),
                 "traffic_source": ("ncu DRAM read+write of one layer's grouped launch times 28 layers, a "
                                    "constant taken on this sketch.cu and common.cuh" if traffic_val is not None
                                    else "no ncu capture on this sketch.cu")})

    out = {
        "metric": metric(),
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, fp32 accumulate", "data": "synthetic (seeded; see synthetic.py)",
        "config": {**workload_config(args, rows, tokens_step), "parallelism": f"dp{world}",
                   "l2": f"inputs larger than L2 ({(m['sk_bytes'] * MB + m['kl_bytes'] + m['mg_bytes']) / 1e9:.0f} "
                         "GB touched per step, no flush needed)"},
        "phases": phases,
        "roofline": roof,
        "gpu_launches": run.launches_per_step * args.steps,
        "clocks": clocks,
        "setup_s": round(setup_s, 1),
    }
    out["config"]["streams"] = 1 if args.sketch == "group" else args.streams
    out["config"]["sketch"] = ("one launch per phase over all matrices (plan), one stream" if args.sketch == "group"
                               else f"one call per {'unit' if args.share_x else 'matrix'} over {args.streams} streams")
    out["config"]["merge"] = ("one launch over all weights (plan)" if run.merge_mode == "group"
                              else "one launch per weight")
    out["config"]["projection"] = run.projection_desc()
    if args.momentum is not None:
        out["config"]["momentum"] = args.momentum

    # ---- the second rank of the 7B workload (r = 256), timed in the same run
    # with the signs rebuilt on chip (no projection stored in HBM)
    if (WORKLOAD == "qwen7b" and r != 256 and not args.no_r256 and args.projection == "fixed"
            and args.momentum is None):
        run256 = StepRunner(args, lg, dp, dev, stream, mats, inputs, units, weights, kl, 256, False, world)
        steps256 = max(3, min(args.steps, 5))
        ms256, clk256 = run256.measure(steps256, 3, local_rank)
        ph256, m256 = run256.phases()
        t256 = TRAFFIC.get((WORKLOAD, "sketch", 256))
        if t256 and t256[1] == sha:
            ph256["sketch_accum"]["dram_traffic_bytes"] = t256[0]
            ph256["sketch_accum"]["traffic_source"] = ("ncu DRAM read+write of one layer's grouped launch times 28 "
                                                       "layers, a constant taken on this sketch.cu and common.cuh")
        out["phases_r256"] = {
            "rank": 256, "steps": steps256, "warmup": 3, "ms_per_step": round(ms256, 3),
            "tokens_per_s": round(tokens_step / (ms256 / 1e3), 1), "projection": run256.projection_desc(),
            "merge": ("one launch over all weights (plan)" if run256.merge_mode == "group"
                      else "one launch per weight"),
            "clocks": clk256, **ph256}
        run256.free()
        del run256
        torch.cuda.empty_cache()

    if not args.no_autograd and args.projection == "fixed" and args.momentum is None and not args.share_x:
        out["autograd_sketch"] = run_autograd(args, lg, dev, stream, mats, inputs, weights, r)
        torch.cuda.empty_cache()
    if not args.no_e2e and not args.share_x and args.projection == "fixed" and args.momentum is None:
        out["e2e"] = run_e2e(args, lg, dev, stream, run)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args, r, budget_s=args.cpu_budget)
    return out


def run_autograd(args, lg, dev, stream, mats, inputs, weights, r):
    """The sketch driven by autograd: every matrix of the set as a
    SketchedLinearGroup fed its resident input, the forward, then the
    backward with the step's dY inside a SketchBatch (one stream; the
    input-gradient GEMMs run in the same backward).  CUDA events time the
    backward and each grouped sketch launch within it."""
    from rank_gradient_sketching_gb300.autograd import SketchBatch, SketchedLinearGroup

    T = synthetic.WORKLOADS[WORKLOAD]["tokens"]
    groups = [SketchedLinearGroup([weights[j]], r, seeds=[m[5]], stream_ids=[m[4]]) for j, m in enumerate(mats)]
    flush_bytes = 32 << 30

    def microbatch(ev):
        leaves = [X.detach().requires_grad_(True) for (X, _) in inputs]
        ys = [g(x)[0] for g, x in zip(groups, leaves)]
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        with SketchBatch(flush_bytes=flush_bytes, timing=True) as sb:
            torch.autograd.backward(ys, [dY for (_, dY) in inputs])
        b1.record(stream)
        ev.append((b0, b1, sb))
        del ys, leaves

    warm, n = 1, max(1, args.autograd_microbatches)
    ev = []
    for _ in range(warm):
        microbatch([])
    torch.cuda.synchronize()
    for _ in range(n):
        microbatch(ev)
    torch.cuda.synchronize()
    if lg.logra_device_error() != 0:
        raise RuntimeError("a kernel recorded a device error in the autograd block")
    bw_ms = statistics.mean(b0.elapsed_time(b1) for b0, b1, _ in ev)
    sk_ms = statistics.mean(sum(e0.elapsed_time(e1) for e0, e1 in sb.events) for _, _, sb in ev)
    sk_bytes = sum(2 * T * (d + k) + 8 * d * r for (_, _, d, k, _, _) in mats)
    hbm = _peaks()[0]
    out = {"rank": r, "microbatches": n, "warmup_microbatches": warm,
           "backward_ms_per_microbatch": round(bw_ms, 3),
           "backward_tokens_per_s": round(T / (bw_ms / 1e3), 1),
           "sketch_ms_per_microbatch": round(sk_ms, 4),
           "sketch_tokens_per_s": round(T / (sk_ms / 1e3), 1),
           "sketch_GB_per_s": round(sk_bytes / (sk_ms / 1e3) / 1e9, 1),
           "sketch_hbm_frac": round(sk_bytes / (sk_ms / 1e3) / 1e9 / hbm, 4),
           "flushes_per_microbatch": round(statistics.mean(sb.flushes for _, _, sb in ev), 2),
           "note": "backward of the 196 matrices as SketchedLinearGroup modules on one stream: input-gradient "
                   "GEMMs (cuBLAS) and the sketches deferred into a SketchBatch (grouped launches, flushed every "
                   f"{flush_bytes >> 30} GiB of inputs); the sketch time is the sum of the grouped launches"}
    del groups
    return out


def run_e2e(args, lg, dev, stream, run):
    """Same step through the public API with the step's inputs copied in from
    pinned host memory every step and q(D), α read back to the host.  Host
    buffers hold one layer's X/dY and one 4096-row block of logits; every
    layer and block is copied from them, so the bytes moved equal the full
    inputs of the step.  All copies run on a side stream (the sketch inputs one
    layer ahead of the kernels, then the logits), so the host link, which
    bounds this number, does not wait on the kernels.  It runs as many steps as
    the device-timed region unless that would take more than about a minute
    (each step moves ~0.7 TB over the host link, ~3.3 s)."""
    mats, inputs, T, MB, world = run.mats, run.inputs, run.T, run.MB, run.world
    cur, prop, kl_ws, q_buf, ae_buf, deltas = run.cur, run.prop, run.kl_ws, run.q_buf, run.ae_buf, run.deltas
    layer0 = [(X.cpu().pin_memory(), dY.cpu().pin_memory()) for (X, dY), m in zip(inputs, mats) if m[0] == 0]
    nmat = len(layer0)
    blk = 4096
    rows = cur.shape[0]
    cur_h = cur[:blk].cpu().pin_memory()
    prop_h = prop[:blk].cpu().pin_memory()
    copy = torch.cuda.Stream(dev)
    out_h = torch.empty(2, dtype=torch.float64).pin_memory()
    h2d = 0
    layers = len(mats) // nmat
    done = [torch.cuda.Event() for _ in range(layers)]
    # with --sketch group each layer's matrices are one plan (one launch per
    # phase on the launch stream), launched as that layer's inputs arrive
    layer_plans = None
    if run.sketch_plan is not None:
        layer_plans = [lg.logra_sketch_group_plan(
            [(inputs[j][0], inputs[j][1], run.sketches[j], run.step_seeds[j], mats[j][4])
             for j in range(L * nmat, (L + 1) * nmat)], run.r, stream=stream) for L in range(layers)]
    kl_done = torch.cuda.Event()

    def step(i):
        nonlocal h2d
        run.s_flat.zero_()
        for mb in range(MB):
            ready = []
            for L in range(layers):
                copy.wait_event(done[L])  # the previous micro-batch has finished reading layer L
                with torch.cuda.stream(copy):
                    for j in range(nmat):
                        X, dY = inputs[L * nmat + j]
                        X.copy_(layer0[j][0], non_blocking=True)
                        dY.copy_(layer0[j][1], non_blocking=True)
                        h2d += layer0[j][0].numel() * 2 + layer0[j][1].numel() * 2
                    e = torch.cuda.Event()
                    e.record(copy)
                ready.append(e)
            for L in range(layers):
                stream.wait_event(ready[L])
                if layer_plans is not None:
                    lg.logra_sketch_accumulate_group(layer_plans[L], stream=stream)
                else:
                    run.fan_out(run.sketch_one, range(L * nmat, (L + 1) * nmat))
                done[L].record(stream)
        # the logits follow the sketch inputs on the copy stream, so the host
        # link stays busy while the last micro-batch is sketched
        copy.wait_event(kl_done)  # the previous step's KL has read them
        with torch.cuda.stream(copy):
            for b in range(0, rows, blk):
                n = min(blk, rows - b)
                cur[b:b + n].copy_(cur_h[:n], non_blocking=True)
                prop[b:b + n].copy_(prop_h[:n], non_blocking=True)
                h2d += 2 * n * cur.shape[1] * 2
            logits_in = torch.cuda.Event()
            logits_in.record(copy)
        stream.wait_event(logits_in)
        lg.logra_predicted_kl(cur, prop, TEMPERATURE, q_out=q_buf, workspace=kl_ws)
        kl_done.record(stream)
        alpha = torch.empty((), dtype=torch.float64, device=dev)
        lg.logra_step_size_device(q_buf, deltas[i % len(deltas)], ALPHA_MAX, ETA, ae_buf, alpha)
        run.do_merge()
        out_h[0].copy_(q_buf, non_blocking=True)
        out_h[1].copy_(alpha, non_blocking=True)
        torch.cuda.synchronize()
        return float(out_h[0]), float(out_h[1])

    warm = 1
    want = args.steps if args.e2e_steps is None else max(1, args.e2e_steps)
    for i in range(warm):
        t_w = time.perf_counter()
        step(i)
        t_w = time.perf_counter() - t_w
    steps = max(1, min(want, int(60.0 / max(t_w, 1e-3))))
    h2d = 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        step(warm + i)
    dt = time.perf_counter() - t0
    return {"value": round(T * MB * world * steps / dt, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d // steps,
            "d2h_bytes_per_step": 16, "steps": steps, "warmup": warm,
            "note": "host wall clock around the steps; inputs copied from pinned host memory every step"
                    + ("" if steps == want else f"; {steps} of the {want} steps asked, to keep it near a minute")}


# ------------------------------------------------------------ oracle (CPU)

def _oracle_sample(r, mb, rng_seed=0):
    """Times the fp64 oracle on a bounded sample of one step and scales it to
    the full step: (seconds for a full step, description)."""
    from oracle import kl as okl
    from oracle import merge as omerge
    from oracle import philox as oph
    from oracle import sketch as osk

    w = synthetic.WORKLOADS[WORKLOAD]
    kw = synthetic.KL_WORKLOADS[KL_WORKLOAD]
    mats = layer_set()
    T_s, d, k = 4096, 3584, 3584
    X, dY = synthetic.microbatch(WORKLOAD, 0, "q", 0, T_s, d, k, "cpu")
    Xn, dYn = X.double().numpy(), dY.double().numpy()
    t0 = time.perf_counter()
    A = oph.projection(100, 0, r, k)
    osk.sketch_accumulate(np.zeros((d, r)), [(Xn, dYn)], A)
    t_sk = time.perf_counter() - t0
    # dense G costs 2·T·d·k and dominates; scale by Σ d·k and by tokens
    dk_total = sum(dd * kk for (_, _, dd, kk, _, _) in mats)
    sk_full = t_sk * (w["tokens"] / T_s) * (dk_total / (d * k)) * mb

    rows_s = 16
    cur, prop = synthetic.kl_logits(KL_WORKLOAD, kw["eps"][0], rows=rows_s)
    t0 = time.perf_counter()
    okl.predicted_kl(cur.double().numpy(), prop.double().numpy(), TEMPERATURE)
    kl_full = (time.perf_counter() - t0) * kw["rows"] / rows_s

    Wt = synthetic.weight(WORKLOAD, 0, "q", d, k, "cpu").double().numpy()
    S = np.random.default_rng(rng_seed).standard_normal((d, r))
    t0 = time.perf_counter()
    omerge.merge(Wt, S, A, 2e-4)
    mg_full = (time.perf_counter() - t0) * dk_total / (d * k)
    desc = (f"oracle sketch of one 3584x3584 matrix on {T_s} tokens (scaled by tokens and by sum d*k over the 196 "
            f"matrices, x{mb} micro-batches) + oracle KL on {rows_s} rows (scaled to {kw['rows']}) + "
            "oracle merge of one 3584x3584 matrix (scaled by sum d*k)")
    return sk_full + kl_full + mg_full, desc, t_sk


def _cores():
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count()


def cpu_baseline(args, r, budget_s=30.0):
    w = synthetic.WORKLOADS[WORKLOAD]
    secs, desc, _ = _oracle_sample(r, args.microbatches)
    return {"value": round(w["tokens"] * args.microbatches / secs, 3), "unit": "tokens/s", "cores": _cores(),
            "kind": "oracle", "sample": desc}


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle on the host cores.  Each step is one
    bounded sample of the step (see _oracle_sample); `ms_per_step` is the
    measured wall time of one sample, and `value` the step's tokens over the
    full step's time extrapolated from the samples (recorded under
    `extrapolation`)."""
    if rank != 0:
        return None
    w = synthetic.WORKLOADS[WORKLOAD]
    warm = min(args.warmup, 1)
    for _ in range(warm):
        _oracle_sample(args.rank, args.microbatches)
    vals, walls, desc = [], [], ""
    t0 = time.perf_counter()
    for i in range(args.steps):
        ts = time.perf_counter()
        secs, desc, _ = _oracle_sample(args.rank, args.microbatches, i)
        walls.append(time.perf_counter() - ts)
        vals.append(secs)
        if time.perf_counter() - t0 > args.cpu_budget * 4:
            break
    secs = statistics.mean(vals)
    value = w["tokens"] * args.microbatches / secs
    kw = synthetic.KL_WORKLOADS[KL_WORKLOAD]
    sample_ms = statistics.mean(walls) * 1e3
    return {"impl": "reference", "metric": metric(),
            "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1, "steps": len(vals), "warmup": warm,
            "ms_per_step": round(sample_ms, 1), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded; see synthetic.py)",
            "config": {**workload_config(args, kw["rows"] // world if world > 1 else kw["rows"],
                                         w["tokens"] * args.microbatches * world),
                       "parallelism": "none (oracle on the host cores of rank 0)"},
            "extrapolation": {"samples_run": len(vals), "sample_ms": round(sample_ms, 1),
                              "full_step_ms_extrapolated": round(secs * 1e3, 1),
                              "note": "each step is a bounded sample of the workload; value = tokens of a full "
                                      "step / the full step's time scaled up from the samples, which were the only "
                                      "work run"},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_kernel_case(args):
    """One kernel on one matrix shape of the 7B set (for profiling): the q
    projection (3584×3584, 16384 tokens) for the sketch, the seven matrices
    of one layer in one plan for the grouped sketch, the gate projection
    (18944×3584) for the merge, the 14 weights of two 1.5B-set layers in one
    launch for the grouped merge, 4096 full-vocabulary rows for the KL.  Times
    `--steps` launches with CUDA events on the launch stream and prints one
    JSON line."""
    import rank_gradient_sketching_gb300 as lg

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    T, d, k, r = 16384, 3584, 3584, args.rank
    name = args.kernel_case
    gauss = args.projection == "gaussian"
    if name == "sketch":
        X, dY = synthetic.microbatch(WORKLOAD, 0, "q", 0, T, d, k, dev)
        S = torch.zeros((d, r), dtype=torch.float32, device=dev)
        ws = lg.sketch_workspace(T, d, k, r, dev)
        if gauss or args.cache_projection == "on":
            A = lg.logra_regen_projection(100, 0, r, k, lg.LOGRA_PROJ_GAUSS_BF16 if gauss else lg.LOGRA_PROJ_SIGN_BF16)
            fn = lambda: lg.logra_sketch_accumulate_proj(X, dY, S, A, r, ws)  # noqa: E731
        else:
            fn = lambda: lg.logra_sketch_accumulate(X, dY, S, 100, 0, r, ws)  # noqa: E731
        nbytes = 2 * T * (d + k) + 8 * d * r
    elif name == "sketch-group":
        # the seven projections of one 7B layer, one launch per phase
        w7 = synthetic.WORKLOADS["qwen7b"]
        tg = []
        for (nm, dd, kk, sid) in w7["layers"][0]:
            Xj, dYj = synthetic.microbatch("qwen7b", 0, nm, 0, T, dd, kk, dev)
            tg.append((Xj, dYj, torch.zeros((dd, r), dtype=torch.float32, device=dev), 100, sid))
        plan = lg.logra_sketch_group_plan(tg, r)
        fn = lambda: lg.logra_sketch_accumulate_group(plan)  # noqa: E731
        nbytes = sum(2 * T * (dd + kk) + 8 * dd * r for (_, dd, kk, _) in w7["layers"][0])
    elif name == "merge":
        d = 18944  # the gate projection: W (136 MB) is larger than L2
        W = synthetic.weight(WORKLOAD, 0, "gate", d, k, dev)
        S = torch.randn((d, r), device=dev) * 0.1
        if gauss:
            A = lg.logra_regen_projection(100, 0, r, k, lg.LOGRA_PROJ_GAUSS_BF16)
            fn = lambda: lg.logra_merge_update_proj(W, S, A, r, 2e-4)  # noqa: E731
        else:
            fn = lambda: lg.logra_merge_update(W, S, 100, 0, r, 2e-4)  # noqa: E731
        nbytes = 4 * d * k + 4 * d * r
    elif name == "merge-group":
        # one launch over the first two layers of the 1.5B set (14 weights,
        # 185 MB of bf16 weights, larger than L2)
        w15 = synthetic.WORKLOADS["qwen1.5b"]
        mats15 = [(layer, nm, dd, kk, sid) for layer, ms in enumerate(w15["layers"][:2]) for (nm, dd, kk, sid) in ms]
        Ws = [synthetic.weight("qwen1.5b", layer, nm, dd, kk, dev) for (layer, nm, dd, kk, _) in mats15]
        Ss = [torch.randn((dd, r), device=dev) * 0.1 for (_, _, dd, _, _) in mats15]
        plan = lg.logra_merge_group_plan([(W, S, w15["seeds"][layer], sid)
                                          for (layer, _, _, _, sid), W, S in zip(mats15, Ws, Ss)], r)
        fn = lambda: lg.logra_merge_update_group(plan, 2e-4)  # noqa: E731
        nbytes = sum(4 * dd * kk + 4 * dd * r for (_, _, dd, kk, _) in mats15)
    elif name == "norm":
        # squared norm of the gate-shaped bf16 matrix (the diagnostic's ‖R‖²)
        d = 18944
        R = synthetic.weight(WORKLOAD, 0, "gate", d, k, dev)
        out = torch.zeros(1, dtype=torch.float64, device=dev)
        nw = torch.empty(int(lg.lib.logra_sum_squares_workspace_bytes()), dtype=torch.uint8, device=dev)
        fn = lambda: lg.logra_sum_squares(R, out, workspace=nw)  # noqa: E731
        nbytes = 2 * d * k
    elif name == "momentum":
        # the flat buffer of every sketch of the 7B set (Σd = 1,390,592 rows)
        rows_all = sum(m[2] for m in layer_set())
        M = torch.zeros((rows_all, r), device=dev)
        S = torch.randn((rows_all, r), device=dev)
        fn = lambda: lg.logra_sketch_momentum(M, S, 0.9, clear_s=True)  # noqa: E731
        nbytes = 16 * rows_all * r
    else:
        cur, prop = synthetic.kl_logits(KL_WORKLOAD, 0.01, rows=4096, device=dev)
        q = torch.zeros((), dtype=torch.float64, device=dev)
        fn = lambda: lg.logra_predicted_kl(cur, prop, 1.0, q_out=q)  # noqa: E731
        nbytes = 2 * cur.numel() * 2
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    if lg.logra_device_error() != 0:
        raise RuntimeError("device error")
    ms = a.elapsed_time(b) / args.steps
    hbm = _peaks()[0]
    print(json.dumps({"kernel_case": name, "rank": r, "projection": args.projection, "ms": round(ms, 4),
                      "GB_per_s": round(nbytes / ms / 1e6, 1),
                      "hbm_frac": round(nbytes / ms / 1e6 / hbm, 4), "bytes": nbytes}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--rank", type=int, default=64, choices=[4, 16, 64, 256])
    ap.add_argument("--microbatches", type=int, default=None, help="default: the workload's (8 for qwen7b)")
    ap.add_argument("--workload", default="qwen7b", choices=["qwen7b", "qwen1.5b"])
    ap.add_argument("--streams", type=int, default=8)
    ap.add_argument("--share-x", action="store_true",
                    help="q/k/v and gate/up read one shared input per layer (one sketch call per group)")
    ap.add_argument("--projection", default="fixed", choices=["fixed", "refreshed", "gaussian"],
                    help="projection basis: fixed Rademacher (default), refreshed every step, or refreshed Gaussian")
    ap.add_argument("--cache-projection", default="off", choices=["on", "off"],
                    help="on: read the signs as a cached bf16 operand in HBM (a variant; by default every kernel "
                         "rebuilds them on chip and no projection is stored)")
    ap.add_argument("--momentum", type=float, default=None,
                    help="heavy-ball momentum on the sketch (U = M, M = beta*M + S) with this beta")
    ap.add_argument("--sketch", default="group", choices=["streams", "group"],
                    help="the sketch of a micro-batch: one launch per phase over all matrices (a plan) on one "
                         "stream (default), or one call per matrix over --streams worker streams")
    ap.add_argument("--merge", default="auto", choices=["auto", "group", "per-weight"],
                    help="merge every weight in one launch over a plan, or one launch per weight (auto: one launch "
                         "when the mean weight holds fewer than 2^24 elements)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="end-to-end steps (default: as many as --steps, capped near a minute)")
    ap.add_argument("--no-r256", action="store_true",
                    help="skip the r = 256 phases timed after the main rank (7B set)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-autograd", action="store_true",
                    help="skip the autograd-driven sketch (SketchedLinearGroup backward into a SketchBatch)")
    ap.add_argument("--autograd-microbatches", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=30.0)
    ap.add_argument("--kernel-case", choices=["sketch", "sketch-group", "merge", "merge-group", "kl", "momentum", "norm"],
                    default=None,
                    help="time one kernel on one 7B-set shape (sketch-group: the seven matrices of one layer; "
                         "merge-group: one launch over two layers of the 1.5B set) instead of the step (for "
                         "profiling)")
    args = ap.parse_args()
    global WORKLOAD
    WORKLOAD = args.workload
    if args.microbatches is None:
        args.microbatches = synthetic.WORKLOADS[WORKLOAD]["microbatches"]
    if args.kernel_case:
        run_kernel_case(args)
        return
    if args.share_x and args.sketch == "group":
        args.sketch = "streams"  # the shared-input calls run per unit over the worker streams
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
