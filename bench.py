#!/usr/bin/env python3
"""Benchmark of the decode-FFN weight stream on GB300 (one JSON line on stdout).

Default workload (--workload stack52_m1): one decode token through a 52-layer
FFN stack of the Muser book's model shape (hidden 6656, FFN 19968).  Per layer:
input RMSNorm (layer 0 only) -> Q4_K gate/up 19968x6656 with SiLU gating ->
Q6_K down 6656x19968 with the dual-eps fused tail.  A step streams the 52
layers' 13.44 GB of distinct weights (far larger than the 129 MB L2).
`--workload stack52_m16` runs the same stack at M = 16 (speculative verify).
`--workload attn52_m1` / `attn52_m16` run the attention side of the same
layers (Q, K, V, gate projections; o_proj with the first dual-eps tail).
`--workload lmhead_m1` runs the LM head (202,048 x 6,656 Q6_K, soft cap).
`--workload down_tail_q4k` / `down_tail_q6k` chain 52 instances of the
standalone down projection + dual-eps tail (Q4_K or Q6_K W_down 6656x19968);
`matvec_q5k` chains 52 plain Q5_K matvecs of the same shape.
`--workload kv_restore` restores one session's K/V planes at 130,815 tokens
(13 head-major NoPE planes, 39 wrapped 2,048-row SWA rings) from detached rows.

Arms:
  --impl native     libmuser (CUDA, sm_103a) through its C ABI.
  --impl reference  the fp64 CPU oracle on the host cores (a bounded row
                    sample of the same workload per step) -- the only other
                    place this script runs oracle/ besides the cpu_baseline leg.

Multi-GPU (torchrun): replicas only -- every rank runs the whole workload on
its own GPU; the value is the sum over ranks, timed by the slowest rank.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import shutil
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

H, F, NL = synth.HIDDEN, synth.FFN, synth.N_LAYERS
Q4K_MAT = H * (F // 256) * 144          # 74,760,192 B (gate or up; same count as Q4_K down)
Q6K_MAT = H * (F // 256) * 210          # 109,025,280 B
LAYER_W = 2 * Q4K_MAT + Q6K_MAT         # 258,545,664 B
PROBES = 4                              # layers per step whose two launches are event-timed
METRIC = "weight-stream GB/s (% of GB300 HBM peak); decode FFN tokens/sec, 1 GPU"

# ncu DRAM traffic of the dominant kernel, per launch, with the source hash it
# was captured on (profiles/ summary); reported as null once the kernel changed.
# The capture ran 4 layers; the traffic per layer is the same, so the 52-layer
# launch's figure is 13 x the captured launch's.
NCU_TRAFFIC = {"kernel": "mvs_kernel<Q4_K,Q6_K>", "bytes_per_launch": 13 * 1038162688, "layers": 52,
               "captured_layers": 4,
               "source_sha256": "064b9000264b591a7c1ed77c6aad4184a76070b4220ccd0c527787d0430ed589",
               "profile": "profiles/mvs_stack_m1_4layers.md"}


def _env_int(k, d):
    try:
        return int(os.environ.get(k, d))
    except ValueError:
        return d


def max_over_ranks(value: float, dist, device="cuda") -> float:
    """The slowest rank's figure: with a process group every rank gets the
    maximum over ranks (an all-reduce MAX); alone, the value itself."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_rank: int, ms: float) -> float:
    """Replicas: every rank streams `bytes_per_rank` per step; the job's rate
    is all ranks' bytes over the slowest rank's step time."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


def algorithmic_bytes(M: int):
    """Per layer and per kernel: weights read + activations read/written (f32).

    M = 1 runs each layer's tail inside the next layer's gate/up kernel:
    (gate/up with the previous tail, plain down projection) per layer, and
    the entry norm plus the last tail once per step.  M = 16 runs (gate/up,
    down + tail) per layer and the entry norm once."""
    if M == 1:
        gate_up = 2 * Q4K_MAT + 4 * H * 6 + 4 * F  # Wg, Wu; p, r in/out, w1, w2, x out; mid out
        down = Q6K_MAT + 4 * F + 4 * H             # Wd, mid in, proj out
        entry = 4 * H * 3 + 4 * H * 6              # rms_norm (r, w, x); the last tail (p, r r/w, w1, w2, out)
        return gate_up, down, entry
    gate_up = 2 * Q4K_MAT + 4 * M * H + 4 * M * F           # Wg, Wu, x in, mid out
    down_tail = Q6K_MAT + 4 * M * F + 4 * M * H * 5 + 4 * 2 * H  # Wd, mid, proj w, p r, r r/w, out w, w1/w2
    entry = 4 * M * H * 2 + 4 * H
    return gate_up, down_tail, entry


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# Sources that define the persistent stack kernel (mvs): a change to any of
# them makes the recorded DRAM traffic stale.
MVS_SOURCES = ("common.cuh", "kernels.cuh", "mv1_core.cuh", "mvs.cu")


def source_sha():
    h = hashlib.sha256()
    for f in MVS_SOURCES:
        with open(os.path.join(ROOT, "quantized_weight_streaming_q4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.gpu_id = gpu_id
        self.path = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="muser_clocks_", suffix=".csv")
        os.close(fd)
        cmd = [exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        self.fh = open(self.path, "w")
        self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- native
def make_layers(n_layers: int, seed: int = 0, workload: int = 4):
    """The stack's seeded weights on the device: per layer Wg, Wu (Q4_K), Wd
    (Q6_K), the post-FFN norm w1 and the next norm (the next layer's input
    norm) w_next."""
    import torch
    layers = []
    for l in range(n_layers):
        Ld = synth.ffn_layer(l, H, F, seed=seed, workload=workload)
        d = {k: torch.from_numpy(v).cuda() for k, v in Ld.items()}
        d["w_next"] = torch.from_numpy(synth.input_norm_weight(l + 1, H, seed=seed, workload=workload)).cuda()
        layers.append(d)
    return layers


class NativeStack:
    """The workload on the GPU, driven through libmuser's C ABI."""

    def __init__(self, M: int, layers, seed: int = 0, workload: int = 4):
        import torch
        import quantized_weight_streaming_q4_gb300 as mu
        self.torch, self.mu, self.M, self.nl = torch, mu, M, len(layers)
        self.L = mu.lib()
        self.layers = layers
        self.structs = [mu.FfnLayer(d["Wg"].data_ptr(), d["Wu"].data_ptr(), d["Wd"].data_ptr(),
                                    d["w1"].data_ptr(), d["w_next"].data_ptr(), mu.MUSER_Q4_K, mu.MUSER_Q6_K)
                        for d in layers]
        self.w_in = torch.from_numpy(synth.input_norm_weight(0, H, seed=seed, workload=workload)).cuda()
        self.r0 = synth.residual_rows(M, H, seed=seed, workload=workload)
        self.resid = torch.from_numpy(self.r0).cuda()
        self.out = torch.empty(M, H, dtype=torch.float32, device="cuda")
        self.x = [torch.empty(M, H, dtype=torch.float32, device="cuda") for _ in range(2)]
        self.mid = torch.empty(M, F, dtype=torch.float32, device="cuda")
        self.proj = torch.empty(M, H, dtype=torch.float32, device="cuda")
        # the per-layer path relays the residual between two rows (each fused
        # boundary reads one and writes the other through residual_out)
        self.resid_b = torch.empty_like(self.resid)
        self.gu_scratch_bytes = mu.muser_gate_up_scratch_bytes(mu.MUSER_Q4_K, F, H, M)
        self.gu_scratch = torch.zeros(max(self.gu_scratch_bytes, 16) // 4, dtype=torch.float32, device="cuda")
        self.scratch_bytes = mu.muser_scratch_bytes(H, M)
        self.scratch = torch.zeros(self.scratch_bytes // 4 + 64, dtype=torch.float32, device="cuda")
        wsb = mu.muser_ffn_workspace_bytes(H, F, M)
        self.ws = torch.zeros(wsb // 4 + 64, dtype=torch.float32, device="cuda")
        self.wsb = wsb
        self.stream = torch.cuda.current_stream()
        self.sh = self.stream.cuda_stream
        self.arr = (mu.FfnLayer * self.nl)(*self.structs)
        # launches of one per-layer step: the entry norm, two per layer, and
        # (M = 1) the last tail on its own
        self.per_layer_launches = 1 + 2 * self.nl + (1 if M == 1 else 0)

    def _rc(self, name, rc):
        if rc != 0:
            raise RuntimeError(f"{name}: {self.mu.muser_last_error()}")

    def step_public(self):
        """One token (M rows) through every layer: the public one-call entry point."""
        self._rc("ffn_stack", self.L.muser_ffn_stack(
            self.arr, self.nl, self.w_in.data_ptr(), H, F, self.M, self.resid.data_ptr(),
            self.out.data_ptr(), 1e-5, 1e-8, self.ws.data_ptr(), self.wsb, self.sh))

    def step_layers(self, events=None):
        """The same token as per-layer calls.  `events` maps a few layers to an
        event triple that brackets their gate/up and down launches (the others
        run back to back, overlapped by PDL)."""
        if self.M == 1:
            return self._layers_m1(events)
        L, M, sh = self.L, self.M, self.sh
        self._rc("rms_norm", L.muser_rms_norm(self.resid.data_ptr(), self.w_in.data_ptr(),
                                              self.x[0].data_ptr(), H, M, 1e-5, sh))
        x, xn = self.x[0], self.x[1]
        for l, d in enumerate(self.layers):
            ev = events.get(l) if events is not None else None
            if ev is not None:
                ev[0].record(self.stream)
            self._rc("gate_up", L.muser_ffn_gate_up_silu_scratch(
                12, d["Wg"].data_ptr(), d["Wu"].data_ptr(), F, H, x.data_ptr(), M, self.mid.data_ptr(),
                self.gu_scratch.data_ptr(), self.gu_scratch_bytes, sh))
            if ev is not None:
                ev[1].record(self.stream)
            dst = self.out if l == self.nl - 1 else xn
            self._rc("down_tail", L.muser_qmatvec_residual_dual_rmsnorm(
                14, d["Wd"].data_ptr(), H, F, self.mid.data_ptr(), M, self.proj.data_ptr(),
                self.resid.data_ptr(), dst.data_ptr(), d["w1"].data_ptr(), d["w_next"].data_ptr(),
                1e-8, 1e-5, self.scratch.data_ptr(), self.scratch_bytes, sh))
            if ev is not None:
                ev[2].record(self.stream)
            x, xn = xn, x

    def _layers_m1(self, events=None):
        """One row of x as per-layer calls: the entry norm, then per layer
        gate/up (with the previous layer's tail fused in, from layer 1, its
        residual relayed to the other row) and the plain down projection, then
        the last layer's tail, in place on the row the relay ended in, which it
        copies back to self.resid when that is the other row."""
        L, M, sh = self.L, self.M, self.sh
        self._rc("rms_norm", L.muser_rms_norm(self.resid.data_ptr(), self.w_in.data_ptr(),
                                              self.x[0].data_ptr(), H, M, 1e-5, sh))
        rows = (self.resid, self.resid_b)
        cur = 0
        prev = None
        for l, d in enumerate(self.layers):
            ev = events.get(l) if events is not None else None
            if ev is not None:
                ev[0].record(self.stream)
            if prev is None:
                self._rc("gate_up", L.muser_ffn_gate_up_silu(
                    12, d["Wg"].data_ptr(), d["Wu"].data_ptr(), F, H, self.x[0].data_ptr(), M,
                    self.mid.data_ptr(), sh))
            else:
                self._rc("gate_up_tail", L.muser_ffn_gate_up_silu_tail(
                    12, d["Wg"].data_ptr(), d["Wu"].data_ptr(), F, H, self.proj.data_ptr(),
                    rows[cur].data_ptr(), rows[1 - cur].data_ptr(), prev["w1"].data_ptr(),
                    prev["w_next"].data_ptr(), 1e-8, 1e-5, self.x[1].data_ptr(), M, self.mid.data_ptr(),
                    None, 0, sh))
                cur = 1 - cur
            if ev is not None:
                ev[1].record(self.stream)
            self._rc("down", L.muser_qmatvec(14, d["Wd"].data_ptr(), H, F, self.mid.data_ptr(), M,
                                             self.proj.data_ptr(), sh))
            if ev is not None:
                ev[2].record(self.stream)
            prev = d
        self._rc("tail", L.muser_fused_residual_dual_rmsnorm(
            rows[cur].data_ptr(), self.proj.data_ptr(), self.out.data_ptr(), prev["w1"].data_ptr(),
            prev["w_next"].data_ptr(), H, M, 1e-8, 1e-5, sh))
        if cur:
            self.resid.copy_(self.resid_b)


NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal (context beside the measured copy peak)
REPS = 5                   # counted repetitions of the timed region (mean and coefficient of variation)


def timed_reps(stream, steps: int, fn):
    """Time exactly `steps` calls of fn() on `stream`, split into up to REPS
    consecutive repetitions bracketed by CUDA events (no synchronisation
    between them).  Returns (total ms, per-rep ms per step)."""
    import torch
    nrep = max(1, min(REPS, steps))
    sizes = [steps // nrep + (1 if r < steps % nrep else 0) for r in range(nrep)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(nrep + 1)]
    ev[0].record(stream)
    for r, n in enumerate(sizes):
        for _ in range(n):
            fn()
        ev[r + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[r].elapsed_time(ev[r + 1]) / n for r, n in enumerate(sizes)]
    return ev[0].elapsed_time(ev[-1]), per


def rep_stats(per):
    m = statistics.mean(per)
    cv = statistics.pstdev(per) / m if len(per) > 1 and m > 0 else 0.0
    return {"reps": len(per), "ms_per_step_mean": round(m, 4), "cv": round(cv, 4),
            "ms_per_step_each": [round(v, 4) for v in per]}


def gpu_uuid():
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        return None


def measure_stack(S, steps: int, warmup: int, barrier, with_probes: bool = True):
    """The headline, probe-free: `steps` tokens through muser_ffn_stack after
    `warmup`, then a separate probe pass (per-launch events, per-layer event
    triples) and the end-to-end pass with host copies."""
    import torch
    M, nl = S.M, S.nl
    for _ in range(warmup):
        S.step_public()
    barrier()
    clocks = ClockSampler(gpu_uuid())
    clocks.start()
    time.sleep(0.3)
    barrier()
    total_ms, per = timed_reps(S.stream, steps, S.step_public)
    barrier()
    clock = clocks.stop()
    res = {"ms": total_ms / steps, "reps": rep_stats(per), "clocks": clock}
    if with_probes:
        # one stack call per event pair: the duration of the whole call
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(max(3, min(steps, 10)))]
        for a, b in pairs:
            a.record(S.stream)
            S.step_public()
            b.record(S.stream)
        barrier()
        res["call_ms"] = statistics.mean(a.elapsed_time(b) for a, b in pairs)
        # per-layer composition, PROBES layers per step bracketed by event triples
        probes = min(PROBES, nl)
        for _ in range(2):
            S.step_layers()
        evs = []
        for k in range(max(3, min(steps, 10))):
            ls = sorted({(k + j * max(1, nl // probes)) % nl for j in range(probes)})
            evs.append({l: [torch.cuda.Event(enable_timing=True) for _ in range(3)] for l in ls})
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(S.stream)
        for e in evs:
            S.step_layers(e)
        t1.record(S.stream)
        barrier()
        res["layers_ms"] = t0.elapsed_time(t1) / len(evs)
        res["gu_ms"] = statistics.mean(t[0].elapsed_time(t[1]) for e in evs for t in e.values())
        res["dn_ms"] = statistics.mean(t[1].elapsed_time(t[2]) for e in evs for t in e.values())
    # e2e: host residual in (pinned), the public call, host output out
    h_in = torch.from_numpy(S.r0.copy()).pin_memory()
    h_out = torch.empty(M, H, dtype=torch.float32).pin_memory()

    def e2e_step():
        S.resid.copy_(h_in, non_blocking=True)
        S.step_public()
        h_out.copy_(S.out, non_blocking=True)
    for _ in range(max(1, min(3, warmup))):
        e2e_step()
    barrier()
    e_total, _ = timed_reps(S.stream, steps, e2e_step)
    barrier()
    assert np.isfinite(h_out.numpy()).all()
    res["e2e_ms"] = e_total / steps
    return res


def run_native(args, rank, world):
    import torch
    import quantized_weight_streaming_q4_gb300 as mu
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
        dist.init_process_group("nccl")
    mu.build()
    M = 16 if args.workload == "stack52_m16" else 1
    nl = args.layers
    t0 = time.time()
    layers = make_layers(nl)
    gen_s = time.time() - t0
    S = NativeStack(M, layers)
    gu_bytes, dt_bytes, entry_bytes = algorithmic_bytes(M)
    step_bytes = nl * (gu_bytes + dt_bytes) + entry_bytes
    weight_bytes = nl * LAYER_W

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    r = measure_stack(S, args.steps, args.warmup, barrier)
    ms = max_over_ranks(r["ms"], dist)
    e2e_ms = max_over_ranks(r["e2e_ms"], dist)
    status = mu.muser_device_status()
    peak, peak_kind = read_peaks()
    one_launch = S.L.muser_ffn_stack_launches(S.arr, nl, H, F, M)
    # the dominant kernel: the whole stack when one launch carries it, else the gate/up kernel
    if M == 1 and one_launch == 1:
        kname = "muser_ffn_stack (the persistent one-token stack kernel: every layer's gate/up, down and tail)"
        k_bytes, k_ms = step_bytes, r["call_ms"]
    elif M == 1:
        kname = ("muser_ffn_gate_up_silu_tail (mv1 Q4_K gate+up, previous layer's dual-eps tail in the prologue, "
                 "SiLU epilogue)")
        k_bytes, k_ms = gu_bytes, r["gu_ms"]
    else:
        kname = "muser_ffn_gate_up_silu_scratch (mvt Q4_K gate+up, SiLU epilogue)"
        k_bytes, k_ms = gu_bytes, r["gu_ms"]
    achieved = k_bytes / (k_ms * 1e-3) / 1e9
    traffic = None
    if (M == 1 and one_launch == 1 and nl == NCU_TRAFFIC["layers"] and
            NCU_TRAFFIC["source_sha256"] == source_sha()):
        traffic = NCU_TRAFFIC["bytes_per_launch"]
    gbs = whole_job_gbs(world, weight_bytes, ms)
    result = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("f32 activations in and out, exact f32 dequantised weights; inside the kernels x is held as "
                  + ("24-bit block fixed point (dp4a digits, <= 2^-23 of each 64-input slice's max)" if M == 1 else
                     "two binary16 parts per super-block (<= 2^-22 of the block max) for the tensor cores")),
        "data": "synthetic (seeded; Q4_K/Q6_K fields and activations drawn per the workload recipe)",
        "config": {
            "workload": f"decode-FFN stack: {nl} layers x [rms_norm(layer 0) -> Q4_K gate/up {F}x{H} + SiLU "
                        f"-> Q6_K down {H}x{F} + dual-eps tail], M={M}",
            "api": "muser_ffn_stack, one C call per token (device-resident input)",
            "layers": nl, "hidden": H, "ffn": F, "M": M,
            "weight_bytes_per_step": weight_bytes,
            "algorithmic_bytes_per_step": step_bytes,
            "l2": f"inputs larger than L2: {weight_bytes / 1e9:.2f} GB of distinct weights per step vs 129 MB L2",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "tokens_per_s": round(world * M / (ms * 1e-3), 3),
        "hbm_frac_of_" + peak_kind: round(gbs / world / peak, 4),
        "hbm_frac_of_nominal_8000": round(gbs / world / NOMINAL_HBM_GBS, 4),
        "repetitions": r["reps"],
        "roofline": {
            "bound": "hbm",
            "kernel": kname,
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": (f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                          else "fallback 6.8 TB/s"),
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "frac_of_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": k_bytes,
            "mean_launch_us": round(k_ms * 1e3, 2),
            "timing": "CUDA events around each launch in a probe pass after the timed region",
        },
        "per_layer_calls": {
            "ms_per_step": round(r["layers_ms"], 4),
            "value": round(weight_bytes / (r["layers_ms"] * 1e-3) / 1e9, 2),
            "gate_up": {"name": ("muser_ffn_gate_up_silu[_tail] (mv1)" if M == 1 else
                                 "muser_ffn_gate_up_silu_scratch (mvt)"),
                        "mean_launch_us": round(r["gu_ms"] * 1e3, 2),
                        "achieved_gbs": round(gu_bytes / (r["gu_ms"] * 1e-3) / 1e9, 1),
                        "algorithmic_bytes_per_launch": gu_bytes},
            "down": {"name": ("muser_qmatvec (mv1 Q6_K)" if M == 1 else
                              "muser_qmatvec_residual_dual_rmsnorm (mvt Q6_K + tail)"),
                     "mean_launch_us": round(r["dn_ms"] * 1e3, 2),
                     "achieved_gbs": round(dt_bytes / (r["dn_ms"] * 1e-3) / 1e9, 1),
                     "algorithmic_bytes_per_launch": dt_bytes},
            "timing": "probe pass: event triples around 4 layers per step (they stop PDL overlap there)",
        },
        "e2e": {"value": round(whole_job_gbs(world, weight_bytes, e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": 4 * M * H,
                "d2h_bytes_per_step": 4 * M * H,
                "api": ("muser_ffn_stack, one C call per token on device buffers; the residual row is copied in "
                        "from pinned host memory and the output row out (torch copies on the same stream)")},
        "gpu_launches": args.steps * one_launch,
        "clocks": r["clocks"],
        "device_status": status,
        "weights_generation_s": round(gen_s, 1),
    }
    if M == 1 and not args.no_sub and world == 1:
        # config 4 (16 rows, speculative-verify shape) through the same weights
        S16 = NativeStack(16, layers)
        r16 = measure_stack(S16, max(3, min(args.steps, 8)), 3, barrier)
        g16, d16, e16 = algorithmic_bytes(16)
        result["sub_results"] = [{
            "workload": f"decode-FFN stack: {nl} layers, M=16 (speculative-verify shape), same weights",
            "value": round(weight_bytes / (r16["ms"] * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(r16["ms"], 4), "row_tokens_per_s": round(16 / (r16["ms"] * 1e-3), 1),
            "hbm_frac_of_" + peak_kind: round(weight_bytes / (r16["ms"] * 1e-3) / 1e9 / peak, 4),
            "repetitions": r16["reps"],
            "gate_up": {"mean_launch_us": round(r16["gu_ms"] * 1e3, 2),
                        "achieved_gbs": round(g16 / (r16["gu_ms"] * 1e-3) / 1e9, 1)},
            "down_tail": {"mean_launch_us": round(r16["dn_ms"] * 1e3, 2),
                          "achieved_gbs": round(d16 / (r16["dn_ms"] * 1e-3) / 1e9, 1)},
            "e2e": {"value": round(weight_bytes / (r16["e2e_ms"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "ms_per_step": round(r16["e2e_ms"], 4)},
            "clocks": r16["clocks"]}]
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return result


# ------------------------------------------------------------- CPU oracle
def _oracle_layer_sample(frac_rows: float, seed=0):
    """A bounded sample of one layer: the first rows of gate/up/down, the
    norm vectors and a residual row."""
    wl = 4
    rg = max(8, int(F * frac_rows))
    rd = max(8, int(H * frac_rows))
    Wg = synth.q4k_matrix(F, H, seed=seed, workload=wl, layer=0, tensor=synth.T_GATE)[:rg]
    Wu = synth.q4k_matrix(F, H, seed=seed, workload=wl, layer=0, tensor=synth.T_UP)[:rg]
    Wd = synth.q6k_matrix(H, F, seed=seed, workload=wl, layer=0, tensor=synth.T_DOWN)[:rd]
    return {"Wg": np.ascontiguousarray(Wg), "Wu": np.ascontiguousarray(Wu), "Wd": np.ascontiguousarray(Wd),
            "rg": rg, "rd": rd, "r": synth.residual_rows(1, H, seed=seed, workload=wl),
            "w_in": synth.input_norm_weight(0, H, seed=seed, workload=wl),
            "w1": synth.norm_weight(H, seed=seed, workload=wl, tensor=synth.T_W1),
            "w2": synth.input_norm_weight(1, H, seed=seed, workload=wl),
            "p": synth.normal((1, H), seed=3) * np.float32(2.5e6), "mid": synth.normal((1, F), seed=2)}


def _oracle_step(oracle, s):
    """One sampled pass of the whole path in the oracle: the input norm, the
    sampled gate/up rows and SiLU, the sampled down rows (on a full-length
    intermediate row) and the dual-eps tail.  Returns the weight bytes read."""
    x = oracle.rms_norm(s["r"], s["w_in"], 1e-5)
    g = oracle.qmatvec("q4_k", s["Wg"], s["rg"], H, x)
    u = oracle.qmatvec("q4_k", s["Wu"], s["rg"], H, x)
    oracle.silu_mul(g, u)
    oracle.qmatvec("q6_k", s["Wd"], s["rd"], F, s["mid"])
    oracle.dual_tail(s["r"], s["p"], s["w1"], s["w2"], 1e-8, 1e-5)
    return s["Wg"].nbytes + s["Wu"].nbytes + s["Wd"].nbytes


def _time_oracle(oracle, s, seconds: float):
    nbytes, t_tot, reps = 0, 0.0, 0
    while t_tot < seconds or reps < 1:
        t0 = time.perf_counter()
        nbytes += _oracle_step(oracle, s)
        t_tot += time.perf_counter() - t0
        reps += 1
    return nbytes / t_tot / 1e9, reps, t_tot


def cpu_baseline(seconds: float, frac_rows: float = 0.125):
    """The fp64 oracle on the host cores: all cores (OpenMP over output rows)
    and one core, each about `seconds` of work on a bounded row sample of one
    layer, scaled to GB/s of weights."""
    import oracle
    s = _oracle_layer_sample(frac_rows)
    nthreads = oracle.num_threads()
    gbs, reps, t_tot = _time_oracle(oracle, s, seconds)
    oracle.set_num_threads(1)
    try:
        gbs1, reps1, t1 = _time_oracle(oracle, s, seconds / 2)
    finally:
        oracle.set_num_threads(nthreads)
    wmb = (s["Wg"].nbytes + s["Wu"].nbytes + s["Wd"].nbytes) / 1e6
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "tokens_per_s": round(gbs * 1e9 / (NL * LAYER_W), 6),
            "sample": f"{reps} passes of the fp64 oracle over one layer's path: input rms_norm, the first "
                      f"{frac_rows:.3f} of the gate/up rows + SiLU and of the down rows ({wmb:.1f} MB of weights), "
                      f"the dual-eps tail; {t_tot:.1f} s",
            "one_core": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                         "tokens_per_s": round(gbs1 * 1e9 / (NL * LAYER_W), 6),
                         "sample": f"{reps1} passes of the same sample on one thread, {t1:.1f} s"}}


QD, KVD = synth.Q_DIM, synth.KV_DIM
ATTN_W = (2 * QD + 2 * KVD) * (H // 256) * 144 + H * (QD // 256) * 144  # Q, K, V, gate, o_proj (Q4_K)


def run_attn(args, rank, world):
    """The attention-side weight stream of one decode token through the
    layers (Ch 10 Figure 10.1 boxes 4, 9, 10): per layer the Q, K, V and gate
    projections as one group (muser_qmatvec_group; from layer 1 with the
    previous layer's post-attention tail fused in, muser_qmatvec_group_tail),
    then o_proj (muser_qmatvec); the last tail once per step.  With 16 rows
    of x the group is one tensor-core launch split over every SM (from layer
    1 muser_qmatvec_group_tail, whose tail also builds the launch's B image)
    and o_proj a muser_qmatvec_scratch call.  The tail's
    output (the FFN input in the model) stands in for the next layer's normed
    input.  Attention itself is outside the path: o_proj reads a seeded
    stand-in for its output."""
    import torch
    import quantized_weight_streaming_q4_gb300 as mu
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
        dist.init_process_group("nccl")
    mu.build()
    L = mu.lib()
    M = 16 if args.workload == "attn52_m16" else 1
    nl, wl = args.layers, synth.ATTN_WORKLOAD
    t0 = time.time()
    layers = []
    for l in range(nl):
        A = synth.attn_layer(l, H)
        d = {k: torch.from_numpy(v).cuda() for k, v in A.items()}
        d["w_ffn"] = torch.from_numpy(synth.input_norm_weight(l + 1, H, workload=wl)).cuda()
        layers.append(d)
    gen_s = time.time() - t0
    w_in = torch.from_numpy(synth.input_norm_weight(0, H, workload=wl)).cuda()
    r0 = synth.residual_rows(M, H, workload=wl)
    resid = torch.from_numpy(r0).cuda()
    attn = torch.from_numpy(synth.attn_output(M)).cuda()
    x = torch.empty(M, H, dtype=torch.float32, device="cuda")
    q, g = (torch.empty(M, QD, dtype=torch.float32, device="cuda") for _ in range(2))
    k, v = (torch.empty(M, KVD, dtype=torch.float32, device="cuda") for _ in range(2))
    proj = torch.empty(M, H, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def rc(name, r):
        if r != 0:
            raise RuntimeError(f"{name}: {mu.muser_last_error()}")

    rows4 = (ctypes.c_int64 * 4)(QD, KVD, KVD, QD)
    ys4 = (ctypes.c_void_p * 4)(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr())
    w4 = [(ctypes.c_void_p * 4)(*[d[n].data_ptr() for n in ("Wq", "Wk", "Wv", "Wg")]) for d in layers]
    nscr = max([mu.muser_qmatvec_scratch_bytes(12, r, c, M) for r, c in ((QD, H), (KVD, H), (H, QD))] +
               [L.muser_qmatvec_group_scratch_bytes(12, 4, rows4, H, M)])
    scratch = torch.zeros(max(nscr, 16) // 4 + 64, dtype=torch.float32, device="cuda")
    outs4 = (q, k, v, g)
    # one row of x: each fused boundary reads the residual from one row and
    # writes it to the other (residual_out); the step ends in the row it
    # reached, which the next step starts from
    rows_r = (resid, torch.empty_like(resid))
    cur = [0]

    def split_mv(W, rows, cols, xin, y):
        rc("qmatvec_scratch", L.muser_qmatvec_scratch(12, W.data_ptr(), rows, cols, xin.data_ptr(), M, y.data_ptr(),
                                                      scratch.data_ptr(), nscr, sh))

    def step(events=None):
        r = rows_r[cur[0]]
        rc("rms_norm", L.muser_rms_norm(r.data_ptr(), w_in.data_ptr(), x.data_ptr(), H, M, 1e-5, sh))
        prev = None
        for l, d in enumerate(layers):
            ev = events.get(l) if events is not None else None
            if ev is not None:
                ev[0].record(stream)
            if M > 1:
                # Q, K, V and gate as one tensor-core launch on the shared x;
                # from layer 1 after the previous tail (in place), which also
                # builds that launch's B image
                if prev is None:
                    rc("qkvg", L.muser_qmatvec_group_scratch(12, 4, w4[l], rows4, H, x.data_ptr(), M, ys4,
                                                             scratch.data_ptr(), nscr, sh))
                else:
                    rc("qkvg_tail", L.muser_qmatvec_group_tail(
                        12, 4, w4[l], rows4, H, proj.data_ptr(), r.data_ptr(), None, prev["w_post"].data_ptr(),
                        prev["w_ffn"].data_ptr(), 1e-8, 1e-5, x.data_ptr(), M, ys4, scratch.data_ptr(), nscr, sh))
            elif prev is None:
                rc("qkvg", L.muser_qmatvec_group(12, 4, w4[l], rows4, H, x.data_ptr(), M, ys4, sh))
            else:
                cur[0] = 1 - cur[0]
                r_next = rows_r[cur[0]]
                rc("qkvg_tail", L.muser_qmatvec_group_tail(
                    12, 4, w4[l], rows4, H, proj.data_ptr(), r.data_ptr(), r_next.data_ptr(),
                    prev["w_post"].data_ptr(), prev["w_ffn"].data_ptr(), 1e-8, 1e-5, x.data_ptr(), M, ys4,
                    None, 0, sh))
                r = r_next
            if ev is not None:
                ev[1].record(stream)
            if M > 1:
                split_mv(d["Wo"], H, QD, attn, proj)
            else:
                rc("o_proj", L.muser_qmatvec(12, d["Wo"].data_ptr(), H, QD, attn.data_ptr(), M, proj.data_ptr(),
                                             sh))
            if ev is not None:
                ev[2].record(stream)
            prev = d
        rc("tail", L.muser_fused_residual_dual_rmsnorm(r.data_ptr(), proj.data_ptr(), x.data_ptr(),
                                                       prev["w_post"].data_ptr(), prev["w_ffn"].data_ptr(),
                                                       H, M, 1e-8, 1e-5, sh))

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    barrier()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    barrier()
    # the headline: the steps alone, nothing recorded between their launches
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for kk in range(args.steps):
        step()
    t_end.record(stream)
    barrier()
    ms = t_start.elapsed_time(t_end) / args.steps
    clock = clocks.stop()
    ms = max_over_ranks(ms, dist)
    # a separate probe pass: event triples around PROBES layers per step (they
    # stop the programmatic overlap at the probed launches)
    probes = min(PROBES, nl)
    events = []
    for kk in range(args.steps):
        ls = sorted({(kk + j * max(1, nl // probes)) % nl for j in range(probes)})
        events.append({l: [torch.cuda.Event(enable_timing=True) for _ in range(3)] for l in ls})
    for kk in range(args.steps):
        step(events[kk])
    barrier()
    q_ms = statistics.mean(t[0].elapsed_time(t[1]) for ev in events for t in ev.values())
    o_ms = statistics.mean(t[1].elapsed_time(t[2]) for ev in events for t in ev.values())
    # e2e: the same calls with the residual in from pinned host memory and x out
    h_in = torch.from_numpy(r0.copy()).pin_memory()
    h_out = torch.empty(M, H, dtype=torch.float32).pin_memory()
    for _ in range(max(1, min(3, args.warmup))):
        rows_r[cur[0]].copy_(h_in, non_blocking=True)
        step()
        h_out.copy_(x, non_blocking=True)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        rows_r[cur[0]].copy_(h_in, non_blocking=True)
        step()
        h_out.copy_(x, non_blocking=True)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    assert np.isfinite(h_out.numpy()).all()
    peak, peak_kind = read_peaks()
    weight_bytes = nl * ATTN_W
    # the group with the previous tail: four matrices; p, r in/out, w1, w2, x out; four outputs
    q_bytes = (2 * QD + 2 * KVD) * (H // 256) * 144 + 4 * M * H * 6 + 4 * M * (2 * QD + 2 * KVD)
    o_bytes = H * (QD // 256) * 144 + 4 * M * QD + 4 * M * H
    gbs = whole_job_gbs(world, weight_bytes, ms)
    achieved = q_bytes / (q_ms * 1e-3) / 1e9
    return {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Q4_K fields per the workload recipe; a seeded stand-in for the attention output)",
        "config": {"workload": f"attention-side weight stream: {nl} layers x [previous dual-eps tail -> Q {QD}x{H}, "
                               f"K {KVD}x{H}, V {KVD}x{H}, gate {QD}x{H} (Q4_K) -> o_proj {H}x{QD} (Q4_K)], M={M}",
                   "layers": nl, "hidden": H, "M": M, "weight_bytes_per_step": weight_bytes,
                   "l2": f"inputs larger than L2: {weight_bytes / 1e9:.2f} GB of distinct weights per step vs 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tokens_per_s": round(world * M / (ms * 1e-3), 3),
        "hbm_frac_of_" + peak_kind: round(gbs / world / peak, 4),
        "roofline": {"bound": "hbm", "kernel": ("muser_qmatvec_group_tail (Q, K, V, gate Q4_K with the previous "
                                                "tail: one launch)" if M == 1 else
                                                f"muser_qmatvec_group_tail: the previous tail with the B image of its "
                                                f"output, then Q, K, V, gate as one tensor-core launch (units split "
                                                f"over the SMs), M={M}"),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None, "algorithmic_bytes_per_launch": q_bytes, "mean_launch_us": round(q_ms * 1e3, 2),
                     "timing": "probe pass after the timed region: event triples around 4 layers per step",
                     "second_kernel": {"name": "muser_qmatvec (o_proj)" if M == 1 else
                                               "muser_qmatvec_scratch (o_proj)",
                                       "achieved_gbs": round(o_bytes / (o_ms * 1e-3) / 1e9, 1),
                                       "mean_launch_us": round(o_ms * 1e3, 2),
                                       "algorithmic_bytes_per_launch": o_bytes}},
        "e2e": {"value": round(whole_job_gbs(world, weight_bytes, e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": 4 * M * H, "d2h_bytes_per_step": 4 * M * H,
                "api": ("per-layer muser_qmatvec_group[_tail] / muser_qmatvec calls" if M == 1 else
                        "per-layer muser_qmatvec_group_tail and muser_qmatvec_scratch calls") +
                       ", host residual in, x out"},
        # M = 16: the entry norm; layer 0 the grouped Q/K/V/gate launch (1,768 units, above 8 per CTA: its B
        # image built before it and cleared after, three launches), later layers the tail that also builds the
        # image, the grouped launch and the clear; o_proj (832 units, one launch) per layer; the last tail
        "gpu_launches": args.steps * ((2 + 2 * nl) if M == 1 else (2 + 4 * nl)),
        "clocks": clock, "device_status": mu.muser_device_status(), "weights_generation_s": round(gen_s, 1),
    }


VOCAB = 202048
LMHEAD_W = VOCAB * (H // 256) * 210  # Q6_K
# The model's logit scale and soft cap as the book prints them (Ch 10 Figure
# 10.1 box 15): logits = cap * tanh(l * scale / cap).
LOGIT_SCALE, SOFTCAP = 0.196116, 20.0


def run_lmhead(args, rank, world):
    """The LM head of one decode token (Ch 10 Figure 10.1 boxes 14-15): the
    202,048 x 6,656 Q6_K matvec of the final normed row with the logit scale
    and soft cap as its epilogue (muser_lm_head), 1.09 GB per step."""
    import torch
    import quantized_weight_streaming_q4_gb300 as mu
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
        dist.init_process_group("nccl")
    mu.build()
    L = mu.lib()
    VOCAB = args.vocab                      # the model's 202,048 unless a smaller case is asked for
    LMHEAD_W = VOCAB * (H // 256) * 210     # Q6_K
    t0 = time.time()
    W = torch.from_numpy(synth.q6k_matrix(VOCAB, H, seed=0, workload=7)).cuda()
    gen_s = time.time() - t0
    x = torch.from_numpy(synth.normal((1, H), seed=0, workload=7) * np.float32(0.02)).cuda()
    logits = torch.empty(VOCAB, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    scale, cap = LOGIT_SCALE, SOFTCAP

    def step():
        r = L.muser_lm_head(14, W.data_ptr(), VOCAB, H, x.data_ptr(), 1, logits.data_ptr(), scale, cap, sh)
        if r != 0:
            raise RuntimeError(f"lm_head: {mu.muser_last_error()}")

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    barrier()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    for a, b in evs:
        a.record(stream)
        step()
        b.record(stream)
    barrier()
    clock = clocks.stop()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    ms = max_over_ranks(ms, dist)
    h_in = torch.from_numpy(x.cpu().numpy()).pin_memory()
    h_out = torch.empty(VOCAB, dtype=torch.float32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        x.copy_(h_in, non_blocking=True)
        step()
        h_out.copy_(logits, non_blocking=True)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    assert np.isfinite(h_out.numpy()).all()
    peak, peak_kind = read_peaks()
    nbytes = LMHEAD_W + 4 * H + 4 * VOCAB
    gbs = whole_job_gbs(world, LMHEAD_W, ms)
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded Q6_K fields per the workload recipe)",
        "config": {"workload": f"LM head: Q6_K {VOCAB}x{H} matvec with the logit scale and soft cap, M=1",
                   "vocab": VOCAB, "hidden": H, "M": 1, "weight_bytes_per_step": LMHEAD_W,
                   "l2": f"inputs larger than L2: {LMHEAD_W / 1e9:.2f} GB of weights per step vs 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tokens_per_s": round(world / (ms * 1e-3), 3),
        "hbm_frac_of_" + peak_kind: round(gbs / world / peak, 4),
        "roofline": {"bound": "hbm", "kernel": "muser_lm_head (mv1 Q6_K, soft-cap epilogue)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None, "algorithmic_bytes_per_launch": nbytes, "mean_launch_us": round(ms * 1e3, 2)},
        "e2e": {"value": round(whole_job_gbs(world, LMHEAD_W, e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": 4 * H, "d2h_bytes_per_step": 4 * VOCAB,
                "api": "muser_lm_head with the hidden row in from pinned host memory and the logits out"},
        "gpu_launches": args.steps, "clocks": clock, "device_status": mu.muser_device_status(),
        "weights_generation_s": round(gen_s, 1),
    }


def run_down_tail(args, rank, world):
    """The stand-alone down projection with the fused dual-eps tail at M = 1
    (muser_qmatvec_residual_dual_rmsnorm; Ch 19 §19.4, §19.6), Q4_K or Q6_K
    W_down 6656 x 19968: a chain of `--layers` calls on distinct seeded
    weights, each one updating the residual in place, so a step streams more
    than L2 holds.  `matvec_q5k`: the same chain of plain Q5_K matvecs
    (muser_qmatvec), the k-quant the book's registry names beside Q4_K and
    Q6_K (Ch 4 §4.4)."""
    import torch
    import quantized_weight_streaming_q4_gb300 as mu
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
        dist.init_process_group("nccl")
    mu.build()
    L = mu.lib()
    q5 = args.workload == "matvec_q5k"
    q4 = args.workload == "down_tail_q4k"
    qname = "Q5_K" if q5 else ("Q4_K" if q4 else "Q6_K")
    qt = {"Q4_K": 12, "Q5_K": 13, "Q6_K": 14}[qname]
    wbytes = H * (F // 256) * {"Q4_K": 144, "Q5_K": 176, "Q6_K": 210}[qname]
    nl = args.layers
    t0 = time.time()
    layers = []
    for l in range(nl):
        c = synth.down_tail_case(qname.lower(), H, F, 1, seed=0, workload=1 if q4 else 2, layer=l)
        a, b = c["a"].astype(np.float32), c["b"].astype(np.float32)
        mid = (a / (np.float32(1) + np.exp(-a)) * b).astype(np.float32)   # the FFN intermediate input
        layers.append({k: torch.from_numpy(np.ascontiguousarray(v)).cuda()
                       for k, v in (("W", c["W"]), ("mid", mid), ("w1", c["w1"]), ("w2", c["w2"]))})
        if l == 0:
            r0 = c["resid"].astype(np.float32)
    gen_s = time.time() - t0
    resid = torch.from_numpy(r0.copy()).cuda()
    out = torch.empty(H, dtype=torch.float32, device="cuda")
    proj = torch.empty(H, dtype=torch.float32, device="cuda")
    nscr = mu.muser_scratch_bytes(H, 1)
    scratch = torch.zeros(nscr // 4 + 64, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def call(d):
        if q5:
            return L.muser_qmatvec(qt, d["W"].data_ptr(), H, F, d["mid"].data_ptr(), 1, out.data_ptr(), sh)
        return L.muser_qmatvec_residual_dual_rmsnorm(
            qt, d["W"].data_ptr(), H, F, d["mid"].data_ptr(), 1, proj.data_ptr(), resid.data_ptr(),
            out.data_ptr(), d["w1"].data_ptr(), d["w2"].data_ptr(), 1e-8, 1e-5, scratch.data_ptr(), nscr, sh)

    def step():
        for d in layers:
            r = call(d)
            if r != 0:
                raise RuntimeError(f"{args.workload}: {mu.muser_last_error()}")

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        resid.copy_(torch.from_numpy(r0))
        step()
    barrier()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    clock = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, dist)
    assert torch.isfinite(out).all() and torch.isfinite(resid).all()
    # end to end: the residual row in from pinned host memory, the normed row out, every call
    h_in = torch.from_numpy(r0.copy()).pin_memory()
    h_x = [d["mid"].cpu().pin_memory() for d in layers] if q5 else None
    h_out = torch.empty(H, dtype=torch.float32).pin_memory()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        for li, d in enumerate(layers):
            if q5:
                d["mid"].copy_(h_x[li], non_blocking=True)
            else:
                resid.copy_(h_in, non_blocking=True)
            r = call(d)
            if r != 0:
                raise RuntimeError(f"{args.workload}: {mu.muser_last_error()}")
            h_out.copy_(out, non_blocking=True)
    f1.record(stream)
    barrier()
    e2e_ms = f0.elapsed_time(f1) / args.steps
    peak, peak_kind = read_peaks()
    # W, mid; p, r in/out, out; w1, w2 (a plain matvec: W, x, y)
    per_launch = wbytes + 4 * F + (4 * H if q5 else 5 * 4 * H + 2 * 4 * H)
    launch_ms = ms / nl
    gbs = world * nl * wbytes / (ms * 1e-3) / 1e9
    achieved = per_launch / (launch_ms * 1e-3) / 1e9
    return {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; fields drawn per the workload recipe)",
        "config": {"workload": (f"{nl} x [{qname} {H}x{F} matvec], M=1, distinct weights per call" if q5 else
                                f"{nl} x [{qname} W_down {H}x{F} matvec + dual-eps fused tail], M=1, "
                                "distinct weights per call"),
                   "hidden": H, "ffn": F, "M": 1, "calls_per_step": nl, "weight_bytes_per_step": nl * wbytes,
                   "l2": f"inputs larger than L2: {nl * wbytes / 1e9:.2f} GB of distinct weights per step "
                         "vs 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        ("matvecs_per_s" if q5 else "matvec_tail_per_s"): round(world * nl / (ms * 1e-3), 1),
        "hbm_frac_of_" + peak_kind: round(gbs / world / peak, 4),
        "roofline": {"bound": "hbm", "kernel": (f"muser_qmatvec (mv1 {qname}, store)" if q5 else
                                                f"muser_qmatvec_residual_dual_rmsnorm (mv1 {qname}, one-pass "
                                                "last-CTA tail)"),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None, "algorithmic_bytes_per_launch": per_launch,
                     "mean_launch_us": round(launch_ms * 1e3, 2),
                     "timing": "step time / calls per step (back-to-back launches)"},
        "e2e": {"value": round(world * nl * wbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": 4 * (F if q5 else H) * nl,
                "d2h_bytes_per_step": 4 * H * nl,
                "api": ("muser_qmatvec, the input row in and the output row out per call" if q5 else
                        "muser_qmatvec_residual_dual_rmsnorm, residual in and normed row out per call")},
        "gpu_launches": args.steps * nl, "clocks": clock, "device_status": mu.muser_device_status(),
        "weights_generation_s": round(gen_s, 1),
    }


# One session slot's K/V planes (Ch 15 §15.7): 13 NoPE layers with head-major
# planes of max_context rows, 39 sliding layers with 2,048-row token-major rings;
# kv_dim 256 halves (2 KV heads x 128), K and V.
KV_TOKENS = 130815          # the deep handoff's context depth (Ch 15 §15.7)
KV_MAX_CONTEXT = 131072
KV_SWA_CAP = 2048
KV_DIM, KV_HEAD_DIM = 256, 128
KV_NOPE, KV_SWA = 13, 39


def run_kv_restore(args, rank, world):
    """Rotation-preserving restore of one session slot (Ch 15 §15.6): every
    layer's detached logical rows installed into its plane pair, the sliding
    rings at rotation origin % 2,048.  The value counts the bytes each restore
    reads and writes, 2 x 1.82 GB per step, against the measured copy
    bandwidth (also read + write bytes)."""
    import torch
    import quantized_weight_streaming_q4_gb300 as mu
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
        dist.init_process_group("nccl")
    mu.build()
    L = mu.lib()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234 + rank)
    swa_len = min(KV_TOKENS, KV_SWA_CAP)
    swa_origin = KV_TOKENS - swa_len
    layers = []  # (plane, k_rows, v_rows, origin, len)
    for layer in range(KV_NOPE + KV_SWA):
        nope = layer < KV_NOPE
        cap, n, origin = (KV_MAX_CONTEXT, KV_TOKENS, 0) if nope else (KV_SWA_CAP, swa_len, swa_origin)
        key = torch.zeros(cap * KV_DIM, dtype=torch.int16, device="cuda")
        val = torch.zeros_like(key)
        kr = torch.randint(-32768, 32767, (n * KV_DIM,), dtype=torch.int16, device="cuda", generator=gen)
        vr = torch.randint(-32768, 32767, (n * KV_DIM,), dtype=torch.int16, device="cuda", generator=gen)
        plane = mu.KvPlane(key.data_ptr(), val.data_ptr(), cap, 0, 0, 0, KV_DIM, KV_HEAD_DIM,
                           1 if nope else 0, 0)
        layers.append((plane, key, val, kr, vr, origin, n, nope))
    row_bytes = sum(2 * 2 * n * KV_DIM for (_, _, _, _, _, _, n, _) in layers)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def restore(rows=None):
        for i, (plane, _, _, kr, vr, origin, n, _) in enumerate(layers):
            k_ptr, v_ptr = (kr.data_ptr(), vr.data_ptr()) if rows is None else rows[i]
            r = L.muser_kv_restore(ctypes.byref(plane), k_ptr, v_ptr, origin, n, sh)
            if r != 0:
                raise RuntimeError(f"kv_restore: {mu.muser_last_error()}")

    def snapshot():
        for plane, _, _, kr, vr, origin, n, _ in layers:
            r = L.muser_kv_snapshot(ctypes.byref(plane), origin, n, kr.data_ptr(), vr.data_ptr(), sh)
            if r != 0:
                raise RuntimeError(f"kv_snapshot: {mu.muser_last_error()}")

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        restore()
        snapshot()
    barrier()
    # the restored planes hold the rows at their rotation (a sampled check; the
    # bit-exact comparison against the oracle is in the GPU tests)
    plane, key, _, kr, _, origin, n, _ = layers[-1]
    rot = origin % plane.capacity
    assert (plane.len, plane.origin_logical, plane.origin_physical) == (n, origin, rot)
    assert torch.equal(key.view(-1, KV_DIM)[rot], kr.view(-1, KV_DIM)[0])
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    for a, b in evs:
        a.record(stream)
        restore()
        b.record(stream)
    barrier()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in sev:
        a.record(stream)
        snapshot()
        b.record(stream)
    barrier()
    clock = clocks.stop()
    snap_ms = statistics.mean(a.elapsed_time(b) for a, b in sev)
    # one NoPE plane restore alone: the dominant launch
    one = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    plane0, _, _, kr0, vr0, _, n0, _ = layers[0]
    for a, b in one:
        a.record(stream)
        L.muser_kv_restore(ctypes.byref(plane0), kr0.data_ptr(), vr0.data_ptr(), 0, n0, sh)
        b.record(stream)
    barrier()
    one_ms = statistics.mean(a.elapsed_time(b) for a, b in one)
    ms = max_over_ranks(ms, dist)
    # end to end: the detached rows arrive in pinned host memory (as from the wire)
    host_rows = [(torch.empty(n * KV_DIM, dtype=torch.int16).pin_memory(),
                  torch.empty(n * KV_DIM, dtype=torch.int16).pin_memory())
                 for (_, _, _, _, _, _, n, _) in layers]
    for (hk, hv), (_, _, _, kr, vr, _, _, _) in zip(host_rows, layers):
        hk.copy_(kr)
        hv.copy_(vr)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        for (hk, hv), (_, _, _, kr, vr, _, _, _) in zip(host_rows, layers):
            kr.copy_(hk, non_blocking=True)
            vr.copy_(hv, non_blocking=True)
        restore()
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    peak, peak_kind = read_peaks()
    moved = 2 * row_bytes
    gbs = whole_job_gbs(world, moved, ms)
    one_bytes = 2 * 2 * 2 * n0 * KV_DIM
    achieved = one_bytes / (one_ms * 1e-3) / 1e9
    return {
        "metric": "K/V bytes moved GB/s (read + write, % of GB300 HBM copy peak), 1 GPU", "value": round(gbs, 2),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16",
        "data": "synthetic (seeded random binary16 bit patterns)",
        "config": {"workload": f"K/V restore of one session at {KV_TOKENS} tokens: {KV_NOPE} head-major NoPE planes "
                               f"({KV_MAX_CONTEXT} rows) and {KV_SWA} token-major SWA rings ({KV_SWA_CAP} rows, "
                               f"origin {swa_origin}, rotation {swa_origin % KV_SWA_CAP})",
                   "kv_dim": KV_DIM, "head_dim": KV_HEAD_DIM, "row_bytes_per_step": row_bytes,
                   "l2": f"inputs larger than L2: {row_bytes / 1e9:.2f} GB of rows per step vs 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hbm_frac_of_" + peak_kind: round(gbs / world / peak, 4),
        "snapshot": {"ms_per_step": round(snap_ms, 4), "value": round(moved / (snap_ms * 1e-3) / 1e9, 2),
                     "unit": "GB/s", "api": "muser_kv_snapshot of every layer's live window"},
        "roofline": {"bound": "hbm", "kernel": "kv_window_kernel<8, restore> (one NoPE plane pair, 268 MB moved)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None, "algorithmic_bytes_per_launch": one_bytes,
                     "mean_launch_us": round(one_ms * 1e3, 2)},
        "e2e": {"value": round(whole_job_gbs(world, moved, e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": row_bytes, "d2h_bytes_per_step": 0,
                "api": "muser_kv_restore with the detached rows in from pinned host memory"},
        "gpu_launches": args.steps * len(layers), "clocks": clock, "device_status": mu.muser_device_status(),
    }


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    smp = _oracle_layer_sample(args.ref_frac)
    for _ in range(args.warmup):
        _oracle_step(oracle, smp)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += _oracle_step(oracle, smp)
    dt = time.perf_counter() - t0
    gbs = nbytes / dt / 1e9
    M = 16 if args.workload == "stack52_m16" else 1
    sample = (f"each step: the fp64 oracle over one layer's path (input rms_norm, the first {args.ref_frac:.3f} "
              f"of the gate/up rows + SiLU and of the down rows, the dual-eps tail), "
              f"{nbytes / args.steps / 1e6:.1f} MB of weights, M=1")
    return {
        "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": f"decode-FFN stack: {args.layers} layers, M={M} (bounded row sample per step)",
                   "layers": args.layers, "hidden": H, "ffn": F, "M": M},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "kind": "oracle",
                         "cores": oracle.num_threads(), "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=["stack52_m1", "stack52_m16", "attn52_m1", "attn52_m16", "lmhead_m1",
                                           "kv_restore", "down_tail_q4k", "down_tail_q6k", "matvec_q5k"],
                    default="stack52_m1")
    ap.add_argument("--layers", type=int, default=NL)
    ap.add_argument("--vocab", type=int, default=VOCAB,
                    help="lmhead_m1: output rows (the model's 202,048; smaller for profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-frac", type=float, default=0.0625)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="skip the M = 16 sub-result of the default workload")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world = _env_int("RANK", 0), _env_int("WORLD_SIZE", 1)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    elif args.workload.startswith("attn"):
        res = run_attn(args, rank, world)
    elif args.workload == "lmhead_m1":
        res = run_lmhead(args, rank, world)
    elif args.workload == "kv_restore":
        res = run_kv_restore(args, rank, world)
    elif args.workload.startswith("down_tail") or args.workload == "matvec_q5k":
        res = run_down_tail(args, rank, world)
    else:
        res = run_native(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
