#!/usr/bin/env python
"""Benchmark of the group-limited MoE block (Beam shapes) on B300.

One step = one forward of the whole block (router, dispatch, gather, gate/up
GEMM + SwiGLU, down GEMM, combine) over one batch of synthetic tokens, with
every input already resident in HBM.  The headline workload is the decode
layer (T=64, H=5120, I=2560, 256 BF16 experts); the prefill layer (T=8192),
the NVFP4-expert layer (T=4096) and the skewed-routing layer (T=32768, Zipf
router bias) are measured the same way and reported under "prefill", "nvfp4"
and "skew", each with its rooflines, per-stage times and a bounded oracle
sample with the workload's near-tie count.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the block does not shard); the barrier and the max-over-ranks time are the
only collectives.  ``--impl reference`` times the CPU oracle (the plain FP64
definition) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "MoE-layer tokens/s (T=64 decode, T=8192 prefill); % HBM / tensor-core roofline"
STAGES = ("route", "dispatch", "gather", "gate_up", "down", "combine")


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML while running."""

    REASONS = {
        "gpu_idle": 0x1, "applications_clocks_setting": 0x2, "sw_power_cap": 0x4, "hw_slowdown": 0x8,
        "sync_boost": 0x10, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
        "hw_power_brake_slowdown": 0x80, "display_clock_setting": 0x100,
    }

    def __init__(self, index: int, period_s: float = 0.01):
        self.period = period_s
        self.samples = []
        self.max_mhz = None
        self.index = index
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._nvml = None
        try:
            import pynvml

            pynvml.nvmlInit()
            self._h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self._nvml = pynvml
            self.source = "nvml"
        except Exception as exc:  # fall back to nvidia-smi's sampling loop
            print(f"bench: NVML unavailable ({exc!r}); sampling clocks with nvidia-smi", file=sys.stderr)

    def _run(self):
        nv = self._nvml
        while not self._stop.is_set():
            try:
                mhz = nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM)
                reasons = nv.nvmlDeviceGetCurrentClocksEventReasons(self._h)
                self.samples.append((mhz, reasons))
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        else:
            import subprocess

            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index),
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                time.sleep(0.3)  # let the first sample land
            except Exception as exc:
                print(f"bench: no clock sampling ({exc!r})", file=sys.stderr)
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()
        if self._proc is not None:
            time.sleep(0.05)
            self._proc.terminate()
            out, _ = self._proc.communicate(timeout=10)
            for line in out.splitlines():
                parts = [q.strip() for q in line.split(",")]
                try:
                    mhz, mx, rs = float(parts[0]), float(parts[1]), int(parts[2], 16)
                except (ValueError, IndexError):
                    continue
                self.max_mhz = mx
                self.samples.append((mhz, rs))

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        mhz = [s[0] for s in self.samples]
        active = 0
        for _, r in self.samples:
            active |= int(r)
        names = [n for n, bit in self.REASONS.items() if active & bit and n != "gpu_idle"]
        return {"sm_mhz": float(statistics.median(mhz)), "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(mhz), "source": self.source}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
WEIGHTS_LAYOUT = "tiled"  # set from --weights-layout
RESIDUAL_STEP = 105  # step of the stream at the last sublayer of a 52-layer stack


def make_layer(wl, dev, layout=None):
    """Inputs and a reusable forward call.  With the tiled layout the expert
    weights are regrouped once here (a model-load step, outside any timing);
    ``d`` keeps the row-major arrays the oracle reads."""
    import group_limited_routing_03_b300 as moe
    from group_limited_routing_03_b300 import inputs

    d = inputs.generate(wl, dev)
    sh = moe.shape(wl.T, wl.H, wl.I)
    weights = d
    if (layout or WEIGHTS_LAYOUT) == "tiled":
        weights = moe.pack_weights(sh, d)
        torch.cuda.synchronize()
    if wl.acts == "nvfp4":  # W4A4: the GEMM inputs quantised to NVFP4 at run time
        weights = dict(weights, activations="nvfp4")
    ws = moe.alloc_workspace(sh, wl.w_dtype if wl.w_dtype in ("nvfp4", "fp8") else "bf16", dev)
    y = torch.empty((wl.T, wl.H), dtype=d["x"].dtype, device=dev)
    ids = torch.empty((wl.T, 8), dtype=torch.int32, device=dev)
    w = torch.empty((wl.T, 8), dtype=torch.float32, device=dev)
    call = moe.ForwardCall(sh, d["x"], d["router_w"], d.get("bias"), weights, y, ids, w, ws)
    return d, sh, ws, y, ids, w, call


def measure(wl, steps, warmup, dev, world, sampler_index, state=None, residual_step=None):
    """Device-timed steps through the per-stage C-ABI calls, events between
    the stages on the launching stream.  Returns a dict of timings.  With
    ``residual_step`` k the combine stage also applies the post-norm residual
    update at step k, in place on a seeded stream (no y written), reusing the
    layer of ``state``."""
    import group_limited_routing_03_b300 as moe
    from group_limited_routing_03_b300 import inputs

    if state is None:
        state = make_layer(wl, dev)
    d, sh, ws, y, ids, w, call = state
    if residual_step is not None:
        resid, g = inputs.residual_inputs(wl, dev)
        call = moe.ForwardCall(sh, d["x"], d["router_w"], d.get("bias"), call.weights, None, ids, w, ws,
                               residual=(resid, resid, g, inputs.RESIDUAL_EPS, residual_step))
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for i in range(len(STAGES)):
            call.stage(i)
    torch.cuda.synchronize()
    code, where = moe.beam_moe_read_device_status(ws)
    if code != 0:
        raise RuntimeError(f"device status {code} at {where} during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(sampler_index) as clk:
        for k in range(steps):
            ev = evs[k]
            ev[0].record(stream)
            for i in range(len(STAGES)):
                call.stage(i)
                ev[i + 1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    total_ms = evs[0][0].elapsed_time(evs[-1][-1])
    stage_ms = [statistics.fmean(ev[i].elapsed_time(ev[i + 1]) for ev in evs) for i in range(len(STAGES))]
    code, where = moe.beam_moe_read_device_status(ws)
    if code != 0:
        raise RuntimeError(f"device status {code} at {where} in the timed region")
    ids_h = ids.cpu()
    touched = int(torch.unique(ids_h).numel())
    xdt = moe.BEAM_BF16 if d["x"].dtype == torch.bfloat16 else moe.BEAM_F32
    launches = sum(moe.beam_moe_stage_kernel_count(sh, i, xdt, call.weights) for i in range(len(STAGES)))
    out = dict(total_ms=total_ms, stage_ms=stage_ms, touched=touched, launches_per_step=launches,
               clocks=clk.summary(), counts=torch.bincount(ids_h.reshape(-1).long(), minlength=256))
    return out, state


def measure_graph(wl, state, steps, warmup):
    """The same step recorded once in a CUDA graph (GraphedForward) and
    replayed: x copied into the graph's input, then one graph launch."""
    import group_limited_routing_03_b300 as moe

    d, sh, ws, y, ids, w, call = state
    layer = moe.BeamMoE(d["router_w"], d.get("bias"), call.weights, max_tokens=wl.T)
    graphed = moe.GraphedForward(layer, wl.T, dtype=d["x"].dtype)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        graphed(d["x"])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        graphed(d["x"])
    e1.record(stream)
    torch.cuda.synchronize()
    code, where = moe.beam_moe_read_device_status(layer.workspace)
    if code != 0:
        raise RuntimeError(f"device status {code} at {where} in the graph replays")
    ms = e0.elapsed_time(e1) / steps
    out = dict(value=wl.T / (ms * 1e-3), unit="tokens/s", ms_per_step=round(ms, 4), steps=steps,
               note="one CUDA-graph replay per step (the library's launches recorded once), x copied in first")
    del graphed, layer
    return out


def measure_dense(wl, steps, warmup, dev, pk):
    """The dense SwiGLU MLP (one expert taking every row) through
    beam_dense_mlp_forward, device-timed per call; weights in the tiled layout."""
    import group_limited_routing_03_b300 as moe
    from group_limited_routing_03_b300 import inputs

    d = inputs.generate(wl, dev)
    w = {k: d[k] for k in ("gate", "up", "down")}
    mlp = moe.DenseMLP(w, max_tokens=wl.T, pack=True)
    x = d["x"]
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        mlp(x, y)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0.record(stream)
        for _ in range(steps):
            mlp(x, y)
        e1.record(stream)
        torch.cuda.synchronize()
    code, where = moe.beam_moe_read_device_status(mlp.workspace)
    if code != 0:
        raise RuntimeError(f"device status {code} at {where} in the dense MLP")
    ms = e0.elapsed_time(e1) / steps
    wbytes = 3 * wl.H * wl.I * 2
    flops = 2.0 * wl.T * 3 * wl.H * wl.I
    gbs = (wbytes + 2 * wl.T * wl.H * 2 + 2 * wl.T * wl.I * 2) / (ms * 1e-3) / 1e9
    tfs = flops / (ms * 1e-3) / 1e12
    out = dict(value=wl.T / (ms * 1e-3), unit="tokens/s", ms_per_call=round(ms, 4), steps=steps,
               config={"workload": f"{wl.name} T={wl.T} H={wl.H} I={wl.I} dense SwiGLU MLP, BF16", "T": wl.T},
               gpu_launches=steps * moe.dense_kernel_count(moe.dense_shape(wl.T, wl.H, wl.I), "bf16"),
               clocks=clk.summary())
    if wl.T <= 256:
        out["roofline"] = dict(bound="hbm", achieved=round(gbs, 1), peak=pk["hbm"], unit="GB/s",
                               frac=round(gbs / pk["hbm"], 4), peak_source=pk["source"])
    else:
        out["roofline"] = dict(bound="tensor", achieved=round(tfs, 1), peak=pk["bf16"], unit="TFLOP/s",
                               frac=round(tfs / pk["bf16"], 4), peak_sustained=pk["bf16_sustained"],
                               frac_sustained=round(tfs / pk["bf16_sustained"], 4), peak_source=pk["source"])
    del d, mlp
    return out


def workload_record(name, steps, warmup, dev, world, pk, small, cpu_budget_s=None, note="", residual=False):
    """One more workload measured like the headline: device-timed steps
    through the per-stage calls, the gate/up kernel's HBM and tensor
    rooflines, the whole step's numbers, optionally the same steps with the
    residual update fused into the combine, and, on rank 0 of a 1-GPU run, a
    bounded sample of the oracle (with the workload's near-tie count)."""
    from group_limited_routing_03_b300 import inputs

    wl = inputs.workload(name, **small)
    m, state = measure(wl, steps, warmup, dev, world, torch.cuda.current_device())
    t_ms = max_over_ranks(m["total_ms"], world)
    hbm, tc = roofline(wl, m, pk)
    desc = {"bf16": "bf16 experts", "nvfp4": "nvfp4 experts (W4A16)",
            "fp8": "fp8 experts (E4M3 + row scales), E4M3 activations per row"}[wl.w_dtype]
    if wl.acts == "nvfp4":
        desc = "nvfp4 experts, NVFP4 activations per row (W4A4; FP16 tensor cores)"
    rec = dict(value=wl.T * steps * world / (t_ms * 1e-3), unit="tokens/s",
               config={"workload": f"{name} T={wl.T} H={wl.H} I={wl.I} E=256 {desc}" + (f", {note}" if note else ""),
                       "T": wl.T},
               roofline=tc, roofline_hbm=hbm, clocks=m["clocks"], gpu_launches=m["launches_per_step"] * steps,
               **step_numbers(wl, m, steps, pk))
    if residual:
        rm, _ = measure(wl, steps, warmup, dev, world, torch.cuda.current_device(), state=state,
                        residual_step=RESIDUAL_STEP)
        rec["residual_epilogue"] = residual_numbers(wl, m, rm, steps, pk, RESIDUAL_STEP)
    if cpu_budget_s is not None and world == 1 and int(os.environ.get("RANK", "0")) == 0:
        rec["cpu_baseline"] = oracle_sample(wl, state[0], budget_s=cpu_budget_s)
    del state
    torch.cuda.empty_cache()
    return rec


def measure_route_noalloc(dev, steps=50):
    """beam_moe_route (workspace) against beam_moe_route_noalloc (static
    scratch, hidden dimension split across at most 4096 / T CTAs per tile):
    device time per call at H=5120, BF16 x, FP32 router."""
    import group_limited_routing_03_b300 as moe
    from group_limited_routing_03_b300 import inputs

    out = {}
    stream = torch.cuda.current_stream()
    for T in (64, 2048, 4096):
        wl = inputs.workload("prefill", T=T)
        d = inputs.generate(wl, dev, experts=False)
        sh = moe.shape(T, wl.H, wl.I)
        ws = moe.alloc_workspace(sh, "bf16", dev)
        ids = torch.empty((T, 8), dtype=torch.int32, device=dev)
        w = torch.empty((T, 8), dtype=torch.float32, device=dev)
        res = {}
        for label, fn in (("route_ms", lambda: moe.beam_moe_route(sh, d["x"], d["router_w"], None, ids, w, ws)),
                          ("noalloc_ms", lambda: moe.beam_moe_route_noalloc(sh, d["x"], d["router_w"], None, ids, w))):
            for _ in range(5):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            res[label] = round(e0.elapsed_time(e1) / steps, 4)
        out[f"T={T}"] = res
        del d, ws
    torch.cuda.empty_cache()
    return out


def residual_numbers(wl, m_plain, m_res, steps, pk, k):
    """The post-norm residual update fused into the combine: its stage time
    against the plain combine's in the same step, and its own HBM roofline.
    Algorithmic bytes per launch: the 8 expert-output rows of every token
    (BF16), the stream read and written (x's dtype), the norm scale, and the
    routing weights and positions."""
    c = STAGES.index("combine")
    ms = m_res["stage_ms"][c]
    xb = 2 if wl.x_dtype == "bf16" else 4
    alg = wl.T * 8 * wl.H * 2 + 2 * wl.T * wl.H * xb + wl.H * 4 + wl.T * 8 * 8
    gbs = alg / (ms * 1e-3) / 1e9
    return dict(step_k=k, in_place=True, combine_ms=round(m_plain["stage_ms"][c], 4), combine_residual_ms=round(ms, 4),
                ms_per_step=round(m_res["total_ms"] / steps, 4),
                roofline=dict(bound="hbm", achieved=round(gbs, 1), peak=pk["hbm"], unit="GB/s",
                              frac=round(gbs / pk["hbm"], 4), algorithmic_bytes=alg, launch_ms=round(ms, 4),
                              kernel="combine_residual_kernel", peak_source=pk["source"]),
                clocks=m_res["clocks"])


def measure_e2e(wl, state, steps, warmup, dev):
    """Same step through the public call with host buffers: every step copies
    its x in from pinned host memory and its y / ids / weights out, inside the
    timed region.  As a serving loop would, the copies run on two copy streams
    with double-buffered device and host buffers, so step i+1's input copy and
    step i-1's output copy overlap step i's compute."""
    import group_limited_routing_03_b300 as moe

    d, sh, ws, y, ids, w, call = state
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    x_host = [d["x"].cpu().pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(d["x"]) for _ in range(2)]
    outs = [(torch.empty_like(y), torch.empty_like(ids), torch.empty_like(w)) for _ in range(2)]
    outs_host = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in o) for o in outs]
    calls = [moe.ForwardCall(sh, x_dev[b], d["router_w"], d.get("bias"), call.weights, *outs[b], ws) for b in range(2)]
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("h2d", "comp", "d2h")}

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev["comp"][b])  # the slot's previous step no longer reads x
            x_dev[b].copy_(x_host[b], non_blocking=True)
            ev["h2d"][b].record(s_in)
        comp.wait_event(ev["h2d"][b])
        if i >= 2:
            comp.wait_event(ev["d2h"][b])  # the slot's previous outputs have been read out
        calls[b].run()
        ev["comp"][b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][b])
            for dst, src in zip(outs_host[b], outs[b]):
                dst.copy_(src, non_blocking=True)
            ev["d2h"][b].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    for i in range(steps):
        step(i)
    comp.wait_event(ev["d2h"][(steps - 1) % 2])  # the last step's results are on the host
    e1.record(comp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    h2d = x_host[0].numel() * x_host[0].element_size()
    d2h = sum(t.numel() * t.element_size() for t in outs_host[0])
    return ms, h2d, d2h


def weight_bytes_per_expert(wl):
    if wl.w_dtype == "nvfp4":
        return 3 * wl.H * wl.I // 2 + 3 * wl.H * wl.I // 16 + 12
    if wl.w_dtype == "fp8":  # E4M3 codes + FP32 row scales
        return 3 * wl.H * wl.I + 4 * (2 * wl.I + wl.H)
    return 3 * wl.H * wl.I * 2


def code_hash(texts) -> str:
    """sha256 of C/CUDA sources with comments removed and white space
    collapsed: it changes with the code the compiler sees, not with its
    comments.  String and character literals are kept as they are."""
    out = []
    for text in texts:
        i, n = 0, len(text)
        while i < n:
            c = text[i]
            if text.startswith("//", i):
                j = text.find("\n", i)
                i = n if j < 0 else j
            elif text.startswith("/*", i):
                j = text.find("*/", i + 2)
                i = n if j < 0 else j + 2
                out.append(" ")
            elif c in "\"'":
                j = i + 1
                while j < n and text[j] != c:
                    j += 2 if text[j] == "\\" else 1
                out.append(text[i:j + 1])
                i = j + 1
            else:
                out.append(c)
                i += 1
        out.append("\n")
    return hashlib.sha256(" ".join("".join(out).split()).encode()).hexdigest()


def traffic_record(kernel: str, workload: str, algorithmic_bytes: float):
    """Per-launch DRAM bytes of `kernel`: the ratio of DRAM to algorithmic
    bytes ncu measured on a small case of the workload (committed summary),
    times this launch's algorithmic bytes; None when there is no record or
    the kernel's code (its sources, comments aside) changed since the
    capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload, {}).get(kernel)
    if not ent:
        return None
    csrc = os.path.join(ROOT, "group_limited_routing_03_b300", "csrc")
    srcs = [os.path.join(csrc, name) for name in ent["sources"]]
    if not all(os.path.exists(f) for f in srcs):
        return None
    if code_hash(open(f).read() for f in srcs) != ent["code_sha256"]:
        return None
    return round(float(ent["dram_ratio"]) * algorithmic_bytes, 1)


def roofline(wl, m, pk):
    """Dominant kernel: the gate/up GEMM (2/3 of the weight bytes and FLOPs)."""
    R = wl.T * 8
    ms = m["stage_ms"][STAGES.index("gate_up")]
    # gate + up weights of the touched experts: BF16 2 bytes per element,
    # NVFP4 half a byte plus one E4M3 scale per 16 elements, FP8 one byte
    # (+ an FP32 scale per row); activations: the route rows in (BF16, or
    # E4M3 codes for FP8) and h out (BF16)
    per_elem = {"nvfp4": 0.5 + 1.0 / 16, "fp8": 1.0}.get(wl.w_dtype, 2.0)
    wbytes = int(m["touched"] * 2 * wl.I * wl.H * per_elem) + (m["touched"] * 2 * wl.I * 4 if wl.w_dtype == "fp8" else 0)
    act_bytes = R * wl.H * (1 if wl.w_dtype == "fp8" else 2) + R * wl.I * 2
    flops = 2.0 * R * 2 * wl.I * wl.H
    gbs = (wbytes + act_bytes) / (ms * 1e-3) / 1e9
    tfs = flops / (ms * 1e-3) / 1e12
    hbm = dict(bound="hbm", achieved=round(gbs, 1), peak=pk["hbm"], unit="GB/s", frac=round(gbs / pk["hbm"], 4),
               traffic=traffic_record("moe_gemm_gate_up", wl.name, wbytes + act_bytes),
               kernel="moe_gemm_kernel<0> (gate/up + SwiGLU)",
               algorithmic_bytes=wbytes + act_bytes, launch_ms=round(ms, 4), peak_source=pk["source"])
    # FP8 MMAs: the measured BF16 peak times the nominal FP8 / BF16 ratio (2).
    # peak: the burst GEMM figure (the headline fraction); peak_sustained: the
    # same GEMM run for seconds under the power cap, for steps whose clock
    # record shows sw_power_cap
    ratio = 2.0 if wl.w_dtype == "fp8" else 1.0
    tpk, tpk_s = pk["bf16"] * ratio, pk["bf16_sustained"] * ratio
    tc = dict(bound="tensor", achieved=round(tfs, 1), peak=round(tpk, 1), unit="TFLOP/s", frac=round(tfs / tpk, 4),
              peak_sustained=round(tpk_s, 1), frac_sustained=round(tfs / tpk_s, 4),
              traffic=hbm["traffic"], kernel=hbm["kernel"], algorithmic_flops=flops, launch_ms=round(ms, 4),
              peak_source=pk["source"] + (" bf16 x 2 (nominal fp8 / bf16 ratio)" if wl.w_dtype == "fp8" else ""))
    return hbm, tc


def step_numbers(wl, m, steps, pk=None):
    """Whole-step numbers: algorithmic bytes (touched experts' weights, x in,
    y out, router weight) and FLOPs (three expert GEMMs per route, the router
    GEMV per token) over the device time of one step, and, with the peaks,
    their fractions of the HBM and tensor peaks."""
    R = wl.T * 8
    ms = m["total_ms"] / steps
    wbytes = m["touched"] * weight_bytes_per_expert(wl)
    xb = 2 if wl.x_dtype == "bf16" else 4
    bytes_alg = wbytes + wl.T * wl.H * xb * 2 + wl.E * wl.H * 4
    flops = 2.0 * R * 3 * wl.I * wl.H + 2.0 * wl.T * wl.E * wl.H
    gbs = bytes_alg / (ms * 1e-3) / 1e9
    tfs = flops / (ms * 1e-3) / 1e12
    out = dict(ms_per_step=round(ms, 4), tokens_per_s=wl.T / (ms * 1e-3),
               step_gbs=round(gbs, 1), step_tflops=round(tfs, 1),
               touched_experts=m["touched"], stage_ms={s: round(v, 4) for s, v in zip(STAGES, m["stage_ms"])})
    if pk is not None:
        ratio = 2.0 if wl.w_dtype == "fp8" else 1.0
        out["step_frac_hbm"] = round(gbs / pk["hbm"], 4)
        out["step_frac_tensor"] = round(tfs / (pk["bf16"] * ratio), 4)
        out["step_frac_tensor_sustained"] = round(tfs / (pk["bf16_sustained"] * ratio), 4)
    return out


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(wl, d, budget_s=12.0, max_tokens=None):
    """Time the FP64 oracle on a bounded sample of the workload: routing of all
    T tokens, then whole tokens (8 experts + combine) one by one until the
    budget is spent.  Host copies of the inputs are made outside the timing.
    Also counts the workload's near-tie tokens (oracle margin <= 1e-5)."""
    import numpy as np

    import oracle
    from group_limited_routing_03_b300 import inputs  # noqa: F401

    def host(t):
        t = t.detach().cpu().contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    x = host(d["x"])
    wr = d["router_w"].cpu().numpy()
    b = None if d.get("bias") is None else d["bias"].cpu().numpy()
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    r = oracle.route(x, wr, b, threads=threads)
    t_route = time.perf_counter() - t0
    order = np.random.default_rng(wl.seed).permutation(wl.T)
    done, t_ffn = 0, 0.0
    for t in order[: (max_tokens or wl.T)]:
        mats = {}
        for e in r["ids"][t]:
            e = int(e)
            if wl.w_dtype == "nvfp4":
                mats[e] = ([d[n][e].cpu().numpy() for n in ("gate", "up", "down")],
                           dict(scales=[d[n + "_sf"][e].cpu().numpy() for n in ("gate", "up", "down")],
                                global_scales=[float(d[n + "_gs"][e]) for n in ("gate", "up", "down")]))
            else:
                mats[e] = ([host(d[n][e]) for n in ("gate", "up", "down")], {})
        t1 = time.perf_counter()
        ffn = oracle.expert_ffn_w4a4 if wl.acts == "nvfp4" else oracle.expert_ffn
        o = np.stack([ffn(x[t:t + 1], *mats[int(e)][0], threads=threads, **mats[int(e)][1])[0]
                      for e in r["ids"][t]])[None]
        oracle.combine(r["weights"][t:t + 1], o)
        t_ffn += time.perf_counter() - t1
        done += 1
        if t_ffn + t_route * done / wl.T >= budget_s:
            break
    sec = t_route * done / wl.T + t_ffn
    return dict(value=done / sec, unit="tokens/s", cores=threads, kind="oracle",
                sample=f"{wl.name}: routing of all {wl.T} tokens (time pro-rated to the sample), then "
                       f"{done} whole tokens (8 experts each, FP64) on {threads} threads; {sec:.2f} s of CPU time",
                near_ties=int((r["margin"] <= 1e-5).sum()), near_tie_tokens_of=wl.T)


def line_problems(line: dict, full: bool = True) -> list:
    """What the printed line lacks of the contract: the top-level keys and
    their types, the roofline object, and (``full``) the cpu_baseline and e2e
    objects.  Empty when the line is well formed."""
    out = []
    for k, t in (("metric", str), ("value", (int, float)), ("unit", str), ("n_gpus", int), ("steps", int),
                 ("warmup", int), ("ms_per_step", (int, float)), ("higher_is_better", bool), ("scaling", str),
                 ("dtype", str), ("data", str), ("config", dict), ("gpu_launches", int), ("clocks", dict)):
        if not isinstance(line.get(k), t):
            out.append(f"{k}: {type(line.get(k)).__name__}")
    if not isinstance(line.get("config", {}).get("workload"), str):
        out.append("config.workload missing")
    r = line.get("roofline")
    if not isinstance(r, dict) or not all(k in r for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")):
        out.append("roofline malformed")
    if full:
        c = line.get("cpu_baseline")
        if not isinstance(c, dict) or not all(k in c for k in ("value", "unit", "cores", "kind", "sample")):
            out.append(f"cpu_baseline malformed: {type(c).__name__}")
        e = line.get("e2e")
        if not isinstance(e, dict) or not all(k in e for k in ("value", "unit", "h2d_bytes_per_step",
                                                               "d2h_bytes_per_step")):
            out.append(f"e2e malformed: {type(e).__name__}")
    return out


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle on the host cores (rank 0 only)."""
    if rank != 0:
        return
    from group_limited_routing_03_b300 import inputs

    wl = inputs.workload(args.workload)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    d = inputs.generate(wl, dev)
    per_step = []
    for k in range(args.warmup + args.steps):
        res = oracle_sample(wl, d, budget_s=1e9, max_tokens=1)
        if k >= args.warmup:
            per_step.append(1.0 / res["value"])
    sec = sum(per_step)
    value = args.steps / sec
    cores = res["cores"]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wl.name} T={wl.T} H={wl.H} I={wl.I} E=256 {wl.w_dtype} experts",
                       "T": wl.T, "H": wl.H, "I": wl.I},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: routing of {wl.T} tokens pro-rated to one token plus one whole "
                                       f"token through its 8 experts and the combine, FP64"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v, world):
    """The slowest replica's time: the whole job finishes when it does."""
    if world == 1:
        return v
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_replica_step, steps, world, max_ms):
    """Whole-job tokens/s: every replica processes its own batch each step."""
    return tokens_per_replica_step * steps * world / (max_ms * 1e-3)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-more", action="store_true",
                    help="skip the NVFP4 layer (T=4096) and the skewed-routing layer (T=32768)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay of the headline step")
    ap.add_argument("--no-dense", action="store_true",
                    help="skip the dense SwiGLU MLP (decode T=64 and prefill T=8192, I=20480)")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the FP8-weight layers (decode T=64 and prefill T=8192) and the NVFP4 decode layer")
    ap.add_argument("--no-residual", action="store_true",
                    help="skip the extra steps with the post-norm residual update fused into the combine")
    ap.add_argument("--small", action="store_true",
                    help="profiling shape H=2048, I=1024 (3.2 GB of experts) instead of 5120/2560")
    ap.add_argument("--weights-layout", choices=("tiled", "rows"), default="tiled",
                    help="expert weights regrouped once into contiguous GEMM tiles (default), or row-major")
    args = ap.parse_args()
    global WEIGHTS_LAYOUT
    WEIGHTS_LAYOUT = args.weights_layout
    args.warmup = max(args.warmup, 3)

    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())

    from group_limited_routing_03_b300 import _build, inputs

    _build.build()
    pk = peaks()
    small = dict(H=2048, I=1024) if args.small else {}
    wl = inputs.workload(args.workload, **small)
    m, state = measure(wl, args.steps, args.warmup, dev, world, torch.cuda.current_device())
    total_ms = max_over_ranks(m["total_ms"], world)
    sn = step_numbers(wl, m, args.steps, pk)
    value = job_throughput(wl.T, args.steps, world, total_ms)
    hbm, tc = roofline(wl, m, pk)

    e2e = None
    if not args.no_e2e:
        e_ms, h2d, d2h = measure_e2e(wl, state, args.steps, args.warmup, dev)
        e_ms = max_over_ranks(e_ms, world)
        e2e = {"value": wl.T * args.steps * world / (e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(wl, state[0])
    graph = None
    try:
        if not args.no_graph:
            graph = measure_graph(wl, state, args.steps, args.warmup)
    except Exception as e:  # an auxiliary number: record why it is missing
        graph = {"unavailable": f"{type(e).__name__}: {e}"[:300]}
    residual = None
    if not args.no_residual:
        rm, _ = measure(wl, args.steps, args.warmup, dev, world, torch.cuda.current_device(), state=state,
                        residual_step=RESIDUAL_STEP)
        residual = residual_numbers(wl, m, rm, args.steps, pk, RESIDUAL_STEP)
    del state
    torch.cuda.empty_cache()

    prefill = None
    if not args.no_prefill:
        psteps = max(3, args.steps // 2)
        prefill = workload_record("prefill", psteps, args.warmup, dev, world, pk, small,
                                  cpu_budget_s=None if args.no_cpu_baseline else 3.0,
                                  residual=not args.no_residual)

    # the NVFP4 layer (T=4096) and the skewed-routing stress layer (T=32768)
    more = {}
    if not args.no_more:
        for name, steps, note in (("nvfp4", max(3, args.steps // 2), ""),
                                  ("skew", max(3, args.steps // 4), "Zipf(1.1) router bias in [0, 3]")):
            more[name] = workload_record(name, steps, args.warmup, dev, world, pk, small,
                                         cpu_budget_s=None if args.no_cpu_baseline else 3.0, note=note)

    fp8 = None
    if not args.no_fp8 and not args.small:
        fp8 = {}
        for name, steps in (("fp8_decode", args.steps), ("fp8", max(3, args.steps // 2)), ("nvfp4_dec", args.steps),
                            ("nvfp4_a4", max(3, args.steps // 2))):
            budget = None if args.no_cpu_baseline or name != "nvfp4_a4" else 3.0  # the W4A4 oracle timed as well
            fp8[name] = workload_record(name, steps, args.warmup, dev, world, pk, {}, cpu_budget_s=budget)

    route_noalloc = None
    if not args.small:
        route_noalloc = measure_route_noalloc(dev)

    dense = None
    if not args.no_dense and not args.small:
        dense = {name: measure_dense(inputs.workload(name), args.steps if name == "dense_dec" else max(3, args.steps // 2),
                                     args.warmup, dev, pk) for name in ("dense_dec", "dense")}
        torch.cuda.empty_cache()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{wl.name} T={wl.T} H={wl.H} I={wl.I} E=256 {wl.w_dtype} experts, FP32 router",
                   "T": wl.T, "H": wl.H, "I": wl.I, "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "weights_layout": WEIGHTS_LAYOUT,
                   "l2": "no flush: each step streams the touched experts' weights "
                         f"({m['touched']} x {weight_bytes_per_expert(wl) / 1e6:.1f} MB), far larger than L2"},
        "roofline": hbm, "roofline_tensor": tc, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": m["launches_per_step"] * args.steps, "clocks": m["clocks"],
        "step": sn, "graph": graph, "residual_epilogue": residual, "prefill": prefill,
        "nvfp4": more.get("nvfp4"), "skew": more.get("skew"), "weight_formats": fp8, "dense": dense,
        "route_noalloc": route_noalloc,
    }
    problems = line_problems(line, full=not (args.no_cpu_baseline or args.no_e2e))
    if problems:
        raise SystemExit("bench line malformed: " + "; ".join(problems))
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
