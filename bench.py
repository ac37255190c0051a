"""Benchmark of the MoGE layer forward on B300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one whole layer forward (routing, permutation, gather, grouped
gate/up GEMM with SwiGLU, grouped down GEMM, combine, imbalance score) over one
batch of seeded synthetic tokens, through the C ABI (moge_layer_forward).  The
headline workload is the prefill layer (T=8192, d=4096, N=64 in 8 groups,
K'=2, I=1408, bf16 with fp32 accumulation); the decode layer (T=32, same
weights) is measured in the same run and reported under "decode".

Under torchrun (N>1) every rank runs an independent replica of the layer on
its own GPU (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import signal
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import WORKLOADS, DEFAULT_SEED  # noqa: E402

METRIC = "MoGE layer tokens/s (decode T=32, prefill T=8192); % of HBM / bf16 TC roofline"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "ncu_traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
KERNEL_SRC = os.path.join(ROOT, "sparse_router_gemm_global_b300", "csrc", "ffn_tc.cu")
SHARED_EXPERTS = 4   # Pangu Pro MoE: 64 routed + 4 shared experts (explainer, section 2)


# --------------------------------------------------------------------------------------------
# environment helpers
# --------------------------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms: float, dist: bool, device) -> float:
    """The slowest rank's time (weak-scaling replicas: the job is done when every rank is)."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput of `world` independent replicas: all tokens over the slowest rank's time."""
    return tokens_per_rank * world / (ms_max / 1e3)


def peaks():
    if os.path.exists(PEAKS_PATH):
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return p, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_hash() -> str:
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(key: str):
    """DRAM bytes per launch from an ncu capture, if taken on the current kernel source."""
    if not os.path.exists(TRAFFIC_PATH):
        return None
    with open(TRAFFIC_PATH) as f:
        rec = json.load(f)
    ent = rec.get(key)
    if not ent or ent.get("kernel_sha256_16") != kernel_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed region runs.  Every sample carries
    nvidia-smi's own timestamp, so only samples taken inside the marked region are summarised
    (the tool's start-up time and output buffering do not matter)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moge_clocks_{os.getpid()}.csv")
        self.t_start = self.t_end = None

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(1.0)  # let the tool start before the region begins
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def mark_start(self):
        import datetime
        self.t_start = datetime.datetime.now()

    def mark_end(self):
        import datetime
        self.t_end = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.send_signal(signal.SIGINT)  # lets the tool flush its output
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        import datetime
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]), parts[6:10]))
                except ValueError:
                    continue
        os.unlink(self.path)
        lo = self.t_start - datetime.timedelta(seconds=0.05) if self.t_start else None
        hi = self.t_end + datetime.timedelta(seconds=0.15) if self.t_end else None
        inside = [r for r in rows if lo is None or (lo <= r[0] <= hi)]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "samples_total": len(rows),
                    "reasons": ["no sample inside the timed region"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[4]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "power_w_max": max(r[3] for r in inside), "samples": len(inside), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------------------------

def upload(inp, device):
    import torch
    out = {}
    for k, v in inp.items():
        v = np.ascontiguousarray(v)
        if v.dtype == np.uint16:
            out[k] = torch.from_numpy(v.view(np.int16)).to(device).view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(v).to(device)
    return out


class Layer:
    """Device buffers of one workload and the C-ABI call of one step (with n_shared shared experts
    when n_shared > 0; the weight tensors then hold N + n_shared experts)."""

    def __init__(self, w, d_inp, device, n_shared=0, residual=False):
        import torch
        import sparse_router_gemm_global_b300 as moge
        self.moge, self.w, self.dev, self.n_shared = moge, w, device, n_shared
        self.cfg = moge.make_config(w.T, w.d, w.N, w.M, w.kpg, w.I, w.dtype)
        self.ws = moge.alloc_workspace(self.cfg, device, n_shared=n_shared)
        self.d = d_inp
        self.x = d_inp["x"][: w.T].contiguous()
        self.y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=device)
        # residual stream of the same shape (a copy of the tokens; y = r + layer, out of place)
        self.r = self.x.clone() if residual else None
        self.aux = {"counts": torch.empty(w.N, dtype=torch.int32, device=device),
                    "group_load": torch.empty(w.M, dtype=torch.int32, device=device),
                    "score": torch.empty(4, dtype=torch.float32, device=device)}

    def step(self, x=None, y=None):
        d = self.d
        x = self.x if x is None else x
        y = self.y if y is None else y
        if self.r is not None:
            self.moge.moge_layer_forward_residual(self.cfg, self.n_shared, x, self.r, d["w_router"], d["bias"],
                                                  d["w_gate"], d["w_up"], d["w_down"], y, self.ws, aux=self.aux)
        elif self.n_shared:
            self.moge.moge_layer_forward_shared(self.cfg, self.n_shared, x, d["w_router"], d["bias"], d["w_gate"],
                                                d["w_up"], d["w_down"], y, self.ws, aux=self.aux)
        else:
            self.moge.moge_layer_forward(self.cfg, x, d["w_router"], d["bias"], d["w_gate"], d["w_up"],
                                         d["w_down"], y, self.ws, aux=self.aux)


EVENT_STRIDE = 10  # the gate/up GEMM is timed on every 10th step of the timed region
# Minimum warm-up time before each timed region (on top of --warmup steps).  Measured on a B300:
# from idle, 5 warm-up steps left the prefill step 0.8 % faster than its steady state (4.28 vs
# 4.32 ms); right after the prefill, the decode step needs ~100 steps (30 ms) to recover from
# 0.337 to 0.317 ms.
WARM_S = {"prefill": 0.5, "decode": 0.2}


def warm_up(layer, steps, min_seconds):
    """At least `steps` steps and at least `min_seconds` of them: under the power cap the SM clock
    takes tens of milliseconds to settle after a change of load (up from idle, or down to a
    lighter layer after a heavy one), and the timed region should see the layer's own steady
    state, not the previous one."""
    import torch
    t0 = time.perf_counter()
    for _ in range(steps):
        layer.step()
    torch.cuda.synchronize()
    while time.perf_counter() - t0 < min_seconds:
        for _ in range(10):
            layer.step()
        torch.cuda.synchronize()


def timed_steps(layer, steps, warmup, dist, clock=None, min_warm_s=0.0):
    """K steps bracketed by barrier + synchronize, after warm_up(warmup, min_warm_s).  Inside the
    timed region the library records the two events around the grouped gate/up GEMM (the roofline
    kernel), on its own stream, on every EVENT_STRIDE-th step: each recorded event costs the step a
    few microseconds, so the step time carries almost none of that instrumentation while the GEMM
    is still timed live.  Returns (ms/step max over ranks, gate/up ms per launch, kernel launches
    in the region)."""
    import torch
    moge = layer.moge
    warm_up(layer, warmup, min_warm_s)
    gu, dn = moge.STAGE_NAMES.index("gate_up"), moge.STAGE_NAMES.index("down")
    evs = []
    for i in range(steps):
        if i % EVENT_STRIDE:
            evs.append(None)
            continue
        row = [None] * (moge.MOGE_NUM_STAGES + 1)
        row[gu], row[gu + 1] = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for e in (row[gu], row[gu + 1]):
            e.record()  # torch creates the CUDA event on first record: do that outside the timed region
        evs.append(row)
    assert gu + 1 == dn
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    n0 = moge.moge_kernel_launch_count()
    if clock:
        clock.mark_start()
    start.record()
    for i in range(steps):
        moge.moge_set_stage_events(evs[i])
        layer.step()
    end.record()
    torch.cuda.synchronize()
    if clock:
        clock.mark_end()
    moge.moge_set_stage_events(None)
    evs = [e for e in evs if e is not None]
    launches = moge.moge_kernel_launch_count() - n0
    if dist:
        torch.distributed.barrier()
    ms = max_over_ranks(start.elapsed_time(end) / steps, dist, layer.dev)
    gate_up_ms = statistics.fmean(e[gu].elapsed_time(e[gu + 1]) for e in evs)
    if moge.moge_query_device_status(layer.ws) != 0:
        raise RuntimeError("device status reports a timed-out wait")
    return ms, gate_up_ms, launches


def stage_breakdown(layer, steps):
    """Device time of every stage (events at every stage boundary; outside the timed region,
    since each recorded event adds a few microseconds to the step)."""
    import torch
    moge = layer.moge
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moge.MOGE_NUM_STAGES + 1)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        moge.moge_set_stage_events(evs[i])
        layer.step()
    torch.cuda.synchronize()
    moge.moge_set_stage_events(None)
    return {name: round(statistics.fmean(e[s].elapsed_time(e[s + 1]) for e in evs), 5)
            for s, name in enumerate(moge.STAGE_NAMES)}


def step_distribution(layer, steps, min_warm_s):
    """Median / min / max of single steps, from a separate pass with one event pair around each
    step, after its own warm-up: after even a second of idle (the clock sampler shutting down) the
    SM clock is up at its boost value and the first ~100 ms of steps run faster than the layer's
    power-capped steady state (measured: a 3.43 ms median without this warm-up against 4.17 ms)."""
    import torch
    warm_up(layer, 3, min_warm_s)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record()
        layer.step()
        b.record()
    torch.cuda.synchronize()
    t = sorted(a.elapsed_time(b) for a, b in evs)
    return {"median": round(statistics.median(t), 5), "min": round(t[0], 5), "max": round(t[-1], 5), "steps": steps}


def graph_steps(layer, steps, dist, min_warm_s=0.0):
    """The same step captured once into a CUDA graph and replayed `steps` times: no host work per
    step (no argument checks, tensor-map encoding or launch calls).  Warm-up: at least 3 replays
    and min_warm_s seconds of them.  ms per step from CUDA events around the replays, max over
    ranks."""
    import torch
    layer.moge.moge_set_stage_events(None)
    layer.step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.step()
    t0 = time.perf_counter()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    while time.perf_counter() - t0 < min_warm_s:
        for _ in range(10):
            g.replay()
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start.record()
    for _ in range(steps):
        g.replay()
    end.record()
    torch.cuda.synchronize()
    if layer.moge.moge_query_device_status(layer.ws) != 0:
        raise RuntimeError("device status word set during the graph replays")
    del g
    return max_over_ranks(start.elapsed_time(end) / steps, dist, layer.dev)


def e2e_steps(layer, steps, dist):
    """Same metric through the public call with host buffers.  Every step copies its input x from
    pinned host memory to the device and its output y back to pinned host memory.  The copies run
    on their own streams, two buffers deep: the upload of step i+1 and the download of step i-1
    overlap the layer of step i (what a serving loop does), and each buffer is reused only after
    the step that last touched it is done with it."""
    import torch
    w = layer.w
    nb = 2
    x_host = [layer.x.cpu().pin_memory() for _ in range(nb)]
    y_host = [torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    x_dev = [torch.empty_like(layer.x) for _ in range(nb)]
    y_dev = [torch.empty_like(layer.y) for _ in range(nb)]
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ev_in, ev_comp, ev_out = [ev() for _ in range(nb)], [ev() for _ in range(nb)], [ev() for _ in range(nb)]
    for b in range(nb):  # all "previous use" events start completed
        ev_comp[b].record(comp)
        ev_out[b].record(comp)

    def run(n):
        for i in range(n):
            b = i % nb
            up.wait_event(ev_comp[b])            # step i-nb has finished reading x_dev[b]
            with torch.cuda.stream(up):
                x_dev[b].copy_(x_host[b], non_blocking=True)
            ev_in[b].record(up)
            comp.wait_event(ev_in[b])
            comp.wait_event(ev_out[b])           # step i-nb's output has left y_dev[b]
            layer.step(x=x_dev[b], y=y_dev[b])
            ev_comp[b].record(comp)
            down.wait_event(ev_comp[b])
            with torch.cuda.stream(down):
                y_host[b].copy_(y_dev[b], non_blocking=True)
            ev_out[b].record(down)
        for b in range(nb):
            comp.wait_event(ev_out[b])

    t0 = time.perf_counter()  # warm-up: at least 3 steps and WARM_S["prefill"] seconds
    run(3)
    torch.cuda.synchronize()
    while time.perf_counter() - t0 < WARM_S["prefill"]:
        run(10)
        torch.cuda.synchronize()
    if dist:
        torch.distributed.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    up.wait_stream(comp)
    run(steps)
    end.record(comp)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end) / steps, dist, layer.dev)
    return ms, x_host[0].numel() * 2, y_host[0].numel() * 2


def imbalance_study(batches, device):
    """moge_imbalance_study over `batches` batches of the routing workload's shape (T=16384,
    N=64 in 8 groups, K'=2, the same popularity bias): device time and the distribution of the
    imbalance score for MoGE and for global top-16."""
    import torch
    import sparse_router_gemm_global_b300 as moge
    w = WORKLOADS["routing_16k"]
    c = moge.make_config(w.T, 0, w.N, w.M, w.kpg, 0, "f32")
    bias = torch.from_numpy(synth.router_bias(DEFAULT_SEED, w.N)).to(device)
    lg = torch.empty((batches, w.M), dtype=torch.int32, device=device)
    lc = torch.empty_like(lg)
    ig = torch.empty(batches, dtype=torch.float32, device=device)
    ic = torch.empty_like(ig)
    moge.moge_imbalance_study(c, batches, DEFAULT_SEED, bias, lg, lc, ig, ic)  # warm-up
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    moge.moge_imbalance_study(c, batches, DEFAULT_SEED, bias, lg, lc, ig, ic)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e)
    g, glob = ig.cpu().numpy(), ic.cpu().numpy()
    return {"workload": f"{w.name} x {batches} batches", "batches": batches, "ms": round(ms, 3),
            "tokens_per_s": round(batches * w.T / (ms / 1e3), 1),
            "moge": {"mean": float(g.mean()), "max": float(g.max())},
            "global_topk": {"mean": round(float(glob.mean()), 4), "min": round(float(glob.min()), 4),
                            "max": round(float(glob.max()), 4), "frac_above_zero": float((glob > 0).mean())}}


def gate_up_roofline(w, counts, stage_ms, pk, peak_kind, sm_mhz=None):
    """Roofline of the dominant kernel (grouped gate/up GEMM + SwiGLU) from its launch time in the
    timed region.  Tensor-bound shapes: `frac` against the measured burst bf16 figure (cuBLAS timed
    alone), `frac_sustained` against the seconds-long power-capped figure, and the SM clock
    sampled in the timed region beside the clock the sustained figure was measured at (the
    sustained denominator is only comparable at the same clock)."""
    P = w.P
    touched = int((counts > 0).sum())
    flops = 4.0 * P * w.d * w.I
    bytes_alg = touched * 2 * w.I * w.d * 2 + P * w.d * 2 + P * w.I * 2
    sec = stage_ms / 1e3
    if w.T >= 1024:  # tensor-core bound shape
        achieved = flops / sec / 1e12
        peak = pk["bf16_tflops"]
        rl = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
              "frac": round(achieved / peak, 4), "peak_kind": f"bf16 burst, {peak_kind}",
              "frac_sustained": round(achieved / pk["bf16_tflops_sustained"], 4),
              "sm_mhz_timed_region": sm_mhz,
              "sm_mhz_of_sustained_peak": (pk.get("clocks_under_load") or {}).get("sm_mhz_median"),
              "algorithmic_per_launch": {"flop": flops}, "kernel": "gate_up grouped GEMM + SwiGLU"}
    else:
        achieved = bytes_alg / sec / 1e9
        peak = pk["hbm_gbs"]
        rl = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
              "frac": round(achieved / peak, 4), "peak_kind": f"HBM copy, {peak_kind}",
              "algorithmic_per_launch": {"bytes": bytes_alg, "touched_experts": touched},
              "kernel": "gate_up grouped GEMM + SwiGLU"}
    rl["traffic"] = recorded_traffic(w.name + ":gate_up")
    rl["launch_ms"] = round(stage_ms, 5)
    return rl


def layer_roofline(w, counts, ms, pk):
    """Whole-layer fractions: FLOP (grouped GEMMs + router) against the bf16 peaks (burst and
    sustained), touched expert weight bytes against the HBM peak, and the fraction of the
    max(tensor time, HBM time) roofline."""
    touched = int((counts > 0).sum())
    flops = 6.0 * w.P * w.d * w.I + 2.0 * w.T * w.d * w.N
    wbytes = touched * 3 * w.I * w.d * 2
    sec = ms / 1e3
    t_roof = max(flops / (pk["bf16_tflops"] * 1e12), wbytes / (pk["hbm_gbs"] * 1e9))
    return {"tflops": round(flops / sec / 1e12, 2),
            "tc_frac": round(flops / sec / 1e12 / pk["bf16_tflops"], 4),
            "tc_frac_sustained": round(flops / sec / 1e12 / pk["bf16_tflops_sustained"], 4),
            "weight_gbs": round(wbytes / sec / 1e9, 1), "hbm_frac": round(wbytes / sec / 1e9 / pk["hbm_gbs"], 4),
            "roofline_ms": round(t_roof * 1e3, 4), "roofline_frac": round(t_roof / sec, 4),
            "touched_experts": touched, "flop": flops, "weight_bytes": wbytes}


def _time_loop(step, steps, min_warm_s=0.1):
    """ms per call of step() from CUDA events around `steps` calls, after at least 3 calls and
    min_warm_s seconds of warm-up."""
    import torch
    t0 = time.perf_counter()
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    while time.perf_counter() - t0 < min_warm_s:
        for _ in range(10):
            step()
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        step()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def routing_bench(steps, device, pk):
    """The routing workload (Pangu Pro MoE explainer, section 1): 16384 tokens, fp32 scores
    N(0,1) + the popularity bias over 64 experts in 8 groups.  One step = moge_route from the
    given scores + moge_permute (counts, offsets, pair rows, row tokens) + moge_imbalance_score,
    for MoGE routing at K'=2 and K'=1 and for plain global top-K (K = 16, 8) on the same scores.
    The 4 MiB of scores and the outputs stay in L2 between steps (stated, not flushed)."""
    import torch
    import sparse_router_gemm_global_b300 as moge
    w = WORKLOADS["routing_16k"]
    logits = torch.from_numpy(synth.route_logits(DEFAULT_SEED, w.T, w.N)).to(device)
    out = {"workload": w.name, "T": w.T, "N": w.N, "M": w.M, "unit": "tokens/s", "steps": steps,
           "step": "moge_route (given fp32 scores) + moge_permute (no row copy) + moge_imbalance_score",
           "l2": "L2-resident: 4 MiB of scores, at most 7 MiB of outputs"}
    i32 = torch.int32
    for kpg in (2, 1):
        c = moge.make_config(w.T, 0, w.N, w.M, kpg, 0, "f32")
        ws = moge.alloc_workspace(c, device)
        K = w.M * kpg
        idx = torch.empty((w.T, K), dtype=i32, device=device)
        gate = torch.empty((w.T, K), dtype=torch.float32, device=device)
        counts = torch.empty(w.N, dtype=i32, device=device)
        offsets = torch.empty(w.N + 1, dtype=i32, device=device)
        pair_row = torch.empty((w.T, K), dtype=i32, device=device)
        row_token = torch.empty(w.T * K, dtype=i32, device=device)
        loads = torch.empty(w.M, dtype=i32, device=device)
        score = torch.empty(4, dtype=torch.float32, device=device)
        for mode, name in ((moge.MOGE_ROUTE_GROUPED, f"moge_k{kpg}"), (moge.MOGE_ROUTE_GLOBAL_TOPK, f"global_top{K}")):
            def step():
                moge.moge_route(c, mode, None, None, None, logits, idx, gate, ws)
                moge.moge_permute(c, idx, None, counts, offsets, pair_row, row_token, None, ws)
                moge.moge_imbalance_score(c, counts, loads, score)
            ms = _time_loop(step, steps)
            # bytes each step must move at least: scores in, idx + gate + pair_row + row_token out
            alg = w.T * w.N * 4 + 4 * w.T * K * 4
            out[name] = {"K": K, "ms_per_step": round(ms, 5), "value": round(w.T / (ms / 1e3), 1),
                         "imbalance_score": round(float(score[0].item()), 5),
                         "gbs": round(alg / (ms / 1e3) / 1e9, 1),
                         "hbm_frac": round(alg / (ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)}
        del ws
    return out


def tiny_bench(steps, device):
    """The tiny all-fp32 layer (T=64, d=256, N=16 in 4 groups, K'=1, I=128; CUDA-core FMA path):
    one moge_layer_forward per step, inputs resident and L2-resident (6.3 MB of weights)."""
    import torch
    import sparse_router_gemm_global_b300 as moge
    w = WORKLOADS["tiny_fp32"]
    d = upload(synth.layer_inputs(w, seed=DEFAULT_SEED), device)
    c = moge.make_config(w.T, w.d, w.N, w.M, w.kpg, w.I, w.dtype)
    ws = moge.alloc_workspace(c, device)
    y = torch.empty((w.T, w.d), dtype=torch.float32, device=device)

    def step():
        moge.moge_layer_forward(c, d["x"], d["w_router"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], y, ws)
    ms = _time_loop(step, steps)
    return {"workload": w.name, "dtype": "f32", "value": round(w.T / (ms / 1e3), 1), "unit": "tokens/s",
            "ms_per_step": round(ms, 5), "steps": steps, "l2": "L2-resident (6.3 MB of fp32 weights)"}


def stress_bench(steps, warmup, dist, device, pk, ws_n, cpu=False):
    """The large-sparse stress layer (T=4096, d=7680, N=256 in 8 groups of 32, K'=1, I=2048; the
    dimensions of the Pangu Ultra MoE page with MoGE routing imposed): one moge_layer_forward per
    step, 24 GB of expert weights resident (larger than L2).  Both roofline fractions: FLOP of the
    grouped GEMMs + router against the bf16 peaks, and the weight bytes of the touched experts
    against the HBM peak; `roofline_frac` = max(tensor time, HBM time) / step time.  With `cpu`,
    also the oracle on this layer (routing of every token + the FFN of 8 tokens per thread)."""
    w = WORKLOADS["stress_n256"]
    inp = synth.layer_inputs(w, seed=DEFAULT_SEED)
    d_inp = upload(inp, device)
    L = Layer(w, d_inp, device)
    ms, _, launches = timed_steps(L, steps, warmup, dist, min_warm_s=WARM_S["prefill"])
    counts = L.aux["counts"].cpu().numpy()
    res = {"workload": w.name, "T": w.T, "d": w.d, "N": w.N, "M": w.M, "k_per_group": w.kpg, "K": w.K, "I": w.I,
           "value": round(job_tokens_per_s(w.T, ws_n, ms), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
           "steps": steps, "gpu_launches": int(launches), "rows_per_expert_max": int(counts.max()),
           "experts_with_at_most_64_rows": int(((counts > 0) & (counts <= 64)).sum()),
           "layer_roofline": layer_roofline(w, counts, ms, pk)}
    del L, d_inp
    if cpu:
        import oracle
        sec, t_route, t_ffn, n = oracle_layer_rate(w, inp, REF_TOKENS_PER_THREAD * oracle.num_threads(),
                                                   np.random.default_rng(0))
        res["cpu_baseline"] = {"value": round(1.0 / sec, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
                               "kind": "oracle", "route_s": round(t_route, 3), "ffn_s": round(t_ffn, 3),
                               "sample": f"routing of all {w.T} tokens + FFN and combine of {n} sampled tokens, "
                                         f"per-token cost extrapolated"}
    del inp
    return res


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or "unknown"


def oracle_layer_rate(w, inp, n_ffn, rng):
    """The oracle on one workload: routing of all T tokens (the permutation needs every token),
    then the expert FFN + combine of n_ffn tokens (all T when n_ffn >= T, else a seeded sample).
    Returns (seconds per token with the FFN cost extrapolated to T, routing s, FFN s, FFN tokens)."""
    import oracle
    t0 = time.perf_counter()
    r = oracle.route(oracle.router_logits(inp["x"], inp["w_router"], inp["bias"]), w.M, w.kpg)
    t_route = time.perf_counter() - t0
    n = min(max(1, n_ffn), w.T)
    sample = np.arange(w.T, dtype=np.int32) if n == w.T else \
        np.sort(rng.choice(w.T, n, replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    oracle.combine_tokens(sample, r["idx"], r["gate64"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"])
    t_ffn = time.perf_counter() - t0
    return t_route / w.T + t_ffn / n, t_route, t_ffn, n


REF_TOKENS_PER_THREAD = 8  # oracle FFN tokens per thread in a reference-arm step


def cpu_baseline(w, inp, wd, budget_s=8.0):
    """The oracle as it stands on this host's cores, at every thread and at one thread: the
    prefill layer (routing of every token + the FFN of a token sample sized to ~budget_s,
    extrapolated per token) and the decode layer in full (all threads; one thread: a sample)."""
    import oracle
    cores = oracle.num_threads()
    rng = np.random.default_rng(0)
    d_inp = {k: (v[: wd.T] if k == "x" else v) for k, v in inp.items()}
    res = {"unit": "tokens/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model()}
    try:
        for threads in (cores, 1):
            oracle.set_num_threads(threads)
            # prefill FFN sample: REF_TOKENS_PER_THREAD tokens per thread (the reference arm's
            # sample, so that the two agree), more while a 2-token probe says budget_s allows
            # (a quarter of it at one thread), always a whole number of tokens per thread
            _, _, t_probe, _ = oracle_layer_rate(wd, d_inp, 2, rng)
            budget = budget_s if threads > 1 else budget_s / 4
            per_thread = max(REF_TOKENS_PER_THREAD, int(budget / max(t_probe / 2, 1e-9) / threads))
            n = int(min(w.T, threads * per_thread if threads > 1 else 3))
            sec, t_route, t_ffn, n = oracle_layer_rate(w, inp, n, rng)
            dn = wd.T if threads > 1 else 4
            dsec, dt_route, dt_ffn, dn = oracle_layer_rate(wd, d_inp, dn, rng)
            key = "threads_all" if threads > 1 else "threads_1"
            res[key] = {
                "threads": threads,
                "prefill": {"value": round(1.0 / sec, 3), "route_s": round(t_route, 3), "ffn_s": round(t_ffn, 3),
                            "ffn_tokens": n, "extrapolated": n < w.T},
                "decode": {"value": round(1.0 / dsec, 3), "route_s": round(dt_route, 4), "ffn_s": round(dt_ffn, 3),
                           "ffn_tokens": dn, "extrapolated": dn < wd.T}}
    finally:
        oracle.set_num_threads(cores)
    # the tiny all-fp32 layer in full, and the routing workload in full (scores given: softmax,
    # group top-K', gates, permutation, imbalance score)
    wt = WORKLOADS["tiny_fp32"]
    sec, _, _, _ = oracle_layer_rate(wt, synth.layer_inputs(wt, seed=DEFAULT_SEED), wt.T, rng)
    res["tiny_fp32"] = {"value": round(1.0 / sec, 1), "tokens": wt.T}
    wr = WORKLOADS["routing_16k"]
    logits = synth.route_logits(DEFAULT_SEED, wr.T, wr.N)
    t0 = time.perf_counter()
    oracle.route(logits, wr.M, wr.kpg)
    res["routing_16k"] = {"value": round(wr.T / (time.perf_counter() - t0), 1), "tokens": wr.T, "k_per_group": wr.kpg}
    res["value"] = res["threads_all"]["prefill"]["value"]
    a = res["threads_all"]["prefill"]
    res["sample"] = (f"{w.name}: routing of all {w.T} tokens + expert FFN and combine of {a['ffn_tokens']} sampled "
                     f"tokens on {cores} threads, per-token cost extrapolated to T={w.T}; {wd.name}, tiny_fp32 and "
                     f"routing_16k in full; threads_1: prefill and decode at one thread (FFN on samples); the "
                     f"stress layer's figure is under stress.cpu_baseline")
    return res


def workload_config(w, ws_n):
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": w.name, "T": w.T, "d": w.d, "N": w.N, "M": w.M, "k_per_group": w.kpg, "K": w.K, "I": w.I,
            "seed": DEFAULT_SEED, "parallelism": f"replicas x{ws_n}",
            "l2": "inputs larger than L2 (2.2 GB of expert weights, 1 GB permuted activations)"}


def run_ours(args):
    import torch
    for k in WARM_S:
        WARM_S[k] *= max(args.warm_scale, 0.0)
    ws_n, rank, local = dist_env()
    dist = ws_n > 1
    if dist:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pk, peak_kind = peaks()

    wp = WORKLOADS[args.workload]
    if args.tokens:  # a smaller token count of the same layer (profiling captures)
        wp = wp.with_(name=f"{wp.name}[T={args.tokens}]", T=args.tokens)
    wd = WORKLOADS["decode_t32"]
    # decode reuses the same weights and the first 32 tokens; the weight tensors also hold the
    # shared experts of the shared-expert measurement (the routed layer reads the first N)
    inp = synth.layer_inputs(wp, seed=DEFAULT_SEED, n_shared=SHARED_EXPERTS)
    d_inp = upload(inp, device)

    prefill = Layer(wp, d_inp, device)
    phys = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local] if dist else \
        os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
    gpu_index = int(phys) if phys.isdigit() else local
    with ClockSampler(gpu_index) as clk:
        ms, gate_up_ms, launches = timed_steps(prefill, args.steps, args.warmup, dist, clock=clk,
                                               min_warm_s=WARM_S["prefill"])
    clocks = clk.summary()
    step_dist = step_distribution(prefill, min(max(args.steps, 20), 100), WARM_S["prefill"])
    stages = stage_breakdown(prefill, min(args.steps, 50))
    counts = prefill.aux["counts"].cpu().numpy()
    score = float(prefill.aux["score"][0].item())

    # decode shape, same weights
    decode = None
    if args.decode_steps > 0:
        dec = Layer(wd, d_inp, device)
        dms, dgate_up_ms, dlaunches = timed_steps(dec, args.decode_steps, max(args.warmup, 3), dist,
                                                  min_warm_s=WARM_S["decode"])
        dstep_dist = step_distribution(dec, min(max(args.decode_steps, 20), 200), WARM_S["decode"])
        dstages = stage_breakdown(dec, min(args.decode_steps, 100))
        dgraph = None
        if args.graph_steps > 0:
            dgms = graph_steps(dec, 3 * args.graph_steps, dist, min_warm_s=WARM_S["decode"])
            dgraph = {"value": round(job_tokens_per_s(wd.T, ws_n, dgms), 1), "unit": "tokens/s",
                      "ms_per_step": round(dgms, 4), "steps": 3 * args.graph_steps}
        dcounts = dec.aux["counts"].cpu().numpy()
        decode = {"workload": wd.name, "value": round(job_tokens_per_s(wd.T, ws_n, dms), 1), "unit": "tokens/s",
                  "ms_per_step": round(dms, 4), "steps": args.decode_steps,
                  "roofline": gate_up_roofline(wd, dcounts, dgate_up_ms, pk, peak_kind),
                  "layer_roofline": layer_roofline(wd, dcounts, dms, pk),
                  "step_ms_distribution": dstep_dist,
                  "stage_share_ms": dstages, "cuda_graph": dgraph, "gpu_launches": int(dlaunches)}

    # the prefill step captured as a CUDA graph (after the decode timing: its replays are a
    # seconds-long load that would leave the short decode window starting power-throttled)
    graph = None
    if args.graph_steps > 0:
        gms = graph_steps(prefill, args.graph_steps, dist, min_warm_s=WARM_S["prefill"])
        graph = {"value": round(job_tokens_per_s(wp.T, ws_n, gms), 1), "unit": "tokens/s",
                 "ms_per_step": round(gms, 4), "steps": args.graph_steps}

    # the same layers with Pangu Pro's 4 shared experts added (every token visits each of them)
    shared = None
    if args.shared_steps > 0:
        shared = {"n_shared": SHARED_EXPERTS}
        for name, w, n in (("prefill", wp, args.shared_steps), ("decode", wd, 3 * args.shared_steps)):
            L = Layer(w, d_inp, device, n_shared=SHARED_EXPERTS)
            sms, _, _ = timed_steps(L, n, max(args.warmup, 3), dist, min_warm_s=WARM_S[name])
            rows = w.P + SHARED_EXPERTS * w.T
            shared[name] = {"workload": f"{w.name}+{SHARED_EXPERTS}shared",
                            "value": round(job_tokens_per_s(w.T, ws_n, sms), 1), "unit": "tokens/s",
                            "ms_per_step": round(sms, 4), "steps": n,
                            "tflops": round(6.0 * rows * w.d * w.I / (sms / 1e3) / 1e12, 2)}
            del L

    # Pangu Pro MoE's own dimensions: hidden 5120, top-1 per group (K = 8), 4 shared experts, the
    # output added to a residual stream (the whole MoE block of one Pangu Pro layer)
    pangu = None
    if args.pangu_steps > 0:
        pangu = {"n_shared": SHARED_EXPERTS}
        wpp, wpd = WORKLOADS["pangu_k1_t8192"], WORKLOADS["pangu_k1_t32"]
        p_inp = upload(synth.layer_inputs(wpp, seed=DEFAULT_SEED, n_shared=SHARED_EXPERTS), device)
        for name, w, n in (("prefill", wpp, args.pangu_steps), ("decode", wpd, 3 * args.pangu_steps)):
            L = Layer(w, p_inp, device, n_shared=SHARED_EXPERTS, residual=True)
            pms, _, _ = timed_steps(L, n, max(args.warmup, 3), dist, min_warm_s=WARM_S[name])
            rows = w.P + SHARED_EXPERTS * w.T
            touched = int((L.aux["counts"].cpu().numpy() > 0).sum()) + SHARED_EXPERTS
            pangu[name] = {"workload": f"{w.name}+{SHARED_EXPERTS}shared+residual", "d": w.d, "I": w.I, "K": w.K,
                           "value": round(job_tokens_per_s(w.T, ws_n, pms), 1), "unit": "tokens/s",
                           "ms_per_step": round(pms, 4), "steps": n,
                           "tflops": round(6.0 * rows * w.d * w.I / (pms / 1e3) / 1e12, 2),
                           "weight_gbs": round(touched * 3 * w.d * w.I * 2 / (pms / 1e3) / 1e9, 1),
                           "touched_experts": touched}
            del L
        del p_inp

    # Monte-Carlo imbalance study on the routing workload's shape (MoGE vs global top-K)
    study = None
    if args.study_batches > 0:
        study = imbalance_study(args.study_batches, device)

    # the routing workload (route + permute + imbalance score) and the tiny all-fp32 layer
    routing = routing_bench(args.routing_steps, device, pk) if args.routing_steps > 0 else None
    tiny = tiny_bench(args.tiny_steps, device) if args.tiny_steps > 0 else None

    # end to end through the public call with host buffers
    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = e2e_steps(prefill, max(3, args.steps // 2), dist)
        e2e = {"value": round(job_tokens_per_s(wp.T, ws_n, e2e_ms), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
               "copies": "pinned host buffers; upload of step i+1 and download of step i-1 overlap step i"}

    # the large-sparse stress layer (24 GB of weights, generated last so the other layers' inputs
    # are released first)
    stress = None
    if args.stress_steps > 0:
        del prefill, d_inp
        stress = stress_bench(args.stress_steps, max(args.warmup, 3), dist, device, pk, ws_n,
                              cpu=rank == 0 and ws_n == 1 and not args.no_cpu_baseline)

    res = {
        "metric": METRIC,
        "value": round(job_tokens_per_s(wp.T, ws_n, ms), 1),
        "unit": "tokens/s",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "warmup_min_seconds": WARM_S,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded splitmix64 + Box-Muller; random-init weights N(0,1/fan_in), "
                "router bias 1.5 ln(1/rank_e))",
        "config": workload_config(wp, ws_n),
        "roofline": gate_up_roofline(wp, counts, gate_up_ms, pk, peak_kind, sm_mhz=clocks.get("sm_mhz")),
        "layer_roofline": layer_roofline(wp, counts, ms, pk),
        "step_ms_distribution": step_dist,
        "stage_share_ms": stages,
        "stage_share_note": ("stage durations from a separate pass with events at every stage boundary "
                             "(those events break the launch overlap): shares of the step, not absolute "
                             "times in the timed region"),
        "cuda_graph": graph,
        "imbalance_score": score,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "decode": decode,
        "shared_experts": shared,
        "pangu_dims_k1": pangu,
        "imbalance_study": study,
        "stress": stress,
        "routing": routing,
        "tiny_fp32": tiny,
    }
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wp, inp, wd, budget_s=args.cpu_budget)
    if dist:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


# --------------------------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands (no reference code exists to install)
# --------------------------------------------------------------------------------------------

def run_reference(args):
    """The CPU oracle as it stands, on the host cores.  Each step routes all T tokens and runs the
    expert FFN + combine of a token sample (8 tokens per oracle thread by default, so that every
    core works, as in the CPU baseline of our arm); `ms_per_step` is the wall time of the step
    actually run, and the per-token cost extrapolated to a whole T-token layer is reported
    separately as `extrapolated_layer_ms`."""
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = WORKLOADS[args.workload]
    inp = synth.layer_inputs(w, seed=DEFAULT_SEED)
    cores = oracle.num_threads()
    rng = np.random.default_rng(0)
    n_sample = args.ref_tokens if args.ref_tokens > 0 else REF_TOKENS_PER_THREAD * cores
    for _ in range(args.warmup):
        oracle_layer_rate(w, inp, n_sample, rng)
    per_tok, wall = [], []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        sec, _, _, _ = oracle_layer_rate(w, inp, n_sample, rng)
        wall.append(time.perf_counter() - t0)
        per_tok.append(sec)
    sec = statistics.fmean(per_tok)
    value = round(1.0 / sec, 3)
    sample_desc = (f"{w.name}: each step routes all {w.T} tokens and runs the expert FFN + combine of "
                   f"{n_sample} sampled tokens on {cores} threads; tokens/s = per-token cost extrapolated "
                   f"to T={w.T}")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.fmean(wall) * 1e3, 2),
        "extrapolated_layer_ms": round(sec * w.T * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": workload_config(w, ws_n),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample_desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# --------------------------------------------------------------------------------------------
# DRAM traffic of the grouped GEMM from an ncu capture (profiles/ncu_traffic.json)
# --------------------------------------------------------------------------------------------

def traffic_stage(name: str, prev_key):
    """The record key of one grouped-GEMM launch of an ncu capture of this bench, from its kernel
    name and the key of the GEMM launch before it (launch order: the prefill layer's CTA-pair
    gate/up, its small-expert weights-as-M gate/up, the pair down, the small-expert down; then the
    decode layer's weights-as-M gate/up, gathering its rows, and down).  Returns (key, counts the
    stage's launches) or None for other kernels."""
    if "ffn_tc_pair_kernel<1" in name:     # <GLU = 1, regions>
        return "prefill_t8192:gate_up", True
    if "ffn_tc_pair_kernel<0" in name:
        return "prefill_t8192:down", True
    if "ffn_tc_kernel<2, 32, 1>" in name:
        return "decode_t32:gate_up", True
    if "ffn_tc_kernel<2, 32, 0>" in name:   # small experts of the prefill layer
        return "prefill_t8192:gate_up", False
    if "ffn_tc_kernel<3, 32, 0>" in name:   # small experts of the prefill layer, or the decode down
        return ("decode_t32:down", True) if prev_key == "decode_t32:gate_up" else ("prefill_t8192:down", False)
    return None


def record_traffic(csv_path: str, command: str) -> None:
    """dram__bytes_read.sum + dram__bytes_write.sum per stage of each grouped GEMM in an ncu --csv
    capture of this bench at full size, stamped with the kernel source hash.  A prefill stage is
    one launch of the CTA-pair kernel plus one of the small-expert kernel: the stage's bytes are the
    total over both divided by the pair kernel's launches."""
    import csv
    total, launches = {}, {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(f) if len(r) > 10]
    hdr = rows[0]
    ki, ii, mi, vi = (hdr.index(k) for k in ("Kernel Name", "ID", "Metric Name", "Metric Value"))
    stage_of, prev_key = {}, None
    for r in rows[1:]:  # one stage per launch id, in launch order
        if r[ii] in stage_of:
            continue
        hit = traffic_stage(r[ki], prev_key)
        stage_of[r[ii]] = hit
        if hit is not None:
            prev_key = hit[0]
    for r in rows[1:]:
        hit = stage_of[r[ii]]
        if hit is None or not r[mi].startswith("dram__bytes_"):
            continue
        key, main_kernel = hit
        total[key] = total.get(key, 0.0) + float(r[vi].replace(",", ""))
        if main_kernel:
            launches.setdefault(key, set()).add(r[ii])
    rec = {"command": command, "kernel_sha256_16": kernel_hash()}
    for key in total:
        n = len(launches.get(key, ()))
        if n:
            rec[key] = {"kernel_sha256_16": kernel_hash(), "launches": n, "dram_bytes_per_launch": total[key] / n}
    with open(TRAFFIC_PATH, "w") as f:
        json.dump(rec, f, indent=1)
    print(json.dumps(rec, indent=1))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--decode-steps", type=int, default=300)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill_t8192", choices=["prefill_t8192"])
    ap.add_argument("--tokens", type=int, default=0, help="override T (small profiling cases)")
    ap.add_argument("--shared-steps", type=int, default=50, help="steps of the shared-expert layers (0: skip)")
    ap.add_argument("--warm-scale", type=float, default=1.0,
                    help="scale of the minimum warm-up times (0: only --warmup steps; for profiling captures)")
    ap.add_argument("--graph-steps", type=int, default=100,
                    help="replays of the step captured as a CUDA graph (decode: 3x; 0: skip)")
    ap.add_argument("--study-batches", type=int, default=1000, help="Monte-Carlo study batches (0: skip)")
    ap.add_argument("--pangu-steps", type=int, default=30, help="steps at Pangu Pro dims, K'=1 (0: skip)")
    ap.add_argument("--stress-steps", type=int, default=50, help="steps of the N=256 stress layer (0: skip)")
    ap.add_argument("--routing-steps", type=int, default=200, help="steps of the routing workload (0: skip)")
    ap.add_argument("--tiny-steps", type=int, default=200, help="steps of the tiny fp32 layer (0: skip)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=8.0, help="seconds of oracle FFN work")
    ap.add_argument("--ref-tokens", type=int, default=0,
                    help="FFN tokens per reference-arm step (0: 8 per oracle thread)")
    ap.add_argument("--record-traffic", metavar="CSV", help="write profiles/ncu_traffic.json from an ncu csv")
    ap.add_argument("--traffic-command", default="", help="the ncu command that made the csv")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(args.record_traffic, args.traffic_command)
        return
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
