"""Throughput benchmark of the attention forward on one GB300 (or N replicas).

One step = the whole hot path over one batch of synthetic input at the
Wan-2.1-720p shape (B=1, H=40, S=76112, D=128, 5 % outlier tokens x8):
    attn_fwd_bf16(Q, K, V)            BF16 flash attention
    sage_prepare(Q, K, V)             INT8 Q/K, e4m3 V
    sage_attn_fwd(prepared)           INT8 QK^T / FP8 PV attention
The metric is attention TFLOPS, 4*B*H*S^2*D per attention evaluation; a step
evaluates attention twice (BF16 and Sage), so value = 2 * 4*B*H*S^2*D * steps
/ time, summed over ranks.  Per-call times and TFLOPS are reported under
"providers".  Inputs are resident in HBM and larger than L2 (779 MB each).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (FP64 attention, plain C) on the host
cores, on bounded row samples of the same workload, in the same metric.
Under torchrun (N > 1) every rank runs an independent replica (the op has no
exchange step); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOPS (4·B·H·S²·D/s) at S=76112,H=40,D=128; % of tensor peak"
KERNELS_PER_STEP = 4  # attn_fwd (BF16), prep_qk_vmax, prep_v, attn_fwd (Sage FP8)


def kernel_traffic(record: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary profiles/<record>_traffic.json,
    or None when a source file the record lists changed since the counters were taken
    (or there is no record)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{record}_traffic.json")
    if workload != "wan720p" or not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    srcs = rec.get("sources", [])
    if not srcs or not all(os.path.exists(os.path.join(ROOT, p)) for p in srcs):
        return None
    h = hashlib.sha256(b"".join(open(os.path.join(ROOT, p), "rb").read() for p in srcs)).hexdigest()
    if h != rec.get("kernel_source_sha256"):
        return None
    return rec["dram_bytes_per_launch_wan720p_scaled"]


# ----------------------------------------------------------------------------- ranks
# One process per GPU (torchrun).  Ranks are independent replicas: nothing crosses
# between them but the barrier around the timed region and the maximum of the ranks'
# times, which these helpers carry (NCCL on the GPU path; any backend works).
def rank_info() -> tuple:
    """(rank, world size, local rank) from the launcher's environment (1 process if unset)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time: the whole job finishes when its last replica does."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, steps: int, ms: float) -> float:
    """Work of all ranks (each runs the full step) over the slowest rank's time, in TFLOPS."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


def workload_config(wl, world: int) -> dict:
    """The `config` object of the JSON line; both arms report the same one."""
    return {"workload": f"{wl.name}: B={wl.B} H={wl.H} S={wl.S} D={wl.D}"
                        + (", 5% outlier tokens x8" if wl.outlier_frac else ""),
            "B": wl.B, "H": wl.H, "S": wl.S, "D": wl.D,
            "step": "attn_fwd_bf16 + sage_attention (prepare + forward in one call; two attention evaluations)",
            "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(bf16=float(p["bf16_tflops"]), bf16_sustained=float(p["bf16_tflops_sustained"]),
                    hbm=float(p["hbm_gbs"]), source="measured")
    return dict(bf16=1900.0, bf16_sustained=1700.0, hbm=6800.0, source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
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

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------- ours
class SmClock:
    """Average SM clock over a stretch of the stream, from the library's SM clock sampler
    (every SM's %clock64 against %globaltimer): sample() before and after, mhz() once
    both have completed.  The samples are enqueued outside the event-timed spans."""

    def __init__(self, sa, torch, dev, n_sms):
        self.sa, self.torch, self.dev, self.n = sa, torch, dev, max(n_sms, 1) + 32

    def sample(self, stream):
        buf = self.torch.empty((self.n, 2), dtype=self.torch.int64, device=self.dev)
        return self.sa.sm_clock_sample(buf, stream=stream)

    def mhz(self, a, b):
        return self.sa.sm_clock_mhz(a.cpu().numpy(), b.cpu().numpy())


def time_providers(calls, stream, clk, rounds=3, warm=2, reps=5):
    """Each provider alone: `warm` warm-up calls, then `reps` calls between two events
    (and two SM clock samples); the providers take turns within each of `rounds` rounds.
    Returns name -> {"ms": median per-call ms, "sm_mhz": median clock, "mcycles": median
    per-call SM cycles / 1e6}."""
    import torch
    got = {name: [] for name in calls}
    for _ in range(rounds):
        for name, fn in calls.items():
            for _ in range(warm):
                fn()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            c0 = clk.sample(stream)
            ev[0].record(stream)
            for _ in range(reps):
                fn()
            ev[1].record(stream)
            c1 = clk.sample(stream)
            ev[1].synchronize()
            torch.cuda.synchronize()
            ms = ev[0].elapsed_time(ev[1]) / reps
            mhz = clk.mhz(c0, c1)
            got[name].append((ms, mhz, ms * mhz / 1e3 if mhz else None))
    out = {}
    for name, t in got.items():
        cyc = [c for _, _, c in t if c is not None]
        mh = [m for _, m, _ in t if m is not None]
        out[name] = {"ms": statistics.median([m for m, _, _ in t]),
                     "sm_mhz": statistics.median(mh) if mh else None,
                     "mcycles": statistics.median(cyc) if cyc else None}
    return out


def run_ours(args, rank, world):
    import torch
    import sage_attention_forward_gb300 as sa
    from sage_attention_forward_gb300 import roofline
    from workloads import WORKLOADS, make_inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    wl = WORKLOADS[args.workload]
    B, H, S, D = wl.B, wl.H, wl.S, wl.D
    inp = make_inputs(wl, device=dev)          # drawn on the device: inputs resident in HBM
    q, k, v = inp.q, inp.k, inp.v
    scale = wl.softmax_scale
    S_pad = sa.sage_padded_len(S)
    o_bf16 = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
    o_sage = torch.empty_like(o_bf16)
    prep = sa.Prepared.empty(B, H, S, S_pad, dev)
    ws_p = sa.prepare_workspace(B, H, dev)
    ws_a = sa.attn_workspace(B, H, S_pad, dev)
    ws_1 = sa.sage_attention_workspace(B, H, S, dev)
    kw = norm_rope_kwargs(inp, wl)
    stream = torch.cuda.current_stream()
    clk = SmClock(sa, torch, dev, n_sms)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        sa.attn_fwd_bf16(q, k, v, out=o_bf16, softmax_scale=scale)
        if ev is not None:
            ev[1].record(stream)
        sa.sage_attention(q, k, v, softmax_scale=scale, out=o_sage, workspace=ws_1, **kw)
        if ev is not None:
            ev[2].record(stream)

    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    sa.attn_get_device_status()
    barrier()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as smi:
        barrier()
        c_start = clk.sample(stream)
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        c_end = clk.sample(stream)
        barrier()
    sa.attn_get_device_status()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    region_mhz = clk.mhz(c_start, c_end)

    # the step's own split (each call timed inside the interleaved step)
    per = {"bf16": [], "sage": []}
    for e in evs:
        per["bf16"].append(e[0].elapsed_time(e[1]))
        per["sage"].append(e[1].elapsed_time(e[2]))
    F = roofline.attention_flops(B, H, S, D)
    step_ms = {k2: statistics.mean(v2) for k2, v2 in per.items()}
    peaks = load_peaks()

    # the same split with each call's own SM clock (clock samples between the calls of a
    # few more steps, outside the timed region): cycles take the power cap's clock out
    split = {"bf16": [], "sage": []}
    for _ in range(3):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        c0 = clk.sample(stream)
        ev[0].record(stream)
        sa.attn_fwd_bf16(q, k, v, out=o_bf16, softmax_scale=scale)
        ev[1].record(stream)
        c1 = clk.sample(stream)
        ev[2].record(stream)
        sa.sage_attention(q, k, v, softmax_scale=scale, out=o_sage, workspace=ws_1, **kw)
        ev[3].record(stream)
        c2 = clk.sample(stream)
        torch.cuda.synchronize()
        for name, a, b, e0, e1 in (("bf16", c0, c1, ev[0], ev[1]), ("sage", c1, c2, ev[2], ev[3])):
            ms = e0.elapsed_time(e1)
            mhz = clk.mhz(a, b)
            split[name].append((ms, mhz, ms * mhz / 1e3 if mhz else None))
    in_step = {name: {"ms": statistics.median([t[0] for t in v2]),
                      "sm_mhz": statistics.median([t[1] for t in v2 if t[1]]) if any(t[1] for t in v2) else None,
                      "mcycles": statistics.median([t[2] for t in v2 if t[2]]) if any(t[2] for t in v2) else None}
               for name, v2 in split.items()}

    # providers, each timed on its own: 2 warm-up + 5 back-to-back calls, 3 rounds with the
    # providers interleaved, median.  Inside the step the GPU's power management carries
    # clock headroom from one kernel into the next, which skews a per-call split; the
    # cycle counts (time x the call's own average SM clock) do not depend on it.
    o_pv16 = torch.empty_like(o_bf16)
    prep_s = sa.Prepared.empty(B, H, S, S_pad, dev)
    ws_s = sa.prepare_workspace(B, H, dev, S_pad, smooth_k=True)
    ws_16 = sa.sage_attention_workspace(B, H, S, dev, pv="bf16")
    ws_ql = sa.sage_attention_workspace(B, H, S, dev, q_on_load=True)
    ws_kl = sa.sage_attention_workspace(B, H, S, dev, q_on_load=True, k_on_load=True)
    sa.sage_prepare(q, k, v, softmax_scale=scale, S_pad=S_pad, out=prep, workspace=ws_p, **kw)
    calls = {
        "bf16": lambda: sa.attn_fwd_bf16(q, k, v, out=o_bf16, softmax_scale=scale),
        "sage": lambda: sa.sage_attention(q, k, v, softmax_scale=scale, out=o_sage, workspace=ws_1, **kw),
        "sage_two_calls": lambda: (sa.sage_prepare(q, k, v, softmax_scale=scale, S_pad=S_pad, out=prep,
                                                   workspace=ws_p, **kw),
                                   sa.sage_attn_fwd(prep, out=o_sage, workspace=ws_a)),
        "sage_pv16": lambda: sa.sage_attention(q, k, v, softmax_scale=scale, out=o_pv16, workspace=ws_16, pv="bf16",
                                               **kw),
        "sage_q_on_load": lambda: sa.sage_attention(q, k, v, softmax_scale=scale, out=o_pv16, workspace=ws_ql,
                                                    q_on_load=True, **kw),
        "sage_qk_on_load": lambda: sa.sage_attention(q, k, v, softmax_scale=scale, out=o_pv16, workspace=ws_kl,
                                                     k_on_load=True, **kw),
        "sage_core": lambda: sa.sage_attn_fwd(prep, out=o_sage, workspace=ws_a),
        "sage_pv16_core": lambda: sa.sage_attn_fwd_pv16(prep, v, out=o_pv16, workspace=ws_a),
        "prepare": lambda: sa.sage_prepare(q, k, v, softmax_scale=scale, S_pad=S_pad, out=prep, workspace=ws_p,
                                           **kw),
        "prepare_smooth_k": lambda: sa.sage_prepare(q, k, v, softmax_scale=scale, S_pad=S_pad, out=prep_s,
                                                    workspace=ws_s, smooth_k=True, **kw),
    }
    timed = time_providers(calls, stream, clk)
    sa.attn_get_device_status()
    prep_bytes = roofline.prepare_bytes(B, H, S, S_pad, D, wl.rms_norm, wl.rope_dim)
    smooth_bytes = roofline.prepare_smooth_k_bytes(B, H, S, S_pad, D, wl.rms_norm, wl.rope_dim)
    rate_bf16 = roofline.TC_FLOP_PER_CLK_SM["f16"]
    rate_sage = roofline.sage_flop_per_clk_sm()

    def attn_entry(name, rate=None, call=None):
        t = timed[name]
        e = {"ms": t["ms"], "tflops": F / (t["ms"] * 1e-3) / 1e12, "sm_mhz": t["sm_mhz"], "mcycles": t["mcycles"]}
        if rate is not None and t["sm_mhz"]:
            e["frac_of_clock_peak"] = e["tflops"] / roofline.clock_peak_tflops(rate, n_sms, t["sm_mhz"])
        if call:
            e["call"] = call
        return e

    def hbm_entry(name, nbytes):
        t = timed[name]
        gbs = nbytes / (t["ms"] * 1e-3) / 1e9
        return {"ms": t["ms"], "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm"], "sm_mhz": t["sm_mhz"]}

    providers = {
        "bf16": attn_entry("bf16", rate_bf16),
        "sage": attn_entry("sage", None, "sage_attention (prepare + forward, one call)"),
        "sage_two_calls": attn_entry("sage_two_calls", None, "sage_prepare, then sage_attn_fwd"),
        "sage_pv16": attn_entry("sage_pv16", None, "sage_attention(pv=bf16)"),
        "sage_q_on_load": attn_entry("sage_q_on_load", None, "sage_attention(q_on_load=True): Q coded by the forward"),
        "sage_qk_on_load": attn_entry("sage_qk_on_load", None,
                                      "sage_attention(k_on_load=True): Q and K coded by the forward"),
        # Q K^T on the FP16 MMA (the kind::f16 rate), P V on the e4m3 MMA (twice that rate)
        "sage_core": attn_entry("sage_core", rate_sage),
        "sage_pv16_core": attn_entry("sage_pv16_core", rate_bf16),
        "prepare": hbm_entry("prepare", prep_bytes),
        "prepare_smooth_k": hbm_entry("prepare_smooth_k", smooth_bytes),
        "timing": "each provider alone: 2 warm-up + 5 calls, 3 interleaved rounds, median; sm_mhz: the call's own "
                  "average SM clock (SM cycle counters against the GPU timer), mcycles = ms x sm_mhz / 1e3",
        "in_step_ms": step_ms,
        "in_step": in_step,
    }
    providers["sage_vs_bf16"] = {
        "alone_time_ratio": timed["sage"]["ms"] / timed["bf16"]["ms"],
        "alone_cycle_ratio": (timed["sage"]["mcycles"] / timed["bf16"]["mcycles"]
                              if timed["sage"]["mcycles"] and timed["bf16"]["mcycles"] else None),
        "in_step_time_ratio": in_step["sage"]["ms"] / in_step["bf16"]["ms"],
        "in_step_cycle_ratio": (in_step["sage"]["mcycles"] / in_step["bf16"]["mcycles"]
                                if in_step["sage"]["mcycles"] and in_step["bf16"]["mcycles"] else None),
        "note": "one-call Sage (prepare included) over BF16; below 1 means Sage is faster",
    }
    del prep_s, ws_s, o_pv16, ws_16, ws_ql, ws_kl

    # ------------------------------------------------------------- end to end
    e2e = run_e2e(args, sa, torch, dev, inp, scale, S_pad, kw, F, world, dist)

    # the roofline of the dominant kernel: the BF16 forward's average launch inside the
    # timed step, against the measured sustained BF16 peak and against the per-clock
    # tcgen05 rate at the SM clock averaged over the timed region
    roof_tflops = F / (step_ms["bf16"] * 1e-3) / 1e12
    roof = {"bound": "tensor", "kernel": "attn_fwd_bf16 (average launch inside the timed step)",
            "achieved": roof_tflops, "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
            "frac": roof_tflops / peaks["bf16_sustained"],
            "traffic": kernel_traffic("attn_fwd_bf16", wl.name),
            "peak_source": f"{peaks['source']} bf16 sustained (of {peaks['source']})"}
    if region_mhz:
        cp = roofline.clock_peak_tflops(rate_bf16, n_sms, region_mhz)
        roof.update({"sm_mhz": region_mhz, "clock_peak": cp, "frac_of_clock_peak": roof_tflops / cp,
                     "clock_peak_source": f"tcgen05 kind::f16 {rate_bf16:.0f} FLOP/clk/SM (probe) x {n_sms} SMs x "
                                          "the SM clock averaged over the timed region"})
    # the Sage forward alone: half the FLOPs at the FP16 rate, half at the e4m3 rate; the
    # measured BF16 burst peak / 0.75 is that mix at the measured rate
    sc = timed["sage_core"]
    sage_tflops = F / (sc["ms"] * 1e-3) / 1e12
    roof_sage = {"bound": "tensor", "kernel": "attn_fwd_kernel Sage FP8 mode (sage_core, timed alone)",
                 "achieved": sage_tflops, "peak": peaks["bf16"] / 0.75, "unit": "TFLOP/s",
                 "frac": sage_tflops / (peaks["bf16"] / 0.75),
                 "traffic": kernel_traffic("attn_fwd_sage_fp8", wl.name),
                 "peak_source": f"{peaks['source']} bf16 burst / 0.75 (half the FLOPs at the e4m3 rate, twice the "
                                f"BF16 rate; no INT8 tensor-core MMA on sm_103a)"}
    if sc["sm_mhz"]:
        cp = roofline.clock_peak_tflops(rate_sage, n_sms, sc["sm_mhz"])
        roof_sage.update({"sm_mhz": sc["sm_mhz"], "clock_peak": cp, "frac_of_clock_peak": sage_tflops / cp,
                          "clock_peak_source": f"{rate_sage:.0f} FLOP/clk/SM (harmonic mean of the probe's kind::f16 "
                                               f"and e4m3 rates) x {n_sms} SMs x the call's SM clock"})

    result = {
        "metric": METRIC,
        "value": whole_job_tflops(world, 2 * F, args.steps, elapsed_ms),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16+int8/e4m3",
        "data": "synthetic",
        "config": workload_config(wl, world),
        "providers": providers,
        "roofline": roof,
        "roofline_sage": roof_sage,
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "e2e": e2e,
    }
    result["clocks"] = smi.summary()
    result["clocks"]["sm_mhz_probe"] = region_mhz
    # the secondary bound of either attention path: one exp2 per score, B*H*S^2 of them, at
    # the MUFU rate measured on this part (30 results per clock per SM, f32 or packed f16x2)
    exps = wl.B * wl.H * wl.S * wl.S
    sm_hz = (region_mhz or result["clocks"].get("sm_mhz") or 2070.0) * 1e6
    result["exp_bound"] = {"exps": exps, "results_per_clk_per_sm": 30, "sm_mhz": sm_hz / 1e6,
                           "floor_ms": exps / (30 * n_sms * sm_hz) * 1e3,
                           "frac_of_bf16_step_time": exps / (30 * n_sms * sm_hz) * 1e3 / step_ms["bf16"]}
    if not args.no_per_workload:
        del prep, ws_p, ws_a, ws_1, o_bf16, o_sage, inp, q, k, v
        torch.cuda.empty_cache()
        result["per_workload"] = per_workload(sa, roofline, torch, dev, stream, clk, n_sms, wl.name)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, seconds=args.cpu_seconds)
    return result


def norm_rope_kwargs(inp, wl):
    kw = {}
    if inp.q_norm_w is not None:
        kw.update(q_norm_w=inp.q_norm_w, k_norm_w=inp.k_norm_w, rms_eps=wl.rms_eps)
    if inp.rope_cos is not None:
        kw.update(rope_cos=inp.rope_cos, rope_sin=inp.rope_sin, rope_dim=wl.rope_dim)
    return kw


PER_WORKLOADS = ("flux1024", "flux2048", "hunyuan720p")


def per_workload(sa, roofline, torch, dev, stream, clk, n_sms, skip):
    """The pages' other DiT shapes (the handbook's byte table): BF16 forward, one-call Sage
    (with the fused RMSNorm + RoPE where the workload has it) and the Sage forward alone,
    each timed on its own, with SM clocks and clock-normalised roof fractions."""
    from workloads import WORKLOADS, make_inputs
    out = {}
    for name in PER_WORKLOADS:
        if name == skip:
            continue
        wl = WORKLOADS[name]
        B, H, S, D = wl.B, wl.H, wl.S, wl.D
        inp = make_inputs(wl, device=dev)
        kw = norm_rope_kwargs(inp, wl)
        S_pad = sa.sage_padded_len(S)
        o1 = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
        o2 = torch.empty_like(o1)
        ws_1 = sa.sage_attention_workspace(B, H, S, dev)
        prep = sa.sage_prepare(inp.q, inp.k, inp.v, softmax_scale=wl.softmax_scale, **kw)
        ws_a = sa.attn_workspace(B, H, S_pad, dev)
        calls = {
            "bf16": lambda: sa.attn_fwd_bf16(inp.q, inp.k, inp.v, out=o1, softmax_scale=wl.softmax_scale),
            "sage": lambda: sa.sage_attention(inp.q, inp.k, inp.v, softmax_scale=wl.softmax_scale, out=o2,
                                              workspace=ws_1, **kw),
            "sage_core": lambda: sa.sage_attn_fwd(prep, out=o2, workspace=ws_a),
        }
        t = time_providers(calls, stream, clk)
        sa.attn_get_device_status()
        F = roofline.attention_flops(B, H, S, D)
        entry = {"config": f"B={B} H={H} S={S} D={D}" + (f", RMSNorm + RoPE {wl.rope_dim} fused" if kw else "")
                           + (", head-major [B,H,S,D] storage" if wl.head_major_storage else "")}
        for prov, rate in (("bf16", roofline.TC_FLOP_PER_CLK_SM["f16"]), ("sage", None),
                           ("sage_core", roofline.sage_flop_per_clk_sm())):
            e = {"ms": t[prov]["ms"], "tflops": F / (t[prov]["ms"] * 1e-3) / 1e12, "sm_mhz": t[prov]["sm_mhz"],
                 "mcycles": t[prov]["mcycles"]}
            if rate is not None and t[prov]["sm_mhz"]:
                e["frac_of_clock_peak"] = e["tflops"] / roofline.clock_peak_tflops(rate, n_sms, t[prov]["sm_mhz"])
            entry[prov] = e
        entry["sage_vs_bf16_cycle_ratio"] = (t["sage"]["mcycles"] / t["bf16"]["mcycles"]
                                             if t["sage"]["mcycles"] and t["bf16"]["mcycles"] else None)
        out[name] = entry
        del inp, o1, o2, ws_1, prep, ws_a, calls
        torch.cuda.empty_cache()
    return out


def run_e2e(args, sa, torch, dev, inp, scale, S_pad, kw, F, world, dist):
    """Same step through the public API from pinned host buffers: every step copies its
    Q, K, V in (H2D), runs both attention paths and copies both outputs out (D2H), all
    inside the timed region.  As a user streaming many steps would, consecutive steps
    overlap on three streams with double-buffered device tensors: step i+1's inputs
    arrive while step i computes, step i-1's outputs leave meanwhile, and a step's BF16
    output leaves while its Sage call runs."""
    B, S, H, D = inp.q.shape
    hq = inp.q.contiguous().cpu().pin_memory()
    hk = inp.k.contiguous().cpu().pin_memory()
    hv = inp.v.contiguous().cpu().pin_memory()
    ho1 = torch.empty((B, S, H, D), dtype=torch.bfloat16).pin_memory()
    ho2 = torch.empty_like(ho1).pin_memory()
    shape = (B, S, H, D)
    din = [[torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(3)] for _ in range(2)]
    dout = [[torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(2)] for _ in range(2)]
    ws_1 = sa.sage_attention_workspace(B, H, S, dev)
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done, bf16_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def run(n):
        for i in range(n):
            bf = i % 2
            dq, dk, dv = din[bf]
            o1, o2 = dout[bf]
            if i >= 2:
                s_in.wait_event(comp_done[bf])        # step i-2 no longer reads these inputs
            with torch.cuda.stream(s_in):
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                in_done[bf].record(s_in)
            comp.wait_event(in_done[bf])
            if i >= 2:
                comp.wait_event(out_done[bf])         # step i-2's outputs have left these buffers
            sa.attn_fwd_bf16(dq, dk, dv, out=o1, softmax_scale=scale, stream=comp)
            bf16_done[bf].record(comp)
            sa.sage_attention(dq, dk, dv, softmax_scale=scale, out=o2, workspace=ws_1, stream=comp, **kw)
            comp_done[bf].record(comp)
            # the BF16 output leaves while the Sage call runs, the Sage output after it
            s_out.wait_event(bf16_done[bf])
            with torch.cuda.stream(s_out):
                ho1.copy_(o1, non_blocking=True)
            s_out.wait_event(comp_done[bf])
            with torch.cuda.stream(s_out):
                ho2.copy_(o2, non_blocking=True)
                out_done[bf].record(s_out)
        comp.wait_event(out_done[(n - 1) % 2])
        if n >= 2:
            comp.wait_event(out_done[(n - 2) % 2])

    # as many steps as the device-side measurement (at most 10), so that the one H2D before
    # the first step and the one D2H after the last are spread the same way
    steps = max(3, min(args.steps, 10))
    run(2)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    s_in.wait_event(t0)
    run(steps)
    t1.record(comp)
    torch.cuda.synchronize()
    sa.attn_get_device_status()
    ms = max_over_ranks(t0.elapsed_time(t1), dist, dev)
    in_bytes = 3 * hq.numel() * 2
    out_bytes = 2 * ho1.numel() * 2
    return {"value": whole_job_tflops(world, 2 * F, steps, ms), "unit": "TFLOPS",
            "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes, "steps": steps,
            "ms_per_step": ms / steps,
            "overlap": "H2D, compute and D2H of consecutive steps on three streams, double-buffered device "
                       "tensors; the first step's H2D and the last step's D2H are inside the timed region"}


# ----------------------------------------------------------------------------- CPU oracle
def _oracle_rows(wl, n, seed):
    import torch
    from workloads import sample_rows
    return sample_rows(wl, n, seed=seed, must_include_tail=False)


def cpu_baseline(wl, seconds: float = 15.0, inputs=None, full_workloads=("tiny", "flux1024"), flux2048_rows=2048):
    """Time the oracle's FP64 attention on sampled query rows of the workload
    (every row a full softmax over all S keys), on all host cores; then the whole
    tiny and FLUX-1024 workloads (every row, all cores) and a bounded row sample of
    FLUX-2048, whose full run (about 7e12 FP64 FLOP) takes minutes."""
    import oracle
    from workloads import make_inputs
    from sage_attention_forward_gb300 import roofline

    if inputs is None:
        inputs = make_inputs(wl)
    q, k, v = inputs.q, inputs.k, inputs.v
    per_row = roofline.attention_flops(1, 1, wl.S, wl.D) / wl.S      # 4*S*D per query row
    t0 = time.perf_counter()
    oracle.attention(q, k, v, wl.softmax_scale, rows=_oracle_rows(wl, 64, 1))
    dt = time.perf_counter() - t0
    n = max(64, int(64 * seconds / max(dt, 1e-3)))
    rows = _oracle_rows(wl, n, 2)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, wl.softmax_scale, rows=rows)
    dt = time.perf_counter() - t0
    out = {"value": n * per_row / dt / 1e12, "unit": "TFLOPS", "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"{n} query rows of {wl.name} (each a full FP64 softmax over S={wl.S} keys), {dt:.1f} s",
           # the whole workload's rows at the sampled rate (not measured: extrapolated)
           "extrapolated_full_s": dt * (wl.B * wl.S * wl.H) / n}
    from workloads import WORKLOADS
    # the whole tiny workload (B=1 H=2 S=512) on one thread
    tw = WORKLOADS["tiny"]
    ti = make_inputs(tw)
    t0 = time.perf_counter()
    oracle.attention(ti.q, ti.k, ti.v, tw.softmax_scale, nthreads=1)
    dt1 = time.perf_counter() - t0
    out["single_thread_tiny"] = {"value": roofline.attention_flops(tw.B, tw.H, tw.S, tw.D) / dt1 / 1e12,
                                 "unit": "TFLOPS", "seconds": dt1, "sample": "all rows of tiny, 1 thread"}
    # full tensors where the oracle finishes in seconds, all host cores
    full = {}
    for name in full_workloads:
        fw = WORKLOADS[name]
        fi = ti if name == "tiny" else make_inputs(fw)
        t0 = time.perf_counter()
        oracle.attention(fi.q, fi.k, fi.v, fw.softmax_scale)
        dtf = time.perf_counter() - t0
        full[name] = {"value": roofline.attention_flops(fw.B, fw.H, fw.S, fw.D) / dtf / 1e12, "unit": "TFLOPS",
                      "seconds": dtf, "cores": oracle.num_threads(),
                      "sample": f"every row of {name} (B={fw.B} H={fw.H} S={fw.S}), measured"}
    # FLUX-2048: a bounded row sample, extrapolated to the full tensor and labelled so
    fw = WORKLOADS["flux2048"]
    fi = make_inputs(fw)
    n2 = flux2048_rows
    t0 = time.perf_counter()
    oracle.attention(fi.q, fi.k, fi.v, fw.softmax_scale, rows=_oracle_rows(fw, n2, 3))
    dt2 = time.perf_counter() - t0
    full["flux2048"] = {"value": n2 * 4 * fw.S * fw.D / dt2 / 1e12, "unit": "TFLOPS", "seconds": dt2,
                        "cores": oracle.num_threads(),
                        "sample": f"{n2} query rows of flux2048 (each over all S={fw.S} keys), measured",
                        "extrapolated_full_s": dt2 * (fw.B * fw.S * fw.H) / n2}
    out["per_workload"] = full
    return out


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on bounded samples of the same workload."""
    import oracle
    from workloads import WORKLOADS, make_inputs
    from sage_attention_forward_gb300 import roofline

    wl = WORKLOADS[args.workload]
    inputs = make_inputs(wl)
    per_row = roofline.attention_flops(1, 1, wl.S, wl.D) / wl.S
    rows_per_step = args.ref_rows
    for i in range(args.warmup):
        oracle.attention(inputs.q, inputs.k, inputs.v, wl.softmax_scale, rows=_oracle_rows(wl, 32, 100 + i))
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.attention(inputs.q, inputs.k, inputs.v, wl.softmax_scale, rows=_oracle_rows(wl, rows_per_step, 200 + i))
    dt = time.perf_counter() - t0
    value = rows_per_step * args.steps * per_row / dt / 1e12
    sample = (f"{rows_per_step} query rows per step of {wl.name} (each a full FP64 softmax over S={wl.S} keys); "
              f"{args.steps} steps in {dt:.1f} s")
    return {"metric": METRIC, "value": value, "unit": "TFLOPS", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, world),
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="wan720p")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-rows", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true")
    args = ap.parse_args()

    rank, world, local_rank = rank_info()
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
