"""Benchmark of the differentiable 3DGS rasterizer hot path on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 3] [--impl reference]

A step is one pass of the whole hot path over one synthetic view: gs_project,
gs_bin_sort, gs_rasterize_fwd, gs_rasterize_bwd (dL/dimage = w, loss = sum w*img)
and gs_project_bwd, on the 1.5M-Gaussian 1297x840 SH-3 scene by default (inputs
resident in HBM; they are larger than L2, 354 MB of parameters plus 354 MB of
gradients per step).  The metric is tile-Gaussian pairs per second (higher is
better); ms_per_step is the matching ms/iter.

Rank 0 prints ONE JSON line.  Under torchrun (N > 1) every rank renders its own
replica of the view (the path does not shard across GPUs: replicas only), the
time is the max over ranks and `value` counts the pairs of all ranks.

--impl reference times the CPU oracle (oracle/, plain C; its unmodified calls on every
host core, over disjoint tiles and Gaussians) on the same workload (a bounded sample of
the larger scenes) and prints the same line with "impl": "reference".

--train-step times a whole training step instead: the same calls with the L1 + SSIM
loss against a synthetic target between forward and backward (gs_loss_l1_ssim), and
the chain rule fused with an Adam step on the raw parameters (gs_project_bwd_adam).
"""

from __future__ import annotations

import argparse
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic_scenes as ss  # noqa: E402

METRIC = "raster fwd+bwd ms/iter & tile-Gaussian pairs/s, 1.5M Gaussians @1297×840"
UNIT = "pairs/s"

# Algorithmic work per contributing pixel-splat pair E, counted from the oracle's scalar
# formulas.  The roofline is the op model of the hot-path table: fp32 ops (an FMA is one
# op, one lane-cycle) against SMs x 128 lanes x the SM clock, and SFU ops (ex2, rcp)
# against SMs x 16 x the clock:
#   forward : dx, dy 2; the quadratic 5 (u1, u2, q); exponent 1; clamp 1; w 1; C 3; T 1 = 14
#             fp32 ops + 1 SFU (ex2)
#   backward: per pixel the quadratic, exponent and clamp 8; 1 - alpha, T_k, w 3; c.G 3;
#             dL/dalpha 2; colour behind 1; the nine outputs and their sums 23 = 40 fp32
#             ops + 2 SFU (ex2, 1 / (1 - alpha))
OPS_FWD_PER_E = 14
OPS_BWD_PER_E = 40
SFU_FWD_PER_E = 1
SFU_BWD_PER_E = 2
FP32_LANES_PER_SM = 128
SFU_LANES_PER_SM = 16
# The same work as flops (an FMA counted as 2; the SFU not counted), reported beside the
# op model: forward 22, backward 48
FLOPS_FWD_PER_E = 22
FLOPS_BWD_PER_E = 48
# The L1 + SSIM loss per pixel: per channel, the window's 11 taps along rows and then
# columns for five moments (x, y, x^2, y^2, xy) and again for the three derivative
# maps of SSIM, 16 x 11 FMA = 352 flops; three channels
LOSS_FLOPS_PER_PIXEL = 3 * 16 * 11 * 2


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--config", type=int, default=3)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--sh-bf16", action="store_true",
                   help="SH coefficients stored as bfloat16 (gs_project_sh16, gs_project_bwd_sh16)")
    p.add_argument("--train-step", action="store_true",
                   help="a whole training step: the hot path with the L1 + SSIM loss against a "
                        "target image between forward and backward, and the chain rule fused "
                        "with an Adam step on the raw parameters (gs_project_bwd_adam)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time (every rank gets it); ms itself outside a process group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, pairs_per_rank: int, ms_per_step: float) -> float:
    """Whole-job pairs/s: every rank renders its own replica of the view (weak scaling)."""
    return world * pairs_per_rank / (ms_per_step * 1e-3)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import differentiable_gaussian_splatting_gb300 as gs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    sc, cam = ss.make_config(args.config)
    w = ss.loss_weights(args.config, cam.height, cam.width)
    H, W = cam.height, cam.width

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    inputs = [to_dev(x) for x in (sc.means, sc.scales, sc.quats, sc.opacities, sc.sh)]
    if args.sh_bf16:
        inputs[4] = inputs[4].to(torch.bfloat16)
    project = gs.gs_project_sh16 if args.sh_bf16 else gs.gs_project
    project_bwd = gs.gs_project_bwd_sh16 if args.sh_bf16 else gs.gs_project_bwd
    dimg = to_dev(w)
    r = gs.Rasterizer(cam, sc.sh_degree, sc.n, device=dev)
    r.forward(*inputs)  # sizes the pair list (one host sync, outside the timed region)
    n_pairs = r.n_pairs
    cap = int(n_pairs * 1.25) + 1024
    r._alloc_pairs(cap)
    r.forward(*inputs)
    torch.cuda.synchronize()
    E = int(r.n_contrib.sum().item())  # contributing pixel-splat pairs
    stream = torch.cuda.current_stream()

    def step(ev=None):
        n = r.n
        if ev:
            ev[0].record(stream)
        project(r.cam, n, r.sh_degree, *inputs, r.splats, r.depths, r.radii, r.tiles_touched)
        if ev:
            ev[1].record(stream)
        gs.gs_bin_sort(r.cam, n, r.splats, r.depths, r.tiles_touched, r.bin_ws, r.sorted_ids,
                       r.capacity, r.tile_ranges, r.lpt_order, r.counts, sync_pairs=False)
        if ev:
            ev[2].record(stream)
        gs.gs_rasterize_fwd(r.cam, n, r.splats, r.sorted_ids, r.tile_ranges, r.lpt_order,
                            r.raster_ws, r.image, r.t_final, r.n_contrib, r.last_idx, r.settings)
        if ev:
            ev[3].record(stream)
        gs.gs_rasterize_bwd(r.cam, n, r.splats, r.sorted_ids, r.tile_ranges, r.lpt_order,
                            r.raster_ws, r.t_final, r.last_idx, dimg, None, r.grad2d, r.touched,
                            r.settings)
        if ev:
            ev[4].record(stream)
        project_bwd(r.cam, n, r.sh_degree, *inputs, r.tiles_touched, r.grad2d, r.touched, *grads)
        if ev:
            ev[5].record(stream)

    K = (sc.sh_degree + 1) ** 2
    grads = [torch.empty((sc.n, 3), device=dev), torch.empty((sc.n, 3), device=dev),
             torch.empty((sc.n, 4), device=dev), torch.empty(sc.n, device=dev),
             torch.empty((sc.n, K, 3), device=dev)]
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = start.elapsed_time(stop)
    # the split by call, from as many further steps with an event between the calls
    # (outside the timed region: the events break the launch overlap at the call
    # boundaries)
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    counts = r.counts.cpu().numpy()
    assert counts[1] == n_pairs and counts[1] <= r.capacity, counts
    calls = ["gs_project", "gs_bin_sort", "gs_rasterize_fwd", "gs_rasterize_bwd", "gs_project_bwd"]
    per_call = {c: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
                for j, c in enumerate(calls)}
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = job_value(world, n_pairs, ms_per_step)

    # roofline of the dominant call (all its work is one kernel launch after small set-up)
    peaks = measured_peaks()
    clocks = clk.summary()
    props = torch.cuda.get_device_properties(dev)
    sm_mhz = clocks["sm_mhz"] or peaks.get("clocks_under_load", {}).get("sm_mhz_median") or 1462.0
    dom = max(per_call, key=per_call.get)
    M = int((r.tiles_touched > 0).sum().item())
    T = int((r.touched != 0).sum().item())
    roof = roofline(dom, per_call[dom], sc, M, n_pairs, E, H, W, peaks,
                    props.multi_processor_count, sm_mhz, T)
    launches = kernel_launches(sc.n, r.capacity, W, H)
    step_roof = step_roofline(ms_per_step, sc, M, n_pairs, E, H, W, peaks,
                              props.multi_processor_count, sm_mhz, T=T)
    roof["per_call"] = per_call_fractions(per_call, sc, M, n_pairs, E, H, W, peaks,
                                          props.multi_processor_count, sm_mhz, T)
    load = imbalance(r.stats(), r.n_tiles)  # the last forward's frame (synchronises)

    e2e = None if args.no_e2e else run_e2e(gs, r, sc, cam, w, dev, args, n_pairs)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # the whole view up to the 1.5M scene, every 16th tile of the larger ones
        cpu = cpu_baseline(sc, cam, w, stride=1 if args.config <= 3 else 16)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(args, sc, W, H, n_pairs,
                                      "replicas" if world > 1 else "single"),
            "contributing_pairs": E,
            "per_call_ms": per_call,
            # the two blend calls alone, the figure the pages quote per stage
            "rast_only_ms": per_call["gs_rasterize_fwd"] + per_call["gs_rasterize_bwd"],
            "roofline": roof,
            "step_roofline": step_roof,
            "imbalance": load,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                       "reasons": clocks["reasons"]},
            "gpu_launches": launches * args.steps,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def roofline(call, ms, sc, M, n_pairs, E, H, W, peaks, n_sm, sm_mhz, T=None):
    """Algorithmic work of one launch / its average duration, against the binding peak.
    M: visible Gaussians; T: Gaussians the backward touched (its chain rule reads the
    parameters and grad2d of those only; M when not given).
    The blend kernels: fp32 ops of the op model against SMs x 128 lanes x the sampled SM
    clock (Tops/s, reported in the TFLOP/s unit), with the SFU fraction and the flop-model
    fraction beside it."""
    if call in ("gs_rasterize_fwd", "gs_rasterize_bwd"):
        fwd = call == "gs_rasterize_fwd"
        ops_e = OPS_FWD_PER_E if fwd else OPS_BWD_PER_E
        flops_e = FLOPS_FWD_PER_E if fwd else FLOPS_BWD_PER_E
        ops = ops_e * E
        sfu = (SFU_FWD_PER_E if fwd else SFU_BWD_PER_E) * E
        flops = flops_e * E
        hz = n_sm * sm_mhz * 1e6
        peak = FP32_LANES_PER_SM * hz / 1e12
        achieved = ops / (ms * 1e-3) / 1e12
        return {"kernel": call, "bound": "alu", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": profiled_traffic(call),
                "peak_source": f"{n_sm} SMs x {FP32_LANES_PER_SM} fp32 lanes x {sm_mhz:.0f} MHz "
                               f"(sampled), one op per lane per cycle",
                "work": f"{ops_e} fp32 ops (an FMA is one op) x {E} contributing pairs",
                "sfu_frac": sfu / (ms * 1e-3) / (SFU_LANES_PER_SM * hz),
                "flop_model": {"frac": flops / (ms * 1e-3) / (2 * FP32_LANES_PER_SM * hz),
                               "work": f"{flops_e} flops (an FMA is two) x {E} pairs, "
                                       f"against 2 x the fp32 lanes"}}
    if call == "gs_loss_l1_ssim":
        flops = LOSS_FLOPS_PER_PIXEL * H * W
        peak = 2.0 * FP32_LANES_PER_SM * n_sm * sm_mhz * 1e6 / 1e12
        achieved = flops / (ms * 1e-3) / 1e12
        return {"kernel": call, "bound": "alu", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": profiled_traffic(call),
                "peak_source": f"{n_sm} SMs x {FP32_LANES_PER_SM} fp32 lanes x 2 x {sm_mhz:.0f} MHz (sampled)",
                "work": f"{LOSS_FLOPS_PER_PIXEL} flops x {H * W} pixels"}
    N, G = sc.n, 44 + 12 * (sc.sh_degree + 1) ** 2  # G: parameter bytes per Gaussian
    T = M if T is None else T
    if call == "gs_project_bwd_adam":
        # grad2d of the touched, the two flags, parameters and both moments read and
        # written, the activated scales and opacities written
        byts = 36 * T + 5 * N + 6 * G * N + 16 * N
        achieved = byts / (ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        return {"kernel": call, "bound": "hbm", "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "traffic": profiled_traffic(call),
                "peak_source": f"{peaks['source']} copy bandwidth"}
    if call == "gs_project":
        # geometry of every Gaussian, SH of the visible; every row of the outputs
        # (record, depth, radii, tile count: 64 B) is written, culled rows as zeros
        byts = 44 * N + (G - 44) * M + 64 * N
    elif call == "gs_project_bwd":
        # grad2d and parameters of the touched, every gradient row written, the two flags
        byts = 36 * T + G * T + G * N + 5 * N
    else:  # gs_bin_sort
        byts = 8 * M * 8 + 8 * n_pairs * 5
    achieved = byts / (ms * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    return {"kernel": call, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": profiled_traffic(call),
            "peak_source": f"{peaks['source']} copy bandwidth"}


def imbalance(stats: dict, n_tiles: int) -> dict:
    """Per-frame tile load (Ryu & Yoo, Sec. 3.1): the heaviest tile against the mean, the
    lightest non-empty tile and the per-CTA share N_total / K; the split policy's choice
    (Eq. 6) and what the forward did with the 256-splat batches of split tiles."""
    K = max(int(stats["resident_ctas"]), 1)
    tot, nmax = int(stats["n_total"]), int(stats["n_max"])
    nz, nmin = int(stats["nonempty_tiles"]), int(stats["n_min_nonempty"])
    return {"tiles": n_tiles, "nonempty_tiles": nz, "n_max": nmax,
            "n_mean": tot / max(n_tiles, 1), "n_mean_nonempty": tot / max(nz, 1),
            "n_min_nonempty": nmin, "max_over_min": nmax / max(nmin, 1),
            "max_over_share": nmax / (tot / K) if tot else 0.0, "resident_ctas": K,
            "h": int(stats["h"]), "k": int(stats["k"]),
            "batches": {k: int(stats["batches_" + k]) for k in
                        ("tiles", "chunks", "skipped_on_flag", "skipped_done", "discarded")}}


def per_call_fractions(per_call, sc, M, n_pairs, E, H, W, peaks, n_sm, sm_mhz, T=None) -> dict:
    """Each call's roofline fraction (bound and frac) from its own event time."""
    out = {}
    for call, ms in per_call.items():
        r = roofline(call, ms, sc, M, n_pairs, E, H, W, peaks, n_sm, sm_mhz, T)
        out[call] = {"bound": r["bound"], "frac": r["frac"], "ms": ms}
    return out


# The kernel each single-kernel call runs, its sources, and its ncu summary.
PROFILED = {
    "gs_rasterize_fwd": ("raster_fwd_kernel", ["gs_raster.cu", "gs_device.cuh", "gs_internal.h"]),
    "gs_rasterize_bwd": ("raster_bwd_kernel", ["gs_raster.cu", "gs_device.cuh", "gs_internal.h"]),
    "gs_project": ("project_kernel", ["gs_project.cu", "gs_device.cuh", "gs_internal.h"]),
    "gs_project_bwd": ("project_bwd_kernel", ["gs_project.cu", "gs_device.cuh", "gs_internal.h"]),
    "gs_loss_l1_ssim": ("loss_ssim_kernel", ["gs_loss.cu", "gs_device.cuh", "gs_internal.h"]),
    "gs_project_bwd_adam": ("project_bwd_adam", ["gs_project.cu", "gs_device.cuh",
                                                 "gs_internal.h", "gs_project_variants.h"]),
}


def sources_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "differentiable_gaussian_splatting_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(call, workload="scene-1.5M-1297x840"):
    """DRAM bytes (read + write) of one launch, from the committed ncu summary of the call's
    kernel; None when there is none or the kernel's sources changed since it was taken."""
    if call not in PROFILED:
        return None
    kernel, files = PROFILED[call]
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            for key in ("traffic_bytes_per_launch", "sources_sha256"):
                if line.startswith(f"- {key}:"):
                    fields[key] = line.split(":", 1)[1].split()[0].strip("`")
    if fields.get("sources_sha256") != sources_digest(files):
        return None
    return int(fields["traffic_bytes_per_launch"]) if "traffic_bytes_per_launch" in fields else None


def step_roofline(ms, sc, M, I, E, H, W, peaks, n_sm, sm_mhz, train=False, T=None):
    """Whole-step roofline: per phase the largest of bytes / HBM, fp32 flops / fp32 peak and
    SFU ops / SFU peak, summed over the phases; frac = that time / the measured step.
    train: the training step (loss phase; Adam on parameters and moments in place of the
    gradient rows)."""
    N, P = sc.n, H * W
    T = M if T is None else T  # Gaussians the backward touched
    G = 44 + 12 * (sc.sh_degree + 1) ** 2  # parameter bytes per Gaussian
    hbm = float(peaks["hbm_gbs"]) * 1e9
    fp32 = FP32_LANES_PER_SM * n_sm * sm_mhz * 1e6  # fp32 ops (an FMA is one)
    sfu = SFU_LANES_PER_SM * n_sm * sm_mhz * 1e6
    phases = {
        # 44 B of geometry per Gaussian, SH only for the visible, 64 B of outputs per
        # Gaussian (culled rows are written as zeros)
        "project": (44 * N + (G - 44) * M + 64 * N, 0, 0),
        # depth sort of the M visible (8 B, 4 passes, read + write) and the pair list
        # (emitted once, then 2 passes read + write)
        "bin_sort": (8 * M * 8 + 8 * I * 5, 0, 0),
        "forward": (48 * I + 24 * P, OPS_FWD_PER_E * E, SFU_FWD_PER_E * E),
        # raster backward and the chain rule: records, pixel state and dL/dimage, grad2d,
        # parameters of the touched, every gradient row written
        "backward": (48 * I + 36 * P + 36 * T + G * T + G * N, OPS_BWD_PER_E * E,
                     SFU_BWD_PER_E * E),
    }
    if train:
        phases["loss"] = (36 * P, LOSS_FLOPS_PER_PIXEL * P // 2, 0)  # its FMAs
        phases["backward"] = (48 * I + 36 * P + 36 * T + 5 * N + 6 * G * N + 16 * N,
                              OPS_BWD_PER_E * E, SFU_BWD_PER_E * E)
    out, total = {}, 0.0
    for k, (b, f, x) in phases.items():
        t = max(b / hbm, f / fp32, x / sfu) * 1e3
        out[k] = t
        total += t
    return {"ms": total, "frac": total / ms, "phases_ms": out,
            "model": "per phase max(bytes/HBM, fp32 ops/(SMs x 128 x clock), SFU ops/(SMs x 16 "
                     "x clock)), summed; an FMA is one op"}


def kernel_launches(n, capacity, W, H) -> int:
    """Kernels one step launches."""
    if capacity >= 8 << 20:
        # long lists, two-stage radix sort: compaction count / scan / write, 4 depth passes,
        # pair count / scan / offsets, emission, 1-3 tile passes, ranges, empty ranges, 2 LPT
        tiles = ((W + 15) // 16) * ((H + 15) // 16)
        tile_passes = (max(1, (tiles - 1).bit_length()) + 7) // 8
        bin_sort = 3 + 4 + 3 + 1 + tile_passes + 2 + 2
    else:
        # buckets: counter reset, span pass, scan, scatter, two slice sorts, two LPT kernels,
        # the long-slice plan and chunk sort, and one merge round per doubling up to min(n, capacity)
        rounds, w = 0, 4096
        while w < min(n, capacity):
            rounds, w = rounds + 1, 2 * w
        bin_sort = 1 + 1 + 1 + 1 + 2 + 2 + 2 + rounds
    # project 1, policy + forward 2, accumulator reset + backward 2, project backward 1
    return 1 + bin_sort + 2 + 2 + 1


def run_e2e(gs, r, sc, cam, w, dev, args, n_pairs):
    """Same metric through the public API with host buffers.  Every step copies its
    inputs (parameters and dL/dimage) from pinned host memory to the device and reads
    its result, the rendered image, back to pinned host memory; the parameter gradients
    stay on the device, where an optimizer step would consume them.  The input copy of
    step k + 1 runs on a second stream into the other of two device buffers while step
    k computes, as a training loop that prefetches its next view would."""
    import torch

    host_in = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
               for a in (sc.means, sc.scales, sc.quats, sc.opacities, sc.sh, w)]
    if args.sh_bf16:
        host_in[4] = host_in[4].to(torch.bfloat16).pin_memory()
    dev_in = [[torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host_in] for _ in range(2)]
    host_img = torch.empty((cam.height, cam.width, 3), dtype=torch.float32).pin_memory()
    bi = sum(h.numel() * h.element_size() for h in host_in)
    bo = host_img.numel() * host_img.element_size()
    compute = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def upload(k):
        b = k % 2
        with torch.cuda.stream(copy):
            copy.wait_event(consumed[b])  # step k - 2 is done with this buffer
            for h, d in zip(host_in, dev_in[b]):
                d.copy_(h, non_blocking=True)
            copied[b].record(copy)

    def step(k, last):
        b = k % 2
        if k + 1 < last:
            upload(k + 1)
        compute.wait_event(copied[b])
        r.forward(*dev_in[b][:5], sync_pairs=False)
        r.backward(dev_in[b][5])
        consumed[b].record(compute)
        host_img.copy_(r.image, non_blocking=True)

    for b in range(2):
        consumed[b].record(compute)
    nw = max(3, args.warmup)
    upload(0)
    for k in range(nw):
        step(k, nw)
    torch.cuda.synchronize()
    # the timed region holds exactly the timed steps' copies (the first is not overlapped)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(compute)
    copy.wait_event(s)
    upload(nw)
    for k in range(nw, nw + args.steps):
        step(k, nw + args.steps)
    e.record(compute)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.steps
    return {"value": n_pairs / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "overlap": "input copy of the next step on a second stream"}


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
L2_BYTES = 129e6  # the GB300's L2


def l2_note(sc, second: str, factor: int) -> str:
    """How the timed steps avoid a warm L2: whether the parameters and the arrays of the
    same size that each step writes (gradients, or the two Adam moments) exceed it."""
    mb = sum(a.nbytes for a in (sc.means, sc.scales, sc.quats, sc.opacities, sc.sh)) / 1e6
    fits = "larger than" if (1 + factor) * mb * 1e6 > L2_BYTES else "smaller than"
    return f"inputs {fits} L2 ({mb:.3g} MB parameters + {factor * mb:.3g} MB {second})"


def workload_config(args, sc, W, H, n_pairs, parallelism):
    """The workload both arms time: scene, image, SH storage and the view's tile-Gaussian
    pair count (an integer both sides reproduce bit for bit)."""
    return {"workload": ss.CONFIG_NAMES[args.config], "gaussians": sc.n, "image": f"{W}x{H}",
            "sh_degree": sc.sh_degree, "tile_pairs": int(n_pairs),
            "sh_storage": "bf16" if args.sh_bf16 else "f32", "parallelism": parallelism,
            "l2": l2_note(sc, "gradients", 1)}


def _row_chunks(n: int, parts: int):
    step = max(1, -(-n // max(1, parts)))
    return [np.arange(i, min(n, i + step)) for i in range(0, n, step)]


def _threads(fn, items, workers):
    from concurrent.futures import ThreadPoolExecutor

    # the oracle's C calls release the GIL (ctypes): the items run on separate cores
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, items))


def oracle_sample_step(sc, cam, w, tile_stride: int, workers: int = 1):
    """One bounded oracle step: projection and binning of the whole view, then the
    forward and backward blend of every tile_stride-th tile (in LPT order, so the
    sample spans heavy and light tiles), then the chain rule.  With workers > 1 the
    unmodified oracle calls run on that many host threads: the projection and the chain
    rule over disjoint ranges of Gaussians, the blends over disjoint sets of tiles (the
    oracle's tile_parts), per-Gaussian float64 sums added at the end.  Returns (pairs
    processed, seconds, pairs of the whole view)."""
    import oracle

    t0 = time.perf_counter()
    if workers > 1:
        chunks = _row_chunks(sc.n, 4 * workers)
        ps = _threads(lambda rows: oracle.project(sc.subset(rows), cam), chunks, workers)
        proj = oracle.Projection(*(np.concatenate([getattr(p, f) for p in ps])
                                   for f in ("splat", "rgb", "radii", "tiles_touched")))
    else:
        proj = oracle.project(sc, cam)
    ntx, nty = oracle.n_tiles(cam)
    if tile_stride == 1:
        b = oracle.bin_sort(cam, proj)
        sel = np.ones(ntx * nty, np.uint8)
        counts = b
    else:
        counts = oracle.bin_sort(cam, proj, np.zeros(ntx * nty, np.uint8))
        sel = np.zeros(ntx * nty, np.uint8)
        sel[counts.lpt_order[::tile_stride]] = 1
        b = oracle.bin_sort(cam, proj, sel)
    # the method's gradient only (the error-bound sums the parity tests use are not formed)
    if workers > 1:
        oracle.blend_parallel(cam, proj, b, workers=workers)
        g2 = oracle.blend_bwd_parallel(cam, proj, b, w, workers=workers, bounds=False).grad2d

        def chain(rows):
            p = oracle.Projection(proj.splat[rows], proj.rgb[rows], proj.radii[rows],
                                  proj.tiles_touched[rows])
            return oracle.project_bwd(sc.subset(rows), cam, p, g2[rows])

        _threads(chain, _row_chunks(sc.n, 4 * workers), workers)
    else:
        oracle.blend(cam, proj, b)
        g2 = oracle.blend_bwd_bounds(cam, proj, b, w, bounds=False).grad2d
        oracle.project_bwd(sc, cam, proj, g2)
    dt = time.perf_counter() - t0
    return int(b.counts[sel.astype(bool)].sum()), dt, int(counts.counts.sum())


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(sc, cam, w, stride: int = 1):
    """The oracle over the whole view, on every host core (the headline) and on one."""
    cores = host_cores()
    what = "every tile" if stride == 1 else f"every {stride}th tile in LPT order"
    if stride > 1:
        # the sampled step is short beside the first touch of the large scenes' arrays:
        # one untimed pass first, so that neither variant pays it
        oracle_sample_step(sc, cam, w, stride, workers=cores)
    pairs1, dt1, _ = oracle_sample_step(sc, cam, w, stride, workers=1)
    pairs, dt, _ = oracle_sample_step(sc, cam, w, stride, workers=cores)
    return {"value": pairs / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"one view: all projections and tile counts, forward + backward of "
                      f"{what} ({pairs} pairs) and the chain rule, the unmodified oracle calls "
                      f"on {cores} host threads (disjoint tiles / Gaussians), {dt:.2f} s",
            "single_core": {"value": pairs1 / dt1, "unit": UNIT, "cores": 1,
                            "sample": f"the same view on one thread, {dt1:.1f} s"}}


# Adam settings of the training step: the learning rates 3DGS trains with (means, scales,
# rotations, opacities, SH band 0, SH bands 1-3), beta1 0.9, beta2 0.999, eps 1e-15
TRAIN_LR = dict(lr_means=1.6e-4, lr_scales=5e-3, lr_quats=1e-3, lr_opacities=5e-2,
                lr_sh0=2.5e-3, lr_shN=1.25e-4)


def run_train(args):
    """A whole training step per timed step: gs_project on the activated parameters,
    gs_bin_sort, gs_rasterize_fwd, gs_loss_l1_ssim against a synthetic target image,
    gs_rasterize_bwd of the loss's gradient and gs_project_bwd_adam, which steps the raw
    parameters and both moments in place and writes the activated scales and opacities
    the next step's projection reads."""
    import torch
    import torch.distributed as dist

    import differentiable_gaussian_splatting_gb300 as gs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    sc, cam = ss.make_config(args.config)
    H, W = cam.height, cam.width
    _, target = ss.image_pair(np.random.default_rng(200 + args.config), H, W)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)

    log_s = np.log(sc.scales.astype(np.float64))
    o = sc.opacities.astype(np.float64).reshape(-1)
    raw = [to_dev(sc.means), to_dev(log_s), to_dev(sc.quats), to_dev(np.log(o / (1 - o))),
           to_dev(sc.sh)]
    act_s, act_o = to_dev(sc.scales), to_dev(o)
    mom_m = [torch.zeros_like(t) for t in raw]
    mom_v = [torch.zeros_like(t) for t in raw]
    tgt = to_dev(target)
    dimg = torch.empty_like(tgt)
    loss_out = torch.zeros(4, dtype=torch.float32, device=dev)
    loss_ws = torch.empty(gs.gs_loss_workspace_bytes(W, H), dtype=torch.uint8, device=dev)
    adam = gs.AdamSettings(**TRAIN_LR, beta1=0.9, beta2=0.999, eps=1e-15, step=1)

    r = gs.Rasterizer(cam, sc.sh_degree, sc.n, device=dev)
    r.forward(raw[0], act_s, raw[2], act_o, raw[4])  # sizes the pair list (one host sync)
    n_pairs = r.n_pairs
    r._alloc_pairs(int(n_pairs * 1.25) + 1024)
    stream = torch.cuda.current_stream()
    t_step = [0]

    def step(ev=None):
        n = r.n
        t_step[0] += 1
        adam.step = t_step[0]
        marks = iter(ev) if ev else None

        def mark():
            if marks:
                next(marks).record(stream)

        mark()
        gs.gs_project(r.cam, n, r.sh_degree, raw[0], act_s, raw[2], act_o, raw[4], r.splats,
                      r.depths, r.radii, r.tiles_touched)
        mark()
        gs.gs_bin_sort(r.cam, n, r.splats, r.depths, r.tiles_touched, r.bin_ws, r.sorted_ids,
                       r.capacity, r.tile_ranges, r.lpt_order, r.counts, sync_pairs=False)
        mark()
        gs.gs_rasterize_fwd(r.cam, n, r.splats, r.sorted_ids, r.tile_ranges, r.lpt_order,
                            r.raster_ws, r.image, r.t_final, r.n_contrib, r.last_idx, r.settings)
        mark()
        gs.gs_loss_l1_ssim(W, H, r.image, tgt, dimg, loss_out, loss_ws)
        mark()
        gs.gs_rasterize_bwd(r.cam, n, r.splats, r.sorted_ids, r.tile_ranges, r.lpt_order,
                            r.raster_ws, r.t_final, r.last_idx, dimg, None, r.grad2d, r.touched,
                            r.settings)
        mark()
        gs.gs_project_bwd_adam(r.cam, n, r.sh_degree, *raw, r.tiles_touched, r.grad2d,
                               r.touched, mom_m, mom_v, adam, scales_out=act_s,
                               opacities_out=act_o)
        mark()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    loss0 = float(loss_out[0].item())
    pairs0 = int(r.counts[1].item())
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = start.elapsed_time(stop)
    loss1 = float(loss_out[0].item())
    counts = r.counts.cpu().numpy()
    if counts[1] > r.capacity:
        raise RuntimeError(f"pair list outgrew its capacity during training: {counts[1]}")
    pairs1 = int(counts[1])
    calls = ["gs_project", "gs_bin_sort", "gs_rasterize_fwd", "gs_loss_l1_ssim",
             "gs_rasterize_bwd", "gs_project_bwd_adam"]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
           for _ in range(args.steps)]
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    per_call = {c: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
                for j, c in enumerate(calls)}
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps
    # pairs of the timed steps: the count moves a little as the parameters train
    pairs = 0.5 * (pairs0 + pairs1)
    value = world * pairs / (ms_per_step * 1e-3)
    peaks = measured_peaks()
    clocks = clk.summary()
    props = torch.cuda.get_device_properties(dev)
    sm_mhz = clocks["sm_mhz"] or peaks.get("clocks_under_load", {}).get("sm_mhz_median") or 1462.0
    dom = max(per_call, key=per_call.get)
    M = int((r.tiles_touched > 0).sum().item())
    T = int((r.touched != 0).sum().item())
    E = int(r.n_contrib.sum().item())
    roof = roofline(dom, per_call[dom], sc, M, pairs1, E, H, W, peaks,
                    props.multi_processor_count, sm_mhz, T)
    step_roof = step_roofline(ms_per_step, sc, M, pairs1, E, H, W, peaks,
                              props.multi_processor_count, sm_mhz, train=True, T=T)
    roof["per_call"] = per_call_fractions(per_call, sc, M, pairs1, E, H, W, peaks,
                                          props.multi_processor_count, sm_mhz, T)
    launches = kernel_launches(sc.n, r.capacity, W, H) + 2  # the loss: tiles + final sum
    if rank == 0:
        print(json.dumps({
            "metric": "training step (hot path + L1/SSIM loss + fused chain rule and Adam), "
                      "tile-Gaussian pairs/s",
            "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": ss.CONFIG_NAMES[args.config], "gaussians": sc.n,
                       "image": f"{W}x{H}", "sh_degree": sc.sh_degree,
                       "tile_pairs": [pairs0, pairs1], "contributing_pairs": E,
                       "loss": [loss0, loss1], "adam": TRAIN_LR,
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": l2_note(sc, "moments", 2)},
            "per_call_ms": per_call,
            "roofline": roof,
            "step_roofline": step_roof,
            "cpu_baseline": None,
            "e2e": None,
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                       "reasons": clocks["reasons"]},
            "gpu_launches": launches * args.steps,
        }))
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    sc, cam = ss.make_config(args.config)
    if args.sh_bf16:
        # the oracle reads the same coefficients the bfloat16 path stores, widened to float
        import dataclasses

        import torch
        sh = torch.from_numpy(np.ascontiguousarray(sc.sh, np.float32))
        sc = dataclasses.replace(sc, sh=sh.to(torch.bfloat16).float().numpy())
    w = ss.loss_weights(args.config, cam.height, cam.width)
    # the whole view up to the 1.5M scene; every 4th tile (in LPT order) of the larger ones
    stride = 1 if args.config <= 3 else 4
    cores = host_cores()
    for _ in range(args.warmup):
        oracle_sample_step(sc, cam, w, stride, workers=cores)
    tot_pairs, tot_s = 0, 0.0
    for _ in range(args.steps):
        p, dt, view_pairs = oracle_sample_step(sc, cam, w, stride, workers=cores)
        tot_pairs += p
        tot_s += dt
    value = tot_pairs / tot_s
    what = "every tile" if stride == 1 else f"every {stride}th tile in LPT order"
    sample = (f"each step: all projections and tile counts, forward + backward of {what} "
              f"({tot_pairs // args.steps} pairs) and the chain rule, on {cores} host threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(args, sc, cam.width, cam.height, view_pairs, "single"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    elif a.train_step:
        run_train(a)
    else:
        run_gpu(a)
