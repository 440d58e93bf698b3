"""Benchmark of the update phase (SS-HSDP: f0 momentum, fragment gather,
batched Newton-Schulz, scatter + f2, MXFP8 requant) on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one update phase over the whole workload through
muon_update_units with the fused stages (f0 + gather in one pass, batched
Newton-Schulz, f2 + MXFP8 requant in one pass), inputs resident in HBM; an
unfused stage-by-stage pass afterwards gives the per-kernel HBM table.  Prints one JSON line on rank 0.  Under
torchrun each rank runs an independent replica on its own GPU (the path has
no cross-GPU exchange on one box): whole-job params/s = ranks * P * K / max
over ranks of the timed region.

--impl reference times the CPU oracle (plain NumPy) on the host cores on a
bounded sample of the same workload, scaled to params/s.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "update-phase params/sec; NS TFLOP/s and requant GB/s as % of GB300 peak"
UNIT = "params/s"


def ns_flops(cfg, steps: int) -> float:
    """Algorithmic Newton-Schulz FLOP of one update: per unit and iteration
    4 m^2 n (X X^T and B X) + 2 m^3 (A A), m = min, n = max of its shape."""
    tot = 0.0
    for u in cfg.units:
        m, n = min(u.rows, u.cols), max(u.rows, u.cols)
        tot += steps * (4.0 * m * m * n + 2.0 * m ** 3)
    return tot


def ns_executed_flops(cfg, steps: int) -> float:
    """Tensor-core FLOP the kernels actually issue per update, by the kernel
    a shape class runs on (Gram size mp = m rounded up to 128):
    - single-CTA GEMMs (mp = 128, or mp not a multiple of 256): 128 x BN tiles
      (BN = 256 once mp >= 256) on or above the diagonal for X X^T and
      bA + cAA, 128 x BN3 tiles of B X, K padded to 64;
    - CTA pairs (mp a multiple of 256): 256 x 256 tiles, the upper triangle
      for the symmetric products and the full grid of B X."""
    classes = {}
    for u in cfg.units:
        key = (min(u.rows, u.cols), max(u.rows, u.cols))
        classes[key] = classes.get(key, 0) + 1
    tot = 0.0
    for (m, n), cnt in classes.items():
        mp, np_ = -(-m // 128) * 128, -(-n // 64) * 64
        if mp <= 128 or mp % 256:
            bn = 256 if mp >= 256 else 128
            bn3 = 256 if np_ >= 256 else 128
            sym = sum(1 for tm in range(mp // 128) for tn in range(-(-mp // bn)) if tn * bn + bn - 1 >= tm * 128)
            per_it = (sym * 2.0 * 128 * bn * (np_ + mp) +
                      (mp // 128) * -(-np_ // bn3) * 2.0 * 128 * bn3 * mp)
        else:
            t2 = -(-mp // 256)
            tri = t2 * (t2 + 1) // 2
            per_it = tri * 2.0 * 256 * 256 * (np_ + mp) + t2 * -(-np_ // 256) * 2.0 * 256 * 256 * mp
        tot += cnt * steps * per_it
    return tot


def straddling_elems(cfg, plan_info) -> int:
    return int(plan_info.staging_elems)


# DRAM bytes (read + write) of one Newton-Schulz stage of the Video-DiT x8
# workload with f2 and G folded into its last products (the timed update's
# second call: the one-launch head-class kernel and 15 CTA-pair GEMMs): an ncu
# launch list of dram__bytes_read.sum + dram__bytes_write.sum over the timed
# update of one Video-DiT layer (18.84 GB), scaled by the units processed (x8);
# valid only for the kernel source it was measured on (sha256 prefix of hm_ns.cu).
NS_STAGE_TRAFFIC = {"workload": "video_dit", "bytes": 1.507e+11, "hm_ns_sha256": "ac4f979a729147d1",
                    "how": "one Video-DiT layer measured, x8 by units"}


def ns_stage_traffic(cfg):
    import hashlib
    src = os.path.join(ROOT, "head_muon_mxfp8_gb300", "csrc", "hm_ns.cu")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if cfg.name != NS_STAGE_TRAFFIC["workload"] or sha != NS_STAGE_TRAFFIC["hm_ns_sha256"]:
        return None
    return NS_STAGE_TRAFFIC["bytes"]


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of one float over all ranks (a scalar, not data)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, numel: int, steps: int, ms: float) -> float:
    """Whole-job parameters per second: every rank updates numel parameters per
    step; the job takes the slowest rank's time."""
    return world * numel * steps / (ms / 1e3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in self.rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in self.rows for k in range(4) if r[5 + k].lower().startswith("active")})
        pw = [num(r[3]) for r in self.rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows), "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------------------
# CPU oracle on a bounded sample (cpu_baseline and --impl reference)
# ----------------------------------------------------------------------------
def oracle_sample_step(cfg, rng_seed: int = 0):
    """One pass of the oracle over a bounded sample of the workload; returns
    (seconds, extrapolated seconds for the whole workload, description).

    Sample: every stage on a 262,144-element slice (f0, f2, MXFP8 requant;
    gather is a copy), Newton-Schulz in full for one unit of the smallest
    shape class, and for every larger class one product of each of the three
    kinds on an m x m slice; the class's time is extrapolated by its
    algorithmic FLOP."""
    from oracle import muon as OM
    from oracle import mxfp8 as OX
    rng = np.random.default_rng(rng_seed)
    t_start = time.perf_counter()
    n_el = 1 << 18
    w = (rng.standard_normal(n_el) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n_el) * 1e-3).astype(np.float32)
    m = np.zeros(n_el, np.float32)
    t0 = time.perf_counter()
    m, u = OM.momentum(m, g, 0.95)
    v = OM.bf16_bits_to_f32(u)
    w = OM.main_weight_update(w, v, 0.02, 1.0)
    OX.requant_list(w, [(0, n_el // 4096, 4096)])
    t_elem = (time.perf_counter() - t0) / n_el
    h = cfg.muon
    classes = {}
    for un in cfg.units:
        key = (min(un.rows, un.cols), max(un.rows, un.cols))
        classes[key] = classes.get(key, 0) + 1
    t_ns = 0.0
    for (mm, nn), cnt in sorted(classes.items()):
        if mm <= 256:
            x = rng.standard_normal((mm, nn)).astype(np.float32) * np.float32(1e-3)
            t0 = time.perf_counter()
            OM.newton_schulz(x, h.ns_steps, h.ns_a, h.ns_b, h.ns_c, h.eps)
            t_ns += (time.perf_counter() - t0) * cnt
        else:
            x = rng.standard_normal((mm, mm)).astype(np.float32) * np.float32(1e-3)
            t0 = time.perf_counter()
            A = x @ x.T
            B = np.float32(h.ns_b) * A + np.float32(h.ns_c) * (A @ A)
            _ = np.float32(h.ns_a) * x + B @ x
            dt = time.perf_counter() - t0
            sample_flops = 6.0 * mm ** 3
            class_flops = cnt * h.ns_steps * (4.0 * mm * mm * nn + 2.0 * mm ** 3)
            t_ns += dt * class_flops / sample_flops
    total = t_elem * cfg.numel + t_ns
    desc = ("oracle f0+f2+MXFP8 on 262144 elements, full Newton-Schulz on one unit per small class, one "
            "X X^T / A A / B X triple on an m x m slice per large class; extrapolated by elements and FLOP")
    return time.perf_counter() - t_start, total, desc


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample_step(cfg)
    times, totals = [], []
    desc = ""
    t0 = time.perf_counter()
    for k in range(args.steps):
        dt, total, desc = oracle_sample_step(cfg, rng_seed=k)
        times.append(dt)
        totals.append(total)
    wall = time.perf_counter() - t0
    per_step = statistics.median(totals)
    value = cfg.numel / per_step
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": cfg.name, "params": cfg.numel, "units": len(cfg.units)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": desc, "sample_wall_s": wall},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def run_ours(args, cfg):
    import torch

    from head_muon_mxfp8_gb300 import abi
    from head_muon_mxfp8_gb300.session import MuonSession, muon_hparams

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    abi.lib()

    sess = MuonSession.from_config(cfg, device=dev, canaries=False)
    data = workloads.generate_device(cfg, dev, seed=cfg.seed + rank)
    sess.load("w", data["w"])
    sess.load("g", data["g"])
    sess.m.zero_()
    del data
    hp = muon_hparams(cfg.muon)
    stream = torch.cuda.Stream(device=dev)
    info = sess.info
    front = abi.HM_STAGE_F0 | abi.HM_STAGE_GATHER | abi.HM_STAGE_FUSED
    back = abi.HM_STAGE_F2 | abi.HM_STAGE_REQUANT | abi.HM_STAGE_FUSED
    # HM_STAGE_STEP as two calls: f0 (u of straddling units into their staging
    # only), then Newton-Schulz with f2 and G in its last products (v skipped)
    front_s = front | abi.HM_STAGE_SCRATCH
    ns_back = abi.HM_STAGE_STEP & ~(abi.HM_STAGE_F0 | abi.HM_STAGE_GATHER)

    def step(ev=None):
        """One update phase, fused: f0 with the gather folded in, then
        batched Newton-Schulz whose last product applies f2 and the MXFP8
        requant itself (HM_STAGE_STEP: v never stored)."""
        if ev is None:
            sess.run(hp, abi.HM_STAGE_STEP, stream)
            return
        ev[0].record(stream)
        sess.run(hp, front_s, stream)
        ev[1].record(stream)
        sess.run(hp, ns_back, stream)
        ev[2].record(stream)

    def step_through_v(ev):
        """The same update with v stored by the last product and read back by
        one f2 + G pass (HM_STAGE_ALL_FUSED, as three calls)."""
        ev[0].record(stream)
        sess.run(hp, front, stream)
        ev[1].record(stream)
        sess.run(hp, abi.HM_STAGE_NS, stream)
        ev[2].record(stream)
        sess.run(hp, back, stream)
        ev[3].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    if abi.hm_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    launches0 = abi.hm_kernel_launches()
    for k in range(args.steps):
        step(evs[k])
    launches = abi.hm_kernel_launches() - launches0
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks.stop()
    ms = t_begin.elapsed_time(t_end)
    stage_ms = {"f0_gather": statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
                "ns_f2_requant": statistics.mean(e[1].elapsed_time(e[2]) for e in evs)}
    if abi.hm_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")

    # the same update through v (a separate, shorter timed loop): Newton-Schulz
    # alone and the f2 + G pass get their own events
    n_v = min(3, args.steps)
    vev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_v)]
    with torch.cuda.stream(stream):
        for e in vev:
            step_through_v(e)
    torch.cuda.synchronize()
    through_v_ms = {"f0_gather": statistics.mean(e[0].elapsed_time(e[1]) for e in vev),
                    "ns": statistics.mean(e[1].elapsed_time(e[2]) for e in vev),
                    "f2_requant": statistics.mean(e[2].elapsed_time(e[3]) for e in vev)}
    through_v_ms["step"] = sum(through_v_ms.values())

    # per-kernel breakdown: the unfused stages, one call each, CUDA events between
    # them (a separate, shorter timed loop after the headline one)
    n_unfused = min(3, args.steps)
    uev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_unfused)]
    with torch.cuda.stream(stream):
        for e in uev:
            e[0].record(stream)
            for j, st_flag in enumerate((abi.HM_STAGE_F0, abi.HM_STAGE_GATHER, abi.HM_STAGE_NS, abi.HM_STAGE_F2,
                                         abi.HM_STAGE_REQUANT)):
                sess.run(hp, st_flag, stream)
                e[j + 1].record(stream)
    torch.cuda.synchronize()
    unfused_ms = {name: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in uev)
                  for j, name in enumerate(("f0", "gather", "ns", "f2", "requant"))}

    ms = max_over_ranks(ms, dist, dev)
    ms_per_step = ms / args.steps
    value = whole_job_rate(world, cfg.numel, args.steps, ms)

    # ---- optional: the same fused step captured once in a CUDA graph and
    # replayed (no per-kernel launch cost; matters for small workloads) ----
    graph = None
    if args.graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            sess.run(hp, abi.HM_STAGE_STEP, stream)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                g.replay()
            ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ga.record(stream)
            for _ in range(args.steps):
                g.replay()
            gb.record(stream)
        torch.cuda.synchronize()
        if abi.hm_device_error() != 0:
            raise RuntimeError("device error word set during graph replay")
        gms = max_over_ranks(ga.elapsed_time(gb), dist, dev)
        graph = {"value": whole_job_rate(world, cfg.numel, args.steps, gms), "unit": UNIT,
                 "ms_per_step": gms / args.steps,
                 "note": "one fused update captured in a CUDA graph, replayed steps times"}
        del g

    # ---- end to end: host gradient in, host MXFP8 runtime weight out -----
    # as many steps as the headline: the first upload and the last download
    # are not overlapped, so fewer steps would weigh them more
    e2e_steps = max(2, args.steps)
    e2e_ms, copy_rates = e2e_pipelined(sess, hp, stream, e2e_steps, dist)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = whole_job_rate(world, cfg.numel, e2e_steps, e2e_ms)
    h2d = sess.total * 4
    d2h = sess.total + sess.total // 32

    # ---- the NEXT-row kernels on the same workload (their own timed loops) --
    extra = {} if args.skip_extra else bench_next_rows(cfg, sess, dev, stream)

    # ---- AdamW on the flat 64M shard (its own small timed loop) ----------
    adamw = None
    if not args.skip_adamw:
        adamw = bench_adamw(dev, stream)

    peaks = load_peaks()
    flops = ns_flops(cfg, cfg.muon.ns_steps)
    ns_tflops = flops / (stage_ms["ns_f2_requant"] / 1e3) / 1e12
    exec_flops = ns_executed_flops(cfg, cfg.muon.ns_steps)
    exec_tflops = exec_flops / (stage_ms["ns_f2_requant"] / 1e3) / 1e12
    P = cfg.numel
    strad = straddling_elems(cfg, info)
    kern = {
        "f0": {"gbs": 14.0 * P / (unfused_ms["f0"] / 1e3) / 1e9, "bytes_per_elem": 14},
        "gather": {"gbs": 4.0 * strad / (unfused_ms["gather"] / 1e3) / 1e9 if strad else None,
                   "bytes_per_straddling_elem": 4},
        "f2_scatter": {"gbs": 12.0 * P / (unfused_ms["f2"] / 1e3) / 1e9, "bytes_per_elem": 12},
        "mxfp8_requant": {"gbs": 5.03125 * P / (unfused_ms["requant"] / 1e3) / 1e9, "bytes_per_elem": 5.03125},
        "f0_gather_fused": {"gbs": 14.0 * P / (stage_ms["f0_gather"] / 1e3) / 1e9,
                            "bytes_per_elem": "14 (u of straddling units to their staging instead of the root)"},
        "f2_requant_fused": {"gbs": 13.03125 * P / (through_v_ms["f2_requant"] / 1e3) / 1e9,
                             "bytes_per_elem": 13.03125, "note": "the pass through v (HM_STAGE_ALL_FUSED)"},
    }
    for k in kern:
        if kern[k]["gbs"] is not None:
            kern[k]["frac"] = kern[k]["gbs"] / peaks["hbm_gbs"]
    kern["ns_unfused"] = {"tflops": flops / (unfused_ms["ns"] / 1e3) / 1e12, "ms": unfused_ms["ns"],
                          "frac": flops / (unfused_ms["ns"] / 1e3) / 1e12 / peaks["bf16_sustained"]}
    kern["ns_through_v"] = {"tflops": flops / (through_v_ms["ns"] / 1e3) / 1e12, "ms": through_v_ms["ns"],
                            "frac": flops / (through_v_ms["ns"] / 1e3) / 1e12 / peaks["bf16_sustained"],
                            "executed_frac": exec_flops / (through_v_ms["ns"] / 1e3) / 1e12 /
                            peaks["bf16_sustained"]}
    if adamw:
        kern["adamw_flat_64M"] = adamw
        adamw["frac"] = adamw["gbs"] / peaks["hbm_gbs"]
    for k, v in extra.items():
        v["frac"] = v["gbs"] / peaks["hbm_gbs"]
        kern[k] = v
    # the same HBM rates against the nominal 8 TB/s of GB300's HBM3e
    for v in kern.values():
        if v.get("gbs") is not None:
            v["frac_of_8tbs"] = v["gbs"] / 8000.0
    roofline = {"bound": "tensor", "achieved": ns_tflops, "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
                "frac": ns_tflops / peaks["bf16_sustained"], "traffic": ns_stage_traffic(cfg),
                "traffic_unit": "DRAM bytes per Newton-Schulz stage (one update), ncu: " + NS_STAGE_TRAFFIC["how"],
                "kernel": "Newton-Schulz stage (the step's second call): per shape class ns_small_kernel (Gram size "
                          "128: every iteration in one launch) or ns_gemm_kernel / ns_gemm_pair_kernel (3 products "
                          "x 5 iterations); the last product also applies f2 and the MXFP8 requant (timed with them); "
                          "X0 and the unit scales come from the first call (f0 inside the input pass)",
                "peak_kind": f"bf16 dense sustained ({peaks['source']})",
                "frac_of_burst": ns_tflops / peaks["bf16"],
                "note": "achieved counts the algorithmic 5(4m^2n+2m^3) FLOP per unit; the kernels skip the "
                        "below-diagonal tiles of the symmetric A and B, so executed tensor FLOP are lower",
                "executed_tflops": exec_tflops, "executed_frac": exec_tflops / peaks["bf16_sustained"],
                "executed_frac_of_burst": exec_tflops / peaks["bf16"]}

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        t0 = time.perf_counter()
        _, total, desc = oracle_sample_step(cfg)
        cpu = {"value": cfg.numel / total, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
               "sample": desc, "sample_wall_s": time.perf_counter() - t0}

    resident_gb = (sess.total * 21 + sess.ws_bytes) / 1e9
    n_classes, n_strad = info.n_classes, info.n_straddling
    sess.close()
    del sess
    torch.cuda.empty_cache()
    # ---- every shape class alone, and the other workloads (N = 1 only) ----
    classes, configs = {}, None
    if world == 1 and not args.skip_configs:
        classes = ns_class_table(cfg, dev, stream, peaks)
        configs = bench_other_configs(dev, stream, peaks)
    kern.update(classes)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16+fp32", "data": "synthetic (seeded N(0,0.02) w, N(0,1e-3) g)",
                "config": {"workload": f"{cfg.name}: {cfg.description}", "params": P, "units": len(cfg.units),
                           "shape_classes": n_classes, "straddling_units": n_strad,
                           "emulated_ranks": cfg.so, "parallelism": f"replica x{world}",
                           "l2": "inputs larger than L2 (resident state ~%.0f GB)" % resident_gb},
                "ns_tflops": ns_tflops, "ns_flops_per_step": flops, "ns_executed_flops_per_step": exec_flops,
                "stages_ms": stage_ms, "through_v_stages_ms": through_v_ms, "unfused_stages_ms": unfused_ms,
                "kernels": kern,
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
                        "copy_rates_gbs": copy_rates,
                        "note": "host gradient in, host MXFP8 weights + scales out, every step; copies on their own "
                                "streams overlap the previous / next step's Newton-Schulz stage"},
                "gpu_launches": launches, "clocks": clocks.summary()}
        if graph is not None:
            line["graph"] = graph
        if configs is not None:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def e2e_pipelined(sess, hp, stream, steps, dist):
    """Update phases fed from and returned to pinned host memory: every step
    copies its gradient in (9.2 GB for Video-DiT) and its MXFP8 weights and
    scales out.  The copies run on their own streams with double-buffered
    device gradients, MXFP8 weights and scales, so step k+1's upload and step
    k's download overlap the Newton-Schulz stages; every step's copies are
    inside the timed region, which runs from the first upload to the last
    download."""
    import torch

    from head_muon_mxfp8_gb300 import abi
    dev = sess.device
    g_dev = [sess.g, torch.empty_like(sess.g)]
    g_dev[1].copy_(sess.g)
    # q and s double-buffered too: the last products of step k+1 write them
    # while step k's are still on their way to the host
    q_dev = [sess.q, torch.empty_like(sess.q)]
    s_dev = [sess.s, torch.empty_like(sess.s)]
    g_host = torch.empty(sess.total, dtype=torch.float32, pin_memory=True)
    g_host.copy_(sess.g)
    q_host = [torch.empty(sess.total, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    s_host = [torch.empty(sess.total // 32, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    bufs = []
    for b in range(2):
        bufs.append(abi.hm_muon_bufs(sess.w.data_ptr(), sess.m.data_ptr(), g_dev[b].data_ptr(), sess.u.data_ptr(),
                                     sess.v.data_ptr(), q_dev[b].data_ptr(), s_dev[b].data_ptr()))
    cs_in = torch.cuda.Stream(device=dev)
    cs_out = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)
    front = abi.HM_STAGE_F0 | abi.HM_STAGE_GATHER | abi.HM_STAGE_FUSED | abi.HM_STAGE_SCRATCH
    ns_back = abi.HM_STAGE_STEP & ~(abi.HM_STAGE_F0 | abi.HM_STAGE_GATHER)

    def run(stages, b):
        abi.muon_update_units(sess.plan, bufs[b], hp, sess.ws, sess.ws_bytes, stages, sh)

    def pipeline(n, t0=None, t1=None):
        ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
        g_free = [None, None]
        out_done = [None, None]
        last_out = None
        if t0 is not None:
            t0.record(cs_in)
        for k in range(n):
            b = k % 2
            in_done = ev()
            with torch.cuda.stream(cs_in):
                if g_free[b] is not None:
                    cs_in.wait_event(g_free[b])
                g_dev[b].copy_(g_host, non_blocking=True)
                in_done.record(cs_in)
            stream.wait_event(in_done)
            run(front, b)
            g_free[b] = ev()
            g_free[b].record(stream)
            if out_done[b] is not None:
                stream.wait_event(out_done[b])  # step k-2's download has left q[b] and s[b]
            run(ns_back, b)
            back_done = ev()
            back_done.record(stream)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(back_done)
                q_host[b].copy_(q_dev[b], non_blocking=True)
                s_host[b].copy_(s_dev[b], non_blocking=True)
                out_done[b] = last_out = ev()
                last_out.record(cs_out)
        if t1 is not None:
            cs_out.wait_event(last_out)
            t1.record(cs_out)

    pipeline(1)  # warm-up
    torch.cuda.synchronize()
    # the box's copy rates alone (one gradient upload, one weight download),
    # which bound the pipelined step when they are below ~100 GB/s
    # (three of each: the rate of a shared host link dips now and then)
    rates = {}
    for name, dst, src in (("h2d_gbs", g_dev[1], g_host), ("d2h_gbs", q_host[0], sess.q)):
        rates[name] = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(cs_in):
                a.record(cs_in)
                dst.copy_(src, non_blocking=True)
                b.record(cs_in)
            torch.cuda.synchronize()
            rates[name].append(round(src.numel() * src.element_size() / (a.elapsed_time(b) * 1e6), 1))
    if dist:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    pipeline(steps, t0, t1)
    torch.cuda.synchronize()
    del g_dev[1], q_dev[1], s_dev[1]
    return t0.elapsed_time(t1), rates


def _time_calls(fn, stream, reps: int = 3):
    import torch
    with torch.cuda.stream(stream):
        fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def bench_next_rows(cfg, sess, dev, stream):
    """32 x 32 MXFP8 requant over the rank segments, the 128 x 4 scale relayout
    of every tensor's 1 x 32 scales, and the emulated gradient reduce-scatter
    (4 contributions in 2 nodes, BF16 stochastic rounding, accumulate), each
    timed with CUDA events on the bench stream."""
    import torch

    from head_muon_mxfp8_gb300 import abi
    sh = int(stream.cuda_stream)
    P = cfg.numel
    out = {}
    tensors, s_off = [], 0
    for m in cfg.members:
        tensors.append((m.offset, 0, s_off, m.rows, m.cols))
        s_off += (m.rows // 32) * (m.cols // 32)
    sc32 = torch.empty(s_off, dtype=torch.uint8, device=dev)
    ms = _time_calls(lambda: abi.mxfp8_requant_32x32(sess.chain, sess.w.data_ptr(), sess.q.data_ptr(),
                                                     sc32.data_ptr(), tensors, sh), stream)
    out["mxfp8_requant_32x32"] = {"gbs": 5.0 * P / (ms / 1e3) / 1e9, "ms": ms, "bytes_per_elem": 5}
    items, src_off, dst_off = [], 0, 0
    for m in cfg.members:
        kb = m.cols // 32
        items.append((src_off, dst_off, m.rows, kb, 1))
        src_off += m.rows * kb
        dst_off += -(-m.rows // 128) * -(-kb // 4) * 512
    src = torch.zeros(src_off, dtype=torch.uint8, device=dev)
    dst = torch.empty(dst_off, dtype=torch.uint8, device=dev)
    ms = _time_calls(lambda: abi.mxfp8_scale_relayout(src.data_ptr(), dst.data_ptr(), items, sh), stream)
    out["mxfp8_scale_relayout"] = {"gbs": (src_off + dst_off) / (ms / 1e3) / 1e9, "ms": ms,
                                   "bytes": "scales read + tiled scales written"}
    del src, dst, sc32
    parts = torch.empty((4, P), dtype=torch.float32, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    parts.normal_(0.0, 1e-3, generator=gen)
    ms = _time_calls(lambda: abi.reduce_scatter_grad(sess.chain, parts.data_ptr(), 4, 2, sess.g.data_ptr(),
                                                     abi.HM_RS_BF16_SR, True, 1234, 0, sh), stream)
    out["grad_reduce_scatter_bf16sr"] = {"gbs": 24.0 * P / (ms / 1e3) / 1e9, "ms": ms,
                                         "bytes_per_elem": "4 contributions x 4 + g read and written"}
    del parts
    return out


def bench_adamw(dev, stream, steps: int = 10):
    import torch

    from head_muon_mxfp8_gb300 import abi
    from head_muon_mxfp8_gb300.session import adamw_hparams
    cfg = workloads.flat_adamw()
    n = cfg.numel
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    w = torch.empty(n, device=dev).normal_(0, 0.02, generator=gen)
    g = torch.empty(n, device=dev).normal_(0, 1e-3, generator=gen).to(torch.bfloat16)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    hp = adamw_hparams(cfg.adamw, 1)
    sh = int(stream.cuda_stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            abi.adamw_update_flat(w.data_ptr(), g.data_ptr(), abi.HM_BF16, m.data_ptr(), v.data_ptr(), n, hp, sh)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            abi.adamw_update_flat(w.data_ptr(), g.data_ptr(), abi.HM_BF16, m.data_ptr(), v.data_ptr(), n, hp, sh)
        b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"gbs": 26.0 * n / (ms / 1e3) / 1e9, "ms": ms, "bytes_per_elem": 26,
            "workload": "flat_adamw 67,108,864 fp32 params, bf16 grads (inputs larger than L2)"}


def time_muon_update(cfg, dev, stream, steps: int, warmup: int):
    """Times `steps` whole update phases of cfg on its own session, exactly as
    the headline step runs (HM_STAGE_STEP as two calls, CUDA events on the
    launching stream around each, inputs resident in HBM), with the SM clocks
    sampled meanwhile.  The session is freed before returning."""
    import torch

    from head_muon_mxfp8_gb300 import abi
    from head_muon_mxfp8_gb300.session import MuonSession, muon_hparams
    sess = MuonSession.from_config(cfg, device=dev, canaries=False)
    data = workloads.generate_device(cfg, dev, seed=cfg.seed)
    sess.load("w", data["w"])
    sess.load("g", data["g"])
    sess.m.zero_()
    del data
    hp = muon_hparams(cfg.muon)
    front_s = abi.HM_STAGE_F0 | abi.HM_STAGE_GATHER | abi.HM_STAGE_FUSED | abi.HM_STAGE_SCRATCH
    ns_back = abi.HM_STAGE_STEP & ~(abi.HM_STAGE_F0 | abi.HM_STAGE_GATHER)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            sess.run(hp, abi.HM_STAGE_STEP, stream)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    launches0 = abi.hm_kernel_launches()
    with torch.cuda.stream(stream):
        for e in evs:
            e[0].record(stream)
            sess.run(hp, front_s, stream)
            e[1].record(stream)
            sess.run(hp, ns_back, stream)
            e[2].record(stream)
    launches = abi.hm_kernel_launches() - launches0
    torch.cuda.synchronize()
    clocks.stop()
    if abi.hm_device_error() != 0:
        raise RuntimeError(f"device error word set while timing {cfg.name}")
    out = {"f0_gather_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
           "ns_ms": statistics.mean(e[1].elapsed_time(e[2]) for e in evs),
           "step_ms": evs[0][0].elapsed_time(evs[-1][2]) / steps,
           "launches_per_step": launches / steps, "clocks": clocks.summary(),
           "n_classes": int(sess.info.n_classes), "n_straddling": int(sess.info.n_straddling)}
    sess.close()
    del sess
    torch.cuda.empty_cache()
    return out


def ns_class_table(cfg, dev, stream, peaks, steps: int = 5, warmup: int = 2):
    """Every Newton-Schulz shape class of cfg timed alone (its members as a
    workload of their own, the same step as the headline).  Beside the tensor
    fractions each class reports an HBM fraction against the traffic of the
    iteration run product by product: per iteration X X^T reads X (2mn bytes)
    and writes A (2m^2), bA + cAA reads A and writes B (4m^2), B X reads B and
    X and writes X' (2m^2 + 4mn); plus u in (2mn) and, for the last product
    with f2 and G folded in, w read and written, q and s written
    (8mn + mn + mn/32) -- per unit."""
    classes = {}
    for u in cfg.units:
        k = (min(u.rows, u.cols), max(u.rows, u.cols))
        classes[k] = classes.get(k, 0) + 1
    if len(classes) < 2:
        return {}
    out = {}
    steps_ns = cfg.muon.ns_steps
    for (m, n), cnt in sorted(classes.items()):
        sub = workloads.class_subset(cfg, m, n)
        t = time_muon_update(sub, dev, stream, steps, warmup)
        sec = t["ns_ms"] / 1e3
        alg = ns_flops(sub, steps_ns)
        exe = ns_executed_flops(sub, steps_ns)
        io = cnt * (steps_ns * (6.0 * m * n + 8.0 * m * m) + 2.0 * m * n + (10.0 + 1 / 32) * m * n)
        out[f"ns_class_{m}x{n}"] = {
            "units": cnt, "ms": t["ns_ms"], "tflops": alg / sec / 1e12,
            "frac": alg / sec / 1e12 / peaks["bf16_sustained"],
            "executed_tflops": exe / sec / 1e12, "executed_frac": exe / sec / 1e12 / peaks["bf16_sustained"],
            "hbm_bytes_product_by_product": io, "gbs": io / sec / 1e9, "hbm_frac": io / sec / 1e9 / peaks["hbm_gbs"],
            "sm_mhz": t["clocks"]["sm_mhz"]}
    return out


def bench_other_configs(dev, stream, peaks, steps: int = 10, warmup: int = 3):
    """The other workloads, each timed like the headline after its session is
    freed: params/s of the whole update phase, the Newton-Schulz stage's
    tensor fractions, the fused f0 + gather pass's HBM fraction, the clocks
    seen, and the CPU oracle on a bounded sample of the same workload.  Flat
    AdamW is one AdamW step over the 64 M shard followed by the MXFP8 requant
    of the 64 M weights as 16384 x 4096 row-major blocks."""
    out = {}
    for name, k in (("tiny", 50), ("lm_layer", steps), ("moe_layer", steps)):
        cfg = workloads.get(name)
        t = time_muon_update(cfg, dev, stream, k, warmup)
        classes = ns_class_table(cfg, dev, stream, peaks) if name == "lm_layer" else {}
        P = cfg.numel
        alg = ns_flops(cfg, cfg.muon.ns_steps)
        exe = ns_executed_flops(cfg, cfg.muon.ns_steps)
        sec = t["ns_ms"] / 1e3
        t0 = time.perf_counter()
        _, total, desc = oracle_sample_step(cfg)
        cpu = {"value": P / total, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle", "sample": desc,
               "sample_wall_s": time.perf_counter() - t0}
        out[name] = {
            "params": P, "units": len(cfg.units), "shape_classes": t["n_classes"],
            "straddling_units": t["n_straddling"], "emulated_ranks": cfg.so, "steps": k,
            "value": P * 1e3 / t["step_ms"], "unit": UNIT, "ms_per_step": t["step_ms"],
            "stages_ms": {"f0_gather": t["f0_gather_ms"], "ns_f2_requant": t["ns_ms"]},
            "ns": {"tflops": alg / sec / 1e12, "frac": alg / sec / 1e12 / peaks["bf16_sustained"],
                   "executed_tflops": exe / sec / 1e12,
                   "executed_frac": exe / sec / 1e12 / peaks["bf16_sustained"]},
            "f0_gather_fused": {"gbs": 14.0 * P / (t["f0_gather_ms"] / 1e3) / 1e9,
                                "frac": 14.0 * P / (t["f0_gather_ms"] / 1e3) / 1e9 / peaks["hbm_gbs"]},
            "gpu_launches_per_step": t["launches_per_step"], "clocks": t["clocks"], "cpu_baseline": cpu,
            "ns_classes": classes,
            "l2": ("inputs larger than L2" if P * 21 > 129e6 else
                   "state fits in L2 (no flush between steps; launch-bound)")}
    out["flat_adamw"] = bench_flat_adamw_config(dev, stream, peaks)
    return out


def bench_flat_adamw_config(dev, stream, peaks, steps: int = 10):
    import torch

    from head_muon_mxfp8_gb300 import abi
    from head_muon_mxfp8_gb300.session import adamw_hparams
    from oracle import adamw as OA
    from oracle import mxfp8 as OX
    cfg = workloads.flat_adamw()
    n = cfg.numel
    rows, k = 16384, n // 16384
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed)
    w = torch.empty(n, device=dev).normal_(0, cfg.w_std, generator=gen)
    g = torch.empty(n, device=dev).normal_(0, cfg.g_std, generator=gen).to(torch.bfloat16)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    q = torch.empty(n, dtype=torch.uint8, device=dev)
    sc = torch.empty(n // 32, dtype=torch.uint8, device=dev)
    sh = int(stream.cuda_stream)
    h = cfg.adamw
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    clocks = ClockSampler(dev.index or 0)
    with torch.cuda.stream(stream):
        for t in range(3):
            abi.adamw_update_flat(w.data_ptr(), g.data_ptr(), abi.HM_BF16, m.data_ptr(), v.data_ptr(), n,
                                  adamw_hparams(h, t + 1), sh)
            abi.mxfp8_requant_packed(w.data_ptr(), q.data_ptr(), sc.data_ptr(), [(0, 0, 0, rows, k)], sh)
        torch.cuda.synchronize()
        clocks.start()
        time.sleep(0.3)
        for j, e in enumerate(evs):
            e[0].record(stream)
            abi.adamw_update_flat(w.data_ptr(), g.data_ptr(), abi.HM_BF16, m.data_ptr(), v.data_ptr(), n,
                                  adamw_hparams(h, 4 + j), sh)
            e[1].record(stream)
            abi.mxfp8_requant_packed(w.data_ptr(), q.data_ptr(), sc.data_ptr(), [(0, 0, 0, rows, k)], sh)
            e[2].record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    a_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    r_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    step_ms = evs[0][0].elapsed_time(evs[-1][2]) / steps
    del w, g, m, v, q, sc
    torch.cuda.empty_cache()
    # the oracle on a 262,144-element slice (AdamW in float64, then the requant), scaled by elements
    rng = np.random.default_rng(0)
    ns = 1 << 18
    t0 = time.perf_counter()
    w0 = (rng.standard_normal(ns) * cfg.w_std).astype(np.float32)
    g0 = (rng.standard_normal(ns) * cfg.g_std).astype(np.float32)
    t1 = time.perf_counter()
    w1, _, _ = OA.adamw_step(w0, g0, np.zeros(ns), np.zeros(ns), h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, 1)
    OX.requant_list(w1.astype(np.float32), [(0, ns // k, k)])
    per_el = (time.perf_counter() - t1) / ns
    return {"params": n, "steps": steps, "value": n * 1e3 / step_ms, "unit": UNIT, "ms_per_step": step_ms,
            "stages_ms": {"adamw": a_ms, "mxfp8_requant": r_ms},
            "kernels": {"adamw": {"gbs": 26.0 * n / (a_ms / 1e3) / 1e9, "bytes_per_elem": 26,
                                  "frac": 26.0 * n / (a_ms / 1e3) / 1e9 / peaks["hbm_gbs"]},
                        "mxfp8_requant": {"gbs": 5.03125 * n / (r_ms / 1e3) / 1e9, "bytes_per_elem": 5.03125,
                                          "frac": 5.03125 * n / (r_ms / 1e3) / 1e9 / peaks["hbm_gbs"]}},
            "clocks": clocks.summary(),
            "cpu_baseline": {"value": 1.0 / per_el, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": "oracle AdamW (float64) + MXFP8 requant on 262144 elements, scaled by elements",
                             "sample_wall_s": time.perf_counter() - t0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="video_dit", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-adamw", action="store_true")
    ap.add_argument("--skip-extra", action="store_true", help="skip the 32x32 / relayout / reduce-scatter timings")
    ap.add_argument("--graph", action="store_true", help="also time the fused step replayed from a CUDA graph")
    ap.add_argument("--skip-configs", action="store_true",
                    help="skip the per-class Newton-Schulz table and the other workloads (N = 1 only)")
    args = ap.parse_args()
    cfg = workloads.get(args.workload)
    if cfg.optimizer != "muon":
        raise SystemExit("bench workloads are Muon tensor lists")
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
