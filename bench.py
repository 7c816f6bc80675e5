"""Benchmark of the work-decomposed BF16 GEMM on GB300.

One step = one sk_gemm call: the whole hot path (schedule walk, TMA/tcgen05 MAC loop,
partial-tile fixup, epilogue) over the workload's synthetic BF16 inputs, resident in HBM.
Default workload: the wave-quantized GEMM 2048 x 2432 x 4096 (304 tiles of 128 x 128 =
2 waves + 8 on 148 SMs), BF16 out, the hybrid rule on 148 SMs, computed with 256 x 256
CTA-pair tiles (80 tiles on 74 pairs: again 2 waves with a short tail); the per-schedule
table also reports the pages' 128 x 128 tile. The headline steps run back to back on one
stream, step i on input set i mod R, where the R copies of A, B and C (R = 12 here, 560 MB)
are at least 4x the L2, so each step reads its operands from HBM. Each launch overlaps the
one before it (programmatic dependent launch; --overlap 0 turns it off). One pair of CUDA
events on the launching stream brackets the K steps; the headline value is TFLOP/s = 2MNK
/ (time / K). `--timing flush` times one launch per event pair with a 256 MiB L2 flush
before each instead (also reported, as `isolated_launch`).

Prints ONE JSON line (rank 0). `--impl reference` times the CPU oracle (FP64 dot products
over the BF16 inputs) on a bounded row sample of the same workload instead.
Multi-GPU (torchrun): the job is one GEMM of N * 2048 rows split by rows over the N ranks
(m_shard), B replicated, no collective on the data path (weak scaling: each rank's share is
the headline shape); a barrier brackets the timed region and the slowest rank's time is
reported.
"""
from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

PEAKS_FALLBACK = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "bf16_tflops_sustained": 1700.0}
METRIC = "BF16 GEMM TFLOP/s and % tensor peak vs tile count, per schedule, 1xGB300"
WORKLOADS = {"waveq": synth.WAVEQ, "skinny": synth.SKINNY, "large": synth.LARGE,
             "smallm96": synth.SMALLM_96, "smallm256": synth.SMALLM_256, "toy": synth.TOY}
# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the GEMM kernel
# from one ncu capture, keyed by workload/schedule; valid only for the kernel source it
# was taken on (sha256 of sk_kernels.cu, first 16 hex digits).
# Nominal dense BF16 tensor peak and HBM bandwidth of one GB300, for context beside the measured
# peaks (MEASURED_PEAKS.json) that the roofline fractions use.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0
TRAFFIC = {
    "waveq_2048x2432x4096/hybrid/tile2@148": {"bytes": 36822016 + 1379328, "kernel_sha": "06e5f6597b0a0f4a",
                                              "profile": "profiles/sk_gemm_kernel_waveq_2048x2432x4096_pair256_hybrid148.md"},
    "waveq_2048x2432x4096/dp/tile2@148": {"bytes": 36804864 + 3328, "kernel_sha": "06e5f6597b0a0f4a",
                                          "profile": "profiles/sk_gemm_kernel_waveq_2048x2432x4096_pair256_dp148_vs_hybrid.md"},
    "waveq_2048x2432x4096/hybrid/tile0@148": {"bytes": 36821504 + 398336, "kernel_sha": "06e5f6597b0a0f4a",
                                              "profile": "profiles/sk_gemm_kernel_waveq_2048x2432x4096_tile128_hybrid148.md"},
    "skinny_512x512x65536/splitk/s16p1/tile2@148": {"bytes": 134333696 + 4358656, "kernel_sha": "06e5f6597b0a0f4a",
                                                    "profile": "profiles/sk_reduce_kernel_skinny_512x512x65536_pair256_splitk16.md"},
    "large_8192x8192x8192/dp/tile2@148": {"bytes": 2030805760 + 130338048, "kernel_sha": "06e5f6597b0a0f4a",
                                          "profile": "profiles/sk_gemm_kernel_large_8192_pair256_dp148_raster.md"},
    "large_8192x8192x8192/dp/tile2@148/r0s8": {"bytes": 1036968704 + 126036224, "kernel_sha": "06e5f6597b0a0f4a",
                                               "profile": "profiles/sk_gemm_kernel_large_8192_pair256_dp148_raster.md"},
}


def graph_upload(graph, stream):
    """Upload an instantiated CUDA graph to the device (cuGraphUpload), so that its first replay
    does not pay for it. Best effort: without the handle or the driver entry point the first
    replay uploads the graph itself."""
    try:
        import ctypes
        h = graph.raw_cuda_graph_exec()
        cu = ctypes.CDLL("libcuda.so.1")
        cu.cuGraphUpload.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        return cu.cuGraphUpload(ctypes.c_void_p(int(h)), ctypes.c_void_p(int(stream.cuda_stream))) == 0
    except Exception:
        return False


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def kernel_sha():
    p = os.path.join(ROOT, "gemm_work_decomposition_gb300", "csrc", "sk_kernels.cu")
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.idx = gpu_id
        self.proc = None
        self.lines = []

    def _query(self, loop=False):
        cmd = ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits"]
        if loop:
            cmd.append("-lms=100")
        return cmd

    def start(self):
        try:
            self.lines += subprocess.run(self._query(), capture_output=True, text=True, timeout=20).stdout.splitlines()
            self.proc = subprocess.Popen(self._query(True), stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=10)
                self.lines += out.splitlines()
            except Exception:
                self.proc.kill()
        try:
            self.lines += subprocess.run(self._query(), capture_output=True, text=True, timeout=20).stdout.splitlines()
        except Exception:
            pass

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        mhz, mx, reasons = [], 0.0, set()
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(mhz)) if mhz else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(mhz)}


def m_shard(M: int, world: int, rank: int):
    """Rows of C (and of A) that rank `rank` computes when a GEMM's M is split over `world`
    devices with B replicated: (first row, row count), divmod split with the first M % world
    ranks one row longer. The shards tile [0, M) in rank order; no data is exchanged."""
    q, big = divmod(M, world)
    return rank * q + min(rank, big), q + (1 if rank < big else 0)


def sharded_workload(w, world: int):
    """The job on `world` devices: one GEMM of world * M rows (the workload's seed and value
    recipe, rows added), each device computing its M-row shard against the whole B."""
    import dataclasses
    return dataclasses.replace(w, name=f"{w.name}_msplit{world}", M=w.M * world)


def max_over_ranks(x: float, dist, device) -> float:
    """The slowest rank's value (float64 all-reduce MAX); x itself on one rank."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_step: float, steps: int, total_ms: float) -> float:
    """Whole-job throughput: every rank's steps over the slowest rank's time."""
    return world * flops_per_step * steps / (total_ms / 1e3) / 1e12


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def cpu_oracle_sample(w, seconds: float, rows_per_block: int = 256):
    """Time the oracle's FP64 GEMM on row blocks of the workload for about `seconds`."""
    from oracle import gemm as og
    A_bits, B_bits = synth.make_inputs(w)
    rows = min(rows_per_block, w.M)
    flops = 0.0
    t0 = time.perf_counter()
    n = 0
    while True:
        r0 = (n * rows) % max(1, w.M - rows + 1)
        og.ref_gemm(A_bits[r0:r0 + rows], B_bits, w.layout)
        flops += 2.0 * rows * w.N * w.K
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return flops / el / 1e12, el, n, rows


MODE_IDS = {"dp": 0, "splitk": 1, "streamk": 2, "hybrid": 3}
TILE_NAMES = {0: "128x128", 1: "256x128 CTA pair", 2: "256x256 CTA pair", 3: "128x256"}


def schedule_config(args, w, plan, sms: int) -> dict:
    """The config keys that name the workload and its schedule (shared by both arms); `plan`
    is the work-unit map's header (sk_plan's, or the oracle's, which equals it)."""
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "layout": w.layout, "out": w.out,
            "schedule": args.mode, "split_partials": args.partials, "reduction": args.reduction, "num_sms": sms,
            "tile": TILE_NAMES[args.tile], "tile_m": int(plan[12]), "tile_n": int(plan[13]),
            "ctas_per_tile": int(plan[14]), "raster": "along_n" if args.raster == 0 else "along_m",
            "swizzle": args.swizzle, "sk_groups": int(plan[17]), "tiles": int(plan[2]), "iters": int(plan[3]),
            "workers": int(plan[4]), "resolved_mode": int(plan[1]), "sk_tiles": int(plan[5]),
            "sk_units": int(plan[6]), "accumulate": "fp32"}


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    from oracle import schedule as osch
    sms = args.sms or 148
    plan = osch.plan_map(osch.build_plan(w.M, w.N, w.K, sms, MODE_IDS[args.mode],
                                         splits=args.splits if args.mode == "splitk" else 1,
                                         split_partials=args.partials, tile=args.tile, raster=args.raster,
                                         swizzle=args.swizzle, sk_groups=args.sk_groups))
    seconds = args.ref_seconds
    for _ in range(args.warmup):
        cpu_oracle_sample(w, 0.0)
    times, flops = [], 0.0
    rows = min(256, w.M)
    for _ in range(args.steps):
        v, el, n, rows = cpu_oracle_sample(w, seconds / max(1, args.steps))
        times.append(el / n)
        flops = 2.0 * rows * w.N * w.K
    ms = float(np.mean(times)) * 1e3
    value = flops / (ms / 1e3) / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(schedule_config(args, w, plan, sms),
                       step=f"FP64 oracle GEMM on {rows} rows of C (bounded sample)"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} x {w.N} x {w.K} FP64 per step (numpy matmul, default BLAS threads)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


SWEEP_COMPACT = (1024, 1536, 2048, 2304, 2432, 3072, 3840, 4096)
# (name, mode, splits, split_partials); splits None: the CUTLASS page's Split-K factor for the
# shape (sk_split_k_slices, clamped to the K loop). The `_slabs` rows are Split-K with FP32
# [s, M, N] slabs summed by the reduction pass (split_partials 1).
SWEEP_SCHEDULES = (("dp", 0, 1, 0), ("splitk2", 1, 2, 0), ("splitk4", 1, 4, 0), ("splitk_cutlass", 1, None, 0),
                   ("splitk2_slabs", 1, 2, 1), ("splitk4_slabs", 1, 4, 1), ("streamk", 2, 1, 0), ("hybrid", 3, 1, 0))


def sweep_points(sk, torch, dev, red, flush, stream, peak_tf, l2_bytes, sizes, configs, flushed=0, b2b=40,
                 library=False):
    """Tile-count sweep over square M = N in `sizes`, K = 4096 (the tile-count sweep
    workload): every schedule of SWEEP_SCHEDULES (data-parallel, Split-K s = 2 and 4 with the
    owner fixup and with FP32 slabs and the reduction pass, Split-K with the CUTLASS page's
    factor heuristic, Stream-K
    and the hybrid rule, which is the decision rule's own choice) for each (num_sms, tile) of
    `configs`. Each point is timed `b2b` overlapped launches back to back over rotating copies
    of A, B and C that together exceed 4x the L2 (the headline's method, mean per launch),
    and, with `flushed` > 0, as the median of that many single launches with the L2 flushed
    before each. Yields one dict per point (and per size a cuBLAS row with `library`)."""
    for m in sizes:
        ww = synth.sweep(m)
        A_bits, B_bits = synth.make_inputs(ww)
        A = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        C = torch.empty((m, m), dtype=torch.bfloat16, device=dev)
        set_b = (A.numel() + B.numel() + C.numel()) * 2
        rot = [(A, B, C)] + [(A.clone(), B.clone(), torch.empty_like(C))
                             for _ in range(max(2, -(-4 * l2_bytes // set_b)) - 1)]
        fl = 2.0 * m * m * ww.K
        for nsms, tile in configs:
            for name, mode, s, parts in SWEEP_SCHEDULES:
                if s is None:
                    s = min(sk.sk_split_k_slices(m, m, ww.K, nsms), -(-ww.K // 64))
                sch = sk.schedule(mode, s, split_partials=parts, tile=tile)
                nb = sk.sk_workspace_size(m, m, ww.K, nsms, sch, red)
                ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
                plan = sk.sk_plan(m, m, ww.K, nsms, sch)
                row = {"M": m, "N": m, "K": ww.K, "tile": tile, "tiles": int(plan[2]), "num_sms": nsms,
                       "schedule": name, "splits": s if mode == 1 else None, "resolved_mode": int(plan[1]),
                       "label": int(plan[9])}
                if flushed:
                    for _ in range(5):
                        sk.sk_gemm(A, B, C, sk.SK_BF16, m, m, ww.K, sk.SK_NN, sch, red, nsms, ws, nb, stream)
                    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                          for _ in range(flushed)]
                    for a, b in ev:
                        flush.zero_()
                        a.record(stream)
                        sk.sk_gemm(A, B, C, sk.SK_BF16, m, m, ww.K, sk.SK_NN, sch, red, nsms, ws, nb, stream)
                        b.record(stream)
                    torch.cuda.synchronize(dev)
                    t = float(np.median([a.elapsed_time(b) for a, b in ev]))
                    row.update({"us": t * 1e3, "tflops": fl / (t / 1e3) / 1e12,
                                "frac_of_measured_peak": fl / (t / 1e3) / 1e12 / peak_tf})
                sch_o = sk.schedule(mode, s, split_partials=parts, tile=tile, overlap=1)
                for i in range(10):
                    a_, b_, c_ = rot[i % len(rot)]
                    sk.sk_gemm(a_, b_, c_, sk.SK_BF16, m, m, ww.K, sk.SK_NN, sch_o, red, nsms, ws, nb, stream)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for i in range(b2b):
                    a_, b_, c_ = rot[i % len(rot)]
                    sk.sk_gemm(a_, b_, c_, sk.SK_BF16, m, m, ww.K, sk.SK_NN, sch_o, red, nsms, ws, nb, stream)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                assert sk.sk_status(ws, stream) == sk.SK_OK
                tb = e0.elapsed_time(e1) / b2b
                tfb = fl / (tb / 1e3) / 1e12
                row.update({"us_b2b": tb * 1e3, "tflops_b2b": tfb, "frac_of_measured_peak_b2b": tfb / peak_tf,
                            "rotating_sets": len(rot)})
                yield row
        if library:
            # The library GEMM (cuBLAS through torch.matmul, BF16 out) on the same operands,
            # timed the same two ways: context for the schedules, outside any timed step.
            t, tb = library_timed(torch, dev, flush, stream, rot, m, m, flushed=max(flushed, 10), b2b=b2b)
            yield {"M": m, "N": m, "K": ww.K, "tile": None, "num_sms": None, "schedule": "cublas",
                   "us": t * 1e3, "tflops": fl / (t / 1e3) / 1e12, "frac_of_measured_peak": fl / (t / 1e3) / 1e12 / peak_tf,
                   "us_b2b": tb * 1e3, "tflops_b2b": fl / (tb / 1e3) / 1e12,
                   "frac_of_measured_peak_b2b": fl / (tb / 1e3) / 1e12 / peak_tf, "rotating_sets": len(rot)}
        del rot, A, B, C


def run_sweep(sk, torch, dev, path, red, flush, stream, peak_tf, dev_sms, l2_bytes):
    """The full tile-count sweep: M = N = 128 .. 4096 step 128, K = 4096, every schedule with
    the pages' 128 x 128 tile and the 256 x 256 CTA-pair tile, on 148 SMs and on the device's
    SM count; one JSON line per point, 30 flushed single launches and 60 back to back."""
    with open(path, "w") as f:
        for row in sweep_points(sk, torch, dev, red, flush, stream, peak_tf, l2_bytes, synth.SWEEP_SIZES,
                                ((148, 0), (dev_sms, 0), (148, 2), (dev_sms, 2)), flushed=30, b2b=60, library=True):
            f.write(json.dumps(row) + "\n")
            f.flush()


def run_sweep_compact(sk, torch, dev, red, flush, stream, peak_tf, l2_bytes):
    """The tile-count sweep in the default bench line: M = N in SWEEP_COMPACT, K = 4096, the
    schedules of SWEEP_SCHEDULES with the pages' 128 x 128 tile and the 256 x 256 CTA-pair tile
    on 148 SMs,
    back to back (40 launches per point). Per size: TFLOP/s and fraction of the measured peak
    per schedule and tile, the rule's choice, and the best."""
    table = {}
    for row in sweep_points(sk, torch, dev, red, flush, stream, peak_tf, l2_bytes, SWEEP_COMPACT,
                            ((148, 0), (148, 2)), flushed=0, b2b=40, library=True):
        key = str(row["M"])
        ent = table.setdefault(key, {"tiles_128x128": (row["M"] // 128) ** 2})
        if row["schedule"] == "cublas":
            ent["cublas_tflops"] = round(row["tflops_b2b"], 1)
            continue
        tname = {0: "128x128", 2: "pair256x256"}[row["tile"]]
        ent[f"{tname}/{row['schedule']}"] = {"us": round(row["us_b2b"], 2), "tflops": round(row["tflops_b2b"], 1),
                                             "frac_of_measured_peak": round(row["frac_of_measured_peak_b2b"], 4)}
        if row["splits"] is not None:
            ent[f"{tname}/{row['schedule']}"]["splits"] = row["splits"]
        if row["schedule"] == "hybrid":
            ent[f"{tname}/rule_choice"] = {0: "dp", 3: "hybrid"}.get(row["resolved_mode"], str(row["resolved_mode"]))
    for ent in table.values():
        pts = {k: v for k, v in ent.items() if isinstance(v, dict)}
        best = max(pts, key=lambda k: pts[k]["tflops"])
        ent["best"] = {"schedule": best, **pts[best]}
    return {"K": 4096, "num_sms": 148, "timing": "back to back, 40 overlapped launches over rotating inputs >= 4x L2",
            "sizes": table}


def library_timed(torch, dev, flush, stream, rot, M, N, nt=False, flushed=30, b2b=60):
    """torch.matmul (cuBLAS) on the rotating sets `rot` of (A, B, C) with BF16 C: the median of
    `flushed` single calls with the L2 flushed before each, and the mean of `b2b` calls back to
    back over the sets; both in ms. With `nt` B is stored N x K and passed transposed."""
    def call(i):
        a_, b_, c_ = rot[i % len(rot)]
        torch.matmul(a_, b_.t() if nt else b_, out=c_)

    with torch.cuda.stream(stream):
        for i in range(10):
            call(i)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(flushed)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            call(0)
            b.record(stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(b2b):
            call(i)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return float(np.median([a.elapsed_time(b) for a, b in ev])), e0.elapsed_time(e1) / b2b


def run_smallm(sk, torch, dev, flush, stream, dev_sms, rounds=9, samples=40, warmup=20):
    """The split-K report's shapes (B stored [N,K], FP32 out): M = 96 and 256, N = 512,
    K = 2048. The [splits, M, N] slab chain at s = 2, 4, 8, 16 (every split stores its
    slab; a reduction pass sums them, two launches), the same slabs summed inside the one
    launch (the splits of a tile share the sum when all run at once, else the last to
    arrive sums it), and the owner-wait fixups.

    Timed with the report's confirmation protocol ("Consecutive-B split-K NAX GEMM",
    Confirmation): every arm gets `warmup` untimed calls; then `rounds` rounds of `samples`
    samples, each sample running every arm once, with the arm order rotated by one from one
    sample to the next; a second direction repeats this with the arm order reversed. An
    arm-sample takes two event-timed measurements behind an L2 flush: pack 1, one whole
    GEMM, and pack 8, eight whole GEMMs over the same inputs, divided by eight. Reported per
    arm: median, p10 and p90 of pack 1 and of pack 8 over all samples of both directions, and
    (`us_b2b`) the mean of 200 overlapped launches back to back over rotating inputs of at
    least 4x the L2. Each arm's C is compared bit for bit before and after its timing."""
    out = {}
    for w in (synth.SMALLM_96, synth.SMALLM_256):
        A_bits, B_bits = synth.make_inputs(w)
        A = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        set_b = A.numel() * 2 + B.numel() * 2 + w.M * w.N * 4
        rot = [(A.clone(), B.clone(), torch.empty((w.M, w.N), dtype=torch.float32, device=dev))
               for _ in range(-(-4 * (129 << 20) // set_b))]
        fl = 2.0 * w.M * w.N * w.K
        kws = [(f"slabs_s{s}", dict(mode=sk.SK_SPLITK, splits=s, split_partials=1)) for s in (2, 4, 8, 16)]
        kws += [(f"slabs_1launch_s{s}", dict(mode=sk.SK_SPLITK, splits=s, split_partials=2)) for s in (2, 4, 8, 16)]
        kws += [("splitk8_fixup", dict(mode=sk.SK_SPLITK, splits=8)), ("streamk", dict(mode=sk.SK_STREAMK)),
                ("streamk_pass", dict(mode=sk.SK_STREAMK, split_partials=1)), ("hybrid", dict(mode=sk.SK_HYBRID))]
        arms = []
        for name, kw in kws:
            sch = sk.schedule(**kw)
            nb = sk.sk_workspace_size(w.M, w.N, w.K, dev_sms, sch, 0)
            ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
            C = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)
            arms.append(dict(name=name, sch=sch, sch_o=sk.schedule(overlap=1, **kw), ws=ws, nb=nb, C=C,
                             one=[], pack8=[]))

        def call(arm, a_=A, b_=B, c_=None, sch=None):
            sk.sk_gemm(a_, b_, arm["C"] if c_ is None else c_, sk.SK_F32, w.M, w.N, w.K, sk.SK_NT,
                       sch or arm["sch"], 0, dev_sms, arm["ws"], arm["nb"], stream)

        for arm in arms:
            for _ in range(warmup):
                call(arm)
        torch.cuda.synchronize(dev)
        before = [arm["C"].clone() for arm in arms]
        n = len(arms)
        for direction in (1, -1):
            order0 = list(range(n)) if direction == 1 else list(range(n - 1, -1, -1))
            for _ in range(rounds):
                pending = []
                for j in range(samples):
                    for a in order0[j % n:] + order0[:j % n]:
                        arm = arms[a]
                        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                        flush.zero_()
                        ev[0].record(stream)
                        call(arm)
                        ev[1].record(stream)
                        flush.zero_()
                        ev[2].record(stream)
                        for _ in range(8):
                            call(arm)
                        ev[3].record(stream)
                        pending.append((arm, ev))
                torch.cuda.synchronize(dev)
                for arm, ev in pending:
                    arm["one"].append(ev[0].elapsed_time(ev[1]) * 1e3)
                    arm["pack8"].append(ev[2].elapsed_time(ev[3]) * 1e3 / 8)
        rows = {}
        for arm, c0 in zip(arms, before):
            assert torch.equal(arm["C"], c0), f"{w.name}/{arm['name']}: C changed during timing"
            for i in range(20):
                a_, b_, c_ = rot[i % len(rot)]
                call(arm, a_, b_, c_, arm["sch_o"])
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(200):
                a_, b_, c_ = rot[i % len(rot)]
                call(arm, a_, b_, c_, arm["sch_o"])
            e1.record(stream)
            torch.cuda.synchronize(dev)
            b2b = e0.elapsed_time(e1) / 200 * 1e3
            assert sk.sk_status(arm["ws"], stream) == sk.SK_OK
            one, p8 = np.asarray(arm["one"]), np.asarray(arm["pack8"])
            name = arm["name"]
            launches = 2 if (name.startswith("slabs_s") or name.endswith("_pass")) else 1
            med = float(np.median(one))
            rows[name] = {"us": med, "us_p10": float(np.percentile(one, 10)), "us_p90": float(np.percentile(one, 90)),
                          "us_pack8": float(np.median(p8)), "us_pack8_p10": float(np.percentile(p8, 10)),
                          "us_pack8_p90": float(np.percentile(p8, 90)), "samples": int(one.size),
                          "us_b2b": b2b, "launches": launches,
                          "tflops": fl / (med / 1e6) / 1e12, "tflops_b2b": fl / (b2b / 1e6) / 1e12}
        out[w.name] = rows
    out["protocol"] = (f"per arm {warmup} warm-ups, then {rounds} rounds x {samples} samples in each of two "
                       "directions (arm order rotated every sample; reversed in the second direction); pack 1 and "
                       "pack 8 each behind an L2 flush; median, p10, p90; C checked bit for bit before and after")
    return out


def run_fixups(sk, torch, dev, flush, stream, peak_tf, peak_gbs, l2_bytes):
    """Partial-tile merges compared on the skinny shape 512 x 512 x 65536 (many contributors per
    tile) and on the wave-quantized shape. Stream-K (hybrid rule on the wave-quantized shape):
    the owner waits and sums in k order, FP32 atomics, and the separate fixup pass (every
    partial to its slot, then a second launch sums each tile in k order), with 128 x 128 and
    256 x 256 pair tiles on 148 SMs, with one Stream-K group and with up to 8 groups
    (`/groupsG`: the first page's max_sk_groups_). On the skinny shape also Split-K in 16 FP32
    slabs, summed by the reduction pass or inside the launch, and the pass chain with
    `overlap = 2` (`/overlap2`: the steps' operands are independent; reported apart, as
    `best_deterministic_independent_operands`). Each entry is timed back to back
    (60 steps over rotating input sets of at least 4x the L2, behind a flush queued before the
    start event, as the headline) and one flushed launch at a time (median of 20)."""
    out = {}
    for w, mode in ((synth.SKINNY, sk.SK_STREAMK), (synth.WAVEQ, sk.SK_HYBRID)):
        A_bits, B_bits = synth.make_inputs(w)
        A = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        C = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
        set_bytes = A.numel() * 2 + B.numel() * 2 + C.numel() * 2
        n_sets = max(2, -(-4 * l2_bytes // set_bytes))
        sets = [(A, B, C)] + [(A.clone(), B.clone(), torch.empty_like(C)) for _ in range(n_sets - 1)]
        fl = 2.0 * w.M * w.N * w.K
        # The shape's roofline time: the larger of its tensor time at the measured peak and the
        # time to move A, B and C once at the measured HBM bandwidth.
        hbm_bytes = 2.0 * (w.M * w.K + w.K * w.N) + 2.0 * w.M * w.N
        bound_us = max(fl / (peak_tf * 1e12), hbm_bytes / (peak_gbs * 1e9)) * 1e6
        rows = {"roofline_us": bound_us}
        cases = []
        for (tile, tname), groups in itertools.product(((0, "128x128"), (2, "pair256x256")), (0, 8)):
            for name, part, red in (("owner", 0, sk.SK_DETERMINISTIC), ("atomic", 0, sk.SK_ATOMIC),
                                    ("pass", 1, sk.SK_DETERMINISTIC)):
                cases.append((tname, name, sk.schedule(mode, split_partials=part, tile=tile, sk_groups=groups,
                                                       overlap=1), red, groups))
        if w is synth.SKINNY:
            for tile, tname in ((2, "pair256x256"), (0, "128x128")):
                cases.append((tname, "splitk16_slabs_pass",
                              sk.schedule(sk.SK_SPLITK, 16, split_partials=1, tile=tile, overlap=1),
                              sk.SK_DETERMINISTIC, 0))
            cases.append(("pair256x256", "splitk16_slabs_in_launch",
                          sk.schedule(sk.SK_SPLITK, 16, split_partials=2, tile=2, overlap=1), sk.SK_DETERMINISTIC, 0))
            # The same chain when the steps' operands are independent (overlap = 2): the next
            # GEMM's first segments start while the reduction runs on the SMs this one leaves.
            cases.append(("pair256x256", "splitk16_slabs_pass/overlap2",
                          sk.schedule(sk.SK_SPLITK, 16, split_partials=1, tile=2, overlap=2), sk.SK_DETERMINISTIC, 0))
        best = best2 = None
        for tname, name, sch, red, groups in cases:
            plan = sk.sk_plan(w.M, w.N, w.K, 148, sch)
            contrib = plan[-sk.SK_MAP_TILE * int(plan[2]) + 1::sk.SK_MAP_TILE]
            gname = f"/groups{int(plan[17])}" if groups else ""
            nb = sk.sk_workspace_size(w.M, w.N, w.K, 148, sch, red)
            ws = torch.zeros(nb, dtype=torch.uint8, device=dev)

            def g(i):
                a, b, c = sets[i % n_sets]
                sk.sk_gemm(a, b, c, sk.SK_BF16, w.M, w.N, w.K, sk.SK_NN, sch, red, 148, ws, nb, stream)
            for i in range(5):
                g(i)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
            for a0, a1 in ev:
                flush.zero_()
                a0.record(stream)
                g(0)
                a1.record(stream)
            torch.cuda.synchronize(dev)
            flushed = float(np.median([a0.elapsed_time(a1) for a0, a1 in ev])) * 1e3
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush.zero_()
            b0.record(stream)
            for i in range(60):
                g(i)
            b1.record(stream)
            torch.cuda.synchronize(dev)
            assert sk.sk_status(ws, stream) == sk.SK_OK
            us = b0.elapsed_time(b1) * 1e3 / 60
            key = f"{tname}/{name}{gname}"
            rows[key] = {"us": us, "tflops": fl / (us / 1e6) / 1e12, "frac_of_roofline": bound_us / us,
                         "us_flushed": flushed, "launches": 2 if sch.split_partials == 1 else 1,
                         "max_contributors_per_tile": int(max(contrib)),
                         "deterministic": red == sk.SK_DETERMINISTIC}
            if red == sk.SK_DETERMINISTIC and sch.overlap == 1 and (best is None or us < rows[best]["us"]):
                best = key
            if red == sk.SK_DETERMINISTIC and (best2 is None or us < rows[best2]["us"]):
                best2 = key
        rows["best_deterministic"] = {"schedule": best, "us": rows[best]["us"],
                                      "frac_of_roofline": rows[best]["frac_of_roofline"]}
        rows["best_deterministic_independent_operands"] = {"schedule": best2, "us": rows[best2]["us"],
                                                           "frac_of_roofline": rows[best2]["frac_of_roofline"]}
        out[w.name] = rows
    return out


def run_raster(sk, torch, dev, flush, stream, peak_tf):
    """Tile-id order on the 8192^3 GEMM (A and B, 268 MB, exceed the 129 MB L2): data-parallel
    256 x 256 pair tiles on 148 SMs, along N or M, with and without swizzled strips; and the
    same GEMM as pure Stream-K (the hybrid rule keeps it data-parallel) with one and with up to
    8 Stream-K groups (`streamk/groupsG`: the first page's max_sk_groups_)."""
    w = synth.LARGE
    A_bits, B_bits = synth.make_inputs(w)
    A = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    C = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
    fl = 2.0 * w.M * w.N * w.K
    out = {}
    cases = [(f"{'along_n' if raster == 0 else 'along_m'}/swizzle{sw}", sk.schedule(sk.SK_DP, tile=2, raster=raster,
                                                                                      swizzle=sw))
             for raster, sw in ((0, 0), (0, 2), (0, 4), (0, 8), (0, 16), (1, 0), (1, 4), (1, 8))]
    for groups in (0, 8):
        sch = sk.schedule(sk.SK_STREAMK, tile=2, sk_groups=groups)
        used = int(sk.sk_plan(w.M, w.N, w.K, 148, sch)[17])
        cases.append((f"streamk/groups{used}", sch))
    for key, sch in cases:
        nb = sk.sk_workspace_size(w.M, w.N, w.K, 148, sch, sk.SK_DETERMINISTIC)
        ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
        g = lambda: sk.sk_gemm(A, B, C, sk.SK_BF16, w.M, w.N, w.K, sk.SK_NN, sch, sk.SK_DETERMINISTIC, 148, ws, nb, stream)
        for _ in range(3):
            g()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(15)]
        for a0, a1 in ev:
            flush.zero_()
            a0.record(stream)
            g()
            a1.record(stream)
        torch.cuda.synchronize(dev)
        assert sk.sk_status(ws, stream) == sk.SK_OK
        us = float(np.median([a0.elapsed_time(a1) for a0, a1 in ev])) * 1e3
        out[key] = {"us": us, "tflops": fl / (us / 1e6) / 1e12, "frac_of_measured_peak": fl / (us / 1e6) / 1e12 / peak_tf}
    return out


def run_experiments(sk, torch, dev, flush, stream, path):
    """The first page's "Try this" simulator experiments, timed on the GPU. M x 4096 x 4096
    with the 128 x 128 tile and the schedule built for 132 units (the page's H100 count):
    data-parallel, Split-K s = 2 and 4, Stream-K and the hybrid rule's choice. At M = 128
    also Split-K whose reduction is a second launch (slabs, s = 2, 4, 8), Split-K with the
    owner's fixup, and Stream-K with the owner's fixup and with the separate fixup pass.
    One JSON line per measurement; the cost model's makespans for the same shapes come
    from the schedule simulator, outside this run."""
    SMS, N, K = 132, 4096, 4096
    ms = list(range(128, 2049, 128)) + [2432, 2944, 4096]
    big = synth.Workload("mxk", max(ms), N, K, "NN", "normal_sqrtk", 7)
    A_bits, B_bits = synth.make_inputs(big)
    A_all = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).to(dev)

    def timed(m, sch):
        A = A_all[:m]
        C = torch.empty((m, N), dtype=torch.bfloat16, device=dev)
        nb = sk.sk_workspace_size(m, N, K, SMS, sch, sk.SK_DETERMINISTIC)
        ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
        g = lambda: sk.sk_gemm(A, B, C, sk.SK_BF16, m, N, K, sk.SK_NN, sch, sk.SK_DETERMINISTIC, SMS, ws, nb, stream)
        for _ in range(5):
            g()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(30)]
        for a0, a1 in ev:
            flush.zero_()
            a0.record(stream)
            g()
            a1.record(stream)
        torch.cuda.synchronize(dev)
        assert sk.sk_status(ws, stream) == sk.SK_OK
        plan = sk.sk_plan(m, N, K, SMS, sch)
        return float(np.median([a0.elapsed_time(a1) for a0, a1 in ev])) * 1e3, plan

    def line(f, **kw):
        f.write(json.dumps(kw) + "\n")
        f.flush()

    with open(path, "w") as f:
        for m in ms:
            for name, sch in (("data-parallel", sk.schedule(sk.SK_DP)), ("split-K s=2", sk.schedule(sk.SK_SPLITK, 2)),
                              ("split-K s=4", sk.schedule(sk.SK_SPLITK, 4)), ("stream-K", sk.schedule(sk.SK_STREAMK)),
                              ("rule", sk.schedule(sk.SK_HYBRID))):
                us, plan = timed(m, sch)
                line(f, experiment="rule_vs_four", M=m, N=N, K=K, num_sms=SMS, tile="128x128", schedule=name,
                     us=us, tiles=int(plan[2]), iters=int(plan[3]), resolved_mode=int(plan[1]), label=int(plan[9]),
                     sk_tiles=int(plan[5]), sk_units=int(plan[6]))
        m = 128
        cases = [(f"split-K s={s} separate reduction", sk.schedule(sk.SK_SPLITK, s, split_partials=1)) for s in (2, 4, 8)]
        cases += [(f"split-K s={s} owner fixup", sk.schedule(sk.SK_SPLITK, s)) for s in (2, 4, 8)]
        cases += [("stream-K owner fixup", sk.schedule(sk.SK_STREAMK)),
                  ("stream-K separate pass", sk.schedule(sk.SK_STREAMK, split_partials=1))]
        for name, sch in cases:
            us, plan = timed(m, sch)
            line(f, experiment="separate_reduction_m128", M=m, N=N, K=K, num_sms=SMS, tile="128x128", schedule=name,
                 us=us, launches=2 if "separate" in name else 1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="waveq", choices=sorted(WORKLOADS))
    ap.add_argument("--sms", type=int, default=148, help="SM count the schedule is built for (0 = device)")
    ap.add_argument("--mode", default="hybrid", choices=["dp", "splitk", "streamk", "hybrid"])
    ap.add_argument("--splits", type=int, default=2)
    ap.add_argument("--tile", type=int, default=2, choices=[0, 1, 2, 3],
                    help="work-tile shape: 0 = 128x128 (one CTA), 1 = 256x128 (CTA pair), "
                         "2 = 256x256 (CTA pair), 3 = 128x256 (one CTA)")
    ap.add_argument("--reduction", default="deterministic", choices=["deterministic", "atomic"])
    ap.add_argument("--raster", type=int, default=0, choices=[0, 1], help="tile ids along N (0) or M (1)")
    ap.add_argument("--swizzle", type=int, default=0, help="tile-id strips this many tiles deep (0: none)")
    ap.add_argument("--partials", type=int, default=0, choices=[0, 1, 2],
                    help="split_partials of the timed schedule (Split-K slabs; Stream-K/hybrid separate fixup pass)")
    ap.add_argument("--sk-groups", type=int, default=0, help="Stream-K groups of the timed schedule (0: one group)")
    ap.add_argument("--overlap", type=int, default=1, choices=[0, 1, 2],
                    help="launch each step overlapped with the one before it (programmatic dependent launch); "
                         "2: and load A and B before it completes (each step's operands are independent)")
    ap.add_argument("--timing", default="graph", choices=["graph", "stream", "flush"],
                    help="graph: the K steps' calls captured as one CUDA graph (outside the timed region) "
                         "and replayed once, back to back over rotating input sets of at least 4x the L2; "
                         "stream: the same K calls launched one by one; "
                         "flush: one event pair per step with a 256 MiB L2 flush before each")
    ap.add_argument("--no-extras", action="store_true", help="skip the schedule table, e2e and CPU baseline")
    ap.add_argument("--ref-seconds", type=float, default=10.0)
    ap.add_argument("--sweep", default="", help="also write the tile-count sweep (JSON lines) to this file")
    ap.add_argument("--experiments", default="",
                    help="also write the simulator experiments timed on the GPU (JSON lines) to this file")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank, world, local = dist_info()
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import torch
    import torch.distributed as dist

    import gemm_work_decomposition_gb300 as sk
    from gemm_work_decomposition_gb300 import build as skbuild

    skbuild.build()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    props = torch.cuda.get_device_properties(dev)
    dev_sms = props.multi_processor_count
    sms = args.sms if args.sms > 0 else dev_sms
    peaks, peaks_src = load_peaks()
    peak_tf = float(peaks["bf16_tflops"])

    modes = {"dp": sk.SK_DP, "splitk": sk.SK_SPLITK, "streamk": sk.SK_STREAMK, "hybrid": sk.SK_HYBRID}
    red = sk.SK_DETERMINISTIC if args.reduction == "deterministic" else sk.SK_ATOMIC
    out_code = sk.SK_BF16 if w.out == "bf16" else sk.SK_F32
    lay = sk.SK_NN if w.layout == "NN" else sk.SK_NT
    flops = 2.0 * w.M * w.N * w.K

    # Inputs, copied once into HBM. On several devices the job is one GEMM with world * M rows,
    # split by rows (B replicated, output tiles independent, so no collective): this rank
    # generates its row block of A and the whole B.
    wg = sharded_workload(w, world) if world > 1 else w
    r0, rows = m_shard(wg.M, world, rank)
    assert rows == w.M
    A_bits, B_bits = synth.make_row_block(wg, r0, r0 + rows)
    A_host = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    B_host = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    A = A_host.to(dev)
    B = B_host.to(dev)
    cdt = torch.bfloat16 if w.out == "bf16" else torch.float32
    C = torch.empty((w.M, w.N), dtype=cdt, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # Rotating input sets for back-to-back timing: enough copies of A, B and C that one pass
    # over them is at least 4x the L2, so every step finds its operands in HBM, not in L2.
    l2_bytes = int(getattr(props, "L2_cache_size", 0) or (129 << 20))
    set_bytes = A.numel() * 2 + B.numel() * 2 + C.numel() * C.element_size()
    n_sets = max(2, -(-4 * l2_bytes // set_bytes))
    sets = [(A, B, C)] + [(A.clone(), B.clone(), torch.empty_like(C)) for _ in range(n_sets - 1)]

    def make(mode_name, nsms, splits=1, tile=args.tile, raster=args.raster, swizzle=args.swizzle, overlap=0,
             groups=args.sk_groups):
        sch = sk.schedule(modes[mode_name], splits if mode_name == "splitk" else 1, tile=tile, raster=raster,
                          swizzle=swizzle, overlap=overlap, sk_groups=groups)
        nb = sk.sk_workspace_size(w.M, w.N, w.K, nsms, sch, red)
        ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
        return sch, ws, nb

    def timed(sch, ws, nb, nsms, steps, warmup):
        for _ in range(warmup):
            sk.sk_gemm(A, B, C, out_code, w.M, w.N, w.K, lay, sch, red, nsms, ws, nb, stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize(dev)
        for s, e in ev:
            flush.zero_()
            s.record(stream)
            sk.sk_gemm(A, B, C, out_code, w.M, w.N, w.K, lay, sch, red, nsms, ws, nb, stream)
            e.record(stream)
        torch.cuda.synchronize(dev)
        st = sk.sk_status(ws, stream)
        if st != sk.SK_OK:
            raise RuntimeError(f"device status {sk.sk_strerror(st)}")
        return np.array([s.elapsed_time(e) for s, e in ev])  # ms

    # Device addresses of the rotating sets and the stream handle, taken once: the public entry
    # point accepts plain integers, which keeps the host's per-step enqueue short.
    set_ptrs = [(a_.data_ptr(), b_.data_ptr(), c_.data_ptr()) for a_, b_, c_ in sets]
    stream_h = stream.cuda_stream

    def launch_set(i, sch, ws, nb, nsms):
        a_, b_, c_ = set_ptrs[i % n_sets]
        sk.sk_gemm(a_, b_, c_, out_code, w.M, w.N, w.K, lay, sch, red, nsms, ws if isinstance(ws, int) else ws.data_ptr(),
                   nb, stream_h)

    def stream_timed(sch, ws, nb, nsms, steps, warmup):
        """Mean ms per step of `steps` launches back to back over the rotating sets."""
        for i in range(warmup):
            launch_set(i, sch, ws, nb, nsms)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        t0.record(stream)
        for i in range(steps):
            launch_set(i, sch, ws, nb, nsms)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        st = sk.sk_status(ws, stream)
        if st != sk.SK_OK:
            raise RuntimeError(f"device status {sk.sk_strerror(st)}")
        return t0.elapsed_time(t1) / steps

    sch, ws, nb = make(args.mode, sms, args.splits, overlap=args.overlap)
    if args.partials:
        sch = sk.schedule(modes[args.mode], args.splits if args.mode == "splitk" else 1, split_partials=args.partials,
                          tile=args.tile, raster=args.raster, swizzle=args.swizzle, overlap=args.overlap,
                          sk_groups=args.sk_groups)
        nb = sk.sk_workspace_size(w.M, w.N, w.K, sms, sch, red)
        ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    plan = sk.sk_plan(w.M, w.N, w.K, sms, sch)
    # One persistent GEMM kernel per step, plus the reduction or fixup pass when partials are
    # summed in a second launch.
    launches_per_step = 2 if args.partials == 1 else 1

    # ---- the K steps as one CUDA graph (--timing graph): the same K public-API calls, captured
    # on a side stream and uploaded to the device before the timed region, then replayed once
    # inside it. The graph keeps each launch's programmatic dependency on the one before it.
    graph = None
    if args.timing == "graph":
        cap = torch.cuda.Stream(dev)
        cap_h = cap.cuda_stream
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(graph, stream=cap):
            for i in range(args.steps):
                a_, b_, c_ = set_ptrs[i % n_sets]
                sk.sk_gemm(a_, b_, c_, out_code, w.M, w.N, w.K, lay, sch, red, sms, ws.data_ptr(), nb, cap_h)
        graph_upload(graph, stream)
        torch.cuda.synchronize(dev)

    # ---- the timed region: K steps, barrier + synchronize on both sides. The clock sampler
    # starts first (starting nvidia-smi takes a while), so the warm-up steps run right before
    # the region and the GPU does not sit idle between them.
    clocks = ClockSampler(f"GPU-{props.uuid}")
    clocks.start()
    if world > 1:
        dist.barrier()
    for i in range(args.warmup):
        launch_set(i, sch, ws, nb, sms)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    wall0 = time.perf_counter()
    if args.timing in ("stream", "graph"):
        # One event pair around K launches back to back; step i uses input set i mod n_sets.
        # The L2 flush queued ahead of the start event keeps the device busy while the host
        # enqueues the event and the K steps, so the start stamp is not taken on an idle
        # device before the first step has even been submitted.
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))]
        flush.zero_()
        ev[0][0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                launch_set(i, sch, ws, nb, sms)
        enqueue_s = time.perf_counter() - wall0
        ev[0][1].record(stream)
    else:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for s, e in ev:
            flush.zero_()
            s.record(stream)
            sk.sk_gemm(A, B, C, out_code, w.M, w.N, w.K, lay, sch, red, sms, ws, nb, stream)
            e.record(stream)
        enqueue_s = time.perf_counter() - wall0
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks.stop()
    status = sk.sk_status(ws, stream)
    if status != sk.SK_OK:
        raise RuntimeError(f"device status {sk.sk_strerror(status)}")
    step_ms = np.array([s.elapsed_time(e) for s, e in ev])
    if red == sk.SK_DETERMINISTIC and args.timing != "flush":  # every set's C is the same, bit for bit
        for _, _, c_ in sets[1:min(n_sets, max(args.warmup, args.steps))]:
            assert torch.equal(c_, C)
    total_ms = max_over_ranks(float(step_ms.sum()), dist if world > 1 else None, dev)
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, flops, args.steps, total_ms)
    kernel_tflops = flops / (ms_per_step / 1e3) / 1e12

    extras = {}
    if args.timing == "graph" and rank == 0:
        # ---- the same K steps launched one call at a time (no graph), timed the same way
        for i in range(args.warmup):
            launch_set(i, sch, ws, nb, sms)
        torch.cuda.synchronize(dev)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        s0.record(stream)
        for i in range(args.steps):
            launch_set(i, sch, ws, nb, sms)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        sms_ = s0.elapsed_time(s1) / args.steps
        extras["stream_launches"] = {"ms_per_step": sms_, "tflops": flops / (sms_ / 1e3) / 1e12,
                                     "frac_of_measured_peak": flops / (sms_ / 1e3) / 1e12 / peak_tf,
                                     "how": "the timed region's K steps launched one sk_gemm call at a time"}
        if args.overlap == 1:
            # ---- the same K steps with overlap = 2: each step's A and B are independent of the
            # step before, so its first segments may load and multiply before that step ends
            sch2 = sk.schedule(sch.mode, sch.splits, sch.units, sch.min_iters, sch.split_partials, sch.tile,
                               sch.raster, sch.swizzle, 2, sch.sk_groups)
            C_ref = C.clone()
            g2 = torch.cuda.CUDAGraph()
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g2, stream=cap):
                for i in range(args.steps):
                    a_, b_, c_ = set_ptrs[i % n_sets]
                    sk.sk_gemm(a_, b_, c_, out_code, w.M, w.N, w.K, lay, sch2, red, sms, ws.data_ptr(), nb, cap_h)
            graph_upload(g2, stream)
            for i in range(args.warmup):
                launch_set(i, sch2, ws, nb, sms)
            torch.cuda.synchronize(dev)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush.zero_()
            s0.record(stream)
            g2.replay()
            s1.record(stream)
            torch.cuda.synchronize(dev)
            if sk.sk_status(ws, stream) != sk.SK_OK:
                raise RuntimeError("device status after the overlap = 2 steps")
            if red == sk.SK_DETERMINISTIC:  # the same bits as the overlap = 1 steps
                for _, _, c_ in sets[:min(n_sets, args.steps)]:
                    assert torch.equal(c_, C_ref)
            ms2 = s0.elapsed_time(s1) / args.steps
            extras["independent_operands"] = {
                "ms_per_step": ms2, "tflops": flops / (ms2 / 1e3) / 1e12,
                "frac_of_measured_peak": flops / (ms2 / 1e3) / 1e12 / peak_tf,
                "how": "the timed region's K steps with sk_schedule.overlap = 2 (each step's A and B are not written "
                       "by the step before, so its first segments' loads and MMAs start before that step completes; "
                       "stores still wait), one CUDA graph, timed the same way"}
            del g2
    if not args.no_extras and rank == 0:
        # ---- per-schedule table (the metric is per schedule)
        table = {}
        tile_names = {0: "128x128", 1: "pair256x128", 2: "pair256x256", 3: "128x256"}
        for tile, name, nsms in ((0, "dp", 148), (0, "splitk2", 148), (0, "streamk", 148), (0, "hybrid", 148),
                                 (0, "dp", dev_sms), (0, "hybrid", dev_sms),
                                 (2, "dp", 148), (2, "splitk2", 148), (2, "streamk", 148), (2, "hybrid", 148),
                                 (2, "dp", dev_sms), (2, "hybrid", dev_sms),
                                 (3, "hybrid", 148), (1, "hybrid", 148)):
            mname = "splitk" if name.startswith("splitk") else name
            s2, ws2, nb2 = make(mname, nsms, 2, tile)
            t = timed(s2, ws2, nb2, nsms, 200, 10)
            med = float(np.median(t))
            table[f"{tile_names[tile]}/{name}@{nsms}"] = {"us_median": med * 1e3, "us_p10": float(np.percentile(t, 10)) * 1e3,
                                       "us_p90": float(np.percentile(t, 90)) * 1e3,
                                       "tflops": flops / (med / 1e3) / 1e12,
                                       "frac_of_measured_peak": flops / (med / 1e3) / 1e12 / peak_tf,
                                       "frac_of_nominal_peak": flops / (med / 1e3) / 1e12 / NOMINAL_BF16_TFLOPS}
        extras["schedules"] = table

        # ---- the same launches back to back over the rotating sets, without and with the
        # overlapped launch (1), and with operand loads ahead of the previous step (2, the
        # steps' operands being independent): what a stream of GEMMs pays per step beyond the
        # kernel itself.
        b2b = {}
        for tile, name, nsms in ((2, "hybrid", 148), (2, "dp", 148), (2, "streamk", 148), (0, "hybrid", 148),
                                 (0, "dp", 148), (2, "hybrid", dev_sms)):
            mname = "splitk" if name.startswith("splitk") else name
            row = {}
            for ov in (0, 1, 2):
                s2, ws2, nb2 = make(mname, nsms, 2, tile, overlap=ov)
                ms = stream_timed(s2, ws2, nb2, nsms, 400, 24)
                row[f"overlap{ov}"] = {"us": ms * 1e3, "tflops": flops / (ms / 1e3) / 1e12,
                                       "frac_of_measured_peak": flops / (ms / 1e3) / 1e12 / peak_tf}
            b2b[f"{tile_names[tile]}/{name}@{nsms}"] = row
        extras["back_to_back"] = {"sets": n_sets, "set_mb": set_bytes / 1e6, "steps": 400, "table": b2b}

        # ---- the library GEMM on the same shape, output type and rotating sets (context only)
        if out_code == sk.SK_BF16:
            t, tb = library_timed(torch, dev, flush, stream, sets, w.M, w.N, nt=lay == sk.SK_NT, b2b=400)
            extras["library_gemm"] = {"what": "torch.matmul (cuBLAS), BF16 out",
                                      "us_b2b": tb * 1e3, "tflops_b2b": flops / (tb / 1e3) / 1e12,
                                      "frac_of_measured_peak_b2b": flops / (tb / 1e3) / 1e12 / peak_tf,
                                      "us_isolated_median": t * 1e3, "tflops_isolated": flops / (t / 1e3) / 1e12}

        # ---- the headline schedule timed one launch at a time, L2 flushed before each
        iso = timed(sch, ws, nb, sms, 200, 10)
        extras["isolated_launch"] = {"us_median": float(np.median(iso)) * 1e3, "us_mean": float(iso.mean()) * 1e3,
                                     "tflops_median": flops / (float(np.median(iso)) / 1e3) / 1e12,
                                     "how": "one event pair per launch, 256 MiB L2 flush before each; includes the "
                                            "launch latency that back-to-back steps hide"}

        # ---- tail-wave idle SM-time from one traced launch each (outside the timed region):
        # sum over SMs of (last SM's end - this SM's end), DP against the headline schedule.
        def idle(mode_name, nsms, tile):
            s3, ws3, nb3 = make(mode_name, nsms, 2, tile)
            plan3 = sk.sk_plan(w.M, w.N, w.K, nsms, s3)
            ncta = int(plan3[4]) * int(plan3[14])
            tr = torch.zeros(ncta * sk.SK_TRACE_WORDS, dtype=torch.int64, device=dev)
            vals = []
            for _ in range(5):
                flush.zero_()
                sk.sk_gemm_debug(A, B, C, out_code, w.M, w.N, w.K, lay, s3, red, nsms, ws3, nb3, stream, trace=tr)
                torch.cuda.synchronize(dev)
                T = tr.cpu().numpy().reshape(ncta, sk.SK_TRACE_WORDS).astype(np.int64)
                # A CTA ends no earlier than any stamp it wrote: the compiler may schedule a
                # %globaltimer read ahead of the exit barrier, so the exit stamp alone can read early.
                nseg = np.minimum(T[:, 2], sk.SK_TRACE_SEGS).astype(np.int64)
                last = np.array([T[c, 4:4 + 4 * nseg[c]].max(initial=0) for c in range(ncta)])
                end = (np.maximum(T[:, 1], last) - T[:, 0].min()) / 1e3
                # SMs without a CTA idle for the whole span
                vals.append((float(np.sum(end.max() - end)) + (dev_sms - ncta) * float(end.max()), float(end.max())))
            assert sk.sk_status(ws3, stream) == sk.SK_OK
            v = sorted(vals)[len(vals) // 2]
            return {"tail_idle_sm_us": v[0], "span_us": v[1], "ctas": ncta}
        dp_idle = idle("dp", sms, args.tile)
        hd_idle = idle(args.mode, sms, args.tile)
        # ---- timeline of two consecutive launches inside a back-to-back run of the timed
        # schedule (launches 20 and 21 over the rotating sets), with and without the
        # overlapped launch: the gap between launches, the cold start, and how the units' ends
        # spread after their last MMA (the epilogue work each unit has left).
        def b2b_timeline(ov):
            s4 = sk.schedule(modes[args.mode], args.splits if args.mode == "splitk" else 1, units=0,
                             split_partials=args.partials, tile=args.tile, raster=args.raster, swizzle=args.swizzle,
                             overlap=ov, sk_groups=args.sk_groups)
            nb4 = sk.sk_workspace_size(w.M, w.N, w.K, sms, s4, red)
            ws4 = torch.zeros(nb4, dtype=torch.uint8, device=dev)
            plan4 = sk.sk_plan(w.M, w.N, w.K, sms, s4)
            cg = int(plan4[14])
            ncta = int(plan4[4]) * cg
            trs = [torch.zeros(ncta * sk.SK_TRACE_WORDS, dtype=torch.int64, device=dev) for _ in range(2)]
            torch.cuda.synchronize(dev)
            for i in range(24):
                a_, b_, c_ = sets[i % n_sets]
                if i in (20, 21):
                    sk.sk_gemm_debug(a_, b_, c_, out_code, w.M, w.N, w.K, lay, s4, red, sms, ws4, nb4, stream,
                                     trace=trs[i - 20])
                else:
                    sk.sk_gemm(a_, b_, c_, out_code, w.M, w.N, w.K, lay, s4, red, sms, ws4, nb4, stream)
            torch.cuda.synchronize(dev)
            assert sk.sk_status(ws4, stream) == sk.SK_OK
            segs = {}
            for i in range(int(plan4[7])):
                r = plan4[sk.SK_MAP_HEADER + sk.SK_MAP_SEG * i: sk.SK_MAP_HEADER + sk.SK_MAP_SEG * (i + 1)]
                segs.setdefault(int(r[0]), []).append((int(r[1]), "FOPS"[int(r[5])] + str(int(r[4]) - int(r[3]))))
            out = []
            for tr in trs:
                T = tr.cpu().numpy().reshape(ncta, sk.SK_TRACE_WORDS).astype(np.int64)
                nseg = np.minimum(T[:, 2], sk.SK_TRACE_SEGS)
                st = [T[c, 4:4 + 4 * nseg[c]].reshape(-1, 4) for c in range(ncta)]
                end = np.array([max(T[c, 1], st[c].max(initial=0)) for c in range(ncta)])
                lead = [c for c in range(ncta) if c % cg == 0 and nseg[c] > 0]
                first = np.array([st[c][0, 0] - T[c, 0] for c in lead]) / 1e3
                commit = np.array([st[c][-1, 1] for c in lead])
                tail = np.array([end[c] - st[c][-1, 1] for c in lead]) / 1e3
                late = sorted(lead, key=lambda c: -end[c])[:3]
                span = np.maximum(T[:, 1] - T[:, 0], 1)
                out.append({"start": int(T[:, 0].min()), "end": int(end.max()),
                            # SM clock while each CTA ran (its cycle count over its span): under a
                            # full tensor load it sits below the clock nvidia-smi samples report.
                            "sm_clock_mhz_in_kernel_median": float(np.median(T[:, 3] / span * 1e3)),
                            "first_mma_after_start_us_median": float(np.median(first)),
                            "last_commit_spread_us": float((commit.max() - commit.min()) / 1e3),
                            "end_spread_us": float((end.max() - end.min()) / 1e3),
                            "end_after_last_commit_us": {"median": float(np.median(tail)), "max": float(tail.max())},
                            "latest_units": [" ".join(s for _, s in sorted(segs.get(c // cg, []))) for c in late]})
            return {"overlap": ov, "gap_between_launches_us": (out[1]["start"] - out[0]["end"]) / 1e3,
                    "launch": [{k: v for k, v in o.items() if k not in ("start", "end")} for o in out]}
        extras["b2b_timeline"] = [b2b_timeline(1), b2b_timeline(0)]

        extras["tail_idle"] = {"dp": dp_idle, args.mode: hd_idle,
                               "dp_over_schedule": dp_idle["tail_idle_sm_us"] / max(1e-9, hd_idle["tail_idle_sm_us"]),
                               "definition": "sum over the device's SMs of (kernel end - SM end), per-CTA globaltimer"}

        # ---- e2e: host buffers, copies inside the timed region, through the C ABI's host-buffer
        # call (sk_gemm_host). Every step copies its A and B from pinned host memory into a
        # device staging set and its C back. Pipelined (depth 2): step i+1's uploads and step
        # i-1's download run on two copy streams while step i's GEMM runs, over two staging
        # sets. Timed by device events on the GEMM stream around the one call (the call makes
        # that stream wait for the last download). The serial chain (depth 1, everything on one
        # stream) is reported beside it.
        n_e2e = max(10, min(200, args.steps))
        h2d_bytes = int(A.numel() * 2 + B.numel() * 2)
        d2h_bytes = int(C.numel() * C.element_size())
        C_host = [torch.empty((w.M, w.N), dtype=cdt).pin_memory() for _ in range(2)]
        stage = {d: sk.sk_host_staging_size(w.M, w.N, w.K, out_code, d) for d in (1, 2)}
        staging = torch.empty(stage[2], dtype=torch.uint8, device=dev)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_host(n, depth):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            sk.sk_gemm_host([A_host] * n, [B_host] * n, [C_host[i % 2] for i in range(n)], out_code, w.M, w.N, w.K,
                            lay, sch, red, sms, staging, stage[depth], depth, ws, nb, stream,
                            s_in if depth == 2 else None, s_out if depth == 2 else None)
            t1.record(stream)
            torch.cuda.synchronize(dev)
            return t0.elapsed_time(t1) / n

        e2e_host(3, 2)
        e2e_host(3, 1)
        pipe_ms = e2e_host(n_e2e, 2)
        if red == sk.SK_DETERMINISTIC:  # the last step's result matches the timed kernel's, bit for bit
            assert torch.equal(C_host[(n_e2e - 1) % 2], C.cpu())
        serial_ms = e2e_host(n_e2e, 1)
        extras["e2e"] = {"value": flops / (pipe_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                         "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "ms_per_step": pipe_ms,
                         "steps": n_e2e,
                         "how": "sk_gemm_host over pinned host buffers, depth 2: A and B uploads on one copy stream "
                                "and the C download on another overlap the GEMM of the neighbouring steps; device "
                                "events on the GEMM stream around the call",
                         "h2d_plus_d2h_gbs": (h2d_bytes + d2h_bytes) / (pipe_ms / 1e3) / 1e9,
                         "serial": {"value": flops / (serial_ms / 1e3) / 1e12, "ms_per_step": serial_ms,
                                    "how": "sk_gemm_host, depth 1: every copy and GEMM in order on one stream"}}
        assert sk.sk_status(ws, stream) == sk.SK_OK

        # ---- CPU oracle baseline on a bounded sample
        cpu_v, cpu_s, cpu_n, cpu_rows = cpu_oracle_sample(w, args.ref_seconds)
        extras["cpu_baseline"] = {"value": cpu_v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                                  "sample": f"{cpu_n} x FP64 GEMM of {cpu_rows} rows x {w.N} x {w.K} "
                                            f"({cpu_s:.1f} s, numpy matmul, default BLAS threads)"}

        extras["smallm_nt"] = run_smallm(sk, torch, dev, flush, stream, dev_sms)
        extras["fixups"] = run_fixups(sk, torch, dev, flush, stream, peak_tf, float(peaks["hbm_gbs"]), l2_bytes)
        extras["raster_8192"] = run_raster(sk, torch, dev, flush, stream, peak_tf)
        extras["sweep"] = run_sweep_compact(sk, torch, dev, red, flush, stream, peak_tf, l2_bytes)
    if rank == 0 and args.sweep:
        run_sweep(sk, torch, dev, args.sweep, red, flush, stream, peak_tf, dev_sms, l2_bytes)
    if rank == 0 and args.experiments:
        run_experiments(sk, torch, dev, flush, stream, args.experiments)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    sha = kernel_sha()
    order = "" if (args.raster, args.swizzle) in ((0, 0), (0, 1)) else f"/r{args.raster}s{args.swizzle}"
    split = f"/s{args.splits}p{args.partials}" if args.mode == "splitk" else ""
    tr = TRAFFIC.get(f"{w.name}/{args.mode}{split}/tile{args.tile}@{sms}{order}")
    traffic = tr["bytes"] if tr and tr.get("kernel_sha") == sha else None
    # The roofline that bounds the step: the tensor time of 2MNK at the measured BF16 peak, or
    # (long-K shapes such as 512 x 512 x 65536) the time to read A and B and write C once at the
    # measured HBM bandwidth, whichever is longer.
    hbm_gbs = float(peaks["hbm_gbs"])
    algo_bytes = 2.0 * (w.M * w.K + w.K * w.N) + (2.0 if w.out == "bf16" else 4.0) * w.M * w.N
    kernel_name = "sk_gemm_kernel" + (" + its second launch" if launches_per_step == 2 else "")
    if algo_bytes / (hbm_gbs * 1e9) > flops / (peak_tf * 1e12):
        achieved_gbs = algo_bytes / (ms_per_step / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_gbs, "unit": "GB/s",
                    "frac": achieved_gbs / hbm_gbs, "traffic": traffic, "algorithmic_bytes": algo_bytes,
                    "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved_gbs / NOMINAL_HBM_GBS,
                    "peak_source": f"{peaks_src} HBM copy", "kernel": kernel_name,
                    "tflops": kernel_tflops, "frac_of_bf16_peak": kernel_tflops / peak_tf}
    else:
        roofline = {"bound": "tensor", "achieved": kernel_tflops, "peak": peak_tf, "unit": "TFLOP/s",
                    "frac": kernel_tflops / peak_tf, "traffic": traffic,
                    "nominal_peak": NOMINAL_BF16_TFLOPS, "frac_of_nominal": kernel_tflops / NOMINAL_BF16_TFLOPS,
                    "peak_source": f"{peaks_src} bf16 burst", "kernel": kernel_name}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**schedule_config(args, w, plan, sms), "device_sms": dev_sms,
                   "overlap": args.overlap, "timing": args.timing,
                   "parallelism": (f"M-split over {world} GPUs: one {wg.M} x {w.N} x {w.K} GEMM, {rows} rows of A and C "
                                   f"per GPU, B replicated, no collective" if world > 1 else "one GPU"),
                   "l2": (f"inputs larger than L2: {n_sets} rotating sets of A, B and C ({n_sets * set_bytes / 1e6:.0f} MB, "
                          f">= 4x the {l2_bytes / 1e6:.0f} MB L2), launched back to back"
                          if args.timing != "flush" else "flushed between timed steps (256 MiB write)"),
                   "launch": ({"graph": "the K steps' sk_gemm calls captured as one CUDA graph before the timed region "
                                        "(uploaded there) and replayed once inside it; a 256 MiB L2 flush queued "
                                        "before the start event covers the host's enqueue",
                               "stream": "K sk_gemm calls launched one by one inside the timed region, behind a "
                                         "256 MiB L2 flush queued before the start event",
                               "flush": "one sk_gemm call per event pair"}[args.timing]),
                   "accumulate": "fp32"},
        "roofline": roofline,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks.summary(),
        "wall_s_timed_region": wall,
        "host_enqueue_us_per_step": enqueue_s / args.steps * 1e6,
    }
    line.update(extras)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
