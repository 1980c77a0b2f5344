"""Benchmark of the weight-delta hot path: whole-model encode + apply.

Default workload: the Llama-3-8B-shaped tensor set (291 tensors,
8,030,261,248 FP32 master params, N(0, 0.02) weights, RMSNorm 1 + N(0, 0.01)),
one Adam-sized step eta = 3e-6, synthetic data drawn on the device.

One step = pulse_encode_multi (FP32 -> BF16 RNE, bitwise compare,
order-preserving compaction, prev refresh) + pulse_apply_multi_device
(scatter into the sampler's BF16 weights), one launch each over the whole
model. Before every step prev and the sampler weights are restored from a
pristine copy (untimed), so every timed step encodes the same real update.
Inputs (48 GB) are far larger than L2 (129 MB), so no L2 flush is needed;
a workload whose buffers fit in a few L2s (the single 2^20 tensor) gets a
1 GiB scratch write after the restore, before every step.

Printed: one JSON line with params/s (value), the roofline of the encode
kernel against measured HBM copy bandwidth, the same step at eta = 3e-7
(about 1 % of the view changed, the pages' steady state), the XOR-mask path, the MXFP8,
MXFP4 and NVFP4 serving views of the same step (their own encode + apply),
the sidecar catch-up legs, index packing, PULSELoCo, an end-to-end number
through host buffers, the CPU oracle baseline, and the SM clocks sampled
during the timed region. The flat 2^28 workload (--config 4) adds the
encode + apply cost at every update scale of the density sweep.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "encode+apply params/s"
UNIT = "params/s"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1024 * 1024
FLUSH_BYTES = 1024 * 1024 * 1024
SPARSE_ETA = 3e-7
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "encode_traffic.json")
ENCODE_SRCS = [os.path.join(ROOT, "rl_post_trainer_gb300", "csrc", f)
               for f in ("encode.cu", "encode_common.cuh", "pulse_device.cuh")]
# the encode kernel's part of the internal header: everything before this line
INTERNAL_H = os.path.join(ROOT, "rl_post_trainer_gb300", "csrc", "pulse_internal.h")
INTERNAL_H_ENCODE_END = b"// ------------------------------------------------------- MX view encode"


# ------------------------------------------------------------- utilities

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def encode_source_hash() -> str:
    """sha256 over the encode kernel's sources, in a fixed order (the shared
    internal header up to its encode section's end only)."""
    h = hashlib.sha256()
    for path in ENCODE_SRCS:
        with open(path, "rb") as f:
            h.update(f.read())
    with open(INTERNAL_H, "rb") as f:
        h.update(f.read().split(INTERNAL_H_ENCODE_END)[0])
    return h.hexdigest()


def profiled_traffic():
    """DRAM bytes per whole-model encode launch (profiles/encode_traffic.json,
    written by --record-traffic from an ncu capture), if the encode sources
    are unchanged since that capture; else None."""
    try:
        with open(TRAFFIC_JSON, encoding="utf-8") as f:
            rec = json.load(f)
        if rec.get("source_sha256") != encode_source_hash():
            return None
        return float(rec["traffic_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        return None


def record_traffic(csv_path: str, captured_config: int, target_config: int = 3) -> dict:
    """Reads an ncu CSV (--metrics dram__bytes_read.sum,dram__bytes_write.sum)
    of encode_kernel launches on a smaller workload, scales the mean traffic
    per launch to the target workload by its element count (the same weight
    distribution and update scale, so the changed fraction and the touched
    sectors grow in proportion), and writes profiles/encode_traffic.json."""
    import csv
    per_launch = {}
    with open(csv_path, newline="", encoding="utf-8") as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(lines):
        if "encode_kernel" not in row.get("Kernel Name", ""):
            continue
        name = row.get("Metric Name", "")
        if name in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            unit = row.get("Metric Unit", "byte")
            scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(unit, 1.0)
            val = float(row["Metric Value"].replace(",", "")) * scale
            per_launch.setdefault(row["ID"], {})[name] = val
    totals = [d["dram__bytes_read.sum"] + d["dram__bytes_write.sum"] for d in per_launch.values()
              if len(d) == 2]
    if not totals:
        raise SystemExit(f"no encode_kernel DRAM counters in {csv_path}")
    cap_cfg = workloads.CONFIGS[captured_config]
    tgt_cfg = workloads.CONFIGS[target_config]
    n_cap = workloads.total_params(cap_cfg["specs"]())
    n_tgt = workloads.total_params(tgt_cfg["specs"]())
    mean = float(np.mean(totals))
    rec = {
        "kernel": "encode_kernel<multi>",
        "traffic_bytes_per_launch": mean * n_tgt / n_cap,
        "workload": tgt_cfg["name"],
        "captured": {"workload": cap_cfg["name"], "params": n_cap, "launches": len(totals),
                     "dram_bytes_per_launch": mean},
        "scaling": f"x {n_tgt} / {n_cap} elements (same distributions and update scale)",
        "source_sha256": encode_source_hash(),
        "csv": os.path.basename(csv_path),
    }
    with open(TRAFFIC_JSON, "w", encoding="utf-8") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() in ("active", "1"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# -------------------------------------------------------------- workload

class Workload:
    """Device buffers of one model: trainer (master, prev), sampler (w),
    patch segments, XOR buffers, and a pristine copy of the initial view."""

    def __init__(self, specs, seed, eta, dev, xor=True):
        import rl_post_trainer_gb300 as pulse
        self.specs = specs
        self.n = workloads.total_params(specs)
        pairs = workloads.torch_model(specs, seed, eta, dev)
        self.master = [m for m, _ in pairs]
        self.prev0 = [p for _, p in pairs]
        self.prev = [p.clone() for p in self.prev0]
        self.w = [p.clone() for p in self.prev0]
        self.idx = [torch.empty(s.numel, dtype=torch.int32, device=dev) for s in specs]
        self.val = [torch.empty(s.numel, dtype=torch.int16, device=dev) for s in specs]
        self.plan = pulse.Plan([pulse.TensorSlot(s.numel, master=self.master[i], prev=self.prev[i],
                                                 w=self.w[i], idx=self.idx[i], val=self.val[i])
                                for i, s in enumerate(specs)])
        self.counts = torch.zeros(len(specs), dtype=torch.int64, device=dev)
        self.xor = xor
        if xor:
            self.prev_x = [p.clone() for p in self.prev0]
            self.w_x = [p.clone() for p in self.prev0]
            self.mask = [torch.empty(s.numel, dtype=torch.int16, device=dev) for s in specs]
            self.xplan = pulse.Plan([pulse.TensorSlot(s.numel, master=self.master[i],
                                                      prev=self.prev_x[i], w=self.w_x[i],
                                                      mask=self.mask[i])
                                     for i, s in enumerate(specs)])

    def release_views(self):
        """Drop the BF16 views and the BF16 plan (legs that only need the
        FP32 masters and the index buffers run after this)."""
        self.plan.close()
        self.prev = self.prev0 = self.w = []
        torch.cuda.empty_cache()

    def restore(self):
        for p, w, p0 in zip(self.prev, self.w, self.prev0):
            p.copy_(p0)
            w.copy_(p0)

    def restore_xor(self):
        for p, w, p0 in zip(self.prev_x, self.w_x, self.prev0):
            p.copy_(p0)
            w.copy_(p0)

    def sectors_touched(self, counts_np) -> int:
        """Distinct 32-byte sectors of the BF16 arrays holding a changed element
        (buffers are 512-byte aligned, so sector = index // 16)."""
        total = 0
        for t, k in enumerate(counts_np):
            k = int(k)
            if k == 0:
                continue
            s = self.idx[t][:k].to(torch.int64) // 16
            total += 1 + int((s[1:] != s[:-1]).sum().item())
        return total


def barrier(dist_on):
    if dist_on:
        torch.distributed.barrier()


def _reduce(x: float, op, dist_on) -> float:
    if not dist_on:
        return x
    on_gpu = torch.distributed.get_backend() == "nccl"
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    torch.distributed.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(x: float, dist_on) -> float:
    """Slowest rank's time: the job is done when every rank is done."""
    return _reduce(x, torch.distributed.ReduceOp.MAX if dist_on else None, dist_on)


def sum_over_ranks(x: float, dist_on) -> float:
    """Work of all ranks (weak scaling: each rank runs its own model replica)."""
    return _reduce(x, torch.distributed.ReduceOp.SUM if dist_on else None, dist_on)


# ------------------------------------------------------------ CPU oracle

def oracle_sample(specs, seed, eta, max_params, dev):
    """First tensors of the model (list order) up to max_params, host copies
    of (master, prev0) drawn with the same generator as the device workload."""
    chosen, total = [], 0
    for s in specs:
        if chosen and total + s.numel > max_params:
            break
        chosen.append(s)
        total += s.numel
    if dev is not None:
        pairs = workloads.torch_model(chosen, seed, eta, dev)
        host = [(m.cpu().numpy(), p.cpu().numpy().view(np.uint16)) for m, p in pairs]
        del pairs
    else:
        rng = np.random.default_rng(seed)
        host = []
        for s in chosen:
            w0 = workloads.np_init(s, rng)
            host.append((workloads.np_update(w0, eta, rng), workloads.np_bf16_view_torch(w0)))
    return chosen, host, total


def time_oracle(host_pairs, threads):
    """Wall time of the oracle's encode + apply over the sample, tensor by
    tensor. threads == 1: the plain single-threaded calls. Otherwise every
    tensor is split into 4 x threads contiguous chunks run on `threads` host
    threads: a count pass, an exclusive scan of the chunk counts, an emit pass
    into place, then the apply over ranges of the patch (the same scalar C
    loops; oracle.encode_chunked / apply_chunked)."""
    import oracle
    oracle.build()
    work = [(m, p.copy(), p.copy()) for m, p in host_pairs]
    k = 0
    t0 = time.perf_counter()
    if threads == 1:
        for m, prev, w in work:
            idx, val = oracle.encode(m, prev)
            oracle.apply(w, idx, val)
            k += idx.size
    else:
        with ThreadPoolExecutor(max_workers=threads) as pool:
            for m, prev, w in work:
                idx, val = oracle.encode_chunked(m, prev, pool, 4 * threads)
                oracle.apply_chunked(w, idx, val, pool, 4 * threads)
                k += idx.size
    return time.perf_counter() - t0, k


# ----------------------------------------------------------------- arms

def run_reference(args, cfg, specs, rank, world, dist_on):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else None
    cores = host_cores()
    chosen, host, total = oracle_sample(specs, cfg["seed"], cfg["eta"], args.cpu_sample_params, dev)
    threads = cores
    for _ in range(args.warmup):
        time_oracle(host, threads)
    times, ks = [], []
    for _ in range(args.steps):
        t, k = time_oracle(host, threads)
        times.append(t)
        ks.append(k)
    tt = sum(times)
    value = total * args.steps / tt
    sample = (f"first {len(chosen)} tensors of {cfg['name']} ({total} of "
              f"{workloads.total_params(specs)} params), encode+apply tensor by tensor, each "
              f"tensor chunk-parallel on {threads} threads (count pass, scan, emit pass)")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic",
        "config": {"workload": cfg["name"], "params": workloads.total_params(specs),
                   "tensors": len(specs), "eta": cfg["eta"], "sample_params": total},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "density": float(np.mean(ks)) / total,
    }


def run_ours(args, cfg, specs, rank, world, dist_on):
    import rl_post_trainer_gb300 as pulse
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = Workload(specs, cfg["seed"] + 1000 * rank, cfg["eta"], dev, xor=not args.no_xor)
    n = wl.n
    stream = torch.cuda.current_stream(dev)
    # trainer + sampler buffers of one step: master, prev, w, patch capacity
    footprint = 14 * n
    flush = (torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
             if footprint < 4 * L2_BYTES else None)
    if flush is None:
        l2_note = (f"step buffers ({footprint / 1e9:.3g} GB: master, prev, w, patch) larger than "
                   "L2; prev and w restored untimed before each step")
    else:
        l2_note = ("L2 flushed by a 1 GiB write after the untimed restore of prev and w, "
                   "before each encode + apply step")

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        wl.plan.encode(wl.counts)
        if ev is not None:
            ev[1].record(stream)
        wl.plan.apply(wl.counts)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        wl.restore()
        step()
    torch.cuda.synchronize()
    if wl.plan.get_error() != 0:
        raise RuntimeError("device error during warm-up")
    counts_np = wl.counts.cpu().numpy()
    k = int(counts_np.sum())

    t_enc, t_app = [], []
    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        for _ in range(args.steps):
            wl.restore()
            if flush is not None:
                flush.fill_(1)
            torch.cuda.synchronize()
            barrier(dist_on)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            step(ev)
            torch.cuda.synchronize()
            barrier(dist_on)
            t_enc.append(ev[0].elapsed_time(ev[1]) * 1e-3)
            t_app.append(ev[1].elapsed_time(ev[2]) * 1e-3)
    if wl.plan.get_error() != 0:
        raise RuntimeError("device error during the timed steps")
    # the sampler holds the trainer's new view after every step
    for t in range(len(specs)):
        if not torch.equal(wl.w[t], wl.prev[t]):
            raise RuntimeError(f"sampler weights differ from the trainer view (tensor {t})")

    step_s = max_over_ranks(sum(t_enc) + sum(t_app), dist_on)
    total_params = sum_over_ranks(float(n), dist_on)
    value = total_params * args.steps / step_s
    enc_s = float(np.mean(t_enc))
    app_s = float(np.mean(t_app))
    S = wl.sectors_touched(counts_np)
    enc_alg = 6.0 * n + 8.0 * k
    enc_sec = 6.0 * n + 32.0 * S + 6.0 * k
    app_alg = 8.0 * k
    app_sec = 6.0 * k + 32.0 * S
    app_rmw = 6.0 * k + 64.0 * S
    peak, peak_kind = measured_peak_gbs()
    achieved = enc_alg / enc_s / 1e9
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic",
        "config": {"workload": cfg["name"], "params": n, "tensors": len(specs), "eta": cfg["eta"],
                   "density": k / n, "patch_entries": k, "parallelism": f"replicas{world}",
                   "l2": l2_note},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(),
                     "kernel": "encode_kernel<multi>", "peak_kind": peak_kind,
                     "bytes_model": "6n+8k",
                     # the same launch time against the sector-granular minimum (prev is
                     # written back in whole 32-byte sectors), and the highest frac the
                     # algorithmic model allows if those bytes moved at the copy peak
                     "frac_sector": enc_sec / enc_s / 1e9 / peak,
                     "frac_cap": enc_alg / enc_sec},
        "encode": {"ms": 1e3 * enc_s, "params_per_s": n / enc_s,
                   "gbs_algorithmic": enc_alg / enc_s / 1e9, "gbs_sector": enc_sec / enc_s / 1e9,
                   "frac_measured_peak": enc_alg / enc_s / 1e9 / peak,
                   "frac_nominal_8tbs": enc_alg / enc_s / 1e9 / NOMINAL_HBM_GBS,
                   "frac_sector_measured_peak": enc_sec / enc_s / 1e9 / peak,
                   "frac_sector_nominal_8tbs": enc_sec / enc_s / 1e9 / NOMINAL_HBM_GBS},
        "apply": {"ms": 1e3 * app_s, "params_per_s": n / app_s,
                  "gbs_algorithmic": app_alg / app_s / 1e9, "gbs_sector": app_sec / app_s / 1e9,
                  "gbs_sector_rmw": app_rmw / app_s / 1e9,
                  "frac_sector_rmw_measured_peak": app_rmw / app_s / 1e9 / peak,
                  "frac_sector_rmw_nominal_8tbs": app_rmw / app_s / 1e9 / NOMINAL_HBM_GBS},
        "sectors_touched": S,
        # one encode launch and one apply launch per step
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(),
    }

    if wl.xor:
        tm, ta = [], []
        for _ in range(max(1, args.steps)):
            wl.restore_xor()
            torch.cuda.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            wl.xplan.xor_mask()
            ev[1].record(stream)
            wl.xplan.xor_apply()
            ev[2].record(stream)
            torch.cuda.synchronize()
            tm.append(ev[0].elapsed_time(ev[1]) * 1e-3)
            ta.append(ev[1].elapsed_time(ev[2]) * 1e-3)
        xm, xa = float(np.mean(tm)), float(np.mean(ta))
        xm_bytes = 8.0 * n + 32.0 * S
        xa_bytes = 2.0 * n + 64.0 * S
        out["xor"] = {"mask_ms": 1e3 * xm, "apply_ms": 1e3 * xa,
                      "params_per_s": n / (xm + xa),
                      "mask_gbs_sector": xm_bytes / xm / 1e9,
                      "mask_frac_measured_peak": xm_bytes / xm / 1e9 / peak,
                      "apply_gbs_sector_rmw": xa_bytes / xa / 1e9,
                      "apply_frac_measured_peak": xa_bytes / xa / 1e9 / peak}
        for t in range(len(specs)):
            if not torch.equal(wl.w_x[t], wl.prev[t]):
                raise RuntimeError(f"XOR path disagrees with the patch path (tensor {t})")
        del wl.prev_x, wl.w_x, wl.mask
        wl.xplan.close()

    if cfg.get("sparse_eta") and not args.no_sparse:
        out["sparse"] = run_sparse(args, cfg, specs, wl, dev, rank, peak, cfg["sparse_eta"])
    if cfg.get("sweep"):
        out["sweep"] = run_sweep(args, specs, cfg["seed"], dev, peak)
    if not args.no_mx:
        out["mxfp8"] = run_mx(args, cfg, specs, wl, dev, rank, peak, pulse.MX_E4M3)
        out["mxfp4"] = run_mx(args, cfg, specs, wl, dev, rank, peak, pulse.MX_E2M1)
        out["nvfp4"] = run_mx(args, cfg, specs, wl, dev, rank, peak, pulse.MX_NVFP4)

    if not args.no_e2e:
        out["e2e"] = e2e(args, wl, counts_np, dist_on)
    if not args.no_pack:
        out["pack"] = run_pack(args, wl, counts_np, dev)
    if not args.no_compose:
        out["compose"] = run_compose(args, wl, dev)   # advances the masters
    if not args.no_loco:
        wl.release_views()
        out["loco"] = run_loco(args, cfg, specs, wl, dev, rank, peak,
                               local_steps=1 if args.no_compose else 4)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = host_cores()
        chosen, host, total = oracle_sample(specs, cfg["seed"], cfg["eta"], args.cpu_sample_params, dev)
        threads = cores
        t, _ = time_oracle(host, threads)
        # the same sample through the plain single-threaded oracle
        t1, _ = time_oracle(host, 1)
        del host
        out["cpu_baseline"] = {
            "value": total / t, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {len(chosen)} tensors ({total} params) of {cfg['name']}, "
                      f"encode+apply tensor by tensor, each tensor chunk-parallel on {threads} "
                      "threads (count pass, scan, emit pass, apply over patch ranges)",
            "value_one_thread": total / t1,
            "sample_one_thread": "the same sample, plain single-threaded oracle calls",
            "speedup": t1 / t}
    return out


def regen_masters(wl, specs, seed, eta, dev):
    """Redraw the FP32 masters in place at update scale `eta`: the generator
    sequence of the workload (per tensor: w0, then z), so the saved view of
    w0 (prev0) still holds."""
    gen = workloads.torch_generator(dev, seed)
    for m, spec in zip(wl.master, specs):
        workloads.torch_init_(m, spec, gen)
        workloads.torch_update_(m, eta, gen)


def run_sparse(args, cfg, specs, wl, dev, rank, peak, eta):
    """The same model and initial weights at a smaller update scale (about
    1 % of the BF16 view changes at eta = 3e-7, the pages' steady-state
    regime): encode + apply timed like the headline step (prev and w restored
    untimed before every step). The masters are redrawn at `eta` first and at
    the workload's own scale afterwards."""
    seed = cfg["seed"] + 1000 * rank
    regen_masters(wl, specs, seed, eta, dev)
    stream = torch.cuda.current_stream(dev)
    n = wl.n
    for _ in range(args.warmup):
        wl.restore()
        wl.plan.encode(wl.counts)
        wl.plan.apply(wl.counts)
    torch.cuda.synchronize()
    counts_np = wl.counts.cpu().numpy()
    k = int(counts_np.sum())
    te, ta = [], []
    for _ in range(args.steps):
        wl.restore()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(stream)
        wl.plan.encode(wl.counts)
        ev[1].record(stream)
        wl.plan.apply(wl.counts)
        ev[2].record(stream)
        torch.cuda.synchronize()
        te.append(ev[0].elapsed_time(ev[1]) * 1e-3)
        ta.append(ev[1].elapsed_time(ev[2]) * 1e-3)
    if wl.plan.get_error() != 0:
        raise RuntimeError("device error in the sparse-regime steps")
    for t in range(len(specs)):
        if not torch.equal(wl.w[t], wl.prev[t]):
            raise RuntimeError(f"sampler weights differ from the trainer view (tensor {t})")
    S = wl.sectors_touched(counts_np)
    regen_masters(wl, specs, seed, cfg["eta"], dev)
    e_s, a_s = float(np.mean(te)), float(np.mean(ta))
    enc_alg, enc_sec = 6.0 * n + 8.0 * k, 6.0 * n + 32.0 * S + 6.0 * k
    app_rmw = 6.0 * k + 64.0 * S
    return {
        "eta": eta, "density": k / n, "patch_entries": k, "sectors_touched": S,
        "encode_ms": 1e3 * e_s, "apply_ms": 1e3 * a_s, "params_per_s": n / (e_s + a_s),
        "encode_gbs_algorithmic": enc_alg / e_s / 1e9,
        "encode_frac_measured_peak": enc_alg / e_s / 1e9 / peak,
        "encode_frac_sector_measured_peak": enc_sec / e_s / 1e9 / peak,
        "apply_gbs_sector_rmw": app_rmw / a_s / 1e9,
        "apply_frac_sector_rmw_measured_peak": app_rmw / a_s / 1e9 / peak,
        "bytes_model": "encode 6n + 8k (sector 6n + 32S + 6k); apply 6k + 64S",
        "gpu_launches": 2 * args.steps,
    }


def run_mx(args, cfg, specs, wl, dev, rank, peak, fmt=0):
    """A low-precision serving view (fmt 0: MXFP8, 1: MXFP4, 2: NVFP4) of the
    same model and step: whole-model encode (pulse_mx_encode_multi, or
    pulse_nvfp4_encode_multi: tensor maxima pass + encode) and
    pulse_mx_apply_multi_device, timed like the BF16 step (previous view and
    receiver restored untimed before each step). The BF16 patch buffers are
    reused for the code segments."""
    import rl_post_trainer_gb300 as pulse
    n = wl.n
    name = {pulse.MX_E4M3: "MXFP8", pulse.MX_E2M1: "MXFP4", pulse.MX_NVFP4: "NVFP4"}[fmt]
    epb = 1 if fmt == pulse.MX_E4M3 else 2   # elements per code byte
    stream = torch.cuda.current_stream(dev)
    # the view before the step: the same generator sequence as the workload
    # (per tensor: w0, then z), quantizing each w0 as it is drawn
    gen = workloads.torch_generator(dev, cfg["seed"] + 1000 * rank)
    c0, s0 = [], []
    tmp = torch.empty(max(s.numel for s in specs), dtype=torch.float32, device=dev)
    for spec in specs:
        w0 = tmp[:spec.numel]
        workloads.torch_init_(w0, spec, gen)
        if fmt == pulse.MX_NVFP4:
            c, sc, _ = pulse.nvfp4_quantize(w0)
            c, sc = c.clone(), sc.clone()
        else:
            c, sc = pulse.mx_quantize(w0, fmt=fmt)
        c0.append(c)
        s0.append(sc)
        workloads.torch_update_(w0, cfg["eta"], gen)   # advances the generator past z
    del tmp
    prev_c = [c.clone() for c in c0]
    prev_s = [x.clone() for x in s0]
    codes = [c.clone() for c in c0]
    scales = [x.clone() for x in s0]
    nb = [pulse.mx_scale_count(s.numel, fmt) for s in specs]
    sidx = [torch.empty(max(b, 1), dtype=torch.int32, device=dev) for b in nb]
    sval = [torch.empty(max(b, 1), dtype=torch.uint8, device=dev) for b in nb]
    plan = pulse.MxPlan([pulse.MxTensorSlot(s.numel, master=wl.master[i], prev_codes=prev_c[i],
                                            prev_scales=prev_s[i], codes=codes[i], scales=scales[i],
                                            idx=wl.idx[i], val=wl.val[i].view(torch.uint8),
                                            sidx=sidx[i], sval=sval[i])
                         for i, s in enumerate(specs)], fmt=fmt)
    counts = torch.zeros(2 * len(specs), dtype=torch.int64, device=dev)

    def restore():
        for a, b in zip(prev_c, c0):
            a.copy_(b)
        for a, b in zip(prev_s, s0):
            a.copy_(b)
        for a, b in zip(codes, c0):
            a.copy_(b)
        for a, b in zip(scales, s0):
            a.copy_(b)

    for _ in range(args.warmup):
        restore()
        plan.encode(counts)
        plan.apply(counts)
    torch.cuda.synchronize()
    te, ta = [], []
    for _ in range(args.steps):
        restore()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(stream)
        plan.encode(counts)
        ev[1].record(stream)
        plan.apply(counts)
        ev[2].record(stream)
        torch.cuda.synchronize()
        te.append(ev[0].elapsed_time(ev[1]) * 1e-3)
        ta.append(ev[1].elapsed_time(ev[2]) * 1e-3)
    if plan.get_error() != 0:
        raise RuntimeError(f"device error in the {name} steps")
    for t in range(len(specs)):
        if not (torch.equal(codes[t], prev_c[t]) and torch.equal(scales[t], prev_s[t])):
            raise RuntimeError(f"{name} receiver differs from the trainer view (tensor {t})")
    cn = counts.cpu().numpy()
    k, ks = int(cn[0::2].sum()), int(cn[1::2].sum())
    # distinct 32-byte sectors holding a changed code / scale (1-byte arrays,
    # allocations 512-byte aligned: sector = index // 32)
    sc_codes = sc_scales = 0
    for t in range(len(specs)):
        for cnt, arr in ((int(cn[2 * t]), wl.idx[t]), (int(cn[2 * t + 1]), sidx[t])):
            if cnt:
                sec = arr[:cnt].to(torch.int64) // 32
                val = 1 + int((sec[1:] != sec[:-1]).sum().item())
                if arr is sidx[t]:
                    sc_scales += val
                else:
                    sc_codes += val
    nblocks = float(sum(nb))
    e_s, a_s = float(np.mean(te)), float(np.mean(ta))
    # master read (twice for NVFP4: the tensor maxima first) + previous view read
    view = (4.0 + 1.0 / epb) * n + nblocks + (4.0 * n if fmt == pulse.MX_NVFP4 else 0.0)
    enc_alg = view + 6.0 * k + 6.0 * ks
    enc_sec = view + 32.0 * (sc_codes + sc_scales) + 5.0 * k + 5.0 * ks
    app_rmw = 5.0 * (k + ks) + 64.0 * (sc_codes + sc_scales)
    plan.close()
    model = {pulse.MX_E4M3: "5n + n/32", pulse.MX_E2M1: "4.5n + n/32",
             pulse.MX_NVFP4: "8.5n + n/16"}[fmt]
    fmt_name = {
        pulse.MX_E4M3: "MXFP8 (E4M3 codes, E8M0 scale per 32 elements)",
        pulse.MX_E2M1: "MXFP4 (E2M1 codes two per byte, E8M0 scale per 32 elements; code entries "
                       "are bytes)",
        pulse.MX_NVFP4: "NVFP4 (E2M1 codes two per byte, E4M3 scale per 16 elements, FP32 scale "
                        "per tensor; code entries are bytes; encode includes the tensor-maximum "
                        "pass)"}[fmt]
    return {
        "format": fmt_name,
        "encode_ms": 1e3 * e_s, "apply_ms": 1e3 * a_s,
        "params_per_s": n / (e_s + a_s),
        "code_density": k / (n / epb), "scale_density": ks / nblocks,
        "code_entries": k, "scale_entries": ks,
        "encode_gbs_algorithmic": enc_alg / e_s / 1e9,
        "encode_gbs_sector": enc_sec / e_s / 1e9,
        "encode_frac_measured_peak": enc_alg / e_s / 1e9 / peak,
        "encode_frac_sector_measured_peak": enc_sec / e_s / 1e9 / peak,
        "apply_gbs_sector_rmw": app_rmw / a_s / 1e9,
        "apply_frac_sector_rmw_measured_peak": app_rmw / a_s / 1e9 / peak,
        "sectors_touched": sc_codes + sc_scales,
        "bytes_model": f"encode {model} + 6k + 6ks (sector: {model} + 32S + 5k + 5ks); "
                       "apply 5k + 5ks + 64S (each touched 32-byte sector read and written)",
        "gpu_launches": (3 if fmt == pulse.MX_NVFP4 else 2) * args.steps,
    }


def run_compose(args, wl, dev, versions: int = 4):
    """Sidecar catch-up over `versions` missing versions of the whole model:
    encode `versions` consecutive steps (untimed), then time (a) the chained
    apply (pulse_apply_chain_multi: every version in one pass over w, the
    catch-up path the library recommends), (b) applying the patches one after
    another, and (c) the k-way composition into one patch
    (pulse_compose_chain_multi) plus one apply of it. The pairwise fold
    (pulse_compose_multi, folded left) runs once, untimed, as the reference
    the k-way composition is checked against."""
    import rl_post_trainer_gb300 as pulse
    specs = wl.specs
    T = len(specs)
    stream = torch.cuda.current_stream(dev)
    wl.restore()
    chain = []   # per version: (idx list, val list, host counts)
    for v in range(versions):
        if v > 0:
            workloads.torch_step_(wl.master, 500 + v)
        wl.plan.encode(wl.counts)
        ks = wl.counts.cpu().tolist()
        chain.append(([wl.idx[t][:ks[t]].clone() for t in range(T)],
                      [wl.val[t][:ks[t]].clone() for t in range(T)], ks))
    final_view = [p.clone() for p in wl.prev]
    # ping-pong outputs sized for the largest possible composition
    cap = [sum(c[2][t] for c in chain) for t in range(T)]
    outs = [([torch.empty(max(cap[t], 1), dtype=torch.int32, device=dev) for t in range(T)],
             [torch.empty(max(cap[t], 1), dtype=torch.int16, device=dev) for t in range(T)])
            for _ in range(2)]
    apply_plan = pulse.Plan([pulse.TensorSlot(s.numel, w=wl.w[t], idx=wl.idx[t], val=wl.val[t])
                             for t, s in enumerate(specs)])

    def compose_chain():
        cur_i, cur_v, cur_k = chain[0]
        for v in range(1, versions):
            oi, ov = outs[v % 2]
            nxt_i, nxt_v, nxt_k = chain[v]
            segs = [(cur_i[t], cur_v[t], cur_k[t], nxt_i[t], nxt_v[t], nxt_k[t], oi[t], ov[t])
                    for t in range(T)]
            counts = pulse.compose_multi(segs)
            out_k = counts.cpu().tolist()     # host counts feed the next fold
            cur_i, cur_v, cur_k = oi, ov, out_k
        return cur_i, cur_v, cur_k

    last_i, last_v = outs[(versions - 1) % 2]
    composed_plan = pulse.Plan([pulse.TensorSlot(s.numel, w=wl.w[t], idx=last_i[t], val=last_v[t])
                                for t, s in enumerate(specs)])

    chain_plan = pulse.Plan([pulse.TensorSlot(s.numel, w=wl.w[t]) for t, s in enumerate(specs)])
    chain_refs = chain_plan.prepare_chain([[(c[0][t], c[1][t], c[2][t]) for t in range(T)]
                                           for c in chain])

    kway_out = [(torch.empty(max(cap[t], 1), dtype=torch.int32, device=dev),
                 torch.empty(max(cap[t], 1), dtype=torch.int16, device=dev)) for t in range(T)]
    kway_prep = chain_plan.prepare_compose(chain_refs, kway_out)
    kway_counts = torch.empty(T, dtype=torch.int64, device=dev)

    def compose_kway():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        chain_plan.compose_chain(kway_prep, counts_out=kway_counts)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3

    def apply_chained():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        chain_plan.apply_chain(chain_refs)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3

    def apply_seq():
        for idx_l, val_l, ks in chain:
            for t in range(T):
                wl.idx[t][:ks[t]].copy_(idx_l[t])
                wl.val[t][:ks[t]].copy_(val_l[t])
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            apply_plan.apply(ks)
            e1.record(stream)
            torch.cuda.synchronize()
            yield e0.elapsed_time(e1) * 1e-3

    # the reference composition (pairwise fold), once
    ci, cv, ck = compose_chain()
    torch.cuda.synchronize()
    t_app1, t_seq, t_chain, t_kway = [], [], [], []
    reps = max(1, min(args.steps, 3))
    for r in range(reps + 1):          # the first round is a warm-up
        for w, p0 in zip(wl.w, wl.prev0):
            w.copy_(p0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        composed_plan.apply(ck)
        e1.record(stream)
        torch.cuda.synchronize()
        ta = e0.elapsed_time(e1) * 1e-3
        for t in range(T):
            if not torch.equal(wl.w[t], final_view[t]):
                raise RuntimeError(f"composed catch-up differs from the final view (tensor {t})")
        for w, p0 in zip(wl.w, wl.prev0):
            w.copy_(p0)
        ts = sum(apply_seq())
        for t in range(T):
            if not torch.equal(wl.w[t], final_view[t]):
                raise RuntimeError(f"sequential catch-up differs from the final view (tensor {t})")
        for w, p0 in zip(wl.w, wl.prev0):
            w.copy_(p0)
        torch.cuda.synchronize()
        tch = apply_chained()
        for t in range(T):
            if not torch.equal(wl.w[t], final_view[t]):
                raise RuntimeError(f"chained catch-up differs from the final view (tensor {t})")
        tk = compose_kway()
        kc = kway_counts.cpu().tolist()
        for t in range(T):
            if kc[t] != ck[t] or not (torch.equal(kway_out[t][0][:kc[t]], ci[t][:ck[t]]) and
                                      torch.equal(kway_out[t][1][:kc[t]], cv[t][:ck[t]])):
                raise RuntimeError(f"k-way composition differs from the folded one (tensor {t})")
        if r > 0:
            t_app1.append(ta)
            t_seq.append(ts)
            t_chain.append(tch)
            t_kway.append(tk)
    if pulse.get_error(dev) != 0:
        raise RuntimeError("device error in the compose leg")
    if chain_plan.get_error() != 0:
        raise RuntimeError("device error in the chained apply")
    # sectors of w that any version touches: the composed patch's distinct idx / 16
    s_union = 0
    for t in range(T):
        if ck[t] > 0:
            sec = ci[t][:ck[t]] // 16
            s_union += 1 + int(torch.count_nonzero(sec[1:] != sec[:-1]))
    apply_plan.close()
    composed_plan.close()
    chain_plan.close()
    k_in = [sum(c[2]) for c in chain]
    k_out = sum(ck)
    tam, tsm = float(np.mean(t_app1)), float(np.mean(t_seq))
    tchm = float(np.mean(t_chain))
    tkm = float(np.mean(t_kway))
    kway_bytes = 6 * sum(k_in) + 6 * k_out
    chain_bytes = 6 * sum(k_in) + 64 * s_union
    return {
        "versions": versions, "patch_entries": k_in, "composed_entries": k_out,
        "catch_up_chained_ms": 1e3 * tchm, "catch_up_sequential_ms": 1e3 * tsm,
        "apply_composed_ms": 1e3 * tam,
        "compose_kway_ms": 1e3 * tkm, "compose_kway_bytes": kway_bytes,
        "compose_kway_gbs": kway_bytes / tkm / 1e9,
        "catch_up_kway_composed_ms": 1e3 * (tkm + tam),
        "sectors_union": s_union,
        "chained_bytes_model": "6 * sum(k) + 64 * S_union", "chained_bytes": chain_bytes,
        "chained_gbs": chain_bytes / tchm / 1e9,
        "timing": "CUDA events. chained: one pulse_apply_chain_multi call on a prepared chain "
                  "(partition + apply launch); sequential: one whole-model apply per version; "
                  "k-way: one pulse_compose_chain_multi call over all versions (partition + "
                  "compose launch), checked equal to a pairwise fold of the same chain, then "
                  "one apply of the composed patch",
    }


def run_sweep(args, specs, seed, dev, peak):
    """Encode + apply of one flat tensor at every update scale of the density
    sweep: w0 from `seed`, the i-th scale's z from sweep_seed(i) (the draws of
    the parity tests). prev and w restored untimed before every step; the
    inputs (1.6 GB and up) are larger than L2. CUDA events, mean over steps."""
    import rl_post_trainer_gb300 as pulse
    (spec,) = specs
    n = spec.numel
    gen = workloads.torch_generator(dev, seed)
    w0 = torch.empty(n, dtype=torch.float32, device=dev)
    workloads.torch_init_(w0, spec, gen)
    p0 = torch.empty(n, dtype=torch.int16, device=dev)
    workloads.torch_bf16_view_(p0, w0)
    m = torch.empty_like(w0)
    prev, w = torch.empty_like(p0), torch.empty_like(p0)
    idx = torch.empty(n, dtype=torch.int32, device=dev)
    val = torch.empty(n, dtype=torch.int16, device=dev)
    counts = torch.zeros(1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    rows = []
    with pulse.Plan([pulse.TensorSlot(n, master=m, prev=prev, w=w, idx=idx, val=val)]) as plan:
        for i, eta in enumerate(workloads.ETA_SWEEP):
            m.copy_(w0)
            workloads.torch_update_(m, eta, workloads.torch_generator(dev, workloads.sweep_seed(i)))
            te, ta = [], []
            for it in range(args.warmup + args.steps):
                prev.copy_(p0)
                w.copy_(p0)
                torch.cuda.synchronize()
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                ev[0].record(stream)
                plan.encode(counts)
                ev[1].record(stream)
                plan.apply(counts)
                ev[2].record(stream)
                torch.cuda.synchronize()
                if it >= args.warmup:
                    te.append(ev[0].elapsed_time(ev[1]) * 1e-3)
                    ta.append(ev[1].elapsed_time(ev[2]) * 1e-3)
            if plan.get_error() != 0:
                raise RuntimeError(f"device error in the sweep at eta={eta}")
            if not torch.equal(w, prev):
                raise RuntimeError(f"sampler weights differ from the trainer view at eta={eta}")
            k = int(counts.item())
            sec = idx[:k].to(torch.int64) // 16
            S = 0 if k == 0 else 1 + int((sec[1:] != sec[:-1]).sum().item())
            del sec
            enc_s, app_s = float(np.mean(te)), float(np.mean(ta))
            enc_sec = 6.0 * n + 32.0 * S + 6.0 * k
            app_rmw = 6.0 * k + 64.0 * S
            rows.append({"eta": eta, "density": k / n, "patch_entries": k, "sectors_touched": S,
                         "encode_ms": 1e3 * enc_s, "apply_ms": 1e3 * app_s,
                         "params_per_s": n / (enc_s + app_s),
                         "encode_gbs_algorithmic": (6.0 * n + 8.0 * k) / enc_s / 1e9,
                         "encode_frac_sector_measured_peak": enc_sec / enc_s / 1e9 / peak,
                         "apply_frac_sector_rmw_measured_peak": app_rmw / app_s / 1e9 / peak})
    return {"workload": f"one flat tensor of {n} params", "rows": rows,
            "bytes_model": "encode 6n+8k (sector 6n+32S+6k); apply sector read-modify-write 6k+64S",
            "gpu_launches": 2 * len(rows) * (args.warmup + args.steps)}


def run_pack(args, wl, counts_np, dev):
    """Codec-friendly packing of the step's patch indices (every tensor's
    segment in one pulse_pack_indices_multi launch), and the receiver's
    unpack (one pulse_unpack_indices_multi launch), checked to round-trip.
    CUDA events around each call."""
    import rl_post_trainer_gb300 as pulse
    stream = torch.cuda.current_stream(dev)
    wl.restore()
    wl.plan.encode(wl.counts)          # the step's patch into wl.idx / wl.val
    ks = wl.counts.cpu().tolist()
    T = len(ks)
    job = pulse.PackJob([(wl.idx[t], ks[t]) for t in range(T)])

    tp, tu = [], []
    for r in range(args.warmup + args.steps):
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(stream)
        job.pack()
        ev[1].record(stream)
        job.unpack()
        ev[2].record(stream)
        torch.cuda.synchronize()
        if r >= args.warmup:
            tp.append(ev[0].elapsed_time(ev[1]) * 1e-3)
            tu.append(ev[1].elapsed_time(ev[2]) * 1e-3)
    if pulse.get_error(dev) != 0:
        raise RuntimeError("device error in the packing leg")
    for t in range(T):
        if ks[t] and not torch.equal(job.unpacked[t][:ks[t]], wl.idx[t][:ks[t]]):
            raise RuntimeError(f"unpack differs from the patch indices (tensor {t})")
    k = sum(ks)
    payload = int(job.payload_bytes.sum().item())
    headers = sum(5 * ((kk + 127) // 128) + 8 * ((kk + 4095) // 4096) for kk in ks)
    tpm, tum = float(np.mean(tp)), float(np.mean(tu))
    return {
        "entries": k, "index_bytes_raw": 4 * k, "index_bytes_packed": payload + headers,
        "bits_per_index": 8.0 * (payload + headers) / max(k, 1),
        "patch_bytes_raw": 6 * k, "patch_bytes_packed": payload + headers + 2 * k,
        "pack_ms": 1e3 * tpm, "unpack_ms": 1e3 * tum,
        "pack_gbs_in": 4.0 * k / tpm / 1e9, "unpack_gbs_out": 4.0 * k / tum / 1e9,
        "launches": 2, "timing": f"all {T} segments in one pack and one unpack launch, CUDA events",
    }


def run_loco(args, cfg, specs, wl, dev, rank, peak, local_steps):
    """The PULSELoCo sender gate over the whole model (pulse_loco_gate_multi)
    and the receiver's accumulation (pulse_loco_accumulate_multi): global =
    the starting weights w0 (the same generator draws), local = the current
    master (`local_steps` Adam-sized steps past w0), error buffer zero. The error buffer and the accumulator
    are restored untimed before each step. Reuses the BF16 patch index
    buffers for the sent indices."""
    import rl_post_trainer_gb300 as pulse
    n = wl.n
    stream = torch.cuda.current_stream(dev)
    gen = workloads.torch_generator(dev, cfg["seed"] + 1000 * rank)
    glob, err, val, acc = [], [], [], []
    for spec in specs:
        w0 = torch.empty(spec.numel, dtype=torch.float32, device=dev)
        workloads.torch_init_(w0, spec, gen)
        glob.append(w0)
        workloads.torch_update_(w0.clone(), cfg["eta"], gen)   # advances past this tensor's z
        err.append(torch.zeros(spec.numel, dtype=torch.float32, device=dev))
        val.append(torch.empty(spec.numel, dtype=torch.float32, device=dev))
        acc.append(w0.clone())
    plan = pulse.LocoPlan([pulse.LocoTensorSlot(s.numel, global_w=glob[t], local_w=wl.master[t],
                                                err=err[t], idx=wl.idx[t], val=val[t], acc=acc[t])
                           for t, s in enumerate(specs)])
    counts = torch.zeros(len(specs), dtype=torch.int64, device=dev)

    def restore():
        for e in err:
            e.zero_()
        for a_, g_ in zip(acc, glob):
            a_.copy_(g_)

    for _ in range(args.warmup):
        restore()
        plan.gate(counts)
        plan.accumulate(counts)
    torch.cuda.synchronize()
    tg, ta = [], []
    for _ in range(args.steps):
        restore()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(stream)
        plan.gate(counts)
        ev[1].record(stream)
        plan.accumulate(counts)
        ev[2].record(stream)
        torch.cuda.synchronize()
        tg.append(ev[0].elapsed_time(ev[1]) * 1e-3)
        ta.append(ev[1].elapsed_time(ev[2]) * 1e-3)
    if plan.get_error() != 0:
        raise RuntimeError("device error in the PULSELoCo steps")
    k = int(counts.sum().item())
    plan.close()
    g_s, a_s = float(np.mean(tg)), float(np.mean(ta))
    gate_bytes = 16.0 * n + 8.0 * k      # read global, local, err; write err; sent entries
    acc_bytes = 16.0 * k                 # read idx, val, acc; write acc (entry-granular)
    return {
        "local_steps": local_steps,
        "gate_ms": 1e3 * g_s, "accumulate_ms": 1e3 * a_s, "sent": k, "sent_fraction": k / n,
        "gate_params_per_s": n / g_s, "gate_gbs": gate_bytes / g_s / 1e9,
        "gate_frac_measured_peak": gate_bytes / g_s / 1e9 / peak,
        "accumulate_gbs_entry": acc_bytes / a_s / 1e9,
        "bytes_model": "gate 16n + 8k; accumulate 16k (entry-granular)",
        "gpu_launches": 2 * args.steps,
    }


def e2e(args, wl, counts_np, dist_on, groups: int = 16):
    """Same metric through the public API with HOST buffers: every step copies
    the new FP32 master from pinned host memory, encodes, reads the patch back
    to pinned host memory (the wire), copies it to the sampler and applies.

    The model is cut into `groups` groups of tensors of about equal size, one
    plan each, so the transfers overlap the work of other groups: masters go
    up on one stream; each group's encode waits for its masters, its count
    comes down at once, and as soon as the host has it the group's patch goes
    down and back up and is applied on other streams."""
    import rl_post_trainer_gb300 as pulse
    try:
        host_master = []
        for m in wl.master:
            h = torch.empty(m.shape, dtype=m.dtype, pin_memory=True)
            h.copy_(m)
            host_master.append(h)
        cap = [int(c * 1.05) + 1024 for c in counts_np]
        h_idx = [torch.empty(c, dtype=torch.int32, pin_memory=True) for c in cap]
        h_val = [torch.empty(c, dtype=torch.int16, pin_memory=True) for c in cap]
    except RuntimeError as exc:  # not enough pinnable host memory
        return {"value": None, "unit": UNIT, "error": str(exc)[:200]}
    n = wl.n
    T = len(wl.specs)
    dev = wl.master[0].device
    # groups of consecutive tensors with about n / groups params each
    bounds, acc, target = [0], 0, n / groups
    for t, s_ in enumerate(wl.specs):
        acc += s_.numel
        if acc >= target * len(bounds) and t + 1 < T:
            bounds.append(t + 1)
    bounds.append(T)
    G = len(bounds) - 1
    plans = [pulse.Plan([pulse.TensorSlot(wl.specs[t].numel, master=wl.master[t], prev=wl.prev[t],
                                          w=wl.w[t], idx=wl.idx[t], val=wl.val[t])
                         for t in range(bounds[g], bounds[g + 1])]) for g in range(G)]
    counts_d = [torch.zeros(bounds[g + 1] - bounds[g], dtype=torch.int64, device=dev) for g in range(G)]
    counts_h = [torch.zeros(bounds[g + 1] - bounds[g], dtype=torch.int64, pin_memory=True) for g in range(G)]
    # the receiver's copy of the counts, taken from the host side like the patch
    counts_r = [torch.zeros(bounds[g + 1] - bounds[g], dtype=torch.int64, device=dev) for g in range(G)]
    s_in, s_enc, s_out, s_back = (torch.cuda.Stream(dev) for _ in range(4))

    def one_step():
        ev_in = [torch.cuda.Event() for _ in range(G)]
        ev_cnt = [torch.cuda.Event() for _ in range(G)]
        ev_out = [torch.cuda.Event() for _ in range(G)]
        with torch.cuda.stream(s_in):
            for g in range(G):
                for t in range(bounds[g], bounds[g + 1]):
                    wl.master[t].copy_(host_master[t], non_blocking=True)
                ev_in[g].record(s_in)
        with torch.cuda.stream(s_enc):
            for g in range(G):
                s_enc.wait_event(ev_in[g])
                plans[g].encode(counts_d[g])
                counts_h[g].copy_(counts_d[g], non_blocking=True)
                ev_cnt[g].record(s_enc)
        ktot = 0
        for g in range(G):
            ev_cnt[g].synchronize()
            ks = counts_h[g].tolist()
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cnt[g])
                for j, t in enumerate(range(bounds[g], bounds[g + 1])):
                    k = ks[j]
                    if k > cap[t]:
                        raise RuntimeError("patch larger than the staging buffer")
                    h_idx[t][:k].copy_(wl.idx[t][:k], non_blocking=True)
                    h_val[t][:k].copy_(wl.val[t][:k], non_blocking=True)
                ev_out[g].record(s_out)
            with torch.cuda.stream(s_back):
                s_back.wait_event(ev_out[g])
                for j, t in enumerate(range(bounds[g], bounds[g + 1])):
                    k = ks[j]
                    wl.idx[t][:k].copy_(h_idx[t][:k], non_blocking=True)
                    wl.val[t][:k].copy_(h_val[t][:k], non_blocking=True)
                # counts from pinned host memory: an asynchronous copy, so the
                # host never waits for this stream to drain
                counts_r[g].copy_(counts_h[g], non_blocking=True)
                plans[g].apply(counts_r[g])
            ktot += sum(ks)
        torch.cuda.synchronize()
        return ktot

    for _ in range(args.warmup):
        wl.restore()
        one_step()
    times, ktot = [], 0
    for _ in range(args.steps):
        wl.restore()
        torch.cuda.synchronize()
        barrier(dist_on)
        t0 = time.perf_counter()
        ktot = one_step()
        times.append(time.perf_counter() - t0)
        barrier(dist_on)
    for t in range(T):
        if not torch.equal(wl.w[t], wl.prev[t]):
            raise RuntimeError(f"e2e: sampler weights differ from the trainer view (tensor {t})")
    for p_ in plans:
        p_.close()
    tt = max_over_ranks(sum(times), dist_on)
    total_params = sum_over_ranks(float(n), dist_on)
    return {"value": total_params * args.steps / tt, "unit": UNIT,
            "h2d_bytes_per_step": int(4 * n + 6 * ktot + 8 * T),
            "d2h_bytes_per_step": int(6 * ktot + 8 * T),
            "ms_per_step": 1e3 * tt / args.steps, "groups": G,
            "pipeline": "per-group plans; masters up on one stream, encode + counts down on a "
                        "second, patches down on a third, up again and applied on a fourth"}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-xor", action="store_true")
    ap.add_argument("--no-sparse", action="store_true",
                    help="skip the eta = 3e-7 (about 1 %% dense) leg of the 8B workload")
    ap.add_argument("--no-mx", action="store_true", help="skip the MXFP8-, MXFP4- and NVFP4-view legs")
    ap.add_argument("--no-compose", action="store_true", help="skip the patch-chain leg")
    ap.add_argument("--no-loco", action="store_true", help="skip the PULSELoCo leg")
    ap.add_argument("--no-pack", action="store_true", help="skip the index-packing leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-params", type=float, default=1.2e9)
    ap.add_argument("--eta", type=float, default=None,
                    help="override the workload's update scale (small-case captures)")
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="write profiles/encode_traffic.json from an ncu CSV of encode_kernel "
                         "launches on --config (no GPU work) and exit")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, args.config)))
        return
    cfg = dict(workloads.CONFIGS[args.config])
    if args.eta is not None:
        cfg["eta"] = args.eta
    if cfg["eta"] is None:  # the density sweep: the headline at the default scale, then every scale
        cfg["eta"] = workloads.ETA_DEFAULT
        cfg["sweep"] = True
    if args.config == 3:
        # the same model at the pages' steady-state density (about 1 % changed)
        cfg["sparse_eta"] = SPARSE_ETA
    specs = cfg["specs"]()

    if args.impl == "reference":
        # the oracle runs on rank 0's host cores; other ranks have no work
        if rank == 0:
            out = run_reference(args, cfg, specs, rank, world, False)
            print(json.dumps(out), flush=True)
        return

    dist_on = world > 1
    if dist_on:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend=backend)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    out = run_ours(args, cfg, specs, rank, world, dist_on)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist_on:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
