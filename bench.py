"""Benchmark: fused attention forward on GB300, one JSON line on stdout (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--no-sweep] [--no-cpu-baseline] [--no-e2e] [--no-clocks]

A step is one launch of the fused forward over one batch of the workload (inputs
resident in HBM).  Default workload: causal GQA prefill, Hq=32, Hkv=8, d=128, bf16,
S=8192, B=4 (B*S = 32768 tokens) -- the prefill configuration that runs the most of
the path at once (scheduler with longest-first causal order, causal bit masking and
tile skipping, GQA head mapping, both tensor-core contractions, online softmax,
correction, epilogue).  The line's headline fields are that workload's; its "sweep" key
times every workload of the pages' benchmarks the same way (10 warm-up launches, the
median of 50 timed ones), with each one's roofline fraction and, for the custom-mask
workloads, the number of skipped tiles against the oracle's count.

Under torchrun (--gpus N > 1) every rank runs its own replica of the workload on its
own GPU (weak scaling, no collective on the data path); the timed region is bracketed
by barriers and the slowest rank's time is reported; there is no sweep.

--impl reference times the fp64 CPU oracle (the only reference implementation this
project has) on a bounded random row sample of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS (GB300, 1 GPU) and % of dense BF16 peak / roofline"
DEFAULT_WORKLOAD = "gqa8_causal_S8192"
L2_BYTES = 129 * 1024 * 1024


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch size")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--e2e-buffers", type=int, default=2, help="device buffer sets in the end-to-end pipeline")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target length of the oracle sample")
    ap.add_argument("--sweep-only", default=None, metavar="NAME",
                    help="time one workload of the sweep (the pages' or an extension) with --warmup / --steps "
                         "launches and print its row as one JSON line instead of the bench line")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank's replica draws its own inputs (weak scaling: the per-GPU work is fixed)."""
    return base_seed + 7919 * rank


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- workload helpers

def workload(name: str, batch: int = 0):
    from dataclasses import replace
    from attention_forward_07_gb300 import inputs as inp
    if name not in inp.WORKLOADS:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(inp.WORKLOADS)}")
    w = inp.WORKLOADS[name]
    if batch:
        w = replace(w, B=batch)
    return w, list(inp.WORKLOADS).index(name)


def live_fraction(w, bits) -> float:
    """Fraction of (batch entry, 16-row block) pairs of a custom mask that keep anything
    (1.0 without a mask): the query rows the kernel has to read and compute."""
    if bits is None:
        return 1.0
    nz = np.asarray(bits).reshape(w.B, w.S, -1).any(axis=2)  # rows that keep anything
    pad = (-w.S) % 16
    if pad:
        nz = np.concatenate([nz, np.zeros((w.B, pad), bool)], axis=1)
    return float(nz.reshape(w.B, -1, 16).any(axis=2).mean())


def algorithmic_bytes(w, live: float = 1.0) -> int:
    """Compulsory HBM traffic of one launch: K, V, the mask words and the Q rows of the
    16-row blocks that keep anything read once, O and LSE written once."""
    el = 2
    q = w.B * w.Hq * w.S * w.d * el
    kv = 2 * w.B * w.Hkv * w.S * w.d * el
    o = q
    lse = w.B * w.Hq * w.S * 4
    mask = w.B * w.S * ((w.S + 31) // 32) * 4 if w.mask != "none" else 0
    return int(round(q * live)) + kv + o + lse + mask


def algorithmic_flops(w, live: float = 1.0) -> float:
    """The two contractions over the query rows that keep anything: the dense count
    4*B*Hq*S^2*d (halved for causal) times the live fraction."""
    return w.flops() * live


def config_dict(w, name, n):
    return {"workload": name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "d": w.d,
            "causal": w.causal, "mask": w.mask,
            "dtype_in": {0: "f16", 1: "bf16"}[w.dtype], "global_batch": w.B * n, "seq_len": w.S,
            "parallelism": f"replicas x{n}" if n > 1 else "single GPU",
            "l2": ("inputs larger than L2, no flush" if needs_flush(w) is False
                   else "L2 flushed (256 MiB write) between timed launches")}


def needs_flush(w) -> bool:
    return algorithmic_bytes(w) <= 2 * L2_BYTES


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["bf16_tflops"]), float(m["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, enabled: bool = True):
        self.proc = None
        self.lines = []
        self.index = index
        if enabled:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self.proc = None
        self.t_start = self.t_end = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for nm, val in zip(names, r[5:9]):
                if val.strip() == "Active":
                    reasons.add(nm)
        # keep the samples taken under load (clock above idle) if any
        load = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------- the oracle baseline

def cpu_baseline(w, seed, target_seconds: float):
    """The fp64 oracle, as it stands, on the host cores.  The short workloads are evaluated
    whole.  For the prefill workloads the whole oracle would take hours, so it runs on the
    row sample the measurement protocol names -- for every (batch, head): rows 0, 1, 127,
    128, S-1 and 64 seeded random rows -- repeated until about target_seconds have passed,
    and the whole-workload time is extrapolated from its rows per second.
    Returns a dict for the JSON line."""
    import oracle
    from attention_forward_07_gb300 import inputs as inp
    q, k, v, bits = w.make(seed)
    total_rows = w.B * w.Hq * w.S
    args = (inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), w.dtype)
    whole = total_rows <= 16 * 16 * 512
    rows = (np.arange(total_rows, dtype=np.int64) if whole
            else inp.sample_rows(w.B, w.Hq, w.S, 64, seed=seed))
    passes, dt = 0, 0.0
    while passes == 0 or (not whole and dt < target_seconds):
        t0 = time.perf_counter()
        oracle.attn_rows(*args, rows, bits, w.causal, w.scale)
        dt += time.perf_counter() - t0
        passes += 1
    per_pass = dt / passes
    full_seconds = per_pass * total_rows / len(rows)
    out = {"value": w.flops() / full_seconds / 1e12, "unit": "TFLOPS", "cores": oracle.num_threads(),
           "kind": "oracle", "rows_per_second": len(rows) / per_pass, "seconds": dt}
    if whole:
        out["sample"] = f"the whole workload ({total_rows} rows), fp64"
    else:
        out["sample"] = (f"{len(rows)} rows of {total_rows} (every (b, hq): rows 0, 1, 127, 128, S-1 and 64 "
                         f"seeded random rows), fp64, {passes} passes")
        out["extrapolated"] = True
        out["extrapolated_seconds"] = full_seconds
    return out


def cpu_single_thread(w, seed):
    """The whole oracle on one host thread (small workloads only), TFLOPS-equivalent."""
    import oracle
    from attention_forward_07_gb300 import inputs as inp
    q, k, v, bits = w.make(seed)
    rows = np.arange(w.B * w.Hq * w.S, dtype=np.int64)
    t0 = time.perf_counter()
    oracle.attn_rows(inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), w.dtype, rows, bits, w.causal, w.scale,
                     nthreads=1)
    return w.flops() / (time.perf_counter() - t0) / 1e12


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w, idx = workload(args.workload, args.batch)
    import oracle
    from attention_forward_07_gb300 import inputs as inp
    oracle.build()
    seed = w.seed(idx)
    q, k, v, bits = w.make(seed)
    a = (inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), w.dtype)
    total_rows = w.B * w.Hq * w.S
    rng = np.random.default_rng(seed)
    per_step = int(min(total_rows, 2048))
    times = []
    for step in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(total_rows, size=per_step, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.attn_rows(*a, rows, bits, w.causal, w.scale)
        if step >= args.warmup:
            times.append(time.perf_counter() - t0)
    dt = sum(times)
    flops = w.flops() * per_step / total_rows * len(times)
    value = flops / dt / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * dt / max(1, len(times)), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": config_dict(w, args.workload, 1),
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{per_step} random rows of {total_rows} per step (seeded), fp64"},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm

# DRAM bytes (read + write) per launch from `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum`,
# keyed by the sha1 of the kernel sources they were taken on; a changed kernel reports null.
MEASURED_TRAFFIC = {
    # dram__bytes_read.sum + dram__bytes_write.sum of one attention-kernel launch, captured at
    # full size (one launch, metrics-only, 1 pass) on the kernel with this source hash
    "bf31ac772055": {"B4_Hq32_Hkv8_S8192_d128_causal_none": 1338.56e6 + 236.14e6,
                     "B16_Hq16_Hkv16_S512_d64_full_bernoulli": 50.94e6 + 0.26e6,
                     "B16_Hq16_Hkv16_S512_d64_full_block90": 36.91e6 + 0.00e6},
}


def kernel_hash() -> str:
    """Hash of the kernel sources with comments and blank lines removed, so that the measured
    figures keyed by it stay attached to the code they were taken on."""
    import hashlib
    import re
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "attention_forward_07_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(name.encode() + text.encode())
    return h.hexdigest()[:12]


def roofline(w, seconds_per_launch, live: float = 1.0):
    """The slower of the tensor and HBM bounds for the algorithmic FLOP and bytes, and the
    fraction of it this launch time reaches."""
    p_tensor, p_hbm, src = peaks()
    flops, nbytes = algorithmic_flops(w, live), algorithmic_bytes(w, live)
    t_tensor = flops / (p_tensor * 1e12)
    t_hbm = nbytes / (p_hbm * 1e9)
    traffic = MEASURED_TRAFFIC.get(kernel_hash(), {}).get(config_key(w))
    common = {"traffic": traffic, "algorithmic_flops": flops, "algorithmic_bytes": nbytes, "live_fraction": live,
              "roofline_ms": 1e3 * max(t_tensor, t_hbm)}
    if t_tensor >= t_hbm:
        ach = flops / seconds_per_launch / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": p_tensor, "unit": "TFLOP/s", "frac": ach / p_tensor,
                "peak_source": f"{src} bf16 dense (burst)", **common}
    ach = nbytes / seconds_per_launch / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": p_hbm, "unit": "GB/s", "frac": ach / p_hbm,
            "peak_source": f"{src} HBM copy", **common}


def kernels_per_step(w) -> int:
    """This library's kernels in one forward call: the attention kernel, plus the mask
    pre-pass and the row compaction when a custom mask is given."""
    return 3 if w.mask != "none" else 1


def config_key(w):
    return f"B{w.B}_Hq{w.Hq}_Hkv{w.Hkv}_S{w.S}_d{w.d}_{'causal' if w.causal else 'full'}_{w.mask}"


def device_inputs(torch, dev, w, seed):
    q, k, v, bits = w.make(seed)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = None if bits is None else torch.from_numpy(bits.view(np.int32)).to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=dev)
    return (q, k, v, bits), (qd, kd, vd, md, o, lse)


def launch_times(torch, dev, step, warmup, timed, flush_buf):
    """Per-launch device times (ms) of `timed` launches after `warmup` untimed ones, CUDA
    events on the launching stream around each launch; the L2 is flushed between launches
    (by writing flush_buf, outside the events) when a buffer is given."""
    for _ in range(max(warmup, 0)):
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(timed)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(timed)]
    torch.cuda.synchronize(dev)
    for i in range(timed):
        if flush_buf is not None:
            flush_buf.fill_(i & 0xFF)
        starts[i].record()
        step()
        ends[i].record()
    torch.cuda.synchronize(dev)
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def skip_counts(af, torch, dev, w, tensors):
    """Blocks computed and skipped by the kernel (attn_fwd_visited, outside any timing)
    next to the oracle's counts for the same seeded mask (tests/golden/skip_counts.json,
    written by tests/golden/make_skip_counts.py)."""
    import hashlib
    qd, kd, vd, md, o, lse = tensors
    bm, bn = af.attn_tile_shape(w.d)
    vis = torch.zeros((w.B, w.Hq, -(-w.S // bm), -(-w.S // bn)), dtype=torch.uint8, device=dev)
    af.attn_fwd_visited(qd, kd, vd, o, lse, md, w.causal, w.scale, vis)
    af.attn_check()
    computed = int(vis.sum().item())
    out = {"blocks": vis.numel(), "computed": computed, "skipped": vis.numel() - computed}
    try:
        with open(os.path.join(ROOT, "tests", "golden", "skip_counts.json")) as f:
            ref = json.load(f)[w.name]
        bits = md.cpu().numpy().view(np.uint32)
        if ref["mask_sha1"] == hashlib.sha1(bits.tobytes()).hexdigest():
            out["oracle_skipped"] = ref["skipped"]
            out["match"] = ref["skipped"] == out["skipped"] and ref["computed"] == computed
        else:
            out["oracle_skipped"] = None  # the stored count is for other mask words
    except (OSError, KeyError):
        out["oracle_skipped"] = None
    return out


def run_sweep(af, torch, dev, warmup=10, timed=50, names=None):
    """Every workload of the pages' benchmarks, timed like the headline one (only `names` when
    given)."""
    from attention_forward_07_gb300 import inputs as inp
    rows = {}
    fbuf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for idx, (name, w) in enumerate(inp.WORKLOADS.items()):
        if names is not None and name not in names:
            continue
        (_, _, _, bits), t = device_inputs(torch, dev, w, w.seed(idx))
        qd, kd, vd, md, o, lse = t

        def step():
            af.attn_fwd(qd, kd, vd, o, lse, md, causal=w.causal, scale=w.scale)

        ms = launch_times(torch, dev, step, warmup, timed, fbuf if needs_flush(w) else None)
        af.attn_check()
        live = live_fraction(w, bits)
        med = statistics.median(ms)
        rf = roofline(w, med / 1e3, live)
        row = {"ms_median": med, "ms_mean": statistics.mean(ms), "value": w.flops() / (med / 1e3) / 1e12,
               "unit": "TFLOPS", "bound": rf["bound"], "achieved": rf["achieved"], "achieved_unit": rf["unit"],
               "frac": rf["frac"], "frac_of_mean": rf["frac"] * med / statistics.mean(ms),
               "live_fraction": live, "traffic": rf["traffic"], "launches": timed * kernels_per_step(w)}
        if w.mask != "none":
            row["tiles"] = skip_counts(af, torch, dev, w, t)
        rows[name] = row
        del t, qd, kd, vd, md, o, lse
        torch.cuda.empty_cache()
    for name, xw in inp.EX_WORKLOADS.items():
        # this library's extensions through attn_fwd_ex (not the pages' configurations)
        if names is not None and name not in names:
            continue
        q, k, v, bits = xw.make(2000 + xw.Sq % 1000)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        md = None if bits is None else torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).to(dev)
        o = torch.empty_like(qd)
        lse = torch.empty((xw.B, xw.Hq, xw.Sq), dtype=torch.float32, device=dev)

        def xstep():
            af.attn_fwd_ex(qd, kd, vd, o, lse, md, xw.per_head_mask, xw.causal, xw.window_left, -1, xw.scale)

        ms = launch_times(torch, dev, xstep, warmup, timed, None)
        af.attn_check()
        med = statistics.median(ms)
        p_tensor, _, _ = peaks()
        ach = xw.flops() / (med / 1e3) / 1e12
        rows[name] = {"ms_median": med, "ms_mean": statistics.mean(ms), "value": ach, "unit": "TFLOPS",
                      "bound": "tensor", "achieved": ach, "achieved_unit": "TFLOP/s", "frac": ach / p_tensor,
                      "B": xw.B, "Hq": xw.Hq, "Hkv": xw.Hkv, "Sq": xw.Sq, "Sk": xw.Sk, "d": xw.d,
                      "causal": xw.causal, "window_left": xw.window_left, "per_head_mask": xw.per_head_mask,
                      "flops": "4*d per kept (row, key) pair of the band, custom bits counted dense",
                      "extension": "attn_fwd_ex case (not one of the pages' configurations)",
                      "launches": timed * (3 if xw.per_head_mask else 1)}
        del qd, kd, vd, md, o, lse
        torch.cuda.empty_cache()
    for name, pw in inp.PACKED_WORKLOADS.items():
        # this library's extension: a packed variable-length batch, through attn_fwd_packed
        if names is not None and name not in names:
            continue
        q, k, v, cu = pw.make(1000 + len(pw.lengths))
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        cud = torch.from_numpy(cu).to(dev)
        o = torch.empty_like(qd)
        lse = torch.empty((pw.Hq, pw.total), dtype=torch.float32, device=dev)
        mx = max(pw.lengths)

        def pstep():
            af.attn_fwd_packed(qd, kd, vd, o, cud, cud, mx, mx, lse=lse, causal=pw.causal, scale=pw.scale)

        ms = launch_times(torch, dev, pstep, warmup, timed, None)
        af.attn_check()
        med = statistics.median(ms)
        p_tensor, _, _ = peaks()
        ach = pw.flops() / (med / 1e3) / 1e12
        rows[name] = {"ms_median": med, "ms_mean": statistics.mean(ms), "value": ach, "unit": "TFLOPS",
                      "bound": "tensor", "achieved": ach, "achieved_unit": "TFLOP/s", "frac": ach / p_tensor,
                      "lengths": list(pw.lengths), "Hq": pw.Hq, "Hkv": pw.Hkv, "d": pw.d, "causal": pw.causal,
                      "extension": "packed variable-length batch (not one of the pages' configurations)",
                      "launches": timed * 2}
        del qd, kd, vd, cud, o, lse
        torch.cuda.empty_cache()
    return rows


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if args.gpus != world:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch N>1 through torchrun")
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import attention_forward_07_gb300 as af
    af.library()  # fail loudly here if the CUDA library is missing
    if args.sweep_only:
        from attention_forward_07_gb300 import inputs as inp
        known = set(inp.WORKLOADS) | set(inp.EX_WORKLOADS) | set(inp.PACKED_WORKLOADS)
        if args.sweep_only not in known:
            raise SystemExit(f"--sweep-only: unknown workload {args.sweep_only!r}")
        rows = run_sweep(af, torch, dev, warmup=args.warmup, timed=args.steps, names={args.sweep_only})
        if rank == 0:
            print(json.dumps({"workload": args.sweep_only, "kernel": kernel_hash(), **rows[args.sweep_only]}))
        return 0
    w, idx = workload(args.workload, args.batch)
    seed = replica_seed(w.seed(idx), rank)
    (q, k, v, bits), t = device_inputs(torch, dev, w, seed)
    qd, kd, vd, md, o, lse = t
    flush = needs_flush(w)
    fbuf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
    live = live_fraction(w, bits)

    def step():
        af.attn_fwd(qd, kd, vd, o, lse, md, causal=w.causal, scale=w.scale)

    for _ in range(max(args.warmup, 0)):
        step()
    af.attn_check()

    sampler = ClockSampler(local, enabled=not args.no_clocks)
    time.sleep(0.4 if sampler.proc else 0)
    K = args.steps
    barrier(world)
    sampler.mark_start()
    per_launch_ms = launch_times(torch, dev, step, 0, K, fbuf)
    barrier(world)
    sampler.mark_end()
    af.attn_check()
    t_ms = sum(per_launch_ms)
    t_ms = max_over_ranks(t_ms, world, dev)
    clocks = sampler.stop() if sampler.proc else None
    value = world * w.flops() * K / (t_ms / 1e3) / 1e12

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(af, torch, dev, w, q, k, v, bits, o, lse, max(3, min(K, 20)), world, args.e2e_buffers)

    mean_ms, med_ms = statistics.mean(per_launch_ms), statistics.median(per_launch_ms)
    line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": t_ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": {0: "f16", 1: "bf16"}[w.dtype], "data": "synthetic",
            "config": config_dict(w, args.workload, world),
            "roofline": roofline(w, mean_ms / 1e3, live),
            "gpu_launches": K * kernels_per_step(w), "clocks": clocks, "e2e": e2e, "kernel": kernel_hash()}
    line["roofline"]["launch_ms_mean"] = mean_ms
    line["roofline"]["launch_ms_median"] = med_ms
    line["roofline"]["frac_of_median"] = line["roofline"]["frac"] * mean_ms / med_ms
    if kernels_per_step(w) > 1:
        # the events bracket the whole call (mask pre-pass, compaction, attention), so the
        # achieved rate is that of the step, a lower bound for the attention kernel's own
        line["roofline"]["timed"] = "whole step (mask pre-pass + compaction + attention kernel)"
    if w.mask != "none":
        line["tiles"] = skip_counts(af, torch, dev, w, t)
    del t, qd, kd, vd, md, o, lse, fbuf
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, seed, args.cpu_seconds)
        if w.B * w.Hq * w.S <= 4096:  # the tiny workload: also the whole oracle on one thread
            line["cpu_baseline"]["single_thread_value"] = cpu_single_thread(w, seed)
    else:
        line["cpu_baseline"] = None
    if world == 1 and not args.no_sweep:
        line["sweep"] = run_sweep(af, torch, dev)
        line["sweep_protocol"] = ("each workload: its seeded inputs, 10 warm-up launches, 50 timed launches (CUDA "
                                  "events per launch, L2 flushed between launches when a launch's data fits in "
                                  "twice the L2); value and frac from the median launch")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def measure_e2e(af, torch, dev, w, q, k, v, bits, o, lse, steps, world, nb=2):
    """Same metric through the public API with host buffers.  Every step copies its Q, K, V
    (and mask) from pinned host memory to the device, runs the forward, and copies O and LSE
    back; steps are pipelined the way a serving loop runs them: nb sets of device buffers,
    H2D copies on one stream, the forward on another, D2H copies on a third, so the copies
    of neighbouring steps overlap the current step's kernel.  The timed region runs
    from before the first H2D copy to the end of the last D2H copy."""
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    mh = None if bits is None else torch.from_numpy(bits.view(np.int32)).pin_memory()
    din = [[torch.empty_like(t, device=dev) for t in (qh, kh, vh)] + [None if mh is None else torch.empty_like(mh, device=dev)]
           for _ in range(nb)]
    dout = [(torch.empty_like(o), torch.empty_like(lse)) for _ in range(nb)]
    hout = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(), torch.empty(lse.shape, dtype=lse.dtype).pin_memory())
            for _ in range(nb)]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    cmp_done = [None] * nb
    out_done = [None] * nb

    def run(n):
        for i in range(n):
            b = i % nb
            with torch.cuda.stream(s_in):
                if cmp_done[b] is not None:
                    s_in.wait_event(cmp_done[b])  # inputs of step i-nb consumed
                for dst, src in zip(din[b], (qh, kh, vh, mh)):
                    if src is not None:
                        dst.copy_(src, non_blocking=True)
                in_done = ev()
                in_done.record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_done)
                if out_done[b] is not None:
                    s_cmp.wait_event(out_done[b])  # outputs of step i-nb copied out
                qd, kd, vd, md = din[b]
                af.attn_fwd(qd, kd, vd, dout[b][0], dout[b][1], md, causal=w.causal, scale=w.scale, stream=s_cmp)
                cmp_done[b] = ev()
                cmp_done[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[b])
                hout[b][0].copy_(dout[b][0], non_blocking=True)
                hout[b][1].copy_(dout[b][1], non_blocking=True)
                out_done[b] = ev()
                out_done[b].record(s_out)

    run(nb)
    torch.cuda.synchronize(dev)
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    s_cmp.wait_event(start)
    s_out.wait_event(start)
    run(steps)
    end.record(s_out)
    torch.cuda.synchronize(dev)
    af.attn_check(s_cmp)
    ms = max_over_ranks(start.elapsed_time(end), world, dev) / steps
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh)) + (0 if mh is None else mh.numel() * 4)
    d2h = o.numel() * o.element_size() + lse.numel() * 4
    return {"value": world * w.flops() / (ms / 1e3) / 1e12, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "pipelining": f"{nb} device buffer sets; H2D, forward and D2H on three streams"}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
