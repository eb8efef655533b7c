#!/usr/bin/env python3
"""Throughput benchmark of the fused exact-attention forward pass on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * C4: bf16, causal, B=1, H=16, N_q=N_k=16384, d=128   (attn_fwd)
  * C5: e4m3, non-causal, B=2, H=16, N_q=N_k=8192, d=128, per-(b,h) descales
        (attn_fwd_fp8_ws: V widened to fp16 once into a workspace, then the
        attention kernel; both launches are inside the timed step)
i.e. the bf16 + causal + FP8 variants the metric names.  FLOPs are counted as
4*B*H*N_q*N_k*d, halved for causal; value = counted TFLOP / device seconds.

Timing: W warm-up steps, then K steps bracketed by a barrier and
torch.cuda.synchronize(), timed with CUDA events on the launching stream; the
per-kernel events give each kernel's average duration (roofline).  Q/K/V of
one step are 288 MiB (> the 129 MB L2), so no L2 flush is needed.
Multi-GPU (torchrun): every rank runs its own shard (its own seeds), no
collective on the data path; value = all ranks' FLOPs / max-over-ranks time.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload: there is no upstream code to run, so the oracle is the reference arm.
"""

from __future__ import annotations

import argparse
import dataclasses
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

METRIC = "attention fwd TFLOPS and % of GB300 tensor peak at 1 GPU (bf16, causal, FP8)"
UNIT = "TFLOPS"
WORKLOAD = ("C4", "C5")
WORKLOAD_DESC = ("C4 bf16 causal B1 H16 N16384 d128 + C5 e4m3 non-causal B2 H16 N8192 d128 "
                 "(per-(b,h) descales, 0.1% x10 outliers); one attention call each per step")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 4.5 / 2.25     # nominal dense ratio
TC_SOURCES = ("io_aware_exact_03_gb300/csrc/attn_tc.cu", "io_aware_exact_03_gb300/csrc/tc_ptx.cuh",
              "io_aware_exact_03_gb300/csrc/bounded_wait.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_attn_tc_bf16_causal_d128.txt")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--sustained-s", type=float, default=1.5,
                    help="seconds of back-to-back steps for the sustained clock record (0: skip)")
    ap.add_argument("--case", choices=["C1", "C2", "C3", "C4", "C5", "LKV", "D256", "D256F", "BWD"], default=None,
                    help="measure one workload case alone instead of the C4 + C5 step")
    ap.add_argument("--splits", type=int, default=1,
                    help="with --case: split each query tile's K/V range over this many CTAs "
                         "(0: the count attn_splitkv_num_splits suggests for the case on this GPU)")
    return ap.parse_args()


def workload(args):
    """(case names, description) of one step."""
    if args.case:
        c = case_by_name(args.case)
        sp = f", split-KV over {args.splits} CTAs" if args.splits > 1 else ""
        return (args.case,), (f"{c.name} {c.dtype} {'causal' if c.causal else 'non-causal'} "
                              f"B{c.B} H{c.H} N_q{c.N_q} N_k{c.N_k} d{c.d}{sp}; one attention call per step")
    return WORKLOAD, WORKLOAD_DESC


# The backward pass does five matrix products per (query tile, key tile) pair
# (S, dP, dV, dK, dQ; the usual count) against the forward's two.
BWD_FLOP_FACTOR = 2.5


def launches_per_call(c, splits):
    """Kernels one call of case c launches: the backward pass three (prep, dk/dv,
    dq); split-KV the attention kernel and the combine; e4m3 at d <= 128 the V
    widening and the attention kernel (attn_fwd_fp8_ws); otherwise one."""
    if c.name == "BWD":
        return 3
    if splits > 1:
        return 2
    if c.dtype == "e4m3" and c.d in (64, 128) and c.N_k > 0:
        return 2
    return 1


def work_flops(c):
    """Counted FLOPs of one call on case c (forward, or backward for BWD)."""
    return c.flops * BWD_FLOP_FACTOR if c.name == "BWD" else c.flops


def case_by_name(name):
    import synthetic
    return synthetic.CASES.get(name) or synthetic.EXTRA_CASES[name]


# ------------------------------------------------------- multi-rank helpers
def shard_seed(case_seed: int, rank: int) -> int:
    """Each rank draws its own shard of (batch, head) work: seed offset by rank."""
    return case_seed + 100 * rank


def max_over_ranks(torch, dist, ms: float, device) -> float:
    """The slowest rank's time (the job is done when every rank is done)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step: float, steps: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank's FLOPs over the slowest rank's time."""
    return world * flops_per_rank_step * steps / (ms_max / 1e3) / 1e12


def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def tc_source_sha():
    h = hashlib.sha256()
    for rel in TC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def read_traffic():
    """dram bytes per C4 launch from the committed ncu summary, if the kernel is unchanged."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256") != tc_source_sha():
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 20 ms, each with its own timestamp; only the
    samples that fall inside the timed region are reported."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out_path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")
        self.window = None

    def start(self):
        """Start sampling; returns once the first sample has been written."""
        try:
            self.fh = open(self.out_path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0:
            time.sleep(0.02)
            try:
                if os.path.getsize(self.out_path) > 0:
                    break
            except OSError:
                pass

    def mark(self, t0: float, t1: float):
        """Host wall-clock bounds of the timed region."""
        self.window = (t0, t1)

    @staticmethod
    def _stamp(text):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.out_path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.remove(self.out_path)
        if self.window is not None:
            t0, t1 = self.window
            inside = [r for r in rows if (ts := self._stamp(r[0])) is not None and t0 <= ts <= t1]
        else:
            inside = rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no sample inside the timed region"],
                    "samples": 0}
        num = lambda x: x.replace(".", "").isdigit()
        sm = [float(r[1]) for r in inside if num(r[1])]
        smax = [float(r[2]) for r in inside if num(r[2])]
        power = [float(r[3]) for r in inside if num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside),
                "power_w_median": statistics.median(power) if power else None,
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------ CPU oracle leg
def oracle_rows_rate(counts, seed):
    """Time the fp64 CPU oracle on sampled rows of the named cases; returns (flops, seconds, threads)."""
    import numpy as np
    import oracle
    import synthetic

    threads = oracle.default_threads()
    flops = 0.0
    secs = 0.0
    for j, (name, n) in enumerate(counts.items()):
        case = case_by_name(name)
        q, k, v = _f64_inputs(name)
        rows = synthetic.sample_rows(case, n, seed=seed + 7 * j)
        keys = np.array([_allowed(case, int(i)) for i in rows[:, 2]], dtype=np.float64)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, case.scale, case.causal, rows, n_threads=threads)
        secs += time.perf_counter() - t0
        flops += float((4.0 * case.d * keys).sum())
    return flops, secs, threads


_F64 = {}


def _f64_inputs(name):
    if name not in _F64:
        import oracle
        import synthetic
        _F64[name] = oracle.case_inputs_f64(synthetic.make_inputs(case_by_name(name)))
    return _F64[name]


def _allowed(case, i):
    if not case.causal:
        return case.N_k
    return max(0, min(case.N_k, i + case.N_k - case.N_q + 1))


def cpu_baseline(names, target_s=12.0):
    # enough rows that every thread has several (a few rows per thread
    # understate the rate, and the scaled run would fall short of target_s)
    base = {n: (512 if i == 0 else 256) for i, n in enumerate(names)}
    for n in names:
        _f64_inputs(n)
    f, s, thr = oracle_rows_rate(base, seed=11)                # calibration
    scale = max(1.0, target_s / max(s, 1e-3))
    counts = {n: int(c * scale) for n, c in base.items()}
    f, s, thr = oracle_rows_rate(counts, seed=12)
    desc = " and ".join(f"{c} of {n}" for n, c in counts.items())
    return {"value": f / s / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"seeded query rows ({desc}; full key range each), fp64 one-pass oracle, "
                      f"{s:.1f} s"}


# ----------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    import io_aware_exact_03_gb300 as attn
    import synthetic

    rank, world, local = env_rank()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    attn.build()
    attn.lib()
    if args.splits == 0:
        c0 = case_by_name(args.case) if args.case else None
        args.splits = attn.attn_splitkv_num_splits(c0.B, c0.H, c0.N_q, c0.N_k, c0.d) if c0 else 1

    names, desc = workload(args)
    cases = [case_by_name(n) for n in names]
    host, dev, outs = [], [], []
    bwd_ws = None
    for c in cases:
        c_r = dataclasses.replace(c, seed=shard_seed(c.seed, rank))
        inp = synthetic.make_inputs(c_r)
        d_in = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        out_dtype = torch.float16 if c.dtype == "fp16" else torch.bfloat16
        if c.name == "BWD":
            # inputs of the backward pass: q, k, v, the forward's o and lse, dO
            o, lse = attn.attn_fwd(d_in["q"], d_in["k"], d_in["v"], scale=c.scale, causal=c.causal)
            d_in.update(o=o, lse=lse, dO=synthetic.make_grad(c_r).cuda())
            inp = dict(inp, o=o.cpu(), lse=lse.cpu(), dO=d_in["dO"].cpu())
            outs.append((torch.empty_like(d_in["q"]), torch.empty_like(d_in["k"]),
                         torch.empty_like(d_in["v"])))
            bwd_ws = torch.empty(attn.attn_bwd_workspace_bytes(c.B, c.H, c.N_q), dtype=torch.uint8,
                                 device="cuda")
        else:
            outs.append((torch.empty((c.B, c.N_q, c.H, c.d), dtype=out_dtype, device="cuda"),
                         torch.empty((c.B, c.H, c.N_q), dtype=torch.float32, device="cuda")))
        host.append(inp)
        dev.append(d_in)
    stream = torch.cuda.current_stream()
    ws = None
    if args.splits > 1:
        need = max(attn.attn_splitkv_workspace_bytes(c.B, c.H, c.N_q, c.d, args.splits) for c in cases)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    # e4m3 cases: the fp16 copy of V (attn_fwd_fp8_ws), allocated once like any workspace
    fp8_ws = {i: torch.empty(max(1, attn.attn_fwd_fp8_workspace_bytes(c.B, c.H, c.N_k, c.d)),
                             dtype=torch.uint8, device="cuda")
              for i, c in enumerate(cases) if c.dtype == "e4m3" and c.name != "BWD"}

    def call(i, d):
        c = cases[i]
        if c.name == "BWD":
            dq, dk, dv = outs[i]
            attn.attn_bwd(d["q"], d["k"], d["v"], d["o"], d["lse"], d["dO"], scale=c.scale,
                          causal=c.causal, dq=dq, dk=dk, dv=dv, workspace=bwd_ws, stream=stream)
            return
        o, lse = outs[i]
        if args.splits > 1:
            attn.attn_fwd_splitkv(d["q"], d["k"], d["v"], args.splits, o=o, lse=lse,
                                  scale=c.scale, causal=c.causal, q_descale=d.get("q_descale"),
                                  k_descale=d.get("k_descale"), v_descale=d.get("v_descale"),
                                  workspace=ws, stream=stream)
        elif c.dtype == "e4m3":
            attn.attn_fwd_fp8_ws(d["q"], d["k"], d["v"], d["q_descale"], d["k_descale"],
                                 d["v_descale"], o=o, lse=lse, scale=c.scale, causal=c.causal,
                                 workspace=fp8_ws[i], stream=stream)
        else:
            attn.attn_fwd(d["q"], d["k"], d["v"], o=o, lse=lse, scale=c.scale,
                          causal=c.causal, stream=stream)

    for _ in range(args.warmup):
        for i in range(len(cases)):
            call(i, dev[i])
    attn.attn_check_status()

    K = args.steps
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)] for _ in cases]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    gpu_id = _gpu_id(torch, local)
    sampler = ClockSampler(gpu_id)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.time()
    t_start.record(stream)
    for s in range(K):
        for i in range(len(cases)):
            ev[i][s][0].record(stream)
            call(i, dev[i])
            ev[i][s][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    sampler.mark(wall0, time.time())
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    attn.attn_check_status()
    ms_total = max_over_ranks(torch, dist, t_start.elapsed_time(t_end), "cuda")
    kern_ms = [statistics.fmean(a.elapsed_time(b) for a, b in ev[i]) for i in range(len(cases))]
    flops_step = sum(work_flops(c) for c in cases)
    value = job_tflops(flops_step, K, world, ms_total)

    # ---- the same step back to back for a sustained period (>= 1.5 s), with
    # its own clock record: the short timed region above cannot show the
    # power draw and the clock a long run settles at.
    sustained = None
    if args.sustained_s > 0:
        sustained = run_sustained(torch, cases, dev, call, stream, gpu_id, ms_total / K,
                                  work_flops_step=sum(work_flops(c) for c in cases),
                                  seconds=args.sustained_s)

    # ---- end to end through the public API: pinned host -> device -> kernel -> host
    e2e = run_e2e(torch, attn, cases, host, outs, stream, args.e2e_steps, call, world,
                  host_api=args.splits <= 1)

    peaks, peak_src = read_peaks()
    bf16_peak = peaks["bf16_tflops"]
    fp8_peak = bf16_peak * FP8_OVER_BF16
    per_kernel = {}
    for i, c in enumerate(cases):
        ach = work_flops(c) / (kern_ms[i] / 1e3) / 1e12
        pk = fp8_peak if c.dtype == "e4m3" else bf16_peak
        per_kernel[c.name] = {"dtype": c.dtype, "causal": c.causal, "ms": round(kern_ms[i], 4),
                              "tflops": round(ach, 1), "peak_tflops": round(pk, 1),
                              "frac_of_peak": round(ach / pk, 4)}
    dom = max(range(len(cases)), key=lambda i: kern_ms[i])
    dc = cases[dom]
    dom_peak = fp8_peak if dc.dtype == "e4m3" else bf16_peak
    dom_ach = work_flops(dc) / (kern_ms[dom] / 1e3) / 1e12
    traffic = read_traffic() if (dc.name == "C4" and len(cases) == 2) else None
    roofline = {"bound": "tensor", "achieved": round(dom_ach, 1), "peak": round(dom_peak, 1),
                "unit": "TFLOP/s", "frac": round(dom_ach / dom_peak, 4), "traffic": traffic,
                "kernel": (f"attn_bwd: bwd_prep + bwd_dkdv + bwd_dq ({dc.dtype}, causal={dc.causal})"
                           if dc.name == "BWD" else f"attn_tc_kernel {dc.name} ({dc.dtype}, causal={dc.causal})"),
                "peak_source": f"{peak_src} bf16 burst" + (" x 2 (fp8/bf16 nominal)" if dc.dtype == "e4m3" else ""),
                "algorithmic_flops_per_launch": work_flops(dc)}
    # mixed roofline of the whole step: time at peak for each kernel over actual time
    t_peak = sum(work_flops(c) / ((fp8_peak if c.dtype == "e4m3" else bf16_peak) * 1e12) for c in cases)
    step_frac = t_peak / (ms_total / K / 1e3)

    result = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(names)
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_total / K, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16,e4m3", "data": "synthetic (seeded N(0,1); C5 with 0.1% x10 outliers)",
            "config": {"workload": desc, "global_batch": sum(c.B * c.H for c in cases) * world,
                       "seq_len": [c.N_q for c in cases], "parallelism": f"dp{world} (independent shards)",
                       "l2": f"Q/K/V of one step: {sum(3 * c.B * c.H * c.N_q * c.d * (1 if c.dtype == 'e4m3' else 2) for c in cases) / 2**20:.0f} MiB (L2 is 129 MB); no flush"},
            "pct_of_tensor_peak_step": round(100 * step_frac, 2),
            "per_kernel": per_kernel,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "sustained": sustained,
            "gpu_launches": sum(launches_per_call(c, args.splits) for c in cases) * K,
            "clocks": clocks,
        }
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def run_sustained(torch, cases, dev, call, stream, gpu_id, ms_step, work_flops_step,
                  seconds=1.5):
    """Back-to-back steps for about `seconds`, timed with CUDA events, with
    nvidia-smi clock / power samples taken inside that window.  Reported
    beside the short timed region; it does not replace `value`."""
    n = max(20, int(seconds * 1e3 / max(ms_step, 1e-3)) + 1)
    sampler = ClockSampler(gpu_id)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.time()
    a.record(stream)
    for _ in range(n):
        for i in range(len(cases)):
            call(i, dev[i])
    b.record(stream)
    torch.cuda.synchronize()
    sampler.mark(wall0, time.time())
    clocks = sampler.stop()
    ms = a.elapsed_time(b)
    return {"steps": n, "seconds": round(ms / 1e3, 3), "ms_per_step": round(ms / n, 4),
            "value": round(work_flops_step * n / (ms / 1e3) / 1e12, 2), "unit": UNIT,
            "clocks": clocks}


def run_e2e(torch, attn, cases, host, outs, stream, steps, call, world, host_api=True):
    """The step end to end from pinned host memory.  Forward cases go through
    attn_fwd_host (copies to and from the device pipelined against the kernel
    over chunks of heads, inside the library); the backward case copies its
    inputs in, runs, and copies the gradients out on the stream."""
    steps = max(1, steps)
    pinned = []
    h2d = d2h = 0
    for i, c in enumerate(cases):
        hp = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in host[i].items()}
        use_host = host_api and c.name != "BWD"
        if use_host:
            names = ["q", "k", "v"] + (["q_descale", "k_descale", "v_descale"] if c.dtype == "e4m3" else [])
            hp = {k: hp[k].contiguous() for k in names}
            dd = torch.empty(attn.attn_fwd_host_workspace_bytes(c.B, c.H, c.N_q, c.N_k, c.d,
                                                                {"bf16": 0, "fp16": 1, "e4m3": 2}[c.dtype]),
                             dtype=torch.uint8, device="cuda")
        else:
            dd = {k: (torch.empty_like(v, device="cuda") if isinstance(v, torch.Tensor) else v)
                  for k, v in hp.items()}
        hout = [torch.empty_like(t, device="cpu").pin_memory() for t in outs[i]]
        pinned.append((use_host, hp, dd, hout))
        h2d += sum(v.numel() * v.element_size() for v in hp.values() if isinstance(v, torch.Tensor))
        d2h += sum(t.numel() * t.element_size() for t in outs[i])

    # The step's independent forward calls go on a stream each, and steps are
    # issued back to back, as a server issues requests: each call's stream
    # orders its own steps (a call's copies start after the same call of the
    # step before has been copied out), and the library's copy streams queue
    # one call's transfers right behind the other's, so the host link stays
    # busy while a call finishes its last chunk.  The caller's stream waits for
    # every step at the end of the timed region.
    side = [torch.cuda.Stream() for _ in cases]
    fork = torch.cuda.Event()
    joins = [torch.cuda.Event() for _ in cases]

    def issue_step():
        for i, c in enumerate(cases):
            use_host, hp, dd, hout = pinned[i]
            if use_host:
                attn.attn_fwd_host(hp["q"], hp["k"], hp["v"], o=hout[0], lse=hout[1], scale=c.scale,
                                   causal=c.causal, q_descale=hp.get("q_descale"),
                                   k_descale=hp.get("k_descale"), v_descale=hp.get("v_descale"),
                                   workspace=dd, stream=side[i])
                continue
            for k, v in hp.items():
                if isinstance(v, torch.Tensor):
                    dd[k].copy_(v, non_blocking=True)
            call(i, dd)
            for h, t in zip(hout, outs[i]):
                h.copy_(t, non_blocking=True)

    def run_steps(n):
        fork.record(stream)
        for s in side:
            s.wait_event(fork)
        for _ in range(n):
            issue_step()
        for i in range(len(cases)):
            joins[i].record(side[i])
            stream.wait_event(joins[i])

    run_steps(1)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run_steps(steps)
    b.record(stream)
    torch.cuda.synchronize()
    attn.attn_check_status()
    import torch.distributed as dist
    ms = max_over_ranks(torch, dist, a.elapsed_time(b), "cuda")
    flops = sum(work_flops(c) for c in cases)
    return {"value": round(job_tflops(flops, steps, world, ms), 2), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": round(ms / steps, 4),
            "path": ("attn_fwd_host per forward call (pinned host buffers; copies pipelined with the "
                     "kernel inside the library), one stream per call, steps issued back to back and "
                     "joined at the end"
                     if any(p[0] for p in pinned) else "copies and the call on one stream")}


def _gpu_id(torch, local):
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[local]
        return str(local)


# ----------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = env_rank()
    if rank != 0:
        return None
    import oracle
    names, desc = workload(args)
    counts = {n: (32 if i == 0 else 16) for i, n in enumerate(names)}
    for n in names:
        _f64_inputs(n)
    for s in range(args.warmup):
        oracle_rows_rate(counts, seed=1000 + s)
    flops = secs = 0.0
    thr = oracle.default_threads()
    for s in range(args.steps):
        f, t, thr = oracle_rows_rate(counts, seed=5000 + s)
        flops += f
        secs += t
    value = flops / secs / 1e12
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1); C5 with 0.1% x10 outliers)",
        "config": {"workload": desc, "parallelism": "CPU host cores, rank 0 only"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                         "sample": "per step " + " and ".join(f"{c} seeded query rows of {n}" for n, c in counts.items())
                                   + " (full key range), fp64 one-pass oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)
    return result


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
