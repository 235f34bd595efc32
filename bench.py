"""Benchmark of the exact-attention hot path (fa_fwd + fa_bwd) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...      # the float64 CPU oracle, timed
    python bench.py --workload decode32k      # the split-KV decode path (its own line)
    python bench.py --workload sparse8k       # the block-sparse forward (its own line)
    python bench.py --workload fp8_8k         # the FP8 (e4m3) forward (its own line)

A step is one training forward plus one backward pass over one batch of the
workload (default: B4 Hq32 Hkv8 N8192 d128 causal -- the N >= 8192, d = 128
regime), inputs resident in HBM.  Timing: CUDA events on the launching stream
around each kernel, L2 flushed (a 256 MiB write) before every step outside
the timed events, the K timed steps bracketed by a barrier and a synchronize,
max over ranks.  Prints one JSON line.

Multi-GPU: the path shards into independent (batch, kv-head group) problems,
so N ranks each run their own batch with no data-path collective ("weak"
scaling); the only collective is the max of the timings.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import fa_workloads as W  # noqa: E402

METRIC = "attention fwd/bwd TFLOPS and % of GB300 BF16 tensor peak at N=2k–128k, d=64/128"
SPARSE_METRIC = ("block-sparse attention forward: TFLOPS of the computed 128x128 blocks and % of "
                 "GB300 BF16 tensor peak")
# block-sparse forward: the gqa8k shape with a synthetic block mask
SPARSE_WORKLOADS = {"sparse8k": ("gqa8k", 24)}
FP8_METRIC = ("FP8 (e4m3) attention forward: nominal TFLOPS (4*B*H*N^2*d, halved causal) and % of "
              "GB300 FP8 tensor peak (measured bf16 peak x the nominal fp8/bf16 ratio 2)")
FP8_WORKLOADS = {"fp8_8k": "gqa8k"}
DECODE_METRIC = ("split-KV decode attention: GB/s of the compulsory HBM bytes (K, V, Q, O, lse) "
                 "and % of the measured HBM copy bandwidth")
DEFAULT_WORKLOAD = "gqa8k"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


def rank_workload(base: W.Workload, rank: int) -> W.Workload:
    """Rank r's share under weak scaling: the same workload shape, its own
    batch (seed offset by 1000 * r)."""
    return base.with_(seed=base.seed + 1000 * rank)


def aggregate(step_ms_local: float, flops_per_rank: float, world_size: int, reduce_max=None):
    """Whole-job throughput: the units all ranks processed divided by the
    slowest rank's time.  reduce_max maps a local float to the max over ranks
    (None for one process)."""
    slowest = reduce_max(step_ms_local) if reduce_max else step_ms_local
    return world_size * flops_per_rank / (slowest * 1e-3) / 1e12, slowest


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons (every 100 ms) and keeps
    the samples whose timestamps fall inside the timed window."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.window = None

    def start(self):
        # the raw samples are kept in FA_BENCH_CLOCKS_DIR when it is set, else
        # in a temporary file removed once the summary is taken
        try:
            keep = os.environ.get("FA_BENCH_CLOCKS_DIR")
            d = keep or tempfile.gettempdir()
            os.makedirs(d, exist_ok=True)
            self.keep = bool(keep)
            self.path = os.path.join(d, f"clocks_{os.getpid()}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        from datetime import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]),
                                 [n for n, v in zip(names, parts[6:10]) if v.lower() == "active"]))
                except ValueError:
                    continue
        if not self.keep:
            os.remove(self.path)
        if not rows:
            return None
        inside = [r for r in rows if self.window and self.window[0] <= r[0] <= self.window[1]]
        use = inside if inside else rows
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted({n for r in use for n in r[3]}),
                "samples": len(use), "window": "timed region" if inside else "whole run"}


def oracle_sample(w: W.Workload, heads: int):
    """A bounded, self-contained piece of the workload for the CPU oracle: one
    batch element drawn with the workload's recipe, key/value head 0 and the
    first `heads` query heads of its group, full sequence.  Returns (inputs,
    nominal FLOPs, description)."""
    heads = max(1, min(heads, w.Hq // w.Hkv))
    x = W.make_inputs(w.with_(B=1))
    sub = {"q": x["q"][:1, :, :heads].contiguous(), "k": x["k"][:1, :, :1].contiguous(),
           "v": x["v"][:1, :, :1].contiguous(), "dout": x["dout"][:1, :, :heads].contiguous()}
    sw = w.with_(B=1, Hq=heads, Hkv=1)
    flops = W.fwd_flops(sw) + (W.bwd_flops(sw) if w.backward else 0.0)
    step = W.fwd_flops(w) + (W.bwd_flops(w) if w.backward else 0.0)
    desc = (f"one batch element, kv head 0 with {heads} query head(s), full N={w.N}, "
            f"{'fwd+bwd' if w.backward else 'fwd'} ({flops / 1e9:.1f} nominal GFLOP, "
            f"{flops / step:.4g} of a step)")
    return sub, flops, desc


def time_oracle_once(sub, w: W.Workload) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.attn_fwd(sub["q"], sub["k"], sub["v"], w.causal, w.scale)
    if w.backward:
        oracle.attn_bwd(sub["q"], sub["k"], sub["v"], sub["dout"], w.causal, w.scale)
    return time.perf_counter() - t0


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = W.WORKLOADS[args.workload]
    sub, flops, desc = oracle_sample(w, heads=1)
    oracle.build()
    for _ in range(args.warmup):
        time_oracle_once(sub, w)
    times = [time_oracle_once(sub, w) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms * 1e-3) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.workload, "shape": W.describe(w), "sample": desc},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def tensor_bytes(*ts) -> int:
    return sum(t.numel() * t.element_size() for t in ts)


# event-timed slots of a step.  The forward slot of a training step is the
# fa_fwd_train call: the maxima and fp16 copies of q, k, v (f16_absmax_kernel,
# f16_convert_kernel), then fa_fwd_kernel -- three launches, named for the
# call; a forward-only workload times the fa_fwd call, one fa_fwd_kernel.
# The backward's slots are the fa_bwd_stage steps: D with max |dO|, dQ (which
# also writes the fp16 copy of dO), dK/dV.
FWD_TRAIN_SLOT = "fa_fwd_train_call"
KERNELS = (FWD_TRAIN_SLOT, "fa_bwd_dsum_kernel", "fa_bwd_dq_kernel", "fa_bwd_dkdv_kernel")
KERNEL_SOURCES = {"fa_fwd_kernel": "fa_fwd.cu", FWD_TRAIN_SLOT: "fa_fwd.cu",
                  "fa_bwd_dsum_kernel": "fa_bwd.cu",
                  "fa_decode_split_kernel": "fa_decode.cu", "fa_fp8_fwd_kernel": "fa_fp8.cu",
                  "fa_bwd_dkdv_kernel": "fa_bwd_dkdv.cu", "fa_bwd_dq_kernel": "fa_bwd_dq.cu"}
LAUNCHES = {FWD_TRAIN_SLOT: 3, "fa_fwd_kernel": 1, "fa_bwd_dsum_kernel": 1,
            "fa_bwd_dkdv_kernel": 1, "fa_bwd_dq_kernel": 1}
# the arithmetic of the training step, which the "dtype" key names
TRAIN_DTYPE = "bf16 I/O; P, dS as fp16 against exact scaled fp16 copies; fp32 accumulate"


def kernel_work(w: W.Workload, name: str):
    """(bound, algorithmic work per launch) of one kernel at workload w.
    Tensor kernels: FLOPs of the GEMMs the kernel must do (2*N^2*d per head per
    GEMM, halved under the causal mask): fwd 2 GEMMs, dK/dV 4, dQ 3.  dsum:
    bytes of O, o_lo and dO read plus D written."""
    g1 = W.fwd_flops(w) / 2.0  # one N x N x d GEMM over all heads
    if name in ("fa_fwd_kernel", FWD_TRAIN_SLOT):
        return "tensor", 2 * g1
    if name == "fa_bwd_dkdv_kernel":
        return "tensor", 4 * g1
    if name == "fa_bwd_dq_kernel":
        return "tensor", 3 * g1
    # dsum slot: read dO, O, o_lo (max |dO| on the way); write D
    return "hbm", 3 * w.B * w.N * w.Hq * w.d * 2 + 4 * w.B * w.Hq * w.N


def source_hash(name: str) -> str:
    """Hash of the code (comments and whitespace removed) of a kernel's source
    file and the shared headers: the stored DRAM counts stay valid across
    edits that change only comments."""
    import hashlib
    import re
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "exact_io_aware_35_gb300", "csrc")
    for f in (KERNEL_SOURCES[name], "sm103_ptx.cuh", "fa_internal.h", "fa_bwd_common.cuh"):
        with open(os.path.join(csrc, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def measured_traffic(name: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t[workload][name]
        return e["dram_bytes_per_launch"] if e.get("source_hash") == source_hash(name) else None
    except Exception:
        return None


def roofline(w: W.Workload, kern_ms: dict, peaks: dict):
    name = max(kern_ms, key=kern_ms.get)  # dominant kernel by measured time
    bound, work = kernel_work(w, name)
    ms = kern_ms[name]
    if bound == "tensor":
        achieved = work / (ms * 1e-3) / 1e12
        peak, unit = peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved = work / (ms * 1e-3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    return {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": peaks["source"] + " burst",
            "launch_ms": ms, "algorithmic_work_per_launch": work,
            "traffic": measured_traffic(name, w.name)}


def run_gpu(args):
    import exact_io_aware_35_gb300 as fa
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks = load_peaks()
    base = W.WORKLOADS[args.workload]
    if args.batch:
        base = base.with_(B=args.batch)
    w = rank_workload(base, rank)
    x = W.make_inputs(w, with_dout=w.backward)
    host = {n: t.pin_memory() for n, t in x.items()}
    dvc = {n: t.to(dev) for n, t in host.items()}
    q, k, v = dvc["q"], dvc["k"], dvc["v"]
    do = dvc.get("dout")
    o = torch.empty_like(q)
    o_lo = torch.empty_like(q) if w.backward else None  # training forward
    lse = torch.empty((w.B, w.Hq, w.N), device=dev, dtype=torch.float32)
    if w.backward:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wsb = torch.empty(fa.fa_bwd_workspace_size(w.B, w.Hq, w.Hkv, w.N, w.d), dtype=torch.uint8,
                          device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > 129 MB of L2
    nk = 1 + (3 if w.backward else 0)  # timed slots per step

    def fwd():
        fa.fa_fwd(q, k, v, causal=w.causal, scale=w.scale, o=o, lse=lse, o_lo=o_lo,
                  workspace=wsb if w.backward else None)

    # the training pair on one workspace: fa_fwd_train leaves the fp16 copies of
    # q, k, v there, so the backward copies only dout
    def bwd(stages=fa.FA_BWD_AFTER_FWD_TRAIN):
        fa.fa_bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, dq=dq, dk=dk, dv=dv,
                  workspace=wsb, stages=stages, o_lo=o_lo)

    # the backward's slots, in the order of KERNELS[1:]
    bwd_stages = (fa.FA_BWD_PREP_DOUT | fa.FA_BWD_DSUM, fa.FA_BWD_DQ, fa.FA_BWD_DKDV)
    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        fwd()
        if w.backward:
            bwd()
    st = fa.fa_get_device_error()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {fa.status_string(st)} during warm-up")

    # timed steps: events between the kernels (fwd | dsum | dQ | dK,dV) so each
    # kernel's duration is measured on the stream it runs on
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(K)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_timed0 = time.time()
    for i in range(K):
        flush.zero_()
        ev[i][0].record()
        fwd()
        ev[i][1].record()
        if w.backward:
            for n, stage in enumerate(bwd_stages):
                bwd(stage)
                ev[i][2 + n].record()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    st = fa.fa_get_device_error()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {fa.status_string(st)} in the timed region")
    kern_ms = [sum(ev[i][n].elapsed_time(ev[i][n + 1]) for i in range(K)) / K for n in range(nk)]
    fwd_ms = kern_ms[0]
    bwd_ms = sum(kern_ms[1:])
    step_ms = fwd_ms + bwd_ms

    # ---- end to end through the public API, inputs from pinned host memory
    outs = {"o": o, "lse": lse}
    if w.backward:
        outs.update({"dq": dq, "dk": dk, "dv": dv})
    h2d = tensor_bytes(*host.values())
    d2h = tensor_bytes(*outs.values())
    # two device sets of the step's inputs and results; the fp16 copies and D
    # (workspace) and o_lo live within one step on the compute stream
    sets = [dict(dvc, **outs),
            {n: torch.empty_like(t) for n, t in list(dvc.items()) + list(outs.items())}]
    out_host = [{n: torch.empty_like(t, device="cpu").pin_memory() for n, t in outs.items()}
                for _ in sets]

    def compute(s):
        fa.fa_fwd(s["q"], s["k"], s["v"], causal=w.causal, scale=w.scale, o=s["o"], lse=s["lse"],
                  o_lo=o_lo, workspace=wsb if w.backward else None)
        if w.backward:
            fa.fa_bwd(s["q"], s["k"], s["v"], s["o"], s["dout"], s["lse"], causal=w.causal,
                      scale=w.scale, dq=s["dq"], dk=s["dk"], dv=s["dv"], workspace=wsb,
                      stages=fa.FA_BWD_AFTER_FWD_TRAIN, o_lo=o_lo)

    def e2e_serial(i):
        s = sets[0]
        for n, t in host.items():
            s[n].copy_(t, non_blocking=True)
        compute(s)
        for n in outs:
            out_host[0][n].copy_(s[n], non_blocking=True)

    # pipelined: the upload of step i+1 and the download of step i run on
    # their own streams while step i's kernels run; events order each buffer
    # set's reuse (upload after the kernels of step i-2 have read it, kernels
    # after the download of step i-2 has read the results)
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    done = [None, None]     # kernels of the set's last step finished
    fetched = [None, None]  # download of the set's last results finished

    def e2e_pipelined(i):
        b = i & 1
        s = sets[b]
        with torch.cuda.stream(up):
            if done[b] is not None:
                up.wait_event(done[b])
            for n, t in host.items():
                s[n].copy_(t, non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(up)
        comp.wait_event(loaded)
        if fetched[b] is not None:
            comp.wait_event(fetched[b])
        compute(s)
        done[b] = torch.cuda.Event()
        done[b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(done[b])
            for n in outs:
                out_host[b][n].copy_(s[n], non_blocking=True)
            fetched[b] = torch.cuda.Event()
            fetched[b].record(down)

    def time_e2e(step):
        step(0)
        step(1)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        up.wait_event(e0)  # no copy starts before the timed region
        for i in range(K):
            step(i)
        for f in fetched:
            if f is not None:
                comp.wait_event(f)  # the last download is inside the region
        e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    e2e_serial_ms = time_e2e(e2e_serial)
    e2e_ms = time_e2e(e2e_pipelined)
    clocks.mark(t_timed0, time.time())
    clk = clocks.stop()

    flops_step = W.fwd_flops(w) + (W.bwd_flops(w) if w.backward else 0.0)
    t = torch.tensor([step_ms, e2e_ms, e2e_serial_ms] + kern_ms, dtype=torch.float64, device=dev)
    if ws > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    vals = [float(u) for u in t.tolist()]
    step_ms, e2e_ms, e2e_serial_ms, kern_ms = vals[0], vals[1], vals[2], vals[3:]
    fwd_ms, bwd_ms = kern_ms[0], sum(kern_ms[1:])
    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0

    peak = peaks["bf16_tflops"]
    slots = KERNELS[:nk] if w.backward else ("fa_fwd_kernel",)
    value, _ = aggregate(step_ms, flops_step, ws)
    fwd_tf = W.fwd_flops(w) / (fwd_ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": TRAIN_DTYPE if w.backward else "bf16 (bf16 P; fp32 accumulate)",
            "data": "synthetic (seeded N(0,1) bf16, shape of the workload)",
            "config": {"workload": args.workload, "shape": W.describe(w),
                       "global_batch": w.B * ws, "seq_len": w.N,
                       "parallelism": f"replicas x{ws} (independent batches, no collective)",
                       "l2": "flushed by a 256 MiB write before every timed step"},
            "frac_of_peak": value / ws / peak,
            "fwd_tflops": fwd_tf, "fwd_frac_of_peak": fwd_tf / peak, "fwd_ms": fwd_ms,
            "peak_tflops": peak, "peak_source": peaks["source"] + " burst bf16",
            "gpu_launches": K * sum(LAUNCHES[n] for n in slots)}
    if w.backward:
        bwd_tf = W.bwd_flops(w) / (bwd_ms * 1e-3) / 1e12
        line.update({"bwd_tflops": bwd_tf, "bwd_frac_of_peak": bwd_tf / peak, "bwd_ms": bwd_ms})
    km = dict(zip(slots, kern_ms))
    line["kernel_ms"] = km
    line["roofline"] = roofline(w, km, peaks)
    line["e2e"] = {"value": aggregate(e2e_ms, flops_step, ws)[0], "unit": "TFLOPS",
                   "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "overlap": "upload of step i+1 and download of step i on their own streams "
                              "during step i's kernels (two device buffer sets); every step's "
                              "copies inside the timed region",
                   "serial_ms_per_step": e2e_serial_ms,
                   "serial_value": aggregate(e2e_serial_ms, flops_step, ws)[0]}
    if clk is not None:
        line["clocks"] = clk
    if ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        sub, sflops, desc = oracle_sample(base, heads=base.Hq // base.Hkv)
        secs = time_oracle_once(sub, base)
        line["cpu_baseline"] = {"value": sflops / secs / 1e12, "unit": "TFLOPS",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": desc, "seconds": secs}
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def decode_oracle_sample(w: W.DecodeWorkload):
    """Batch element 0 of the decode workload (all heads) for the CPU oracle."""
    x = W.make_decode_inputs(w.with_(B=1))
    sw = w.with_(B=1)
    flops = W.decode_flops(sw)
    desc = (f"batch element 0 of {w.B}, all {w.Hq} heads, Nq={w.Nq}, Nk={w.Nk} "
            f"({flops / 1e9:.2f} nominal GFLOP, {1 / w.B:.4g} of a step)")
    return x, flops, desc


def time_decode_oracle(x, w: W.DecodeWorkload) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.attn_fwd_kv(x["q"], x["k"], x["v"], w.causal, w.scale)
    return time.perf_counter() - t0


def run_decode_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = W.DECODE_WORKLOADS[args.workload]
    x, flops, desc = decode_oracle_sample(w)
    oracle.build()
    for _ in range(args.warmup):
        time_decode_oracle(x, w)
    times = [time_decode_oracle(x, w) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    gbs = W.decode_min_bytes(w.with_(B=1)) / (ms * 1e-3) / 1e9
    line = {"impl": "reference", "metric": DECODE_METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.workload, "shape": W.describe_decode(w), "sample": desc},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_decode(args):
    """One step = one fa_fwd_splitkv call (split kernel + combine kernel) over
    the decode workload, inputs resident in HBM, L2 flushed before each."""
    import exact_io_aware_35_gb300 as fa
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks = load_peaks()
    base = W.DECODE_WORKLOADS[args.workload]
    if args.batch:
        base = base.with_(B=args.batch)
    w = base.with_(seed=base.seed + 1000 * rank)
    x = W.make_decode_inputs(w)
    host = {n: t.pin_memory() for n, t in x.items()}
    dvc = {n: t.to(dev) for n, t in host.items()}
    q, k, v = dvc["q"], dvc["k"], dvc["v"]
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Nq), device=dev, dtype=torch.float32)
    splits = fa.fa_fwd_splitkv_num_splits(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.causal)
    wsb = fa.fa_fwd_splitkv_workspace_size(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.causal)
    wsp = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        fa.fa_fwd_splitkv(q, k, v, causal=w.causal, scale=w.scale, o=o, lse=lse, workspace=wsp)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        step()
    if fa.fa_get_device_error() != fa.FA_OK:
        raise RuntimeError("device status error during warm-up")
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_timed0 = time.time()
    # the call takes ~0.2 ms of GPU time, about what the host needs to enqueue
    # it: a GPU-side wait ahead of each start event keeps the host's enqueue
    # out of the device time (the e2e number below includes it)
    hold = getattr(torch.cuda, "_sleep", None)
    for i in range(K):
        flush.zero_()
        if hold is not None:
            hold(1_000_000)
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    if fa.fa_get_device_error() != fa.FA_OK:
        raise RuntimeError("device status error in the timed region")
    ms = sum(a.elapsed_time(b) for a, b in ev) / K

    out_host = {"o": torch.empty_like(o, device="cpu").pin_memory(),
                "lse": torch.empty_like(lse, device="cpu").pin_memory()}
    h2d = tensor_bytes(*host.values())
    d2h = tensor_bytes(o, lse)

    def e2e_step():
        for n, t in host.items():
            dvc[n].copy_(t, non_blocking=True)
        step()
        out_host["o"].copy_(o, non_blocking=True)
        out_host["lse"].copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    clocks.mark(t_timed0, time.time())
    clk = clocks.stop()
    e2e_ms = e0.elapsed_time(e1) / K
    t = torch.tensor([ms, e2e_ms], dtype=torch.float64, device=dev)
    if ws > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms, e2e_ms = (float(u) for u in t.tolist())
    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0
    nbytes = W.decode_min_bytes(w) * ws
    flops = W.decode_flops(w) * ws
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {"metric": DECODE_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16, shape of the workload)",
            "config": {"workload": args.workload, "shape": W.describe_decode(w),
                       "global_batch": w.B * ws, "seq_len": w.Nk, "splits": splits,
                       "parallelism": f"replicas x{ws} (independent batches, no collective)",
                       "l2": "flushed by a 256 MiB write before every timed step",
                       "timing": "CUDA events around each call, a GPU-side wait ahead of the "
                                 "start event so the host's enqueue is not timed"},
            "frac_of_peak": gbs / ws / peaks["hbm_gbs"], "tflops": flops / (ms * 1e-3) / 1e12,
            "peak_gbs": peaks["hbm_gbs"], "peak_source": peaks["source"] + " HBM copy",
            "gpu_launches": K * (2 if splits > 1 else 1),
            "roofline": {"kernel": "fa_decode_split_kernel + fa_decode_combine_kernel",
                         "bound": "hbm", "achieved": gbs / ws, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / ws / peaks["hbm_gbs"],
                         "peak_source": peaks["source"] + " copy", "launch_ms": ms,
                         "algorithmic_work_per_launch": W.decode_min_bytes(w),
                         "traffic": measured_traffic("fa_decode_split_kernel", args.workload)},
            "e2e": {"value": nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}}
    if clk is not None:
        line["clocks"] = clk
    if ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        xs, sflops, desc = decode_oracle_sample(base)
        secs = time_decode_oracle(xs, base)
        line["cpu_baseline"] = {"value": W.decode_min_bytes(base.with_(B=1)) / secs / 1e9,
                                "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": desc, "seconds": secs}
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_sparse(args):
    """One step = one fa_fwd_blocksparse call over the gqa8k shape under a
    local-window + first-block + random block mask; the dense causal fa_fwd
    on the same inputs is timed beside it for the saving."""
    import exact_io_aware_35_gb300 as fa
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks = load_peaks()
    wname, mseed = SPARSE_WORKLOADS[args.workload]
    base = W.WORKLOADS[wname]
    if args.batch:
        base = base.with_(B=args.batch)
    w = base.with_(seed=base.seed + 1000 * rank)
    x = W.make_inputs(w, with_dout=False)
    mask_h = W.block_sparse_mask(w.Hq, w.N, seed=mseed)
    host = {n: t.pin_memory() for n, t in x.items()}
    dvc = {n: t.to(dev) for n, t in host.items()}
    q, k, v = dvc["q"], dvc["k"], dvc["v"]
    mask = mask_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), device=dev, dtype=torch.float32)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        fa.fa_fwd_blocksparse(q, k, v, mask, causal=w.causal, scale=w.scale, o=o, lse=lse)

    def dense():
        fa.fa_fwd(q, k, v, causal=w.causal, scale=w.scale, o=o, lse=lse)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        step()
        dense()
    if fa.fa_get_device_error() != fa.FA_OK:
        raise RuntimeError("device status error during warm-up")
    K = args.steps

    def timed(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        for i in range(K):
            flush.zero_()
            ev[i][0].record()
            fn()
            ev[i][1].record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / K

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_timed0 = time.time()
    ms = timed(step)
    dense_ms = timed(dense)
    if ws > 1:
        torch.distributed.barrier()
    if fa.fa_get_device_error() != fa.FA_OK:
        raise RuntimeError("device status error in the timed region")
    out_host = {"o": torch.empty_like(o, device="cpu").pin_memory(),
                "lse": torch.empty_like(lse, device="cpu").pin_memory()}
    h2d = tensor_bytes(*host.values())
    d2h = tensor_bytes(o, lse)

    def e2e_step():
        for n, t in host.items():
            dvc[n].copy_(t, non_blocking=True)
        step()
        out_host["o"].copy_(o, non_blocking=True)
        out_host["lse"].copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    clocks.mark(t_timed0, time.time())
    clk = clocks.stop()
    e2e_ms = e0.elapsed_time(e1) / K
    t = torch.tensor([ms, e2e_ms, dense_ms], dtype=torch.float64, device=dev)
    if ws > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms, e2e_ms, dense_ms = (float(u) for u in t.tolist())
    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0
    flops = W.block_sparse_flops(mask_h, w.N, w.d, w.B, w.causal) * ws
    tf = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    nb = (w.N + 127) // 128
    tri = torch.tril(torch.ones(nb, nb)) if w.causal else torch.ones(nb, nb)
    density = float((mask_h.float() * tri).sum() / (w.Hq * tri.sum()))
    line = {"metric": SPARSE_METRIC, "value": tf, "unit": "TFLOPS", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16, shape of the workload; seeded block mask)",
            "config": {"workload": args.workload, "shape": W.describe(w),
                       "mask": f"local window +-2 blocks, key block 0, 10% random; "
                               f"{density:.3f} of the causal blocks",
                       "global_batch": w.B * ws, "seq_len": w.N,
                       "parallelism": f"replicas x{ws} (independent batches, no collective)",
                       "l2": "flushed by a 256 MiB write before every timed step"},
            "frac_of_peak": tf / ws / peak, "peak_tflops": peak,
            "peak_source": peaks["source"] + " burst bf16",
            "dense_causal_ms": dense_ms, "speedup_vs_dense": dense_ms / ms,
            "gpu_launches": K,
            "roofline": {"kernel": "fa_fwd_kernel (block-mask walk)", "bound": "tensor",
                         "achieved": tf / ws, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / ws / peak, "peak_source": peaks["source"] + " burst",
                         "launch_ms": ms, "algorithmic_work_per_launch": flops / ws,
                         "traffic": measured_traffic("fa_fwd_kernel", args.workload)},
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}}
    if clk is not None:
        line["clocks"] = clk
    if ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        # one head of batch element 0 under its mask row
        xs = W.make_inputs(base.with_(B=1), with_dout=False)
        sub = (xs["q"][:, :, :1], xs["k"][:, :, :1], xs["v"][:, :, :1])
        t0 = time.perf_counter()
        oracle.attn_fwd_blockmask(*sub, mask_h[:1].numpy(), 128, w.causal, w.scale)
        secs = time.perf_counter() - t0
        sflops = W.block_sparse_flops(mask_h[:1], w.N, w.d, 1, w.causal)
        line["cpu_baseline"] = {"value": sflops / secs / 1e12, "unit": "TFLOPS",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": "batch element 0, head 0 under its mask", "seconds": secs}
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def reference_line(args, metric, value, unit, ms, shape, desc):
    """The JSON line of a reference arm: the oracle timed on the host cores."""
    import oracle
    return {"impl": "reference", "metric": metric, "value": value, "unit": unit,
            "n_gpus": dist_env()[0], "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "shape": shape, "sample": desc},
            "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_sparse_reference(args):
    """The block-mask oracle on one head of batch element 0 under its mask row
    (the sample the GPU line's CPU baseline uses)."""
    if dist_env()[1] != 0:
        return 0
    import oracle
    wname, mseed = SPARSE_WORKLOADS[args.workload]
    w = W.WORKLOADS[wname]
    mask_h = W.block_sparse_mask(w.Hq, w.N, seed=mseed)
    xs = W.make_inputs(w.with_(B=1), with_dout=False)
    sub = (xs["q"][:, :, :1], xs["k"][:, :, :1], xs["v"][:, :, :1])
    oracle.build()

    def once():
        t0 = time.perf_counter()
        oracle.attn_fwd_blockmask(*sub, mask_h[:1].numpy(), 128, w.causal, w.scale)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        once()
    ms = 1e3 * sum(once() for _ in range(args.steps)) / args.steps
    sflops = W.block_sparse_flops(mask_h[:1], w.N, w.d, 1, w.causal)
    desc = (f"batch element 0, head 0 under its mask, full N={w.N} "
            f"({sflops / 1e9:.1f} GFLOP of computed blocks)")
    print(json.dumps(reference_line(args, SPARSE_METRIC, sflops / (ms * 1e-3) / 1e12, "TFLOPS",
                                    ms, W.describe(w), desc)), flush=True)
    return 0


def run_fp8_reference(args):
    """The float64 model of the FP8 forward (block quantisation, rotation,
    lazy rescale, e4m3 P) on one head over the first 2048 positions of batch
    element 0: the model walks rows and blocks in Python, so the sample is
    kept well under a second per step."""
    if dist_env()[1] != 0:
        return 0
    w = W.WORKLOADS[FP8_WORKLOADS[args.workload]]
    once, flops, desc = fp8_model_sample(w)
    for _ in range(args.warmup):
        once()
    ms = 1e3 * sum(once() for _ in range(args.steps)) / args.steps
    print(json.dumps(reference_line(args, FP8_METRIC, flops / (ms * 1e-3) / 1e12, "TFLOPS", ms,
                                    W.describe(w), desc)), flush=True)
    return 0


def fp8_model_sample(w: W.Workload, n: int = 2048):
    """(timed call, nominal FLOPs, description) of the float64 FP8 model on
    head 0 of batch element 0 over its first n positions."""
    from oracle import fp8 as ofp8
    n = min(n, w.N)
    xs = W.make_inputs(w.with_(B=1), with_dout=False)
    q, k, v = (xs[c][:, :n, :1].contiguous() for c in ("q", "k", "v"))

    def once():
        t0 = time.perf_counter()
        ofp8.attn_fwd_fp8(q, k, v, w.causal, w.scale, rotate=True)
        return time.perf_counter() - t0

    flops = W.fwd_flops(w.with_(B=1, Hq=1, Hkv=1, N=n))
    desc = (f"batch element 0, head 0, positions 0..{n - 1} through the float64 model of the "
            f"FP8 forward ({flops / 1e9:.2f} nominal GFLOP)")
    return once, flops, desc


def run_fp8(args):
    """One step = one fa_fwd_fp8 call (quantisation of q, k, v + the FP8
    forward) over the gqa8k shape; the bf16 inference fa_fwd on the same
    inputs is timed beside it."""
    import exact_io_aware_35_gb300 as fa
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks = load_peaks()
    base = W.WORKLOADS[FP8_WORKLOADS[args.workload]]
    if args.batch:
        base = base.with_(B=args.batch)
    w = base.with_(seed=base.seed + 1000 * rank)
    x = W.make_inputs(w, with_dout=False)
    host = {n: t.pin_memory() for n, t in x.items()}
    dvc = {n: t.to(dev) for n, t in host.items()}
    q, k, v = dvc["q"], dvc["k"], dvc["v"]
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), device=dev, dtype=torch.float32)
    wsp = torch.empty(fa.fa_fwd_fp8_workspace_size(w.B, w.Hq, w.Hkv, w.N, w.d),
                      dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        fa.fa_fwd_fp8(q, k, v, causal=w.causal, scale=w.scale, rotate=True, o=o, lse=lse,
                      workspace=wsp)

    def quant():
        fa.fa_fwd_fp8(q, k, v, causal=w.causal, scale=w.scale, rotate=True, o=o, lse=lse,
                      workspace=wsp, stage=fa.FA_FP8_QUANTIZE_ONLY)

    def attend():
        fa.fa_fwd_fp8(q, k, v, causal=w.causal, scale=w.scale, rotate=True, o=o, lse=lse,
                      workspace=wsp, stage=fa.FA_FP8_ATTEND_ONLY)

    def bf16():
        fa.fa_fwd(q, k, v, causal=w.causal, scale=w.scale, o=o, lse=lse)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        step()
        bf16()
    if fa.fa_get_device_error() != fa.FA_OK:
        raise RuntimeError("device status error during warm-up")
    K = args.steps

    def timed(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        for i in range(K):
            flush.zero_()
            ev[i][0].record()
            fn()
            ev[i][1].record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / K

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_timed0 = time.time()
    ms = timed(step)
    quant_ms = timed(quant)
    attn_ms = timed(attend)
    bf16_ms = timed(bf16)
    if ws > 1:
        torch.distributed.barrier()
    if fa.fa_get_device_error() != fa.FA_OK:
        raise RuntimeError("device status error in the timed region")
    out_host = {"o": torch.empty_like(o, device="cpu").pin_memory(),
                "lse": torch.empty_like(lse, device="cpu").pin_memory()}
    h2d = tensor_bytes(*host.values())
    d2h = tensor_bytes(o, lse)

    def e2e_step():
        for n, t in host.items():
            dvc[n].copy_(t, non_blocking=True)
        step()
        out_host["o"].copy_(o, non_blocking=True)
        out_host["lse"].copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    clocks.mark(t_timed0, time.time())
    clk = clocks.stop()
    e2e_ms = e0.elapsed_time(e1) / K
    t = torch.tensor([ms, e2e_ms, bf16_ms, quant_ms, attn_ms], dtype=torch.float64, device=dev)
    if ws > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms, e2e_ms, bf16_ms, quant_ms, attn_ms = (float(u) for u in t.tolist())
    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0
    flops = W.fwd_flops(w) * ws
    tf = flops / (ms * 1e-3) / 1e12
    attn_tf = flops / ws / (attn_ms * 1e-3) / 1e12
    peak8 = 2.0 * peaks["bf16_tflops"]
    line = {"metric": FP8_METRIC, "value": tf, "unit": "TFLOPS", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (bf16 in and out)",
            "data": "synthetic (seeded N(0,1) bf16, shape of the workload)",
            "config": {"workload": args.workload, "shape": W.describe(w),
                       "global_batch": w.B * ws, "seq_len": w.N,
                       "quantisation": "q, k per 128-row block and head, rotated; v per head",
                       "parallelism": f"replicas x{ws} (independent batches, no collective)",
                       "l2": "flushed by a 256 MiB write before every timed step"},
            "frac_of_peak": tf / ws / peak8, "peak_tflops": peak8,
            "peak_source": peaks["source"] + " burst bf16 x 2 (nominal fp8/bf16 ratio)",
            "bf16_fwd_ms": bf16_ms, "speedup_vs_bf16": bf16_ms / ms,
            "quantise_ms": quant_ms, "attention_ms": attn_ms,
            "attention_tflops": attn_tf, "attention_speedup_vs_bf16": bf16_ms / attn_ms,
            "gpu_launches": K * 5,
            "roofline": {"kernel": "fa_fp8_fwd_kernel (FA_FP8_ATTEND_ONLY call)",
                         "bound": "tensor", "achieved": attn_tf, "peak": peak8,
                         "unit": "TFLOP/s", "frac": attn_tf / peak8,
                         "peak_source": peaks["source"] + " burst bf16 x 2", "launch_ms": attn_ms,
                         "algorithmic_work_per_launch": flops / ws,
                         "traffic": measured_traffic("fa_fp8_fwd_kernel", args.workload)},
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}}
    if clk is not None:
        line["clocks"] = clk
    if ws == 1 and not args.no_cpu_baseline:
        import oracle
        once, sflops, desc = fp8_model_sample(w)
        secs = once()
        line["cpu_baseline"] = {"value": sflops / secs / 1e12, "unit": "TFLOPS",
                                "cores": oracle.num_threads(), "kind": "oracle (float64 FP8 model)",
                                "sample": desc, "seconds": secs}
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(W.WORKLOADS) + sorted(W.DECODE_WORKLOADS) +
                    sorted(SPARSE_WORKLOADS) + sorted(FP8_WORKLOADS))
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (profiling cases)")
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.workload in W.DECODE_WORKLOADS:
        return run_decode_reference(args) if args.impl == "reference" else run_decode(args)
    if args.workload in SPARSE_WORKLOADS:
        return run_sparse_reference(args) if args.impl == "reference" else run_sparse(args)
    if args.workload in FP8_WORKLOADS:
        return run_fp8_reference(args) if args.impl == "reference" else run_fp8(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
