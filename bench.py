#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300.

One step = one chunked forward (saving chunk-start states) plus the matching
backward over the fwd+bwd workload B=1, T=32768, H=96, d=128 (bf16 I/O, fp32
state and gradients, nonzero initial state), through the C ABI with buffers
resident in HBM. The decode/verify workload (256 sequences x 96 heads, 4 tokens
per call) is measured in the same run and reported under "decode".

Prints ONE JSON line (rank 0). Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 run under torch.distributed.run: every rank runs an independent
replica on its own GPU (weak scaling; the heads and sequences of KDA are
independent, so there is no data-path collective).
"""
from __future__ import annotations

import argparse
import ctypes as C
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "fwdbwd-bf16-T32768-H96"
DECODE = "decode-bf16-N256-L4-H96"
D = 128
# algorithmic bytes per token and head (inputs read once, outputs written once)
FWD_BYTES = 3 * 256 + 512 + 4 + 256          # q,k,v bf16 + g fp32 + beta + o bf16        = 1540
BWD_BYTES = 3 * 256 + 512 + 4 + 256 + 3 * 512 + 512 + 4   # + dO, dq/dk/dv/dg fp32, dbeta = 3592
FWD_BYTES_F32 = 3 * 512 + 512 + 4 + 512      # the same tensors with fp32 q, k, v, o      = 2564
BWD_BYTES_F32 = 3 * 512 + 512 + 4 + 512 + 3 * 512 + 512 + 4   # fp32 q, k, v, dO            = 4616
FWD_FLOP = 10 * 64 * D + 6 * D * D           # 180,224
BWD_FLOP = 24 * 64 * D + 12 * D * D          # 393,216
DEC_BYTES = 2 * D * D * 4 + 4 * (3 * 256 + 512 + 4 + 256)   # per (sequence, head) per 4-token call
# per-kernel share of the algorithmic bytes (which kernel reads/writes which tensor)
KERNEL_BYTES = {
    "fwd.prep": 256 + 256 + 512 + 4,         # q, k, g, beta
    "fwd.scan": 256 + 256,                   # v in, o out
    "bwd.dscan": 256 + 512,                  # dO in, dv out
    "bwd.chunk": 256 + 256 + 256 + 512 + 4 + 3 * 512 + 4,   # v, q, k, g, beta in; dq, dk, dg, dbeta out
}
FWD_STAGES = ["fwd.table", "fwd.prep", "fwd.scan"]
BWD_STAGES = ["bwd.table", "bwd.dscan", "bwd.chunk"]
KERNEL_SRC = {"fwd.prep": "kda_prep_tc.cu", "fwd.scan": "kda_scan_tc.cu",
              "bwd.dscan": "kda_scan_tc.cu", "bwd.chunk": "kda_bwd_tc.cu",
              "fwd.prep.inference": "kda_prep_tc.cu", "fwd.scan.inference": "kda_scan_tc.cu",
              "decode": "kda_step.cu", "attnres.fwd": "kda_attnres.cu", "attnres.bwd": "kda_attnres.cu",
              "conv.fwd": "kda_conv.cu", "conv.bwd": "kda_conv.cu", "conv.step": "kda_conv.cu"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def src_hash(name):
    path = os.path.join(ROOT, "gated_delta_rule_chunked_gb300", "csrc", name)
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:12]


def recorded_traffic(kernel):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged.

    Summaries under profiles/ carry lines `traffic <kernel> <bytes_per_launch> <source-sha12> <scale>`.
    """
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".txt", ".md")):
            continue
        for line in open(os.path.join(pdir, fn)):
            m = re.match(r"^traffic\s+(\S+)\s+([0-9.eE+]+)\s+([0-9a-f]{12})", line.strip())
            if m and m.group(1) == kernel and m.group(3) == src_hash(KERNEL_SRC[kernel]):
                return float(m.group(2))
    return None


def scaled_traffic(kernel, units, ref_units=32768 * 96):
    """Recorded DRAM bytes per launch of the T=32768 x 96-head workload, scaled to `units`
    token-heads (the chunk-parallel and scan kernels move a fixed amount per chunk-head)."""
    t = recorded_traffic(kernel)
    return None if t is None else t * units / ref_units


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.06)
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        mhz = [float(r[0]) for r in rows if len(r) >= 8 and r[0].strip().replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if len(r) >= 8 and r[1].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) >= 8 for i in range(4) if "Active" in r[4 + i]
                          and "Not" not in r[4 + i]})
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- ours
class ChunkedCase:
    """Resident buffers of one chunked workload, two input sets (different seeds) that the
    timed steps alternate between, so no step re-reads the previous step's inputs. `mode`
    "fwdbwd": training forward (saves what the backward needs) + backward; "fwd": the
    inference forward (no saved, records in the workspace)."""

    def __init__(self, lib, dev, name, mode, status, seq_len=0, over=None):
        import torch
        import gated_delta_rule_chunked_gb300 as kda
        from gated_delta_rule_chunked_gb300.inputs import make_workload, WORKLOADS
        over = dict(over or {})
        if seq_len:
            over["seq_lens"] = (seq_len,)
        seed = WORKLOADS[name].seed
        self.sets = [make_workload(name, device=dev, **over, **({"seed": seed + 5000} if i else {}))
                     for i in range(2)]
        b = self.sets[0]
        self.T, self.H, self.N = b.total, b.heads, b.n_seqs
        self.mode = mode
        f32io = b.q.dtype == torch.float32
        self.fwd_bytes = FWD_BYTES_F32 if f32io else FWD_BYTES
        self.bwd_bytes = BWD_BYTES_F32 if f32io else BWD_BYTES
        f32 = dict(dtype=torch.float32, device=dev)
        self.o = torch.empty_like(b.v)
        self.hT = torch.empty((self.N, self.H, D, D), **f32)
        fa = kda.fwd_args(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.h0, self.o, self.hT)
        self.saved = (torch.empty(lib.kda_saved_size(C.byref(fa)), dtype=torch.uint8, device=dev)
                      if mode == "fwdbwd" else None)
        fa = kda.fwd_args(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.h0, self.o, self.hT, self.saved)
        self.fws = torch.empty(lib.kda_fwd_workspace_size(C.byref(fa)), dtype=torch.uint8, device=dev)
        self.fa, self.ba = [], []
        if mode == "fwdbwd":
            self.grads = {n: torch.empty(sh, **f32) for n, sh in
                          (("dq", b.q.shape), ("dk", b.k.shape), ("dv", b.v.shape), ("dg", b.g.shape),
                           ("dbeta", b.beta.shape), ("dh0", (self.N, self.H, D, D)))}
        for x in self.sets:
            a = kda.fwd_args(x.q, x.k, x.v, x.beta, x.g, x.cu_seqlens, x.h0, self.o, self.hT, self.saved, self.fws,
                             dev_status=status)
            self.fa.append(a)
            if mode == "fwdbwd":
                gr = self.grads
                ba = kda.bwd_args(a, x.dO, gr["dq"], gr["dk"], gr["dv"], gr["dbeta"], gr["dg"], gr["dh0"])
                if not hasattr(self, "bws"):
                    self.bws = torch.empty(lib.kda_bwd_workspace_size(C.byref(ba)), dtype=torch.uint8, device=dev)
                self.ba.append(kda.bwd_args(a, x.dO, gr["dq"], gr["dk"], gr["dv"], gr["dbeta"], gr["dg"], gr["dh0"],
                                            None, self.bws))

    def stages(self):
        return FWD_STAGES + (BWD_STAGES if self.mode == "fwdbwd" else [])

    def step(self, lib, sptr, i, arrays=None):
        from gated_delta_rule_chunked_gb300 import _lib
        k = i & 1
        if arrays is not None:
            lib.kda_set_profile_events(C.cast(arrays[0], C.c_void_p), len(FWD_STAGES))
        _lib.check(lib.kda_fwd(C.byref(self.fa[k]), sptr))
        if self.mode == "fwdbwd":
            if arrays is not None:
                lib.kda_set_profile_events(C.cast(arrays[1], C.c_void_p), len(BWD_STAGES))
            _lib.check(lib.kda_bwd(C.byref(self.ba[k]), sptr))
        if arrays is not None:
            lib.kda_set_profile_events(None, 0)


def time_case(case, lib, dev, stream, K, W, world=1, on_start=None):
    """W untimed steps, then K timed steps bracketed by a barrier and synchronisation; per-kernel
    device times from the events the library records after each launch. Returns (ms per step
    as the max over ranks, per-kernel ms)."""
    import torch
    sptr = stream.cuda_stream
    names = case.stages()
    nst = 1 + len(names)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(K)]
    for row in evs:
        for e in row:
            e.record(stream)          # materialise the events so their handles exist
    torch.cuda.synchronize(dev)
    arrays = [((C.c_void_p * len(FWD_STAGES))(*[e.cuda_event for e in row[1:1 + len(FWD_STAGES)]]),
               (C.c_void_p * len(BWD_STAGES))(*[e.cuda_event for e in row[1 + len(FWD_STAGES):]]))
              for row in evs]
    for i in range(W):
        case.step(lib, sptr, i)
    torch.cuda.synchronize(dev)
    barrier(world)
    extra = on_start() if on_start else None
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for i in range(K):
        evs[i][0].record(stream)
        case.step(lib, sptr, W + i, arrays[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    ms_local = t_start.elapsed_time(t_end) / K
    barrier(world)
    per = {n: 0.0 for n in names}
    for row in evs:
        for j in range(1, nst):
            per[names[j - 1]] += row[j - 1].elapsed_time(row[j]) / K
    return reduce_max(ms_local, world), per, extra


def summarize(case, per, peaks, ms=None):
    """tokens/s, algorithmic GB/s and roofline fractions of one timed chunked workload."""
    units = case.T * case.H
    fwd_ms = sum(per[n] for n in FWD_STAGES)
    out = {"fwd": {"ms": fwd_ms, "tokens_per_s": case.T / (fwd_ms * 1e-3),
                   "gbs_algorithmic": case.fwd_bytes * units / (fwd_ms * 1e-3) / 1e9,
                   "roofline_frac": case.fwd_bytes * units / (fwd_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}}
    if case.mode == "fwdbwd":
        bwd_ms = sum(per[n] for n in BWD_STAGES)
        out["bwd"] = {"ms": bwd_ms, "tokens_per_s": case.T / (bwd_ms * 1e-3),
                      "gbs_algorithmic": case.bwd_bytes * units / (bwd_ms * 1e-3) / 1e9,
                      "roofline_frac": case.bwd_bytes * units / (bwd_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    if ms is not None:
        byts = (case.fwd_bytes + (case.bwd_bytes if case.mode == "fwdbwd" else 0)) * units
        out["step"] = {"ms": ms, "tokens_per_s": case.T / (ms * 1e-3), "gbs_algorithmic": byts / (ms * 1e-3) / 1e9,
                       "roofline_frac": byts / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    out["kernels_ms"] = {k: round(v, 4) for k, v in per.items()}
    return out


def bench_range(args, lib, dev, stream, peaks, status):
    """The pages' sequence-length range (4K-128K tokens) and the inference forward: the
    T=4096 forward, the T=32768 forward without saved (inference), the 131,072 packed
    varlen tokens (8 sequences) fwd+bwd and one 131,072-token sequence fwd+bwd. Every
    line alternates two resident input sets per timed step."""
    import torch
    res = {}
    want = set(x for x in args.range_lines.split(",") if x)
    for name, mode, key in (("fwd-bf16-T4096-H96", "fwd", "fwd_T4096"),
                            ("fwdbwd-bf16-T32768-H96", "fwd", "fwd_T32768_inference"),
                            ("fwdbwd-bf16-varlen8-T131072-H96", "fwdbwd", "fwdbwd_varlen8_T131072"),
                            ("fwdbwd-bf16-T131072-H96", "fwdbwd", "fwdbwd_T131072")):
        if (args.seq_len and "131072" in name) or (want and key not in want):
            continue
        case = ChunkedCase(lib, dev, name, mode, status, seq_len=args.seq_len if "T32768" in name else 0)
        K = max(3, min(args.steps, 20 if case.T <= 32768 else 5))
        ms, per, _ = time_case(case, lib, dev, stream, K, max(args.warmup, 3))
        if int(status.item()) != 0:
            raise SystemExit(f"device status {int(status.item())} in {name}: no number reported")
        line = {"workload": name, "mode": "training fwd + bwd" if mode == "fwdbwd" else "inference forward (no saved)",
                "tokens": case.T, "sequences": case.N, "steps": K, **summarize(case, per, peaks, ms)}
        dom = max((k for k in per if k in KERNEL_BYTES), key=lambda n: per[n])
        ach = KERNEL_BYTES[dom] * case.T * case.H / (per[dom] * 1e-3) / 1e9
        line["roofline"] = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": ach / peaks["hbm_gbs"],
                            "traffic": scaled_traffic(dom if mode == "fwdbwd" else dom + ".inference",
                                                      case.T * case.H)}
        res[key] = line
        del case
        torch.cuda.empty_cache()
    # fp32 I/O fwd + bwd: the fp32 workload's recipe at 4096 tokens x 96 heads
    if want and "fwdbwd_f32_T4096" not in want:
        return res
    case = ChunkedCase(lib, dev, "fwd-f32-T512-H2", "fwdbwd", status,
                       over={"kind": "fwdbwd", "seq_lens": (4096,), "heads": 96})
    K = max(3, min(args.steps, 10))
    ms, per, _ = time_case(case, lib, dev, stream, K, max(args.warmup, 3))
    if int(status.item()) != 0:
        raise SystemExit(f"device status {int(status.item())} in the fp32 line: no number reported")
    res["fwdbwd_f32_T4096"] = {
        "workload": "fwdbwd-f32-T4096-H96 (the recipe of fwd-f32-T512-H2 at 4096 tokens x 96 heads, dO drawn after)",
        "mode": "training fwd + bwd, fp32 I/O", "tokens": case.T, "sequences": case.N, "steps": K,
        **summarize(case, per, peaks, ms),
        "note": "fp32 products on the CUDA cores (the 1e-4 tolerance of fp32 I/O); bwd.dscan includes the "
                "backward's re-run of the chunk prep, bwd.chunk its state-side and intra-chunk kernels"}
    del case
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    import gated_delta_rule_chunked_gb300 as kda

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = kda.library()
    stream = torch.cuda.current_stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)   # a kernel that gives up a bounded wait writes here

    case = ChunkedCase(lib, dev, WORKLOAD, "fwdbwd", status, seq_len=args.seq_len)
    T, H, N = case.T, case.H, case.N
    K = args.steps
    clocks_box = []
    ms_step, per, _ = time_case(case, lib, dev, stream, K, args.warmup, world,
                                on_start=lambda: clocks_box.append(ClockSampler(local_rank) if rank == 0 else None))
    ck = clocks_box[0].stop() if clocks_box and clocks_box[0] else None
    if int(status.item()) != 0:
        raise SystemExit(f"device status {int(status.item())}: a kernel gave up a bounded wait; no number reported")

    peaks = load_peaks()
    tok = T
    units = T * H
    summ = summarize(case, per, peaks)
    fwd_ms, bwd_ms = summ["fwd"]["ms"], summ["bwd"]["ms"]
    dom = max(KERNEL_BYTES, key=lambda n: per[n])
    dom_bytes = KERNEL_BYTES[dom] * units
    achieved = dom_bytes / (per[dom] * 1e-3) / 1e9
    traffic = recorded_traffic(dom) if not args.seq_len else None   # recorded for T = 32768
    step_bytes = (FWD_BYTES + BWD_BYTES) * units
    out = {
        "metric": "KDA fwd+bwd tokens/s (H=96, d=128, T=32768, bf16 I/O, fp32 state/grads)",
        "value": world * tok / (ms_step * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; q,k,v,dO ~ N(0,1) bf16, beta=sigmoid(N(0,1)), g=logsigmoid(N(3,1)), h0 ~ N(0,0.02))",
        "config": {"workload": WORKLOAD, "batch": N, "seq_len": T, "heads": H, "head_dim": D, "chunk": 64,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs (4.8 GB per set) larger than L2; no flush; the timed steps alternate between two "
                         "resident input sets drawn with different seeds"},
        "fwd": summ["fwd"],
        "bwd": summ["bwd"],
        "kernels_ms": summ["kernels_ms"],
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "algorithmic_bytes_per_launch": dom_bytes, "peak_source": peaks["source"]},
        "roofline_step": {"bound": "hbm", "achieved": step_bytes / (ms_step * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                          "unit": "GB/s", "frac": step_bytes / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"],
                          "flop_frac_of_bf16": (FWD_FLOP + BWD_FLOP) * units / (ms_step * 1e-3) / 1e12
                          / peaks["bf16_tflops_sustained"]},
        "gpu_launches": K * (len(FWD_STAGES) + len(BWD_STAGES)),
        "clocks": ck,
    }
    if args.seq_len:
        out["config"]["workload"] += f" (T overridden to {T})"
    host = None
    if not args.no_e2e:
        b = case.sets[0]
        host = {n: getattr(b, n).to("cpu").pin_memory() for n in ("q", "k", "v", "beta", "g", "h0", "dO")}
        host["cu_seqlens"] = b.cu_seqlens.to("cpu")
    del case
    torch.cuda.empty_cache()
    if host is not None:   # first after the step, on an empty allocator cache
        out["e2e"] = bench_e2e(args, dev, world, host)
        del host
        torch.cuda.empty_cache()
    if not args.no_range:
        out["range"] = bench_range(args, lib, dev, stream, peaks, status)
    if not args.no_decode:
        out["decode"] = bench_decode(args, dev, lib, stream, peaks)
    if not args.no_cp:
        out["cp_forward"] = bench_cp(args, dev, peaks, out["fwd"]["ms"])
    small = {"T": args.seq_len} if args.seq_len else {}   # profiling runs only
    if not args.no_attnres:
        out["attnres"] = bench_attnres(args, dev, peaks, **small)
    if not args.no_conv:
        out["short_conv"] = bench_conv(args, dev, peaks, **small)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args)
    return out


def bench_attnres(args, dev, peaks, T=32768, S=9, d=7168):
    """Attention Residuals at the K3 width: 9 sources x 7168 channels per token, bf16.
    Algorithmic bytes: forward reads the sources once and writes out; backward reads the
    sources and d_out once and writes every d_source (the [T, S] statistics are negligible)."""
    import torch
    import gated_delta_rule_chunked_gb300 as kda
    gen = torch.Generator(device=dev).manual_seed(7168)
    src = [torch.randn(T, d, generator=gen, device=dev).to(torch.bfloat16) for _ in range(S)]
    w = torch.randn(d, generator=gen, device=dev) / d ** 0.5
    g = torch.randn(T, d, generator=gen, device=dev).to(torch.bfloat16)
    K = max(args.steps, 10)
    res = {}
    for name in ("fwd", "bwd"):
        out, stats = kda.attnres_fwd(src, w)
        run = (lambda: kda.attnres_fwd(src, w)) if name == "fwd" else (lambda: kda.attnres_bwd(src, w, stats, g))
        for _ in range(max(args.warmup, 3)):
            run()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        s.record()
        for _ in range(K):
            run()
        e.record()
        torch.cuda.synchronize(dev)
        ms = s.elapsed_time(e) / K
        byts = T * d * 2 * ((S + 1) if name == "fwd" else (2 * S + 1))
        gbs = byts / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "gbs_algorithmic": gbs, "algorithmic_bytes_per_launch": byts,
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": gbs / peaks["hbm_gbs"],
                                  "traffic": recorded_traffic(f"attnres.{name}") if T == 32768 else None}}
    return {"workload": f"attnres-bf16-T{T}-S{S}-d{d}", **res,
            "tokens_per_s_fwd_bwd": T / ((res["fwd"]["ms"] + res["bwd"]["ms"]) * 1e-3),
            "l2": "sources (4.2 GB) larger than L2; no flush"}


def _time_ms(run, dev, warmup, K):
    import torch
    for _ in range(max(warmup, 3)):
        run()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    s.record()
    for _ in range(K):
        run()
    e.record()
    torch.cuda.synchronize(dev)
    return s.elapsed_time(e) / K


def bench_conv(args, dev, peaks, T=32768, H=96, d=128, W=4, N=256, L=4):
    """Short convolution of the KDA input side on q, k, v side by side (C = 3 x H x d), width
    4, SiLU, bf16, one sequence of T tokens with its state; and the decode step of N sequences
    x L slots from a state pool. Algorithmic bytes: forward reads x, writes y; backward reads x
    and dy, writes dx (fp32); the step reads x and the states, writes y and the states (the
    weights, bias and [N, W-1, C] states of the training calls are included, all small)."""
    import torch
    import gated_delta_rule_chunked_gb300 as kda
    C = 3 * H * d
    gen = torch.Generator(device=dev).manual_seed(C)
    x = torch.randn(T, C, generator=gen, device=dev).to(torch.bfloat16)
    dy = torch.randn(T, C, generator=gen, device=dev).to(torch.bfloat16)
    w = torch.randn(C, W, generator=gen, device=dev) / 2
    b = torch.randn(C, generator=gen, device=dev) * 0.1
    st = torch.randn(1, W - 1, C, generator=gen, device=dev).to(torch.bfloat16)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    K = max(args.steps, 10)
    small = C * W * 4 + C * 4 + 2 * (W - 1) * C * 2
    res = {}
    for name, run, byts in (
            ("fwd", lambda: kda.conv_fwd(x, w, b, cu, st), T * C * 4 + small),
            ("bwd", lambda: kda.conv_bwd(x, w, b, dy, cu, st, None), T * C * 8 + small + (W - 1) * C * 4)):
        ms = _time_ms(run, dev, args.warmup, K)
        gbs = byts / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "gbs_algorithmic": gbs, "algorithmic_bytes_per_launch": byts,
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": gbs / peaks["hbm_gbs"],
                                  "traffic": recorded_traffic(f"conv.{name}") if T == 32768 else None}}
    xs = torch.randn(N, L, C, generator=gen, device=dev).to(torch.bfloat16)
    pool = torch.randn(N, W - 1, C, generator=gen, device=dev).to(torch.bfloat16)
    acc = torch.randint(1, L + 1, (N,), generator=gen, device=dev, dtype=torch.int32)
    ys = torch.empty_like(xs)
    ms = _time_ms(lambda: kda.conv_step(xs, w, b, pool, acc, out=ys), dev, args.warmup, max(K, 50))
    byts = N * L * C * 4 + N * (W - 1) * C * 4 + C * W * 4 + C * 4
    gbs = byts / (ms * 1e-3) / 1e9
    res["step"] = {"workload": f"conv-step-bf16-N{N}-L{L}-C{C}", "ms": ms, "gbs_algorithmic": gbs,
                   "algorithmic_bytes_per_launch": byts,
                   "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": gbs / peaks["hbm_gbs"], "traffic": recorded_traffic("conv.step")},
                   "note": f"{byts / 1e6:.0f} MB per call (inputs, outputs and pool together larger than L2); no flush"}
    return {"workload": f"conv-bf16-T{T}-C{C}-W{W}-silu", **res,
            "tokens_per_s_fwd_bwd": T / ((res["fwd"]["ms"] + res["bwd"]["ms"]) * 1e-3),
            "l2": "x and dy (2.4 GB each) larger than L2; no flush"}


def bench_cp(args, dev, peaks, fwd_ms, P=4):
    """Context-parallel forward emulated on one GPU: the sequence cut into P segments,
    each segment's (M, b) from two forward passes, the combine, and a forward over the
    segments from their incoming states (what each of P devices would run on its own
    segment, plus the state exchange)."""
    import torch
    import gated_delta_rule_chunked_gb300 as kda
    from gated_delta_rule_chunked_gb300.inputs import make_workload
    b = make_workload(WORKLOAD, device=dev)
    T = b.q.shape[0]
    cu = b.cu_seqlens.cpu()
    run = lambda: kda.kda_fwd_cp(b.q, b.k, b.v, b.beta, b.g, cu, b.h0, n_segments=P)
    for _ in range(max(args.warmup, 3)):
        run()
    K = max(3, min(args.steps, 10))
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    s.record()
    for _ in range(K):
        run()
    e.record()
    torch.cuda.synchronize(dev)
    ms = s.elapsed_time(e) / K
    H = b.q.shape[1]
    gbs = FWD_BYTES * T * H / (ms * 1e-3) / 1e9
    return {"workload": f"cp{P}-{WORKLOAD.replace('fwdbwd', 'fwd')}", "segments": P, "ms": ms,
            "unsplit_fwd_ms": fwd_ms, "tokens_per_s": T / (ms * 1e-3), "gbs_algorithmic": gbs,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"]},
            "note": "one GPU runs all P segments: the chunk records, the segment maps and offsets (one paired scan "
                    "launch), the combine, and the final forward pass"}


def bench_decode(args, dev, lib, stream, peaks):
    import torch
    import gated_delta_rule_chunked_gb300 as kda
    from gated_delta_rule_chunked_gb300 import _lib
    from gated_delta_rule_chunked_gb300.inputs import make_workload
    d = make_workload(DECODE, device=dev)
    N, L, H, _ = d.q.shape
    o = torch.empty_like(d.v)
    a = kda.step_args(d.q, d.k, d.v, d.beta, d.g, d.state, d.accept_len, o)
    sptr = stream.cuda_stream
    K = max(args.steps, 20)
    for _ in range(max(args.warmup, 3)):
        _lib.check(lib.kda_step(C.byref(a), sptr))
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    s.record(stream)
    for _ in range(K):
        _lib.check(lib.kda_step(C.byref(a), sptr))
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = s.elapsed_time(e) / K
    gbs = DEC_BYTES * N * H / (ms * 1e-3) / 1e9
    out = {"workload": DECODE, "ms_per_call": ms, "gbs_algorithmic": gbs, "unit": "GB/s",
           "roofline": {"kernel": "decode", "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "traffic": recorded_traffic("decode")},
           "tokens_per_s": N * L / (ms * 1e-3), "gpu_launches": K,
           "state_bytes": N * H * D * D * 4, "l2": "state (1.6 GB) larger than L2; no flush"}
    del d, o, a
    out["replay_verify"] = bench_replay_verify(args, dev, lib, stream, peaks, N, L, H)
    return out


def bench_replay_verify(args, dev, lib, stream, peaks, N, L, H, P=512):
    """Two-phase draft/verify over a paged state pool: each call replays the a_i accepted
    tokens of the previous L-token draft (right-aligned after padding) and verifies the next
    L-token draft, committing after the replay; states sit in random distinct slots of a pool
    of P. Algorithmic bytes: the state read and written once, and every real token slot's
    inputs and output."""
    import torch
    from gated_delta_rule_chunked_gb300 import _lib
    from gated_delta_rule_chunked_gb300.inputs import make_decode_batch
    import gated_delta_rule_chunked_gb300 as kda
    d = make_decode_batch(N, 2 * L, H, "bf16", seed=4242, device=dev)
    gen = torch.Generator().manual_seed(4243)
    pool = (torch.randn(P, H, D, D, generator=gen) * 0.02).to(dev)
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32).to(dev)
    acc_prev = torch.randint(1, L + 1, (N,), generator=gen, dtype=torch.int32)
    first = (L - acc_prev).to(torch.int32).to(dev)
    commit = torch.full((N,), L, dtype=torch.int32, device=dev)
    o = torch.empty_like(d.v)
    a = kda.step_args(d.q, d.k, d.v, d.beta, d.g, pool, commit, o, 1.0, idx, first)
    sptr = stream.cuda_stream
    K = max(args.steps, 20)
    for _ in range(max(args.warmup, 3)):
        _lib.check(lib.kda_step(C.byref(a), sptr))
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    s.record(stream)
    for _ in range(K):
        _lib.check(lib.kda_step(C.byref(a), sptr))
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = s.elapsed_time(e) / K
    real = int(acc_prev.sum()) + N * L                     # real token slots per head
    byts = H * (N * 2 * D * D * 4 + real * (3 * 256 + 512 + 4 + 256))
    gbs = byts / (ms * 1e-3) / 1e9
    return {"workload": f"decode-replay-verify-bf16-N{N}-P{P}-L{L}+{L}-H{H}", "ms_per_call": ms,
            "gbs_algorithmic": gbs, "unit": "GB/s",
            "roofline": {"kernel": "decode", "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"]},
            "draft_tokens_per_s": N * L / (ms * 1e-3), "replayed_tokens_per_call": int(acc_prev.sum()),
            "gpu_launches": K, "pool_bytes": P * H * D * D * 4}


def bench_e2e(args, dev, world, host):
    """Same step through the public Python API with host buffers: every step copies its
    inputs host->device from pinned memory, runs kda_fwd + kda_bwd and copies the
    gradients device->host. Steps are pipelined the way a training loop would run them:
    step i's inputs move on a copy-in stream and step i-1's gradients on a copy-out
    stream while step i-1 / i compute, with two device input buffers and two pinned
    output buffers."""
    import torch
    import gated_delta_rule_chunked_gb300 as kda
    names = ("q", "k", "v", "beta", "g", "h0", "dO", "cu_seqlens")
    host["cu_seqlens"] = host["cu_seqlens"].to(torch.int32).pin_memory()
    total = host["q"].shape[0]
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    K = max(2, min(args.steps, 8))
    link = host_link_gbs(dev)   # before the pipeline's own pinned and device buffers exist
    s_in, s_c, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dev_in = [{n: torch.empty(host[n].shape, dtype=host[n].dtype, device=dev) for n in names} for _ in range(2)]
    out_host = [None, None]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_c = [torch.cuda.Event() for _ in range(2)]
    d2h = 0
    spans = []   # per step: (copy-in start, end, copy-out start, end) events, to report the link rate seen

    def issue(i):
        nonlocal d2h
        slot = i & 1
        d = dev_in[slot]
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        spans.append(ev)
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_c[slot])          # step i-2 has finished reading this buffer
            ev[0].record(s_in)
            for n in names:
                d[n].copy_(host[n], non_blocking=True)
            ev[1].record(s_in)
            ev_in[slot].record(s_in)
        with torch.cuda.stream(s_c):
            s_c.wait_event(ev_in[slot])
            ev[4].record(s_c)
            cu = d["cu_seqlens"]
            o, hT, saved = kda.kda_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], cu, d["h0"], save=True)
            gr = kda.kda_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["dO"], saved, cu, d["h0"])
            ev[5].record(s_c)
            ev_c[slot].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[slot])
            if out_host[slot] is None:
                out_host[slot] = {n: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for n, v in gr.items()
                                  if v is not None}
                d2h = sum(v.numel() * v.element_size() for v in out_host[slot].values())
            ev[2].record(s_out)
            for n, v in gr.items():
                if v is not None:
                    out_host[slot][n].copy_(v, non_blocking=True)
                    v.record_stream(s_out)
            ev[3].record(s_out)

    W = 4                                              # warm-up: both slots allocated and used twice
    for i in range(W):
        issue(i)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(W, W + K):
        issue(i)
    end.record(s_out)
    torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end) / K
    ms = reduce_max(ms, world)
    timed = spans[W:]
    cin = sorted(ev[0].elapsed_time(ev[1]) for ev in timed)
    cout = sorted(ev[2].elapsed_time(ev[3]) for ev in timed)
    seen = {"h2d": round(h2d / (cin[len(cin) // 2] * 1e-3) / 1e9, 1),
            "d2h": round(d2h / (cout[len(cout) // 2] * 1e-3) / 1e9, 1),
            "copy_in_ms": round(cin[len(cin) // 2], 2), "copy_out_ms": round(cout[len(cout) // 2], 2)}
    # per timed step, ms from the start of the timed region: copy-in, compute and copy-out spans
    timeline = [[round(start.elapsed_time(ev[a]), 1) for a in (0, 1, 4, 5, 2, 3)] for ev in timed]
    return {"value": world * total / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "pipelining": "copy-in, compute and copy-out on three streams, two buffers each",
            "host_link_gbs": link,
            "link_during_steps_gbs": seen,
            "timeline_ms": {"columns": ["in_start", "in_end", "compute_start", "compute_end", "out_start",
                                        "out_end"], "steps": timeline},
            "note": "bound by the host link (inputs in, fp32 gradients out) and by how the copies overlap the "
                    "compute kernels; host_link_gbs is the pinned copy rate measured alone before the pipeline starts, "
                    "link_during_steps_gbs the median rate of the timed steps' own copies (the two directions overlap)"}


def host_link_gbs(dev, n=1 << 30):
    """Pinned host<->device copy rate right now (one direction at a time, best of 3)."""
    import torch
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    out = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        best = None
        for _ in range(3):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            dst.copy_(src, non_blocking=True)
            e.record()
            torch.cuda.synchronize(dev)
            ms = s.elapsed_time(e)
            best = ms if best is None else min(best, ms)
        out[name] = round(n / (best * 1e-3) / 1e9, 1)
    del h, d
    return out


# ----------------------------------------------------------------------------- oracle
def cpu_baseline(args, steps=1, sample_tokens=None, heads_per_core=4):
    """The fp64 oracle as it stands, timed on this host's cores on a bounded sample of
    the workload: `sample_tokens` tokens of `heads_per_core` x cores heads (at most 96),
    drawn with the workload's recipe and seed."""
    import torch
    import oracle
    from gated_delta_rule_chunked_gb300.inputs import make_seq_batch
    cores = oracle.default_threads()
    Ts = sample_tokens or args.cpu_sample_tokens
    heads = min(96, heads_per_core * cores)
    b = make_seq_batch([Ts], heads=heads, io_dtype="bf16", seed=1002, h0=True, grad=True)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.fwd(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.h0, n_threads=cores)
        oracle.bwd(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.dO, b.h0, n_threads=cores)
    el = (time.perf_counter() - t0) / steps
    # tokens/s of the full 96-head workload = sampled token-heads per second / 96
    val = Ts * heads / el / 96
    return {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fwd+bwd of one {Ts}-token sequence x {heads} heads drawn with the recipe and seed of "
                      f"{WORKLOAD} ({cores} threads, one (sequence, head) task per thread at a time); "
                      f"value = sampled token-heads per second / 96 heads", "seconds": el}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    ms = []
    for _ in range(args.warmup):
        cpu_baseline(args, sample_tokens=args.ref_sample_tokens, heads_per_core=1)
    for _ in range(args.steps):
        r = cpu_baseline(args, sample_tokens=args.ref_sample_tokens, heads_per_core=1)
        ms.append(r["seconds"] * 1e3)
    ms_step = statistics.mean(ms)
    cores = r["cores"]
    val = args.ref_sample_tokens * min(96, cores) / (ms_step * 1e-3) / 96
    return {"impl": "reference", "metric": "KDA fwd+bwd tokens/s (H=96, d=128, T=32768, bf16 I/O, fp32 state/grads)",
            "value": val, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded, same recipe)",
            "config": {"workload": WORKLOAD, "seq_len": 32768, "heads": 96, "head_dim": D},
            "cpu_baseline": {"kind": "oracle", "cores": cores, "value": val, "unit": "tokens/s",
                             "sample": r["sample"]},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- dist
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cp", action="store_true", help="skip the context-parallel forward emulation")
    ap.add_argument("--no-attnres", action="store_true", help="skip the Attention Residuals workload")
    ap.add_argument("--no-conv", action="store_true", help="skip the short-convolution workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-range", action="store_true", help="skip the 4K / inference / 128K / varlen lines")
    ap.add_argument("--range-lines", default="", help="comma-separated keys of the range lines to run "
                    "(fwd_T4096, fwd_T32768_inference, fwdbwd_varlen8_T131072, fwdbwd_T131072, fwdbwd_f32_T4096; "
                    "default all; profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=16384)
    ap.add_argument("--ref-sample-tokens", type=int, default=2048)
    ap.add_argument("--seq-len", type=int, default=0, help="override T (profiling runs only)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        if args.warmup < 3:
            raise SystemExit("--warmup must be >= 3")
        out = run_ours(args, rank, world, local_rank)
    if rank == 0 and out is not None:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
