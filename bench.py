"""Benchmark of the continuous softmax attention forward pass on GB300.

One step = one csa_forward call (the whole hot path: TMA staging, QK^T on
tensor cores, halo + correction b + online softmax, PV on tensor cores,
epilogue) over the headline workload B=1, H=32, T=8192, d=128, bf16,
scale 1/sqrt(d), zero sink, with inputs resident in HBM.  L2 is flushed
(a 512 MiB write) before every timed step; each step is timed with CUDA
events on the launching stream and the steps are summed.

Also reported on the same JSON line:
  e2e          the same metric through the C ABI with host buffers
               (csa_forward_host_ex): pinned host -> device copies of q, k,
               v, the kernels, and the device -> host copy of o and lse, all
               inside the timed region, overlapped by chunks of 8 heads and,
               through two alternating workspaces, across consecutive steps
  std          the library's standard causal attention kernel (eq. (12)) at
               the same shape, and the ratio continuous / standard
  short_conv, symmetric, log_domain
               the other forms of the same step: the first-order reading of
               eq. (13), the symmetric interval, and the interval weights
               formed in the log domain (the reference evaluation)
  roofline     tensor-core bound: algorithmic matmul flops / kernel time
               against the measured dense bf16 peak
  cpu_baseline the CPU oracle (double precision, all host cores) on a
               bounded sample of rows of the same workload
  clocks       nvidia-smi SM clocks and throttle reasons sampled during the
               timed region
  decode       the decode step (csa_decode: the newest token of 16 sequences
               of lengths in [4096, 8192] against their KV cache, H=32,
               d=128), an HBM-bound path: cache bytes read / call time
               against the measured copy bandwidth, plus its own e2e (the
               queries from pinned host memory, outputs back to the host;
               the cache stays resident as it would while serving)
  backward     the backward pass (csa_backward) at the same shape
  workloads    every other workload of the evaluation plan: the continuous
               and standard kernels at the mid (4 x 16 x 2048 x 128, RoPE)
               and long (1 x 8 x 32768 x 64, per-head sink) workloads, with
               tokens/s and an oracle baseline on sampled rows; the tiny
               (fp32, 1 x 1 x 64 x 16) and stress (2 x 4 x 512 x 64, scale
               x sink-mode sweep) workloads with the oracle's full run timed
               beside them

`--impl reference` times the CPU oracle alone (the reference arm).
Multi-GPU (torchrun), two modes:
  default      weak scaling of replicas: every rank runs its own copy of the
               workload (the (b, h) problems are independent; no collective
               on the data path), the time is the max over ranks, and value
               = all ranks' flops / that time
  --shard      strong scaling: the headline's B*H problems are split into N
               contiguous shards (continuous_softmax_attention_gb300.dist:
               the partition forward_sharded uses, no gather in the timed
               region), each rank times the forward and standard kernels on
               its shard, and value = the whole workload's flops / the max
               over ranks; the decode, backward and other-workload legs are
               left out
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

METRIC = "continuous-attn fwd TFLOP/s (B=1,H=32,T=8192,d=128, bf16, causal)"
UNIT = "TFLOP/s"
WORKLOAD = "headline"
E2E_HEADS_PER_CHUNK = 8  # pipeline granularity of the host-buffer path
FALLBACK_BF16_TFLOPS = 1900.0


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "csa_forward_headline.md")
KERNEL_SOURCES = ["csa_tc.cu", "csa_tc_common.cuh", "csa_device.cuh"]
DECODE_PROFILE = os.path.join(ROOT, "profiles", "decode_chunk_bench.md")
DECODE_SOURCES = ["csa_decode.cu", "csa_device.cuh"]
BACKWARD_PROFILE = os.path.join(ROOT, "profiles", "backward_headline.md")
BACKWARD_SOURCES = ["csa_tc_bwd.cu", "csa_tc_common.cuh", "csa_device.cuh"]


def kernel_source_hash(names=KERNEL_SOURCES):
    """sha256 over the sources of one kernel."""
    import hashlib

    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "continuous_softmax_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_figure(path, key, sources):
    """A figure recorded in a committed ncu summary (lines `key: value` and
    `source_sha256: ...`), or None when the kernel's sources changed since
    the counters were taken."""
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                line = line.strip().strip("`")
                for k in (key + ":", "source_sha256:"):
                    if line.startswith(k):
                        fields[k] = line[len(k):].strip()
        if fields.get("source_sha256:") != kernel_source_hash(sources):
            return None
        return float(fields[key + ":"])
    except Exception:
        return None


def recorded_traffic():
    """DRAM bytes per launch of the headline kernel, or None."""
    v = recorded_figure(PROFILE_SUMMARY, "traffic_bytes_per_launch", KERNEL_SOURCES)
    return None if v is None else int(v)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (every 100 ms)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.tmp is None:
            return None
        try:
            rows = [l.strip().split(", ") for l in open(self.tmp.name) if l.strip()]
            os.unlink(self.tmp.name)
        except Exception:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def run_shard_plan(args, ws, rank):
    """Without a GPU (gloo): the partition --shard times, every rank's
    [start, stop) of the headline's flattened (b, h) problems gathered to
    rank 0.  Checks the argument handling and the partition; nothing is
    timed and nothing is computed."""
    import torch.distributed as dist

    from continuous_softmax_attention_gb300.dist import head_shard
    from continuous_softmax_attention_gb300.inputs import WORKLOADS

    w = WORKLOADS[WORKLOAD]
    n = w.B * w.H
    mine = head_shard(n, ws, rank) if args.shard else (0, n)
    ranges = [mine]
    if ws > 1:
        ranges = [None] * ws
        dist.all_gather_object(ranges, mine)
        dist.destroy_process_group()
    if rank != 0:
        return None
    return {"plan": "shard" if args.shard else "replicas", "n_gpus": ws,
            "scaling": "strong" if args.shard else "weak",
            "config": {"workload": WORKLOAD, "B": w.B, "H": w.H, "T": w.T, "d": w.d},
            "ranges": [list(r) for r in ranges], "timed": False}


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import continuous_softmax_attention_gb300 as csa
    from continuous_softmax_attention_gb300.dist import max_over_ranks
    from continuous_softmax_attention_gb300.inputs import WORKLOADS, algorithmic_flops, workload_inputs

    ws, rank, local = _dist_env()
    if ws > 1:
        dist.init_process_group(args.backend)
    if args.backend == "gloo" and not torch.cuda.is_available():  # argument handling only
        return run_shard_plan(args, ws, rank)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[WORKLOAD]
    B, H, T, d = w.B, w.H, w.T, w.d
    scale = 1.0 / math.sqrt(d)
    x = workload_inputs(WORKLOAD)
    flops = algorithmic_flops(B, H, T, d, continuous=True)
    flops_std = algorithmic_flops(B, H, T, d, continuous=False)
    # per-rank work: the whole workload (replicas), or this rank's shard
    rep_world = ws
    if args.shard:
        from continuous_softmax_attention_gb300.dist import shard_inputs

        qs, ks, vs, k0s, v0s, (start, stop) = shard_inputs(x["q"], x["k"], x["v"], x["k0"],
                                                           x["v0"], ws, rank)
        x = {"q": qs.contiguous(), "k": ks.contiguous(), "v": vs.contiguous(),
             "k0": k0s.contiguous(), "v0": v0s.contiguous()}
        B, H = 1, stop - start
        rep_world = 1  # every rank's flops are a share of the one workload
        args.no_decode = args.no_backward = args.no_workloads = True
    g = {k: v.to(dev) for k, v in x.items()}
    out = torch.empty_like(g["q"])
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    e2e_hpc = max(c for c in range(1, min(E2E_HEADS_PER_CHUNK, H) + 1) if H % c == 0)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def timed(fn, steps):
        ms = []
        for _ in range(steps):
            flush.fill_(1.0)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return ms

    csa_call = lambda: csa.forward(g["q"], g["k"], g["v"], mode=w.modes[0], scale=scale, out=out, lse=lse)
    sc_call = lambda: csa.forward(g["q"], g["k"], g["v"], mode=w.modes[0], scale=scale, out=out,
                                  lse=lse, short_conv=True)
    sym_call = lambda: csa.forward_symmetric(g["q"], g["k"], g["v"], scale=scale, out=out, lse=lse)
    ld_call = lambda: csa.forward(g["q"], g["k"], g["v"], mode=w.modes[0], scale=scale, out=out,
                                  lse=lse, log_domain=True)
    std_call = lambda: csa.std_forward(g["q"], g["k"], g["v"], scale=scale, out=out, lse=lse)

    dec = None if args.no_decode else DecodeBench(csa, dev, stream, flush)
    more = None if args.no_workloads else WorkloadBench(csa, dev)
    bwd = None if args.no_backward else BackwardBench(csa, g, out, lse, scale, w.modes[0], dev)

    # end to end through the C ABI with host buffers (csa_forward_host_ex: the
    # copies of one chunk of heads overlap the kernel of another, and with two
    # workspaces one step's copies in overlap the previous step's kernels)
    pin = {k: x[k].pin_memory() for k in ("q", "k", "v")}
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    host_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    pipe = csa.HostForwardPipeline(B, H, T, d, dev, heads_per_chunk=e2e_hpc, stream=stream)

    def e2e_call():
        pipe(pin["q"], pin["k"], pin["v"], host_out, host_lse, mode=w.modes[0], scale=scale)

    def timed_region(fn, steps):
        """steps calls back to back as one timed region: consecutive calls
        overlap, so they are not separated by a synchronisation or a flush
        (every step copies its 201 MB of inputs from the host anyway)."""
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pipe.s_h2d.wait_event(a)  # no copy starts before the region does
        for _ in range(steps):
            fn()
        b.record(stream)
        b.synchronize()
        return [a.elapsed_time(b)]

    h2d = sum(pin[n].numel() * pin[n].element_size() for n in pin)
    d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * host_lse.element_size()

    for _ in range(args.warmup):
        csa_call()
        std_call()
        sc_call()
        sym_call()
        ld_call()
        e2e_call()
        if dec is not None:
            dec.call()
            dec.e2e_call()
        if bwd is not None:
            bwd.call()
        if more is not None:
            more.warm()
    torch.cuda.synchronize()
    assert csa.device_status() == 0

    barrier()
    t_wall = time.perf_counter()
    with ClockSampler(local) as clk:
        ms_csa = timed(csa_call, args.steps)
        ms_std = timed(std_call, args.steps)
        ms_sc = timed(sc_call, args.steps)
        ms_sym = timed(sym_call, args.steps)
        ms_ld = timed(ld_call, args.steps)
        ms_e2e = timed_region(e2e_call, args.steps)
        if dec is not None:
            dec.ms = timed(dec.call, args.decode_steps)
            dec.ms_e2e = timed(dec.e2e_call, args.decode_steps)
        if bwd is not None:
            bwd.ms = timed(bwd.call, args.backward_steps)
        if more is not None:
            more.time(timed, args.workload_steps)
    barrier()
    t_wall = time.perf_counter() - t_wall
    status = csa.device_status()

    def total(ms):
        return max_over_ranks(sum(ms), device=dev)

    tot_csa, tot_std, tot_e2e = total(ms_csa), total(ms_std), total(ms_e2e)
    tot_sc = total(ms_sc)
    tot_sym = total(ms_sym)
    tot_ld = total(ms_ld)
    # every rank takes part in the max over ranks of every leg before the
    # process group goes away
    if dec is not None:
        dec.tot, dec.tot_e2e = total(dec.ms), total(dec.ms_e2e)
    if bwd is not None:
        bwd.tot = total(bwd.ms)
    if more is not None:
        more.reduce(total)
    if ws > 1:
        dist.destroy_process_group()
    if rank != 0:
        return None
    K = args.steps
    ms_step = tot_csa / K
    value = rep_world * flops * K / (tot_csa * 1e-3) / 1e12
    std_value = rep_world * flops_std * K / (tot_std * 1e-3) / 1e12
    e2e_value = rep_world * flops * K / (tot_e2e * 1e-3) / 1e12
    burst, sustained, src = _peaks()
    clocks = clk.summary()
    # the kernel's own rate: this rank's flops per launch over its time
    rank_flops = algorithmic_flops(B, H, T, d, continuous=True)
    rank_flops_std = algorithmic_flops(B, H, T, d, continuous=False)
    achieved = rank_flops / (ms_step * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "strong" if args.shard else "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": w.B, "H": w.H, "T": T, "d": d, "scale": scale,
                   "k0_mode": "zero", "causal": True,
                   "per_gpu": (f"shard of the B*H problems ({H} of {w.B * w.H} on rank 0), "
                               "no gather in the timed region" if args.shard else
                               "full workload per rank (replicas)"),
                   "l2": "flushed (512 MiB write) before every timed step; inputs 192 MiB > L2"},
        "tokens_per_s": round((w.B * T if args.shard else ws * B * T) * K / (tot_csa * 1e-3), 1),
        "pct_bf16_peak": round(100.0 * achieved / burst, 2),
        "std": {"value": round(std_value, 3), "unit": UNIT, "ms_per_step": round(tot_std / K, 5),
                "ratio_continuous_over_std": round(value / std_value, 4)},
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "ms_per_step": round(tot_e2e / K, 5),
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "api": (f"csa_forward_host_ex (CSA_HOST_NO_ENTRY_WAIT), {E2E_HEADS_PER_CHUNK} heads "
                        "per pipeline chunk, two workspaces alternating: each step's copies in "
                        "overlap the previous step's kernels and copies out"),
                "timed": "the K steps back to back as one CUDA-event region"},
        "short_conv": {"value": round(rep_world * flops * K / (tot_sc * 1e-3) / 1e12, 3), "unit": UNIT,
                       "ms_per_step": round(tot_sc / K, 5),
                       "ratio_over_std": round((flops / tot_sc) / (flops_std / tot_std), 4),
                       "note": "first-order (eq. (13)) reading of the same step, csa_forward_short_conv"},
        "symmetric": {"value": round(rep_world * flops_std * K / (tot_sym * 1e-3) / 1e12, 3),
                      "unit": UNIT, "ms_per_step": round(tot_sym / K, 5),
                      "note": "eq. (2) over [1/2, t+1/2] (csa_forward_symmetric); flops over its "
                              "B*H*T(T+1)/2 pairs (no sink)"},
        "log_domain": {"value": round(rep_world * flops * K / (tot_ld * 1e-3) / 1e12, 3), "unit": UNIT,
                       "ms_per_step": round(tot_ld / K, 5),
                       "note": "the same step with z = a + b formed in the log domain "
                               "(csa_forward_logdomain), the reference evaluation of the weights"},
        "gpu_launches": 5 * K + K * (B * H // e2e_hpc) +
                        (0 if dec is None else 2 * 2 * args.decode_steps) +
                        (0 if bwd is None else bwd.launches * args.backward_steps) +
                        (0 if more is None else more.launches * args.workload_steps),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": burst,
                     "unit": "TFLOP/s", "frac": round(achieved / burst, 4),
                     "peak_source": f"{src} bf16 dense (burst)",
                     "traffic": recorded_traffic() if (B, H) == (w.B, w.H) else None,
                     "traffic_unit": "bytes per launch (ncu dram read+write)",
                     "algorithmic_bytes": 2 * 4 * B * H * T * d + 4 * B * H * T},
        "clocks": clocks,
        "device_status": status,
        "wall_s": round(t_wall, 3),
    }
    if dec is not None:
        line["decode"] = dec.summary(ws, args.decode_steps)
    if bwd is not None:
        line["backward"] = bwd.summary(ws, args.backward_steps, burst, src)
    if more is not None:
        line["workloads"] = more.summary(ws, args.workload_steps, burst, src)
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_baseline(x, scale, budget_s=args.cpu_seconds)
        if more is not None:
            more.cpu_baselines(line["workloads"])
        line["short_conv"]["cpu_baseline"] = cpu_baseline_form(x, scale, "short_conv")
        line["symmetric"]["cpu_baseline"] = cpu_baseline_form(x, scale, "symmetric")
        if bwd is not None:
            line["backward"]["cpu_baseline"] = cpu_baseline_backward(x, scale, w.modes[0])
        if dec is not None:
            line["decode"]["cpu_baseline"] = cpu_baseline_decode(dec)
    return line


class WorkloadBench:
    """Every other workload of the evaluation plan on the same line:
      mid    B=4, H=16, T=2048, d=128, RoPE, zero sink
      long   B=1, H=8, T=32768, d=64, per-head sink
    the continuous and standard kernels (the launches their parity tests
    run), with tokens/s and, at N = 1, the oracle on rows sampled from the
    workload; and
      tiny   B=1, H=1, T=64, d=16, fp32 (CUDA-core kernels), scale 1/4
      stress B=2, H=4, T=512, d=64, bf16, scale {1/8, 1, 4} x sink {zero,
             copy-first}
    each run timed on the GPU beside the oracle's full run of the same
    workload (these finish in well under a second on the host)."""

    NAMES = ("mid", "long")

    def __init__(self, csa, dev):
        import torch

        from continuous_softmax_attention_gb300.inputs import (WORKLOADS, algorithmic_flops,
                                                               workload_inputs)
        self.legs = []
        for name in self.NAMES:
            w = WORKLOADS[name]
            x = workload_inputs(name)
            g = {k: t.to(dev) for k, t in x.items()}
            scale = 1.0 / math.sqrt(w.d)
            out = torch.empty_like(g["q"])
            lse = torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=dev)
            mode = w.modes[0]
            cont = (lambda g=g, mode=mode, scale=scale, out=out, lse=lse:
                    csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"], mode=mode, scale=scale,
                                out=out, lse=lse))
            std = (lambda g=g, scale=scale, out=out, lse=lse:
                   csa.std_forward(g["q"], g["k"], g["v"], scale=scale, out=out, lse=lse))
            self.legs.append({"name": name, "w": w, "mode": mode, "calls": (cont, std), "x": x,
                              "scale": scale,
                              "flops": (algorithmic_flops(w.B, w.H, w.T, w.d, continuous=True),
                                        algorithmic_flops(w.B, w.H, w.T, w.d, continuous=False)),
                              "bytes": 3 * g["q"].numel() * 2})
        # the small workloads: one run per (scale, mode)
        self.small = []
        for name in ("tiny", "stress"):
            w = WORKLOADS[name]
            x = workload_inputs(name)
            g = {k: t.to(dev) for k, t in x.items()}
            scales = w.scales or (1.0 / math.sqrt(w.d),)
            runs = []
            for sc in scales:
                for mode in w.modes:
                    runs.append({"scale": sc, "mode": mode,
                                 "call": (lambda g=g, sc=sc, mode=mode:
                                          csa.forward(g["q"], g["k"], g["v"], g["k0"], g["v0"],
                                                      mode=mode, scale=sc))})
                runs[-1]["std"] = (lambda g=g, sc=sc: csa.std_forward(g["q"], g["k"], g["v"],
                                                                      scale=sc))
            self.small.append({"name": name, "w": w, "x": x, "runs": runs,
                               "flops": (algorithmic_flops(w.B, w.H, w.T, w.d, continuous=True),
                                         algorithmic_flops(w.B, w.H, w.T, w.d, continuous=False))})
        n_small = sum(len(sm["runs"]) + sum(1 for r in sm["runs"] if "std" in r)
                      for sm in self.small)
        self.launches = 2 * len(self.legs) + n_small

    def warm(self):
        for leg in self.legs:
            for c in leg["calls"]:
                c()
        for sm in self.small:
            for r in sm["runs"]:
                r["call"]()
                if "std" in r:
                    r["std"]()

    def time(self, timed, steps):
        for leg in self.legs:
            leg["ms"] = [timed(c, steps) for c in leg["calls"]]
        for sm in self.small:
            for r in sm["runs"]:
                r["ms"] = timed(r["call"], steps)
                if "std" in r:
                    r["ms_std"] = timed(r["std"], steps)

    def reduce(self, total):
        for leg in self.legs:
            leg["tot"] = [total(ms) for ms in leg["ms"]]
        for sm in self.small:
            for r in sm["runs"]:
                r["tot"] = total(r["ms"])
                if "std" in r:
                    r["tot_std"] = total(r["ms_std"])

    def summary(self, world, steps, peak, src):
        out = {}
        for leg in self.legs:
            w = leg["w"]
            (fc, fs), (tc, ts) = leg["flops"], leg["tot"]
            vc = world * fc * steps / (tc * 1e-3) / 1e12
            vs = world * fs * steps / (ts * 1e-3) / 1e12
            out[leg["name"]] = {
                "config": {"B": w.B, "H": w.H, "T": w.T, "d": w.d,
                           "k0_mode": ("zero", "copy_first", "given")[leg["mode"]],
                           "rope": bool(w.rope)},
                "value": round(vc, 3), "unit": UNIT, "ms_per_step": round(tc / steps, 5),
                "tokens_per_s": round(world * w.B * w.T * steps / (tc * 1e-3), 1),
                "pct_bf16_peak": round(100.0 * (fc / (tc / steps * 1e-3) / 1e12) / peak, 2),
                "peak_source": f"{src} bf16 dense (burst)",
                "std": {"value": round(vs, 3), "ms_per_step": round(ts / steps, 5)},
                "ratio_continuous_over_std": round(vc / vs, 4),
                "l2": (f"flushed (512 MiB write) before every timed step; q, k, v "
                       f"{leg['bytes'] / 2**20:.0f} MiB"),
            }
        for sm in self.small:
            w = sm["w"]
            fc, fs = sm["flops"]
            runs = []
            std_of = {r["scale"]: r["tot_std"] for r in sm["runs"] if "std" in r}
            for r in sm["runs"]:
                ms = r["tot"] / steps
                entry = {"scale": r["scale"], "k0_mode": ("zero", "copy_first", "given")[r["mode"]],
                         "value": round(world * fc / (ms * 1e-3) / 1e12, 4), "ms_per_step": round(ms, 5),
                         "tokens_per_s": round(world * w.B * w.T / (ms * 1e-3), 1),
                         "pct_bf16_peak": round(100.0 * (fc / (ms * 1e-3) / 1e12) / peak, 4)}
                if r["scale"] in std_of:  # the standard kernel at this scale (no sink)
                    ms_s = std_of[r["scale"]] / steps
                    entry["std"] = {"value": round(world * fs / (ms_s * 1e-3) / 1e12, 4),
                                    "ms_per_step": round(ms_s, 5)}
                    entry["ratio_continuous_over_std"] = round((fc / ms) / (fs / ms_s), 4)
                runs.append(entry)
            out[sm["name"]] = {
                "config": {"B": w.B, "H": w.H, "T": w.T, "d": w.d, "dtype": w.dtype},
                "unit": UNIT, "runs": runs,
                "note": ("fp32 CUDA-core kernels" if w.dtype == "f32" else
                         "bf16 tensor-core kernels") + "; small enough that launch latency "
                        "dominates the GPU time",
                "l2": "flushed (512 MiB write) before every timed step",
            }
        return out

    def cpu_baselines(self, line):
        """The oracle beside each workload: sampled rows for mid and long (as
        the headline's cpu_baseline), the full run of every tiny and stress
        case."""
        import oracle

        cores = oracle.default_threads()
        for leg in self.legs:
            cb = cpu_baseline(leg["x"], leg["scale"], budget_s=4.0, mode=leg["mode"])
            line[leg["name"]]["cpu_baseline"] = cb
        for sm, (name, runs) in zip(self.small, ((s["name"], line[s["name"]]["runs"])
                                                  for s in self.small)):
            x, w = sm["x"], sm["w"]
            fc = sm["flops"][0]
            for r, entry in zip(sm["runs"], runs):
                t0 = time.perf_counter()
                oracle.forward(x["q"], x["k"], x["v"], x["k0"], x["v0"], scale=r["scale"],
                               mode=r["mode"])
                dt = time.perf_counter() - t0
                entry["cpu_baseline"] = {"value": fc / dt / 1e12, "unit": UNIT, "cores": cores,
                                         "kind": "oracle", "seconds": round(dt, 4),
                                         "sample": "the whole workload (eq. (8) in double)"}


class BackwardBench:
    """The backward pass at the headline shape: dq, dk, dv from q, k, v, the
    forward's out and lse, and a seeded upstream gradient (inputs resident)."""

    launches = 3  # D row dot, the tensor-core kernel, the dq conversion

    def __init__(self, csa, g, out, lse, scale, mode, dev):
        import torch

        self.csa, self.g, self.scale, self.mode = csa, g, scale, mode
        B, H, T, d = g["q"].shape
        gen = torch.Generator().manual_seed(7)
        self.dout = torch.randn(B, H, T, d, generator=gen).to(torch.bfloat16).to(dev)
        self.out = torch.empty_like(out)
        self.lse = torch.empty_like(lse)
        csa.forward(g["q"], g["k"], g["v"], mode=mode, scale=scale, out=self.out, lse=self.lse)
        self.grads = [torch.empty_like(g["q"]) for _ in range(3)]
        self.ws = torch.empty(csa.backward_workspace_bytes(B, H, T, d), dtype=torch.uint8,
                              device=dev)
        self.shape = (B, H, T, d)
        self.ms = None

    def call(self):
        g = self.g
        self.csa.backward(g["q"], g["k"], g["v"], self.out, self.lse, self.dout, mode=self.mode,
                          scale=self.scale, dq=self.grads[0], dk=self.grads[1], dv=self.grads[2],
                          workspace=self.ws)

    def summary(self, world, steps, peak, src):
        B, H, T, d = self.shape
        pairs = B * H * T * (T + 3) // 2
        flops = 10 * d * pairs  # S, dP, dV, dK, dQ: 2 d flops each per (query, key) pair
        tot = self.tot  # max over ranks of the timed steps
        ms = tot / steps
        achieved = flops / (ms * 1e-3) / 1e12
        per_head = recorded_figure(BACKWARD_PROFILE, "traffic_bytes_per_head", BACKWARD_SOURCES)
        traffic = None if per_head is None else int(per_head * B * H)
        return {
            "metric": f"continuous-attn bwd TFLOP/s (B={B},H={H},T={T},d={d}, bf16, causal)",
            "value": round(world * achieved, 3), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
            "steps": steps,
            "flops_per_step": flops,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                         "peak_source": f"{src} bf16 dense (burst)", "traffic": traffic,
                         "traffic_unit": "bytes per call (ncu dram read+write of the tensor-core "
                                         "kernel per head, times this workload's heads)",
                         "algorithmic_bytes": 2 * 8 * B * H * T * d + 4 * B * H * T,
                         "timed": "whole csa_backward call (D row dot, tensor-core kernel, dq "
                                  "conversion)"},
            "gpu_launches_per_step": self.launches,
        }


class DecodeBench:
    """The decode workload: resident cache, one csa_decode call per step."""

    def __init__(self, csa, dev, stream, flush):
        import torch

        from continuous_softmax_attention_gb300.inputs import (DECODE_WORKLOADS, decode_bytes,
                                                               decode_workload_inputs)

        self.w = w = DECODE_WORKLOADS["decode"]
        x = decode_workload_inputs("decode")
        self.lens = x["seqlens"].tolist()
        self.host = x
        self.bytes = decode_bytes(self.lens, w.H, w.d)
        g = {k: t.to(dev) for k, t in x.items()}
        self.q, self.k, self.v, self.sl = g["q"], g["k"], g["v"], g["seqlens"]
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
        self.ws = torch.empty(csa.decode_workspace_bytes(w.B, w.H, w.T, w.d), dtype=torch.uint8,
                              device=dev)
        self.pin_q = x["q"].pin_memory()
        self.dq = torch.empty_like(self.q)
        self.host_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.host_lse = torch.empty(self.lse.shape, dtype=self.lse.dtype).pin_memory()
        self.csa = csa
        self.ms = self.ms_e2e = None

    def call(self):
        self.csa.decode(self.q, self.k, self.v, seqlens=self.sl, mode=self.w.mode, out=self.out,
                        lse=self.lse, workspace=self.ws)

    def e2e_call(self):
        self.dq.copy_(self.pin_q, non_blocking=True)
        self.csa.decode(self.dq, self.k, self.v, seqlens=self.sl, mode=self.w.mode, out=self.out,
                        lse=self.lse, workspace=self.ws)
        self.host_out.copy_(self.out, non_blocking=True)
        self.host_lse.copy_(self.lse, non_blocking=True)

    def summary(self, world, steps):
        w = self.w
        tot, tot_e2e = self.tot, self.tot_e2e  # max over ranks of the timed steps
        ms = tot / steps
        gbs = world * self.bytes * steps / (tot * 1e-3) / 1e9
        gbs_e2e = world * self.bytes * steps / (tot_e2e * 1e-3) / 1e9
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                peak, src = float(json.load(f)["hbm_gbs"]), "measured"
        except Exception:
            peak, src = 6800.0, "fallback"
        achieved = self.bytes / (ms * 1e-3) / 1e9
        per_pos = recorded_figure(DECODE_PROFILE, "traffic_bytes_per_position", DECODE_SOURCES)
        traffic = None if per_pos is None else int(per_pos * sum(self.lens) * w.H)
        h2d = self.pin_q.numel() * self.pin_q.element_size()
        d2h = (self.host_out.numel() * self.host_out.element_size() +
               self.host_lse.numel() * self.host_lse.element_size())
        return {
            "metric": f"continuous-attn decode step HBM GB/s (B={w.B},H={w.H},T<={w.T},d={w.d}, bf16)",
            "value": round(gbs, 2), "unit": "GB/s", "ms_per_step": round(ms, 5), "steps": steps,
            "tokens_per_s": round(world * w.B * steps / (tot * 1e-3), 1),
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T_capacity": w.T, "d": w.d,
                       "lengths": f"uniform in [{w.len_lo}, {w.T}], total {sum(self.lens)}",
                       "k0_mode": "zero", "l2": "512 MiB flush before every step; cache "
                       f"{2 * sum(self.lens) * w.H * w.d * 2 / 2**30:.2f} GiB > L2"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": f"{src} copy bandwidth", "traffic": traffic,
                         "traffic_unit": "bytes per call (ncu dram read+write of the chunk "
                                         "kernel per (b, h, position), times this workload's)",
                         "algorithmic_bytes": self.bytes,
                         "timed": "whole csa_decode call (chunk kernel + merge kernel)"},
            "e2e": {"value": round(gbs_e2e, 2), "unit": "GB/s", "ms_per_step": round(tot_e2e / steps, 5),
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "note": "queries copied in and outputs copied out each step; cache resident"},
            "gpu_launches_per_step": 2,
        }


def _sample_rows(T, H, nrows, seed=0):
    import numpy as np

    rng = np.random.default_rng(seed)
    picks = [(0, int(h), int(r)) for h, r in zip(rng.integers(0, H, nrows), rng.integers(0, T, nrows))]
    return picks


def cpu_baseline(x, scale, budget_s=15.0, seed=0, mode=0):
    """The oracle (eq. (8), double, all host cores) on rows sampled uniformly
    from the workload; rate = algorithmic flops of those rows / wall time."""
    import numpy as np

    import oracle

    B, H, T, d = x["q"].shape
    q = x["q"].float().numpy()
    k = x["k"].float().numpy()
    v = x["v"].float().numpy()
    k0 = x["k0"].float().numpy() if mode == 2 else None
    v0 = x["v0"].float().numpy() if mode == 2 else None
    cores = oracle.default_threads()
    # calibrate on a small sample, then size the timed one to the budget
    n = 16 * cores
    while True:
        picks = _sample_rows(T, H, n, seed)
        rows = oracle.flat_rows(B, H, T, picks)
        t0 = time.perf_counter()
        oracle.forward_rows(q, k, v, rows, k0, v0, scale=scale, mode=mode, nthreads=cores)
        dt = time.perf_counter() - t0
        if dt > 0.25 * budget_s or n >= 1 << 20:
            break
        n = int(n * min(8.0, max(2.0, 0.5 * budget_s / max(dt, 1e-3))))
    pairs = sum(r + 2 for (_, _, r) in picks)
    rate = 4.0 * d * pairs / dt / 1e12
    return {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(picks)} rows drawn uniformly from the {B}x{H}x{T}x{d} workload "
                      f"(eq. (8) in double, {dt:.1f} s)",
            "seconds": round(dt, 3)}


def cpu_baseline_form(x, scale, form, budget_s=4.0, seed=1):
    """The oracle of the short-conv or symmetric form on rows sampled from the
    workload (double, all host cores); rate = algorithmic flops / wall time."""
    import oracle

    B, H, T, d = x["q"].shape
    q, k, v = (x[n].float().numpy() for n in ("q", "k", "v"))
    cores = oracle.default_threads()
    fn = oracle.forward_short_conv_rows if form == "short_conv" else oracle.forward_symmetric_rows
    per_row = (lambda r: r + 2) if form == "short_conv" else (lambda r: r + 1)
    n = 16 * cores
    while True:
        picks = _sample_rows(T, H, n, seed)
        rows = oracle.flat_rows(B, H, T, picks)
        t0 = time.perf_counter()
        fn(q, k, v, rows, scale=scale, nthreads=cores)
        dt = time.perf_counter() - t0
        if dt > 0.25 * budget_s or n >= 1 << 20:
            break
        n = int(n * min(8.0, max(2.0, 0.5 * budget_s / max(dt, 1e-3))))
    rate = 4.0 * d * sum(per_row(r) for (_, _, r) in picks) / dt / 1e12
    return {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(picks)} rows drawn uniformly from the {B}x{H}x{T}x{d} workload "
                      f"({form} form in double, {dt:.1f} s)",
            "seconds": round(dt, 3)}


def cpu_baseline_backward(x, scale, mode, T_sample=1024):
    """The backward oracle (chain rule, double) on causal prefixes of one head
    per host core (the heads run in parallel); rate = 10 d flops per pair /
    wall time."""
    import torch

    import oracle

    cores = oracle.default_threads()
    B, H, T, d = x["q"].shape
    hs = min(H, cores)
    Ts = min(T, T_sample)
    sl = lambda t: t[:, :hs, :Ts].contiguous()
    g = torch.randn(1, hs, Ts, d, generator=torch.Generator().manual_seed(3))
    t0 = time.perf_counter()
    oracle.backward(sl(x["q"]), sl(x["k"]), sl(x["v"]), g, x["k0"][:hs], x["v0"][:hs],
                    scale=scale, mode=mode, nthreads=cores)
    dt = time.perf_counter() - t0
    flops = 10.0 * d * hs * Ts * (Ts + 3) / 2
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": min(cores, hs), "kind": "oracle",
            "sample": f"{hs} heads x the first {Ts} rows of the {B}x{H}x{T}x{d} workload "
                      f"(chain rule in double, {dt:.1f} s)",
            "seconds": round(dt, 3)}


def cpu_baseline_decode(dec, budget_s=4.0):
    """The oracle (eq. (8) row n_b of each sequence, double, all host cores)
    on the decode workload's first sequences; rate = their cache bytes /
    wall time."""
    import torch

    import oracle

    cores = oracle.default_threads()
    x, w = dec.host, dec.w
    done, nbytes, t_all = 0, 0, 0.0
    while done < w.B and t_all < budget_s:
        n = dec.lens[done]
        qf = torch.zeros(1, w.H, n, w.d)
        qf[0, :, n - 1] = x["q"][done].float()
        rows = oracle.flat_rows(1, w.H, n, [(0, h, n - 1) for h in range(w.H)])
        t0 = time.perf_counter()
        oracle.forward_rows(qf, x["k"][done:done + 1, :, :n], x["v"][done:done + 1, :, :n], rows,
                            scale=1.0 / math.sqrt(w.d), nthreads=cores)
        t_all += time.perf_counter() - t0
        nbytes += 2 * n * w.H * w.d * 2
        done += 1
    return {"value": round(nbytes / t_all / 1e9, 3), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"the first {done} of {w.B} sequences, all {w.H} heads (eq. (8) row n_b "
                      f"in double, {t_all:.1f} s; the conversion of the cache to float32 is not "
                      f"timed)",
            "seconds": round(t_all, 3)}


def run_reference(args):
    """Reference arm: the CPU oracle on bounded samples of the same workload."""
    import numpy as np

    from continuous_softmax_attention_gb300.inputs import WORKLOADS, workload_inputs

    import oracle

    ws, rank, _ = _dist_env()
    if rank != 0:
        return None
    w = WORKLOADS[WORKLOAD]
    x = workload_inputs(WORKLOAD)
    q, k, v = (x[n].float().numpy() for n in ("q", "k", "v"))
    B, H, T, d = q.shape
    scale = 1.0 / math.sqrt(d)
    cores = oracle.default_threads()
    rows_per_step = max(cores, int(args.ref_rows))
    for s in range(args.warmup):
        picks = _sample_rows(T, H, max(cores, rows_per_step // 8), seed=100 + s)
        oracle.forward_rows(q, k, v, oracle.flat_rows(B, H, T, picks), scale=scale, nthreads=cores)
    tot = 0.0
    flops = 0.0
    for s in range(args.steps):
        picks = _sample_rows(T, H, rows_per_step, seed=s)
        rows = oracle.flat_rows(B, H, T, picks)
        t0 = time.perf_counter()
        oracle.forward_rows(q, k, v, rows, scale=scale, nthreads=cores)
        tot += time.perf_counter() - t0
        flops += 4.0 * d * sum(r + 2 for (_, _, r) in picks)
    value = flops / tot / 1e12
    sample = (f"{rows_per_step} rows per step drawn uniformly from the {B}x{H}x{T}x{d} workload "
              f"(eq. (8) in double on {cores} host threads)")
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "T": T, "d": d, "scale": scale,
                   "k0_mode": "zero", "causal": True},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-rows", type=int, default=256, help="oracle rows per reference step")
    ap.add_argument("--decode-steps", type=int, default=200, help="timed steps of the decode workload")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode workload")
    ap.add_argument("--backward-steps", type=int, default=50, help="timed steps of the backward pass")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward pass")
    ap.add_argument("--workload-steps", type=int, default=20,
                    help="timed steps of each kernel at the mid and long workloads")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads (mid, long, tiny, stress)")
    ap.add_argument("--shard", action="store_true",
                    help="strong scaling: split the headline's (b, h) problems over the ranks")
    ap.add_argument("--backend", choices=["nccl", "gloo"], default="nccl",
                    help="process-group backend (gloo without a GPU checks the shard plan only)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
