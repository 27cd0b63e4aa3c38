#!/usr/bin/env python3
"""Benchmark of the packed varlen causal attention path on GB300.

One step = the whole hot path over one synthetic packed batch:
  positions + labels  ->  forward attention (work list, RoPE table, k rotated once, tcgen05
  kernel rotating the q tiles, which also returns q', k')  ->  backward attention on q', k'
  (work lists, delta, dQ pass, dK/dV pass).  --rope once instead rotates q, k by one pass
  before the forward.
Metric: effective TFLOP/s counting only in-segment causal FLOPs of real (non-pad)
segments, 4*d*H*pairs (forward) + 10*d*H*pairs (backward); packed real tokens/s
is reported beside it.  Default workload: the pretraining-window forward+backward pack
(32 x 4096 tokens, lognormal(400, 0.8) document lengths clipped to [32, 4096] and packed
first-fit-decreasing, H=32, d=128, with dO), the largest single-GPU shape with a backward.
The line's extras also time the forward alone on the 4K-window pack and on the
131072-token long-context buffer (per-iteration CUDA events over >= 300 iterations,
median and min), in both RoPE forms: rotation fused into the forward kernel, and q, k
rotated once by a separate pass followed by the kernel on the rotated operands.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

With --impl reference the fp64 CPU oracle is timed on the host cores instead (a
bounded sample of the same workload per step).  Under torchrun each rank runs its
own independently seeded pack on its own GPU (weak scaling, no collective on the
data path); rank 0 prints one JSON line.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from variable_length_causal_gb300 import synth  # noqa: E402

METRIC = "varlen causal attn effective TFLOP/s (in-segment FLOPs only); packed tokens/s"
UNIT = "TFLOP/s"
WORKLOAD_BY_NAME = {n: i for i, n in enumerate(synth.WORKLOAD_NAMES)}
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ----------------------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
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
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workload
def make_inputs(w: synth.Workload, device, rank: int):
    seed = 1000 + max(w.index, 0) + 7919 * rank
    q, k, v, g = synth.make_tensors(w, device=device, seed=seed, with_grad=True)
    tokens = torch.from_numpy(synth.make_tokens(w, seed=2000 + w.index + rank)).to(device)
    cu = torch.from_numpy(w.cu).to(device)
    ign = torch.from_numpy(w.seg_ignore).to(device)
    return q, k, v, g, tokens, cu, ign


class Step:
    """Pre-allocated buffers and one call per path step (no allocation inside the step)."""

    def __init__(self, vlc, w, q, k, v, g, tokens, cu, ign, fwd_only=False, rope="once"):
        self.vlc, self.w = vlc, w
        self.q, self.k, self.v, self.g, self.tokens, self.cu, self.ign = q, k, v, g, tokens, cu, ign
        dev = q.device
        self.o = torch.empty_like(q)
        self.lse = torch.empty((w.H, w.total), dtype=torch.float32, device=dev)
        self.fwd_only = fwd_only
        # "once": q, k rotated by one pass for both directions; "fused": RoPE in the forward kernel,
        # which returns q', k' for the backward (forward-only: the plain forward with RoPE in the kernel)
        self.rope = rope
        if fwd_only:
            self.dq = self.dk = self.dv = None
        else:
            self.dq, self.dk, self.dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        self.ws_f = vlc.new_workspace(w.nseg, w.total, w.H, w.d, w.max_seqlen, False, dev)
        # q' and k' for the step: rotated once, read by the forward and the backward
        self.qr, self.kr = torch.empty_like(q), torch.empty_like(k)
        self.ws_b = None if fwd_only else vlc.new_workspace(w.nseg, w.total, w.H, w.d, w.max_seqlen, True, dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    fwd_only = False

    def __call__(self, ev=None):
        vlc, w = self.vlc, self.w
        if ev is not None:
            ev[0].record()
        self.pos, self.lab = vlc.build_positions_labels(self.cu, self.tokens, self.ign, err=self.err)
        if ev is not None:
            ev[1].record()
        once = self.rope == "once"
        if once:
            vlc.rope_qk(self.q, self.k, self.cu, w.max_seqlen, rope_theta=w.theta, out=(self.qr, self.kr),
                        workspace=self.ws_f, check=False)
            vlc.varlen_attn_fwd(self.qr, self.kr, self.v, self.cu, w.max_seqlen, rope_theta=w.theta, out=self.o,
                                lse=self.lse, workspace=self.ws_f, check=False, qk_rotated=True)
        elif self.fwd_only:
            vlc.varlen_attn_fwd(self.q, self.k, self.v, self.cu, w.max_seqlen, rope_theta=w.theta, out=self.o,
                                lse=self.lse, workspace=self.ws_f, check=False)
        else:   # RoPE in the forward kernel, which also returns q', k' for the backward
            vlc.varlen_attn_fwd_rot(self.q, self.k, self.v, self.cu, w.max_seqlen, rope_theta=w.theta,
                                    out=self.o, lse=self.lse, rotated_out=(self.qr, self.kr), workspace=self.ws_f,
                                    check=False)
        if ev is not None:
            ev[2].record()
        if not self.fwd_only:
            vlc.varlen_attn_bwd(self.g, self.qr, self.kr, self.v, self.o, self.lse, self.cu, w.max_seqlen,
                                rope_theta=w.theta, dq=self.dq, dk=self.dk, dv=self.dv, workspace=self.ws_b,
                                check=False, qk_rotated=True)
        if ev is not None:
            ev[3].record()

    def check_errors(self):
        for ws in (self.ws_f,) + (() if self.ws_b is None else (self.ws_b,)):
            st, bits = self.vlc.get_error(ws)
            if st != 0:
                raise RuntimeError(f"device error status {st} bits 0x{bits:x}")
        if int(self.err.item()) != 0:
            raise RuntimeError("positions/labels reported invalid cu_seqlens")


# posl; rotation (worklist and table in one launch + q'/k'); forward (worklist + attention);
# backward (2 worklists and table in one launch + delta + dq + dkdv).  With RoPE in the
# kernels there is no rotation pass; the forward adds its pass that rotates k once (the
# attention kernel rotates the q tiles).
def launches_per_step(w, fwd_only, rope):
    rot = 2 if rope == "once" else 0
    krot = 1 if rope == "fused" else 0
    return 1 + rot + 2 + krot + (0 if fwd_only else 4)


# ----------------------------------------------------------------------------- oracle arm
# Legal (query, key) pairs in one oracle sample: about 5 s of fp64 forward + backward on 16
# host cores.  Both the cpu_baseline leg and the reference arm time this same sample, so
# they report one number.
ORACLE_SAMPLE_PAIRS = 40_000_000


def oracle_sample(w: synth.Workload, threads: int):
    """(segment, head) pairs of real segments, drawn in a seeded order until they hold
    ORACLE_SAMPLE_PAIRS legal pairs and at least 8 pairs per host thread; returned longest
    segment first, so that the host threads' dynamic schedule ends together.  The same
    workload and thread count always give the same sample (no timing decides it)."""
    rng = np.random.default_rng(12345)
    real = np.nonzero(w.seg_ignore == 0)[0]
    order = rng.permutation(len(real))
    heads = rng.integers(0, w.H, size=len(order))
    pairs, total_pairs = [], 0
    for i, h in zip(order, heads):
        r = int(real[i])
        L = int(w.lengths[r])
        pairs.append((r, int(h)))
        total_pairs += L * (L + 1) // 2
        if total_pairs >= ORACLE_SAMPLE_PAIRS and len(pairs) >= 8 * threads:
            break
    pairs.sort(key=lambda p: (-int(w.lengths[p[0]]), p[0], p[1]))
    return pairs, total_pairs


def _sample_text(w, pairs, npairs):
    return (f"{len(pairs)} (segment, head) pairs of the {w.name} pack ({npairs} legal pairs, "
            f"drawn with a fixed seed, longest first): fwd + bwd in fp64, plus positions/labels "
            f"of the whole pack")


def run_oracle_step(w, q, k, v, g, tokens_np, pairs):
    import oracle

    oracle.positions_labels(w.cu, tokens_np, w.seg_ignore)
    oracle.attn_fwd(q, k, v, w.cu, seg_heads=pairs)
    oracle.attn_bwd(g, q, k, v, w.cu, seg_heads=pairs)


def reference_arm(args, w, world, rank):
    if rank != 0:
        return
    import oracle

    oracle.build()
    q, k, v, g = (oracle.bf16_bits(t) for t in synth.make_tensors(w, seed=1000 + w.index, with_grad=True))
    tokens_np = synth.make_tokens(w)
    pairs, npairs = oracle_sample(w, oracle.num_threads())
    for _ in range(args.warmup):
        run_oracle_step(w, q, k, v, g, tokens_np, pairs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle_step(w, q, k, v, g, tokens_np, pairs)
    dt = (time.perf_counter() - t0) / args.steps
    flops = 14.0 * w.d * npairs
    value = flops / dt / 1e12
    tok = sum(int(w.lengths[r]) for r, _ in pairs) / w.H
    sample = _sample_text(w, pairs, npairs) + f"; one sample per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w, world, "oracle sample"),
        "tokens_per_s": tok / dt,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(w, world, flush):
    return {"workload": f"{w.name}: {w.description}", "nseg": w.nseg, "real_segments": int((w.seg_ignore == 0).sum()),
            "total_tokens": w.total, "real_tokens": int(w.real_lengths.sum()), "H": w.H, "head_dim": w.d,
            "max_seqlen": w.max_seqlen, "rope_theta": w.theta, "legal_pairs": synth.causal_pairs(w.real_lengths),
            "tile_efficiency_128": round(synth.tile_efficiency(w), 4),
            "slot_efficiency": round(float(w.real_lengths.sum()) / w.total, 4),
            "parallelism": f"dp{world} (independent packs per GPU)", "l2": flush}


# ----------------------------------------------------------------------------- GPU arm
def gpu_arm(args, w, world, rank, local):
    import variable_length_causal_gb300 as vlc

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    vlc.load_library()
    peaks = _peaks()
    q, k, v, g, tokens, cu, ign = make_inputs(w, dev, rank)
    if args.fwd_only:
        g = None
    step = Step(vlc, w, q, k, v, g, tokens, cu, ign, fwd_only=args.fwd_only, rope=args.rope)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    step.check_errors()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for i in range(args.steps):
            step(evs[i])
        stop.record()
        torch.cuda.synchronize()
    barrier(world)
    step.check_errors()
    ms_local = start.elapsed_time(stop) / args.steps
    ms = max_over_ranks(ms_local, world, dev)
    per_pos = [e[0].elapsed_time(e[1]) for e in evs]
    per_fwd = [e[1].elapsed_time(e[2]) for e in evs]
    per_bwd = [e[2].elapsed_time(e[3]) for e in evs]
    t_pos, t_fwd, t_bwd = (statistics.mean(x) for x in (per_pos, per_fwd, per_bwd))

    fl_f, fl_b = synth.fwd_flops(w), (0.0 if args.fwd_only else synth.bwd_flops(w))
    flops_all = sum_over_ranks(fl_f + fl_b, world, dev)
    real_tok = sum_over_ranks(float(w.real_lengths.sum()), world, dev)
    value = flops_all / (ms * 1e-3) / 1e12

    # ---- end to end through the public API, pinned host buffers in and out
    e2e = None if args.no_e2e else e2e_measure(vlc, w, step, args.steps, world, dev, args.e2e_readback)

    if rank != 0:
        return
    tb = w.total * w.H
    fwd_tflops = fl_f / (t_fwd * 1e-3) / 1e12
    bwd_tflops = fl_b / (t_bwd * 1e-3) / 1e12 if t_bwd > 0 and fl_b > 0 else 0.0
    pos_bytes = 20.0 * w.total
    kernels = {
        "positions_labels": {"ms": t_pos, "GB/s": pos_bytes / (t_pos * 1e-3) / 1e9},
        "attn_fwd_call": {"ms": t_fwd, "ms_median": statistics.median(per_fwd), "ms_min": min(per_fwd),
                          "eff_TFLOP/s": fwd_tflops,
                          "kernels": ("rotation (meta_kernel: work list + RoPE table; rope_qk_kernel) + meta_kernel "
                                      "(work list) + attn_fwd_kernel" if args.rope == "once" else
                                      "meta_kernel (work list + RoPE table) + rope_qk_kernel (k only) + attn_fwd_kernel "
                                      "(q rotated in the kernel)")},
        "attn_bwd_call": {"ms": t_bwd, "ms_median": statistics.median(per_bwd), "ms_min": min(per_bwd),
                          "eff_TFLOP/s": bwd_tflops,
                          "kernels": "meta_kernel (2 work lists + RoPE tables) + prep_kernel (delta) + dq_kernel + dkdv_kernel"},
    }
    dominant = "attn_bwd_call" if t_bwd >= t_fwd else "attn_fwd_call"
    ach = bwd_tflops if dominant == "attn_bwd_call" else fwd_tflops
    traffic = (_traffic_from_profiles(dominant if args.rope == "once" else dominant + "_fused", w.name)
               if args.bins is None else None)
    roofline = {"bound": "tensor", "kernel": dominant, "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "traffic": traffic,
                "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                "peak_source": f"{peaks['source']} bf16 burst",
                "algorithmic": ("10*d*H*pairs" if dominant == "attn_bwd_call" else "4*d*H*pairs")
                + " FLOP per call, real segments only"}
    roofline_fwd = {"bound": "tensor", "achieved": fwd_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": fwd_tflops / peaks["bf16_tflops"],
                    "frac_of_sustained": fwd_tflops / peaks["bf16_tflops_sustained"]}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _config(w, world, f"inputs larger than L2 ({4 * tb * w.d * 2 / 2**30:.1f} GiB q/k/v/dO vs 129 MB)"),
        "tokens_per_s": real_tok / (ms * 1e-3),
        "fwd_eff_tflops": fwd_tflops, "bwd_eff_tflops": bwd_tflops,
        "kernels": kernels, "roofline": roofline, "roofline_fwd": roofline_fwd,
        "gpu_launches": launches_per_step(w, args.fwd_only, args.rope) * args.steps,
        "rope": ("q, k rotated once per step (vlc_rope_qk), both passes on the rotated operands"
                 if args.rope == "once" else
                 "RoPE in the forward kernel (k rotated by its k pass, q tiles inside the kernel), which returns "
                 "q', k'; the backward runs on them"),
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    if not args.no_extras and args.bins is None and world == 1:
        which = EXTRAS if args.extras == "all" else tuple(args.extras.split(","))
        line["extras"] = extra_measurements(vlc, w, dev, peaks, q, k, v, step, which)
        if "forward_configs" in which:
            line["extras"]["forward_configs"] = forward_configs(vlc, dev, peaks)
        if "step_form" in which and not args.fwd_only:
            line["extras"]["step_other_rope_form"] = step_form_measurement(
                vlc, w, q, k, v, g, tokens, cu, ign, "fused" if args.rope == "once" else "once")
        if "cp" in which:
            line["extras"]["context_parallel"] = context_parallel_measurement(vlc, dev, peaks)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, q, k, v, g, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def _time_ms(fn, reps: int) -> float:
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _time_events(fn, reps: int):
    """Per-iteration CUDA events around ``reps`` back-to-back calls (no synchronisation
    between them): (median ms, min ms)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in evs:
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    ts = [a.elapsed_time(b) for a, b in evs]
    return statistics.median(ts), min(ts)


def forward_configs(vlc, dev, peaks, reps: int = 300):
    """The forward alone on the 4K-window pack (32 x 4096 tokens) and on the 131072-token
    long-context buffer, H = 32, d = 128, RoPE theta 10000 with the per-segment reset, in
    both forms: ``fused_rope`` (vlc_attn_fwd: the rotation runs on the staged tiles inside
    the attention kernel) and ``rotate_once`` (vlc_rope_qk writes q', k', then the kernel
    runs on them; the form a training step uses, since the backward reuses q', k').
    Effective TFLOP/s = 4 d H pairs / median call time; frac against the measured bf16
    burst peak; traffic = DRAM bytes per call from the committed ncu capture, when it was
    taken on the current sources."""
    out = {}
    with ClockSampler(dev.index or 0) as clk:
        for name in ("pt", "long"):
            w = synth.workload(WORKLOAD_BY_NAME[name])
            q, k, v = synth.make_tensors(w, device=dev, seed=1000 + w.index)
            cu = torch.from_numpy(w.cu).to(dev)
            o = torch.empty_like(q)
            lse = torch.empty((w.H, w.total), dtype=torch.float32, device=dev)
            qr, kr = torch.empty_like(q), torch.empty_like(k)
            ws = vlc.new_workspace(w.nseg, w.total, w.H, w.d, w.max_seqlen, False, dev)

            def fused():
                vlc.varlen_attn_fwd(q, k, v, cu, w.max_seqlen, rope_theta=w.theta, out=o, lse=lse, workspace=ws,
                                    check=False)

            def rotate_once():
                vlc.rope_qk(q, k, cu, w.max_seqlen, rope_theta=w.theta, out=(qr, kr), workspace=ws, check=False)
                vlc.varlen_attn_fwd(qr, kr, v, cu, w.max_seqlen, rope_theta=w.theta, out=o, lse=lse, workspace=ws,
                                    check=False, qk_rotated=True)

            fl = synth.fwd_flops(w)
            res = {"workload": f"{w.name}: {w.description}", "total_tokens": w.total,
                   "legal_pairs": synth.causal_pairs(w.real_lengths), "reps": reps}
            for form, fn in (("fused_rope", fused), ("rotate_once", rotate_once)):
                med, mn = _time_events(fn, reps)
                st, bits = vlc.get_error(ws)
                if st != 0:
                    raise RuntimeError(f"{name} {form}: device error status {st} bits 0x{bits:x}")
                tf = fl / (med * 1e-3) / 1e12
                res[form] = {"ms_median": med, "ms_min": mn, "eff_TFLOP/s": tf,
                             "eff_TFLOP/s_at_min": fl / (mn * 1e-3) / 1e12,
                             "frac": tf / peaks["bf16_tflops"],
                             "frac_of_sustained": tf / peaks["bf16_tflops_sustained"],
                             "traffic": _traffic_from_profiles(f"fwd_{form}", name)}
            out[name] = res
            del q, k, v, o, lse, qr, kr, ws
            torch.cuda.empty_cache()
    out["clocks"] = clk.summary()
    out["peak"] = {"bf16_tflops": peaks["bf16_tflops"], "source": f"{peaks['source']} bf16 burst",
                   "bf16_tflops_sustained": peaks["bf16_tflops_sustained"]}
    return out


def step_form_measurement(vlc, w, q, k, v, g, tokens, cu, ign, rope, reps: int = 30):
    """The same step with the other RoPE form (median of per-step CUDA events)."""
    st = Step(vlc, w, q, k, v, g, tokens, cu, ign, rope=rope)
    med, mn = _time_events(st, reps)
    st.check_errors()
    fl = synth.fwd_flops(w) + synth.bwd_flops(w)
    return {"rope": rope, "ms_median": med, "ms_min": mn, "eff_TFLOP/s": fl / (med * 1e-3) / 1e12}


def context_parallel_measurement(vlc, dev, peaks, L: int = 131072, cp: int = 4, H: int = 32, d: int = 128,
                                 reps: int = 5):
    """One 131072-token document split over a 4-rank context-parallel group (2 cp chunks, rank i
    holding chunks i and 2cp-1-i), the ranks' work run one after another on this GPU: every
    rank rotates its rows by their positions in the document, computes its blocks of the ring
    (the chunk's own causal block, and every earlier chunk with all keys visible) and merges
    the partial results.  The backward of a rank: every block's backward with the merged O and
    LSE of its query half, its dq parts summed and taken back through R(pos)^T, and the dk / dv
    parts of its own key halves summed (as many as the ring's blocks deliver; on one GPU the
    parts summed are stand-ins of the right shape and count, the arithmetic is the same) and dk
    taken back through R(pos)^T.  No communication is timed (one GPU).  Compared with the whole
    document's causal forward / backward on this GPU: balance = max rank time / mean rank time,
    and split overhead = cp * mean rank time / whole-document time."""
    w = synth.custom_workload([L], H, d)
    q, k, v, g = synth.make_tensors(w, device=dev, seed=4321, with_grad=True)
    cu = torch.from_numpy(w.cu).to(dev)
    qr, kr = vlc.rope_qk(q, k, cu, L)
    o1 = torch.empty_like(q)
    l1 = torch.empty((H, L), dtype=torch.float32, device=dev)
    ws1 = vlc.new_workspace(1, L, H, d, L, False, dev)
    full_ms, _ = _time_events(lambda: vlc.varlen_attn_fwd(qr, kr, v, cu, L, out=o1, lse=l1, workspace=ws1,
                                                          check=False, qk_rotated=True), reps)
    wsb1 = vlc.new_workspace(1, L, H, d, L, True, dev)
    gq1, gk1, gv1 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    full_bwd_ms, _ = _time_events(lambda: vlc.varlen_attn_bwd(g, qr, kr, v, o1, l1, cu, L, dq=gq1, dk=gk1, dv=gv1,
                                                              workspace=wsb1, check=False, qk_rotated=True), reps)
    del o1, l1, ws1, wsb1, gq1, gk1, gv1
    locs = {}
    for r in range(cp):
        rows, pos, cu_chunk = vlc.cp_partition(w.cu, cp, r)
        rows_d = torch.from_numpy(rows).to(dev)
        locs[r] = (rows_d, torch.from_numpy(pos).to(dev), torch.from_numpy(cu_chunk).to(dev), q[rows_d].contiguous(),
                   k[rows_d].contiguous(), v[rows_d].contiguous(), g[rows_d].contiguous())
    half = L // cp // 2
    m = L // (2 * cp)
    # how many block gradients reach each key half (rank, half) in the ring
    into = {(s2, kh): 0 for s2 in range(cp) for kh in (0, 1)}
    for r2 in range(cp):
        for qh in (0, 1):
            for s2 in range(cp):
                for kh in (0, 1):
                    if vlc.cp_block_mode(cp, r2, qh, s2, kh) != vlc.binding.CP_BLOCK_NONE:
                        into[(s2, kh)] += 1
    rank_ms, rank_bwd_ms = [], []
    for r in range(cp):
        rows_d, pos_d, cuc, ql, kl, vl, gl = locs[r]
        qrl, krl = torch.empty_like(ql), torch.empty_like(kl)
        wsr = torch.empty(vlc.load_library().vlc_rope_pos_workspace_bytes(L - 1, d), dtype=torch.uint8, device=dev)
        # every other rank's rotated k/v halves, as the ring would deliver them
        peers = {}
        for s2 in range(cp):
            _, p2, _, _, k2, v2, _ = locs[s2]
            peers[s2] = (vlc.rope_pos(k2, p2, L - 1), v2)
        blocks = []
        for qh in (0, 1):
            for step in range(cp):
                src = (r - step) % cp
                for kh in (0, 1):
                    mode = vlc.cp_block_mode(cp, r, qh, src, kh)
                    if mode != vlc.binding.CP_BLOCK_NONE:
                        blocks.append((qh, src, kh, mode))
        outs = {qh: [] for qh in (0, 1)}
        wsb = vlc.new_workspace(1, m, H, d, m, False, dev, total_kv=m, max_seqlen_kv=m)
        for qh, src, kh, mode in blocks:
            outs[qh].append((torch.empty((half, H, d), dtype=torch.bfloat16, device=dev),
                             torch.empty((H, half), dtype=torch.float32, device=dev)))
        om = [torch.empty((half, H, d), dtype=torch.bfloat16, device=dev) for _ in (0, 1)]
        lm = [torch.empty((H, half), dtype=torch.float32, device=dev) for _ in (0, 1)]

        def rank_fwd():
            vlc.rope_pos(ql, pos_d, L - 1, out=qrl, workspace=wsr, check=False)
            vlc.rope_pos(kl, pos_d, L - 1, out=krl, workspace=wsr, check=False)
            cnt = {0: 0, 1: 0}
            for qh, src, kh, mode in blocks:
                o_p, l_p = outs[qh][cnt[qh]]
                cnt[qh] += 1
                kk, vv = peers[src]
                vlc.varlen_attn_fwd(qrl[qh * half:(qh + 1) * half], kk[kh * half:(kh + 1) * half],
                                    vv[kh * half:(kh + 1) * half], cuc, m, out=o_p, lse=l_p, workspace=wsb,
                                    check=False, cu_seqlens_kv=cuc, max_seqlen_kv=m, qk_rotated=True,
                                    keys_all_visible=mode == vlc.binding.CP_BLOCK_ALL)
            for qh in (0, 1):
                vlc.lse_merge([a for a, _ in outs[qh]], [b for _, b in outs[qh]], out=om[qh], lse=lm[qh])

        ms, _ = _time_events(rank_fwd, reps)
        st, bits = vlc.get_error(wsb)
        if st != 0:
            raise RuntimeError(f"context-parallel block: device error status {st} bits 0x{bits:x}")
        rank_ms.append(ms)
        # backward: block gradients into preallocated parts, then the sums and R(pos)^T
        wsbb = vlc.new_workspace(1, m, H, d, m, True, dev, total_kv=m, max_seqlen_kv=m)
        nb = len(blocks)
        gparts = [tuple(torch.empty((half, H, d), dtype=torch.bfloat16, device=dev) for _ in range(3))
                  for _ in range(nb)]
        recv = {kh: [torch.zeros((half, H, d), dtype=torch.bfloat16, device=dev) for _ in range(into[(r, kh)])]
                for kh in (0, 1)}
        dq_h = [torch.empty((half, H, d), dtype=torch.bfloat16, device=dev) for _ in (0, 1)]
        dk_h = [torch.empty((half, H, d), dtype=torch.bfloat16, device=dev) for _ in (0, 1)]
        dv_h = [torch.empty((half, H, d), dtype=torch.bfloat16, device=dev) for _ in (0, 1)]
        gsum = torch.empty((half, H, d), dtype=torch.bfloat16, device=dev)

        def rank_bwd():
            for i, (qh, src, kh, mode) in enumerate(blocks):
                kk, vv = peers[src]
                gq, gk, gv = gparts[i]
                vlc.varlen_attn_bwd(gl[qh * half:(qh + 1) * half], qrl[qh * half:(qh + 1) * half],
                                    kk[kh * half:(kh + 1) * half], vv[kh * half:(kh + 1) * half], om[qh], lm[qh],
                                    cuc, m, rope_theta=0.0, dq=gq, dk=gk, dv=gv, workspace=wsbb, check=False,
                                    cu_seqlens_kv=cuc, max_seqlen_kv=m,
                                    keys_all_visible=mode == vlc.binding.CP_BLOCK_ALL)
            for qh in (0, 1):
                vlc.sum_parts([gparts[i][0] for i, b in enumerate(blocks) if b[0] == qh], out=gsum)
                vlc.rope_pos(gsum, pos_d[qh * half:(qh + 1) * half], L - 1, out=dq_h[qh], workspace=wsr,
                             check=False, transpose=True)
            for kh in (0, 1):
                vlc.sum_parts(recv[kh], out=gsum)
                vlc.rope_pos(gsum, pos_d[kh * half:(kh + 1) * half], L - 1, out=dk_h[kh], workspace=wsr,
                             check=False, transpose=True)
                vlc.sum_parts(recv[kh], out=dv_h[kh])

        rank_fwd()
        bms, _ = _time_events(rank_bwd, reps)
        st, bits = vlc.get_error(wsbb)
        if st != 0:
            raise RuntimeError(f"context-parallel block backward: device error status {st} bits 0x{bits:x}")
        rank_bwd_ms.append(bms)
        del peers, outs, om, lm, qrl, krl, wsb, wsbb, gparts, recv, dq_h, dk_h, dv_h, gsum
    mean = sum(rank_ms) / cp
    bmean = sum(rank_bwd_ms) / cp
    fl = 4.0 * d * H * L * (L + 1) / 2
    return {"document_tokens": L, "cp": cp, "H": H, "head_dim": d, "whole_forward_ms": full_ms,
            "whole_forward_eff_TFLOP/s": fl / (full_ms * 1e-3) / 1e12, "rank_forward_ms": rank_ms,
            "balance_max_over_mean": max(rank_ms) / mean, "split_overhead": cp * mean / full_ms,
            "whole_backward_ms": full_bwd_ms, "whole_backward_eff_TFLOP/s": 2.5 * fl / (full_bwd_ms * 1e-3) / 1e12,
            "rank_backward_ms": rank_bwd_ms, "backward_balance_max_over_mean": max(rank_bwd_ms) / bmean,
            "backward_split_overhead": cp * bmean / full_bwd_ms,
            "note": "ranks run one after another on one GPU; communication not included; the dk / dv sums of a "
                    "rank's key halves take stand-in parts of the ring's count"}


EXTRAS = ("positions", "ce", "variants", "packer", "padded", "forward_configs", "step_form", "cp")


def extra_measurements(vlc, w, dev, peaks, q, k, v, step, which=EXTRAS):
    """Positions/labels bandwidth on large packs with the workload's length mix, and (long-context
    workload) the padded comparator: every document padded to the buffer length costs one full
    causal run of that length, and the whole pack run as one causal segment ignores the boundaries."""
    out = {}
    sweep = {}
    lens = np.diff(w.cu).astype(np.int64)
    for logT in ((24, 26) if "positions" in which else ()):
        T = 1 << logT
        reps = -(-T // int(lens.sum()))
        L = np.tile(lens, reps)
        cut = np.searchsorted(np.cumsum(L), T)
        L = L[:cut + 1].copy()
        L[-1] -= int(L.sum()) - T
        L = L[L > 0]
        cu = torch.from_numpy(np.concatenate([[0], np.cumsum(L)]).astype(np.int32)).to(dev)
        tok = torch.randint(0, 32000, (T,), dtype=torch.int64, device=dev)
        pos = torch.empty(T, dtype=torch.int32, device=dev)
        lab = torch.empty(T, dtype=torch.int64, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ms = _time_ms(lambda: vlc.build_positions_labels(cu, tok, None, err=err, out=(pos, lab)), 20)
        gbs = 20.0 * T / (ms * 1e-3) / 1e9
        sweep[f"T=2^{logT}"] = {"ms": ms, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]}
        del cu, tok, pos, lab
    if sweep:
        out["positions_labels_sweep"] = sweep
    if "ce" in which:
        out["shifted_cross_entropy"] = ce_measurement(vlc, w, dev, peaks, step)
    if "variants" in which:
        out["varlen_variants"] = variant_measurements(vlc, w, dev, peaks, step)
    if "packer" in which:
        out["host_packer"] = packer_measurement(vlc)
    if w.name == "long" and "padded" in which:
        out["padded_comparator"] = padded_comparator(vlc, w, dev, q, k, v, step)
    return out


def ce_measurement(vlc, w, dev, peaks, step):
    """Shifted cross-entropy over this pack's labels with a 32000-token vocabulary (bf16 logits)."""
    V = 32000
    gen = torch.Generator(device=dev).manual_seed(4242)
    logits = (torch.randn((w.total, V), generator=gen, device=dev) * 2.0).to(torch.bfloat16)
    ws_ce = torch.empty(vlc.load_library().vlc_ce_workspace_bytes(w.total, w.nseg), dtype=torch.uint8,
                        device=dev)
    ms_ce = _time_ms(lambda: vlc.shifted_cross_entropy(logits, step.lab, step.cu, workspace=ws_ce,
                                                       check=False), 10)
    rows_read = int((step.lab != -100).sum().item())
    ce_bytes = rows_read * V * 2.0 + w.total * (8 + 4 + 1 + 4 + 1)
    return {"vocab": V, "rows_read": rows_read, "ms": ms_ce, "GB/s": ce_bytes / (ms_ce * 1e-3) / 1e9,
            "frac_hbm": ce_bytes / (ms_ce * 1e-3) / 1e9 / peaks["hbm_gbs"]}


def padded_comparator(vlc, w, dev, q, k, v, step):
    """Every document padded to the buffer length costs one full causal run of that length; the
    whole pack run as one causal segment ignores the boundaries."""
    cu1 = torch.tensor([0, w.total], dtype=torch.int32, device=dev)
    o1 = torch.empty_like(q)
    lse1 = torch.empty((w.H, w.total), dtype=torch.float32, device=dev)
    ws1 = vlc.new_workspace(1, w.total, w.H, w.d, w.total, False, dev)
    ms1 = _time_ms(lambda: vlc.varlen_attn_fwd(q, k, v, cu1, w.total, out=o1, lse=lse1, workspace=ws1,
                                                check=False), 3)
    docs = int((w.seg_ignore == 0).sum())
    ms_packed = _time_ms(lambda: vlc.varlen_attn_fwd(q, k, v, step.cu, w.max_seqlen, out=step.o, lse=step.lse,
                                                      workspace=step.ws_f, check=False), 5)
    res = {
        "docs": docs,
        "causal_run_ms": ms1,
        "padded_forward_ms": ms1 * docs,
        "whole_pack_causal_forward_ms": ms1,
        "packed_forward_ms": ms_packed,
        "speedup_packed_vs_padded": ms1 * docs / ms_packed,
        "causal_run_tflops": 4.0 * w.d * w.H * (w.total * (w.total + 1) / 2) / (ms1 * 1e-3) / 1e12,
    }
    del o1, lse1, ws1
    return res


def packer_measurement(vlc, n: int = 10_000_000, capacity: int = 4096, ranks: int = 8):
    """Host packer on n samples of the SFT length mix (lognormal median 300, sigma 1.0, clipped to
    [16, capacity - 1], one reserved token each): first-fit decreasing into windows, then the
    windows to ranks by sum of squared lengths.  Host code, one thread: samples/s, not a roofline."""
    rng = np.random.default_rng(77)
    L = np.clip(np.round(rng.lognormal(np.log(300), 1.0, size=n)), 16, capacity - 1).astype(np.int32)
    t0 = time.perf_counter()
    p = vlc.pack(L, capacity, extra=1)
    t1 = time.perf_counter()
    _, load = vlc.shard_packs(L, p, ranks)
    t2 = time.perf_counter()
    nf = vlc.pack(L, capacity, extra=1, mode="next_fit")
    return {"samples": n, "capacity": capacity, "pack_ms": (t1 - t0) * 1e3,
            "samples_per_s": n / (t1 - t0), "windows": p.nbins, "eta": p.eta,
            "eta_next_fit": nf.eta, "shard_ms": (t2 - t1) * 1e3, "ranks": ranks,
            "sumsq_load_max_over_min": float(load.max() / load.min())}


def variant_measurements(vlc, w, dev, peaks, step):
    """Forward and backward of the varlen variants on this workload's pack (4 d H pairs forward,
    10 d H pairs backward over the legal (query, key) pairs of the real segments): the
    interleaved RoPE pairing, grouped key/value heads (H / 4 of them), a padded layout with every
    segment's slot rounded up to a multiple of 64 rows (same pairs), and bottom-right aligned
    queries that are the last quarter of each segment against all its keys (chunked prefill)."""
    pairs = synth.causal_pairs(w.real_lengths)
    mx = w.max_seqlen

    def run(name, q, k, v, g, cu, n_pairs=pairs, max_q=mx, **kw):
        f_fl, b_fl = 4.0 * w.d * w.H * n_pairs, 10.0 * w.d * w.H * n_pairs
        o = torch.empty_like(q)
        lse = torch.empty((w.H, q.shape[0]), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        kvw = {}
        if "cu_seqlens_kv" in kw:
            kvw = {"total_kv": k.shape[0], "max_seqlen_kv": kw["max_seqlen_kv"]}
        wsf = vlc.new_workspace(w.nseg, q.shape[0], w.H, w.d, max_q, False, dev, k.shape[1], **kvw)
        wsb = vlc.new_workspace(w.nseg, q.shape[0], w.H, w.d, max_q, True, dev, k.shape[1], **kvw)
        fwd = lambda: vlc.varlen_attn_fwd(q, k, v, cu, max_q, out=o, lse=lse, workspace=wsf, check=False, **kw)
        fwd()
        vlc.get_error(wsf)
        bwd = lambda: vlc.varlen_attn_bwd(g, q, k, v, o, lse, cu, max_q, dq=dq, dk=dk, dv=dv, workspace=wsb,
                                          check=False, **kw)
        ms_f, ms_b = _time_ms(fwd, 5), _time_ms(bwd, 5)
        for ws in (wsf, wsb):
            st, bits = vlc.get_error(ws)
            if st != 0:
                raise RuntimeError(f"{name}: device error status {st} bits 0x{bits:x}")
        return {"fwd_ms": ms_f, "bwd_ms": ms_b, "fwd_eff_TFLOP/s": f_fl / (ms_f * 1e-3) / 1e12,
                "bwd_eff_TFLOP/s": b_fl / (ms_b * 1e-3) / 1e12}

    res = {"interleaved_rope": run("interleaved", step.q, step.k, step.v, step.g, step.cu, rope_interleaved=True)}
    hk = max(1, w.H // 4)
    k4, v4 = step.k[:, :hk].contiguous(), step.v[:, :hk].contiguous()
    res[f"gqa_{w.H}q_{hk}kv"] = run("gqa", step.q, k4, v4, step.g, step.cu)
    del k4, v4
    lens = np.diff(w.cu).astype(np.int64)
    slots = lens + (-lens) % 64
    cp = np.concatenate([[0], np.cumsum(slots)])
    idx = torch.from_numpy(np.concatenate([np.arange(a, a + n) for a, n in zip(cp[:-1], lens)])).to(dev)
    padded = []
    for x in (step.q, step.k, step.v, step.g):
        y = torch.zeros((int(cp[-1]),) + tuple(x.shape[1:]), dtype=x.dtype, device=dev)
        y[idx] = x
        padded.append(y)
    cpt = torch.from_numpy(cp.astype(np.int32)).to(dev)
    r = run("padded", *padded, step.cu, cu_seqlens_padded=cpt)
    r["padding_rows"] = int(cp[-1] - w.total)
    res["padded_slots_x64"] = r
    del padded
    # chunked prefill: the last quarter of each real segment's tokens as queries
    real = w.seg_ignore == 0
    lq = np.maximum(1, lens // 4)
    qidx = torch.from_numpy(np.concatenate([np.arange(b - n, b) for b, n in zip(w.cu[1:], lq)])).to(dev)
    off = (lens - lq)[real]
    lqr = lq[real]
    qk_pairs = int(np.sum(lqr * (off + 1) + lqr * (lqr - 1) // 2))
    cuq = torch.from_numpy(np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)).to(dev)
    qq, gq = step.q[qidx].contiguous(), step.g[qidx].contiguous()
    r = run("qkv", qq, step.k, step.v, gq, cuq, n_pairs=qk_pairs, max_q=int(lq.max()),
            cu_seqlens_kv=step.cu, max_seqlen_kv=mx)
    r["query_rows"] = int(lq.sum())
    res["qkv_last_quarter"] = r
    del qq, gq
    return res


def e2e_measure(vlc, w, step, steps, world, dev, readback="result"):
    """Same metric through the public API with pinned host buffers: every step copies this
    step's inputs host->device and reads its result back device->host.  The result is the
    step's per-row log-normalisers (LSE, [H, total] fp32), the attention step's loss-like
    statistic; the gradients stay on the device, as they do in training, where the next
    layer's backward consumes them (readback="all" also reads O, dq, dk, dv, positions and
    labels back).  Steps are pipelined over three streams (copy-in, compute, copy-out) with
    two device buffer sets, so step k's result travels back while step k+1 computes and step
    k+2's inputs arrive."""
    sets = [step, Step(vlc, w, *(torch.empty_like(t) if t is not None else None
                                 for t in (step.q, step.k, step.v, step.g, step.tokens, step.cu, step.ign)),
                       fwd_only=step.fwd_only, rope=step.rope)]
    host_in = [t.cpu().pin_memory() for t in (step.q, step.k, step.v, step.g, step.tokens, step.cu, step.ign)
               if t is not None]

    def dev_in(s):
        return [t for t in (s.q, s.k, s.v, s.g, s.tokens, s.cu, s.ign) if t is not None]

    def dev_out(s):
        if readback == "result":
            return [s.lse]
        return [t for t in (s.o, s.lse, s.dq, s.dk, s.dv) if t is not None]

    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out(step)]
    host_pos = torch.empty(w.total, dtype=torch.int32).pin_memory()
    host_lab = torch.empty(w.total, dtype=torch.int64).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out) + (w.total * 12 if readback == "all" else 0)
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done = [torch.cuda.Event() for _ in sets]
    cmp_done = [torch.cuda.Event() for _ in sets]
    out_done = [torch.cuda.Event() for _ in sets]

    def one(k):
        s = sets[k % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(cmp_done[k % 2])          # the previous user of this set is done computing
            for d, h in zip(dev_in(s), host_in):
                d.copy_(h, non_blocking=True)
            in_done[k % 2].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(in_done[k % 2])
            s_cmp.wait_event(out_done[k % 2])         # its outputs of two steps ago were read back
            s()
            cmp_done[k % 2].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(cmp_done[k % 2])
            for h, d in zip(host_out, dev_out(s)):
                h.copy_(d, non_blocking=True)
            if readback == "all":
                host_pos.copy_(s.pos, non_blocking=True)
                host_lab.copy_(s.lab, non_blocking=True)
            s.pos.record_stream(s_out)                # allocated per call on the compute stream
            s.lab.record_stream(s_out)
            out_done[k % 2].record(s_out)

    for k in range(2):
        one(k)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(steps):
        one(k)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    dt = max_over_ranks(dt, world, dev)
    for s in sets:
        s.check_errors()
    flops = sum_over_ranks(synth.fwd_flops(w) + (0.0 if step.fwd_only else synth.bwd_flops(w)), world, dev)
    return {"value": flops / dt / 1e12, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": dt * 1e3,
            "pipelining": "copy-in, compute and copy-out streams, two device buffer sets",
            "readback": ("the step's LSE (per-row log-normalisers); gradients stay on the device"
                         if readback == "result" else "every output: O, LSE, dq, dk, dv, positions, labels")}


def cpu_baseline(w, q, k, v, g, seconds):
    """The oracle on the host cores, on the same fixed sample the reference arm times: the
    sample is run until ``seconds`` have passed (at least twice); the median run gives the
    rate."""
    import oracle

    oracle.build()
    qc, kc, vc, gc = (oracle.bf16_bits(t) for t in (q, k, v, g))
    pairs, npairs = oracle_sample(w, oracle.num_threads())
    tokens_np = synth.make_tokens(w)
    runs = []
    t_start = time.perf_counter()
    while len(runs) < 2 or (time.perf_counter() - t_start < seconds and len(runs) < 10):
        t0 = time.perf_counter()
        run_oracle_step(w, qc, kc, vc, gc, tokens_np, pairs)
        runs.append(time.perf_counter() - t0)
    dt = statistics.median(runs)
    return {"value": 14.0 * w.d * npairs / dt / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": _sample_text(w, pairs, npairs) + f"; median of {len(runs)} runs of {dt:.1f} s"}


def _source_digest() -> str:
    """sha256 over the kernel sources and the C header (names and bytes)."""
    import glob
    import hashlib

    files = sorted(glob.glob(os.path.join(ROOT, "variable_length_causal_gb300", "csrc", "*")))
    files.append(os.path.join(ROOT, "include", "vlc.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic_from_profiles(kernel: str, workload: str):
    """DRAM bytes per call from the committed ncu capture (profiles/traffic.json), or None when
    that capture was taken on other kernel sources or another workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            doc = json.load(f)
        if doc.get("source_sha256") != _source_digest():
            return None
        return doc["workloads"][workload][kernel]
    except Exception:
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="vlc", choices=["vlc", "reference"])
    ap.add_argument("--workload", default="pt_bwd", choices=synth.WORKLOAD_NAMES)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--rope", choices=("once", "fused"), default="fused",
                    help="fused: RoPE in the forward kernel (k rotated by its k pass, the q tiles inside the "
                         "kernel), which returns q', k' for the backward; once: the step rotates q, k by one "
                         "pass and both directions run on q', k'")
    ap.add_argument("--fwd-only", action="store_true",
                    help="step = positions/labels + forward only (for profiling the forward kernel)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--e2e-readback", choices=("result", "all"), default="result",
                    help="end-to-end leg: read back the step's LSE only (result) or every output (all)")
    ap.add_argument("--extras", default="all",
                    help="comma-separated subset of " + ",".join(EXTRAS) + " (default: all)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the positions/labels sweep and the padded comparator")
    ap.add_argument("--bins", type=int, default=None,
                    help="number of 4096-token windows (default: the workload's own); for small profiling runs")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "vlc" else args.warmup
    world, rank, local = dist_setup()
    w = synth.workload(WORKLOAD_BY_NAME[args.workload], bins=args.bins)
    if args.impl == "reference":
        reference_arm(args, w, world, rank)
    else:
        gpu_arm(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
