"""Benchmark of the KDA operator on one node (one process per GPU).

Default workload (the headline): chunkwise prefill, B=1, H=96, T=8192,
d_k=d_v=128, bf16 q/k/v, fp32 log_alpha/beta, fp32 state, S0 = 0 -- metric
tokens/s.  The same JSON line carries a ``decode`` object: one decode step for
64 sessions x 96 heads (fp32 state [64, 96, 128, 128], 403 MB, in place) --
metric state-GB/s = 2 * state bytes / step time -- and a ``draft`` object:
speculative decode on the same state, verify 8 draft tokens then commit them
(kda_verify_tokens + kda_commit_tokens), metric draft tokens/s -- and a
``segment_parallel`` object: the long prefill of 12 heads (B=1, T=131072) with
kda_fwd_cp against the plain kda_fwd -- and ``epilogue``, ``long`` and
``varlen`` objects: the layer's output epilogue fused against a separate pass,
the long prefill with carry-in (T=131072) and the varlen batch (16 packed
sequences, then 256 decode steps on the returned states).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload prefill|decode|long|long_tp8|varlen]

A step is one kda_fwd over the whole workload (the set-up kernel plus the
prefill kernel).  Inputs are generated on the device before timing and are
larger than L2, so no L2 flush is needed between steps.  Timing: CUDA events
on the launching stream, barrier + synchronize on both sides, max over ranks.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_attention_recurrence_chunkwise_gb300 import inputs as I  # noqa: E402

METRIC = "KDA prefill tokens/s and decode state GB/s (H=96,d=128) vs roofline"
_CSRC = "linear_attention_recurrence_chunkwise_gb300/csrc/"
KERNEL_SOURCES = {  # every source file a kernel is compiled from
    "prefill_tc": (_CSRC + "kda_prefill_tc.cu", _CSRC + "kda_solve.cuh", _CSRC + "kda_sm100.cuh",
                   _CSRC + "kda_serial.cuh"),
    "prefill_tc64": (_CSRC + "kda_prefill_tc64.cu", _CSRC + "kda_sm100.cuh"),
    "prefill_simt": (_CSRC + "kda_prefill_simt.cu", _CSRC + "kda_serial.cuh"),
    "decode": (_CSRC + "kda_decode.cu",),
    "multitoken": (_CSRC + "kda_multitoken.cu",),
}


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def source_hash(rels):
    h = hashlib.sha256()
    for rel in rels:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel_key, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(kernel_key, {}).get(workload)
    if not rec or rec.get("source_sha256_16") != source_hash(KERNEL_SOURCES[kernel_key]):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background (200 ms period)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.tmp is None:
            return None
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(",") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup(n_gpus):
    """One process per GPU under torchrun (RANK / LOCAL_RANK / WORLD_SIZE from the
    environment): NCCL on GPUs; gloo where no GPU is present (the host-side
    multi-rank path, exercised by the CPU tests)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The largest x over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def nbytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts if t is not None)


# ------------------------------------------------------------------ workloads

def make_workload(name, seed, device):
    w = _make_workload(name, seed, device)
    if torch.cuda.is_available():
        torch.cuda.synchronize()  # generated on the current stream; timed on another
    return w


def _make_workload(name, seed, device):
    if name == "decode":
        p = I.PRESETS["decode"]
        S = I.decode_state(p["N"], p["H"], p["d"], p["d"], p["s0_std"], seed, device)
        steps = [I.decode_token(p["N"], p["H"], p["d"], p["d"], p["dtype"], p["la"], seed, s,
                                device) for s in range(8)]
        return dict(kind="decode", S=S, tokens=steps, N=p["N"], H=p["H"], d=p["d"],
                    label=f"decode step N={p['N']} H={p['H']} d={p['d']} {p['dtype']} "
                          f"fp32 state (in place)")
    prob = I.preset_problem(name, seed=seed, device=device)
    Ttot = prob.q.shape[0] * prob.q.shape[1] if prob.q.dim() == 4 else prob.q.shape[0]
    H, d = prob.q.shape[-2], prob.q.shape[-1]
    lab = {"prefill": "prefill B=1 H=96 T=8192 d=128 bf16, S0=0",
           "long": "long prefill B=1 H=96 T=131072 d=128 bf16, S0~N(0,0.02)",
           "long_tp8": "long prefill B=1 H=12 T=131072 d=128 bf16, S0~N(0,0.02) "
                       "(12 of K3's 96 heads: 8-way tensor parallel)",
           "varlen": f"varlen prefill 16 seqs (sum T={Ttot}) H=96 d=128 bf16",
           "tiny": "tiny prefill B=1 H=2 T=256 d=64 fp32"}[name]
    return dict(kind="prefill", prob=prob, Ttot=Ttot, H=H, d=d, label=lab)


def line_config(w, world):
    """The `config` object of the JSON line (identical for both arms)."""
    c = {"workload": w["label"], "l2": "inputs larger than L2, no flush",
         "parallelism": f"replicas x{world} (independent problems per rank)"}
    if w["kind"] == "prefill":
        c.update(tokens_per_step=w["Ttot"], heads=w["H"], d=w["d"])
    else:
        c.update(sessions=w["N"], heads=w["H"], d=w["d"])
    return c


def time_calls(fn, reps, stream, warm=2, warm_s=0.3):
    """Mean device time of one call of fn (CUDA events on `stream`), after at
    least `warm` calls and `warm_s` seconds of untimed calls (the clocks ramp
    up from idle after the CPU-only phases of the run)."""
    torch.cuda.synchronize()  # inputs made on another stream are complete
    t_end = time.time() + warm_s
    with torch.cuda.stream(stream):
        while warm > 0:
            for _ in range(warm):
                fn()
            stream.synchronize()
            if time.time() >= t_end:
                break
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
    stream.synchronize()
    return a.elapsed_time(b) / reps


def hbm_roof(alg, ms, pk, **extra):
    gbs = alg / (ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
            "frac": round(gbs / pk["hbm"], 4), "algorithmic_bytes_per_launch": alg, **extra}


def prefill_alg_bytes(w):
    p = w["prob"]
    return nbytes(p.q, p.k, p.v, p.log_alpha, p.beta, p.S0, p.cu_seqlens) + \
        nbytes(p.v) + p.n_seq * w["H"] * w["d"] * w["d"] * 4  # o and S_T


def prefill_flops(w):
    """Chunk-kernel FLOPs per head 6 T d^2 + 3 T C d + T C^2 (C = 64), as the
    pages give them ("Kimi Delta Attention 完全拆解", prefill complexity)."""
    T, d, C = w["Ttot"], w["d"], 64
    return w["H"] * (6 * T * d * d + 3 * T * C * d + T * C * C)


def decode_alg_bytes(w):
    S = w["S"]
    x = w["tokens"][0]
    return 2 * nbytes(S) + nbytes(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"]) + \
        nbytes(x["v"])


# ------------------------------------------------------------------ our arm

def resolve_segments(kda, w, segments):
    """None for the plain kda_fwd; else the segment count of kda_fwd_cp ('auto':
    the library's suggestion for this workload)."""
    if segments is None:
        return None
    if segments == "auto":
        return kda.kda_fwd_cp_segments(w["prob"].n_seq, w["H"], w["Ttot"])
    return int(segments)


def time_prefill(kda, w, steps, warmup, stream, segments=None):
    p = w["prob"]
    o = torch.empty_like(p.v)
    ST = torch.empty((p.n_seq, w["H"], w["d"], w["d"]), dtype=torch.float32, device="cuda")
    nbytes_ws = kda.kda_fwd_workspace_bytes(p.n_seq) if segments is None else \
        kda.kda_fwd_cp_workspace_bytes(p.n_seq, w["H"], w["d"], w["d"], segments)
    ws = torch.empty(nbytes_ws, dtype=torch.uint8, device="cuda")

    def call():
        if segments is None:
            kda.kda_fwd(p.q, p.k, p.v, p.log_alpha, p.beta, p.S0, p.cu_seqlens, o=o, S_T=ST,
                        workspace=ws, stream=stream)
        else:
            kda.kda_fwd_cp(p.q, p.k, p.v, p.log_alpha, p.beta, p.S0, p.cu_seqlens,
                           segments=segments, o=o, S_T=ST, workspace=ws, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    return call, ev, (o, ST, ws)


def run_ours(args, world, rank):
    from linear_attention_recurrence_chunkwise_gb300 import build as kbuild
    kbuild.build()
    from linear_attention_recurrence_chunkwise_gb300 import kda
    kda.load()
    pk = peaks()
    stream = torch.cuda.Stream()
    w = make_workload(args.workload, seed=args.seed + rank, device="cuda")
    torch.cuda.synchronize()

    if w["kind"] == "prefill":
        segments = resolve_segments(kda, w, args.segments)
        call, ev, bufs = time_prefill(kda, w, args.steps, args.warmup, stream, segments)
        # plain: set-up + prefill kernel; segment-parallel: plan, pass A, scan, pass D
        launches_per_step = 2 if segments is None or segments == 1 else 4
    else:
        S = w["S"]
        toks = w["tokens"]
        o = torch.empty_like(toks[0]["v"])
        ctr = [0]

        def call():
            x = toks[ctr[0] % len(toks)]
            ctr[0] += 1
            kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S, o=o,
                                stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                call()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        launches_per_step = 1

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        time.sleep(0.1)  # the sampler's first reading
        with torch.cuda.stream(stream):
            # untimed steps for at least 0.3 s right before the timed ones: the
            # clocks have ramped up from idle when the first timed step starts,
            # and the sampler reads them under this load
            t_end = time.time() + 0.3
            while True:
                for _ in range(max(args.warmup, 1)):
                    call()
                stream.synchronize()
                if time.time() >= t_end:
                    break
            start.record(stream)
            for i in range(args.steps):
                ev[i][0].record(stream)
                call()
                ev[i][1].record(stream)
            stop.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
    barrier(world)
    total_ms = start.elapsed_time(stop)
    per_call = [a.elapsed_time(b) for a, b in ev]  # events around each call's launches
    per_launch_ms = statistics.mean(per_call)
    total_ms = max_over_ranks(total_ms, world)
    ms_step = total_ms / args.steps

    if w["kind"] == "prefill":
        units = w["Ttot"]
        value = units * world / (ms_step / 1e3)
        unit = "tokens/s"
        alg = prefill_alg_bytes(w)
        flops = prefill_flops(w)
        # the engine kda_fwd's AUTO choice runs: tensor cores for bf16 at d = 128
        # and for any dtype at d = 64, CUDA cores otherwise
        bf16 = w["prob"].q.dtype == torch.bfloat16
        kernel_key = "prefill_tc" if (bf16 and w["d"] == 128) else \
            "prefill_tc64" if w["d"] == 64 else "prefill_simt"
    else:
        value = 2 * nbytes(w["S"]) * world / (ms_step / 1e3) / 1e9
        unit = "GB/s"
        alg = decode_alg_bytes(w)
        flops = None
        kernel_key = "decode"
    achieved_gbs = alg / (per_launch_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": pk["hbm"],
                "unit": "GB/s", "frac": round(achieved_gbs / pk["hbm"], 4),
                "traffic": traffic_for(kernel_key, args.workload),
                "peak_source": f"{pk['source']} (MEASURED_PEAKS.json hbm_gbs)"
                if pk["source"] == "measured" else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": alg, "kernel": kernel_key,
                "avg_launch_ms": round(per_launch_ms, 4),
                "launch_timing": "CUDA events around each call on its stream: the dominant "
                                 "kernel plus, for a prefill, its 2-3 us set-up kernel"}
    if flops is not None:
        tf = flops / (per_launch_ms / 1e3) / 1e12
        roofline["tensor"] = {"achieved_tflops": round(tf, 2), "peak_tflops": pk["bf16"],
                              "frac": round(tf / pk["bf16"], 4),
                              "flops_per_launch": flops,
                              "flop_count": "6Td^2+3TCd+TC^2 per head (pages' formula)"}

    line = {"metric": METRIC, "value": round(value, 1), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "ms_per_step_p50": round(statistics.median(per_call), 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if args.workload != "tiny" else "f32",
            "data": "synthetic (seeded, device-generated)",
            "config": line_config(w, world),
            "roofline": roofline, "clocks": clk.summary(),
            "gpu_launches": launches_per_step * args.steps}
    if w["kind"] == "prefill":
        if segments is not None:
            line["config"]["segments"] = segments
            line["config"]["call"] = "kda_fwd_cp (segment-parallel)"
        e2e_steps = max(2, min(args.steps, 5))
        if segments is None and w["prob"].cu_seqlens is None and w["prob"].n_seq == 1:
            line["e2e"] = e2e_prefill_pipelined(kda, w, e2e_steps, stream, world)
        else:
            line["e2e"] = e2e_prefill(kda, w, e2e_steps, stream, world, segments)
        if args.workload == "prefill" and not args.no_decode:
            cpu = rank == 0 and world == 1 and not args.no_cpu
            line["decode"] = decode_sub(kda, args, stream, pk, cpu)
            line["draft"] = draft_sub(kda, args, stream, pk, line["decode"]["us_per_step"])
            line["segment_parallel"] = cp_sub(kda, args, stream, pk)
            line["epilogue"] = epilogue_sub(kda, args, stream, pk)
            line["prologue"] = prologue_sub(kda, args, stream, pk)
            line["wide_gates"] = wide_gates_sub(kda, args, stream, pk)
            line["long"] = long_sub(kda, args, stream, pk, cpu)
            line["tiny"] = tiny_sub(kda, args, stream, pk, cpu)
            line["varlen"] = varlen_sub(kda, args, stream, pk, cpu)
    else:
        line["e2e"] = e2e_decode(kda, w, max(2, min(args.steps, 20)), stream, world)
        if not args.no_decode:
            line["draft"] = draft_sub(kda, args, stream, pk, ms_step * 1e3)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, args)
    return line


def decode_sub(kda, args, stream, pk, cpu=False):
    w = make_workload("decode", seed=args.seed, device="cuda")
    S, toks = w["S"], w["tokens"]
    o = torch.empty_like(toks[0]["v"])
    steps = 1000  # back to back, in place; an event between steps gives the median

    def run(states):
        with torch.cuda.stream(stream):
            for i in range(5):
                x = toks[i % len(toks)]
                kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                    states[i % len(states)], o=o, stream=stream)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(steps):
                x = toks[i % len(toks)]
                kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                    states[i % len(states)], o=o, stream=stream)
                ev[i + 1].record(stream)
        stream.synchronize()
        ms = ev[0].elapsed_time(ev[-1]) / steps
        p50 = statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))
        return ms, p50
    ms, p50 = run([S])
    # two states taken in turn (806 MB, over six times the L2): no block of the
    # state a step reads can still sit in L2 from the step before
    S2 = I.decode_state(w["N"], w["H"], w["d"], w["d"], I.PRESETS["decode"]["s0_std"],
                        args.seed + 1, "cuda")
    torch.cuda.synchronize()
    ms2, p50_2 = run([S, S2])
    del S2
    alg = decode_alg_bytes(w)
    out = {"metric": "decode state GB/s", "value": round(2 * nbytes(S) / (ms / 1e3) / 1e9, 1),
           "unit": "GB/s", "us_per_step": round(ms * 1e3, 2),
           "us_per_step_p50": round(p50 * 1e3, 2), "steps": steps,
           "workload": w["label"],
           "roofline": hbm_roof(alg, ms, pk, traffic=traffic_for("decode", "decode")),
           "alternating_states": {
               "value": round(2 * nbytes(S) / (ms2 / 1e3) / 1e9, 1), "unit": "GB/s",
               "us_per_step": round(ms2 * 1e3, 2), "us_per_step_p50": round(p50_2 * 1e3, 2),
               "states": 2, "roofline": hbm_roof(alg, ms2, pk),
               "note": "steps alternate between two 403 MB states, so no state block is "
                       "re-read from L2"}}
    if cpu:
        out["cpu_baseline"] = cpu_baseline(w, args, target_s=5.0)
    return out


def draft_sub(kda, args, stream, pk, decode_us):
    """Speculative decode on the decode state: verify K draft tokens (outputs,
    state read once and kept), then commit all K (state read and written once;
    every session accepting everything is the commit's slowest case)."""
    p = I.PRESETS["draft"]
    N, K, H, d = p["N"], p["K"], p["H"], p["d"]
    S = I.decode_state(N, H, d, d, p["s0_std"], args.seed, "cuda")
    x = I.draft_tokens(N, K, H, d, d, p["dtype"], p["la"], args.seed + 1, "cuda")
    torch.cuda.synchronize()
    ins = (x["q"], x["k"], x["v"], x["log_alpha"], x["beta"])
    o = torch.empty_like(x["v"])
    acc = torch.full((N,), K, dtype=torch.int32, device="cuda")
    reps = 30
    with torch.cuda.stream(stream):
        for _ in range(3):
            kda.kda_verify_tokens(*ins, S, o=o, stream=stream)
            kda.kda_commit_tokens(*ins, S, n_accept=acc, stream=stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    with torch.cuda.stream(stream):
        for e in ev:
            e[0].record(stream)
            kda.kda_verify_tokens(*ins, S, o=o, stream=stream)
            e[1].record(stream)
            kda.kda_commit_tokens(*ins, S, n_accept=acc, stream=stream)
            e[2].record(stream)
    stream.synchronize()
    ver_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    com_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    alg_v = nbytes(S, *ins, o)
    alg_c = 2 * nbytes(S) + nbytes(x["k"], x["v"], x["log_alpha"], x["beta"], acc)

    def roof(alg, ms):
        gbs = alg / (ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                "frac": round(gbs / pk["hbm"], 4), "traffic": None,
                "algorithmic_bytes_per_launch": alg, "avg_launch_us": round(ms * 1e3, 2)}
    rv, rc = roof(alg_v, ver_ms), roof(alg_c, com_ms)
    rv["traffic"] = traffic_for("multitoken", "verify")
    rc["traffic"] = traffic_for("multitoken", "commit")
    spec_us = (ver_ms + com_ms) * 1e3
    return {"metric": "draft tokens/s (verify + commit)",
            "value": round(N * K / (spec_us / 1e6), 1), "unit": "tokens/s",
            "workload": f"verify K={K} draft tokens then commit all, N={N} H={H} d={d} "
                        f"{p['dtype']} fp32 state (in place)",
            "us_per_verify_commit": round(spec_us, 2),
            "us_for_K_decode_steps": round(K * decode_us, 2),
            "verify": rv, "commit": rc, "reps": reps}


def cp_sub(kda, args, stream, pk):
    """Segment-parallel forward on the long prefill of the 12 heads one GPU holds
    under 8-way tensor parallelism (B=1, H=12, T=131072): kda_fwd_cp with the
    suggested segment count against the plain kda_fwd (12 blocks, one per head)."""
    w = make_workload("long_tp8", seed=args.seed, device="cuda")
    p = w["prob"]
    N, H, d = p.n_seq, w["H"], w["d"]
    P = kda.kda_fwd_cp_segments(N, H, w["Ttot"])
    o = torch.empty_like(p.v)
    ST = torch.empty((N, H, d, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(kda.kda_fwd_cp_workspace_bytes(N, H, d, d, P), dtype=torch.uint8,
                     device="cuda")
    plain = lambda: kda.kda_fwd(p.q, p.k, p.v, p.log_alpha, p.beta, p.S0, o=o, S_T=ST,
                                workspace=ws, stream=stream)
    cp = lambda: kda.kda_fwd_cp(p.q, p.k, p.v, p.log_alpha, p.beta, p.S0, segments=P, o=o,
                                S_T=ST, workspace=ws, stream=stream)
    out = {}
    for name, fn in (("plain", plain), ("cp", cp)):
        with torch.cuda.stream(stream):
            for _ in range(2):
                fn()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(3):
                fn()
            b.record(stream)
        stream.synchronize()
        out[name] = a.elapsed_time(b) / 3
    alg = prefill_alg_bytes(w)
    gbs = alg / (out["cp"] / 1e3) / 1e9
    return {"metric": "tokens/s", "value": round(w["Ttot"] / (out["cp"] / 1e3), 1),
            "unit": "tokens/s", "workload": w["label"], "segments": P,
            "ms_segment_parallel": round(out["cp"], 3), "ms_plain": round(out["plain"], 3),
            "speedup": round(out["plain"] / out["cp"], 2),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"],
                         "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4),
                         "algorithmic_bytes_per_call": alg,
                         "note": "the operator's bytes over the whole call (three kernels "
                                 "of passes A and D plus the scan)"}}


def prefill_roofline(w, ms, pk):
    r = hbm_roof(prefill_alg_bytes(w), ms, pk)
    tf = prefill_flops(w) / (ms / 1e3) / 1e12
    r["tensor"] = {"achieved_tflops": round(tf, 2), "peak_tflops": pk["bf16"],
                   "frac": round(tf / pk["bf16"], 4), "flops_per_launch": prefill_flops(w),
                   "flop_count": "6Td^2+3TCd+TC^2 per head (pages' formula)"}
    return r


def epilogue_sub(kda, args, stream, pk):
    """The layer's output epilogue (head-wise RMSNorm times a sigmoid gate) on
    the prefill and decode workloads, fused into the kernel against a separate
    pass, same box: the A/B behind KDA_EPILOGUE_AUTO's choice."""
    out = {"metric": "us per call", "unit": "us"}
    w = make_workload("prefill", seed=args.seed, device="cuda")
    p = w["prob"]
    gen = torch.Generator(device="cuda").manual_seed(args.seed + 7)
    g = (2 * torch.randn(p.v.shape, generator=gen, device="cuda")).to(p.v.dtype)
    nw = torch.rand(w["d"], generator=gen, device="cuda") + 0.5
    y = torch.empty_like(p.v)
    ST = torch.empty((p.n_seq, w["H"], w["d"], w["d"]), dtype=torch.float32, device="cuda")
    ws = torch.empty(kda.kda_fwd_workspace_bytes(p.n_seq), dtype=torch.uint8, device="cuda")
    for mode in ("fused", "separate"):
        ms = time_calls(lambda: kda.kda_fwd_gated(p.q, p.k, p.v, p.log_alpha, p.beta, p.S0,
                                                  g=g, norm_weight=nw, y=y, S_T=ST,
                                                  workspace=ws, epilogue=mode, stream=stream),
                        10, stream)
        out[f"prefill_{mode}_us"] = round(ms * 1e3, 2)
    out["prefill_plain_us"] = round(time_calls(
        lambda: kda.kda_fwd(p.q, p.k, p.v, p.log_alpha, p.beta, p.S0, o=y, S_T=ST, workspace=ws,
                            stream=stream), 10, stream) * 1e3, 2)
    del w, p, g, y, ST
    wd = make_workload("decode", seed=args.seed, device="cuda")
    x = wd["tokens"][0]
    gd = (2 * torch.randn(x["v"].shape, generator=gen, device="cuda")).to(x["v"].dtype)
    yd = torch.empty_like(x["v"])
    for mode in ("fused", "separate"):
        ms = time_calls(lambda: kda.kda_decode_step_gated(
            x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], wd["S"], g=gd, norm_weight=nw,
            y=yd, epilogue=mode, stream=stream), 100, stream)
        out[f"decode_{mode}_us"] = round(ms * 1e3, 2)
    out["decode_plain_us"] = round(time_calls(
        lambda: kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], wd["S"],
                                    o=yd, stream=stream), 100, stream) * 1e3, 2)
    out["workloads"] = "prefill B=1 H=96 T=8192 d=128 bf16; decode step N=64 H=96 d=128"
    out["auto_choice"] = {"prefill": "separate", "decode": "fused"}
    del wd
    torch.cuda.empty_cache()
    return out


def prologue_sub(kda, args, stream, pk):
    """The layer's input prologue (ShortConv(4), Swish, L2Norm of q and k) on
    the prefill shape (B=1, T=8192, H=96, d=128, bf16; a pass of its own that
    reads the three projected streams and writes q, k, v) and one decode token
    for 64 sessions x 96 heads (the conv state moved on in place)."""
    out = {"metric": "GB/s", "unit": "GB/s"}
    T, H, d, N = 8192, 96, 128, 64
    gen = torch.Generator(device="cuda").manual_seed(args.seed + 11)
    xs = [torch.randn((1, T, H, d), generator=gen, device="cuda").to(torch.bfloat16)
          for _ in range(3)]
    ws = [0.5 * torch.randn((H, d, 4), generator=gen, device="cuda") for _ in range(3)]
    c0 = torch.randn((1, 3, 3, H, d), generator=gen, device="cuda")
    ys = [torch.empty_like(xs[0]) for _ in range(3)]
    cT = torch.empty_like(c0)
    wsp = torch.empty(kda.kda_fwd_workspace_bytes(1), dtype=torch.uint8, device="cuda")
    ms = time_calls(lambda: kda.kda_short_conv(*xs, *ws, c0, q=ys[0], k=ys[1], v=ys[2],
                                               conv_T=cT, workspace=wsp, stream=stream),
                    10, stream)
    alg = 3 * 2 * xs[0].numel() * 2 + 3 * H * d * 4 * 4 + 2 * c0.numel() * 4
    out["prefill"] = {"workload": "prologue of B=1 T=8192 H=96 d=128 bf16 (q, k, v streams)",
                      "us_per_call": round(ms * 1e3, 2), "value": round(alg / (ms / 1e3) / 1e9, 1),
                      "roofline": hbm_roof(alg, ms, pk)}
    del xs, ys
    xd = [torch.randn((N, H, d), generator=gen, device="cuda").to(torch.bfloat16)
          for _ in range(3)]
    yd = [torch.empty_like(xd[0]) for _ in range(3)]
    conv = torch.randn((N, 3, 3, H, d), generator=gen, device="cuda")
    ms = time_calls(lambda: kda.kda_short_conv_step(*xd, *ws, conv, q=yd[0], k=yd[1], v=yd[2],
                                                    stream=stream), 100, stream)
    alg = 3 * 2 * xd[0].numel() * 2 + 3 * H * d * 4 * 4 + 2 * conv.numel() * 4
    out["decode_step"] = {"workload": "prologue of one token, N=64 sessions H=96 d=128 bf16, "
                                      "conv state [64,3,3,96,128] fp32 in place",
                          "us_per_call": round(ms * 1e3, 2),
                          "value": round(alg / (ms / 1e3) / 1e9, 1),
                          "roofline": hbm_roof(alg, ms, pk),
                          "note": "the 28 MB conv state fits in L2, so repeated steps may "
                                  "re-read it from L2"}
    # the whole layer step for one token: prologue, recurrence and epilogue in
    # one kernel, against the prologue step followed by the gated decode step
    wd = make_workload("decode", seed=args.seed, device="cuda")
    x = wd["tokens"][0]
    gate = (2 * torch.randn((N, H, d), generator=gen, device="cuda")).to(torch.bfloat16)
    nw = torch.rand(d, generator=gen, device="cuda") + 0.5
    y = torch.empty_like(gate)
    fused = time_calls(lambda: kda.kda_decode_layer_step(
        *xd, *ws, conv, x["log_alpha"], x["beta"], wd["S"], gate, nw, y=y, stream=stream),
        100, stream)

    def separate():
        kda.kda_short_conv_step(*xd, *ws, conv, q=yd[0], k=yd[1], v=yd[2], stream=stream)
        kda.kda_decode_step_gated(yd[0], yd[1], yd[2], x["log_alpha"], x["beta"], wd["S"], g=gate,
                                  norm_weight=nw, y=y, stream=stream)
    sep = time_calls(separate, 100, stream)
    out["layer_step"] = {"workload": "one decode token, N=64 sessions H=96 d=128 bf16: "
                                     "prologue, recurrence on the 403 MB state, epilogue",
                         "fused_us": round(fused * 1e3, 2), "separate_us": round(sep * 1e3, 2)}
    del xd, yd, conv, wd
    torch.cuda.empty_cache()
    return out


def wide_gates_sub(kda, args, stream, pk):
    """K3-strength gates (per-token log-decay in U(-5, -0.5): every 64-token
    chunk leaves the chunk form's range) on the prefill shape, B=1, H=96,
    T=8192: the tensor-core engine with the blocked path against the plain one
    (which recomputes such heads token by token), and the blocked-path
    engine's cost on in-range gates."""
    out = {"metric": "ms per call", "unit": "ms",
           "workload": "prefill B=1 H=96 T=8192 d=128 bf16, log alpha in U(-5, -0.5)"}
    for la, tag in (((-5.0, -0.5), "wide"), ((-0.5, -0.001), "in_range")):
        prob = I.prefill_problem(1, 8192, 96, 128, 128, "bf16", la, None, args.seed, "cuda")
        torch.cuda.synchronize()
        o = torch.empty_like(prob.v)
        ST = torch.empty((1, 96, 128, 128), dtype=torch.float32, device="cuda")
        ws = torch.empty(kda.kda_fwd_workspace_bytes(1), dtype=torch.uint8, device="cuda")
        engines = ("tensorcore_wide", "tensorcore") if tag == "wide" else ("tensorcore_wide",)
        for eng in engines:
            ms = time_calls(lambda: kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha,
                                                prob.beta, None, o=o, S_T=ST, workspace=ws,
                                                engine=eng, stream=stream), 5, stream)
            out[f"{tag}_{eng}_ms"] = round(ms, 4)
        del prob, o, ST
    out["note"] = ("tensorcore: heads with such chunks are recomputed token by token; "
                   "tensorcore_wide: such chunks take the blocked path on the tensor cores")
    torch.cuda.empty_cache()
    return out


def tiny_sub(kda, args, stream, pk, cpu=False):
    """The tiny fp32 recurrence, B=1, H=2, T=256, d=64: the d = 64 tensor-core
    engine that AUTO runs for fp32 at d = 64, the CUDA-core engine beside it,
    and both at the prefill size (B=1, H=96, T=8192, d=64, fp32)."""
    w = make_workload("tiny", seed=args.seed, device="cuda")
    p = w["prob"]
    o = torch.empty_like(p.v)
    ST = torch.empty((p.n_seq, w["H"], w["d"], w["d"]), dtype=torch.float32, device="cuda")
    ws = torch.empty(kda.kda_fwd_workspace_bytes(p.n_seq), dtype=torch.uint8, device="cuda")

    def per_engine(q, k, v, la, beta, o, ST, reps):
        # (the sub-benchmarks before this one have ramped the clocks: a short warm-up)
        return {eng: time_calls(lambda: kda.kda_fwd(q, k, v, la, beta, None, o=o, S_T=ST,
                                                     workspace=ws, engine=eng, stream=stream),
                                reps, stream, warm=3, warm_s=0.0)
                for eng in ("tensorcore", "cudacore")}
    t = per_engine(p.q, p.k, p.v, p.log_alpha, p.beta, o, ST, 200)
    roof = prefill_roofline(w, t["tensorcore"], pk)
    roof["traffic"] = traffic_for("prefill_tc64", "tiny")
    roof["note"] = "latency-bound: 2 CTAs walk their 4 chunks in series"
    out = {"metric": "tokens/s", "value": round(w["Ttot"] / (t["tensorcore"] / 1e3), 1),
           "unit": "tokens/s", "workload": w["label"] + " (tensor-core engine)",
           "ms_per_call": round(t["tensorcore"], 4),
           "cudacore_ms_per_call": round(t["cudacore"], 4), "roofline": roof}
    big = I.prefill_problem(1, 8192, 96, 64, 64, "f32", (-0.5, -0.001), None, args.seed, "cuda")
    ob = torch.empty_like(big.v)
    STb = torch.empty((1, 96, 64, 64), dtype=torch.float32, device="cuda")
    tb = per_engine(big.q, big.k, big.v, big.log_alpha, big.beta, ob, STb, 10)
    wb = dict(kind="prefill", prob=big, Ttot=8192, H=96, d=64, label="")
    out["prefill_size"] = {"workload": "prefill B=1 H=96 T=8192 d=64 fp32, S0=0",
                           "tensorcore_ms": round(tb["tensorcore"], 4),
                           "cudacore_ms": round(tb["cudacore"], 4),
                           "tokens_per_s": round(8192 / (tb["tensorcore"] / 1e3), 1),
                           "roofline": hbm_roof(prefill_alg_bytes(wb), tb["tensorcore"], pk)}
    if cpu:
        out["cpu_baseline"] = cpu_baseline(w, args, target_s=2.0)
    del w, p, o, ST, big, ob, STb
    torch.cuda.empty_cache()
    return out


def long_sub(kda, args, stream, pk, cpu=False):
    """The long prefill with carry-in: B=1, H=96, T=131072, S0 ~ N(0, 0.02),
    long-memory gates (one kda_fwd per call)."""
    w = make_workload("long", seed=args.seed, device="cuda")
    p = w["prob"]
    o = torch.empty_like(p.v)
    ST = torch.empty_like(p.S0)
    ws = torch.empty(kda.kda_fwd_workspace_bytes(p.n_seq), dtype=torch.uint8, device="cuda")
    ms = time_calls(lambda: kda.kda_fwd(p.q, p.k, p.v, p.log_alpha, p.beta, p.S0, o=o, S_T=ST,
                                        workspace=ws, stream=stream), 10, stream)
    out = {"metric": "tokens/s", "value": round(w["Ttot"] / (ms / 1e3), 1), "unit": "tokens/s",
           "workload": w["label"], "ms_per_call": round(ms, 3),
           "roofline": prefill_roofline(w, ms, pk)}
    if cpu:
        out["cpu_baseline"] = cpu_baseline(w, args, target_s=4.0, tokens=16384)
    del w, p, o, ST
    torch.cuda.empty_cache()
    return out


def varlen_sub(kda, args, stream, pk, cpu=False):
    """The varlen batch: 16 packed sequences (lengths log-uniform in [1024,
    65536]), H=96, per-sequence S0; then 256 decode steps on the 16 returned
    states (B=16)."""
    w = make_workload("varlen", seed=args.seed, device="cuda")
    p = w["prob"]
    o = torch.empty_like(p.v)
    ST = torch.empty_like(p.S0)
    ws = torch.empty(kda.kda_fwd_workspace_bytes(p.n_seq), dtype=torch.uint8, device="cuda")
    ms = time_calls(lambda: kda.kda_fwd(p.q, p.k, p.v, p.log_alpha, p.beta, p.S0,
                                        p.cu_seqlens, o=o, S_T=ST, workspace=ws,
                                        stream=stream), 10, stream)
    pv = I.PRESETS["varlen"]
    N, H, d = p.n_seq, w["H"], w["d"]
    toks = [I.decode_token(N, H, d, d, pv["dtype"], pv["la"], args.seed + 1, s, "cuda")
            for s in range(pv["decode_steps"])]
    torch.cuda.synchronize()
    od = torch.empty_like(toks[0]["v"])
    S = ST.clone()
    ctr = [0]

    def dec():
        x = toks[ctr[0] % len(toks)]
        ctr[0] += 1
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S, o=od,
                            stream=stream)
    ctr[0] = 0
    dms = time_calls(dec, pv["decode_steps"], stream, warm=0)  # the 256 steps, once
    x = toks[0]
    dalg = 2 * nbytes(S) + nbytes(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], od)
    out = {"metric": "tokens/s", "value": round(w["Ttot"] / (ms / 1e3), 1), "unit": "tokens/s",
           "workload": w["label"], "ms_per_call": round(ms, 3),
           "sequence_lengths": (p.cu_seqlens[1:] - p.cu_seqlens[:-1]).tolist(),
           "roofline": prefill_roofline(w, ms, pk),
           "decode": {"metric": "decode state GB/s",
                      "value": round(2 * nbytes(S) / (dms / 1e3) / 1e9, 1), "unit": "GB/s",
                      "us_per_step": round(dms * 1e3, 2), "steps": pv["decode_steps"],
                      "workload": f"256 decode steps, N={N} H={H} d={d} {pv['dtype']} on the "
                                  f"returned fp32 states (in place)",
                      "roofline": hbm_roof(dalg, dms, pk, note="the 16 x 96 states (101 MB) "
                                           "fit in L2, so steps may re-read them from L2")}}
    if cpu:
        out["cpu_baseline"] = cpu_baseline(w, args, target_s=4.0, heads=4)
        dw = dict(kind="decode", S=ST, tokens=toks[:1], N=N, H=H, d=d, label="")
        out["decode"]["cpu_baseline"] = cpu_baseline(dw, args, target_s=2.0)
    del w, p, o, ST, S, toks
    torch.cuda.empty_cache()
    return out


def e2e_prefill(kda, w, steps, stream, world, segments=None):
    """Same metric through the public API with pinned host buffers: H2D of the
    step's inputs, kda_fwd (kda_fwd_cp with `segments`), D2H of o and S_T, all
    inside the timed region."""
    p = w["prob"]
    host = {n: getattr(p, n).to("cpu").pin_memory()
            for n in ("q", "k", "v", "log_alpha", "beta")}
    host_S0 = None if p.S0 is None else p.S0.to("cpu").pin_memory()
    host_cu = None if p.cu_seqlens is None else p.cu_seqlens.to("cpu").pin_memory()
    o_h = torch.empty(p.v.shape, dtype=p.v.dtype).pin_memory()
    ST_h = torch.empty((p.n_seq, w["H"], w["d"], w["d"]), dtype=torch.float32).pin_memory()
    h2d = nbytes(*host.values(), host_S0, host_cu)
    d2h = nbytes(o_h, ST_h)

    def step():
        dev = {n: t.to("cuda", non_blocking=True) for n, t in host.items()}
        S0 = None if host_S0 is None else host_S0.to("cuda", non_blocking=True)
        cu = None if host_cu is None else host_cu.to("cuda", non_blocking=True)
        fwd = kda.kda_fwd if segments is None else \
            (lambda *a, **kw: kda.kda_fwd_cp(*a, segments=segments, **kw))
        o, ST = fwd(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"], S0, cu,
                    stream=stream)
        o_h.copy_(o, non_blocking=True)
        ST_h.copy_(ST, non_blocking=True)
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
    stream.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / steps, world)
    return {"value": round(w["Ttot"] * world / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3)}


def e2e_prefill_pipelined(kda, w, steps, stream, world, segments=8):
    """The e2e metric for one sequence (B = 1), with the prompt uploaded in token
    segments: kda_fwd runs on each segment as soon as its inputs have landed,
    the state passing from one call to the next through S_T -> S0 (the result
    is compared with one call over the whole prompt afterwards), while the next segment uploads and the
    previous segment's o downloads.  Every step still copies all its inputs in
    from pinned host memory and o and S_T out, inside the timed region."""
    p = w["prob"]
    T, H, d = w["Ttot"], w["H"], w["d"]
    seg = -(-T // segments // 64) * 64  # segment length, whole chunks
    bounds = [(t, min(t + seg, T)) for t in range(0, T, seg)]
    names = ("q", "k", "v", "log_alpha", "beta")
    host = {n: getattr(p, n).reshape(T, *getattr(p, n).shape[2:]).to("cpu").pin_memory()
            for n in names}
    dev = {n: torch.empty_like(host[n], device="cuda") for n in names}
    host_S0 = None if p.S0 is None else p.S0.to("cpu").pin_memory()
    S0_d = None if host_S0 is None else torch.empty_like(host_S0, device="cuda")
    o_d = torch.empty((T, H, d), dtype=p.v.dtype, device="cuda")
    o_h = torch.empty((T, H, d), dtype=p.v.dtype).pin_memory()
    S_d = [torch.empty((1, H, d, d), dtype=torch.float32, device="cuda") for _ in range(2)]
    ST_h = torch.empty((1, H, d, d), dtype=torch.float32).pin_memory()
    ws = torch.empty(kda.kda_fwd_workspace_bytes(1), dtype=torch.uint8, device="cuda")
    h2d = nbytes(*host.values(), host_S0)
    d2h = nbytes(o_h, ST_h)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def step():
        ev_in, ev_done = [], []
        with torch.cuda.stream(s_in):
            s_in.wait_stream(stream)
            if host_S0 is not None:
                S0_d.copy_(host_S0, non_blocking=True)
            for t0, t1 in bounds:
                for n in names:
                    dev[n][t0:t1].copy_(host[n][t0:t1], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in)
                ev_in.append(e)
        for i, (t0, t1) in enumerate(bounds):
            stream.wait_event(ev_in[i])
            S0 = S0_d if i == 0 else S_d[(i - 1) % 2]
            kda.kda_fwd(dev["q"][t0:t1], dev["k"][t0:t1], dev["v"][t0:t1],
                        dev["log_alpha"][t0:t1], dev["beta"][t0:t1], S0, o=o_d[t0:t1],
                        S_T=S_d[i % 2], workspace=ws, stream=stream)
            e = torch.cuda.Event()
            e.record(stream)
            ev_done.append(e)
        with torch.cuda.stream(s_out):
            for i, (t0, t1) in enumerate(bounds):
                s_out.wait_event(ev_done[i])
                o_h[t0:t1].copy_(o_d[t0:t1], non_blocking=True)
            ST_h.copy_(S_d[(len(bounds) - 1) % 2], non_blocking=True)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
    stream.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / steps, world)
    # the segmented result against one kda_fwd call over the whole prompt
    with torch.cuda.stream(stream):
        o1, ST1 = kda.kda_fwd(p.q, p.k, p.v, p.log_alpha, p.beta, p.S0, stream=stream)
    stream.synchronize()
    same = bool(torch.equal(o1.reshape(T, H, d).cpu(), o_h) and torch.equal(ST1.cpu(), ST_h))
    return {"value": round(T * world / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "method": f"prompt uploaded in {len(bounds)} token segments, kda_fwd per segment "
                      f"as each lands (state chained through S_T -> S0), o downloaded behind",
            "bitwise_equal_to_one_call": same}


def e2e_decode(kda, w, steps, stream, world):
    S_dev = w["S"]
    host = [{n: t.to("cpu").pin_memory() for n, t in x.items()} for x in w["tokens"]]
    o_h = torch.empty(w["tokens"][0]["v"].shape, dtype=w["tokens"][0]["v"].dtype).pin_memory()
    h2d = nbytes(*host[0].values())
    d2h = nbytes(o_h)

    def step(i):
        x = {n: t.to("cuda", non_blocking=True) for n, t in host[i % len(host)].items()}
        o = kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S_dev,
                                stream=stream)
        o_h.copy_(o, non_blocking=True)
    with torch.cuda.stream(stream):
        step(0)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    with torch.cuda.stream(stream):
        a.record(stream)
        for i in range(steps):
            step(i)
        b.record(stream)
    stream.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / steps, world)
    return {"value": round(2 * nbytes(S_dev) * world / (ms / 1e3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4)}


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(w, heads=None, tokens=None):
    """Bounded sample of the workload for the fp64 oracle: the first `heads`
    heads (default 2 per core) over the first `tokens` tokens of a single
    sequence (default all), or every sequence of a packed batch; for decode,
    one session per core.  Returns (run, fraction of the workload, text, cores)."""
    import oracle
    cores = oracle.max_threads()
    if w["kind"] == "prefill":
        p = w["prob"]
        H = w["H"]
        nh = min(H, heads or max(1, 2 * cores))
        idx = torch.arange(nh, device=p.q.device)
        sl = lambda t: t
        T_s = w["Ttot"]
        if tokens is not None and p.cu_seqlens is None and p.q.dim() == 4 and p.q.shape[0] == 1:
            T_s = min(tokens, p.q.shape[1])
            sl = lambda t: t[:, :T_s]
        q, k, v = (sl(t).index_select(-2, idx) for t in (p.q, p.k, p.v))
        g = sl(p.log_alpha).index_select(-2, idx)
        b = sl(p.beta).index_select(-1, idx)
        S0 = None if p.S0 is None else p.S0.index_select(1, idx)
        cu = None if p.cu_seqlens is None else p.cu_seqlens.cpu().numpy()
        args = [oracle._f64(x) for x in (q, k, v, g, b)]
        s0 = None if S0 is None else oracle._f64(S0)

        def run():
            oracle.fwd(*args, s0, cu)
        tok = f"all {w['Ttot']} tokens" if T_s == w["Ttot"] else \
            f"the first {T_s} of {w['Ttot']} tokens"
        return run, (nh / H) * (T_s / w["Ttot"]), f"{nh} of {H} heads, {tok}", cores
    S = w["S"]
    x = w["tokens"][0]
    nsess = min(S.shape[0], max(1, cores))
    args = [oracle._f64(t[:nsess]) for t in (x["q"], x["k"], x["v"], x["log_alpha"],
                                              x["beta"])]
    S_h = oracle._f64(S[:nsess])

    def run():
        oracle.decode_step(*args, S_h)
    return run, nsess / S.shape[0], f"{nsess} of {S.shape[0]} sessions, all heads", cores


def cpu_baseline(w, args, target_s=10.0, max_repeats=50, heads=None, tokens=None):
    """The oracle on a bounded sample, repeated for about target_s seconds of CPU
    work, scaled to the whole workload."""
    run, frac, sample, cores = oracle_sample(w, heads, tokens)
    run()  # warm (and builds the oracle library if needed)
    repeats = 0
    t0 = time.perf_counter()
    while True:
        run()
        repeats += 1
        elapsed = time.perf_counter() - t0
        if elapsed >= target_s or repeats >= max_repeats:
            break
    dt = elapsed / repeats / frac  # seconds for the whole workload
    extra = {"cores": cores, "kind": "oracle", "sample": f"{sample}, {repeats} repeats",
             "seconds_sampled": round(elapsed, 2)}
    if w["kind"] == "prefill":
        return {"value": round(w["Ttot"] / dt, 2), "unit": "tokens/s", **extra}
    return {"value": round(2 * nbytes(w["S"]) / dt / 1e9, 4), "unit": "GB/s", **extra}


def run_reference(args, world, rank):
    """The oracle, as it stands, on the host cores (rank 0 only).  A step is the
    oracle over a bounded sample of the workload; `ms_per_step` is the
    sample's own time, and `value` scales the sample's throughput to the
    workload's unit (`sample_fraction` gives the factor)."""
    if rank != 0:
        return None
    w = make_workload(args.workload, seed=args.seed,
                      device="cuda" if torch.cuda.is_available() else "cpu")
    run, frac, sample, cores = oracle_sample(w)
    for _ in range(max(1, args.warmup)):  # untimed (the first builds the oracle library)
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt_sample = (time.perf_counter() - t0) / args.steps
    dt = dt_sample / frac  # the whole workload at this rate
    if w["kind"] == "prefill":
        value, unit = w["Ttot"] / dt, "tokens/s"
    else:
        value, unit = 2 * nbytes(w["S"]) / dt / 1e9, "GB/s"
    return {"metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt_sample * 1e3, 2),
            "sample_fraction": round(frac, 6),
            "ms_per_workload": round(dt * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded)", "impl": "reference",
            "config": line_config(w, world),
            "cpu_baseline": {"value": round(value, 3), "unit": unit, "cores": cores,
                             "kind": "oracle",
                             "sample": sample + " per step (ms_per_step is the sample's "
                                                "time; value is scaled to the workload)"},
            "e2e": {"value": round(value, 3), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload",
                    choices=["prefill", "decode", "long", "long_tp8", "varlen", "tiny"],
                    default="prefill")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--segments", default=None,
                    help="prefill workloads: time kda_fwd_cp with this many segments per "
                         "sequence ('auto': the library's suggestion) instead of kda_fwd")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode, draft and segment-parallel sub-benchmarks")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, _ = dist_setup(args.gpus)
    line = run_reference(args, world, rank) if args.impl == "reference" else \
        run_ours(args, world, rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
