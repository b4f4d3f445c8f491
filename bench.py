"""Prefill throughput benchmark.

One step = one whole prefill forward pass (embed -> every decoder layer ->
output norm -> lm_head logits [T, n_vocab] f32) of the 8B-shape dense decoder
over T = 4096 synthetic tokens, through the C ABI.  Weights are random-init
(seeded N(0, 0.02), norm scales 1 + N(0, 0.1)) with that architecture; tokens
are seeded uniform ids.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dtp|reference]

N > 1 runs under torchrun as independent replicas (one sequence per rank, no
collective on the data path); value = tokens of all ranks / max rank time.
`--impl reference` times the CPU oracle (float64 numpy) on a bounded sample
of the same workload, on the host cores, rank 0 only.
Prints one JSON line on rank 0.
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

import synth  # noqa: E402

METRIC = "prefill tokens/s and TFLOP/s vs GB300 peak (1 GPU), logits vs CPU oracle"
UNIT = "tokens/s"
# device logit buffers of the end-to-end leg (2.49 GB each at the 8B shape)
E2E_DEVICE_BUFFERS = 8


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def profiled_traffic(profile: str, sources) -> float | None:
    """DRAM bytes per launch recorded by an ncu capture under profiles/, or None if
    the kernel sources changed since (their hash no longer matches) or there is none."""
    import hashlib
    import re

    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    m = re.search(r"traffic_bytes_per_launch=(\d+) source_sha256_16=([0-9a-f]+)", open(path).read())
    if not m:
        return None
    h = hashlib.sha256()
    for f in sources:
        h.update(open(os.path.join(ROOT, "dense_transformer_prefill_gb300", "csrc", f), "rb").read())
    return float(m.group(1)) if h.hexdigest()[:16] == m.group(2) else None


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """Maximum of a per-rank float over the process group (identity when world == 1)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, tokens_per_rank_step: int, steps: int, max_ms: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank_step * steps / (max_ms / 1000.0)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle timing
class OracleSample:
    """A bounded sample of the workload for the float64 oracle, scaled to the whole
    pass: one decoder layer over the first S_l tokens (t_layer), of which the
    attention alone takes t_attn (timed on its own at the same shape), and the
    lm_head over S_h rows x a V_s-row slice of the vocabulary (t_head).  The
    layer's projections and FFN grow linearly in T and its attention
    quadratically, so the whole pass is extrapolated as
      n_layer * ((t_layer - t_attn) * T/S_l + t_attn * (T/S_l)^2)
      + t_head * (T/S_h) * (V/V_s),
    and tokens/s = T / that."""

    def __init__(self, cfg, s_layer: int = 1024, s_head: int = 512, v_slice: int = 8192):
        self.cfg = cfg
        self.mode = {"bf16_operands": cfg.precision == "bf16",
                     "tf32_operands": cfg.precision == "tf32",
                     "fp8_operands": cfg.precision == "e4m3"}
        self.sl = min(cfg.T, s_layer)
        self.sh = min(cfg.T, s_head)
        self.vs = min(cfg.n_vocab, v_slice)
        self.lw = synth.layer_weights(cfg, 0)
        toks = synth.tokens(cfg)[:self.sl]
        self.x = synth.tok_embd(cfg)[toks].astype(np.float64)
        self.W = synth.normal(0, synth.TID_OUTPUT, (self.vs, cfg.n_embd), std=0.02)
        self.hn = synth.normal(0, 99, (self.sh, cfg.n_embd))
        hd = cfg.head_dim
        self.q = synth.normal(0, 97, (self.sl, cfg.n_head * hd)).astype(np.float64)
        self.kv = synth.normal(0, 98, (self.sl, cfg.n_head_kv * hd)).astype(np.float64)

    def run(self) -> dict:
        import oracle

        cfg, T = self.cfg, self.cfg.T
        t0 = time.perf_counter()
        oracle.forward_layer(cfg, self.lw, self.x, np.arange(self.sl), **self.mode)
        t_layer = time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle.sdpa_causal_gqa(self.q, self.kv, self.kv, cfg.n_head, cfg.n_head_kv, cfg.head_dim,
                               cfg.head_dim ** -0.5)
        t_attn = min(time.perf_counter() - t0, t_layer)
        t0 = time.perf_counter()
        rnd = {"bf16": oracle.round_bf16, "tf32": oracle.round_tf32,
               "e4m3": oracle.fake_quant_rows_e4m3}.get(cfg.precision, lambda a: a)
        oracle.linear(rnd(self.hn), rnd(self.W))
        t_head = time.perf_counter() - t0
        r = T / self.sl
        total = (cfg.n_layer * ((t_layer - t_attn) * r + t_attn * r * r)
                 + t_head * (T / self.sh) * (cfg.n_vocab / self.vs))
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        return {"value": T / total, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample_s": t_layer + t_attn + t_head, "extrapolated_step_s": total,
                "sample": (f"float64 numpy oracle ({cfg.precision} operand mode,"
                           f" BLAS on all {cores} host cores) on {cfg.name}: 1 decoder layer over "
                           f"the first {self.sl} tokens ({t_layer:.2f} s, of which attention "
                           f"{t_attn:.2f} s) + lm_head over {self.sh} rows x {self.vs} vocab rows "
                           f"({t_head:.2f} s), extrapolated to {cfg.n_layer} layers x {T} tokens "
                           f"(attention quadratic, the rest linear in T) and the full "
                           f"{cfg.n_vocab} vocab")}


def attention_sweep(dtp, dev, peak, Ts=(1024, 4096, 8192, 16384), reps=5) -> dict:
    """Causal GQA flash attention alone at the sweep shape (h=32, g=8, hd=128,
    q/k/v ~ N(0,1) bf16): mean kernel time over `reps` launches (CUDA events on the
    launch stream, after warm-up) and TFLOP/s against h*2*hd*T*(T+1)."""
    import torch

    sw = synth.ATTN_SWEEP
    nh, nkv, hd = sw["n_head"], sw["n_head_kv"], sw["head_dim"]
    out = {}
    for T in Ts:
        inp = synth.attention_inputs(T, nh, nkv, hd)
        q, k, v = (torch.as_tensor(inp[n], device=dev).bfloat16() for n in ("q", "k", "v"))
        o = torch.empty_like(q)
        ws = torch.empty(dtp.sdpa_workspace_size(T, nkv, hd, dtp.DTP_BF16), dtype=torch.uint8,
                         device=dev)
        for _ in range(3):
            dtp.sdpa_causal_gqa(q, k, v, o, nh, nkv, hd, hd ** -0.5, ws)
        torch.cuda.synchronize(dev)
        dtp.timer_enable(["attn"], reps)
        for _ in range(reps):
            dtp.sdpa_causal_gqa(q, k, v, o, nh, nkv, hd, hd ** -0.5, ws)
        torch.cuda.synchronize(dev)
        n, ms = dtp.timer_read("attn")
        dtp.timer_disable()
        dtp.check()
        flops = nh * 2.0 * hd * T * (T + 1)
        tf = flops / (ms / n / 1000.0) / 1e12
        out[str(T)] = {"ms": ms / n, "tflops": tf, "frac": tf / peak if peak else None}
    return out


def span_summary(fwd, cpy) -> dict:
    """Where an end-to-end batch's time goes, from per-prompt (start, end) spans in
    ms: each prompt's pass on the compute stream and each logits copy on the copy
    stream.  idle = compute-stream gaps between passes; a copy overlaps the next
    pass when it starts before that pass ends."""
    if not fwd:
        return {}
    f_ms = [e - b for b, e in fwd]
    c_ms = [e - b for b, e in cpy]
    idle = [max(0.0, fwd[j + 1][0] - fwd[j][1]) for j in range(len(fwd) - 1)]
    overlap = [max(0.0, min(cpy[j][1], fwd[j + 1][1]) - max(cpy[j][0], fwd[j + 1][0]))
               for j in range(min(len(cpy), len(fwd) - 1))]
    wait = [max(0.0, cpy[j][0] - fwd[j][1]) for j in range(min(len(cpy), len(fwd)))]
    end = max([e for _, e in fwd] + [e for _, e in cpy])
    return {"prompts": len(fwd), "span_ms": end,
            "forward_ms_mean": statistics.mean(f_ms), "forward_ms_max": max(f_ms),
            "copy_ms_mean": statistics.mean(c_ms) if c_ms else None,
            "copy_ms_max": max(c_ms) if c_ms else None,
            "compute_idle_ms_total": sum(idle),
            "copy_start_after_ready_ms_mean": statistics.mean(wait) if wait else None,
            "copy_overlapped_with_next_forward_ms_total": sum(overlap),
            "per_prompt_ms": [[round(b, 1), round(e, 1)] for b, e in fwd],
            "per_copy_ms": [[round(b, 1), round(e, 1)] for b, e in cpy]}


def l2_note(cfg) -> str:
    """Whether a step's inputs exceed the 129 MB L2 (then no flush is needed
    between timed steps): the packed GEMM weights alone, in the step's operand type."""
    eb = {"e4m3": 1, "bf16": 2}.get(cfg.precision, 4)
    wbytes = cfg.gemm_flops(1) / 2 * eb          # gemm_flops(1) = 2 * weight elements
    if wbytes > 129e6:
        return f"inputs larger than L2 (packed weights {wbytes / 1e9:.1f} GB exceed 129 MB)"
    return f"inputs smaller than L2 (packed weights {wbytes / 1e6:.1f} MB): steps after the first run L2-warm"


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="dtp", choices=["dtp", "reference"])
    ap.add_argument("--workload", default="qwen3-8b-shape", choices=sorted(synth.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-attn-sweep", action="store_true")
    ap.add_argument("--n-layer", type=int, default=None,
                    help="override the layer count (profiling captures of a small case)")
    ap.add_argument("--precision", default=None, choices=["bf16", "tf32", "e4m3", "f32"],
                    help="arithmetic (default: the workload's, bf16 for the model shapes)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = synth.CONFIGS[args.workload]
    if args.n_layer is not None:
        cfg = cfg.replace(n_layer=args.n_layer)
    if args.precision is not None:
        cfg = cfg.replace(precision=args.precision)
    config = {"workload": cfg.name, "T": cfg.T, "n_layer": cfg.n_layer, "n_embd": cfg.n_embd,
              "n_head": cfg.n_head, "n_head_kv": cfg.n_head_kv, "head_dim": cfg.head_dim,
              "n_ff": cfg.n_ff, "n_vocab": cfg.n_vocab, "sequences_per_gpu": 1,
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
              "l2": l2_note(cfg)}

    if args.impl == "reference":
        if rank != 0:
            return
        config["l2"] = "not applicable (CPU oracle)"
        sampler = OracleSample(cfg)
        for _ in range(args.warmup):          # untimed samples (BLAS thread pool, page-in)
            sampler.run()
        samples = [sampler.run() for _ in range(args.steps)]
        v = statistics.median(s["value"] for s in samples)
        cb = dict(samples[0])
        cb["value"] = v
        # each step is one bounded sample; ms_per_step is the whole pass
        # extrapolated from it (see cpu_baseline.sample), not a timed full pass
        print(json.dumps({"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": 1000.0 * cfg.T / v,
                          "ms_per_step_kind": "extrapolated from one bounded sample per step",
                          "sample_ms_per_step": 1000.0 * statistics.median(
                              s["sample_s"] for s in samples),
                          "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "impl": "reference", "config": config,
                          "cpu_baseline": cb,
                          "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return

    import torch
    import dense_transformer_prefill_gb300 as dtp

    dtp.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ------------------------------------------------------------------ setup (untimed)
    t_setup = time.perf_counter()
    m = dtp.Model(cfg, device=dev)
    for l in range(cfg.n_layer):
        m.load_layer(l, synth.layer_weights(cfg, l))
    m.load_globals(synth.tok_embd(cfg), synth.output_norm(cfg), synth.output_weight(cfg))
    toks_np = synth.tokens(cfg, seed=1000 + rank).astype(np.int32)
    toks = torch.as_tensor(toks_np, device=dev)
    logits = torch.empty((cfg.T, cfg.n_vocab), dtype=torch.float32, device=dev)
    m.workspace(cfg.T)
    setup_s = time.perf_counter() - t_setup
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        m.forward(toks, logits)
    torch.cuda.synchronize(dev)
    dtp.check()

    # ------------------------------------------------------------------ timed region
    gpu_index = local_rank
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local_rank])
        except (ValueError, IndexError):
            pass
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        n0 = dtp.launch_count()
        start.record(stream)
        for _ in range(args.steps):
            m.forward(toks, logits)
        end.record(stream)
        torch.cuda.synchronize(dev)
        launches = dtp.launch_count() - n0
        barrier()
    dtp.check()
    ms = max_over_ranks(start.elapsed_time(end), world, dev)
    ms_per_step = ms / args.steps
    value = replica_throughput(world, cfg.T, args.steps, ms)

    # ------------------------------------------------------------------ per-kernel times
    # A second pass of the same steps with a CUDA event pair around every launch
    # (on the launch stream): the per-kernel durations and the roofline come from
    # here; `value` above is measured without the events.
    kinds = ["gemm_qkv", "attn", "gemm_o", "gemm_gateup", "gemm_down", "gemm_lmhead", "rmsnorm",
             "embed", "other"]
    dtp.timer_enable(kinds, capacity=args.steps * (cfg.n_layer + 1) * 2)
    i_start, i_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    i_start.record(stream)
    for _ in range(args.steps):
        m.forward(toks, logits)
    i_end.record(stream)
    torch.cuda.synchronize(dev)
    dtp.check()
    instrumented_ms_per_step = i_start.elapsed_time(i_end) / args.steps
    kstats = {k: dtp.timer_read(k) for k in kinds}
    dtp.timer_disable()

    # ------------------------------------------------------------------ end to end (host buffers)
    e2e = None
    if not args.no_e2e:
        # one prompt per step, host to host: tokens in, the forward pass, all
        # logits out; the batch call overlaps prompt j's logits copy with the next
        # forward passes (two pinned host logit buffers, used alternately; eight
        # device logit buffers, so a copy slowed on the host side holds the
        # passes back only after seven more have finished)
        tok_h = [torch.as_tensor(synth.tokens(cfg, seed=2000 + 97 * rank + j).astype(np.int32))
                 .pin_memory() for j in range(args.steps)]
        log_h = [torch.empty((cfg.T, cfg.n_vocab), dtype=torch.float32).pin_memory()
                 for _ in range(2)]
        ws_h = torch.empty(dtp.workspace_size_host_batch(m.c, cfg.T, E2E_DEVICE_BUFFERS),
                           dtype=torch.uint8, device=dev)
        outs = [log_h[j % 2] for j in range(args.steps)]
        dtp.fwd_prefill_host_batch(m.c, m.packed, tok_h[:2], log_h, ws_h)
        torch.cuda.synchronize(dev)
        barrier()
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_start.record(stream)
        h0 = time.perf_counter()
        dtp.fwd_prefill_host_batch(m.c, m.packed, tok_h, outs, ws_h)
        host_enqueue_ms = (time.perf_counter() - h0) * 1e3
        e_end.record(stream)
        torch.cuda.synchronize(dev)
        dtp.check()
        ems = max_over_ranks(e_start.elapsed_time(e_end), world, dev)
        # the same call once more with a span around every prompt's pass (caller's
        # stream) and every logits copy (the library's copy stream): where the
        # end-to-end time goes
        dtp.timer_enable(["prompt", "d2h"], args.steps)
        d0 = time.perf_counter()
        dtp.fwd_prefill_host_batch(m.c, m.packed, tok_h, outs, ws_h)
        diag_enqueue_ms = (time.perf_counter() - d0) * 1e3
        torch.cuda.synchronize(dev)
        dtp.check()
        fwd = dtp.timer_spans("prompt", "prompt")
        cpy = dtp.timer_spans("d2h", "prompt")
        dtp.timer_disable()
        e2e_spans = span_summary(fwd, cpy)
        e2e_spans["host_enqueue_ms"] = diag_enqueue_ms
        # the device-to-host copy of one step's logits on its own: e2e is bound by
        # max(forward pass, this copy), and the copy depends on the host's memory
        c_start, c_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c_start.record(stream)
        log_h[0].copy_(logits, non_blocking=True)
        c_end.record(stream)
        torch.cuda.synchronize(dev)
        d2h_ms = c_start.elapsed_time(c_end)
        e2e = {"value": replica_throughput(world, cfg.T, args.steps, ems), "unit": UNIT,
               "ms_per_step": ems / args.steps,
               "host_enqueue_ms_per_step": host_enqueue_ms / args.steps,
               "spans": e2e_spans,
               "d2h_ms_per_step_alone": d2h_ms,
               "d2h_gbs_alone": log_h[0].numel() * 4 / d2h_ms / 1e6,
               "device_logit_buffers": E2E_DEVICE_BUFFERS,
               "h2d_bytes_per_step": int(tok_h[0].numel() * 4),
               "d2h_bytes_per_step": int(log_h[0].numel() * 4),
               "path": "dtp_fwd_prefill_host_batch: one prompt per step, pinned host tokens in, "
                       "all pinned host logits out; each prompt's logits copy overlaps the next "
                       "prompts' forward passes"}
        del log_h, outs, ws_h

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    # ------------------------------------------------------------------ roofline
    peaks = load_peaks()
    T, d, F = cfg.T, cfg.n_embd, cfg.n_ff
    gu_n, gu_ms = kstats["gemm_gateup"]
    gu_flops = 2.0 * T * (2 * F) * d
    achieved = gu_flops / (gu_ms / gu_n / 1000.0) / 1e12 if gu_n else None
    # GEMM peak of the operand type: the measured bf16 figure, times the nominal
    # dense ratio for tf32 (1.1 / 2.25) and e4m3 (4.5 / 2.25); attention runs bf16
    # tensor cores in bf16 and e4m3 modes
    bf16_peak = peaks["bf16_tflops_sustained"]
    peak = {"bf16": bf16_peak, "tf32": bf16_peak * 1.1 / 2.25,
            "e4m3": bf16_peak * 2.0}.get(cfg.precision)
    attn_peak = bf16_peak if cfg.precision in ("bf16", "e4m3") else None
    is8b = cfg.name == "qwen3-8b-shape" and cfg.T == 4096
    roofline = {"kernel": "gemm_tc_kernel (gate/up projection, %s operands)" % cfg.precision,
                "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if (achieved and peak) else None,
                "traffic": profiled_traffic("gemm_tc_gateup_qwen3-8b-shape.md",
                                            ["gemm_tc.cu", "ptx.cuh", "internal.h"]) if is8b else None,
                "algorithmic_bytes_per_launch": 2.0 * (T * d + 2 * F * d + T * F),
                "flops_per_launch": gu_flops,
                "peak_source": f"bf16_tflops_sustained of {peaks['source']} peaks"
                               + ("" if cfg.precision == "bf16" else
                                  f" x the nominal {cfg.precision}/bf16 dense ratio"),
                "avg_launch_ms": gu_ms / gu_n if gu_n else None}
    clocks = clk.summary()
    burst = {"bf16": peaks["bf16_tflops"], "tf32": peaks["bf16_tflops"] * 1.1 / 2.25,
             "e4m3": peaks["bf16_tflops"] * 2.0}.get(cfg.precision)
    roofline["frac_burst"] = (achieved / burst) if (achieved and burst) else None
    # the sustained peak was measured at its own median SM clock; compare per MHz
    peak_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
    if achieved and peak and peak_mhz and clocks.get("sm_mhz"):
        roofline["frac_at_equal_clock"] = (achieved / clocks["sm_mhz"]) / (peak / peak_mhz)
        roofline["clock_note"] = (f"this run's median SM clock {clocks['sm_mhz']:.0f} MHz; the "
                                  f"sustained peak's {peak_mhz:.0f} MHz")
    at_n, at_ms = kstats["attn"]
    at_flops = cfg.attn_flops() / cfg.n_layer
    at_ach = at_flops / (at_ms / at_n / 1000.0) / 1e12 if at_n else None
    roofline_attn = {"kernel": "attn_tc_kernel<%d> (causal GQA flash attention, one layer)"
                     % cfg.head_dim, "bound": "tensor", "achieved": at_ach, "peak": attn_peak,
                     "unit": "TFLOP/s",
                     "frac": (at_ach / attn_peak) if (at_ach and attn_peak) else None,
                     "traffic": profiled_traffic("attn_tc_qwen3-8b-shape.md",
                                                 ["attn_tc.cu", "ptx.cuh", "internal.h"]) if is8b else None,
                     "flops_per_launch": at_flops,
                     "avg_launch_ms": at_ms / at_n if at_n else None}
    if at_ach and cfg.precision in ("bf16", "e4m3"):
        roofline_attn["frac_burst"] = at_ach / peaks["bf16_tflops"]
    per_kernel = {}
    step_flops = 0.0
    for k, (n, kms) in kstats.items():
        if n:
            per_kernel[k] = {"launches_per_step": n / args.steps, "ms_per_step": kms / args.steps}
    gemm_flops = cfg.gemm_flops()
    attn_flops = cfg.attn_flops()
    step_flops = gemm_flops + attn_flops
    gemm_ms = sum(kstats[k][1] for k in ("gemm_qkv", "gemm_o", "gemm_gateup", "gemm_down",
                                         "gemm_lmhead")) / args.steps
    attn_ms = kstats["attn"][1] / args.steps
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.precision,
        "data": "synthetic (seeded random-init weights of the architecture, uniform token ids)",
        "config": config, "roofline": roofline, "roofline_attn": roofline_attn,
        "tflops": {"step": step_flops / (ms_per_step / 1000.0) / 1e12,
                   "gemm": gemm_flops / (gemm_ms / 1000.0) / 1e12 if gemm_ms else None,
                   "attn": attn_flops / (attn_ms / 1000.0) / 1e12 if attn_ms else None,
                   "gemm_frac_of_peak": (gemm_flops / (gemm_ms / 1000.0) / 1e12 / peak)
                   if (gemm_ms and peak) else None,
                   "attn_frac_of_peak": (attn_flops / (attn_ms / 1000.0) / 1e12 / attn_peak)
                   if (attn_ms and attn_peak) else None},
        "kernels": per_kernel,
        "instrumented_ms_per_step": instrumented_ms_per_step,
        "clocks": clocks,
        "gpu_launches": int(launches),
        "e2e": e2e,
        "setup_s": setup_s,
    }
    if not args.no_attn_sweep and cfg.precision == "bf16":
        # timed alone, launch after launch: compared with the burst peak
        burst = peaks["bf16_tflops"]
        out["attention_sweep"] = {"shape": "h=32, g=8, hd=128, bf16, causal; kernel time only",
                                  "peak": burst,
                                  "peak_source": f"bf16_tflops (burst) of {peaks['source']} peaks",
                                  "T": attention_sweep(dtp, dev, burst)}
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = OracleSample(cfg).run()
    print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
