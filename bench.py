#!/usr/bin/env python3
"""Benchmark of the KDA forward (chunked WY prefill) and the KDA decode step on GB300.

One step = one chunked forward over the prefill workload (B8 H32 T4096 K=V=128,
chunk 64, bf16 I/O, fp32 state) through the C ABI: gate, intra-chunk WY,
inter-chunk carry and output.  After the timed prefill steps the decode
workload (B256 H32 K=V=128, fp32 state 512 MiB updated in place) is timed for
64 consecutive single-token steps and reported in the same JSON line under
"decode", the long-sequence workload (B1 H32 T65536, h0 given; the split
chunk-parallel form) under "long", and the backward of the prefill workload
(kda_chunk_backward: every input's gradient from dL/do and dL/dhT) under "backward".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs the whole workload on its own GPU (weak
scaling, no data-path collective); rank 0 prints one JSON line.

--impl reference times the f64 CPU oracle (the token-by-token recurrence) on the
host cores, on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA fwd tokens/s & TFLOP/s (% bf16 peak); decode state GB/s (% HBM)"
WORKLOAD = "prefill_bf16"
# Algorithmic work per token-head of the chunked forward (C = 64, K = V = 128):
#   FLOPs 6KV + 3CK + 2CV + C^2/3 (triangular counts) and the essential HBM bytes:
#   q, k, v, z read and o written in bf16 (5 x 256 B) plus beta (2 B).
def flops_per_token_head(C, K, V):
    return 6 * K * V + 3 * C * K + 2 * C * V + C * C / 3.0


# Algorithmic work per token-head of the backward (chunks of C = 16): the state terms are
# twice the forward's (dDelta, dKt, dQg, dY S^T and the two products of the dS update:
# 12KV) plus the intra-chunk terms counted as for the forward.
def bwd_flops_per_token_head(C, K, V):
    return 12 * K * V + 3 * C * K + 2 * C * V + C * C / 3.0


# fp32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 FLOPs at the maximum SM clock
def fp32_peak_tflops(sm_mhz=2070.0):
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


def bytes_per_token_head(K, V, io_bytes=2):
    return io_bytes * (3 * K + V) + io_bytes * V + io_bytes


def measured_traffic(kernel, source, key="dram_bytes_per_launch"):
    """DRAM bytes of `kernel` from the committed ncu summary (profiles/traffic.json), or None
    when a source it was built from has changed since those counters were taken.  `source`
    is one file name or a tuple of them (all must match)."""
    import hashlib
    sources = (source,) if isinstance(source, str) else tuple(source)
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            entry = json.load(fh)[kernel]
        for src in sources:
            with open(os.path.join(ROOT, "gated_delta_rule_26_gb300", "csrc", src), "rb") as fh:
                digest = hashlib.sha256(fh.read()).hexdigest()
            if entry.get("source_sha256", {}).get(src) != digest:
                return None
    except (OSError, KeyError, ValueError, AttributeError):
        return None
    return entry.get(key)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for ln in fh:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    from gated_delta_rule_26_gb300 import dist as kdist
    return kdist.env()


def timed(fn, steps, stream, events=True):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


def oracle_sample(inp, n_pairs, threads, T=None):
    """Run the f64 oracle on n_pairs (b, h) sequences of the workload; returns (seconds, tokens)."""
    import oracle
    T = T or inp.T
    pairs = [(i % inp.B, (i * 7) % inp.H) for i in range(n_pairs)]
    bs = [p[0] for p in pairs]
    hs = [p[1] for p in pairs]
    g = lambda t: t[bs, hs, :T].unsqueeze(0)
    h0 = None if inp.h0 is None else inp.h0[bs, hs].unsqueeze(0)
    args = (g(inp.q), g(inp.k), g(inp.v), g(inp.z), inp.beta[bs, hs, :T].unsqueeze(0),
            inp.A_log[hs], inp.dt_bias[hs])
    args = tuple(oracle.f64(a) for a in args)
    t0 = time.perf_counter()
    oracle.forward(*args, inp.scale, h0, threads=threads)
    dt = time.perf_counter() - t0
    # tokens of the workload's unit: one token-head sequence of T tokens is T / H "tokens"
    return dt, n_pairs * T / inp.H


def cpu_baseline(inp, budget_s=12.0):
    """Oracle as it stands, on the host cores, on a bounded sample; tokens/s (B*T tokens)."""
    threads = os.cpu_count() or 1
    # calibrate: one thread, one (b, h) sequence of 256 tokens
    dt, _ = oracle_sample(inp, 1, 1, T=256)
    sec_per_token = dt / 256
    T = inp.T
    rounds = max(1, int(budget_s / max(sec_per_token * T, 1e-9)))
    n = threads * rounds
    dt, tokens = oracle_sample(inp, n, threads, T=T)
    return {"value": tokens / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} (b,h) sequences x T={T} of the {WORKLOAD} workload "
                      f"({n * T} token-heads, {dt:.1f} s); tokens = token-heads / H"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from gated_delta_rule_26_gb300 import inputs
    inp = inputs.workload(WORKLOAD)
    threads = os.cpu_count() or 1
    # one step = a bounded sample: `threads` (b, h) sequences of 1024 tokens
    T = 1024
    for _ in range(args.warmup):
        oracle_sample(inp, threads, threads, T=T)
    tot_s, tot_tok = 0.0, 0.0
    for _ in range(args.steps):
        dt, tok = oracle_sample(inp, threads, threads, T=T)
        tot_s += dt
        tot_tok += tok
    value = tot_tok / tot_s
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{WORKLOAD} B8 H32 T4096 K=V=128 chunk 64 (sampled)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle",
                             "sample": f"per step {threads} (b,h) sequences x T={T}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_decode(args, kda, inputs, peaks, ws, barrier):
    """Time `decode_steps` consecutive in-place decode steps on the fp32 state."""
    import torch
    stream = torch.cuda.current_stream()
    dec = inputs.decode(steps=args.decode_steps, B=args.decode_batch)

    dq, dk, dv, dz, db = (t.cuda() for t in (dec.q, dec.k, dec.v, dec.z, dec.beta))
    dA, ddt = dec.A_log.cuda(), dec.dt_bias.cuda()
    state = dec.state.cuda()
    dout = torch.empty(dec.B, dec.H, 1, dec.V, device="cuda", dtype=torch.bfloat16)
    it = [0]

    def dstep():
        s = it[0] % dec.steps
        kda.recurrent_step(dq[s], dk[s], dv[s], dz[s], db[s], dA, ddt, state, dec.scale, out=dout)
        it[0] += 1

    for _ in range(3):
        dstep()
    barrier()
    dsecs = timed(dstep, dec.steps, stream)
    from gated_delta_rule_26_gb300 import dist as kdist
    dsecs = kdist.max_over_ranks(dsecs, device="cuda")
    dper = dsecs / dec.steps
    dbytes = 2 * dec.B * dec.H * dec.K * dec.V * 4 + dec.B * dec.H * (3 * dec.K + 2 * dec.V + 1) * 2
    decode = {"value": ws * dec.B / dper, "unit": "tokens/s", "us_per_step": dper * 1e6,
              "state_GBps": dbytes / dper / 1e9,
              "roofline": {"bound": "hbm", "achieved": dbytes / dper / 1e9,
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": dbytes / dper / 1e9 / peaks["hbm_gbs"],
                           "traffic": measured_traffic("decode_stream_kernel",
                                                         ("decode.cu", "tc_ptx.cuh", "common.cuh"))
                           if dec.B == 256 else None,
                           "algorithmic_bytes": dbytes},
              "config": {"workload": f"decode_bf16 B{dec.B} H{dec.H} K={dec.K} V={dec.V}, "
                                     f"{dec.steps} consecutive steps",
                         "bytes_per_step": dbytes}}

    return decode


def run_long(args, kda, inputs, peaks, ws, barrier):
    """Time the long-sequence workload (few heads, 65536 tokens, h0 given) through the public
    entry point, which takes the split form here; reported under "long"."""
    import torch
    stream = torch.cuda.current_stream()
    inp = inputs.workload("long_bf16", **({"T": args.long_T} if args.long_T else {}))
    B, H, T, K, V, C = inp.B, inp.H, inp.T, inp.K, inp.V, inp.chunk
    d = inp.to("cuda")
    out = torch.empty(B, H, T, V, device="cuda", dtype=torch.bfloat16)
    hT = torch.empty(B, H, K, V, device="cuda", dtype=torch.float32)

    def step():
        kda.chunk_forward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, inp.scale, d.h0, C,
                          out=out, hT=hT)

    # at least 3 warm-up steps and 0.2 s of them, so that the clocks have left any idle state
    # (this leg may start right after the inputs' upload, with the GPU idle for seconds)
    t_end = time.perf_counter() + 0.2
    for i in range(1000):
        step()
        if i >= 2:
            torch.cuda.synchronize()
            if time.perf_counter() >= t_end:
                break
    barrier()
    n0 = kda.launch_count()
    secs = timed(step, args.long_steps, stream)
    launches = kda.launch_count() - n0
    from gated_delta_rule_26_gb300 import dist as kdist
    secs = kdist.max_over_ranks(secs, device="cuda")
    per = secs / args.long_steps
    th = B * H * T
    alg_bytes = th * bytes_per_token_head(K, V) + 2 * B * H * K * V * 4
    flops = th * flops_per_token_head(C, K, V)
    gbs = alg_bytes / per / 1e9
    res = {"value": ws * B * T / per, "unit": "tokens/s", "ms_per_step": per * 1e3,
           "steps": args.long_steps, "tflops": flops / per / 1e12,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"],
                        "traffic": measured_traffic("split_form_long_bf16",
                                                    ("chunk_tc.cu", "chunk_carry.cu",
                                                     "chunk_tiles.cuh", "tc_ptx.cuh"),
                                                    key="dram_bytes_per_step")
                        if T == 65536 else None,
                        "traffic_scope": "all kernels of one step (prep + carry), DRAM read + write",
                        "algorithmic_bytes": alg_bytes, "kernel": "kda chunked forward, split form",
                        "kernels_per_step": launches / args.long_steps,
                        "peak_source": peaks["source"]},
           "gpu_launches": launches,
           "config": {"workload": f"long_bf16 B{B} H{H} T{T} K={K} V={V} chunk {C}, h0 given",
                      "form": "split (chosen by kda_chunk_forward for this shape)"}}
    del d, out, hT
    torch.cuda.empty_cache()
    res["few_heads"] = run_long_few_heads(args, kda, inputs, peaks, ws, barrier)
    return res


def run_long_few_heads(args, kda, inputs, peaks, ws, barrier, H=4):
    """The long workload with few heads (B1 H4 T65536): kda_chunk_forward takes the split form
    with the chunk-parallel state scan here; the split form without it is timed beside it."""
    import torch
    stream = torch.cuda.current_stream()
    inp = inputs.workload("long_bf16", H=H, **({"T": args.long_T} if args.long_T else {}))
    B, T, K, V, C = inp.B, inp.T, inp.K, inp.V, inp.chunk
    d = inp.to("cuda")
    out = torch.empty(B, H, T, V, device="cuda", dtype=torch.bfloat16)
    hT = torch.empty(B, H, K, V, device="cuda", dtype=torch.float32)
    res = {}
    for form in ("auto", "split"):
        def step():
            kda.chunk_forward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, inp.scale, d.h0, C,
                              out=out, hT=hT, form=form)
        for _ in range(3):
            step()
        barrier()
        n0 = kda.launch_count()
        secs = timed(step, args.long_steps, stream)
        launches = kda.launch_count() - n0
        from gated_delta_rule_26_gb300 import dist as kdist
        per = kdist.max_over_ranks(secs, device="cuda") / args.long_steps
        alg_bytes = B * H * T * bytes_per_token_head(K, V) + 2 * B * H * K * V * 4
        res[form] = {"ms_per_step": per * 1e3, "value": ws * B * T / per, "unit": "tokens/s",
                     "hbm_frac": alg_bytes / per / 1e9 / peaks["hbm_gbs"],
                     "kernels_per_step": launches / args.long_steps}
    res["config"] = {"workload": f"long_bf16 B{B} H{H} T{T} K={K} V={V} chunk {C}, h0 given",
                     "forms": "auto = kda_chunk_forward (the split form with the state scan for "
                              "this shape); split = kda_chunk_forward_split"}
    del d, out, hT
    torch.cuda.empty_cache()
    return res


def run_backward(args, kda, inputs, peaks, ws, barrier):
    """Time the backward of the prefill workload (gradients of every input from seeded dL/do
    and dL/dhT) through kda_chunk_backward; reported under "backward"."""
    import torch
    stream = torch.cuda.current_stream()
    inp = inputs.workload(WORKLOAD, **({"T": args.backward_T} if args.backward_T else {}))
    adj = inputs.adjoints(inp, seed=77)
    B, H, T, K, V = inp.B, inp.H, inp.T, inp.K, inp.V
    d = inp.to("cuda")
    d_o, dhT = adj.d_o.to("cuda"), adj.dhT.to("cuda")

    from gated_delta_rule_26_gb300 import dist as kdist

    def step():
        g = kda.chunk_backward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, d_o, inp.scale,
                               h0=d.h0, dhT=dhT)
        # data parallel over ranks: the gate parameters' gradients are summed over all ranks'
        # batches (one all-reduce of H + H K floats; nothing on one GPU)
        kdist.sum_param_grads(g)

    for _ in range(2):
        step()
    barrier()
    n0 = kda.launch_count()
    secs = timed(step, args.backward_steps, stream)
    launches = kda.launch_count() - n0
    secs = kdist.max_over_ranks(secs, device="cuda")
    per = secs / args.backward_steps
    C = 16
    flops = B * H * T * bwd_flops_per_token_head(C, K, V)
    achieved = flops / per / 1e12
    tensor = K == 128 and V == 128  # the tensor-core form; other shapes run on the CUDA cores
    if tensor:
        # the contractions with the state (12KV of the count) are tcgen05 products, each as the
        # four bf16 products of hi/lo operand halves; the rest runs on the CUDA cores
        roof = {"bound": "tensor", "peak": peaks["bf16_tflops"],
                "peak_source": f"bf16 dense, {peaks['source']} (burst)",
                "kernel": "kda_chunk_bwd_tc_kernel (+ the batch sum of dA_log, ddt_bias)",
                "tensor_products_per_state_product": 4,
                "fp32_cuda_core_frac": achieved / fp32_peak_tflops(),
                "traffic": measured_traffic("kda_chunk_bwd_tc_kernel",
                                            ("chunk_bwd.cu", "chunk_tiles.cuh", "tc_ptx.cuh",
                                             "common.cuh")) if T == 4096 else None}
    else:
        roof = {"bound": "alu", "peak": fp32_peak_tflops(),
                "peak_source": "fp32 FMA: 152 SMs x 128 lanes x 2 x 2070 MHz",
                "kernel": "kda_chunk_bwd_kernel (+ the batch sum of dA_log, ddt_bias)",
                "traffic": None}
    roof.update({"achieved": achieved, "unit": "TFLOP/s", "frac": achieved / roof["peak"],
                 "flops_convention": "12KV+3CK+2CV+C^2/3 per token-head, C=16"})
    res = {"value": ws * B * T / per, "unit": "tokens/s", "ms_per_step": per * 1e3,
           "steps": args.backward_steps,
           "roofline": roof,
           "gpu_launches": launches,
           "config": {"workload": f"{WORKLOAD} backward B{B} H{H} T{T} K={K} V={V}, "
                                  "bf16 inputs, fp32 gradients, dL/dhT given",
                      "parallelism": (f"data parallel x{ws}: batch per rank, dA_log and "
                                      "ddt_bias all-reduced") if ws > 1 else "single GPU"}}
    del d, d_o, dhT
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-steps", type=int, default=64)
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="decode batch B (default: the decode workload's 256)")
    ap.add_argument("--long-steps", type=int, default=5,
                    help="timed steps of the long-sequence workload")
    ap.add_argument("--long-T", type=int, default=None,
                    help="sequence length of the long-sequence workload (default 65536; smaller "
                         "for profiler captures)")
    ap.add_argument("--backward-steps", type=int, default=3,
                    help="timed steps of the backward workload")
    ap.add_argument("--backward-T", type=int, default=None,
                    help="sequence length of the backward workload (default 4096; smaller for "
                         "profiler captures)")
    ap.add_argument("--only", default="all", choices=["all", "prefill", "decode", "long",
                                                      "backward"],
                    help="time only one of the two workloads (for profiler captures)")
    ap.add_argument("--prefill-T", type=int, default=None,
                    help="sequence length of the prefill workload (default 4096; smaller for "
                         "profiler captures)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from gated_delta_rule_26_gb300 import build as kbuild
    kbuild.build()
    from gated_delta_rule_26_gb300 import inputs, kda

    from gated_delta_rule_26_gb300 import dist as kdist

    def barrier():
        kdist.barrier()

    peaks = load_peaks()
    if args.only == "long":
        res = run_long(args, kda, inputs, peaks, ws, barrier)
        if rank == 0:
            print(json.dumps({"metric": "long only", "long": res}), flush=True)
        return 0
    if args.only == "backward":
        res = run_backward(args, kda, inputs, peaks, ws, barrier)
        if rank == 0:
            print(json.dumps({"metric": "backward only", "backward": res}), flush=True)
        return 0
    if args.only == "decode":
        decode = run_decode(args, kda, inputs, peaks, ws, barrier)
        if rank == 0:
            print(json.dumps({"metric": "decode only", "decode": decode}), flush=True)
        return 0
    inp_cpu = inputs.workload(WORKLOAD, **({"T": args.prefill_T} if args.prefill_T else {}))
    B, H, T, K, V, C = inp_cpu.B, inp_cpu.H, inp_cpu.T, inp_cpu.K, inp_cpu.V, inp_cpu.chunk
    d = inp_cpu.to("cuda")
    stream = torch.cuda.current_stream()
    out = torch.empty(B, H, T, V, device="cuda", dtype=torch.bfloat16)
    hT = torch.empty(B, H, K, V, device="cuda", dtype=torch.float32)

    def step():
        kda.chunk_forward(d.q, d.k, d.v, d.z, d.beta, d.A_log, d.dt_bias, inp_cpu.scale, d.h0, C,
                          out=out, hT=hT)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    barrier()
    n0 = kda.launch_count()
    secs = timed(step, args.steps, stream)
    launches = kda.launch_count() - n0
    clocks = sampler.stop()
    barrier()
    secs = kdist.max_over_ranks(secs, device="cuda")
    per_step = secs / args.steps
    tokens = B * T
    token_heads = B * H * T
    value = ws * tokens / per_step
    flops = token_heads * flops_per_token_head(C, K, V)
    alg_bytes = token_heads * bytes_per_token_head(K, V) + B * H * K * V * 4 * (
        2 if inp_cpu.h0 is not None else 1)
    kernels_per_step = launches / args.steps
    # Dominant kernel: the chunked forward launches `kernels_per_step` kernels per step; with one
    # kernel the step time is that kernel's time.
    achieved_gbs = alg_bytes / per_step / 1e9
    roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"],
                "traffic": measured_traffic("kda_chunk_tc_kernel", ("chunk_tc.cu", "chunk_tiles.cuh",
                                                                     "tc_ptx.cuh")),
                "algorithmic_bytes": alg_bytes,
                "kernel": "kda chunked forward", "kernels_per_step": kernels_per_step,
                "peak_source": peaks["source"]}
    tflops = flops / per_step / 1e12

    if args.only == "prefill":
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "ms_per_step": per_step * 1e3,
                "config": {"workload": f"{WORKLOAD} B{B} H{H} T{T}"}, "roofline": roofline,
                "gpu_launches": launches}
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0
    # ---- end to end through the public API: pinned host inputs -> device -> forward -> host.
    # Every step uploads its inputs and reads its output and final state back; two slots on
    # three streams let step i+1's uploads run under step i's forward and read-back.
    host = {n: getattr(inp_cpu, n).pin_memory() for n in ("q", "k", "v", "z", "beta", "A_log",
                                                         "dt_bias")}
    slots = []
    for _ in range(2):
        slots.append({
            "dev": {n: torch.empty_like(t, device="cuda") for n, t in host.items()},
            "out": torch.empty(B, H, T, V, device="cuda", dtype=torch.bfloat16),
            "hT": torch.empty(B, H, K, V, device="cuda", dtype=torch.float32),
            "out_h": torch.empty(B, H, T, V, dtype=torch.bfloat16).pin_memory(),
            "hT_h": torch.empty(B, H, K, V, dtype=torch.float32).pin_memory(),
            "up": torch.cuda.Event(), "run": torch.cuda.Event(), "down": torch.cuda.Event()})
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = slots[0]["out_h"].numel() * 2 + slots[0]["hT_h"].numel() * 4
    s_up, s_run, s_down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_steps_run(n):
        for i in range(n):
            sl = slots[i % 2]
            with torch.cuda.stream(s_up):
                s_up.wait_event(sl["run"])  # this slot's inputs were read by its last forward
                for name, t in host.items():
                    sl["dev"][name].copy_(t, non_blocking=True)
                sl["up"].record(s_up)
            s_run.wait_event(sl["up"])
            s_run.wait_event(sl["down"])  # this slot's outputs were read back
            dv = sl["dev"]
            kda.chunk_forward(dv["q"], dv["k"], dv["v"], dv["z"], dv["beta"], dv["A_log"],
                              dv["dt_bias"], inp_cpu.scale, None, C, out=sl["out"], hT=sl["hT"],
                              stream=s_run)
            sl["run"].record(s_run)
            with torch.cuda.stream(s_down):
                s_down.wait_event(sl["run"])
                sl["out_h"].copy_(sl["out"], non_blocking=True)
                sl["hT_h"].copy_(sl["hT"], non_blocking=True)
                sl["down"].record(s_down)

    e2e_steps_run(2)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 10))
    barrier()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(s_up)
    e2e_steps_run(e2e_steps)
    s_up.wait_stream(s_down)
    t_end.record(s_up)
    torch.cuda.synchronize()
    e2e_secs = t_start.elapsed_time(t_end) / 1e3
    e2e_secs = kdist.max_over_ranks(e2e_secs, device="cuda")
    e2e = {"value": ws * tokens / (e2e_secs / e2e_steps), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "pipelining": "two slots: uploads of step i+1 overlap the forward and read-back "
                         "of step i; the uploads (host-to-device ~190 GB/s) bound the step"}
    del host, slots

    decode = None if args.only == "prefill" else run_decode(args, kda, inputs, peaks, ws, barrier)
    del d
    torch.cuda.empty_cache()
    long_res = run_long(args, kda, inputs, peaks, ws, barrier)
    backward = None if args.only == "prefill" else run_backward(args, kda, inputs, peaks, ws, barrier)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"{WORKLOAD} B{B} H{H} T{T} K={K} V={V} chunk {C}",
                       "B": B, "H": H, "T": T, "K": K, "V": V, "chunk": C,
                       "state": "fp32", "h0": "zero",
                       "l2": "inputs larger than L2 (%.2f GB per step)" % (alg_bytes / 1e9),
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
            "tflops": tflops, "tflops_frac_bf16_burst": tflops / peaks["bf16_tflops"],
            "tflops_convention": "algorithmic (triangular) FLOPs 6KV+3CK+2CV+C^2/3 per token-head",
            "roofline": roofline, "e2e": e2e, "clocks": clocks, "gpu_launches": launches,
            "decode": decode, "long": long_res, "backward": backward}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp_cpu)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
