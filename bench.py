#!/usr/bin/env python3
"""Throughput of the MoE layer forward on GB300: tokens/s on the Mixtral-8x7B-shaped prefill layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME] [--T T] [--ep]

One step = one colibri_moe_forward (router, gather, grouped up-GEMM, grouped down-GEMM, combine) over
a batch of T tokens already resident in HBM.  Prints one JSON line (rank 0).  Under torchrun each
rank runs the same workload on its own GPU (replicas, weak scaling, no data-path collective); the
reported time is the max over ranks and the value counts every rank's tokens.

--impl reference times the CPU oracle (fp64 C, OpenMP) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# stdout carries exactly one JSON line: keep NCCL's banner off it unless the caller asks for its logs
os.environ.setdefault("NCCL_DEBUG", "WARN")
sys.path.insert(0, os.path.join(ROOT, "tests"))

METRIC = "MoE-layer tokens/s at Mixtral-8x7B shape; % of bf16 tensor peak / HBM BW"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_BF16_TFLOPS = 2250.0  # GB300 dense bf16 tensor rate, datasheet (no sparsity)
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e, datasheet
# a timed region shorter than this is a burst: the GPU has not yet settled at its power cap, so a
# contraction is compared with the burst cuBLAS rate; longer regions with the sustained one
SUSTAINED_AFTER_S = 1.0
STAGES = ["router", "gather", "gemm_up", "gemm_down", "combine"]
# (the cooperative decode kernel runs inside the "gemm_up" stage: up GEMM, activation, down GEMM and
# combine in one launch, the other stages empty)
# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture of the kernel as it now
# stands; None where no capture of the current kernel exists.
DOM_EVERY = 8  # the dominant kernel is timed with events on every 8th step of the timed region
NCU_TRAFFIC = {("mixtral-prefill", 8192, "gemm_up", "2sm"): 2.618e9, ("mixtral-prefill", 8192, "gemm_down", "2sm"): 2.816e9,
               ("mixtral-decode", 1, "gemm_up", "1kernel"): 0.7092e9, ("mixtral-decode", 16, "gemm_up", "1kernel"): 2.8339e9,
               ("1.3b-8e", 512, "gemm_up", "2sm"): 0.3911e9, ("1.3b-8e", 512, "gemm_down", "2sm"): 0.2076e9,
               ("1.3b-8e", 512, "gemm_up", "1kernel"): 0.5947e9, ("skewed-16e", 4096, "gemm_up", "1kernel"): 0.4574e9}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="mixtral-prefill")
    p.add_argument("--T", type=int, default=None, help="tokens per step (default: the workload's)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU work budget of the oracle baseline")
    p.add_argument("--top-k", type=int, default=None, help="routed experts per token (default: the workload's, 2)")
    p.add_argument("--gate-mode", type=int, default=None, help="0 softmax over the selected experts, 1 full softmax")
    p.add_argument("--shared-expert", action="store_true", help="add an always-on shared expert")
    p.add_argument("--ep", action="store_true",
                   help="expert parallelism over the launched ranks (E / N experts per GPU, NCCL all-to-alls); "
                        "each rank routes its own batch of T tokens")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the decode sweep and the other workloads' step times that follow the main line")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(s, T):
    act = "SwiGLU" if s.act == 1 else "ReLU+bias"
    return (f"{s.name}: T={T} d_model={s.d_model} d_ff={s.d_ff} E={s.num_experts} top-{s.top_k} {act} {s.dtype}"
            + (" router-bias zipf" if s.zipf_router_bias else "")
            + (" full-softmax gates" if s.gate_mode == 1 else "")
            + (" +1 shared expert" if s.shared_expert else ""))


def algorithmic(s, T, active_experts=None):
    """FLOPs and bytes of one forward counting routed work only (no padding rows)."""
    n_up = 2 if s.act == 1 else 1
    es = 2 if s.dtype == "bf16" else 4
    rows = (s.top_k + int(s.shared_expert)) * T          # routed rows (+ the shared expert's)
    flops_up = 2.0 * rows * s.d_model * s.d_ff * n_up
    flops_down = 2.0 * rows * s.d_model * s.d_ff
    flops_router = 2.0 * T * s.num_experts * s.d_model
    n_act = (s.num_experts if active_experts is None else active_experts) + int(s.shared_expert)
    w_bytes_expert = (n_up + 1) * s.d_model * s.d_ff * es
    bytes_total = n_act * w_bytes_expert + T * s.d_model * es + T * s.d_model * 4 + s.num_experts * s.d_model * es
    return dict(flops_up=flops_up, flops_down=flops_down, flops_router=flops_router,
                flops=flops_up + flops_down + flops_router, bytes=bytes_total,
                w_bytes_up=n_act * n_up * s.d_model * s.d_ff * es, w_bytes_expert=w_bytes_expert)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank number over all ranks (the job takes as long as its slowest replica)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, tokens_per_rank_step: int, steps: int, seconds: float) -> float:
    """Tokens/s of the whole job: every replica processes its own batch each step (weak scaling)."""
    return world * tokens_per_rank_step * steps / seconds


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", *sel], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception as e:  # no nvidia-smi: report nothing rather than fail the bench
            log("clock sampler unavailable:", e)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        loaded = [c for c in sm if c > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------- CPU oracle
def oracle_rate(li, T, seconds, tokens_per_round=None, rounds=None, seed=0):
    """Time the oracle on a sample of the workload's tokens: routing (logits + top-2) of the sampled
    tokens and their two experts each.  Returns (tokens/s, tokens timed, wall seconds, threads)."""
    import numpy as np
    import oracle
    L = oracle.OracleLayer.from_inputs(li)
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    rng = np.random.default_rng(seed)

    def one(n):
        toks = np.sort(rng.choice(T, size=n, replace=False)).astype(np.int32)
        xs = li.x_f32[toks]
        t0 = time.perf_counter()
        logits = L.router_logits(xs)
        idx, gate = L.top2(logits)
        L.forward_rows(xs, idx, gate, np.arange(n, dtype=np.int32))
        return time.perf_counter() - t0

    if tokens_per_round is None:
        probe = max(1, min(threads, T))
        dt = one(probe)
        per_tok = dt / probe
        tokens_per_round = max(1, min(T, int(seconds / per_tok)))
        rounds = 1
    done, wall = 0, 0.0
    for _ in range(rounds):
        wall += one(tokens_per_round)
        done += tokens_per_round
    return done / wall, done, wall, min(threads, tokens_per_round)


def run_reference(args, shape, T):
    """--impl reference: the oracle as it stands, each step a bounded sample of the workload."""
    import testgen
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    li = testgen.make_inputs(shape.with_T(T), want_bits=False)
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    # size each step from one probe so the whole run stays within ~2-3 minutes
    rate, n, wall, _ = oracle_rate(li, T, 1.0)
    per_step = max(1, min(T, int(rate * 120.0 / max(1, args.steps + args.warmup))))
    for _ in range(args.warmup):
        oracle_rate(li, T, 0, tokens_per_round=per_step, rounds=1, seed=1)
    rate, n, wall, used = oracle_rate(li, T, 0, tokens_per_round=per_step, rounds=args.steps, seed=2)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(shape, T), "sample_tokens_per_step": per_step},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": f"{per_step} random tokens of {T} per step (routing + both experts, fp64)"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------- GPU arm
def time_forwards(layer, x_ptr, out_ptr, T, stream, steps, warmup):
    """ms per forward over `steps` back-to-back forwards, CUDA events on the launching stream."""
    import torch
    for _ in range(max(3, warmup)):
        layer.forward_ptr(x_ptr, out_ptr, T, stream.cuda_stream)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        layer.forward_ptr(x_ptr, out_ptr, T, stream.cuda_stream)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def decode_sweep(layer, shape, x, out, stream, hbm_gbs, steps):
    """The decode-shaped layer: the same weights, the first T rows of the batch, T in 1, 4, 16, 32.
    HBM fraction over the bytes of the distinct experts the batch activates (each read once)."""
    import testgen
    res = {}
    for Td in testgen.DECODE_TOKENS:
        ms = time_forwards(layer, x.data_ptr(), out.data_ptr(), Td, stream, steps, 10)
        counts = layer.get_routing(Td)["counts"].cpu().numpy()
        active = int((counts > 0).sum())
        wbytes = active * algorithmic(shape, Td)["w_bytes_expert"]
        res[str(Td)] = {"us_per_step": ms * 1e3, "tokens_per_s": Td / (ms / 1e3), "active_experts": active,
                        "weight_bytes": wbytes, "hbm_gbs": wbytes / (ms / 1e3) / 1e9,
                        "hbm_frac": wbytes / (ms / 1e3) / 1e9 / hbm_gbs, "steps": steps,
                        "kernels_per_step": layer.last_kernel_count(), "gemm_form": layer.last_gemm()}
    return res


def other_workloads(peaks, steps, device: int):
    """Step time of the benchmark's other layers (each with its own seeded weights), for the record."""
    import torch
    import testgen
    from moe_check import host_weights, x_device
    import mixture_experts_gemm_gb300 as moe
    dev = torch.device("cuda", device)
    stream = torch.cuda.current_stream(dev)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    res = {}
    for name in ("tiny-moe-4e2r", "1.3b-8e", "skewed-16e"):
        s = testgen.CONFIGS[name]
        li = testgen.make_inputs(s, want_f32=s.dtype == "f32")
        layer = moe.MoELayer(s.d_model, s.d_ff, s.num_experts, s.T, dtype=s.dtype,
                             act="swiglu" if s.act == testgen.ACT_SWIGLU else "relu_bias",
                             has_router_bias=s.zipf_router_bias, out_dtype="f32", device=device, top_k=s.top_k,
                             gate_mode=s.gate_mode, shared_expert=s.shared_expert)
        layer.load_weights(**host_weights(li))
        x = x_device(li).to(dev)
        out = torch.empty((s.T, s.d_model), dtype=torch.float32, device=dev)
        ms = time_forwards(layer, x.data_ptr(), out.data_ptr(), s.T, stream, steps, 10)
        counts = layer.get_routing(s.T)["counts"].cpu().numpy()
        alg = algorithmic(s, s.T, int((counts > 0).sum()))
        sec = ms / 1e3
        r = {"workload": workload_desc(s, s.T), "us_per_step": ms * 1e3, "tokens_per_s": s.T / sec,
             "tflops": alg["flops"] / sec / 1e12, "steps": steps, "kernels_per_step": layer.last_kernel_count(),
             "gemm_form": layer.last_gemm()}
        if s.dtype == "bf16":
            r["hbm_frac_over_weights"] = alg["bytes"] / sec / 1e9 / hbm
            r["tensor_frac_of_burst"] = alg["flops"] / sec / 1e12 / burst
            r["bound"] = "hbm" if alg["flops"] / alg["bytes"] < burst * 1e12 / (hbm * 1e9) else "tensor"
        else:
            r["bound"] = "latency (weights fit in L2; fp32 SIMT path)"
        res[name] = r
        layer.close()
        del x, out
        torch.cuda.empty_cache()
    return res


def ep_phases(li, shape, x, steps, device: int):
    """Expert parallelism on this one GPU: ep_size ranks of T / ep_size tokens each (the experts split
    in ep_size blocks), emulated in one process with the all-to-alls as device copies.  CUDA events
    time each phase of every rank: dispatch (router + pack), experts (regroup, up GEMM, down GEMM,
    unregroup), combine, and the copies standing in for the exchange."""
    import numpy as np
    import torch
    import mixture_experts_gemm_gb300 as moe
    from moe_check import host_weights
    n = 2
    T = x.shape[0] // n
    dev = torch.device("cuda", device)
    stream = torch.cuda.current_stream(dev)
    w = host_weights(li)
    El = shape.num_experts // n
    layers = []
    for r in range(n):
        L = moe.MoELayer(shape.d_model, shape.d_ff, shape.num_experts, T, dtype=shape.dtype, act="swiglu",
                         out_dtype="f32", device=device, top_k=shape.top_k, ep_rank=r, ep_size=n)
        own = lambda lst: None if lst is None else [t if r * El <= e < (r + 1) * El else None for e, t in enumerate(lst)]
        L.load_weights(w["w_router"], own(w["w1"]), own(w["w2"]), w3=own(w["w3"]), b_router=w["b_router"])
        layers.append(L)
    xs = [x[r * T:(r + 1) * T].contiguous() for r in range(n)]
    ev = lambda: torch.cuda.Event(enable_timing=True)
    acc = {"dispatch": 0.0, "exchange": 0.0, "experts": 0.0, "combine": 0.0}
    rows_recv = 0
    for it in range(steps + 3):
        e0, e1, e2, e3, e4, e5 = ev(), ev(), ev(), ev(), ev(), ev()
        e0.record(stream)
        sends = [L.ep_dispatch(xr) for L, xr in zip(layers, xs)]
        e1.record(stream)
        counts = [sc.cpu().numpy().astype(np.int64).reshape(n, -1) for _, sc in sends]
        per = [c.sum(axis=1) for c in counts]
        starts = [np.concatenate([[0], np.cumsum(p)[:-1]]) for p in per]
        e2.record(stream)
        recv = [torch.cat([sends[p][0][int(starts[p][q]):int(starts[p][q] + per[p][q])] for p in range(n)])
                for q in range(n)]
        rc = [np.stack([counts[p][q] for p in range(n)]).astype(np.int32) for q in range(n)]
        e3.record(stream)
        ys = [layers[q].ep_experts(recv[q], rc[q]) for q in range(n)]
        e4.record(stream)
        backs = []
        for p in range(n):
            pieces = []
            for q in range(n):
                before = int(sum(per[s][q] for s in range(p)))
                pieces.append(ys[q][before:before + int(per[p][q])])
            backs.append(torch.cat(pieces))
        e5.record(stream)
        outs = [layers[p].ep_combine(backs[p]) for p in range(n)]
        e6 = ev()
        e6.record(stream)
        torch.cuda.synchronize(dev)
        if it >= 3:
            acc["dispatch"] += e0.elapsed_time(e1)
            acc["exchange"] += e2.elapsed_time(e3) + e4.elapsed_time(e5)
            acc["experts"] += e3.elapsed_time(e4)
            acc["combine"] += e5.elapsed_time(e6)
            rows_recv = sum(int(r.shape[0]) for r in recv)
    status = max(L.device_status() for L in layers)
    for L in layers:
        L.close()
    us = {k: v / steps * 1e3 for k, v in acc.items()}  # all ranks, per step
    return {"ranks": n, "tokens_per_rank": T, "experts_per_rank": El, "rows_exchanged_per_step": rows_recv,
            "us_per_step_all_ranks": us,
            "us_per_rank_compute": (us["dispatch"] + us["experts"] + us["combine"]) / n,
            "steps": steps, "device_status": status,
            "note": "ranks emulated one after another on this GPU; the exchange as device copies (NCCL unmeasured)"}


def run_ep(args, shape, T):
    """--ep: one expert-parallel step per iteration on every rank (ep_dispatch, count and row
    all-to-alls, ep_experts, all-to-all back, ep_combine), each rank with its own T tokens (weak
    scaling).  Without torchrun it runs as a one-rank group (the exchange is then NCCL to itself)."""
    import socket
    import torch
    import torch.distributed as dist
    import testgen
    import mixture_experts_gemm_gb300 as moe
    from mixture_experts_gemm_gb300 import ep
    from moe_check import host_weights, torch_from_bits
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if "MASTER_ADDR" in os.environ:
        dist.init_process_group(backend="nccl", device_id=dev)
    else:
        with socket.socket() as so:
            so.bind(("127.0.0.1", 0))
            port = so.getsockname()[1]
        dist.init_process_group(backend="nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                                device_id=dev)
    if shape.num_experts % world or shape.shared_expert or shape.dtype != "bf16":
        raise SystemExit("--ep needs E divisible by the number of ranks, bf16 and no shared expert")
    li = testgen.make_inputs(shape.with_T(T * world), want_f32=False)
    El = shape.num_experts // world
    layer = moe.MoELayer(shape.d_model, shape.d_ff, shape.num_experts, T, dtype="bf16",
                         act="swiglu" if shape.act == testgen.ACT_SWIGLU else "relu_bias",
                         has_router_bias=shape.zipf_router_bias, out_dtype="f32", device=local, top_k=shape.top_k,
                         gate_mode=shape.gate_mode, ep_rank=rank, ep_size=world)
    w = host_weights(li)
    own = lambda lst: None if lst is None else [t if rank * El <= e < (rank + 1) * El else None
                                                for e, t in enumerate(lst)]
    layer.load_weights(w["w_router"], own(w["w1"]), own(w["w2"]), w3=own(w["w3"]), b_router=w["b_router"],
                       b1=own(w["b1"]), b2=own(w["b2"]))
    x = torch_from_bits(li.x_bits)[rank * T:(rank + 1) * T].contiguous().to(dev)
    backend = ep.LayerEP(layer)
    for _ in range(max(3, args.warmup)):
        ep.ep_forward(backend, x)
    stream = torch.cuda.current_stream(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(args.steps):
        ep.ep_forward(backend, x)
    b.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    status = layer.device_status()
    layer.close()
    if rank == 0:
        line = {"metric": METRIC, "value": whole_job_rate(world, T, args.steps, ms / 1e3), "unit": UNIT,
                "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
                "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": workload_desc(shape, T), "tokens_per_step_per_gpu": T,
                           "parallelism": f"expert parallel x{world} ({El} experts per GPU, NCCL all-to-alls)"},
                "gpu_launches": args.steps * 7, "device_status": status}
        print(json.dumps(line), flush=True)
    dist.destroy_process_group()


def main():
    args = parse_args()
    import dataclasses
    import testgen
    shape = testgen.CONFIGS[args.workload]
    if args.top_k is not None or args.gate_mode is not None or args.shared_expert:
        shape = dataclasses.replace(shape, top_k=args.top_k or shape.top_k,
                                    gate_mode=shape.gate_mode if args.gate_mode is None else args.gate_mode,
                                    shared_expert=args.shared_expert or shape.shared_expert)
    T = args.T if args.T is not None else shape.T
    if args.impl == "reference":
        run_reference(args, shape, T)
        return
    if args.ep:
        run_ep(args, shape, T)
        return

    import numpy as np
    import torch
    import torch.distributed as dist
    from moe_check import host_weights, x_device
    import mixture_experts_gemm_gb300 as moe

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def barrier():
        if world > 1:
            dist.barrier()

    # inputs: the layer's weights and one batch of T tokens, generated on the host, copied to HBM
    li = testgen.make_inputs(shape.with_T(T), want_f32=shape.dtype == "f32")
    layer = moe.MoELayer(shape.d_model, shape.d_ff, shape.num_experts, T, dtype=shape.dtype,
                         act="swiglu" if shape.act == testgen.ACT_SWIGLU else "relu_bias",
                         has_router_bias=shape.zipf_router_bias, out_dtype="f32", device=local, top_k=shape.top_k,
                         gate_mode=shape.gate_mode, shared_expert=shape.shared_expert)
    layer.load_weights(**host_weights(li))
    x = x_device(li).to(dev)
    out = torch.empty((T, shape.d_model), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    n_st = layer.num_stages()

    for _ in range(max(3, args.warmup)):
        layer.forward_ptr(x.data_ptr(), out.data_ptr(), T, sh)
    torch.cuda.synchronize(dev)
    routing = layer.get_routing(T)
    counts = routing["counts"].cpu().numpy()
    active = int((counts > 0).sum())

    import ctypes
    lib = moe.lib()

    def event_array(evs):
        for e in evs:
            if e is not None:
                e.record(stream)  # makes torch create the underlying cudaEvent_t
        return (ctypes.c_void_p * (n_st + 1))(*[None if e is None else e.cuda_event for e in evs])

    # 1) stage breakdown: a short pass with an event at every stage boundary
    n_prof = min(args.steps, 50)
    prof_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(n_st + 1)] for _ in range(n_prof)]
    prof_arrs = [event_array(evs) for evs in prof_sets]
    torch.cuda.synchronize(dev)
    for k in range(n_prof):
        lib.colibri_moe_set_stage_events(layer._h, ctypes.cast(prof_arrs[k], ctypes.c_void_p), n_st + 1)
        layer.forward_ptr(x.data_ptr(), out.data_ptr(), T, sh)
    torch.cuda.synchronize(dev)
    stage_ms = np.array([[evs[i].elapsed_time(evs[i + 1]) for i in range(n_st)] for evs in prof_sets])
    step_ms_prof = np.array([evs[0].elapsed_time(evs[n_st]) for evs in prof_sets])
    dominant = int(np.argmax(stage_ms.mean(axis=0)))

    # 2) the timed region: K back-to-back forwards; events around the dominant kernel on every
    # DOM_EVERY-th step only (an event between two kernels ends their programmatic-launch overlap,
    # which costs a few microseconds per step on decode-sized batches)
    dom_steps = list(range(0, args.steps, DOM_EVERY))
    dom_sets = [[torch.cuda.Event(enable_timing=True) if i in (dominant, dominant + 1) else None
                 for i in range(n_st + 1)] for _ in dom_steps]
    dom_arrs = [event_array(evs) for evs in dom_sets]
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for k in range(args.steps):
        if k % DOM_EVERY == 0:
            lib.colibri_moe_set_stage_events(layer._h, ctypes.cast(dom_arrs[k // DOM_EVERY], ctypes.c_void_p),
                                             n_st + 1)
        elif k % DOM_EVERY == 1:
            lib.colibri_moe_set_stage_events(layer._h, None, 0)
        layer.forward_ptr(x.data_ptr(), out.data_ptr(), T, sh)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    kernels_per_step = layer.last_kernel_count()  # (later legs run other batch sizes on this layer)
    gemm_form = layer.last_gemm()
    both_in_one = gemm_form in ("decode_fused", "weight_major_fused")  # one launch, both projections
    lib.colibri_moe_set_stage_events(layer._h, None, 0)
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    dom_ms = np.array([evs[dominant].elapsed_time(evs[dominant + 1]) for evs in dom_sets])
    ms_per_step = ms_total / args.steps
    value = whole_job_rate(world, T, args.steps, ms_total / 1e3)

    # end to end through the C ABI with host buffers (pinned): every step copies its x host->device,
    # runs the forward and copies out device->host; forward_host_async overlaps one step's copies
    # with the neighbouring steps' forwards (three staging slots), host_sync ends the timed region
    e2e = None
    if not args.no_e2e:
        if shape.dtype == "bf16":
            from moe_check import torch_from_bits
            xh = torch_from_bits(li.x_bits).pin_memory()
        else:
            xh = torch.from_numpy(li.x_f32).pin_memory()
        oh = torch.empty((T, shape.d_model), dtype=torch.float32).pin_memory()
        for _ in range(3):
            layer.forward_host(xh, oh, stream)
        k_e2e = max(1, min(args.steps, 100))
        barrier()
        t0 = time.perf_counter()
        for _ in range(k_e2e):
            layer.forward_host_async(xh, oh, stream)
        layer.host_sync()
        el = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": whole_job_rate(world, T, k_e2e, el), "unit": UNIT,
               "h2d_bytes_per_step": xh.numel() * xh.element_size(),
               "d2h_bytes_per_step": oh.numel() * oh.element_size(),
               "mode": "colibri_moe_forward_host_async: three staging slots; the copies of step i overlap the forwards of the steps around it"}
    clk = clocks.stop()
    status = layer.device_status()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    alg = algorithmic(shape, T, active)
    peaks, peak_src = load_peaks()
    mean_stage = stage_ms.mean(axis=0)
    dur = float(dom_ms.mean()) / 1e3  # live, inside the timed region
    timed_note = f"CUDA events around the kernel on {len(dom_steps)} of the {args.steps} timed steps"
    # the binding roofline follows the layer's arithmetic intensity against the ridge point of the
    # measured peaks: tensor above it, HBM over the active experts' weights below it
    ridge = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])) * 1e12 / \
        (float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])) * 1e9)
    tensor_bound = alg["flops"] / alg["bytes"] > ridge
    if shape.dtype == "bf16" and tensor_bound and dominant in (2, 3):
        fl = alg["flops_up"] + alg["flops_down"] if both_in_one else \
            (alg["flops_up"] if dominant == 2 else alg["flops_down"])
        ach = fl / dur / 1e12
        burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        # the peak that fits the timed region: the burst rate for a region shorter than a second (the
        # GPU has not settled at its power cap yet), the sustained rate for a longer loop
        region_s = ms_total / 1e3
        long_region = region_s >= SUSTAINED_AFTER_S
        peak = sustained if long_region else burst
        gemm = {"single_cta": "1sm", "weight_major_fused": "1kernel"}.get(gemm_form, "2sm")
        roof = {"bound": "tensor", "kernel": STAGES[dominant] + (" (both projections, one launch)" if both_in_one else ""),
                "gemm_form": gemm_form, "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": NCU_TRAFFIC.get((shape.name, T, STAGES[dominant], gemm)),
                "peak_source": (f"{peak_src} bf16 {'sustained' if long_region else 'burst'}: timed region "
                                f"{region_s:.3f} s {'>=' if long_region else '<'} {SUSTAINED_AFTER_S:.0f} s"),
                "frac_of_burst": ach / burst, "frac_of_sustained": ach / sustained,
                "frac_of_nominal": ach / NOMINAL_BF16_TFLOPS,
                "nominal_note": f"frac_of_nominal: against the {NOMINAL_BF16_TFLOPS:.0f} TFLOP/s dense bf16 datasheet rate",
                "algorithmic_flops_per_launch": fl, "dominant_ms": dur * 1e3, "timing": timed_note,
                "layer_tflops": alg["flops"] / (ms_per_step / 1e3) / 1e12,
                "layer_frac": alg["flops"] / (ms_per_step / 1e3) / 1e12 / peak}
    else:
        # weight streaming: bytes of the distinct active experts' weights this stage reads
        n_up = 2 if shape.act == 1 else 1
        es = 2 if shape.dtype == "bf16" else 4
        n_w = active + int(shape.shared_expert)
        byts = {2: n_w * n_up * shape.d_model * shape.d_ff * es,
                3: n_w * shape.d_model * shape.d_ff * es}.get(dominant, alg["bytes"])
        if both_in_one:  # one kernel streams both projections' weights: the cooperative decode
            # kernel, or the fused weight-major GEMM
            byts = n_w * (n_up + 1) * shape.d_model * shape.d_ff * es
        ach = byts / dur / 1e9
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        path = "1kernel" if both_in_one else {"single_cta": "1sm"}.get(gemm_form, "2sm")
        roof = {"bound": "hbm", "kernel": STAGES[dominant] + (" (both projections, one launch)" if both_in_one else ""),
                "gemm_form": gemm_form, "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak, "traffic": NCU_TRAFFIC.get((shape.name, T, STAGES[dominant], path)),
                "peak_source": f"{peak_src} copy", "algorithmic_bytes_per_launch": byts,
                "dominant_ms": dur * 1e3, "frac_of_nominal": ach / NOMINAL_HBM_GBS,
                "step_frac_of_hbm": alg["bytes"] / (ms_per_step / 1e3) / 1e9 / peak, "timing": timed_note}

    roof["layer_flop_per_byte"] = alg["flops"] / alg["bytes"]
    roof["ridge_flop_per_byte"] = ridge

    extra = {}
    if not args.no_extra and world == 1 and args.impl == "ours":
        peaks_x, _ = load_peaks()
        n_x = max(50, min(args.steps, 200))
        if shape.name == "mixtral-prefill" and shape.top_k == 2 and not shape.shared_expert and shape.gate_mode == 0:
            extra["decode"] = decode_sweep(layer, shape, x, out, stream,
                                           float(peaks_x.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])), n_x)
        extra["workloads"] = other_workloads(peaks_x, n_x, local)
        if shape.name == "mixtral-prefill" and shape.top_k == 2 and not shape.shared_expert and shape.gate_mode == 0:
            extra["ep"] = ep_phases(li, shape, x, 20, local)

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        li32 = li if li.x_f32 is not None and (li.w1_f32 and li.w1_f32[0] is not None) else \
            testgen.make_inputs(shape.with_T(T), want_bits=False)
        rate, n, wall, used = oracle_rate(li32, T, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": used, "kind": "oracle",
               "sample": f"{n} random tokens of the {T}-token batch: fp64 routing + both experts, {wall:.1f} s"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": shape.dtype, "data": "synthetic",
        "config": {"workload": workload_desc(shape, T), "tokens_per_step_per_gpu": T,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2: {alg['bytes'] / 1e9:.2f} GB of weights and activations per step",
                   "active_experts": active},
        "tflops": alg["flops"] / (ms_per_step / 1e3) / 1e12,
        "roofline": roof,
        "stages_us": {n: float(v * 1e3) for n, v in zip(STAGES, mean_stage)},
        "stages_note": "stage split from a separate 50-step pass with an event at every stage boundary",
        "spread_us": {
            "step_p10": float(np.percentile(step_ms_prof, 10) * 1e3),
            "step_p50": float(np.percentile(step_ms_prof, 50) * 1e3),
            "step_p90": float(np.percentile(step_ms_prof, 90) * 1e3),
            "dominant_p10": float(np.percentile(dom_ms, 10) * 1e3),
            "dominant_p50": float(np.percentile(dom_ms, 50) * 1e3),
            "dominant_p90": float(np.percentile(dom_ms, 90) * 1e3),
            "note": "step: per-step times of the stage pass (50 steps with an event at every stage boundary, "
                    "which ends the programmatic-launch overlap between kernels: a few microseconds per kernel; "
                    "it runs before the timed region, so at a cooler clock it can also come out below "
                    "ms_per_step); dominant: the kernel timed for the roofline, inside the timed region"},
        "e2e": e2e,
        "gpu_launches": args.steps * kernels_per_step,
        "clocks": clk,
        "cpu_baseline": cpu,
        "device_status": status,
    }
    if extra:
        line["decode"] = extra.get("decode")
        line["workloads"] = extra.get("workloads")
        line["ep"] = extra.get("ep")
        line["extra_note"] = ("decode: the Mixtral-shaped layer's weights on the first T rows of the batch, HBM "
                              "fraction over the distinct active experts' weights; workloads: the other layers' "
                              "step times; ep: the expert-parallel calls on two emulated ranks; all timed after "
                              "the main region with CUDA events")
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
