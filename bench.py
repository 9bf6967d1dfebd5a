#!/usr/bin/env python3
"""Stable LatentMoE layer forward throughput on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lmoe|reference]
                    [--workload NAME] [--cpu-tokens T] [--no-cpu-baseline]

One step = one lmoe_forward (router GEMM, cutoffs, top-K, segments, W_down, grouped
expert gate/up + SiTU-GLU, expert down, RMSNorm + combine, shared experts, W_up +
shared down) over one synthetic batch already resident in HBM.  Prints one JSON line
(rank 0).  N > 1 (torchrun) runs N independent replicas, one per GPU, each with its own
batch: the cutoffs are per batch, so the layer has no data-parallel exchange step.

--impl reference times the fp64 CPU oracle on the host cores instead (each step a
bounded sample of the same workload); it is a deliberately slow correctness program."""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import FFN_WORKLOADS, WORKLOADS, make_ffn_inputs, make_inputs, make_x  # noqa: E402

DEFAULT_WORKLOAD = "full_prefill_bt8192"
METRIC = "LatentMoE layer fwd tokens/s on 1 B300; % of bf16 TC peak (or HBM BW)"


# ----------------------------------------------------------------------------- arithmetic

def algorithmic(shape, bt, n_touched, fp8_experts=False, mxfp4_experts=False):
    """Algorithmic FLOPs and bytes of one layer call and of each stage (2*M*N*K per GEMM;
    bytes = what each stage must read and write at least once).  n_touched = experts
    with at least one token.  For the routed-expert GEMMs the bytes are the touched experts'
    weights only, the per-expert unit of the layer's byte count: their token rows and
    activations are intermediates of the layer (implementation traffic, which the measured
    DRAM traffic shows on top).  With fp8 experts the weights are one byte per value plus
    4-byte row scales; with MXFP4 experts half a byte per value plus one scale byte per 32
    values (17/32 byte per value)."""
    d, L, E, K, I, S, Is = (shape.d, shape.latent, shape.n_experts, shape.top_k, shape.expert_inter,
                            shape.n_shared, shape.shared_inter)
    b = 2 if shape.dtype == "bf16" else 4
    if fp8_experts or mxfp4_experts:
        # per value, per output row
        ev, er = (17 / 32, 0) if mxfp4_experts else (1, 4)
        st = {
            "router_gemm": (2 * bt * E * d, (bt * d + E * d) * b + 2 * bt * E * 4),
            "cutoff_topk_segments": (0, 2 * bt * E * 4 + bt * K * 16),
            "w_down_gemm": (2 * bt * L * d, (bt * d + L * d + bt * L) * b),
            "token_gather": (0, bt * L * b + 2 * bt * L + bt * K * L),
            "expert_gate_up_gemm": (2 * bt * K * 2 * I * L, n_touched * 2 * I * (L * ev + er)),
            "expert_down_gemm": (2 * bt * K * L * I, n_touched * L * (I * ev + er)),
            "rmsnorm_combine": (0, (bt * K * L + bt * L) * b + bt * K * 8),
            "shared_gate_up_gemm": (2 * bt * S * 2 * Is * d, (S * 2 * Is * d + bt * d + bt * S * Is) * b),
            "up_shared_down_gemm": (2 * bt * d * (L + S * Is), (d * (L + S * Is) + bt * (L + S * Is) + bt * d) * b),
        }
        flops = 2 * bt * (E * d + L * d + K * 3 * L * I + d * L + S * 3 * d * Is)
        weight_bytes = (E * d + 2 * L * d + L + S * 3 * d * Is) * b + n_touched * 3 * L * I * ev + n_touched * (2 * I + L) * er
        return flops, weight_bytes + 2 * bt * d * b, st
    st = {
        "router_gemm": (2 * bt * E * d, (bt * d + E * d) * b + 2 * bt * E * 4),
        "cutoff_topk_segments": (0, 2 * bt * E * 4 + bt * K * 16),
        "w_down_gemm": (2 * bt * L * d, (bt * d + L * d + bt * L) * b),
        "token_gather": (0, (bt * L + bt * K * L) * b),
        "expert_gate_up_gemm": (2 * bt * K * 2 * I * L, n_touched * 2 * I * L * b),
        "expert_down_gemm": (2 * bt * K * L * I, n_touched * L * I * b),
        "rmsnorm_combine": (0, (bt * K * L + bt * L) * b + bt * K * 8),
        "shared_gate_up_gemm": (2 * bt * S * 2 * Is * d, (S * 2 * Is * d + bt * d + bt * S * Is) * b),
        "up_shared_down_gemm": (2 * bt * d * (L + S * Is), (d * (L + S * Is) + bt * (L + S * Is) + bt * d) * b),
    }
    flops = 2 * bt * (E * d + L * d + K * 3 * L * I + d * L + S * 3 * d * Is)
    weight_bytes = (E * d + 2 * L * d + L + n_touched * 3 * L * I + S * 3 * d * Is) * b
    layer_bytes = weight_bytes + 2 * bt * d * b
    return flops, layer_bytes, st


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return dict(hbm=j["hbm_gbs"], tc=j["bf16_tflops"], tc_sustained=j["bf16_tflops_sustained"],
                    source="measured")
    print("bench.py: MEASURED_PEAKS.json not found; roofline fractions use the fallback peaks "
          "(6400 GB/s, 1800 / 1400 TFLOP/s) and say so in peak_source", file=sys.stderr, flush=True)
    return dict(hbm=6400.0, tc=1800.0, tc_sustained=1400.0, source="fallback")


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons of this process's GPU, sampled every 100 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        pr = torch.cuda.get_device_properties(device)
        self.bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        self.proc = None
        self.path = None

    def start(self):
        try:
            self.path = f"/tmp/lmoe_clocks_{os.getpid()}.csv"
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.bus, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(v):
            try:
                return float(v)
            except ValueError:
                return float("nan")
        sm = [num(r[0]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(num(r[1]) for r in rows),
                "power_w_max": max(num(r[2]) for r in rows), "samples": len(rows),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- distributed

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(v: float, ws: int, device) -> float:
    if ws == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v: float, ws: int, device) -> float:
    if ws == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle

def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        n = [i.get("num_threads", 0) for i in info if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def oracle_sample_time(w, x, weights, bias, n_tokens: int, offset: int = 0):
    """Wall time of the fp64 oracle on n_tokens tokens of the batch (routing over those
    tokens, then the layer), fetching each needed expert's weights from device memory
    and upcasting them as it goes (the oracle's weight source)."""
    from oracle import lmoe_oracle as O

    class PerIndex:
        def __init__(self, t):
            self.t = t

        def __getitem__(self, i):
            return self.t[int(i)].cpu().to(torch.float64).numpy()

        def __len__(self):
            return self.t.shape[0]

    bt = x.shape[0]
    rows = (np.arange(n_tokens) * max(1, bt // n_tokens) + offset) % bt
    xs = x[torch.as_tensor(rows, device=x.device)].cpu().to(torch.float64).numpy()
    t0 = time.perf_counter()
    W = {k: (PerIndex(v) if v.dim() == 3 else v.cpu().to(torch.float64).numpy()) for k, v in weights.items()}
    b = None if bias is None else bias.cpu().to(torch.float64).numpy()
    s = w.shape
    O.forward(xs, W, s.top_k, router_bias=b, beta=s.beta, beta_u=s.beta_u, eps=s.rms_eps)
    return time.perf_counter() - t0


# ----------------------------------------------------------------------------- traffic record

def kernel_traffic(stage: str, workload: str, experts: str):
    """DRAM bytes per launch of `stage` from the committed ncu summary, if it was scaled to this
    workload and expert format and the kernel source it was taken from is unchanged (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(stage)
    if not rec or rec.get("workload") != workload or rec.get("experts") != experts:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src) or hashlib.sha1(open(src, "rb").read()).hexdigest() != rec["source_sha1"]:
        return None
    return rec["dram_bytes_per_launch"]


# ----------------------------------------------------------------------------- main

def run_reference(args, ws, rank):
    """The oracle as the reference arm: rank 0 only."""
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    device = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    x, weights, bias = make_inputs(w, device)
    n = args.cpu_tokens_ref
    for i in range(args.warmup):
        oracle_sample_time(w, x, weights, bias, n, offset=i)
    total = 0.0
    for i in range(args.steps):
        total += oracle_sample_time(w, x, weights, bias, n, offset=args.warmup + i)
    value = n * args.steps / total
    cores = _blas_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "bt": w.bt, "d": w.shape.d, "latent": w.shape.latent,
                       "n_experts": w.shape.n_experts, "top_k": w.shape.top_k,
                       "expert_inter": w.shape.expert_inter, "n_shared": w.shape.n_shared,
                       "shared_inter": w.shape.shared_inter, "parallelism": "single process, host cores"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} tokens of the batch per step (routing over the sample), "
                                       "expert weights fetched from HBM and upcast inside the timing"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ffn(args, ws, rank, local):
    """The dense first-layer SiTU-GLU FFN (out = W_down act(W_gate x, W_up x)) through
    lmoe_ffn_forward: same timing rules as the layer; the reference arm times the oracle."""
    from oracle import lmoe_oracle as O

    w = FFN_WORKLOADS[args.workload]
    flops = 2 * w.bt * 3 * w.d * w.inter
    metric = "dense SiTU-GLU FFN fwd tokens/s on 1 B300"
    cfg = {"workload": w.name, "bt": w.bt, "d": w.d, "inter": w.inter, "global_batch": w.bt * ws,
           "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"}
    if args.impl == "reference":
        if rank != 0:
            return 0
        x, wg, wu, wd = make_ffn_inputs(w, "cuda" if torch.cuda.is_available() else "cpu", 8)
        W = [t.cpu().to(torch.float64).numpy() for t in (wg, wu, wd)]
        xs = x.cpu().to(torch.float64).numpy()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            O.dense_ffn(xs[:2], *W, w.beta, w.beta_u)
        dt = time.perf_counter() - t0
        value = 2 * args.steps / dt
        print(json.dumps({"impl": "reference", "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": cfg,
                          "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _blas_threads(),
                                           "kind": "oracle", "sample": "2 tokens per step"},
                          "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    from sparse_moe_layer_cutoff_b300 import DenseFFN

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    x, wg, wu, wd = make_ffn_inputs(w, device)
    ffn = DenseFFN(w.d, w.inter, wg, wu, wd, max_bt=w.bt, beta=w.beta, beta_u=w.beta_u)
    out = torch.empty((w.bt, w.d), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        ffn.forward(x, out)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        ffn.forward(x, out)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(ws)
    if ffn.sync_status() != 0:
        raise RuntimeError("device status set in the timed region")
    ms = max_over_ranks(e0.elapsed_time(e1), ws, device)
    value = sum_over_ranks(float(w.bt * args.steps), ws, device) / (ms / 1e3)
    step_s = ms / 1e3 / args.steps
    pk = peaks()
    tc_peak = pk["tc_sustained"] if ms / 1e3 > 2.0 else pk["tc"]
    achieved = flops / step_s / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved / tc_peak,
            "traffic": None, "kernel": "dense_ffn (SiTU-GLU + down)", "ms_per_launch": step_s * 1e3,
            "algorithmic_flops": flops,
            "peak_source": pk["source"] + (" sustained" if ms / 1e3 > 2.0 else " burst")}
    xh = x.cpu().pin_memory()
    oh = torch.empty((w.bt, w.d), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(x)
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.e2e_steps):
        xd.copy_(xh, non_blocking=True)
        ffn.forward(xd, out)
        oh.copy_(out, non_blocking=True)
    e3.record(stream)
    torch.cuda.synchronize()
    e2e = w.bt * args.e2e_steps / (e2.elapsed_time(e3) / 1e3)
    if rank == 0:
        print(json.dumps({"metric": metric, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
                          "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                          "config": cfg, "roofline": roof, "cpu_baseline": None,
                          "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": w.bt * w.d * 2,
                                  "d2h_bytes_per_step": w.bt * w.d * 2},
                          "gpu_launches": 2 * args.steps, "clocks": clk}), flush=True)
    ffn.close()
    return 0


def time_forwards(layer, xs, out, steps, warmup, local, ws):
    """W untimed forwards, then K forwards timed with CUDA events on the launch stream
    (synchronised and barriered on both sides), with the per-stage record and a clock
    sample over the timed region.  Returns (local ms, stage ms summed, calls, launches, clocks)."""
    from sparse_moe_layer_cutoff_b300.lmoe import lmoe_profile, lmoe_profile_read

    stream = torch.cuda.current_stream()
    for i in range(warmup):
        layer.forward(xs[i % len(xs)], out)
    torch.cuda.synchronize()
    if layer.sync_status() != 0:
        raise RuntimeError("device status set during warm-up")
    clocks = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize()
    lmoe_profile(layer.ctx, True)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        layer.forward(xs[i % len(xs)], out)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    lmoe_profile(layer.ctx, False)
    barrier(ws)
    st, stage_ms, calls, launches = lmoe_profile_read(layer.ctx)
    status = layer.sync_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    return e0.elapsed_time(e1), stage_ms, calls, launches, clk


def routing_stats(layer, xs):
    """Experts touched (for the algorithmic byte count) and the load range, from the route of
    each batch."""
    touched, load_max, load_min = [], [], []
    for xb in xs:
        c = layer.route(xb)["counts"]
        touched.append(int((c > 0).sum().item()))
        load_max.append(int(c.max().item()))
        load_min.append(int(c.min().item()))
    return sum(touched) / len(touched), max(load_max), min(load_min)


def layer_fractions(shape, bt, n_touched, step_s, pk, fp8_experts=False, mxfp4_experts=False):
    """The layer's achieved TFLOP/s and GB/s and their fractions of the measured bf16 tensor and
    HBM peaks; `bound` is the roof that binds (the larger of the two ideal times) and `frac`
    the fraction of that roof."""
    flops, layer_bytes, _ = algorithmic(shape, bt, n_touched, fp8_experts=fp8_experts, mxfp4_experts=mxfp4_experts)
    tc_frac = flops / step_s / 1e12 / pk["tc"]
    hbm_frac = layer_bytes / step_s / 1e9 / pk["hbm"]
    bound = "tensor" if flops / (pk["tc"] * 1e12) > layer_bytes / (pk["hbm"] * 1e9) else "hbm"
    return {"tflops": flops / step_s / 1e12, "tc_frac": tc_frac, "gbs": layer_bytes / step_s / 1e9,
            "hbm_frac": hbm_frac, "bound": bound, "frac": tc_frac if bound == "tensor" else hbm_frac,
            "algorithmic_flops": flops, "algorithmic_bytes": layer_bytes, "experts_touched": n_touched}


def extra_workload(name, weights, steps, warmup, local, ws, device, pk, experts="bf16"):
    """One more line of the layer on the bench's weights: the named workload's token batch (its
    own seed, and for the skewed one the Zipf logit bias and the repeated-token block), timed
    as the headline is; experts "fp8" / "mxfp4" quantize the routed experts first (the
    quantization is not timed).  Returns a dict for the JSON line."""
    from sparse_moe_layer_cutoff_b300 import LatentMoE
    from sparse_moe_layer_cutoff_b300.lmoe import quantize_experts_fp8, quantize_experts_mxfp4
    from workloads import make_bias

    w = WORKLOADS[name]
    s = w.shape
    lowp = {}
    if experts == "fp8":
        lowp["fp8_experts"] = quantize_experts_fp8(weights)
    elif experts == "mxfp4":
        lowp["mxfp4_experts"] = quantize_experts_mxfp4(weights)
    layer = LatentMoE(s, weights, max_bt=w.bt, router_bias=make_bias(w, device), **lowp)
    xs = [make_x(w, device), make_x(w, device, seed_offset=1)]
    out = torch.empty((w.bt, s.d), dtype=layer.dtype, device=device)
    n_touched, lmax, lmin = routing_stats(layer, xs)
    ms, stage_ms, calls, launches, clk = time_forwards(layer, xs, out, steps, warmup, local, ws)
    layer.close()
    del xs, out, lowp, layer
    torch.cuda.empty_cache()
    step_s = ms / 1e3 / steps
    fr = layer_fractions(s, w.bt, n_touched, step_s, pk, fp8_experts=experts == "fp8",
                         mxfp4_experts=experts == "mxfp4")
    return {"workload": w.name, "experts": experts, "bt": w.bt, "steps": steps, "warmup": warmup,
            "ms_per_step": ms / steps,
            "tokens_s": w.bt / step_s, "tc_frac": fr["tc_frac"], "hbm_frac": fr["hbm_frac"],
            "bound": fr["bound"], "frac": fr["frac"], "experts_touched": n_touched,
            "expert_load": {"max": lmax, "min": lmin, "target": w.bt * s.top_k / s.n_experts},
            "stage_ms_per_step": {k: v / max(calls, 1) for k, v in stage_ms.items()},
            "gpu_launches": launches, "clocks": clk,
            "inputs": "the headline's weights" +
                      ("" if experts == "bf16" else f" (routed experts quantized to {experts}, not timed)") +
                      "; x drawn with this workload's seed" +
                      (", Zipf(1.1) logit bias and 25 % identical tokens" if w.zipf_bias else "")}


# extra figures of the default line: (JSON key, workload, routed-expert format)
EXTRA_WORKLOADS = (("decode_bt64", "full_decode_bt64", "bf16"), ("skewed_bt16384", "full_skewed_bt16384", "bf16"),
                   ("decode_bt64_fp8_experts", "full_decode_bt64", "fp8"),
                   ("decode_bt64_mxfp4_experts", "full_decode_bt64", "mxfp4"))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="lmoe", choices=["lmoe", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS) + sorted(FFN_WORKLOADS))
    ap.add_argument("--cpu-tokens", type=int, default=12, help="oracle sample for cpu_baseline")
    ap.add_argument("--cpu-tokens-ref", type=int, default=2, help="oracle sample per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None, help="default: --steps")
    ap.add_argument("--fp8-experts", action="store_true",
                    help="routed experts in e4m3 (lmoe_create_fp8); a separate line, not the bf16 headline")
    ap.add_argument("--mxfp4-experts", action="store_true",
                    help="routed experts in MXFP4 (lmoe_create_mxfp4); a separate line, not the bf16 headline")
    ap.add_argument("--bt", type=int, default=None,
                    help="tokens per step instead of the workload's (same shape and recipe); a separate line")
    ap.add_argument("--latent-norm", default="expert", choices=["expert", "combined"],
                    help="latent RMSNorm placement; 'combined' (one norm of the weighted sum) is a separate line")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the extra figures of the default line (64-token decode with bf16, e4m3 and MXFP4 experts; 16384-token skewed forward)")
    args = ap.parse_args(argv)
    if args.e2e_steps is None:
        args.e2e_steps = args.steps
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.fp8_experts and args.mxfp4_experts:
        ap.error("--fp8-experts and --mxfp4-experts are exclusive")
    lowp = args.fp8_experts or args.mxfp4_experts
    ws, rank, local = dist_setup()
    if args.workload in FFN_WORKLOADS:
        return run_ffn(args, ws, rank, local)
    if args.impl == "reference":
        rc = run_reference(args, ws, rank)
        barrier(ws)
        return rc

    from sparse_moe_layer_cutoff_b300 import LatentMoE
    from sparse_moe_layer_cutoff_b300.lmoe import lmoe_build_info

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    if args.bt is not None:
        if args.bt <= 0:
            ap.error("--bt must be positive")
        w = w.with_(bt=args.bt, name=f"{w.name} at bt={args.bt}")
    s = w.shape
    x, weights, bias = make_inputs(w, device)
    xs = [x, make_x(w, device, seed_offset=1 + rank)]
    if args.fp8_experts:
        from sparse_moe_layer_cutoff_b300.lmoe import quantize_experts_fp8
        f8 = quantize_experts_fp8(weights)
        for n in ("exp_gate", "exp_up", "exp_down"):
            del weights[n]
        torch.cuda.empty_cache()
        layer = LatentMoE(s, weights, max_bt=w.bt, router_bias=bias, fp8_experts=f8)
    elif args.mxfp4_experts:
        from sparse_moe_layer_cutoff_b300.lmoe import quantize_experts_mxfp4
        mx = quantize_experts_mxfp4(weights)
        for n in ("exp_gate", "exp_up", "exp_down"):
            del weights[n]
        torch.cuda.empty_cache()
        layer = LatentMoE(s, weights, max_bt=w.bt, router_bias=bias, mxfp4_experts=mx)
    else:
        layer = LatentMoE(s, weights, max_bt=w.bt, router_bias=bias)
    if args.latent_norm != "expert":
        layer.set_latent_norm(args.latent_norm)
    out = torch.empty((w.bt, s.d), dtype=layer.dtype, device=device)
    stream = torch.cuda.current_stream(device)

    n_touched, load_max, load_min = routing_stats(layer, xs)
    ms_local, stage_ms, calls, launches, clk = time_forwards(layer, xs, out, args.steps, args.warmup, local, ws)
    ms = max_over_ranks(ms_local, ws, device)
    tokens_all = sum_over_ranks(float(w.bt * args.steps), ws, device)
    value = tokens_all / (ms / 1e3)

    # ---- roofline of the dominant kernel (largest share of the timed region)
    pk = peaks()
    flops, layer_bytes, per_stage = algorithmic(s, w.bt, n_touched, fp8_experts=args.fp8_experts,
                                                mxfp4_experts=args.mxfp4_experts)
    dom = max(stage_ms, key=lambda k: stage_ms[k])
    dom_ms = stage_ms[dom] / max(calls, 1)
    f, b = per_stage[dom]
    long_step = ms / 1e3 > 2.0
    tc_peak = pk["tc_sustained"] if long_step else pk["tc"]
    # the e4m3 (and e2m1 x e4m3) expert GEMMs take the fp8 peak: the measured bf16 peak x the
    # nominal fp8 / bf16 dense ratio (4.5 / 2.25 PFLOP/s)
    f8_kernel = lowp and dom in ("expert_gate_up_gemm", "expert_down_gemm")
    if f8_kernel:
        tc_peak *= 2.0
    if f / (tc_peak * 1e12) > b / (pk["hbm"] * 1e9):
        roof = {"bound": "tensor", "achieved": f / (dom_ms / 1e3) / 1e12, "peak": tc_peak, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": b / (dom_ms / 1e3) / 1e9, "peak": pk["hbm"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = kernel_traffic(dom, w.name, "fp8" if args.fp8_experts else "mxfp4" if args.mxfp4_experts else "bf16")
    roof.update({"kernel": dom, "ms_per_launch": dom_ms, "algorithmic_flops": f, "algorithmic_bytes": b,
                 "peak_source": pk["source"] + (" sustained" if (roof["bound"] == "tensor" and long_step) else
                                                " burst" if roof["bound"] == "tensor" else "")
                 + (" bf16 x 2 (nominal fp8 / bf16 ratio)" if (roof["bound"] == "tensor" and f8_kernel) else "")})
    step_s = ms / 1e3 / args.steps
    layer_roof = layer_fractions(s, w.bt, n_touched, step_s, pk, fp8_experts=args.fp8_experts,
                                 mxfp4_experts=args.mxfp4_experts)
    layer_roof["expert_load"] = {"max": load_max, "min": load_min, "target": w.bt * s.top_k / s.n_experts}

    # ---- end to end through the C ABI host-buffer call (lmoe_forward_host): every step copies
    # its input from pinned host memory and its output back to pinned host memory.  Wall clock
    # with the device synchronised on both sides (the input copies run on the library's copy
    # stream, which events on the caller's stream would not bracket).
    xh = [t.cpu().pin_memory() for t in xs]
    oh = torch.empty((w.bt, s.d), dtype=layer.dtype).pin_memory()
    for i in range(2):
        layer.forward_host(xh[i], oh)
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        layer.forward_host(xh[i % 2], oh)
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3
    barrier(ws)
    e2e_ms = max_over_ranks(e2e_ms, ws, device)
    e2e_value = sum_over_ranks(float(w.bt * args.e2e_steps), ws, device) / (e2e_ms / 1e3)
    layer.forward(xs[(args.e2e_steps - 1) % 2], out)
    torch.cuda.synchronize()
    if not torch.equal(oh, out.cpu()):
        raise RuntimeError("host-buffer forward differs from the device-buffer forward")
    xbytes = w.bt * s.d * (2 if s.dtype == "bf16" else 4)

    # ---- CPU oracle baseline (rank 0, one GPU only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not lowp and args.latent_norm == "expert":
        t = oracle_sample_time(w, x, weights, bias, args.cpu_tokens)
        cpu = {"value": args.cpu_tokens / t, "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
               "sample": f"{args.cpu_tokens} tokens spread over the batch, routed among themselves, "
                         f"{t:.1f} s wall; expert weights fetched from HBM and upcast to fp64 inside the timing"}

    extras = {}
    default_line = (args.workload == DEFAULT_WORKLOAD and args.bt is None and not lowp and
                    args.latent_norm == "expert" and not args.no_extra)
    if default_line:
        layer.close()
        del xs, out, xh, oh
        torch.cuda.empty_cache()
        for key, name, experts in EXTRA_WORKLOADS:
            extras[key] = extra_workload(name, weights, args.steps, args.warmup, local, ws, device, pk, experts)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": s.dtype, "data": "synthetic",
                "config": {"workload": w.name, "bt": w.bt, "d": s.d, "latent": s.latent, "n_experts": s.n_experts,
                           "top_k": s.top_k, "expert_inter": s.expert_inter, "n_shared": s.n_shared,
                           "shared_inter": s.shared_inter, "global_batch": w.bt * ws,
                           "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                           "l2": "no flush: every step streams the whole weight set "
                                 f"({layer_bytes / 1e9:.1f} GB algorithmic) through a 126 MB L2"},
                "roofline": roof, "layer_roofline": layer_roof,
                "stage_ms_per_step": {k: v / max(calls, 1) for k, v in stage_ms.items()},
                "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": xbytes,
                        "d2h_bytes_per_step": xbytes, "api": "lmoe_forward_host, pinned host buffers",
                        "timer": "wall clock, device synchronised on both sides", "steps": args.e2e_steps},
                "gpu_launches": launches, "clocks": clk, "engine": lmoe_build_info()}
        if args.fp8_experts:
            line["dtype"] = "bf16 (routed experts e4m3)"
            line["metric"] = METRIC + " [fp8 routed experts]"
        if args.mxfp4_experts:
            line["dtype"] = "bf16 (routed experts e2m1 x e4m3, ue8m0 block scales)"
            line["metric"] = METRIC + " [MXFP4 routed experts]"
        if args.latent_norm != "expert":
            line["metric"] += f" [latent norm: {args.latent_norm}]"
            line["config"]["latent_norm"] = args.latent_norm
        line.update(extras)
        print(json.dumps(line), flush=True)
    if not default_line:
        layer.close()
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
