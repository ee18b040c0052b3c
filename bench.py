#!/usr/bin/env python
"""One MLA layer decode step on B300: append -> absorb -> decode attention
(split-KV + LSE combine) -> W_UV up-projection, through the C ABI.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl native|reference]

Prints one JSON line (rank 0). The step runs on inputs resident in HBM; L2 is
flushed (a 512 MiB write) before every timed step, outside its events. The
decode call is timed on its own with CUDA events on the launching stream for
the roofline figure. ``e2e`` repeats the step with the step's inputs copied
from pinned host memory and the output copied back inside the timed region.
Multi-GPU runs are independent replicas (the decode step has no exchange).
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
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import mla_inputs as W  # noqa: E402

METRIC = "MLA decode TFLOP/s + HBM GB/s as % of B300 roofline; µs per layer decode step"
DEFAULT_WORKLOAD = W.DSV2_B16.name
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
ACT = {"f32": 0, "bf16": 1}
CACHE = {"f32": 0, "bf16": 1, "fp8_e4m3": 2}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def decode_traffic(workload: str):
    """DRAM bytes per launch of the decode kernel on `workload` from the committed
    ncu record, or None when there is no record for it or the kernel source has
    changed since the counters were taken."""
    import hashlib
    rec_path = os.path.join(ROOT, "profiles", "tc_decode_kernel_counters.json")
    src_path = os.path.join(ROOT, "mla_latent_kv_80_b300", "csrc", "tc_decode.cu")
    try:
        with open(rec_path) as f:
            rec = json.load(f)
        with open(src_path, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    w = rec.get("workloads", {}).get(workload)
    if rec.get("source_sha256") != sha or w is None:
        return None
    return w["dram_bytes_read_per_launch"] + w["dram_bytes_write_per_launch"]


def cache_bytes_per_token(w: W.Workload) -> int:
    if w.cache_dtype == "fp8_e4m3":
        return w.d_c + 2 * w.d_rope + 4
    return (w.d_c + w.d_rope) * (4 if w.cache_dtype == "f32" else 2)


def visible_keys(w: W.Workload, seq_lens) -> list:
    out = []
    for L in seq_lens:
        for j in range(w.q_per_seq):
            out.append(max(int(L) - w.q_per_seq + j + 1, 0))
    return out


def decode_work(w: W.Workload, seq_lens):
    """Algorithmic bytes and FLOPs of one decode-attention call."""
    act = 4 if w.act_dtype == "f32" else 2
    keys = visible_keys(w, seq_lens)
    rows = len(keys)
    cache_tokens = sum(int(L) for L in seq_lens)  # each cached token is read once per sequence
    bytes_ = (cache_tokens * cache_bytes_per_token(w)
              + rows * w.n_h * (w.d_c + w.d_rope) * act      # q_abs read
              + rows * w.n_h * w.d_c * act + rows * w.n_h * 4)  # o_lat + lse written
    flops = sum(keys) * 2 * w.n_h * ((w.d_c + w.d_rope) + w.d_c)
    return bytes_, flops


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_units(x: dict, seconds: float, units_per_call: int = 1):
    """Time the float64 oracle on (sequence, head) units of the workload until
    ``seconds`` elapsed. Returns (seconds per unit, units timed, threads)."""
    import numpy as np
    from oracle import mla_oracle as O
    from tests.oracle_io import oracle_inputs
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:  # pragma: no cover
        threads = os.cpu_count() or 1
    w = x["workload"]
    inp = oracle_inputs(x)
    t0 = time.perf_counter()
    units = 0
    h = 0
    while True:
        b = (units // w.n_h) % w.batch
        heads = [(h + i) % w.n_h for i in range(units_per_call)]
        O.decode_step(inp, sequences=[b], heads=heads)
        units += units_per_call * w.q_per_seq
        h += units_per_call
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return dt / units, units, threads


def full_step_units(w: W.Workload) -> int:
    return w.batch * w.q_per_seq * w.n_h


# ---------------------------------------------------------------- native arm
def run_native(args, rank, world):
    import mla_latent_kv_80_b300 as M
    w = W.BY_NAME[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    x = W.generate(w)
    d = lambda t: None if t is None else t.to(dev).contiguous()
    dims = M.make_dims(w.n_h, w.d_h, w.d_rope, w.d_c, w.d_v, w.d_model, w.page_size,
                       ACT[w.act_dtype], CACHE[w.cache_dtype], w.softmax_scale, w.rope_theta)
    cache_t = {k: d(v) for k, v in x["cache"].items()}
    cache = M.make_cache(cache_t["ckv"], cache_t["kr"], cache_t["scale"], x["num_pages"])
    bt, seq_lens = d(x["block_table"]), d(x["seq_lens"])
    h, seq_idx, pos = d(x["new_h"]), d(x["new_seq_idx"]), d(x["new_pos"])
    w_dkv, w_kr, w_uk, w_uv = (d(x[k]) for k in ("w_dkv", "w_kr", "w_uk", "w_uv"))
    if x["q"] is None:
        raise SystemExit("bench workloads draw their queries directly")
    q = d(x["q"])
    q_pos = d(W.query_positions(x["seq_lens"], w.q_per_seq))
    step = M.DecodeStep(dims, w.batch, w.q_per_seq, h.shape[0], args.num_splits, dev)
    flush = torch.empty(W.l2_flush_bytes() // 4, dtype=torch.float32, device=dev)

    def pre():
        step.prepare(cache, h, w_dkv, w_kr, seq_idx, pos, q, q_pos, w_uk, bt)

    def dec():
        step.decode(cache, bt, seq_lens)

    def post():
        step.out_proj(w_uv)

    def whole():
        pre(); dec(); post()

    # End-to-end inputs and output in pinned host memory.
    h_host = x["new_h"].pin_memory()
    q_host = x["q"].pin_memory()
    small_host = [t.pin_memory() for t in (x["new_seq_idx"], x["new_pos"], x["seq_lens"],
                                           W.query_positions(x["seq_lens"], w.q_per_seq))]
    small_dev = [seq_idx, pos, seq_lens, q_pos]
    o_host = torch.empty(step.o.shape, dtype=step.o.dtype).pin_memory()

    def e2e():
        h.copy_(h_host, non_blocking=True)
        q.copy_(q_host, non_blocking=True)
        for s_h, s_d in zip(small_host, small_dev):
            s_d.copy_(s_h, non_blocking=True)
        whole()
        o_host.copy_(step.o, non_blocking=True)

    step.status.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(args.warmup):
            e2e()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0, "device status after warm-up"
    # One CUDA graph per timed unit: the ABI calls only enqueue work, so a whole
    # step (or one stage of it) replays with no host work between kernels.
    graphs = {}
    for name, fn in (("step", whole), ("pre", pre), ("dec", dec), ("post", post), ("e2e", e2e)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs[name] = g
    for g in graphs.values():
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def timed(name, n):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for k in range(n):
            flush.zero_()
            evs[k][0].record(stream)
            graphs[name].replay()
            evs[k][1].record(stream)
        torch.cuda.synchronize()
        return [e[0].elapsed_time(e[1]) for e in evs]

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    step_ms = timed("step", args.steps)
    dec_ms = timed("dec", args.steps)
    pre_ms = timed("pre", args.steps)
    post_ms = timed("post", args.steps)
    e2e_ms = timed("e2e", args.steps)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    # The same step issued call by call from Python (host work between launches).
    eager_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        eager_ev[k][0].record(stream)
        e2e()
        eager_ev[k][1].record(stream)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0, "device status after the timed steps"
    eager_ms = [e[0].elapsed_time(e[1]) for e in eager_ev]
    h2d = sum(t.numel() * t.element_size() for t in [h_host, q_host] + small_host)
    d2h = o_host.numel() * o_host.element_size()

    def agg(v):
        t = torch.tensor([statistics.mean(v)], dtype=torch.float64, device=dev)
        if world > 1:
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())

    step_mean, dec_mean, e2e_mean = agg(step_ms), agg(dec_ms), agg(e2e_ms)
    if rank != 0:
        return None
    pk, src = peaks()
    bytes_, flops = decode_work(w, x["seq_lens"].tolist())
    traffic = decode_traffic(w.name)
    achieved = bytes_ / (dec_mean * 1e-3) / 1e9
    tflops = flops / (dec_mean * 1e-3) / 1e12
    out = {
        "metric": METRIC,
        "value": round(step_mean * 1e3 / world, 3),
        "unit": "us/step",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_mean, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": w.act_dtype if w.cache_dtype != "fp8_e4m3" else "bf16+fp8cache",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch,
                   "seq_len": w.seq_len or list(w.seq_len_range or w.seq_lens),
                   "q_per_seq": w.q_per_seq, "n_h": w.n_h, "d_c": w.d_c, "d_rope": w.d_rope,
                   "page_size": w.page_size, "cache_dtype": w.cache_dtype,
                   "append_tokens": int(h.shape[0]),
                   "l2": "flushed by a 512 MiB write before every timed step (outside its events)",
                   "parallelism": f"replicas x{world}"},
        "breakdown_us": {"append+absorb": round(statistics.mean(pre_ms) * 1e3, 2),
                         "decode_attn": round(dec_mean * 1e3, 2),
                         "out_proj": round(statistics.mean(post_ms) * 1e3, 2)},
        "roofline": {"kernel": "mla_decode_attn (plan + main + combine launches)",
                     "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": pk["hbm_gbs"], "peak_source": src, "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": traffic,
                     "traffic_note": "dram bytes read+written by tc_decode_kernel per launch, from "
                                     "profiles/tc_decode_kernel_counters.json (null if the kernel changed)",
                     "algorithmic_bytes": bytes_, "flops": flops,
                     "tflops": round(tflops, 2),
                     "tensor_frac": round(tflops / pk["bf16_tflops"], 4)},
        "e2e": {"value": round(e2e_mean * 1e3 / world, 3), "unit": "us/step",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "pinned-host inputs copied in, the four ABI calls, output copied out; one CUDA graph per step",
                "eager_value": round(statistics.mean(eager_ms) * 1e3 / world, 3)},
        "gpu_launches": args.steps * 7,
        "timing": "CUDA events around one CUDA-graph replay per step on the launching stream",
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        per_unit, units, threads = oracle_units(x, args.cpu_seconds)
        out["cpu_baseline"] = {
            "value": round(per_unit * full_step_units(w) * 1e6, 1), "unit": "us/step",
            "cores": threads, "kind": "oracle",
            "sample": f"{units} (sequence, head) rows of this workload through the float64 oracle "
                      f"in {args.cpu_seconds:.0f}s, scaled to the {full_step_units(w)} rows of one step"}
    return out


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    w = W.BY_NAME[args.workload]
    x = W.generate(w)
    per_step_s = max(1.0, 60.0 / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        oracle_units(x, per_step_s / 4)
    vals = []
    threads = 1
    units_total = 0
    for _ in range(args.steps):
        per_unit, units, threads = oracle_units(x, per_step_s)
        vals.append(per_unit * full_step_units(w) * 1e6)
        units_total += units
    v = statistics.mean(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us/step",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch,
                   "seq_len": w.seq_len or list(w.seq_len_range or w.seq_lens),
                   "q_per_seq": w.q_per_seq, "n_h": w.n_h, "page_size": w.page_size,
                   "cache_dtype": w.cache_dtype, "parallelism": "none (CPU)"},
        "cpu_baseline": {"value": round(v, 1), "unit": "us/step", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {per_step_s:.1f}s of (sequence, head) rows of this "
                                   f"workload through the float64 oracle, scaled to one full step "
                                   f"({units_total} rows timed in total)"},
        "e2e": {"value": round(v, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.BY_NAME))
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    out = run_native(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
