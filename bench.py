#!/usr/bin/env python
"""One MLA layer decode step on B300: append -> absorb -> decode attention
(split-KV + LSE combine) -> W_UV up-projection, through the C ABI. With a
chunked-prefill workload (--workload dsv2_bf16_prefill_b4_l8192_c512) the
step is append -> mla_prefill_attn instead.

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
DEFAULT_WORKLOAD = W.DSV2_VARLEN.name
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
class _CtypesNvml:
    """The few read-only NVML queries the sampler makes, through the driver's
    libnvidia-ml directly (for hosts without the Python bindings)."""
    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")

    def _ok(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed: {rc}")

    def nvmlInit(self):
        self._ok(self.lib.nvmlInit_v2(), "nvmlInit_v2")

    def nvmlDeviceGetHandleByUUID(self, uuid):
        h = self.c.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByUUID(self.c.c_char_p(uuid), self.c.byref(h)), "by uuid")
        return h

    def nvmlDeviceGetHandleByPciBusId(self, bus):
        h = self.c.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByPciBusId_v2(self.c.c_char_p(bus), self.c.byref(h)), "by pci")
        return h

    def nvmlDeviceGetMaxClockInfo(self, h, kind):
        v = self.c.c_uint()
        self._ok(self.lib.nvmlDeviceGetMaxClockInfo(h, kind, self.c.byref(v)), "max clock")
        return v.value

    def nvmlDeviceGetClockInfo(self, h, kind):
        v = self.c.c_uint()
        self._ok(self.lib.nvmlDeviceGetClockInfo(h, kind, self.c.byref(v)), "clock")
        return v.value

    def nvmlDeviceGetPowerUsage(self, h):
        v = self.c.c_uint()
        self._ok(self.lib.nvmlDeviceGetPowerUsage(h, self.c.byref(v)), "power")
        return v.value

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        v = self.c.c_ulonglong()
        self._ok(self.lib.nvmlDeviceGetCurrentClocksThrottleReasons(h, self.c.byref(v)), "reasons")
        return v.value


class ClockSampler:
    """Samples the SM clock, its maximum, board power and the clock-event
    reasons of one GPU every few milliseconds while the timed region runs.
    Read-only NVML queries; falls back to `nvidia-smi -lms 100`."""
    REASONS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
               "sw_power_cap": 0x4}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int, period_s: float = 0.002):
        import threading
        self.samples = []
        self.proc = None
        self.source = "nvml"
        self._stop = threading.Event()
        try:
            try:
                import pynvml
            except ImportError:
                pynvml = _CtypesNvml()
            pynvml.nvmlInit()
            props = torch.cuda.get_device_properties(dev_index)
            try:
                self.h = pynvml.nvmlDeviceGetHandleByUUID(("GPU-" + str(props.uuid)).encode())
            except Exception:
                self.h = pynvml.nvmlDeviceGetHandleByPciBusId(
                    f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode())
            self.nv = pynvml
            self.smax = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.thread = threading.Thread(target=self._run, args=(period_s,), daemon=True)
            self.thread.start()
        except Exception:
            self.nv = None
            self.source = "nvidia-smi"
            self.path = tempfile.mktemp(suffix=".csv")
            try:
                self.f = open(self.path, "w")
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={dev_index}", f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                    stderr=subprocess.DEVNULL)
            except (OSError, FileNotFoundError):
                self.proc = None

    def _run(self, period_s):
        nv = self.nv
        while not self._stop.is_set():
            try:
                sm = nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)
                pw = nv.nvmlDeviceGetPowerUsage(self.h) / 1000.0
                rs = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                self.samples.append((sm, pw, rs))
            except Exception:
                pass
            time.sleep(period_s)

    def stop(self) -> dict:
        if self.nv is not None:
            self._stop.set()
            self.thread.join(timeout=2)
            sm = [x[0] for x in self.samples]
            reasons = sorted({n for _, _, r in self.samples for n, bit in self.REASONS.items() if r & bit})
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.smax,
                    "power_w_max": max((x[1] for x in self.samples), default=None),
                    "samples": len(sm), "source": "nvml, every 2 ms during the timed region",
                    "reasons": reasons}
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
                "samples": len(sm), "source": "nvidia-smi -lms 100", "reasons": sorted(reasons)}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_units(x: dict, seconds: float, start: int = 0):
    """Time the float64 oracle on (sequence, head) rows of the workload until
    ``seconds`` elapsed, visiting sequences in a seeded shuffled order from
    ``start``. Returns (seconds per visible key and head, rows timed, threads,
    next start). A row's cost is proportional to the keys it sees, so the
    per-key-head time extrapolates to any mix of sequence lengths."""
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
    keys = visible_keys(w, x["seq_lens"].tolist())
    order = np.random.default_rng(12345).permutation(w.batch * w.n_h)
    t0 = time.perf_counter()
    rows = key_heads = 0
    k = start
    while True:
        b, h = divmod(int(order[k % order.size]), w.n_h)
        O.decode_step(inp, sequences=[b], heads=[h])
        rows += w.q_per_seq
        key_heads += sum(keys[b * w.q_per_seq:(b + 1) * w.q_per_seq])
        k += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return dt / max(key_heads, 1), rows, threads, k


def full_step_key_heads(w: W.Workload, seq_lens) -> int:
    return sum(visible_keys(w, seq_lens.tolist())) * w.n_h


# ---------------------------------------------------------------- replicas (N > 1)
def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of one value over the ranks of the job (each rank is an
    independent replica on its own GPU; the job's step time is the slowest
    replica's). With one rank, the value itself."""
    t = torch.tensor([value], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_aggregate(step_ms: float, world: int) -> dict:
    """Whole-job rate of N independent replicas, each running one layer step
    in `step_ms` (the max-over-ranks time): their step rates add up."""
    return {"steps_per_s": round(world * 1e3 / step_ms, 1),
            "note": "N independent replicas, one layer step each; value is the "
                    "max-over-replicas time of one step"}


# ---------------------------------------------------------------- shared config
def config_of(w: W.Workload, parallelism: str, seq_lens) -> dict:
    """The `config` object of both arms' JSON lines (same workload, same keys)."""
    append_tokens = sum(min(w.append_new, int(L)) if w.append_new >= 0 else int(L)
                        for L in seq_lens.tolist())
    return {"workload": w.name, "batch": w.batch,
            "seq_len": w.seq_len or list(w.seq_len_range or w.seq_lens),
            "q_per_seq": w.q_per_seq, "n_h": w.n_h, "d_c": w.d_c, "d_rope": w.d_rope,
            "page_size": w.page_size, "cache_dtype": w.cache_dtype,
            "append_tokens": append_tokens,
            "l2": "flushed by a 512 MiB write before every timed step (outside its events)",
            "parallelism": parallelism}


class Packed:
    """Several host tensors behind ONE pinned host buffer and one device buffer,
    so that a step's inputs cross the link in a single cudaMemcpyAsync."""

    def __init__(self, tensors, dev):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        self.host = torch.empty(max(n, 256), dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
        self.views = []
        for t, o in zip(tensors, offs):
            nb = t.numel() * t.element_size()
            self.host[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
            self.views.append(self.dev[o:o + nb].view(t.dtype).view(t.shape))
        self.nbytes = n

    def upload(self):
        self.dev.copy_(self.host, non_blocking=True)


# ---------------------------------------------------------------- native arm
LAUNCHES = {"step": 7, "pre": 3, "dec": 3, "post": 1, "e2e": 7, "wo": 3}  # library kernels per graph


def decode_roofline(bytes_, flops, gbs, tflops, pk, src, traffic):
    """The decode call against the roofline that bounds it: the larger of its
    bytes over the HBM peak and its flops over the bf16 tensor peak (the cache
    is read once; an fp8 cache is converted to bf16 before the MMAs)."""
    hbm_frac, tensor_frac = gbs / pk["hbm_gbs"], tflops / pk["bf16_tflops"]
    tensor = flops / (pk["bf16_tflops"] * 1e12) > bytes_ / (pk["hbm_gbs"] * 1e9)
    r = {"kernel": "mla_decode_attn (all launches of the call)"}
    if tensor:
        r.update({"bound": "tensor", "achieved": round(tflops, 2), "peak": pk["bf16_tflops"],
                  "peak_source": src + " bf16 burst (the call is timed alone)", "unit": "TFLOP/s",
                  "frac": round(tensor_frac, 4)})
    else:
        r.update({"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "peak_source": src,
                  "unit": "GB/s", "frac": round(hbm_frac, 4)})
    r.update({"traffic": traffic,
              "traffic_note": "dram bytes read+written by the decode kernel per launch, from "
                              "profiles/tc_decode_kernel_counters.json (null if the kernel changed)",
              "algorithmic_bytes": bytes_, "flops": flops, "gbs": round(gbs, 1), "tflops": round(tflops, 2),
              "hbm_frac": round(hbm_frac, 4), "tensor_frac": round(tensor_frac, 4)})
    return r


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
    q_pos_host = W.query_positions(x["seq_lens"], w.q_per_seq)
    q_pos = d(q_pos_host)
    w_o = d(W.output_weight(w))
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

    def wo():  # W_UV then W_O: the layer's output projection, timed apart from the step
        step.out_proj_wo(w_uv, w_o)

    # End to end: the step's inputs start in pinned host memory, packed per
    # consumer: what the append needs (hidden states, slots, lengths) crosses on
    # the caller's stream, the queries on the side stream where the absorb runs,
    # so their copy overlaps the append. The output o comes back at the end.
    pa = Packed([x["new_h"], x["new_seq_idx"], x["new_pos"], x["seq_lens"]], dev)
    pb = Packed([x["q"], q_pos_host], dev)
    e_h, e_seq_idx, e_pos, e_seq_lens = pa.views
    e_q, e_q_pos = pb.views
    o_host = torch.empty(step.o.shape, dtype=step.o.dtype).pin_memory()
    side = torch.cuda.Stream(device=dev)

    def e2e():
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        with torch.cuda.stream(side):
            pb.upload()
            step.absorb(e_q, e_q_pos, w_uk, side)
        pa.upload()
        step.append(cache, e_h, w_dkv, w_kr, e_seq_idx, e_pos, bt, main)
        main.wait_stream(side)
        step.decode(cache, bt, e_seq_lens)
        step.out_proj(w_uv)
        o_host.copy_(step.o, non_blocking=True)

    step.status.zero_()
    warm = torch.cuda.Stream(device=dev)
    warm.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(warm):
        for _ in range(args.warmup):
            e2e()
    torch.cuda.current_stream().wait_stream(warm)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0, "device status after warm-up"
    # One CUDA graph per timed unit: the ABI calls only enqueue work, so a whole
    # step (or one stage of it) replays with no host work between kernels.
    graphs = {}
    wo()
    for name, fn in (("step", whole), ("pre", pre), ("dec", dec), ("post", post), ("e2e", e2e), ("wo", wo)):
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
    time.sleep(0.05 if sampler else 0)
    step_ms = timed("step", args.steps)
    dec_ms = timed("dec", args.steps)
    pre_ms = timed("pre", args.steps)
    post_ms = timed("post", args.steps)
    e2e_ms = timed("e2e", args.steps)
    wo_ms = timed("wo", args.steps)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    # The same end-to-end step issued call by call from Python (host work between launches).
    eager_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        eager_ev[k][0].record(stream)
        e2e()
        eager_ev[k][1].record(stream)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0, "device status after the timed steps"
    eager_ms = [e[0].elapsed_time(e[1]) for e in eager_ev]
    h2d = pa.nbytes + pb.nbytes
    d2h = o_host.numel() * o_host.element_size()
    # Host link rate for the same bytes (pinned, one copy each way), for
    # comparing the end-to-end gap with the copies it contains.
    link = []
    for _ in range(max(args.steps, 5)):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(stream)
        pa.upload(); pb.upload()
        ev[1].record(stream)
        o_host.copy_(step.o, non_blocking=True)
        ev[2].record(stream)
        torch.cuda.synchronize()
        link.append((ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])))
    h2d_ms = statistics.median(x[0] for x in link)
    d2h_ms = statistics.median(x[1] for x in link)

    def agg(v):
        return max_over_ranks(statistics.mean(v), world, dev)

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
        "value": round(step_mean * 1e3, 3),
        "unit": "us/step",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_mean, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": w.act_dtype if w.cache_dtype != "fp8_e4m3" else "bf16+fp8cache",
        "data": "synthetic",
        "config": config_of(w, f"replicas x{world}", x["seq_lens"]),
        "aggregate": replica_aggregate(step_mean, world),
        "breakdown_us": {"append+absorb": round(statistics.mean(pre_ms) * 1e3, 2),
                         "decode_attn": round(dec_mean * 1e3, 2),
                         "out_proj": round(statistics.mean(post_ms) * 1e3, 2)},
        "out_proj_wo": {"us": round(statistics.mean(wo_ms) * 1e3, 2),
                        "weight_bytes": (w_o.numel() + w_uv.numel()) * w_o.element_size(),
                        "gbs": round((w_o.numel() + w_uv.numel()) * w_o.element_size()
                                     / (statistics.mean(wo_ms) * 1e-3) / 1e9, 1),
                        "note": "W_UV then W_O (mla_out_proj_wo), timed on its own; not part of the step"},
        "roofline": decode_roofline(bytes_, flops, achieved, tflops, pk, src, traffic),
        "e2e": {"value": round(e2e_mean * 1e3, 3), "unit": "us/step",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "two packed pinned-host input copies (the queries' on the absorb stream, "
                       "overlapping the append), the four ABI calls, o copied out; one CUDA graph per step",
                "eager_value": round(statistics.mean(eager_ms) * 1e3, 3),
                "link": {"h2d_us": round(h2d_ms * 1e3, 2), "d2h_us": round(d2h_ms * 1e3, 2),
                         "h2d_gbs": round(h2d / (h2d_ms * 1e-3) / 1e9, 2),
                         "d2h_gbs": round(d2h / (d2h_ms * 1e-3) / 1e9, 2),
                         "how": "the same pinned copies alone, serialised on one stream"}},
        "gpu_launches": args.steps * sum(LAUNCHES.values()),
        "gpu_launches_note": "library kernels inside the timed region: per step, the whole step (7), "
                             "append+absorb (3), decode call (3), out-proj (1), end to end (7), "
                             "out-proj with W_O (3)",
        "timing": "CUDA events around one CUDA-graph replay per step on the launching stream",
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        per_kh, rows, threads, _ = oracle_units(x, args.cpu_seconds)
        total = full_step_key_heads(w, x["seq_lens"])
        out["cpu_baseline"] = {
            "value": round(per_kh * total * 1e6, 1), "unit": "us/step",
            "cores": threads, "kind": "oracle",
            "sample": f"{rows} (query, head) rows of this workload, sequences in a seeded random "
                      f"order, through the float64 oracle in {args.cpu_seconds:.0f}s; time per visible "
                      f"key and head scaled to the {total} key-heads of one step"}
    return out


# ---------------------------------------------------------------- chunked prefill
PREFILL_METRIC = "MLA chunked-prefill TFLOP/s as % of B300 roofline; µs per layer prefill step"
PREFILL_LAUNCHES = {"step": 6, "app": 2, "att": 4, "abs": 4, "e2e": 6}  # library kernels per graph


def prefill_flops(w: W.Workload, seq_lens):
    """(explicit-form flops, absorbed-form flops, visible pairs) of one prefill call:
    per visible (query, key) pair 2 n_h (d_h + d_rope + d_v) explicit / 2 n_h
    (2 d_c + d_rope) absorbed; plus 2 n_h (d_h + d_v) d_c per cached token
    (forming keys and values) explicit / per query (absorbing W_UK, applying
    W_UV) absorbed."""
    pairs = sum(visible_keys(w, seq_lens))
    per = 2 * w.n_h * (w.d_h + w.d_v) * w.d_c
    tokens = sum(int(L) for L in seq_lens)
    rows = w.batch * w.q_per_seq
    explicit = per * tokens + 2 * w.n_h * (w.d_h + w.d_rope + w.d_v) * pairs
    absorbed = per * rows + 2 * w.n_h * (2 * w.d_c + w.d_rope) * pairs
    return explicit, absorbed, pairs


def prefill_oracle_units(x: dict, seconds: float, start: int = 0):
    """Time the float64 oracle's explicit prefill on whole (sequence, head)
    pairs (all C queries) until ``seconds`` elapsed; returns (seconds per
    (sequence, head), pairs timed, threads, next start)."""
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
    order = np.random.default_rng(12345).permutation(w.batch * w.n_h)
    t0 = time.perf_counter()
    k = start
    n = 0
    while True:
        b, h = divmod(int(order[k % order.size]), w.n_h)
        O.prefill_step(inp, sequences=[b], heads=[h])
        n += 1
        k += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return (time.perf_counter() - t0) / n, n, threads, k


def run_prefill_native(args, rank, world):
    """One layer's chunked-prefill step: append the chunk's tokens to the cache,
    then attend (the cheaper form by mla_prefill_form: explicit here)."""
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
    q = d(x["q"])
    B, C, T = w.batch, w.q_per_seq, h.shape[0]
    L_max = int(x["seq_lens"].max())
    form = M.mla_prefill_form(dims, C, L_max)
    ws_a_bytes = M.mla_cache_append_workspace_size(dims, T)
    ws_a = torch.empty(max(ws_a_bytes, 256), dtype=torch.uint8, device=dev)
    ws_p_bytes = M.mla_prefill_workspace_size(dims, B, C, L_max)
    ws_p = torch.empty(ws_p_bytes, dtype=torch.uint8, device=dev)
    o = torch.empty((B * C, w.n_h, w.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B * C, w.n_h), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    step_abs = M.DecodeStep(dims, B, C, 0, args.num_splits, dev)
    q_pos_host = W.query_positions(x["seq_lens"], C)
    q_pos = d(q_pos_host)
    flush = torch.empty(W.l2_flush_bytes() // 4, dtype=torch.float32, device=dev)

    def app(h_=h, seq_idx_=seq_idx, pos_=pos, stream=None):
        M.mla_cache_append(dims, cache, T, h_, w_dkv, w_kr, seq_idx_, pos_, bt, bt.shape[1], ws_a, ws_a_bytes,
                           status, stream)

    def att(q_=q, seq_lens_=seq_lens):
        M.mla_prefill_attn(dims, cache, B, C, L_max, q_, w_uk, w_uv, bt, bt.shape[1], seq_lens_, ws_p, ws_p_bytes,
                           o, lse, status)

    def whole():
        app(); att()

    def absorbed():
        step_abs.absorb(q, q_pos, w_uk)
        step_abs.decode(cache, bt, seq_lens)
        step_abs.out_proj(w_uv)

    pa = Packed([x["new_h"], x["new_seq_idx"], x["new_pos"], x["seq_lens"], x["q"]], dev)
    e_h, e_seq_idx, e_pos, e_seq_lens, e_q = pa.views
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()

    def e2e():
        pa.upload()
        app(e_h, e_seq_idx, e_pos)
        att(e_q, e_seq_lens)
        o_host.copy_(o, non_blocking=True)

    status.zero_()
    step_abs.status.zero_()
    warm = torch.cuda.Stream(device=dev)
    warm.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(warm):
        for _ in range(args.warmup):
            e2e()
            absorbed()
    torch.cuda.current_stream().wait_stream(warm)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(step_abs.status.item()) == 0, "device status after warm-up"
    graphs = {}
    for name, fn in (("step", whole), ("app", app), ("att", att), ("abs", absorbed), ("e2e", e2e)):
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
    step_ms = timed("step", args.steps)
    app_ms = timed("app", args.steps)
    att_ms = timed("att", args.steps)
    abs_ms = timed("abs", args.steps)
    e2e_ms = timed("e2e", args.steps)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    assert int(status.item()) == 0 and int(step_abs.status.item()) == 0, "device status after the timed steps"

    def agg(v):
        return max_over_ranks(statistics.mean(v), world, dev)

    step_mean, att_mean, e2e_mean = agg(step_ms), agg(att_ms), agg(e2e_ms)
    if rank != 0:
        return None
    pk, src = peaks()
    f_exp, f_abs, pairs = prefill_flops(w, x["seq_lens"].tolist())
    achieved = f_exp / (att_mean * 1e-3) / 1e12
    abs_mean = statistics.mean(abs_ms)
    out = {
        "metric": PREFILL_METRIC,
        "value": round(step_mean * 1e3, 3), "unit": "us/step",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_mean, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": w.act_dtype, "data": "synthetic",
        "config": config_of(w, f"replicas x{world}", x["seq_lens"]),
        "aggregate": replica_aggregate(step_mean, world),
        "form": "explicit" if form else "absorbed",
        "breakdown_us": {"append": round(statistics.mean(app_ms) * 1e3, 2),
                         "prefill_attn": round(att_mean * 1e3, 2),
                         "note": "each timed alone"},
        "absorbed_form": {"us": round(abs_mean * 1e3, 2),
                          "tflops": round(f_abs / (abs_mean * 1e-3) / 1e12, 1),
                          "note": "the same chunk through mla_absorb_q, mla_decode_attn (q_per_seq = C) "
                                  "and mla_out_proj, timed alone"},
        "roofline": {"kernel": "mla_prefill_attn (gather, cos/sin table, key/value expansion, attention)",
                     "bound": "tensor", "achieved": round(achieved, 1), "peak": pk["bf16_tflops"],
                     "peak_source": src + " bf16 burst (the call is timed alone)", "unit": "TFLOP/s",
                     "frac": round(achieved / pk["bf16_tflops"], 4), "traffic": None,
                     "algorithmic_flops": f_exp, "visible_pairs": pairs},
        "e2e": {"value": round(e2e_mean * 1e3, 3), "unit": "us/step",
                "h2d_bytes_per_step": pa.nbytes, "d2h_bytes_per_step": o_host.numel() * o_host.element_size(),
                "how": "one packed pinned-host input copy (hidden states, slots, lengths, queries), append, "
                       "prefill attention, o copied out; one CUDA graph per step"},
        "gpu_launches": args.steps * sum(PREFILL_LAUNCHES.values()),
        "gpu_launches_note": "library kernels inside the timed region: per step, the whole step (6: append "
                             "GEMM and epilogue, gather, cos/sin table, expansion, attention), the append (2), "
                             "the prefill call (4), the absorbed form (4), end to end (6)",
        "timing": "CUDA events around one CUDA-graph replay per step on the launching stream",
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        per_bh, n, threads, _ = prefill_oracle_units(x, args.cpu_seconds)
        out["cpu_baseline"] = {
            "value": round(per_bh * B * w.n_h * 1e6, 1), "unit": "us/step", "cores": threads, "kind": "oracle",
            "sample": f"{n} whole (sequence, head) pairs ({C} queries each) of this workload through the "
                      f"float64 oracle's explicit prefill in {args.cpu_seconds:.0f}s, scaled to the "
                      f"{B * w.n_h} pairs of one step (the append is not counted)"}
    return out


def run_prefill_reference(args):
    w = W.BY_NAME[args.workload]
    x = W.generate(w)
    per_step_s = max(1.0, 60.0 / max(args.steps + args.warmup, 1))
    k = 0
    for _ in range(args.warmup):
        _, _, _, k = prefill_oracle_units(x, per_step_s / 4, k)
    vals, n_total, threads = [], 0, 1
    for _ in range(args.steps):
        per_bh, n, threads, k = prefill_oracle_units(x, per_step_s, k)
        vals.append(per_bh * w.batch * w.n_h * 1e6)
        n_total += n
    v = statistics.mean(vals)
    return {
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(v, 1), "unit": "us/step",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, "replicas x1", x["seq_lens"]), "extrapolated": True,
        "cpu_baseline": {"value": round(v, 1), "unit": "us/step", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {per_step_s:.1f}s of whole (sequence, head) pairs through the "
                                   f"float64 oracle's explicit prefill, scaled to the {w.batch * w.n_h} pairs "
                                   f"of one step ({n_total} pairs timed in all)"},
        "e2e": {"value": round(v, 1), "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    w = W.BY_NAME[args.workload]
    x = W.generate(w)
    total = full_step_key_heads(w, x["seq_lens"])
    per_step_s = max(1.0, 60.0 / max(args.steps + args.warmup, 1))
    k = 0
    for _ in range(args.warmup):
        _, _, _, k = oracle_units(x, per_step_s / 4, k)
    vals = []
    threads = 1
    rows_total = 0
    for _ in range(args.steps):
        per_kh, rows, threads, k = oracle_units(x, per_step_s, k)
        vals.append(per_kh * total * 1e6)
        rows_total += rows
    v = statistics.mean(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us/step",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_of(w, "replicas x1", x["seq_lens"]),
        "extrapolated": True,
        "cpu_baseline": {"value": round(v, 1), "unit": "us/step", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {per_step_s:.1f}s of (query, head) rows of this workload "
                                   f"(sequences in a seeded random order) through the float64 oracle; "
                                   f"the time per visible key and head is extrapolated to the {total} "
                                   f"key-heads of one full step ({rows_total} rows timed in all)"},
        "e2e": {"value": round(v, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
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
    prefill = W.BY_NAME[args.workload] in W.PREFILL_WORKLOADS
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_prefill_reference(args) if prefill else run_reference(args)), flush=True)
        return
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    out = run_prefill_native(args, rank, world) if prefill else run_native(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
