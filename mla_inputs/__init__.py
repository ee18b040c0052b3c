"""Seeded synthetic workloads for MLA decode over a paged latent cache.

This module is shared by the CPU oracle, the GPU tests and the benchmark. It
only draws random numbers and lays them out (shapes, page pools, block tables,
sentinels); it holds none of the method's arithmetic (no projection, RoPE,
softmax or quantisation).

Shapes follow DeepSeek-V2 as the MLA pages state them ("MLA 是什么", table of
DeepSeek-V2 hyper-parameters: n_h=128, d_h=128, d_c=512, d_h^R=64) plus a tiny
fp32 case. Every tensor is a torch CPU tensor; callers move what they need to
the device.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

F32, BF16, FP8 = "f32", "bf16", "fp8_e4m3"
NAN_BF16_BITS = 0x7FC0
NAN_E4M3_CODE = 0x7F


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    act_dtype: str
    cache_dtype: str
    d_model: int
    n_h: int
    d_h: int
    d_rope: int
    d_c: int
    d_v: int
    batch: int
    seq_lens: Optional[tuple] = None          # explicit lengths
    seq_len: Optional[int] = None             # uniform length
    seq_len_range: Optional[tuple] = None     # inclusive uniform integer range
    q_per_seq: int = 1
    page_size: int = 64
    pool_tokens: Optional[int] = None         # page-pool size; None = just what is used
    block_table: str = "contiguous"           # contiguous | permutation
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    append_new: int = 1                       # trailing tokens per sequence written by append (-1 = all)
    rope_theta: float = 10000.0

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d_h + self.d_rope)

    @property
    def d_qk(self) -> int:
        return self.d_c + self.d_rope


TINY = Workload(
    name="tiny_fp32_b2", seed=0, act_dtype=F32, cache_dtype=F32,
    d_model=256, n_h=8, d_h=32, d_rope=16, d_c=64, d_v=32,
    batch=2, seq_lens=(37, 128), q_per_seq=1, page_size=16,
    block_table="permutation", append_new=-1)

DSV2_B16 = Workload(
    name="dsv2_bf16_b16_l4096", seed=1, act_dtype=BF16, cache_dtype=BF16,
    d_model=5120, n_h=128, d_h=128, d_rope=64, d_c=512, d_v=128,
    batch=16, seq_len=4096, q_per_seq=1, page_size=64, block_table="contiguous",
    append_new=1)

DSV2_VARLEN = Workload(
    name="dsv2_bf16_paged_varlen_b64", seed=2, act_dtype=BF16, cache_dtype=BF16,
    d_model=5120, n_h=128, d_h=128, d_rope=64, d_c=512, d_v=128,
    batch=64, seq_len_range=(1024, 16384), q_per_seq=1, page_size=64,
    pool_tokens=1_200_000, block_table="permutation", append_new=1)

DSV2_LONG = Workload(
    name="dsv2_bf16_long_b4_l131072", seed=3, act_dtype=BF16, cache_dtype=BF16,
    d_model=5120, n_h=128, d_h=128, d_rope=64, d_c=512, d_v=128,
    batch=4, seq_len=131072, q_per_seq=1, page_size=64, block_table="contiguous",
    outlier_frac=0.01, outlier_scale=8.0, append_new=0)

DSV2_FP8_Q2 = Workload(
    name="dsv2_fp8cache_q2_b128_l8192", seed=4, act_dtype=BF16, cache_dtype=FP8,
    d_model=5120, n_h=128, d_h=128, d_rope=64, d_c=512, d_v=128,
    batch=128, seq_len=8192, q_per_seq=2, page_size=64, block_table="contiguous",
    append_new=2)

WORKLOADS = [TINY, DSV2_B16, DSV2_VARLEN, DSV2_LONG, DSV2_FP8_Q2]

# Chunked prefill: four sequences of 8192 tokens whose last 512 tokens are the
# chunk (appended, then attending causally over the whole sequence).
DSV2_PREFILL = Workload(
    name="dsv2_bf16_prefill_b4_l8192_c512", seed=5, act_dtype=BF16, cache_dtype=BF16,
    d_model=5120, n_h=128, d_h=128, d_rope=64, d_c=512, d_v=128,
    batch=4, seq_len=8192, q_per_seq=512, page_size=64, block_table="permutation",
    append_new=512)
PREFILL_WORKLOADS = [DSV2_PREFILL]
BY_NAME = {w.name: w for w in WORKLOADS + PREFILL_WORKLOADS}


def shrink(w: Workload, **kw) -> Workload:
    """Same workload with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **kw)


def _torch_dtype(name: str) -> torch.dtype:
    return {F32: torch.float32, BF16: torch.bfloat16}[name]


def _randn(g: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32) * std


def _seq_lens(w: Workload, g: torch.Generator) -> torch.Tensor:
    if w.seq_lens is not None:
        return torch.tensor(w.seq_lens, dtype=torch.int32)
    if w.seq_len is not None:
        return torch.full((w.batch,), w.seq_len, dtype=torch.int32)
    lo, hi = w.seq_len_range
    return torch.randint(lo, hi + 1, (w.batch,), generator=g, dtype=torch.int64).to(torch.int32)


def _block_table(w: Workload, g: torch.Generator, seq_lens: torch.Tensor):
    P = w.page_size
    n_pages = [(int(L) + P - 1) // P for L in seq_lens]
    need = sum(n_pages)
    pool_pages = need if w.pool_tokens is None else max(need, w.pool_tokens // P)
    if w.block_table == "contiguous":
        order = torch.arange(pool_pages, dtype=torch.int64)
    elif w.block_table == "permutation":
        order = torch.randperm(pool_pages, generator=g)
    else:
        raise ValueError(w.block_table)
    max_pages = max(max(n_pages), 1)
    bt = torch.full((w.batch, max_pages), -1, dtype=torch.int32)
    k = 0
    for b, n in enumerate(n_pages):
        bt[b, :n] = order[k:k + n].to(torch.int32)
        k += n
    return bt, pool_pages


def generate(w: Workload, device_friendly: bool = True) -> dict:
    """Draw every input of one decode step of workload ``w``.

    Returns a dict of CPU tensors:
      weights   w_dkv [d_c,d_model], w_kr [d_rope,d_model], w_uk [n_h,d_h,d_c],
                w_uv [n_h,d_v,d_c], w_q [n_h,d_h+d_rope,d_model] (tiny case only),
                all ~ N(0, 1/fan_in) in the activation dtype
      seq_lens  [B] int32 (keys visible to the last query of each sequence)
      block_table [B, max_pages] int32, -1 past each sequence's pages
      cache     pool tensors in slot order (slot = page*page_size + offset):
                f32/bf16: ckv [num_slots, d_c+d_rope] with k_R in the last d_rope columns
                fp8:      ckv [num_slots, d_c] uint8 E4M3 codes, kr [num_slots, d_rope] bf16,
                          scale [num_slots] fp32
                Slots that hold no history token are NaN sentinels.
      new_h, new_seq_idx, new_pos  tokens that the append step writes
      q         [B*q_per_seq, n_h, d_h+d_rope] ~ N(0,1) (None for the tiny case,
                whose queries come from W_Q)
    """
    g = torch.Generator().manual_seed(w.seed)
    adt = _torch_dtype(w.act_dtype)
    out: dict = {"workload": w}

    out["w_dkv"] = _randn(g, (w.d_c, w.d_model), 1 / math.sqrt(w.d_model)).to(adt)
    out["w_kr"] = _randn(g, (w.d_rope, w.d_model), 1 / math.sqrt(w.d_model)).to(adt)
    out["w_uk"] = _randn(g, (w.n_h, w.d_h, w.d_c), 1 / math.sqrt(w.d_c)).to(adt)
    out["w_uv"] = _randn(g, (w.n_h, w.d_v, w.d_c), 1 / math.sqrt(w.d_c)).to(adt)
    if w.append_new < 0:
        out["w_q"] = _randn(g, (w.n_h, w.d_h + w.d_rope, w.d_model),
                            1 / math.sqrt(w.d_model)).to(adt)
    else:
        out["w_q"] = None

    seq_lens = _seq_lens(w, g)
    bt, pool_pages = _block_table(w, g, seq_lens)
    out["seq_lens"], out["block_table"], out["num_pages"] = seq_lens, bt, pool_pages
    P = w.page_size
    num_slots = pool_pages * P

    # Which slots hold history tokens (drawn directly) and which the append writes.
    hist_mask = torch.zeros(num_slots, dtype=torch.bool)
    new_slots = []
    new_seq, new_pos = [], []
    for b in range(w.batch):
        L = int(seq_lens[b])
        n_new = L if w.append_new < 0 else min(w.append_new, L)
        n_hist = L - n_new
        pages = bt[b].to(torch.int64)
        if n_hist > 0:
            t = torch.arange(n_hist)
            hist_mask[pages[t // P] * P + t % P] = True
        for t in range(n_hist, L):
            new_seq.append(b)
            new_pos.append(t)

    T = len(new_pos)
    out["new_seq_idx"] = torch.tensor(new_seq, dtype=torch.int32)
    out["new_pos"] = torch.tensor(new_pos, dtype=torch.int32)
    out["new_h"] = _randn(g, (T, w.d_model)).to(adt)

    # Cache pool, filled page-chunk by page-chunk to bound host memory.
    if w.cache_dtype in (F32, BF16):
        cdt = _torch_dtype(w.cache_dtype)
        ckv = torch.empty((num_slots, w.d_c + w.d_rope), dtype=cdt)
        step = 1 << 18
        for s0 in range(0, num_slots, step):
            s1 = min(num_slots, s0 + step)
            ckv[s0:s1] = _randn(g, (s1 - s0, w.d_c + w.d_rope)).to(cdt)
        if w.outlier_frac > 0:
            idx = torch.nonzero(hist_mask).flatten()
            n_out = int(round(w.outlier_frac * idx.numel()))
            pick = idx[torch.randperm(idx.numel(), generator=g)[:n_out]]
            ckv[pick] = (ckv[pick].float() * w.outlier_scale).to(cdt)
        ckv[~hist_mask] = float("nan")
        out["cache"] = {"ckv": ckv, "kr": None, "scale": None}
    elif w.cache_dtype == FP8:
        codes = torch.empty((num_slots, w.d_c), dtype=torch.uint8)
        step = 1 << 18
        for s0 in range(0, num_slots, step):
            s1 = min(num_slots, s0 + step)
            x = (_randn(g, (s1 - s0, w.d_c)) * 64.0).clamp(-448.0, 448.0)
            codes[s0:s1] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        kr = _randn(g, (num_slots, w.d_rope)).to(torch.bfloat16)
        scale = (torch.rand((num_slots,), generator=g) * 1.5 + 0.5) / 64.0
        codes[~hist_mask] = NAN_E4M3_CODE
        kr[~hist_mask] = float("nan")
        scale[~hist_mask] = float("nan")
        out["cache"] = {"ckv": codes, "kr": kr, "scale": scale}
    else:
        raise ValueError(w.cache_dtype)

    if w.append_new >= 0:
        out["q"] = _randn(g, (w.batch * w.q_per_seq, w.n_h, w.d_h + w.d_rope)).to(adt)
    else:
        out["q"] = None
    out["hist_mask"] = hist_mask
    return out


def output_weight(w: Workload) -> torch.Tensor:
    """W_O [d_model, n_h * d_v] ~ N(0, 1/fan_in) in the activation dtype, from a
    generator of its own (the other inputs of a workload do not change)."""
    g = torch.Generator().manual_seed(w.seed + 5000)
    fan_in = w.n_h * w.d_v
    return _randn(g, (w.d_model, fan_in), 1 / math.sqrt(fan_in)).to(_torch_dtype(w.act_dtype))


def query_positions(seq_lens: torch.Tensor, q_per_seq: int) -> torch.Tensor:
    """Position of each query row: query j of sequence b sits at seq_lens[b]-q+j."""
    B = seq_lens.numel()
    j = torch.arange(q_per_seq, dtype=torch.int32)
    return (seq_lens.view(B, 1) - q_per_seq + j.view(1, -1)).reshape(-1).to(torch.int32)


def l2_flush_bytes() -> int:
    """Bytes to write between timed iterations so that nothing stays in a 126 MB L2."""
    return 512 << 20


def stage_inputs(w: Workload, rows: int, seed_offset: int = 1000) -> dict:
    """Seeded inputs for checking one ABI stage on its own, in the activation dtype:
    q_abs [rows, n_h, d_c+d_rope] with the latent part ~ N(0, 1/4) and the RoPE
    part ~ N(0, 1) (the spread W_UK^T q has for q ~ N(0,1), W_UK ~ N(0, 1/d_c),
    d_h = 128), and o_lat [rows, n_h, d_c] ~ N(0, 1)."""
    g = torch.Generator().manual_seed(w.seed + seed_offset)
    adt = _torch_dtype(w.act_dtype)
    q_lat = _randn(g, (rows, w.n_h, w.d_c), 0.5)
    q_rot = _randn(g, (rows, w.n_h, w.d_rope))
    return {"q_abs": torch.cat([q_lat, q_rot], dim=-1).to(adt),
            "o_lat": _randn(g, (rows, w.n_h, w.d_c)).to(adt)}
