"""The decode entry point that allocates nothing.

Some callers cannot allocate device memory when they run a decode step (for
example code that is handed only its input and output buffers by a host
framework that owns the allocator). mla_decode_attn_noalloc serves them with
its scratch in a fixed-size array inside the library. This test calls it
through the C ABI twice in a row, on two different workloads (so the second
call runs over the first call's leftover scratch contents), and checks both
results against mla_decode_attn with a caller-allocated workspace, within the
same bf16 / fp32 tolerances the parity tests use. It also checks that a
request needing more scratch than the array holds is refused.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_inputs as W
from tests.gpu_harness import GpuRun, check_bf16, check_fp32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import mla_latent_kv_80_b300 as M
    return M


def _decode_both(M, w, num_splits):
    x = W.generate(w)
    run = GpuRun(M, x, num_splits=num_splits)
    s = run.step
    rows = w.batch * w.q_per_seq
    q_abs = W.stage_inputs(w, rows)["q_abs"].cuda()
    s.q_abs.copy_(q_abs)
    s.status.zero_()
    s.decode(run.cache, run.bt, run.seq_lens)
    torch.cuda.synchronize()
    assert int(s.status.item()) == 0
    ref_lat = s.o_lat.float().cpu().numpy()
    ref_lse = s.lse.cpu().numpy()
    o_lat = torch.full_like(s.o_lat, float("nan"))
    lse = torch.full_like(s.lse, float("nan"))
    M.mla_decode_attn_noalloc(run.dims, run.cache, w.batch, w.q_per_seq, q_abs, run.bt,
                              run.bt.shape[1], run.seq_lens, num_splits, o_lat, lse, s.status)
    torch.cuda.synchronize()
    assert int(s.status.item()) == 0
    return o_lat.float().cpu().numpy(), lse.cpu().numpy(), ref_lat, ref_lse, run


def test_noalloc_decode_matches_workspace_decode_twice(M):
    first = W.shrink(W.DSV2_VARLEN, batch=5, seq_len_range=(1, 900), pool_tokens=64 * 120,
                     append_new=0)
    second = W.shrink(W.DSV2_B16, batch=3, seq_len=700, append_new=0)
    for w, splits in ((first, 0), (second, 7)):
        o_lat, lse, ref_lat, ref_lse, _ = _decode_both(M, w, splits)
        check_bf16(o_lat, ref_lat, f"{w.name} o_lat")
        check_bf16(lse, ref_lse, f"{w.name} lse", stored_bf16=False)


def test_noalloc_decode_fp32_path(M):
    w = W.shrink(W.TINY, append_new=0)
    for splits in (0, 3):
        o_lat, lse, ref_lat, ref_lse, _ = _decode_both(M, w, splits)
        check_fp32(o_lat, ref_lat, "tiny o_lat")
        check_fp32(lse, ref_lse, "tiny lse")


def test_noalloc_rejects_requests_beyond_its_scratch(M):
    w = W.shrink(W.DSV2_B16, batch=2, seq_len=128, append_new=0)
    x = W.generate(w)
    run = GpuRun(M, x)
    limit = M.mla_decode_noalloc_scratch_bytes()
    splits = 1
    while M.mla_decode_workspace_size(run.dims, w.batch, 1, splits) <= limit:
        splits *= 2
    with pytest.raises(M.MlaError) as ei:
        M.mla_decode_attn_noalloc(run.dims, run.cache, w.batch, 1, run.step.q_abs, run.bt,
                                  run.bt.shape[1], run.seq_lens, splits, run.step.o_lat,
                                  run.step.lse, run.step.status)
    assert ei.value.code == -3
