"""The decode entry point that allocates nothing.

Some callers cannot allocate device memory when they run a decode step (for
example code that is handed only its input and output buffers by a host
framework that owns the allocator). mla_decode_attn_noalloc serves them with
its scratch in a fixed-size array inside the library. This test calls it
through the C ABI twice in a row, on two different workloads (so the second
call runs over the first call's leftover scratch contents), and checks both
results against mla_decode_attn with a caller-allocated workspace and the same
worker count: the two run the same kernels with the same plan, so the results
must be bit-identical (which also shows that nothing left in the array by the
first call leaks into the second). With num_splits = 0 and a default worker
count whose scratch does not fit the array (the CUDA-core path on DeepSeek-V2
shapes), the call must use the largest worker count that fits. It also checks
that a request needing more scratch than the array holds is refused.
"""

import numpy as np
import pytest
import torch

import mla_inputs as W
from tests.gpu_harness import DeviceRun, dims_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import mla_latent_kv_80_b300 as M
    return M


def _expected_workers(M, dims, w, num_splits):
    """Worker count the no-alloc call uses: the request, or with num_splits = 0
    the default when its scratch fits the array, else the largest that fits."""
    if num_splits:
        return num_splits
    limit = M.mla_decode_noalloc_scratch_bytes()
    g = M.mla_decode_default_splits(dims)
    while g > 1 and M.mla_decode_workspace_size(dims, w.batch, w.q_per_seq, g) > limit:
        g -= 1
    return g


def _decode_both(M, w, num_splits):
    x = W.generate(w)
    run = DeviceRun(M, x, num_splits=_expected_workers(M, dims_of(M, w), w, num_splits))
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
        np.testing.assert_array_equal(o_lat, ref_lat, err_msg=f"{w.name} o_lat")
        np.testing.assert_array_equal(lse, ref_lse, err_msg=f"{w.name} lse")


def test_noalloc_decode_fp32_path(M):
    w = W.shrink(W.TINY, append_new=0)
    for splits in (0, 3):
        o_lat, lse, ref_lat, ref_lse, _ = _decode_both(M, w, splits)
        np.testing.assert_array_equal(o_lat, ref_lat)
        np.testing.assert_array_equal(lse, ref_lse)


def test_noalloc_default_splits_fit_the_array_on_the_cuda_core_path(M):
    """DeepSeek-V2 shapes on the CUDA-core path (fp32 activations and cache):
    its default of one worker per SM needs more scratch than the array holds,
    so the call must pick the largest worker count that fits, not refuse."""
    w = W.shrink(W.DSV2_B16, name="dsv2_f32_small", act_dtype="f32", cache_dtype="f32",
                 batch=2, seq_len=300, append_new=0)
    dims = dims_of(M, w)
    limit = M.mla_decode_noalloc_scratch_bytes()
    assert M.mla_decode_workspace_size(dims, w.batch, 1, 0) > limit
    o_lat, lse, ref_lat, ref_lse, _ = _decode_both(M, w, 0)
    np.testing.assert_array_equal(o_lat, ref_lat)
    np.testing.assert_array_equal(lse, ref_lse)


def test_noalloc_rejects_requests_beyond_its_scratch(M):
    w = W.shrink(W.DSV2_B16, batch=2, seq_len=128, append_new=0)
    x = W.generate(w)
    run = DeviceRun(M, x)
    limit = M.mla_decode_noalloc_scratch_bytes()
    splits = 1
    while M.mla_decode_workspace_size(run.dims, w.batch, 1, splits) <= limit:
        splits *= 2
    with pytest.raises(M.MlaError) as ei:
        M.mla_decode_attn_noalloc(run.dims, run.cache, w.batch, 1, run.step.q_abs, run.bt,
                                  run.bt.shape[1], run.seq_lens, splits, run.step.o_lat,
                                  run.step.lse, run.step.status)
    assert ei.value.code == -3
