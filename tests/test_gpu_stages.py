"""Each ABI stage on its own: the decode and output stages are fed seeded
stage inputs (not results of earlier GPU stages) and compared with the oracle."""
import numpy as np
import pytest
import torch

import mla_inputs as W
from oracle import mla_oracle as O
from tests.gpu_harness import GpuRun, check_bf16, check_fp32, check_fp8, dims_of
from tests.oracle_io import oracle_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import mla_latent_kv_80_b300 as M
    return M


CASES = {
    "tiny_fp32": (W.shrink(W.TINY, append_new=0), None),
    "b16_small": (W.shrink(W.DSV2_B16, batch=3, seq_len=777, append_new=0), [0, 33, 127]),
    "varlen_paged": (W.shrink(W.DSV2_VARLEN, batch=6, seq_len_range=(1, 900), pool_tokens=64 * 120,
                              append_new=0), [1, 64, 126]),
    "fp8_q2": (W.shrink(W.DSV2_FP8_Q2, batch=2, seq_len=500, append_new=0), [0, 99]),
    "bench_b16_l4096": (W.shrink(W.DSV2_B16, append_new=0), [7, 120]),
}


def _check(w):
    if w.act_dtype == "f32":
        return check_fp32
    return check_fp8 if w.cache_dtype == "fp8_e4m3" else check_bf16


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("splits", [0, 5])
def test_decode_stage(M, name, splits):
    w, heads = CASES[name]
    x = W.generate(w)
    run = GpuRun(M, x, num_splits=splits)
    rows = w.batch * w.q_per_seq
    qa = W.stage_inputs(w, rows)["q_abs"]
    run.step.q_abs.copy_(qa.cuda())
    run.step.status.zero_()
    run.step.decode(run.cache, run.bt, run.seq_lens)
    torch.cuda.synchronize()
    assert int(run.step.status.item()) == 0
    o_lat = run.step.o_lat.float().cpu().numpy()
    lse = run.step.lse.cpu().numpy()
    inp = oracle_inputs(x)
    qa64 = qa.double().numpy()
    heads = list(range(w.n_h)) if heads is None else heads
    got_l, ref_l, got_s, ref_s = [], [], [], []
    for b in range(w.batch):
        L = int(x["seq_lens"][b])
        c, kr = O.gather_sequence(inp["cache"], w.cache_dtype, inp["block_table"], b, L,
                                  w.page_size, w.d_c)
        for j in range(w.q_per_seq):
            vis = max(L - w.q_per_seq + j + 1, 0)
            row = b * w.q_per_seq + j
            lat, l = O.absorbed_attention(qa64[row, heads], c[:vis], kr[:vis], w.softmax_scale)
            got_l.append(o_lat[row, heads]); ref_l.append(lat)
            got_s.append(lse[row, heads]); ref_s.append(l)
    chk = _check(w)
    chk(np.concatenate(got_l), np.concatenate(ref_l), f"{name} o_lat")
    if chk is check_bf16:
        check_bf16(np.concatenate(got_s), np.concatenate(ref_s), f"{name} lse", stored_bf16=False)
    else:
        chk(np.concatenate(got_s), np.concatenate(ref_s), f"{name} lse")


@pytest.mark.parametrize("name", ["tiny_fp32", "b16_small", "fp8_q2"])
def test_output_stage(M, name):
    w, heads = CASES[name]
    rows = w.batch * w.q_per_seq
    si = W.stage_inputs(w, rows)
    x = W.generate(w)
    dims = dims_of(M, w)
    o = torch.empty((rows, w.n_h, w.d_v), dtype=si["o_lat"].dtype, device="cuda")
    M.mla_out_proj(dims, rows, si["o_lat"].cuda(), x["w_uv"].cuda(), o)
    torch.cuda.synchronize()
    w_uv = x["w_uv"].double().numpy()
    lat = si["o_lat"].double().numpy()
    ref = np.einsum("hvc,thc->thv", w_uv, lat)
    got = o.float().cpu().numpy()
    chk = check_fp32 if w.act_dtype == "f32" else check_bf16
    chk(got, ref, f"{name} o")


@pytest.mark.parametrize("name", ["tiny_fp32", "b16_small", "fp8_q2"])
def test_absorb_stage(M, name):
    w, heads = CASES[name]
    x = W.generate(w)
    rows = w.batch * w.q_per_seq
    q = x["q"] if x["q"] is not None else torch.randn(rows, w.n_h, w.d_h + w.d_rope)
    pos = W.query_positions(x["seq_lens"], w.q_per_seq)
    dims = dims_of(M, w)
    qa = torch.empty((rows, w.n_h, w.d_c + w.d_rope), dtype=q.dtype, device="cuda")
    M.mla_absorb_q(dims, rows, q.cuda(), pos.cuda(), x["w_uk"].cuda(), qa)
    torch.cuda.synchronize()
    q64 = q.double().numpy()
    ref = np.concatenate([O.absorbed_query(q64[..., :w.d_h], x["w_uk"].double().numpy()),
                          O.rope(q64[..., w.d_h:], pos.numpy(), w.rope_theta)], axis=-1)
    chk = check_fp32 if w.act_dtype == "f32" else check_bf16
    chk(qa.float().cpu().numpy(), ref, f"{name} q_abs")
