"""Each ABI stage on its own: the decode and output stages are fed seeded
stage inputs (not results of earlier GPU stages) and compared with the oracle."""
import numpy as np
import pytest
import torch

import mla_inputs as W
from oracle import mla_oracle as O
from tests.gpu_harness import DeviceRun, check_bf16, check_fp32, check_fp8, dims_of
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
    run = DeviceRun(M, x, num_splits=splits)
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
    g = torch.Generator().manual_seed(w.seed + 2000)
    q = x["q"] if x["q"] is not None else torch.randn(rows, w.n_h, w.d_h + w.d_rope, generator=g)
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


# Token counts that span two 128-token tiles with a ragged tail, and positions
# from 0 up to 2^23 - 1 (RoPE's single-precision angle reduction).
WIDE_POS = [0, 1, 2, 4095, 131071, (1 << 20) + 12345, (1 << 23) - 1]


@pytest.mark.parametrize("name,T", [("tiny_fp32", 7), ("b16_small", 64), ("b16_small", 200)])
def test_absorb_stage_many_tokens_and_large_positions(M, name, T):
    w, _ = CASES[name]
    x = W.generate(w)
    g = torch.Generator().manual_seed(w.seed + 3000 + T)
    dt = torch.float32 if w.act_dtype == "f32" else torch.bfloat16
    q = torch.randn(T, w.n_h, w.d_h + w.d_rope, generator=g).to(dt)
    pos = torch.tensor([WIDE_POS[i % len(WIDE_POS)] + 17 * (i // len(WIDE_POS)) for i in range(T)],
                       dtype=torch.int32).clamp_(max=(1 << 23) - 1)
    dims = dims_of(M, w)
    qa = torch.full((T, w.n_h, w.d_c + w.d_rope), float("nan"), dtype=dt, device="cuda")
    M.mla_absorb_q(dims, T, q.cuda(), pos.cuda(), x["w_uk"].cuda(), qa)
    torch.cuda.synchronize()
    q64 = q.double().numpy()
    ref = np.concatenate([O.absorbed_query(q64[..., :w.d_h], x["w_uk"].double().numpy()),
                          O.rope(q64[..., w.d_h:], pos.numpy(), w.rope_theta)], axis=-1)
    chk = check_fp32 if w.act_dtype == "f32" else check_bf16
    got = qa.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    chk(got[..., :w.d_c], ref[..., :w.d_c], f"{name} T={T} q_lat")
    chk(got[..., w.d_c:], ref[..., w.d_c:], f"{name} T={T} rotated q_rope")


@pytest.mark.parametrize("T", [64, 200, 300])
def test_output_stage_many_tokens(M, T):
    w, _ = CASES["b16_small"]
    x = W.generate(w)
    g = torch.Generator().manual_seed(w.seed + 4000 + T)
    lat = torch.randn(T, w.n_h, w.d_c, generator=g).to(torch.bfloat16)
    o = torch.full((T, w.n_h, w.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    M.mla_out_proj(dims_of(M, w), T, lat.cuda(), x["w_uv"].cuda(), o)
    torch.cuda.synchronize()
    ref = np.einsum("hvc,thc->thv", x["w_uv"].double().numpy(), lat.double().numpy())
    check_bf16(o.float().cpu().numpy(), ref, f"out-proj T={T}")


@pytest.mark.parametrize("name,T", [("tiny_fp32", 5), ("b16_small", 3), ("b16_small", 64), ("b16_small", 200),
                                    ("b16_small", 300)])
def test_out_proj_wo_stage(M, name, T):
    """W_UV then W_O in one call: o against W_UV o_lat, out against W_O applied to
    the heads of o joined in head order (the oracle fed o as the ABI stores it)."""
    w, _ = CASES[name]
    x = W.generate(w)
    w_o = W.output_weight(w)
    g = torch.Generator().manual_seed(w.seed + 6000 + T)
    dt = torch.float32 if w.act_dtype == "f32" else torch.bfloat16
    lat = torch.randn(T, w.n_h, w.d_c, generator=g).to(dt)
    dims = dims_of(M, w)
    o = torch.full((T, w.n_h, w.d_v), float("nan"), dtype=dt, device="cuda")
    out = torch.full((T, w.d_model), float("nan"), dtype=dt, device="cuda")
    ws_bytes = M.mla_out_proj_wo_workspace_size(dims, T)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.mla_out_proj_wo(dims, T, lat.cuda(), x["w_uv"].cuda(), w_o.cuda(), o, out, ws, ws_bytes, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref = np.einsum("hvc,thc->thv", x["w_uv"].double().numpy(), lat.double().numpy())
    o_st = O.round_to_storage(o_ref, w.act_dtype)
    out_ref = O.output_projection(o_st, w_o.double().numpy())
    chk = check_fp32 if w.act_dtype == "f32" else check_bf16
    chk(o.float().cpu().numpy(), o_ref, f"{name} T={T} o")
    chk(out.float().cpu().numpy(), out_ref, f"{name} T={T} out")
