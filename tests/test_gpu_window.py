"""Decode over a window (mla_decode_attn_window): each sequence's keys before
its start position are invisible, and the pages that hold only such keys are
freed (-1 in the block table) and must never be read. The decode stage is fed
seeded q_abs and compared with the oracle's attention over the window's keys."""
import numpy as np
import pytest
import torch

import mla_inputs as W
from oracle import mla_oracle as O
from tests.gpu_harness import DeviceRun, check_bf16, check_fp32, check_fp8
from tests.oracle_io import oracle_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import mla_latent_kv_80_b300 as M
    return M


CASES = {
    # (workload, window starts per sequence, heads checked)
    "bf16_page64": (W.shrink(W.DSV2_VARLEN, batch=7, seq_len_range=(60, 900), pool_tokens=64 * 120,
                             append_new=0), [0, 37, 64, 128, 10 ** 6, -4, None], [0, 41, 127]),
    "bf16_page16": (W.shrink(W.DSV2_VARLEN, batch=4, seq_len_range=(100, 500), page_size=16,
                             pool_tokens=16 * 200, append_new=0), [5, 16, 200, None], [3, 100]),
    "fp8_q2": (W.shrink(W.DSV2_FP8_Q2, batch=3, seq_len=333, append_new=0), [100, 331, 0], [0, 77]),
    "tiny_fp32": (W.shrink(W.TINY, append_new=0), [20, 127], None),
}


def _starts(x, spec):
    """Window starts: None stands for 'the last key only' (seq_len - 1)."""
    lens = x["seq_lens"].tolist()
    return [L - 1 if s is None else s for s, L in zip(spec, lens)]


def _free_pages_before(x, w, starts):
    """Marks the block-table entries of pages wholly before each start as freed."""
    bt = x["block_table"].clone()
    for b, s in enumerate(starts):
        n = max(0, s) // w.page_size
        bt[b, :min(n, bt.shape[1])] = -1
    return bt


def _check(w):
    if w.act_dtype == "f32":
        return check_fp32
    return check_fp8 if w.cache_dtype == "fp8_e4m3" else check_bf16


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("splits", [0, 1, 5])
def test_window_decode_matches_oracle(M, name, splits):
    w, spec, heads = CASES[name]
    x = W.generate(w)
    starts = _starts(x, spec)
    inp = oracle_inputs(x)  # the oracle gathers through the original table
    x = dict(x)
    x["block_table"] = _free_pages_before(x, w, starts)
    run = DeviceRun(M, x, num_splits=splits)
    rows = w.batch * w.q_per_seq
    qa = W.stage_inputs(w, rows)["q_abs"]
    run.step.q_abs.copy_(qa.cuda())
    run.step.status.zero_()
    st = torch.tensor(starts, dtype=torch.int32, device="cuda")
    run.step.decode(run.cache, run.bt, run.seq_lens, seq_start=st)
    torch.cuda.synchronize()
    assert int(run.step.status.item()) == 0, "a freed page was read or a wait gave up"
    o_lat = run.step.o_lat.float().cpu().numpy()
    lse = run.step.lse.cpu().numpy()
    qa64 = qa.double().numpy()
    heads = list(range(w.n_h)) if heads is None else heads
    got_l, ref_l, got_s, ref_s = [], [], [], []
    for b in range(w.batch):
        L = int(x["seq_lens"][b])
        c, kr = O.gather_sequence(inp["cache"], w.cache_dtype, inp["block_table"], b, L, w.page_size, w.d_c)
        for j in range(w.q_per_seq):
            vis = max(L - w.q_per_seq + j + 1, 0)
            lo = min(max(starts[b], 0), vis)
            row = b * w.q_per_seq + j
            lat, l = O.absorbed_attention(qa64[row, heads], c[lo:vis], kr[lo:vis], w.softmax_scale)
            if lo == vis:
                assert np.all(lse[row, heads] == -np.inf) and not np.any(o_lat[row, heads])
                continue
            got_l.append(o_lat[row, heads]); ref_l.append(lat)
            got_s.append(lse[row, heads]); ref_s.append(l)
    chk = _check(w)
    chk(np.concatenate(got_l), np.concatenate(ref_l), f"{name} window o_lat")
    if chk is check_bf16:
        check_bf16(np.concatenate(got_s), np.concatenate(ref_s), f"{name} window lse", stored_bf16=False)
    else:
        chk(np.concatenate(got_s), np.concatenate(ref_s), f"{name} window lse")


def test_window_of_one_key_is_that_key_exactly(M):
    """A window holding only the last key: softmax weight 1, o_lat is its latent."""
    w = W.shrink(W.DSV2_B16, batch=3, seq_len=300, append_new=0)
    x = W.generate(w)
    run = DeviceRun(M, x)
    run.step.q_abs.copy_(W.stage_inputs(w, w.batch)["q_abs"].cuda())
    run.step.status.zero_()
    st = (run.seq_lens - 1).to(torch.int32)
    run.step.decode(run.cache, run.bt, run.seq_lens, seq_start=st)
    torch.cuda.synchronize()
    assert int(run.step.status.item()) == 0
    o_lat = run.step.o_lat.float().cpu().numpy()
    for b in range(w.batch):
        slot = int(x["block_table"][b, 299 // w.page_size]) * w.page_size + 299 % w.page_size
        c = x["cache"]["ckv"][slot, :w.d_c].float().numpy()
        np.testing.assert_array_equal(o_lat[b], np.broadcast_to(c, o_lat[b].shape))
