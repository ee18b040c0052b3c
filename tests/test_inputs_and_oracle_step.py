"""Host-side checks of the seeded workloads and of the oracle's whole decode step."""
import math

import numpy as np
import pytest
import torch

import mla_inputs as W
from oracle import mla_oracle as O
from tests.oracle_io import oracle_inputs


def test_generation_is_deterministic_and_shaped():
    a = W.generate(W.TINY)
    b = W.generate(W.TINY)
    for k in ("w_dkv", "w_kr", "w_uk", "w_uv", "w_q", "new_h", "block_table"):
        assert torch.equal(a[k], b[k]), k
    w = W.TINY
    assert a["w_q"].shape == (w.n_h, w.d_h + w.d_rope, w.d_model)
    assert a["new_h"].shape == (37 + 128, w.d_model)
    assert a["cache"]["ckv"].shape == (a["num_pages"] * w.page_size, w.d_c + w.d_rope)
    # Every slot is a NaN sentinel before the tiny case appends all its tokens.
    assert torch.isnan(a["cache"]["ckv"]).all()
    # The block table is a permutation of the pool's pages.
    bt = a["block_table"]
    used = sorted(int(x) for x in bt.flatten() if x >= 0)
    assert used == list(range(a["num_pages"]))


def test_small_varlen_pool_sentinels():
    w = W.shrink(W.DSV2_VARLEN, batch=3, seq_len_range=(70, 200), pool_tokens=64 * 20,
                 d_model=64, n_h=2, d_h=8, d_v=8)
    x = W.generate(w)
    P = w.page_size
    ckv, bt = x["cache"]["ckv"], x["block_table"]
    for b in range(w.batch):
        L = int(x["seq_lens"][b])
        for t in range(L):
            row = ckv[int(bt[b, t // P]) * P + t % P]
            if t == L - 1:
                assert torch.isnan(row).all()       # appended by the decode step
            else:
                assert not torch.isnan(row).any()
    assert int(torch.isfinite(ckv[:, 0]).sum()) == int(x["seq_lens"].sum()) - w.batch


def test_outlier_fraction():
    w = W.shrink(W.DSV2_LONG, batch=2, seq_len=2000, d_model=64, n_h=2, d_h=8, d_v=8)
    x = W.generate(w)
    norms = x["cache"]["ckv"].float().abs().amax(dim=1)
    finite = norms[torch.isfinite(norms)]
    frac = float((finite > 6.0).float().mean())
    assert 0.005 < frac < 0.02


def test_oracle_step_on_tiny_workload():
    x = W.generate(W.TINY)
    inp = oracle_inputs(x)
    res = O.decode_step(inp)
    w = W.TINY
    assert set(res["rows"]) == {(0, 0), (1, 0)}
    for (b, j), r in res["rows"].items():
        assert r["o"].shape == (w.n_h, w.d_v)
        assert r["o_lat"].shape == (w.n_h, w.d_c)
        assert np.all(np.isfinite(r["o"]))
        # o = W_UV[h] (sum_t a_t c_t) for every head (value absorption).
        for h in range(w.n_h):
            np.testing.assert_allclose(r["o"][h], inp["w_uv"][h] @ r["o_lat"][h], atol=1e-12)
    # Appended entries: c_KV = W_DKV h for every token, stored as fp32.
    c_st = res["entries"][0]
    np.testing.assert_allclose(c_st, (inp["new_h"] @ inp["w_dkv"].T).astype(np.float32), atol=0)


def test_query_positions():
    pos = W.query_positions(torch.tensor([5, 9], dtype=torch.int32), 2)
    assert pos.tolist() == [3, 4, 7, 8]
