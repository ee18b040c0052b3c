"""Pins for the CPU oracle: values, identities and library routines it must agree with.

Each test ties the oracle to something other than itself: numbers the MLA
pages print, closed forms, identities the pages state (absorption, RoPE
relativity), brute force on tiny inputs, or an independent library routine.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import e4m3
from oracle import mla_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- worked example
def test_dgblog_worked_example_projections():
    g = load("worked_example_dgblog.json")
    c = O.joint_kv_latent(np.array([g["h"]]), np.array(g["W_DKV"]))[0]
    assert c.tolist() == g["c_KV"]
    k = O.up_project(c[None], np.array(g["W_UK"]))[0]
    v = O.up_project(c[None], np.array(g["W_UV"]))[0]
    assert k.tolist() == g["k"]
    assert v.tolist() == g["v"]
    assert (len(k) + len(v)) / len(c) == g["compression_ratio"]


def test_dgblog_worked_example_single_token_attention():
    """One cached token: the softmax weight is 1, so o = W_UV c exactly."""
    g = load("worked_example_dgblog.json")
    c = np.array([g["c_KV"]], dtype=np.float64)
    w_uk = np.array(g["W_UK"], dtype=np.float64)
    w_uv = np.array(g["W_UV"], dtype=np.float64)
    q = np.array([0.3, -1.0, 2.0])
    o, a, lse, lat = O.attend_head(q, np.zeros(0), c, np.zeros((1, 0)), w_uk, w_uv, 0.5)
    assert a.tolist() == [1.0]
    assert o.tolist() == g["v"]
    assert lat.tolist() == g["c_KV"]
    assert lse == pytest.approx(0.5 * float(np.dot(q, g["k"])), abs=1e-15)


# ---------------------------------------------------------------- cache sizes
def test_cache_element_counts():
    g = load("cache_sizes.json")
    n_h, d_h, d_c, d_r = g["n_h"], g["d_h"], g["d_c"], g["d_rope"]
    assert d_c + d_r == g["mla_elements_per_token_layer"]
    assert 2 * n_h * d_h == g["mha_elements_per_token_layer"]
    assert n_h * (d_h + d_r + d_h) == g["mha_equivalent_with_rope_and_v"]
    assert 2 * 2 * n_h * d_h == g["mha_bytes_bf16_per_token_layer"]
    assert 2 * 8 * 128 * 80 * 2 == g["llama2_70b_gqa_bytes_per_token"]
    assert (d_c + d_r) / (2 * d_h) == g["gqa_equivalent_groups"]
    assert round(100 * (d_c + d_r) / (2 * n_h * d_h), 1) == 1.8
    # The oracle reads exactly d_c + d_rope values per cached token.
    pool = {"ckv": rng.standard_normal((4, d_c + d_r)).astype(np.float32)}
    c, kr = O.gather_sequence(pool, "f32", np.array([[0]]), 0, 3, 4, d_c)
    assert c.shape[1] + kr.shape[1] == g["mla_elements_per_token_layer"]


# ---------------------------------------------------------------- absorption identities
def _random_head(L=37, d_h=8, d_c=12, d_r=4, d_v=6):
    return dict(q_nope=rng.standard_normal(d_h), q_r=rng.standard_normal(d_r),
                c=rng.standard_normal((L, d_c)), kr=rng.standard_normal((L, d_r)),
                w_uk=rng.standard_normal((d_h, d_c)), w_uv=rng.standard_normal((d_v, d_c)))


def test_key_absorption_matches_explicit_scores():
    """score = q^T (W_UK c) = (W_UK^T q)^T c ("第二步，推理时的吸收")."""
    x = _random_head()
    scale = 0.3
    o, a, lse, lat = O.attend_head(x["q_nope"], x["q_r"], x["c"], x["kr"], x["w_uk"], x["w_uv"], scale)
    q_lat = x["w_uk"].T @ x["q_nope"]
    s_abs = scale * (x["c"] @ q_lat + x["kr"] @ x["q_r"])
    a_abs = np.exp(s_abs - s_abs.max())
    a_abs /= a_abs.sum()
    np.testing.assert_allclose(a, a_abs, rtol=0, atol=1e-12)
    m = s_abs.max()
    assert lse == pytest.approx(m + math.log(np.exp(s_abs - m).sum()), abs=1e-12)


def test_value_absorption_matches_explicit_output():
    """o = sum_j a_j W_UV c_j = W_UV (sum_j a_j c_j)."""
    x = _random_head()
    o, a, lse, lat = O.attend_head(x["q_nope"], x["q_r"], x["c"], x["kr"], x["w_uk"], x["w_uv"], 0.7)
    np.testing.assert_allclose(o, x["w_uv"] @ (a @ x["c"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lat, a @ x["c"], rtol=0, atol=1e-12)


def test_absorbed_query_is_transpose_product_per_head():
    w_uk = rng.standard_normal((3, 5, 7))
    q = rng.standard_normal((2, 3, 5))
    got = O.absorbed_query(q, w_uk)
    for t in range(2):
        for h in range(3):
            np.testing.assert_allclose(got[t, h], w_uk[h].T @ q[t, h], atol=1e-13)


# ---------------------------------------------------------------- RoPE
def test_rope_closed_form_values():
    one = O.rope(np.array([[1.0, 0.0]]), [1])[0]
    np.testing.assert_allclose(one, [math.cos(1), math.sin(1)], atol=1e-15)
    two = O.rope(np.array([[0.0, 1.0]]), [1])[0]
    np.testing.assert_allclose(two, [-math.sin(1), math.cos(1)], atol=1e-15)
    # Pair i=1 of a 4-wide key turns at 10000^(-2/4) = 0.01 rad per position.
    third = O.rope(np.array([[0.0, 0.0, 1.0, 0.0]]), [100])[0]
    np.testing.assert_allclose(third, [0, 0, math.cos(1), math.sin(1)], atol=1e-13)
    # theta^(-2i/d) at the last pair of a 64-wide key.
    ang = O.rope_angles([1], 64)[0]
    assert ang[31] == pytest.approx(10000.0 ** (-62 / 64), rel=1e-15)


def test_rope_position_zero_is_identity_and_preserves_norm():
    x = rng.standard_normal((5, 64))
    np.testing.assert_array_equal(O.rope(x, [0] * 5), x)
    y = O.rope(x, [3, 77, 4095, 65536, 131071])
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_scores_depend_only_on_relative_position():
    """(R_i q)^T (R_j k) = q^T R_{j-i} k: shifting every position leaves scores alone."""
    q = rng.standard_normal(64)
    k = rng.standard_normal((20, 64))
    pos_k = np.arange(20) * 37
    pos_q = 1000
    base = O.rope(k, pos_k) @ O.rope(q[None], [pos_q])[0]
    for delta in (1, 1000, 123457):
        shifted = O.rope(k, pos_k + delta) @ O.rope(q[None], [pos_q + delta])[0]
        np.testing.assert_allclose(shifted, base, rtol=0, atol=1e-10 * np.abs(base).max())


# ---------------------------------------------------------------- softmax attention
def test_matches_library_einsum_formulation_without_rope():
    """With d_rope = 0 the explicit oracle equals torch's einsum/softmax attention in float64."""
    B, L, H, d_c, d = 2, 11, 3, 6, 4
    c = rng.standard_normal((B, L, d_c))
    q = rng.standard_normal((B, 1, H, d))
    w_uk = rng.standard_normal((H, d, d_c))
    w_uv = rng.standard_normal((H, d, d_c))
    tc = torch.from_numpy(c)
    k = torch.einsum("hdc,blc->blhd", torch.from_numpy(w_uk), tc)
    v = torch.einsum("hdc,blc->blhd", torch.from_numpy(w_uv), tc)
    scores = torch.einsum("bqhd,bkhd->bhqk", torch.from_numpy(q), k) / math.sqrt(d)
    ref = torch.einsum("bhqk,bkhd->bqhd", torch.softmax(scores, dim=-1), v).numpy()
    for b in range(B):
        r = O.decode_rows(q[b, 0], np.zeros((H, 0)), 5, c[b], np.zeros((L, 0)), w_uk, w_uv,
                          1 / math.sqrt(d))
        np.testing.assert_allclose(r["o"], ref[b, 0], rtol=0, atol=1e-12)


def test_hand_computed_two_token_case():
    """Scores 0 and ln 3 give weights 1/4, 3/4; W_UV = 2 gives o = 1.5 ln 3."""
    c = np.array([[0.0], [math.log(3.0)]])
    o, a, lse, _ = O.attend_head(np.array([1.0]), np.zeros(0), c, np.zeros((2, 0)),
                                 np.array([[1.0]]), np.array([[2.0]]), 1.0)
    np.testing.assert_allclose(a, [0.25, 0.75], atol=1e-15)
    assert o[0] == pytest.approx(1.5 * math.log(3.0), abs=1e-15)
    assert lse == pytest.approx(math.log(4.0), abs=1e-15)


def test_hand_computed_rope_only_score():
    """q_nope = 0: the score is the RoPE part alone, cos(1) against a key at position 0."""
    c = np.array([[1.0], [-1.0]])
    kr = np.array([[1.0, 0.0], [0.0, 0.0]])
    r = O.decode_rows(np.zeros((1, 1)), np.array([[1.0, 0.0]]), 1, c, kr,
                      np.ones((1, 1, 1)), np.ones((1, 1, 1)), 1.0)
    e = math.exp(math.cos(1.0))
    expect = (e * 1.0 + 1.0 * -1.0) / (e + 1.0)
    assert r["o"][0, 0] == pytest.approx(expect, abs=1e-15)
    assert r["lse"][0] == pytest.approx(math.log(e + 1.0), abs=1e-15)


def test_lse_matches_scipy_and_weights_sum_to_one():
    from scipy.special import logsumexp
    x = _random_head(L=200)
    for scale in (0.1, 3.0):
        o, a, lse, _ = O.attend_head(x["q_nope"], x["q_r"], x["c"], x["kr"], x["w_uk"], x["w_uv"], scale)
        s = scale * ((x["c"] @ x["w_uk"].T) @ x["q_nope"] + x["kr"] @ x["q_r"])
        assert lse == pytest.approx(logsumexp(s), abs=1e-12)
        assert a.sum() == pytest.approx(1.0, abs=1e-14)


def test_empty_key_set():
    o, a, lse, lat = O.attend_head(np.ones(2), np.ones(2), np.zeros((0, 3)), np.zeros((0, 2)),
                                   np.ones((2, 3)), np.ones((4, 3)), 1.0)
    assert lse == -math.inf and not o.any() and o.shape == (4,)


def test_causal_second_query_sees_one_more_key():
    """q = 2: query 0 sits at L-2 and must not see the key at L-1."""
    L, d_c, d_r = 6, 4, 2
    c = rng.standard_normal((L, d_c))
    kr = np.zeros((L, d_r))
    c[L - 1] = 50.0  # a key that would dominate if it were visible
    w = np.eye(d_c)[None]
    r0 = O.decode_rows(np.ones((1, d_c)), np.zeros((1, d_r)), L - 2, c[:L - 1], kr[:L - 1], w, w, 1.0)
    assert np.all(np.abs(r0["o"]) < 10)
    r1 = O.decode_rows(np.ones((1, d_c)), np.zeros((1, d_r)), L - 1, c, kr, w, w, 1.0)
    np.testing.assert_allclose(r1["o"][0], c[L - 1], atol=1e-12)


# ---------------------------------------------------------------- paged addressing
def test_slot_index_by_hand():
    bt = np.array([[3, 0, -1], [1, 2, 4]])
    assert O.slot_index(bt, 0, 0, 16) == 48
    assert O.slot_index(bt, 0, 17, 16) == 1
    assert O.slot_index(bt, 1, 15, 16) == 31
    assert O.slot_index(bt, 1, 40, 16) == 72
    np.testing.assert_array_equal(O.slot_index(bt, 1, [0, 16, 32], 16), [16, 32, 64])


def test_gather_follows_block_table():
    P, d = 4, 3
    pool = np.arange(5 * P * d, dtype=np.float32).reshape(5 * P, d)
    bt = np.array([[2, 4]])
    c, kr = O.gather_sequence({"ckv": pool}, "f32", bt, 0, 6, P, 2)
    np.testing.assert_array_equal(c[:, 0], pool[[8, 9, 10, 11, 16, 17], 0])
    np.testing.assert_array_equal(kr[:, 0], pool[[8, 9, 10, 11, 16, 17], 2])


# ---------------------------------------------------------------- storage formats
def test_bf16_rounding_matches_torch_cast():
    x = rng.standard_normal(100000).astype(np.float32) * np.exp(rng.uniform(-20, 20, 100000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_bf16(x), ref)


def test_bf16_bits_decode():
    t = torch.tensor([1.0, -2.5, 3.140625, 0.0], dtype=torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(O.bf16_bits_to_f64(bits), [1.0, -2.5, 3.140625, 0.0])


def test_e4m3_known_codes():
    assert e4m3.decode_code(0x7E) == 448.0
    assert e4m3.decode_code(0x08) == 2.0 ** -6
    assert e4m3.decode_code(0x01) == 2.0 ** -9
    assert e4m3.decode_code(0x38) == 1.0
    assert e4m3.decode_code(0xB8) == -1.0
    assert math.isnan(e4m3.decode_code(0x7F)) and math.isnan(e4m3.decode_code(0xFF))
    assert e4m3.decode_code(0x77) == 240.0  # exponent 14, mantissa 7: 1.875 * 2^7


def test_e4m3_rounding_ties_and_saturation():
    enc = e4m3.encode_satfinite_rne
    assert enc(np.array([1.0625]))[0] == 0x38     # tie between 1.0 (even) and 1.125
    assert enc(np.array([1.1875]))[0] == 0x3A     # tie between 1.125 and 1.25 (even)
    assert enc(np.array([1.07]))[0] == 0x39
    assert enc(np.array([460.0]))[0] == 0x7E      # saturates to 448
    assert enc(np.array([1e30]))[0] == 0x7E
    assert enc(np.array([-1e30]))[0] == 0xFE
    assert enc(np.array([2.0 ** -10]))[0] == 0x00  # tie between 0 (even) and 2^-9
    assert enc(np.array([3 * 2.0 ** -10]))[0] == 0x02  # tie between 2^-9 and 2^-8 (even)


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    np.testing.assert_array_equal(e4m3.encode_satfinite_rne(e4m3.decode(codes)), codes)


def test_e4m3_matches_library_cast_on_every_bf16_value_in_range():
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 448.0)]
    ref = torch.from_numpy(vals.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = e4m3.encode_satfinite_rne(vals)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_matches_library_cast_on_random_fp32():
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(e4m3.encode_satfinite_rne(x), ref)


def test_quantize_rows_recipe():
    x = rng.standard_normal((50, 512)).astype(np.float32)
    codes, scale = e4m3.quantize_rows(x)
    amax = np.abs(x).max(axis=1)
    np.testing.assert_array_equal(scale, (amax / np.float32(448)).astype(np.float32))
    # The largest element maps to +-448 (code 0x7E or 0xFE).
    i = np.abs(x).argmax(axis=1)
    assert set((codes[np.arange(50), i] & 0x7F).tolist()) == {0x7E}
    deq = e4m3.dequantize_rows(codes, scale)
    # Half a step of the top binade [256, 448] is 16, i.e. 16/448 of amax.
    assert np.max(np.abs(deq - x) / amax[:, None]) <= 16 / 448 * (1 + 1e-6)
    z, zs = e4m3.quantize_rows(np.zeros((1, 8), np.float32))
    assert zs[0] == 1.0 and not z.any()


# ---------------------------------------------------------------- append entries
def test_append_entries_definitions():
    h = rng.standard_normal((3, 16))
    w_dkv = rng.standard_normal((8, 16))
    w_kr = rng.standard_normal((4, 16))
    c, kr, _, _ = O.append_entries(h, w_dkv, w_kr, [0, 5, 9], "f32")
    np.testing.assert_allclose(c, (h @ w_dkv.T).astype(np.float32), rtol=0, atol=0)
    # Position 0: RoPE is the identity.
    np.testing.assert_allclose(kr[0], (w_kr @ h[0]).astype(np.float32), rtol=0, atol=0)
    # Position 5 rotates pair 0 by 5 rad.
    raw = w_kr @ h[1]
    assert kr[1][0] == pytest.approx(raw[0] * math.cos(5) - raw[1] * math.sin(5), rel=1e-6)


# ---------------------------------------------------------------- planted mistakes
def test_pins_catch_a_wrong_output_index_in_up_projection(monkeypatch):
    monkeypatch.setattr(O, "up_project", lambda c, w: (np.asarray(c) @ np.asarray(w).T)[..., ::-1])
    with pytest.raises(AssertionError):
        test_dgblog_worked_example_projections()


def test_pins_catch_a_flipped_rope_sign(monkeypatch):
    real = O.rope_angles
    monkeypatch.setattr(O, "rope_angles", lambda pos, d, theta=10000.0: -real(pos, d, theta))
    with pytest.raises(AssertionError):
        test_rope_closed_form_values()


def test_pins_catch_a_dropped_rope_term(monkeypatch):
    real = O.attend_head
    monkeypatch.setattr(O, "attend_head",
                        lambda qn, qr, c, kr, wuk, wuv, s: real(qn, np.zeros_like(qr), c, kr, wuk, wuv, s))
    with pytest.raises(AssertionError):
        test_hand_computed_rope_only_score()


def test_absorbed_attention_equals_explicit_form():
    """The latent-space attention the GPU runs equals the explicit form (both identities)."""
    H, L, d_h, d_c, d_r, d_v = 4, 50, 8, 12, 4, 6
    q_nope = rng.standard_normal((H, d_h))
    q_rot = rng.standard_normal((H, d_r))
    c = rng.standard_normal((L, d_c))
    kr = rng.standard_normal((L, d_r))
    w_uk = rng.standard_normal((H, d_h, d_c))
    w_uv = rng.standard_normal((H, d_v, d_c))
    q_abs = np.concatenate([O.absorbed_query(q_nope, w_uk), q_rot], axis=1)
    lat, lse = O.absorbed_attention(q_abs, c, kr, 0.4)
    for h in range(H):
        o, a, l, lat_h = O.attend_head(q_nope[h], q_rot[h], c, kr, w_uk[h], w_uv[h], 0.4)
        np.testing.assert_allclose(lat[h], lat_h, atol=1e-12)
        np.testing.assert_allclose(w_uv[h] @ lat[h], o, atol=1e-12)
        assert lse[h] == pytest.approx(l, abs=1e-12)


def test_stage_results_with_f32_storage_match_end_to_end():
    x = _random_head(L=40)
    w_uk = rng.standard_normal((3, 8, 12))
    w_uv = rng.standard_normal((3, 6, 12))
    r = O.decode_rows(rng.standard_normal((3, 8)), rng.standard_normal((3, 4)), 7, x["c"], x["kr"],
                      w_uk, w_uv, 0.3, act_dtype="f32")
    np.testing.assert_allclose(r["o_lat_s"], r["o_lat"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(r["o_s"], r["o"], rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------- query projection
def test_query_projection_equals_linear_then_head_view_without_rope():
    """With d_rope = 0 the per-head query is page 3's listing: one nn.Linear of
    width n_heads * d_n applied to x, then viewed as [.., n_heads, d_n] ("MLA 是什么
    | dg's Blog", "完整代码"). torch's linear and view are the independent side."""
    T, n_h, d, d_model = 5, 4, 6, 10
    x = rng.standard_normal((T, d_model))
    w_full = rng.standard_normal((n_h * d, d_model))  # nn.Linear weight [out x in]
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(w_full)).view(T, n_h, d)
    q_nope, q_rope = O.query_projection(x, w_full.reshape(n_h, d, d_model), d)
    assert q_rope.shape == (T, n_h, 0)
    np.testing.assert_allclose(q_nope, ref.numpy(), rtol=0, atol=1e-12)


def test_query_projection_splits_nope_then_rope_per_head():
    """Each head's d_h + d_rope outputs are [q_nope ; q_rope] in that order, and
    head h owns outputs h*(d_h+d_rope) .. of the full projection. Hand-built
    weights: output o of head h reads input (3h + o) mod 4 with gain 10h + o + 1."""
    n_h, d_h, d_rope, d_model = 2, 2, 1, 4
    w_q = np.zeros((n_h, d_h + d_rope, d_model))
    for h in range(n_h):
        for o in range(d_h + d_rope):
            w_q[h, o, (3 * h + o) % 4] = 10 * h + o + 1
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    q_nope, q_rope = O.query_projection(x, w_q, d_h)
    # head 0: outputs read x0*1, x1*2, x2*3; head 1: x3*11, x0*12, x1*13
    assert q_nope[0].tolist() == [[1.0, 4.0], [44.0, 12.0]]
    assert q_rope[0].tolist() == [[9.0], [26.0]]


def test_pins_catch_swapped_nope_and_rope(monkeypatch):
    real = O.query_projection

    def swapped(h, w_q, d_h):
        qn, qr = real(h, w_q, d_h)
        return np.concatenate([qr, qn], axis=-1)[..., :d_h], np.concatenate([qr, qn], axis=-1)[..., d_h:]

    monkeypatch.setattr(O, "query_projection", swapped)
    with pytest.raises(AssertionError):
        test_query_projection_splits_nope_then_rope_per_head()


# ---------------------------------------------------------------- output projection W_O
def test_output_projection_equals_linear_on_joined_heads():
    """Page 3's listing: out.reshape(batch, seq, -1) then self.W_O(out); torch's
    linear on the head-major joined vector is the independent side."""
    T, n_h, d_v, d_model = 4, 3, 5, 7
    o = rng.standard_normal((T, n_h, d_v))
    w_o = rng.standard_normal((d_model, n_h * d_v))
    ref = torch.nn.functional.linear(torch.from_numpy(o).reshape(T, -1), torch.from_numpy(w_o))
    np.testing.assert_allclose(O.output_projection(o, w_o), ref.numpy(), rtol=0, atol=1e-12)


def test_output_projection_joins_heads_in_head_order():
    """Two heads of width 2: W_O picks input k = 2h + i with gain k + 1, so
    output k reads head k // 2, component k % 2."""
    o = np.array([[[1.0, 2.0], [3.0, 4.0]]])
    w_o = np.diag([1.0, 2.0, 3.0, 4.0])
    assert O.output_projection(o, w_o).tolist() == [[1.0, 4.0, 9.0, 16.0]]


def test_pins_catch_heads_joined_in_the_wrong_order(monkeypatch):
    real = O.output_projection
    monkeypatch.setattr(O, "output_projection", lambda o, w: real(np.swapaxes(o, 1, 2), w))
    with pytest.raises(AssertionError):
        test_output_projection_joins_heads_in_head_order()


# ---------------------------------------------------------------- decode over a window
def _window_inputs(L=9, B=2):
    """A small generated workload (fp32) for the windowed decode step."""
    import mla_inputs as W
    from tests.oracle_io import oracle_inputs
    w = W.shrink(W.TINY, batch=B, seq_lens=tuple([L] * B), append_new=1, block_table="contiguous")
    x = W.generate(w)
    inp = oracle_inputs(x)
    inp["q"] = np.asarray(np.random.default_rng(5).standard_normal((B, w.n_h, w.d_h + w.d_rope)))
    return w, x, inp


def test_window_start_zero_is_the_full_attention():
    w, x, inp = _window_inputs()
    full = O.decode_step(inp)["rows"]
    win = O.decode_step(inp, seq_start=[0, -3])["rows"]
    for k in full:
        np.testing.assert_array_equal(full[k]["o_lat"], win[k]["o_lat"])


def test_window_matches_library_softmax_over_the_window_keys():
    """torch's softmax attention restricted to the keys at positions >= start."""
    w, x, inp = _window_inputs(L=11)
    start = [4, 10]
    got = O.decode_step(inp, seq_start=start)["rows"]
    for b in range(w.batch):
        L = int(x["seq_lens"][b])
        c, kr = O.gather_sequence(inp["cache"], "f32", inp["block_table"], b, L, w.page_size, w.d_c)
        ent = O.append_entries(inp["new_h"], inp["w_dkv"], inp["w_kr"], inp["new_pos"], "f32")
        mine = np.nonzero(inp["new_seq_idx"] == b)[0]
        c, kr = O.overwrite_positions(c, kr, inp["new_pos"][mine], ent, mine)
        q_abs = got[(b, 0)]["q_abs"]
        keys = torch.from_numpy(np.concatenate([c, kr], axis=1)[start[b]:L])
        s = w.softmax_scale * torch.from_numpy(q_abs) @ keys.T
        ref = torch.softmax(s, dim=-1) @ torch.from_numpy(c[start[b]:L])
        np.testing.assert_allclose(got[(b, 0)]["o_lat"], ref.numpy(), rtol=0, atol=1e-12)


def test_window_of_one_key_returns_that_key():
    w, x, inp = _window_inputs(L=7)
    r = O.decode_step(inp, seq_start=[6, 7])["rows"]
    ent = O.append_entries(inp["new_h"], inp["w_dkv"], inp["w_kr"], inp["new_pos"], "f32")
    # position 6 is the token the step appended for sequence 0
    k = int(np.nonzero((inp["new_seq_idx"] == 0) & (inp["new_pos"] == 6))[0][0])
    np.testing.assert_allclose(r[(0, 0)]["o_lat"], np.broadcast_to(ent[0][k], r[(0, 0)]["o_lat"].shape),
                               rtol=0, atol=1e-12)
    # a start past the query's position leaves no keys
    assert np.all(r[(1, 0)]["lse"] == -np.inf) and not np.any(r[(1, 0)]["o_lat"])


def test_pins_catch_a_window_off_by_one(monkeypatch):
    real = O.decode_rows
    monkeypatch.setattr(O, "decode_rows", lambda qn, qr, p, c, kr, *a, **k: real(qn, qr, p, c[1:], kr[1:], *a, **k))
    with pytest.raises(AssertionError):
        test_window_of_one_key_returns_that_key()


# ---------------------------------------------------------------- chunked prefill (explicit form)
def _prefill_case(C=5, L=9, d_h=8, d_r=4, d_c=12, d_v=6, seed=7):
    g = np.random.default_rng(seed)
    q_n = g.standard_normal((C, d_h))
    q_r = g.standard_normal((C, d_r))
    c = g.standard_normal((L, d_c))
    kr = g.standard_normal((L, d_r))
    w_uk = g.standard_normal((d_h, d_c)) / math.sqrt(d_c)
    w_uv = g.standard_normal((d_v, d_c)) / math.sqrt(d_c)
    pos = L - C + np.arange(C)
    return q_n, q_r, pos, c, kr, w_uk, w_uv


def test_prefill_matches_library_causal_attention():
    """torch's scaled_dot_product_attention on the explicit keys [W_UK c ; k_R]
    and values W_UV c, with a mask that lets query i see keys up to its position."""
    q_n, q_r, pos, c, kr, w_uk, w_uv = _prefill_case()
    scale = 0.37
    o, lse = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, scale)
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    q = torch.cat([t(q_n), t(q_r)], 1)[None, None]
    k = torch.cat([t(c) @ t(w_uk).T, t(kr)], 1)[None, None]
    v = (t(c) @ t(w_uv).T)[None, None]
    mask = torch.arange(c.shape[0])[None, :] <= torch.from_numpy(pos)[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)[0, 0]
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)
    s = (q[0, 0] @ k[0, 0].T) * scale
    ref_lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_prefill_rows_equal_single_query_attention():
    """Each query of the chunk equals one explicit decode over the keys up to its position."""
    q_n, q_r, pos, c, kr, w_uk, w_uv = _prefill_case(C=4, L=7)
    o, lse = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, 0.5)
    for i, p in enumerate(pos):
        oh, _, lh, _ = O.attend_head(q_n[i], q_r[i], c[:p + 1], kr[:p + 1], w_uk, w_uv, 0.5)
        np.testing.assert_allclose(o[i], oh, rtol=1e-12, atol=1e-13)
        assert abs(lse[i] - lh) < 1e-12


def test_prefill_first_query_of_a_fresh_sequence_returns_its_own_value():
    """A sequence prefilled from empty: query 0 sees only key 0, so o = W_UV c_0 and
    lse = its one score; query 1 mixes two values with the logistic weight."""
    q_n, q_r, _, c, kr, w_uk, w_uv = _prefill_case(C=2, L=2)
    pos = np.array([0, 1])
    o, lse = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, 1.0)
    v = c @ w_uv.T
    s = np.array([[q_n[i] @ (w_uk @ c[t]) + q_r[i] @ kr[t] for t in range(2)] for i in range(2)])
    np.testing.assert_allclose(o[0], v[0], rtol=1e-13)
    assert abs(lse[0] - s[0, 0]) < 1e-13
    a1 = 1.0 / (1.0 + math.exp(s[1, 0] - s[1, 1]))
    np.testing.assert_allclose(o[1], (1 - a1) * v[0] + a1 * v[1], rtol=1e-12)


def test_prefill_is_causal():
    """Changing the keys after a query's position leaves its row alone; changing
    the key at its position does not."""
    q_n, q_r, pos, c, kr, w_uk, w_uv = _prefill_case(C=4, L=8)
    o0, _ = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, 0.5)
    c2, kr2 = c.copy(), kr.copy()
    c2[pos[1] + 1:] += 3.0
    kr2[pos[1] + 1:] -= 2.0
    o1, _ = O.explicit_prefill_head(q_n, q_r, pos, c2, kr2, w_uk, w_uv, 0.5)
    np.testing.assert_array_equal(o1[:2], o0[:2])
    assert np.max(np.abs(o1[2:] - o0[2:])) > 1e-3


def test_prefill_query_before_every_key_sees_nothing():
    q_n, q_r, _, c, kr, w_uk, w_uv = _prefill_case(C=3, L=2)
    pos = np.array([-1, 0, 1])                      # a chunk longer than the sequence
    o, lse = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, 0.5)
    assert np.all(o[0] == 0) and lse[0] == -math.inf
    assert np.isfinite(lse[1:]).all()


def test_prefill_storage_hook_rounds_what_it_says():
    """With f32 storage every formed quantity is rounded to fp32 only: the
    result moves by fp32 rounding, not more; with bf16 by about bf16's."""
    q_n, q_r, pos, c, kr, w_uk, w_uv = _prefill_case(C=6, L=40, d_h=32, d_c=64, d_v=32)
    o, _ = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, 0.3)
    o32, _ = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, 0.3,
                                     store=lambda x: O.round_to_storage(x, "f32"))
    o16, _ = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, 0.3,
                                     store=lambda x: O.round_to_storage(x, "bf16"))
    e32 = np.max(np.abs(o32 - o)) / np.max(np.abs(o))
    e16 = np.max(np.abs(o16 - o)) / np.max(np.abs(o))
    assert 0 < e32 < 1e-6 and 1e-5 < e16 < 3e-2


def test_pins_catch_a_causal_off_by_one(monkeypatch):
    real = O.explicit_prefill_head
    monkeypatch.setattr(O, "explicit_prefill_head",
                        lambda qn, qr, pos, *a, **k: real(qn, qr, np.asarray(pos) - 1, *a, **k))
    with pytest.raises(AssertionError):
        test_prefill_matches_library_causal_attention()


def test_pins_catch_values_formed_with_the_key_weight(monkeypatch):
    real = O.explicit_prefill_head
    monkeypatch.setattr(O, "explicit_prefill_head",
                        lambda qn, qr, pos, c, kr, wuk, wuv, *a, **k: real(qn, qr, pos, c, kr, wuk, wuk[:wuv.shape[0]],
                                                                         *a, **k))
    with pytest.raises(AssertionError):
        test_prefill_matches_library_causal_attention()


def test_prefill_window_matches_library_attention_over_the_window():
    """With a first visible position lo, query i sees keys lo .. q_pos[i]: the
    library's causal attention with that window mask; lo = 0 is the full form."""
    q_n, q_r, pos, c, kr, w_uk, w_uv = _prefill_case(C=6, L=14)
    lo, scale = 5, 0.4
    o, lse = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, scale, lo=lo)
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    q = torch.cat([t(q_n), t(q_r)], 1)[None, None]
    k = torch.cat([t(c) @ t(w_uk).T, t(kr)], 1)[None, None]
    v = (t(c) @ t(w_uv).T)[None, None]
    kp = torch.arange(c.shape[0])[None, :]
    mask = (kp <= torch.from_numpy(pos)[:, None]) & (kp >= lo)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)[0, 0]
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)
    full, _ = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, scale, lo=0)
    base, _ = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, scale)
    np.testing.assert_array_equal(full, base)


def test_prefill_window_ignores_evicted_keys():
    """Keys before the window change nothing (they may be gone); a query whose
    position is before the window sees no key."""
    q_n, q_r, pos, c, kr, w_uk, w_uv = _prefill_case(C=4, L=9)
    o0, l0 = O.explicit_prefill_head(q_n, q_r, pos, c, kr, w_uk, w_uv, 0.5, lo=7)
    c2, kr2 = c.copy(), kr.copy()
    c2[:7], kr2[:7] = np.nan, np.nan
    o1, l1 = O.explicit_prefill_head(q_n, q_r, pos, c2, kr2, w_uk, w_uv, 0.5, lo=7)
    np.testing.assert_array_equal(o0, o1)
    assert np.all(o0[pos < 7] == 0) and np.all(np.isneginf(l0[pos < 7]))


def test_pins_catch_a_prefill_window_off_by_one(monkeypatch):
    real = O.explicit_prefill_head
    monkeypatch.setattr(O, "explicit_prefill_head",
                        lambda *a, lo=0, **k: real(*a, lo=lo + 1 if lo else lo, **k))
    with pytest.raises(AssertionError):
        test_prefill_window_matches_library_attention_over_the_window()
