"""Chunked prefill in the explicit form (mla_prefill_attn) against the oracle.

Each case generates a DeepSeek-V2-shaped cache (the chunk's own tokens already
in it) and C queries per sequence, runs the C ABI on the GPU, and compares o and
lse element by element with the oracle: against the oracle fed the formats the
call keeps its intermediates in (rotated query, latent, formed keys and values
in bf16) at the bf16 bound, and against the exact oracle at the derived
end-to-end bound."""
import math

import numpy as np
import pytest
import torch

import mla_inputs as W
from oracle import mla_oracle as O
from tests.gpu_harness import END_TO_END_REL_BF16, check_bf16, check_fp8, dims_of
from tests.oracle_io import oracle_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import mla_latent_kv_80_b300 as M
    return M


def workload(base, **kw):
    kw.setdefault("append_new", 0)
    kw.setdefault("pool_tokens", None)
    kw.setdefault("seq_len_range", None)
    kw.setdefault("seq_len", None)
    return W.shrink(base, **kw)


def run_prefill(M, x, max_seq_len=None, table=None, status_ok=True, seq_start=None):
    w = x["workload"]
    dev = torch.device("cuda")
    dims = dims_of(M, w)
    d = lambda t: None if t is None else t.to(dev).contiguous()
    cache_t = {k: d(v) for k, v in x["cache"].items()}
    cache = M.make_cache(cache_t["ckv"], cache_t["kr"], cache_t["scale"], x["num_pages"])
    B, C = w.batch, w.q_per_seq
    L_max = int(x["seq_lens"].max()) if max_seq_len is None else max_seq_len
    bt = d(x["block_table"] if table is None else table)
    ws_bytes = M.mla_prefill_workspace_size(dims, B, C, L_max)
    ws = torch.full((ws_bytes,), 0xFF, dtype=torch.uint8, device=dev)  # NaN-patterned scratch
    o = torch.full((B * C, w.n_h, w.d_v), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((B * C, w.n_h), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if seq_start is None:
        M.mla_prefill_attn(dims, cache, B, C, L_max, d(x["q"]), d(x["w_uk"]), d(x["w_uv"]), bt, bt.shape[1],
                           d(x["seq_lens"]), ws, ws_bytes, o, lse, status)
    else:
        st = torch.tensor(seq_start, dtype=torch.int32, device=dev)
        M.mla_prefill_attn_window(dims, cache, B, C, L_max, d(x["q"]), d(x["w_uk"]), d(x["w_uv"]), bt, bt.shape[1],
                                  d(x["seq_lens"]), st, ws, ws_bytes, o, lse, status)
    torch.cuda.synchronize()
    st = int(status.item())
    if status_ok:
        assert st == 0, f"device status {st}"
    return o.float().cpu().numpy(), lse.cpu().numpy(), st


def compare(o, lse, x, heads, sequences=None, fp8=False, seq_start=None):
    w = x["workload"]
    ref = O.prefill_step(oracle_inputs(x), sequences=sequences, heads=heads, seq_start=seq_start)
    C = w.q_per_seq
    got_o = np.concatenate([o[b * C:(b + 1) * C][:, heads] for b in ref])
    got_l = np.concatenate([lse[b * C:(b + 1) * C][:, heads] for b in ref])
    r = {k: np.concatenate([ref[b][k] for b in ref]) for k in ("o", "lse", "o_s", "lse_s")}
    seen = np.isfinite(r["lse"])
    assert np.array_equal(np.isfinite(got_l), seen), "rows with and without visible keys differ"
    assert np.all(got_o[~seen] == 0), "a query that sees no key must return o = 0"
    if fp8:
        check_fp8(got_o, r["o"], "o (fp8 cache)")
        check_fp8(got_l[seen], r["lse"][seen], "lse (fp8 cache)")
        return
    check_bf16(got_o, r["o_s"], "o (stored-format oracle)")
    check_bf16(got_l[seen], r["lse_s"][seen], "lse (stored-format oracle)", stored_bf16=False)
    check_bf16(got_o, r["o"], "o (exact oracle)", rel_bound=END_TO_END_REL_BF16)
    check_bf16(got_l[seen], r["lse"][seen], "lse (exact oracle)", stored_bf16=False)


HEADS = [0, 1, 37, 64, 100, 127]


def test_ragged_sequences_two_query_blocks(M):
    # C = 130: two query blocks per sequence, the second with 2 rows; lengths
    # span several key tiles with ragged last tiles; a shuffled page pool.
    w = workload(W.DSV2_VARLEN, name="prefill_ragged", batch=3, seq_lens=(300, 517, 131), q_per_seq=130,
                 block_table="permutation")
    x = W.generate(w)
    o, lse, _ = run_prefill(M, x)
    compare(o, lse, x, HEADS)


def test_chunk_is_the_whole_sequence(M):
    # A fresh prefill: every cached token is one of the chunk's queries.
    w = workload(W.DSV2_B16, name="prefill_fresh", batch=2, seq_lens=(200, 256), q_per_seq=200,
                 block_table="permutation")
    x = W.generate(w)
    # The second sequence is 256 long with a 200-query chunk: positions 56..255.
    o, lse, _ = run_prefill(M, x)
    compare(o, lse, x, HEADS)


def test_chunk_longer_than_the_sequence(M):
    # Queries at negative positions see no key: o = 0, lse = -inf.
    w = workload(W.DSV2_B16, name="prefill_short", batch=2, seq_lens=(50, 140), q_per_seq=64)
    x = W.generate(w)
    o, lse, _ = run_prefill(M, x)
    assert np.all(np.isneginf(lse[:14])) and np.all(o[:14] == 0)
    compare(o, lse, x, HEADS)


def test_one_query_per_sequence_matches_decode_oracle(M):
    w = workload(W.DSV2_B16, name="prefill_c1", batch=4, seq_lens=(1, 127, 128, 1000), q_per_seq=1)
    x = W.generate(w)
    o, lse, _ = run_prefill(M, x)
    compare(o, lse, x, HEADS)


def test_fp8_cache(M):
    w = workload(W.DSV2_FP8_Q2, name="prefill_fp8", batch=2, seq_lens=(400, 333), q_per_seq=150)
    x = W.generate(w)
    o, lse, _ = run_prefill(M, x)
    compare(o, lse, x, HEADS, fp8=True)


def test_larger_max_seq_len_than_needed(M):
    # The workspace sized for longer sequences: the padded rows are never read.
    w = workload(W.DSV2_B16, name="prefill_pad", batch=2, seq_lens=(190, 70), q_per_seq=40)
    x = W.generate(w)
    o, lse, _ = run_prefill(M, x, max_seq_len=1000)
    compare(o, lse, x, HEADS)


def test_full_size_sampled_rows(M):
    # Four sequences of 8192 tokens with a 512-token chunk at the end: sampled
    # (query, head) rows against the oracle computed for those rows alone.
    w = workload(W.DSV2_B16, name="prefill_b4_l8192_c512", batch=4, seq_len=8192, q_per_seq=512,
                 block_table="permutation")
    x = W.generate(w)
    o, lse, _ = run_prefill(M, x)
    inp = oracle_inputs(x)
    C, d_h = w.q_per_seq, w.d_h
    rows = [0, 1, 127, 128, 255, 300, 511]
    for b in (0, 3):
        L = int(x["seq_lens"][b])
        c, kr = O.gather_sequence(inp["cache"], "bf16", inp["block_table"], b, L, w.page_size, w.d_c)
        pos = L - C + np.array(rows)
        q = inp["q"][b * C + np.array(rows)]
        q_rot = O.rope(q[:, :, d_h:], pos, w.rope_theta)
        for h in (0, 77, 127):
            ref_o, ref_l = O.explicit_prefill_head(q[:, h, :d_h], q_rot[:, h], pos, c, kr, inp["w_uk"][h],
                                                   inp["w_uv"][h], w.softmax_scale)
            got = o[b * C + np.array(rows), h]
            check_bf16(got, ref_o, f"seq {b} head {h} o", rel_bound=END_TO_END_REL_BF16)
            check_bf16(lse[b * C + np.array(rows), h], ref_l, f"seq {b} head {h} lse", stored_bf16=False)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_explicit_and_absorbed_forms_agree(M):
    # The same chunk through absorb -> decode -> out-proj (q_per_seq = C).
    w = workload(W.DSV2_B16, name="prefill_vs_absorbed", batch=2, seq_lens=(260, 390), q_per_seq=70)
    x = W.generate(w)
    o, lse, _ = run_prefill(M, x)
    dev = torch.device("cuda")
    dims = dims_of(M, w)
    d = lambda t: t.to(dev).contiguous()
    cache = M.make_cache(d(x["cache"]["ckv"]), None, None, x["num_pages"])
    step = M.DecodeStep(dims, w.batch, w.q_per_seq, 0, 0, dev)
    q_pos = W.query_positions(x["seq_lens"], w.q_per_seq)
    step.status.zero_()
    step.absorb(d(x["q"]), d(q_pos), d(x["w_uk"]))
    step.decode(cache, d(x["block_table"]), d(x["seq_lens"]))
    step.out_proj(d(x["w_uv"]))
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    o_abs = step.o.float().cpu().numpy()
    check_bf16(o, o_abs, "explicit vs absorbed o", rel_bound=END_TO_END_REL_BF16)
    check_bf16(lse, step.lse.cpu().numpy(), "explicit vs absorbed lse", stored_bf16=False,
               rel_bound=END_TO_END_REL_BF16)


def test_bad_page_and_overlong_sequence_set_status(M):
    w = workload(W.DSV2_B16, name="prefill_bad", batch=2, seq_lens=(130, 200), q_per_seq=8)
    x = W.generate(w)
    bt = x["block_table"].clone()
    bt[1, 1] = 10 ** 6
    _, _, st = run_prefill(M, x, table=bt, status_ok=False)
    assert st == -5  # MLA_ERR_BAD_PAGE
    _, lse, st = run_prefill(M, x, max_seq_len=150, status_ok=False)
    assert st == -1  # MLA_ERR_INVALID_ARG: seq_lens[1] = 200 > max_seq_len
    assert np.all(np.isfinite(lse[:8]))


def test_page_size_16(M):
    # Small pages: a 128-row key tile spans eight pages of a shuffled pool.
    w = workload(W.DSV2_VARLEN, name="prefill_page16", batch=3, seq_lens=(700, 257, 1000), q_per_seq=150,
                 page_size=16, block_table="permutation")
    x = W.generate(w)
    o, lse, _ = run_prefill(M, x)
    compare(o, lse, x, [0, 63, 127])


def test_page_size_128_fp8(M):
    # Large pages over an fp8 cache: a page holds a whole 128-row key tile.
    w = workload(W.DSV2_FP8_Q2, name="prefill_page128_fp8", batch=2, seq_lens=(600, 389), q_per_seq=260,
                 page_size=128)
    x = W.generate(w)
    o, lse, _ = run_prefill(M, x)
    compare(o, lse, x, [0, 64, 127], fp8=True)


def test_fp8_cache_longer_sequences(M):
    # fp8 codes times the per-token scale, dequantised when gathered; several
    # key tiles per query block and a ragged chunk.
    w = workload(W.DSV2_FP8_Q2, name="prefill_fp8_long", batch=2, seq_lens=(3000, 2222), q_per_seq=300)
    x = W.generate(w)
    o, lse, _ = run_prefill(M, x)
    compare(o, lse, x, [0, 77, 127], fp8=True)


def test_window_with_evicted_pages(M):
    # First visible positions per sequence; the pages wholly before them are
    # gone from the block table (-1) and must not be read.
    w = workload(W.DSV2_VARLEN, name="prefill_window", batch=3, seq_lens=(700, 517, 300), q_per_seq=150,
                 block_table="permutation")
    x = W.generate(w)
    starts = [300, 0, 280]
    bt = x["block_table"].clone()
    for b, lo in enumerate(starts):
        bt[b, : lo // w.page_size] = -1
    o, lse, _ = run_prefill(M, x, table=bt, seq_start=starts)
    # Sequence 2: positions 150..299 with a window from 280: queries before 280 see nothing.
    assert np.all(np.isneginf(lse[2 * 150:2 * 150 + 130]))
    compare(o, lse, x, HEADS, seq_start=starts)


def test_window_from_zero_equals_the_plain_call(M):
    w = workload(W.DSV2_B16, name="prefill_window0", batch=2, seq_lens=(200, 333), q_per_seq=70)
    x = W.generate(w)
    o0, l0, _ = run_prefill(M, x)
    o1, l1, _ = run_prefill(M, x, seq_start=[0, -5])
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)
