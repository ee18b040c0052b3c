"""The device-built split plan (scheduler reading R10), read back from the decode
workspace and compared integer for integer with a plain restatement of that
reading; plus the invariants every plan must satisfy."""
import math

import numpy as np
import pytest
import torch

import mla_inputs as W
from tests.gpu_harness import dims_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import mla_latent_kv_80_b300 as M
    return M


def prefix(xs):
    out = [0]
    for v in xs:
        out.append(out[-1] + v)
    return out


def plan_reference(seq_lens, q, tile_n, seg_cost, G, seq_start=None):
    """Reading R10: the problems' tiles in order, cut into G contiguous worker
    ranges of equal cost; a range costs its tiles plus seg_cost per problem it
    touches. A problem's tiles are the tile_n-wide key blocks that meet its
    visible positions [lo, len). Returns the plan words in the workspace layout."""
    P = len(seq_lens) * q
    lens = [max(0, int(seq_lens[p // q]) - q + (p % q) + 1) for p in range(P)]
    starts = [0] * len(seq_lens) if seq_start is None else list(seq_start)
    los = [min(max(int(starts[p // q]), 0), lens[p]) for p in range(P)]
    tfs = [lo // tile_n for lo in los]
    tiles = [(n + tile_n - 1) // tile_n - tf if lo < n else 0 for n, lo, tf in zip(lens, los, tfs)]
    cum = prefix(tiles)
    vcum = prefix([t + seg_cost if t > 0 else 0 for t in tiles])
    total, total_v = cum[P], vcum[P]
    per_v = max(1, math.ceil(total_v / G)) if G > 0 else max(1, total_v)
    wstart = [total] * (G + 1)
    first = [P] * G
    for p in range(P):
        v0, v1 = vcum[p], vcum[p + 1]
        if v1 <= v0:
            continue
        # cost position w * per_v inside problem p's cost range [v0, v1)
        for w in range(G):
            pos = w * per_v
            if v0 <= pos < v1:
                wstart[w] = cum[p] + max(0, pos - v0 - seg_cost)
                first[w] = p
    pw0, pcnt = [0] * P, [0] * P
    for p in range(P):
        c0, c1 = cum[p], cum[p + 1]
        if c1 <= c0:
            continue
        # the workers whose range [wstart[w], wstart[w+1]) meets [c0, c1)
        ws = [w for w in range(G) if wstart[w] < c1 and wstart[w + 1] > c0 and wstart[w + 1] > wstart[w]]
        pw0[p], pcnt[p] = ws[0], len(ws)
    pbase = prefix([c if c >= 2 else 0 for c in pcnt])
    return np.array([P, total, seg_cost, G] + cum + pbase + lens + first + wstart + pw0 + pcnt + vcum + los + tfs,
                    dtype=np.int64)


def device_plan(M, w, seq_lens, num_splits, seq_start=None):
    """Runs one decode call over `seq_lens` (and window starts) and returns the plan words it built."""
    x = W.generate(w)
    B = len(seq_lens)
    dev = torch.device("cuda")
    dims = dims_of(M, w)
    cache_t = {k: (None if v is None else v.to(dev)) for k, v in x["cache"].items()}
    cache = M.make_cache(cache_t["ckv"], cache_t["kr"], cache_t["scale"], x["num_pages"])
    # Enough pages for the longest sequence, all of them valid pool pages (the
    # attention values are not checked here, only the plan and the status).
    max_pages = max(1, -(-max(seq_lens) // w.page_size))
    bt = (torch.arange(B * max_pages, dtype=torch.int32) % int(x["num_pages"])).reshape(B, max_pages)
    sl = torch.tensor(seq_lens, dtype=torch.int32)
    step = M.DecodeStep(dims, B, w.q_per_seq, 0, num_splits, dev)
    step.q_abs.zero_()
    st = None if seq_start is None else torch.tensor(seq_start, dtype=torch.int32, device=dev)
    step.decode(cache, bt.to(dev), sl.to(dev), seq_start=st)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    P = B * w.q_per_seq
    G = int(step.ws_decode[12:16].view(torch.int32).item())
    n = 8 + 8 * P + 2 * G
    return step.ws_decode[: 4 * n].view(torch.int32).cpu().numpy().astype(np.int64), G


def check_invariants(words):
    P, total, _, G = (int(v) for v in words[:4])
    o = 4
    cum = words[o:o + P + 1]; o += P + 1
    pbase = words[o:o + P + 1]; o += P + 1
    o += P  # lens
    o += G  # first
    wstart = words[o:o + G + 1]; o += G + 1
    pw0 = words[o:o + P]; o += P
    pcnt = words[o:o + P]
    assert wstart[0] == 0 and wstart[G] == total
    assert np.all(np.diff(wstart) >= 0), "worker ranges overlap"
    for p in range(P):
        if cum[p + 1] > cum[p]:
            assert pcnt[p] >= 1
            lo, hi = int(pw0[p]), int(pw0[p] + pcnt[p])
            assert wstart[lo] <= cum[p] < wstart[lo + 1]
            assert wstart[hi - 1] < cum[p + 1] <= wstart[hi]
    assert pbase[P] <= 2 * G, "more partial slots than the workspace holds"


CASES = [
    ([4096] * 16, 0),
    ([4096] * 16, 5),
    ([1, 63, 64, 65, 0, 700, 129, 4000], 0),
    ([1, 63, 64, 65, 0, 700, 129, 4000], 3),
    ([0, 0, 0, 0], 0),
    ([131072, 2048], 0),
    ([17] * 40, 0),
]


@pytest.mark.parametrize("seq_lens,splits", CASES)
def test_tensor_core_plan_matches_reading(M, seq_lens, splits):
    w = W.shrink(W.DSV2_B16, batch=len(seq_lens), seq_len=64)
    words, G = device_plan(M, w, seq_lens, splits)
    ref = plan_reference(seq_lens, w.q_per_seq, 64, 4, G)
    np.testing.assert_array_equal(words, ref)
    check_invariants(words)


@pytest.mark.parametrize("seq_lens,splits", [([37, 128], 0), ([37, 128], 3), ([5, 0, 90], 7)])
def test_simt_plan_matches_reading(M, seq_lens, splits):
    w = W.shrink(W.TINY, batch=len(seq_lens), seq_lens=tuple(max(1, s) for s in seq_lens))
    words, G = device_plan(M, w, seq_lens, splits)
    ref = plan_reference(seq_lens, w.q_per_seq, 32, 0, G)
    np.testing.assert_array_equal(words, ref)
    check_invariants(words)


WINDOW_CASES = [
    ([4096] * 4, [0, 1, 64, 4095], 0),
    ([1, 63, 64, 65, 0, 700, 129, 4000], [0, 62, 64, 64, 3, 699, 200, 3000], 0),
    ([1000, 2000, 3000], [-5, 1999, 2937], 5),
]


@pytest.mark.parametrize("seq_lens,starts,splits", WINDOW_CASES)
def test_tensor_core_plan_with_window_starts(M, seq_lens, starts, splits):
    w = W.shrink(W.DSV2_B16, batch=len(seq_lens), seq_len=64)
    words, G = device_plan(M, w, seq_lens, splits, starts)
    ref = plan_reference(seq_lens, w.q_per_seq, 64, 4, G, starts)
    np.testing.assert_array_equal(words, ref)
    check_invariants(words)
