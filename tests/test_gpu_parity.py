"""GPU parity: the C-ABI path against the float64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import mla_inputs as W
from oracle import e4m3
from oracle import mla_oracle as O
from tests.gpu_harness import DeviceRun, check_bf16, check_fp32, check_fp8, compare, oracle_for

pytestmark = pytest.mark.gpu

HEADS = [0, 1, 37, 64, 127]


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import mla_latent_kv_80_b300 as M
    return M


def pool_bytes(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy().reshape(t.shape[0], -1)


def check_append_placement(run: DeviceRun, ref):
    """Bit-exact placement: exactly the new tokens' slots changed; values within tolerance."""
    x, w = run.x, run.w
    bt = x["block_table"].numpy()
    want = {}
    for i, (b, p) in enumerate(zip(x["new_seq_idx"].tolist(), x["new_pos"].tolist())):
        want[int(O.slot_index(bt, b, p, w.page_size))] = i
    changed = set()
    for key in ("ckv", "kr", "scale"):
        before = x["cache"][key]
        if before is None:
            continue
        after = run.cache_t[key]
        a = pool_bytes(after)
        bb = pool_bytes(before if before.dim() > 1 else before.view(-1, 1))
        a = a.reshape(bb.shape)
        changed |= set(np.nonzero(np.any(a != bb, axis=1))[0].tolist())
    assert changed == set(want), f"slots changed {sorted(changed)[:8]} != expected {sorted(want)[:8]}"
    if not want:
        return
    slots = np.array(sorted(want))
    rows = np.array([want[s] for s in slots])
    c_ref, kr_ref, codes_ref, scale_ref = ref["entries"]
    if w.cache_dtype in ("f32", "bf16"):
        got = run.cache_t["ckv"][torch.from_numpy(slots).cuda()].float().cpu().numpy()
        chk = check_fp32 if w.cache_dtype == "f32" else check_bf16
        chk(got[:, :w.d_c], c_ref[rows], "appended c_KV")
        chk(got[:, w.d_c:], kr_ref[rows], "appended k_R")
    else:
        idx = torch.from_numpy(slots).cuda()
        codes = run.cache_t["ckv"][idx].cpu().numpy()
        scale = run.cache_t["scale"][idx].cpu().numpy()
        np.testing.assert_allclose(scale, scale_ref[rows], rtol=1e-5)
        check_fp8(e4m3.dequantize_rows(codes, scale), c_ref[rows], "appended fp8 c_KV")
        kr = run.cache_t["kr"][idx].float().cpu().numpy()
        check_bf16(kr, kr_ref[rows], "appended k_R")


# ------------------------------------------------------------------ tiny fp32 workload
def test_tiny_fp32_all_heads(M):
    x = W.generate(W.TINY)
    run = DeviceRun(M, x)
    out = run.run()
    ref = oracle_for(x)
    compare(out, ref, W.TINY, "tiny")
    check_append_placement(run, ref)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_tiny_fp32_split_counts(M, splits):
    x = W.generate(W.TINY)
    out = DeviceRun(M, x, num_splits=splits).run()
    compare(out, oracle_for(x), W.TINY, f"tiny splits={splits}")


# ------------------------------------------------------------------ DeepSeek-V2 shapes, small batches
SMALL = {
    "b16_small": W.shrink(W.DSV2_B16, batch=3, seq_len=1000),
    "varlen_small": W.shrink(W.DSV2_VARLEN, batch=5, seq_len_range=(1, 700), pool_tokens=64 * 80),
    "long_small": W.shrink(W.DSV2_LONG, batch=2, seq_len=3000),
    "fp8_q2_small": W.shrink(W.DSV2_FP8_Q2, batch=3, seq_len=333),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_dsv2_small(M, name):
    w = SMALL[name]
    x = W.generate(w)
    run = DeviceRun(M, x)
    out = run.run()
    ref = oracle_for(x, heads=HEADS)
    compare(out, ref, w, name)
    check_append_placement(run, ref)


# Page sizes 32 and 128 (the tensor-core decode loads a 64-token tile as two
# boxes, or as half of a page), for both cache formats, with appends landing
# in the last page.
@pytest.mark.parametrize("page_size", [32, 128])
@pytest.mark.parametrize("base", ["varlen", "fp8_q2"])
def test_page_sizes_32_and_128(M, page_size, base):
    if base == "varlen":
        w = W.shrink(W.DSV2_VARLEN, name=f"varlen_page{page_size}", batch=4, seq_len_range=(70, 650),
                     pool_tokens=page_size * (4 * (700 // page_size + 2)), page_size=page_size)
    else:
        w = W.shrink(W.DSV2_FP8_Q2, name=f"fp8_page{page_size}", batch=3, seq_len=333, page_size=page_size)
    x = W.generate(w)
    run = DeviceRun(M, x)
    out = run.run()
    ref = oracle_for(x, heads=HEADS)
    compare(out, ref, w, w.name)
    check_append_placement(run, ref)


# The combine takes its narrow form (two pieces per thread) while the worker
# count is at most twice the problem count (here 5 problems) and its wide form
# above that: 10 and 11 sit on either side of the switch.
@pytest.mark.parametrize("splits", [1, 2, 7, 10, 11, 64])
def test_split_count_invariance(M, splits):
    w = SMALL["varlen_small"]
    x = W.generate(w)
    out = DeviceRun(M, x, num_splits=splits).run()
    compare(out, oracle_for(x, heads=HEADS), w, f"splits={splits}")


def test_page_placement_does_not_change_results(M):
    """Same tokens in a shuffled vs a contiguous page layout: bit-identical outputs."""
    w = W.shrink(W.DSV2_VARLEN, batch=4, seq_len_range=(100, 400), pool_tokens=64 * 40, append_new=0)
    x = W.generate(w)
    out_perm = DeviceRun(M, x).run()
    bt = x["block_table"]
    P = w.page_size
    new_bt = torch.full_like(bt, -1)
    ckv = torch.full_like(x["cache"]["ckv"], float("nan"))
    k = 0
    for b in range(w.batch):
        for i in range(bt.shape[1]):
            pg = int(bt[b, i])
            if pg < 0:
                continue
            new_bt[b, i] = k
            ckv[k * P:(k + 1) * P] = x["cache"]["ckv"][pg * P:(pg + 1) * P]
            k += 1
    x2 = dict(x)
    x2["block_table"] = new_bt
    x2["cache"] = {"ckv": ckv, "kr": None, "scale": None}
    out_cont = DeviceRun(M, x2).run()
    for a, b in zip(out_perm, out_cont):
        np.testing.assert_array_equal(a, b)


def test_empty_and_single_token_sequences(M):
    w = W.shrink(W.DSV2_B16, batch=3, seq_len=None, seq_lens=(0, 1, 130), append_new=0)
    x = W.generate(w)
    o, o_lat, lse, q_abs = DeviceRun(M, x).run()
    ref = oracle_for(x, heads=HEADS)
    assert np.all(lse[0] == -np.inf) and not np.any(o_lat[0]) and not np.any(o[0])
    rows = {k: v for k, v in ref["rows"].items() if k[0] > 0}
    compare((o, o_lat, lse, q_abs), {"rows": rows}, w, "single/short")
    # One key: o_lat is that key's latent exactly (softmax weight 1).
    c1 = x["cache"]["ckv"][int(x["block_table"][1, 0]) * w.page_size, :w.d_c].float().numpy()
    np.testing.assert_allclose(o_lat[1], np.broadcast_to(c1, o_lat[1].shape), rtol=0, atol=0)


def test_bad_page_sets_status_without_fault(M):
    w = W.shrink(W.DSV2_B16, batch=2, seq_len=200)
    x = W.generate(w)
    x["block_table"][1, 2] = x["num_pages"] + 7
    run = DeviceRun(M, x)
    s = run.step
    s.status.zero_()
    s.run(run.cache, run.h, run.w_dkv, run.w_kr, run.seq_idx, run.pos, run.q, run.q_pos,
          run.w_uk, run.w_uv, run.bt, run.seq_lens)
    torch.cuda.synchronize()
    assert int(s.status.item()) == -5


# ------------------------------------------------------------------ fp8 codec
def test_fp8_quantizer_bit_exact_on_every_bf16_value(M):
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 448.0)]
    cols = 512
    n = (vals.size + cols - 2) // (cols - 1)
    x = np.zeros((n, cols), np.float32)
    x[:, 0] = 448.0  # amax 448 makes the scale exactly 1
    flat = np.zeros(n * (cols - 1), np.float32)
    flat[:vals.size] = vals
    x[:, 1:] = flat.reshape(n, cols - 1)
    rng = np.random.default_rng(7)
    r = (rng.standard_normal((300, cols)) * np.exp(rng.uniform(-30, 30, (300, 1)))).astype(np.float32)
    x = np.concatenate([x, r, np.zeros((1, cols), np.float32)])
    xt = torch.from_numpy(x).cuda()
    codes = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(x.shape[0], dtype=torch.float32, device="cuda")
    M.mla_quantize_fp8_rows(xt, x.shape[0], cols, codes, scales)
    torch.cuda.synchronize()
    ref_codes, ref_scale = e4m3.quantize_rows(x)
    np.testing.assert_array_equal(scales.cpu().numpy(), ref_scale)
    np.testing.assert_array_equal(codes.cpu().numpy(), ref_codes)


# ------------------------------------------------------------------ full-size workloads, sampled rows
FULL = {
    "dsv2_bf16_b16_l4096": (W.DSV2_B16, [0, 15], [0, 77, 127]),
    "dsv2_bf16_paged_varlen_b64": (W.DSV2_VARLEN, [0, 31, 63], [5, 127]),
    "dsv2_bf16_long_b4_l131072": (W.DSV2_LONG, [1], [0, 100]),
    "dsv2_fp8cache_q2_b128_l8192": (W.DSV2_FP8_Q2, [0, 127], [3, 90]),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled(M, name):
    w, seqs, heads = FULL[name]
    x = W.generate(w)
    run = DeviceRun(M, x)
    out = run.run()
    ref = oracle_for(x, sequences=seqs, heads=heads)
    compare(out, ref, w, name)
    check_append_placement(run, oracle_for(x, sequences=[]))
