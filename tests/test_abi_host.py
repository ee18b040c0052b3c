"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "mla.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"MLA_API\s+(?:const\s+char\s*\*|int|size_t)\s+(mla_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def M():
    import mla_latent_kv_80_b300 as M
    return M


def test_header_declares_the_four_calls():
    names = declared_symbols()
    for n in ("mla_cache_append", "mla_absorb_q", "mla_decode_attn", "mla_out_proj"):
        assert n in names


def test_library_exports_every_declared_symbol(M):
    lib = ctypes.CDLL(M.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) <= set(M.EXPORTED)
    assert M.abi_version() == 1


def test_status_strings(M):
    assert M.status_string(0) == "ok"
    assert "workspace" in M.status_string(-3)
    assert "page" in M.status_string(-5)
    assert M.status_string(12345) == "unknown status"


def tiny_dims(M, **kw):
    args = dict(n_h=8, d_h=32, d_rope=16, d_c=64, d_v=32, d_model=256, page_size=16,
                act_dtype=M.MLA_F32, cache_dtype=M.MLA_F32)
    args.update(kw)
    return M.make_dims(**args)


def test_workspace_sizes_are_consistent(M):
    d = tiny_dims(M)
    assert M.mla_cache_append_workspace_size(d, 0) == 0
    a = M.mla_cache_append_workspace_size(d, 165)
    assert a >= 165 * 80 * 4 and a % 256 == 0
    w1 = M.mla_decode_workspace_size(d, 2, 1, 1)
    w7 = M.mla_decode_workspace_size(d, 2, 1, 7)
    assert 0 < w1 < w7


def rc_of(fn):
    with pytest.raises(Exception) as ei:
        fn()
    return ei.value.code


def test_invalid_dims_rejected(M):
    for bad in (dict(d_c=60), dict(d_rope=15), dict(page_size=24), dict(n_h=0),
                dict(d_c=1024), dict(d_rope=128), dict(d_model=100),
                dict(softmax_scale=0.0), dict(softmax_scale=-0.1), dict(softmax_scale=float("nan")),
                dict(softmax_scale=float("inf")), dict(rope_theta=0.0), dict(rope_theta=float("nan"))):
        d = tiny_dims(M, **bad)
        assert rc_of(lambda: M.mla_decode_workspace_size(d, 2, 1, 0)) == -1, bad
    d = tiny_dims(M, act_dtype=M.MLA_F32, cache_dtype=M.MLA_BF16)
    assert rc_of(lambda: M.mla_decode_workspace_size(d, 2, 1, 0)) == -2
    d = tiny_dims(M, act_dtype=M.MLA_FP8_E4M3, cache_dtype=M.MLA_FP8_E4M3)
    assert rc_of(lambda: M.mla_decode_workspace_size(d, 2, 1, 0)) == -2


def test_null_pointers_and_small_workspace_rejected(M):
    d = tiny_dims(M)
    fake = 0x10000  # never dereferenced: validation fails before any launch
    cache = M.make_cache(fake, num_pages=4)
    # Null q_abs.
    assert rc_of(lambda: M.mla_decode_attn(d, cache, 2, 1, None, fake, 4, fake, 0, fake, 1 << 30,
                                           fake, fake, fake, stream=0)) == -1
    # Workspace one byte short.
    need = M.mla_decode_workspace_size(d, 2, 1, 3)
    assert rc_of(lambda: M.mla_decode_attn(d, cache, 2, 1, fake, fake, 4, fake, 3, fake, need - 1,
                                           fake, fake, fake, stream=0)) == -3
    need_a = M.mla_cache_append_workspace_size(d, 5)
    assert rc_of(lambda: M.mla_cache_append(d, cache, 5, fake, fake, fake, fake, fake, fake, 4,
                                            fake, need_a - 1, fake, stream=0)) == -3
    # Misaligned cache base and a null cache.
    bad_cache = M.make_cache(fake + 2, num_pages=4)
    assert rc_of(lambda: M.mla_decode_attn(d, bad_cache, 2, 1, fake, fake, 4, fake, 0, fake, 1 << 30,
                                           fake, fake, fake, stream=0)) == -1
    # fp8 cache without its k_R / scale pools.
    d8 = tiny_dims(M, act_dtype=M.MLA_BF16, cache_dtype=M.MLA_FP8_E4M3)
    assert rc_of(lambda: M.mla_decode_attn(d8, cache, 2, 1, fake, fake, 4, fake, 0, fake, 1 << 30,
                                           fake, fake, fake, stream=0)) == -1
    # Negative sizes.
    assert rc_of(lambda: M.mla_absorb_q(d, -1, fake, fake, fake, fake, stream=0)) == -1
    assert rc_of(lambda: M.mla_out_proj(d, -1, fake, fake, fake, stream=0)) == -1
    assert rc_of(lambda: M.mla_quantize_fp8_rows(fake, 1, 5000, fake, fake, stream=0)) == -1


def test_zero_sized_calls_are_no_ops(M):
    d = tiny_dims(M)
    M.mla_absorb_q(d, 0, None, None, None, None, stream=0)
    M.mla_out_proj(d, 0, None, None, None, stream=0)
    M.mla_quantize_fp8_rows(None, 0, 16, None, None, stream=0)


def test_out_proj_wo_workspace_and_argument_checks(M):
    d = tiny_dims(M)
    assert M.mla_out_proj_wo_workspace_size(d, 0) == 0
    w = M.mla_out_proj_wo_workspace_size(d, 5)
    assert w >= 5 * 256 * 4 and w % 256 == 0
    # T = 0 is a no-op; null pointers and a short workspace are refused before any launch.
    assert M.raw_call("mla_out_proj_wo", ctypes.byref(d), 0, None, None, None, None, None, None, 0,
                      None, None) == 0
    assert M.raw_call("mla_out_proj_wo", ctypes.byref(d), 5, None, None, None, None, None, None, w,
                      None, None) == -1
    p = ctypes.c_void_p(16)
    assert M.raw_call("mla_out_proj_wo", ctypes.byref(d), 5, p, p, p, p, p, p, w - 1, None, None) == -3


def dsv2_dims(M, **kw):
    args = dict(n_h=128, d_h=128, d_rope=64, d_c=512, d_v=128, d_model=5120, page_size=64,
                act_dtype=M.MLA_BF16, cache_dtype=M.MLA_BF16)
    args.update(kw)
    return M.make_dims(**args)


def test_prefill_form_follows_the_flop_count(M):
    """Explicit form: 2 n_h (d_h + d_v) d_c per cached token plus 2 n_h (d_h + d_rope + d_v)
    per visible (query, key) pair; absorbed form: 2 n_h (d_h + d_v) d_c per query plus
    2 n_h (2 d_c + d_rope) per pair."""
    d = dsv2_dims(M)
    n_h, d_h, d_r, d_c, d_v = 128, 128, 64, 512, 128
    for C, L in [(1, 4096), (64, 8192), (160, 8192), (180, 8192), (512, 8192), (300, 300), (2048, 100)]:
        pairs = sum(max(L - C + j + 1, 0) for j in range(C))
        explicit = 2 * n_h * (d_h + d_v) * d_c * L + 2 * n_h * (d_h + d_r + d_v) * pairs
        absorbed = 2 * n_h * (d_h + d_v) * d_c * C + 2 * n_h * (2 * d_c + d_r) * pairs
        assert M.mla_prefill_form(d, C, L) == int(explicit < absorbed), (C, L)
    # Decode-sized chunks stay absorbed; long chunks go explicit (crossover near 170 at 8K).
    assert M.mla_prefill_form(d, 160, 8192) == 0 and M.mla_prefill_form(d, 180, 8192) == 1
    assert rc_of(lambda: M.mla_prefill_form(d, 0, 10)) == -1
    assert rc_of(lambda: M.mla_prefill_form(d, 4, -1)) == -1


def test_prefill_workspace_and_argument_checks(M):
    d = dsv2_dims(M)
    B, C, L = 3, 130, 517
    need = M.mla_prefill_workspace_size(d, B, C, L)
    l_pad = 768  # 517 rounded up to a multiple of 256 rows
    assert need >= B * l_pad * (576 * 2 + 128 * 256 * 2)
    assert need % 256 == 0
    assert M.mla_prefill_workspace_size(d, B, C, 768) == need
    assert rc_of(lambda: M.mla_prefill_workspace_size(d, -1, C, L)) == -1
    assert rc_of(lambda: M.mla_prefill_workspace_size(d, B, 0, L)) == -1
    fake = 0x10000
    cache = M.make_cache(fake, num_pages=4)
    assert rc_of(lambda: M.mla_prefill_attn(d, cache, -1, C, L, fake, fake, fake, fake, 9, fake, fake, need,
                                            fake, fake, fake, stream=0)) == -1
    # Dims the explicit kernels are not built for (fp32 tiny shapes).
    t = tiny_dims(M)
    assert rc_of(lambda: M.mla_prefill_attn(t, cache, 1, 4, 64, fake, fake, fake, fake, 4, fake, fake, 1 << 20,
                                            fake, fake, fake, stream=0)) == -2


def test_cache_struct_keeps_its_tensors_alive(M):
    import gc
    import torch
    c = M.make_cache(torch.zeros(128, 576, dtype=torch.bfloat16), torch.zeros(128, 64), None, 2)
    gc.collect()
    assert c.ckv == c._tensors[0].data_ptr() and c.kr == c._tensors[1].data_ptr() and c.scale is None
