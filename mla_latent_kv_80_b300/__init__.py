"""Python binding of libmla (B300 MLA decode over a paged latent cache).

Argument marshalling only: every function below forwards to the C ABI in
``include/mla.h`` under the same name; all computation runs in the library's
CUDA kernels. Tensors are torch tensors on the CUDA device (PyTorch supplies
device memory and streams). Importing fails loudly when ``libmla.so`` has not
been built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

MLA_F32, MLA_BF16, MLA_FP8_E4M3 = 0, 1, 2
STATUS = {0: "MLA_OK", -1: "MLA_ERR_INVALID_ARG", -2: "MLA_ERR_UNSUPPORTED",
          -3: "MLA_ERR_WORKSPACE_TOO_SMALL", -4: "MLA_ERR_CUDA", -5: "MLA_ERR_BAD_PAGE",
          -6: "MLA_ERR_DEVICE_TIMEOUT", -7: "MLA_ERR_NO_DEVICE", -8: "MLA_ERR_NO_PAGES"}

EXPORTED = ["mla_cache_append_workspace_size", "mla_cache_append", "mla_absorb_q",
            "mla_decode_default_splits", "mla_decode_workspace_size", "mla_decode_attn", "mla_out_proj",
            "mla_quantize_fp8_rows", "mla_status_string", "mla_abi_version",
            "mla_decode_noalloc_scratch_bytes", "mla_decode_attn_noalloc",
            "mla_out_proj_wo_workspace_size", "mla_out_proj_wo", "mla_decode_attn_window",
            "mla_pool_create", "mla_pool_destroy", "mla_pool_new_seq", "mla_pool_reserve", "mla_pool_fork",
            "mla_pool_evict_before", "mla_pool_free_seq", "mla_pool_block_table", "mla_pool_seq_info",
            "mla_pool_page_refs", "mla_pool_free_pages", "mla_pool_take_copies", "mla_copy_pages",
            "mla_prefill_form", "mla_prefill_workspace_size", "mla_prefill_attn", "mla_selftest_bounded_wait",
            "mla_prefill_attn_window"]

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libmla.so is not built ({LIB_PATH}); run `python mla_latent_kv_80_b300/build.py`")
_lib = ctypes.CDLL(LIB_PATH)


class MlaDims(ctypes.Structure):
    _fields_ = [("n_h", ctypes.c_int32), ("d_h", ctypes.c_int32), ("d_rope", ctypes.c_int32),
                ("d_c", ctypes.c_int32), ("d_v", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("act_dtype", ctypes.c_int32),
                ("cache_dtype", ctypes.c_int32)]


class MlaCache(ctypes.Structure):
    _fields_ = [("ckv", ctypes.c_void_p), ("kr", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("num_pages", ctypes.c_int64)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_SZ = ctypes.c_size_t
_SIGS = {
    "mla_cache_append_workspace_size": [ctypes.POINTER(MlaDims), _I, ctypes.POINTER(_SZ)],
    "mla_cache_append": [ctypes.POINTER(MlaDims), ctypes.POINTER(MlaCache), _I, _P, _P, _P, _P, _P,
                         _P, _I, _P, _SZ, _P, _P],
    "mla_absorb_q": [ctypes.POINTER(MlaDims), _I, _P, _P, _P, _P, _P],
    "mla_decode_default_splits": [ctypes.POINTER(MlaDims), ctypes.POINTER(_I)],
    "mla_decode_workspace_size": [ctypes.POINTER(MlaDims), _I, _I, _I, ctypes.POINTER(_SZ)],
    "mla_decode_attn": [ctypes.POINTER(MlaDims), ctypes.POINTER(MlaCache), _I, _I, _P, _P, _I, _P,
                        _I, _P, _SZ, _P, _P, _P, _P],
    "mla_decode_attn_window": [ctypes.POINTER(MlaDims), ctypes.POINTER(MlaCache), _I, _I, _P, _P, _I, _P,
                               _P, _I, _P, _SZ, _P, _P, _P, _P],
    "mla_decode_noalloc_scratch_bytes": [],
    "mla_decode_attn_noalloc": [ctypes.POINTER(MlaDims), ctypes.POINTER(MlaCache), _I, _I, _P, _P, _I,
                                _P, _I, _P, _P, _P, _P],
    "mla_out_proj": [ctypes.POINTER(MlaDims), _I, _P, _P, _P, _P],
    "mla_out_proj_wo_workspace_size": [ctypes.POINTER(MlaDims), _I, ctypes.POINTER(_SZ)],
    "mla_out_proj_wo": [ctypes.POINTER(MlaDims), _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P],
    "mla_quantize_fp8_rows": [_P, _I, _I, _P, _P, _P],
    "mla_status_string": [ctypes.c_int],
    "mla_pool_create": [ctypes.c_int64, _I, _I, _I, ctypes.POINTER(_P)],
    "mla_pool_destroy": [_P],
    "mla_pool_new_seq": [_P, ctypes.POINTER(_I)],
    "mla_pool_reserve": [_P, _I, _I],
    "mla_pool_fork": [_P, _I, _I, ctypes.POINTER(_I)],
    "mla_pool_evict_before": [_P, _I, _I],
    "mla_pool_free_seq": [_P, _I],
    "mla_pool_block_table": [_P, _P],
    "mla_pool_seq_info": [_P, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)],
    "mla_pool_page_refs": [_P, _I, ctypes.POINTER(_I)],
    "mla_pool_free_pages": [_P, ctypes.POINTER(ctypes.c_int64)],
    "mla_pool_take_copies": [_P, _P, _P, _I, ctypes.POINTER(_I)],
    "mla_copy_pages": [ctypes.POINTER(MlaDims), ctypes.POINTER(MlaCache), _I, _P, _P, _P, _P],
    "mla_prefill_form": [ctypes.POINTER(MlaDims), _I, ctypes.c_int64, ctypes.POINTER(_I)],
    "mla_prefill_workspace_size": [ctypes.POINTER(MlaDims), _I, _I, _I, ctypes.POINTER(_SZ)],
    "mla_prefill_attn": [ctypes.POINTER(MlaDims), ctypes.POINTER(MlaCache), _I, _I, _I, _P, _P, _P, _P, _I,
                         _P, _P, _SZ, _P, _P, _P, _P],
    "mla_selftest_bounded_wait": [ctypes.c_uint64, _P, _P],
    "mla_prefill_attn_window": [ctypes.POINTER(MlaDims), ctypes.POINTER(MlaCache), _I, _I, _I, _P, _P, _P, _P, _I,
                                _P, _P, _P, _SZ, _P, _P, _P, _P],
    "mla_abi_version": [],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = {"mla_status_string": ctypes.c_char_p,
                  "mla_decode_noalloc_scratch_bytes": ctypes.c_size_t,
                  "mla_pool_destroy": None}.get(_name, ctypes.c_int)


class MlaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({status_string(code)})")
        self.code = code


def status_string(code: int) -> str:
    return _lib.mla_status_string(int(code)).decode()


def abi_version() -> int:
    return _lib.mla_abi_version()


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int):
    if rc != 0:
        raise MlaError(fn, rc)


def make_dims(n_h, d_h, d_rope, d_c, d_v, d_model, page_size, act_dtype, cache_dtype,
              softmax_scale=None, rope_theta=10000.0) -> MlaDims:
    if softmax_scale is None:
        softmax_scale = 1.0 / (d_h + d_rope) ** 0.5
    return MlaDims(n_h, d_h, d_rope, d_c, d_v, d_model, page_size, softmax_scale, rope_theta,
                   act_dtype, cache_dtype)


def make_cache(ckv, kr=None, scale=None, num_pages=0) -> MlaCache:
    """The cache struct of the C ABI. It holds references to the tensors it
    points into, so that a cache built from temporaries stays valid for as long
    as the struct is alive."""
    c = MlaCache(_ptr(ckv), _ptr(kr), _ptr(scale), int(num_pages))
    c._tensors = (ckv, kr, scale)
    return c


# ------------------------------------------------------------------ the ABI calls
def mla_cache_append_workspace_size(dims: MlaDims, T: int) -> int:
    out = _SZ(0)
    _check("mla_cache_append_workspace_size",
           _lib.mla_cache_append_workspace_size(ctypes.byref(dims), int(T), ctypes.byref(out)))
    return out.value


def mla_cache_append(dims, cache, T, h, w_dkv, w_kr, seq_idx, pos, block_table,
                     max_pages_per_seq, workspace, workspace_bytes, status, stream=None):
    _check("mla_cache_append", _lib.mla_cache_append(
        ctypes.byref(dims), ctypes.byref(cache), int(T), _ptr(h), _ptr(w_dkv), _ptr(w_kr),
        _ptr(seq_idx), _ptr(pos), _ptr(block_table), int(max_pages_per_seq), _ptr(workspace),
        int(workspace_bytes), _ptr(status), _stream(stream)))


def mla_absorb_q(dims, T, q, pos, w_uk, q_abs, stream=None):
    _check("mla_absorb_q", _lib.mla_absorb_q(ctypes.byref(dims), int(T), _ptr(q), _ptr(pos),
                                             _ptr(w_uk), _ptr(q_abs), _stream(stream)))


def mla_decode_default_splits(dims) -> int:
    out = _I(0)
    _check("mla_decode_default_splits", _lib.mla_decode_default_splits(ctypes.byref(dims), ctypes.byref(out)))
    return out.value


def mla_decode_workspace_size(dims, B, q_per_seq, num_splits=0) -> int:
    out = _SZ(0)
    _check("mla_decode_workspace_size", _lib.mla_decode_workspace_size(
        ctypes.byref(dims), int(B), int(q_per_seq), int(num_splits), ctypes.byref(out)))
    return out.value


def mla_decode_attn(dims, cache, B, q_per_seq, q_abs, block_table, max_pages_per_seq, seq_lens,
                    num_splits, workspace, workspace_bytes, o_lat, lse, status, stream=None):
    _check("mla_decode_attn", _lib.mla_decode_attn(
        ctypes.byref(dims), ctypes.byref(cache), int(B), int(q_per_seq), _ptr(q_abs),
        _ptr(block_table), int(max_pages_per_seq), _ptr(seq_lens), int(num_splits),
        _ptr(workspace), int(workspace_bytes), _ptr(o_lat), _ptr(lse), _ptr(status),
        _stream(stream)))


def mla_decode_attn_window(dims, cache, B, q_per_seq, q_abs, block_table, max_pages_per_seq, seq_lens,
                           seq_start, num_splits, workspace, workspace_bytes, o_lat, lse, status, stream=None):
    _check("mla_decode_attn_window", _lib.mla_decode_attn_window(
        ctypes.byref(dims), ctypes.byref(cache), int(B), int(q_per_seq), _ptr(q_abs), _ptr(block_table),
        int(max_pages_per_seq), _ptr(seq_lens), _ptr(seq_start), int(num_splits), _ptr(workspace),
        int(workspace_bytes), _ptr(o_lat), _ptr(lse), _ptr(status), _stream(stream)))


def mla_decode_noalloc_scratch_bytes() -> int:
    return int(_lib.mla_decode_noalloc_scratch_bytes())


def mla_decode_attn_noalloc(dims, cache, B, q_per_seq, q_abs, block_table, max_pages_per_seq,
                            seq_lens, num_splits, o_lat, lse, status, stream=None):
    """mla_decode_attn without a workspace argument: the scratch is a fixed array
    inside the library (for callers that cannot allocate device memory)."""
    _check("mla_decode_attn_noalloc", _lib.mla_decode_attn_noalloc(
        ctypes.byref(dims), ctypes.byref(cache), int(B), int(q_per_seq), _ptr(q_abs),
        _ptr(block_table), int(max_pages_per_seq), _ptr(seq_lens), int(num_splits), _ptr(o_lat),
        _ptr(lse), _ptr(status), _stream(stream)))


def mla_out_proj(dims, T, o_lat, w_uv, o, stream=None):
    _check("mla_out_proj", _lib.mla_out_proj(ctypes.byref(dims), int(T), _ptr(o_lat), _ptr(w_uv),
                                             _ptr(o), _stream(stream)))


def mla_out_proj_wo_workspace_size(dims, T) -> int:
    out = _SZ(0)
    _check("mla_out_proj_wo_workspace_size",
           _lib.mla_out_proj_wo_workspace_size(ctypes.byref(dims), int(T), ctypes.byref(out)))
    return out.value


def mla_out_proj_wo(dims, T, o_lat, w_uv, w_o, o, out, workspace, workspace_bytes, status=None, stream=None):
    _check("mla_out_proj_wo", _lib.mla_out_proj_wo(
        ctypes.byref(dims), int(T), _ptr(o_lat), _ptr(w_uv), _ptr(w_o), _ptr(o), _ptr(out), _ptr(workspace),
        int(workspace_bytes), _ptr(status), _stream(stream)))


def mla_prefill_form(dims, q_per_seq, seq_len) -> int:
    """1 when the explicit form costs fewer flops for this chunk, else 0."""
    out = _I(0)
    _check("mla_prefill_form", _lib.mla_prefill_form(ctypes.byref(dims), int(q_per_seq), int(seq_len),
                                                     ctypes.byref(out)))
    return out.value


def mla_prefill_workspace_size(dims, B, q_per_seq, max_seq_len) -> int:
    out = _SZ(0)
    _check("mla_prefill_workspace_size", _lib.mla_prefill_workspace_size(
        ctypes.byref(dims), int(B), int(q_per_seq), int(max_seq_len), ctypes.byref(out)))
    return out.value


def mla_prefill_attn(dims, cache, B, q_per_seq, max_seq_len, q, w_uk, w_uv, block_table, max_pages_per_seq,
                     seq_lens, workspace, workspace_bytes, o, lse, status, stream=None):
    _check("mla_prefill_attn", _lib.mla_prefill_attn(
        ctypes.byref(dims), ctypes.byref(cache), int(B), int(q_per_seq), int(max_seq_len), _ptr(q), _ptr(w_uk),
        _ptr(w_uv), _ptr(block_table), int(max_pages_per_seq), _ptr(seq_lens), _ptr(workspace),
        int(workspace_bytes), _ptr(o), _ptr(lse), _ptr(status), _stream(stream)))


def mla_prefill_attn_window(dims, cache, B, q_per_seq, max_seq_len, q, w_uk, w_uv, block_table,
                            max_pages_per_seq, seq_lens, seq_start, workspace, workspace_bytes, o, lse, status,
                            stream=None):
    _check("mla_prefill_attn_window", _lib.mla_prefill_attn_window(
        ctypes.byref(dims), ctypes.byref(cache), int(B), int(q_per_seq), int(max_seq_len), _ptr(q), _ptr(w_uk),
        _ptr(w_uv), _ptr(block_table), int(max_pages_per_seq), _ptr(seq_lens), _ptr(seq_start), _ptr(workspace),
        int(workspace_bytes), _ptr(o), _ptr(lse), _ptr(status), _stream(stream)))


def mla_selftest_bounded_wait(limit_ns, status, stream=None):
    _check("mla_selftest_bounded_wait", _lib.mla_selftest_bounded_wait(int(limit_ns), _ptr(status), _stream(stream)))


def mla_quantize_fp8_rows(x, rows, cols, codes, scales, stream=None):
    _check("mla_quantize_fp8_rows", _lib.mla_quantize_fp8_rows(
        _ptr(x), int(rows), int(cols), _ptr(codes), _ptr(scales), _stream(stream)))


def mla_copy_pages(dims, cache, n, src, dst, status=None, stream=None):
    _check("mla_copy_pages", _lib.mla_copy_pages(ctypes.byref(dims), ctypes.byref(cache), int(n), _ptr(src),
                                                 _ptr(dst), _ptr(status), _stream(stream)))


class PagePool:
    """The library's host-side page pool (mla_pool_*): page ids for block
    tables, reference-counted prefix sharing and eviction. Marshalling only."""

    def __init__(self, num_pages, page_size, max_seqs, max_pages_per_seq):
        self._h = _P()
        _check("mla_pool_create", _lib.mla_pool_create(int(num_pages), int(page_size), int(max_seqs),
                                                       int(max_pages_per_seq), ctypes.byref(self._h)))
        self.max_seqs, self.max_pages = int(max_seqs), int(max_pages_per_seq)

    def close(self):
        if self._h:
            _lib.mla_pool_destroy(self._h)
            self._h = _P()

    def __del__(self):
        try:
            self.close()
        except Exception:  # pragma: no cover  (interpreter shutdown)
            pass

    def new_seq(self) -> int:
        s = _I(0)
        _check("mla_pool_new_seq", _lib.mla_pool_new_seq(self._h, ctypes.byref(s)))
        return s.value

    def reserve(self, seq, length):
        _check("mla_pool_reserve", _lib.mla_pool_reserve(self._h, int(seq), int(length)))

    def fork(self, parent, shared_tokens) -> int:
        c = _I(0)
        _check("mla_pool_fork", _lib.mla_pool_fork(self._h, int(parent), int(shared_tokens), ctypes.byref(c)))
        return c.value

    def evict_before(self, seq, pos):
        _check("mla_pool_evict_before", _lib.mla_pool_evict_before(self._h, int(seq), int(pos)))

    def free_seq(self, seq):
        _check("mla_pool_free_seq", _lib.mla_pool_free_seq(self._h, int(seq)))

    def block_table(self) -> torch.Tensor:
        t = torch.empty((self.max_seqs, self.max_pages), dtype=torch.int32)
        _check("mla_pool_block_table", _lib.mla_pool_block_table(self._h, t.data_ptr()))
        return t

    def seq_info(self, seq):
        cap, st = _I(0), _I(0)
        _check("mla_pool_seq_info", _lib.mla_pool_seq_info(self._h, int(seq), ctypes.byref(cap), ctypes.byref(st)))
        return cap.value, st.value

    def page_refs(self, page) -> int:
        r = _I(0)
        _check("mla_pool_page_refs", _lib.mla_pool_page_refs(self._h, int(page), ctypes.byref(r)))
        return r.value

    def free_pages(self) -> int:
        n = ctypes.c_int64(0)
        _check("mla_pool_free_pages", _lib.mla_pool_free_pages(self._h, ctypes.byref(n)))
        return n.value

    def take_copies(self):
        """Pending page copies (src, dst) as int32 host tensors; the queue is emptied."""
        n = _I(0)
        rc = _lib.mla_pool_take_copies(self._h, None, None, 0, ctypes.byref(n))
        if rc == 0:
            return torch.empty(0, dtype=torch.int32), torch.empty(0, dtype=torch.int32)
        src = torch.empty(n.value, dtype=torch.int32)
        dst = torch.empty(n.value, dtype=torch.int32)
        _check("mla_pool_take_copies", _lib.mla_pool_take_copies(self._h, src.data_ptr(), dst.data_ptr(),
                                                                 n.value, ctypes.byref(n)))
        return src, dst


def raw_call(name: str, *args) -> int:
    """Call an ABI function with raw ctypes-compatible arguments; returns its status."""
    return getattr(_lib, name)(*args)


# ------------------------------------------------------------------ one decode step
class DecodeStep:
    """Owns the scratch buffers of one decode step and issues its four ABI calls.

    Buffers are torch CUDA tensors sized for B sequences, q_per_seq queries and
    T appended tokens. ``run`` enqueues the four calls on the given (or current)
    stream and returns (o, o_lat, lse, q_abs): the absorb call, which needs
    neither the cache nor the append's output, runs on a second stream forked
    from and joined back to that one, alongside the append.
    """

    def __init__(self, dims: MlaDims, B: int, q_per_seq: int, T_new: int, num_splits: int = 0,
                 device="cuda"):
        self.dims, self.B, self.q, self.T_new, self.num_splits = dims, B, q_per_seq, T_new, num_splits
        act = torch.float32 if dims.act_dtype == MLA_F32 else torch.bfloat16
        rows = B * q_per_seq
        self.q_abs = torch.empty((rows, dims.n_h, dims.d_c + dims.d_rope), dtype=act, device=device)
        self.o_lat = torch.empty((rows, dims.n_h, dims.d_c), dtype=act, device=device)
        self.lse = torch.empty((rows, dims.n_h), dtype=torch.float32, device=device)
        self.o = torch.empty((rows, dims.n_h, dims.d_v), dtype=act, device=device)
        self.ws_append_bytes = mla_cache_append_workspace_size(dims, max(T_new, 0))
        self.ws_decode_bytes = mla_decode_workspace_size(dims, B, q_per_seq, num_splits)
        self.ws_append = torch.empty(max(self.ws_append_bytes, 256), dtype=torch.uint8, device=device)
        self.ws_decode = torch.empty(max(self.ws_decode_bytes, 256), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self._side = torch.cuda.Stream(device=device)

    def append(self, cache, h, w_dkv, w_kr, seq_idx, pos, block_table, stream=None):
        T = h.shape[0]
        if T:
            mla_cache_append(self.dims, cache, T, h, w_dkv, w_kr, seq_idx, pos, block_table,
                             block_table.shape[1], self.ws_append, self.ws_append_bytes,
                             self.status, stream)

    def absorb(self, q, q_pos, w_uk, stream=None):
        mla_absorb_q(self.dims, self.B * self.q, q, q_pos, w_uk, self.q_abs, stream)

    def decode(self, cache, block_table, seq_lens, stream=None, seq_start=None):
        """Decode attention; with ``seq_start`` ([B] int32) only the keys at
        positions from seq_start[b] on are visible (mla_decode_attn_window)."""
        if seq_start is None:
            mla_decode_attn(self.dims, cache, self.B, self.q, self.q_abs, block_table,
                            block_table.shape[1], seq_lens, self.num_splits, self.ws_decode,
                            self.ws_decode_bytes, self.o_lat, self.lse, self.status, stream)
        else:
            mla_decode_attn_window(self.dims, cache, self.B, self.q, self.q_abs, block_table,
                                   block_table.shape[1], seq_lens, seq_start, self.num_splits,
                                   self.ws_decode, self.ws_decode_bytes, self.o_lat, self.lse,
                                   self.status, stream)

    def out_proj(self, w_uv, stream=None):
        mla_out_proj(self.dims, self.B * self.q, self.o_lat, w_uv, self.o, stream)

    def out_proj_wo(self, w_uv, w_o, stream=None):
        """W_UV then W_O: self.o and self.out ([rows][d_model]) are written."""
        rows = self.B * self.q
        if getattr(self, "out", None) is None:
            self.out = torch.empty((rows, self.dims.d_model), dtype=self.o.dtype, device=self.o.device)
            self.ws_wo_bytes = mla_out_proj_wo_workspace_size(self.dims, rows)
            self.ws_wo = torch.empty(max(self.ws_wo_bytes, 256), dtype=torch.uint8, device=self.o.device)
        mla_out_proj_wo(self.dims, rows, self.o_lat, w_uv, w_o, self.o, self.out, self.ws_wo, self.ws_wo_bytes,
                        self.status, stream)
        return self.out

    def attend(self, cache, q, q_pos, w_uk, w_uv, block_table, seq_lens, stream=None):
        self.absorb(q, q_pos, w_uk, stream)
        self.decode(cache, block_table, seq_lens, stream)
        self.out_proj(w_uv, stream)
        return self.o, self.o_lat, self.lse, self.q_abs

    def prepare(self, cache, h, w_dkv, w_kr, seq_idx, pos, q, q_pos, w_uk, block_table,
                stream=None):
        """append on `stream` and absorb on a side stream, joined back into `stream`."""
        main = torch.cuda.current_stream() if stream is None else stream
        if isinstance(main, int):
            main = torch.cuda.ExternalStream(main)
        self._side.wait_stream(main)
        self.append(cache, h, w_dkv, w_kr, seq_idx, pos, block_table, main)
        self.absorb(q, q_pos, w_uk, self._side)
        main.wait_stream(self._side)

    def run(self, cache, h, w_dkv, w_kr, seq_idx, pos, q, q_pos, w_uk, w_uv, block_table,
            seq_lens, stream=None):
        self.prepare(cache, h, w_dkv, w_kr, seq_idx, pos, q, q_pos, w_uk, block_table, stream)
        self.decode(cache, block_table, seq_lens, stream)
        self.out_proj(w_uv, stream)
        return self.o, self.o_lat, self.lse, self.q_abs
