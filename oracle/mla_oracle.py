"""Plain double-precision CPU oracle for MLA decode over a paged latent cache.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module. It shares no code with
the CUDA library and never imports it.

What it computes is the explicit, non-absorbed form of Multi-head Latent
Attention as the pages define it (DeepSeek-V2):

* "MLA 之后，KV cache 确实得重新理解一遍", section "MLA 的三步 / 第一步": the
  joint latent c_kv(t) = W_DKV x(t) and the up-projections k = W_UK c_kv,
  v = W_UV c_kv;
* same page, section "RoPE 为什么必须解耦": the decoupled key
  k_R(t) = RoPE(W_KR x(t)) of width 64 shared by all heads, and the split
  score q_C.k_C + q_R.k_R;
* "MLA 是什么 | dg's Blog", sections "1. 下采样" / "2. 上采样" (shapes, the
  [out x in] weight convention) and "PyTorch 代码示例" (scores scaled by
  1/sqrt(d), softmax over keys, weighted sum of v);
* the interview-answer page on MLA and KV Cache, section "先区分 KV Cache 与
  MLA": a decode step appends the current token's entry first and then attends
  over history plus the current token.

Every head's keys and values are rebuilt explicitly from the cached latent and
a textbook max-subtracted softmax runs in float64. The absorbed quantities the
GPU path produces (q_lat = W_UK^T q_nope, the latent weighted sum sum_t a_t c_t,
the log-sum-exp) are also returned, each computed by its plain definition, so
that every GPU stage can be compared on its own.

Readings where the pages are silent (each one is listed in the design notes):
  * softmax scale 1/sqrt(d_h + d_rope);
  * RoPE rotates interleaved pairs (2i, 2i+1) by pos * theta^(-2i/d_rope), theta = 10000;
  * positions count from 0; query j of sequence b sits at seq_len_b - q + j and
    sees keys at positions <= its own;
  * W_UK[h] is [d_h x d_c] and W_UV[h] is [d_v x d_c] (nn.Linear [out x in]);
  * q_rope is rotated at the query's own position;
  * an empty key set gives o = 0 and lse = -inf;
  * cached values are stored in the cache dtype: bf16 rounds to nearest even
    from the exact value; fp8 c_KV follows the per-token E4M3 recipe in ``e4m3``.
"""
from __future__ import annotations

import math

import numpy as np

from . import e4m3


# --------------------------------------------------------------------------
# Rounding helpers for the cache storage formats
# --------------------------------------------------------------------------
def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (nearest, ties to even) via exact fp32.

    The double is first rounded to fp32 (RNE), then the fp32 bit pattern is
    rounded to its top 16 bits (RNE). Double rounding can differ from a single
    RNE only in exact-midpoint cases that random data does not hit.
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    out = np.where(np.isnan(f), np.float32("nan"), out)
    return out.astype(np.float64)


# --------------------------------------------------------------------------
# Projections and RoPE (page 2 "第一步", "RoPE 为什么必须解耦"; page 3 "1. 下采样")
# --------------------------------------------------------------------------
def joint_kv_latent(h: np.ndarray, w_dkv: np.ndarray) -> np.ndarray:
    """c_KV,t = W_DKV h_t for each row of h [T, d_model]; W_DKV is [d_c, d_model]."""
    return np.asarray(h, np.float64) @ np.asarray(w_dkv, np.float64).T


def rope_angles(pos, d_rope: int, theta: float = 10000.0) -> np.ndarray:
    """Angle pos * theta^(-2i/d_rope) for pair i, shape [len(pos), d_rope/2]."""
    i = np.arange(d_rope // 2, dtype=np.float64)
    inv_freq = np.power(float(theta), -2.0 * i / d_rope)
    return np.asarray(pos, dtype=np.float64).reshape(-1, 1) * inv_freq.reshape(1, -1)


def rope(x: np.ndarray, pos, theta: float = 10000.0) -> np.ndarray:
    """Rotate each interleaved pair (x[2i], x[2i+1]) of the last axis by the angle of ``pos``.

    ``x`` is [n, d_rope] or [n, heads, d_rope]; ``pos`` has n entries. The
    rotation is R_pos acting on the key or query, so that
    (R_i q)^T (R_j k) = q^T R_{j-i} k (page 2, "RoPE 为什么必须解耦").
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = rope_angles(pos, d, theta)
    if x.ndim == 3:
        ang = ang[:, None, :]
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def decoupled_rope_key(h: np.ndarray, w_kr: np.ndarray, pos, theta: float = 10000.0) -> np.ndarray:
    """k_R,t = RoPE(W_KR h_t) at the token's own position; shared by all heads."""
    return rope(np.asarray(h, np.float64) @ np.asarray(w_kr, np.float64).T, pos, theta)


def query_projection(h: np.ndarray, w_q: np.ndarray, d_h: int):
    """Per-head query q_h = W_Q[h] h split into (q_nope [d_h], q_rope [d_rope]).

    Page 3's listing projects the query directly from the hidden state; the
    tiny workload keeps that and orders each head's output as [nope ; rope].
    """
    q = np.einsum("hod,td->tho", np.asarray(w_q, np.float64), np.asarray(h, np.float64))
    return q[..., :d_h], q[..., d_h:]


def up_project(c: np.ndarray, w_u_h: np.ndarray) -> np.ndarray:
    """k^C_t = W_UK[h] c_t or v_t = W_UV[h] c_t for each cached token (rows of c)."""
    return np.asarray(c, np.float64) @ np.asarray(w_u_h, np.float64).T


def absorbed_query(q_nope: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """q_lat[.., h, :] = W_UK[h]^T q_nope[.., h, :] (page 2, "第二步，推理时的吸收")."""
    return np.einsum("hkc,...hk->...hc", np.asarray(w_uk, np.float64), np.asarray(q_nope, np.float64))


def output_projection(o: np.ndarray, w_o: np.ndarray) -> np.ndarray:
    """Layer output W_O . [o_1 ; o_2 ; ... ; o_n_h] for each token.

    ``o`` is [T, n_h, d_v] (each head's W_UV[h] o_lat); the heads are joined
    in head order into one n_h * d_v vector and W_O [d_model, n_h * d_v]
    (nn.Linear [out x in]) maps it to d_model: page 3's listing reshapes the
    per-head outputs to (batch, seq, n_heads * d_n) and applies self.W_O
    ("MLA 是什么 | dg's Blog", "完整代码").
    """
    o = np.asarray(o, np.float64)
    return o.reshape(o.shape[0], -1) @ np.asarray(w_o, np.float64).T


# --------------------------------------------------------------------------
# Paged cache addressing
# --------------------------------------------------------------------------
def slot_index(block_table: np.ndarray, b: int, pos, page_size: int) -> np.ndarray:
    """Pool slot of (sequence b, position pos): page table entry times page size plus offset."""
    pos = np.asarray(pos, dtype=np.int64)
    pages = np.asarray(block_table, dtype=np.int64)[b, pos // page_size]
    return pages * page_size + pos % page_size


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) to float64: the top half of an fp32 pattern."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gather_sequence(cache: dict, cache_dtype: str, block_table, b: int, length: int,
                    page_size: int, d_c: int, first: int = 0):
    """Cached (c_KV, k_R) of sequence b's positions ``first`` .. ``length`` - 1, float64.

    ``cache`` holds numpy pools in slot order: "f32" float32 rows, "bf16" uint16
    bit patterns (k_R in the last columns of each row), or for fp8 uint8 codes
    ``ckv``, bf16 bits ``kr`` and float32 ``scale``.
    """
    slots = slot_index(block_table, b, np.arange(first, length), page_size)
    if cache_dtype == "f32":
        rows = np.asarray(cache["ckv"])[slots].astype(np.float64)
        return rows[:, :d_c], rows[:, d_c:]
    if cache_dtype == "bf16":
        rows = bf16_bits_to_f64(np.asarray(cache["ckv"])[slots])
        return rows[:, :d_c], rows[:, d_c:]
    codes = np.asarray(cache["ckv"])[slots]
    scale = np.asarray(cache["scale"], dtype=np.float32)[slots]
    c = e4m3.dequantize_rows(codes, scale)
    kr = bf16_bits_to_f64(np.asarray(cache["kr"])[slots])
    return c, kr


# --------------------------------------------------------------------------
# Attention for one head: explicit keys/values, textbook softmax
# --------------------------------------------------------------------------
def attend_head(q_nope_h, q_rope_rot_h, c, k_r, w_uk_h, w_uv_h, scale: float):
    """Explicit attention of one query head over cached tokens.

    k_t = [W_UK[h] c_t ; k_R,t] and v_t = W_UV[h] c_t are rebuilt for every
    token; s_t = scale * q.k_t; a = softmax(s); o = sum_t a_t v_t.
    Returns (o [d_v], a [L], lse, latent_sum [d_c]).
    """
    L = c.shape[0]
    d_v = w_uv_h.shape[0]
    if L == 0:
        return np.zeros(d_v), np.zeros(0), -math.inf, np.zeros(c.shape[1])
    k_c = up_project(c, w_uk_h)
    v = up_project(c, w_uv_h)
    s = scale * (k_c @ np.asarray(q_nope_h, np.float64) + np.asarray(k_r, np.float64) @ np.asarray(q_rope_rot_h, np.float64))
    m = np.max(s)
    e = np.exp(s - m)
    z = np.sum(e)
    a = e / z
    o = a @ v
    lse = m + math.log(z)
    latent_sum = a @ c
    return o, a, lse, latent_sum


def decode_rows(q_nope, q_rope, q_pos, c, k_r, w_uk, w_uv, scale, theta=10000.0, heads=None,
                act_dtype="f32"):
    """Attention of one query token (all or selected heads) over its visible keys.

    q_nope [n_h, d_h], q_rope [n_h, d_rope] (not yet rotated), q_pos its position;
    c [L, d_c] and k_r [L, d_rope] are the cached entries it sees.

    Returns, for the selected heads:
      end to end (explicit keys and values, no intermediate rounding):
        o [H, d_v], o_lat [H, d_c] (= sum_t a_t c_t), lse [H]
      per ABI stage, each fed the previous stage's result as the ABI stores it
      (``act_dtype``):
        q_abs [H, d_c+d_rope]              absorb stage
        o_lat_s [H, d_c], lse_s [H]        decode stage on round(q_abs)
        o_s [H, d_v]                       output stage on round(o_lat_s)
    """
    n_h = q_nope.shape[0]
    heads = list(range(n_h)) if heads is None else list(heads)
    q_rot = rope(np.asarray(q_rope, np.float64)[None], [q_pos], theta)[0]
    q_lat = absorbed_query(q_nope, w_uk)
    o, o_lat, lse, q_abs = [], [], [], []
    for h in heads:
        oh, _, lh, lat = attend_head(q_nope[h], q_rot[h], c, k_r, w_uk[h], w_uv[h], scale)
        o.append(oh)
        o_lat.append(lat)
        lse.append(lh)
        q_abs.append(np.concatenate([q_lat[h], q_rot[h]]))
    q_abs = np.array(q_abs)
    o_lat_s, lse_s = absorbed_attention(round_to_storage(q_abs, act_dtype), c, k_r, scale)
    lat_st = round_to_storage(o_lat_s, act_dtype)
    o_s = np.array([up_project(lat_st[i][None], w_uv[h])[0] for i, h in enumerate(heads)])
    return {"o": np.array(o), "o_lat": np.array(o_lat), "lse": np.array(lse), "q_abs": q_abs,
            "o_lat_s": o_lat_s, "lse_s": lse_s, "o_s": o_s, "heads": heads}


def absorbed_attention(q_abs, c, k_r, scale: float):
    """Attention in latent space (page 2, "第二步，推理时的吸收"): for each head,
    s_t = scale * q_abs . [c_t ; k_R,t], a = softmax(s), o_lat = sum_t a_t c_t.

    q_abs [H, d_c + d_rope]. Returns (o_lat [H, d_c], lse [H]). With the exact
    q_abs this equals the explicit form (the absorption identity).
    """
    q_abs = np.asarray(q_abs, np.float64)
    H, d_c = q_abs.shape[0], c.shape[1]
    if c.shape[0] == 0:
        return np.zeros((H, d_c)), np.full(H, -math.inf)
    keys = np.concatenate([np.asarray(c, np.float64), np.asarray(k_r, np.float64)], axis=1)
    s = scale * (q_abs @ keys.T)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=1, keepdims=True)
    return (e / z) @ c, (m + np.log(z))[:, 0]


def round_to_storage(x, act_dtype: str) -> np.ndarray:
    """Value of x once stored in the activation dtype of the ABI ("f32" or "bf16")."""
    if act_dtype == "bf16":
        return round_to_bf16(x)
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Cache append (what one decode step writes before attending)
# --------------------------------------------------------------------------
def append_entries(h, w_dkv, w_kr, pos, cache_dtype: str, theta=10000.0):
    """Cache entries of new tokens: c_KV = W_DKV h and k_R = RoPE(W_KR h, pos).

    Returns (c_stored [T, d_c] float64, k_r_stored [T, d_rope] float64, codes, scale):
    the values as the cache holds them (rounded to the storage format) plus,
    for fp8, the E4M3 codes and per-token scales computed from the fp32-rounded
    exact latent.
    """
    c = joint_kv_latent(h, w_dkv)
    kr = decoupled_rope_key(h, w_kr, pos, theta)
    if cache_dtype == "f32":
        return c.astype(np.float32).astype(np.float64), kr.astype(np.float32).astype(np.float64), None, None
    if cache_dtype == "bf16":
        return round_to_bf16(c), round_to_bf16(kr), None, None
    codes, scale = e4m3.quantize_rows(c.astype(np.float32))
    return e4m3.dequantize_rows(codes, scale), round_to_bf16(kr), codes, scale


def overwrite_positions(c, k_r, positions, entries, rows):
    """Sequence view with the appended entries placed at their positions.

    ``c``/``k_r`` are one sequence's gathered cache rows; ``rows`` selects which
    appended entries belong to it and ``positions`` gives their positions.
    """
    c_st, kr_st, _, _ = entries
    c = np.array(c, copy=True)
    k_r = np.array(k_r, copy=True)
    for i, p in zip(rows, positions):
        c[int(p)] = c_st[i]
        k_r[int(p)] = kr_st[i]
    return c, k_r


# --------------------------------------------------------------------------
# One whole decode step of a workload (append, then attend)
# --------------------------------------------------------------------------
def decode_step(inp: dict, sequences=None, heads=None, seq_start=None) -> dict:
    """Expected results of one decode step for the selected sequences and heads.

    ``seq_start`` (optional, one int per sequence) is each sequence's first
    visible key position: a query at position p then attends to the keys at
    positions seq_start[b] .. p only (keys before it evicted, or a sliding
    window; "MLA 之后，KV cache 确实得重新理解一遍", "所以 cache 逻辑到底哪里要重写").

    ``inp`` holds numpy arrays (weights float64, pools as described in
    ``gather_sequence``) and the scalars ``page_size``, ``q_per_seq``,
    ``cache_dtype``, ``softmax_scale``, ``rope_theta``, ``d_h``, ``d_c``.
    The new tokens' cache entries are computed here from their hidden states
    (append first), then each query attends over every key at a position up to
    its own. Returns {"entries": ..., "rows": {(b, j): decode_rows(...)}}.
    """
    P, q_per_seq = inp["page_size"], inp["q_per_seq"]
    theta, scale, d_h, d_c = inp["rope_theta"], inp["softmax_scale"], inp["d_h"], inp["d_c"]
    seq_lens = np.asarray(inp["seq_lens"], dtype=np.int64)
    new_seq = np.asarray(inp["new_seq_idx"], dtype=np.int64)
    new_pos = np.asarray(inp["new_pos"], dtype=np.int64)
    entries = append_entries(inp["new_h"], inp["w_dkv"], inp["w_kr"], new_pos,
                             inp["cache_dtype"], theta) if new_pos.size else None
    B = seq_lens.size
    sequences = range(B) if sequences is None else sequences
    rows = {}
    for b in sequences:
        L = int(seq_lens[b])
        c, kr = gather_sequence(inp["cache"], inp["cache_dtype"], inp["block_table"], b, L, P, d_c)
        mine = np.nonzero(new_seq == b)[0]
        if entries is not None and mine.size:
            c, kr = overwrite_positions(c, kr, new_pos[mine], entries, mine)
        for j in range(q_per_seq):
            p = L - q_per_seq + j
            if inp.get("q") is not None:
                qrow = np.asarray(inp["q"][b * q_per_seq + j], np.float64)
                q_nope, q_rope = qrow[:, :d_h], qrow[:, d_h:]
            else:
                k = int(np.nonzero((new_seq == b) & (new_pos == p))[0][0])
                qn, qr = query_projection(inp["new_h"][k:k + 1], inp["w_q"], d_h)
                q_nope, q_rope = qn[0], qr[0]
            vis = max(p + 1, 0)
            lo = 0 if seq_start is None else min(max(int(seq_start[b]), 0), vis)
            rows[(b, j)] = decode_rows(q_nope, q_rope, p, c[lo:vis], kr[lo:vis], inp["w_uk"],
                                       inp["w_uv"], scale, theta, heads,
                                       inp.get("act_dtype", "f32"))
            rows[(b, j)]["q_nope"], rows[(b, j)]["q_rope"] = q_nope, q_rope
    return {"entries": entries, "rows": rows}


# --------------------------------------------------------------------------
# Chunked prefill: many query tokens per sequence, explicit keys and values
# --------------------------------------------------------------------------
def explicit_prefill_head(q_nope_h, q_rope_rot_h, q_pos, c, k_r, w_uk_h, w_uv_h, scale: float,
                          store=None, lo: int = 0):
    """Causal attention of a chunk of queries of one head in the explicit form.

    The training-time form ("MLA 之后，KV cache 确实得重新理解一遍", "第一步，训练时";
    "MLA 是什么 | dg's Blog", "完整代码"): every cached token's key
    k_t = [W_UK[h] c_t ; k_R,t] and value v_t = W_UV[h] c_t are formed once,
    and query i (at position q_pos[i]) attends over the keys at positions
    lo .. q_pos[i] with a max-subtracted softmax (``lo`` > 0: the keys before
    it evicted, or a sliding window; "MLA 之后，KV cache 确实得重新理解一遍",
    "所以 cache 逻辑到底哪里要重写").

    q_nope_h [C, d_h], q_rope_rot_h [C, d_rope] (rotated at q_pos), c [L, d_c],
    k_r [L, d_rope]. ``store`` (optional) is applied to c, to the rotated
    query and to the formed keys and values, modelling a format they are kept
    in. Returns (o [C, d_v], lse [C]); a query that sees no key gets o = 0 and
    lse = -inf.
    """
    keep = (lambda x: np.asarray(x, np.float64)) if store is None else store
    c = keep(c)
    q_n = np.asarray(q_nope_h, np.float64)
    q_r = keep(q_rope_rot_h)
    k_c = keep(up_project(c, w_uk_h))
    v = keep(up_project(c, w_uv_h))
    k_r = np.asarray(k_r, np.float64)
    C, L, d_v = q_n.shape[0], c.shape[0], v.shape[1]
    s = scale * (q_n @ k_c.T + q_r @ k_r.T)                         # [C, L]
    t = np.arange(L)[None, :]
    visible = (t <= np.asarray(q_pos, np.int64)[:, None]) & (t >= lo)
    o = np.zeros((C, d_v))
    lse = np.full(C, -math.inf)
    for i in range(C):
        si = s[i, visible[i]]
        if si.size == 0:
            continue
        m = np.max(si)
        e = np.exp(si - m)
        z = np.sum(e)
        o[i] = (e / z) @ v[visible[i]]
        lse[i] = m + math.log(z)
    return o, lse


def prefill_step(inp: dict, sequences=None, heads=None, act_dtype: str = "bf16", seq_start=None) -> dict:
    """Expected results of one chunked-prefill attention call.

    Sequence b's cache holds its first seq_lens[b] tokens (the chunk's own
    tokens already appended); its q_per_seq = C queries sit at positions
    seq_lens[b] - C + j, as for decode, and each sees the keys up to its own
    position (and, with ``seq_start``, from seq_start[b] on). ``inp`` is as for
    ``decode_step`` (queries ``q`` [B*C, n_h, d_h + d_rope], RoPE part not yet
    rotated).

    Returns {b: {"o": [C, H, d_v], "lse": [C, H], "o_s": ..., "lse_s": ...,
    "heads": [...]}}: "o"/"lse" exact; "o_s"/"lse_s" with the query's rotated
    part, c and the formed keys and values kept in the activation format
    (``act_dtype``), as an implementation that stores them would see them.
    """
    P, C = inp["page_size"], inp["q_per_seq"]
    theta, scale, d_h, d_c = inp["rope_theta"], inp["softmax_scale"], inp["d_h"], inp["d_c"]
    seq_lens = np.asarray(inp["seq_lens"], dtype=np.int64)
    n_h = np.asarray(inp["w_uk"]).shape[0]
    heads = list(range(n_h)) if heads is None else list(heads)
    sequences = range(seq_lens.size) if sequences is None else sequences
    store = lambda x: round_to_storage(x, act_dtype)
    out = {}
    for b in sequences:
        L = int(seq_lens[b])
        lo = 0 if seq_start is None else min(max(int(seq_start[b]), 0), L)
        # Positions before the window are never read (their pages may be gone).
        d_r = np.asarray(inp["q"]).shape[-1] - d_h
        c, kr = np.zeros((L, d_c)), np.zeros((L, d_r))
        if L > lo:
            cw, krw = gather_sequence(inp["cache"], inp["cache_dtype"], inp["block_table"], b, L, P, d_c,
                                      first=lo)
            c[lo:], kr[lo:] = cw, krw
        pos = L - C + np.arange(C)
        q = np.asarray(inp["q"][b * C:(b + 1) * C], np.float64)
        q_rot = rope(q[:, :, d_h:], pos, theta)
        res = {k: [] for k in ("o", "lse", "o_s", "lse_s")}
        for h in heads:
            o, l = explicit_prefill_head(q[:, h, :d_h], q_rot[:, h], pos, c, kr, inp["w_uk"][h], inp["w_uv"][h], scale,
                                         lo=lo)
            o_s, l_s = explicit_prefill_head(q[:, h, :d_h], q_rot[:, h], pos, c, kr, inp["w_uk"][h], inp["w_uv"][h],
                                             scale, store=store, lo=lo)
            for k, v in (("o", o), ("lse", l), ("o_s", o_s), ("lse_s", l_s)):
                res[k].append(v)
        out[b] = {k: np.stack(v, axis=1) for k, v in res.items()}
        out[b]["heads"] = heads
    return out
