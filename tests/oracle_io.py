"""Conversion of generated torch inputs into the numpy form the oracle reads."""
import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def to_f64(t):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return t.to(torch.float32).numpy().astype(np.float64)
    return t.numpy().astype(np.float64)


def oracle_inputs(x: dict) -> dict:
    """Numpy view of a generated workload for ``oracle.mla_oracle.decode_step``."""
    w = x["workload"]
    c = x["cache"]
    if w.cache_dtype == "bf16":
        cache = {"ckv": bf16_bits(c["ckv"])}
    elif w.cache_dtype == "f32":
        cache = {"ckv": c["ckv"].numpy()}
    else:
        cache = {"ckv": c["ckv"].numpy(), "kr": bf16_bits(c["kr"]), "scale": c["scale"].numpy()}
    return {
        "page_size": w.page_size, "q_per_seq": w.q_per_seq, "cache_dtype": w.cache_dtype,
        "act_dtype": w.act_dtype,
        "softmax_scale": w.softmax_scale, "rope_theta": w.rope_theta, "d_h": w.d_h, "d_c": w.d_c,
        "seq_lens": x["seq_lens"].numpy(), "block_table": x["block_table"].numpy(),
        "new_seq_idx": x["new_seq_idx"].numpy(), "new_pos": x["new_pos"].numpy(),
        "new_h": to_f64(x["new_h"]), "w_dkv": to_f64(x["w_dkv"]), "w_kr": to_f64(x["w_kr"]),
        "w_uk": to_f64(x["w_uk"]), "w_uv": to_f64(x["w_uv"]), "w_q": to_f64(x["w_q"]),
        "q": to_f64(x["q"]), "cache": cache,
    }
