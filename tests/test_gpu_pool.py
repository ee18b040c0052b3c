"""The page pool on a real cache: a forked sequence shares its parent's full
pages and gets a copy of the partial one (mla_copy_pages, byte for byte);
appends land only in each sequence's own slots; decode over both, and over the
parent after its leading pages are evicted, matches the oracle."""
import numpy as np
import pytest
import torch

import mla_inputs as W
from oracle import mla_oracle as O
from tests.gpu_harness import check_bf16, dims_of
from tests.oracle_io import bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import mla_latent_kv_80_b300 as M
    return M


def test_forked_sequences_share_pages_and_decode_correctly(M):
    w = W.shrink(W.DSV2_B16, batch=2, seq_len=300, append_new=0)
    x = W.generate(w)  # weights and queries of DeepSeek-V2 shape
    dims = dims_of(M, w)
    P, NP = w.page_size, 24
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(77)
    ckv = torch.full((NP * P, w.d_c + w.d_rope), float("nan"), dtype=torch.bfloat16, device=dev)
    cache = M.make_cache(ckv, None, None, NP)
    pool = M.PagePool(NP, P, max_seqs=4, max_pages_per_seq=8)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    a = pool.new_seq()
    pool.reserve(a, 300)
    tab = pool.block_table()
    slots_a = torch.tensor([int(tab[a, t // P]) * P + t % P for t in range(300)], device=dev)
    ckv[slots_a] = torch.randn(300, w.d_c + w.d_rope, generator=g).to(torch.bfloat16).to(dev)

    b = pool.fork(a, 250)  # pages 0-2 shared; page 3 (positions 192-255) copied
    src, dst = pool.take_copies()
    assert src.tolist() == [int(tab[a, 3])] and len(dst) == 1
    M.mla_copy_pages(dims, cache, 1, src.to(dev), dst.to(dev), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    s0, d0 = int(src[0]) * P, int(dst[0]) * P
    before = ckv.clone()
    assert torch.equal(ckv[d0:d0 + P].view(torch.int16), ckv[s0:s0 + P].view(torch.int16))
    tab = pool.block_table()
    assert tab[b, :3].tolist() == tab[a, :3].tolist() and int(tab[b, 3]) == int(dst[0])
    assert [pool.page_refs(int(p)) for p in tab[a, :4]] == [2, 2, 2, 1]

    # One new token each: the parent at position 300, the child at 250.
    pool.reserve(a, 301)
    pool.reserve(b, 251)
    tab = pool.block_table()
    h = torch.randn(2, w.d_model, generator=g).to(torch.bfloat16)
    seq_idx = torch.tensor([a, b], dtype=torch.int32)
    pos = torch.tensor([300, 250], dtype=torch.int32)
    ws_bytes = M.mla_cache_append_workspace_size(dims, 2)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    M.mla_cache_append(dims, cache, 2, h.to(dev), x["w_dkv"].to(dev), x["w_kr"].to(dev), seq_idx.to(dev),
                       pos.to(dev), tab.to(dev), tab.shape[1], ws, ws_bytes, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    new_a = int(tab[a, 300 // P]) * P + 300 % P
    new_b = int(tab[b, 250 // P]) * P + 250 % P
    changed = torch.nonzero(torch.any(ckv.view(torch.int16) != before.view(torch.int16), dim=1)).flatten()
    assert sorted(changed.tolist()) == sorted([new_a, new_b]), "an append touched another slot"
    c_new, kr_new, _, _ = O.append_entries(h.double().numpy(), x["w_dkv"].double().numpy(),
                                           x["w_kr"].double().numpy(), pos.numpy(), "bf16")
    got_new = ckv[[new_a, new_b]].float().cpu().numpy()
    check_bf16(got_new[:, :w.d_c], c_new, "appended c_KV")
    check_bf16(got_new[:, w.d_c:], kr_new, "appended k_R")

    # Decode both over the pool's table rows, then the parent over a window
    # after its first two pages are evicted (the child still holds them).
    heads = [0, 64, 127]
    qa = W.stage_inputs(w, 2)["q_abs"]
    seq_lens = torch.tensor([301, 251], dtype=torch.int32)
    cache_host = {"ckv": bf16_bits(ckv.cpu())}
    full_tab = pool.block_table()[[a, b]].numpy()

    def decode(table, start):
        step = M.DecodeStep(dims, 2, 1, 0, 0, dev)
        step.q_abs.copy_(qa.to(dev))
        step.status.zero_()
        st = None if start is None else torch.tensor(start, dtype=torch.int32, device=dev)
        step.decode(cache, table.to(dev), seq_lens.to(dev), seq_start=st)
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        return step.o_lat.float().cpu().numpy(), step.lse.cpu().numpy()

    def check(o_lat, lse, starts, what):
        for r in range(2):
            L = int(seq_lens[r])
            c, kr = O.gather_sequence(cache_host, "bf16", full_tab, r, L, P, w.d_c)
            lat, l = O.absorbed_attention(qa.double().numpy()[r, heads], c[starts[r]:L], kr[starts[r]:L],
                                          w.softmax_scale)
            check_bf16(o_lat[r, heads], lat, f"{what} row {r} o_lat")
            check_bf16(lse[r, heads], l, f"{what} row {r} lse", stored_bf16=False)

    o_lat, lse = decode(pool.block_table()[[a, b]], None)
    check(o_lat, lse, [0, 0], "shared prefix")
    free0 = pool.free_pages()
    pool.evict_before(a, 130)
    assert pool.seq_info(a) == (301, 130) and pool.free_pages() == free0
    win_tab = pool.block_table()[[a, b]]
    assert win_tab[0, :2].tolist() == [-1, -1]
    o_lat, lse = decode(win_tab, [pool.seq_info(a)[1], 0])
    check(o_lat, lse, [130, 0], "after eviction")
    pool.free_seq(b)
    assert pool.free_pages() == free0 + 3  # pages 0-1 and the child's copied page
