"""Where the end-to-end bf16 bound comes from (CPU only, oracle arithmetic).

The stated bf16 bound is a mean relative error of at most 2e-3 (relative L1
against the reference rounded to bf16). The C ABI itself fixes three bf16
roundings on the way from the query to the output, whatever kernel implements
it: q_abs is a bf16 tensor between the absorb and decode calls, the
probabilities P enter a bf16 tensor-core product with c_KV, and o_lat is a bf16
tensor between the decode and output calls. This test applies exactly those
roundings to the float64 oracle on DeepSeek-V2 shapes and shows that

  * the decode stage alone (its own bf16 P, compared with the oracle fed the
    same bf16 q_abs) stays under 2e-3;
  * the raw end-to-end output o, compared with the exact oracle, exceeds 2e-3,
    so no implementation of this ABI meets 2e-3 end to end, but it stays under
    the derived bound END_TO_END_REL_BF16 = 4e-3 that the GPU tests use;
  * o against the oracle's chained stage result o_s (two chained bf16 stages:
    decode then output) also stays under that derived bound.
"""
import numpy as np
import pytest

import mla_inputs as W
from oracle import mla_oracle as O
from tests.gpu_harness import END_TO_END_REL_BF16, _bf16, rel_l1
from tests.oracle_io import oracle_inputs

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.fixture(scope="module")
def chain():
    L = 2000
    w = W.shrink(W.DSV2_B16, batch=1, seq_len=L)
    x = W.generate(w)
    inp = oracle_inputs(x)
    heads = list(range(0, 128, 4))
    ref = O.decode_step(inp, sequences=[0], heads=heads)
    r = ref["rows"][(0, 0)]
    c, kr = O.gather_sequence(inp["cache"], "bf16", inp["block_table"], 0, L, w.page_size, w.d_c)
    mine = np.nonzero(inp["new_seq_idx"] == 0)[0]
    c, kr = O.overwrite_positions(c, kr, inp["new_pos"][mine], ref["entries"], mine)
    keys = np.concatenate([c, kr], axis=1)
    # The ABI's roundings, nothing else: bf16 q_abs, bf16 P in P.c_KV (the row
    # sum l adds the unrounded probabilities), bf16 o_lat, bf16 o.
    q_abs = O.round_to_bf16(r["q_abs"])
    s = w.softmax_scale * (q_abs @ keys.T)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    o_lat = O.round_to_bf16((O.round_to_bf16(e) @ c) / e.sum(axis=1, keepdims=True))
    o = O.round_to_bf16(np.stack([inp["w_uv"][h] @ o_lat[i] for i, h in enumerate(heads)]))
    return {"o_lat": o_lat, "o": o, "ref": r}


def test_decode_stage_alone_meets_the_stated_bound(chain):
    assert rel_l1(chain["o_lat"], _bf16(chain["ref"]["o_lat_s"])) < 2e-3


def test_end_to_end_needs_the_derived_bound(chain):
    e2e = rel_l1(chain["o"], _bf16(chain["ref"]["o"]))
    assert 2e-3 < e2e < END_TO_END_REL_BF16


def test_chained_stages_stay_under_the_derived_bound(chain):
    assert rel_l1(chain["o"], _bf16(chain["ref"]["o_s"])) < END_TO_END_REL_BF16
    assert rel_l1(chain["o_lat"], _bf16(chain["ref"]["o_lat"])) < END_TO_END_REL_BF16
