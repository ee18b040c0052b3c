"""The failure path without a fault: a bounded device wait that runs out sets
MLA_ERR_DEVICE_TIMEOUT in the status word, and the context stays usable (a
decode step right after it is correct)."""
import pytest
import torch

import mla_inputs as W
from tests.gpu_harness import DeviceRun, compare, oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import mla_latent_kv_80_b300 as M
    return M


def test_bounded_wait_times_out_and_the_context_stays_usable(M):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.mla_selftest_bounded_wait(1_000_000, status)  # 1 ms on a barrier nothing arrives on
    torch.cuda.synchronize()
    assert int(status.item()) == -6  # MLA_ERR_DEVICE_TIMEOUT
    # An earlier error is kept: the status word records the first failure.
    M.mla_selftest_bounded_wait(1_000_000, status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    w = W.shrink(W.DSV2_B16, batch=2, seq_len=300)
    x = W.generate(w)
    out = DeviceRun(M, x).run()
    compare(out, oracle_for(x, heads=[0, 127]), w, "after a timed-out wait")


def test_limit_is_checked_on_the_host(M):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(M.MlaError) as e:
        M.mla_selftest_bounded_wait(3_000_000_000, status)
    assert e.value.code == -1
