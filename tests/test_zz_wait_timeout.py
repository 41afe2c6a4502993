"""The failure path of the kernels' bounded waits, run on the GPU without a fault.

mla_selftest_wait_timeout makes one thread wait, through the same bounded wait every kernel uses,
on an mbarrier nothing arrives on. The wait must give up at its limit (about 2 s), the status word
must report MLA_ERR_TIMEOUT, and once the status is cleared the same context must still run the
prefill correctly.

The file name makes pytest collect it after every other test, so a failure here cannot leave a
recorded timeout behind for them.
"""

import numpy as np
import pytest
import torch

import mla_inputs as mi
from tests import parity

pytestmark = pytest.mark.gpu

MLA_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    import sparse_latent_attention_norm_b300 as m
    from sparse_latent_attention_norm_b300 import build
    build.build()
    m.clear_status()
    return m


def test_bounded_wait_gives_up_and_context_survives(mla, oracle_lib):
    mla.clear_status()
    try:
        completed, ms = mla.selftest_wait_timeout()
        status = mla.get_status()
    finally:
        mla.clear_status()
    assert completed == 0
    assert 1500 <= ms <= 10000, ms
    assert status == MLA_ERR_TIMEOUT
    assert mla.get_status() == 0
    # the same context runs the prefill afterwards, within the parity tolerances
    w = mi.custom("after_timeout", 1, 200, 4, 48, "uniform", stress=False, seed_id=77)
    inp = mi.make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out, lse, nk = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"],
                                      n_keys=True)
    torch.cuda.synchronize()
    assert mla.get_status() == 0
    ref_out, ref_lse, ref_n = oracle_lib.prefill(inp)
    assert np.array_equal(nk.cpu().numpy().reshape(-1), ref_n)
    parity.compare(out.float().cpu().numpy().reshape(-1, 4, 128), lse.cpu().numpy().reshape(-1, 4), ref_out, ref_lse,
                   "after the timeout")
