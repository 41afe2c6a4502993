"""The allocation-free prefill entry point, mla_sparse_prefill_noalloc, called through the C ABI.

It exists for callers that cannot allocate device memory when they run the prefill (code running
inside an allocator or memory-pool callback, engines that fix their device footprint ahead of
time, hosts that forbid cudaMalloc during a step): its scratch is a device array the library owns.
Two calls in a row, on different shapes, must give the same bits as the workspace-taking entry
point and match the oracle within the parity tolerances; a problem too large for that array must
be refused before any launch.

The file name makes pytest collect it last, so a run that stops at the first failure has already
run every other test.
"""

import ctypes

import pytest
import torch

import mla_inputs as mi
from tests import parity

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(L, mla, d, out, lse, dims):
    return L.mla_sparse_prefill_noalloc(_ptr(d["q"]), _ptr(d["c_kv"]), _ptr(d["k_pe"]), _ptr(d["gamma"]),
                                        _ptr(d["wkv_b"]), _ptr(d["topk_idx"]), _ptr(out), _ptr(lse), dims,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    import sparse_latent_attention_norm_b300 as m
    from sparse_latent_attention_norm_b300 import build
    build.build()
    m.clear_status()
    return m


def test_noalloc_matches_workspace_entry_point_on_two_calls(mla, oracle_lib):
    # Both entry points launch the same kernels on the same inputs, so their results must be the
    # same bits; each is also checked against the oracle within the parity tolerances.
    L = mla.lib()
    workloads = [mi.WORKLOADS["tiny"], mi.custom("noalloc_ragged", 2, 333, 5, 48, "uniform", seed_id=301)]
    for w in workloads:                                           # call 1, then call 2 on another shape
        inp = mi.make_inputs(w)
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        assert mla.workspace_size(w.B, w.T, w.H, w.K) <= 64 << 20
        ref_out, ref_lse = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"],
                                              workspace=mla.alloc_workspace(w.B, w.T, w.H, w.K))
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = _noalloc(L, mla, d, out, lse, mla.Dims(w.B, w.T, w.H, w.K))
        assert rc == 0, mla.status_string(rc)
        torch.cuda.synchronize()
        assert mla.get_status() == 0
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), f"noalloc {w.name}: bits differ"
        n = w.B * w.T
        o_out, o_lse, _ = oracle_lib.prefill(inp)
        parity.compare(out.float().cpu().numpy().reshape(n, w.H, 128), lse.cpu().numpy().reshape(n, w.H),
                       o_out, o_lse, f"noalloc {w.name} vs oracle")


def test_noalloc_refuses_problems_beyond_its_scratch(mla):
    L = mla.lib()
    w = mi.WORKLOADS["tiny"]
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in mi.make_inputs(w).items()}
    out = torch.empty((1, 64, 4, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 64, 4), dtype=torch.float32, device="cuda")
    big = mla.Dims(1, 4096, 128, 2048)                            # needs ~337 MB of scratch
    assert mla.workspace_size(1, 4096, 128, 2048) > 64 << 20
    assert _noalloc(L, mla, d, out, lse, big) == 6                # MLA_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert mla.get_status() == 0
