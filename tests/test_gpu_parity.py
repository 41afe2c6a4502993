"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on seeded inputs.

Small and ragged shapes are compared on every output element; the full-size workloads (at the
launch configuration the benchmark times) on sampled query rows that the oracle computes one by
one. Tolerances are in tests/parity.py.
"""

import numpy as np
import pytest
import torch

import mla_inputs as mi
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    import sparse_latent_attention_norm_b300 as m
    from sparse_latent_attention_norm_b300 import build
    build.build()
    m.clear_status()
    return m


def to_dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def out_f64(out, rows, B, T, H):
    o = out.float().cpu().numpy().reshape(B * T, H, 128)
    return o[rows] if rows is not None else o


def run_and_compare(mla, oracle_lib, inp, rows=None, heads=None, what=""):
    d = to_dev(inp)
    B, T, H, _ = inp["q"].shape
    out, lse, nk = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"],
                                      n_keys=True)
    torch.cuda.synchronize()
    assert mla.get_status() == 0
    ref_out, ref_lse, ref_n = oracle_lib.prefill(inp, rows=rows, heads=heads)
    sel = np.arange(B * T) if rows is None else np.asarray(rows)
    h0, h1 = (0, H) if heads is None else heads
    og = out.float().cpu().numpy().reshape(B * T, H, 128)[sel][:, h0:h1]
    lg = lse.cpu().numpy().reshape(B * T, H)[sel][:, h0:h1]
    assert np.array_equal(nk.cpu().numpy().reshape(-1)[sel], ref_n), f"{what}: n_keys differ"
    return parity.compare(og, lg, ref_out, ref_lse, what)


SMALL = [
    ("tiny", mi.WORKLOADS["tiny"]),
    ("ragged_b2", mi.custom("ragged_b2", 2, 333, 5, 48, "uniform", seed_id=201)),
    ("stress_small", mi.custom("stress_small", 1, 520, 4, 64, "uniform", stress=True, seed_id=202)),
    ("clustered_small", mi.custom("clustered_small", 1, 1100, 2, 128, "clustered", recent=256, seed_id=203)),
    ("dense_small", mi.custom("dense_small", 1, 200, 2, 256, "dense", seed_id=204)),
    ("single_query", mi.custom("single_query", 1, 1, 3, 4, "tiny", seed_id=205)),
    ("one_tile_edge", mi.custom("one_tile_edge", 1, 129, 1, 16, "uniform", seed_id=206)),
]


@pytest.mark.parametrize("name,w", SMALL, ids=[s[0] for s in SMALL])
def test_small_all_elements(mla, oracle_lib, name, w):
    inp = mi.make_inputs(w)
    run_and_compare(mla, oracle_lib, inp, what=name)


FULL = ["dense_causal", "headline", "stress", "long_context"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(mla, oracle_lib, name):
    w = mi.WORKLOADS[name]
    inp = mi.make_inputs(w)
    rows = parity.sample_rows(w.B, w.T, w.K, n_random=16, seed=w.seed_id)
    heads = (0, 16) if name == "long_context" else None
    run_and_compare(mla, oracle_lib, inp, rows=rows, heads=heads, what=name)


@pytest.mark.parametrize("name", ["tiny", "headline", "long_context"])
def test_selection_bitsets_bit_exact(mla, oracle_lib, name):
    w = mi.WORKLOADS[name] if name != "tiny" else mi.custom("sel", 2, 300, 1, 80, "uniform", stress=True, seed_id=7)
    topk = mi.make_topk(w)
    if name == "tiny":
        topk[0, 5, :10] = [-3, 299, 300, 10_000, 5, 5, 4, -1, 6, 7]   # out of range, non-causal, dups
    bits, nk = mla.canon_select(torch.from_numpy(topk).cuda(), w.T)
    want_bits, want_n = parity.expected_bits(topk, w.T, oracle_lib)
    got = bits.cpu().numpy().view(np.uint32)
    W = got.shape[-1]
    for b in range(w.B):
        for t in range(w.T):
            words = (t // 128 + 1) * 4
            assert np.array_equal(got[b, t, :words], want_bits[b, t, :words]), (b, t)
    assert np.array_equal(nk.cpu().numpy(), want_n)
    assert W == (w.T + 127) // 128 * 4


def test_kvnorm_wkvb_against_oracle(mla, oracle_lib):
    for w in [mi.custom("k1a", 1, 200, 3, 8, "uniform", seed_id=11),
              mi.custom("k1b", 2, 4096 + 77, 2, 8, "uniform", stress=True, seed_id=12)]:
        inp = mi.make_inputs(w)
        d = to_dev(inp)
        kv, klo = mla.kvnorm_wkvb(d["c_kv"], d["gamma"], d["wkv_b"])
        kn = mla.k_nope_from(kv, klo).double().cpu().numpy()            # [B, H, T, 128]
        v = kv[..., 128:].double().cpu().numpy()
        y = oracle_lib.kv_norm(inp["c_kv"].reshape(-1, 512), inp["gamma"].numpy())
        rkn, rv = oracle_lib.up_proj(y, inp["wkv_b"])                     # [B*T, H, 128]
        rkn = rkn.reshape(w.B, w.T, w.H, 128).transpose(0, 2, 1, 3)
        rv = rv.reshape(w.B, w.T, w.H, 128).transpose(0, 2, 1, 3)
        # k_nope: fp32 accumulation + hi/lo representation (about 2^-14 relative)
        ek = np.abs(kn - rkn)
        assert ek.max() <= 2e-4 * max(1.0, np.abs(rkn).max()), ek.max()
        assert np.linalg.norm(kn - rkn) / np.linalg.norm(rkn) < 1e-4
        # v: fp16 rounding (2^-11 relative) on top of the fp32 accumulation (absolute ~1e-6)
        ev = np.abs(v - rv) - 2.0 ** -11 * np.abs(rv)
        assert ev.max() <= 1e-5, ev.max()


def test_staged_calls_equal_fused_call(mla):
    w = mi.custom("staged", 2, 300, 3, 40, "uniform", seed_id=13)
    d = to_dev(mi.make_inputs(w))
    out, lse = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"])
    bits, _ = mla.canon_select(d["topk_idx"], w.T)
    kv, klo = mla.kvnorm_wkvb(d["c_kv"], d["gamma"], d["wkv_b"])
    out2, lse2 = mla.sparse_attention(d["q"], d["k_pe"], kv, klo, bits)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_order_and_duplicate_invariance_bit_identical(mla):
    w = mi.custom("perm", 1, 700, 2, 96, "uniform", seed_id=14)
    inp = mi.make_inputs(w)
    d = to_dev(inp)
    out, lse = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"])
    topk = inp["topk_idx"].numpy().copy()
    rng = np.random.default_rng(3)
    for t in range(w.T):
        rng.shuffle(topk[0, t])
    topk = np.concatenate([topk, topk[..., :17]], axis=-1)   # appended duplicates
    out2, lse2 = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"],
                                    torch.from_numpy(np.ascontiguousarray(topk)).cuda())
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_empty_rows_and_invalid_indices(mla, oracle_lib):
    w = mi.custom("empty", 1, 260, 2, 8, "tiny", seed_id=15)
    inp = mi.make_inputs(w)
    topk = inp["topk_idx"].numpy().copy()
    topk[0, 3] = [5, 6, 7, 8, 9, 10, 11, 12]        # all after t = 3: empty set
    topk[0, 200] = [-1, -5, 201, 259, 300, 250, 220, 210]   # negative, non-causal, >= T
    inp["topk_idx"] = torch.from_numpy(topk)
    run_and_compare(mla, oracle_lib, inp, what="empty rows")
    d = to_dev(inp)
    mla.clear_status()
    mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"])
    assert mla.get_status() == 0                    # ignored without validation
    mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"], validate=True)
    assert mla.get_status() == 4                    # MLA_ERR_INDEX
    mla.clear_status()
    assert mla.get_status() == 0


def test_library_allocated_workspace_and_host_path(mla):
    w = mi.custom("host", 1, 256, 2, 32, "uniform", seed_id=16)
    inp = mi.make_inputs(w)
    d = to_dev(inp)
    ws = mla.alloc_workspace(w.B, w.T, w.H, w.K)
    out1, lse1 = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"], workspace=ws)
    out2, lse2 = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"])
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    hp = mla.HostPrefill(w.B, w.T, w.H, w.K)
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out3, lse3 = hp(host)
    assert torch.equal(out3, out1.cpu()) and torch.equal(lse3, lse1.cpu())


def test_pipelined_host_path_matches_direct_calls(mla):
    # five steps with different inputs through the three-stream pipeline (two buffer sets): each
    # step's host results equal the direct device call on the same inputs
    ws = [mi.custom("pipe", 1, 300, 2, 48, "uniform", seed_id=40 + i) for i in range(5)]
    inps = [mi.make_inputs(w) for w in ws]
    refs = []
    for inp in inps:
        d = to_dev(inp)
        o, l = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"])
        refs.append((o.cpu(), l.cpu()))
    pipe = mla.HostPrefillPipeline(1, 300, 2, 48)
    hosts = [{k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()} for inp in inps]
    handles = []
    for i, h in enumerate(hosts):
        handles.append(pipe.submit(h))
        if i >= 1:   # results of a step are read before its host buffers come round again
            out, lse = pipe.result(handles[i - 1])
            assert torch.equal(out, refs[i - 1][0]) and torch.equal(lse, refs[i - 1][1])
    out, lse = pipe.result(handles[-1])
    assert torch.equal(out, refs[-1][0]) and torch.equal(lse, refs[-1][1])
    assert mla.get_status() == 0


def test_run_on_side_stream(mla):
    w = mi.custom("stream", 1, 384, 2, 64, "uniform", seed_id=17)
    d = to_dev(mi.make_inputs(w))
    out1, lse1 = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out2, lse2 = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"], stream=s)
    s.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
