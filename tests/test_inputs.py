"""The seeded input generator: determinism and the workload recipes (CPU only)."""

import numpy as np
import torch

import mla_inputs as mi


def _sets(topk, b, t):
    return {int(j) for j in topk[b, t] if 0 <= j <= t}


def test_deterministic():
    w = mi.WORKLOADS["tiny"]
    a, b = mi.make_inputs(w), mi.make_inputs(w)
    for k in ["q", "c_kv", "k_pe", "gamma", "wkv_b", "topk_idx"]:
        assert torch.equal(a[k], b[k])


def test_shapes_and_dtypes():
    w = mi.WORKLOADS["tiny"]
    x = mi.make_inputs(w)
    assert x["q"].shape == (1, 64, 4, 192) and x["q"].dtype == torch.bfloat16
    assert x["c_kv"].shape == (1, 64, 512) and x["k_pe"].shape == (1, 64, 64)
    assert x["wkv_b"].shape == (4 * 256, 512) and x["gamma"].dtype == torch.float32
    assert x["topk_idx"].shape == (1, 64, 32) and x["topk_idx"].dtype == torch.int32
    g = x["gamma"]
    assert torch.equal(g, g.to(torch.bfloat16).float()) and g.min() >= 0.5 and g.max() <= 1.5


def test_tiny_recipe_counts():
    x = mi.make_inputs(mi.WORKLOADS["tiny"])
    topk = x["topk_idx"].numpy()
    n = [len(_sets(topk, 0, t)) for t in range(64)]
    assert n == [min(t + 1, 32) for t in range(64)] and sum(n) == 1552
    for t in range(64):
        assert t in topk[0, t] and len(set(topk[0, t].tolist())) == 32   # distinct entries


def test_uniform_recipe_small():
    w = mi.custom("u", 1, 300, 2, 64, pattern="uniform", seed_id=3)
    topk = mi.make_topk(w)
    for t in range(300):
        row = topk[0, t]
        assert t in row and len(set(row.tolist())) == 64
        if t >= 63:
            assert row[0] == t
            assert all(0 <= j < t for j in row[1:])
        else:
            assert set(range(t + 1)) <= set(row.tolist()) and all(j < 300 for j in row)


def test_clustered_recipe_small():
    w = mi.custom("c", 1, 600, 2, 64, pattern="clustered", recent=128, seed_id=4)
    topk = mi.make_topk(w)
    for t in range(63, 600):
        row = topk[0, t]
        assert row[0] == t and len(set(row.tolist())) == 64
        recent = sum(1 for j in row if t - 127 <= j <= t)
        if t - 127 >= 32:
            assert recent == 32                    # t + 31 from the recent window, 32 earlier


def test_dense_recipe_covers_all_causal_keys():
    w = mi.custom("d", 1, 40, 2, 64, pattern="dense", seed_id=5)
    topk = mi.make_topk(w)
    for t in range(40):
        assert _sets(topk, 0, t) == set(range(t + 1))


def test_stress_recipe_has_duplicates_and_shuffles():
    w = mi.custom("s", 1, 200, 2, 60, pattern="uniform", stress=True, seed_id=6)
    topk = mi.make_topk(w)
    n_dup = int(0.05 * 60)
    for t in range(200):
        row = topk[0, t]
        assert t in row
        assert len(set(row.tolist())) >= 60 - n_dup and len(set(row.tolist())) < 60
    assert sum(topk[0, t, 0] == t for t in range(200)) < 50     # t no longer always first
