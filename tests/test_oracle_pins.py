"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test is built so that a plausible mistake in the oracle fails it: a dropped term, a wrong
sign, index, axis or constant, a transposed operand, a lost normalisation. None of them retypes
the oracle's own code path: they use printed values, closed forms, invariants, a library routine
(numpy matmul) and an independent dense restatement of the pages' prefill excerpt.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import mla_inputs as mi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "constants.json")


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64).numpy()


def small_inputs(B=1, T=48, H=3, K=24, pattern="tiny", seed=7, stress=False):
    w = mi.custom("pin", B, T, H, K, pattern=pattern, seed_id=seed, stress=stress)
    return mi.make_inputs(w)


# --------------------------------------------------------------------------------------------
# Literal restatement of the pages' MHA prefill (model.py 574-589) with a dense [T, T] mask, in
# numpy fp64. It shares nothing with the oracle: its own RMSNorm, a numpy matmul for wkv_b, the
# einsum scores, scatter-built index mask plus causal mask, dense softmax, einsum with v.
# --------------------------------------------------------------------------------------------
def round_bf16(x):
    import oracle
    return oracle.round_to_bf16(x)


def rmsnorm_fp32(x, gamma, eps=1e-6):
    """RMSNorm as the excerpt writes it, in fp32 (x.float()): mean of squares summed in ascending
    feature order, x * (1 / sqrt(var + eps)), weight * x. numpy float32 ops are IEEE-rounded."""
    x = np.asarray(x, dtype=np.float32)
    g = np.asarray(gamma, dtype=np.float32)
    ss = np.zeros(x.shape[:-1], dtype=np.float32)
    for c in range(x.shape[-1]):
        ss = (ss + x[..., c] * x[..., c]).astype(np.float32)
    var = (ss / np.float32(x.shape[-1])).astype(np.float32)
    r = (np.float32(1.0) / np.sqrt((var + np.float32(eps)).astype(np.float32))).astype(np.float32)
    return (g * (x * r[..., None]).astype(np.float32)).astype(np.float32).astype(np.float64)


def literal_prefill(inp, eps=1e-6):
    q = f64(inp["q"])
    B, T, H, _ = q.shape
    c_kv = f64(inp["c_kv"])
    k_pe = f64(inp["k_pe"])
    gamma = inp["gamma"].numpy().astype(np.float64)
    W = f64(inp["wkv_b"])
    topk = np.asarray(inp["topk_idx"]).astype(np.int64)
    kv = round_bf16(rmsnorm_fp32(c_kv, gamma, eps))            # x.float() ... .to(dtype)
    kv = kv @ W.T                                               # wkv_b, weight [out, in]
    kv = kv.reshape(B, T, H, 256)
    k_nope, v = kv[..., :128], kv[..., 128:]
    k = np.concatenate([k_nope, np.broadcast_to(k_pe[:, :, None, :], (B, T, H, 64))], axis=-1)
    m = 0.1 * 1.0 * math.log(40.0) + 1.0
    scale = 192 ** -0.5 * m * m
    scores = np.einsum("bshd,bthd->bsht", q, k) * scale
    index_mask = np.full((B, T, T), -np.inf)
    for b in range(B):
        for s in range(T):
            for j in topk[b, s]:
                if 0 <= j < T:
                    index_mask[b, s, j] = 0.0
    causal = np.triu(np.full((T, T), -np.inf), k=1)
    index_mask = index_mask + causal
    scores = scores + index_mask[:, :, None, :]
    mx = scores.max(-1, keepdims=True)
    e = np.exp(scores - mx)
    z = e.sum(-1, keepdims=True)
    p = e / z
    out = np.einsum("bsht,bthd->bshd", p, v)
    lse = (mx + np.log(z))[..., 0]
    return out, lse


def test_scale_matches_printed_m_squared(oracle_lib):
    g = json.load(open(GOLDEN))
    m2 = oracle_lib.softmax_scale() * math.sqrt(g["qk_head_dim"]["value"])
    assert round(m2, g["m_squared_printed"]["digits"]) == g["m_squared_printed"]["value"]


def test_scale_reaches_the_scores(oracle_lib):
    """t = 0 with only the rotary dims of q set: lse = s_00 = scale * <q_pe, k_pe[0]>."""
    g = json.load(open(GOLDEN))
    inp = small_inputs(T=4, H=2, K=4)
    q = torch.zeros_like(inp["q"])
    q[..., 128:] = inp["q"][..., 128:]
    inp["q"] = q
    _, lse, nk = oracle_lib.prefill(inp, rows=[0])
    assert nk[0] == 1
    dot = (f64(q[0, 0, :, 128:]) * f64(inp["k_pe"][0, 0])[None, :]).sum(-1)
    m2 = lse[0] / dot * math.sqrt(192)
    assert np.all(np.round(m2, 3) == g["m_squared_printed"]["value"])


# ---------------------------------------------- kv_norm ------------------------------------
def test_kv_norm_unit_rms_with_unit_gain(oracle_lib):
    rng = np.random.default_rng(1)
    x = bf16(rng.standard_normal((64, 512)))
    y = oracle_lib.kv_norm(x, np.ones(512, np.float32), precast=True)
    rms = np.sqrt((y ** 2).mean(-1))
    ms = (f64(x) ** 2).mean(-1)
    np.testing.assert_allclose(rms, np.sqrt(ms / (ms + 1e-6)), rtol=2e-6)
    assert np.all(np.abs(rms - 1) < 3e-6)


def test_kv_norm_constant_row_closed_form(oracle_lib):
    """x = a everywhere: y = gamma * a / sqrt(a^2 + eps). At a = 2^-10, eps = 1e-6 matters."""
    g = json.load(open(GOLDEN))
    eps = g["rms_eps_code_default"]["value"]
    rng = np.random.default_rng(2)
    gamma = bf16(rng.uniform(0.5, 1.5, 512)).float().numpy()
    for a in [2.0 ** -10, 0.75, -3.0, 2.0 ** -6]:
        y = oracle_lib.kv_norm(bf16(np.full((1, 512), a)), gamma, precast=True)
        np.testing.assert_allclose(y[0], gamma.astype(np.float64) * a / math.sqrt(a * a + eps), rtol=1e-6)


def test_kv_norm_single_channel_closed_form(oracle_lib):
    """x = a e_c: mean of squares = a^2 / 512, so y_c = gamma_c a / sqrt(a^2/512 + eps)."""
    gamma = np.linspace(0.5, 1.5, 512).astype(np.float32)
    for c, a in [(0, 1.0), (311, -2.5), (511, 0.03125)]:
        x = np.zeros((1, 512))
        x[0, c] = a
        y = oracle_lib.kv_norm(bf16(x), gamma, precast=True)[0]
        expect = np.zeros(512)
        expect[c] = float(gamma[c]) * a / math.sqrt(a * a / 512 + 1e-6)
        np.testing.assert_allclose(y, expect, rtol=1e-6, atol=0)


def test_kv_norm_gain_is_elementwise_and_scale_invariant(oracle_lib):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((8, 512))
    gamma = bf16(rng.uniform(0.5, 1.5, 512)).float().numpy()
    y1 = oracle_lib.kv_norm(bf16(x), np.ones(512, np.float32), precast=True)
    yg = oracle_lib.kv_norm(bf16(x), gamma, precast=True)
    np.testing.assert_allclose(yg, y1 * gamma.astype(np.float64), rtol=2e-7)
    y4 = oracle_lib.kv_norm(bf16(x * 4.0), gamma, precast=True)   # x4 is exact in bf16
    np.testing.assert_allclose(y4, yg, rtol=2e-6)   # only eps breaks the invariance


def test_kv_norm_is_the_fp32_computation_of_the_excerpt(oracle_lib):
    """Bit-exact against an independent fp32 restatement (numpy float32, ascending order)."""
    rng = np.random.default_rng(10)
    x = bf16(rng.standard_normal((64, 512)) * np.exp(rng.uniform(-3, 3, (64, 1))))
    gamma = bf16(rng.uniform(0.5, 1.5, 512)).float().numpy()
    pre = oracle_lib.kv_norm(x, gamma, precast=True)
    assert np.array_equal(pre, rmsnorm_fp32(x.float().numpy(), gamma))


def test_kv_norm_output_is_the_bf16_cast(oracle_lib):
    """RMSNorm.forward ends with .to(dtype): the output is the pre-cast value rounded to bf16."""
    rng = np.random.default_rng(8)
    x = bf16(rng.standard_normal((16, 512)) * 3)
    gamma = bf16(rng.uniform(0.5, 1.5, 512)).float().numpy()
    y = oracle_lib.kv_norm(x, gamma)
    pre = oracle_lib.kv_norm(x, gamma, precast=True)
    assert np.array_equal(y, oracle_lib.round_to_bf16(pre))
    assert np.array_equal(y, bf16(y).double().numpy())            # every value is a bf16 value
    assert 0 < np.abs(y - pre).max() <= 2.0 ** -8 * np.abs(pre).max()


def test_round_to_bf16_matches_torch_and_ties_to_even(oracle_lib):
    rng = np.random.default_rng(9)
    f = (rng.standard_normal(20000) * np.exp(rng.uniform(-60, 60, 20000))).astype(np.float32)
    f = np.concatenate([f, np.float32([1e-40, -3e-39, 3.3e38, -3.4e38, 0.0])])
    want = torch.from_numpy(f).to(torch.bfloat16).double().numpy()     # one rounding, fp32 -> bf16
    got = oracle_lib.round_to_bf16(f.astype(np.float64))
    assert np.array_equal(got, want)
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(2 + 2.0 ** -7), 1 + 2.0 ** -8 + 2.0 ** -30])
    assert oracle_lib.round_to_bf16(ties).tolist() == [1.0, 1 + 2.0 ** -6, -2.0, 1 + 2.0 ** -7]


# ---------------------------------------------- wkv_b --------------------------------------
def test_up_proj_one_hot_layout(oracle_lib):
    """W[h*256 + f, c] = [c == (f + 7h) mod 512]: k_nope[h, d] = y[(d + 7h) % 512] and
    v[h, d] = y[(128 + d + 7h) % 512]. Fails for a transposed W, a wrong head stride or a
    swapped k_nope / v split."""
    H = 3
    W = np.zeros((H * 256, 512))
    for h in range(H):
        for f in range(256):
            W[h * 256 + f, (f + 7 * h) % 512] = 1.0
    rng = np.random.default_rng(4)
    y = rng.standard_normal((5, 512))
    kn, v = oracle_lib.up_proj(y, bf16(W))
    for h in range(H):
        d = np.arange(128)
        np.testing.assert_array_equal(kn[:, h, :], y[:, (d + 7 * h) % 512])
        np.testing.assert_array_equal(v[:, h, :], y[:, (128 + d + 7 * h) % 512])


def test_up_proj_matches_numpy_matmul(oracle_lib):
    rng = np.random.default_rng(5)
    H = 4
    W = bf16(rng.standard_normal((H * 256, 512)) / math.sqrt(512))
    y = rng.standard_normal((17, 512))
    kn, v = oracle_lib.up_proj(y, W)
    ref = (y @ f64(W).T).reshape(17, H, 256)
    np.testing.assert_allclose(kn, ref[..., :128], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(v, ref[..., 128:], rtol=1e-12, atol=1e-13)


# ---------------------------------------------- selection ----------------------------------
def test_canon_row_is_the_causal_set(oracle_lib):
    rng = np.random.default_rng(6)
    for _ in range(200):
        t = int(rng.integers(0, 300))
        idx = rng.integers(-20, 400, size=int(rng.integers(1, 90))).astype(np.int32)
        expect = sorted({int(j) for j in idx if 0 <= j <= t})
        got = oracle_lib.canon_row(idx, t)
        assert got.tolist() == expect


def test_counts_match_set_count(oracle_lib):
    inp = small_inputs(T=64, H=2, K=40, pattern="uniform", stress=True)
    _, _, nk = oracle_lib.prefill(inp)
    topk = inp["topk_idx"].numpy()
    expect = [len({int(j) for j in topk[0, t] if 0 <= j <= t}) for t in range(64)]
    assert nk.tolist() == expect


# ---------------------------------------------- prefill ------------------------------------
@pytest.mark.parametrize("pattern,T,H,K,stress", [
    ("tiny", 64, 4, 32, False),
    ("uniform", 50, 2, 16, False),
    ("uniform", 40, 3, 24, True),
    ("dense", 33, 2, 48, False),
])
def test_prefill_equals_literal_dense_mask(oracle_lib, pattern, T, H, K, stress):
    inp = small_inputs(T=T, H=H, K=K, pattern=pattern, stress=stress, seed=11)
    out, lse, _ = oracle_lib.prefill(inp)
    ref_out, ref_lse = literal_prefill(inp)
    np.testing.assert_allclose(out.reshape(ref_out.shape), ref_out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(ref_lse.shape), ref_lse, rtol=1e-11, atol=1e-12)


def test_dense_limit_is_textbook_causal_attention(oracle_lib):
    """K >= T with every causal key selected: plain causal softmax attention, no index logic."""
    inp = small_inputs(T=70, H=2, K=96, pattern="dense", seed=12)
    out, lse, nk = oracle_lib.prefill(inp)
    assert nk.tolist() == list(range(1, 71))
    y = oracle_lib.kv_norm(inp["c_kv"], inp["gamma"].numpy())[0]
    kv = (y @ f64(inp["wkv_b"]).T).reshape(70, 2, 256)
    q = f64(inp["q"])[0]
    kp = f64(inp["k_pe"])[0]
    for h in range(2):
        k = np.concatenate([kv[:, h, :128], kp], axis=1)
        s = q[:, h, :] @ k.T * oracle_lib.softmax_scale()
        s[np.triu_indices(70, 1)] = -np.inf
        p = np.exp(s - s.max(1, keepdims=True))
        o = (p @ kv[:, h, 128:]) / p.sum(1, keepdims=True)
        np.testing.assert_allclose(out[:, h, :], o, rtol=1e-11, atol=1e-12)


def test_softmax_rows_sum_to_one(oracle_lib):
    """Identical latent rows give identical v for every key; any softmax row that sums to 1 then
    returns exactly that v, whatever the (varying) scores are."""
    inp = small_inputs(T=40, H=2, K=24, pattern="uniform", seed=13)
    inp["c_kv"][:] = inp["c_kv"][0, 0]
    out, _, _ = oracle_lib.prefill(inp)
    y = oracle_lib.kv_norm(inp["c_kv"][0, :1], inp["gamma"].numpy())
    _, v = oracle_lib.up_proj(y, inp["wkv_b"])
    for t in range(40):
        np.testing.assert_allclose(out[t], v[0], rtol=1e-12, atol=1e-13)


def test_zero_query_gives_mean_of_values_and_log_count(oracle_lib):
    inp = small_inputs(T=48, H=2, K=20, pattern="uniform", seed=14, stress=True)
    inp["q"] = torch.zeros_like(inp["q"])
    out, lse, nk = oracle_lib.prefill(inp)
    np.testing.assert_allclose(lse, np.log(nk.astype(np.float64))[:, None].repeat(2, 1), rtol=0, atol=1e-13)
    y = oracle_lib.kv_norm(inp["c_kv"][0], inp["gamma"].numpy())
    _, v = oracle_lib.up_proj(y, inp["wkv_b"])
    topk = inp["topk_idx"].numpy()[0]
    for t in [0, 5, 31, 47]:
        S = sorted({int(j) for j in topk[t] if 0 <= j <= t})
        np.testing.assert_allclose(out[t], v[S].mean(0), rtol=1e-12, atol=1e-13)


def test_first_row_is_v0(oracle_lib):
    inp = small_inputs(T=16, H=3, K=8, pattern="tiny", seed=15)
    out, _, nk = oracle_lib.prefill(inp, rows=[0])
    assert nk[0] == 1
    y = oracle_lib.kv_norm(inp["c_kv"][0, :1], inp["gamma"].numpy())
    _, v = oracle_lib.up_proj(y, inp["wkv_b"])
    np.testing.assert_allclose(out[0], v[0], rtol=1e-13, atol=1e-14)


def test_order_and_duplicates_are_bit_invariant(oracle_lib):
    inp = small_inputs(T=64, H=2, K=32, pattern="uniform", seed=16)
    out, lse, nk = oracle_lib.prefill(inp)
    rng = np.random.default_rng(0)
    topk = inp["topk_idx"].numpy().copy()
    for t in range(64):
        row = topk[0, t]
        row[rng.integers(1, 32, size=5)] = row[rng.integers(0, 32, size=5)]   # some duplicates
        rng.shuffle(row)
    inp2 = dict(inp, topk_idx=torch.from_numpy(topk))
    out2, lse2, nk2 = oracle_lib.prefill(inp2)
    changed = nk2 != nk   # rows whose set lost members to the duplicates are not comparable
    keep = ~changed
    assert keep.sum() > 0
    assert np.array_equal(out[keep], out2[keep]) and np.array_equal(lse[keep], lse2[keep])
    # pure permutation: every row bit-identical
    topk3 = inp["topk_idx"].numpy().copy()
    for t in range(64):
        rng.shuffle(topk3[0, t])
    out3, lse3, nk3 = oracle_lib.prefill(dict(inp, topk_idx=torch.from_numpy(topk3)))
    assert np.array_equal(out, out3) and np.array_equal(lse, lse3) and np.array_equal(nk, nk3)
    # appended duplicates of existing entries: every row bit-identical
    topk4 = np.concatenate([inp["topk_idx"].numpy(), inp["topk_idx"].numpy()[..., :7]], axis=-1)
    out4, lse4, nk4 = oracle_lib.prefill(dict(inp, topk_idx=torch.from_numpy(topk4)))
    assert np.array_equal(out, out4) and np.array_equal(lse, lse4) and np.array_equal(nk, nk4)


def test_head_permutation_equivariance(oracle_lib):
    inp = small_inputs(T=32, H=4, K=16, pattern="uniform", seed=17)
    out, lse, _ = oracle_lib.prefill(inp)
    perm = [2, 0, 3, 1]
    W = inp["wkv_b"].reshape(4, 256, 512)[perm].reshape(1024, 512)
    inp2 = dict(inp, q=inp["q"][:, :, perm].contiguous(), wkv_b=W.contiguous())
    out2, lse2, _ = oracle_lib.prefill(inp2)
    assert np.array_equal(out[:, perm], out2) and np.array_equal(lse[:, perm], lse2)


def test_empty_selection_row(oracle_lib):
    """A row whose indices are all non-causal or negative: n = 0, out = 0, lse = -inf."""
    inp = small_inputs(T=16, H=2, K=6, pattern="tiny", seed=18)
    topk = inp["topk_idx"].numpy().copy()
    topk[0, 5] = [9, 10, -1, 15, 11, 6]
    out, lse, nk = oracle_lib.prefill(dict(inp, topk_idx=torch.from_numpy(topk)), rows=[5, 6])
    assert nk.tolist()[0] == 0 and nk[1] > 0
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_row_and_head_subsets_match_full_run(oracle_lib):
    inp = small_inputs(B=2, T=40, H=4, K=16, pattern="uniform", seed=19)
    out, lse, nk = oracle_lib.prefill(inp)
    rows = [79, 3, 40, 0, 55]
    o2, l2, n2 = oracle_lib.prefill(inp, rows=rows, heads=(1, 3))
    assert np.array_equal(o2, out[rows][:, 1:3]) and np.array_equal(l2, lse[rows][:, 1:3])
    assert np.array_equal(n2, nk[rows])


def test_multibatch_matches_literal(oracle_lib):
    inp = small_inputs(B=2, T=24, H=2, K=12, pattern="uniform", seed=20)
    out, lse, _ = oracle_lib.prefill(inp)
    ref_out, ref_lse = literal_prefill(inp)
    np.testing.assert_allclose(out.reshape(ref_out.shape), ref_out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(ref_lse.shape), ref_lse, rtol=1e-11, atol=1e-12)


def test_threads_do_not_change_bits(oracle_lib):
    inp = small_inputs(T=64, H=4, K=32, pattern="uniform", seed=21)
    a = oracle_lib.prefill(inp, threads=1)
    b = oracle_lib.prefill(inp, threads=5)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_kv_norm_agrees_with_torch_running_the_excerpt(oracle_lib):
    # torch's own fp32 execution of the RMSNorm excerpt ("Key-value RMSNorm" page, model.py
    # 281-293: x.float(), x.pow(2).mean(-1, keepdim=True), x * torch.rsqrt(var + eps), weight * x,
    # .to(dtype)) sums the squares in its own order and uses its own rsqrt: the oracle's fixed
    # order (ascending features, 1 / sqrt) is one fp32 reading of the same step. The bf16 outputs
    # may differ only where an fp32 result lies next to a bf16 rounding boundary: by one bf16 unit,
    # on a small fraction of the elements.
    inp = small_inputs(B=1, T=2048, H=1, K=4, stress=True, seed=41)
    x = inp["c_kv"].reshape(-1, 512)
    gamma = inp["gamma"]
    ref = oracle_lib.kv_norm(x, gamma.numpy())
    xf = x.float()
    var = xf.pow(2).mean(-1, keepdim=True)
    yt = (gamma * (xf * torch.rsqrt(var + 1e-6))).to(torch.bfloat16).to(torch.float64).numpy()
    diff = np.abs(yt - ref)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    assert (diff <= ulp * 1.0001).all()
    assert (diff > 0).mean() < 0.01
