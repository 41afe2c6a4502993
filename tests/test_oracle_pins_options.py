"""Pins of the oracle's optional steps (CPU only): the FP8 e4m3 format, the FP8 round trip of the
latent (KV-cache excerpt, "Keys" page), the FP8 block-scaled wkv_b (Linear excerpt, "Key-value
down-projection" page) and YaRN RoPE (ModelArgs on the "Keys" page; apply_rotary_emb call site on
the "Key-value down-projection" page).

Each test checks the oracle against something other than its own code: torch's float8 type (a
library routine), closed forms and invariants of the formats, YaRN's defining rotation counts,
and the oracle's main path fed with inputs prepared another way.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import mla_inputs as mi

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "constants.json")))


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


# ------------------------------------------------------------------------------------ e4m3 format
def test_e4m3_code_values_match_torch_float8(oracle_lib):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle_lib.e4m3_values()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.nanmax(got) == 448.0 and got[1] == 2.0 ** -9   # largest finite, smallest subnormal


def test_e4m3_rounding_matches_torch_cast(oracle_lib):
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.normal(0, 50, 20000), rng.uniform(-448, 448, 20000), rng.normal(0, 0.01, 20000),
                        np.array([0.0, 448.0, -448.0, 2.0 ** -10, 2.0 ** -9 * 1.5, 17.0, 18.0, 19.0])])
    x = x.astype(np.float32).astype(np.float64)          # fp32 values, as the kernels round them
    want = torch.from_numpy(x).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle_lib.round_to_e4m3(x), want)


def test_e4m3_grid_values_round_trip_and_saturate(oracle_lib):
    v = oracle_lib.e4m3_values()
    v = v[~np.isnan(v)]
    assert np.array_equal(oracle_lib.round_to_e4m3(v), v)
    assert np.array_equal(oracle_lib.round_to_e4m3(np.array([449.0, 1e6, -500.0])), np.array([448.0, 448.0, -448.0]))


# -------------------------------------------------------------------- FP8 round trip of the latent
def latent_inputs(N=64, seed=3, outliers=False):
    w = mi.custom("pin_lat", 1, N, 1, 4, "tiny", seed_id=seed, stress=outliers)
    inp = mi.make_inputs(w)
    return inp["c_kv"].reshape(N, 512), inp["gamma"]


@pytest.mark.parametrize("outliers", [False, True])
def test_fp8_latent_keeps_each_block_max_and_bounds_the_error(oracle_lib, outliers):
    c_kv, gamma = latent_inputs(outliers=outliers)
    y = oracle_lib.latent(c_kv, gamma)
    y8 = oracle_lib.latent(c_kv, gamma, fp8_latent=True)
    B = GOLDEN["fp8_block_size"]["value"]
    for r in range(y.shape[0]):
        for b0 in range(0, 512, B):
            blk, blk8 = y[r, b0:b0 + B], y8[r, b0:b0 + B]
            amax = np.abs(blk).max()
            i = np.argmax(np.abs(blk))
            assert blk8[i] == blk[i]                       # the block max maps to +-448 * scale exactly
            scale = amax / 448.0
            # e4m3 keeps 4 significant bits (relative 2^-4 at most), subnormals step 2^-9 * scale;
            # the bf16 cast adds at most 2^-9 relative
            err = np.abs(blk8 - blk)
            bound = np.maximum(np.abs(blk) * (2.0 ** -4 + 2.0 ** -8), 2.0 ** -10 * scale * 1.01)
            assert (err <= bound).all()


def test_fp8_latent_blocks_are_independent_and_zero_stays_zero(oracle_lib):
    c_kv, gamma = latent_inputs(N=8)
    y8 = oracle_lib.latent(c_kv, gamma, fp8_latent=True)
    # a gain of zero on block 2 zeroes that block of y; the other blocks' round trip is unchanged
    g2 = gamma.clone()
    g2[256:384] = 0.0
    y8b = oracle_lib.latent(c_kv, g2, fp8_latent=True)
    assert (y8b[:, 256:384] == 0.0).all()
    keep = np.r_[0:256, 384:512]
    assert np.array_equal(y8b[:, keep], y8[:, keep])


def test_fp8_latent_of_grid_values_is_the_identity(oracle_lib):
    # rows whose kv_norm output already lies on the e4m3 grid of its block scale come back unchanged:
    # with unit gain and a row of +-1 and +-0.5 entries the RMS is fixed and every value is a power
    # of two times an e4m3 value, block max included
    x = np.where(np.arange(512) % 3 == 0, 1.0, 0.5) * np.where(np.arange(512) % 2 == 0, 1.0, -1.0)
    c_kv = bf16(x[None, :])
    gamma = torch.ones(512)
    y = oracle_lib.latent(c_kv, gamma)
    y8 = oracle_lib.latent(c_kv, gamma, fp8_latent=True)
    assert np.array_equal(y, y8)


# --------------------------------------------------------------------- FP8 block-scaled wkv_b
def fp8_weight_inputs(H=2, seed=9):
    rng = np.random.default_rng(seed)
    rows = H * 256
    w = rng.normal(0, 1, (rows, 512)).astype(np.float32)
    W8 = torch.from_numpy(w).to(torch.float8_e4m3fn).view(torch.uint8)
    scale = (rng.uniform(0.5, 2.0, ((rows + 127) // 128, 4)) / 448).astype(np.float32)
    return W8, torch.from_numpy(scale)


def test_fp8_weight_unit_scale_is_the_e4m3_value(oracle_lib):
    W8, scale = fp8_weight_inputs()
    one = torch.ones_like(scale)
    w = oracle_lib.fp8_weight(W8, one)
    assert np.array_equal(w, W8.view(torch.float8_e4m3fn).to(torch.float64).numpy())


def test_fp8_weight_scale_applies_per_128_block(oracle_lib):
    W8, scale = fp8_weight_inputs()
    one = torch.ones_like(scale)
    base = W8.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    # a power-of-two scale on one block scales exactly that 128 x 128 block
    s = one.clone()
    s[2, 1] = 0.25
    w = oracle_lib.fp8_weight(W8, s)
    want = base.copy()
    want[256:384, 128:256] *= 0.25
    assert np.array_equal(w, want)
    # a general scale: the fp32 product rounded to bf16 (torch's casts as the library routine)
    w = oracle_lib.fp8_weight(W8, scale)
    full = scale.repeat_interleave(128, 0).repeat_interleave(128, 1)[:W8.shape[0], :512]
    want = (W8.view(torch.float8_e4m3fn).to(torch.float32) * full).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(w, want)


# ---------------------------------------------------------------------------------- YaRN RoPE
def test_yarn_frequencies_follow_the_rotation_counts(oracle_lib):
    # YaRN's definition: a pair that turns more than beta_fast times over the original context keeps
    # RoPE's frequency theta^(-2i/d); one turning fewer than beta_slow times is divided by the
    # factor; in between the frequency lies strictly between the two, falling with i
    theta = GOLDEN["rope_theta"]["value"]
    d = GOLDEN["qk_rope_head_dim"]["value"]
    L = GOLDEN["original_seq_len"]["value"]
    factor = GOLDEN["rope_factor"]["value"]
    fast, slow = GOLDEN["beta_fast"]["value"], GOLDEN["beta_slow"]["value"]
    f = oracle_lib.yarn_inv_freq()
    assert f.shape == (d // 2,)
    base = theta ** (-2.0 * np.arange(d // 2) / d)
    turns = L * base / (2 * math.pi)
    kept, divided = turns > fast, turns < slow
    assert kept.sum() >= 10 and divided.sum() >= 8
    # the pair just below the fast boundary rounds outward (the lower dim is floored): kept too
    assert np.allclose(f[kept], base[kept], rtol=1e-15, atol=0)
    assert np.allclose(f[divided], base[divided] / factor, rtol=1e-15, atol=0)
    mid = ~(kept | divided)
    assert mid.sum() >= 10 and (f[mid] < base[mid]).all() and (f[mid] > base[mid] / factor).all()
    assert (np.diff(f) < 0).all()


def test_rope_position_zero_is_the_identity(oracle_lib):
    x = bf16(np.random.default_rng(1).normal(0, 1, (16, 64)))
    y = oracle_lib.rope(x, np.zeros(16, dtype=np.int32))
    assert np.array_equal(y, x.to(torch.float64).numpy())


def test_rope_is_a_rotation_of_adjacent_pairs(oracle_lib):
    # against numpy's complex exponential at the oracle's frequencies: (x_2i + i x_2i+1) e^{i t f_i},
    # within the fp32 product and bf16 cast; pair norms are kept
    rng = np.random.default_rng(2)
    x = bf16(rng.normal(0, 1, (64, 64)))
    pos = rng.integers(0, 16384, 64).astype(np.int32)
    y = oracle_lib.rope(x, pos)
    xf = x.to(torch.float64).numpy()
    f = oracle_lib.yarn_inv_freq()
    z = (xf[:, 0::2] + 1j * xf[:, 1::2]) * np.exp(1j * pos[:, None] * f[None, :])
    want = np.stack([z.real, z.imag], axis=-1).reshape(64, 64)
    assert np.abs(y - want).max() <= 2.0 ** -8 * np.abs(want).max()
    ny = np.hypot(y[:, 0::2], y[:, 1::2])
    nx = np.hypot(xf[:, 0::2], xf[:, 1::2])
    assert np.abs(ny - nx).max() <= 2.0 ** -7 * nx.max()


def test_rope_inner_products_depend_on_relative_position(oracle_lib):
    rng = np.random.default_rng(4)
    q = bf16(rng.normal(0, 1, (1, 64)))
    k = bf16(rng.normal(0, 1, (1, 64)))
    dots = []
    for t, s in [(700, 100), (1600, 1000), (9600, 9000)]:
        dots.append(float((oracle_lib.rope(q, np.array([t], np.int32)) @ oracle_lib.rope(k, np.array([s], np.int32)).T)[0, 0]))
    assert max(dots) - min(dots) <= 0.05 * max(1.0, abs(dots[0]))


# --------------------------------------------------------------- the options wired into the path
def test_prefill_rope_equals_prefill_on_prerotated_inputs(oracle_lib):
    w = mi.custom("pin_rope", 1, 80, 2, 24, "tiny", seed_id=31)
    inp = mi.make_inputs(w)
    out, lse, _ = oracle_lib.prefill(inp, rope=True)
    T = w.T
    q = inp["q"].clone()
    qpe = q[..., 128:].reshape(-1, 64)
    pos_q = np.repeat(np.arange(T, dtype=np.int32), w.H)
    q[..., 128:] = bf16(oracle_lib.rope(qpe, pos_q)).reshape(1, T, w.H, 64)
    k_pe = bf16(oracle_lib.rope(inp["k_pe"].reshape(-1, 64), np.arange(T, dtype=np.int32))).reshape(1, T, 64)
    out2, lse2, _ = oracle_lib.prefill(dict(inp, q=q, k_pe=k_pe))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    out3, _, _ = oracle_lib.prefill(inp)
    assert not np.array_equal(out, out3)


def test_prefill_fp8_weight_equals_prefill_on_its_bf16_weight(oracle_lib):
    w = mi.custom("pin_w8", 1, 60, 2, 20, "tiny", seed_id=32)
    inp = mi.make_inputs(w)
    W8, scale = fp8_weight_inputs(H=2, seed=33)
    Weff = bf16(oracle_lib.fp8_weight(W8, scale))
    out, lse, _ = oracle_lib.prefill(dict(inp, wkv_b_fp8=W8, wkv_b_scale=scale))
    out2, lse2, _ = oracle_lib.prefill(dict(inp, wkv_b=Weff))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_prefill_fp8_latent_attends_over_the_round_tripped_latent(oracle_lib):
    # a textbook attention (numpy) over k_nope / v up-projected from the oracle's round-tripped
    # latent equals the oracle's prefill with the FP8 round trip, and differs from the one without
    w = mi.custom("pin_lat8", 1, 40, 2, 40, "dense", seed_id=34)
    inp = mi.make_inputs(w)
    out, lse, _ = oracle_lib.prefill(inp, fp8_latent=True)
    y8 = oracle_lib.latent(inp["c_kv"].reshape(-1, 512), inp["gamma"], fp8_latent=True)
    W = inp["wkv_b"].to(torch.float64).numpy().reshape(w.H, 256, 512)
    q = inp["q"].to(torch.float64).numpy()[0]
    kpe = inp["k_pe"].to(torch.float64).numpy()[0]
    scale = oracle_lib.softmax_scale()
    for h in range(w.H):
        kv = y8 @ W[h].T
        k = np.concatenate([kv[:, :128], kpe], axis=1)
        s = (q[:, h] @ k.T) * scale
        s[np.triu_indices(w.T, 1)] = -np.inf
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        o = (p @ kv[:, 128:]) / p.sum(axis=1, keepdims=True)
        assert np.allclose(out[:, h], o, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse[:, h], m[:, 0] + np.log(p.sum(axis=1)), rtol=1e-12, atol=1e-12)
    out0, _, _ = oracle_lib.prefill(inp)
    assert not np.array_equal(out, out0)


# ------------------------------------------------------- rounding emulation (diagnostic mode)
def test_emulation_with_zero_queries_is_the_rounded_mean(oracle_lib):
    # q = 0 makes every score 0 exactly: the pages' bf16 softmax gives every selected key the bf16
    # value of 1/n, out is bf16(bf16(1/n) * sum of the bf16-rounded v), lse = ln n
    w = mi.custom("pin_emul", 1, 40, 2, 40, "dense", seed_id=35)
    inp = mi.make_inputs(w)
    inp["q"] = torch.zeros_like(inp["q"])
    out, lse, nk = oracle_lib.prefill(inp, emulate_bf16=True)
    y = oracle_lib.kv_norm(inp["c_kv"].reshape(-1, 512), inp["gamma"].numpy())
    _, v = oracle_lib.up_proj(y, inp["wkv_b"])                      # [T, H, 128], exact
    vb = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    for t in range(w.T):
        n = t + 1
        p = float(torch.tensor(1.0 / n, dtype=torch.float64).to(torch.bfloat16).to(torch.float64))
        want = torch.from_numpy(p * vb[:n].sum(axis=0)).to(torch.bfloat16).to(torch.float64).numpy()
        assert np.array_equal(out[t], want)
        assert np.allclose(lse[t], math.log(n), rtol=0, atol=1e-12)


def test_emulation_outputs_are_bf16_and_near_the_exact_result(oracle_lib):
    w = mi.custom("pin_emul2", 1, 200, 3, 48, "uniform", seed_id=36)
    inp = mi.make_inputs(w)
    out, lse, _ = oracle_lib.prefill(inp)
    oe, le, _ = oracle_lib.prefill(inp, emulate_bf16=True)
    assert np.array_equal(oracle_lib.round_to_bf16(oe), oe)
    assert not np.array_equal(oe, out)
    # bf16 keeps 8 significant bits: each rounding moves a value by at most 2^-9 of itself
    assert np.abs(oe - out).max() <= 0.1 * max(1.0, np.abs(out).max())
    assert np.abs(le - lse).max() <= 2.0 ** -6 * max(1.0, np.abs(lse).max())
