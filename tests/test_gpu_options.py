"""Parity of the optional steps of the path with the oracle, through the C ABI (GPU):

  * FP8 block-scaled wkv_b ("Key-value down-projection" page, Linear excerpt): the dequantised
    weight bit-exact, the prefill within the parity tolerances;
  * the KV cache's FP8 round trip of the normalised latent ("Keys" page, KV-cache excerpt): the
    latent written to kv_cache bit-exact, the prefill within tolerance;
  * YaRN RoPE of k_pe and q's rotary tail (apply_rotary_emb call site; ModelArgs): the rotated
    k_pe and pe_cache, the prefill within tolerance;
  * all of them at once, on small shapes and on the full-size headline workload.

Tolerances are in tests/parity.py.
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


def fp8_weight(H, seed):
    """An FP8 block-scaled wkv_b: e4m3 codes of N(0, 100^2) values (clipped to e4m3's +-448) and
    per-block scales U(0.9, 1.1) / (100 sqrt(512)), so that the effective weight has the
    N(0, 1/512) spread of the bf16 workloads (wider weights make |v|, and so |out|, larger; out's
    bound of 2e-2 is below bf16's rounding step once |out| passes 8)."""
    rng = np.random.default_rng(seed)
    rows = H * 256
    w = np.clip(rng.normal(0, 100.0, (rows, 512)), -448, 448).astype(np.float32)
    w8 = torch.from_numpy(w).to(torch.float8_e4m3fn).view(torch.uint8)
    scale = (rng.uniform(0.9, 1.1, (rows // 128, 4)) / (100.0 * np.sqrt(512))).astype(np.float32)
    return w8, torch.from_numpy(scale)


def run(mla, inp, **kw):
    d = to_dev(inp)
    extra = {}
    if "wkv_b_fp8" in inp:
        extra = dict(wkv_b_scale=d["wkv_b_scale"])
        wkv_b = d["wkv_b_fp8"]
    else:
        wkv_b = d["wkv_b"]
    out, lse, nk = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], wkv_b, d["topk_idx"], n_keys=True,
                                      **extra, **kw)
    torch.cuda.synchronize()
    assert mla.get_status() == 0
    return out, lse, nk


def compare(out, lse, nk, ref, B, T, H, what):
    ref_out, ref_lse, ref_n = ref
    assert np.array_equal(nk.cpu().numpy().reshape(-1), ref_n), f"{what}: n_keys differ"
    return parity.compare(out.float().cpu().numpy().reshape(B * T, H, 128), lse.cpu().numpy().reshape(B * T, H),
                          ref_out, ref_lse, what)


# ------------------------------------------------------------------------- FP8 block-scaled wkv_b
def test_fp8_weight_dequantisation_is_bit_exact(mla, oracle_lib):
    for H, seed in [(1, 1), (5, 2), (128, 3)]:
        w8, scale = fp8_weight(H, seed)
        w = mla.dequant_wkvb_fp8(w8.cuda(), scale.cuda())
        torch.cuda.synchronize()
        want = oracle_lib.fp8_weight(w8, scale)
        assert np.array_equal(w.double().cpu().numpy(), want), H


@pytest.mark.parametrize("T,H,K,pattern", [(333, 5, 48, "uniform"), (600, 3, 96, "clustered")])
def test_prefill_with_fp8_weight(mla, oracle_lib, T, H, K, pattern):
    w = mi.custom("fp8w", 1, T, H, K, pattern, recent=256, seed_id=400 + T)
    inp = mi.make_inputs(w)
    w8, scale = fp8_weight(H, 7 + T)
    inp8 = dict(inp, wkv_b_fp8=w8, wkv_b_scale=scale)
    out, lse, nk = run(mla, inp8)
    compare(out, lse, nk, oracle_lib.prefill(inp8), 1, T, H, "fp8 weight")
    # the same bits as the bf16 path fed the dequantised weight
    weff = mla.dequant_wkvb_fp8(w8.cuda(), scale.cuda()).cpu()
    out2, lse2, _ = run(mla, dict(inp, wkv_b=weff))
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


# ------------------------------------------------------------------ FP8 round trip of the latent
@pytest.mark.parametrize("fp8_latent", [False, True])
def test_kv_cache_holds_the_latent_bit_exact(mla, oracle_lib, fp8_latent):
    w = mi.custom("kvc", 2, 300, 3, 8, "uniform", stress=True, seed_id=410)
    inp = mi.make_inputs(w)
    d = to_dev(inp)
    L = 320
    cache = torch.full((2, L, 512), -7.0, dtype=torch.bfloat16, device="cuda")
    kv, klo = mla.kvnorm_wkvb(d["c_kv"], d["gamma"], d["wkv_b"], fp8_latent=fp8_latent, kv_cache=cache)
    torch.cuda.synchronize()
    assert mla.get_status() == 0
    y = oracle_lib.latent(inp["c_kv"], inp["gamma"], fp8_latent=fp8_latent)       # [2, 300, 512]
    got = cache.double().cpu().numpy()
    assert np.array_equal(got[:, :300], y)
    assert (got[:, 300:] == -7.0).all()                                           # positions >= T untouched
    # k_nope / v from that latent, as in the GEMM-stage test
    kn = mla.k_nope_from(kv, klo).double().cpu().numpy()
    rkn, rv = oracle_lib.up_proj(y.reshape(-1, 512), inp["wkv_b"])
    rkn = rkn.reshape(2, 300, 3, 128).transpose(0, 2, 1, 3)
    rv = rv.reshape(2, 300, 3, 128).transpose(0, 2, 1, 3)
    assert np.abs(kn - rkn).max() <= 2e-4 * max(1.0, np.abs(rkn).max())
    assert (np.abs(kv[..., 128:].double().cpu().numpy() - rv) - 2.0 ** -11 * np.abs(rv)).max() <= 1e-5


@pytest.mark.parametrize("T,H,K,stress", [(333, 5, 48, False), (520, 4, 64, True)])
def test_prefill_with_fp8_latent(mla, oracle_lib, T, H, K, stress):
    w = mi.custom("fp8lat", 1, T, H, K, "uniform", stress=stress, seed_id=420 + T)
    inp = mi.make_inputs(w)
    out, lse, nk = run(mla, inp, fp8_latent=True)
    compare(out, lse, nk, oracle_lib.prefill(inp, fp8_latent=True), 1, T, H, "fp8 latent")


# ------------------------------------------------------------------------------------ YaRN RoPE
def test_yarn_frequencies_match_the_oracle(mla, oracle_lib):
    np.testing.assert_allclose(mla.yarn_frequencies(), oracle_lib.yarn_inv_freq(), rtol=1e-15, atol=0)


def test_rotated_k_pe_and_table(mla, oracle_lib):
    B, T = 2, 16384          # every position of the model's context
    k_pe = torch.from_numpy(np.random.default_rng(11).normal(0, 1, (B, T, 64)).astype(np.float32)).to(torch.bfloat16)
    L = T + 8
    pe_cache = torch.zeros((B, L, 64), dtype=torch.bfloat16, device="cuda")
    rot, cs = mla.rope_k_pe(k_pe.cuda(), pe_cache=pe_cache)
    torch.cuda.synchronize()
    assert mla.get_status() == 0
    want = oracle_lib.rope(k_pe.reshape(-1, 64), np.tile(np.arange(T, dtype=np.int32), B)).reshape(B, T, 64)
    got = rot.double().cpu().numpy()
    # the rotation's only rounding-sensitive inputs are fp32 cos / sin of the fp64 angle: they may
    # differ from the oracle's in the last place on rare positions, which moves a bf16 result by at
    # most one unit where its exact value lies next to a rounding boundary
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(want), 1e-30))) - 7)
    assert (np.abs(got - want) <= ulp).all()
    assert (got == want).mean() >= 0.9999
    assert torch.equal(pe_cache[:, :T], rot) and (pe_cache[:, T:] == 0).all()
    f = oracle_lib.yarn_inv_freq()
    ang = np.arange(T)[:, None] * f[None, :]
    table = cs.cpu().numpy()
    assert (table[..., 0] == np.cos(ang).astype(np.float32)).mean() >= 0.9999
    assert (table[..., 1] == np.sin(ang).astype(np.float32)).mean() >= 0.9999
    assert np.abs(table[..., 0] - np.cos(ang)).max() <= 2.0 ** -24 and np.abs(table[..., 1] - np.sin(ang)).max() <= 2.0 ** -24


@pytest.mark.parametrize("T,H,K,pattern", [(333, 5, 48, "uniform"), (4200, 2, 256, "clustered")])
def test_prefill_with_rope(mla, oracle_lib, T, H, K, pattern):
    w = mi.custom("rope", 1, T, H, K, pattern, recent=1024, seed_id=430 + T)
    inp = mi.make_inputs(w)
    pe_cache = torch.zeros((1, T, 64), dtype=torch.bfloat16, device="cuda")
    out, lse, nk = run(mla, inp, rope=True, pe_cache=pe_cache)
    compare(out, lse, nk, oracle_lib.prefill(inp, rope=True), 1, T, H, "rope")
    rot, _ = mla.rope_k_pe(inp["k_pe"].cuda())
    assert torch.equal(pe_cache, rot)
    # the staged form: rotated k_pe and the table into the attention stage
    d = to_dev(inp)
    bits, _ = mla.canon_select(d["topk_idx"], T)
    kv, klo = mla.kvnorm_wkvb(d["c_kv"], d["gamma"], d["wkv_b"])
    rot, cs = mla.rope_k_pe(d["k_pe"])
    out2, lse2 = mla.sparse_attention(d["q"], rot, kv, klo, bits, rope_cs=cs)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


# ----------------------------------------------------------------------------------- all at once
def all_options_inputs(w, seed):
    inp = mi.make_inputs(w)
    w8, scale = fp8_weight(w.H, seed)
    return dict(inp, wkv_b_fp8=w8, wkv_b_scale=scale)


def test_prefill_with_every_option_small(mla, oracle_lib):
    w = mi.custom("allopt", 2, 333, 5, 48, "uniform", stress=True, seed_id=440)
    inp = all_options_inputs(w, 441)
    L = 400
    kv_cache = torch.zeros((2, L, 512), dtype=torch.bfloat16, device="cuda")
    pe_cache = torch.zeros((2, L, 64), dtype=torch.bfloat16, device="cuda")
    out, lse, nk = run(mla, inp, fp8_latent=True, rope=True, kv_cache=kv_cache, pe_cache=pe_cache)
    compare(out, lse, nk, oracle_lib.prefill(inp, rope=True, fp8_latent=True), 2, 333, 5, "all options")
    y = oracle_lib.latent(inp["c_kv"], inp["gamma"], fp8_latent=True)
    assert np.array_equal(kv_cache[:, :333].double().cpu().numpy(), y)


def test_prefill_with_every_option_headline(mla, oracle_lib):
    # the full-size headline workload with the model's own steps switched on, every element
    w = mi.WORKLOADS["headline"]
    inp = all_options_inputs(w, 442)
    out, lse, nk = run(mla, inp, fp8_latent=True, rope=True)
    og = out.view(w.T, w.H, 128)
    lg = lse.view(w.T, w.H).cpu().numpy()
    nkh = nk.cpu().numpy().reshape(-1)
    for h0 in range(0, w.H, 64):
        ref_out, ref_lse, ref_n = oracle_lib.prefill(inp, heads=(h0, h0 + 64), rope=True, fp8_latent=True)
        if h0 == 0:
            assert np.array_equal(nkh, ref_n)
        parity.compare(og[:, h0:h0 + 64].float().cpu().numpy(), lg[:, h0:h0 + 64], ref_out, ref_lse,
                       f"headline all options heads {h0}..")
