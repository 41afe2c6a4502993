"""The C-ABI library loads and exports every declared entry point; host-side argument checks
(CPU only: no call here reaches the device)."""

import ctypes
import json
import math
import os
import re

import numpy as np

import pytest

import sparse_latent_attention_norm_b300 as mla
from sparse_latent_attention_norm_b300 import build as mla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    mla_build.build()
    return mla.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    return re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text)


def test_every_declared_symbol_is_exported(L):
    declared = header_functions()
    assert len(declared) >= 10
    assert sorted(declared) == sorted(mla.SYMBOLS)
    for name in declared:
        assert hasattr(L, name), name


def test_no_oracle_symbols_in_library(L):
    for name in ["oracle_prefill", "oracle_kv_norm", "oracle_up_proj"]:
        with pytest.raises(AttributeError):
            getattr(L, name)


def test_status_strings(L):
    for code, name in mla.STATUS_NAMES.items():
        assert mla.status_string(code).startswith(name)


def test_softmax_scale_matches_printed_m_squared(L):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "constants.json")))
    assert round(mla.softmax_scale() * math.sqrt(192), 3) == g["m_squared_printed"]["value"]


def test_workspace_size():
    for B, T, H, K in [(1, 64, 4, 32), (1, 4096, 128, 2048), (2, 16384, 128, 2048), (3, 333, 5, 7)]:
        kv = B * H * T * 256 * 2
        klo = B * H * T * 128
        bits = B * T * ((T + 127) // 128 * 4) * 4
        up = lambda x: (x + 1023) // 1024 * 1024
        sched = 1024   # the attention stage's tile counter
        assert mla.workspace_size(B, T, H, K) == up(kv) + up(klo) + up(bits) + sched
    assert mla.workspace_size(0, 64, 4, 32) == 0
    assert mla.workspace_size(1, 64, 129, 32) == 0
    assert mla.workspace_size(1, 65537, 4, 32) == 0


def _call_prefill(L, ptrs, dims, ws=None, ws_bytes=0, nk=None, flags=0):
    P = ctypes.c_void_p
    return L.mla_sparse_prefill_ex(*[P(p) if p else None for p in ptrs], dims, P(ws) if ws else None, ws_bytes,
                                   None, P(nk) if nk else None, flags)


def test_argument_errors_return_before_any_device_work(L):
    good = [0x100000 * (i + 1) for i in range(8)]    # never dereferenced: every call below fails early
    d = mla.Dims(1, 64, 4, 32)
    for i in range(8):
        ptrs = list(good)
        ptrs[i] = 0
        assert _call_prefill(L, ptrs, d) == 1                       # null pointer
        ptrs = list(good)
        ptrs[i] += 8
        if i != 7:                                                   # lse needs only 4-byte alignment
            assert _call_prefill(L, ptrs, d) == 1                   # misaligned
    assert _call_prefill(L, good, mla.Dims(0, 64, 4, 32)) == 1
    assert _call_prefill(L, good, mla.Dims(1, 0, 4, 32)) == 1
    assert _call_prefill(L, good, mla.Dims(1, 64, 4, 0)) == 1
    assert _call_prefill(L, good, mla.Dims(1, 64, 129, 32)) == 2
    assert _call_prefill(L, good, mla.Dims(1, 65537, 4, 32)) == 2
    assert _call_prefill(L, good, mla.Dims(1 << 20, 65536, 128, 1 << 20)) == 2
    assert _call_prefill(L, good, d, flags=2) == 1                  # unknown flag
    need = mla.workspace_size(1, 64, 4, 32)
    assert _call_prefill(L, good, d, ws=0x200000 + 512, ws_bytes=need) == 6   # misaligned workspace
    assert _call_prefill(L, good, d, ws=0x200000, ws_bytes=need - 1) == 6    # too small
    P = ctypes.c_void_p
    assert L.mla_canon_select(None, d, P(good[0]), None, 0, None) == 1
    assert L.mla_kvnorm_wkvb(P(good[0]), None, P(good[1]), d, P(good[2]), P(good[3]), None) == 1
    assert L.mla_kvnorm_wkvb(P(good[0]), P(good[1]), P(good[2]), d, P(good[3]), None, None) == 1
    assert L.mla_sparse_attention(P(good[0]), P(good[1]), P(good[2]), P(good[3]), P(good[4]), P(good[5]), None, d,
                                  None) == 1
    assert L.mla_selftest_wait_timeout(None, None) == 1             # null result
    assert L.mla_selftest_wait_timeout(P(good[0] + 2), None) == 1    # misaligned result


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    x = torch.zeros(1, 64, 4, 192, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        mla.sparse_prefill(x, x, x, x, x, torch.zeros(1, 64, 32, dtype=torch.int32))


def test_q_and_out_need_32_byte_alignment(L):
    good = [0x100000 * (i + 1) for i in range(8)]
    d = mla.Dims(1, 64, 4, 32)
    for i in (0, 6):                                                  # q, out: 32-byte vector accesses
        ptrs = list(good)
        ptrs[i] += 16
        assert _call_prefill(L, ptrs, d) == 1


def test_options_workspace_sizes(L):
    up = lambda x: (x + 1023) // 1024 * 1024
    for B, T, H, K in [(1, 64, 4, 32), (2, 333, 5, 7), (1, 4096, 128, 2048)]:
        base = mla.workspace_size(B, T, H, K)
        assert mla.workspace_size_opt(B, T, H, K, None) == base
        assert mla.workspace_size_opt(B, T, H, K, mla.options()) == base
        assert mla.workspace_size_opt(B, T, H, K, mla.options(flags=mla.FLAG_FP8_LATENT)) == base
        rope = mla.workspace_size_opt(B, T, H, K, mla.options(flags=mla.FLAG_ROPE))
        assert rope == base + up(T * 32 * 8) + up(B * T * 64 * 2)
        scale = ctypes.c_float(1.0)   # any host address: the size query only tests it against NULL
        opt = mla.PrefillOptions(0, None, ctypes.addressof(scale), None, None, 0)
        assert mla.workspace_size_opt(B, T, H, K, opt) == base + up(H * 256 * 512 * 2)
    assert mla.workspace_size_opt(1, 64, 4, 32, mla.options(flags=8)) == 0          # unknown flag
    kv = 0x400000
    bad = mla.PrefillOptions(0, None, None, kv, None, 63)                          # cache shorter than T
    assert mla.workspace_size_opt(1, 64, 4, 32, bad) == 0


def test_option_argument_errors(L):
    P = ctypes.c_void_p
    good = [0x100000 * (i + 1) for i in range(8)]
    d = mla.Dims(1, 64, 4, 32)

    def call(opt):
        return L.mla_sparse_prefill_opt(*[P(p) for p in good], d, None, 0, None, ctypes.byref(opt))
    assert call(mla.PrefillOptions(16, None, None, None, None, 0)) == 1            # unknown flag
    assert call(mla.PrefillOptions(0, None, None, 0x400010, None, 64)) == 1         # kv_cache not 32-aligned
    assert call(mla.PrefillOptions(0, None, None, None, 0x400002, 64)) == 1         # pe_cache not 4-aligned
    assert call(mla.PrefillOptions(0, None, None, 0x400000, None, 10)) == 1         # cache_len < T
    assert call(mla.PrefillOptions(0, 0x400002, None, None, None, 0)) == 1          # n_keys misaligned
    assert L.mla_sparse_prefill_ex(*[P(p) for p in good], d, None, 0, None, None, mla.FLAG_ROPE) == 1   # _ex: validate only
    assert L.mla_dequant_wkvb_fp8(P(good[0]), P(good[1]), 100, P(good[2]), None) == 1  # rows not a multiple of 128
    assert L.mla_dequant_wkvb_fp8(None, P(good[1]), 256, P(good[2]), None) == 1
    assert L.mla_dequant_wkvb_fp8(P(good[0]), P(good[1]), 256, P(good[2] + 16), None) == 1
    assert L.mla_kvnorm_wkvb_opt(P(good[0]), P(good[1]), P(good[2]), d, P(good[3]), P(good[4]), 4, None, 0, None) == 1
    assert L.mla_kvnorm_wkvb_opt(P(good[0]), P(good[1]), P(good[2]), d, P(good[3]), P(good[4]), 2,
                                 P(good[5]), 10, None) == 1                          # cache_len < T
    assert L.mla_rope_k_pe(P(good[0]), d, P(good[1]), P(good[2] + 16), None, 0, None) == 1   # table misaligned
    assert L.mla_rope_k_pe(None, d, P(good[1]), P(good[2]), None, 0, None) == 1
    assert L.mla_sparse_attention_opt(*[P(p) for p in good[:7]], d, P(good[7] + 8), None) == 1


def test_host_yarn_frequencies_follow_the_rotation_counts(L):
    # the library's own YaRN frequencies (host, fp64): RoPE's theta^(-2i/64) for pairs that turn
    # more than 32 times over the 4096 original positions, divided by 40 below one turn
    f = mla.yarn_frequencies()
    base = 10000.0 ** (-2.0 * np.arange(32) / 64)
    turns = 4096 * base / (2 * math.pi)
    assert np.allclose(f[turns > 32], base[turns > 32], rtol=1e-15, atol=0)
    assert np.allclose(f[turns < 1], base[turns < 1] / 40, rtol=1e-15, atol=0)
