"""The C-ABI library loads and exports every declared entry point; host-side argument checks
(CPU only: no call here reaches the device)."""

import ctypes
import json
import math
import os
import re

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
