"""fp64 CPU oracle of the DeepSeek-V3.2-Exp sparse latent attention (MLA) prefill.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this package. It never imports the CUDA library and the CUDA library
never calls it. The arithmetic lives in ``mla_oracle.cpp`` (plain C++, fp64); this module only
compiles it, loads it with ctypes and marshals numpy arrays.

Every function follows the model atlas pages' DeepSeek-V3.2-Exp ``inference/model.py`` excerpts:
RMSNorm (model.py 281-293), MLA ``__init__`` (523-539), the MHA prefill branch (574-589) and
the "Scale scores" page. See ``mla_oracle.cpp`` for the per-step citations and readings.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "libmla_oracle.so")
_lib = None

LATENT, NOPE, ROPE, QK, V = 512, 128, 64, 192, 128


def build(force: bool = False) -> str:
    """Compile mla_oracle.cpp into libmla_oracle.so next to it (g++, -O3, pthreads)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["g++", "-O3", "-march=x86-64-v3", "-ffp-contract=off", "-std=c++17", "-shared", "-fPIC", "-pthread",
               _SRC, "-o", _LIB_PATH + ".tmp"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        lib.oracle_softmax_scale.restype = ctypes.c_double
        lib.oracle_softmax_scale.argtypes = []
        lib.oracle_kv_norm.restype = None
        lib.oracle_kv_norm.argtypes = [P, P, ctypes.c_int64, P]
        lib.oracle_kv_norm_precast.restype = None
        lib.oracle_kv_norm_precast.argtypes = [P, P, ctypes.c_int64, P]
        lib.oracle_round_to_bf16.restype = None
        lib.oracle_round_to_bf16.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_up_proj.restype = None
        lib.oracle_up_proj.argtypes = [P, P, ctypes.c_int, ctypes.c_int64, P, P]
        lib.oracle_canon_row.restype = ctypes.c_int
        lib.oracle_canon_row.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
        lib.oracle_prefill.restype = ctypes.c_int
        lib.oracle_prefill.argtypes = [ctypes.c_int] * 4 + [P] * 6 + [ctypes.c_int64, P, ctypes.c_int,
                                                                   ctypes.c_int, P, P, P, ctypes.c_int]
        lib.oracle_prefill_opt.restype = ctypes.c_int
        lib.oracle_prefill_opt.argtypes = [ctypes.c_int] * 4 + [P] * 8 + [ctypes.c_int64, P] + [ctypes.c_int] * 3 + \
            [P, P, P, ctypes.c_int]
        lib.oracle_latent.restype = None
        lib.oracle_latent.argtypes = [P, P, ctypes.c_int64, ctypes.c_int, P]
        lib.oracle_round_to_e4m3.restype = None
        lib.oracle_round_to_e4m3.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_e4m3_values.restype = None
        lib.oracle_e4m3_values.argtypes = [P]
        lib.oracle_fp8_weight.restype = None
        lib.oracle_fp8_weight.argtypes = [P, P, ctypes.c_int, P]
        lib.oracle_yarn_inv_freq.restype = None
        lib.oracle_yarn_inv_freq.argtypes = [P]
        lib.oracle_rope.restype = None
        lib.oracle_rope.argtypes = [P, P, ctypes.c_int64, P]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(a) -> np.ndarray:
    """bf16 tensor (torch) or uint16 bit array -> contiguous uint16 numpy array of bit patterns."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch  # plumbing only: read the bf16 bit patterns of a CPU tensor
    assert a.dtype == torch.bfloat16
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def softmax_scale() -> float:
    """MLA ``__init__``: 192 ** -0.5 * mscale**2, mscale = 0.1 * 1 * ln 40 + 1."""
    return _load().oracle_softmax_scale()


def kv_norm(x, gamma, precast: bool = False) -> np.ndarray:
    """RMSNorm(512), eps 1e-6, on bf16 rows ``x`` [..., 512] with fp32 ``gamma`` [512].

    Returns the bf16 output values as fp64 (the excerpt's final ``.to(dtype)``), or with
    ``precast=True`` the fp32 values before that cast (the excerpt computes the norm in fp32)."""
    xb = _bits(x)
    shape = xb.shape
    assert shape[-1] == LATENT
    g = np.ascontiguousarray(np.asarray(gamma, dtype=np.float32))
    n = int(np.prod(shape[:-1]))
    y = np.empty((n, LATENT), dtype=np.float64)
    fn = _load().oracle_kv_norm_precast if precast else _load().oracle_kv_norm
    fn(_ptr(xb), _ptr(g), n, _ptr(y))
    return y.reshape(shape)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """The oracle's round-to-nearest-even bf16 rounding, elementwise (fp64 in, fp64 out)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_round_to_bf16(_ptr(x), x.size, _ptr(y))
    return y


def up_proj(y: np.ndarray, W) -> tuple[np.ndarray, np.ndarray]:
    """wkv_b on fp64 rows ``y`` [N, 512] with bf16 ``W`` [H*256, 512] -> (k_nope, v) [N, H, 128]."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    wb = _bits(W)
    H = wb.shape[0] // (NOPE + V)
    assert wb.shape == (H * (NOPE + V), LATENT)
    n = y.shape[0]
    kn = np.empty((n, H, NOPE), dtype=np.float64)
    vv = np.empty((n, H, V), dtype=np.float64)
    _load().oracle_up_proj(_ptr(y), _ptr(wb), H, n, _ptr(kn), _ptr(vv))
    return kn, vv


def canon_row(idx: np.ndarray, t: int) -> np.ndarray:
    """Selected key set of query ``t``: distinct entries of ``idx`` in [0, t], ascending."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    sel = np.empty(max(idx.size, 1), dtype=np.int32)
    n = _load().oracle_canon_row(_ptr(idx), idx.size, int(t), _ptr(sel))
    return sel[:n].copy()


def prefill(inputs: dict, rows=None, heads=None, threads: int = 0, rope: bool = False, fp8_latent: bool = False,
            emulate_bf16: bool = False):
    """Run the oracle prefill.

    ``inputs`` holds q [B,T,H,192], c_kv [B,T,512], k_pe [B,T,64] (bf16), gamma [512] fp32,
    topk_idx [B,T,K] int32 and either wkv_b [H*256,512] bf16 or, for an FP8 block-scaled weight,
    wkv_b_fp8 [H*256,512] (e4m3 bytes, uint8) with wkv_b_scale [2H,4] fp32 (torch CPU tensors or
    numpy arrays). ``rows``: flat row ids b*T+t (default: all). ``heads``: (h_begin, h_end)
    (default: all). ``rope``: q[..., 128:] and k_pe are unrotated and get YaRN RoPE at their
    positions. ``fp8_latent``: the normalised latent goes through the KV cache's FP8 round trip.
    ``emulate_bf16``: the diagnostic rounding-emulation mode (the pages' bf16 tensors rounded where
    the MHA prefill excerpt would hold them: wkv_b's output, the scores before and after the scale,
    the softmax weights, out); not a parity reference.
    Returns (out [R,Hs,128] fp64, lse [R,Hs] fp64, n_keys [R] int32).
    """
    q = _bits(inputs["q"])
    B, T, H, _ = q.shape
    c_kv = _bits(inputs["c_kv"])
    k_pe = _bits(inputs["k_pe"])
    if inputs.get("wkv_b_fp8") is not None:
        W = None
        W8 = _bytes(inputs["wkv_b_fp8"])
        Ws = np.ascontiguousarray(np.asarray(inputs["wkv_b_scale"], dtype=np.float32))
        assert W8.shape == (H * (NOPE + V), LATENT) and Ws.shape == ((H * (NOPE + V) + 127) // 128, LATENT // 128)
    else:
        W = _bits(inputs["wkv_b"])
        W8 = Ws = None
    g = np.ascontiguousarray(np.asarray(inputs["gamma"], dtype=np.float32))
    topk = np.ascontiguousarray(np.asarray(inputs["topk_idx"], dtype=np.int32))
    K = topk.shape[-1]
    assert c_kv.shape == (B, T, LATENT) and k_pe.shape == (B, T, ROPE) and topk.shape == (B, T, K)
    if rows is None:
        rows_arr = None
        nr = B * T
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nr = rows_arr.size
    h0, h1 = (0, H) if heads is None else heads
    out = np.empty((nr, h1 - h0, V), dtype=np.float64)
    lse = np.empty((nr, h1 - h0), dtype=np.float64)
    nk = np.empty(nr, dtype=np.int32)
    opts = (1 if rope else 0) | (2 if fp8_latent else 0) | (4 if emulate_bf16 else 0)
    rc = _load().oracle_prefill_opt(B, T, H, K, _ptr(q), _ptr(c_kv), _ptr(k_pe), _ptr(g),
                                    None if W is None else _ptr(W), None if W8 is None else _ptr(W8),
                                    None if Ws is None else _ptr(Ws), _ptr(topk), nr,
                                    None if rows_arr is None else _ptr(rows_arr), h0, h1, opts,
                                    _ptr(out), _ptr(lse), _ptr(nk), int(threads))
    if rc != 0:
        raise ValueError("oracle_prefill rejected its arguments")
    return out, lse, nk


def _bytes(a) -> np.ndarray:
    """uint8 tensor (torch) or array -> contiguous uint8 numpy array."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint8
        return np.ascontiguousarray(a)
    import torch  # plumbing only: the bytes of a CPU tensor
    if a.dtype != torch.uint8:
        a = a.view(torch.uint8)
    return np.ascontiguousarray(a.detach().cpu().contiguous().numpy())


def latent(c_kv, gamma, fp8_latent: bool = False) -> np.ndarray:
    """The normalised latent the path up-projects (and the KV-cache excerpt stores): kv_norm, then
    with ``fp8_latent`` the FP8 round trip. c_kv bf16 [..., 512] -> bf16 values as fp64."""
    xb = _bits(c_kv)
    shape = xb.shape
    n = int(np.prod(shape[:-1]))
    g = np.ascontiguousarray(np.asarray(gamma, dtype=np.float32))
    y = np.empty((n, LATENT), dtype=np.float64)
    _load().oracle_latent(_ptr(xb), _ptr(g), n, 1 if fp8_latent else 0, _ptr(y))
    return y.reshape(shape)


def round_to_e4m3(x: np.ndarray) -> np.ndarray:
    """The oracle's e4m3 rounding (nearest, ties to even, saturating at 448), elementwise."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_round_to_e4m3(_ptr(x), x.size, _ptr(y))
    return y


def e4m3_values() -> np.ndarray:
    """The value of each of the 256 e4m3 byte codes (NaN for 0x7F and 0xFF)."""
    v = np.empty(256, dtype=np.float64)
    _load().oracle_e4m3_values(_ptr(v))
    return v


def fp8_weight(W8, scale) -> np.ndarray:
    """Effective bf16 weight of an FP8 block-scaled wkv_b: e4m3 bytes [rows, 512] and fp32 scales
    [ceil(rows/128), 4] -> [rows, 512] bf16 values as fp64."""
    w8 = _bytes(W8)
    sc = np.ascontiguousarray(np.asarray(scale, dtype=np.float32))
    rows = w8.shape[0]
    assert w8.shape == (rows, LATENT) and sc.shape == ((rows + 127) // 128, LATENT // 128)
    w = np.empty((rows, LATENT), dtype=np.float64)
    _load().oracle_fp8_weight(_ptr(w8), _ptr(sc), rows, _ptr(w))
    return w


def yarn_inv_freq() -> np.ndarray:
    """The 32 YaRN rotary frequencies (radians per position) of the 64-wide rotary key."""
    f = np.empty(ROPE // 2, dtype=np.float64)
    _load().oracle_yarn_inv_freq(_ptr(f))
    return f


def rope(x, positions) -> np.ndarray:
    """YaRN rotary embedding of bf16 vectors x [N, 64] at integer positions [N] -> bf16 values
    as fp64 [N, 64]."""
    xb = _bits(x)
    n = xb.shape[0]
    assert xb.shape == (n, ROPE)
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int32))
    assert pos.shape == (n,)
    y = np.empty((n, ROPE), dtype=np.float64)
    _load().oracle_rope(_ptr(xb), _ptr(pos), n, _ptr(y))
    return y
