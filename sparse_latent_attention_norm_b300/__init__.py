"""Python binding of libmla, the B300 (sm_103a) MLA sparse-prefill library.

Argument marshalling only: every step of the path (selection, kv_norm + wkv_b, attention) runs in
the CUDA kernels behind the C ABI declared in ``include/mla.h``. PyTorch supplies device memory
and streams. There is no CPU fallback: if ``libmla.so`` is missing or no CUDA device is present,
the calls raise.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

LATENT, NOPE, ROPE, QK, V = 512, 128, 64, 192, 128
FLAG_VALIDATE_INDICES = 1
FLAG_FP8_LATENT = 2
FLAG_ROPE = 4

STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CUDA",
                4: "MLA_ERR_INDEX", 5: "MLA_ERR_TIMEOUT", 6: "MLA_ERR_WORKSPACE", 7: "MLA_ERR_RANGE",
                8: "MLA_ERR_BOUNDS"}

# every entry point include/mla.h declares
SYMBOLS = ("mla_sparse_prefill_workspace_size", "mla_sparse_prefill", "mla_sparse_prefill_ex", "mla_canon_select",
           "mla_kvnorm_wkvb", "mla_sparse_attention", "mla_get_status", "mla_clear_status", "mla_softmax_scale",
           "mla_status_string", "mla_sparse_prefill_noalloc", "mla_selftest_wait_timeout",
           "mla_sparse_prefill_opt_workspace_size", "mla_sparse_prefill_opt", "mla_dequant_wkvb_fp8",
           "mla_kvnorm_wkvb_opt", "mla_rope_k_pe", "mla_yarn_frequencies", "mla_sparse_attention_opt")


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("K", ctypes.c_int32)]


class PrefillOptions(ctypes.Structure):
    """mla_prefill_options (include/mla.h)."""
    _fields_ = [("flags", ctypes.c_uint), ("n_keys", ctypes.c_void_p), ("wkv_b_scale", ctypes.c_void_p),
                ("kv_cache", ctypes.c_void_p), ("pe_cache", ctypes.c_void_p), ("cache_len", ctypes.c_int32)]


_lib = None
LIB_CHECKS_PATH = os.path.join(_HERE, "libmla_checks.so")


def load(path: str) -> ctypes.CDLL:
    """Load a build of libmla from `path` and declare its entry points' argument types."""
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} is not built ({path}); run "
                           "`python -m sparse_latent_attention_norm_b300.build`")
    L = ctypes.CDLL(path)
    P, I, U, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
    L.mla_sparse_prefill_workspace_size.restype = S
    L.mla_sparse_prefill_workspace_size.argtypes = [Dims]
    L.mla_sparse_prefill.restype = I
    L.mla_sparse_prefill.argtypes = [P] * 8 + [Dims, P, S, P]
    L.mla_sparse_prefill_ex.restype = I
    L.mla_sparse_prefill_ex.argtypes = [P] * 8 + [Dims, P, S, P, P, U]
    L.mla_canon_select.restype = I
    L.mla_canon_select.argtypes = [P, Dims, P, P, U, P]
    L.mla_kvnorm_wkvb.restype = I
    L.mla_kvnorm_wkvb.argtypes = [P, P, P, Dims, P, P, P]
    L.mla_sparse_attention.restype = I
    L.mla_sparse_attention.argtypes = [P] * 7 + [Dims, P]
    L.mla_get_status.restype = I
    L.mla_get_status.argtypes = []
    L.mla_clear_status.restype = I
    L.mla_clear_status.argtypes = []
    L.mla_softmax_scale.restype = ctypes.c_double
    L.mla_softmax_scale.argtypes = []
    L.mla_status_string.restype = ctypes.c_char_p
    L.mla_status_string.argtypes = [I]
    L.mla_sparse_prefill_noalloc.restype = I
    L.mla_sparse_prefill_noalloc.argtypes = [P] * 8 + [Dims, P]
    L.mla_selftest_wait_timeout.restype = I
    L.mla_selftest_wait_timeout.argtypes = [P, P]
    OP = ctypes.POINTER(PrefillOptions)
    L.mla_sparse_prefill_opt_workspace_size.restype = S
    L.mla_sparse_prefill_opt_workspace_size.argtypes = [Dims, OP]
    L.mla_sparse_prefill_opt.restype = I
    L.mla_sparse_prefill_opt.argtypes = [P] * 8 + [Dims, P, S, P, OP]
    L.mla_dequant_wkvb_fp8.restype = I
    L.mla_dequant_wkvb_fp8.argtypes = [P, P, ctypes.c_int32, P, P]
    L.mla_kvnorm_wkvb_opt.restype = I
    L.mla_kvnorm_wkvb_opt.argtypes = [P, P, P, Dims, P, P, U, P, ctypes.c_int32, P]
    L.mla_rope_k_pe.restype = I
    L.mla_rope_k_pe.argtypes = [P, Dims, P, P, P, ctypes.c_int32, P]
    L.mla_yarn_frequencies.restype = None
    L.mla_yarn_frequencies.argtypes = [P]
    L.mla_sparse_attention_opt.restype = I
    L.mla_sparse_attention_opt.argtypes = [P] * 7 + [Dims, P, P]
    return L


def lib() -> ctypes.CDLL:
    """The loaded libmla.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MlaError(status, where)


def _ptr(t) -> ctypes.c_void_p | None:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, shape=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def dims_of(q, topk_idx) -> Dims:
    B, T, H, _ = q.shape
    return Dims(B, T, H, topk_idx.shape[-1])


def softmax_scale() -> float:
    return lib().mla_softmax_scale()


def status_string(status: int) -> str:
    return lib().mla_status_string(status).decode()


def workspace_size(B: int, T: int, H: int, K: int) -> int:
    return lib().mla_sparse_prefill_workspace_size(Dims(B, T, H, K))


def get_status() -> int:
    """Device status word of the current device (synchronizes)."""
    return lib().mla_get_status()


def clear_status() -> None:
    _check(lib().mla_clear_status(), "mla_clear_status")


def selftest_wait_timeout(stream=None) -> tuple[int, int]:
    """Run mla_selftest_wait_timeout and wait for it: (1 if the wait completed else 0, milliseconds
    waited). It leaves MLA_ERR_TIMEOUT in the status word; clear_status() resets it."""
    import torch
    res = torch.zeros(2, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream() if stream is None else stream
    _check(lib().mla_selftest_wait_timeout(ctypes.c_void_p(res.data_ptr()), ctypes.c_void_p(s.cuda_stream)),
           "mla_selftest_wait_timeout")
    s.synchronize()
    completed, ms = (int(x) for x in res.cpu().tolist())
    return completed, ms


def options(*, flags: int = 0, n_keys=None, wkv_b_scale=None, kv_cache=None, pe_cache=None,
            cache_len: int = 0) -> PrefillOptions:
    """mla_prefill_options from tensors (or None)."""
    return PrefillOptions(flags, _ptr(n_keys), _ptr(wkv_b_scale), _ptr(kv_cache), _ptr(pe_cache), cache_len)


def workspace_size_opt(B: int, T: int, H: int, K: int, opt: PrefillOptions | None = None) -> int:
    return lib().mla_sparse_prefill_opt_workspace_size(Dims(B, T, H, K), None if opt is None else ctypes.byref(opt))


def alloc_workspace(B: int, T: int, H: int, K: int, device=None, opt: PrefillOptions | None = None):
    """A workspace tensor (uint8) of the size mla_sparse_prefill (or, given `opt`,
    mla_sparse_prefill_opt) needs, 1024-byte aligned."""
    import torch
    n = workspace_size(B, T, H, K) if opt is None else workspace_size_opt(B, T, H, K, opt)
    if n == 0:
        raise MlaError(1, "workspace_size")
    raw = torch.empty(n + 1024, dtype=torch.uint8, device=device or "cuda")
    off = (-raw.data_ptr()) % 1024
    return raw[off:off + n]


def sparse_prefill(q, c_kv, k_pe, gamma, wkv_b, topk_idx, *, out=None, lse=None, workspace=None,
                   n_keys: bool = False, validate: bool = False, stream=None, fp8_latent: bool = False,
                   rope: bool = False, wkv_b_scale=None, kv_cache=None, pe_cache=None):
    """kv_norm -> wkv_b -> sparse causal attention. Returns (out, lse) or (out, lse, n_keys).

    Options (mla_sparse_prefill_opt): fp8_latent (FP8 round trip of the normalised latent), rope
    (q's rotary tail and k_pe arrive unrotated), wkv_b_scale (wkv_b is then uint8 e4m3 bytes with
    these [2H, 4] fp32 block scales), kv_cache [B, L, 512] / pe_cache [B, L, 64] bf16 (positions
    0..T-1 written)."""
    import torch
    B, T, H, _ = q.shape
    K = topk_idx.shape[-1]
    _need(q, "q", torch.bfloat16, (B, T, H, QK))
    _need(c_kv, "c_kv", torch.bfloat16, (B, T, LATENT))
    _need(k_pe, "k_pe", torch.bfloat16, (B, T, ROPE))
    _need(gamma, "gamma", torch.float32, (LATENT,))
    if wkv_b_scale is None:
        _need(wkv_b, "wkv_b", torch.bfloat16, (H * (NOPE + V), LATENT))
    else:
        _need(wkv_b, "wkv_b", torch.uint8, (H * (NOPE + V), LATENT))
        _need(wkv_b_scale, "wkv_b_scale", torch.float32, (2 * H, LATENT // 128))
    _need(topk_idx, "topk_idx", torch.int32, (B, T, K))
    if out is None:
        out = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, (B, T, H, V))
    _need(lse, "lse", torch.float32, (B, T, H))
    cache_len = 0
    if kv_cache is not None:
        _need(kv_cache, "kv_cache", torch.bfloat16)
        cache_len = kv_cache.shape[1]
        if kv_cache.shape[0] != B or kv_cache.shape[2] != LATENT:
            raise ValueError("kv_cache must be [B, cache_len, 512]")
    if pe_cache is not None:
        _need(pe_cache, "pe_cache", torch.bfloat16)
        if cache_len and pe_cache.shape[1] != cache_len:
            raise ValueError("kv_cache and pe_cache must have the same cache length")
        cache_len = pe_cache.shape[1]
        if pe_cache.shape[0] != B or pe_cache.shape[2] != ROPE:
            raise ValueError("pe_cache must be [B, cache_len, 64]")
    nk = torch.empty((B, T), dtype=torch.int32, device=q.device) if n_keys else None
    flags = (FLAG_VALIDATE_INDICES if validate else 0) | (FLAG_FP8_LATENT if fp8_latent else 0) | \
        (FLAG_ROPE if rope else 0)
    opt = options(flags=flags, n_keys=nk, wkv_b_scale=wkv_b_scale, kv_cache=kv_cache, pe_cache=pe_cache,
                  cache_len=cache_len)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().mla_sparse_prefill_opt(_ptr(q), _ptr(c_kv), _ptr(k_pe), _ptr(gamma), _ptr(wkv_b), _ptr(topk_idx),
                                      _ptr(out), _ptr(lse), Dims(B, T, H, K), _ptr(workspace), ws_bytes,
                                      _stream(stream), ctypes.byref(opt))
    _check(st, "mla_sparse_prefill_opt")
    return (out, lse, nk) if n_keys else (out, lse)


def dequant_wkvb_fp8(w8, scale, *, stream=None):
    """FP8 block-scaled weight (uint8 e4m3 bytes [rows, 512], fp32 scales [rows/128, 4]) -> its bf16
    weight [rows, 512]."""
    import torch
    rows = w8.shape[0]
    _need(w8, "w8", torch.uint8, (rows, LATENT))
    _need(scale, "scale", torch.float32, ((rows + 127) // 128, LATENT // 128))
    w = torch.empty((rows, LATENT), dtype=torch.bfloat16, device=w8.device)
    _check(lib().mla_dequant_wkvb_fp8(_ptr(w8), _ptr(scale), rows, _ptr(w), _stream(stream)), "mla_dequant_wkvb_fp8")
    return w


def rope_k_pe(k_pe, *, pe_cache=None, stream=None):
    """YaRN RoPE of k_pe [B, T, 64] at positions 0..T-1 -> (rotated k_pe, (cos, sin) table [T, 32, 2])."""
    import torch
    B, T, _ = k_pe.shape
    _need(k_pe, "k_pe", torch.bfloat16, (B, T, ROPE))
    rot = torch.empty_like(k_pe)
    cs = torch.empty((T, ROPE // 2, 2), dtype=torch.float32, device=k_pe.device)
    cache_len = 0 if pe_cache is None else pe_cache.shape[1]
    _check(lib().mla_rope_k_pe(_ptr(k_pe), Dims(B, T, 1, 1), _ptr(rot), _ptr(cs), _ptr(pe_cache), cache_len,
                               _stream(stream)), "mla_rope_k_pe")
    return rot, cs


def yarn_frequencies():
    """The 32 YaRN rotary frequencies libmla uses (host computation, fp64)."""
    import numpy as np
    f = np.empty(ROPE // 2, dtype=np.float64)
    lib().mla_yarn_frequencies(f.ctypes.data_as(ctypes.c_void_p))
    return f


def canon_select(topk_idx, T: int | None = None, *, n_keys: bool = True, validate: bool = False, stream=None):
    """Selection bitsets [B, T, W] uint32 (as int32 storage) and n_keys [B, T]."""
    import torch
    B, T_, K = topk_idx.shape
    T = T_ if T is None else T
    _need(topk_idx, "topk_idx", torch.int32)
    W = (T + 127) // 128 * 4
    bits = torch.zeros((B, T, W), dtype=torch.int32, device=topk_idx.device)
    nk = torch.empty((B, T), dtype=torch.int32, device=topk_idx.device) if n_keys else None
    _check(lib().mla_canon_select(_ptr(topk_idx), Dims(B, T, 1, K), _ptr(bits), _ptr(nk),
                                  FLAG_VALIDATE_INDICES if validate else 0, _stream(stream)), "mla_canon_select")
    return bits, nk


def kvnorm_wkvb(c_kv, gamma, wkv_b, *, fp8_latent: bool = False, kv_cache=None, stream=None):
    """kv_norm + wkv_b -> (kv [B, H, T, 256] fp16, klo [B, H, T, 128] uint8).

    kv[..., :128] = k_hi = fp16(k_nope), kv[..., 128:] = fp16(v); klo holds e4m3 bytes of
    (k_nope - k_hi) * 2^11. fp8_latent: the FP8 round trip of the normalised latent first;
    kv_cache [B, L, 512] bf16: receives the latent the GEMM consumed."""
    import torch
    B, T, _ = c_kv.shape
    H = wkv_b.shape[0] // (NOPE + V)
    _need(c_kv, "c_kv", torch.bfloat16, (B, T, LATENT))
    _need(gamma, "gamma", torch.float32, (LATENT,))
    _need(wkv_b, "wkv_b", torch.bfloat16, (H * (NOPE + V), LATENT))
    kv = torch.empty((B, H, T, NOPE + V), dtype=torch.float16, device=c_kv.device)
    klo = torch.empty((B, H, T, NOPE), dtype=torch.uint8, device=c_kv.device)
    cache_len = 0
    if kv_cache is not None:
        _need(kv_cache, "kv_cache", torch.bfloat16)
        cache_len = kv_cache.shape[1]
    _check(lib().mla_kvnorm_wkvb_opt(_ptr(c_kv), _ptr(gamma), _ptr(wkv_b), Dims(B, T, H, 1), _ptr(kv), _ptr(klo),
                                     FLAG_FP8_LATENT if fp8_latent else 0, _ptr(kv_cache), cache_len,
                                     _stream(stream)), "mla_kvnorm_wkvb_opt")
    return kv, klo


def k_nope_from(kv, klo):
    """k_nope (fp32) from kvnorm_wkvb's outputs: k_hi + e4m3(klo) * 2^-11 (torch, for inspection)."""
    import torch
    return kv[..., :NOPE].float() + klo.view(torch.float8_e4m3fn).float() * (2.0 ** -11)


def sparse_attention(q, k_pe, kv, klo, sel_bits, *, rope_cs=None, stream=None):
    """Attention stage alone from kvnorm_wkvb's (kv, klo) and canon_select's bitsets -> (out, lse).
    rope_cs: the table rope_k_pe returned (q's rotary tail is then rotated here; k_pe must be the
    rotated one)."""
    import torch
    B, T, H, _ = q.shape
    _need(q, "q", torch.bfloat16, (B, T, H, QK))
    _need(k_pe, "k_pe", torch.bfloat16, (B, T, ROPE))
    _need(kv, "kv", torch.float16, (B, H, T, NOPE + V))
    _need(klo, "klo", torch.uint8, (B, H, T, NOPE))
    _need(sel_bits, "sel_bits", torch.int32)
    if rope_cs is not None:
        _need(rope_cs, "rope_cs", torch.float32, (T, ROPE // 2, 2))
    out = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    _check(lib().mla_sparse_attention_opt(_ptr(q), _ptr(k_pe), _ptr(kv), _ptr(klo), _ptr(sel_bits), _ptr(out),
                                          _ptr(lse), Dims(B, T, H, 1), _ptr(rope_cs), _stream(stream)),
           "mla_sparse_attention_opt")
    return out, lse


# The model's weights (kv_norm's gain and wkv_b) and the per-step activations of the prefill.
WEIGHTS = ("gamma", "wkv_b")
ACTIVATIONS = ("q", "c_kv", "k_pe", "topk_idx")


class HostPrefill:
    """End-to-end use from host memory: per call, copy the inputs from (pinned) host tensors to the
    device, run mla_sparse_prefill and copy out / lse back to pinned host tensors. Device buffers
    and the workspace are allocated once for the shapes given at construction. After
    set_weights(gamma, wkv_b) the weights stay on the device and a call copies the activations
    (q, c_kv, k_pe, topk_idx) only."""

    def __init__(self, B: int, T: int, H: int, K: int, device="cuda"):
        import torch
        self.dims = (B, T, H, K)
        dev = torch.device(device)
        self.d = {
            "q": torch.empty((B, T, H, QK), dtype=torch.bfloat16, device=dev),
            "c_kv": torch.empty((B, T, LATENT), dtype=torch.bfloat16, device=dev),
            "k_pe": torch.empty((B, T, ROPE), dtype=torch.bfloat16, device=dev),
            "gamma": torch.empty((LATENT,), dtype=torch.float32, device=dev),
            "wkv_b": torch.empty((H * (NOPE + V), LATENT), dtype=torch.bfloat16, device=dev),
            "topk_idx": torch.empty((B, T, K), dtype=torch.int32, device=dev),
        }
        self.out = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
        self.ws = alloc_workspace(B, T, H, K, device=dev)
        self.out_h = torch.empty(self.out.shape, dtype=torch.bfloat16, pin_memory=True)
        self.lse_h = torch.empty(self.lse.shape, dtype=torch.float32, pin_memory=True)
        self.resident = False

    def set_weights(self, gamma, wkv_b) -> None:
        """Copy the weights to the device once; later calls copy the activations only."""
        self.d["gamma"].copy_(gamma)
        self.d["wkv_b"].copy_(wkv_b)
        self.resident = True

    def _copied(self):
        return ACTIVATIONS if self.resident else ACTIVATIONS + WEIGHTS

    def h2d_bytes(self, inputs) -> int:
        """Bytes a call copies host -> device."""
        return sum(inputs[k].numel() * inputs[k].element_size() for k in self._copied())

    def d2h_bytes(self) -> int:
        return self.out.numel() * 2 + self.lse.numel() * 4

    def __call__(self, inputs, stream=None):
        """inputs: dict of host tensors (pinned for asynchronous copies). Returns host (out, lse)
        after the stream has finished."""
        import torch
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            for k in self._copied():
                self.d[k].copy_(inputs[k], non_blocking=True)
            sparse_prefill(self.d["q"], self.d["c_kv"], self.d["k_pe"], self.d["gamma"], self.d["wkv_b"],
                           self.d["topk_idx"], out=self.out, lse=self.lse, workspace=self.ws, stream=s)
            self.out_h.copy_(self.out, non_blocking=True)
            self.lse_h.copy_(self.lse, non_blocking=True)
        s.synchronize()
        return self.out_h, self.lse_h


class HostPrefillPipeline:
    """Pipelined end-to-end use from host memory. Each submitted step copies its inputs from
    (pinned) host tensors to the device, runs mla_sparse_prefill and copies out / lse back to
    pinned host tensors, like HostPrefill, but on three streams: the host->device copies of step
    i run while step i-1 computes and step i-2's results travel back. Device input and output
    buffers are double-buffered (`depth` sets); the steps compute in submission order on one
    stream and share one workspace.

        pipe = HostPrefillPipeline(B, T, H, K)
        h = pipe.submit(inputs)          # returns at once
        out, lse = pipe.result(h)        # waits for that step's results on the host

    The host tensors a step returns are reused `depth` submissions later. After
    set_weights(gamma, wkv_b) the weights stay on the device (one copy shared by the buffer sets)
    and a step copies the activations (q, c_kv, k_pe, topk_idx) only."""

    def __init__(self, B: int, T: int, H: int, K: int, device="cuda", depth: int = 2):
        import torch
        if depth < 1:
            raise ValueError("depth must be >= 1")
        self.depth = depth
        self.dev = torch.device(device)
        self.slots = []
        for _ in range(depth):
            d = {
                "q": torch.empty((B, T, H, QK), dtype=torch.bfloat16, device=self.dev),
                "c_kv": torch.empty((B, T, LATENT), dtype=torch.bfloat16, device=self.dev),
                "k_pe": torch.empty((B, T, ROPE), dtype=torch.bfloat16, device=self.dev),
                "gamma": torch.empty((LATENT,), dtype=torch.float32, device=self.dev),
                "wkv_b": torch.empty((H * (NOPE + V), LATENT), dtype=torch.bfloat16, device=self.dev),
                "topk_idx": torch.empty((B, T, K), dtype=torch.int32, device=self.dev),
            }
            self.slots.append({
                "in": d,
                "out": torch.empty((B, T, H, V), dtype=torch.bfloat16, device=self.dev),
                "lse": torch.empty((B, T, H), dtype=torch.float32, device=self.dev),
                "out_h": torch.empty((B, T, H, V), dtype=torch.bfloat16, pin_memory=True),
                "lse_h": torch.empty((B, T, H), dtype=torch.float32, pin_memory=True),
                "in_free": None,    # event: the step that last used this slot has read its inputs
                "out_free": None,   # event: that step's results have reached the host
            })
        self.ws = alloc_workspace(B, T, H, K, device=self.dev)
        self.weights = None   # device (gamma, wkv_b) once set_weights has run
        self.s_h2d = torch.cuda.Stream(device=self.dev)
        self.s_comp = torch.cuda.Stream(device=self.dev)
        self.s_d2h = torch.cuda.Stream(device=self.dev)
        self.n = 0

    def set_weights(self, gamma, wkv_b) -> None:
        """Copy the weights to the device once (ordered before every later step); later steps
        copy the activations only."""
        import torch
        w = {"gamma": torch.empty_like(self.slots[0]["in"]["gamma"]),
             "wkv_b": torch.empty_like(self.slots[0]["in"]["wkv_b"])}
        with torch.cuda.stream(self.s_h2d):
            w["gamma"].copy_(gamma, non_blocking=True)
            w["wkv_b"].copy_(wkv_b, non_blocking=True)
        self.s_h2d.synchronize()
        self.weights = w

    def _copied(self):
        return ACTIVATIONS if self.weights is not None else ACTIVATIONS + WEIGHTS

    def h2d_bytes(self, inputs) -> int:
        """Bytes a step copies host -> device."""
        return sum(inputs[k].numel() * inputs[k].element_size() for k in self._copied())

    def d2h_bytes(self) -> int:
        o = self.slots[0]
        return o["out"].numel() * 2 + o["lse"].numel() * 4

    def submit(self, inputs):
        """Enqueue one step (inputs: dict of host tensors, pinned for asynchronous copies). Returns
        a handle for result()."""
        import torch
        slot = self.slots[self.n % self.depth]
        self.n += 1
        if slot["in_free"] is not None:
            self.s_h2d.wait_event(slot["in_free"])
        with torch.cuda.stream(self.s_h2d):
            for k in self._copied():
                slot["in"][k].copy_(inputs[k], non_blocking=True)
        copied = torch.cuda.Event()
        copied.record(self.s_h2d)
        self.s_comp.wait_event(copied)
        if slot["out_free"] is not None:
            self.s_comp.wait_event(slot["out_free"])
        d = dict(slot["in"], **self.weights) if self.weights is not None else slot["in"]
        sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"], out=slot["out"],
                       lse=slot["lse"], workspace=self.ws, stream=self.s_comp)
        computed = torch.cuda.Event()
        computed.record(self.s_comp)
        slot["in_free"] = computed
        self.s_d2h.wait_event(computed)
        with torch.cuda.stream(self.s_d2h):
            slot["out_h"].copy_(slot["out"], non_blocking=True)
            slot["lse_h"].copy_(slot["lse"], non_blocking=True)
        back = torch.cuda.Event()
        back.record(self.s_d2h)
        slot["out_free"] = back
        return (slot, back)

    def result(self, handle):
        """Host (out, lse) of a submitted step, once it has arrived."""
        slot, back = handle
        back.synchronize()
        return slot["out_h"], slot["lse_h"]
