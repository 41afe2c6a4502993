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

STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CUDA",
                4: "MLA_ERR_INDEX", 5: "MLA_ERR_TIMEOUT", 6: "MLA_ERR_WORKSPACE"}

# every entry point include/mla.h declares
SYMBOLS = ("mla_sparse_prefill_workspace_size", "mla_sparse_prefill", "mla_sparse_prefill_ex", "mla_canon_select",
           "mla_kvnorm_wkvb", "mla_sparse_attention", "mla_get_status", "mla_clear_status", "mla_softmax_scale",
           "mla_status_string", "mla_sparse_prefill_noalloc", "mla_selftest_wait_timeout")


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("K", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmla.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmla.so is not built ({LIB_PATH}); run "
                               "`python -m sparse_latent_attention_norm_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
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
        _lib = L
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


def alloc_workspace(B: int, T: int, H: int, K: int, device=None):
    """A workspace tensor (uint8) of the size mla_sparse_prefill needs, 1024-byte aligned."""
    import torch
    n = workspace_size(B, T, H, K)
    if n == 0:
        raise MlaError(1, "workspace_size")
    raw = torch.empty(n + 1024, dtype=torch.uint8, device=device or "cuda")
    off = (-raw.data_ptr()) % 1024
    return raw[off:off + n]


def sparse_prefill(q, c_kv, k_pe, gamma, wkv_b, topk_idx, *, out=None, lse=None, workspace=None,
                   n_keys: bool = False, validate: bool = False, stream=None):
    """kv_norm -> wkv_b -> sparse causal attention. Returns (out, lse) or (out, lse, n_keys)."""
    import torch
    B, T, H, _ = q.shape
    K = topk_idx.shape[-1]
    _need(q, "q", torch.bfloat16, (B, T, H, QK))
    _need(c_kv, "c_kv", torch.bfloat16, (B, T, LATENT))
    _need(k_pe, "k_pe", torch.bfloat16, (B, T, ROPE))
    _need(gamma, "gamma", torch.float32, (LATENT,))
    _need(wkv_b, "wkv_b", torch.bfloat16, (H * (NOPE + V), LATENT))
    _need(topk_idx, "topk_idx", torch.int32, (B, T, K))
    if out is None:
        out = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, (B, T, H, V))
    _need(lse, "lse", torch.float32, (B, T, H))
    nk = torch.empty((B, T), dtype=torch.int32, device=q.device) if n_keys else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().mla_sparse_prefill_ex(_ptr(q), _ptr(c_kv), _ptr(k_pe), _ptr(gamma), _ptr(wkv_b), _ptr(topk_idx),
                                     _ptr(out), _ptr(lse), Dims(B, T, H, K), _ptr(workspace), ws_bytes,
                                     _stream(stream), _ptr(nk), FLAG_VALIDATE_INDICES if validate else 0)
    _check(st, "mla_sparse_prefill_ex")
    return (out, lse, nk) if n_keys else (out, lse)


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


def kvnorm_wkvb(c_kv, gamma, wkv_b, *, stream=None):
    """kv_norm + wkv_b -> (kv [B, H, T, 256] fp16, klo [B, H, T, 128] uint8).

    kv[..., :128] = k_hi = fp16(k_nope), kv[..., 128:] = fp16(v); klo holds e4m3 bytes of
    (k_nope - k_hi) * 2^11."""
    import torch
    B, T, _ = c_kv.shape
    H = wkv_b.shape[0] // (NOPE + V)
    _need(c_kv, "c_kv", torch.bfloat16, (B, T, LATENT))
    _need(gamma, "gamma", torch.float32, (LATENT,))
    _need(wkv_b, "wkv_b", torch.bfloat16, (H * (NOPE + V), LATENT))
    kv = torch.empty((B, H, T, NOPE + V), dtype=torch.float16, device=c_kv.device)
    klo = torch.empty((B, H, T, NOPE), dtype=torch.uint8, device=c_kv.device)
    _check(lib().mla_kvnorm_wkvb(_ptr(c_kv), _ptr(gamma), _ptr(wkv_b), Dims(B, T, H, 1), _ptr(kv), _ptr(klo),
                                 _stream(stream)), "mla_kvnorm_wkvb")
    return kv, klo


def k_nope_from(kv, klo):
    """k_nope (fp32) from kvnorm_wkvb's outputs: k_hi + e4m3(klo) * 2^-11 (torch, for inspection)."""
    import torch
    return kv[..., :NOPE].float() + klo.view(torch.float8_e4m3fn).float() * (2.0 ** -11)


def sparse_attention(q, k_pe, kv, klo, sel_bits, *, stream=None):
    """Attention stage alone from kvnorm_wkvb's (kv, klo) and canon_select's bitsets -> (out, lse)."""
    import torch
    B, T, H, _ = q.shape
    _need(q, "q", torch.bfloat16, (B, T, H, QK))
    _need(k_pe, "k_pe", torch.bfloat16, (B, T, ROPE))
    _need(kv, "kv", torch.float16, (B, H, T, NOPE + V))
    _need(klo, "klo", torch.uint8, (B, H, T, NOPE))
    _need(sel_bits, "sel_bits", torch.int32)
    out = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    _check(lib().mla_sparse_attention(_ptr(q), _ptr(k_pe), _ptr(kv), _ptr(klo), _ptr(sel_bits), _ptr(out), _ptr(lse),
                                      Dims(B, T, H, 1), _stream(stream)), "mla_sparse_attention")
    return out, lse


class HostPrefill:
    """End-to-end use from host memory: per call, copy the inputs from (pinned) host tensors to the
    device, run mla_sparse_prefill and copy out / lse back to pinned host tensors. Device buffers
    and the workspace are allocated once for the shapes given at construction."""

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

    def h2d_bytes(self, inputs) -> int:
        return sum(inputs[k].numel() * inputs[k].element_size() for k in self.d)

    def d2h_bytes(self) -> int:
        return self.out.numel() * 2 + self.lse.numel() * 4

    def __call__(self, inputs, stream=None):
        """inputs: dict of host tensors (pinned for asynchronous copies). Returns host (out, lse)
        after the stream has finished."""
        import torch
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            for k, dst in self.d.items():
                dst.copy_(inputs[k], non_blocking=True)
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

    The host tensors a step returns are reused `depth` submissions later."""

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
        self.s_h2d = torch.cuda.Stream(device=self.dev)
        self.s_comp = torch.cuda.Stream(device=self.dev)
        self.s_d2h = torch.cuda.Stream(device=self.dev)
        self.n = 0

    def h2d_bytes(self, inputs) -> int:
        return sum(inputs[k].numel() * inputs[k].element_size() for k in self.slots[0]["in"])

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
            for k, dst in slot["in"].items():
                dst.copy_(inputs[k], non_blocking=True)
        copied = torch.cuda.Event()
        copied.record(self.s_h2d)
        self.s_comp.wait_event(copied)
        if slot["out_free"] is not None:
            self.s_comp.wait_event(slot["out_free"])
        d = slot["in"]
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
