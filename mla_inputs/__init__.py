"""Seeded synthetic inputs for the MLA sparse prefill (shared by the tests, the benchmark and the
oracle harness).

This module holds no step of the method: it draws random tensors and top-k index rows with the
shapes and distributions of the five workloads below and nothing else. Random values come from
numpy's PCG64 generator, seeded per (workload, tensor); floating-point tensors are drawn in
fp32 and rounded to bf16 (round-to-nearest-even, by torch's conversion).

Workloads (DeepSeek-V3.2-Exp MLA: latent 512, 128 nope + 64 rope key dims, 128 value dims):
  tiny          B=1 T=64    H=4   K=32
  dense_causal  B=1 T=1024  H=128 K=2048  (K >= T: every causal key selected)
  headline      B=1 T=4096  H=128 K=2048  (uniform top-k over the causal prefix)
  long_context  B=2 T=16384 H=128 K=2048  (half recent 4096 positions, half earlier prefix)
  stress        B=1 T=8192  H=128 K=2048  (outlier channels, x4 q/k_pe, shuffled rows, 5% dups)

Value distributions: q, c_kv, k_pe ~ N(0, 1); gamma ~ U(0.5, 1.5) rounded to bf16 values and
held as fp32; wkv_b ~ N(0, 1/512).
"""

from __future__ import annotations

import dataclasses

import numpy as np

LATENT, NOPE, ROPE, QK, V = 512, 128, 64, 192, 128
SEED_BASE = 0x4D4C4100

# tensor ids for per-tensor seeds
_T_Q, _T_CKV, _T_KPE, _T_GAMMA, _T_W, _T_IDX, _T_OUTLIER, _T_DUP = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    pattern: str            # "tiny" | "dense" | "uniform" | "clustered"
    recent: int = 4096      # clustered: size of the recent window (t included)
    stress: bool = False    # outlier channels, x4 q and k_pe, duplicates, shuffled rows
    seed_id: int = 0

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "T": self.T, "H": self.H, "K": self.K,
                "latent": LATENT, "d_qk": QK, "d_v": V, "pattern": self.pattern,
                "stress": self.stress}


WORKLOADS = {
    "tiny": Workload("tiny", 1, 64, 4, 32, "tiny", seed_id=0),
    "dense_causal": Workload("dense_causal", 1, 1024, 128, 2048, "dense", seed_id=1),
    "headline": Workload("headline", 1, 4096, 128, 2048, "uniform", seed_id=2),
    "long_context": Workload("long_context", 2, 16384, 128, 2048, "clustered", seed_id=3),
    "stress": Workload("stress", 1, 8192, 128, 2048, "uniform", stress=True, seed_id=4),
}


def _rng(w: Workload, tensor_id: int, extra: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + 16 * w.seed_id + tensor_id + (extra << 32)))


def _to_bf16(a: np.ndarray):
    import torch  # plumbing: fp32 -> bf16 rounding (RNE) and CPU tensors
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _normal_bf16(w: Workload, tensor_id: int, shape, std: float = 1.0, chunk_rows: int = 1 << 20):
    """N(0, std^2) drawn in fp32 chunk by chunk (bounded host memory), rounded to bf16."""
    import torch
    rng = _rng(w, tensor_id)
    rows = int(np.prod(shape[:-1]))
    cols = shape[-1]
    out = torch.empty((rows, cols), dtype=torch.bfloat16)
    step = max(1, chunk_rows // max(1, cols // 64))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = rng.standard_normal((r1 - r0, cols), dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[r0:r1] = _to_bf16(x)
    return out.reshape(shape)


def _distinct(rng: np.random.Generator, lo: int, hi: int, m: int) -> np.ndarray:
    """m distinct integers drawn uniformly from [lo, hi)."""
    if m <= 0 or hi <= lo:
        return np.empty(0, dtype=np.int64)
    return rng.choice(hi - lo, size=m, replace=False) + lo


def topk_row(w: Workload, t: int, rng: np.random.Generator) -> np.ndarray:
    """One top-k index row of length K for query t, following the workload's recipe."""
    T, K = w.T, w.K
    if w.pattern == "tiny":
        # t, min(K-1, t) distinct picks from [0, t), padded with distinct picks from (t, T)
        m = min(K - 1, t)
        row = [np.array([t]), _distinct(rng, 0, t, m)]
        pad = K - 1 - m
        row.append(_distinct(rng, t + 1, T, pad))
        r = np.concatenate(row)
    elif w.pattern == "dense":
        # every causal key [0, t], then padding that cycles through (t, T) (repeats t if empty)
        head = np.arange(t + 1)
        pad = K - (t + 1)
        if pad > 0:
            if t + 1 < T:
                tail = (t + 1) + (np.arange(pad) % (T - t - 1))
            else:
                tail = np.full(pad, t)
            r = np.concatenate([head, tail])
        else:
            r = head[:K]
    else:
        if t < K - 1:
            # all of [0, t], padded with distinct picks from (t, T) that the causal mask removes
            pad = K - (t + 1)
            avail = T - t - 1
            tail = _distinct(rng, t + 1, T, min(pad, avail))
            if tail.size < pad:
                tail = np.concatenate([tail, np.full(pad - tail.size, t)])
            r = np.concatenate([np.arange(t + 1), tail])
        elif w.pattern == "uniform":
            r = np.concatenate([[t], _distinct(rng, 0, t, K - 1)])
        elif w.pattern == "clustered":
            lo_recent = max(0, t - (w.recent - 1))
            n_recent_pool = t - lo_recent          # R = [lo_recent, t)
            n_prefix_pool = lo_recent              # P = [0, lo_recent)
            want_r, want_p = K // 2 - 1, K // 2
            take_p = min(want_p, n_prefix_pool)
            take_r = min(n_recent_pool, want_r + (want_p - take_p))
            take_p = min(n_prefix_pool, take_p + (want_r + want_p - take_p - take_r))
            r = np.concatenate([[t], _distinct(rng, lo_recent, t, take_r), _distinct(rng, 0, lo_recent, take_p)])
        else:
            raise ValueError(w.pattern)
    return r.astype(np.int32)


def make_topk(w: Workload) -> np.ndarray:
    """topk_idx [B, T, K] int32."""
    out = np.empty((w.B, w.T, w.K), dtype=np.int32)
    for b in range(w.B):
        rng = _rng(w, _T_IDX, extra=b + 1)
        for t in range(w.T):
            out[b, t] = topk_row(w, t, rng)
        if w.stress:
            drng = _rng(w, _T_DUP, extra=b + 1)
            n_dup = int(0.05 * w.K)
            for t in range(w.T):
                row = out[b, t]
                # overwrite n_dup entries other than the one holding t with copies of entries
                # that are kept, then shuffle the row (Fisher-Yates, numpy's shuffle)
                pos_t = int(np.flatnonzero(row == t)[0])
                victims = drng.choice(np.delete(np.arange(w.K), pos_t), size=n_dup, replace=False)
                keep = np.setdiff1d(np.arange(w.K), victims, assume_unique=True)
                row[victims] = row[drng.choice(keep, size=n_dup, replace=True)]
                drng.shuffle(row)
    return out


def make_inputs(w: Workload) -> dict:
    """All inputs of the workload as CPU tensors (bf16 / fp32) plus topk_idx as int32 numpy/torch."""
    import torch
    B, T, H = w.B, w.T, w.H
    q = _normal_bf16(w, _T_Q, (B, T, H, QK))
    c_kv = _normal_bf16(w, _T_CKV, (B, T, LATENT))
    k_pe = _normal_bf16(w, _T_KPE, (B, T, ROPE))
    g = _rng(w, _T_GAMMA).uniform(0.5, 1.5, size=LATENT).astype(np.float32)
    gamma = _to_bf16(g).to(torch.float32)
    wkv_b = _normal_bf16(w, _T_W, (H * (NOPE + V), LATENT), std=float(1.0 / np.sqrt(LATENT)))
    if w.stress:
        ch = _rng(w, _T_OUTLIER).choice(LATENT, size=8, replace=False)
        c_kv[..., torch.from_numpy(np.sort(ch))] *= 50.0
        q *= 4.0          # exact in bf16 (power of two)
        k_pe *= 4.0
    topk = torch.from_numpy(make_topk(w))
    return {"q": q, "c_kv": c_kv, "k_pe": k_pe, "gamma": gamma, "wkv_b": wkv_b, "topk_idx": topk,
            "workload": w}


def custom(name: str, B: int, T: int, H: int, K: int, pattern: str = "uniform", stress: bool = False,
           seed_id: int = 100, recent: int = 4096) -> Workload:
    """A workload with one of the recipes above at other sizes (tests: ragged tails, edge cases)."""
    return Workload(name, B, T, H, K, pattern, recent=recent, stress=stress, seed_id=seed_id)
