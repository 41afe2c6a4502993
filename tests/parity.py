"""Comparison helpers shared by the GPU parity tests, the smoke check and the benchmark's
full-size parity sample. Tolerances (bf16 path against the fp64 oracle):
  out : max |delta| <= 2e-2 and ||delta||_2 / ||ref||_2 <= 1e-2
  lse : |delta| <= 1e-3 * max(1, |ref|)   (-inf exactly where the selected set is empty)
  n_keys : bit-exact
"""

from __future__ import annotations

import numpy as np

OUT_MAX_ABS = 2e-2
OUT_REL_L2 = 1e-2
LSE_REL = 1e-3


def sample_rows(B: int, T: int, K: int, n_random: int = 24, seed: int = 0) -> np.ndarray:
    """Flat row ids b*T + t: tile edges, the top-k boundary, the last rows, plus seeded random rows."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, K - 2, K - 1, K, T // 2, T - 129, T - 128, T - 1]
    rows = set()
    for b in range(B):
        for t in fixed:
            if 0 <= t < T:
                rows.add(b * T + t)
    rows.update(int(r) for r in rng.integers(0, B * T, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what: str = "") -> dict:
    """out_*: [R, H, 128]; lse_*: [R, H]. Raises AssertionError with the figures on failure."""
    og = np.asarray(out_gpu, dtype=np.float64)
    orf = np.asarray(out_ref, dtype=np.float64)
    lg = np.asarray(lse_gpu, dtype=np.float64)
    lr = np.asarray(lse_ref, dtype=np.float64)
    assert og.shape == orf.shape and lg.shape == lr.shape, (og.shape, orf.shape, lg.shape, lr.shape)
    diff = og - orf
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    ref_norm = float(np.linalg.norm(orf))
    rel_l2 = float(np.linalg.norm(diff) / ref_norm) if ref_norm > 0 else float(np.linalg.norm(diff))
    empty = np.isneginf(lr)
    assert np.array_equal(np.isneginf(lg), empty), f"{what}: lse -inf pattern differs"
    fin = ~empty
    lse_err = np.abs(lg[fin] - lr[fin]) / np.maximum(1.0, np.abs(lr[fin])) if fin.any() else np.zeros(1)
    lse_worst = float(lse_err.max())
    res = {"out_max_abs": max_abs, "out_rel_l2": rel_l2, "lse_rel_max": lse_worst,
           "rows": int(og.shape[0]), "empty_rows": int(empty.any(axis=-1).sum())}
    assert np.isfinite(og).all(), f"{what}: non-finite out"
    assert max_abs <= OUT_MAX_ABS, f"{what}: out max-abs {max_abs:.3e} > {OUT_MAX_ABS} ({res})"
    assert rel_l2 <= OUT_REL_L2, f"{what}: out rel-L2 {rel_l2:.3e} > {OUT_REL_L2} ({res})"
    assert lse_worst <= LSE_REL, f"{what}: lse rel {lse_worst:.3e} > {LSE_REL} ({res})"
    return res


def expected_bits(topk: np.ndarray, T: int, oracle) -> tuple[np.ndarray, np.ndarray]:
    """Selection bitsets [B, T, W] (uint32, words the kernel writes) and counts, from the oracle's
    canonical sets."""
    B = topk.shape[0]
    W = (T + 127) // 128 * 4
    bits = np.zeros((B, T, W), dtype=np.uint32)
    counts = np.zeros((B, T), dtype=np.int32)
    for b in range(B):
        for t in range(T):
            sel = oracle.canon_row(topk[b, t], t)
            counts[b, t] = sel.size
            if sel.size:
                np.bitwise_or.at(bits[b, t], sel >> 5, (np.uint32(1) << (sel & 31).astype(np.uint32)))
    return bits, counts
