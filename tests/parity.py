"""Shared comparison helpers for the GPU-vs-oracle parity tests."""
from __future__ import annotations

import numpy as np

# Floating-point bar: |gpu - oracle| <= RTOL * (1 + |oracle|) per logit.
RTOL = 1e-4


def assert_logits_close(gpu: np.ndarray, ref: np.ndarray, what: str = "logits"):
    gpu = np.asarray(gpu, np.float32)
    ref = np.asarray(ref, np.float32)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    ninf_r = np.isneginf(ref)
    ninf_g = np.isneginf(gpu)
    bad_mask = np.argwhere(ninf_r != ninf_g)
    assert bad_mask.size == 0, f"{what}: -inf mask differs at {bad_mask[:5].tolist()}"
    fin = ~ninf_r
    assert np.isfinite(gpu[fin]).all(), f"{what}: non-finite GPU value where oracle is finite"
    err = np.abs(gpu[fin].astype(np.float64) - ref[fin].astype(np.float64))
    bound = RTOL * (1.0 + np.abs(ref[fin].astype(np.float64)))
    if err.size:
        worst = int(np.argmax(err / bound))
        assert (err <= bound).all(), (
            f"{what}: {(err > bound).sum()} values out of tolerance; worst |d|={err[worst]:.3g} "
            f"bound={bound[worst]:.3g} ref={ref[fin][worst]:.6g}")
    return float(err.max()) if err.size else 0.0


def topk_sets(idx: np.ndarray) -> list[np.ndarray]:
    """Per row: the sorted selected indices (padding -1 removed)."""
    return [np.sort(r[r >= 0]) for r in np.asarray(idx)]


def assert_topk_exact(gpu_idx: np.ndarray, ora_idx: np.ndarray, what: str = "topk"):
    """Bit-exact set equality plus the GPU's own layout contract: ascending
    indices, then -1 padding."""
    g = np.asarray(gpu_idx)
    for r, (a, b) in enumerate(zip(topk_sets(g), topk_sets(ora_idx))):
        assert np.array_equal(a, b), f"{what}: row {r} differs ({len(a)} vs {len(b)} selected)"
        row = g[r]
        n = len(a)
        assert np.array_equal(row[:n], a), f"{what}: row {r} not in ascending index order"
        assert (row[n:] == -1).all(), f"{what}: row {r} padding is not -1"


def assert_topk_near_tie(gpu_idx, ora_idx, ora_logits, lengths, k, what="topk"):
    """End-to-end top-k (each side on its own logits): the sets must match
    exactly unless the k-th and (k+1)-th oracle logits are closer than the
    logits tolerance; then only entries within that band may differ."""
    exempt = 0
    for r, (a, b) in enumerate(zip(topk_sets(gpu_idx), topk_sets(ora_idx))):
        if np.array_equal(a, b):
            continue
        row = np.asarray(ora_logits[r, :lengths[r]], np.float64)
        fin = np.sort(row[np.isfinite(row)])[::-1]
        assert len(fin) > k, f"{what}: row {r} differs although every finite entry fits"
        vk, vk1 = fin[k - 1], fin[k]
        tol = RTOL * (1.0 + abs(vk))
        assert abs(vk - vk1) < tol, f"{what}: row {r} differs with a clear gap {vk - vk1:.3g}"
        diff = np.setxor1d(a, b)
        assert (np.abs(row[diff] - vk) <= 2 * tol).all(), f"{what}: row {r} far swap"
        exempt += 1
    return exempt
