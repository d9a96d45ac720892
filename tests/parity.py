"""Acceptance rules shared by the GPU parity tests.

* Index sets: a query at position t gets exactly min(t+1, k) distinct keys in
  [0, t], then -1 padding.  Every key in the symmetric difference between the
  GPU set and the oracle's top-k set must be a near-tie: its oracle score lies
  within 1e-3 (relative) of the k-th score s_k; when s_k == 0 only exact zeros
  qualify.
* Floating-point outputs: max-abs <= 2e-2 and relative L2 <= 1e-2 against the
  float64 oracle; log-sum-exp within 1e-3 absolute.
"""

from __future__ import annotations

import numpy as np

TIE_REL = 1e-3
MAX_ABS = 2e-2
REL_L2 = 1e-2
LSE_ABS = 1e-3


def check_index_row(gpu_row: np.ndarray, scores: np.ndarray, n_valid: int, k: int,
                    oracle_row: np.ndarray, kth: float, where: str = "") -> int:
    """Check one query's GPU index row; returns the number of near-tie swaps."""
    gpu_row = np.asarray(gpu_row)
    m = min(n_valid, k)
    head, tail = gpu_row[:m], gpu_row[m:]
    assert np.all(tail == -1), f"{where}: padding is not -1"
    assert np.all(head >= 0) and np.all(head < n_valid), f"{where}: index out of [0, t]"
    g = set(int(v) for v in head)
    assert len(g) == m, f"{where}: duplicate indices"
    o = set(int(v) for v in oracle_row if v >= 0)
    assert len(o) == m
    diff = g ^ o
    if not diff:
        return 0
    assert n_valid > k, f"{where}: a query with <= k keys must keep all of them"
    if kth == 0.0:
        bad = [s for s in diff if scores[s] != 0.0]
    else:
        tol = TIE_REL * abs(kth)
        bad = [s for s in diff if abs(scores[s] - kth) > tol]
    assert not bad, (f"{where}: {len(bad)} keys differ beyond the near-tie band; e.g. key {bad[0]} "
                     f"score {scores[bad[0]]!r} vs k-th {kth!r}")
    return len(diff) // 2


def check_close(gpu: np.ndarray, ref: np.ndarray, what: str, max_abs: float = MAX_ABS,
                rel_l2: float = REL_L2):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU values"
    err = np.abs(gpu - ref)
    ma = float(err.max()) if err.size else 0.0
    den = float(np.linalg.norm(ref))
    rl = float(np.linalg.norm(gpu - ref) / den) if den > 0 else float(np.linalg.norm(gpu))
    assert ma <= max_abs, f"{what}: max-abs {ma:.3g} > {max_abs}"
    assert rl <= rel_l2, f"{what}: rel-L2 {rl:.3g} > {rel_l2}"
    return ma, rl


def check_lse(gpu: np.ndarray, ref: np.ndarray, what: str):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    inf = np.isinf(ref)
    assert np.array_equal(np.isinf(gpu), inf), f"{what}: -inf pattern differs"
    d = np.abs(gpu[~inf] - ref[~inf])
    m = float(d.max()) if d.size else 0.0
    assert m <= LSE_ABS, f"{what}: lse max-abs {m:.3g} > {LSE_ABS}"
    return m
