"""Acceptance rules shared by the GPU parity tests.

* Index sets: a query at position t gets exactly min(t+1, k) distinct keys in
  [0, t], then -1 padding.  Every key in the symmetric difference between the
  GPU set and the oracle's top-k set must be a near-tie: its oracle score lies
  within 1e-3 (relative) of the k-th score s_k; when s_k == 0 only exact zeros
  qualify.
* Floating-point outputs: max-abs <= 2e-2 and relative L2 <= 1e-2 against the
  float64 oracle; log-sum-exp within 1e-3 absolute.
* BF16 results of an FP32 computation (the indexer-key LayerNorm): equal to the
  oracle's rounding of its float64 value, except next to a rounding midpoint.
"""

from __future__ import annotations

import numpy as np

from workloads import bf16_to_f32

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


# BF16 results of an FP32 computation (the indexer-key LayerNorm) against the
# float64 value v: the GPU's BF16 must lie between the round-to-nearest-even
# BF16 values of v - delta and v + delta, where delta bounds the FP32
# computation's own error.  For y = (x - mean) / sqrt(var + eps) computed in FP32
# (a tree sum of at most 128 terms for the mean, one subtraction, a correctly
# rounded square root, division and product) the error is below
#   inv * (8 * 2^-24 * mean|x| + 2^-24 * |x - mean|) + 4 * 2^-24 * |y|,
# inv = 1/sqrt(var + eps); the tests use 2^-20 in place of 8 * 2^-24 and
# 2^-22 for the others, so near-zero outputs (x close to the mean, where the
# subtraction cancels) get an absolute allowance and the rest a few 2^-24.
def layernorm_delta(x: np.ndarray, v: np.ndarray, eps: float) -> np.ndarray:
    x = np.asarray(x, np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    inv = 1.0 / np.sqrt(((x - mean) ** 2).mean(axis=-1, keepdims=True) + eps)
    mabs = np.abs(x).mean(axis=-1, keepdims=True)
    return inv * (2.0 ** -20 * mabs + 2.0 ** -22 * np.abs(x - mean)) + 2.0 ** -22 * np.abs(v)


def check_bf16_of(gpu_bits: np.ndarray, v: np.ndarray, delta: np.ndarray, what: str):
    import oracle
    gpu_bits = np.asarray(gpu_bits, np.uint16).ravel()
    v = np.asarray(v, np.float64).ravel()
    delta = np.asarray(delta, np.float64).ravel()
    lo = bf16_to_f32(oracle.bf16_rne(v - delta)).astype(np.float64)
    hi = bf16_to_f32(oracle.bf16_rne(v + delta)).astype(np.float64)
    g = bf16_to_f32(gpu_bits).astype(np.float64)
    ok = (g >= lo) & (g <= hi)
    assert ok.all(), (f"{what}: {int((~ok).sum())} BF16 values outside rounding of the exact "
                      f"value +- delta, e.g. gpu={g[~ok][:4]} exact={v[~ok][:4]} delta={delta[~ok][:4]}")
    return int((gpu_bits != oracle.bf16_rne(v)).sum())
