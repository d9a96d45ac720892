"""GPU parity of the split-K path of sparse_mla_fwd at every split count.

With B*Tq queries below the SM count, each query's index list is processed in
nsplit = min(8, SMs // (B*Tq)) key ranges whose partial results (BF16 outputs,
FP32 log-sum-exps) are then combined.  On a 152-SM part the batches below give
every split count from 8 down to 1 (1..19 -> 8, 21 -> 7, 25 -> 6, 30 -> 5,
38 -> 4, 50 -> 3, 76 -> 2, 151 -> 1).  Context lengths are ragged: lists
shorter than one block (so that some splits get no block at all), lists of
exactly 2,048 and 2,049 keys, one empty list, -1 entries scattered through the
lists and the entries in random order.  Sampled rows are checked against the
oracle, every row for finiteness, and the empty list gives o = 0, lse = -inf.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import bf, check_mla_rows, i32, to_u16
from workloads import normal_bf16

pytestmark = pytest.mark.gpu

TOPK = 2048
H = 96
SCALE = 1.0 / np.sqrt(192.0)


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_serving_gb300 as m
    return m


def _lists(seed, lens, empty):
    """Per request (query at position L-1): min(L, k) distinct keys of [0, L)
    in random slots of the k-entry list, the rest -1; request `empty` has none."""
    rng = np.random.default_rng([seed, 1])
    B = len(lens)
    idx = np.full((B, 1, TOPK), -1, np.int32)
    for b, L in enumerate(lens):
        if b == empty:
            continue
        n = min(int(L), TOPK)
        keys = rng.permutation(int(L))[:n]
        slots = np.sort(rng.choice(TOPK, n, replace=False)) if rng.random() < 0.5 \
            else np.arange(n)
        idx[b, 0, slots] = keys
        rng.shuffle(idx[b, 0, :slots[-1] + 1] if n else idx[b, 0, :0])
    return idx


@pytest.mark.parametrize("B", [1, 2, 4, 5, 8, 19, 21, 25, 30, 38, 50, 76, 151])
def test_split_counts(dsa, B):
    seed = 700 + B
    rng = np.random.default_rng(seed)
    lens = rng.integers(1900, 2300, size=B).astype(np.int32)
    edge = [1, 64, 65, 2048, 2049, 300]
    n_edge = min(len(edge), max(B - 1, 0))
    lens[:n_edge] = edge[:n_edge]
    empty = min(6, B - 1) if B > 1 else -1
    S = int(lens.max())
    kv = normal_bf16(seed, "kv", (B, S, 576))
    q = normal_bf16(seed, "q_lat", (B, 1, H, 576))
    idx = _lists(seed, lens, empty)
    qs, kl = lens - 1, lens
    o, lse = dsa.sparse_mla_fwd(bf(q), dsa.Rows(bf(kv)), i32(idx), i32(qs), i32(kl), S, SCALE)
    torch.cuda.synchronize()
    og, lg = to_u16(o), lse.cpu().numpy()
    rows = np.unique(np.array([0, 1, 2, 3, 4, 5, B // 2, B - 1]) % B)
    rows = rows[rows != empty]
    check_mla_rows(og, lg, q, kv, idx, qs, kl, SCALE, rows, f"split B={B}")
    if empty >= 0:
        assert np.all(og[empty] == 0) and np.all(np.isneginf(lg[empty]))
    keep = np.arange(B) != empty
    assert np.all(np.isfinite(lg[keep]))
