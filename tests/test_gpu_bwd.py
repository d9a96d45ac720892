"""GPU parity of sparse_mla_bwd against the oracle's float64 gradient.

The GPU backward takes its own forward's o_lat and lse (as a training step
would); the oracle recomputes everything in float64 from the same BF16 inputs
and the same index set.  dq and dkv must each satisfy, against the float64
values: relative L2 error <= 1e-2 and max-abs error <= 2e-2 of the largest
reference magnitude (the output bar of the forward, applied relative to the
gradient's scale, which grows with the number of queries sharing a row).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bf, i32
from workloads import normal_bf16, page_table, to_pages

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS_REL = 2e-2


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_serving_gb300 as m
    return m


def _check(gpu, ref, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    err = np.abs(gpu - ref)
    scale = float(np.abs(ref).max()) or 1.0
    rl = float(np.linalg.norm(gpu - ref) / (np.linalg.norm(ref) or 1.0))
    assert err.max() <= MAX_ABS_REL * scale, f"{what}: max-abs {err.max():.3g} > {MAX_ABS_REL} x {scale:.3g}"
    assert rl <= REL_L2, f"{what}: rel-L2 {rl:.3g}"
    return rl


def _indices(seed, B, Tq, q0, k, frac_short=0.25):
    """A causal index set per query (distinct positions in [0, t]), -1 padded;
    some queries keep fewer than k entries, and the order is shuffled."""
    rng = np.random.default_rng([seed, 7])
    idx = np.full((B, Tq, k), -1, np.int32)
    for b in range(B):
        for i in range(Tq):
            t = q0 + i
            n = min(t + 1, k)
            if rng.random() < frac_short:
                n = int(rng.integers(0, n + 1))
            c = rng.permutation(t + 1)[:n]
            idx[b, i, :n] = c
            rng.shuffle(idx[b, i])
    return idx


def bwd_workspace(dsa, path, B, Tq, S, H, k):
    """"tc": as large as dsa_workspace_bytes reports (at 96 heads this selects the
    tcgen05 kernels); "warp": the bare status header (the warp-level MMA path)."""
    n = dsa.workspace_bytes(dsa.OP_SPARSE_MLA_BWD, B, Tq, S, H, k) if path == "tc" else 256
    return dsa.new_workspace(n)


def _run(dsa, q, kv_rows_dev, idx, q_start, kv_len, S, dO, dkv_shape, scale, path="tc"):
    qt, dOt = bf(q), bf(dO)
    it, qs, kl = i32(idx), i32(q_start), i32(kv_len)
    o_lat, lse = dsa.sparse_mla_fwd(qt, kv_rows_dev, it, qs, kl, S, scale)
    dkv = torch.zeros(dkv_shape, dtype=torch.float32, device="cuda")
    B, Tq, H = q.shape[:3]
    ws = bwd_workspace(dsa, path, B, Tq, S, H, idx.shape[-1])
    dq = dsa.sparse_mla_bwd(qt, kv_rows_dev, it, qs, kl, S, o_lat, lse, dOt, dkv, scale,
                            workspace=ws)
    code, where, detail = dsa.read_device_status(ws)
    return dq.cpu().numpy(), dkv.cpu().numpy(), code


@pytest.mark.parametrize("B,T,H,k,path", [(1, 256, 8, 64, "warp"), (2, 300, 96, 64, "warp"),
                                          (1, 160, 96, 200, "warp"), (2, 300, 96, 64, "tc"),
                                          (1, 160, 96, 200, "tc"), (1, 520, 96, 384, "tc")])
def test_bwd_contiguous(dsa, B, T, H, k, path):
    """Contiguous latent rows; ragged key counts (some queries keep fewer than k,
    some none), k not a multiple of the 32-key (warp path) or 128-key (tensor-core
    path) block."""
    seed = 100 + T + H
    q = normal_bf16(seed, "q_lat", (B, T, H, 576))
    kv = normal_bf16(seed, "kv", (B, T, 576))
    dO = normal_bf16(seed, "w", (B, T, H, 512))
    idx = _indices(seed, B, T, 0, k)
    q_start, kv_len = np.zeros(B, np.int32), np.full(B, T, np.int32)
    scale = 1.0 / np.sqrt(192.0)
    dq, dkv, code = _run(dsa, q, dsa.Rows(bf(kv)), idx, q_start, kv_len, T, dO, (B, T, 576), scale,
                         path)
    assert code == dsa.DSA_OK
    rdq, rdkv = oracle.sparse_mla_bwd(q, kv, idx, q_start, kv_len, scale, dO)
    _check(dq, rdq, "dq")
    _check(dkv, rdkv, "dkv")
    # queries with no valid entry have zero dq
    empty = (idx < 0).all(axis=-1)
    assert np.all(dq[empty] == 0.0)


def test_bwd_paged_chunk(dsa):
    """Queries 256..383 of a sequence over a paged latent cache (q_start > 0);
    dkv is a page pool and is added to, not overwritten."""
    B, S, q0, Tq, H, k = 1, 384, 256, 128, 96, 128
    seed = 131
    kv_log = normal_bf16(seed, "kv", (B, S, 576))
    q = normal_bf16(seed, "q_lat", (B, Tq, H, 576))
    dO = normal_bf16(seed, "w", (B, Tq, H, 512))
    idx = _indices(seed, B, Tq, q0, k)
    lens = np.full(B, S, np.int32)
    bt, npages = page_table(seed, lens)
    pool = to_pages(kv_log, lens, bt, npages)
    q_start, kv_len = np.full(B, q0, np.int32), np.full(B, q0 + Tq, np.int32)
    scale = 1.0 / np.sqrt(192.0)
    rows = dsa.Rows(bf(pool), i32(bt))
    qt, dOt = bf(q), bf(dO)
    it, qs, kl = i32(idx), i32(q_start), i32(kv_len)
    o_lat, lse = dsa.sparse_mla_fwd(qt, rows, it, qs, kl, S, scale)
    base = np.random.default_rng(5).standard_normal((npages, 64, 576)).astype(np.float32)
    dkv = torch.from_numpy(base.copy()).cuda()
    dq = dsa.sparse_mla_bwd(qt, rows, it, qs, kl, S, o_lat, lse, dOt, dkv, scale)
    torch.cuda.synchronize()
    rdq, rdkv = oracle.sparse_mla_bwd(q, kv_log[:, :q0 + Tq], idx, q_start, kv_len, scale, dO)
    _check(dq.cpu().numpy(), rdq, "dq")
    got = dkv.cpu().numpy() - base
    want = np.zeros_like(base, dtype=np.float64)
    for s in range(q0 + Tq):
        want[bt[0, s // 64], s % 64] = rdkv[0, s]
    _check(got, want, "dkv (pool, added)")


@pytest.mark.parametrize("H,path", [(8, "warp"), (96, "tc")])
def test_bwd_bad_index_is_flagged_and_skipped(dsa, H, path):
    """A non-causal entry: DSA_ERR_BAD_INDEX, and the gradients equal those of
    the index set without it."""
    B, T, k = 1, 96, 32
    seed = 141
    q = normal_bf16(seed, "q_lat", (B, T, H, 576))
    kv = normal_bf16(seed, "kv", (B, T, 576))
    dO = normal_bf16(seed, "w", (B, T, H, 512))
    idx = _indices(seed, B, T, 0, k, frac_short=0.0)
    clean = idx.copy()
    idx[0, 40, 3] = 77          # key 77 is in the future of query 40
    clean[0, 40, 3] = -1
    q_start, kv_len = np.zeros(B, np.int32), np.full(B, T, np.int32)
    scale = 1.0 / np.sqrt(192.0)
    rows = dsa.Rows(bf(kv))
    qt, dOt = bf(q), bf(dO)
    qs, kl = i32(q_start), i32(kv_len)
    # the forward on the clean set (it would flag the bad entry too)
    o_lat, lse = dsa.sparse_mla_fwd(qt, rows, i32(clean), qs, kl, T, scale)
    dkv = torch.zeros((B, T, 576), dtype=torch.float32, device="cuda")
    ws = bwd_workspace(dsa, path, B, T, T, H, k)
    dq = dsa.sparse_mla_bwd(qt, rows, i32(idx), qs, kl, T, o_lat, lse, dOt, dkv, scale, workspace=ws)
    code, where, detail = dsa.read_device_status(ws)
    assert code == dsa.DSA_ERR_BAD_INDEX and detail == 77
    rdq, rdkv = oracle.sparse_mla_bwd(q, kv, clean, q_start, kv_len, scale, dO)
    _check(dq.cpu().numpy(), rdq, "dq")
    _check(dkv.cpu().numpy(), rdkv, "dkv")


def test_bwd_with_sink(dsa):
    """The backward of the learnable-sink forward: the same kernels, fed the sink
    forward's o_lat and lse (the sink is in the denominator; it has no value and
    depends on neither q nor the latent rows), against the oracle with the sink."""
    B, T, H, k = 1, 200, 96, 64
    seed = 151
    q = normal_bf16(seed, "q_lat", (B, T, H, 576))
    kv = normal_bf16(seed, "kv", (B, T, 576))
    dO = normal_bf16(seed, "w", (B, T, H, 512))
    idx = _indices(seed, B, T, 0, k)
    sink = np.random.default_rng(seed).normal(0.0, 2.0, H).astype(np.float32)
    sink[0], sink[1] = -np.inf, 40.0
    q_start, kv_len = np.zeros(B, np.int32), np.full(B, T, np.int32)
    scale = 1.0 / np.sqrt(192.0)
    rows = dsa.Rows(bf(kv))
    qt, dOt, it, qs, kl = bf(q), bf(dO), i32(idx), i32(q_start), i32(kv_len)
    o_lat, lse = dsa.sparse_mla_fwd(qt, rows, it, qs, kl, T, scale,
                                    sink=torch.from_numpy(sink).cuda())
    dkv = torch.zeros((B, T, 576), dtype=torch.float32, device="cuda")
    dq = dsa.sparse_mla_bwd(qt, rows, it, qs, kl, T, o_lat, lse, dOt, dkv, scale)
    torch.cuda.synchronize()
    rdq, rdkv = oracle.sparse_mla_bwd(q, kv, idx, q_start, kv_len, scale, dO,
                                      sink=sink.astype(np.float64))
    _check(dq.cpu().numpy(), rdq, "dq (sink)")
    _check(dkv.cpu().numpy(), rdkv, "dkv (sink)")
