"""GPU parity at the full sizes of the five workloads, in the launch configuration
bench.py times, checked on sampled rows the oracle computes one by one."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_helpers import bf, check_gate_rows, check_indexer_rows, check_mla_rows, i32, to_u16
from workloads import CONFIGS, chunked, decode, gate_inputs, prefill

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_serving_gb300 as m
    return m


def _sample_rows(B, T, topk, n, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, topk - 2, topk - 1, topk, T - 1]
    rows = [b * T + t for b in range(B) for t in fixed if t < T]
    rows += list(rng.integers(0, B * T, n))
    return np.unique(np.array(rows, np.int64))


@pytest.mark.parametrize("name", ["val4096", "head8192"])
def test_prefill_fullsize(dsa, name):
    cfg = CONFIGS[name]
    B, T, N = cfg.B, cfg.T, cfg.B * cfg.T
    d = prefill(cfg)
    g = gate_inputs(cfg, N)
    qs, kl = i32(d["q_start"]), i32(d["kv_len"])
    ws = dsa.new_workspace(max(dsa.workspace_bytes(op, B, T, T, h, cfg.topk) for op, h in
                               ((dsa.OP_INDEXER_TOPK, cfg.H_I), (dsa.OP_SPARSE_MLA, cfg.H))))
    idx = dsa.dsa_indexer_topk(bf(d["q_idx"]), bf(d["w"]), dsa.Rows(bf(d["k_idx"])), qs, kl,
                               cfg.topk, T, workspace=ws)
    o_lat, lse = dsa.sparse_mla_fwd(bf(d["q_lat"]), dsa.Rows(bf(d["kv"])), idx, qs, kl, T,
                                    cfg.scale, workspace=ws)
    out = dsa.mla_gate_apply(bf(g["x"]), bf(g["W_g"]), o_lat.view(N, cfg.H, 512), bf(g["W_uv"]),
                             workspace=ws)
    assert dsa.read_device_status(ws)[0] == dsa.DSA_OK
    gi = idx.cpu().numpy()
    # properties that hold for every row: counts, range, uniqueness
    valid = gi >= 0
    t_pos = np.arange(T)[None, :, None]
    assert np.array_equal(valid.sum(-1), np.minimum(np.arange(T) + 1, cfg.topk)[None].repeat(B, 0))
    assert np.all(np.where(valid, gi <= t_pos, True))
    srt = np.sort(np.where(valid, gi, -1 - np.arange(cfg.topk)[None, None]), axis=-1)
    assert np.all(np.diff(srt, axis=-1) != 0)
    rows = _sample_rows(B, T, cfg.topk, 24, 1)
    check_indexer_rows(gi, d["q_idx"], d["w"], d["k_idx"], d["q_start"], d["kv_len"], cfg.topk,
                       rows, name)
    ol = to_u16(o_lat)
    # the persistent sparse MLA kernel: CTA c takes queries c, c + P, c + 2P, ...
    # (P = SM count), and each unit's start overlaps the previous unit's tail, so
    # check the first two and the last unit of a few CTAs as well
    P = torch.cuda.get_device_properties(0).multi_processor_count
    unit_rows = []
    for c in (0, 1, P // 2, P - 1):
        last = c + P * ((N - 1 - c) // P)
        unit_rows += [c, c + P, last]
    mla_rows = np.unique(np.concatenate([rows, np.array(unit_rows, np.int64)]))
    check_mla_rows(ol, lse.cpu().numpy(), d["q_lat"], d["kv"], gi, d["q_start"], d["kv_len"],
                   cfg.scale, mla_rows, name)
    # the gate: every row of three whole 128-token tiles (first, middle, last)
    tiles = [0, (N // 128 // 2) * 128, N - 128]
    gate_rows = np.concatenate([np.arange(t0, t0 + 128) for t0 in tiles]).astype(np.int64)
    check_gate_rows(to_u16(out), g["x"], g["W_g"], ol.reshape(N, cfg.H, 512), g["W_uv"],
                    gate_rows, name)


def test_chunked_32k_fullsize(dsa):
    """Last and first chunks of the 32,768-token chunked prefill over the paged cache."""
    cfg = CONFIGS["chunk32k"]
    for c in (3, 0):
        d = chunked(cfg, c)
        qs, kl = i32(d["q_start"]), i32(d["kv_len"])
        bt = i32(d["block_table"])
        idx = dsa.dsa_indexer_topk(bf(d["q_idx"]), bf(d["w"]), dsa.Rows(bf(d["k_pool"]), bt), qs,
                                   kl, cfg.topk, cfg.T)
        o_lat, lse = dsa.sparse_mla_fwd(bf(d["q_lat"]), dsa.Rows(bf(d["kv_pool"]), bt), idx, qs,
                                        kl, cfg.T, cfg.scale)
        torch.cuda.synchronize()
        gi = idx.cpu().numpy()
        rows = _sample_rows(1, cfg.chunk, cfg.topk, 6, 2 + c)
        check_indexer_rows(gi, d["q_idx"], d["w"], d["k_logical"], d["q_start"], d["kv_len"],
                           cfg.topk, rows, f"chunk{c}")
        check_mla_rows(to_u16(o_lat), lse.cpu().numpy(), d["q_lat"], d["kv_logical"], gi,
                       d["q_start"], d["kv_len"], cfg.scale, rows, f"chunk{c}")


def test_decode64_fullsize(dsa):
    from workloads import from_pages
    cfg = CONFIGS["decode64"]
    d = decode(cfg)
    qs, kl = i32(d["q_start"]), i32(d["kv_len"])
    bt = i32(d["block_table"])
    S = int(d["kv_len"].max())
    idx = dsa.dsa_indexer_topk(bf(d["q_idx"]), bf(d["w"]), dsa.Rows(bf(d["k_pool"]), bt), qs, kl,
                               cfg.topk, S)
    o_lat, lse = dsa.sparse_mla_fwd(bf(d["q_lat"]), dsa.Rows(bf(d["kv_pool"]), bt), idx, qs, kl,
                                    S, cfg.scale)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    ol, ls = to_u16(o_lat), lse.cpu().numpy()
    # the split sparse MLA cuts the 64 x 32 list blocks into one contiguous range
    # per CTA, so each request's partials come from 3 or 4 CTAs with different
    # range boundaries: check the attention of a dozen requests spread over the
    # batch, the indexer of three
    for b in (0, 1, 2, 9, 17, 30, 31, 32, 47, 55, 62, 63):
        L = int(d["kv_len"][b])
        kv_log = from_pages(d["kv_pool"], d["block_table"], b, L)[None]
        one = lambda a: a[b:b + 1]
        if b in (0, 17, 63):
            k_log = from_pages(d["k_pool"], d["block_table"], b, L)[None]
            check_indexer_rows(one(gi), one(d["q_idx"]), one(d["w"]), k_log, one(d["q_start"]),
                               one(d["kv_len"]), cfg.topk, np.array([0]), f"decode req {b}")
        check_mla_rows(one(ol), one(ls), one(d["q_lat"]), kv_log, one(gi), one(d["q_start"]),
                       one(d["kv_len"]), cfg.scale, np.array([0]), f"decode req {b}")


def test_decode64_fp8_fullsize(dsa):
    """The FP8 indexer on the full decode64 cache, checked on three requests.  The
    checked requests' pages hold the oracle's quantisation of the seeded BF16 keys;
    the other pages hold seeded random codes and scales (their results are not
    checked), so no FP8 operand comes from the CUDA path."""
    import oracle
    from workloads import from_pages
    cfg = CONFIGS["decode64"]
    d = decode(cfg)
    S = int(d["kv_len"].max())
    npages = d["num_pages"]
    rng = np.random.default_rng(64)
    kc_pool = rng.integers(0, 0x7F, (npages, 64, 128), dtype=np.uint8)   # finite codes
    ks_pool = rng.uniform(1e-3, 1e-2, (npages, 64)).astype(np.float32)
    checked = (0, 17, 63)
    for b in checked:
        L = int(d["kv_len"][b])
        pages = d["block_table"][b, :(L + 63) // 64]
        c, sc = oracle.quant_fp8(d["k_pool"][pages])
        kc_pool[pages], ks_pool[pages] = c, sc
    qc, qsc = oracle.quant_fp8(d["q_idx"])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bt = i32(d["block_table"])
    idx = dsa.dsa_indexer_topk_fp8(dev(qc), dev(qsc), bf(d["w"]), dsa.Rows(dev(kc_pool), bt),
                                   dev(ks_pool), i32(d["q_start"]), i32(d["kv_len"]), cfg.topk, S)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    from parity import check_index_row
    for b in checked:
        L = int(d["kv_len"][b])
        kc = from_pages(kc_pool, d["block_table"], b, L)[None]
        ks = from_pages(ks_pool[..., None], d["block_table"], b, L)[None, :, 0]
        one = lambda a: a[b:b + 1]
        o_idx, kth, sc, nv = oracle.indexer_topk_fp8(one(qc), one(qsc), one(d["w"]), kc, ks,
                                                     one(d["q_start"]), one(d["kv_len"]),
                                                     cfg.topk, np.array([0]))
        check_index_row(gi[b, 0], sc[0], int(nv[0]), cfg.topk, o_idx[0], kth[0],
                        f"fp8 decode req {b}")


@pytest.mark.parametrize("path", ["tc", "warp"])
def test_bwd_fullsize_slice(dsa, path):
    """The backward on full-size index sets: the indexer and forward run on the whole
    val4096 sequence; the backward takes its last 8 queries (each with k = 2,048
    selected keys) and is checked against the float64 gradient, on the tcgen05
    kernels and on the warp-level MMA path."""
    import oracle
    from test_gpu_bwd import _check, bwd_workspace
    cfg = CONFIGS["val4096"]
    T, nq = cfg.T, 8
    d = prefill(cfg)
    qs, kl = i32(d["q_start"]), i32(d["kv_len"])
    idx = dsa.dsa_indexer_topk(bf(d["q_idx"]), bf(d["w"]), dsa.Rows(bf(d["k_idx"])), qs, kl,
                               cfg.topk, T)
    kvrows = dsa.Rows(bf(d["kv"]))
    o_lat, lse = dsa.sparse_mla_fwd(bf(d["q_lat"]), kvrows, idx, qs, kl, T, cfg.scale)
    q0 = T - nq
    sl = lambda t: t[:, q0:].contiguous()
    dO = np.random.default_rng(4096).standard_normal((1, nq, cfg.H, 512)).astype(np.float32)
    from workloads import bf16_round
    dO = bf16_round(dO)
    dkv = torch.zeros((1, T, 576), dtype=torch.float32, device="cuda")
    ws = bwd_workspace(dsa, path, 1, nq, T, cfg.H, cfg.topk)
    dq = dsa.sparse_mla_bwd(sl(bf(d["q_lat"])), kvrows, sl(idx), i32([q0]), i32([T]), T, sl(o_lat),
                            sl(lse), bf(dO), dkv, cfg.scale, workspace=ws)
    assert dsa.read_device_status(ws)[0] == dsa.DSA_OK
    gi = idx[:, q0:].cpu().numpy()
    rdq, rdkv = oracle.sparse_mla_bwd(d["q_lat"][:, q0:], d["kv"], gi, np.array([q0], np.int32),
                                      np.array([T], np.int32), cfg.scale, dO)
    _check(dq.cpu().numpy(), rdq, "dq (val4096 slice)")
    _check(dkv.cpu().numpy(), rdkv, "dkv (val4096 slice)")
