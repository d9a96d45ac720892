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
    ws = dsa.new_workspace(1 << 20)
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
    check_mla_rows(ol, lse.cpu().numpy(), d["q_lat"], d["kv"], gi, d["q_start"], d["kv_len"],
                   cfg.scale, rows, name)
    check_gate_rows(to_u16(out), g["x"], g["W_g"], ol.reshape(N, cfg.H, 512), g["W_uv"],
                    rows[:12], name)


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
    for b in (0, 17, 63):
        L = int(d["kv_len"][b])
        k_log = from_pages(d["k_pool"], d["block_table"], b, L)[None]
        kv_log = from_pages(d["kv_pool"], d["block_table"], b, L)[None]
        one = lambda a: a[b:b + 1]
        check_indexer_rows(one(gi), one(d["q_idx"]), one(d["w"]), k_log, one(d["q_start"]),
                           one(d["kv_len"]), cfg.topk, np.array([0]), f"decode req {b}")
        check_mla_rows(one(ol), one(ls), one(d["q_lat"]), kv_log, one(gi), one(d["q_start"]),
                       one(d["kv_len"]), cfg.scale, np.array([0]), f"decode req {b}")
