"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Small shapes that still span several tiles and a ragged
tail, plus the edge cases of the method."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bf, check_gate_rows, check_indexer_rows, check_mla_rows, i32, to_u16
from parity import check_close
from workloads import (CONFIGS, Config, bf16_to_f32, gate_inputs, normal_bf16, page_table, prefill,
                       prefill_keys, prefill_queries, to_pages)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_serving_gb300 as m
    return m


def _run_prefill(dsa, d, cfg, with_gate=True):
    B, T = cfg.B, cfg.T
    q_idx, w, k_idx = bf(d["q_idx"]), bf(d["w"]), bf(d["k_idx"])
    q_lat, kv = bf(d["q_lat"]), bf(d["kv"])
    qs, kl = i32(d["q_start"]), i32(d["kv_len"])
    idx = dsa.dsa_indexer_topk(q_idx, w, dsa.Rows(k_idx), qs, kl, cfg.topk, T)
    o_lat, lse = dsa.sparse_mla_fwd(q_lat, dsa.Rows(kv), idx, qs, kl, T, cfg.scale)
    out = None
    g = None
    if with_gate:
        g = gate_inputs(cfg, B * T)
        out = dsa.mla_gate_apply(bf(g["x"]), bf(g["W_g"]), o_lat.view(B * T, cfg.H, 512),
                                 bf(g["W_uv"]))
    torch.cuda.synchronize()
    res = {"idx": idx.cpu().numpy(), "o_lat": to_u16(o_lat), "lse": lse.cpu().numpy()}
    if with_gate:
        res["out"] = to_u16(out)
        res["gate"] = g
    return res


def test_tiny_full_pipeline(dsa):
    cfg = CONFIGS["tiny"]
    d = prefill(cfg)
    r = _run_prefill(dsa, d, cfg)
    rows = np.arange(cfg.B * cfg.T)
    check_indexer_rows(r["idx"], d["q_idx"], d["w"], d["k_idx"], d["q_start"], d["kv_len"],
                       cfg.topk, rows, "tiny indexer")
    check_mla_rows(r["o_lat"], r["lse"], d["q_lat"], d["kv"], r["idx"], d["q_start"], d["kv_len"],
                   cfg.scale, rows, "tiny mla")
    g = r["gate"]
    check_gate_rows(r["out"], g["x"], g["W_g"], r["o_lat"].reshape(cfg.B * cfg.T, cfg.H, 512),
                    g["W_uv"], rows, "tiny")


def test_tiny128_keeps_every_key_and_equals_dense(dsa):
    """T <= k: every query keeps all its causal keys, so sparse MLA equals dense MLA."""
    cfg = CONFIGS["tiny128"]
    d = prefill(cfg)
    r = _run_prefill(dsa, d, cfg, with_gate=False)
    for t in range(cfg.T):
        row = r["idx"][0, t]
        assert sorted(row[:t + 1].tolist()) == list(range(t + 1))
        assert np.all(row[t + 1:] == -1)
    o_ref, lse_ref = oracle.dense_mla(d["q_lat"], d["kv"], d["q_start"], d["kv_len"], cfg.scale)
    check_close(bf16_to_f32(r["o_lat"][0]), o_ref, "tiny128 vs dense")


def test_sparse_mla_on_oracle_indices(dsa):
    """Sparse MLA alone, fed the oracle's index sets (independent of the GPU indexer)."""
    cfg = CONFIGS["tiny"]
    d = prefill(cfg)
    rows = np.arange(cfg.T)
    o_idx, _, _, _ = oracle.indexer_topk(d["q_idx"], d["w"], d["k_idx"], d["q_start"], d["kv_len"],
                                         cfg.topk, rows)
    idx = o_idx.reshape(1, cfg.T, cfg.topk)
    o_lat, lse = dsa.sparse_mla_fwd(bf(d["q_lat"]), dsa.Rows(bf(d["kv"])), i32(idx),
                                    i32(d["q_start"]), i32(d["kv_len"]), cfg.T, cfg.scale)
    check_mla_rows(to_u16(o_lat), lse.cpu().numpy(), d["q_lat"], d["kv"], idx, d["q_start"],
                   d["kv_len"], cfg.scale, rows, "mla/oracle-idx")


@pytest.mark.parametrize("T,topk,H_I,D_I,H", [(300, 64, 64, 128, 96), (777, 256, 4, 64, 8),
                                               (1000, 512, 64, 128, 96)])
def test_ragged_prefill(dsa, T, topk, H_I, D_I, H):
    """Sequence lengths that are not multiples of any tile, several sequences."""
    cfg = Config("ragged", B=2, T=T, topk=topk, H_I=H_I, D_I=D_I, H=H, hid=1024, seed=77)
    d = prefill(cfg)
    r = _run_prefill(dsa, d, cfg)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, T - 1, T, 2 * T - 1, topk - 1, topk, T + topk],
                                     rng.integers(0, 2 * T, 24)]))
    rows = rows[rows < 2 * T]
    check_indexer_rows(r["idx"], d["q_idx"], d["w"], d["k_idx"], d["q_start"], d["kv_len"], topk,
                       rows, "ragged indexer")
    check_mla_rows(r["o_lat"], r["lse"], d["q_lat"], d["kv"], r["idx"], d["q_start"], d["kv_len"],
                   cfg.scale, rows, "ragged mla")
    g = r["gate"]
    check_gate_rows(r["out"], g["x"], g["W_g"], r["o_lat"].reshape(2 * T, H, 512), g["W_uv"], rows,
                    "ragged")


def test_sparse_mla_edge_index_lists(dsa):
    """Empty index lists (all -1) give o = 0 and lse = -inf; -1 entries scattered
    anywhere are skipped; the order of the entries does not matter."""
    cfg = Config("edge", B=1, T=200, topk=96, H_I=4, D_I=64, H=96, hid=1024, seed=12)
    d = prefill(cfg)
    T, k = cfg.T, cfg.topk
    rng = np.random.default_rng(3)
    idx = np.full((1, T, k), -1, np.int32)
    for t in range(T):
        mode = t % 4
        if mode == 0:
            continue  # empty
        n = min(t + 1, k) if mode == 1 else int(rng.integers(1, min(t + 1, k) + 1))
        sel = rng.choice(t + 1, n, replace=False)
        pos = rng.choice(k, n, replace=False)
        idx[0, t, pos] = sel
    o_lat, lse = dsa.sparse_mla_fwd(bf(d["q_lat"]), dsa.Rows(bf(d["kv"])), i32(idx),
                                    i32(d["q_start"]), i32(d["kv_len"]), T, cfg.scale)
    rows = np.arange(T)
    check_mla_rows(to_u16(o_lat), lse.cpu().numpy(), d["q_lat"], d["kv"], idx, d["q_start"],
                   d["kv_len"], cfg.scale, rows, "edge")
    og = to_u16(o_lat)[0]
    assert np.all(og[0::4] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[0, 0::4]))


def test_bad_index_is_flagged_and_skipped(dsa):
    """A non-causal index is reported through the device status word and skipped."""
    cfg = Config("bad", B=1, T=64, topk=16, H_I=4, D_I=64, H=8, hid=1024, seed=13)
    d = prefill(cfg)
    T, k = cfg.T, cfg.topk
    idx = np.full((1, T, k), -1, np.int32)
    for t in range(T):
        idx[0, t, :min(t + 1, k)] = np.arange(min(t + 1, k))
    idx[0, 5, 7] = 40  # not causal for the query at position 5
    ws = dsa.new_workspace(dsa.workspace_bytes(dsa.OP_SPARSE_MLA, 1, T, T, cfg.H, k))
    o_lat, lse = dsa.sparse_mla_fwd(bf(d["q_lat"]), dsa.Rows(bf(d["kv"])), i32(idx),
                                    i32(d["q_start"]), i32(d["kv_len"]), T, cfg.scale,
                                    workspace=ws)
    code, where, detail = dsa.read_device_status(ws)
    assert code == dsa.DSA_ERR_BAD_INDEX and detail == 40
    assert dsa.read_device_status(ws)[0] == dsa.DSA_OK  # reading clears it
    ref_idx = idx.copy()
    ref_idx[0, 5, 7] = -1
    check_mla_rows(to_u16(o_lat), lse.cpu().numpy(), d["q_lat"], d["kv"], ref_idx, d["q_start"],
                   d["kv_len"], cfg.scale, np.arange(T), "bad-index")


def test_chunked_prefill_paged_small(dsa):
    """A chunk of queries against a paged cache with permuted pages (q_start > 0)."""
    cfg = Config("chunk-small", B=1, T=1024, topk=256, H_I=64, D_I=128, H=96, hid=1024,
                 chunk=256, paged=True, seed=14)
    keys = prefill_keys(cfg)
    lens = np.array([cfg.T])
    bt, npages = page_table(cfg.seed, lens, spare=3)
    k_pool = to_pages(keys["k_idx"], lens, bt, npages)
    kv_pool = to_pages(keys["kv"], lens, bt, npages)
    for c in (1, 3):
        q0 = c * cfg.chunk
        q = prefill_queries(cfg, q0, cfg.chunk)
        qs, kl = np.array([q0], np.int32), np.array([q0 + cfg.chunk], np.int32)
        idx = dsa.dsa_indexer_topk(bf(q["q_idx"]), bf(q["w"]), dsa.Rows(bf(k_pool), i32(bt)),
                                   i32(qs), i32(kl), cfg.topk, cfg.T)
        o_lat, lse = dsa.sparse_mla_fwd(bf(q["q_lat"]), dsa.Rows(bf(kv_pool), i32(bt)), idx,
                                        i32(qs), i32(kl), cfg.T, cfg.scale)
        torch.cuda.synchronize()
        gi = idx.cpu().numpy()
        rows = np.array([0, 1, 100, 200, cfg.chunk - 1])
        check_indexer_rows(gi, q["q_idx"], q["w"], keys["k_idx"], qs, kl, cfg.topk, rows,
                           f"chunk{c} indexer")
        check_mla_rows(to_u16(o_lat), lse.cpu().numpy(), q["q_lat"], keys["kv"], gi, qs, kl,
                       cfg.scale, rows, f"chunk{c} mla")


def test_decode_small_paged(dsa):
    """Decode: one query per request at position L-1 over paged caches."""
    cfg = Config("decode-small", B=5, T=1, topk=512, H_I=64, D_I=128, H=96, hid=1024, paged=True,
                 decode=True, L_min=300, L_max=3000, seed=15)
    rng = np.random.default_rng(cfg.seed)
    lens = rng.integers(cfg.L_min, cfg.L_max + 1, size=cfg.B).astype(np.int32)
    lens[0] = 100  # fewer keys than k
    bt, npages = page_table(cfg.seed, lens)
    S = int(lens.max())
    k_log = normal_bf16(cfg.seed, "k_idx", (cfg.B, S, cfg.D_I))
    kv_log = normal_bf16(cfg.seed, "kv", (cfg.B, S, 576))
    k_pool = to_pages(k_log, lens, bt, npages)
    kv_pool = to_pages(kv_log, lens, bt, npages)
    q = prefill_queries(Config(**{**cfg.__dict__, "T": 1}), 0, 1)
    qs, kl = lens - 1, lens
    idx = dsa.dsa_indexer_topk(bf(q["q_idx"]), bf(q["w"]), dsa.Rows(bf(k_pool), i32(bt)), i32(qs),
                               i32(kl), cfg.topk, S)
    o_lat, lse = dsa.sparse_mla_fwd(bf(q["q_lat"]), dsa.Rows(bf(kv_pool), i32(bt)), idx, i32(qs),
                                    i32(kl), S, cfg.scale)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    rows = np.arange(cfg.B)
    check_indexer_rows(gi, q["q_idx"], q["w"], k_log, qs, kl, cfg.topk, rows, "decode indexer")
    check_mla_rows(to_u16(o_lat), lse.cpu().numpy(), q["q_lat"], kv_log, gi, qs, kl, cfg.scale,
                   rows, "decode mla")


def test_decode_select_ties_and_equal_scores(dsa):
    """Decode top-k on score rows with heavy ties: request 0 draws its keys from
    two distinct rows (about 10,000 keys share the k-th score, more than the
    select kernel keeps in shared memory), request 1 has one key row repeated
    (every score equal), request 2 is ordinary.  Any choice among tied keys is
    valid; the near-tie rule checks the sets."""
    cfg = Config("decode-ties", B=3, T=1, topk=2048, H_I=64, D_I=128, H=96, hid=1024, seed=23)
    lens = np.array([20000, 20000, 5000], np.int32)
    S = int(lens.max())
    k_log = normal_bf16(cfg.seed, "k_idx", (cfg.B, S, cfg.D_I))
    rng = np.random.default_rng([cfg.seed, 99])
    pick = rng.integers(0, 2, size=S)
    k_log[0] = k_log[0, pick]          # two distinct key rows
    k_log[1] = k_log[1, :1]            # one key row everywhere
    q = prefill_queries(Config(**{**cfg.__dict__, "T": 1}), 0, 1)
    qs, kl = lens - 1, lens
    idx = dsa.dsa_indexer_topk(bf(q["q_idx"]), bf(q["w"]), dsa.Rows(bf(k_log)), i32(qs), i32(kl),
                               cfg.topk, S)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    check_indexer_rows(gi, q["q_idx"], q["w"], k_log, qs, kl, cfg.topk, np.arange(cfg.B),
                       "decode ties")


def test_gate_zero_weight_gives_half(dsa):
    """W_g = 0: out = 0.5 * (W_uv_h . o_lat_h) exactly up to BF16 rounding."""
    cfg = CONFIGS["tiny"]
    N = 200
    g = gate_inputs(cfg, N)
    o_lat = normal_bf16(99, "q_lat", (N, cfg.H, 512), std=0.1)
    Wg0 = np.zeros_like(g["W_g"])
    out = dsa.mla_gate_apply(bf(g["x"]), bf(Wg0), bf(o_lat), bf(g["W_uv"]))
    torch.cuda.synchronize()
    u = np.einsum("her,nhr->nhe", bf16_to_f32(g["W_uv"]).astype(np.float64),
                  bf16_to_f32(o_lat).astype(np.float64)).reshape(N, -1)
    check_close(bf16_to_f32(to_u16(out)), 0.5 * u, "gate W_g=0")
