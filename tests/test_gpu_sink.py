"""GPU parity of sparse_mla_fwd_sink (learnable attention sink, "Kimi K3.1 Pro"
archdiff blueprint, "Output gate + sink") against the oracle: prefill (one CTA
per query, sink applied in the epilogue) and decode (split-K, sink applied once
in the combine), a sink of -inf reproducing sparse_mla_fwd bit for bit, and a
query with no valid entry."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bf, check_mla_rows, i32, to_u16
from workloads import CONFIGS, Config, normal_bf16, page_table, prefill, prefill_queries, to_pages

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_serving_gb300 as m
    return m


def _sinks(H, seed):
    s = np.random.default_rng(seed).normal(0.0, 2.0, H)
    s[0] = -np.inf        # this head behaves as without a sink
    s[1] = 40.0           # this head puts nearly all weight on the sink
    return s.astype(np.float32)


def _oracle_indices(d, cfg, dsa):
    qs, kl = i32(d["q_start"]), i32(d["kv_len"])
    idx = dsa.dsa_indexer_topk(bf(d["q_idx"]), bf(d["w"]), dsa.Rows(bf(d["k_idx"])), qs, kl,
                               cfg.topk, cfg.T)
    return idx, qs, kl


@pytest.mark.parametrize("name", ["tiny", "sink96"])
def test_sink_prefill(dsa, name):
    cfg = CONFIGS["tiny"] if name == "tiny" else Config("sink96", B=1, T=700, topk=256, H_I=64,
                                                        D_I=128, H=96, hid=1024, seed=51)
    d = prefill(cfg)
    idx, qs, kl = _oracle_indices(d, cfg, dsa)
    sink = _sinks(cfg.H, 52)
    o, lse = dsa.sparse_mla_fwd(bf(d["q_lat"]), dsa.Rows(bf(d["kv"])), idx, qs, kl, cfg.T,
                                cfg.scale, sink=torch.from_numpy(sink).cuda())
    torch.cuda.synchronize()
    rows = np.unique(np.r_[0, 1, 5, np.linspace(0, cfg.T - 1, 12).astype(int)])
    check_mla_rows(to_u16(o), lse.cpu().numpy(), d["q_lat"], d["kv"], idx.cpu().numpy(),
                   d["q_start"], d["kv_len"], cfg.scale, rows, f"{name} sink",
                   sink=sink.astype(np.float64))


def test_sink_minus_infinity_is_bitwise_no_sink(dsa):
    cfg = CONFIGS["tiny"]
    d = prefill(cfg)
    idx, qs, kl = _oracle_indices(d, cfg, dsa)
    q, kv = bf(d["q_lat"]), dsa.Rows(bf(d["kv"]))
    o0, l0 = dsa.sparse_mla_fwd(q, kv, idx, qs, kl, cfg.T, cfg.scale)
    o1, l1 = dsa.sparse_mla_fwd(q, kv, idx, qs, kl, cfg.T, cfg.scale,
                                sink=torch.full((cfg.H,), float("-inf"), device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0, l1)


def test_sink_decode_split(dsa):
    """Decode over paged caches: the split-K path merges partials and adds the sink
    once in the combine."""
    cfg = Config("sink-dec", B=4, T=1, topk=512, H_I=64, D_I=128, H=96, hid=1024, paged=True,
                 decode=True, L_min=600, L_max=3000, seed=53)
    lens = np.array([700, 1500, 2999, 3000], np.int32)
    bt, npages = page_table(cfg.seed, lens)
    S = int(lens.max())
    k_log = normal_bf16(cfg.seed, "k_idx", (cfg.B, S, cfg.D_I))
    kv_log = normal_bf16(cfg.seed, "kv", (cfg.B, S, 576))
    q = prefill_queries(Config(**{**cfg.__dict__, "T": 1}), 0, 1)
    qs, kl = lens - 1, lens
    btt = i32(bt)
    idx = dsa.dsa_indexer_topk(bf(q["q_idx"]), bf(q["w"]),
                               dsa.Rows(bf(to_pages(k_log, lens, bt, npages)), btt), i32(qs),
                               i32(kl), cfg.topk, S)
    sink = _sinks(cfg.H, 54)
    o, lse = dsa.sparse_mla_fwd(bf(q["q_lat"]), dsa.Rows(bf(to_pages(kv_log, lens, bt, npages)), btt),
                                idx, i32(qs), i32(kl), S, cfg.scale, sink=torch.from_numpy(sink).cuda())
    torch.cuda.synchronize()
    check_mla_rows(to_u16(o), lse.cpu().numpy(), q["q_lat"], kv_log, idx.cpu().numpy(), qs, kl,
                   cfg.scale, np.arange(cfg.B), "decode sink", sink=sink.astype(np.float64))


def test_sink_empty_list(dsa):
    """Every entry -1: o = 0 and lse = sink (prefill and split decode paths)."""
    for T, B in ((200, 1), (1, 3)):   # one CTA per query (200 >= SMs), and split-K
        H = 96
        q = normal_bf16(55, "q_lat", (B, T, H, 576))
        kv = normal_bf16(55, "kv", (B, max(T, 8), 576))
        idx = torch.full((B, T, 64), -1, dtype=torch.int32, device="cuda")
        qs = i32(np.full(B, 0 if T > 1 else 7, np.int32))
        kl = i32(np.full(B, max(T, 8), np.int32))
        sink = _sinks(H, 56)
        o, lse = dsa.sparse_mla_fwd(bf(q), dsa.Rows(bf(kv)), idx, qs, kl, max(T, 8), 0.1,
                                    sink=torch.from_numpy(sink).cuda())
        torch.cuda.synchronize()
        assert torch.count_nonzero(o.view(torch.int16)).item() == 0
        want = np.broadcast_to(sink, (B, T, H))
        np.testing.assert_allclose(lse.cpu().numpy(), want, rtol=1e-6, atol=0)
