"""GPU parity of dsa_cache_append (indexer-key LayerNorm + cache append) against
the oracle: the latent rows bit for bit, the keys within BF16 rounding of the
float64 LayerNorm, every other cache row untouched."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bf, i32, to_u16
from parity import check_bf16_of, layernorm_delta
from workloads import append_inputs, page_table

pytestmark = pytest.mark.gpu

EPS = 1e-5


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_serving_gb300 as m
    return m


def _sentinel(shape, seed):
    return np.random.default_rng(seed).integers(0, 0x7F7F, shape, dtype=np.uint16)


def _run(dsa, inp, q_start, k_cache, kv_cache, bt=None):
    kc_t, vc_t = bf(k_cache), bf(kv_cache)
    bt_t = None if bt is None else i32(bt)
    ws = dsa.dsa_cache_append(torch.from_numpy(inp["k_pre"]).cuda(), bf(inp["kv_new"]),
                              dsa.Rows(kc_t, bt_t), dsa.Rows(vc_t, bt_t), i32(q_start), EPS)
    code, where, detail = dsa.read_device_status(ws)
    return to_u16(kc_t), to_u16(vc_t), code


def _check(inp, q_start, k_cache, kv_cache, gk, gv, bt=None, what=""):
    ek, ev, k_ln = oracle.cache_append(inp["k_pre"], inp["kv_new"], q_start, EPS, k_cache,
                                       kv_cache, bt, bt)
    np.testing.assert_array_equal(gv, ev, err_msg=f"{what}: latent rows")
    # key caches: equal everywhere except the written rows, which follow the BF16 rule
    B, Tq, D = inp["k_pre"].shape
    written = np.zeros(ek.shape[:2], bool)
    for b in range(B):
        for i in range(Tq):
            pos = int(q_start[b]) + i
            if bt is None:
                written[b, pos] = True
            else:
                written[bt[b, pos // 64], pos % 64] = True
    np.testing.assert_array_equal(gk[~written], ek[~written], err_msg=f"{what}: untouched key rows")
    # oracle float64 values (and their FP32 error allowance) in cache order
    delta_all = layernorm_delta(inp["k_pre"], k_ln, EPS)
    v = np.zeros(ek.shape, np.float64)
    dl = np.zeros(ek.shape, np.float64)
    for b in range(B):
        for i in range(Tq):
            pos = int(q_start[b]) + i
            idx = (b, pos) if bt is None else (bt[b, pos // 64], pos % 64)
            v[idx], dl[idx] = k_ln[b, i], delta_all[b, i]
    return check_bf16_of(gk[written], v[written], dl[written], f"{what}: keys")


def test_append_decode_paged(dsa):
    """Decode: one new token per request at position L-1, paged caches."""
    lens = np.array([1, 64, 65, 300, 2049], np.int32)
    B, D = len(lens), 128
    bt, npages = page_table(41, lens)
    inp = append_inputs(41, B, 1, D)
    k_pool, kv_pool = _sentinel((npages, 64, D), 1), _sentinel((npages, 64, 576), 2)
    q_start = lens - 1
    gk, gv, code = _run(dsa, inp, q_start, k_pool, kv_pool, bt)
    assert code == dsa.DSA_OK
    _check(inp, q_start, k_pool, kv_pool, gk, gv, bt, "decode paged")


def test_append_prefill_chunk_contiguous(dsa):
    """A prefill chunk of 300 tokens per sequence into contiguous caches (D_I = 64)."""
    B, Tq, D, S = 2, 300, 64, 700
    inp = append_inputs(42, B, Tq, D)
    k_c, kv_c = _sentinel((B, S, D), 3), _sentinel((B, S, 576), 4)
    q_start = np.array([0, 377], np.int32)
    gk, gv, code = _run(dsa, inp, q_start, k_c, kv_c)
    assert code == dsa.DSA_OK
    _check(inp, q_start, k_c, kv_c, gk, gv, None, "chunk contiguous")


def test_append_full_chunk_paged(dsa):
    """An 8,192-token chunk (the long-context chunk size) over a paged cache."""
    B, Tq, D = 1, 8192, 128
    lens = np.array([3 * 8192], np.int32)
    bt, npages = page_table(43, lens)
    inp = append_inputs(43, B, Tq, D)
    k_pool, kv_pool = _sentinel((npages, 64, D), 5), _sentinel((npages, 64, 576), 6)
    q_start = np.array([8192], np.int32)
    gk, gv, code = _run(dsa, inp, q_start, k_pool, kv_pool, bt)
    assert code == dsa.DSA_OK
    near = _check(inp, q_start, k_pool, kv_pool, gk, gv, bt, "8192 chunk")
    assert near < 0.01 * Tq * D, near  # midpoint cases are rare


def test_append_bad_page_is_flagged_and_skipped(dsa):
    """A block-table entry outside the pool: that row is not written, the others are,
    and the status word reports DSA_ERR_BAD_INDEX."""
    lens = np.array([70, 130], np.int32)
    bt, npages = page_table(44, lens)
    bt = bt.copy()
    bt[1, 2] = npages + 5          # page of position 129 of sequence 1
    inp = append_inputs(44, 2, 1, 128)
    k_pool, kv_pool = _sentinel((npages, 64, 128), 7), _sentinel((npages, 64, 576), 8)
    q_start = lens - 1
    gk, gv, code = _run(dsa, inp, q_start, k_pool, kv_pool, bt)
    assert code == dsa.DSA_ERR_BAD_INDEX
    v = oracle.layernorm(inp["k_pre"][0, 0], EPS)
    check_bf16_of(gk[bt[0, 1], 5], v, layernorm_delta(inp["k_pre"][0, 0], v, EPS),
                  "bad-page call, good row")
    np.testing.assert_array_equal(gv[bt[0, 1], 5], inp["kv_new"][0, 0])
    np.testing.assert_array_equal(gk, np.where(np.arange(npages)[:, None, None] == bt[0, 1], gk, k_pool))
