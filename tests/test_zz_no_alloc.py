"""sparse_mla_fwd_noalloc: the allocation-free variant of sparse_mla_fwd.

Some callers cannot allocate device memory where they run attention (a server
that gives all device memory to its own pool at start-up, a plugin interface
with no scratch hook).  For them the library keeps the split-K scratch in a
fixed array of its own.  This file is collected last on purpose, so a run that
stops at the first failure has already run every other test.  It must pass on
its own in a fresh process as well as after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import bf, check_mla_rows, i32, to_u16
from parity import check_close, check_lse
from workloads import (Config, bf16_to_f32, from_pages, normal_bf16, page_table, prefill_queries,
                       to_pages)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_serving_gb300 as m
    lib = m.lib
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.sparse_mla_fwd_noalloc.argtypes = [P, ctypes.POINTER(m._Rows), P, P, P, I, I, I, I, I,
                                           ctypes.c_float, P, P, P, P]
    lib.sparse_mla_fwd_noalloc.restype = I
    return m


def _decode_case(seed, B=6, topk=512):
    cfg = Config("noalloc", B=B, T=1, topk=topk, H_I=64, D_I=128, H=96, hid=1024, paged=True,
                 decode=True, L_min=200, L_max=2500, seed=seed)
    rng = np.random.default_rng(seed)
    lens = rng.integers(cfg.L_min, cfg.L_max + 1, size=B).astype(np.int32)
    bt, npages = page_table(seed, lens)
    S = int(lens.max())
    kv_log = normal_bf16(seed, "kv", (B, S, 576))
    kv_pool = to_pages(kv_log, lens, bt, npages)
    q = prefill_queries(Config(**{**cfg.__dict__, "T": 1}), 0, 1)
    idx = np.full((B, 1, topk), -1, np.int32)
    for b in range(B):
        n = min(int(lens[b]), topk)
        idx[b, 0, :n] = rng.choice(int(lens[b]), n, replace=False)
    return cfg, q["q_lat"], kv_pool, bt, lens, idx, S


def _noalloc(dsa, q_lat, rows, idx, qs, kl, S, scale, status=None):
    B, Tq, H, _ = q_lat.shape
    o = torch.empty((B, Tq, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Tq, H), dtype=torch.float32, device="cuda")
    r = rows.c()
    rc = dsa.lib.sparse_mla_fwd_noalloc(
        q_lat.data_ptr(), ctypes.byref(r), idx.data_ptr(), qs.data_ptr(), kl.data_ptr(), B, Tq,
        H, idx.shape[-1], S, ctypes.c_float(scale), o.data_ptr(), lse.data_ptr(),
        None if status is None else status.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, o, lse


def _check_oracle(o, l, q_lat, kv_pool, bt, lens, idx, scale, what):
    """Every request of the decode case against the float64 oracle, each over its
    own logical rows read back from the page pool."""
    for b in range(len(lens)):
        L = int(lens[b])
        kv_log = from_pages(kv_pool, bt, b, L)[None]
        one = lambda a: a[b:b + 1]
        check_mla_rows(one(to_u16(o)), one(l.cpu().numpy()), one(q_lat), kv_log, one(idx),
                       one(lens - 1), one(lens), scale, np.array([0]), f"{what} req {b}")


def test_noalloc_matches_workspace_entry_point_twice(dsa):
    for call, seed in enumerate((21, 22)):  # two calls in a row, different inputs
        cfg, q_lat, kv_pool, bt, lens, idx, S = _decode_case(seed)
        qd, kvr = bf(q_lat), dsa.Rows(bf(kv_pool), i32(bt))
        ix, qs, kl = i32(idx), i32(lens - 1), i32(lens)
        o_ref, l_ref = dsa.sparse_mla_fwd(qd, kvr, ix, qs, kl, S, cfg.scale)
        status = torch.zeros(3, dtype=torch.int32, device="cuda")
        rc, o, l = _noalloc(dsa, qd, kvr, ix, qs, kl, S, cfg.scale, status)
        assert rc == dsa.DSA_OK, dsa.status_string(rc)
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        check_close(bf16_to_f32(to_u16(o)), bf16_to_f32(to_u16(o_ref)), f"call {call} o_lat")
        check_lse(l.cpu().numpy(), l_ref.cpu().numpy(), f"call {call} lse")
        # and against the oracle itself, not only against the other entry point
        _check_oracle(o, l, q_lat, kv_pool, bt, lens, idx, cfg.scale, f"call {call}")


def test_noalloc_without_status_pointer(dsa):
    """device_status = NULL: errors go to the array's own header, which the call
    clears first; the output must still match the workspace entry point."""
    cfg, q_lat, kv_pool, bt, lens, idx, S = _decode_case(23, B=3)
    qd, kvr = bf(q_lat), dsa.Rows(bf(kv_pool), i32(bt))
    ix, qs, kl = i32(idx), i32(lens - 1), i32(lens)
    o_ref, l_ref = dsa.sparse_mla_fwd(qd, kvr, ix, qs, kl, S, cfg.scale)
    for _ in range(2):
        rc, o, l = _noalloc(dsa, qd, kvr, ix, qs, kl, S, cfg.scale, None)
        assert rc == dsa.DSA_OK, dsa.status_string(rc)
        torch.cuda.synchronize()
        check_close(bf16_to_f32(to_u16(o)), bf16_to_f32(to_u16(o_ref)), "no status o_lat")
        check_lse(l.cpu().numpy(), l_ref.cpu().numpy(), "no status lse")


def test_noalloc_unsplit_prefill(dsa):
    """B*Tq at or above the SM count: no split, so no scratch is used at all."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T, topk = sms + 37, 64
    cfg = Config("noalloc_pf", B=1, T=T, topk=topk, H_I=4, D_I=64, H=8, hid=1024, seed=31)
    q = prefill_queries(cfg, 0, T)
    kv = normal_bf16(cfg.seed, "kv", (1, T, 576))
    rng = np.random.default_rng(31)
    idx = np.full((1, T, topk), -1, np.int32)
    for t in range(T):
        n = min(t + 1, topk)
        idx[0, t, :n] = rng.choice(t + 1, n, replace=False)
    qd, kvr = bf(q["q_lat"]), dsa.Rows(bf(kv))
    ix, qs, kl = i32(idx), i32([0]), i32([T])
    o_ref, l_ref = dsa.sparse_mla_fwd(qd, kvr, ix, qs, kl, T, cfg.scale)
    status = torch.zeros(3, dtype=torch.int32, device="cuda")
    rc, o, l = _noalloc(dsa, qd, kvr, ix, qs, kl, T, cfg.scale, status)
    assert rc == dsa.DSA_OK, dsa.status_string(rc)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    check_close(bf16_to_f32(to_u16(o)), bf16_to_f32(to_u16(o_ref)), "unsplit o_lat")
    check_lse(l.cpu().numpy(), l_ref.cpu().numpy(), "unsplit lse")
    rows = np.array([0, 1, 63, 64, T // 2, T - 1])
    check_mla_rows(to_u16(o), l.cpu().numpy(), q["q_lat"], kv, idx, np.array([0]),
                   np.array([T]), cfg.scale, rows, "unsplit")


def test_noalloc_bad_index_recorded(dsa):
    """A non-causal entry is flagged in the caller's status and left out."""
    cfg, q_lat, kv_pool, bt, lens, idx, S = _decode_case(24, B=2)
    bad = idx.copy()
    bad[1, 0, 5] = int(lens[1]) + 3          # beyond the query position
    qd, kvr = bf(q_lat), dsa.Rows(bf(kv_pool), i32(bt))
    qs, kl = i32(lens - 1), i32(lens)
    status = torch.zeros(3, dtype=torch.int32, device="cuda")
    rc, o, l = _noalloc(dsa, qd, kvr, i32(bad), qs, kl, S, cfg.scale, status)
    assert rc == dsa.DSA_OK, dsa.status_string(rc)
    torch.cuda.synchronize()
    assert int(status[0]) == dsa.DSA_ERR_BAD_INDEX
    kept = bad.copy()
    kept[1, 0, 5] = -1
    _check_oracle(o, l, q_lat, kv_pool, bt, lens, kept, cfg.scale, "bad index")
