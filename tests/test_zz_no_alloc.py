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

from gpu_helpers import bf, i32, to_u16
from parity import check_close, check_lse
from workloads import Config, bf16_to_f32, normal_bf16, page_table, prefill_queries, to_pages

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
