"""The C ABI library loads, exports every entry point include/dsa.h declares,
and rejects bad arguments on the host before any launch.  CPU only: no call
here reaches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_serving_gb300 as m
    return m


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s+(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_three_entry_points():
    names = declared_functions()
    for n in ("dsa_indexer_topk", "sparse_mla_fwd", "mla_gate_apply"):
        assert n in names


def test_every_declared_symbol_is_exported(dsa):
    lib = ctypes.CDLL(dsa.LIB_PATH)
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dsa.h but not exported"
    for n in dsa.EXPORTS:
        assert n in names


def test_status_strings(dsa):
    assert dsa.lib.dsa_abi_version() == 1
    for code in range(7):
        assert dsa.status_string(code) and dsa.status_string(code) != "unknown status"
    assert dsa.status_string(99) == "unknown status"


def test_workspace_bytes_has_header(dsa):
    for op in (dsa.OP_INDEXER_TOPK, dsa.OP_SPARSE_MLA, dsa.OP_GATE, dsa.OP_SPARSE_MLA_BWD):
        n = dsa.workspace_bytes(op, 2, 8192, 8192, 96, 2048)
        assert n >= 256 and n % 256 == 0


def test_workspace_bytes_prefill_indexer_and_backward(dsa):
    """The prefill indexer's candidate buffers (one slice per persistent CTA, at
    most one CTA per 4-query work item) and the tensor-core backward's p and dz
    of up to 512 queries are part of the reported size."""
    per_cta = 4 * 8192 * 8
    small = dsa.workspace_bytes(dsa.OP_INDEXER_TOPK, 1, 8, 8, 64, 2048)   # 2 work items
    assert small >= 256 + 2 * per_cta
    big = dsa.workspace_bytes(dsa.OP_INDEXER_TOPK, 2, 8192, 8192, 64, 2048)
    assert big >= 256 + 100 * per_cta          # one slice per SM (any GPU has 100+ here)
    assert big < 256 + 1024 * per_cta          # bounded by the SM count, not by the sequence
    # decode (Tq == 1) has no candidate buffers, only its score vectors
    assert dsa.workspace_bytes(dsa.OP_INDEXER_TOPK, 4, 1, 4096, 64, 2048) >= 256 + 4 * 4096 * 4
    per_q = 2 * 96 * 2048 * 2
    assert dsa.workspace_bytes(dsa.OP_SPARSE_MLA_BWD, 1, 8, 4096, 96, 2048) == 256 + 8 * per_q
    assert dsa.workspace_bytes(dsa.OP_SPARSE_MLA_BWD, 2, 8192, 8192, 96, 2048) == 256 + 512 * per_q
    # topk rounded up to a multiple of 128 entries
    assert dsa.workspace_bytes(dsa.OP_SPARSE_MLA_BWD, 1, 8, 4096, 96, 200) == 256 + 8 * 2 * 96 * 256 * 2
    # other head counts take the warp-level path: the header only
    assert dsa.workspace_bytes(dsa.OP_SPARSE_MLA_BWD, 1, 8, 4096, 8, 2048) == 256


def _rows(base=0, bt=0, stride=0, maxp=0, page=0, npages=0):
    from sparse_attention_serving_gb300 import _Rows
    return _Rows(base, stride, bt, maxp, page, npages)


def test_host_argument_checks(dsa):
    lib = dsa.lib
    P = ctypes.c_void_p
    fake = P(1 << 20)  # aligned, never dereferenced: every call below fails its host checks
    ws = P(1 << 24)
    r = _rows(base=1 << 20, stride=128)
    # null pointers
    assert lib.dsa_indexer_topk(None, fake, ctypes.byref(r), fake, fake, 1, 128, 64, 128, 128, 64,
                                fake, ws, 1 << 20, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    # unsupported indexer dims
    assert lib.dsa_indexer_topk(fake, fake, ctypes.byref(r), fake, fake, 1, 128, 32, 128, 128, 64,
                                fake, ws, 1 << 20, None) == dsa.DSA_ERR_UNSUPPORTED
    # top-k not a multiple of 4 / above 2048
    assert lib.dsa_indexer_topk(fake, fake, ctypes.byref(r), fake, fake, 1, 128, 64, 128, 128, 62,
                                fake, ws, 1 << 20, None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_indexer_topk(fake, fake, ctypes.byref(r), fake, fake, 1, 128, 64, 128, 128, 4096,
                                fake, ws, 1 << 20, None) == dsa.DSA_ERR_UNSUPPORTED
    # contiguous stride shorter than max_kv_len
    assert lib.dsa_indexer_topk(fake, fake, ctypes.byref(_rows(base=1 << 20, stride=64)), fake,
                                fake, 1, 128, 64, 128, 128, 64, fake, ws, 1 << 20,
                                None) == dsa.DSA_ERR_INVALID_ARGUMENT
    # paged store with a page size other than 64
    assert lib.dsa_indexer_topk(fake, fake,
                                ctypes.byref(_rows(base=1 << 20, bt=1 << 20, maxp=4, page=32,
                                                   npages=8)),
                                fake, fake, 1, 128, 64, 128, 128, 64, fake, ws, 1 << 20,
                                None) == dsa.DSA_ERR_UNSUPPORTED
    # workspace too small / misaligned
    assert lib.dsa_indexer_topk(fake, fake, ctypes.byref(r), fake, fake, 1, 128, 64, 128, 128, 64,
                                fake, ws, 16, None) == dsa.DSA_ERR_WORKSPACE_TOO_SMALL
    assert lib.dsa_indexer_topk(fake, fake, ctypes.byref(r), fake, fake, 1, 128, 64, 128, 128, 64,
                                fake, P((1 << 24) + 8), 1 << 20, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    # sparse MLA: unsupported heads, bad scale, misaligned q
    kvr = _rows(base=1 << 20, stride=128)
    assert lib.sparse_mla_fwd(fake, ctypes.byref(kvr), fake, fake, fake, 1, 128, 64, 128, 128,
                              ctypes.c_float(0.07), fake, None, ws, 1 << 20,
                              None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.sparse_mla_fwd(fake, ctypes.byref(kvr), fake, fake, fake, 1, 128, 96, 128, 128,
                              ctypes.c_float(-1.0), fake, None, ws, 1 << 20,
                              None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert lib.sparse_mla_fwd(P((1 << 20) + 2), ctypes.byref(kvr), fake, fake, fake, 1, 128, 96,
                              128, 128, ctypes.c_float(0.07), fake, None, ws, 1 << 20,
                              None) == dsa.DSA_ERR_INVALID_ARGUMENT
    # gate: dv other than 128, odd head count, hid not a multiple of 64
    assert lib.mla_gate_apply(fake, fake, fake, fake, 16, 1024, 8, 64, fake, ws, 1 << 20,
                              None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.mla_gate_apply(fake, fake, fake, fake, 16, 1024, 7, 128, fake, ws, 1 << 20,
                              None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.mla_gate_apply(fake, fake, fake, fake, 16, 1000, 8, 128, fake, ws, 1 << 20,
                              None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.mla_gate_apply(fake, fake, None, fake, 16, 1024, 8, 128, fake, ws, 1 << 20,
                              None) == dsa.DSA_ERR_INVALID_ARGUMENT


def test_host_argument_checks_fp8(dsa):
    lib = dsa.lib
    P = ctypes.c_void_p
    fake = P(1 << 20)
    ws = P(1 << 24)
    r = _rows(base=1 << 20, stride=128)

    def topk8(q=fake, qs=fake, ks=fake, rows=r, B=1, Tq=1, H_I=64, D_I=128, S=128, k=64):
        return lib.dsa_indexer_topk_fp8(q, qs, fake, ctypes.byref(rows), ks, fake, fake, B, Tq,
                                        H_I, D_I, S, k, fake, ws, 1 << 20, None)

    assert topk8(qs=None) == dsa.DSA_ERR_INVALID_ARGUMENT       # scales are required
    assert topk8(ks=None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert topk8(ks=P((1 << 20) + 4)) == dsa.DSA_ERR_INVALID_ARGUMENT  # key scales 16-byte aligned
    assert topk8(H_I=4, D_I=64) == dsa.DSA_ERR_UNSUPPORTED      # (64, 128) only
    # contiguous keys with a row stride that is not a multiple of 4
    assert topk8(rows=_rows(base=1 << 20, stride=130), S=128) == dsa.DSA_ERR_UNSUPPORTED
    # quantizer: D other than 64 / 128, misaligned input, negative row count
    assert lib.dsa_quant_fp8(fake, 16, 96, fake, fake, None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_quant_fp8(P((1 << 20) + 2), 16, 128, fake, fake, None) == \
        dsa.DSA_ERR_INVALID_ARGUMENT
    assert lib.dsa_quant_fp8(fake, -1, 128, fake, fake, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert lib.dsa_quant_fp8(fake, 0, 128, fake, fake, None) == dsa.DSA_OK   # nothing to do
    # FP8 cache append needs its scale array
    assert lib.dsa_cache_append_fp8(fake, fake, ctypes.byref(r), None, ctypes.byref(r), fake, 1, 1,
                                    128, ctypes.c_float(1e-5), ws, 1 << 20,
                                    None) == dsa.DSA_ERR_INVALID_ARGUMENT


def test_host_argument_checks_bwd(dsa):
    lib = dsa.lib
    P = ctypes.c_void_p
    fake = P(1 << 20)
    ws = P(1 << 24)
    r = _rows(base=1 << 20, stride=128)

    def bwd(q=fake, dkv=fake, H=96, k=64, scale=0.07, d_o=fake):
        return lib.sparse_mla_bwd(q, ctypes.byref(r), fake, fake, fake, 1, 128, H, k, 128,
                                  ctypes.c_float(scale), fake, fake, d_o, fake, dkv, ws, 1 << 20,
                                  None)

    assert bwd(d_o=None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert bwd(dkv=P((1 << 20) + 4)) == dsa.DSA_ERR_INVALID_ARGUMENT   # dkv 16-byte aligned
    assert bwd(scale=0.0) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert bwd(H=160) == dsa.DSA_ERR_UNSUPPORTED
    assert bwd(k=4096) == dsa.DSA_ERR_UNSUPPORTED
