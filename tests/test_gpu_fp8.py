"""GPU parity of the FP8 (E4M3) indexer variant against the oracle.

* dsa_quant_fp8: codes and scales bit for bit (both sides use the same IEEE
  float operations and the same E4M3 rounding).
* dsa_cache_append_fp8: the codes and scale of the BF16 LayerNorm row.  Where
  the FP32 LayerNorm may round an element to either of two BF16 values (the
  BF16 rule of the BF16 append), every such choice is quantised by the oracle
  and the GPU row must equal one of them; elsewhere, bit for bit.
* dsa_indexer_topk_fp8: index sets under the near-tie rule against the
  oracle's FP8 scores (the dequantised rows in float64).

The FP8 operands are produced on the CPU by the oracle's quantiser from the
seeded BF16 inputs, never by the CUDA path.
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bf, i32, to_u16
from parity import check_index_row, layernorm_delta
from workloads import (Config, append_inputs, bf16_round, normal_bf16, page_table,
                       prefill_queries, to_pages)

pytestmark = pytest.mark.gpu

EPS = 1e-5


@pytest.fixture(scope="module")
def dsa():
    import sparse_attention_serving_gb300 as m
    return m


def u8(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda()


def f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


# ----------------------------------------------------------------------------
# quantiser
# ----------------------------------------------------------------------------

def _quant_rows(D, n, seed):
    x = normal_bf16(seed, "q_idx", (n, D))
    rng = np.random.default_rng(seed)
    x[0] = 0                                                          # all zero
    x[1] = bf16_round(np.full(D, 3.0, np.float32))                    # constant
    x[2] = bf16_round((rng.standard_normal(D) * 1e37).astype(np.float32))   # huge
    x[3] = bf16_round((rng.standard_normal(D) * 1e-35).astype(np.float32))  # below the floor
    x[4] = bf16_round((rng.standard_normal(D) * 1e-39).astype(np.float32))  # BF16 subnormals
    x[5] = bf16_round((rng.standard_normal(D) * 1e-3).astype(np.float32))
    x[6] = 0
    x[6, :2] = bf16_round(np.array([0.19140625, 0.08544921875], np.float32))  # x*inv != x/scale
    for r in range(7, min(n, 40)):                                    # mixed magnitudes
        x[r] = bf16_round((rng.standard_normal(D) * 10.0 ** rng.uniform(-6, 6, D)).astype(np.float32))
    return x


@pytest.mark.parametrize("D,n", [(128, 4099), (64, 777)])
def test_quant_fp8_bit_exact(dsa, D, n):
    x = _quant_rows(D, n, 60 + D)
    codes, scale = dsa.dsa_quant_fp8(bf(x))
    torch.cuda.synchronize()
    ec, es = oracle.quant_fp8(x)
    np.testing.assert_array_equal(scale.cpu().numpy().view(np.uint32), es.view(np.uint32))
    np.testing.assert_array_equal(codes.cpu().numpy(), ec)


def test_quant_fp8_query_shape(dsa):
    """A [B, Tq, H_I, D_I] query block quantises row by row (one scale per head)."""
    x = normal_bf16(62, "q_idx", (2, 3, 64, 128))
    codes, scale = dsa.dsa_quant_fp8(bf(x))
    ec, es = oracle.quant_fp8(x)
    assert tuple(scale.shape) == (2, 3, 64)
    np.testing.assert_array_equal(codes.cpu().numpy(), ec)
    np.testing.assert_array_equal(scale.cpu().numpy(), es)


# ----------------------------------------------------------------------------
# cache append
# ----------------------------------------------------------------------------

def _expected_fp8_rows(k_pre, eps):
    """Per new token: the list of (codes, scale) the GPU may write -- one entry
    unless the FP32 LayerNorm may round some elements either way."""
    v = oracle.layernorm(k_pre, eps)
    dl = layernorm_delta(k_pre, v, eps)
    lo, hi = oracle.bf16_rne(v - dl), oracle.bf16_rne(v + dl)
    mid = oracle.bf16_rne(v)
    B, Tq, D = k_pre.shape
    out = {}
    for b in range(B):
        for i in range(Tq):
            amb = np.nonzero(lo[b, i] != hi[b, i])[0]
            assert len(amb) <= 8, "too many elements next to a BF16 midpoint"
            cands = []
            for choice in itertools.product(*[(lo[b, i, d], hi[b, i, d]) for d in amb]):
                row = mid[b, i].copy()
                row[amb] = choice
                cands.append(row)
            c, s = oracle.quant_fp8(np.stack(cands))
            out[b, i] = (c, s)
    return out


def _check_append_fp8(dsa, inp, q_start, D, bt=None, S=None, what=""):
    B, Tq, _ = inp["k_pre"].shape
    rng = np.random.default_rng(7)
    if bt is None:
        kshape, sshape, vshape = (B, S, D), (B, S), (B, S, 576)
    else:
        npages = int(bt.max()) + 1
        kshape, sshape, vshape = (npages, 64, D), (npages, 64), (npages, 64, 576)
    k0 = rng.integers(0, 256, kshape).astype(np.uint8)
    s0 = rng.standard_normal(sshape).astype(np.float32)
    v0 = rng.integers(0, 0x7F7F, vshape).astype(np.uint16)
    kc, sc, vc = u8(k0), f32(s0), bf(v0)
    bt_t = None if bt is None else i32(bt)
    ws = dsa.dsa_cache_append_fp8(torch.from_numpy(inp["k_pre"]).cuda(), bf(inp["kv_new"]),
                                  dsa.Rows(kc, bt_t), sc, dsa.Rows(vc, bt_t), i32(q_start), EPS)
    code, where, detail = dsa.read_device_status(ws)
    assert code == dsa.DSA_OK, (code, hex(where), detail)
    gk, gs, gv = kc.cpu().numpy(), sc.cpu().numpy(), to_u16(vc)
    exp = _expected_fp8_rows(inp["k_pre"], EPS)
    written = np.zeros(sshape, bool)
    ambiguous = 0
    for b in range(B):
        for i in range(Tq):
            pos = int(q_start[b]) + i
            at = (b, pos) if bt is None else (bt[b, pos // 64], pos % 64)
            written[at] = True
            c, s = exp[b, i]
            ok = [j for j in range(len(s)) if s[j] == gs[at] and np.array_equal(c[j], gk[at])]
            assert ok, f"{what}: token ({b},{i}) codes/scale match no admissible BF16 row"
            ambiguous += len(s) > 1
            np.testing.assert_array_equal(gv[at], inp["kv_new"][b, i], err_msg=f"{what}: latent")
    np.testing.assert_array_equal(gk[~written], k0[~written], err_msg=f"{what}: untouched codes")
    np.testing.assert_array_equal(gs[~written], s0[~written], err_msg=f"{what}: untouched scales")
    np.testing.assert_array_equal(gv[~written], v0[~written], err_msg=f"{what}: untouched latent")
    return ambiguous


def test_append_fp8_decode_paged(dsa):
    lens = np.array([1, 64, 65, 300, 2049], np.int32)
    bt, _ = page_table(51, lens)
    inp = append_inputs(51, len(lens), 1, 128)
    _check_append_fp8(dsa, inp, lens - 1, 128, bt=bt, what="decode paged")


@pytest.mark.parametrize("D", [128, 64])
def test_append_fp8_chunk_contiguous(dsa, D):
    inp = append_inputs(52, 2, 300, D)
    # rows with an element next to a BF16 midpoint are checked against every
    # admissible rounding (at most 8 such elements per row, asserted above)
    _check_append_fp8(dsa, inp, np.array([0, 377], np.int32), D, S=700,
                      what=f"chunk contiguous D={D}")


# ----------------------------------------------------------------------------
# decode indexer
# ----------------------------------------------------------------------------

def _decode_fp8(dsa, lens, seed, topk, paged=True, stride_pad=0):
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    cfg = Config("decode-fp8", B=B, T=1, topk=topk, H_I=64, D_I=128, H=96, hid=1024, seed=seed)
    S = int(lens.max())
    k_log = normal_bf16(seed, "k_idx", (B, S, 128))
    q = prefill_queries(cfg, 0, 1)
    kc, ks = oracle.quant_fp8(k_log)
    qc, qsc = oracle.quant_fp8(q["q_idx"])
    qs, kl = lens - 1, lens
    if paged:
        bt, npages = page_table(seed, lens)
        kc_dev = dsa.Rows(u8(to_pages(kc, lens, bt, npages)), i32(bt))
        ks_dev = f32(to_pages(ks[..., None], lens, bt, npages)[..., 0])
    else:
        Sp = (S + stride_pad + 3) // 4 * 4
        kcp = np.zeros((B, Sp, 128), np.uint8)
        ksp = np.zeros((B, Sp), np.float32)
        kcp[:, :S], ksp[:, :S] = kc, ks
        kc_dev, ks_dev = dsa.Rows(u8(kcp)), f32(ksp)
    idx = dsa.dsa_indexer_topk_fp8(u8(qc), f32(qsc), bf(q["w"]), kc_dev, ks_dev, i32(qs), i32(kl),
                                   topk, S)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy().reshape(B, topk)
    rows = np.arange(B)
    o_idx, kth, sc, nv = oracle.indexer_topk_fp8(qc, qsc, q["w"], kc, ks, qs, kl, topk, rows)
    swaps = 0
    for r in rows:
        swaps += check_index_row(gi[r], sc[r], int(nv[r]), topk, o_idx[r], kth[r],
                                 f"fp8 decode request {r} (L={lens[r]})")
    return swaps


def test_decode_fp8_paged_ragged(dsa):
    """Requests shorter than k, at k, one past k and long ones with ragged tails."""
    _decode_fp8(dsa, [1, 100, 2048, 2049, 5000, 9001, 12345], 53, 2048)


def test_decode_fp8_contiguous(dsa):
    """Contiguous key codes (row stride padded to a multiple of 4 past the longest request)."""
    _decode_fp8(dsa, [777, 3000, 4099], 54, 512, paged=False, stride_pad=1)


def test_decode_fp8_small_topk(dsa):
    _decode_fp8(dsa, [300, 1000, 2500], 55, 64)


def test_decode_fp8_rejects_bad_stride(dsa):
    qc = torch.zeros((1, 1, 64, 128), dtype=torch.uint8, device="cuda")
    qs = torch.ones((1, 1, 64), dtype=torch.float32, device="cuda")
    w = torch.zeros((1, 1, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 130, 128), dtype=torch.uint8, device="cuda")
    ks = torch.ones((1, 130), dtype=torch.float32, device="cuda")
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_indexer_topk_fp8(qc, qs, w, dsa.Rows(kc), ks, i32([1]), i32([2]), 64, 128)
    assert e.value.code == dsa.DSA_ERR_UNSUPPORTED                   # row stride 130


# ----------------------------------------------------------------------------
# prefill indexer
# ----------------------------------------------------------------------------

def _prefill_fp8(dsa, B, T, topk, seed, rows, q0=0, nq=None, paged=False):
    """Queries [q0, q0+nq) of B sequences of T keys (a chunk when q0 > 0)."""
    nq = T - q0 if nq is None else nq
    cfg = Config("prefill-fp8", B=B, T=T, topk=topk, H_I=64, D_I=128, H=96, hid=1024, seed=seed)
    q = prefill_queries(cfg, q0, nq)
    k_log = normal_bf16(seed, "k_idx", (B, T, 128))
    kc, ks = oracle.quant_fp8(k_log)
    qc, qsc = oracle.quant_fp8(q["q_idx"])
    q_start = np.full(B, q0, np.int32)
    kv_len = np.full(B, q0 + nq, np.int32)
    if paged:
        lens = np.full(B, T, np.int32)
        bt, npages = page_table(seed, lens)
        kc_dev = dsa.Rows(u8(to_pages(kc, lens, bt, npages)), i32(bt))
        ks_dev = f32(to_pages(ks[..., None], lens, bt, npages)[..., 0])
    else:
        Sp = (T + 3) // 4 * 4
        kcp = np.zeros((B, Sp, 128), np.uint8)
        ksp = np.zeros((B, Sp), np.float32)
        kcp[:, :T], ksp[:, :T] = kc, ks
        kc_dev, ks_dev = dsa.Rows(u8(kcp)), f32(ksp)
    idx = dsa.dsa_indexer_topk_fp8(u8(qc), f32(qsc), bf(q["w"]), kc_dev, ks_dev, i32(q_start),
                                   i32(kv_len), topk, T)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy().reshape(B * nq, topk)
    o_idx, kth, sc, nv = oracle.indexer_topk_fp8(qc, qsc, q["w"], kc[:, :q0 + nq], ks[:, :q0 + nq],
                                                 q_start, kv_len, topk, rows)
    swaps = 0
    for r, row in enumerate(rows):
        swaps += check_index_row(gi[row], sc[r], int(nv[r]), topk, o_idx[r], kth[r],
                                 f"fp8 prefill row {row}")
    return swaps


def test_prefill_fp8_ragged_contiguous(dsa):
    """Two sequences of 777 keys (a ragged last tile), top-256: rows below, at and
    far past k, both sequences."""
    T = 777
    rows = np.array([0, 1, 100, 255, 256, 257, 500, 700, 775, 776, T, T + 300, 2 * T - 1])
    _prefill_fp8(dsa, 2, T, 256, 56, rows)


def test_prefill_fp8_topk_2048(dsa):
    """k = 2,048 with T = 2,600: the head keeps every key, the tail selects."""
    T = 2600
    rows = np.array([0, 2046, 2047, 2048, 2049, 2300, 2599])
    _prefill_fp8(dsa, 1, T, 2048, 57, rows)


def test_prefill_fp8_chunk_paged(dsa):
    """Chunk 2 of a paged chunked prefill: queries 1,024..1,535 over 1,536 keys."""
    rows = np.array([0, 1, 200, 511])
    _prefill_fp8(dsa, 1, 1536, 512, 58, rows, q0=1024, nq=512, paged=True)
