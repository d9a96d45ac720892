"""CPU oracle for the gated DSA attention step -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never loads it and has no fallback to it.

The arithmetic lives in ``dsa_oracle.c`` (plain C, double precision, one query
row per thread, compiled with gcc); this module only compiles it, marshals
numpy arrays and wraps each entry point.  Each wrapper names the passage its
C function follows.  The oracle shares no code with the CUDA path.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

RLAT, VLAT = 576, 512


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc (portable flags: no -march, no intrinsics)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, src, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library and declare its signatures."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_indexer_scores.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i64, P, P]
        lib.oracle_topk.argtypes = [P, P, i64, i32, i32, P, P]
        lib.oracle_sparse_mla.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, f64, i64, P, P, P]
        lib.oracle_dense_mla.argtypes = [P, P, P, P, i32, i32, i32, i32, f64, i64, P, P, P]
        lib.oracle_explicit_mla.argtypes = [P, P, P, P, P, P, P, i64, i32, i32, i32, i32, i32,
                                            i32, f64, P]
        lib.oracle_gate.argtypes = [P, P, P, P, i64, i32, i32, i32, i32, i64, P, P]
        lib.oracle_sparse_mla_sink.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, f64, P,
                                               i64, P, P, P]
        lib.oracle_layernorm.argtypes = [P, i64, i32, f64, P]
        lib.oracle_bf16_rne.argtypes = [P, i64, P]
        lib.oracle_e4m3_encode.argtypes = [P, i64, P]
        lib.oracle_e4m3_decode.argtypes = [P, i64, P]
        lib.oracle_quant_fp8.argtypes = [P, i64, i32, P, P]
        lib.oracle_indexer_scores_fp8.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                                  i64, P, P]
        lib.oracle_sparse_mla_f64.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, f64, P, i64,
                                              P, P, P]
        lib.oracle_sparse_mla_bwd.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, f64, P, P, P,
                                              P]
        lib.oracle_set_threads.argtypes = [i32]
        for f in ("oracle_indexer_scores", "oracle_topk", "oracle_sparse_mla", "oracle_dense_mla",
                  "oracle_explicit_mla", "oracle_gate", "oracle_set_threads",
                  "oracle_get_threads"):
            getattr(lib, f).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc == 2:
        raise OracleError(f"{what}: an index is out of range or not causal")
    if rc != 0:
        raise OracleError(f"{what}: error code {rc}")


def set_threads(n: int, lib=None) -> None:
    (lib or load()).oracle_set_threads(int(n))


def get_threads(lib=None) -> int:
    return int((lib or load()).oracle_get_threads())


def _rows(rows, B, Tq):
    if rows is None:
        rows = np.arange(B * Tq, dtype=np.int64)
    return _c(rows, np.int64)


def indexer_scores(q_idx, w, k_idx, q_start, kv_len, rows=None, lib=None):
    """Indexer scores I[t,s] = sum_j w[t,j]*max(0, q[t,j].k[s]) for every causal key.

    Follows "Kimi-K3.1-Pro" (NeMo AutoModel), Implementation Limits, bullet 2
    (BF16 inputs, every causal key scored), with the head-weighted ReLU form as
    the stated reading.  Returns [n_rows, S_max] float64, NaN beyond t.
    """
    lib = lib or load()
    B, Tq, H_I, D_I = q_idx.shape
    S_max = k_idx.shape[1]
    rows = _rows(rows, B, Tq)
    out = np.empty((len(rows), S_max), np.float64)
    q, ww, k = _c(q_idx, np.uint16), _c(w, np.uint16), _c(k_idx, np.uint16)
    qs, kl = _c(q_start, np.int32), _c(kv_len, np.int32)
    _check(lib.oracle_indexer_scores(_p(q), _p(ww), _p(k), _p(qs), _p(kl), B, Tq, S_max, H_I, D_I,
                                     len(rows), _p(rows), _p(out)), "indexer_scores")
    return out


def topk(scores, n_valid, k, lib=None):
    """Top-k per row by (score desc, index asc); a row with <= k keys keeps all.

    Follows "Kimi-K3.1-Pro" (NeMo AutoModel), Implementation Limits, bullets 1
    (top-k coordinates) and 4 (short sequences keep every causal key).
    Returns (idx [n_rows, k] int32 -1 padded, kth [n_rows] float64).
    """
    lib = lib or load()
    sc = _c(scores, np.float64)
    nv = _c(n_valid, np.int32)
    n_rows, S_max = sc.shape
    idx = np.empty((n_rows, k), np.int32)
    kth = np.empty(n_rows, np.float64)
    _check(lib.oracle_topk(_p(sc), _p(nv), n_rows, S_max, k, _p(idx), _p(kth)), "topk")
    return idx, kth


def sparse_mla(q_lat, kv, idx, q_start, kv_len, scale, rows=None, lib=None, sink=None):
    """Latent-space attention over the selected rows only (value = first 512 dims).

    Follows "Kimi-K3.1-Pro" (NeMo AutoModel), Implementation Limits, bullets 1-2;
    dims from KimiK3TextConfig (v0.4 API); no rotation ("Kimi K3.1 Pro",
    archdiff summary: no positional encoding).  Returns (o [n,H,512], lse [n,H]).
    sink: optional [H] learnable sink logits ("Kimi K3.1 Pro" archdiff blueprint,
    "Output gate + sink"): one more term in the softmax denominator, no value.
    """
    lib = lib or load()
    B, Tq, H, R = q_lat.shape
    assert R == RLAT
    S_max = kv.shape[1]
    topk_ = idx.shape[-1]
    rows = _rows(rows, B, Tq)
    o = np.empty((len(rows), H, VLAT), np.float64)
    lse = np.empty((len(rows), H), np.float64)
    q, k, ix = _c(q_lat, np.uint16), _c(kv, np.uint16), _c(idx, np.int32)
    qs, kl = _c(q_start, np.int32), _c(kv_len, np.int32)
    if sink is None:
        _check(lib.oracle_sparse_mla(_p(q), _p(k), _p(ix), _p(qs), _p(kl), B, Tq, S_max, H, topk_,
                                     float(scale), len(rows), _p(rows), _p(o), _p(lse)), "sparse_mla")
    else:
        sk = _c(sink, np.float64)
        assert sk.shape == (H,)
        _check(lib.oracle_sparse_mla_sink(_p(q), _p(k), _p(ix), _p(qs), _p(kl), B, Tq, S_max, H,
                                          topk_, float(scale), _p(sk), len(rows), _p(rows), _p(o),
                                          _p(lse)), "sparse_mla_sink")
    return o, lse


def dense_mla(q_lat, kv, q_start, kv_len, scale, rows=None, lib=None):
    """Dense causal latent attention over every key s <= t (the dense-mask reference)."""
    lib = lib or load()
    B, Tq, H, R = q_lat.shape
    assert R == RLAT
    S_max = kv.shape[1]
    rows = _rows(rows, B, Tq)
    o = np.empty((len(rows), H, VLAT), np.float64)
    lse = np.empty((len(rows), H), np.float64)
    q, k = _c(q_lat, np.uint16), _c(kv, np.uint16)
    qs, kl = _c(q_start, np.int32), _c(kv_len, np.int32)
    _check(lib.oracle_dense_mla(_p(q), _p(k), _p(qs), _p(kl), B, Tq, S_max, H, float(scale),
                                len(rows), _p(rows), _p(o), _p(lse)), "dense_mla")
    return o, lse


def explicit_mla(q_nope, q_pe, W_UK, W_UV, c_kv, k_pe, sel, scale, lib=None):
    """Non-absorbed MLA: per-head keys W_UK_h c_kv and values W_UV_h c_kv expanded.

    The path "Kimi-K3.1-Pro", Implementation Limits, bullet 2 says sparse MLA
    avoids; used to pin the absorbed latent form.  Returns [n, H, dv].
    """
    lib = lib or load()
    n, H, dn = q_nope.shape
    dr = q_pe.shape[2]
    R = c_kv.shape[1]
    dv = W_UV.shape[1]
    K = sel.shape[1]
    out = np.empty((n, H, dv), np.float64)
    a = [_c(v, np.float64) for v in (q_nope, q_pe, W_UK, W_UV, c_kv, k_pe)]
    s = _c(sel, np.int32)
    _check(lib.oracle_explicit_mla(*[_p(v) for v in a], _p(s), n, H, dn, dr, R, dv, K,
                                   float(scale), _p(out)), "explicit_mla")
    return out


def gate(x, W_g, o_lat, W_uv, rows=None, lib=None):
    """out[t, h*dv+e] = sigmoid(x[t].W_g[h*dv+e]) * (W_uv[h,e].o_lat[t,h]).

    Follows "Kimi K3.1 Pro" (archdiff), blueprint entry for the output gate,
    and KimiK3TextConfig (v0.4 API) ``mla_use_output_gate``, ``v_head_dim``.
    o_lat is float64 [N, H, 512].  Returns [n_rows, H*dv].
    """
    lib = lib or load()
    N, hid = x.shape
    H, dv, R = W_uv.shape
    rows = _rows(rows, N, 1)
    out = np.empty((len(rows), H * dv), np.float64)
    xx, wg, wu = _c(x, np.uint16), _c(W_g, np.uint16), _c(W_uv, np.uint16)
    ol = _c(o_lat, np.float64)
    assert ol.shape == (N, H, R)
    _check(lib.oracle_gate(_p(xx), _p(wg), _p(ol), _p(wu), N, hid, H, dv, R, len(rows), _p(rows),
                           _p(out)), "gate")
    return out


def indexer_topk(q_idx, w, k_idx, q_start, kv_len, k, rows=None, lib=None):
    """Scores and top-k for the given rows; returns (idx, kth, scores, n_valid)."""
    B, Tq = q_idx.shape[:2]
    rows = _rows(rows, B, Tq)
    sc = indexer_scores(q_idx, w, k_idx, q_start, kv_len, rows, lib=lib)
    qs = np.asarray(q_start, np.int64)
    n_valid = (qs[rows // Tq] + rows % Tq + 1).astype(np.int32)
    idx, kth = topk(sc, n_valid, k, lib=lib)
    return idx, kth, sc, n_valid


def layernorm(x, eps, lib=None) -> np.ndarray:
    """x [..., D] float32 -> float64 LayerNorm over the last axis (unit gain, zero
    bias, population variance) ("Kimi K3.1 Pro" archdiff blueprint: LayerNorm on
    the indexer key)."""
    lib = lib or load()
    x = _c(x, np.float32)
    D = x.shape[-1]
    y = np.empty(x.shape, np.float64)
    _check(lib.oracle_layernorm(_p(x), x.size // D, D, float(eps), _p(y)), "oracle_layernorm")
    return y


def bf16_rne(v, lib=None) -> np.ndarray:
    """float64 -> BF16 bit patterns, round to nearest, ties to even."""
    lib = lib or load()
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    _check(lib.oracle_bf16_rne(_p(v), v.size, _p(out)), "oracle_bf16_rne")
    return out


def cache_append(k_pre, kv_new, q_start, eps, k_cache, kv_cache, k_block_table=None,
                 kv_block_table=None, page=64, lib=None):
    """The cache append that precedes the indexer, on copies of the caches.

    k_pre [B,Tq,D] float32, kv_new [B,Tq,576] BF16 bits, q_start [B]; caches are
    contiguous [B,S,W] or page pools [P,page,W] with block tables [B,max_pages].
    Row q_start[b]+i of sequence b receives BF16(LayerNorm(k_pre[b,i])) and
    kv_new[b,i].  Returns (k_cache', kv_cache', (k_ln float64, positions))."""
    lib = lib or load()
    k_ln = layernorm(k_pre, eps, lib)
    k_bits = bf16_rne(k_ln, lib)
    kc, vc = np.array(k_cache, copy=True), np.array(kv_cache, copy=True)
    B, Tq, _ = k_pre.shape

    def place(cache, bt, b, pos, row):
        if bt is None:
            cache[b, pos] = row
        else:
            cache[bt[b, pos // page], pos % page] = row

    for b in range(B):
        for i in range(Tq):
            pos = int(q_start[b]) + i
            place(kc, k_block_table, b, pos, k_bits[b, i])
            place(vc, kv_block_table, b, pos, kv_new[b, i])
    return kc, vc, k_ln


# ---------------------------------------------------------------------------
# FP8 indexer variant ("Kimi-K3.1-Pro", NeMo AutoModel, Implementation Limits,
# bullet 2: the FP8 indexer of some serving kernels, against the BF16 one).
# Format and scaling are readings stated in dsa_oracle.c.
# ---------------------------------------------------------------------------

def e4m3_encode(x, lib=None) -> np.ndarray:
    """float32 -> E4M3 codes (uint8), round to nearest even, saturating at +-448."""
    lib = lib or load()
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _check(lib.oracle_e4m3_encode(_p(x), x.size, _p(out)), "oracle_e4m3_encode")
    return out


def e4m3_decode(c, lib=None) -> np.ndarray:
    """E4M3 codes -> float64 values."""
    lib = lib or load()
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    _check(lib.oracle_e4m3_decode(_p(c), c.size, _p(out)), "oracle_e4m3_decode")
    return out


def quant_fp8(x, lib=None):
    """BF16 rows [..., D] -> (codes [..., D] uint8, scale [...] float32): one FP32
    scale per row, scale = max(amax, 2^-100)/448, code = E4M3(x * (1/scale))."""
    lib = lib or load()
    x = _c(x, np.uint16)
    D = x.shape[-1]
    n = x.size // D
    codes = np.empty(x.shape, np.uint8)
    scale = np.empty(x.shape[:-1], np.float32)
    _check(lib.oracle_quant_fp8(_p(x), n, D, _p(codes), _p(scale)), "oracle_quant_fp8")
    return codes, scale


def indexer_scores_fp8(q_codes, q_scale, w, k_codes, k_scale, q_start, kv_len, rows=None,
                       lib=None):
    """Indexer scores of the dequantised FP8 rows: I[t,s] = sum_j w[t,j] *
    max(0, (q_scale[t,j] q[t,j]) . (k_scale[s] k[s])).  k_codes [B,S,D_I],
    k_scale [B,S].  Returns [n_rows, S_max] float64, NaN beyond t."""
    lib = lib or load()
    B, Tq, H_I, D_I = q_codes.shape
    S_max = k_codes.shape[1]
    rows = _rows(rows, B, Tq)
    out = np.empty((len(rows), S_max), np.float64)
    q, qs = _c(q_codes, np.uint8), _c(q_scale, np.float32)
    ww = _c(w, np.uint16)
    k, ks = _c(k_codes, np.uint8), _c(k_scale, np.float32)
    assert qs.shape == (B, Tq, H_I) and ks.shape == (B, S_max)
    qst, kl = _c(q_start, np.int32), _c(kv_len, np.int32)
    _check(lib.oracle_indexer_scores_fp8(_p(q), _p(qs), _p(ww), _p(k), _p(ks), _p(qst), _p(kl),
                                         B, Tq, S_max, H_I, D_I, len(rows), _p(rows), _p(out)),
           "indexer_scores_fp8")
    return out


def indexer_topk_fp8(q_codes, q_scale, w, k_codes, k_scale, q_start, kv_len, k, rows=None,
                     lib=None):
    """FP8 scores and top-k for the given rows; returns (idx, kth, scores, n_valid)."""
    B, Tq = q_codes.shape[:2]
    rows = _rows(rows, B, Tq)
    sc = indexer_scores_fp8(q_codes, q_scale, w, k_codes, k_scale, q_start, kv_len, rows, lib=lib)
    qs = np.asarray(q_start, np.int64)
    n_valid = (qs[rows // Tq] + rows % Tq + 1).astype(np.int32)
    idx, kth = topk(sc, n_valid, k, lib=lib)
    return idx, kth, sc, n_valid


# ---------------------------------------------------------------------------
# Sparse MLA backward ("Kimi-K3.1-Pro", NeMo AutoModel, Implementation Limits:
# bullets 1-2 (attention over the selected rows only), the paragraph after
# bullet 4 (a native 96-head backward), bullet 3 (hard top-k gives the indexer
# no gradient, so the index set is a constant here)).
# ---------------------------------------------------------------------------

def _as_f64(a):
    """BF16 bit patterns (uint16) -> float64, exactly; float arrays pass through."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return _c(a, np.float64)


def _sink(sink, H):
    if sink is None:
        return None
    sk = _c(sink, np.float64)
    assert sk.shape == (H,)
    return sk


def sparse_mla_f64(q_lat, kv, idx, q_start, kv_len, scale, rows=None, lib=None, sink=None):
    """The sparse MLA forward on exact (float64) values: (o [n,H,512], lse [n,H]);
    sink: optional [H] learnable sink logits (natural log)."""
    lib = lib or load()
    q, k = _as_f64(q_lat), _as_f64(kv)
    B, Tq, H, R = q.shape
    assert R == RLAT
    S_max = k.shape[1]
    topk_ = idx.shape[-1]
    rows = _rows(rows, B, Tq)
    o = np.empty((len(rows), H, VLAT), np.float64)
    lse = np.empty((len(rows), H), np.float64)
    ix = _c(idx, np.int32)
    qs, kl = _c(q_start, np.int32), _c(kv_len, np.int32)
    sk = _sink(sink, H)
    _check(lib.oracle_sparse_mla_f64(_p(q), _p(k), _p(ix), _p(qs), _p(kl), B, Tq, S_max, H, topk_,
                                     float(scale), None if sk is None else _p(sk), len(rows),
                                     _p(rows), _p(o), _p(lse)), "sparse_mla_f64")
    return o, lse


def sparse_mla_bwd(q_lat, kv, idx, q_start, kv_len, scale, dO, lib=None, sink=None):
    """Gradients of sum(dO * o) for the sparse MLA forward with a fixed index set:
    (dq [B,Tq,H,576], dkv [B,S,576]), float64.  Inputs may be BF16 bits or floats.
    sink: optional [H] learnable sink logits of the forward (natural log)."""
    lib = lib or load()
    q, k, g = _as_f64(q_lat), _as_f64(kv), _as_f64(dO)
    B, Tq, H, R = q.shape
    assert R == RLAT and g.shape == (B, Tq, H, VLAT)
    S_max = k.shape[1]
    topk_ = idx.shape[-1]
    dq = np.empty(q.shape, np.float64)
    dkv = np.empty(k.shape, np.float64)
    ix = _c(idx, np.int32)
    qs, kl = _c(q_start, np.int32), _c(kv_len, np.int32)
    sk = _sink(sink, H)
    _check(lib.oracle_sparse_mla_bwd(_p(q), _p(k), _p(ix), _p(qs), _p(kl), B, Tq, S_max, H, topk_,
                                     float(scale), None if sk is None else _p(sk), _p(g), _p(dq),
                                     _p(dkv)), "sparse_mla_bwd")
    return dq, dkv
