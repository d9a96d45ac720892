"""Python binding of libdsa.so, the gated DSA attention step on GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/dsa.h``.  PyTorch supplies device
memory and streams.  There is no CPU or PyTorch fallback: importing this
package without a built ``libdsa.so`` raises, and calling an entry point
without a CUDA device fails.

Entry points (same names as the C ABI):
  dsa_indexer_topk  lightning indexer scores + top-k key positions
  sparse_mla_fwd    latent-space attention over the selected rows
  mla_gate_apply    sigmoid output gate applied after the per-head up-projection
  dsa_cache_append  LayerNorm of new indexer keys + append of keys and latent rows
  dsa_quant_fp8, dsa_cache_append_fp8, dsa_indexer_topk_fp8
                    the FP8 (E4M3, one FP32 scale per row) indexer variant
  sparse_mla_bwd    gradients of sparse MLA for q_lat and the latent rows
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

DSA_OK = 0
DSA_ERR_INVALID_ARGUMENT = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_CUDA = 3
DSA_ERR_DEVICE_TIMEOUT = 4
DSA_ERR_BAD_INDEX = 5
DSA_ERR_WORKSPACE_TOO_SMALL = 6

OP_INDEXER_TOPK, OP_SPARSE_MLA, OP_GATE, OP_CACHE_APPEND, OP_SPARSE_MLA_BWD = 0, 1, 2, 3, 4
INDEXER_KEY_EPS = 1e-5   # KimiK3TextConfig rms_norm_eps
RLAT, VLAT, PAGE = 576, 512, 64
MLA_SCALE = 1.0 / math.sqrt(128 + 64)   # qk_nope_head_dim + qk_rope_head_dim


class DsaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (code {code})")


class _Rows(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("seq_stride", ctypes.c_int64),
                ("block_table", ctypes.c_void_p), ("max_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


EXPORTS = ("dsa_abi_version", "dsa_status_string", "dsa_workspace_bytes", "dsa_workspace_init",
           "dsa_read_device_status", "dsa_indexer_topk", "sparse_mla_fwd", "mla_gate_apply",
           "dsa_cache_append", "sparse_mla_fwd_sink", "dsa_selftest_wait_timeout",
           "dsa_quant_fp8", "dsa_cache_append_fp8", "dsa_indexer_topk_fp8", "sparse_mla_bwd")


def _load(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python sparse_attention_serving_gb300/build.py`"
                          " (there is no fallback path)")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.dsa_abi_version.restype = I
    lib.dsa_status_string.argtypes = [I]
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.dsa_workspace_bytes.restype = Z
    lib.dsa_workspace_init.argtypes = [P, Z, P]
    lib.dsa_read_device_status.argtypes = [P, P, P, P]
    lib.dsa_indexer_topk.argtypes = [P, P, ctypes.POINTER(_Rows), P, P, I, I, I, I, I, I, P, P, Z, P]
    lib.sparse_mla_fwd.argtypes = [P, ctypes.POINTER(_Rows), P, P, P, I, I, I, I, I,
                                   ctypes.c_float, P, P, P, Z, P]
    lib.sparse_mla_fwd_sink.argtypes = [P, ctypes.POINTER(_Rows), P, P, P, I, I, I, I, I,
                                        ctypes.c_float, P, P, P, P, Z, P]
    lib.mla_gate_apply.argtypes = [P, P, P, P, I, I, I, I, P, P, Z, P]
    lib.dsa_cache_append.argtypes = [P, P, ctypes.POINTER(_Rows), ctypes.POINTER(_Rows), P, I, I, I,
                                     ctypes.c_float, P, Z, P]
    lib.dsa_selftest_wait_timeout.argtypes = [P, Z, ctypes.c_uint64, P]
    lib.dsa_quant_fp8.argtypes = [P, ctypes.c_int64, I, P, P, P]
    lib.dsa_cache_append_fp8.argtypes = [P, P, ctypes.POINTER(_Rows), P, ctypes.POINTER(_Rows), P,
                                         I, I, I, ctypes.c_float, P, Z, P]
    lib.dsa_indexer_topk_fp8.argtypes = [P, P, P, ctypes.POINTER(_Rows), P, P, P, I, I, I, I, I, I,
                                         P, P, Z, P]
    lib.sparse_mla_bwd.argtypes = [P, ctypes.POINTER(_Rows), P, P, P, I, I, I, I, I,
                                   ctypes.c_float, P, P, P, P, P, P, Z, P]
    for f in ("sparse_mla_bwd", "dsa_workspace_init", "dsa_read_device_status", "dsa_indexer_topk",
              "sparse_mla_fwd", "mla_gate_apply", "dsa_cache_append", "sparse_mla_fwd_sink",
              "dsa_selftest_wait_timeout", "dsa_quant_fp8", "dsa_cache_append_fp8",
              "dsa_indexer_topk_fp8"):
        getattr(lib, f).restype = I
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.dsa_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != DSA_OK:
        raise DsaError(code, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise DsaError(DSA_ERR_INVALID_ARGUMENT, f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise DsaError(DSA_ERR_INVALID_ARGUMENT, f"{name} must be contiguous")


class Rows:
    """A per-token row store: contiguous ``[B, S, width]`` or a paged pool
    ``[num_pages, 64, width]`` with ``block_table [B, max_pages]`` (int32).
    BF16 rows, or uint8 rows of E4M3 codes for the FP8 indexer variant."""

    def __init__(self, base: torch.Tensor, block_table: torch.Tensor | None = None,
                 seq_stride: int | None = None):
        _need(base, torch.uint8 if base.dtype == torch.uint8 else torch.bfloat16, "rows.base")
        self.base = base
        self.block_table = block_table
        if block_table is None:
            if base.dim() != 3:
                raise ValueError("contiguous rows must be [B, S, width]")
            self.seq_stride = base.shape[1] if seq_stride is None else seq_stride
            self.num_pages = 0
            self.max_pages = 0
        else:
            _need(block_table, torch.int32, "block_table")
            if base.dim() != 3 or base.shape[1] != PAGE:
                raise ValueError("paged rows must be [num_pages, 64, width]")
            self.seq_stride = 0
            self.num_pages = base.shape[0]
            self.max_pages = block_table.shape[1]

    def c(self) -> _Rows:
        return _Rows(self.base.data_ptr(), int(self.seq_stride),
                     0 if self.block_table is None else self.block_table.data_ptr(),
                     int(self.max_pages), PAGE if self.block_table is not None else 0,
                     int(self.num_pages))


def workspace_bytes(op: int, B: int, Tq: int, max_kv_len: int, heads: int, topk: int) -> int:
    return int(lib.dsa_workspace_bytes(op, B, Tq, max_kv_len, heads, topk))


def new_workspace(nbytes: int, device=None, stream=None) -> torch.Tensor:
    """Allocate (through torch) and initialise a workspace of at least nbytes."""
    nbytes = max(256, (int(nbytes) + 255) // 256 * 256)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
    _check(lib.dsa_workspace_init(_ptr(ws), nbytes, _stream(stream)), "dsa_workspace_init")
    return ws


def read_device_status(workspace: torch.Tensor, stream=None):
    """Synchronise the stream, return (code, where, detail) and clear the status."""
    where, detail = ctypes.c_uint32(0), ctypes.c_uint32(0)
    code = lib.dsa_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(where),
                                      ctypes.byref(detail))
    return int(code), int(where.value), int(detail.value)


def selftest_wait_timeout(workspace: torch.Tensor, limit_ns: int = 20_000_000, stream=None):
    """Run the device failure-path self-test; returns (code, where, detail) read back."""
    _check(lib.dsa_selftest_wait_timeout(_ptr(workspace), workspace.numel(), int(limit_ns),
                                         _stream(stream)), "dsa_selftest_wait_timeout")
    return read_device_status(workspace, stream)


def _ws(workspace, op, B, Tq, max_kv_len, heads, topk, device, stream):
    need = workspace_bytes(op, B, Tq, max_kv_len, heads, topk)
    if workspace is None:
        workspace = new_workspace(need, device, stream)
    _need(workspace, torch.uint8, "workspace")
    return workspace


def dsa_indexer_topk(q_idx, w, k_idx: Rows, q_start, kv_len, topk: int, max_kv_len: int,
                     out_idx=None, workspace=None, stream=None):
    """q_idx [B,Tq,H_I,D_I] bf16, w [B,Tq,H_I] bf16, k_idx Rows (width D_I),
    q_start/kv_len [B] int32 -> out_idx [B,Tq,topk] int32 (-1 padded)."""
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(w, torch.bfloat16, "w")
    _need(q_start, torch.int32, "q_start")
    _need(kv_len, torch.int32, "kv_len")
    B, Tq, H_I, D_I = q_idx.shape
    if out_idx is None:
        out_idx = torch.empty((B, Tq, topk), dtype=torch.int32, device=q_idx.device)
    _need(out_idx, torch.int32, "out_idx")
    ws = _ws(workspace, OP_INDEXER_TOPK, B, Tq, max_kv_len, H_I, topk, q_idx.device, stream)
    rows = k_idx.c()
    _check(lib.dsa_indexer_topk(_ptr(q_idx), _ptr(w), ctypes.byref(rows), _ptr(q_start),
                                _ptr(kv_len), B, Tq, H_I, D_I, int(max_kv_len), int(topk),
                                _ptr(out_idx), _ptr(ws), ws.numel(), _stream(stream)),
           "dsa_indexer_topk")
    return out_idx


def sparse_mla_fwd(q_lat, kv: Rows, idx, q_start, kv_len, max_kv_len: int, scale: float = MLA_SCALE,
                   o_lat=None, lse=None, want_lse: bool = True, workspace=None, stream=None,
                   sink=None):
    """q_lat [B,Tq,H,576] bf16, kv Rows (width 576), idx [B,Tq,topk] int32 ->
    (o_lat [B,Tq,H,512] bf16, lse [B,Tq,H] float32 or None).  sink: optional [H]
    float32 learnable sink logits (calls sparse_mla_fwd_sink)."""
    _need(q_lat, torch.bfloat16, "q_lat")
    _need(idx, torch.int32, "idx")
    _need(q_start, torch.int32, "q_start")
    _need(kv_len, torch.int32, "kv_len")
    B, Tq, H, R = q_lat.shape
    topk = idx.shape[-1]
    if o_lat is None:
        o_lat = torch.empty((B, Tq, H, VLAT), dtype=torch.bfloat16, device=q_lat.device)
    _need(o_lat, torch.bfloat16, "o_lat")
    if lse is None and want_lse:
        lse = torch.empty((B, Tq, H), dtype=torch.float32, device=q_lat.device)
    if lse is not None:
        _need(lse, torch.float32, "lse")
    ws = _ws(workspace, OP_SPARSE_MLA, B, Tq, max_kv_len, H, topk, q_lat.device, stream)
    rows = kv.c()
    if sink is None:
        _check(lib.sparse_mla_fwd(_ptr(q_lat), ctypes.byref(rows), _ptr(idx), _ptr(q_start),
                                  _ptr(kv_len), B, Tq, H, topk, int(max_kv_len), float(scale),
                                  _ptr(o_lat), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)),
               "sparse_mla_fwd")
    else:
        _need(sink, torch.float32, "sink")
        if tuple(sink.shape) != (H,):
            raise ValueError("sink must be [H]")
        _check(lib.sparse_mla_fwd_sink(_ptr(q_lat), ctypes.byref(rows), _ptr(idx), _ptr(q_start),
                                       _ptr(kv_len), B, Tq, H, topk, int(max_kv_len),
                                       float(scale), _ptr(sink), _ptr(o_lat), _ptr(lse),
                                       _ptr(ws), ws.numel(), _stream(stream)),
               "sparse_mla_fwd_sink")
    return o_lat, lse


def mla_gate_apply(x, W_g, o_lat, W_uv, out=None, workspace=None, stream=None):
    """x [N,hid] bf16, W_g [H*dv,hid] bf16, o_lat [N,H,512] bf16, W_uv [H,dv,512] bf16
    -> out [N, H*dv] bf16."""
    for t, n in ((x, "x"), (W_g, "W_g"), (o_lat, "o_lat"), (W_uv, "W_uv")):
        _need(t, torch.bfloat16, n)
    N, hid = x.shape
    H, dv, R = W_uv.shape
    if out is None:
        out = torch.empty((N, H * dv), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    ws = _ws(workspace, OP_GATE, N, 1, 0, H, 0, x.device, stream)
    _check(lib.mla_gate_apply(_ptr(x), _ptr(W_g), _ptr(o_lat), _ptr(W_uv), N, hid, H, dv,
                              _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "mla_gate_apply")
    return out


def dsa_cache_append(k_pre, kv_new, k_cache: Rows, kv_cache: Rows, q_start,
                     eps: float = INDEXER_KEY_EPS, workspace=None, stream=None):
    """k_pre [B,Tq,D_I] float32, kv_new [B,Tq,576] bf16, caches as Rows (written in
    place), q_start [B] int32: LayerNorm'd BF16 keys and the latent rows land at
    positions q_start[b]+i.  Returns the workspace (its status word holds any
    BAD_INDEX raised for rows the caches do not have)."""
    _need(k_pre, torch.float32, "k_pre")
    _need(kv_new, torch.bfloat16, "kv_new")
    _need(q_start, torch.int32, "q_start")
    B, Tq, D_I = k_pre.shape
    if tuple(kv_new.shape) != (B, Tq, RLAT):
        raise ValueError("kv_new must be [B, Tq, 576]")
    ws = _ws(workspace, OP_CACHE_APPEND, B, Tq, 0, 0, 0, k_pre.device, stream)
    kr, vr = k_cache.c(), kv_cache.c()
    _check(lib.dsa_cache_append(_ptr(k_pre), _ptr(kv_new), ctypes.byref(kr), ctypes.byref(vr),
                                _ptr(q_start), B, Tq, D_I, float(eps), _ptr(ws), ws.numel(),
                                _stream(stream)), "dsa_cache_append")
    return ws


# ---------------------------------------------------------------------------
# FP8 (E4M3) indexer variant
# ---------------------------------------------------------------------------

def dsa_quant_fp8(x, codes=None, scale=None, stream=None):
    """x [..., D] bf16 (D in {64, 128}) -> (codes [..., D] uint8, scale [...] float32):
    scale = max(amax, 2^-100)/448 per row, code = E4M3(x * (1/scale))."""
    _need(x, torch.bfloat16, "x")
    D = x.shape[-1]
    n = x.numel() // D if D else 0
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _need(codes, torch.uint8, "codes")
    _need(scale, torch.float32, "scale")
    _check(lib.dsa_quant_fp8(_ptr(x), n, D, _ptr(codes), _ptr(scale), _stream(stream)),
           "dsa_quant_fp8")
    return codes, scale


def dsa_cache_append_fp8(k_pre, kv_new, k_codes: Rows, k_scale, kv_cache: Rows, q_start,
                         eps: float = INDEXER_KEY_EPS, workspace=None, stream=None):
    """dsa_cache_append with the key stored as E4M3 codes (k_codes, uint8 rows of
    D_I) plus one float32 scale per row (k_scale, laid out like k_codes' rows:
    [B, S] contiguous or [num_pages, 64] paged).  Returns the workspace."""
    _need(k_pre, torch.float32, "k_pre")
    _need(kv_new, torch.bfloat16, "kv_new")
    _need(q_start, torch.int32, "q_start")
    _need(k_scale, torch.float32, "k_scale")
    B, Tq, D_I = k_pre.shape
    if tuple(kv_new.shape) != (B, Tq, RLAT):
        raise ValueError("kv_new must be [B, Tq, 576]")
    ws = _ws(workspace, OP_CACHE_APPEND, B, Tq, 0, 0, 0, k_pre.device, stream)
    kr, vr = k_codes.c(), kv_cache.c()
    _check(lib.dsa_cache_append_fp8(_ptr(k_pre), _ptr(kv_new), ctypes.byref(kr), _ptr(k_scale),
                                    ctypes.byref(vr), _ptr(q_start), B, Tq, D_I, float(eps),
                                    _ptr(ws), ws.numel(), _stream(stream)),
           "dsa_cache_append_fp8")
    return ws


def dsa_indexer_topk_fp8(q_codes, q_scale, w, k_codes: Rows, k_scale, q_start, kv_len, topk: int,
                         max_kv_len: int, out_idx=None, workspace=None, stream=None):
    """q_codes [B,Tq,H_I,D_I] uint8, q_scale [B,Tq,H_I] float32, w [B,Tq,H_I] bf16,
    k_codes Rows (uint8, width D_I), k_scale float32 laid out like k_codes' rows
    -> out_idx [B,Tq,topk] int32 (-1 padded)."""
    _need(q_codes, torch.uint8, "q_codes")
    _need(q_scale, torch.float32, "q_scale")
    _need(w, torch.bfloat16, "w")
    _need(k_scale, torch.float32, "k_scale")
    _need(q_start, torch.int32, "q_start")
    _need(kv_len, torch.int32, "kv_len")
    B, Tq, H_I, D_I = q_codes.shape
    if out_idx is None:
        out_idx = torch.empty((B, Tq, topk), dtype=torch.int32, device=q_codes.device)
    _need(out_idx, torch.int32, "out_idx")
    ws = _ws(workspace, OP_INDEXER_TOPK, B, Tq, max_kv_len, H_I, topk, q_codes.device, stream)
    rows = k_codes.c()
    _check(lib.dsa_indexer_topk_fp8(_ptr(q_codes), _ptr(q_scale), _ptr(w), ctypes.byref(rows),
                                    _ptr(k_scale), _ptr(q_start), _ptr(kv_len), B, Tq, H_I, D_I,
                                    int(max_kv_len), int(topk), _ptr(out_idx), _ptr(ws),
                                    ws.numel(), _stream(stream)), "dsa_indexer_topk_fp8")
    return out_idx


def sparse_mla_bwd(q_lat, kv: Rows, idx, q_start, kv_len, max_kv_len: int, o_lat, lse, d_o,
                   dkv, scale: float = MLA_SCALE, dq=None, workspace=None, stream=None):
    """Backward of sparse_mla_fwd for a fixed index set: returns dq [B,Tq,H,576]
    float32 and ADDS the latent-row gradients into dkv (float32, laid out like
    kv's rows: [B, S, 576] or [num_pages, 64, 576]; zero it first)."""
    _need(q_lat, torch.bfloat16, "q_lat")
    _need(idx, torch.int32, "idx")
    _need(o_lat, torch.bfloat16, "o_lat")
    _need(lse, torch.float32, "lse")
    _need(d_o, torch.bfloat16, "d_o")
    _need(dkv, torch.float32, "dkv")
    _need(q_start, torch.int32, "q_start")
    _need(kv_len, torch.int32, "kv_len")
    B, Tq, H, _ = q_lat.shape
    topk = idx.shape[-1]
    if dq is None:
        dq = torch.empty((B, Tq, H, RLAT), dtype=torch.float32, device=q_lat.device)
    _need(dq, torch.float32, "dq")
    ws = _ws(workspace, OP_SPARSE_MLA_BWD, B, Tq, 0, 0, 0, q_lat.device, stream)
    rows = kv.c()
    _check(lib.sparse_mla_bwd(_ptr(q_lat), ctypes.byref(rows), _ptr(idx), _ptr(q_start),
                              _ptr(kv_len), B, Tq, H, topk, int(max_kv_len), float(scale),
                              _ptr(o_lat), _ptr(lse), _ptr(d_o), _ptr(dq), _ptr(dkv), _ptr(ws),
                              ws.numel(), _stream(stream)), "sparse_mla_bwd")
    return dq
