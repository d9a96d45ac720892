"""Helpers for the GPU tests: upload seeded inputs, run the CUDA path through the
binding, and evaluate the oracle on the same bits."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_attention_serving_gb300 as dsa
from parity import check_close, check_index_row, check_lse
from workloads import bf16_to_f32


def bf(a: np.ndarray) -> torch.Tensor:
    """uint16 BF16 bits -> CUDA bfloat16 tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def to_u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_indexer_rows(gpu_idx: np.ndarray, q_idx, w, k_logical, q_start, kv_len, topk, rows,
                       what=""):
    """Oracle scores + top-k on `rows` (flat b*Tq+i), checked against the GPU rows."""
    B, Tq = q_idx.shape[:2]
    o_idx, kth, sc, nv = oracle.indexer_topk(q_idx, w, k_logical, q_start, kv_len, topk, rows)
    swaps = 0
    flat = gpu_idx.reshape(B * Tq, topk)
    for r, row in enumerate(rows):
        swaps += check_index_row(flat[row], sc[r], int(nv[r]), topk, o_idx[r], kth[r],
                                 f"{what} row {row}")
    return swaps


def check_mla_rows(o_gpu: np.ndarray, lse_gpu: np.ndarray, q_lat, kv_logical, idx, q_start,
                   kv_len, scale, rows, what="", sink=None):
    B, Tq, H, _ = q_lat.shape
    o_ref, lse_ref = oracle.sparse_mla(q_lat, kv_logical, idx, q_start, kv_len, scale, rows,
                                       sink=sink)
    og = bf16_to_f32(o_gpu.reshape(B * Tq, H, 512)[rows])
    ma, rl = check_close(og, o_ref, f"{what} o_lat")
    if lse_gpu is not None:
        check_lse(lse_gpu.reshape(B * Tq, H)[rows], lse_ref, f"{what} lse")
    return ma, rl


def check_gate_rows(out_gpu: np.ndarray, x, W_g, o_lat_u16, W_uv, rows, what=""):
    o64 = bf16_to_f32(o_lat_u16).astype(np.float64)
    ref = oracle.gate(x, W_g, o64, W_uv, rows)
    return check_close(bf16_to_f32(out_gpu[rows]), ref, f"{what} gate")
