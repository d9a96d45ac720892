"""Seeded synthetic inputs for the gated DSA attention step.

This module holds random draws and storage-format conversions only (BF16
rounding, paged-cache layout, length draws): none of the method's arithmetic.
Both the CPU oracle (``oracle/``) and the CUDA path consume the buffers it
returns, so a parity test feeds the two sides the same bits.

Workload shapes follow the pages' workloads:

* "Kimi-K3.1-Pro" (NeMo AutoModel model coverage), *Validation and Training*:
  single-document inputs of 4,096 and 8,192 tokens.
* Same page, *Implementation Limits*: a sequence needs more than 2,048 valid
  tokens before top-k selection drops anything.
* "nemo_automodel.components.models.kimi_k3" (v0.4 API), *KimiK3TextConfig*:
  ``num_attention_heads 96``, ``kv_lora_rank 512``, ``qk_rope_head_dim 64``,
  ``v_head_dim 128``, ``hidden_size 7168``.

Every array has its own streams ``default_rng([seed, stream_id, sub, slab])``
(PCG64), so any array, or any chunk of the queries, can be drawn without
drawing the others first.  Activations are N(0, 1), weights N(0, 0.02), all
rounded to BF16 by round-to-nearest-even and stored as ``uint16``.
The indexer key is drawn directly as the output of a LayerNorm with unit gain
and zero bias: i.i.d. N(0, 1) entries (the boundary takes normalised keys).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

R_LAT = 576      # latent KV row: 512 c_kv + 64 unrotated k_pe
V_LAT = 512      # value = the first 512 latent dims
PAGE = 64        # tokens per cache page

# one stream id per array; never reuse an id for a different array
_STREAM = {
    "x": 1, "W_g": 2, "W_uv": 3, "q_idx": 4, "w": 5, "k_idx": 6,
    "q_lat": 7, "kv": 8, "pages": 9, "lens": 10, "k_pre": 11, "kv_new": 12,
}


@dataclass(frozen=True)
class Config:
    name: str
    B: int            # sequences (or decode requests)
    T: int            # tokens per sequence (prefill) / unused for decode
    topk: int
    H_I: int          # indexer heads
    D_I: int          # indexer head dim
    H: int            # MLA query heads
    hid: int          # gate input width (hidden size)
    dv: int = 128     # per-head value dim after W_UV
    chunk: int = 0    # >0: chunked prefill with this many queries per chunk
    paged: bool = False
    decode: bool = False
    L_min: int = 0
    L_max: int = 0
    seed: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        # qk_nope_head_dim 128 + qk_rope_head_dim 64 = 192
        return 1.0 / math.sqrt(192.0)


CONFIGS = {
    # 1: tiny prefill, and its T <= k variant
    "tiny": Config("tiny", B=1, T=512, topk=128, H_I=4, D_I=64, H=8, hid=1024, seed=1),
    "tiny128": Config("tiny128", B=1, T=128, topk=128, H_I=4, D_I=64, H=8, hid=1024, seed=11),
    # 2: validation-length prefill
    "val4096": Config("val4096", B=1, T=4096, topk=2048, H_I=64, D_I=128, H=96, hid=7168, seed=2),
    # 3: headline prefill
    "head8192": Config("head8192", B=2, T=8192, topk=2048, H_I=64, D_I=128, H=96, hid=7168, seed=3),
    # 4: long-context chunked prefill over a paged cache
    "chunk32k": Config("chunk32k", B=1, T=32768, topk=2048, H_I=64, D_I=128, H=96, hid=7168,
                       chunk=8192, paged=True, seed=4),
    # 5: serving decode over paged caches
    "decode64": Config("decode64", B=64, T=1, topk=2048, H_I=64, D_I=128, H=96, hid=7168,
                       paged=True, decode=True, L_min=16384, L_max=131072, seed=5),
    # the same request mix at 16 requests (about 2 GB of caches): the profiling case
    "decode16": Config("decode16", B=16, T=1, topk=2048, H_I=64, D_I=128, H=96, hid=7168,
                       paged=True, decode=True, L_min=16384, L_max=131072, seed=6),
}


# ----------------------------------------------------------------------------
# storage format
# ----------------------------------------------------------------------------

def bf16_round(a: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bits (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """BF16 bits (uint16) -> float32, exact."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_trunc_check(a: np.ndarray) -> bool:
    """True when every value is exactly representable in BF16."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return bool(np.all((u & np.uint32(0xFFFF)) == 0))


def _rng(seed: int, name: str, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, _STREAM[name], sub])


def normal_bf16(seed: int, name: str, shape, std: float = 1.0, sub: int = 0) -> np.ndarray:
    """Seeded N(0, std^2) draw rounded to BF16.

    The array is drawn in slabs of 2^22 values; slab i comes from its own stream
    default_rng([seed, stream_id, sub, i]), so slabs are drawn in parallel and
    the result does not depend on the thread count.
    """
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    slab = 1 << 22
    nslab = (n + slab - 1) // slab

    def one(i):
        o = i * slab
        m = min(slab, n - o)
        v = np.random.default_rng([seed, _STREAM[name], sub, i]).standard_normal(m, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[o:o + m] = bf16_round(v)

    if nslab <= 1:
        for i in range(nslab):
            one(i)
    else:
        import concurrent.futures as cf
        import os
        with cf.ThreadPoolExecutor(max_workers=min(nslab, os.cpu_count() or 1, 32)) as ex:
            list(ex.map(one, range(nslab)))
    return out.reshape(shape)


# ----------------------------------------------------------------------------
# prefill inputs
# ----------------------------------------------------------------------------

def prefill_queries(cfg: Config, q0: int = 0, nq: int | None = None) -> dict:
    """Query-side inputs for queries [q0, q0+nq) of every sequence.

    Rows of a query array are drawn per query position, so a chunk of queries
    has the same bits whether drawn alone or as part of the whole sequence.
    """
    if nq is None:
        nq = cfg.T - q0
    B = cfg.B
    q_idx = np.empty((B, nq, cfg.H_I, cfg.D_I), np.uint16)
    w = np.empty((B, nq, cfg.H_I), np.uint16)
    q_lat = np.empty((B, nq, cfg.H, R_LAT), np.uint16)
    blk = 256  # query rows per draw block (sub-stream = block number)
    jobs = [(b, t0) for b in range(B) for t0 in range((q0 // blk) * blk, q0 + nq, blk)]

    def one(job):
        b, t0 = job
        sub = b * (1 << 20) + t0 // blk
        a = normal_bf16(cfg.seed, "q_idx", (blk, cfg.H_I, cfg.D_I), sub=sub)
        c = normal_bf16(cfg.seed, "w", (blk, cfg.H_I), sub=sub)
        d = normal_bf16(cfg.seed, "q_lat", (blk, cfg.H, R_LAT), sub=sub)
        lo, hi = max(t0, q0), min(t0 + blk, q0 + nq)
        q_idx[b, lo - q0:hi - q0] = a[lo - t0:hi - t0]
        w[b, lo - q0:hi - q0] = c[lo - t0:hi - t0]
        q_lat[b, lo - q0:hi - q0] = d[lo - t0:hi - t0]

    import concurrent.futures as cf
    import os
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 1, 16)) as ex:
        list(ex.map(one, jobs))
    return {"q_idx": q_idx, "w": w, "q_lat": q_lat}


def prefill_keys(cfg: Config, S: int | None = None) -> dict:
    """Key-side inputs: LayerNorm'd indexer keys [B,S,D_I] and latent rows [B,S,576]."""
    S = cfg.T if S is None else S
    k_idx = normal_bf16(cfg.seed, "k_idx", (cfg.B, S, cfg.D_I))
    kv = normal_bf16(cfg.seed, "kv", (cfg.B, S, R_LAT))
    return {"k_idx": k_idx, "kv": kv}


def gate_inputs(cfg: Config, N: int) -> dict:
    """Gate inputs: x [N,hid], W_g [H*dv, hid] (row = output feature), W_uv [H, dv, 512]."""
    x = normal_bf16(cfg.seed, "x", (N, cfg.hid))
    W_g = normal_bf16(cfg.seed, "W_g", (cfg.H * cfg.dv, cfg.hid), std=0.02)
    W_uv = normal_bf16(cfg.seed, "W_uv", (cfg.H, cfg.dv, V_LAT), std=0.02)
    return {"x": x, "W_g": W_g, "W_uv": W_uv}


def prefill(cfg: Config) -> dict:
    """All inputs of a single (unchunked) prefill: q_start = 0, kv_len = T."""
    d = prefill_queries(cfg)
    d.update(prefill_keys(cfg))
    d["q_start"] = np.zeros(cfg.B, np.int32)
    d["kv_len"] = np.full(cfg.B, cfg.T, np.int32)
    return d


# ----------------------------------------------------------------------------
# paged caches
# ----------------------------------------------------------------------------

def page_table(seed: int, lens: np.ndarray, page: int = PAGE, spare: int = 0):
    """Seeded random assignment of physical pages to the logical pages of each sequence.

    Returns (block_table [B, max_pages] int32, num_pages).  Unused table slots
    hold -1.  ``spare`` extra physical pages are left unassigned.
    """
    lens = np.asarray(lens, dtype=np.int64)
    npg = (lens + page - 1) // page
    total = int(npg.sum()) + spare
    perm = _rng(seed, "pages").permutation(total).astype(np.int32)
    maxp = int(npg.max()) if len(npg) else 0
    bt = np.full((len(lens), max(maxp, 1)), -1, np.int32)
    o = 0
    for b, n in enumerate(npg):
        bt[b, :n] = perm[o:o + n]
        o += int(n)
    return bt, total


def to_pages(logical: np.ndarray, lens: np.ndarray, block_table: np.ndarray, num_pages: int,
             page: int = PAGE) -> np.ndarray:
    """Scatter logical rows [B, S, W] into a page pool [num_pages, page, W] (layout only)."""
    B, S, W = logical.shape
    pool = np.zeros((num_pages, page, W), logical.dtype)
    for b in range(B):
        L = int(lens[b])
        for p in range((L + page - 1) // page):
            n = min(page, L - p * page)
            pool[block_table[b, p], :n] = logical[b, p * page:p * page + n]
    return pool


def from_pages(pool: np.ndarray, block_table: np.ndarray, b: int, L: int, page: int = PAGE) -> np.ndarray:
    """Logical rows [L, W] of sequence b read back from a page pool (layout only)."""
    idx = np.arange(L)
    return pool[block_table[b, idx // page], idx % page]


def decode_lengths(cfg: Config) -> np.ndarray:
    return _rng(cfg.seed, "lens").integers(cfg.L_min, cfg.L_max + 1, size=cfg.B).astype(np.int32)


def decode(cfg: Config) -> dict:
    """Decode inputs: one query per request at position L-1 over paged caches of length L.

    The page pools are drawn directly in physical order (entries are i.i.d., so
    this has the same distribution as paging a logically drawn cache).
    """
    lens = decode_lengths(cfg)
    bt, num_pages = page_table(cfg.seed, lens)
    k_pool = normal_bf16(cfg.seed, "k_idx", (num_pages, PAGE, cfg.D_I))
    kv_pool = normal_bf16(cfg.seed, "kv", (num_pages, PAGE, R_LAT))
    q = prefill_queries(Config(**{**cfg.__dict__, "T": 1}), 0, 1)
    return {
        "q_idx": q["q_idx"], "w": q["w"], "q_lat": q["q_lat"],
        "k_pool": k_pool, "kv_pool": kv_pool, "block_table": bt, "num_pages": num_pages,
        "q_start": (lens - 1).astype(np.int32), "kv_len": lens,
    }


def chunked(cfg: Config, c: int) -> dict:
    """Chunk c of a chunked prefill: queries [c*chunk, (c+1)*chunk) over a paged cache
    holding keys [0, (c+1)*chunk).  The cache pages are those of the whole sequence
    (the tail beyond (c+1)*chunk is simply not yet visible)."""
    assert cfg.chunk > 0
    q0 = c * cfg.chunk
    S = cfg.T
    keys = prefill_keys(cfg, S)
    lens = np.full(cfg.B, S, np.int64)
    bt, num_pages = page_table(cfg.seed, lens)
    d = prefill_queries(cfg, q0, cfg.chunk)
    d["k_logical"], d["kv_logical"] = keys["k_idx"], keys["kv"]
    d["k_pool"] = to_pages(keys["k_idx"], lens, bt, num_pages)
    d["kv_pool"] = to_pages(keys["kv"], lens, bt, num_pages)
    d["block_table"], d["num_pages"] = bt, num_pages
    d["q_start"] = np.full(cfg.B, q0, np.int32)
    d["kv_len"] = np.full(cfg.B, q0 + cfg.chunk, np.int32)
    return d


def append_inputs(seed: int, B: int, Tq: int, D_I: int) -> dict:
    """New tokens for the cache append: raw indexer keys k_pre [B, Tq, D_I] FP32
    (each row N(mu, sigma^2) with its own mu ~ U(-2, 2) and sigma ~ U(0.2, 4), so
    that centring and scaling both matter) and latent rows kv_new [B, Tq, 576]
    BF16 ~ N(0, 1)."""
    r = _rng(seed, "k_pre")
    mu = r.uniform(-2.0, 2.0, (B, Tq, 1))
    sigma = r.uniform(0.2, 4.0, (B, Tq, 1))
    k_pre = (r.standard_normal((B, Tq, D_I)) * sigma + mu).astype(np.float32)
    kv_new = normal_bf16(seed, "kv_new", (B, Tq, R_LAT))
    return {"k_pre": k_pre, "kv_new": kv_new}
