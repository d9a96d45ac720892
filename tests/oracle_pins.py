"""Pins that tie the CPU oracle to facts fixed outside itself.

Each ``pin_*`` function takes a loaded oracle library and raises
AssertionError when the oracle disagrees with a hand-worked example, a closed
form, an invariant, a library routine or a brute force on tiny inputs.  The
same functions run against the real oracle (test_oracle_pins.py) and against
copies with a planted mistake (test_oracle_mutants.py), which must each fail at
least one pin.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
from workloads import bf16_round, bf16_to_f32, normal_bf16

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
SCALE = 1.0 / math.sqrt(192.0)


def _bf(a):
    a = np.asarray(a, np.float32)
    h = bf16_round(a)
    assert np.array_equal(bf16_to_f32(h), a), "fixture value not exact in BF16"
    return h


# ----------------------------------------------------------------------------
# indexer
# ----------------------------------------------------------------------------

def pin_indexer_worked_example(lib):
    """Hand-worked example in tests/golden/indexer_worked.json."""
    g = json.load(open(os.path.join(GOLDEN, "indexer_worked.json")))
    q = np.array(g["q"], np.float32)              # [H_I, D_I]
    T = len(g["k"])
    q_idx = _bf(np.broadcast_to(q, (1, T) + q.shape).copy())
    w = _bf(np.broadcast_to(np.array(g["w"], np.float32), (1, T, q.shape[0])).copy())
    k = _bf(np.array(g["k"], np.float32)[None])
    qs, kl = np.zeros(1, np.int32), np.full(1, T, np.int32)
    sc = oracle.indexer_scores(q_idx, w, k, qs, kl, lib=lib)
    for t in range(T):
        for s in range(T):
            e = g["scores"][t][s]
            if e is None:
                assert math.isnan(sc[t, s]), (t, s, sc[t, s])
            else:
                assert sc[t, s] == e, (t, s, sc[t, s], e)
    idx, kth = oracle.topk(sc, np.arange(1, T + 1, dtype=np.int32), g["topk"], lib=lib)
    for t in range(T):
        got = [int(v) for v in idx[t] if v >= 0]
        assert sorted(got) == sorted(g["selected"][t]), (t, got)
        if g["kth"][t] is None:
            assert kth[t] == -math.inf
        else:
            assert kth[t] == g["kth"][t]


def pin_indexer_single_head_is_relu_dot(lib):
    """H_I = 1, w = 1 reduces to ReLU(q.k): compare with a numpy matmul."""
    rng = np.random.default_rng(7)
    T, D = 40, 64
    q = bf16_round(rng.standard_normal((1, T, 1, D), dtype=np.float32))
    k = bf16_round(rng.standard_normal((1, T, D), dtype=np.float32))
    w = bf16_round(np.ones((1, T, 1), np.float32))
    sc = oracle.indexer_scores(q, w, k, np.zeros(1, np.int32), np.full(1, T, np.int32), lib=lib)
    ref = np.maximum(bf16_to_f32(q[0, :, 0]).astype(np.float64)
                     @ bf16_to_f32(k[0]).astype(np.float64).T, 0.0)
    for t in range(T):
        np.testing.assert_allclose(sc[t, :t + 1], ref[t, :t + 1], rtol=1e-12, atol=1e-12)
        assert np.all(np.isnan(sc[t, t + 1:]))


def pin_indexer_invariances(lib):
    """Permuting heads (q and w together) leaves scores unchanged; doubling w doubles
    them exactly; a head whose weight is negative lowers the score."""
    cfg_T, H, D = 24, 4, 64
    q = normal_bf16(3, "q_idx", (1, cfg_T, H, D))
    w = normal_bf16(3, "w", (1, cfg_T, H))
    k = normal_bf16(3, "k_idx", (1, cfg_T, D))
    qs, kl = np.zeros(1, np.int32), np.full(1, cfg_T, np.int32)
    base = oracle.indexer_scores(q, w, k, qs, kl, lib=lib)
    perm = np.array([2, 0, 3, 1])
    sc_p = oracle.indexer_scores(q[:, :, perm], w[:, :, perm], k, qs, kl, lib=lib)
    np.testing.assert_allclose(sc_p, base, rtol=1e-12, atol=1e-12, equal_nan=True)
    w2 = bf16_round(bf16_to_f32(w) * 2.0)
    sc2 = oracle.indexer_scores(q, w2, k, qs, kl, lib=lib)
    np.testing.assert_array_equal(sc2, 2.0 * base)
    # all weights negative and all dots positive -> strictly negative scores
    qpos = bf16_round(np.abs(bf16_to_f32(q)) + 0.5)
    kpos = bf16_round(np.abs(bf16_to_f32(k)) + 0.5)
    wneg = bf16_round(-np.abs(bf16_to_f32(w)) - 0.25)
    scn = oracle.indexer_scores(qpos, wneg, kpos, qs, kl, lib=lib)
    for t in range(cfg_T):
        assert np.all(scn[t, :t + 1] < 0)


def pin_indexer_relu_clips(lib):
    """When every q.k is negative the ReLU zeroes every head: scores are exactly 0,
    whatever the (possibly negative) head weights."""
    T, H, D = 16, 4, 64
    q = bf16_round(np.full((1, T, H, D), 0.5, np.float32))
    k = bf16_round(-np.abs(bf16_to_f32(normal_bf16(5, "k_idx", (1, T, D)))) - 0.125)
    w = normal_bf16(5, "w", (1, T, H))
    sc = oracle.indexer_scores(q, w, k, np.zeros(1, np.int32), np.full(1, T, np.int32), lib=lib)
    for t in range(T):
        assert np.all(sc[t, :t + 1] == 0.0)


def pin_indexer_causal_window(lib):
    """Query i of a chunk sits at q_start+i and scores keys 0..q_start+i (self included)."""
    T, H, D = 32, 2, 64
    q_start = 20
    q = normal_bf16(9, "q_idx", (1, 4, H, D))
    w = normal_bf16(9, "w", (1, 4, H))
    k = normal_bf16(9, "k_idx", (1, T, D))
    sc = oracle.indexer_scores(q, w, k, np.array([q_start], np.int32),
                               np.array([q_start + 4], np.int32), lib=lib)
    for i in range(4):
        t = q_start + i
        assert not np.isnan(sc[i, t]), "the query's own key must be scored"
        assert np.all(~np.isnan(sc[i, :t + 1]))
        assert np.all(np.isnan(sc[i, t + 1:]))
        # brute force for key s = t
        qq = bf16_to_f32(q[0, i]).astype(np.float64)
        kk = bf16_to_f32(k[0, t]).astype(np.float64)
        ww = bf16_to_f32(w[0, i]).astype(np.float64)
        e = sum(ww[j] * max(0.0, float(qq[j] @ kk)) for j in range(H))
        assert abs(sc[i, t] - e) <= 1e-12 * max(1.0, abs(e))


# ----------------------------------------------------------------------------
# top-k
# ----------------------------------------------------------------------------

def pin_topk_planted_permutation(lib):
    """H_I = 1, w = 1, q = e_0 and k[s,0] = a seeded permutation of 1..n: the score of
    key s is its planted value, so the top-k set is known by construction."""
    n, D, k = 200, 64, 50
    vals = np.random.default_rng(11).permutation(n).astype(np.float32) + 1.0  # exact in BF16
    kk = np.zeros((1, n, D), np.float32)
    kk[0, :, 0] = vals
    q = np.zeros((1, n, 1, D), np.float32)
    q[..., 0] = 1.0
    w = np.ones((1, n, 1), np.float32)
    idx, kth, sc, nv = oracle.indexer_topk(_bf(q), _bf(w), _bf(kk), np.zeros(1, np.int32),
                                           np.full(1, n, np.int32), k, lib=lib)
    for t in range(n):
        if t + 1 <= k:
            expect = set(range(t + 1))
        else:
            order = np.argsort(-vals[:t + 1], kind="stable")
            expect = set(order[:k].tolist())
            assert kth[t] == np.sort(vals[:t + 1])[::-1][k - 1]
        got = set(int(v) for v in idx[t] if v >= 0)
        assert got == expect, t
        assert len([v for v in idx[t] if v >= 0]) == min(t + 1, k)


def pin_topk_brute_force_rank(lib):
    """Brute force on tiny rows with many exact ties: key s is selected iff fewer than
    k keys beat it, where s' beats s when its score is larger, or equal with s' < s."""
    rng = np.random.default_rng(13)
    n_rows, S, k = 60, 30, 7
    scores = rng.integers(-3, 4, size=(n_rows, S)).astype(np.float64)
    n_valid = rng.integers(1, S + 1, size=n_rows).astype(np.int32)
    idx, kth = oracle.topk(scores, n_valid, k, lib=lib)
    for r in range(n_rows):
        n = int(n_valid[r])
        expect = set()
        for s in range(n):
            beats = sum(1 for s2 in range(n)
                        if scores[r, s2] > scores[r, s] or (scores[r, s2] == scores[r, s] and s2 < s))
            if beats < k:
                expect.add(s)
        got = [int(v) for v in idx[r] if v >= 0]
        assert len(got) == len(set(got)) == min(n, k)
        assert set(got) == expect, r
        assert np.all(idx[r, len(got):] == -1)
        if n > k:
            assert kth[r] == sorted(scores[r, :n], reverse=True)[k - 1]


def pin_topk_all_equal_takes_lowest(lib):
    """All scores equal: the tie rule keeps the k smallest key indices."""
    S, k = 64, 10
    scores = np.full((1, S), 1.5)
    idx, kth = oracle.topk(scores, np.array([S], np.int32), k, lib=lib)
    assert sorted(int(v) for v in idx[0]) == list(range(k))
    assert kth[0] == 1.5


# ----------------------------------------------------------------------------
# sparse / dense latent attention
# ----------------------------------------------------------------------------

def _mla_inputs(seed, T, H):
    q = normal_bf16(seed, "q_lat", (1, T, H, 576))
    kv = normal_bf16(seed, "kv", (1, T, 576))
    return q, kv, np.zeros(1, np.int32), np.full(1, T, np.int32)


def pin_mla_single_key(lib):
    """One selected key: the output is that key's 512 value dims exactly, lse = its logit."""
    T, H = 12, 3
    q, kv, qs, kl = _mla_inputs(21, T, H)
    idx = np.full((1, T, 4), -1, np.int32)
    sel = [min(t, (5 * t) % (t + 1)) for t in range(T)]
    idx[0, :, 2] = sel
    o, lse = oracle.sparse_mla(q, kv, idx, qs, kl, SCALE, lib=lib)
    kvf = bf16_to_f32(kv[0]).astype(np.float64)
    for t in range(T):
        s = sel[t]
        for h in range(H):
            np.testing.assert_array_equal(o[t, h], kvf[s, :512])
            z = float(bf16_to_f32(q[0, t, h]).astype(np.float64) @ kvf[s]) * SCALE
            assert abs(lse[t, h] - z) <= 1e-12 * max(1.0, abs(z))


def pin_mla_uniform_logits(lib):
    """q = 0 makes every logit 0: output = mean of the selected values, lse = ln(n)."""
    T, H = 10, 2
    _, kv, qs, kl = _mla_inputs(22, T, H)
    q = np.zeros((1, T, H, 576), np.uint16)
    o, lse = oracle.dense_mla(q, kv, qs, kl, SCALE, lib=lib)
    kvf = bf16_to_f32(kv[0]).astype(np.float64)
    for t in range(T):
        np.testing.assert_allclose(o[t, 0], kvf[:t + 1, :512].mean(0), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[t], math.log(t + 1), rtol=0, atol=1e-14)


def pin_mla_two_keys_closed_form(lib):
    """Two keys whose logits differ by a known amount: p0 = 1 / (1 + exp(z1 - z0)).
    Key 0 has 1 in a rope dim and key 1 has 0 there, so the rope dims must enter the
    logits, and the 1/sqrt(192) scale is checked exactly."""
    H = 1
    q = np.zeros((1, 2, H, 576), np.float32)
    q[0, 1, 0, 540] = 16.0            # a rope dim (>= 512)
    kv = np.zeros((1, 2, 576), np.float32)
    kv[0, 0, 540] = 1.0
    kv[0, 0, :512] = np.linspace(-1, 1, 512, dtype=np.float32)
    kv[0, 1, :512] = 0.5
    qh, kvh = _bf(q), bf16_round(kv)
    o, lse = oracle.dense_mla(qh, kvh, np.zeros(1, np.int32), np.full(1, 2, np.int32), SCALE,
                              lib=lib)
    z0 = 16.0 / math.sqrt(192.0)
    p0 = 1.0 / (1.0 + math.exp(-z0))
    v = bf16_to_f32(kvh[0]).astype(np.float64)
    np.testing.assert_allclose(o[1, 0], p0 * v[0, :512] + (1 - p0) * v[1, :512], rtol=1e-13,
                               atol=1e-15)
    assert abs(lse[1, 0] - (z0 + math.log1p(math.exp(-z0)))) < 1e-13


def pin_mla_dense_matches_library_sdpa(lib):
    """Dense causal MLA against torch's scaled_dot_product_attention in float64 (CPU),
    with the latent rows as a single shared key/value head (value = first 512 dims)."""
    import torch
    T, H = 20, 4
    q, kv, qs, kl = _mla_inputs(23, T, H)
    o, lse = oracle.dense_mla(q, kv, qs, kl, SCALE, lib=lib)
    qf = torch.from_numpy(bf16_to_f32(q[0]).astype(np.float64))        # [T,H,576]
    kf = torch.from_numpy(bf16_to_f32(kv[0]).astype(np.float64))       # [T,576]
    Q = qf.permute(1, 0, 2)[None]                                       # [1,H,T,576]
    K = kf[None, None].expand(1, H, T, 576)
    V = kf[None, None, :, :512].expand(1, H, T, 512)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=SCALE)
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    logits = (Q @ K.transpose(-1, -2)) * SCALE
    mask = torch.ones(T, T, dtype=torch.bool).tril()
    ref_lse = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1)[0].T
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def pin_mla_sparse_full_set_equals_dense(lib):
    """T <= k: every causal key is selected, so sparse MLA equals dense causal MLA
    ("Kimi-K3.1-Pro", Implementation Limits, bullet 4).  The index order and -1
    padding must not matter."""
    T, H, k = 24, 3, 32
    q, kv, qs, kl = _mla_inputs(24, T, H)
    rng = np.random.default_rng(5)
    idx = np.full((1, T, k), -1, np.int32)
    for t in range(T):
        pos = rng.permutation(k)[:t + 1]
        idx[0, t, pos] = rng.permutation(t + 1)
    o_s, l_s = oracle.sparse_mla(q, kv, idx, qs, kl, SCALE, lib=lib)
    o_d, l_d = oracle.dense_mla(q, kv, qs, kl, SCALE, lib=lib)
    np.testing.assert_allclose(o_s, o_d, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l_s, l_d, rtol=1e-13, atol=1e-13)


def pin_mla_subset_brute_force(lib):
    """A strict subset of keys: brute-force softmax over exactly that subset."""
    T, H = 16, 2
    q, kv, qs, kl = _mla_inputs(25, T, H)
    sel = {t: sorted({0, t, t // 2, (3 * t) // 4}) for t in range(T)}
    idx = np.full((1, T, 4), -1, np.int32)
    for t in range(T):
        idx[0, t, :len(sel[t])] = sel[t]
    o, lse = oracle.sparse_mla(q, kv, idx, qs, kl, SCALE, lib=lib)
    kvf = bf16_to_f32(kv[0]).astype(np.float64)
    for t in (3, 9, 15):
        for h in range(H):
            qv = bf16_to_f32(q[0, t, h]).astype(np.float64)
            z = np.array([qv @ kvf[s] for s in sel[t]]) * SCALE
            e = np.exp(z - z.max())
            ref = (e[:, None] * kvf[sel[t], :512]).sum(0) / e.sum()
            np.testing.assert_allclose(o[t, h], ref, rtol=1e-12, atol=1e-13)
            assert abs(lse[t, h] - (z.max() + math.log(e.sum()))) < 1e-12


def pin_mla_rejects_noncausal_index(lib):
    """An index beyond the query's position is not a causal key: the oracle refuses."""
    T, H = 8, 1
    q, kv, qs, kl = _mla_inputs(26, T, H)
    idx = np.full((1, T, 2), -1, np.int32)
    idx[0, 3, 0] = 5
    try:
        oracle.sparse_mla(q, kv, idx, qs, kl, SCALE, lib=lib)
    except oracle.OracleError:
        return
    raise AssertionError("non-causal index accepted")


def pin_absorbed_equals_explicit(lib):
    """The absorbed latent form (q_lat = [W_UK^T q_nope | q_pe], values = c_kv, then
    W_UV) equals explicit per-head expansion of K and V ("Kimi-K3.1-Pro",
    Implementation Limits, bullet 2).  Inputs are chosen so q_lat is exact in BF16."""
    rng = np.random.default_rng(31)
    H, dn, dr, R, dv, S, n = 2, 128, 64, 512, 128, 9, 5
    W_UK = rng.integers(-1, 2, size=(H, dn, R)).astype(np.float64) * (rng.random((H, dn, R)) < 0.05)
    q_nope = rng.integers(-2, 3, size=(n, H, dn)).astype(np.float64) * 0.125
    q_pe = bf16_to_f32(bf16_round(rng.standard_normal((n, H, dr), dtype=np.float32))).astype(np.float64)
    c_kv = bf16_to_f32(bf16_round(rng.standard_normal((S, R), dtype=np.float32))).astype(np.float64)
    k_pe = bf16_to_f32(bf16_round(rng.standard_normal((S, dr), dtype=np.float32))).astype(np.float64)
    W_UV = rng.standard_normal((H, dv, R)) * 0.02
    q_abs = np.einsum("nha,har->nhr", q_nope, W_UK)
    q_lat = np.concatenate([q_abs, q_pe], axis=-1)                     # [n,H,576]
    q_lat_bf = bf16_round(q_lat.astype(np.float32))
    assert np.array_equal(bf16_to_f32(q_lat_bf).astype(np.float64), q_lat)
    kv = np.concatenate([c_kv, k_pe], axis=-1)
    kv_bf = bf16_round(kv.astype(np.float32))
    sel = np.full((n, 6), -1, np.int32)
    for i in range(n):  # query i sits at position S-n+i
        sel[i, :4] = np.sort(rng.choice(S - n + i + 1, 4, replace=False))
    o_lat, _ = oracle.sparse_mla(q_lat_bf[None], kv_bf[None], sel[None],
                                 np.array([S - n], np.int32), np.array([S], np.int32),
                                 SCALE, lib=lib)
    absorbed = np.einsum("her,nhr->nhe", W_UV, o_lat)
    explicit = oracle.explicit_mla(q_nope, q_pe, W_UK, W_UV, c_kv, k_pe, sel, SCALE, lib=lib)
    np.testing.assert_allclose(absorbed, explicit, rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------------------
# gate
# ----------------------------------------------------------------------------

def _gate_inputs(seed, N, hid, H, dv):
    x = normal_bf16(seed, "x", (N, hid))
    W_g = normal_bf16(seed, "W_g", (H * dv, hid), std=0.02)
    W_uv = normal_bf16(seed, "W_uv", (H, dv, 512), std=0.02)
    o_lat = np.random.default_rng(seed).standard_normal((N, H, 512)) * 0.1
    return x, W_g, W_uv, o_lat


def pin_gate_zero_weight_is_half(lib):
    """W_g = 0 gives sigma(0) = 1/2: out = 0.5 * (W_uv_h . o_lat_h)."""
    N, hid, H, dv = 6, 64, 3, 16
    x, _, W_uv, o_lat = _gate_inputs(41, N, hid, H, dv)
    W_g = np.zeros((H * dv, hid), np.uint16)
    out = oracle.gate(x, W_g, o_lat, W_uv, lib=lib)
    u = np.einsum("her,nhr->nhe", bf16_to_f32(W_uv).astype(np.float64), o_lat).reshape(N, H * dv)
    np.testing.assert_allclose(out, 0.5 * u, rtol=1e-13, atol=1e-15)


def pin_gate_matches_library(lib):
    """Against torch.sigmoid / torch matmul in float64 on the CPU."""
    import torch
    N, hid, H, dv = 7, 96, 2, 32
    x, W_g, W_uv, o_lat = _gate_inputs(42, N, hid, H, dv)
    out = oracle.gate(x, W_g, o_lat, W_uv, lib=lib)
    X = torch.from_numpy(bf16_to_f32(x).astype(np.float64))
    G = torch.from_numpy(bf16_to_f32(W_g).astype(np.float64))
    U = torch.from_numpy(bf16_to_f32(W_uv).astype(np.float64))
    O = torch.from_numpy(o_lat)
    ref = torch.sigmoid(X @ G.T) * torch.einsum("her,nhr->nhe", U, O).reshape(N, H * dv)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-14)


def pin_gate_row_subset(lib):
    """Evaluating a subset of rows gives the same values as the full evaluation."""
    N, hid, H, dv = 9, 32, 2, 8
    x, W_g, W_uv, o_lat = _gate_inputs(43, N, hid, H, dv)
    full = oracle.gate(x, W_g, o_lat, W_uv, lib=lib)
    rows = np.array([8, 0, 4])
    part = oracle.gate(x, W_g, o_lat, W_uv, rows=rows, lib=lib)
    np.testing.assert_array_equal(part, full[rows])




# ---------------------------------------------------------------------------
# Indexer-key LayerNorm, BF16 rounding and the cache append
# ("Kimi K3.1 Pro" archdiff blueprint: LayerNorm on the indexer key;
#  KimiK3TextConfig rms_norm_eps)
# ---------------------------------------------------------------------------

def pin_layernorm_worked_example(lib):
    g = json.load(open(os.path.join(GOLDEN, "layernorm_worked.json")))
    y = oracle.layernorm(np.array([g["x"]], np.float32), g["eps"], lib)[0]
    assert np.max(np.abs(y - np.array(g["y"]))) < g["y_tol"], y
    bits = oracle.bf16_rne(y, lib)
    assert [int(b, 16) for b in g["bf16"]] == bits.tolist(), [hex(b) for b in bits]


def pin_layernorm_moments_closed_form(lib):
    """mean(y) = 0 and mean(y^2) = var/(var + eps) for every row."""
    rng = np.random.default_rng(31)
    x = (rng.standard_normal((50, 128)) * rng.uniform(0.01, 5, (50, 1)) + rng.uniform(-3, 3, (50, 1)))
    x = x.astype(np.float32)
    eps = 1e-5
    y = oracle.layernorm(x, eps, lib)
    xd = x.astype(np.float64)
    var = xd.var(axis=1)
    assert np.max(np.abs(y.mean(axis=1))) < 1e-12
    np.testing.assert_allclose((y * y).mean(axis=1), var / (var + eps), rtol=1e-12)


def pin_layernorm_constant_row_is_zero(lib):
    y = oracle.layernorm(np.full((3, 64), 2.75, np.float32), 1e-5, lib)
    assert np.all(y == 0.0)


def pin_layernorm_matches_library(lib):
    import torch
    rng = np.random.default_rng(32)
    x = rng.standard_normal((20, 64)).astype(np.float32) * 3 + 1
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x.astype(np.float64)), (64,), eps=1e-5)
    np.testing.assert_allclose(oracle.layernorm(x, 1e-5, lib), ref.numpy(), rtol=0, atol=1e-12)


def pin_bf16_rounding_definition(lib):
    """Ties to even at the two midpoints next to 1.0, and agreement with torch's
    float32 -> bfloat16 conversion on values a float32 holds exactly."""
    import torch
    b = oracle.bf16_rne(np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -1.5, 0.0, -0.0]), lib)
    assert b.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xBFC0, 0x0000, 0x8000], [hex(v) for v in b]
    rng = np.random.default_rng(33)
    v = (rng.standard_normal(4000) * np.exp(rng.uniform(-20, 20, 4000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_rne(v.astype(np.float64), lib), ref)


def pin_cache_append_places_rows(lib):
    """Rows land at q_start[b]+i through the block table; nothing else changes."""
    rng = np.random.default_rng(34)
    B, Tq, D, page = 2, 3, 64, 64
    bt = np.array([[3, 0], [1, 2]], np.int32)
    pool_k = rng.integers(0, 65535, (4, page, D), dtype=np.uint16)
    pool_v = rng.integers(0, 65535, (4, page, 576), dtype=np.uint16)
    k_pre = rng.standard_normal((B, Tq, D)).astype(np.float32)
    kv_new = rng.integers(0, 65535, (B, Tq, 576), dtype=np.uint16)
    q_start = np.array([62, 10], np.int32)
    kc, vc, k_ln = oracle.cache_append(k_pre, kv_new, q_start, 1e-5, pool_k, pool_v, bt, bt, page, lib)
    touched = {(3, 62), (3, 63), (0, 0), (1, 10), (1, 11), (1, 12)}
    for p_ in range(4):
        for s in range(page):
            if (p_, s) not in touched:
                assert np.array_equal(kc[p_, s], pool_k[p_, s]) and np.array_equal(vc[p_, s], pool_v[p_, s])
    assert np.array_equal(vc[0, 0], kv_new[0, 2]) and np.array_equal(vc[1, 12], kv_new[1, 2])
    assert np.array_equal(kc[3, 63], oracle.bf16_rne(k_ln[0, 1], lib))


# ---------------------------------------------------------------------------
# Learnable sink ("Kimi K3.1 Pro" archdiff blueprint, "Output gate + sink")
# ---------------------------------------------------------------------------

def pin_sink_minus_infinity_is_no_sink(lib):
    T, H = 9, 3
    q, kv, qs, kl = _mla_inputs(61, T, H)
    idx = np.tile(np.arange(T, dtype=np.int32), (1, T, 1))
    idx[0] = np.where(idx[0] <= np.arange(T)[:, None], idx[0], -1)
    a = oracle.sparse_mla(q, kv, idx, qs, kl, SCALE, lib=lib)
    b = oracle.sparse_mla(q, kv, idx, qs, kl, SCALE, lib=lib, sink=np.full(H, -np.inf))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def pin_sink_single_key_closed_form(lib):
    """One key with logit z and a sink s: o = v * sigma(z - s), lse = log(e^z + e^s)."""
    T, H = 6, 2
    q, kv, qs, kl = _mla_inputs(62, T, H)
    idx = np.full((1, T, 4), -1, np.int32)
    idx[0, :, 1] = np.arange(T) // 2
    sink = np.array([0.7, -3.5])
    o, lse = oracle.sparse_mla(q, kv, idx, qs, kl, SCALE, lib=lib, sink=sink)
    kvf = bf16_to_f32(kv[0]).astype(np.float64)
    for t in range(T):
        s_ = t // 2
        for h in range(H):
            z = float(bf16_to_f32(q[0, t, h]).astype(np.float64) @ kvf[s_]) * SCALE
            p = 1.0 / (1.0 + math.exp(sink[h] - z))
            np.testing.assert_allclose(o[t, h], p * kvf[s_, :512], rtol=1e-12, atol=1e-15)
            want = max(z, sink[h]) + math.log1p(math.exp(-abs(z - sink[h])))
            assert abs(lse[t, h] - want) < 1e-12


def pin_sink_uniform_logits(lib):
    """q = 0: n keys of logit 0 and a sink s give o = mean(v) * n / (n + e^s) and
    lse = log(n + e^s); with no attended key, o = 0 and lse = s."""
    T, H = 7, 1
    _, kv, qs, kl = _mla_inputs(63, T, H)
    q = np.zeros((1, T, H, 576), np.uint16)
    idx = np.full((1, T, T), -1, np.int32)
    for t in range(1, T):
        idx[0, t, :t] = np.arange(t)          # query t attends to keys 0..t-1; query 0 to none
    sink = np.array([1.25])
    o, lse = oracle.sparse_mla(q, kv, idx, qs, kl, SCALE, lib=lib, sink=sink)
    kvf = bf16_to_f32(kv[0]).astype(np.float64)
    assert np.all(o[0] == 0.0) and lse[0, 0] == 1.25
    for t in range(1, T):
        w = t / (t + math.exp(1.25))
        np.testing.assert_allclose(o[t, 0], kvf[:t, :512].mean(0) * w, rtol=1e-12, atol=1e-15)
        assert abs(lse[t, 0] - math.log(t + math.exp(1.25))) < 1e-12


def pin_sink_dominant_limit(lib):
    """A sink far above every logit takes all the weight: o = 0, lse = the sink
    (finite: the sink must enter the running maximum, not overflow e^{s - m})."""
    T, H = 4, 2
    q, kv, qs, kl = _mla_inputs(64, T, H)
    idx = np.zeros((1, T, 1), np.int32)
    o, lse = oracle.sparse_mla(q, kv, idx, qs, kl, SCALE, lib=lib, sink=np.array([1000.0, 1000.0]))
    assert np.all(o == 0.0)
    np.testing.assert_array_equal(lse, np.full((T, H), 1000.0))


# ----------------------------------------------------------------------------
# FP8 (E4M3) indexer variant
# ----------------------------------------------------------------------------

def _e4m3_grid():
    """The 127 finite non-negative E4M3 magnitudes, in code order."""
    g = json.load(open(os.path.join(GOLDEN, "e4m3_codes.json")))["codes"]
    assert g["0x7e"] == 448.0
    return oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def pin_e4m3_format_table(lib):
    """Hand-worked code values of the OFP8 E4M3 format (tests/golden/e4m3_codes.json)."""
    g = json.load(open(os.path.join(GOLDEN, "e4m3_codes.json")))["codes"]
    codes = np.array([int(k, 16) for k in g], np.uint8)
    vals = oracle.e4m3_decode(codes, lib=lib)
    for c, v, e in zip(codes, vals, g.values()):
        if e == "nan":
            assert math.isnan(v), (hex(c), v)
        else:
            assert v == e and math.copysign(1.0, v) == math.copysign(1.0, e), (hex(c), v, e)


def pin_e4m3_roundtrip_and_order(lib):
    """Every finite code encodes back to itself; magnitudes rise with the code."""
    allc = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_decode(allc, lib=lib)
    fin = ~np.isnan(v)
    assert fin.sum() == 254
    back = oracle.e4m3_encode(v[fin].astype(np.float32), lib=lib)
    assert np.array_equal(back, allc[fin])
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)


def pin_e4m3_rounding_matches_library(lib):
    """Round to nearest, ties to even, against torch's float8_e4m3fn cast (in
    range) and saturation to +-448 beyond it; midpoints and their neighbours."""
    import torch
    grid = _e4m3_grid()
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    xs = [grid.astype(np.float32), mids, np.nextafter(mids, np.float32(0)),
          np.nextafter(mids, np.float32(1e30))]
    rng = np.random.default_rng(81)
    xs.append((rng.standard_normal(4000) * 60).astype(np.float32))
    xs.append((rng.standard_normal(4000) * 0.01).astype(np.float32))
    x = np.concatenate(xs)
    x = np.concatenate([x, -x])
    inr = np.abs(x) < 464
    got = oracle.e4m3_encode(x, lib=lib)
    ref = torch.from_numpy(x[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[inr], ref), np.nonzero(got[inr] != ref)[0][:5]
    big = np.array([464.0, 1000.0, 3e38], np.float32)
    assert np.array_equal(oracle.e4m3_encode(big, lib=lib), [0x7E] * 3)
    assert np.array_equal(oracle.e4m3_encode(-big, lib=lib), [0xFE] * 3)
    # ties: midpoint of codes 0x38 / 0x39 goes to the even 0x38, of 0x39 / 0x3a to 0x3a
    assert list(oracle.e4m3_encode(np.array([1.0625, 1.1875, 2.0 ** -10], np.float32),
                                   lib=lib)) == [0x38, 0x3A, 0x00]


def pin_quant_fp8_definition(lib):
    """Per-row scale and codes recomputed with numpy float32 arithmetic and
    torch's E4M3 cast: scale = max(amax, 2^-100)/448, code = E4M3(x * (1/scale))."""
    import torch
    rng = np.random.default_rng(82)
    x = normal_bf16(82, "q_idx", (37, 128))
    x[3] = 0                                   # an all-zero row
    x[5] = bf16_round(np.full(128, -2.5, np.float32))
    x[7, :] = bf16_round((rng.standard_normal(128) * 1e-3).astype(np.float32))
    # rows where x * (1/scale) and x / scale round to different codes: the
    # pin fixes the two-step form (found by search over BF16 pairs)
    for r, (amax_, xv) in enumerate([(0.19140625, 0.08544921875), (0.26953125, 0.2021484375),
                                     (0.40625, 0.076171875)]):
        x[10 + r, :] = 0
        x[10 + r, :2] = bf16_round(np.array([amax_, xv], np.float32))
    codes, scale = oracle.quant_fp8(x, lib=lib)
    xf = bf16_to_f32(x)
    amax = np.max(np.abs(xf), axis=1).astype(np.float32)
    s_ref = np.maximum(amax, np.float32(2.0 ** -100)) / np.float32(448.0)
    assert np.array_equal(scale, s_ref.astype(np.float32))
    inv = (np.float32(1.0) / s_ref).astype(np.float32)
    t = (xf * inv[:, None]).astype(np.float32)
    t = np.clip(t, -448.0, 448.0)           # the saturation (values past 448 round to it)
    ref = torch.from_numpy(np.ascontiguousarray(t)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    assert np.all(codes[3] == 0)
    # the row maximum lands on +-448 (code 0x7e / 0xfe)
    for r in (0, 5, 7):
        assert (codes[r, np.argmax(np.abs(xf[r]))] & 0x7F) == 0x7E


def pin_indexer_fp8_equals_bf16_on_exact_values(lib):
    """With power-of-two scales the dequantised values are exact BF16 numbers,
    and the FP8 scores then equal the BF16 indexer's scores exactly."""
    rng = np.random.default_rng(83)
    B, T, H_I, D_I = 1, 24, 3, 16
    qc = rng.integers(0, 256, (B, T, H_I, D_I)).astype(np.uint8)
    kc = rng.integers(0, 256, (B, T, D_I)).astype(np.uint8)
    qc[(qc & 0x7F) == 0x7F] = 0x38            # no NaN codes
    kc[(kc & 0x7F) == 0x7F] = 0x40
    qs = (2.0 ** rng.integers(-6, 3, (B, T, H_I))).astype(np.float32)
    ks = (2.0 ** rng.integers(-6, 3, (B, T))).astype(np.float32)
    w = normal_bf16(83, "w", (B, T, H_I))
    qv = oracle.e4m3_decode(qc, lib=lib) * qs[..., None]
    kv = oracle.e4m3_decode(kc, lib=lib) * ks[..., None]
    q16, k16 = _bf(qv.astype(np.float32)), _bf(kv.astype(np.float32))
    q_start, kv_len = np.zeros(B, np.int32), np.full(B, T, np.int32)
    a = oracle.indexer_scores_fp8(qc, qs, w, kc, ks, q_start, kv_len, lib=lib)
    b = oracle.indexer_scores(q16, w, k16, q_start, kv_len, lib=lib)
    assert np.array_equal(np.isnan(a), np.isnan(b))
    assert np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])
    # the scales matter: doubling one key's scale doubles its column of scores
    ks2 = ks.copy()
    ks2[0, 5] *= 2
    c = oracle.indexer_scores_fp8(qc, qs, w, kc, ks2, q_start, kv_len, lib=lib)
    assert np.array_equal(c[5:, 5], 2 * a[5:, 5])
    assert np.array_equal(c[:, 6:], a[:, 6:], equal_nan=True)


# ----------------------------------------------------------------------------
# sparse MLA backward
# ----------------------------------------------------------------------------

def _bwd_case(seed, T, H, k, amp=0.25, full=False):
    """Float64 inputs with a random causal index set (or every causal key)."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, T, H, 576)) * amp
    kv = rng.standard_normal((1, T, 576)) * amp
    dO = rng.standard_normal((1, T, H, 512))
    idx = np.full((1, T, k), -1, np.int32)
    for t in range(T):
        c = np.arange(t + 1) if full else rng.permutation(t + 1)[:k]
        idx[0, t, :len(c)] = c
    return q, kv, dO, idx, np.zeros(1, np.int32), np.full(1, T, np.int32)


def pin_mla_f64_forward_matches_bf16_forward(lib):
    """The float64-input forward (the function the backward differentiates) agrees
    with the BF16-input forward on BF16 values."""
    T, H = 40, 8
    q = normal_bf16(91, "q_lat", (1, T, H, 576))
    kv = normal_bf16(91, "kv", (1, T, 576))
    rng = np.random.default_rng(91)
    idx = np.full((1, T, 16), -1, np.int32)
    for t in range(T):
        c = rng.permutation(t + 1)[:16]
        idx[0, t, :len(c)] = c
    qs, kl = np.zeros(1, np.int32), np.full(1, T, np.int32)
    o1, l1 = oracle.sparse_mla(q, kv, idx, qs, kl, SCALE, lib=lib)
    o2, l2 = oracle.sparse_mla_f64(q, kv, idx, qs, kl, SCALE, lib=lib)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)


def pin_mla_bwd_finite_differences(lib):
    """Central differences of sum(dO * o) through the float64 forward, at query
    and latent coordinates in the value dims and in the 64 k_pe dims."""
    q, kv, dO, idx, qs, kl = _bwd_case(92, 6, 2, 3, amp=0.5)
    scale = 0.3
    dq, dkv = oracle.sparse_mla_bwd(q, kv, idx, qs, kl, scale, dO, lib=lib)

    def loss(qq, kk):
        o, _ = oracle.sparse_mla_f64(qq, kk, idx, qs, kl, scale, lib=lib)
        return float(np.sum(o * dO.reshape(o.shape)))

    eps = 1e-6
    for (t, h, d) in [(5, 1, 3), (3, 0, 540), (4, 1, 511), (2, 0, 575)]:
        qp, qm = q.copy(), q.copy()
        qp[0, t, h, d] += eps
        qm[0, t, h, d] -= eps
        fd = (loss(qp, kv) - loss(qm, kv)) / (2 * eps)
        assert abs(fd - dq[0, t, h, d]) <= 1e-7 * max(1.0, abs(fd)), ("dq", t, h, d, fd, dq[0, t, h, d])
    used = sorted(set(int(v) for v in idx.ravel() if v >= 0))
    for (s, d) in [(used[0], 7), (used[1], 530), (used[-1], 200), (used[2], 575)]:
        kp, km = kv.copy(), kv.copy()
        kp[0, s, d] += eps
        km[0, s, d] -= eps
        fd = (loss(q, kp) - loss(q, km)) / (2 * eps)
        assert abs(fd - dkv[0, s, d]) <= 1e-7 * max(1.0, abs(fd)), ("dkv", s, d, fd, dkv[0, s, d])


def pin_mla_bwd_matches_library_autograd(lib):
    """With every causal key selected the sparse forward is dense causal attention;
    torch float64 autograd of that dense attention (K = the latent row, V = its
    first 512 dims, one shared tensor) gives the same gradients."""
    import torch
    T, H = 7, 3
    q, kv, dO, idx, qs, kl = _bwd_case(93, T, H, T, full=True)
    dq, dkv = oracle.sparse_mla_bwd(q, kv, idx, qs, kl, SCALE, dO, lib=lib)
    tq = torch.tensor(q[0].transpose(1, 0, 2), requires_grad=True)      # [H, T, 576]
    tk = torch.tensor(kv[0], requires_grad=True)                         # [T, 576]
    z = torch.einsum("htd,sd->hts", tq, tk) * SCALE
    mask = torch.triu(torch.ones(T, T, dtype=torch.bool), diagonal=1)
    pr = torch.softmax(z.masked_fill(mask, float("-inf")), dim=-1)
    o = torch.einsum("hts,sd->htd", pr, tk[:, :512])
    (o * torch.tensor(dO[0].transpose(1, 0, 2))).sum().backward()
    assert np.allclose(tq.grad.numpy().transpose(1, 0, 2), dq[0], rtol=0, atol=1e-10)
    assert np.allclose(tk.grad.numpy(), dkv[0], rtol=0, atol=1e-10)


def pin_mla_bwd_single_key_closed_form(lib):
    """One selected key per query: p = 1, so dq = 0, the k_pe dims get nothing,
    and the key's value dims receive the sum of the upstream gradients."""
    T, H = 9, 4
    q, kv, dO, _, qs, kl = _bwd_case(94, T, H, 1)
    idx = (np.arange(T) // 2).astype(np.int32).reshape(1, T, 1)   # query t selects key t // 2
    dq, dkv = oracle.sparse_mla_bwd(q, kv, idx, qs, kl, SCALE, dO, lib=lib)
    assert np.allclose(dq, 0.0, atol=1e-12)
    want = np.zeros((T, 512))
    for t in range(T):
        want[t // 2] += dO[0, t].sum(axis=0)
    assert np.allclose(dkv[0, :, :512], want, rtol=0, atol=1e-12)
    assert np.allclose(dkv[0, :, 512:], 0.0, atol=1e-12)


def pin_mla_bwd_sum_rules(lib):
    """Summed over keys: the k_pe-dim gradients cancel (sum_j dz_j = 0 per query
    head) and the value-dim gradients add up to sum_t,h dO (sum_j p_j = 1)."""
    T, H = 14, 3
    q, kv, dO, idx, qs, kl = _bwd_case(95, T, H, 5, amp=0.6)
    idx[0, 6] = -1                                  # a query with no valid entry
    _, dkv = oracle.sparse_mla_bwd(q, kv, idx, qs, kl, 0.4, dO, lib=lib)
    assert np.allclose(dkv[0, :, 512:].sum(axis=0), 0.0, atol=1e-10)
    live = [t for t in range(T) if (idx[0, t] >= 0).any()]
    want = dO[0, live].sum(axis=(0, 1))
    assert np.allclose(dkv[0, :, :512].sum(axis=0), want, rtol=0, atol=1e-10)


def pin_mla_bwd_with_sink(lib):
    """With a learnable sink: a sink of -inf is exactly no sink; the float64
    forward agrees with the BF16 sink forward; central differences of the sink
    forward agree with the backward."""
    T, H = 30, 8
    q16 = normal_bf16(96, "q_lat", (1, T, H, 576))
    kv16 = normal_bf16(96, "kv", (1, T, 576))
    rng = np.random.default_rng(96)
    idx = np.full((1, T, 8), -1, np.int32)
    for t in range(T):
        c = rng.permutation(t + 1)[:8]
        idx[0, t, :len(c)] = c
    idx[0, 11] = -1                                   # a query with no valid entry
    qs, kl = np.zeros(1, np.int32), np.full(1, T, np.int32)
    sink = rng.uniform(-1.0, 3.0, H)
    o1, l1 = oracle.sparse_mla(q16, kv16, idx, qs, kl, SCALE, lib=lib, sink=sink)
    o2, l2 = oracle.sparse_mla_f64(q16, kv16, idx, qs, kl, SCALE, lib=lib, sink=sink)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)
    assert np.allclose(l2[11], sink) and np.all(o2[11] == 0.0)
    dO = rng.standard_normal((1, T, H, 512))
    a = oracle.sparse_mla_bwd(q16, kv16, idx, qs, kl, SCALE, dO, lib=lib)
    b = oracle.sparse_mla_bwd(q16, kv16, idx, qs, kl, SCALE, dO, lib=lib, sink=np.full(H, -np.inf))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # central differences on a small float64 case with a sink
    q, kv, dO2, idx2, qs2, kl2 = _bwd_case(97, 6, 2, 3, amp=0.5)
    sk = np.array([0.7, -0.4])
    scale = 0.3
    dq, dkv = oracle.sparse_mla_bwd(q, kv, idx2, qs2, kl2, scale, dO2, lib=lib, sink=sk)

    def loss(qq, kk):
        o, _ = oracle.sparse_mla_f64(qq, kk, idx2, qs2, kl2, scale, lib=lib, sink=sk)
        return float(np.sum(o * dO2.reshape(o.shape)))

    eps = 1e-6
    for (t, h, d) in [(5, 1, 3), (4, 0, 550)]:
        qp, qm = q.copy(), q.copy()
        qp[0, t, h, d] += eps
        qm[0, t, h, d] -= eps
        fd = (loss(qp, kv) - loss(qm, kv)) / (2 * eps)
        assert abs(fd - dq[0, t, h, d]) <= 1e-7 * max(1.0, abs(fd)), ("dq", t, h, d, fd)
    s0 = int(idx2[0, 5, 0])
    for d in (9, 560):
        kp, km = kv.copy(), kv.copy()
        kp[0, s0, d] += eps
        km[0, s0, d] -= eps
        fd = (loss(q, kp) - loss(q, km)) / (2 * eps)
        assert abs(fd - dkv[0, s0, d]) <= 1e-7 * max(1.0, abs(fd)), ("dkv", s0, d, fd)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
