"""Pins for the CPU oracle, independent of the oracle's own code paths.

Each test checks the oracle against something the pages or mathematics fix: closed
forms, invariants, brute force on tiny inputs, and the pages' worked examples stored
under tests/golden/ (each with its citation).
"""
import json
import math
import os

import numpy as np
import pytest

import dflash_inputs as di
from oracle import dflash_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_cfg(**kw):
    base = dict(name="pin", D=32, Dt=16, L=3, N=2, Hq=4, Hkv=2, hd=8, F=24, V=64, B=6, nb=3,
                C=10)
    base.update(kw)
    return di.Workload(**base)


def rand_weights(cfg, seed=0, std=0.3):
    rng = np.random.default_rng(seed)
    W = {}
    for k, shp in di.weight_shapes(cfg).items():
        base = k.rsplit(".", 1)[-1]
        if base.startswith("g_"):
            W[k] = 1.0 + 0.1 * rng.standard_normal(shp)
        elif base == "base":
            b = 0.1 * rng.standard_normal(shp)
            b[0] += 1.0
            W[k] = b
        else:
            W[k] = std * rng.standard_normal(shp)
    return W


def fill_cache(cfg, cache, C, rng):
    for n in range(cfg.N):
        for i in range(len(cache.K[n])):
            cache.K[n][i][:, :C] = rng.standard_normal(cache.K[n][i][:, :C].shape)
            cache.V[n][i][:, :C] = rng.standard_normal(cache.V[n][i][:, :C].shape)


# ----------------------------------------------------------------------------- RMSNorm

def test_rmsnorm_closed_form_constant_vector():
    rng = np.random.default_rng(1)
    g = rng.standard_normal(17)
    for c in (0.5, -3.0, 1e-3):
        y = orc.rmsnorm(np.full(17, c), g, 1e-6)
        np.testing.assert_allclose(y, g * c / math.sqrt(c * c + 1e-6), rtol=1e-14)


def test_rmsnorm_hand_value_and_scale_invariance():
    y = orc.rmsnorm(np.array([3.0, 4.0]), np.ones(2), 0.0)
    np.testing.assert_allclose(y, [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=1e-15)
    x = np.random.default_rng(2).standard_normal((3, 9))
    np.testing.assert_allclose(orc.rmsnorm(7.5 * x, np.ones(9), 0.0), orc.rmsnorm(x, np.ones(9), 0.0),
                               rtol=1e-13)


# ----------------------------------------------------------------------------- RoPE

def test_rope_hand_value_hd4():
    # hd = 4: pairs (0, 2) and (1, 3); angles p * base^0 and p * base^(-1/2).
    x = np.array([1.0, 2.0, 3.0, 4.0])
    p, base = 3, 100.0
    t0, t1 = 3.0, 3.0 / 10.0
    want = [1 * math.cos(t0) - 3 * math.sin(t0), 2 * math.cos(t1) - 4 * math.sin(t1),
            3 * math.cos(t0) + 1 * math.sin(t0), 4 * math.cos(t1) + 2 * math.sin(t1)]
    np.testing.assert_allclose(orc.rope(x, p, base), want, rtol=1e-14)


def test_rope_identity_at_zero_and_pair_norms():
    x = np.random.default_rng(3).standard_normal((5, 3, 16))
    np.testing.assert_array_equal(orc.rope(x, np.zeros(5, int), 1e4), x)
    y = orc.rope(x, np.arange(5) * 1000 + 7, 1e4)
    np.testing.assert_allclose(x[..., :8] ** 2 + x[..., 8:] ** 2, y[..., :8] ** 2 + y[..., 8:] ** 2,
                               rtol=1e-12)


def test_rope_scores_depend_only_on_offset():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(32), rng.standard_normal(32)
    s1 = orc.rope(q, 50, 1e4) @ orc.rope(k, 20, 1e4)
    s2 = orc.rope(q, 1050, 1e4) @ orc.rope(k, 1020, 1e4)
    assert abs(s1 - s2) < 1e-9


# ----------------------------------------------------------------------------- attention

def scalar_rope(vec, pos, base):
    """Rotate pairs (d, d + hd/2) by pos * base^(-2d/hd), one scalar at a time."""
    hd = len(vec)
    half = hd // 2
    out = np.array(vec, dtype=float)
    for d in range(half):
        th = pos * base ** (-2.0 * d / hd)
        out[d] = vec[d] * math.cos(th) - vec[d + half] * math.sin(th)
        out[d + half] = vec[d + half] * math.cos(th) + vec[d] * math.sin(th)
    return out


def brute_attention(q, K, V):
    nq, hd = q.shape
    out = np.zeros((nq, V.shape[1]))
    for a in range(nq):
        sc = [sum(q[a, d] * K[b, d] for d in range(hd)) / math.sqrt(hd) for b in range(K.shape[0])]
        m = max(sc)
        w = [math.exp(s - m) for s in sc]
        tot = sum(w)
        for b in range(K.shape[0]):
            for d in range(V.shape[1]):
                out[a, d] += w[b] / tot * V[b, d]
    return out


def test_attention_brute_force():
    rng = np.random.default_rng(5)
    q, K, V = rng.standard_normal((3, 4)), rng.standard_normal((7, 4)), rng.standard_normal((7, 4))
    np.testing.assert_allclose(orc.softmax_attention(q, K, V), brute_attention(q, K, V), rtol=1e-12)


def test_attention_equal_keys_gives_mean_and_single_key_gives_row():
    rng = np.random.default_rng(6)
    q, V = rng.standard_normal((5, 8)), rng.standard_normal((9, 8))
    K = np.tile(rng.standard_normal(8), (9, 1))
    np.testing.assert_allclose(orc.softmax_attention(q, K, V), np.tile(V.mean(0), (5, 1)), rtol=1e-12)
    np.testing.assert_allclose(orc.softmax_attention(q, K[:1], V[:1]), np.tile(V[0], (5, 1)), rtol=1e-14)


def layer_once(cfg, W, x, Kc, Vc, C):
    return orc.drafter_layer(cfg, W, 0, x, Kc, Vc, C)


def test_layer_context_permutation_invariance():
    cfg = small_cfg()
    W = rand_weights(cfg)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((cfg.B, cfg.D))
    Kc = rng.standard_normal((cfg.Hkv, 12, cfg.hd))
    Vc = rng.standard_normal((cfg.Hkv, 12, cfg.hd))
    perm = rng.permutation(12)
    a = layer_once(cfg, W, x, Kc, Vc, 12)
    b = layer_once(cfg, W, x, Kc[:, perm], Vc[:, perm], 12)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_layer_empty_context_is_block_self_attention():
    cfg = small_cfg()
    W = rand_weights(cfg)
    rng = np.random.default_rng(8)
    x = rng.standard_normal((cfg.B, cfg.D))
    garbage = rng.standard_normal((cfg.Hkv, 5, cfg.hd))
    got = layer_once(cfg, W, x, garbage, garbage, 0)
    # brute force: the same layer written with scalar loops over the block keys only
    p = "layer0."
    u = x / np.sqrt((x * x).mean(1, keepdims=True) + cfg.eps) * W[p + "g_attn"]
    qkv = u @ W[p + "W_qkv"].T
    Hq, Hkv, hd = cfg.Hq, cfg.Hkv, cfg.hd
    q = qkv[:, :Hq * hd].reshape(cfg.B, Hq, hd)
    k = qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(cfg.B, Hkv, hd)
    v = qkv[:, (Hq + Hkv) * hd:].reshape(cfg.B, Hkv, hd)
    def rot(vec, pos):
        return scalar_rope(vec, pos, cfg.rope_base)

    o = np.zeros((cfg.B, Hq * hd))
    for h in range(Hq):
        g = h // (Hq // Hkv)
        qs = np.array([rot(q[j, h], j) for j in range(cfg.B)])
        ks = np.array([rot(k[j, g], j) for j in range(cfg.B)])
        o[:, h * hd:(h + 1) * hd] = brute_attention(qs, ks, v[:, g])
    x1 = x + o @ W[p + "W_o"].T
    u = x1 / np.sqrt((x1 * x1).mean(1, keepdims=True) + cfg.eps) * W[p + "g_ffn"]
    gt, up = u @ W[p + "W_gate"].T, u @ W[p + "W_up"].T
    want = x1 + (gt / (1 + np.exp(-gt)) * up) @ W[p + "W_down"].T
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-10)


def test_zero_output_projections_make_identity_layers():
    cfg = small_cfg()
    W = rand_weights(cfg)
    for n in range(cfg.N):
        W[f"layer{n}.W_o"][:] = 0
        W[f"layer{n}.W_down"][:] = 0
    rng = np.random.default_rng(9)
    cache = orc.KVCache(cfg.N, cfg.nb, cfg.Hkv, 16, cfg.hd)
    fill_cache(cfg, cache, 10, rng)
    ids = rng.integers(0, cfg.V, (cfg.nb, cfg.B))
    out = orc.draft_block(cfg, W, ids, np.full(cfg.nb, 10), cache)
    x = W["E"][ids]
    np.testing.assert_allclose(out, x / np.sqrt((x * x).mean(-1, keepdims=True) + cfg.eps) * W["g_final"],
                               rtol=1e-12)


def test_batch_independence():
    cfg = small_cfg()
    W = rand_weights(cfg)
    rng = np.random.default_rng(10)
    cache = orc.KVCache(cfg.N, cfg.nb, cfg.Hkv, 16, cfg.hd)
    fill_cache(cfg, cache, 16, rng)
    ids = rng.integers(0, cfg.V, (cfg.nb, cfg.B))
    lens = np.array([3, 10, 16])
    a = orc.draft_block(cfg, W, ids, lens, cache)
    ids2 = ids.copy()
    ids2[1:] = rng.integers(0, cfg.V, (cfg.nb - 1, cfg.B))
    for n in range(cfg.N):
        cache.K[n][2][:] = 0
    b = orc.draft_block(cfg, W, ids2, np.array([3, 7, 9]), cache)
    np.testing.assert_array_equal(a[0], b[0])


# ----------------------------------------------------------------------------- conv

def test_conv_identity_and_shift():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((6, 32))
    Z = np.zeros((2, 32))
    base = np.zeros((2, 32))
    base[0] = 1
    np.testing.assert_array_equal(orc.dyn_conv(x, Z, Z, base), x)
    base = np.zeros((2, 32))
    base[1] = 1
    want = np.vstack([np.zeros(32), x[:-1]])
    np.testing.assert_array_equal(orc.dyn_conv(x, Z, Z, base), want)


def test_conv_correction_shared_per_16_channels():
    # one correction value per 16 channels: a W0 row that picks channel 0 scales the
    # first 16 channels by (1 + x_t[0]) and leaves the next 16 at base 1.
    x = np.random.default_rng(12).standard_normal((3, 32))
    W0 = np.zeros((2, 32))
    W0[0, 0] = 1.0
    base = np.zeros((2, 32))
    base[0] = 1
    y = orc.dyn_conv(x, W0, np.zeros((2, 32)), base)
    for t in range(3):
        np.testing.assert_allclose(y[t, :16], (1 + x[t, 0]) * x[t, :16], rtol=1e-15)
        np.testing.assert_array_equal(y[t, 16:], x[t, 16:])


# ----------------------------------------------------------------------------- top-k / accept

def test_topk_matches_python_sort_with_ties():
    rng = np.random.default_rng(13)
    vals = rng.integers(0, 6, (4, 40)).astype(float)  # many exact ties
    ids, v = orc.topk(vals, 7)
    for r in range(4):
        order = sorted(range(40), key=lambda c: (-vals[r, c], c))[:7]
        assert list(ids[r]) == order
        assert list(v[r]) == [vals[r, c] for c in order]


def test_accept_golden_cases():
    g = json.load(open(os.path.join(GOLDEN, "accept_cases.json")))
    for c in g["cases"]:
        tau, bonus = orc.accept(np.array([c["draft"]]), np.array([c["target"]]))
        assert (int(tau[0]), int(bonus[0])) == (c["tau"], c["bonus"]), c["why"]


def test_accept_tau_range_and_bonus():
    rng = np.random.default_rng(14)
    B = 16
    d = rng.integers(0, 3, (500, B - 1))
    t = rng.integers(0, 3, (500, B))
    tau, bonus = orc.accept(d, t)
    assert tau.min() >= 1 and tau.max() <= B
    for i in range(500):
        m = int(tau[i]) - 1
        assert np.array_equal(d[i, :m], t[i, :m])
        assert m == B - 1 or d[i, m] != t[i, m]
        assert bonus[i] == t[i, m]


# ----------------------------------------------------------------------------- relay

def test_relay_placement_matches_dflow_example():
    g = json.load(open(os.path.join(GOLDEN, "relay_positions.json")))
    cfg = small_cfg(B=g["B"], nb=1)
    W = rand_weights(cfg)
    rng = np.random.default_rng(15)
    hv = rng.standard_normal((1, cfg.B, cfg.L * cfg.Dt))
    a = g["accepted"]
    cache = orc.KVCache(cfg.N, 1, cfg.Hkv, 32, cfg.hd)
    start = g["prev_block_start"]
    new_len, x0r = orc.ctx_project(cfg, W, hv, [a + 1], [start], cache, relay_a=[a])
    assert int(new_len[0]) == g["next_block_start"]
    h = orc.fuse_context(cfg, W, hv[0])
    placed = {}
    for e in g["relayed"]:
        assert e["new_pos"] == e["prev_pos"] + 1
        assert e["new_pos"] == g["next_block_start"] + e["new_offset"]
        np.testing.assert_array_equal(x0r[0, e["new_offset"]], h[e["prev_row"]])
        placed[e["new_offset"]] = True
    for j in range(cfg.B):
        if j not in placed:
            assert not x0r[0, j].any()


def test_relay_inactive_when_nearly_all_accepted():
    cfg = small_cfg(nb=2)
    W = rand_weights(cfg)
    rng = np.random.default_rng(16)
    hv = rng.standard_normal((2, cfg.B, cfg.L * cfg.Dt))
    cache = orc.KVCache(cfg.N, 2, cfg.Hkv, 32, cfg.hd)
    _, x0r = orc.ctx_project(cfg, W, hv, [cfg.B - 1, cfg.B], [0, 0], cache,
                             relay_a=[cfg.B - 2, cfg.B - 1])
    assert not x0r.any()


def test_ctx_project_cache_rows():
    cfg = small_cfg(nb=1)
    W = rand_weights(cfg)
    rng = np.random.default_rng(17)
    hv = rng.standard_normal((1, 4, cfg.L * cfg.Dt))
    cache = orc.KVCache(cfg.N, 1, cfg.Hkv, 16, cfg.hd)
    new_len, _ = orc.ctx_project(cfg, W, hv, [3], [5], cache)
    assert int(new_len[0]) == 8
    # h by block decomposition of W_c over the L concatenated layers
    Wc = W["W_c"]
    pre = sum(Wc[:, l * cfg.Dt:(l + 1) * cfg.Dt] @ hv[0, :, l * cfg.Dt:(l + 1) * cfg.Dt].T
              for l in range(cfg.L)).T
    h = pre / np.sqrt((pre * pre).mean(-1, keepdims=True) + cfg.eps) * W["g_ctx"]
    for n in range(cfg.N):
        for j in range(3):
            v = (W[f"layer{n}.Wv_c"] @ h[j]).reshape(cfg.Hkv, cfg.hd)
            np.testing.assert_allclose(cache.V[n][0][:, 5 + j], v, rtol=1e-12)
            k = (W[f"layer{n}.Wk_c"] @ h[j]).reshape(cfg.Hkv, cfg.hd)
            kc = cache.K[n][0][:, 5 + j]
            for g in range(cfg.Hkv):
                np.testing.assert_allclose(kc[g], scalar_rope(k[g], 5 + j, cfg.rope_base),
                                           rtol=1e-10, atol=1e-12)
        assert not cache.K[n][0][:, 8:].any() and not cache.K[n][0][:, :5].any()


# ----------------------------------------------------------------------------- paged cache

def test_paged_rows_hand_case():
    """Pages of 4 rows, 2 heads, hd 1; pool[p, h, r] = 100 p + 10 h + r. Table row 0 is
    [2, 0]: its rows 0..3 come from page 2, rows 4..7 from page 0."""
    pool = np.array([[[[100.0 * p + 10 * h + r] for r in range(4)] for h in range(2)] for p in range(4)])
    table = [[2, 0], [1, 3]]
    got = orc.paged_rows(pool, table, 0, 7, page_rows=4)
    assert got.shape == (2, 7, 1)
    assert got[0, :, 0].tolist() == [200, 201, 202, 203, 0, 1, 2]
    assert got[1, :, 0].tolist() == [210, 211, 212, 213, 10, 11, 12]
    got = orc.paged_rows(pool, table, 1, 8, page_rows=4)
    assert got[1, :, 0].tolist() == [110, 111, 112, 113, 310, 311, 312, 313]


def test_paged_identity_table_is_the_contiguous_layout():
    """With table[i][q] = i * pages_per_seq + q the pool is the contiguous cache
    [nb][Hkv][Cmax][hd] cut into pages: a reshape, whatever the contents."""
    rng = np.random.default_rng(31)
    N, nb, Hkv, pps, hd = 2, 3, 2, 3, 4
    Cmax = pps * orc.PAGE_ROWS
    poolK = rng.standard_normal((N, nb * pps, Hkv, orc.PAGE_ROWS, hd))
    poolV = rng.standard_normal((N, nb * pps, Hkv, orc.PAGE_ROWS, hd))
    table = [[i * pps + q for q in range(pps)] for i in range(nb)]
    c = orc.cache_from_pages(poolK, poolV, table, nb, Cmax)
    contK = poolK.reshape(N, nb, pps, Hkv, orc.PAGE_ROWS, hd).transpose(0, 1, 3, 2, 4, 5)
    contK = contK.reshape(N, nb, Hkv, Cmax, hd)
    contV = poolV.reshape(N, nb, pps, Hkv, orc.PAGE_ROWS, hd).transpose(0, 1, 3, 2, 4, 5)
    contV = contV.reshape(N, nb, Hkv, Cmax, hd)
    for n in range(N):
        for i in range(nb):
            assert np.array_equal(c.K[n][i], contK[n, i])
            assert np.array_equal(c.V[n][i], contV[n, i])


def test_paged_relabelling_and_shared_prefix():
    """Renaming the physical pages (pool and table permuted together) changes no logical
    row; two sequences whose tables share their first pages read the same prefix rows."""
    rng = np.random.default_rng(32)
    P, Hkv, hd = 6, 2, 3
    pool = rng.standard_normal((P, Hkv, orc.PAGE_ROWS, hd))
    table = [[4, 1, 5], [4, 1, 0]]
    perm = rng.permutation(P)                      # page q moves to slot perm[q]
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    table2 = [[int(perm[q]) for q in row] for row in table]
    n = 3 * orc.PAGE_ROWS
    for i in range(2):
        assert np.array_equal(orc.paged_rows(pool, table, i, n), orc.paged_rows(pool2, table2, i, n))
    a, b = orc.paged_rows(pool, table, 0, n), orc.paged_rows(pool, table, 1, n)
    assert np.array_equal(a[:, :2 * orc.PAGE_ROWS], b[:, :2 * orc.PAGE_ROWS])
    assert not np.array_equal(a[:, 2 * orc.PAGE_ROWS:], b[:, 2 * orc.PAGE_ROWS:])


# ----------------------------------------------------------------------------- FiLM relay

def test_layer_norm_closed_forms():
    eps = 1e-6
    # a constant row has zero deviation from its mean
    assert not orc.layer_norm(np.full((1, 8), 3.7), eps).any()
    # +-c alternating: mean 0, population variance c^2
    x = np.array([3.0, -3.0] * 4)
    np.testing.assert_allclose(orc.layer_norm(x, eps), x / math.sqrt(9.0 + eps), rtol=1e-15)
    # 1, 2, 3, 4: mean 5/2, population variance 5/4 (not the sample variance 5/3)
    got = orc.layer_norm(np.array([1.0, 2.0, 3.0, 4.0]), eps)
    np.testing.assert_allclose(got, np.array([-1.5, -0.5, 0.5, 1.5]) / math.sqrt(1.25 + eps),
                               rtol=1e-15)


def test_layer_norm_moments_and_invariance():
    rng = np.random.default_rng(30)
    x = rng.standard_normal((5, 64)) * 3 + 2
    y = orc.layer_norm(x, 0.0)
    np.testing.assert_allclose(y.mean(-1), 0.0, atol=1e-14)
    np.testing.assert_allclose((y * y).mean(-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(orc.layer_norm(4.0 * x - 7.0, 0.0), y, rtol=1e-12, atol=1e-13)


def film_cfg(**kw):
    return small_cfg(flags=di.FLAG_RELAY | di.FLAG_FILM, film_dim=32, **kw)


def film_case(cfg, seed):
    W = rand_weights(cfg, seed)
    rng = np.random.default_rng(seed + 1)
    hv = rng.standard_normal((cfg.nb, cfg.B, cfg.L * cfg.Dt))
    b = rng.integers(0, cfg.V - 1, cfg.nb)
    y = rng.integers(0, cfg.V - 1, cfg.nb)
    return W, hv, b, y


def project(cfg, W, hv, a, b=None, y=None):
    cache = orc.KVCache(cfg.N, cfg.nb, cfg.Hkv, 32, cfg.hd)
    return orc.ctx_project(cfg, W, hv, [a[i] + 1 for i in range(cfg.nb)], [3] * cfg.nb, cache,
                           relay_a=a, relay_b=b, relay_y=y)[1]


def selection(D, blocks):
    """[D, len(blocks) * D] with an identity in each block marked 1."""
    return np.concatenate([np.eye(D) if on else np.zeros((D, D)) for on in blocks], axis=1)


def test_film_selection_weights_pick_each_input():
    """Selection-matrix weights turn the FiLM row into closed forms, one input at a time:
    gamma = silu(h) alone; beta = silu(E[b]) or silu(E[y]) times LN(h). A swapped
    concatenation order, a swapped beta/gamma split, a missing LN or a wrong relay row
    fails one of them."""
    from scipy.special import expit
    cfg = film_cfg(nb=3)
    D = cfg.D
    a = [0, 2, 1]
    W, hv, b, y = film_case(cfg, 31)
    plain = project(cfg, W, hv, a)
    zero = np.zeros((D, D))
    eye = np.eye(D)
    relayed = np.abs(plain).sum(-1) > 0

    W["film.W1"] = selection(D, (0, 0, 1))
    W["film.W2"] = np.concatenate([zero, eye])
    got = project(cfg, W, hv, a, b, y)
    np.testing.assert_allclose(got, plain * expit(plain), rtol=1e-13, atol=1e-15)

    def ln(v):
        return (v - v.mean(-1, keepdims=True)) / np.sqrt(v.var(-1, keepdims=True) + cfg.eps)

    W["film.W2"] = np.concatenate([eye, zero])
    for blocks, tok in (((1, 0, 0), b), ((0, 1, 0), y)):
        W["film.W1"] = selection(D, blocks)
        got = project(cfg, W, hv, a, b, y)
        e = W["E"][tok]
        want = (e * expit(e))[:, None, :] * ln(plain)
        np.testing.assert_allclose(got[relayed], want[relayed], rtol=1e-12, atol=1e-14)
        assert not got[~relayed].any()


def test_film_zero_output_layer_turns_relay_off():
    """W2 = 0 gives beta = gamma = 0: the relayed input is the mask embedding alone, so the
    whole draft equals the draft with no relay."""
    cfg = film_cfg(nb=2)
    a = [1, 0]
    W, hv, b, y = film_case(cfg, 32)
    W["film.W2"] = np.zeros_like(W["film.W2"])
    assert not project(cfg, W, hv, a, b, y).any()
    ids = np.full((cfg.nb, cfg.B), cfg.mask_id, np.int32)
    ids[:, 0] = [5, 9]
    outs = []
    for relay in (False, True):
        cache = orc.KVCache(cfg.N, cfg.nb, cfg.Hkv, 32, cfg.hd)
        fill_cache(cfg, cache, 3, np.random.default_rng(34))
        kw = dict(relay_a=a, relay_b=b, relay_y=y) if relay else {}
        outs.append(orc.draft_step(cfg, W, hv, [2, 1], [3, 3], cache, ids,
                                   np.zeros((cfg.nb, cfg.B), np.int32), **kw)["hidden"])
    np.testing.assert_array_equal(outs[0], outs[1])


def test_film_brute_force_tiny():
    """Scalar loops over a D = 2, film width 3 case with random (non-symmetric) weights:
    catches a transposed W1 or W2 block that identity selections cannot."""
    cfg = small_cfg(D=2, Dt=2, L=1, Hq=1, Hkv=1, hd=2, F=2, V=5, B=4, nb=1,
                    flags=di.FLAG_RELAY | di.FLAG_FILM, film_dim=3)
    rng = np.random.default_rng(35)
    W = rand_weights(cfg, 36, std=0.7)
    h = rng.standard_normal(2)
    b, y = 3, 1
    c = [W["E"][b][0], W["E"][b][1], W["E"][y][0], W["E"][y][1], h[0], h[1]]
    hid = []
    for r in range(3):
        t = 0.0
        for q in range(6):
            t += W["film.W1"][r][q] * c[q]
        hid.append(t / (1.0 + math.exp(-t)))
    out = []
    for r in range(4):
        t = 0.0
        for q in range(3):
            t += W["film.W2"][r][q] * hid[q]
        out.append(t)
    mean = (h[0] + h[1]) / 2
    var = ((h[0] - mean) ** 2 + (h[1] - mean) ** 2) / 2
    want = [out[d] * (h[d] - mean) / math.sqrt(var + cfg.eps) + out[2 + d] for d in range(2)]
    np.testing.assert_allclose(orc.film_relay_row(cfg, W, h, b, y), want, rtol=1e-12)


def test_film_weight_shapes():
    w = di.FILM_RELAY
    s = di.weight_shapes(w)
    assert s["film.W1"] == (w.D // 4, 3 * w.D)
    assert s["film.W2"] == (2 * w.D, w.D // 4)
    assert "film.W1" not in di.weight_shapes(di.QWEN3_8B)


# ----------------------------------------------------------------------------- sampling

def test_philox_known_answer_vectors():
    g = json.load(open(os.path.join(GOLDEN, "philox_kat.json")))
    for case in g["cases"]:
        ctr = [int(x, 16) for x in case["ctr"]]
        key = [int(x, 16) for x in case["key"]]
        got = [int(x) for x in orc.philox4x32(ctr, key)]
        assert got == [int(x, 16) for x in case["out"]], case


def test_uniforms_are_uniform_and_streams_independent():
    from scipy import stats
    u = orc.uniforms(12345, orc.STREAM_DRAFT, 7, 200000)
    assert u.min() > 0.0 and u.max() < 1.0
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    # one Philox call covers four consecutive indices: the words must not repeat
    assert len(np.unique(u[:4])) == 4
    v = orc.uniforms(12345, orc.STREAM_ACCEPT, 7, 200000)
    w = orc.uniforms(12345, orc.STREAM_DRAFT, 8, 200000)
    x = orc.uniforms(12346, orc.STREAM_DRAFT, 7, 200000)
    for o in (v, w, x):
        assert abs(np.corrcoef(u, o)[0, 1]) < 0.01


@pytest.mark.parametrize("T", [1.0, 0.5, 2.0])
def test_gumbel_draws_follow_softmax(T):
    from scipy import stats
    logits = np.array([1.0, 0.2, -0.5, 2.0, 0.0])
    n = 20000
    draws = np.array([orc.gumbel_argmax(logits / T + orc.gumbel(orc.uniforms(99, 0, r, 5)))[0]
                      for r in range(n)])
    p = np.exp(logits / T) / np.exp(logits / T).sum()
    obs = np.bincount(draws, minlength=5)
    assert stats.chisquare(obs, p * n).pvalue > 1e-4


def test_sample_candidates_rows_and_log_probs():
    rng = np.random.default_rng(40)
    U = rng.standard_normal((2, 3, 50)) * 2
    ids, lse, logq, _ = orc.sample_candidates(U, 1.0, 7)
    for i in range(2):
        for t in range(3):
            q = np.exp(U[i, t]) / np.exp(U[i, t]).sum()
            assert math.isclose(logq[i, t], math.log(q[ids[i, t]]), rel_tol=1e-12)
    # rows are distinct streams: the same logits in two rows draw independently
    same = np.repeat(U[:1, :1], 400, axis=1)
    ids2, _, _, _ = orc.sample_candidates(same, 1.0, 7)
    assert len(np.unique(ids2)) > 10


def verify_inputs(nb, B, V, seed, scale=1.5):
    rng = np.random.default_rng(seed)
    U = rng.standard_normal((nb, B - 1, V)) * scale
    Z = rng.standard_normal((nb, B, V)) * scale
    return U, Z


def test_verify_equal_distributions_accept_every_candidate():
    """p_j = q_{j+1} gives ratio 1 > u: every candidate is accepted, tau = B."""
    U, Z = verify_inputs(3, 6, 40, 41)
    Z[:, :5] = U
    cand, _, _, _ = orc.sample_candidates(U, 1.0, 3)
    tau, token = orc.verify_sample(U, cand, Z, 1.0, 3)
    assert (tau == 6).all()
    assert ((token >= 0) & (token < 40)).all()


def test_verify_zero_target_probability_rejects_there():
    """A candidate the target gives probability 0 is rejected, and the re-drawn token is
    never that candidate (its residual max(0, 0 - q) is 0)."""
    U, Z = verify_inputs(4, 6, 40, 42)
    Z[:, :5] = U
    cand, _, _, _ = orc.sample_candidates(U, 1.0, 5)
    for i in range(4):
        Z[i, 2, cand[i, 2]] = -np.inf
    tau, token = orc.verify_sample(U, cand, Z, 1.0, 5)
    assert (tau == 3).all()
    assert (token != cand[:, 2]).all()


def test_verify_is_lossless_monte_carlo():
    """The first emitted token (accepted candidate, or the re-drawn one) follows the target
    distribution p_0 whatever q is, and the acceptance rate is sum_v min(p_0, q_1)."""
    from scipy import stats
    zp = np.log(np.array([0.5, 0.3, 0.15, 0.05]))
    zq = np.log(np.array([0.1, 0.2, 0.3, 0.4]))
    U = zq[None, None, :]
    Z = np.stack([zp, zp])[None]
    n = 6000
    first = np.zeros(n, np.int64)
    acc = 0
    for s in range(n):
        cand, _, _, _ = orc.sample_candidates(U, 1.0, s)
        tau, token = orc.verify_sample(U, cand, Z, 1.0, s)
        first[s] = cand[0, 0] if tau[0] > 1 else token[0]
        acc += int(tau[0] > 1)
    p = np.exp(zp)
    assert stats.chisquare(np.bincount(first, minlength=4), p * n).pvalue > 1e-4
    a = np.minimum(p, np.exp(zq)).sum()
    assert abs(acc / n - a) < 4 * math.sqrt(a * (1 - a) / n)


def test_verify_temperature_scales_logits():
    """Logits times T at temperature T are the same distributions as at T = 1."""
    U, Z = verify_inputs(3, 5, 30, 43)
    cand, _, _, _ = orc.sample_candidates(U, 1.0, 9)
    c2, _, _, _ = orc.sample_candidates(U * 0.7, 0.7, 9)
    assert np.array_equal(cand, c2)
    t1 = orc.verify_sample(U, cand, Z, 1.0, 9)
    t2 = orc.verify_sample(U * 0.7, cand, Z * 0.7, 0.7, 9)
    assert np.array_equal(t1[0], t2[0]) and np.array_equal(t1[1], t2[1])


# ----------------------------------------------------------------------------- selector

def test_selector_without_pair_term_is_per_position_argmax():
    cfg = small_cfg(flags=di.FLAG_SELECT, sel_dim=8)
    W = rand_weights(cfg)
    W["W_A"][:] = 0
    rng = np.random.default_rng(18)
    ids = np.stack([rng.permutation(cfg.V)[:5] for _ in range(cfg.nb * (cfg.B - 1))])
    ids = ids.reshape(cfg.nb, cfg.B - 1, 5)
    vals = rng.integers(0, 3, ids.shape).astype(float)
    hid = rng.standard_normal((cfg.nb, cfg.B, cfg.D))
    path = orc.select_path(cfg, W, ids, vals, hid, np.zeros(cfg.nb, int))
    for i in range(cfg.nb):
        for t in range(cfg.B - 1):
            best = sorted(range(5), key=lambda c: (-vals[i, t, c], ids[i, t, c]))[0]
            assert path[i, t] == ids[i, t, best]


def test_selector_pair_term_prefers_coherent_successor():
    # E rows one-hot, W_A = W_B = 4*I, W_G = 0 (gate 1/2): the pair term adds 8 when
    # b == a and 0 otherwise, so the walk repeats the anchor whenever it is a candidate
    # unless some other logit leads by more than 8.
    cfg = small_cfg(D=8, V=8, B=4, nb=1, flags=di.FLAG_SELECT, sel_dim=8)
    W = rand_weights(cfg)
    W["E"] = np.eye(8)
    W["W_A"] = 4 * np.eye(8)
    W["W_B"] = 4 * np.eye(8)
    W["W_G"] = np.zeros((8, 8))
    ids = np.array([[[1, 3], [3, 5], [5, 6]]])
    vals = np.array([[[1.0, 0.0], [0.5, 0.0], [0.0, 9.0]]])
    path = orc.select_path(cfg, W, ids, vals, np.zeros((1, 4, 8)), np.array([3]))
    # t=1: S(3,1)=1, S(3,3)=0+8 -> 3; t=2: S(3,3)=0.5+8, S(3,5)=0 -> 3;
    # t=3: S(3,5)=0, S(3,6)=9 -> 6
    assert path.tolist() == [[3, 3, 6]]


# ----------------------------------------------------------------------------- shapes

def test_shape_pins_from_pages():
    g = json.load(open(os.path.join(GOLDEN, "shape_pins.json")))
    p = g["W_c_bytes"]
    w = di.Workload("p", D=p["D"], Dt=p["D"], L=p["L"], N=1, Hq=16, Hkv=8, hd=128, F=8, V=8, B=16,
                    nb=1, C=1)
    shp = di.weight_shapes(w)["W_c"]
    mb = shp[0] * shp[1] * p["bytes_per_param"] / 1e6
    assert abs(mb - p["quoted_MB"]) / p["quoted_MB"] < p["rel_tol"]

    q = g["conv_params"]
    w = di.QWEN3_4B.with_(flags=di.FLAG_CONV)
    assert w.D == q["D"] and w.N == q["N"]
    n = sum(int(np.prod(s)) for k, s in di.weight_shapes(w).items() if ".conv" in k)
    assert abs(n / 1e6 - q["quoted_M"]) < q["abs_tol_M"]

    s = g["selector_params"]
    w = di.QWEN3_4B.with_(flags=di.FLAG_SELECT)
    n = sum(int(np.prod(v)) for k, v in di.weight_shapes(w).items() if k in ("W_A", "W_B", "W_G"))
    assert abs(n / 1e6 - s["quoted_M"]) < s["abs_tol_M"]


# ----------------------------------------------------------------------------- sampling walk

def walk_case(seed=50, nb=2, B=5, k=4, D=8, V=40):
    cfg = small_cfg(D=D, V=V, B=B, nb=nb, flags=di.FLAG_SELECT, sel_dim=8)
    W = rand_weights(cfg, seed, std=0.5)
    rng = np.random.default_rng(seed + 1)
    cand = np.stack([np.stack([rng.choice(V, k, replace=False) for _ in range(B - 1)])
                     for _ in range(nb)]).astype(np.int32)
    vals = rng.standard_normal((nb, B - 1, k)) * 1.5
    hid = rng.standard_normal((nb, B, D))
    anchor = rng.integers(0, V, nb)
    return cfg, W, cand, vals, hid, anchor


def test_walk_without_pair_term_draws_from_candidate_softmax():
    """W_A = 0 removes the pair term: S_t(a, b_c) = U_t(b_c) whatever a, so the walk's
    log q is log softmax(U_t / T) on the candidates and its draws follow it."""
    from scipy import stats
    cfg, W, cand, vals, hid, anchor = walk_case()
    W["W_A"] = np.zeros_like(W["W_A"])
    T = 0.8
    _, logq, _ = orc.select_walk_sample(cfg, W, cand, vals, hid, anchor, T, 3)
    x = vals / T
    want = x - np.log(np.exp(x).sum(-1, keepdims=True))
    np.testing.assert_allclose(logq, want, rtol=1e-12, atol=1e-12)
    n = 3000
    first = [orc.select_walk_sample(cfg, W, cand[:1], vals[:1], hid[:1], anchor[:1], T, s)[0][0, 0]
             for s in range(n)]
    slots = [int(np.nonzero(cand[0, 0] == c)[0][0]) for c in first]
    p = np.exp(want[0, 0])
    assert stats.chisquare(np.bincount(slots, minlength=4), p * n).pvalue > 1e-4


def test_walk_draws_of_different_offsets_are_independent():
    """Each step has its own Philox row: with the pair term off and the same candidate
    scores at offsets 1 and 2, the two draws are independent (chi-square on the joint
    counts), not copies of each other."""
    from scipy import stats
    cfg, W, cand, vals, hid, anchor = walk_case(seed=54, nb=1, B=3, k=3)
    W["W_A"] = np.zeros_like(W["W_A"])
    vals[0, 1] = vals[0, 0] = np.array([0.3, 0.0, -0.2])
    cand[0, 1] = cand[0, 0]
    n = 3000
    joint = np.zeros((3, 3))
    for sd in range(n):
        path, _, _ = orc.select_walk_sample(cfg, W, cand, vals, hid, anchor, 1.0, sd)
        s1 = int(np.nonzero(cand[0, 0] == path[0, 0])[0][0])
        s2 = int(np.nonzero(cand[0, 1] == path[0, 1])[0][0])
        joint[s1, s2] += 1
    assert stats.chi2_contingency(joint).pvalue > 1e-4
    assert np.trace(joint) < 0.6 * n


def test_walk_at_low_temperature_is_the_greedy_walk():
    cfg, W, cand, vals, hid, anchor = walk_case(seed=51, nb=3)
    greedy, margins = orc.select_path(cfg, W, cand, vals, hid, anchor, return_margins=True)
    path, logq, _ = orc.select_walk_sample(cfg, W, cand, vals, hid, anchor, 1e-5, 9)
    assert (margins > 1e-2).all()
    assert np.array_equal(path, greedy)
    np.testing.assert_allclose(np.exp(logq).sum(-1), 1.0, rtol=1e-12)


def test_verify_walk_equals_dense_verify_with_minus_inf_logits():
    """The walk's sparse q, written as dense logits (log q on the candidates, -inf
    elsewhere), gives the dense verify the same distribution: identical tau and token."""
    cfg, W, cand, vals, hid, anchor = walk_case(seed=52, nb=6, B=6, k=4, V=30)
    path, logq, _ = orc.select_walk_sample(cfg, W, cand, vals, hid, anchor, 1.0, 4)
    rng = np.random.default_rng(53)
    Z = rng.standard_normal((6, 6, 30)) * 1.5
    for i in range(6):  # make acceptance likely: the target favours the walked tokens
        for t in range(5):
            Z[i, t, path[i, t]] += 2.0
    dense = np.full((6, 5, 30), -np.inf)
    for i in range(6):
        for t in range(5):
            dense[i, t, cand[i, t]] = logq[i, t]
    a = orc.verify_sample_walk(cand, logq, path, Z, 1.0, 11)
    b = orc.verify_sample(dense, path, Z, 1.0, 11)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert len(np.unique(a[0])) > 1


def test_verify_walk_is_lossless_monte_carlo():
    from scipy import stats
    p = np.array([0.4, 0.25, 0.2, 0.1, 0.05])
    cand = np.array([[[3, 0, 2]]], np.int32)
    q = np.array([0.5, 0.2, 0.3])
    logq = np.log(q)[None, None]
    Z = np.log(np.stack([p, p]))[None]
    n = 6000
    first = np.zeros(n, np.int64)
    for s in range(n):
        c = cand[0, 0, orc.gumbel_argmax(logq[0, 0] + orc.gumbel(orc.uniforms(s, 3, 0, 3)))[0]]
        tau, tok = orc.verify_sample_walk(cand, logq, np.array([[c]], np.int32), Z, 1.0, s)
        first[s] = c if tau[0] > 1 else tok[0]
    assert stats.chisquare(np.bincount(first, minlength=5), p * n).pvalue > 1e-4


def test_recall_at_k_hand_case():
    cand = np.array([[[1, 2], [3, 4], [5, 6]],     # targets 2, 4, 9: hits at 1, 2; miss at 3
                     [[1, 2], [3, 4], [5, 6]],     # targets 7, ...: miss at 1, stops
                     [[7, 8], [9, 1], [2, 3]]],    # targets 8, 1, 3: all three hit
                    np.int32)
    target = np.array([[2, 4, 9], [7, 4, 5], [8, 1, 3]])
    hits, eligible = orc.recall_at_k(cand, target)
    assert list(hits) == [2, 2, 1] and list(eligible) == [3, 2, 2]


# ----------------------------------------------------------------------------- LM head rows

def test_lm_logits_rows_are_mask_offsets_one_to_b_minus_one():
    # [DFlash] 四、推理流程, dflash_cycle: the draft takes the LM head of the block's
    # hidden rows from offset 1 on (the anchor at offset 0 is already known and yields no
    # candidate). Offset j of sequence i carries a one-hot at column c(i, j); W_lm is a
    # non-symmetric permutation (row perm[c] reads column c), so logits row (i, t-1) peaks
    # at vocabulary id perm[c(i, t)]. Offsets 0..B-2 instead of 1..B-1, or W_lm applied
    # transposed, move every peak.
    D, B, nb = 16, 6, 2
    rng = np.random.default_rng(31)
    perm = rng.permutation(D)
    while np.array_equal(perm[perm], np.arange(D)):  # not an involution: W_lm != W_lm^T
        perm = rng.permutation(D)
    W = {"W_lm": np.zeros((D, D))}
    W["W_lm"][perm, np.arange(D)] = 1.0
    col = np.array([[(5 * i + 3 * j + 1) % D for j in range(B)] for i in range(nb)])
    hidden = np.zeros((nb, B, D))
    for i in range(nb):
        for j in range(B):
            hidden[i, j, col[i, j]] = 2.0 + j + (50.0 if j == 0 else 0.0)  # the anchor row is loud
    logits = orc.lm_logits(W, hidden)
    assert logits.shape == (nb, B - 1, D)
    for i in range(nb):
        for t in range(1, B):
            assert int(np.argmax(logits[i, t - 1])) == perm[col[i, t]]
            assert logits[i, t - 1].max() == 2.0 + t
    assert logits.max() < 50.0  # the anchor row never reaches the logits


# ----------------------------------------------------------------------------- whole step

def test_draft_step_accept_reads_the_selector_path():
    # [DFlash2] 洞察一: with the selector on, the greedy walk's path replaces the per-offset
    # top-1 as the draft that the verifier checks. Large W_A / W_B make the pair term
    # dominate, so the path leaves the top-1 at offset 1 of some sequence; a target row that
    # repeats the path then accepts every candidate (tau = B, bonus = T[B-1]), and one that
    # repeats the top-1 stops at the first offset where they differ.
    import copy
    cfg = small_cfg(flags=di.FLAG_SELECT, sel_dim=8, k_top=6, nb=4)
    W = rand_weights(cfg, seed=5)
    W["W_A"] = 3.0 * np.random.default_rng(6).standard_normal(W["W_A"].shape)
    W["W_B"] = 3.0 * np.random.default_rng(7).standard_normal(W["W_B"].shape)
    rng = np.random.default_rng(8)
    cache = orc.KVCache(cfg.N, cfg.nb, cfg.Hkv, 40, cfg.hd)
    fill_cache(cfg, cache, 12, rng)
    hv = rng.standard_normal((cfg.nb, 3, cfg.L * cfg.Dt))
    ids = rng.integers(0, cfg.V - 1, (cfg.nb, cfg.B)).astype(np.int32)
    ids[:, 1:] = cfg.V - 1
    args = (hv, [3] * cfg.nb, [12] * cfg.nb)
    first = orc.draft_step(cfg, W, *args, copy.deepcopy(cache), ids, np.zeros((cfg.nb, cfg.B), np.int32))
    path, top1 = first["path"], first["ids"][..., 0]
    differs = path[:, 0] != top1[:, 0]
    assert differs.any()
    assert np.array_equal(first["draft"], path)
    bonus_tok = np.arange(cfg.nb, dtype=np.int32) + 7
    t_path = np.concatenate([path, bonus_tok[:, None]], axis=1).astype(np.int32)
    o = orc.draft_step(cfg, W, *args, copy.deepcopy(cache), ids, t_path)
    assert np.array_equal(o["path"], path)
    assert o["tau"].tolist() == [cfg.B] * cfg.nb
    assert o["bonus"].tolist() == bonus_tok.tolist()
    t_top1 = np.concatenate([top1, bonus_tok[:, None]], axis=1).astype(np.int32)
    o = orc.draft_step(cfg, W, *args, copy.deepcopy(cache), ids, t_top1)
    for i in range(cfg.nb):
        m = int(np.argmax(path[i] != top1[i])) if (path[i] != top1[i]).any() else cfg.B - 1
        assert int(o["tau"][i]) == m + 1
        assert int(o["bonus"][i]) == int(t_top1[i, m])
    assert (o["tau"][differs] == 1).all()



def test_tiny_step_runs_and_is_deterministic():
    cfg = di.TINY
    bits = di.make_weights(cfg)
    W = orc.widen_all(bits)
    cache = orc.KVCache(cfg.N, cfg.nb, cfg.Hkv, 80, cfg.hd)
    hv = orc.widen(di.verifier_rows(cfg, cfg.C))
    lens, _ = orc.ctx_project(cfg, W, hv[:, :cfg.C - 3], [cfg.C - 3], [0], cache)
    ids = di.block_ids(cfg, di.anchors(cfg))
    out1 = orc.draft_step(cfg, W, hv[:, cfg.C - 3:], [3], lens,
                          cache, ids, np.zeros((1, cfg.B), np.int32))
    assert int(out1["ctx_len"][0]) == cfg.C
    assert 1 <= int(out1["tau"][0]) <= cfg.B
    assert np.isfinite(out1["hidden"]).all()
