"""GPU parity of every step call against the CPU oracle, on seeded synthetic inputs.

Each test calls libdflash through its C ABI (ctypes binding) and the oracle on the
same bf16 values. Sizes span several GEMM tiles, ragged tails (F, V and L*Dt not
multiples of the tile), ragged and empty contexts, and the small tiny workload.
"""
import numpy as np
import pytest
import torch

import dflash_inputs as di
from _parity import assert_close, check_topk
from oracle import dflash_oracle as orc

pytestmark = pytest.mark.gpu

MEDIUM = di.Workload("medium_d512_hd128_gqa4", D=512, Dt=192, L=5, N=2, Hq=8, Hkv=2, hd=128,
                     F=1000, V=5003, B=16, nb=3, C=300)
MEDIUM_B8 = MEDIUM.with_(name="medium_b8", B=8, nb=5)
MEDIUM_ALL = MEDIUM.with_(name="medium_relay_conv_select",
                          flags=di.FLAG_RELAY | di.FLAG_CONV | di.FLAG_SELECT)
MEDIUM_G8 = MEDIUM.with_(name="medium_gqa8_128_query_rows", Hq=16)  # (Hq/Hkv)*B = 128
MEDIUM_FILM = MEDIUM.with_(name="medium_film_relay", flags=di.FLAG_RELAY | di.FLAG_FILM)
TINY_FILM = di.TINY.with_(name="tiny_film_relay_nb4", nb=4, flags=di.FLAG_RELAY | di.FLAG_FILM)


def lib():
    from block_diffusion_speculative_project_gb300 import dflash, drafter
    return dflash, drafter


def make(w, Cmax, max_proj_rows, seed=0, max_batch=None, max_spin=0, flags_extra=0, bits=None,
         num_pages=0):
    _, drafter = lib()
    bits = di.make_weights(w, seed) if bits is None else bits
    dev = {k: drafter.to_device_bf16(v) for k, v in bits.items()}
    shape = w.with_(flags=w.flags | flags_extra) if flags_extra else w
    dr = drafter.Drafter(shape, dev, max_batch or w.nb, Cmax, max_proj_rows, max_spin=max_spin,
                         num_pages=num_pages)
    return dr, orc.widen_all(bits), bits


def i32(a):
    return torch.tensor(np.asarray(a, dtype=np.int32), device="cuda")


def bf16(bits):
    _, drafter = lib()
    return drafter.to_device_bf16(bits)


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def random_cache(w, nb, Cmax, seed=0):
    shp = (w.N, nb, w.Hkv, Cmax, w.hd)
    return di.normal_bf16("kcache", shp, 1.0, seed=seed), di.normal_bf16("vcache", shp, 1.0, seed=seed)


def oracle_cache(w, kb, vb, Cmax):
    c = orc.KVCache(w.N, kb.shape[1], w.Hkv, Cmax, w.hd)
    K, V = orc.widen(kb), orc.widen(vb)
    for n in range(w.N):
        for i in range(kb.shape[1]):
            c.K[n][i][:] = K[n, i]
            c.V[n][i][:] = V[n, i]
    return c


# ----------------------------------------------------------------------------- accept / top-k

def test_accept_matches_oracle_exactly():
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "accept_cases.json")))
    dr, _, _ = make(di.TINY, 80, 8)
    B = g["B"]
    d = np.array([c["draft"] for c in g["cases"]], np.int32)
    t = np.array([c["target"] for c in g["cases"]], np.int32)
    rng = np.random.default_rng(1)
    d = np.vstack([d, rng.integers(0, 3, (300, B - 1))]).astype(np.int32)
    t = np.vstack([t, rng.integers(0, 3, (300, B))]).astype(np.int32)
    tau, bonus = torch.empty(len(d), dtype=torch.int32, device="cuda"), torch.empty(len(d), dtype=torch.int32, device="cuda")
    dr.accept(len(d), i32(d), i32(t), tau, bonus)
    ot, ob = orc.accept(d, t)
    assert np.array_equal(tau.cpu().numpy(), ot)
    assert np.array_equal(bonus.cpu().numpy(), ob)
    for c, tt, bb in zip(g["cases"], tau.cpu().numpy(), bonus.cpu().numpy()):
        assert (tt, bb) == (c["tau"], c["bonus"])


@pytest.mark.parametrize("k", [1, 5, 16])
def test_accept_topk_reads_the_first_entry_of_each_list(k):
    # dflash_accept_topk on [nb, B-1, k] lists equals the oracle's accept of their first
    # column; the other entries (set to match the target everywhere) must not be read
    dr, _, _ = make(di.TINY, 80, 8)
    B = di.TINY.B
    rng = np.random.default_rng(10 + k)
    n = 257
    t = rng.integers(0, 3, (n, B)).astype(np.int32)
    d = np.where(rng.random((n, B - 1)) < 0.8, t[:, :B - 1], rng.integers(0, 3, (n, B - 1))).astype(np.int32)
    lists = np.repeat(t[:, :B - 1, None], k, axis=2).astype(np.int32)
    lists[:, :, 0] = d
    tau = torch.empty(n, dtype=torch.int32, device="cuda")
    bonus = torch.empty(n, dtype=torch.int32, device="cuda")
    dr.accept_topk(n, i32(lists), k, i32(t), tau, bonus)
    ot, ob = orc.accept(d, t)
    assert np.array_equal(tau.cpu().numpy(), ot)
    assert np.array_equal(bonus.cpu().numpy(), ob)
    assert (ot < B).any() and (ot == B).any()  # both a rejection and a full acceptance occur


@pytest.mark.parametrize("rows,cols,k", [(7, 5000, 16), (1, 151936, 16), (3, 17, 16), (5, 300, 1)])
def test_topk_exact_with_ties(rows, cols, k):
    dr, _, _ = make(di.TINY, 80, 8)
    rng = np.random.default_rng(cols)
    logits = rng.integers(-3, 4, (rows, cols)).astype(np.float32)  # dense exact ties
    ids = torch.empty(rows, k, dtype=torch.int32, device="cuda")
    vals = torch.empty(rows, k, dtype=torch.float32, device="cuda")
    dr.topk(rows, cols, torch.tensor(logits, device="cuda"), k, ids, vals)
    oi, ov = orc.topk(logits.astype(np.float64), k)
    assert np.array_equal(ids.cpu().numpy(), oi)
    assert np.array_equal(vals.cpu().numpy(), ov.astype(np.float32))


# ----------------------------------------------------------------------------- LM head

@pytest.mark.parametrize("w", [di.TINY, MEDIUM, MEDIUM_B8], ids=lambda w: w.name)
def test_lm_head_topk_stage(w):
    bits = di.make_weights(w)
    # duplicate LM-head rows: exact logit ties that must resolve to the lower id
    bits["W_lm"][w.V - 2] = bits["W_lm"][5]
    bits["W_lm"][w.V - 3] = bits["W_lm"][5]
    dr, W, _ = make(w, 64, w.B, bits=bits)
    hid_bits = di.normal_bf16("hidden", (w.nb, w.B, w.D), 1.0)
    hid = bf16(hid_bits)
    k = w.k_top
    ids = torch.empty(w.nb, w.B - 1, k, dtype=torch.int32, device="cuda")
    vals = torch.empty(w.nb, w.B - 1, k, dtype=torch.float32, device="cuda")
    logits = torch.empty(w.nb, w.B - 1, w.V, dtype=torch.float32, device="cuda")
    dr.lm_head_topk(w.nb, hid, k, ids, vals, logits)
    ol = orc.lm_logits(W, orc.widen(hid_bits))
    err = assert_close(logits.cpu().numpy(), ol, "logits")
    assert err < 1e-3, f"fp32-accumulated logits drift {err}"
    und = check_topk(ids.cpu().numpy(), vals.cpu().numpy(), ol, k, "lm_head top-k", abs_delta=2e-3)
    print(f"{w.name}: {und} top-k positions within 2e-3 of the next value")
    gi = ids.cpu().numpy().reshape(-1, k)
    gl = logits.cpu().numpy().reshape(-1, w.V)
    assert np.array_equal(gi, own_logits_topk(gl, k)), "fused selection differs from the kernel's own logits"
    for r in range(gi.shape[0]):
        assert np.array_equal(gl[r, 5], gl[r, w.V - 2]), "duplicate rows must tie exactly"
        row = gi[r].tolist()
        for dup in (w.V - 2, w.V - 3):
            if dup in row:
                assert 5 in row and row.index(5) < row.index(dup)


def own_logits_topk(gl, k):
    """Top-k of each row of the GPU's own fp32 logits: value descending, ties to the lower id."""
    ids = np.zeros((gl.shape[0], k), np.int64)
    for r in range(gl.shape[0]):
        ids[r] = np.lexsort((np.arange(gl.shape[1]), -gl[r].astype(np.float64)))[:k]
    return ids


@pytest.mark.parametrize("V", [4096, 151936])
def test_lm_head_topk_dense_ties_exact(V):
    """W_lm rows drawn from seven distinct rows: every row's logits take seven values, so
    the top-16 is decided by the lower-id rule across chunks, epilogue groups and
    vocabulary ranges. The fused selection must equal, exactly, the top-k of the kernel's
    own fp32 logits and the oracle's top-k of the fp64 logits (seven values far apart)."""
    w = di.TINY.with_(name=f"tiny_ties_v{V}", V=V, nb=4)
    bits = di.make_weights(w)
    rng = np.random.default_rng(V)
    pick = rng.integers(0, 7, V)
    bits["W_lm"] = di.normal_bf16("wlm_ties", (7, w.D), 1.0)[pick].copy()
    dr, W, _ = make(w, 64, w.B, bits=bits)
    hid_bits = di.normal_bf16("hidden_ties", (w.nb, w.B, w.D), 1.0)
    k = w.k_top
    ids = torch.empty(w.nb, w.B - 1, k, dtype=torch.int32, device="cuda")
    vals = torch.empty(w.nb, w.B - 1, k, dtype=torch.float32, device="cuda")
    logits = torch.empty(w.nb, w.B - 1, w.V, dtype=torch.float32, device="cuda")
    dr.lm_head_topk(w.nb, bf16(hid_bits), k, ids, vals, logits)
    gi = ids.cpu().numpy().reshape(-1, k)
    gv = vals.cpu().numpy().reshape(-1, k)
    gl = logits.cpu().numpy().reshape(-1, V)
    want = own_logits_topk(gl, k)
    assert np.array_equal(gi, want)
    assert np.array_equal(gv, np.take_along_axis(gl, want, 1))
    ol = orc.lm_logits(W, orc.widen(hid_bits)).reshape(-1, V)
    oi, _ = orc.topk(ol, k)
    # rows whose seven values are all more than 1e-2 apart in fp64 (fp32 cannot reorder them)
    gaps = np.array([np.diff(np.unique(r)).min() for r in ol])
    far = gaps > 1e-2
    assert far.mean() > 0.5
    assert np.array_equal(gi[far], oi[far])


@pytest.mark.parametrize("V,k", [(1000, 16), (1000, 5), (4096, 1)])
def test_lm_head_topk_few_ranges(V, k):
    """Fewer vocabulary ranges than k (every candidate reaches the final placement) and
    small k, against the oracle's logits of the same seeded hidden rows (exact selection
    wherever the oracle's margin exceeds the fp32-versus-fp64 difference)."""
    w = di.TINY.with_(name=f"tiny_v{V}", V=V)
    dr, W, _ = make(w, 64, w.B)
    hid_bits = di.normal_bf16("hidden_fr", (w.nb, w.B, w.D), 1.0)
    ids = torch.empty(w.nb, w.B - 1, k, dtype=torch.int32, device="cuda")
    vals = torch.empty(w.nb, w.B - 1, k, dtype=torch.float32, device="cuda")
    logits = torch.empty(w.nb, w.B - 1, w.V, dtype=torch.float32, device="cuda")
    dr.lm_head_topk(w.nb, bf16(hid_bits), k, ids, vals, logits)
    ol = orc.lm_logits(W, orc.widen(hid_bits)).reshape(-1, V)
    err = assert_close(logits.cpu().numpy().reshape(-1, V), ol, "logits")
    assert err < 1e-3
    check_topk(ids.cpu().numpy(), vals.cpu().numpy(), ol, k, "few-range top-k", abs_delta=2e-3)


# ----------------------------------------------------------------------------- ctx_project

@pytest.mark.parametrize("w", [di.TINY, MEDIUM, MEDIUM_ALL, TINY_FILM, MEDIUM_FILM],
                         ids=lambda w: w.name)
def test_ctx_project_stage(w):
    Cmax, R = 96, w.B
    dr, W, _ = make(w, Cmax, R)
    rng = np.random.default_rng(2)
    nb = w.nb
    hv_bits = di.verifier_rows(w, R, name="hv_stage")
    n_commit = rng.integers(0, R + 1, nb).astype(np.int32)
    n_commit[0] = R
    if nb > 1:
        n_commit[1] = 0
    c0 = rng.integers(0, Cmax - R, nb).astype(np.int32)
    relay = (w.flags & di.FLAG_RELAY) != 0
    a = rng.integers(0, w.B, nb).astype(np.int32) if relay else None
    film = {}
    if w.flags & di.FLAG_FILM:
        b, y = rng.integers(0, w.V, (2, nb)).astype(np.int32)
        film = dict(relay_b=b, relay_y=y)
        a[0] = 0  # the most relayed rows
    ctx = i32(c0)
    x0 = torch.full((nb, w.B, w.D), float("nan"), dtype=torch.bfloat16, device="cuda") if relay else None
    dr.ctx_project(nb, R, bf16(hv_bits), i32(n_commit), ctx, relay_a=None if a is None else i32(a),
                   x0_relay=x0, **{k: i32(v) for k, v in film.items()})
    assert dr.status() == 0
    cache = orc.KVCache(w.N, nb, w.Hkv, Cmax, w.hd)
    new_len, x0r = orc.ctx_project(w, W, orc.widen(hv_bits), n_commit, c0, cache, relay_a=a,
                                   **film)
    assert np.array_equal(ctx.cpu().numpy(), new_len)
    K, V = f64(dr.kcache), f64(dr.vcache)
    for n in range(w.N):
        for i in range(nb):
            lo, hi = c0[i], c0[i] + n_commit[i]
            assert_close(K[n, i][:, lo:hi], cache.K[n][i][:, lo:hi], f"K_c layer {n} seq {i}")
            assert_close(V[n, i][:, lo:hi], cache.V[n][i][:, lo:hi], f"V_c layer {n} seq {i}")
            assert not K[n, i][:, :lo].any() and not K[n, i][:, hi:].any(), "rows outside the append"
    if relay:
        g = f64(x0)
        assert_close(g, x0r, "x0_relay")
        assert np.array_equal(g == 0, x0r == 0), "relay placement"


def test_film_relay_short_rows_and_bad_tokens():
    """FiLM relay with fewer projected rows than the block (the k < R cut), every a from 0
    to B-1 (B-1 and B-2 relay nothing), then an out-of-range token: reported, read as zeros."""
    dflash, _ = lib()
    w = TINY_FILM.with_(nb=8)
    R = 5
    dr, W, _ = make(w, 64, R)
    hv_bits = di.verifier_rows(w, R, name="hv_film")
    a = np.array([0, 1, 2, 3, 4, 5, 6, 7], np.int32)
    b, y = di.relay_tokens(w)
    n_commit = np.full(w.nb, R, np.int32)
    x0 = torch.full((w.nb, w.B, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    dr.ctx_project(w.nb, R, bf16(hv_bits), i32(n_commit), i32(np.zeros(w.nb)), relay_a=i32(a),
                   x0_relay=x0, relay_b=i32(b), relay_y=i32(y))
    assert dr.status() == 0
    cache = orc.KVCache(w.N, w.nb, w.Hkv, 64, w.hd)
    _, x0r = orc.ctx_project(w, W, orc.widen(hv_bits), n_commit, np.zeros(w.nb), cache,
                             relay_a=a, relay_b=b, relay_y=y)
    g = f64(x0)
    assert_close(g, x0r, "x0_relay (FiLM)")
    assert np.array_equal(np.abs(g).sum(-1) > 0, np.abs(x0r).sum(-1) > 0), "relay placement"
    assert (np.abs(x0r).sum(-1) > 0).sum() == 3 + 2 + 1  # a = 0, 1, 2 with k < R = 5
    bad_b = b.copy()
    bad_b[0] = w.V
    dr.ctx_project(w.nb, R, bf16(hv_bits), i32(np.zeros(w.nb)), i32(np.zeros(w.nb)), relay_a=i32(a),
                   x0_relay=x0, relay_b=i32(bad_b), relay_y=i32(y))
    assert dr.status() == dflash.DFLASH_ERR_DEVICE_CHECK
    W0 = dict(W)  # the kernel reads the out-of-range row as zeros: an appended zero row E[V]
    W0["E"] = np.concatenate([W["E"], np.zeros((1, w.D))])
    _, x0z = orc.ctx_project(w, W0, orc.widen(hv_bits), np.zeros(w.nb), np.zeros(w.nb),
                             orc.KVCache(w.N, w.nb, w.Hkv, 64, w.hd), relay_a=a, relay_b=bad_b,
                             relay_y=y)
    assert_close(f64(x0)[0], x0z[0], "x0_relay with an out-of-range b")


# ----------------------------------------------------------------------------- draft_block

@pytest.mark.parametrize("w", [di.TINY, MEDIUM, MEDIUM_B8, MEDIUM_ALL], ids=lambda w: w.name)
def test_draft_block_stage(w):
    Cmax = 320
    dr, W, _ = make(w, Cmax, w.B)
    kb, vb = random_cache(w, w.nb, Cmax)
    dr.kcache.copy_(bf16(kb))
    dr.vcache.copy_(bf16(vb))
    lens = np.array([Cmax - w.B, 0, 65, 300, 64, 1, 63][: w.nb], dtype=np.int32)
    ids = di.block_ids(w, di.anchors(w))
    x0_bits = None
    if w.flags & di.FLAG_RELAY:
        x0_bits = di.normal_bf16("x0_relay", (w.nb, w.B, w.D), 1.0)
    out = torch.empty(w.nb, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(w.nb, i32(ids), i32(lens), out, x0_relay=None if x0_bits is None else bf16(x0_bits),
                   max_ctx_hint=Cmax)
    assert dr.status() == 0
    oc = oracle_cache(w, kb, vb, Cmax)
    want = orc.draft_block(w, W, ids, lens, oc, None if x0_bits is None else orc.widen(x0_bits))
    assert_close(f64(out), want, f"hidden {w.name}")


def test_draft_block_other_sequences_do_not_leak():
    """A sequence's hidden does not depend on the other sequences' tokens or caches
    (bitwise, same context lengths); with other lengths only the attention's split
    points move, so it stays within the stated tolerance of the oracle."""
    w = MEDIUM
    Cmax = 320
    dr, W, _ = make(w, Cmax, w.B)
    kb, vb = random_cache(w, w.nb, Cmax)
    dr.kcache.copy_(bf16(kb))
    dr.vcache.copy_(bf16(vb))
    oc = oracle_cache(w, kb, vb, Cmax)
    ids = di.block_ids(w, di.anchors(w))
    lens = np.array([200, 17, 300], np.int32)
    out1 = torch.empty(w.nb, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(w.nb, i32(ids), i32(lens), out1, max_ctx_hint=Cmax)
    ids2 = ids.copy()
    ids2[1:, 0] = (ids2[1:, 0] + 7) % (w.V - 1)
    dr.kcache[:, 1:].normal_()
    dr.vcache[:, 1:].normal_()
    out2 = torch.empty_like(out1)
    dr.draft_block(w.nb, i32(ids2), i32(lens), out2, max_ctx_hint=Cmax)
    assert torch.equal(out1[0], out2[0])
    out3 = torch.empty_like(out1)
    dr.draft_block(w.nb, i32(ids2), i32(np.array([200, 40, 90], np.int32)), out3, max_ctx_hint=Cmax)
    want = orc.draft_block(w, W, ids[:1], lens[:1], oc)
    assert_close(f64(out3[:1]), want, "hidden of sequence 0 with other lengths")
    assert dr.status() == 0


def test_draft_block_long_ragged():
    """Thousands of context rows per sequence, ragged down to 1 row: many 64-key units
    per attention CTA and several (sequence, kv head) segments per CTA."""
    w = MEDIUM.with_(name="medium_long_ragged", nb=6)
    Cmax = 4200
    dr, W, _ = make(w, Cmax, w.B)
    kb, vb = random_cache(w, w.nb, Cmax, seed=3)
    dr.kcache.copy_(bf16(kb))
    dr.vcache.copy_(bf16(vb))
    lens = np.array([4000, 1, 2500, 3333, 64, Cmax - w.B], np.int32)
    ids = di.block_ids(w, di.anchors(w))
    out = torch.empty(w.nb, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(w.nb, i32(ids), i32(lens), out, max_ctx_hint=Cmax)
    assert dr.status() == 0
    want = orc.draft_block(w, W, ids, lens, oracle_cache(w, kb, vb, Cmax))
    assert_close(f64(out), want, "hidden, long ragged contexts")


@pytest.mark.parametrize("w", [MEDIUM, MEDIUM_B8, MEDIUM_G8, di.TINY], ids=lambda w: w.name)
def test_attention_stage_spikes_ragged_nan_tail(w):
    """The attention stage on given bf16 q, K, V. Key rows carry spikes of growing size
    along the context (a common direction per kv head), so the running row maxima keep
    rising past the rescale threshold; lengths are ragged (0, 1, 63..65 context rows,
    the maximum); every cache row past ctx_len + B holds NaN, which must not reach the
    output (masked scores, zeroed V rows)."""
    nb, Cmax, layer = 6, 2200, 1
    dr, _, _ = make(w, Cmax, w.B, max_batch=nb)
    lens = np.array([Cmax - w.B, 0, 1, 63, 64, 1500][:nb], np.int32)
    shp = (w.N, nb, w.Hkv, Cmax, w.hd)
    K = 0.1 * orc.widen(di.normal_bf16("kspike", shp, 1.0, seed=5))
    V = orc.widen(di.normal_bf16("vspike", shp, 1.0, seed=5))
    r = orc.widen(di.normal_bf16("spike_dir", (w.N, w.Hkv, w.hd), 1.0, seed=5))
    for m, pos in enumerate(range(40, Cmax, 150)):
        K[:, :, :, pos, :] = (8.0 * (m + 1)) * r[:, None, :, :]
    for i, L in enumerate(lens + w.B):
        K[:, i, :, L:, :] = np.nan
        V[:, i, :, L:, :] = np.nan
    kb = di.f32_to_bf16_bits(K.astype(np.float32))
    vb = di.f32_to_bf16_bits(V.astype(np.float32))
    qb = di.normal_bf16("qspike", (nb, w.B, w.Hq, w.hd), 1.0, seed=5)
    dr.kcache.copy_(bf16(kb))
    dr.vcache.copy_(bf16(vb))
    out = torch.empty(nb, w.B, w.Hq, w.hd, dtype=torch.bfloat16, device="cuda")
    dr.attention(nb, layer, bf16(qb), i32(lens), out, max_ctx_hint=Cmax)
    assert dr.status() == 0
    q, Kw, Vw = orc.widen(qb), orc.widen(kb), orc.widen(vb)
    grp = w.Hq // w.Hkv
    want = np.zeros((nb, w.B, w.Hq, w.hd))
    for i in range(nb):
        L = int(lens[i]) + w.B
        for h in range(w.Hq):
            g = h // grp
            want[i, :, h] = orc.softmax_attention(q[i, :, h], Kw[layer, i, g, :L], Vw[layer, i, g, :L])
    assert_close(f64(out), want, f"attention {w.name}")


# ----------------------------------------------------------------------------- conv / select

def test_conv_stage():
    w = MEDIUM_ALL
    dr, W, _ = make(w, 64, w.B)
    M = w.nb * w.B
    x0 = np.random.default_rng(3).standard_normal((M, w.D)).astype(np.float32)
    x = torch.tensor(x0, device="cuda")
    dr.conv(1, 2, w.nb, x)
    assert dr.status() == 0
    p = "layer1.conv2."
    xf = x0.astype(np.float64).reshape(w.nb, w.B, w.D)
    got = x.cpu().numpy().reshape(w.nb, w.B, w.D)
    for i in range(w.nb):
        want = orc.dyn_conv(xf[i], W[p + "W0"], W[p + "W1"], W[p + "base"], w.conv_group)
        assert_close(got[i], want, f"conv seq {i}")


def test_select_stage():
    w = MEDIUM_ALL
    dr, W, _ = make(w, 64, w.B)
    rng = np.random.default_rng(4)
    k = w.k_top
    cand = np.stack([rng.permutation(w.V)[:k] for _ in range(w.nb * (w.B - 1))]).reshape(w.nb, w.B - 1, k)
    vals = rng.standard_normal((w.nb, w.B - 1, k)).astype(np.float32)
    hid_bits = di.normal_bf16("sel_hidden", (w.nb, w.B, w.D), 1.0)
    ids = di.block_ids(w, di.anchors(w))
    path = torch.empty(w.nb, w.B - 1, dtype=torch.int32, device="cuda")
    dr.select(w.nb, k, i32(cand), torch.tensor(vals, device="cuda"), bf16(hid_bits), i32(ids), path)
    assert dr.status() == 0
    want, margin = orc.select_path(w, W, cand, vals.astype(np.float64), orc.widen(hid_bits),
                                   ids[:, 0], return_margins=True)
    got = path.cpu().numpy()
    decided = 0
    for i in range(w.nb):
        for t in range(w.B - 1):
            if margin[i, t] <= 1e-2 * max(1.0, abs(vals[i, t]).max()):
                assert got[i, t] in cand[i, t]
                break
            assert got[i, t] == want[i, t], f"seq {i} offset {t + 1}"
            decided += 1
    assert decided > 0


# ----------------------------------------------------------------------------- whole step

@pytest.mark.parametrize("w", [di.TINY, MEDIUM_ALL, MEDIUM_FILM], ids=lambda w: w.name)
def test_full_step(w):
    """Prefill through ctx_project, then one draft step (append, draft, LM head, accept)."""
    Cmax, C = 96, 70
    dr, W, _ = make(w, Cmax, C)
    nb = w.nb
    hv_pre = di.verifier_rows(w, C, name="hv_prefill")
    tp = np.minimum(di.tau_prev(w), w.B).astype(np.int32)
    ctx = i32(np.zeros(nb, np.int32))
    dr.ctx_project(nb, C, bf16(hv_pre), i32(C - tp), ctx)
    cache = orc.KVCache(w.N, nb, w.Hkv, Cmax, w.hd)
    lens, _ = orc.ctx_project(w, W, orc.widen(hv_pre), C - tp, np.zeros(nb), cache)
    relay = (w.flags & di.FLAG_RELAY) != 0
    hv = di.verifier_rows(w, w.B, name="hv_step")
    a = (tp - 1).astype(np.int32)
    x0 = torch.empty(nb, w.B, w.D, dtype=torch.bfloat16, device="cuda") if relay else None
    film = {}
    if w.flags & di.FLAG_FILM:
        b, y = di.relay_tokens(w)
        film = dict(relay_b=b, relay_y=y)
    dr.ctx_project(nb, w.B, bf16(hv), i32(tp), ctx, relay_a=i32(a) if relay else None, x0_relay=x0,
                   **{k: i32(v) for k, v in film.items()})
    ids = di.block_ids(w, di.anchors(w))
    out = torch.empty(nb, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(nb, i32(ids), ctx, out, x0_relay=x0, max_ctx_hint=C)
    k = w.k_top
    tid = torch.empty(nb, w.B - 1, k, dtype=torch.int32, device="cuda")
    tv = torch.empty(nb, w.B - 1, k, dtype=torch.float32, device="cuda")
    tl = torch.empty(nb, w.B - 1, w.V, dtype=torch.float32, device="cuda")
    dr.lm_head_topk(nb, out, k, tid, tv, tl)
    assert dr.status() == 0
    o = orc.draft_step(w, W, orc.widen(hv), tp, lens, cache, ids, np.zeros((nb, w.B), np.int32),
                       relay_a=a if relay else None, **film)
    assert np.array_equal(ctx.cpu().numpy(), o["ctx_len"])
    assert int(o["ctx_len"].max()) <= C
    if relay:
        assert_close(f64(x0), o["x0_relay"], "x0_relay")
    assert_close(f64(out), o["hidden"], "hidden")
    assert_close(tl.cpu().numpy(), o["logits"], "logits")
    und = check_topk(tid.cpu().numpy(), tv.cpu().numpy(), o["logits"], k, "top-k")
    draft = tid[..., 0].contiguous()
    if w.flags & di.FLAG_SELECT:
        path = torch.empty(nb, w.B - 1, dtype=torch.int32, device="cuda")
        dr.select(nb, k, tid, tv, out, i32(ids), path)
        draft = path
    # the target rows come from the oracle's draft; tau compares wherever the GPU drafted
    # the oracle's tokens
    target = di.target_row_from_draft(o["draft"], w.V)
    tau = torch.empty(nb, dtype=torch.int32, device="cuda")
    bonus = torch.empty(nb, dtype=torch.int32, device="cuda")
    dr.accept(nb, draft, i32(target), tau, bonus)
    ot, ob = orc.accept(o["draft"], target)
    gd = draft.cpu().numpy()
    same = np.array([(gd[j, :min(int(ot[j]), w.B - 1)] == o["draft"][j, :min(int(ot[j]), w.B - 1)]).all()
                     for j in range(nb)])
    assert np.array_equal(tau.cpu().numpy()[same], ot[same]) and np.array_equal(bonus.cpu().numpy()[same], ob[same])
    tau2 = torch.empty(nb, dtype=torch.int32, device="cuda")
    bonus2 = torch.empty(nb, dtype=torch.int32, device="cuda")
    dr.accept(nb, i32(o["draft"]), i32(target), tau2, bonus2)  # both sides read the oracle's draft
    assert np.array_equal(tau2.cpu().numpy(), ot) and np.array_equal(bonus2.cpu().numpy(), ob)
    print(f"{w.name}: {und} of {nb * (w.B - 1) * k} top-k positions under the decision margin")


# ----------------------------------------------------------------------------- failure paths

def test_argument_errors():
    dflash, drafter = lib()
    dr, _, _ = make(di.TINY, 80, 8)
    with pytest.raises(dflash.DflashError) as e:
        dr.ctx_project(5, 8, torch.empty(1, device="cuda"), i32([1]), i32([0]))
    assert e.value.code == dflash.DFLASH_ERR_INVALID_ARG
    with pytest.raises(dflash.DflashError) as e:
        dr.lm_head_topk(1, torch.empty(8, 256, dtype=torch.bfloat16, device="cuda"), 17,
                        i32([0]), i32([0]))
    assert e.value.code == dflash.DFLASH_ERR_INVALID_ARG
    bad = dflash.dflash_config.from_buffer_copy(dr.cfg)
    bad.B = 17
    with pytest.raises(dflash.DflashError) as e:
        dflash.dflash_create(bad)
    assert e.value.code == dflash.DFLASH_ERR_UNSUPPORTED_SHAPE


def test_context_beyond_hint_is_reported():
    dflash, _ = lib()
    w = di.TINY
    dr, _, _ = make(w, 80, 8)
    out = torch.empty(1, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(1, i32(di.block_ids(w, [3])), i32([50]), out, max_ctx_hint=40)
    assert dr.status() == dflash.DFLASH_ERR_DEVICE_CHECK
    assert dr.status() == dflash.DFLASH_OK  # status clears on read


def test_bounded_wait_times_out_and_context_survives():
    """A wait that nothing signals runs out, reports TIMEOUT, and the GPU stays usable."""
    dflash, _ = lib()
    w = di.TINY
    dr, W, bits = make(w, 80, 8, max_spin=2000, flags_extra=dflash.FLAG_TEST_STALL)
    out = torch.empty(1, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(1, i32(di.block_ids(w, [3])), i32([0]), out, max_ctx_hint=16)
    assert dr.status() == dflash.DFLASH_ERR_TIMEOUT
    del dr
    dr2, W, _ = make(w, 80, 8, bits=bits)
    dr2.draft_block(1, i32(di.block_ids(w, [3])), i32([0]), out, max_ctx_hint=16)
    assert dr2.status() == dflash.DFLASH_OK
    want = orc.draft_block(w, W, di.block_ids(w, [3]), [0], orc.KVCache(w.N, 1, w.Hkv, 80, w.hd))
    assert_close(f64(out), want, "hidden after a timed-out call")


# ----------------------------------------------------------------------------- shared K/V projection

def test_shared_context_and_block_kv_projection():
    """The shared-projection variant ([DFlash] 二、块扩散草稿: the attention equations write
    W^K_c, W^V_c for the context and W^K_b, W^V_b for the block; reading c4 keeps them
    separate and obtains the shared form by aliasing): every layer's Wk_c / Wv_c pointers
    are the k_b / v_b row blocks of the same layer's fused W_qkv. The oracle runs with the
    same aliased matrices; a whole step (prefill, append, draft, LM head) matches it."""
    _, drafter = lib()
    w = MEDIUM
    bits = di.make_weights(w)
    qd, kd = w.Hq * w.hd, w.Hkv * w.hd
    for n in range(w.N):
        qkv = bits[f"layer{n}.W_qkv"]
        bits[f"layer{n}.Wk_c"] = qkv[qd:qd + kd]
        bits[f"layer{n}.Wv_c"] = qkv[qd + kd:qd + 2 * kd]
    dev = {k: drafter.to_device_bf16(v) for k, v in bits.items() if ".Wk_c" not in k and ".Wv_c" not in k}
    for n in range(w.N):  # views into W_qkv: the library reads the same memory for both
        qkv = dev[f"layer{n}.W_qkv"]
        dev[f"layer{n}.Wk_c"] = qkv[qd:qd + kd]
        dev[f"layer{n}.Wv_c"] = qkv[qd + kd:qd + 2 * kd]
        assert dev[f"layer{n}.Wk_c"].data_ptr() == qkv.data_ptr() + qd * w.D * 2
    Cmax, C = 96, 70
    dr = drafter.Drafter(w, dev, w.nb, Cmax, C)
    W = orc.widen_all(bits)
    nb = w.nb
    hv_pre = di.verifier_rows(w, C, name="hv_prefill_shared")
    tp = np.minimum(di.tau_prev(w), w.B).astype(np.int32)
    ctx = i32(np.zeros(nb, np.int32))
    dr.ctx_project(nb, C, bf16(hv_pre), i32(C - tp), ctx)
    cache = orc.KVCache(w.N, nb, w.Hkv, Cmax, w.hd)
    lens, _ = orc.ctx_project(w, W, orc.widen(hv_pre), C - tp, np.zeros(nb), cache)
    hv = di.verifier_rows(w, w.B, name="hv_step_shared")
    dr.ctx_project(nb, w.B, bf16(hv), i32(tp), ctx)
    ids = di.block_ids(w, di.anchors(w))
    out = torch.empty(nb, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(nb, i32(ids), ctx, out, max_ctx_hint=C)
    k = w.k_top
    tid = torch.empty(nb, w.B - 1, k, dtype=torch.int32, device="cuda")
    tv = torch.empty(nb, w.B - 1, k, dtype=torch.float32, device="cuda")
    tl = torch.empty(nb, w.B - 1, w.V, dtype=torch.float32, device="cuda")
    dr.lm_head_topk(nb, out, k, tid, tv, tl)
    assert dr.status() == 0
    o = orc.draft_step(w, W, orc.widen(hv), tp, lens, cache, ids, np.zeros((nb, w.B), np.int32))
    assert np.array_equal(ctx.cpu().numpy(), o["ctx_len"])
    gk = f64(dr.kcache)
    for n in range(w.N):  # the appended context rows use the shared (block) projection
        for i in range(nb):
            assert_close(gk[n, i, :, :int(o["ctx_len"][i])], cache.K[n][i][:, :int(o["ctx_len"][i])],
                         f"K_c layer {n} seq {i}")
    assert_close(f64(out), o["hidden"], "hidden (shared projection)")
    assert_close(tl.cpu().numpy(), o["logits"], "logits (shared projection)")
    check_topk(tid.cpu().numpy(), tv.cpu().numpy(), o["logits"], k, "top-k (shared projection)")


# ----------------------------------------------------------------------------- stacked tiles

def test_wide_batch_takes_stacked_tiles():
    """320 sequences of the medium drafter (22,400 prefill rows, 5,120 block rows): the
    context projection's W_c and K/V GEMMs (prefill and step) and the SwiGLU gate|up GEMM run
    256-row M-stacked tiles, every GEMM visits its tiles in groups of row tiles, and the LM
    head has 38 row tiles. Sequences are independent, so three of them (first, middle,
    last) against the oracle fix the result: appended K/V rows, hidden, logits and top-k."""
    w = MEDIUM.with_(name="medium_wide_batch_nb320", nb=320)
    nb, B, k = w.nb, w.B, w.k_top
    Cmax, C = 96, 70
    dr, W, _ = make(w, Cmax, C)
    sample = [0, nb // 2 - 3, nb - 1]
    hv_pre = di.verifier_rows(w, C, name="hv_prefill_wide")
    tp = np.minimum(di.tau_prev(w), B).astype(np.int32)
    pre = (C - tp).astype(np.int32)
    ctx = i32(np.zeros(nb, np.int32))
    dr.ctx_project(nb, C, bf16(hv_pre), i32(pre), ctx)
    hv = di.verifier_rows(w, B, name="hv_step_wide")
    dr.ctx_project(nb, B, bf16(hv), i32(tp), ctx)
    ids = di.block_ids(w, di.anchors(w))
    out = torch.empty(nb, B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(nb, i32(ids), ctx, out, max_ctx_hint=C)
    tid = torch.empty(nb, B - 1, k, dtype=torch.int32, device="cuda")
    tv = torch.empty(nb, B - 1, k, dtype=torch.float32, device="cuda")
    tl = torch.empty(nb, B - 1, w.V, dtype=torch.float32, device="cuda")
    dr.lm_head_topk(nb, out, k, tid, tv, tl)
    assert dr.status() == 0
    s = np.array(sample)
    cache = orc.KVCache(w.N, len(sample), w.Hkv, Cmax, w.hd)
    lens, _ = orc.ctx_project(w, W, orc.widen(hv_pre[s]), pre[s], np.zeros(len(sample)), cache)
    o = orc.draft_step(w, W, orc.widen(hv[s]), tp[s], lens, cache, ids[s], np.zeros((len(sample), B), np.int32))
    assert np.array_equal(ctx.cpu().numpy()[s], o["ctx_len"])
    gk, gv = dr.kcache, dr.vcache
    for si, i in enumerate(sample):
        L = int(o["ctx_len"][si])
        for n in range(w.N):
            assert_close(f64(gk[n, i, :, :L]), cache.K[n][si][:, :L], f"K rows seq {i} layer {n}")
            assert_close(f64(gv[n, i, :, :L]), cache.V[n][si][:, :L], f"V rows seq {i} layer {n}")
    assert_close(f64(out[s]), o["hidden"], "hidden (stacked tiles)")
    assert_close(tl[s].cpu().numpy(), o["logits"], "logits (stacked tiles)")
    check_topk(tid[s].cpu().numpy(), tv[s].cpu().numpy(), o["logits"], k, "top-k (stacked tiles)")
