"""Paged KV cache through the C ABI: pools of 64-row pages and a block table per
sequence, against the oracle's paged view (oracle.paged_rows / cache_from_pages).

Pages are handed out in a seeded random order, two sequences share their first pages
(a common prefix that no call writes), and spare pages belong to no sequence: after a
context append (ctx_project) and a draft block (which appends the block's K/V rows and
attends through the table) the appended rows and the hidden match the oracle, and every
page the step does not write keeps its bits.
"""
import numpy as np
import pytest
import torch

import dflash_inputs as di
from _parity import assert_close
from oracle import dflash_oracle as orc
from test_gpu_parity import MEDIUM, MEDIUM_G8, bf16, f64, i32, lib, make

pytestmark = pytest.mark.gpu

PR = orc.PAGE_ROWS


def page_plan(nb, pps, spare, shared, seed):
    """Block table [nb, pps] over nb * pps - shared * (nb > 1) + spare pages in a seeded
    random order; sequence 1 reuses sequence 0's first `shared` pages."""
    rng = np.random.default_rng(seed)
    need = nb * pps - (shared if nb > 1 else 0)
    P = need + spare
    ids = rng.permutation(P)
    table = np.empty((nb, pps), np.int32)
    k = 0
    for i in range(nb):
        for q in range(pps):
            if i == 1 and q < shared:
                table[i, q] = table[0, q]
            else:
                table[i, q] = ids[k]
                k += 1
    return table, P


def pools(w, P, seed):
    shp = (w.N, P, w.Hkv, PR, w.hd)
    return di.normal_bf16("kpool", shp, 1.0, seed=seed), di.normal_bf16("vpool", shp, 1.0, seed=seed)


def written_pages(table, lo, hi):
    """Pages holding rows [lo[i], hi[i]) of each sequence."""
    out = set()
    for i in range(len(lo)):
        for r in range(int(lo[i]), int(hi[i])):
            out.add(int(table[i, r // PR]))
    return out


@pytest.mark.parametrize("w", [MEDIUM, MEDIUM_G8, di.TINY.with_(name="tiny_nb3", nb=3)],
                         ids=lambda w: w.name)
def test_paged_append_and_draft(w):
    nb, Cmax, R = w.nb, 320, w.B
    pps = Cmax // PR
    shared = 2 if nb > 1 else 0
    table, P = page_plan(nb, pps, spare=3, shared=shared, seed=11)
    dr, W, _ = make(w, Cmax, R, num_pages=P)
    kp, vp = pools(w, P, seed=12)
    dr.kcache.copy_(bf16(kp))
    dr.vcache.copy_(bf16(vp))
    dr.set_block_table(i32(table))
    # appends start past the shared prefix; one sequence ends exactly at Cmax
    base = np.array([shared * PR + 5, shared * PR, 150, 40, 7][:nb], np.int32)
    n_commit = np.array([R, 3, 0, R, 1][:nb], np.int32)
    base[-1] = Cmax - w.B - n_commit[-1]
    hv = di.verifier_rows(w, R, name="hv_paged")
    ctx = i32(base)
    dr.ctx_project(nb, R, bf16(hv), i32(n_commit), ctx)
    ids = di.block_ids(w, di.anchors(w))
    out = torch.empty(nb, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(nb, i32(ids), ctx, out, max_ctx_hint=Cmax - w.B)
    assert dr.status() == 0

    cache = orc.cache_from_pages(orc.widen(kp), orc.widen(vp), table, nb, Cmax)
    new_len, _ = orc.ctx_project(w, W, orc.widen(hv), n_commit, base, cache)
    assert np.array_equal(ctx.cpu().numpy(), new_len)
    want = orc.draft_block(w, W, ids, new_len, cache)
    assert_close(f64(out), want, f"hidden, paged {w.name}")

    gk, gv = f64(dr.kcache), f64(dr.vcache)
    # appended context rows, read back through the table (the block's own K/V rows are
    # compared with the contiguous layout in test_paged_matches_contiguous_bitwise)
    for n in range(w.N):
        for i in range(nb):
            lo, hi = int(base[i]), int(new_len[i])
            assert_close(orc.paged_rows(gk[n], table, i, hi)[:, lo:], cache.K[n][i][:, lo:hi], f"K rows seq {i}")
            assert_close(orc.paged_rows(gv[n], table, i, hi)[:, lo:], cache.V[n][i][:, lo:hi], f"V rows seq {i}")
    # every other page keeps its bits: spare pages, the shared prefix, untouched rows
    wp = written_pages(table, base, new_len + w.B)
    kb = dr.kcache.view(torch.int16).cpu().numpy().view(np.uint16)
    vb = dr.vcache.view(torch.int16).cpu().numpy().view(np.uint16)
    for pg in range(P):
        if pg not in wp:
            assert np.array_equal(kb[:, pg], kp[:, pg]) and np.array_equal(vb[:, pg], vp[:, pg]), f"page {pg}"
    for i in range(nb):
        lo, hi = int(base[i]), int(new_len[i]) + w.B
        for r in list(range(lo - lo % PR, lo)) + list(range(hi, min(Cmax, hi + PR - hi % PR if hi % PR else hi))):
            pg, rr = table[i, r // PR], r % PR
            assert np.array_equal(kb[:, pg, :, rr], kp[:, pg, :, rr]), f"row {r} of seq {i}"


def test_paged_matches_contiguous_bitwise():
    """The same caches laid out contiguously and as shuffled pages give the same hidden
    and the same cache rows after the block's K/V append, bit for bit (same units and
    split points; only the addresses differ)."""
    w = MEDIUM
    nb, Cmax = w.nb, 320
    pps = Cmax // PR
    table, P = page_plan(nb, pps, spare=2, shared=0, seed=21)
    drc, _, bits = make(w, Cmax, w.B)
    drp, _, _ = make(w, Cmax, w.B, bits=bits, num_pages=P)
    kc, vc = di.normal_bf16("kc_cont", (w.N, nb, w.Hkv, Cmax, w.hd), 1.0), \
        di.normal_bf16("vc_cont", (w.N, nb, w.Hkv, Cmax, w.hd), 1.0)
    drc.kcache.copy_(bf16(kc))
    drc.vcache.copy_(bf16(vc))
    kp = np.zeros((w.N, P, w.Hkv, PR, w.hd), np.uint16)
    vp = np.zeros_like(kp)
    for i in range(nb):
        for q in range(pps):
            kp[:, table[i, q]] = kc[:, i, :, q * PR:(q + 1) * PR]
            vp[:, table[i, q]] = vc[:, i, :, q * PR:(q + 1) * PR]
    drp.kcache.copy_(bf16(kp))
    drp.vcache.copy_(bf16(vp))
    drp.set_block_table(i32(table))
    lens = np.array([Cmax - w.B, 1, 200], np.int32)[:nb]
    ids = di.block_ids(w, di.anchors(w))
    oc = torch.empty(nb, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    op = torch.empty_like(oc)
    drc.draft_block(nb, i32(ids), i32(lens), oc, max_ctx_hint=Cmax - w.B)
    drp.draft_block(nb, i32(ids), i32(lens), op, max_ctx_hint=Cmax - w.B)
    assert drc.status() == 0 and drp.status() == 0
    assert torch.equal(oc, op)
    kcb = drc.kcache.view(torch.int16).cpu().numpy()
    vcb = drc.vcache.view(torch.int16).cpu().numpy()
    kpb = drp.kcache.view(torch.int16).cpu().numpy()
    vpb = drp.vcache.view(torch.int16).cpu().numpy()
    for n in range(w.N):
        for i in range(nb):
            L = int(lens[i]) + w.B
            assert np.array_equal(orc.paged_rows(kpb[n], table, i, L), kcb[n, i, :, :L]), f"K layer {n} seq {i}"
            assert np.array_equal(orc.paged_rows(vpb[n], table, i, L), vcb[n, i, :, :L]), f"V layer {n} seq {i}"


def test_paged_errors_and_bad_page_reported():
    """No table: refused before any launch. A table entry outside the pool that the step
    reaches: reported by the status word, never dereferenced."""
    dflash, _ = lib()
    w = di.TINY
    Cmax = 128
    dr, _, _ = make(w, Cmax, w.B, max_batch=1, num_pages=3)
    out = torch.empty(1, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    ids = i32(di.block_ids(w, [3]))
    with pytest.raises(dflash.DflashError) as e:
        dr.draft_block(1, ids, i32([10]), out, max_ctx_hint=Cmax - w.B)
    assert e.value.code == dflash.DFLASH_ERR_INVALID_ARG
    for bad in (3, -1):
        dr.set_block_table(i32([[0, bad]]))
        dr.draft_block(1, ids, i32([70]), out, max_ctx_hint=Cmax - w.B)  # rows 70..77: page 1
        assert dr.status() == dflash.DFLASH_ERR_DEVICE_CHECK
    dr.set_block_table(i32([[0, 2]]))
    dr.draft_block(1, ids, i32([70]), out, max_ctx_hint=Cmax - w.B)
    assert dr.status() == dflash.DFLASH_OK
    drc, _, _ = make(w, Cmax, w.B, max_batch=1)
    with pytest.raises(dflash.DflashError) as e:
        drc.set_block_table(i32([[0, 1]]))
    assert e.value.code == dflash.DFLASH_ERR_INVALID_ARG
    bad = dflash.dflash_config.from_buffer_copy(dr.cfg)
    bad.Cmax = 100
    with pytest.raises(dflash.DflashError) as e:
        dflash.dflash_create(bad)
    assert e.value.code == dflash.DFLASH_ERR_UNSUPPORTED_SHAPE
