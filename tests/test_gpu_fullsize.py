"""Full-size parity: each workload at its full shape and batch, through the same C-ABI
calls and batch sizes bench.py times, with the oracle computing sampled sequences one
by one (sequences are independent, so a sample fixes them exactly).

Stage-wise checks, where both sides consume the same seeded inputs, use the stated
tolerance |g - o| <= 2e-2 + 1e-2|o|: appended K/V rows and relay rows (same verifier rows),
the LM-head logits and top-k at the full vocabulary on seeded hidden rows, the selector on
seeded candidates, values and hidden rows. Accept runs on targets built from the oracle's
draft and compares wherever the GPU drafted the oracle's tokens. The end-to-end drafter
hidden after N = 5 layers at D = 2560..4096 carries the bf16 storage error of about
20 rounding points. tests/bf16_storage_model.py rounds the fp64 oracle to bf16 at exactly
the kernel path's storage points; on the sampled sequences of these workloads it deviates
from fp64 by max 0.044-0.072, max |err|/(1+|o|) 0.034-0.056, mean 0.0083-0.0098, with
96.0-98.5% of elements within the stated tolerance. The GPU adds an independent rounding
noise of the same size (its pre-rounding values are fp32, not fp64, so some bf16 roundings
land on the other side; RoPE angles in fp32), so its error is expected within sqrt(2) of
the model's. Measured, the GPU's hidden deviates as the model's does (max 0.044-0.076,
mean 0.0082-0.0101, 95.9-98.6% within the stated tolerance on the seven workloads), so the
end-to-end comparison requires |g - o| <= 0.08 (1 + |o|) (the model's largest 0.056 with
40% margin), a mean error <= 0.0125 (1.25 x the model's largest mean) and >= 95% of the
elements within the stated tolerance.

End-to-end ids: the GPU's logits drift from the oracle's by eps = max_v |z_gpu - z_oracle|
per row (the hidden difference seen through W_lm; 0.056-0.091 measured, up to 0.074 in
the storage model), above the stated delta = 1e-2 max(1, |v|) ~ 0.05 at the top of the
vocabulary. So: the GPU's top-k is checked exactly against the fp64 logits of its own
hidden rows (delta 2e-3); every top-k decision whose oracle margin exceeds 2 eps + 2e-3
must be the oracle's; and the draft ids (top-1) must equal the oracle's wherever the
oracle's margin exceeds the stated delta.

Context caches are seeded random values for the sampled sequences (the same bf16 bits
on both sides) and device-generated values for the others; the step then appends the
previous round's committed rows through ctx_project, drafts, runs the LM head with
top-k (and the selector), and accepts against a seeded target row. The paged workloads
run the same step through the bench's seeded shuffled block table.
"""
import numpy as np
import pytest
import torch

import dflash_inputs as di
from _parity import assert_close, check_topk
from oracle import dflash_oracle as orc

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HIDDEN_ATOL = 0.08
HIDDEN_RTOL = 0.08
HIDDEN_MEAN = 0.0125
STATED_FRACTION = 0.95
# End-to-end logit drift bound: the bf16 storage model's logits of the sampled sequences
# deviate from the exact oracle's by up to 0.053 (Qwen3-4B shape) and 0.074 (Qwen3-8B
# shape) at any vocabulary entry; twice the larger.
LOGIT_DRIFT = 0.15

_W = {}


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def weights_for(w):
    key = (w.D, w.N, w.V, w.F, w.flags & (di.FLAG_CONV | di.FLAG_SELECT | di.FLAG_FILM))
    if key not in _W:
        _W.clear()
        bits = di.make_weights(w)
        _W[key] = (bits, orc.widen_all(bits))
    return _W[key]


def seq_rows(pool, n, i, table):
    """Cache rows [Hkv, Cmax, hd] of sequence i in layer n: a view of the contiguous
    cache, or the sequence's pages gathered through the block table (a copy)."""
    if table is None:
        return pool[n, i]
    pages = pool[n, torch.as_tensor(table[i], dtype=torch.long, device=pool.device)]  # [pps, Hkv, 64, hd]
    return pages.permute(1, 0, 2, 3).reshape(pool.shape[2], -1, pool.shape[4])


def set_seq_rows(pool, n, i, table, rows):
    """Write rows [Hkv, Cmax, hd] of sequence i in layer n (through the table when paged)."""
    if table is None:
        pool[n, i].copy_(rows)
        return
    pr = pool.shape[3]
    for q, pg in enumerate(table[i]):
        pool[n, int(pg)].copy_(rows[:, q * pr:(q + 1) * pr])


def run_case(w, sample):
    from block_diffusion_speculative_project_gb300 import drafter
    bits, W = weights_for(w)
    nb, B, k = w.nb, w.B, w.k_top
    ctx = di.context_lengths(w).astype(np.int32)
    tp = di.tau_prev(w).astype(np.int32)
    relay = bool(w.flags & di.FLAG_RELAY)
    select = bool(w.flags & di.FLAG_SELECT)
    a = None
    if relay:
        a = di.accepted_prev(w).astype(np.int32)
        tp = a + 1
    fb = fy = None
    if w.flags & di.FLAG_FILM:
        fb, fy = di.relay_tokens(w)
    base = ctx - tp
    Cmax = int(ctx.max()) + B
    if w.paged:
        Cmax = -(-Cmax // di.PAGE_ROWS) * di.PAGE_ROWS
    dev = {n: drafter.to_device_bf16(v) for n, v in bits.items()}
    pps = Cmax // di.PAGE_ROWS
    dr = drafter.Drafter(w, dev, nb, Cmax, B, num_pages=nb * pps if w.paged else 0)
    i32 = lambda x: torch.tensor(np.asarray(x, np.int32), device="cuda")
    table = None
    if w.paged:  # the bench's seeded shuffled pages
        table = di.block_table(nb, Cmax, 0)
        dr.set_block_table(i32(table))
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    dr.kcache.normal_(generator=g)
    dr.vcache.normal_(generator=g)
    cache = orc.KVCache(w.N, len(sample), w.Hkv, Cmax, w.hd)
    for si, i in enumerate(sample):
        for n in range(w.N):
            kb = di.normal_bf16(f"kc{i}_{n}", (w.Hkv, Cmax, w.hd), 1.0)
            vb = di.normal_bf16(f"vc{i}_{n}", (w.Hkv, Cmax, w.hd), 1.0)
            set_seq_rows(dr.kcache, n, i, table, drafter.to_device_bf16(kb))
            set_seq_rows(dr.vcache, n, i, table, drafter.to_device_bf16(vb))
            cache.K[n][si][:] = orc.widen(kb)
            cache.V[n][si][:] = orc.widen(vb)
    hv = di.verifier_rows(w, B, name="hv_full")
    ctx_len = i32(base)
    x0 = torch.empty(nb, B, w.D, dtype=torch.bfloat16, device="cuda") if relay else None
    film = {} if fb is None else dict(relay_b=i32(fb), relay_y=i32(fy))
    dr.ctx_project(nb, B, drafter.to_device_bf16(hv), i32(tp), ctx_len,
                   relay_a=i32(a) if relay else None, x0_relay=x0, **film)
    ids = di.block_ids(w, di.anchors(w))
    hid = torch.empty(nb, B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(nb, i32(ids), ctx_len, hid, x0_relay=x0, max_ctx_hint=int(ctx.max()))
    tid = torch.empty(nb, B - 1, k, dtype=torch.int32, device="cuda")
    tv = torch.empty(nb, B - 1, k, dtype=torch.float32, device="cuda")
    dr.lm_head_topk(nb, hid, k, tid, tv)
    assert dr.status() == 0
    assert np.array_equal(ctx_len.cpu().numpy(), ctx), "ctx_len after the append"

    # oracle on the sample
    s = np.array(sample)
    new_len, x0r = orc.ctx_project(w, W, orc.widen(hv[s]), tp[s], base[s], cache,
                                   relay_a=None if a is None else a[s],
                                   relay_b=None if fb is None else fb[s],
                                   relay_y=None if fy is None else fy[s])
    assert np.array_equal(new_len, ctx[s])
    ohid = orc.draft_block(w, W, ids[s], new_len, cache, x0r)
    for si, i in enumerate(sample):
        lo, hi = int(base[i]), int(ctx[i])
        for n in range(w.N):
            gK, gV = seq_rows(dr.kcache, n, i, table), seq_rows(dr.vcache, n, i, table)
            assert_close(gK[:, lo:hi].float().cpu().numpy(), cache.K[n][si][:, lo:hi], f"K_c seq {i}")
            assert_close(gV[:, lo:hi].float().cpu().numpy(), cache.V[n][si][:, lo:hi], f"V_c seq {i}")
        if relay:
            assert_close(x0[i].float().cpu().numpy(), x0r[si], f"x0_relay seq {i}")
        gh = hid[i].float().cpu().numpy().astype(np.float64)
        assert_close(gh, ohid[si], f"hidden seq {i} (derived bf16 bound)", atol=HIDDEN_ATOL, rtol=HIDDEN_RTOL)
        mean_err = np.abs(gh - ohid[si]).mean()
        assert mean_err <= HIDDEN_MEAN, f"hidden seq {i}: mean error {mean_err:.4f}"
        within = (np.abs(gh - ohid[si]) <= 2e-2 + 1e-2 * np.abs(ohid[si])).mean()
        assert within >= STATED_FRACTION, f"hidden seq {i}: only {within:.4f} within the stated tolerance"
        print(f"seq {i}: hidden max err {np.abs(gh - ohid[si]).max():.4f}, mean {mean_err:.5f}, "
              f"{within:.4f} within stated")
    ol = orc.lm_logits(W, ohid)                  # [sample, B-1, V] from the oracle's hidden
    odraft, _ = orc.topk(ol, 1)
    odraft = odraft[..., 0]

    # End to end. The GPU's step carries its own hidden (bf16 storage, fp32 accumulation),
    # bounded against the oracle's exact hidden above, so the two sides' logits differ per
    # row by eps = max_v |z_gpu - z_oracle| (the hidden difference seen through W_lm).
    #  (1) The LM head and top-k on the step's own hidden: the GPU's ids and values against
    #      the fp64 logits of the GPU's hidden rows, margin rule with delta = 2e-3 (same
    #      inputs on both sides, fp32 against fp64 accumulation).
    #  (2) Against the oracle: every top-k decision whose oracle margin exceeds 2 eps + 2e-3
    #      must be the oracle's (a drift of eps cannot reorder it); eps is bounded by
    #      LOGIT_DRIFT. The draft ids (top-1) must equal the oracle's wherever the oracle's
    #      margin exceeds the stated delta = 1e-2 max(1, |v|); with top-1 gaps distributed
    #      as the spacing of the largest of V Gaussian logits (mean ~0.26 here), 70-95% of
    #      the offsets have a margin above delta, and at least 60% is required.
    ns = len(sample)
    s_ids, s_vals = tid[s].cpu().numpy(), tv[s].cpu().numpy()
    gl = orc.lm_logits(W, f64(hid[s]))
    und_self = check_topk(s_ids, s_vals, gl, k, "top-k on the step's own hidden", abs_delta=2e-3)
    eps = np.abs(gl - ol).max(axis=-1)                      # [ns, B-1]
    assert eps.max() <= LOGIT_DRIFT, f"end-to-end logit drift {eps.max():.4f} > {LOGIT_DRIFT}"
    cols = np.arange(w.V)
    und_e2e = 0
    top1_fixed = np.zeros((ns, B - 1), bool)               # top-1 margin above 2 eps + 2e-3
    top1_stated = np.zeros((ns, B - 1), bool)              # top-1 margin above the stated delta
    for si in range(ns):
        for t in range(B - 1):
            order = np.lexsort((cols, -ol[si, t]))[:k + 1]
            v = ol[si, t, order]
            thr = 2 * eps[si, t] + 2e-3
            top1_stated[si, t] = v[0] - v[1] > 1e-2 * max(1.0, abs(v[0]))
            for j in range(k):
                if (j == 0 or v[j - 1] - v[j] > thr) and v[j] - v[j + 1] > thr:
                    assert s_ids[si, t, j] == order[j], (f"end-to-end top-k seq {sample[si]} offset {t + 1} "
                                                         f"pos {j}: {s_ids[si, t, j]} vs {order[j]}")
                    top1_fixed[si, t] |= j == 0
                else:
                    und_e2e += 1
    agree_stated = (s_ids[..., 0] == odraft)[top1_stated].mean() if top1_stated.any() else 1.0
    # the draft itself (top-1): the GPU's id equals the oracle's wherever the oracle's margin
    # exceeds the stated delta (every sampled workload meets this although eps can exceed
    # delta: a top-1 gap is rarely within the drift)
    assert agree_stated == 1.0, f"end-to-end draft ids differ above the stated margin: {agree_stated:.3f}"
    assert top1_stated.mean() >= 0.6, f"only {top1_stated.mean():.3f} of the top-1 margins exceed delta"
    print(f"{w.name}: logit drift eps max {eps.max():.4f} mean {eps.mean():.4f}; top-1 above the stated "
          f"delta {top1_stated.mean():.3f} (GPU equal there {agree_stated:.3f}), above 2 eps "
          f"{top1_fixed.mean():.3f}; top-k positions within the drift {und_e2e}/{ns * (B - 1) * k}; "
          f"own-hidden top-k under 2e-3: {und_self}")

    # LM head at full vocabulary, stage-wise on seeded hidden rows both sides read
    hs_bits = di.normal_bf16(f"hidden_stage_{w.name}", (ns, B, w.D), 1.0)
    sid = torch.empty(ns, B - 1, k, dtype=torch.int32, device="cuda")
    sv = torch.empty(ns, B - 1, k, dtype=torch.float32, device="cuda")
    sl = torch.empty(ns, B - 1, w.V, dtype=torch.float32, device="cuda")
    dr.lm_head_topk(ns, drafter.to_device_bf16(hs_bits), k, sid, sv, sl)
    slog = orc.lm_logits(W, orc.widen(hs_bits))
    err = assert_close(sl.cpu().numpy(), slog, "stage logits")
    assert err < 1e-3, f"stage logits: fp32-accumulated logits drift {err}"
    und = check_topk(sid.cpu().numpy(), sv.cpu().numpy(), slog, k, "stage top-k", abs_delta=2e-3)

    if select:  # the selector stage on seeded candidates, values and hidden rows
        rng = np.random.default_rng(17)
        cand = np.stack([rng.permutation(w.V)[:k] for _ in range(ns * (B - 1))]).reshape(ns, B - 1, k)
        cvals = (rng.standard_normal((ns, B - 1, k)) * 2).astype(np.float32)
        path = torch.empty(ns, B - 1, dtype=torch.int32, device="cuda")
        dr.select(ns, k, i32(cand), torch.tensor(cvals, device="cuda"), drafter.to_device_bf16(hs_bits),
                  i32(ids[s]), path)
        opath, margin = orc.select_path(w, W, cand, cvals.astype(np.float64), orc.widen(hs_bits), ids[s, 0],
                                        return_margins=True)
        gp = path.cpu().numpy()
        for si in range(ns):
            for t in range(B - 1):
                if margin[si, t] <= 1e-2 * max(1.0, float(np.abs(cvals[si, t]).max())):
                    assert gp[si, t] in cand[si, t]
                    break
                assert gp[si, t] == opath[si, t], f"selector seq {sample[si]} offset {t + 1}"

    # accept: the target rows are built from the oracle's draft; the GPU's accept runs on its
    # own draft, so the two compare wherever the GPU drafted the oracle's tokens
    target = di.target_row_from_draft(odraft, w.V)
    gdraft = tid[s][..., 0].contiguous()
    tau = i32(np.zeros(ns))
    bonus = i32(np.zeros(ns))
    dr.accept(ns, gdraft, i32(target), tau, bonus)
    ot, ob = orc.accept(odraft, target)
    # accept reads the draft up to its first mismatch only: compare where the GPU's draft
    # equals the oracle's on that examined prefix
    gd = gdraft.cpu().numpy()
    same = np.array([(gd[j, :min(int(ot[j]), B - 1)] == odraft[j, :min(int(ot[j]), B - 1)]).all()
                     for j in range(ns)])
    # a sequence whose examined prefix is decided at every offset must have drafted the
    # oracle's tokens there (checked above), so it takes part in the comparison
    decided_prefix = np.array([top1_fixed[j, :min(int(ot[j]), B - 1)].all() for j in range(ns)])
    assert same[decided_prefix].all(), f"drafts equal on the examined prefix: {same}, decided {decided_prefix}"
    assert np.array_equal(tau.cpu().numpy()[same], ot[same]) and np.array_equal(bonus.cpu().numpy()[same], ob[same])
    # the accept stage at this shape on the oracle's draft, which both sides read: exact
    tau2 = i32(np.zeros(ns))
    bonus2 = i32(np.zeros(ns))
    dr.accept(ns, i32(odraft), i32(target), tau2, bonus2)
    assert np.array_equal(tau2.cpu().numpy(), ot) and np.array_equal(bonus2.cpu().numpy(), ob)
    print(f"{w.name}: sample {sample}: {und} of {ns * (B - 1) * k} stage top-k positions under the margin; "
          f"{int(same.sum())}/{ns} drafts equal to the oracle's on the examined prefix "
          f"({int(decided_prefix.sum())} decided there)")


def test_fullsize_qwen3_4b_b16_nb1():
    run_case(di.QWEN3_4B, [0])


def test_fullsize_qwen3_8b_b16_nb8():
    run_case(di.QWEN3_8B, [0, 5])


def test_fullsize_qwen3_8b_b8_ragged_nb64():
    ctx = di.context_lengths(di.SWEEP_NB64)
    run_case(di.SWEEP_NB64, [int(np.argmin(ctx)), int(np.argmax(ctx))])


def test_fullsize_paged_qwen3_8b_b16_nb8():
    """The 8-sequence workload with the caches as page pools behind the bench's seeded
    shuffled block table ([DFlash] 四、推理流程, the engineering note on reusing projected K/V)."""
    run_case(di.PAGED_KV, [0, 5])


def test_fullsize_paged_b8_ragged_nb64():
    ctx = di.context_lengths(di.PAGED_KV_NB64)
    run_case(di.PAGED_KV_NB64, [int(np.argmin(ctx)), int(np.argmax(ctx))])


def test_fullsize_relay_dflash2_nb32():
    run_case(di.RELAY_DFLASH2, [3])


def test_fullsize_film_relay_nb32():
    a = di.accepted_prev(di.FILM_RELAY)
    run_case(di.FILM_RELAY, [int(np.argmin(a)), 3])  # the most relayed rows, and sequence 3


@pytest.mark.parametrize("nb,R,paged", [(2, 2048, False), (3, 2048, False), (5, 1500, False), (2, 2048, True)])
def test_fullsize_prefill_qwen3_8b_2048_rows(nb, R, paged):
    """The large-context path: dflash_ctx_project over R prompt rows per sequence at the
    Qwen3-8B shape (M = 4096, 6144 or 7500 rows through the W_c and K/V GEMMs), sequences
    starting at positions 0, 100, 37, 5, 250 and committing R, R - 548, R - 48, R / 2 and
    R - 1 rows. At 4096 rows the K/V GEMM takes the wide 256 x 256 tiles and W_c the
    256 x 128 ones; at 6144 rows both take the wide tiles, and at 7500 rows the last wide
    row tile is ragged. The oracle computes sampled rows one by one (rows are independent):
    h, then K_c / V_c of every layer at those positions, compared at the stated tolerance;
    rows outside the appended range stay untouched. The paged case writes the same rows
    through a shuffled block table of 64-row pages."""
    from block_diffusion_speculative_project_gb300 import drafter
    w = di.QWEN3_8B.with_(nb=nb)
    bits, W = weights_for(w)
    start = np.array([0, 100, 37, 5, 250][:nb], np.int32)
    commit = np.array([R, R - 548, R - 48, R // 2, R - 1][:nb], np.int32)
    Cmax = int((start + commit).max()) + w.B + 8
    Cmax = (Cmax + 63) // 64 * 64
    dev = {n: drafter.to_device_bf16(v) for n, v in bits.items()}
    table = di.block_table(nb, Cmax, 0) if paged else None
    dr = drafter.Drafter(w, dev, w.nb, Cmax, R, num_pages=nb * (Cmax // 64) if paged else 0)
    if paged:
        dr.set_block_table(torch.tensor(table, device="cuda"))
    hv = di.verifier_rows(w, R, name=f"hv_prefill_{R}")
    ctx = torch.tensor(start, device="cuda")
    dr.ctx_project(w.nb, R, drafter.to_device_bf16(hv), torch.tensor(commit, device="cuda"), ctx)
    assert dr.status() == 0
    assert np.array_equal(ctx.cpu().numpy(), start + commit)
    rows = [r for r in (0, 1, 63, 64, 127, 128, 129, 700, 749, 750, 1023, 1024, 1451, 1452, 1499, 1500, 2046, 2047)
            if r < R]
    K, V = dr.kcache, dr.vcache
    for i in range(w.nb):
        sel = [r for r in rows if r < commit[i]]
        h = orc.fuse_context(w, W, orc.widen(hv[i, sel]))
        end = int(start[i] + commit[i])
        for n in range(w.N):
            Kn, Vn = seq_rows(K, n, i, table), seq_rows(V, n, i, table)
            for j, r in enumerate(sel):
                pos = int(start[i]) + r
                k = (W[f"layer{n}.Wk_c"] @ h[j]).reshape(w.Hkv, w.hd)
                v = (W[f"layer{n}.Wv_c"] @ h[j]).reshape(w.Hkv, w.hd)
                ok = orc.rope(k[None], pos, w.rope_base)[0]
                assert_close(Kn[:, pos].float().cpu().numpy(), ok, f"K_c seq {i} row {r} layer {n}")
                assert_close(Vn[:, pos].float().cpu().numpy(), v, f"V_c seq {i} row {r} layer {n}")
            assert not Kn[:, end:].float().abs().sum().item(), "rows past the append"
            assert not Kn[:, :int(start[i])].float().abs().sum().item(), "rows before the append"


def test_fullsize_sampling_launch_shapes_qwen3_8b():
    """The sampling workload's launches at their bench shapes (8 sequences, B = 16,
    V = 151936): the draw over 120 logit rows, the verify of 8 blocks and the DFlash 2
    walk's verify at k = 16, on seeded logits both sides read. Decisions compare exactly
    where the oracle's margin exceeds 1e-3 (fp32 against fp64 scores), otherwise the GPU's
    choice must lie within that margin; the acceptance counts must vary."""
    from block_diffusion_speculative_project_gb300 import drafter
    w = di.SAMPLING_T1
    nb, B, V, k, T, seed = w.nb, w.B, w.V, w.k_top, w.temperature, 0x5EED
    small = di.TINY.with_(V=V, B=B)
    dev = {n: drafter.to_device_bf16(v) for n, v in di.make_weights(small).items()}
    dr = drafter.Drafter(small, dev, nb, 80, 8)
    t32 = lambda x: torch.tensor(np.asarray(x, np.float32), device="cuda")
    i32 = lambda x: torch.tensor(np.asarray(x, np.int32), device="cuda")
    U = di.normal_f32("fs_draft_logits", (nb, B - 1, V), 2.0).astype(np.float64)
    Z = di.target_logits(w).astype(np.float64)
    Z[:, :B - 1] = U + 0.3 * Z[:, :B - 1]           # the target leans toward the draft
    cand = i32(np.zeros((nb, B - 1)))
    lse = t32(np.zeros((nb, B - 1)))
    dr.sample(nb * (B - 1), t32(U), T, seed, cand, lse)
    oc, olse, _, om = orc.sample_candidates(U, T, seed)
    gc = cand.cpu().numpy()
    dec = om > 1e-3
    assert np.array_equal(gc[dec], oc[dec]) and dec.mean() > 0.95
    np.testing.assert_allclose(lse.cpu().numpy(), olse, rtol=1e-5, atol=1e-4)
    tau = i32(np.zeros(nb))
    tok = i32(np.zeros(nb))
    dr.verify_sample(nb, t32(U), t32(olse), i32(oc), t32(Z), T, seed, tau, tok)
    otau, otok, am, em = orc.verify_sample(U, oc, Z, T, seed, return_detail=True)
    gt, gk = tau.cpu().numpy(), tok.cpu().numpy()
    for i in range(nb):
        if (am[i, :min(int(otau[i]), B - 1)] > 1e-3).all():
            assert gt[i] == otau[i], f"seq {i}: tau {gt[i]} vs {otau[i]}"
            if em[i] > 1e-3:
                assert gk[i] == otok[i], f"seq {i}: token {gk[i]} vs {otok[i]}"
    assert len(np.unique(otau)) > 1
    # the DFlash 2 walk's verify at the same shapes
    rng = np.random.default_rng(23)
    cids = np.stack([rng.permutation(V)[:k] for _ in range(nb * (B - 1))]).reshape(nb, B - 1, k).astype(np.int32)
    x = rng.standard_normal((nb, B - 1, k)) * 1.5
    logq = (x - np.log(np.exp(x).sum(-1, keepdims=True))).astype(np.float32).astype(np.float64)
    path = cids[..., 0]
    Zw = Z.copy()
    for i in range(nb):
        for t in range(B - 1):
            Zw[i, t, path[i, t]] += 12.0 if (i + t) % 5 else 0.0  # mostly accepted walked tokens
    dr.verify_sample_walk(nb, k, i32(cids), t32(logq), i32(path), t32(Zw), T, seed, tau, tok)
    wt, wk_, wam, wem = orc.verify_sample_walk(cids, logq, path, Zw.astype(np.float32).astype(np.float64), T, seed,
                                               return_detail=True)
    gt, gk = tau.cpu().numpy(), tok.cpu().numpy()
    for i in range(nb):
        if (wam[i, :min(int(wt[i]), B - 1)] > 1e-3).all():
            assert gt[i] == wt[i], f"walk seq {i}: tau {gt[i]} vs {wt[i]}"
            if wem[i] > 1e-3:
                assert gk[i] == wk_[i], f"walk seq {i}: token {gk[i]} vs {wk_[i]}"
    assert len(np.unique(wt)) > 1
    assert dr.status() == 0
    print(f"sampling launch shapes: draws {dec.sum()}/{dec.size} exact; tau {list(otau)}; walk tau {list(wt)}")


def test_fullsize_attention_repeats_bitwise_qwen3_8b_nb32():
    """The attention stage at the 32-sequence Qwen3-8B shape (C = 4096, B = 16): 65 key
    units per (sequence, kv head) pair over 152 CTAs, 109.5 units each, so some CTAs run
    three segments, the last only a few units long, right after a whole pair. Each half's
    final PV into O must have completed before O is read at a segment's end; a read that
    runs ahead of it gives outputs that change from run to run. Four runs on the same
    inputs must agree bit for bit, and sequences 0 and 4 (which hold such short segments,
    on kv head 5) match the oracle."""
    from block_diffusion_speculative_project_gb300 import drafter
    w = di.QWEN3_8B.with_(name="attn_nb32", N=1, V=4096, L=1, nb=32, B=16)
    nb, B, C = w.nb, w.B, 4096
    Cmax = C + B
    dev = {n: drafter.to_device_bf16(v) for n, v in di.make_weights(w).items()}
    dr = drafter.Drafter(w, dev, nb, Cmax, B)
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    dr.kcache.normal_(generator=g)
    dr.vcache.normal_(generator=g)
    sample = [0, 4]
    kv = {}
    for i in sample:
        kb = di.normal_bf16(f"attn_k{i}", (w.Hkv, Cmax, w.hd), 1.0)
        vb = di.normal_bf16(f"attn_v{i}", (w.Hkv, Cmax, w.hd), 1.0)
        dr.kcache[0, i].copy_(drafter.to_device_bf16(kb))
        dr.vcache[0, i].copy_(drafter.to_device_bf16(vb))
        kv[i] = (orc.widen(kb), orc.widen(vb))
    qb = di.normal_bf16("attn_q_nb32", (nb, B, w.Hq, w.hd), 1.0)
    q = drafter.to_device_bf16(qb)
    ctx = torch.full((nb,), C, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(4):
        o = torch.zeros(nb, B, w.Hq, w.hd, dtype=torch.bfloat16, device="cuda")
        dr.attention(nb, 0, q, ctx, o, max_ctx_hint=C)
        outs.append(o)
    torch.cuda.synchronize()
    assert dr.status() == 0
    ref = outs[0].view(torch.int16)
    for r in range(1, len(outs)):
        diff = (outs[r].view(torch.int16) != ref).any(dim=(1, 3)).nonzero().tolist()
        assert not diff, f"run {r}: (sequence, query head) outputs differ from run 0: {diff[:8]}"
    qw = orc.widen(qb)
    grp = w.Hq // w.Hkv
    for i in sample:
        K, V = kv[i]
        want = np.stack([orc.softmax_attention(qw[i, :, h], K[h // grp], V[h // grp]) for h in range(w.Hq)], 1)
        assert_close(f64(outs[0][i]), want, f"attention nb32 seq {i}")

