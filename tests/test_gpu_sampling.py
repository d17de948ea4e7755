"""GPU parity of sampling at temperature T: dflash_sample (Gumbel-max draft candidates)
and dflash_verify_sample (lossless rejection sampling), through the C ABI, against the
oracle on the same seeded fp32 logits and the same Philox streams.

Decisions that floating point takes (a Gumbel argmax, an acceptance test) are compared
exactly wherever the oracle's margin exceeds DELTA; the kernel computes the scores in fp32
(logits / T, -log(-log u) with u exact in fp32, log p - log q), about 1e-5 from the fp64
values, so DELTA = 1e-3 leaves a wide gap. Below the margin the GPU's choice must still be
one the oracle's scores allow within DELTA. lse and log q are compared at 1e-4 relative.
"""
import numpy as np
import pytest
import torch

import dflash_inputs as di
from oracle import dflash_oracle as orc

pytestmark = pytest.mark.gpu

DELTA = 1e-3


def handle(V, B=16, max_batch=64):
    from block_diffusion_speculative_project_gb300 import drafter
    w = di.TINY.with_(V=V, B=B)
    bits = di.make_weights(w, names=[n for n in di.weight_shapes(w)])
    dev = {k: drafter.to_device_bf16(v) for k, v in bits.items()}
    return drafter.Drafter(w, dev, max_batch, 80, 8)


def t32(a):
    return torch.tensor(np.asarray(a, np.float32), device="cuda")


def i32(a):
    return torch.tensor(np.asarray(a, np.int32), device="cuda")


def logits_rows(name, shape, scale):
    return di.normal_f32(name, shape, scale).astype(np.float64)


def check_draws(gpu_ids, scores_fn, oracle_ids, margins, what):
    """Exact where the oracle's margin exceeds DELTA, else a choice within DELTA."""
    close = 0
    for r in range(len(oracle_ids)):
        if margins[r] > DELTA:
            assert gpu_ids[r] == oracle_ids[r], f"{what} row {r}: {gpu_ids[r]} vs {oracle_ids[r]}"
        else:
            sc = scores_fn(r)
            assert sc[gpu_ids[r]] >= sc.max() - DELTA, f"{what} row {r}: not a near-best choice"
            close += 1
    return close


@pytest.mark.parametrize("V,rows,T,row0", [(151936, 3, 1.0, 0), (5003, 40, 1.0, 0),
                                           (5003, 17, 0.7, 5), (7, 5, 1.0, 0),
                                           (4097, 9, 1.3, 0)])
def test_sample_stage(V, rows, T, row0):
    dr = handle(V)
    U = logits_rows(f"sample_{V}_{rows}", (rows, V), 2.0)
    U[0, :3] = -np.inf  # probability-0 tokens
    seed = 0x1234_5678_9ABC + V
    ids = i32(np.zeros(rows))
    lse = t32(np.zeros(rows))
    logq = t32(np.zeros(rows))
    dr.sample(rows, t32(U), T, seed, ids, lse, logq, row0=row0)
    assert dr.status() == 0
    gi = ids.cpu().numpy()
    # the oracle draws row r of a [1, row0 + rows, V] block; rows before row0 are padding
    pad = np.concatenate([np.zeros((row0, V)), U])[None]
    oi, olse, ologq, om = orc.sample_candidates(pad, T, seed)
    oi, olse, ologq, om = oi[0, row0:], olse[0, row0:], ologq[0, row0:], om[0, row0:]
    np.testing.assert_allclose(lse.cpu().numpy(), olse, rtol=1e-4, atol=1e-4)

    def scores(r):
        return U[r] / T + orc.gumbel(orc.uniforms(seed, orc.STREAM_DRAFT, row0 + r, V))

    close = check_draws(gi, scores, oi, om, "draw")
    same = gi == oi
    np.testing.assert_allclose(logq.cpu().numpy()[same], ologq[same], rtol=1e-4, atol=1e-4)
    assert not np.isin(gi[:1], [0, 1, 2]).any(), "a probability-0 token was drawn"
    print(f"V={V} rows={rows}: {close} draws under the margin")


def verify_case(nb, B, V, seed, noise=0.3):
    """Draft logits, target logits close to them (so acceptance runs vary), the oracle's
    candidates and draft lse."""
    U = logits_rows(f"vU_{nb}_{V}", (nb, B - 1, V), 2.0)
    Z = logits_rows(f"vZ_{nb}_{V}", (nb, B, V), 2.0)
    Z[:, :B - 1] = U + noise * Z[:, :B - 1]
    cand, lse, _, _ = orc.sample_candidates(U, 1.0, seed)
    return U, Z, cand, lse


def run_verify(dr, U, Z, cand, lse, T, seed):
    nb = U.shape[0]
    tau = i32(np.zeros(nb))
    tok = i32(np.zeros(nb))
    dr.verify_sample(nb, t32(U), t32(lse), i32(cand), t32(Z), T, seed, tau, tok)
    assert dr.status() == 0
    return tau.cpu().numpy(), tok.cpu().numpy()


def compare_verify(U, Z, cand, T, seed, gtau, gtok):
    otau, otok, am, em = orc.verify_sample(U, cand, Z, T, seed, return_detail=True)
    exact = 0
    for i in range(len(otau)):
        n = otau[i] - 1
        decided = am[i, :min(n + 1, U.shape[1])]
        if (decided > DELTA).all():
            assert gtau[i] == otau[i], f"seq {i}: tau {gtau[i]} vs {otau[i]}"
            if em[i] > DELTA:
                assert gtok[i] == otok[i], f"seq {i}: token {gtok[i]} vs {otok[i]}"
                exact += 1
    return exact, otau


def test_verify_stage_many_sequences():
    nb, B, V, seed = 64, 16, 5003, 77
    dr = handle(V, B)
    U, Z, cand, lse = verify_case(nb, B, V, seed)
    gtau, gtok = run_verify(dr, U, Z, cand, lse, 1.0, seed)
    exact, otau = compare_verify(U, Z, cand, 1.0, seed, gtau, gtok)
    assert exact >= 0.9 * nb, f"only {exact} of {nb} sequences decided above the margin"
    assert len(np.unique(otau)) >= 4, "acceptance lengths should vary in this case"
    print(f"tau histogram {np.bincount(otau, minlength=B + 1)}; {exact}/{nb} compared exactly")


def test_verify_stage_full_vocabulary_and_temperature():
    nb, B, V, seed = 4, 8, 151936, 78
    dr = handle(V, B)
    U, Z, cand, _ = verify_case(nb, B, V, seed, noise=0.1)
    T = 0.8
    cand, lse, _, _ = orc.sample_candidates(U, T, seed)
    gtau, gtok = run_verify(dr, U, Z, cand, lse, T, seed)
    exact, _ = compare_verify(U, Z, cand, T, seed, gtau, gtok)
    assert exact >= nb - 1


def test_verify_accept_all_and_zero_probability_reject():
    nb, B, V, seed = 6, 8, 999, 79
    dr = handle(V, B)
    U, Z, cand, lse = verify_case(nb, B, V, seed)
    Z[:, :B - 1] = U            # p_j = q_{j+1}: every candidate accepted, tau = B
    gtau, gtok = run_verify(dr, U, Z, cand, lse, 1.0, seed)
    assert (gtau == B).all()
    otau, otok = orc.verify_sample(U, cand, Z, 1.0, seed)
    assert np.array_equal(gtok, otok)  # the bonus draw from p_{B-1}
    for i in range(nb):
        Z[i, 3, cand[i, 3]] = -np.inf  # the target gives c_4 probability 0
    gtau, gtok = run_verify(dr, U, Z, cand, lse, 1.0, seed)
    assert (gtau == 4).all()
    assert (gtok != cand[:, 3]).all()
    otau, otok, _, em = orc.verify_sample(U, cand, Z, 1.0, seed, return_detail=True)
    assert np.array_equal(gtau, otau)
    assert np.array_equal(gtok[em > DELTA], otok[em > DELTA])


def test_verify_rejects_out_of_vocabulary_candidate():
    nb, B, V, seed = 2, 4, 300, 80
    dr = handle(V, B)
    U, Z, cand, lse = verify_case(nb, B, V, seed)
    Z[:, :B - 1] = U
    cand = cand.copy()
    cand[0, 1] = V + 5
    cand[1, 0] = -1
    gtau, _ = run_verify(dr, U, Z, cand, lse, 1.0, seed)
    assert list(gtau) == [2, 1]


def test_sampling_argument_errors():
    from block_diffusion_speculative_project_gb300 import dflash
    dr = handle(64, 4, max_batch=2)
    x = t32(np.zeros((2, 64)))
    out = i32(np.zeros(2))
    with pytest.raises(dflash.DflashError) as e:
        dr.sample(2, x, 0.0, 1, out, t32(np.zeros(2)))
    assert e.value.code == dflash.DFLASH_ERR_INVALID_ARG
    with pytest.raises(dflash.DflashError) as e:
        dr.sample(2 * 4 + 1, x, 1.0, 1, out, t32(np.zeros(2)))
    assert e.value.code == dflash.DFLASH_ERR_INVALID_ARG


def test_sampling_full_step_medium():
    """ctx_project -> draft_block -> LM head logits -> draw -> verify against seeded target
    logits, end to end against the oracle's step. The GPU's logits differ from the oracle's
    by the bf16 path error (within 2e-2 + 1e-2|o|, checked in test_full_step), so the
    decisions compare exactly where the oracle's margin exceeds DELTA_E2E = 0.1."""
    from block_diffusion_speculative_project_gb300 import drafter
    DELTA_E2E = 0.1
    w = di.Workload("medium_sampling", D=512, Dt=192, L=5, N=2, Hq=8, Hkv=2, hd=128, F=1000,
                    V=5003, B=16, nb=6, C=300, temperature=1.0)
    bits = di.make_weights(w)
    W = orc.widen_all(bits)
    dev = {k: drafter.to_device_bf16(v) for k, v in bits.items()}
    Cmax, C = 96, 70
    dr = drafter.Drafter(w, dev, w.nb, Cmax, C)
    nb, B, V, T, seed = w.nb, w.B, w.V, w.temperature, 4242
    hv_pre = di.verifier_rows(w, C, name="hv_prefill")
    tp = np.minimum(di.tau_prev(w), B).astype(np.int32)
    ctx = i32(np.zeros(nb))
    dr.ctx_project(nb, C, drafter.to_device_bf16(hv_pre), i32(C - tp), ctx)
    cache = orc.KVCache(w.N, nb, w.Hkv, Cmax, w.hd)
    lens, _ = orc.ctx_project(w, W, orc.widen(hv_pre), C - tp, np.zeros(nb), cache)
    hv = di.verifier_rows(w, B, name="hv_step")
    dr.ctx_project(nb, B, drafter.to_device_bf16(hv), i32(tp), ctx)
    ids = di.block_ids(w, di.anchors(w))
    out = torch.empty(nb, B, w.D, dtype=torch.bfloat16, device="cuda")
    dr.draft_block(nb, i32(ids), ctx, out, max_ctx_hint=C)
    k = w.k_top
    logits = torch.empty(nb, B - 1, V, dtype=torch.float32, device="cuda")
    dr.lm_head_topk(nb, out, k, i32(np.zeros((nb, B - 1, k))), t32(np.zeros((nb, B - 1, k))), logits)
    cand = i32(np.zeros((nb, B - 1)))
    lse = t32(np.zeros((nb, B - 1)))
    dr.sample(nb * (B - 1), logits, T, seed, cand, lse)
    Zb = di.target_logits(w).astype(np.float64)
    tau = i32(np.zeros(nb))
    tok = i32(np.zeros(nb))
    dr.verify_sample(nb, logits, lse, cand, t32(Zb), T, seed, tau, tok)
    assert dr.status() == 0

    o = orc.draft_step(w, W, orc.widen(hv), tp, lens, cache, ids, np.zeros((nb, B), np.int32))
    oc, _, _, om = orc.sample_candidates(o["logits"], T, seed)
    gc = cand.cpu().numpy()
    decided = om > DELTA_E2E
    assert np.array_equal(gc[decided], oc[decided]), "draws above the end-to-end margin"
    assert decided.mean() > 0.8, f"only {decided.mean():.2f} of the draws above the margin"
    otau, otok, am, em = orc.verify_sample(o["logits"], oc, Zb, T, seed, return_detail=True)
    gt, gk = tau.cpu().numpy(), tok.cpu().numpy()
    compared = 0
    for i in range(nb):
        n = otau[i] - 1
        steps = range(min(n + 1, B - 1))
        if all(decided[i, j] and am[i, j] > DELTA_E2E for j in steps):
            assert gt[i] == otau[i], f"seq {i}: tau {gt[i]} vs {otau[i]}"
            if em[i] > DELTA_E2E:
                assert gk[i] == otok[i], f"seq {i}: token {gk[i]} vs {otok[i]}"
            compared += 1
    assert compared >= nb // 2
    print(f"end-to-end sampling: {decided.sum()}/{decided.size} draws and {compared}/{nb} "
          f"verifies compared exactly; tau {list(gt)}")


def test_philox_uniforms_bit_exact_and_gumbel_error():
    """The kernels' random numbers against the oracle's Philox4x32-10: uniforms bit-exact
    (both are ((w >> 9) + 1/2) / 2^23, exact in fp32) over 4M elements of three streams,
    Gumbel values within 5e-6 of the fp64 -log(-log u)."""
    from block_diffusion_speculative_project_gb300 import dflash
    n = 1 << 22
    for seed, stream, row in ((0x0123_4567_89AB_CDEF, 0, 3), (7, 1, 0), (2 ** 63 + 5, 2, 65535)):
        u = torch.empty(n, dtype=torch.float32, device="cuda")
        g = torch.empty(n, dtype=torch.float32, device="cuda")
        dflash.dflash_draw_gumbel(n, seed, stream, row, u, g)
        torch.cuda.synchronize()
        ou = orc.uniforms(seed, stream, row, n)
        assert np.array_equal(u.cpu().numpy().astype(np.float64), ou), f"uniforms stream {stream}"
        err = np.abs(g.cpu().numpy().astype(np.float64) - orc.gumbel(ou))
        assert err.max() < 5e-6, f"Gumbel error {err.max():.2e} stream {stream}"
        print(f"stream {stream}: Gumbel max abs error {err.max():.2e}")


@pytest.mark.parametrize("V,nb,B,T", [(151936, 2, 16, 1.0), (5003, 9, 16, 0.6), (4097, 5, 8, 1.0)])
def test_lm_head_fused_draw(V, nb, B, T):
    """dflash_lm_head_sample on seeded bf16 hidden rows against the oracle's LM head and
    draw: the fp32-accumulated logits are within 1e-3 of the fp64 ones, so the draws
    compare exactly where the oracle's margin exceeds 2e-3; lse within 1e-3."""
    from block_diffusion_speculative_project_gb300 import drafter
    w = di.TINY.with_(V=V, B=B, nb=nb)
    bits = di.make_weights(w)
    dev = {k: drafter.to_device_bf16(v) for k, v in bits.items()}
    dr = drafter.Drafter(w, dev, nb, 80, 8)
    hid = di.normal_bf16(f"hid_draw_{V}", (nb, B, w.D), 1.0)
    seed = 99 + V
    cand = i32(np.zeros((nb, B - 1)))
    lse = t32(np.zeros((nb, B - 1)))
    logq = t32(np.zeros((nb, B - 1)))
    logits = torch.empty(nb, B - 1, V, dtype=torch.float32, device="cuda")
    ids = i32(np.zeros((nb, B - 1, w.k_top)))
    vals = t32(np.zeros((nb, B - 1, w.k_top)))
    dr.lm_head_sample(nb, drafter.to_device_bf16(hid), T, seed, cand, lse, logq, logits, w.k_top, ids, vals)
    assert dr.status() == 0
    W = orc.widen_all({"W_lm": bits["W_lm"]})
    ol = orc.lm_logits(W, orc.widen(hid))
    assert np.abs(logits.cpu().numpy() - ol).max() < 1e-3
    oc, olse, ologq, om = orc.sample_candidates(ol, T, seed)
    gc = cand.cpu().numpy()
    dec = om > 2e-3
    assert np.array_equal(gc[dec], oc[dec])
    assert dec.mean() > 0.9
    np.testing.assert_allclose(lse.cpu().numpy(), olse, atol=1e-3, rtol=1e-5)
    same = gc == oc
    np.testing.assert_allclose(logq.cpu().numpy()[same], ologq[same], atol=2e-3)
    # the top-k of the same launch is unchanged by the draw
    oi, _ = orc.topk(ol, w.k_top)
    assert (ids.cpu().numpy()[..., 0] == oi[..., 0]).mean() > 0.95
    # the draw from the written logits (dflash_sample) is the same draw
    c2 = i32(np.zeros((nb, B - 1)))
    l2 = t32(np.zeros((nb, B - 1)))
    dr.sample(nb * (B - 1), logits, T, seed, c2, l2)
    assert np.array_equal(c2.cpu().numpy(), gc)
    np.testing.assert_allclose(l2.cpu().numpy(), lse.cpu().numpy(), rtol=1e-5, atol=1e-5)


# ----------------------------------------------------------------------------- DFlash 2 sampling walk

SEL = di.Workload("medium_select_walk", D=512, Dt=192, L=5, N=1, Hq=8, Hkv=2, hd=128, F=1000,
                  V=5003, B=16, nb=6, C=300, flags=di.FLAG_SELECT)


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_select_walk_sample_stage(T):
    """dflash2_select_sample against the oracle's walk on the same candidates, values and
    hidden rows. The scores come from bf16 GEMMs (within 1e-2 (1 + |U|) of fp64), so the
    walks agree step by step while the oracle's Gumbel margin exceeds that; after the first
    step under it the prefixes may part and the rest of that sequence is not compared."""
    from block_diffusion_speculative_project_gb300 import drafter
    w = SEL
    bits = di.make_weights(w)
    W = orc.widen_all(bits)
    dev = {k: drafter.to_device_bf16(v) for k, v in bits.items()}
    dr = drafter.Drafter(w, dev, w.nb, 64, w.B)
    rng = np.random.default_rng(61)
    k = w.k_top
    cand = np.stack([rng.permutation(w.V)[:k] for _ in range(w.nb * (w.B - 1))]).reshape(w.nb, w.B - 1, k)
    vals = (rng.standard_normal((w.nb, w.B - 1, k)) * 2).astype(np.float32)
    hid_bits = di.normal_bf16("walk_hidden", (w.nb, w.B, w.D), 1.0)
    ids = di.block_ids(w, di.anchors(w))
    seed = 2024
    path = i32(np.zeros((w.nb, w.B - 1)))
    logq = t32(np.zeros((w.nb, w.B - 1, k)))
    dr.select_sample(w.nb, k, i32(cand), torch.tensor(vals, device="cuda"), drafter.to_device_bf16(hid_bits),
                     i32(ids), T, seed, path, logq)
    assert dr.status() == 0
    opath, ologq, margin = orc.select_walk_sample(w, W, cand, vals.astype(np.float64), orc.widen(hid_bits),
                                                  ids[:, 0], T, seed)
    gp, gl = path.cpu().numpy(), logq.cpu().numpy()
    decided = 0
    for i in range(w.nb):
        for t in range(w.B - 1):
            err = np.abs(gl[i, t] - ologq[i, t])
            assert (err <= 2e-2 / T + 1e-2 * np.abs(ologq[i, t])).all(), (
                f"log q seq {i} offset {t + 1}: max err {err.max():.3e}; gpu {gl[i, t][:4]} oracle {ologq[i, t][:4]}")
            if margin[i, t] <= 1e-2 * max(1.0, abs(vals[i, t]).max()) / T:
                assert gp[i, t] in cand[i, t]
                break
            assert gp[i, t] == opath[i, t], f"seq {i} offset {t + 1}"
            decided += 1
    assert decided >= w.nb * (w.B - 1) // 2
    print(f"T={T}: {decided}/{w.nb * (w.B - 1)} walk steps compared exactly")


def test_verify_sample_walk_stage():
    """dflash_verify_sample_walk on the oracle's walk (candidates, log q, path) and seeded
    target logits that favour the walked tokens, against the oracle's sparse verify."""
    nb, B, V, k, seed = 48, 16, 5003, 16, 81
    dr = handle(V, B)
    rng = np.random.default_rng(82)
    cand = np.stack([rng.permutation(V)[:k] for _ in range(nb * (B - 1))]).reshape(nb, B - 1, k).astype(np.int32)
    x = rng.standard_normal((nb, B - 1, k)) * 1.5
    logq = x - np.log(np.exp(x).sum(-1, keepdims=True))
    slot = np.array([[orc.gumbel_argmax(logq[i, t] + orc.gumbel(orc.uniforms(seed, 3, i * (B - 1) + t, k)))[0]
                      for t in range(B - 1)] for i in range(nb)])
    path = np.take_along_axis(cand, slot[..., None], -1)[..., 0]
    Z = logits_rows("walkZ", (nb, B, V), 1.0)
    for i in range(nb):
        for t in range(B - 1):
            Z[i, t, cand[i, t]] += 4.0 + x[i, t]      # the target leans toward the candidates
    lq32 = logq.astype(np.float32).astype(np.float64)
    tau = i32(np.zeros(nb))
    tok = i32(np.zeros(nb))
    dr.verify_sample_walk(nb, k, i32(cand), t32(lq32), i32(path), t32(Z), 1.0, seed, tau, tok)
    assert dr.status() == 0
    otau, otok, am, em = orc.verify_sample_walk(cand, lq32, path, Z.astype(np.float32).astype(np.float64),
                                                1.0, seed, return_detail=True)
    gt, gk = tau.cpu().numpy(), tok.cpu().numpy()
    exact = 0
    for i in range(nb):
        n = otau[i] - 1
        if (am[i, :min(n + 1, B - 1)] > DELTA).all():
            assert gt[i] == otau[i], f"seq {i}: tau {gt[i]} vs {otau[i]}"
            if em[i] > DELTA:
                assert gk[i] == otok[i], f"seq {i}: token {gk[i]} vs {otok[i]}"
                exact += 1
    assert exact >= 0.9 * nb
    assert len(np.unique(otau)) >= 4
    print(f"walk verify: tau histogram {np.bincount(otau, minlength=B + 1)}; {exact}/{nb} exact")


def test_recall_at_k_counts():
    nb, B, V, k = 40, 8, 999, 4
    dr = handle(V, B)
    rng = np.random.default_rng(83)
    cand = np.stack([rng.permutation(V)[:k] for _ in range(nb * (B - 1))]).reshape(nb, B - 1, k).astype(np.int32)
    target = rng.integers(0, V, (nb, B)).astype(np.int32)
    hit = rng.random((nb, B - 1)) < 0.8                      # plant hits at 80% of the offsets
    for i in range(nb):
        for t in range(B - 1):
            if hit[i, t]:
                target[i, t] = cand[i, t, rng.integers(0, k)]
    hits = i32(np.zeros(B - 1))
    elig = i32(np.zeros(B - 1))
    dr.recall_at_k(nb, k, i32(cand), i32(target), hits, elig)
    dr.recall_at_k(nb, k, i32(cand), i32(target), hits, elig)  # counts accumulate
    oh, oe = orc.recall_at_k(cand, target)
    assert np.array_equal(hits.cpu().numpy(), 2 * oh) and np.array_equal(elig.cpu().numpy(), 2 * oe)
    assert oe[0] == nb and oh[-1] > 0
