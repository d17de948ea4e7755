"""CPU model of the GPU path's bf16 storage points, used to derive the tolerance of the
full-size end-to-end hidden comparison (tests/test_gpu_fullsize.py).

It builds the same inputs as that test for one sampled sequence and computes the drafter
hidden twice with oracle functions: exactly (the fp64 oracle) and with every value that
the kernel path stores in bf16 rounded to bf16 at that point (h and the appended K_c, V_c
rows of the context projection; with the FiLM relay its MLP hidden and the relay row; per layer the conv inputs of the correction GEMMs, the
normalised GEMM input (u = RMSNorm(x) * g, or without the convs after layer 0's attention
norm bf16(x * g) with the rsqrt(mean x^2 + eps) row factor applied after the GEMM), q,
k_b, v_b, P, o and act; the final hidden). Everything else stays fp64.
It prints the model's deviation from the exact oracle.

    python tests/bf16_storage_model.py WORKLOAD SEQUENCE

It calls only oracle/ and the seeded input generators; nothing here runs on a GPU.
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import dflash_inputs as di  # noqa: E402
from oracle import dflash_oracle as orc  # noqa: E402


def rb(x):
    return orc.widen(di.f32_to_bf16_bits(np.asarray(x, np.float32)))


def model(w, si):
    bits = di.make_weights(w)
    W = orc.widen_all(bits)
    B, Hq, Hkv, hd = w.B, w.Hq, w.Hkv, w.hd
    ctx = di.context_lengths(w).astype(np.int64)
    tp = di.tau_prev(w).astype(np.int64)
    relay, conv = bool(w.flags & di.FLAG_RELAY), bool(w.flags & di.FLAG_CONV)
    a = None
    if relay:
        a = di.accepted_prev(w).astype(np.int64)
        tp = a + 1
    fb = fy = None
    film = bool(w.flags & di.FLAG_FILM)
    if film:
        fb, fy = di.relay_tokens(w)
    base = ctx - tp
    Cmax = int(ctx.max()) + B
    hv = orc.widen(di.verifier_rows(w, B, name="hv_full")[si:si + 1])
    ids = di.block_ids(w, di.anchors(w))[si:si + 1]
    cache = orc.KVCache(w.N, 1, Hkv, Cmax, hd)
    for n in range(w.N):
        cache.K[n][0][:] = orc.widen(di.normal_bf16(f"kc{si}_{n}", (Hkv, Cmax, hd), 1.0))
        cache.V[n][0][:] = orc.widen(di.normal_bf16(f"vc{si}_{n}", (Hkv, Cmax, hd), 1.0))
    Ke = [cache.K[n][0].copy() for n in range(w.N)]
    Ve = [cache.V[n][0].copy() for n in range(w.N)]
    new_len, x0r = orc.ctx_project(w, W, hv, tp[si:si + 1], base[si:si + 1], cache,
                                   relay_a=None if a is None else a[si:si + 1],
                                   relay_b=None if fb is None else fb[si:si + 1],
                                   relay_y=None if fy is None else fy[si:si + 1])
    exact = orc.draft_block(w, W, ids, new_len, cache, x0r)[0]

    # the same step with the kernel path's bf16 storage points
    C0, nc = int(base[si]), int(tp[si])
    C = C0 + nc
    h = rb(orc.rmsnorm(hv[0] @ W["W_c"].T, W["g_ctx"], w.eps))
    for j in range(nc):
        for n in range(w.N):
            k = (W[f"layer{n}.Wk_c"] @ h[j]).reshape(Hkv, hd)
            v = (W[f"layer{n}.Wv_c"] @ h[j]).reshape(Hkv, hd)
            Ke[n][:, C0 + j] = rb(orc.rope(k[None], C0 + j, w.rope_base)[0])
            Ve[n][:, C0 + j] = rb(v)
    x = W["E"][ids[0]].copy()
    if relay:
        aa = int(a[si])
        for j in range(2, B - aa):
            if j + aa < B:
                hk = h[j + aa]
                if film:  # bf16 MLP hidden and relay row; beta, gamma in fp32 (here exact)
                    cond = np.concatenate([W["E"][fb[si]], W["E"][fy[si]], hk])
                    z = rb(orc.silu(cond @ W["film.W1"].T)) @ W["film.W2"].T
                    x[j] = x[j] + rb(z[:w.D] * orc.layer_norm(hk, w.eps) + z[w.D:])
                else:
                    x[j] = x[j] + hk

    def dconv(x, p):
        xb = rb(x)
        k0 = W[p + "base"][0][None, :] + np.repeat(xb @ W[p + "W0"].T, w.conv_group, axis=1)
        k1 = W[p + "base"][1][None, :] + np.repeat(xb @ W[p + "W1"].T, w.conv_group, axis=1)
        prev = np.zeros_like(x)
        prev[1:] = x[:-1]
        return k0 * x + k1 * prev

    def rms(x):
        return 1.0 / np.sqrt((x * x).mean(axis=1, keepdims=True) + w.eps)

    pos = C + np.arange(B)
    grp = Hq // Hkv
    for n in range(w.N):
        p = f"layer{n}."
        if conv:
            x = dconv(x, p + "conv0.")
        if conv or n == 0:
            qkv = rb(orc.rmsnorm(x, W[p + "g_attn"], w.eps)) @ W[p + "W_qkv"].T
        else:  # deferred norm: bf16(x * g) times the row factor after the GEMM
            qkv = (rb(x * W[p + "g_attn"]) @ W[p + "W_qkv"].T) * rms(x)
        q = rb(orc.rope(qkv[:, :Hq * hd].reshape(B, Hq, hd), pos, w.rope_base))
        kb = rb(orc.rope(qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(B, Hkv, hd), pos, w.rope_base))
        vb = rb(qkv[:, (Hq + Hkv) * hd:].reshape(B, Hkv, hd))
        o = np.zeros((B, Hq, hd))
        for hh in range(Hq):
            g = hh // grp
            K = np.concatenate([Ke[n][g, :C], kb[:, g]])
            V = np.concatenate([Ve[n][g, :C], vb[:, g]])
            s = q[:, hh] @ K.T / np.sqrt(hd)
            pe = np.exp(s - s.max(1, keepdims=True))
            o[:, hh] = (rb(pe) @ V) / pe.sum(1, keepdims=True)
        x = x + rb(o.reshape(B, -1)) @ W[p + "W_o"].T
        if conv:
            x = dconv(dconv(x, p + "conv1."), p + "conv2.")
        if conv:
            u = rb(orc.rmsnorm(x, W[p + "g_ffn"], w.eps))
            gate, up = u @ W[p + "W_gate"].T, u @ W[p + "W_up"].T
        else:
            ug, r = rb(x * W[p + "g_ffn"]), rms(x)
            gate, up = (ug @ W[p + "W_gate"].T) * r, (ug @ W[p + "W_up"].T) * r
        x = x + rb(orc.silu(gate) * up) @ W[p + "W_down"].T
        if conv:
            x = dconv(x, p + "conv3.")
    return exact, rb(orc.rmsnorm(x, W["g_final"], w.eps))


if __name__ == "__main__":
    w = di.WORKLOADS[sys.argv[1]]
    si = int(sys.argv[2])
    exact, emu = model(w, si)
    err = np.abs(emu - exact)
    within = (err <= 2e-2 + 1e-2 * np.abs(exact)).mean()
    print(f"{w.name} seq {si}: max {err.max():.4f}  mean {err.mean():.5f}  "
          f"max err/(1+|o|) {(err / (1 + np.abs(exact))).max():.4f}  within stated {within:.4f}")
