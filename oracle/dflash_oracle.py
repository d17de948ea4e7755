"""Oracle for the one-pass block-diffusion draft step (DFlash, DFlow relay, DFlash 2).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` import this module; the product path (the CUDA library and its
binding) never does, and shares no code with it.

What it is: a plain, slow CPU statement of what the draft step computes, written out
per sequence and per head with numpy in float64 (``dtype`` may be set to float32 for
the timed CPU baseline). It consumes the same bf16 values the GPU consumes, widened
exactly, and rounds nothing in between. Library primitives used as steps: matrix
products, exp/sqrt/sin/cos, and ``np.lexsort`` for ordering.

Sources (page title, section):
  [DFlash]  "DFlash 投机解码：块扩散草稿与 KV 注入" (caijizhuo.github.io):
            符号约定 table; 二、块扩散草稿 -- attention equations; 三、KV 注入 -- the H_c
            equation and the W_c size; 四、推理流程 -- draft_forward and dflash_cycle.
  [DFlow]   "DFlow 完全拆解" (pinghaoyang.com.cn/aigc/posts/dflow): 第一步 -- the h_i
            projection; 第二步 -- the one-position shift; 第三步 -- the FiLM relay
            ([beta; gamma] = MLP_phi([E(b); E(y); h_i]), x = E_mask + beta * LN(h_i) + gamma);
            推理循环可以怎么实现 -- relay placement by absolute position; 问题不在拒绝 --
            the accept / bonus split.
  [DFlash2] "DFlash 2：正确 token 已在候选里" (bowenzhou.top/papers/2026/DFlash2):
            洞察一 -- the S_t(a,b) selector score and the greedy walk; 洞察二 -- the
            two-tap dynamic convolution; 洞察一 and Results -- sampling at temperature 1
            with lossless rejection sampling.
  [Philox]  Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
            (SC 2011): the Philox4x32-10 counter-based generator, used for every random
            number the sampling path draws.

Readings where the pages are silent or disagree:
  * block layout [anchor, mask x (B-1)] at absolute positions C..C+B-1, C = context
    rows after the append; offset 0 yields no candidate ([DFlash] 符号约定, dflash_cycle);
  * pre-norm residual layer x += Attn(RMSNorm(x)); x += FFN(RMSNorm(x)); final RMSNorm;
    no QK-norm; RMSNorm eps 1e-6; RoPE rotate-half with theta_d = base^(-2d/hd) on q,
    k_b and k_c at absolute positions; q-head h reads kv-head h // (Hq/Hkv);
  * tau counts the bonus token (1 <= tau <= B); T[j] verifies candidate c_{j+1};
  * relay rows k in [a+2, B-1] of the previous verify go to new offset j = k - a
    (plain add onto the mask embedding); top-k ties and selector ties go to the lower id;
  * FiLM relay: MLP_phi = W2 silu(W1 c) (two bias-free linear layers, hidden width
    film_dim), output split [beta; gamma] in that order; LN without its own gain or bias
    (beta and gamma are the affine), eps as RMSNorm's; conditioning row h_i is the same
    projected row h_k the plain form adds;
  * four convs per layer acting on the residual stream (before/after each sublayer),
    correction linear in the conv input, x_{-1} = 0 at offset 0;
  * selector A = W_A E[a], B = W_B E[b], G = sigmoid(W_G z_t), U_t = raw logit;
  * sampling at temperature T: q_t = softmax(U_t / T) over the whole vocabulary,
    candidates drawn independently per offset (Gumbel-max); verify accepts c_{j+1} when
    u_j < p_j(c_{j+1}) / q_{j+1}(c_{j+1}), p_j = softmax(Z_j / T) of the target row j;
    the first rejection n emits a draw from max(0, p_n - q_{n+1}) (renormalised), or
    from p_n when that is zero everywhere; all accepted emits a draw from p_{B-1};
  * sampling walk (DFlash 2): step t draws among the k candidates of offset t from
    softmax_c(S_t(a_{t-1}, b_c) / T); the walk's draft distribution is that softmax on the
    candidates and 0 elsewhere, and the verify uses it in place of softmax(U_t / T);
  * Recall@k at offset t: the target token is among the k candidates, counted over the
    blocks whose offsets before t all held their target token among theirs;
  * random numbers: Philox4x32-10 keyed by the 64-bit seed, counter (v // 4, row,
    stream, 0), output word v % 4; u = ((x >> 9) + 1/2) / 2^23 (exact in fp32, so both
    sides start from the same u); Gumbel g = -log(-log u).
  * paged cache: the projected K/V of a sequence sit in pages of PAGE_ROWS = 64 rows (one
    attention key unit); a per-sequence block table names the page of each run of 64
    rows, so sequences with a common prefix can point at the same pages.

Parity status: every function here is pinned by tests/test_oracle.py (closed forms,
invariants, brute force on tiny inputs, the pages' worked examples under tests/golden/).
"""
from __future__ import annotations

import math

import numpy as np

from dflash_inputs import bf16_bits_to_f32

FLAG_RELAY = 1
FLAG_CONV = 2
FLAG_SELECT = 4
FLAG_FILM = 8


def widen(bits, dtype=np.float64) -> np.ndarray:
    """bf16 bit patterns -> float array (exact)."""
    return bf16_bits_to_f32(bits).astype(dtype)


def widen_all(bits: dict, dtype=np.float64) -> dict:
    return {k: widen(v, dtype) for k, v in bits.items()}


# ----------------------------------------------------------------------------- pieces

def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: g * x / sqrt(mean(x^2) + eps).

    [DFlash] 三、KV 注入, the H_c equation (RMSNorm after W_c); eps is not given on
    the pages, 1e-6 is used.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return g * x / np.sqrt(ms + eps)


def rope(x: np.ndarray, pos, base: float) -> np.ndarray:
    """Rotary position embedding, rotate-half pairing (d, d + hd/2).

    x: [..., hd] with leading axis matching ``pos`` (scalar or [rows]); any axes in
    between (heads) are broadcast. Angle for pair d at position p: p * base^(-2d/hd).
    """
    hd = x.shape[-1]
    h = hd // 2
    d = np.arange(h, dtype=np.float64)
    inv = np.power(float(base), -2.0 * d / hd)
    p = np.asarray(pos, dtype=np.float64)
    ang = p.reshape(p.shape + (1,) * (x.ndim - 1 - p.ndim) + (1,)) * inv
    c = np.cos(ang).astype(x.dtype)
    s = np.sin(ang).astype(x.dtype)
    x1 = x[..., :h]
    x2 = x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """softmax(q K^T / sqrt(hd)) V with no mask. q [nq, hd], K/V [nk, hd].

    [DFlash] 二、块扩散草稿: Q from the block only, K = [K_c; K_b], V = [V_c; V_b],
    bidirectional inside the block (no causal mask).
    """
    s = (q @ K.T) / math.sqrt(q.shape[-1])
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ V


def silu(x):
    return x / (1.0 + np.exp(-x))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def layer_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """LayerNorm over the last axis, (x - mean) / sqrt(var + eps), population variance.

    [DFlow] 第三步, the LN(h_i) of the relay input. The page gives no LN gain or bias;
    beta and gamma already scale and shift every channel, so none is applied here.
    """
    mu = np.mean(x, axis=-1, keepdims=True)
    var = np.mean((x - mu) ** 2, axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def film_mlp(W: dict, cond: np.ndarray):
    """[beta; gamma] = MLP_phi(cond) = W2 silu(W1 cond), split in that order.

    [DFlow] 第三步: a light MLP of the concatenation [E(b); E(y_{a+1}); h_i]; its depth
    and width are not given on the page: two bias-free linear layers with SiLU between.
    cond: [..., 3D] -> (beta [..., D], gamma [..., D]).
    """
    z = silu(cond @ W["film.W1"].T) @ W["film.W2"].T
    D = z.shape[-1] // 2
    return z[..., :D], z[..., D:]


def film_relay_row(cfg, W: dict, h_i: np.ndarray, b: int, y: int) -> np.ndarray:
    """Relayed row beta * LN(h_i) + gamma ([DFlow] 第三步, the x^{(r+1)}_i equation without
    its E_mask term, which the block input adds).

    b: the verifier's correction token, y: the draft's first rejected guess.
    """
    cond = np.concatenate([W["E"][b], W["E"][y], h_i])
    beta, gamma = film_mlp(W, cond)
    return beta * layer_norm(h_i, cfg.eps) + gamma


def dyn_conv(x: np.ndarray, W0: np.ndarray, W1: np.ndarray, base: np.ndarray,
             group: int = 16) -> np.ndarray:
    """Two-tap dynamic depthwise convolution over one block's rows.

    [DFlash2] 洞察二: x'_t = k_{t,0} * x_t + k_{t,1} * x_{t-1}, each tap k_{t,j} =
    base_j + a correction computed from the current hidden state, one correction value
    shared by every 16 channels. x: [B, D] (block offsets in order); x_{-1} = 0.
    """
    c0 = x @ W0.T                      # [B, D/group]
    c1 = x @ W1.T
    k0 = base[0][None, :] + np.repeat(c0, group, axis=1)
    k1 = base[1][None, :] + np.repeat(c1, group, axis=1)
    prev = np.zeros_like(x)
    prev[1:] = x[:-1]
    return k0 * x + k1 * prev


# ----------------------------------------------------------------------------- cache

class KVCache:
    """Drafter context cache holding projected K_c (RoPE applied) and V_c.

    [DFlash] 四、推理流程, the engineering note: the projected K/V of H_c are what the
    drafter's cache stores, not the raw H_c. Layout per (layer, sequence):
    [Hkv, Cmax, hd]; rows at or beyond the sequence's ctx_len are ignored.
    """

    def __init__(self, N: int, nb: int, Hkv: int, Cmax: int, hd: int, dtype=np.float64):
        self.K = [[np.zeros((Hkv, Cmax, hd), dtype) for _ in range(nb)] for _ in range(N)]
        self.V = [[np.zeros((Hkv, Cmax, hd), dtype) for _ in range(nb)] for _ in range(N)]


PAGE_ROWS = 64


def paged_rows(pool: np.ndarray, table, i: int, n_rows: int, page_rows: int = PAGE_ROWS) -> np.ndarray:
    """Rows 0..n_rows-1 of sequence i, read from a paged pool of one layer.

    [DFlash] 四、推理流程, the engineering note: the drafter's cache holds the projected
    K/V, and requests that share a prefix reuse them through a radix cache. Reading: the
    cache is cut into pages of page_rows rows, pool [P][Hkv][page_rows][hd], and table[i][q]
    names the page that holds rows q*page_rows .. (q+1)*page_rows - 1 of sequence i.
    Returns [Hkv][n_rows][hd].
    """
    out = np.empty((pool.shape[1], n_rows, pool.shape[3]), pool.dtype)
    for r in range(n_rows):
        out[:, r, :] = pool[table[i][r // page_rows], :, r % page_rows, :]
    return out


def cache_from_pages(poolK: np.ndarray, poolV: np.ndarray, table, nb: int, Cmax: int) -> KVCache:
    """The per-sequence cache a paged pool and block table describe. poolK, poolV:
    [N][P][Hkv][PAGE_ROWS][hd]; sequence i of the result is rows 0..Cmax-1 of table row i."""
    N, _, Hkv, _, hd = poolK.shape
    c = KVCache(N, nb, Hkv, Cmax, hd, poolK.dtype)
    for n in range(N):
        for i in range(nb):
            c.K[n][i][:] = paged_rows(poolK[n], table, i, Cmax)
            c.V[n][i][:] = paged_rows(poolV[n], table, i, Cmax)
    return c


# ----------------------------------------------------------------------------- step

def fuse_context(cfg, W: dict, hv_rows: np.ndarray) -> np.ndarray:
    """h = RMSNorm(W_c [H^{l1}; ...; H^{lL}]) per row.

    [DFlash] 三、KV 注入 (H_c equation); [DFlow] 第一步 (the same projection for the
    rejected-suffix rows). hv_rows: [R, L*Dt] with the L layers concatenated.
    """
    return rmsnorm(hv_rows @ W["W_c"].T, W["g_ctx"], cfg.eps)


def ctx_project(cfg, W: dict, hv: np.ndarray, n_commit, ctx_len, cache: KVCache,
                relay_a=None, relay_b=None, relay_y=None):
    """Append committed verifier rows to the context cache; build the relay input.

    hv: [nb, R, L*Dt]. Rows 0..n_commit[i]-1 of sequence i become context rows at
    absolute positions ctx_len[i] + j: K_c = RoPE(Wk_c h), V_c = Wv_c h for every layer.
    With ``relay_a`` (the previous round's accepted count a per sequence), rows
    k in [a+2, B-1] move to new block offset j = k - a ([DFlow] 第二步: the verifier
    row at position p serves draft position p+1; 推理循环: rejected suffix after the
    first rejection), giving x0_relay[i, j] = h_k (plain add form), or with ``relay_b``
    and ``relay_y`` (per sequence: the verifier's correction b, the draft's rejected
    guess y) the FiLM form film_relay_row(h_k, b, y) ([DFlow] 第三步).

    Returns (new_ctx_len [nb], x0_relay [nb, B, D] or None). ``cache`` is updated.
    """
    nb, R, _ = hv.shape
    B, D, Hkv, hd = cfg.B, cfg.D, cfg.Hkv, cfg.hd
    new_len = np.array(ctx_len, dtype=np.int64).copy()
    x0r = None if relay_a is None else np.zeros((nb, B, D), dtype=hv.dtype)
    for i in range(nb):
        h = fuse_context(cfg, W, hv[i])                      # [R, D]
        c0 = int(ctx_len[i])
        nc = int(n_commit[i])
        for j in range(nc):
            pos = c0 + j
            for n in range(cfg.N):
                k = (W[f"layer{n}.Wk_c"] @ h[j]).reshape(Hkv, hd)
                v = (W[f"layer{n}.Wv_c"] @ h[j]).reshape(Hkv, hd)
                cache.K[n][i][:, pos, :] = rope(k[None], pos, cfg.rope_base)[0]
                cache.V[n][i][:, pos, :] = v
        new_len[i] = c0 + nc
        if x0r is not None:
            a = int(relay_a[i])
            for j in range(2, B - a):
                k = j + a
                if k < R:
                    if relay_b is None:
                        x0r[i, j] = h[k]
                    else:
                        x0r[i, j] = film_relay_row(cfg, W, h[k], int(relay_b[i]),
                                                   int(relay_y[i]))
    return new_len, x0r


def block_input(cfg, W: dict, block_ids: np.ndarray, x0_relay=None) -> np.ndarray:
    """x0 = E[block ids] (+ relay rows): [anchor, m_1..m_{B-1}] ([DFlash] 二, the block)."""
    x = W["E"][np.asarray(block_ids)]
    if x0_relay is not None:
        x = x + x0_relay
    return x


def drafter_layer(cfg, W: dict, n: int, x: np.ndarray, Kc: np.ndarray, Vc: np.ndarray,
                  C: int) -> np.ndarray:
    """One drafter layer for one sequence. x: [B, D]; Kc/Vc: [Hkv, >=C, hd].

    [DFlash] 二 attention equations and 四 draft_forward: Q = W_Q H_b from the block only,
    K = [K_c; K_b], V = [V_c; V_b], no mask; SwiGLU FFN. Pre-norm residual form.
    """
    p = f"layer{n}."
    B = x.shape[0]
    Hq, Hkv, hd = cfg.Hq, cfg.Hkv, cfg.hd
    conv = bool(cfg.flags & FLAG_CONV)
    pos = C + np.arange(B)
    if conv:
        x = dyn_conv(x, W[p + "conv0.W0"], W[p + "conv0.W1"], W[p + "conv0.base"], cfg.conv_group)
    u = rmsnorm(x, W[p + "g_attn"], cfg.eps)
    qkv = u @ W[p + "W_qkv"].T
    q = qkv[:, : Hq * hd].reshape(B, Hq, hd)
    kb = qkv[:, Hq * hd: (Hq + Hkv) * hd].reshape(B, Hkv, hd)
    vb = qkv[:, (Hq + Hkv) * hd:].reshape(B, Hkv, hd)
    q = rope(q, pos, cfg.rope_base)
    kb = rope(kb, pos, cfg.rope_base)
    o = np.zeros((B, Hq, hd), dtype=x.dtype)
    grp = Hq // Hkv
    for h in range(Hq):
        g = h // grp
        K = np.concatenate([Kc[g, :C], kb[:, g]], axis=0)
        V = np.concatenate([Vc[g, :C], vb[:, g]], axis=0)
        o[:, h] = softmax_attention(q[:, h], K, V)
    x = x + o.reshape(B, Hq * hd) @ W[p + "W_o"].T
    if conv:
        x = dyn_conv(x, W[p + "conv1.W0"], W[p + "conv1.W1"], W[p + "conv1.base"], cfg.conv_group)
        x = dyn_conv(x, W[p + "conv2.W0"], W[p + "conv2.W1"], W[p + "conv2.base"], cfg.conv_group)
    u = rmsnorm(x, W[p + "g_ffn"], cfg.eps)
    x = x + (silu(u @ W[p + "W_gate"].T) * (u @ W[p + "W_up"].T)) @ W[p + "W_down"].T
    if conv:
        x = dyn_conv(x, W[p + "conv3.W0"], W[p + "conv3.W1"], W[p + "conv3.base"], cfg.conv_group)
    return x


def draft_block(cfg, W: dict, block_ids: np.ndarray, ctx_len, cache: KVCache,
                x0_relay=None, seqs=None) -> np.ndarray:
    """One-pass draft of every block: returns the final-normed hidden [nb, B, D].

    ``seqs`` restricts the computation to a subset of sequences (the others stay zero);
    sequences are independent.
    """
    nb = block_ids.shape[0]
    out = np.zeros((nb, cfg.B, cfg.D), dtype=W["E"].dtype)
    for i in (range(nb) if seqs is None else seqs):
        x = block_input(cfg, W, block_ids[i], None if x0_relay is None else x0_relay[i])
        C = int(ctx_len[i])
        for n in range(cfg.N):
            x = drafter_layer(cfg, W, n, x, cache.K[n][i], cache.V[n][i], C)
        out[i] = rmsnorm(x, W["g_final"], cfg.eps)
    return out


def lm_logits(W: dict, hidden: np.ndarray) -> np.ndarray:
    """Shared LM head on mask offsets 1..B-1: [nb, B-1, V] ([DFlash] dflash_cycle, [1:])."""
    return hidden[:, 1:, :] @ W["W_lm"].T


def topk(values: np.ndarray, k: int):
    """Top-k per row, sorted by value descending, ties to the lower id."""
    rows = values.reshape(-1, values.shape[-1])
    ids = np.zeros((rows.shape[0], k), dtype=np.int32)
    vals = np.zeros((rows.shape[0], k), dtype=values.dtype)
    col = np.arange(rows.shape[1])
    for r in range(rows.shape[0]):
        order = np.lexsort((col, -rows[r]))[:k]
        ids[r] = order
        vals[r] = rows[r, order]
    return ids.reshape(values.shape[:-1] + (k,)), vals.reshape(values.shape[:-1] + (k,))


def accept(draft: np.ndarray, target: np.ndarray):
    """Greedy exact-match accept.

    draft [nb, B-1] = candidates c_1..c_{B-1}; target [nb, B] = the verifier's greedy
    tokens, T[j] predicted from block offset j, so T[j] verifies c_{j+1}. n = number of
    leading matches; tau = n + 1 (accepted plus the bonus token, 1 <= tau <= B);
    bonus = T[n]. ([DFlash] 符号约定 and dflash_cycle step ④; [DFlow] 问题不在拒绝.)
    """
    nb, bm1 = draft.shape
    tau = np.zeros(nb, dtype=np.int32)
    bonus = np.zeros(nb, dtype=np.int32)
    for i in range(nb):
        n = 0
        while n < bm1 and int(draft[i, n]) == int(target[i, n]):
            n += 1
        tau[i] = n + 1
        bonus[i] = target[i, n]
    return tau, bonus


def select_path(cfg, W: dict, cand_ids: np.ndarray, cand_vals: np.ndarray,
                hidden: np.ndarray, anchor: np.ndarray, return_margins: bool = False):
    """DFlash 2 path selector, greedy walk ([DFlash2] 洞察一).

    cand_ids/cand_vals: [nb, B-1, k] top-k candidates and their logits U_t(b) for
    offsets t = 1..B-1; hidden: [nb, B, D] final-normed drafter states z_t.
    S_t(a, b) = U_t(b) + sum_d A(a)_d G_t,d B(b)_d with A(a) = W_A E[a],
    B(b) = W_B E[b], G_t = sigmoid(W_G z_t). Walk: a_0 = anchor,
    a_t = argmax_b S_t(a_{t-1}, b) over the candidates of offset t, ties to the lower id.
    With ``return_margins`` also returns, per step, the best score minus the runner-up.
    """
    nb, bm1, k = cand_ids.shape
    path = np.zeros((nb, bm1), dtype=np.int32)
    margins = np.full((nb, bm1), np.inf)
    for i in range(nb):
        a = int(anchor[i])
        for t in range(1, bm1 + 1):
            G = sigmoid(W["W_G"] @ hidden[i, t])
            Aa = W["W_A"] @ W["E"][a]
            best_b, best_s = None, None
            scores = []
            for c in range(k):
                b = int(cand_ids[i, t - 1, c])
                s = cand_vals[i, t - 1, c] + np.sum(Aa * G * (W["W_B"] @ W["E"][b]))
                scores.append(s)
                if best_s is None or s > best_s or (s == best_s and b < best_b):
                    best_b, best_s = b, s
            path[i, t - 1] = best_b
            if k > 1:
                margins[i, t - 1] = best_s - sorted(scores)[-2]
            a = best_b
    return (path, margins) if return_margins else path


# ----------------------------------------------------------------------------- sampling

PHILOX_M = (0xD2511F53, 0xCD9E8D57)   # [Philox] round multipliers of Philox4x32
PHILOX_W = (0x9E3779B9, 0xBB67AE85)   # [Philox] Weyl key increments
_M32 = np.uint64(0xFFFFFFFF)

STREAM_DRAFT = 0     # candidate draws, row = sequence * (B-1) + offset - 1
STREAM_ACCEPT = 1    # acceptance uniforms, row = sequence, index = step n
STREAM_EMIT = 2      # residual / bonus draw, row = sequence
STREAM_WALK = 3      # selector walk draws, row = sequence * (B-1) + offset - 1, index = slot


def philox4x32(ctr, key, rounds: int = 10):
    """Philox4x32-R of [Philox], vectorised: ctr is four uint arrays (broadcastable),
    key two ints. Each round: (hi, lo) of M0 * c0 and M1 * c2 give
    (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); the key gains (W0, W1) before every round
    after the first. Returns four uint64 arrays holding 32-bit words."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _M32 for c in ctr)
    k0, k1 = np.uint64(key[0] & 0xFFFFFFFF), np.uint64(key[1] & 0xFFFFFFFF)
    m0, m1 = np.uint64(PHILOX_M[0]), np.uint64(PHILOX_M[1])
    for r in range(rounds):
        if r:
            k0 = (k0 + np.uint64(PHILOX_W[0])) & _M32
            k1 = (k1 + np.uint64(PHILOX_W[1])) & _M32
        p0 = m0 * c0            # < 2^64: exact in uint64
        p1 = m1 * c2
        c0, c1, c2, c3 = ((p1 >> np.uint64(32)) ^ c1 ^ k0, p1 & _M32,
                          (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & _M32)
    return c0, c1, c2, c3


def uniforms(seed: int, stream: int, row: int, n: int) -> np.ndarray:
    """u_v in (0, 1) for v = 0..n-1 of (seed, stream, row): word v % 4 of Philox4x32-10
    at counter (v // 4, row, stream, 0), key (seed low, seed high); u = ((w >> 9) + 0.5) / 2^23
    (23 random bits, never 0 or 1, exactly representable in fp32)."""
    v = np.arange(n, dtype=np.uint64)
    words = philox4x32((v >> np.uint64(2), np.uint64(row), np.uint64(stream), np.uint64(0)),
                       (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    w = np.choose((v & np.uint64(3)).astype(np.int64), words)
    return ((w >> np.uint64(9)).astype(np.float64) + 0.5) / float(1 << 23)


def gumbel(u: np.ndarray) -> np.ndarray:
    return -np.log(-np.log(u))


def logsumexp(x: np.ndarray) -> float:
    m = np.max(x)
    return float(m + np.log(np.sum(np.exp(x - m))))


def gumbel_argmax(score: np.ndarray):
    """argmax with ties to the lower id, and the margin to the runner-up."""
    best = int(np.argmax(score))   # first index of the maximum = lowest id
    if score.size < 2:
        return best, np.inf
    top2 = np.partition(score, -2)[-2:]
    return best, float(top2[1] - top2[0])


def sample_candidates(logits: np.ndarray, T: float, seed: int):
    """Draft sampling at temperature T ([DFlash2] 洞察一 / Results: sampling at T = 1).

    logits [nb, B-1, V] = U_t for offsets t = 1..B-1. Each offset draws independently
    from q_t = softmax(U_t / T) by Gumbel-max: c_t = argmax_v U_t(v)/T + g_v with g from
    stream STREAM_DRAFT, row i*(B-1) + t-1. Returns ids [nb, B-1], lse [nb, B-1]
    (logsumexp of U_t / T), logq [nb, B-1] (log q_t(c_t)) and the Gumbel margins."""
    nb, bm1, V = logits.shape
    ids = np.zeros((nb, bm1), np.int32)
    lse = np.zeros((nb, bm1))
    logq = np.zeros((nb, bm1))
    margin = np.zeros((nb, bm1))
    for i in range(nb):
        for t in range(bm1):
            x = logits[i, t] / T
            row = i * bm1 + t
            c, m = gumbel_argmax(x + gumbel(uniforms(seed, STREAM_DRAFT, row, V)))
            ids[i, t], margin[i, t] = c, m
            lse[i, t] = logsumexp(x)
            logq[i, t] = x[c] - lse[i, t]
    return ids, lse, logq, margin


def verify_sample(draft_logits: np.ndarray, cand: np.ndarray, target_logits: np.ndarray,
                  T: float, seed: int, return_detail: bool = False):
    """Lossless rejection sampling of a drafted block ([DFlash2] Results: lossless
    rejection sampling at T = 1; [DFlash] 四、推理流程 dflash_cycle step ④, the rejected
    position is re-drawn from the target and the last step yields the bonus token).

    draft_logits [nb, B-1, V] (offsets 1..B-1), cand [nb, B-1], target_logits [nb, B, V]
    (row j = the target's distribution after block offset j). With p_j = softmax(Z_j/T),
    q_t = softmax(U_t/T): step n accepts c_{n+1} when u_n < p_n(c) / q_{n+1}(c), u_n the
    uniform of stream STREAM_ACCEPT, row i, index n. At the first rejection n the emitted
    token is argmax_v log r(v) + g_v over r = max(0, p_n - q_{n+1}) > 0 (or over log p_n
    when r is zero everywhere); with every candidate accepted it is a draw from p_{B-1};
    g from stream STREAM_EMIT, row i. Returns (tau = n + 1, token) and, with
    ``return_detail``, the per-step acceptance margins |log u - log(p/q)| and the
    emitted draw's Gumbel margin."""
    nb, bm1, V = draft_logits.shape
    tau = np.zeros(nb, np.int32)
    token = np.zeros(nb, np.int32)
    acc_margin = np.full((nb, bm1), np.inf)
    emit_margin = np.zeros(nb)
    for i in range(nb):
        u = uniforms(seed, STREAM_ACCEPT, i, bm1)
        n = 0
        while n < bm1:
            c = int(cand[i, n])
            zp = target_logits[i, n] / T
            zq = draft_logits[i, n] / T
            log_ratio = (zp[c] - logsumexp(zp)) - (zq[c] - logsumexp(zq))
            acc_margin[i, n] = abs(math.log(u[n]) - log_ratio)
            if math.log(u[n]) < log_ratio:
                n += 1
            else:
                break
        g = gumbel(uniforms(seed, STREAM_EMIT, i, V))
        if n < bm1:
            zp = target_logits[i, n] / T
            zq = draft_logits[i, n] / T
            r = np.exp(zp - logsumexp(zp)) - np.exp(zq - logsumexp(zq))
            if (r > 0).any():
                with np.errstate(divide="ignore"):
                    score = np.where(r > 0, np.log(np.where(r > 0, r, 1.0)), -np.inf) + g
            else:
                score = zp + g
        else:
            score = target_logits[i, bm1] / T + g
        token[i], emit_margin[i] = gumbel_argmax(score)
        tau[i] = n + 1
    if return_detail:
        return tau, token, acc_margin, emit_margin
    return tau, token


def selector_scores(cfg, W: dict, cand_ids, cand_vals, hidden, i: int, t: int, a: int):
    """S_t(a, b_c) for the k candidates c of offset t of sequence i ([DFlash2] 洞察一):
    U_t(b) + sum_d A(a)_d G_t,d B(b)_d, A = W_A E[a], B = W_B E[b], G = sigmoid(W_G z_t)."""
    G = sigmoid(W["W_G"] @ hidden[i, t])
    Aa = W["W_A"] @ W["E"][a]
    k = cand_ids.shape[-1]
    return np.array([cand_vals[i, t - 1, c] + np.sum(Aa * G * (W["W_B"] @ W["E"][int(cand_ids[i, t - 1, c])]))
                     for c in range(k)])


def select_walk_sample(cfg, W: dict, cand_ids, cand_vals, hidden, anchor, T: float, seed: int):
    """DFlash 2 sampling walk ([DFlash2] 洞察一: sampling draws from the same score
    distribution the greedy walk maximises). From a_0 = anchor, step t draws slot
    c_t = argmax_c S_t(a_{t-1}, b_c)/T + g_c (Gumbel, stream STREAM_WALK, row
    i*(B-1) + t-1, index c; ties to the lower token id) and a_t = b_{c_t}.
    Returns path [nb, B-1], walk_logq [nb, B-1, k] = log softmax_c(S_t(a_{t-1}, b_c)/T) on
    the walked prefix, and the Gumbel margins."""
    nb, bm1, k = cand_ids.shape
    path = np.zeros((nb, bm1), np.int32)
    logq = np.zeros((nb, bm1, k))
    margin = np.zeros((nb, bm1))
    for i in range(nb):
        a = int(anchor[i])
        for t in range(1, bm1 + 1):
            x = selector_scores(cfg, W, cand_ids, cand_vals, hidden, i, t, a) / T
            sc = x + gumbel(uniforms(seed, STREAM_WALK, i * bm1 + t - 1, k))
            ids = cand_ids[i, t - 1].astype(np.int64)
            order = np.lexsort((ids, -sc))          # best score first, ties to the lower id
            c = int(order[0])
            margin[i, t - 1] = sc[order[0]] - sc[order[1]] if k > 1 else np.inf
            logq[i, t - 1] = x - logsumexp(x)
            path[i, t - 1] = ids[c]
            a = int(ids[c])
    return path, logq, margin


def verify_sample_walk(cand_ids, walk_logq, path, target_logits, T: float, seed: int,
                       return_detail: bool = False):
    """verify_sample with the sampling walk's draft distribution: q_{t}(v) =
    exp(walk_logq[t-1, c]) for v = cand_ids[t-1, c], 0 for every other token. The
    acceptance test, the residual max(0, p - q), the fallback and the bonus draw, their
    streams and ties are those of verify_sample."""
    nb, bm1, k = cand_ids.shape
    V = target_logits.shape[-1]
    tau = np.zeros(nb, np.int32)
    token = np.zeros(nb, np.int32)
    acc_margin = np.full((nb, bm1), np.inf)
    emit_margin = np.zeros(nb)
    for i in range(nb):
        u = uniforms(seed, STREAM_ACCEPT, i, bm1)
        n = 0
        while n < bm1:
            c = int(path[i, n])
            zp = target_logits[i, n] / T
            slot = int(np.nonzero(cand_ids[i, n] == c)[0][0])
            log_ratio = (zp[c] - logsumexp(zp)) - walk_logq[i, n, slot]
            acc_margin[i, n] = abs(math.log(u[n]) - log_ratio)
            if math.log(u[n]) < log_ratio:
                n += 1
            else:
                break
        g = gumbel(uniforms(seed, STREAM_EMIT, i, V))
        if n < bm1:
            zp = target_logits[i, n] / T
            p = np.exp(zp - logsumexp(zp))
            q = np.zeros(V)
            q[cand_ids[i, n].astype(np.int64)] = np.exp(walk_logq[i, n])
            r = p - q
            if (r > 0).any():
                with np.errstate(divide="ignore"):
                    score = np.where(r > 0, np.log(np.where(r > 0, r, 1.0)), -np.inf) + g
            else:
                score = zp + g
        else:
            score = target_logits[i, bm1] / T + g
        token[i], emit_margin[i] = gumbel_argmax(score)
        tau[i] = n + 1
    if return_detail:
        return tau, token, acc_margin, emit_margin
    return tau, token


def recall_at_k(cand_ids, target):
    """Recall@k instrumentation ([DFlash2] Why DFlash 2, the Recall@1 / Recall@16 table):
    at offset t the target token T[t-1] is among the k candidates of offset t, counted over
    the blocks whose offsets 1..t-1 all held their target token. Returns (hits [B-1],
    eligible [B-1]) summed over the nb blocks."""
    nb, bm1, k = cand_ids.shape
    hits = np.zeros(bm1, np.int64)
    eligible = np.zeros(bm1, np.int64)
    for i in range(nb):
        for t in range(bm1):
            eligible[t] += 1
            if int(target[i, t]) in set(int(x) for x in cand_ids[i, t]):
                hits[t] += 1
            else:
                break
    return hits, eligible


def draft_step(cfg, W: dict, hv, n_commit, ctx_len, cache: KVCache, block_ids, target,
               relay_a=None, seqs=None, relay_b=None, relay_y=None):
    """One whole draft step: ctx_project -> draft_block -> LM head + top-k ->
    (selector) -> accept. Returns a dict of every stage's output."""
    new_len, x0r = ctx_project(cfg, W, hv, n_commit, ctx_len, cache, relay_a, relay_b,
                               relay_y)
    hidden = draft_block(cfg, W, block_ids, new_len, cache, x0r, seqs)
    logits = lm_logits(W, hidden)
    ids, vals = topk(logits, cfg.k_top)
    draft = ids[..., 0]
    path = None
    if cfg.flags & FLAG_SELECT:
        path = select_path(cfg, W, ids, vals, hidden, np.asarray(block_ids)[:, 0])
        draft = path
    tau, bonus = accept(draft, target)
    return dict(ctx_len=new_len, x0_relay=x0r, hidden=hidden, logits=logits, ids=ids,
                vals=vals, path=path, draft=draft, tau=tau, bonus=bonus)
