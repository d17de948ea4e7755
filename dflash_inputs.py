"""Seeded synthetic inputs for the one-pass block-diffusion draft step.

This module is shared by the tests, the benchmark and the oracle checks. It holds
no arithmetic of the method: only random draws from named, seeded streams, the
round-to-nearest-even narrowing of those draws to bf16 (the storage format both
sides consume), and the shapes of the named workloads.

Every tensor is drawn from its own stream: the master seed and a CRC32 of the
tensor's name seed a numpy SeedSequence; large tensors are split into fixed
16M-element chunks, each chunk with its own spawned PCG64 stream, so the values
do not depend on how many threads fill them.

Value recipe (the pages give no trained weights; these stand in for them):
  * weights                  ~ N(0, 0.02)
  * RMSNorm gains            ~ 1 + N(0, 0.02)
  * conv base kernel (2, D)  ~ (1, 0) + N(0, 0.02)
  * conv correction W_j      ~ N(0, (0.02 / sqrt(D))^2): the correction is small next
                               to the base kernel, as the DFlash 2 page describes it; at
                               N(0, 0.02) the two-tap conv is quadratic in x and the
                               residual stream diverges within two layers
  * verifier hidden states   ~ N(0, 1)
  * target logits (sampling verify) ~ 2 N(0, 1), fp32
  * anchors                  ~ U{0 .. V-2};  mask id = V-1
  * FiLM relay MLP           W1 ~ N(0, 1/(3D)), W2 ~ N(0, 4/film_dim): fan-in scaled so
                               that beta and gamma come out O(1), the size of the plain
                               relay's h (at N(0, 0.02) they would be ~0.03, below what a
                               bf16 comparison resolves); conditioning tokens ~ U{0 .. V-2}
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

CHUNK = 1 << 24  # elements per independent stream chunk

FLAG_RELAY = 1
FLAG_CONV = 2
FLAG_SELECT = 4
FLAG_FILM = 8


@dataclass(frozen=True)
class Workload:
    """Shape of one named workload (drafter architecture plus batch)."""

    name: str
    D: int
    Dt: int
    L: int
    N: int
    Hq: int
    Hkv: int
    hd: int
    F: int
    V: int
    B: int
    nb: int
    C: int            # context rows attended per sequence (mean when ragged)
    C_lo: int = 0     # ragged contexts: C_i ~ U[C_lo, C_hi]; 0 = all C
    C_hi: int = 0
    flags: int = 0
    k_top: int = 16
    rope_base: float = 1.0e4
    eps: float = 1.0e-6
    sel_dim: int = 256
    conv_group: int = 16
    film_dim: int = 0  # hidden width of the FiLM relay MLP; 0 = D/4
    temperature: float = 0.0  # 0: greedy draft and exact-match accept; > 0: sampling
    paged: bool = False  # caches as pools of 64-row pages behind a block table

    @property
    def film_width(self) -> int:
        return self.film_dim if self.film_dim > 0 else self.D // 4

    @property
    def mask_id(self) -> int:
        return self.V - 1

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload("tiny_d256_n2_b8_c64", D=256, Dt=256, L=5, N=2, Hq=4, Hkv=4, hd=64,
                F=688, V=4096, B=8, nb=1, C=64)
QWEN3_4B = Workload("qwen3_4b_shaped_b16_c2048_nb1", D=2560, Dt=2560, L=5, N=5, Hq=32,
                    Hkv=8, hd=128, F=9728, V=151936, B=16, nb=1, C=2048)
QWEN3_8B = Workload("qwen3_8b_shaped_b16_c4096_nb8", D=4096, Dt=4096, L=5, N=5, Hq=32,
                    Hkv=8, hd=128, F=12288, V=151936, B=16, nb=8, C=4096)
SWEEP_NB16 = QWEN3_8B.with_(name="qwen3_8b_shaped_b8_ragged1024_8192_nb16", B=8, nb=16,
                            C=4608, C_lo=1024, C_hi=8192)
SWEEP_NB32 = SWEEP_NB16.with_(name="qwen3_8b_shaped_b8_ragged1024_8192_nb32", nb=32)
SWEEP_NB64 = SWEEP_NB16.with_(name="qwen3_8b_shaped_b8_ragged1024_8192_nb64", nb=64)
RELAY_DFLASH2 = QWEN3_8B.with_(name="qwen3_8b_shaped_relay_dflash2_b16_c4096_nb32", nb=32,
                               flags=FLAG_RELAY | FLAG_CONV | FLAG_SELECT)
FILM_RELAY = QWEN3_8B.with_(name="qwen3_8b_shaped_film_relay_b16_c4096_nb32", nb=32,
                            flags=FLAG_RELAY | FLAG_FILM)
SAMPLING_T1 = QWEN3_8B.with_(name="qwen3_8b_shaped_sampling_t1_b16_c4096_nb8", temperature=1.0)
DFLASH2_SAMPLING_T1 = QWEN3_8B.with_(name="qwen3_8b_shaped_dflash2_sampling_t1_b16_c4096_nb8",
                                     temperature=1.0, flags=FLAG_CONV | FLAG_SELECT)
PAGED_KV = QWEN3_8B.with_(name="qwen3_8b_shaped_paged_kv_b16_c4096_nb8", paged=True)
PAGED_KV_NB64 = SWEEP_NB64.with_(name="qwen3_8b_shaped_paged_kv_b8_ragged1024_8192_nb64", paged=True)

WORKLOADS = {w.name: w for w in (TINY, QWEN3_4B, QWEN3_8B, SWEEP_NB16, SWEEP_NB32,
                                  SWEEP_NB64, RELAY_DFLASH2, FILM_RELAY, SAMPLING_T1,
                                  DFLASH2_SAMPLING_T1, PAGED_KV, PAGED_KV_NB64)}

PAGE_ROWS = 64


def block_table(nb: int, Cmax: int, seed: int = 0, name: str = "pages") -> np.ndarray:
    """int32 [nb, Cmax / 64]: every sequence's pages, handed out in a seeded random order
    (as a free list that has seen many requests come and go would), no page shared."""
    pps = Cmax // PAGE_ROWS
    g = np.random.Generator(np.random.PCG64(_seedseq(name, seed)))
    return g.permutation(nb * pps).astype(np.int32).reshape(nb, pps)


# --------------------------------------------------------------------------- streams

def _seedseq(name: str, seed: int) -> np.random.SeedSequence:
    return np.random.SeedSequence([seed & 0xFFFFFFFF, zlib.crc32(name.encode())])


def _threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def _fill_normal(name: str, n: int, seed: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK
    children = _seedseq(name, seed).spawn(max(1, nchunks))

    def work(c):
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        g = np.random.Generator(np.random.PCG64(children[c]))
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    if nchunks <= 1:
        if n:
            work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(name: str, shape, std: float, mean: float = 0.0, seed: int = 0) -> np.ndarray:
    """bf16 bits of mean + std * N(0, 1), drawn from the stream `name`."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    x = _fill_normal(name, n, seed)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return f32_to_bf16_bits(x).reshape(shape)


def normal_f32(name: str, shape, std: float = 1.0, seed: int = 0) -> np.ndarray:
    """float32 std * N(0, 1) from the stream `name`, for inputs the path takes in fp32
    (logit rows of the sampling calls)."""
    shape = tuple(int(s) for s in shape)
    x = _fill_normal(name, int(np.prod(shape)) if shape else 1, seed)
    if std != 1.0:
        x *= np.float32(std)
    return x.reshape(shape)


def uniform_int(name: str, shape, lo: int, hi: int, seed: int = 0) -> np.ndarray:
    """int32 draws uniform on [lo, hi] inclusive."""
    g = np.random.Generator(np.random.PCG64(_seedseq(name, seed)))
    return g.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.int32)


# --------------------------------------------------------------------------- weights

def layer_names(n: int):
    p = f"layer{n}."
    return [p + s for s in ("W_qkv", "Wk_c", "Wv_c", "W_o", "W_gate", "W_up", "W_down",
                            "g_attn", "g_ffn")]


def weight_shapes(w: Workload) -> dict:
    """Name -> shape of every weight tensor (row-major, [out, in] for matrices)."""
    s = {
        "W_c": (w.D, w.L * w.Dt),
        "g_ctx": (w.D,),
        "E": (w.V, w.D),
        "W_lm": (w.V, w.D),
        "g_final": (w.D,),
    }
    for n in range(w.N):
        p = f"layer{n}."
        s[p + "W_qkv"] = ((w.Hq + 2 * w.Hkv) * w.hd, w.D)
        s[p + "Wk_c"] = (w.Hkv * w.hd, w.D)
        s[p + "Wv_c"] = (w.Hkv * w.hd, w.D)
        s[p + "W_o"] = (w.D, w.Hq * w.hd)
        s[p + "W_gate"] = (w.F, w.D)
        s[p + "W_up"] = (w.F, w.D)
        s[p + "W_down"] = (w.D, w.F)
        s[p + "g_attn"] = (w.D,)
        s[p + "g_ffn"] = (w.D,)
        if w.flags & FLAG_CONV:
            for c in range(4):
                s[p + f"conv{c}.W0"] = (w.D // w.conv_group, w.D)
                s[p + f"conv{c}.W1"] = (w.D // w.conv_group, w.D)
                s[p + f"conv{c}.base"] = (2, w.D)
    if w.flags & FLAG_FILM:
        s["film.W1"] = (w.film_width, 3 * w.D)
        s["film.W2"] = (2 * w.D, w.film_width)
    if w.flags & FLAG_SELECT:
        s["W_A"] = (w.sel_dim, w.D)
        s["W_B"] = (w.sel_dim, w.D)
        s["W_G"] = (w.sel_dim, w.D)
    return s


def make_weight(name: str, shape, seed: int = 0) -> np.ndarray:
    """bf16 bits of one weight tensor, following the value recipe above."""
    base = name.rsplit(".", 1)[-1]
    if base.startswith("g_"):
        return normal_bf16(name, shape, 0.02, mean=1.0, seed=seed)
    if ".conv" in name and base in ("W0", "W1"):
        return normal_bf16(name, shape, 0.02 / float(np.sqrt(shape[1])), seed=seed)
    if name == "film.W1":
        return normal_bf16(name, shape, 1.0 / float(np.sqrt(shape[1])), seed=seed)
    if name == "film.W2":
        return normal_bf16(name, shape, 2.0 / float(np.sqrt(shape[1])), seed=seed)
    if base == "base":
        x = _fill_normal(name, int(np.prod(shape)), seed).reshape(shape) * np.float32(0.02)
        x[0] += np.float32(1.0)
        return f32_to_bf16_bits(x)
    return normal_bf16(name, shape, 0.02, seed=seed)


def make_weights(w: Workload, seed: int = 0, names=None) -> dict:
    shapes = weight_shapes(w)
    names = list(shapes) if names is None else names
    return {k: make_weight(k, shapes[k], seed) for k in names}


# --------------------------------------------------------------------------- step inputs

def context_lengths(w: Workload, seed: int = 0) -> np.ndarray:
    """C_i per sequence: fixed C, or U[C_lo, C_hi] for the ragged sweep."""
    if w.C_hi > 0:
        return uniform_int("ctx_len", (w.nb,), w.C_lo, w.C_hi, seed)
    return np.full((w.nb,), w.C, dtype=np.int32)


def tau_prev(w: Workload, seed: int = 0) -> np.ndarray:
    """Previous round's accept length per sequence, U{1..B}."""
    return uniform_int("tau_prev", (w.nb,), 1, w.B, seed)


def accepted_prev(w: Workload, seed: int = 0) -> np.ndarray:
    """Previous round's accepted draft count a per sequence, U{0..B-1} (relay workload)."""
    return uniform_int("a_prev", (w.nb,), 0, w.B - 1, seed)


def relay_tokens(w: Workload, seed: int = 0):
    """FiLM relay conditioning tokens per sequence (relay workload): the verifier's
    correction b and the draft's first rejected guess, each U{0..V-2}."""
    return (uniform_int("relay_b", (w.nb,), 0, w.V - 2, seed),
            uniform_int("relay_y", (w.nb,), 0, w.V - 2, seed))


def target_logits(w: Workload, seed: int = 0) -> np.ndarray:
    """Target-model logits of the verify pass [nb, B, V] (fp32), 2 * N(0, 1): the target
    model itself is not part of the draft step, its output row j (the distribution after
    block offset j) is an input of the sampling verify."""
    return normal_f32("target_logits", (w.nb, w.B, w.V), 2.0, seed)


def verifier_rows(w: Workload, rows: int, seed: int = 0, name: str = "hv") -> np.ndarray:
    """Verifier hidden states [nb, rows, L*Dt] (bf16 bits), N(0, 1)."""
    return normal_bf16(name, (w.nb, rows, w.L * w.Dt), 1.0, seed=seed)


def anchors(w: Workload, seed: int = 0) -> np.ndarray:
    return uniform_int("anchor", (w.nb,), 0, w.V - 2, seed)


def block_ids(w: Workload, anchor: np.ndarray) -> np.ndarray:
    """[anchor, mask, ..., mask] per sequence, int32 [nb, B]."""
    ids = np.full((len(anchor), w.B), w.mask_id, dtype=np.int32)
    ids[:, 0] = anchor
    return ids


def target_row_from_draft(draft: np.ndarray, V: int, seed: int = 0,
                          name: str = "target") -> np.ndarray:
    """Synthetic verifier greedy tokens T [nb, B] with a seeded first mismatch.

    draft is [nb, B-1] (candidates c_1..c_{B-1}). The first mismatch index m is
    uniform on {0..B-1}: T[j] = c_{j+1} for j < m; T[m] differs from c_{m+1}
    when m <= B-2; every other entry is a uniform id.
    """
    nb, bm1 = draft.shape
    B = bm1 + 1
    g = np.random.Generator(np.random.PCG64(_seedseq(name, seed)))
    m = g.integers(0, B, size=nb)
    T = g.integers(0, V, size=(nb, B)).astype(np.int32)
    for i in range(nb):
        for j in range(int(m[i])):
            T[i, j] = draft[i, j]
        if m[i] <= B - 2:
            T[i, m[i]] = (int(draft[i, m[i]]) + 1) % V
    return T
