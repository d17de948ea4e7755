"""Python binding of libdflash (include/dflash.h): argument marshalling only.

Every function here has the name of the C entry point it calls and forwards torch
tensors as raw device pointers (``tensor.data_ptr()``) with the current CUDA stream.
No step of the draft computation runs in Python. If the shared library is missing
the import of this module raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdflash.so")

DFLASH_OK = 0
DFLASH_ERR_INVALID_ARG = -1
DFLASH_ERR_UNSUPPORTED_SHAPE = -2
DFLASH_ERR_CUDA = -3
DFLASH_ERR_TIMEOUT = -4
DFLASH_ERR_DEVICE_CHECK = -5

FLAG_RELAY = 1
FLAG_CONV = 2
FLAG_SELECT = 4
FLAG_FILM = 8
FLAG_TEST_STALL = 1 << 30


class DflashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dflash error {code}: {msg}")
        self.code = code


class dflash_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("D", "Dt", "L", "N", "Hq", "Hkv", "hd", "F", "V", "B",
                                            "k_top")] + [
        ("rope_base", ctypes.c_float), ("eps", ctypes.c_float)] + [
        (n, ctypes.c_int) for n in ("mask_id", "Cmax", "max_batch", "max_proj_rows", "conv_group",
                                    "sel_dim")] + [
        ("flags", ctypes.c_uint), ("max_spin", ctypes.c_int), ("film_dim", ctypes.c_int),
        ("num_pages", ctypes.c_int)]


DFLASH_PAGE_ROWS = 64


_P = ctypes.c_void_p


class dflash_layer_weights(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("W_qkv", "Wk_c", "Wv_c", "W_o", "W_gate", "W_up", "W_down",
                                  "g_attn", "g_ffn")] + [
        ("conv_W0", _P * 4), ("conv_W1", _P * 4), ("conv_base", _P * 4)]


class dflash_weights(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("W_c", "g_ctx", "E", "W_lm", "g_final", "W_A", "W_B", "W_G")] + [
        ("layers", ctypes.POINTER(dflash_layer_weights)), ("film_W1", _P), ("film_W2", _P)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m block_diffusion_speculative_project_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    i, p, sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    sig = {
        "dflash_create": (i, [ctypes.POINTER(dflash_config), ctypes.POINTER(p)]),
        "dflash_destroy": (i, [p]),
        "dflash_set_weights": (i, [p, ctypes.POINTER(dflash_weights)]),
        "dflash_set_block_table": (i, [p, p]),
        "dflash_workspace_size": (i, [p, ctypes.POINTER(sz)]),
        "dflash_status": (i, [p, p, p, ctypes.POINTER(i)]),
        "dflash_last_error": (ctypes.c_char_p, []),
        "dflash_ctx_project": (i, [p, i, i, p, p, p, p, p, p, p, p, sz, p]),
        "dflash_ctx_project_film": (i, [p, i, i, p, p, p, p, p, p, p, p, p, p, sz, p]),
        "dflash_draft_block": (i, [p, i, p, p, p, p, p, i, p, p, sz, p]),
        "dflash_lm_head_topk": (i, [p, i, p, i, p, p, p, p, sz, p]),
        "dflash_lm_head_topk_noalloc": (i, [p, i, p, i, p, p, p, p]),
        "dflash_attention": (i, [p, i, i, p, p, p, p, i, p, p, sz, p]),
        "dflash_topk": (i, [p, i, i, p, i, p, p, p, sz, p]),
        "dflash_accept": (i, [p, i, p, p, p, p, p]),
        "dflash_accept_topk": (i, [p, i, p, i, p, p, p, p]),
        "dflash_sample": (i, [p, i, p, ctypes.c_float, ctypes.c_uint64, i, p, p, p, p, sz, p]),
        "dflash_lm_head_sample": (i, [p, i, p, ctypes.c_float, ctypes.c_uint64, p, p, p, p, i, p, p, p,
                                      sz, p]),
        "dflash_draw_gumbel": (i, [i, ctypes.c_uint64, i, i, p, p, p]),
        "dflash_verify_sample": (i, [p, i, p, p, p, p, ctypes.c_float, ctypes.c_uint64, p, p, p, sz,
                                     p]),
        "dflash2_conv": (i, [p, i, i, i, p, p, sz, p]),
        "dflash2_select": (i, [p, i, i, p, p, p, p, p, p, sz, p]),
        "dflash2_select_sample": (i, [p, i, i, p, p, p, p, ctypes.c_float, ctypes.c_uint64, p, p, p, sz,
                                      p]),
        "dflash_verify_sample_walk": (i, [p, i, i, p, p, p, p, ctypes.c_float, ctypes.c_uint64, p, p, p,
                                          sz, p]),
        "dflash_recall_at_k": (i, [p, i, i, p, p, p, p, p]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


LIB = _load()
EXPORTED = ("dflash_create", "dflash_destroy", "dflash_set_weights", "dflash_set_block_table",
            "dflash_workspace_size",
            "dflash_status", "dflash_last_error", "dflash_ctx_project", "dflash_ctx_project_film",
            "dflash_draft_block",
            "dflash_lm_head_topk", "dflash_lm_head_topk_noalloc", "dflash_attention", "dflash_topk", "dflash_accept", "dflash_accept_topk", "dflash_sample", "dflash_verify_sample",
            "dflash_lm_head_sample", "dflash_draw_gumbel", "dflash2_select_sample",
            "dflash_verify_sample_walk", "dflash_recall_at_k", "dflash2_conv",
            "dflash2_select")


def _check(rc: int):
    if rc != DFLASH_OK:
        raise DflashError(rc, LIB.dflash_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


# ----------------------------------------------------------------------------- lifecycle

def dflash_create(cfg: dflash_config) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(LIB.dflash_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h


def dflash_destroy(h) -> None:
    _check(LIB.dflash_destroy(h))


def dflash_set_weights(h, w: dflash_weights) -> None:
    _check(LIB.dflash_set_weights(h, ctypes.byref(w)))


def dflash_set_block_table(h, table) -> None:
    """table: int32 device tensor [max_batch, Cmax / DFLASH_PAGE_ROWS] (borrowed)."""
    _check(LIB.dflash_set_block_table(h, _ptr(table)))


def dflash_workspace_size(h) -> int:
    n = ctypes.c_size_t()
    _check(LIB.dflash_workspace_size(h, ctypes.byref(n)))
    return n.value


def dflash_status(h, ws, stream=None) -> int:
    code = ctypes.c_int()
    _check(LIB.dflash_status(h, _ptr(ws), _stream(stream), ctypes.byref(code)))
    return code.value


# ----------------------------------------------------------------------------- step calls

def dflash_ctx_project(h, nb, R, hv, n_commit, relay_a, ctx_len, kcache, vcache, x0_relay, ws,
                       stream=None) -> None:
    _check(LIB.dflash_ctx_project(h, nb, R, _ptr(hv), _ptr(n_commit), _ptr(relay_a), _ptr(ctx_len),
                                  _ptr(kcache), _ptr(vcache), _ptr(x0_relay), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)))


def dflash_ctx_project_film(h, nb, R, hv, n_commit, relay_a, relay_b, relay_y, ctx_len, kcache,
                            vcache, x0_relay, ws, stream=None) -> None:
    _check(LIB.dflash_ctx_project_film(h, nb, R, _ptr(hv), _ptr(n_commit), _ptr(relay_a),
                                       _ptr(relay_b), _ptr(relay_y), _ptr(ctx_len), _ptr(kcache),
                                       _ptr(vcache), _ptr(x0_relay), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(stream)))


def dflash_draft_block(h, nb, block_ids, x0_relay, kcache, vcache, ctx_len, max_ctx_hint,
                       out_hidden, ws, stream=None) -> None:
    _check(LIB.dflash_draft_block(h, nb, _ptr(block_ids), _ptr(x0_relay), _ptr(kcache), _ptr(vcache),
                                  _ptr(ctx_len), int(max_ctx_hint), _ptr(out_hidden), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)))


def dflash_lm_head_topk(h, nb, hidden, k, out_ids, out_vals, out_logits, ws, stream=None) -> None:
    _check(LIB.dflash_lm_head_topk(h, nb, _ptr(hidden), k, _ptr(out_ids), _ptr(out_vals),
                                   _ptr(out_logits), _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(stream)))


def dflash_lm_head_topk_noalloc(h, nb, hidden, k, out_ids, out_vals, out_status=None,
                                stream=None) -> None:
    _check(LIB.dflash_lm_head_topk_noalloc(h, nb, _ptr(hidden), k, _ptr(out_ids), _ptr(out_vals),
                                           _ptr(out_status), _stream(stream)))


def dflash_attention(h, nb, layer, q, kcache, vcache, ctx_len, max_ctx_hint, out_o, ws,
                     stream=None) -> None:
    _check(LIB.dflash_attention(h, nb, layer, _ptr(q), _ptr(kcache), _ptr(vcache), _ptr(ctx_len),
                                max_ctx_hint, _ptr(out_o), _ptr(ws), ws.numel() * ws.element_size(),
                                _stream(stream)))


def dflash_topk(h, rows, cols, logits, k, out_ids, out_vals, ws=None, stream=None) -> None:
    _check(LIB.dflash_topk(h, rows, cols, _ptr(logits), k, _ptr(out_ids), _ptr(out_vals), _ptr(ws),
                           0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def dflash_accept(h, nb, draft, target, out_tau, out_bonus, stream=None) -> None:
    _check(LIB.dflash_accept(h, nb, _ptr(draft), _ptr(target), _ptr(out_tau), _ptr(out_bonus),
                             _stream(stream)))


def dflash_accept_topk(h, nb, topk_ids, k, target, out_tau, out_bonus, stream=None) -> None:
    _check(LIB.dflash_accept_topk(h, nb, _ptr(topk_ids), int(k), _ptr(target), _ptr(out_tau), _ptr(out_bonus),
                                  _stream(stream)))


def dflash_sample(h, rows, logits, temperature, seed, row0, out_ids, out_lse, out_logq, ws,
                  stream=None) -> None:
    _check(LIB.dflash_sample(h, rows, _ptr(logits), float(temperature), int(seed), int(row0),
                             _ptr(out_ids), _ptr(out_lse), _ptr(out_logq), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream)))


def dflash_lm_head_sample(h, nb, hidden, temperature, seed, out_cand, out_lse, out_logq, out_logits,
                          k, out_ids, out_vals, ws, stream=None) -> None:
    _check(LIB.dflash_lm_head_sample(h, nb, _ptr(hidden), float(temperature), int(seed),
                                     _ptr(out_cand), _ptr(out_lse), _ptr(out_logq), _ptr(out_logits),
                                     int(k), _ptr(out_ids), _ptr(out_vals), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)))


def dflash_draw_gumbel(n, seed, stream_id, row, out_u, out_g, stream=None) -> None:
    _check(LIB.dflash_draw_gumbel(int(n), int(seed), int(stream_id), int(row), _ptr(out_u), _ptr(out_g),
                                  _stream(stream)))


def dflash_verify_sample(h, nb, draft_logits, draft_lse, cand, target_logits, temperature, seed,
                         out_tau, out_token, ws, stream=None) -> None:
    _check(LIB.dflash_verify_sample(h, nb, _ptr(draft_logits), _ptr(draft_lse), _ptr(cand),
                                    _ptr(target_logits), float(temperature), int(seed),
                                    _ptr(out_tau), _ptr(out_token), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)))


def dflash2_select_sample(h, nb, k, topk_ids, topk_vals, hidden, block_ids, temperature, seed,
                          out_path, out_walk_logq, ws, stream=None) -> None:
    _check(LIB.dflash2_select_sample(h, nb, k, _ptr(topk_ids), _ptr(topk_vals), _ptr(hidden),
                                     _ptr(block_ids), float(temperature), int(seed), _ptr(out_path),
                                     _ptr(out_walk_logq), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)))


def dflash_verify_sample_walk(h, nb, k, cand_ids, walk_logq, path, target_logits, temperature, seed,
                              out_tau, out_token, ws, stream=None) -> None:
    _check(LIB.dflash_verify_sample_walk(h, nb, k, _ptr(cand_ids), _ptr(walk_logq), _ptr(path),
                                         _ptr(target_logits), float(temperature), int(seed),
                                         _ptr(out_tau), _ptr(out_token), _ptr(ws),
                                         ws.numel() * ws.element_size(), _stream(stream)))


def dflash_recall_at_k(h, nb, k, cand_ids, target, hits, eligible, stream=None) -> None:
    _check(LIB.dflash_recall_at_k(h, nb, k, _ptr(cand_ids), _ptr(target), _ptr(hits), _ptr(eligible),
                                  _stream(stream)))


def dflash2_conv(h, layer, which, nb, x, ws, stream=None) -> None:
    _check(LIB.dflash2_conv(h, layer, which, nb, _ptr(x), _ptr(ws), ws.numel() * ws.element_size(),
                            _stream(stream)))


def dflash2_select(h, nb, k, topk_ids, topk_vals, hidden, block_ids, out_path, ws, stream=None) -> None:
    _check(LIB.dflash2_select(h, nb, k, _ptr(topk_ids), _ptr(topk_vals), _ptr(hidden), _ptr(block_ids),
                              _ptr(out_path), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream)))
