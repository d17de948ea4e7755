"""Holder for one libdflash handle: device weights, KV caches and workspace.

PyTorch supplies device memory and the stream; every step is a call into the C ABI
(see dflash.py). Weight tensors are borrowed by the handle and kept alive here.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import dflash as _d


def to_device_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 bit patterns (uint16 numpy) -> bf16 torch tensor on the device."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


class Drafter:
    """One handle with its caches [N, max_batch, Hkv, Cmax, hd] and workspace; with
    ``num_pages`` > 0 the caches are page pools [N, num_pages, Hkv, 64, hd] read and
    written through the block table given to ``set_block_table``.

    ``shape`` is any object with the workload fields D, Dt, L, N, Hq, Hkv, hd, F, V,
    B, k_top, rope_base, eps, mask_id, flags, conv_group, sel_dim and film_width.
    ``weights`` maps the weight names of dflash_inputs.weight_shapes to bf16 device
    tensors.
    """

    def __init__(self, shape, weights: dict, max_batch: int, Cmax: int, max_proj_rows: int,
                 max_spin: int = 0, device="cuda", num_pages: int = 0):
        self.shape = shape
        s = shape
        self.cfg = _d.dflash_config(
            D=s.D, Dt=s.Dt, L=s.L, N=s.N, Hq=s.Hq, Hkv=s.Hkv, hd=s.hd, F=s.F, V=s.V, B=s.B,
            k_top=s.k_top, rope_base=s.rope_base, eps=s.eps, mask_id=s.mask_id, Cmax=Cmax,
            max_batch=max_batch, max_proj_rows=max_proj_rows, conv_group=s.conv_group,
            sel_dim=s.sel_dim, flags=s.flags, max_spin=max_spin, film_dim=s.film_width,
            num_pages=num_pages)
        self.h = _d.dflash_create(self.cfg)
        self.weights = weights
        P = lambda name: ctypes.c_void_p(weights[name].data_ptr()) if name in weights else None
        layers = (_d.dflash_layer_weights * s.N)()
        for n in range(s.N):
            p = f"layer{n}."
            L = layers[n]
            for f in ("W_qkv", "Wk_c", "Wv_c", "W_o", "W_gate", "W_up", "W_down", "g_attn", "g_ffn"):
                setattr(L, f, P(p + f))
            for q in range(4):
                L.conv_W0[q] = P(p + f"conv{q}.W0")
                L.conv_W1[q] = P(p + f"conv{q}.W1")
                L.conv_base[q] = P(p + f"conv{q}.base")
        self._layers = layers
        self.wstruct = _d.dflash_weights(W_c=P("W_c"), g_ctx=P("g_ctx"), E=P("E"), W_lm=P("W_lm"),
                                         g_final=P("g_final"), W_A=P("W_A"), W_B=P("W_B"),
                                         W_G=P("W_G"), layers=layers, film_W1=P("film.W1"),
                                         film_W2=P("film.W2"))
        _d.dflash_set_weights(self.h, self.wstruct)
        nbytes = _d.dflash_workspace_size(self.h)
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        cshape = ((s.N, num_pages, s.Hkv, _d.DFLASH_PAGE_ROWS, s.hd) if num_pages > 0
                  else (s.N, max_batch, s.Hkv, Cmax, s.hd))
        self.kcache = torch.zeros(cshape, dtype=torch.bfloat16, device=device)
        self.vcache = torch.zeros(cshape, dtype=torch.bfloat16, device=device)
        self.max_batch, self.Cmax, self.max_proj_rows = max_batch, Cmax, max_proj_rows
        self.num_pages = num_pages
        self.block_table = None

    def set_block_table(self, table: torch.Tensor):
        """Register the int32 device block table [max_batch, Cmax / 64] (kept alive here)."""
        assert table.dtype == torch.int32 and table.is_cuda and table.is_contiguous()
        assert tuple(table.shape) == (self.max_batch, self.Cmax // _d.DFLASH_PAGE_ROWS)
        self.block_table = table
        _d.dflash_set_block_table(self.h, table)

    def __del__(self):
        try:
            if getattr(self, "h", None):
                _d.dflash_destroy(self.h)
                self.h = None
        except Exception:
            pass

    # thin forwards -------------------------------------------------------------
    def ctx_project(self, nb, R, hv, n_commit, ctx_len, relay_a=None, x0_relay=None, stream=None,
                    relay_b=None, relay_y=None):
        if relay_b is not None or relay_y is not None:
            _d.dflash_ctx_project_film(self.h, nb, R, hv, n_commit, relay_a, relay_b, relay_y, ctx_len,
                                       self.kcache, self.vcache, x0_relay, self.ws, stream)
        else:
            _d.dflash_ctx_project(self.h, nb, R, hv, n_commit, relay_a, ctx_len, self.kcache,
                                  self.vcache, x0_relay, self.ws, stream)

    def draft_block(self, nb, block_ids, ctx_len, out_hidden, x0_relay=None, max_ctx_hint=0,
                    stream=None):
        _d.dflash_draft_block(self.h, nb, block_ids, x0_relay, self.kcache, self.vcache, ctx_len,
                              max_ctx_hint, out_hidden, self.ws, stream)

    def lm_head_topk(self, nb, hidden, k, out_ids, out_vals, out_logits=None, stream=None):
        _d.dflash_lm_head_topk(self.h, nb, hidden, k, out_ids, out_vals, out_logits, self.ws, stream)

    def accept(self, nb, draft, target, out_tau, out_bonus, stream=None):
        _d.dflash_accept(self.h, nb, draft, target, out_tau, out_bonus, stream)

    def accept_topk(self, nb, topk_ids, k, target, out_tau, out_bonus, stream=None):
        _d.dflash_accept_topk(self.h, nb, topk_ids, k, target, out_tau, out_bonus, stream)

    def sample(self, rows, logits, temperature, seed, out_ids, out_lse, out_logq=None, row0=0,
               stream=None):
        _d.dflash_sample(self.h, rows, logits, temperature, seed, row0, out_ids, out_lse, out_logq,
                         self.ws, stream)

    def lm_head_sample(self, nb, hidden, temperature, seed, out_cand, out_lse, out_logq=None,
                       out_logits=None, k=0, out_ids=None, out_vals=None, stream=None):
        _d.dflash_lm_head_sample(self.h, nb, hidden, temperature, seed, out_cand, out_lse, out_logq,
                                 out_logits, k, out_ids, out_vals, self.ws, stream)

    def verify_sample(self, nb, draft_logits, draft_lse, cand, target_logits, temperature, seed,
                      out_tau, out_token, stream=None):
        _d.dflash_verify_sample(self.h, nb, draft_logits, draft_lse, cand, target_logits, temperature,
                                seed, out_tau, out_token, self.ws, stream)

    def conv(self, layer, which, nb, x, stream=None):
        _d.dflash2_conv(self.h, layer, which, nb, x, self.ws, stream)

    def select(self, nb, k, topk_ids, topk_vals, hidden, block_ids, out_path, stream=None):
        _d.dflash2_select(self.h, nb, k, topk_ids, topk_vals, hidden, block_ids, out_path, self.ws,
                          stream)

    def select_sample(self, nb, k, topk_ids, topk_vals, hidden, block_ids, temperature, seed, out_path,
                      out_walk_logq, stream=None):
        _d.dflash2_select_sample(self.h, nb, k, topk_ids, topk_vals, hidden, block_ids, temperature, seed,
                                 out_path, out_walk_logq, self.ws, stream)

    def verify_sample_walk(self, nb, k, cand_ids, walk_logq, path, target_logits, temperature, seed,
                           out_tau, out_token, stream=None):
        _d.dflash_verify_sample_walk(self.h, nb, k, cand_ids, walk_logq, path, target_logits, temperature,
                                     seed, out_tau, out_token, self.ws, stream)

    def recall_at_k(self, nb, k, cand_ids, target, hits, eligible, stream=None):
        _d.dflash_recall_at_k(self.h, nb, k, cand_ids, target, hits, eligible, stream)

    def attention(self, nb, layer, q, ctx_len, out_o, max_ctx_hint=0, stream=None):
        _d.dflash_attention(self.h, nb, layer, q, self.kcache, self.vcache, ctx_len, max_ctx_hint,
                            out_o, self.ws, stream)

    def topk(self, rows, cols, logits, k, out_ids, out_vals, stream=None):
        _d.dflash_topk(self.h, rows, cols, logits, k, out_ids, out_vals, None, stream)

    def status(self, stream=None) -> int:
        return _d.dflash_status(self.h, self.ws, stream)
