"""The allocation-free LM head (dflash_lm_head_topk_noalloc) against the workspace one.

Some callers cannot give the library a workspace: code recorded into a CUDA graph,
where a cudaMalloc is not allowed; processes whose device memory is entirely owned
by another pool allocator; threads that must not risk the device synchronisation an
allocation can cause. For them the LM head keeps its scratch in a static device
array. This test calls that entry point through the C ABI twice in a row, on
different inputs, and checks each result against dflash_lm_head_topk on the same
inputs (ids exactly, logits within the parity tolerance) and against the oracle's
logits of the same hidden rows (ids by the margin rule, values within the tolerance);
the second call passes no status word, so the entry point clears the one inside its
own scratch. It is collected last and also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import dflash_inputs as di
from _parity import assert_close, check_topk
from oracle import dflash_oracle as orc

pytestmark = pytest.mark.gpu

SHAPE = di.Workload("noalloc_check_d512_v5003_b16", D=512, Dt=192, L=5, N=1, Hq=8, Hkv=2, hd=128,
                    F=1000, V=5003, B=16, nb=3, C=64)


def test_noalloc_lm_head_matches_workspace_lm_head_on_two_calls():
    from block_diffusion_speculative_project_gb300 import dflash, drafter
    w = SHAPE
    bits = di.make_weights(w)
    dev = {k: drafter.to_device_bf16(v) for k, v in bits.items()}
    dr = drafter.Drafter(w, dev, w.nb, 64, w.B)
    W = orc.widen_all(bits)
    k = w.k_top
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        hid_bits = di.normal_bf16(f"noalloc_hidden{call}", (w.nb, w.B, w.D), 1.0)
        hid = drafter.to_device_bf16(hid_bits)
        ids_ws = torch.empty(w.nb, w.B - 1, k, dtype=torch.int32, device="cuda")
        vals_ws = torch.empty(w.nb, w.B - 1, k, dtype=torch.float32, device="cuda")
        dr.lm_head_topk(w.nb, hid, k, ids_ws, vals_ws)
        ids_na = torch.full_like(ids_ws, -1)
        vals_na = torch.full_like(vals_ws, float("nan"))
        # the first call reports device errors into the caller's word, the second into the
        # word inside the entry point's own scratch (not read back)
        dflash.dflash_lm_head_topk_noalloc(dr.h, w.nb, hid, k, ids_na, vals_na, status if call == 0 else None)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert dr.status() == 0
        assert np.array_equal(ids_na.cpu().numpy(), ids_ws.cpu().numpy()), f"call {call}: ids differ"
        assert_close(vals_na.cpu().numpy(), vals_ws.cpu().numpy(), f"call {call}: values")
        logits = orc.lm_logits(W, orc.widen(hid_bits))
        und = check_topk(ids_na.cpu().numpy(), vals_na.cpu().numpy(), logits, k, f"call {call}: oracle",
                         abs_delta=2e-3)
        # deep top-k positions have small gaps; most decisions are still above the margin
        assert und < w.nb * (w.B - 1) * k // 2, f"call {call}: {und} positions under the margin"


def test_noalloc_lm_head_rejects_shapes_beyond_its_scratch():
    from block_diffusion_speculative_project_gb300 import dflash, drafter
    # 33000 LM-head rows in one call: more row tiles than SMs, so the partial lists
    # need 33000 * 16 * 8 bytes, beyond the 4 MiB static scratch
    w = SHAPE.with_(name="noalloc_too_big", B=2, nb=33000)
    shapes = di.weight_shapes(w)
    dev = {n: torch.zeros(s, dtype=torch.bfloat16, device="cuda") for n, s in shapes.items()}
    dr = drafter.Drafter(w, dev, w.nb, 16, w.B)
    hid = torch.zeros(w.nb, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(w.nb, w.B - 1, 16, dtype=torch.int32, device="cuda")
    vals = torch.empty(w.nb, w.B - 1, 16, dtype=torch.float32, device="cuda")
    del dev
    with pytest.raises(dflash.DflashError) as e:
        dflash.dflash_lm_head_topk_noalloc(dr.h, w.nb, hid, 16, ids, vals)
    assert e.value.code == dflash.DFLASH_ERR_UNSUPPORTED_SHAPE
