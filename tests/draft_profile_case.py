"""Small case of the drafter layer's kernels for profiling: one Qwen3-8B-shaped layer
(D = 4096, 32/8 heads of 128, F = 12288) with a 4096-token vocabulary, 8 sequences of
B = 16 over 4096 context rows, so the QKV, attention, O, gate|up and down launches have the
bench workload's shapes while the device holds about 0.6 GB. Calls dflash_draft_block a
few times and prints the time of the last call.

    python tests/draft_profile_case.py

Not a test; it uses the C-ABI binding only.
"""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import dflash_inputs as di  # noqa: E402
from block_diffusion_speculative_project_gb300 import drafter  # noqa: E402


def main():
    w = di.QWEN3_8B.with_(N=1, V=4096, L=1)
    C = w.C
    dev = {k: drafter.to_device_bf16(v) for k, v in di.make_weights(w).items()}
    dr = drafter.Drafter(w, dev, w.nb, C + w.B, w.B)
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    dr.kcache.normal_(generator=g)
    dr.vcache.normal_(generator=g)
    ids = torch.tensor(di.block_ids(w, di.anchors(w)), dtype=torch.int32, device="cuda")
    ctx = torch.full((w.nb,), C, dtype=torch.int32, device="cuda")
    out = torch.empty(w.nb, w.B, w.D, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream()
    for _ in range(3):
        dr.draft_block(w.nb, ids, ctx, out, max_ctx_hint=C)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    dr.draft_block(w.nb, ids, ctx, out, max_ctx_hint=C)
    e1.record(s)
    torch.cuda.synchronize()
    print(f"draft_block, one layer: {e0.elapsed_time(e1) * 1e3:.1f} us (host launch time included); "
          f"status {dr.status()}; finite {bool(torch.isfinite(out.float()).all())}")


if __name__ == "__main__":
    main()
