"""Small case of the sampling kernels for profiling: a handle with a 151936-token
vocabulary (tiny drafter weights otherwise) and 16 sequences of B = 16, so the draft logits
(146 MB) and the target logits (156 MB) both exceed L2 while the device holds well under
1 GB. Runs dflash_sample and dflash_verify_sample a few times and prints their times.

    python tests/sampling_profile_case.py

Not a test (no assertions on values); it uses the C-ABI binding only.
"""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import dflash_inputs as di  # noqa: E402
from block_diffusion_speculative_project_gb300 import drafter  # noqa: E402

V, B, NB = 151936, 16, 16


def main():
    w = di.TINY.with_(V=V, B=B, nb=NB)
    dev = {k: drafter.to_device_bf16(v) for k, v in di.make_weights(w).items()}
    dr = drafter.Drafter(w, dev, NB, 80, 8)
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    U = torch.randn(NB, B - 1, V, device="cuda", generator=g) * 2
    Z = torch.randn(NB, B, V, device="cuda", generator=g) * 2
    cand = torch.zeros(NB, B - 1, dtype=torch.int32, device="cuda")
    lse = torch.zeros(NB, B - 1, device="cuda")
    tau = torch.zeros(NB, dtype=torch.int32, device="cuda")
    tok = torch.zeros_like(tau)
    s = torch.cuda.current_stream()
    for it in range(3):
        dr.sample(NB * (B - 1), U, 1.0, 7 + it, cand, lse)
        dr.verify_sample(NB, U, lse, cand, Z, 1.0, 7 + it, tau, tok)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    ev[0].record(s)
    dr.sample(NB * (B - 1), U, 1.0, 99, cand, lse)
    ev[1].record(s)
    dr.verify_sample(NB, U, lse, cand, Z, 1.0, 99, tau, tok)
    ev[2].record(s)
    torch.cuda.synchronize()
    print(f"draw {ev[0].elapsed_time(ev[1]) * 1e3:.1f} us, verify {ev[1].elapsed_time(ev[2]) * 1e3:.1f} us "
          f"(host launch time included); status {dr.status()}")


if __name__ == "__main__":
    main()
