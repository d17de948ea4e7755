"""Host-side arithmetic of bench.py, checked without a GPU: the roofline's algorithmic
bytes per step against the figures derived from the workload shapes by hand (weights read
once, each context K/V row read once per layer), and the launch count per step against
the ncu launch list of the default step (117 launches of the library over 3 steps)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import dflash_inputs as di  # noqa: E402


def _weights_by_hand(D, N, Hq, Hkv, hd, F, V, L, Dt):
    per_layer = (Hq + 2 * Hkv) * hd * D + D * Hq * hd + 3 * F * D + 2 * Hkv * hd * D
    norms = 2 * D * N + 2 * D          # attention and FFN gains per layer, g_ctx and g_final
    return 2 * (N * per_layer + D * L * Dt + V * D + norms)


def test_default_step_bytes():
    w = di.QWEN3_8B
    ctx = di.context_lengths(w).astype(np.int32)
    tp = di.tau_prev(w).astype(np.int32)
    total, flops, wbytes, kv = bench.step_bytes_flops(w, ctx, tp)
    assert wbytes == _weights_by_hand(4096, 5, 32, 8, 128, 12288, 151936, 5, 4096)
    assert abs(wbytes / 1e9 - 3.426) < 5e-4       # Qwen3-8B-shaped drafter: 3.426 GB
    assert kv == 8 * 4096 * 5 * 2 * 8 * 128 * 2    # 8 sequences x 4096 rows: 0.671 GB
    assert 0 < total - wbytes - kv < 0.01 * total  # inputs and outputs are small
    assert flops > 2 * 8 * 15 * 151936 * 4096      # at least the LM head


def test_4b_and_ragged_step_bytes():
    w = di.QWEN3_4B
    ctx = di.context_lengths(w).astype(np.int32)
    _, _, wbytes, kv = bench.step_bytes_flops(w, ctx, di.tau_prev(w).astype(np.int32))
    assert wbytes == _weights_by_hand(2560, 5, 32, 8, 128, 9728, 151936, 5, 2560)
    assert kv == 2048 * 5 * 2 * 8 * 128 * 2
    w = di.SWEEP_NB64
    ctx = di.context_lengths(w).astype(np.int32)
    assert ctx.min() >= 1024 and ctx.max() <= 8192
    _, _, _, kv = bench.step_bytes_flops(w, ctx, di.tau_prev(w).astype(np.int32))
    assert kv == int(ctx.sum()) * 5 * 2 * 8 * 128 * 2


def test_optional_weights_are_counted():
    base = bench.step_bytes_flops(di.QWEN3_8B, np.full(8, 4096), np.ones(8, np.int32))[2]
    film = bench.step_bytes_flops(di.FILM_RELAY.with_(nb=8), np.full(8, 4096), np.ones(8, np.int32))[2]
    assert film - base == 2 * 5 * 4096 * 1024     # W1 [1024, 3D] and W2 [2D, 1024]
    sel = bench.step_bytes_flops(di.QWEN3_8B.with_(flags=di.FLAG_SELECT), np.full(8, 4096),
                                 np.ones(8, np.int32))[2]
    assert sel - base == 2 * 3 * 256 * 4096        # W_A, W_B, W_G


def test_launches_per_default_step_match_the_launch_list():
    assert bench.kernels_per_step(di.QWEN3_8B) == 117 // 3
    assert bench.kernels_per_step(di.PAGED_KV) == bench.kernels_per_step(di.QWEN3_8B)


def test_step_summary_of_a_measured_workload():
    """The `workloads` entry of the bench line: blocks/s = sequences / step time and the
    step's roofline fraction = max(bytes / HBM, FLOPs / sustained bf16) / step time."""
    w = di.SWEEP_NB64
    ctx = di.context_lengths(w).astype(np.int32)
    tp = di.tau_prev(w).astype(np.int32)
    m = dict(w=w, ctx=ctx, tp=tp, ms_step=2.5, clk=None, tau=np.full(w.nb, 3))
    out = bench.step_summary(m, world=1)
    assert abs(out["value"] - 64 / 2.5e-3) < 1e-6 * out["value"]
    assert out["draft_tokens_per_s"] == round(out["value"] * 7, 1)
    hbm, tf_burst, tf_sus, _ = bench.load_peaks()
    total, flops, _, _ = bench.step_bytes_flops(w, ctx, tp)
    roof = max(total / (hbm * 1e9), flops / ((tf_sus or tf_burst) * 1e12))
    assert abs(out["step_roofline"]["frac"] - round(roof * 1e3 / 2.5, 4)) < 1e-9
    assert out["config"]["nb_per_gpu"] == 64 and out["config"]["B"] == 8
