"""Helpers shared by the GPU parity tests: tolerance checks and the top-k margin rule.

Continuous outputs: |gpu - oracle| <= 2e-2 + 1e-2 * |oracle| (the draft step's stated
bf16 tolerance). Discrete outputs decided by floating point (top-k ids, selector
path): bit-exact wherever the oracle's decision margin exceeds
delta = 1e-2 * max(1, |v|); below that margin the GPU's choice must be a valid one
within delta under the oracle's values, and such positions are counted.
"""
import numpy as np

ATOL = 2e-2
RTOL = 1e-2


def assert_close(g, o, what="", atol=ATOL, rtol=RTOL):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    assert g.shape == o.shape, f"{what}: shape {g.shape} vs {o.shape}"
    if g.size == 0:
        return 0.0
    assert np.isfinite(g).all(), f"{what}: non-finite GPU values"
    err = np.abs(g - o)
    bad = err > atol + rtol * np.abs(o)
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} outside tolerance, "
                           f"max abs err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def check_topk(gpu_ids, gpu_vals, logits, k, what="", abs_delta=None):
    """Rule-D check of a top-k result against oracle logits [rows, V] (float64).

    delta = 1e-2 * max(1, |v|) when the logits come from different inputs (end to end);
    ``abs_delta`` replaces it when both sides computed the logits from the same inputs,
    so only fp32-versus-fp64 accumulation separates them."""
    logits = np.asarray(logits, dtype=np.float64).reshape(-1, logits.shape[-1])
    gpu_ids = np.asarray(gpu_ids).reshape(-1, k)
    gpu_vals = np.asarray(gpu_vals, dtype=np.float64).reshape(-1, k)
    undecided = 0
    cols = np.arange(logits.shape[1])
    for r in range(logits.shape[0]):
        order = np.lexsort((cols, -logits[r]))[: k + 1]
        v = logits[r, order]
        assert len(set(gpu_ids[r].tolist())) == k, f"{what}: duplicate ids in row {r}"
        for j in range(k):
            delta = abs_delta if abs_delta is not None else 1e-2 * max(1.0, abs(v[j]))
            lo_ok = j == 0 or (v[j - 1] - v[j]) > delta
            hi_ok = (v[j] - v[j + 1]) > delta if j + 1 < len(v) else True
            gid = int(gpu_ids[r, j])
            assert 0 <= gid < logits.shape[1], f"{what}: id {gid} out of range"
            if lo_ok and hi_ok:
                assert gid == int(order[j]), (f"{what}: row {r} pos {j}: gpu id {gid} vs oracle "
                                              f"{int(order[j])} (margin above delta)")
            else:
                undecided += 1
                assert abs(logits[r, gid] - v[j]) <= delta, (f"{what}: row {r} pos {j}: gpu id {gid} "
                                                             "is not a valid choice within delta")
            assert abs(gpu_vals[r, j] - logits[r, gid]) <= ATOL + RTOL * abs(logits[r, gid]), \
                f"{what}: row {r} pos {j}: value {gpu_vals[r, j]} vs {logits[r, gid]}"
    return undecided
