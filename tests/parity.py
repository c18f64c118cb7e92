"""Comparison rules shared by the GPU parity tests (no method arithmetic here beyond
checking results against the oracle).

* votes / cumulative scores: |gpu - oracle| <= 1e-5 * |oracle| + 1e-9;
* kept or evicted index sets: identical, except swaps between candidates whose fp64
  (pooled) score lies within 1e-4 relative of the selection boundary;
* attention outputs from bf16 inputs: |gpu - oracle| <= 2e-2 + 1e-2 * |oracle|.
"""

import numpy as np

VOTE_RTOL, VOTE_ATOL = 1e-5, 1e-9
BAND = 1e-4
OUT_ATOL, OUT_RTOL = 2e-2, 1e-2


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_votes_close(gpu, ref, what="votes"):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    bad = err > VOTE_RTOL * np.abs(ref) + VOTE_ATOL
    if bad.any():
        i = int(np.argmax(err / (np.abs(ref) + VOTE_ATOL)))
        raise AssertionError("%s: %d of %d outside 1e-5 rel; worst at %d: gpu %.9g ref %.9g"
                             % (what, int(bad.sum()), bad.size, i, gpu.flat[i], ref.flat[i]))


def assert_outputs_close(gpu, ref, what="attention output"):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    bad = err > OUT_ATOL + OUT_RTOL * np.abs(ref)
    if bad.any():
        i = int(np.argmax(err))
        raise AssertionError("%s: %d of %d outside 2e-2 abs + 1e-2 rel; worst %.4g (gpu %.6g ref %.6g)"
                             % (what, int(bad.sum()), bad.size, err.flat[i], gpu.flat[i], ref.flat[i]))


def check_selected_set(gpu_pos, ref_pos, pooled, k, what="kept set"):
    """gpu_pos/ref_pos: chosen prefix positions (k each).  pooled: the oracle's fp64
    pooled vote over the candidates.  Returns the number of in-band swaps."""
    g, r = set(int(x) for x in gpu_pos), set(int(x) for x in ref_pos)
    assert len(g) == len(gpu_pos) == k, "%s: %d positions, %d distinct, want %d" % (
        what, len(gpu_pos), len(g), k)
    assert list(gpu_pos) == sorted(gpu_pos), "%s: not ascending" % what
    if g == r:
        return 0
    boundary = np.sort(pooled)[::-1][k - 1]
    for j in g ^ r:
        assert abs(pooled[j] - boundary) <= BAND * abs(boundary), (
            "%s: position %d (pooled %.9g) differs outside the 1e-4 band of the boundary %.9g"
            % (what, j, pooled[j], boundary))
    return len(g ^ r) // 2
