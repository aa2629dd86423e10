"""Host-side accounting of the benchmark (no GPU): the visible-pair count
behind every algorithmic TFLOP/s and roofline figure, and the counted FLOPs
of the headline metric."""
import itertools

import pytest

import bench
import fa_inputs


def brute_force_pairs(Tq, Tkv, causal, window, rows=None):
    # key j is hidden from query i when (causal and j > i) or (window > 0 and
    # i >= j and i - j >= window)
    lo, hi = (0, Tq) if rows is None else rows
    n = 0
    for i in range(lo, hi):
        for j in range(Tkv):
            if causal and j > i:
                continue
            if window > 0 and i >= j and i - j >= window:
                continue
            n += 1
    return n


@pytest.mark.parametrize("Tq,Tkv,causal,window", list(itertools.product(
    [1, 7, 64, 130], [1, 9, 64, 200], [False, True], [0, 1, 5, 70])))
def test_visible_pairs_match_the_mask(Tq, Tkv, causal, window):
    w = fa_inputs.Workload("p", 1, 1, 1, Tq, Tkv, 64, "fp16", causal, window)
    assert bench.visible_pairs_per_head(w) == brute_force_pairs(Tq, Tkv, causal, window)


def test_visible_pairs_row_range():
    w = fa_inputs.Workload("p", 1, 1, 1, 300, 250, 64, "bf16", True, 40)
    assert bench.visible_pairs_per_head(w, rows=(100, 180)) == \
        brute_force_pairs(300, 250, True, 40, rows=(100, 180))


def test_headline_counted_flops():
    """4 B Hq Tq Tkv D for the forward, halved under the causal mask, and 2.5
    times that for the backward: 1.924 TFLOP per step at the headline shape."""
    w = fa_inputs.WORKLOADS[fa_inputs.HEADLINE]
    fwd, bwd = bench.counted_flops(w)
    assert fwd == 4 * 4 * 32 * 4096 * 4096 * 128 / 2
    assert bwd == 2.5 * fwd
    assert abs((fwd + bwd) / 1e12 - 1.924) < 1e-3
    # the visible pairs of one causal head are T (T + 1) / 2
    assert bench.visible_pairs_per_head(w) == 4096 * 4097 // 2
