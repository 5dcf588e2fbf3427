"""The seeded input recipes: the routed-expert segment counts (Zipf(1.1) by
rank over 64 experts, capped at the 16,384 tokens that top-8 routing can send
to one expert, excess re-spread, largest-remainder rounding) and the
distributions of the named workloads."""
import numpy as np

import workloads


def test_zipf_counts_cap_and_total():
    c = workloads.zipf_segment_counts()
    assert c.sum() == 16384 * 8 and len(c) == 64
    assert c.max() == 16384 and (c <= 16384).all() and (c > 0).all()
    assert (np.diff(c) <= 0).all()                       # non-increasing by rank
    assert list(c[:8]) == [16384, 16384, 11625, 8471, 6628, 5423, 4577, 3952]
    assert list(c[-3:]) == [416, 408, 401]


def test_zipf_counts_follow_the_power_law_where_uncapped():
    c = workloads.zipf_segment_counts().astype(np.float64)
    e = np.arange(64) + 1.0
    free = c < 16384
    # uncapped experts share the remainder in proportion to (e)^-1.1, to within rounding
    k = c[free].sum() / (e[free] ** -1.1).sum()
    assert np.max(np.abs(c[free] - k * e[free] ** -1.1)) < 1.0


def test_plain_zipf_would_exceed_the_cap():
    """Uncapped Zipf(1.1) over 64 ranks gives the top expert about a quarter
    of the rows, more than one token can route to it."""
    w = (np.arange(64) + 1.0) ** -1.1
    assert 131072 * w[0] / w.sum() > 16384


def test_segment_offsets():
    c = workloads.zipf_segment_counts()
    seg = workloads.segment_offsets(c)
    assert seg.dtype == np.int32 and seg[0] == 0 and seg[-1] == 131072
    assert (np.diff(seg) == c).all()


def test_named_workload_distributions():
    x, dy = workloads.isolated_hbm("f16", n=1 << 20)
    xv = x.view(np.float16).astype(np.float64)
    out = np.abs(xv) > 12          # beyond 4 sigma: the 1 % U[-40, 40] outliers, 28/40 of them
    assert 0.006 < out.mean() < 0.008 and np.abs(xv).max() <= 40
    core = xv[~out]
    assert abs(core.std() - 3.0) < 0.05
    assert abs(dy.view(np.float16).astype(np.float64).std() - 1.0) < 0.01
