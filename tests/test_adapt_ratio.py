"""Run-time adaptation of r = BP/BH (no GPU).

The oracle's statement of the rule is pinned to a hand-worked trace and to
closed forms; the library's adapter (pure host code in the C ABI) must give
the oracle's r after every window of synthetic bandwidth traces."""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "adapt_ratio.json")


@pytest.fixture(scope="module")
def ft():
    from expert_cache_host_gb300 import build as ftbuild
    ftbuild.build()
    import expert_cache_host_gb300 as lib
    lib.load()
    return lib


def test_oracle_hand_worked_trace():
    g = json.load(open(GOLD))
    bp = [w["bp"] for w in g["windows"]]
    bh = [w["bh"] for w in g["windows"]]
    got = oracle.adapt_ratio_trace(bp, bh, g["alpha"], g["r_den"], g["r_num_max"])
    assert got.tolist() == [w["r_num"] for w in g["windows"]], [w["why"] for w in g["windows"]]


def test_oracle_closed_forms():
    # a constant trace gives r = BP/BH from the first window with both samples
    got = oracle.adapt_ratio_trace([210.0] * 5, [70.0] * 5, 0.3)
    assert got.tolist() == [768] * 5
    # alpha = 1: r follows the last samples alone
    bp = np.array([100.0, 300.0, 50.0, 200.0])
    bh = np.array([100.0, 100.0, 200.0, 25.0])
    assert oracle.adapt_ratio_trace(bp, bh, 1.0).tolist() == [256, 768, 64, 2048]
    # the cap, and r = 0 never arises from positive samples unless BP/BH < 1/(2 r_den)
    assert oracle.adapt_ratio_trace([1e6], [1.0], 0.5, 256, 1000).tolist() == [1000]
    assert oracle.adapt_ratio_trace([1.0], [1e6], 0.5).tolist() == [0]
    # monotone in BP for a fixed BH
    rs = [oracle.adapt_ratio_trace([x], [100.0], 0.5)[0] for x in np.linspace(1.0, 400.0, 50)]
    assert all(a <= b for a, b in zip(rs, rs[1:]))


def test_library_adapter_matches_oracle_on_synthetic_traces(ft):
    rng = np.random.default_rng(7)
    for trial in range(20):
        n = int(rng.integers(1, 60))
        alpha = float(rng.choice([1.0, 0.5, 0.25, 0.1, 0.9]))
        # link rates around 100-220 GB/s and host rates around 20-400 GB/s, with windows that carry no sample
        bp = np.where(rng.random(n) < 0.2, 0.0, rng.uniform(90.0, 220.0, n))
        bh = np.where(rng.random(n) < 0.4, 0.0, rng.uniform(20.0, 400.0, n))
        r_den, r_max = int(rng.choice([1, 16, 256, 1024])), int(rng.choice([4, 1000, 16384]))
        want = oracle.adapt_ratio_trace(bp, bh, alpha, r_den, r_max)
        a = ft.ft_ratio_adapter_init(alpha, r_den, r_max)
        prev = -1
        for i in range(n):
            changed = ft.ft_ratio_adapter_update(a, float(bp[i]), float(bh[i]))
            assert a.r_num == want[i], f"trial {trial} window {i}"
            assert changed == int(a.r_num != prev)
            prev = a.r_num


def test_library_adapter_golden_and_bad_arguments(ft):
    g = json.load(open(GOLD))
    a = ft.ft_ratio_adapter_init(g["alpha"], g["r_den"], g["r_num_max"])
    for w in g["windows"]:
        ft.ft_ratio_adapter_update(a, w["bp"], w["bh"])
        assert a.r_num == w["r_num"], w["why"]
    for bad in ((0.0, 256, 10), (1.5, 256, 10), (0.5, 0, 10), (0.5, 256, -1)):
        with pytest.raises(ft.FtError):
            ft.ft_ratio_adapter_init(*bad)
    with pytest.raises(ft.FtError):
        ft.ft_ratio_adapter_update(ft.ft_ratio_adapter(), 1.0, 1.0)  # never initialised
