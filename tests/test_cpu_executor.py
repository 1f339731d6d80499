"""The CPU expert executor's arithmetic (ft_cpu_experts: host arrays, no
context, no GPU) against the oracle's CPU partial sum.

The executor computes, for the routes of a step that got no cache slot, the
sum over those routes of w * SwiGLU expert(hidden) in fp32 on the host cores
(FreeToken article, section "设计 1", Decode bullet: the misses that are not
filled run on the CPU and their partial sum is merged exactly).  The oracle's
moe_forward returns the same quantity in fp64 as its third output.
"""
import numpy as np
import pytest

import ftsynth
import oracle
import expert_cache_host_gb300 as ft
from expert_cache_host_gb300 import build as ftbuild

# fp32 dot products of length <= 2048 against fp64: errors of a few ulp of the
# row sums; this bound is far below the decode path's tolerance
CPU_MAX_REL = 1e-4
CPU_NORMWISE = 1e-5


@pytest.fixture(scope="module")
def lib():
    ftbuild.build()
    return ft.load()


def _case(dtype, E=8, k=3, d=256, f=128, L=2, T=5, seed=1):
    pool = ftsynth.make_pool(seed, L, E, d, f, dtype, 0.05, threads=2)
    ids, w = oracle.route(ftsynth.test_logits(seed + 3, 0, T, E), k)
    w32 = w.astype(np.float32)
    hid = ftsynth.normal_bf16(seed + 5, 6, 0, 0, T * d).reshape(T, d)
    return pool, ids, w32, hid


def _oracle_cpu(pool, layer, E, dtype, d, f, ids, w32, hid, sid):
    bx = ftsynth.expert_bytes(d, f, dtype)
    layer_pool = pool[layer * E * bx:(layer + 1) * E * bx]
    _, _, cpu = oracle.moe_forward(layer_pool, bx, dtype, d, f, ids, w32.astype(np.float64), hid, slot_ids=sid)
    return cpu


@pytest.mark.parametrize("dtype", [0, 1])
def test_matches_oracle_cpu_partial(lib, dtype):
    E, k, d, f, L, T = 8, 3, 256, 128, 2, 5
    pool, ids, w32, hid = _case(dtype, E, k, d, f, L, T)
    rng = np.random.default_rng(7)
    for layer in range(L):
        for _ in range(3):
            sid = np.where(rng.random((T, k)) < 0.5, -1, 2).astype(np.int32)
            got = ft.ft_cpu_experts(pool, E, k, d, f, dtype, layer, ids, w32, sid, hid, threads=3)
            ref = _oracle_cpu(pool, layer, E, dtype, d, f, ids, w32, hid, sid)
            assert oracle.max_rel_err(got, ref) <= CPU_MAX_REL
            assert oracle.normwise_err(got, ref) <= CPU_NORMWISE
            # tokens with every route on the GPU get exactly zero
            for t in range(T):
                if np.all(sid[t] >= 0):
                    assert np.all(got[t] == 0)


@pytest.mark.parametrize("dtype", [0, 1])
def test_result_does_not_depend_on_threads(lib, dtype):
    E, k, d, f, T = 8, 4, 512, 256, 3
    pool, ids, w32, hid = _case(dtype, E, k, d, f, 1, T, seed=4)
    sid = np.full((T, k), -1, dtype=np.int32)
    one = ft.ft_cpu_experts(pool, E, k, d, f, dtype, 0, ids, w32, sid, hid, threads=1)
    for n in (2, 5, 16):
        assert np.array_equal(ft.ft_cpu_experts(pool, E, k, d, f, dtype, 0, ids, w32, sid, hid, threads=n), one)


def test_all_gpu_routes_give_zero_and_bad_ids_are_skipped(lib):
    E, k, d, f, T = 8, 2, 256, 128, 4
    pool, ids, w32, hid = _case(0, E, k, d, f, 1, T, seed=9)
    got = ft.ft_cpu_experts(pool, E, k, d, f, 0, 0, ids, w32, np.zeros((T, k), np.int32), hid)
    assert np.all(got == 0)
    # a route id outside [0, E) contributes nothing (the control kernel treats it as absent)
    bad = ids.copy()
    bad[:, 1] = E + 3
    sid = np.full((T, k), -1, dtype=np.int32)
    got = ft.ft_cpu_experts(pool, E, k, d, f, 0, 0, bad, w32, sid, hid)
    only0 = np.array([[-1, 0]] * T, dtype=np.int32)
    ref = ft.ft_cpu_experts(pool, E, k, d, f, 0, 0, ids, w32, only0, hid)
    assert np.array_equal(got, ref)


def test_single_expert_closed_form(lib):
    """One route, weight 1, a bf16 expert whose gate and up rows are unit
    vectors and whose down matrix is the identity: y = silu(x_a) * x_b placed
    at the rows the down matrix selects."""
    d, f, E, k = 256, 128, 2, 1
    bx = ftsynth.expert_bytes(d, f, 0)
    pool = np.zeros(E * bx, dtype=np.uint8)
    ex = pool[bx:2 * bx].view(np.uint16)  # expert 1
    one = 0x3F80  # bf16 1.0
    wg = ex[:f * d].reshape(f, d)
    wu = ex[f * d:2 * f * d].reshape(f, d)
    wd = ex[2 * f * d:].reshape(d, f)
    for i in range(f):
        wg[i, i] = one
        wu[i, i + 1] = one
        wd[i, i] = one
    x = ftsynth.normal_bf16(2, 6, 0, 0, d).reshape(1, d)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)[0]
    got = ft.ft_cpu_experts(pool, E, k, d, f, 0, 0, np.array([[1]], np.int32), np.array([[1.0]], np.float32),
                            np.array([[-1]], np.int32), x)
    want = np.zeros(d)
    want[:f] = xf[:f] / (1 + np.exp(-xf[:f])) * xf[1:f + 1]
    np.testing.assert_allclose(got[0], want, rtol=1e-6, atol=1e-7)


def test_argument_errors(lib):
    pool = np.zeros(16, dtype=np.uint8)
    ids = np.zeros((1, 1), np.int32)
    w = np.ones((1, 1), np.float32)
    hid = np.zeros((1, 256), np.uint16)
    with pytest.raises(ft.FtError) as ei:
        ft.ft_cpu_experts(pool, 1, 1, 250, 128, 0, 0, ids, w, ids, np.zeros((1, 250), np.uint16))
    assert ei.value.code == ft.FT_E_ARG
    with pytest.raises(ft.FtError) as ei:
        ft.ft_cpu_experts(pool, 1, 1, 256, 128, 2, 0, ids, w, ids, hid)
    assert ei.value.code == ft.FT_E_ARG
    with pytest.raises(ft.FtError) as ei:
        ft.ft_cpu_experts(pool, 1, 1, 256, 128, 0, 0, ids, w, ids, hid, threads=0)
    assert ei.value.code == ft.FT_E_ARG


def test_mxfp4_nan_scale_propagates(lib):
    """OCP MX v1.0: the e8m0 byte 255 is NaN; a route through a row group with
    that scale yields NaN in the executor as in the oracle, and other tokens
    stay finite."""
    E, k, d, f, T = 4, 1, 256, 128, 2
    bx = ftsynth.expert_bytes(d, f, 1)
    pool = ftsynth.make_pool(3, 1, E, d, f, 1, 0.05, threads=2)
    df = d * f
    pool[2 * bx + 3 * df // 2] = 255  # expert 2: first gate scale byte (row 0, group 0)
    ids = np.array([[2], [1]], np.int32)
    w = np.ones((T, k), np.float32)
    sid = np.full((T, k), -1, np.int32)
    hid = ftsynth.normal_bf16(4, 6, 0, 0, T * d).reshape(T, d)
    got = ft.ft_cpu_experts(pool, E, k, d, f, 1, 0, ids, w, sid, hid)
    ref = _oracle_cpu(pool, 0, E, 1, d, f, ids, w, hid, sid)
    assert np.isnan(got[0]).any() and np.isnan(ref[0]).any()
    assert np.isfinite(got[1]).all()
    assert oracle.max_rel_err(got[1:], ref[1:]) <= CPU_MAX_REL
