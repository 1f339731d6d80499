"""GPU parity of the decode path against the oracle, through the C ABI.

Control state (routes, unique/hit/miss lists, fetch set, victims, evicted
experts, rewritten slot ids, the whole residency table and clock) must match
bit for bit after every step; expert outputs within max relative error 2e-2
and normwise 5e-3 of the fp64 oracle.
"""
import numpy as np
import pytest

import ftsynth
import oracle
from harness import (check_output, compare_step, compare_table, dev_view, make_model, step_to_host)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ft():
    from expert_cache_host_gb300 import build as ftbuild
    ftbuild.build()
    import expert_cache_host_gb300 as lib
    lib.load()
    return lib


# ------------------------------------------------------------------ routing

@pytest.mark.parametrize("T,E,k", [(1, 16, 2), (64, 128, 8), (100, 256, 6), (33, 1000, 32), (5, 7, 7)])
def test_route_parity(ft, T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    lg = ftsynth.test_logits(11, E, T, E)
    # plant ties and signed zeros
    lg[:, ::3] = np.round(lg[:, ::3] * 2) / 2
    lg[0, :min(E, 4)] = 0.0
    if E > 5:
        lg[0, 5] = -0.0
    ref_ids, ref_w = oracle.route(lg, k)
    d_lg = torch.from_numpy(lg).cuda()
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ft.ft_route(d_lg.data_ptr(), T, E, k, ids.data_ptr(), w.data_ptr(), st.data_ptr())
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-7)
    assert int(st.item()) == 0


def test_route_nan_sets_status(ft):
    lg = np.zeros((3, 16), dtype=np.float32)
    lg[1, 4] = np.nan
    d_lg = torch.from_numpy(lg).cuda()
    ids = torch.empty((3, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((3, 2), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ft.ft_route(d_lg.data_ptr(), 3, 16, 2, ids.data_ptr(), w.data_ptr(), st.data_ptr())
    torch.cuda.synchronize()
    assert int(st.item()) & ft.FT_ST_NAN


@pytest.mark.parametrize("T,E,k", [(1, 16, 2), (4, 64, 4), (16, 128, 8), (2, 1000, 32)])
def test_cache_step_routes_and_nan(ft, T, E, k):
    """Routing inside the control kernel (by rank for few tokens, a warp per
    token otherwise): ids bit-exact and weights equal to the oracle's on random
    logits with ties; a NaN logit sets FT_ST_NAN."""
    cfg = ft.make_config(num_layers=1, num_experts=E, top_k=k, hidden=256, inter=128, num_slots=4, k_max=4, t_max=T)
    pool = np.zeros(E * ftsynth.expert_bytes(256, 128, 0), dtype=np.uint8)
    ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
    try:
        rng = np.random.default_rng(E + T)
        lg = rng.integers(-8, 8, size=(T, E)).astype(np.float32) * 0.25  # many ties
        res = ft.ft_cache_step(ctx, 0, torch.from_numpy(lg).cuda().data_ptr(), T)
        torch.cuda.synchronize()
        ref_ids, ref_w = oracle.route(lg, k)
        g = step_to_host(res, T, k, E, 4)
        assert np.array_equal(g["ids"], ref_ids)
        np.testing.assert_allclose(g["w"], ref_w, rtol=2e-6, atol=1e-7)
        assert ft.ft_get_status(ctx, clear=True) == 0
        lg[T - 1, E // 2] = np.nan
        ft.ft_cache_step(ctx, 0, torch.from_numpy(lg).cuda().data_ptr(), T)
        torch.cuda.synchronize()
        assert ft.ft_get_status(ctx) & ft.FT_ST_NAN
    finally:
        ft.ft_moe_destroy(ctx)


# ------------------------------------------------------------------ decode steps

def run_decode(ft, model, S, K_max, r, steps, T=1, fill_mode=0, check_every=1, out_tokens=None, rho=0.9,
               rebuild_at=None, graph=False, r_at=None, fill_order=0, cpu_exec=0, decode_path=0, fill_ctas=0):
    """Decode `steps` steps over all layers through the library and the oracle
    side by side; compare control state every step and outputs every
    `check_every` steps.  r_at: {step: (r_num, r_den)} changes r (ft_set_ratio)
    before that step.  cpu_exec > 0: the context's CPU expert executor (that
    many threads) computes the CPU routes' partial sum; no partial is passed."""
    L, E, k, d, f = model.L, model.E, model.k, model.d, model.f
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, dtype=model.dtype, num_slots=S,
                         k_max=K_max, t_max=T, r_num=r[0], r_den=r[1], fill_mode=fill_mode, fill_order=fill_order,
                         decode_path=decode_path, fill_ctas=fill_ctas)
    ctx = ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)
    try:
        if fill_mode == 0 and (model.dtype == 0 or model.d % 512 == 0):
            assert ft.ft_decode_path(ctx) == decode_path
        if cpu_exec:
            ft.ft_cpu_executor(ctx, cpu_exec)
            check_every = 1
        cache = oracle.Cache(L * E, S)
        hid = np.stack([np.stack([ftsynth.ar1_hidden(model.seed, l, b, steps, d, rho) for b in range(T)], axis=1)
                        for l in range(L)], axis=1)  # [steps, L, T, d]
        logits = np.stack([ftsynth.router_logits(hid[:, l], model.wr[l]) for l in range(L)], axis=1)  # [steps,L,T,E]
        d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
        d_lg = torch.from_numpy(logits).cuda()
        out = torch.empty((T, d), dtype=torch.float32, device="cuda")
        partial = torch.empty((T, d), dtype=torch.float32, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        worst = (0.0, 0.0)
        for s in range(steps):
            if r_at and s in r_at:
                r = r_at[s]
                ft.ft_set_ratio(ctx, r[0], r[1], stream)
            if rebuild_at is not None and s == rebuild_at[0]:
                if len(rebuild_at) > 2 and rebuild_at[2] == "retain":
                    ft.ft_cache_rebuild_retain(ctx, rebuild_at[1])
                    cache = cache.rebuild_retain(rebuild_at[1])
                else:
                    ft.ft_cache_rebuild(ctx, rebuild_at[1])
                    cache = oracle.Cache(L * E, rebuild_at[1])
                S = rebuild_at[1]
                compare_table(ft, ctx, cache, f"after the rebuild at step {s}")
            for l in range(L):
                res = ft.ft_cache_step(ctx, l, d_lg[s, l].data_ptr(), T, stream)
                ref_ids, ref_w = oracle.route(logits[s, l], k)
                ref = cache.step(l, E, ref_ids, r[0], r[1], K_max, fill_order=fill_order)
                torch.cuda.synchronize()
                g = step_to_host(res, T, k, E, K_max)
                where = f"step {s} layer {l}"
                assert np.array_equal(g["ids"], ref_ids), where
                np.testing.assert_allclose(g["w"], ref_w, rtol=2e-6, atol=1e-7)
                compare_step(g, ref, where)
                check = (s % check_every == 0)
                if check:
                    full, gpu_part, cpu_part = oracle.moe_forward(model.layer_pool(l), model.bx, model.dtype, d, f,
                                                                  ref_ids, ref_w, hid[s, l],
                                                                  slot_ids=ref.slot_ids.reshape(T, k))
                    partial.copy_(torch.from_numpy(cpu_part.astype(np.float32)))
                else:
                    partial.zero_()
                ft.ft_moe_forward(ctx, l, ft.FT_DECODE_CACHED, 0, d_hid[s, l].data_ptr(), T,
                                  0 if cpu_exec else partial.data_ptr(), out.data_ptr(), stream)
                torch.cuda.synchronize()
                if check:
                    y = out.cpu().numpy().astype(np.float64)
                    mr, nw = check_output(y, full, where)
                    worst = (max(worst[0], mr), max(worst[1], nw))
            compare_table(ft, ctx, cache, f"after step {s}")
        assert ft.ft_get_status(ctx) == 0
        return ctx, cache, worst
    except Exception:
        ft.ft_moe_destroy(ctx)
        raise


def test_tiny_decode_all_fill(ft):
    """1 layer, d=256, E=16, top-2, f=128, 8 slots, BP/BH = 1, 32 steps."""
    model = make_model(1, 16, 2, 256, 128, seed=0)
    ctx, cache, worst = run_decode(ft, model, S=8, K_max=16, r=(1, 1), steps=32)
    cnt = ft.ft_get_counters(ctx, 1)
    assert cnt[0, 5] == 32 and cnt[0, 3] == 0  # all misses filled at r = 1
    ft.ft_moe_destroy(ctx)


PATHS = [0, 1]  # FT_DECODE_FUSED, FT_DECODE_SPLIT


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("r,K_max", [((1, 2), 16), ((1, 1), 1), ((0, 1), 4)])
def test_tiny_decode_cpu_split(ft, r, K_max, path):
    """Misses left to the CPU arrive as an external partial sum and merge exactly."""
    model = make_model(2, 16, 2, 256, 128, seed=1)
    ctx, cache, worst = run_decode(ft, model, S=6, K_max=K_max, r=r, steps=20, decode_path=path)
    cnt = ft.ft_get_counters(ctx, 2)
    assert cnt[:, 3].sum() > 0  # some routes did go to the CPU
    ft.ft_moe_destroy(ctx)


def test_ratio_changes_at_run_time(ft):
    """ft_set_ratio between steps: the fill/CPU split follows the new r from
    the next step on (all-fill, half, none, 2x), against the oracle run with
    the same r per step."""
    model = make_model(2, 16, 2, 256, 128, seed=8)
    ctx, _, _ = run_decode(ft, model, S=6, K_max=16, r=(1, 1), steps=10,
                           r_at={2: (1, 2), 4: (0, 1), 6: (2, 1), 8: (3, 4)})
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("r,K_max", [((1, 2), 16), ((1, 1), 2), ((1, 3), 8)])
def test_fill_order_most_routed(ft, r, K_max):
    """FT_FILL_ORDER_MOST_ROUTED with several tokens per step (route counts
    differ): control state bit-exact and outputs against the oracle run with
    the same fill order, while q < m (r < 1, or K_max below the misses)."""
    model = make_model(2, 16, 3, 256, 128, seed=12)
    ctx, _, _ = run_decode(ft, model, S=8, K_max=K_max, r=r, steps=8, T=4, fill_order=ft.FT_FILL_ORDER_MOST_ROUTED)
    ft.ft_moe_destroy(ctx)


def test_tiny_decode_copy_engine_fill(ft):
    model = make_model(2, 16, 2, 256, 128, seed=2)
    ctx, _, _ = run_decode(ft, model, S=5, K_max=16, r=(1, 1), steps=12, fill_mode=ft.FT_FILL_COPY_ENGINE)
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("path", PATHS)
def test_batch16_decode_groups(ft, path):
    """16 tokens per step: tokens share experts, so groups hold several routes."""
    model = make_model(2, 16, 4, 256, 256, seed=3)
    ctx, _, _ = run_decode(ft, model, S=12, K_max=8, r=(1, 1), steps=6, T=16, decode_path=path)
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("d,f,T,k", [(512, 256, 1, 2), (1024, 128, 16, 4), (768, 128, 4, 2), (2048, 128, 16, 8),
                                     (8192, 128, 2, 2)])
def test_decode_shapes(ft, d, f, T, k, path):
    """Hidden sizes of 2, 3, 4, 8 and 32 column blocks, f of 4 to 8 chunks, and
    T = 16, which puts several token batches through one CTA."""
    model = make_model(2, 16, k, d, f, seed=7 + d)
    ctx, _, _ = run_decode(ft, model, S=max(6, 2 * k), K_max=16, r=(1, 1), steps=5, T=T, decode_path=path)
    ft.ft_moe_destroy(ctx)


def test_rebuild_mid_run(ft):
    """A rebuild at a safe point resets the cache cold at the new size; the
    results stay equal to a fresh oracle cache of that size."""
    model = make_model(2, 16, 2, 256, 128, seed=4)
    ctx, cache, _ = run_decode(ft, model, S=8, K_max=16, r=(1, 1), steps=10, rebuild_at=(5, 3))
    assert ft.ft_get_epoch(ctx) == 1 and ft.ft_num_slots(ctx) == 3
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("new_S", [3, 12, 20])
def test_rebuild_retain_mid_run(ft, new_S):
    """ft_cache_rebuild_retain: the most recently used residents stay (fewer,
    equal or more slots); the table equals the oracle's retaining rebuild and
    the steps after it (hits on the kept experts, whose bytes moved to new
    slots) keep matching the oracle."""
    model = make_model(2, 16, 2, 256, 128, seed=13)
    ctx, cache, _ = run_decode(ft, model, S=8, K_max=16, r=(1, 1), steps=12, rebuild_at=(6, new_S, "retain"))
    assert ft.ft_get_epoch(ctx) == 1 and ft.ft_num_slots(ctx) == new_S
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("path,fill_ctas", [(0, 0), (0, 1), (0, 150), (1, 0)])
def test_ragged_shapes_and_larger_model(ft, path, fill_ctas):
    """d=2048, f=768 (24 chunks), E=128, top-8: the A3B expert shape, 3 layers;
    the fused path with the default number of fill CTAs, with one, and with
    all but one or two of the grid."""
    model = make_model(3, 128, 8, 2048, 768, seed=5)
    ctx, _, worst = run_decode(ft, model, S=20, K_max=128, r=(1, 2), steps=4, decode_path=path, fill_ctas=fill_ctas)
    ft.ft_moe_destroy(ctx)


# ------------------------------------------------------------------ control alone

@pytest.mark.parametrize("S,K_max,r,s_zipf,T", [(64, 64, (1, 1), 1.2, 64), (40, 8, (1, 2), 0.6, 64),
                                                  (300, 512, (1, 1), 0.6, 64), (6144, 128, (1, 1), 1.2, 64),
                                                  (64, 64, (1, 1), 0.6, 16), (300, 128, (1, 1), 1.2, 16),
                                                  (40, 8, (1, 1), 0.6, 1)])
def test_control_zipf_stress_small(ft, S, K_max, r, s_zipf, T):
    """The control kernel alone on Zipf route streams: T tokens x top-8 x E=128
    (64 tokens take the full block, 16 and 1 the half block; both victim
    searches, block arg-min rounds for q <= 4 and radix select above, run)."""
    L, E, k, steps = 4, 128, 8, 25
    d, f = 256, 128  # the control path never reads expert bytes: smallest legal expert shape
    bx = ftsynth.expert_bytes(d, f, 0)
    pool = np.zeros(L * E * bx, dtype=np.uint8)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=K_max,
                         t_max=T, r_num=r[0], r_den=r[1])
    ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
    routes = np.stack([ftsynth.zipf_routes(0, l, E, T, k, s_zipf, 0, steps, threads=4) for l in range(L)], axis=1)
    d_routes = torch.from_numpy(routes).cuda()
    cache = oracle.Cache(L * E, S)
    stream = torch.cuda.current_stream().cuda_stream
    for s in range(steps):
        for l in range(L):
            res = ft.ft_cache_control(ctx, l, d_routes[s, l].data_ptr(), T, stream)
            ref = cache.step(l, E, routes[s, l], r[0], r[1], K_max)
            torch.cuda.synchronize()
            compare_step(step_to_host(res, T, k, E, K_max), ref, f"step {s} layer {l}")
        compare_table(ft, ctx, cache, f"after step {s}")
    assert ft.ft_get_status(ctx) == 0
    ft.ft_moe_destroy(ctx)


def test_control_out_of_range_route_sets_status(ft):
    L, E, k, T, S = 1, 16, 2, 2, 4
    d, f = 256, 128
    pool = np.zeros(L * E * ftsynth.expert_bytes(d, f, 0), dtype=np.uint8)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, t_max=T)
    ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
    ids = torch.tensor([[1, 99], [2, 3]], dtype=torch.int32, device="cuda")
    res = ft.ft_cache_control(ctx, 0, ids.data_ptr(), T, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    g = step_to_host(res, T, k, E, 16)
    assert ft.ft_get_status(ctx, clear=True) & ft.FT_ST_ROUTE_RANGE
    assert g["slot_ids"][0, 1] == -1 and g["counts"][0] == 3  # the bad route is treated as absent
    assert ft.ft_get_status(ctx) == 0
    ft.ft_moe_destroy(ctx)


def test_forward_without_step_is_rejected(ft):
    model = make_model(1, 16, 2, 256, 128, seed=6)
    cfg = ft.make_config(num_layers=1, num_experts=16, top_k=2, hidden=256, inter=128, num_slots=4)
    ctx = ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)
    out = torch.empty((1, 256), dtype=torch.float32, device="cuda")
    hid = torch.zeros((1, 256), dtype=torch.int16, device="cuda")
    with pytest.raises(ft.FtError) as ei:
        ft.ft_moe_forward(ctx, 0, ft.FT_DECODE_CACHED, 0, hid.data_ptr(), 1, 0, out.data_ptr())
    assert ei.value.code == ft.FT_E_STATE
    with pytest.raises(ft.FtError):
        ft.ft_cache_step(ctx, 3, hid.data_ptr(), 1)  # bad layer
    ft.ft_moe_destroy(ctx)


# ------------------------------------------------------------------ MXFP4 experts

@pytest.mark.parametrize("path", PATHS)
def test_mxfp4_decode_small(ft, path):
    """MXFP4 experts (e2m1 codes uniform over all 16 values, e8m0 scales 119..121)."""
    model = make_model(2, 16, 2, 512, 128, dtype=1, seed=21)
    ctx, _, worst = run_decode(ft, model, S=6, K_max=16, r=(1, 1), steps=10, decode_path=path)
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("path", PATHS)
def test_mxfp4_decode_batch16_groups(ft, path):
    """16 tokens per step, top-6: groups of several routes share one pass over the weights."""
    model = make_model(1, 32, 6, 1024, 256, dtype=1, seed=22)
    ctx, _, worst = run_decode(ft, model, S=40, K_max=64, r=(1, 2), steps=4, T=16, decode_path=path)
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("path", PATHS)
def test_mxfp4_decode_v4_expert_shape(ft, path):
    """d=4096, f=2048 (the V4-Flash-style expert), top-6 of 16 experts, 3 steps."""
    model = make_model(1, 16, 6, 4096, 2048, dtype=1, seed=23)
    ctx, _, worst = run_decode(ft, model, S=8, K_max=16, r=(1, 1), steps=3, decode_path=path)
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("path", PATHS)
def test_mxfp4_decode_cpu_split(ft, path):
    """r = 1/2: half of the misses arrive as the oracle's CPU partial sum and
    merge exactly; MXFP4 experts, several tokens per step."""
    model = make_model(2, 16, 4, 512, 256, dtype=1, seed=25)
    ctx, _, _ = run_decode(ft, model, S=8, K_max=16, r=(1, 2), steps=8, T=4, decode_path=path)
    cnt = ft.ft_get_counters(ctx, 2)
    assert cnt[:, 3].sum() > 0  # some routes did go to the CPU
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", [1, 4])
def test_mxfp4_decode_wide_scale_range(ft, path, T):
    """Scale bytes drawn uniformly from [100, 140] for every (row, 32-element
    group) of every matrix: the gate/up scales the kernels stage per chunk and
    the down scales they read per row must pair with the right codes."""
    model = make_model(2, 16, 2, 1024, 256, dtype=1, seed=26)
    d, f, bx = model.d, model.f, model.bx
    rng = np.random.default_rng(77)
    for e in range(model.L * model.E):
        base = e * bx + 3 * d * f // 2
        model.pool[base:base + 3 * d * f // 32] = rng.integers(100, 141, 3 * d * f // 32, dtype=np.uint8)
    ctx, _, _ = run_decode(ft, model, S=6, K_max=16, r=(1, 1), steps=5, T=T, decode_path=path)
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("d,f,T", [(1536, 256, 1), (1536, 256, 16), (8192, 128, 2)])
def test_mxfp4_decode_shapes(ft, path, d, f, T):
    """An odd number of 256-byte column blocks per gate row (d = 1536: a
    half-filled last gate/up stage and down stage) and the largest hidden size
    of the fused kernel (d = 8192)."""
    model = make_model(2, 16, 4, d, f, dtype=1, seed=27 + d)
    ctx, _, _ = run_decode(ft, model, S=10, K_max=16, r=(1, 1), steps=4, T=T, decode_path=path)
    ft.ft_moe_destroy(ctx)


def test_mxfp4_rebuild_retain_fused(ft):
    """A retaining rebuild mid-run on the fused MXFP4 path: the kept experts'
    bytes move to new slots and the steps after it hit on them."""
    model = make_model(2, 16, 2, 512, 128, dtype=1, seed=28)
    ctx, _, _ = run_decode(ft, model, S=8, K_max=16, r=(1, 1), steps=10, rebuild_at=(5, 6, "retain"))
    assert ft.ft_get_epoch(ctx) == 1 and ft.ft_num_slots(ctx) == 6
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("fill_ctas", [1, 150])
def test_mxfp4_decode_fused_fill_ctas(ft, fill_ctas):
    """Fused MXFP4 path with one fill CTA (every installed item waits on a long
    fill) and with all but two CTAs filling; steps that hit and fill."""
    model = make_model(2, 32, 6, 1024, 512, dtype=1, seed=24)
    ctx, _, worst = run_decode(ft, model, S=20, K_max=64, r=(1, 1), steps=6, fill_ctas=fill_ctas)
    ft.ft_moe_destroy(ctx)


# ------------------------------------------------------------------ mixed hit / fill steps

@pytest.mark.parametrize("path", PATHS)
def test_mixed_steps_a3b_expert_shape(ft, path):
    """A3B expert shape over steps that both hit and fill: the resident experts
    stream from HBM through the TMA ring while the fill shares the GPU (split
    path: the same SMs; fused path: installed experts start as soon as their
    own bytes are in the slot), and every slot's bytes equal the pool's."""
    model = make_model(2, 128, 8, 2048, 768, seed=32)
    ctx, cache, _ = run_decode(ft, model, S=20, K_max=128, r=(1, 1), steps=6, decode_path=path)
    if path == 0:
        m = ft.ft_decode_meters(ctx)
        assert m["fill_launches"] > 0 and m["fill_bytes"] > 0 and m["fill_s"] > 0
        assert m["resident_launches"] > 0 and m["resident_bytes"] > 0 and m["resident_s"] > 0
    so, eo, lu, now = ft.ft_get_table(ctx, 256, 20)
    bx = model.bx
    for s in range(20):
        if eo[s] >= 0:
            got = dev_view(ft.ft_slot_ptr(ctx, s), (bx,), "|u1").cpu().numpy()
            assert np.array_equal(got, model.pool[int(eo[s]) * bx:(int(eo[s]) + 1) * bx]), f"slot {s}"
    ft.ft_moe_destroy(ctx)


# ------------------------------------------------------------------ pool in memory pinned before the write

def test_decode_from_host_alloc_pool(ft):
    """A pool written into ft_host_alloc memory is used as is (no registration)
    and gives the same answers; the memory outlives the context."""
    from harness import Model
    L, E, k, d, f = 2, 16, 2, 256, 128
    hp = ft.HostPool(L * E * ftsynth.expert_bytes(d, f, 0))
    try:
        pool = ftsynth.make_pool(41, L, E, d, f, 0, out=hp.array)
        model = Model(L, E, k, d, f, 0, pool, ftsynth.router_weights(41, L, E, d, 0.02), 41)
        ctx, _, _ = run_decode(ft, model, S=6, K_max=16, r=(1, 1), steps=6)
        ft.ft_moe_destroy(ctx)
        assert np.array_equal(hp.array[:64], ftsynth.make_pool(41, L, E, d, f, 0)[:64])  # still mapped and intact
    finally:
        hp.free()  # nothing above holds the context any more


# ------------------------------------------------------------------ CUDA graph replay

@pytest.mark.parametrize("path", PATHS)
def test_graph_replay_matches_oracle(ft, path):
    """One decode step of every layer captured once as a CUDA graph and
    replayed with new inputs: control state and outputs equal the oracle's at
    every replay; an ft_set_ratio between replays is seen by the graph (the
    fused path is a cooperative kernel node)."""
    L, E, k, d, f, T, S, K_max = 2, 16, 2, 256, 128, 1, 6, 16
    model = make_model(L, E, k, d, f, seed=9)
    steps, r = 8, (1, 1)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=K_max, t_max=T,
                         r_num=r[0], r_den=r[1], decode_path=path)
    ctx = ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)
    try:
        cache = oracle.Cache(L * E, S)
        hid = np.stack([ftsynth.ar1_hidden(model.seed, l, 0, steps, d)[:, None, :] for l in range(L)], axis=1)
        logits = np.stack([ftsynth.router_logits(hid[:, l], model.wr[l]) for l in range(L)], axis=1)
        cur_hid = torch.empty((L, T, d), dtype=torch.int16, device="cuda")
        cur_lg = torch.empty((L, T, E), dtype=torch.float32, device="cuda")
        partial = torch.zeros((L, T, d), dtype=torch.float32, device="cuda")
        out = torch.empty((L, T, d), dtype=torch.float32, device="cuda")
        stream = torch.cuda.Stream()
        res = [None] * L

        def step(st):
            for l in range(L):
                res[l] = ft.ft_cache_step(ctx, l, cur_lg[l].data_ptr(), T, st)
                ft.ft_moe_forward(ctx, l, ft.FT_DECODE_CACHED, 0, cur_hid[l].data_ptr(), T, partial[l].data_ptr(),
                                  out[l].data_ptr(), st)

        graph = None
        with torch.cuda.stream(stream):
            for s in range(steps):
                if s == 5:
                    r = (1, 2)
                    ft.ft_set_ratio(ctx, r[0], r[1], stream.cuda_stream)
                refs, fulls = [], []
                for l in range(L):  # oracle first: its CPU part is an input of the step
                    ids, w = oracle.route(logits[s, l], k)
                    ref = cache.step(l, E, ids, r[0], r[1], K_max)
                    full, _, cpu_part = oracle.moe_forward(model.layer_pool(l), model.bx, 0, d, f, ids, w, hid[s, l],
                                                           slot_ids=ref.slot_ids.reshape(T, k))
                    partial[l].copy_(torch.from_numpy(cpu_part.astype(np.float32)))
                    refs.append((ids, ref))
                    fulls.append(full)
                cur_hid.copy_(torch.from_numpy(hid[s].view(np.int16)))
                cur_lg.copy_(torch.from_numpy(logits[s]))
                if s == 0:
                    step(stream.cuda_stream)  # eager: kernel attributes are set outside the capture
                else:
                    if graph is None:
                        graph = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(graph, stream=stream):
                            step(torch.cuda.current_stream().cuda_stream)
                    graph.replay()
                stream.synchronize()
                for l in range(L):
                    g = step_to_host(res[l], T, k, E, K_max)
                    assert np.array_equal(g["ids"], refs[l][0]), f"step {s} layer {l}"
                    compare_step(g, refs[l][1], f"step {s} layer {l}")
                    check_output(out[l].cpu().numpy().astype(np.float64), fulls[l], f"step {s} layer {l}")
                compare_table(ft, ctx, cache, f"after step {s}")
        assert ft.ft_get_status(ctx) == 0
    finally:
        ft.ft_moe_destroy(ctx)


# ------------------------------------------------------------------ CPU expert executor

@pytest.mark.parametrize("dtype,d,f,r,K_max", [(0, 256, 128, (1, 2), 16), (0, 256, 128, (0, 1), 4),
                                               (1, 512, 128, (1, 2), 16)])
def test_cpu_executor_decode_split(ft, dtype, d, f, r, K_max):
    """The misses left to the CPU run on the context's CPU expert executor
    (host function in the stream order) instead of arriving as a partial sum:
    outputs equal the oracle's full sum (GPU routes + CPU routes) every step,
    control state bit-exact."""
    model = make_model(2, 16, 2, d, f, dtype=dtype, seed=21)
    ctx, _, worst = run_decode(ft, model, S=6, K_max=K_max, r=r, steps=12, cpu_exec=3)
    try:
        cnt = ft.ft_get_counters(ctx, 2)
        assert cnt[:, 3].sum() > 0  # some routes did go to the CPU
        prof = ft.ft_profile_read(ctx, reset=True)
        assert set(prof) >= {"cpu"}
    finally:
        ft.ft_moe_destroy(ctx)


def test_cpu_executor_batch_and_profile(ft):
    """Four tokens per step (several CPU routes per token), the executor's
    stream profiled under ft_profile_enable."""
    model = make_model(2, 16, 3, 256, 128, seed=22)
    ctx, _, _ = run_decode(ft, model, S=8, K_max=8, r=(1, 3), steps=6, T=4, cpu_exec=2)
    try:
        ft.ft_profile_enable(ctx, 1)
        hid = torch.zeros((4, 256), dtype=torch.int16, device="cuda")
        lg = torch.zeros((4, 16), dtype=torch.float32, device="cuda")
        out = torch.empty((4, 256), dtype=torch.float32, device="cuda")
        ft.ft_cache_step(ctx, 0, lg.data_ptr(), 4)
        ft.ft_moe_forward(ctx, 0, ft.FT_DECODE_CACHED, 0, hid.data_ptr(), 4, 0, out.data_ptr(), 0)
        prof = ft.ft_profile_read(ctx, reset=True)
        assert prof["cpu"][1] == 1 and prof["cpu"][0] > 0
        assert np.isfinite(out.cpu().numpy()).all()
    finally:
        ft.ft_moe_destroy(ctx)


def test_cpu_executor_rejects_partial_and_disables(ft):
    model = make_model(1, 16, 2, 256, 128, seed=23)
    cfg = ft.make_config(num_layers=1, num_experts=16, top_k=2, hidden=256, inter=128, num_slots=4, k_max=4, t_max=1,
                         r_num=1, r_den=2)
    ctx = ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)
    try:
        ft.ft_cpu_executor(ctx, 2)
        hid = torch.zeros((1, 256), dtype=torch.int16, device="cuda")
        lg = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
        part = torch.zeros((1, 256), dtype=torch.float32, device="cuda")
        out = torch.empty((1, 256), dtype=torch.float32, device="cuda")
        ft.ft_cache_step(ctx, 0, lg.data_ptr(), 1)
        with pytest.raises(ft.FtError) as ei:
            ft.ft_moe_forward(ctx, 0, ft.FT_DECODE_CACHED, 0, hid.data_ptr(), 1, part.data_ptr(), out.data_ptr(), 0)
        assert ei.value.code == ft.FT_E_ARG
        ft.ft_cpu_executor(ctx, 0)  # off again: the caller's partial is accepted
        ft.ft_moe_forward(ctx, 0, ft.FT_DECODE_CACHED, 0, hid.data_ptr(), 1, part.data_ptr(), out.data_ptr(), 0)
        torch.cuda.synchronize()
        with pytest.raises(ft.FtError):
            ft.ft_cpu_executor(ctx, -1)
    finally:
        ft.ft_moe_destroy(ctx)


def test_cpu_executor_graph_replay(ft):
    """A token of every layer captured once as a CUDA graph with the executor
    on (copies and the host function become graph nodes) and replayed with new
    inputs: outputs equal the oracle's full sum at every replay."""
    L, E, k, d, f, T, S, K_max = 2, 16, 2, 256, 128, 1, 5, 16
    model = make_model(L, E, k, d, f, seed=24)
    steps, r = 8, (1, 2)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=K_max, t_max=T,
                         r_num=r[0], r_den=r[1])
    ctx = ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)
    try:
        ft.ft_cpu_executor(ctx, 2)
        cache = oracle.Cache(L * E, S)
        hid = np.stack([ftsynth.ar1_hidden(model.seed, l, 0, steps, d)[:, None, :] for l in range(L)], axis=1)
        logits = np.stack([ftsynth.router_logits(hid[:, l], model.wr[l]) for l in range(L)], axis=1)
        cur_hid = torch.empty((L, T, d), dtype=torch.int16, device="cuda")
        cur_lg = torch.empty((L, T, E), dtype=torch.float32, device="cuda")
        out = torch.empty((L, T, d), dtype=torch.float32, device="cuda")
        stream = torch.cuda.Stream()
        cpu_routes = 0

        def step(st):
            for l in range(L):
                ft.ft_cache_step(ctx, l, cur_lg[l].data_ptr(), T, st)
                ft.ft_moe_forward(ctx, l, ft.FT_DECODE_CACHED, 0, cur_hid[l].data_ptr(), T, 0, out[l].data_ptr(), st)

        graph = None
        with torch.cuda.stream(stream):
            for s in range(steps):
                fulls = []
                for l in range(L):
                    ids, w = oracle.route(logits[s, l], k)
                    ref = cache.step(l, E, ids, r[0], r[1], K_max)
                    cpu_routes += int((ref.slot_ids < 0).sum())
                    full, _, _ = oracle.moe_forward(model.layer_pool(l), model.bx, 0, d, f, ids, w, hid[s, l],
                                                    slot_ids=ref.slot_ids.reshape(T, k))
                    fulls.append(full)
                cur_hid.copy_(torch.from_numpy(hid[s].view(np.int16)))
                cur_lg.copy_(torch.from_numpy(logits[s]))
                if s == 0:
                    step(stream.cuda_stream)
                else:
                    if graph is None:
                        graph = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(graph, stream=stream):
                            step(torch.cuda.current_stream().cuda_stream)
                    graph.replay()
                stream.synchronize()
                for l in range(L):
                    check_output(out[l].cpu().numpy().astype(np.float64), fulls[l], f"step {s} layer {l}")
                compare_table(ft, ctx, cache, f"after step {s}")
        assert cpu_routes > 0
        assert ft.ft_get_status(ctx) == 0
    finally:
        ft.ft_moe_destroy(ctx)


def test_cpu_executor_with_caller_routes(ft):
    """ft_cache_control steps (routes from the caller, read in place; weights
    written by the caller into out->weights) with the executor on: the route
    arrays are not adjacent, so they reach the host by separate copies; the
    outputs equal the oracle's full sum."""
    L, E, k, d, f, T, S, K_max, steps, r = 2, 16, 2, 256, 128, 3, 6, 16, 8, (1, 2)
    model = make_model(L, E, k, d, f, seed=25)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=K_max, t_max=T,
                         r_num=r[0], r_den=r[1])
    ctx = ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)
    try:
        ft.ft_cpu_executor(ctx, 3)
        cache = oracle.Cache(L * E, S)
        hid = np.stack([np.stack([ftsynth.ar1_hidden(model.seed, l, b, steps, d) for b in range(T)], axis=1)
                        for l in range(L)], axis=1)  # [steps, L, T, d]
        logits = np.stack([ftsynth.router_logits(hid[:, l], model.wr[l]) for l in range(L)], axis=1)
        d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
        ids_dev = torch.empty((T, k), dtype=torch.int32, device="cuda")
        out = torch.empty((T, d), dtype=torch.float32, device="cuda")
        cpu_routes = 0
        for s in range(steps):
            for l in range(L):
                ids, w = oracle.route(logits[s, l], k)
                ids_dev.copy_(torch.from_numpy(ids))
                res = ft.ft_cache_control(ctx, l, ids_dev.data_ptr(), T)
                dev_view(res.weights, (T * k,), "<f4").copy_(torch.from_numpy(w.astype(np.float32).reshape(-1)))
                ref = cache.step(l, E, ids, r[0], r[1], K_max)
                cpu_routes += int((ref.slot_ids < 0).sum())
                full, _, _ = oracle.moe_forward(model.layer_pool(l), model.bx, 0, d, f, ids,
                                                w.astype(np.float32).astype(np.float64), hid[s, l],
                                                slot_ids=ref.slot_ids.reshape(T, k))
                ft.ft_moe_forward(ctx, l, ft.FT_DECODE_CACHED, 0, d_hid[s, l].data_ptr(), T, 0, out.data_ptr())
                torch.cuda.synchronize()
                check_output(out.cpu().numpy().astype(np.float64), full, f"step {s} layer {l}")
        assert cpu_routes > 0
        assert ft.ft_get_status(ctx) == 0
    finally:
        ft.ft_moe_destroy(ctx)
