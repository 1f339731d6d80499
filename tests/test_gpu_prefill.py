"""GPU parity of the prefill path (full-layer buffers, dispatch, tcgen05 grouped
GEMMs, combine) against the oracle, through the C ABI.

Outputs within max relative error 2e-2 and normwise 5e-3 of the fp64 oracle
(the intermediate H is rounded to bf16 as the operand of the down GEMM);
routing ids bit-exact; the decode cache is never touched by prefill.
"""
import numpy as np
import pytest

import ftsynth
import oracle
from harness import check_output, make_model

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ft():
    from expert_cache_host_gb300 import build as ftbuild
    ftbuild.build()
    import expert_cache_host_gb300 as lib
    lib.load()
    return lib


def make_ctx(ft, model, T, buffers=2, S=4):
    cfg = ft.make_config(num_layers=model.L, num_experts=model.E, top_k=model.k, hidden=model.d, inter=model.f,
                         dtype=model.dtype, num_slots=S, k_max=4, t_max=1, prefill_buffers=buffers, prefill_t_max=T)
    return ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)


def prefill_layers(ft, ctx, model, T, layers, seed=0, partial=None, logits_fn=None, tokens=None):
    """Run ft_moe_forward(PREFILL) over `layers` in order; compare each layer
    with the oracle on the selected tokens (all if None)."""
    stream = torch.cuda.current_stream().cuda_stream
    worst = (0.0, 0.0)
    for l in layers:
        hid = ftsynth.prefill_hidden(seed, l, T, model.d, threads=8)
        lg = ftsynth.router_logits(hid, model.wr[l]) if logits_fn is None else logits_fn(l, hid)
        d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
        d_lg = torch.from_numpy(lg).cuda()
        out = torch.empty((T, model.d), dtype=torch.float32, device="cuda")
        d_part = None if partial is None else torch.from_numpy(partial).cuda()
        ft.ft_moe_forward(ctx, l, ft.FT_PREFILL_LAYER, d_lg.data_ptr(), d_hid.data_ptr(), T,
                          0 if d_part is None else d_part.data_ptr(), out.data_ptr(), stream)
        torch.cuda.synchronize()
        ids, w = oracle.route(lg, model.k)
        sel = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, dtype=np.int32)
        full, _, _ = oracle.moe_forward(model.layer_pool(l), model.bx, model.dtype, model.d, model.f, ids, w, hid, tokens=sel)
        if partial is not None:
            full = full + partial[sel].astype(np.float64)
        y = out.cpu().numpy()[sel].astype(np.float64)
        mr, nw = check_output(y, full, f"layer {l}")
        worst = (max(worst[0], mr), max(worst[1], nw))
    assert ft.ft_get_status(ctx) == 0
    return worst


def test_tiny_prefill_chunk(ft):
    """1 layer, d=256, E=16, top-2, f=128: one 64-token prefill chunk."""
    model = make_model(1, 16, 2, 256, 128, seed=0)
    ctx = make_ctx(ft, model, 64)
    prefill_layers(ft, ctx, model, 64, [0])
    ft.ft_moe_destroy(ctx)


def test_tiny_prefill_with_partial_and_ragged_tokens(ft):
    model = make_model(2, 16, 2, 256, 128, seed=1)
    T = 77
    ctx = make_ctx(ft, model, T)
    partial = ftsynth.test_partial(3, T, 256)
    prefill_layers(ft, ctx, model, T, [0, 1], partial=partial)
    ft.ft_moe_destroy(ctx)


@pytest.mark.parametrize("buffers", [2, 1])
def test_a3b_expert_shape_layers(ft, buffers):
    """d=2048, f=768, E=128, top-8 over 3 layers: segments of ~8-16 rows, some
    experts empty; single and double layer buffers give the same answers."""
    model = make_model(3, 128, 8, 2048, 768, seed=2)
    T = 200
    ctx = make_ctx(ft, model, T, buffers=buffers)
    prefill_layers(ft, ctx, model, T, [0, 1, 2], tokens=np.arange(0, T, 7))
    ft.ft_moe_destroy(ctx)


def test_skewed_routing_long_segments(ft):
    """Every token routes to the same k experts: segments of T rows, several
    128-row tiles plus a ragged one; the other experts are empty."""
    model = make_model(1, 32, 4, 512, 256, seed=3)
    T = 700

    def skew(l, hid):
        lg = ftsynth.router_logits(hid, model.wr[l])
        lg[:, [3, 9, 17, 30]] += 100.0
        return lg

    ctx = make_ctx(ft, model, T)
    prefill_layers(ft, ctx, model, T, [0], logits_fn=skew, tokens=np.arange(0, T, 5))
    ft.ft_moe_destroy(ctx)


def test_prefill_leaves_cache_untouched(ft):
    model = make_model(2, 16, 2, 256, 128, seed=4)
    ctx = make_ctx(ft, model, 64, S=5)
    before = ft.ft_get_table(ctx, 32, 5)
    prefill_layers(ft, ctx, model, 64, [0, 1, 0])
    after = ft.ft_get_table(ctx, 32, 5)
    for a, b in zip(before[:3], after[:3]):
        assert np.array_equal(a, b)
    assert before[3] == after[3] == 0
    ft.ft_moe_destroy(ctx)


def test_prefill_rejects_oversized_chunk(ft):
    model = make_model(1, 16, 2, 256, 128, seed=5)
    ctx = make_ctx(ft, model, 32)
    x = torch.zeros((64, 256), dtype=torch.int16, device="cuda")
    lg = torch.zeros((64, 16), dtype=torch.float32, device="cuda")
    out = torch.empty((64, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(ft.FtError) as ei:
        ft.ft_moe_forward(ctx, 0, ft.FT_PREFILL_LAYER, lg.data_ptr(), x.data_ptr(), 64, 0, out.data_ptr())
    assert ei.value.code == ft.FT_E_ARG
    ft.ft_moe_destroy(ctx)


# --- MXFP4 experts: codes and scales dequantised to bf16 in shared memory,
# --- then the same tcgen05 GEMMs (activations stay bf16)

def test_mxfp4_prefill_ragged_and_full_tiles(ft):
    """E = 8, top-2, d = f = 512, 700 tokens: ~175 rows per expert (one full
    128-row tile and a ragged one), two layers through the double buffer."""
    model = make_model(2, 8, 2, 512, 512, dtype=1, seed=6)
    T = 700
    ctx = make_ctx(ft, model, T)
    prefill_layers(ft, ctx, model, T, [0, 1], tokens=np.arange(0, T, 3))
    ft.ft_moe_destroy(ctx)


def test_mxfp4_prefill_skewed_long_segments_with_partial(ft):
    """Every token routes to the same 4 of 16 experts: segments of 600 rows
    (four full tiles and a ragged one), plus a caller partial sum."""
    model = make_model(1, 16, 4, 1024, 512, dtype=1, seed=7)
    T = 600

    def skew(l, hid):
        lg = ftsynth.router_logits(hid, model.wr[l])
        lg[:, [1, 6, 11, 15]] += 100.0
        return lg

    ctx = make_ctx(ft, model, T)
    partial = ftsynth.test_partial(8, T, 1024)
    prefill_layers(ft, ctx, model, T, [0], logits_fn=skew, partial=partial, tokens=np.arange(0, T, 4))
    ft.ft_moe_destroy(ctx)


def test_mxfp4_prefill_wide_scale_range(ft):
    """Scale bytes drawn uniformly from [100, 140] (2^-27 .. 2^13) for every
    (row, 32-element group): a scale read from the wrong row or group, or
    applied twice, moves the outputs far outside the tolerance."""
    model = make_model(1, 8, 2, 512, 512, dtype=1, seed=9)
    d, f, E, bx = model.d, model.f, model.E, model.bx
    rng = np.random.default_rng(1234)
    for e in range(E):
        base = e * bx + 3 * d * f // 2
        model.pool[base:base + 3 * d * f // 32] = rng.integers(100, 141, 3 * d * f // 32, dtype=np.uint8)
    T = 300
    ctx = make_ctx(ft, model, T)
    prefill_layers(ft, ctx, model, T, [0], tokens=np.arange(0, T, 2))
    ft.ft_moe_destroy(ctx)


def test_mxfp4_prefill_v4_expert_shape_8192_tokens(ft):
    """V4-Flash-style expert shape (E = 256, top-6, d = 4096, f = 2048, MXFP4),
    one 8192-token chunk: ~192 rows per expert (a full tile and a ragged
    one).  Compared with the oracle on the first and last routed token of 24
    experts plus a spread of others."""
    from concurrent.futures import ThreadPoolExecutor
    L, E, k, d, f, dt, T = 1, 256, 6, 4096, 2048, 1, 8192
    bx = ftsynth.expert_bytes(d, f, dt)
    hp = ft.HostPool(L * E * bx)
    ctx = None
    try:
        pool = ftsynth.make_pool(0, L, E, d, f, dt, out=hp.array)
        wr = ftsynth.router_weights(0, L, E, d)
        cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, dtype=dt, num_slots=1, k_max=1,
                             t_max=1, prefill_buffers=2, prefill_t_max=T)
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        st = torch.cuda.current_stream().cuda_stream
        hid = ftsynth.prefill_hidden(0, 0, T, d, threads=8)
        lg = ftsynth.router_logits(hid, wr[0])
        d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
        d_lg = torch.from_numpy(lg).cuda()
        out = torch.empty((T, d), dtype=torch.float32, device="cuda")
        ft.ft_moe_forward(ctx, 0, ft.FT_PREFILL_LAYER, d_lg.data_ptr(), d_hid.data_ptr(), T, 0, out.data_ptr(), st)
        torch.cuda.synchronize()
        assert ft.ft_get_status(ctx) == 0
        ids, w = oracle.route(lg, k)
        some = range(0, E, E // 24)
        first = [int(np.argmax((ids == e).any(1))) for e in some]
        last = [T - 1 - int(np.argmax((ids[::-1] == e).any(1))) for e in some]
        sel = np.unique(np.concatenate([first, last, np.arange(0, T, 1023), [T - 1]])).astype(np.int32)
        parts = np.array_split(sel, 8)
        with ThreadPoolExecutor(8) as ex:  # the oracle's C call runs without the GIL
            fulls = list(ex.map(lambda s: oracle.moe_forward(pool, bx, dt, d, f, ids, w, hid, tokens=s)[0], parts))
        check_output(out.cpu().numpy()[sel].astype(np.float64), np.concatenate(fulls), "V4 prefill")
    finally:
        if ctx is not None:
            ft.ft_moe_destroy(ctx)
        hp.free()
