"""The allocation-free decode entry point against the oracle and the context path.

ft_decode_experts_noalloc serves callers that cannot allocate device memory
when they run the step (a runtime with a fixed memory budget, a framework that
owns every buffer, code inside a global-mode stream capture).  It keeps its
scratch in a fixed array inside the library, so on the same slots, routes and
weights it must give the oracle's GPU-side sum plus the caller's partial, and
the same output as ft_moe_forward(FT_DECODE_CACHED) -- checked here on two
calls in a row, within the tolerances of the other tests.  A route whose slot
id is out of range must be reported and add nothing, even though the shared
scratch still holds an earlier call's partial sums.  This file is collected
last so a failure here stops a run only after every other test has run; it
also passes alone in a fresh process.
"""
import numpy as np
import pytest

import ftsynth
import oracle
from harness import MAX_REL, NORMWISE, check_output, dev_view, make_model

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ft():
    from expert_cache_host_gb300 import build as ftbuild
    ftbuild.build()
    import expert_cache_host_gb300 as lib
    lib.load()
    return lib


def _oracle_gpu_sum(model, cache, logits, hid, k, slot_override=None):
    """The oracle's route, cache step and GPU-side expert sum for one token.
    slot_override: {route index: slot id} applied to the oracle's slot ids
    (a route set to -1 is left out of the GPU sum)."""
    ids, w = oracle.route(logits, k)
    ref = cache.step(0, model.E, ids, 1, 1, 16) if cache is not None else None
    sid = ref.slot_ids.reshape(1, k).copy()
    for r, v in (slot_override or {}).items():
        sid[0, r] = v
    _, gpu, _ = oracle.moe_forward(model.layer_pool(0), model.bx, 0, model.d, model.f, ids, w, hid,
                                   slot_ids=np.where(sid >= 0, sid, -1).astype(np.int32))
    return ref, gpu


def test_noalloc_matches_oracle_and_context_path_two_calls(ft):
    L, E, k, d, f, S, T = 1, 32, 8, 2048, 768, 24, 1
    model = make_model(L, E, k, d, f, seed=11)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=16, t_max=T)
    ctx = ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)
    cache = oracle.Cache(L * E, S)
    try:
        hid = ftsynth.ar1_hidden(11, 0, 0, 2, d)
        logits = ftsynth.router_logits(hid, model.wr[0])
        d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
        d_lg = torch.from_numpy(logits).cuda()
        partial_np = ftsynth.test_partial(5, T, d)
        partial = torch.from_numpy(partial_np).cuda()
        st = torch.cuda.current_stream().cuda_stream
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        arena = ft.ft_slot_ptr(ctx, 0)
        for call, use_partial in enumerate((False, True)):
            res = ft.ft_cache_step(ctx, 0, d_lg[call].data_ptr(), T, st)
            ref = torch.empty((T, d), dtype=torch.float32, device="cuda")
            got = torch.full((T, d), float("nan"), dtype=torch.float32, device="cuda")
            p_ptr = partial.data_ptr() if use_partial else 0
            ft.ft_moe_forward(ctx, 0, ft.FT_DECODE_CACHED, 0, d_hid[call].data_ptr(), T, p_ptr, ref.data_ptr(), st)
            ft.ft_decode_experts_noalloc(arena, S, d, f, k, T, res.slot_ids, res.weights, d_hid[call].data_ptr(), p_ptr,
                                         got.data_ptr(), status.data_ptr(), st)
            torch.cuda.synchronize()
            y, r = got.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
            assert np.isfinite(y).all()
            # the oracle: same routes and slots (bit-exact), its fp64 GPU-side sum plus the partial
            oref, gpu = _oracle_gpu_sum(model, cache, logits[call:call + 1], hid[call:call + 1], k)
            sid = dev_view(res.slot_ids, (T * k,), "<i4").cpu().numpy()
            assert np.array_equal(sid, oref.slot_ids), f"call {call}: slot ids"
            want = gpu + (partial_np.astype(np.float64) if use_partial else 0.0)
            check_output(y, want, f"call {call} vs oracle")
            assert oracle.max_rel_err(y, r) <= MAX_REL and oracle.normwise_err(y, r) <= NORMWISE, f"call {call}"
            # every route of this token had a slot (all-fill at BP/BH = 1), so the expert sum was computed
            assert (sid >= 0).all()
        assert int(status.item()) == 0
        assert ft.ft_get_status(ctx) == 0
    finally:
        ft.ft_moe_destroy(ctx)


def test_noalloc_out_of_range_slot_adds_nothing(ft):
    """A call with valid slots fills the shared scratch; the next call names a
    slot id >= num_slots for one route: that route is reported
    (FT_ST_BAD_SLOT) and the output is the sum over the other routes."""
    L, E, k, d, f, S, T = 1, 32, 8, 2048, 768, 24, 1
    model = make_model(L, E, k, d, f, seed=12)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=16, t_max=T)
    ctx = ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)
    cache = oracle.Cache(L * E, S)
    try:
        hid = ftsynth.ar1_hidden(12, 0, 0, 1, d)
        logits = ftsynth.router_logits(hid, model.wr[0])
        d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
        d_lg = torch.from_numpy(logits).cuda()
        st = torch.cuda.current_stream().cuda_stream
        res = ft.ft_cache_step(ctx, 0, d_lg[0].data_ptr(), T, st)
        out = torch.empty((T, d), dtype=torch.float32, device="cuda")
        ft.ft_moe_forward(ctx, 0, ft.FT_DECODE_CACHED, 0, d_hid[0].data_ptr(), T, 0, out.data_ptr(), st)
        arena = ft.ft_slot_ptr(ctx, 0)
        sid = dev_view(res.slot_ids, (T * k,), "<i4").clone()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = torch.full((T, d), float("nan"), dtype=torch.float32, device="cuda")
        # first call: every slot valid (leaves partial sums for all k routes in the scratch)
        ft.ft_decode_experts_noalloc(arena, S, d, f, k, T, sid.data_ptr(), res.weights, d_hid[0].data_ptr(), 0,
                                     got.data_ptr(), status.data_ptr(), st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        bad = 3
        sid[bad] = S + 5
        ft.ft_decode_experts_noalloc(arena, S, d, f, k, T, sid.data_ptr(), res.weights, d_hid[0].data_ptr(), 0,
                                     got.data_ptr(), status.data_ptr(), st)
        torch.cuda.synchronize()
        assert int(status.item()) & ft.FT_ST_BAD_SLOT
        _, want = _oracle_gpu_sum(model, cache, logits[0:1], hid[0:1], k, slot_override={bad: -1})
        check_output(got.cpu().numpy().astype(np.float64), want, "out-of-range slot")
    finally:
        ft.ft_moe_destroy(ctx)


def test_noalloc_rejects_oversized_scratch(ft):
    x = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(ft.FtError) as ei:
        # 64 tokens x top-8 x 24 chunks x 2048 x 4 B = 100 MB > the fixed 8 MiB
        ft.ft_decode_experts_noalloc(x.data_ptr(), 4, 2048, 768, 8, 64, x.data_ptr(), x.data_ptr(), x.data_ptr(), 0,
                                     x.data_ptr())
    assert ei.value.code == ft.FT_E_ARG and "static scratch" in str(ei.value)
