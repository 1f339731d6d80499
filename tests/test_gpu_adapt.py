"""Run-time r = BP/BH on the GPU: the context measures the fill kernel's link
rate (BP) and the CPU expert executor's rate (BH); ft_adapt_ratio turns them
into r between decode steps.  The measured values are not deterministic, so
the test records the r in effect at every step and has the oracle replay the
cache with that same r sequence: the control state must agree bit-exactly
and the outputs (GPU routes + CPU routes) must match the oracle's full sum,
in eager steps and in CUDA-graph replays that pick up the new r from device
memory."""
import numpy as np
import pytest

import ftsynth
import oracle
from harness import check_output, compare_step, compare_table, make_model, step_to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ft():
    from expert_cache_host_gb300 import build as ftbuild
    ftbuild.build()
    import expert_cache_host_gb300 as lib
    lib.load()
    return lib


@pytest.mark.parametrize("dtype,d", [(0, 256), (1, 512)])
def test_adaptive_ratio_follows_oracle_with_the_same_r_sequence(ft, dtype, d):
    """bf16 and MXFP4 experts (the fused decode path, the CPU expert executor
    and a graph captured before r changes)."""
    L, E, k, f, T, S, K_max = 2, 16, 2, 128, 1, 5, 16
    model = make_model(L, E, k, d, f, dtype=dtype, seed=31)
    steps, r = 16, (1, 2)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, dtype=dtype, num_slots=S,
                         k_max=K_max, t_max=T, r_num=r[0], r_den=r[1])
    ctx = ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)
    try:
        ft.ft_cpu_executor(ctx, 2)
        a = ft.ft_ratio_adapter_init(0.5, 256, 256 * 64)
        cache = oracle.Cache(L * E, S)
        hid = np.stack([ftsynth.ar1_hidden(model.seed, l, 0, steps, d)[:, None, :] for l in range(L)], axis=1)
        logits = np.stack([ftsynth.router_logits(hid[:, l], model.wr[l]) for l in range(L)], axis=1)
        cur_hid = torch.empty((L, T, d), dtype=torch.int16, device="cuda")
        cur_lg = torch.empty((L, T, E), dtype=torch.float32, device="cuda")
        out = torch.empty((L, T, d), dtype=torch.float32, device="cuda")
        stream = torch.cuda.Stream()
        res = [None] * L
        r_seq, samples = [], []

        def step(st):
            for l in range(L):
                res[l] = ft.ft_cache_step(ctx, l, cur_lg[l].data_ptr(), T, st)
                ft.ft_moe_forward(ctx, l, ft.FT_DECODE_CACHED, 0, cur_hid[l].data_ptr(), T, 0, out[l].data_ptr(), st)

        graph = None
        with torch.cuda.stream(stream):
            for s in range(steps):
                if s > 0 and s % 2 == 0:
                    ft.ft_adapt_ratio(ctx, a, stream.cuda_stream)
                    samples.append((a.bp_gbs, a.bh_gbs))
                    if a.r_num >= 0:
                        r = (a.r_num, a.r_den)
                r_seq.append(r)
                refs, fulls = [], []
                for l in range(L):
                    ids, w = oracle.route(logits[s, l], k)
                    ref = cache.step(l, E, ids, r[0], r[1], K_max)
                    full, _, _ = oracle.moe_forward(model.layer_pool(l), model.bx, dtype, d, f, ids, w, hid[s, l],
                                                    slot_ids=ref.slot_ids.reshape(T, k))
                    refs.append((ids, ref))
                    fulls.append(full)
                cur_hid.copy_(torch.from_numpy(hid[s].view(np.int16)))
                cur_lg.copy_(torch.from_numpy(logits[s]))
                if s < steps // 2:
                    step(stream.cuda_stream)  # eager half
                else:
                    if graph is None:
                        graph = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(graph, stream=stream):
                            step(torch.cuda.current_stream().cuda_stream)
                    graph.replay()
                stream.synchronize()
                for l in range(L):
                    g = step_to_host(res[l], T, k, E, K_max)
                    compare_step(g, refs[l][1], f"step {s} layer {l} (r = {r[0]}/{r[1]})")
                    check_output(out[l].cpu().numpy().astype(np.float64), fulls[l], f"step {s} layer {l}")
                compare_table(ft, ctx, cache, f"after step {s}")
        # both bandwidths were measured and r was set from them at least once
        assert a.updates > 0 and a.bp_gbs > 0 and a.bh_gbs > 0, samples
        assert len({x for x in r_seq[2:]}) >= 1 and r_seq[-1] == (a.r_num, a.r_den)
        assert ft.ft_get_status(ctx) == 0
    finally:
        ft.ft_moe_destroy(ctx)


def test_measured_bandwidths_window_and_reset(ft):
    """BP comes from fills only: after a window of steps that fill, BP > 0;
    after a reset and no further fill, both read 0 (no sample)."""
    L, E, k, d, f, S = 1, 16, 2, 256, 128, 8
    model = make_model(L, E, k, d, f, seed=32)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=16, t_max=1)
    ctx = ft.ft_moe_init(cfg, model.pool.ctypes.data, model.pool.nbytes)
    try:
        hid = ftsynth.ar1_hidden(32, 0, 0, 4, d)
        lg = torch.from_numpy(ftsynth.router_logits(hid, model.wr[0])).cuda()
        h = torch.from_numpy(hid.view(np.int16)).cuda()
        out = torch.empty((1, d), dtype=torch.float32, device="cuda")
        for s in range(4):
            ft.ft_cache_step(ctx, 0, lg[s].data_ptr(), 1)
            ft.ft_moe_forward(ctx, 0, ft.FT_DECODE_CACHED, 0, h[s].data_ptr(), 1, 0, out.data_ptr(), 0)
        bp, bh = ft.ft_measured_bandwidths(ctx, reset=True)
        assert bp > 0.0 and bh == 0.0  # fills happened; no CPU executor, nothing reported
        assert ft.ft_measured_bandwidths(ctx, reset=False) == (0.0, 0.0)
        ft.ft_report_host_rate(ctx, 2.0e9, 0.5)
        assert ft.ft_measured_bandwidths(ctx, reset=True)[1] == pytest.approx(4.0)
        with pytest.raises(ft.FtError):
            ft.ft_report_host_rate(ctx, 1.0, 0.0)
    finally:
        ft.ft_moe_destroy(ctx)
