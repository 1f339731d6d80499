"""Parity at the full decode configurations, in the launch configuration
bench.py times (one CUDA graph per token replayed with new inputs, the pool in
ft_host_alloc memory):
  - A3B-style bf16: 48 layers, E = 128, top-8, d = 2048, f = 768, S = 1536,
    K_max = 128, BP/BH = 1 (58 GB pool);
  - V4-Flash-style MXFP4: 43 layers, E = 256, top-6, d = 4096, f = 2048,
    S = 2393, K_max = 256 (147 GB pool), where the host holds it.
Every layer's control state is compared bit-exactly at every token; every
layer's output at the last tokens (the oracle evaluates the routed experts
one by one)."""
import numpy as np
import pytest

import ftsynth
import oracle
from harness import check_output, compare_step, compare_table, step_to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ft():
    from expert_cache_host_gb300 import build as ftbuild
    ftbuild.build()
    import expert_cache_host_gb300 as lib
    lib.load()
    return lib


def _host_available() -> int:
    with open("/proc/meminfo") as fh:
        for line in fh:
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    return 0


@pytest.mark.parametrize("shape", ["a3b", "v4"])
def test_full_size_graph_replay(ft, shape):
    if shape == "a3b":
        L, E, k, d, f, dt, S, K_max, steps, check_from = 48, 128, 8, 2048, 768, 0, 1536, 128, 6, 4
    else:
        L, E, k, d, f, dt, S, K_max, steps, check_from = 43, 256, 6, 4096, 2048, 1, 2393, 256, 4, 3
    T, r = 1, (1, 1)
    bx = ftsynth.expert_bytes(d, f, dt)
    if L * E * bx + (24 << 30) > _host_available():
        pytest.skip(f"host memory cannot hold the {L * E * bx / 1e9:.0f} GB pool")
    hp = ft.HostPool(L * E * bx)
    ctx = None
    try:
        pool = ftsynth.make_pool(0, L, E, d, f, dt, out=hp.array)
        wr = ftsynth.router_weights(0, L, E, d)
        hid = np.stack([ftsynth.ar1_hidden(0, l, 0, steps, d)[:, None, :] for l in range(L)], axis=1)
        logits = np.stack([ftsynth.router_logits(hid[:, l], wr[l]) for l in range(L)], axis=1)
        cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, dtype=dt, num_slots=S,
                             k_max=K_max, t_max=T, r_num=r[0], r_den=r[1])
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        cache = oracle.Cache(L * E, S)
        cur_hid = torch.empty((L, T, d), dtype=torch.int16, device="cuda")
        cur_lg = torch.empty((L, T, E), dtype=torch.float32, device="cuda")
        partial = torch.zeros((L, T, d), dtype=torch.float32, device="cuda")
        out = torch.empty((L, T, d), dtype=torch.float32, device="cuda")
        stream = torch.cuda.Stream()
        res = [None] * L

        def token(st):
            for l in range(L):
                res[l] = ft.ft_cache_step(ctx, l, cur_lg[l].data_ptr(), T, st)
                ft.ft_moe_forward(ctx, l, ft.FT_DECODE_CACHED, 0, cur_hid[l].data_ptr(), T, partial[l].data_ptr(),
                                  out[l].data_ptr(), st)

        graph = None
        with torch.cuda.stream(stream):
            for s in range(steps):
                refs, fulls = [], []
                for l in range(L):
                    ids, w = oracle.route(logits[s, l], k)
                    ref = cache.step(l, E, ids, r[0], r[1], K_max)
                    if s >= check_from:
                        full, _, cpu_part = oracle.moe_forward(pool[l * E * bx:(l + 1) * E * bx], bx, dt, d, f, ids,
                                                               w, hid[s, l], slot_ids=ref.slot_ids.reshape(T, k))
                        partial[l].copy_(torch.from_numpy(cpu_part.astype(np.float32)))
                        fulls.append(full)
                    else:
                        assert ref.counts[4] == 0  # all-fill: no CPU part to supply
                    refs.append((ids, ref))
                cur_hid.copy_(torch.from_numpy(hid[s].view(np.int16)))
                cur_lg.copy_(torch.from_numpy(logits[s]))
                if s == 0:
                    token(stream.cuda_stream)  # eager: kernel attributes are set outside the capture
                else:
                    if graph is None:
                        graph = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(graph, stream=stream):
                            token(torch.cuda.current_stream().cuda_stream)
                    graph.replay()
                stream.synchronize()
                for l in range(L):
                    g = step_to_host(res[l], T, k, E, K_max)
                    assert np.array_equal(g["ids"], refs[l][0]), f"step {s} layer {l}"
                    compare_step(g, refs[l][1], f"step {s} layer {l}")
                    if s >= check_from:
                        check_output(out[l].cpu().numpy().astype(np.float64), fulls[l], f"step {s} layer {l}")
                compare_table(ft, ctx, cache, f"after step {s}")
        assert ft.ft_get_status(ctx) == 0
    finally:
        if ctx is not None:
            ft.ft_moe_destroy(ctx)
        hp.free()


def test_prefill_8192_token_chunk_a3b(ft):
    """The prefill chunk bench.py times: 8192 tokens, A3B-style expert shape
    (E = 128, top-8, d = 2048, f = 768), full-layer double buffer, two layers
    (layer 1's upload overlaps layer 0's GEMMs), pool in ft_host_alloc memory.
    About 512 rows per expert: full 128-row tiles and ragged tails.  Compared
    with the oracle on every expert's first and last routed token plus a
    spread of others."""
    L, E, k, d, f, T = 2, 128, 8, 2048, 768, 8192
    bx = ftsynth.expert_bytes(d, f, 0)
    hp = ft.HostPool(L * E * bx)
    ctx = None
    try:
        pool = ftsynth.make_pool(0, L, E, d, f, 0, out=hp.array)
        wr = ftsynth.router_weights(0, L, E, d)
        cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=1, k_max=1, t_max=1,
                             prefill_buffers=2, prefill_t_max=T)
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        st = torch.cuda.current_stream().cuda_stream
        outs, inputs = [], []
        for l in range(L):
            hid = ftsynth.prefill_hidden(0, l, T, d, threads=8)
            lg = ftsynth.router_logits(hid, wr[l])
            d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
            d_lg = torch.from_numpy(lg).cuda()
            out = torch.empty((T, d), dtype=torch.float32, device="cuda")
            ft.ft_moe_forward(ctx, l, ft.FT_PREFILL_LAYER, d_lg.data_ptr(), d_hid.data_ptr(), T, 0, out.data_ptr(), st)
            outs.append(out)
            inputs.append((hid, lg, d_hid, d_lg))
        torch.cuda.synchronize()
        assert ft.ft_get_status(ctx) == 0
        for l in range(L):
            hid, lg = inputs[l][:2]
            ids, w = oracle.route(lg, k)
            first = [int(np.argmax((ids == e).any(1))) for e in range(E) if (ids == e).any()]
            last = [T - 1 - int(np.argmax((ids[::-1] == e).any(1))) for e in range(E) if (ids == e).any()]
            assert len(first) == E  # iid hidden states route every expert
            sel = np.unique(np.concatenate([first, last, np.arange(0, T, 257), [T - 1]])).astype(np.int32)
            full, _, _ = oracle.moe_forward(pool[l * E * bx:(l + 1) * E * bx], bx, 0, d, f, ids, w, hid, tokens=sel)
            check_output(outs[l].cpu().numpy()[sel].astype(np.float64), full, f"layer {l}")
    finally:
        if ctx is not None:
            ft.ft_moe_destroy(ctx)
        hp.free()


def test_v4_mxfp4_batch16_graph_replay(ft):
    """V4-Flash-style MXFP4 expert shape (E = 256, top-6, d = 4096, f = 2048)
    at batch 16 (16 independent AR(1) streams), two layers, S = 2393, K_max =
    256, one CUDA graph per step as bench.py --workload v4 --batch 16 runs it;
    control state bit-exact every step, all 16 tokens' outputs checked after
    the first step."""
    L, E, k, d, f, dt, S, K_max, T, steps = 2, 256, 6, 4096, 2048, 1, 2393, 256, 16, 3
    bx = ftsynth.expert_bytes(d, f, dt)
    hp = ft.HostPool(L * E * bx)
    ctx = None
    try:
        pool = ftsynth.make_pool(0, L, E, d, f, dt, out=hp.array)
        wr = ftsynth.router_weights(0, L, E, d)
        hid = np.stack([np.stack([ftsynth.ar1_hidden(0, l, b, steps, d) for b in range(T)], axis=1)
                        for l in range(L)], axis=1)  # [steps, L, T, d]
        logits = np.stack([ftsynth.router_logits(hid[:, l], wr[l]) for l in range(L)], axis=1)
        cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, dtype=dt, num_slots=S,
                             k_max=K_max, t_max=T)
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        cache = oracle.Cache(L * E, S)
        cur_hid = torch.empty((L, T, d), dtype=torch.int16, device="cuda")
        cur_lg = torch.empty((L, T, E), dtype=torch.float32, device="cuda")
        out = torch.empty((L, T, d), dtype=torch.float32, device="cuda")
        stream = torch.cuda.Stream()
        res = [None] * L

        def step_fn(st):
            for l in range(L):
                res[l] = ft.ft_cache_step(ctx, l, cur_lg[l].data_ptr(), T, st)
                ft.ft_moe_forward(ctx, l, ft.FT_DECODE_CACHED, 0, cur_hid[l].data_ptr(), T, 0, out[l].data_ptr(), st)

        graph = None
        with torch.cuda.stream(stream):
            for s in range(steps):
                cur_hid.copy_(torch.from_numpy(hid[s].view(np.int16)))
                cur_lg.copy_(torch.from_numpy(logits[s]))
                if s == 0:
                    step_fn(stream.cuda_stream)
                else:
                    if graph is None:
                        graph = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(graph, stream=stream):
                            step_fn(torch.cuda.current_stream().cuda_stream)
                    graph.replay()
                stream.synchronize()
                for l in range(L):
                    ids, w = oracle.route(logits[s, l], k)
                    ref = cache.step(l, E, ids, 1, 1, K_max)
                    g = step_to_host(res[l], T, k, E, K_max)
                    assert np.array_equal(g["ids"], ids), f"step {s} layer {l}"
                    compare_step(g, ref, f"step {s} layer {l}")
                    assert ref.counts[4] == 0
                    if s >= 1:
                        full, _, _ = oracle.moe_forward(pool[l * E * bx:(l + 1) * E * bx], bx, dt, d, f, ids, w,
                                                        hid[s, l], slot_ids=ref.slot_ids.reshape(T, k))
                        check_output(out[l].cpu().numpy().astype(np.float64), full, f"step {s} layer {l}")
                compare_table(ft, ctx, cache, f"after step {s}")
        assert ft.ft_get_status(ctx) == 0
    finally:
        if ctx is not None:
            ft.ft_moe_destroy(ctx)
        hp.free()
