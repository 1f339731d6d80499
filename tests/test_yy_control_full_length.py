"""The cache-control stress workload at full length, checked every step.

48 layers x 64 tokens x top-8 routes per step over E = 128 experts per layer,
Zipf(s) route streams, 10 000 steps (480 000 layer steps), the control kernel
alone replayed as one CUDA graph per step -- the launch configuration bench.py
times.  Inside the graph every layer's step outputs (slot id of every route,
counts, fetch list, victims, evicted experts) are copied to a per-step record
on the device; afterwards the oracle replays the same route stream and every
layer step is compared bit-exactly.  Those outputs determine the residency
table's evolution (hits touch the slots their routes name, fills rewrite the
victims), and the whole table is also compared every 1000 steps and at the
end.  The second case runs a smaller cache (1536 slots, BP/BH = 1/2) where
LRU evicts and leaves routes to the CPU at every step.
"""
import numpy as np
import pytest

import ftsynth
import oracle
from harness import dev_view

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ft():
    from expert_cache_host_gb300 import build as ftbuild
    ftbuild.build()
    import expert_cache_host_gb300 as lib
    lib.load()
    return lib


@pytest.mark.parametrize("S,K_max,s_zipf,r,steps", [(6144, 512, 1.2, (1, 1), 10000),
                                                     (1536, 128, 0.6, (1, 2), 3000)])
def test_control_stress_every_step(ft, S, K_max, s_zipf, r, steps):
    L, E, k, T = 48, 128, 8, 64
    d, f = 256, 128  # the control kernel never reads expert bytes: smallest legal expert shape
    R = T * k
    W = R + 8 + 3 * K_max  # record per layer: slot ids, counts, fetch, victims, evicted
    pool = np.zeros(L * E * ftsynth.expert_bytes(d, f, 0), dtype=np.uint8)
    routes = np.ascontiguousarray(
        np.stack([ftsynth.zipf_routes(0, l, E, T, k, s_zipf, 0, steps, threads=8) for l in range(L)], axis=1))
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=K_max,
                         t_max=T, r_num=r[0], r_den=r[1])
    ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
    try:
        d_routes = torch.from_numpy(routes).cuda()  # [steps, L, T, k]
        cur = torch.empty((L, T, k), dtype=torch.int32, device="cuda")
        rec = torch.zeros((L, W), dtype=torch.int32, device="cuda")
        big = torch.empty((steps, L, W), dtype=torch.int32, device="cuda")
        stream = torch.cuda.Stream()
        tables = {}

        views = []  # the context's step buffers (fixed per layer), viewed once outside the capture

        def step_fn(st):
            for l in range(L):
                o = ft.ft_cache_control(ctx, l, cur[l].data_ptr(), T, st)
                if len(views) < L:
                    views.append((dev_view(o.slot_ids, (R,), "<i4"), dev_view(o.counts, (8,), "<i4"),
                                  dev_view(o.fetch, (K_max,), "<i4"), dev_view(o.victims, (K_max,), "<i4"),
                                  dev_view(o.evicted, (K_max,), "<i4")))
                v = views[l]
                rec[l, :R].copy_(v[0])
                rec[l, R:R + 8].copy_(v[1])
                rec[l, R + 8:R + 8 + K_max].copy_(v[2])
                rec[l, R + 8 + K_max:R + 8 + 2 * K_max].copy_(v[3])
                rec[l, R + 8 + 2 * K_max:].copy_(v[4])

        with torch.cuda.stream(stream):
            cur.copy_(d_routes[0])
            step_fn(stream.cuda_stream)  # step 0 eager (kernel attributes are set outside the capture)
            big[0].copy_(rec)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step_fn(torch.cuda.current_stream().cuda_stream)
            for s in range(1, steps):
                cur.copy_(d_routes[s])
                g.replay()
                big[s].copy_(rec)
                if (s + 1) % 1000 == 0 or s == steps - 1:
                    stream.synchronize()
                    tables[s] = ft.ft_get_table(ctx, L * E, S)
            stream.synchronize()
        assert ft.ft_get_status(ctx) == 0
        got = big.cpu().numpy()
        del big
        cache = oracle.Cache(L * E, S)
        for s in range(steps):
            for l in range(L):
                ref = cache.step(l, E, routes[s, l], r[0], r[1], K_max)
                row = got[s, l]
                q = int(ref.counts[3])
                where = f"step {s} layer {l}"
                assert row[R:R + 5].tolist() == ref.counts.tolist(), f"{where}: counts {row[R:R + 5]} vs {ref.counts}"
                assert np.array_equal(row[:R], ref.slot_ids), f"{where}: slot ids"
                assert np.array_equal(row[R + 8:R + 8 + q], ref.fetch), f"{where}: fetch"
                assert np.array_equal(row[R + 8 + K_max:R + 8 + K_max + q], ref.victims), f"{where}: victims"
                assert np.array_equal(row[R + 8 + 2 * K_max:R + 8 + 2 * K_max + q], ref.evicted), f"{where}: evicted"
            if s in tables:
                so, eo, lu, now = tables[s]
                assert now == int(cache.now[0]), f"after step {s}: clock"
                assert np.array_equal(so, cache.slot_of), f"after step {s}: slot_of"
                assert np.array_equal(eo, cache.expert_of), f"after step {s}: expert_of"
                assert np.array_equal(lu, cache.last_use), f"after step {s}: last_use"
        # the stream exercised the path it is meant to: compulsory misses only
        # with the whole pool cached, evictions and CPU routes with 1536 slots
        cnt = ft.ft_get_counters(ctx, L)
        if S == L * E:
            assert cnt[:, 4].sum() == 0
        else:
            assert cnt[:, 4].sum() > 0 and cnt[:, 3].sum() > 0
    finally:
        ft.ft_moe_destroy(ctx)
