#!/usr/bin/env python
"""Benchmark of the MoE expert-cache layer step on GB300.

One JSON line on stdout.  The headline (value) is A3B-style decode: 48 MoE
layers, d=2048, E=128 routed experts, top-8, SwiGLU f=768, bf16 weights
N(0, 0.02) in a 57.98 GB pinned host pool, batch 1, AR(1) hidden states
(rho = 0.9), a shared LRU cache of 1536 slots (25% of 48x128), BP/BH = 1,
K_max = 128.  One step is one decode token through all 48 layers -- routing,
cache control, fills from the host pool, expert FFNs and merge -- replayed as
one CUDA graph per token.  `e2e` runs the same tokens from the same cache state
on a twin context with the token's inputs copied in from pinned host memory and
every layer's output copied back inside the timed region.

The same run adds, as components, every other workload of the method:
  - the whole 512-token decode sequence from a cold cache, and A3B decode at
    BP/BH = 1/2 and 2;
  - the 8192-token prefill chunk of the same model (full-layer double buffer
    on and off, grouped GEMM throughput with weights resident);
  - route + control alone, graph-timed, at batch 1 and 16;
  - the cache-control stress workload (48 layers x 64 tokens x top-8, 6144
    slots, Zipf routes, 10 000 steps);
  - the tiny single-layer model (64-token prefill chunk, 32 decode steps);
  - V4-Flash-style MXFP4 decode at batch 1 and 16 (147 GB pool, built after the
    A3B pool is freed);
  - the host link measured over the whole pool, with the pool's memory node.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the decode
workload on its own GPU (the path has no exchange step); rank 0 prints the
line with value = tokens of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import ftsynth  # noqa: E402

METRIC = "MoE decode tok/s (A3B-style, batch 1, GPU side; CPU-routed experts arrive as a partial sum)"
V4 = dict(L=43, E=256, k=6, d=4096, f=2048, dtype=1, S=2393, K_max=256, T=1, rho=0.9, r=(1, 1), seq=256,
          desc="V4-Flash-style decode: 43 layers, d=4096, E=256, top-6, f=2048, MXFP4 experts (147 GB pool), "
               "S=2393 (32 GB budget), BP/BH=1, K_max=256, AR(1) rho=0.9")
A3B = dict(L=48, E=128, k=8, d=2048, f=768, dtype=0, S=1536, K_max=128, T=1, rho=0.9, r=(1, 1), seq=512,
           desc="A3B-style decode: 48 layers, d=2048, E=128, top-8, f=768, bf16, batch 1, "
                "S=1536 (25% of 6144), BP/BH=1, K_max=128, AR(1) rho=0.9")
L2_BYTES = 129 * 2 ** 20

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) over algorithmic
# bytes for the launches of one ncu capture, with the kernel source it was
# taken from (first 16 hex digits of its sha256) and the summary that records
# it.  A launch's traffic is reported as ratio x its algorithmic bytes only
# while the source is unchanged; otherwise traffic is null.
NCU_TRAFFIC = {
    # split decode path: three bf16 expert launches (11 experts), two MXFP4 launches (6 experts)
    "decode_experts": dict(ratio=105_966_592 / 103_809_024, src="expert_cache_host_gb300/csrc/expert_decode.cu",
                           sha16="8b886874d489e037", profile="profiles/decode_experts_a3b.md"),
    "decode_experts_mxfp4": dict(ratio=81_504_000 / 80_216_064, src="expert_cache_host_gb300/csrc/expert_decode_mxfp4.cu",
                                 sha16="e7d6809da31fca43", profile="profiles/decode_experts_mxfp4_v4.md"),
    # two all-hit launches of the fused decode layer kernel (8 resident experts each)
    "decode_layer": dict(ratio=154_340_864 / 150_994_944, src="expert_cache_host_gb300/csrc/decode_layer.cu",
                         sha16="21f6d1d1675fdf2c", profile="profiles/decode_layer_a3b.md"),
    # both prefill GEMMs of one layer (gate/up + down): the A3B 8192-token chunk, and the V4 shape with 64
    # experts and 2048 tokens (192 rows per expert, as in its 8192-token chunk)
    "grouped_gemm": dict(ratio=2_153_847_296 / 2_214_592_512, src="expert_cache_host_gb300/csrc/grouped_gemm.cu",
                         sha16="5f68d3782a496771", profile="profiles/grouped_gemm_prefill_a3b.md"),
    "grouped_gemm_mxfp4": dict(ratio=1_215_293_952 / 1_258_291_200, src="expert_cache_host_gb300/csrc/grouped_gemm.cu",
                               sha16="5f68d3782a496771", profile="profiles/grouped_gemm_prefill_mxfp4_v4.md"),
    # four all-hit launches of the fused kernel's MXFP4 instantiation (6 resident V4 experts each)
    "decode_layer_mxfp4": dict(ratio=331_816_960 / 320_864_256, src="expert_cache_host_gb300/csrc/decode_layer.cu",
                               sha16="21f6d1d1675fdf2c", profile="profiles/decode_layer_mxfp4_v4.md"),
}


# ----------------------------------------------------------------------------- helpers

def dist_env():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def replica_reduce(elapsed_s: float, units: float, world_size: int):
    """Max of the elapsed time and sum of the units over ranks (replicas only:
    this is the only cross-rank communication)."""
    if world_size == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def ncu_traffic(kernel: str, algorithmic_bytes: float):
    """(traffic bytes or None, note) for one launch of `kernel`."""
    t = NCU_TRAFFIC[kernel]
    if t["ratio"] is None:
        return None, f"no ncu capture of {t['src']} yet"
    with open(os.path.join(ROOT, t["src"]), "rb") as fh:
        sha = hashlib.sha256(fh.read()).hexdigest()[:16]
    if sha != t["sha16"]:
        return None, f"{t['src']} changed since the ncu capture in {t['profile']}"
    return round(t["ratio"] * algorithmic_bytes), f"ncu DRAM bytes / algorithmic bytes = {t['ratio']:.4f} " \
                                                  f"({t['profile']}, source sha256 {sha}) x algorithmic bytes per launch"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu, self.proc, self.path = gpu_index, None, None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="ftclk", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as fh:
                rows = [p for p in ([x.strip() for x in line.split(",")] for line in fh) if len(p) >= 9]
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        num = lambda s: s.replace(".", "", 1).isdigit()
        sm = [float(r[1]) for r in rows if num(r[1])]
        mx = [float(r[2]) for r in rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def decode_inputs(w, n_steps, seed=0):
    """AR(1) hidden [steps, L, T, d] bf16 and logits [steps, L, T, E] float32."""
    L, E, d, T = w["L"], w["E"], w["d"], w["T"]
    wr = ftsynth.router_weights(seed, L, E, d)
    hid = np.empty((n_steps, L, T, d), dtype=np.uint16)
    for l in range(L):
        for b in range(T):
            hid[:, l, b, :] = ftsynth.ar1_hidden(seed, l, b, n_steps, d, w["rho"])
    lg = np.stack([ftsynth.router_logits(hid[:, l], wr[l]) for l in range(L)], axis=1)
    return hid, np.ascontiguousarray(lg)


def timed(stream, fn, reps=1):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream.synchronize()
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3


def pool_placement(pool):
    """Host-side record of where the pool's pages live: the memory nodes this
    process sees, the GPU's nearest node, and the pages of the pool's mapping
    per node (/proc/self/numa_maps)."""
    import torch
    rec = {}
    try:
        with open("/sys/devices/system/node/online") as fh:
            rec["nodes_online"] = fh.read().strip()
    except OSError:
        rec["nodes_online"] = None
    try:
        bus = torch.cuda.get_device_properties(torch.cuda.current_device()).pci_bus_id.lower()
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as fh:
            rec["gpu_numa_node"] = int(fh.read().strip())
    except (OSError, AttributeError, ValueError):
        rec["gpu_numa_node"] = None
    base = pool.ctypes.data
    try:
        with open("/proc/self/numa_maps") as fh:
            for line in fh:
                parts = line.split()
                start = int(parts[0], 16)
                if start <= base < start + pool.nbytes and start >= base - (1 << 30):
                    rec["pool_pages_per_node"] = {p.split("=")[0]: int(p.split("=")[1]) for p in parts
                                                  if p.startswith("N") and "=" in p}
                    rec["page_kb"] = next((int(p.split("=")[1]) for p in parts if p.startswith("kernelpagesize_kB")), None)
                    rec["policy"] = parts[1]
                    break
    except OSError:
        pass
    return rec


def host_link_profile(pool, chunk=1 << 30):
    """Host -> device copy-engine rate over the WHOLE pool: every 1 GiB chunk
    copied once, each timed with CUDA events (the rate the pool can stream at,
    which prefill uploads and decode fills see), plus the best of three copies
    of the first 1.21 GB (a burst from a region touched just before)."""
    import torch
    n = pool.nbytes // chunk
    src = torch.from_numpy(pool[:n * chunk]).view(n, chunk)
    dst = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    s.synchronize()
    ev[0].record(s)
    for i in range(n):
        dst.copy_(src[i], non_blocking=True)
        ev[i + 1].record(s)
    ev[n].synchronize()
    per = [chunk / (ev[i].elapsed_time(ev[i + 1]) / 1e3) / 1e9 for i in range(n)]
    whole = n * chunk / (ev[0].elapsed_time(ev[n]) / 1e3) / 1e9
    burst_bytes = min(pool.nbytes, 1_207_959_552)
    b = torch.from_numpy(pool[:burst_bytes])
    bd = torch.empty(burst_bytes, dtype=torch.uint8, device="cuda")
    burst = burst_bytes / min(timed(s, lambda: bd.copy_(b, non_blocking=True)) for _ in range(3)) / 1e9
    del dst, bd
    slow = [i for i, g in enumerate(per) if g < 150.0]
    srt = sorted(per)
    return {"whole_pool_gbs": round(whole, 1), "chunks": n, "chunk_gbs_min": round(srt[0], 1),
            "chunk_gbs_median": round(srt[n // 2], 1), "chunk_gbs_max": round(srt[-1], 1),
            "slow_chunks": {"count_below_150_gbs": len(slow), "first_indices": slow[:16],
                            "gbs": [round(per[i], 1) for i in slow[:16]]},
            "burst_first_1p21gb_gbs": round(burst, 1),
            "how": "pinned H2D cudaMemcpyAsync of every 1 GiB chunk of the pool once, CUDA events"}


def experts_alone(w, pool, hid, reps=40):
    """The bf16 decode expert kernel with its merge, outside the step: the
    first k experts of layer 0 resident in a scratch arena, one token, L2
    flushed (256 MB written) before every call, CUDA events around the call
    (route grouping + experts + merge of the allocation-free entry).  Returns
    {experts: median seconds} for k and for 2 experts."""
    import torch

    import expert_cache_host_gb300 as ft
    d, f, k = w["d"], w["f"], w["k"]
    bx = ftsynth.expert_bytes(d, f, 0)
    arena = torch.from_numpy(pool[:k * bx]).cuda()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    x = torch.from_numpy(hid[0, 0, :1].view(np.int16)).cuda()
    out = torch.empty((1, d), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    res = {}
    for n in (k, 2):
        sid = torch.arange(n, dtype=torch.int32, device="cuda")
        wt = torch.full((n,), 1.0 / n, dtype=torch.float32, device="cuda")
        ts = []
        for r in range(reps + 3):
            flush.add_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            ft.ft_decode_experts_noalloc(arena.data_ptr(), k, d, f, n, 1, sid.data_ptr(), wt.data_ptr(), x.data_ptr(),
                                         0, out.data_ptr(), 0, st.cuda_stream)
            e1.record(st)
            e1.synchronize()
            if r >= 3:
                ts.append(e0.elapsed_time(e1) / 1e3)
        res[n] = statistics.median(ts)
    del arena, flush
    return res


# ----------------------------------------------------------------------------- decode

class DecodeRun:
    """One context over the decode workload, its per-token CUDA graph, and the
    device copies of the step inputs."""

    def __init__(self, w, pool, d_hid, d_lg):
        import torch

        import expert_cache_host_gb300 as ft
        self.ft, self.w = ft, w
        L, E, k, d, f, T = w["L"], w["E"], w["k"], w["d"], w["f"], w["T"]
        cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, dtype=w["dtype"],
                             num_slots=w["S"], k_max=w["K_max"], t_max=T, r_num=w["r"][0], r_den=w["r"][1],
                             decode_path=w.get("decode_path", 0), fill_ctas=w.get("fill_ctas", 0))
        t0 = time.time()
        self.ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        self.t_init = time.time() - t0
        self.d_hid, self.d_lg = d_hid, d_lg
        self.cur_hid = torch.empty((L, T, d), dtype=torch.int16, device="cuda")
        self.cur_lg = torch.empty((L, T, E), dtype=torch.float32, device="cuda")
        self.out = torch.empty((L, T, d), dtype=torch.float32, device="cuda")
        self.stream = torch.cuda.Stream()
        self.graph = None

    def token(self, st):
        ft, L, T = self.ft, self.w["L"], self.w["T"]
        for l in range(L):
            ft.ft_cache_step(self.ctx, l, self.cur_lg[l].data_ptr(), T, st)
            ft.ft_moe_forward(self.ctx, l, ft.FT_DECODE_CACHED, 0, self.cur_hid[l].data_ptr(), T, 0,
                              self.out[l].data_ptr(), st)

    def begin(self):
        """Token 0 eagerly (kernel attributes are set outside any capture), then
        capture one token as a graph.  Returns the next token index."""
        import torch
        with torch.cuda.stream(self.stream):
            self.cur_hid.copy_(self.d_hid[0])
            self.cur_lg.copy_(self.d_lg[0])
            self.token(self.stream.cuda_stream)
            self.stream.synchronize()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=self.stream):
                self.token(torch.cuda.current_stream().cuda_stream)
        return 1

    def step(self, s):
        self.cur_hid.copy_(self.d_hid[s])
        self.cur_lg.copy_(self.d_lg[s])
        self.graph.replay()

    def counters(self):
        return self.ft.ft_get_counters(self.ctx, self.w["L"])

    def destroy(self):
        if self.ctx:
            self.ft.ft_moe_destroy(self.ctx)
            self.ctx = None


def _window(c0, c1):
    dc = (c1 - c0).astype(np.float64)
    hits, misses, fills, cpu = (dc[:, i].sum() for i in range(4))
    return hits, misses, fills, cpu


def run_decode_leg(args, w, world, local, pool, hid, lg, with_e2e=True, seq=True, profile=True):
    """Headline decode measurement.  Context A times K tokens after W warm-up
    tokens (device inputs, graph replays).  With the end-to-end twin B (stepped through the
    same W warm-up tokens; pinned host inputs in, every layer's output out) the
    two contexts step tokens W..W+2K-1 and take turns to lead: A is timed on
    the K tokens it leads, B on the other K.  A then runs P profiled tokens
    eagerly (per-kernel CUDA events) and, from a cold rebuild, the whole decode
    sequence."""
    import torch

    import expert_cache_host_gb300 as ft

    L, d, f, T = w["L"], w["d"], w["f"], w["T"]
    bx = ftsynth.expert_bytes(d, f, w["dtype"])
    W, K = args.warmup, args.steps
    P = min(K, args.profile_steps) if profile else 0
    d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
    d_lg = torch.from_numpy(lg).cuda()
    A = DecodeRun(w, pool, d_hid, d_lg)
    B = DecodeRun(w, pool, d_hid, d_lg) if with_e2e else None
    res = {}
    try:
        if args.cpu_exec:
            ft.ft_cpu_executor(A.ctx, args.cpu_exec)
            if B:
                ft.ft_cpu_executor(B.ctx, args.cpu_exec)
        s = A.begin()
        if B:
            B.begin()
        with torch.cuda.stream(A.stream):
            for i in range(s, W):
                A.step(i)
                if B:
                    with torch.cuda.stream(B.stream):
                        B.step(i)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        c0 = A.counters()
        ft.ft_decode_meters(A.ctx, reset=True)
        e2e_elapsed = None
        if B:
            h_hid = torch.from_numpy(hid.view(np.int16)).pin_memory()
            h_lg = torch.from_numpy(lg).pin_memory()
            h_out = torch.empty((L, T, d), dtype=torch.float32).pin_memory()
            cb0 = B.counters()
            e2e_elapsed = 0.0

            def e2e_step(i):
                B.cur_hid.copy_(h_hid[i], non_blocking=True)
                B.cur_lg.copy_(h_lg[i], non_blocking=True)
                B.graph.replay()
                h_out.copy_(B.out, non_blocking=True)

        with ClockSampler(local) as clk:
            if not B:
                it = iter(range(W, W + K))
                with torch.cuda.stream(A.stream):
                    elapsed = timed(A.stream, lambda: A.step(next(it)), K)
                dA = A.counters() - c0
                meters = ft.ft_decode_meters(A.ctx, reset=True)
            else:
                # The two contexts step the same 2K tokens and take turns to go
                # first: A leads the even tokens, B (end to end) the odd ones,
                # and each is timed only on the tokens it leads.  The context
                # that follows reads the pool pages the leader has just read
                # and runs a few per cent faster, so no follower token is
                # timed, and both sums see the same host-link conditions.
                elapsed = 0.0
                dA = np.zeros_like(c0)
                dB = np.zeros_like(c0)  # the control counters of the tokens B leads
                meters = None
                for j in range(2 * K):
                    i = W + j
                    if j % 2 == 0:
                        ca = A.counters()
                        ft.ft_decode_meters(A.ctx, reset=True)
                        with torch.cuda.stream(A.stream):
                            elapsed += timed(A.stream, lambda: A.step(i))
                        m = ft.ft_decode_meters(A.ctx, reset=True)
                        meters = m if meters is None else {n: meters[n] + m[n] for n in m}
                        dA += A.counters() - ca
                        with torch.cuda.stream(B.stream):
                            e2e_step(i)
                        B.stream.synchronize()
                    else:
                        cb = B.counters()
                        with torch.cuda.stream(B.stream):
                            e2e_elapsed += timed(B.stream, lambda: e2e_step(i))
                        dB += B.counters() - cb
                        with torch.cuda.stream(A.stream):
                            A.step(i)
                        A.stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        res["meters"] = meters  # fill and resident-expert phases of the timed tokens
        res["path"] = "fused" if ft.ft_decode_path(A.ctx) == ft.FT_DECODE_FUSED else "split"
        clocks = clk.summary()
        hits, misses, fills, cpu = _window(np.zeros_like(dA), dA)
        end = W + K
        if B:
            end = W + 2 * K
            # same tokens from the same cache state: the control streams agree
            res["e2e_same_window"] = bool(np.array_equal(B.counters() - cb0, A.counters() - c0))
            # the two timed token sets differ: their fills per token, side by side
            res["e2e_fills"] = (_window(np.zeros_like(dB), dB)[2], fills)
            B.destroy()
            B = None

        prof = None
        if P:
            ft.ft_profile_enable(A.ctx, True)
            ft.ft_profile_read(A.ctx, reset=True)
            cp0 = A.counters()
            with torch.cuda.stream(A.stream):
                for i in range(end, end + P):
                    A.cur_hid.copy_(d_hid[i])
                    A.cur_lg.copy_(d_lg[i])
                    A.token(A.stream.cuda_stream)
            prof = ft.ft_profile_read(A.ctx, reset=True)
            cp1 = A.counters()
            ft.ft_profile_enable(A.ctx, False)
            dp = (cp1 - cp0).astype(np.float64)
            groups_p, fills_p = dp[:, 0].sum() + dp[:, 2].sum(), dp[:, 2].sum()

        if seq:
            res["sequence"] = _sequence(A, w, hid.shape[0])
        status = ft.ft_get_status(A.ctx)
        t_init = A.t_init
    finally:
        A.destroy()
        if B:
            B.destroy()

    elapsed_max, units = replica_reduce(elapsed, K * T, world)
    res.update(value=units / elapsed_max, elapsed=elapsed_max, K=K, W=W, T=T, stride=2 if with_e2e else 1,
               clocks=clocks, status=status,
               t_init=t_init, hits=hits, misses=misses, fills=fills, cpu=cpu, P=P, bx=bx)
    if B is None and e2e_elapsed is not None:
        res.update(e2e=K * T / e2e_elapsed, h2d=int(lg[0].nbytes + hid[0].nbytes), d2h=int(L * T * d * 4))
    if prof:
        tot_ms = sum(v[0] for v in prof.values())
        ex_ms, ex_n = prof["experts"]
        fill_ms, fill_n = prof["fill"]
        res.update(shares={n: round(v[0] / tot_ms, 4) for n, v in prof.items() if v[1]},
                   ms_per_token={n: round(v[0] / P, 4) for n, v in prof.items() if v[1]},
                   launches={n: v[1] for n, v in prof.items() if v[1]},
                   ex_bytes=groups_p * bx, ex_ms=ex_ms, ex_n=ex_n, fill_bytes=fills_p * bx, fill_ms=fill_ms,
                   fill_n=fill_n, control_us=prof["control"][0] / max(1, prof["control"][1]) * 1e3,
                   eager_ms=tot_ms / P)
    return res


def _sequence(A, w, n_avail):
    """The configured decode sequence from a cold cache (ft_cache_rebuild
    resets the table; the graph is captured again): tokens [0, 64) and [64, N)
    timed separately, with the hit rate of each part."""
    import torch
    ft = A.ft
    N = min(w["seq"], n_avail)
    ft.ft_cache_rebuild(A.ctx, w["S"])
    A.begin()  # token 0 eagerly and a new capture (the rebuild changed the epoch)
    cut = min(64, N)
    out = {}
    with torch.cuda.stream(A.stream):
        c_prev = None
        for name, lo, hi in (("first", 1, cut), ("rest", cut, N)):
            if hi <= lo:
                continue
            c0 = A.counters() if c_prev is None else c_prev
            it = iter(range(lo, hi))
            el = timed(A.stream, lambda: A.step(next(it)), hi - lo)
            c1 = A.counters()
            c_prev = c1
            h, m, fi, _ = _window(c0, c1)
            out[name] = dict(tokens=[lo, hi], tok_s=round((hi - lo) * w["T"] / el, 3),
                             hit_rate=round(h / max(1.0, h + m), 4), fills_per_token=round(fi / ((hi - lo) * w["T"]), 3))
    tot = sum(v["tokens"][1] - v["tokens"][0] for v in out.values())
    t_all = sum((v["tokens"][1] - v["tokens"][0]) * w["T"] / v["tok_s"] for v in out.values())
    return dict(tokens=N, tok_s_tokens_1_to_N=round(tot * w["T"] / t_all, 3), **out,
                note="token 0 runs eagerly before the capture and is not timed")


def run_adaptive_leg(args, w, pool, hid, lg, threads=8, every=4):
    """Run-time r = BP/BH: A3B decode with the context's CPU expert executor,
    starting from r = 1/2; every `every` tokens ft_adapt_ratio reads the
    measured fill rate (BP) and CPU expert rate (BH) and sets r (graphs pick
    it up from device memory).  The adaptation calls are inside the timed
    region (they synchronise)."""
    import torch

    import expert_cache_host_gb300 as ft
    wr = dict(w, r=(1, 2))
    d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
    d_lg = torch.from_numpy(lg).cuda()
    A = DecodeRun(wr, pool, d_hid, d_lg)
    try:
        ft.ft_cpu_executor(A.ctx, threads)
        a = ft.ft_ratio_adapter_init(0.5, 256, 256 * 64)
        r_seq = []
        s = A.begin()
        W, K = args.warmup, args.steps

        def tok(i):
            if i % every == 0:
                ft.ft_adapt_ratio(A.ctx, a, A.stream.cuda_stream)
            r_seq.append(a.r_num)
            A.step(i)

        with torch.cuda.stream(A.stream):
            for i in range(s, W):
                tok(i)
            c0 = A.counters()
            it = iter(range(W, W + K))
            el = timed(A.stream, lambda: tok(next(it)), K)
            c1 = A.counters()
        h, m, fi, cpu = _window(c0, c1)
        return dict(workload=wr["desc"].replace("BP/BH=1", "BP/BH adapted at run time from 1/2") +
                    f", CPU expert executor ({threads} host threads), r updated every {every} tokens",
                    tok_s=round(K * w["T"] / el, 3), timed_tokens=K, warmup_tokens=W,
                    r_den=a.r_den, r_num_at_tokens={str(i + s): x for i, x in enumerate(r_seq) if
                                                    i == 0 or x != r_seq[i - 1]},
                    bp_gbs_estimate=round(a.bp_gbs, 1), bh_gbs_estimate=round(a.bh_gbs, 1),
                    hit_rate=round(h / max(1.0, h + m), 4), fills_per_token=round(fi / (K * w["T"]), 3),
                    cpu_routes_per_token=round(cpu / (K * w["T"]), 3), device_status=ft.ft_get_status(A.ctx))
    finally:
        A.destroy()


def run_route_control_leg(w, batches=(1, 16), n=128):
    """Route + control (one fused kernel per layer step) alone, graph-timed:
    one CUDA graph of the L ft_cache_step calls replayed over n decode steps
    with new logits, CUDA events around the replays; microseconds per layer
    step.  The cache state follows the same route stream as in decode."""
    import torch

    import expert_cache_host_gb300 as ft
    L, E, k = w["L"], w["E"], w["k"]
    pool = np.zeros(L * E * ftsynth.expert_bytes(256, 128, 0), dtype=np.uint8)  # never read by the control path
    out = []
    for T in batches:
        _, lg = decode_inputs(dict(w, T=T), n)
        d_lg = torch.from_numpy(lg).cuda()
        cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=256, inter=128, num_slots=w["S"],
                             k_max=w["K_max"], t_max=T)
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        try:
            cur = torch.empty((L, T, E), dtype=torch.float32, device="cuda")
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                cur.copy_(d_lg[0])
                for l in range(L):
                    ft.ft_cache_step(ctx, l, cur[l].data_ptr(), T, st.cuda_stream)
                st.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=st):
                    for l in range(L):
                        ft.ft_cache_step(ctx, l, cur[l].data_ptr(), T, torch.cuda.current_stream().cuda_stream)
                i = 1

                def step():
                    nonlocal i
                    cur.copy_(d_lg[i])
                    g.replay()
                    i += 1

                for _ in range(8):
                    step()
                el = timed(st, step, n - 9)
            out.append(dict(T=T, S=w["S"], K_max=w["K_max"], us_per_layer_step=round(el / ((n - 9) * L) * 1e6, 3),
                            layer_steps=(n - 9) * L, status=ft.ft_get_status(ctx)))
        finally:
            ft.ft_moe_destroy(ctx)
    return out


# ----------------------------------------------------------------------------- prefill chunk

def run_prefill_leg(args, w, pool):
    import torch

    import expert_cache_host_gb300 as ft

    L = args.prefill_layers or w["L"]
    E, k, d, f, T = w["E"], w["k"], w["d"], w["f"], args.prefill_tokens
    dt = w["dtype"]
    bx = ftsynth.expert_bytes(d, f, dt)
    wr = ftsynth.router_weights(0, L, E, d)
    hid = np.stack([ftsynth.prefill_hidden(0, l, T, d) for l in range(L)])
    lg = np.stack([ftsynth.router_logits(hid[l], wr[l]) for l in range(L)])
    d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
    d_lg = torch.from_numpy(lg).cuda()
    del hid, lg
    out = torch.empty((T, d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    # The double- and the single-buffer context take turns, three timed chunks
    # each, and each reports its median: the host link has slow spells of
    # seconds, which would otherwise land on one setting only.
    ctxs, times = {}, {2: [], 1: []}
    try:
        for buffers in (2, 1):
            cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, dtype=dt, num_slots=1,
                                 k_max=1, t_max=1, prefill_buffers=buffers, prefill_t_max=T)
            ctxs[buffers] = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        with torch.cuda.stream(stream):
            st = stream.cuda_stream

            def chunk(ctx):
                for l in range(L):
                    ft.ft_moe_forward(ctx, l, ft.FT_PREFILL_LAYER, d_lg[l].data_ptr(), d_hid[l].data_ptr(), T, 0,
                                      out.data_ptr(), st)

            for buffers in (2, 1):
                chunk(ctxs[buffers])  # warm-up chunk (each chunk re-uploads the whole pool)
            for _ in range(3):
                for buffers in (2, 1):
                    times[buffers].append(timed(stream, lambda: chunk(ctxs[buffers])))
            # upload rate and grouped-GEMM throughput, weights resident (layer 0 twice in a row)
            ctx = ctxs[2]
            ft.ft_profile_enable(ctx, True)
            ft.ft_profile_read(ctx, reset=True)
            chunk(ctx)
            prof_chunk = ft.ft_profile_read(ctx, reset=True)
            for _ in range(3):
                ft.ft_moe_forward(ctx, 0, ft.FT_PREFILL_LAYER, d_lg[0].data_ptr(), d_hid[0].data_ptr(), T, 0,
                                  out.data_ptr(), st)
            ft.ft_moe_forward(ctx, 0, ft.FT_PREFILL_LAYER, d_lg[0].data_ptr(), d_hid[0].data_ptr(), T, 0,
                              out.data_ptr(), st)
            prof_res = ft.ft_profile_read(ctx, reset=True)
            ft.ft_profile_enable(ctx, False)
        status = max(ft.ft_get_status(c) for c in ctxs.values())
    finally:
        for c in ctxs.values():
            ft.ft_moe_destroy(c)
    res = {b_: statistics.median(v) for b_, v in times.items()}
    pool_bytes = L * E * bx
    # algorithmic bytes of one layer's two GEMMs: X in, the layer's experts, H out and back in, Y out
    gemm_bytes = T * k * d * 2 + E * bx + 2 * T * k * f * 2 + T * k * d * 4
    gemm_traffic, gemm_traffic_note = ncu_traffic("grouped_gemm" if dt == 0 else "grouped_gemm_mxfp4", gemm_bytes)
    up_ms, up_n = prof_chunk["upload"]
    gemm_ms, gemm_n = prof_res["gemm"]
    flops_layer = T * k * 3 * d * f * 2  # 3 matrices of d*f MACs per (token, expert), 2 flops per MAC
    gemm_tflops = flops_layer / (gemm_ms / gemm_n / 1e3) / 1e12 if gemm_n else 0.0
    upload_gbs = up_n * E * bx / (up_ms / 1e3) / 1e9 if up_n else 0.0
    return dict(L=L, T=T, chunk_s=res[2], chunk_s_single_buffer=res[1], pool_bytes=pool_bytes,
                link_gbs=pool_bytes / res[2] / 1e9, upload_gbs=upload_gbs, gemm_tflops=gemm_tflops,
                gemm_ms_per_layer=gemm_ms / max(1, gemm_n), status=status, gemm_bytes_per_layer=gemm_bytes,
                gemm_traffic_per_layer=gemm_traffic, gemm_traffic_source=gemm_traffic_note,
                chunk_s_runs={"double": [round(t, 4) for t in times[2]], "single": [round(t, 4) for t in times[1]]},
                overlap_loss_without_double_buffer=1.0 - res[2] / res[1])


# ----------------------------------------------------------------------------- control stress

def run_control_leg(args):
    import torch

    import expert_cache_host_gb300 as ft

    L, E, k, T, steps = 48, 128, 8, 64, args.control_steps
    d, f = 256, 128  # the control kernel never reads expert bytes: smallest legal expert shape
    pool = np.zeros(L * E * ftsynth.expert_bytes(d, f, 0), dtype=np.uint8)
    stream = torch.cuda.Stream()
    cases = [(6144, km, s) for s in (0.6, 1.2) for km in (8, 64, 128, 512)] + \
            [(S, 128, s) for S in (1536, 512) for s in (0.6, 1.2)]
    routes = {}
    for s in (0.6, 1.2):
        r = np.stack([ftsynth.zipf_routes(0, l, E, T, k, s, 0, steps) for l in range(L)], axis=1)
        routes[s] = torch.from_numpy(r).cuda()  # [steps, L, T, k]
    out = []
    for S, km, s in cases:
        cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=km, t_max=T)
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        try:
            cur = torch.empty((L, T, k), dtype=torch.int32, device="cuda")
            with torch.cuda.stream(stream):
                cur.copy_(routes[s][0])
                for l in range(L):
                    ft.ft_cache_control(ctx, l, cur[l].data_ptr(), T, stream.cuda_stream)
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for l in range(L):
                        ft.ft_cache_control(ctx, l, cur[l].data_ptr(), T, torch.cuda.current_stream().cuda_stream)
                i = 1

                def step():
                    nonlocal i
                    cur.copy_(routes[s][i])
                    g.replay()
                    i += 1

                warm = min(100, steps // 4)
                for _ in range(warm):
                    step()
                c0 = ft.ft_get_counters(ctx, L)
                el = timed(stream, step, steps - 1 - warm)
                c1 = ft.ft_get_counters(ctx, L)
            dc = (c1 - c0).astype(np.float64)
            n_ls = (steps - 1 - warm) * L
            out.append(dict(S=S, K_max=km, zipf_s=s, us_per_layer_step=round(el / n_ls * 1e6, 3),
                            miss_rate=round(dc[:, 1].sum() / max(1.0, dc[:, 0].sum() + dc[:, 1].sum()), 4),
                            fills_per_layer_step=round(dc[:, 2].sum() / n_ls, 3), status=ft.ft_get_status(ctx)))
        finally:
            ft.ft_moe_destroy(ctx)
    return out


# ----------------------------------------------------------------------------- tiny model

def run_tiny_leg():
    """The tiny single-layer model: d=256, E=16, top-2, f=128, bf16, S=8,
    BP/BH=1.  One 64-token prefill chunk (median of 20, events), then 32
    batch-1 decode steps from a cold cache as graph replays (AR(1) hidden)."""
    import torch

    import expert_cache_host_gb300 as ft
    L, E, k, d, f, S, Tp, n_dec = 1, 16, 2, 256, 128, 8, 64, 32
    pool = ftsynth.make_pool(0, L, E, d, f, 0, 0.02, threads=4)
    wr = ftsynth.router_weights(0, L, E, d)
    hp = ftsynth.prefill_hidden(0, 0, Tp, d)
    lp = ftsynth.router_logits(hp, wr[0])
    hd = ftsynth.ar1_hidden(0, 0, 0, n_dec + 1, d)
    ld = ftsynth.router_logits(hd, wr[0])
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=16, t_max=1,
                         prefill_buffers=1, prefill_t_max=Tp)
    ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
    try:
        st = torch.cuda.Stream()
        d_hp, d_lp = torch.from_numpy(hp.view(np.int16)).cuda(), torch.from_numpy(lp).cuda()
        d_hd, d_ld = torch.from_numpy(hd.view(np.int16)).cuda(), torch.from_numpy(ld).cuda()
        out_p = torch.empty((Tp, d), dtype=torch.float32, device="cuda")
        out = torch.empty((1, d), dtype=torch.float32, device="cuda")
        cur_h, cur_l = torch.empty((1, d), dtype=torch.int16, device="cuda"), torch.empty((1, E), device="cuda")
        with torch.cuda.stream(st):
            pf = lambda: ft.ft_moe_forward(ctx, 0, ft.FT_PREFILL_LAYER, d_lp.data_ptr(), d_hp.data_ptr(), Tp, 0,
                                           out_p.data_ptr(), st.cuda_stream)
            pf()
            pre = statistics.median(timed(st, pf) for _ in range(20))

            def tok(s):
                ft.ft_cache_step(ctx, 0, cur_l.data_ptr(), 1, s)
                ft.ft_moe_forward(ctx, 0, ft.FT_DECODE_CACHED, 0, cur_h.data_ptr(), 1, 0, out.data_ptr(), s)

            cur_h.copy_(d_hd[0:1])
            cur_l.copy_(d_ld[0:1])
            tok(st.cuda_stream)
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                tok(torch.cuda.current_stream().cuda_stream)
            i = 1

            def step():
                nonlocal i
                cur_h.copy_(d_hd[i:i + 1])
                cur_l.copy_(d_ld[i:i + 1])
                g.replay()
                i += 1

            el = timed(st, step, n_dec)
        c = ft.ft_get_counters(ctx, 1)[0]
        return dict(workload="tiny: 1 layer, d=256, E=16, top-2, f=128, bf16, S=8, BP/BH=1",
                    prefill_chunk_64_us=round(pre * 1e6, 2), decode_us_per_step=round(el / n_dec * 1e6, 2),
                    decode_steps=n_dec + 1, hits=int(c[0]), misses=int(c[1]), fills=int(c[2]),
                    status=ft.ft_get_status(ctx))
    finally:
        ft.ft_moe_destroy(ctx)


# ----------------------------------------------------------------------------- oracle (CPU baseline / reference arm)

def oracle_decode_rate(w, pool, hid, lg, budget_s, min_layer_steps=1, warmup_tokens=0, steps=None,
                       layers_per_step=None):
    """Time the oracle on the decode workload (routing, cache step and fp64
    experts of every layer step), after warmup_tokens untimed tokens from a
    cold cache.  steps=None: layer steps in token order until budget_s has
    passed (at least min_layer_steps); else exactly `steps` steps, each the
    first layers_per_step layers of one token.  Returns (tokens/s, tokens
    timed -- fractional when a step covers part of a token, seconds, threads)."""
    import oracle
    L, E, k, d, f, T = w["L"], w["E"], w["k"], w["d"], w["f"], w["T"]
    bx = ftsynth.expert_bytes(d, f, w["dtype"])
    cache = oracle.Cache(L * E, w["S"])

    def layer_step(s, l):
        ids, wt = oracle.route(lg[s, l], k)
        ref = cache.step(l, E, ids, w["r"][0], w["r"][1], w["K_max"])
        oracle.moe_forward(pool[l * E * bx:(l + 1) * E * bx], bx, w["dtype"], d, f, ids, wt, hid[s, l],
                           slot_ids=ref.slot_ids.reshape(T, k))

    Ls = layers_per_step or L
    for s in range(warmup_tokens):
        for l in range(Ls):
            layer_step(s, l)
    done, t_spent = 0, 0.0
    for s in range(warmup_tokens, hid.shape[0] if steps is None else warmup_tokens + steps):
        for l in range(Ls):
            t0 = time.time()
            layer_step(s, l)
            t_spent += time.time() - t0
            done += 1
            if steps is None and done >= min_layer_steps and t_spent >= budget_s:
                break
        else:
            continue
        break
    # the expert evaluations of one layer run in parallel over its T*k routes
    threads = min(oracle.threads(), T * k)
    tokens = done / L
    return tokens * T / t_spent, tokens, t_spent, threads


def line_config(args, w, world):
    """The `config` object both arms print (the same workload, in the same words)."""
    bx = ftsynth.expert_bytes(w["d"], w["f"], w["dtype"])
    return {"workload": w["desc"], "batch": w["T"], "graph": "one CUDA graph per token",
            "l2": "inputs larger than L2: %.2f GB of expert weights per token" % (w["L"] * w["k"] * bx / 1e9),
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


def run_reference(args, w, world):
    """The oracle as the reference arm: same metric, unit, config and step
    counts -- W untimed warm-up steps from a cold cache, then exactly K timed
    steps -- on the host cores.  A step is one decode token through all
    layers, or, when W + K whole tokens would take longer than --ref-budget-s,
    the first layers of one token (the oracle's cost per layer step does not
    depend on the layer), and tok/s counts the layers actually run."""
    import oracle
    pool = ftsynth.make_pool(0, w["L"], w["E"], w["d"], w["f"], w["dtype"], 0.02)
    W, K = args.warmup, args.steps
    hid, lg = decode_inputs(w, W + K)
    # cost of one layer step, from a throwaway one
    bx = ftsynth.expert_bytes(w["d"], w["f"], w["dtype"])
    ids, wt = oracle.route(lg[0, 0], w["k"])
    t0 = time.time()
    oracle.moe_forward(pool[:w["E"] * bx], bx, w["dtype"], w["d"], w["f"], ids, wt, hid[0, 0])
    per_layer = time.time() - t0
    Ls = max(1, min(w["L"], int(args.ref_budget_s / max(1e-9, (W + K) * per_layer))))
    rate, _, t, threads = oracle_decode_rate(w, pool, hid, lg, args.ref_budget_s, warmup_tokens=W, steps=K,
                                              layers_per_step=Ls)
    what = "decode tokens" if Ls == w["L"] else f"steps of the first {Ls} of {w['L']} layers of a decode token"
    sample = f"{K} timed {what} after {W} warm-up steps from a cold cache ({t:.1f} s of oracle work)"
    return {
        "impl": "reference", "metric": metric_name(args, w), "value": round(rate, 5), "unit": "tok/s", "n_gpus": world,
        "steps": int(K), "warmup": int(W), "ms_per_step": round(t / K * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": line_config(args, w, world),
        "cpu_baseline": {"value": round(rate, 5), "unit": "tok/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(rate, 5), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- sweeps (report mode)

def run_sweep(args, w, world, local):
    """One JSON line per point.  capacity: the decode step at S = 5, 10, 25 and
    50 % of the pool's experts (the synthetic counterpart of the article's
    miss rate versus cache capacity, Figure 4b); prompt: the prefill chunk at
    4096, 8192 and 16384 tokens with and without the double buffer (Figure 4a)."""
    hp, pool, _ = make_host_pool(args, w)
    try:
        if args.sweep == "capacity":
            e_tot = w["L"] * w["E"]
            hid, lg = decode_inputs(w, args.warmup + args.steps + min(args.steps, args.profile_steps))
            for pct in (5, 10, 25, 50):
                ws = dict(w, S=max(w["k"] * w["T"], e_tot * pct // 100))
                dec = run_decode_leg(args, ws, world, local, pool, hid, lg, with_e2e=False, seq=False, profile=False)
                routes = dec["hits"] + dec["misses"]
                print(json.dumps({
                    "sweep": "capacity", "workload": w["desc"].split(":")[0], "slots": ws["S"],
                    "capacity_pct": pct, "tok_s": round(dec["value"], 3),
                    "expert_miss_rate": round(dec["misses"] / max(1.0, routes), 4),
                    "fills_per_token": round(dec["fills"] / (dec["K"] * dec["T"]), 3),
                    "timed_tokens": dec["K"], "warmup_tokens": dec["W"], "device_status": dec["status"]}), flush=True)
        elif args.sweep == "fill":
            hid, lg = decode_inputs(w, args.warmup + args.steps + min(args.steps, args.profile_steps))
            peaks = measured_peaks()
            # split path: the fill kernel's CTAs (0 = the library's choice); fused path: fill CTAs of the grid
            split_n = [int(x) for x in args.split_fill_points.split(",") if x]
            points = [("split", n) for n in split_n]
            points += [("fused", n) for n in (19, 38, 57, 76)]
            for rep in range(2):  # the link varies over minutes: every point twice, interleaved
                for path, n in points:
                    ws = dict(w, decode_path=0 if path == "fused" else 1, fill_ctas=n)
                    dec = run_decode_leg(args, ws, world, local, pool, hid, lg, with_e2e=False, seq=False,
                                         profile=path == "split")
                    ex, _ = experts_rate(dec)
                    print(json.dumps({
                        "sweep": "fill", "workload": w["desc"].split(":")[0], "decode_path": dec["path"],
                        "fill_ctas": n, "rep": rep, "tok_s": round(dec["value"], 3),
                        "fill_gbs": round(fill_rate(dec), 1), "experts_gbs": round(ex, 1),
                        "experts_frac_of_hbm": round(ex / peaks["hbm_gbs"], 4),
                        "timed_tokens": dec["K"], "warmup_tokens": dec["W"], "device_status": dec["status"]}),
                        flush=True)
        else:
            w = dict(w, dtype=0)
            for tokens in (4096, 8192, 16384):
                args.prefill_tokens = tokens
                pre = run_prefill_leg(args, w, pool)
                print(json.dumps({
                    "sweep": "prompt", "tokens": tokens, "chunk_s": round(pre["chunk_s"], 4),
                    "chunk_s_single_buffer": round(pre["chunk_s_single_buffer"], 4),
                    "tok_s": round(tokens / pre["chunk_s"], 1), "link_gbs": round(pre["link_gbs"], 1),
                    "gemm_tflops": round(pre["gemm_tflops"], 1), "device_status": pre["status"]}), flush=True)
    finally:
        if hp:
            del pool
            hp.free()


# ----------------------------------------------------------------------------- main

def make_host_pool(args, w):
    """The expert pool, written in the canonical layout.  "pinned": into
    ft_host_alloc memory (mapped in the GPU page tables before the write);
    "registered": into pageable memory that ft_moe_init pins after the write.
    Returns (HostPool or None, uint8 array, seconds to allocate and write)."""
    import expert_cache_host_gb300 as ft
    t0 = time.time()
    n = w["L"] * w["E"] * ftsynth.expert_bytes(w["d"], w["f"], w["dtype"])
    hp = ft.HostPool(n) if args.pool == "pinned" else None
    pool = ftsynth.make_pool(0, w["L"], w["E"], w["d"], w["f"], w["dtype"], 0.02, out=hp.array if hp else None)
    return hp, pool, time.time() - t0


def host_available() -> int:
    with open("/proc/meminfo") as fh:
        for line in fh:
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    return 0


def metric_name(args, w):
    m = METRIC.replace("batch 1", f"batch {w['T']}") if w["dtype"] == 0 else \
        METRIC.replace("A3B-style, batch 1", f"V4-Flash-style MXFP4, batch {w['T']}")
    if args.cpu_exec:
        m = m.replace("GPU side; CPU-routed experts arrive as a partial sum", "GPU + CPU expert executor")
    return m


def fill_rate(dec):
    """GB/s of the decode fill over the timed window: bytes over the summed
    spans of the fill launches (device clock; the fused kernel's fill CTAs or
    the split path's fill kernel)."""
    m = dec.get("meters")
    if m and m["fill_s"] > 0:
        return m["fill_bytes"] / m["fill_s"] / 1e9
    if dec.get("fill_ms"):
        return dec["fill_bytes"] / (dec["fill_ms"] / 1e3) / 1e9
    return 0.0


def experts_rate(dec):
    """(GB/s, how) of the decode experts.  Fused path: the experts resident
    before the step, over the span from the first compute CTA start to the
    last resident work item end, summed over the timed window's launches
    (device clock).  Split path: every executed expert over the expert
    launches' CUDA-event durations (profiled tokens)."""
    m = dec.get("meters")
    if dec.get("path") == "fused":
        if not m or m["resident_s"] <= 0:
            return 0.0, None
        # a phase of less than one resident expert per layer on average (hit rate ~0: the step's experts
        # are installed by its own fill and run behind it) measures start-up, not streaming
        per_launch = m["resident_bytes"] / max(1, m.get("resident_launches", 0))
        if per_launch < dec.get("bx", 0):
            return 0.0, None
        return (m["resident_bytes"] / m["resident_s"] / 1e9,
                "fused path: resident experts' bytes / resident phase span (first compute CTA start to last "
                "resident item end), device clock, timed window")
    if dec.get("ex_ms"):
        return dec["ex_bytes"] / (dec["ex_ms"] / 1e3) / 1e9, "expert launches' bytes / CUDA-event durations, profiled tokens"
    return 0.0, None


def experts_traffic(w, dec):
    """(bytes per launch, bytes from ncu or None, note) of the decode experts:
    fused path, the resident experts of a launch; split path, an expert launch."""
    if dec.get("path") == "fused":
        m = dec.get("meters") or {}
        per = m.get("resident_bytes", 0.0) / max(1, m.get("resident_launches", 0))
        key = "decode_layer" if w["dtype"] == 0 else "decode_layer_mxfp4"
    else:
        per = dec.get("ex_bytes", 0.0) / max(1, dec.get("ex_n", 0))
        key = "decode_experts" if w["dtype"] == 0 else "decode_experts_mxfp4"
    if per <= 0:
        return per, None, "no resident experts in the timed window"
    tr, note = ncu_traffic(key, per)
    return per, tr, note


def decode_summary(w, dec, peaks, link_gbs):
    """Per-workload decode figures (component form)."""
    r = dict(workload=w["desc"], tok_s=round(dec["value"], 3), timed_tokens=dec["K"], warmup_tokens=dec["W"],
             hit_rate=round(dec["hits"] / max(1.0, dec["hits"] + dec["misses"]), 4),
             fills_per_token=round(dec["fills"] / (dec["K"] * dec["T"]), 3),
             cpu_routes_per_token=round(dec["cpu"] / (dec["K"] * dec["T"]), 3), device_status=dec["status"])
    ex_gbs, ex_how = experts_rate(dec)
    if ex_gbs:
        r["experts_gbs"] = round(ex_gbs, 1)
        r["experts_frac_of_hbm"] = round(ex_gbs / peaks["hbm_gbs"], 4)
        r["experts_how"] = ex_how
    fill_gbs = fill_rate(dec)
    if fill_gbs:
        r["fill_gbs"] = round(fill_gbs, 1)
        r["fill_frac_of_link"] = round(fill_gbs / link_gbs, 4) if link_gbs else None
    r["decode_path"] = dec.get("path")
    if "sequence" in dec:
        r["sequence"] = dec["sequence"]
    return r


def fill_link_peak(link):
    """The host-link peak of the decode fill fractions: the median rate of the
    pool's 1 GiB chunks (a fill reads experts scattered over the pool; a
    few slow regions pull the whole-pool rate down but not the median)."""
    return link["chunk_gbs_median"] if link else 0.0


def build_line(args, w, world, dec, link, pre, ctl, peaks, comps=None):
    """The bench line.  `link` is the host-link record (host_link_profile);
    its median 1 GiB chunk rate is the peak of the fill's host-link fraction,
    its whole-pool rate that of the prefill's."""
    link_gbs = fill_link_peak(link)
    ex_gbs, ex_how = experts_rate(dec)
    fill_gbs = fill_rate(dec)
    fused = dec.get("path") == "fused"
    m = dec.get("meters") or {}
    ex_per_launch, traffic, traffic_src = experts_traffic(w, dec)
    if fused:
        ex_us = m.get("resident_s", 0.0) / max(1, m.get("resident_launches", 0)) * 1e6
    else:
        ex_us = dec["ex_ms"] / max(1, dec.get("ex_n", 0)) * 1e3 if dec.get("ex_ms") else None
    hits, misses = dec["hits"], dec["misses"]
    cfg = line_config(args, w, world)
    line = {
        "metric": metric_name(args, w),
        "value": round(dec["value"], 3), "unit": "tok/s", "n_gpus": world, "steps": dec["K"],
        "warmup": dec["W"], "ms_per_step": round(dec["elapsed"] / dec["K"] * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w["dtype"] == 0 else "e2m1*e8m0 x bf16 -> f16/f32",
        "data": "synthetic", "config": cfg,
        # with the end-to-end twin, value's K tokens are every second token of a 2K-token range
        "timed_window": {"tokens": [dec["W"], dec["W"] + dec.get("stride", 1) * dec["K"]],
                         "every": dec.get("stride", 1), "of_sequence": w["seq"],
                         "hit_rate": round(hits / max(1.0, hits + misses), 4),
                         "fills_per_token": round(dec["fills"] / (dec["K"] * dec["T"]), 3)},
        # the dominant kernel by time is the fill: host-link bound
        "roofline": {"bound": "host_link",
                     "kernel": "decode fill (host pool -> slots)" + (": the fill CTAs of the fused decode layer kernel"
                                                                     if fused else ""),
                     "achieved": round(fill_gbs, 1), "peak": link_gbs, "unit": "GB/s",
                     "frac": round(fill_gbs / link_gbs, 4) if link_gbs else None, "traffic": None,
                     "traffic_note": "DRAM counters do not see the host link; its bytes per fill launch equal q x B_x "
                                     "to 0.001 % (system-memory read sectors, profiles/fill_host_link_a3b.md)",
                     "achieved_how": "bytes filled / summed fill spans (first fill CTA start to last fill CTA end, "
                                     "device clock) over the timed window",
                     "peak_source": "measured in this run: the median rate of the pool's 1 GiB chunks, each "
                                    "streamed host -> device once by the copy engine (whole-pool rate: host_link)",
                     "share": dec.get("shares", {}).get("experts" if fused else "fill")},
        "roofline_experts": {"bound": "hbm",
                             "kernel": ("decode experts resident before the step (fused decode layer kernel, compute "
                                        "CTAs)" if fused else "decode experts (in the step, beside the fill)"),
                             "achieved": round(ex_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(ex_gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
                             "traffic_source": traffic_src, "peak_source": peaks["source"], "achieved_how": ex_how,
                             "bytes_per_launch": round(ex_per_launch),
                             "avg_us_per_launch": round(ex_us, 2) if ex_us else None,
                             "share": dec.get("shares", {}).get("experts")},
        "components": {
            "kernel_share": dec.get("shares"),
            "kernel_ms_per_token": {n: round(v / dec["T"], 4) for n, v in dec.get("ms_per_token", {}).items()},
            "route_control_us_per_layer_step_eager": round(dec["control_us"], 3) if "control_us" in dec else None,
            "hit_rate": round(hits / max(1.0, hits + misses), 4),
            "fills_per_token": round(dec["fills"] / (dec["K"] * dec["T"]), 3),
            "cpu_routes_per_token": round(dec["cpu"] / (dec["K"] * dec["T"]), 3),
            "fills_per_step": round(dec["fills"] / dec["K"], 3), "tokens_per_step": dec["T"],
            "eager_ms_per_token_profiled": round(dec["eager_ms"] / dec["T"], 4) if dec.get("eager_ms") else None,
            "init_pin_s": round(dec["t_init"], 2), "device_status": dec["status"],
        },
        "clocks": dec["clocks"],
        # per layer: route + control (one kernel), then the fused decode layer kernel (fill + experts) and the
        # merge, or on the split path the fill, the resident and installed expert launches and the merge
        "gpu_launches": int(dec["K"] * w["L"] * (3 if fused else 5)),
    }
    if "e2e" in dec:
        line["e2e"] = {"value": round(dec["e2e"], 3), "unit": "tok/s", "h2d_bytes_per_step": dec["h2d"],
                       "d2h_bytes_per_step": dec["d2h"]}
        if dec.get("e2e_fills"):
            fb, fa = dec["e2e_fills"]
            line["components"]["e2e_fills_per_token"] = {"e2e_tokens": round(fb / (dec["K"] * dec["T"]), 3),
                                                          "value_tokens": round(fa / (dec["K"] * dec["T"]), 3)}
        line["components"]["e2e_how"] = ("a twin context (host copies in and out) and the device-timed context step the "
                                         "same 2K tokens and take turns to go first; each is timed on the K "
                                         "tokens it leads; control streams identical: %s"
                                         % dec.get("e2e_same_window"))
    if "sequence" in dec:
        line["components"]["sequence"] = dec["sequence"]
    if link:
        line["host_link"] = link
    if pre:
        pre_link = pre.get("link_profile_gbs") or link_gbs
        line["prefill"] = {
            "workload": f"{pre['T']}-token chunk, A3B-style, {pre['L']} layers, full-layer double buffer",
            "chunk_s": round(pre["chunk_s"], 4), "chunk_s_single_buffer": round(pre["chunk_s_single_buffer"], 4),
            "chunk_s_runs": pre["chunk_s_runs"],
            "chunk_timing": "median of three chunks per setting, double and single buffer taking turns",
            "loss_without_double_buffer": round(pre["overlap_loss_without_double_buffer"], 4),
            "tok_s": round(pre["T"] / pre["chunk_s"], 1), "pool_gb": round(pre["pool_bytes"] / 1e9, 2),
            "link_gbs_effective": round(pre["link_gbs"], 1), "upload_gbs": round(pre["upload_gbs"], 1),
            "link_frac": round(pre["link_gbs"] / pre_link, 4) if pre_link else None,
            "link_peak_gbs": pre_link, "device_status": pre["status"],
            "link_peak_how": "the fastest of three whole-pool host -> device streams: the run's host_link pass and "
                             "two just before and just after the prefill leg", "link_around": pre.get("link_around"),
            "roofline_gemm": {"bound": "tensor", "kernel": "grouped SwiGLU GEMMs (tcgen05), weights resident",
                              "achieved": round(pre["gemm_tflops"], 1), "peak": peaks["bf16_tflops"],
                              "unit": "TFLOP/s", "frac": round(pre["gemm_tflops"] / peaks["bf16_tflops"], 4),
                              "ms_per_layer": round(pre["gemm_ms_per_layer"], 3),
                              "traffic": pre["gemm_traffic_per_layer"], "traffic_unit": "bytes per layer (both GEMMs)",
                              "algorithmic_bytes_per_layer": pre["gemm_bytes_per_layer"],
                              "traffic_source": pre["gemm_traffic_source"],
                              "peak_source": peaks["source"] + " (burst bf16)"},
        }
    if ctl:
        line["control_stress"] = {
            "workload": "control kernel alone, 48 layers x 64 tokens x top-8, E=128, Zipf routes, graph replay",
            "steps": args.control_steps, "cases": ctl,
        }
    if comps:
        line["components"].update(comps)
    return line


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=448)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--profile-steps", type=int, default=32)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-budget-s", type=float, default=150.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-control", action="store_true")
    ap.add_argument("--no-components", action="store_true", help="the headline decode leg only")
    ap.add_argument("--no-v4", action="store_true", help="skip the V4 MXFP4 components")
    ap.add_argument("--prefill-tokens", type=int, default=8192)
    ap.add_argument("--prefill-layers", type=int, default=0)
    ap.add_argument("--control-steps", type=int, default=10000)
    ap.add_argument("--prefill-only", action="store_true", help="profiling case: the prefill leg alone")
    ap.add_argument("--workload", choices=("a3b", "v4"), default="a3b",
                    help="a3b: bf16 A3B-style decode (default line); v4: MXFP4 V4-Flash-style decode")
    ap.add_argument("--batch", type=int, default=0, help="decode tokens per step (default 1)")
    ap.add_argument("--layers", type=int, default=0, help="override L (small profiling cases, not a bench line)")
    ap.add_argument("--slots", type=int, default=0, help="override S (small profiling cases, not a bench line)")
    ap.add_argument("--experts", type=int, default=0, help="override E (small profiling cases, not a bench line)")
    ap.add_argument("--sweep", choices=("capacity", "prompt", "fill"), default=None,
                    help="report mode (not the bench line): decode miss rate and tok/s over cache capacities of "
                         "5/10/25/50%% of the pool, or prefill chunk time over prompt lengths 4k/8k/16k with and "
                         "without the double buffer; or decode on the split path and on the fused path with 19 to 76 "
                         "fill CTAs")
    ap.add_argument("--ratio", default=None, help="r = BP/BH as NUM/DEN for the decode workload (default 1/1: every "
                    "miss filled)")
    ap.add_argument("--cpu-exec", type=int, default=0, help="variant: the context's CPU expert executor with this many "
                    "host threads computes the misses that are not filled (not the bench line)")
    ap.add_argument("--repeat-tokens", action="store_true",
                    help="profiling case (not a bench line): every decode token's inputs twice in a row, so the "
                         "second pass hits on every expert and runs with no fill")
    ap.add_argument("--decode-path", choices=("fused", "split"), default="fused",
                    help="fused: one cooperative kernel per layer runs the fill and the experts (bf16); split: a "
                         "fill kernel beside two expert launches")
    ap.add_argument("--fill-ctas", type=int, default=0, help="CTAs that fill (0 = the library's choice)")
    ap.add_argument("--split-fill-points", default="0,76,57,38",
                    help="--sweep fill: fill CTA counts of the split path (0 = the library's choice)")
    ap.add_argument("--pool", choices=("pinned", "registered"), default="pinned",
                    help="pinned: pool written into ft_host_alloc memory; registered: pageable pool pinned by "
                         "ft_moe_init after the write")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    w = dict(A3B if args.workload == "a3b" else V4)
    if args.batch:
        w["T"] = args.batch
        w["desc"] = w["desc"].replace("batch 1, ", "") + f", batch {args.batch}"
    if args.workload == "v4":
        # keep the per-layer shapes; drop layers only if the host cannot hold the pinned pool
        per_layer = w["E"] * ftsynth.expert_bytes(w["d"], w["f"], 1)
        fit = int(max(0, host_available() - (24 << 30)) // per_layer)
        if fit < w["L"]:
            w["L"] = max(1, fit)
            w["desc"] += f" [host RAM holds {w['L']} of the 43 layers]"
        args.no_prefill = args.no_control = args.no_components = True
    if args.ratio:
        num, den = (int(x) for x in args.ratio.split("/"))
        w["r"] = (num, den)
        w["desc"] = w["desc"].replace("BP/BH=1", f"BP/BH={num}/{den}")
    if args.cpu_exec:
        w["desc"] += f", CPU executor with {args.cpu_exec} host threads for the unfilled misses"
    w["decode_path"] = 0 if args.decode_path == "fused" else 1
    w["fill_ctas"] = args.fill_ctas
    if args.decode_path == "split" or args.fill_ctas:
        w["desc"] += f" [decode path {args.decode_path}" + (f", {args.fill_ctas} fill CTAs]" if args.fill_ctas else "]")
    if args.layers or args.slots or args.experts:
        w["L"], w["S"], w["E"] = args.layers or w["L"], args.slots or w["S"], args.experts or w["E"]
        w["desc"] += f" [profiling case: L={w['L']}, S={w['S']}, E={w['E']}]"
        args.no_components = True

    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w, world)), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import torch

    from expert_cache_host_gb300 import build as ftbuild
    ftbuild.build()
    torch.cuda.set_device(local)
    if args.prefill_only:
        # profiling case: the prefill leg alone on the first --prefill-layers layers (not a bench line)
        w["L"] = args.prefill_layers or w["L"]
        hp, pool, _ = make_host_pool(args, w)
        print(json.dumps({"profiling_case": "prefill", **run_prefill_leg(args, w, pool)}), flush=True)
        if hp:
            del pool
            hp.free()
        return
    if args.sweep:
        run_sweep(args, w, world, local)
        return
    hp, pool, t_pool = make_host_pool(args, w)
    n_in = max(args.warmup + 2 * args.steps + min(args.steps, args.profile_steps), w["seq"])
    hid, lg = decode_inputs(w, n_in)
    if args.repeat_tokens:
        hid = np.ascontiguousarray(np.repeat(hid[:(n_in + 1) // 2], 2, axis=0)[:n_in])
        lg = np.ascontiguousarray(np.repeat(lg[:(n_in + 1) // 2], 2, axis=0)[:n_in])
        w["desc"] += " [profiling case: every token twice]"
        args.no_components = True
    seq = rank == 0 and not args.no_components
    dec = run_decode_leg(args, w, world, local, pool, hid, lg, with_e2e=True, seq=seq)
    # components time at most 128 tokens after at most 32 warm-up tokens
    cargs = argparse.Namespace(**vars(args))
    cargs.steps, cargs.warmup = min(args.steps, 128), min(args.warmup, 32)
    pre = ctl = alone = link = None
    comps = {}
    if rank == 0:
        import expert_cache_host_gb300 as ft
        # the pool is registered (pinned, mapped) for the measurement below by a throwaway context
        cfg = ft.make_config(num_layers=w["L"], num_experts=w["E"], top_k=w["k"], hidden=w["d"], inter=w["f"],
                             dtype=w["dtype"], num_slots=1, k_max=1, t_max=1)
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        try:
            link = host_link_profile(pool)
            link["placement"] = pool_placement(pool)
        finally:
            ft.ft_moe_destroy(ctx)
        if w["dtype"] == 0 and not args.no_components:
            alone = experts_alone(w, pool, hid)
            for rr in ((1, 2), (2, 1)):
                wr_ = dict(w, r=rr, desc=w["desc"].replace("BP/BH=1", f"BP/BH={rr[0]}/{rr[1]}"))
                d_r = run_decode_leg(cargs, wr_, 1, local, pool, hid, lg, with_e2e=False, seq=False)
                comps[f"decode_r_{rr[0]}_{rr[1]}"] = decode_summary(wr_, d_r, measured_peaks(), fill_link_peak(link))
            comps["decode_adaptive_r"] = run_adaptive_leg(cargs, w, pool, hid, lg)
            comps["route_control_graph"] = run_route_control_leg(w)
            comps["tiny"] = run_tiny_leg()
        if not args.no_prefill and not args.no_components:
            ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
            try:
                before = host_link_profile(pool)
                pre = run_prefill_leg(args, w, pool)
                after = host_link_profile(pool)
            finally:
                ft.ft_moe_destroy(ctx)
            # the link drifts within minutes: the peak is the fastest whole-pool pass of the run
            pre["link_profile_gbs"] = max(before["whole_pool_gbs"], after["whole_pool_gbs"], link["whole_pool_gbs"])
            pre["link_around"] = {"before": before, "after": after}
        if not args.no_control and not args.no_components:
            ctl = run_control_leg(args)
    peaks = measured_peaks()
    line = None
    if rank == 0:
        line = build_line(args, w, world, dec, link, pre, ctl, peaks, comps)
        if alone:
            bx = ftsynth.expert_bytes(w["d"], w["f"], 0)
            t8 = alone[w["k"]]
            line["roofline_experts_alone"] = {
                "bound": "hbm", "kernel": f"decode experts + merge outside the step ({w['k']} resident experts, "
                                          "batch 1, L2 flushed; allocation-free entry: route grouping, experts, merge)",
                "achieved": round(w["k"] * bx / t8 / 1e9, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(w["k"] * bx / t8 / 1e9 / peaks["hbm_gbs"], 4), "us": round(t8 * 1e6, 2),
                "us_2_experts": round(alone[2] * 1e6, 2), "peak_source": peaks["source"]}
        if not args.no_cpu_baseline:
            rate, n, t, threads = oracle_decode_rate(w, pool, hid, lg, args.cpu_budget_s, min_layer_steps=1)
            line["cpu_baseline"] = {"value": round(rate, 5), "unit": "tok/s", "cores": threads, "kind": "oracle",
                                    "sample": f"{n:.2f} decode tokens x {w['L']} layers from a cold cache, "
                                              f"{t:.1f} s of oracle work"}
        line["components"]["pool"] = (f"{args.pool}: {pool.nbytes / 1e9:.2f} GB, allocated and written in "
                                      f"{t_pool:.1f} s")
    del hid, lg
    if hp:
        del pool
        hp.free()
    if rank == 0 and not args.no_components and not args.no_v4:
        line["components"]["v4"] = run_v4_components(cargs, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_v4_components(args, local):
    """V4-Flash-style MXFP4 decode at batch 1 and 16 and an 8192-token prefill
    chunk, after the A3B pool is freed: the 147 GB pool in ft_host_alloc
    memory (fewer layers only if the host cannot hold it, said in the
    workload)."""
    w = dict(V4)
    per_layer = w["E"] * ftsynth.expert_bytes(w["d"], w["f"], 1)
    fit = int(max(0, host_available() - (24 << 30)) // per_layer)
    if fit < 1:
        return {"unavailable": "host memory cannot hold one V4 layer"}
    if fit < w["L"]:
        w["L"] = fit
        w["desc"] += f" [host RAM holds {w['L']} of the 43 layers]"
    hp, pool, t_pool = make_host_pool(args, w)
    out = {"pool": f"{pool.nbytes / 1e9:.2f} GB, allocated and written in {t_pool:.1f} s"}
    try:
        peaks = measured_peaks()
        import expert_cache_host_gb300 as ft
        cfg = ft.make_config(num_layers=w["L"], num_experts=w["E"], top_k=w["k"], hidden=w["d"], inter=w["f"],
                             dtype=1, num_slots=1, k_max=1, t_max=1)
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        try:
            # a freshly written pool can still hold slow pages on the first full pass: two passes, the faster counts
            passes = [host_link_profile(pool) for _ in range(2)]
            link = dict(max(passes, key=lambda p: p["whole_pool_gbs"]))
            link["passes_whole_pool_gbs"] = [p["whole_pool_gbs"] for p in passes]
            link["placement"] = pool_placement(pool)
        finally:
            ft.ft_moe_destroy(ctx)
        out["host_link"] = link
        for T in (1, 16):
            wt = dict(w, T=T)
            if T > 1:
                wt["desc"] = wt["desc"] + f", batch {T}"
            n_in = max(args.warmup + args.steps + min(args.steps, args.profile_steps), w["seq"] if T == 1 else 0)
            hid, lg = decode_inputs(wt, n_in)
            d = run_decode_leg(args, wt, 1, local, pool, hid, lg, with_e2e=False, seq=(T == 1))
            s = decode_summary(wt, d, peaks, fill_link_peak(link))
            _, tr, note = experts_traffic(wt, d)
            s["experts_traffic_per_launch"], s["experts_traffic_source"] = tr, note
            out[f"batch_{T}"] = s
            del hid, lg
        if not args.no_prefill:
            pre = run_prefill_leg(args, w, pool)
            bf16_peak = peaks["bf16_tflops"]
            out["prefill"] = {
                "workload": f"{pre['T']}-token chunk, V4-Flash-style MXFP4, {pre['L']} layers, full-layer double "
                            "buffer",
                "chunk_s": round(pre["chunk_s"], 4), "chunk_s_single_buffer": round(pre["chunk_s_single_buffer"], 4),
                "chunk_s_runs": pre["chunk_s_runs"],
                "chunk_timing": "median of three chunks per setting, double and single buffer taking turns",
                "tok_s": round(pre["T"] / pre["chunk_s"], 1), "pool_gb": round(pre["pool_bytes"] / 1e9, 2),
                "link_gbs_effective": round(pre["link_gbs"], 1), "upload_gbs": round(pre["upload_gbs"], 1),
                "link_frac": round(pre["link_gbs"] / link["whole_pool_gbs"], 4), "device_status": pre["status"],
                "roofline_gemm": {"bound": "tensor", "kernel": "grouped SwiGLU GEMMs (tcgen05 kind::f16), MXFP4 "
                                  "weights dequantised exactly to bf16 in shared memory, weights resident",
                                  "achieved": round(pre["gemm_tflops"], 1), "peak": bf16_peak, "unit": "TFLOP/s",
                                  "frac": round(pre["gemm_tflops"] / bf16_peak, 4),
                                  "ms_per_layer": round(pre["gemm_ms_per_layer"], 3),
                                  "traffic": pre["gemm_traffic_per_layer"],
                                  "traffic_unit": "bytes per layer (both GEMMs)",
                                  "algorithmic_bytes_per_layer": pre["gemm_bytes_per_layer"],
                                  "traffic_source": pre["gemm_traffic_source"],
                                  "peak_source": peaks["source"] + " (burst bf16)"},
            }
    finally:
        del pool
        hp.free()
    return out


if __name__ == "__main__":
    main()
