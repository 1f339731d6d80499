"""Shared helpers for the tests: workload construction, device views, and the
oracle-vs-library comparison of one MoE layer step.

The oracle is only ever called from here and from tests; the library under
test is called through its C ABI (expert_cache_host_gb300)."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import ftsynth
import oracle

MAX_REL = 2e-2     # max_i |y - ref| / max(|ref_i|, rms(ref))
NORMWISE = 5e-3    # ||y - ref|| / ||ref||


def dev_view(ptr: int, shape, dtype: str):
    """Zero-copy torch view of library-owned device memory."""
    import torch

    class _A:
        __cuda_array_interface__ = {"shape": tuple(shape), "typestr": dtype, "data": (int(ptr), False), "version": 3}

    return torch.as_tensor(_A(), device="cuda")


@dataclass
class Model:
    L: int
    E: int
    k: int
    d: int
    f: int
    dtype: int
    pool: np.ndarray
    wr: np.ndarray  # [L, E, d] bf16 router weights
    seed: int = 0

    @property
    def bx(self) -> int:
        return ftsynth.expert_bytes(self.d, self.f, self.dtype)

    def layer_pool(self, l: int) -> np.ndarray:
        return self.pool[l * self.E * self.bx:(l + 1) * self.E * self.bx]


def make_model(L, E, k, d, f, dtype=0, seed=0, std=0.02, threads=None) -> Model:
    pool = ftsynth.make_pool(seed, L, E, d, f, dtype, std, threads=threads)
    wr = ftsynth.router_weights(seed, L, E, d, 0.02)
    return Model(L, E, k, d, f, dtype, pool, wr, seed)


def step_to_host(out, T, k, E, K_max):
    """Copy a ft_step_out's device buffers to numpy (ids, w, slot_ids, lists, counts)."""
    cnt = dev_view(out.counts, (8,), "<i4").cpu().numpy()
    n, h, m, q, c = (int(x) for x in cnt[:5])
    g = lambda p, ln, t="<i4": dev_view(p, (ln,), t).cpu().numpy() if ln > 0 else np.zeros(0, dtype=np.int32)
    return dict(
        counts=cnt,
        ids=g(out.ids, T * k).reshape(T, k),
        w=g(out.weights, T * k, "<f4").reshape(T, k),
        slot_ids=g(out.slot_ids, T * k).reshape(T, k),
        uniq=g(out.uniq, n),
        hit_list=g(out.hit_list, h),
        fetch=g(out.fetch, q),
        victims=g(out.victims, q),
        evicted=g(out.evicted, q),
        cpu_list=g(out.cpu_list, c),
    )


def compare_step(gpu: dict, ref: oracle.StepResult, where: str):
    assert gpu["counts"][:5].tolist() == ref.counts.tolist(), f"{where}: counts {gpu['counts'][:5]} vs {ref.counts}"
    for key in ("uniq", "hit_list", "fetch", "victims", "evicted", "cpu_list"):
        assert np.array_equal(gpu[key], getattr(ref, key)), f"{where}: {key} {gpu[key]} vs {getattr(ref, key)}"
    assert np.array_equal(gpu["slot_ids"].reshape(-1), ref.slot_ids), f"{where}: slot_ids"


def compare_table(lib, ctx, cache: oracle.Cache, where: str):
    so, eo, lu, now = lib.ft_get_table(ctx, cache.E_tot, cache.S)
    assert now == int(cache.now[0]), f"{where}: clock {now} vs {int(cache.now[0])}"
    assert np.array_equal(so, cache.slot_of), f"{where}: slot_of"
    assert np.array_equal(eo, cache.expert_of), f"{where}: expert_of"
    assert np.array_equal(lu, cache.last_use), f"{where}: last_use"


def check_output(y: np.ndarray, ref: np.ndarray, where: str):
    mr = oracle.max_rel_err(y, ref)
    nw = oracle.normwise_err(y, ref)
    assert mr <= MAX_REL and nw <= NORMWISE, f"{where}: max rel {mr:.3e} normwise {nw:.3e}"
    return mr, nw
