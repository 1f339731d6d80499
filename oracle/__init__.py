"""ORACLE -- test infrastructure only.

A plain, slow, fp64 CPU statement of the FreeToken expert-cache layer step
(routing, shared LRU residency table, q* split, K-LRU victims, route rewrite,
SwiGLU experts with bf16 or MXFP4 weights, merge of partial sums).  It shares
no code with the CUDA library and never imports it.  Only tests/, the smoke
check and the benchmark's CPU-baseline leg may import this package; the
product path never calls it.

The arithmetic lives in ftoracle.c (compiled here with gcc, OpenMP over
expert evaluations when the compiler supports it); this file marshals numpy
arrays through ctypes and keeps the cache state between calls.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libftoracle.so")
_SRC = os.path.join(_HERE, "ftoracle.c")
_lock = threading.Lock()
_lib = None

OR_OK, OR_EARG, OR_ENAN, OR_ERANGE, OR_EWRAP = 0, -1, -2, -3, -4
DTYPE_BF16, DTYPE_MXFP4 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc; OpenMP if available, plain otherwise."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(tmp, _SO)
    return _SO


def _l():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, u64, vp, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_double
            lib.or_route.argtypes = [vp, i32, i32, i32, vp, vp]
            lib.or_cache_step.argtypes = [i32, i32, i32, vp, i64, i64, i32, vp, i32, vp, vp, i32, vp,
                                          vp, vp, vp, vp, vp, vp, vp, vp, vp, i32]
            lib.or_e2m1_value.argtypes = [i32]
            lib.or_e2m1_value.restype = dbl
            lib.or_e8m0_value.argtypes = [i32]
            lib.or_e8m0_value.restype = dbl
            lib.or_expert_ffn.argtypes = [vp, i32, i32, i32, vp, vp]
            lib.or_moe_forward.argtypes = [vp, u64, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp]
            lib.or_dense_moe.argtypes = [vp, u64, i32, i32, i32, i32, i32, vp, vp, vp]
            lib.or_threads.argtypes = []
            lib.or_threads.restype = i32
            lib.or_adapt_ratio.argtypes = [i32, vp, vp, dbl, i32, i32, vp]
            for fn in ("or_route", "or_cache_step", "or_expert_ffn", "or_moe_forward", "or_dense_moe",
                       "or_adapt_ratio"):
                getattr(lib, fn).restype = i32
            _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != OR_OK:
        raise OracleError(f"{what} returned {rc}")


def threads() -> int:
    """Threads the oracle's expert evaluations may use."""
    return int(_l().or_threads())


# ------------------------------------------------------------------ routing

def route(logits: np.ndarray, k: int):
    """Top-k routing of float32 logits [T, E] -> (ids int32 [T,k], w float64 [T,k])."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _check(_l().or_route(_p(logits), T, E, k, _p(ids), _p(w)), "or_route")
    return ids, w


# ------------------------------------------------------------ cache control

@dataclass
class StepResult:
    uniq: np.ndarray
    counts: np.ndarray  # n, hits, m, q, cpu
    hit_list: np.ndarray
    miss_list: np.ndarray
    fetch: np.ndarray
    victims: np.ndarray
    evicted: np.ndarray
    cpu_list: np.ndarray
    slot_ids: np.ndarray


@dataclass
class Cache:
    """Residency table of the shared expert cache (all layers, one clock)."""

    E_tot: int
    S: int
    slot_of: np.ndarray = field(init=False)
    expert_of: np.ndarray = field(init=False)
    last_use: np.ndarray = field(init=False)
    now: np.ndarray = field(init=False)

    def __post_init__(self):
        self.slot_of = np.full(self.E_tot, -1, dtype=np.int32)
        self.expert_of = np.full(self.S, -1, dtype=np.int32)
        self.last_use = np.zeros(self.S, dtype=np.uint32)
        self.now = np.zeros(1, dtype=np.uint32)

    def step(self, layer: int, E: int, ids: np.ndarray, r_num: int, r_den: int, K_max: int,
             fill_order: int = 0) -> StepResult:
        """One control step; fill_order 0 fills the first q misses in ascending
        id, 1 the q misses with the most routes in the step (ties: lower id)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
        nr = ids.size
        cap = max(1, nr)
        uniq = np.empty(cap, dtype=np.int32)
        counts = np.zeros(5, dtype=np.int32)
        hit = np.empty(cap, dtype=np.int32)
        miss = np.empty(cap, dtype=np.int32)
        fetch = np.empty(max(1, K_max), dtype=np.int32)
        vict = np.empty(max(1, K_max), dtype=np.int32)
        evic = np.empty(max(1, K_max), dtype=np.int32)
        cpu = np.empty(cap, dtype=np.int32)
        sid = np.empty(cap, dtype=np.int32)
        rc = _l().or_cache_step(layer, E, nr, _p(ids), r_num, r_den, K_max, _p(self.slot_of), self.E_tot,
                                _p(self.expert_of), _p(self.last_use), self.S, _p(self.now), _p(uniq),
                                _p(counts), _p(hit), _p(miss), _p(fetch), _p(vict), _p(evic), _p(cpu), _p(sid),
                                fill_order)
        _check(rc, "or_cache_step")
        n, h, m, q, c = (int(x) for x in counts)
        return StepResult(uniq[:n].copy(), counts, hit[:h].copy(), miss[:m].copy(), fetch[:q].copy(),
                          vict[:q].copy(), evic[:q].copy(), cpu[:c].copy(), sid[:nr].copy())

    def rebuild_retain(self, new_S: int) -> "Cache":
        """A rebuild at new_S slots that keeps the most recently used residents
        (the variant of the article's runtime cache rebuild, section
        "弹性边缘资源管理": GPU memory changes only performance, so any subset
        of the residents may stay).  Residents are taken in order of last use,
        most recent first, ties to the lower slot; the i-th kept one moves to
        slot i with its last use; the clock is unchanged."""
        kept = sorted((s for s in range(self.S) if self.expert_of[s] >= 0),
                      key=lambda s: (-int(self.last_use[s]), s))[:new_S]
        n = Cache(self.E_tot, new_S)
        n.now[:] = self.now
        for i, s in enumerate(kept):
            u = int(self.expert_of[s])
            n.expert_of[i] = u
            n.slot_of[u] = i
            n.last_use[i] = self.last_use[s]
        return n


# ---------------------------------------------------------------- experts

def e2m1_value(code: int) -> float:
    return _l().or_e2m1_value(int(code))


def e8m0_value(e: int) -> float:
    return _l().or_e8m0_value(int(e))


def expert_ffn(expert: np.ndarray, dtype: int, d: int, f: int, x_bf16: np.ndarray) -> np.ndarray:
    expert = np.ascontiguousarray(expert, dtype=np.uint8)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    y = np.empty(d, dtype=np.float64)
    _check(_l().or_expert_ffn(_p(expert), dtype, d, f, _p(x), _p(y)), "or_expert_ffn")
    return y


def moe_forward(layer_pool: np.ndarray, expert_bytes: int, dtype: int, d: int, f: int, ids: np.ndarray,
                w: np.ndarray, hidden_bf16: np.ndarray, slot_ids: np.ndarray | None = None,
                tokens: np.ndarray | None = None):
    """Routed SwiGLU MoE of one layer: returns (out_full, out_gpu, out_cpu) float64 [n_sel, d].

    layer_pool: uint8 bytes of the layer's E experts (expert e at e*expert_bytes).
    """
    layer_pool = np.ascontiguousarray(layer_pool).view(np.uint8).reshape(-1)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    w = np.ascontiguousarray(w, dtype=np.float64)
    hid = np.ascontiguousarray(hidden_bf16, dtype=np.uint16)
    sid = None if slot_ids is None else np.ascontiguousarray(slot_ids, dtype=np.int32).reshape(T, k)
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n_sel = T if tok is None else tok.size
    full = np.empty((n_sel, d), dtype=np.float64)
    gpu = np.empty((n_sel, d), dtype=np.float64)
    cpu = np.empty((n_sel, d), dtype=np.float64)
    rc = _l().or_moe_forward(_p(layer_pool), expert_bytes, dtype, d, f, T, k, _p(ids), _p(w), _p(sid), _p(hid),
                             _p(tok), n_sel, _p(full), _p(gpu), _p(cpu))
    _check(rc, "or_moe_forward")
    return full, gpu, cpu


def dense_moe(layer_pool, expert_bytes, dtype, d, f, E, gates, hidden_bf16) -> np.ndarray:
    layer_pool = np.ascontiguousarray(layer_pool).view(np.uint8).reshape(-1)
    gates = np.ascontiguousarray(gates, dtype=np.float64)
    hid = np.ascontiguousarray(hidden_bf16, dtype=np.uint16)
    T = hid.shape[0]
    out = np.empty((T, d), dtype=np.float64)
    _check(_l().or_dense_moe(_p(layer_pool), expert_bytes, dtype, d, f, T, E, _p(gates), _p(hid), _p(out)),
           "or_dense_moe")
    return out


# ---------------------------------------------------------------- tolerances

def max_rel_err(y: np.ndarray, ref: np.ndarray) -> float:
    """max_i |y_i - ref_i| / max(|ref_i|, rms(ref)) -- the rms floor keeps near-zero
    reference entries from dominating."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    den = np.maximum(np.abs(ref), rms)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(np.abs(y - ref) / den)) if ref.size else 0.0


def normwise_err(y: np.ndarray, ref: np.ndarray) -> float:
    """||y - ref||_2 / ||ref||_2."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    n = float(np.linalg.norm(ref))
    return float(np.linalg.norm(y - ref)) / n if n > 0 else float(np.linalg.norm(y - ref))


# ------------------------------------------------------- run-time r = BP/BH

def adapt_ratio_trace(bp, bh, alpha: float, r_den: int = 256, r_num_max: int = 256 * 64) -> np.ndarray:
    """r_num after each measurement window of (BP, BH) samples (<= 0 = none);
    -1 until both have a sample.  See or_adapt_ratio."""
    bp = np.ascontiguousarray(bp, dtype=np.float64)
    bh = np.ascontiguousarray(bh, dtype=np.float64)
    assert bp.shape == bh.shape
    out = np.empty(bp.size, dtype=np.int32)
    _check(_l().or_adapt_ratio(bp.size, _p(bp), _p(bh), float(alpha), r_den, r_num_max, _p(out)), "or_adapt_ratio")
    return out
