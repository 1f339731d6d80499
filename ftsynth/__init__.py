"""Seeded synthetic inputs shared by the CUDA library's tests/bench and the oracle.

Nothing here computes any part of the MoE expert-cache method: this module
only draws weights, hidden-state streams, router logits and route streams.
Every draw is a pure function of (seed, tensor id, layer, expert/sequence,
element index) through Philox4x32-10, so one expert can be regenerated on its
own and the CUDA path and the oracle always see the same bytes.

Tensor ids: 1/2/3 gate/up/down bf16 weights, 4 router weights, 5 decode
innovations, 6 prefill hidden, 7/8/9 MXFP4 codes, 10/11/12 MXFP4 scales,
13 test partial sums, 14 test logits, 15/16 Zipf ranks/noise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libftsynth.so")
_SRCS = [os.path.join(_HERE, "synth.c"), os.path.join(_HERE, "zipf.c")]
_lock = threading.Lock()
_lib = None

DTYPE_BF16 = 0
DTYPE_MXFP4 = 1

T_GATE, T_UP, T_DOWN, T_ROUTER, T_INNOV, T_PREFILL, T_PARTIAL, T_LOGITS = 1, 2, 3, 4, 5, 6, 13, 14


def build(force: bool = False) -> str:
    """Compile the generator library with gcc (portable C, no arch flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(s) for s in _SRCS)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o", tmp, *_SRCS, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _l():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u32, u64, i32, dbl, vp = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.ftsynth_philox4x32_10.argtypes = [vp, vp, vp]
            lib.ftsynth_normal_f64.argtypes = [u32, u32, u32, u32, u64, u64, dbl, vp]
            lib.ftsynth_normal_bf16.argtypes = [u32, u32, u32, u32, u64, u64, dbl, vp]
            lib.ftsynth_bytes.argtypes = [u32, u32, u32, u32, u64, u64, vp]
            lib.ftsynth_scale_bytes.argtypes = [u32, u32, u32, u32, u64, u64, u32, u32, vp]
            lib.ftsynth_ar1_bf16.argtypes = [u32, u32, u32, u32, u64, u64, dbl, vp]
            lib.ftsynth_fill_pool.argtypes = [u32, i32, i32, i32, i32, i32, i32, dbl, u64, vp, i32]
            lib.ftsynth_fill_pool.restype = i32
            lib.ftsynth_normal_bf16_par.argtypes = [u32, u32, u32, u32, u64, u64, dbl, vp, i32]
            lib.ftsynth_normal_bf16_par.restype = i32
            lib.ftsynth_zipf_ranks.argtypes = [u32, u32, i32, vp]
            lib.ftsynth_zipf_routes.argtypes = [u32, i32, i32, i32, i32, dbl, u64, u64, vp, i32]
            lib.ftsynth_zipf_routes.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def _threads(n: int | None) -> int:
    return int(n) if n else (os.cpu_count() or 1)


# ---------------------------------------------------------------- primitives

def philox4x32_10(counter, key) -> np.ndarray:
    c = np.asarray(counter, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _l().ftsynth_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def normal_f64(seed, tensor, a, b, n, std=1.0, offset=0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _l().ftsynth_normal_f64(seed, tensor, a, b, offset, n, std, _ptr(out))
    return out


def normal_bf16(seed, tensor, a, b, n, std=1.0, offset=0) -> np.ndarray:
    """bf16 bit patterns (uint16) of bf16(float(std * z))."""
    out = np.empty(n, dtype=np.uint16)
    _l().ftsynth_normal_bf16(seed, tensor, a, b, offset, n, std, _ptr(out))
    return out


def normal_bf16_rows(seed, tensor, a, b, rows, cols, std=1.0, threads=None) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.uint16)
    _l().ftsynth_normal_bf16_par(seed, tensor, a, b, rows, cols, std, _ptr(out), _threads(threads))
    return out


def uniform_bytes(seed, tensor, a, b, n, offset=0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    _l().ftsynth_bytes(seed, tensor, a, b, offset, n, _ptr(out))
    return out


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even narrowing of float32 to bf16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


# ---------------------------------------------------------------- workloads

def expert_bytes(d: int, f: int, dtype: int) -> int:
    """Bytes of one expert in the canonical layout: bf16 6df; MXFP4 3df/2 + 3df/32."""
    if dtype == DTYPE_BF16:
        return 6 * d * f
    return 3 * d * f // 2 + 3 * d * f // 32


def fill_pool(pool: np.ndarray, seed: int, L: int, E: int, d: int, f: int, dtype: int,
              std: float = 0.02, first_layer: int = 0, threads=None) -> np.ndarray:
    """Write layers first_layer .. first_layer+L-1 into a uint8 host array of L*E*B_x bytes."""
    bx = expert_bytes(d, f, dtype)
    assert pool.dtype == np.uint8 and pool.size >= L * E * bx
    rc = _l().ftsynth_fill_pool(seed, first_layer, L, E, d, f, dtype, std, bx, _ptr(pool), _threads(threads))
    assert rc == 0
    return pool


def make_pool(seed, L, E, d, f, dtype, std=0.02, threads=None, out: np.ndarray | None = None) -> np.ndarray:
    """Generate the pool into `out` (a uint8 array of at least L*E*B_x bytes,
    e.g. a view of pinned host memory) or into a new pageable array."""
    n = L * E * expert_bytes(d, f, dtype)
    pool = np.empty(n, dtype=np.uint8) if out is None else out[:n]
    return fill_pool(pool, seed, L, E, d, f, dtype, std, 0, threads)


def router_weights(seed, L, E, d, std=0.02) -> np.ndarray:
    """[L, E, d] bf16 bit patterns; layer l is stream (seed, 4, l, 0)."""
    return np.stack([normal_bf16(seed, T_ROUTER, l, 0, E * d, std).reshape(E, d) for l in range(L)])


def ar1_hidden(seed, layer, seq, steps, d, rho=0.9) -> np.ndarray:
    """[steps, d] bf16 AR(1) stream h_0 = eps_0, h_t = rho h_{t-1} + eps_t, eps ~ N(0, I)."""
    out = np.empty((steps, d), dtype=np.uint16)
    _l().ftsynth_ar1_bf16(seed, T_INNOV, layer, seq, steps, d, rho, _ptr(out))
    return out


def decode_hidden(seed, L, steps, d, batch=1, rho=0.9) -> np.ndarray:
    """[steps, L, batch, d] bf16: one AR(1) stream per (layer, sequence)."""
    out = np.empty((steps, L, batch, d), dtype=np.uint16)
    for l in range(L):
        for b in range(batch):
            out[:, l, b, :] = ar1_hidden(seed, l, b, steps, d, rho)
    return out


def prefill_hidden(seed, layer, T, d, threads=None) -> np.ndarray:
    """[T, d] bf16 iid N(0, 1) for one layer of a prefill chunk."""
    return normal_bf16_rows(seed, T_PREFILL, layer, 0, T, d, 1.0, threads)


def router_logits(hidden_bf16: np.ndarray, wr_bf16: np.ndarray) -> np.ndarray:
    """float32 logits = bf16(h) . W_r^T, computed once by the harness (fp32 matmul).

    hidden_bf16 [..., d], wr_bf16 [E, d] -> [..., E] float32.  The logits are an
    input of the path: the CUDA library and the oracle receive the same array.
    """
    h = bf16_to_f32(hidden_bf16)
    w = bf16_to_f32(wr_bf16)
    return np.ascontiguousarray(np.matmul(h, w.T, dtype=np.float32))


def zipf_ranks(seed, layer, E) -> np.ndarray:
    out = np.empty(E, dtype=np.int32)
    _l().ftsynth_zipf_ranks(seed, layer, E, _ptr(out))
    return out


def zipf_routes(seed, layer, E, T, k, s, step0, nsteps, threads=None) -> np.ndarray:
    """[nsteps, T, k] int32 local expert ids, Zipf(s) without replacement."""
    out = np.empty((nsteps, T, k), dtype=np.int32)
    rc = _l().ftsynth_zipf_routes(seed, layer, E, T, k, s, step0, nsteps, _ptr(out), _threads(threads))
    assert rc == 0
    return out


def test_partial(seed, T, d, std=0.05) -> np.ndarray:
    """[T, d] float32 values used as an externally supplied partial sum in tests."""
    return normal_f64(seed, T_PARTIAL, 0, 0, T * d, std).astype(np.float32).reshape(T, d)


def test_logits(seed, layer, T, E, std=1.0) -> np.ndarray:
    return normal_f64(seed, T_LOGITS, layer, 0, T * E, std).astype(np.float32).reshape(T, E)
