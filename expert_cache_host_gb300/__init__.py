"""Python binding of libftmoe.so, the GB300 MoE expert-cache layer step.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  The functions carry the C names (ft_moe_init, ft_cache_step,
ft_moe_forward, ft_cache_rebuild, ...) and take plain integers for device and
host pointers (e.g. torch's tensor.data_ptr() and
torch.cuda.current_stream().cuda_stream).  Errors raise FtError with the
library's message.  If the compiled library is missing, the first call raises
ImportError: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libftmoe.so")

FT_OK, FT_E_ARG, FT_E_PIN, FT_E_NOMEM, FT_E_CUDA, FT_E_STATE, FT_E_UNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
FT_ST_ROUTE_RANGE, FT_ST_NAN, FT_ST_CLOCK_WRAP, FT_ST_BAD_SLOT = 1, 2, 4, 8
FT_DTYPE_BF16, FT_DTYPE_MXFP4 = 0, 1
FT_DECODE_CACHED, FT_PREFILL_LAYER = 0, 1
FT_FILL_KERNEL, FT_FILL_COPY_ENGINE = 0, 1
FT_FILL_ORDER_ID, FT_FILL_ORDER_MOST_ROUTED = 0, 1
FT_DECODE_FUSED, FT_DECODE_SPLIT = 0, 1
COUNTS = ("n", "hits", "m", "q", "cpu", "n_groups", "now")

# Every symbol include/ft_moe.h declares.
EXPORTS = (
    "ft_moe_init", "ft_moe_destroy", "ft_cache_step", "ft_cache_control", "ft_moe_forward", "ft_cache_rebuild",
    "ft_get_status", "ft_get_counters", "ft_get_table", "ft_slot_ptr", "ft_get_epoch", "ft_num_slots", "ft_route",
    "ft_profile_enable", "ft_profile_read", "ft_decode_experts_noalloc", "ft_host_alloc", "ft_host_free", "ft_set_ratio",
    "ft_cache_rebuild_retain", "ft_cpu_executor", "ft_cpu_experts",
    "ft_ratio_adapter_init", "ft_ratio_adapter_update", "ft_report_host_rate", "ft_measured_bandwidths",
    "ft_adapt_ratio", "ft_decode_meters", "ft_decode_path",
    "ft_last_error",
)
FT_K_ROUTE, FT_K_CONTROL, FT_K_FILL, FT_K_EXPERTS, FT_K_MERGE, FT_K_UPLOAD, FT_K_PREFILL, FT_K_GEMM, FT_K_CPU = range(9)
FT_K_COUNT = 9
KERNEL_CLASSES = ("route", "control", "fill", "experts", "merge", "upload", "prefill", "gemm", "cpu")


class FtError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class ft_config(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("num_slots", ctypes.c_int32), ("k_max", ctypes.c_int32), ("t_max", ctypes.c_int32),
        ("r_num", ctypes.c_int32), ("r_den", ctypes.c_int32), ("prefill_buffers", ctypes.c_int32),
        ("prefill_t_max", ctypes.c_int32), ("fill_mode", ctypes.c_int32), ("fill_order", ctypes.c_int32),
        ("decode_path", ctypes.c_int32), ("fill_ctas", ctypes.c_int32), ("reserved", ctypes.c_int32 * 1),
    ]


class ft_ratio_adapter(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_double), ("r_den", ctypes.c_int32), ("r_num_max", ctypes.c_int32),
                ("bp_gbs", ctypes.c_double), ("bh_gbs", ctypes.c_double), ("r_num", ctypes.c_int32),
                ("updates", ctypes.c_int32)]


class ft_step_out(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "ids", "weights", "slot_ids", "uniq", "hit_list", "fetch", "victims", "evicted", "cpu_list", "counts")]


_lib = None
_lock = threading.Lock()


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled library (build it with expert_cache_host_gb300.build.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"libftmoe.so not built at {p}; run expert_cache_host_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i32, sz, u32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
        sig = {
            "ft_moe_init": ([ctypes.POINTER(ft_config), vp, sz, ctypes.POINTER(vp)], i32),
            "ft_moe_destroy": ([vp], i32),
            "ft_cache_step": ([vp, i32, vp, i32, ctypes.POINTER(ft_step_out), vp], i32),
            "ft_cache_control": ([vp, i32, vp, i32, ctypes.POINTER(ft_step_out), vp], i32),
            "ft_moe_forward": ([vp, i32, i32, vp, vp, i32, vp, vp, vp], i32),
            "ft_cache_rebuild": ([vp, i32], i32),
            "ft_get_status": ([vp, u32p, i32], i32),
            "ft_get_counters": ([vp, vp], i32),
            "ft_get_table": ([vp, vp, vp, vp, vp], i32),
            "ft_slot_ptr": ([vp, i32], vp),
            "ft_get_epoch": ([vp], i32),
            "ft_num_slots": ([vp], i32),
            "ft_route": ([vp, i32, i32, i32, vp, vp, vp, vp], i32),
            "ft_profile_enable": ([vp, i32], i32),
            "ft_profile_read": ([vp, vp, vp, i32], i32),
            "ft_decode_experts_noalloc": ([vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp], i32),
            "ft_host_alloc": ([sz, ctypes.POINTER(vp)], i32),
            "ft_set_ratio": ([vp, i32, i32, vp], i32),
            "ft_cache_rebuild_retain": ([vp, i32], i32),
            "ft_cpu_executor": ([vp, i32], i32),
            "ft_cpu_experts": ([vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i32], i32),
            "ft_host_free": ([vp], i32),
            "ft_ratio_adapter_init": ([ctypes.POINTER(ft_ratio_adapter), ctypes.c_double, i32, i32], i32),
            "ft_ratio_adapter_update": ([ctypes.POINTER(ft_ratio_adapter), ctypes.c_double, ctypes.c_double], i32),
            "ft_report_host_rate": ([vp, ctypes.c_double, ctypes.c_double], i32),
            "ft_measured_bandwidths": ([vp, vp, vp, i32], i32),
            "ft_adapt_ratio": ([vp, ctypes.POINTER(ft_ratio_adapter), vp, vp], i32),
            "ft_decode_meters": ([vp, vp, i32], i32),
            "ft_decode_path": ([vp], i32),
            "ft_last_error": ([], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _chk(rc: int) -> int:
    if rc != FT_OK:
        raise FtError(rc, load().ft_last_error().decode(errors="replace"))
    return rc


def make_config(**kw) -> ft_config:
    c = ft_config()
    defaults = dict(num_layers=1, num_experts=16, top_k=2, hidden=256, inter=128, dtype=FT_DTYPE_BF16, num_slots=8,
                    k_max=16, t_max=1, r_num=1, r_den=1, prefill_buffers=0, prefill_t_max=0, fill_mode=FT_FILL_KERNEL,
                    fill_order=FT_FILL_ORDER_ID)
    defaults.update(kw)
    for k, v in defaults.items():
        setattr(c, k, int(v))
    return c


def ft_moe_init(cfg: ft_config, host_pool_ptr: int, pool_bytes: int) -> int:
    ctx = ctypes.c_void_p()
    _chk(load().ft_moe_init(ctypes.byref(cfg), ctypes.c_void_p(host_pool_ptr), pool_bytes, ctypes.byref(ctx)))
    return ctx.value


def ft_moe_destroy(ctx: int) -> None:
    _chk(load().ft_moe_destroy(ctypes.c_void_p(ctx)))


def ft_cache_step(ctx: int, layer: int, logits_ptr: int, T: int, stream: int = 0) -> ft_step_out:
    out = ft_step_out()
    _chk(load().ft_cache_step(ctypes.c_void_p(ctx), layer, ctypes.c_void_p(logits_ptr), T, ctypes.byref(out),
                              ctypes.c_void_p(stream)))
    return out


def ft_cache_control(ctx: int, layer: int, ids_ptr: int, T: int, stream: int = 0) -> ft_step_out:
    out = ft_step_out()
    _chk(load().ft_cache_control(ctypes.c_void_p(ctx), layer, ctypes.c_void_p(ids_ptr), T, ctypes.byref(out),
                                 ctypes.c_void_p(stream)))
    return out


def ft_moe_forward(ctx: int, layer: int, mode: int, logits_ptr: int, hidden_ptr: int, T: int, partial_ptr: int,
                   out_ptr: int, stream: int = 0) -> None:
    _chk(load().ft_moe_forward(ctypes.c_void_p(ctx), layer, mode, ctypes.c_void_p(logits_ptr or None),
                               ctypes.c_void_p(hidden_ptr), T, ctypes.c_void_p(partial_ptr or None),
                               ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream)))


def ft_cache_rebuild(ctx: int, new_slots: int) -> None:
    _chk(load().ft_cache_rebuild(ctypes.c_void_p(ctx), new_slots))


def ft_cache_rebuild_retain(ctx: int, new_slots: int) -> None:
    _chk(load().ft_cache_rebuild_retain(ctypes.c_void_p(ctx), new_slots))


def ft_get_status(ctx: int, clear: bool = False) -> int:
    v = ctypes.c_uint32()
    _chk(load().ft_get_status(ctypes.c_void_p(ctx), ctypes.byref(v), int(clear)))
    return v.value


def ft_get_counters(ctx: int, num_layers: int):
    import numpy as np
    a = np.zeros((num_layers, 6), dtype=np.uint64)
    _chk(load().ft_get_counters(ctypes.c_void_p(ctx), ctypes.c_void_p(a.ctypes.data)))
    return a


def ft_get_table(ctx: int, E_tot: int, S: int):
    """(slot_of int32 [E_tot], expert_of int32 [S], last_use uint32 [S], now int)."""
    import numpy as np
    so = np.empty(E_tot, dtype=np.int32)
    eo = np.empty(S, dtype=np.int32)
    lu = np.empty(S, dtype=np.uint32)
    now = np.empty(1, dtype=np.uint32)
    _chk(load().ft_get_table(ctypes.c_void_p(ctx), ctypes.c_void_p(so.ctypes.data), ctypes.c_void_p(eo.ctypes.data),
                             ctypes.c_void_p(lu.ctypes.data), ctypes.c_void_p(now.ctypes.data)))
    return so, eo, lu, int(now[0])


def ft_slot_ptr(ctx: int, slot: int) -> int:
    return load().ft_slot_ptr(ctypes.c_void_p(ctx), slot) or 0


def ft_set_ratio(ctx: int, r_num: int, r_den: int, stream: int = 0) -> None:
    _chk(load().ft_set_ratio(ctypes.c_void_p(ctx), r_num, r_den, ctypes.c_void_p(stream)))


def ft_ratio_adapter_init(alpha: float, r_den: int = 256, r_num_max: int = 256 * 64) -> ft_ratio_adapter:
    a = ft_ratio_adapter()
    _chk(load().ft_ratio_adapter_init(ctypes.byref(a), alpha, r_den, r_num_max))
    return a


def ft_ratio_adapter_update(a: ft_ratio_adapter, bp_gbs: float, bh_gbs: float) -> int:
    """1 if r_num changed, 0 if not."""
    rc = load().ft_ratio_adapter_update(ctypes.byref(a), bp_gbs, bh_gbs)
    if rc < 0:
        _chk(rc)
    return rc


def ft_report_host_rate(ctx: int, nbytes: float, seconds: float) -> None:
    _chk(load().ft_report_host_rate(ctypes.c_void_p(ctx), nbytes, seconds))


def ft_measured_bandwidths(ctx: int, reset: bool = False):
    """(BP, BH) in GB/s measured since the last reset (0 = no sample)."""
    bp, bh = ctypes.c_double(), ctypes.c_double()
    _chk(load().ft_measured_bandwidths(ctypes.c_void_p(ctx), ctypes.byref(bp), ctypes.byref(bh), int(reset)))
    return bp.value, bh.value


def ft_decode_meters(ctx: int, reset: bool = False) -> dict:
    """Device-side decode meters since the last reset: fill bytes / seconds /
    launches and resident-expert bytes / seconds / launches (fused path)."""
    a = (ctypes.c_double * 6)()
    _chk(load().ft_decode_meters(ctypes.c_void_p(ctx), a, int(reset)))
    return dict(fill_bytes=a[0], fill_s=a[1], fill_launches=int(a[2]), resident_bytes=a[3], resident_s=a[4],
                resident_launches=int(a[5]))


def ft_decode_path(ctx: int) -> int:
    rc = load().ft_decode_path(ctypes.c_void_p(ctx))
    if rc < 0:
        _chk(rc)
    return rc


def ft_adapt_ratio(ctx: int, a: ft_ratio_adapter, stream: int = 0) -> int:
    """One adaptation step; 1 if r changed (and was set on `stream`), else 0."""
    ch = ctypes.c_int()
    _chk(load().ft_adapt_ratio(ctypes.c_void_p(ctx), ctypes.byref(a), ctypes.c_void_p(stream), ctypes.byref(ch)))
    return ch.value


def ft_cpu_executor(ctx: int, threads: int) -> None:
    """Enable (threads >= 1) or disable (0) the context's CPU expert executor."""
    _chk(load().ft_cpu_executor(ctypes.c_void_p(ctx), threads))


def ft_cpu_experts(pool, num_experts: int, top_k: int, hidden: int, inter: int, dtype: int, layer: int,
                   ids, weights, slot_ids, hidden_rows, threads: int = 1):
    """The executor's sum over the routes with slot id < 0, on host numpy
    arrays: returns partial float32 [T, hidden]."""
    import numpy as np
    pool = np.ascontiguousarray(pool).view(np.uint8).reshape(-1)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T = ids.shape[0]
    w = np.ascontiguousarray(weights, dtype=np.float32).reshape(T, top_k)
    sid = np.ascontiguousarray(slot_ids, dtype=np.int32).reshape(T, top_k)
    hid = np.ascontiguousarray(hidden_rows).view(np.uint16).reshape(T, hidden)
    out = np.empty((T, hidden), dtype=np.float32)
    v = ctypes.c_void_p
    _chk(load().ft_cpu_experts(v(pool.ctypes.data), num_experts, top_k, hidden, inter, dtype, layer, T,
                               v(ids.ctypes.data), v(w.ctypes.data), v(sid.ctypes.data), v(hid.ctypes.data),
                               v(out.ctypes.data), threads))
    return out


def ft_get_epoch(ctx: int) -> int:
    return load().ft_get_epoch(ctypes.c_void_p(ctx))


def ft_num_slots(ctx: int) -> int:
    return load().ft_num_slots(ctypes.c_void_p(ctx))


def ft_route(logits_ptr: int, T: int, E: int, k: int, ids_ptr: int, w_ptr: int, status_ptr: int = 0,
             stream: int = 0) -> None:
    _chk(load().ft_route(ctypes.c_void_p(logits_ptr), T, E, k, ctypes.c_void_p(ids_ptr), ctypes.c_void_p(w_ptr),
                         ctypes.c_void_p(status_ptr or None), ctypes.c_void_p(stream)))


def ft_profile_enable(ctx: int, on: bool = True) -> None:
    _chk(load().ft_profile_enable(ctypes.c_void_p(ctx), int(on)))


def ft_profile_read(ctx: int, reset: bool = True) -> dict:
    """{class name: (total ms, launches)} recorded since the last reset."""
    ms = (ctypes.c_double * FT_K_COUNT)()
    n = (ctypes.c_uint64 * FT_K_COUNT)()
    _chk(load().ft_profile_read(ctypes.c_void_p(ctx), ms, n, int(reset)))
    return {name: (ms[i], int(n[i])) for i, name in enumerate(KERNEL_CLASSES)}


def ft_decode_experts_noalloc(arena_ptr: int, num_slots: int, hidden: int, inter: int, top_k: int, T: int,
                              slot_ids_ptr: int, weights_ptr: int, hidden_ptr: int, partial_ptr: int, out_ptr: int,
                              status_ptr: int = 0, stream: int = 0) -> None:
    """Decode experts + merge with no device allocation (scratch is a fixed
    array inside the library; see include/ft_moe.h for the limits)."""
    v = ctypes.c_void_p
    _chk(load().ft_decode_experts_noalloc(v(arena_ptr), num_slots, hidden, inter, top_k, T, v(slot_ids_ptr),
                                          v(weights_ptr), v(hidden_ptr), v(partial_ptr or None), v(out_ptr),
                                          v(status_ptr or None), v(stream)))


class HostPool:
    """Pinned, device-mapped host memory from ft_host_alloc, viewed as a uint8
    numpy array (``.array``).  Free it (``.free()``) only after every context
    using it has been destroyed; the array must not be used afterwards."""

    def __init__(self, nbytes: int):
        import numpy as np
        p = ctypes.c_void_p()
        _chk(load().ft_host_alloc(nbytes, ctypes.byref(p)))
        self.ptr, self.nbytes = p.value, nbytes
        self.array = np.ctypeslib.as_array((ctypes.c_uint8 * nbytes).from_address(self.ptr))

    def free(self) -> None:
        if self.ptr:
            self.array = None
            _chk(load().ft_host_free(ctypes.c_void_p(self.ptr)))
            self.ptr = 0


def ft_last_error() -> str:
    return load().ft_last_error().decode(errors="replace")
