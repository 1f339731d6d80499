"""The C-ABI library loads and exports every symbol its header declares (no GPU)."""
import ctypes
import os
import re

import pytest

import expert_cache_host_gb300 as ft
from expert_cache_host_gb300 import build as ftbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ftbuild.build()
    return ft.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "ft_moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ft_[a-z_]+)\s*\(", src)))


def test_header_declares_the_four_calls():
    names = header_functions()
    for n in ("ft_moe_init", "ft_cache_step", "ft_moe_forward", "ft_cache_rebuild"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert set(names) == set(ft.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_bad_config_rejected_on_host(lib):
    pool = (ctypes.c_uint8 * 16)()
    for bad in (dict(num_experts=0), dict(top_k=3, num_experts=2), dict(hidden=100), dict(inter=96),
                dict(num_slots=0), dict(k_max=0), dict(t_max=0), dict(r_den=0), dict(dtype=7),
                dict(prefill_buffers=3)):
        cfg = ft.make_config(**bad)
        with pytest.raises(ft.FtError) as ei:
            ft.ft_moe_init(cfg, ctypes.addressof(pool), 16)
        assert ei.value.code == ft.FT_E_ARG, bad


def test_mxfp4_prefill_shape_rejected_on_host(lib):
    """MXFP4 prefill GEMMs read the scales of 8 K steps per TMA box: hidden and
    inter must be multiples of 512."""
    pool = (ctypes.c_uint8 * 16)()
    for shape in (dict(hidden=768, inter=512), dict(hidden=512, inter=384)):
        cfg = ft.make_config(dtype=ft.FT_DTYPE_MXFP4, prefill_buffers=2, prefill_t_max=64, **shape)
        with pytest.raises(ft.FtError) as ei:
            ft.ft_moe_init(cfg, ctypes.addressof(pool), 16)
        assert ei.value.code == ft.FT_E_UNSUPPORTED, shape


def test_small_pool_rejected(lib):
    pool = (ctypes.c_uint8 * 16)()
    cfg = ft.make_config()
    with pytest.raises(ft.FtError) as ei:
        ft.ft_moe_init(cfg, ctypes.addressof(pool), 16)
    assert ei.value.code == ft.FT_E_ARG and "pool_bytes" in str(ei.value)


def test_route_shape_rejected_on_host(lib):
    with pytest.raises(ft.FtError) as ei:
        ft.ft_route(8, 4, 2000, 2, 8, 8)
    assert ei.value.code == ft.FT_E_ARG


def test_host_alloc_arguments_checked_on_host(lib):
    import ctypes
    p = ctypes.c_void_p()
    assert lib.ft_host_alloc(0, ctypes.byref(p)) == ft.FT_E_ARG
    assert lib.ft_host_alloc(4096, None) == ft.FT_E_ARG
    assert lib.ft_host_free(None) == ft.FT_OK


def test_set_ratio_arguments_checked_on_host(lib):
    assert lib.ft_set_ratio(None, 1, 1, None) == ft.FT_E_ARG


def test_cpu_executor_arguments_checked_on_host(lib):
    assert lib.ft_cpu_executor(None, 4) == ft.FT_E_ARG
    null = None
    assert lib.ft_cpu_experts(null, 8, 2, 256, 128, 0, 0, 1, null, null, null, null, null, 1) == ft.FT_E_ARG
    assert "null" in lib.ft_last_error().decode()
