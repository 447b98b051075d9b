"""The C-ABI library builds, loads, and exports every entry point that
include/pa.h declares (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pa.h"), encoding="utf-8").read()
    return re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", src)


def test_header_declares_the_entry_points():
    names = set(_declared())
    assert {"pa_reshape_and_cache", "pa_decode", "pa_copy_blocks",
            "pa_decode_workspace_size", "pa_status_string"} <= names


def test_library_loads_and_exports_every_declared_symbol():
    from paged_kv_cache_54_gb300 import build as B
    if not os.path.exists(B.LIB):
        B.build()
    lib = ctypes.CDLL(B.LIB)
    for name in _declared():
        assert hasattr(lib, name), name
    import paged_kv_cache_54_gb300 as pa
    assert set(pa.EXPORTED) == set(_declared())
    lib = pa.load_library()
    assert pa.pa_status_string(0) == "ok"


def test_host_validation_needs_no_gpu():
    import paged_kv_cache_54_gb300 as pa
    lib = pa.load_library()
    # sizes the library rejects return 0 workspace bytes
    assert lib.pa_decode_workspace_size(4, 4, 4, 64, 100, 0) > 0
    assert lib.pa_decode_workspace_size(4, 4, 4, 64, 100, 100) == 0   # not a multiple of 64
    assert lib.pa_decode_workspace_size(-1, 4, 4, 64, 100, 0) == 0
    # a null cache description is rejected before any CUDA call
    st = lib.pa_copy_blocks(None, None, None, None, 1, None, None)
    assert st == 1
    desc = pa.PaCacheDesc(16, 2, 16, 64, 0, 1.0, 1.0)
    assert lib.pa_copy_blocks(None, None, ctypes.byref(desc), None, 0, None, None) == 0
    assert lib.pa_copy_blocks(None, None, ctypes.byref(desc), None, 3, None, None) == 1
    bad = pa.PaCacheDesc(16, 2, 24, 64, 0, 1.0, 1.0)   # block size outside the supported set
    assert lib.pa_reshape_and_cache(16, 16, 0, 8, 1, 16, 16, ctypes.byref(bad), None, None) == 2


def test_partition_size_choice_is_deterministic():
    import paged_kv_cache_54_gb300 as pa
    a = pa.pa_decode_workspace_size(64, 32, 32, 128, 4096)
    b = pa.pa_decode_workspace_size(64, 32, 32, 128, 4096)
    assert a == b > 0


def test_scale_descriptions_are_validated_on_the_host():
    import paged_kv_cache_54_gb300 as pa
    lib = pa.load_library()

    def rc(desc):   # zero tokens: only the description is checked
        return lib.pa_reshape_and_cache(16, 16, 0, 8, 0, 16, 16, ctypes.byref(desc), None, None)

    assert rc(pa.PaCacheDesc(16, 2, 16, 64, pa.PA_INT8, 0.05, 0.05)) == 0
    assert rc(pa.PaCacheDesc(16, 2, 16, 64, pa.PA_INT8, 0.05, 0.05, 4096, 8192)) == 0
    assert rc(pa.PaCacheDesc(16, 2, 16, 64, 5, 1.0, 1.0)) == 1          # unknown dtype
    assert rc(pa.PaCacheDesc(16, 2, 16, 64, pa.PA_INT8, 0.0, 1.0)) == 1  # scale must be > 0
    assert rc(pa.PaCacheDesc(16, 2, 16, 64, pa.PA_INT8, 1.0, 1.0, 4096, None)) == 1  # K without V
    assert rc(pa.PaCacheDesc(16, 2, 16, 64, pa.PA_FP8_E4M3, 1.0, 1.0, 4098, 8192)) == 1  # misaligned
    assert rc(pa.PaCacheDesc(16, 2, 16, 64, pa.PA_F16, 1.0, 1.0, 4096, 8192)) == 1  # 16-bit: no scales


def test_binding_marshals_per_head_scales():
    import torch
    import paged_kv_cache_54_gb300 as pa
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.uint8)
    d = pa.cache_desc(kc, "int8", 0.25, 0.5)
    assert (d.dtype, d.k_scale, d.v_scale, d.k_head_scales, d.v_head_scales) == (4, 0.25, 0.5, None, None)
    with pytest.raises(ValueError):   # per-head scales must live on the device
        pa.cache_desc(kc, "int8", torch.ones(2), torch.ones(2))
    assert pa.cache_desc(torch.zeros((4, 2, 16, 64), dtype=torch.int8)).dtype == pa.PA_INT8
