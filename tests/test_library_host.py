"""Host-side checks of libdms.so that need no GPU: it builds for sm_103a, loads,
exports every entry point declared in include/dms.h, and rejects bad handles
and arguments without touching the device."""
import ctypes
import os
import re

import pytest
import torch

from learned_kv_cache_eviction_b300 import build, dms

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_entry_points():
    text = open(os.path.join(ROOT, "include", "dms.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dms_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return dms.load_library()


def test_library_exports_every_declared_symbol(lib):
    names = _declared_entry_points()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dms.h but not exported"
    assert sorted(dms.SIGNATURES) == names


def test_error_strings(lib):
    for code in range(0, -7, -1):
        s = lib.dms_error_string(code)
        assert s and s != b"unknown error"
    assert lib.dms_error_string(-99) == b"unknown error"


def test_null_handle_rejected_without_device(lib):
    assert lib.dms_append(None, None, None, None, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_append_chunk(None, None, None, None, 4, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_decode_attention(None, None, None, 1.0, 4, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_cache_lengths(None, None, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_cache_slot_positions(None, None, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_cache_export_kv(None, None, None, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_cache_status(None, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_cache_selftest_wait(None, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_prefill(None, None, None, None, None, 4, None, 1.0, 4, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_cache_export_scales(None, None, None, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_cache_kv_format(None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_step(None, None, None, None, None, None, 1.0, 4, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_step_host(None, None, None, None, None, None, 1.0, 4, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_step_host_join(None, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_step_graph_launch(None, None) == dms.DMS_ERR_BAD_HANDLE
    assert lib.dms_step_graph_create(None, 0, None, None, None, None, None, 1.0, 4) is None
    assert lib.dms_last_error() == dms.DMS_ERR_INVALID_ARG
    lib.dms_step_graph_destroy(None)  # ignored
    assert lib.dms_cache_position(None) == -1
    lib.dms_cache_destroy(None)  # ignored
    fake = ctypes.c_void_p(0x1000)  # never returned by dms_cache_create
    assert lib.dms_append(fake, None, None, None, None) == dms.DMS_ERR_BAD_HANDLE


def test_create_rejects_bad_sizes(lib):
    for args in [(0, 8, 16, 128, 16), (1, 0, 16, 128, 16), (1, 8, 0, 128, 16), (1, 8, 16, 96, 16),
                 (1, 8, 16, 128, 0), (1 << 16, 1 << 10, 1 << 12, 128, 16)]:
        assert lib.dms_cache_create(*args) is None
        assert lib.dms_last_error() == dms.DMS_ERR_INVALID_ARG
    for fmt in (-1, 2, 7):  # unknown storage format
        assert lib.dms_cache_create_ex(1, 8, 16, 128, 16, fmt) is None
        assert lib.dms_last_error() == dms.DMS_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device failure path")
def test_create_without_device_reports_cuda_error(lib):
    assert lib.dms_cache_create(1, 2, 16, 64, 16) is None
    assert lib.dms_last_error() == dms.DMS_ERR_CUDA
    with pytest.raises(RuntimeError):  # DmsError, or torch's own "no driver" error
        dms.DmsCache(1, 2, 16, 64, 16)


def test_binding_refuses_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        saved = dms._lib
        dms._lib = None
        try:
            dms.load_library(str(tmp_path / "libdms.so"))
        finally:
            dms._lib = saved
