"""CPU-side checks of the C ABI library: it builds, loads, exports every
declared symbol, and host-side argument checks answer without a GPU
(no compute call is made here)."""

import ctypes
import os
import re

import numpy as np
import pytest

from int2_rotated_kv_oscar_gb300 import abi, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "oscar.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oscar_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load(build_if_missing=False)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("oscar_kv_append", "oscar_decode_attention", "oscar_load_rotation", "oscar_create",
                     "oscar_destroy", "oscar_decode_workspace_bytes", "oscar_check_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(abi.library_path())
    for name in _declared_functions():
        assert hasattr(raw, name), name
    assert set(_declared_functions()) == set(abi.SIGNATURES)


def test_status_strings(lib):
    assert abi.oscar_status_string(0) == "ok"
    assert "workspace" in abi.oscar_status_string(6)
    assert abi.oscar_status_string(99) == "unknown status"


def test_host_checks_need_no_gpu(lib):
    # null / bad arguments are rejected before any CUDA call
    assert lib.oscar_create(None, None) == 1
    cfg = abi.oscar_config(num_layers=1, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=64, sink=64,
                           recent=256, group=64, device=0)
    h = ctypes.c_void_p()
    assert lib.oscar_create(ctypes.byref(cfg), ctypes.byref(h)) == 1      # head_dim must be 128
    cfg.head_dim = 128
    cfg.num_q_heads = 24                                                   # GQA ratio 12 > 8
    assert lib.oscar_create(ctypes.byref(cfg), ctypes.byref(h)) == 1
    u = np.eye(128, dtype=np.float32)
    assert lib.oscar_load_rotation(None, 0, u.ctypes.data, u.ctypes.data, 1.0, 1.0, 7) == 1
    assert lib.oscar_kv_append(None, 0, None, None, None) == 1
    assert lib.oscar_decode_attention(None, 0, None, None, None, 0, None) == 1
    assert lib.oscar_decode_workspace_bytes(None, 1, 10) == 0
    assert lib.oscar_check_device_error(None, None, None) == 1
    assert lib.oscar_selftest_bounded_wait(None, 1024, None) == 1
    assert lib.oscar_device_sm_count(None) == 0
    # calibration: sizes out of range give 0 bytes, null arguments are rejected
    assert lib.oscar_calib_workspace_bytes(0, 1, 1, 1) == 0
    assert lib.oscar_calib_workspace_bytes(1, 1, 1, (1 << 20) + 1) == 0
    assert lib.oscar_calib_workspace_bytes(2048, 2048, 8, 8 * 2048) >= 8 * 2048 * 128 * 4
    assert lib.oscar_calib_covariances(None, None, 1, None, None, 1, 1, 1.0, None, None, None, 0, None) == 1
    tau = ctypes.c_double(0.0)
    assert lib.oscar_calib_clip_threshold(None, None, 1, u.ctypes.data, 7, 99.9, ctypes.byref(tau), None, 0,
                                          None) == 1
    lib.oscar_destroy(None)


def test_struct_layouts_match_the_header():
    # field order and sizes of the ctypes mirrors (x86-64 / aarch64 LP64 ABI)
    assert ctypes.sizeof(abi.oscar_config) == 9 * 4
    assert abi.oscar_cache_view.batch.offset == 96
    assert abi.oscar_cache_view.recent_page_table.offset == 104 and ctypes.sizeof(abi.oscar_cache_view) == 112
    assert ctypes.sizeof(abi.oscar_append_args) == 8 * 4 + 3 * 4 + 4
    assert ctypes.sizeof(abi.oscar_decode_args) == 3 * 8 + 8


def test_binding_constants_match_the_header():
    # every #define the header gives a C caller (device error bits, flags,
    # block layout, sizes) has the same value in the binding, where it has one
    text = open(HEADER).read()
    defines = dict(re.findall(r"#define\s+(OSCAR_[A-Z0-9_]+)\s+\(?([0-9]+)u?\s*(?:<<\s*([0-9]+))?", text) and
                   [(n, v) for n, v, _ in re.findall(r"#define\s+(OSCAR_[A-Z0-9_]+)\s+\(?([0-9]+)u?\s*(?:<<\s*([0-9]+))?", text)])
    shifts = {n: int(s) for n, _, s in re.findall(r"#define\s+(OSCAR_[A-Z0-9_]+)\s+\(?([0-9]+)u?\s*(?:<<\s*([0-9]+))?", text) if s}
    bits = sorted(n for n in defines if n.startswith("OSCAR_DEVERR_"))
    assert bits == ["OSCAR_DEVERR_LENGTH", "OSCAR_DEVERR_PAGE", "OSCAR_DEVERR_RING", "OSCAR_DEVERR_SINK",
                    "OSCAR_DEVERR_TIMEOUT", "OSCAR_DEVERR_TOKENS"]
    values = []
    for name, v in defines.items():
        value = int(v) << shifts.get(name, 0)
        if hasattr(abi, name):
            assert getattr(abi, name) == value, name
        if name.startswith("OSCAR_DEVERR_"):
            values.append(value)
            assert getattr(abi, name) == value, name  # the binding decodes every bit
    # the error bits are distinct single bits
    assert all(v & (v - 1) == 0 for v in values) and len(set(values)) == len(values)
