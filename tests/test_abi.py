"""The C-ABI library loads and exports every entry point that include/ekv.h declares;
host-side argument checks that need no GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "ekv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ekv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ["ekv_create", "ekv_destroy", "ekv_paged_decode", "ekv_gather_prefill",
                 "ekv_demote_pages", "ekv_get_error"]:
        assert name in syms


def test_library_exports_every_declared_symbol(ekv_lib):
    lib = ctypes.CDLL(ekv_lib.LIB_PATH)
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, f"not exported: {missing}"
    assert sorted(ekv_lib.EXPORTED) == declared_symbols()


def test_status_strings(ekv_lib):
    s = ekv_lib._lib.ekv_status_string
    assert s(0) == b"EKV_OK" and s(3) == b"EKV_ERR_CAPACITY" and s(99) == b"EKV_UNKNOWN_STATUS"


def test_null_arguments_are_rejected_without_a_gpu(ekv_lib):
    L = ekv_lib._lib
    assert L.ekv_create(None, None) == ekv_lib.EKV_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert L.ekv_create(ctypes.byref(h), None) == ekv_lib.EKV_ERR_INVALID_ARG and h.value is None
    assert L.ekv_paged_decode(None, *([None] * 3), 0, 0, None, 0, None, 0, None, 0, None, 1,
                              ctypes.c_float(0), None, None, None) == ekv_lib.EKV_ERR_INVALID_ARG
    assert L.ekv_demote_pages(None, None, 0, 0, None, 0, None, None, None) == ekv_lib.EKV_ERR_INVALID_ARG
    assert L.ekv_set_pdl(None, 1) == ekv_lib.EKV_ERR_INVALID_ARG
    assert L.ekv_set_decode_variant(None, 0) == ekv_lib.EKV_ERR_INVALID_ARG
    ms = ctypes.c_double(-1.0)
    assert L.ekv_profile_launch_floor(None, 8, None, ctypes.byref(ms)) == ekv_lib.EKV_ERR_INVALID_ARG
    assert ms.value == -1.0
    assert L.ekv_destroy(None) == ekv_lib.EKV_OK


@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 96), (48, 16, 128), (32, 4, 256), (40, 4, 128), (6, 4, 64)])
def test_unsupported_shapes_are_refused_before_any_cuda_call(ekv_lib, hq, hkv, d):
    cfg = ekv_lib.ekv_config(hq, hkv, d, 8)
    h = ctypes.c_void_p()
    assert ekv_lib._lib.ekv_create(ctypes.byref(h), ctypes.byref(cfg)) == ekv_lib.EKV_ERR_UNSUPPORTED


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "mixed_precision_paged_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.findall(r"^\s*(?:from|import)\s+(\w+)", src, flags=re.M)
