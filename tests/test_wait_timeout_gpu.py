"""The bounded pipeline wait, made to run out on purpose in the allowed way.

Every ring wait of the decode gives up after a time bound, reports EKV_DETAIL_TIMEOUT,
lets its own copies in flight land and winds the kernel down, so that no barrier is left
waiting and the context stays usable. Here that path runs on a GPU without any fault: the
test library libekv_waittest.so (built beside libekv.so from the same sources, with the
bound cut to 5 ms) can raise the byte count of one ring barrier's first phase by 16 bytes
that no copy delivers (CTA 0, warp 0, slot 0). The data of every copy still lands and
nothing is left in flight; only that wait runs out. The call must return, ekv_get_error
must report the timeout, and the next calls on the same context must match the oracle
(the tickets of the call that wound down are cleared).
"""

import ctypes
import os
import time

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl

from _helpers import assert_close, oracle_decode, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def waitlib(ekv_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    path = os.path.join(os.path.dirname(ekv_lib.LIB_PATH), "libekv_waittest.so")
    assert os.path.exists(path), "the test library is built with libekv.so"
    lib = ctypes.CDLL(path)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.ekv_create.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(ekv_lib.ekv_config)]
    lib.ekv_destroy.argtypes = [vp]
    lib.ekv_set_pdl.argtypes = [vp, i]
    lib.ekv_paged_decode.argtypes = [vp, vp, vp, vp, ctypes.c_longlong, i, vp, i, vp, i, vp, i, vp, i,
                                     ctypes.c_float, vp, vp, vp]
    lib.ekv_get_error.argtypes = [vp, ctypes.POINTER(i), ctypes.POINTER(i)]
    lib.ekv_test_inject_wait_timeout.argtypes = [i]
    for f in ("ekv_create", "ekv_destroy", "ekv_set_pdl", "ekv_paged_decode", "ekv_get_error",
              "ekv_test_inject_wait_timeout"):
        getattr(lib, f).restype = i
    return lib, torch


def _decode(lib, torch, ctx, case, d, out, lse):
    st = torch.cuda.current_stream().cuda_stream
    s = lib.ekv_paged_decode(ctx, d.q.data_ptr(), d.k_pages.data_ptr(), d.v_pages.data_ptr(), case.v_page_stride,
                             case.num_pages, None if d.v_scales is None else d.v_scales.data_ptr(),
                             case.scale_mode, None if d.page_mode is None else d.page_mode.data_ptr(),
                             case.uniform_mode, d.block_table.data_ptr(), case.block_table.shape[1],
                             d.seq_lens.data_ptr(), case.batch, 0.0, out.data_ptr(), lse.data_ptr(), st)
    assert s == 0


def _error(lib, ctx):
    code, detail = ctypes.c_int(-1), ctypes.c_int(-1)
    assert lib.ekv_get_error(ctx, ctypes.byref(code), ctypes.byref(detail)) == 0
    return code.value, detail.value


@pytest.mark.parametrize("fmt,scale_mode,pdl", [("e4m3", 0, 0), ("mixed", 1, 0), ("mixed", 1, 1)])
def test_wait_runs_out_and_the_context_recovers(ekv_lib, waitlib, fmt, scale_mode, pdl):
    lib, torch = waitlib
    lens = [900, 1, 2500, 37, 610, 1300]
    hq, hkv, d = 32, 8, 128
    case = wl.make_decode_case(lens, hq, hkv, d, v_format=fmt, scale_mode=scale_mode, seed=930,
                               pool_pages=sum((x + 15) // 16 for x in lens) + 3)
    dv = to_device(case)
    cfg = ekv_lib.ekv_config(hq, hkv, d, len(lens))
    ctx = ctypes.c_void_p()
    assert lib.ekv_create(ctypes.byref(ctx), ctypes.byref(cfg)) == 0
    assert lib.ekv_set_pdl(ctx, pdl) == 0
    B = case.batch
    out = torch.empty((B, hq, d), dtype=torch.float16, device="cuda")
    lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    ref_out, ref_lse = oracle_decode(case)
    try:
        _decode(lib, torch, ctx, case, dv, out, lse)       # a clean call first
        assert _error(lib, ctx) == (0, 0)
        assert_close(out, lse, ref_out, ref_lse)
        for _ in range(2):
            assert lib.ekv_test_inject_wait_timeout(1) == 0
            t0 = time.perf_counter()
            _decode(lib, torch, ctx, case, dv, out, lse)
            code, detail = _error(lib, ctx)                # synchronises: the call has returned
            assert time.perf_counter() - t0 < 5.0
            assert (code, detail) == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_TIMEOUT)
            assert _error(lib, ctx) == (0, 0)              # read once, then cleared
            for _ in range(2):                             # the context is usable again
                out.fill_(float("nan"))
                lse.fill_(float("nan"))
                _decode(lib, torch, ctx, case, dv, out, lse)
                assert _error(lib, ctx) == (0, 0)
                assert_close(out, lse, ref_out, ref_lse)
    finally:
        lib.ekv_destroy(ctx)
