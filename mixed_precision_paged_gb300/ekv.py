"""Thin ctypes binding of the ekv C ABI (include/ekv.h).

Argument marshalling only: every step of the decode, gather and demotion runs in the
library's CUDA kernels. Tensors are passed as raw device pointers (``data_ptr()``);
``page_range`` of the gather is a host array. Importing this module fails loudly when
``libekv.so`` is missing: there is no fallback path.
"""

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libekv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"ekv CUDA library not found at {LIB_PATH}; build it with "
        "`python -c 'import __graft_entry__ as g; g.build()'` "
        "(or `python -m mixed_precision_paged_gb300.build`)")

_lib = ctypes.CDLL(LIB_PATH)

EKV_OK = 0
EKV_ERR_INVALID_ARG = 1
EKV_ERR_UNSUPPORTED = 2
EKV_ERR_CAPACITY = 3
EKV_ERR_CUDA = 4
EKV_ERR_DEVICE_CHECK = 5

EKV_MODE_TARGET_FP16 = 0
EKV_MODE_COMPACT_E4M3 = 1
EKV_MODE_BASE = 2
EKV_SCALE_PER_TENSOR = 0
EKV_SCALE_PER_PAGE_HEAD = 1

EKV_DETAIL_NONE = 0
EKV_DETAIL_PAGE_ID = 1
EKV_DETAIL_SCALE = 2
EKV_DETAIL_SEQ_LEN = 3
EKV_DETAIL_NONFINITE_PAGE = 4
EKV_DETAIL_TIMEOUT = 5
EKV_DETAIL_PAGE_MODE = 6

EXPORTED = ["ekv_create", "ekv_destroy", "ekv_paged_decode", "ekv_gather_prefill",
            "ekv_demote_pages", "ekv_get_error", "ekv_profile_enable", "ekv_profile_read",
            "ekv_set_decode_variant", "ekv_query", "ekv_paged_decode_noalloc",
            "ekv_demote_pages_base", "ekv_promote_pages", "ekv_append_kv", "ekv_paged_decode_elastic",
            "ekv_transition_pages", "ekv_prefill_attention", "ekv_gather_prefill_elastic",
            "ekv_set_pdl", "ekv_profile_launch_floor", "ekv_status_string"]


class ekv_config(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("max_batch", ctypes.c_int)]


_vp = ctypes.c_void_p
_i = ctypes.c_int
_ll = ctypes.c_longlong

_lib.ekv_create.argtypes = [ctypes.POINTER(_vp), ctypes.POINTER(ekv_config)]
_lib.ekv_destroy.argtypes = [_vp]
_lib.ekv_paged_decode.argtypes = [_vp, _vp, _vp, _vp, _ll, _i, _vp, _i, _vp, _i, _vp, _i, _vp,
                                  _i, ctypes.c_float, _vp, _vp, _vp]
_lib.ekv_gather_prefill.argtypes = [_vp, _vp, _vp, _ll, _i, _vp, _i, _vp, _i, _vp, _i, _i, _vp,
                                    _i, _vp, _vp, _vp, _i, _i, _vp]
_lib.ekv_gather_prefill_elastic.argtypes = [_vp, _vp, _vp, _ll, _i, _i, _vp, _i, _vp, _i, _vp, _vp, _i, _vp,
                                            _i, _i, _vp, _i, _vp, _vp, _vp, _i, _i, _vp]
_lib.ekv_demote_pages.argtypes = [_vp, _vp, _ll, _i, _vp, _i, _vp, _vp, _vp]
_lib.ekv_demote_pages_base.argtypes = [_vp, _vp, _ll, _i, _vp, _i, _vp, _vp, _vp]
_lib.ekv_promote_pages.argtypes = [_vp, _vp, _ll, _i, _vp, _i, _vp, _vp, _vp]
_lib.ekv_paged_decode_elastic.argtypes = [_vp, _vp, _vp, _vp, _ll, _i, _i, _vp, _i, _vp, _i, _vp, _vp, _i, _vp,
                                          _i, _vp, _i, ctypes.c_float, _vp, _vp, _vp]
_lib.ekv_transition_pages.argtypes = [_vp, _i, _vp, _ll, _i, _i, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp]
_lib.ekv_prefill_attention.argtypes = [_vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, ctypes.c_float, _vp, _vp, _vp]
_lib.ekv_append_kv.argtypes = [_vp, _vp, _vp, _vp, _vp, _ll, _i, _vp, _i, _vp, _i, _vp, _i, _vp, _i, _vp]
_lib.ekv_paged_decode_noalloc.argtypes = [_i, _i, _i, _vp, _vp, _vp, _ll, _i, _vp, _i, _vp, _i, _vp, _i,
                                          _vp, _i, ctypes.c_float, _vp, _vp, _vp, _vp]
_lib.ekv_get_error.argtypes = [_vp, ctypes.POINTER(_i), ctypes.POINTER(_i)]
_lib.ekv_profile_enable.argtypes = [_vp, _i]
_lib.ekv_profile_read.argtypes = [_vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_ll)]
_lib.ekv_profile_launch_floor.argtypes = [_vp, _i, _vp, ctypes.POINTER(ctypes.c_double)]
_lib.ekv_set_decode_variant.argtypes = [_vp, _i]
_lib.ekv_set_pdl.argtypes = [_vp, _i]
_lib.ekv_query.argtypes = [_vp, ctypes.POINTER(_i), ctypes.POINTER(_i)]
_lib.ekv_status_string.argtypes = [_i]
_lib.ekv_status_string.restype = ctypes.c_char_p
for _n in EXPORTED[:-1]:
    getattr(_lib, _n).restype = _i


class EkvError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {_lib.ekv_status_string(status).decode()}")


def _check(status, what):
    if status != EKV_OK:
        raise EkvError(status, what)


def _ptr(x):
    """Device/host address of a tensor or array, an int address, or None -> NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def ekv_create(num_q_heads, num_kv_heads, head_dim, max_batch):
    """Create a context on the current CUDA device; returns its handle (int)."""
    cfg = ekv_config(num_q_heads, num_kv_heads, head_dim, max_batch)
    h = _vp()
    _check(_lib.ekv_create(ctypes.byref(h), ctypes.byref(cfg)), "ekv_create")
    return h.value


def ekv_destroy(ctx):
    _check(_lib.ekv_destroy(ctx), "ekv_destroy")


def ekv_paged_decode(ctx, q, k_pages, v_pages, v_page_stride_bytes, num_pages, v_scales,
                     scale_mode, page_mode, uniform_mode, block_table, block_table_stride,
                     seq_lens, batch, sm_scale, out, lse=None, stream=None):
    _check(_lib.ekv_paged_decode(ctx, _ptr(q), _ptr(k_pages), _ptr(v_pages), v_page_stride_bytes,
                                 num_pages, _ptr(v_scales), scale_mode, _ptr(page_mode),
                                 uniform_mode, _ptr(block_table), block_table_stride,
                                 _ptr(seq_lens), batch, float(sm_scale), _ptr(out), _ptr(lse),
                                 _stream(stream)), "ekv_paged_decode")


def ekv_paged_decode_noalloc(num_q_heads, num_kv_heads, head_dim, q, k_pages, v_pages,
                             v_page_stride_bytes, num_pages, v_scales, scale_mode, page_mode,
                             uniform_mode, block_table, block_table_stride, seq_lens, batch,
                             sm_scale, out, lse=None, err_out=None, stream=None):
    """Decode with no context and no device allocation: the split-K scratch is a fixed
    array inside the library (see include/ekv.h). For callers that may not allocate
    device memory on this path."""
    _check(_lib.ekv_paged_decode_noalloc(num_q_heads, num_kv_heads, head_dim, _ptr(q), _ptr(k_pages),
                                         _ptr(v_pages), v_page_stride_bytes, num_pages, _ptr(v_scales),
                                         scale_mode, _ptr(page_mode), uniform_mode, _ptr(block_table),
                                         block_table_stride, _ptr(seq_lens), batch, float(sm_scale),
                                         _ptr(out), _ptr(lse), _ptr(err_out), _stream(stream)),
           "ekv_paged_decode_noalloc")


def ekv_gather_prefill(ctx, k_pages, v_pages, v_page_stride_bytes, num_pages, v_scales,
                       scale_mode, page_mode, uniform_mode, block_table, block_table_stride,
                       block_table_rows, page_range, ws_k, ws_v, ws_indices, ws_pages,
                       apply_scale=1, stream=None):
    pr = np.ascontiguousarray(np.asarray(page_range, dtype=np.int32).reshape(-1, 3))
    _check(_lib.ekv_gather_prefill(ctx, _ptr(k_pages), _ptr(v_pages), v_page_stride_bytes,
                                   num_pages, _ptr(v_scales), scale_mode, _ptr(page_mode),
                                   uniform_mode, _ptr(block_table), block_table_stride,
                                   block_table_rows, pr.ctypes.data, pr.shape[0], _ptr(ws_k),
                                   _ptr(ws_v), _ptr(ws_indices), ws_pages, int(apply_scale),
                                   _stream(stream)), "ekv_gather_prefill")


def ekv_gather_prefill_elastic(ctx, k_pages, v_pages, v_page_stride_bytes, num_pages, num_v_slots,
                               v_scales, scale_mode, page_mode, uniform_mode, block_table, v_block_table,
                               block_table_stride, boundaries, has_base, block_table_rows, page_range,
                               ws_k, ws_v, ws_indices, ws_pages, apply_scale=1, stream=None):
    pr = np.ascontiguousarray(np.asarray(page_range, dtype=np.int32).reshape(-1, 3))
    _check(_lib.ekv_gather_prefill_elastic(ctx, _ptr(k_pages), _ptr(v_pages), v_page_stride_bytes,
                                           num_pages, num_v_slots, _ptr(v_scales), scale_mode,
                                           _ptr(page_mode), uniform_mode, _ptr(block_table),
                                           _ptr(v_block_table), block_table_stride, _ptr(boundaries),
                                           int(has_base), block_table_rows, pr.ctypes.data, pr.shape[0],
                                           _ptr(ws_k), _ptr(ws_v), _ptr(ws_indices), ws_pages,
                                           int(apply_scale), _stream(stream)), "ekv_gather_prefill_elastic")


def ekv_demote_pages(ctx, v_pages, v_page_stride_bytes, num_pages, page_ids, n, page_mode,
                     scale_out, stream=None):
    _check(_lib.ekv_demote_pages(ctx, _ptr(v_pages), v_page_stride_bytes, num_pages,
                                 _ptr(page_ids), n, _ptr(page_mode), _ptr(scale_out),
                                 _stream(stream)), "ekv_demote_pages")


def ekv_demote_pages_base(ctx, v_pages, v_page_stride_bytes, num_pages, page_ids, n, page_mode,
                          low_out=None, stream=None):
    """TARGET -> BASE in place; row i of ``low_out`` receives page_ids[i]'s low bytes."""
    _check(_lib.ekv_demote_pages_base(ctx, _ptr(v_pages), v_page_stride_bytes, num_pages,
                                      _ptr(page_ids), n, _ptr(page_mode), _ptr(low_out),
                                      _stream(stream)), "ekv_demote_pages_base")


def ekv_promote_pages(ctx, v_pages, v_page_stride_bytes, num_pages, page_ids, n, page_mode, low_in,
                      stream=None):
    """BASE -> TARGET in place from the low bytes ``low_in`` (row i for page_ids[i])."""
    _check(_lib.ekv_promote_pages(ctx, _ptr(v_pages), v_page_stride_bytes, num_pages,
                                  _ptr(page_ids), n, _ptr(page_mode), _ptr(low_in),
                                  _stream(stream)), "ekv_promote_pages")


def ekv_paged_decode_elastic(ctx, q, k_pages, v_pages, v_page_stride_bytes, num_pages, num_v_slots, v_scales,
                             scale_mode, page_mode, uniform_mode, block_table, v_block_table,
                             block_table_stride, boundaries, has_base, seq_lens, batch, sm_scale, out,
                             lse=None, stream=None):
    """Decode over the pair-structured value layout (values located through v_block_table)."""
    _check(_lib.ekv_paged_decode_elastic(ctx, _ptr(q), _ptr(k_pages), _ptr(v_pages), v_page_stride_bytes,
                                         num_pages, num_v_slots, _ptr(v_scales), scale_mode, _ptr(page_mode),
                                         uniform_mode, _ptr(block_table), _ptr(v_block_table),
                                         block_table_stride, _ptr(boundaries), int(has_base), _ptr(seq_lens),
                                         batch, float(sm_scale), _ptr(out), _ptr(lse), _stream(stream)),
           "ekv_paged_decode_elastic")


def ekv_transition_pages(ctx, op, v_pages, v_page_stride_bytes, num_slots, num_pages, page_ids, src_loc,
                         dst_loc, n, page_mode, scale_out=None, low=None, stream=None):
    """Located mode transition: op 0 -> E4M3, 1 -> BASE, 2 promote (see include/ekv.h)."""
    _check(_lib.ekv_transition_pages(ctx, op, _ptr(v_pages), v_page_stride_bytes, num_slots, num_pages,
                                     _ptr(page_ids), _ptr(src_loc), _ptr(dst_loc), n, _ptr(page_mode),
                                     _ptr(scale_out), _ptr(low), _stream(stream)), "ekv_transition_pages")


def ekv_prefill_attention(ctx, q, ws_k, ws_v, ws_pages, cu_seqlens, page_off, n, max_len, sm_scale, out,
                          lse=None, stream=None):
    """FP16 causal prefill of whole prompts over the gathered workspace."""
    _check(_lib.ekv_prefill_attention(ctx, _ptr(q), _ptr(ws_k), _ptr(ws_v), ws_pages, _ptr(cu_seqlens),
                                      _ptr(page_off), n, max_len, float(sm_scale), _ptr(out), _ptr(lse),
                                      _stream(stream)), "ekv_prefill_attention")


def ekv_append_kv(ctx, k_new, v_new, k_pages, v_pages, v_page_stride_bytes, num_pages, v_scales,
                  scale_mode, page_mode, uniform_mode, block_table, block_table_stride, positions, batch,
                  stream=None):
    """Write one new token per sequence (positions[b] < 0: none) into the paged cache."""
    _check(_lib.ekv_append_kv(ctx, _ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages),
                              v_page_stride_bytes, num_pages, _ptr(v_scales), scale_mode, _ptr(page_mode),
                              uniform_mode, _ptr(block_table), block_table_stride, _ptr(positions), batch,
                              _stream(stream)), "ekv_append_kv")


def ekv_get_error(ctx):
    """(code, detail) of the sticky device error word, which is then cleared."""
    code, detail = _i(0), _i(0)
    _check(_lib.ekv_get_error(ctx, ctypes.byref(code), ctypes.byref(detail)), "ekv_get_error")
    return code.value, detail.value


def ekv_profile_enable(ctx, enable=True):
    _check(_lib.ekv_profile_enable(ctx, 1 if enable else 0), "ekv_profile_enable")


def ekv_profile_read(ctx):
    ms, n = ctypes.c_double(0), _ll(0)
    _check(_lib.ekv_profile_read(ctx, ctypes.byref(ms), ctypes.byref(n)), "ekv_profile_read")
    return ms.value, n.value


def ekv_set_decode_variant(ctx, variant):
    _check(_lib.ekv_set_decode_variant(ctx, variant), "ekv_set_decode_variant")


def ekv_profile_launch_floor(ctx, reps=64, stream=None):
    """Average ms between the CUDA events of one empty launch shaped like the split kernel."""
    ms = ctypes.c_double(0.0)
    _check(_lib.ekv_profile_launch_floor(ctx, int(reps), _stream(stream), ctypes.byref(ms)),
           "ekv_profile_launch_floor")
    return ms.value


def ekv_set_pdl(ctx, enable):
    _check(_lib.ekv_set_pdl(ctx, int(enable)), "ekv_set_pdl")


def ekv_query(ctx):
    a, b = _i(0), _i(0)
    _check(_lib.ekv_query(ctx, ctypes.byref(a), ctypes.byref(b)), "ekv_query")
    return a.value, b.value


def raw_status(fn_name, *args):
    """Call a C entry point directly and return its status (used by the error tests)."""
    return getattr(_lib, fn_name)(*args)


# ----------------------------------------------------------------- convenience layer
class Context:
    """Owns one ekv context; methods take torch tensors and the case's metadata."""

    def __init__(self, num_q_heads, num_kv_heads, head_dim, max_batch, variant=0, pdl=False):
        self.handle = ekv_create(num_q_heads, num_kv_heads, head_dim, max_batch)
        self.num_q_heads, self.num_kv_heads, self.head_dim = num_q_heads, num_kv_heads, head_dim
        if variant:
            ekv_set_decode_variant(self.handle, variant)
        if pdl:
            ekv_set_pdl(self.handle, 1)

    def close(self):
        if self.handle:
            ekv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def decode(self, case, out, lse=None, sm_scale=0.0, stream=None):
        """Decode one ``workloads.DecodeCase`` whose arrays are device tensors."""
        ekv_paged_decode(self.handle, case.q, case.k_pages, case.v_pages, case.v_page_stride,
                         case.num_pages, case.v_scales, case.scale_mode, case.page_mode,
                         case.uniform_mode, case.block_table, int(case.block_table.shape[1]),
                         case.seq_lens, case.batch, sm_scale, out, lse, stream)

    def error(self):
        return ekv_get_error(self.handle)
