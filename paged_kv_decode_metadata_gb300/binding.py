"""Python binding of the C ABI in include/pa.h (argument marshalling only).

Each function here has the name of the C entry point it calls, takes torch tensors,
checks that they are CUDA tensors of the expected dtype and layout, and passes their
device pointers through ctypes.  All arithmetic runs in the library's kernels; there
is no fallback: if ``_build/libpa.so`` is missing the first call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_SCRATCH_LIMIT = 0, 1, 2, 3, 4
PA_STATIC_SCRATCH_BYTES = 16 * 1024 * 1024
PA_KV_BF16, PA_KV_INT8 = 0, 1
PA_Q_MODE_NONE, PA_Q_MODE_CUMSUM, PA_Q_MODE_STRIDED = 0, 1, 2
PA_PRODUCER_AUTO, PA_PRODUCER_FMA, PA_PRODUCER_MMA = 0, 1, 2
DEVERR_PAGE_OUT_OF_RANGE = 0x1
DEVERR_POOL_ROW_OUT_OF_RANGE = 0x2
DEVERR_SLOT_OUT_OF_RANGE = 0x4
DEVERR_WAIT_TIMEOUT = 0x8
DEVERR_SEQLEN_OUT_OF_RANGE = 0x10

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class PAError(RuntimeError):
    def __init__(self, func: str, status: int, lib=None):
        self.status = status
        detail = ""
        if status == PA_ERR_CUDA:
            detail = ": " + (lib or load()).pa_last_error_string().decode()
        super().__init__(f"{func} failed: {status_string(status)} ({status}){detail}")


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libpa.so (built by ``build.build()``, or the file named by the PA_LIBRARY
    environment variable); raise if it is not there."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("PA_LIBRARY") or _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing; build it with "
                    "`python -m paged_kv_decode_metadata_gb300.build`")
            _lib = _declare(ctypes.CDLL(path))
    return _lib


_ts_lib: Optional[ctypes.CDLL] = None


def load_instrumented() -> ctypes.CDLL:
    """Load the timestamp-instrumented build ``_build/libpa_ts.so`` (same entry points
    plus pa_set_timestamp_buffer, include/pa_timestamps.h); raise if it is missing."""
    global _ts_lib
    with _lock:
        if _ts_lib is None:
            path = _build.TS_LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"instrumented library {path} is missing; build it with "
                                   "`python -m paged_kv_decode_metadata_gb300.build --ts`")
            lib = _declare(ctypes.CDLL(path))
            lib.pa_set_timestamp_buffer.argtypes = [ctypes.c_void_p]
            lib.pa_set_timestamp_buffer.restype = ctypes.c_int
            lib.pa_set_test_hold_loads.argtypes = [ctypes.c_int32]
            lib.pa_set_test_hold_loads.restype = ctypes.c_int
            lib.pa_set_test_no_persist.argtypes = [ctypes.c_int32]
            lib.pa_set_test_no_persist.restype = ctypes.c_int
            _ts_lib = lib
    return _ts_lib


def _declare(lib):
    vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
    lib.pa_build_metadata.argtypes = [vp, vp, vp, i64, i64, vp, i64, vp, vp, vp, i64, vp, i64,
                                      i32, i32, i32, i32, vp, i32]
    lib.pa_build_metadata_full.argtypes = [vp, vp, i32, vp, i64, i64, vp, i64, vp, i64, vp, vp,
                                           vp, vp, vp, i64, vp, i64, vp, i64, i32, i32, i32,
                                           i32, i32, i32, vp, i32]
    lib.pa_decode_splitk.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, vp, i32, i32, i32, i32,
                                     i32, i64, i32, i32, f32, vp, vp, vp, vp, i32]
    lib.pa_decode_splitk_multi.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, vp, vp, i32, i32,
                                           i32, i32, i32, i32, i64, i32, i32, f32, vp, vp, vp,
                                           vp, i32]
    lib.pa_decode_splitk_window.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, vp, vp, i32, i32,
                                            i32, i32, i32, i32, i64, i32, i32, i32, f32, vp, vp,
                                            vp, vp, i32]
    lib.pa_window_pages.argtypes = [i32, i32, i32, i32]
    lib.pa_window_pages.restype = i32
    lib.pa_reduce.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, i32]
    lib.pa_decode_step.argtypes = [vp, vp, vp, i64, i64, vp, i64, i32, i32, vp, vp, vp, i64,
                                   vp, i64, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                   i64, i32, f32, vp, sz, vp, vp, vp, i32]
    lib.pa_decode_step_host.argtypes = [vp, vp, vp, vp, vp] + lib.pa_decode_step.argtypes
    step = lib.pa_decode_step.argtypes
    lib.pa_decode_step_host_packed.argtypes = [vp, vp, vp, vp] + step[2:15] + step[16:31] + \
        step[33:35]
    lib.pa_packed_input_bytes.argtypes = [i32, i32, i32]
    lib.pa_packed_input_bytes.restype = sz
    lib.pa_packed_output_bytes.argtypes = [i32, i32, i32]
    lib.pa_packed_output_bytes.restype = sz
    lib.pa_decode_step_multi.argtypes = [vp, vp, vp, i64, i64, vp, i64, i32, i32, vp, vp, vp,
                                         i64, vp, i64, vp, i32, i32, vp, vp, i32, i32, vp, vp,
                                         vp, vp, i32, i32, i32, i32, i32, i32, i64, i32, f32, vp,
                                         sz, vp, vp, vp, i32]
    lib.pa_decode_step_window.argtypes = [vp, vp, vp, i64, i64, vp, i64, i32, i32, vp, vp, vp,
                                          i64, vp, i64, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                          i32, i32, i64, i32, i32, f32, vp, sz, vp, vp, vp, i32]
    lib.pa_decode_step_static_scratch.argtypes = [vp, vp, vp, i64, i64, vp, i64, i32, i32, vp,
                                                  vp, vp, i64, vp, i64, vp, vp, vp, vp, vp, i32,
                                                  i32, i32, i32, i32, i32, i64, i32, f32, vp, vp,
                                                  vp, i32]
    lib.pa_decode_step_static_scratch.restype = ctypes.c_int
    lib.pa_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.pa_workspace_bytes.restype = sz
    lib.pa_choose_splits.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.pa_choose_splits.restype = i32
    lib.pa_select_producer.argtypes = [i32]
    lib.pa_select_producer.restype = i32
    lib.pa_last_error_string.argtypes = []
    lib.pa_last_error_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [i32]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_read_error_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
    for name in ("pa_build_metadata", "pa_build_metadata_full", "pa_decode_splitk",
                 "pa_decode_splitk_multi", "pa_decode_splitk_window", "pa_reduce",
                 "pa_decode_step", "pa_decode_step_host", "pa_decode_step_host_packed",
                 "pa_decode_step_multi",
                 "pa_decode_step_window",
                 "pa_read_error_flags"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def _check(func: str, status: int, lib=None):
    if status != PA_OK:
        raise PAError(func, status, lib)


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _io_ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    """Pointer of a step input or output that the kernels may also reach in pinned host
    memory (q, req_pool_indices, seq_lens, out, lse): a CUDA tensor, or a pinned CPU
    tensor, which the kernels then read or write over the host link (no copy)."""
    if t is not None and not t.is_cuda:
        if not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
        if dtype is not None and t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return t.data_ptr()
    return _ptr(t, dtype, name)


def _row_stride(t: torch.Tensor, name: str) -> int:
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be 2-D with unit column stride")
    return t.stride(0)


def _ptr2d(t: torch.Tensor, dtype, name: str) -> int:
    """Pointer of a row-strided 2-D CUDA tensor (rows may be padded)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    _row_stride(t, name)
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def pa_build_metadata(req_pool_indices, seq_lens, req_to_token, cache_seqlens, cu_seqlens_k,
                      page_table, *, seqlen_offset: int, max_seq_pages: int, page_size: int,
                      full_to_swa_mapping=None, swa_page_table=None, stream=None,
                      use_pdl: bool = True):
    """Fused metadata update; see include/pa.h.  Outputs are written in place."""
    return pa_build_metadata_full(req_pool_indices, seq_lens, req_to_token, cache_seqlens,
                                  cu_seqlens_k, page_table, seqlen_offset=seqlen_offset,
                                  max_seq_pages=max_seq_pages, page_size=page_size,
                                  full_to_swa_mapping=full_to_swa_mapping,
                                  swa_page_table=swa_page_table, stream=stream, use_pdl=use_pdl)


def pa_build_metadata_full(req_pool_indices, seq_lens, req_to_token, cache_seqlens,
                           cu_seqlens_k, page_table, *, seqlen_offset: int, max_seq_pages: int,
                           page_size: int, full_to_swa_mapping=None, swa_page_table=None,
                           cu_seqlens_q=None, qlens=None, q_mode: int = PA_Q_MODE_NONE,
                           q_stride: int = 0, out_cache_loc=None, swa_out_cache_loc=None,
                           stream=None, use_pdl: bool = True):
    lib = load()
    bs = req_pool_indices.shape[0]
    pt_stride = _row_stride(page_table, "page_table")
    swa_stride = _row_stride(swa_page_table, "swa_page_table") if swa_page_table is not None else 0
    idx_dtype = req_pool_indices.dtype
    if idx_dtype not in (torch.int64, torch.int32):
        raise ValueError("req_pool_indices must be int64 or int32")
    st = lib.pa_build_metadata_full(
        _io_ptr(req_pool_indices, idx_dtype, "req_pool_indices"),
        _io_ptr(seq_lens, idx_dtype, "seq_lens"), 64 if idx_dtype == torch.int64 else 32,
        _ptr2d(req_to_token, torch.int32, "req_to_token"),
        req_to_token.shape[0], req_to_token.stride(0),
        _ptr(full_to_swa_mapping, torch.int64, "full_to_swa_mapping"),
        full_to_swa_mapping.numel() if full_to_swa_mapping is not None else 0,
        _ptr(out_cache_loc, torch.int64, "out_cache_loc"),
        out_cache_loc.numel() if out_cache_loc is not None else 0,
        _ptr(qlens, idx_dtype, "qlens"),
        _ptr(cache_seqlens, torch.int32, "cache_seqlens"),
        _ptr(cu_seqlens_k, torch.int32, "cu_seqlens_k"),
        _ptr(cu_seqlens_q, torch.int32, "cu_seqlens_q"),
        _ptr2d(page_table, torch.int32, "page_table"), pt_stride,
        _ptr2d(swa_page_table, torch.int32, "swa_page_table") if swa_page_table is not None else None,
        swa_stride,
        _ptr(swa_out_cache_loc, torch.int64, "swa_out_cache_loc"),
        swa_out_cache_loc.numel() if swa_out_cache_loc is not None else 0,
        bs, int(seqlen_offset), int(max_seq_pages), int(page_size), int(q_mode), int(q_stride),
        _stream(stream), int(bool(use_pdl)))
    _check("pa_build_metadata_full", st)


def _kv_args(k_cache, v_cache, k_scale, v_scale):
    if k_cache.dtype == torch.bfloat16:
        return PA_KV_BF16, None, None
    if k_cache.dtype == torch.int8:
        if k_scale is None or v_scale is None:
            raise ValueError("int8 KV needs k_scale and v_scale")
        return PA_KV_INT8, _ptr(k_scale, torch.float32, "k_scale"), _ptr(v_scale, torch.float32, "v_scale")
    raise ValueError(f"unsupported KV dtype {k_cache.dtype}")


def pa_decode_splitk(q, k_cache, v_cache, page_table, cache_seqlens, scratch_m, scratch_l,
                     scratch_acc, *, max_seq_pages: int, num_splits: int, sm_scale: float,
                     k_scale=None, v_scale=None, stream=None, use_pdl: bool = True):
    """Split-K producer: writes per-split (m, l, acc) partials; see include/pa.h."""
    lib = load()
    kv_dtype, ks, vs = _kv_args(k_cache, v_cache, k_scale, v_scale)
    bs, hq, d = q.shape
    num_pages, hkv, page_size, _ = k_cache.shape
    st = lib.pa_decode_splitk(
        _io_ptr(q, torch.bfloat16, "q"), _ptr(k_cache, None, "k_cache"), _ptr(v_cache, None, "v_cache"),
        ks, vs, kv_dtype, _ptr2d(page_table, torch.int32, "page_table"),
        _row_stride(page_table, "page_table"),
        _ptr(cache_seqlens, torch.int32, "cache_seqlens"), bs, hq, hkv, d, page_size, num_pages,
        int(max_seq_pages), int(num_splits), float(sm_scale),
        _ptr(scratch_m, torch.float32, "scratch_m"), _ptr(scratch_l, torch.float32, "scratch_l"),
        _ptr(scratch_acc, torch.float32, "scratch_acc"), _stream(stream), int(bool(use_pdl)))
    _check("pa_decode_splitk", st)


def pa_decode_splitk_multi(q, k_cache, v_cache, page_table, cache_seqlens, cu_seqlens_q,
                           scratch_m, scratch_l, scratch_acc, *, max_q_len: int,
                           max_seq_pages: int, num_splits: int, sm_scale: float, k_scale=None,
                           v_scale=None, stream=None, use_pdl: bool = True):
    """Split-K producer for several query tokens per request (rows from cu_seqlens_q,
    causal within the request's newest tokens); see include/pa.h."""
    lib = load()
    kv_dtype, ks, vs = _kv_args(k_cache, v_cache, k_scale, v_scale)
    total_q, hq, d = q.shape
    bs = cache_seqlens.shape[0]
    num_pages, hkv, page_size, _ = k_cache.shape
    st = lib.pa_decode_splitk_multi(
        _io_ptr(q, torch.bfloat16, "q"), _ptr(k_cache, None, "k_cache"), _ptr(v_cache, None, "v_cache"),
        ks, vs, kv_dtype, _ptr2d(page_table, torch.int32, "page_table"),
        _row_stride(page_table, "page_table"), _ptr(cache_seqlens, torch.int32, "cache_seqlens"),
        _ptr(cu_seqlens_q, torch.int32, "cu_seqlens_q"), bs, int(max_q_len), hq, hkv, d,
        page_size, num_pages, int(max_seq_pages), int(num_splits), float(sm_scale),
        _ptr(scratch_m, torch.float32, "scratch_m"), _ptr(scratch_l, torch.float32, "scratch_l"),
        _ptr(scratch_acc, torch.float32, "scratch_acc"), _stream(stream), int(bool(use_pdl)))
    _check("pa_decode_splitk_multi", st)


def pa_decode_splitk_window(q, k_cache, v_cache, page_table, cache_seqlens, scratch_m,
                            scratch_l, scratch_acc, *, sliding_window: int, max_seq_pages: int,
                            num_splits: int, sm_scale: float, cu_seqlens_q=None,
                            max_q_len: int = 1, k_scale=None, v_scale=None, stream=None,
                            use_pdl: bool = True):
    """Split-K producer of a sliding-window layer: reads the sliding-window pool
    (``k_cache``/``v_cache``) through the sliding-window page table; one query per
    request, or the rows ``cu_seqlens_q`` assigns.  See include/pa.h."""
    lib = load()
    kv_dtype, ks, vs = _kv_args(k_cache, v_cache, k_scale, v_scale)
    rows, hq, d = q.shape
    bs = cache_seqlens.shape[0]
    num_pages, hkv, page_size, _ = k_cache.shape
    st = lib.pa_decode_splitk_window(
        _io_ptr(q, torch.bfloat16, "q"), _ptr(k_cache, None, "k_cache"), _ptr(v_cache, None, "v_cache"),
        ks, vs, kv_dtype, _ptr2d(page_table, torch.int32, "page_table"),
        _row_stride(page_table, "page_table"), _ptr(cache_seqlens, torch.int32, "cache_seqlens"),
        _ptr(cu_seqlens_q, torch.int32, "cu_seqlens_q"), bs, int(max_q_len), hq, hkv, d,
        page_size, num_pages, int(max_seq_pages), int(sliding_window), int(num_splits),
        float(sm_scale), _ptr(scratch_m, torch.float32, "scratch_m"),
        _ptr(scratch_l, torch.float32, "scratch_l"), _ptr(scratch_acc, torch.float32, "scratch_acc"),
        _stream(stream), int(bool(use_pdl)))
    _check("pa_decode_splitk_window", st)


def pa_window_pages(sliding_window: int, max_q_len: int, page_size: int,
                    max_seq_pages: int) -> int:
    """Pages a sliding-window split partition spans; see include/pa.h."""
    return int(load().pa_window_pages(int(sliding_window), int(max_q_len), int(page_size),
                                      int(max_seq_pages)))


def pa_reduce(scratch_m, scratch_l, scratch_acc, out, lse=None, *, stream=None,
              use_pdl: bool = True):
    """Log-sum-exp reducer: writes out (bf16) and lse (fp32); see include/pa.h."""
    lib = load()
    bs, hq, s = scratch_m.shape
    d = scratch_acc.shape[-1]
    st = lib.pa_reduce(_ptr(scratch_m, torch.float32, "scratch_m"),
                       _ptr(scratch_l, torch.float32, "scratch_l"),
                       _ptr(scratch_acc, torch.float32, "scratch_acc"), bs, hq, d, s,
                       _io_ptr(out, torch.bfloat16, "out"), _io_ptr(lse, torch.float32, "lse"),
                       _stream(stream), int(bool(use_pdl)))
    _check("pa_reduce", st)


def pa_decode_step(*, lib=None, **kw):
    """Metadata + split-K producer + reducer in one call; see include/pa.h.  ``lib``
    selects another build of the library (e.g. ``load_instrumented()``).  Keyword
    arguments: those of ``_decode_step_args``."""
    lib = lib or load()
    _check("pa_decode_step", lib.pa_decode_step(*_decode_step_args(**kw)), lib)


def _decode_step_args(*, req_pool_indices, seq_lens, req_to_token, seqlen_offset: int,
                      max_seq_pages: int, cache_seqlens, cu_seqlens_k, page_table, q, k_cache,
                      v_cache, num_splits: int, sm_scale: float, workspace, out, lse=None,
                      k_scale=None, v_scale=None, full_to_swa_mapping=None, swa_page_table=None,
                      stream=None, use_pdl: bool = True):
    kv_dtype, ks, vs = _kv_args(k_cache, v_cache, k_scale, v_scale)
    bs, hq, d = q.shape
    num_pages, hkv, page_size, _ = k_cache.shape
    return (
        _io_ptr(req_pool_indices, torch.int64, "req_pool_indices"),
        _io_ptr(seq_lens, torch.int64, "seq_lens"), _ptr2d(req_to_token, torch.int32, "req_to_token"),
        req_to_token.shape[0], req_to_token.stride(0),
        _ptr(full_to_swa_mapping, torch.int64, "full_to_swa_mapping"),
        full_to_swa_mapping.numel() if full_to_swa_mapping is not None else 0,
        int(seqlen_offset), int(max_seq_pages), _ptr(cache_seqlens, torch.int32, "cache_seqlens"),
        _ptr(cu_seqlens_k, torch.int32, "cu_seqlens_k"), _ptr2d(page_table, torch.int32, "page_table"),
        _row_stride(page_table, "page_table"),
        _ptr2d(swa_page_table, torch.int32, "swa_page_table") if swa_page_table is not None else None,
        _row_stride(swa_page_table, "swa_page_table") if swa_page_table is not None else 0,
        _io_ptr(q, torch.bfloat16, "q"), _ptr(k_cache, None, "k_cache"),
        _ptr(v_cache, None, "v_cache"), ks, vs, kv_dtype, bs, hq, hkv, d, page_size, num_pages,
        int(num_splits), float(sm_scale), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _io_ptr(out, torch.bfloat16, "out"),
        _io_ptr(lse, torch.float32, "lse"), _stream(stream), int(bool(use_pdl)))


def _host_ptr(t, dtype, name):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _decode_step_host_args(*, h_q, h_req_pool_indices, h_seq_lens, h_out, h_lse=None, **kw):
    return (_host_ptr(h_q, torch.bfloat16, "h_q"),
            _host_ptr(h_req_pool_indices, torch.int64, "h_req_pool_indices"),
            _host_ptr(h_seq_lens, torch.int64, "h_seq_lens"),
            _host_ptr(h_out, torch.bfloat16, "h_out"),
            _host_ptr(h_lse, torch.float32, "h_lse")) + _decode_step_args(**kw)


def pa_decode_step_host(*, lib=None, **kw):
    """pa_decode_step with host inputs (h_q, h_req_pool_indices, h_seq_lens) and host
    outputs (h_out, h_lse), copies enqueued on the same stream; see include/pa.h.  The
    other keyword arguments are those of ``pa_decode_step``."""
    lib = lib or load()
    _check("pa_decode_step_host", lib.pa_decode_step_host(*_decode_step_host_args(**kw)), lib)


def _decode_step_host_packed_args(*, h_inputs, inputs, h_outputs, outputs, **kw):
    """``kw``: the arguments of ``pa_decode_step``, whose q, req_pool_indices and
    seq_lens must be the views of ``inputs``, and out and lse those of ``outputs``, that
    the packed layout defines (their pointers are not passed; only shapes are read)."""
    a = _decode_step_args(**kw)
    bs, hq, d = a[21], a[22], a[24]
    lib = load()
    for t, name, n in ((h_inputs, "h_inputs", lib.pa_packed_input_bytes(bs, hq, d)),
                       (h_outputs, "h_outputs", lib.pa_packed_output_bytes(bs, hq, d))):
        if t.is_cuda or not t.is_contiguous() or t.numel() * t.element_size() < n:
            raise ValueError(f"{name} must be a contiguous host buffer of {n} bytes")
    for t, name, n in ((inputs, "inputs", lib.pa_packed_input_bytes(bs, hq, d)),
                       (outputs, "outputs", lib.pa_packed_output_bytes(bs, hq, d))):
        if not t.is_cuda or not t.is_contiguous() or t.numel() * t.element_size() < n:
            raise ValueError(f"{name} must be a contiguous device buffer of {n} bytes")
    if a[15] != inputs.data_ptr() or a[0] != inputs.data_ptr() + d * hq * bs * 2 or \
            a[31] != outputs.data_ptr() or (a[32] is not None and
                                            a[32] != outputs.data_ptr() + d * hq * bs * 2):
        raise ValueError("q / req_pool_indices / seq_lens and out / lse must be the packed views")
    return (h_inputs.data_ptr(), inputs.data_ptr(), h_outputs.data_ptr(),
            outputs.data_ptr()) + a[2:15] + a[16:31] + a[33:35]


def pa_decode_step_multi(*, req_pool_indices, seq_lens, req_to_token, seqlen_offset: int,
                         max_seq_pages: int, cache_seqlens, cu_seqlens_k, page_table,
                         cu_seqlens_q, q, max_q_len: int, k_cache, v_cache, num_splits: int,
                         sm_scale: float, workspace, out, lse=None, qlens=None,
                         q_mode: int = PA_Q_MODE_CUMSUM, q_stride: int = 0, k_scale=None,
                         v_scale=None, full_to_swa_mapping=None, swa_page_table=None,
                         stream=None, use_pdl: bool = True):
    """Metadata (with cu_seqlens_q) + multi-query producer + reducer over the q rows;
    see include/pa.h."""
    lib = load()
    kv_dtype, ks, vs = _kv_args(k_cache, v_cache, k_scale, v_scale)
    total_q, hq, d = q.shape
    bs = cache_seqlens.shape[0]
    num_pages, hkv, page_size, _ = k_cache.shape
    st = lib.pa_decode_step_multi(
        _io_ptr(req_pool_indices, torch.int64, "req_pool_indices"),
        _io_ptr(seq_lens, torch.int64, "seq_lens"), _ptr2d(req_to_token, torch.int32, "req_to_token"),
        req_to_token.shape[0], req_to_token.stride(0),
        _ptr(full_to_swa_mapping, torch.int64, "full_to_swa_mapping"),
        full_to_swa_mapping.numel() if full_to_swa_mapping is not None else 0,
        int(seqlen_offset), int(max_seq_pages), _ptr(cache_seqlens, torch.int32, "cache_seqlens"),
        _ptr(cu_seqlens_k, torch.int32, "cu_seqlens_k"), _ptr2d(page_table, torch.int32, "page_table"),
        _row_stride(page_table, "page_table"),
        _ptr2d(swa_page_table, torch.int32, "swa_page_table") if swa_page_table is not None else None,
        _row_stride(swa_page_table, "swa_page_table") if swa_page_table is not None else 0,
        _ptr(qlens, torch.int64, "qlens"), int(q_mode), int(q_stride),
        _ptr(cu_seqlens_q, torch.int32, "cu_seqlens_q"), _io_ptr(q, torch.bfloat16, "q"), total_q,
        int(max_q_len), _ptr(k_cache, None, "k_cache"), _ptr(v_cache, None, "v_cache"), ks, vs,
        kv_dtype, bs, hq, hkv, d, page_size, num_pages, int(num_splits), float(sm_scale),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _io_ptr(out, torch.bfloat16, "out"), _io_ptr(lse, torch.float32, "lse"), _stream(stream),
        int(bool(use_pdl)))
    _check("pa_decode_step_multi", st)


def pa_decode_step_window(*, lib=None, **kw):
    """Metadata + sliding-window producer + reducer in one call; see include/pa.h.
    Keyword arguments: those of ``_decode_step_window_args``."""
    lib = lib or load()
    _check("pa_decode_step_window", lib.pa_decode_step_window(*_decode_step_window_args(**kw)),
           lib)


def _decode_step_window_args(*, req_pool_indices, seq_lens, req_to_token, seqlen_offset: int,
                             max_seq_pages: int, cache_seqlens, cu_seqlens_k, page_table,
                             full_to_swa_mapping, swa_page_table, q, k_swa, v_swa,
                             sliding_window: int, num_splits: int, sm_scale: float, workspace,
                             out, lse=None, k_swa_scale=None, v_swa_scale=None, stream=None,
                             use_pdl: bool = True):
    kv_dtype, ks, vs = _kv_args(k_swa, v_swa, k_swa_scale, v_swa_scale)
    bs, hq, d = q.shape
    num_pages, hkv, page_size, _ = k_swa.shape
    return (
        _io_ptr(req_pool_indices, torch.int64, "req_pool_indices"),
        _io_ptr(seq_lens, torch.int64, "seq_lens"), _ptr2d(req_to_token, torch.int32, "req_to_token"),
        req_to_token.shape[0], req_to_token.stride(0),
        _ptr(full_to_swa_mapping, torch.int64, "full_to_swa_mapping"),
        full_to_swa_mapping.numel(), int(seqlen_offset), int(max_seq_pages),
        _ptr(cache_seqlens, torch.int32, "cache_seqlens"),
        _ptr(cu_seqlens_k, torch.int32, "cu_seqlens_k"), _ptr2d(page_table, torch.int32, "page_table"),
        _row_stride(page_table, "page_table"), _ptr2d(swa_page_table, torch.int32, "swa_page_table"),
        _row_stride(swa_page_table, "swa_page_table"), _io_ptr(q, torch.bfloat16, "q"),
        _ptr(k_swa, None, "k_swa"), _ptr(v_swa, None, "v_swa"), ks, vs, kv_dtype, bs, hq, hkv, d,
        page_size, num_pages, int(sliding_window), int(num_splits), float(sm_scale),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _io_ptr(out, torch.bfloat16, "out"), _io_ptr(lse, torch.float32, "lse"), _stream(stream),
        int(bool(use_pdl)))


class PreparedCall:
    """One entry point with its arguments marshalled once: calling it repeats the call
    on the same tensors, stream and options, without re-validating or re-converting the
    Python arguments.  The call holds references to the tensors it was prepared with
    (``keep``), so their memory stays allocated; they must stay in place (in-place
    updates are fine)."""

    def __init__(self, name: str, args: tuple, lib=None, keep: tuple = ()):
        self.lib = lib or load()
        self.name = name
        self.fn = getattr(self.lib, name)
        self.args = tuple(t(a) if a is not None else None
                          for t, a in zip(self.fn.argtypes, args))
        self._keep = tuple(k for k in keep if isinstance(k, torch.Tensor))

    def __call__(self):
        st = self.fn(*self.args)
        if st != PA_OK:
            raise PAError(self.name, st, self.lib)


def prepare_decode_step(*, lib=None, **kw) -> PreparedCall:
    """``pa_decode_step`` with the given keyword arguments, marshalled once."""
    return PreparedCall("pa_decode_step", _decode_step_args(**kw), lib, keep=tuple(kw.values()))


def prepare_decode_step_host(*, lib=None, **kw) -> PreparedCall:
    """``pa_decode_step_host`` with the given keyword arguments, marshalled once."""
    return PreparedCall("pa_decode_step_host", _decode_step_host_args(**kw), lib, keep=tuple(kw.values()))


def prepare_decode_step_host_packed(*, lib=None, **kw) -> PreparedCall:
    """``pa_decode_step_host_packed`` with the given keyword arguments, marshalled once."""
    return PreparedCall("pa_decode_step_host_packed", _decode_step_host_packed_args(**kw), lib, keep=tuple(kw.values()))


def prepare_decode_step_window(*, lib=None, **kw) -> PreparedCall:
    """``pa_decode_step_window`` with the given keyword arguments, marshalled once."""
    return PreparedCall("pa_decode_step_window", _decode_step_window_args(**kw), lib, keep=tuple(kw.values()))


def pa_decode_step_static_scratch(*, req_pool_indices, seq_lens, req_to_token,
                                  seqlen_offset: int, max_seq_pages: int, cache_seqlens,
                                  cu_seqlens_k, page_table, q, k_cache, v_cache,
                                  num_splits: int, sm_scale: float, out, lse=None, k_scale=None,
                                  v_scale=None, full_to_swa_mapping=None, swa_page_table=None,
                                  stream=None, use_pdl: bool = True):
    """pa_decode_step without a workspace argument, for callers that cannot allocate:
    the split-K scratch is the library's built-in array (see include/pa.h).  Calls
    share that array, so calls must not overlap on the GPU."""
    lib = load()
    kv_dtype, ks, vs = _kv_args(k_cache, v_cache, k_scale, v_scale)
    bs, hq, d = q.shape
    num_pages, hkv, page_size, _ = k_cache.shape
    st = lib.pa_decode_step_static_scratch(
        _io_ptr(req_pool_indices, torch.int64, "req_pool_indices"),
        _io_ptr(seq_lens, torch.int64, "seq_lens"), _ptr2d(req_to_token, torch.int32, "req_to_token"),
        req_to_token.shape[0], req_to_token.stride(0),
        _ptr(full_to_swa_mapping, torch.int64, "full_to_swa_mapping"),
        full_to_swa_mapping.numel() if full_to_swa_mapping is not None else 0,
        int(seqlen_offset), int(max_seq_pages), _ptr(cache_seqlens, torch.int32, "cache_seqlens"),
        _ptr(cu_seqlens_k, torch.int32, "cu_seqlens_k"), _ptr2d(page_table, torch.int32, "page_table"),
        _row_stride(page_table, "page_table"),
        _ptr2d(swa_page_table, torch.int32, "swa_page_table") if swa_page_table is not None else None,
        _row_stride(swa_page_table, "swa_page_table") if swa_page_table is not None else 0,
        _io_ptr(q, torch.bfloat16, "q"), _ptr(k_cache, None, "k_cache"),
        _ptr(v_cache, None, "v_cache"), ks, vs, kv_dtype, bs, hq, hkv, d, page_size, num_pages,
        int(num_splits), float(sm_scale), _io_ptr(out, torch.bfloat16, "out"),
        _io_ptr(lse, torch.float32, "lse"), _stream(stream), int(bool(use_pdl)))
    _check("pa_decode_step_static_scratch", st)


def pa_workspace_bytes(bs: int, num_q_heads: int, head_dim: int, num_splits: int) -> int:
    return int(load().pa_workspace_bytes(bs, num_q_heads, head_dim, num_splits))


def pa_choose_splits(bs: int, num_kv_heads: int, max_seq_pages: int, page_size: int,
                     kv_dtype: int = 0, sm_count: int = 0) -> int:
    """Split count heuristic; kv_dtype PA_KV_BF16 (0) or PA_KV_INT8 (1)."""
    return int(load().pa_choose_splits(bs, num_kv_heads, max_seq_pages, page_size, kv_dtype,
                                       sm_count))


def pa_select_producer(producer: int) -> int:
    """Choose the split-K producer implementation (PA_PRODUCER_AUTO / _FMA / _MMA) for
    later calls; returns the previous choice."""
    return int(load().pa_select_producer(int(producer)))


class producer:
    """Context manager: run a block with one producer implementation selected."""

    def __init__(self, which: int):
        self.which = which

    def __enter__(self):
        self.prev = pa_select_producer(self.which)
        return self

    def __exit__(self, *exc):
        pa_select_producer(self.prev)


def pa_status_string(status: int) -> str:
    return status_string(status)


def pa_read_error_flags(reset: bool = True, lib=None) -> int:
    """Device error word (synchronises the device); see include/pa.h.  ``lib`` reads the
    word of another build of the library (each build has its own)."""
    v = ctypes.c_uint32(0)
    lib = lib or load()
    _check("pa_read_error_flags", lib.pa_read_error_flags(ctypes.byref(v), int(bool(reset))), lib)
    return int(v.value)
