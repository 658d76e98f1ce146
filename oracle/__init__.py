"""CPU oracle for the decode-step paged-KV attention path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline`` /
``--impl reference`` legs may import this package.  It never imports the product
package, and the product never imports it.

The arithmetic lives in ``pa_oracle.cpp`` (plain C++ loops, double precision); this
module compiles it with the host compiler and wraps it for numpy arrays.  Which
passage each function follows is stated in the C++ source.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off keeps a*b+c as two rounded operations on every host (gcc on
# aarch64 would otherwise fuse them), so the oracle gives the same bits on the
# x86 build box and on the Arm GPU host.
_CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off"]


def build(source: str = _SRC, out_path: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile ``source`` into the shared library ``out_path`` with g++."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["g++", *_CXXFLAGS, *extra_flags, source, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def _stale(lib_path: str, src_path: str) -> bool:
    return (not os.path.exists(lib_path)) or os.path.getmtime(lib_path) < os.path.getmtime(src_path)


def _p(arr):
    return ctypes.c_void_p(arr.ctypes.data) if arr is not None else ctypes.c_void_p(0)


def load(lib_path: str | None = None) -> ctypes.CDLL:
    """Return the oracle library, compiling it first if it is missing or stale.

    ``lib_path`` loads another build of the same source (the planted-mistake tests
    compile modified copies and load them through this function).
    """
    global _lib
    if lib_path is not None:
        return _declare(ctypes.CDLL(lib_path))
    with _lock:
        if _lib is None:
            if _stale(_LIB_PATH, _SRC):
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_build_metadata.argtypes = [vp, vp, vp, i64, vp, vp, vp, vp, i64, vp, i64,
                                          i32, i32, i32, i32]
    lib.oracle_cu_seqlens_q.argtypes = [vp, vp, i32, i32, i32]
    lib.oracle_swa_out_cache_loc.argtypes = [vp, i64, vp, vp, i64]
    lib.oracle_paged_attention.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, vp, i32, i32,
                                           i32, i32, i32, f64, vp, vp]
    lib.oracle_paged_attention_multi.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, vp, vp, i32,
                                                 i32, i32, i32, i32, f64, vp, vp]
    lib.oracle_splitk_partials.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, vp, i32, i32,
                                           i32, i32, i32, i32, i32, f64, vp, vp, vp]
    lib.oracle_paged_attention_window.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, vp, vp,
                                                  i32, i32, i32, i32, i32, i32, f64, vp, vp]
    lib.oracle_splitk_partials_window.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, vp, vp,
                                                  i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                                  f64, vp, vp, vp]
    lib.oracle_combine_splits.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp]
    for name in ("oracle_build_metadata", "oracle_cu_seqlens_q", "oracle_swa_out_cache_loc",
                 "oracle_paged_attention", "oracle_paged_attention_multi",
                 "oracle_splitk_partials", "oracle_combine_splits",
                 "oracle_paged_attention_window", "oracle_splitk_partials_window"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def _c(arr, dtype):
    arr = np.ascontiguousarray(arr)
    if arr.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {arr.dtype}")
    return arr


def build_metadata(req_pool_indices, seq_lens, req_to_token, seqlen_offset, max_seq_pages,
                   page_size, full_to_swa_mapping=None, page_table_stride=None,
                   cu_seqlens_k_init=None, lib=None):
    """Fused metadata update; returns a dict of numpy int32 arrays.

    ``cu_seqlens_k_init`` presets the output buffer (the oracle writes every entry,
    index 0 included, so the preset is only there to show that it is overwritten).
    """
    lib = lib or load()
    rpi = _c(req_pool_indices, np.int64)
    sl = _c(seq_lens, np.int64)
    r2t = _c(req_to_token, np.int32)
    bs = rpi.shape[0]
    stride_pt = page_table_stride or max(max_seq_pages, 1)
    cache_seqlens = np.zeros(bs, np.int32)
    cu = np.zeros(bs + 1, np.int32) if cu_seqlens_k_init is None else np.array(cu_seqlens_k_init, np.int32)
    page_table = np.zeros((bs, stride_pt), np.int32)
    swa = None
    mapping = None
    if full_to_swa_mapping is not None:
        mapping = _c(full_to_swa_mapping, np.int64)
        swa = np.zeros((bs, stride_pt), np.int32)
    lib.oracle_build_metadata(_p(rpi), _p(sl), _p(r2t), r2t.shape[1], _p(mapping),
                              _p(cache_seqlens), _p(cu), _p(page_table), stride_pt,
                              _p(swa), stride_pt, bs, int(seqlen_offset), int(max_seq_pages),
                              int(page_size))
    out = {"cache_seqlens": cache_seqlens, "cu_seqlens_k": cu,
           "page_table": page_table[:, :max_seq_pages]}
    if swa is not None:
        out["swa_page_table"] = swa[:, :max_seq_pages]
    return out


def cu_seqlens_q(qlens, bs, q_mode, q_stride=0, init=None, lib=None):
    lib = lib or load()
    ql = _c(qlens, np.int64) if qlens is not None else None
    cu = np.zeros(bs + 1, np.int32) if init is None else np.array(init, np.int32)
    lib.oracle_cu_seqlens_q(_p(ql), _p(cu), bs, q_mode, q_stride)
    return cu


def swa_out_cache_loc(out_cache_loc, full_to_swa_mapping, swa_out_len, lib=None):
    lib = lib or load()
    loc = _c(out_cache_loc, np.int64)
    mapping = _c(full_to_swa_mapping, np.int64)
    out = np.full(swa_out_len, 12345, np.int64)
    lib.oracle_swa_out_cache_loc(_p(loc), loc.shape[0], _p(mapping), _p(out), swa_out_len)
    return out


def _attention_args(q_bits, k_cache, v_cache, k_scale, v_scale):
    q = _c(q_bits, np.uint16)
    if k_cache.dtype == np.int8:
        kv_dtype = 1
        k = _c(k_cache, np.int8)
        v = _c(v_cache, np.int8)
        ks = _c(k_scale, np.float32)
        vs = _c(v_scale, np.float32)
    else:
        kv_dtype = 0
        k = _c(k_cache, np.uint16)
        v = _c(v_cache, np.uint16)
        ks = vs = None
    return q, k, v, ks, vs, kv_dtype


def paged_attention(q_bits, k_cache, v_cache, page_table, cache_seqlens, sm_scale,
                    k_scale=None, v_scale=None, lib=None):
    """softmax(q K^T sm_scale) V and the natural-log LSE, in float64.

    ``q_bits`` [bs, Hq, d] uint16 (bf16 bit patterns); ``k_cache``/``v_cache``
    [num_pages, Hkv, page_size, d] as uint16 bf16 bits or int8 codes (then
    ``k_scale``/``v_scale`` [num_pages, Hkv, page_size] float32).
    """
    lib = lib or load()
    q, k, v, ks, vs, kv_dtype = _attention_args(q_bits, k_cache, v_cache, k_scale, v_scale)
    pt = _c(page_table, np.int32)
    cl = _c(cache_seqlens, np.int32)
    bs, hq, d = q.shape
    _, hkv, page_size, _ = k.shape
    out = np.zeros((bs, hq, d), np.float64)
    lse = np.zeros((bs, hq), np.float64)
    lib.oracle_paged_attention(_p(q), _p(k), _p(v), _p(ks), _p(vs), kv_dtype, _p(pt),
                               pt.shape[1], _p(cl), bs, hq, hkv, d, page_size,
                               float(sm_scale), _p(out), _p(lse))
    return out, lse


def paged_attention_multi(q_bits, k_cache, v_cache, page_table, cache_seqlens, cu_seqlens_q,
                          sm_scale, k_scale=None, v_scale=None, lib=None):
    """Several query tokens per request, causal within the request's newest tokens.

    ``q_bits`` [total_q, Hq, d] uint16; ``cu_seqlens_q`` [bs + 1] int32.  Returns
    (out [total_q, Hq, d], lse [total_q, Hq]) in float64.
    """
    lib = lib or load()
    q, k, v, ks, vs, kv_dtype = _attention_args(q_bits, k_cache, v_cache, k_scale, v_scale)
    pt = _c(page_table, np.int32)
    cl = _c(cache_seqlens, np.int32)
    cq = _c(cu_seqlens_q, np.int32)
    total_q, hq, d = q.shape
    _, hkv, page_size, _ = k.shape
    out = np.zeros((total_q, hq, d), np.float64)
    lse = np.zeros((total_q, hq), np.float64)
    lib.oracle_paged_attention_multi(_p(q), _p(k), _p(v), _p(ks), _p(vs), kv_dtype, _p(pt),
                                     pt.shape[1], _p(cl), _p(cq), cl.shape[0], hq, hkv, d,
                                     page_size, float(sm_scale), _p(out), _p(lse))
    return out, lse


def paged_attention_window(q_bits, k_cache, v_cache, page_table, cache_seqlens, window,
                           sm_scale, cu_seqlens_q=None, k_scale=None, v_scale=None, lib=None):
    """Sliding-window attention through a sliding-window page table (-1 pages skipped).

    ``q_bits`` [rows, Hq, d] uint16: one row per request, or the rows ``cu_seqlens_q``
    [bs + 1] int32 assigns.  ``k_cache``/``v_cache`` is the sliding-window pool.
    Returns (out [rows, Hq, d], lse [rows, Hq]) in float64.
    """
    lib = lib or load()
    q, k, v, ks, vs, kv_dtype = _attention_args(q_bits, k_cache, v_cache, k_scale, v_scale)
    pt = _c(page_table, np.int32)
    cl = _c(cache_seqlens, np.int32)
    cq = _c(cu_seqlens_q, np.int32) if cu_seqlens_q is not None else None
    rows, hq, d = q.shape
    _, hkv, page_size, _ = k.shape
    out = np.zeros((rows, hq, d), np.float64)
    lse = np.zeros((rows, hq), np.float64)
    lib.oracle_paged_attention_window(_p(q), _p(k), _p(v), _p(ks), _p(vs), kv_dtype, _p(pt),
                                      pt.shape[1], _p(cl), _p(cq), cl.shape[0], hq, hkv, d,
                                      page_size, int(window), float(sm_scale), _p(out), _p(lse))
    return out, lse


def splitk_partials_window(q_bits, k_cache, v_cache, page_table, cache_seqlens, window,
                           sm_scale, max_seq_pages, num_splits, cu_seqlens_q=None,
                           max_q_len=1, k_scale=None, v_scale=None, lib=None):
    """Per-split (m, l, acc) of the sliding-window attention over the window's split
    partition; shapes [rows,Hq,S], [rows,Hq,S], [rows,Hq,S,d] in float64."""
    lib = lib or load()
    q, k, v, ks, vs, kv_dtype = _attention_args(q_bits, k_cache, v_cache, k_scale, v_scale)
    pt = _c(page_table, np.int32)
    cl = _c(cache_seqlens, np.int32)
    cq = _c(cu_seqlens_q, np.int32) if cu_seqlens_q is not None else None
    rows, hq, d = q.shape
    _, hkv, page_size, _ = k.shape
    m = np.zeros((rows, hq, num_splits), np.float64)
    l = np.zeros((rows, hq, num_splits), np.float64)
    acc = np.zeros((rows, hq, num_splits, d), np.float64)
    lib.oracle_splitk_partials_window(_p(q), _p(k), _p(v), _p(ks), _p(vs), kv_dtype, _p(pt),
                                      pt.shape[1], _p(cl), _p(cq), cl.shape[0], int(max_q_len),
                                      hq, hkv, d, page_size, int(max_seq_pages), int(window),
                                      int(num_splits), float(sm_scale), _p(m), _p(l), _p(acc))
    return m, l, acc


def splitk_partials(q_bits, k_cache, v_cache, page_table, cache_seqlens, sm_scale,
                    max_seq_pages, num_splits, k_scale=None, v_scale=None, lib=None):
    """Per-split (m, l, acc) in float64; shapes [bs,Hq,S], [bs,Hq,S], [bs,Hq,S,d]."""
    lib = lib or load()
    q, k, v, ks, vs, kv_dtype = _attention_args(q_bits, k_cache, v_cache, k_scale, v_scale)
    pt = _c(page_table, np.int32)
    cl = _c(cache_seqlens, np.int32)
    bs, hq, d = q.shape
    _, hkv, page_size, _ = k.shape
    m = np.zeros((bs, hq, num_splits), np.float64)
    l = np.zeros((bs, hq, num_splits), np.float64)
    acc = np.zeros((bs, hq, num_splits, d), np.float64)
    lib.oracle_splitk_partials(_p(q), _p(k), _p(v), _p(ks), _p(vs), kv_dtype, _p(pt),
                               pt.shape[1], _p(cl), bs, hq, hkv, d, page_size,
                               int(max_seq_pages), int(num_splits), float(sm_scale),
                               _p(m), _p(l), _p(acc))
    return m, l, acc


def combine_splits(m, l, acc, lib=None):
    """Log-sum-exp combination; returns (out [bs,Hq,d], lse [bs,Hq]) in float64."""
    lib = lib or load()
    m = _c(m, np.float64)
    l = _c(l, np.float64)
    acc = _c(acc, np.float64)
    bs, hq, s, d = acc.shape
    out = np.zeros((bs, hq, d), np.float64)
    lse = np.zeros((bs, hq), np.float64)
    lib.oracle_combine_splits(_p(m), _p(l), _p(acc), bs, hq, d, s, _p(out), _p(lse))
    return out, lse
