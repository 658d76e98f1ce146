"""Shared test helpers: oracle calls on synthetic workloads and parity checks."""

from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances of the attention outputs against the float64 oracle: bf16 output max-abs
# error 1e-2, natural-log LSE max-abs error 1e-3.  The 1e-2 bounds the arithmetic; the
# final conversion to bf16 (8 significant bits) adds at most half a bf16 ulp of the
# value on top, which no bf16 output can avoid (for |out| >= 4 half an ulp alone is
# 2^-6 > 1e-2).  Bound per element: 1e-2 + ulp_bf16(ref) / 2.
O_ATOL = 1e-2
LSE_ATOL = 1e-3


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (normal range)."""
    _, e = np.frexp(np.abs(x))            # |x| = m * 2**e, m in [0.5, 1)
    return np.ldexp(1.0, e - 8)


def out_tolerance(ref: np.ndarray) -> np.ndarray:
    return O_ATOL + 0.5 * bf16_ulp(ref)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def kv_np(wl):
    if wl.spec.kv_dtype == "int8":
        return wl.k_cache.numpy(), wl.v_cache.numpy(), wl.k_scale.numpy(), wl.v_scale.numpy()
    return bits(wl.k_cache), bits(wl.v_cache), None, None


def oracle_metadata(wl, max_seq_pages=None):
    m = wl.full_to_swa_mapping
    return oracle.build_metadata(wl.req_pool_indices.numpy(), wl.seq_lens.numpy(),
                                 wl.req_to_token.numpy(), wl.spec.seqlen_offset,
                                 max_seq_pages or wl.max_seq_pages, wl.spec.page_size,
                                 None if m is None else m.numpy())


def oracle_attention(wl, meta, rows=None):
    """Oracle output/LSE for the requests in ``rows`` (all by default)."""
    rows = np.arange(wl.spec.bs) if rows is None else np.asarray(rows)
    k, v, ks, vs = kv_np(wl)
    q = bits(wl.q)[rows]
    return oracle.paged_attention(q, k, v, meta["page_table"][rows], meta["cache_seqlens"][rows],
                                  wl.sm_scale, ks, vs)


def oracle_partials(wl, meta, num_splits, rows=None):
    rows = np.arange(wl.spec.bs) if rows is None else np.asarray(rows)
    k, v, ks, vs = kv_np(wl)
    q = bits(wl.q)[rows]
    return oracle.splitk_partials(q, k, v, meta["page_table"][rows], meta["cache_seqlens"][rows],
                                  wl.sm_scale, wl.max_seq_pages, num_splits, ks, vs)


def assert_attention_close(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.float().cpu().numpy().astype(np.float64)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: empty-row pattern differs"
    if empty.any():
        assert np.all(o[empty] == 0.0), f"{what}: empty rows must be 0"
    full = ~empty
    o_err = np.abs(o[full] - out_ref[full]).max() if full.any() else 0.0
    l_err = np.abs(lse[full] - lse_ref[full]).max() if full.any() else 0.0
    excess = (np.abs(o[full] - out_ref[full]) - out_tolerance(out_ref[full])).max() if full.any() else 0.0
    assert excess <= 0, f"{what}: out max abs err {o_err} beyond tolerance by {excess}"
    assert l_err <= LSE_ATOL, f"{what}: lse max abs err {l_err}"
    return o_err, l_err
