"""Shared test helpers: oracle calls on synthetic workloads and parity checks.

Attention tolerance against the float64 oracle (``out_tolerance``):

* LSE: max-abs error <= 1e-3, everywhere.
* O (bf16): max-abs error <= 1e-2 for every element whose reference has |ref| < 4, the
  stated bound taken literally.  There half a bf16 ulp of the value is at most 2^-7, so
  a correctly rounded output leaves room for the arithmetic.
* O at |ref| >= 4: half a bf16 ulp alone is >= 2^-6 > 1e-2, so no bf16 output can meet
  1e-2 there.  The bound is the output rounding plus the kernel's arithmetic:
  ``ulp_bf16(|ref| + E) / 2 + E`` with ``E = (u_w + 2^-13) * A``, where
  ``A[c] = sum_j softmax_j |v_j[c]|`` is the oracle's output with every V element
  replaced by its magnitude.  Derivation: the producer accumulates the normaliser
  ``l`` from the fp32 weights p_j and feeds the PV product each weight as two MMA
  operands, the weight rounded to the operand type and its rounding residual rounded
  again (bf16 KV: p_j, relative error u_w <= 2^-8 * 2^-8 = 2^-16; int8 KV: p_j times
  the V scale in fp16, u_w <= 2^-11 * 2^-11 = 2^-22); int8 codes are exact in fp16.
  So the output is ``sum_j p_j (1 + d_j) v_j / l`` with |d_j| <= u_w, off by at most
  ``u_w * A``.  The 2^-13 * A term covers the fp32 parts (score rounding, exp2, the
  MMA accumulation over a split's 16-token slices and the split merges; each is a
  relative error far below 2^-13 for scores of magnitude below ~100 and splits below
  ~65536 tokens).  ``ulp(|ref| + E)`` allows for the computed value lying across a
  binade boundary from the reference.
  int8 adds one absolute term: the fp16 weights are scaled so that the largest V scale
  seen maps to [64, 128), and a weight part below fp16's normal range (2^-14) is
  rounded with absolute error <= 2^-25 in those units, 2^-31 * max(v_scale) in V units
  per unit code; over n <= max(cache_seqlens) tokens of codes <= 127 and a normaliser
  >= 1 that is at most ``2^-31 * max(v_scale) * 127 * n`` (``Expected.abs_floor``).
  Below |ref| = 4 these bounds are at most 2^-7 + 1.4e-4 * A + the floor, inside 1e-2
  for any |V| <= 15: the literal bound is guaranteed, not just observed.
"""

from __future__ import annotations

import concurrent.futures
import json
import os

import numpy as np
import torch

import oracle

O_ATOL = 1e-2
LSE_ATOL = 1e-3
# |ref| from which half a bf16 ulp (2^-6 at 4) exceeds O_ATOL
ULP_BAND = 4.0
# relative error of the PV weights in the tensor-core producer (a weight and its residual,
# each rounded to the MMA operand type), by KV type; "fp32" for arithmetic that rounds
# no weight (the reducer alone)
WEIGHT_UNIT = {"bf16": 2.0 ** -16, "int8": 2.0 ** -22, "fp32": 0.0}
FP32_MARGIN = 2.0 ** -13

BANDS = [(0.0, 0.5), (0.5, 1.0), (1.0, 2.0), (2.0, 4.0), (4.0, np.inf)]

# per-band maximum O errors seen in this process (written out at session end when the
# PA_PARITY_REPORT environment variable names a file)
PARITY_RECORD: list[dict] = []


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (normal range)."""
    _, e = np.frexp(np.abs(x))            # |x| = m * 2**e, m in [0.5, 1)
    return np.ldexp(1.0, e - 8)


def out_tolerance(ref: np.ndarray, abs_ref: np.ndarray | None, weight: str,
                  abs_floor: float = 0.0) -> np.ndarray:
    """Per-element O bound (see the module docstring); ``abs_ref`` is needed only where
    |ref| >= 4."""
    tol = np.full(ref.shape, O_ATOL)
    big = np.abs(ref) >= ULP_BAND
    if big.any():
        if abs_ref is None:
            raise AssertionError("reference values >= 4 need the oracle's |V| output")
        e = (WEIGHT_UNIT[weight] + FP32_MARGIN) * abs_ref[big] + abs_floor
        tol[big] = 0.5 * bf16_ulp(np.abs(ref[big]) + e) + e
    return tol


def subnormal_floor(weight: str, v_scale, cache_seqlens) -> float:
    """The int8 producer's absolute bound for PV weights below fp16's normal range (see
    the module docstring); 0 for other weight types."""
    if weight != "int8" or v_scale is None or np.size(cache_seqlens) == 0:
        return 0.0
    return 2.0 ** -31 * float(np.max(v_scale)) * 127.0 * float(max(1, np.max(cache_seqlens)))


def abs_values(v: np.ndarray) -> np.ndarray:
    """|V| in the oracle's input encoding: int8 code magnitudes, or bf16 bit patterns
    with the sign bit cleared."""
    if v.dtype == np.int8:
        return np.minimum(np.abs(v.astype(np.int16)), 127).astype(np.int8)
    return (v & np.uint16(0x7FFF)).astype(np.uint16)


class Expected:
    """The oracle's (out, lse) for one call, and, computed only when needed, the same
    oracle call on |V| (the A of the tolerance).  ``fn`` is an oracle function whose
    third positional argument is the V cache (or, for ``combine_splits``, the acc
    partials); ``weight`` names the producer's weight rounding (by KV type)."""

    def __init__(self, fn, *args, weight=None, **kwargs):
        self.fn, self.args, self.kwargs = fn, args, kwargs
        v = args[2]
        self.weight = weight or ("int8" if v.dtype == np.int8 else "bf16")
        self.out, self.lse = fn(*args, **kwargs)
        self._abs = None
        # v_scale is the last positional argument and cache_seqlens the fifth of every
        # oracle attention function
        self.abs_floor = subnormal_floor(self.weight, args[-1], args[4]) \
            if self.weight == "int8" else 0.0

    def abs_out(self) -> np.ndarray:
        if self._abs is None:
            args = list(self.args)
            args[2] = np.abs(args[2]) if args[2].dtype == np.float64 else abs_values(args[2])
            self._abs = self.fn(*args, **self.kwargs)[0]
        return self._abs


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


def threads() -> int:
    return max(1, os.cpu_count() or 1)


def rows_threaded(fn, q, k, v, pt, cl, *args, **kwargs):
    """An oracle function with one query row per request (q [bs, Hq, d], page table
    [bs, ...], lengths [bs]) called one request per task on every host core (the
    oracle's C call releases the interpreter lock).  Same values as one call."""
    bs = q.shape[0]
    if bs <= 2:
        return fn(q, k, v, pt, cl, *args, **kwargs)

    def one(r):
        return fn(q[r:r + 1], k, v, pt[r:r + 1], cl[r:r + 1], *args, **kwargs)
    with concurrent.futures.ThreadPoolExecutor(min(threads(), bs)) as ex:
        parts = list(ex.map(one, range(bs)))
    return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))


def paged_attention_threaded(q, k, v, pt, cl, sm_scale, k_scale=None, v_scale=None):
    """oracle.paged_attention over all rows, spread over the host cores."""
    return rows_threaded(oracle.paged_attention, q, k, v, pt, cl, sm_scale, k_scale, v_scale)


def paged_attention_window_threaded(q, k, v, pt, cl, window, sm_scale, k_scale=None,
                                    v_scale=None):
    """oracle.paged_attention_window (one query per request) spread over the host cores."""
    return rows_threaded(oracle.paged_attention_window, q, k, v, pt, cl, window, sm_scale,
                         None, k_scale, v_scale)


def oracle_attention(wl, meta, rows=None) -> Expected:
    """Oracle output/LSE for the requests in ``rows`` (all by default)."""
    rows = np.arange(wl.spec.bs) if rows is None else np.asarray(rows)
    k, v, ks, vs = kv_np(wl)
    q = bits(wl.q)[rows]
    return Expected(paged_attention_threaded, q, k, v, meta["page_table"][rows],
                    meta["cache_seqlens"][rows], wl.sm_scale, ks, vs)


def oracle_partials(wl, meta, num_splits, rows=None, v_override=None):
    rows = np.arange(wl.spec.bs) if rows is None else np.asarray(rows)
    k, v, ks, vs = kv_np(wl)
    if v_override is not None:
        v = v_override
    q = bits(wl.q)[rows]
    return oracle.splitk_partials(q, k, v, meta["page_table"][rows], meta["cache_seqlens"][rows],
                                  wl.sm_scale, wl.max_seq_pages, num_splits, ks, vs)


def assert_partials_close(m, l, acc, m_ref, l_ref, acc_ref, acc_abs, weight, what="",
                          abs_floor=0.0):
    """Split partials (m natural-log max, l sum of exponentials, acc unnormalised output)
    against the oracle's: m within 1e-4 (relative, at least 1e-4 absolute), l within 1e-4
    relative, and acc = sum_j p_j v_j within (u_w + 2^-13) * sum_j p_j |v_j| (each PV
    weight carried as two MMA operands, see the module docstring; ``acc_abs`` is the
    oracle's acc over |V|, same split partition and maximum; ``abs_floor``: the int8
    subnormal-weight term, ``subnormal_floor``).  Empty splits: m = -inf, l = 0."""
    m, l, acc = (np.asarray(t, np.float64) for t in (m, l, acc))
    empty = np.isneginf(m_ref)
    assert np.array_equal(np.isneginf(m), empty), f"{what}: empty-split pattern differs"
    assert np.all(l[empty] == 0), f"{what}: empty split with l != 0"
    full = ~empty
    if not full.any():
        return
    m_err = np.abs(m[full] - m_ref[full]).max()
    assert m_err <= 1e-4 * max(1.0, np.abs(m_ref[full]).max()), f"{what}: m err {m_err}"
    l_rel = (np.abs(l[full] - l_ref[full]) / l_ref[full]).max()
    assert l_rel <= 1e-4, f"{what}: l relative err {l_rel}"
    err = np.abs(acc[full] - acc_ref[full])
    tol = (WEIGHT_UNIT[weight] + FP32_MARGIN) * acc_abs[full] + abs_floor + 1e-30
    ratio = err / tol
    if ratio.max() > 1:
        i = np.unravel_index(np.argmax(ratio), ratio.shape)
        raise AssertionError(
            f"{what}: acc error {err[i]:.3e} > bound {tol[i]:.3e} (ratio {ratio[i]:.2f}) at "
            f"split row {i[0]} channel {i[1]}: got {acc[full][i]:.6e}, oracle "
            f"{acc_ref[full][i]:.6e}, oracle over |V| {acc_abs[full][i]:.6e}, l "
            f"{l_ref[full][i[0]]:.6e}, m {m_ref[full][i[0]]:.6f}; err/acc_abs max "
            f"{(err / np.maximum(acc_abs[full], 1e-30)).max():.3e}")


def band_errors(o: np.ndarray, ref: np.ndarray) -> dict:
    """Max |o - ref| per |ref| band (bands with no element are left out)."""
    err = np.abs(o - ref)
    mag = np.abs(ref)
    out = {}
    for lo, hi in BANDS:
        m = (mag >= lo) & (mag < hi)
        if m.any():
            out[f"[{lo:g},{hi:g})"] = float(err[m].max())
    return out


def assert_attention_close(out_gpu, lse_gpu, ref, what=""):
    """``ref``: an ``Expected`` (or an (out, lse) pair when every |ref| < 4)."""
    if isinstance(ref, tuple):
        out_ref, lse_ref, abs_fn, weight, floor = ref[0], ref[1], None, "bf16", 0.0
    else:
        out_ref, lse_ref, abs_fn, weight = ref.out, ref.lse, ref.abs_out, ref.weight
        floor = ref.abs_floor
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.float().cpu().numpy().astype(np.float64)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: empty-row pattern differs"
    if empty.any():
        assert np.all(o[empty] == 0.0), f"{what}: empty rows must be 0"
    full = ~empty
    if not full.any():
        return 0.0, 0.0
    o_f, r_f = o[full], out_ref[full]
    big = np.abs(r_f) >= ULP_BAND
    abs_f = abs_fn()[full] if big.any() else None
    tol = out_tolerance(r_f, abs_f, weight, floor)
    err = np.abs(o_f - r_f)
    o_err = float(err.max())
    l_err = float(np.abs(lse[full] - lse_ref[full]).max())
    bands = band_errors(o_f, r_f)
    PARITY_RECORD.append({"case": what, "weight": weight, "out_max_err_by_band": bands,
                          "lse_max_err": l_err, "elements": int(r_f.size)})
    excess = float((err - tol).max())
    assert excess <= 0, (f"{what}: out max abs err {o_err} beyond tolerance by {excess}; "
                         f"max err per |ref| band {bands}")
    assert l_err <= LSE_ATOL, f"{what}: lse max abs err {l_err}; out max err per band {bands}"
    return o_err, l_err


def write_parity_report():
    path = os.environ.get("PA_PARITY_REPORT")
    if not path or not PARITY_RECORD:
        return
    worst = {}
    for rec in PARITY_RECORD:
        for band, e in rec["out_max_err_by_band"].items():
            worst[band] = max(worst.get(band, 0.0), e)
    with open(path, "w") as f:
        json.dump({"cases": len(PARITY_RECORD), "out_max_err_by_band": worst,
                   "lse_max_err": max(r["lse_max_err"] for r in PARITY_RECORD),
                   "records": PARITY_RECORD}, f, indent=1)
