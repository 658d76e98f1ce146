"""GPU parity of the sliding-window producer (attention through the sliding-window page
table) against the float64 oracle: outputs and LSE within the attention tolerance,
split partials on the window's partition, skipped (-1) pages, multi-token queries,
PDL on/off bit-identical, and the full-size int8 ragged batch with window 4096."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_metadata_gb300 import binding as B
from paged_kv_decode_metadata_gb300 import build, synthetic
from paged_kv_decode_metadata_gb300.runtime import WindowStep

from helpers import (Expected, abs_values, assert_attention_close, assert_partials_close, bits,
                     oracle_metadata, paged_attention_window_threaded, subnormal_floor)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    B.load()
    B.pa_read_error_flags(reset=True)
    yield
    assert B.pa_read_error_flags(reset=True) == 0


def _swa_np(wl):
    if wl.spec.kv_dtype == "int8":
        return (wl.k_swa.numpy(), wl.v_swa.numpy(), wl.k_swa_scale.numpy(),
                wl.v_swa_scale.numpy())
    return bits(wl.k_swa), bits(wl.v_swa), None, None


def _case(seed, kv, grp, P, window, max_q_len=None, holes=0, bs=4, ctx_max=700):
    spec = synthetic.Spec(f"win{seed}", bs=bs, num_q_heads=2 * grp, num_kv_heads=2,
                          num_pages=bs * (-(-ctx_max // P)) + 2, ragged=(1, ctx_max),
                          page_size=P, kv_dtype=kv, seqlen_offset=seed % 2,
                          swa_window=window, seed=1200 + seed)
    wl = synthetic.make(spec, with_cache=False, with_swa_cache=True)
    meta = oracle_metadata(wl)
    table = meta["swa_page_table"].copy()
    g = torch.Generator().manual_seed(seed)
    for _ in range(holes):          # knock out mapped pages: the producer must skip them
        b = int(torch.randint(0, bs, (1,), generator=g))
        mapped = sorted(wl.swa_pages[b])
        table[b, mapped[int(torch.randint(0, len(mapped), (1,), generator=g))]] = -1
    cu_q, q = None, wl.q
    if max_q_len is not None:
        qlens = synthetic.draw_query_lengths(bs, max_q_len, 1300 + seed)
        cu_q = oracle.cu_seqlens_q(qlens.numpy(), bs, 1)
        q = synthetic.draw_queries(int(cu_q[-1]), spec.num_q_heads, spec.head_dim, 1400 + seed)
    return wl, meta, table, q, cu_q


def _run(wl, meta, table, q, cu_q, num_splits, use_pdl=True, max_q_len=None):
    """GPU: window producer + reducer over the given table; returns out, lse, m, l, acc.
    ``max_q_len`` (the bound the query lengths were drawn under) fixes the split
    partition; by default the longest drawn query count."""
    dev = "cuda"
    rows, hq, d = q.shape
    f32 = dict(dtype=torch.float32, device=dev)
    m = torch.empty((rows, hq, num_splits), **f32)
    l = torch.empty((rows, hq, num_splits), **f32)
    acc = torch.empty((rows, hq, num_splits, d), **f32)
    out = torch.empty((rows, hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((rows, hq), **f32)
    ks = wl.k_swa_scale.to(dev) if wl.k_swa_scale is not None else None
    vs = wl.v_swa_scale.to(dev) if wl.v_swa_scale is not None else None
    mql = 1 if cu_q is None else (max_q_len or int(np.diff(cu_q).max()))
    B.pa_decode_splitk_window(
        q.to(dev), wl.k_swa.to(dev), wl.v_swa.to(dev), torch.from_numpy(table).to(dev),
        torch.from_numpy(meta["cache_seqlens"]).to(dev), m, l, acc,
        sliding_window=wl.spec.swa_window, max_seq_pages=wl.max_seq_pages,
        num_splits=num_splits, sm_scale=wl.sm_scale,
        cu_seqlens_q=None if cu_q is None else torch.from_numpy(cu_q).to(dev), max_q_len=mql,
        k_scale=ks, v_scale=vs, use_pdl=use_pdl)
    B.pa_reduce(m, l, acc, out, lse, use_pdl=use_pdl)
    torch.cuda.synchronize()
    return out, lse, m, l, acc


def _oracle(wl, meta, table, q, cu_q, window=None):
    k, v, ks, vs = _swa_np(wl)
    return Expected(oracle.paged_attention_window, bits(q), k, v, table, meta["cache_seqlens"],
                    window or wl.spec.swa_window, wl.sm_scale, cu_q, ks, vs)


CASES = [  # seed, kv, group, page_size, window, max_q_len, holes, splits
    (1, "bf16", 4, 64, 150, None, 0, 3), (2, "int8", 8, 64, 150, None, 2, 2),
    (3, "bf16", 8, 16, 37, None, 3, 4), (4, "int8", 4, 32, 100, None, 1, 5),
    (5, "bf16", 1, 128, 300, None, 0, 1), (6, "int8", 16, 64, 64, None, 2, 3),
    (7, "bf16", 2, 16, 1, None, 0, 2), (8, "int8", 8, 128, 5000, None, 0, 3),
    (9, "bf16", 4, 64, 150, 4, 2, 3), (10, "int8", 8, 32, 90, 2, 1, 4),
    (11, "bf16", 1, 16, 20, 16, 0, 2), (12, "int8", 2, 128, 130, 8, 3, 6),
]


@pytest.mark.parametrize("seed,kv,grp,P,window,mql,holes,splits", CASES)
def test_window_matches_oracle(seed, kv, grp, P, window, mql, holes, splits):
    wl, meta, table, q, cu_q = _case(seed, kv, grp, P, window, mql, holes)
    out, lse, *_ = _run(wl, meta, table, q, cu_q, splits)
    assert_attention_close(out, lse, _oracle(wl, meta, table, q, cu_q), wl.spec.name)


@pytest.mark.parametrize("seed,kv,grp,P,window,mql,holes,splits",
                         [CASES[1], CASES[2], CASES[9], CASES[11]])
def test_window_partials_match_oracle(seed, kv, grp, P, window, mql, holes, splits):
    wl, meta, table, q, cu_q = _case(seed, kv, grp, P, window, mql, holes)
    _, _, m, l, acc = _run(wl, meta, table, q, cu_q, splits, max_q_len=mql)
    k, v, ks, vs = _swa_np(wl)
    m_ref, l_ref, acc_ref = oracle.splitk_partials_window(
        bits(q), k, v, table, meta["cache_seqlens"], window, wl.sm_scale, wl.max_seq_pages,
        splits, cu_q, mql or 1, ks, vs)
    _, _, acc_abs = oracle.splitk_partials_window(
        bits(q), k, abs_values(v), table, meta["cache_seqlens"], window, wl.sm_scale,
        wl.max_seq_pages, splits, cu_q, mql or 1, ks, vs)
    assert_partials_close(m.cpu(), l.cpu(), acc.cpu(), m_ref, l_ref, acc_ref, acc_abs, kv,
                          wl.spec.name, subnormal_floor(kv, vs, meta["cache_seqlens"]))


def test_every_page_skipped_gives_empty_rows():
    wl, meta, table, q, cu_q = _case(21, "bf16", 4, 64, 150)
    table[1, :] = -1
    out, lse, *_ = _run(wl, meta, table, q, cu_q, 3)
    ref = _oracle(wl, meta, table, q, cu_q)
    assert np.all(np.isneginf(ref.lse[1]))
    assert_attention_close(out, lse, ref, "all skipped")


def test_window_pdl_on_off_identical():
    wl, meta, table, q, cu_q = _case(22, "int8", 8, 16, 200, 2, 2)
    a = _run(wl, meta, table, q, cu_q, 4, use_pdl=True)
    b = _run(wl, meta, table, q, cu_q, 4, use_pdl=False)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_window_step_bs64_ragged_int8():
    """The int8 ragged batch (64 requests, lengths U[1, 16384], 64/8 heads) through its
    sliding-window layer (window 4096): metadata, window producer and reducer in one
    call, every request against the oracle (spread over the host cores)."""
    wl = synthetic.make(synthetic.WORKLOADS["bs64_ragged16k_int8_swa"], with_cache=False,
                        with_swa_cache=True)
    ws = WindowStep(wl)
    ws.step(use_pdl=True)
    torch.cuda.synchronize()
    assert B.pa_read_error_flags(reset=True) == 0
    meta = oracle_metadata(wl)
    assert np.array_equal(ws.swa_page_table.cpu().numpy(), meta["swa_page_table"])
    k, v, ks, vs = _swa_np(wl)
    ref = Expected(paged_attention_window_threaded, bits(wl.q), k, v, meta["swa_page_table"],
                   meta["cache_seqlens"], wl.spec.swa_window, wl.sm_scale, ks, vs)
    assert_attention_close(ws.out, ws.lse, ref, "bs64 window")
    # the same step with q / req_pool_indices / seq_lens / out / lse in pinned host
    # memory (no copies): the same bits
    h_in, h_outs, (h_q, h_rpi, h_sl, h_out, h_lse) = ws.host_buffers()
    h_q.copy_(ws.q)
    h_rpi.copy_(ws.req_pool_indices)
    h_sl.copy_(ws.seq_lens)
    ws.prepare_host_io_step(h_in, h_outs, use_pdl=True)()
    torch.cuda.synchronize()
    assert torch.equal(h_out, ws.out.cpu()) and torch.equal(h_lse, ws.lse.cpu())
    assert B.pa_read_error_flags(reset=True) == 0


def test_window_rejects_bad_arguments():
    wl, meta, table, q, cu_q = _case(23, "bf16", 4, 64, 150)
    dev = "cuda"
    f32 = dict(dtype=torch.float32, device=dev)
    args = (q.to(dev), wl.k_swa.to(dev), wl.v_swa.to(dev), torch.from_numpy(table).to(dev),
            torch.from_numpy(meta["cache_seqlens"]).to(dev), torch.empty((4, 8, 2), **f32),
            torch.empty((4, 8, 2), **f32), torch.empty((4, 8, 2, 128), **f32))
    with pytest.raises(B.PAError) as e:
        B.pa_decode_splitk_window(*args, sliding_window=0, max_seq_pages=wl.max_seq_pages,
                                  num_splits=2, sm_scale=wl.sm_scale)
    assert e.value.status == B.PA_ERR_INVALID
    with B.producer(B.PA_PRODUCER_FMA):
        with pytest.raises(B.PAError) as e:
            B.pa_decode_splitk_window(*args, sliding_window=10, max_seq_pages=wl.max_seq_pages,
                                      num_splits=2, sm_scale=wl.sm_scale)
    assert e.value.status == B.PA_ERR_UNSUPPORTED


def test_window_out_of_range_page_sets_error_flag_without_fault():
    """A sliding-window table entry past the pool is replaced by a safe page and flagged;
    nothing outside the pool is read."""
    wl, meta, table, q, cu_q = _case(24, "int8", 8, 64, 300)
    b = 2
    table[b, sorted(wl.swa_pages[b])[-1]] = wl.swa_num_pages + 7
    B.pa_read_error_flags(reset=True)
    _run(wl, meta, table, q, cu_q, 2)
    assert B.pa_read_error_flags(reset=True) & B.DEVERR_PAGE_OUT_OF_RANGE


def test_window_split_longer_than_the_cached_page_list():
    """A 20000-token window at page size 16 in one split (1251 pages): page indices past
    the first 256 come from the sliding-window table in global memory."""
    wl, meta, table, q, cu_q = _case(25, "bf16", 4, 16, 20000, holes=2, ctx_max=40000)
    assert B.pa_window_pages(20000, 1, 16, wl.max_seq_pages) > 256
    out, lse, *_ = _run(wl, meta, table, q, cu_q, 1)
    assert_attention_close(out, lse, _oracle(wl, meta, table, q, cu_q), "long window")
