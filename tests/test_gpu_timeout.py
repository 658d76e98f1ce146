"""Failure detection without a GPU fault: every wait of the split-K producer gives up
after a time limit, records it in the device error word and returns, and the context
stays usable.  The instrumented build's test hook makes the producer issue no copies,
so the consumers' first wait runs out (a stage that nothing fills)."""

import ctypes
import time

import pytest
import torch

from paged_kv_decode_metadata_gb300 import binding as B
from paged_kv_decode_metadata_gb300 import build, synthetic

from helpers import assert_attention_close, oracle_attention, oracle_metadata

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    build.build(instrumented=True)
    lib = B.load_instrumented()
    B.pa_read_error_flags(reset=True, lib=lib)
    yield lib
    lib.pa_set_test_hold_loads(0)


def _splitk(lib, wl, meta, dev_bufs, splits):
    q, k, v, pt, cl, m, l, acc = dev_bufs
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.pa_decode_splitk(p(q), p(k), p(v), None, None, B.PA_KV_BF16, p(pt), pt.stride(0),
                                p(cl), wl.spec.bs, wl.spec.num_q_heads, wl.spec.num_kv_heads,
                                128, wl.spec.page_size, wl.spec.num_pages, wl.max_seq_pages,
                                splits, wl.sm_scale, p(m), p(l), p(acc), None, 0)


def test_wait_limit_reports_and_returns(ts):
    spec = synthetic.Spec("stall", bs=1, num_q_heads=8, num_kv_heads=1, num_pages=4, ctx=128,
                          num_splits=1, seed=77)
    wl = synthetic.make(spec)
    meta = oracle_metadata(wl)
    dev = "cuda"
    f32 = dict(dtype=torch.float32, device=dev)
    bufs = (wl.q.to(dev), wl.k_cache.to(dev), wl.v_cache.to(dev),
            torch.from_numpy(meta["page_table"]).to(dev),
            torch.from_numpy(meta["cache_seqlens"]).to(dev),
            torch.empty((1, 8, 1), **f32), torch.empty((1, 8, 1), **f32),
            torch.empty((1, 8, 1, 128), **f32))
    with B.producer(B.PA_PRODUCER_MMA):
        assert ts.pa_set_test_hold_loads(1) == B.PA_OK
        try:
            t0 = time.perf_counter()
            assert _splitk(ts, wl, meta, bufs, 1) == B.PA_OK
            torch.cuda.synchronize()
            waited = time.perf_counter() - t0
        finally:
            ts.pa_set_test_hold_loads(0)
        flags = B.pa_read_error_flags(reset=True, lib=ts)
        assert flags & B.DEVERR_WAIT_TIMEOUT, hex(flags)
        assert 1.0 < waited < 60.0, waited          # one wait limit, then a bounded drain
        # the same context, the hook off: a normal launch and the right answer
        assert _splitk(ts, wl, meta, bufs, 1) == B.PA_OK
        out = torch.empty((1, 8, 128), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((1, 8), **f32)
        p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
        assert ts.pa_reduce(p(bufs[5]), p(bufs[6]), p(bufs[7]), 1, 8, 128, 1, p(out), p(lse),
                            None, 0) == B.PA_OK
        torch.cuda.synchronize()
        assert B.pa_read_error_flags(reset=True, lib=ts) == 0
    assert_attention_close(out, lse, oracle_attention(wl, meta), "after timeout")


def test_persistent_form_recovers_after_timeout(ts):
    """An int8 batch large enough for the persistent form (one CTA per resident slot
    claiming items from a per-launch counter slot): with the hook on, every CTA's
    consumers time out and the launch reports it; with the hook off, the next 70
    launches (every counter slot reused at least once) each give the oracle's answer."""
    spec = synthetic.Spec("stall8", bs=32, num_q_heads=64, num_kv_heads=8, num_pages=300,
                          ctx=512, kv_dtype="int8", num_splits=4, seed=78)
    wl = synthetic.make(spec)
    meta = oracle_metadata(wl)
    dev = "cuda"
    f32 = dict(dtype=torch.float32, device=dev)
    S = spec.num_splits
    q, k, v = wl.q.to(dev), wl.k_cache.to(dev), wl.v_cache.to(dev)
    ks, vs = wl.k_scale.to(dev), wl.v_scale.to(dev)
    pt = torch.from_numpy(meta["page_table"]).to(dev)
    cl = torch.from_numpy(meta["cache_seqlens"]).to(dev)
    m = torch.empty((spec.bs, spec.num_q_heads, S), **f32)
    l = torch.empty((spec.bs, spec.num_q_heads, S), **f32)
    acc = torch.empty((spec.bs, spec.num_q_heads, S, 128), **f32)
    out = torch.empty((spec.bs, spec.num_q_heads, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((spec.bs, spec.num_q_heads), **f32)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    def splitk():
        return ts.pa_decode_splitk(p(q), p(k), p(v), p(ks), p(vs), B.PA_KV_INT8, p(pt),
                                   pt.stride(0), p(cl), spec.bs, spec.num_q_heads,
                                   spec.num_kv_heads, 128, spec.page_size, spec.num_pages,
                                   wl.max_seq_pages, S, wl.sm_scale, p(m), p(l), p(acc),
                                   None, 0)

    with B.producer(B.PA_PRODUCER_MMA):
        assert ts.pa_set_test_hold_loads(1) == B.PA_OK
        try:
            assert splitk() == B.PA_OK
            torch.cuda.synchronize()
        finally:
            ts.pa_set_test_hold_loads(0)
        flags = B.pa_read_error_flags(reset=True, lib=ts)
        assert flags & B.DEVERR_WAIT_TIMEOUT, hex(flags)
        ref = oracle_attention(wl, meta)
        for rep in range(70):
            acc.fill_(float("nan"))
            assert splitk() == B.PA_OK
            if rep % 10 == 9 or rep == 0:
                assert ts.pa_reduce(p(m), p(l), p(acc), spec.bs, spec.num_q_heads, 128, S,
                                    p(out), p(lse), None, 0) == B.PA_OK
                torch.cuda.synchronize()
                assert B.pa_read_error_flags(reset=True, lib=ts) == 0
                assert_attention_close(out, lse, ref, f"launch {rep} after timeout")
