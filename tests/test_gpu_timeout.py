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
