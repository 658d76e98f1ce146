"""PDL wiring, checked with the timestamp-instrumented build: a stage never passes its
wait on the previous grid before that grid's last warp has finished, and the
instrumented build computes exactly what the production build computes."""

import numpy as np
import pytest
import torch

from paged_kv_decode_metadata_gb300 import binding as B
from paged_kv_decode_metadata_gb300 import build, synthetic
from paged_kv_decode_metadata_gb300.runtime import DeviceStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts_lib():
    build.build()
    build.build(instrumented=True)
    B.load()
    return B.load_instrumented()


def _stamps(buf):
    return buf.cpu().numpy().view(np.uint64).reshape(3, 3).astype(np.int64)


@pytest.mark.parametrize("use_pdl", [True, False])
@pytest.mark.parametrize("graph", [True, False])
@pytest.mark.parametrize("name", ["bs8_ctx1k", "bs1_ctx8k"])
def test_stages_wait_for_their_predecessor(ts_lib, name, graph, use_pdl):
    wl = synthetic.make(synthetic.WORKLOADS[name])
    ds = DeviceStep(wl)
    ds.step(use_pdl=use_pdl)                     # production build
    torch.cuda.synchronize()
    want = (ds.out.clone(), ds.lse.clone(), ds.page_table.clone())
    buf = torch.empty(9, dtype=torch.int64, device="cuda")
    init = torch.tensor([-1, -1, 0] * 3, dtype=torch.int64, device="cuda")
    assert ts_lib.pa_set_timestamp_buffer(buf.data_ptr()) == 0
    try:
        stream = torch.cuda.Stream()
        g = None
        if graph:
            with torch.cuda.stream(stream):
                ds.step(use_pdl=use_pdl, lib=ts_lib)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                ds.step(use_pdl=use_pdl, lib=ts_lib)
        for _ in range(5):
            ds.out.zero_()
            with torch.cuda.stream(stream):
                buf.copy_(init)
                if graph:
                    g.replay()
                else:
                    ds.step(use_pdl=use_pdl, lib=ts_lib)
            stream.synchronize()
            ts = _stamps(buf)
            entry, ready, exit_ = ts[:, 0], ts[:, 1], ts[:, 2]
            assert np.all(entry <= ready) and np.all(ready <= exit_), ts
            assert ready[1] >= exit_[0], ts        # producer waited for the metadata grid
            assert ready[2] >= exit_[1], ts        # reducer waited for the producer grid
            assert torch.equal(ds.out, want[0]) and torch.equal(ds.lse, want[1])
            assert torch.equal(ds.page_table, want[2])
    finally:
        ts_lib.pa_set_timestamp_buffer(None)
