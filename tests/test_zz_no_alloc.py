"""pa_decode_step_static_scratch, the decode step for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run a decode step: runtimes whose device
memory belongs entirely to their own allocator, latency-critical paths that cannot take
cudaMalloc's implicit synchronisation, plain C hosts without a device allocator.  This
entry point takes its split-K scratch from an array built into the library instead of a
workspace argument.  The test runs it through the C ABI twice in a row and checks each
result against pa_decode_step's on the same inputs.  Both run the same kernels with the
same split count, so the outputs must be identical bit for bit (tighter than the
attention tolerances the other tests use).  This file is named to be collected last; it
builds and loads everything it needs, so it also passes on its own.
"""

import pytest
import torch

from paged_kv_decode_metadata_gb300 import binding as B
from paged_kv_decode_metadata_gb300 import build, synthetic
from paged_kv_decode_metadata_gb300.runtime import DeviceStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return B.load()


def _static_step(ds, out, lse):
    B.pa_decode_step_static_scratch(
        req_pool_indices=ds.req_pool_indices, seq_lens=ds.seq_lens, req_to_token=ds.req_to_token,
        seqlen_offset=ds.seqlen_offset, max_seq_pages=ds.max_seq_pages,
        cache_seqlens=ds.cache_seqlens, cu_seqlens_k=ds.cu_seqlens_k, page_table=ds.page_table,
        q=ds.q, k_cache=ds.k_cache, v_cache=ds.v_cache, num_splits=ds.num_splits,
        sm_scale=ds.sm_scale, out=out, lse=lse, k_scale=ds.k_scale, v_scale=ds.v_scale,
        full_to_swa_mapping=ds.full_to_swa_mapping, swa_page_table=ds.swa_page_table)


@pytest.mark.parametrize("spec", [
    synthetic.WORKLOADS["bs8_ctx1k"],
    synthetic.Spec("int8_ragged", bs=6, num_q_heads=32, num_kv_heads=4, num_pages=300,
                   ragged=(1, 3000), kv_dtype="int8", num_splits=7, swa_window=512, seed=4242),
])
def test_static_scratch_step_matches_workspace_step(spec):
    wl = synthetic.make(spec)
    ds = DeviceStep(wl)
    assert B.pa_workspace_bytes(ds.bs, ds.num_q_heads, ds.head_dim, ds.num_splits) \
        <= B.PA_STATIC_SCRATCH_BYTES
    ds.step()                                   # the existing entry point, own workspace
    torch.cuda.synchronize()
    want_out, want_lse = ds.out.clone(), ds.lse.clone()
    for _ in range(2):                          # two calls in a row share the array
        out = torch.full_like(ds.out, float("nan"))
        lse = torch.full_like(ds.lse, float("nan"))
        _static_step(ds, out, lse)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), want_out.view(torch.int16)), spec.name
        assert torch.equal(lse, want_lse), spec.name
    assert B.pa_read_error_flags(reset=True) == 0


def test_static_scratch_rejects_steps_that_do_not_fit(lib):
    fake = 1 << 20                              # never dereferenced: rejected first
    need = B.pa_workspace_bytes(64, 64, 128, 64)
    assert need > B.PA_STATIC_SCRATCH_BYTES
    st = lib.pa_decode_step_static_scratch(
        fake, fake, fake, 64, 16384, None, 0, 0, 256, fake, fake, fake, 256, None, 0, fake, fake,
        fake, None, None, 0, 64, 64, 8, 128, 64, 20000, 64, 0.088, fake, None, None, 1)
    assert st == B.PA_ERR_SCRATCH_LIMIT
    assert B.pa_status_string(st).startswith("step needs more scratch")
