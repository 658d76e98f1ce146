"""The persistent form of the tensor-core producer (one CTA per resident slot claiming
items of a largest-first work list; the library runs it for large int8 full-context
grids).  With the instrumented build's hook the same steps run with one block per item:
both forms must give the same bits, and the oracle's answer."""

import pytest
import torch

from paged_kv_decode_metadata_gb300 import binding as B
from paged_kv_decode_metadata_gb300 import build, synthetic
from paged_kv_decode_metadata_gb300.runtime import DeviceStep

from helpers import assert_attention_close, oracle_attention, oracle_metadata

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts_lib():
    build.build()
    build.build(instrumented=True)
    B.load()
    lib = B.load_instrumented()
    yield lib
    lib.pa_set_test_no_persist(0)


def _run(ds, lib, no_persist):
    """One decode step through `lib` (pa_decode_step); returns (out, lse)."""
    assert lib.pa_set_test_no_persist(int(no_persist)) == B.PA_OK
    ds.out.fill_(float("nan"))
    ds.lse.fill_(float("nan"))
    ds.step(use_pdl=True, lib=lib)
    torch.cuda.synchronize()
    assert B.pa_read_error_flags(reset=True, lib=lib) == 0
    return ds.out.clone(), ds.lse.clone()


@pytest.mark.parametrize("spec", [
    synthetic.WORKLOADS["bs64_ragged16k_int8_swa"],
    # many empty splits: most CTAs of the persistent grid find no item at all
    synthetic.Spec("persist_sparse", bs=128, num_q_heads=8, num_kv_heads=1, num_pages=128 * 4 + 2,
                   ragged=(1, 200), kv_dtype="int8", num_splits=16, seed=4343),
    # every request the same length: a work list of full splits only
    synthetic.Spec("persist_uniform", bs=40, num_q_heads=32, num_kv_heads=8, num_pages=40 * 40,
                   ctx=2560, kv_dtype="int8", num_splits=5, seed=4344),
])
def test_persistent_form_matches_one_block_per_item(ts_lib, spec):
    wl = synthetic.make(spec)
    ds = DeviceStep(wl)
    blocks = ds.num_splits * spec.num_kv_heads * spec.bs
    assert blocks >= 2 * 3 * torch.cuda.get_device_properties(0).multi_processor_count
    a = _run(ds, ts_lib, no_persist=False)
    b = _run(ds, ts_lib, no_persist=True)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16)) and torch.equal(a[1], b[1])
    # once more: the work-claim counter must have been handed back clean
    c = _run(ds, ts_lib, no_persist=False)
    assert torch.equal(a[0].view(torch.int16), c[0].view(torch.int16)) and torch.equal(a[1], c[1])
    meta = oracle_metadata(wl)
    ds.out.copy_(a[0])
    ds.lse.copy_(a[1])
    assert_attention_close(ds.out, ds.lse, oracle_attention(wl, meta), spec.name)


def test_persistent_form_in_a_cuda_graph_of_steps(ts_lib):
    """Eight steps with PDL in one CUDA graph (the benchmark's configuration) through the
    production library: the graph's replays equal the eager step bit for bit."""
    wl = synthetic.make(synthetic.WORKLOADS["bs64_ragged16k_int8_swa"])
    ds = DeviceStep(wl)
    ds.step(use_pdl=True)
    torch.cuda.synchronize()
    want = (ds.out.clone(), ds.lse.clone())
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(8):
            ds.step(use_pdl=True)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(8):
            ds.step(use_pdl=True)
    for _ in range(3):
        ds.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(ds.out, want[0]) and torch.equal(ds.lse, want[1])
    assert B.pa_read_error_flags(reset=True) == 0


def _persist_spec(seed):
    """A random int8 full-context batch big enough for the persistent form: G in
    {1, 2, 4, 8}, Hkv in {1, 2, 4, 8}, page 16-128, ragged lengths, 2-24 splits."""
    g = torch.Generator().manual_seed(70_000 + seed)
    pick = lambda xs: xs[int(torch.randint(0, len(xs), (1,), generator=g))]  # noqa: E731
    grp, hkv, P = pick([1, 2, 4, 8]), pick([1, 2, 4, 8]), pick([16, 32, 64, 128])
    ctx_max = pick([300, 2000, 9000])
    slots = 3 * torch.cuda.get_device_properties(0).multi_processor_count
    splits = int(torch.randint(2, 25, (1,), generator=g))
    bs = max(int(torch.randint(1, 129, (1,), generator=g)), -(-2 * slots // (splits * hkv)))
    bs = min(bs, 128)
    return synthetic.Spec(f"persist_fuzz{seed}", bs=bs, num_q_heads=grp * hkv, num_kv_heads=hkv,
                          num_pages=bs * (-(-ctx_max // P)) + 2, ragged=(1, ctx_max),
                          page_size=P, kv_dtype="int8", num_splits=splits,
                          seqlen_offset=int(torch.randint(0, 2, (1,), generator=g)),
                          seed=71_000 + seed)


# 8 seeds by default; PA_PERSIST_SEEDS=n draws n
@pytest.mark.parametrize("seed", range(int(__import__("os").environ.get("PA_PERSIST_SEEDS", "8"))))
def test_persistent_form_random_batches(ts_lib, seed):
    """Random batches that take the persistent form (at least two blocks per resident
    slot, at most 128 requests): the same bits as one block per item, every request
    against the oracle."""
    spec = _persist_spec(seed)
    wl = synthetic.make(spec)
    ds = DeviceStep(wl)
    if ds.num_splits * spec.num_kv_heads * spec.bs < 2 * 3 * torch.cuda.get_device_properties(0).multi_processor_count:
        pytest.skip("grid too small for the persistent form")
    a = _run(ds, ts_lib, no_persist=False)
    b = _run(ds, ts_lib, no_persist=True)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16)) and torch.equal(a[1], b[1])
    ds.out.copy_(a[0])
    ds.lse.copy_(a[1])
    assert_attention_close(ds.out, ds.lse, oracle_attention(wl, oracle_metadata(wl)), spec.name)
