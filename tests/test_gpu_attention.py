"""GPU parity of the split-K producer, the reducer and the whole decode step against
the float64 oracle (O max-abs <= 1e-2, LSE <= 1e-3), plus the properties the CUDA path
must have exactly: PDL on/off, eager vs CUDA-graph replay, page relabelling."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_metadata_gb300 import binding as B
from paged_kv_decode_metadata_gb300 import build, synthetic
from paged_kv_decode_metadata_gb300.runtime import DeviceStep

from helpers import (Expected, abs_values, assert_attention_close, assert_partials_close, kv_np,
                     oracle_attention, oracle_metadata, oracle_partials, subnormal_floor)

pytestmark = pytest.mark.gpu

_CACHE = {}


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    B.load()
    B.pa_read_error_flags(reset=True)
    yield
    _CACHE.clear()
    torch.cuda.empty_cache()


def named(name):
    if name not in _CACHE:
        _CACHE.clear()                      # keep at most one large workload resident
        torch.cuda.empty_cache()
        wl = synthetic.make(synthetic.WORKLOADS[name])
        _CACHE[name] = (wl, DeviceStep(wl))
    return _CACHE[name]


def _check_flags():
    assert B.pa_read_error_flags(reset=True) == 0


PRODUCERS = {"mma": B.PA_PRODUCER_MMA, "fma": B.PA_PRODUCER_FMA}


# ---- whole step on the five workloads --------------------------------------------------

@pytest.mark.parametrize("impl", sorted(PRODUCERS))
@pytest.mark.parametrize("name", synthetic.WORKLOAD_ORDER)
def test_decode_step_matches_oracle(name, impl):
    wl, ds = named(name)
    with B.producer(PRODUCERS[impl]):
        ds.step(use_pdl=True)
    torch.cuda.synchronize()
    _check_flags()
    meta = oracle_metadata(wl)
    assert np.array_equal(ds.cache_seqlens.cpu().numpy(), meta["cache_seqlens"])
    assert np.array_equal(ds.page_table.cpu().numpy()[:, :wl.max_seq_pages], meta["page_table"])
    if ds.swa_page_table is not None:
        assert np.array_equal(ds.swa_page_table.cpu().numpy(), meta["swa_page_table"])
    # every request of the step, the oracle spread over the host cores
    assert_attention_close(ds.out, ds.lse, oracle_attention(wl, meta), f"{name} {impl}")


@pytest.mark.parametrize("impl", sorted(PRODUCERS))
@pytest.mark.parametrize("name", ["bs1_ctx1k", "bs8_ctx1k", "bs1_ctx8k"])
def test_splitk_scratch_matches_oracle_partials(name, impl):
    wl, ds = named(name)
    ds.metadata()
    with B.producer(PRODUCERS[impl]):
        ds.splitk()
    torch.cuda.synchronize()
    _check_flags()
    meta = oracle_metadata(wl)
    m_ref, l_ref, acc_ref = oracle_partials(wl, meta, ds.num_splits)
    _, _, acc_abs = oracle_partials(wl, meta, ds.num_splits, v_override=abs_values(kv_np(wl)[1]))
    assert_partials_close(ds.scratch_m.cpu(), ds.scratch_l.cpu(), ds.scratch_acc.cpu(), m_ref,
                          l_ref, acc_ref, acc_abs, wl.spec.kv_dtype, f"{name} {impl}",
                          subnormal_floor(wl.spec.kv_dtype, kv_np(wl)[3], meta["cache_seqlens"]))


def test_reduce_alone_matches_oracle_combine():
    g = torch.Generator().manual_seed(3)
    bs, hq, S, d = 3, 8, 37, 128
    m = torch.randn(bs, hq, S, generator=g, dtype=torch.float64) * 4
    m[0, 0, :] = -np.inf                      # a row with no tokens
    m[1, :, ::3] = -np.inf                    # empty splits among full ones
    l = torch.rand(bs, hq, S, generator=g, dtype=torch.float64) * 50 + 1
    l[torch.isinf(m)] = 0
    acc = torch.randn(bs, hq, S, d, generator=g, dtype=torch.float64) * l[..., None]
    acc[torch.isinf(m)] = float("nan")        # must never be read
    m32, l32, acc32 = (t.float() for t in (m, l, acc))
    out = torch.empty(bs, hq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(bs, hq, dtype=torch.float32, device="cuda")
    B.pa_reduce(m32.cuda(), l32.cuda(), acc32.cuda(), out, lse)
    torch.cuda.synchronize()
    ref = Expected(oracle.combine_splits, m32.double().numpy(), l32.double().numpy(),
                   acc32.double().numpy(), weight="fp32")
    assert_attention_close(out, lse, ref, "reduce")


# ---- small random shapes: every group size, page size and KV type ---------------------

SMALL = [(seed, kv, grp, P) for seed, (kv, grp, P) in enumerate(
    [(kv, grp, P) for kv in ("bf16", "int8") for grp in (1, 2, 4, 8, 16)
     for P in (16, 32, 64, 128)])]


@pytest.mark.parametrize("impl", sorted(PRODUCERS))
@pytest.mark.parametrize("seed,kv,grp,P", SMALL)
def test_small_shapes_match_oracle(seed, kv, grp, P, impl):
    if impl == "fma" and grp > 8:
        pytest.skip("the CUDA-core producer covers G <= 8")
    spec = synthetic.small_spec(500 + seed, kv_dtype=kv, group=grp, page_size=P, ctx_max=330)
    wl = synthetic.make(spec)
    ds = DeviceStep(wl, page_table_stride=wl.max_seq_pages + 2)
    with B.producer(PRODUCERS[impl]):
        ds.step()
    torch.cuda.synchronize()
    _check_flags()
    meta = oracle_metadata(wl)
    assert_attention_close(ds.out, ds.lse, oracle_attention(wl, meta), spec.name)


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 16, 40])
def test_split_count_does_not_change_result(splits):
    """Default (tensor-core) producer."""
    spec = synthetic.Spec("splits", bs=3, num_q_heads=16, num_kv_heads=4, num_pages=40,
                          ragged=(100, 700), num_splits=splits, seed=900)
    wl = synthetic.make(spec)
    ds = DeviceStep(wl)
    ds.step()
    torch.cuda.synchronize()
    meta = oracle_metadata(wl)
    assert_attention_close(ds.out, ds.lse, oracle_attention(wl, meta), f"S={splits}")


@pytest.mark.parametrize("impl", sorted(PRODUCERS))
@pytest.mark.parametrize("kv,P,splits", [("bf16", 64, 1), ("int8", 16, 2), ("bf16", 16, 3),
                                         ("int8", 64, 1)])
def test_splits_longer_than_the_cached_page_list(kv, P, splits, impl):
    """Splits of more than 256 pages (up to 1250): the producers cache 256 page indices
    in shared memory and read the rest from the page table in global memory."""
    spec = synthetic.Spec(f"long{kv}{P}", bs=2, num_q_heads=16, num_kv_heads=2,
                          num_pages=2 * (-(-40000 // P)) + 3, ragged=(20000, 40000),
                          page_size=P, kv_dtype=kv, num_splits=splits, seed=905 + P + splits)
    wl = synthetic.make(spec)
    assert -(-wl.max_seq_pages // splits) > 256
    ds = DeviceStep(wl)
    with B.producer(PRODUCERS[impl]):
        ds.step()
    torch.cuda.synchronize()
    _check_flags()
    meta = oracle_metadata(wl)
    assert_attention_close(ds.out, ds.lse, oracle_attention(wl, meta), spec.name)


@pytest.mark.parametrize("impl", sorted(PRODUCERS))
@pytest.mark.parametrize("q_mult", [3e5, 1e-6])
def test_int8_query_magnitudes_outside_fp16(q_mult, impl):
    """The int8 path feeds Q to fp16 MMAs: queries far above fp16's 65504 or below its
    normal range (2^-14) must still give the oracle's answer (the K scales are set so
    that the scores stay of order one)."""
    spec = synthetic.Spec("qrange", bs=3, num_q_heads=16, num_kv_heads=2, num_pages=30,
                          ragged=(1, 600), kv_dtype="int8", num_splits=3, seed=906)
    wl = synthetic.make(spec)
    wl.q = (wl.q.float() * q_mult).to(torch.bfloat16)
    wl.k_scale = (wl.k_scale.double() / q_mult).float()
    assert wl.q.float().abs().max() > 65504 if q_mult > 1 else wl.q.float().abs().max() < 2 ** -14
    ds = DeviceStep(wl)
    with B.producer(PRODUCERS[impl]):
        ds.step()
    torch.cuda.synchronize()
    _check_flags()
    meta = oracle_metadata(wl)
    assert_attention_close(ds.out, ds.lse, oracle_attention(wl, meta), f"q x {q_mult} {impl}")


def test_empty_and_single_token_requests():
    spec = synthetic.Spec("edge", bs=4, num_q_heads=8, num_kv_heads=2, num_pages=20,
                          ragged=(1, 200), num_splits=3, seed=901)
    wl = synthetic.make(spec)
    # request 0 attends to nothing, request 1 to a single token
    wl.seq_lens[0] = -spec.seqlen_offset
    wl.seq_lens[1] = 1 - spec.seqlen_offset
    wl.ctx[0], wl.ctx[1] = 0, 1
    ds = DeviceStep(wl)
    ds.step()
    torch.cuda.synchronize()
    _check_flags()
    meta = oracle_metadata(wl)
    ref = oracle_attention(wl, meta)
    assert np.all(np.isneginf(ref.lse[0]))
    assert_attention_close(ds.out, ds.lse, ref, "edge")


# ---- exact properties of the CUDA path --------------------------------------------------

def _outputs(ds):
    return [t.clone() for t in (ds.cache_seqlens, ds.cu_seqlens_k, ds.page_table, ds.out, ds.lse)]


@pytest.mark.parametrize("name", ["bs1_ctx8k", "bs64_ragged16k_int8_swa"])
def test_pdl_on_off_bit_identical(name):
    wl, ds = named(name)
    ds.step(use_pdl=True)
    a = _outputs(ds)
    ds.out.zero_()
    ds.step(use_pdl=False)
    b = _outputs(ds)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.uint8) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.uint8) if y.dtype == torch.bfloat16 else y)


@pytest.mark.parametrize("use_pdl", [True, False])
def test_graph_replay_bit_identical_to_eager(use_pdl):
    wl, ds = named("bs8_ctx1k")
    ds.step(use_pdl=use_pdl)
    torch.cuda.synchronize()
    eager = _outputs(ds)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        ds.step(use_pdl=use_pdl)            # warm up on the capture stream
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        ds.step(use_pdl=use_pdl)
    ds.out.zero_()
    ds.lse.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for x, y in zip(eager, _outputs(ds)):
        assert torch.equal(x, y)


@pytest.mark.parametrize("name", ["bs32_ctx8k", "bs64_ragged16k_int8_swa"])
def test_benchmark_launch_configuration_matches_oracle(name):
    """The configuration bench.py times: the full-size workload, the heuristic split
    count, a CUDA graph of 8 consecutive steps with PDL.  After the replays the outputs
    equal one eager step bit for bit, and every request matches the oracle."""
    wl, ds = named(name)
    stream = torch.cuda.Stream()

    def steps():
        for _ in range(8):
            ds.step(use_pdl=True)
    with torch.cuda.stream(stream):
        steps()
    torch.cuda.synchronize()
    eager = _outputs(ds)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        steps()
    ds.out.zero_()
    ds.lse.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    _check_flags()
    for x, y in zip(eager, _outputs(ds)):
        assert torch.equal(x, y)
    meta = oracle_metadata(wl)
    assert_attention_close(ds.out, ds.lse, oracle_attention(wl, meta), name + " graph")


@pytest.mark.parametrize("packed", [False, True])
def test_host_buffer_step_matches_device_step(packed):
    """pa_decode_step_host (separate buffers, one copy per buffer) and
    pa_decode_step_host_packed (one input and one output buffer, one copy each way):
    host inputs copied in, the step, outputs copied back; the outputs equal
    pa_decode_step's bit for bit, on two calls in a row with new inputs."""
    wl, ds = named("bs8_ctx1k")
    for call in range(2):
        q = synthetic.draw_queries(wl.spec.bs, wl.spec.num_q_heads, wl.spec.head_dim, 70 + call)
        ds.out.zero_()
        if packed:
            h_in, h_outs, (h_q, h_rpi, h_sl, h_out, h_lse) = ds.host_buffers()
            h_q.copy_(q)
            h_rpi.copy_(wl.req_pool_indices)
            h_sl.copy_(wl.seq_lens)
            ds.prepare_packed_host_step(h_in, h_outs)()
        else:
            h_q, h_rpi = q.pin_memory(), wl.req_pool_indices.clone().pin_memory()
            h_sl = wl.seq_lens.clone().pin_memory()
            h_out = torch.empty(ds.out.shape, dtype=torch.bfloat16).pin_memory()
            h_lse = torch.empty(ds.lse.shape, dtype=torch.float32).pin_memory()
            ds.prepare_host_step(h_q, h_rpi, h_sl, h_out, h_lse)()
        torch.cuda.synchronize()
        assert torch.equal(ds.q.cpu(), q)
        ds.step()
        torch.cuda.synchronize()
        assert torch.equal(h_out, ds.out.cpu()) and torch.equal(h_lse, ds.lse.cpu())
    ds.q.copy_(wl.q)
    _check_flags()


def test_host_packed_step_in_cuda_graph():
    """pa_decode_step_host_packed captured once into a CUDA graph: every replay copies
    the host inputs as they are at that replay and writes the host outputs, bit for bit
    pa_decode_step's on the same inputs."""
    wl, ds = named("bs8_ctx1k")
    h_in, h_outs, (h_q, h_rpi, h_sl, h_out, h_lse) = ds.host_buffers()
    h_rpi.copy_(wl.req_pool_indices)
    h_sl.copy_(wl.seq_lens)
    stream = torch.cuda.Stream()
    call = ds.prepare_packed_host_step(h_in, h_outs, use_pdl=True, stream=stream)
    h_q.copy_(wl.q)
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    torch.cuda.synchronize()
    for rep in range(2):
        q = synthetic.draw_queries(wl.spec.bs, wl.spec.num_q_heads, wl.spec.head_dim, 90 + rep)
        h_q.copy_(q)
        h_out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(ds.q.cpu(), q)
        ds.step()
        torch.cuda.synchronize()
        assert torch.equal(h_out, ds.out.cpu()) and torch.equal(h_lse, ds.lse.cpu())
    del graph
    ds.q.copy_(wl.q)
    _check_flags()


@pytest.mark.parametrize("name", ["bs8_ctx1k", "bs64_ragged16k_int8_swa"])
def test_host_io_step_matches_device_step(name):
    """pa_decode_step with q, req_pool_indices, seq_lens, out and lse in pinned host
    memory (the kernels read and write them over the host link; no copies), eager and
    from a CUDA graph: bit for bit pa_decode_step's on device buffers."""
    wl, ds = named(name)
    ds.step()
    torch.cuda.synchronize()
    ref_out, ref_lse = ds.out.cpu(), ds.lse.cpu()
    h_in, h_outs, (h_q, h_rpi, h_sl, h_out, h_lse) = ds.host_buffers()
    h_q.copy_(ds.q)
    h_rpi.copy_(ds.req_pool_indices)
    h_sl.copy_(ds.seq_lens)
    stream = torch.cuda.Stream()
    call = ds.prepare_host_io_step(h_in, h_outs, use_pdl=True, stream=stream)
    call()
    stream.synchronize()
    assert torch.equal(h_out, ref_out) and torch.equal(h_lse, ref_lse)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    torch.cuda.synchronize()
    h_out.zero_()
    h_lse.zero_()
    with torch.cuda.stream(stream):
        graph.replay()
    stream.synchronize()
    assert torch.equal(h_out, ref_out) and torch.equal(h_lse, ref_lse)
    del graph
    _check_flags()


def test_page_relabelling_bit_identical_on_gpu():
    spec = synthetic.Spec("relabel", bs=4, num_q_heads=32, num_kv_heads=8, num_pages=80,
                          ragged=(300, 1200), num_splits=5, seed=902)
    wl = synthetic.make(spec)
    ds = DeviceStep(wl)
    ds.step()
    out1, lse1 = ds.out.clone(), ds.lse.clone()
    perm = torch.randperm(spec.num_pages, generator=torch.Generator().manual_seed(1))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(spec.num_pages)
    wl2 = synthetic.make(spec)
    wl2.k_cache = wl.k_cache[perm].contiguous()
    wl2.v_cache = wl.v_cache[perm].contiguous()
    P = spec.page_size
    r2t = wl.req_to_token.clone()
    for i in range(spec.bs):
        n = wl.ctx[i]
        t = r2t[int(wl.req_pool_indices[i]), :n]
        r2t[int(wl.req_pool_indices[i]), :n] = inv[(t // P).long()].to(torch.int32) * P + t % P
    wl2.req_to_token = r2t
    ds2 = DeviceStep(wl2)
    ds2.step()
    torch.cuda.synchronize()
    assert torch.equal(out1, ds2.out) and torch.equal(lse1, ds2.lse)


def test_out_of_range_page_sets_error_flag_without_fault():
    spec = synthetic.Spec("badpage", bs=2, num_q_heads=8, num_kv_heads=2, num_pages=12,
                          ctx=200, num_splits=2, seed=903)
    wl = synthetic.make(spec)
    ds = DeviceStep(wl)
    ds.metadata()
    ds.page_table[1, 2] = spec.num_pages + 5   # a page the pool does not have
    B.pa_read_error_flags(reset=True)
    ds.splitk()
    ds.reduce()
    flags = B.pa_read_error_flags(reset=True)
    assert flags & B.DEVERR_PAGE_OUT_OF_RANGE
    # request 0 is unaffected
    meta = oracle_metadata(wl)
    assert_attention_close(ds.out[:1], ds.lse[:1], oracle_attention(wl, meta, [0]), "request 0")
