"""GPU parity of the multi-token-query producer (several query tokens per request,
causal within the request's newest tokens) against the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_metadata_gb300 import binding as B
from paged_kv_decode_metadata_gb300 import build, synthetic
from paged_kv_decode_metadata_gb300.runtime import DeviceStep

from helpers import Expected, assert_attention_close, bits, kv_np, oracle_metadata

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    B.load()
    B.pa_read_error_flags(reset=True)
    yield
    assert B.pa_read_error_flags(reset=True) == 0


def _run_multi(wl, qlens, q, num_splits, use_pdl=True, host_io=False):
    """GPU: metadata (with cu_seqlens_q from qlens), multi-query producer, reducer.
    host_io: q, out and lse in pinned host memory (the kernels read and write them over
    the host link)."""
    dev = "cuda"
    spec = wl.spec
    i32 = dict(dtype=torch.int32, device=dev)
    bs, msp = spec.bs, wl.max_seq_pages
    cl, cu = torch.empty(bs, **i32), torch.empty(bs + 1, **i32)
    cq, pt = torch.empty(bs + 1, **i32), torch.empty((bs, msp), **i32)
    B.pa_build_metadata_full(wl.req_pool_indices.to(dev), wl.seq_lens.to(dev),
                             wl.req_to_token.to(dev), cl, cu, pt,
                             seqlen_offset=spec.seqlen_offset, max_seq_pages=msp,
                             page_size=spec.page_size, cu_seqlens_q=cq, qlens=qlens.to(dev),
                             q_mode=B.PA_Q_MODE_CUMSUM, use_pdl=use_pdl)
    total_q, hq, d = q.shape
    f32 = dict(dtype=torch.float32, device=dev)
    m = torch.empty((total_q, hq, num_splits), **f32)
    l = torch.empty((total_q, hq, num_splits), **f32)
    acc = torch.empty((total_q, hq, num_splits, d), **f32)
    if host_io:
        out = torch.empty((total_q, hq, d), dtype=torch.bfloat16).pin_memory()
        lse = torch.empty((total_q, hq), dtype=torch.float32).pin_memory()
        q_in = q.contiguous().pin_memory()
    else:
        out = torch.empty((total_q, hq, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((total_q, hq), **f32)
        q_in = q.to(dev)
    k = wl.k_cache.to(dev)
    v = wl.v_cache.to(dev)
    ks = wl.k_scale.to(dev) if wl.k_scale is not None else None
    vs = wl.v_scale.to(dev) if wl.v_scale is not None else None
    B.pa_decode_splitk_multi(q_in, k, v, pt, cl, cq, m, l, acc,
                             max_q_len=int(qlens.max()), max_seq_pages=msp,
                             num_splits=num_splits, sm_scale=wl.sm_scale, k_scale=ks, v_scale=vs,
                             use_pdl=use_pdl)
    B.pa_reduce(m, l, acc, out, lse, use_pdl=use_pdl)
    torch.cuda.synchronize()
    assert np.array_equal(cq.cpu().numpy(), oracle.cu_seqlens_q(qlens.numpy(), bs, 1))
    return out, lse


def _oracle_multi(wl, qlens, q):
    meta = oracle_metadata(wl)
    k, v, ks, vs = kv_np(wl)
    cu_q = oracle.cu_seqlens_q(qlens.numpy(), wl.spec.bs, 1)
    return Expected(oracle.paged_attention_multi, bits(q), k, v, meta["page_table"],
                    meta["cache_seqlens"], cu_q, wl.sm_scale, ks, vs)


CASES = [  # seed, kv, group, max_q_len, page_size, splits
    (1, "bf16", 4, 4, 64, 3), (2, "bf16", 8, 2, 64, 4), (3, "int8", 8, 2, 64, 3),
    (4, "int8", 4, 4, 16, 5), (5, "bf16", 1, 16, 128, 2), (6, "bf16", 2, 8, 32, 7),
    (7, "int8", 16, 1, 64, 3), (8, "int8", 2, 5, 128, 1),
]


@pytest.mark.parametrize("seed,kv,grp,max_q,P,splits", CASES)
def test_multi_query_matches_oracle(seed, kv, grp, max_q, P, splits):
    spec = synthetic.Spec(f"mq{seed}", bs=4, num_q_heads=2 * grp, num_kv_heads=2,
                          num_pages=4 * (-(-700 // P)) + 2, ragged=(1, 700), page_size=P,
                          kv_dtype=kv, num_splits=splits, seqlen_offset=seed % 2, seed=700 + seed)
    wl = synthetic.make(spec)
    qlens = synthetic.draw_query_lengths(spec.bs, max_q, 800 + seed)
    q = synthetic.draw_queries(int(qlens.sum()), spec.num_q_heads, spec.head_dim, 900 + seed)
    out, lse = _run_multi(wl, qlens, q, splits)
    assert_attention_close(out, lse, _oracle_multi(wl, qlens, q), spec.name)


def test_queries_beyond_the_context_are_empty():
    spec = synthetic.Spec("short", bs=3, num_q_heads=8, num_kv_heads=2, num_pages=6,
                          ragged=(1, 5), num_splits=2, seed=31)
    wl = synthetic.make(spec)
    qlens = torch.tensor([4, 4, 4], dtype=torch.int64)   # more queries than cached tokens
    q = synthetic.draw_queries(12, 8, 128, 32)
    out, lse = _run_multi(wl, qlens, q, 2)
    ref = _oracle_multi(wl, qlens, q)
    assert np.isneginf(ref.lse).any()
    assert_attention_close(out, lse, ref, "short")


def test_one_query_per_request_equals_decode_bit_for_bit():
    wl = synthetic.make(synthetic.WORKLOADS["bs8_ctx1k"])
    ds = DeviceStep(wl)
    ds.step()
    qlens = torch.ones(wl.spec.bs, dtype=torch.int64)
    out, lse = _run_multi(wl, qlens, wl.q, ds.num_splits)
    assert torch.equal(out, ds.out) and torch.equal(lse, ds.lse)


def test_multi_query_pdl_on_off_identical():
    spec = synthetic.Spec("mqpdl", bs=6, num_q_heads=16, num_kv_heads=4, num_pages=80,
                          ragged=(200, 800), num_splits=4, seed=41)
    wl = synthetic.make(spec)
    qlens = synthetic.draw_query_lengths(spec.bs, 4, 42)
    q = synthetic.draw_queries(int(qlens.sum()), 16, 128, 43)
    a = _run_multi(wl, qlens, q, 4, use_pdl=True)
    b = _run_multi(wl, qlens, q, 4, use_pdl=False)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_multi_query_unsupported_shapes(lib):
    wl = synthetic.make(synthetic.small_spec(3, group=8))
    qlens = torch.full((wl.spec.bs,), 3, dtype=torch.int64)  # 8 heads x 3 queries > 16 columns
    q = synthetic.draw_queries(int(qlens.sum()), wl.spec.num_q_heads, 128, 4)
    with pytest.raises(B.PAError) as e:
        _run_multi(wl, qlens, q, 2)
    assert e.value.status == B.PA_ERR_UNSUPPORTED


@pytest.mark.parametrize("q_mode", ["cumsum", "strided", "preset"])
def test_multi_step_one_call_matches_stages(q_mode):
    """pa_decode_step_multi (metadata with cu_seqlens_q, multi-query producer, reducer)
    equals the three calls made one by one, bit for bit, and the oracle."""
    spec = synthetic.Spec("mqstep", bs=5, num_q_heads=16, num_kv_heads=4, num_pages=120,
                          ragged=(1, 900), num_splits=3, seqlen_offset=1, seed=51)
    wl = synthetic.make(spec)
    dev = "cuda"
    if q_mode == "strided":
        qlens = torch.full((spec.bs,), 3, dtype=torch.int64)
    else:
        qlens = synthetic.draw_query_lengths(spec.bs, 4, 52)
    q = synthetic.draw_queries(int(qlens.sum()), spec.num_q_heads, spec.head_dim, 53)
    out_ref, lse_ref = _run_multi(wl, qlens, q, 3)
    i32 = dict(dtype=torch.int32, device=dev)
    bs, msp = spec.bs, wl.max_seq_pages
    cl, cu, pt = torch.empty(bs, **i32), torch.empty(bs + 1, **i32), torch.empty((bs, msp), **i32)
    cq = torch.empty(bs + 1, **i32)
    if q_mode == "preset":
        cq.copy_(torch.from_numpy(oracle.cu_seqlens_q(qlens.numpy(), bs, 1)))
    total_q, hq, d = q.shape
    ws = torch.empty(B.pa_workspace_bytes(total_q, hq, d, 3), dtype=torch.uint8, device=dev)
    out = torch.empty((total_q, hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((total_q, hq), dtype=torch.float32, device=dev)
    mode = {"cumsum": B.PA_Q_MODE_CUMSUM, "strided": B.PA_Q_MODE_STRIDED,
            "preset": B.PA_Q_MODE_NONE}[q_mode]
    B.pa_decode_step_multi(req_pool_indices=wl.req_pool_indices.to(dev),
                           seq_lens=wl.seq_lens.to(dev), req_to_token=wl.req_to_token.to(dev),
                           seqlen_offset=spec.seqlen_offset, max_seq_pages=msp, cache_seqlens=cl,
                           cu_seqlens_k=cu, page_table=pt, cu_seqlens_q=cq, q=q.to(dev),
                           max_q_len=int(qlens.max()), k_cache=wl.k_cache.to(dev),
                           v_cache=wl.v_cache.to(dev), num_splits=3, sm_scale=wl.sm_scale,
                           workspace=ws, out=out, lse=lse,
                           qlens=qlens.to(dev) if q_mode == "cumsum" else None, q_mode=mode,
                           q_stride=3)
    torch.cuda.synchronize()
    assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref)
    assert_attention_close(out, lse, _oracle_multi(wl, qlens, q), f"step multi {q_mode}")


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_multi_query_host_io_bit_identical(kv):
    """q, out and lse in pinned host memory: the same bits as device buffers."""
    spec = synthetic.Spec(f"mq_host_{kv}", bs=5, num_q_heads=16, num_kv_heads=4, num_pages=5 * 16,
                          ragged=(200, 900), kv_dtype=kv, num_splits=3, seed=61)
    wl = synthetic.make(spec)
    qlens = synthetic.draw_query_lengths(spec.bs, 3, 62)
    q = synthetic.draw_queries(int(qlens.sum()), spec.num_q_heads, spec.head_dim, 63)
    a = _run_multi(wl, qlens, q, 3)
    b = _run_multi(wl, qlens, q, 3, host_io=True)
    assert torch.equal(a[0].cpu().view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].cpu(), b[1])
