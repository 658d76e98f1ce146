"""Seeded random shapes against the oracle: every producer form (decode with either
producer, several query tokens per request, sliding window with -1 holes) over random
KV type, page size, GQA group, batch, lengths, split count and seqlen_offset."""

import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_metadata_gb300 import binding as B
from paged_kv_decode_metadata_gb300 import build, synthetic
from paged_kv_decode_metadata_gb300.runtime import DeviceStep

from helpers import Expected, assert_attention_close, bits, kv_np, oracle_metadata, \
    paged_attention_threaded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    B.load()
    B.pa_read_error_flags(reset=True)
    yield
    assert B.pa_read_error_flags(reset=True) == 0


def _draw(seed):
    g = torch.Generator().manual_seed(50_000 + seed)
    pick = lambda xs: xs[int(torch.randint(0, len(xs), (1,), generator=g))]  # noqa: E731
    kv = pick(["bf16", "int8"])
    P = pick([16, 32, 64, 128])
    grp = pick([1, 2, 4, 8, 16])
    hkv = pick([1, 2])
    bs = int(torch.randint(1, 7, (1,), generator=g))
    ctx_max = pick([40, 300, 1500])
    splits = int(torch.randint(1, 13, (1,), generator=g))
    mode = pick(["decode", "multi", "window"])
    spec = synthetic.Spec(f"fuzz{seed}", bs=bs, num_q_heads=grp * hkv, num_kv_heads=hkv,
                          num_pages=bs * (-(-ctx_max // P)) + 2, ragged=(1, ctx_max), page_size=P,
                          kv_dtype=kv, num_splits=splits,
                          seqlen_offset=int(torch.randint(0, 2, (1,), generator=g)),
                          swa_window=int(torch.randint(1, 2 * ctx_max, (1,), generator=g))
                          if mode == "window" else None,
                          seed=60_000 + seed)
    max_q = max(1, 16 // grp) if mode == "multi" else 1
    if mode == "multi":
        max_q = int(torch.randint(1, max_q + 1, (1,), generator=g))
    return spec, mode, max_q, g


def _run_window(wl, meta, g, splits):
    table = meta["swa_page_table"].copy()
    for b in range(wl.spec.bs):                       # a -1 hole in about half the requests
        mapped = sorted(wl.swa_pages[b])
        if mapped and bool(torch.rand(1, generator=g) < 0.5):
            table[b, mapped[int(torch.randint(0, len(mapped), (1,), generator=g))]] = -1
    dev = "cuda"
    hq, d = wl.spec.num_q_heads, wl.spec.head_dim
    f32 = dict(dtype=torch.float32, device=dev)
    m = torch.empty((wl.spec.bs, hq, splits), **f32)
    l, acc = torch.empty_like(m), torch.empty((wl.spec.bs, hq, splits, d), **f32)
    out = torch.empty((wl.spec.bs, hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.spec.bs, hq), **f32)
    sc = (lambda t: t.to(dev) if t is not None else None)
    B.pa_decode_splitk_window(wl.q.to(dev), wl.k_swa.to(dev), wl.v_swa.to(dev),
                              torch.from_numpy(table).to(dev),
                              torch.from_numpy(meta["cache_seqlens"]).to(dev), m, l, acc,
                              sliding_window=wl.spec.swa_window, max_seq_pages=wl.max_seq_pages,
                              num_splits=splits, sm_scale=wl.sm_scale,
                              k_scale=sc(wl.k_swa_scale), v_scale=sc(wl.v_swa_scale))
    B.pa_reduce(m, l, acc, out, lse)
    torch.cuda.synchronize()
    if wl.spec.kv_dtype == "int8":
        k, v = wl.k_swa.numpy(), wl.v_swa.numpy()
        ks, vs = wl.k_swa_scale.numpy(), wl.v_swa_scale.numpy()
    else:
        k, v, ks, vs = bits(wl.k_swa), bits(wl.v_swa), None, None
    ref = Expected(oracle.paged_attention_window, bits(wl.q), k, v, table,
                   meta["cache_seqlens"], wl.spec.swa_window, wl.sm_scale, None, ks, vs)
    return (out, lse), ref


def _run_multi(wl, meta, max_q, g, splits):
    qlens = synthetic.draw_query_lengths(wl.spec.bs, max_q, int(torch.randint(0, 1 << 30, (1,), generator=g)))
    cu_q = oracle.cu_seqlens_q(qlens.numpy(), wl.spec.bs, 1)
    q = synthetic.draw_queries(int(cu_q[-1]), wl.spec.num_q_heads, wl.spec.head_dim,
                               int(torch.randint(0, 1 << 30, (1,), generator=g)))
    dev = "cuda"
    rows, hq, d = q.shape
    f32 = dict(dtype=torch.float32, device=dev)
    m = torch.empty((rows, hq, splits), **f32)
    l, acc = torch.empty_like(m), torch.empty((rows, hq, splits, d), **f32)
    out = torch.empty((rows, hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((rows, hq), **f32)
    sc = (lambda t: t.to(dev) if t is not None else None)
    B.pa_decode_splitk_multi(q.to(dev), wl.k_cache.to(dev), wl.v_cache.to(dev),
                             torch.from_numpy(meta["page_table"]).to(dev),
                             torch.from_numpy(meta["cache_seqlens"]).to(dev),
                             torch.from_numpy(cu_q).to(dev), m, l, acc, max_q_len=max_q,
                             max_seq_pages=wl.max_seq_pages, num_splits=splits,
                             sm_scale=wl.sm_scale, k_scale=sc(wl.k_scale), v_scale=sc(wl.v_scale))
    B.pa_reduce(m, l, acc, out, lse)
    torch.cuda.synchronize()
    k, v, ks, vs = kv_np(wl)
    ref = Expected(oracle.paged_attention_multi, bits(q), k, v, meta["page_table"],
                   meta["cache_seqlens"], cu_q, wl.sm_scale, ks, vs)
    return (out, lse), ref


# 36 seeds by default; PA_FUZZ_SEEDS=n draws n (a longer sweep of the same generator)
@pytest.mark.parametrize("seed", range(int(os.environ.get("PA_FUZZ_SEEDS", "36"))))
def test_random_shapes_match_oracle(seed):
    spec, mode, max_q, g = _draw(seed)
    wl = synthetic.make(spec, with_cache=mode != "window", with_swa_cache=mode == "window")
    meta = oracle_metadata(wl)
    splits = spec.num_splits
    if mode == "window":
        got, ref = _run_window(wl, meta, g, splits)
    elif mode == "multi":
        got, ref = _run_multi(wl, meta, max_q, g, splits)
    else:
        impl = B.PA_PRODUCER_FMA if (seed % 2 and spec.num_q_heads // spec.num_kv_heads <= 8) \
            else B.PA_PRODUCER_MMA
        ds = DeviceStep(wl)
        with B.producer(impl):
            ds.step()
        torch.cuda.synchronize()
        k, v, ks, vs = kv_np(wl)
        ref = Expected(oracle.paged_attention, bits(wl.q), k, v, meta["page_table"],
                       meta["cache_seqlens"], wl.sm_scale, ks, vs)
        got = (ds.out, ds.lse)
    assert_attention_close(got[0], got[1], ref, f"{spec.name} {mode}")
    assert B.pa_read_error_flags(reset=True) == 0


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_large_batch_all_rows(kv):
    """1024 requests (grid depth 1024, four scan tiles in the metadata kernel) with short
    ragged lengths: metadata bit-exact, every request against the oracle."""
    spec = synthetic.Spec(f"bs1024{kv}", bs=1024, num_q_heads=32, num_kv_heads=8,
                          num_pages=1024 * 5 + 2, ragged=(1, 300), kv_dtype=kv, seed=70_001)
    wl = synthetic.make(spec)
    ds = DeviceStep(wl)
    ds.step()
    torch.cuda.synchronize()
    meta = oracle_metadata(wl)
    assert np.array_equal(ds.cache_seqlens.cpu().numpy(), meta["cache_seqlens"])
    assert np.array_equal(ds.cu_seqlens_k.cpu().numpy(), meta["cu_seqlens_k"])
    assert np.array_equal(ds.page_table.cpu().numpy(), meta["page_table"])
    k, v, ks, vs = kv_np(wl)
    ref = Expected(paged_attention_threaded, bits(wl.q), k, v, meta["page_table"],
                   meta["cache_seqlens"], wl.sm_scale, ks, vs)
    assert_attention_close(ds.out, ds.lse, ref, spec.name)
