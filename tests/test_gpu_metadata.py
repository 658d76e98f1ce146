"""GPU parity of the fused metadata stage against the oracle: bit-exact."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_metadata_gb300 import binding as B
from paged_kv_decode_metadata_gb300 import build, synthetic

from helpers import oracle_metadata

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    B.load()
    B.pa_read_error_flags(reset=True)
    yield
    assert B.pa_read_error_flags(reset=True) == 0


def _run(wl, stride_pad=0, use_pdl=True, with_swa=True, canary=-777):
    dev = "cuda"
    bs, msp = wl.spec.bs, wl.max_seq_pages
    pts = msp + stride_pad
    i32 = dict(dtype=torch.int32, device=dev)
    cache_seqlens = torch.full((bs,), canary, **i32)
    cu = torch.full((bs + 1,), canary, **i32)
    pt = torch.full((bs, pts), canary, **i32)
    mapping = wl.full_to_swa_mapping if with_swa else None
    swa = torch.full((bs, pts), canary, **i32) if mapping is not None else None
    B.pa_build_metadata(wl.req_pool_indices.to(dev), wl.seq_lens.to(dev), wl.req_to_token.to(dev),
                        cache_seqlens, cu, pt, seqlen_offset=wl.spec.seqlen_offset,
                        max_seq_pages=msp, page_size=wl.spec.page_size,
                        full_to_swa_mapping=None if mapping is None else mapping.to(dev),
                        swa_page_table=swa, use_pdl=use_pdl)
    torch.cuda.synchronize()
    out = {"cache_seqlens": cache_seqlens.cpu().numpy(), "cu_seqlens_k": cu.cpu().numpy(),
           "page_table": pt.cpu().numpy()}
    if swa is not None:
        out["swa_page_table"] = swa.cpu().numpy()
    return out


def _compare(got, want, msp):
    for key in want:
        g = got[key][:, :msp] if got[key].ndim == 2 else got[key]
        assert np.array_equal(g, want[key]), key


@pytest.mark.parametrize("name", synthetic.WORKLOAD_ORDER)
def test_metadata_bit_exact_on_workloads(name):
    wl = synthetic.make(synthetic.WORKLOADS[name], with_cache=False)
    got = _run(wl)
    _compare(got, oracle_metadata(wl), wl.max_seq_pages)


@pytest.mark.parametrize("seed", range(6))
def test_metadata_bit_exact_small_and_padded(seed):
    wl = synthetic.make(synthetic.small_spec(100 + seed), with_cache=False)
    got = _run(wl, stride_pad=5)
    _compare(got, oracle_metadata(wl), wl.max_seq_pages)
    assert np.all(got["page_table"][:, wl.max_seq_pages:] == -777)   # untouched columns


def test_metadata_swa_small_windows():
    for seed in range(3):
        spec = synthetic.Spec(f"swa{seed}", bs=5, num_q_heads=8, num_kv_heads=8, num_pages=60,
                              ragged=(1, 700), swa_window=100 + 37 * seed, seed=300 + seed)
        wl = synthetic.make(spec, with_cache=False)
        _compare(_run(wl, stride_pad=3), oracle_metadata(wl), wl.max_seq_pages)


def test_metadata_hand_example_and_full_surface():
    fx = json.load(open(os.path.join(GOLDEN, "metadata_hand_example.json")))
    dev = "cuda"
    i32 = dict(dtype=torch.int32, device=dev)
    rpi = torch.tensor(fx["req_pool_indices"], dtype=torch.int64, device=dev)
    sl = torch.tensor(fx["seq_lens"], dtype=torch.int64, device=dev)
    r2t = torch.tensor(fx["req_to_token"], dtype=torch.int32, device=dev)
    mapping = torch.tensor(fx["full_to_swa_mapping"], dtype=torch.int64, device=dev)
    cl, cu = torch.full((2,), 9, **i32), torch.full((3,), 9, **i32)
    pt, swa = torch.full((2, 3), 9, **i32), torch.full((2, 3), 9, **i32)
    cq = torch.full((3,), 9, **i32)
    B.pa_build_metadata_full(rpi, sl, r2t, cl, cu, pt, seqlen_offset=fx["seqlen_offset"],
                             max_seq_pages=fx["max_seq_pages"], page_size=fx["page_size"],
                             full_to_swa_mapping=mapping, swa_page_table=swa)
    torch.cuda.synchronize()
    e = fx["expected"]
    assert cl.tolist() == e["cache_seqlens"] and cu.tolist() == e["cu_seqlens_k"]
    assert pt.tolist() == e["page_table"] and swa.tolist() == e["swa_page_table"]
    # cu_seqlens_q modes and swa_out_cache_loc (bs 3 over the same table)
    rpi3 = torch.tensor([0, 1, 2], dtype=torch.int64, device=dev)
    sl3 = torch.tensor([1, 2, 3], dtype=torch.int64, device=dev)
    cl3, cu3, pt3 = torch.empty(3, **i32), torch.empty(4, **i32), torch.empty((3, 3), **i32)
    swa3 = torch.empty((3, 3), **i32)
    cq = torch.full((4,), 9, **i32)
    qc = fx["cu_seqlens_q"]
    so = fx["swa_out_cache_loc"]
    loc = torch.tensor(so["out_cache_loc"], dtype=torch.int64, device=dev)
    swa_out = torch.full((so["swa_out_len"],), 99, dtype=torch.int64, device=dev)
    B.pa_build_metadata_full(rpi3, sl3, r2t, cl3, cu3, pt3, seqlen_offset=0, max_seq_pages=3,
                             page_size=4, full_to_swa_mapping=mapping, swa_page_table=swa3,
                             cu_seqlens_q=cq, qlens=torch.tensor(qc["qlens"], dtype=torch.int64, device=dev),
                             q_mode=B.PA_Q_MODE_CUMSUM, out_cache_loc=loc, swa_out_cache_loc=swa_out)
    torch.cuda.synchronize()
    assert cq.tolist() == qc["cumsum"]
    assert swa_out.tolist() == so["expected"]
    B.pa_build_metadata_full(rpi3, sl3, r2t, cl3, cu3, pt3, seqlen_offset=0, max_seq_pages=3,
                             page_size=4, cu_seqlens_q=cq, q_mode=B.PA_Q_MODE_STRIDED,
                             q_stride=qc["q_stride"])
    torch.cuda.synchronize()
    assert cq.tolist() == qc["strided"]


@pytest.mark.parametrize("idx", [torch.int64, torch.int32])
def test_metadata_full_surface_against_oracle(idx):
    """Large batch (several scan tiles), random qlens, long swa_out_cache_loc; index
    inputs as int64 and as int32 (the module's kernel takes either)."""
    g = torch.Generator().manual_seed(77)
    spec = synthetic.Spec("scan", bs=700, num_q_heads=8, num_kv_heads=8, num_pages=12000,
                          ragged=(0, 900), swa_window=200, seqlen_offset=1, seed=78)
    wl = synthetic.make(spec, with_cache=False)
    dev = "cuda"
    qlens = torch.randint(0, 9, (spec.bs,), generator=g, dtype=torch.int64)
    full = wl.full_to_swa_mapping
    loc = torch.randint(-3, full.numel(), (1500,), generator=g, dtype=torch.int64)
    i32 = dict(dtype=torch.int32, device=dev)
    msp = wl.max_seq_pages
    cl, cu, cq = torch.empty(spec.bs, **i32), torch.empty(spec.bs + 1, **i32), torch.empty(spec.bs + 1, **i32)
    pt, swa = torch.empty((spec.bs, msp), **i32), torch.empty((spec.bs, msp), **i32)
    swa_out = torch.full((1700,), 5, dtype=torch.int64, device=dev)
    B.pa_build_metadata_full(wl.req_pool_indices.to(dev, idx), wl.seq_lens.to(dev, idx),
                             wl.req_to_token.to(dev), cl, cu, pt, seqlen_offset=1,
                             max_seq_pages=msp, page_size=64, full_to_swa_mapping=full.to(dev),
                             swa_page_table=swa, cu_seqlens_q=cq, qlens=qlens.to(dev, idx),
                             q_mode=B.PA_Q_MODE_CUMSUM, out_cache_loc=loc.to(dev),
                             swa_out_cache_loc=swa_out)
    torch.cuda.synchronize()
    want = oracle_metadata(wl)
    _compare({"cache_seqlens": cl.cpu().numpy(), "cu_seqlens_k": cu.cpu().numpy(),
              "page_table": pt.cpu().numpy(), "swa_page_table": swa.cpu().numpy()}, want, msp)
    assert np.array_equal(cq.cpu().numpy(), oracle.cu_seqlens_q(qlens.numpy(), spec.bs, 1))
    assert np.array_equal(swa_out.cpu().numpy(), oracle.swa_out_cache_loc(loc.numpy(), full.numpy(), 1700))


def test_metadata_pdl_on_off_identical():
    wl = synthetic.make(synthetic.WORKLOADS["bs64_ragged16k_int8_swa"], with_cache=False)
    a, b = _run(wl, use_pdl=True), _run(wl, use_pdl=False)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_metadata_out_of_range_row_sets_error_flag():
    wl = synthetic.make(synthetic.small_spec(5), with_cache=False)
    wl.req_pool_indices[0] = wl.req_to_token.shape[0] + 3     # outside the table
    B.pa_read_error_flags(reset=True)
    _run(wl)
    assert B.pa_read_error_flags(reset=True) & B.DEVERR_POOL_ROW_OUT_OF_RANGE


def test_empty_batch_is_a_no_op():
    i32 = dict(dtype=torch.int32, device="cuda")
    e64 = torch.empty(0, dtype=torch.int64, device="cuda")
    B.pa_build_metadata(e64, e64, torch.zeros((1, 64), **i32), torch.empty(0, **i32),
                        torch.full((1,), 3, **i32), torch.empty((0, 1), **i32), seqlen_offset=0,
                        max_seq_pages=1, page_size=64)
    torch.cuda.synchronize()


def test_metadata_long_rows_and_many_requests():
    """Rows longer than the 1024 columns a row block reads before its PDL wait (the
    rest is read after it) and more requests than one 256-wide scan tile (later tiles
    of lengths are read after the wait): still bit-exact, sliding-window table too."""
    spec = synthetic.Spec("long_rows", bs=300, num_q_heads=8, num_kv_heads=8,
                          num_pages=400000, ragged=(1, 20000), page_size=16,
                          swa_window=5000, seqlen_offset=1, seed=404)
    wl = synthetic.make(spec, with_cache=False)
    assert wl.max_seq_pages > 1024
    for use_pdl in (True, False):
        _compare(_run(wl, stride_pad=2, use_pdl=use_pdl), oracle_metadata(wl), wl.max_seq_pages)
