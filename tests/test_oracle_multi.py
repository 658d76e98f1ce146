"""Pins for the multi-token-query oracle (several query tokens per request, causal
within the request's newest tokens).

* one query per request reduces exactly to the decode oracle;
* each query row equals the decode oracle over the request cut to the tokens that
  query may see (n - q_len + i + 1), and torch's scaled_dot_product_attention in
  float64 with the causal-offset mask;
* planted mistakes in the causal limit or the query row are caught.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_metadata_gb300 import synthetic

from test_oracle_pins import _bits, _dense_kv, _kv_np, _oracle_metadata, plant_source


def _case(seed, kv="bf16", max_q_len=4):
    spec = synthetic.Spec(f"mq{seed}", bs=3, num_q_heads=8, num_kv_heads=2, num_pages=24,
                          ragged=(1, 400), kv_dtype=kv, num_splits=3, seed=seed)
    wl = synthetic.make(spec)
    qlens = synthetic.draw_query_lengths(spec.bs, max_q_len, seed + 1)
    cu_q = oracle.cu_seqlens_q(qlens.numpy(), spec.bs, 1)
    q = synthetic.draw_queries(int(cu_q[-1]), spec.num_q_heads, spec.head_dim, seed + 2)
    return wl, q, cu_q


def _multi(wl, q, cu_q, lib=None):
    meta = _oracle_metadata(wl, lib)
    k, v, ks, vs = _kv_np(wl)
    return oracle.paged_attention_multi(_bits(q), k, v, meta["page_table"],
                                        meta["cache_seqlens"], cu_q, wl.sm_scale, ks, vs,
                                        lib=lib), meta


def check_single_query_is_decode(lib=None):
    wl, _, _ = _case(5)
    cu_q = np.arange(wl.spec.bs + 1, dtype=np.int32)
    (out, lse), meta = _multi(wl, wl.q, cu_q, lib)
    k, v, ks, vs = _kv_np(wl)
    out1, lse1 = oracle.paged_attention(_bits(wl.q), k, v, meta["page_table"],
                                        meta["cache_seqlens"], wl.sm_scale, ks, vs, lib=lib)
    assert np.array_equal(out, out1) and np.array_equal(lse, lse1)


def check_rows_are_prefix_decodes(seed, kv="bf16", lib=None):
    wl, q, cu_q = _case(seed, kv)
    (out, lse), meta = _multi(wl, q, cu_q, lib)
    k, v, ks, vs = _kv_np(wl)
    for b in range(wl.spec.bs):
        q_len = cu_q[b + 1] - cu_q[b]
        for i in range(q_len):
            r = cu_q[b] + i
            limit = max(0, int(meta["cache_seqlens"][b]) - q_len + i + 1)
            o1, l1 = oracle.paged_attention(_bits(q[r:r + 1]), k, v, meta["page_table"][b:b + 1],
                                            np.array([limit], np.int32), wl.sm_scale, ks, vs,
                                            lib=lib)
            np.testing.assert_array_equal(out[r], o1[0])
            np.testing.assert_array_equal(lse[r], l1[0])


def check_against_torch_sdpa(seed, kv="bf16", lib=None):
    wl, q, cu_q = _case(seed, kv)
    (out, lse), _ = _multi(wl, q, cu_q, lib)
    g = wl.spec.num_q_heads // wl.spec.num_kv_heads
    for b in range(wl.spec.bs):
        kd, vd = _dense_kv(wl, b)                       # [Hkv, n, d]
        n = kd.shape[1]
        rows = q[cu_q[b]:cu_q[b + 1]].to(torch.float64)  # [q_len, Hq, d]
        q_len = rows.shape[0]
        pos = torch.arange(n)
        mask = pos[None, :] < (n - q_len + torch.arange(q_len) + 1)[:, None]   # [q_len, n]
        ref = torch.nn.functional.scaled_dot_product_attention(
            rows.permute(1, 0, 2)[None], kd[None], vd[None], attn_mask=mask[None, None],
            scale=wl.sm_scale, enable_gqa=True)[0].permute(1, 0, 2)
        scores = torch.einsum("qhd,hnd->qhn", rows, kd.repeat_interleave(g, dim=0)) * wl.sm_scale
        ref_lse = torch.logsumexp(scores.masked_fill(~mask[:, None, :], float("-inf")), dim=-1)
        np.testing.assert_allclose(out[cu_q[b]:cu_q[b + 1]], ref.numpy(), rtol=0, atol=1e-10)
        np.testing.assert_allclose(lse[cu_q[b]:cu_q[b + 1]], ref_lse.numpy(), rtol=0, atol=1e-10)


def test_single_query_is_decode():
    check_single_query_is_decode()


@pytest.mark.parametrize("seed,kv", [(11, "bf16"), (12, "int8"), (13, "bf16")])
def test_rows_are_prefix_decodes(seed, kv):
    check_rows_are_prefix_decodes(seed, kv)


@pytest.mark.parametrize("seed,kv", [(21, "bf16"), (22, "int8")])
def test_against_torch_sdpa(seed, kv):
    check_against_torch_sdpa(seed, kv)


def test_queries_longer_than_context_are_empty():
    spec = synthetic.Spec("short", bs=1, num_q_heads=2, num_kv_heads=1, num_pages=2, ctx=3,
                          num_splits=1, seed=3)
    wl = synthetic.make(spec)
    cu_q = np.array([0, 5], np.int32)                  # 5 queries, 3 cached tokens
    q = synthetic.draw_queries(5, 2, 128, 4)
    (out, lse), _ = _multi(wl, q, cu_q)
    assert np.all(np.isneginf(lse[:2])) and np.all(out[:2] == 0)
    assert np.all(np.isfinite(lse[2:]))


MULTI_PLANTS = {
    "causal_limit_off_by_one": ("static_cast<int64_t>(cache_seqlens[b]) - q_len + i + 1;",
                                "static_cast<int64_t>(cache_seqlens[b]) - q_len + i;"),
    "query_row_of_first_token": ("const int64_t row = q_begin + i;", "const int64_t row = q_begin;"),
    "no_causal_mask": ("static_cast<int64_t>(cache_seqlens[b]) - q_len + i + 1;",
                       "static_cast<int64_t>(cache_seqlens[b]);"),
}


@pytest.mark.parametrize("plant", sorted(MULTI_PLANTS))
def test_multi_plants_are_caught(plant, tmp_path):
    before, after = MULTI_PLANTS[plant]
    src = open(oracle._SRC).read()
    path = tmp_path / f"{plant}.cpp"
    path.write_text(plant_source(src, before, after, "oracle_paged_attention_multi"))
    lib = oracle.load(oracle.build(str(path), str(tmp_path / f"lib{plant}.so")))
    with pytest.raises(AssertionError):
        check_single_query_is_decode(lib)
        check_rows_are_prefix_decodes(11, lib=lib)
        check_against_torch_sdpa(21, lib=lib)
