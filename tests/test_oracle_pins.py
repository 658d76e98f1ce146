"""Pins for the CPU oracle: it is checked against things other than itself.

* hand-worked metadata and attention examples (tests/golden/, each with its citation);
* the generator's own record of which pages a request owns and which pages the
  sliding window covers (not the metadata formula);
* torch's scaled_dot_product_attention and logsumexp in float64 on densely gathered
  K/V (a library routine standing in for brute force);
* closed forms (one token; identical keys);
* invariants (split count, page relabelling, request order, empty contexts).

``test_planted_mistakes_are_caught`` compiles modified copies of the oracle, each
with one plausible mistake, and checks that these pins reject every one.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_metadata_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _kv_np(wl):
    if wl.spec.kv_dtype == "int8":
        return (wl.k_cache.numpy(), wl.v_cache.numpy(), wl.k_scale.numpy(), wl.v_scale.numpy())
    return _bits(wl.k_cache), _bits(wl.v_cache), None, None


def _oracle_metadata(wl, lib=None):
    m = wl.full_to_swa_mapping
    return oracle.build_metadata(wl.req_pool_indices.numpy(), wl.seq_lens.numpy(),
                                 wl.req_to_token.numpy(), wl.spec.seqlen_offset,
                                 wl.max_seq_pages, wl.spec.page_size,
                                 None if m is None else m.numpy(), lib=lib)


def _oracle_attention(wl, meta, lib=None):
    k, v, ks, vs = _kv_np(wl)
    return oracle.paged_attention(_bits(wl.q), k, v, meta["page_table"],
                                  meta["cache_seqlens"], wl.sm_scale, ks, vs, lib=lib)


def _dense_kv(wl, b):
    """K/V of request b gathered through the generator's page list, float64."""
    P = wl.spec.page_size
    n = wl.ctx[b]
    pages = torch.tensor([wl.pages[b][j // P] for j in range(n)], dtype=torch.long)
    offs = torch.arange(n) % P
    k = wl.k_cache[pages, :, offs, :].to(torch.float64)      # [n, Hkv, d]
    v = wl.v_cache[pages, :, offs, :].to(torch.float64)
    if wl.spec.kv_dtype == "int8":
        k = k * wl.k_scale[pages, :, offs].to(torch.float64)[..., None]
        v = v * wl.v_scale[pages, :, offs].to(torch.float64)[..., None]
    return k.permute(1, 0, 2), v.permute(1, 0, 2)            # [Hkv, n, d]


def _library_attention(wl, b):
    """torch SDPA output and torch.logsumexp LSE for request b (float64)."""
    k, v = _dense_kv(wl, b)
    q = wl.q[b].to(torch.float64)                            # [Hq, d]
    g = wl.spec.num_q_heads // wl.spec.num_kv_heads
    out = torch.nn.functional.scaled_dot_product_attention(
        q[None, :, None, :], k[None], v[None], scale=wl.sm_scale, enable_gqa=True)[0, :, 0, :]
    scores = torch.einsum("hd,hnd->hn", q, k.repeat_interleave(g, dim=0)) * wl.sm_scale
    lse = torch.logsumexp(scores, dim=-1)
    return out.numpy(), lse.numpy()


# --------------------------------------------------------------------------------------
# Checks, written once and used both on the real oracle and on planted-mistake builds.
# Each returns normally when the pin holds and raises AssertionError otherwise.
# --------------------------------------------------------------------------------------

def check_metadata_hand_example(lib=None):
    fx = _fixture("metadata_hand_example.json")
    out = oracle.build_metadata(
        np.array(fx["req_pool_indices"], np.int64), np.array(fx["seq_lens"], np.int64),
        np.array(fx["req_to_token"], np.int32), fx["seqlen_offset"], fx["max_seq_pages"],
        fx["page_size"], np.array(fx["full_to_swa_mapping"], np.int64),
        cu_seqlens_k_init=[77, 77, 77], lib=lib)
    for key, want in fx["expected"].items():
        np.testing.assert_array_equal(out[key], np.array(want, np.int32), err_msg=key)
    cq = fx["cu_seqlens_q"]
    np.testing.assert_array_equal(
        oracle.cu_seqlens_q(np.array(cq["qlens"], np.int64), 3, 1, lib=lib), cq["cumsum"])
    np.testing.assert_array_equal(
        oracle.cu_seqlens_q(None, 3, 2, cq["q_stride"], lib=lib), cq["strided"])
    so = fx["swa_out_cache_loc"]
    np.testing.assert_array_equal(
        oracle.swa_out_cache_loc(np.array(so["out_cache_loc"], np.int64),
                                 np.array(fx["full_to_swa_mapping"], np.int64),
                                 so["swa_out_len"], lib=lib), so["expected"])


def check_negative_token_reading(lib=None):
    """A -1 token (never a real slot) divides with C truncation: page 0; its SWA entry
    is -1.  Only the first slot of each page (column p * page_size) is read."""
    r2t = np.array([[0, 1, -1, 3]], np.int32)
    mapping = np.arange(10, dtype=np.int64)
    out = oracle.build_metadata(np.array([0], np.int64), np.array([4], np.int64), r2t, 0, 2, 2,
                                mapping, lib=lib)
    np.testing.assert_array_equal(out["page_table"], [[0, 0]])
    np.testing.assert_array_equal(out["swa_page_table"], [[0, -1]])


def check_metadata_against_generator(wl, lib=None):
    meta = _oracle_metadata(wl, lib)
    P = wl.spec.page_size
    cl = meta["cache_seqlens"]
    np.testing.assert_array_equal(cl, np.array(wl.ctx, np.int32))
    cu = meta["cu_seqlens_k"]
    assert cu[0] == 0
    np.testing.assert_array_equal(np.diff(cu.astype(np.int64)), cl.astype(np.int64))
    assert cu[-1] == sum(wl.ctx)
    for b in range(wl.spec.bs):
        npg = len(wl.pages[b])
        np.testing.assert_array_equal(meta["page_table"][b, :npg], np.array(wl.pages[b]))
        # the unused tail of a request-to-token row is 0, so its columns read page 0
        np.testing.assert_array_equal(meta["page_table"][b, npg:], 0)
        if wl.full_to_swa_mapping is not None:
            for p in range(wl.max_seq_pages):
                # a column past the request's pages reads the zero-filled tail: slot 0
                slot = wl.pages[b][p] * P if p < npg else 0
                assert meta["swa_page_table"][b, p] == _swa_page_of_slot(wl, slot), (b, p)
    return meta


def _swa_page_of_slot(wl, slot):
    """Sliding-window page of a full-pool slot, from the generator's own record (the
    pool maps whole pages: every page holding a token of the window)."""
    P = wl.spec.page_size
    for r, pages in enumerate(wl.pages):
        if slot // P in pages:
            return wl.swa_pages[r].get(pages.index(slot // P), -1)
    return -1


def check_attention_tiny(lib=None):
    fx = _fixture("attention_tiny.json")
    q = torch.tensor(fx["q"], dtype=torch.bfloat16)
    k = torch.tensor(fx["k_cache"], dtype=torch.bfloat16)
    v = torch.tensor(fx["v_cache"], dtype=torch.bfloat16)
    out, lse = oracle.paged_attention(_bits(q), _bits(k), _bits(v),
                                      np.array(fx["page_table"], np.int32),
                                      np.array(fx["cache_seqlens"], np.int32), fx["sm_scale"],
                                      lib=lib)
    np.testing.assert_allclose(out, fx["expected_out"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, fx["expected_lse"], rtol=0, atol=1e-12)


def check_attention_against_library(wl, lib=None):
    meta = _oracle_metadata(wl, lib)
    out, lse = _oracle_attention(wl, meta, lib)
    for b in range(wl.spec.bs):
        if wl.ctx[b] == 0:
            continue
        ref_out, ref_lse = _library_attention(wl, b)
        np.testing.assert_allclose(out[b], ref_out, rtol=0, atol=1e-10)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=0, atol=1e-10)
    return out, lse


def check_split_invariance(wl, splits=(1, 2, 3, 4, 7, 32), lib=None):
    meta = _oracle_metadata(wl, lib)
    out, lse = _oracle_attention(wl, meta, lib)
    k, v, ks, vs = _kv_np(wl)
    for s in splits:
        m, l, acc = oracle.splitk_partials(_bits(wl.q), k, v, meta["page_table"],
                                           meta["cache_seqlens"], wl.sm_scale,
                                           wl.max_seq_pages, s, ks, vs, lib=lib)
        o2, lse2 = oracle.combine_splits(m, l, acc, lib=lib)
        np.testing.assert_allclose(o2, out, rtol=0, atol=1e-12, err_msg=f"S={s}")
        np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12, err_msg=f"S={s}")


def check_closed_forms(lib=None):
    d, P = 128, 64
    g = torch.Generator().manual_seed(7)
    # one token: out = v0, lse = x0
    q = torch.randn(1, 2, d, generator=g).to(torch.bfloat16)
    k = torch.randn(3, 1, P, d, generator=g).to(torch.bfloat16)
    v = torch.randn(3, 1, P, d, generator=g).to(torch.bfloat16)
    pt = np.array([[2]], np.int32)
    out, lse = oracle.paged_attention(_bits(q), _bits(k), _bits(v), pt,
                                      np.array([1], np.int32), 0.125, lib=lib)
    v0 = v[2, 0, 0].double().numpy()
    np.testing.assert_allclose(out[0, 0], v0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[0, 1], v0, rtol=0, atol=1e-12)
    x0 = 0.125 * (q[0].double() @ k[2, 0, 0].double()).numpy()
    np.testing.assert_allclose(lse[0], x0, rtol=0, atol=1e-12)
    # n identical keys: out = mean(v), lse = x + ln n
    n = 150
    kk = torch.randn(1, 1, 1, d, generator=g).to(torch.bfloat16).expand(3, 1, P, d).contiguous()
    pt = np.array([[1, 0, 2]], np.int32)
    out, lse = oracle.paged_attention(_bits(q), _bits(kk), _bits(v), pt,
                                      np.array([n], np.int32), 0.125, lib=lib)
    pages = [1, 0, 2]
    vs = torch.stack([v[pages[j // P], 0, j % P] for j in range(n)]).double()
    np.testing.assert_allclose(out[0, 0], vs.mean(0).numpy(), rtol=0, atol=1e-12)
    x = 0.125 * (q[0].double() @ kk[0, 0, 0].double()).numpy()
    np.testing.assert_allclose(lse[0], x + math.log(n), rtol=0, atol=1e-12)


def check_empty_context(lib=None):
    d, P = 128, 64
    q = torch.ones(2, 1, d, dtype=torch.bfloat16)
    k = torch.ones(1, 1, P, d, dtype=torch.bfloat16)
    pt = np.zeros((2, 1), np.int32)
    out, lse = oracle.paged_attention(_bits(q), _bits(k), _bits(k), pt,
                                      np.array([0, 1], np.int32), 0.5, lib=lib)
    assert np.all(out[0] == 0) and lse[0, 0] == -np.inf
    assert np.all(out[1] == 1.0) and lse[1, 0] == pytest.approx(0.5 * d)
    m = np.full((1, 1, 3), -np.inf)
    o2, lse2 = oracle.combine_splits(m, np.zeros((1, 1, 3)), np.full((1, 1, 3, 4), np.nan),
                                     lib=lib)
    assert np.all(o2 == 0) and lse2[0, 0] == -np.inf


def _small(seed, kv="bf16", **kw):
    return synthetic.make(synthetic.small_spec(seed, kv_dtype=kv, **kw))


def _gqa_small(seed, kv="bf16"):
    """Two KV heads, four query heads each: a wrong head grouping changes the result."""
    spec = synthetic.Spec(f"gqa{seed}", bs=2, num_q_heads=8, num_kv_heads=2, num_pages=12,
                          ragged=(1, 300), kv_dtype=kv, num_splits=2, seed=seed)
    return synthetic.make(spec)


def _swa_small(seed):
    spec = synthetic.Spec(f"swa{seed}", bs=4, num_q_heads=4, num_kv_heads=2, num_pages=40,
                          ragged=(1, 600), page_size=64, kv_dtype="int8", num_splits=3,
                          swa_window=130, seed=seed)
    return synthetic.make(spec)


# --------------------------------------------------------------------------------------
# Tests on the real oracle
# --------------------------------------------------------------------------------------

def test_metadata_hand_example():
    check_metadata_hand_example()


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_metadata_matches_generator(seed):
    check_metadata_against_generator(_small(seed))


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_metadata_swa_matches_window_construction(seed):
    check_metadata_against_generator(_swa_small(seed))


def test_metadata_negative_token_reading():
    check_negative_token_reading()


def test_metadata_int32_wraps():
    """cache_seqlens is an int32 cast and cu_seqlens_k an int32 running sum."""
    big = 2**31 - 10
    out = oracle.build_metadata(np.array([0, 1], np.int64), np.array([big, 100], np.int64),
                                np.zeros((2, 4), np.int32), 20, 1, 4)
    np.testing.assert_array_equal(out["cache_seqlens"], [np.int32(-2**31 + 10), 120])
    np.testing.assert_array_equal(out["cu_seqlens_k"], [0, np.int32(-2**31 + 10), np.int32(-2**31 + 130)])


def test_attention_tiny_example():
    check_attention_tiny()


@pytest.mark.parametrize("seed,kv", [(21, "bf16"), (22, "bf16"), (23, "int8"), (24, "int8")])
def test_attention_matches_torch_sdpa(seed, kv):
    check_attention_against_library(_small(seed, kv))


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_attention_gqa_matches_torch_sdpa(kv):
    check_attention_against_library(_gqa_small(25, kv))


def test_attention_swa_workload_matches_torch_sdpa():
    check_attention_against_library(_swa_small(31))


def test_attention_closed_forms():
    check_closed_forms()


def test_empty_context():
    check_empty_context()


@pytest.mark.parametrize("seed,kv", [(41, "bf16"), (42, "int8")])
def test_split_count_invariance(seed, kv):
    check_split_invariance(_small(seed, kv, ctx_max=700))


def test_page_relabelling_is_bit_identical():
    wl = _small(51, ctx_max=400)
    meta = _oracle_metadata(wl)
    out, lse = _oracle_attention(wl, meta)
    perm = torch.randperm(wl.spec.num_pages, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(len(perm))
    k2 = wl.k_cache[perm]            # new page i holds old page perm[i]
    v2 = wl.v_cache[perm]
    pt2 = inv.numpy().astype(np.int32)[meta["page_table"]]
    out2, lse2 = oracle.paged_attention(_bits(wl.q), _bits(k2), _bits(v2), pt2,
                                        meta["cache_seqlens"], wl.sm_scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_request_order_permutes_outputs():
    wl = _small(61, bs_max=5)
    meta = _oracle_metadata(wl)
    out, lse = _oracle_attention(wl, meta)
    order = np.arange(wl.spec.bs)[::-1].copy()
    k, v, _, _ = _kv_np(wl)
    out2, lse2 = oracle.paged_attention(_bits(wl.q[order]), k, v, meta["page_table"][order],
                                        meta["cache_seqlens"][order], wl.sm_scale)
    assert np.array_equal(out2, out[order]) and np.array_equal(lse2, lse[order])


# --------------------------------------------------------------------------------------
# Planted mistakes: each modified oracle must fail at least one pin.
# --------------------------------------------------------------------------------------

PLANTS = {
    "drop_sm_scale": ("x[j] = sm_scale * dot;", "x[j] = dot;"),
    "gqa_modulo": ("const int32_t kv_head = h / group;\n      const uint16_t* qrow = q + (static_cast<int64_t>(b) * num_q_heads + h) * head_dim;\n      double* orow",
                   "const int32_t kv_head = h % num_kv_heads;\n      const uint16_t* qrow = q + (static_cast<int64_t>(b) * num_q_heads + h) * head_dim;\n      double* orow"),
    "page_offset_shift": ("const int32_t off = j % page_size;\n        double dot",
                          "const int32_t off = (j + 1) % page_size;\n        double dot"),
    "lse_log2": ("x_max + std::log(denom)", "x_max + std::log2(denom)"),
    "page_table_floor_div": ("= token / page_size;", "= (token >= 0 ? token / page_size : token / page_size - 1);"),
    "page_table_wrong_column": ("static_cast<int64_t>(p) * page_size];", "static_cast<int64_t>(p) * page_size + 1];"),
    "cu_seqlens_exclusive": ("running += static_cast<uint32_t>(cache_seqlens[i]);\n    cu_seqlens_k[i + 1] = static_cast<int32_t>(running);",
                             "cu_seqlens_k[i + 1] = static_cast<int32_t>(running);\n    running += static_cast<uint32_t>(cache_seqlens[i]);"),
    "no_seqlen_offset": ("seq_lens[i] + static_cast<int64_t>(seqlen_offset)", "seq_lens[i]"),
    "swa_no_negative_guard": ("swa_token < 0 ? -1 : static_cast<int32_t>(swa_token / page_size)",
                              "static_cast<int32_t>(swa_token / page_size)"),
    "int8_scale_of_wrong_row": ("return static_cast<double>(scale[row]) * code;",
                                "return static_cast<double>(scale[row / page_size]) * code;"),
    "combine_forgets_rescale": ("total += l_in[bh * num_splits + s] * w;",
                                "total += l_in[bh * num_splits + s];"),
    "split_drops_last_token": ("const int64_t end = (begin + split_tokens < n) ? begin + split_tokens : n;",
                               "const int64_t end = (begin + split_tokens < n) ? begin + split_tokens : n - 1;"),
    "softmax_missing_exp": ("const double w = std::exp(x[j] - x_max) / denom;",
                            "const double w = (x[j] - x_max + 1.0) / denom;"),
}


def plant_source(src, before, after, function=None):
    """``src`` with the first occurrence of ``before`` (after the start of ``function``
    when given) replaced by ``after``; the occurrence must lie inside that function's
    definition (before the next top-level ``int oracle_`` definition)."""
    start = src.find(f"int {function}(") if function else 0
    assert start >= 0, function
    site = src.find(before, start)
    assert site >= 0, before
    head = src.rfind("\nint oracle_", 0, site)
    nxt = src.find("\nint oracle_", head + 1)
    assert nxt == -1 or site < nxt, before
    if function:
        assert src.rfind(f"\nint {function}(", 0, site) == head, (function, before)
    return src[:site] + after + src[site + len(before):]


def _run_all_pins(lib):
    check_metadata_hand_example(lib)
    check_negative_token_reading(lib)
    for seed in (1, 2):
        check_metadata_against_generator(_small(seed), lib)
    check_metadata_against_generator(_swa_small(11), lib)
    check_attention_tiny(lib)
    check_closed_forms(lib)
    check_empty_context(lib)
    for seed, kv in ((21, "bf16"), (23, "int8")):
        check_attention_against_library(_small(seed, kv), lib)
    check_attention_against_library(_gqa_small(25), lib)
    check_split_invariance(_small(41, "bf16", ctx_max=700), splits=(1, 3, 7), lib=lib)


def test_unplanted_build_passes_all_pins(tmp_path):
    src = open(oracle._SRC).read()
    path = tmp_path / "clean.cpp"
    path.write_text(src)
    lib = oracle.load(oracle.build(str(path), str(tmp_path / "libclean.so")))
    _run_all_pins(lib)


@pytest.mark.parametrize("plant", sorted(PLANTS))
def test_planted_mistakes_are_caught(plant, tmp_path):
    before, after = PLANTS[plant]
    src = open(oracle._SRC).read()
    # the site is unique, or (for lines later functions repeat) its first occurrence,
    # inside the first function that holds it
    path = tmp_path / f"{plant}.cpp"
    path.write_text(plant_source(src, before, after))
    lib = oracle.load(oracle.build(str(path), str(tmp_path / f"lib{plant}.so")))
    with pytest.raises(AssertionError):
        _run_all_pins(lib)
