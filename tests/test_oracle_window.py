"""Pins for the sliding-window oracle (attention through the sliding-window page table
and the window's split partials).

* torch's scaled_dot_product_attention in float64, with K/V gathered from the
  sliding-window pool through the generator's own page record (not the metadata
  stage's table) and a band mask, for decode and multi-token queries, bf16 and int8,
  with and without -1 holes in the table;
* a window of one token gives exactly that token's V and its score as lse;
* a window covering the whole context, read through the full table and pool, is the
  decode (and multi-query) oracle exactly;
* the split partials combine to the windowed attention for any split count, and a
  hand-worked example fixes which positions each split holds;
* planted mistakes in the window bounds, the hole skip, the query position and the
  split partition are caught.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_metadata_gb300 import synthetic

from test_oracle_pins import _bits, _dense_kv, _oracle_metadata, plant_source


def _kv(k, v, ks, vs):
    if k.dtype == torch.int8:
        return k.numpy(), v.numpy(), ks.numpy(), vs.numpy()
    return _bits(k), _bits(v), None, None


def _case(seed, kv="bf16", window=150, page_size=16, max_q_len=None, holes=0):
    """A small ragged batch with a sliding-window pool; returns (wl, q, cu_q, table)."""
    spec = synthetic.Spec(f"w{seed}", bs=3, num_q_heads=8, num_kv_heads=2, num_pages=80,
                          ragged=(1, 400), page_size=page_size, kv_dtype=kv,
                          swa_window=window, seed=seed)
    wl = synthetic.make(spec, with_swa_cache=True)
    table = _oracle_metadata(wl)["swa_page_table"].copy()
    g = torch.Generator().manual_seed(seed + 5)
    for _ in range(holes):        # knock out mapped pages of random requests
        b = int(torch.randint(0, spec.bs, (1,), generator=g))
        mapped = sorted(wl.swa_pages[b])
        table[b, mapped[int(torch.randint(0, len(mapped), (1,), generator=g))]] = -1
    if max_q_len is None:
        return wl, wl.q, None, table
    qlens = synthetic.draw_query_lengths(spec.bs, max_q_len, seed + 1)
    cu_q = oracle.cu_seqlens_q(qlens.numpy(), spec.bs, 1)
    q = synthetic.draw_queries(int(cu_q[-1]), spec.num_q_heads, spec.head_dim, seed + 2)
    return wl, q, cu_q, table


def _window_oracle(wl, q, cu_q, table, lib=None, window=None):
    k, v, ks, vs = _kv(wl.k_swa, wl.v_swa, wl.k_swa_scale, wl.v_swa_scale)
    return oracle.paged_attention_window(_bits(q), k, v, table, np.array(wl.ctx, np.int32),
                                         window or wl.spec.swa_window, wl.sm_scale, cu_q, ks, vs,
                                         lib=lib)


def _rows(wl, cu_q, b):
    if cu_q is None:
        return b, 1
    return int(cu_q[b]), int(cu_q[b + 1] - cu_q[b])


def check_against_torch_sdpa(seed, kv="bf16", max_q_len=None, holes=0, lib=None):
    wl, q, cu_q, table = _case(seed, kv, max_q_len=max_q_len, holes=holes)
    out, lse = _window_oracle(wl, q, cu_q, table, lib)
    P, W = wl.spec.page_size, wl.spec.swa_window
    g = wl.spec.num_q_heads // wl.spec.num_kv_heads
    for b in range(wl.spec.bs):
        n = wl.ctx[b]
        # K/V of every position the pool holds, through the generator's page record
        held = [j for j in range(n) if j // P in wl.swa_pages[b] and table[b, j // P] >= 0]
        sp = torch.tensor([wl.swa_pages[b][j // P] for j in held], dtype=torch.long)
        off = torch.tensor([j % P for j in held], dtype=torch.long)
        kd = wl.k_swa[sp, :, off, :].to(torch.float64)
        vd = wl.v_swa[sp, :, off, :].to(torch.float64)
        if kv == "int8":
            kd = kd * wl.k_swa_scale[sp, :, off].to(torch.float64)[..., None]
            vd = vd * wl.v_swa_scale[sp, :, off].to(torch.float64)[..., None]
        kd, vd = kd.permute(1, 0, 2), vd.permute(1, 0, 2)           # [Hkv, held, d]
        r0, q_len = _rows(wl, cu_q, b)
        rows = q[r0:r0 + q_len].to(torch.float64)                   # [q_len, Hq, d]
        pos = torch.tensor(held, dtype=torch.long)
        qpos = n - q_len + torch.arange(q_len)
        mask = (pos[None, :] <= qpos[:, None]) & (pos[None, :] > qpos[:, None] - W)
        for i in range(q_len):
            if not bool(mask[i].any()):
                assert np.all(np.isneginf(lse[r0 + i])) and np.all(out[r0 + i] == 0)
                continue
            m = mask[i]
            ref = torch.nn.functional.scaled_dot_product_attention(
                rows[i][None, :, None, :], kd[None][:, :, m], vd[None][:, :, m],
                scale=wl.sm_scale, enable_gqa=True)[0, :, 0, :]
            scores = torch.einsum("hd,hnd->hn", rows[i], kd[:, m].repeat_interleave(g, dim=0))
            ref_lse = torch.logsumexp(scores * wl.sm_scale, dim=-1)
            np.testing.assert_allclose(out[r0 + i], ref.numpy(), rtol=0, atol=1e-10)
            np.testing.assert_allclose(lse[r0 + i], ref_lse.numpy(), rtol=0, atol=1e-10)


def check_window_of_one(lib=None):
    wl, q, cu_q, table = _case(31, "bf16", max_q_len=3)
    out, lse = _window_oracle(wl, q, cu_q, table, lib, window=1)
    P = wl.spec.page_size
    g = wl.spec.num_q_heads // wl.spec.num_kv_heads
    for b in range(wl.spec.bs):
        r0, q_len = _rows(wl, cu_q, b)
        for i in range(q_len):
            pos = wl.ctx[b] - q_len + i
            if pos < 0:
                assert np.all(np.isneginf(lse[r0 + i]))
                continue
            sp, o = wl.swa_pages[b][pos // P], pos % P
            for h in range(wl.spec.num_q_heads):
                vrow = wl.v_swa[sp, h // g, o].to(torch.float64).numpy()
                krow = wl.k_swa[sp, h // g, o].to(torch.float64)
                assert np.array_equal(out[r0 + i, h], vrow)
                score = float((q[r0 + i, h].to(torch.float64) * krow).sum()) * wl.sm_scale
                assert abs(lse[r0 + i, h] - score) <= 1e-12 * max(1.0, abs(score))


def check_full_window_is_full_attention(lib=None):
    spec = synthetic.Spec("wfull", bs=3, num_q_heads=8, num_kv_heads=2, num_pages=30,
                          ragged=(1, 400), kv_dtype="int8", seed=41)
    wl = synthetic.make(spec)
    meta = _oracle_metadata(wl)
    k, v, ks, vs = _kv(wl.k_cache, wl.v_cache, wl.k_scale, wl.v_scale)
    big = max(wl.ctx) + 5
    o1, l1 = oracle.paged_attention_window(_bits(wl.q), k, v, meta["page_table"],
                                           meta["cache_seqlens"], big, wl.sm_scale, None, ks, vs,
                                           lib=lib)
    o0, l0 = oracle.paged_attention(_bits(wl.q), k, v, meta["page_table"], meta["cache_seqlens"],
                                    wl.sm_scale, ks, vs)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)
    qlens = synthetic.draw_query_lengths(spec.bs, 4, 42)
    cu_q = oracle.cu_seqlens_q(qlens.numpy(), spec.bs, 1)
    q = synthetic.draw_queries(int(cu_q[-1]), 8, 128, 43)
    o1, l1 = oracle.paged_attention_window(_bits(q), k, v, meta["page_table"],
                                           meta["cache_seqlens"], big, wl.sm_scale, cu_q, ks, vs,
                                           lib=lib)
    o0, l0 = oracle.paged_attention_multi(_bits(q), k, v, meta["page_table"],
                                          meta["cache_seqlens"], cu_q, wl.sm_scale, ks, vs)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)


def check_partials_combine(seed, kv, max_q_len, splits, lib=None):
    wl, q, cu_q, table = _case(seed, kv, max_q_len=max_q_len, holes=2)
    k, v, ks, vs = _kv(wl.k_swa, wl.v_swa, wl.k_swa_scale, wl.v_swa_scale)
    cl = np.array(wl.ctx, np.int32)
    out, lse = _window_oracle(wl, q, cu_q, table, lib)
    for S in splits:
        m, l, acc = oracle.splitk_partials_window(_bits(q), k, v, table, cl, wl.spec.swa_window,
                                                  wl.sm_scale, wl.max_seq_pages, S, cu_q,
                                                  max_q_len or 1, ks, vs, lib=lib)
        assert np.all(l[np.isneginf(m)] == 0)
        o2, l2 = oracle.combine_splits(m, l, acc)
        np.testing.assert_allclose(o2, out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l2, lse, rtol=0, atol=1e-12)


def check_partition_hand_example(lib=None):
    """page_size 4, one kv head, 13 cached tokens on pages 0..3 (identity table; page 2,
    positions 8..11, a hole in one case), max_seq_pages 4.  K = 0, so every visible
    token has weight exactly 1, and V_j = e_j (channel j) makes acc the indicator of
    the positions a split holds.

    window 6, two splits: window_pages = min(4, (6 + max_q_len - 2) // 4 + 2) = 3 for
    max_q_len 1..3, split_tokens = 4 * ceil(3 / 2) = 8.
      decode: the query at position 12 sees 7..12; base = 4 * floor(7 / 4) = 4, so
        split 0 = [4, 12) holds 7..11 and split 1 = [12, 20) holds 12.
      three queries (positions 10, 11, 12): the first visible position is 5, base 4:
        query 0 sees 5..10 -> split 0: 5..10, split 1: none
        query 1 sees 6..11 -> split 0: 6..11, split 1: none
        query 2 sees 7..12 -> split 0: 7..11, split 1: 12
      the same with page 2 a hole: query 0 -> 5, 6, 7 | none; query 1 -> 6, 7 | none;
        query 2 -> 7 | 12.
    window 8, three queries, one split: window_pages = min(4, (8 + 3 - 2) // 4 + 2) = 4,
    split_tokens = 16; first visible 3, base 0: the split holds 3..10, 4..11 and 5..12.
    """
    P, d = 4, 128
    k = np.zeros((4, 1, P, d), np.uint16)
    vals = np.zeros((4, 1, P, d), np.float32)
    for j in range(16):
        vals[j // P, 0, j % P, j] = 1.0
    v = (vals.view(np.uint32) >> 16).astype(np.uint16)
    cl = np.array([13], np.int32)
    ident = np.array([[0, 1, 2, 3]], np.int32)
    three = np.array([0, 3], np.int32)

    def tokens(m, l, acc, row, s):
        if np.isneginf(m[row, 0, s]):
            assert l[row, 0, s] == 0
            return []
        assert m[row, 0, s] == 0
        idx = np.nonzero(acc[row, 0, s])[0].tolist()
        assert np.all(acc[row, 0, s, idx] == 1.0) and l[row, 0, s] == len(idx)
        return idx

    r = lambda a, b: list(range(a, b + 1))
    cases = [  # table, cu_seqlens_q, max_q_len, window, splits, positions per row and split
        (ident, None, 1, 6, 2, [[r(7, 11), [12]]]),
        (ident, three, 3, 6, 2, [[r(5, 10), []], [r(6, 11), []], [r(7, 11), [12]]]),
        (np.array([[0, 1, -1, 3]], np.int32), three, 3, 6, 2,
         [[[5, 6, 7], []], [[6, 7], []], [[7], [12]]]),
        (ident, three, 3, 8, 1, [[r(3, 10)], [r(4, 11)], [r(5, 12)]]),
    ]
    for table, cu_q, mql, window, S, want in cases:
        rows = len(want)
        q = np.full((rows, 1, d), 0x3F80, np.uint16)            # 1.0
        m, l, acc = oracle.splitk_partials_window(q, k, v, table, cl, window, 1.0, 4, S, cu_q,
                                                  mql, lib=lib)
        for row in range(rows):
            got = [tokens(m, l, acc, row, s) for s in range(S)]
            assert got == want[row], (row, table.tolist(), window, S, got)


def test_against_torch_sdpa_decode():
    check_against_torch_sdpa(51, "bf16")


@pytest.mark.parametrize("seed,kv,mql,holes", [(52, "int8", None, 3), (53, "bf16", 4, 2),
                                               (54, "int8", 3, 0)])
def test_against_torch_sdpa(seed, kv, mql, holes):
    check_against_torch_sdpa(seed, kv, mql, holes)


def test_window_of_one_token():
    check_window_of_one()


def test_window_covering_the_context_is_full_attention():
    check_full_window_is_full_attention()


@pytest.mark.parametrize("seed,kv,mql", [(61, "bf16", None), (62, "int8", 4)])
def test_partials_combine_to_window_attention(seed, kv, mql):
    check_partials_combine(seed, kv, mql, (1, 2, 3, 7, 40))


def test_partition_hand_example():
    check_partition_hand_example()


WINDOW_PLANTS = {
    "window_start_off_by_one": ("oracle_paged_attention_window",
                                "const int64_t lo = pos - window + 1 > 0 ? pos - window + 1 : 0;",
                                "const int64_t lo = pos - window > 0 ? pos - window : 0;"),
    "window_excludes_query": ("oracle_paged_attention_window",
                              "for (int64_t j = lo; j <= pos; ++j) {",
                              "for (int64_t j = lo; j < pos; ++j) {"),
    "hole_read_as_page_zero": ("oracle_paged_attention_window",
                               "if (page < 0) continue;\n        tok.push_back(j);\n        pg.push_back(page);",
                               "tok.push_back(j);\n        pg.push_back(page < 0 ? 0 : page);"),
    "query_positions_reversed": ("oracle_paged_attention_window",
                                 "const int64_t pos = n - q_len + i;",
                                 "const int64_t pos = n - 1 - i;"),
    "split_base_not_page_aligned": ("oracle_splitk_partials_window",
                                    "const int64_t base = first / page_size * page_size;",
                                    "const int64_t base = first;"),
    "split_window_pages_without_queries": ("oracle_splitk_partials_window",
                                           "(static_cast<int64_t>(window) + max_q_len - 2) / page_size + 2;",
                                           "(static_cast<int64_t>(window) - 1) / page_size + 2;"),
    "split_window_start_off_by_one": ("oracle_splitk_partials_window",
                                      "const int64_t lo = pos - window + 1 > 0 ? pos - window + 1 : 0;",
                                      "const int64_t lo = pos - window > 0 ? pos - window : 0;"),
}


def _run_window_pins(lib):
    check_against_torch_sdpa(51, "bf16", lib=lib)
    check_against_torch_sdpa(53, "bf16", 4, 2, lib=lib)
    check_window_of_one(lib)
    check_full_window_is_full_attention(lib)
    check_partials_combine(62, "int8", 4, (1, 3), lib=lib)
    check_partition_hand_example(lib)


@pytest.mark.parametrize("plant", sorted(WINDOW_PLANTS))
def test_window_plants_are_caught(plant, tmp_path):
    function, before, after = WINDOW_PLANTS[plant]
    src = open(oracle._SRC).read()
    path = tmp_path / f"{plant}.cpp"
    path.write_text(plant_source(src, before, after, function))
    lib = oracle.load(oracle.build(str(path), str(tmp_path / f"lib{plant}.so")))
    with pytest.raises(AssertionError):
        _run_window_pins(lib)
