"""Writes the hand-worked fixtures in this folder.

The values are worked by hand from the formulas the fixtures cite (integer metadata
by direct substitution; the tiny attention case by its closed form with math.exp /
math.log).  Nothing here calls the CUDA path or the oracle.

    python tests/golden/make_golden.py
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def metadata_fixture():
    P = 4

    def row(pages):
        return [pages[j // P] * P + j % P for j in range(12)]

    mapping = [-1] * (9 * P + P + 1)
    for page, swa in ((6, 0), (8, 1), (7, 2)):
        for off in range(P):
            mapping[page * P + off] = swa * P + off
    return {
        "citation": "sglang trtllm_mha_graph_metadata.py: module docstring (cache_seqlens, "
                    "cu_seqlens_k, page_table, swa_page_table, swa_out_cache_loc, cu_seqlens_q "
                    "formulas) and the launcher's num_out_tokens = min(swa_out_len, "
                    "len(out_cache_loc)). Values worked by hand from those formulas.",
        "derivation": [
            "req_to_token rows have stride 12 and page_size 4; row r holds page[j/4]*4 + j%4 for the page lists below.",
            "row 0 pages [5,2,7]; row 1 pages [1,3,0]; row 2 pages [4,6,8].",
            "request 0 uses pool row 2 -> page_table row [16/4, 24/4, 32/4] = [4,6,8]; request 1 uses row 0 -> [20/4, 8/4, 28/4] = [5,2,7].",
            "cache_seqlens = seq_lens + 1 = [10, 6]; cu_seqlens_k = [0, 10, 16].",
            "full_to_swa_mapping has 9*4+4+1 = 41 entries; slots of page 6 map to swa slots 0..3, page 8 to 4..7, page 7 to 8..11, all others -1.",
            "swa row 0: map[16]=-1 -> -1, map[24]=0 -> 0, map[32]=4 -> 1; swa row 1: map[20]=-1, map[8]=-1, map[28]=8 -> 2.",
            "cu_seqlens_q cumsum mode with qlens [3,1,2] -> [0,3,4,6]; strided mode with q_stride 4 -> [0,4,8,12].",
            "swa_out_cache_loc with out_cache_loc [24,-1,29,17] and swa_out_len 6 -> [map[24]=0, -1, map[29]=9, map[17]=-1, 0, 0].",
        ],
        "page_size": P,
        "req_to_token": [row([5, 2, 7]), row([1, 3, 0]), row([4, 6, 8])],
        "req_pool_indices": [2, 0],
        "seq_lens": [9, 5],
        "seqlen_offset": 1,
        "max_seq_pages": 3,
        "full_to_swa_mapping": mapping,
        "expected": {
            "cache_seqlens": [10, 6],
            "cu_seqlens_k": [0, 10, 16],
            "page_table": [[4, 6, 8], [5, 2, 7]],
            "swa_page_table": [[-1, 0, 1], [-1, -1, 2]],
        },
        "cu_seqlens_q": {"qlens": [3, 1, 2], "cumsum": [0, 3, 4, 6], "q_stride": 4,
                         "strided": [0, 4, 8, 12]},
        "swa_out_cache_loc": {"out_cache_loc": [24, -1, 29, 17], "swa_out_len": 6,
                              "expected": [0, -1, 9, -1, 0, 0]},
    }


def attention_fixture():
    e = math.e
    Z = 1 + e + e * e
    return {
        "citation": "Scaled dot-product attention by its definition, softmax(q K^T * sm_scale) V "
                    "with LSE = ln sum exp(scores); the split-K producer/reducer pair it is "
                    "computed by is named in lmdeploy PR #4861 (Changes: Split-K paged "
                    "attention). Worked by hand.",
        "derivation": [
            "head_dim 2, page_size 2, one request of 3 tokens, one query head and one KV head, sm_scale 1.",
            "tokens 0,1 live in page 1 and token 2 in page 0, so page_table = [[1, 0]].",
            "q = [1,0]; k0 = [1,0], k1 = [0,1], k2 = [2,0]  -> scores x = [1, 0, 2].",
            "v0 = [1,0], v1 = [0,1], v2 = [1,1].",
            "Z = e^1 + e^0 + e^2; out = [(e + e^2)/Z, (1 + e^2)/Z]; lse = ln Z.",
        ],
        "head_dim": 2, "page_size": 2, "sm_scale": 1.0,
        "q": [[[1.0, 0.0]]],
        "k_cache": [[[[2.0, 0.0], [0.0, 0.0]]], [[[1.0, 0.0], [0.0, 1.0]]]],
        "v_cache": [[[[1.0, 1.0], [0.0, 0.0]]], [[[1.0, 0.0], [0.0, 1.0]]]],
        "page_table": [[1, 0]],
        "cache_seqlens": [3],
        "expected_out": [[[(e + e * e) / Z, (1 + e * e) / Z]]],
        "expected_lse": [[math.log(Z)]],
    }


if __name__ == "__main__":
    for name, fx in (("metadata_hand_example.json", metadata_fixture()),
                     ("attention_tiny.json", attention_fixture())):
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(fx, f, indent=1)
            f.write("\n")
