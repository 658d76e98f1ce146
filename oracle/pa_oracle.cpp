// Plain, slow CPU oracle for the decode-step paged-KV attention path.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
// CPU-baseline leg load this library.  It shares no code, header, table or
// helper with the CUDA path, and the CUDA path never calls it.
//
// Every function is a direct statement of what the path computes, written as
// nested loops with double-precision accumulation:
//
//   * oracle_build_metadata   - the fused metadata update described by the sglang
//     module "trtllm_mha_graph_metadata.py" (module docstring, and the kernel
//     update_trtllm_mha_graph_metadata_kernel: row program, scan program, SWA
//     branch, swa_out_cache_loc branch, cu_seqlens_q modes).
//   * oracle_paged_attention  - softmax(q K^T * sm_scale) V per request and query
//     head over the tokens the page table addresses, plus the natural-log
//     log-sum-exp of the scaled scores.  The pages name the split-K paged
//     attention producer and reducer (lmdeploy PR #4861, "perf(cuda): use PDL for
//     paged attention and V4 prefill", section Changes / Split-K paged attention)
//     but do not print the attention arithmetic, so this is the textbook
//     definition of scaled dot-product attention with grouped KV heads.
//   * oracle_paged_attention_multi - the same attention for several query tokens per
//     request (rows given by cu_seqlens_q, the module's query-length output), causal
//     within the request's newest tokens.
//   * oracle_paged_attention_window - sliding-window attention through the SWA page
//     table the metadata module builds (swa_page_table): each query sees only its
//     `window` newest positions, read from the sliding-window pool, and skips pages
//     whose table entry is -1.  The pages build the table but do not print the
//     attention that reads it; the window reading is stated at the function.
//   * oracle_splitk_partials  - the per-split partial results (running max m,
//     sum of exponentials l, unnormalised accumulator acc) that the split-K
//     producer writes to scratch, for a given split of the context.
//   * oracle_splitk_partials_window - the same partials for the sliding-window
//     attention, over the window's split partition.
//   * oracle_combine_splits   - the log-sum-exp combination the reducer performs.
//
// Parity pins: every function here is checked by CPU tests against hand-worked
// examples, closed forms, library routines and invariants (tests/test_oracle_*).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

// bf16 is the upper 16 bits of an IEEE-754 binary32 value; widening is exact.
double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof(f));
  return static_cast<double>(f);
}

// Element (page, kv_head, offset, c) of a paged cache laid out as
// [num_pages][num_kv_heads][page_size][head_dim].
// kv_dtype 0: bf16 values.  kv_dtype 1: int8 codes times an fp32 scale stored per
// (page, kv_head, offset), the symmetric per-token-per-head quantisation.
double kv_element(const void* cache, const float* scale, int32_t kv_dtype,
                  int64_t page, int32_t kv_head, int32_t off, int32_t c,
                  int32_t num_kv_heads, int32_t page_size, int32_t head_dim) {
  const int64_t row = (page * num_kv_heads + kv_head) * page_size + off;
  const int64_t idx = row * head_dim + c;
  if (kv_dtype == 0) {
    return bf16_bits_to_double(static_cast<const uint16_t*>(cache)[idx]);
  }
  const double code = static_cast<double>(static_cast<const int8_t*>(cache)[idx]);
  return static_cast<double>(scale[row]) * code;
}

}  // namespace

extern "C" {

// Fused metadata update (sglang trtllm_mha_graph_metadata.py, module docstring):
//   cache_seqlens[i]  = int32(seq_lens[i] + seqlen_offset)
//   cu_seqlens_k[0]   = 0, cu_seqlens_k[i+1] = cu_seqlens_k[i] + cache_seqlens[i]
//                       (int32 running sum, wrapping like 32-bit hardware adds)
//   page_table[i, p]  = req_to_token[req_pool_indices[i], p * page_size] / page_size
//                       for p < max_seq_pages (C truncating division)
//   swa_page_table[i, p] (only when full_to_swa_mapping is given):
//                       t = req_to_token[...] as above; s = t >= 0 ? map[t] : -1;
//                       s < 0 ? -1 : int32(s / page_size)
// Returns 0.  bs == 0 writes nothing (the launcher returns early for an empty batch).
int oracle_build_metadata(const int64_t* req_pool_indices, const int64_t* seq_lens,
                          const int32_t* req_to_token, int64_t req_to_token_stride,
                          const int64_t* full_to_swa_mapping,
                          int32_t* cache_seqlens, int32_t* cu_seqlens_k,
                          int32_t* page_table, int64_t page_table_stride,
                          int32_t* swa_page_table, int64_t swa_page_table_stride,
                          int32_t bs, int32_t seqlen_offset, int32_t max_seq_pages,
                          int32_t page_size) {
  if (bs <= 0) return 0;
  for (int32_t i = 0; i < bs; ++i) {
    const int64_t sum = seq_lens[i] + static_cast<int64_t>(seqlen_offset);
    cache_seqlens[i] = static_cast<int32_t>(static_cast<uint32_t>(static_cast<uint64_t>(sum)));
  }
  uint32_t running = 0;
  cu_seqlens_k[0] = 0;
  for (int32_t i = 0; i < bs; ++i) {
    running += static_cast<uint32_t>(cache_seqlens[i]);
    cu_seqlens_k[i + 1] = static_cast<int32_t>(running);
  }
  for (int32_t i = 0; i < bs; ++i) {
    const int64_t row = req_pool_indices[i];
    for (int32_t p = 0; p < max_seq_pages; ++p) {
      const int32_t token =
          req_to_token[row * req_to_token_stride + static_cast<int64_t>(p) * page_size];
      page_table[static_cast<int64_t>(i) * page_table_stride + p] = token / page_size;
      if (full_to_swa_mapping != nullptr) {
        const int64_t swa_token = token >= 0 ? full_to_swa_mapping[token] : -1;
        const int32_t swa_page =
            swa_token < 0 ? -1 : static_cast<int32_t>(swa_token / page_size);
        swa_page_table[static_cast<int64_t>(i) * swa_page_table_stride + p] = swa_page;
      }
    }
  }
  return 0;
}

// cu_seqlens_q in the two computed modes of the same module (cu_seqlens_q[0] is
// written as 0 here; the module leaves it preset):
//   mode 1 (cumsum):  cu_seqlens_q[i+1] = sum_{j<=i} int32(qlens[j])
//   mode 2 (strided): cu_seqlens_q[i+1] = (i + 1) * q_stride
// Mode 0 leaves the buffer untouched.
int oracle_cu_seqlens_q(const int64_t* qlens, int32_t* cu_seqlens_q, int32_t bs,
                        int32_t q_mode, int32_t q_stride) {
  if (bs <= 0 || q_mode == 0) return 0;
  cu_seqlens_q[0] = 0;
  uint32_t running = 0;
  for (int32_t i = 0; i < bs; ++i) {
    if (q_mode == 1) {
      running += static_cast<uint32_t>(static_cast<int32_t>(qlens[i]));
      cu_seqlens_q[i + 1] = static_cast<int32_t>(running);
    } else {
      cu_seqlens_q[i + 1] = static_cast<int32_t>(
          static_cast<uint32_t>(i + 1) * static_cast<uint32_t>(q_stride));
    }
  }
  return 0;
}

// swa_out_cache_loc translation of the same module: for idx < swa_out_len,
// idx < num_out_tokens  -> loc = out_cache_loc[idx]; loc < 0 ? -1 : map[loc]
// otherwise             -> 0 (zero padding), with
// num_out_tokens = min(swa_out_len, out_cache_loc_len).
int oracle_swa_out_cache_loc(const int64_t* out_cache_loc, int64_t out_cache_loc_len,
                             const int64_t* full_to_swa_mapping,
                             int64_t* swa_out_cache_loc, int64_t swa_out_len) {
  const int64_t num_out_tokens =
      out_cache_loc_len < swa_out_len ? out_cache_loc_len : swa_out_len;
  for (int64_t idx = 0; idx < swa_out_len; ++idx) {
    if (idx < num_out_tokens) {
      const int64_t loc = out_cache_loc[idx];
      swa_out_cache_loc[idx] = loc < 0 ? -1 : full_to_swa_mapping[loc];
    } else {
      swa_out_cache_loc[idx] = 0;
    }
  }
  return 0;
}

// Decode attention over a paged KV cache, one query token per request.
//   q       [bs][num_q_heads][head_dim]                      bf16 bits
//   k/v     [num_pages][num_kv_heads][page_size][head_dim]    bf16 bits or int8
//   scales  [num_pages][num_kv_heads][page_size]              fp32 (int8 only)
// Token j (0 <= j < cache_seqlens[b]) of request b lives in page
// page_table[b, j / page_size] at offset j % page_size.  Query head h reads KV head
// h / (num_q_heads / num_kv_heads).
//   x_j      = sm_scale * sum_c q[b,h,c] * K_j[c]
//   out[b,h] = sum_j exp(x_j - max x) V_j / sum_j exp(x_j - max x)
//   lse[b,h] = ln sum_j exp(x_j)
// An empty context gives out = 0 and lse = -inf.
int oracle_paged_attention(const uint16_t* q, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, int32_t kv_dtype,
                           const int32_t* page_table, int64_t page_table_stride,
                           const int32_t* cache_seqlens, int32_t bs, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                           double sm_scale, double* out, double* lse) {
  const int32_t group = num_q_heads / num_kv_heads;
  for (int32_t b = 0; b < bs; ++b) {
    const int32_t n = cache_seqlens[b];
    for (int32_t h = 0; h < num_q_heads; ++h) {
      const int32_t kv_head = h / group;
      const uint16_t* qrow = q + (static_cast<int64_t>(b) * num_q_heads + h) * head_dim;
      double* orow = out + (static_cast<int64_t>(b) * num_q_heads + h) * head_dim;
      std::vector<double> x(n > 0 ? n : 0);
      double x_max = -std::numeric_limits<double>::infinity();
      for (int32_t j = 0; j < n; ++j) {
        const int64_t page = page_table[b * page_table_stride + j / page_size];
        const int32_t off = j % page_size;
        double dot = 0.0;
        for (int32_t c = 0; c < head_dim; ++c) {
          dot += bf16_bits_to_double(qrow[c]) *
                 kv_element(k_cache, k_scale, kv_dtype, page, kv_head, off, c,
                            num_kv_heads, page_size, head_dim);
        }
        x[j] = sm_scale * dot;
        if (x[j] > x_max) x_max = x[j];
      }
      for (int32_t c = 0; c < head_dim; ++c) orow[c] = 0.0;
      if (n <= 0) {
        lse[static_cast<int64_t>(b) * num_q_heads + h] =
            -std::numeric_limits<double>::infinity();
        continue;
      }
      double denom = 0.0;
      for (int32_t j = 0; j < n; ++j) denom += std::exp(x[j] - x_max);
      for (int32_t j = 0; j < n; ++j) {
        const int64_t page = page_table[b * page_table_stride + j / page_size];
        const int32_t off = j % page_size;
        const double w = std::exp(x[j] - x_max) / denom;
        for (int32_t c = 0; c < head_dim; ++c) {
          orow[c] += w * kv_element(v_cache, v_scale, kv_dtype, page, kv_head, off, c,
                                    num_kv_heads, page_size, head_dim);
        }
      }
      lse[static_cast<int64_t>(b) * num_q_heads + h] = x_max + std::log(denom);
    }
  }
  return 0;
}

// Several query tokens per request (speculative verify / extend steps).  Query rows of
// request b are q[cu_seqlens_q[b] .. cu_seqlens_q[b+1]) ([total_q][num_q_heads][head_dim]);
// they are the last q_len = cu_seqlens_q[b+1] - cu_seqlens_q[b] tokens of the request's
// cache, so query i attends causally to token positions j < n - q_len + i + 1 with
// n = cache_seqlens[b] (an empty range gives out = 0 and lse = -inf).  Everything else
// is oracle_paged_attention.  out [total_q][num_q_heads][head_dim], lse [total_q][num_q_heads].
int oracle_paged_attention_multi(const uint16_t* q, const void* k_cache, const void* v_cache,
                                 const float* k_scale, const float* v_scale, int32_t kv_dtype,
                                 const int32_t* page_table, int64_t page_table_stride,
                                 const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
                                 int32_t bs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t page_size, double sm_scale,
                                 double* out, double* lse) {
  const int32_t group = num_q_heads / num_kv_heads;
  for (int32_t b = 0; b < bs; ++b) {
    const int32_t q_begin = cu_seqlens_q[b];
    const int32_t q_len = cu_seqlens_q[b + 1] - q_begin;
    for (int32_t i = 0; i < q_len; ++i) {
      const int64_t row = q_begin + i;
      const int64_t limit = static_cast<int64_t>(cache_seqlens[b]) - q_len + i + 1;
      const int32_t n = limit > 0 ? static_cast<int32_t>(limit) : 0;
      for (int32_t h = 0; h < num_q_heads; ++h) {
        const int32_t kv_head = h / group;
        const uint16_t* qrow = q + (row * num_q_heads + h) * head_dim;
        double* orow = out + (row * num_q_heads + h) * head_dim;
        for (int32_t c = 0; c < head_dim; ++c) orow[c] = 0.0;
        if (n == 0) {
          lse[row * num_q_heads + h] = -std::numeric_limits<double>::infinity();
          continue;
        }
        std::vector<double> x(n);
        double x_max = -std::numeric_limits<double>::infinity();
        for (int32_t j = 0; j < n; ++j) {
          const int64_t page = page_table[b * page_table_stride + j / page_size];
          double dot = 0.0;
          for (int32_t c = 0; c < head_dim; ++c) {
            dot += bf16_bits_to_double(qrow[c]) *
                   kv_element(k_cache, k_scale, kv_dtype, page, kv_head, j % page_size, c,
                              num_kv_heads, page_size, head_dim);
          }
          x[j] = sm_scale * dot;
          if (x[j] > x_max) x_max = x[j];
        }
        double denom = 0.0;
        for (int32_t j = 0; j < n; ++j) denom += std::exp(x[j] - x_max);
        for (int32_t j = 0; j < n; ++j) {
          const int64_t page = page_table[b * page_table_stride + j / page_size];
          const double w = std::exp(x[j] - x_max) / denom;
          for (int32_t c = 0; c < head_dim; ++c) {
            orow[c] += w * kv_element(v_cache, v_scale, kv_dtype, page, kv_head, j % page_size, c,
                                      num_kv_heads, page_size, head_dim);
          }
        }
        lse[row * num_q_heads + h] = x_max + std::log(denom);
      }
    }
  }
  return 0;
}

// Per-split partial results of the split-K decomposition of the same attention.
// Split s of request b covers token positions
//   [s * split_tokens, min((s + 1) * split_tokens, cache_seqlens[b]))
// with split_tokens = page_size * ceil(max_seq_pages / num_splits).
// For each (b, h, s):
//   m   = max_j x_j              (-inf for an empty split)
//   l   = sum_j exp(x_j - m)      (0 for an empty split)
//   acc = sum_j exp(x_j - m) V_j  (0 for an empty split)
// Layouts: m, l [bs][num_q_heads][num_splits]; acc [bs][num_q_heads][num_splits][head_dim].
int oracle_splitk_partials(const uint16_t* q, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, int32_t kv_dtype,
                           const int32_t* page_table, int64_t page_table_stride,
                           const int32_t* cache_seqlens, int32_t bs, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                           int32_t max_seq_pages, int32_t num_splits, double sm_scale,
                           double* m_out, double* l_out, double* acc_out) {
  const int32_t group = num_q_heads / num_kv_heads;
  const int64_t pages_per_split = (max_seq_pages + num_splits - 1) / num_splits;
  const int64_t split_tokens = pages_per_split * page_size;
  for (int32_t b = 0; b < bs; ++b) {
    const int64_t n = cache_seqlens[b];
    for (int32_t h = 0; h < num_q_heads; ++h) {
      const int32_t kv_head = h / group;
      const uint16_t* qrow = q + (static_cast<int64_t>(b) * num_q_heads + h) * head_dim;
      for (int32_t s = 0; s < num_splits; ++s) {
        const int64_t slot = (static_cast<int64_t>(b) * num_q_heads + h) * num_splits + s;
        double* acc = acc_out + slot * head_dim;
        for (int32_t c = 0; c < head_dim; ++c) acc[c] = 0.0;
        const int64_t begin = s * split_tokens;
        const int64_t end = (begin + split_tokens < n) ? begin + split_tokens : n;
        if (begin >= end) {
          m_out[slot] = -std::numeric_limits<double>::infinity();
          l_out[slot] = 0.0;
          continue;
        }
        std::vector<double> x(end - begin);
        double x_max = -std::numeric_limits<double>::infinity();
        for (int64_t j = begin; j < end; ++j) {
          const int64_t page = page_table[b * page_table_stride + j / page_size];
          const int32_t off = static_cast<int32_t>(j % page_size);
          double dot = 0.0;
          for (int32_t c = 0; c < head_dim; ++c) {
            dot += bf16_bits_to_double(qrow[c]) *
                   kv_element(k_cache, k_scale, kv_dtype, page, kv_head, off, c,
                              num_kv_heads, page_size, head_dim);
          }
          x[j - begin] = sm_scale * dot;
          if (x[j - begin] > x_max) x_max = x[j - begin];
        }
        double l = 0.0;
        for (int64_t j = begin; j < end; ++j) {
          const int64_t page = page_table[b * page_table_stride + j / page_size];
          const int32_t off = static_cast<int32_t>(j % page_size);
          const double w = std::exp(x[j - begin] - x_max);
          l += w;
          for (int32_t c = 0; c < head_dim; ++c) {
            acc[c] += w * kv_element(v_cache, v_scale, kv_dtype, page, kv_head, off, c,
                                     num_kv_heads, page_size, head_dim);
          }
        }
        m_out[slot] = x_max;
        l_out[slot] = l;
      }
    }
  }
  return 0;
}

// Sliding-window attention through the sliding-window page table.
// Request b has n = cache_seqlens[b] cached tokens and q_len query rows: rows
// cu_seqlens_q[b] .. cu_seqlens_q[b+1] when cu_seqlens_q is given, else the single row b
// (q_len = 1).  The queries are the request's newest tokens, so query i sits at position
// pos = n - q_len + i and attends positions j with
//   max(0, pos - window + 1) <= j <= pos          (its `window` newest positions)
// whose page entry page_table[b, j / page_size] is >= 0 (a -1 entry is a page the
// sliding-window pool does not hold: its tokens are skipped).  Token j is row
// j % page_size of that page of the sliding-window pool (k/v laid out as for
// oracle_paged_attention).  Scores, softmax, output and lse as in
// oracle_paged_attention; a query with no visible token gets out = 0, lse = -inf.
// out [rows][num_q_heads][head_dim], lse [rows][num_q_heads].
int oracle_paged_attention_window(const uint16_t* q, const void* k_cache, const void* v_cache,
                                  const float* k_scale, const float* v_scale, int32_t kv_dtype,
                                  const int32_t* page_table, int64_t page_table_stride,
                                  const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
                                  int32_t bs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t page_size, int32_t window,
                                  double sm_scale, double* out, double* lse) {
  const int32_t group = num_q_heads / num_kv_heads;
  for (int32_t b = 0; b < bs; ++b) {
    const int64_t q_begin = cu_seqlens_q != nullptr ? cu_seqlens_q[b] : b;
    const int64_t q_len = cu_seqlens_q != nullptr ? cu_seqlens_q[b + 1] - q_begin : 1;
    const int64_t n = cache_seqlens[b];
    for (int64_t i = 0; i < q_len; ++i) {
      const int64_t row = q_begin + i;
      const int64_t pos = n - q_len + i;
      const int64_t lo = pos - window + 1 > 0 ? pos - window + 1 : 0;
      // the visible tokens and their pages
      std::vector<int64_t> tok, pg;
      for (int64_t j = lo; j <= pos; ++j) {
        const int64_t page = page_table[b * page_table_stride + j / page_size];
        if (page < 0) continue;
        tok.push_back(j);
        pg.push_back(page);
      }
      for (int32_t h = 0; h < num_q_heads; ++h) {
        const int32_t kv_head = h / group;
        const uint16_t* qrow = q + (row * num_q_heads + h) * head_dim;
        double* orow = out + (row * num_q_heads + h) * head_dim;
        for (int32_t c = 0; c < head_dim; ++c) orow[c] = 0.0;
        if (tok.empty()) {
          lse[row * num_q_heads + h] = -std::numeric_limits<double>::infinity();
          continue;
        }
        std::vector<double> x(tok.size());
        double x_max = -std::numeric_limits<double>::infinity();
        for (size_t t = 0; t < tok.size(); ++t) {
          const int32_t off = static_cast<int32_t>(tok[t] % page_size);
          double dot = 0.0;
          for (int32_t c = 0; c < head_dim; ++c) {
            dot += bf16_bits_to_double(qrow[c]) *
                   kv_element(k_cache, k_scale, kv_dtype, pg[t], kv_head, off, c,
                              num_kv_heads, page_size, head_dim);
          }
          x[t] = sm_scale * dot;
          if (x[t] > x_max) x_max = x[t];
        }
        double denom = 0.0;
        for (size_t t = 0; t < tok.size(); ++t) denom += std::exp(x[t] - x_max);
        for (size_t t = 0; t < tok.size(); ++t) {
          const int32_t off = static_cast<int32_t>(tok[t] % page_size);
          const double w = std::exp(x[t] - x_max) / denom;
          for (int32_t c = 0; c < head_dim; ++c) {
            orow[c] += w * kv_element(v_cache, v_scale, kv_dtype, pg[t], kv_head, off, c,
                                      num_kv_heads, page_size, head_dim);
          }
        }
        lse[row * num_q_heads + h] = x_max + std::log(denom);
      }
    }
  }
  return 0;
}

// Split partials of the sliding-window attention.  The splits cover the window of the
// request rather than its whole context: with
//   window_pages = min(max_seq_pages, (window + max_q_len - 2) / page_size + 2)
// (the most pages that the positions any query of a request can see, at most
// window + max_q_len - 1 consecutive ones, can touch) and
//   split_tokens = page_size * ceil(window_pages / num_splits),
// split s of request b covers positions
//   [base + s * split_tokens, base + (s + 1) * split_tokens),
//   base = page_size * floor(max(0, n - q_len - window + 1) / page_size),
// i.e. the splits start at the page holding the first position the request's earliest
// query sees.  Each query sees, within its split, the positions and pages
// oracle_paged_attention_window lets it see; m, l, acc per (row, head, split) as in
// oracle_splitk_partials.  Rows as in oracle_paged_attention_window (cu_seqlens_q or one
// per request).
int oracle_splitk_partials_window(const uint16_t* q, const void* k_cache, const void* v_cache,
                                  const float* k_scale, const float* v_scale, int32_t kv_dtype,
                                  const int32_t* page_table, int64_t page_table_stride,
                                  const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
                                  int32_t bs, int32_t max_q_len, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                  int32_t max_seq_pages, int32_t window, int32_t num_splits,
                                  double sm_scale, double* m_out, double* l_out,
                                  double* acc_out) {
  const int32_t group = num_q_heads / num_kv_heads;
  int64_t window_pages = (static_cast<int64_t>(window) + max_q_len - 2) / page_size + 2;
  if (window_pages > max_seq_pages) window_pages = max_seq_pages;
  const int64_t split_tokens = (window_pages + num_splits - 1) / num_splits * page_size;
  for (int32_t b = 0; b < bs; ++b) {
    const int64_t q_begin = cu_seqlens_q != nullptr ? cu_seqlens_q[b] : b;
    const int64_t q_len = cu_seqlens_q != nullptr ? cu_seqlens_q[b + 1] - q_begin : 1;
    const int64_t n = cache_seqlens[b];
    const int64_t first = n - q_len - window + 1 > 0 ? n - q_len - window + 1 : 0;
    const int64_t base = first / page_size * page_size;
    for (int64_t i = 0; i < q_len; ++i) {
      const int64_t row = q_begin + i;
      const int64_t pos = n - q_len + i;
      const int64_t lo = pos - window + 1 > 0 ? pos - window + 1 : 0;
      for (int32_t h = 0; h < num_q_heads; ++h) {
        const int32_t kv_head = h / group;
        const uint16_t* qrow = q + (row * num_q_heads + h) * head_dim;
        for (int32_t s = 0; s < num_splits; ++s) {
          const int64_t slot = (row * num_q_heads + h) * num_splits + s;
          double* acc = acc_out + slot * head_dim;
          for (int32_t c = 0; c < head_dim; ++c) acc[c] = 0.0;
          const int64_t begin = base + s * split_tokens;
          const int64_t end = begin + split_tokens;
          std::vector<int64_t> tok, pg;
          for (int64_t j = begin; j < end; ++j) {
            if (j < lo || j > pos) continue;
            const int64_t page = page_table[b * page_table_stride + j / page_size];
            if (page < 0) continue;
            tok.push_back(j);
            pg.push_back(page);
          }
          if (tok.empty()) {
            m_out[slot] = -std::numeric_limits<double>::infinity();
            l_out[slot] = 0.0;
            continue;
          }
          std::vector<double> x(tok.size());
          double x_max = -std::numeric_limits<double>::infinity();
          for (size_t t = 0; t < tok.size(); ++t) {
            const int32_t off = static_cast<int32_t>(tok[t] % page_size);
            double dot = 0.0;
            for (int32_t c = 0; c < head_dim; ++c) {
              dot += bf16_bits_to_double(qrow[c]) *
                     kv_element(k_cache, k_scale, kv_dtype, pg[t], kv_head, off, c,
                                num_kv_heads, page_size, head_dim);
            }
            x[t] = sm_scale * dot;
            if (x[t] > x_max) x_max = x[t];
          }
          double l = 0.0;
          for (size_t t = 0; t < tok.size(); ++t) {
            const int32_t off = static_cast<int32_t>(tok[t] % page_size);
            const double w = std::exp(x[t] - x_max);
            l += w;
            for (int32_t c = 0; c < head_dim; ++c) {
              acc[c] += w * kv_element(v_cache, v_scale, kv_dtype, pg[t], kv_head, off, c,
                                       num_kv_heads, page_size, head_dim);
            }
          }
          m_out[slot] = x_max;
          l_out[slot] = l;
        }
      }
    }
  }
  return 0;
}

// Log-sum-exp combination of split partials (the reducer):
//   M = max_s m_s,  L = sum_s l_s exp(m_s - M)
//   out = sum_s acc_s exp(m_s - M) / L,  lse = M + ln L
// Splits with m_s = -inf contribute nothing; if every split is empty, out = 0 and
// lse = -inf.
int oracle_combine_splits(const double* m_in, const double* l_in, const double* acc_in,
                          int32_t bs, int32_t num_q_heads, int32_t head_dim,
                          int32_t num_splits, double* out, double* lse) {
  const double neg_inf = -std::numeric_limits<double>::infinity();
  for (int64_t bh = 0; bh < static_cast<int64_t>(bs) * num_q_heads; ++bh) {
    double* orow = out + bh * head_dim;
    for (int32_t c = 0; c < head_dim; ++c) orow[c] = 0.0;
    double m_max = neg_inf;
    for (int32_t s = 0; s < num_splits; ++s) {
      const double m = m_in[bh * num_splits + s];
      if (m > m_max) m_max = m;
    }
    if (m_max == neg_inf) {
      lse[bh] = neg_inf;
      continue;
    }
    double total = 0.0;
    for (int32_t s = 0; s < num_splits; ++s) {
      const double m = m_in[bh * num_splits + s];
      if (m == neg_inf) continue;
      const double w = std::exp(m - m_max);
      total += l_in[bh * num_splits + s] * w;
      const double* acc = acc_in + (bh * num_splits + s) * head_dim;
      for (int32_t c = 0; c < head_dim; ++c) orow[c] += acc[c] * w;
    }
    for (int32_t c = 0; c < head_dim; ++c) orow[c] /= total;
    lse[bh] = m_max + std::log(total);
  }
  return 0;
}

}  // extern "C"
