// Paged decode attention: the CPU oracle.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
// call this file; only the tests, the smoke check and the benchmark's CPU
// baseline do. It shares no code, header or table with the CUDA library.
//
// What it states, in plain FP64 loops, and where the pages say so:
//
//  * The KV cache is a shared pool of physical pages; each page holds 16
//    tokens of K and V for one layer, and a block table per sequence and
//    layer maps logical page i of a sequence to a physical page id.
//    [samir-vllm: Build LLM Inference From Scratch in C++ and CUDA,
//     "Architecture walkthrough", KV cache paragraph; 6 Hours of YouTube and
//     85 handtyped pages of notes on LLM Inference - Start here, README
//     feature list, shared BF16 KV page pool bullet]
//  * Decode appends one new token's K/V at its absolute position into the
//    slot its block table names (same two passages).
//  * Decode attention reads each sequence's cached pages through the block
//    table, with no contiguous gather; the result it reaches is ordinary
//    softmax attention over the sequence's tokens, grouped-query: each query
//    head reads the K/V head of its group.
//    [6 Hours of YouTube ..., README feature list, direct paged decode
//     attention bullet; samir-vllm: Build LLM Inference ..., "TL;DR" table,
//     Decode and Kernels rows]
//
// Because the online softmax the pages describe reaches exactly (up to
// rounding order) plain softmax attention, this file is that definition
// written out: gather, scores, max-subtracted exponentials, normalised
// weighted sum. It does not restate the streaming algorithm.
//
// Readings where the pages are silent (each is also listed with the design
// notes):
//  * query head h reads KV head h / (Hq / Hkv) (consecutive grouping);
//  * the score scale is 1 / sqrt(head_dim);
//  * seq_lens[b] is the attended length after the append, so the token just
//    appended sits at position seq_lens[b] - 1 and is attended;
//  * page ids are global over one pool shared by every layer; the block
//    table's layer index selects the mapping;
//  * pool layout is [page][kv_head][token-in-page][dim], K and V in separate
//    pools; block tables are [layer][max_batch][max_pages_per_seq] int32;
//  * BF16 values arrive as their 16-bit patterns and are widened exactly.
//
// Rotary position embedding (the pages have the decode step write the new
// token at its absolute rotary position but do not print the rotation). Reading: the
// rotate-half convention of Llama implementations, pairing dim i with
// i + D/2, with the angles supplied as FP32 tables cos_t[p][i], sin_t[p][i]
// (i < D/2) because the pages fix neither the base nor Llama 3.2's scaling:
//   x'[i] = x[i] cos - x[i + D/2] sin,   x'[i + D/2] = x[i + D/2] cos + x[i] sin.
// The appended key is stored in BF16, so its rotation is stated in the
// precision in which that rounding is decided: FP32 products and sum, each
// rounded, no fused multiply-add, then round to nearest even. Queries are not
// stored and are rotated in FP64.
//
// The split variant computes, per contiguous range of logical pages, the
// unnormalised partial (o, m, l) and merges the partials with the
// log-sum-exp rule; it exists so that the merge algebra can be checked in
// FP64 against the unsplit definition.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

extern "C" {

typedef struct {
  int num_layers;
  int num_pages;
  int page_size;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int max_batch;
  int max_pages_per_seq;
} pkv_oracle_geometry;

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_OUT_OF_RANGE = 2 };

}  // extern "C"

namespace {

double bf16_bits_to_double(uint16_t bits) {
  uint32_t word = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &word, sizeof f);
  return static_cast<double>(f);
}

bool geometry_ok(const pkv_oracle_geometry* g) {
  return g && g->num_layers > 0 && g->num_pages > 0 && g->page_size > 0 &&
         g->num_q_heads > 0 && g->num_kv_heads > 0 && g->head_dim > 0 &&
         g->num_q_heads % g->num_kv_heads == 0 && g->max_batch > 0 &&
         g->max_pages_per_seq > 0;
}

size_t pool_index(const pkv_oracle_geometry* g, long page, int kv_head, int slot, int d) {
  return ((static_cast<size_t>(page) * g->num_kv_heads + kv_head) * g->page_size + slot) *
             g->head_dim + d;
}

// Physical page holding logical token t of sequence b in layer l, or -1 when
// the block table names a page outside the pool.
long physical_page(const pkv_oracle_geometry* g, const int32_t* block_tables, int layer, int b,
                   int t) {
  int logical = t / g->page_size;
  if (logical >= g->max_pages_per_seq) return -1;
  size_t at = (static_cast<size_t>(layer) * g->max_batch + b) * g->max_pages_per_seq + logical;
  long page = block_tables[at];
  if (page < 0 || page >= g->num_pages) return -1;
  return page;
}

// Gathered K and V rows of one (sequence, kv head), widened to double:
// rows[t * D + d] for t < len.
bool gather_head(const pkv_oracle_geometry* g, const uint16_t* k_pool, const uint16_t* v_pool,
                 const int32_t* block_tables, int layer, int b, int kv_head, int len,
                 std::vector<double>& k_rows, std::vector<double>& v_rows) {
  const int D = g->head_dim;
  k_rows.assign(static_cast<size_t>(len) * D, 0.0);
  v_rows.assign(static_cast<size_t>(len) * D, 0.0);
  for (int t = 0; t < len; ++t) {
    long page = physical_page(g, block_tables, layer, b, t);
    if (page < 0) return false;
    int slot = t % g->page_size;
    for (int d = 0; d < D; ++d) {
      k_rows[static_cast<size_t>(t) * D + d] =
          bf16_bits_to_double(k_pool[pool_index(g, page, kv_head, slot, d)]);
      v_rows[static_cast<size_t>(t) * D + d] =
          bf16_bits_to_double(v_pool[pool_index(g, page, kv_head, slot, d)]);
    }
  }
  return true;
}

// Softmax attention of one query row over len gathered rows:
//   s_t = (q . K_t) / sqrt(D),  w_t = exp(s_t - max s) / sum_u exp(s_u - max s),
//   out = sum_t w_t V_t.
// Also returns lse = log sum_t exp(s_t) and the sum of the weights.
void attend_row(const double* q, const double* k_rows, const double* v_rows, int len, int D,
                double* out, double* lse, double* wsum) {
  const double scale = 1.0 / std::sqrt(static_cast<double>(D));
  std::vector<double> s(len);
  for (int t = 0; t < len; ++t) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q[d] * k_rows[static_cast<size_t>(t) * D + d];
    s[t] = dot * scale;
  }
  double m = -std::numeric_limits<double>::infinity();
  for (int t = 0; t < len; ++t) m = s[t] > m ? s[t] : m;
  double z = 0.0;
  for (int t = 0; t < len; ++t) z += std::exp(s[t] - m);
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  double total = 0.0;
  for (int t = 0; t < len; ++t) {
    double w = std::exp(s[t] - m) / z;
    total += w;
    for (int d = 0; d < D; ++d) out[d] += w * v_rows[static_cast<size_t>(t) * D + d];
  }
  if (lse) *lse = m + std::log(z);
  if (wsum) *wsum = total;
}

// All query heads of one sequence.
int attend_sequence(const pkv_oracle_geometry* g, int layer, const uint16_t* q,
                    const uint16_t* k_pool, const uint16_t* v_pool, const int32_t* block_tables,
                    const int32_t* seq_lens, int b, double* out, double* lse, double* wsum,
                    const double* q64 = nullptr) {
  const int D = g->head_dim;
  const int group = g->num_q_heads / g->num_kv_heads;
  const int len = seq_lens[b];
  if (len < 1 || len > g->max_pages_per_seq * g->page_size) return ORACLE_OUT_OF_RANGE;
  std::vector<double> k_rows, v_rows, q_row(D);
  for (int kv = 0; kv < g->num_kv_heads; ++kv) {
    if (!gather_head(g, k_pool, v_pool, block_tables, layer, b, kv, len, k_rows, v_rows))
      return ORACLE_OUT_OF_RANGE;
    for (int h = kv * group; h < (kv + 1) * group; ++h) {
      size_t row = static_cast<size_t>(b) * g->num_q_heads + h;
      for (int d = 0; d < D; ++d)
        q_row[d] = q64 ? q64[row * D + d] : bf16_bits_to_double(q[row * D + d]);
      attend_row(q_row.data(), k_rows.data(), v_rows.data(), len, D, out + row * D,
                 lse ? lse + row : nullptr, wsum ? wsum + row : nullptr);
    }
  }
  return ORACLE_OK;
}

float bf16_bits_to_float(uint16_t bits) {
  uint32_t word = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &word, sizeof f);
  return f;
}

// FP32 -> BF16 bit pattern, round to nearest, ties to even (finite inputs).
uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

}  // namespace

extern "C" {

// Decode-time append: for each sequence b and kv head, the new token at
// absolute position positions[b] is written to
//   pool[block_tables[layer][b][pos / P]][kv][pos % P][:].
// k_new, v_new: BF16 bit patterns [batch][Hkv][D]. The pools are modified in
// place. Returns ORACLE_OUT_OF_RANGE (and writes nothing for that sequence)
// when the position or the page id falls outside the pool.
int pkv_oracle_append(const pkv_oracle_geometry* g, int layer, const uint16_t* k_new,
                      const uint16_t* v_new, uint16_t* k_pool, uint16_t* v_pool,
                      const int32_t* block_tables, const int32_t* positions, int batch) {
  if (!geometry_ok(g) || layer < 0 || layer >= g->num_layers || batch < 0 ||
      batch > g->max_batch)
    return ORACLE_BAD_ARG;
  int status = ORACLE_OK;
  const int D = g->head_dim;
  for (int b = 0; b < batch; ++b) {
    int pos = positions[b];
    if (pos < 0 || pos >= g->max_pages_per_seq * g->page_size) {
      status = ORACLE_OUT_OF_RANGE;
      continue;
    }
    long page = physical_page(g, block_tables, layer, b, pos);
    if (page < 0) {
      status = ORACLE_OUT_OF_RANGE;
      continue;
    }
    int slot = pos % g->page_size;
    for (int kv = 0; kv < g->num_kv_heads; ++kv) {
      for (int d = 0; d < D; ++d) {
        size_t src = (static_cast<size_t>(b) * g->num_kv_heads + kv) * D + d;
        k_pool[pool_index(g, page, kv, slot, d)] = k_new[src];
        v_pool[pool_index(g, page, kv, slot, d)] = v_new[src];
      }
    }
  }
  return status;
}

// Decode attention for one layer: out[b][h][:] = softmax attention of query
// head h of sequence b over tokens 0..seq_lens[b]-1 of KV head h / group,
// gathered through the block table. q: BF16 bit patterns [batch][Hq][D].
// out: double [batch][Hq][D]; lse and wsum (optional): double [batch][Hq].
int pkv_oracle_decode_attention(const pkv_oracle_geometry* g, int layer, const uint16_t* q,
                                const uint16_t* k_pool, const uint16_t* v_pool,
                                const int32_t* block_tables, const int32_t* seq_lens, int batch,
                                double* out, double* lse, double* wsum) {
  if (!geometry_ok(g) || layer < 0 || layer >= g->num_layers || batch < 0 ||
      batch > g->max_batch || !out)
    return ORACLE_BAD_ARG;
  int status = ORACLE_OK;
  for (int b = 0; b < batch; ++b) {
    int r = attend_sequence(g, layer, q, k_pool, v_pool, block_tables, seq_lens, b, out, lse,
                            wsum);
    if (r != ORACLE_OK) status = r;
  }
  return status;
}

// The same computation with the sequences shared out over nthreads host
// threads (sequence b goes to thread b % nthreads). Each sequence is
// computed exactly as above; used to time the oracle on all host cores.
int pkv_oracle_decode_attention_mt(const pkv_oracle_geometry* g, int layer, const uint16_t* q,
                                   const uint16_t* k_pool, const uint16_t* v_pool,
                                   const int32_t* block_tables, const int32_t* seq_lens,
                                   int batch, double* out, int nthreads) {
  if (!geometry_ok(g) || layer < 0 || layer >= g->num_layers || batch < 0 ||
      batch > g->max_batch || !out || nthreads < 1)
    return ORACLE_BAD_ARG;
  std::vector<int> status(nthreads, ORACLE_OK);
  std::vector<std::thread> pool;
  for (int w = 0; w < nthreads; ++w) {
    pool.emplace_back([&, w]() {
      for (int b = w; b < batch; b += nthreads) {
        int r = attend_sequence(g, layer, q, k_pool, v_pool, block_tables, seq_lens, b, out,
                                nullptr, nullptr);
        if (r != ORACLE_OK) status[w] = r;
      }
    });
  }
  for (auto& th : pool) th.join();
  for (int s : status)
    if (s != ORACLE_OK) return s;
  return ORACLE_OK;
}

// Split-KV statement of the same attention. For sequence b with
// np = ceil(len / P) logical pages and S splits, split s covers logical pages
// [s * C, min(np, (s + 1) * C)) with C = ceil(np / S). Per split and head:
//   m_s = max of its scores, l_s = sum exp(s_t - m_s),
//   o_s = sum exp(s_t - m_s) V_t        (unnormalised);
// an empty split has m_s = -inf, l_s = 0, o_s = 0. The merge is
//   M = max_s m_s,  out = sum_s exp(m_s - M) o_s / sum_s exp(m_s - M) l_s.
// part_o [batch][Hq][S][D], part_m and part_l [batch][Hq][S] are optional.
int pkv_oracle_decode_attention_split(const pkv_oracle_geometry* g, int layer,
                                      const uint16_t* q, const uint16_t* k_pool,
                                      const uint16_t* v_pool, const int32_t* block_tables,
                                      const int32_t* seq_lens, int batch, int num_splits,
                                      double* out, double* part_o, double* part_m,
                                      double* part_l) {
  if (!geometry_ok(g) || layer < 0 || layer >= g->num_layers || batch < 0 ||
      batch > g->max_batch || !out || num_splits < 1)
    return ORACLE_BAD_ARG;
  const int D = g->head_dim;
  const int P = g->page_size;
  const int S = num_splits;
  const int group = g->num_q_heads / g->num_kv_heads;
  const double scale = 1.0 / std::sqrt(static_cast<double>(D));
  const double neg_inf = -std::numeric_limits<double>::infinity();
  int status = ORACLE_OK;
  std::vector<double> k_rows, v_rows, q_row(D), o(static_cast<size_t>(S) * D), m(S), l(S);
  for (int b = 0; b < batch; ++b) {
    const int len = seq_lens[b];
    if (len < 1 || len > g->max_pages_per_seq * P) {
      status = ORACLE_OUT_OF_RANGE;
      continue;
    }
    const int np = (len + P - 1) / P;
    const int chunk = (np + S - 1) / S;
    for (int kv = 0; kv < g->num_kv_heads; ++kv) {
      if (!gather_head(g, k_pool, v_pool, block_tables, layer, b, kv, len, k_rows, v_rows)) {
        status = ORACLE_OUT_OF_RANGE;
        continue;
      }
      for (int h = kv * group; h < (kv + 1) * group; ++h) {
        size_t row = static_cast<size_t>(b) * g->num_q_heads + h;
        for (int d = 0; d < D; ++d) q_row[d] = bf16_bits_to_double(q[row * D + d]);
        for (int s = 0; s < S; ++s) {
          int t0 = s * chunk * P;
          int t1 = (s + 1) * chunk * P;
          if (t1 > len) t1 = len;
          m[s] = neg_inf;
          l[s] = 0.0;
          for (int d = 0; d < D; ++d) o[static_cast<size_t>(s) * D + d] = 0.0;
          std::vector<double> sc;
          for (int t = t0; t < t1; ++t) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += q_row[d] * k_rows[static_cast<size_t>(t) * D + d];
            sc.push_back(dot * scale);
            if (sc.back() > m[s]) m[s] = sc.back();
          }
          for (int t = t0; t < t1; ++t) {
            double e = std::exp(sc[t - t0] - m[s]);
            l[s] += e;
            for (int d = 0; d < D; ++d)
              o[static_cast<size_t>(s) * D + d] += e * v_rows[static_cast<size_t>(t) * D + d];
          }
          if (part_m) part_m[row * S + s] = m[s];
          if (part_l) part_l[row * S + s] = l[s];
          if (part_o)
            for (int d = 0; d < D; ++d)
              part_o[(row * S + s) * D + d] = o[static_cast<size_t>(s) * D + d];
        }
        double big = neg_inf;
        for (int s = 0; s < S; ++s) big = m[s] > big ? m[s] : big;
        double denom = 0.0;
        for (int s = 0; s < S; ++s)
          if (l[s] > 0.0) denom += std::exp(m[s] - big) * l[s];
        for (int d = 0; d < D; ++d) {
          double num = 0.0;
          for (int s = 0; s < S; ++s)
            if (l[s] > 0.0) num += std::exp(m[s] - big) * o[static_cast<size_t>(s) * D + d];
          out[row * D + d] = num / denom;
        }
      }
    }
  }
  return status;
}

// Softmax attention of one sequence over a CONTIGUOUS cache (no pages):
// q [Hq][D], k and v [len][Hkv][D] (BF16 bit patterns), out double [Hq][D].
// Used to check that the paged gather reaches the same result.
int pkv_oracle_contiguous_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    int len, int num_q_heads, int num_kv_heads, int head_dim,
                                    double* out) {
  if (len < 1 || num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads || !out)
    return ORACLE_BAD_ARG;
  const int D = head_dim;
  const int group = num_q_heads / num_kv_heads;
  std::vector<double> k_rows(static_cast<size_t>(len) * D), v_rows(k_rows.size()), q_row(D);
  for (int kv = 0; kv < num_kv_heads; ++kv) {
    for (int t = 0; t < len; ++t)
      for (int d = 0; d < D; ++d) {
        size_t src = (static_cast<size_t>(t) * num_kv_heads + kv) * D + d;
        k_rows[static_cast<size_t>(t) * D + d] = bf16_bits_to_double(k[src]);
        v_rows[static_cast<size_t>(t) * D + d] = bf16_bits_to_double(v[src]);
      }
    for (int h = kv * group; h < (kv + 1) * group; ++h) {
      for (int d = 0; d < D; ++d) q_row[d] = bf16_bits_to_double(q[static_cast<size_t>(h) * D + d]);
      attend_row(q_row.data(), k_rows.data(), v_rows.data(), len, D,
                 out + static_cast<size_t>(h) * D, nullptr, nullptr);
    }
  }
  return ORACLE_OK;
}

}  // extern "C"

extern "C" {

// Decode-time append with the key rotated to its position first: as
// pkv_oracle_append, with k_new[b][kv] rotated by the angles of position
// positions[b] (tables cos_t, sin_t: FP32 [table_len][D/2]) in the FP32
// statement above, then rounded to BF16. V is copied unchanged.
int pkv_oracle_append_rope(const pkv_oracle_geometry* g, int layer, const uint16_t* k_new,
                           const uint16_t* v_new, uint16_t* k_pool, uint16_t* v_pool,
                           const int32_t* block_tables, const int32_t* positions, int batch,
                           const float* cos_t, const float* sin_t, int table_len) {
  if (!geometry_ok(g) || g->head_dim % 2 != 0 || !cos_t || !sin_t || batch < 0 ||
      batch > g->max_batch)
    return ORACLE_BAD_ARG;
  const int D = g->head_dim;
  const int half = D / 2;
  std::vector<uint16_t> rotated(static_cast<size_t>(batch) * g->num_kv_heads * D);
  for (int b = 0; b < batch; ++b) {
    const int pos = positions[b];
    for (int kv = 0; kv < g->num_kv_heads; ++kv) {
      const size_t row = (static_cast<size_t>(b) * g->num_kv_heads + kv) * D;
      for (int i = 0; i < D; ++i) rotated[row + i] = k_new[row + i];
      if (pos < 0 || pos >= table_len) continue;   // the append reports the range error
      for (int i = 0; i < half; ++i) {
        const float c = cos_t[static_cast<size_t>(pos) * half + i];
        const float s = sin_t[static_cast<size_t>(pos) * half + i];
        const float x = bf16_bits_to_float(k_new[row + i]);
        const float y = bf16_bits_to_float(k_new[row + i + half]);
        const float xc = x * c, ys = y * s, yc = y * c, xs = x * s;
        rotated[row + i] = float_to_bf16_rne(xc - ys);
        rotated[row + i + half] = float_to_bf16_rne(yc + xs);
      }
    }
  }
  return pkv_oracle_append(g, layer, rotated.data(), v_new, k_pool, v_pool, block_tables,
                           positions, batch);
}

// Queries rotated to their positions, in double: q [batch][Hq][D] BF16 bit
// patterns -> q_out double [batch][Hq][D].
int pkv_oracle_rope_queries(const uint16_t* q, int batch, int num_q_heads, int head_dim,
                            const int32_t* positions, const float* cos_t, const float* sin_t,
                            int table_len, double* q_out) {
  if (!q || !q_out || !cos_t || !sin_t || head_dim % 2 != 0 || batch < 0) return ORACLE_BAD_ARG;
  const int half = head_dim / 2;
  int status = ORACLE_OK;
  for (int b = 0; b < batch; ++b) {
    const int pos = positions[b];
    for (int h = 0; h < num_q_heads; ++h) {
      const size_t row = (static_cast<size_t>(b) * num_q_heads + h) * head_dim;
      for (int i = 0; i < head_dim; ++i) q_out[row + i] = bf16_bits_to_double(q[row + i]);
      if (pos < 0 || pos >= table_len) {
        status = ORACLE_OUT_OF_RANGE;
        continue;
      }
      for (int i = 0; i < half; ++i) {
        const double c = cos_t[static_cast<size_t>(pos) * half + i];
        const double s = sin_t[static_cast<size_t>(pos) * half + i];
        const double x = bf16_bits_to_double(q[row + i]);
        const double y = bf16_bits_to_double(q[row + i + half]);
        q_out[row + i] = x * c - y * s;
        q_out[row + i + half] = y * c + x * s;
      }
    }
  }
  return status;
}

// pkv_oracle_decode_attention with the queries given in double (q64
// [batch][Hq][D]), e.g. after the rotation above.
int pkv_oracle_decode_attention_q64(const pkv_oracle_geometry* g, int layer, const double* q64,
                                    const uint16_t* k_pool, const uint16_t* v_pool,
                                    const int32_t* block_tables, const int32_t* seq_lens,
                                    int batch, double* out) {
  if (!geometry_ok(g) || layer < 0 || layer >= g->num_layers || batch < 0 ||
      batch > g->max_batch || !out || !q64)
    return ORACLE_BAD_ARG;
  int status = ORACLE_OK;
  for (int b = 0; b < batch; ++b) {
    int r = attend_sequence(g, layer, nullptr, k_pool, v_pool, block_tables, seq_lens, b, out,
                            nullptr, nullptr, q64);
    if (r != ORACLE_OK) status = r;
  }
  return status;
}

}  // extern "C"

// ---------------------------------------------------------------- prefill
// Prefill over pages [samir-vllm: Build LLM Inference From Scratch in C++ and
// CUDA, "Architecture walkthrough", Prefill and KV cache paragraphs; 6 Hours
// of YouTube and 85 handtyped pages of notes on LLM Inference - Start here,
// README feature list, dense causal prefill and shared BF16 KV page pool
// bullets]: prefill fills the prompt's pages with its K/V, and each prompt
// token attends causally to every token up to and including itself.
//
// Readings: a call carries, for each sequence b, a chunk of n_b tokens packed
// at rows cu_tokens[b] .. cu_tokens[b+1] - 1 of q/k/v, at absolute positions
// start_pos[b] .. start_pos[b] + n_b - 1 (start_pos > 0 continues a prompt
// whose earlier tokens are already in the pages: chunked prefill); the fill
// is the decode append applied to every token of the chunk; token i of the
// chunk attends to keys 0 .. start_pos[b] + i, read through the block table
// (so the fill of the same chunk comes first).
extern "C" {

int pkv_oracle_prefill_fill(const pkv_oracle_geometry* g, int layer, const uint16_t* k,
                            const uint16_t* v, uint16_t* k_pool, uint16_t* v_pool,
                            const int32_t* block_tables, const int32_t* cu_tokens,
                            const int32_t* start_pos, int batch) {
  if (!geometry_ok(g) || layer < 0 || layer >= g->num_layers || batch < 0 ||
      batch > g->max_batch || !k || !v || !k_pool || !v_pool || !cu_tokens || !start_pos)
    return ORACLE_BAD_ARG;
  const int D = g->head_dim;
  int status = ORACLE_OK;
  for (int b = 0; b < batch; ++b) {
    for (int row = cu_tokens[b]; row < cu_tokens[b + 1]; ++row) {
      const int pos = start_pos[b] + (row - cu_tokens[b]);
      const long page = pos < 0 ? -1 : physical_page(g, block_tables, layer, b, pos);
      if (page < 0) {
        status = ORACLE_OUT_OF_RANGE;
        continue;
      }
      for (int h = 0; h < g->num_kv_heads; ++h)
        for (int d = 0; d < D; ++d) {
          const size_t src = (static_cast<size_t>(row) * g->num_kv_heads + h) * D + d;
          k_pool[pool_index(g, page, h, pos % g->page_size, d)] = k[src];
          v_pool[pool_index(g, page, h, pos % g->page_size, d)] = v[src];
        }
    }
  }
  return status;
}

// Causal attention of every chunk token over the pages: out [total][Hq][D]
// (double), total = cu_tokens[batch]. (sequence, kv head) pairs are spread
// over `nthreads` host threads; each output row is computed the same way
// whatever the thread count.
int pkv_oracle_prefill_attention(const pkv_oracle_geometry* g, int layer, const uint16_t* q,
                                 const uint16_t* k_pool, const uint16_t* v_pool,
                                 const int32_t* block_tables, const int32_t* cu_tokens,
                                 const int32_t* start_pos, int batch, double* out,
                                 int nthreads) {
  if (!geometry_ok(g) || layer < 0 || layer >= g->num_layers || batch < 0 ||
      batch > g->max_batch || !q || !k_pool || !v_pool || !cu_tokens || !start_pos || !out)
    return ORACLE_BAD_ARG;
  const int D = g->head_dim;
  const int Hq = g->num_q_heads;
  const int group = Hq / g->num_kv_heads;
  const int units = batch * g->num_kv_heads;
  if (nthreads < 1) nthreads = 1;
  std::vector<int> status(static_cast<size_t>(nthreads), ORACLE_OK);
  auto work = [&](int w) {
    std::vector<double> k_rows, v_rows, q_row(D);
    for (int u = w; u < units; u += nthreads) {
      const int b = u / g->num_kv_heads;
      const int kv = u % g->num_kv_heads;
      const int n = cu_tokens[b + 1] - cu_tokens[b];
      if (n == 0) continue;
      const int len = start_pos[b] + n;          // keys the last token sees
      if (start_pos[b] < 0 ||
          !gather_head(g, k_pool, v_pool, block_tables, layer, b, kv, len, k_rows, v_rows)) {
        status[w] = ORACLE_OUT_OF_RANGE;
        continue;
      }
      for (int i = 0; i < n; ++i) {
        const size_t row = static_cast<size_t>(cu_tokens[b] + i);
        for (int h = kv * group; h < (kv + 1) * group; ++h) {
          for (int d = 0; d < D; ++d) q_row[d] = bf16_bits_to_double(q[(row * Hq + h) * D + d]);
          attend_row(q_row.data(), k_rows.data(), v_rows.data(), start_pos[b] + i + 1, D,
                     out + (row * Hq + h) * D, nullptr, nullptr);
        }
      }
    }
  };
  if (nthreads == 1) {
    work(0);
  } else {
    std::vector<std::thread> pool;
    for (int w = 0; w < nthreads; ++w) pool.emplace_back(work, w);
    for (auto& t : pool) t.join();
  }
  for (int s : status)
    if (s != ORACLE_OK) return s;
  return ORACLE_OK;
}

}  // extern "C"
