// lt_oracle.cpp -- CPU oracle for the indexer top-k (Lightning TopK) and its
// two-level, candidate-restricted variant.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the library under
// sparse_attention_indexer_lt_gb300/ links, loads or calls this file; only the
// tests, the smoke check in __graft_entry__.py and the CPU-baseline leg of
// bench.py do. It shares no code, header, table or helper with the CUDA path.
//
// What it computes (plain definitions, written out; no blocking or reordering):
//
//   * Per-row top-k. "CSA: 4:1 compression + TopK selection" (AICon 2026
//     Shenzhen speaker page, aicon.infoq.cn, abstract and outline section 1.1)
//     and "LightningTopK" (SGLang DeepSeek-V4 inference talk notes,
//     devpress.csdn.net, section 3.2) select, for one query row of indexer
//     scores, the k highest-scoring compressed positions. The pages give no
//     tie rule and no output order; this oracle takes the plainest reading:
//     order positions i in [0, L) by score descending, ties by index
//     ascending (a stable sort of the index-ordered row), keep the first
//     min(k, L), pad the rest with (-1, -inf). Under that rule the answer is
//     unique.
//
//   * Two-level selection. In the cross-layer sharing of DeepSeek-V4.1 one
//     layer picks at most 2048 candidate blocks of eight positions and the
//     later indexer-source layers take their top-512 only among the positions
//     of those blocks (SGLang and Miles day-0 support for DeepSeek-V4.1,
//     xhh.club, Q&A on cross-layer sharing). Literal steps, in the order the
//     page gives them: (1) block score = max of the block's valid scores;
//     (2) stable-sort blocks by block score descending, keep the first
//     min(k_blocks, nblocks) (ties: lowest block index); (3) gather the
//     valid positions of the kept blocks in ascending index order; (4) stable
//     sort those by score descending, keep min(k, ncand).
//
//   * Candidate-restricted selection with the candidates given (the later
//     layers' side of that sharing, where the block list arrives from the
//     earlier layer). The pages say nothing about the list's form; reading:
//     block ids outside [0, nblocks) are ignored (-1 pads a short list),
//     repeated ids count once, the list's order does not matter. Steps (3)
//     and (4) above on the listed blocks.
//
// Float order (the pages are silent; the reading taken here):
// IEEE order on numbers, so -0.0 == +0.0 and +-inf are ordinary extremes;
// denormals compare as themselves; NaN ranks below every number (below -inf)
// and NaNs tie with each other. The comparator below uses float compares,
// never an integer re-encoding of the float, so it is independent of the key
// transform the GPU uses.
//
// Parity pins: every function here is pinned by tests under tests/ against
// brute force (Python sorted over tuples, numpy lexsort), library routines
// (numpy sort, torch.topk values, argmax), invariants and special cases.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// a ranks strictly above b by score alone (index ignored).
inline bool score_above(float a, float b) {
  const bool a_nan = std::isnan(a);
  const bool b_nan = std::isnan(b);
  if (a_nan) return false;  // NaN is never above anything
  if (b_nan) return true;   // any number is above NaN
  return a > b;             // IEEE compare: -0 == +0
}

inline int64_t row_length(const int32_t* lengths, int64_t r, int64_t row_stride) {
  if (lengths == nullptr) return row_stride;
  int64_t L = lengths[r];
  if (L < 0) L = 0;
  if (L > row_stride) L = row_stride;
  return L;
}

// Stable sort of the given positions by score descending; ties keep the
// incoming (ascending-index) order.
void stable_sort_desc(const float* s, std::vector<int64_t>& pos) {
  std::stable_sort(pos.begin(), pos.end(),
                   [s](int64_t a, int64_t b) { return score_above(s[a], s[b]); });
}

void write_row(const float* s, const std::vector<int64_t>& picked, int64_t k,
               int32_t* out_idx, float* out_val) {
  const int64_t n = std::min<int64_t>(k, (int64_t)picked.size());
  for (int64_t j = 0; j < n; ++j) {
    out_idx[j] = (int32_t)picked[j];
    if (out_val) std::memcpy(&out_val[j], &s[picked[j]], sizeof(float));  // copy bits
  }
  for (int64_t j = n; j < k; ++j) {
    out_idx[j] = -1;
    if (out_val) out_val[j] = -std::numeric_limits<float>::infinity();
  }
}

void topk_row(const float* s, int64_t L, int64_t k, int32_t* out_idx, float* out_val) {
  std::vector<int64_t> pos(L);
  for (int64_t i = 0; i < L; ++i) pos[i] = i;
  stable_sort_desc(s, pos);
  write_row(s, pos, k, out_idx, out_val);
}

void blocked_row(const float* s, int64_t L, int64_t B, int64_t k_blocks, int64_t k,
                 int32_t* out_idx, float* out_val, int32_t* out_blocks) {
  // (1) block score: max over the block's valid positions, in the float order.
  const int64_t nb = (L + B - 1) / B;
  std::vector<float> bs(nb);
  for (int64_t j = 0; j < nb; ++j) {
    float m = s[j * B];
    for (int64_t i = j * B + 1; i < std::min(L, (j + 1) * B); ++i)
      if (score_above(s[i], m)) m = s[i];
    bs[j] = m;
  }
  // (2) stable sort of block ids by block score descending; keep the first.
  std::vector<int64_t> blocks(nb);
  for (int64_t j = 0; j < nb; ++j) blocks[j] = j;
  stable_sort_desc(bs.data(), blocks);
  const int64_t kept = std::min<int64_t>(k_blocks, nb);
  blocks.resize(kept);
  std::sort(blocks.begin(), blocks.end());  // ascending block ids
  if (out_blocks) {
    for (int64_t j = 0; j < k_blocks; ++j) out_blocks[j] = j < kept ? (int32_t)blocks[j] : -1;
  }
  // (3) valid positions of the kept blocks, ascending.
  std::vector<int64_t> cand;
  cand.reserve(kept * B);
  for (int64_t b : blocks)
    for (int64_t i = b * B; i < std::min(L, (b + 1) * B); ++i) cand.push_back(i);
  // (4) stable sort by score descending; keep the first min(k, ncand).
  stable_sort_desc(s, cand);
  write_row(s, cand, k, out_idx, out_val);
}

void candidates_row(const float* s, int64_t L, int64_t B, const int32_t* listed, int64_t n_listed,
                    int64_t k, int32_t* out_idx, float* out_val) {
  // the listed blocks that hold valid positions, each once, ascending
  const int64_t nb = (L + B - 1) / B;
  std::vector<int64_t> blocks;
  blocks.reserve(n_listed);
  for (int64_t j = 0; j < n_listed; ++j)
    if (listed[j] >= 0 && listed[j] < nb) blocks.push_back(listed[j]);
  std::sort(blocks.begin(), blocks.end());
  blocks.erase(std::unique(blocks.begin(), blocks.end()), blocks.end());
  // (3) their valid positions, ascending; (4) stable sort by score descending
  std::vector<int64_t> cand;
  cand.reserve(blocks.size() * B);
  for (int64_t b : blocks)
    for (int64_t i = b * B; i < std::min(L, (b + 1) * B); ++i) cand.push_back(i);
  stable_sort_desc(s, cand);
  write_row(s, cand, k, out_idx, out_val);
}

template <class F>
void parallel_rows(int64_t rows, int32_t nthreads, F f) {
  if (nthreads <= 1 || rows <= 1) {
    for (int64_t r = 0; r < rows; ++r) f(r);
    return;
  }
  const int64_t nt = std::min<int64_t>(nthreads, rows);
  std::vector<std::thread> pool;
  pool.reserve(nt);
  for (int64_t t = 0; t < nt; ++t)
    pool.emplace_back([=]() {
      for (int64_t r = t; r < rows; r += nt) f(r);
    });
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Returns 0 on success, 1 on an invalid argument. All pointers are host memory.
int lt_oracle_topk(const float* scores, const int32_t* lengths, int64_t rows,
                   int64_t row_stride, int64_t k, int32_t* out_idx, float* out_val,
                   int32_t nthreads) {
  if (rows < 0 || row_stride < 0 || k < 1 || (rows > 0 && (!scores || !out_idx))) return 1;
  parallel_rows(rows, nthreads, [=](int64_t r) {
    topk_row(scores + r * row_stride, row_length(lengths, r, row_stride), k,
             out_idx + r * k, out_val ? out_val + r * k : nullptr);
  });
  return 0;
}

int lt_oracle_topk_blocked(const float* scores, const int32_t* lengths, int64_t rows,
                           int64_t row_stride, int64_t block, int64_t k_blocks, int64_t k,
                           int32_t* out_idx, float* out_val, int32_t* out_blocks,
                           int32_t nthreads) {
  if (rows < 0 || row_stride < 0 || block < 1 || k_blocks < 1 || k < 1 ||
      (rows > 0 && (!scores || !out_idx)))
    return 1;
  parallel_rows(rows, nthreads, [=](int64_t r) {
    blocked_row(scores + r * row_stride, row_length(lengths, r, row_stride), block, k_blocks,
                k, out_idx + r * k, out_val ? out_val + r * k : nullptr,
                out_blocks ? out_blocks + r * k_blocks : nullptr);
  });
  return 0;
}

// cand_blocks: n_cand block ids per row (row-major), host memory.
int lt_oracle_topk_candidates(const float* scores, const int32_t* lengths, int64_t rows,
                              int64_t row_stride, int64_t block, const int32_t* cand_blocks,
                              int64_t n_cand, int64_t k, int32_t* out_idx, float* out_val,
                              int32_t nthreads) {
  if (rows < 0 || row_stride < 0 || block < 1 || n_cand < 0 || k < 1 ||
      (rows > 0 && (!scores || !out_idx || (n_cand > 0 && !cand_blocks))))
    return 1;
  parallel_rows(rows, nthreads, [=](int64_t r) {
    candidates_row(scores + r * row_stride, row_length(lengths, r, row_stride), block,
                   cand_blocks ? cand_blocks + r * n_cand : nullptr, n_cand, k, out_idx + r * k,
                   out_val ? out_val + r * k : nullptr);
  });
  return 0;
}

}  // extern "C"
