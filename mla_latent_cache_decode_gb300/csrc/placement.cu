// KV-load-aware placement of requests on data-parallel attention ranks (host
// code only; see mla_place_requests in mla.h).
//
// Longest request first, each to the least loaded rank that can still hold
// it: list scheduling in decreasing order (Graham 1969), the load being the
// cached tokens a rank's decodes read [dp-attention-expert-parallel-mla-kv-
// replication (inferenceinterviews.com), "What it costs"].  The least loaded
// rank is kept in a binary min-heap on (load, rank).
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "mla.h"

namespace mla {
void set_error_detail(const char *msg);
}

namespace {

struct RankHeap {
  // (load, rank) pairs; the smallest on top, ties to the lower rank
  std::vector<std::pair<int64_t, int32_t>> h;
  static bool after(const std::pair<int64_t, int32_t> &a, const std::pair<int64_t, int32_t> &b) {
    return a.first != b.first ? a.first > b.first : a.second > b.second;
  }
  void push(int64_t load, int32_t rank) {
    h.emplace_back(load, rank);
    std::push_heap(h.begin(), h.end(), after);
  }
  std::pair<int64_t, int32_t> top() const { return h.front(); }
  void replace_top(int64_t load) {
    std::pop_heap(h.begin(), h.end(), after);
    h.back().first = load;
    std::push_heap(h.begin(), h.end(), after);
  }
};

bool fits(int64_t load, int64_t tokens, int64_t capacity) {
  return capacity == 0 || tokens <= capacity - load;
}

}  // namespace

extern "C" {

mla_status_t mla_place_requests(const int64_t *kv_tokens, int32_t n, int32_t ranks,
                                int64_t capacity_tokens, int32_t *rank_of, int64_t *rank_load,
                                int32_t *unplaced) {
  mla::set_error_detail("");
  if (n < 0 || ranks < 1 || capacity_tokens < 0 || !rank_load ||
      (n > 0 && (!kv_tokens || !rank_of))) {
    mla::set_error_detail("n < 0, ranks < 1, capacity < 0 or a null array");
    return MLA_ERR_INVALID_ARGUMENT;
  }
  for (int32_t i = 0; i < n; ++i)
    if (kv_tokens[i] < 0) {
      mla::set_error_detail("negative kv_tokens");
      return MLA_ERR_INVALID_ARGUMENT;
    }
  std::vector<int32_t> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return kv_tokens[a] > kv_tokens[b]; });
  RankHeap heap;
  heap.h.reserve(ranks);
  for (int32_t r = 0; r < ranks; ++r) heap.push(0, r);
  std::vector<int64_t> load(ranks, 0);
  int32_t left = 0;
  for (int32_t i : order) {
    const auto least = heap.top();
    if (!fits(least.first, kv_tokens[i], capacity_tokens)) {
      rank_of[i] = -1;
      ++left;
      continue;
    }
    rank_of[i] = least.second;
    load[least.second] = least.first + kv_tokens[i];
    heap.replace_top(load[least.second]);
  }
  std::copy(load.begin(), load.end(), rank_load);
  if (unplaced) *unplaced = left;
  return MLA_OK;
}

mla_status_t mla_place_one(const int64_t *rank_load, int32_t ranks, int64_t capacity_tokens,
                           int64_t kv_tokens, int32_t *rank) {
  mla::set_error_detail("");
  if (ranks < 1 || !rank_load || !rank || capacity_tokens < 0 || kv_tokens < 0) {
    mla::set_error_detail("ranks < 1, a null pointer, or a negative length or capacity");
    return MLA_ERR_INVALID_ARGUMENT;
  }
  int32_t best = 0;
  for (int32_t r = 0; r < ranks; ++r) {
    if (rank_load[r] < 0) {
      mla::set_error_detail("negative rank load");
      return MLA_ERR_INVALID_ARGUMENT;
    }
    if (rank_load[r] < rank_load[best]) best = r;
  }
  *rank = fits(rank_load[best], kv_tokens, capacity_tokens) ? best : -1;
  return MLA_OK;
}

}  // extern "C"
