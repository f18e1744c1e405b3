// Host packing planners: order-preserving next-fit and best-fit-decreasing.
//
// "Packing与 FlashAttention Varlen", section 2: packing only decides which whole
// samples share a pack (the samples stay independent sequences); `sequential`
// is order-preserving next-fit and the default `binpack` is best-fit-decreasing.
// "Pack sequences without joining their contexts", "Fill only the current row":
// a new row starts when an example does not fit the room left; oversize
// examples fail, never split; an exact fill opens no extra row.
#include <algorithm>
#include <numeric>
#include <set>
#include <utility>
#include <vector>

#include "varlen_attn.h"

namespace va {
void set_error(const char* msg);
}

namespace {

va_status check(const int32_t* lengths, int32_t n, int32_t capacity, int32_t* order,
                int32_t* offsets, int32_t* n_packs) {
  if (n < 0 || capacity <= 0 || !n_packs || (n > 0 && (!lengths || !order || !offsets)) ||
      (n == 0 && !offsets)) {
    va::set_error("planner: null pointer or bad size");
    return VA_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n; ++i) {
    if (lengths[i] <= 0) {
      va::set_error("planner: document length must be positive");
      return VA_ERR_INVALID_ARG;
    }
    if (lengths[i] > capacity) {
      va::set_error("planner: document longer than the pack capacity (never split)");
      return VA_ERR_CAPACITY;
    }
  }
  return VA_OK;
}

}  // namespace

extern "C" va_status varlen_pack_next_fit(const int32_t* lengths, int32_t n, int32_t capacity,
                                          int32_t* order, int32_t* offsets, int32_t* n_packs) {
  va_status st = check(lengths, n, capacity, order, offsets, n_packs);
  if (st != VA_OK) return st;
  int32_t packs = 0;
  int64_t used = 0;
  offsets[0] = 0;
  for (int32_t i = 0; i < n; ++i) {
    // a document opens a new pack when it does not fit the room left
    if (i > 0 && lengths[i] > capacity - used) {
      offsets[++packs] = i;
      used = 0;
    }
    order[i] = i;
    used += lengths[i];
  }
  if (n > 0) offsets[++packs] = n;
  *n_packs = packs;
  return VA_OK;
}

extern "C" va_status varlen_pack_best_fit_decreasing(const int32_t* lengths, int32_t n,
                                                     int32_t capacity, int32_t* order,
                                                     int32_t* offsets, int32_t* n_packs) {
  va_status st = check(lengths, n, capacity, order, offsets, n_packs);
  if (st != VA_OK) return st;
  std::vector<int32_t> idx(n);
  std::iota(idx.begin(), idx.end(), 0);
  std::stable_sort(idx.begin(), idx.end(),
                   [&](int32_t a, int32_t b) { return lengths[a] > lengths[b]; });
  // open packs keyed by (room left, opening index): lower_bound({L, 0}) is the
  // pack with the least room >= L, ties to the earliest opened.
  std::set<std::pair<int32_t, int32_t>> open;
  std::vector<int32_t> room;
  std::vector<std::vector<int32_t>> members;
  for (int32_t i : idx) {
    const int32_t L = lengths[i];
    auto it = open.lower_bound({L, 0});
    if (it == open.end()) {
      room.push_back(capacity - L);
      members.push_back({i});
      open.insert({capacity - L, static_cast<int32_t>(room.size()) - 1});
    } else {
      const int32_t p = it->second;
      open.erase(it);
      room[p] -= L;
      members[p].push_back(i);
      open.insert({room[p], p});
    }
  }
  int32_t k = 0;
  offsets[0] = 0;
  for (size_t p = 0; p < members.size(); ++p) {
    for (int32_t i : members[p]) order[k++] = i;
    offsets[p + 1] = k;
  }
  *n_packs = static_cast<int32_t>(members.size());
  return VA_OK;
}
