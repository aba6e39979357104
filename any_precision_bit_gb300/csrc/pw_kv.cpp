// pw_kv.cpp -- KV-block allocator sharing the device budget with the weight pages (host).
//
// PagedWeight Sec. 3.3 (asynchronous page movement): the planner follows the free KV
// blocks, the allocator headroom and the pending KV growth, and the GPU pages an offload
// retires become headroom the KV blocks can take.  Sec. 3.2, Eq. 7: the free-block count
// F_blk against the reserve T_blk sets the bytes the planner must release.  Here one budget
// S holds the weight pages (W bytes) and the KV blocks (B bytes each):
//   C = floor(max(0, S - W) / B),  F_blk = C - U - P,  headroom = S - W - U B,
// with U the blocks held and P the blocks announced as pending growth.  A grow draws on the
// request's own announcement first and must otherwise fit in F_blk; it is all or nothing.
// Ids are logical and the lowest free one is granted first: ids below the high-water mark
// that were released are kept in an ordered set, so memory grows with the ids in use, not
// with the budget.
#include <stdint.h>

#include <iterator>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "../../include/pw.h"

struct pw_kv {
  int64_t S = 0, B = 0, W = 0;
  int64_t n_ids = 0;
  pw_ctx *ctx = nullptr;  // W is read from here when set
  int64_t U = 0, P = 0;
  int32_t next_id = 0;              // ids >= next_id were never granted
  std::set<int32_t> freed;          // released ids below next_id
  std::unordered_map<int64_t, std::vector<int32_t>> held;
  std::unordered_map<int64_t, int64_t> announced;
};

namespace {

pw_status refresh_weights(pw_kv *kv) {
  if (!kv->ctx) return PW_OK;
  pw_mem_info mi;
  if (pw_status st = pw_memory(kv->ctx, &mi)) return st;
  kv->W = mi.held_bytes;
  return PW_OK;
}

int64_t capacity(const pw_kv *kv) { return kv->S > kv->W ? (kv->S - kv->W) / kv->B : 0; }

int32_t take_lowest(pw_kv *kv) {
  if (!kv->freed.empty()) {
    const int32_t id = *kv->freed.begin();
    kv->freed.erase(kv->freed.begin());
    return id;
  }
  return kv->next_id++;
}

}  // namespace

extern "C" pw_status pw_kv_create(int64_t budget_bytes, int64_t block_bytes, pw_kv **out) {
  if (!out || budget_bytes < 0 || block_bytes <= 0 || budget_bytes / block_bytes >= (int64_t(1) << 31))
    return PW_ERR_INVALID;
  pw_kv *kv = new (std::nothrow) pw_kv;
  if (!kv) return PW_ERR_OOM;
  kv->S = budget_bytes;
  kv->B = block_bytes;
  kv->n_ids = budget_bytes / block_bytes;
  *out = kv;
  return PW_OK;
}

extern "C" void pw_kv_destroy(pw_kv *kv) { delete kv; }

extern "C" pw_status pw_kv_set_weight_bytes(pw_kv *kv, int64_t weight_bytes) {
  if (!kv || weight_bytes < 0) return PW_ERR_INVALID;
  kv->ctx = nullptr;
  kv->W = weight_bytes;
  return PW_OK;
}

extern "C" pw_status pw_kv_attach(pw_kv *kv, pw_ctx *ctx) {
  if (!kv) return PW_ERR_INVALID;
  kv->ctx = ctx;
  if (pw_status st = refresh_weights(kv)) {
    kv->ctx = nullptr;
    return st;
  }
  return PW_OK;
}

extern "C" pw_status pw_kv_announce(pw_kv *kv, int64_t request, int64_t n_blocks) {
  if (!kv || n_blocks < 0) return PW_ERR_INVALID;
  auto it = kv->announced.find(request);
  const int64_t old = it == kv->announced.end() ? 0 : it->second;
  kv->P += n_blocks - old;
  if (n_blocks == 0) {
    if (it != kv->announced.end()) kv->announced.erase(it);
  } else {
    kv->announced[request] = n_blocks;
  }
  return PW_OK;
}

extern "C" pw_status pw_kv_grow(pw_kv *kv, int64_t request, int64_t n_blocks, int32_t *ids_out) {
  if (!kv || n_blocks < 0) return PW_ERR_INVALID;
  if (pw_status st = refresh_weights(kv)) return st;
  auto it = kv->announced.find(request);
  const int64_t own = it == kv->announced.end() ? 0 : it->second;
  const int64_t c = n_blocks < own ? n_blocks : own;
  const int64_t free_blocks = capacity(kv) - kv->U - kv->P;
  if (n_blocks - c > free_blocks) return PW_ERR_OOM;
  // U + n <= C <= n_ids, so the ids below n_ids suffice
  std::vector<int32_t> &mine = kv->held[request];
  try {
    mine.reserve(mine.size() + (size_t)n_blocks);
  } catch (...) {
    return PW_ERR_OOM;
  }
  for (int64_t k = 0; k < n_blocks; ++k) {
    const int32_t id = take_lowest(kv);
    mine.push_back(id);
    if (ids_out) ids_out[k] = id;
  }
  kv->U += n_blocks;
  if (c > 0) pw_kv_announce(kv, request, own - c);
  return PW_OK;
}

extern "C" pw_status pw_kv_release(pw_kv *kv, int64_t request, int64_t *n_released) {
  if (!kv) return PW_ERR_INVALID;
  int64_t n = 0;
  auto it = kv->held.find(request);
  if (it != kv->held.end()) {
    n = (int64_t)it->second.size();
    for (int32_t id : it->second) kv->freed.insert(id);
    kv->held.erase(it);
  }
  // the high-water mark comes back down over released ids at its top
  while (kv->next_id > 0 && !kv->freed.empty() && *kv->freed.rbegin() == kv->next_id - 1) {
    kv->freed.erase(std::prev(kv->freed.end()));
    --kv->next_id;
  }
  kv->U -= n;
  pw_kv_announce(kv, request, 0);
  if (n_released) *n_released = n;
  return PW_OK;
}

extern "C" pw_status pw_kv_request(const pw_kv *kv, int64_t request, int64_t *held, int64_t *announced) {
  if (!kv) return PW_ERR_INVALID;
  if (held) {
    auto it = kv->held.find(request);
    *held = it == kv->held.end() ? 0 : (int64_t)it->second.size();
  }
  if (announced) {
    auto it = kv->announced.find(request);
    *announced = it == kv->announced.end() ? 0 : it->second;
  }
  return PW_OK;
}

extern "C" pw_status pw_kv_blocks(const pw_kv *kv, int64_t request, int32_t *ids_out, int64_t capacity_out,
                                  int64_t *n) {
  if (!kv || !n || capacity_out < 0 || (capacity_out > 0 && !ids_out)) return PW_ERR_INVALID;
  auto it = kv->held.find(request);
  *n = it == kv->held.end() ? 0 : (int64_t)it->second.size();
  for (int64_t k = 0; k < *n && k < capacity_out; ++k) ids_out[k] = it->second[(size_t)k];
  return PW_OK;
}

extern "C" pw_status pw_kv_get_stats(pw_kv *kv, pw_kv_stats *out) {
  if (!kv || !out) return PW_ERR_INVALID;
  if (pw_status st = refresh_weights(kv)) return st;
  out->budget_bytes = kv->S;
  out->block_bytes = kv->B;
  out->weight_bytes = kv->W;
  out->capacity_blocks = capacity(kv);
  out->used_blocks = kv->U;
  out->pending_blocks = kv->P;
  out->free_blocks = out->capacity_blocks - kv->U - kv->P;
  out->headroom_bytes = kv->S - kv->W - kv->U * kv->B;
  return PW_OK;
}
