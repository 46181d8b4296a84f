// kvp_block_manager.cpp -- host-side block allocator with reference counts and
// copy-on-write (plain C++, no CUDA).  It produces what the GPU entry points
// consume: block tables, slot mappings and copy pairs.
//
//   * Free pool and per-request block lists, ceil(tokens / block_size) blocks
//     per request, blocks returned when a request ends ("ATB KV Cache
//     management", "BlockManager 的调度").
//   * A request's blocks come from the largest free contiguous range that can
//     hold them, else the lowest free ids ("显存碎片问题": contiguous first,
//     scattered otherwise).  A new block for a growing request prefers the id
//     right after its current last block.
//   * Allocation fails cleanly, leaving the state unchanged, when the pool is
//     short ("KV Cache 优化与显存管理", 三: allocate returns nothing; "ATB
//     PagedAttention", "ATB 的 PagedAttention 实现": Status::OUT_OF_MEMORY).
//   * Reference counts: sharing increments, release decrements and frees at 0;
//     releasing a block a request does not hold is an error ("踩坑二").
//   * Appending into a shared block first moves the request onto a private
//     copy ("踩坑三", ExtendKVPage: copy-on-write only when the count > 1).
#include <algorithm>
#include <cstdint>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "kvp.h"

struct kvp_bm {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  int64_t bytes_per_block = 0;
  std::vector<int32_t> ref;        // reference count per block
  std::set<int32_t> free_ids;      // blocks with ref == 0, ordered
  struct Req {
    std::vector<int32_t> blocks;
    int32_t tokens = 0;
  };
  std::unordered_map<int64_t, Req> reqs;
  int64_t refs = 0;                // sum of reference counts

  int32_t take(int32_t id) {
    free_ids.erase(id);
    ref[id] = 1;
    ++refs;
    return id;
  }
  void drop(int32_t id) {
    --refs;
    if (--ref[id] == 0) free_ids.insert(id);
  }
  // Lowest free id, or `prefer` if it is free.
  int32_t pick_one(int32_t prefer) const {
    if (prefer >= 0 && prefer < num_blocks && ref[prefer] == 0) return prefer;
    return free_ids.empty() ? -1 : *free_ids.begin();
  }
};

extern "C" {

kvp_bm* kvp_bm_create(int32_t num_blocks, int32_t block_size, int64_t bytes_per_block) {
  if (num_blocks <= 0 || block_size <= 0 || bytes_per_block < 0) return nullptr;
  kvp_bm* bm = new (std::nothrow) kvp_bm();
  if (bm == nullptr) return nullptr;
  try {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->bytes_per_block = bytes_per_block;
    bm->ref.assign(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) bm->free_ids.insert(bm->free_ids.end(), i);
  } catch (...) {
    delete bm;
    return nullptr;
  }
  return bm;
}

void kvp_bm_destroy(kvp_bm* bm) { delete bm; }

kvp_status kvp_bm_allocate(kvp_bm* bm, int64_t req, int32_t num_tokens, int32_t reserve_blocks) {
  if (bm == nullptr || num_tokens < 0 || reserve_blocks < 0) return KVP_ERR_INVALID_ARG;
  if (bm->reqs.count(req)) return KVP_ERR_INVALID_ARG;
  const int64_t need =
      (static_cast<int64_t>(num_tokens) + bm->block_size - 1) / bm->block_size + reserve_blocks;
  if (need > static_cast<int64_t>(bm->free_ids.size())) return KVP_ERR_OOM;
  kvp_bm::Req r;
  r.tokens = num_tokens;
  // largest free run of consecutive ids
  int32_t best_start = -1, best_len = 0, run_start = -1, run_len = 0, prev = -2;
  for (int32_t id : bm->free_ids) {
    if (id == prev + 1) {
      ++run_len;
    } else {
      run_start = id;
      run_len = 1;
    }
    if (run_len > best_len) {
      best_len = run_len;
      best_start = run_start;
    }
    prev = id;
  }
  if (need > 0 && best_len >= need) {
    for (int64_t i = 0; i < need; ++i) r.blocks.push_back(bm->take(best_start + static_cast<int32_t>(i)));
  } else {
    for (int64_t i = 0; i < need; ++i) r.blocks.push_back(bm->take(*bm->free_ids.begin()));
  }
  bm->reqs.emplace(req, std::move(r));
  return KVP_OK;
}

kvp_status kvp_bm_share_prefix(kvp_bm* bm, int64_t src, int64_t dst, int32_t num_tokens) {
  if (bm == nullptr || num_tokens < 0) return KVP_ERR_INVALID_ARG;
  auto it = bm->reqs.find(src);
  if (it == bm->reqs.end()) return KVP_ERR_NOT_FOUND;
  if (bm->reqs.count(dst) || num_tokens > it->second.tokens) return KVP_ERR_INVALID_ARG;
  const int32_t nb = (num_tokens + bm->block_size - 1) / bm->block_size;
  kvp_bm::Req r;
  r.tokens = num_tokens;
  r.blocks.assign(it->second.blocks.begin(), it->second.blocks.begin() + nb);
  for (int32_t id : r.blocks) {
    ++bm->ref[id];
    ++bm->refs;
  }
  bm->reqs.emplace(dst, std::move(r));
  return KVP_OK;
}

kvp_status kvp_bm_append_slot(kvp_bm* bm, int64_t req, int32_t* slot, int32_t* cow_src,
                              int32_t* cow_dst) {
  if (bm == nullptr || slot == nullptr || cow_src == nullptr || cow_dst == nullptr)
    return KVP_ERR_INVALID_ARG;
  auto it = bm->reqs.find(req);
  if (it == bm->reqs.end()) return KVP_ERR_NOT_FOUND;
  kvp_bm::Req& r = it->second;
  const int32_t pos = r.tokens;
  const int32_t bi = pos / bm->block_size;
  *cow_src = -1;
  *cow_dst = -1;
  if (bi >= static_cast<int32_t>(r.blocks.size())) {
    // capacity exceeded: a new block, right after the last one when possible
    const int32_t id = bm->pick_one(r.blocks.empty() ? -1 : r.blocks.back() + 1);
    if (id < 0) return KVP_ERR_OOM;
    r.blocks.push_back(bm->take(id));
  } else if (bm->ref[r.blocks[bi]] > 1) {
    // the block receiving the token is shared: copy-on-write
    const int32_t old = r.blocks[bi];
    const int32_t id = bm->pick_one(-1);
    if (id < 0) return KVP_ERR_OOM;
    bm->take(id);
    bm->drop(old);
    r.blocks[bi] = id;
    *cow_src = old;
    *cow_dst = id;
  }
  *slot = r.blocks[bi] * bm->block_size + pos % bm->block_size;
  r.tokens = pos + 1;
  return KVP_OK;
}

kvp_status kvp_bm_free(kvp_bm* bm, int64_t req) {
  if (bm == nullptr) return KVP_ERR_INVALID_ARG;
  auto it = bm->reqs.find(req);
  if (it == bm->reqs.end()) return KVP_ERR_NOT_FOUND;
  for (int32_t id : it->second.blocks) bm->drop(id);
  bm->reqs.erase(it);
  return KVP_OK;
}

kvp_status kvp_bm_release_block(kvp_bm* bm, int64_t req, int32_t block) {
  if (bm == nullptr) return KVP_ERR_INVALID_ARG;
  auto it = bm->reqs.find(req);
  if (it == bm->reqs.end()) return KVP_ERR_NOT_FOUND;
  auto& blocks = it->second.blocks;
  auto pos = std::find(blocks.begin(), blocks.end(), block);
  if (pos == blocks.end()) return KVP_ERR_REFCOUNT;
  // the request gives up `block` and everything after it in its table
  const int32_t keep = static_cast<int32_t>(pos - blocks.begin());
  for (auto p = pos; p != blocks.end(); ++p) bm->drop(*p);
  blocks.resize(keep);
  it->second.tokens = std::min(it->second.tokens, keep * bm->block_size);
  return KVP_OK;
}

int32_t kvp_bm_block_table(const kvp_bm* bm, int64_t req, int32_t* out, int32_t cap) {
  if (bm == nullptr) return -1;
  auto it = bm->reqs.find(req);
  if (it == bm->reqs.end()) return -1;
  const auto& blocks = it->second.blocks;
  const int32_t n = static_cast<int32_t>(blocks.size());
  if (out != nullptr) {
    for (int32_t i = 0; i < n && i < cap; ++i) out[i] = blocks[i];
  }
  return n;
}

int32_t kvp_bm_num_tokens(const kvp_bm* bm, int64_t req) {
  if (bm == nullptr) return -1;
  auto it = bm->reqs.find(req);
  return it == bm->reqs.end() ? -1 : it->second.tokens;
}

int32_t kvp_bm_ref_count(const kvp_bm* bm, int32_t block) {
  if (bm == nullptr || block < 0 || block >= bm->num_blocks) return -1;
  return bm->ref[block];
}

void kvp_bm_stats(const kvp_bm* bm, kvp_bm_stats_t* out) {
  if (bm == nullptr || out == nullptr) return;
  out->total_blocks = bm->num_blocks;
  out->free_blocks = static_cast<int32_t>(bm->free_ids.size());
  out->used_blocks = bm->num_blocks - out->free_blocks;
  out->active_requests = static_cast<int32_t>(bm->reqs.size());
  out->block_refs = bm->refs;
  out->utilization = static_cast<double>(out->used_blocks) / bm->num_blocks;
  out->bytes_per_block = bm->bytes_per_block;
  out->total_memory_gb = static_cast<double>(bm->num_blocks) * bm->bytes_per_block / 1e9;
}

}  // extern "C"
