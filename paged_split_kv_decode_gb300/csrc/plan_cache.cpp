// Decode-plan cache: detection and cascade planning memoised across layers and steps.
//
// The pages leave this as a follow-up: the plan cache holds the page table, but the
// detection scan re-runs per layer per step (mlxcel PR #1004, Left out / unsure names
// a cascade-plan entry in that cache as the follow-up).  Another page reports a bug in
// exactly such a cache: it was keyed by rows, although split-KV also depends on the
// KV length (FreeToken issue #750, Layer-major prefill for offloaded MoE, Attention
// batching section).  So the key here is everything psd_plan_decode reads: the
// resolved switch, both thresholds, the tile and page sizes, the batch, and the full
// contents of page_indptr, page_indices and last_page_len.  A 64-bit hash picks the
// candidate entry and an exact comparison of the key confirms it, so a hit always
// returns the plan that planning from scratch would return.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <memory>
#include <vector>

#include "psd_internal.h"

namespace {

struct Entry {
  uint64_t hash = 0;
  int64_t generation = -1;    // caller's table generation at planning time, or -1
  int32_t args[5] = {0, 0, 0, 0, 0};  // tile_tokens, enable, thresholds, batch
  std::vector<int32_t> key;
  std::vector<int32_t> members, row_base, o_indptr;
  std::vector<psd_work_item> l0, l1;
  psd_cascade_plan plan{};  // arrays point into the vectors above
  uint64_t last_use = 0;
  bool valid = false;
};

// Four independent multiply-xor lanes over 64-bit words, so the chain of dependent
// multiplies is a quarter as long; a tail shorter than 32 bytes goes word by word.
uint64_t hash_bytes(const void *data, size_t bytes, uint64_t seed) {
  const uint8_t *p = static_cast<const uint8_t *>(data);
  uint64_t h[4] = {seed ^ 0x9E3779B97F4A7C15ull, seed ^ 0xBF58476D1CE4E5B9ull,
                   seed ^ 0x94D049BB133111EBull, seed ^ 0x2545F4914F6CDD1Dull};
  size_t i = 0;
  for (; i + 32 <= bytes; i += 32) {
    for (int l = 0; l < 4; ++l) {
      uint64_t w;
      std::memcpy(&w, p + i + 8 * l, 8);
      h[l] = (h[l] ^ w) * 0xFF51AFD7ED558CCDull;
      h[l] ^= h[l] >> 32;
    }
  }
  uint64_t r = h[0] ^ (h[1] * 3) ^ (h[2] * 5) ^ (h[3] * 7) ^ bytes;
  for (; i < bytes; ++i) r = (r ^ p[i]) * 0x100000001B3ull;
  return r ^ (r >> 31);
}

}  // namespace

struct psd_plan_cache {
  std::vector<std::unique_ptr<Entry>> entries;
  uint64_t clock = 0;
  int64_t hits = 0, misses = 0;
};

extern "C" psd_status psd_plan_cache_create(psd_plan_cache **cache, int32_t capacity) {
  psd::clear_error();
  if (!cache) return psd::fail(PSD_ERR_INVALID_ARG, "psd_plan_cache_create: NULL");
  *cache = nullptr;
  if (capacity < 1 || capacity > 1024)
    return psd::fail(PSD_ERR_INVALID_ARG, "psd_plan_cache_create: capacity %d outside [1, 1024]", capacity);
  psd_plan_cache *c = new psd_plan_cache();
  c->entries.resize(size_t(capacity));
  for (auto &e : c->entries) e.reset(new Entry());
  *cache = c;
  return PSD_OK;
}

extern "C" psd_status psd_plan_cache_destroy(psd_plan_cache *cache) {
  psd::clear_error();
  delete cache;
  return PSD_OK;
}

namespace {

psd_status lookup(psd_plan_cache *cache, int64_t generation, const psd_page_table *host,
                  int32_t tile_tokens, int32_t enable, int32_t min_shared_pages, int32_t min_members,
                  const psd_cascade_plan **plan, int32_t *hit) {
  psd::clear_error();
  if (!cache || !plan || !host) return psd::fail(PSD_ERR_INVALID_ARG, "psd_plan_cache_lookup: NULL");
  *plan = nullptr;
  if (hit) *hit = 0;
  if (enable < 0) enable = psd_cascade_env_enabled(0);
  const int32_t args[5] = {tile_tokens, enable, min_shared_pages, min_members, host->batch};
  if (generation >= 0) {  // the caller vouches that this generation's table is unchanged
    ++cache->clock;
    for (auto &e : cache->entries) {
      if (e->valid && e->generation == generation && std::memcmp(e->args, args, sizeof(args)) == 0) {
        e->last_use = cache->clock;
        ++cache->hits;
        *plan = &e->plan;
        if (hit) *hit = 1;
        return PSD_OK;
      }
    }
  }
  // The table is checked before any of its arrays is read into the key.
  psd_status st = psd::validate_table(host, -1);
  if (st != PSD_OK) return st;
  const int32_t B = host->batch, nnz = host->page_indptr[B];
  const int32_t header[6] = {B, host->page_size, tile_tokens, enable, min_shared_pages, min_members};
  // key = header | page_indptr[B+1] | page_indices[nnz] | last_page_len[B], hashed and
  // compared in place; only a miss copies it.
  const size_t nb_ptr = sizeof(int32_t) * size_t(B + 1), nb_idx = sizeof(int32_t) * size_t(nnz),
               nb_last = sizeof(int32_t) * size_t(B);
  uint64_t h = hash_bytes(header, sizeof(header), 1);
  h = hash_bytes(host->page_indptr, nb_ptr, h);
  h = hash_bytes(host->page_indices, nb_idx, h);
  h = hash_bytes(host->last_page_len, nb_last, h);
  ++cache->clock;
  auto same_key = [&](const std::vector<int32_t> &k) {
    if (k.size() != 6 + size_t(B + 1) + size_t(nnz) + size_t(B)) return false;
    const int32_t *q = k.data();
    return std::memcmp(q, header, sizeof(header)) == 0 &&
           std::memcmp(q + 6, host->page_indptr, nb_ptr) == 0 &&
           std::memcmp(q + 6 + (B + 1), host->page_indices, nb_idx) == 0 &&
           std::memcmp(q + 6 + (B + 1) + nnz, host->last_page_len, nb_last) == 0;
  };

  for (auto &e : cache->entries) {
    if (e->valid && e->hash == h && same_key(e->key)) {
      if (generation >= 0) e->generation = generation;
      e->last_use = cache->clock;
      ++cache->hits;
      *plan = &e->plan;
      if (hit) *hit = 1;
      return PSD_OK;
    }
  }

  // Miss: plan into the empty or least recently used entry.
  Entry *v = cache->entries.front().get();
  for (auto &e : cache->entries) {
    if (!e->valid) {
      v = e.get();
      break;
    }
    if (e->last_use < v->last_use) v = e.get();
  }
  v->valid = false;
  const size_t bc = size_t(std::max(B, 1)), ic = size_t(std::max(nnz, 1));
  v->members.assign(bc, 0);
  v->row_base.assign(bc, 0);
  v->o_indptr.assign(bc + 1, 0);
  v->l0.assign(ic, psd_work_item{});
  v->l1.assign(ic, psd_work_item{});
  psd_cascade_plan &p = v->plan;
  p = psd_cascade_plan{};
  p.batch_capacity = int32_t(bc);
  p.item_capacity = int32_t(ic);
  p.members = v->members.data();
  p.member_row_base = v->row_base.data();
  p.l0_items = v->l0.data();
  p.l1_items = v->l1.data();
  p.o_indptr = v->o_indptr.data();
  st = psd_plan_decode(host, tile_tokens, enable, min_shared_pages, min_members, &p);
  if (st != PSD_OK) return st;
  v->key.assign(header, header + 6);
  v->key.insert(v->key.end(), host->page_indptr, host->page_indptr + B + 1);
  v->key.insert(v->key.end(), host->page_indices, host->page_indices + nnz);
  v->key.insert(v->key.end(), host->last_page_len, host->last_page_len + B);
  v->hash = h;
  v->generation = generation >= 0 ? generation : -1;
  std::memcpy(v->args, args, sizeof(args));
  v->last_use = cache->clock;
  v->valid = true;
  ++cache->misses;
  *plan = &p;
  return PSD_OK;
}

}  // namespace

extern "C" psd_status psd_plan_cache_lookup(psd_plan_cache *cache, const psd_page_table *host,
                                            int32_t tile_tokens, int32_t enable,
                                            int32_t min_shared_pages, int32_t min_members,
                                            const psd_cascade_plan **plan, int32_t *hit) {
  return lookup(cache, -1, host, tile_tokens, enable, min_shared_pages, min_members, plan, hit);
}

extern "C" psd_status psd_plan_cache_lookup_gen(psd_plan_cache *cache, int64_t generation,
                                                const psd_page_table *host, int32_t tile_tokens,
                                                int32_t enable, int32_t min_shared_pages,
                                                int32_t min_members, const psd_cascade_plan **plan,
                                                int32_t *hit) {
  return lookup(cache, generation, host, tile_tokens, enable, min_shared_pages, min_members, plan, hit);
}

extern "C" psd_status psd_plan_cache_stats(const psd_plan_cache *cache, int64_t *hits, int64_t *misses,
                                           int32_t *entries) {
  psd::clear_error();
  if (!cache) return psd::fail(PSD_ERR_INVALID_ARG, "psd_plan_cache_stats: NULL");
  if (hits) *hits = cache->hits;
  if (misses) *misses = cache->misses;
  if (entries) {
    int32_t n = 0;
    for (auto &e : cache->entries) n += e->valid ? 1 : 0;
    *entries = n;
  }
  return PSD_OK;
}
