// Minimal KV block allocator (the "KDA" of §2.4): a host free list of block
// ids that hands out the lowest free ids first, so a fresh pool fills from the
// bottom and freed blocks are reused before untouched ones.
#include <cstdint>
#include <new>
#include <set>
#include <vector>

#include "../../include/dsa.h"

struct dsa_kv_alloc {
  int32_t num_blocks;
  std::set<int32_t> free_ids;
  std::vector<uint8_t> in_use;
};

extern "C" {

dsa_status dsa_kv_alloc_create(int32_t num_blocks, dsa_kv_alloc** out) {
  if (!out || num_blocks < 1) return DSA_ERR_INVALID_ARG;
  dsa_kv_alloc* a = new (std::nothrow) dsa_kv_alloc;
  if (!a) return DSA_ERR_OOM;
  a->num_blocks = num_blocks;
  a->in_use.assign((size_t)num_blocks, 0);
  for (int32_t i = 0; i < num_blocks; ++i) a->free_ids.insert(a->free_ids.end(), i);
  *out = a;
  return DSA_OK;
}

dsa_status dsa_kv_alloc_blocks(dsa_kv_alloc* a, int32_t n, int32_t* out_ids) {
  if (!a || n < 0 || (n > 0 && !out_ids)) return DSA_ERR_INVALID_ARG;
  if ((size_t)n > a->free_ids.size()) return DSA_ERR_OOM;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = *a->free_ids.begin();
    a->free_ids.erase(a->free_ids.begin());
    a->in_use[(size_t)id] = 1;
    out_ids[i] = id;
  }
  return DSA_OK;
}

dsa_status dsa_kv_free_blocks(dsa_kv_alloc* a, const int32_t* ids, int32_t n) {
  if (!a || n < 0 || (n > 0 && !ids)) return DSA_ERR_INVALID_ARG;
  // Check the whole call first so that a bad id changes nothing.
  std::set<int32_t> seen;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= a->num_blocks || !a->in_use[(size_t)id] || !seen.insert(id).second)
      return DSA_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n; ++i) {
    a->in_use[(size_t)ids[i]] = 0;
    a->free_ids.insert(ids[i]);
  }
  return DSA_OK;
}

int32_t dsa_kv_alloc_num_free(const dsa_kv_alloc* a) { return a ? (int32_t)a->free_ids.size() : 0; }

void dsa_kv_alloc_destroy(dsa_kv_alloc* a) { delete a; }

}  // extern "C"
