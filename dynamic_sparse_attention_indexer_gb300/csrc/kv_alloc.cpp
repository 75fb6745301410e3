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

// Block allocator with one block bitmap per (layer, KV head) (§2.4: the
// allocator knows the layer and the head and keeps an independent block bitmap
// per head, so that heads do not overwrite one another's blocks).  A (layer,
// head) owns the head-h slices of the blocks its bitmap marks; the same block
// id can be held by several heads at once, for different positions.  A request
// takes the lowest free ids of that (layer, head); a release must name blocks
// that (layer, head) holds, each once, else nothing changes.
struct dsa_kv_bitmap {
  int32_t num_layers, num_heads, num_blocks, words;
  std::vector<uint64_t> bits;  // [layer][head][words]
  std::vector<int32_t> used;   // [layer][head] blocks held
  uint64_t* map(int32_t l, int32_t h) { return bits.data() + ((size_t)l * num_heads + h) * words; }
  bool valid(int32_t l, int32_t h) const { return l >= 0 && l < num_layers && h >= 0 && h < num_heads; }
};

extern "C" {

dsa_status dsa_kv_bitmap_create(int32_t num_layers, int32_t num_heads, int32_t num_blocks, dsa_kv_bitmap** out) {
  if (!out || num_layers < 1 || num_heads < 1 || num_blocks < 1) return DSA_ERR_INVALID_ARG;
  if ((int64_t)num_layers * num_heads > (1 << 20)) return DSA_ERR_UNSUPPORTED;
  dsa_kv_bitmap* a = new (std::nothrow) dsa_kv_bitmap;
  if (!a) return DSA_ERR_OOM;
  a->num_layers = num_layers;
  a->num_heads = num_heads;
  a->num_blocks = num_blocks;
  a->words = (num_blocks + 63) / 64;
  try {
    a->bits.assign((size_t)num_layers * num_heads * a->words, 0);
    a->used.assign((size_t)num_layers * num_heads, 0);
  } catch (...) {
    delete a;
    return DSA_ERR_OOM;
  }
  *out = a;
  return DSA_OK;
}

dsa_status dsa_kv_bitmap_alloc(dsa_kv_bitmap* a, int32_t layer, int32_t head, int32_t n, int32_t* out_ids) {
  if (!a || !a->valid(layer, head) || n < 0 || (n > 0 && !out_ids)) return DSA_ERR_INVALID_ARG;
  int32_t& used = a->used[(size_t)layer * a->num_heads + head];
  if (n > a->num_blocks - used) return DSA_ERR_OOM;
  uint64_t* m = a->map(layer, head);
  int32_t got = 0;
  for (int32_t w = 0; w < a->words && got < n; ++w) {
    uint64_t free_bits = ~m[w];
    if (w == a->words - 1 && (a->num_blocks & 63)) free_bits &= (1ull << (a->num_blocks & 63)) - 1;
    while (free_bits && got < n) {
      const int b = __builtin_ctzll(free_bits);
      free_bits &= free_bits - 1;
      m[w] |= 1ull << b;
      out_ids[got++] = w * 64 + b;
    }
  }
  used += got;
  return DSA_OK;
}

dsa_status dsa_kv_bitmap_free(dsa_kv_bitmap* a, int32_t layer, int32_t head, const int32_t* ids, int32_t n) {
  if (!a || !a->valid(layer, head) || n < 0 || (n > 0 && !ids)) return DSA_ERR_INVALID_ARG;
  uint64_t* m = a->map(layer, head);
  // Check the whole call first (held, each once) so that a bad id changes nothing.
  std::vector<uint64_t> seen((size_t)a->words, 0);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= a->num_blocks) return DSA_ERR_INVALID_ARG;
    const uint64_t bit = 1ull << (id & 63);
    if (!(m[id >> 6] & bit) || (seen[(size_t)(id >> 6)] & bit)) return DSA_ERR_INVALID_ARG;
    seen[(size_t)(id >> 6)] |= bit;
  }
  for (int32_t i = 0; i < n; ++i) m[ids[i] >> 6] &= ~(1ull << (ids[i] & 63));
  a->used[(size_t)layer * a->num_heads + head] -= n;
  return DSA_OK;
}

int32_t dsa_kv_bitmap_num_free(const dsa_kv_bitmap* a, int32_t layer, int32_t head) {
  if (!a || !a->valid(layer, head)) return -1;
  return a->num_blocks - a->used[(size_t)layer * a->num_heads + head];
}

dsa_status dsa_kv_bitmap_words(const dsa_kv_bitmap* a, int32_t layer, int32_t head, uint64_t* words,
                               int32_t n_words) {
  if (!a || !a->valid(layer, head) || !words || n_words < a->words) return DSA_ERR_INVALID_ARG;
  const uint64_t* m = const_cast<dsa_kv_bitmap*>(a)->map(layer, head);
  for (int32_t w = 0; w < a->words; ++w) words[w] = m[w];
  return DSA_OK;
}

void dsa_kv_bitmap_destroy(dsa_kv_bitmap* a) { delete a; }

}  // extern "C"
