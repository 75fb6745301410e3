// The C ABI: argument checks, workspace layout, launch order.
//
// Nothing here touches the GPU before every argument has been checked, so the
// error paths run (and are tested) on machines without a GPU.
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/dsa.h"
#include "internal.h"

namespace {

thread_local std::string g_msg;

dsa_status fail(dsa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_msg = buf;
  return s;
}

dsa_status cuda_fail(const char* where, cudaError_t e) {
  return fail(DSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Kernel attributes are set once per device, before the first launch there.
dsa_status ensure_setup() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= 64) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d >= 64", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return DSA_OK;
  if ((e = dsa::setup_index_kernels()) != cudaSuccess) return cuda_fail("setup (index kernels)", e);
  if ((e = dsa::setup_topk_kernels()) != cudaSuccess) return cuda_fail("setup (top-k kernels)", e);
  if ((e = dsa::setup_attn_kernels()) != cudaSuccess) return cuda_fail("setup (attention kernels)", e);
  if ((e = dsa::setup_prefix_kernels()) != cudaSuccess) return cuda_fail("setup (prefix kernel)", e);
  if ((e = dsa::setup_dense_kernels()) != cudaSuccess) return cuda_fail("setup (dense prefill kernel)", e);
  if ((e = dsa::setup_pselect_kernels()) != cudaSuccess) return cuda_fail("setup (fused prefill selection)", e);
  done[dev] = true;
  return DSA_OK;
}

dsa_status check_kv(const dsa_paged_kv* kv, dsa::KV* out) {
  if (!kv) return fail(DSA_ERR_INVALID_ARG, "kv descriptor is NULL");
  if (kv->block_size != 64) return fail(DSA_ERR_UNSUPPORTED, "block_size %d: only 64 is supported", kv->block_size);
  if (kv->head_dim != 128) return fail(DSA_ERR_UNSUPPORTED, "head_dim %d: only 128 is supported", kv->head_dim);
  if (kv->idx_dim != 64) return fail(DSA_ERR_UNSUPPORTED, "idx_dim %d: only 64 is supported", kv->idx_dim);
  if (kv->num_blocks < 1 || kv->num_kv_heads < 1 || kv->batch < 1 || kv->max_blocks_per_seq < 1)
    return fail(DSA_ERR_INVALID_ARG, "num_blocks, num_kv_heads, batch and max_blocks_per_seq must be >= 1");
  if (kv->num_kv_heads != 1 && kv->num_kv_heads != 2 && kv->num_kv_heads != 4 && kv->num_kv_heads != 8)
    return fail(DSA_ERR_UNSUPPORTED, "num_kv_heads %d: only 1, 2, 4 or 8 are supported", kv->num_kv_heads);
  if ((int64_t)kv->num_blocks * kv->num_kv_heads * 64 >= (int64_t(1) << 31))
    return fail(DSA_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * 64 must stay below 2^31 rows");
  if ((int64_t)kv->max_blocks_per_seq * 64 >= (int64_t(1) << 30))
    return fail(DSA_ERR_UNSUPPORTED, "max_blocks_per_seq * 64 must stay below 2^30 positions");
  if (kv->max_context_len < 1 || (int64_t)kv->max_context_len > (int64_t)kv->max_blocks_per_seq * 64)
    return fail(DSA_ERR_INVALID_ARG, "max_context_len %d outside [1, max_blocks_per_seq * 64]", kv->max_context_len);
  if (!kv->k_cache || !kv->v_cache || !kv->idx_cache || !kv->block_table || !kv->context_lens)
    return fail(DSA_ERR_INVALID_ARG, "a cache, block_table or context_lens pointer is NULL");
  if (!aligned16(kv->k_cache) || !aligned16(kv->v_cache) || !aligned16(kv->idx_cache))
    return fail(DSA_ERR_INVALID_ARG, "k_cache, v_cache and idx_cache must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(kv->block_table) & 3u) || (reinterpret_cast<uintptr_t>(kv->context_lens) & 3u))
    return fail(DSA_ERR_INVALID_ARG, "block_table and context_lens must be 4-byte aligned");
  const int32_t row = kv->num_kv_heads * 128;
  const int32_t stride = kv->kv_row_stride == 0 ? row : kv->kv_row_stride;
  if (stride < row || stride % 8 != 0)
    return fail(DSA_ERR_INVALID_ARG, "kv_row_stride %d: must be 0 or a multiple of 8 >= num_kv_heads * 128 (%d)",
                kv->kv_row_stride, row);
  if ((int64_t)kv->num_blocks * 64 * stride >= (int64_t(1) << 40))
    return fail(DSA_ERR_UNSUPPORTED, "num_blocks * 64 * kv_row_stride must stay below 2^40 values");
  out->k_cache = kv->k_cache;
  out->v_cache = kv->v_cache;
  out->idx_cache = kv->idx_cache;
  out->block_table = kv->block_table;
  out->context_lens = kv->context_lens;
  out->num_blocks = kv->num_blocks;
  out->hkv = kv->num_kv_heads;
  out->max_blocks = kv->max_blocks_per_seq;
  out->batch = kv->batch;
  out->max_ctx = kv->max_context_len;
  out->row_stride = stride;
  out->adjacent = stride == 2 * row &&
                  static_cast<const char*>(kv->v_cache) == static_cast<const char*>(kv->k_cache) + 2 * (size_t)row;
  return DSA_OK;
}

dsa_status check_qs(const dsa_query_set* qs, const dsa::KV& kv, dsa::QS* out) {
  if (!qs) return fail(DSA_ERR_INVALID_ARG, "query set is NULL");
  if (qs->mode == DSA_MODE_DECODE) {
    if (qs->n_q != kv.batch) return fail(DSA_ERR_INVALID_ARG, "decode: n_q (%d) must equal batch (%d)", qs->n_q, kv.batch);
    if (kv.batch > dsa::kMaxDecodeBatch)
      return fail(DSA_ERR_UNSUPPORTED, "decode: batch %d above %d", kv.batch, dsa::kMaxDecodeBatch);
    if (kv.max_ctx > dsa::kMaxDecodeCtx)
      return fail(DSA_ERR_UNSUPPORTED, "decode: max_context_len above %d", dsa::kMaxDecodeCtx);
  } else if (qs->mode == DSA_MODE_PREFILL) {
    if (qs->n_q < 1) return fail(DSA_ERR_INVALID_ARG, "prefill: n_q must be >= 1");
    if (qs->seq < 0 || qs->seq >= kv.batch) return fail(DSA_ERR_INVALID_ARG, "prefill: seq %d outside [0, batch)", qs->seq);
    if (qs->pos0 < 0 || (int64_t)qs->pos0 + qs->n_q > (int64_t)kv.max_blocks * 64)
      return fail(DSA_ERR_INVALID_ARG, "prefill: positions [pos0, pos0 + n_q) must lie in [0, max_blocks_per_seq * 64)");
  } else {
    return fail(DSA_ERR_INVALID_ARG, "unknown query-set mode %d", qs->mode);
  }
  out->mode = qs->mode;
  out->n_q = qs->n_q;
  out->seq = qs->seq;
  out->pos0 = qs->pos0;
  return DSA_OK;
}

// Largest position + 1 any query of the set can see.
int64_t positions_needed(const dsa::KV& kv, const dsa::QS& qs) {
  return qs.mode == DSA_MODE_DECODE ? (int64_t)kv.max_ctx : (int64_t)qs.pos0 + qs.n_q;
}

dsa_status check_scores(const int32_t* scores, int32_t ld, const dsa::KV& kv, const dsa::QS& qs) {
  if (!scores || !aligned16(scores)) return fail(DSA_ERR_INVALID_ARG, "scores must be non-NULL and 16-byte aligned");
  if (ld % 4 != 0) return fail(DSA_ERR_INVALID_ARG, "ld (%d) must be a multiple of 4", ld);
  if ((int64_t)ld < positions_needed(kv, qs))
    return fail(DSA_ERR_INVALID_ARG, "ld (%d) below the largest position + 1 (%lld)", ld,
                (long long)positions_needed(kv, qs));
  return DSA_OK;
}

// Workspace regions.  Decode top-k: [coarse histograms]; attention: [selected
// slots | partials].  The histograms must be zero when a call starts; every
// call leaves them zero again.
struct Layout {
  size_t coarse = 0, slot = 0;
  size_t pre_ml = 0, pre_o = 0;  // 0 size: none
  bool pre = false;
  size_t part_o = 0, part_ml = 0;
  size_t sel_end = 0, attn_begin = 0, total = 0;
};

Layout layout(const dsa::KV& kv, const dsa::QS& qs, int k, int hq, int prefix) {
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = up256(off + bytes);
    return o;
  };
  if (qs.mode == DSA_MODE_DECODE) {
    const size_t B = (size_t)kv.batch;
    L.coarse = take(B * dsa::kCoarseBinsHost * 4);
  }
  L.sel_end = off;
  L.attn_begin = off;
  if (qs.mode == DSA_MODE_DECODE)  // the fused decode step's selected cache slots
    L.slot = take((size_t)qs.n_q * (size_t)k * 4);
  if (qs.mode == DSA_MODE_PREFILL && prefix > 0) {  // the prefix part of every query, per tile of queries
    L.pre = true;
    L.pre_ml = take((size_t)qs.n_q * (size_t)hq * 8);
    L.pre_o = take((size_t)qs.n_q * (size_t)hq * 128 * 4);
  }
  // two partial slots per CTA and pass; decode may walk two passes
  const size_t slots = qs.mode == DSA_MODE_DECODE ? 4 : 2;
  L.part_o = take((size_t)dsa::kMaxAttnCtas * slots * (size_t)hq * 128 * 4);
  L.part_ml = take((size_t)dsa::kMaxAttnCtas * slots * (size_t)hq * 8);
  L.total = off;
  return L;
}

dsa::SelState sel_state(const Layout& L, void* ws, bool with_slot) {
  char* w = static_cast<char*>(ws);
  dsa::SelState s;
  s.coarse = reinterpret_cast<int*>(w + L.coarse);
  s.slot = with_slot ? reinterpret_cast<int*>(w + L.slot) : nullptr;
  return s;
}

// The fused decode step's overlap: the selection's clusters are capped so
// that they hold at most half of the SMs, and the attention's first pass (the
// prefix rows, before its wait) runs over the CTAs that find an SM free
// while the selection runs.
void overlap_shape(const dsa::KV& kv, int prefix, int* c_cap, int* prefix_ctas) {
  const int sms = dsa::attn_grid_ctas();
  int c = 16;
  while (c > 1 && c * kv.batch > sms / 2) c >>= 1;
  *c_cap = c;
  const int held = dsa::decode_select_ctas(kv, prefix, c);
  if (held <= kv.batch) {
    // one CTA per sequence already fills half of the SMs: one pass, nothing
    // to overlap (8K, B = 32: one pass 48.5 us, two passes 48.9 us).  The
    // clusters are then capped so that the selection is about one wave of
    // CTAs at two per SM (per-KV-head step, 64 rows of 128K: clusters of 16
    // 168 us, of 8 157 us, of 4 153 us, of 2 155 us).
    int cap = 16;
    while (cap > 1 && cap * kv.batch > 2 * sms) cap >>= 1;
    *c_cap = cap;
    *prefix_ctas = 0;
    return;
  }
  const int free_ctas = sms - held;
  *prefix_ctas = free_ctas > sms / 4 ? free_ctas : sms / 4;
}

dsa::AttnWs attn_ws(const Layout& L, void* ws) {
  char* w = static_cast<char*>(ws);
  dsa::AttnWs a;
  a.pre_ml = L.pre ? reinterpret_cast<float2*>(w + L.pre_ml) : nullptr;
  a.pre_o = L.pre ? reinterpret_cast<float*>(w + L.pre_o) : nullptr;
  a.part_o = reinterpret_cast<float*>(w + L.part_o);
  a.part_ml = reinterpret_cast<float2*>(w + L.part_ml);
  return a;
}

dsa_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return DSA_OK;
  if (!ws || !aligned16(ws)) return fail(DSA_ERR_WORKSPACE, "workspace must be non-NULL and 16-byte aligned");
  if (ws_bytes < need) return fail(DSA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return DSA_OK;
}

dsa_status check_k_prefix(int32_t k, int32_t prefix) {
  if (k < 1) return fail(DSA_ERR_INVALID_ARG, "k (%d) must be >= 1", k);
  if (prefix < 0) return fail(DSA_ERR_INVALID_ARG, "prefix_len (%d) must be >= 0", prefix);
  if ((int64_t)prefix + k > (int64_t(1) << 24)) return fail(DSA_ERR_UNSUPPORTED, "prefix_len + k above 2^24");
  return DSA_OK;
}

// The attention kernel walks the attended-row slots of all queries, n_q * (prefix + k), in 32-bit.
dsa_status check_tiles(const dsa::KV& kv, const dsa::QS& qs, int32_t k, int32_t prefix) {
  (void)kv;
  if ((int64_t)qs.n_q * ((int64_t)prefix + k) >= (int64_t(1) << 31))
    return fail(DSA_ERR_UNSUPPORTED, "n_q * (prefix_len + k) must stay below 2^31");
  return DSA_OK;
}

// The attention kernel stages one query's Q (all heads) in a shared-memory
// slot sized for dsa::kMaxQHeads heads, so more heads are refused here, before
// anything is launched.
dsa_status check_heads(int32_t hq, const dsa::KV& kv) {
  if (hq < 1 || hq % kv.hkv != 0)
    return fail(DSA_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)", hq, kv.hkv);
  if (hq > dsa::kMaxQHeads)
    return fail(DSA_ERR_UNSUPPORTED, "num_q_heads %d above %d", hq, dsa::kMaxQHeads);
  if (hq / kv.hkv > 16) return fail(DSA_ERR_UNSUPPORTED, "GQA group %d > 16 query heads per KV head", hq / kv.hkv);
  return DSA_OK;
}

#define DSA_TRY(x)                  \
  do {                              \
    const dsa_status s_ = (x);      \
    if (s_ != DSA_OK) return s_;    \
  } while (0)

#define DSA_CUDA(where, x)                        \
  do {                                            \
    const cudaError_t e_ = (x);                   \
    if (e_ != cudaSuccess) return cuda_fail(where, e_); \
  } while (0)

// Prefill attention runs its first n_dense queries as a masked dense pass over
// every causal position (k_dense.cu) and the rest by gathering their attended
// rows (k_prefix.cu + k_attn.cu).  Per (query, KV head) and position the dense
// pass costs about 1/kDenseRatio of a gathered row on GB300 (16K chunk: 0.72 ns
// against 7.6 ns of SM time), and a query at position pos attends
// min(P, pos + 1) + min(k, pos + 1 - P) rows out of pos + 1, so the dense pass
// is the cheaper one while
//   pos + 1 <= kDenseRatio * (P + k)   (always when pos < P + k).
// The split falls on a whole dense tile pair unless every query goes dense.
constexpr int64_t kDenseRatio = 10;

struct PrefillPlan {
  int n_dense = 0;       // queries [0, n_dense) dense
  size_t mask = 0;       // bytes of the dense pass's bitmap (workspace offset 0)
  dsa::QS rest{};        // the gathered queries
  Layout L;              // their workspace, at offset `mask`
  size_t total = 0;
};

// The dense pass addresses cache slots through a tensor map, whose dimensions
// stop at 2^32 elements: larger pools take the gathered path only.
bool dense_pool_ok(const dsa::KV& kv) { return (int64_t)kv.num_blocks * 64 <= (int64_t(1) << 32); }

int auto_dense_queries(const dsa::KV& kv, const dsa::QS& qs, int32_t k, int32_t hq, int32_t prefix) {
  if (!dense_pool_ok(kv)) return 0;
  const int64_t lim = kDenseRatio * ((int64_t)prefix + k) - qs.pos0;
  if (lim <= 0) return 0;
  if (lim >= qs.n_q) return qs.n_q;
  const int pair = 2 * dsa::dense_tile_queries(hq / kv.hkv);
  return (int)(lim / pair * pair);
}

PrefillPlan prefill_plan(const dsa::KV& kv, const dsa::QS& qs, int32_t k, int32_t hq, int32_t prefix, int n_dense) {
  PrefillPlan pl;
  pl.n_dense = n_dense;
  pl.mask = up256(dsa::dense_mask_bytes(qs, n_dense));
  pl.rest = dsa::QS{qs.mode, qs.n_q - n_dense, qs.seq, qs.pos0 + n_dense};
  if (pl.rest.n_q > 0) pl.L = layout(kv, pl.rest, k, hq, prefix);
  pl.total = pl.mask + pl.L.total;
  return pl;
}

dsa_status attn_impl(const dsa_paged_kv* kv_, const dsa_query_set* qs_, const void* q, int32_t hq,
                     const int32_t* idx, const int32_t* n_sel, int32_t k, int32_t prefix, float scale, void* out,
                     int32_t out_dtype, float* lse, void* ws, size_t ws_bytes, cudaStream_t stream,
                     int32_t n_dense = -1, bool mask_ready = false) {
  dsa::KV kv{};
  dsa::QS qs{};
  DSA_TRY(check_kv(kv_, &kv));
  DSA_TRY(check_qs(qs_, kv, &qs));
  DSA_TRY(check_k_prefix(k, prefix));
  DSA_TRY(check_heads(hq, kv));
  DSA_TRY(check_tiles(kv, qs, k, prefix));
  if (!q || !aligned16(q) || !out || !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
  if (!idx || !n_sel) return fail(DSA_ERR_INVALID_ARG, "idx and n_sel must be non-NULL");
  if (out_dtype != DSA_OUT_BF16 && out_dtype != DSA_OUT_F32)
    return fail(DSA_ERR_INVALID_ARG, "out_dtype %d is neither DSA_OUT_BF16 nor DSA_OUT_F32", out_dtype);
  if (!std::isfinite(scale)) return fail(DSA_ERR_INVALID_ARG, "softmax_scale must be finite");
  if (qs.mode == DSA_MODE_PREFILL) {
    if (n_dense < -1 || n_dense > qs.n_q)
      return fail(DSA_ERR_INVALID_ARG, "n_dense (%d) must be -1 (automatic) or in [0, n_q]", n_dense);
    if (n_dense < 0) n_dense = auto_dense_queries(kv, qs, k, hq, prefix);
    if (n_dense > 0 && !dense_pool_ok(kv))
      return fail(DSA_ERR_UNSUPPORTED, "the dense prefill pass needs num_blocks * 64 <= 2^32");
    const PrefillPlan pl = prefill_plan(kv, qs, k, hq, prefix, n_dense);
    DSA_TRY(check_ws(ws, ws_bytes, pl.total));
    DSA_TRY(ensure_setup());
    dsa::AttnArgs a;
    a.kv = kv;
    a.qs = qs;
    a.q = q;
    a.hq = hq;
    a.idx = idx;
    a.n_sel = n_sel;
    a.slot = nullptr;
    a.k = k;
    a.prefix = prefix;
    a.scale = scale;
    a.out = out;
    a.out_dtype = out_dtype;
    a.lse = lse;
    if (pl.n_dense > 0)
      DSA_CUDA("dense prefill attention launch", dsa::launch_dense_attn(a, pl.n_dense, ws, stream, 0, mask_ready));
    if (pl.rest.n_q == 0) return DSA_OK;
    const size_t nd = (size_t)pl.n_dense, row = (size_t)hq * 128;
    a.qs = pl.rest;
    a.q = static_cast<const char*>(q) + nd * row * 2;
    a.idx = idx + nd * (size_t)k;
    a.n_sel = n_sel + nd;
    a.out = static_cast<char*>(out) + nd * row * (out_dtype == DSA_OUT_F32 ? 4 : 2);
    a.lse = lse ? lse + nd * (size_t)hq : nullptr;
    a.ws = attn_ws(pl.L, static_cast<char*>(ws) + pl.mask);
    DSA_CUDA("sparse attention launch", dsa::launch_sparse_attn(a, stream));
    return DSA_OK;
  }
  const Layout L = layout(kv, qs, k, hq, prefix);
  DSA_TRY(check_ws(ws, ws_bytes, L.total));
  DSA_TRY(ensure_setup());
  dsa::AttnArgs a;
  a.kv = kv;
  a.qs = qs;
  a.q = q;
  a.hq = hq;
  a.idx = idx;
  a.n_sel = n_sel;
  a.slot = nullptr;
  a.k = k;
  a.prefix = prefix;
  a.scale = scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.lse = lse;
  a.ws = attn_ws(L, ws);
  DSA_CUDA("sparse attention launch", dsa::launch_sparse_attn(a, stream));
  return DSA_OK;
}

// Local sliding-window attention (the hybrid attention's local sibling): decode
// workspace = index lists [B][window] + counts [B] + the attention partials.
// Decode window attention: the attention's own workspace only (the window's
// rows are walked from each context's end, with no index lists).
struct WindowLayout {
  size_t attn = 0, total = 0;
  Layout L;
};

WindowLayout window_layout(const dsa::KV& kv, int32_t hq, int32_t window) {
  WindowLayout W;
  const dsa::QS qs{DSA_MODE_DECODE, kv.batch, 0, 0};
  W.L = layout(kv, qs, 0, hq, window);
  W.total = W.L.total;
  return W;
}

dsa_status check_window_call(int32_t window, const void* q, const void* out, int32_t out_dtype, float scale) {
  if (window < 1) return fail(DSA_ERR_INVALID_ARG, "window (%d) must be >= 1", window);
  if (window > (1 << 24)) return fail(DSA_ERR_UNSUPPORTED, "window above 2^24");
  if (!q || !aligned16(q) || !out || !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
  if (out_dtype != DSA_OUT_BF16 && out_dtype != DSA_OUT_F32)
    return fail(DSA_ERR_INVALID_ARG, "out_dtype %d is neither DSA_OUT_BF16 nor DSA_OUT_F32", out_dtype);
  if (!std::isfinite(scale)) return fail(DSA_ERR_INVALID_ARG, "softmax_scale must be finite");
  return DSA_OK;
}

// Per-KV-head indexer decode: the (sequence, KV head) pairs run the scoring and
// selection as sequences of their own (virtual block table and context lengths
// in the workspace), the attention as one query per pair over its KV head.
struct HeadsPlan {
  dsa::KV kv2;    // the virtual sequences (scoring and selection)
  dsa::QS qs2;
  dsa::KV kva;    // the attention's view of the cache: one KV head per query
  size_t sel = 0, total = 0;
  Layout L;
};

dsa_status heads_plan(const dsa::KV& kv, int32_t hq, int32_t k, int32_t prefix, HeadsPlan* out) {
  if ((int64_t)kv.batch * kv.hkv > dsa::kMaxDecodeBatch)
    return fail(DSA_ERR_UNSUPPORTED, "per-head indexer: batch x num_kv_heads above %d", dsa::kMaxDecodeBatch);
  if ((int64_t)kv.num_blocks * kv.hkv >= (int64_t(1) << 31) / 64)
    return fail(DSA_ERR_UNSUPPORTED, "per-head indexer: num_blocks x num_kv_heads x 64 must stay below 2^31");
  HeadsPlan h;
  h.kv2 = kv;
  h.kv2.num_blocks = kv.num_blocks * kv.hkv;
  h.kv2.batch = kv.batch * kv.hkv;
  h.qs2 = dsa::QS{DSA_MODE_DECODE, h.kv2.batch, 0, 0};
  h.kva = kv;
  h.kva.hkv = 1;
  h.kva.adjacent = false;
  h.sel = 0;
  h.L = layout(h.kv2, h.qs2, k, hq / kv.hkv, prefix);
  h.total = h.sel + h.L.total;
  *out = h;
  return DSA_OK;
}

}  // namespace

namespace dsa {

// Argument checks and scratch layout of a decode top-k, for entry points that
// bring their own scratch (the allocation-free variant).  On success *st points
// into `base`, *bytes is the scratch size and *clear_bytes the leading part
// (histograms and counters) that must be zero when the call starts.
dsa_status prepare_decode_topk(const dsa_paged_kv* kv_, const int32_t* scores, int32_t ld, int32_t prefix,
                               int32_t k, const int32_t* idx, const int32_t* n_sel, KV* kv_out, size_t* bytes,
                               size_t* clear_bytes) {
  KV kv{};
  QS qs{};
  DSA_TRY(check_kv(kv_, &kv));
  const dsa_query_set qs_ = {DSA_MODE_DECODE, kv.batch, 0, 0};
  DSA_TRY(check_qs(&qs_, kv, &qs));
  DSA_TRY(check_k_prefix(k, prefix));
  DSA_TRY(check_scores(scores, ld, kv, qs));
  if (!idx || !n_sel) return fail(DSA_ERR_INVALID_ARG, "idx and n_sel must be non-NULL");
  const Layout L = layout(kv, qs, k, kv.hkv, prefix);
  *kv_out = kv;
  *bytes = L.sel_end;
  *clear_bytes = L.sel_end;  // the histograms
  return DSA_OK;
}

SelState decode_topk_state(const KV& kv, int32_t k, int32_t prefix, void* base) {
  const dsa_query_set qs_ = {DSA_MODE_DECODE, kv.batch, 0, 0};
  QS qs{qs_.mode, qs_.n_q, qs_.seq, qs_.pos0};
  return sel_state(layout(kv, qs, k, kv.hkv, prefix), base, false);
}

dsa_status set_error(dsa_status s, const char* msg) { return fail(s, "%s", msg); }

dsa_status setup_device() { return ensure_setup(); }

}  // namespace dsa

extern "C" {

const char* dsa_status_string(dsa_status s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_OOM: return "DSA_ERR_OOM";
    case DSA_ERR_BAD_BLOCK_TABLE: return "DSA_ERR_BAD_BLOCK_TABLE";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
  }
  return "DSA_ERR_UNKNOWN";
}

const char* dsa_last_error_message(void) { return g_msg.c_str(); }

int32_t dsa_abi_version(void) { return DSA_ABI_VERSION; }

dsa_status dsa_check_device_status(cudaStream_t stream, int32_t* code) {
  if (!code) return fail(DSA_ERR_INVALID_ARG, "code is NULL");
  int c = 0;
  DSA_CUDA("status (index)", dsa::read_clear_status_index(&c, stream));
  DSA_CUDA("status (top-k)", dsa::read_clear_status_topk(&c, stream));
  DSA_CUDA("status (attention)", dsa::read_clear_status_attn(&c, stream));
  DSA_CUDA("status (prefix attention)", dsa::read_clear_status_prefix(&c, stream));
  DSA_CUDA("status (cache)", dsa::read_clear_status_misc(&c, stream));
  DSA_CUDA("status (dense prefill attention)", dsa::read_clear_status_dense(&c, stream));
  DSA_CUDA("status (fused prefill selection)", dsa::read_clear_status_pselect(&c, stream));
  *code = c;
  return DSA_OK;
}

size_t dsa_workspace_size(int32_t op, const dsa_paged_kv* kv_, const dsa_query_set* qs_, int32_t k, int32_t hq,
                          int32_t prefix) {
  dsa::KV kv{};
  dsa::QS qs{};
  if (check_kv(kv_, &kv) != DSA_OK || check_qs(qs_, kv, &qs) != DSA_OK) return 0;
  if (op == DSA_OP_INDEX_SCORES) return 0;
  if (check_k_prefix(k, prefix) != DSA_OK || check_heads(hq, kv) != DSA_OK) return 0;
  const Layout L = layout(kv, qs, k, hq, prefix);
  if (qs.mode == DSA_MODE_PREFILL && (op == DSA_OP_SPARSE_ATTN || op == DSA_OP_PREFILL_STEP))
    return prefill_plan(kv, qs, k, hq, prefix, auto_dense_queries(kv, qs, k, hq, prefix)).total;
  switch (op) {
    case DSA_OP_TOPK_SELECT: return L.sel_end;
    case DSA_OP_SPARSE_ATTN:
    case DSA_OP_DECODE_STEP:
    case DSA_OP_PREFILL_STEP: return L.total;
    default: fail(DSA_ERR_INVALID_ARG, "unknown op %d", op); return 0;
  }
}

dsa_status dsa_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (ws_bytes == 0) return DSA_OK;
  if (!ws) return fail(DSA_ERR_WORKSPACE, "workspace is NULL");
  DSA_CUDA("workspace memset", cudaMemsetAsync(ws, 0, ws_bytes, stream));
  return DSA_OK;
}

dsa_status dsa_kv_write(const dsa_paged_kv* kv_, const int32_t* slots, int32_t ntok, const void* k, const void* v,
                        const int8_t* idx_k, cudaStream_t stream) {
  dsa::KV kv{};
  DSA_TRY(check_kv(kv_, &kv));
  if (ntok < 0) return fail(DSA_ERR_INVALID_ARG, "ntok (%d) must be >= 0", ntok);
  if (ntok == 0) return DSA_OK;
  if (!slots || !k || !v || !idx_k) return fail(DSA_ERR_INVALID_ARG, "slot_mapping, k, v and idx_k must be non-NULL");
  if (!aligned16(k) || !aligned16(v) || !aligned16(idx_k))
    return fail(DSA_ERR_INVALID_ARG, "k, v and idx_k must be 16-byte aligned");
  DSA_TRY(ensure_setup());
  DSA_CUDA("kv_write launch", dsa::launch_kv_write(kv, slots, ntok, k, v, idx_k, stream));
  return DSA_OK;
}

dsa_status dsa_kv_write_heads(const dsa_paged_kv* kv_, const int32_t* slots, int32_t ntok, const void* k,
                              const void* v, const int8_t* idx_k, cudaStream_t stream) {
  dsa::KV kv{};
  DSA_TRY(check_kv(kv_, &kv));
  if (ntok < 0) return fail(DSA_ERR_INVALID_ARG, "ntok (%d) must be >= 0", ntok);
  if (ntok == 0) return DSA_OK;
  if (!slots || !k || !v || !idx_k)
    return fail(DSA_ERR_INVALID_ARG, "slot_mapping_heads, k, v and idx_k must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(slots) & 3) || !aligned16(k) || !aligned16(v) || !aligned16(idx_k))
    return fail(DSA_ERR_INVALID_ARG, "slot_mapping_heads must be 4-byte aligned, k, v and idx_k 16-byte aligned");
  DSA_TRY(ensure_setup());
  DSA_CUDA("kv_write_heads launch", dsa::launch_kv_write_heads(kv, slots, ntok, k, v, idx_k, stream));
  return DSA_OK;
}

dsa_status dsa_index_scores(const dsa_paged_kv* kv_, const dsa_query_set* qs_, const int8_t* q_idx, int32_t prefix,
                            int32_t* scores, int32_t ld, void* ws, size_t ws_bytes, cudaStream_t stream) {
  (void)ws;
  (void)ws_bytes;
  dsa::KV kv{};
  dsa::QS qs{};
  DSA_TRY(check_kv(kv_, &kv));
  DSA_TRY(check_qs(qs_, kv, &qs));
  if (prefix < 0) return fail(DSA_ERR_INVALID_ARG, "prefix_len (%d) must be >= 0", prefix);
  if (!q_idx || !aligned16(q_idx)) return fail(DSA_ERR_INVALID_ARG, "q_idx must be non-NULL and 16-byte aligned");
  DSA_TRY(check_scores(scores, ld, kv, qs));
  DSA_TRY(ensure_setup());
  if (qs.mode == DSA_MODE_DECODE)
    DSA_CUDA("index_scores launch", dsa::launch_decode_index(kv, q_idx, prefix, scores, ld, nullptr, 0, stream));
  else
    DSA_CUDA("index_scores launch", dsa::launch_prefill_index(kv, qs, q_idx, prefix, scores, ld, stream));
  return DSA_OK;
}

dsa_status dsa_topk_select(const dsa_paged_kv* kv_, const dsa_query_set* qs_, const int32_t* scores, int32_t ld,
                           int32_t prefix, int32_t k, int32_t* idx, int32_t* n_sel, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  dsa::KV kv{};
  dsa::QS qs{};
  DSA_TRY(check_kv(kv_, &kv));
  DSA_TRY(check_qs(qs_, kv, &qs));
  DSA_TRY(check_k_prefix(k, prefix));
  DSA_TRY(check_scores(scores, ld, kv, qs));
  if (!idx || !n_sel) return fail(DSA_ERR_INVALID_ARG, "idx and n_sel must be non-NULL");
  if (qs.mode == DSA_MODE_DECODE) {
    const Layout L = layout(kv, qs, k, kv.hkv, prefix);
    DSA_TRY(check_ws(ws, ws_bytes, L.sel_end));
    DSA_TRY(ensure_setup());
    const dsa::SelState s = sel_state(L, ws, false);
    DSA_CUDA("top-k histogram launch", dsa::launch_decode_hist(kv, scores, ld, prefix, k, s, stream));
    DSA_CUDA("top-k selection launch", dsa::launch_decode_select(kv, scores, ld, prefix, k, s, idx, n_sel, stream));
  } else {
    DSA_TRY(ensure_setup());
    DSA_CUDA("top-k launch", dsa::launch_prefill_topk(qs, scores, ld, prefix, k, idx, n_sel, stream));
  }
  return DSA_OK;
}

dsa_status dsa_prefill_step(const dsa_paged_kv* kv_, const dsa_query_set* qs_, const void* q, const int8_t* q_idx,
                            int32_t hq, int32_t prefix, int32_t k, float scale, int32_t* scores, int32_t ld,
                            int32_t* idx, int32_t* n_sel, void* out, int32_t out_dtype, float* lse, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  dsa::KV kv{};
  dsa::QS qs{};
  DSA_TRY(check_kv(kv_, &kv));
  if (qs_ && qs_->mode != DSA_MODE_PREFILL)
    return fail(DSA_ERR_INVALID_ARG, "dsa_prefill_step needs a DSA_MODE_PREFILL query set");
  DSA_TRY(check_qs(qs_, kv, &qs));
  DSA_TRY(check_k_prefix(k, prefix));
  DSA_TRY(check_heads(hq, kv));
  DSA_TRY(check_tiles(kv, qs, k, prefix));
  if (!q_idx || !aligned16(q_idx)) return fail(DSA_ERR_INVALID_ARG, "q_idx must be non-NULL and 16-byte aligned");
  DSA_TRY(check_scores(scores, ld, kv, qs));
  if (!idx || !n_sel) return fail(DSA_ERR_INVALID_ARG, "idx and n_sel must be non-NULL");
  if (!q || !aligned16(q) || !out || !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
  if (out_dtype != DSA_OUT_BF16 && out_dtype != DSA_OUT_F32)
    return fail(DSA_ERR_INVALID_ARG, "out_dtype %d is neither DSA_OUT_BF16 nor DSA_OUT_F32", out_dtype);
  if (!std::isfinite(scale)) return fail(DSA_ERR_INVALID_ARG, "softmax_scale must be finite");
  const int n_dense = auto_dense_queries(kv, qs, k, hq, prefix);
  const PrefillPlan pl = prefill_plan(kv, qs, k, hq, prefix, n_dense);
  DSA_TRY(check_ws(ws, ws_bytes, pl.total));
  DSA_TRY(ensure_setup());
  // The top-k writes the dense queries' attended-position bitmap as it writes
  // their index lists (the attention then needs no pass over the lists).
  uint64_t* mask = n_dense > 0 ? static_cast<uint64_t*>(ws) : nullptr;
  if (mask) DSA_CUDA("bitmap clear", cudaMemsetAsync(mask, 0, dsa::dense_mask_bytes(qs, n_dense), stream));
  DSA_CUDA("index_scores launch", dsa::launch_prefill_index(kv, qs, q_idx, prefix, scores, ld, stream));
  DSA_CUDA("top-k launch", dsa::launch_prefill_topk(qs, scores, ld, prefix, k, idx, n_sel, stream, mask, n_dense,
                                                   (n_dense + 1) & ~1));
  return attn_impl(kv_, qs_, q, hq, idx, n_sel, k, prefix, scale, out, out_dtype, lse, ws, ws_bytes, stream, n_dense,
                   true);
}

dsa_status dsa_kv_gather(const dsa_paged_kv* kv_, const dsa_query_set* qs_, const int32_t* idx, const int32_t* n_sel,
                         int32_t k, int32_t prefix, void* k_out, void* v_out, cudaStream_t stream) {
  dsa::KV kv{};
  dsa::QS qs{};
  DSA_TRY(check_kv(kv_, &kv));
  DSA_TRY(check_qs(qs_, kv, &qs));
  DSA_TRY(check_k_prefix(k, prefix));
  if (!idx || !n_sel) return fail(DSA_ERR_INVALID_ARG, "idx and n_sel must be non-NULL");
  if (!k_out || !v_out || !aligned16(k_out) || !aligned16(v_out))
    return fail(DSA_ERR_INVALID_ARG, "k_out and v_out must be non-NULL and 16-byte aligned");
  DSA_TRY(ensure_setup());
  DSA_CUDA("kv_gather launch", dsa::launch_kv_gather(kv, qs, idx, n_sel, k, prefix, k_out, v_out, stream));
  return DSA_OK;
}

// Device-side address of one end of a staging copy: device or managed memory
// as it is, page-locked host memory through its device mapping; anything else
// (pageable host memory, unknown pointers) is refused before any launch.
static dsa_status staging_address(const void* ptr, const char* name, const void** out) {
  cudaPointerAttributes at{};
  const cudaError_t e = cudaPointerGetAttributes(&at, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DSA_ERR_INVALID_ARG, "%s: not a pointer the CUDA runtime knows (%s)", name, cudaGetErrorString(e));
  }
  if (at.type == cudaMemoryTypeDevice) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != at.device)
      return fail(DSA_ERR_INVALID_ARG, "%s is device memory of device %d, not of the current device %d", name,
                  at.device, dev);
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    *out = ptr;
    return DSA_OK;
  }
  if (at.type == cudaMemoryTypeHost && at.devicePointer) {
    *out = at.devicePointer;
    return DSA_OK;
  }
  return fail(DSA_ERR_INVALID_ARG, "%s must be device memory or page-locked host memory", name);
}

dsa_status dsa_copy_async(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
  if (!dst || !src) return fail(DSA_ERR_INVALID_ARG, "dst and src must be non-NULL");
  if (!aligned16(dst) || !aligned16(src) || bytes % 16 != 0)
    return fail(DSA_ERR_INVALID_ARG, "dst and src must be 16-byte aligned and bytes a multiple of 16 (got %zu)", bytes);
  if (bytes == 0) return DSA_OK;
  const void* d_src = nullptr;
  const void* d_dst = nullptr;
  DSA_TRY(staging_address(src, "src", &d_src));
  DSA_TRY(staging_address(dst, "dst", &d_dst));
  if (!aligned16(d_src) || !aligned16(d_dst))
    return fail(DSA_ERR_INVALID_ARG, "the device-side addresses of dst and src must be 16-byte aligned");
  const char* s0 = static_cast<const char*>(d_src);
  const char* d0 = static_cast<const char*>(d_dst);
  if (s0 < d0 + bytes && d0 < s0 + bytes) return fail(DSA_ERR_INVALID_ARG, "dst and src overlap");
  DSA_TRY(ensure_setup());
  DSA_CUDA("staging copy launch", dsa::launch_stage_copy(const_cast<void*>(d_dst), d_src, bytes, stream));
  return DSA_OK;
}

dsa_status dsa_sparse_attn_decode(const dsa_paged_kv* kv, const void* q, int32_t hq, const int32_t* idx,
                                  const int32_t* n_sel, int32_t k, int32_t prefix, float scale, void* out,
                                  int32_t out_dtype, float* lse, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!kv) return fail(DSA_ERR_INVALID_ARG, "kv descriptor is NULL");
  dsa_query_set qs = {DSA_MODE_DECODE, kv->batch, 0, 0};
  return attn_impl(kv, &qs, q, hq, idx, n_sel, k, prefix, scale, out, out_dtype, lse, ws, ws_bytes, stream);
}

dsa_status dsa_sparse_attn_prefill(const dsa_paged_kv* kv, const dsa_query_set* qs, const void* q, int32_t hq,
                                   const int32_t* idx, const int32_t* n_sel, int32_t k, int32_t prefix, float scale,
                                   void* out, int32_t out_dtype, float* lse, void* ws, size_t ws_bytes,
                                   cudaStream_t stream) {
  if (qs && qs->mode != DSA_MODE_PREFILL)
    return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_attn_prefill needs a DSA_MODE_PREFILL query set");
  return attn_impl(kv, qs, q, hq, idx, n_sel, k, prefix, scale, out, out_dtype, lse, ws, ws_bytes, stream);
}

dsa_status dsa_sparse_attn_prefill_split(const dsa_paged_kv* kv, const dsa_query_set* qs, const void* q,
                                         int32_t hq, const int32_t* idx, const int32_t* n_sel, int32_t k,
                                         int32_t prefix, float scale, int32_t n_dense, void* out, int32_t out_dtype,
                                         float* lse, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (qs && qs->mode != DSA_MODE_PREFILL)
    return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_attn_prefill_split needs a DSA_MODE_PREFILL query set");
  return attn_impl(kv, qs, q, hq, idx, n_sel, k, prefix, scale, out, out_dtype, lse, ws, ws_bytes, stream, n_dense);
}

int32_t dsa_prefill_dense_queries(const dsa_paged_kv* kv_, const dsa_query_set* qs_, int32_t k, int32_t hq,
                                  int32_t prefix) {
  dsa::KV kv{};
  dsa::QS qs{};
  if (check_kv(kv_, &kv) != DSA_OK || check_qs(qs_, kv, &qs) != DSA_OK || qs.mode != DSA_MODE_PREFILL) return -1;
  if (check_k_prefix(k, prefix) != DSA_OK || check_heads(hq, kv) != DSA_OK) return -1;
  return auto_dense_queries(kv, qs, k, hq, prefix);
}

size_t dsa_prefill_attn_workspace_size(const dsa_paged_kv* kv_, const dsa_query_set* qs_, int32_t k, int32_t hq,
                                       int32_t prefix, int32_t n_dense) {
  dsa::KV kv{};
  dsa::QS qs{};
  if (check_kv(kv_, &kv) != DSA_OK || check_qs(qs_, kv, &qs) != DSA_OK) return 0;
  if (qs.mode != DSA_MODE_PREFILL) {
    fail(DSA_ERR_INVALID_ARG, "dsa_prefill_attn_workspace_size needs a DSA_MODE_PREFILL query set");
    return 0;
  }
  if (check_k_prefix(k, prefix) != DSA_OK || check_heads(hq, kv) != DSA_OK) return 0;
  if (n_dense < -1 || n_dense > qs.n_q) {
    fail(DSA_ERR_INVALID_ARG, "n_dense (%d) must be -1 (automatic) or in [0, n_q = %d]", n_dense, qs.n_q);
    return 0;
  }
  if (n_dense < 0) n_dense = auto_dense_queries(kv, qs, k, hq, prefix);
  return prefill_plan(kv, qs, k, hq, prefix, n_dense).total;
}

dsa_status dsa_prefill_select(const dsa_paged_kv* kv_, const dsa_query_set* qs_, const int8_t* q_idx,
                              int32_t prefix, int32_t k, int32_t* idx, int32_t* n_sel, cudaStream_t stream) {
  dsa::KV kv{};
  dsa::QS qs{};
  DSA_TRY(check_kv(kv_, &kv));
  if (qs_ && qs_->mode != DSA_MODE_PREFILL)
    return fail(DSA_ERR_INVALID_ARG, "dsa_prefill_select needs a DSA_MODE_PREFILL query set");
  DSA_TRY(check_qs(qs_, kv, &qs));
  DSA_TRY(check_k_prefix(k, prefix));
  if (!q_idx || !aligned16(q_idx)) return fail(DSA_ERR_INVALID_ARG, "q_idx must be non-NULL and 16-byte aligned");
  if (!idx || !n_sel) return fail(DSA_ERR_INVALID_ARG, "idx and n_sel must be non-NULL");
  DSA_TRY(ensure_setup());
  DSA_CUDA("fused prefill selection launch", dsa::launch_prefill_select(kv, qs, q_idx, prefix, k, idx, n_sel, stream));
  return DSA_OK;
}

size_t dsa_heads_workspace_size(const dsa_paged_kv* kv_, int32_t hq, int32_t k, int32_t prefix) {
  dsa::KV kv{};
  if (check_kv(kv_, &kv) != DSA_OK || check_heads(hq, kv) != DSA_OK || check_k_prefix(k, prefix) != DSA_OK) return 0;
  HeadsPlan h;
  if (heads_plan(kv, hq, k, prefix, &h) != DSA_OK) return 0;
  return h.total;
}

dsa_status dsa_decode_step_heads(const dsa_paged_kv* kv_, const void* q, const int8_t* q_idx,
                                 const int32_t* block_table_heads, int32_t hq, int32_t prefix, int32_t k, float scale,
                                 int32_t* scores, int32_t ld, int32_t* idx,
                                 int32_t* n_sel, void* out, int32_t out_dtype, float* lse, void* ws, size_t ws_bytes,
                                 cudaStream_t stream) {
  dsa::KV kv{};
  DSA_TRY(check_kv(kv_, &kv));
  const dsa_query_set qs_ = {DSA_MODE_DECODE, kv.batch, 0, 0};
  dsa::QS qs{};
  DSA_TRY(check_qs(&qs_, kv, &qs));
  DSA_TRY(check_k_prefix(k, prefix));
  DSA_TRY(check_heads(hq, kv));
  HeadsPlan h;
  DSA_TRY(heads_plan(kv, hq, k, prefix, &h));
  DSA_TRY(check_tiles(kv, h.qs2, k, prefix));
  if (!q_idx || !aligned16(q_idx)) return fail(DSA_ERR_INVALID_ARG, "q_idx must be non-NULL and 16-byte aligned");
  if (block_table_heads && (reinterpret_cast<uintptr_t>(block_table_heads) & 3))
    return fail(DSA_ERR_INVALID_ARG, "block_table_heads must be 4-byte aligned");
  DSA_TRY(check_scores(scores, ld, h.kv2, h.qs2));
  if (!idx || !n_sel) return fail(DSA_ERR_INVALID_ARG, "idx and n_sel must be non-NULL");
  if (!q || !aligned16(q) || !out || !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
  if (out_dtype != DSA_OUT_BF16 && out_dtype != DSA_OUT_F32)
    return fail(DSA_ERR_INVALID_ARG, "out_dtype %d is neither DSA_OUT_BF16 nor DSA_OUT_F32", out_dtype);
  if (!std::isfinite(scale)) return fail(DSA_ERR_INVALID_ARG, "softmax_scale must be finite");
  DSA_TRY(check_ws(ws, ws_bytes, h.total));
  DSA_TRY(ensure_setup());
  char* w = static_cast<char*>(ws);
  // The (sequence, KV head) pairs are the rows of the scoring and the
  // selection: row b * Hkv + h scores head h's indexer keys (block blk * Hkv + h
  // of the indexer cache, blk from the shared table or from head h's own) with
  // its sequence's context length; the attention reads head h's K and V rows
  // of the same blocks.  The kernels map the rows themselves, so the scoring
  // kernel starts early as in dsa_decode_step.
  const dsa::KV kv2 = h.kv2;
  const dsa::SelState s2 = sel_state(h.L, w + h.sel, false);  // no cache slots: the attention resolves positions
  DSA_CUDA("decode index launch", dsa::launch_decode_index(kv2, q_idx, prefix, scores, ld, &s2, k, stream, true,
                                                           kv.hkv, block_table_heads));
  int c_cap, prefix_ctas;
  overlap_shape(h.kv2, prefix, &c_cap, &prefix_ctas);
  DSA_CUDA("decode selection launch",
           dsa::launch_decode_select(kv2, scores, ld, prefix, k, s2, idx, n_sel, stream, c_cap, kv.hkv));
  dsa::AttnArgs a;
  a.prefix_ctas = prefix_ctas;
  a.kv = h.kva;
  if (block_table_heads) {  // head h of sequence b reads row h * batch + b of the per-head tables
    a.kv.block_table = block_table_heads;
    a.bt_head_rows = kv.batch;
  }
  a.qs = h.qs2;
  a.q = q;
  a.hq = hq / kv.hkv;
  a.idx = idx;
  a.n_sel = n_sel;
  a.slot = nullptr;
  a.k = k;
  a.prefix = prefix;
  a.scale = scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.lse = lse;
  a.ws = attn_ws(h.L, w + h.sel);
  a.hsplit = kv.hkv;
  DSA_CUDA("decode attention launch", dsa::launch_sparse_attn(a, stream));
  return DSA_OK;
}

size_t dsa_window_workspace_size(const dsa_paged_kv* kv_, int32_t hq, int32_t window) {
  dsa::KV kv{};
  if (check_kv(kv_, &kv) != DSA_OK || check_heads(hq, kv) != DSA_OK) return 0;
  if (window < 1 || window > (1 << 24)) {
    fail(DSA_ERR_INVALID_ARG, "window (%d) must be in [1, 2^24]", window);
    return 0;
  }
  return window_layout(kv, hq, window).total;
}

dsa_status dsa_window_attn_decode(const dsa_paged_kv* kv_, const void* q, int32_t hq, int32_t window, float scale,
                                  void* out, int32_t out_dtype, float* lse, void* ws, size_t ws_bytes,
                                  cudaStream_t stream) {
  dsa::KV kv{};
  DSA_TRY(check_kv(kv_, &kv));
  const dsa_query_set qs_ = {DSA_MODE_DECODE, kv.batch, 0, 0};
  dsa::QS qs{};
  DSA_TRY(check_qs(&qs_, kv, &qs));
  DSA_TRY(check_heads(hq, kv));
  DSA_TRY(check_window_call(window, q, out, out_dtype, scale));
  DSA_TRY(check_tiles(kv, qs, window, 0));
  const WindowLayout W = window_layout(kv, hq, window);
  DSA_TRY(check_ws(ws, ws_bytes, W.total));
  DSA_TRY(ensure_setup());
  char* w = static_cast<char*>(ws);
  // The window's rows are contiguous: the attention walks them as the
  // query's prefix part from the window's start, with no index lists.
  dsa::AttnArgs a;
  a.kv = kv;
  a.qs = qs;
  a.q = q;
  a.hq = hq;
  a.idx = nullptr;
  a.n_sel = nullptr;
  a.slot = nullptr;
  a.window = window;
  a.k = 0;
  a.prefix = window;
  a.scale = scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.lse = lse;
  a.ws = attn_ws(W.L, w + W.attn);
  DSA_CUDA("window attention launch", dsa::launch_sparse_attn(a, stream));
  return DSA_OK;
}

dsa_status dsa_window_attn_prefill(const dsa_paged_kv* kv_, const dsa_query_set* qs_, const void* q, int32_t hq,
                                   int32_t window, float scale, void* out, int32_t out_dtype, float* lse,
                                   cudaStream_t stream) {
  dsa::KV kv{};
  dsa::QS qs{};
  DSA_TRY(check_kv(kv_, &kv));
  if (qs_ && qs_->mode != DSA_MODE_PREFILL)
    return fail(DSA_ERR_INVALID_ARG, "dsa_window_attn_prefill needs a DSA_MODE_PREFILL query set");
  DSA_TRY(check_qs(qs_, kv, &qs));
  DSA_TRY(check_heads(hq, kv));
  DSA_TRY(check_window_call(window, q, out, out_dtype, scale));
  if (!dense_pool_ok(kv)) return fail(DSA_ERR_UNSUPPORTED, "window prefill needs num_blocks * 64 <= 2^32");
  DSA_TRY(ensure_setup());
  dsa::AttnArgs a;
  a.kv = kv;
  a.qs = qs;
  a.q = q;
  a.hq = hq;
  a.idx = nullptr;
  a.n_sel = nullptr;
  a.slot = nullptr;
  a.k = 0;
  a.prefix = 0;
  a.scale = scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.lse = lse;
  DSA_CUDA("window prefill launch", dsa::launch_dense_attn(a, qs.n_q, nullptr, stream, window));
  return DSA_OK;
}

dsa_status dsa_decode_step(const dsa_paged_kv* kv_, const void* q, const int8_t* q_idx, int32_t hq, int32_t prefix,
                           int32_t k, float scale, int32_t* scores, int32_t ld, int32_t* idx, int32_t* n_sel,
                           void* out, int32_t out_dtype, float* lse, void* ws, size_t ws_bytes, cudaStream_t stream) {
  dsa::KV kv{};
  DSA_TRY(check_kv(kv_, &kv));
  const dsa_query_set qs_ = {DSA_MODE_DECODE, kv.batch, 0, 0};
  dsa::QS qs{};
  DSA_TRY(check_qs(&qs_, kv, &qs));
  DSA_TRY(check_k_prefix(k, prefix));
  DSA_TRY(check_heads(hq, kv));
  DSA_TRY(check_tiles(kv, qs, k, prefix));
  if (!q_idx || !aligned16(q_idx)) return fail(DSA_ERR_INVALID_ARG, "q_idx must be non-NULL and 16-byte aligned");
  DSA_TRY(check_scores(scores, ld, kv, qs));
  if (!idx || !n_sel) return fail(DSA_ERR_INVALID_ARG, "idx and n_sel must be non-NULL");
  if (!q || !aligned16(q) || !out || !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
  if (out_dtype != DSA_OUT_BF16 && out_dtype != DSA_OUT_F32)
    return fail(DSA_ERR_INVALID_ARG, "out_dtype %d is neither DSA_OUT_BF16 nor DSA_OUT_F32", out_dtype);
  if (!std::isfinite(scale)) return fail(DSA_ERR_INVALID_ARG, "softmax_scale must be finite");
  const Layout L = layout(kv, qs, k, hq, prefix);
  DSA_TRY(check_ws(ws, ws_bytes, L.total));
  DSA_TRY(ensure_setup());
  const dsa::SelState s = sel_state(L, ws, true);
  int c_cap, prefix_ctas;
  overlap_shape(kv, prefix, &c_cap, &prefix_ctas);
  DSA_CUDA("decode index launch", dsa::launch_decode_index(kv, q_idx, prefix, scores, ld, &s, k, stream));
  DSA_CUDA("decode selection launch",
           dsa::launch_decode_select(kv, scores, ld, prefix, k, s, idx, n_sel, stream, c_cap));
  dsa::AttnArgs a;
  a.prefix_ctas = prefix_ctas;
  a.kv = kv;
  a.qs = qs;
  a.q = q;
  a.hq = hq;
  a.idx = idx;
  a.n_sel = n_sel;
  a.slot = s.slot;
  a.k = k;
  a.prefix = prefix;
  a.scale = scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.lse = lse;
  a.ws = attn_ws(L, ws);
  DSA_CUDA("decode attention launch", dsa::launch_sparse_attn(a, stream));
  return DSA_OK;
}

}  // extern "C"
