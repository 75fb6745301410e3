// Host-side interface between the C ABI (api.cpp) and the kernel files.
#pragma once

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dsa.h"

namespace dsa {

struct KV {
  const void* k_cache;
  const void* v_cache;
  const int8_t* idx_cache;
  const int32_t* block_table;
  const int32_t* context_lens;
  int num_blocks, hkv, max_blocks, batch, max_ctx;
  int row_stride;  // bf16 values between the K (or V) rows of consecutive slots
  bool adjacent;   // V row right after the K row of the same slot: one piece of 2 * hkv * 256 bytes
};

struct QS {
  int mode, n_q, seq, pos0;
};

// Decode selection state kept in the workspace between the scoring and the
// selection kernels.
struct SelState {
  int* coarse;  // [B][kCoarseBins] coarse score histogram of each sequence; zero between calls
  int* slot;    // [B][k] cache slot (block * 64 + row) of each selected position, or nullptr
};

constexpr int kMaxDecodeBatch = 2048;
constexpr int kMaxDecodeCtx = 1 << 21;  // longest decode context (positions)
constexpr int kMaxAttnCtas = 320;       // persistent attention grid cap (partials are sized for it)
constexpr int kCoarseBinsHost = 1024;   // coarse histogram bins (host-side copy of the device constant)
constexpr int kMaxQHeads = 64;          // query heads per token the attention kernels hold (Q slot in shared memory)

struct AttnWs {
  float2* pre_ml;   // prefill with a prefix: [n_q][Hq] prefix part (max in log2 units, sum), else null
  float* pre_o;     // [n_q][Hq][128] its unnormalised output
  float* part_o;    // [kMaxAttnCtas][slots][Hq][128]  per-CTA partials of split queries (unnormalised O);
                    // two slots per pass: 4 in decode (two passes), 2 in prefill
  float2* part_ml;  // [kMaxAttnCtas][slots][Hq]       (max in log2 units, sum of weights)
};

struct AttnArgs {
  KV kv;
  QS qs;
  const void* q;
  int hq;
  const int32_t* idx;
  const int32_t* n_sel;
  const int32_t* slot;     // cache slots of idx (the fused decode step), or null: the
                           // attention kernel resolves the positions idx itself
  int k, prefix;
  float scale;
  void* out;
  int out_dtype;
  float* lse;
  AttnWs ws;
  int hsplit = 1;  // decode with a per-KV-head indexer: query qi is (sequence qi / hsplit, KV head qi % hsplit)
  int bt_per_query = 0;  // kv.block_table has one row per query (qi), not per sequence
  int bt_head_rows = 0;  // decode, per-head block tables: query qi = (b, h) reads row h * bt_head_rows + b
  int prefix_ctas = 0;  // decode: > 0 walks the prefix rows first, over that many CTAs, before the wait on
                        // the previous kernel (only where that kernel is the step's own selection)
  int window = 0;  // decode: > 0 attends each query's last `window` positions (prefix = window, k = 0,
                   // no index lists): the local sliding-window sibling
};

// Kernel launches (return the launch error, if any).
// hsplit > 1: the per-KV-head indexer over kv.batch = sequences x hsplit rows
// (kv.num_blocks = the KV cache's blocks x hsplit, kv.block_table and
// kv.context_lens those of the sequences; bt_heads: per-head tables or null).
cudaError_t launch_decode_index(const KV& kv, const int8_t* q_idx, int prefix, int* scores, int ld,
                                const SelState* sel, int k, cudaStream_t st, bool early = true, int hsplit = 1,
                                const int32_t* bt_heads = nullptr);
cudaError_t launch_decode_hist(const KV& kv, const int32_t* scores, int ld, int prefix, int k,
                               const SelState& sel, cudaStream_t st);
// Whether the decode selection of this batch runs with one CTA per SM.
bool decode_select_spread(const KV& kv, int prefix);
// c_cap: at most that many CTAs per sequence (the fused step leaves SMs to the
// attention's first pass).
// csplit > 1: kv.batch = sequences x csplit rows, kv.context_lens per sequence.
cudaError_t launch_decode_select(const KV& kv, const int32_t* scores, int ld, int prefix, int k,
                                 const SelState& sel, int32_t* idx, int32_t* n_sel, cudaStream_t st,
                                 int c_cap = 16, int csplit = 1);
// CTAs the decode selection of this batch launches with that cap.
int decode_select_ctas(const KV& kv, int prefix, int c_cap);
// CTAs of the persistent attention grid on the current device.
int attn_grid_ctas();
cudaError_t launch_prefill_index(const KV& kv, const QS& qs, const int8_t* q_idx, int prefix,
                                 int* scores, int ld, cudaStream_t st);
// mask: the dense pass's attended-position bitmap (dense_mask_bytes, zeroed), set
// here for the first n_dense queries (nq_pad as in the dense pass), or null.
cudaError_t launch_prefill_topk(const QS& qs, const int32_t* scores, int ld, int prefix, int k,
                                int32_t* idx, int32_t* n_sel, cudaStream_t st, uint64_t* mask = nullptr,
                                int n_dense = 0, int nq_pad = 0);
cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_prefix_attn(const KV& kv, const QS& qs, const void* q, int hq, int prefix, float scale,
                               float2* pre_ml, float* pre_o, cudaStream_t st);
// Prefill attention of the first n_dense queries of the set as a masked dense
// pass on tcgen05 (k_dense.cu).  window <= 0: the attended sets of the
// selections (a.idx, a.n_sel, a.prefix), with mask_ws holding
// dense_mask_bytes(qs, n_dense); window > 0: the causal window of that many
// positions ending at each query (no workspace).
cudaError_t launch_dense_attn(const AttnArgs& a, int n_dense, void* mask_ws, cudaStream_t st, int window = 0,
                              bool mask_ready = false);  // mask_ready: the bitmap is already in mask_ws
// Decode window attention's index lists: idx[b][j] = L_b - min(window, L_b) + j,
// n_sel[b] = min(window, L_b), -1 past it (k_misc.cu).
size_t dense_mask_bytes(const QS& qs, int n_dense);
int dense_tile_queries(int group);
// Prefill index scores and top-k in one kernel, the scores never written (k_pselect.cu).
cudaError_t launch_prefill_select(const KV& kv, const QS& qs, const int8_t* q_idx, int prefix, int k, int32_t* idx,
                                  int32_t* n_sel, cudaStream_t st);
// Per-head write: slots [ntok][hkv], k / v [ntok][hkv][128], idx_k [ntok][hkv][64]
// into the head slices (indexer cache [blocks][hkv][64][64]).
cudaError_t launch_kv_write_heads(const KV& kv, const int32_t* slots, int ntok, const void* k, const void* v,
                                  const int8_t* idx_k, cudaStream_t st);
cudaError_t launch_kv_write(const KV& kv, const int32_t* slots, int ntok, const void* k, const void* v,
                            const int8_t* idx_k, cudaStream_t st);
// Staging copy by a kernel (device or page-locked host memory on either side;
// device-side addresses, 16-byte aligned, bytes a multiple of 16).
cudaError_t launch_stage_copy(void* dst, const void* src, size_t bytes, cudaStream_t st);
cudaError_t launch_kv_gather(const KV& kv, const QS& qs, const int32_t* idx, const int32_t* n_sel, int k,
                             int prefix, void* k_out, void* v_out, cudaStream_t st);

// One-time per-device kernel attribute setup (dynamic shared memory limits).
cudaError_t setup_index_kernels();
cudaError_t setup_topk_kernels();
cudaError_t setup_attn_kernels();
cudaError_t setup_prefix_kernels();
cudaError_t setup_dense_kernels();
cudaError_t setup_pselect_kernels();

// Device status words, one per kernel file: each reads its word into *code
// (if *code is still 0) and clears it.
cudaError_t read_clear_status_index(int* code, cudaStream_t st);
cudaError_t read_clear_status_topk(int* code, cudaStream_t st);
cudaError_t read_clear_status_attn(int* code, cudaStream_t st);
cudaError_t read_clear_status_prefix(int* code, cudaStream_t st);
cudaError_t read_clear_status_misc(int* code, cudaStream_t st);
cudaError_t read_clear_status_dense(int* code, cudaStream_t st);
cudaError_t read_clear_status_pselect(int* code, cudaStream_t st);

// Used by the allocation-free top-k entry point (defined in api.cpp).
dsa_status prepare_decode_topk(const dsa_paged_kv* kv, const int32_t* scores, int32_t ld, int32_t prefix,
                               int32_t k, const int32_t* idx, const int32_t* n_sel, KV* kv_out, size_t* bytes,
                               size_t* clear_bytes);
SelState decode_topk_state(const KV& kv, int32_t k, int32_t prefix, void* base);
dsa_status set_error(dsa_status s, const char* msg);
dsa_status setup_device();

}  // namespace dsa
