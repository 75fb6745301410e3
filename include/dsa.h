/*
 * dsa.h — C ABI of the dynamic sparse attention (DSA) hot path on GB300 (sm_103a).
 *
 * The method is the one dissected in the article
 *   "国产AI芯片完成前沿大模型Day-0适配:稀疏注意力与混合精度推理全解析" (ruibaoantu.com),
 * section 2; "§2.x" below refers to its sub-sections:
 *   §2.1  index selection on the GPU: a tensor-core similarity score of the query
 *         against every key, then a reduction that picks the top-k positions;
 *   §2.2  the KV cache in fixed blocks (e.g. 64 x 128) of consecutive positions, and
 *         a batched gather of the selected rows ("gather first, then compute");
 *   §2.3  separate prefill (fused select + gather + attention, with the next block
 *         prefetched while the current one is computed) and decode (bandwidth-bound:
 *         load only the active KV, asynchronously) paths;
 *   §2.4  a KV block allocator ("KDA"), and the vision-token prefix that is always
 *         attended in full and never takes part in index selection.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE memory owned by the caller; the library never
 *     allocates, frees or keeps them.  Host pointers are marked "host".
 *   - Hot-path calls are asynchronous on the given stream, never synchronise and
 *     never allocate; they may be captured in a CUDA graph once the library has
 *     made one call on the device (its first call sets kernel attributes).
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED / DSA_ERR_WORKSPACE
 *     and dsa_last_error_message() (per host thread) says which.
 *   - Kernels never trap.  A block-table entry outside [0, num_blocks) read on the
 *     device, or a bounded wait that ran out, sets a device status word and the
 *     kernel goes on with block 0 in its place (outputs then undefined);
 *     dsa_check_device_status() reads and clears it.
 *   - Launch failures return DSA_ERR_CUDA with the CUDA error text.
 *   - Kernels are launched with programmatic dependent launch: each one waits
 *     (griddepcontrol.wait) for the previous kernel of the stream before it touches
 *     anything that kernel may write, and may let the next kernel launch before it
 *     finishes.  Kernels of the caller that follow a call on the same stream either
 *     are launched without that attribute (the default: they start after the call
 *     has completed) or must wait the same way before they read its outputs.
 *
 * Data layout (row-major, innermost last)
 *   k_cache, v_cache : bf16 rows of num_kv_heads * 128 values (every KV head of one position,
 *                      head h at h * 128), one row per cache slot (slot = block * 64 + row),
 *                      slot s at k_cache + s * kv_row_stride (v_cache likewise).  Two layouts:
 *                        separate  kv_row_stride = num_kv_heads * 128 (or 0): k_cache and
 *                                  v_cache are [num_blocks][64][num_kv_heads][128] each;
 *                        adjacent  kv_row_stride = 2 * num_kv_heads * 128 and
 *                                  v_cache = k_cache + num_kv_heads * 128: one array
 *                                  [num_blocks][64][2][num_kv_heads][128], the K and V of a
 *                                  slot one contiguous 2 * num_kv_heads * 256-byte piece, which
 *                                  the attention kernels gather with one copy per position
 *                                  (fewer, larger copies: the faster layout);
 *                      any other stride >= num_kv_heads * 128 (multiple of 8) is accepted too
 *   idx_cache        : int8 [num_blocks][64][64]                   indexer key per position
 *   block_table      : int32 [batch][max_blocks_per_seq]           position t of sequence b is
 *                      row t % 64 of block block_table[b][t / 64]
 *   context_lens     : int32 [batch]                               tokens in the cache per sequence
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 4

typedef enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,      /* null/misaligned pointer, bad size or range        */
  DSA_ERR_UNSUPPORTED = 2,      /* valid but not implemented (e.g. head_dim != 128)  */
  DSA_ERR_OOM = 3,              /* block allocator has too few free blocks           */
  DSA_ERR_BAD_BLOCK_TABLE = 4,  /* device saw a block id outside [0, num_blocks)     */
  DSA_ERR_CUDA = 5,             /* a CUDA call failed                                */
  DSA_ERR_TIMEOUT = 6,          /* a bounded device wait ran out                     */
  DSA_ERR_WORKSPACE = 7         /* workspace pointer null/misaligned or too small    */
} dsa_status;

enum { DSA_MODE_DECODE = 0, DSA_MODE_PREFILL = 1 };
enum { DSA_OUT_BF16 = 0, DSA_OUT_F32 = 1 };
enum {
  DSA_OP_INDEX_SCORES = 0, DSA_OP_TOPK_SELECT = 1, DSA_OP_SPARSE_ATTN = 2,
  DSA_OP_DECODE_STEP = 3, DSA_OP_PREFILL_STEP = 4
};

/* The paged KV cache, described (not owned).  Fixed sizes: block_size 64,
 * head_dim 128, idx_dim 64 (others return DSA_ERR_UNSUPPORTED).
 * max_context_len is a HOST upper bound of context_lens[] (decode) used to size
 * grids; it must be <= max_blocks_per_seq * 64.  kv_row_stride: bf16 values
 * between the K (or V) rows of consecutive slots (see the data layout above;
 * 0 = num_kv_heads * 128). */
typedef struct dsa_paged_kv {
  void* k_cache;
  void* v_cache;
  int8_t* idx_cache;
  const int32_t* block_table;
  const int32_t* context_lens;
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t idx_dim;
  int32_t max_blocks_per_seq;
  int32_t batch;
  int32_t max_context_len;
  int32_t kv_row_stride;
} dsa_paged_kv;

/* Which query tokens a call serves.
 *   DSA_MODE_DECODE : n_q == batch; query b is the newest token of sequence b, at
 *                     position context_lens[b] - 1 (its K, V and indexer key are
 *                     already in the cache).  seq and pos0 are ignored.
 *   DSA_MODE_PREFILL: n_q query tokens of sequence `seq` at positions pos0 .. pos0+n_q-1;
 *                     query i sees keys [0, pos0 + i] (causal, also inside the prefix);
 *                     pos0 + n_q <= max_blocks_per_seq * 64. */
typedef struct dsa_query_set {
  int32_t mode;
  int32_t n_q;
  int32_t seq;
  int32_t pos0;
} dsa_query_set;

/* ---------------------------------------------------------------- status --- */
const char* dsa_status_string(dsa_status s);
/* Message of the last failed call on this host thread ("" if none). */
const char* dsa_last_error_message(void);
int32_t dsa_abi_version(void);
/* Synchronises `stream`, then reads and clears the device status word of the
 * current device.  *code (host) receives DSA_OK, DSA_ERR_BAD_BLOCK_TABLE or
 * DSA_ERR_TIMEOUT; the return value reports CUDA failures only. */
dsa_status dsa_check_device_status(cudaStream_t stream, int32_t* code);

/* --------------------------------------------- block allocator (§2.4 KDA) --- */
/* Host-side free list of block ids [0, num_blocks).  Not thread-safe. */
typedef struct dsa_kv_alloc dsa_kv_alloc;
dsa_status dsa_kv_alloc_create(int32_t num_blocks, dsa_kv_alloc** out /* host */);
/* Takes n free ids into out_ids (host, n entries), lowest ids first.  If fewer
 * than n are free it takes none and returns DSA_ERR_OOM. */
dsa_status dsa_kv_alloc_blocks(dsa_kv_alloc* a, int32_t n, int32_t* out_ids);
/* Returns ids to the free list.  An id out of range or already free makes the
 * whole call fail with DSA_ERR_INVALID_ARG and change nothing. */
dsa_status dsa_kv_free_blocks(dsa_kv_alloc* a, const int32_t* ids /* host */, int32_t n);
int32_t dsa_kv_alloc_num_free(const dsa_kv_alloc* a);
void dsa_kv_alloc_destroy(dsa_kv_alloc* a);

/* Block allocator with one block bitmap per (layer, KV head) (§2.4: the
 * allocator knows the layer and the head and keeps an independent block bitmap
 * per head, so that heads do not overwrite one another's blocks).  A (layer,
 * head) holds the head-h slices of the blocks its bitmap marks, so the same
 * block id may be held by several heads at once for different positions; the
 * per-KV-head decode step (dsa_decode_step_heads) reads each head's blocks
 * through that head's own block table.  Host-side, not thread-safe.
 * create: num_layers, num_heads, num_blocks >= 1 (num_layers x num_heads <=
 * 2^20), else DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED.
 * alloc: the n lowest free ids of (layer, head) into out_ids (host, ascending);
 * DSA_ERR_OOM and nothing taken when fewer are free; layer or head out of
 * range, n < 0 or out_ids NULL with n > 0: DSA_ERR_INVALID_ARG.
 * free: ids (host) must be held by (layer, head), each once; otherwise
 * DSA_ERR_INVALID_ARG and nothing changes.
 * num_free: free ids of (layer, head), -1 for a bad handle or index.
 * words: copies the bitmap (bit i of word i / 64 set when block i is held)
 * into words (host, at least ceil(num_blocks / 64) entries). */
typedef struct dsa_kv_bitmap dsa_kv_bitmap;
dsa_status dsa_kv_bitmap_create(int32_t num_layers, int32_t num_heads, int32_t num_blocks,
                                dsa_kv_bitmap** out /* host */);
dsa_status dsa_kv_bitmap_alloc(dsa_kv_bitmap* a, int32_t layer, int32_t head, int32_t n, int32_t* out_ids);
dsa_status dsa_kv_bitmap_free(dsa_kv_bitmap* a, int32_t layer, int32_t head, const int32_t* ids /* host */,
                              int32_t n);
int32_t dsa_kv_bitmap_num_free(const dsa_kv_bitmap* a, int32_t layer, int32_t head);
dsa_status dsa_kv_bitmap_words(const dsa_kv_bitmap* a, int32_t layer, int32_t head, uint64_t* words /* host */,
                               int32_t n_words);
void dsa_kv_bitmap_destroy(dsa_kv_bitmap* a);

/* ------------------------------------------------------- cache write (§2.2) --- */
/* Scatters ntok new tokens into the cache: token j goes to slot slot_mapping[j]
 * = block_id * 64 + row.  k, v: bf16 [ntok][num_kv_heads][128]; idx_k: int8
 * [ntok][64].  Slots outside the pool set DSA_ERR_BAD_BLOCK_TABLE on the device
 * and are skipped. */
dsa_status dsa_kv_write(const dsa_paged_kv* kv, const int32_t* slot_mapping, int32_t ntok,
                        const void* k, const void* v, const int8_t* idx_k, cudaStream_t stream);
/* Per-head write, for caches whose heads keep their own block tables (the
 * per-(layer, head) block bitmaps, dsa_kv_bitmap_*): token j's head-h K, V and
 * indexer key go to the head-h slice of slot slot_mapping_heads[j][h] only, so
 * heads given the same block never overwrite one another.  slot_mapping_heads:
 * int32 [ntok][num_kv_heads] (device); k, v: bf16 [ntok][num_kv_heads][128];
 * idx_k: int8 [ntok][num_kv_heads][64]; kv->idx_cache: int8
 * [num_blocks][num_kv_heads][64][64] (the per-KV-head indexer's layout).
 * Slots outside the pool set DSA_ERR_BAD_BLOCK_TABLE on the device and are
 * skipped; two (token, head) pairs naming the same slot and head write in no
 * set order. */
dsa_status dsa_kv_write_heads(const dsa_paged_kv* kv, const int32_t* slot_mapping_heads, int32_t ntok,
                              const void* k, const void* v, const int8_t* idx_k, cudaStream_t stream);

/* -------------------------------------------------------------- workspace --- */
/* Bytes of workspace an op needs for these sizes (0 when it needs none, or on
 * invalid arguments: see the message).  A buffer sized for DSA_OP_DECODE_STEP
 * serves every decode op, one sized for DSA_OP_PREFILL_STEP every prefill op.
 * index_scores never needs one; pass NULL / 0 there.  What it holds: per
 * decode sequence a 4 KB coarse score histogram; for the fused decode step the
 * selected cache slots (4 B per query and k); the attention's partial states
 * of queries split over CTAs (about 330 KB per query head); and in prefill
 * with a prefix, the prefix part of every (query, head): 520 B each (272 MB
 * for 16K queries x 32 heads). */
size_t dsa_workspace_size(int32_t op, const dsa_paged_kv* kv, const dsa_query_set* qs,
                          int32_t k, int32_t num_q_heads, int32_t prefix_len);
/* Zeroes a workspace (async on `stream`).  Required once before first use: the
 * ops leave the counters they use at zero again when they finish, so a
 * workspace stays ready; after a failed or interrupted call, call it again. */
dsa_status dsa_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/* ----------------------------------------------------- step 1: scores (§2.1) --- */
/* scores[i * ld + t] = sum_d q_idx[i][d] * key(t)[d] (exact int32) for every
 * candidate key t of query i: t in [prefix_len, pos_i].  Other entries of the row
 * are left untouched.  q_idx: int8 [n_q][64].  ld >= max position + 1, ld % 4 == 0,
 * scores 16-byte aligned. */
dsa_status dsa_index_scores(const dsa_paged_kv* kv, const dsa_query_set* qs, const int8_t* q_idx,
                            int32_t prefix_len, int32_t* scores, int32_t ld,
                            void* ws, size_t ws_bytes, cudaStream_t stream);

/* --------------------------------------------------- step 2: top-k (§2.1, §2.4) --- */
/* For each query: the k candidates t in [prefix_len, pos_i] with the largest
 * scores, ties to the lower position (all candidates when there are <= k).
 * idx: int32 [n_q][k], ascending positions, padded with -1; n_sel: int32 [n_q].
 * The prefix [0, min(prefix_len, pos_i + 1)) is not part of idx: it is always
 * attended (the attention calls add it). */
dsa_status dsa_topk_select(const dsa_paged_kv* kv, const dsa_query_set* qs, const int32_t* scores,
                           int32_t ld, int32_t prefix_len, int32_t k, int32_t* idx, int32_t* n_sel,
                           void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------- prefill steps 1 + 2 without the score matrix --- */
/* The result of dsa_index_scores followed by dsa_topk_select for a prefill
 * query set (same idx / n_sel contract: the k largest scores over
 * [prefix_len, pos_i], ties to the lower position, ascending, -1 padded), with
 * the scores never written: one kernel recomputes each 128-query x 256-key
 * score tile on the tensor cores in three walks over the keys (a 256-bin
 * histogram per query, one-score bins inside the threshold bin, the selected
 * positions), selection fused with scoring as in §2.3's prefill path.  Exact
 * for any int8 values (a CTA whose scores leave [-8192, 8191] runs a
 * three-level radix select instead of the first two walks).  No workspace, no
 * scores buffer.  On GB300 at a 16K chunk it takes 1.19 ms against 0.62 ms for
 * the two separate calls: it trades the score matrix's memory, not time. */
dsa_status dsa_prefill_select(const dsa_paged_kv* kv, const dsa_query_set* qs, const int8_t* q_idx,
                              int32_t prefix_len, int32_t k, int32_t* idx, int32_t* n_sel,
                              cudaStream_t stream);

/* --------------------------------------------------- step 3: gather (§2.2) --- */
/* Copies the attended rows of each query into contiguous buffers
 * k_out, v_out: bf16 [n_q][num_kv_heads][prefix_len + k][128].  Row r of query i:
 * r < P_i = min(prefix_len, pos_i + 1) is position r; P_i <= r < P_i + n_sel[i] is
 * position idx[i][r - P_i]; later rows are zero. */
dsa_status dsa_kv_gather(const dsa_paged_kv* kv, const dsa_query_set* qs, const int32_t* idx,
                         const int32_t* n_sel, int32_t k, int32_t prefix_len,
                         void* k_out, void* v_out, cudaStream_t stream);

/* ------------------------------------------------ step 4: attention (§2.3) --- */
/* out[i][h] = softmax(softmax_scale * q[i][h] . K_S^T) V_S over the attended set
 * S_i = prefix part + idx[i][0 .. n_sel[i]), read straight from the paged cache
 * (the gather is fused).  Query head h uses KV head h / (num_q_heads / num_kv_heads).
 * q: bf16 [n_q][num_q_heads][128]; out: [n_q][num_q_heads][128] bf16 (RNE) or f32;
 * lse: f32 [n_q][num_q_heads] natural-log softmax denominator (may be NULL).
 * Heads: num_q_heads <= 64 (one query's Q, all heads, is staged in a 16 KB
 * shared-memory slot) and num_q_heads / num_kv_heads <= 16; more return
 * DSA_ERR_UNSUPPORTED before anything is launched.
 * Decode form (query set = decode of the whole batch): */
dsa_status dsa_sparse_attn_decode(const dsa_paged_kv* kv, const void* q, int32_t num_q_heads,
                                  const int32_t* idx, const int32_t* n_sel, int32_t k,
                                  int32_t prefix_len, float softmax_scale, void* out,
                                  int32_t out_dtype, float* lse, void* ws, size_t ws_bytes,
                                  cudaStream_t stream);
/* Prefill form: the queries of `qs` (mode DSA_MODE_PREFILL), in two parts
 * (§2.3: selection, gather and attention fused per prefill chunk):
 *   - the first n_dense queries (those at positions below about
 *     10 * (prefix_len + k), where the attended set is a large share of the causal
 *     range; see dsa_prefill_dense_queries) as a masked dense pass on the tensor
 *     cores: every causal position of a tile of queries is read once per tile
 *     and weighted zero unless it is in the query's attended set.  This part
 *     reads the K and V rows of every position up to the tile's last one, so
 *     those rows must hold finite values (any written cache row does); a
 *     selected position outside [0, pos_i] is left out and sets
 *     DSA_ERR_BAD_BLOCK_TABLE on the device;
 *   - the others by gathering their attended rows: with a prefix, the prefix
 *     part of every query first, once per tile of 128 (query, head) rows (§2.4:
 *     the prefix is attended in full by every query), then the selected rows
 *     added to it.
 * The workspace holds the dense part's attended-position bitmap (8 bytes per
 * query and 64 positions) and the gathered part's partial states (see
 * dsa_workspace_size, which sizes the automatic split). */
dsa_status dsa_sparse_attn_prefill(const dsa_paged_kv* kv, const dsa_query_set* qs, const void* q,
                                   int32_t num_q_heads, const int32_t* idx, const int32_t* n_sel,
                                   int32_t k, int32_t prefix_len, float softmax_scale, void* out,
                                   int32_t out_dtype, float* lse, void* ws, size_t ws_bytes,
                                   cudaStream_t stream);
/* The same with the split given: queries [0, n_dense) by the dense pass, the
 * rest by the gather (n_dense = 0: all gathered; n_dense = n_q: all dense;
 * -1: the automatic split).  The workspace must hold
 * dsa_prefill_attn_workspace_size(..., n_dense) bytes. */
dsa_status dsa_sparse_attn_prefill_split(const dsa_paged_kv* kv, const dsa_query_set* qs, const void* q,
                                         int32_t num_q_heads, const int32_t* idx, const int32_t* n_sel,
                                         int32_t k, int32_t prefix_len, float softmax_scale,
                                         int32_t n_dense, void* out, int32_t out_dtype, float* lse,
                                         void* ws, size_t ws_bytes, cudaStream_t stream);
/* The automatic split of dsa_sparse_attn_prefill: the number of leading queries
 * of `qs` it runs as the dense pass (-1 on invalid arguments). */
int32_t dsa_prefill_dense_queries(const dsa_paged_kv* kv, const dsa_query_set* qs, int32_t k,
                                  int32_t num_q_heads, int32_t prefix_len);
/* Workspace bytes of dsa_sparse_attn_prefill_split with this n_dense (-1: the
 * automatic split; 0 on invalid arguments). */
size_t dsa_prefill_attn_workspace_size(const dsa_paged_kv* kv, const dsa_query_set* qs, int32_t k,
                                       int32_t num_q_heads, int32_t prefix_len, int32_t n_dense);

/* ------------------------------- local sliding-window attention (sibling) --- */
/* The hybrid attention's local sub-module ("Qwen3.5在摩尔线程MTT S5000上的原生推理
 * 优化实践", §2.3: global sparse attention, local sliding-window attention and
 * cross-modal attention side by side).  The page gives no definition; the
 * reading taken: query token i at position pos_i attends the causal window
 * [max(0, pos_i - window + 1), pos_i] of its own sequence, no prefix, no
 * selection.  Same q / out / lse layout, head rules (num_q_heads <= 64, group
 * <= 16) and softmax as the sparse attention above; window in [1, 2^24].
 * Decode form: the newest token of every sequence (pos = context_len - 1),
 * through the sparse attention kernels, which walk the window's rows from the
 * end of each context (contiguous positions: no index lists); the workspace
 * holds the attention partials, dsa_window_workspace_size bytes. */
size_t dsa_window_workspace_size(const dsa_paged_kv* kv, int32_t num_q_heads, int32_t window);
dsa_status dsa_window_attn_decode(const dsa_paged_kv* kv, const void* q, int32_t num_q_heads,
                                  int32_t window, float softmax_scale, void* out, int32_t out_dtype,
                                  float* lse, void* ws, size_t ws_bytes, cudaStream_t stream);
/* Prefill form: the queries of `qs` (mode DSA_MODE_PREFILL) through the masked
 * dense pass of dsa_sparse_attn_prefill, its mask the window, its position range
 * starting at the block of each query tile's first window position; no
 * workspace.  As there, the K and V rows of every position in a tile's range
 * must be finite (any written cache row is). */
dsa_status dsa_window_attn_prefill(const dsa_paged_kv* kv, const dsa_query_set* qs, const void* q,
                                   int32_t num_q_heads, int32_t window, float softmax_scale, void* out,
                                   int32_t out_dtype, float* lse, cudaStream_t stream);

/* ---------------------------------------------------- prefill step --- */
/* Steps 1-4 for one prefill chunk (a DSA_MODE_PREFILL query set) in one call:
 * scores (written to `scores`, [n_q][ld]), top-k (idx, n_sel) and attention
 * (out, lse) with the automatic split of dsa_sparse_attn_prefill (the first
 * dsa_prefill_dense_queries() queries through the masked dense pass, the rest
 * gathered).  The top-k writes the dense pass's attended-position bitmap as it
 * writes the index lists, so the attention needs no pass over them.  Same
 * argument rules as the single calls; the workspace is
 * dsa_prefill_attn_workspace_size(kv, qs, k, num_q_heads, prefix_len, -1)
 * bytes.  Results equal those of the three calls in sequence (indices bit for
 * bit; outputs within rounding). */
dsa_status dsa_prefill_step(const dsa_paged_kv* kv, const dsa_query_set* qs, const void* q, const int8_t* q_idx,
                            int32_t num_q_heads, int32_t prefix_len, int32_t k, float softmax_scale,
                            int32_t* scores, int32_t ld, int32_t* idx, int32_t* n_sel, void* out,
                            int32_t out_dtype, float* lse, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------- staging copy --- */
/* Copies `bytes` from src to dst with a kernel on `stream`: the staging of a
 * step's inputs and outputs in a serving loop, without the copy engines.
 * Either side may be device memory or page-locked host memory (cudaHostAlloc,
 * cudaMallocHost or cudaHostRegister; the exception to "device memory only"
 * above), which the kernel reaches through its device mapping; pageable host
 * memory, device memory of another device and overlapping ranges return
 * DSA_ERR_INVALID_ARG before anything is launched.  dst and src 16-byte aligned, bytes a multiple of 16 (0: nothing
 * happens).  Launched with programmatic dependent launch like every kernel
 * here: it reads src only after the previous kernel of the stream has
 * completed, so a step's outputs can be copied right behind it.  The host sees
 * a copy into its memory once it has synchronised with the stream. */
dsa_status dsa_copy_async(void* dst, const void* src, size_t bytes, cudaStream_t stream);

/* ---------------------------------------------------- fused decode step --- */
/* Steps 1-4 for one decode token per sequence, in one call: scores (written to
 * `scores`, [batch][ld]), top-k (idx, n_sel) and attention (out, lse), with the
 * score histogram built while scoring.  Same argument rules as the single steps
 * (num_q_heads <= 64, group <= 16).
 * Overlap with the previous kernel: the kernels are launched with programmatic
 * dependent launch, and the first one (the scoring, as in dsa_index_scores in
 * decode mode) reads context_lens, block_table and the indexer cache rows other
 * than each sequence's newest position before it waits for the previous kernel
 * of the stream to finish.  These inputs must therefore be complete before that
 * kernel starts: written by host copies, by kernels launched without early
 * completion (every kernel not launched with programmatic dependent launch, and
 * dsa_kv_write), or earlier.  Everything else (the newest token's cache rows,
 * q, q_idx, the workspace and the outputs) is touched only after the wait.
 * Inside the step the attention walks every sequence's prefix rows first (of
 * sequences whose context reaches past the prefix), while the selection still
 * runs on part of the SMs, and the selected rows after it; by then the scoring
 * kernel, and so every kernel before the step, has completed.  The selection's
 * clusters are kept to at most half of the SMs to leave room for that pass.
 * The step's last kernel (the merge) lets the next kernel of the stream launch
 * before it finishes: a kernel launched after the step with programmatic
 * dependent launch must wait for it (griddepcontrol.wait) before it reads out,
 * lse or anything else the step writes. */
dsa_status dsa_decode_step(const dsa_paged_kv* kv, const void* q, const int8_t* q_idx,
                           int32_t num_q_heads, int32_t prefix_len, int32_t k,
                           float softmax_scale, int32_t* scores, int32_t ld, int32_t* idx,
                           int32_t* n_sel, void* out, int32_t out_dtype, float* lse,
                           void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------ per-KV-head indexer, decode --- */
/* The fused decode step with one indexer head per KV head (§2.4 keeps the KV
 * state per head; whether the selection is per head the article does not say,
 * and dsa_decode_step reads it as one selection per token): KV head g scores
 * its own indexer keys against its own indexer query, selects its own top-k
 * (same rule as dsa_topk_select: ties to the lower position, the prefix never
 * scored) and its num_q_heads / num_kv_heads query heads attend the prefix plus
 * that selection.  Layouts that differ from dsa_decode_step:
 *   kv->idx_cache : int8 [num_blocks][num_kv_heads][64][64] (a head's keys of a
 *                   block contiguous)
 *   q_idx         : int8 [batch][num_kv_heads][64]
 *   scores        : int32 [batch * num_kv_heads][ld], ld >= max_context_len
 *   idx, n_sel    : int32 [batch][num_kv_heads][k] and [batch][num_kv_heads]
 * q / out / lse as in dsa_decode_step.  batch * num_kv_heads <= 2048.  The
 * workspace (dsa_heads_workspace_size bytes) holds the histograms of the
 * (sequence, head) pairs and the attention partials; the kernels map each pair
 * onto its sequence's context length and block-table row themselves.  The same
 * overlap with the previous kernel as dsa_decode_step (block tables, context
 * lengths and the cache outside the newest positions must be complete before
 * the call's first kernel starts).  The attention copies each selected row per
 * KV head (256-byte K and V pieces) instead of one piece per position.
 * block_table_heads (device, or NULL): one block table per KV head, int32
 * [num_kv_heads][batch][max_blocks_per_seq], the tables of the per-(layer,
 * head) block bitmaps (dsa_kv_bitmap_*): head g then reads its positions'
 * indexer keys, K and V from the head-g slices of the blocks its own table
 * names, so that one physical block can hold different positions for
 * different heads.  NULL: every head uses kv->block_table.  Ids outside the
 * pool are reported through the device status, as for kv->block_table.
 * (ABI version 3 added this argument.) */
size_t dsa_heads_workspace_size(const dsa_paged_kv* kv, int32_t num_q_heads, int32_t k, int32_t prefix_len);
dsa_status dsa_decode_step_heads(const dsa_paged_kv* kv, const void* q, const int8_t* q_idx,
                                 const int32_t* block_table_heads /* device or NULL */,
                                 int32_t num_q_heads, int32_t prefix_len, int32_t k, float softmax_scale,
                                 int32_t* scores, int32_t ld, int32_t* idx, int32_t* n_sel, void* out,
                                 int32_t out_dtype, float* lse, void* ws, size_t ws_bytes,
                                 cudaStream_t stream);

/* ------------------------------------------- decode top-k without scratch --- */
/* The article has no counterpart to this call.  It is for callers that cannot
 * allocate device memory: for example a plugin running inside a serving process
 * whose device memory is all owned by the host framework's pool and which is
 * handed no allocator, or a latency-critical path that cannot take cudaMalloc's
 * implicit synchronisation and unbounded cost.  It returns exactly what
 * dsa_topk_select returns in decode mode (query b = newest token of sequence
 * b); the caller passes inputs and outputs only.  Its scratch is a static
 * device array of DSA_TOPK_STATIC_SCRATCH_BYTES inside the library, which every
 * GPU that loads the library keeps until the process exits; the call makes no
 * cudaMalloc, cudaFree or other allocating call.
 *   - Scratch needed: exactly 4096 bytes per sequence (its 1024-bin coarse
 *     score histogram, nothing else), so the 4 MiB array serves batches of
 *     up to 1024 sequences; batch 1025 and above return DSA_ERR_UNSUPPORTED
 *     before anything is launched (checked on the host).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and sets kernel attributes: make that first call
 *     before any stream capture.
 *   - Every call uses the same array, which keeps the last call's contents;
 *     each call first zeroes the histograms and counters it relies on.  Calls
 *     whose work overlaps on the GPU (other streams, other host threads) race
 *     on the array and give wrong results: serialise them. */
#define DSA_TOPK_STATIC_SCRATCH_BYTES (4u << 20)
dsa_status dsa_topk_select_decode_noalloc(const dsa_paged_kv* kv, const int32_t* scores, int32_t ld,
                                          int32_t prefix_len, int32_t k, int32_t* idx, int32_t* n_sel,
                                          cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H */
