// Steps 3 + 4 of DSA (§2.2 gather, §2.3 attention): GQA attention of each query
// token over its attended rows, read straight from the paged KV cache.
//
// The cache keeps, for every slot (block * 64 + row), the K rows of all KV heads
// side by side (and the same for V), so one attended position is one contiguous
// piece of Hkv * 256 bytes of K and one of V; where the cache stores a slot's V
// row right after its K row the two are one piece, fetched with one copy.  A query has P + k attended-row
// slots, its causal prefix rows then its selected rows (slots past its actual
// rows are empty).  A persistent grid (one CTA per SM) takes one contiguous
// range of the row slots of all queries per CTA (the same number of rows to
// within one for every CTA) and walks it in tiles of up to 128 / Hkv rows
// (64 KB of K and V whatever Hkv is) that break at query boundaries, so the
// copy pipeline runs on across queries (§2.3 decode: load only the active KV,
// asynchronously).  In prefill the prefix part of every query comes from the
// prefix pass (k_prefix.cu) as the query's starting state, and only the
// selected rows are walked here.
//
// Warp roles.  Four producer warps gather: every attended position of a tile is
// two bulk copies (cp.async.bulk, K piece and V piece) into a three-stage ring of
// shared memory, tracked by mbarriers, ahead of the math (§2.3 prefetch of the
// next block); each row's cache slot is fetched two tiles before its copy (a
// position given by the caller is resolved through the block table by a
// second, dependent load).  In decode every producer thread walks every tile
// and issues its share of the copies; in prefill one producer warp per stage
// takes every third tile (see the PS parameter).  One consumer warp per KV
// head computes, for each 16-row chunk, S^T = K Q^T and O^T = V^T P^T on the
// tensor cores (mma.sync m16n8k16 bf16, fp32 accumulate; P enters as two bf16
// terms, hi + lo, so it keeps ~16 mantissa bits), so the attended rows fill the
// 16-row M side and the G query heads of the group the 8-wide N side; P^T
// reaches its operand layout through movmatrix.  The online softmax runs per
// head column in base 2, reduced over the row groups with warp shuffles, and O
// is rescaled only when a running max moved.  A query whose rows all fall in
// one CTA is written out directly; a query cut by range boundaries leaves one
// partial (max, sum, unnormalised O) per CTA, and attn_combine_kernel,
// launched right behind (programmatic dependent launch), merges them.
#include "attn_tile.cuh"
#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

__device__ int g_status;

constexpr int kProducerWarps = 4;
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr int kStages = 3;
constexpr int kTileRowsMax = 128;                 // 128 / Hkv rows per tile
constexpr int kRowPad = 16;                       // shared-memory row pitch = Hkv * 256 + 16 (conflict-free ldmatrix)
constexpr int kPieceMax = 8 * kHeadDim * 2;       // K (or V) bytes of one position, Hkv <= 8
constexpr int kStageBytes = 2 * kTileRowsMax * (kHeadDim * 2 + kRowPad);  // largest stage (Hkv = 1): 69,632
constexpr int kMaxHq = kMaxQHeads;              // the host refuses more heads (check_heads)
constexpr int kQBytes = kMaxHq * kHeadDim * 2;    // one query's Q, all heads: 16 KB
constexpr int kSmemBytes = kStages * kStageBytes + kQBytes + 8 * (2 * kStages + 2) + 16;
static_assert(kProducerWarps == kStages + 1, "one producer warp per stage, plus the query copier");
static_assert(2 * 16 * (kPieceMax + kRowPad) <= kStageBytes, "Hkv = 8 stage must fit");
static_assert(kTileRowsMax * (2 * kHeadDim * 2 + kRowPad) <= kStageBytes, "adjacent K/V stage (Hkv = 1) must fit");
static_assert(kSmemBytes <= 232448, "attention shared memory above the 227 KB per-CTA limit");

struct AttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  const int32_t* bt;
  const int32_t* ctx;
  const int32_t* nsel;
  const int32_t* slot;  // cache slot of every selected position, [n_q][k], or null:
  const int32_t* idx;   // then the selected positions themselves, [n_q][k]
  int mode, seq, pos0;
  int max_blocks, num_blocks, hkv, hq, group, k, prefix, max_ctx;
  int rows;          // attended rows per tile: 128 / hkv
  int piece;         // bytes of one position's K (or V): hkv * 256
  int row_stride;    // bf16 values between the K (or V) rows of consecutive cache slots
  int per_row;       // copies per attended row: 1 (K and V adjacent in the cache, one piece) or 2
  int cbytes;        // bytes of one copy: 2 * piece or piece
  int pitch;         // shared-memory row pitch: cbytes + 16 (adjacent) or piece + 16
  int v_off;         // shared-memory offset of a row's V from its K: piece (adjacent) or rows * pitch
  float scale_log2;
  int units;         // n_q * rows_per_q attended-row slots (< 2^31, checked on the host)
  int rows_per_q;    // prefix + k (k when the prefix part comes from pre_ml); with two passes
                     // the second pass's: max(k, min(prefix, max_ctx))
  int two_pass;      // decode: the prefix rows first, before the wait on the previous kernel
  int units1;        // first pass: n_q * prefix row slots, over CTAs [0, grid1)
  int grid1;
  float* part_o;     // [grid][passes][2 slots][hq][128]
  float2* part_ml;   // [grid][passes][2 slots][hq]
  void* out;
  int out_dtype;
  float* lse;
  const float2* pre_ml;  // prefill: the prefix part of every query, computed per tile of
  const float* pre_o;    // queries beforehand ([n_q][hq] and [n_q][hq][128]), or null
  int hsplit;            // decode, per-KV-head indexer: query qi is (sequence qi / hsplit, head qi % hsplit)
  int bt_per_query;      // the block table has one row per query, not per sequence
  int bt_head_rows;      // per-head block tables [Hkv][batch]: query (b, h) reads row h * bt_head_rows + b
  int window;            // decode: > 0 attends the last `window` positions of each context, no selection
};

// 32-bit division when the products fit (the common case), 64-bit otherwise;
// the 64-bit forms stay out of line so that the kernels' code keeps one copy.
__device__ __noinline__ int range_begin64(int T, int G, int c) { return (int)((long long)T * c / G); }
__device__ __noinline__ int cta_of64(int T, int G, int x) { return (int)(((long long)(x + 1) * G - 1) / T); }
__device__ __forceinline__ int range_begin(int T, int G, int c) {
  if ((unsigned long long)T * G < (1ull << 31)) return (int)((unsigned)(T * c) / (unsigned)G);
  return range_begin64(T, G, c);
}
__device__ __forceinline__ int cta_of(int T, int G, int x) {
  if ((unsigned long long)T * G < (1ull << 31)) return (int)((unsigned)((x + 1) * G - 1) / (unsigned)T);
  return cta_of64(T, G, x);
}

struct QueryInfo {
  int qi, seq, n_pre, rows;
  int pre_off;  // position of the query's first prefix-part row (the window's start; else 0)
  int bt_row;  // row of the block table: the query's (per-head tables) or its sequence's
  int hoff;  // bf16 offset of the query's KV head inside a cache row (per-head indexer), else 0
};
// pass 0 (two-pass decode only): the query's prefix rows when its context
// reaches past the prefix, else none; pass 1 then holds its selected rows, or
// (context inside the prefix) its whole causal range.  The first pass reads
// no selection output: it runs before the wait on the previous kernel.
// PS: prefill (queries of one sequence, the prefix part possibly from pre_ml);
// else decode (one query per sequence, or per (sequence, KV head) with hsplit).
// TP: two-pass decode.
template <bool PS, bool TP>
__device__ __forceinline__ QueryInfo query_info(const AttnParams& p, int qi, int pass) {
  QueryInfo qf;
  qf.qi = qi;
  const int hh = !PS && p.hsplit > 1 ? qi % p.hsplit : 0;
  qf.seq = PS ? p.seq : p.hsplit > 1 ? (qi - hh) / p.hsplit : qi;
  qf.bt_row = PS ? qf.seq : p.bt_head_rows ? hh * p.bt_head_rows + qf.seq : p.bt_per_query ? qi : qf.seq;
  qf.hoff = hh * kHeadDim;
  const int pos = PS ? p.pos0 + qi : min(__ldg(p.ctx + qf.seq), p.max_ctx) - 1;
  qf.pre_off = 0;
  if (!PS && p.window > 0) {  // the window [pos + 1 - n, pos]: contiguous rows, no index list
    qf.n_pre = max(0, min(p.window, pos + 1));
    qf.pre_off = pos + 1 - qf.n_pre;
    qf.rows = qf.n_pre;
    return qf;
  }
  if constexpr (TP) {
    const bool past = pos + 1 > p.prefix;
    if (pass == 0) {
      qf.n_pre = past ? p.prefix : 0;
      qf.rows = qf.n_pre;
    } else {
      qf.n_pre = past ? 0 : max(0, pos + 1);
      qf.rows = qf.n_pre + (past ? min(max(__ldg(p.nsel + qi), 0), p.k) : 0);
    }
    return qf;
  }
  qf.n_pre = PS && p.pre_ml ? 0 : max(0, min(p.prefix, pos + 1));  // with pre_ml every row is a selected one
  qf.rows = qf.n_pre + min(max(__ldg(p.nsel + qi), 0), p.k);
  return qf;
}

enum : int { kFirst = 1, kLast = 2, kWhole = 4, kHead = 8 };  // kHead: the segment starts the query

// The work of all queries is the sequence of their attended-row slots, P + k
// per query (slots past a query's actual row count are empty).  A CTA takes
// one contiguous range of it and walks it in tiles of up to `rows` rows that
// break at query boundaries, so every CTA gets the same number of rows to
// within one.  Empty tiles are skipped, but a segment's last tile is always
// kept so that the segment closes.  A segment is the run of a query's rows
// inside one CTA's range.
// Two-pass decode walks two such sequences one after the other: first the
// prefix row slots (P per query) over CTAs [0, grid1), then the selected-row
// slots over every CTA; each pass leaves its own partials, and a query is
// never written out directly (the combine merges both passes).
struct Cursor {
  int x, x_begin, x_end, qi, seg_start, pass, rpq;
  QueryInfo qf;
  bool fresh;
  bool hold;  // stop at the end of the prefix pass instead of waiting for the second
};
struct Tile {
  QueryInfo qf;
  int r0, nvalid, flags, slot;  // slot: partial index of this CTA, (pass, first / later segment)
};

__device__ __forceinline__ void cursor_pass(Cursor& c, const AttnParams& p, int pass) {
  c.pass = pass;
  if (pass == 0) {
    const int g1 = p.grid1;
    c.x_begin = (int)blockIdx.x < g1 ? range_begin(p.units1, g1, blockIdx.x) : 0;
    c.x_end = (int)blockIdx.x < g1 ? range_begin(p.units1, g1, blockIdx.x + 1) : 0;
    c.rpq = p.prefix;
  } else {
    c.x_begin = range_begin(p.units, gridDim.x, blockIdx.x);
    c.x_end = range_begin(p.units, gridDim.x, blockIdx.x + 1);
    c.rpq = p.rows_per_q;
  }
  c.x = c.x_begin;
  c.qi = -1;
  c.seg_start = c.x_begin;
  c.fresh = false;
}
template <bool TP>
__device__ __forceinline__ void cursor_init(Cursor& c, const AttnParams& p) {
  c.hold = false;
  cursor_pass(c, p, TP ? 0 : 1);
}

template <bool PS, bool TP>
__device__ __forceinline__ bool next_tile(Cursor& c, const AttnParams& p, Tile* t) {
  for (;;) {
    if (c.x >= c.x_end) {
      if (!TP || c.pass == 1 || c.hold) return false;
      // The selected rows come from the previous kernel of the stream.
      pdl_wait();
      cursor_pass(c, p, 1);
      continue;
    }
    const int RPQ = c.rpq;
    const int x = c.x;
    const int qi = x / RPQ;
    const int r = x - qi * RPQ;
    const int q_end = (qi + 1) * RPQ;
    c.x = x + min(min(c.x_end, q_end) - x, p.rows);
    if (qi != c.qi) {
      c.qi = qi;
      c.qf = query_info<PS, TP>(p, qi, c.pass);
      c.seg_start = x;
      c.fresh = true;
    }
    const int nvalid = min(max(c.qf.rows - r, 0), c.x - x);
    const bool last = c.x == c.x_end || c.x == q_end;
    if (nvalid == 0 && !last) continue;
    t->qf = c.qf;
    t->r0 = r;
    t->nvalid = nvalid;
    t->flags = (c.fresh ? kFirst : 0) | (last ? kLast : 0) |
               (!TP && last && c.seg_start == qi * RPQ && c.x == q_end ? kWhole : 0) |
               (c.fresh && c.seg_start == qi * RPQ ? kHead : 0);
    t->slot = (TP ? 2 * c.pass : 0) + (c.seg_start == c.x_begin ? 0 : 1);
    c.fresh = false;
    return true;
  }
}

// Cache slots are fetched two tiles ahead of their use, in up to two
// dependent loads: fetch_first issues the first (the block id of a prefix
// row; the slot of a selected row, or its position when the call brings
// positions instead of slots), fetch_second the second (the block id of a
// selected position), and resolve makes the slot, validated against the pool,
// when the copy is issued.
struct RowRef {
  int a;   // block id (lo >= 0) or cache slot (lo < 0), not yet validated
  int lo;  // row inside the block, or -1
};
__device__ __forceinline__ int fetch_first(const AttnParams& p, const QueryInfo& qf, int r) {
  if (r < qf.n_pre) return __ldg(p.bt + (size_t)qf.bt_row * p.max_blocks + ((qf.pre_off + r) >> 6));
  const size_t e = (size_t)qf.qi * p.k + (r - qf.n_pre);
  return p.slot ? __ldg(p.slot + e) : __ldg(p.idx + e);
}
__device__ __forceinline__ RowRef fetch_second(const AttnParams& p, const QueryInfo& qf, int r, int first) {
  if (r < qf.n_pre) return RowRef{first, (qf.pre_off + r) & 63};  // prefix-part row r is position pre_off + r
  if (p.slot) return RowRef{first, -1};
  int pos = first;
  if ((unsigned)pos >= (unsigned)p.max_blocks * kBlock) {
    set_status(&g_status, kStBadBlock);
    pos = 0;
  }
  return RowRef{__ldg(p.bt + (size_t)qf.bt_row * p.max_blocks + (pos >> 6)), pos & 63};
}
__device__ __forceinline__ int resolve(const AttnParams& p, RowRef v) {
  if (v.lo < 0) {
    if ((unsigned)v.a >= (unsigned)p.num_blocks * kBlock) {
      set_status(&g_status, kStBadBlock);
      return 0;
    }
    return v.a;
  }
  if ((unsigned)v.a >= (unsigned)p.num_blocks) {
    set_status(&g_status, kStBadBlock);
    return v.lo;
  }
  return v.a * kBlock + v.lo;
}

__device__ __forceinline__ void write_out(const AttnParams& p, size_t head, int d, float v) {
  if (p.out_dtype == 0)
    reinterpret_cast<__nv_bfloat16*>(p.out)[head * kHeadDim + d] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(p.out)[head * kHeadDim + d] = v;
}

// NT: 8-head column tiles of a KV group (1 for G <= 8, 2 for G <= 16).
// PS: producer layout.  false (decode): every producer thread walks every
// tile and issues its share of the copies; Q rides on the segment's first
// tile.  true (prefill, where L2-resident rows make the producer's per-tile
// chain the limit): one producer warp per ring stage, each with kStages tile
// times per tile, and Q copied by its own warp through a one-slot ring.
// TP (decode only): two passes, the prefix rows before the wait on the
// previous kernel, then the selected rows.
template <int NT, bool PS, bool TP>
__global__ void __launch_bounds__(kProducerThreads + 8 * 32, 1) sparse_attn_kernel(const AttnParams p) {
  static_assert(!(PS && TP), "two passes are a decode form");
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* s_q = smem + kStages * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_q + kQBytes);
  uint64_t* empty = full + kStages;
  uint64_t* q_empty = empty + kStages;
  uint64_t* q_full = q_empty + 1;
  volatile int* s_abort = reinterpret_cast<volatile int*>(q_full + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.group;
  const bool none1 = !TP || (int)blockIdx.x >= p.grid1 ||
                     range_begin(p.units1, p.grid1, blockIdx.x) >= range_begin(p.units1, p.grid1, blockIdx.x + 1);
  if (none1 && range_begin(p.units, gridDim.x, blockIdx.x) >= range_begin(p.units, gridDim.x, blockIdx.x + 1)) return;

  // Set-up that touches no global memory runs before the wait on the previous kernel.
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], PS ? 32 : kProducerThreads);
      mbar_init(&empty[s], p.hkv);
    }
    mbar_init(q_empty, p.hkv);
    if (PS) mbar_init(q_full, 1);
    *s_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // Two-pass decode: the prefix rows, Q, context lengths and block table are
  // inputs no kernel of the step writes (a context inside the prefix, whose
  // newest row the step's cache write may have just written, has its rows in
  // the second pass), and this kernel starts only after the selection kernel
  // has passed its own wait, i.e. after the scoring kernel and everything
  // before it completed.  The first pass therefore runs before the wait; each
  // thread waits when its walk reaches the second pass.
  if (!TP) pdl_wait();
  pdl_trigger();

  if (warp < kProducerWarps) {
    // ---------------------------------------------------------- producers
    if constexpr (!PS) {
      // Copy c of a tile (row c / per_row: its K and V in one piece when they
      // are adjacent in the cache, else K if c is even and V if odd) is issued
      // by thread (c % 4) * 32 + (c / 4) % 32, so the copies spread over the warps.
      // Rows from the valid count up to the next multiple of 16 (the rest of the
      // last 16-row chunk the consumers read) get the last valid row again, so
      // that every row the math touches holds finite cache values; their
      // probabilities are zero.
      const int pt = lane * kProducerWarps + warp;
      const int shift = p.per_row - 1;  // 0 or 1
      const int n_copies = p.rows << shift;
      auto filled = [&](const Tile& tl) { return min((tl.nvalid + 15) & ~15, p.rows); };
      auto active = [&](const Tile& tl, int u) {
        const int c = pt + u * kProducerThreads;
        return c < n_copies && (c >> shift) < filled(tl);
      };
      auto row_of = [&](const Tile& tl, int u) {
        return tl.r0 + min((pt + u * kProducerThreads) >> shift, tl.nvalid - 1);
      };
      // Two-pass decode: the look-ahead stops at the end of the prefix pass, so
      // that every prefix tile goes out before the wait on the previous kernel
      // (looking two tiles ahead into the second pass held the last prefix
      // tiles back until the selection ended); the second phase then starts
      // its own look-ahead behind the wait.
      Cursor cur;
      cursor_init<TP>(cur, p);
      cur.hold = TP;
      const uint32_t q_bytes = (uint32_t)p.hq * kHeadDim * 2;
      // Decode reads each attended row once per call: evict-first keeps the
      // partial states, block table and selection in L2 around the stream.
      const uint64_t stream_policy = l2_evict_first();
      int n = 0, seg = 0;
      for (int phase = 0; phase < 2 && !*s_abort; ++phase) {
      if (phase == 1) {
        if (!TP) break;
        cur.hold = false;  // the next tile switches to the second pass, after the wait
      }
      Tile t0, t1, t2;  // issued now, next, the one after
      bool h0 = next_tile<PS, TP>(cur, p, &t0);
      bool h1 = h0 && next_tile<PS, TP>(cur, p, &t1);
      bool h2 = h1 && next_tile<PS, TP>(cur, p, &t2);
      RowRef v0[2];  // rows of t0, both loads issued
      int f1[2];     // first loads of t1
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        v0[u] = RowRef{0, -1};
        f1[u] = 0;
        if (h0 && active(t0, u)) v0[u] = fetch_second(p, t0.qf, row_of(t0, u), fetch_first(p, t0.qf, row_of(t0, u)));
        if (h1 && active(t1, u)) f1[u] = fetch_first(p, t1.qf, row_of(t1, u));
      }
      while (h0) {
        const int s = n % kStages;
        if (n >= kStages && !mbar_wait(&empty[s], ((n / kStages) - 1) & 1)) {
          set_status(&g_status, kStTimeout);
          *s_abort = 1;
          break;
        }
        if (*s_abort) break;
        const bool first = t0.flags & kFirst;
        uint32_t bytes = 0;
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if (active(t0, u)) bytes += p.cbytes;
        if (first && pt == 0) {
          if (seg > 0 && !mbar_wait(q_empty, (seg - 1) & 1)) {
            set_status(&g_status, kStTimeout);
            *s_abort = 1;
          }
          bytes += q_bytes;
        }
        seg += first;
        mbar_arrive_expect_tx(&full[s], bytes);
        uint8_t* st = smem + s * kStageBytes;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int c = pt + u * kProducerThreads;
          if (active(t0, u)) {
            const int r = c >> shift, part = c & shift;  // part 1: the V of a separate layout
            const size_t sl = (size_t)resolve(p, v0[u]);
            const __nv_bfloat16* src = (part ? p.vc : p.kc) + sl * p.row_stride + t0.qf.hoff;
            bulk_g2s_hint(st + r * p.pitch + part * p.v_off, src, p.cbytes, &full[s], stream_policy);
          }
        }
        if (first && pt == 0)
          bulk_g2s(s_q, p.q + (size_t)t0.qf.qi * p.hq * kHeadDim, q_bytes, &full[s]);
        ++n;
        // Advance: second loads of the next tile, first loads of the one after.
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (h1 && active(t1, u)) v0[u] = fetch_second(p, t1.qf, row_of(t1, u), f1[u]);
          if (h2 && active(t2, u)) f1[u] = fetch_first(p, t2.qf, row_of(t2, u));
        }
        const bool more = h2;
        t0 = t1;
        h0 = h1;
        t1 = t2;
        h1 = h2;
        h2 = more && next_tile<PS, TP>(cur, p, &t2);
      }
      }
    } else {
      // Producer warp w < kStages issues the tiles n with n % kStages == w, all
      // into stage w, so it waits only on its own stage's previous use (no
      // mbarrier phase of another warp's tile can alias) and has kStages tile
      // times for each of its tiles.  Its lanes take the tile's rows in turn
      // (row r by lane r % 32) and issue one bulk copy for the row's K and one
      // for its V.  The cache slots of its next tile are fetched while the
      // current one is issued, i.e. kStages tiles ahead (the second load of a
      // position, its block id, then has kStages tile times as well), and those
      // of the tile after it 2 * kStages tiles ahead.  Rows from the valid count
      // up to the next multiple of 16 (the rest of the last 16-row chunk the
      // consumers read) get the last valid row again, so that every row the math
      // touches holds finite cache values; their probabilities are zero.  Warp
      // kStages copies each segment's Q, in order, through a one-slot ring of
      // its own (q_full / q_empty).
      if (warp < kStages) {
        const int w = warp;
        const int R = (p.rows + 31) >> 5;  // rows per lane: 1 .. 4
        auto filled = [&](const Tile& tl) { return min((tl.nvalid + 15) & ~15, p.rows); };
        auto active = [&](const Tile& tl, int i) { return i < R && lane + 32 * i < filled(tl); };
        auto row_of = [&](const Tile& tl, int i) { return tl.r0 + min(lane + 32 * i, tl.nvalid - 1); };
        Cursor cur;
        cursor_init<TP>(cur, p);
        int n_walk = 0;
        auto next_own = [&](Tile* t) {
          Tile x;
          while (next_tile<PS, TP>(cur, p, &x))
            if (n_walk++ % kStages == w) {
              *t = x;
              return true;
            }
          return false;
        };
        Tile t0, t1, t2;  // this warp's tile issued now, its next, the one after
        bool h0 = next_own(&t0);
        bool h1 = h0 && next_own(&t1);
        bool h2 = h1 && next_own(&t2);
        RowRef v0[4];  // rows of t0, both loads issued
        int f1[4];     // first loads of t1
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v0[i] = RowRef{0, -1};
          f1[i] = 0;
          if (h0 && active(t0, i)) v0[i] = fetch_second(p, t0.qf, row_of(t0, i), fetch_first(p, t0.qf, row_of(t0, i)));
          if (h1 && active(t1, i)) f1[i] = fetch_first(p, t1.qf, row_of(t1, i));
        }
        uint8_t* st = smem + w * kStageBytes;
        for (int j = 0; h0; ++j) {
          if (j > 0 && !mbar_wait(&empty[w], (j - 1) & 1)) {
            set_status(&g_status, kStTimeout);
            *s_abort = 1;
            break;
          }
          if (*s_abort) break;
          uint32_t bytes = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (active(t0, i)) bytes += 2 * p.piece;
          mbar_arrive_expect_tx(&full[w], bytes);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (active(t0, i)) {
              const int r = lane + 32 * i;
              const size_t off = (size_t)resolve(p, v0[i]) * p.row_stride;
              bulk_g2s(st + r * p.pitch, p.kc + off, p.cbytes, &full[w]);
              if (p.per_row == 2) bulk_g2s(st + r * p.pitch + p.v_off, p.vc + off, p.piece, &full[w]);
            }
          // Advance: second loads of the next tile, first loads of the one after.
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (h1 && active(t1, i)) v0[i] = fetch_second(p, t1.qf, row_of(t1, i), f1[i]);
            if (h2 && active(t2, i)) f1[i] = fetch_first(p, t2.qf, row_of(t2, i));
          }
          const bool more = h2;
          t0 = t1;
          h0 = h1;
          t1 = t2;
          h1 = h2;
          h2 = more && next_own(&t2);
        }
      } else if (lane == 0) {
        const uint32_t q_bytes = (uint32_t)p.hq * kHeadDim * 2;
        Cursor cur;
        cursor_init<TP>(cur, p);
        Tile t;
        for (int seg = 0; next_tile<PS, TP>(cur, p, &t);) {
          if (!(t.flags & kFirst)) continue;
          if (seg > 0 && !mbar_wait(q_empty, (seg - 1) & 1)) {
            set_status(&g_status, kStTimeout);
            *s_abort = 1;
            break;
          }
          if (*s_abort) break;
          mbar_arrive_expect_tx(q_full, q_bytes);
          bulk_g2s(s_q, p.q + (size_t)t.qf.qi * p.hq * kHeadDim, q_bytes, q_full);
          ++seg;
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int g = warp - kProducerWarps;  // KV head
  if (g >= p.hkv) return;
  const int hc = 2 * (lane & 3);  // first head column of this lane in an 8-head tile
  HeadState<NT> hs;
  Cursor cur;
  cursor_init<TP>(cur, p);
  Tile t;
  int seg = 0;
  for (int n = 0; next_tile<PS, TP>(cur, p, &t); ++n) {
    const int s = n % kStages;
    if (!mbar_wait(&full[s], (n / kStages) & 1)) {
      set_status(&g_status, kStTimeout);
      *s_abort = 1;
      break;
    }
    if (t.flags & kFirst) {
      if constexpr (PS) {
        if (!mbar_wait(q_full, seg & 1)) {
          set_status(&g_status, kStTimeout);
          *s_abort = 1;
          break;
        }
        ++seg;
      }
      load_q(hs, s_q, g, G, lane);
      // The slot is refilled by a bulk copy (async proxy): order the ldmatrix
      // reads before it (without the proxy fence, the next segment's Q was
      // seen landing while a warp still read the slot).
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_empty);
      reset_state(hs);
      if (PS && p.pre_ml && (t.flags & kHead)) {
        // The query's prefix part is the starting state of the segment that
        // begins the query (its sum sits in one row group of lanes).
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = j * 8 + hc + e;
            if (h >= G) continue;
            const size_t head = (size_t)t.qf.qi * p.hq + (size_t)g * G + h;
            const float2 ml = __ldg(p.pre_ml + head);
            hs.m[j][e] = ml.x;
            hs.l[j][e] = (lane >> 2) == 0 ? ml.y : 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int d = 16 * i + (lane >> 2);
              hs.o[i][j][e] = __ldg(p.pre_o + head * kHeadDim + d);
              hs.o[i][j][e + 2] = __ldg(p.pre_o + head * kHeadDim + d + 8);
            }
          }
      }
    }
    const uint8_t* sk = smem + s * kStageBytes + g * (kHeadDim * 2);
    attend_rows(hs, sk, sk + p.v_off, p.pitch, t.nvalid, p.scale_log2, lane);
    fence_proxy_async_smem();  // the stage is refilled by bulk copies as well
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    if (t.flags & kLast) {
      total_sums(hs);
      const size_t head0 = (size_t)t.qf.qi * p.hq + (size_t)g * G;
      const size_t sl = (size_t)blockIdx.x * (TP ? 4 : 2) + t.slot;
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = j * 8 + hc + e;
          if (h >= G) continue;
          if (t.flags & kWhole) {
            const float r = 1.f / hs.l[j][e];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int d = 16 * i + (lane >> 2);
              write_out(p, head0 + h, d, hs.o[i][j][e] * r);
              write_out(p, head0 + h, d + 8, hs.o[i][j][e + 2] * r);
            }
            if (lane < 4 && p.lse) p.lse[head0 + h] = (hs.m[j][e] + log2f(hs.l[j][e])) * 0.69314718055994531f;
          } else {
            const size_t ph = sl * p.hq + (size_t)g * G + h;
            store_partial(hs, j, e, lane, p.part_ml + ph, p.part_o + ph * kHeadDim);
          }
        }
    }
  }
}

// Merge of the partials of split queries.  Block c stands for the range
// boundary between CTAs c and c + 1 of the attention grid.  A query cut by the
// nb boundaries c_lo .. c_hi - 1 has n = nb + 1 partials (one per CTA
// c_lo .. c_hi); the block of its j-th boundary merges the query heads
// h = j, j + nb, j + 2 nb, ..., four at a time.  A head has four warps: warp
// s of the head takes the partials i = s, s + 4, s + 8, ..., each lane four
// columns (one 16-byte load per partial), and the four running states
// (max, sum, accumulator) meet in shared memory.  A thread keeps up to
// kCombBatch partials in flight, so up to 32 partials are one round trip.
constexpr int kCombHeads = 4;                                // heads merged at once
constexpr int kCombSplit = 4;                                // warps per head
constexpr int kCombThreads = 32 * kCombHeads * kCombSplit;  // 512
constexpr int kCombBatch = 8;                                // partials in flight per thread

__device__ __forceinline__ void write_out4(const AttnParams& p, size_t head, int lane, float4 v) {
  if (p.out_dtype == 0) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p.out)[head * (kHeadDim / 4) + lane] = u;
  } else {
    reinterpret_cast<float4*>(p.out)[head * (kHeadDim / 4) + lane] = v;
  }
}

__global__ void __launch_bounds__(kCombThreads) attn_combine_kernel(const AttnParams p, int grid_ctas) {
  __shared__ float4 s_acc[kCombHeads][kCombSplit][32];
  __shared__ float2 s_ml[kCombHeads][kCombSplit];
  // The boundary arithmetic reads no memory: it runs before the wait on the
  // attention kernel, and blocks with no cut query leave without waiting.
  const int T = p.units, TP = p.rows_per_q;
  const int x = range_begin(T, grid_ctas, blockIdx.x + 1);  // first row slot of CTA blockIdx.x + 1
  const int qi = x / TP;
  if (x == qi * TP) return;  // no query is cut at this boundary
  const int first = qi * TP;
  const int c_lo = cta_of(T, grid_ctas, first), c_hi = cta_of(T, grid_ctas, first + TP - 1);
  const int j = (int)blockIdx.x - c_lo, nb = c_hi - c_lo, n = nb + 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hg = warp / kCombSplit, sub = warp % kCombSplit;
  // The partial of CTA c for this query sits in slot 0 if the query's segment
  // starts the CTA's range, else in slot 1.
  const int c_first = range_begin(T, grid_ctas, c_lo) >= first ? 0 : 1;  // slot of CTA c_lo
  const float4* part_o = reinterpret_cast<const float4*>(p.part_o);
  // The next kernel may start its own set-up while the merge waits: whatever it
  // reads before its wait on this kernel, no kernel here writes.
  pdl_trigger();
  pdl_wait();
  // The trip count depends on hg only, so the four warps of a head meet at
  // the same named barriers.
  for (int h = j + hg * nb; h < p.hq; h += kCombHeads * nb) {
    float M = -INFINITY, Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = sub; i0 < n; i0 += kCombSplit * kCombBatch) {
      float2 ml[kCombBatch];
      float4 v[kCombBatch];
#pragma unroll
      for (int u = 0; u < kCombBatch; ++u) {
        const int i = i0 + u * kCombSplit;
        if (i < n) {
          const int ph = ((c_lo + i) * 2 + (i == 0 ? c_first : 0)) * p.hq + h;  // < 2 * 320 * 64
          ml[u] = __ldg(&p.part_ml[ph]);
          v[u] = __ldg(&part_o[ph * (kHeadDim / 4) + lane]);
        }
      }
      float Mb = M;
#pragma unroll
      for (int u = 0; u < kCombBatch; ++u)
        if (i0 + u * kCombSplit < n) Mb = fmaxf(Mb, ml[u].x);
      const float Ms = Mb == -INFINITY ? 0.f : Mb;
      const float a = exp2f(M - Ms);  // rescale of what earlier batches summed
      Lsum *= a;
      acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
#pragma unroll
      for (int u = 0; u < kCombBatch; ++u)
        if (i0 + u * kCombSplit < n) {
          const float w = exp2f(ml[u].x - Ms);
          Lsum += w * ml[u].y;
          acc.x += w * v[u].x; acc.y += w * v[u].y; acc.z += w * v[u].z; acc.w += w * v[u].w;
        }
      M = Mb;
    }
    s_acc[hg][sub][lane] = acc;
    if (lane == 0) s_ml[hg][sub] = make_float2(M, Lsum);
    named_bar_sync(1 + hg, 32 * kCombSplit);
    if (sub == 0) {
      float Mx = -INFINITY;
#pragma unroll
      for (int s = 0; s < kCombSplit; ++s) Mx = fmaxf(Mx, s_ml[hg][s].x);
      const float Ms = Mx == -INFINITY ? 0.f : Mx;
      float L = 0.f;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s = 0; s < kCombSplit; ++s) {
        const float2 st = s_ml[hg][s];
        const float4 av = s_acc[hg][s][lane];
        const float w = exp2f(st.x - Ms);
        L += w * st.y;
        o.x += w * av.x; o.y += w * av.y; o.z += w * av.z; o.w += w * av.w;
      }
      const float r = 1.f / L;
      const size_t head = (size_t)qi * p.hq + h;
      write_out4(p, head, lane, make_float4(o.x * r, o.y * r, o.z * r, o.w * r));
      if (lane == 0 && p.lse) p.lse[head] = (Ms + log2f(L)) * 0.69314718055994531f;
    }
    named_bar_sync(1 + hg, 32 * kCombSplit);  // shared state is rewritten by the next head
  }
}

// Merge for two-pass decode: block (qi, hb) merges query heads hb * 4 ..
// hb * 4 + 3 of query qi over the partials of both passes (the CTAs whose
// prefix range and whose selected range cut the query); a head has four
// warps as above, warp s taking the partials s, s + 4, ... of the combined list.
__global__ void __launch_bounds__(kCombThreads) attn_combine2_kernel(const AttnParams p, int grid_ctas) {
  __shared__ float4 s_acc[kCombHeads][kCombSplit][32];
  __shared__ float2 s_ml[kCombHeads][kCombSplit];
  const int qi = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hg = warp / kCombSplit, sub = warp % kCombSplit;
  const int h = blockIdx.y * kCombHeads + hg;
  // CTA ranges over each pass's row slots: c0 .. c0 + n0 - 1 (prefix pass, grid1
  // CTAs), c1 .. c1 + n1 - 1 (selected pass, every CTA); the first CTA of a
  // range holds the query in its slot 0 if its range starts with the query.
  int n0 = 0, c0 = 0, f0 = 0;
  if (p.grid1 > 0 && p.units1 > 0) {
    const int first = qi * p.prefix;
    c0 = cta_of(p.units1, p.grid1, first);
    n0 = cta_of(p.units1, p.grid1, first + p.prefix - 1) - c0 + 1;
    f0 = range_begin(p.units1, p.grid1, c0) >= first ? 0 : 1;
  }
  const int first1 = qi * p.rows_per_q;
  const int c1 = cta_of(p.units, grid_ctas, first1);
  const int n1 = cta_of(p.units, grid_ctas, first1 + p.rows_per_q - 1) - c1 + 1;
  const int f1 = range_begin(p.units, grid_ctas, c1) >= first1 ? 0 : 1;
  const int n = n0 + n1;
  const float4* part_o = reinterpret_cast<const float4*>(p.part_o);
  pdl_trigger();  // as in attn_combine_kernel
  pdl_wait();
  if (h < p.hq) {
    float M = -INFINITY, Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = sub; i0 < n; i0 += kCombSplit * kCombBatch) {
      float2 ml[kCombBatch];
      float4 v[kCombBatch];
#pragma unroll
      for (int u = 0; u < kCombBatch; ++u) {
        const int i = i0 + u * kCombSplit;
        if (i < n) {
          const int sl = i < n0 ? (c0 + i) * 4 + (i == 0 ? f0 : 0)
                                : (c1 + i - n0) * 4 + 2 + (i == n0 ? f1 : 0);
          const int ph = sl * p.hq + h;  // < 4 * 320 * 64
          ml[u] = __ldg(&p.part_ml[ph]);
          v[u] = __ldg(&part_o[ph * (kHeadDim / 4) + lane]);
        }
      }
      float Mb = M;
#pragma unroll
      for (int u = 0; u < kCombBatch; ++u)
        if (i0 + u * kCombSplit < n) Mb = fmaxf(Mb, ml[u].x);
      const float Ms = Mb == -INFINITY ? 0.f : Mb;
      const float a = exp2f(M - Ms);
      Lsum *= a;
      acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
#pragma unroll
      for (int u = 0; u < kCombBatch; ++u)
        if (i0 + u * kCombSplit < n) {
          const float w = exp2f(ml[u].x - Ms);
          Lsum += w * ml[u].y;
          acc.x += w * v[u].x; acc.y += w * v[u].y; acc.z += w * v[u].z; acc.w += w * v[u].w;
        }
      M = Mb;
    }
    s_acc[hg][sub][lane] = acc;
    if (lane == 0) s_ml[hg][sub] = make_float2(M, Lsum);
  }
  __syncthreads();
  if (h < p.hq && sub == 0) {
    float Mx = -INFINITY;
#pragma unroll
    for (int s = 0; s < kCombSplit; ++s) Mx = fmaxf(Mx, s_ml[hg][s].x);
    const float Ms = Mx == -INFINITY ? 0.f : Mx;
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kCombSplit; ++s) {
      const float2 st = s_ml[hg][s];
      const float4 av = s_acc[hg][s][lane];
      const float w = exp2f(st.x - Ms);
      L += w * st.y;
      o.x += w * av.x; o.y += w * av.y; o.z += w * av.z; o.w += w * av.w;
    }
    const float r = 1.f / L;
    const size_t head = (size_t)qi * p.hq + h;
    write_out4(p, head, lane, make_float4(o.x * r, o.y * r, o.z * r, o.w * r));
    if (lane == 0 && p.lse) p.lse[head] = (Ms + log2f(L)) * 0.69314718055994531f;
  }
}

int g_attn_grid[64] = {};

}  // namespace

cudaError_t setup_attn_kernels() {
  cudaError_t e = cudaSuccess;
  auto smem = [&](auto kernel) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  };
  smem(sparse_attn_kernel<1, false, false>);
  smem(sparse_attn_kernel<2, false, false>);
  smem(sparse_attn_kernel<1, false, true>);
  smem(sparse_attn_kernel<2, false, true>);
  smem(sparse_attn_kernel<1, true, false>);
  smem(sparse_attn_kernel<2, true, false>);
  int dev = 0, sms = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && dev >= 0 && dev < 64) g_attn_grid[dev] = sms < kMaxAttnCtas ? sms : kMaxAttnCtas;
  return e;
}

int attn_grid_ctas() {
  int dev = 0;
  cudaGetDevice(&dev);
  return (dev >= 0 && dev < 64 && g_attn_grid[dev] > 0) ? g_attn_grid[dev] : 148;
}

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t st) {
  AttnParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kc = static_cast<const __nv_bfloat16*>(a.kv.k_cache);
  p.vc = static_cast<const __nv_bfloat16*>(a.kv.v_cache);
  p.bt = a.kv.block_table;
  p.ctx = a.kv.context_lens;
  p.nsel = a.n_sel;
  p.slot = a.slot;
  p.idx = a.idx;
  p.mode = a.qs.mode;
  p.seq = a.qs.seq;
  p.pos0 = a.qs.pos0;
  p.max_blocks = a.kv.max_blocks;
  p.num_blocks = a.kv.num_blocks;
  p.hkv = a.kv.hkv;
  p.hq = a.hq;
  p.group = a.hq / a.kv.hkv;
  p.k = a.k;
  p.prefix = a.prefix;
  p.max_ctx = a.kv.max_ctx;
  p.rows = kTileRowsMax / a.kv.hkv;
  p.piece = a.kv.hkv * kHeadDim * 2;
  p.row_stride = a.kv.row_stride;
  p.per_row = a.kv.adjacent ? 1 : 2;
  p.cbytes = a.kv.adjacent ? 2 * p.piece : p.piece;
  p.pitch = p.cbytes + kRowPad;
  p.v_off = a.kv.adjacent ? p.piece : p.rows * p.pitch;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.pre_ml = a.ws.pre_ml;
  p.pre_o = a.ws.pre_o;
  p.hsplit = a.hsplit > 1 ? a.hsplit : 1;
  p.bt_per_query = a.bt_per_query;
  p.bt_head_rows = a.bt_head_rows;
  p.window = a.qs.mode == DSA_MODE_DECODE ? a.window : 0;
  p.rows_per_q = p.pre_ml ? a.k : a.prefix + a.k;
  p.two_pass = 0;
  p.units1 = 0;
  p.grid1 = 0;
  if (a.prefix_ctas > 0 && a.qs.mode == DSA_MODE_DECODE && !p.pre_ml && a.prefix > 0 && a.kv.max_ctx > a.prefix) {
    p.two_pass = 1;
    p.rows_per_q = a.k > a.prefix ? a.k : a.prefix;
    p.units1 = (int)((long long)a.qs.n_q * a.prefix);
  }
  p.units = (int)((long long)a.qs.n_q * p.rows_per_q);
  p.part_o = a.ws.part_o;
  p.part_ml = a.ws.part_ml;
  p.out = a.out;
  p.out_dtype = a.out_dtype;
  p.lse = a.lse;
  int dev = 0;
  cudaGetDevice(&dev);
  int grid = (dev >= 0 && dev < 64 && g_attn_grid[dev] > 0) ? g_attn_grid[dev] : 148;
  if (grid > p.units) grid = p.units;
  if (p.two_pass) {
    p.grid1 = a.prefix_ctas < grid ? a.prefix_ctas : grid;
    if (p.grid1 > p.units1) p.grid1 = p.units1;
  }
  cudaError_t e;
  if (p.pre_ml) {  // prefill: the prefix part of every query first, per tile of queries
    e = launch_prefix_attn(a.kv, a.qs, a.q, a.hq, a.prefix, a.scale, a.ws.pre_ml, a.ws.pre_o, st);
    if (e != cudaSuccess) return e;
  }
  const dim3 block(kProducerThreads + 32 * a.kv.hkv);
  const bool ps = a.qs.mode == DSA_MODE_PREFILL;
  const bool tp = p.two_pass;
  if (p.group <= 8)
    e = ps   ? launch_pdl(sparse_attn_kernel<1, true, false>, dim3(grid), block, kSmemBytes, st, 1, p)
        : tp ? launch_pdl(sparse_attn_kernel<1, false, true>, dim3(grid), block, kSmemBytes, st, 1, p)
             : launch_pdl(sparse_attn_kernel<1, false, false>, dim3(grid), block, kSmemBytes, st, 1, p);
  else
    e = ps   ? launch_pdl(sparse_attn_kernel<2, true, false>, dim3(grid), block, kSmemBytes, st, 1, p)
        : tp ? launch_pdl(sparse_attn_kernel<2, false, true>, dim3(grid), block, kSmemBytes, st, 1, p)
             : launch_pdl(sparse_attn_kernel<2, false, false>, dim3(grid), block, kSmemBytes, st, 1, p);
  if (e != cudaSuccess) return e;
  if (p.two_pass)
    return launch_pdl(attn_combine2_kernel, dim3(a.qs.n_q, (a.hq + kCombHeads - 1) / kCombHeads),
                      dim3(kCombThreads), 0, st, 1, p, grid);
  if (grid < 2) return e;
  return launch_pdl(attn_combine_kernel, dim3(grid - 1), dim3(kCombThreads), 0, st, 1, p, grid);
}

cudaError_t read_clear_status_attn(int* code, cudaStream_t st) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v != 0) {
    const int z = 0;
    e = cudaMemcpyToSymbolAsync(g_status, &z, sizeof(int), 0, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (*code == 0) *code = v;
  }
  return e;
}

}  // namespace dsa
