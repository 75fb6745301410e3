// Step 1 of DSA (§2.1): indexer scores of each query against every causal
// non-prefix key, read from the paged int8 indexer cache (§2.2 blocks).
//
// Decode: one int8 dot product of 64 per position, a pure HBM stream of 64 B
// per position.  Whole 4 KB cache blocks are staged into shared memory with
// mbarrier-tracked bulk copies by a producer warp, eight 16 KB stages in flight
// per SM; consumer warps score one position per thread with __dp4a.  The fused
// variant also builds the coarse score histogram the top-k needs (per-warp
// shared-memory bins added into a per-sequence global histogram), so the
// selection needs no extra pass over the scores to find its threshold window.
//
// Prefill: the causal [T x 64] . [64 x L] int8 product on the fifth-generation
// tensor cores (tcgen05.mma, e4m3 or f16 operands, fp32 accumulation in tensor
// memory, exact), 128 x 256 output tiles, fully masked tiles skipped.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "score_walk.cuh"
#include "tc.cuh"

namespace dsa {
namespace {

__device__ int g_status;

// ---------------------------------------------------------------- decode ---
// Persistent scoring: the candidate blocks of all sequences, [P / 64, ceil(L_b / 64))
// for each b, are laid end to end and cut into one contiguous range per CTA (one
// CTA per SM).  Warp roles: lanes 0-3 of warp 0 stage groups of up to four
// whole 4 KB blocks of one sequence with bulk copies into a ring of
// kIdxStages 16 KB stages (mbarrier full / empty per stage); the eight
// consumer warps score one position per thread with __dp4a and release the
// stage, with no CTA-wide barrier per group.  Every warp walks the same group
// sequence, computed from the block ranges.  With the histogram, each consumer
// warp counts its scores into its own shared 1024-bin coarse histogram; when
// the sequence changes (and at the end) the eight are summed and added to the
// sequence's global histogram (fire-and-forget atomics; the selection kernel
// reads the completed histogram).
constexpr int kIdxConsumers = 8;                               // consumer warps
constexpr int kIdxThreads = 32 * (1 + kIdxConsumers);          // 288
constexpr int kIdxStages = 8;          // ring stages; 6 where the selection CTAs are to fit beside
constexpr int kIdxStagesShared = 6;    // a scoring CTA (they are then resident before it ends)
constexpr int kIdxBlockBytes = kBlock * kIdxDim;               // 4096
constexpr int kIdxStageBytes = kGroupBlocks * kIdxBlockBytes;  // 16 KB
constexpr int kMaxRange = 2048;                                // candidate blocks per CTA at most
constexpr int kScratchInts = 64;

constexpr int idx_smem_bytes(int stages = kIdxStages) {
  return stages * kIdxStageBytes + 16 * stages /*bars*/ + 4 * (2 * kMaxDecodeBatch + 1) /*seg_start, len*/ +
         4 * kMaxRange /*ids*/ + 4 * kIdxConsumers * kCoarseBins /*hist*/ + 4 * kScratchInts + 16;
}

struct DecodeIndexParams {
  const int8_t* idx_cache;
  const int32_t* bt;
  const int32_t* ctx;
  const int8_t* q_idx;
  int* scores;
  int* coarse;  // [B][kCoarseBins] global histograms, or nullptr
  int ld, max_blocks, num_blocks, prefix, max_ctx, batch, k;
  // Per-KV-head indexer (hsplit = Hkv > 1): row v = b * hsplit + h scores head
  // h's keys, block id blk * hsplit + h of the indexer cache, blk from the
  // shared table (row b) or from head h's own table (bt_heads[h][b]); ctx per
  // sequence; num_blocks counts the KV cache's blocks.
  int hsplit, real_batch;
  const int32_t* bt_heads;
};

// Block id of block-table slot j of row v, checked against the pool.
__device__ __forceinline__ int row_block(const DecodeIndexParams& p, int v, int j) {
  if (p.hsplit <= 1) return load_block(p.bt, v, p.max_blocks, j, p.num_blocks, &g_status);
  const int b = v / p.hsplit, h = v - b * p.hsplit;
  const int blk = p.bt_heads ? load_block(p.bt_heads, h * p.real_batch + b, p.max_blocks, j, p.num_blocks, &g_status)
                             : load_block(p.bt, b, p.max_blocks, j, p.num_blocks, &g_status);
  return blk * p.hsplit + h;
}

// Sums the consumer warps' histograms of one sequence into its global one
// (called by all consumer threads, ct = 0 .. 255); with `clear` the warp
// histograms are zeroed for the next sequence before anyone counts again.
__device__ __forceinline__ void flush_cta_hist(int* hist, int* gh, int ct, bool clear) {
  constexpr int kConsumerThreads = 32 * kIdxConsumers;
  named_bar_sync(1, kConsumerThreads);  // every warp's counts are in
  for (int i = ct; i < kCoarseBins; i += kConsumerThreads) {
    int sum = 0;
#pragma unroll
    for (int w = 0; w < kIdxConsumers; ++w) {
      sum += hist[w * kCoarseBins + i];
      if (clear) hist[w * kCoarseBins + i] = 0;
    }
    if (sum) atomicAdd(gh + i, sum);
  }
  if (clear) named_bar_sync(1, kConsumerThreads);
}

template <bool kHist, int kStg>
__global__ void __launch_bounds__(kIdxThreads, 1) decode_index_kernel(const DecodeIndexParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStg * kIdxStageBytes);
  uint64_t* empty = full + kStg;
  int* seg_start = reinterpret_cast<int*>(empty + kStg);
  int* len = seg_start + kMaxDecodeBatch + 1;
  int* ids = len + kMaxDecodeBatch;
  int* hist = ids + kMaxRange;
  int* scratch = hist + kIdxConsumers * kCoarseBins;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = p.prefix, jb_base = P / kBlock;
  // Set-up before the wait on the previous kernel of the stream, so that it
  // overlaps that kernel's tail: shared memory, then the inputs no kernel of
  // the step writes (context lengths, block table, the indexer cache outside
  // each sequence's newest position; the caller's contract in dsa.h).  The
  // scores and histograms are written only after the wait.
  if (kHist)
    for (int i = tid; i < kIdxConsumers * kCoarseBins; i += kIdxThreads) hist[i] = 0;
  if (tid == 0) {
    for (int s = 0; s < kStg; ++s) {
      mbar_init(&full[s], kGroupBlocks);
      mbar_init(&empty[s], kIdxConsumers);
    }
    mbar_fence_init();
  }
  candidate_blocks(p.ctx, p.batch, p.max_ctx, P, seg_start, len, scratch, p.hsplit);
  const long long T = seg_start[p.batch];
  const int f_begin = (int)(T * blockIdx.x / gridDim.x), f_end = (int)(T * (blockIdx.x + 1) / gridDim.x);
  if (f_begin >= f_end) return;
  int b_first = 0;  // sequence of the range's first block
  {
    int lo = 0, hi = p.batch - 1;  // last b with seg_start[b] <= f_begin
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (seg_start[mid] <= f_begin) lo = mid; else hi = mid - 1;
    }
    b_first = lo;
  }
  // Block ids of the whole range, loaded in parallel (validated against the pool).
  for (int f = f_begin + tid; f < f_end; f += kIdxThreads) {
    int lo = b_first, hi = p.batch - 1;  // last b with seg_start[b] <= f
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (seg_start[mid] <= f) lo = mid; else hi = mid - 1;
    }
    ids[f - f_begin] = row_block(p, lo, f - seg_start[lo] + jb_base);
  }
  __syncthreads();
  GroupCursor cur{f_begin, f_end, b_first};
  Group g;

  if (warp == 0) {
    // ---- producer: lane i < 4 copies block i of each group.  The first
    // groups are copied before the wait on the previous kernel, up to the ring
    // size or the first group holding a sequence's newest position (which the
    // cache write of this step may be the previous kernel to write).
    if (lane >= kGroupBlocks) return;
    const uint64_t stream_policy = l2_evict_first();  // each key block is read once per call
    bool waited = false;
    for (int n = 0; next_group(cur, seg_start, jb_base, &g); ++n) {
      const int s = n % kStg;
      const int newest_jb = (len[g.b] - 1) >> 6;
      if (!waited && (n >= kStg || (newest_jb >= g.jb && newest_jb < g.jb + g.count))) {
        pdl_wait();
        pdl_trigger();
        waited = true;
      }
      if (n >= kStg && !mbar_wait(&empty[s], ((n / kStg) - 1) & 1)) {
        set_status(&g_status, kStTimeout);
        return;
      }
      const bool mine = lane < g.count;
      mbar_arrive_expect_tx(&full[s], mine ? kIdxBlockBytes : 0);
      if (mine) {
        const int f = cur.f - g.count + lane;  // flattened block of this lane
        bulk_g2s_hint(stages + s * kIdxStageBytes + lane * kIdxBlockBytes,
                      p.idx_cache + (size_t)ids[f - f_begin] * kIdxBlockBytes, kIdxBlockBytes, &full[s],
                      stream_policy);
      }
    }
    return;
  }

  pdl_wait();
  pdl_trigger();
  // ---- consumers: warp cw scores rows 32 (cw % 2) .. + 31 of block cw / 2 of each
  // group.  Four lanes share a row, lane l taking the 16-byte chunk l % 4 of the
  // key (so its query chunk is fixed and the warp's shared-memory reads are 512
  // contiguous bytes), and a two-step shuffle sums the four partial dot products.
  const int cw = warp - 1;
  const int blk = cw >> 1, row0 = (cw & 1) * 32;
  int* whist = hist + cw * kCoarseBins;
  int qb = -1;
  int4 qc = make_int4(0, 0, 0, 0);  // chunk lane % 4 of the current sequence's query
  int hist_b = -1;                  // sequence whose counts sit in whist
  for (int n = 0; next_group(cur, seg_start, jb_base, &g); ++n) {
    const int s = n % kStg;
    const int b = g.b, L = len[b];
    const bool want_hist = kHist && L - P > p.k;
    if (kHist && b != hist_b) {  // the same group sequence in every consumer warp: uniform
      if (hist_b >= 0) flush_cta_hist(hist, p.coarse + (size_t)hist_b * kCoarseBins, tid - 32, true);
      hist_b = want_hist ? b : -1;
    }
    if (b != qb) {
      qc = __ldg(reinterpret_cast<const int4*>(p.q_idx + (size_t)b * kIdxDim) + (lane & 3));
      qb = b;
    }
    if (!mbar_wait(&full[s], (n / kStg) & 1)) {
      set_status(&g_status, kStTimeout);
      break;
    }
    if (blk < g.count) {
      const uint8_t* base = stages + s * kIdxStageBytes + blk * kIdxBlockBytes + row0 * kIdxDim;
      int mine = 0;  // score of row row0 + lane
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int4 kv = *reinterpret_cast<const int4*>(base + (8 * i + (lane >> 2)) * kIdxDim + (lane & 3) * 16);
        int acc = dot4(kv.x, qc.x, 0);
        acc = dot4(kv.y, qc.y, acc);
        acc = dot4(kv.z, qc.z, acc);
        acc = dot4(kv.w, qc.w, acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        const int v = __shfl_sync(0xffffffffu, acc, 4 * (lane & 7));  // row 8 i + lane % 8
        if ((lane >> 3) == i) mine = v;
      }
      const int t = (g.jb + blk) * kBlock + row0 + lane;
      if (t >= P && t < L) {
        p.scores[(size_t)b * p.ld + t] = mine;
        if (want_hist) atomicAdd(&whist[coarse_bin(mine)], 1);
      }
    }
    fence_proxy_async_smem();  // the stage is refilled by bulk copies
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (kHist && hist_b >= 0) flush_cta_hist(hist, p.coarse + (size_t)hist_b * kCoarseBins, tid - 32, false);
}

// Coarse histogram of existing scores (the stand-alone top-k call): one CTA per
// chunk of kHistChunk positions of a sequence, added to the sequence's global
// histogram with fire-and-forget atomics.
constexpr int kHistChunk = 2048;
struct DecodeHistParams {
  const int32_t* scores;
  const int32_t* ctx;
  int* coarse;
  int ld, prefix, k, max_ctx;
};

__global__ void __launch_bounds__(256) decode_hist_kernel(const DecodeHistParams p) {
  __shared__ int hist[kCoarseBins];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.y, c = blockIdx.x;
  const int L = min(__ldg(p.ctx + b), p.max_ctx);
  const int n_cand = L - p.prefix;
  if (n_cand <= p.k) return;  // the selection takes every candidate
  const int t_lo = max(p.prefix, c * kHistChunk), t_hi = min(L, (c + 1) * kHistChunk);
  if (t_lo >= t_hi) return;
  for (int i = threadIdx.x; i < kCoarseBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int32_t* row = p.scores + (size_t)b * p.ld;
  for (int t = t_lo + threadIdx.x; t < t_hi; t += blockDim.x) atomicAdd(&hist[coarse_bin(__ldg(row + t))], 1);
  __syncthreads();
  int* gh = p.coarse + (size_t)b * kCoarseBins;
  for (int i = threadIdx.x; i < kCoarseBins; i += blockDim.x)
    if (hist[i]) atomicAdd(gh + i, hist[i]);
}

// --------------------------------------------------------------- prefill ---
// The causal [T x 64] . [64 x L] product on the fifth-generation tensor cores:
// one CTA per tile of 128 queries x 256 keys (tiles wholly above the diagonal
// or inside the prefix are skipped).  The four warps load the tile's int8 rows
// (the keys through the block table), check whether every value lies in
// [-16, 16], and convert them into the tensor-core operand layout: e4m3 when
// they do (exact: e4m3 holds every integer up to 16), f16 otherwise (exact for
// every int8).  One thread issues the MMAs (tcgen05.mma kind::f8f6f4, 2 x K=32,
// or kind::f16, 4 x K=16), accumulating in fp32 in tensor memory: every product
// and partial sum is an integer below 2^24 in magnitude (64 x 128 x 128 = 2^20),
// so the fp32 result is the exact integer.  The epilogue reads the 128 x 256
// accumulator back (each thread one query row) and stores the causal,
// non-prefix part as int32.
constexpr int kTcM = 128, kTcN = 256, kTcThreads = 128;
constexpr int kTcSmem = 1024 + 16384 + 32768 + 64;  // alignment slack, A, B (f16 sizes), barrier + TMEM slot
// One or two CTAs per SM: their accumulators (256 TMEM columns each) fit the
// 512 columns of an SM, so no CTA waits for tensor memory.
constexpr int kTcSmemAlloc = 80 * 1024;

struct PrefillIndexParams {
  const int8_t* idx_cache;
  const int32_t* bt;
  const int8_t* q_idx;
  int* scores;
  int ld, max_blocks, num_blocks, prefix, seq, pos0, n_q;
};

__device__ __forceinline__ bool any_above16(int4 v) {
  const int w[4] = {v.x, v.y, v.z, v.w};
  bool big = false;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int x = (int)(int8_t)((unsigned)w[i] >> (8 * b));
      big |= x > 16 || x < -16;
    }
  return big;
}
__device__ __forceinline__ int sx8(int w, int b) { return (int)(int8_t)((unsigned)w >> (8 * b)); }

// Row r of an operand: 64 int8 values (4 int4) to e4m3 (64 bytes, 64-byte
// swizzle) or to f16 (128 bytes, 128-byte swizzle).
__device__ __forceinline__ void store_row_e4m3(uint8_t* op, int r, const int4 (&v)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = (uint32_t)e4m3x2((float)sx8(w[i], 0), (float)sx8(w[i], 1)) |
             ((uint32_t)e4m3x2((float)sx8(w[i], 2), (float)sx8(w[i], 3)) << 16);
    *reinterpret_cast<uint4*>(op + (r >> 3) * 512 + (r & 7) * 64 + ((c ^ ((r & 7) >> 1)) << 4)) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}
__device__ __forceinline__ void store_row_f16(uint8_t* op, int r, const int4 (&v)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // int4 c holds values 16 c .. 16 c + 15: f16 chunks 2 c and 2 c + 1
    const int w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 lo = __halves2half2(__int2half_rn(sx8(w[i], 0)), __int2half_rn(sx8(w[i], 1)));
      const __half2 hi = __halves2half2(__int2half_rn(sx8(w[i], 2)), __int2half_rn(sx8(w[i], 3)));
      o[2 * i] = *reinterpret_cast<const uint32_t*>(&lo);
      o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hi);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ch = 2 * c + h;
      *reinterpret_cast<uint4*>(op + (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4)) =
          make_uint4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]);
    }
  }
}

__global__ void __launch_bounds__(kTcThreads) prefill_index_kernel(const PrefillIndexParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = base;          // A: 128 query rows
  uint8_t* sb = base + 16384;  // B: 256 key rows
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + 16384 + 32768);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kTcN, i0 = blockIdx.y * kTcM;
  const int i_last = min(p.n_q, i0 + kTcM) - 1;
  const int t_max = p.pos0 + i_last;  // largest key any query of the tile sees
  if (t0 > t_max || t0 + kTcN - 1 < p.prefix) return;

  if (warp == 0) tmem_alloc(tslot, kTcN);
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  // Rows: query i0 + tid; keys t0 + tid and t0 + 128 + tid (zero past the
  // last query / the last key the tile needs).
  int4 qv[4], kv[2][4];
  {
    const int i = i0 + tid;
    const int4* src = reinterpret_cast<const int4*>(p.q_idx + (size_t)min(i, p.n_q - 1) * kIdxDim);
#pragma unroll
    for (int c = 0; c < 4; ++c) qv[c] = i < p.n_q ? __ldg(src + c) : make_int4(0, 0, 0, 0);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = t0 + 128 * h + tid;
      const bool ok = t <= t_max;
      const int blk = ok ? load_block(p.bt, p.seq, p.max_blocks, t >> 6, p.num_blocks, &g_status) : 0;
      const int4* ks = reinterpret_cast<const int4*>(p.idx_cache + ((size_t)blk * kBlock + (t & 63)) * kIdxDim);
#pragma unroll
      for (int c = 0; c < 4; ++c) kv[h][c] = ok ? __ldg(ks + c) : make_int4(0, 0, 0, 0);
    }
  }
  bool big = false;
#pragma unroll
  for (int c = 0; c < 4; ++c) big |= any_above16(qv[c]) | any_above16(kv[0][c]) | any_above16(kv[1][c]);
  const bool f16 = __syncthreads_or(big) != 0;
  if (!f16) {
    store_row_e4m3(sa, tid, qv);
    store_row_e4m3(sb, tid, kv[0]);
    store_row_e4m3(sb, tid + 128, kv[1]);
  } else {
    store_row_f16(sa, tid, qv);
    store_row_f16(sb, tid, kv[0]);
    store_row_f16(sb, tid + 128, kv[1]);
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) {
    if (!f16) {
      constexpr uint32_t idesc = mma_idesc(kTcM, kTcN, 0);
#pragma unroll
      for (int k = 0; k < 2; ++k)
        mma_f8(tmem, smem_desc(smem_u32(sa) + 32 * k, 512, kSwizzle64), smem_desc(smem_u32(sb) + 32 * k, 512, kSwizzle64),
               idesc, k > 0);
    } else {
      constexpr uint32_t idesc = mma_idesc(kTcM, kTcN, 0);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_f16(tmem, smem_desc(smem_u32(sa) + 32 * k, 1024, kSwizzle128),
                smem_desc(smem_u32(sb) + 32 * k, 1024, kSwizzle128), idesc, k > 0);
    }
    mma_commit(bar);
  }
  if (!mbar_wait(bar, 0)) set_status(&g_status, kStTimeout);
  tc_fence_after();
  // Epilogue, 8 chunks of 32 keys: each thread reads its query row's 32
  // accumulators from tensor memory into the warp's staging area (the operand
  // memory is free now; row pitch 33 words: conflict-free both ways), then the
  // warp stores 4 rows of 128 bytes per instruction (8 lanes per row).
  int* stage = reinterpret_cast<int*>(base) + warp * 32 * 33;
  const int sub_r = lane >> 3, sub_c = (lane & 7) * 4;
#pragma unroll 1
  for (int c = 0; c < kTcN / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * c, r);
#pragma unroll
    for (int j = 0; j < 32; ++j) stage[lane * 33 + j] = __float2int_rn(__uint_as_float(r[j]));
    __syncwarp();
    const int t = t0 + 32 * c + sub_c;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int rw = 4 * m + sub_r;
      const int i = i0 + 32 * warp + rw;
      const int pos = p.pos0 + i;
      const int* sv = stage + rw * 33 + sub_c;
      if (i < p.n_q && t + 3 >= p.prefix && t <= pos) {
        int* dst = p.scores + (size_t)i * p.ld + t;
        if (t >= p.prefix && t + 3 <= pos) {
          *reinterpret_cast<int4*>(dst) = make_int4(sv[0], sv[1], sv[2], sv[3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (t + q >= p.prefix && t + q <= pos) dst[q] = sv[q];
        }
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTcN);
}

}  // namespace

namespace {
int g_index_grid[64] = {};  // persistent indexer CTAs per device (SMs x resident CTAs)
}

cudaError_t setup_index_kernels() {
  cudaError_t e = cudaFuncSetAttribute(prefill_index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemAlloc);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_index_kernel<true, kIdxStages>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, idx_smem_bytes());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_index_kernel<false, kIdxStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             idx_smem_bytes());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_index_kernel<true, kIdxStagesShared>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, idx_smem_bytes(kIdxStagesShared));
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_index_kernel<true, kIdxStages>, kIdxThreads,
                                                      idx_smem_bytes());
  if (e == cudaSuccess && dev >= 0 && dev < 64) g_index_grid[dev] = sms * (per_sm > 0 ? per_sm : 1);
  return e;
}

static int index_grid(const KV& kv, int prefix) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int base = (dev >= 0 && dev < 64 && g_index_grid[dev] > 0) ? g_index_grid[dev] : 148;
  // Upper bound of the candidate blocks; every CTA range must fit kMaxRange ids.
  const long long per_seq = (kv.max_ctx + kBlock - 1) / kBlock - prefix / kBlock;
  const long long t_max = (long long)kv.batch * (per_seq > 0 ? per_seq : 0);
  const long long need = (t_max + kMaxRange - 1) / kMaxRange;
  return (int)(need > base ? need : base);
}

cudaError_t launch_decode_index(const KV& kv, const int8_t* q_idx, int prefix, int* scores, int ld,
                                const SelState* sel, int k, cudaStream_t st, bool early, int hsplit,
                                const int32_t* bt_heads) {
  DecodeIndexParams p;
  p.hsplit = hsplit > 1 ? hsplit : 1;
  p.real_batch = kv.batch / p.hsplit;
  p.bt_heads = bt_heads;
  p.idx_cache = kv.idx_cache;
  p.bt = kv.block_table;
  p.ctx = kv.context_lens;
  p.q_idx = q_idx;
  p.scores = scores;
  p.coarse = sel ? sel->coarse : nullptr;
  p.ld = ld;
  p.max_blocks = kv.max_blocks;
  p.num_blocks = kv.num_blocks / p.hsplit;
  p.prefix = prefix;
  p.max_ctx = kv.max_ctx;
  p.batch = kv.batch;
  p.k = k;
  const int grid = index_grid(kv, prefix);
  // In the fused step, where the selection packs its CTAs (they do not each
  // take an SM), a smaller ring lets them be resident beside the scoring CTAs
  // before those end (measured at 128K, B = 8: step 48.3 -> 47.9 us; where the
  // selection has one CTA per SM the larger ring streams faster).
  auto kern = sel && !decode_select_spread(kv, prefix) ? decode_index_kernel<true, kIdxStagesShared>
               : sel                                    ? decode_index_kernel<true, kIdxStages>
                                                        : decode_index_kernel<false, kIdxStages>;
  const size_t smem = sel && !decode_select_spread(kv, prefix) ? idx_smem_bytes(kIdxStagesShared) : idx_smem_bytes();
  // early = false: the block table or context lengths come from the previous
  // kernel of the stream, so the pre-wait reads must not start before it ends.
  if (!early) return launch_ordered(kern, dim3(grid), dim3(kIdxThreads), smem, st, p);
  return launch_pdl(kern, dim3(grid), dim3(kIdxThreads), smem, st, 1, p);
}

cudaError_t launch_decode_hist(const KV& kv, const int32_t* scores, int ld, int prefix, int k,
                               const SelState& sel, cudaStream_t st) {
  DecodeHistParams p;
  p.scores = scores;
  p.ctx = kv.context_lens;
  p.coarse = sel.coarse;
  p.ld = ld;
  p.prefix = prefix;
  p.k = k;
  p.max_ctx = kv.max_ctx;
  dim3 grid((kv.max_ctx + kHistChunk - 1) / kHistChunk, kv.batch);
  return launch_pdl(decode_hist_kernel, grid, dim3(256), 0, st, 1, p);
}

cudaError_t launch_prefill_index(const KV& kv, const QS& qs, const int8_t* q_idx, int prefix, int* scores,
                                 int ld, cudaStream_t st) {
  PrefillIndexParams p;
  p.idx_cache = kv.idx_cache;
  p.bt = kv.block_table;
  p.q_idx = q_idx;
  p.scores = scores;
  p.ld = ld;
  p.max_blocks = kv.max_blocks;
  p.num_blocks = kv.num_blocks;
  p.prefix = prefix;
  p.seq = qs.seq;
  p.pos0 = qs.pos0;
  p.n_q = qs.n_q;
  const int last_pos = qs.pos0 + qs.n_q - 1;
  static_assert(kTcSmem <= kTcSmemAlloc, "prefill indexer shared memory");
  dim3 grid(last_pos / kTcN + 1, (qs.n_q + kTcM - 1) / kTcM);
  prefill_index_kernel<<<grid, kTcThreads, kTcSmemAlloc, st>>>(p);
  return cudaGetLastError();
}

cudaError_t read_clear_status_index(int* code, cudaStream_t st) {
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
