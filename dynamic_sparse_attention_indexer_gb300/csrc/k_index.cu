// Step 1 of DSA (§2.1): indexer scores of each query against every causal
// non-prefix key, read from the paged int8 indexer cache (§2.2 blocks).
//
// Decode: one int8 dot product of 64 per position, a pure HBM stream of 64 B
// per position.  Whole 4 KB cache blocks are staged into shared memory with
// mbarrier-tracked bulk copies, several blocks in flight per CTA; each thread
// scores one position with __dp4a.  The fused variant also builds the score
// histogram the top-k needs (shared-memory bins merged into a per-sequence
// global histogram); the last CTA of a sequence turns it into the selection
// threshold, so no extra pass over the scores is needed.
//
// Prefill: the causal [T x 64] . [64 x L] int8 product on the tensor cores
// (mma.sync m16n8k32 s8, exact int32), 128 x 128 output tiles, fully masked
// tiles skipped.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace dsa {
namespace {

__device__ int g_status;

// ---------------------------------------------------------------- decode ---
// Persistent scoring: the candidate blocks of all sequences, [P / 64, ceil(L_b / 64))
// for each b, are laid end to end and cut into one contiguous range per CTA.  A CTA
// stages whole 4 KB blocks into shared memory with bulk copies (groups of up to four
// blocks of one sequence, five groups in flight), each thread scores one position.
constexpr int kIdxThreads = 256;
constexpr int kIdxStages = 5;
constexpr int kGroupBlocks = 4;                                // cache blocks per stage
constexpr int kIdxBlockBytes = kBlock * kIdxDim;               // 4096
constexpr int kIdxStageBytes = kGroupBlocks * kIdxBlockBytes;  // 16 KB
constexpr int kMaxRange = 1024;                                // candidate blocks per CTA at most
constexpr int kScratchInts = 264;

constexpr int idx_smem_bytes() {
  return kIdxStages * kIdxStageBytes + 16 * kIdxStages /*meta*/ + 8 * kIdxStages /*bars*/ +
         4 * (2 * kMaxDecodeBatch + 1) /*seg_start, len*/ + 4 * kMaxRange /*ids*/ + 4 * kCoarseBins /*hist*/ +
         4 * kScratchInts;
}

struct DecodeIndexParams {
  const int8_t* idx_cache;
  const int32_t* bt;
  const int32_t* ctx;
  const int8_t* q_idx;
  int* scores;
  int ld, max_blocks, num_blocks, prefix, max_ctx, batch, k;
  SelState sel;
};

// Candidate blocks of every sequence and their prefix sums: seg_start[b] is the
// first flattened block of sequence b, seg_start[batch] the total.
__device__ void candidate_blocks(const int32_t* __restrict__ ctx, int batch, int max_ctx, int prefix,
                                 int* seg_start, int* len, int* scratch) {
  int carry = 0;
  for (int base = 0; base < batch; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int nb = 0;
    if (b < batch) {
      const int L = min(__ldg(ctx + b), max_ctx);
      len[b] = L;
      nb = L > prefix ? (L + kBlock - 1) / kBlock - prefix / kBlock : 0;
    }
    int tot;
    const int ex = block_exclusive_scan(nb, scratch, &tot);
    if (b < batch) seg_start[b] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) seg_start[batch] = carry;
  __syncthreads();
}

// Selection of sequence b from its complete coarse histogram (the CTA whose
// counts completed it); leaves the histogram and the counter at zero.
__device__ void decode_finish(const SelState& st, int b, const int* cand_scores, int n_cand, int k,
                              int* scratch) {
  int* gh = st.coarse + (size_t)b * kCoarseBins;
  int beta, above;
  hist_threshold_bin<kCoarseBins>([gh](int i) { return __ldcg(gh + i); }, k, scratch, &beta, &above);
  if (beta > 0 && beta < kCoarseBins - 1) {
    if (threadIdx.x == 0) st.sel[b] = make_int4(kSelCoarse, (beta - kCoarseOff) * kFineBins, kFineBins, above);
  } else {
    int tau, n_gt;
    block_radix_select(cand_scores, n_cand, k, scratch, &tau, &n_gt);
    if (threadIdx.x == 0) st.sel[b] = make_int4(kSelExact, tau, 1, n_gt);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kCoarseBins; i += blockDim.x) gh[i] = 0;
  if (threadIdx.x == 0) st.done_idx[b] = 0;
}

// Adds this CTA's histogram of sequence b (covering `counted` candidates) to the
// sequence's and, if that completes it, computes the selection.
__device__ void flush_hist(const SelState& st, int* hist, int b, int counted, const int* cand_scores, int n_cand,
                           int k, int* scratch) {
  __syncthreads();
  int* gh = st.coarse + (size_t)b * kCoarseBins;
  for (int i = threadIdx.x; i < kCoarseBins; i += blockDim.x) {
    const int h = hist[i];
    if (h) {
      atomicAdd(gh + i, h);
      hist[i] = 0;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) scratch[263] = (atomicAdd(st.done_idx + b, counted) + counted == n_cand);
  __syncthreads();
  const bool last = scratch[263] != 0;
  __syncthreads();
  if (last) {
    __threadfence();
    decode_finish(st, b, cand_scores, n_cand, k, scratch);
    __syncthreads();
  }
}

template <bool kHist>
__global__ void __launch_bounds__(kIdxThreads) decode_index_kernel(const DecodeIndexParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  int4* meta = reinterpret_cast<int4*>(smem + kIdxStages * kIdxStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(meta + kIdxStages);
  int* seg_start = reinterpret_cast<int*>(bars + kIdxStages);
  int* len = seg_start + kMaxDecodeBatch + 1;
  int* ids = len + kMaxDecodeBatch;
  int* hist = ids + kMaxRange;
  int* scratch = hist + kCoarseBins;

  const int tid = threadIdx.x;
  const int P = p.prefix, jb_base = P / kBlock;
  candidate_blocks(p.ctx, p.batch, p.max_ctx, P, seg_start, len, scratch);
  const long long T = seg_start[p.batch];
  const int f_begin = (int)(T * blockIdx.x / gridDim.x), f_end = (int)(T * (blockIdx.x + 1) / gridDim.x);
  if (f_begin >= f_end) return;

  // Block ids of the whole range, loaded in parallel (validated against the pool).
  {
    int b = 0;
    for (int f = f_begin + tid; f < f_end; f += kIdxThreads) {
      int lo = 0, hi = p.batch - 1;  // last b with seg_start[b] <= f
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg_start[mid] <= f) lo = mid; else hi = mid - 1;
      }
      b = lo;
      ids[f - f_begin] = load_block(p.bt, b, p.max_blocks, f - seg_start[b] + jb_base, p.num_blocks, &g_status);
    }
  }
  if (kHist)
    for (int i = tid; i < kCoarseBins; i += kIdxThreads) hist[i] = 0;
  if (tid == 0) {
    for (int s = 0; s < kIdxStages; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  // Producer state (thread 0): next block to issue and its sequence.
  int f_next = f_begin, b_next = 0;
  if (tid == 0) {
    int lo = 0, hi = p.batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (seg_start[mid] <= f_next) lo = mid; else hi = mid - 1;
    }
    b_next = lo;
  }
  int n_groups_issued = 0;  // thread 0
  auto issue = [&]() {      // thread 0 only; returns false at the end of the range
    if (f_next >= f_end) return false;
    while (seg_start[b_next + 1] <= f_next) ++b_next;  // skip sequences without candidates
    const int s = n_groups_issued % kIdxStages;
    const int count = min(kGroupBlocks, min(f_end, seg_start[b_next + 1]) - f_next);
    meta[s] = make_int4(b_next, f_next - seg_start[b_next] + jb_base, count, 0);
    mbar_arrive_expect_tx(&bars[s], count * kIdxBlockBytes);
    for (int i = 0; i < count; ++i)
      bulk_g2s(stages + s * kIdxStageBytes + i * kIdxBlockBytes,
               p.idx_cache + (size_t)ids[f_next - f_begin + i] * kIdxBlockBytes, kIdxBlockBytes, &bars[s]);
    f_next += count;
    ++n_groups_issued;
    return true;
  };
  if (tid == 0)
    for (int s = 0; s < kIdxStages; ++s)
      if (!issue()) break;

  const int slot = tid >> 6, r = tid & 63;
  int qb = -1;
  int4 q[4];
  int hist_b = -1, counted = 0;  // sequence whose counts sit in `hist`, candidates counted
  for (int g = 0;; ++g) {
    // All threads learn whether group g exists: thread 0 issued it before this point.
    if (tid == 0) scratch[262] = g < n_groups_issued;
    __syncthreads();
    if (!scratch[262]) break;
    const int s = g % kIdxStages;
    const bool ok = mbar_wait(&bars[s], (g / kIdxStages) & 1);
    if (!ok) set_status(&g_status, kStTimeout);
    const int4 m = meta[s];
    const int b = m.x, L = len[m.x];
    const int n_cand = L - P;
    const bool want_hist = kHist && n_cand > p.k;
    if (kHist && b != hist_b) {
      if (hist_b >= 0 && counted > 0)
        flush_hist(p.sel, hist, hist_b, counted, p.scores + (size_t)hist_b * p.ld + P, len[hist_b] - P, p.k,
                   scratch);
      hist_b = want_hist ? b : -1;
      counted = 0;
    }
    const int t = (m.y + slot) * kBlock + r;
    const bool valid = ok && slot < m.z && t >= P && t < L;
    if (valid) {
      if (b != qb) {
        const int4* src = reinterpret_cast<const int4*>(p.q_idx + (size_t)b * kIdxDim);
        q[0] = __ldg(src), q[1] = __ldg(src + 1), q[2] = __ldg(src + 2), q[3] = __ldg(src + 3);
        qb = b;
      }
      const int4* row = reinterpret_cast<const int4*>(stages + s * kIdxStageBytes + slot * kIdxBlockBytes + r * kIdxDim);
      int acc = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int jj = (j + (r >> 1)) & 3;  // rotate 16-B chunks: conflict-free smem reads
        const int4 kv = row[jj];
        const int4 qv = jj == 0 ? q[0] : jj == 1 ? q[1] : jj == 2 ? q[2] : q[3];
        acc = dot4(kv.x, qv.x, acc);
        acc = dot4(kv.y, qv.y, acc);
        acc = dot4(kv.z, qv.z, acc);
        acc = dot4(kv.w, qv.w, acc);
      }
      p.scores[(size_t)b * p.ld + t] = acc;
      if (want_hist) atomicAdd(&hist[coarse_bin(acc)], 1);
    }
    if (want_hist) {
      // Candidates of this group: positions [max(P, first), min(L, last + 1)).
      const int first = max(P, m.y * kBlock), last = min(L, (m.y + m.z) * kBlock);
      counted += last - first;
    }
    if (__syncthreads_or(!ok)) {
      // A wait ran out: give the copies in flight a bounded chance to land, then leave.
      if (tid == 0)
        for (int gg = g; gg < n_groups_issued; ++gg) mbar_wait(&bars[gg % kIdxStages], (gg / kIdxStages) & 1);
      return;
    }
    if (tid == 0) issue();
  }
  if (kHist && hist_b >= 0 && counted > 0)
    flush_hist(p.sel, hist, hist_b, counted, p.scores + (size_t)hist_b * p.ld + P, len[hist_b] - P, p.k, scratch);
}

// Coarse histogram of existing scores (the stand-alone top-k call): one CTA per
// chunk of kCompactChunk positions of a sequence.
struct DecodeHistParams {
  const int32_t* scores;
  const int32_t* ctx;
  int ld, prefix, k, max_ctx;
  SelState sel;
};

__global__ void __launch_bounds__(256) decode_hist_kernel(const DecodeHistParams p) {
  __shared__ int hist[kCoarseBins];
  __shared__ int scratch[kScratchInts];
  const int b = blockIdx.y, c = blockIdx.x;
  const int L = min(__ldg(p.ctx + b), p.max_ctx);
  const int n_cand = L - p.prefix;
  if (n_cand <= p.k) return;  // the compaction takes every candidate
  const int t_lo = max(p.prefix, c * kCompactChunk), t_hi = min(L, (c + 1) * kCompactChunk);
  if (t_lo >= t_hi) return;
  for (int i = threadIdx.x; i < kCoarseBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int32_t* row = p.scores + (size_t)b * p.ld;
  for (int t = t_lo + threadIdx.x; t < t_hi; t += blockDim.x) atomicAdd(&hist[coarse_bin(__ldg(row + t))], 1);
  flush_hist(p.sel, hist, b, t_hi - t_lo, row + p.prefix, n_cand, p.k, scratch);
}

// --------------------------------------------------------------- prefill ---
constexpr int kPT = 128;  // query rows and key columns per tile

struct PrefillIndexParams {
  const int8_t* idx_cache;
  const int32_t* bt;
  const int8_t* q_idx;
  int* scores;
  int ld, max_blocks, num_blocks, prefix, seq, pos0, n_q;
};

// 64-byte rows, 16-byte chunks swizzled by (row >> 1) & 3: conflict-free ldmatrix.
__device__ __forceinline__ int swz64(int row, int chunk) { return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4); }

__global__ void __launch_bounds__(256) prefill_index_kernel(const PrefillIndexParams p) {
  __shared__ __align__(128) int8_t sA[kPT * kIdxDim];
  __shared__ __align__(128) int8_t sB[kPT * kIdxDim];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kPT, i0 = blockIdx.y * kPT;
  const int i_last = min(p.n_q, i0 + kPT) - 1;
  const int t_max = p.pos0 + i_last;  // largest key any query of the tile sees
  if (t0 > t_max || t0 + kPT - 1 < p.prefix) return;

  for (int cidx = tid; cidx < kPT * 4; cidx += 256) {
    const int row = cidx >> 2, ch = cidx & 3;
    const int i = i0 + row;
    cp_async16(sA + swz64(row, ch), p.q_idx + (size_t)min(i, p.n_q - 1) * kIdxDim + ch * 16, i < p.n_q ? 16u : 0u);
    const int t = t0 + row;
    const bool kv = t <= t_max;
    const int blk = kv ? load_block(p.bt, p.seq, p.max_blocks, t >> 6, p.num_blocks, &g_status) : 0;
    cp_async16(sB + swz64(row, ch), p.idx_cache + (size_t)blk * kIdxBlockBytes + (t & 63) * kIdxDim + ch * 16,
               kv ? 16u : 0u);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  const int wm = warp & 3, wn = warp >> 2;  // warp tile: 32 rows x 64 cols
  int acc[2][8][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[a][n][e] = 0;

  const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    uint32_t af[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int row = wm * 32 + mt * 16 + (mi & 1) * 8 + rr;
      ldsm_x4(smem_u32(sA + swz64(row, ks * 2 + (mi >> 1))), af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
    }
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b0, b1, b2, b3;
      const int row = wn * 64 + (2 * np + (mi >> 1)) * 8 + rr;
      ldsm_x4(smem_u32(sB + swz64(row, ks * 2 + (mi & 1))), b0, b1, b2, b3);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        mma_s8_16832(acc[mt][2 * np], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
        mma_s8_16832(acc[mt][2 * np + 1], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b2, b3);
      }
    }
  }

#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int i = i0 + wm * 32 + mt * 16 + hh * 8 + (lane >> 2);
      if (i >= p.n_q) continue;
      const int pos = p.pos0 + i;
      int* out = p.scores + (size_t)i * p.ld;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int t = t0 + wn * 64 + nt * 8 + (lane & 3) * 2;
        const int v0 = acc[mt][nt][2 * hh], v1 = acc[mt][nt][2 * hh + 1];
        if (t >= p.prefix && t + 1 <= pos) {
          *reinterpret_cast<int2*>(out + t) = make_int2(v0, v1);
        } else {
          if (t >= p.prefix && t <= pos) out[t] = v0;
          if (t + 1 >= p.prefix && t + 1 <= pos) out[t + 1] = v1;
        }
      }
    }
}

}  // namespace

namespace {
int g_index_grid[64] = {};  // persistent indexer CTAs per device (SMs x resident CTAs)
}

cudaError_t setup_index_kernels() {
  cudaError_t e = cudaFuncSetAttribute(decode_index_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       idx_smem_bytes());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_index_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             idx_smem_bytes());
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_index_kernel<true>, kIdxThreads,
                                                      idx_smem_bytes());
  if (e == cudaSuccess && dev >= 0 && dev < 64) g_index_grid[dev] = sms * (per_sm > 0 ? per_sm : 1);
  return e;
}

static int index_grid(const KV& kv, int prefix) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int base = (dev >= 0 && dev < 64 && g_index_grid[dev] > 0) ? g_index_grid[dev] : 304;
  // Upper bound of the candidate blocks; every CTA range must fit kMaxRange ids.
  const long long per_seq = (kv.max_ctx + kBlock - 1) / kBlock - prefix / kBlock;
  const long long t_max = (long long)kv.batch * (per_seq > 0 ? per_seq : 0);
  const long long need = (t_max + kMaxRange - 1) / kMaxRange;
  return (int)(need > base ? need : base);
}

cudaError_t launch_decode_index(const KV& kv, const int8_t* q_idx, int prefix, int* scores, int ld,
                                const SelState* sel, int k, cudaStream_t st) {
  DecodeIndexParams p;
  p.idx_cache = kv.idx_cache;
  p.bt = kv.block_table;
  p.ctx = kv.context_lens;
  p.q_idx = q_idx;
  p.scores = scores;
  p.ld = ld;
  p.max_blocks = kv.max_blocks;
  p.num_blocks = kv.num_blocks;
  p.prefix = prefix;
  p.max_ctx = kv.max_ctx;
  p.batch = kv.batch;
  p.k = k;
  if (sel) p.sel = *sel;
  const int grid = index_grid(kv, prefix);
  if (sel)
    decode_index_kernel<true><<<grid, kIdxThreads, idx_smem_bytes(), st>>>(p);
  else
    decode_index_kernel<false><<<grid, kIdxThreads, idx_smem_bytes(), st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_hist(const KV& kv, const int32_t* scores, int ld, int prefix, int k,
                               const SelState& sel, cudaStream_t st) {
  DecodeHistParams p;
  p.scores = scores;
  p.ctx = kv.context_lens;
  p.ld = ld;
  p.prefix = prefix;
  p.k = k;
  p.max_ctx = kv.max_ctx;
  p.sel = sel;
  dim3 grid((kv.max_ctx + kCompactChunk - 1) / kCompactChunk, kv.batch);
  decode_hist_kernel<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
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
  dim3 grid(last_pos / kPT + 1, (qs.n_q + kPT - 1) / kPT);
  prefill_index_kernel<<<grid, 256, 0, st>>>(p);
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
