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
constexpr int kIdxThreads = 256;
constexpr int kIdxStages = 4;
constexpr int kGroupBlocks = 4;                              // cache blocks per stage
constexpr int kIdxBlockBytes = kBlock * kIdxDim;             // 4096
constexpr int kIdxStageBytes = kGroupBlocks * kIdxBlockBytes;  // 16 KB
constexpr int kScratchInts = 264;

constexpr int idx_smem_bytes(bool hist) {
  return kIdxStages * kIdxStageBytes + 64 + 8 * kIdxStages + 4 * kScratchInts +
         (hist ? 4 * kHistBins : 0);
}

struct DecodeIndexParams {
  const int8_t* idx_cache;
  const int32_t* bt;
  const int32_t* ctx;
  const int8_t* q_idx;
  int* scores;
  int ld, max_blocks, num_blocks, prefix, chunk, k, max_ctx;
  SelState sel;
};

// Last CTA of sequence b: histogram -> selection, then leave the histogram and
// the ticket at zero for the next call.
__device__ void decode_finish(const SelState& st, int b, const int* cand_scores, int n_cand, int k,
                              int* scratch) {
  int* gh = st.hist + (size_t)b * kHistBins;
  auto ld = [gh](int i) { return __ldcg(gh + i); };
  const Sel s = selection_from_hist(ld, cand_scores, n_cand, k, scratch);
  if (threadIdx.x == 0) st.sel[b] = make_int4(s.mode, s.tau, s.n_gt, s.quota);
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) gh[i] = 0;
  if (threadIdx.x == 0) st.ticket_h[b] = 0;
}

// Merge a CTA's shared histogram into the sequence's and, if this CTA is the
// last of the sequence to do so, compute the selection.
__device__ void merge_and_finish(const SelState& st, const int* hist, int b, const int* cand_scores,
                                 int n_cand, int k, int* scratch) {
  __syncthreads();
  int* gh = st.hist + (size_t)b * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) {
    const int h = hist[i];
    if (h) atomicAdd(gh + i, h);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) scratch[263] = (atomicAdd(st.ticket_h + b, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (scratch[263]) {
    __threadfence();
    decode_finish(st, b, cand_scores, n_cand, k, scratch);
  }
}

template <bool kHist>
__global__ void __launch_bounds__(kIdxThreads) decode_index_kernel(const DecodeIndexParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  int4* q_s = reinterpret_cast<int4*>(smem + kIdxStages * kIdxStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kIdxStages * kIdxStageBytes + 64);
  int* scratch = reinterpret_cast<int*>(smem + kIdxStages * kIdxStageBytes + 64 + 8 * kIdxStages);
  int* hist = scratch + kScratchInts;

  const int tid = threadIdx.x, b = blockIdx.y, c = blockIdx.x;
  const int L = min(__ldg(p.ctx + b), p.max_ctx);  // never past the host bound
  const int t_lo = max(p.prefix, c * p.chunk), t_hi = min(L, (c + 1) * p.chunk);
  const int jb0 = t_lo / kBlock;
  const int nb = t_lo < t_hi ? (t_hi - 1) / kBlock - jb0 + 1 : 0;
  const int ngroups = (nb + kGroupBlocks - 1) / kGroupBlocks;

  if (kHist)
    for (int i = tid; i < kHistBins; i += kIdxThreads) hist[i] = 0;
  if (tid < 4) q_s[tid] = __ldg(reinterpret_cast<const int4*>(p.q_idx + (size_t)b * kIdxDim) + tid);
  if (tid == 0) {
    for (int s = 0; s < kIdxStages; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  auto issue = [&](int g) {
    const int s = g % kIdxStages;
    const int n_in = min(kGroupBlocks, nb - g * kGroupBlocks);
    mbar_arrive_expect_tx(&bars[s], n_in * kIdxBlockBytes);
    for (int i = 0; i < n_in; ++i) {
      const int blk = load_block(p.bt, b, p.max_blocks, jb0 + g * kGroupBlocks + i, p.num_blocks, &g_status);
      bulk_g2s(stages + s * kIdxStageBytes + i * kIdxBlockBytes, p.idx_cache + (size_t)blk * kIdxBlockBytes,
               kIdxBlockBytes, &bars[s]);
    }
  };
  int issued = 0;  // used by thread 0 only
  if (tid == 0)
    for (; issued < min(kIdxStages, ngroups); ++issued) issue(issued);

  const int slot = tid >> 6, r = tid & 63;
  int* out = p.scores + (size_t)b * p.ld;
  for (int g = 0; g < ngroups; ++g) {
    const int s = g % kIdxStages;
    const bool ok = mbar_wait(&bars[s], (g / kIdxStages) & 1);
    if (!ok) set_status(&g_status, kStTimeout);
    const int jb = g * kGroupBlocks + slot;
    const int t = (jb0 + jb) * kBlock + r;
    if (ok && jb < nb && t >= t_lo && t < t_hi) {
      const int4* row =
          reinterpret_cast<const int4*>(stages + s * kIdxStageBytes + slot * kIdxBlockBytes + r * kIdxDim);
      int acc = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int jj = (j + (r >> 1)) & 3;  // rotate 16-B chunks: conflict-free smem reads
        const int4 kv = row[jj];
        const int4 qv = q_s[jj];
        acc = dot4(kv.x, qv.x, acc);
        acc = dot4(kv.y, qv.y, acc);
        acc = dot4(kv.z, qv.z, acc);
        acc = dot4(kv.w, qv.w, acc);
      }
      out[t] = acc;
      if (kHist) atomicAdd(&hist[hist_bin(acc)], 1);
    }
    if (__syncthreads_or(!ok)) {
      // A wait ran out: give the copies still in flight a bounded chance to land, then leave.
      if (tid == 0)
        for (int gg = g; gg < issued; ++gg) mbar_wait(&bars[gg % kIdxStages], (gg / kIdxStages) & 1);
      return;
    }
    if (tid == 0 && issued < ngroups) issue(issued++);
  }
  if (kHist)
    merge_and_finish(p.sel, hist, b, p.scores + (size_t)b * p.ld + p.prefix, max(0, L - p.prefix), p.k,
                     scratch);
}

// Histogram of existing scores (the stand-alone top-k call).
struct DecodeHistParams {
  const int32_t* scores;
  const int32_t* ctx;
  int ld, prefix, chunk, k, max_ctx;
  SelState sel;
};

__global__ void __launch_bounds__(256) decode_hist_kernel(const DecodeHistParams p) {
  __shared__ int hist[kHistBins];
  __shared__ int scratch[kScratchInts];
  const int b = blockIdx.y, c = blockIdx.x;
  const int L = min(__ldg(p.ctx + b), p.max_ctx);
  const int t_lo = max(p.prefix, c * p.chunk), t_hi = min(L, (c + 1) * p.chunk);
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int32_t* row = p.scores + (size_t)b * p.ld;
  for (int t = t_lo + threadIdx.x; t < t_hi; t += blockDim.x) atomicAdd(&hist[hist_bin(__ldg(row + t))], 1);
  merge_and_finish(p.sel, hist, b, row + p.prefix, max(0, L - p.prefix), p.k, scratch);
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

int decode_index_chunk(int batch, int max_ctx) {
  const long long total = (long long)batch * max_ctx;
  int ch = 512;
  while (ch < 16384 && total / ch > 512) ch *= 2;
  return ch;
}

cudaError_t setup_index_kernels() {
  cudaError_t e = cudaFuncSetAttribute(decode_index_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       idx_smem_bytes(true));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_index_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              idx_smem_bytes(false));
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
  p.chunk = decode_index_chunk(kv.batch, kv.max_ctx);
  p.k = k;
  p.max_ctx = kv.max_ctx;
  if (sel) p.sel = *sel;
  dim3 grid((kv.max_ctx + p.chunk - 1) / p.chunk, kv.batch);
  if (sel)
    decode_index_kernel<true><<<grid, kIdxThreads, idx_smem_bytes(true), st>>>(p);
  else
    decode_index_kernel<false><<<grid, kIdxThreads, idx_smem_bytes(false), st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_hist(const KV& kv, const int32_t* scores, int ld, int prefix, int k,
                               const SelState& sel, cudaStream_t st) {
  DecodeHistParams p;
  p.scores = scores;
  p.ctx = kv.context_lens;
  p.ld = ld;
  p.prefix = prefix;
  p.chunk = decode_index_chunk(kv.batch, kv.max_ctx);
  p.k = k;
  p.max_ctx = kv.max_ctx;
  p.sel = sel;
  dim3 grid((kv.max_ctx + p.chunk - 1) / p.chunk, kv.batch);
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
