// Step 2 of DSA (§2.1 top-k, §2.4 prefix never selected): turn scores and the
// selection threshold into the ascending list of selected positions.
//
// Decode (few queries, long rows): many CTAs per sequence.  Each compaction CTA
// owns 2048 positions and writes, in position order, every candidate at or
// above the threshold together with its rank among the ties of its chunk.  The
// last CTA of a sequence (ticket counter, no spin) lays the runs end to end:
// ties before a chunk decide how many of its ties are kept, so the lower
// positions win, and the result is deterministic and ascending.
//
// Prefill (many rows of at most a few ten thousand candidates): one CTA per
// query row builds its histogram in shared memory, finds the threshold and
// compacts the row in order with block-wide scans.
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace dsa {
namespace {

__device__ int g_status;

constexpr int kPer = kCompactChunk / kCompactThreads;  // 8 consecutive positions per thread
static_assert(kPer == 8, "compaction assumes 8 positions per thread");
constexpr int kStageEntries = 4096;                      // merge entries staged in shared memory
constexpr int kMaxChunks = 1024;                         // compaction chunks per sequence at most

struct CompactParams {
  const int32_t* scores;
  const int32_t* ctx;
  const int32_t* bt;
  int ld, prefix, k, max_ctx, max_blocks, num_blocks, hkv;
  SelState sel;
  int32_t* idx;
  int32_t* n_sel;
};

// Cache slot (block * 64 + row) of position t of sequence b.
__device__ __forceinline__ int slot_of(const CompactParams& p, int b, int t) {
  return load_block(p.bt, b, p.max_blocks, t >> 6, p.num_blocks, &g_status) * kBlock + (t & 63);
}

struct MergeSmem {
  int ent_pos[kStageEntries];
  int ent_score[kStageEntries];
  int run_off[kMaxChunks + 1];
  int fine[kFineBins];
  int misc[8];
  int scratch[40];
};

// Run entry e (flattened over the chunks of sequence b, in position order).
__device__ __forceinline__ void load_entry(const CompactParams& p, const MergeSmem& sm, int b, int nch, int e,
                                           bool staged, int* pos, int* score) {
  if (staged) {
    *pos = sm.ent_pos[e];
    *score = sm.ent_score[e];
    return;
  }
  int lo = 0, hi = nch - 1;  // last chunk with run_off <= e
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.run_off[mid] <= e) lo = mid; else hi = mid - 1;
  }
  const size_t at = ((size_t)b * nch + lo) * kCompactChunk + (e - sm.run_off[lo]);
  *pos = __ldcg(p.sel.run_pos + at);
  *score = __ldcg(p.sel.run_score + at);
}

// The last compaction CTA of sequence b: exact threshold from the fine bins,
// then every candidate run, in position order, filtered and written out.
__device__ void merge_runs(const CompactParams& p, int b, const int4 sel, MergeSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nch = p.sel.n_chunks;
  const int lo = sel.y, width = sel.z, above = sel.w;
  if (tid < kFineBins) sm.fine[tid] = 0;
  __syncthreads();
  // Fine-bin totals and run offsets (chunks in order).
  int carry = 0;
  for (int base = 0; base < nch; base += kCompactThreads) {
    const int c = base + tid;
    int run_len = 0;
    if (c < nch) {
      const int* rec = p.sel.chunk_rec + ((size_t)b * nch + c) * kRecInts;
      run_len = __ldcg(rec);
      for (int f = 0; f < width; ++f) {
        const int v = __ldcg(rec + 2 + f);
        if (v) atomicAdd(&sm.fine[f], v);
      }
    }
    int tot;
    const int ex = block_exclusive_scan(run_len, sm.scratch, &tot);
    if (c < nch) sm.run_off[c] = carry + ex;
    carry += tot;
  }
  __syncthreads();
  const int E = carry;
  if (tid == 0) {
    sm.run_off[nch] = E;
    // The k-th largest lies in fine bin f*: fewer than k - above candidates sit above it.
    const int kk = p.k - above;
    int cum = 0, fstar = 0;
    for (int f = width - 1; f >= 0; --f) {
      if (cum + sm.fine[f] >= kk) {
        fstar = f;
        break;
      }
      cum += sm.fine[f];
    }
    sm.misc[0] = lo + fstar;        // tau
    sm.misc[1] = p.k - above - cum;  // quota of ties at tau
  }
  __syncthreads();
  const int tau = sm.misc[0], quota = sm.misc[1];
  const bool staged = E <= kStageEntries;
  if (staged) {
    for (int c = warp; c < nch; c += kCompactThreads / 32) {
      const size_t run = ((size_t)b * nch + c) * kCompactChunk;
      const int off = sm.run_off[c], n = sm.run_off[c + 1] - off;
      for (int j = lane; j < n; j += 32) {
        sm.ent_pos[off + j] = __ldcg(p.sel.run_pos + run + j);
        sm.ent_score[off + j] = __ldcg(p.sel.run_score + run + j);
      }
    }
    __syncthreads();
  }
  // Each thread owns a contiguous slice of the entries.
  const int per = (E + kCompactThreads - 1) / kCompactThreads;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int n_eq = 0;
  for (int e = e0; e < e1; ++e) {
    int pos, sc;
    load_entry(p, sm, b, nch, e, staged, &pos, &sc);
    n_eq += sc == tau;
  }
  int tot;
  int tie = block_exclusive_scan(n_eq, sm.scratch, &tot);  // ties before this slice
  int n_take = 0;
  for (int e = e0, tr = tie; e < e1; ++e) {
    int pos, sc;
    load_entry(p, sm, b, nch, e, staged, &pos, &sc);
    if (sc > tau) ++n_take;
    else if (sc == tau) n_take += tr++ < quota;
  }
  int o = block_exclusive_scan(n_take, sm.scratch, &tot);
  int32_t* out = p.idx + (size_t)b * p.k;
  for (int e = e0, tr = tie; e < e1; ++e) {
    int pos, sc;
    load_entry(p, sm, b, nch, e, staged, &pos, &sc);
    const bool take = sc > tau || (sc == tau && tr++ < quota);
    if (take && o < p.k) {
      out[o] = pos;
      if (p.sel.slot) p.sel.slot[(size_t)b * p.k + o] = slot_of(p, b, pos);
    }
    o += take;
  }
  const int n_out = min(tot, p.k);
  for (int r = n_out + tid; r < p.k; r += kCompactThreads) out[r] = -1;
  if (tid == 0) {
    p.n_sel[b] = n_out;
    p.sel.done_cmp[b] = 0;
  }
}

__global__ void __launch_bounds__(kCompactThreads) decode_compact_kernel(const CompactParams p) {
  __shared__ MergeSmem sm;
  __shared__ int s_fine[kFineBins];
  __shared__ int s_last;
  const int tid = threadIdx.x, b = blockIdx.y, c = blockIdx.x;
  const int L = min(__ldg(p.ctx + b), p.max_ctx);
  const int n_cand = max(0, L - p.prefix);
  const int t_lo = max(p.prefix, c * kCompactChunk), t_hi = min(L, (c + 1) * kCompactChunk);
  int32_t* out = p.idx + (size_t)b * p.k;

  if (n_cand <= p.k) {  // every candidate is selected: position t goes to slot t - prefix
    for (int t = t_lo + tid; t < t_hi; t += kCompactThreads) {
      out[t - p.prefix] = t;
      if (p.sel.slot) p.sel.slot[(size_t)b * p.k + (t - p.prefix)] = slot_of(p, b, t);
    }
    if (c == 0) {
      for (int r = n_cand + tid; r < p.k; r += kCompactThreads) out[r] = -1;
      if (tid == 0) p.n_sel[b] = n_cand;
    }
    return;
  }

  const int4 sel = __ldcg(p.sel.sel + b);
  const int lo = sel.y, hi = sel.y + sel.z;  // candidates: s >= lo; fine bins: lo <= s < hi
  if (tid < kFineBins) s_fine[tid] = 0;
  const int t_base = c * kCompactChunk + tid * kPer;
  int v[kPer];
  if (t_base >= t_lo && t_base + kPer <= t_hi) {
    const int4* src = reinterpret_cast<const int4*>(p.scores + (size_t)b * p.ld + t_base);
    const int4 a = __ldg(src), bb = __ldg(src + 1);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = bb.x, v[5] = bb.y, v[6] = bb.z, v[7] = bb.w;
  } else {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int t = t_base + j;
      v[j] = (t >= t_lo && t < t_hi) ? __ldg(p.scores + (size_t)b * p.ld + t) : INT_MIN;
    }
  }
  __syncthreads();
  uint32_t cand = 0;
  int n_above = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int t = t_base + j;
    if (t >= t_lo && t < t_hi && v[j] >= lo) {
      cand |= 1u << j;
      if (v[j] >= hi) ++n_above;
      else atomicAdd(&s_fine[v[j] - lo], 1);
    }
  }
  int tot_len, tot_above;
  const int off = block_exclusive_scan(__popc(cand), sm.scratch, &tot_len);
  block_exclusive_scan(n_above, sm.scratch, &tot_above);
  const size_t run = ((size_t)b * p.sel.n_chunks + c) * kCompactChunk;
  int o = off;
#pragma unroll
  for (int j = 0; j < kPer; ++j)
    if ((cand >> j) & 1) {
      p.sel.run_pos[run + o] = t_base + j;
      p.sel.run_score[run + o] = v[j];
      ++o;
    }
  int* rec = p.sel.chunk_rec + ((size_t)b * p.sel.n_chunks + c) * kRecInts;
  if (tid == 0) {
    rec[0] = tot_len;
    rec[1] = tot_above;
  }
  if (tid < kFineBins) rec[2 + tid] = s_fine[tid];
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.sel.done_cmp + b, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  merge_runs(p, b, sel, sm);
}

// ---------------------------------------------------------------- prefill ---
constexpr int kRowThreads = 512;
constexpr int kScratchIntsTopk = 264;

struct RowTopkParams {
  const int32_t* scores;
  int ld, prefix, k, pos0, n_q;
  int32_t* idx;
  int32_t* n_sel;
};

__global__ void __launch_bounds__(kRowThreads) prefill_topk_kernel(const RowTopkParams p) {
  __shared__ int hist[kHistBins];
  __shared__ int scratch[kScratchIntsTopk];
  const int i = blockIdx.x, tid = threadIdx.x;
  const int pos = p.pos0 + i;
  const int n_cand = max(0, pos - p.prefix + 1);
  int32_t* out = p.idx + (size_t)i * p.k;
  const int32_t* row = p.scores + (size_t)i * p.ld + p.prefix;  // candidate j is position prefix + j
  if (n_cand <= p.k) {
    for (int j = tid; j < p.k; j += kRowThreads) out[j] = j < n_cand ? p.prefix + j : -1;
    if (tid == 0) p.n_sel[i] = n_cand;
    return;
  }
  for (int j = tid; j < kHistBins; j += kRowThreads) hist[j] = 0;
  __syncthreads();
  for (int j = tid; j < n_cand; j += kRowThreads) atomicAdd(&hist[hist_bin(__ldg(row + j))], 1);
  __syncthreads();
  auto lds = [&](int b) { return hist[b]; };
  const Sel s = selection_from_hist(lds, row, n_cand, p.k, scratch);

  // Ordered compaction: segments of kRowThreads * 8 candidates, 8 per thread.
  int carry_ties = 0, carry_out = 0;
  for (int seg = 0; seg < n_cand; seg += kRowThreads * 8) {
    const int j0 = seg + tid * 8;
    uint32_t gt_m = 0, eq_m = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u;
      if (j < n_cand) {
        const int v = __ldg(row + j);
        if (v > s.tau) gt_m |= 1u << u;
        if (v == s.tau) eq_m |= 1u << u;
      }
    }
    int tot;
    const int ties_before = block_exclusive_scan(__popc(eq_m), scratch, &tot) + carry_ties;
    carry_ties += tot;
    // Keep ties while the row-wide tie rank is below the quota.
    uint32_t keep = gt_m;
    int tr = ties_before;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if ((eq_m >> u) & 1) {
        if (tr < s.quota) keep |= 1u << u;
        ++tr;
      }
    const int off = block_exclusive_scan(__popc(keep), scratch, &tot) + carry_out;
    carry_out += tot;
    int o = off;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if ((keep >> u) & 1) {
        if (o < p.k) out[o] = p.prefix + j0 + u;
        ++o;
      }
  }
  carry_out = min(carry_out, p.k);
  for (int j = carry_out + tid; j < p.k; j += kRowThreads) out[j] = -1;
  if (tid == 0) p.n_sel[i] = carry_out;
}

}  // namespace

cudaError_t setup_topk_kernels() { return cudaSuccess; }

cudaError_t launch_decode_compact(const KV& kv, const int32_t* scores, int ld, int prefix, int k,
                                  const SelState& sel, int32_t* idx, int32_t* n_sel, cudaStream_t st) {
  CompactParams p;
  p.scores = scores;
  p.ctx = kv.context_lens;
  p.bt = kv.block_table;
  p.ld = ld;
  p.prefix = prefix;
  p.k = k;
  p.max_ctx = kv.max_ctx;
  p.max_blocks = kv.max_blocks;
  p.num_blocks = kv.num_blocks;
  p.hkv = kv.hkv;
  p.sel = sel;
  p.idx = idx;
  p.n_sel = n_sel;
  dim3 grid(sel.n_chunks, kv.batch);
  decode_compact_kernel<<<grid, kCompactThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill_topk(const QS& qs, const int32_t* scores, int ld, int prefix, int k, int32_t* idx,
                                int32_t* n_sel, cudaStream_t st) {
  RowTopkParams p;
  p.scores = scores;
  p.ld = ld;
  p.prefix = prefix;
  p.k = k;
  p.pos0 = qs.pos0;
  p.n_q = qs.n_q;
  p.idx = idx;
  p.n_sel = n_sel;
  prefill_topk_kernel<<<qs.n_q, kRowThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t read_clear_status_topk(int* code, cudaStream_t st) {
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
