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
#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace dsa {
namespace {

__device__ int g_status;

constexpr int kPer = kCompactChunk / kCompactThreads;  // 8 consecutive positions per thread
static_assert(kPer == 8, "compaction assumes 8 positions per thread");

struct CompactParams {
  const int32_t* scores;
  const int32_t* ctx;
  int ld, prefix, k, max_ctx;
  SelState sel;
  int32_t* idx;
  int32_t* n_sel;
};

// Lays the runs of sequence b end to end (the last compaction CTA of b).
__device__ void merge_runs(const CompactParams& p, int b, const int4 sel) {
  __shared__ int s_take[kCompactThreads], s_off[kCompactThreads], s_len[kCompactThreads];
  __shared__ int scratch[40];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nch = p.sel.n_chunks;
  const int quota = sel.w;
  int carry_ties = 0, carry_out = 0;
  int32_t* out = p.idx + (size_t)b * p.k;
  for (int base = 0; base < nch; base += kCompactThreads) {
    const int c = base + tid;
    int2 cnt = make_int2(0, 0);
    if (c < nch) cnt = __ldcg(p.sel.chunk_cnt + (size_t)b * nch + c);
    int tot;
    const int ties_before = block_exclusive_scan(cnt.y, scratch, &tot) + carry_ties;
    carry_ties += tot;
    const int take = min(max(quota - ties_before, 0), cnt.y);
    const int off = block_exclusive_scan(cnt.x + take, scratch, &tot) + carry_out;
    carry_out += tot;
    s_take[tid] = take;
    s_off[tid] = off;
    s_len[tid] = cnt.x + cnt.y;
    __syncthreads();
    const int ngrp = min(kCompactThreads, nch - base);
    for (int cc = warp; cc < ngrp; cc += kCompactThreads / 32) {
      const size_t run = ((size_t)b * nch + base + cc) * kCompactChunk;
      const int len = s_len[cc], tk = s_take[cc], o = s_off[cc];
      for (int j = lane; j < len; j += 32) {
        const int pos = __ldcg(p.sel.run_pos + run + j);
        const int info = __ldcg(p.sel.run_info + run + j);
        const int e = info >> 1;
        const int dst = o + (j - e) + min(e, tk);
        if ((!(info & 1) || e < tk) && dst < p.k) out[dst] = pos;  // bound holds unless the workspace was dirty
      }
    }
    __syncthreads();
  }
  carry_out = min(carry_out, p.k);
  for (int r = carry_out + tid; r < p.k; r += kCompactThreads) out[r] = -1;
  if (tid == 0) {
    p.n_sel[b] = carry_out;
    p.sel.ticket_c[b] = 0;
  }
}

__global__ void __launch_bounds__(kCompactThreads) decode_compact_kernel(const CompactParams p) {
  __shared__ int scratch[40];
  __shared__ int s_last;
  const int tid = threadIdx.x, b = blockIdx.y, c = blockIdx.x;
  const int L = min(__ldg(p.ctx + b), p.max_ctx);
  const int4 sel = __ldcg(p.sel.sel + b);
  const bool all = sel.x == kSelAll;
  const int tau = sel.y;
  const int t_lo = max(p.prefix, c * kCompactChunk), t_hi = min(L, (c + 1) * kCompactChunk);
  const int t_base = c * kCompactChunk + tid * kPer;

  int v[kPer];
  if (t_base + kPer <= t_hi && t_base >= t_lo) {
    const int4* src = reinterpret_cast<const int4*>(p.scores + (size_t)b * p.ld + t_base);
    const int4 a = __ldg(src), bb = __ldg(src + 1);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = bb.x, v[5] = bb.y, v[6] = bb.z, v[7] = bb.w;
  } else {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int t = t_base + j;
      v[j] = (t >= t_lo && t < t_hi) ? __ldg(p.scores + (size_t)b * p.ld + t) : 0;
    }
  }
  uint32_t gt_m = 0, eq_m = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int t = t_base + j;
    const bool in = t >= t_lo && t < t_hi;
    if (in && (all || v[j] > tau)) gt_m |= 1u << j;
    if (in && !all && v[j] == tau) eq_m |= 1u << j;
  }
  const int n_gt = __popc(gt_m), n_eq = __popc(eq_m);
  int tot_len, tot_eq;
  const int off = block_exclusive_scan(n_gt + n_eq, scratch, &tot_len);
  const int eq_off = block_exclusive_scan(n_eq, scratch, &tot_eq);
  const size_t run = ((size_t)b * p.sel.n_chunks + c) * kCompactChunk;
  int o = off, e = eq_off;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const bool g = (gt_m >> j) & 1, q = (eq_m >> j) & 1;
    if (g || q) {
      p.sel.run_pos[run + o] = t_base + j;
      p.sel.run_info[run + o] = (e << 1) | (q ? 1 : 0);
      ++o;
      e += q;
    }
  }
  if (tid == 0) p.sel.chunk_cnt[(size_t)b * p.sel.n_chunks + c] = make_int2(tot_len - tot_eq, tot_eq);
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.sel.ticket_c + b, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  merge_runs(p, b, sel);
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
  p.ld = ld;
  p.prefix = prefix;
  p.k = k;
  p.max_ctx = kv.max_ctx;
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
