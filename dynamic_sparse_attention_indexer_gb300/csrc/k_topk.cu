// Step 2 of DSA (§2.1 top-k, §2.4 prefix never selected): turn scores and the
// selection threshold into the ascending list of selected positions.
//
// Decode (few queries, long rows): one cluster of CTAs per sequence, the CTAs
// exchanging their counts through distributed shared memory (below).  The
// result is deterministic and ascending; among equal scores the lower
// positions win.
//
// Prefill (many rows of at most a few ten thousand candidates): one warp per
// query row, histogram, threshold and ordered compaction all within the warp.
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace dsa {
namespace {

__device__ int g_status;

// Decode selection: one thread-block cluster of C CTAs per sequence (C = 1 ..
// 16, chosen from the longest context so that a CTA reads about one round of
// 8192 scores).  CTA rank r owns the r-th of C equal parts of the candidates
// [prefix, L).  Every CTA reads the sequence's coarse histogram (built by the
// scoring kernel, bins 16 scores wide) and finds the bin that holds the k-th
// largest score: the window [lo, lo + 16) and the number of candidates above
// it (an edge bin sends the sequence to an exact radix select over its
// scores, window one score wide).  Then:
//   1. every CTA counts, in its part, the candidates in each one-score-wide
//      fine bin of the window and those above it, and keeps the part's
//      candidates at or above the window (about 2% of the positions at 128K)
//      in position order in shared memory, with their cache slots;
//   2. the counts of all ranks are exchanged through distributed shared
//      memory; each CTA derives the exact threshold tau (the k-th largest
//      score), the number of ties at tau to keep (quota), and how many
//      selected positions and ties at tau lie in the parts before its own;
//   3. each CTA writes its selected positions, in order, at that offset (ties
//      at tau are kept while their rank over the whole sequence is below the
//      quota, so the lower positions win).
// A part with more than kSelCap kept candidates rescans its scores in step 3.
// Global loads that do not depend on one another (the first round of scores,
// their block ids, the histogram) are issued together, and the next round's
// scores are loaded while the current one is processed: on this GPU a
// dependent global access costs on the order of a microsecond.  No global
// atomics, no fences; the only hand-off between CTAs is the pushed count
// exchange before one cluster barrier.
// A round is 8192 positions: 512 threads x 16, or (where the launch has one
// CTA per SM anyway) 1024 threads x 8, which shortens each thread's serial part.
constexpr int kSelRound = 8192;                      // positions per round
constexpr int kSelThreads = 512;                     // threads of the packed launch
constexpr int kCounts = 1 + kFineBins;               // above, fine bins
constexpr int kSelCap = 4096;                        // kept candidates per CTA in shared memory
constexpr int kSelSmem = kSelCap * 3 * 4;
constexpr int kSelSmemSpread = 120 * 1024;  // over half an SM's shared memory: one CTA per SM

struct SelectParams {
  const int32_t* scores;
  const int32_t* ctx;
  const int32_t* bt;
  int* coarse;  // [B][kCoarseBins], zeroed again here after use
  int ld, prefix, k, max_ctx, max_blocks, num_blocks;
  int32_t* idx;
  int32_t* n_sel;
  int32_t* slot;  // cache slots of the selected positions, or nullptr
  int csplit;     // row b's context length is ctx[b / csplit] (per-KV-head rows: csplit = Hkv)
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Barrier over every thread of the cluster; orders shared-memory writes before
// it with reads after it, across the cluster's CTAs.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Cache slot (block * 64 + row) of position t of sequence b.
__device__ __forceinline__ int slot_of(const SelectParams& p, int b, int t) {
  return load_block(p.bt, b, p.max_blocks, t >> 6, p.num_blocks, &g_status) * kBlock + (t & 63);
}
// Writes v to CTA `rank`'s shared memory at the address of `p` in this CTA.
__device__ __forceinline__ void st_remote(int* p, uint32_t rank, int v) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Raw scores of positions t .. t + 15 (t a multiple of 16); chunks wholly outside
// [lo_t, hi_t) are not read.  mask_scores applies the range later, where the
// values are used, so that no instruction waits on the loads before that.
template <int PER>
__device__ __forceinline__ void load_raw(const int32_t* row, int ld, int t, int lo_t, int hi_t, int4* x) {
#pragma unroll
  for (int q = 0; q < PER / 4; ++q) {
    const int tq = t + 4 * q;
    x[q] = make_int4(INT_MIN, INT_MIN, INT_MIN, INT_MIN);
    if (tq < ld && tq + 4 > lo_t && tq < hi_t) x[q] = __ldg(reinterpret_cast<const int4*>(row + tq));
  }
}
template <int PER>
__device__ __forceinline__ void mask_scores(const int4* x, int t, int lo_t, int hi_t, int* v) {
#pragma unroll
  for (int q = 0; q < PER / 4; ++q) {
    const int tq = t + 4 * q;
    v[4 * q] = tq >= lo_t && tq < hi_t ? x[q].x : INT_MIN;
    v[4 * q + 1] = tq + 1 >= lo_t && tq + 1 < hi_t ? x[q].y : INT_MIN;
    v[4 * q + 2] = tq + 2 >= lo_t && tq + 2 < hi_t ? x[q].z : INT_MIN;
    v[4 * q + 3] = tq + 3 >= lo_t && tq + 3 < hi_t ? x[q].w : INT_MIN;
  }
}
// Scores of positions t .. t + 15 (t a multiple of 16) kept where lo_t <= t' < hi_t,
// INT_MIN elsewhere; never reads past the row's ld entries.
template <int PER>
__device__ __forceinline__ void load_scores(const int32_t* row, int ld, int t, int lo_t, int hi_t, int* v) {
#pragma unroll
  for (int q = 0; q < PER / 4; ++q) {
    const int tq = t + 4 * q;
    int4 x = make_int4(INT_MIN, INT_MIN, INT_MIN, INT_MIN);
    if (tq < ld && tq + 4 > lo_t && tq < hi_t) x = __ldg(reinterpret_cast<const int4*>(row + tq));
    v[4 * q] = tq >= lo_t && tq < hi_t ? x.x : INT_MIN;
    v[4 * q + 1] = tq + 1 >= lo_t && tq + 1 < hi_t ? x.y : INT_MIN;
    v[4 * q + 2] = tq + 2 >= lo_t && tq + 2 < hi_t ? x.z : INT_MIN;
    v[4 * q + 3] = tq + 3 >= lo_t && tq + 3 < hi_t ? x.w : INT_MIN;
  }
}

template <int C, int NTH>
__global__ void __launch_bounds__(NTH) decode_select_kernel(const SelectParams p) {
  constexpr int kSelThreads = NTH;               // threads of this launch
  constexpr int kSelPer = kSelRound / NTH;       // consecutive positions per thread per round
  extern __shared__ __align__(16) int s_ent[];     // [kSelCap] positions | scores | slots
  __shared__ int s_hist[kCoarseBins];
  __shared__ int s_counts[kCounts];                // this rank's: above, fine bins
  __shared__ int s_all[C][kCounts];                // every rank's
  __shared__ int s_misc[4];                        // tau, quota, ties before, output base
  __shared__ int s_scratch[264];
  int* e_pos = s_ent;
  int* e_sc = s_ent + kSelCap;
  int* e_slot = s_ent + 2 * kSelCap;
  const int tid = threadIdx.x, lane = tid & 31, b = blockIdx.y;
  const int r = C > 1 ? (int)cluster_rank() : 0;
  const int L = min(__ldg(p.ctx + (p.csplit > 1 ? b / p.csplit : b)), p.max_ctx);
  const int n_cand = max(0, L - p.prefix);
  const int tb = p.prefix + (int)((long long)n_cand * r / C);
  const int te = p.prefix + (int)((long long)n_cand * (r + 1) / C);
  int32_t* out = p.idx + (size_t)b * p.k;
  int32_t* out_slot = p.slot ? p.slot + (size_t)b * p.k : nullptr;
  const int a0 = tb & ~(kSelPer - 1);
  int t = a0 + tid * kSelPer;  // kSelPer positions inside one 64-position block
  const int bt0 = (out_slot && t < te) ? __ldg(p.bt + (size_t)b * p.max_blocks + (t >> 6)) : 0;
  // The context length and the block table are inputs no kernel of the step
  // writes: they are read before the wait on the scoring kernel.  This kernel
  // lets the next one start only after its own wait (the attention's first
  // pass relies on that).
  pdl_wait();
  pdl_trigger();

  if (n_cand <= p.k) {  // every candidate is selected: position t goes to entry t - prefix
    for (int t = tb + tid; t < te; t += kSelThreads) {
      out[t - p.prefix] = t;
      if (out_slot) out_slot[t - p.prefix] = slot_of(p, b, t);
    }
    if (r == 0) {
      for (int j = n_cand + tid; j < p.k; j += kSelThreads) out[j] = -1;
      if (tid == 0) p.n_sel[b] = n_cand;
    }
    return;  // the whole cluster takes this branch: no cluster barrier is pending
  }

  const int32_t* row = p.scores + (size_t)b * p.ld;
  int* gh = p.coarse + (size_t)b * kCoarseBins;
  // First round of scores and slots, then the histogram: all in flight together.
  constexpr int kHB = kCoarseBins / kSelThreads;  // histogram bins per thread
  int hreg[kHB];
#pragma unroll
  for (int i = 0; i < kHB; ++i) hreg[i] = __ldcg(gh + tid + i * kSelThreads);
  int v[kSelPer];
  int4 xr[kSelPer / 4];
  load_raw<kSelPer>(row, p.ld, t, tb, te, xr);
#pragma unroll
  for (int i = 0; i < kHB; ++i) s_hist[tid + i * kSelThreads] = hreg[i];
  if (tid < kCounts) s_counts[tid] = 0;
  __syncthreads();
  if (tid < 32) {  // one warp finds the threshold bin
    int bb, ab;
    warp_hist_threshold(s_hist, kCoarseBins, p.k, lane, &bb, &ab);
    if (lane == 0) s_misc[0] = bb;
  }
  __syncthreads();
  const int beta = s_misc[0];
  int slot0 = 0;  // slot of t; t + j is slot0 + j
  if (out_slot && t < te) {
    slot0 = bt0;
    if ((unsigned)slot0 >= (unsigned)p.num_blocks) {
      set_status(&g_status, kStBadBlock);
      slot0 = 0;
    }
    slot0 = slot0 * kBlock + (t & 63);
  }
  int lo, width;
  if (beta > 0 && beta < kCoarseBins - 1) {
    lo = (beta - kCoarseOff) << kCoarseShift;
    width = kFineBins;
  } else {  // the k-th largest lies outside the histogram's range: exact radix select
    int tau, n_gt;
    block_radix_select(row + p.prefix, n_cand, p.k, s_scratch, &tau, &n_gt);
    lo = tau;
    width = 1;
  }
  const int hi = lo + width;
  // 1. this part's candidates (s >= lo), in position order, into shared memory;
  //    counts per fine bin of the window and above it.
  mask_scores<kSelPer>(xr, t, tb, te, v);
  int n_keep = 0, my_above = 0;
  for (int t0 = a0; t0 < te; t0 += kSelRound) {
    int vn[kSelPer];  // next round, loaded while this one is processed
    const int tn = t + kSelRound;
    int slot_n = 0;
    if (t0 + kSelRound < te) {
      load_scores<kSelPer>(row, p.ld, tn, tb, te, vn);
      slot_n = (out_slot && tn < te) ? slot_of(p, b, tn) : 0;
    }
    uint32_t cmask = 0;
#pragma unroll
    for (int j = 0; j < kSelPer; ++j) cmask |= (uint32_t)(v[j] >= lo) << j;
    int tot;
    int o = block_exclusive_scan(__popc(cmask), s_scratch, &tot) + n_keep;
    n_keep += tot;
    if (__any_sync(0xffffffffu, cmask != 0)) {
#pragma unroll
      for (int j = 0; j < kSelPer; ++j)
        if ((cmask >> j) & 1) {
          if (v[j] >= hi) ++my_above;
          else atomicAdd(&s_counts[1 + v[j] - lo], 1);
          if (o < kSelCap) {
            e_pos[o] = t + j;
            e_sc[o] = v[j];
            e_slot[o] = slot0 + j;
          }
          ++o;
        }
    }
#pragma unroll
    for (int j = 0; j < kSelPer; ++j) v[j] = vn[j];
    t = tn;
    slot0 = slot_n;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) my_above += __shfl_xor_sync(0xffffffffu, my_above, o);
  if (lane == 0 && my_above) atomicAdd(&s_counts[0], my_above);
  __syncthreads();
  // 2. this rank's counts go to row r of every rank's table; after the cluster
  //    barrier each CTA reads only its own shared memory, so no CTA touches
  //    another's after it and none has to wait for the others before leaving.
  for (int e = tid; e < C * kCounts; e += kSelThreads) {
    const int rr = e / kCounts, f = e - rr * kCounts;
    if (C > 1) st_remote(&s_all[r][f], rr, s_counts[f]);
    else s_all[0][f] = s_counts[f];
  }
  if (C > 1) cluster_sync(); else __syncthreads();  // every rank's counts are in place
  if (r == 0)  // every rank has read the histogram: leave it zero for the next call
    for (int i = tid; i < kCoarseBins; i += kSelThreads) gh[i] = 0;
  if (tid < 32) {
    // Warp 0, lanes as fine bins: totals, suffix sums from the top of the window.
    int fine_f = 0;
#pragma unroll
    for (int rr = 0; rr < C; ++rr) fine_f += lane < width ? s_all[rr][1 + (lane & 15)] : 0;
    int above = lane < C ? s_all[lane][0] : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
    int suf = fine_f;  // candidates in fine bins lane .. width - 1
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += y;
    }
    // The k-th largest lies in fine bin f*, the highest bin whose suffix reaches
    // k - above; cum = candidates above it inside the window.
    const int kk = p.k - above;
    const uint32_t reach = __ballot_sync(0xffffffffu, lane < width && suf >= kk);
    const int fstar = reach ? 31 - __clz(reach) : 0;
    const int cum = __shfl_sync(0xffffffffu, suf, fstar + 1);  // fstar + 1 <= 16: suffix past the window is 0
    const int quota = kk - cum;
    // Lanes as ranks: candidates above tau and at tau in each part, then the
    // ties and the selected entries in the parts before this CTA's.
    int gt = 0, eq = 0;
    if (lane < C) {
      gt = s_all[lane][0];
#pragma unroll
      for (int f = 0; f < kFineBins; ++f) gt += (f > fstar && f < width) ? s_all[lane][1 + f] : 0;
      eq = s_all[lane][1 + fstar];
    }
    int eq_incl = eq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, eq_incl, o);
      if (lane >= o) eq_incl += y;
    }
    const int ties_before = eq_incl - eq;
    const int taken = gt + min(max(quota - ties_before, 0), eq);
    int tk_incl = taken;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, tk_incl, o);
      if (lane >= o) tk_incl += y;
    }
    if (lane == r) {
      s_misc[2] = ties_before;
      s_misc[3] = tk_incl - taken;
    }
    if (lane == 0) {
      s_misc[0] = lo + fstar;
      s_misc[1] = quota;
    }
  }
  __syncthreads();
  const int tau = s_misc[0], quota = s_misc[1];
  int carry_ties = s_misc[2], carry_out = s_misc[3];
  // 3. ordered write of this part's selection
  if (n_keep <= kSelCap) {
    // From the kept candidates: thread i takes entries [i * per, (i + 1) * per).
    // One scan of (above tau, at tau) pairs, 16 bits each (n_keep <= 4096):
    // ties in this CTA before the thread's entries, and of them those kept
    // (global tie rank below the quota), give its output offset.
    const int per = (n_keep + kSelThreads - 1) / kSelThreads;
    const int e0 = min(n_keep, tid * per), e1 = min(n_keep, e0 + per);
    int n_gt = 0, n_eq = 0;
    for (int e = e0; e < e1; ++e) {
      n_gt += e_sc[e] > tau;
      n_eq += e_sc[e] == tau;
    }
    int tot;
    const int ex = block_exclusive_scan((n_eq << 16) | n_gt, s_scratch, &tot);
    const int eq_before = ex >> 16, gt_before = ex & 0xffff;
    const int tot_eq = tot >> 16, tot_gt = tot & 0xffff;
    const int tie_room = max(quota - carry_ties, 0);  // ties this CTA may still keep
    int tr = carry_ties + eq_before;
    int o = carry_out + gt_before + min(eq_before, tie_room);
    carry_out += tot_gt + min(tot_eq, tie_room);
    for (int e = e0; e < e1; ++e) {
      const int sc = e_sc[e];
      const bool take = sc > tau || (sc == tau && tr++ < quota);
      if (take) {
        if (o < p.k) {
          out[o] = e_pos[e];
          if (out_slot) out_slot[o] = e_slot[e];
        }
        ++o;
      }
    }
  } else {
    // More candidates than the stage holds: rescan the scores of this part.
    for (int t0 = a0; t0 < te; t0 += kSelRound) {
      const int tt = t0 + tid * kSelPer;
      int w[kSelPer];
      load_scores<kSelPer>(row, p.ld, tt, tb, te, w);
      const int s0 = (out_slot && tt < te) ? slot_of(p, b, tt) : 0;
      uint32_t gt_m = 0, eq_m = 0;
#pragma unroll
      for (int j = 0; j < kSelPer; ++j) {
        gt_m |= (uint32_t)(w[j] > tau) << j;
        eq_m |= (uint32_t)(w[j] == tau) << j;
      }
      int tot;
      int tr = block_exclusive_scan(__popc(eq_m), s_scratch, &tot) + carry_ties;
      carry_ties += tot;
      uint32_t keep = gt_m;
#pragma unroll
      for (int j = 0; j < kSelPer; ++j)
        if ((eq_m >> j) & 1) {
          if (tr < quota) keep |= 1u << j;
          ++tr;
        }
      int o = block_exclusive_scan(__popc(keep), s_scratch, &tot) + carry_out;
      carry_out += tot;
#pragma unroll
      for (int j = 0; j < kSelPer; ++j)
        if ((keep >> j) & 1) {
          if (o < p.k) {
            out[o] = tt + j;
            if (out_slot) out_slot[o] = s0 + j;
          }
          ++o;
        }
    }
  }
  if (r == C - 1) {  // the last part ends the list: pad, count
    for (int j = carry_out + tid; j < p.k; j += kSelThreads) out[j] = -1;
    if (tid == 0) p.n_sel[b] = min(carry_out, p.k);
  }
}

// ---------------------------------------------------------------- prefill ---
// One CTA of 256 threads per query row, heaviest rows first: a 1024-bin coarse
// histogram of the row's scores in shared memory and the threshold window from
// it; the counts per one-score bin of the window and above it, which give the
// exact threshold tau and the tie quota; then an ordered compaction, each thread
// over its own contiguous run of the row after scans of its counts above and at
// tau.  The first pass reads the row from HBM with the whole CTA, and the later
// passes follow at once, while the row is still in L2: with one warp per row
// (about 7,300 rows in flight) the rows of a 16K chunk fell out of L2 between
// passes (16K chunk: 0.454 -> 0.383 ms).  An edge bin falls back to an exact
// block radix select.
constexpr int kRowThreads = 256;

struct RowTopkParams {
  const int32_t* scores;
  int ld, prefix, k, pos0, n_q;
  uint64_t* mask;  // or null: the dense pass's attended-position bitmap [block][nq_pad] (zeroed), rows < n_dense
  int n_dense, nq_pad;
  int32_t* idx;
  int32_t* n_sel;
};

// Candidate scores of one row, four per 16-byte chunk c (positions 4c .. 4c + 3),
// INT_MIN outside [t_lo, t_hi).
__device__ __forceinline__ int4 row_chunk(const int32_t* row, int c, int t_lo, int t_hi) {
  int4 x = __ldcg(reinterpret_cast<const int4*>(row) + c);
  const int t = 4 * c;
  x.x = t >= t_lo && t < t_hi ? x.x : INT_MIN;
  x.y = t + 1 >= t_lo && t + 1 < t_hi ? x.y : INT_MIN;
  x.z = t + 2 >= t_lo && t + 2 < t_hi ? x.z : INT_MIN;
  x.w = t + 3 >= t_lo && t + 3 < t_hi ? x.w : INT_MIN;
  return x;
}

__global__ void __launch_bounds__(kRowThreads) prefill_topk_kernel(const RowTopkParams p) {
  __shared__ int s_hist[kCoarseBins];
  __shared__ int s_cnt[1 + kFineBins];  // above the window, fine bins
  __shared__ int s_misc[4];
  __shared__ int s_scratch[272];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = p.n_q - 1 - (int)blockIdx.x;  // the longest rows first
  const int pos = p.pos0 + i;
  const int n_cand = max(0, pos - p.prefix + 1);
  int32_t* out = p.idx + (size_t)i * p.k;
  uint64_t* mrow = p.mask && i < p.n_dense ? p.mask + i : nullptr;  // word c of this row at mrow[c * nq_pad]
  if (n_cand <= p.k) {  // every candidate is selected
    for (int j = tid; j < p.k; j += kRowThreads) out[j] = j < n_cand ? p.prefix + j : -1;
    if (tid == 0) p.n_sel[i] = n_cand;
    if (mrow) {  // the prefix and every candidate: the whole causal range [0, pos]
      const int n = pos + 1;
      for (int c = tid; c < ((n + 63) >> 6); c += kRowThreads)
        mrow[(size_t)c * p.nq_pad] = (c + 1) * 64 <= n ? ~0ull : (1ull << (n & 63)) - 1ull;
    }
    return;
  }
  if (mrow) {  // the prefix [0, min(P, pos + 1)): whole words stored, the partial one OR-ed
    const int npre = min(p.prefix, pos + 1);
    for (int c = tid; c < (npre >> 6); c += kRowThreads) mrow[(size_t)c * p.nq_pad] = ~0ull;
    if (tid == 0 && (npre & 63))
      atomicOr(reinterpret_cast<unsigned long long*>(&mrow[(size_t)(npre >> 6) * p.nq_pad]), (1ull << (npre & 63)) - 1ull);
  }
  const int32_t* row = p.scores + (size_t)i * p.ld;
  const int t_lo = p.prefix, t_hi = pos + 1;
  const int c0 = t_lo >> 2, c1 = (t_hi + 3) >> 2;  // chunks covering [t_lo, t_hi), all inside the row's ld entries
  // Pass 1: coarse histogram.
  for (int b = tid; b < kCoarseBins; b += kRowThreads) s_hist[b] = 0;
  if (tid <= kFineBins) s_cnt[tid] = 0;
  __syncthreads();
#pragma unroll 4
  for (int c = c0 + tid; c < c1; c += kRowThreads) {
    const int4 x = row_chunk(row, c, t_lo, t_hi);
    if (x.x != INT_MIN) atomicAdd(&s_hist[coarse_bin(x.x)], 1);
    if (x.y != INT_MIN) atomicAdd(&s_hist[coarse_bin(x.y)], 1);
    if (x.z != INT_MIN) atomicAdd(&s_hist[coarse_bin(x.z)], 1);
    if (x.w != INT_MIN) atomicAdd(&s_hist[coarse_bin(x.w)], 1);
  }
  __syncthreads();
  if (warp == 0) {
    int beta, above_win;
    warp_hist_threshold(s_hist, kCoarseBins, p.k, lane, &beta, &above_win);
    if (lane == 0) s_misc[0] = beta;
  }
  __syncthreads();
  const int beta = s_misc[0];
  int lo, width;
  if (beta > 0 && beta < kCoarseBins - 1) {
    lo = (beta - kCoarseOff) << kCoarseShift;
    width = kFineBins;
  } else {  // the k-th largest lies outside the histogram's range: exact radix select
    int tau_r, n_gt_r;
    block_radix_select(row + t_lo, n_cand, p.k, s_scratch, &tau_r, &n_gt_r);
    lo = tau_r;
    width = 1;
  }
  // Pass 2: counts per one-score bin of the window and above it.
  int my_above = 0;
#pragma unroll 4
  for (int c = c0 + tid; c < c1; c += kRowThreads) {
    const int4 x = row_chunk(row, c, t_lo, t_hi);
    const int v4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v4[u];
      if (v >= lo + width) ++my_above;
      else if (v >= lo) atomicAdd(&s_cnt[1 + v - lo], 1);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) my_above += __shfl_xor_sync(0xffffffffu, my_above, o);
  if (lane == 0 && my_above) atomicAdd(&s_cnt[0], my_above);
  __syncthreads();
  // Lanes of warp 0 as fine bins: the k-th largest lies in bin f*, the highest
  // whose suffix reaches k - above; cum = candidates above it inside the window.
  if (warp == 0) {
    const int kk = p.k - s_cnt[0];
    int suf = lane < width ? s_cnt[1 + (lane & 15)] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += y;
    }
    const uint32_t reach = __ballot_sync(0xffffffffu, lane < width && suf >= kk);
    const int fstar = reach ? 31 - __clz(reach) : 0;
    const int cum = __shfl_sync(0xffffffffu, suf, fstar + 1);  // fstar + 1 <= 16: the suffix past the window is 0
    if (lane == 0) {
      s_misc[1] = lo + fstar;
      s_misc[2] = kk - cum;
    }
  }
  __syncthreads();
  const int tau = s_misc[1], quota = s_misc[2];
  // Pass 3: ordered compaction.  Thread t takes the chunks [a, e) of the row;
  // scans of its counts at and above tau give the ties and the selected
  // positions before it.
  const int per = (c1 - c0 + kRowThreads - 1) / kRowThreads;
  const int a = min(c1, c0 + tid * per), e = min(c1, a + per);
  int n_gt = 0, n_eq = 0;
  for (int c = a; c < e; ++c) {
    const int4 x = row_chunk(row, c, t_lo, t_hi);
    n_gt += (x.x > tau) + (x.y > tau) + (x.z > tau) + (x.w > tau);
    n_eq += (x.x == tau) + (x.y == tau) + (x.z == tau) + (x.w == tau);
  }
  int tot_eq, tot_gt;
  const int eq_before = block_exclusive_scan(n_eq, s_scratch, &tot_eq);
  const int gt_before = block_exclusive_scan(n_gt, s_scratch, &tot_gt);
  int tr = eq_before;
  int o = gt_before + min(eq_before, quota);
  int mword = -1;            // bitmap word being gathered (this thread's run spans few words)
  unsigned long long mbits = 0;
  for (int c = a; c < e; ++c) {
    const int4 x = row_chunk(row, c, t_lo, t_hi);
    const int v4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v4[u];
      if (v > tau || (v == tau && tr++ < quota)) {
        const int t = 4 * c + u;
        if (o < p.k) out[o] = t;
        ++o;
        if (mrow) {
          if ((t >> 6) != mword) {
            if (mbits) atomicOr(reinterpret_cast<unsigned long long*>(&mrow[(size_t)mword * p.nq_pad]), mbits);
            mword = t >> 6;
            mbits = 0;
          }
          mbits |= 1ull << (t & 63);
        }
      }
    }
  }
  if (mbits) atomicOr(reinterpret_cast<unsigned long long*>(&mrow[(size_t)mword * p.nq_pad]), mbits);
  const int n_out = min(tot_gt + min(tot_eq, quota), p.k);
  for (int j = n_out + tid; j < p.k; j += kRowThreads) out[j] = -1;
  if (tid == 0) p.n_sel[i] = n_out;
}

}  // namespace

// Per device: clusters of 16 selection CTAs can be scheduled at all, and how
// many clusters of 1, 2, 4, 8, 16 CTAs fit at once with one CTA per SM.
bool g_sel16[64] = {};
int g_spread_cap[64][5] = {};

constexpr int kSelThreadsSpread = 1024;  // threads of a launch with one CTA per SM

template <int C>
int spread_capacity() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, 1);
  cfg.blockDim = dim3(kSelThreadsSpread);
  cfg.dynamicSmemBytes = kSelSmemSpread;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_select_kernel<C, kSelThreadsSpread>, &cfg) != cudaSuccess) n = 0;
  return n;
}

cudaError_t setup_topk_kernels() {
  cudaError_t e = cudaSuccess;
  auto smem = [&](auto kernel) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelSmemSpread);
  };
  smem(decode_select_kernel<1, kSelThreads>);
  smem(decode_select_kernel<2, kSelThreads>);
  smem(decode_select_kernel<4, kSelThreads>);
  smem(decode_select_kernel<8, kSelThreads>);
  smem(decode_select_kernel<16, kSelThreads>);
  smem(decode_select_kernel<1, kSelThreadsSpread>);
  smem(decode_select_kernel<2, kSelThreadsSpread>);
  smem(decode_select_kernel<4, kSelThreadsSpread>);
  smem(decode_select_kernel<8, kSelThreadsSpread>);
  smem(decode_select_kernel<16, kSelThreadsSpread>);
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaSuccess;
  // Clusters of 16 are beyond the portable size: use them only where the
  // occupancy query says at least one fits.
  if (cudaFuncSetAttribute(decode_select_kernel<16, kSelThreads>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
          cudaSuccess &&
      cudaFuncSetAttribute(decode_select_kernel<16, kSelThreadsSpread>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                           1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1);
    cfg.blockDim = dim3(kSelThreads);
    cfg.dynamicSmemBytes = kSelSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    g_sel16[dev] =
        cudaOccupancyMaxActiveClusters(&n, decode_select_kernel<16, kSelThreads>, &cfg) == cudaSuccess && n > 0;
  }
  g_spread_cap[dev][0] = spread_capacity<1>();
  g_spread_cap[dev][1] = spread_capacity<2>();
  g_spread_cap[dev][2] = spread_capacity<4>();
  g_spread_cap[dev][3] = spread_capacity<8>();
  g_spread_cap[dev][4] = g_sel16[dev] ? spread_capacity<16>() : 0;
  cudaGetLastError();  // a refused query leaves no error behind
  return cudaSuccess;
}

// CTAs per sequence (about one round of scores each, at most 8, 16 where
// supported, at most c_cap) and whether every cluster fits with one CTA per SM.
static void select_shape(const KV& kv, int prefix, int c_cap, int* c_out, bool* spread) {
  int dev = 0;
  cudaGetDevice(&dev);
  const bool known = dev >= 0 && dev < 64;
  int c_max = (known && g_sel16[dev]) ? 16 : 8;
  if (c_cap < c_max) c_max = c_cap < 1 ? 1 : c_cap;
  const long long n_max = (long long)kv.max_ctx - prefix;
  int c = 1;
  while (c < c_max && n_max > (long long)c * kSelRound) c *= 2;
  const int ci = c == 1 ? 0 : c == 2 ? 1 : c == 4 ? 2 : c == 8 ? 3 : 4;
  *c_out = c;
  *spread = known && g_spread_cap[dev][ci] >= kv.batch;
}

bool decode_select_spread(const KV& kv, int prefix) {
  int c;
  bool spread;
  select_shape(kv, prefix, 16, &c, &spread);
  return spread;
}

int decode_select_ctas(const KV& kv, int prefix, int c_cap) {
  int c;
  bool spread;
  select_shape(kv, prefix, c_cap, &c, &spread);
  return c * kv.batch;
}

cudaError_t launch_decode_select(const KV& kv, const int32_t* scores, int ld, int prefix, int k,
                                 const SelState& sel, int32_t* idx, int32_t* n_sel, cudaStream_t st, int c_cap,
                                 int csplit) {
  SelectParams p;
  p.csplit = csplit > 1 ? csplit : 1;
  p.scores = scores;
  p.ctx = kv.context_lens;
  p.bt = kv.block_table;
  p.coarse = sel.coarse;
  p.ld = ld;
  p.prefix = prefix;
  p.k = k;
  p.max_ctx = kv.max_ctx;
  p.max_blocks = kv.max_blocks;
  p.num_blocks = kv.num_blocks;
  p.idx = idx;
  p.n_sel = n_sel;
  p.slot = sel.slot;
  // The selection is a chain of dependent steps: a CTA sharing its SM with
  // another runs it markedly slower (measured).  Where every cluster of the
  // launch fits with one CTA per SM, ask for enough shared memory to get that,
  // and give the CTA 1024 threads (8 positions each instead of 16).
  int c;
  bool spread;
  select_shape(kv, prefix, c_cap, &c, &spread);
  const dim3 grid(c, kv.batch);
  if (spread) {
    const dim3 block(kSelThreadsSpread);
    const int sm = kSelSmemSpread;
    switch (c) {
      case 1: return launch_pdl(decode_select_kernel<1, kSelThreadsSpread>, grid, block, sm, st, 1, p);
      case 2: return launch_pdl(decode_select_kernel<2, kSelThreadsSpread>, grid, block, sm, st, 2, p);
      case 4: return launch_pdl(decode_select_kernel<4, kSelThreadsSpread>, grid, block, sm, st, 4, p);
      case 8: return launch_pdl(decode_select_kernel<8, kSelThreadsSpread>, grid, block, sm, st, 8, p);
      default: return launch_pdl(decode_select_kernel<16, kSelThreadsSpread>, grid, block, sm, st, 16, p);
    }
  }
  const dim3 block(kSelThreads);
  switch (c) {
    case 1: return launch_pdl(decode_select_kernel<1, kSelThreads>, grid, block, kSelSmem, st, 1, p);
    case 2: return launch_pdl(decode_select_kernel<2, kSelThreads>, grid, block, kSelSmem, st, 2, p);
    case 4: return launch_pdl(decode_select_kernel<4, kSelThreads>, grid, block, kSelSmem, st, 4, p);
    case 8: return launch_pdl(decode_select_kernel<8, kSelThreads>, grid, block, kSelSmem, st, 8, p);
    default: return launch_pdl(decode_select_kernel<16, kSelThreads>, grid, block, kSelSmem, st, 16, p);
  }
}

cudaError_t launch_prefill_topk(const QS& qs, const int32_t* scores, int ld, int prefix, int k, int32_t* idx,
                                int32_t* n_sel, cudaStream_t st, uint64_t* mask, int n_dense, int nq_pad) {
  RowTopkParams p;
  p.mask = mask;
  p.n_dense = mask ? n_dense : 0;
  p.nq_pad = nq_pad;
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
