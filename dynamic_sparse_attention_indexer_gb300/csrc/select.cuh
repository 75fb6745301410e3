// Exact top-k threshold search over int32 indexer scores.
//
// The selection rule (§2.1 top-k, ties to the lower position) is decided by a
// threshold tau and a tie quota: every candidate with score > tau is taken,
// and of those with score == tau the `quota` lowest positions are taken.  The
// threshold is found from a 1-wide score histogram when it falls inside the
// histogram window, else by an exact 4-pass radix select over the scores.
#pragma once

#include "common.cuh"

namespace dsa {

// Highest bin b with sum(bins >= b) >= k among nb (256 or 1024) bins in shared
// memory, and the count above it; one warp.  *bin = -1 when the total is below k.
__device__ __forceinline__ void warp_hist_threshold(const int* h, int nb, int k, int lane, int* bin, int* above) {
  const int gs = nb / 32;  // bins per lane group (8 or 32)
  // Four independent sums over the group's bins, read in a lane-rotated order
  // (no bank conflicts).
  int s4[4] = {0, 0, 0, 0};
  for (int i = 0; i < gs; i += 4)
#pragma unroll
    for (int u = 0; u < 4; ++u) s4[u] += h[gs * lane + ((i + u + lane) & (gs - 1))];
  int suf = (s4[0] + s4[1]) + (s4[2] + s4[3]);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += y;
  }
  const uint32_t reach = __ballot_sync(0xffffffffu, suf >= k);
  if (!reach) {
    *bin = -1;
    *above = 0;
    return;
  }
  const int ls = 31 - __clz(reach);
  const int above_grp = ls < 31 ? __shfl_sync(0xffffffffu, suf, ls + 1) : 0;
  int suf2 = lane < gs ? h[gs * ls + lane] : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, suf2, o);
    if (lane + o < 32) suf2 += y;
  }
  const uint32_t reach2 = __ballot_sync(0xffffffffu, lane < gs && above_grp + suf2 >= k);
  const int b = 31 - __clz(reach2);
  *bin = gs * ls + b;
  *above = above_grp + (b < 31 ? __shfl_sync(0xffffffffu, suf2, b + 1) : 0);
}

// Selection of one query: mode kSelAll takes every candidate.
struct Sel {
  int mode, tau, n_gt, quota;
};

// Finds the histogram bin beta holding the k-th largest score: the count above
// beta is < k and the count from beta up is >= k.  All threads of the CTA call;
// blockDim.x must divide NB.  `ld` loads bin i.  Requires sum >= k.
// Returns beta (or -1 if the counts do not reach k) and the count above it.
template <int NB = kHistBins, class Load>
__device__ __forceinline__ void hist_threshold_bin(Load ld, int k, int* scratch, int* beta_out,
                                                   int* above_out) {
  const int per = NB / blockDim.x;
  const int base = threadIdx.x * per;
  int local = 0;
  for (int i = 0; i < per; ++i) local += ld(base + i);
  int total;
  const int below = block_exclusive_scan(local, scratch, &total);
  const int above_thread = total - below - local;  // bins owned by higher threads
  if (threadIdx.x == 0) scratch[40] = -1;
  __syncthreads();
  if (above_thread < k && above_thread + local >= k) {
    int acc = above_thread;
    for (int i = per - 1; i >= 0; --i) {
      const int h = ld(base + i);
      if (acc + h >= k) {
        scratch[40] = base + i;
        scratch[41] = acc;
        break;
      }
      acc += h;
    }
  }
  __syncthreads();
  *beta_out = scratch[40];
  *above_out = scratch[41];
  __syncthreads();
}

// Exact k-th largest of x[0..n) (1 <= k <= n): 4 passes of 8-bit radix digits
// over the order-preserving unsigned key u = s ^ 0x80000000.  Returns tau and
// the number of elements strictly greater than tau.  All threads call; sh holds
// >= 258 ints.  Slow path for scores outside the histogram window.
__device__ __forceinline__ void block_radix_select(const int* __restrict__ x, int n, int k, int* sh,
                                                   int* tau_out, int* n_gt_out) {
  uint32_t prefix = 0, mask = 0;
  int kk = k, above = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint32_t u = (uint32_t)__ldcg(x + i) ^ 0x80000000u;
      if ((u & mask) == prefix) atomicAdd(&sh[(u >> shift) & 255], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = 0, dsel = 0;
      for (int dg = 255; dg >= 0; --dg) {
        const int h = sh[dg];
        if (acc + h >= kk) {
          dsel = dg;
          break;
        }
        acc += h;
      }
      sh[256] = dsel;
      sh[257] = acc;
    }
    __syncthreads();
    const int dsel = sh[256], acc = sh[257];
    above += acc;
    kk -= acc;
    prefix |= (uint32_t)dsel << shift;
    mask |= 0xFFu << shift;
    __syncthreads();
  }
  *tau_out = (int)(prefix ^ 0x80000000u);
  *n_gt_out = above;
}

// Selection of one query from its complete histogram (or the radix fallback).
// x/n: the query's candidate scores, read only on the fallback.
template <class Load>
__device__ __forceinline__ Sel selection_from_hist(Load ld, const int* x, int n_cand, int k, int* scratch) {
  Sel s;
  if (n_cand <= k) {
    s.mode = kSelAll;
    s.tau = 0;
    s.n_gt = n_cand;
    s.quota = 0;
    return s;
  }
  int beta, above;
  hist_threshold_bin(ld, k, scratch, &beta, &above);
  s.mode = kSelThreshold;
  if (beta > 0 && beta < kHistBins - 1) {
    s.tau = beta - kHistOff;
    s.n_gt = above;
  } else {
    block_radix_select(x, n_cand, k, scratch, &s.tau, &s.n_gt);
  }
  s.quota = k - s.n_gt;
  return s;
}

}  // namespace dsa
