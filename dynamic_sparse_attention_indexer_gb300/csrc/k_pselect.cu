// Prefill index selection without materialising the scores: the indexer
// product and the top-k in one kernel.
//
// The article ("国产AI芯片完成前沿大模型Day-0适配:稀疏注意力与混合精度推理全解析")
// scores every query against every key on the tensor cores and reduces the
// scores to the top-k (§2.1), with the vision prefix never scored (§2.4) and,
// in prefill, selection fused with what follows (§2.3).  Written out, the score
// matrix of a 16K chunk is 442 MB, read back three times by a separate top-k.
// Here one CTA owns 128 query rows (four threads per row, 64 columns of a tile
// each) and walks its key tiles (256 positions) in ascending order several
// times, the product of the next tile in flight while one is visited, recomputing the exact scores on tcgen05 each
// time (the product is ~0.2 us of tensor time per tile; the 64-dim indexer
// makes recomputation far cheaper than a round trip through HBM), and runs a
// radix select on per-row histograms held in shared memory:
//   pass 1  a 256-bin histogram per row, bins 64 scores wide over
//           [-8192, 8191] (the indexer values of the pages' workloads, int8 in
//           [-8, 8], give |s| <= 4096), which fixes the bin holding the k-th
//           largest score and how many candidates lie above it;
//   pass 2  one-score bins inside that bin: the exact threshold and how many
//           candidates equal to it are taken (ties: the lower positions);
//   pass 3  the selected positions, written in ascending order as the tiles
//           are walked.
// If any row of the CTA has a candidate score outside [-8192, 8191] the CTA
// instead runs an exact radix select over the key s + 2^20 (|s| <= 2^20 for
// any int8 values, so the key lies in [0, 2^21]), 8, 8 and 6 bits per level
// (bits 21-14, 13-6, 5-0), before the same final pass.
// Rows with at most k candidates take all of them (no selection).
//
// Measured on GB300 at the 16K chunk: 1.19 ms, against 0.62 ms for the
// separate scoring (0.17 ms, its time the 442 MB of score writes) and top-k
// (0.45 ms): the per-score histogram work of three walks (about 30 instructions
// per score over the walks, at 0.4 issued per cycle) costs more than the HBM
// round trip it saves, and one CTA per 128 queries leaves the causal
// imbalance (the last CTA walks twice the average).  It is kept as the
// allocation-light form (no score matrix, no workspace).
//
// Scores are exact: int8 values converted to e4m3 (kind::f8f6f4) when every
// value of the tile lies in [-16, 16], to f16 (kind::f16) otherwise, fp32
// accumulation of integer products (exact below 2^24).  The query rows are
// kept in both formats for the whole kernel.
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dsa {
namespace {

__device__ int g_status;

constexpr int kRows = 128;      // query rows per CTA (M of the product, TMEM lanes)
constexpr int kKeys = 256;      // key positions per tile (N of the product)
constexpr int kThreads = 512;   // four threads per query row
constexpr int kBins = 256;
constexpr int kPitch = kBins + 1;  // histogram row pitch in words: same-bin reads across rows hit distinct banks
constexpr int kFastShift = 6;      // pass-1 bins 64 scores wide
constexpr int kFastLo = -8192;     // pass-1 window [-8192, 8191]
constexpr int kGenOff = 1 << 20;   // exact fallback: key s + 2^20 in [0, 2^21]

// Shared memory: histograms, then the operands (1024-byte aligned).
constexpr uint32_t kHistBytes = kRows * kPitch * 4;            // 131,584
constexpr uint32_t kOffA8 = (kHistBytes + 1023) & ~1023u;      // query rows, e4m3, 64-byte swizzle: 8 KB
constexpr uint32_t kOffA16 = kOffA8 + 8192;                    // query rows, f16, 128-byte swizzle: 16 KB
constexpr uint32_t kOffB = kOffA16 + 16384;                    // key rows, two buffers: 16 KB (e4m3) or 32 KB (f16) each
constexpr uint32_t kOffCnt = kOffB + 2 * 32768;                 // per-tile counts of the final walk: 4 KB
constexpr uint32_t kOffBar = kOffCnt + kRows * 4 * 8;
constexpr uint32_t kSmem = kOffBar + 32 + 1024;  // + two barriers, TMEM slot, alignment slack
static_assert(kSmem <= 227 * 1024, "shared memory budget");

struct PSelParams {
  const int8_t* idx_cache;
  const int32_t* bt;  // block-table row of the sequence
  const int8_t* q_idx;
  int32_t* idx;
  int32_t* n_sel;
  int num_blocks, prefix, pos0, n_q, k, n_tiles;
};

__device__ __forceinline__ int sx8(int w, int b) { return (int)(int8_t)((unsigned)w >> (8 * b)); }
__device__ __forceinline__ bool above16(const int4 (&v)[4]) {
  bool big = false;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int x = sx8(w[i], b);
        big |= x > 16 || x < -16;
      }
  }
  return big;
}

// Row r of an operand: 64 int8 values to e4m3 (64 bytes, 64-byte swizzle) or
// f16 (128 bytes, 128-byte swizzle), K-major.
__device__ __forceinline__ void put_e4m3(uint8_t* op, int r, const int4 (&v)[4]) {
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
__device__ __forceinline__ void put_f16(uint8_t* op, int r, const int4 (&v)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
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

// Walks a row's histogram from the highest bin down: the bin holding the
// need-th largest entry, and how many entries lie in the bins above it.
__device__ __forceinline__ void find_bin(const uint32_t* h, int nbins, int need, int* bin, int* above) {
  int acc = 0, b = nbins - 1;
  for (; b > 0; --b) {
    const int c = (int)h[b];
    if (acc + c >= need) break;
    acc += c;
  }
  *bin = b;
  *above = acc;
}

// One CTA per 128 query rows, heaviest (latest) rows first.  Four threads per
// row (warps w, w + 4, w + 8, w + 12 share TMEM lanes 32 (w % 4) ..): quarter q
// of a row handles columns 64q .. 64q + 63 of each 256-position tile.
__global__ void __launch_bounds__(kThreads, 1) prefill_select_kernel(const PSelParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a8 = base + kOffA8;
  uint8_t* a16 = base + kOffA16;
  uint8_t* sb = base + kOffB;
  int2* qcnt = reinterpret_cast<int2*>(base + kOffCnt);  // [row][quarter]: (above, equal) of a tile
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + kOffBar);  // [buffer]: its product is done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp >> 2, r = ((warp & 3) << 5) | lane;  // this thread's row and column quarter
  const int i0 = (p.n_tiles - 1 - (int)blockIdx.x) * kRows;
  const int i = i0 + r;
  const bool row_ok = i < p.n_q;
  const int pos = p.pos0 + i;
  const int n_c = row_ok ? max(0, pos + 1 - p.prefix) : 0;  // candidates [prefix, pos]
  const bool all = n_c <= p.k;                                // every candidate is taken
  const bool sel = row_ok && !all;
  uint32_t* hist = reinterpret_cast<uint32_t*>(base) + r * kPitch;
  const int i_last = min(p.n_q, i0 + kRows) - 1;
  const int t_max = p.pos0 + i_last;  // largest position any row of the CTA sees
  pdl_wait();
  pdl_trigger();

  if (!__syncthreads_or(sel)) {
    // No row needs a selection: the candidates themselves, a row at a time per
    // warp (coalesced).
    for (int rr = warp; rr < kRows; rr += kThreads / 32) {
      const int ir = i0 + rr;
      if (ir >= p.n_q) break;
      const int nr = max(0, p.pos0 + ir + 1 - p.prefix);
      int32_t* out = p.idx + (size_t)ir * p.k;
      for (int j = lane; j < p.k; j += 32) out[j] = j < nr ? p.prefix + j : -1;
      if (lane == 0) p.n_sel[ir] = nr;
    }
    return;
  }

  // The query rows (operand row m = query i0 + m), kept in both formats.
  bool bq = false;
  if (tid < kRows) {
    int4 qv[4];
    const int iq = i0 + tid;
    const int4* src = reinterpret_cast<const int4*>(p.q_idx + (size_t)min(iq, p.n_q - 1) * kIdxDim);
#pragma unroll
    for (int c = 0; c < 4; ++c) qv[c] = iq < p.n_q ? __ldg(src + c) : make_int4(0, 0, 0, 0);
    bq = above16(qv);
    put_e4m3(a8, tid, qv);
    put_f16(a16, tid, qv);
  }
  const bool big_q = __syncthreads_or(bq) != 0;
  if (warp == 0) tmem_alloc(tslot, 2 * kKeys);
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_fence_init();
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t col_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 64 * quarter;
  const int tb = p.prefix / kKeys, te = t_max / kKeys;  // key tiles holding candidates
  uint32_t n_issued = 0, n_done = 0;  // products issued / waited for, over all walks: product n uses buffer n & 1
  bool ok = true;

  // Key row `tid` of tile `tile` (threads 0 .. 255; zero past the CTA's last position).
  auto load_key = [&](int tile, int4 (&kv)[4]) {
    const int t = tile * kKeys + tid;
    const bool in = tid < kKeys && tile <= te && t <= t_max;
    const int blk = in ? load_block(p.bt, 0, 0, t >> 6, p.num_blocks, &g_status) : 0;
    const int4* ks = reinterpret_cast<const int4*>(p.idx_cache + ((size_t)blk * kBlock + (t & 63)) * kIdxDim);
#pragma unroll
    for (int c = 0; c < 4; ++c) kv[c] = in ? __ldg(ks + c) : make_int4(0, 0, 0, 0);
  };
  // Converts the key rows in registers into operand buffer n & 1 and issues
  // product n (tile scores into accumulator n & 1).  Every thread calls it.
  auto issue = [&](const int4 (&kv)[4]) {
    uint8_t* b = sb + (n_issued & 1u) * 32768u;
    const bool f16 = __syncthreads_or(big_q || (tid < kKeys && above16(kv))) != 0;
    if (tid < kKeys) {
      if (f16) put_f16(b, tid, kv);
      else put_e4m3(b, tid, kv);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      constexpr uint32_t idesc = mma_idesc(kRows, kKeys, 0);
      const uint32_t d = tmem + (n_issued & 1u) * kKeys;
      if (!f16) {
#pragma unroll
        for (int k = 0; k < 2; ++k)
          mma_f8(d, smem_desc(smem_u32(a8) + 32 * k, 512, kSwizzle64), smem_desc(smem_u32(b) + 32 * k, 512, kSwizzle64),
                 idesc, k > 0);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16(d, smem_desc(smem_u32(a16) + 32 * k, 1024, kSwizzle128),
                  smem_desc(smem_u32(b) + 32 * k, 1024, kSwizzle128), idesc, k > 0);
      }
      mma_commit(&bar[n_issued & 1u]);
    }
    ++n_issued;
  };
  // One walk over the key tiles in ascending order, software-pipelined: the
  // product of tile + 1 runs on the tensor core while the threads visit tile's
  // scores, on_tile(t0, jlo, jhi, s[64]) with this thread's 64 scores (columns
  // 64 quarter + e) and its row's candidate columns [jlo, jhi].  on_tile is
  // called by every thread (it may synchronise the CTA).
  auto walk = [&](auto&& on_tile) {
    int4 kv[4];
    load_key(tb, kv);
    issue(kv);
    load_key(tb + 1, kv);
    for (int tile = tb; tile <= te; ++tile) {
      const int t0 = tile * kKeys;
      if (tile + 1 <= te) {  // operand buffer and accumulator of product n + 1 were last used by tile - 1: done
        issue(kv);
        load_key(tile + 2, kv);
      }
      const uint32_t buf = n_done & 1u;
      if (!mbar_wait(&bar[buf], (n_done >> 1) & 1u)) ok = false;
      ++n_done;
      tc_fence_after();
      uint32_t sv[64];
      {
        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
        tmem_ld32_nowait(col_addr + buf * kKeys, lo);
        tmem_ld32_nowait(col_addr + buf * kKeys + 32, hi);
        tmem_wait_ld();
      }
      const int jlo = row_ok ? max(p.prefix - t0, 0) : 1, jhi = row_ok ? min(pos - t0, kKeys - 1) : 0;
      on_tile(t0, jlo, jhi, sv);
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  };
  // A histogram walk: visit(s) for every candidate score of this thread's columns.
  auto hist_walk = [&](auto&& visit) {
    walk([&](int, int jlo, int jhi, const uint32_t (&sv)[64]) {
      const int j0 = 64 * quarter;
      if (jlo <= j0 && jhi >= j0 + 63) {  // every column a candidate (all but the diagonal and prefix tiles)
#pragma unroll
        for (int e = 0; e < 64; ++e) visit(__float2int_rn(__uint_as_float(sv[e])));
      } else if (jlo <= j0 + 63 && jhi >= j0) {
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (j0 + e >= jlo && j0 + e <= jhi) visit(__float2int_rn(__uint_as_float(sv[e])));
      }
    });
  };
  // (histogram updates are shared-memory atomics with the result unused: one
  // instruction each, and the row's four threads share the row's histogram)
  auto clear = [&] {  // after a barrier: every thread has read the histograms
    __syncthreads();
    if (quarter == 0)
      for (int b = 0; b <= kBins; ++b) hist[b] = 0u;
  };

  int need = p.k;  // entries still to take at or below the current bin
  int thr = 0;     // the k-th largest score of the row
  clear();
  bool wide = false;
  hist_walk([&](int s) {
    const unsigned u = (unsigned)(s - kFastLo);
    wide |= u >= (unsigned)(kBins << kFastShift);
    atomicAdd(&hist[min(u >> kFastShift, (unsigned)kBins)], 1u);  // past the window: the pad word
  });
  if (!__syncthreads_or(sel && wide)) {
    int b0 = 0, above = 0;
    if (sel) find_bin(hist, kBins, need, &b0, &above);
    need -= above;
    const int lo = kFastLo + (b0 << kFastShift);
    clear();
    hist_walk([&](int s) {
      const unsigned d = (unsigned)(s - lo);
      atomicAdd(&hist[min(d, (unsigned)kBins)], 1u);  // outside the bin: the pad word (never read)
    });
    int b1 = 0;
    above = 0;
    if (sel) find_bin(hist, 1 << kFastShift, need, &b1, &above);
    need -= above;
    thr = lo + b1;
  } else {
    // exact radix select over the key s + 2^20 in [0, 2^21]: bits 21-14, 13-6, 5-0
    int a = 0, b = 0, c = 0, above = 0;
    clear();
    hist_walk([&](int s) { atomicAdd(&hist[(unsigned)(s + kGenOff) >> 14], 1u); });
    if (sel) find_bin(hist, kBins, need, &a, &above);
    need -= above;
    clear();
    hist_walk([&](int s) {
      const unsigned u = (unsigned)(s + kGenOff);
      if ((int)(u >> 14) == a) atomicAdd(&hist[(u >> 6) & 255u], 1u);
    });
    above = 0;
    if (sel) find_bin(hist, kBins, need, &b, &above);
    need -= above;
    clear();
    hist_walk([&](int s) {
      const unsigned u = (unsigned)(s + kGenOff);
      if ((int)(u >> 6) == ((a << 8) | b)) atomicAdd(&hist[u & 63u], 1u);
    });
    above = 0;
    if (sel) find_bin(hist, 64, need, &c, &above);
    need -= above;
    thr = ((a << 14) | (b << 6) | c) - kGenOff;
  }
  // Final walk: the selected positions in ascending order.  Per tile each
  // quarter counts its candidates above and at the threshold; from the four
  // counts every quarter derives its output offset and how many of its
  // threshold-equal candidates it takes (ties: the lowest positions of the
  // row, `need` of them in all).
  int row_cnt = 0, eq_seen = 0;
  int32_t* out = p.idx + (size_t)(row_ok ? i : 0) * p.k;
  walk([&](int t0, int jlo, int jhi, const uint32_t (&sv)[64]) {
    int gt = 0, eq = 0;
#pragma unroll
    for (int e = 0; e < 64; ++e) {
      const int j = 64 * quarter + e;
      const int s = __float2int_rn(__uint_as_float(sv[e]));
      if (j >= jlo && j <= jhi) {
        gt += (all || s > thr) ? 1 : 0;
        eq += (!all && s == thr) ? 1 : 0;
      }
    }
    qcnt[r * 4 + quarter] = make_int2(gt, eq);
    __syncthreads();
    int off = row_cnt, eqb = eq_seen, my_off = 0, my_eq = 0;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const int2 cq = qcnt[r * 4 + qq];
      const int te_q = min(max(need - eqb, 0), cq.y);
      if (qq == quarter) {
        my_off = off;
        my_eq = te_q;
      }
      off += cq.x + te_q;
      eqb += cq.y;
    }
    row_cnt = off;
    eq_seen = eqb;
    int taken_eq = 0;
#pragma unroll
    for (int e = 0; e < 64; ++e) {
      const int j = 64 * quarter + e;
      const int s = __float2int_rn(__uint_as_float(sv[e]));
      if (j >= jlo && j <= jhi) {
        bool take = all || s > thr;
        if (!take && s == thr) take = taken_eq++ < my_eq;
        if (take) out[my_off++] = t0 + j;
      }
    }
  });
  if (row_ok) {
    for (int j = row_cnt + quarter; j < p.k; j += 4) out[j] = -1;
    if (quarter == 0) p.n_sel[i] = row_cnt;
  }
  if (!ok && tid == 0) set_status(&g_status, kStTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 2 * kKeys);
}

}  // namespace

cudaError_t setup_pselect_kernels() {
  return cudaFuncSetAttribute(prefill_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
}

cudaError_t launch_prefill_select(const KV& kv, const QS& qs, const int8_t* q_idx, int prefix, int k, int32_t* idx,
                                  int32_t* n_sel, cudaStream_t st) {
  PSelParams p;
  p.idx_cache = kv.idx_cache;
  p.bt = kv.block_table + (size_t)qs.seq * kv.max_blocks;
  p.q_idx = q_idx;
  p.idx = idx;
  p.n_sel = n_sel;
  p.num_blocks = kv.num_blocks;
  p.prefix = prefix;
  p.pos0 = qs.pos0;
  p.n_q = qs.n_q;
  p.k = k;
  p.n_tiles = (qs.n_q + kRows - 1) / kRows;
  return launch_pdl(prefill_select_kernel, dim3(p.n_tiles), dim3(kThreads), kSmem, st, 1, p);
}

cudaError_t read_clear_status_pselect(int* code, cudaStream_t st) {
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
