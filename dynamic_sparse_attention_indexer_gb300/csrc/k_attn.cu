// Steps 3 + 4 of DSA (§2.2 gather, §2.3 attention): GQA attention of each query
// token over its attended rows, read straight from the paged KV cache.
//
// Work is cut into 64-row tiles of (query, KV head) pairs; a pair's tiles cover
// the causal prefix rows then the selected rows.  A persistent grid (two CTAs per
// SM) takes one contiguous range of the (pair, tile) sequence per CTA, so every
// CTA streams about the same number of bytes and the copy pipeline runs on
// across pair boundaries (§2.3 decode: load only the active KV, asynchronously).
//
// All four warps of a CTA gather: each tile's 256-byte K and V rows arrive by
// 16-byte cp.async in an XOR-swizzled three-stage shared-memory ring, two tiles
// ahead of the math (§2.3 prefetch), and the row addresses of a tile are fetched
// one tile earlier still, so their latency hides behind the math too.  Each warp
// then computes its 16 rows of the tile on the tensor cores (mma.sync m16n8k16
// bf16, fp32 accumulate) in transposed form, S^T = K Q^T and O^T = V^T P^T, so
// the attended rows fill the 16-row M side and the G query heads the 8-wide N
// side (no padded heads); P^T reaches its operand layout through movmatrix.  The
// online softmax runs per head column in base 2, reduced across the row groups
// with warp shuffles, and O is rescaled only when a running max moved.  When a pair's
// segment ends the four warps merge their (max, sum, O) states through shared
// memory; a pair wholly inside the CTA is written out directly, a pair cut by a
// range boundary leaves one partial per CTA in the workspace, and the CTA that
// completes the pair's tile count (a ticket, no spinning) merges those.
#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

__device__ int g_status;

constexpr int kWarps = kAttnWarps;
constexpr int kAttnThreads = kWarps * 32;
constexpr int kTileRows = 64;                      // 16 rows per warp
constexpr int kStages = 3;
constexpr int kRowBytes = kHeadDim * 2;            // 256 B per K or V row
constexpr int kTileBytes = kTileRows * kRowBytes;  // 16 KB
constexpr int kQBytes = 16 * kRowBytes;            // G <= 16 query rows
constexpr int kStageBytes = 2 * kTileBytes;        // K and V tiles
constexpr int kQSlots = 2;                         // Q of the current and the next segment
constexpr int kMergeFloats = 16 * kHeadDim;        // one warp's O (G <= 16 heads)
// ring | Q slots | merge O | merge (m, l) | flag
constexpr int kSmemBytes = kStages * kStageBytes + kQSlots * kQBytes + 4 * kMergeFloats + 4 * 16 * 2 + 16;
constexpr int kRowsPerThread = kTileRows * 16 / kAttnThreads;  // 8 rows (one 16-B chunk each) per tile

struct AttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  const int32_t* bt;
  const int32_t* ctx;
  const int32_t* idx;
  const int32_t* nsel;
  const int32_t* rowbase;  // cache row (KV head 0) of every selected position, [n_q][k]
  int mode, seq, pos0;
  int max_blocks, num_blocks, hkv, hq, group, k, prefix, max_ctx;
  float scale_log2;
  int tiles;        // pairs * tiles_per_pair (< 2^31, checked on the host)
  int tiles_per_pair;
  float* part_o;    // [grid][2 slots][G][128]
  float2* part_ml;  // [grid][2 slots][G]
  int* pair_cnt;
  void* out;
  int out_dtype;
  float* lse;
};

// 256-byte rows of 16 chunks; chunk c of row r lives at chunk c ^ (r & 7).
__device__ __forceinline__ int swz(int row, int chunk) { return row * kRowBytes + ((chunk ^ (row & 7)) << 4); }

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

__device__ __forceinline__ int range_begin(int T, int G, int c) { return (int)((long long)T * c / G); }
__device__ __forceinline__ int cta_of(int T, int G, int x) { return (int)(((long long)(x + 1) * G - 1) / T); }

struct PairInfo {
  int qi, g, seq, n_pre, rows;
};
__device__ __forceinline__ PairInfo pair_info(const AttnParams& p, int pair) {
  PairInfo pi;
  pi.qi = pair / p.hkv;
  pi.g = pair - pi.qi * p.hkv;
  pi.seq = p.mode == 0 ? pi.qi : p.seq;
  const int pos = p.mode == 0 ? min(__ldg(p.ctx + pi.qi), p.max_ctx) - 1 : p.pos0 + pi.qi;
  pi.n_pre = max(0, min(p.prefix, pos + 1));
  pi.rows = pi.n_pre + min(max(__ldg(p.nsel + pi.qi), 0), p.k);
  return pi;
}

enum : int { kFirst = 1, kLast = 2, kFinal = 4, kWhole = 8 };

// The tiles a CTA handles, in order, without the empty ones (a segment's last
// tile is always kept so that the segment closes).
struct Cursor {
  int ti, t_begin, t_end, pair, seg_start;
  PairInfo pi;
  bool fresh;
};
struct Tile {
  int pair;
  PairInfo pi;
  int r0, nvalid, flags, seg_tiles, slot;
};

__device__ __forceinline__ bool next_tile(Cursor& c, const AttnParams& p, Tile* t) {
  const int TP = p.tiles_per_pair;
  while (c.ti < c.t_end) {
    const int ti = c.ti++;
    const int pair = ti / TP;
    const int tt = ti - pair * TP;
    if (pair != c.pair) {
      c.pair = pair;
      c.pi = pair_info(p, pair);
      c.seg_start = ti;
      c.fresh = true;
    }
    const int nvalid = min(max(c.pi.rows - tt * kTileRows, 0), kTileRows);
    const bool last = ti == c.t_end - 1 || tt == TP - 1;
    if (nvalid == 0 && !last) continue;
    t->pair = pair;
    t->pi = c.pi;
    t->r0 = tt * kTileRows;
    t->nvalid = nvalid;
    t->flags = (c.fresh ? kFirst : 0) | (last ? kLast : 0) | (ti == c.t_end - 1 ? kFinal : 0) |
               (last && c.seg_start == pair * TP && tt == TP - 1 ? kWhole : 0);
    t->seg_tiles = ti - c.seg_start + 1;
    t->slot = c.seg_start == c.t_begin ? 0 : 1;
    c.fresh = false;
    return true;
  }
  return false;
}

// Cache rows are fetched one tile ahead of their use: fetch_raw only issues the
// load (the block id of a prefix row, the pre-resolved row of a selected one),
// resolve turns it into the cache row of KV head g when the copy is issued.
__device__ __forceinline__ int fetch_raw(const AttnParams& p, const PairInfo& pi, int r) {
  return r < pi.n_pre ? __ldg(p.bt + (size_t)pi.seq * p.max_blocks + (r >> 6))
                      : __ldg(p.rowbase + (size_t)pi.qi * p.k + (r - pi.n_pre));
}
__device__ __forceinline__ int resolve(const AttnParams& p, const PairInfo& pi, int r, int raw) {
  if (r >= pi.n_pre) return raw + pi.g * kBlock;
  if ((unsigned)raw >= (unsigned)p.num_blocks) {
    set_status(&g_status, kStBadBlock);
    raw = 0;
  }
  return (raw * p.hkv + pi.g) * kBlock + (r & 63);
}

__device__ __forceinline__ void write_out(const AttnParams& p, size_t head, int d, float v) {
  if (p.out_dtype == 0)
    reinterpret_cast<__nv_bfloat16*>(p.out)[head * kHeadDim + d] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(p.out)[head * kHeadDim + d] = v;
}

// Merge the n partials of one pair (slots slot_of(0 .. n-1)) into the output.
// s_w holds 2048 floats, s_ml 32.  All threads of the CTA call.
template <class SlotOf>
__device__ void combine(const AttnParams& p, size_t head0, int n, SlotOf slot_of, float* s_w, float* s_ml) {
  const int tid = threadIdx.x, G = p.group;
  float2* s_pml = reinterpret_cast<float2*>(s_w);  // (max, sum) of partial i, head h at i * G + h
  const bool staged = n * G <= 1024;
  if (staged) {
    for (int e = tid; e < n * G; e += blockDim.x) s_pml[e] = __ldcg(&p.part_ml[(size_t)slot_of(e / G) * G + e % G]);
    __syncthreads();
  }
  auto ml_of = [&](int i, int h) {
    return staged ? s_pml[i * G + h] : __ldcg(&p.part_ml[(size_t)slot_of(i) * G + h]);
  };
  if (tid < G) {  // per head: the largest max and the total weight
    float M = -INFINITY;
    for (int i = 0; i < n; ++i) M = fmaxf(M, ml_of(i, tid).x);
    const float Ms = M == -INFINITY ? 0.f : M;
    float L = 0.f;
    for (int i = 0; i < n; ++i) {
      const float2 ml = ml_of(i, tid);
      L += exp2f(ml.x - Ms) * ml.y;
    }
    s_ml[2 * tid] = Ms;
    s_ml[2 * tid + 1] = L;
  }
  __syncthreads();
  const int d = tid;  // one output column per thread, all heads at once
  float acc[16];
#pragma unroll
  for (int h = 0; h < 16; ++h) acc[h] = 0.f;
  for (int i = 0; i < n; ++i) {
    const size_t base = (size_t)slot_of(i) * G * kHeadDim + d;
#pragma unroll
    for (int h = 0; h < 16; ++h)
      if (h < G) acc[h] += exp2f(ml_of(i, h).x - s_ml[2 * h]) * __ldcg(p.part_o + base + (size_t)h * kHeadDim);
  }
#pragma unroll
  for (int h = 0; h < 16; ++h)
    if (h < G) {
      write_out(p, head0 + h, d, acc[h] / s_ml[2 * h + 1]);
      if (d == 0 && p.lse) p.lse[head0 + h] = (s_ml[2 * h] + log2f(s_ml[2 * h + 1])) * 0.69314718055994531f;
    }
  __syncthreads();
}

__device__ __forceinline__ uint32_t transpose8x8(uint32_t v) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(v));
  return d;
}

// NT: 8-head column tiles (1 for G <= 8, 2 for G <= 16).
template <int NT>
__global__ void __launch_bounds__(kAttnThreads, 2) sparse_attn_kernel(const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* s_q = smem + kStages * kStageBytes;                                  // [kQSlots][16 rows]
  float* s_mo = reinterpret_cast<float*>(s_q + kQSlots * kQBytes);              // merge O [16 heads][128]
  float* s_mml = s_mo + kMergeFloats;                                           // merge (m, l) [16][2]
  volatile int* s_flag = reinterpret_cast<volatile int*>(s_mml + 32);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = p.tiles;
  const int TP = p.tiles_per_pair, G = p.group;
  Cursor ic, cc;  // issue cursor (runs ahead) and compute cursor
  ic.t_begin = cc.t_begin = range_begin(T, gridDim.x, blockIdx.x);
  ic.t_end = cc.t_end = range_begin(T, gridDim.x, blockIdx.x + 1);
  if (ic.t_begin >= ic.t_end) return;
  ic.ti = cc.ti = ic.t_begin;
  ic.pair = cc.pair = -1;
  ic.seg_start = cc.seg_start = ic.t_begin;
  ic.fresh = cc.fresh = false;

  // Masked rows and unused head rows must read as finite numbers: clear once.
  for (int i = tid; i < (kStages * kStageBytes + kQSlots * kQBytes) / 16; i += kAttnThreads)
    reinterpret_cast<int4*>(smem)[i] = make_int4(0, 0, 0, 0);
  __syncthreads();

  // This thread copies chunk `ch` of rows row0 + 8 i of every tile.
  const int ch = tid & 15, row0 = tid >> 4;
  int addr[kRowsPerThread];  // raw row loads of the next tile to issue
  Tile nt;                   // that tile
  bool have_next = next_tile(ic, p, &nt);
  auto fetch_addrs = [&](const Tile& t) {
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int rr = row0 + 8 * i;
      addr[i] = rr < t.nvalid ? fetch_raw(p, t.pi, t.r0 + rr) : 0;
    }
  };
  if (have_next) fetch_addrs(nt);
  int n_issued = 0, q_issue = 0;
  auto issue = [&]() {  // copy tile `nt` into the next stage, then fetch the following tile's rows
    if (have_next) {
      uint8_t* st = smem + (n_issued % kStages) * kStageBytes;
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int rr = row0 + 8 * i;
        if (rr < nt.nvalid) {
          const size_t off = (size_t)resolve(p, nt.pi, nt.r0 + rr, addr[i]) * kHeadDim + ch * 8;
          cp_async16(st + swz(rr, ch), p.kc + off, 16u);
          cp_async16(st + kTileBytes + swz(rr, ch), p.vc + off, 16u);
        }
      }
      if (nt.flags & kFirst) {
        const __nv_bfloat16* qsrc = p.q + ((size_t)nt.pi.qi * p.hq + (size_t)nt.pi.g * G) * kHeadDim;
        uint8_t* qdst = s_q + (q_issue & 1) * kQBytes;
        for (int c = tid; c < G * 16; c += kAttnThreads) cp_async16(qdst + swz(c >> 4, c & 15), qsrc + c * 8, 16u);
        ++q_issue;
      }
      ++n_issued;
      have_next = next_tile(ic, p, &nt);
      if (have_next) fetch_addrs(nt);
    }
    cp_async_commit();
  };
  for (int s = 0; s < kStages - 1; ++s) issue();

  // Fragment coordinates: S^T rows (attended rows) r = lane / 4 (+ 8); head
  // columns 2 (lane % 4) (+ 1) of each 8-head tile; O^T rows d = 16 i + lane / 4 (+ 8).
  const int mi = lane >> 3, rr8 = lane & 7, wrow = warp * 16;
  const int hc = 2 * (lane & 3);  // first head column of this lane in a tile
  uint32_t qb[NT][8][2];
  float o[8][NT][4];
  float m[NT][2], l[NT][2];
  Tile t;
  int q_use = 0;
  for (int n = 0; next_tile(cc, p, &t); ++n) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    if (t.flags & kFirst) {
      // Q into registers before the issue below may refill this Q slot.
      const uint8_t* sq = s_q + (q_use & 1) * kQBytes;
      ++q_use;
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int ks = 0; ks < 8; ks += 2)
          ldsm_x4(smem_u32(sq + swz(j * 8 + rr8, 2 * ks + mi)), qb[j][ks][0], qb[j][ks][1], qb[j][ks + 1][0],
                  qb[j][ks + 1][1]);
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j) o[i][j][0] = o[i][j][1] = o[i][j][2] = o[i][j][3] = 0.f;
#pragma unroll
      for (int j = 0; j < NT; ++j) m[j][0] = m[j][1] = -INFINITY, l[j][0] = l[j][1] = 0.f;
      __syncthreads();
    }
    issue();  // the stage consumed last iteration is free for the tile two ahead
    const uint8_t* sk = smem + (n % kStages) * kStageBytes;
    const uint8_t* sv = sk + kTileBytes;
    if (t.nvalid > wrow) {
      // S^T = K Q^T: this warp's 16 rows x 8 NT heads.
      float sacc[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(smem_u32(sk + swz(wrow + (mi & 1) * 8 + rr8, 2 * ks + (mi >> 1))), a0, a1, a2, a3);
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_bf16_16816(sacc[j], a0, a1, a2, a3, qb[j][ks][0], qb[j][ks][1]);
      }
      // Online softmax per head column (base 2), reduced over the 8 row groups.
      const int ra = wrow + (lane >> 2);  // tile rows of elements 0,1 (ra) and 2,3 (ra + 8)
      const bool va = ra < t.nvalid, vb = ra + 8 < t.nvalid;
      float alpha[NT][2], ms[NT][2];
      bool moved = false;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        sacc[j][0] = va ? sacc[j][0] * p.scale_log2 : -INFINITY;
        sacc[j][1] = va ? sacc[j][1] * p.scale_log2 : -INFINITY;
        sacc[j][2] = vb ? sacc[j][2] * p.scale_log2 : -INFINITY;
        sacc[j][3] = vb ? sacc[j][3] * p.scale_log2 : -INFINITY;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float mx = fmaxf(sacc[j][e], sacc[j][e + 2]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m[j][e], mx);
          ms[j][e] = mn == -INFINITY ? 0.f : mn;
          alpha[j][e] = exp2f(m[j][e] - ms[j][e]);
          moved |= mn != m[j][e];
          m[j][e] = mn;
        }
      }
      if (__any_sync(0xffffffffu, moved)) {  // rescale only when a running max moved
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            o[i][j][0] *= alpha[j][0];
            o[i][j][1] *= alpha[j][1];
            o[i][j][2] *= alpha[j][0];
            o[i][j][3] *= alpha[j][1];
          }
#pragma unroll
        for (int j = 0; j < NT; ++j) l[j][0] *= alpha[j][0], l[j][1] *= alpha[j][1];
      }
      uint32_t pb[NT][2];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const float p0 = exp2f(sacc[j][0] - ms[j][0]), p1 = exp2f(sacc[j][1] - ms[j][1]);
        const float p2 = exp2f(sacc[j][2] - ms[j][0]), p3 = exp2f(sacc[j][3] - ms[j][1]);
        l[j][0] += p0 + p2;
        l[j][1] += p1 + p3;
        // P^T rows (attended rows) x head columns -> B fragments (rows as K).
        pb[j][0] = transpose8x8(pack_bf16x2(p0, p1));
        pb[j][1] = transpose8x8(pack_bf16x2(p2, p3));
      }
      // O^T += V^T P^T: d in 8 tiles of 16.
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(smem_u32(sv + swz(wrow + (mi >> 1) * 8 + rr8, 2 * i + (mi & 1))), a0, a1, a2, a3);
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_bf16_16816(o[i][j], a0, a1, a2, a3, pb[j][0], pb[j][1]);
      }
    }

    if (t.flags & kLast) {
      // ---- the pair's segment ends: merge the warps' states into warp 0
      // (pairs of warps through shared memory: 1 -> 0, 3 -> 2, 2 -> 0).
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = l[j][e];
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 16);
          l[j][e] = v;
        }
#pragma unroll
      for (int step = 0; step < 3; ++step) {
        const int from = step == 0 ? 1 : (step == 1 ? 3 : 2), dst = step == 1 ? 2 : 0;
        if (warp == from) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            if (lane < 4) {
              s_mml[2 * (j * 8 + hc)] = m[j][0];
              s_mml[2 * (j * 8 + hc) + 1] = l[j][0];
              s_mml[2 * (j * 8 + hc + 1)] = m[j][1];
              s_mml[2 * (j * 8 + hc + 1) + 1] = l[j][1];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int d = 16 * i + (lane >> 2);
              s_mo[(j * 8 + hc) * kHeadDim + d] = o[i][j][0];
              s_mo[(j * 8 + hc + 1) * kHeadDim + d] = o[i][j][1];
              s_mo[(j * 8 + hc) * kHeadDim + d + 8] = o[i][j][2];
              s_mo[(j * 8 + hc + 1) * kHeadDim + d + 8] = o[i][j][3];
            }
          }
        }
        __syncthreads();
        if (warp == dst) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            float a[2], b[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float om = s_mml[2 * (j * 8 + hc + e)], ol = s_mml[2 * (j * 8 + hc + e) + 1];
              const float M = fmaxf(m[j][e], om);
              const float S = M == -INFINITY ? 0.f : M;
              a[e] = exp2f(m[j][e] - S);
              b[e] = exp2f(om - S);
              m[j][e] = M;
              l[j][e] = l[j][e] * a[e] + ol * b[e];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int d = 16 * i + (lane >> 2);
              o[i][j][0] = o[i][j][0] * a[0] + s_mo[(j * 8 + hc) * kHeadDim + d] * b[0];
              o[i][j][1] = o[i][j][1] * a[1] + s_mo[(j * 8 + hc + 1) * kHeadDim + d] * b[1];
              o[i][j][2] = o[i][j][2] * a[0] + s_mo[(j * 8 + hc) * kHeadDim + d + 8] * b[0];
              o[i][j][3] = o[i][j][3] * a[1] + s_mo[(j * 8 + hc + 1) * kHeadDim + d + 8] * b[1];
            }
          }
        }
        __syncthreads();
      }
      const size_t head0 = (size_t)t.pi.qi * p.hq + (size_t)t.pi.g * G;
      if (t.flags & kWhole) {
        if (warp == 0) {
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int h = j * 8 + hc + e;
              if (h >= G) continue;
              const float r = 1.f / l[j][e];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int d = 16 * i + (lane >> 2);
                write_out(p, head0 + h, d, o[i][j][e] * r);
                write_out(p, head0 + h, d + 8, o[i][j][e + 2] * r);
              }
              if (lane < 4 && p.lse) p.lse[head0 + h] = (m[j][e] + log2f(l[j][e])) * 0.69314718055994531f;
            }
        }
      } else {
        if (warp == 0) {
          const size_t sl = (size_t)blockIdx.x * 2 + t.slot;
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int h = j * 8 + hc + e;
              if (h >= G) continue;
              if (lane < 4) p.part_ml[sl * G + h] = make_float2(m[j][e], l[j][e]);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int d = 16 * i + (lane >> 2);
                p.part_o[(sl * G + h) * kHeadDim + d] = o[i][j][e];
                p.part_o[(sl * G + h) * kHeadDim + d + 8] = o[i][j][e + 2];
              }
            }
          __threadfence();
        }
        __syncthreads();
        if (tid == 0) *s_flag = atomicAdd(p.pair_cnt + t.pair, t.seg_tiles) + t.seg_tiles == TP;
        __syncthreads();
        if (*s_flag) {
          // Every segment of the pair has landed: merge them in CTA order.
          __threadfence();
          const int first = t.pair * TP;
          const int c_lo = cta_of(T, gridDim.x, first), c_hi = cta_of(T, gridDim.x, first + TP - 1);
          const int nG = gridDim.x;
          combine(
              p, head0, c_hi - c_lo + 1,
              [&](int i) {
                const int c = c_lo + i;
                return c * 2 + (range_begin(T, nG, c) >= first ? 0 : 1);
              },
              s_mo, s_mml);
          if (tid == 0) p.pair_cnt[t.pair] = 0;
        }
        __syncthreads();  // merge buffers and the flag are free again
      }
    }
  }
  cp_async_wait<0>();
}

int g_attn_grid[64] = {};

// Selected positions -> cache rows (KV head 0), validated against the pool.
__global__ void resolve_rows_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ nsel,
                                    const int32_t* __restrict__ bt, const int32_t* __restrict__ ctx, int mode,
                                    int seq0, int n_q, int k, int max_blocks, int num_blocks, int hkv,
                                    int32_t* __restrict__ rowbase) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)n_q * k) return;
  const int qi = (int)(e / k), j = (int)(e - (long long)qi * k);
  if (j >= min(max(__ldg(nsel + qi), 0), k)) return;
  const int seq = mode == 0 ? qi : seq0;
  const int t = __ldg(idx + e);
  int blk = 0;
  if (t >= 0 && t < max_blocks * kBlock)
    blk = load_block(bt, seq, max_blocks, t >> 6, num_blocks, &g_status);
  else
    set_status(&g_status, kStBadBlock);
  rowbase[e] = blk * hkv * kBlock + (t & 63);
  (void)ctx;
}

}  // namespace

cudaError_t setup_attn_kernels() {
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(sparse_attn_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sparse_attn_kernel<2>, kAttnThreads, kSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) {
    const int g = sms * (per_sm > 0 ? per_sm : 1);
    g_attn_grid[dev] = g < kMaxAttnCtas ? g : kMaxAttnCtas;
  }
  return e;
}

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t st) {
  AttnParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kc = static_cast<const __nv_bfloat16*>(a.kv.k_cache);
  p.vc = static_cast<const __nv_bfloat16*>(a.kv.v_cache);
  p.bt = a.kv.block_table;
  p.ctx = a.kv.context_lens;
  p.idx = a.idx;
  p.nsel = a.n_sel;
  p.rowbase = a.rowbase ? a.rowbase : a.ws.rowbase;
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
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.tiles_per_pair = (a.prefix + a.k + kTileRows - 1) / kTileRows;
  p.tiles = (int)((long long)a.qs.n_q * a.kv.hkv * p.tiles_per_pair);
  p.part_o = a.ws.part_o;
  p.part_ml = a.ws.part_ml;
  p.pair_cnt = a.ws.pair_cnt;
  p.out = a.out;
  p.out_dtype = a.out_dtype;
  p.lse = a.lse;
  int dev = 0;
  cudaGetDevice(&dev);
  int grid = (dev >= 0 && dev < 64 && g_attn_grid[dev] > 0) ? g_attn_grid[dev] : 296;
  if (grid > p.tiles) grid = p.tiles;
  if (!a.rowbase) {  // stand-alone call: resolve the selected positions first
    const long long n = (long long)a.qs.n_q * a.k;
    resolve_rows_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
        a.idx, a.n_sel, a.kv.block_table, a.kv.context_lens, a.qs.mode, a.qs.seq, a.qs.n_q, a.k, a.kv.max_blocks,
        a.kv.num_blocks, a.kv.hkv, a.ws.rowbase);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.group <= 8)
    sparse_attn_kernel<1><<<grid, kAttnThreads, kSmemBytes, st>>>(p);
  else
    sparse_attn_kernel<2><<<grid, kAttnThreads, kSmemBytes, st>>>(p);
  return cudaGetLastError();
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
