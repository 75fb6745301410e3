// Prefill attention as a masked dense pass on the fifth-generation tensor cores.
//
// The article ("国产AI芯片完成前沿大模型Day-0适配:稀疏注意力与混合精度推理全解析", §2.3)
// fuses selection, gather and attention in prefill.  On GB300 the rows a query
// attends in a prefill chunk are a large share of its causal range (at a 16K
// chunk with k = 2048 and a 576-position prefix, 2624 of ~8200 positions on
// average), and gathering them row by row moves each cached row through L2 once
// per query (62 GB for the chunk).  This pass instead reads every cached
// position once per tile of 2 x 128 (query, head) rows and runs
//   S = Q K^T  and  O += P V
// on tcgen05.mma (bf16 operands, fp32 accumulators in tensor memory) over all
// of the tile's causal positions, with P = 0 wherever the position is not in
// the query's attended set.  The result is the same softmax over the same set:
// masked positions contribute exactly zero weight.
//
// Attended set of a query at position pos: the prefix [0, min(P, pos + 1))
// and its selected positions (§2.1, §2.4).  dense_mask_kernel writes it as a
// bitmap, word [c][i] holding positions 64c .. 64c + 63 of dense query i.
//
// dense_attn_kernel, one CTA per (KV head, two tiles of QT = floor(128 / G)
// queries), heaviest (latest) tiles first, 352 threads:
//   warp 8       K producer: TMA loads of the two Q tiles (once), then per
//                chunk of 64 positions the K block of the KV head (two 8 KB
//                boxes, 128-byte swizzle) with the tiles' mask words into a
//                4-stage ring, released as soon as S is computed;
//   warp 10      V producer: the chunk's V block into a 3-stage ring, released
//                after P V.  Separate issuers keep the K loads several chunks
//                ahead of their use;
//   warp 9       one thread issues the MMAs: S_t(j) = Q_t K(j)^T (A and B from
//                shared memory) and O_t += P_t(j) V(j) with P in tensor memory
//                as two bf16 terms, hi and the residual lo (V an MN-major
//                operand in shared memory), each group committed to an mbarrier;
//   warps 0-7    softmax, one thread per (query, head) row (TMEM lane), warps
//                0-3 tile 0 and 4-7 tile 1: masked online softmax in base 2 with a
//                lazy rescale of O (only when the running max grows by more than
//                2^8), P = hi + lo (about 16 significant bits, as in the gathered
//                path: a single bf16 P costs 2^-9 |v| per dominant weight, more
//                than the attention's tolerance when few keys carry the softmax)
//                stored into tensor memory, and at the end O / l and the
//                log-sum-exp.
// Tensor memory, per tile t at column 256 t: S (64 fp32 columns), P_hi and P_lo
// (32 columns each, two bf16 per column), O (128 fp32 columns).  Keeping P in
// tensor memory keeps shared-memory traffic to the K, V and Q operand reads:
// with P stored to and read back from shared memory, that traffic (about 320 KB
// per 64 positions of a tile pair) held the tensor pipe to a third of its rate.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dsa {
namespace {

__device__ int g_status;

constexpr int kKStages = 4;
constexpr int kVStages = 3;
constexpr int kThreads = 352;
constexpr uint32_t kQHalf = 16384;   // 128 rows x 128 bytes: one 64-wide half of the head dim
constexpr uint32_t kKVHalf = 8192;   // 64 positions x 128 bytes
constexpr uint32_t kKVStage = 2 * kKVHalf;
constexpr uint32_t kMaskStage = 2048;  // up to 2 x 128 mask words
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = 4 * kQHalf;
constexpr uint32_t kOffV = kOffK + kKStages * kKVStage;
constexpr uint32_t kOffMask = kOffV + kVStages * kKVStage;
constexpr uint32_t kOffBar = kOffMask + kKStages * kMaskStage;
constexpr uint32_t kNumBars = 1 + 3 * kKStages + 2 * kVStages + 2 + 2 + 2 + 2 + 2;
constexpr uint32_t kSmem = kOffBar + kNumBars * 8 + 16 + 1024;  // + TMEM address slot + alignment slack
// tensor-memory columns of tile t: base + 256 t + ...
constexpr uint32_t kColS = 0, kColPHi = 64, kColPLo = 96, kColO = 128;
static_assert(kSmem <= 227 * 1024, "shared memory budget");
constexpr float kRescaleLog2 = 8.f;  // O is rescaled only when the max grows by more than this (base-2 units)

struct DenseParams {
  const int32_t* bt;      // block-table row of the sequence
  const uint64_t* mask;   // [chunks][nq_pad] attended-position bitmap of the dense queries
  void* out;
  float* lse;
  int num_blocks, n_dense, nq_pad, pos0, hq, hkv, group, qt, n_super, out_dtype;
  float scale_log2;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 lanes in one 64-bit register, and the packed fp32x2 arithmetic of
// sm_100-class GPUs (one instruction for both lanes).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Waits for phase `parity` of `bar` for at most ~2 s, the thread suspended in
// the hardware between checks (try_wait with a suspend-time hint of 100 us: it
// returns as soon as the phase completes).  A polling wait here took issue
// slots from the thread that issues the MMAs on the same SM sub-partition and
// halved the tensor-core rate.
__device__ __forceinline__ bool mbar_sleep_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(100000u)
        : "memory");
    if (ok) return true;
    if (global_ns() - t0 > 2000000000ull) return false;
  }
}

// The same with every lane of the warp; the result is warp-uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_sleep_wait(bar, parity));
}

__global__ void __launch_bounds__(kThreads, 1)
    dense_attn_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const DenseParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;  // K block and mask words of a chunk landed
  uint64_t* k_empty = k_full + kKStages;
  uint64_t* m_free = k_empty + kKStages;  // mask words read, one arrival per softmax warp
  uint64_t* v_full = m_free + kKStages;
  uint64_t* v_empty = v_full + kVStages;
  uint64_t* s_full = v_empty + kVStages;  // [tile]
  uint64_t* s_free = s_full + 2;          // [tile], one arrival per softmax warp
  uint64_t* p_full = s_free + 2;          // [tile], one arrival per softmax warp
  uint64_t* p_free = p_full + 2;          // [tile]
  uint64_t* drain = p_free + 2;
  uint64_t* tail = drain + 1;             // V rows past the tiles' last position zeroed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(tail + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x % p.hkv;
  const int q0 = (p.n_super - 1 - blockIdx.x / p.hkv) * 2 * p.qt;  // heaviest tiles first
  const int q_last = min(q0 + 2 * p.qt, p.n_dense) - 1;
  const int nc = (p.pos0 + q_last) / kBlock + 1;  // chunks of 64 positions the tiles see
  const int last_rows = p.pos0 + q_last - (nc - 1) * kBlock + 1;  // positions of the last chunk in range
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&m_free[s], 8);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], 4);
      mbar_init(&p_full[t], 4);
      mbar_init(&p_free[t], 1);
    }
    mbar_init(drain, 1);
    mbar_init(tail, 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  pdl_wait();  // the bitmap comes from the previous kernel
  pdl_trigger();

  if (warp == 8) {
    // ---------------------------------------------------------- K producer
    const int rows = p.group * p.qt;
    const int mwords = min(2 * p.qt, p.nq_pad - q0);  // even: q0 and nq_pad are even
    if (lane == 0) {
      tma_prefetch_map(&qmap);
      tma_prefetch_map(&kmap);
      tma_prefetch_map(&vmap);
      mbar_arrive_expect_tx(q_full, 4u * (uint32_t)rows * 128u);
      for (int t = 0; t < 2; ++t)
        for (int x = 0; x < 2; ++x)
          tma_load_4d(base + kOffQ + (t * 2 + x) * kQHalf, &qmap, 0, x, g * p.group, q0 + t * p.qt, q_full);
    }
    int blk_next = 0;
    int k_issued = 0;
    for (int j = 0; j < nc; ++j) {
      if ((j & 31) == 0) blk_next = j + lane < nc ? load_block(p.bt, 0, 0, j + lane, p.num_blocks, &g_status) : 0;
      const int blk = __shfl_sync(0xffffffffu, blk_next, j & 31);
      const int sk = j % kKStages;
      if (j >= kKStages && !(warp_wait(&k_empty[sk], ((j / kKStages) + 1) & 1) &&
                             warp_wait(&m_free[sk], ((j / kKStages) + 1) & 1)))
        break;
      if (lane == 0) {
        uint8_t* st = base + kOffK + sk * kKVStage;
        mbar_arrive_expect_tx(&k_full[sk], kKVStage + (uint32_t)mwords * 8u);
        for (int x = 0; x < 2; ++x) tma_load_4d(st + x * kKVHalf, &kmap, 0, x, g, blk * kBlock, &k_full[sk]);
        bulk_g2s(base + kOffMask + sk * kMaskStage, p.mask + (size_t)j * p.nq_pad + q0, (uint32_t)mwords * 8u,
                 &k_full[sk]);
      }
      k_issued = j + 1;
    }
    if (k_issued < nc && lane == 0) set_status(&g_status, kStTimeout);
    // every copy this warp started has landed before the CTA ends
    bool landed = true;
    for (int j = max(k_issued - kKStages, 0); j < k_issued; ++j)
      if (!warp_wait(&k_full[j % kKStages], (j / kKStages) & 1)) landed = false;
    if (!landed && lane == 0) set_status(&g_status, kStTimeout);
  } else if (warp == 10) {
    // ---------------------------------------------------------- V producer
    int blk_next = 0;
    int v_issued = 0;
    for (int j = 0; j < nc; ++j) {
      if ((j & 31) == 0) blk_next = j + lane < nc ? load_block(p.bt, 0, 0, j + lane, p.num_blocks, &g_status) : 0;
      const int blk = __shfl_sync(0xffffffffu, blk_next, j & 31);
      const int sv = j % kVStages;
      if (j >= kVStages && !warp_wait(&v_empty[sv], ((j / kVStages) + 1) & 1)) break;
      if (lane == 0) {
        uint8_t* st = base + kOffV + sv * kKVStage;
        mbar_arrive_expect_tx(&v_full[sv], kKVStage);
        for (int x = 0; x < 2; ++x) tma_load_4d(st + x * kKVHalf, &vmap, 0, x, g, blk * kBlock, &v_full[sv]);
      }
      v_issued = j + 1;
    }
    if (v_issued < nc && lane == 0) set_status(&g_status, kStTimeout);
    bool landed = true;
    for (int j = max(v_issued - kVStages, 0); j < v_issued; ++j)
      if (!warp_wait(&v_full[j % kVStages], (j / kVStages) & 1)) landed = false;
    if (!landed && lane == 0) set_status(&g_status, kStTimeout);
    // Positions of the last block past the tiles' last position may hold anything
    // (unwritten slots); P is zero there, and their V rows are zeroed so that no
    // non-finite value meets a zero weight in the product.
    if (landed && v_issued == nc && last_rows < kBlock) {
      uint8_t* vt = base + kOffV + ((nc - 1) % kVStages) * kKVStage;
      const int n16 = (kBlock - last_rows) * 8;  // 16-byte pieces per half
      for (int e = lane; e < 2 * n16; e += 32)
        *reinterpret_cast<uint4*>(vt + (e / n16) * kKVHalf + last_rows * 128 + (e % n16) * 16) =
            make_uint4(0, 0, 0, 0);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(tail);
    }
  } else if (warp == 9) {
    // -------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc_s = mma_idesc(128, 64, kFmtBF16);
      constexpr uint32_t idesc_o = mma_idesc(128, 128, kFmtBF16, 0, 1);
      bool ok = mbar_sleep_wait(q_full, 0);
      tc_fence_after();
      // descriptors computed once; a byte offset o added to the start address adds o >> 4
      const uint64_t dq = smem_desc(smem_u32(base + kOffQ), 1024, kSwizzle128);
      const uint64_t dk = smem_desc(smem_u32(base + kOffK), 1024, kSwizzle128);
      const uint64_t dv = smem_desc_mn(smem_u32(base + kOffV), kKVHalf, 1024);
      for (int j = 0; ok && j <= nc; ++j) {
        if (j < nc) {  // S_t(j) = Q_t K(j)^T, once softmax_t has read S_t(j - 1)
          const int s = j % kKStages;
          ok = mbar_sleep_wait(&k_full[s], (j / kKStages) & 1);
          tc_fence_after();
          const uint64_t kb = dk + (uint64_t)(s * (kKVStage >> 4));
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!(ok = ok && mbar_sleep_wait(&s_free[t], (j & 1) ^ 1))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16(tmem + t * 256 + kColS, dq + (uint64_t)((t * 2 * kQHalf + (kk >> 2) * kQHalf + (kk & 3) * 32) >> 4),
                      kb + (uint64_t)(((kk >> 2) * kKVHalf + (kk & 3) * 32) >> 4), idesc_s, kk > 0);
            mma_commit(&s_full[t]);
          }
          mma_commit(&k_empty[s]);
        }
        if (j > 0 && ok) {  // O_t += (P_hi + P_lo)_t(j - 1) V(j - 1)
          const int jp = j - 1, s = jp % kVStages;
          ok = mbar_sleep_wait(&v_full[s], (jp / kVStages) & 1);
          if (ok && jp == nc - 1 && last_rows < kBlock) ok = mbar_sleep_wait(tail, 0);
          tc_fence_after();
          const uint64_t vb = dv + (uint64_t)(s * (kKVStage >> 4));
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!(ok = ok && mbar_sleep_wait(&p_full[t], jp & 1))) break;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16_ts(tmem + t * 256 + kColO, tmem + t * 256 + (h ? kColPLo : kColPHi) + kk * 8,
                           vb + (uint64_t)((kk * 2048) >> 4), idesc_o, jp > 0 || h > 0 || kk > 0);
            mma_commit(&p_free[t]);
          }
          mma_commit(&v_empty[s]);
        }
      }
      if (!ok) set_status(&g_status, kStTimeout);
      mma_commit(drain);  // every MMA issued above is complete before the CTA ends
      if (!mbar_sleep_wait(drain, 0)) set_status(&g_status, kStTimeout);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ---------------------------------------------------------------- softmax
    const int t = warp >> 2;
    const int r = ((warp & 3) << 5) | lane;  // row = TMEM lane
    const int qi = r / p.group;
    const int qd = q0 + t * p.qt + qi;  // dense query index
    const bool valid = qi < p.qt && qd < p.n_dense;
    const int mword = t * p.qt + qi;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    const bool pos_scale = p.scale_log2 > 0.f;
    for (int j = 0; j < nc; ++j) {
      const int s = j % kKStages;
      if (!(ok = warp_wait(&s_full[t], j & 1))) break;
      tc_fence_after();
      uint32_t sv[64];
      {
        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
        tmem_ld32(lane_addr + t * 256 + kColS, lo);
        tmem_ld32(lane_addr + t * 256 + kColS + 32, hi);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[t]);
      // the chunk's mask words came with its K block (phase j / kKStages of k_full[s]); the producer
      // refills the stage only after every softmax warp has read them (m_free)
      if (!(ok = warp_wait(&k_full[s], (j / kKStages) & 1))) break;
      uint64_t w = 0;
      if (valid) w = reinterpret_cast<const uint64_t*>(base + kOffMask + s * kMaskStage)[mword];
      __syncwarp();
      if (lane == 0) mbar_arrive(&m_free[s]);
      const uint32_t wlo = (uint32_t)w, whi = (uint32_t)(w >> 32);
      // x = the raw score where the position is attended, -inf elsewhere; with a
      // positive scale the scaled max is the scale times the raw max
      float x[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const uint32_t bit = i < 32 ? (wlo >> i) & 1u : (whi >> (i - 32)) & 1u;
        x[i] = bit ? __uint_as_float(sv[i]) : -INFINITY;
      }
      float mx;
      if (pos_scale) {
        float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; i += 8) {
          a0 = max3(a0, x[i], x[i + 1]);
          a1 = max3(a1, x[i + 2], x[i + 3]);
          a2 = max3(a2, x[i + 4], x[i + 5]);
          a3 = max3(a3, x[i + 6], x[i + 7]);
        }
        mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * p.scale_log2;
      } else {  // scale <= 0: scale first (a masked -inf stays -inf)
        mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          x[i] = x[i] == -INFINITY ? -INFINITY : x[i] * p.scale_log2;
          mx = fmaxf(mx, x[i]);
        }
      }
      float factor = 1.f;
      bool rescale = false;
      if (mx > m + kRescaleLog2) {  // also the first finite max (m = -inf)
        if (m != -INFINITY) {
          factor = ex2(m - mx);
          l *= factor;
          rescale = true;
        }
        m = mx;
      }
      const float m_use = m == -INFINITY ? 0.f : m;
      // p = 2^(scale x - m) two at a time; P = hi + lo with hi the truncated top
      // 16 bits of p (exact bf16) and lo = p - hi rounded to bf16 (~16 bits in all)
      const uint64_t c2 = pos_scale ? f2_pack(p.scale_log2, p.scale_log2) : f2_pack(1.f, 1.f);
      const uint64_t nm2 = f2_pack(-m_use, -m_use);
      uint64_t sum2 = f2_pack(0.f, 0.f);
      uint32_t pk[32], pl[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float a, c;
        f2_unpack(f2_fma(f2_pack(x[2 * i], x[2 * i + 1]), c2, nm2), a, c);
        a = ex2(a);
        c = ex2(c);
        const uint64_t pp = f2_pack(a, c);
        sum2 = f2_add(sum2, pp);
        const uint32_t ab = __float_as_uint(a), cb = __float_as_uint(c);
        pk[i] = __byte_perm(ab, cb, 0x7632);
        float la, lc;
        f2_unpack(f2_sub(pp, f2_pack(__uint_as_float(ab & 0xffff0000u), __uint_as_float(cb & 0xffff0000u))), la, lc);
        pl[i] = pack_bf16x2(la, lc);
      }
      {
        float s0, s1;
        f2_unpack(sum2, s0, s1);
        l += s0 + s1;
      }
      // P(j) overwrites P(j - 1) and O may be rescaled only once O += P(j - 1) V(j - 1) is done
      if (j > 0 && !(ok = warp_wait(&p_free[t], (j - 1) & 1))) break;
      tc_fence_after();
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_addr + t * 256 + kColO + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          tmem_st32(lane_addr + t * 256 + kColO + c * 32, o);
        }
      }
      tmem_st32(lane_addr + t * 256 + kColPHi, pk);
      tmem_st32(lane_addr + t * 256 + kColPLo, pl);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    // ---- epilogue: O / l, log-sum-exp
    if (ok && (ok = warp_wait(&p_free[t], (nc - 1) & 1))) {
      tc_fence_after();
      const int head = g * p.group + (r - qi * p.group);
      const size_t row = (size_t)qd * p.hq + head;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + t * 256 + kColO + c * 32, o);
        if (!valid) continue;
        if (p.out_dtype == DSA_OUT_F32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + row * kHeadDim + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                 __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + row * kHeadDim + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * e]) * inv, __uint_as_float(o[8 * e + 1]) * inv),
                                pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv),
                                pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv),
                                pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv));
        }
      }
      if (valid && p.lse) p.lse[row] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
    if (!ok && lane == 0) set_status(&g_status, kStTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// One warp per dense query: the prefix words and the selected positions into
// the zeroed [chunk][nq_pad] bitmap.  Runs of selected positions in the same
// word are OR-ed within the warp first, so each word takes one atomic per run.
__global__ void __launch_bounds__(256) dense_mask_kernel(const int32_t* __restrict__ idx,
                                                          const int32_t* __restrict__ n_sel, int k, int prefix,
                                                          int pos0, int n_dense, int nq_pad, uint64_t* mask) {
  pdl_wait();
  pdl_trigger();
  const int i = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (i >= n_dense) return;
  const int pos = pos0 + i;
  const int npre = min(prefix, pos + 1);
  for (int c = lane; c < (npre >> 6); c += 32) mask[(size_t)c * nq_pad + i] = ~0ull;
  if (lane == 0 && (npre & 63)) atomicOr(reinterpret_cast<unsigned long long*>(&mask[(size_t)(npre >> 6) * nq_pad + i]),
                                         (1ull << (npre & 63)) - 1ull);
  const int ns = min(max(__ldg(n_sel + i), 0), k);
  for (int e0 = 0; e0 < ns; e0 += 32) {
    const int e = e0 + lane;
    int c = -1;
    unsigned long long v = 0;
    if (e < ns) {
      const int t = __ldg(idx + (size_t)i * k + e);
      if ((unsigned)t > (unsigned)pos) {
        set_status(&g_status, kStBadBlock);  // outside the query's causal range: left out
      } else {
        c = t >> 6;
        v = 1ull << (t & 63);
      }
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long vo = __shfl_down_sync(0xffffffffu, v, o);
      const int co = __shfl_down_sync(0xffffffffu, c, o);
      if (lane + o < 32 && co == c) v |= vo;
    }
    const int cp = __shfl_up_sync(0xffffffffu, c, 1);
    if (c >= 0 && (lane == 0 || cp != c))
      atomicOr(reinterpret_cast<unsigned long long*>(&mask[(size_t)c * nq_pad + i]), v);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 4-D bf16 map over rows of `heads` x 128 values, `row_bytes` apart, viewed as
// (64 values, 2 halves, heads, rows); box (64, 1, box_heads, box_rows), 128-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* base, int heads, uint64_t rows, uint64_t row_bytes, int box_heads,
                 int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {64, 2, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[3] = {128, 256, (cuuint64_t)row_bytes};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int dense_tile_queries(int group) { return 128 / group; }

size_t dense_mask_bytes(const QS& qs, int n_dense) {
  if (n_dense <= 0) return 0;
  const size_t nq_pad = (size_t)((n_dense + 1) & ~1);
  const size_t chunks = (size_t)(qs.pos0 + n_dense - 1) / kBlock + 1;
  return nq_pad * chunks * 8;
}

cudaError_t setup_dense_kernels() {
  return cudaFuncSetAttribute(dense_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
}

cudaError_t launch_dense_attn(const AttnArgs& a, int n_dense, void* mask_ws, cudaStream_t st) {
  if (n_dense <= 0) return cudaSuccess;
  const int group = a.hq / a.kv.hkv;
  const int qt = dense_tile_queries(group);
  const int nq_pad = (n_dense + 1) & ~1;
  const size_t chunks = (size_t)(a.qs.pos0 + n_dense - 1) / kBlock + 1;
  uint64_t* mask = static_cast<uint64_t*>(mask_ws);
  CUtensorMap qmap, kmap, vmap;
  const uint64_t slot_bytes = (uint64_t)a.kv.row_stride * 2;
  if (!encode_rows(&qmap, a.q, a.hq, (uint64_t)a.qs.n_q, (uint64_t)a.hq * 256, group, qt) ||
      !encode_rows(&kmap, a.kv.k_cache, a.kv.hkv, (uint64_t)a.kv.num_blocks * kBlock, slot_bytes, 1, kBlock) ||
      !encode_rows(&vmap, a.kv.v_cache, a.kv.hkv, (uint64_t)a.kv.num_blocks * kBlock, slot_bytes, 1, kBlock))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(mask, 0, (size_t)nq_pad * chunks * 8, st);
  if (e != cudaSuccess) return e;
  e = launch_pdl(dense_mask_kernel, dim3((n_dense + 7) / 8), dim3(256), 0, st, 1, a.idx, a.n_sel, a.k, a.prefix,
                 a.qs.pos0, n_dense, nq_pad, mask);
  if (e != cudaSuccess) return e;
  DenseParams p;
  p.bt = a.kv.block_table + (size_t)a.qs.seq * a.kv.max_blocks;
  p.mask = mask;
  p.out = a.out;
  p.lse = a.lse;
  p.num_blocks = a.kv.num_blocks;
  p.n_dense = n_dense;
  p.nq_pad = nq_pad;
  p.pos0 = a.qs.pos0;
  p.hq = a.hq;
  p.hkv = a.kv.hkv;
  p.group = group;
  p.qt = qt;
  p.n_super = (n_dense + 2 * qt - 1) / (2 * qt);
  p.out_dtype = a.out_dtype;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  return launch_pdl(dense_attn_kernel, dim3(p.n_super * a.kv.hkv), dim3(kThreads), kSmem, st, 1, qmap, kmap, vmap,
                    p);
}

cudaError_t read_clear_status_dense(int* code, cudaStream_t st) {
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
