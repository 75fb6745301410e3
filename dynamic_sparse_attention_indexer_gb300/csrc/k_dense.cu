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
// queries), heaviest (latest) tiles first, 320 threads, in steps of 128
// positions (two cache blocks):
//   warp 8       producer: TMA loads of the two Q tiles (once), then per step
//                the two K blocks of the KV head (8 KB boxes, 128-byte swizzle)
//                with the tiles' mask words, and the two V blocks, into 2-stage
//                rings (K stage i + 1 and V stage i free up together: the
//                products of step i - 1 and the S of step i are issued back to
//                back);
//   warp 9       one thread issues the MMAs, per tile t: O_t += P_t(i) V(i) (P
//                in tensor memory as two bf16 terms, hi and the residual lo; V
//                an MN-major operand) and then S_t(i + 1) = Q_t K(i + 1)^T
//                (M = 128, N = 128, K = 16 per instruction, the shape at which
//                one issuing thread keeps the tensor core at its full rate: an
//                issue costs ~63 cycles, an N = 64 product only 34), each group
//                committed to an mbarrier.  The tiles alternate, so one tile's
//                softmax overlaps the other tile's products;
//   warps 0-7    softmax, one thread per (query, head) row (TMEM lane), warps
//                0-3 tile 0 and 4-7 tile 1: masked online softmax in base 2 with a
//                lazy rescale of O (only when the running max grows by more than
//                2^8) and P = hi + lo (about 16 significant bits, as in the
//                gathered path: a single bf16 P costs 2^-9 |v| per dominant
//                weight, more than the attention's tolerance when few keys carry
//                the softmax), written over S in tensor memory, and at the end
//                O / l and the log-sum-exp.
// Tensor memory per tile t at column 256 t: S (128 fp32 columns), overwritten
// by P in place, 32 positions at a time: positions 32c .. 32c + 31 as P_hi in
// columns 32c .. 32c + 15 and P_lo in 32c + 16 .. 32c + 31 (two bf16 per
// column); O in columns 128 .. 255.  S(i + 1) overwrites P(i): the tcgen05.mma
// operations of one thread run in issue order, so P V reads P first.
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

constexpr int kStages = 2;       // K and V ring stages, one 128-position step each
constexpr int kThreads = 320;
constexpr uint32_t kQHalf = 16384;   // 128 rows x 128 bytes: one 64-wide half of the head dim
constexpr uint32_t kKVBlockHalf = 8192;            // 64 positions x 128 bytes
constexpr uint32_t kKVHalf = 2 * kKVBlockHalf;     // 128 positions x 128 bytes
constexpr uint32_t kKVStage = 2 * kKVHalf;
constexpr uint32_t kMaskChunk = 2048;  // up to 2 x 128 mask words of one block
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = 4 * kQHalf;
constexpr uint32_t kOffV = kOffK + kStages * kKVStage;
constexpr uint32_t kOffMask = kOffV + kStages * kKVStage;
constexpr uint32_t kOffBar = kOffMask + kStages * 2 * kMaskChunk;
constexpr uint32_t kNumBars = 1 + 5 * kStages + 2 + 2 + 2;
constexpr uint32_t kSmem = kOffBar + kNumBars * 8 + 16 + 1024;  // + TMEM address slot + alignment slack
static_assert(kSmem <= 227 * 1024, "shared memory budget");
constexpr uint32_t kColO = 128;  // tensor-memory column of O within a tile's 256
constexpr float kRescaleLog2 = 8.f;  // O is rescaled only when the max grows by more than this (base-2 units)

struct DenseParams {
  const int32_t* bt;      // block-table row of the sequence
  const uint64_t* mask;   // [chunks][nq_pad] attended-position bitmap of the dense queries
  void* out;
  float* lse;
  int num_blocks, n_dense, nq_pad, pos0, hq, hkv, group, qt, n_super, out_dtype;
  int window;  // > 0: the attended set is the causal window [pos - window + 1, pos] (no bitmap)
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
__device__ __forceinline__ bool mbar_try_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(100000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_sleep_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_sleep(bar, parity)) return true;  // the usual case: no timer read
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_sleep(bar, parity)) return true;
    if (global_ns() - t0 > 2000000000ull) return false;
  }
}

// The same with every lane of the warp; the result is warp-uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_sleep_wait(bar, parity));
}

// POS_SCALE: softmax_scale > 0 (the usual case: the max of the scaled scores is
// the scale times the raw max); otherwise every score is scaled first.
template <bool POS_SCALE>
__global__ void __launch_bounds__(kThreads, 1)
    dense_attn_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const DenseParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;  // K blocks and mask words of a step landed
  uint64_t* k_empty = k_full + kStages;
  uint64_t* m_free = k_empty + kStages;  // mask words read, one arrival per softmax warp
  uint64_t* v_full = m_free + kStages;
  uint64_t* v_empty = v_full + kStages;
  uint64_t* s_full = v_empty + kStages;  // [tile]: S(i) computed (and every earlier product done)
  uint64_t* p_full = s_full + 2;         // [tile]: P(i) written, one arrival per softmax warp
  uint64_t* drain = p_full + 2;
  uint64_t* tail = drain + 1;            // V rows past the tiles' last position zeroed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(tail + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x % p.hkv;
  const int q0 = (p.n_super - 1 - blockIdx.x / p.hkv) * 2 * p.qt;  // heaviest tiles first
  const int q_last = min(q0 + 2 * p.qt, p.n_dense) - 1;
  const int pos_last = p.pos0 + q_last;
  // blocks of 64 positions the tiles see: from block 0, or, with a window, from
  // the block holding the first query's first window position
  const int c_begin = p.window > 0 ? max(0, p.pos0 + q0 - p.window + 1) / kBlock : 0;
  const int nc = pos_last / kBlock + 1 - c_begin;
  const int ns = (nc + 1) / 2;  // steps of two blocks
  const int last_rows = pos_last - c_begin * kBlock - (ns - 1) * 2 * kBlock + 1;  // positions of the last step in range (1..128)
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&m_free[s], 8);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
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
    // ------------------------------------------------------------- producer
    const int mwords = p.window > 0 ? 0 : min(2 * p.qt, p.nq_pad - q0);  // even: q0 and nq_pad are even
    if (lane == 0) {
      tma_prefetch_map(&qmap);
      tma_prefetch_map(&kmap);
      tma_prefetch_map(&vmap);
      mbar_arrive_expect_tx(q_full, 4u * (uint32_t)(p.group * p.qt) * 128u);
      for (int t = 0; t < 2; ++t)
        for (int x = 0; x < 2; ++x)
          tma_load_4d(base + kOffQ + (t * 2 + x) * kQHalf, &qmap, 0, x, g * p.group, q0 + t * p.qt, q_full);
    }
    int blk_next = 0;
    int k_issued = 0, v_issued = 0;
    for (int i = 0; i < ns; ++i) {
      const int c0 = 2 * i, nb = c0 + 1 < nc ? 2 : 1;  // blocks in this step
      if ((c0 & 31) == 0)
        blk_next = c0 + lane < nc ? load_block(p.bt, 0, 0, c_begin + c0 + lane, p.num_blocks, &g_status) : 0;
      const int b0 = __shfl_sync(0xffffffffu, blk_next, c0 & 31);
      const int b1 = __shfl_sync(0xffffffffu, blk_next, (c0 + 1) & 31);
      const int s = i % kStages;
      const uint32_t par = ((i / kStages) + 1) & 1;
      if (i >= kStages && !(warp_wait(&k_empty[s], par) && warp_wait(&m_free[s], par))) break;
      if (lane == 0) {
        uint8_t* st = base + kOffK + s * kKVStage;
        mbar_arrive_expect_tx(&k_full[s], (uint32_t)nb * (2 * kKVBlockHalf + (uint32_t)mwords * 8u));
        for (int a = 0; a < nb; ++a) {
          for (int x = 0; x < 2; ++x)
            tma_load_4d(st + x * kKVHalf + a * kKVBlockHalf, &kmap, 0, x, g, (a ? b1 : b0) * kBlock, &k_full[s]);
          if (mwords > 0)
            bulk_g2s(base + kOffMask + (s * 2 + a) * kMaskChunk, p.mask + (size_t)(c_begin + c0 + a) * p.nq_pad + q0,
                     (uint32_t)mwords * 8u, &k_full[s]);
        }
      }
      k_issued = i + 1;
      if (i >= kStages && !warp_wait(&v_empty[s], par)) break;
      if (lane == 0) {
        uint8_t* st = base + kOffV + s * kKVStage;
        mbar_arrive_expect_tx(&v_full[s], (uint32_t)nb * 2 * kKVBlockHalf);
        for (int a = 0; a < nb; ++a)
          for (int x = 0; x < 2; ++x)
            tma_load_4d(st + x * kKVHalf + a * kKVBlockHalf, &vmap, 0, x, g, (a ? b1 : b0) * kBlock, &v_full[s]);
      }
      v_issued = i + 1;
    }
    if (v_issued < ns && lane == 0) set_status(&g_status, kStTimeout);
    // every copy this warp started has landed before the CTA ends
    bool landed = true;
    for (int i = max(k_issued - kStages, 0); i < k_issued; ++i)
      if (!warp_wait(&k_full[i % kStages], (i / kStages) & 1)) landed = false;
    for (int i = max(v_issued - kStages, 0); i < v_issued; ++i)
      if (!warp_wait(&v_full[i % kStages], (i / kStages) & 1)) landed = false;
    if (!landed && lane == 0) set_status(&g_status, kStTimeout);
    // Positions of the last step past the tiles' last position (a block not
    // loaded, or unwritten slots of the last block) may hold anything; P is zero
    // there, and their V rows are zeroed so that no non-finite value meets a
    // zero weight in the product.
    if (landed && v_issued == ns && last_rows < 2 * kBlock) {
      uint8_t* vt = base + kOffV + ((ns - 1) % kStages) * kKVStage;
      const int n16 = (2 * kBlock - last_rows) * 8;  // 16-byte pieces per half
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
      constexpr uint32_t idesc_s = mma_idesc(128, 128, kFmtBF16);
      constexpr uint32_t idesc_o = mma_idesc(128, 128, kFmtBF16, 0, 1);
      bool ok = mbar_sleep_wait(q_full, 0);
      tc_fence_after();
      // descriptors computed once; a byte offset o added to the start address adds o >> 4
      const uint64_t dq = smem_desc(smem_u32(base + kOffQ), 1024, kSwizzle128);
      const uint64_t dk = smem_desc(smem_u32(base + kOffK), 1024, kSwizzle128);
      const uint64_t dv = smem_desc_mn(smem_u32(base + kOffV), kKVHalf, 1024);
      auto issue_qk = [&](int t, int i) {  // S_t(i) = Q_t K(i)^T
        const uint64_t kb = dk + (uint64_t)((i % kStages) * (kKVStage >> 4));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_f16(tmem + t * 256, dq + (uint64_t)((t * 2 * kQHalf + (kk >> 2) * kQHalf + (kk & 3) * 32) >> 4),
                  kb + (uint64_t)(((kk >> 2) * kKVHalf + (kk & 3) * 32) >> 4), idesc_s, kk > 0);
        mma_commit(&s_full[t]);
      };
      if (ok) ok = mbar_sleep_wait(&k_full[0], 0);
      tc_fence_after();
      if (ok) {
        issue_qk(0, 0);
        issue_qk(1, 0);
        mma_commit(&k_empty[0]);
      }
      for (int i = 0; ok && i < ns; ++i) {
        const int sv = i % kStages;
        ok = mbar_sleep_wait(&v_full[sv], (i / kStages) & 1);
        if (ok && i == ns - 1 && last_rows < 2 * kBlock) ok = mbar_sleep_wait(tail, 0);
        if (ok && i + 1 < ns) ok = mbar_sleep_wait(&k_full[(i + 1) % kStages], ((i + 1) / kStages) & 1);
        tc_fence_after();
        const uint64_t vb = dv + (uint64_t)(sv * (kKVStage >> 4));
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!(ok = ok && mbar_sleep_wait(&p_full[t], i & 1))) break;
          tc_fence_after();
          // O_t += (P_hi + P_lo)_t(i) V(i): 8 steps of 16 positions, P columns of
          // positions 16kk .. 16kk + 15 at 32 (kk / 2) + 8 (kk % 2) (+ 16 for lo)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ts(tmem + t * 256 + kColO, tmem + t * 256 + 32 * (kk >> 1) + 8 * (kk & 1) + 16 * h,
                         vb + (uint64_t)((kk * 2048) >> 4), idesc_o, i > 0 || h > 0 || kk > 0);
          if (i + 1 < ns) issue_qk(t, i + 1);  // overwrites P_t(i) after the products above have read it
          else mma_commit(&s_full[t]);         // the last products done: the epilogue's signal
        }
        mma_commit(&v_empty[sv]);
        if (i + 1 < ns) mma_commit(&k_empty[(i + 1) % kStages]);
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
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + t * 256;
    constexpr bool pos_scale = POS_SCALE;
    const uint64_t c2 = pos_scale ? f2_pack(p.scale_log2, p.scale_log2) : f2_pack(1.f, 1.f);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < ns; ++i) {
      const int s = i % kStages;
      if (!(ok = warp_wait(&s_full[t], i & 1))) break;
      tc_fence_after();
      // the step's mask words came with its K blocks (phase i / kStages of k_full[s]); the producer
      // refills the stage only after every softmax warp has read them (m_free)
      if (!(ok = warp_wait(&k_full[s], (i / kStages) & 1))) break;
      uint64_t w[2] = {0ull, 0ull};
      if (valid && p.window > 0) {  // the window [qpos - window + 1, qpos] within each block of the step
        const int qpos = p.pos0 + qd;
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          const int first = (c_begin + 2 * i + a) * kBlock;
          const int lo = max(qpos - p.window + 1 - first, 0), hi = min(qpos - first, kBlock - 1);
          if (2 * i + a < nc && lo <= hi)
            w[a] = (hi == kBlock - 1 ? ~0ull : (1ull << (hi + 1)) - 1ull) & ~((1ull << lo) - 1ull);
        }
      } else if (valid) {
        w[0] = reinterpret_cast<const uint64_t*>(base + kOffMask + (s * 2) * kMaskChunk)[mword];
        if (2 * i + 1 < nc) w[1] = reinterpret_cast<const uint64_t*>(base + kOffMask + (s * 2 + 1) * kMaskChunk)[mword];
      }
      fence_proxy_async_smem();  // the mask words are refilled by a bulk copy
      __syncwarp();
      if (lane == 0) mbar_arrive(&m_free[s]);
      // The step's 128 positions in two halves of 64.  Each half's S is read from
      // tensor memory once (P is written over it): tensor-memory reads from the
      // threads compete with the products for its bandwidth, so a separate max
      // pass over S cost more than it saved, and holding all 128 scores in
      // registers spilled.  When the second half raises the running max past the
      // lazy threshold, the first half's P is rescaled together with O.
      uint64_t sum2 = f2_pack(0.f, 0.f);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t sv[2][32];
        tmem_ld32_nowait(lane_addr + 64 * hh, sv[0]);
        tmem_ld32_nowait(lane_addr + 64 * hh + 32, sv[1]);
        tmem_wait_ld();
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t wb = q ? (uint32_t)(w[hh] >> 32) : (uint32_t)w[hh];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float x = (wb >> e) & 1u ? __uint_as_float(sv[q][e]) : -INFINITY;
            if (!pos_scale) x = x == -INFINITY ? -INFINITY : x * p.scale_log2;
            sv[q][e] = __float_as_uint(x);
          }
          float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            a0 = max3(a0, __uint_as_float(sv[q][e]), __uint_as_float(sv[q][e + 1]));
            a1 = max3(a1, __uint_as_float(sv[q][e + 2]), __uint_as_float(sv[q][e + 3]));
          }
          mx = max3(mx, a0, a1);
        }
        if (pos_scale) mx *= p.scale_log2;  // -inf stays -inf
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
        // O (the products of the previous steps are complete: s_full of this step
        // came after them) and, in the second half, this step's first-half P.  The
        // tensor-memory loads and stores are warp-wide, so the warp rescales if any
        // row needs it, the other rows by 1.
        if (__any_sync(0xffffffffu, rescale)) {
          if (hh == 1) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t hl[32];  // [0, 16): hi, [16, 32): lo of positions 32c .. 32c + 31, two per column
              tmem_ld32(lane_addr + 32 * c, hl);
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float a = (__uint_as_float(hl[e] << 16) + __uint_as_float(hl[16 + e] << 16)) * factor;
                const float b =
                    (__uint_as_float(hl[e] & 0xffff0000u) + __uint_as_float(hl[16 + e] & 0xffff0000u)) * factor;
                const uint32_t ab = __float_as_uint(a), bb = __float_as_uint(b);
                hl[e] = __byte_perm(ab, bb, 0x7632);
                hl[16 + e] =
                    pack_bf16x2(a - __uint_as_float(ab & 0xffff0000u), b - __uint_as_float(bb & 0xffff0000u));
              }
              tmem_st32(lane_addr + 32 * c, hl);
            }
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_addr + kColO + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
            tmem_st32(lane_addr + kColO + c * 32, o);
          }
        }
        const float m_use = m == -INFINITY ? 0.f : m;
        const uint64_t nm2 = f2_pack(-m_use, -m_use);
        // p = 2^(scale s - m); P = hi + lo with hi the truncated top 16 bits of p
        // (exact bf16) and lo = p - hi rounded to bf16 (~16 bits in all)
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {  // positions 64 hh + 16 c8 .. + 15
          const int q = c8 >> 1, o = 16 * (c8 & 1);
          uint32_t ph[8], pl[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float a, b;
            f2_unpack(
                f2_fma(f2_pack(__uint_as_float(sv[q][o + 2 * e]), __uint_as_float(sv[q][o + 2 * e + 1])), c2, nm2), a,
                b);
            a = ex2(a);
            b = ex2(b);
            const uint64_t pp = f2_pack(a, b);
            sum2 = f2_add(sum2, pp);
            const uint32_t ab = __float_as_uint(a), bb = __float_as_uint(b);
            ph[e] = __byte_perm(ab, bb, 0x7632);
            float la, lb;
            f2_unpack(f2_sub(pp, f2_pack(__uint_as_float(ab & 0xffff0000u), __uint_as_float(bb & 0xffff0000u))), la,
                      lb);
            pl[e] = pack_bf16x2(la, lb);
          }
          // positions 32c + o .. + 15 (c = 2 hh + q): hi in columns 32c + o / 2 .. + 7, lo 16 columns further
          const int c = 2 * hh + q;
          tmem_st8_nowait(lane_addr + 32 * c + o / 2, ph);
          tmem_st8_nowait(lane_addr + 32 * c + 16 + o / 2, pl);
        }
        if (hh == 0) {  // the first half's weights into l before a possible rescale in the second
          float s0, s1;
          f2_unpack(sum2, s0, s1);
          l += s0 + s1;
          sum2 = f2_pack(0.f, 0.f);
          tmem_wait_st();  // its P is in tensor memory before the second half may rescale it
        }
      }
      {
        float s0, s1;
        f2_unpack(sum2, s0, s1);
        l += s0 + s1;
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    // ---- epilogue: O / l, log-sum-exp, once the last products are done
    if (ok && (ok = warp_wait(&s_full[t], ns & 1))) {
      tc_fence_after();
      const int head = g * p.group + (r - qi * p.group);
      const size_t row = (size_t)qd * p.hq + head;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + kColO + c * 32, o);
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
  cudaError_t e = cudaFuncSetAttribute(dense_attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dense_attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  return e;
}

cudaError_t launch_dense_attn(const AttnArgs& a, int n_dense, void* mask_ws, cudaStream_t st, int window,
                              bool mask_ready) {
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
  if (window <= 0 && !mask_ready) {  // the attended-position bitmap of the selections
    cudaError_t e = cudaMemsetAsync(mask, 0, (size_t)nq_pad * chunks * 8, st);
    if (e != cudaSuccess) return e;
    e = launch_pdl(dense_mask_kernel, dim3((n_dense + 7) / 8), dim3(256), 0, st, 1, a.idx, a.n_sel, a.k, a.prefix,
                   a.qs.pos0, n_dense, nq_pad, mask);
    if (e != cudaSuccess) return e;
  }
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
  p.window = window > 0 ? window : 0;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  return launch_pdl(p.scale_log2 > 0.f ? dense_attn_kernel<true> : dense_attn_kernel<false>,
                    dim3(p.n_super * a.kv.hkv), dim3(kThreads), kSmem, st, 1, qmap, kmap, vmap, p);
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
