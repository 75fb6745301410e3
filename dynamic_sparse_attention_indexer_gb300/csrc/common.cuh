// Device-side building blocks shared by the DSA kernels (sm_103a).
//
// Inline PTX for the Blackwell data-movement path: mbarrier-tracked bulk
// copies (cp.async.bulk) into shared memory, 16-byte cp.async with zero fill,
// ldmatrix, and the warp-level mma.sync shapes the kernels use.  Every wait is
// bounded by the global timer; a wait that runs out records DSA_ERR_TIMEOUT in
// the caller's status word instead of hanging.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

namespace dsa {

constexpr int kBlock = 64;      // positions per KV block
constexpr int kHeadDim = 128;   // attention head dim
constexpr int kIdxDim = 64;     // indexer dim (int8)

// Score histogram: bin = clamp(s + kHistOff, 0, kHistBins - 1).  Interior bins
// are one score wide (exact for s in [-4095, 4094]); the two edge bins collect
// everything outside and trigger an exact radix refinement.
constexpr int kHistBins = 8192;
constexpr int kHistOff = 4096;

// Coarse score histogram of the decode top-k: bins 16 scores wide,
// bin = clamp((s >> 4) + 512, 0, 1023).  Interior bin b holds the scores
// [(b - 512) * 16, (b - 512) * 16 + 15]; the edge bins 0 and 1023 collect the
// rest and send the selection to the exact radix fallback.
constexpr int kCoarseBins = 1024;
constexpr int kCoarseShift = 4;
constexpr int kCoarseOff = 512;
constexpr int kFineBins = 1 << kCoarseShift;

enum : int { kStOk = 0, kStBadBlock = 4, kStTimeout = 6 };
enum : int { kSelAll = 1, kSelThreshold = 0 };

__device__ __forceinline__ int hist_bin(int s) {
  return min(max(s + kHistOff, 0), kHistBins - 1);
}
__device__ __forceinline__ int coarse_bin(int s) {
  return min(max((s >> kCoarseShift) + kCoarseOff, 0), kCoarseBins - 1);
}

// Record the first error only.
__device__ __forceinline__ void set_status(int* st, int code) { atomicCAS(st, 0, code); }

// Block id of block-table slot j of sequence `seq`, checked against the pool.
__device__ __forceinline__ int load_block(const int32_t* __restrict__ bt, int seq, int max_blocks,
                                          int j, int num_blocks, int* status) {
  int blk = __ldg(bt + (size_t)seq * max_blocks + j);
  if ((unsigned)blk >= (unsigned)num_blocks) {
    set_status(status, kStBadBlock);
    blk = 0;
  }
  return blk;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy ones (bulk copies into the same buffer once it is released).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Barrier over the first `count` threads of the CTA (count a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Waits for phase `parity` of `bar` to complete, for at most ~2 s.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > 2000000000ull) return false;
  }
}

// Bulk copy global -> this CTA's shared memory, completion counted on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// The same with an L2 cache policy made by createpolicy (l2_evict_first below).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// L2 policy for data streamed once per call (the decode step's indexer keys and
// K/V rows): those lines go first, so that the small data a call writes and
// reads back (scores, histograms, partial states, block tables) stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

// ------------------------------------------- programmatic dependent launch
// A kernel launched with launch_pdl may start while the previous kernel of the
// stream is still running; pdl_wait() blocks until that kernel has completed
// and its writes are visible, so every kernel calls it before its first global
// memory access.  pdl_trigger() lets the next kernel start launching early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// With cluster_x > 1 the grid is launched in clusters of cluster_x CTAs along x.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster_x > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same launch without programmatic dependent launch: the kernel starts only
// once the previous work of the stream has completed (for a kernel that reads
// inputs before its dependency wait, when the previous kernel produces them).
template <typename... Params, typename... Args>
cudaError_t launch_ordered(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                           Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------ cp.async
// 16-byte async copy; src_bytes = 0 writes zeros (zero fill) without reading.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ ldmatrix
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// --------------------------------------------------------------------- mma
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A(16x32 s8, row) * B(32x8 s8, col) + D, s32 accumulate (exact).
__device__ __forceinline__ void mma_s8_16832(int* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------ integer dot product
// Sum of four int8 products, accumulated in int32 (exact).
__device__ __forceinline__ int dot4(int a, int b, int c) { return __dp4a(a, b, c); }

// ------------------------------------------------------------ block scans
// Exclusive prefix sum over the CTA (blockDim.x threads, multiple of 32).
// `scratch` holds at least blockDim.x / 32 + 1 ints.  Returns the total in *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) scratch[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  int base = warp > 0 ? scratch[warp - 1] : 0;
  int t = scratch[nw - 1];
  __syncthreads();
  *total = t;
  return base + x - v;
}

}  // namespace dsa
