// Peak-rate microbenchmarks for the roofline denominators the measurement
// reports beside the DSA kernels (built as its own library, libdsa_probe.so;
// not part of the dsa_* interface).
//
//   probe_mma_s8    warp-level int8 tensor-core rate: mma.sync m16n8k32 s8
//                   with s32 accumulate, the instruction the prefill indexer GEMM
//                   uses (tcgen05 has no int8 kind on sm_103a).
//   probe_mma_bf16  the same for mma.sync m16n8k16 bf16 / f32 accumulate (the
//                   prefill prefix pass).
//   probe_tc        fifth-generation tensor-core rate: back-to-back tcgen05.mma
//                   of 128 x 256 tiles issued by one thread per CTA, kind::f8f6f4
//                   (e4m3, K = 32) or kind::f16 (f16, K = 16), fp32 accumulation
//                   in tensor memory (the prefill indexer's instructions).
//   probe_gather    bulk copies (cp.async.bulk into shared memory) of `piece`
//                   bytes from random offsets of a buffer: with a buffer that fits
//                   the L2 this is the rate at which the SMs can gather rows that
//                   L2 holds (the prefill attention's selected rows).
//
// Each function launches on the given stream and returns elapsed milliseconds
// measured with CUDA events on that stream (negative on a CUDA error).  The
// caller passes every buffer; nothing is allocated here.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "tc.cuh"

namespace {

constexpr int kMmaWarps = 8;   // warps per CTA
constexpr int kChains = 8;     // independent accumulators per warp

__global__ void __launch_bounds__(32 * kMmaWarps) mma_s8_kernel(int iters, int* sink) {
  const int lane = threadIdx.x & 31;
  uint32_t a0 = 0x01020304u * (lane + 1), a1 = a0 ^ 0x5a5a5a5au, a2 = a0 + 7, a3 = a1 - 3;
  uint32_t b0 = 0x03010204u ^ lane, b1 = b0 * 3u;
  int acc[kChains][4] = {};
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) dsa::mma_s8_16832(acc[c], a0, a1, a2, a3, b0, b1);
  }
  int s = 0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += acc[c][0] + acc[c][1] + acc[c][2] + acc[c][3];
  if (s == 0x7fffffff) *sink = s;  // keeps the chains live
}

__global__ void __launch_bounds__(32 * kMmaWarps) mma_bf16_kernel(int iters, int* sink) {
  const int lane = threadIdx.x & 31;
  const uint32_t a0 = dsa::pack_bf16x2(0.5f + lane, 1.f), a1 = dsa::pack_bf16x2(0.25f, -1.f);
  const uint32_t a2 = a0 ^ 0x00010001u, a3 = a1 ^ 0x00010001u;
  const uint32_t b0 = dsa::pack_bf16x2(0.125f, 2.f), b1 = dsa::pack_bf16x2(-0.5f, 1.f);
  float acc[kChains][4] = {};
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) dsa::mma_bf16_16816(acc[c], a0, a1, a2, a3, b0, b1);
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += acc[c][0] + acc[c][1] + acc[c][2] + acc[c][3];
  if (s == 1.2345f) *sink = 1;
}

// Four issuing warps (the attention kernel's producer count) share the pieces
// of each 64 KB stage; `stages` stages in flight per CTA; the offsets come from
// a per-thread linear congruential sequence masked to a power-of-two number of
// pieces.  A wait that runs out sets *sink and stops.
constexpr int kGatherStage = 64 * 1024;
constexpr int kGatherThreads = 128;

__global__ void __launch_bounds__(kGatherThreads, 1) gather_kernel(const uint8_t* src, uint64_t n_pieces_pow2,
                                                                 int piece, int stages, int iters, int* sink) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * kGatherStage);
  const int tid = threadIdx.x;
  const int per_stage = kGatherStage / piece;  // 16 .. 64 pieces
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) dsa::mbar_init(&full[s], 1);
    dsa::mbar_fence_init();
  }
  __syncthreads();
  uint64_t x = 0x9E3779B97F4A7C15ull * (blockIdx.x * kGatherThreads + tid + 1);
  const uint64_t mask = n_pieces_pow2 - 1;
  for (int n = 0; n < iters; ++n) {
    const int s = n % stages;
    if (n >= stages && !dsa::mbar_wait(&full[s], ((n / stages) - 1) & 1)) {
      atomicExch(sink, 1);
      return;
    }
    if (tid == 0) dsa::mbar_arrive_expect_tx(&full[s], (uint32_t)kGatherStage);
    for (int j = tid; j < per_stage; j += kGatherThreads) {
      x = x * 6364136223846793005ull + 1442695040888963407ull;
      const uint64_t pi = (x >> 24) & mask;
      dsa::bulk_g2s(smem + (size_t)s * kGatherStage + (size_t)j * piece, src + pi * piece, (uint32_t)piece, &full[s]);
    }
  }
  for (int n = iters > stages ? iters - stages : 0; n < iters; ++n) {
    const int s = n % stages;
    if (!dsa::mbar_wait(&full[s], (n / stages) & 1)) {
      atomicExch(sink, 2);
      return;
    }
  }
}

// One thread per CTA issues `iters` MMAs of 128 x 256 x K into one 256-column
// accumulator, then waits for them; the operands are zero (the rate does not
// depend on the values).
template <bool F8>
__global__ void __launch_bounds__(128, 1) tc_kernel(int iters, int* sink) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = base;
  uint8_t* sb = base + 16384;
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + 16384 + 32768);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x;
  for (int i = tid; i < (16384 + 32768) / 16; i += 128) reinterpret_cast<uint4*>(base)[i] = make_uint4(0, 0, 0, 0);
  if (tid < 32) dsa::tmem_alloc(tslot, 256);
  if (tid == 0) {
    dsa::mbar_init(bar, 1);
    dsa::mbar_fence_init();
  }
  dsa::fence_proxy_async();
  dsa::tc_fence_before();
  __syncthreads();
  dsa::tc_fence_after();
  const uint32_t tmem = *tslot;
  if (tid == 0) {
    constexpr uint32_t idesc = dsa::mma_idesc(128, 256, 0);
    for (int it = 0; it < iters; ++it) {
      const uint32_t k = it & 1;
      if (F8)
        dsa::mma_f8(tmem, dsa::smem_desc(dsa::smem_u32(sa) + 32 * k, 512, dsa::kSwizzle64),
                    dsa::smem_desc(dsa::smem_u32(sb) + 32 * k, 512, dsa::kSwizzle64), idesc, it > 0);
      else
        dsa::mma_f16(tmem, dsa::smem_desc(dsa::smem_u32(sa) + 32 * k, 1024, dsa::kSwizzle128),
                     dsa::smem_desc(dsa::smem_u32(sb) + 32 * k, 1024, dsa::kSwizzle128), idesc, it > 0);
    }
    dsa::mma_commit(bar);
  }
  if (!dsa::mbar_wait(bar, 0)) atomicExch(sink, 3);
  dsa::tc_fence_before();
  __syncthreads();
  dsa::tc_fence_after();
  if (tid < 32) dsa::tmem_dealloc(tmem, 256);
}

template <typename F>
float timed(cudaStream_t st, F launch) {
  cudaEvent_t a, b;
  if (cudaEventCreate(&a) != cudaSuccess) return -1.f;
  if (cudaEventCreate(&b) != cudaSuccess) {
    cudaEventDestroy(a);
    return -1.f;
  }
  float ms = -1.f;
  cudaEventRecord(a, st);
  launch();
  cudaEventRecord(b, st);
  if (cudaGetLastError() == cudaSuccess && cudaEventSynchronize(b) == cudaSuccess) cudaEventElapsedTime(&ms, a, b);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  return ms;
}

}  // namespace

extern "C" {

// Elapsed ms of `ctas` CTAs x 8 warps x iters x 8 mma.sync m16n8k32 s8
// (2 * 16 * 8 * 32 = 8192 integer operations each).
float probe_mma_s8(int ctas, int iters, int* sink, cudaStream_t st) {
  return timed(st, [&] { mma_s8_kernel<<<ctas, 32 * kMmaWarps, 0, st>>>(iters, sink); });
}

// Elapsed ms of `ctas` CTAs x 8 warps x iters x 8 mma.sync m16n8k16 bf16
// (2 * 16 * 8 * 16 = 4096 flops each).
float probe_mma_bf16(int ctas, int iters, int* sink, cudaStream_t st) {
  return timed(st, [&] { mma_bf16_kernel<<<ctas, 32 * kMmaWarps, 0, st>>>(iters, sink); });
}

// Elapsed ms of `ctas` CTAs (at most one per SM) x iters tcgen05.mma of
// 128 x 256 x K: e4m3 (f8 != 0; K = 32, 2 * 128 * 256 * 32 operations each)
// or f16 (K = 16, 2 * 128 * 256 * 16 flops each).
float probe_tc(int f8, int ctas, int iters, int* sink, cudaStream_t st) {
  auto kern = f8 ? tc_kernel<true> : tc_kernel<false>;
  // 80 KB of shared memory keeps to one or two CTAs per SM (256 TMEM columns each).
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 80 * 1024) != cudaSuccess) return -1.f;
  return timed(st, [&] { kern<<<ctas, 128, 80 * 1024, st>>>(iters, sink); });
}

// Elapsed ms of `ctas` CTAs each gathering iters x 64 KB in `piece`-byte bulk
// copies from random piece offsets of src (n_pieces_pow2 pieces, a power of
// two; src 16-byte aligned; piece a multiple of 16 dividing 64 KB, >= 1024).
float probe_gather(const void* src, unsigned long long n_pieces_pow2, int piece, int stages, int ctas, int iters,
                   int* sink, cudaStream_t st) {
  if (piece < 1024 || kGatherStage % piece || stages < 1 || stages > 3 || (n_pieces_pow2 & (n_pieces_pow2 - 1)))
    return -1.f;
  const size_t smem = (size_t)stages * kGatherStage + 8 * stages;
  if (cudaFuncSetAttribute(gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return -1.f;
  return timed(st, [&] {
    gather_kernel<<<ctas, kGatherThreads, smem, st>>>(static_cast<const uint8_t*>(src), n_pieces_pow2, piece, stages,
                                                     iters, sink);
  });
}

}  // extern "C"
