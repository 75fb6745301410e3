// Cache maintenance and the stand-alone gather.
//
// kv_write scatters new tokens into their paged slots (§2.2 blocks of
// consecutive positions).  kv_gather is the literal "gather first" step of
// §2.2: the attended rows of every query copied into a contiguous buffer,
// 16 bytes per thread, prefix rows first, then the selected rows in order.
// The attention kernels do not need it (they gather into shared memory).
#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

__device__ int g_status;

struct WriteParams {
  __nv_bfloat16* kc;
  __nv_bfloat16* vc;
  int8_t* ic;
  const int32_t* slots;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int8_t* ik;
  int ntok, hkv, num_blocks, row_stride;
};

// One CTA per token: Hkv x 16 chunks of K, the same of V, 4 chunks of the indexer key.
// A slot's K (and V) row holds all KV heads contiguously (row_stride values apart
// from the next slot's), so both copies are straight runs.
__global__ void kv_write_kernel(const WriteParams p) {
  const int j = blockIdx.x;
  const int slot = __ldg(p.slots + j);
  const int blk = slot >> 6, row = slot & 63;
  if (slot < 0 || blk >= p.num_blocks) {
    if (threadIdx.x == 0) set_status(&g_status, kStBadBlock);
    return;
  }
  const int kv_chunks = p.hkv * 16;
  for (int c = threadIdx.x; c < 2 * kv_chunks + 4; c += blockDim.x) {
    if (c < 2 * kv_chunks) {
      const bool is_v = c >= kv_chunks;
      const int cc = is_v ? c - kv_chunks : c;
      const __nv_bfloat16* src = (is_v ? p.v : p.k) + (size_t)j * p.hkv * kHeadDim + cc * 8;
      __nv_bfloat16* dst = (is_v ? p.vc : p.kc) + (size_t)slot * p.row_stride + cc * 8;
      *reinterpret_cast<int4*>(dst) = __ldg(reinterpret_cast<const int4*>(src));
    } else {
      const int ch = c - 2 * kv_chunks;
      *reinterpret_cast<int4*>(p.ic + ((size_t)blk * kBlock + row) * kIdxDim + ch * 16) =
          __ldg(reinterpret_cast<const int4*>(p.ik + (size_t)j * kIdxDim + ch * 16));
    }
  }
}

// Per-head write (the write side of the per-head block bitmaps): one CTA per
// token, head h's K and V (16 chunks each) into the head-h slice of slot
// slots[j][h], and its indexer key (4 chunks) into the head-h keys of that block
// (indexer cache [blocks][hkv][64][64]).  Other heads' slices are not touched.
__global__ void kv_write_heads_kernel(const WriteParams p) {
  const int j = blockIdx.x;
  for (int c = threadIdx.x; c < p.hkv * 36; c += blockDim.x) {
    const int h = c / 36, r = c - h * 36;
    const int slot = __ldg(p.slots + (size_t)j * p.hkv + h);
    const int blk = slot >> 6, row = slot & 63;
    if (slot < 0 || blk >= p.num_blocks) {
      if (r == 0) set_status(&g_status, kStBadBlock);
      continue;
    }
    if (r < 32) {
      const bool is_v = r >= 16;
      const int cc = r & 15;
      const __nv_bfloat16* src = (is_v ? p.v : p.k) + ((size_t)j * p.hkv + h) * kHeadDim + cc * 8;
      __nv_bfloat16* dst = (is_v ? p.vc : p.kc) + (size_t)slot * p.row_stride + h * kHeadDim + cc * 8;
      *reinterpret_cast<int4*>(dst) = __ldg(reinterpret_cast<const int4*>(src));
    } else {
      const int ch = r - 32;
      *reinterpret_cast<int4*>(p.ic + (((size_t)blk * p.hkv + h) * kBlock + row) * kIdxDim + ch * 16) =
          __ldg(reinterpret_cast<const int4*>(p.ik + ((size_t)j * p.hkv + h) * kIdxDim + ch * 16));
    }
  }
}

struct GatherParams {
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  const int32_t* bt;
  const int32_t* ctx;
  const int32_t* idx;
  const int32_t* nsel;
  __nv_bfloat16* ko;
  __nv_bfloat16* vo;
  int mode, seq, pos0, max_blocks, num_blocks, hkv, k, prefix, rows_out, max_ctx, row_stride;
};

// CTA: 8 output rows of one (query, KV head); 16 threads per row.
__global__ void __launch_bounds__(128) kv_gather_kernel(const GatherParams p) {
  const int qi = blockIdx.z, g = blockIdx.y;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 4), ch = threadIdx.x & 15;
  if (r >= p.rows_out) return;
  const int seq = p.mode == 0 ? qi : p.seq;
  const int pos = p.mode == 0 ? min(__ldg(p.ctx + qi), p.max_ctx) - 1 : p.pos0 + qi;
  const int n_pre = max(0, min(p.prefix, pos + 1));
  const int ns = min(max(__ldg(p.nsel + qi), 0), p.k);
  const size_t o = (((size_t)qi * p.hkv + g) * p.rows_out + r) * kHeadDim + ch * 8;
  int4 kval = make_int4(0, 0, 0, 0), vval = kval;
  if (r < n_pre + ns) {
    const int t = r < n_pre ? r : __ldg(p.idx + (size_t)qi * p.k + (r - n_pre));
    int blk = 0;
    if (t >= 0 && t < p.max_blocks * kBlock)
      blk = load_block(p.bt, seq, p.max_blocks, t >> 6, p.num_blocks, &g_status);
    else
      set_status(&g_status, kStBadBlock);
    const size_t src = ((size_t)blk * kBlock + (t & 63)) * p.row_stride + (size_t)g * kHeadDim + ch * 8;
    kval = __ldg(reinterpret_cast<const int4*>(p.kc + src));
    vval = __ldg(reinterpret_cast<const int4*>(p.vc + src));
  }
  *reinterpret_cast<int4*>(p.ko + o) = kval;
  *reinterpret_cast<int4*>(p.vo + o) = vval;
}

}  // namespace

cudaError_t launch_kv_write_heads(const KV& kv, const int32_t* slots, int ntok, const void* k, const void* v,
                                  const int8_t* idx_k, cudaStream_t st) {
  WriteParams p;
  p.kc = static_cast<__nv_bfloat16*>(const_cast<void*>(kv.k_cache));
  p.vc = static_cast<__nv_bfloat16*>(const_cast<void*>(kv.v_cache));
  p.ic = const_cast<int8_t*>(kv.idx_cache);
  p.slots = slots;
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.ik = idx_k;
  p.ntok = ntok;
  p.hkv = kv.hkv;
  p.num_blocks = kv.num_blocks;
  p.row_stride = kv.row_stride;
  kv_write_heads_kernel<<<ntok, 128, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_kv_write(const KV& kv, const int32_t* slots, int ntok, const void* k, const void* v,
                            const int8_t* idx_k, cudaStream_t st) {
  WriteParams p;
  p.kc = static_cast<__nv_bfloat16*>(const_cast<void*>(kv.k_cache));
  p.vc = static_cast<__nv_bfloat16*>(const_cast<void*>(kv.v_cache));
  p.ic = const_cast<int8_t*>(kv.idx_cache);
  p.slots = slots;
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.ik = idx_k;
  p.ntok = ntok;
  p.hkv = kv.hkv;
  p.num_blocks = kv.num_blocks;
  p.row_stride = kv.row_stride;
  kv_write_kernel<<<ntok, 128, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_kv_gather(const KV& kv, const QS& qs, const int32_t* idx, const int32_t* n_sel, int k,
                             int prefix, void* k_out, void* v_out, cudaStream_t st) {
  GatherParams p;
  p.kc = static_cast<const __nv_bfloat16*>(kv.k_cache);
  p.vc = static_cast<const __nv_bfloat16*>(kv.v_cache);
  p.bt = kv.block_table;
  p.ctx = kv.context_lens;
  p.idx = idx;
  p.nsel = n_sel;
  p.ko = static_cast<__nv_bfloat16*>(k_out);
  p.vo = static_cast<__nv_bfloat16*>(v_out);
  p.mode = qs.mode;
  p.seq = qs.seq;
  p.pos0 = qs.pos0;
  p.max_blocks = kv.max_blocks;
  p.num_blocks = kv.num_blocks;
  p.hkv = kv.hkv;
  p.k = k;
  p.prefix = prefix;
  p.rows_out = prefix + k;
  p.max_ctx = kv.max_ctx;
  p.row_stride = kv.row_stride;
  dim3 grid((p.rows_out + 7) / 8, kv.hkv, qs.n_q);
  kv_gather_kernel<<<grid, 128, 0, st>>>(p);
  return cudaGetLastError();
}

// Staging copy between device memory and page-locked host memory (or device to
// device) by the SMs: 16-byte loads and stores over a grid-stride loop, after
// the wait on the previous kernel of the stream (which may have written src).
// Host memory is reached through its device-side address (unified addressing).
namespace {
__global__ void __launch_bounds__(256) stage_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                         size_t n16) {
  pdl_wait();
  pdl_trigger();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) dst[i] = src[i];
}
}  // namespace

cudaError_t launch_stage_copy(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  const size_t n16 = bytes / 16;
  size_t blocks = (n16 + 255) / 256;
  const size_t cap = 4 * (size_t)attn_grid_ctas();
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(stage_copy_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1,
                    static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
}

cudaError_t read_clear_status_misc(int* code, cudaStream_t st) {
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
