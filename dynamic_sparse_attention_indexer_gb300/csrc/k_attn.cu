// Step 3 + 4 of DSA (§2.2 gather, §2.3 attention): GQA attention of each query
// token over its attended rows, read straight from the paged KV cache.
//
// One CTA owns (query, KV head, split of the attended rows) and serves all G
// query heads of that KV head, so every selected row is read from HBM once per
// token (§2.3 decode: load only the active KV).  Rows are gathered with 16-byte
// cp.async into an XOR-swizzled shared-memory ring of 64-row tiles, several
// tiles in flight, so the next tile's gather overlaps the current tile's math
// (§2.3 prefetch).  The contraction runs on the tensor cores (mma.sync m16n8k16
// bf16, fp32 accumulate) with the G heads as the M dimension; the softmax is
// online in fp32 (base 2), reduced across the quad with warp shuffles.  Warps
// merge through shared memory; splits merge in a second small kernel.
#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

__device__ int g_status;

constexpr int kAttnThreads = 128;  // 4 warps x 16 rows of each 64-row tile
constexpr int kTileRows = 64;
constexpr int kStages = 3;
constexpr int kRowBytes = kHeadDim * 2;                 // 256 B per K or V row
constexpr int kTileBytes = kTileRows * kRowBytes;       // 16 KB
constexpr int kStageBytes = 2 * kTileBytes;             // K + V
constexpr int kQBytes = 16 * kRowBytes;                 // 16 head rows (G <= 16, zero padded)
constexpr int kMaxRowsPerSplit = 4096;

struct AttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  const int32_t* bt;
  const int32_t* ctx;
  const int32_t* idx;
  const int32_t* nsel;
  int mode, seq, pos0;
  int max_blocks, num_blocks, hkv, hq, group, k, prefix, max_ctx;
  float scale_log2;
  int rows_per_split, max_splits;
  float* part_o;
  float2* part_ml;
  void* out;
  int out_dtype;
  float* lse;
};

__host__ __device__ constexpr int attn_smem_bytes(int rows_per_split) {
  return kStages * kStageBytes + kQBytes + 4 * rows_per_split;
}

// 256-byte rows of 16 chunks; chunk c of row r lives at chunk c ^ (r & 7).
__device__ __forceinline__ int swz256(int row, int chunk) { return row * kRowBytes + ((chunk ^ (row & 7)) << 4); }

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

__global__ void __launch_bounds__(kAttnThreads, 2) sparse_attn_kernel(const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* q_s = smem + kStages * kStageBytes;
  int* row_off = reinterpret_cast<int*>(q_s + kQBytes);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.y, qi = blockIdx.z;
  const int G = p.group;
  const int seq = p.mode == 0 ? qi : p.seq;
  const int pos = p.mode == 0 ? min(__ldg(p.ctx + qi), p.max_ctx) - 1 : p.pos0 + qi;
  const int n_pre = max(0, min(p.prefix, pos + 1));
  const int ns = min(max(__ldg(p.nsel + qi), 0), p.k);
  const int R = n_pre + ns;
  const int r0 = split * p.rows_per_split;
  const int nrows = min(R, r0 + p.rows_per_split) - r0;
  const size_t head0 = (size_t)qi * p.hq + (size_t)g * G;  // first query head of this KV head

  if (nrows <= 0) {  // empty split: neutral partial for the combine pass
    if (p.max_splits > 1 && tid < G)
      p.part_ml[(head0 + tid) * p.max_splits + split] = make_float2(-INFINITY, 0.f);
    return;
  }

  // Row r of this split -> row index of the K/V caches ((block * Hkv + g) * 64 + t % 64).
  const int pos_limit = p.max_blocks * kBlock;
  for (int r = tid; r < nrows; r += kAttnThreads) {
    const int rr = r0 + r;
    const int t = rr < n_pre ? rr : __ldg(p.idx + (size_t)qi * p.k + (rr - n_pre));
    int blk = 0;
    if (t >= 0 && t < pos_limit)
      blk = load_block(p.bt, seq, p.max_blocks, t >> 6, p.num_blocks, &g_status);
    else
      set_status(&g_status, kStBadBlock);
    row_off[r] = (blk * p.hkv + g) * kBlock + (t & 63);
  }
  // Q rows of the G heads, zero padded to 16 rows.
  for (int c = tid; c < 16 * 16; c += kAttnThreads) {
    const int row = c >> 4, ch = c & 15;
    const __nv_bfloat16* src = p.q + (head0 + min(row, G - 1)) * kHeadDim + ch * 8;
    cp_async16(q_s + swz256(row, ch), src, row < G ? 16u : 0u);
  }
  __syncthreads();  // row_off visible to every thread

  const int ntiles = (nrows + kTileRows - 1) / kTileRows;
  auto load_tile = [&](int tile) {
    uint8_t* sk = smem + (tile % kStages) * kStageBytes;
    uint8_t* sv = sk + kTileBytes;
    for (int c = tid; c < kTileRows * 16; c += kAttnThreads) {
      const int row = c >> 4, ch = c & 15;
      const int r = tile * kTileRows + row;
      const bool valid = r < nrows;
      const size_t off = valid ? (size_t)row_off[r] * kHeadDim + ch * 8 : 0;
      cp_async16(sk + swz256(row, ch), p.kc + off, valid ? 16u : 0u);
      cp_async16(sv + swz256(row, ch), p.vc + off, valid ? 16u : 0u);
    }
  };
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) load_tile(s);
    cp_async_commit();
  }

  uint32_t qf[8][4];
  float oacc[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int mi = lane >> 3, rr8 = lane & 7;
  const int wrow = warp * 16;

  for (int tile = 0; tile < ntiles; ++tile) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    if (tile == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        ldsm_x4(smem_u32(q_s + swz256((mi & 1) * 8 + rr8, 2 * ks + (mi >> 1))), qf[ks][0], qf[ks][1], qf[ks][2],
                qf[ks][3]);
    }
    if (tile + kStages - 1 < ntiles) load_tile(tile + kStages - 1);
    cp_async_commit();

    const uint8_t* sk = smem + (tile % kStages) * kStageBytes;
    const uint8_t* sv = sk + kTileBytes;

    // S = Q K^T for this warp's 16 rows (two n8 tiles).
    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(smem_u32(sk + swz256(wrow + (mi >> 1) * 8 + rr8, 2 * ks + (mi & 1))), b0, b1, b2, b3);
      mma_bf16_16816(sacc[0], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
      mma_bf16_16816(sacc[1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
    }

    // Online softmax (base 2).  Elements 0,1 belong to head row lane/4, 2,3 to lane/4 + 8.
    const int base_r = tile * kTileRows + wrow + (lane & 3) * 2;
    float x[2][4];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool valid = base_r + j * 8 + (e & 1) < nrows;
        x[j][e] = valid ? sacc[j][e] * p.scale_log2 : -INFINITY;
        if (e < 2) mx0 = fmaxf(mx0, x[j][e]);
        else mx1 = fmaxf(mx1, x[j][e]);
      }
    mx0 = quad_max(mx0);
    mx1 = quad_max(mx1);
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
    const float a0 = exp2f(m0 - ms0), a1 = exp2f(m1 - ms1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      x[j][0] = exp2f(x[j][0] - ms0);
      x[j][1] = exp2f(x[j][1] - ms0);
      x[j][2] = exp2f(x[j][2] - ms1);
      x[j][3] = exp2f(x[j][3] - ms1);
      ps0 += x[j][0] + x[j][1];
      ps1 += x[j][2] + x[j][3];
    }
    l0 = l0 * a0 + ps0;
    l1 = l1 * a1 + ps1;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      oacc[n][0] *= a0;
      oacc[n][1] *= a0;
      oacc[n][2] *= a1;
      oacc[n][3] *= a1;
    }
    const uint32_t pa0 = pack_bf16x2(x[0][0], x[0][1]), pa1 = pack_bf16x2(x[0][2], x[0][3]);
    const uint32_t pa2 = pack_bf16x2(x[1][0], x[1][1]), pa3 = pack_bf16x2(x[1][2], x[1][3]);

    // O += P V over the warp's 16 rows.
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(smem_u32(sv + swz256(wrow + (mi & 1) * 8 + rr8, 2 * np + (mi >> 1))), b0, b1, b2, b3);
      mma_bf16_16816(oacc[2 * np], pa0, pa1, pa2, pa3, b0, b1);
      mma_bf16_16816(oacc[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // stage memory is free from here on

  // Merge the four warps: (m, l, O) per head row through shared memory.
  l0 = quad_sum(l0);
  l1 = quad_sum(l1);
  float* s_o = reinterpret_cast<float*>(smem);               // [4][16][128]
  float* s_ml = reinterpret_cast<float*>(smem + 4 * 16 * 128 * 4);  // [4][16][2]
  const int h0 = lane >> 2, h1 = h0 + 8;
  if ((lane & 3) == 0) {
    s_ml[(warp * 16 + h0) * 2] = m0;
    s_ml[(warp * 16 + h0) * 2 + 1] = l0;
    s_ml[(warp * 16 + h1) * 2] = m1;
    s_ml[(warp * 16 + h1) * 2 + 1] = l1;
  }
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int d = n * 8 + (lane & 3) * 2;
    *reinterpret_cast<float2*>(s_o + (warp * 16 + h0) * 128 + d) = make_float2(oacc[n][0], oacc[n][1]);
    *reinterpret_cast<float2*>(s_o + (warp * 16 + h1) * 128 + d) = make_float2(oacc[n][2], oacc[n][3]);
  }
  __syncthreads();
  const int d = tid;  // one output column per thread
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, s_ml[(w * 16 + h) * 2]);
    float O = 0.f, Lsum = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw = s_ml[(w * 16 + h) * 2];
      if (mw == -INFINITY) continue;
      const float sc = exp2f(mw - M);
      O += sc * s_o[(w * 16 + h) * 128 + d];
      Lsum += sc * s_ml[(w * 16 + h) * 2 + 1];
    }
    const size_t head = head0 + h;
    if (p.max_splits == 1) {
      const float v = O / Lsum;
      if (p.out_dtype == 0)
        reinterpret_cast<__nv_bfloat16*>(p.out)[head * kHeadDim + d] = __float2bfloat16_rn(v);
      else
        reinterpret_cast<float*>(p.out)[head * kHeadDim + d] = v;
      if (d == 0 && p.lse) p.lse[head] = (M + log2f(Lsum)) * 0.69314718055994531f;
    } else {
      p.part_o[(head * p.max_splits + split) * kHeadDim + d] = O;
      if (d == 0) p.part_ml[head * p.max_splits + split] = make_float2(M, Lsum);
    }
  }
}

// Merge the splits of one (query, head): out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
__global__ void __launch_bounds__(kHeadDim) attn_combine_kernel(const float* __restrict__ part_o,
                                                               const float2* __restrict__ part_ml, int max_splits,
                                                               void* out, int out_dtype, float* lse) {
  const size_t head = blockIdx.x;
  const int d = threadIdx.x;
  const float2* ml = part_ml + head * max_splits;
  float M = -INFINITY;
  for (int s = 0; s < max_splits; ++s) M = fmaxf(M, ml[s].x);
  float O = 0.f, L = 0.f;
  for (int s = 0; s < max_splits; ++s) {
    const float2 v = ml[s];
    if (v.x == -INFINITY) continue;
    const float sc = exp2f(v.x - M);
    O += sc * part_o[(head * max_splits + s) * kHeadDim + d];
    L += sc * v.y;
  }
  const float r = O / L;
  if (out_dtype == 0)
    reinterpret_cast<__nv_bfloat16*>(out)[head * kHeadDim + d] = __float2bfloat16_rn(r);
  else
    reinterpret_cast<float*>(out)[head * kHeadDim + d] = r;
  if (d == 0 && lse) lse[head] = (M + log2f(L)) * 0.69314718055994531f;
}

}  // namespace

void attn_split_plan(int pairs, int rows_max, int mode, int* rows_per_split, int* max_splits) {
  auto up64 = [](int x) { return (x + 63) / 64 * 64; };
  if (mode == 1) {  // prefill: thousands of (query, KV head) CTAs already; no split unless rows exceed the cap
    const int n = (rows_max + kMaxRowsPerSplit - 1) / kMaxRowsPerSplit;
    *rows_per_split = up64((rows_max + n - 1) / n);
    *max_splits = n;
    return;
  }
  const int target = 1216;  // 8 CTAs per SM worth of work over 152 SMs
  const int splits = (target + pairs - 1) / pairs;
  int rps = up64((rows_max + splits - 1) / splits);
  rps = rps < 64 ? 64 : (rps > kMaxRowsPerSplit ? kMaxRowsPerSplit : rps);
  *rows_per_split = rps;
  *max_splits = (rows_max + rps - 1) / rps;
}

cudaError_t setup_attn_kernels() {
  return cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              attn_smem_bytes(kMaxRowsPerSplit));
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
  p.rows_per_split = a.rows_per_split;
  p.max_splits = a.max_splits;
  p.part_o = a.ws.part_o;
  p.part_ml = a.ws.part_ml;
  p.out = a.out;
  p.out_dtype = a.out_dtype;
  p.lse = a.lse;
  dim3 grid(a.max_splits, a.kv.hkv, a.qs.n_q);
  sparse_attn_kernel<<<grid, kAttnThreads, attn_smem_bytes(a.rows_per_split), st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.max_splits == 1) return e;
  attn_combine_kernel<<<(unsigned)((size_t)a.qs.n_q * a.hq), kHeadDim, 0, st>>>(a.ws.part_o, a.ws.part_ml,
                                                                                  a.max_splits, a.out,
                                                                                  a.out_dtype, a.lse);
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
