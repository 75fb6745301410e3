// Prefill: attention of every query to the forced vision prefix, computed once
// per tile of queries instead of once per query (§2.4: the prefix is always
// attended in full; §2.3: the prefill path is the compute-heavy one).
//
// In prefill every query of the sequence attends the same prefix rows
// [0, min(P, pos + 1)), so for a tile of queries the prefix part is a dense,
// causally masked attention: S = Q K^T over (query, head) rows x prefix keys,
// then P V.  One CTA takes 128 (query, head) rows of one KV head (128 / G
// queries x the G heads of the group) and streams the prefix keys in chunks of
// 64 (one cache block each), double-buffered with cp.async; eight warps of
// 16 rows run the two products on mma.sync m16n8k16 bf16 with fp32
// accumulation, the online softmax in base 2, and P entered as hi + lo bf16
// terms like the sparse kernel.  The result per (query, head) is a partial
// state (running max in log2 units, sum of weights, unnormalised output in
// fp32) that the sparse kernel takes as its starting state for the query, so
// the selected rows then only add to it.  The same prefix rows thus cross L2
// once per 128 rows instead of once per query.
#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

__device__ int g_status;

constexpr int kPreRows = 128;                      // (query, head) rows per CTA
constexpr int kPreWarps = kPreRows / 16;           // 8
constexpr int kPreThreads = 32 * kPreWarps;        // 256
constexpr int kPreKeys = kBlock;                   // keys per chunk: one cache block
constexpr int kPrePitch = kHeadDim * 2 + 16;       // padded shared row (conflict-free ldmatrix)
constexpr int kPreQBytes = kPreRows * kPrePitch;   // 34,816
constexpr int kPreKVBytes = kPreKeys * kPrePitch;  // 17,408 (K or V of one chunk)
constexpr int kPreSmem = kPreQBytes + 4 * kPreKVBytes;

struct PrefixParams {
  const __nv_bfloat16* q;   // [n_q][hq][128]
  const __nv_bfloat16* kc;  // [num_blocks][64][hkv][128]
  const __nv_bfloat16* vc;
  const int32_t* bt;
  int seq, pos0, n_q, hq, hkv, group, prefix, max_blocks, num_blocks, row_stride;
  float scale_log2;
  float2* pre_ml;  // [n_q][hq] (max in log2 units, sum of weights)
  float* pre_o;    // [n_q][hq][128] unnormalised output
};

__global__ void __launch_bounds__(kPreThreads) prefix_attn_kernel(const PrefixParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* s_q = smem;
  uint8_t* s_kv = smem + kPreQBytes;  // [2 buffers][K, V][64 rows][pitch]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y;                // KV head
  const int G = p.group;
  const int qt = kPreRows / G;             // queries per CTA
  const int q0 = blockIdx.x * qt;          // first query of the tile
  const int nq = min(qt, p.n_q - q0);
  // Keys this tile needs: the prefix part of its last query's causal range.
  const int n_keys = min(p.prefix, p.pos0 + q0 + nq);
  const int n_chunks = (n_keys + kPreKeys - 1) / kPreKeys;
  pdl_wait();
  pdl_trigger();

  // Q rows: row r is (query q0 + r / G, head g * G + r % G); rows past the
  // last query are zero.
  for (int c = tid; c < kPreRows * (kHeadDim / 8); c += kPreThreads) {
    const int r = c / (kHeadDim / 8), ch = c % (kHeadDim / 8);
    const int qi = r / G;
    const __nv_bfloat16* src = p.q + ((size_t)(q0 + min(qi, nq - 1)) * p.hq + g * G + r % G) * kHeadDim + ch * 8;
    cp_async16(s_q + r * kPrePitch + ch * 16, src, qi < nq ? 16u : 0u);
  }
  // One chunk of K and V (rows past the prefix are zero, so that masked
  // weights multiply finite values).
  auto load_chunk = [&](int c, int buf) {
    int blk = __ldg(p.bt + (size_t)p.seq * p.max_blocks + c);
    if ((unsigned)blk >= (unsigned)p.num_blocks) {
      set_status(&g_status, kStBadBlock);
      blk = 0;
    }
    uint8_t* dk = s_kv + buf * 2 * kPreKVBytes;
    uint8_t* dv = dk + kPreKVBytes;
    for (int e = tid; e < kPreKeys * (kHeadDim / 8); e += kPreThreads) {
      const int j = e / (kHeadDim / 8), ch = e % (kHeadDim / 8);
      const bool ok = c * kPreKeys + j < p.prefix;
      const size_t off = ((size_t)blk * kBlock + j) * p.row_stride + (size_t)g * kHeadDim + ch * 8;
      cp_async16(dk + j * kPrePitch + ch * 16, p.kc + off, ok ? 16u : 0u);
      cp_async16(dv + j * kPrePitch + ch * 16, p.vc + off, ok ? 16u : 0u);
    }
  };
  if (n_chunks > 0) load_chunk(0, 0);
  cp_async_commit();

  // This lane's rows of the warp's 16: ra = warp * 16 + lane / 4 and ra + 8,
  // each with its own causal key limit.
  const int ra = warp * 16 + (lane >> 2), rb = ra + 8;
  const int lim_a = min(p.prefix, p.pos0 + q0 + min(ra / G, nq - 1) + 1);
  const int lim_b = min(p.prefix, p.pos0 + q0 + min(rb / G, nq - 1) + 1);
  uint32_t qa[8][4];  // A fragments of Q, 8 steps of 16 columns
  float o[16][4];     // 16 column tiles of 8 (d), C layout
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int c = 0; c < n_chunks; ++c) {
    if (c + 1 < n_chunks) load_chunk(c + 1, (c + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();  // chunk c (and Q) landed for every thread
    if (c == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int col = ks * 16 + ((lane >> 4) & 1) * 8;
        ldsm_x4(smem_u32(s_q + row * kPrePitch + col * 2), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
      }
    }
    const uint8_t* sk = s_kv + (c & 1) * 2 * kPreKVBytes;
    const uint8_t* sv = sk + kPreKVBytes;
    // S = Q K^T: 16 rows x 64 keys in 8 tiles of 8.
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int np = 0; np < 4; ++np) {  // key tiles 2 np, 2 np + 1
        uint32_t b0, b1, b2, b3;
        const int key = np * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int col = ks * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4(smem_u32(sk + key * kPrePitch + col * 2), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
    // Causal mask, scale, online softmax per row (4 lanes share a row).
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = c * kPreKeys + nt * 8 + 2 * (lane & 3) + (e & 1);
        const bool ok = key < (e < 2 ? lim_a : lim_b);
        s[nt][e] = ok ? s[nt][e] * p.scale_log2 : -INFINITY;
        mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
      }
    float ms[2], alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float mn = fmaxf(m[h], mx[h]);
      ms[h] = mn == -INFINITY ? 0.f : mn;
      alpha[h] = exp2f(m[h] - ms[h]);
      m[h] = mn;
      l[h] *= alpha[h];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }
    // P in two bf16 terms (hi + rounding residual), as A fragments: key tiles
    // 2t and 2t + 1 form the 16 keys of step t.
    uint32_t ph[4][4], pl[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float* sc = s[2 * t + half];
        const float p0 = exp2f(sc[0] - ms[0]), p1 = exp2f(sc[1] - ms[0]);
        const float p2 = exp2f(sc[2] - ms[1]), p3 = exp2f(sc[3] - ms[1]);
        l[0] += p0 + p1;
        l[1] += p2 + p3;
        const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
        const float r0 = p0 - __uint_as_float(h01 << 16), r1 = p1 - __uint_as_float(h01 & 0xffff0000u);
        const float r2 = p2 - __uint_as_float(h23 << 16), r3 = p3 - __uint_as_float(h23 & 0xffff0000u);
        ph[t][2 * half] = h01;       // a0 / a2: row lane / 4
        ph[t][2 * half + 1] = h23;   // a1 / a3: row lane / 4 + 8
        pl[t][2 * half] = pack_bf16x2(r0, r1);
        pl[t][2 * half + 1] = pack_bf16x2(r2, r3);
      }
    // O += P V: 16 keys per step, d in 16 tiles of 8.
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {  // d tiles 2 dp, 2 dp + 1
        uint32_t b0, b1, b2, b3;
        const int key = t * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int col = dp * 16 + ((lane >> 4) & 1) * 8;
        ldsm_x4_t(smem_u32(sv + key * kPrePitch + col * 2), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], ph[t][0], ph[t][1], ph[t][2], ph[t][3], b0, b1);
        mma_bf16_16816(o[2 * dp], pl[t][0], pl[t][1], pl[t][2], pl[t][3], b0, b1);
        mma_bf16_16816(o[2 * dp + 1], ph[t][0], ph[t][1], ph[t][2], ph[t][3], b2, b3);
        mma_bf16_16816(o[2 * dp + 1], pl[t][0], pl[t][1], pl[t][2], pl[t][3], b2, b3);
      }
    __syncthreads();  // every warp is done with buffer c & 1 before it is refilled
  }
  cp_async_wait<0>();

  // Row sums over the 4 lanes of a row; write the partial states.
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = h ? rb : ra;
    const int qi = r / G;
    if (qi >= nq) continue;
    const size_t head = (size_t)(q0 + qi) * p.hq + g * G + r % G;
    if ((lane & 3) == 0) p.pre_ml[head] = make_float2(m[h], l[h]);
    float* dst = p.pre_o + head * kHeadDim;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      *reinterpret_cast<float2*>(dst + i * 8 + 2 * (lane & 3)) = make_float2(o[i][2 * h], o[i][2 * h + 1]);
  }
}

}  // namespace

cudaError_t setup_prefix_kernels() {
  return cudaFuncSetAttribute(prefix_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPreSmem);
}

cudaError_t launch_prefix_attn(const KV& kv, const QS& qs, const void* q, int hq, int prefix, float scale,
                               float2* pre_ml, float* pre_o, cudaStream_t st) {
  PrefixParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kc = static_cast<const __nv_bfloat16*>(kv.k_cache);
  p.vc = static_cast<const __nv_bfloat16*>(kv.v_cache);
  p.bt = kv.block_table;
  p.seq = qs.seq;
  p.pos0 = qs.pos0;
  p.n_q = qs.n_q;
  p.hq = hq;
  p.hkv = kv.hkv;
  p.group = hq / kv.hkv;
  p.prefix = prefix;
  p.max_blocks = kv.max_blocks;
  p.num_blocks = kv.num_blocks;
  p.row_stride = kv.row_stride;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.pre_ml = pre_ml;
  p.pre_o = pre_o;
  const int qt = kPreRows / p.group;
  const dim3 grid((unsigned)((qs.n_q + qt - 1) / qt), (unsigned)kv.hkv);
  return launch_pdl(prefix_attn_kernel, grid, dim3(kPreThreads), kPreSmem, st, 1, p);
}

cudaError_t read_clear_status_prefix(int* code, cudaStream_t st) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v != 0) {
    if (*code == 0) *code = v;
    const int z = 0;
    e = cudaMemcpyToSymbolAsync(g_status, &z, sizeof(int), 0, cudaMemcpyHostToDevice, st);
  }
  return e;
}

}  // namespace dsa
