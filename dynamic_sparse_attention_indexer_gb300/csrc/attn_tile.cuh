// GQA attention over staged rows for one KV head (§2.3): the per-warp math that
// the sparse attention kernels run on each tile of attended rows.
//
// A consumer warp owns the G query heads of one KV head.  For each 16-row chunk
// of the tile it computes S^T = K Q^T and O^T = V^T P^T on the tensor cores
// (mma.sync m16n8k16 bf16, fp32 accumulate), so the attended rows fill the
// 16-row M side and the query heads the 8-wide N side (NT tiles of 8 heads).
// P enters the second product as two bf16 terms, hi + lo (lo the rounding
// residual of hi), so it keeps about 16 mantissa bits; P^T reaches its operand
// layout through movmatrix.  The online softmax runs per head column in base 2,
// reduced over the row groups with warp shuffles, and O is rescaled only when
// a running max moved.
//
// Shared-memory layout of a staged tile: K rows then V rows, `pitch` bytes per
// row (a multiple of 16 plus 16, so that ldmatrix is conflict-free), the 128
// dims of this KV head at the byte offset the caller passes in sk / sv.
#pragma once

#include "common.cuh"

namespace dsa {

// The two bf16 halves of a packed pair, as floats (exact).
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t transpose8x8(uint32_t v) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(v));
  return d;
}

// Running state of one consumer warp: Q fragments of its heads, the
// unnormalised output O^T (d in 8 tiles of 16, NT head tiles, C layout) and
// per head column the running max (log2 units) and the lane's share of the sum.
template <int NT>
struct HeadState {
  uint32_t qb[NT][8][2];
  float o[8][NT][4];
  float m[NT][2], l[NT][2];
};

// Q fragments (B operand, heads as N) of KV head g's G heads from the query's
// staged Q (all heads, 256 bytes each).  Heads past G repeat head G - 1; their
// columns are never written out.
template <int NT>
__device__ __forceinline__ void load_q(HeadState<NT>& st, const uint8_t* s_q, int g, int G, int lane) {
  const int mi = lane >> 3, rr8 = lane & 7;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int h = g * G + min(j * 8 + rr8, G - 1);
#pragma unroll
    for (int ks = 0; ks < 8; ks += 2)
      ldsm_x4(smem_u32(s_q + h * (kHeadDim * 2) + (2 * ks + mi) * 16), st.qb[j][ks][0], st.qb[j][ks][1],
              st.qb[j][ks + 1][0], st.qb[j][ks + 1][1]);
  }
}

template <int NT>
__device__ __forceinline__ void reset_state(HeadState<NT>& st) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j) st.o[i][j][0] = st.o[i][j][1] = st.o[i][j][2] = st.o[i][j][3] = 0.f;
#pragma unroll
  for (int j = 0; j < NT; ++j) st.m[j][0] = st.m[j][1] = -INFINITY, st.l[j][0] = st.l[j][1] = 0.f;
}

// Adds the first `nvalid` staged rows (K at sk, V at sv) to the state.  Rows
// from nvalid up to the next multiple of 16 must hold finite values (their
// weights are zero).
template <int NT>
__device__ __forceinline__ void attend_rows(HeadState<NT>& st, const uint8_t* sk, const uint8_t* sv, int pitch,
                                            int nvalid, float scale_log2, int lane) {
  const int mi = lane >> 3, rr8 = lane & 7;
  for (int c16 = 0; c16 < nvalid; c16 += 16) {
    // S^T = K Q^T: 16 rows x 8 NT heads.
    float sacc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(smem_u32(sk + (c16 + (mi & 1) * 8 + rr8) * pitch + (2 * ks + (mi >> 1)) * 16), a0, a1, a2, a3);
#pragma unroll
      for (int j = 0; j < NT; ++j) mma_bf16_16816(sacc[j], a0, a1, a2, a3, st.qb[j][ks][0], st.qb[j][ks][1]);
    }
    // Online softmax per head column (base 2), reduced over the 8 row groups.
    const int ra = c16 + (lane >> 2);  // tile rows of elements 0,1 (ra) and 2,3 (ra + 8)
    const bool va = ra < nvalid, vb = ra + 8 < nvalid;
    float alpha[NT][2], ms[NT][2];
    bool moved = false;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      sacc[j][0] = va ? sacc[j][0] * scale_log2 : -INFINITY;
      sacc[j][1] = va ? sacc[j][1] * scale_log2 : -INFINITY;
      sacc[j][2] = vb ? sacc[j][2] * scale_log2 : -INFINITY;
      sacc[j][3] = vb ? sacc[j][3] * scale_log2 : -INFINITY;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = fmaxf(sacc[j][e], sacc[j][e + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(st.m[j][e], mx);
        ms[j][e] = mn == -INFINITY ? 0.f : mn;
        alpha[j][e] = exp2f(st.m[j][e] - ms[j][e]);
        moved |= mn != st.m[j][e];
        st.m[j][e] = mn;
      }
    }
    if (__any_sync(0xffffffffu, moved)) {  // rescale only when a running max moved
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          st.o[i][j][0] *= alpha[j][0];
          st.o[i][j][1] *= alpha[j][1];
          st.o[i][j][2] *= alpha[j][0];
          st.o[i][j][3] *= alpha[j][1];
        }
#pragma unroll
      for (int j = 0; j < NT; ++j) st.l[j][0] *= alpha[j][0], st.l[j][1] *= alpha[j][1];
    }
    // P in two bf16 terms, P = hi + lo (lo = the rounding residual of hi), so
    // the P.V product carries about 16 mantissa bits of P instead of 8.
    uint32_t pb[NT][2], pl[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float p0 = exp2f(sacc[j][0] - ms[j][0]), p1 = exp2f(sacc[j][1] - ms[j][1]);
      const float p2 = exp2f(sacc[j][2] - ms[j][0]), p3 = exp2f(sacc[j][3] - ms[j][1]);
      st.l[j][0] += p0 + p2;
      st.l[j][1] += p1 + p3;
      const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
      const uint32_t r01 = pack_bf16x2(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
      const uint32_t r23 = pack_bf16x2(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
      // P^T rows (attended rows) x head columns -> B fragments (rows as K).
      pb[j][0] = transpose8x8(h01);
      pb[j][1] = transpose8x8(h23);
      pl[j][0] = transpose8x8(r01);
      pl[j][1] = transpose8x8(r23);
    }
    // O^T += V^T P^T: d in 8 tiles of 16.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(smem_u32(sv + (c16 + (mi >> 1) * 8 + rr8) * pitch + (2 * i + (mi & 1)) * 16), a0, a1, a2, a3);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        mma_bf16_16816(st.o[i][j], a0, a1, a2, a3, pb[j][0], pb[j][1]);
        mma_bf16_16816(st.o[i][j], a0, a1, a2, a3, pl[j][0], pl[j][1]);
      }
    }
  }
}

// Segment end: the total weight per head column over the eight row groups
// (every lane of a column group then holds it).
template <int NT>
__device__ __forceinline__ void total_sums(HeadState<NT>& st) {
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = st.l[j][e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      st.l[j][e] = v;
    }
}

// Stores the state of head column (j, e) of this lane as a partial: (max, sum)
// at *ml (lanes 0-3 only) and the unnormalised output at o_dst[0 .. 128).
template <int NT>
__device__ __forceinline__ void store_partial(const HeadState<NT>& st, int j, int e, int lane, float2* ml,
                                              float* o_dst) {
  if (lane < 4) *ml = make_float2(st.m[j][e], st.l[j][e]);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int d = 16 * i + (lane >> 2);
    o_dst[d] = st.o[i][j][e];
    o_dst[d + 8] = st.o[i][j][e + 2];
  }
}

}  // namespace dsa
