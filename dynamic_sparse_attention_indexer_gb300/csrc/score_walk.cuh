// The decode scoring walk (§2.1 index scores over §2.2 paged blocks): how the
// candidate blocks of all sequences are laid end to end and cut into one
// contiguous range per CTA, and how a range is walked in groups of up to
// kGroupBlocks consecutive blocks of one sequence.
#pragma once

#include "common.cuh"

namespace dsa {

constexpr int kGroupBlocks = 4;  // cache blocks per scoring stage (4 x 4 KB)

// Candidate blocks of every sequence and their prefix sums: seg_start[b] is the
// first flattened block of sequence b, seg_start[batch] the total.  Row b's
// context length is ctx[b / csplit] (csplit > 1: rows are (sequence, KV head)
// pairs of the per-head indexer).
__device__ __forceinline__ void candidate_blocks(const int32_t* __restrict__ ctx, int batch, int max_ctx, int prefix,
                                 int* seg_start, int* len, int* scratch, int csplit = 1) {
  int carry = 0;
  for (int base = 0; base < batch; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int nb = 0;
    if (b < batch) {
      const int L = min(__ldg(ctx + (csplit > 1 ? b / csplit : b)), max_ctx);
      len[b] = L;
      nb = L > prefix ? (L + kBlock - 1) / kBlock - prefix / kBlock : 0;
    }
    int tot;
    const int ex = block_exclusive_scan(nb, scratch, &tot);
    if (b < batch) seg_start[b] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) seg_start[batch] = carry;
  __syncthreads();
}

// The group sequence of a CTA range: groups of up to kGroupBlocks consecutive
// candidate blocks of one sequence.
struct GroupCursor {
  int f, f_end, b;
};
struct Group {
  int b, jb, count;  // sequence, block-table index of the first block, blocks
};
__device__ __forceinline__ bool next_group(GroupCursor& c, const int* seg_start, int jb_base, Group* g) {
  if (c.f >= c.f_end) return false;
  while (seg_start[c.b + 1] <= c.f) ++c.b;  // skip sequences without candidates
  g->b = c.b;
  g->jb = c.f - seg_start[c.b] + jb_base;
  g->count = min(kGroupBlocks, min(c.f_end, seg_start[c.b + 1]) - c.f);
  c.f += g->count;
  return true;
}

}  // namespace dsa
