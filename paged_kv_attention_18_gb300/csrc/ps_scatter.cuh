// The step's KV scatter with its slot mapping, as a device function shared by the
// scatter kernel and the planner's scatter CTAs.
//
// The slot of the token at position pos of a sequence is block_table[pos // 16] * 16 +
// pos % 16, and a step's n query tokens of a sequence are the last n positions of its
// context (PageServe, section 01 "Scheduler loop"; section 03 "Paged KV cache").
#pragma once
#include "ps_common.cuh"
#include "ps_launch.h"

namespace ps {

// Copies of whole buffers by a set of threads (thread index tid of nth): 16-byte words
// where both addresses and the size allow, 4-byte words otherwise. Used by the gather
// kernel and by the planner's copy CTAs; either side may be page-locked host memory seen
// through its device address.
__device__ __forceinline__ void copy_segments(const CopySegments& segs, int64_t tid, int64_t nth) {
  for (int k = 0; k < segs.n; ++k) {
    const CopySegment& c = segs.seg[k];
    const bool wide = ((reinterpret_cast<uintptr_t>(c.dst) | reinterpret_cast<uintptr_t>(c.src) |
                        static_cast<uintptr_t>(c.bytes)) & 15u) == 0;
    if (wide) {
      const uint4* src = static_cast<const uint4*>(c.src);
      uint4* dst = static_cast<uint4*>(c.dst);
      for (int64_t i = tid; i < c.bytes / 16; i += nth) dst[i] = src[i];
    } else {
      const uint32_t* src = static_cast<const uint32_t*>(c.src);
      uint32_t* dst = static_cast<uint32_t*>(c.dst);
      for (int64_t i = tid; i < c.bytes / 4; i += nth) dst[i] = src[i];
    }
  }
}

// Sequence of packed token t: the largest b in [0, B) with qsl[b] <= t (empty sequences
// share their start with the next one), found by the whole warp in 32-way rounds, so a
// batch of B sequences takes ceil(log32(B)) rounds of loads instead of log2(B).
__device__ __forceinline__ int warp_find_seq(const int32_t* __restrict__ qsl, int B, int t,
                                             int lane) {
  int lo = 0, n = B;  // the answer lies in [lo, lo + n); qsl[lo] <= t throughout
  while (n > 1) {
    const int step = (n + 31) / 32;
    const int idx = lo + lane * step;
    const bool le = idx < lo + n && __ldg(qsl + idx) <= t;
    const unsigned m = __ballot_sync(0xffffffffu, le) | 1u;
    const int k = 31 - __clz(m);
    const int end = lo + n;
    lo += k * step;
    n = min(step, end - lo);
  }
  return lo;
}

// Warps first_warp, first_warp + nwarps, ... each take one packed token: find its
// sequence and position, read its block-table entry, write its slot and copy its K and V
// rows (row_vecs 16-byte chunks each) to that slot of the pools.
__device__ __forceinline__ void scatter_step_tokens(
    const uint4* __restrict__ k, const uint4* __restrict__ v,
    const int32_t* __restrict__ block_tables, int max_blocks, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ qsl, int B, int T, int row_vecs, int num_blocks,
    int32_t* __restrict__ slots, uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int* err,
    int first_warp, int nwarps) {
  const int lane = threadIdx.x & 31;
  for (int t = first_warp; t < T; t += nwarps) {
    const int b = warp_find_seq(qsl, B, t, lane);
    int slot = -1;
    if (lane == 0) {
      const int start = __ldg(qsl + b), end = __ldg(qsl + b + 1);
      const int n = end - start, L = __ldg(seq_lens + b);
      const int pos = L - n + (t - start);
      if (t < start || t >= end || n > L || pos < 0 || pos / kBlockSize >= max_blocks) {
        record_error(err, kDevBadSequence);
      } else {
        const int blk =
            __ldg(block_tables + static_cast<int64_t>(b) * max_blocks + pos / kBlockSize);
        if (blk < 0 || blk >= num_blocks) record_error(err, kDevBadBlockId);
        else slot = blk * kBlockSize + pos % kBlockSize;
      }
      slots[t] = slot;
    }
    slot = __shfl_sync(0xffffffffu, slot, 0);
    if (slot < 0) continue;
    const int64_t src = static_cast<int64_t>(t) * row_vecs;
    const int64_t dst = static_cast<int64_t>(slot) * row_vecs;
    for (int c = lane; c < row_vecs; c += 32) {
      const uint4 kk = __ldcs(k + src + c);
      const uint4 vv = __ldcs(v + src + c);
      k_pool[dst + c] = kk;
      v_pool[dst + c] = vv;
    }
  }
}

}  // namespace ps
