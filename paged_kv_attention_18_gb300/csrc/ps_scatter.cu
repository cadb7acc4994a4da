// Slot mapping and KV scatter (reshape_and_cache) kernels.
//
// The slot of a token at position pos of a sequence is
//     block_table[pos // 16] * 16 + pos % 16
// (PageServe, section 01 "Scheduler loop", closing paragraph; section 03 "Paged KV
// cache", attention_wrapper.py code box). A step's n query tokens of a sequence are
// the last n positions of its context (PageServe section 01: every step computes the
// tokens not yet computed). The scatter writes each token's K and V rows into the
// pool [blocks, 16, H_kv, D] at its slot (PageServe section 01 "Execute": the
// backend writes K/V into the pool).
#include "ps_common.cuh"
#include "ps_launch.h"
#include "ps_scatter.cuh"

namespace ps {

// One thread per packed token: find its sequence, its position, then its slot.
__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables, int max_blocks,
                                    const int32_t* __restrict__ seq_lens,
                                    const int32_t* __restrict__ qsl, int B, int T,
                                    int num_blocks, int32_t* __restrict__ slots, int* err) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  // largest b in [0, B) with qsl[b] <= t (empty sequences share their start with the next)
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int start = __ldg(qsl + b), end = __ldg(qsl + b + 1);
  const int n = end - start, L = __ldg(seq_lens + b);
  const int pos = L - n + (t - start);
  if (t < start || t >= end || n > L || pos < 0 || pos / kBlockSize >= max_blocks) {
    record_error(err, kDevBadSequence);
    slots[t] = -1;
    return;
  }
  const int blk = __ldg(block_tables + static_cast<int64_t>(b) * max_blocks + pos / kBlockSize);
  if (blk < 0 || blk >= num_blocks) {
    record_error(err, kDevBadBlockId);
    slots[t] = -1;
    return;
  }
  slots[t] = blk * kBlockSize + pos % kBlockSize;
}

// Each thread moves one 16-byte chunk of one token's K row and the same chunk of its V
// row. Consecutive threads take consecutive chunks of a row, so loads and stores are
// fully coalesced 16-byte accesses.
__global__ void reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                         const int32_t* __restrict__ slots,
                                         uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                         int T, int row_vecs, int64_t num_slots, int* err) {
  pdl_launch_dependents();
  pdl_wait();  // the slots may come from the kernel before this one
  const int64_t total = static_cast<int64_t>(T) * row_vecs;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += stride) {
    const int t = static_cast<int>(i / row_vecs);
    const int c = static_cast<int>(i - static_cast<int64_t>(t) * row_vecs);
    const int s = __ldg(slots + t);
    if (s < 0) continue;  // padding token: nothing to cache
    if (s >= num_slots) {
      record_error(err, kDevBadSlot);
      continue;
    }
    const uint4 kk = __ldcs(k + i);
    const uint4 vv = __ldcs(v + i);
    const int64_t dst = static_cast<int64_t>(s) * row_vecs + c;
    k_pool[dst] = kk;
    v_pool[dst] = vv;
  }
}

// The step's KV scatter with its slot mapping, first in the launch chain of the tile
// kernel's direct mode: one warp per packed token finds the token's sequence and position
// (the last n positions of the context are the step's tokens), reads its block-table
// entry, writes the slot and copies the token's K and V rows there in 16-byte chunks. It
// lets the tile kernel start as soon as the previous work on the stream is done; the tile
// kernel's K/V producers wait for this kernel before their first copy from the pools.
__global__ void __launch_bounds__(256) step_scatter_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v,
    const int32_t* __restrict__ block_tables, int max_blocks, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ qsl, int B, int T, int row_vecs, int num_blocks,
    int32_t* __restrict__ slots, uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int* err) {
  pdl_wait();               // the previous kernel on the stream has finished
  pdl_launch_dependents();  // the planner may start now
  scatter_step_tokens(k, v, block_tables, max_blocks, seq_lens, qsl, B, T, row_vecs, num_blocks,
                      slots, k_pool, v_pool, err, (blockIdx.x * blockDim.x + threadIdx.x) >> 5,
                      gridDim.x * (blockDim.x >> 5));
}

cudaError_t launch_step_scatter(const void* k, const void* v, const int32_t* block_tables,
                                int max_blocks, const int32_t* seq_lens, const int32_t* qsl, int B,
                                int T, int H_kv, int D, int num_blocks, int32_t* slots,
                                void* k_pool, void* v_pool, int* err, int num_sms,
                                cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int threads = 256, per_cta = threads / 32;
  int64_t blocks = (static_cast<int64_t>(T) + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return launch_kernel(step_scatter_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
                       stream, true, static_cast<const uint4*>(k), static_cast<const uint4*>(v),
                       block_tables, max_blocks, seq_lens, qsl, B, T, H_kv * D / 8, num_blocks,
                       slots, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), err);
}

// The host step's copies in one launch: each CTA's threads walk the segments' 16-byte
// chunks (4-byte words for a segment whose addresses or size are not 16-byte multiples),
// reading or writing the page-locked host buffers directly. Launched after the kernel
// that writes its sources, it waits for that kernel first.
__global__ void __launch_bounds__(256) gather_in_kernel(const CopySegments segs) {
  pdl_wait();
  pdl_launch_dependents();
  copy_segments(segs, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                static_cast<int64_t>(gridDim.x) * blockDim.x);
}

cudaError_t launch_gather_in(const CopySegments& segs, int num_sms, cudaStream_t stream,
                             bool pdl) {
  int64_t chunks = 0;
  for (int k = 0; k < segs.n; ++k) chunks += segs.seg[k].bytes / 16 + 1;
  int64_t blocks = (chunks + 255) / 256;
  if (blocks > 2 * static_cast<int64_t>(num_sms)) blocks = 2 * static_cast<int64_t>(num_sms);
  if (blocks < 1) blocks = 1;
  return launch_kernel(gather_in_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                       pdl, segs);
}

cudaError_t launch_slot_mapping(const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                const int32_t* qsl, int B, int T, int num_blocks, int32_t* slots,
                                int* err, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int threads = 256;
  const int grid = (T + threads - 1) / threads;
  slot_mapping_kernel<<<grid, threads, 0, stream>>>(block_tables, max_blocks, seq_lens, qsl, B, T,
                                                    num_blocks, slots, err);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void* k, const void* v, const int32_t* slots,
                                     void* k_pool, void* v_pool, int T, int H_kv, int D,
                                     int num_blocks, int* err, int num_sms,
                                     cudaStream_t stream, bool pdl) {
  if (T == 0) return cudaSuccess;
  const int row_vecs = H_kv * D / 8;  // 16-byte chunks per token row
  const int64_t total = static_cast<int64_t>(T) * row_vecs;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return launch_kernel(reshape_and_cache_kernel, dim3(static_cast<unsigned>(blocks)),
                       dim3(threads), 0, stream, pdl, static_cast<const uint4*>(k),
                       static_cast<const uint4*>(v), slots, static_cast<uint4*>(k_pool),
                       static_cast<uint4*>(v_pool), T, row_vecs,
                       static_cast<int64_t>(num_blocks) * kBlockSize, err);
}

}  // namespace ps
