// Whole-block copies between KV pools. Two uses on the pages:
//   - copy-on-write: a write into a block that several block tables share first copies the
//     block, so writers never corrupt shared readers (tinyserve "How it works"; the
//     "Highlights" table, paged KV-cache row);
//   - preemption by swapping: a preempted sequence's blocks move to a pinned host pool and
//     back when it resumes, losslessly (PageServe section 04 "Phase 9 · Preemption";
//     tinyserve "How it works", "Correctness & testing" table).
// A block is 16 rows x H_kv x D 16-bit values (K and V pools alike); the copy is bit-exact.
// Pools may live in device memory or in pinned host memory: the kernel reads and writes
// them through unified addressing, so a swap is one kernel over the host link.
#include "ps_common.cuh"
#include "ps_launch.h"

namespace ps {

namespace {

// One (pair, tensor) unit per CTA at a time: the CTA streams one block of K or of V. Each
// thread keeps four 16-byte chunks in flight; consecutive threads take consecutive chunks.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(const uint4* sk, const uint4* sv, int src_nb, uint4* dk, uint4* dv,
                       int dst_nb, const int32_t* __restrict__ src_ids,
                       const int32_t* __restrict__ dst_ids, int n, int vecs, int* err) {
  constexpr int kInFlight = 4;
  for (int u = blockIdx.x; u < 2 * n; u += gridDim.x) {
    const int pair = u >> 1, tensor = u & 1;
    const int s = src_ids[pair], d = dst_ids[pair];
    if (s < 0 || s >= src_nb || d < 0 || d >= dst_nb) {
      if (threadIdx.x == 0 && tensor == 0) record_error(err, kDevBadBlockId);
      continue;
    }
    const uint4* src = (tensor ? sv : sk) + static_cast<int64_t>(s) * vecs;
    uint4* dst = (tensor ? dv : dk) + static_cast<int64_t>(d) * vecs;
    for (int c = threadIdx.x; c < vecs; c += kInFlight * blockDim.x) {
      uint4 r[kInFlight];
#pragma unroll
      for (int q = 0; q < kInFlight; ++q) {
        const int cc = c + q * blockDim.x;
        if (cc < vecs) r[q] = src[cc];
      }
#pragma unroll
      for (int q = 0; q < kInFlight; ++q) {
        const int cc = c + q * blockDim.x;
        if (cc < vecs) dst[cc] = r[q];
      }
    }
  }
}

}  // namespace

cudaError_t launch_copy_blocks(const void* src_k, const void* src_v, int src_num_blocks,
                               void* dst_k, void* dst_v, int dst_num_blocks,
                               const int32_t* src_ids, const int32_t* dst_ids, int n, int H_kv,
                               int D, int* err, int num_sms, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int vecs = kBlockSize * H_kv * D * 2 / 16;  // 16-byte chunks per block
  const int64_t units = 2 * static_cast<int64_t>(n);
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(units < cap ? units : cap);
  copy_blocks_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4*>(src_k), static_cast<const uint4*>(src_v), src_num_blocks,
      static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v), dst_num_blocks, src_ids, dst_ids,
      n, vecs, err);
  return cudaGetLastError();
}

}  // namespace ps
