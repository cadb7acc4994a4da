// ps_paged_attention_noalloc: paged attention whose scratch lives in a fixed device
// array compiled into this library, so the call needs no workspace and allocates nothing.
//
// Who needs it: code that is handed only its input and output buffers and may not
// create device memory of its own, for example a plug-in running inside a host
// framework that owns every byte of device memory through its own allocator, or a
// latency-critical serving loop that must never call cudaMalloc/cudaFree because they
// can synchronise the whole device and stall every stream.
//
// How it works: the planner's work lists, the per-token split table and the split
// partials are laid out in `g_noalloc_scratch`, a file-scope __device__ array of
// PS_NOALLOC_SCRATCH_BYTES. Host code cannot use the array's name as a device address,
// so the first call on each device (with that device current) looks the address up with
// cudaGetSymbolAddress, checks the result and caches it; make that first call before
// any stream capture. Every later call reuses the array, which keeps whatever the last
// call left in it: the plan kernel rewrites the work list and resets the work counter
// at the start of every call, and every other entry is written before it is read.
// Because all calls share the one array, calls whose kernels overlap on the device
// (two streams, or two host threads) race on it and must be serialised by the caller.
#include <mutex>

#include "pagedserve.h"
#include "ps_common.cuh"
#include "ps_launch.h"

static __device__ __align__(256) uint8_t g_noalloc_scratch[PS_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
uint8_t* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once).
int scratch_address(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (e != cudaSuccess || !addr) return PS_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<uint8_t*>(addr);
  }
  *out = g_scratch_addr[dev];
  return PS_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int ps_paged_attention_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                          const int32_t* block_tables, int max_blocks_per_seq,
                                          const int32_t* seq_lens, const int32_t* query_start_loc,
                                          int B, int T, int H_q, int H_kv, int D, int num_blocks,
                                          float scale, void* out, int dtype, void* stream) {
  // argument checks: everything is rejected on the host before any device work
  if (H_q <= 0 || H_kv <= 0 || B < 0 || T < 0 || max_blocks_per_seq < 0 || num_blocks <= 0)
    return PS_ERR_ARG;
  if (dtype != PS_F16 && dtype != PS_BF16) return PS_ERR_UNSUPPORTED;
  if ((D != 64 && D != 128) || H_q % H_kv) return PS_ERR_UNSUPPORTED;
  if (B == 0 && T != 0) return PS_ERR_ARG;
  if (static_cast<int64_t>(num_blocks) * PS_BLOCK_SIZE > INT32_MAX) return PS_ERR_ARG;
  if (T == 0) return PS_OK;
  if (!q || !k_pool || !v_pool || !out || !block_tables || !seq_lens || !query_start_loc ||
      max_blocks_per_seq == 0)
    return PS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return PS_ERR_ALIGN;
  // beyond the fixed maximum even without room for splitting: reject before device work
  if (ps::workspace_fixed_bytes(T, B, H_q, H_kv, false, nullptr, nullptr) >
      PS_NOALLOC_SCRATCH_BYTES)
    return PS_ERR_WORKSPACE;

  uint8_t* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc) return rc;
  ps::AttnParams p{};
  p.q = q;
  p.out = out;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.max_blocks = max_blocks_per_seq;
  p.B = B;
  p.T = T;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.D = D;
  p.G = H_q / H_kv;
  p.num_blocks = num_blocks;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.tpt = ps::tile_tokens(p.G);
  if (!ps::layout_workspace(p, ws, PS_NOALLOC_SCRATCH_BYTES, true)) return PS_ERR_WORKSPACE;
  return ps::run_attention(p, const_cast<void*>(k_pool), const_cast<void*>(v_pool),
                           dtype == PS_BF16, static_cast<cudaStream_t>(stream));
}
