// C ABI of the paged KV attention library: argument validation, workspace layout,
// TMA descriptors, kernel launches and the benchmark timing hook.
#include <cudaTypedefs.h>

#include <cstdio>

#include <cmath>
#include <mutex>
#include <initializer_list>
#include <new>
#include <vector>

#include "pagedserve.h"
#include "ps_common.cuh"
#include "ps_launch.h"

namespace {

__device__ int g_device_error;  // the library's device error word (one per device)

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool init = false;
  int num_sms = 0;
  int* err = nullptr;  // device address of g_device_error
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceState& s = g_dev[dev];
  if (!s.init) {
    if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PS_ERR_CUDA;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) return PS_ERR_CUDA;
    s.err = static_cast<int*>(addr);
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return PS_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    s.init = true;
  }
  *out = &s;
  return PS_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------------
// timing hook
// ---------------------------------------------------------------------------------
constexpr int kKinds = 9;
struct Profile {
  bool on = false;
  int cap = 0;
  std::vector<cudaEvent_t> ev[kKinds];  // pairs: start, stop
  int used[kKinds] = {};
  float ms[kKinds] = {};
  int done[kKinds] = {};
};
Profile g_prof;
std::mutex g_prof_mu;

struct Timed {
  cudaEvent_t stop = nullptr;
  cudaStream_t stream;
  Timed(int kind, cudaStream_t s) : stream(s) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (!g_prof.on || g_prof.used[kind] >= g_prof.cap) return;
    const int i = g_prof.used[kind]++;
    cudaEventRecord(g_prof.ev[kind][2 * i], s);
    stop = g_prof.ev[kind][2 * i + 1];
  }
  ~Timed() {
    if (stop) cudaEventRecord(stop, stream);
  }
};

thread_local char g_last_error[256] = "";
int cuda_fail(cudaError_t e, const char* where);

// PS_ERR_CUDA, remembering which step failed and CUDA's message for ps_last_error_message.
int cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e),
           static_cast<int>(e));
  return PS_ERR_CUDA;
}

int cuda_status(cudaError_t e, const char* where = "kernel launch") {
  return e == cudaSuccess ? PS_OK : cuda_fail(e, where);
}

int make_pool_map(CUtensorMap* map, const void* pool, int num_blocks, int H_kv, int D, bool bf16) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(H_kv) * D,
                              static_cast<cuuint64_t>(num_blocks) * PS_BLOCK_SIZE};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(H_kv) * D * 2};
  const cuuint32_t box[2] = {64, PS_BLOCK_SIZE};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(
      map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
      const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) return PS_OK;
  snprintf(g_last_error, sizeof(g_last_error), "pool tensor map: CUresult %d", static_cast<int>(r));
  return PS_ERR_CUDA;
}

// q [T, H_q, D] as a 3-D tensor (D, H_q, T) with boxes of 64 elements x G heads x tpt
// tokens: one box is tpt whole tokens of the G query heads that share one KV head.
int make_q_map(CUtensorMap* map, const void* q, int T, int H_q, int D, int G, int tpt, bool bf16) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H_q),
                              static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(H_q) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(tpt)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(
      map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
      const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) return PS_OK;
  snprintf(g_last_error, sizeof(g_last_error), "query tensor map: CUresult %d", static_cast<int>(r));
  return PS_ERR_CUDA;
}

int check_shapes(int H_q, int H_kv, int D, int dtype) {
  if (H_q <= 0 || H_kv <= 0) return PS_ERR_ARG;
  if (dtype != PS_F16 && dtype != PS_BF16) return PS_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return PS_ERR_UNSUPPORTED;
  if (H_q % H_kv != 0) return PS_ERR_UNSUPPORTED;
  return PS_OK;
}

int check_batch(const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                const int32_t* qsl, int B, int T, int num_blocks) {
  if (B < 0 || T < 0 || max_blocks < 0 || num_blocks <= 0) return PS_ERR_ARG;
  if (B == 0 && T != 0) return PS_ERR_ARG;
  if (static_cast<int64_t>(num_blocks) * PS_BLOCK_SIZE > INT32_MAX) return PS_ERR_ARG;
  if (B > 0 && (!seq_lens || !qsl || !block_tables || max_blocks == 0)) return PS_ERR_ARG;
  return PS_OK;
}

}  // namespace

namespace ps {

namespace {
size_t up256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

size_t workspace_fixed_bytes(int T, int B, int H_q, int H_kv, bool headroom, int* cap_items,
                             int* cap_tile) {
  // every count is taken in 64 bits, so sizes near INT_MAX cannot wrap; a plan whose
  // lists would not be indexable with int gives SIZE_MAX (larger than any workspace)
  const int64_t T64 = T, B64 = B, G = H_q / H_kv;
  const int64_t tpt = tile_tokens(static_cast<int>(G));
  const int64_t split_seqs = B64 < T64 ? B64 : T64;
  int64_t ci = H_kv * ((T64 * G + 15) / 16 + B64);
  int64_t ct = tpt > 0 ? H_kv * ((T64 + tpt - 1) / tpt + B64) : 1;
  if (headroom) {
    ci += H_kv * split_seqs * kSplitGroupLimit * (kMaxSplits - 1);
    if (tpt > 0) {
      // pairs of query tiles: half the query tiles (rounded up per sequence) over at most
      // T G / (16 kTileMinGroups + 1) tile-class sequences (each has n G > 16 kTileMinGroups)
      const int64_t tile_seqs = T64 * G / (16 * kTileMinGroups + 1) + 1;
      const int64_t pairs = ((T64 + tpt - 1) / tpt + 1) / 2 + tile_seqs;
      ct += H_kv * pairs * (kMaxSplits - 1);
    }
  }
  if (ci < 1) ci = 1;
  if (ct < 1) ct = 1;
  if (ci > INT32_MAX || ct > INT32_MAX || T64 < 0 || B64 < 0) return SIZE_MAX;
  if (cap_items) *cap_items = static_cast<int>(ci);
  if (cap_tile) *cap_tile = static_cast<int>(ct);
  const size_t per_seq = static_cast<size_t>(B64 + 1) * 4, per_tok = static_cast<size_t>(T64) * 4;
  size_t o = 256;                                                   // header
  o = up256(o + static_cast<size_t>(ci) * sizeof(WorkItem));        // split items
  o = up256(o + per_seq);                                           // seq_off
  o = up256(o + static_cast<size_t>(ct) * sizeof(WorkItem));        // tile items
  o = up256(o + per_seq);                                           // seq_off_t
  o = up256(o + per_tok);                                           // tok_ns
  o = up256(o + per_tok);                                           // tok_base
  o = up256(o + per_seq);                                           // seq_off_p
  o = up256(o + per_seq);                                           // seq_off_s
  o = up256(o + per_tok);                                           // tok_list
  return o;
}

size_t partial_bytes(int64_t cap_part, int D) {
  return up256(static_cast<size_t>(cap_part) * 4) + static_cast<size_t>(cap_part) * D * 4;
}

bool layout_workspace(AttnParams& p, uint8_t* ws, size_t bytes, bool shrink) {
  int ci = 0, ct = 0;
  size_t fixed = workspace_fixed_bytes(p.T, p.B, p.H_q, p.H_kv, true, &ci, &ct);
  if (fixed > bytes) {
    if (!shrink) return false;
    fixed = workspace_fixed_bytes(p.T, p.B, p.H_q, p.H_kv, false, &ci, &ct);
    if (fixed > bytes) return false;
  }
  size_t o = 256;
  p.hdr = reinterpret_cast<int*>(ws);
  p.items = reinterpret_cast<WorkItem*>(ws + o);
  o = up256(o + static_cast<size_t>(ci) * sizeof(WorkItem));
  p.seq_off = reinterpret_cast<int*>(ws + o);
  o = up256(o + static_cast<size_t>(p.B + 1) * 4);
  p.tile_items = reinterpret_cast<WorkItem*>(ws + o);
  o = up256(o + static_cast<size_t>(ct) * sizeof(WorkItem));
  p.seq_off_t = reinterpret_cast<int*>(ws + o);
  o = up256(o + static_cast<size_t>(p.B + 1) * 4);
  p.tok_ns = reinterpret_cast<int*>(ws + o);
  o = up256(o + static_cast<size_t>(p.T) * 4);
  p.tok_base = reinterpret_cast<int*>(ws + o);
  o = up256(o + static_cast<size_t>(p.T) * 4);
  p.seq_off_p = reinterpret_cast<int*>(ws + o);
  o = up256(o + static_cast<size_t>(p.B + 1) * 4);
  p.seq_off_s = reinterpret_cast<int*>(ws + o);
  o = up256(o + static_cast<size_t>(p.B + 1) * 4);
  p.tok_list = reinterpret_cast<int*>(ws + o);
  o = up256(o + static_cast<size_t>(p.T) * 4);
  // the rest holds split partials
  const size_t left = bytes - o;
  int64_t part = static_cast<int64_t>(left / ((p.D + 1) * 4));
  while (part > 0 && partial_bytes(part, p.D) > left) --part;
  if (part > INT32_MAX) part = INT32_MAX;
  p.part_lse = reinterpret_cast<float*>(ws + o);
  p.part_o = reinterpret_cast<float*>(ws + o + up256(static_cast<size_t>(part) * 4));
  p.cap_items = ci;
  p.cap_tile = ct;
  p.cap_part = static_cast<int>(part);
  return true;
}

int run_attention(const AttnParams& p0, void* k_pool, void* v_pool, bool bf16, cudaStream_t s,
                  const ScatterArgs* scatter) {
  AttnParams p = p0;
  int num_sms = 0;
  int* err = nullptr;
  int rc = current_device(&num_sms, &err);
  if (rc) return rc;
  p.err = err;
  // Only a sequence with more than 16 * kTileMinGroups packed rows (n * G) goes to the tile
  // kernel. With one token or more in every sequence, none has more than T - B + 1 tokens;
  // when even that cannot reach a tile the tile kernel is not launched, and the planner is
  // told so (tpt = 0): should a sequence still have that many rows (other sequences
  // without tokens), the split kernel takes it.
  const bool tiles = p.tpt > 0 && (static_cast<int64_t>(p.T) - p.B + 1) * p.G > 16 * kTileMinGroups;
  if (!tiles) p.tpt = 0;
  CUtensorMap kmap, vmap, qmap;
  if ((rc = make_pool_map(&kmap, k_pool, p.num_blocks, p.H_kv, p.D, bf16))) return rc;
  if ((rc = make_pool_map(&vmap, v_pool, p.num_blocks, p.H_kv, p.D, bf16))) return rc;
  if (tiles && (rc = make_q_map(&qmap, p.q, p.T, p.H_q, p.D, p.G, p.tpt, bf16))) return rc;
  cudaError_t e;
  const CopySegments* pre = scatter != nullptr ? scatter->pre : nullptr;
  const bool direct = direct_fits(p, num_sms), direct_tile = tiles && direct_tile_fits(p, num_sms);
  if (pre != nullptr && pre->n > 0 && (direct || direct_tile) &&
      (e = launch_gather_in(*pre, num_sms, s, false)) != cudaSuccess)
    return cuda_fail(e, "input gather kernel");
  if (direct) {
    // a small batch: the whole step (scatter included) in one launch, without a plan
    p.direct = 1;
    if (scatter) {
      p.new_k = scatter->k;
      p.new_v = scatter->v;
      p.k_pool = k_pool;
      p.v_pool = v_pool;
    }
    Timed tm(3, s);
    if ((e = launch_direct_attention(p, bf16, kmap, vmap, num_sms, s)) != cudaSuccess)
      return cuda_fail(e, "split attention kernel (direct)");
    return PS_OK;
  }
  // A few sequences with query tiles and short contexts: the tile kernel alone, right after
  // the step's scatter, each CTA deriving its items (every sequence unsplit) from seq_lens
  // and qsl. No plan, nothing to combine.
  if (direct_tile) {
    if (scatter) {
      Timed tm(1, s);
      if ((e = launch_step_scatter(scatter->k, scatter->v, p.block_tables, p.max_blocks,
                                   p.seq_lens, p.qsl, p.B, p.T, p.H_kv, p.D, p.num_blocks,
                                   p.slots, k_pool, v_pool, err, num_sms, s)) != cudaSuccess)
        return cuda_fail(e, "KV scatter kernel");
      p.after_scatter = 1;
    }
    Timed tm(5, s);
    if ((e = launch_tile_attention(p, bf16, kmap, vmap, qmap, direct_tile_ctas(p, num_sms), s,
                                   true, true)) != cudaSuccess)
      return cuda_fail(e, "tile attention kernel (direct)");
    return PS_OK;
  }
  // A batch of so few sequences that each could have its own tile item runs on the tile
  // kernel alone: its decode or verify rows become single query tiles (split along the
  // context, since tile items are scarce), and the split kernel is not launched.
  if (tiles && static_cast<int64_t>(p.B) * p.H_kv * 2 <= num_sms) p.all_tiles = 1;
  const int split_grid = split_ctas(p, num_sms);
  const int concurrency = split_grid * attention_warps(p.D);
  // The planner goes first, with the step's KV scatter (if any) on extra CTAs of the same
  // launch; every later launch is chained with programmatic dependent launch.
  {
    AttnParams pp = p;
    if (scatter) {
      pp.new_k = scatter->k;
      pp.new_v = scatter->v;
      pp.k_pool = k_pool;
      pp.v_pool = v_pool;
    }
    Timed tm(2, s);
    if ((e = launch_plan(pp, concurrency, num_sms, num_sms, s, pre)) != cudaSuccess)
      return cuda_fail(e, "plan kernel");
  }
  // One stream, every launch chained with programmatic dependent launch. With both
  // kernels, the tile kernel follows the split kernel and runs beside it: it reads the
  // plan without waiting (the split kernel lets it launch only once the plan is complete),
  // and its CTAs take their items from a counter, so CTAs that start late (on SMs the split
  // kernel still holds) just join in.
  if (!p.all_tiles) {
    Timed tm(3, s);
    if ((e = launch_split_attention(p, bf16, kmap, vmap, split_grid, s, true)) != cudaSuccess)
      return cuda_fail(e, "split attention kernel");
  }
  if (tiles) {
    AttnParams pt = p;
    pt.after_split = !p.all_tiles;
    Timed tm(5, s);
    if ((e = launch_tile_attention(pt, bf16, kmap, vmap, qmap, num_sms, s, true)) != cudaSuccess)
      return cuda_fail(e, "tile attention kernel");
  }
  // A split holds at least kMinSplitPages pages, so with no block table longer than that
  // no row is split and there is nothing to combine.
  if (p.max_blocks > kMinSplitPages) {
    Timed tm(4, s);
    if ((e = launch_combine(p, bf16, num_sms, s, true)) != cudaSuccess)
      return cuda_fail(e, "combine kernel");
  }
  return PS_OK;
}

int current_device(int* num_sms, int** err) {
  DeviceState* ds;
  const int rc = current_device_state(&ds);
  if (rc) return rc;
  *num_sms = ds->num_sms;
  *err = ds->err;
  return PS_OK;
}

int encode_pool_map(CUtensorMap* map, const void* pool, int num_blocks, int H_kv, int D,
                    bool bf16) {
  DeviceState* ds;
  const int rc = current_device_state(&ds);  // makes sure the encoder is resolved
  if (rc) return rc;
  return make_pool_map(map, pool, num_blocks, H_kv, D, bf16);
}
}  // namespace ps

extern "C" {

const char* ps_status_string(int status) {
  switch (status) {
    case PS_OK: return "PS_OK";
    case PS_ERR_ARG: return "PS_ERR_ARG: invalid size, count or pointer";
    case PS_ERR_UNSUPPORTED: return "PS_ERR_UNSUPPORTED: dtype, head_dim or head counts";
    case PS_ERR_ALIGN: return "PS_ERR_ALIGN: tensor pointer not 16-byte aligned";
    case PS_ERR_WORKSPACE: return "PS_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case PS_ERR_CUDA: return "PS_ERR_CUDA: CUDA call or kernel launch failed";
    default: return "unknown ps_status";
  }
}

int ps_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                    const int32_t* query_start_loc, int B, int T, int num_blocks,
                    int32_t* slot_mapping, void* stream) {
  int rc = check_batch(block_tables, max_blocks_per_seq, seq_lens, query_start_loc, B, T,
                       num_blocks);
  if (rc) return rc;
  if (T > 0 && !slot_mapping) return PS_ERR_ARG;
  if (T == 0) return PS_OK;
  DeviceState* ds;
  if ((rc = current_device_state(&ds))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Timed tm(0, s);
  return cuda_status(ps::launch_slot_mapping(block_tables, max_blocks_per_seq, seq_lens,
                                             query_start_loc, B, T, num_blocks, slot_mapping,
                                             ds->err, s),
                     "slot mapping kernel");
}

int ps_reshape_and_cache(const void* k, const void* v, const int32_t* slot_mapping, void* k_pool,
                         void* v_pool, int T, int H_kv, int D, int num_blocks, int dtype,
                         void* stream) {
  int rc = check_shapes(H_kv, H_kv, D, dtype);
  if (rc) return rc;
  if (T < 0 || num_blocks <= 0) return PS_ERR_ARG;
  if (static_cast<int64_t>(num_blocks) * PS_BLOCK_SIZE > INT32_MAX) return PS_ERR_ARG;
  if (T == 0) return PS_OK;
  if (!k || !v || !slot_mapping || !k_pool || !v_pool) return PS_ERR_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool))
    return PS_ERR_ALIGN;
  DeviceState* ds;
  if ((rc = current_device_state(&ds))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Timed tm(1, s);
  return cuda_status(ps::launch_reshape_and_cache(k, v, slot_mapping, k_pool, v_pool, T, H_kv, D,
                                                  num_blocks, ds->err, ds->num_sms, s),
                     "KV scatter kernel");
}

int ps_copy_blocks(const void* src_k, const void* src_v, int src_num_blocks, void* dst_k,
                   void* dst_v, int dst_num_blocks, const int32_t* src_ids,
                   const int32_t* dst_ids, int n, int H_kv, int D, int dtype, void* stream) {
  int rc = check_shapes(H_kv, H_kv, D, dtype);
  if (rc) return rc;
  if (n < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0) return PS_ERR_ARG;
  if (n == 0) return PS_OK;
  if (!src_k || !src_v || !dst_k || !dst_v || !src_ids || !dst_ids) return PS_ERR_ARG;
  if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
    return PS_ERR_ALIGN;
  DeviceState* ds;
  if ((rc = current_device_state(&ds))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Timed tm(6, s);
  return cuda_status(ps::launch_copy_blocks(src_k, src_v, src_num_blocks, dst_k, dst_v,
                                            dst_num_blocks, src_ids, dst_ids, n, H_kv, D,
                                            ds->err, ds->num_sms, s),
                     "block copy kernel");
}

int ps_rope_reshape_and_cache(void* q, const void* k, const void* v, const int32_t* positions,
                              const int32_t* slot_mapping, void* k_pool, void* v_pool, int T,
                              int H_q, int H_kv, int D, int num_blocks, float rope_theta,
                              int dtype, void* stream) {
  int rc = check_shapes(H_q, H_kv, D, dtype);
  if (rc) return rc;
  if (T < 0 || num_blocks <= 0 || !(rope_theta > 1.f) || !std::isfinite(rope_theta))
    return PS_ERR_ARG;
  if (static_cast<int64_t>(num_blocks) * PS_BLOCK_SIZE > INT32_MAX) return PS_ERR_ARG;
  if (T == 0) return PS_OK;
  if (!q || !k || !v || !positions || !slot_mapping || !k_pool || !v_pool) return PS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_pool) ||
      !aligned16(v_pool))
    return PS_ERR_ALIGN;
  DeviceState* ds;
  if ((rc = current_device_state(&ds))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Timed tm(8, s);
  return cuda_status(ps::launch_rope_reshape_and_cache(q, k, v, positions, slot_mapping, k_pool,
                                                       v_pool, T, H_q, H_kv, D, num_blocks,
                                                       rope_theta, dtype == PS_BF16, ds->err,
                                                       ds->num_sms, s),
                     "rotary KV scatter kernel");
}

size_t ps_spec_accept_workspace_size(int B, int k, int V) {
  if (B < 0 || k < 0 || V <= 0) return 0;
  // greedy entries per row: one per run (16-byte rows) or per chunk, whichever is more
  const int per_row = ps::spec_runs(V) > ps::spec_chunks(V) ? ps::spec_runs(V) : ps::spec_chunks(V);
  const size_t rows = static_cast<size_t>(B) * (k + 1) * per_row;
  const size_t runs = static_cast<size_t>(B) * ps::spec_runs(V);
  return ps::up256(runs * 8) + 2 * ps::up256(rows * 4) + ps::up256(static_cast<size_t>(B) * 4);
}

int ps_spec_accept(const float* target_probs, const float* draft_probs,
                   const int32_t* draft_tokens, const uint32_t* random_bits, int B, int k, int V,
                   int greedy, int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                   size_t workspace_bytes, void* stream) {
  if (B < 0 || k < 0 || V <= 0) return PS_ERR_ARG;
  if (k > 31) return PS_ERR_UNSUPPORTED;  // one lane per draft decides the acceptance
  if (V > (1 << 30)) return PS_ERR_UNSUPPORTED;  // token indices stay 32-bit
  if (B == 0) return PS_OK;
  if (!target_probs || !out_tokens || !num_accepted) return PS_ERR_ARG;
  if (k > 0 && !draft_tokens) return PS_ERR_ARG;
  if (!greedy && !random_bits) return PS_ERR_ARG;
  const size_t need = ps_spec_accept_workspace_size(B, k, V);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return PS_ERR_WORKSPACE;
  DeviceState* ds;
  int rc = current_device_state(&ds);
  if (rc) return rc;
  const int per_row = ps::spec_runs(V) > ps::spec_chunks(V) ? ps::spec_runs(V) : ps::spec_chunks(V);
  const size_t rows = static_cast<size_t>(B) * (k + 1) * per_row;
  const size_t runs = ps::up256(static_cast<size_t>(B) * ps::spec_runs(V) * 8);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  ps::SpecParams a = {};
  a.p = target_probs;
  a.q = draft_probs;
  a.drafts = draft_tokens;
  a.rnd = random_bits;
  a.B = B;
  a.k = k;
  a.V = V;
  a.greedy = greedy ? 1 : 0;
  a.out = out_tokens;
  a.num = num_accepted;
  a.wsum = reinterpret_cast<long long*>(ws);
  a.amax_v = reinterpret_cast<float*>(ws + runs);
  a.amax_i = reinterpret_cast<int*>(ws + runs + ps::up256(rows * 4));
  a.acc = reinterpret_cast<int*>(ws + runs + 2 * ps::up256(rows * 4));
  a.num_sms = ds->num_sms;
  a.err = ds->err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Timed tm(7, s);
  return cuda_status(ps::launch_spec_accept(a, s), "speculative acceptance kernels");
}

size_t ps_paged_attention_workspace_size(int T, int B, int H_q, int H_kv, int D,
                                         int max_seq_len) {
  if (T < 0 || B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv || (D != 64 && D != 128))
    return 0;
  const size_t fixed = ps::workspace_fixed_bytes(T, B, H_q, H_kv, true, nullptr, nullptr);
  if (fixed == SIZE_MAX) return 0;  // no workspace can hold the plan
  int64_t splits = (static_cast<int64_t>(max_seq_len) + ps::kBlockSize * ps::kMinSplitPages - 1) /
                   (ps::kBlockSize * ps::kMinSplitPages);
  if (splits > ps::kMaxSplits) splits = ps::kMaxSplits;
  if (splits < 2) splits = 0;  // nothing to split
  const int64_t cap_part = static_cast<int64_t>(T) * H_q * splits;
  return fixed + ps::partial_bytes(cap_part, D);
}

namespace {
// Host-side checks of ps_paged_attention's arguments (T > 0 assumed checked by caller).
int check_attention(const void* q, const void* k_pool, const void* v_pool,
                    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                    const int32_t* query_start_loc, int B, int T, int H_q, int H_kv, int D,
                    int num_blocks, const void* out, const void* workspace,
                    size_t workspace_bytes, int dtype) {
  int rc = check_shapes(H_q, H_kv, D, dtype);
  if (rc) return rc;
  if ((rc = check_batch(block_tables, max_blocks_per_seq, seq_lens, query_start_loc, B, T,
                        num_blocks)))
    return rc;
  if (T == 0) return PS_OK;
  if (!q || !k_pool || !v_pool || !out) return PS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return PS_ERR_ALIGN;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PS_ERR_WORKSPACE;
  if (workspace_bytes < ps::workspace_fixed_bytes(T, B, H_q, H_kv, true, nullptr, nullptr))
    return PS_ERR_WORKSPACE;
  return PS_OK;
}
}  // namespace

int ps_paged_attention(const void* q, const void* k_pool, const void* v_pool,
                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                       const int32_t* query_start_loc, int B, int T, int H_q, int H_kv, int D,
                       int num_blocks, float scale, void* out, void* workspace,
                       size_t workspace_bytes, int dtype, void* stream) {
  int rc = check_attention(q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens,
                           query_start_loc, B, T, H_q, H_kv, D, num_blocks, out, workspace,
                           workspace_bytes, dtype);
  if (rc) return rc;
  if (T == 0) return PS_OK;
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
  if (!ps::layout_workspace(p, static_cast<uint8_t*>(workspace), workspace_bytes, false))
    return PS_ERR_WORKSPACE;
  return ps::run_attention(p, const_cast<void*>(k_pool), const_cast<void*>(v_pool),
                           dtype == PS_BF16, static_cast<cudaStream_t>(stream));
}

namespace {
// The step, with copies still to make before the attention kernels read their
// destinations (`pre`, the host step's queries) or none.
int attention_step_impl(const void* q, const void* k, const void* v, void* k_pool, void* v_pool,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* seq_lens, const int32_t* query_start_loc, int B, int T,
                        int H_q, int H_kv, int D, int num_blocks, float scale, void* out,
                        int32_t* slot_mapping, void* workspace, size_t workspace_bytes, int dtype,
                        void* stream, const ps::CopySegments* pre);
}  // namespace

int ps_attention_step(const void* q, const void* k, const void* v, void* k_pool, void* v_pool,
                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                      const int32_t* query_start_loc, int B, int T, int H_q, int H_kv, int D,
                      int num_blocks, float scale, void* out, int32_t* slot_mapping,
                      void* workspace, size_t workspace_bytes, int dtype, void* stream) {
  return attention_step_impl(q, k, v, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens,
                             query_start_loc, B, T, H_q, H_kv, D, num_blocks, scale, out,
                             slot_mapping, workspace, workspace_bytes, dtype, stream, nullptr);
}

namespace {
int attention_step_impl(const void* q, const void* k, const void* v, void* k_pool, void* v_pool,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* seq_lens, const int32_t* query_start_loc, int B, int T,
                        int H_q, int H_kv, int D, int num_blocks, float scale, void* out,
                        int32_t* slot_mapping, void* workspace, size_t workspace_bytes, int dtype,
                        void* stream, const ps::CopySegments* pre) {
  // validate everything before enqueuing anything
  int rc = check_attention(q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens,
                           query_start_loc, B, T, H_q, H_kv, D, num_blocks, out, workspace,
                           workspace_bytes, dtype);
  if (rc) return rc;
  if (T == 0) return PS_OK;
  if (!k || !v || !slot_mapping) return PS_ERR_ARG;
  if (!aligned16(k) || !aligned16(v)) return PS_ERR_ALIGN;
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
  p.slots = slot_mapping;
  if (!ps::layout_workspace(p, static_cast<uint8_t*>(workspace), workspace_bytes, false))
    return PS_ERR_WORKSPACE;
  const ps::ScatterArgs sc{k, v, pre};
  return ps::run_attention(p, k_pool, v_pool, dtype == PS_BF16, static_cast<cudaStream_t>(stream),
                           &sc);
}
}  // namespace

namespace {
struct StagingLayout {
  size_t q, k, v, bt, sl, qsl, slots, out, ws, total;
};
StagingLayout staging_layout(int T, int B, int max_blocks, int H_q, int H_kv, int D,
                             size_t ws_bytes) {
  StagingLayout l;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  l.q = take(static_cast<size_t>(T) * H_q * D * 2);
  l.k = take(static_cast<size_t>(T) * H_kv * D * 2);
  l.v = take(static_cast<size_t>(T) * H_kv * D * 2);
  l.bt = take(static_cast<size_t>(B) * max_blocks * 4);
  l.sl = take(static_cast<size_t>(B) * 4);
  l.qsl = take(static_cast<size_t>(B + 1) * 4);
  l.slots = take(static_cast<size_t>(T) * 4);
  l.out = take(static_cast<size_t>(T) * H_q * D * 2);
  l.ws = take(ws_bytes);
  l.total = o;
  return l;
}
}  // namespace

size_t ps_attention_step_host_staging_size(int T, int B, int max_blocks_per_seq, int H_q,
                                           int H_kv, int D, int max_seq_len) {
  if (max_blocks_per_seq < 0) return 0;
  const size_t ws = ps_paged_attention_workspace_size(T, B, H_q, H_kv, D, max_seq_len);
  if (ws == 0) return 0;
  return staging_layout(T, B, max_blocks_per_seq, H_q, H_kv, D, ws).total;
}

namespace {
// The device's view of a host buffer the kernels may read directly: page-locked, mapped
// for the device and 4-byte aligned; null otherwise (the buffer is then copied by a
// copy operation). Not called while a graph is being captured.
const void* device_view(const void* h) {
  if (!h || (reinterpret_cast<uintptr_t>(h) & 3u)) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer ||
      (reinterpret_cast<uintptr_t>(a.devicePointer) & 3u))
    return nullptr;
  return a.devicePointer;
}

// The host step. dev[i] is the device's view of host buffer i (q, k, v, block tables,
// lengths, offsets, out) or null: the new K and V rows with a view are read by the step's
// scatter itself, other inputs with a view are gathered by one kernel that reads them
// across the host link, the rest copied one by one; an output with a view is written by
// the step's kernels themselves (up to 4 MB) or by a kernel after them, otherwise copied.
int host_step(const void* q, const void* k, const void* v, const int32_t* block_tables,
              const int32_t* seq_lens, const int32_t* query_start_loc, void* out, void* k_pool,
              void* v_pool, int max_blocks_per_seq, int B, int T, int H_q, int H_kv, int D,
              int num_blocks, float scale, void* staging, size_t staging_bytes, int dtype,
              void* stream, const void* const dev[7]);
}  // namespace

int ps_attention_step_host(const void* q, const void* k, const void* v,
                           const int32_t* block_tables, const int32_t* seq_lens,
                           const int32_t* query_start_loc, void* out, void* k_pool, void* v_pool,
                           int max_blocks_per_seq, int B, int T, int H_q, int H_kv, int D,
                           int num_blocks, float scale, void* staging, size_t staging_bytes,
                           int dtype, void* stream) {
  const void* dev[7] = {device_view(q), device_view(k), device_view(v), device_view(block_tables),
                        device_view(seq_lens), device_view(query_start_loc), device_view(out)};
  return host_step(q, k, v, block_tables, seq_lens, query_start_loc, out, k_pool, v_pool,
                   max_blocks_per_seq, B, T, H_q, H_kv, D, num_blocks, scale, staging,
                   staging_bytes, dtype, stream, dev);
}

namespace {
int host_step(const void* q, const void* k, const void* v, const int32_t* block_tables,
              const int32_t* seq_lens, const int32_t* query_start_loc, void* out, void* k_pool,
              void* v_pool, int max_blocks_per_seq, int B, int T, int H_q, int H_kv, int D,
              int num_blocks, float scale, void* staging, size_t staging_bytes, int dtype,
              void* stream, const void* const dev[7]) {
  int rc = check_shapes(H_q, H_kv, D, dtype);
  if (rc) return rc;
  if ((rc = check_batch(block_tables, max_blocks_per_seq, seq_lens, query_start_loc, B, T,
                        num_blocks)))
    return rc;
  if (T == 0) return PS_OK;
  if (!q || !k || !v || !out || !k_pool || !v_pool) return PS_ERR_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool)) return PS_ERR_ALIGN;
  if (!staging || (reinterpret_cast<uintptr_t>(staging) & 255u)) return PS_ERR_WORKSPACE;
  // the attention workspace takes whatever the inputs leave over
  const StagingLayout l0 = staging_layout(T, B, max_blocks_per_seq, H_q, H_kv, D, 0);
  if (staging_bytes < l0.total) return PS_ERR_WORKSPACE;
  const size_t ws_bytes = staging_bytes - l0.total;
  const StagingLayout l = staging_layout(T, B, max_blocks_per_seq, H_q, H_kv, D, 0);
  uint8_t* st = static_cast<uint8_t*>(staging);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  struct Copy {
    void* dst;
    const void* src;
    size_t bytes;
  } in[] = {
      {st + l.q, q, static_cast<size_t>(T) * H_q * D * 2},
      {st + l.k, k, static_cast<size_t>(T) * H_kv * D * 2},
      {st + l.v, v, static_cast<size_t>(T) * H_kv * D * 2},
      {st + l.bt, block_tables, static_cast<size_t>(B) * max_blocks_per_seq * 4},
      {st + l.sl, seq_lens, static_cast<size_t>(B) * 4},
      {st + l.qsl, query_start_loc, static_cast<size_t>(B + 1) * 4},
  };
  // The new tokens' K and V rows are read once, by the step's KV scatter: with a 16-byte
  // aligned device view, the scatter reads them across the host link itself.
  const bool kv_direct = dev[1] && dev[2] && aligned16(dev[1]) && aligned16(dev[2]);
  // The queries are read only by the attention kernels: their copy goes to the step, which
  // makes it on extra CTAs of the planner's launch (beside the planning), or first when the
  // step has no planner. The other inputs are gathered before the step.
  ps::CopySegments segs{}, pre{};
  for (int i = 0; i < 6; ++i) {
    const Copy& c = in[i];
    if (c.bytes == 0 || (kv_direct && (i == 1 || i == 2))) continue;
    if (dev[i] && c.bytes % 4 == 0) {
      ps::CopySegments& to = i == 0 ? pre : segs;
      to.seg[to.n++] = ps::CopySegment{c.dst, dev[i], static_cast<int64_t>(c.bytes)};
    } else if (cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
      return PS_ERR_CUDA;
    }
  }
  if (segs.n > 0) {
    int num_sms = 0, *err = nullptr;
    if ((rc = ps::current_device(&num_sms, &err))) return rc;
    if (ps::launch_gather_in(segs, num_sms, s, false) != cudaSuccess) return PS_ERR_CUDA;
  }
  // A small output (up to kDirectOutBytes) goes straight from the step's kernels into the
  // page-locked host buffer, so it crosses the host link while the last kernels run. A
  // larger one is written to the staging buffer and then moved by a kernel that follows the
  // step's last kernel (or copied): written directly, its stores would hold the attention
  // kernels back at the link's rate.
  constexpr size_t kDirectOutBytes = size_t(4) << 20;
  const size_t out_bytes = static_cast<size_t>(T) * H_q * D * 2;
  const bool direct_out = dev[6] && aligned16(dev[6]) && out_bytes <= kDirectOutBytes;
  rc = attention_step_impl(st + l.q, kv_direct ? dev[1] : st + l.k,
                           kv_direct ? dev[2] : st + l.v, k_pool, v_pool,
                           reinterpret_cast<const int32_t*>(st + l.bt), max_blocks_per_seq,
                           reinterpret_cast<const int32_t*>(st + l.sl),
                           reinterpret_cast<const int32_t*>(st + l.qsl), B, T, H_q, H_kv, D,
                           num_blocks, scale, direct_out ? const_cast<void*>(dev[6]) : st + l.out,
                           reinterpret_cast<int32_t*>(st + l.slots), st + l.ws, ws_bytes, dtype,
                           stream, pre.n > 0 ? &pre : nullptr);
  if (rc || direct_out) return rc;
  if (dev[6] && out_bytes % 4 == 0) {
    ps::CopySegments o{};
    o.seg[0] = ps::CopySegment{const_cast<void*>(dev[6]), st + l.out,
                               static_cast<int64_t>(out_bytes)};
    o.n = 1;
    int num_sms = 0, *err = nullptr;
    if ((rc = ps::current_device(&num_sms, &err))) return rc;
    if (ps::launch_gather_in(o, num_sms, s, true) != cudaSuccess) return PS_ERR_CUDA;
  } else if (cudaMemcpyAsync(out, st + l.out, out_bytes, cudaMemcpyDeviceToHost, s) !=
             cudaSuccess) {
    return PS_ERR_CUDA;
  }
  return PS_OK;
}
}  // namespace

// One host step in a CUDA graph: the copies in, the step's kernels and the copy out are
// captured from a private stream and instantiated once; each launch replays them with the
// host buffers' contents at that time.
struct HostStepGraph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

int ps_attention_step_host_graph_create(const void* q, const void* k, const void* v,
                                        const int32_t* block_tables, const int32_t* seq_lens,
                                        const int32_t* query_start_loc, void* out,
                                        void* k_pool, void* v_pool, int max_blocks_per_seq,
                                        int B, int T, int H_q, int H_kv, int D, int num_blocks,
                                        float scale, void* staging, size_t staging_bytes,
                                        int dtype, void** graph) {
  if (!graph) return PS_ERR_ARG;
  // argument errors are reported before anything is resolved or recorded
  int rc = check_shapes(H_q, H_kv, D, dtype);
  if (rc) return rc;
  if ((rc = check_batch(block_tables, max_blocks_per_seq, seq_lens, query_start_loc, B, T,
                        num_blocks)))
    return rc;
  // device state (SM count, error word, tensor-map encoder) is resolved before capture
  DeviceState* ds;
  if ((rc = current_device_state(&ds))) return rc;
  // every host buffer the graph copies from or to must be page-locked (null ones are left
  // to the step's own argument checks)
  for (const void* h : {q, k, v, static_cast<const void*>(block_tables),
                        static_cast<const void*>(seq_lens),
                        static_cast<const void*>(query_start_loc),
                        static_cast<const void*>(out)}) {
    if (!h) continue;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
      cudaGetLastError();
      return PS_ERR_ARG;
    }
    if (a.type != cudaMemoryTypeHost) return PS_ERR_ARG;
  }
  const void* dev[7] = {device_view(q), device_view(k), device_view(v), device_view(block_tables),
                        device_view(seq_lens), device_view(query_start_loc), device_view(out)};
  cudaStream_t cs;
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e, "graph stream");
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) {
    cudaStreamDestroy(cs);
    return cuda_fail(e, "graph capture");
  }
  rc = host_step(q, k, v, block_tables, seq_lens, query_start_loc, out, k_pool, v_pool,
                 max_blocks_per_seq, B, T, H_q, H_kv, D, num_blocks, scale, staging,
                 staging_bytes, dtype, cs, dev);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(cs, &g);  // ends the capture whatever the step returned
  cudaStreamDestroy(cs);
  if (rc || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();  // clear the last-error state a failed capture leaves behind
    return rc ? rc : cuda_fail(e != cudaSuccess ? e : cudaErrorUnknown, "graph capture");
  }
  cudaGraphExec_t x;
  e = cudaGraphInstantiate(&x, g, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    return cuda_fail(e, "graph instantiate");
  }
  auto* h = new (std::nothrow) HostStepGraph{g, x};
  if (!h) {
    cudaGraphExecDestroy(x);
    cudaGraphDestroy(g);
    return cuda_fail(cudaErrorMemoryAllocation, "graph handle");
  }
  *graph = h;
  return PS_OK;
}

int ps_graph_launch(void* graph, void* stream) {
  if (!graph) return PS_ERR_ARG;
  const cudaError_t e =
      cudaGraphLaunch(static_cast<HostStepGraph*>(graph)->exec, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PS_OK : cuda_fail(e, "graph launch");
}

int ps_graph_destroy(void* graph) {
  if (!graph) return PS_ERR_ARG;
  auto* h = static_cast<HostStepGraph*>(graph);
  cudaGraphExecDestroy(h->exec);
  cudaGraphDestroy(h->graph);
  delete h;
  return PS_OK;
}

const char* ps_last_error_message(void) { return g_last_error; }

int ps_get_device_error(int* code) {
  if (!code) return PS_ERR_ARG;
  DeviceState* ds;
  int rc = current_device_state(&ds);
  if (rc) return rc;
  int v = 0;
  if (cudaMemcpy(&v, ds->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PS_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(ds->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return PS_ERR_CUDA;
  *code = v;
  return PS_OK;
}

int ps_profile_begin(int max_launches_per_kind) {
  if (max_launches_per_kind <= 0) return PS_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  for (int k = 0; k < kKinds; ++k) {
    for (cudaEvent_t e : g_prof.ev[k]) cudaEventDestroy(e);
    g_prof.ev[k].assign(2 * max_launches_per_kind, nullptr);
    for (auto& e : g_prof.ev[k])
      if (cudaEventCreate(&e) != cudaSuccess) return PS_ERR_CUDA;
    g_prof.used[k] = 0;
    g_prof.ms[k] = 0.f;
    g_prof.done[k] = 0;
  }
  g_prof.cap = max_launches_per_kind;
  g_prof.on = true;
  return PS_OK;
}

int ps_profile_end(void) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof.on = false;
  for (int k = 0; k < kKinds; ++k) {
    float total = 0.f;
    for (int i = 0; i < g_prof.used[k]; ++i) {
      if (cudaEventSynchronize(g_prof.ev[k][2 * i + 1]) != cudaSuccess) return PS_ERR_CUDA;
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, g_prof.ev[k][2 * i], g_prof.ev[k][2 * i + 1]) != cudaSuccess)
        return PS_ERR_CUDA;
      total += ms;
    }
    g_prof.ms[k] = total;
    g_prof.done[k] = g_prof.used[k];
  }
  return PS_OK;
}

int ps_profile_read(int kind, float* total_ms, int* launches) {
  if (kind < 0 || kind >= kKinds || !total_ms || !launches) return PS_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  *total_ms = g_prof.ms[kind];
  *launches = g_prof.done[kind];
  return PS_OK;
}

}  // extern "C"
