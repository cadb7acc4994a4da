// Internal launch interface between the C ABI (ps_abi.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace ps {

struct WorkItem;

// Everything the planner, the attention kernels and the combine kernel read.
struct AttnParams {
  const void* q;                 // [T, H_q, D]
  void* out;                     // [T, H_q, D]
  const int32_t* block_tables;   // [B, max_blocks]
  const int32_t* seq_lens;       // [B]
  const int32_t* qsl;            // [B + 1]
  int max_blocks;
  int B, T, H_q, H_kv, D, G, num_blocks;
  float scale_log2;              // softmax scale * log2(e)
  // workspace
  // [0] split-kernel items, [1] their fetch counter, [2] pages per split, [3] partials,
  // [4] tile-kernel items, [5] their fetch counter, [6] tile pages per split,
  // [7] tokens whose rows are split (entries of tok_list)
  int* hdr;
  WorkItem* items;               // [cap_items] split-kernel work (decode rows)
  int* seq_off;                  // [B + 1] sequence's first split item within its length class
  WorkItem* tile_items;          // [cap_tile] tile-kernel work (prefill / verify rows)
  int* seq_off_t;                // [B + 1] first tile-kernel item of each sequence
  int cap_tile;
  int tpt;                       // query tokens per 128-row tile (0: no tile kernel)
  int all_tiles;                 // every sequence with rows goes to the tile kernel (no split kernel)
  int* tok_ns;                   // [T] splits holding each token's rows (0 = none)
  int* tok_base;                 // [T] first partial entry of each token
  int* seq_off_p;                // [B + 1] first partial entry of each sequence
  int* seq_off_s;                // [B + 1] first tok_list entry of each sequence
  int* tok_list;                 // [T] the tokens whose rows are split, for the combine
  float* part_lse;               // [cap_part] log2-sum-exp of each partial
  float* part_o;                 // [cap_part, D] normalised partial outputs
  int cap_items, cap_part;
  int* err;                      // device error word
  int32_t* slots;                // [T] slot of every token, written by the step's scatter
  // Direct mode (small batches, see launch_direct_attention): the split kernel takes one
  // item per (sequence, KV head) straight from seq_lens and qsl instead of a plan, and,
  // with new_k set, first scatters the step's K/V into the pools.
  int direct;
  // The tile kernel's direct mode was launched right after the step's scatter, which
  // waited for the earlier work on the stream: the step's inputs may be read before the
  // wait for the scatter itself.
  int after_scatter;
  // The tile kernel follows the split kernel on the stream. The split kernel lets its
  // dependents launch only once the plan is complete, so the tile kernel reads the plan
  // without waiting, runs beside the split kernel, and waits for it only before it ends
  // (one thread), so that its completion stands for both for the combine.
  int after_split;
  const void* new_k;             // [T, H_kv, D] the step's K and V, or null
  const void* new_v;
  void* k_pool;                  // [num_blocks, 16, H_kv, D]
  void* v_pool;
};

// Raise `kern`'s dynamic shared-memory limit to `bytes` once per device: the setting lasts
// for the process, and repeating it on every launch only costs host time.
template <typename Kern>
inline cudaError_t ensure_smem_limit(Kern kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return ge;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Launch `kern` on `s`; with `pdl` the launch may overlap the tail of the previous kernel
// on the stream (the kernel waits with pdl_wait before using that kernel's results).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Copies between page-locked host memory (through its device view) and device memory,
// several buffers in one launch; each buffer's address and size must be multiples of 4
// bytes. With pdl, it may start while the kernel before it runs and waits for it before
// reading.
struct CopySegment {
  void* dst;
  const void* src;
  int64_t bytes;
};
struct CopySegments {
  CopySegment seg[8];
  int n;
};
cudaError_t launch_gather_in(const CopySegments& segs, int num_sms, cudaStream_t stream,
                             bool pdl);

cudaError_t launch_slot_mapping(const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                const int32_t* qsl, int B, int T, int num_blocks, int32_t* slots,
                                int* err, cudaStream_t stream);

cudaError_t launch_reshape_and_cache(const void* k, const void* v, const int32_t* slots,
                                     void* k_pool, void* v_pool, int T, int H_kv, int D,
                                     int num_blocks, int* err, int num_sms, cudaStream_t stream,
                                     bool pdl = false);

// The step's KV scatter with its slot mapping (the first kernel of ps_attention_step): the
// slot of every packed token is written to `slots` and its K/V rows to the pools.
cudaError_t launch_step_scatter(const void* k, const void* v, const int32_t* block_tables,
                                int max_blocks, const int32_t* seq_lens, const int32_t* qsl, int B,
                                int T, int H_kv, int D, int num_blocks, int32_t* slots,
                                void* k_pool, void* v_pool, int* err, int num_sms,
                                cudaStream_t stream);

// Copy n whole blocks (16 rows x H_kv x D, K and V): dst block dst_ids[i] of (dst_k, dst_v)
// gets src block src_ids[i] of (src_k, src_v). Pools may be device or pinned host memory.
cudaError_t launch_copy_blocks(const void* src_k, const void* src_v, int src_num_blocks,
                               void* dst_k, void* dst_v, int dst_num_blocks,
                               const int32_t* src_ids, const int32_t* dst_ids, int n, int H_kv,
                               int D, int* err, int num_sms, cudaStream_t stream);

// Rotary embedding of q (in place) and k (into the pool at each token's slot) by position,
// with the V rows copied to their slots.
cudaError_t launch_rope_reshape_and_cache(void* q, const void* k, const void* v,
                                          const int32_t* pos, const int32_t* slots,
                                          void* k_pool, void* v_pool, int T, int H_q, int H_kv,
                                          int D, int num_blocks, float theta, bool bf16,
                                          int* err, int num_sms, cudaStream_t stream);

// Speculative acceptance (rejection rule or greedy) of every sequence's k drafts.
struct SpecParams {
  const float* p;          // [B, k + 1, V] target probabilities of the verify rows
  const float* q;          // [B, k, V] draft probabilities, or null (one-hot drafts)
  const int32_t* drafts;   // [B, k]
  const uint32_t* rnd;     // [B, k + 1] random words (rejection rule only)
  int B, k, V, greedy;
  int chunks, chunk;       // vocabulary chunks, greedy rule with 4-byte rows (set by the launcher)
  int runs;                // 128-token runs per row (set by the launcher)
  int gent;                // greedy (max, token) entries per row (set by the launcher)
  int num_sms;
  int vec;                 // rows as float4 loads: V % 4 == 0, p and q 16-byte aligned
  int32_t* out;            // [B, k + 1] accepted drafts, the final token, then -1
  int32_t* num;            // [B] accepted drafts
  long long* wsum;         // [B, runs] workspace: fixed-point residual sums of the runs
  float* amax_v;           // [B, k + 1, gent] workspace: run or chunk maxima (greedy)
  int* amax_i;             // [B, k + 1, gent] workspace: their tokens
  int* acc;                // [B] workspace: accepted drafts | plain << 8 | invalid << 9
  int* err;
};
int spec_chunks(int V);
int spec_runs(int V);
cudaError_t launch_spec_accept(const SpecParams& a, cudaStream_t stream);

// Number of resident attention CTAs and warps per CTA the split kernel uses.
int attention_ctas(int D, int num_sms);
int attention_warps(int D);

// concurrency: split-kernel warps; tile_ctas: tile-kernel CTAs (work is sized for both).
// With p.new_k set, the same launch also carries the step's KV scatter (p.new_k, p.new_v
// into p.k_pool, p.v_pool, slots to p.slots) on extra CTAs beside the planning ones; with
// `pre`, further CTAs make those copies (inputs that only the later kernels read).
cudaError_t launch_plan(const AttnParams& p, int concurrency, int tile_ctas, int num_sms,
                        cudaStream_t stream, const CopySegments* pre = nullptr);

// Query tokens per 128-row tile for G query heads per KV head (0 = use the split kernel).
int tile_tokens(int G);

// The tile kernel on `ctas` CTAs: from the plan's list, or, in direct mode, every
// sequence unsplit from items each CTA derives from seq_lens and qsl (see
// direct_tile_fits).
cudaError_t launch_tile_attention(const AttnParams& p, bool bf16, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, const CUtensorMap& qmap, int ctas,
                                  cudaStream_t stream, bool pdl, bool direct = false);

// Sequences the tile kernel's direct mode takes at most (one warp lane each).
constexpr int kDirectTileMaxSeqs = 32;

// True when a batch with query tiles fits the tile kernel's direct mode: at most
// kDirectTileMaxSeqs sequences, so few that each could have its own tile items, and no
// block table wider than kDirectMaxPages, so no item is long enough to want a split.
bool direct_tile_fits(const AttnParams& p, int num_sms);

// CTAs for the direct tile mode: the items of the batch, bounded from T, B and the tile
// size, at most one per SM.
int direct_tile_ctas(const AttnParams& p, int num_sms);

// CTAs for the split kernel: the full grid, or fewer when the batch's shape (T, B, the
// block-table width) bounds its work items below one per warp of the full grid.
int split_ctas(const AttnParams& p, int num_sms);

cudaError_t launch_split_attention(const AttnParams& p, bool bf16, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int ctas, cudaStream_t stream,
                                   bool pdl);

cudaError_t launch_combine(const AttnParams& p, bool bf16, int num_sms, cudaStream_t stream,
                           bool pdl);

// Largest block-table width (pages) the direct mode takes: one warp streams a sequence's
// whole context, which for this many pages takes no longer than a plan would.
constexpr int kDirectMaxPages = 64;
// Block-table width (pages) up to which the direct mode's ring has two stages.
constexpr int kDirectSmallPages = 8;

// True when a batch of T packed tokens fits the direct mode: every sequence's rows (n * G
// <= T * G) fit one 16-row group, no block table is wide enough for the planner to split a
// row, and the items fit a few waves of the split kernel's warps.
bool direct_fits(const AttnParams& p, int num_sms);

// The whole step in one launch for such a batch: the split kernel in direct mode (p.direct
// and, for a step with K/V to cache, p.new_k / p.new_v / p.k_pool / p.v_pool set).
cudaError_t launch_direct_attention(const AttnParams& p, bool bf16, const CUtensorMap& kmap,
                                    const CUtensorMap& vmap, int num_sms, cudaStream_t stream);

// Workspace bytes before the split partials (header, work lists, per-token tables);
// `headroom` reserves work-list room for splitting long contexts.
size_t workspace_fixed_bytes(int T, int B, int H_q, int H_kv, bool headroom, int* cap_items,
                             int* cap_tile);
size_t partial_bytes(int64_t cap_part, int D);

// Point p's workspace fields into `ws` (bytes long); the partials take what is left. With
// `shrink`, the work lists fall back to their unsplit size when the headroom does not fit.
// False when even that does not fit.
bool layout_workspace(AttnParams& p, uint8_t* ws, size_t bytes, bool shrink);

// The new tokens' K/V to scatter into the pools (the scatter writes their slots into
// AttnParams::slots), and copies still to make before the attention kernels read their
// destinations (the host step's queries): on extra CTAs of the planner's launch, or by a
// gather kernel first when the step has no planner.
struct ScatterArgs {
  const void* k;
  const void* v;
  const CopySegments* pre = nullptr;
};

// Plan, [KV scatter], split kernel, tile kernel, combine on `s` (p's problem and workspace
// fields set). The kernels after the first are chained with programmatic dependent launch.
int run_attention(const AttnParams& p, void* k_pool, void* v_pool, bool bf16, cudaStream_t s,
                  const ScatterArgs* scatter = nullptr);

// Library state of the current device (set up on first use): SM count and the device
// address of the library's device error word. Returns a ps_status.
int current_device(int* num_sms, int** err);

// TMA descriptor of a pool [num_blocks, 16, H_kv, D] as a 2-D tensor [num_blocks * 16,
// H_kv * D] with 64 x 16 boxes and 128-byte swizzle. Returns a ps_status.
int encode_pool_map(CUtensorMap* map, const void* pool, int num_blocks, int H_kv, int D,
                    bool bf16);

}  // namespace ps
