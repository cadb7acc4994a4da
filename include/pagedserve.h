/*
 * pagedserve.h -- C ABI of the GB300 (sm_103a) paged KV attention library.
 *
 * One attention step over a paged KV cache for a packed ragged batch:
 *   1. ps_slot_mapping       -- the pool slot of every packed token;
 *   2. ps_reshape_and_cache  -- scatter each token's K/V row into the pool at its slot;
 *   3. ps_paged_attention    -- causal grouped-query attention of every packed query row
 *                               over its sequence's context, read through block tables.
 *
 * Sources (three web pages on paged KV serving):
 *   - PageServe, section 01 "Scheduler loop": one packed [1, T] forward per step with
 *     explicit position ids and a slot mapping per token; the forward writes K/V into the
 *     pool and reads context via block tables; a token's slot is
 *     block_table[pos // 16] * 16 + pos % 16; every step computes the tokens that do not
 *     yet have K/V ("num_computed_tokens").
 *   - PageServe, section 03 "Paged KV cache" and development-history phases 6-8: fixed
 *     16-token blocks in one pre-allocated pool [layers, blocks, 16, H, D]; per-sequence
 *     block tables; a custom attention backend that scatters new K/V and attends through
 *     the table.
 *   - tinyserve, "How it works": K/V slabs [layers, blocks x 16, H_kv, D] (the same memory
 *     order); shared prefix blocks referenced from several tables; one fused pass over a
 *     flattened ragged batch mixing prefill chunks and decodes; k+1 speculative-verify
 *     tokens scored at once under a stepped causal mask; grouped-query attention
 *     ("Highlights" table, forward-pass row).
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a DEVICE pointer owned by the caller, unless the argument says
 *     otherwise. The library allocates no device memory and keeps no pointer after return.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and returns PS_OK once its kernels are enqueued, or a negative ps_status.
 *     Host-side argument errors are detected before anything is enqueued.
 *   - Tensors are dense and row-major with the shapes given. 16-bit values are IEEE fp16
 *     or bfloat16 as `dtype` says. Tensor pointers must be 16-byte aligned.
 *   - Block size is 16 tokens. head_dim D is 64 or 128. H_q is a multiple of H_kv; query
 *     head h reads KV head h / (H_q / H_kv).
 *   - Device-side index errors (a block id outside the pool, a slot past the pool, a
 *     sequence with more query tokens than context) never trap: the kernel records the
 *     first such error in the library's device error word (ps_get_device_error) and
 *     skips the access; the affected outputs are left unwritten.
 */
#ifndef PAGEDSERVE_H
#define PAGEDSERVE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PS_BLOCK_SIZE 16

typedef enum { PS_F16 = 0, PS_BF16 = 1 } ps_dtype;

typedef enum {
  PS_OK = 0,
  PS_ERR_ARG = -1,          /* a size, count or required pointer is invalid            */
  PS_ERR_UNSUPPORTED = -2,  /* dtype, head_dim or head counts not supported            */
  PS_ERR_ALIGN = -3,        /* a tensor pointer is not 16-byte aligned                 */
  PS_ERR_WORKSPACE = -4,    /* workspace missing, misaligned or too small              */
  PS_ERR_CUDA = -5          /* a CUDA call or kernel launch failed                     */
} ps_status;

/* Device error codes reported by ps_get_device_error. */
typedef enum {
  PS_DEV_OK = 0,
  PS_DEV_BAD_BLOCK_ID = 1,   /* a block-table entry outside [0, num_blocks)            */
  PS_DEV_BAD_SLOT = 2,       /* a slot_mapping entry >= num_blocks * 16                */
  PS_DEV_BAD_SEQUENCE = 3,   /* query count > context, or context beyond the table     */
  PS_DEV_WAIT_TIMEOUT = 4,   /* a kernel's bounded wait ran out (the kernel returned)  */
  PS_DEV_PLAN_OVERFLOW = 5,  /* the work plan did not fit the workspace                */
  PS_DEV_BAD_TOKEN = 6       /* a draft token id outside [0, V)                          */
} ps_device_error;

/*
 * ps_slot_mapping -- slot of every packed query token (PageServe section 01).
 *
 *   block_tables     int32 [B, max_blocks_per_seq]: physical block ids of each sequence;
 *                    entries past a sequence's context are never read.
 *   seq_lens         int32 [B]: context length of each sequence AFTER this step's tokens.
 *   query_start_loc  int32 [B + 1]: packed offsets, [0] = 0, [B] = T, non-decreasing.
 *                    Sequence b owns packed tokens [query_start_loc[b], query_start_loc[b+1]).
 *   slot_mapping     int32 [T], written: for token i of the n_b tokens of sequence b,
 *                    pos = seq_lens[b] - n_b + i and
 *                    slot = block_tables[b][pos / 16] * 16 + pos % 16;
 *                    -1 (and a device error) where the entry would be invalid.
 *   num_blocks       pool size in blocks, for the bounds check.
 * B = 0 requires T = 0. Returns PS_ERR_ARG for negative sizes or null pointers with T > 0.
 */
int ps_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* seq_lens, const int32_t* query_start_loc, int B, int T,
                    int num_blocks, int32_t* slot_mapping, void* stream);

/*
 * ps_reshape_and_cache -- KV scatter (PageServe section 01 "Execute"; section 03).
 *
 *   k, v          [T, H_kv, D] of dtype: the new tokens' keys and values.
 *   slot_mapping  int32 [T]: destination slot of each token; a negative slot skips the
 *                 token; a slot >= num_blocks * 16 is skipped and recorded as
 *                 PS_DEV_BAD_SLOT.
 *   k_pool, v_pool [num_blocks, 16, H_kv, D] of dtype, updated in place:
 *                 pool[slot / 16, slot % 16, :, :] = k[t] (bit-exact copy).
 * Two tokens mapped to one slot leave one of the two rows (which one is unspecified).
 */
int ps_reshape_and_cache(const void* k, const void* v, const int32_t* slot_mapping,
                         void* k_pool, void* v_pool, int T, int H_kv, int D, int num_blocks,
                         int dtype, void* stream);

/*
 * ps_copy_blocks -- copy whole KV blocks between pools, bit-exact.
 *
 * Copy-on-write of a block that several block tables share, before one of them writes
 * into it (tinyserve "How it works"; "Highlights" table, paged KV-cache row), and the
 * swap of a preempted sequence's blocks to a pinned host pool and back (PageServe
 * section 04 "Phase 9 · Preemption"; tinyserve "How it works": swapped KV is lossless).
 *
 *   src_k, src_v   [src_num_blocks, 16, H_kv, D] of dtype: the source pools.
 *   dst_k, dst_v   [dst_num_blocks, 16, H_kv, D] of dtype: the destination pools, updated
 *                  in place. Source and destination may be the same pools (copy-on-write)
 *                  or different ones. Each pool may be DEVICE memory or PINNED HOST memory
 *                  (page-locked and mapped, e.g. cudaHostAlloc): the kernel reads and
 *                  writes it through unified addressing, so a swap out or in is one call.
 *   src_ids, dst_ids  int32 [n], device-accessible (device or pinned host memory): for
 *                  every i, block dst_ids[i] of both destination pools becomes a copy of
 *                  block src_ids[i] of the source pools (all 16 x H_kv x D values).
 * The pairs are copied concurrently: destination ids must be distinct and no block may be
 * both a source and a destination of one call (otherwise the result is unspecified). An
 * id outside its pool records PS_DEV_BAD_BLOCK_ID and that pair is skipped. n = 0 is a
 * no-op.
 */
int ps_copy_blocks(const void* src_k, const void* src_v, int src_num_blocks, void* dst_k,
                   void* dst_v, int dst_num_blocks, const int32_t* src_ids,
                   const int32_t* dst_ids, int n, int H_kv, int D, int dtype, void* stream);

/*
 * ps_rope_reshape_and_cache -- rotary position embedding fused with the KV scatter.
 *
 * Every new token's query and key are rotated by its position before the key is cached
 * (tinyserve "Highlights" table, forward-pass row: rotary embeddings in the Qwen2
 * decoder; PageServe section 01: explicit position ids per packed token). Rotate-half
 * form, for each head and frequency i < D/2, with a = positions[t] * rope_theta^(-2i/D):
 *     x'[i]       = x[i] cos(a) - x[i + D/2] sin(a)
 *     x'[i + D/2] = x[i + D/2] cos(a) + x[i] sin(a)
 * The angle is formed and reduced in fp64, its cosine and sine taken in fp32, and each
 * output rounded once to dtype: within one unit in the last place of the exact value
 * plus 2^-20 (|x[i]| + |x[i + D/2]|), the fp32 cosine's share.
 *
 *   q             [T, H_q, D] of dtype, rotated IN PLACE.
 *   k, v          [T, H_kv, D] of dtype (k is not modified).
 *   positions     int32 [T]: position of each token.
 *   slot_mapping  int32 [T]: as for ps_reshape_and_cache; the rotated key row and the V
 *                 row go to the slot (a negative slot skips the token's K/V, a slot past
 *                 the pool records PS_DEV_BAD_SLOT; q is rotated either way).
 *   k_pool, v_pool [num_blocks, 16, H_kv, D] of dtype, updated in place.
 *   rope_theta    the rotary base (> 1), e.g. 1e6 for Qwen2.5 models.
 */
int ps_rope_reshape_and_cache(void* q, const void* k, const void* v, const int32_t* positions,
                              const int32_t* slot_mapping, void* k_pool, void* v_pool, int T,
                              int H_q, int H_kv, int D, int num_blocks, float rope_theta,
                              int dtype, void* stream);

/*
 * ps_spec_accept -- speculative-decoding acceptance after the verify pass.
 *
 * tinyserve "How it works" (speculative decoding): draft d_i is accepted with probability
 * min(1, p_i(d_i) / q_i(d_i)); at the first rejection the replacement is drawn from
 * normalize(max(p_i - q_i, 0)); if all k drafts survive, a bonus token is drawn from the
 * last target distribution. The greedy rule (temperature 0) accepts a draft while it
 * equals argmax p_i and emits argmax p_i at the first mismatch, or argmax p_k when all
 * match. Randomness is an input, and every decision is fixed to a precision, so the tokens
 * are reproducible:
 *   - acceptance of draft i: (double)R_i * (double)q_i(d_i) < (double)p_i(d_i) * 2^32,
 *     each product rounded once in fp64 (q = 1 when draft_probs is null);
 *   - residual weights w = max(p - q, 0) in fp32 (q the one-hot of the draft token when
 *     draft_probs is null; w = p for the bonus row), as integers W = trunc(w * 2^40);
 *   - the sample is the first token v whose running sum W_0 + ... + W_v exceeds
 *     floor(R_k * Z / 2^32), Z the sum of all W (if Z = 0, the same draw from p itself);
 *   - argmax ties go to the lowest token.
 *
 *   target_probs  float [B, k + 1, V]: p_0 .. p_k of each sequence (the verify rows).
 *   draft_probs   float [B, k, V]: q_0 .. q_{k-1}, or NULL for a deterministic proposer
 *                 (n-gram drafts: q is the one-hot of the draft token).
 *   draft_tokens  int32 [B, k]; an id outside [0, V) records PS_DEV_BAD_TOKEN and counts
 *                 as rejected, its replacement drawn from p alone.
 *   random_bits   uint32 [B, k + 1]: R_0 .. R_{k-1} for the acceptance tests, R_k for the
 *                 final draw; may be NULL when greedy != 0.
 *   out_tokens    int32 [B, k + 1], written: the accepted drafts, then the replacement or
 *                 bonus token, then -1.
 *   num_accepted  int32 [B], written: accepted drafts (0 .. k); num_accepted + 1 tokens
 *                 are emitted.
 *   workspace     device scratch of ps_spec_accept_workspace_size(B, k, V) bytes,
 *                 256-byte aligned.
 * Probabilities are expected in [0, 1]; other values give unspecified tokens, never a
 * fault. B = 0 is a no-op; k = 0 draws one token from p_0; k > 31 or V > 2^30 returns
 * PS_ERR_UNSUPPORTED. Rows are read as 16-byte words when V is a multiple of 4 and both
 * probability arrays are 16-byte aligned, and as 4-byte words otherwise.
 */
size_t ps_spec_accept_workspace_size(int B, int k, int V);
int ps_spec_accept(const float* target_probs, const float* draft_probs,
                   const int32_t* draft_tokens, const uint32_t* random_bits, int B, int k, int V,
                   int greedy, int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * ps_paged_attention_workspace_size -- bytes of device workspace ps_paged_attention wants
 * for a batch of at most T packed tokens, B sequences and contexts of at most
 * max_seq_len tokens. A smaller workspace (at least the size returned for
 * max_seq_len = 0) still works; the attention then splits long contexts into fewer parts.
 * Returns 0 for invalid sizes or head counts, and for a batch whose plan could not be
 * indexed with 32-bit integers (such a batch is rejected by ps_paged_attention too).
 */
size_t ps_paged_attention_workspace_size(int T, int B, int H_q, int H_kv, int D,
                                         int max_seq_len);

/*
 * ps_paged_attention -- causal paged attention over a packed ragged batch.
 *
 * For packed row r = query_start_loc[b] + i of sequence b (n_b rows, context
 * L_b = seq_lens[b], position p = L_b - n_b + i) and query head h, with G = H_q / H_kv:
 *     out[r, h, :] = sum_{j <= p} softmax_j(scale * q[r, h, :] . K_b[j]) V_b[j]
 * where K_b[j] = k_pool[block_tables[b][j / 16], j % 16, h / G, :] (V likewise).
 * One-token decodes, k+1-token speculative-verify rows and prefill chunks mix freely
 * (PageServe section 01; tinyserve "How it works").
 *
 *   q              [T, H_q, D] of dtype.
 *   k_pool, v_pool [num_blocks, 16, H_kv, D] of dtype (already holding this step's K/V).
 *   block_tables, seq_lens, query_start_loc  as for ps_slot_mapping; 0 <= n_b <= L_b.
 *   scale          softmax scale (normally 1 / sqrt(D)).
 *   out            [T, H_q, D] of dtype, written for every packed row.
 *   workspace      device scratch of workspace_bytes bytes, 256-byte aligned, owned by the
 *                  caller; contents on entry are ignored and on return are undefined.
 *                  Calls that share a workspace must not overlap on the device.
 * Accumulation is fp32; the output is rounded to dtype.
 */
int ps_paged_attention(const void* q, const void* k_pool, const void* v_pool,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* seq_lens, const int32_t* query_start_loc, int B, int T,
                       int H_q, int H_kv, int D, int num_blocks, float scale, void* out,
                       void* workspace, size_t workspace_bytes, int dtype, void* stream);

/*
 * ps_paged_attention_noalloc -- ps_paged_attention for callers that cannot allocate.
 *
 * The pages describe no such call; it exists for users of this library. Some callers
 * are handed only their input and output buffers and may not create device memory:
 * a plug-in inside a host framework whose allocator owns all device memory, or a
 * latency-critical loop that must not call cudaMalloc/cudaFree (they can synchronise
 * the device). This variant takes no workspace: its scratch is a fixed device array of
 * PS_NOALLOC_SCRATCH_BYTES compiled into the library, held by every GPU that loads the
 * library until the process exits. Arguments and results are those of
 * ps_paged_attention without workspace/workspace_bytes.
 *
 *   - Returns PS_ERR_WORKSPACE, before doing anything, when the batch needs more scratch
 *     than the fixed maximum (a work list of about H_kv * (T * H_q / H_kv / 16 + B)
 *     64-byte entries plus 8 bytes per token must fit; long contexts are split into
 *     fewer parts when the partials would not fit).
 *   - The first call on each device (with that device current) looks up the array's
 *     device address with cudaGetSymbolAddress; make that first call before any stream
 *     capture.
 *   - Every call reuses the same array and leaves its contents behind; each call
 *     rewrites what it reads. Calls whose kernels overlap on the device (from two
 *     streams or two host threads) race on the array: the caller must serialise them.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
#define PS_NOALLOC_SCRATCH_BYTES (32u << 20)
int ps_paged_attention_noalloc(const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* seq_lens, const int32_t* query_start_loc, int B,
                               int T, int H_q, int H_kv, int D, int num_blocks, float scale,
                               void* out, int dtype, void* stream);

/*
 * ps_attention_step -- the whole step in one call, with the results of ps_slot_mapping,
 * ps_reshape_and_cache and then ps_paged_attention, on one stream (the slot mapping is
 * computed by the attention planner and the kernels are chained with programmatic
 * dependent launch). k, v are the step's new tokens [T, H_kv, D]; slot_mapping is
 * caller-provided device memory of T int32 (written with the slots). Other arguments as
 * above.
 */
int ps_attention_step(const void* q, const void* k, const void* v, void* k_pool, void* v_pool,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* seq_lens, const int32_t* query_start_loc, int B, int T,
                      int H_q, int H_kv, int D, int num_blocks, float scale, void* out,
                      int32_t* slot_mapping, void* workspace, size_t workspace_bytes,
                      int dtype, void* stream);

/*
 * ps_attention_step_host -- one step from HOST buffers: copies the step's inputs to the
 * device, runs ps_attention_step, and copies the output back, all on `stream`.
 *
 *   q, k, v, block_tables, seq_lens, query_start_loc   HOST pointers (pinned memory lets
 *                  the copies run asynchronously), shapes as for ps_attention_step.
 *   out            HOST pointer [T, H_q, D] of dtype; valid once `stream` has completed.
 *   k_pool, v_pool DEVICE pointers: the resident KV cache, updated in place.
 *   staging        DEVICE scratch of at least ps_attention_step_host_staging_size() bytes,
 *                  256-byte aligned, owned by the caller (inputs, slot mapping, output and
 *                  the attention workspace are placed in it).
 * Host memory must stay valid and unmodified until the stream completes. Page-locked host
 * arrays that the device can address (pinned and mapped, 4-byte aligned) are read by one
 * kernel that gathers all such inputs across the host link; such k and v (16-byte aligned)
 * are instead read by the step's KV scatter directly. Such an `out` (16-byte aligned)
 * is written by the step's kernels themselves when it is at most 4 MB, and otherwise by a
 * kernel after the step's last one; any other array is copied with one cudaMemcpyAsync.
 */
size_t ps_attention_step_host_staging_size(int T, int B, int max_blocks_per_seq, int H_q,
                                           int H_kv, int D, int max_seq_len);

/*
 * ps_attention_step_host_graph_create -- ps_attention_step_host recorded once into a CUDA
 * graph, so that a serving loop pays one graph launch per step instead of the copies' and
 * kernels' launch costs (PageServe, "Next steps": CUDA graphs for decode, against Python
 * and launch overhead at small batch sizes).
 *
 *   Arguments as ps_attention_step_host, without the stream; `graph` receives an opaque
 *   handle. Nothing runs at creation: the pools are not touched.
 *   Each ps_graph_launch(graph, stream) copies the CURRENT contents of the host buffers q,
 *   k, v, block_tables, seq_lens, query_start_loc to the device, runs the step and copies
 *   the output to `out`, as one call of ps_attention_step_host with the same arguments
 *   would. Shapes (T, B, max_blocks_per_seq, heads, D, num_blocks) are fixed at creation;
 *   the contents (lengths, block tables, tokens) may change between launches, with lengths
 *   within the max_seq_len `staging` was sized for (longer ones get fewer splits, and
 *   PS_DEV_PLAN_OVERFLOW if even those do not fit).
 *   The host buffers must be page-locked (cudaHostAlloc, cudaHostRegister); a host pointer
 *   that is not is rejected with PS_ERR_ARG before anything is recorded.
 *   Ownership: the caller keeps every buffer alive, in place and page-locked while the
 *   graph exists; ps_graph_destroy releases the graph.
 * Errors: PS_ERR_ARG for a null `graph` or a host buffer that is not page-locked; those of
 * ps_attention_step_host's argument checks; PS_ERR_CUDA if the capture or instantiation
 * fails. The handle is set only on success.
 */
int ps_attention_step_host_graph_create(const void* q, const void* k, const void* v,
                                        const int32_t* block_tables, const int32_t* seq_lens,
                                        const int32_t* query_start_loc, void* out,
                                        void* k_pool, void* v_pool, int max_blocks_per_seq,
                                        int B, int T, int H_q, int H_kv, int D, int num_blocks,
                                        float scale, void* staging, size_t staging_bytes,
                                        int dtype, void** graph);
/* Launch a graph from ps_attention_step_host_graph_create on `stream` (asynchronous; the
 * output is valid once the stream has completed). PS_ERR_ARG for a null handle. */
int ps_graph_launch(void* graph, void* stream);
/* Release a graph (after its last launch has completed). PS_ERR_ARG for a null handle. */
int ps_graph_destroy(void* graph);
int ps_attention_step_host(const void* q, const void* k, const void* v,
                           const int32_t* block_tables, const int32_t* seq_lens,
                           const int32_t* query_start_loc, void* out, void* k_pool,
                           void* v_pool, int max_blocks_per_seq, int B, int T, int H_q,
                           int H_kv, int D, int num_blocks, float scale, void* staging,
                           size_t staging_bytes, int dtype, void* stream);

/*
 * ps_get_device_error -- read (and clear) the device error word of the current device.
 * Synchronises with the device. *code receives a ps_device_error value. Returns PS_OK or
 * PS_ERR_CUDA / PS_ERR_ARG.
 */
int ps_get_device_error(int* code);

/*
 * ps_last_error_message -- after a call returned PS_ERR_CUDA, the step that failed and
 * CUDA's message, for the calling host thread ("" if none). The string stays valid until
 * the next failing call on the same thread.
 */
const char* ps_last_error_message(void);

/* Human-readable name of a ps_status value. The string is static. */
const char* ps_status_string(int status);

/*
 * Kernel timing hook for benchmarks. ps_profile_begin(n) starts recording CUDA events
 * around the next n launches of each kernel kind (host memory only; events are created
 * here, not in the timed calls). ps_profile_end() waits for the recorded events and
 * stops recording. ps_profile_read(kind, &ms, &launches) then gives the summed device
 * time and the launch count of one kind: 0 slot mapping, 1 KV scatter as its own launch
 * (ps_reshape_and_cache, or the step's scatter ahead of the tile kernel's direct mode),
 * 2 planner (carrying the step's KV scatter when there is one), 3 split attention (decode
 * and verify rows), 4 split combine, 5 tile attention (prefill rows, tcgen05), 6 block
 * copy, 7 speculative acceptance, 8 rotary KV scatter.
 */
int ps_profile_begin(int max_launches_per_kind);
int ps_profile_end(void);
int ps_profile_read(int kind, float* total_ms, int* launches);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDSERVE_H */
