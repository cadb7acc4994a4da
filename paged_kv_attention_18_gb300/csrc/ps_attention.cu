// Paged attention over a packed ragged batch: planner, split kernel, split-combine.
//
// What is computed (PageServe section 01 "Execute": the backend reads each sequence's
// context through its block table; tinyserve "How it works": one fused pass over a
// flattened ragged batch, the stepped causal mask for k+1 verify tokens, grouped-query
// attention): for every packed query row r of sequence b at position
// p = L_b - n_b + i and every query head h,
//     out[r, h] = softmax_j<=p( q[r, h] . K_b[j, h / G] * scale ) . V_b[j, h / G]
// with K_b[j] read from the pool row block_table[b][j / 16] * 16 + j % 16.
//
// Design (GB300): a multi-CTA planner (up to 64 CTAs, each repeating the per-sequence
// scan) turns the batch into work items on the device
// (16 packed rows = query tokens x GQA heads of one KV head, over one split of the
// context); a persistent split kernel lets every warp fetch items from an atomic
// counter and stream the item's K/V pages through its own ring of TMA-filled shared
// memory stages (128-byte swizzled, one mbarrier per stage), computing QK^T and PV with
// mma.sync and an online softmax in registers; a combine kernel merges the splits of
// rows whose context was split, by log-sum-exp weights.
#include "ps_common.cuh"
#include "ps_launch.h"
#include "ps_scatter.cuh"

namespace ps {

// ----------------------------------------------------------------------------------
// planner
// ----------------------------------------------------------------------------------
struct SeqInfo {
  int n, L, valid, groups, pages, tok0, tile, qtiles;
};

// groups: 16-row groups of the split kernel; tile / qtiles: the sequence goes to the tile
// kernel (more than 16 packed rows and a tile size exists) in qtiles 128-row tiles.
__device__ __forceinline__ SeqInfo seq_info(const AttnParams& p, const int* qsl,
                                            const int* lens, int b) {
  SeqInfo s;
  s.tok0 = qsl[b];
  s.n = qsl[b + 1] - s.tok0;
  s.L = lens[b];
  s.pages = (s.L + kBlockSize - 1) / kBlockSize;
  s.valid = s.n >= 0 && s.n <= s.L && s.pages <= p.max_blocks;
  const int rows = s.valid ? s.n * p.G : 0;
  s.groups = (rows + 15) / 16;
  s.tile = p.tpt > 0 && (s.groups > kTileMinGroups || (p.all_tiles && s.groups > 0));
  s.qtiles = s.tile ? (s.n + p.tpt - 1) / p.tpt : 0;
  return s;
}

__device__ __forceinline__ int seq_splits(const SeqInfo& s, int pps_dec, int pps_tile) {
  if (s.groups == 0) return 0;
  int pps;
  if (s.tile) {
    pps = pps_tile;
  } else {
    if (s.groups > kSplitGroupLimit) return 1;
    pps = pps_dec;
  }
  int ns = (s.pages + pps - 1) / pps;
  ns = ns < 1 ? 1 : ns;
  ns = ns > kMaxSplits ? kMaxSplits : ns;
  return ns > s.pages ? s.pages : ns;
}

// largest b in [0, n) with arr[b] <= x (arr non-decreasing, arr[0] <= x)
__device__ __forceinline__ int last_le(const int* arr, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (arr[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Exclusive scan over the block (blockDim.x a multiple of 32, at most 1024).
__device__ int block_exscan(int v, int* sh, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nw ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;
  }
  __syncthreads();
  const int prefix = wid ? sh[wid - 1] : 0;
  total = sh[nw - 1];
  __syncthreads();
  return prefix + x - v;
}

// Exclusive scan of four counters at once (one set of barriers for all four).
__device__ int4 block_exscan4(int4 v, int4* sh, int4& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int4 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, x.x, o), b = __shfl_up_sync(0xffffffffu, x.y, o);
    const int c = __shfl_up_sync(0xffffffffu, x.z, o), d = __shfl_up_sync(0xffffffffu, x.w, o);
    if (lane >= o) {
      x.x += a;
      x.y += b;
      x.z += c;
      x.w += d;
    }
  }
  if (lane == 31) sh[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int4 w = lane < nw ? sh[lane] : make_int4(0, 0, 0, 0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, w.x, o), b = __shfl_up_sync(0xffffffffu, w.y, o);
      const int c = __shfl_up_sync(0xffffffffu, w.z, o), d = __shfl_up_sync(0xffffffffu, w.w, o);
      if (lane >= o) {
        w.x += a;
        w.y += b;
        w.z += c;
        w.w += d;
      }
    }
    sh[lane] = w;
  }
  __syncthreads();
  const int4 pre = wid ? sh[wid - 1] : make_int4(0, 0, 0, 0);
  total = sh[nw - 1];
  __syncthreads();
  return make_int4(pre.x + x.x - v.x, pre.y + x.y - v.y, pre.z + x.z - v.z, pre.w + x.w - v.w);
}

// Token i (0-based within its sequence, at position L - n + i) lies on page (L - n + i) / 16;
// split k of a sequence split ns ways starts at page (k * pages) / ns, so the first token
// that split k covers is first_k = max(0, 16 * start_k - (L - n)). A token's rows are held
// by the splits with first_k <= i; with more than one, each holds H_q partial entries.
__device__ __forceinline__ int split_first_token(const SeqInfo& s, int ns, int k) {
  const int f = (k * s.pages) / ns * kBlockSize - (s.L - s.n);
  return f > 0 ? f : 0;
}

// For token i: the splits holding its rows (*held) and, summed over the tokens before it,
// the splits holding each token held by at least two (the tokens from first_1 on). The
// split starts k * pages / ns are stepped with a running remainder, without dividing.
__device__ __forceinline__ int split_entries_before(const SeqInfo& s, int ns, int i,
                                                    int* held = nullptr) {
  const int q = s.pages / ns, r = s.pages - q * ns, p0 = s.L - s.n;
  const int f1 = max(0, q * kBlockSize - p0);  // start_1 = q (r < ns)
  int acc = 0, cnt = 0, start = 0, rem = 0;
  for (int k = 0; k < ns; ++k) {
    const int fk = max(0, start * kBlockSize - p0);
    cnt += fk <= i ? 1 : 0;
    const int from = fk > f1 ? fk : f1;
    acc += i > from ? i - from : 0;
    start += q;
    rem += r;
    if (rem >= ns) {
      rem -= ns;
      ++start;
    }
  }
  if (held) *held = cnt;
  return acc;
}

// Sums of three values over the block, returned to every thread.
struct Sum3 {
  long long x, y, z;
};
__device__ Sum3 block_sum3_ll(Sum3 v, Sum3* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
  }
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  if (wid == 0) {
    Sum3 w = lane < nw ? sh[lane] : Sum3{0, 0, 0};
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      w.x += __shfl_xor_sync(0xffffffffu, w.x, o);
      w.y += __shfl_xor_sync(0xffffffffu, w.y, o);
      w.z += __shfl_xor_sync(0xffffffffu, w.z, o);
    }
    if (lane == 0) sh[0] = w;
  }
  __syncthreads();
  const Sum3 t = sh[0];
  __syncthreads();
  return t;
}

// Items per worker that the split sizes aim at: more items balance the workers' ends
// better, fewer carry less per-item cost (query load, partial output, combine).
#ifndef PS_SPLIT_ITEMS_PER_WORKER
#define PS_SPLIT_ITEMS_PER_WORKER 4
#endif

__device__ __forceinline__ int pages_per_split(long long work, long long workers, int align) {
  const long long target = workers * PS_SPLIT_ITEMS_PER_WORKER;
  long long pps = (work + target - 1) / (target > 0 ? target : 1);
  if (pps < kMinSplitPages) pps = kMinSplitPages;
  pps = (pps + align - 1) / align * align;
  return static_cast<int>(pps > (1 << 24) ? (1 << 24) : pps);
}

// Split-kernel items go out longest first, by class of their length in pages: 0 for
// items longer than the target (sequences at the split cap), then by quarters of the
// target. Items are fetched in list order, so the short ones fill the workers' ends.
__device__ __forceinline__ int split_class(const SeqInfo& s, int ns, int pps) {
  const int len = (s.pages + ns - 1) / ns;
  return len > pps ? 0 : 4 * len > 3 * pps ? 1 : 2 * len > pps ? 2 : 3;
}
__device__ __forceinline__ int int4_at(const int4& v, int k) {
  return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

__device__ __forceinline__ void store_item(WorkItem* dst_item, const WorkItem& it) {
  const int4* src = reinterpret_cast<const int4*>(&it);
  int4* dst = reinterpret_cast<int4*>(dst_item);
  dst[0] = src[0];
  dst[1] = src[1];
  dst[2] = src[2];
  dst[3] = src[3];
}

// The planner turns the batch into two work lists: split-kernel items (sequences with at
// most 64 packed rows: decodes, verify rows) and tile-kernel items (prefill chunks), plus
// the per-token split table that the combine kernel reads and the slot of every new
// token. Every count is taken per sequence (one scan over the batch); the token table
// follows from closed forms per sequence. Each CTA of the grid repeats the scan (the
// results are identical) and then writes its own share of the tokens and of the
// sequences' items, so no CTA waits on another. The per-sequence metadata is staged in
// shared memory when the batch is small enough (kPlanSmemSeqs sequences).
constexpr int kPlanSmemSeqs = 4096;
constexpr int kPlanSmemArrays = 9;  // qsl, lens, five offset arrays, two tile lists; B + 1 ints each
constexpr int kPlanRankSeqs = 512;  // tile sequences up to which every rank goes rank by rank
constexpr int kPlanMaxCtas = 64;

__global__ void __launch_bounds__(1024) plan_kernel(const AttnParams p, int concurrency,
                                                    int tile_ctas, int plan_ctas,
                                                    const CopySegments pre, int copy_ctas) {
  __shared__ int4 sh4[32];
  __shared__ Sum3 shl[32];
  extern __shared__ int plan_smem[];
  const int tid = threadIdx.x, nth = blockDim.x;
  // First in the chain, every CTA waits for the previous work on the stream before it
  // reads anything. CTAs plan_ctas and up carry the step's KV scatter (when p.new_k is
  // set), beside the planning CTAs: the attention kernels' wait on this grid then covers
  // both, at the cost of one launch. The planning CTAs let the attention kernels launch
  // only once their lists are written: those CTAs, resident early and waiting, slowed the
  // planner's own passes.
  pdl_wait();
  // The last copy_ctas CTAs copy inputs that only the later kernels read (the queries,
  // from page-locked host memory), beside the planning and the scatter.
  const int first_copy = static_cast<int>(gridDim.x) - copy_ctas;
  if (static_cast<int>(blockIdx.x) >= first_copy) {
    copy_segments(pre, static_cast<int64_t>(static_cast<int>(blockIdx.x) - first_copy) * nth + tid,
                  static_cast<int64_t>(copy_ctas) * nth);
    return;
  }
  if (static_cast<int>(blockIdx.x) >= plan_ctas) {
    scatter_step_tokens(static_cast<const uint4*>(p.new_k), static_cast<const uint4*>(p.new_v),
                        p.block_tables, p.max_blocks, p.seq_lens, p.qsl, p.B, p.T,
                        p.H_kv * p.D / 8, p.num_blocks, p.slots, static_cast<uint4*>(p.k_pool),
                        static_cast<uint4*>(p.v_pool), p.err,
                        (static_cast<int>(blockIdx.x) - plan_ctas) * (nth >> 5) + (tid >> 5),
                        (first_copy - plan_ctas) * (nth >> 5));
    return;
  }
  const bool in_smem = p.B <= kPlanSmemSeqs;
  const int* qsl = p.qsl;
  const int* lens = p.seq_lens;
  int* off_d = p.seq_off;
  int* off_t = p.seq_off_t;
  int* off_p = p.seq_off_p;
  int* off_s = p.seq_off_s;
  if (in_smem) {
    int* s_qsl = plan_smem;
    int* s_len = s_qsl + (p.B + 1);
    for (int b = tid; b <= p.B; b += nth) s_qsl[b] = p.qsl[b];
    for (int b = tid; b < p.B; b += nth) s_len[b] = p.seq_lens[b];
    qsl = s_qsl;
    lens = s_len;
    off_d = s_len + (p.B + 1);
    off_t = off_d + (p.B + 1);
    off_p = off_t + (p.B + 1);
    off_s = off_p + (p.B + 1);
    __syncthreads();
  }

  // cost of the batch in pages read, per kernel
  long long wd = 0, wt = 0, pairs = 0;
  for (int b = tid; b < p.B; b += nth) {
    const SeqInfo s = seq_info(p, qsl, lens, b);
    if (!s.valid) {
      record_error(p.err, kDevBadSequence);
      continue;
    }
    if (s.tile) {
      wt += static_cast<long long>(s.qtiles) * s.pages;
      pairs += (s.qtiles + 1) / 2;
    } else {
      wd += static_cast<long long>(s.groups) * s.pages;
    }
  }
  const Sum3 W = block_sum3_ll(Sum3{wd, wt, pairs}, shl);
  const long long Wd = W.x * p.H_kv, Wt = W.y * p.H_kv;
  int pps_d = pages_per_split(Wd, concurrency, 1);
  // Tile items carry a fixed cost (query tiles loaded, the output written), so prefill
  // chunks split their context only when the batch has fewer unsplit tile items than half
  // the tile kernel's CTAs (few short chunks, or short chunks at the end of long contexts).
  int pps_t = 2 * W.z * p.H_kv < tile_ctas ? pages_per_split(Wt, tile_ctas, kTilePagesAlign)
                                            : (1 << 24);
#ifdef PS_TILE_ALL_NOSPLIT
  if (p.all_tiles) pps_t = 1 << 24;
#endif

  // per sequence: split-kernel items, tile-kernel items (pairs of query tiles), partial
  // entries and split tokens; coarser splits while the lists overflow the workspace
  // (split-kernel items: the offset within the sequence's length class, run_d the
  // classes' sizes)
  int4 tot = make_int4(0, 0, 0, 0), run_d = make_int4(0, 0, 0, 0);
  for (int attempt = 0; attempt < 32; ++attempt) {
    int4 run = make_int4(0, 0, 0, 0);
    run_d = make_int4(0, 0, 0, 0);
    for (int base = 0; base < p.B; base += nth) {
      const int b = base + tid;
      int4 c = make_int4(0, 0, 0, 0), cd = make_int4(0, 0, 0, 0);
      int kd = 0;
      if (b < p.B) {
        const SeqInfo s = seq_info(p, qsl, lens, b);
        const int ns = seq_splits(s, pps_d, pps_t);
        if (s.tile) {
          c.y = (s.qtiles + 1) / 2 * ns * p.H_kv;
        } else if (ns > 0) {
          c.x = s.groups * ns * p.H_kv;
          kd = split_class(s, ns, pps_d);
          cd = make_int4(kd == 0 ? c.x : 0, kd == 1 ? c.x : 0, kd == 2 ? c.x : 0,
                         kd == 3 ? c.x : 0);
        }
        if (ns > 1) {
          c.z = split_entries_before(s, ns, s.n) * p.H_q;
          c.w = s.n - split_first_token(s, ns, 1);
        }
      }
      int4 t4, td;
      const int4 ex = block_exscan4(c, sh4, t4);
      const int4 exd = block_exscan4(cd, sh4, td);
      if (b < p.B) {
        off_d[b] = int4_at(run_d, kd) + int4_at(exd, kd);
        off_t[b] = run.y + ex.y;
        off_p[b] = run.z + ex.z;
        off_s[b] = run.w + ex.w;
      }
      run.x += t4.x;
      run.y += t4.y;
      run.z += t4.z;
      run.w += t4.w;
      run_d.x += td.x;
      run_d.y += td.y;
      run_d.z += td.z;
      run_d.w += td.w;
    }
    tot = run;
    if (tot.x <= p.cap_items && tot.y <= p.cap_tile && tot.z <= p.cap_part) break;
    if (pps_d >= (1 << 24) && pps_t >= (1 << 24)) {  // cannot shrink further
      record_error(p.err, kDevPlanOverflow);
      tot = make_int4(0, 0, 0, 0);
      break;
    }
    pps_d = pps_d >= (1 << 23) ? (1 << 24) : 2 * pps_d;
    pps_t = pps_t >= (1 << 23) ? (1 << 24) : 2 * pps_t;
  }
  if (tid == 0) {
    off_d[p.B] = tot.x;
    off_t[p.B] = tot.y;
    off_p[p.B] = tot.z;
    off_s[p.B] = tot.w;
  }
  __syncthreads();
  const bool planned = tot.x > 0 || tot.y > 0;

  // Tile items go out longest first. A sequence's rank-r items are its r-th longest pair
  // of query tiles (for every KV head and split); the items go rank by rank, and within a
  // rank sequence by sequence. Rank r starts after C(r) = sum over tile sequences of
  // width * min(pairs, r) items, and sequence b's block within it after the widths of the
  // earlier sequences that have a rank r. For the ranks every tile sequence has (r < rc)
  // that is r * (total width) + off_w[b]; beyond them it is summed over a compact list of
  // the tile sequences (when there are at most kPlanRankSeqs of them; otherwise those ranks
  // follow sequence by sequence). Batches not staged in shared memory keep rc = 0 and the
  // sequence order.
  __shared__ int s_rc;
  int rc = 0, n_tile = 0;
  int* off_w = in_smem ? off_s + (p.B + 1) : nullptr;   // width prefix (KV heads x splits)
  int* tl_np = in_smem ? off_w + (p.B + 1) : nullptr;   // compact list: pairs of each
  int* tl_w = in_smem ? tl_np + (p.B + 1) : nullptr;    // tile sequence, and its width
  if (planned && tot.y > 0 && in_smem) {
    if (tid == 0) s_rc = 1 << 30;
    __syncthreads();
    int run_w = 0, run_n = 0;
    for (int base = 0; base < p.B; base += nth) {
      const int b = base + tid;
      int wb = 0, npb = 0;
      if (b < p.B) {
        const SeqInfo s = seq_info(p, qsl, lens, b);
        if (s.valid && s.tile) {
          wb = seq_splits(s, pps_d, pps_t) * p.H_kv;
          npb = (s.qtiles + 1) / 2;
          atomicMin(&s_rc, npb);
        }
      }
      int4 t4;
      const int4 ex = block_exscan4(make_int4(wb, wb > 0 ? 1 : 0, 0, 0), sh4, t4);
      if (b < p.B) {
        off_w[b] = run_w + ex.x;
        if (wb > 0) {
          tl_np[run_n + ex.y] = npb;
          tl_w[run_n + ex.y] = wb;
        }
      }
      run_w += t4.x;
      run_n += t4.y;
    }
    if (tid == 0) off_w[p.B] = run_w;
    __syncthreads();
    rc = s_rc;
    n_tile = run_n;
  }

  // tokens: splits holding the rows, first partial entry and the combine's token list. The
  // tokens are dealt to the CTAs in blocks of nth, round robin, four per thread and round.
  constexpr int kTokUnroll = 4;
  const int tok_stride = plan_ctas * nth;
  // the token pass starts from the block's upper half: with few tokens it then runs on
  // other warps than the item pass below, which deals sequences to the low warps first
  const int ttid = (tid + nth / 2) % nth;
  for (int base = blockIdx.x * nth; base < p.T; base += kTokUnroll * tok_stride) {
#pragma unroll
    for (int u = 0; u < kTokUnroll; ++u) {
      const int t = base + u * tok_stride + ttid;
      if (t >= p.T) continue;
      const int b = last_le(qsl, p.B, t);
      const SeqInfo s = seq_info(p, qsl, lens, b);
      const int i = t - s.tok0;
      int ns_t = 0, tb = 0;
      if (planned && s.valid && s.groups > 0) {
        const int ns = seq_splits(s, pps_d, pps_t);
        ns_t = 1;
        if (ns > 1) {
          tb = off_p[b] + split_entries_before(s, ns, i, &ns_t) * p.H_q;
          const int f1 = split_first_token(s, ns, 1);
          if (i >= f1) p.tok_list[off_s[b] + (i - f1)] = t;
        }
      }
      p.tok_ns[t] = ns_t;
      p.tok_base[t] = tb;
    }
  }

  // work items, one warp per sequence: split-kernel items with the group index fastest
  // (rows sharing pages run back to back); tile-kernel items as pairs of consecutive query
  // tiles (A, B), placed in the rank order above
  const int lane = tid & 31, nw = nth >> 5;
  const int gw = (tid >> 5) * plan_ctas + blockIdx.x;  // sequences dealt across the CTAs
  for (int b = planned ? gw : p.B; b < p.B; b += plan_ctas * nw) {
    const SeqInfo s = seq_info(p, qsl, lens, b);
    if (!s.valid || s.groups == 0) continue;
    const int ns = seq_splits(s, pps_d, pps_t);
    if (!s.tile) {
      const int kd = split_class(s, ns, pps_d);
      const int cls_base = (kd > 0 ? run_d.x : 0) + (kd > 1 ? run_d.y : 0) + (kd > 2 ? run_d.z : 0);
      const int cnt = s.groups * ns * p.H_kv, first = cls_base + off_d[b], rows = s.n * p.G;
      for (int local = lane; local < cnt; local += 32) {
        const int j = local % s.groups;
        const int rest = local / s.groups;
        const int kv = rest % p.H_kv;
        const int sp = rest / p.H_kv;
        WorkItem it;
        it.seq = b;
        it.kv = kv;
        it.row0 = 16 * j;
        it.nrows = min(16, rows - 16 * j);
        const int i_last = (it.row0 + it.nrows - 1) / p.G;
        const int page_last = (s.L - s.n + i_last) / kBlockSize;
        it.page_begin = (sp * s.pages) / ns;
        it.page_end = min(((sp + 1) * s.pages) / ns, page_last + 1);
        it.split = sp;
        it.nsplit = ns;
        it.ctx_len = s.L;
        it.n_query = s.n;
        it.tok0 = s.tok0;
        it.pad[0] = it.pad[1] = it.pad[2] = it.pad[3] = it.pad[4] = 0;
        store_item(p.items + first + local, it);
      }
    } else {
      const int npairs = (s.qtiles + 1) / 2;
      const int wb = ns * p.H_kv, cnt = npairs * wb, first = off_t[b];
      const int width = rc > 0 ? off_w[p.B] : 0, ow = rc > 0 ? off_w[b] : 0;
      const bool by_rank = rc > 0 && n_tile <= kPlanRankSeqs;
      for (int local = lane; local < cnt; local += 32) {
        const int r = local % npairs;  // rank: 0 is the longest pair
        const int j = npairs - 1 - r;
        const int rest = local / npairs;  // split * H_kv + KV head
        int pos;
        if (r < rc) {
          pos = r * width + ow + rest;
        } else if (by_rank) {
          // C(r) over every tile sequence, plus the earlier sequences that have rank r;
          // the compact list keeps batch order, so "earlier" is a prefix of width ow
          int c = 0, before = 0, seen_w = 0;
          for (int k = 0; k < n_tile; ++k) {
            const int nk = tl_np[k], wk = tl_w[k];
            c += wk * min(nk, r);
            if (seen_w < ow && nk > r) before += wk;
            seen_w += wk;
          }
          pos = c + before + rest;
        } else {
          pos = rc * width + (first - rc * ow) + (r - rc) * wb + rest;
        }
        const int kv = rest % p.H_kv;
        const int sp = rest / p.H_kv;
        const int qa = 2 * j * p.tpt, qb = qa + p.tpt;  // first query of tiles A and B
        const int na = min(p.tpt, s.n - qa), nb = qb < s.n ? min(p.tpt, s.n - qb) : 0;
        WorkItem it;
        it.seq = b;
        it.kv = kv;
        it.row0 = qa * p.G;
        it.nrows = na * p.G;
        const int i_last = nb > 0 ? qb + nb - 1 : qa + na - 1;
        const int page_last = (s.L - s.n + i_last) / kBlockSize;
        it.page_begin = (sp * s.pages) / ns;
        it.page_end = min(((sp + 1) * s.pages) / ns, page_last + 1);
        it.split = sp;
        it.nsplit = ns;
        it.ctx_len = s.L;
        it.n_query = s.n;
        it.tok0 = s.tok0;
        it.pad[0] = nb * p.G;
        it.pad[1] = it.pad[2] = it.pad[3] = it.pad[4] = 0;
        store_item(p.tile_items + pos, it);
      }
    }
  }
  pdl_launch_dependents();
  if (blockIdx.x == 0 && tid == 0) {
    p.hdr[0] = tot.x;
    p.hdr[1] = 0;
    p.hdr[2] = pps_d;
    p.hdr[3] = tot.z;
    p.hdr[4] = tot.y;
    p.hdr[5] = 0;
    p.hdr[6] = pps_t;
    p.hdr[7] = planned ? tot.w : 0;
  }
}

// ----------------------------------------------------------------------------------
// split kernel: one warp = one work item at a time
// ----------------------------------------------------------------------------------
// Shape of the split kernel: warps per CTA, ring stages per warp (one page of K and V per
// stage) and CTAs per SM. Overridable at build time for tuning sweeps.
#ifndef PS_SPLIT_WARPS
#define PS_SPLIT_WARPS 8
#endif
#ifndef PS_SPLIT_STAGES
#define PS_SPLIT_STAGES 3
#endif
#ifndef PS_SPLIT_CTAS_PER_SM
#define PS_SPLIT_CTAS_PER_SM 1
#endif
template <int D>
struct SplitCfg;
template <>
struct SplitCfg<128> {
  static constexpr int kWarps = PS_SPLIT_WARPS, kStages = PS_SPLIT_STAGES;
};
template <>
struct SplitCfg<64> {
  static constexpr int kWarps = PS_SPLIT_WARPS, kStages = 2 * PS_SPLIT_STAGES;
};

// kS > 0 overrides the ring's stage count (the direct mode's small ring for short
// contexts, see launch_split_attention).
template <int D, int kS = 0>
constexpr int split_stages() {
  return kS > 0 ? kS : SplitCfg<D>::kStages;
}
template <int D, int kS = 0>
constexpr int split_smem_bytes() {
  return 1024 /*alignment slack*/ +
         SplitCfg<D>::kWarps * split_stages<D, kS>() * (2 * kBlockSize * D * 2) +
         SplitCfg<D>::kWarps * split_stages<D, kS>() * 8 +
         SplitCfg<D>::kWarps * (split_stages<D, kS>() + 2) * 64;
}

template <bool kBF16, int D, bool kDirect, int kS = 0>
__global__ void __launch_bounds__(SplitCfg<D>::kWarps * 32, PS_SPLIT_CTAS_PER_SM)
    split_attention_kernel(const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
  constexpr int W = SplitCfg<D>::kWarps;
  constexpr int S = split_stages<D, kS>();
  constexpr int kRing = S + 2;
  constexpr int kPage = kBlockSize * D * 2;  // bytes of one page of K (or V), one head
  constexpr int kStage = 2 * kPage;
  constexpr int kBoxes = D / 64;             // 64-element (128-byte) boxes per row
  constexpr int kKSteps = D / 16;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* tiles = smem + warp * S * kStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + W * S * kStage) + warp * S;
  WorkItem* ring =
      reinterpret_cast<WorkItem*>(smem + W * S * kStage + W * S * 8) + warp * kRing;
  const uint32_t tiles_addr = smem_u32(tiles);

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  __syncwarp();
  pdl_wait();  // the plan (and the KV scatter) before this kernel are complete
  // Dependents launch only now: the tile kernel after this one reads the plan without a
  // wait of its own.
  pdl_launch_dependents();

  // direct mode: one item per (sequence, KV head), handed out round robin; otherwise the
  // plan's list, fetched through its counter
  const int n_items = kDirect ? p.B * p.H_kv : *reinterpret_cast<volatile int*>(p.hdr);
  int direct_next = blockIdx.x * W + warp;
  bool first_fetch = true;
  const bool tile_planned = !kDirect && *reinterpret_cast<volatile int*>(p.hdr + 4) > 0;
  const uint64_t policy = l2_policy_evict_first();

  // ---------------- issue side (runs ahead of compute by up to S pages) -------------
  int iss_page = 0, iss_end = 0, iss_seq = 0, iss_kv = 0;
  int bt_base = 0, bt_reg = -1;
  bool no_more = false;
  uint32_t g_issue = 0, ring_tail = 0;

  auto load_bt = [&](int first) {
    bt_base = first;
    const int pg = first + lane;
    bt_reg = pg < iss_end
                 ? __ldg(p.block_tables + static_cast<int64_t>(iss_seq) * p.max_blocks + pg)
                 : -1;
  };

  // Direct mode: the record of item idx = (sequence idx / H_kv, KV head idx % H_kv), all
  // of the sequence's rows (n * G <= 16) over its whole context, in one split; lane k
  // returns field k, and bt_lane the sequence's block-table entry for page `lane`. With
  // the step's K/V given, the sequence's new rows of this head are written to the pools
  // at their slots (the head-0 warp also records the slots), exactly as the step's scatter
  // does, just before the first page holding one of them is copied (scatter_new below).
  // An invalid sequence records an error, gives an empty item and slots of -1.
  int dir_seq = 0, dir_kv = 0, dir_q0 = 0, dir_n = 0, dir_L = 0, dir_first_new = 0;
  bool dir_pending = false;
  auto scatter_new = [&](int bt_lane, bool bad) {
    constexpr int kVecs = D / 8;  // 16-byte chunks of one head's row
    const int32_t* bt = p.block_tables + static_cast<int64_t>(dir_seq) * p.max_blocks;
    for (int t = 0; t < dir_n; ++t) {
      const int64_t src = (static_cast<int64_t>(dir_q0 + t) * p.H_kv + dir_kv) * kVecs + lane;
      uint4 kk = make_uint4(0, 0, 0, 0), vv = kk;
      if (!bad && lane < kVecs) {
        kk = __ldcs(static_cast<const uint4*>(p.new_k) + src);
        vv = __ldcs(static_cast<const uint4*>(p.new_v) + src);
      }
      int slot = -1;
      if (!bad) {
        const int pos = dir_L - dir_n + t, page = pos / kBlockSize;
        const int e = __shfl_sync(0xffffffffu, bt_lane, page & 31);
        const int blk = page < 32 ? e : __ldg(bt + page);
        if (blk >= 0 && blk < p.num_blocks) slot = blk * kBlockSize + pos % kBlockSize;
        else if (lane == 0) record_error(p.err, kDevBadBlockId);
      }
      if (dir_kv == 0 && lane == 0) p.slots[dir_q0 + t] = slot;
      if (slot >= 0 && lane < kVecs) {
        const int64_t dst = (static_cast<int64_t>(slot) * p.H_kv + dir_kv) * kVecs + lane;
        static_cast<uint4*>(p.k_pool)[dst] = kk;
        static_cast<uint4*>(p.v_pool)[dst] = vv;
      }
    }
    fence_proxy_async_global();  // before the TMA copies of these pages
    __syncwarp();
  };
  auto direct_item = [&](int idx, int& bt_lane) -> int {
    const int b = idx / p.H_kv, kv = idx - b * p.H_kv;
    const int32_t* bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;
    // lengths and the block-table row are loaded together
    const int q0 = __ldg(p.qsl + b), q1 = __ldg(p.qsl + b + 1), L = __ldg(p.seq_lens + b);
    const int bt_raw = lane < p.max_blocks ? __ldg(bt + lane) : -1;
    const int n = q1 - q0, pe = (L + kBlockSize - 1) / kBlockSize;
    if (idx == 0 && lane == 0 && (__ldg(p.qsl) != 0 || __ldg(p.qsl + p.B) != p.T))
      record_error(p.err, kDevBadSequence);  // tokens outside every sequence
    if (q0 < 0 || q1 > p.T || n < 0) {
      if (lane == 0) record_error(p.err, kDevBadSequence);
      return 0;
    }
    const bool bad = n > L || n * p.G > 16 || pe > p.max_blocks;
    if (bad && lane == 0) record_error(p.err, kDevBadSequence);
    bt_lane = !bad && lane < pe ? bt_raw : -1;
    dir_seq = b;
    dir_kv = kv;
    dir_q0 = q0;
    dir_n = n;
    dir_L = L;
    dir_first_new = (L - n) / kBlockSize;
    dir_pending = false;
    if (p.new_k != nullptr && n > 0) {
      if (bad) scatter_new(bt_lane, true);  // slots of -1 only
      else dir_pending = true;
    }
    if (bad || n == 0) return 0;
    int f = 0;
    f = lane == 0 ? b : f;
    f = lane == 1 ? kv : f;
    f = lane == 3 ? n * p.G : f;   // rows; row0 (lane 2) and page_begin (lane 4) are 0
    f = lane == 5 ? pe : f;
    f = lane == 7 ? 1 : f;         // one split (lane 6: split 0)
    f = lane == 8 ? L : f;
    f = lane == 9 ? n : f;
    f = lane == 10 ? q0 : f;
    return f;
  };

  // Issue the next page of work into stage g_issue % S; false when nothing is left.
  auto issue_one = [&]() -> bool {
    while (iss_page >= iss_end) {
      if (no_more) return false;
      int idx = 0;
      if constexpr (kDirect) {
        idx = direct_next;
        direct_next += gridDim.x * W;
      } else if (first_fetch) {
        // each warp's first item is its own, with no trip to the counter: the list is
        // longest first and the kernel's CTAs (one per SM) are all resident by then. With
        // tile items planned, a CTA's warps take consecutive items, so the split work sits
        // on as few SMs as it needs and the rest are free early for the tile kernel;
        // otherwise the items are dealt across the CTAs, so neighbouring items run on
        // different SMs.
        idx = tile_planned ? static_cast<int>(blockIdx.x) * W + warp
                           : warp * static_cast<int>(gridDim.x) + blockIdx.x;
        first_fetch = false;
      } else {
        if (lane == 0) idx = atomicAdd(p.hdr + 1, 1) + static_cast<int>(gridDim.x) * W;
        idx = __shfl_sync(0xffffffffu, idx, 0);
      }
      if (idx >= n_items) {
        no_more = true;
        return false;
      }
      const int* src = reinterpret_cast<const int*>(p.items + idx);
      int bt_direct = -1;
      int v;
      if constexpr (kDirect) v = direct_item(idx, bt_direct);
      else v = lane < 16 ? __ldg(src + lane) : 0;
      const int pb = __shfl_sync(0xffffffffu, v, 4), pe = __shfl_sync(0xffffffffu, v, 5);
      if (pe <= pb) continue;  // no key of this split is visible to these rows
      WorkItem* slot = ring + (ring_tail % kRing);
      if (lane < 16) reinterpret_cast<int*>(slot)[lane] = v;
      ++ring_tail;
      iss_seq = __shfl_sync(0xffffffffu, v, 0);
      iss_kv = __shfl_sync(0xffffffffu, v, 1);
      iss_page = pb;
      iss_end = pe;
      if constexpr (kDirect) {  // pages 0..31 of the sequence, read by direct_item
        bt_base = 0;
        bt_reg = bt_direct;
      } else {
        load_bt(pb);
      }
    }
    if (kDirect && dir_pending && iss_page >= dir_first_new) {
      // direct mode: the new tokens' rows go to the pools before their first page's copy
      scatter_new(bt_base == 0 ? bt_reg : -1, false);
      dir_pending = false;
    }
    if (iss_page - bt_base >= 32) load_bt(iss_page);
    const int blk = __shfl_sync(0xffffffffu, bt_reg, iss_page - bt_base);
    if (lane == 0) {
      int row = blk * kBlockSize;
      if (blk < 0 || blk >= p.num_blocks) {
        record_error(p.err, kDevBadBlockId);
        row = p.num_blocks * kBlockSize;  // past the tensor: the copy reads zeros
      }
      const uint32_t st = g_issue % S;
      uint8_t* dst = tiles + st * kStage;
      mbar_arrive_expect_tx(&full[st], kStage);
#pragma unroll
      for (int x = 0; x < kBoxes; ++x) {
        tma_load_2d_hint(dst + x * (kBlockSize * 128), &kmap, &full[st], iss_kv * D + x * 64,
                         row, policy);
        tma_load_2d_hint(dst + kPage + x * (kBlockSize * 128), &vmap, &full[st],
                         iss_kv * D + x * 64, row, policy);
      }
    }
    ++iss_page;
    ++g_issue;
    return true;
  };

  // ---------------- compute side ---------------------------------------------------
  const int g = lane >> 2, t4 = lane & 3;
  uint32_t g_comp = 0, ring_head = 0;
  int comp_left = 0, comp_page = 0;
  bool have_item = false;
  WorkItem cur;
  // per-thread rows g and g + 8 of the item
  int row_tok[2], row_h[2], row_pos[2];
  float m_run[2], l_run[2];
  float o[D / 8][4];
  uint32_t qa[kKSteps][4];
  const float scale_log2 = p.scale_log2;
  const uint16_t* qptr = static_cast<const uint16_t*>(p.q);

  auto start_item = [&]() {
    __syncwarp();  // the ring slot was written by lanes 0..15
    cur = ring[ring_head % kRing];
    ++ring_head;
    comp_page = cur.page_begin;
    comp_left = cur.page_end - cur.page_begin;
    have_item = true;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int rr = g + 8 * r;
      if (rr < cur.nrows) {
        const int R = cur.row0 + rr;
        const int i = R / p.G;
        row_tok[r] = cur.tok0 + i;
        row_h[r] = cur.kv * p.G + (R - i * p.G);
        row_pos[r] = cur.ctx_len - cur.n_query + i;
      } else {
        row_tok[r] = -1;
        row_h[r] = 0;
        row_pos[r] = -1;
      }
      m_run[r] = -INFINITY;
      l_run[r] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    // query fragments straight from global memory (rows g, g + 8; columns 2*t4 ...)
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        uint32_t lo = 0, hi = 0;
        if (row_tok[r] >= 0) {
          const uint16_t* src =
              qptr + (static_cast<int64_t>(row_tok[r]) * p.H_q + row_h[r]) * D + kk * 16 + 2 * t4;
          lo = __ldg(reinterpret_cast<const uint32_t*>(src));
          hi = __ldg(reinterpret_cast<const uint32_t*>(src + 8));
        }
        qa[kk][r] = lo;       // a0a1 (row g) / a2a3 (row g+8): columns 2t4, 2t4+1
        qa[kk][2 + r] = hi;   // a4a5 / a6a7: columns 2t4+8, 2t4+9
      }
    }
  };

  auto finish_item = [&]() {
    // complete the row sums across the quad of lanes sharing a row
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (row_tok[r] < 0) continue;
      const int tok = row_tok[r];
      const int ns_t = kDirect ? 1 : __ldg(p.tok_ns + tok);
      if (cur.split >= ns_t) continue;  // this split holds no key visible to the row
      const float inv = l_run[r] > 0.f ? 1.f / l_run[r] : 0.f;
      if (ns_t == 1) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(
            static_cast<uint16_t*>(p.out) + (static_cast<int64_t>(tok) * p.H_q + row_h[r]) * D +
            2 * t4);
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
          dst[j * 4] = pack2<kBF16>(o[j][2 * r] * inv, o[j][2 * r + 1] * inv);
      } else {
        const int64_t idx = __ldg(p.tok_base + tok) + cur.split * p.H_q + row_h[r];
        float2* dst = reinterpret_cast<float2*>(p.part_o + idx * D + 2 * t4);
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
          dst[j * 4] = make_float2(o[j][2 * r] * inv, o[j][2 * r + 1] * inv);
        if (t4 == 0)
          p.part_lse[idx] = l_run[r] > 0.f ? m_run[r] + __log2f(l_run[r]) : -INFINITY;
      }
    }
    have_item = false;
  };

  // fill the ring
  for (int s = 0; s < S; ++s)
    if (!issue_one()) break;

  bool aborted = false;
  while (true) {
    if (comp_left == 0) {
      if (have_item) finish_item();
      if (ring_head == ring_tail) break;  // everything issued has been computed
      start_item();
    }
    const uint32_t st = g_comp % S;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (g_comp / S) & 1))) {
      if (lane == 0) record_error(p.err, kDevWaitTimeout);
      aborted = true;
      break;
    }
    const uint32_t kbase = tiles_addr + st * kStage;
    const uint32_t vbase = kbase + kPage;

    // S = Q K^T for the page's 16 keys: two n8 tiles
    // two accumulators per n8 tile (even and odd k steps) halve the dependent mma chain
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int mi = lane >> 3, rr = lane & 7;
      const int key = (mi >> 1) * 8 + rr;
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
        const int chunk = 2 * kk + (mi & 1);
        const uint32_t addr = kbase + (chunk >> 3) * (kBlockSize * 128) + swz128(key, chunk & 7);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(addr, b0, b1, b2, b3);
        float (*acc)[4] = (kk & 1) ? s2 : s;
        mma_16816<kBF16>(acc[0], qa[kk], b0, b1);
        mma_16816<kBF16>(acc[1], qa[kk], b2, b3);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
    }
    // causal mask and row max on the raw scores (the scale is positive, so the max of the
    // scaled scores is the scaled max)
    const int key0 = comp_page * kBlockSize + 2 * t4;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e >> 1;
        const int key = key0 + nt * 8 + (e & 1);
        const float x = key <= row_pos[r] ? s[nt][e] : -INFINITY;
        s[nt][e] = x;
        mx[r] = fmaxf(mx[r], x);
      }
    float alpha[2], m_use[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float m_new = fmaxf(m_run[r], mx[r] == -INFINITY ? -INFINITY : mx[r] * scale_log2);
      m_use[r] = m_new == -INFINITY ? 0.f : m_new;
      alpha[r] = fast_exp2(m_run[r] - m_use[r]);
      m_run[r] = m_new;
    }
    // P = 2^(s * scale * log2 e - m): one packed fma per pair of scores of a row
    const float2 sc2 = make_float2(scale_log2, scale_log2);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float2 x = ffma2(make_float2(s[nt][2 * r], s[nt][2 * r + 1]), sc2,
                               make_float2(-m_use[r], -m_use[r]));
        s[nt][2 * r] = fast_exp2(x.x);
        s[nt][2 * r + 1] = fast_exp2(x.y);
      }
    uint32_t pa[4];
    pa[0] = pack2<kBF16>(s[0][0], s[0][1]);
    pa[1] = pack2<kBF16>(s[0][2], s[0][3]);
    pa[2] = pack2<kBF16>(s[1][0], s[1][1]);
    pa[3] = pack2<kBF16>(s[1][2], s[1][3]);
    // the row sums use the rounded P the tensor core multiplies with (each value widened
    // exactly and added in fp32)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float2 acc = make_float2(l_run[r] * alpha[r], 0.f);
      add_pair_exact<kBF16>(acc, pa[r]);
      add_pair_exact<kBF16>(acc, pa[2 + r]);
      l_run[r] = acc.x + acc.y;
    }
    // O rescaled by packed multiplies (a thread's accumulators pair up by row)
    const float2 a0 = make_float2(alpha[0], alpha[0]), a1 = make_float2(alpha[1], alpha[1]);
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      const float2 u = fmul2(make_float2(o[j][0], o[j][1]), a0);
      const float2 w = fmul2(make_float2(o[j][2], o[j][3]), a1);
      o[j][0] = u.x;
      o[j][1] = u.y;
      o[j][2] = w.x;
      o[j][3] = w.y;
    }
    // O += P V: V page is [key][d], read transposed
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int key = (mi & 1) * 8 + rr;
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        const int chunk = 2 * np + (mi >> 1);
        const uint32_t addr = vbase + (chunk >> 3) * (kBlockSize * 128) + swz128(key, chunk & 7);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(addr, b0, b1, b2, b3);
        mma_16816<kBF16>(o[2 * np], pa, b0, b1);
        mma_16816<kBF16>(o[2 * np + 1], pa, b2, b3);
      }
    }
    ++g_comp;
    ++comp_page;
    --comp_left;
    __syncwarp();
    fence_proxy_async_smem();
    issue_one();
  }
  if (aborted) {
    // let the copies already issued land before the CTA's shared memory goes away
    for (uint32_t gg = g_comp; gg < g_issue; ++gg) mbar_wait(&full[gg % S], (gg / S) & 1, 1u << 20);
  }
}

// ----------------------------------------------------------------------------------
// combine: one warp per (token, head) whose rows were split
// ----------------------------------------------------------------------------------
// A fixed grid walks the planner's list of split tokens, so a batch with no split rows
// costs one small launch.
#ifndef PS_COMBINE_UNROLL
#define PS_COMBINE_UNROLL 8
#endif
constexpr int kCombineUnroll = PS_COMBINE_UNROLL;

template <bool kBF16, int D>
__global__ void __launch_bounds__(256) combine_kernel(const AttnParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  // The warp's list entry is read beside the count (the list has room for T entries, so
  // the read stays in bounds; the entry is used only below the count).
  int tok_next = wid / p.H_q < p.T ? p.tok_list[wid / p.H_q] : 0;
  const int n = *reinterpret_cast<volatile const int*>(p.hdr + 7) * p.H_q;
  constexpr int kPer = D / 32;  // elements per lane
  for (; wid < n; wid += nwarps) {
    const int li = wid / p.H_q, h = wid - li * p.H_q;
    const int tok = tok_next;
    const int li_next = (wid + nwarps) / p.H_q;
    tok_next = li_next < p.T ? p.tok_list[li_next] : 0;
    const int ns = p.tok_ns[tok];
    const int base = p.tok_base[tok];
    // the first round's partials are loaded beside the log-sum-exps (they do not need them)
    auto load = [&](int s) -> float4 {
      const float* src = p.part_o + static_cast<int64_t>(base + s * p.H_q + h) * D + lane * kPer;
      if constexpr (kPer == 4) {
        return *reinterpret_cast<const float4*>(src);
      } else {
        const float2 v2 = *reinterpret_cast<const float2*>(src);
        return make_float4(v2.x, v2.y, 0.f, 0.f);
      }
    };
    float4 v[kCombineUnroll];
#pragma unroll
    for (int u = 0; u < kCombineUnroll; ++u)
      v[u] = u < ns ? load(u) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float lse = lane < ns ? p.part_lse[base + lane * p.H_q + h] : -INFINITY;
    float M = lse;
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = (lane < ns && lse != -INFINITY) ? exp2f(lse - M) : 0.f;
    float Wsum = w;
#pragma unroll
    for (int o = 16; o; o >>= 1) Wsum += __shfl_xor_sync(0xffffffffu, Wsum, o);
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    // kCombineUnroll partials' loads in flight per round
    for (int s0 = 0; s0 < ns; s0 += kCombineUnroll) {
      if (s0 > 0) {
#pragma unroll
        for (int u = 0; u < kCombineUnroll; ++u)
          v[u] = s0 + u < ns ? load(s0 + u) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kCombineUnroll; ++u) {
        const float ws = s0 + u < ns ? __shfl_sync(0xffffffffu, w, (s0 + u) & 31) : 0.f;
        acc[0] += ws * v[u].x;
        acc[1] += ws * v[u].y;
        if constexpr (kPer == 4) {
          acc[2] += ws * v[u].z;
          acc[3] += ws * v[u].w;
        }
      }
    }
    const float inv = Wsum > 0.f ? 1.f / Wsum : 0.f;
    uint16_t* dst = static_cast<uint16_t*>(p.out) + (static_cast<int64_t>(tok) * p.H_q + h) * D +
                    lane * kPer;
    if constexpr (kPer == 4) {
      uint2 o;
      o.x = pack2<kBF16>(acc[0] * inv, acc[1] * inv);
      o.y = pack2<kBF16>(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(dst) = o;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack2<kBF16>(acc[0] * inv, acc[1] * inv);
    }
  }
}

// ----------------------------------------------------------------------------------
// launchers
// ----------------------------------------------------------------------------------
int attention_warps(int D) { return D == 128 ? SplitCfg<128>::kWarps : SplitCfg<64>::kWarps; }
int attention_ctas(int D, int num_sms) { (void)D; return num_sms * PS_SPLIT_CTAS_PER_SM; }

// Threads per planner CTA: a small batch needs fewer (its scans and barriers span fewer
// warps); up to 1024.
// Packed tokens per planning CTA (the token pass's share of each CTA).
#ifndef PS_PLAN_TOKENS_PER_CTA
#define PS_PLAN_TOKENS_PER_CTA 256
#endif
#ifndef PS_PLAN_MIN_THREADS
#define PS_PLAN_MIN_THREADS 256
#endif
static int plan_threads(int B) {
  int t = (B + 31) / 32 * 32;
  t = t < PS_PLAN_MIN_THREADS ? PS_PLAN_MIN_THREADS : t;
  return t > 1024 ? 1024 : t;
}

cudaError_t launch_plan(const AttnParams& p, int concurrency, int tile_ctas, int num_sms,
                        cudaStream_t stream, const CopySegments* pre) {
  const int smem =
      p.B <= kPlanSmemSeqs ? kPlanSmemArrays * (p.B + 1) * static_cast<int>(sizeof(int)) : 0;
  if (smem > 48 * 1024) {
    static std::atomic<uint64_t> done{0};
    const cudaError_t e =
        ensure_smem_limit(plan_kernel, kPlanSmemArrays * (kPlanSmemSeqs + 1) * 4, done);
    if (e != cudaSuccess) return e;
  }
  // enough CTAs that the token and item passes are short (a CTA's warps share its SM's
  // issue slots, and emitting a sequence's items is division-heavy); each repeats the scan
  const int64_t want = 1 + static_cast<int64_t>(p.T) / PS_PLAN_TOKENS_PER_CTA + p.B / 8;
  // (one CTA when the offsets live in global memory: the CTAs' scans would share them)
  const int ctas = p.B > kPlanSmemSeqs ? 1 : static_cast<int>(want < kPlanMaxCtas ? want : kPlanMaxCtas);
  // the scatter CTAs: one warp per token, at most 64 warps per SM in all
  const int threads = plan_threads(p.B), warps = threads / 32;
  int64_t scatter = 0;
  if (p.new_k != nullptr && p.T > 0) {
    scatter = (static_cast<int64_t>(p.T) + warps - 1) / warps;
    const int64_t cap = static_cast<int64_t>(num_sms) * 64 / warps;
    if (scatter > cap) scatter = cap;
  }
  // the copy CTAs: one 16-byte word per thread and round, at most two CTAs per SM
  CopySegments segs{};
  int64_t copies = 0;
  if (pre != nullptr && pre->n > 0) {
    segs = *pre;
    int64_t words = 0;
    for (int k = 0; k < segs.n; ++k) words += segs.seg[k].bytes / 16 + 1;
    copies = (words + threads - 1) / threads;
    const int64_t cap = 2 * static_cast<int64_t>(num_sms);
    if (copies > cap) copies = cap;
  }
  // programmatic dependent launch: the CTAs may start while the kernel before them on the
  // stream finishes (see plan_kernel for what they wait for, and when)
  return launch_kernel(plan_kernel, dim3(static_cast<unsigned>(ctas + scatter + copies)),
                       dim3(threads), static_cast<size_t>(smem), stream, true, p, concurrency,
                       tile_ctas, ctas, segs, static_cast<int>(copies));
}

template <bool kBF16, int D, bool kDirect, int kS = 0>
static cudaError_t launch_split_t(const AttnParams& p, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, int ctas, cudaStream_t stream,
                                  bool pdl) {
  constexpr int smem = split_smem_bytes<D, kS>();
  auto kern = split_attention_kernel<kBF16, D, kDirect, kS>;
  static std::atomic<uint64_t> done{0};
  const cudaError_t e = ensure_smem_limit(kern, smem, done);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(ctas), dim3(SplitCfg<D>::kWarps * 32), smem, stream, pdl, kmap,
                       vmap, p);
}

bool direct_fits(const AttnParams& p, int num_sms) {
  const int64_t items = static_cast<int64_t>(p.B) * p.H_kv;
  return static_cast<int64_t>(p.T) * p.G <= 16 && p.max_blocks <= kDirectMaxPages &&
         items <= static_cast<int64_t>(num_sms) * attention_warps(p.D);
}

cudaError_t launch_direct_attention(const AttnParams& p, bool bf16, const CUtensorMap& kmap,
                                    const CUtensorMap& vmap, int num_sms, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(p.B) * p.H_kv;
  const int warps = attention_warps(p.D);
  int64_t ctas = (items + warps - 1) / warps;
  if (ctas < 1) ctas = 1;
  if (ctas > num_sms) ctas = num_sms;
  return launch_split_attention(p, bf16, kmap, vmap, static_cast<int>(ctas), stream, false);
}

int split_ctas(const AttnParams& p, int num_sms) {
  // items <= H_kv x (sum over sequences of ceil(n G / 16)) x splits, and a sequence splits
  // at most ceil(max_blocks / kMinSplitPages) ways: no more warps than that can find work
  const int64_t per_split = static_cast<int64_t>(p.T) * p.G / 16 + 1 + p.B;
  int64_t splits = (static_cast<int64_t>(p.max_blocks) + kMinSplitPages - 1) / kMinSplitPages;
  splits = splits < 1 ? 1 : (splits > kMaxSplits ? kMaxSplits : splits);
  const int64_t items = static_cast<int64_t>(p.H_kv) * per_split * splits;
  const int warps = attention_warps(p.D);
  const int64_t need = (items + warps - 1) / warps;
  const int full = attention_ctas(p.D, num_sms);
  return static_cast<int>(need < full ? (need < 1 ? 1 : need) : full);
}

cudaError_t launch_split_attention(const AttnParams& p, bool bf16, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int ctas, cudaStream_t stream,
                                   bool pdl) {
  // the direct mode is its own instantiation, so the planned kernel carries none of it;
  // with no block table longer than kDirectSmallPages its ring has two stages: a warp
  // streams at most that many pages, and the smaller footprint starts the launch sooner
  if (p.direct && p.max_blocks <= kDirectSmallPages) {
    if (p.D == 128)
      return bf16 ? launch_split_t<true, 128, true, 2>(p, kmap, vmap, ctas, stream, pdl)
                  : launch_split_t<false, 128, true, 2>(p, kmap, vmap, ctas, stream, pdl);
    return bf16 ? launch_split_t<true, 64, true, 2>(p, kmap, vmap, ctas, stream, pdl)
                : launch_split_t<false, 64, true, 2>(p, kmap, vmap, ctas, stream, pdl);
  }
  if (p.direct) {
    if (p.D == 128)
      return bf16 ? launch_split_t<true, 128, true>(p, kmap, vmap, ctas, stream, pdl)
                  : launch_split_t<false, 128, true>(p, kmap, vmap, ctas, stream, pdl);
    return bf16 ? launch_split_t<true, 64, true>(p, kmap, vmap, ctas, stream, pdl)
                : launch_split_t<false, 64, true>(p, kmap, vmap, ctas, stream, pdl);
  }
  if (p.D == 128)
    return bf16 ? launch_split_t<true, 128, false>(p, kmap, vmap, ctas, stream, pdl)
                : launch_split_t<false, 128, false>(p, kmap, vmap, ctas, stream, pdl);
  return bf16 ? launch_split_t<true, 64, false>(p, kmap, vmap, ctas, stream, pdl)
              : launch_split_t<false, 64, false>(p, kmap, vmap, ctas, stream, pdl);
}

cudaError_t launch_combine(const AttnParams& p, bool bf16, int num_sms, cudaStream_t stream,
                           bool pdl) {
  const int64_t warps = static_cast<int64_t>(p.T) * p.H_q;
  if (warps == 0) return cudaSuccess;
  const int64_t ctas = (warps + 7) / 8;  // 8 warps per CTA
  const dim3 grid(static_cast<unsigned>(ctas < 4 * num_sms ? ctas : 4 * num_sms));
  if (p.D == 128)
    return bf16 ? launch_kernel(combine_kernel<true, 128>, grid, dim3(256), 0, stream, pdl, p)
                : launch_kernel(combine_kernel<false, 128>, grid, dim3(256), 0, stream, pdl, p);
  return bf16 ? launch_kernel(combine_kernel<true, 64>, grid, dim3(256), 0, stream, pdl, p)
              : launch_kernel(combine_kernel<false, 64>, grid, dim3(256), 0, stream, pdl, p);
}

}  // namespace ps
