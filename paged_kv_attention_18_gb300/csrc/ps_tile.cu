// Tile kernel for prefill chunks: tcgen05 MMA with TMEM accumulators, K/V pages fed by
// TMA straight from the paged pool.
//
// One work item is a pair of query tiles of one sequence and one KV head: tile A and the
// tile after it, B, each up to 128 packed rows (whole query tokens x the G query heads
// that share the KV head), over one split of the context. The context is walked in
// tiles of 128 keys (8 pages of 16); each K/V tile serves both query tiles:
//     S_g = Q_g K^T        tcgen05.mma: A = Q_g (smem), B = K (smem)    -> S_g in TMEM
//     P_g = exp2(S_g*scale*log2e - m) with the online row max / sum (softmax group g)
//     O_g += P_g V         tcgen05.mma: A = P_g (TMEM), B = V (smem)    -> O_g in TMEM
// with the causal rule of the pages (key j visible to the query at position p iff
// j <= p: PageServe section 01; tinyserve "How it works") and grouped-query attention
// (tinyserve "Highlights" table).
//
// Warp roles (384 threads):
//   warp 0     hands out work items (longest first, as the planner lists them) and loads
//              Q and K: three K stages, each freed once both S products have read it;
//   warp 2     loads V (two stages); a tile's page copies are spread over the lanes, one
//              TMA copy per lane;
//   warp 1     owns TMEM; one of its threads issues every MMA and, per tile and query
//              tile, waits on nothing but P;
//   warp 3     watches K and V: it adds its arrival to query tile A's P barrier once V
//              tile j and K tile j + 1 have landed, so P also stands for them;
//   warps 4..7 and 8..11  the softmax groups of query tiles A and B, one TMEM lane (one
//              query row) per thread; a warp reaches the 32 TMEM lanes of its warp index
//              mod 4. While one group computes its exponentials the tensor core works on
//              the other group's products. P is written back over S in TMEM and read from
//              there by the PV product. O is rescaled lazily, only when a row's running
//              max grows by more than 2^8. The same warps write the item's output.
#include "ps_common.cuh"
#include "ps_launch.h"
#include "ps_tc05.cuh"

namespace ps {

namespace {

constexpr int kRows = 128;        // query rows per tile (MMA M)
constexpr int kKeys = 128;        // keys per KV tile (MMA N of S, K of PV) = 8 pages
constexpr int kPagesPerTile = kKeys / kBlockSize;
constexpr int kSub = kRows * 128; // bytes of one [128 rows x 64 elements] swizzled sub-tile
constexpr int kKStages = 3;       // K tile stages (freed once both products S have read them)
constexpr int kVStages = 2;       // V tile stages (freed once both products PV have read them)
constexpr int kItemRing = 4;     // item indices handed from the fetching warp to the others
constexpr int kThreads = 384;
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows by > 2^8
// A larger jump inside a tile moves the reference at once; below it P can reach 2^kMove,
// which must stay finite in the 16-bit type (fp16 tops out near 2^16, bf16 near 2^128).
template <bool kBF16>
constexpr float kMoveLog2 = kBF16 ? 64.f : 15.f;
// Largest row sum of a 64-column half of P taken against the current reference without
// looking at the half's max: every P is then at most this (bf16: 2^64, as above; fp16:
// 64 finite values, so none overflowed). A larger (or infinite) sum sends the half
// through the max and the reference move.
template <bool kBF16>
constexpr float kHalfSumMax = kBF16 ? 18446744073709551616.f : 4194304.f;
constexpr uint32_t kTmemCols = 512;

// TMEM columns of softmax group g: S (and P over it) at g*256, O at g*256 + 128
__host__ __device__ constexpr uint32_t col_s(int g) { return g * 256u; }
__host__ __device__ constexpr uint32_t col_o(int g) { return g * 256u + 128u; }

template <int D>
struct TileSmem {
  static constexpr int kQ = (D / 64) * kSub;  // one query tile
  static constexpr int kK = (D / 64) * kSub;  // one K or V tile (128 keys)
  static constexpr int kOffQ = 0;             // query tiles A, B
  static constexpr int kOffK = kOffQ + 2 * kQ;
  static constexpr int kOffV = kOffK + kKStages * kK;
  static constexpr int kOffBar = kOffV + kVStages * kK;
  static constexpr int kOffItems = kOffBar + 512;             // work items in flight
  static constexpr int kBytes = kOffItems + 2 * kItemRing * 64 + 1024;  // + alignment slack
};
static_assert(TileSmem<128>::kBytes <= 232448, "tile kernel shared memory");

struct TileBars {
  uint64_t q_full[2], q_empty[2];  // query tiles A and B, each freed after its last S
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t mma_final;
  uint64_t item_full[kItemRing], item_empty[kItemRing];
  int item_idx[kItemRing];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(TileBars) <= 512, "barrier block");

// An item fits this launch: a sequence and KV head of the batch, a page range inside the
// block table, and query rows inside the packed batch. Every role checks each item the
// same way and skips one that does not fit, so no role reads or writes outside its
// buffers on a plan it cannot use.
__device__ __forceinline__ bool tile_item_ok(const WorkItem& w, const AttnParams& p) {
  if (w.seq < 0 || w.seq >= p.B || w.kv < 0 || w.kv >= p.H_kv) return false;
  if (w.page_begin < 0 || w.page_end > p.max_blocks) return false;
  if (w.tok0 < 0 || w.row0 < 0 || w.nrows <= 0 || w.pad[0] < 0) return false;
  const int last_row = w.row0 + (w.pad[0] > 0 ? p.tpt * p.G + w.pad[0] : w.nrows) - 1;
  return w.tok0 + last_row / p.G < p.T;
}

}  // namespace

// kDirect: no plan. Each CTA derives its items from seq_lens and qsl (every sequence
// unsplit, its query-tile pairs longest first), and only the K/V producers wait for the
// kernel before this one (the step's scatter) before their first copy from the pools.
template <bool kBF16, int D, bool kDirect>
__global__ void __launch_bounds__(kThreads, 1)
    tile_attention_kernel(const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap,
                          const __grid_constant__ CUtensorMap qmap, const AttnParams p) {
  using L = TileSmem<D>;
  constexpr int kHalves = D / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();

  // The set-up (barriers, TMEM, zeroed query rows, descriptor prefetch) touches only this
  // CTA's own state, so it runs while the kernels before this one finish.
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  TileBars* bars = reinterpret_cast<TileBars*>(smem + L::kOffBar);
  // Records of the items in flight: item it's record sits in slot it % (2 * kItemRing).
  // The fetching warp runs at most kItemRing items ahead of the slowest reader (the index
  // ring), so a slot is written again only after every reader has finished with it.
  WorkItem* items = reinterpret_cast<WorkItem*>(smem + L::kOffItems);
  const uint32_t sQ = smem_u32(smem + L::kOffQ);
  const uint32_t sK = smem_u32(smem + L::kOffK);
  const uint32_t sV = smem_u32(smem + L::kOffV);

  if (threadIdx.x == 0) {
    for (int q = 0; q < 2; ++q) {
      mbar_init(&bars->q_full[q], 1);
      mbar_init(&bars->q_empty[q], 1);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&bars->s_full[g], 1);
      mbar_init(&bars->p_full[g], g == 0 ? 5 : 4);  // tile A's: + the K/V watcher
      mbar_init(&bars->o_done[g], 1);
    }
    mbar_init(&bars->mma_final, 1);
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(&bars->item_full[s], 1);
      mbar_init(&bars->item_empty[s], 11);  // V producer, MMA, K/V watcher, 8 softmax warps
    }
    bars->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&qmap);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  {
    // Rows past the G * tpt rows a query tile holds are never written by TMA: zero them
    // once, so that their S is 0 and they go through the softmax like any unmasked row.
    const int rows = p.G * p.tpt;
    const int words = (kRows - rows) * 128 / 16;  // 16-byte words per sub-tile
    for (int i = threadIdx.x; i < 2 * kHalves * words; i += kThreads) {
      const int sub = i / words, wd = i - sub * words;
      reinterpret_cast<uint4*>(smem + L::kOffQ + sub * kSub + rows * 128)[wd] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();  // visible to the tensor core's reads
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;

  int n_items = 0;
  if constexpr (!kDirect) {
    // the plan and the kernels before this one are complete; after the split kernel,
    // which let this kernel launch only once the plan was complete, the plan is read
    // without a wait and the wait for the split kernel comes at the end
    if (!p.after_split) pdl_wait();
    n_items = *reinterpret_cast<volatile const int*>(p.hdr + 4);
    if (n_items == 0) {  // nothing planned for this kernel (uniform across the grid)
      if (warp == 1) tmem_dealloc(tmem, kTmemCols);
      if (p.after_split && blockIdx.x == 0 && threadIdx.x == 0) pdl_wait();
      return;
    }
  } else if (!p.after_scatter) {
    pdl_wait();  // the step's inputs may still be being written by the kernel before
  }

  // Bounded wait with a warp-uniform outcome: if any lane gives up (or another role has
  // given up), the whole warp leaves its loop together.
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    bool ok = !*abort_flag && mbar_wait(bar, parity);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) {
      record_error(p.err, kDevWaitTimeout);
      *abort_flag = 1;
    }
    return ok;
  };
  // next work item from the ring (consumer side); -1 at the end or on a time-out
  auto next_item = [&](int it) -> int {
    const int slot = it % kItemRing;
    if (!wait(&bars->item_full[slot], (it / kItemRing) & 1)) return -1;
    const int idx = bars->item_idx[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    return idx;
  };

  if (warp == 0 || warp == 2) {
    // ===================== producers: warp 0 (items, Q, K), warp 2 (V) ================
    const bool is_k = warp == 0;
    const int n_stages = is_k ? kKStages : kVStages;
    uint32_t g = 0, qa = 0, qb = 0;
    bool waited = !kDirect;  // direct mode: the pools are read after the step's scatter
    // Direct mode: lane b holds sequence b's query tokens n, context L, first token t0 and
    // query-tile pairs (0 for a sequence without rows or an invalid one). Items go rank by
    // rank (rank r: every sequence's r-th longest pair, in batch order, each KV head), so
    // csum(r) = H_kv * sum_b min(pairs_b, r) items come before rank r; CTA c takes items
    // c, c + gridDim.x, ...
    int d_n = 0, d_L = 0, d_t0 = 0, d_pairs = 0, d_max = 0, d_total = 0;
    auto csum = [&](int r) -> int {
      int v = min(d_pairs, r);
#pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      return v * p.H_kv;
    };
    if constexpr (kDirect) {
      if (is_k && lane < p.B) {
        const int q0 = __ldg(p.qsl + lane), q1 = __ldg(p.qsl + lane + 1);
        const int L = __ldg(p.seq_lens + lane), n = q1 - q0;
        const bool valid = n >= 0 && n <= L && (L + kBlockSize - 1) / kBlockSize <= p.max_blocks &&
                           q0 >= 0 && q1 <= p.T;
        if (!valid) {
          if (blockIdx.x == 0) record_error(p.err, kDevBadSequence);
        } else if (n > 0) {
          d_n = n;
          d_L = L;
          d_t0 = q0;
          d_pairs = ((n + p.tpt - 1) / p.tpt + 1) / 2;
        }
      }
      d_max = d_pairs;
#pragma unroll
      for (int o = 16; o; o >>= 1) d_max = max(d_max, __shfl_xor_sync(0xffffffffu, d_max, o));
      d_total = csum(d_max);
    }
    // field `lane` of direct item idx (< d_total)
    auto direct_field = [&](int idx) -> int {
      int lo = 0, hi = d_max - 1;  // rank: the last r with csum(r) <= idx
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (csum(mid) <= idx) lo = mid;
        else hi = mid - 1;
      }
      const int r = lo, k = idx - csum(r);
      const int nth = k / p.H_kv, kv = k - nth * p.H_kv;
      // the nth (from 0) sequence in batch order that has a pair of rank r
      const unsigned has = __ballot_sync(0xffffffffu, d_pairs > r);
      const bool hit = ((has >> lane) & 1u) && __popc(has & ((1u << lane) - 1u)) == nth;
      const int b = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
      const int n = __shfl_sync(0xffffffffu, d_n, b), L = __shfl_sync(0xffffffffu, d_L, b);
      const int t0 = __shfl_sync(0xffffffffu, d_t0, b);
      const int j = __shfl_sync(0xffffffffu, d_pairs, b) - 1 - r;  // rank 0: the last pair
      const int qa_ = 2 * j * p.tpt, qb_ = qa_ + p.tpt;
      const int na = min(p.tpt, n - qa_), nb = qb_ < n ? min(p.tpt, n - qb_) : 0;
      const int i_last = nb > 0 ? qb_ + nb - 1 : qa_ + na - 1;
      const int pe = min((L + kBlockSize - 1) / kBlockSize, (L - n + i_last) / kBlockSize + 1);
      int f = 0;  // seq, kv, row0, nrows, page_begin 0, page_end, split 0, nsplit 1, L, n, t0
      f = lane == 0 ? b : f;
      f = lane == 1 ? kv : f;
      f = lane == 2 ? qa_ * p.G : f;
      f = lane == 3 ? na * p.G : f;
      f = lane == 5 ? pe : f;
      f = lane == 7 ? 1 : f;
      f = lane == 8 ? L : f;
      f = lane == 9 ? n : f;
      f = lane == 10 ? t0 : f;
      f = lane == 11 ? nb * p.G : f;  // rows of query tile B
      return f;
    };
    for (int it = 0;; ++it) {
      int idx = 0;
      if (is_k && kDirect) {
        const int slot = it % kItemRing;
        if (!wait(&bars->item_empty[slot], ((it / kItemRing) & 1) ^ 1)) break;
        idx = blockIdx.x + it * static_cast<int>(gridDim.x);
        if (idx >= d_total) idx = -1;
        if (idx >= 0) {
          const int f = direct_field(idx);
          if (lane < 16) reinterpret_cast<int*>(items + it % (2 * kItemRing))[lane] = f;
        }
        __syncwarp();
        if (lane == 0) {
          bars->item_idx[slot] = idx;
          mbar_arrive(&bars->item_full[slot]);
        }
      } else if (is_k) {
        const int slot = it % kItemRing;
        if (!wait(&bars->item_empty[slot], ((it / kItemRing) & 1) ^ 1)) break;
        if (lane < 4) {
          // lanes 0..3 copy the item's record into its shared-memory slot, lane 0 hands
          // out the index (its arrival orders the copy before every reader's wait)
          if (lane == 0) idx = atomicAdd(p.hdr + 5, 1);
          idx = __shfl_sync(0x0000000fu, idx, 0);
          if (idx >= n_items) idx = -1;
          if (idx >= 0)
            reinterpret_cast<uint4*>(items + it % (2 * kItemRing))[lane] =
                __ldg(reinterpret_cast<const uint4*>(p.tile_items + idx) + lane);
          __syncwarp(0x0000000fu);
          if (lane == 0) {
            bars->item_idx[slot] = idx;
            mbar_arrive(&bars->item_full[slot]);
          }
        }
        __syncwarp();
        idx = __shfl_sync(0xffffffffu, idx, 0);
      } else {
        idx = next_item(it);
      }
      if (idx < 0) break;
      const WorkItem& w = items[it % (2 * kItemRing)];
      const int pb = w.page_begin, pe = w.page_end;
      if (pe <= pb || !tile_item_ok(w, p)) continue;
      const int seq = w.seq, kv = w.kv;
      const int nt = (pe - pb + kPagesPerTile - 1) / kPagesPerTile;
      // query tiles (K warp): whole tokens x the G heads of this KV head. Each tile has its
      // own buffer, refilled as soon as that tile's last S of the previous item has read
      // it. They are loaded after the item's first K tile, whose stage frees earlier.
      auto load_q = [&]() -> bool {
        const bool has_b = w.pad[0] > 0;
        const int tok = w.tok0 + w.row0 / p.G;
        const uint32_t tile_bytes = kHalves * 64 * 2 * p.G * p.tpt;
        for (int q = 0; q < (has_b ? 2 : 1); ++q) {
          if (!wait(&bars->q_empty[q], ((q ? qb : qa) & 1) ^ 1)) return false;
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars->q_full[q], tile_bytes);
            for (int h = 0; h < kHalves; ++h)
              tma_load_3d(smem + L::kOffQ + q * L::kQ + h * kSub, &qmap, &bars->q_full[q],
                          h * 64, kv * p.G, tok + q * p.tpt);
          }
        }
        ++qa;
        if (has_b) ++qb;
        return true;
      };
      // K (or V) tiles of 8 pages; pages past the split read the zero fill. One lane per
      // page copy: lane = page * kHalves + half (64-element half of the head).
      const int32_t* bt = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks;
      int bt_base = -1000, bt_reg = -1;
      bool ok = true;
      const int pp = lane / kHalves, h = lane % kHalves;
      for (int j = 0; j < nt; ++j) {
        const int first = pb + j * kPagesPerTile;
        if (first - bt_base + kPagesPerTile > 32) {
          bt_base = first;
          bt_reg = first + lane < pe ? __ldg(bt + first + lane) : -1;
        }
        const uint32_t st = g % n_stages;
        uint64_t* empty = is_k ? &bars->k_empty[st] : &bars->v_empty[st];
        uint64_t* full = is_k ? &bars->k_full[st] : &bars->v_full[st];
        if (!wait(empty, ((g / n_stages) & 1) ^ 1)) { ok = false; break; }
        if (!waited) {
          pdl_wait();  // the step's scatter has written the new tokens' rows
          waited = true;
        }
        const int blk = __shfl_sync(0xffffffffu, bt_reg, (first - bt_base + pp) & 31);
        uint8_t* dst = smem + (is_k ? L::kOffK : L::kOffV) + st * L::kK;
        if (lane == 0) mbar_arrive_expect_tx(full, L::kK);
        __syncwarp();
        if (lane < kPagesPerTile * kHalves) {
          int row;
          if (first + pp >= pe) {
            row = p.num_blocks * kBlockSize;  // past the pool: zero fill, no HBM read
          } else if (blk < 0 || blk >= p.num_blocks) {
            record_error(p.err, kDevBadBlockId);
            row = p.num_blocks * kBlockSize;
          } else {
            row = blk * kBlockSize;
          }
          tma_load_2d(dst + h * kSub + pp * (kBlockSize * 128), is_k ? &kmap : &vmap, full,
                      kv * D + h * 64, row);
        }
        ++g;
        if (is_k && j == 0 && !load_q()) { ok = false; break; }
      }
      if (!ok) break;
    }
  } else if (warp == 1) {
    // ============================ MMA issuer (one thread) ===========================
    // Issuing one tcgen05.mma occupies the thread for nearly as long as the tensor core
    // takes to run it (M128 N128 K16), so this loop is kept lean: lane 0 alone, with
    // descriptors formed as a base plus constant offsets and waits without warp votes.
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16(kBF16, kRows, kKeys, false);
      constexpr uint32_t idPV = idesc_f16(kBF16, kRows, D, true);
      // bounded single-thread wait; the abort flag is read only on the slow path
      auto wait1 = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        for (uint32_t i = 0; i < (1u << 24); ++i) {
          if (*abort_flag) return false;
          if (mbar_try_wait(bar, parity)) return true;
        }
        record_error(p.err, kDevWaitTimeout);
        *abort_flag = 1;
        return false;
      };
      // descriptor start addresses stay below 2^18 bytes, so offsets added to the 14-bit
      // start field (address / 16) never carry into the next field
      const uint64_t qdesc0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t qdesc1 = sdesc_sw128(sQ + L::kQ, 16, 1024);
      const uint64_t kdesc0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t vdesc0 = sdesc_sw128(sV, kSub, 1024);
      uint32_t g = 0, qa = 0, qb = 0, pc[2] = {0, 0};
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int slot = it % kItemRing;
        if (!wait1(&bars->item_full[slot], (it / kItemRing) & 1)) break;
        const int idx = bars->item_idx[slot];
        mbar_arrive(&bars->item_empty[slot]);
        if (idx < 0) break;
        const WorkItem& w = items[it % (2 * kItemRing)];
        const int pb = w.page_begin, pe = w.page_end;
        if (!tile_item_ok(w, p)) {
          record_error(p.err, kDevPlanOverflow);  // a plan this launch cannot use
          continue;
        }
        if (pe <= pb) continue;
        const bool has_b = w.pad[0] > 0;
        const int ng = has_b ? 2 : 1;
        const int nt = (pe - pb + kPagesPerTile - 1) / kPagesPerTile;
        if (!wait1(&bars->q_full[0], qa & 1)) break;
        const uint32_t g0 = g;
        // S of query tile `grp` against K tile j. Only the item's first K tile is waited
        // for here; P of query tile A for tile j - 1 implies K tile j (the K/V watcher).
        auto issue_s = [&](int grp, int j) -> bool {
          const uint32_t st = (g0 + j) % kKStages;
          if (j == 0 && grp == 0) {
            if (!wait1(&bars->k_full[st], ((g0 + j) / kKStages) & 1)) return false;
            tc_fence_after();
          }
          const uint64_t a0 = grp ? qdesc1 : qdesc0;
          const uint64_t b0 = kdesc0 + ((st * L::kK) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk / 4) * kSub + (kk % 4) * 32) >> 4;
            umma_f16(tmem + col_s(grp), a0 + off, b0 + off, idS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars->s_full[grp]);
          if (j == nt - 1) umma_commit(&bars->q_empty[grp]);  // last read of this Q tile
          if (grp == ng - 1) umma_commit(&bars->k_empty[st]);  // last reader of the K stage
          return true;
        };
        // O of query tile `grp` += P V of K/V tile j. P is the only wait: the softmax
        // warps arrive on it after their epilogue of the previous item has read O, and
        // the K/V watcher adds its arrival to query tile A's once V tile j (and K tile
        // j + 1) have landed.
        auto issue_pv = [&](int grp, int j) -> bool {
          if (!wait1(&bars->p_full[grp], pc[grp] & 1)) return false;
          ++pc[grp];
          const uint32_t st = (g0 + j) % kVStages;
          tc_fence_after();
          const uint64_t b0 = vdesc0 + ((st * L::kK) >> 4);
          const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)
            umma_f16_ts(tmem + col_o(grp), tmem + col_s(grp) + kk * 8, b0 + ((kk * 2048) >> 4),
                        idPV, kk > 0 ? 1u : acc0);
          if (grp == ng - 1) umma_commit(&bars->v_empty[st]);  // last reader of the V stage
          return true;
        };
        for (int q = 0; q < ng && ok; ++q) {
          if (q == 1 && !wait1(&bars->q_full[1], qb & 1)) {
            ok = false;
            break;
          }
          ok = issue_s(q, 0);
        }
        // per K/V tile: PV of A, next S of A, PV of B, next S of B. A query tile's next S
        // overwrites its P in TMEM, so it is issued after that tile's PV (in order).
        // A query tile's O is final after its last PV: its epilogue may start while the
        // other tile's last PV still waits for P.
        for (int j = 0; j < nt && ok; ++j)
          for (int q = 0; q < ng && ok; ++q) {
            ok = issue_pv(q, j);
            if (ok && j + 1 < nt) ok = issue_s(q, j + 1);
            if (ok && j + 1 == nt) umma_commit(&bars->o_done[q]);
          }
        if (!ok) break;
        g += nt;
        ++qa;
        if (ng > 1) ++qb;
      }
      // every MMA issued by this thread has completed before TMEM is released
      umma_commit(&bars->mma_final);
      mbar_wait(&bars->mma_final, 0, 1u << 22);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ============================ K/V watcher ==================================
    // P of query tile A also stands for V tile j and K tile j + 1 having landed: this
    // warp waits for them and adds its arrival to that P barrier, then waits for the
    // barrier's phase to complete so that it never runs a tile ahead. The MMA thread
    // then waits on P alone, and the softmax warps carry no extra waits.
    uint32_t gt = 0, pc = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int idx = next_item(it);
      if (idx < 0) break;
      const WorkItem& w = items[it % (2 * kItemRing)];
      const int pb = w.page_begin, pe = w.page_end;
      if (pe <= pb || !tile_item_ok(w, p)) continue;
      const int nt = (pe - pb + kPagesPerTile - 1) / kPagesPerTile;
      for (int j = 0; j < nt && ok; ++j) {
        const uint32_t gv = gt + j, gk = gv + 1;
        ok = wait(&bars->v_full[gv % kVStages], (gv / kVStages) & 1) &&
             (j + 1 >= nt || wait(&bars->k_full[gk % kKStages], (gk / kKStages) & 1));
        if (!ok) break;
        if (lane == 0) mbar_arrive(&bars->p_full[0]);
        ok = wait(&bars->p_full[0], pc & 1);
        ++pc;
      }
      gt += nt;
    }
  } else if (warp >= 4) {
    // ============================ softmax groups + epilogue =========================
    const int grp = (warp - 4) >> 2;   // 0: query tile A, 1: query tile B
    const int quarter = warp & 3;      // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t tS = trow + col_s(grp), tO = trow + col_o(grp);
    const float sl2 = p.scale_log2;
    uint32_t sc = 0, act = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int idx = next_item(it);
      if (idx < 0) break;
      const WorkItem& w = items[it % (2 * kItemRing)];
      const int pb = w.page_begin, pe = w.page_end;
      if (pe <= pb || !tile_item_ok(w, p)) continue;
      const int nt = (pe - pb + kPagesPerTile - 1) / kPagesPerTile;
      const int nrows = grp == 0 ? w.nrows : w.pad[0];
      if (nrows == 0) continue;  // no query tile B in this item
      // this thread's query row
      const bool valid = r < nrows;
      const int R = w.row0 + grp * p.tpt * p.G + r;  // packed row within the sequence
      const int qtok = R / p.G;                        // query index within the sequence
      const int tok = w.tok0 + qtok;
      const int head = w.kv * p.G + R - qtok * p.G;
      const int pos = valid ? w.ctx_len - w.n_query + qtok : -1;
      const int key_hi = min(pos, pe * kBlockSize - 1);  // last key of the item this row sees
      // the row's split count and partial base, fetched now so that the epilogue's
      // stores do not wait on them
      // (both loads are issued at once; nothing waits for them before the epilogue)
      const int ns_t = !valid ? 0 : kDirect ? 1 : __ldg(p.tok_ns + tok);
      const int tok_part = kDirect || !valid ? 0 : __ldg(p.tok_base + tok);
      // m_ref: the reference max (log2 units) that P, O and l are currently taken against;
      // m_next: a max more than 2^8 above it seen in the last tile, applied before the next
      float m_ref = -INFINITY, m_next = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        // visible columns: c <= lim (a row past the tile's rows is computed unmasked and
        // not written)
        const int lim = valid ? key_hi - (pb * kBlockSize + j * kKeys) : kKeys;
        if (!wait(&bars->s_full[grp], sc & 1)) { ok = false; break; }
        ++sc;
        tc_fence_after();
        // This group's previous PV has completed (this S was issued after it): O is stable.
        auto rescale_o = [&](float alpha) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tO + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st32(tO + c * 32, v);
          }
          tmem_st_wait();
        };
        if (__any_sync(0xffffffffu, m_next > m_ref)) {
          const bool need = m_next > m_ref;
          const float alpha = need ? fast_exp2(m_ref - m_next) : 1.f;
          if (j > 0) rescale_o(alpha);
          l *= alpha;
          if (need) m_ref = m_next;
        }
        // P = 2^(s*scale*log2e - m_ref) as 16-bit pairs written over S; half h of P lands
        // on columns 32h..32h+31, which the loads of halves <= h have already read
        const bool full = __all_sync(0xffffffffu, lim >= kKeys - 1);
        // l holds the earlier tiles' sum; this tile's halves are summed apart, so that a
        // reference moved in half 1 can re-sum the half-0 P it re-rounds
        float l_half0 = 0.f, l_h = 0.f;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t v[64];
          tmem_ld32(tS + 64 * h, v);
          tmem_ld32(tS + 64 * h + 32, v + 32);
          tmem_ld_wait();
          if (!full) {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (64 * h + e > lim) v[e] = __float_as_uint(-INFINITY);
          }
          uint32_t pk[32];
          // P is taken against the row's reference without the half's max; the max (and a
          // move of the reference) is taken only when there is no reference yet, or when
          // the half's sum shows that P outgrew its bound, and P is then taken again
          bool with_max = __any_sync(0xffffffffu, m_ref == -INFINITY);
#pragma unroll 1
          for (int pass = 0; pass < 2; ++pass) {
            if (with_max) {
              // four independent max chains
              float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
              for (int e = 0; e < 64; e += 8)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  mq[k] = fmax3(mq[k], __uint_as_float(v[e + 2 * k]), __uint_as_float(v[e + 2 * k + 1]));
              const float mx = fmax3(fmaxf(mq[0], mq[1]), mq[2], mq[3]);
              const float m_half = mx == -INFINITY ? -INFINITY : mx * sl2;
              // no reference yet, or a jump P could overflow on: move the reference now,
              // rescaling what is already taken against the old one
              const bool move = m_half > m_ref + kMoveLog2<kBF16> ||
                                (m_ref == -INFINITY && m_half != -INFINITY);
              if (__any_sync(0xffffffffu, move)) {
                const float alpha = move && m_ref != -INFINITY ? fast_exp2(m_ref - m_half) : 1.f;
                if (j > 0) rescale_o(alpha);
                l *= alpha;
                if (h == 1) {
                  // the half of P already written (columns 0..31) is scaled and rounded
                  // again; its sum is taken anew from the values the PV product will read
                  uint32_t q[32];
                  tmem_st_wait();
                  tmem_ld32(tS, q);
                  tmem_ld_wait();
                  float2 lq0[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                  for (int e = 0; e < 32; ++e) {
                    q[e] = scale_pair<kBF16>(q[e], alpha);
                    add_pair_exact<kBF16>(lq0[e & 1], q[e]);
                  }
                  l_half0 = (lq0[0].x + lq0[0].y) + (lq0[1].x + lq0[1].y);
                  tmem_st32(tS, q);
                  tmem_st_wait();
                }
                if (move) m_ref = m_half;
              }
            }
            const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
            float2 lq[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // four sums
            // scale and subtract two scores per packed fma; the row sum adds the 16-bit P
            // values the MMA sees, widened exactly
            const float2 sl2x2 = make_float2(sl2, sl2), nm2 = make_float2(neg_m, neg_m);
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
              const float2 x = ffma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                     sl2x2, nm2);
              pk[e / 2] = pack2<kBF16>(fast_exp2(x.x), fast_exp2(x.y));
              add_pair_exact<kBF16>(lq[(e / 2) & 1], pk[e / 2]);
            }
            // P goes out before its sum is checked; a second pass writes it again
            if (pass > 0) tmem_st_wait();
            tmem_st16(tS + 32 * h, pk);
            tmem_st16(tS + 32 * h + 16, pk + 16);
            l_h = (lq[0].x + lq[0].y) + (lq[1].x + lq[1].y);
            if (with_max || __all_sync(0xffffffffu, l_h <= kHalfSumMax<kBF16>)) break;
            with_max = true;
          }
          if (h == 0) l_half0 = l_h;
          else l += l_half0 + l_h;
        }
        // O is rescaled lazily: when this tile's P summed to more than 2^8, the reference
        // moves up by log2 of that sum before the next tile (the new reference is at least
        // the row's max, so P stays at most 1 there)
        const float l_tile = l_half0 + l_h;
        m_next = l_tile > (1 << static_cast<int>(kRescaleLog2)) ? m_ref + __log2f(l_tile) : m_ref;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[grp]);
      }
      if (!ok) break;
      // epilogue: O / l of this group's rows to the output, or to the split partials
      if (!wait(&bars->o_done[grp], act & 1)) break;
      tc_fence_after();
      const bool write = valid && w.split < ns_t && l > 0.f;
      const float inv = write ? 1.f / l : 0.f;
      if (__all_sync(0xffffffffu, !write || ns_t == 1)) {
        // Direct output: each lane writes its own row, 64 columns (128 bytes) per TMEM
        // wait, as 32-byte stores when the output is 32-byte aligned (16-byte stores
        // otherwise), so every store instruction fills whole 32-byte sectors of 32 rows.
        uint16_t* dst = static_cast<uint16_t*>(p.out) + (static_cast<int64_t>(tok) * p.H_q + head) * D;
        const bool wide = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll 1
        for (int c4 = 0; c4 < D / 64; ++c4) {
          uint32_t v[64];
          tmem_ld32(tO + c4 * 64, v);
          tmem_ld32(tO + c4 * 64 + 32, v + 32);
          tmem_ld_wait();
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 x =
                fmul2(make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), inv2);
            w[e] = pack2<kBF16>(x.x, x.y);
          }
          if (write) {
            if (wide) {
#pragma unroll
              for (int q = 0; q < 4; ++q) st_global_v8(dst + c4 * 64 + 16 * q, w + 8 * q);
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(dst + c4 * 64);
#pragma unroll
              for (int q = 0; q < 8; ++q) d4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            }
          }
        }
      } else {
        // split partials (fp32), one row per lane
#pragma unroll 1
        for (int c2 = 0; c2 < D / 64; ++c2) {
          uint32_t v[64];
          tmem_ld32(tO + c2 * 64, v);
          tmem_ld32(tO + c2 * 64 + 32, v + 32);
          tmem_ld_wait();
          if (!write) continue;
          if (ns_t == 1) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                  (static_cast<int64_t>(tok) * p.H_q + head) * D +
                                                  c2 * 64);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_uint4(
                  pack2<kBF16>(__uint_as_float(v[8 * q + 0]) * inv, __uint_as_float(v[8 * q + 1]) * inv),
                  pack2<kBF16>(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv),
                  pack2<kBF16>(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv),
                  pack2<kBF16>(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv));
          } else {
            const int64_t pidx = static_cast<int64_t>(tok_part) + w.split * p.H_q + head;
            float4* dst = reinterpret_cast<float4*>(p.part_o + pidx * D + c2 * 64);
#pragma unroll
            for (int q = 0; q < 16; ++q)
              dst[q] = make_float4(__uint_as_float(v[4 * q]) * inv, __uint_as_float(v[4 * q + 1]) * inv,
                                   __uint_as_float(v[4 * q + 2]) * inv, __uint_as_float(v[4 * q + 3]) * inv);
            if (c2 == 0) p.part_lse[pidx] = m_ref + __log2f(l);
          }
        }
      }
      ++act;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (!kDirect && p.after_split && blockIdx.x == 0 && threadIdx.x == 0) pdl_wait();
}

int tile_tokens(int G) { return G >= 1 && G <= 16 ? kRows / G : 0; }

template <bool kBF16, int D, bool kDirect>
static cudaError_t launch_tile_t(const AttnParams& p, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, const CUtensorMap& qmap, int ctas,
                                 cudaStream_t stream, bool pdl) {
  constexpr int smem = TileSmem<D>::kBytes;
  auto kern = tile_attention_kernel<kBF16, D, kDirect>;
  static std::atomic<uint64_t> done{0};
  const cudaError_t e = ensure_smem_limit(kern, smem, done);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(ctas), dim3(kThreads), smem, stream, pdl, kmap, vmap, qmap, p);
}

template <bool kDirect>
static cudaError_t launch_tile_d(const AttnParams& p, bool bf16, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, const CUtensorMap& qmap, int ctas,
                                 cudaStream_t stream, bool pdl) {
  if (p.D == 128)
    return bf16 ? launch_tile_t<true, 128, kDirect>(p, kmap, vmap, qmap, ctas, stream, pdl)
                : launch_tile_t<false, 128, kDirect>(p, kmap, vmap, qmap, ctas, stream, pdl);
  return bf16 ? launch_tile_t<true, 64, kDirect>(p, kmap, vmap, qmap, ctas, stream, pdl)
              : launch_tile_t<false, 64, kDirect>(p, kmap, vmap, qmap, ctas, stream, pdl);
}

cudaError_t launch_tile_attention(const AttnParams& p, bool bf16, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, const CUtensorMap& qmap, int ctas,
                                  cudaStream_t stream, bool pdl, bool direct) {
  return direct ? launch_tile_d<true>(p, bf16, kmap, vmap, qmap, ctas, stream, pdl)
                : launch_tile_d<false>(p, bf16, kmap, vmap, qmap, ctas, stream, pdl);
}

bool direct_tile_fits(const AttnParams& p, int num_sms) {
  return p.tpt > 0 && p.B <= kDirectTileMaxSeqs && p.max_blocks <= kDirectMaxPages &&
         static_cast<int64_t>(p.B) * p.H_kv * 2 <= num_sms;
}

int direct_tile_ctas(const AttnParams& p, int num_sms) {
  // a sequence of n tokens has ceil(ceil(n / tpt) / 2) <= n / (2 tpt) + 1 pairs
  const int64_t items = static_cast<int64_t>(p.H_kv) * (p.T / (2 * p.tpt) + 1 + p.B);
  return static_cast<int>(items < num_sms ? (items < 1 ? 1 : items) : num_sms);
}

}  // namespace ps
