// Speculative-decoding acceptance after the verify pass (tinyserve "How it works",
// speculative decoding; PageServe "Rejection sampling"): draft d_i is accepted with
// probability min(1, p_i(d_i) / q_i(d_i)); at the first rejection the replacement token is
// drawn from normalize(max(p_i - q_i, 0)); when all k drafts survive, a bonus token is
// drawn from the last target distribution p_k. The greedy rule accepts a draft while it
// equals argmax p_i and emits the argmax at the first mismatch (or p_k's when all match).
//
// Every decision is made in a fixed precision so that any implementation of the same
// rule picks the same tokens: the random draws are caller-provided 32-bit words R; the
// acceptance test is the fp64 comparison R * q < p * 2^32 (products rounded once); the
// residual weights max(p - q, 0) are fp32 and become integers W = trunc(w * 2^40), so
// their sums are exact in any order; the sample is the first token whose running sum of
// W exceeds floor(R * Z / 2^32), Z the total. Argmax ties go to the lowest token.
//
// Two kernels per call. Rejection rule: the first streams the one residual row each
// sequence needs as 128-token runs, spread evenly over about four CTAs per SM, and writes
// every run's fixed-point sum; the second, one CTA per sequence, scans those sums, then
// reads only the run that holds the sample. Greedy: the first, one CTA per (sequence,
// chunk of the vocabulary), takes the chunk argmax of every row; the second combines them.
// Every sum is an exact integer, so how a row is cut into runs never changes the token.
#include "ps_common.cuh"
#include "ps_launch.h"

namespace ps {

namespace {

constexpr int kThreads = 256;  // also the largest chunk count (spec_chunks caps it at 64)
constexpr int kWarps = kThreads / 32;
constexpr int kRun = 128;          // tokens per run: four per lane
#ifndef PS_SPEC_CTAS_PER_SM
#define PS_SPEC_CTAS_PER_SM 4
#endif
constexpr int kCtasPerSm = PS_SPEC_CTAS_PER_SM;        // resident run-kernel CTAs per SM

// trunc(w * 2^40) for w > 0, 0 for w <= 0 and NaN: scaling by 2^40 is exact and the
// conversion truncates toward zero, so this is the exact integer for every w below 2^23.
__device__ __forceinline__ long long fixed_weight(float w) {
  return w > 0.f ? static_cast<long long>(__float2ull_rz(w * 1099511627776.0f)) : 0;
}

// The fixed-point weight of one token: max(p - q_e, 0), q_e the draft's probability of the
// token (1 at the draft token of a one-hot row; 0 on a row drawn from p itself, whose
// weight is then p).
__device__ __forceinline__ long long token_weight(float pv, float qe) {
  return fixed_weight(fmaxf(__fsub_rn(pv, qe), 0.f));
}

// Acceptance of a sequence's drafts under the rejection rule, decided by a warp (one
// lane per draft, k <= 31).
struct Accept {
  int r;         // drafts accepted
  bool plain;    // the final draw is from p itself: every draft survived, or the stopping
  bool invalid;  //   draft id lies outside the vocabulary (then also `invalid`)
  int draft;     // the stopping draft's token (the one-hot row's 1), -1 when plain
};

// One lane's part for sequence b: its draft's token and test. Branch-free, so the loads of
// two sequences can be in flight together; an id outside the vocabulary reads token 0.
struct AcceptLane {
  int d;
  bool ok, bad;
};

__device__ __forceinline__ AcceptLane accept_lane(const SpecParams& a, int b) {
  const int lane = threadIdx.x & 31;
  AcceptLane x = {-1, true, false};
  if (lane < a.k) {
    x.d = a.drafts[b * a.k + lane];
    x.bad = x.d < 0 || x.d >= a.V;
    const int dc = x.bad ? 0 : x.d;
    const float pv = a.p[(static_cast<int64_t>(b) * (a.k + 1) + lane) * a.V + dc];
    const float qv = a.q ? a.q[(static_cast<int64_t>(b) * a.k + lane) * a.V + dc] : 1.f;
    const double lhs = __dmul_rn(static_cast<double>(a.rnd[b * (a.k + 1) + lane]), qv);
    const double rhs = __dmul_rn(static_cast<double>(pv), 4294967296.0);
    x.ok = !x.bad && lhs < rhs;
  }
  return x;
}

__device__ __forceinline__ Accept accept_finish(const SpecParams& a, const AcceptLane& x) {
  const int lane = threadIdx.x & 31;
  const unsigned rej = __ballot_sync(0xffffffffu, lane < a.k && !x.ok);
  Accept y;
  y.r = rej ? __ffs(rej) - 1 : a.k;
  const bool inv = __shfl_sync(0xffffffffu, x.bad ? 1 : 0, y.r & 31) != 0;
  const int d = __shfl_sync(0xffffffffu, x.d, y.r & 31);
  y.invalid = rej != 0 && inv;
  y.plain = rej == 0 || y.invalid;
  y.draft = y.plain ? -1 : d;
  return y;
}

__device__ __forceinline__ Accept accepted_warp(const SpecParams& a, int b) {
  return accept_finish(a, accept_lane(a, b));
}

__device__ __forceinline__ int accept_word(const Accept& y) {
  return y.r | (y.plain ? 1 << 8 : 0) | (y.invalid ? 1 << 9 : 0);
}

template <typename T>
__device__ T block_sum(T v, T* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  T t = 0;
  for (int i = 0; i < nw; ++i) t += sh[i];
  __syncthreads();
  return t;
}

// (value, token) with the larger value, the lower token on ties; NaN never wins
__device__ __forceinline__ void amax_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ void block_argmax(float& v, int& i, float* shv, int* shi) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    amax_merge(v, i, v2, i2);
  }
  if (lane == 0) {
    shv[wid] = v;
    shi[wid] = i;
  }
  __syncthreads();
  v = -INFINITY;
  i = INT32_MAX;
  for (int w = 0; w < nw; ++w) amax_merge(v, i, shv[w], shi[w]);
  __syncthreads();
}

// grid (chunks, B), greedy rule: the argmax of each of sequence b's k + 1 rows over one
// chunk of the vocabulary. With V a multiple of 4 and p 16-byte aligned every row starts
// 16-byte aligned and chunks are multiples of 8 tokens, so rows stream as float4 loads,
// four per thread in flight.
__global__ void __launch_bounds__(kThreads) spec_chunk_kernel(const SpecParams a) {
  __shared__ float shv[kThreads / 32];
  __shared__ int shi[kThreads / 32];
  pdl_launch_dependents();
  const int c = blockIdx.x, b = blockIdx.y;
  const int64_t lo = static_cast<int64_t>(c) * a.chunk;
  const int64_t hi = lo + a.chunk < a.V ? lo + a.chunk : a.V;
  const bool vec = a.vec != 0;
  for (int i = 0; i <= a.k; ++i) {
    const float* row = a.p + (static_cast<int64_t>(b) * (a.k + 1) + i) * a.V;
    float v = -INFINITY;
    int t = INT32_MAX;
    if (vec) {
      // four float4 loads per thread in flight
      const float4* r4 = reinterpret_cast<const float4*>(row);
      for (int64_t x0 = lo / 4 + threadIdx.x; x0 < hi / 4; x0 += 4 * kThreads) {
        float4 f[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t x = x0 + u * kThreads;
          f[u] = x < hi / 4 ? __ldcs(r4 + x) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int base = static_cast<int>(4 * (x0 + u * kThreads));
          amax_merge(v, t, f[u].x, base);
          amax_merge(v, t, f[u].y, base + 1);
          amax_merge(v, t, f[u].z, base + 2);
          amax_merge(v, t, f[u].w, base + 3);
        }
      }
    } else {
      for (int64_t x = lo + threadIdx.x; x < hi; x += kThreads)
        amax_merge(v, t, row[x], static_cast<int>(x));
    }
    block_argmax(v, t, shv, shi);
    if (threadIdx.x == 0) {
      const int64_t o = (static_cast<int64_t>(b) * (a.k + 1) + i) * a.gent + c;
      a.amax_v[o] = v;
      a.amax_i[o] = t;
    }
  }
}

// Sums over the warp of N values per lane: lane l returns the sum of value l / (32 / N)
// (lanes other than the first of each group of 32 / N hold the same sum). Each exchange
// at distance 16, 8, ... halves the values a lane holds, the two halves of the warp
// keeping different ones; the rest is a plain butterfly.
template <int N>
__device__ __forceinline__ long long warp_sum_n(long long (&v)[N]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int half = N / 2, dist = 16; half >= 1; half /= 2, dist /= 2) {
    const bool up = lane & dist;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const long long keep = up ? v[i + half] : v[i];
      const long long send = up ? v[i] : v[i + half];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, dist);
    }
  }
#pragma unroll
  for (int dist = 16 / N; dist >= 1; dist /= 2) v[0] += __shfl_xor_sync(0xffffffffu, v[0], dist);
  return v[0];
}

// trunc(w * 2^40) = hi * 2^20 + lo with hi = floor(y), y = w * 2^20, and lo = floor((y - hi)
// * 2^20), for 0 <= w < 8: adding 2^23 rounded toward zero drops the fraction of any value
// in [0, 2^23), and every other step is exact, so both parts are integers held exactly in
// fp32 and their sums over a few tokens stay exact.
__device__ __forceinline__ void weight_parts(float w, float& hi, float& lo) {
  const float y = w * 1048576.0f;
  hi = __fsub_rn(__fadd_rz(y, 8388608.0f), 8388608.0f);
  const float z = __fsub_rn(y, hi) * 1048576.0f;
  lo = __fsub_rn(__fadd_rz(z, 8388608.0f), 8388608.0f);
}

// weight_parts on two tokens at once (packed fp32 pairs, each lane rounded as the scalar
// form), added into hs and ls: hs += hi, ls += lo per token.
__device__ __forceinline__ void weight_parts2_add(float w0, float w1, float2& hs, float2& ls) {
  asm("{\n\t.reg .b64 w, y, hb, hi, z, lb, lo, c20, c23, hs, ls;\n\t"
      "mov.b64 w, {%4, %5};\n\t"
      "mov.b64 c20, {%6, %6};\n\t"
      "mov.b64 c23, {%7, %7};\n\t"
      "mul.rn.f32x2 y, w, c20;\n\t"
      "add.rz.f32x2 hb, y, c23;\n\t"
      "sub.rn.f32x2 hi, hb, c23;\n\t"
      "sub.rn.f32x2 z, y, hi;\n\t"
      "mul.rn.f32x2 z, z, c20;\n\t"
      "add.rz.f32x2 lb, z, c23;\n\t"
      "sub.rn.f32x2 lo, lb, c23;\n\t"
      "mov.b64 hs, {%0, %1};\n\t"
      "mov.b64 ls, {%2, %3};\n\t"
      "add.rn.f32x2 hs, hs, hi;\n\t"
      "add.rn.f32x2 ls, ls, lo;\n\t"
      "mov.b64 {%0, %1}, hs;\n\t"
      "mov.b64 {%2, %3}, ls;\n\t}"
      : "+f"(hs.x), "+f"(hs.y), "+f"(ls.x), "+f"(ls.y)
      : "f"(w0), "f"(w1), "f"(1048576.0f), "f"(8388608.0f));
}

// p - q on two tokens at once.
__device__ __forceinline__ float2 sub2(float2 p, float2 q) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(p.x), "f"(p.y), "f"(q.x), "f"(q.y));
  return d;
}

// An integer-valued float in [0, 2^23) as an integer: its bits after adding 2^23.
__device__ __forceinline__ int small_int(float x) {
  return __float_as_int(__fadd_rn(x, 8388608.0f)) - 0x4B000000;
}

// Rejection rule, grid G (one wave of resident CTAs). The rows the sequences need are cut
// into runs of 128 tokens, listed sequence by sequence: U = B * runs. CTA j takes the
// runs [j*U/G, (j+1)*U/G), so every CTA streams the same number of bytes; its warp w
// takes runs w*N .. w*N+N-1 of each group of 8N (N = 4 with draft rows q, 8 without), loads
// all N before summing any, and writes each run's fixed-point residual sum. Tokens past the
// end of a row load as zeros, which weigh 0. A warp decides the acceptance of a sequence
// when it first meets one of its runs (the one that holds run 0 records it).
template <bool kQ>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) spec_run_kernel(const SpecParams a) {
  constexpr int kN = kQ ? 4 : 8;  // runs a warp loads before summing any
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t U = static_cast<int64_t>(a.B) * a.runs;
  const int64_t u_lo = U * blockIdx.x / gridDim.x;
  const int64_t u_hi = U * (blockIdx.x + 1) / gridDim.x;
  const bool vec = a.vec != 0;
  // (sequence, run) of the warp's first run of the group, advanced without division
  int64_t u0 = u_lo + warp * kN;
  int b0 = static_cast<int>(u0 / a.runs);
  int m0 = static_cast<int>(u0 - static_cast<int64_t>(b0) * a.runs);
  // the acceptance of the sequence the warp last met, and its row pointers
  int cur_b = -1, draft = -1;
  const float* row = nullptr;
  const float* qrow = nullptr;
  for (; u0 < u_hi; u0 += kWarps * kN) {
    float4 f[kN], g[kQ ? kN : 1];  // p, and q (0 on a row without one)
    int dl[kN];  // the one-hot draft token relative to the run, -1 for none
    int b = b0, m = m0;
#pragma unroll
    for (int t = 0; t < kN; ++t) {
      f[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kQ) g[t] = f[t];
      dl[t] = -1;
      if (t > 0 && ++m == a.runs) {
        m = 0;
        ++b;
      }
      if (u0 + t >= u_hi) continue;  // warp-uniform
      if (b != cur_b) {
        const Accept y = accepted_warp(a, b);
        if (m == 0 && lane == 0) a.acc[b] = accept_word(y);
        cur_b = b;
        row = a.p + (static_cast<int64_t>(b) * (a.k + 1) + y.r) * a.V;
        qrow = (kQ && !y.plain) ? a.q + (static_cast<int64_t>(b) * a.k + y.r) * a.V : nullptr;
        draft = kQ ? -1 : y.draft;
      }
      const int t0 = m * kRun;
      dl[t] = draft >= t0 && draft < t0 + kRun ? draft - t0 : -1;
      if (vec) {
        // lane l: tokens t0 + 4l .. t0 + 4l + 3 (V a multiple of 4: all or none in range)
        const int v = t0 + 4 * lane;
        if (v < a.V) {
          f[t] = __ldcs(reinterpret_cast<const float4*>(row + v));
          if (kQ && qrow) g[t] = __ldcs(reinterpret_cast<const float4*>(qrow + v));
        }
      } else {
        // lane l: tokens t0 + l + 32e, 4-byte loads
        float* fe = &f[t].x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = t0 + lane + 32 * e;
          if (v < a.V) {
            fe[e] = __ldcs(row + v);
            if (kQ && qrow) (&g[t].x)[e] = __ldcs(qrow + v);
          }
        }
      }
    }
    long long s[kN];
#pragma unroll
    for (int t = 0; t < kN; ++t) {
      const float pv[4] = {f[t].x, f[t].y, f[t].z, f[t].w};
      float qv[4] = {0.f, 0.f, 0.f, 0.f};
      if (kQ) {
        qv[0] = g[kQ ? t : 0].x;
        qv[1] = g[kQ ? t : 0].y;
        qv[2] = g[kQ ? t : 0].z;
        qv[3] = g[kQ ? t : 0].w;
      } else if (dl[t] >= 0) {  // warp-uniform: the draft token of a one-hot row is here
        const int l = vec ? dl[t] >> 2 : dl[t] & 31;
        const int e = vec ? dl[t] & 3 : dl[t] >> 5;
        if (lane == l) {
#pragma unroll
          for (int x = 0; x < 4; ++x)
            if (x == e) qv[x] = 1.f;
        }
      }
      float hs = 0.f, ls = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float hi, lo;
        weight_parts(fmaxf(__fsub_rn(pv[e], qv[e]), 0.f), hi, lo);
        hs += hi;
        ls += lo;
      }
      s[t] = (static_cast<long long>(small_int(hs)) << 20) + small_int(ls);
    }
    const long long tot = warp_sum_n<kN>(s);
    const int j = lane / (32 / kN);
    if (lane % (32 / kN) == 0 && u0 + j < u_hi) a.wsum[u0 + j] = tot;
    // (b, m) is the group's last run; the next group starts kWarps * kN runs after its first
    b0 = b;
    m0 = m + (kWarps - 1) * kN + 1;
    while (m0 >= a.runs) {
      m0 -= a.runs;
      ++b0;
    }
  }
}

// ------------------------------------------------------------------------------------
// Rejection rule with rows as 16-byte words: the runs and sums of spec_run_kernel, but the
// rows reach shared memory by bulk copies, so the bytes in flight do not depend on
// registers. A stage holds 16 KB: 16 runs of p and 16 of q, or 32 runs of p.
// ------------------------------------------------------------------------------------
constexpr int kStreamStages = 4;
constexpr int kStageFloats = 4096;
constexpr int kStreamThreads = (kWarps + 1) * 32;  // eight consumer warps, one producer
constexpr int kStreamCtasPerSm = 3;

struct StreamSmem {
  float buf[kStreamStages][kStageFloats];
  uint64_t full[kStreamStages];   // the stage's copies landed (one arrival with the bytes)
  uint64_t empty[kStreamStages];  // the stage was read (one arrival per consumer warp)
  int has_q[kStreamStages];       // q copied into the stage's second half
  int draft[kStreamStages];       // one-hot draft token relative to the stage, -1 for none
};

// One run of sequence rows after another within [u, u_hi): at most `cap` runs, never past
// the end of a row.
struct Chunk {
  int64_t u;
  int b, m, n;
  __device__ __forceinline__ void fit(int64_t u_hi, int runs, int cap) {
    const int64_t left = u_hi - u;
    int k = runs - m < cap ? runs - m : cap;
    n = left <= 0 ? 0 : (left < k ? static_cast<int>(left) : k);
  }
  __device__ __forceinline__ void next(int64_t u_hi, int runs, int cap) {
    u += n;
    m += n;
    if (m == runs) {
      m = 0;
      ++b;
    }
    fit(u_hi, runs, cap);
  }
};

// Wait for the phase with the given parity, the thread suspended in between (it resumes
// when the phase completes, or after at most 20 us per poll), so waiting warps leave the
// issue slots to the others; gives up after `limit` polls (about 1.3 s) and returns false.
__device__ __forceinline__ bool mbar_wait_idle(uint64_t* bar, uint32_t parity,
                                               uint32_t limit = (1u << 16)) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    if (ok) return true;
  }
  return false;
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// What a stream kernel computes per run: the residual sum with draft rows q, the residual
// sum with one-hot drafts (or none), or the argmax of every row (greedy rule).
enum StreamMode { kResidualQ = 0, kResidualOneHot = 1, kArgmax = 2 };

// grid G (one wave of resident CTAs), the same share of runs per CTA as spec_run_kernel
// (greedy: the runs of all k + 1 rows of every sequence). The producer warp decides each
// sequence's acceptance when it meets its first run (rejection rule), then copies each
// chunk of a row (p, and q where the row has one) into the next free stage; consumer warp
// w handles runs w, w + 8, ... of every stage and releases it.
template <int kMode>
__global__ void __launch_bounds__(kStreamThreads, kStreamCtasPerSm)
    spec_stream_kernel(const SpecParams a) {
  constexpr bool kQ = kMode == kResidualQ, kGreedy = kMode == kArgmax;
  constexpr int kCap = kQ ? 16 : 32;  // runs per stage
  constexpr int kPer = kCap / kWarps;  // runs per consumer warp and stage
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StreamSmem& sm = *reinterpret_cast<StreamSmem*>(smem_raw);
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows = kGreedy ? a.B * (a.k + 1) : a.B;
  const int64_t U = static_cast<int64_t>(rows) * a.runs;
  const int64_t u_lo = U * blockIdx.x / gridDim.x;
  const int64_t u_hi = U * (blockIdx.x + 1) / gridDim.x;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStreamStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  Chunk c0;  // c.b: the sequence (rejection rule) or the row b * (k + 1) + i (greedy)
  c0.u = u_lo;
  c0.b = static_cast<int>(u_lo / a.runs);
  c0.m = static_cast<int>(u_lo - static_cast<int64_t>(c0.b) * a.runs);
  c0.fit(u_hi, a.runs, kCap);
  if (warp == kWarps) {
    // producer
    const uint64_t pol = l2_policy_evict_first();
    Accept cur = {0, true, false, -1}, nxt = cur;
    int cur_b = -1, nxt_b = -1;
    if (!kGreedy && c0.n > 0) {
      // the share's first sequence, and the next one when the share reaches it: their
      // loads in flight together
      const bool two = static_cast<int64_t>(c0.b + 1) * a.runs < u_hi;
      const AcceptLane x0 = accept_lane(a, c0.b);
      const AcceptLane x1 = two ? accept_lane(a, c0.b + 1) : x0;
      nxt = accept_finish(a, x0);
      nxt_b = c0.b;
      if (two) {
        cur = nxt;
        cur_b = c0.b;
        if (c0.m == 0 && lane == 0) a.acc[c0.b] = accept_word(cur);
        nxt = accept_finish(a, x1);
        nxt_b = c0.b + 1;
      }
    }
    int r = cur.r, draft = kQ ? -1 : cur.draft;
    bool plain = cur.plain;
    int issued = 0;
    for (Chunk c = c0; c.n > 0; c.next(u_hi, a.runs, kCap)) {
      if (!kGreedy && c.b != cur_b) {
        cur = c.b == nxt_b ? nxt : accepted_warp(a, c.b);
        cur_b = c.b;
        if (c.m == 0 && lane == 0) a.acc[c.b] = accept_word(cur);
        r = cur.r;
        plain = cur.plain;
        draft = kQ ? -1 : cur.draft;
      }
      const int s = issued % kStreamStages, use = issued / kStreamStages;
      bool ok = true;
      if (lane == 0) {
        ok = use == 0 || mbar_wait_idle(&sm.empty[s], (use - 1) & 1);
        if (ok) {
          const int t0 = c.m * kRun;
          const int t1 = (c.m + c.n) * kRun < a.V ? (c.m + c.n) * kRun : a.V;
          const uint32_t bytes = static_cast<uint32_t>(t1 - t0) * 4;  // a multiple of 16
          const bool hq = kQ && !plain;
          sm.has_q[s] = hq ? 1 : 0;
          sm.draft[s] = draft >= t0 && draft < t1 ? draft - t0 : -1;
          mbar_arrive_expect_tx(&sm.full[s], hq ? 2 * bytes : bytes);
          const int64_t prow = kGreedy ? c.b : static_cast<int64_t>(c.b) * (a.k + 1) + r;
          bulk_load(sm.buf[s], a.p + prow * a.V + t0, bytes, &sm.full[s], pol);
          if (hq)
            bulk_load(sm.buf[s] + kStageFloats / 2,
                      a.q + (static_cast<int64_t>(c.b) * a.k + r) * a.V + t0, bytes,
                      &sm.full[s], pol);
        } else {
          record_error(a.err, kDevWaitTimeout);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      ++issued;
    }
    // no copy may still be writing this CTA's shared memory when it exits
    if (lane == 0) {
      const int first = issued > kStreamStages ? issued - kStreamStages : 0;
      for (int i = first; i < issued; ++i)
        mbar_wait_idle(&sm.full[i % kStreamStages], (i / kStreamStages) & 1);
    }
    return;
  }
  // consumers
  int idx = 0;
  for (Chunk c = c0; c.n > 0; c.next(u_hi, a.runs, kCap), ++idx) {
    const int s = idx % kStreamStages;
    if (!mbar_wait_idle(&sm.full[s], (idx / kStreamStages) & 1)) {
      if (lane == 0) record_error(a.err, kDevWaitTimeout);
      break;
    }
    if (kGreedy) {
      // (largest value, lowest token holding it) over the warp's runs of the stage: each
      // lane meets its tokens in increasing order, so a strict comparison keeps the lowest
      // of equal values; then one exchange over the warp, written as the entry of the
      // warp's first run and (-inf, none) for its other runs
      float4 f[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int run = warp + kWarps * j;
        f[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (run < c.n && (c.m + run) * kRun + 4 * lane < a.V)
          f[j] = *reinterpret_cast<const float4*>(&sm.buf[s][run * kRun + 4 * lane]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
      float v = -INFINITY;
      int t = INT32_MAX;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int run = warp + kWarps * j;
        const int base = (c.m + run) * kRun + 4 * lane;
        if (run < c.n && base < a.V) {
          const float x[4] = {f[j].x, f[j].y, f[j].z, f[j].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (x[e] > v) {
              v = x[e];
              t = base + e;
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int t2 = __shfl_xor_sync(0xffffffffu, t, o);
        amax_merge(v, t, v2, t2);
      }
      if (lane < kPer && warp + kWarps * lane < c.n) {
        a.amax_v[c.u + warp + kWarps * lane] = lane == 0 ? v : -INFINITY;
        a.amax_i[c.u + warp + kWarps * lane] = lane == 0 ? t : INT32_MAX;
      }
    } else {
      // each run's fixed-point residual sum
      const bool hq = kQ && sm.has_q[s] != 0;
      const int dd = kMode == kResidualOneHot ? sm.draft[s] : -1;
      long long sums[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int run = warp + kWarps * j;
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f), g = f;
        if (run < c.n && (c.m + run) * kRun + 4 * lane < a.V) {
          f = *reinterpret_cast<const float4*>(&sm.buf[s][run * kRun + 4 * lane]);
          if (hq)
            g = *reinterpret_cast<const float4*>(
                &sm.buf[s][kStageFloats / 2 + run * kRun + 4 * lane]);
        }
        // residual weights max(p - q, 0): q from the stage, or 1 at a one-hot row's
        // draft token and 0 elsewhere
        float2 w01 = make_float2(f.x, f.y), w23 = make_float2(f.z, f.w);
        if (kQ) {
          w01 = sub2(w01, make_float2(g.x, g.y));
          w23 = sub2(w23, make_float2(g.z, g.w));
        } else if (dd >= 0 && (dd >> 7) == run && ((dd & (kRun - 1)) >> 2) == lane) {
          const int e = dd & 3;
          if (e == 0) w01.x = __fsub_rn(w01.x, 1.f);
          if (e == 1) w01.y = __fsub_rn(w01.y, 1.f);
          if (e == 2) w23.x = __fsub_rn(w23.x, 1.f);
          if (e == 3) w23.y = __fsub_rn(w23.y, 1.f);
        }
        float2 hs = make_float2(0.f, 0.f), ls = hs;
        weight_parts2_add(fmaxf(w01.x, 0.f), fmaxf(w01.y, 0.f), hs, ls);
        weight_parts2_add(fmaxf(w23.x, 0.f), fmaxf(w23.y, 0.f), hs, ls);
        sums[j] = (static_cast<long long>(small_int(hs.x + hs.y)) << 20) + small_int(ls.x + ls.y);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
      const long long tot = warp_sum_n<kPer>(sums);
      const int j = lane / (32 / kPer);
      if (lane % (32 / kPer) == 0 && warp + kWarps * j < c.n)
        a.wsum[c.u + warp + kWarps * j] = tot;
    }
  }
}

// Exclusive scan of one value per thread over the block; *total gets the block's sum.
__device__ long long block_exscan_ll(long long v, long long* sh, long long* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sh[wid] = inc;
  __syncthreads();
  long long before = 0, t = 0;
  for (int i = 0; i < nw; ++i) {
    if (i < wid) before += sh[i];
    t += sh[i];
  }
  __syncthreads();
  *total = t;
  return before + inc - v;
}

// Token of the first running sum above `target` along all of row r of p (weights p
// itself, the draw when no residual mass is left); one CTA. Each thread sums 32
// consecutive tokens, a block scan places the target in one thread's run, and that thread
// walks its 32 tokens again.
__device__ int scan_row_p(const SpecParams& a, int b, int r, unsigned long long target,
                          long long* sh) {
  __shared__ int found;
  constexpr int kPer = 32;
  const float* row = a.p + (static_cast<int64_t>(b) * (a.k + 1) + r) * a.V;
  // sum (or, with `locate`, find the token) over the run [first, first + 32)
  auto run_sum = [&](int64_t first, bool locate, long long acc) -> long long {
    long long sum = 0;
    for (int e = 0; e < kPer; ++e) {
      const int64_t x = first + e;
      if (x >= a.V) break;
      sum += token_weight(row[x], 0.f);
      if (locate && static_cast<unsigned long long>(acc + sum) > target) return x;
    }
    return locate ? -1 : sum;
  };
  if (threadIdx.x == 0) found = -1;
  __syncthreads();
  long long run = 0;
  for (int64_t tile = 0; tile < a.V; tile += static_cast<int64_t>(kThreads) * kPer) {
    const int64_t first = tile + static_cast<int64_t>(threadIdx.x) * kPer;
    const long long mine = first < a.V ? run_sum(first, false, 0) : 0;
    long long total;
    const long long acc = run + block_exscan_ll(mine, sh, &total);
    if (mine > 0 && static_cast<unsigned long long>(acc) <= target &&
        static_cast<unsigned long long>(acc + mine) > target)
      found = static_cast<int>(run_sum(first, true, acc));
    __syncthreads();
    if (found >= 0) break;
    run += total;
  }
  return found;
}

// Token of the first running sum above `target` within run m of sequence b's row r, given
// the sum `base` of every weight before the run; the calling warp (lane l holds tokens
// 128m + 4l .. 128m + 4l + 3, in order). -1 when no token reaches the target.
__device__ int run_locate(const SpecParams& a, int b, int r, bool plain, int m, long long base,
                          unsigned long long target) {
  const int lane = threadIdx.x & 31;
  const float* row = a.p + (static_cast<int64_t>(b) * (a.k + 1) + r) * a.V;
  const float* qrow = (!plain && a.q) ? a.q + (static_cast<int64_t>(b) * a.k + r) * a.V : nullptr;
  const int draft = (!plain && !a.q) ? a.drafts[b * a.k + r] : -1;
  const int64_t v0 = static_cast<int64_t>(m) * kRun + 4 * lane;
  long long w[4], mine = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int64_t v = v0 + e;
    w[e] = v < a.V ? token_weight(row[v], v == draft ? 1.f : (qrow ? qrow[v] : 0.f)) : 0;
    mine += w[e];
  }
  long long inc = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  const unsigned hit =
      __ballot_sync(0xffffffffu, static_cast<unsigned long long>(base + inc) > target);
  if (!hit) return -1;
  const int first = __ffs(hit) - 1;
  int tok = -1;
  if (lane == first) {
    long long acc = base + inc - mine;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc += w[e];
      if (tok < 0 && static_cast<unsigned long long>(acc) > target) tok = static_cast<int>(v0 + e);
    }
  }
  return __shfl_sync(0xffffffffu, tok, first);
}

// grid B: acceptance and the final token of each sequence
__global__ void __launch_bounds__(kThreads) spec_final_kernel(const SpecParams a) {
  __shared__ long long shl[kThreads / 32];
  __shared__ float shv[kThreads / 32];
  __shared__ int shi[kThreads / 32];
  __shared__ long long sh_base;
  __shared__ int sh_run;
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x;
  int n_acc = 0, tok = 0;
  if (a.greedy) {
    // argmax of each row from its chunks; accept while the draft equals it
    for (int i = 0; i <= a.k; ++i) {
      float v = -INFINITY;
      int t = INT32_MAX;
      for (int c = threadIdx.x; c < a.gent; c += kThreads) {
        const int64_t o = (static_cast<int64_t>(b) * (a.k + 1) + i) * a.gent + c;
        amax_merge(v, t, a.amax_v[o], a.amax_i[o]);
      }
      block_argmax(v, t, shv, shi);
      tok = t == INT32_MAX ? 0 : t;
      if (i == a.k || a.drafts[b * a.k + i] != tok) break;
      ++n_acc;
    }
  } else {
    // the acceptance recorded with the sequence's first run; thread t sums the run sums
    // [t*per, (t+1)*per) of the row
    const int info = a.acc[b];
    const int r = info & 0xff;
    const bool plain = (info >> 8) & 1, invalid = (info >> 9) & 1;
    if (invalid && threadIdx.x == 0) record_error(a.err, kDevBadToken);
    n_acc = r;
    const unsigned long long R = a.rnd[b * (a.k + 1) + a.k];
    const long long* rs = a.wsum + static_cast<int64_t>(b) * a.runs;
    const int per = (a.runs + kThreads - 1) / kThreads;
    const int m0 = min(static_cast<int>(threadIdx.x) * per, a.runs);
    const int m1 = min(m0 + per, a.runs);
    long long cs = 0;
    for (int m = m0; m < m1; ++m) cs += rs[m];
    if (threadIdx.x == 0) {
      sh_base = 0;
      sh_run = -1;
    }
    long long Z;
    const long long before = block_exscan_ll(cs, shl, &Z);
    tok = -1;
    if (Z > 0) {
      const unsigned long long target = __umul64hi(static_cast<unsigned long long>(Z), R << 32);
      // the run holding the target, found by the thread whose runs hold it
      if (cs > 0 && static_cast<unsigned long long>(before) <= target &&
          static_cast<unsigned long long>(before + cs) > target) {
        long long acc = before;
        for (int m = m0; m < m1; ++m) {
          const long long w = rs[m];
          if (static_cast<unsigned long long>(acc + w) > target) {
            sh_run = m;
            sh_base = acc;
            break;
          }
          acc += w;
        }
      }
      __syncthreads();
      if (threadIdx.x < 32 && sh_run >= 0)
        tok = run_locate(a, b, r, plain, sh_run, sh_base, target);
    } else {
      // no residual mass (p <= q at every token): draw from p_r itself over the row
      long long Zp = 0;
      const float* row = a.p + (static_cast<int64_t>(b) * (a.k + 1) + r) * a.V;
      for (int64_t x = threadIdx.x; x < a.V; x += kThreads)
        Zp += token_weight(row[x], 0.f);
      Zp = block_sum(Zp, shl);
      if (Zp > 0) {
        const unsigned long long target = __umul64hi(static_cast<unsigned long long>(Zp), R << 32);
        tok = scan_row_p(a, b, r, target, shl);
      }
    }
    if (tok < 0) tok = 0;
  }
  if (threadIdx.x == 0) {
    int32_t* out = a.out + static_cast<int64_t>(b) * (a.k + 1);
    for (int i = 0; i <= a.k; ++i)
      out[i] = i < n_acc ? a.drafts[b * a.k + i] : (i == n_acc ? tok : -1);
    a.num[b] = n_acc;
  }
}

}  // namespace

int spec_chunks(int V) {
  const int c = (V + 8191) / 8192;
  return c < 1 ? 1 : (c > 64 ? 64 : c);
}

int spec_runs(int V) { return (V + kRun - 1) / kRun; }

template <int kMode>
static cudaError_t launch_stream(const SpecParams& a, cudaStream_t stream) {
  // one wave of resident CTAs, each at least one stage of runs
  const int cap_runs = kMode == kResidualQ ? 16 : 32;
  const int rows = kMode == kArgmax ? a.B * (a.k + 1) : a.B;
  const int64_t units = static_cast<int64_t>(rows) * a.runs;
  const int64_t by_work = (units + cap_runs - 1) / cap_runs;
  const int64_t cap = kStreamCtasPerSm * static_cast<int64_t>(a.num_sms > 0 ? a.num_sms : 1);
  const int grid = static_cast<int>(by_work < cap ? by_work : cap);
  constexpr int smem = sizeof(StreamSmem);
  static std::atomic<uint64_t> done{0};
  const cudaError_t e = ensure_smem_limit(spec_stream_kernel<kMode>, smem, done);
  if (e != cudaSuccess) return e;
  return launch_kernel(spec_stream_kernel<kMode>, dim3(grid), dim3(kStreamThreads), smem, stream,
                       false, a);
}

cudaError_t launch_spec_accept(const SpecParams& a0, cudaStream_t stream) {
  if (a0.B == 0) return cudaSuccess;
  SpecParams a = a0;
  a.chunks = spec_chunks(a.V);
  a.chunk = ((a.V + a.chunks - 1) / a.chunks + 7) / 8 * 8;  // multiples of 8 tokens
  a.chunks = (a.V + a.chunk - 1) / a.chunk;
  a.runs = spec_runs(a.V);
  a.vec = (a.V & 3) == 0 && (reinterpret_cast<uintptr_t>(a.p) & 15) == 0 &&
          (reinterpret_cast<uintptr_t>(a.q) & 15) == 0;
  // greedy: one (max, token) entry per run with 16-byte rows, per chunk otherwise
  a.gent = a.vec ? a.runs : a.chunks;
  cudaError_t e;
  if (a.greedy) {
    e = a.vec ? launch_stream<kArgmax>(a, stream)
              : launch_kernel(spec_chunk_kernel, dim3(a.chunks, a.B), dim3(kThreads), 0, stream,
                              false, a);
  } else if (a.vec) {
    e = a.q ? launch_stream<kResidualQ>(a, stream) : launch_stream<kResidualOneHot>(a, stream);
  } else {
    // rows as 4-byte words: one wave of resident CTAs, each at least one load group per warp
    const int n = a.q ? 4 : 8;
    const int64_t units = static_cast<int64_t>(a.B) * a.runs;
    const int64_t by_work = (units + kWarps * n - 1) / (kWarps * n);
    const int64_t cap = kCtasPerSm * static_cast<int64_t>(a.num_sms > 0 ? a.num_sms : 1);
    const int grid = static_cast<int>(by_work < cap ? by_work : cap);
    e = a.q ? launch_kernel(spec_run_kernel<true>, dim3(grid), dim3(kThreads), 0, stream, false, a)
            : launch_kernel(spec_run_kernel<false>, dim3(grid), dim3(kThreads), 0, stream, false, a);
  }
  if (e != cudaSuccess) return e;
  return launch_kernel(spec_final_kernel, dim3(a.B), dim3(kThreads), 0, stream, true, a);
}

}  // namespace ps
