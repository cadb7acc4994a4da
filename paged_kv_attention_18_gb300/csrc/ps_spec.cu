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
// Two kernels: the first, one CTA per (sequence, chunk of the vocabulary), reduces its
// chunk of the rows it needs (fixed-point sums of the residual row, or argmaxes of every
// row in greedy mode) so the whole GPU streams the probability rows; the second, one CTA
// per sequence, combines the chunks and scans only the chunk that holds the sample.
#include "ps_common.cuh"
#include "ps_launch.h"

namespace ps {

namespace {

constexpr int kThreads = 256;  // also the largest chunk count (spec_chunks caps it at 64)

// trunc(w * 2^40) for w > 0 (0 otherwise), from the float's fields: a normal w is
// (2^23 + mantissa) * 2^(exponent - 150), so the result is that integer shifted by
// exponent - 110; subnormals (below 2^-126) give 0. Integer shifts only: the same value
// as an exact float-to-integer conversion, without the conversion unit.
__device__ __forceinline__ int64_t fixed_weight(float w) {
  if (!(w > 0.f)) return 0;
  const uint32_t bits = __float_as_uint(w);
  const int e = static_cast<int>(bits >> 23);  // sign bit is 0
  if (e == 0) return 0;
  const uint64_t m = (bits & 0x7fffffu) | 0x800000u;
  const int sh = e - 110;
  if (sh >= 0) return static_cast<int64_t>(m << sh);  // w < 2^23, so sh <= 39
  return sh > -64 ? static_cast<int64_t>(m >> -sh) : 0;
}

// Residual weight of token v at row r: max(p - q, 0) with q the draft distribution, or
// the one-hot of the draft token when there is none (a deterministic proposer), or 0 when
// r is the bonus row or the draft was invalid (the weight is then p itself).
__device__ __forceinline__ float residual(const SpecParams& a, int b, int r, bool bonus,
                                          int64_t v, float pv) {
  if (bonus) return pv;
  float qv;
  if (a.q) {
    qv = a.q[(static_cast<int64_t>(b) * a.k + r) * a.V + v];
  } else {
    qv = v == a.drafts[b * a.k + r] ? 1.f : 0.f;
  }
  return fmaxf(__fsub_rn(pv, qv), 0.f);
}

// Acceptance of sequence b's drafts under the rejection rule, by the calling warp (one
// lane per draft, k <= 31): the number accepted; *plain when the final draw is from p
// itself (every draft survived, or the stopping draft id lies outside the vocabulary,
// then also *invalid).
__device__ int accepted_warp(const SpecParams& a, int b, bool* plain, bool* invalid) {
  const int lane = threadIdx.x & 31;
  bool ok = true, bad = false;
  if (lane < a.k) {
    const int d = a.drafts[b * a.k + lane];
    if (d < 0 || d >= a.V) {
      bad = true;
      ok = false;
    } else {
      const float pv = a.p[(static_cast<int64_t>(b) * (a.k + 1) + lane) * a.V + d];
      const float qv = a.q ? a.q[(static_cast<int64_t>(b) * a.k + lane) * a.V + d] : 1.f;
      const double lhs = __dmul_rn(static_cast<double>(a.rnd[b * (a.k + 1) + lane]), qv);
      const double rhs = __dmul_rn(static_cast<double>(pv), 4294967296.0);
      ok = lhs < rhs;
    }
  }
  const unsigned rej = __ballot_sync(0xffffffffu, lane < a.k && !ok);
  const int r = rej ? __ffs(rej) - 1 : a.k;
  const bool inv = __shfl_sync(0xffffffffu, bad ? 1 : 0, r & 31) != 0;
  *invalid = rej != 0 && inv;
  *plain = rej == 0 || *invalid;
  return r;
}

// The acceptance of sequence b, decided by warp 0 and shared with the block.
__device__ int accepted_block(const SpecParams& a, int b, bool* plain, bool* invalid) {
  __shared__ int sh_r, sh_flags;
  if (threadIdx.x < 32) {
    bool pl, inv;
    const int r = accepted_warp(a, b, &pl, &inv);
    if (threadIdx.x == 0) {
      sh_r = r;
      sh_flags = (pl ? 1 : 0) | (inv ? 2 : 0);
    }
  }
  __syncthreads();
  *plain = sh_flags & 1;
  *invalid = (sh_flags & 2) != 0;
  return sh_r;
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

// grid (chunks, B): chunk statistics of the rows sequence b needs. With V a multiple of 4
// every row starts 16-byte aligned and chunks are multiples of 8 tokens, so rows stream
// as float4 loads, two per thread in flight.
__global__ void __launch_bounds__(kThreads) spec_chunk_kernel(const SpecParams a) {
  __shared__ long long shl[kThreads / 32];
  __shared__ float shv[kThreads / 32];
  __shared__ int shi[kThreads / 32];
  pdl_launch_dependents();
  const int c = blockIdx.x, b = blockIdx.y;
  const int64_t lo = static_cast<int64_t>(c) * a.chunk;
  const int64_t hi = lo + a.chunk < a.V ? lo + a.chunk : a.V;
  const bool vec = (a.V & 3) == 0;
  if (a.greedy) {
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
        const int64_t o = (static_cast<int64_t>(b) * (a.k + 1) + i) * a.chunks + c;
        a.amax_v[o] = v;
        a.amax_i[o] = t;
      }
    }
    return;
  }
  bool plain, invalid;
  const int r = accepted_block(a, b, &plain, &invalid);
  if (c == 0 && threadIdx.x == 0) a.acc[b] = r | (plain ? 1 << 8 : 0) | (invalid ? 1 << 9 : 0);
  const float* row = a.p + (static_cast<int64_t>(b) * (a.k + 1) + r) * a.V;
  const float* qrow = (!plain && a.q) ? a.q + (static_cast<int64_t>(b) * a.k + r) * a.V : nullptr;
  const int draft = (!plain && !a.q) ? a.drafts[b * a.k + r] : -1;
  long long s = 0;
  if (vec) {
    // four float4 loads of p (and of q) per thread in flight
    const float4* p4 = reinterpret_cast<const float4*>(row);
    const float4* q4 = reinterpret_cast<const float4*>(qrow);
    for (int64_t x0 = lo / 4 + threadIdx.x; x0 < hi / 4; x0 += 4 * kThreads) {
      float4 f[4], g[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t x = x0 + u * kThreads;
        const bool in = x < hi / 4;
        f[u] = in ? __ldcs(p4 + x) : make_float4(0.f, 0.f, 0.f, 0.f);
        g[u] = (in && qrow) ? __ldcs(q4 + x) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float pv[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
        const float qv[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t v = 4 * (x0 + u * kThreads) + e;
          const float qe = qrow ? qv[e] : (v == draft ? 1.f : 0.f);
          s += fixed_weight(plain ? pv[e] : fmaxf(__fsub_rn(pv[e], qe), 0.f));
        }
      }
    }
  } else {
    for (int64_t x = lo + threadIdx.x; x < hi; x += kThreads)
      s += fixed_weight(residual(a, b, r, plain, x, row[x]));
  }
  s = block_sum(s, shl);
  if (threadIdx.x == 0) a.wsum[static_cast<int64_t>(b) * a.chunks + c] = s;
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

// Token of the first running sum above `target` within [lo, hi) of row r (weights
// recomputed), given the sum `base` of every weight before lo; one CTA. Each thread sums
// 32 consecutive tokens, a block scan places the target in one thread's run, and that
// thread walks its 32 tokens again.
__device__ int scan_for(const SpecParams& a, int b, int r, bool plain, int64_t lo, int64_t hi,
                        long long base, unsigned long long target, long long* sh) {
  __shared__ int found;
  constexpr int kPer = 32;
  const float* row = a.p + (static_cast<int64_t>(b) * (a.k + 1) + r) * a.V;
  const float* qrow = (!plain && a.q) ? a.q + (static_cast<int64_t>(b) * a.k + r) * a.V : nullptr;
  const int draft = (!plain && !a.q) ? a.drafts[b * a.k + r] : -1;
  const bool vec = (a.V & 3) == 0 && (lo & 7) == 0;
  auto weight = [&](int64_t x, float pv, float qv) -> long long {
    if (x >= hi) return 0;
    if (plain) return fixed_weight(pv);
    const float qe = qrow ? qv : (x == draft ? 1.f : 0.f);
    return fixed_weight(fmaxf(__fsub_rn(pv, qe), 0.f));
  };
  // sum (or, with `target_in`, locate) over the run [first, first + 32)
  auto run_sum = [&](int64_t first, bool locate, long long acc) -> long long {
    long long sum = 0;
    if (vec && first + kPer <= hi) {
      const float4* p4 = reinterpret_cast<const float4*>(row + first);
      const float4* q4 = reinterpret_cast<const float4*>(qrow ? qrow + first : row + first);
#pragma unroll
      for (int e4 = 0; e4 < kPer / 4; ++e4) {
        const float4 f = p4[e4];
        const float4 g = qrow ? q4[e4] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float pv[4] = {f.x, f.y, f.z, f.w};
        const float qv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t x = first + 4 * e4 + e;
          sum += weight(x, pv[e], qv[e]);
          if (locate && static_cast<unsigned long long>(acc + sum) > target) return x;
        }
      }
    } else {
      for (int e = 0; e < kPer; ++e) {
        const int64_t x = first + e;
        if (x >= hi) break;
        sum += weight(x, row[x], qrow ? qrow[x] : 0.f);
        if (locate && static_cast<unsigned long long>(acc + sum) > target) return x;
      }
    }
    return locate ? -1 : sum;
  };
  if (threadIdx.x == 0) found = -1;
  __syncthreads();
  long long run = base;
  for (int64_t tile = lo; tile < hi; tile += static_cast<int64_t>(kThreads) * kPer) {
    const int64_t first = tile + static_cast<int64_t>(threadIdx.x) * kPer;
    const long long mine = first < hi ? run_sum(first, false, 0) : 0;
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

// grid B: acceptance and the final token of each sequence
__global__ void __launch_bounds__(kThreads) spec_final_kernel(const SpecParams a) {
  __shared__ long long shl[kThreads / 32];
  __shared__ float shv[kThreads / 32];
  __shared__ int shi[kThreads / 32];
  __shared__ long long sh_base;
  __shared__ int sh_chunk;
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x;
  int n_acc = 0, tok = 0;
  if (a.greedy) {
    // argmax of each row from its chunks; accept while the draft equals it
    for (int i = 0; i <= a.k; ++i) {
      float v = -INFINITY;
      int t = INT32_MAX;
      for (int c = threadIdx.x; c < a.chunks; c += kThreads) {
        const int64_t o = (static_cast<int64_t>(b) * (a.k + 1) + i) * a.chunks + c;
        amax_merge(v, t, a.amax_v[o], a.amax_i[o]);
      }
      block_argmax(v, t, shv, shi);
      tok = t == INT32_MAX ? 0 : t;
      if (i == a.k || a.drafts[b * a.k + i] != tok) break;
      ++n_acc;
    }
  } else {
    // the acceptance recorded by the first chunk's CTA, and the chunk sums (chunks <=
    // threads) with their scan, loaded together
    const int info = a.acc[b];
    const int r = info & 0xff;
    const bool plain = (info >> 8) & 1, invalid = (info >> 9) & 1;
    if (invalid && threadIdx.x == 0) record_error(a.err, kDevBadToken);
    n_acc = r;
    const unsigned long long R = a.rnd[b * (a.k + 1) + a.k];
    if (threadIdx.x == 0) {
      sh_base = 0;
      sh_chunk = 0;
    }
    const long long cs = threadIdx.x < a.chunks ? a.wsum[static_cast<int64_t>(b) * a.chunks + threadIdx.x] : 0;
    long long Z;
    const long long before = block_exscan_ll(cs, shl, &Z);
    if (Z > 0) {
      const unsigned long long target = __umul64hi(static_cast<unsigned long long>(Z), R << 32);
      // the chunk holding the target
      if (threadIdx.x < a.chunks && cs > 0 && static_cast<unsigned long long>(before) <= target &&
          static_cast<unsigned long long>(before + cs) > target) {
        sh_base = before;
        sh_chunk = threadIdx.x;
      }
      __syncthreads();
      const int64_t lo = static_cast<int64_t>(sh_chunk) * a.chunk;
      const int64_t hi = lo + a.chunk < a.V ? lo + a.chunk : a.V;
      tok = scan_for(a, b, r, plain, lo, hi, sh_base, target, shl);
    } else {
      // no residual mass (p <= q at every token): draw from p_r itself over the row
      long long Zp = 0;
      const float* row = a.p + (static_cast<int64_t>(b) * (a.k + 1) + r) * a.V;
      for (int64_t x = threadIdx.x; x < a.V; x += kThreads) Zp += fixed_weight(row[x]);
      Zp = block_sum(Zp, shl);
      tok = 0;
      if (Zp > 0) {
        const unsigned long long target = __umul64hi(static_cast<unsigned long long>(Zp), R << 32);
        tok = scan_for(a, b, r, true, 0, a.V, 0, target, shl);
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

cudaError_t launch_spec_accept(const SpecParams& a0, cudaStream_t stream) {
  if (a0.B == 0) return cudaSuccess;
  SpecParams a = a0;
  a.chunks = spec_chunks(a.V);
  a.chunk = ((a.V + a.chunks - 1) / a.chunks + 7) / 8 * 8;  // multiples of 8 tokens
  a.chunks = (a.V + a.chunk - 1) / a.chunk;
  cudaError_t e = launch_kernel(spec_chunk_kernel, dim3(a.chunks, a.B), dim3(kThreads), 0,
                                stream, false, a);
  if (e != cudaSuccess) return e;
  return launch_kernel(spec_final_kernel, dim3(a.B), dim3(kThreads), 0, stream, true, a);
}

}  // namespace ps
