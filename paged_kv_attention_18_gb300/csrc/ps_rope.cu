// Rotary position embedding fused with the KV scatter. Every new token's query and key are
// rotated by its position before the key is cached, so the cache holds rotated keys and
// the attention reads them as they are (tinyserve "Highlights" table, forward-pass row:
// rotary embeddings in the Qwen2 decoder; PageServe section 01: explicit position ids per
// packed token). The rotation is the rotate-half form: for frequency i < D/2,
//     x'[i]       = x[i] cos(a) - x[i + D/2] sin(a)
//     x'[i + D/2] = x[i + D/2] cos(a) + x[i] sin(a),   a = pos * theta^(-2i/D).
// Each frequency is held as a 64-bit fixed-point fraction of a turn, F_i = f_i / (2 pi) * 2^64
// (computed once per CTA in fp64); the integer product pos * F_i, wrapping modulo 2^64, is
// the angle reduced modulo one turn, exactly; its top 32 bits as a signed fraction of a turn
// give an fp32 angle in [-pi, pi), whose cosine and sine are taken in fp32. The products are
// fp32 and the result is rounded once to the 16-bit type.
#include "ps_common.cuh"
#include "ps_launch.h"

namespace ps {

namespace {

constexpr int kRopeThreads = 256;

template <bool kBF16>
__device__ __forceinline__ float2 unpack2(uint32_t u) {
  if constexpr (kBF16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&u));
  }
}

// Rotate 8 consecutive pairs: lo holds elements i..i+7, hi elements i+D/2..i+D/2+7.
template <bool kBF16>
__device__ __forceinline__ void rotate8(uint4& lo, uint4& hi, const float* c, const float* s) {
  uint32_t* l = reinterpret_cast<uint32_t*>(&lo);
  uint32_t* h = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float2 a = unpack2<kBF16>(l[w]), b = unpack2<kBF16>(h[w]);
    const float c0 = c[2 * w], c1 = c[2 * w + 1], s0 = s[2 * w], s1 = s[2 * w + 1];
    l[w] = pack2<kBF16>(__fsub_rn(__fmul_rn(a.x, c0), __fmul_rn(b.x, s0)),
                        __fsub_rn(__fmul_rn(a.y, c1), __fmul_rn(b.y, s1)));
    h[w] = pack2<kBF16>(__fadd_rn(__fmul_rn(b.x, c0), __fmul_rn(a.x, s0)),
                        __fadd_rn(__fmul_rn(b.y, c1), __fmul_rn(a.y, s1)));
  }
}

constexpr double kInvTwoPi = 0.15915494309189533576888376337251436203445964574046;
constexpr double kTwoTo64 = 18446744073709551616.0;
constexpr float kTurnToRad = 1.46291807926715968e-09f;  // 2 pi / 2^32
constexpr int kTokensPerPass = 8;
constexpr int kRopeCtasPerSm = 3;
constexpr int kUnits = 4;  // q/k units per thread per round

// One CTA takes a contiguous range of passes of 8 tokens. A pass's q and k rows are
// 8 * (H_q + H_kv) rows of D elements; thread t takes chunk pair t % (D/16) (16-byte chunks
// i..i+7 and i+D/2..i+D/2+7) of rows t / (D/16), + 256 / (D/16), ... A round first issues
// every load of its units and of the V rows, then computes the pass's cosines and sines
// into one of two shared tables while the loads are in flight; after one barrier it
// rotates and stores. The two tables let the next pass start without a second barrier.
template <bool kBF16, int D>
__global__ void __launch_bounds__(kRopeThreads, kRopeCtasPerSm)
    rope_reshape_and_cache_kernel(uint4* __restrict__ q, const uint4* __restrict__ k,
                                  const uint4* __restrict__ v, const int32_t* __restrict__ pos,
                                  const int32_t* __restrict__ slots, uint4* __restrict__ k_pool,
                                  uint4* __restrict__ v_pool, int T, int H_q, int H_kv,
                                  int64_t num_slots, double log2_theta, int* err) {
  constexpr int kHalf = D / 2, kChunks = kHalf / 8;  // 16-byte chunks per half row
  constexpr int kRowsPerRound = kRopeThreads / kChunks;
  __shared__ unsigned long long turns[kHalf];  // f_i / (2 pi) in units of 2^-64 turn
  __shared__ float cs[2][kTokensPerPass][kHalf], sn[2][kTokensPerPass][kHalf];
  for (int i = threadIdx.x; i < kHalf; i += blockDim.x)
    turns[i] = __double2ull_rn(exp2(-(2.0 * i / D) * log2_theta) * kInvTwoPi * kTwoTo64);
  const int heads = H_q + H_kv;
  const int rows = kTokensPerPass * heads;  // q and k rows of a pass
  const int vecs = H_kv * D / 8;            // 16-byte words of a token's V row
  const int ch = threadIdx.x % kChunks, row0 = threadIdx.x / kChunks;
  const int passes = (T + kTokensPerPass - 1) / kTokensPerPass;
  const int p_lo = static_cast<int>(static_cast<int64_t>(passes) * blockIdx.x / gridDim.x);
  const int p_hi = static_cast<int>(static_cast<int64_t>(passes) * (blockIdx.x + 1) / gridDim.x);
  __syncthreads();
  int buf = 0;
  for (int pass = p_lo; pass < p_hi; ++pass, buf ^= 1) {
    const int t0 = pass * kTokensPerPass;
    for (int r0 = 0; r0 < rows; r0 += kUnits * kRowsPerRound) {
      // 1. loads of this round's units, and (first round) of the pass's V rows
      uint4 lo[kUnits], hi[kUnits];
      int slot[kUnits];
#pragma unroll
      for (int j = 0; j < kUnits; ++j) {
        const int row = r0 + row0 + j * kRowsPerRound;
        const int u = row / heads, head = row - u * heads, t = t0 + u;
        slot[j] = -2;  // -2: no unit; -1: a k row with nothing to cache
        if (row >= rows || t >= T) continue;
        const uint4* src;
        if (head < H_q) {
          slot[j] = -3;  // a q row
          src = q + (static_cast<int64_t>(t) * H_q + head) * (D / 8);
        } else {
          const int sl = slots[t];
          slot[j] = sl >= 0 && sl < num_slots ? sl : -1;
          src = k + (static_cast<int64_t>(t) * H_kv + head - H_q) * (D / 8);
          if (slot[j] < 0) continue;
        }
        lo[j] = src[ch];
        hi[j] = src[ch + kChunks];
      }
      constexpr int kV = 1;  // V words per thread per pass held in registers
      uint4 vv[kV];
      int vslot[kV];
      if (r0 == 0) {
#pragma unroll
        for (int j = 0; j < kV; ++j) {
          const int x = threadIdx.x + j * kRopeThreads;
          const int u = x / vecs, w = x - u * vecs, t = t0 + u;
          vslot[j] = -1;
          if (u >= kTokensPerPass || t >= T) continue;
          const int vs = slots[t];
          if (vs >= num_slots) {
            if (w == 0) record_error(err, kDevBadSlot);
            continue;
          }
          vslot[j] = vs;
          if (vs >= 0) vv[j] = v[static_cast<int64_t>(t) * vecs + w];
        }
        // 2. the pass's cosines and sines
        for (int x = threadIdx.x; x < kTokensPerPass * kHalf; x += blockDim.x) {
          const int u = x / kHalf, i = x - u * kHalf;
          const int t = t0 + u;
          if (t >= T) continue;
          const unsigned long long ph =
              static_cast<unsigned long long>(static_cast<uint32_t>(pos[t])) * turns[i];
          const float r = static_cast<float>(static_cast<int32_t>(ph >> 32)) * kTurnToRad;
          float sf, cf;
          sincosf(r, &sf, &cf);
          cs[buf][u][i] = cf;
          sn[buf][u][i] = sf;
        }
        __syncthreads();
      }
      // 3. rotate and store
#pragma unroll
      for (int j = 0; j < kUnits; ++j) {
        if (slot[j] < -2 || slot[j] >= 0) {
          const int row = r0 + row0 + j * kRowsPerRound;
          const int u = row / heads, head = row - u * heads, t = t0 + u;
          const int i0 = ch * 8;
          rotate8<kBF16>(lo[j], hi[j], cs[buf][u] + i0, sn[buf][u] + i0);
          uint4* dst = head < H_q
                           ? q + (static_cast<int64_t>(t) * H_q + head) * (D / 8)
                           : k_pool + (static_cast<int64_t>(slot[j]) * H_kv + head - H_q) * (D / 8);
          dst[ch] = lo[j];
          dst[ch + kChunks] = hi[j];
        }
      }
      if (r0 == 0) {
        // the V rows as they are
#pragma unroll
        for (int j = 0; j < kV; ++j) {
          const int x = threadIdx.x + j * kRopeThreads;
          if (vslot[j] >= 0) v_pool[static_cast<int64_t>(vslot[j]) * vecs + x % vecs] = vv[j];
        }
        // V words beyond what the registers held (more than 256 in a pass)
        for (int x = threadIdx.x + kV * kRopeThreads; x < kTokensPerPass * vecs;
             x += kRopeThreads) {
          const int u = x / vecs, w = x - u * vecs, t = t0 + u;
          if (t >= T) continue;
          const int vs = slots[t];
          if (vs >= num_slots) {
            if (w == 0) record_error(err, kDevBadSlot);
            continue;
          }
          if (vs >= 0) v_pool[static_cast<int64_t>(vs) * vecs + w] = v[static_cast<int64_t>(t) * vecs + w];
        }
      }
    }
  }
}

template <bool kBF16, int D>
cudaError_t launch_rope_t(void* q, const void* k, const void* v, const int32_t* pos,
                          const int32_t* slots, void* k_pool, void* v_pool, int T, int H_q,
                          int H_kv, int num_blocks, float theta, int* err, int num_sms,
                          cudaStream_t stream) {
  // one wave of resident CTAs, each a contiguous range of passes
  const int passes = (T + kTokensPerPass - 1) / kTokensPerPass;
  const int grid = passes < num_sms * kRopeCtasPerSm ? passes : num_sms * kRopeCtasPerSm;
  rope_reshape_and_cache_kernel<kBF16, D><<<grid, kRopeThreads, 0, stream>>>(
      static_cast<uint4*>(q), static_cast<const uint4*>(k), static_cast<const uint4*>(v), pos,
      slots, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), T, H_q, H_kv,
      static_cast<int64_t>(num_blocks) * kBlockSize, log2(static_cast<double>(theta)), err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope_reshape_and_cache(void* q, const void* k, const void* v,
                                          const int32_t* pos, const int32_t* slots,
                                          void* k_pool, void* v_pool, int T, int H_q, int H_kv,
                                          int D, int num_blocks, float theta, bool bf16,
                                          int* err, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (D == 128)
    return bf16 ? launch_rope_t<true, 128>(q, k, v, pos, slots, k_pool, v_pool, T, H_q, H_kv,
                                           num_blocks, theta, err, num_sms, stream)
                : launch_rope_t<false, 128>(q, k, v, pos, slots, k_pool, v_pool, T, H_q, H_kv,
                                            num_blocks, theta, err, num_sms, stream);
  return bf16 ? launch_rope_t<true, 64>(q, k, v, pos, slots, k_pool, v_pool, T, H_q, H_kv,
                                        num_blocks, theta, err, num_sms, stream)
              : launch_rope_t<false, 64>(q, k, v, pos, slots, k_pool, v_pool, T, H_q, H_kv,
                                         num_blocks, theta, err, num_sms, stream);
}

}  // namespace ps
