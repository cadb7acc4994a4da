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

// Each pass of a CTA takes 8 tokens. A thread first issues the loads of its units (a unit
// is one (token, head) pair of 16-byte chunks i..i+7 and i+D/2..i+D/2+7 of q or k), then
// computes the tokens' cosines and sines into shared memory while those loads are in
// flight, and after the barrier rotates and stores; the V rows are copied last.
template <bool kBF16, int D>
__global__ void __launch_bounds__(kRopeThreads)
    rope_reshape_and_cache_kernel(uint4* __restrict__ q, const uint4* __restrict__ k,
                                  const uint4* __restrict__ v, const int32_t* __restrict__ pos,
                                  const int32_t* __restrict__ slots, uint4* __restrict__ k_pool,
                                  uint4* __restrict__ v_pool, int T, int H_q, int H_kv,
                                  int64_t num_slots, double log2_theta, int* err) {
  constexpr int kHalf = D / 2, kChunks = kHalf / 8;  // 16-byte chunks per half row
  constexpr int kUnits = 4;                          // q/k units per thread per round
  __shared__ unsigned long long turns[kHalf];  // f_i / (2 pi) in units of 2^-64 turn
  __shared__ float cs[kTokensPerPass][kHalf], sn[kTokensPerPass][kHalf];
  for (int i = threadIdx.x; i < kHalf; i += blockDim.x)
    turns[i] = __double2ull_rn(exp2(-(2.0 * i / D) * log2_theta) * kInvTwoPi * kTwoTo64);
  __syncthreads();
  const int units_tok = (H_q + H_kv) * kChunks;
  const int units = kTokensPerPass * units_tok;
  const int vecs = H_kv * D / 8;
  for (int t0 = blockIdx.x * kTokensPerPass; t0 < T; t0 += gridDim.x * kTokensPerPass) {
    for (int r0 = 0; r0 < units; r0 += kUnits * kRopeThreads) {
      // 1. loads of this round's units
      uint4 lo[kUnits], hi[kUnits];
      int tok[kUnits], head[kUnits], ch[kUnits], slot[kUnits];
#pragma unroll
      for (int j = 0; j < kUnits; ++j) {
        const int x = r0 + j * kRopeThreads + threadIdx.x;
        const int u = x / units_tok, w = x - u * units_tok;
        tok[j] = (x < units && t0 + u < T) ? t0 + u : -1;
        head[j] = w / kChunks;
        ch[j] = w - head[j] * kChunks;
        slot[j] = -1;
        if (tok[j] < 0) continue;
        const uint4* row;
        if (head[j] < H_q) {
          row = q + (static_cast<int64_t>(tok[j]) * H_q + head[j]) * (D / 8);
        } else {
          slot[j] = slots[tok[j]];
          row = k + (static_cast<int64_t>(tok[j]) * H_kv + head[j] - H_q) * (D / 8);
          if (slot[j] < 0 || slot[j] >= num_slots) {
            tok[j] = -1;  // nothing to cache for this token
            continue;
          }
        }
        lo[j] = row[ch[j]];
        hi[j] = row[ch[j] + kChunks];
      }
      // 2. the tokens' cosines and sines (first round of the pass)
      if (r0 == 0) {
        for (int x = threadIdx.x; x < kTokensPerPass * kHalf; x += blockDim.x) {
          const int u = x / kHalf, i = x - u * kHalf;
          const int t = t0 + u;
          if (t >= T) continue;
          const unsigned long long ph =
              static_cast<unsigned long long>(static_cast<uint32_t>(pos[t])) * turns[i];
          const float r = static_cast<float>(static_cast<int32_t>(ph >> 32)) * kTurnToRad;
          float sf, cf;
          sincosf(r, &sf, &cf);
          cs[u][i] = cf;
          sn[u][i] = sf;
        }
        __syncthreads();
      }
      // 3. rotate and store
#pragma unroll
      for (int j = 0; j < kUnits; ++j) {
        if (tok[j] < 0) continue;
        const int u = tok[j] - t0, i0 = ch[j] * 8;
        rotate8<kBF16>(lo[j], hi[j], cs[u] + i0, sn[u] + i0);
        uint4* dst;
        if (head[j] < H_q)
          dst = q + (static_cast<int64_t>(tok[j]) * H_q + head[j]) * (D / 8);
        else
          dst = k_pool + (static_cast<int64_t>(slot[j]) * H_kv + head[j] - H_q) * (D / 8);
        dst[ch[j]] = lo[j];
        dst[ch[j] + kChunks] = hi[j];
      }
    }
    // the V rows as they are
    for (int x = threadIdx.x; x < kTokensPerPass * vecs; x += blockDim.x) {
      const int u = x / vecs, w = x - u * vecs;
      const int t = t0 + u;
      if (t >= T) continue;
      const int vs = slots[t];
      if (vs >= num_slots) {
        if (w == 0) record_error(err, kDevBadSlot);
        continue;
      }
      if (vs >= 0) v_pool[static_cast<int64_t>(vs) * vecs + w] = v[static_cast<int64_t>(t) * vecs + w];
    }
    __syncthreads();  // the pass's cosines are read before the next pass writes them
  }
}

template <bool kBF16, int D>
cudaError_t launch_rope_t(void* q, const void* k, const void* v, const int32_t* pos,
                          const int32_t* slots, void* k_pool, void* v_pool, int T, int H_q,
                          int H_kv, int num_blocks, float theta, int* err, int num_sms,
                          cudaStream_t stream) {
  const int passes = (T + kTokensPerPass - 1) / kTokensPerPass;
  const int grid = passes < num_sms * 8 ? passes : num_sms * 8;
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
