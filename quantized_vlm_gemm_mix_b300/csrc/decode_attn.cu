// Fused MiX decode attention (one query token per head, GQA) over an MX KV
// cache: the accelerator dataflow of the pchao.org digest of "MiX:
// Micro-Inverted-Scaling ..." (Method section, accelerator bullet: K-mean
// subtraction with the frozen prefill mean, Q-K^T on the dual-format
// matmul, the SFU softmax, MiX requantisation of P, P-V on the dual-format
// matmul) as two kernels and no host round trip.
//
//  attn_qk_kernel   grid (token chunks, KV heads).  Quantises the group's
//                   query heads to MiX-4.5b, appends the new key (K' =
//                   fp32(k) - mean, MXINT4 along head_dim) when this chunk
//                   holds the last token, then S = Eq. (6) shift-add for
//                   every (head, token) of the chunk, and the chunk's softmax
//                   statistics (max, sum of exp) per head.
//  attn_pv_kernel   same grid.  Combines the statistics of all chunks, forms
//                   P = exp(s - m) / l for its chunk, requantises P to
//                   MiX-4.5b (32-token blocks), P-V by Eq. (6) shift-add
//                   against the MXINT4 V plane (blocks along tokens), writes
//                   a partial O; the last CTA of a KV head (an atomic ticket,
//                   no waiting) sums the partials in chunk order.
//
// Every block product is an exact integer (as on the shift-add PE); block
// terms are accumulated in fp32.  The work is tiny and latency-bound: the
// whole 8192-token cache of four KV heads is 4.3 MB.
#include <cuda_runtime.h>

#include "mix_common.cuh"
#include "mix_internal.h"

namespace mixk {
namespace {

constexpr int kD = 128;        // head_dim
constexpr int kChunk = 256;    // tokens per CTA
constexpr int kThreads = 256;
constexpr int kMaxG = 16;      // query heads per KV head

struct AttnArgs {
  const void* q;
  const void* k_new;
  const float* k_mean;
  int bf16;
  uint8_t* k_codes;
  uint8_t* k_scales;
  const uint8_t* v_codes;
  const uint8_t* v_scales;
  int64_t v_ld;
  int64_t T, Tpad;
  int C, HQ, HK, G;
  float sm_scale;
  int q_ebias, p_ebias;
  float* S;        // [HQ][Tpad]
  float2* stats;   // [C][HQ] (chunk max, chunk sum of exp)
  float* opart;    // [C][HQ][D]
  unsigned* tickets;  // [HK]
  float* out;      // [HQ][D]
  uint8_t* p_codes;    // optional [HQ][v_ld / 2]
  uint16_t* p_shared;  // optional [HQ][v_ld / 32]
};

__device__ __forceinline__ uint32_t load_bits(const void* p, bool bf16, int64_t i) {
  return bf16 ? (uint32_t)static_cast<const uint16_t*>(p)[i] << 16 : __float_as_uint(static_cast<const float*>(p)[i]);
}

// MiX element code -> s * 2^(7 - de) (0 for the zero code, +1 for the
// recycled -0 code, one binade below de = 6).
__device__ __forceinline__ int mix_factor(uint32_t c) {
  if (c == 7u) return 0;
  if (c == 15u) return 1;
  const int v = 128 >> (c & 7u);
  return (c & 8u) ? -v : v;
}

// Decode one quantised MiX-4.5b block into factors and (Emax, packed m3s).
__device__ __forceinline__ void mix_unpack(const uint4& cw, uint32_t sh, int ebias, int16_t* f, int2* meta) {
  const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 8; ++i) f[8 * j + i] = (int16_t)mix_factor((w[j] >> (4 * i)) & 0xFu);
  const int mk = (int)(((sh >> 4) & 7u) | (((sh >> 7) & 7u) << 8) | (((sh >> 10) & 7u) << 16) |
                       (((sh >> 13) & 7u) << 24));
  *meta = make_int2((int)(sh & 0xFu) + ebias, mk);
}

// One Eq. (6) block: 32 INT4 weights (two's complement nibbles) against 32
// MiX factors, four 8-way sub-trees each times (8 + m3), one exponent add.
__device__ __forceinline__ float eq6_block(const int* bv, const int16_t* f, int2 meta, int X) {
  int blockv = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += bv[8 * q + i] * (int)f[8 * q + i];
    blockv += s * (8 + ((meta.y >> (8 * q)) & 0xFF));
  }
  return ldexpf((float)blockv, meta.x + X - 12);  // 2^(Emax + X - 10 - c_B), c_B = 2 for MXINT4
}

__device__ __forceinline__ void int4_values(const uint4& cw, int* bv) {
  const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = (int)((w[j] >> (4 * i)) & 0xFu);
      bv[8 * j + i] = (c & 8) ? c - 16 : c;
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__global__ void __launch_bounds__(kThreads) attn_qk_kernel(AttnArgs a) {
  __shared__ __align__(16) int16_t qf[kMaxG][kD];
  __shared__ int2 qmeta[kMaxG][kD / 32];
  __shared__ float red[kThreads / 32];
  const int c = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
  const bool bf16 = a.bf16 != 0;
  if (c == 0 && tid == 0) a.tickets[g] = 0u;  // for attn_pv_kernel, which runs after this grid

  // the group's query heads -> MiX-4.5b, decoded into factors
  if (tid < a.G * 4) {
    const int h = tid >> 2, b = tid & 3;
    uint32_t u[32];
    const int64_t base = (int64_t)(g * a.G + h) * kD + 32 * b;
#pragma unroll
    for (int i = 0; i < 32; ++i) u[i] = load_bits(a.q, bf16, base + i);
    uint4 cw;
    uint32_t sh;
    mix_block32<2>(u, a.q_ebias, true, cw, sh);
    mix_unpack(cw, sh, a.q_ebias, &qf[h][32 * b], &qmeta[h][b]);
  }
  // append the new key: K' = fp32(k) - mean, MXINT4 along head_dim
  const int64_t t_new = a.T - 1;
  if (a.k_new != nullptr && t_new / kChunk == c && tid < 4) {
    const int b = tid;
    uint32_t u[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int64_t e = (int64_t)g * kD + 32 * b + i;
      u[i] = __float_as_uint(__fsub_rn(__uint_as_float(load_bits(a.k_new, bf16, e)), a.k_mean[e]));
    }
    uint4 w;
    uint32_t sc;
    mx_block32<false>(u, MX_RULE_CEIL, w, sc);
    const int64_t row = t_new * a.HK + g;
    *reinterpret_cast<uint4*>(a.k_codes + row * (kD / 2) + 16 * b) = w;
    a.k_scales[row * (kD / 32) + b] = (uint8_t)sc;
  }
  __syncthreads();

  // S for one token per thread
  const int64_t t = (int64_t)c * kChunk + tid;
  const bool valid = t < a.T;
  float acc[kMaxG];
#pragma unroll
  for (int h = 0; h < kMaxG; ++h) acc[h] = 0.0f;
  if (valid) {
    const int64_t row = t * a.HK + g;
    const uint8_t* kc = a.k_codes + row * (kD / 2);
    const uint32_t scw = *reinterpret_cast<const uint32_t*>(a.k_scales + row * (kD / 32));
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint4 cw = *reinterpret_cast<const uint4*>(kc + 16 * b);
      const int X = (int)((scw >> (8 * b)) & 0xFFu) - 127;
      int bv[32];
      int4_values(cw, bv);
#pragma unroll
      for (int h = 0; h < kMaxG; ++h)
        if (h < a.G) acc[h] += eq6_block(bv, &qf[h][32 * b], qmeta[h][b], X);
    }
  }
  // S out, and the chunk's softmax statistics per head
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int h = 0; h < kMaxG; ++h) {
    if (h >= a.G) break;  // uniform across the block
    const int hq = g * a.G + h;
    a.S[(int64_t)hq * a.Tpad + t] = valid ? acc[h] : 0.0f;
    const float z = valid ? __fmul_rn(acc[h], a.sm_scale) : -INFINITY;
    float m = warp_max(z);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red[w]);
    __syncthreads();
    float e = valid ? expf(z - m) : 0.0f;
    e = warp_sum(e);
    if (lane == 0) red[warp] = e;
    __syncthreads();
    if (tid == 0) {
      float l = 0.0f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) l += red[w];
      a.stats[(int64_t)c * a.HQ + hq] = make_float2(m, l);
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads) attn_pv_kernel(AttnArgs a) {
  __shared__ __align__(16) int16_t pf[kMaxG][kChunk];
  __shared__ int2 pmeta[kMaxG][kChunk / 32];
  __shared__ float gm[kMaxG], gl[kMaxG];
  __shared__ int last;
  const int c = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  // softmax statistics over every chunk, one warp per head
  for (int h = warp; h < a.G; h += kThreads / 32) {
    const int hq = g * a.G + h;
    float m = -INFINITY;
    for (int j = lane; j < a.C; j += 32) m = fmaxf(m, a.stats[(int64_t)j * a.HQ + hq].x);
    m = warp_max(m);
    float l = 0.0f;
    for (int j = lane; j < a.C; j += 32) {
      const float2 s = a.stats[(int64_t)j * a.HQ + hq];
      l += s.y * expf(s.x - m);
    }
    l = warp_sum(l);
    if (lane == 0) {
      gm[h] = m;
      gl[h] = l;
    }
  }
  __syncthreads();

  // P for this chunk -> MiX-4.5b, one thread per (head, 32-token block)
  const int64_t t0 = (int64_t)c * kChunk;
  const int nblk = (int)min((int64_t)(kChunk / 32), (a.T - t0 + 31) / 32);  // blocks holding a token
  if (tid < a.G * (kChunk / 32)) {
    const int h = tid >> 3, b = tid & 7;
    const int hq = g * a.G + h;
    if (b < nblk) {
      uint32_t u[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int64_t t = t0 + 32 * b + i;
        float p = 0.0f;
        if (t < a.T) p = __fdiv_rn(expf(__fmul_rn(a.S[(int64_t)hq * a.Tpad + t], a.sm_scale) - gm[h]), gl[h]);
        u[i] = __float_as_uint(p);
      }
      uint4 cw;
      uint32_t sh;
      mix_block32<2>(u, a.p_ebias, true, cw, sh);
      mix_unpack(cw, sh, a.p_ebias, &pf[h][32 * b], &pmeta[h][b]);
      if (a.p_codes != nullptr) {
        const int64_t e = (int64_t)hq * a.v_ld + t0 + 32 * b;
        *reinterpret_cast<uint4*>(a.p_codes + e / 2) = cw;
        a.p_shared[e / 32] = (uint16_t)sh;
      }
    }
  }
  __syncthreads();

  // P-V: thread (d, half) owns channel d for half of the heads
  const int d = tid & (kD - 1), half = tid >> 7;
  const int hper = (a.G + 1) / 2, h0 = half * hper, h1 = min(a.G, h0 + hper);
  float acc[(kMaxG + 1) / 2];
#pragma unroll
  for (int j = 0; j < (kMaxG + 1) / 2; ++j) acc[j] = 0.0f;
  const int64_t vrow = (int64_t)g * kD + d;
  for (int b = 0; b < nblk; ++b) {
    const int64_t e = vrow * a.v_ld + t0 + 32 * b;
    const uint4 cw = *reinterpret_cast<const uint4*>(a.v_codes + e / 2);
    const int X = (int)a.v_scales[e / 32] - 127;
    int bv[32];
    int4_values(cw, bv);
#pragma unroll
    for (int j = 0; j < (kMaxG + 1) / 2; ++j) {
      const int h = h0 + j;
      if (h < h1) acc[j] += eq6_block(bv, &pf[h][32 * b], pmeta[h][b], X);
    }
  }
#pragma unroll
  for (int j = 0; j < (kMaxG + 1) / 2; ++j) {
    const int h = h0 + j;
    if (h < h1) a.opart[((int64_t)c * a.HQ + g * a.G + h) * kD + d] = acc[j];
  }

  // the last CTA of this KV head sums the partials in chunk order
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    last = atomicAdd(&a.tickets[g], 1u) == (unsigned)(a.C - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = tid; i < a.G * kD; i += kThreads) {
    const int h = i / kD, dd = i % kD;
    const int hq = g * a.G + h;
    float s = 0.0f;
    for (int j = 0; j < a.C; ++j) s += __ldcg(a.opart + ((int64_t)j * a.HQ + hq) * kD + dd);
    a.out[(int64_t)hq * kD + dd] = s;
  }
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

size_t decode_attention_ws_bytes(const mix_decode_attn_desc_t& d) {
  const int64_t C = (d.tokens + kChunk - 1) / kChunk, Tpad = C * kChunk;
  return align256((size_t)d.q_heads * Tpad * 4) + align256((size_t)C * d.q_heads * 8) +
         align256((size_t)C * d.q_heads * kD * 4) + align256((size_t)d.kv_heads * 4) + 256;
}

cudaError_t launch_decode_attention(const mix_decode_attn_desc_t& d, void* ws, cudaStream_t st) {
  AttnArgs a{};
  const int64_t C = (d.tokens + kChunk - 1) / kChunk;
  a.q = d.q; a.k_new = d.k_new; a.k_mean = d.k_mean; a.bf16 = d.dtype == MIX_DT_BF16;
  a.k_codes = d.k_codes; a.k_scales = d.k_scales; a.v_codes = d.v_codes; a.v_scales = d.v_scales; a.v_ld = d.v_ld;
  a.T = d.tokens; a.Tpad = C * kChunk; a.C = (int)C; a.HQ = d.q_heads; a.HK = d.kv_heads;
  a.G = d.q_heads / d.kv_heads; a.sm_scale = d.sm_scale; a.q_ebias = d.q_ebias; a.p_ebias = d.p_ebias;
  char* p = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~static_cast<uintptr_t>(255));
  a.S = reinterpret_cast<float*>(p);
  p += align256((size_t)d.q_heads * a.Tpad * 4);
  a.stats = reinterpret_cast<float2*>(p);
  p += align256((size_t)C * d.q_heads * 8);
  a.opart = reinterpret_cast<float*>(p);
  p += align256((size_t)C * d.q_heads * kD * 4);
  a.tickets = reinterpret_cast<unsigned*>(p);
  a.out = d.out; a.p_codes = d.p_codes; a.p_shared = static_cast<uint16_t*>(d.p_shared);
  const dim3 grid((unsigned)C, (unsigned)d.kv_heads);
  attn_qk_kernel<<<grid, kThreads, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_pv_kernel<<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mixk
