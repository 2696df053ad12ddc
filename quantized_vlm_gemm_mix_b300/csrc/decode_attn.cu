// Fused MiX decode attention (one query token per head, GQA) over an MX KV
// cache: the accelerator dataflow of the pchao.org digest of "MiX:
// Micro-Inverted-Scaling ..." (Method section, accelerator bullet: K-mean
// subtraction with the frozen prefill mean, Q-K^T on the dual-format
// matmul, the SFU softmax, MiX requantisation of P, P-V on the dual-format
// matmul) as ONE cooperative kernel and no host round trip.
//
// Grid: KV heads x NC token chunks of TB tokens (TB a multiple of 32, chosen
// so that the grid fills the SMs once); 512 threads.  CTA (g, c):
//   A. loads its chunk of the K' cache (MXINT4 rows along head_dim) and of
//      the V planes (MXINT4 blocks along tokens) into shared memory,
//      quantises the group's query heads to MiX-4.5b, appends the new key
//      (K' = fp32(k) - mean, MXINT4) when the chunk holds the last token,
//      forms S = Eq. (6) shift-add for every (head, token) of the chunk and
//      the chunk's softmax statistics (max, sum of exp) per head;
//   -- grid barrier --
//   B. combines the statistics of every chunk of its KV head in chunk order,
//      forms P = exp(s - m) / l for its tokens, requantises P to MiX-4.5b
//      (32-token blocks) and computes the chunk's partial O by Eq. (6)
//      against the V blocks;
//   -- grid barrier --
//   C. each CTA sums, in chunk order, the partial outputs of a slice of the
//      (query head, channel) outputs.
// The barriers are a counter in the workspace, zeroed by the host before the
// launch; every wait is bounded (bit 11 of the device error word on
// timeout, and the CTA writes nothing more).
//
// Every block product is an exact integer (as on the shift-add PE); block
// terms are accumulated in fp32.  The work is tiny (the 8192-token cache of
// four KV heads is 4.3 MB) and latency-bound: one launch with the keys,
// values and scores kept in shared memory replaces two kernels and the
// global round trip of S.  Loops over heads stay rolled: a version that
// unrolled every head of a thread spent most of its time waiting on
// instruction fetch.
#include <cuda_runtime.h>

#include "mix_common.cuh"
#include "mix_internal.h"

namespace mixk {
namespace {

constexpr int kD = 128;          // head_dim
constexpr int kMaxG = 8;         // query heads per KV head
constexpr int kThreadsD = 512;   // threads of the kernel
constexpr int kDecMaxSmem = 200 * 1024;  // shared memory a CTA of the one-kernel path may use

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
  int64_t T;
  int NC, TB, HQ, HK, G;
  float sm_scale;
  int q_ebias, p_ebias;
  float2* stats;       // [HK][NC][G] (chunk max, chunk sum of exp)
  float* opart;        // [HK][NC][G][D]
  unsigned* counter;   // grid barrier
  unsigned* err;       // device error word
  long long limit;     // bounded waits, SM clocks
  float* out;          // [HQ][D]
  uint8_t* p_codes;    // optional [HQ][v_ld / 2]
  uint16_t* p_shared;  // optional [HQ][v_ld / 32]
  float* p_values;     // optional [HQ][v_ld]: the P that was quantised
};

// Shared memory of one CTA for TB tokens (offsets in bytes, 16-aligned).
struct DecPlan {
  int kc, ksc, vsm, vxs, qf, qmeta, zs, pf, pmeta, stat, red, bytes;
};
__host__ __device__ inline DecPlan dec_plan(int TB) {
  DecPlan p;
  const int nb = TB / 32;
  int o = 0;
  p.kc = o;    o += TB * (kD / 2);                    // K' codes of the chunk
  p.ksc = o;   o += TB * 4;                           // their four scale bytes per token
  p.vsm = o;   o += nb * kD * 16;                     // V words [block][channel]
  p.vxs = o;   o += nb * kD * 4;                      // V exponents [block][channel]
  p.qf = o;    o += kMaxG * kD * 2;                   // MiX factors of the query heads
  p.qmeta = o; o += kMaxG * (kD / 32) * 8;
  p.zs = o;    o += kMaxG * TB * 4;                   // scaled scores, then P
  p.pf = o;    o += kMaxG * TB * 2;                   // MiX factors of P
  p.pmeta = o; o += kMaxG * nb * 8;
  p.stat = o;  o += 2 * kMaxG * 4;                    // global max and sum per head
  p.red = o;   o += 4 * kMaxG * kD * 4;               // P-V sums of four block groups
  p.bytes = (o + 15) & ~15;
  return p;
}

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

// Algorithm 1 (MiX-4.5b) on one 32-element block by four consecutive lanes
// of a fully active warp: lane q holds sub-block q (eight fp32 patterns, no
// NaN).  The same steps as mix_block32<2> -- block maximum (by shuffles),
// Emax and this sub-block's mshared, the element step, canonical zeros --
// with a quarter of the serial work per thread.  Returns this lane's code
// word; sh, the block's shared field, is the same in all four lanes.
__device__ __forceinline__ uint32_t mix_block32_quad(const uint32_t* u, int q, int ebias, bool asym, uint32_t& sh) {
  uint32_t ks = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) ks = max(ks, u[i] & 0x7FFFFFFFu);
  uint32_t kb = max(ks, __shfl_xor_sync(0xFFFFFFFFu, ks, 1));
  kb = max(kb, __shfl_xor_sync(0xFFFFFFFFu, kb, 2));
  int f, m3;
  const bool nz = max_exp_mant(kb, &f, &m3);
  const int emax = clampi(f, ebias, ebias + 15);
  uint32_t word = 0x77777777u, mine = 0u;
  if (nz) {
    int fs, ms;
    if (!max_exp_mant(ks, &fs, &ms)) ms = 0;
    const MixBlk bb = mix_blk(emax, 8 + ms, asym);
    word = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) word |= mix_code_nonan(u[i], u[i] & 0x7FFFFFFFu, bb) << (4 * i);
    if (word != 0x77777777u) mine = (uint32_t)ms << (4 + 3 * q);
  }
  uint32_t allz = word == 0x77777777u ? 1u : 0u;
  allz &= __shfl_xor_sync(0xFFFFFFFFu, allz, 1);
  allz &= __shfl_xor_sync(0xFFFFFFFFu, allz, 2);
  uint32_t bits = mine | __shfl_xor_sync(0xFFFFFFFFu, mine, 1);
  bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 2);
  sh = (nz && !allz) ? ((uint32_t)(emax - ebias) | bits) : 0u;
  return word;
}

// This lane's eight factors of a quad-quantised block, and (lane 0 of the
// quad) the block's (Emax, packed mshared).
__device__ __forceinline__ void mix_unpack_quad(uint32_t word, uint32_t sh, int q, int ebias, int16_t* f, int2* meta) {
#pragma unroll
  for (int i = 0; i < 8; ++i) f[8 * q + i] = (int16_t)mix_factor((word >> (4 * i)) & 0xFu);
  if (q == 0) {
    const int mk = (int)(((sh >> 4) & 7u) | (((sh >> 7) & 7u) << 8) | (((sh >> 10) & 7u) << 16) |
                         (((sh >> 13) & 7u) << 24));
    *meta = make_int2((int)(sh & 0xFu) + ebias, mk);
  }
}

// v * 2^e for an integer-valued v (|v| < 2^24, exact in fp32): one exact
// power-of-two multiply in the normal range, ldexpf outside it.
__device__ __forceinline__ float scale_pow2(float v, int e) {
  return (e >= -126 && e <= 127) ? v * __uint_as_float((uint32_t)(e + 127) << 23) : ldexpf(v, e);
}

// Four INT4 nibbles (bits 0..15 of x) -> four sign-extended int8 lanes.
__device__ __forceinline__ uint32_t nib4_to_s8(uint32_t x) {
  x = (x | (x << 8)) & 0x00FF00FFu;
  x = (x | (x << 4)) & 0x0F0F0F0Fu;
  return __vsub4(x ^ 0x08080808u, 0x08080808u);  // (n ^ 8) - 8 per byte
}

// One Eq. (6) block: 32 INT4 weights (two's complement nibbles of cw)
// against 32 MiX factors (int16, read as 16-byte vectors): each 8-way
// sub-tree is four 2-way 16x8-bit dot products, times (8 + m3), then one
// exponent add.
__device__ __forceinline__ float eq6_block(const uint4& cw, const int16_t* f, int2 meta, int X) {
  const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
  int blockv = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int4 fv = *reinterpret_cast<const int4*>(f + 8 * q);
    const int lo = (int)nib4_to_s8(w[q] & 0xFFFFu), hi = (int)nib4_to_s8(w[q] >> 16);
    int s = __dp2a_lo(fv.x, lo, 0);
    s = __dp2a_hi(fv.y, lo, s);
    s = __dp2a_lo(fv.z, hi, s);
    s = __dp2a_hi(fv.w, hi, s);
    blockv += s * (8 + ((meta.y >> (8 * q)) & 0xFF));
  }
  return scale_pow2((float)blockv, meta.x + X - 12);  // 2^(Emax + X - 10 - c_B), c_B = 2 for MXINT4
}

// The same block product with the 32 INT4 weights already widened to int8
// (eight words of four lanes, nib4_to_s8 of each half-word in order), for a
// weight block used by several heads.
__device__ __forceinline__ void int4x32_to_s8(const uint4& cw, uint32_t* s8) {
  const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    s8[2 * q] = nib4_to_s8(w[q] & 0xFFFFu);
    s8[2 * q + 1] = nib4_to_s8(w[q] >> 16);
  }
}
__device__ __forceinline__ float eq6_block_s8(const uint32_t* s8, const int16_t* f, int2 meta, int X) {
  int blockv = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int4 fv = *reinterpret_cast<const int4*>(f + 8 * q);
    const int lo = (int)s8[2 * q], hi = (int)s8[2 * q + 1];
    int sq = __dp2a_lo(fv.x, lo, 0);
    sq = __dp2a_hi(fv.y, lo, sq);
    sq = __dp2a_lo(fv.z, hi, sq);
    sq = __dp2a_hi(fv.w, hi, sq);
    blockv += sq * (8 + ((meta.y >> (8 * q)) & 0xFF));
  }
  return scale_pow2((float)blockv, meta.x + X - 12);
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


// Bounded grid barrier: every CTA of the cooperative grid arrives once; the
// counter reaches `target` (the host zeroed it; gridDim.x per barrier).
__device__ __forceinline__ bool dec_barrier(const AttnArgs& a, unsigned target, int* ok_s) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    atomicAdd(a.counter, 1u);
    const long long s0 = clock64();
    int ok = 1;
    for (;;) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.counter) : "memory");
      if (v >= target) break;
      if (clock64() - s0 > a.limit) {
        atomicOr(a.err, 2048u);
        ok = 0;
        break;
      }
    }
    *ok_s = ok;
  }
  __syncthreads();
  return *ok_s != 0;
}

__global__ void __launch_bounds__(kThreadsD, 1) attn_decode_kernel(AttnArgs a) {
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ int ok_s;
  const int TB = a.TB, G = a.G, NC = a.NC;
  const DecPlan L = dec_plan(TB);
  uint8_t* kc = dsm + L.kc;
  uint32_t* ksc = reinterpret_cast<uint32_t*>(dsm + L.ksc);
  uint4* vsm = reinterpret_cast<uint4*>(dsm + L.vsm);
  int* vxs = reinterpret_cast<int*>(dsm + L.vxs);
  int16_t* qf = reinterpret_cast<int16_t*>(dsm + L.qf);
  int2* qmeta = reinterpret_cast<int2*>(dsm + L.qmeta);
  float* zs = reinterpret_cast<float*>(dsm + L.zs);
  int16_t* pf = reinterpret_cast<int16_t*>(dsm + L.pf);
  int2* pmeta = reinterpret_cast<int2*>(dsm + L.pmeta);
  float* gm = reinterpret_cast<float*>(dsm + L.stat);
  float* gl = gm + kMaxG;
  const int g = (int)blockIdx.x / NC, c = (int)blockIdx.x % NC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool bf16 = a.bf16 != 0;
  const int64_t t0 = (int64_t)c * TB;
  const int nt = (int)min((int64_t)TB, a.T - t0);  // tokens of this chunk (>= 1)
  const int nblk = (nt + 31) / 32;                 // 32-token blocks holding a token
  const int64_t t_new = a.T - 1;
  const bool appends = a.k_new != nullptr && t_new >= t0 && t_new < t0 + TB;
  const int nb = TB / 32;

  // ---- A. the chunk's keys and values into shared memory
  for (int i = tid; i < nt * 5; i += kThreadsD) {
    const int tt = i / 5, part = i % 5;
    if (appends && t0 + tt == t_new) continue;  // made below
    const int64_t row = (t0 + tt) * a.HK + g;
    if (part < 4)
      reinterpret_cast<uint4*>(kc + tt * (kD / 2))[part] = __ldg(reinterpret_cast<const uint4*>(a.k_codes + row * (kD / 2)) + part);
    else
      ksc[tt] = __ldg(reinterpret_cast<const uint32_t*>(a.k_scales + row * (kD / 32)));
  }
  for (int i = tid; i < nblk * kD; i += kThreadsD) {
    const int d = i / nblk, b = i % nblk;  // blocks of one channel are contiguous
    const int64_t e = ((int64_t)g * kD + d) * a.v_ld + t0 + 32 * b;
    vsm[b * kD + d] = __ldg(reinterpret_cast<const uint4*>(a.v_codes + e / 2));
    vxs[b * kD + d] = (int)__ldg(a.v_scales + e / 32) - 127;
  }
  // the group's query heads -> MiX-4.5b factors: four lanes per 32-element
  // block, sixteen per head, whole warps
  const int q_warps = (G + 1) / 2;
  if (warp < q_warps) {
    const int hh = tid >> 4, b = (tid >> 2) & 3, qq = tid & 3;
    uint32_t u[8] = {};
    if (hh < G) {
      const int64_t base = (int64_t)(g * G + hh) * kD + 32 * b + 8 * qq;
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = load_bits(a.q, bf16, base + i);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if ((u[i] & 0x7FFFFFFFu) > 0x7F800000u) u[i] = 0u;  // NaN codes as zero
    }
    uint32_t sh;
    const uint32_t word = mix_block32_quad(u, qq, a.q_ebias, true, sh);
    if (hh < G) mix_unpack_quad(word, sh, qq, a.q_ebias, &qf[hh * kD + 32 * b], &qmeta[hh * 4 + b]);
  } else if (appends && warp == q_warps && lane < 4) {
    // append the new key: K' = fp32(k) - mean, MXINT4 along head_dim
    const int b = lane;
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
    const int tt = (int)(t_new - t0);
    reinterpret_cast<uint4*>(kc + tt * (kD / 2))[b] = w;
    reinterpret_cast<uint8_t*>(ksc + tt)[b] = (uint8_t)sc;
  }
  __syncthreads();

  // S of every (head, token) of the chunk, scaled for the softmax: one
  // thread per (token, group of up to four heads); the token's K' row is
  // widened to int8 once and serves every head of the group
  const int HG = (G + 3) / 4;
  for (int i = tid; i < nt * HG; i += kThreadsD) {
    const int tt = i % nt, hg = i / nt;
    const uint4* kr = reinterpret_cast<const uint4*>(kc + tt * (kD / 2));
    const uint32_t scw = ksc[tt];
    uint32_t s8[4][8];
#pragma unroll
    for (int b = 0; b < 4; ++b) int4x32_to_s8(kr[b], s8[b]);
    const int h1 = min(G, 4 * hg + 4);
#pragma unroll 1
    for (int h = 4 * hg; h < h1; ++h) {
      float s = 0.0f;
#pragma unroll
      for (int b = 0; b < 4; ++b)
        s += eq6_block_s8(s8[b], &qf[h * kD + 32 * b], qmeta[h * 4 + b], (int)((scw >> (8 * b)) & 0xFFu) - 127);
      zs[h * TB + tt] = __fmul_rn(s, a.sm_scale);
    }
  }
  __syncthreads();
  // the chunk's statistics, one warp per head
  if (warp < G) {
    const int h = warp;
    float m = -INFINITY;
    for (int tt = lane; tt < nt; tt += 32) m = fmaxf(m, zs[h * TB + tt]);
    m = warp_max(m);
    float e = 0.0f;
    for (int tt = lane; tt < nt; tt += 32) e += expf(zs[h * TB + tt] - m);
    e = warp_sum(e);
    if (lane == 0) a.stats[((int64_t)g * NC + c) * G + h] = make_float2(m, e);
  }
  if (!dec_barrier(a, gridDim.x, &ok_s)) return;

  // ---- B. the softmax over every chunk of this KV head, P, P-V
  if (warp < G) {
    // NC <= 160 chunks: each lane holds its (up to five) chunk statistics in
    // registers, so the maximum and the sum need one round of loads
    const int h = warp;
    const float2* st = a.stats + (int64_t)g * NC * G + h;
    float2 v[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      const int j = lane + 32 * i;
      v[i] = j < NC ? __ldcg(st + (int64_t)j * G) : make_float2(-INFINITY, 0.0f);
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 5; ++i) m = fmaxf(m, v[i].x);
    m = warp_max(m);
    float l = 0.0f;
#pragma unroll
    for (int i = 0; i < 5; ++i)
      if (lane + 32 * i < NC) l += v[i].y * expf(v[i].x - m);
    l = warp_sum(l);
    if (lane == 0) {
      gm[h] = m;
      gl[h] = __frcp_rn(l);  // P = exp(z - m) * (1 / l)
    }
  }
  __syncthreads();
  for (int i = tid; i < G * nblk * 32; i += kThreadsD) {
    const int h = i / (nblk * 32), j = i % (nblk * 32);
    const int64_t t = t0 + j;
    const float p = j < nt ? __fmul_rn(expf(zs[h * TB + j] - gm[h]), gl[h]) : 0.0f;
    zs[h * TB + j] = p;
    if (a.p_values != nullptr) a.p_values[(int64_t)(g * G + h) * a.v_ld + t] = p;
  }
  __syncthreads();
  // P -> MiX-4.5b: four lanes per (head, 32-token block), whole warps
  for (int w0 = warp * 8; w0 < G * nblk; w0 += (kThreadsD / 32) * 8) {
    const int blk = w0 + (lane >> 2), qq = lane & 3;
    const bool on = blk < G * nblk;
    const int h = on ? blk / nblk : 0, b = on ? blk % nblk : 0;
    uint32_t u[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      u[i] = on ? __float_as_uint(zs[h * TB + 32 * b + 8 * qq + i]) : 0u;
      if ((u[i] & 0x7FFFFFFFu) > 0x7F800000u) u[i] = 0u;  // NaN codes as zero
    }
    uint32_t sh;
    const uint32_t word = mix_block32_quad(u, qq, a.p_ebias, true, sh);
    if (on) {
      mix_unpack_quad(word, sh, qq, a.p_ebias, &pf[h * TB + 32 * b], &pmeta[h * nb + b]);
      if (a.p_codes != nullptr) {
        const int64_t e = (int64_t)(g * G + h) * a.v_ld + t0 + 32 * b;
        reinterpret_cast<uint32_t*>(a.p_codes + e / 2)[qq] = word;
        if (qq == 0) a.p_shared[e / 32] = (uint16_t)sh;
      }
    }
  }
  __syncthreads();
  // the chunk's partial O of (head, channel): one thread per (channel, group
  // of blocks) widens the group's V words to int8 once for every head, two
  // blocks at a time; the four groups' sums are then added in group order
  constexpr int BG = 4;
  float* red = reinterpret_cast<float*>(dsm + L.red);  // [BG][kMaxG][kD]
  const int bpg = (nblk + BG - 1) / BG;
  for (int i = tid; i < BG * kD; i += kThreadsD) {
    const int d = i % kD, bg = i / kD;
    const int b0 = bg * bpg, b1 = min(nblk, b0 + bpg);
    for (int h = 0; h < G; ++h) red[(bg * kMaxG + h) * kD + d] = 0.0f;
    for (int bb = b0; bb < b1; bb += 2) {
      const bool two = bb + 1 < b1;
      uint32_t v8[2][8];
      int4x32_to_s8(vsm[bb * kD + d], v8[0]);
      int4x32_to_s8(two ? vsm[(bb + 1) * kD + d] : make_uint4(0, 0, 0, 0), v8[1]);
      const int x0 = vxs[bb * kD + d], x1 = two ? vxs[(bb + 1) * kD + d] : 0;
#pragma unroll 1
      for (int h = 0; h < G; ++h) {
        float acc = red[(bg * kMaxG + h) * kD + d];
        acc += eq6_block_s8(v8[0], &pf[h * TB + 32 * bb], pmeta[h * nb + bb], x0);
        if (two) acc += eq6_block_s8(v8[1], &pf[h * TB + 32 * (bb + 1)], pmeta[h * nb + bb + 1], x1);
        red[(bg * kMaxG + h) * kD + d] = acc;
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < G * kD; i += kThreadsD) {
    const int h = i / kD, d = i % kD;
    float acc = 0.0f;
#pragma unroll
    for (int bg = 0; bg < BG; ++bg) acc += red[(bg * kMaxG + h) * kD + d];
    a.opart[(((int64_t)g * NC + c) * G + h) * kD + d] = acc;
  }
  if (!dec_barrier(a, 2u * gridDim.x, &ok_s)) return;

  // ---- C. O = the partial outputs summed over the chunks, a slice of the
  // outputs per CTA and one warp per output: lane l adds chunks l, l + 32, ...
  // (up to five, loaded at once) and the warp's butterfly adds the lanes, the
  // same fixed order for every output
  const int64_t total = (int64_t)a.HQ * kD;
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  const int64_t o0 = (int64_t)blockIdx.x * per, o1 = min(total, o0 + per);
  for (int64_t o = o0 + warp; o < o1; o += kThreadsD / 32) {
    const int hq = (int)(o / kD), d = (int)(o % kD);
    const int gg = hq / G, h = hq % G;
    const float* src = a.opart + ((int64_t)gg * NC * G + h) * kD + d;
    const int64_t step = (int64_t)G * kD;
    float v[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      const int j = lane + 32 * i;
      v[i] = j < NC ? __ldcg(src + (int64_t)j * step) : 0.0f;
    }
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < 5; ++i) sum += v[i];
    sum = warp_sum(sum);
    if (lane == 0) a.out[o] = sum;
  }
}


// ------------------------------------------------------ long caches
// When a chunk of the one-kernel grid no longer fits in shared memory (tens
// of thousands of tokens), the step runs as two kernels instead:
//  attn_qk_kernel  grid (64-token chunks, KV heads), one thread per (query
//                  head, token): quantises the query heads, appends the new
//                  key, S by Eq. (6), the chunk's softmax statistics;
//  attn_pv_kernel  grid (256-token chunks, KV heads), one thread per (query
//                  head, channel): combines the statistics, P, MiX-4.5b
//                  requantisation, P-V by Eq. (6) into a partial O; the last
//                  CTA of a KV head (an atomic ticket, no waiting) sums the
//                  partials in chunk order.
constexpr int kChunkA = 64;      // tokens per CTA of the Q-K^T kernel
constexpr int kChunkB = 256;     // tokens per CTA of the P-V kernel (8 blocks of 32)

struct AttnArgs2 {  // the two-kernel path
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
  int CA, CB, HQ, HK, G;
  float sm_scale;
  int q_ebias, p_ebias;
  float* S;        // [HQ][Tpad]
  float2* stats;   // [CA][HQ] (chunk max, chunk sum of exp)
  float* opart;    // [CB][HQ][D]
  unsigned* tickets;  // [HK]
  float* out;      // [HQ][D]
  uint8_t* p_codes;    // optional [HQ][v_ld / 2]
  uint16_t* p_shared;  // optional [HQ][v_ld / 32]
  float* p_values;     // optional [HQ][v_ld]: the P that was quantised
};

__global__ void __launch_bounds__(kChunkA * kMaxG, 2) attn_qk_kernel(AttnArgs2 a) {
  __shared__ __align__(16) int16_t qf[kMaxG][kD];
  __shared__ int2 qmeta[kMaxG][kD / 32];
  __shared__ float red[2 * kMaxG];
  __shared__ float cmax[kMaxG];
  const int c = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
  const bool bf16 = a.bf16 != 0;
  const int h = tid / kChunkA;                        // query head within the group
  const int64_t t = (int64_t)c * kChunkA + (tid & (kChunkA - 1));
  const bool valid = t < a.T;
  const int64_t t_new = a.T - 1;
  const bool appended = a.k_new != nullptr && t == t_new;
  if (c == 0 && tid == 0) a.tickets[g] = 0u;  // for attn_pv_kernel, which runs after this grid

  // this thread's key row, fetched first (the appended row is made below)
  uint4 kw[4] = {};
  uint32_t scw = 0;
  if (valid && !appended) {
    const int64_t row = t * a.HK + g;
#pragma unroll
    for (int b = 0; b < 4; ++b) kw[b] = __ldg(reinterpret_cast<const uint4*>(a.k_codes + row * (kD / 2)) + b);
    scw = __ldg(reinterpret_cast<const uint32_t*>(a.k_scales + row * (kD / 32)));
  }
  // the group's query heads -> MiX-4.5b, decoded into factors: four lanes per
  // 32-element block (sixteen per head), whole warps
  const int q_warps = (a.G + 1) / 2, warp_id = tid >> 5;
  if (warp_id < q_warps) {
    const int hh = tid >> 4, b = (tid >> 2) & 3, qq = tid & 3;
    uint32_t u[8] = {};
    if (hh < a.G) {
      const int64_t base = (int64_t)(g * a.G + hh) * kD + 32 * b + 8 * qq;
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = load_bits(a.q, bf16, base + i);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if ((u[i] & 0x7FFFFFFFu) > 0x7F800000u) u[i] = 0u;  // NaN codes as zero
    }
    uint32_t sh;
    const uint32_t word = mix_block32_quad(u, qq, a.q_ebias, true, sh);
    if (hh < a.G) mix_unpack_quad(word, sh, qq, a.q_ebias, &qf[hh][32 * b], &qmeta[hh][b]);
  } else if (a.k_new != nullptr && t_new / kChunkA == c && warp_id == 2 * a.G - 1 && (tid & 31) < 4) {
    // append the new key: K' = fp32(k) - mean, MXINT4 along head_dim (four
    // lanes of the block's last warp, never one of the query warps)
    const int b = tid & 31;
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
  if (appended) {
    const int64_t row = t * a.HK + g;
#pragma unroll
    for (int b = 0; b < 4; ++b) kw[b] = reinterpret_cast<const uint4*>(a.k_codes + row * (kD / 2))[b];
    scw = *reinterpret_cast<const uint32_t*>(a.k_scales + row * (kD / 32));
  }

  // S of (head h, token t)
  float s = 0.0f;
  if (valid) {
    // a rolled loop: each pass re-runs the same instructions, which matters
    // more here than the loop overhead (the kernel is instruction-fetch bound
    // when every instruction runs once)
#pragma unroll 1
    for (int b = 0; b < 4; ++b) {
      const uint4 kb = b == 0 ? kw[0] : b == 1 ? kw[1] : b == 2 ? kw[2] : kw[3];
      s += eq6_block(kb, &qf[h][32 * b], qmeta[h][b], (int)((scw >> (8 * b)) & 0xFFu) - 127);
    }
  }
  a.S[(int64_t)(g * a.G + h) * a.Tpad + t] = s;
  // the chunk's softmax statistics: head h's 64 tokens are warps 2h and 2h + 1
  const int lane = tid & 31, warp = tid >> 5;
  const float z = valid ? __fmul_rn(s, a.sm_scale) : -INFINITY;
  const float wm = warp_max(z);
  if (lane == 0) red[warp] = wm;
  __syncthreads();
  if (tid < a.G) cmax[tid] = fmaxf(red[2 * tid], red[2 * tid + 1]);
  __syncthreads();
  const float e = warp_sum(valid ? expf(z - cmax[h]) : 0.0f);
  __syncthreads();  // every read of red above is done
  if (lane == 0) red[warp] = e;
  __syncthreads();
  if (tid < a.G)
    a.stats[(int64_t)c * a.HQ + g * a.G + tid] = make_float2(cmax[tid], red[2 * tid] + red[2 * tid + 1]);
}

__global__ void __launch_bounds__(kD * kMaxG) attn_pv_kernel(AttnArgs2 a) {
  __shared__ __align__(16) int16_t pf[kMaxG][kChunkB];
  __shared__ int2 pmeta[kMaxG][kChunkB / 32];
  __shared__ __align__(16) float pv[kMaxG][kChunkB];
  __shared__ __align__(16) uint4 vsm[kChunkB / 32][kD];   // the chunk's V words, [block][channel]
  __shared__ int vxs[kChunkB / 32][kD];
  __shared__ float gm[kMaxG], gl[kMaxG];
  __shared__ int last;
  const int c = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int64_t t0 = (int64_t)c * kChunkB;
  const int nblk = (int)min((int64_t)(kChunkB / 32), (a.T - t0 + 31) / 32);  // blocks holding a token
  const int d = tid & (kD - 1), h = tid / kD;

  // the chunk's V words and scales into shared memory
  for (int i = tid; i < nblk * kD; i += nthr) {
    const int b = i / kD, dd = i % kD;
    const int64_t e = ((int64_t)g * kD + dd) * a.v_ld + t0 + 32 * b;
    vsm[b][dd] = __ldg(reinterpret_cast<const uint4*>(a.v_codes + e / 2));
    vxs[b][dd] = (int)__ldg(a.v_scales + e / 32) - 127;
  }

  // softmax statistics over every chunk, one warp per head
  if (warp < a.G) {
    const int hq = g * a.G + warp;
    float m = -INFINITY;
    for (int j = lane; j < a.CA; j += 32) m = fmaxf(m, a.stats[(int64_t)j * a.HQ + hq].x);
    m = warp_max(m);
    float l = 0.0f;
    for (int j = lane; j < a.CA; j += 32) {
      const float2 st = a.stats[(int64_t)j * a.HQ + hq];
      l += st.y * expf(st.x - m);
    }
    l = warp_sum(l);
    if (lane == 0) {
      gm[warp] = m;
      gl[warp] = l;
    }
  }
  __syncthreads();

  // P for this chunk: every thread forms some, then four lanes per (head,
  // 32-token block) requantise them to MiX-4.5b
  for (int i = tid; i < a.G * kChunkB; i += nthr) {
    const int hh = i / kChunkB, j = i % kChunkB;
    const int64_t t = t0 + j;
    float p = 0.0f;
    if (t < a.T)
      p = __fdiv_rn(expf(__fmul_rn(a.S[(int64_t)(g * a.G + hh) * a.Tpad + t], a.sm_scale) - gm[hh]), gl[hh]);
    pv[hh][j] = p;
    if (a.p_values != nullptr && j < 32 * nblk) a.p_values[(int64_t)(g * a.G + hh) * a.v_ld + t] = p;
  }
  __syncthreads();
  if (warp < a.G) {  // warp hh: its 8 blocks, four lanes per block
    const int hh = warp, b = lane >> 2, qq = lane & 3;
    uint32_t u[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      u[i] = __float_as_uint(pv[hh][32 * b + 8 * qq + i]);
      if ((u[i] & 0x7FFFFFFFu) > 0x7F800000u) u[i] = 0u;  // NaN codes as zero
    }
    uint32_t sh;
    const uint32_t word = mix_block32_quad(u, qq, a.p_ebias, true, sh);
    if (b < nblk) {
      mix_unpack_quad(word, sh, qq, a.p_ebias, &pf[hh][32 * b], &pmeta[hh][b]);
      if (a.p_codes != nullptr) {
        const int64_t e = (int64_t)(g * a.G + hh) * a.v_ld + t0 + 32 * b;
        reinterpret_cast<uint32_t*>(a.p_codes + e / 2)[qq] = word;
        if (qq == 0) a.p_shared[e / 32] = (uint16_t)sh;
      }
    }
  }
  __syncthreads();

  // P-V of (head h, channel d)
  float acc = 0.0f;
#pragma unroll 1
  for (int b = 0; b < nblk; ++b) acc += eq6_block(vsm[b][d], &pf[h][32 * b], pmeta[h][b], vxs[b][d]);
  a.opart[((int64_t)c * a.HQ + g * a.G + h) * kD + d] = acc;

  // the last CTA of this KV head sums the partials in chunk order
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    last = atomicAdd(&a.tickets[g], 1u) == (unsigned)(a.CB - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const float* src = a.opart + (int64_t)(g * a.G + h) * kD + d;
  const int64_t step = (int64_t)a.HQ * kD;
  float sum = 0.0f;
  for (int j0 = 0; j0 < a.CB; j0 += 8) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = j0 + j < a.CB ? __ldcg(src + (j0 + j) * step) : 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) sum += v[j];
  }
  a.out[(int64_t)(g * a.G + h) * kD + d] = sum;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Chunk length: the smallest multiple of 32 that lets KV heads x chunks fit
// the SMs once.
int dec_chunk(int64_t T, int HK) {
  int64_t per = num_sms() / HK;
  if (per < 1) per = 1;
  if (per > 160) per = 160;  // the kernel's per-lane registers hold at most 160 chunks
  int64_t tb = (T + per - 1) / per;
  tb = (tb + 31) / 32 * 32;
  return (int)(tb < 32 ? 32 : tb);
}

size_t one_ws_bytes(const mix_decode_attn_desc_t& d) {
  const int TB = dec_chunk(d.tokens, d.kv_heads);
  const int64_t NC = (d.tokens + TB - 1) / TB, G = d.q_heads / d.kv_heads;
  return align256((size_t)d.kv_heads * NC * G * 8) + align256((size_t)d.kv_heads * NC * G * kD * 4) + 256 + 256;
}

cudaError_t launch_one(const mix_decode_attn_desc_t& d, void* ws, cudaStream_t st) {
  AttnArgs a{};
  const int TB = dec_chunk(d.tokens, d.kv_heads);
  const int64_t NC = (d.tokens + TB - 1) / TB;
  a.q = d.q; a.k_new = d.k_new; a.k_mean = d.k_mean; a.bf16 = d.dtype == MIX_DT_BF16;
  a.k_codes = d.k_codes; a.k_scales = d.k_scales; a.v_codes = d.v_codes; a.v_scales = d.v_scales; a.v_ld = d.v_ld;
  a.T = d.tokens; a.NC = (int)NC; a.TB = TB; a.HQ = d.q_heads; a.HK = d.kv_heads;
  a.G = d.q_heads / d.kv_heads; a.sm_scale = d.sm_scale; a.q_ebias = d.q_ebias; a.p_ebias = d.p_ebias;
  char* p = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~static_cast<uintptr_t>(255));
  a.stats = reinterpret_cast<float2*>(p);
  p += align256((size_t)d.kv_heads * NC * a.G * 8);
  a.opart = reinterpret_cast<float*>(p);
  p += align256((size_t)d.kv_heads * NC * a.G * kD * 4);
  a.counter = reinterpret_cast<unsigned*>(p);
  a.limit = 1LL << 31;
  a.out = d.out; a.p_codes = d.p_codes; a.p_shared = static_cast<uint16_t*>(d.p_shared);
  a.p_values = d.p_values;
  cudaError_t e = cudaMemsetAsync(a.counter, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  e = device_error_word(&a.err);
  if (e != cudaSuccess) return e;
  const DecPlan L = dec_plan(TB);
  static bool attr_set[64] = {false};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecMaxSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(d.kv_heads * NC));
  cfg.blockDim = dim3(kThreadsD);
  cfg.dynamicSmemBytes = (size_t)L.bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // CTAs wait on one another: all resident at once
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel, a);
}

size_t two_ws_bytes(const mix_decode_attn_desc_t& d) {
  const int64_t CB = (d.tokens + kChunkB - 1) / kChunkB, CA = (d.tokens + kChunkA - 1) / kChunkA;
  const int64_t Tpad = CB * kChunkB;
  return align256((size_t)d.q_heads * Tpad * 4) + align256((size_t)CA * d.q_heads * 8) +
         align256((size_t)CB * d.q_heads * kD * 4) + align256((size_t)d.kv_heads * 4) + 256;
}

cudaError_t launch_two(const mix_decode_attn_desc_t& d, void* ws, cudaStream_t st) {
  AttnArgs2 a{};
  const int64_t CB = (d.tokens + kChunkB - 1) / kChunkB, CA = (d.tokens + kChunkA - 1) / kChunkA;
  a.q = d.q; a.k_new = d.k_new; a.k_mean = d.k_mean; a.bf16 = d.dtype == MIX_DT_BF16;
  a.k_codes = d.k_codes; a.k_scales = d.k_scales; a.v_codes = d.v_codes; a.v_scales = d.v_scales; a.v_ld = d.v_ld;
  a.T = d.tokens; a.Tpad = CB * kChunkB; a.CA = (int)CA; a.CB = (int)CB; a.HQ = d.q_heads; a.HK = d.kv_heads;
  a.G = d.q_heads / d.kv_heads; a.sm_scale = d.sm_scale; a.q_ebias = d.q_ebias; a.p_ebias = d.p_ebias;
  char* p = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~static_cast<uintptr_t>(255));
  a.S = reinterpret_cast<float*>(p);
  p += align256((size_t)d.q_heads * a.Tpad * 4);
  a.stats = reinterpret_cast<float2*>(p);
  p += align256((size_t)CA * d.q_heads * 8);
  a.opart = reinterpret_cast<float*>(p);
  p += align256((size_t)CB * d.q_heads * kD * 4);
  a.tickets = reinterpret_cast<unsigned*>(p);
  a.out = d.out; a.p_codes = d.p_codes; a.p_shared = static_cast<uint16_t*>(d.p_shared);
  a.p_values = d.p_values;
  attn_qk_kernel<<<dim3((unsigned)CA, (unsigned)d.kv_heads), kChunkA * a.G, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_pv_kernel<<<dim3((unsigned)CB, (unsigned)d.kv_heads), kD * a.G, 0, st>>>(a);
  return cudaGetLastError();
}

// The one-kernel path when a chunk fits in shared memory.
bool one_kernel_fits(const mix_decode_attn_desc_t& d) {
  return dec_plan(dec_chunk(d.tokens, d.kv_heads)).bytes <= kDecMaxSmem;
}

}  // namespace

size_t decode_attention_ws_bytes(const mix_decode_attn_desc_t& d) {
  return one_kernel_fits(d) ? one_ws_bytes(d) : two_ws_bytes(d);
}

cudaError_t launch_decode_attention(const mix_decode_attn_desc_t& d, void* ws, cudaStream_t st) {
  return one_kernel_fits(d) ? launch_one(d, ws, st) : launch_two(d, ws, st);
}

}  // namespace mixk
