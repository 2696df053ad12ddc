// K-smoothing (SageAttention's gamma(K) = K - mean(K); Method section,
// accelerator bullet, and Caveats section of the pchao.org digest of "MiX:
// Micro-Inverted-Scaling ...": the mean is taken once over the prefill tokens
// and frozen for decode, so the Key cache is never re-read to update it).
//
// COMPUTE: the tokens are split into chunks across CTAs (the whole tensor has
// to be in flight to reach HBM bandwidth); each CTA sums its chunk per
// channel and writes one partial row to the caller's workspace.  Every sum is
// a double-float (an fp32 pair (hi, lo) kept exact by Knuth's two-sum, about
// 48 bits of precision) because fp64 arithmetic is slow on this part: a
// thread's own run of tokens, the cross-warp sum and the cross-chunk sum.  A
// second kernel adds the partial rows in a fixed order and divides by the
// token count (the one fp64 operation per channel), so the result does not
// depend on scheduling.  APPLY (both modes): k_out = fp32(k) - mean, one fp32
// subtraction per element.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>

#include "mix_internal.h"

namespace mixk {
namespace {

constexpr int kThreads = 256;  // 8 warps x 32 lanes x 8 channels = 256 channels

__device__ __forceinline__ void load8f(const void* base, bool bf16, int64_t elem, float* v) {
  if (bf16) {
    const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem);
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(a[i] << 16);
      v[2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
    const float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// Knuth's two-sum: a + b = s + e exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bv = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bv)), __fsub_rn(b, bv));
}

// (h, l) += (bh, bl) in double-float, renormalised with a second two-sum.
__device__ __forceinline__ void df_add(float& h, float& l, float bh, float bl) {
  float s, e;
  two_sum(h, bh, s, e);
  two_sum(s, __fadd_rn(e, __fadd_rn(l, bl)), h, l);
}

constexpr int kBatch = 8;  // tokens whose loads a thread has in flight at once

// grid (channel tiles of 256, chunks).  Warp w sums tokens t0 + w, t0 + w + 8,
// ... of the chunk, kBatch of them per round of loads; lane l owns channels
// c0 + 8l .. c0 + 8l + 7.  partial[chunk][c] = (hi, lo).
__global__ void __launch_bounds__(kThreads) ksmooth_partial_kernel(
    const void* __restrict__ k, int bf16, int64_t tokens, int64_t C, int64_t ld, int64_t chunk,
    float2* __restrict__ partial) {
  __shared__ float2 red[8][256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 256 + lane * 8;
  const int64_t t0 = (int64_t)blockIdx.y * chunk;
  const int64_t t1 = min(tokens, t0 + chunk);
  float hi[8] = {0, 0, 0, 0, 0, 0, 0, 0}, lo[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (c < C) {
    for (int64_t tb = t0 + warp; tb < t1; tb += 8 * kBatch) {
      float v[kBatch][8];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int64_t t = tb + 8 * b;
        if (t < t1) {
          load8f(k, bf16 != 0, t * ld + c, v[b]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) v[b][i] = 0.0f;  // adding +0 leaves the pair unchanged
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float s, e;
          two_sum(hi[i], v[b][i], s, e);
          hi[i] = s;
          lo[i] = __fadd_rn(lo[i], e);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[warp][lane * 8 + i] = make_float2(hi[i], lo[i]);
  __syncthreads();
  const int64_t cc = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (cc < C) {
    float h = 0.0f, l = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) df_add(h, l, red[w][threadIdx.x].x, red[w][threadIdx.x].y);
    partial[(int64_t)blockIdx.y * C + cc] = make_float2(h, l);
  }
}

// grid ceil(C / 32), 256 threads: lane x owns channel c0 + x and row y
// (threadIdx.x / 32) adds chunks y, y + 8, ... (all of its loads in flight);
// the eight rows are then added in order 0..7.  The one fp64 step is the
// division of the pair's sum by the token count.
__global__ void __launch_bounds__(256) ksmooth_finalize_kernel(const float2* __restrict__ partial,
                                                               int64_t nchunks, int64_t C, int64_t tokens,
                                                               float* __restrict__ mean) {
  __shared__ float2 red[8][32];
  const int x = threadIdx.x & 31, y = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 32 + x;
  float h = 0.0f, l = 0.0f;
  if (c < C) {
    int64_t j = y;
    for (; j + 24 < nchunks; j += 32) {
      float2 p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = __ldg(partial + (j + 8 * i) * C + c);
#pragma unroll
      for (int i = 0; i < 4; ++i) df_add(h, l, p[i].x, p[i].y);
    }
    for (; j < nchunks; j += 8) {
      const float2 p = __ldg(partial + j * C + c);
      df_add(h, l, p.x, p.y);
    }
  }
  red[y][x] = make_float2(h, l);
  __syncthreads();
  if (y == 0 && c < C) {
#pragma unroll
    for (int w = 1; w < 8; ++w) df_add(h, l, red[w][x].x, red[w][x].y);
    mean[c] = (float)(((double)h + (double)l) / (double)tokens);
  }
}

__global__ void __launch_bounds__(kThreads) ksmooth_apply_kernel(
    const void* __restrict__ k, int bf16, int64_t tokens, int64_t C, int64_t ld,
    const float* __restrict__ mean, float* __restrict__ out) {
  const int64_t groups = C / 8;
  const int64_t total = tokens * groups;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = g / groups, c = (g - t * groups) * 8;
    float v[8];
    load8f(k, bf16 != 0, t * ld + c, v);
    const float4 m0 = *reinterpret_cast<const float4*>(mean + c);
    const float4 m1 = *reinterpret_cast<const float4*>(mean + c + 4);
    float4* o = reinterpret_cast<float4*>(out + t * C + c);
    o[0] = make_float4(__fsub_rn(v[0], m0.x), __fsub_rn(v[1], m0.y), __fsub_rn(v[2], m0.z), __fsub_rn(v[3], m0.w));
    o[1] = make_float4(__fsub_rn(v[4], m1.x), __fsub_rn(v[5], m1.y), __fsub_rn(v[6], m1.z), __fsub_rn(v[7], m1.w));
  }
}

// ---------------------------------------------------------------- one pass
// COMPUTE with the keys held in shared memory: one cooperative launch of G
// CTAs (all resident at once), each owning a run of `chunk` tokens.
//   1. load the run once (kept in shared memory as it was read) and sum it
//      per channel (double-float, the partial kernel's order), one partial
//      row per CTA to the workspace;
//   2. a grid barrier (a counter the host zeroes before the launch; bounded
//      wait -- on timeout bit 10 of the device error word is set and the CTA
//      writes nothing more);
//   3. each CTA adds the G partial rows of its share of the channels in a
//      fixed order and writes their mean; after a second barrier every CTA
//      reads the whole mean;
//   4. k_out = fp32(k) - mean from shared memory.
// Used when a CTA's run fits in shared memory (the prefill keys of one layer
// are a few MB); longer inputs take the three-kernel path above.
constexpr int kFusedRunBytes = 32 << 10;    // target bytes of keys per CTA
constexpr int kFusedMaxBytes = 176 << 10;   // shared memory a CTA may use for them

struct FusedPlan {
  int G, chunk;
  size_t smem;
  bool ok;
};

// All CTAs of the (cooperative, hence co-resident) grid arrive; returns once
// the counter reaches `target` (zeroed by the host before the launch, G
// arrivals per barrier).  Bounded: on timeout bit 10 of the device error word
// is set and every thread of the CTA gets false.
__device__ __forceinline__ bool grid_barrier(unsigned* counter, unsigned target, long long limit, unsigned* err,
                                             int* ok_s) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    atomicAdd(counter, 1u);
    const long long s0 = clock64();
    int ok = 1;
    for (;;) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
      if (v >= target) break;
      if (clock64() - s0 > limit) {
        atomicOr(err, 1024u);
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    *ok_s = ok;
  }
  __syncthreads();
  return *ok_s != 0;
}

__global__ void __launch_bounds__(kThreads, 1) ksmooth_fused_kernel(
    const void* __restrict__ k, int bf16, int64_t tokens, int64_t C, int64_t ld, int chunk,
    float2* __restrict__ partial, unsigned* __restrict__ counter, float* __restrict__ mean,
    float* __restrict__ out, long long limit, unsigned* __restrict__ err) {
  extern __shared__ __align__(16) unsigned char fsm[];
  __shared__ float2 red[8][256];
  __shared__ int ok_s;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int esz = bf16 ? 2 : 4;
  const int64_t t0 = (int64_t)blockIdx.x * chunk;
  const int n = (int)min((int64_t)chunk, tokens - t0);  // tokens of this run (>= 1)
  unsigned char* kr = fsm;                              // [n][C] raw keys
  float* msm = reinterpret_cast<float*>(fsm + (((size_t)chunk * C * esz + 15) & ~(size_t)15));  // [C] mean
  // 1. load and sum, 256 channels at a time: lane l owns channels c + 8 l ..
  //    c + 8 l + 7, warp w tokens w, w + 8, ...
  for (int64_t c0 = 0; c0 < C; c0 += 256) {
    const int64_t c = c0 + lane * 8;
    float hi[8] = {0, 0, 0, 0, 0, 0, 0, 0}, lo[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (c < C) {
      for (int tb = warp; tb < n; tb += 8 * kBatch) {
        // every load of the batch in flight first, then keep and add them
        uint4 raw[kBatch][2];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int t = tb + 8 * b;
          raw[b][0] = raw[b][1] = make_uint4(0, 0, 0, 0);
          if (t < n) {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(k) +
                                                              ((t0 + t) * ld + c) * esz);
            raw[b][0] = __ldg(src);
            if (!bf16) raw[b][1] = __ldg(src + 1);
          }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int t = tb + 8 * b;
          if (t < n) {
            uint4* dst = reinterpret_cast<uint4*>(kr + ((size_t)t * C + c) * esz);
            dst[0] = raw[b][0];
            if (!bf16) dst[1] = raw[b][1];
          }
          float v[8];  // +0 for a missing token leaves the pair unchanged
          if (bf16) {
            const uint32_t a[4] = {raw[b][0].x, raw[b][0].y, raw[b][0].z, raw[b][0].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[2 * i] = __uint_as_float(a[i] << 16);
              v[2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
            }
          } else {
            const uint32_t a[8] = {raw[b][0].x, raw[b][0].y, raw[b][0].z, raw[b][0].w,
                                   raw[b][1].x, raw[b][1].y, raw[b][1].z, raw[b][1].w};
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(a[i]);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float s, e;
            two_sum(hi[i], v[i], s, e);
            hi[i] = s;
            lo[i] = __fadd_rn(lo[i], e);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) red[warp][lane * 8 + i] = make_float2(hi[i], lo[i]);
    __syncthreads();
    const int64_t cc = c0 + threadIdx.x;
    if (cc < C) {
      float h = 0.0f, l = 0.0f;
#pragma unroll
      for (int w = 0; w < 8; ++w) df_add(h, l, red[w][threadIdx.x].x, red[w][threadIdx.x].y);
      partial[(int64_t)blockIdx.x * C + cc] = make_float2(h, l);
    }
    __syncthreads();
  }
  // 2. grid barrier
  if (!grid_barrier(counter, gridDim.x, limit, err, &ok_s)) return;
  // 3. the mean: CTA b adds the G partial rows of its channels (warp w takes
  //    rows w, w + 8, ..., then the eight warp sums are added in order -- the
  //    same order for every channel), writes them to `mean`, and after a
  //    second barrier every CTA reads all of them
  const int G = (int)gridDim.x;
  const int64_t cpc = (C + G - 1) / G, cb = (int64_t)blockIdx.x * cpc, ce = min(C, cb + cpc);
  for (int64_t c0 = cb; c0 < ce; c0 += 32) {
    const int64_t c = c0 + lane;
    float h = 0.0f, l = 0.0f;
    if (c < ce) {
      int j = warp;
      for (; j + 56 < G; j += 64) {
        float2 p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) p[i] = __ldcg(partial + (int64_t)(j + 8 * i) * C + c);
#pragma unroll
        for (int i = 0; i < 8; ++i) df_add(h, l, p[i].x, p[i].y);
      }
      for (; j < G; j += 8) {
        const float2 p = __ldcg(partial + (int64_t)j * C + c);
        df_add(h, l, p.x, p.y);
      }
    }
    red[warp][lane] = make_float2(h, l);
    __syncthreads();
    if (warp == 0 && c < ce) {
      float hh = 0.0f, ll = 0.0f;
#pragma unroll
      for (int w = 0; w < 8; ++w) df_add(hh, ll, red[w][lane].x, red[w][lane].y);
      mean[c] = (float)(((double)hh + (double)ll) / (double)tokens);
    }
    __syncthreads();
  }
  __threadfence();
  if (!grid_barrier(counter, 2u * gridDim.x, limit, err, &ok_s)) return;
  for (int64_t c = threadIdx.x; c < C; c += blockDim.x) msm[c] = __ldcg(mean + c);
  __syncthreads();
  // 4. apply from shared memory
  if (out == nullptr) return;
  const int64_t groups = C / 8, total = (int64_t)n * groups;
  for (int64_t g = threadIdx.x; g < total; g += blockDim.x) {
    const int64_t t = g / groups, c = (g - t * groups) * 8;
    float v[8];
    load8f(kr, bf16 != 0, t * C + c, v);
    float4* o = reinterpret_cast<float4*>(out + (t0 + t) * C + c);
    o[0] = make_float4(__fsub_rn(v[0], msm[c]), __fsub_rn(v[1], msm[c + 1]), __fsub_rn(v[2], msm[c + 2]),
                       __fsub_rn(v[3], msm[c + 3]));
    o[1] = make_float4(__fsub_rn(v[4], msm[c + 4]), __fsub_rn(v[5], msm[c + 5]), __fsub_rn(v[6], msm[c + 6]),
                       __fsub_rn(v[7], msm[c + 7]));
  }
}

FusedPlan fused_plan(int64_t tokens, int64_t C, bool bf16) {
  FusedPlan f{};
  f.ok = false;
  if (tokens <= 0 || C <= 0 || C % 8 != 0) return f;
  const int64_t esz = bf16 ? 2 : 4, total = tokens * C * esz;
  int64_t G = (total + kFusedRunBytes - 1) / kFusedRunBytes;
  if (G > num_sms()) G = num_sms();
  if (G < 1) G = 1;
  int64_t chunk = (tokens + G - 1) / G;
  G = (tokens + chunk - 1) / chunk;  // every CTA owns at least one token
  const size_t smem = (((size_t)chunk * C * esz + 15) & ~(size_t)15) + (size_t)C * 4;
  if (smem > (size_t)kFusedMaxBytes + 16 * 1024) return f;
  if ((size_t)chunk * C * esz > (size_t)kFusedMaxBytes) return f;
  f.G = (int)G;
  f.chunk = (int)chunk;
  f.smem = smem;
  f.ok = true;
  return f;
}

size_t fused_ws_bytes(const FusedPlan& f, int64_t C) { return (size_t)f.G * C * sizeof(float2) + 256; }

int64_t ksmooth_chunks(int64_t tokens, int64_t C) {
  const int64_t tiles = (C + 255) / 256;
  int64_t want = (4 * (int64_t)num_sms() + tiles - 1) / tiles;  // about four CTAs per SM
  const int64_t by_len = (tokens + 15) / 16;                    // at least 16 tokens per chunk
  if (want > by_len) want = by_len;
  if (want > 128) want = 128;  // the finalize adds at most 16 rows per thread, four loads in flight
  return want > 0 ? want : 1;
}

}  // namespace

size_t ksmooth_ws_bytes(int64_t tokens, int heads, int head_dim) {
  const int64_t C = (int64_t)heads * head_dim;
  if (tokens <= 0 || C <= 0) return 0;
  const size_t three = (size_t)ksmooth_chunks(tokens, C) * (size_t)C * sizeof(float2);
  // either dtype may come with these sizes: cover the one-pass plan of both
  size_t one = 0;
  for (int b = 0; b < 2; ++b) {
    const FusedPlan f = fused_plan(tokens, C, b != 0);
    if (f.ok && fused_ws_bytes(f, C) > one) one = fused_ws_bytes(f, C);
  }
  return three > one ? three : one;
}

cudaError_t launch_ksmooth(const void* k, bool bf16, int64_t tokens, int heads, int head_dim,
                           int64_t ld, float* mean, int mode, float* k_out, void* ws,
                           cudaStream_t st) {
  const int64_t C = (int64_t)heads * head_dim;
  const FusedPlan fp = fused_plan(tokens, C, bf16);
  if (mode == KSMOOTH_COMPUTE && fp.ok && (ld % 8) == 0) {
    // one cooperative launch; the barrier counter sits after the partial rows
    float2* part = static_cast<float2*>(ws);
    unsigned* counter = reinterpret_cast<unsigned*>(part + (size_t)fp.G * C);
    cudaError_t e = cudaMemsetAsync(counter, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    unsigned* err = nullptr;
    e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    // the kernel's static arrays (16 KB) count against the default 48 KB too;
    // the limit is raised once per device, to the most any plan asks for
    static bool attr_set[64] = {false};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
      e = cudaFuncSetAttribute(ksmooth_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kFusedMaxBytes + 16 * 1024);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)fp.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = fp.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int bf = bf16 ? 1 : 0;
    const long long limit = 1LL << 31;
    e = cudaLaunchKernelEx(&cfg, ksmooth_fused_kernel, k, bf, tokens, C, ld, fp.chunk, part, counter, mean, k_out,
                           limit, err);
    if (e != cudaSuccess && std::getenv("MIX_DEBUG") != nullptr)
      std::fprintf(stderr, "ksmooth one-pass launch (G %d, chunk %d, smem %zu): %s\n", fp.G, fp.chunk, fp.smem,
                   cudaGetErrorString(e));
    return e;
  }
  if (mode == KSMOOTH_COMPUTE) {
    const int64_t nch = ksmooth_chunks(tokens, C);
    const int64_t chunk = (tokens + nch - 1) / nch;
    const int64_t used = (tokens + chunk - 1) / chunk;
    const dim3 grid((unsigned)((C + 255) / 256), (unsigned)used);
    ksmooth_partial_kernel<<<grid, kThreads, 0, st>>>(k, bf16 ? 1 : 0, tokens, C, ld, chunk,
                                                      static_cast<float2*>(ws));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ksmooth_finalize_kernel<<<(unsigned)((C + 31) / 32), 256, 0, st>>>(static_cast<const float2*>(ws), used,
                                                                       C, tokens, mean);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (k_out != nullptr && tokens > 0) {
    const int64_t total = tokens * (C / 8);
    int64_t g = (total + kThreads - 1) / kThreads;
    if (g > (int64_t)num_sms() * 8) g = (int64_t)num_sms() * 8;
    ksmooth_apply_kernel<<<(unsigned)g, kThreads, 0, st>>>(k, bf16 ? 1 : 0, tokens, C, ld, mean, k_out);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace mixk

// ---------------------------------------------------------------------------
// No-allocation variant.  Some callers cannot hand the library device memory:
// hosts whose device memory is all owned by their own allocator, and loops
// that must never call cudaMalloc (it can synchronise the whole device).  For them the partial sums of COMPUTE live
// in a fixed array compiled into the library instead of a caller workspace.
// Every GPU that loads the library keeps this array until the process exits.
// ---------------------------------------------------------------------------
#include <cuda.h>

#include <mutex>

namespace mixk {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)2 << 20;  // 2 MiB
static __device__ __align__(256) float2 g_ksmooth_scratch[kNoAllocScratchBytes / sizeof(float2)];

std::mutex g_scratch_mu;
struct ScratchEntry {
  unsigned long long ctx_id;  // the context the address belongs to
  void* addr;
};
ScratchEntry g_scratch_addr[64] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (0 if it cannot be
// read).  A context created after cudaDeviceReset gets a new id.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(a);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
        qb == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(b);
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur == nullptr || get_id == nullptr || get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_ksmooth_scratch on the current device (in host code
// the symbol is only a host-side stand-in).  Looked up once per device and
// context: an address cached under a context that has since been destroyed
// (cudaDeviceReset) is never handed out; with no readable context id the
// address is looked up on every call.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const unsigned long long id = current_context_id();  // 0 before the context exists
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& ent = g_scratch_addr[dev];
  if (ent.addr == nullptr || ent.ctx_id != id || id == 0) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ksmooth_scratch);  // creates the primary context if needed
    if (e != cudaSuccess) return e;
    ent.addr = p;
    ent.ctx_id = current_context_id();
  }
  *out = ent.addr;
  return cudaSuccess;
}

}  // namespace

size_t ksmooth_noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

cudaError_t launch_ksmooth_noalloc(const void* k, bool bf16, int64_t tokens, int heads, int head_dim,
                                   int64_t ld, float* mean, int mode, float* k_out, cudaStream_t st) {
  void* ws = nullptr;
  if (mode == KSMOOTH_COMPUTE) {
    cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) return e;
  }
  return launch_ksmooth(k, bf16, tokens, heads, head_dim, ld, mean, mode, k_out, ws, st);
}

}  // namespace mixk
