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
  return (size_t)ksmooth_chunks(tokens, C) * (size_t)C * sizeof(float2);
}

cudaError_t launch_ksmooth(const void* k, bool bf16, int64_t tokens, int heads, int head_dim,
                           int64_t ld, float* mean, int mode, float* k_out, void* ws,
                           cudaStream_t st) {
  const int64_t C = (int64_t)heads * head_dim;
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
