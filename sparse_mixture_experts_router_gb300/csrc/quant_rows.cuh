// Shared pieces of the row quantizers (E4M3 in fp8.cu, NVFP4 in nvfp4.cu).
// Both launch one warp per row, or, for up to kQBlockRows rows (decode
// sizes), one block of kQThreads per row, so that a handful of rows still
// spreads over many SMs.
#pragma once
#include "device_util.cuh"
#include "moe_internal.h"

namespace moe {
namespace quant {

constexpr int kQThreads = 256;
constexpr int kQWarps = kQThreads / 32;
constexpr long long kQBlockRows = 1024;

// Max |v| over this thread's 16-byte vectors v0, v0 + step, ... < nv of a
// bf16 row (the caller reduces over the threads of the row).
__device__ __forceinline__ float partial_amax(const uint4* src, int v0, int nv, int step) {
  float m = 0.f;
  for (int v = v0; v < nv; v += step) {
    const uint4 q = __ldg(src + v);
    float f[8];
    bf16x2_to_f32(q.x, f[0], f[1]);
    bf16x2_to_f32(q.y, f[2], f[3]);
    bf16x2_to_f32(q.z, f[4], f[5]);
    bf16x2_to_f32(q.w, f[6], f[7]);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  }
  return m;
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// Source row of output row r, or -1 when the row is not written (past the
// rows in use, or a gather slot without a pair); thread t < clear_n clears
// one of the row's H maxima first.
__device__ __forceinline__ long long source_row(const QuantArgs& a, long long r, int t) {
  if (r >= a.rows) return -1;
  if (a.rows_dev && r >= (long long)__ldg(a.rows_dev)) return -1;
  if (a.clear && t < a.clear_n) a.clear[a.clear_base + t * a.clear_stride + r] = 0u;
  if (!a.gather) return r;
  const int p = __ldg(a.gather + r);
  if (p < 0 || (long long)(p / a.k) >= a.src_rows) return -1;
  return p / a.k;
}

// The row's max |v|: recorded (amax_in) or reduced over the block's
// threads (one row a block; every thread calls it).
__device__ __forceinline__ float block_row_amax(const QuantArgs& a, long long r, const uint4* src) {
  if (a.amax_in) return __uint_as_float(__ldg(a.amax_in + r));
  __shared__ float wmax[kQWarps];
  const int t = threadIdx.x;
  const float m = warp_max(partial_amax(src, t, a.cols / 8, kQThreads));
  if (t % 32 == 0) wmax[t / 32] = m;
  __syncthreads();
  float amax = wmax[0];
#pragma unroll
  for (int w = 1; w < kQWarps; ++w) amax = fmaxf(amax, wmax[w]);
  return amax;
}

}  // namespace quant
}  // namespace moe
