// Row-wise E4M3 quantization: the FP8 form of the expert GEMMs' operands.
//
// Deployed experts are stored and tokens dispatched in FP8 ("MoE inference:
// the call centre with 256 specialists and 8 taking each call", "The maths
// that matters" and "DeepEP, EPLB and Wide-EP"). The pages give no scaling
// rule; the one used here gives every row (a token's activations, an output
// channel of a weight matrix, or a row of H) one fp32 scale
// s = fp32(amax / 448) and codes q = E4M3(fp32(v * fp32(448 / amax))),
// rounded to nearest even and saturated at +-448 (cvt.rn.satfinite); a row
// of zeros gets s = 0 and codes 0. A code's value is decode(q) * s.
//
// One warp per row (one block per row for up to kQBlockRows rows): the
// row's max |v| (or the one the gate/up epilogue recorded for H), then 8
// values per thread and step, 16 bytes of bf16 in and 8 bytes of codes out. The same kernel gathers x_perm rows (row r reads
// token sorted_pair[r] / k) and clears the H maxima of the rows it feeds.
#include "quant_rows.cuh"

namespace moe {
namespace {

using namespace quant;

// Two fp32 values to E4M3 codes: `lo` in the low byte, `hi` in the high one
// (the instruction puts its first source in the upper half).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Vectors v0, v0 + step, ... of row r (8 values each): codes, and the row
// scale from the thread that has v0 = 0.
__device__ __forceinline__ void quantize_vecs(const QuantArgs& a, long long r, const uint4* src,
                                              float amax, int v0, int step) {
  const int nvec = a.cols / 8;
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
  if (v0 == 0) a.scale[r] = __fdiv_rn(amax, 448.f);
  uint2* dst = reinterpret_cast<uint2*>(a.q + r * a.cols);
  for (int v = v0; v < nvec; v += step) {
    if (amax == 0.f) {
      dst[v] = make_uint2(0u, 0u);
      continue;
    }
    const uint4 q = __ldg(src + v);
    float f[8];
    bf16x2_to_f32(q.x, f[0], f[1]);
    bf16x2_to_f32(q.y, f[2], f[3]);
    bf16x2_to_f32(q.z, f[4], f[5]);
    bf16x2_to_f32(q.w, f[6], f[7]);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = e4m3x2(__fmul_rn(f[2 * i], inv), __fmul_rn(f[2 * i + 1], inv));
    dst[v] = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
  }
}

// Many rows: one warp a row.
__global__ void __launch_bounds__(kQThreads) quantize_rows_kernel(const QuantArgs a) {
  const long long r = (long long)blockIdx.x * kQWarps + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  pdl_wait();
  pdl_trigger();
  const long long sr = source_row(a, r, lane);
  if (sr < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(a.src + sr * a.cols);
  const float amax = a.amax_in ? __uint_as_float(__ldg(a.amax_in + r))
                               : warp_max(partial_amax(src, lane, a.cols / 8, 32));
  quantize_vecs(a, r, src, amax, lane, 32);
}

// Few rows: one block a row.
__global__ void __launch_bounds__(kQThreads) quantize_row_block_kernel(const QuantArgs a) {
  const long long r = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const long long sr = source_row(a, r, threadIdx.x);
  if (sr < 0) return;  // the same for the whole block
  const uint4* src = reinterpret_cast<const uint4*>(a.src + sr * a.cols);
  quantize_vecs(a, r, src, block_row_amax(a, r, src), threadIdx.x, kQThreads);
}

}  // namespace

cudaError_t launch_quantize_rows(const QuantArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  ProfScope p(K_QUANTIZE, s);
  if (a.rows <= kQBlockRows)
    return launch_pdl(quantize_row_block_kernel, dim3((unsigned)a.rows), dim3(kQThreads), 0, s, 1,
                      a);
  return launch_pdl(quantize_rows_kernel, dim3((unsigned)((a.rows + kQWarps - 1) / kQWarps)),
                    dim3(kQThreads), 0, s, 1, a);
}

}  // namespace moe
