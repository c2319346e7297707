// Row-wise NVFP4 quantization: the NVFP4 form of the expert GEMMs' operands.
//
// The GB200 deployment keeps its experts in NVFP4 ("MoE inference: the call
// centre with 256 specialists and 8 taking each call", "The maths that
// matters" and "DeepEP, EPLB and Wide-EP"). The format: 4-bit E2M1 elements
// (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) in blocks of 16 consecutive
// elements along the contraction, each block with an unsigned E4M3 scale.
// The pages give no scaling rule; the one used here also gives each row one
// fp32 scale, so that the block scales use E4M3's whole range. For a row
// with max |v| = amax > 0:
//   row scale   s = fp32(amax / 2688)                      (2688 = 6 * 448)
//   block code  b = E4M3(fp32(bmax * fp32(448 / amax)))   (bmax: the block's max |v|)
//   element     q = E2M1(fp32(v * fp32(fp32(2688 / amax) / e4m3(b))))
// both roundings to nearest even and saturating (at 448 and at 6), the sign
// of v kept when q rounds to zero; a block whose scale decodes to 0 has
// codes 0 and a zero row has s = 0 and codes 0. An element stands for
// e2m1(q) * e4m3(b) * s.
//
// Layout: codes packed two a byte, the lower column in the low nibble,
// [rows][cols / 2]; block scales [rows][ld_sf] bytes with zeros past
// cols / 16; row scales [rows] fp32.
//
// One warp per row (one block per row for up to kQBlockRows rows): the
// row's max |v| (or the one the gate/up epilogue recorded for H), then one
// 16-element block per thread and step: 32 bytes of bf16 in, 8 bytes of
// codes and one scale byte out. The E2M1 rounding is the
// conversion instruction's (round to nearest even, saturating, the sign of a
// value that rounds to zero kept), checked bit for bit against the oracle's
// definition of the code. The same kernel gathers
// x_perm rows (row r reads token sorted_pair[r] / k) and clears the H
// maxima of the rows it feeds.
#include "quant_rows.cuh"

namespace moe {
namespace {

using namespace quant;

// E4M3 code of a non-negative fp32 value, rounded to nearest even and
// saturated at 448.
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}
// Value of a non-negative E4M3 code (exponent bias 7; exponent field 0
// holds the subnormals m * 2^-9), exact in fp32.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  if (e == 0) return (float)m * 0.001953125f;
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}
// Eight fp32 values to E2M1 codes packed in 32 bits, value i in bits
// [4i, 4i+4): round to nearest even, saturated at 6 (cvt.rn.satfinite; each
// instruction converts a pair, its first source into the upper nibble).
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                           float v5, float v6, float v7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

// Blocks b0, b0 + step, ... of row r: codes, block scales, and the zero
// padding of the block-scale row.
__device__ __forceinline__ void quantize_blocks(const QuantArgs& a, long long r, const uint4* src,
                                                float amax, int b0, int step) {
  const int nb = a.cols / 16;  // blocks of 16 = two 16-byte vectors
  const float to_block = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
  const float to_code = amax > 0.f ? __fdiv_rn(2688.f, amax) : 0.f;
  if (b0 == 0) a.scale[r] = __fdiv_rn(amax, 2688.f);
  uint2* dst = reinterpret_cast<uint2*>(a.q + r * (a.cols / 2));
  uint8_t* sfrow = a.sf + r * a.ld_sf;
  for (int b = b0; b < nb; b += step) {
    const uint4 q0 = __ldg(src + 2 * b), q1 = __ldg(src + 2 * b + 1);
    float f[16];
    bf16x2_to_f32(q0.x, f[0], f[1]);
    bf16x2_to_f32(q0.y, f[2], f[3]);
    bf16x2_to_f32(q0.z, f[4], f[5]);
    bf16x2_to_f32(q0.w, f[6], f[7]);
    bf16x2_to_f32(q1.x, f[8], f[9]);
    bf16x2_to_f32(q1.y, f[10], f[11]);
    bf16x2_to_f32(q1.z, f[12], f[13]);
    bf16x2_to_f32(q1.w, f[14], f[15]);
    float bmax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(f[i]));
    const uint32_t bc = amax > 0.f ? e4m3_code(__fmul_rn(bmax, to_block)) : 0u;
    const float bv = e4m3_value(bc);
    const float inv = bv > 0.f ? __fdiv_rn(to_code, bv) : 0.f;
    uint32_t w[2] = {0u, 0u};
    if (bv > 0.f) {
#pragma unroll
      for (int i = 0; i < 16; ++i) f[i] = __fmul_rn(f[i], inv);
      w[0] = e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
      w[1] = e2m1x8(f[8], f[9], f[10], f[11], f[12], f[13], f[14], f[15]);
    }
    dst[b] = make_uint2(w[0], w[1]);
    sfrow[b] = (uint8_t)bc;
  }
  for (int b = nb + b0; b < a.ld_sf; b += step) sfrow[b] = 0;
}

// Many rows: one warp a row.
__global__ void __launch_bounds__(kQThreads) quantize_rows_nvf4_kernel(const QuantArgs a) {
  const long long r = (long long)blockIdx.x * kQWarps + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  pdl_wait();
  pdl_trigger();
  const long long sr = source_row(a, r, lane);
  if (sr < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(a.src + sr * a.cols);
  const float amax = a.amax_in ? __uint_as_float(__ldg(a.amax_in + r))
                               : warp_max(partial_amax(src, lane, a.cols / 8, 32));
  quantize_blocks(a, r, src, amax, lane, 32);
}

// Few rows: one block a row.
__global__ void __launch_bounds__(kQThreads) quantize_row_block_nvf4_kernel(const QuantArgs a) {
  const long long r = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const long long sr = source_row(a, r, threadIdx.x);
  if (sr < 0) return;  // the same for the whole block
  const uint4* src = reinterpret_cast<const uint4*>(a.src + sr * a.cols);
  quantize_blocks(a, r, src, block_row_amax(a, r, src), threadIdx.x, kQThreads);
}

}  // namespace

cudaError_t launch_quantize_rows_nvf4(const QuantArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  ProfScope p(K_QUANTIZE, s);
  if (a.rows <= kQBlockRows)
    return launch_pdl(quantize_row_block_nvf4_kernel, dim3((unsigned)a.rows), dim3(kQThreads), 0,
                      s, 1, a);
  return launch_pdl(quantize_rows_nvf4_kernel, dim3((unsigned)((a.rows + kQWarps - 1) / kQWarps)),
                    dim3(kQThreads), 0, s, 1, a);
}

}  // namespace moe
