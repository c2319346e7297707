// K7: grouped SwiGLU experts in fp32 on the CUDA cores.
//
// The same computation as the bf16 tensor-core path (every expert's SwiGLU
// FFN over its row segment, "MoE inference: the call centre with 256
// specialists and 8 taking each call", "The bare mechanism"), kept in fp32
// end to end for fp32 layers: tcgen05 has no fp32-operand kind (kind::tf32
// rounds operands to 10 mantissa bits), so fp32 layers are not tensor-core
// work here.
//
// Each block computes a 32-row x 32-column output tile with 8x8 threads of
// 4x4 outputs, staging 32-wide K slices of the input rows through shared
// memory. A row tile may straddle two experts, so each thread reads the
// weights of its own rows' experts (through L1); rows of a tile are mapped
// to their segment by a binary search over the output-row starts.
#include "device_util.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int TM = 32, TN = 32, TK = 32;

struct FfnArgs {
  const float* a_routed;   // x_perm [P][K]
  const float* a_shared;   // x [T][K]
  const int32_t* seg;
  const float* w0;         // gate (stage 1) or down (stage 2): [E][n_out][K]
  const float* w1;         // up (stage 1) or unused
  const int32_t* sorted_pair;
  const float* topk_w;
  float* out;              // [R][n_out]
  int R, K, n_out, n_routed, n_pairs;
  int stage;               // 1: SwiGLU hidden, 2: down projection
  int a_by_out_row;        // input row index = output row (stage 2 reads H)
};

// Segment of an output row: the largest e with out_row0[e] <= row (empty
// segments share their successor's start, so the largest is non-empty).
__device__ __forceinline__ int seg_of_row(const int32_t* seg, int E, int row) {
  const int32_t* out_row0 = seg + 3 + 3 * E;
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (out_row0[mid] <= row) lo = mid;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(64) simt_ffn_kernel(const FfnArgs a) {
  __shared__ float As[TM][TK + 1];
  pdl_wait();
  pdl_trigger();
  const int E = a.seg[0];
  const int32_t* rows_of = a.seg + 3 + E;
  const int32_t* a_row0 = a.seg + 3 + 2 * E;
  const int32_t* out_row0 = a.seg + 3 + 3 * E;
  const int tx = threadIdx.x % 8, ty = threadIdx.x / 8;
  const int row0 = blockIdx.y * TM, col0 = blockIdx.x * TN;

  // Per-thread rows and their experts.
  int rseg[4];
  const float* arow[4];
  bool rvalid[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = row0 + ty * 4 + i;
    rvalid[i] = row < a.R;
    int s = 0;
    const float* src = a.a_routed;
    if (rvalid[i]) {
      s = seg_of_row(a.seg, E, row);
      const int local = row - out_row0[s];
      rvalid[i] = local < rows_of[s];
      if (a.a_by_out_row)
        src = a.a_routed + (size_t)row * a.K;
      else
        src = (s < a.n_routed ? a.a_routed : a.a_shared) + (size_t)(a_row0[s] + local) * a.K;
    }
    rseg[i] = s;
    arow[i] = src;
  }
  float acc0[4][4], acc1[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc0[i][j] = acc1[i][j] = 0.f;

  for (int k0 = 0; k0 < a.K; k0 += TK) {
    // Stage the input rows of the tile (each thread its 4 rows, 4 columns a pass).
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kk = tx * 4 + q;
        As[ty * 4 + i][kk] = (rvalid[i] && k0 + kk < a.K) ? arow[i][k0 + kk] : 0.f;
      }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < TK; ++kk) {
      if (k0 + kk >= a.K) break;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (!rvalid[i]) continue;
        const float av = As[ty * 4 + i][kk];
        const size_t wbase = (size_t)rseg[i] * a.n_out;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = col0 + tx * 4 + j;
          if (col >= a.n_out) continue;
          const size_t wi = (wbase + col) * a.K + k0 + kk;
          acc0[i][j] = fmaf(av, a.w0[wi], acc0[i][j]);
          if (a.stage == 1) acc1[i][j] = fmaf(av, a.w1[wi], acc1[i][j]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (!rvalid[i]) continue;
    const int row = row0 + ty * 4 + i;
    float scale = 1.f;
    if (a.stage == 2 && a.topk_w && rseg[i] < a.n_routed) {
      const int pair = a.sorted_pair[row];
      scale = (pair >= 0 && pair < a.n_pairs) ? a.topk_w[pair] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = col0 + tx * 4 + j;
      if (col >= a.n_out) continue;
      float v;
      if (a.stage == 1) {
        const float g = acc0[i][j];
        v = (g / (1.0f + expf(-g))) * acc1[i][j];
      } else {
        v = scale * acc0[i][j];
      }
      a.out[(size_t)row * a.n_out + col] = v;
    }
  }
}

}  // namespace

cudaError_t launch_grouped_f32(const moe_config& c, const void* x_perm, const void* x,
                               const int32_t* seg, const int32_t* sorted_pair,
                               const float* topk_w, const void* w_gate, const void* w_up,
                               const void* w_down, void* h, void* y_perm, int* status,
                               cudaStream_t s) {
  (void)status;
  const long long P = (long long)c.T * c.top_k;
  const long long R = P + (long long)c.n_shared * c.T;
  if (R == 0) return cudaSuccess;
  FfnArgs a;
  a.a_routed = static_cast<const float*>(x_perm);
  a.a_shared = static_cast<const float*>(x);
  a.seg = seg;
  a.w0 = static_cast<const float*>(w_gate);
  a.w1 = static_cast<const float*>(w_up);
  a.sorted_pair = sorted_pair;
  a.topk_w = nullptr;
  a.out = static_cast<float*>(h);
  a.R = (int)R;
  a.K = c.d_model;
  a.n_out = c.d_ff;
  a.n_routed = c.n_experts;
  a.n_pairs = (int)P;
  a.stage = 1;
  a.a_by_out_row = 0;
  {
    dim3 grid(ceil_div(c.d_ff, TN), ceil_div(R, TM));
    ProfScope p(K_GATE_UP, s);
    cudaError_t e = launch_pdl(simt_ffn_kernel, grid, dim3(64), 0, s, 1, a);
    if (e != cudaSuccess) return e;
  }
  // Stage 2 reads H rows in output order: input row == output row.
  FfnArgs b = a;
  b.a_routed = static_cast<const float*>(h);
  b.a_shared = static_cast<const float*>(h);
  b.w0 = static_cast<const float*>(w_down);
  b.w1 = nullptr;
  b.topk_w = topk_w;
  b.out = static_cast<float*>(y_perm);
  b.K = c.d_ff;
  b.n_out = c.d_model;
  b.stage = 2;
  b.a_by_out_row = 1;
  {
    dim3 grid(ceil_div(c.d_model, TN), ceil_div(R, TM));
    ProfScope p(K_DOWN, s);
    return launch_pdl(simt_ffn_kernel, grid, dim3(64), 0, s, 1, b);
  }
}

}  // namespace moe
