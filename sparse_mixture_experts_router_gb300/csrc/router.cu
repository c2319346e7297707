// K1: router scores, top-k selection, gate weights and balance statistics.
//
// Follows "Mixture of experts and speculative decoding", steps 1-3 of
// "Following one token through an MoE layer" (score every expert with one
// linear layer, keep the k best, softmax over the kept scores) and section
// "Keeping the experts busy" (f_i and P_i of the balance loss); and "MoE
// inference: the call centre with 256 specialists and 8 taking each call",
// "The bare mechanism" (affinity softmax over all experts, renormalised
// top-k weights, a routing bias that only moves the choice).
//
// One block scores 32 tokens against all N experts on the CUDA cores (fp32
// FMA over d_model, operands staged through shared memory), keeps the
// [32 x N] score tile in shared memory, then each warp selects the top k of
// four tokens with warp shuffles: k rounds of a (key desc, index asc)
// argmax, so equal keys go to the lower index. Counts use shared-memory
// integer atomics (order-free, so exact); the per-expert probability sums
// are added in a fixed order (tokens of a warp, warps of a block, then
// blocks in a separate pass), so results are bitwise reproducible.
#include <float.h>

#include "device_util.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTok = kRouterTokens;          // 32 tokens per block
constexpr int kTokPerWarp = kTok / kWarps;   // 4
constexpr int kKC = 32;                      // d_model chunk staged in smem

struct RouterArgs {
  const void* x;
  const void* w;
  const float* logit_bias;
  const float* sel_bias;
  const float* logits_in;
  float* logits_out;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  float* partials;  // [gridDim.x][N]
  int* status;
  int T, d, N, k, gate_mode;
};

// Four consecutive elements of a row as fp32 (index must be a multiple of 4).
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
  float4 q = *reinterpret_cast<const float4*>(p);
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  uint2 q = *reinterpret_cast<const uint2*>(p);
  bf16x2_to_f32(q.x, v[0], v[1]);
  bf16x2_to_f32(q.y, v[2], v[3]);
}

// (key, index) ordering of the top-k: larger key first, then lower index.
__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// EJ = experts handled per lane (N <= 32 * EJ).
template <typename TX, int EJ>
__global__ void __launch_bounds__(kThreads) router_topk_kernel(const RouterArgs a) {
  extern __shared__ float smem[];
  const int N = a.N;
  const int NP = 32 * EJ;                       // padded expert count
  float* xs = smem;                             // [kTok][kKC]
  float* wsm = xs + kTok * kKC;                 // [NP][kKC + 1]
  float* lt = wsm + NP * (kKC + 1);             // [kTok][NP] scores
  float* wprob = lt + kTok * NP;                // [kWarps][NP]
  int* bcount = reinterpret_cast<int*>(wprob + kWarps * NP);  // [NP]

  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  const int t0 = blockIdx.x * kTok;

  for (int e = tid; e < NP; e += kThreads) bcount[e] = 0;

  // ---- scores -------------------------------------------------------------
  if (a.logits_in == nullptr) {
    const TX* x = static_cast<const TX*>(a.x);
    const TX* w = static_cast<const TX*>(a.w);
    float acc[kTokPerWarp][EJ];
#pragma unroll
    for (int i = 0; i < kTokPerWarp; ++i)
#pragma unroll
      for (int j = 0; j < EJ; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < a.d; k0 += kKC) {
      // x chunk: 32 tokens x 32 columns, 4 columns per thread.
      {
        const int r = tid / 8, c = (tid % 8) * 4;
        const int t = t0 + r;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (t < a.T && k0 + c < a.d) load4(x + (size_t)t * a.d + k0 + c, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) xs[r * kKC + c + q] = v[q];
      }
      // router weight chunk: N rows x 32 columns.
      for (int i = tid; i < NP * 8; i += kThreads) {
        const int r = i / 8, c = (i % 8) * 4;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (r < N && k0 + c < a.d) load4(w + (size_t)r * a.d + k0 + c, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) wsm[r * (kKC + 1) + c + q] = v[q];
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < kKC; ++kk) {
        float xv[kTokPerWarp], wv[EJ];
#pragma unroll
        for (int i = 0; i < kTokPerWarp; ++i) xv[i] = xs[(warp * kTokPerWarp + i) * kKC + kk];
#pragma unroll
        for (int j = 0; j < EJ; ++j) wv[j] = wsm[(lane + 32 * j) * (kKC + 1) + kk];
#pragma unroll
        for (int i = 0; i < kTokPerWarp; ++i)
#pragma unroll
          for (int j = 0; j < EJ; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < kTokPerWarp; ++i)
#pragma unroll
      for (int j = 0; j < EJ; ++j) {
        const int e = lane + 32 * j;
        float r = acc[i][j];
        if (e < N && a.logit_bias) r = __fadd_rn(r, a.logit_bias[e]);
        lt[(warp * kTokPerWarp + i) * NP + e] = r;
      }
  } else {
    for (int i = tid; i < kTok * NP; i += kThreads) {
      const int r = i / NP, e = i % NP;
      const int t = t0 + r;
      lt[i] = (t < a.T && e < N) ? a.logits_in[(size_t)t * N + e] : 0.f;
    }
  }
  __syncthreads();

  if (a.logits_out) {
    for (int i = tid; i < kTok * N; i += kThreads) {
      const int r = i / N, e = i % N;
      if (t0 + r < a.T) a.logits_out[(size_t)(t0 + r) * N + e] = lt[r * NP + e];
    }
  }

  // ---- top-k, gates, statistics: one warp per 4 tokens -----------------------
  float psum[EJ];
#pragma unroll
  for (int j = 0; j < EJ; ++j) psum[j] = 0.f;

  for (int i = 0; i < kTokPerWarp; ++i) {
    const int tl = warp * kTokPerWarp + i;
    const int t = t0 + tl;
    if (t >= a.T) break;  // warp-uniform
    float r[EJ], key[EJ];
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
      const int e = lane + 32 * j;
      r[j] = (e < N) ? lt[tl * NP + e] : -FLT_MAX;
      key[j] = (e < N && a.sel_bias) ? __fadd_rn(r[j], a.sel_bias[e]) : r[j];
    }
    // Full softmax over the N unbiased scores (the affinity probabilities).
    float m = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < EJ; ++j)
      if (lane + 32 * j < N) m = fmaxf(m, r[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float p[EJ];
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
      p[j] = (lane + 32 * j < N) ? expf(r[j] - m) : 0.f;
      z += p[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
      p[j] = p[j] / z;
      psum[j] += p[j];
    }

    // k rounds of warp argmax over (key, index).
    uint32_t taken = 0;
    int sel[kMaxTopK];
    float rsel[kMaxTopK];
    for (int s = 0; s < a.k; ++s) {
      float bk = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < EJ; ++j) {
        const int e = lane + 32 * j;
        if (e < N && !(taken & (1u << j)) && better(key[j], e, bk, bi)) {
          bk = key[j];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ok, oi, bk, bi)) {
          bk = ok;
          bi = oi;
        }
      }
      sel[s] = bi;
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      rsel[s] = lt[tl * NP + bi];
    }
    if (lane == 0) {
      float g[kMaxTopK];
      if (a.gate_mode == MOE_GATE_TOPK_SOFTMAX) {
        float mk = rsel[0];
        for (int s = 1; s < a.k; ++s) mk = fmaxf(mk, rsel[s]);
        float zs = 0.f;
        for (int s = 0; s < a.k; ++s) {
          g[s] = expf(rsel[s] - mk);
          zs += g[s];
        }
        for (int s = 0; s < a.k; ++s) g[s] = g[s] / zs;
      } else {
        float zs = 0.f;
        for (int s = 0; s < a.k; ++s) {
          g[s] = expf(rsel[s] - m) / z;
          zs += g[s];
        }
        for (int s = 0; s < a.k; ++s) g[s] = g[s] / zs;
      }
      for (int s = 0; s < a.k; ++s) {
        a.topk_idx[(size_t)t * a.k + s] = sel[s];
        a.topk_w[(size_t)t * a.k + s] = g[s];
        atomicAdd(&bcount[sel[s]], 1);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < EJ; ++j) wprob[warp * NP + lane + 32 * j] = psum[j];
  __syncthreads();
  for (int e = tid; e < N; e += kThreads) {
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += wprob[w * NP + e];
    a.partials[(size_t)blockIdx.x * N + e] = s;
    if (bcount[e]) atomicAdd(&a.counts[e], bcount[e]);
  }
}

// prob_sum[e] = sum over blocks, in block order.
__global__ void router_reduce_kernel(const float* partials, int nblk, int N, float* prob_sum) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= N) return;
  float s = 0.f;
  for (int b = 0; b < nblk; ++b) s += partials[(size_t)b * N + e];
  prob_sum[e] = s;
}

template <typename TX, int EJ>
cudaError_t launch_t(const RouterArgs& a, int nblk, cudaStream_t s) {
  const int NP = 32 * EJ;
  const size_t smem = sizeof(float) * ((size_t)kTok * kKC + (size_t)NP * (kKC + 1) +
                                       (size_t)kTok * NP + (size_t)kWarps * NP) +
                      sizeof(int) * NP;
  cudaError_t e = cudaFuncSetAttribute(router_topk_kernel<TX, EJ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ProfScope p(K_ROUTER, s);
  router_topk_kernel<TX, EJ><<<nblk, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename TX>
cudaError_t launch_dtype(const RouterArgs& a, int nblk, cudaStream_t s) {
  if (a.N <= 32) return launch_t<TX, 1>(a, nblk, s);
  if (a.N <= 64) return launch_t<TX, 2>(a, nblk, s);
  if (a.N <= 128) return launch_t<TX, 4>(a, nblk, s);
  return launch_t<TX, 8>(a, nblk, s);
}

}  // namespace

size_t router_partials_bytes(const moe_config& c) {
  return sizeof(float) * (size_t)ceil_div(c.T, kTok) * (size_t)c.n_experts;
}

cudaError_t launch_router(const moe_config& c, const void* x, const void* w_router,
                          const float* logit_bias, const float* sel_bias,
                          const float* logits_in, float* logits_out, int32_t* topk_idx,
                          float* topk_w, int32_t* counts, float* prob_sum, float* partials,
                          int* status, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.n_experts, s);
  if (e != cudaSuccess) return e;
  if (c.T == 0) return cudaMemsetAsync(prob_sum, 0, sizeof(float) * c.n_experts, s);
  RouterArgs a;
  a.x = x; a.w = w_router; a.logit_bias = logit_bias; a.sel_bias = sel_bias;
  a.logits_in = logits_in; a.logits_out = logits_out; a.topk_idx = topk_idx;
  a.topk_w = topk_w; a.counts = counts; a.partials = partials; a.status = status;
  a.T = c.T; a.d = c.d_model; a.N = c.n_experts; a.k = c.top_k; a.gate_mode = c.gate_mode;
  const int nblk = ceil_div(c.T, kTok);
  e = (c.dtype == MOE_BF16) ? launch_dtype<__nv_bfloat16>(a, nblk, s) : launch_dtype<float>(a, nblk, s);
  if (e != cudaSuccess) return e;
  {
    ProfScope p(K_ROUTER_REDUCE, s);
    router_reduce_kernel<<<ceil_div(c.n_experts, 256), 256, 0, s>>>(partials, nblk, c.n_experts, prob_sum);
  }
  return cudaGetLastError();
}

}  // namespace moe
