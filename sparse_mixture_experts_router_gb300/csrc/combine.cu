// K5: gate-weighted sum back into token order, and the balance statistics.
//
// y[t] = sum_slot w * y_perm[inv_pos[t*k+slot]] + sum_shared y_perm[T*k+s*T+t]
// ("Mixture of experts and speculative decoding", step 4 and the layer
// equation; "Mixture of Experts and Guided Decoding", the three-expert gated
// sum). One block per token; each output vector accumulates the k + n_shared
// rows' vectors in fp32 in a fixed order (slots, then shared experts) and is
// written exactly once, so there are no atomics and the result is
// reproducible.
#include "device_util.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;

template <typename TE>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int n = 4;
  __device__ static void unpack(const uint4& q, float (&v)[4]) {
    v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
    v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
  }
  __device__ static void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void unpack(const uint4& q, float (&v)[8]) {
    bf16x2_to_f32(q.x, v[0], v[1]);
    bf16x2_to_f32(q.y, v[2], v[3]);
    bf16x2_to_f32(q.z, v[4], v[5]);
    bf16x2_to_f32(q.w, v[6], v[7]);
  }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(f32x2_to_bf16x2(v[0], v[1]), f32x2_to_bf16x2(v[2], v[3]),
                                              f32x2_to_bf16x2(v[4], v[5]), f32x2_to_bf16x2(v[6], v[7]));
  }
};

// One block per token: the token's k slot rows and weights are read once into
// shared memory, then each thread sums whole 16-byte vectors of the output
// row, loading all k + n_shared terms of a vector before adding them in fp32
// in slot order then shared order, and stores once.
template <typename TE>
__global__ void __launch_bounds__(kThreads) combine_kernel(const TE* __restrict__ yp,
                                                           const int32_t* __restrict__ inv_pos,
                                                           const float* __restrict__ topk_w,
                                                           TE* __restrict__ y, int T, int d, int k,
                                                           int n_shared) {
  constexpr int V = Vec<TE>::n;
  constexpr int TERMS = kMaxTopK + kMaxShared;
  __shared__ long long s_row[TERMS];
  __shared__ float s_w[TERMS];
  const int t = blockIdx.x;
  const long long P = (long long)T * k;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < TERMS) {
    const int j = threadIdx.x;
    long long row = -1;
    float w = 1.0f;
    if (j < kMaxTopK) {
      if (j < k) {
        const int pos = inv_pos[(size_t)t * k + j];
        if (pos >= 0 && pos < P) row = pos;  // out of range: contributes zero
        if (topk_w) w = topk_w[(size_t)t * k + j];
      }
    } else if (j - kMaxTopK < n_shared) {
      row = P + (long long)(j - kMaxTopK) * T + t;
    }
    s_row[j] = row;
    s_w[j] = w;
  }
  __syncthreads();
  const int nvec = d / V;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    uint4 raw[TERMS];
#pragma unroll
    for (int j = 0; j < TERMS; ++j)
      raw[j] = s_row[j] >= 0 ? __ldg(reinterpret_cast<const uint4*>(yp + s_row[j] * d) + v)
                             : make_uint4(0, 0, 0, 0);
    float acc[V];
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = 0.f;
#pragma unroll
    for (int j = 0; j < TERMS; ++j) {
      if (s_row[j] < 0) continue;
      float val[V];
      Vec<TE>::unpack(raw[j], val);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] = fmaf(s_w[j], val[q], acc[q]);
    }
    Vec<TE>::store(y + (size_t)t * d + (size_t)v * V, acc);
  }
}

__global__ void balance_stats_kernel(const int32_t* counts, const float* prob_sum, int N, int T,
                                     int k, float alpha, float* f, float* P, float* aux) {
  __shared__ float fp[kMaxExperts];
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    const float fe = T > 0 ? (float)counts[e] / ((float)T * (float)k) : 0.f;
    const float pe = T > 0 ? prob_sum[e] / (float)T : 0.f;
    f[e] = fe;
    P[e] = pe;
    fp[e] = fe * pe;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int e = 0; e < N; ++e) s += fp[e];
    *aux = alpha * (float)N * s;
  }
}

}  // namespace

cudaError_t launch_combine(const moe_config& c, const void* y_perm, const int32_t* inv_pos,
                           const float* topk_w, void* y, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  // one block per token, at most one thread per 16-byte vector of the row
  const int nvec = c.d_model / (c.dtype == MOE_BF16 ? 8 : 4);
  const int threads = nvec >= kThreads ? kThreads : ((nvec + 31) / 32) * 32;
  const int grid = c.T;
  ProfScope p(K_COMBINE, s);
  if (c.dtype == MOE_BF16)
    return launch_pdl(combine_kernel<__nv_bfloat16>, dim3(grid), dim3(threads), 0, s, 1,
                      static_cast<const __nv_bfloat16*>(y_perm), inv_pos, topk_w,
                      static_cast<__nv_bfloat16*>(y), c.T, c.d_model, c.top_k, c.n_shared);
  return launch_pdl(combine_kernel<float>, dim3(grid), dim3(threads), 0, s, 1,
                    static_cast<const float*>(y_perm), inv_pos, topk_w, static_cast<float*>(y),
                    c.T, c.d_model, c.top_k, c.n_shared);
}

cudaError_t launch_balance_stats(int N, int T, int k, const int32_t* counts, const float* prob_sum,
                                 float alpha, float* f, float* P, float* aux, cudaStream_t s) {
  ProfScope p(K_BALANCE, s);
  return launch_pdl(balance_stats_kernel, dim3(1), dim3(256), 0, s, 1, counts, prob_sum, N, T, k,
                    alpha, f, P, aux);
}

}  // namespace moe
