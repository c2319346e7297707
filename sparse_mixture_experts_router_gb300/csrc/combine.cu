// K5: gate-weighted sum back into token order, and the balance statistics.
//
// y[t] = sum_slot w * y_perm[inv_pos[t*k+slot]] + sum_shared y_perm[T*k+s*T+t]
// ("Mixture of experts and speculative decoding", step 4 and the layer
// equation; "Mixture of Experts and Guided Decoding", the three-expert gated
// sum). One warp per token; each output vector accumulates the k + n_shared
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

// WPT warps per token (1, 2 or 4, so that a lane sums about 8 vectors and
// blocks stay short). Lane j of each of the token's warps fetches term j's
// row and weight (slot j for j < k, shared expert j - k after them) and
// shuffles them to the warp; each lane then sums whole 16-byte vectors of
// the output row, loading all NT terms of a vector before adding them in
// fp32 in term order (slots, then shared experts), and stores once. NT is
// k + n_shared rounded up to a template size; terms past the token's own
// count are skipped.
constexpr int kWarpsPerBlock = kThreads / 32;
template <typename TE, int NT, int UNROLL>
__global__ void __launch_bounds__(kThreads) combine_kernel(const TE* __restrict__ yp,
                                                           const int32_t* __restrict__ inv_pos,
                                                           const float* __restrict__ topk_w,
                                                           TE* __restrict__ y, int T, int d, int k,
                                                           int n_shared, int wpt) {
  constexpr int V = Vec<TE>::n;
  const int lane = threadIdx.x % 32;
  const int warp = threadIdx.x / 32;
  const long long t = (long long)blockIdx.x * (kWarpsPerBlock / wpt) + warp / wpt;
  const int part = warp % wpt;
  const long long P = (long long)T * k;
  pdl_wait();
  pdl_trigger();
  if (t >= T) return;
  long long my_row = -1;
  float my_w = 1.0f;
  if (lane < k) {
    const int pos = inv_pos[t * k + lane];
    if (pos >= 0 && pos < P) my_row = pos;  // out of range: contributes zero
    if (topk_w) my_w = topk_w[t * k + lane];
  } else if (lane < k + n_shared) {
    my_row = P + (long long)(lane - k) * T + t;
  }
  const uint4* src[NT];
  float w[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const long long r = __shfl_sync(0xffffffffu, my_row, j);
    w[j] = __shfl_sync(0xffffffffu, my_w, j);
    src[j] = r >= 0 ? reinterpret_cast<const uint4*>(yp + r * d) : nullptr;
  }
  const int nvec = d / V;
  uint4* dst = reinterpret_cast<uint4*>(y + t * d);
#pragma unroll UNROLL
  for (int v = part * 32 + lane; v < nvec; v += 32 * wpt) {
    uint4 raw[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) raw[j] = src[j] ? __ldg(src[j] + v) : make_uint4(0, 0, 0, 0);
    float acc[V];
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = 0.f;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      if (!src[j]) continue;
      float val[V];
      Vec<TE>::unpack(raw[j], val);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] = fmaf(w[j], val[q], acc[q]);
    }
    Vec<TE>::store(reinterpret_cast<TE*>(dst + v), acc);
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

template <typename TE, int NT, int UNROLL>
cudaError_t launch_combine_t(const moe_config& c, const void* y_perm, const int32_t* inv_pos,
                             const float* topk_w, void* y, cudaStream_t s) {
  const int nvec = c.d_model / Vec<TE>::n;
  int wpt = 1;
  while (wpt < 4 && nvec > 32 * 8 * wpt) wpt *= 2;
  return launch_pdl(combine_kernel<TE, NT, UNROLL>, dim3(ceil_div(c.T, kWarpsPerBlock / wpt)),
                    dim3(kThreads), 0, s, 1, static_cast<const TE*>(y_perm), inv_pos, topk_w,
                    static_cast<TE*>(y), c.T, c.d_model, c.top_k, c.n_shared, wpt);
}

template <typename TE>
cudaError_t launch_combine_dt(const moe_config& c, const void* y_perm, const int32_t* inv_pos,
                              const float* topk_w, void* y, cudaStream_t s) {
  const int terms = c.top_k + c.n_shared;
  if (terms <= 2) return launch_combine_t<TE, 2, 4>(c, y_perm, inv_pos, topk_w, y, s);
  if (terms <= 4) return launch_combine_t<TE, 4, 2>(c, y_perm, inv_pos, topk_w, y, s);
  if (terms <= 8) return launch_combine_t<TE, 8, 1>(c, y_perm, inv_pos, topk_w, y, s);
  if (terms == 9) return launch_combine_t<TE, 9, 1>(c, y_perm, inv_pos, topk_w, y, s);
  return launch_combine_t<TE, kMaxTopK + kMaxShared, 1>(c, y_perm, inv_pos, topk_w, y, s);
}

cudaError_t launch_combine(const moe_config& c, const void* y_perm, const int32_t* inv_pos,
                           const float* topk_w, void* y, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  ProfScope p(K_COMBINE, s);
  if (c.dtype == MOE_BF16)
    return launch_combine_dt<__nv_bfloat16>(c, y_perm, inv_pos, topk_w, y, s);
  return launch_combine_dt<float>(c, y_perm, inv_pos, topk_w, y, s);
}

cudaError_t launch_balance_stats(int N, int T, int k, const int32_t* counts, const float* prob_sum,
                                 float alpha, float* f, float* P, float* aux, cudaStream_t s) {
  ProfScope p(K_BALANCE, s);
  return launch_pdl(balance_stats_kernel, dim3(1), dim3(256), 0, s, 1, counts, prob_sum, N, T, k,
                    alpha, f, P, aux);
}

}  // namespace moe
