// Backward of the layer: the CUDA-core steps around the tensor-core GEMMs.
//
// The loss is L = sum(dy * y) + aux_grad * aux with aux = alpha * N *
// sum_i f_i P_i ("Mixture of experts and speculative decoding", the layer
// equation and "Keeping the experts busy"; "Mixture of Experts and Guided
// Decoding", the auxiliary-loss formula: f comes from a hard choice and is
// not differentiated, the gradient flows through P). Routing is held fixed.
//
//  bwd_gate_kernel    dL/dg of every kept pair, <dy[t], o[row]> with o the
//                     unweighted expert output, and dO[row] = g * dy[t]
//                     (dy itself for shared-expert rows);
//  bwd_score_kernel   dL/dr per token: the gates' softmax backward plus the
//                     balance term alpha * N / T * p * (f - <p, f>), stored in
//                     bf16 as dr [T][n_pad] and drT [n_pad][t_pad], the
//                     operands of dx = dr W_r and dW_r = dr^T x (tensor cores,
//                     wgrad_sm103.cu);
//  bwd_dx_kernel      dx[t] += the token's dA rows (kept slots, then shared
//                     experts), on top of dr W_r.
// Every sum runs in a fixed order, so the results are reproducible.
#include "device_util.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per pair (t, slot), then one per shared-expert row.
__global__ void __launch_bounds__(kThreads)
    bwd_gate_kernel(const __nv_bfloat16* __restrict__ dy, const __nv_bfloat16* __restrict__ o,
                    const int32_t* __restrict__ inv_pos, const float* __restrict__ topk_w,
                    float* __restrict__ dg, __nv_bfloat16* __restrict__ dO, int T, int d, int k,
                    int n_shared) {
  const int lane = threadIdx.x % 32;
  const long long w = (long long)blockIdx.x * kWarps + threadIdx.x / 32;
  const long long P = (long long)T * k;
  pdl_wait();
  pdl_trigger();
  if (w >= P + (long long)n_shared * T) return;
  long long t, row;
  float g = 1.0f;
  if (w < P) {
    t = w / k;
    const int pos = inv_pos[w];
    if (pos < 0 || pos >= P) {  // dropped by the capacity cut: not in y
      if (lane == 0) dg[w] = 0.0f;
      return;
    }
    row = pos;
    g = topk_w[w];
  } else {
    const long long q = w - P;
    t = q % T;
    row = w;  // shared expert s owns rows P + s*T + t
  }
  const uint4* py = reinterpret_cast<const uint4*>(dy + t * d);
  const uint4* po = reinterpret_cast<const uint4*>(o + row * d);
  uint4* pd = reinterpret_cast<uint4*>(dO + row * d);
  float dot = 0.0f;
  for (int v = lane; v < d / 8; v += 32) {
    const uint4 a = __ldg(py + v);
    const uint4 b = __ldg(po + v);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float a0, a1, b0, b1;
      bf16x2_to_f32(aw[i], a0, a1);
      bf16x2_to_f32(bw[i], b0, b1);
      dot += a0 * b0 + a1 * b1;
      out[i] = f32x2_to_bf16x2(g * a0, g * a1);
    }
    pd[v] = make_uint4(out[0], out[1], out[2], out[3]);
  }
  dot = warp_sum(dot);
  if (w < P && lane == 0) dg[w] = dot;
}

// One warp per token; lane l holds experts l, l + 32, ... (N <= 256).
__global__ void __launch_bounds__(kThreads)
    bwd_score_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                     const float* __restrict__ topk_w, const float* __restrict__ dg,
                     const int32_t* __restrict__ counts, __nv_bfloat16* __restrict__ dr,
                     __nv_bfloat16* __restrict__ drT, int T, int N, int k, int n_pad, int t_pad,
                     float balance_scale) {
  constexpr int EPL = kMaxExperts / 32;
  const int lane = threadIdx.x % 32;
  const long long t = (long long)blockIdx.x * kWarps + threadIdx.x / 32;
  pdl_wait();
  pdl_trigger();
  if (t >= T) return;
  float r[EPL], acc[EPL];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    r[i] = e < N ? logits[t * N + e] : -INFINITY;
    acc[i] = 0.0f;
    m = fmaxf(m, r[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.0f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    r[i] = (lane + 32 * i < N) ? __expf(r[i] - m) : 0.0f;  // unnormalised p
    z += r[i];
  }
  z = warp_sum(z);
  const float inv_z = 1.0f / z;
  const float inv_tk = 1.0f / ((float)T * (float)k);
  float pf = 0.0f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    r[i] *= inv_z;  // p
    if (e < N) pf += r[i] * (float)counts[e] * inv_tk;
  }
  pf = warp_sum(pf);
  // gates: g = softmax over the kept scores (in both gate modes the kept
  // probabilities renormalised are that softmax), dr_j += g_j (dG_j - <g, dG>)
  float my_g = 0.0f, my_dg = 0.0f;
  int my_e = -1;
  if (lane < k) {
    my_e = topk_idx[t * k + lane];
    my_g = topk_w[t * k + lane];
    my_dg = dg[t * k + lane];
  }
  const float gdg = warp_sum(my_g * my_dg);
  for (int s = 0; s < k; ++s) {
    const int e = __shfl_sync(0xffffffffu, my_e, s);
    const float v = __shfl_sync(0xffffffffu, my_g * (my_dg - gdg), s);
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i == e) acc[i] += v;
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < N) {
      const float f = (float)counts[e] * inv_tk;
      const __nv_bfloat16 v = __float2bfloat16_rn(acc[i] + balance_scale * r[i] * (f - pf));
      dr[t * n_pad + e] = v;
      drT[(long long)e * t_pad + t] = v;
    } else if (e < n_pad) {
      dr[t * n_pad + e] = __float2bfloat16_rn(0.0f);
    }
  }
}

// One warp per token; lanes take 16-byte vectors of the row in turn.
template <int MAXT>
__global__ void __launch_bounds__(kThreads)
    bwd_dx_kernel(const __nv_bfloat16* __restrict__ dA, const int32_t* __restrict__ inv_pos,
                  float* __restrict__ dx, int T, int d, int k, int n_shared) {
  const int lane = threadIdx.x % 32;
  const long long t = (long long)blockIdx.x * kWarps + threadIdx.x / 32;
  const long long P = (long long)T * k;
  pdl_wait();
  pdl_trigger();
  if (t >= T) return;
  long long rows[MAXT];
  int nt = 0;
  for (int s = 0; s < k; ++s) {
    const int pos = inv_pos[t * k + s];
    if (pos >= 0 && pos < P) rows[nt++] = pos;
  }
  for (int q = 0; q < n_shared; ++q) rows[nt++] = P + (long long)q * T + t;
  for (int v = lane; v < d / 8; v += 32) {
    float4* out = reinterpret_cast<float4*>(dx + t * d) + 2 * v;
    const float4 r0 = out[0], r1 = out[1];  // dr W_r
    float acc[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    for (int i = 0; i < nt; ++i) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(dA + rows[i] * d) + v);
      const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float a0, a1;
        bf16x2_to_f32(qw[j], a0, a1);
        acc[2 * j] += a0;
        acc[2 * j + 1] += a1;
      }
    }
    out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

}  // namespace

cudaError_t launch_bwd_gate(const moe_config& c, const void* dy, const void* o,
                            const int32_t* inv_pos, const float* topk_w, float* dg, void* dO,
                            cudaStream_t s) {
  const long long warps = (long long)c.T * c.top_k + (long long)c.n_shared * c.T;
  if (warps == 0) return cudaSuccess;
  ProfScope p(K_BWD_GATE, s);
  return launch_pdl(bwd_gate_kernel, dim3(ceil_div(warps, kWarps)), dim3(kThreads), 0, s, 1,
                    static_cast<const __nv_bfloat16*>(dy), static_cast<const __nv_bfloat16*>(o),
                    inv_pos, topk_w, dg, static_cast<__nv_bfloat16*>(dO), c.T, c.d_model,
                    c.top_k, c.n_shared);
}

cudaError_t launch_bwd_score(const moe_config& c, const float* logits, const int32_t* topk_idx,
                             const float* topk_w, const float* dg, const int32_t* counts,
                             float alpha, float aux_grad, void* dr_bf, void* drT_bf, int n_pad,
                             int t_pad, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  ProfScope p(K_BWD_SCORE, s);
  const float scale = aux_grad * alpha * (float)c.n_experts / (float)c.T;
  return launch_pdl(bwd_score_kernel, dim3(ceil_div(c.T, kWarps)), dim3(kThreads), 0, s, 1,
                    logits, topk_idx, topk_w, dg, counts, static_cast<__nv_bfloat16*>(dr_bf),
                    static_cast<__nv_bfloat16*>(drT_bf), c.T, c.n_experts, c.top_k, n_pad, t_pad,
                    scale);
}

cudaError_t launch_bwd_dx(const moe_config& c, const void* dA, const int32_t* inv_pos, float* dx,
                          cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  ProfScope p(K_BWD_DX, s);
  static_assert(kMaxTopK + kMaxShared <= 12, "term table");
  return launch_pdl(bwd_dx_kernel<12>, dim3(ceil_div(c.T, kWarps)), dim3(kThreads), 0, s, 1,
                    static_cast<const __nv_bfloat16*>(dA), inv_pos, dx, c.T, c.d_model, c.top_k,
                    c.n_shared);
}

}  // namespace moe
