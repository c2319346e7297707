// Decode-sized layers (T <= 8 tokens, N <= 32 routed experts, bf16) in one
// cooperative kernel.
//
// A decode step is weight streaming: every expert a token chooses is read
// once, 3 d d_ff weights for a handful of rows ("MoE inference: the call
// centre with 256 specialists and 8 taking each call", "The maths that
// matters": decode stays memory-bound). The general path spends eight
// launches on it (status, router, permutation, gather, two GEMMs, split-K
// reduction, combine), and their latencies are a third of a T = 1 step. Here
// one kernel does the whole layer, with the same definitions as those kernels
// ("Mixture of experts and speculative decoding", steps 1-4 and the layer
// equation):
//
//  0. Every CTA routes all T tokens itself (T N <= 256 dot products of
//     length d over x staged in shared memory): scores, selection key
//     fp32(r + sel_bias) with NaN below every number and ties to the lower
//     index, gates in either mode, the capacity cut, and the list of active
//     experts with their (token, H row, gate) terms (shared experts last,
//     every token, gate 1). CTA 0 writes topk_idx / topk_w / counts /
//     prob_sum.
//  1. Gate/up: warp-sized units (active expert, half of row j of d_ff); a
//     warp streams that half of W_g[e][j] and of W_u[e][j] with 16-byte
//     loads and stores the two partial dot products (a, b) of each of the
//     expert's terms; the halves are summed when H is staged.
//  2. A grid barrier (an atomic counter, bounded spin, cooperative launch so
//     every CTA is resident).
//  3. Down, in items of (active expert, K chunk, 32 output features), each
//     CTA a contiguous run of them: the chunk of H[term] = bf16(SiLU(a) * b)
//     is staged in shared memory (once for the run's items of one expert and
//     chunk), and each warp stores the partial sums W_d[e][c][chunk] .
//     H[term][chunk] of 4 features.
//  4. A second barrier, then y[t][c] = sum over the token's terms (experts
//     in ascending order, shared ones after) of g times the sum of its
//     partials over the chunks, in fp32 in that order, written once as bf16.
//
// Every sum runs in a fixed order. Weights are read with 16-byte vectors
// that bypass L1; H is read at L2 (it was written by other CTAs).
#include <float.h>

#include <atomic>

#include "device_util.cuh"
#include "moe_internal.h"
#include "sm103_wait.cuh"

namespace moe {
namespace {

constexpr int DF_THREADS = 256;
constexpr int DF_WARPS = DF_THREADS / 32;
constexpr int DF_MAX_T = 8;
constexpr int DF_MAX_N = 32;
constexpr int DF_MAX_ACT = DF_MAX_N + kMaxShared;
// K chunk of a down-projection unit: the largest of 2048, 1024, 512, 256
// dividing d_ff (short units keep the warps' work even).

struct DecodeArgs {
  const __nv_bfloat16* x;
  const __nv_bfloat16* w_router;
  const float* logit_bias;
  const float* sel_bias;
  const __nv_bfloat16* w_gate;
  const __nv_bfloat16* w_up;
  const __nv_bfloat16* w_down;
  __nv_bfloat16* y;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  float* prob_sum;
  float* ab;         // [T * (k + s)][2 halves][a | b][d_ff] fp32 pre-activation halves
  float* part;       // [active experts][MT][d_ff / chunk][d] partial sums
  int chunk;
  int* status;       // [0] status word, [2] grid-barrier counter (zero at launch)
  int T, d, N, k, s, d_ff, gate_mode, capacity;
  // Bounded grid-barrier waits: the limit, and arrivals the barriers wait for
  // beyond the grid's own (0; 1 only under moe_set_decode_barrier_test, an
  // arrival that never comes, so that every wait runs out).
  unsigned long long barrier_limit_ns;
  int barrier_withheld;
};

struct DfShared {
  float score[DF_MAX_T][DF_MAX_N];
  float p[DF_MAX_T][DF_MAX_N];  // softmax over all N scores
  int idx[DF_MAX_T][kMaxTopK];
  float g[DF_MAX_T][kMaxTopK];
  int n_act;
  int act_e[DF_MAX_ACT];
  int act_nt[DF_MAX_ACT];
  int act_tok[DF_MAX_ACT][DF_MAX_T];
  int act_q[DF_MAX_ACT][DF_MAX_T];
  float act_g[DF_MAX_ACT][DF_MAX_T];
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& q, float (&f)[8]) {
  bf16x2_to_f32(q.x, f[0], f[1]);
  bf16x2_to_f32(q.y, f[2], f[3]);
  bf16x2_to_f32(q.z, f[4], f[5]);
  bf16x2_to_f32(q.w, f[6], f[7]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ bool key_better(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + __expf(-v)); }

// Grid barrier: every CTA adds one to the counter and waits (bounded by
// limit_ns) until all have. Returns false if the wait ran out (the status
// word then says so).
__device__ bool grid_barrier(int* counter, int* status, int target, uint64_t limit_ns) {
  __syncthreads();
  __shared__ int ok;
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(counter, 1);
    ok = 1;
    const uint64_t t0 = globaltimer_ns();
    while (*reinterpret_cast<volatile int*>(counter) < target) {
      if (globaltimer_ns() - t0 > limit_ns) {
        set_status(status, MOE_ERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
  return ok != 0;
}

// Routing of all T tokens into `sh` (every CTA); CTA 0 also writes the
// routing outputs. x is staged (fp32) in xs [T][d] first.
__device__ void route_tokens(const DecodeArgs& a, DfShared& sh, float* xs) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int T = a.T, d = a.d, N = a.N, k = a.k;
  const int terms = k + a.s;
  // scores: a warp a (token, expert) pair, x and W_r read straight from
  // global memory (one round trip: the loads do not wait on each other)
  for (int pr = warp; pr < T * N; pr += DF_WARPS) {
    const int t = pr / N, e = pr % N;
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)t * d);
    const uint4* wr = reinterpret_cast<const uint4*>(a.w_router + (size_t)e * d);
    float acc = 0.f;
#pragma unroll 8
    for (int v = lane; v < d / 8; v += 32) {
      float wf[8], xf[8];
      unpack8(__ldg(wr + v), wf);
      unpack8(__ldg(xr + v), xf);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc = fmaf(xf[q], wf[q], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) sh.score[t][e] = a.logit_bias ? __fadd_rn(acc, a.logit_bias[e]) : acc;
  }
  // x in fp32 for the gate/up phase
  for (int i = threadIdx.x; i < T * d / 8; i += DF_THREADS) {
    float f[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(a.x) + i), f);
    reinterpret_cast<float4*>(xs)[2 * i] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(xs)[2 * i + 1] = make_float4(f[4], f[5], f[6], f[7]);
  }
  __syncthreads();
  for (int t = warp; t < T; t += DF_WARPS) {
    const bool in = lane < N;
    const float r = in ? sh.score[t][lane] : -FLT_MAX;
    float key = (in && a.sel_bias) ? __fadd_rn(r, a.sel_bias[lane]) : r;
    if (key != key) key = -INFINITY;  // a NaN key ranks below every number
    float m = in ? r : -FLT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float pe = in ? expf(r - m) : 0.f;
    const float z = warp_sum(pe);
    if (in) sh.p[t][lane] = pe / z;
    bool taken = !in;
    for (int s = 0; s < k; ++s) {  // k rounds of warp argmax over (key, lower index)
      float bk = taken ? -INFINITY : key;
      int bi = taken ? 0x7fffffff : lane;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (key_better(ok, oi, bk, bi)) {
          bk = ok;
          bi = oi;
        }
      }
      const float rs = __shfl_sync(0xffffffffu, r, bi & 31);
      if (lane == 0) {
        sh.idx[t][s] = bi;
        sh.g[t][s] = rs;
      }
      if (bi == lane) taken = true;
    }
    if (lane == 0) {
      // sh.g holds the kept scores; turn them into gates
      float zs = 0.f;
      if (a.gate_mode == MOE_GATE_TOPK_SOFTMAX) {
        float mk = sh.g[t][0];
        for (int s = 1; s < k; ++s) mk = fmaxf(mk, sh.g[t][s]);
        for (int s = 0; s < k; ++s) {
          sh.g[t][s] = expf(sh.g[t][s] - mk);
          zs += sh.g[t][s];
        }
      } else {
        for (int s = 0; s < k; ++s) {
          sh.g[t][s] = expf(sh.g[t][s] - m) / z;
          zs += sh.g[t][s];
        }
      }
      for (int s = 0; s < k; ++s) sh.g[t][s] = sh.g[t][s] / zs;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // the capacity cut (ascending token, then slot, within each expert) and
    // the active experts with their terms
    int n = 0;
    for (int e = 0; e < N; ++e) {
      int taken = 0, nt = 0;
      for (int t = 0; t < T; ++t)
        for (int s = 0; s < k; ++s)
          if (sh.idx[t][s] == e) {
            if (a.capacity == 0 || taken < a.capacity) {
              sh.act_tok[n][nt] = t;
              sh.act_q[n][nt] = t * terms + s;
              sh.act_g[n][nt] = sh.g[t][s];
              ++nt;
            }
            ++taken;
          }
      if (nt > 0) {
        sh.act_e[n] = e;
        sh.act_nt[n] = nt;
        ++n;
      }
    }
    for (int q = 0; q < a.s; ++q) {
      sh.act_e[n] = N + q;
      sh.act_nt[n] = T;
      for (int t = 0; t < T; ++t) {
        sh.act_tok[n][t] = t;
        sh.act_q[n][t] = t * terms + k + q;
        sh.act_g[n][t] = 1.0f;
      }
      ++n;
    }
    sh.n_act = n;
  }
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < T * k; i += DF_THREADS) {
      a.topk_idx[i] = sh.idx[i / k][i % k];
      a.topk_w[i] = sh.g[i / k][i % k];
    }
    for (int e = threadIdx.x; e < N; e += DF_THREADS) {
      int c = 0;
      float ps = 0.f;
      for (int t = 0; t < T; ++t) {
        for (int s = 0; s < k; ++s) c += sh.idx[t][s] == e;
        ps += sh.p[t][e];
      }
      if (a.counts) a.counts[e] = c;
      if (a.prob_sum) a.prob_sum[e] = ps;
    }
  }
  __syncthreads();
}

// MT: the most tokens an expert can have in this launch (T rounded up to 1,
// 2, 4 or 8); the per-token accumulators live in registers.
template <int MT>
__global__ void __launch_bounds__(DF_THREADS, MT <= 2 ? 4 : 2) decode_layer_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* xs = reinterpret_cast<float*>(smem_raw);  // [T][d] fp32
  __shared__ DfShared sh;
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int T = a.T, d = a.d, dff = a.d_ff;
  route_tokens(a, sh, xs);
  const int gw = blockIdx.x * DF_WARPS + warp, GW = gridDim.x * DF_WARPS;
  const int n_act = sh.n_act;
  const int dh = d / 2;  // gate/up units take half a row, so the warps' work stays even

  // ---- 1. gate/up halves: ab[term][half][0|1][j] = W_{g|u}[e][j][half] . x --
  for (int u = gw; u < n_act * dff * 2; u += GW) {
    const int ei = u / (2 * dff);
    const int rem = u - ei * 2 * dff;
    const int j = rem >> 1, hf = rem & 1;
    const int e = sh.act_e[ei], nt = sh.act_nt[ei];
    const size_t off = ((size_t)e * dff + j) * d + (size_t)hf * dh;
    const uint4* wg = reinterpret_cast<const uint4*>(a.w_gate + off);
    const uint4* wu = reinterpret_cast<const uint4*>(a.w_up + off);
    int tok[MT];
#pragma unroll
    for (int i = 0; i < MT; ++i) tok[i] = i < nt ? sh.act_tok[ei][i] : 0;
    float ag[MT], au[MT];
#pragma unroll
    for (int i = 0; i < MT; ++i) ag[i] = au[i] = 0.f;
#pragma unroll 4
    for (int v = lane; v < dh / 8; v += 32) {
      float gf[8], uf[8];
      unpack8(ld_stream(wg + v), gf);
      unpack8(ld_stream(wu + v), uf);
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        if (i < nt) {
          const float4* xr =
              reinterpret_cast<const float4*>(xs + (size_t)tok[i] * d + (size_t)hf * dh) + 2 * v;
          const float4 x0 = xr[0], x1 = xr[1];
          const float xf[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            ag[i] = fmaf(gf[q], xf[q], ag[i]);
            au[i] = fmaf(uf[q], xf[q], au[i]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      if (i < nt) {
        const float gsum = warp_sum(ag[i]), usum = warp_sum(au[i]);
        if (lane == 0) {
          float* abp = a.ab + ((size_t)sh.act_q[ei][i] * 2 + hf) * 2 * dff;
          abp[j] = gsum;
          abp[dff + j] = usum;
        }
      }
    }
  }
  if (!grid_barrier(a.status + 2, a.status, gridDim.x + a.barrier_withheld, a.barrier_limit_ns))
    return;

  // ---- 2. down, in items of (expert, K chunk, 32 output features): the
  // chunk of H (bf16(SiLU(a) * b), a and b the sums of the two halves) of the
  // expert's terms is staged in shared memory, then each warp takes 4
  // features: part[term][chunk][c] = W_d[e][c][chunk] . H[term][chunk]. -----
  float* hs = xs + (size_t)T * d;  // [MT][chunk] fp32
  const int chunk = a.chunk, nch = dff / chunk;
  constexpr int CB = 32;  // features an item
  const int nfb = (d + CB - 1) / CB;
  const int n_items = n_act * nch * nfb;
  // A CTA takes a contiguous run of items: consecutive items share their
  // (expert, chunk) but for one in nfb, so the chunk of H is staged once for
  // the run rather than once an item (3.5% of a Mixtral-shaped step).
  const int it_end = (int)(((long long)(blockIdx.x + 1) * n_items) / gridDim.x);
  int staged = -1;  // the (expert, chunk) whose H is in hs (the same in every thread)
  for (int it = (int)(((long long)blockIdx.x * n_items) / gridDim.x); it < it_end; ++it) {
    const int pr = it / nfb, fb = it - pr * nfb;
    const int ei = pr / nch, ch = pr - ei * nch;
    const int e = sh.act_e[ei], nt = sh.act_nt[ei];
    __syncthreads();  // the previous item's warps are done with hs
    // four h at a time: the four float4 loads of a group go out together
    const int c4 = chunk / 4;
    if (pr != staged)
#pragma unroll 4
      for (int vi = threadIdx.x; vi < nt * c4; vi += DF_THREADS) {
        const int i = vi / c4, jj = ch * chunk + 4 * (vi - i * c4);
        const float* ab0 = a.ab + ((size_t)sh.act_q[ei][i] * 2) * 2 * dff + jj;
        const float4 a0 = __ldcg(reinterpret_cast<const float4*>(ab0));
        const float4 a1 = __ldcg(reinterpret_cast<const float4*>(ab0 + 2 * (size_t)dff));
        const float4 b0 = __ldcg(reinterpret_cast<const float4*>(ab0 + dff));
        const float4 b1 = __ldcg(reinterpret_cast<const float4*>(ab0 + 3 * (size_t)dff));
        const auto hval = [](float av, float bv) {
          return __bfloat162float(__float2bfloat16_rn(silu_f(av) * bv));
        };
        reinterpret_cast<float4*>(hs)[vi] =
            make_float4(hval(a0.x + a1.x, b0.x + b1.x), hval(a0.y + a1.y, b0.y + b1.y),
                        hval(a0.z + a1.z, b0.z + b1.z), hval(a0.w + a1.w, b0.w + b1.w));
      }
    staged = pr;
    __syncthreads();
    for (int cc = warp; cc < CB; cc += DF_WARPS) {
      const int c = fb * CB + cc;
      if (c >= d) break;
      const uint4* wd = reinterpret_cast<const uint4*>(a.w_down + ((size_t)e * d + c) * dff +
                                                       (size_t)ch * chunk);
      float o[MT];
#pragma unroll
      for (int i = 0; i < MT; ++i) o[i] = 0.f;
#pragma unroll 8
      for (int v = lane; v < chunk / 8; v += 32) {
        float wf[8];
        unpack8(ld_stream(wd + v), wf);
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          if (i < nt) {
            const float4* hr = reinterpret_cast<const float4*>(hs + (size_t)i * chunk) + 2 * v;
            const float4 h0 = hr[0], h1 = hr[1];
            const float hf8[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) o[i] = fmaf(wf[q], hf8[q], o[i]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        if (i < nt) {
          const float oi = warp_sum(o[i]);
          if (lane == 0) a.part[((size_t)(ei * MT + i) * nch + ch) * d + c] = oi;
        }
      }
    }
  }
  if (!grid_barrier(a.status + 2, a.status, 2 * gridDim.x + a.barrier_withheld,
                    a.barrier_limit_ns))
    return;

  // ---- 3. y[t][c] = sum over the token's terms (experts ascending, shared
  // last) of g * sum over chunks of part, in that order ---------------------
  for (int idx = blockIdx.x * DF_THREADS + threadIdx.x; idx < T * d;
       idx += gridDim.x * DF_THREADS) {
    const int t = idx / d, c = idx - t * d;
    float y = 0.f;
    for (int ei = 0; ei < n_act; ++ei) {
      const int nt = sh.act_nt[ei];
      for (int i = 0; i < nt; ++i) {
        if (sh.act_tok[ei][i] != t) continue;
        float o = 0.f;
        for (int ch = 0; ch < nch; ++ch)
          o += __ldcg(a.part + ((size_t)(ei * MT + i) * nch + ch) * d + c);
        y = fmaf(sh.act_g[ei][i], o, y);
      }
    }
    a.y[(size_t)t * d + c] = __float2bfloat16_rn(y);
  }
}

constexpr size_t DF_MAX_SMEM = 96 * 1024;  // x of all tokens (fp32)

// Grid-barrier settings of the next launches (moe_set_decode_barrier_test).
std::atomic<unsigned long long> g_barrier_limit_ns{kWaitLimitNs};
std::atomic<int> g_barrier_withheld{0};

int df_chunk(int d_ff) {
  for (int ch = 2048; ch >= 256; ch /= 2)
    if (d_ff % ch == 0) return ch;
  return 0;
}
int df_mt(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8; }

template <int MT>
cudaError_t launch_df(const DecodeArgs& a, size_t smem, cudaStream_t s) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(decode_layer_kernel<MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)DF_MAX_SMEM);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_layer_kernel<MT>,
                                                                DF_THREADS, smem);
  if (e != cudaSuccess) return e;
  per_sm = per_sm < 4 ? per_sm : 4;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(per_sm * num_sms());
  cfg.blockDim = dim3(DF_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel<MT>, a);
}


size_t df_smem(const moe_config& c) {
  return ((size_t)c.T * c.d_model + (size_t)df_mt(c.T) * df_chunk(c.d_ff)) * sizeof(float);
}
size_t df_ab_bytes(const moe_config& c) {
  return align_up((size_t)c.T * (c.top_k + c.n_shared) * 4 * c.d_ff * sizeof(float), 256);
}

}  // namespace

bool decode_fused_applies(const moe_config& c) {
  return c.dtype == MOE_BF16 && c.T >= 1 && c.T <= kDecodeFusedMaxT && c.n_experts <= DF_MAX_N &&
         c.d_model % 256 == 0 && df_chunk(c.d_ff) > 0 && df_smem(c) <= DF_MAX_SMEM;
}

size_t decode_fused_ws_bytes(const moe_config& c) {
  if (!decode_fused_applies(c)) return 0;
  const int act = (c.T * c.top_k < c.n_experts ? c.T * c.top_k : c.n_experts) + c.n_shared;
  return df_ab_bytes(c) +
         (size_t)act * df_mt(c.T) * (c.d_ff / df_chunk(c.d_ff)) * c.d_model * sizeof(float);
}

cudaError_t launch_decode_fused(const moe_config& c, const void* x, const void* w_router,
                                const float* logit_bias, const float* sel_bias,
                                const void* w_gate, const void* w_up, const void* w_down,
                                void* y, int32_t* topk_idx, float* topk_w, int32_t* counts,
                                float* prob_sum, void* ws, int* status, cudaStream_t s) {
  DecodeArgs a;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.w_router = static_cast<const __nv_bfloat16*>(w_router);
  a.logit_bias = logit_bias;
  a.sel_bias = sel_bias;
  a.w_gate = static_cast<const __nv_bfloat16*>(w_gate);
  a.w_up = static_cast<const __nv_bfloat16*>(w_up);
  a.w_down = static_cast<const __nv_bfloat16*>(w_down);
  a.y = static_cast<__nv_bfloat16*>(y);
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.counts = counts;
  a.prob_sum = prob_sum;
  a.ab = static_cast<float*>(ws);
  a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + df_ab_bytes(c));
  a.chunk = df_chunk(c.d_ff);
  a.status = status;
  a.T = c.T;
  a.d = c.d_model;
  a.N = c.n_experts;
  a.k = c.top_k;
  a.s = c.n_shared;
  a.d_ff = c.d_ff;
  a.gate_mode = c.gate_mode;
  a.capacity = c.capacity;
  a.barrier_limit_ns = g_barrier_limit_ns.load();
  a.barrier_withheld = g_barrier_withheld.load();
  const size_t smem = df_smem(c);
  ProfScope p(K_DECODE_FUSED, s);
  switch (df_mt(c.T)) {
    case 1: return launch_df<1>(a, smem, s);
    case 2: return launch_df<2>(a, smem, s);
    case 4: return launch_df<4>(a, smem, s);
    default: return launch_df<8>(a, smem, s);
  }
}

}  // namespace moe

extern "C" void moe_set_decode_barrier_test(int32_t withhold, uint64_t limit_ns) {
  if (withhold == 0 && limit_ns == 0) limit_ns = moe::kWaitLimitNs;
  moe::g_barrier_withheld.store(withhold != 0 ? 1 : 0);
  moe::g_barrier_limit_ns.store(limit_ns);
}
