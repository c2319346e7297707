// K1 for many experts (bf16, 32 < N <= 256) on the tensor cores.
//
// Same computation as router.cu ("Mixture of experts and speculative
// decoding", steps 1-3 and "Keeping the experts busy"; "MoE inference: the
// call centre with 256 specialists and 8 taking each call", "The bare
// mechanism"): scores r = x W_r^T (+ logit_bias), top-k on r + sel_bias
// with ties to the lower index, gate weights from the unbiased scores, and
// the per-expert counts and probability sums.
//
// With N = 256 and d_model = 7168 the scores are a 30 GFLOP dense
// contraction per 8192 tokens, so on CUDA cores they cost several times the
// rest of the routing. Here one CTA scores 128 tokens against all N experts
// with tcgen05.mma (bf16 operands, fp32 accumulation, a 128x256 TMEM
// accumulator fed by a 4-stage TMA ring). Sixteen epilogue warps then route
// the tile: four per TMEM lane group, each thread holding 64 of its token's
// scores in registers. A thread keeps the top 8 of its 64 keys as packed
// 64-bit words (order-preserving key bits above the complemented expert
// index, so one unsigned compare orders by key and then by lower index),
// sorting each group of 8 with a comparator network and merging it into the
// kept list with a bitonic half-cleaner, so selection is short dependency
// chains rather than one element at a time,
// and the four partial maxima, softmax sums and lists of a token meet in the
// shared memory the TMA ring no longer needs. One thread per token merges
// the four sorted lists into the top k. Probability sums over the tile's
// tokens use a butterfly reduce-scatter per 32 columns; every sum runs in a
// fixed order, so results are reproducible.
#include <float.h>

#include "device_util.cuh"
#include "moe_internal.h"
#include "sm103_ptx.cuh"
#include "router_finish.cuh"
#include "topk_select.cuh"
#include "sm103_wait.cuh"

namespace moe {
namespace {

constexpr int RT_BM = 128;                     // tokens per CTA = TMEM lanes
constexpr int RT_BK = 64;                      // K block (one 128-byte swizzle row)
constexpr int RT_STAGES = 4;
constexpr int RT_A_BYTES = RT_BM * RT_BK * 2;  // 16 KB of tokens
constexpr int RT_B_HALF = 128 * RT_BK * 2;     // 16 KB: 128 experts
constexpr int RT_STAGE_BYTES = RT_A_BYTES + 2 * RT_B_HALF;
constexpr size_t RT_SMEM = (size_t)RT_STAGES * RT_STAGE_BYTES + 1024;
constexpr int RT_EPI_WARPS = 16;               // 4 column quarters x 4 TMEM lane groups
constexpr int RT_EPI_THREADS = RT_EPI_WARPS * 32;
constexpr int RT_THREADS = 64 + RT_EPI_THREADS; // TMA warp, MMA warp, epilogue warps
constexpr int RT_QCOLS = 64;                    // scores per epilogue thread
constexpr int RT_LIST = 8;                      // kept per quarter (>= k; the networks are for 8)
constexpr int RT_RSTRIDE = 257;                 // padded row of the staged scores
constexpr int RT_LSTRIDE = 9;                   // padded quarter list
constexpr int RT_TMEM_COLS = 256;
constexpr int RT_NMAX = 256;
constexpr uint32_t RT_IDESC = ptx::idesc_bf16_f32(RT_BM, RT_NMAX);

struct RouterTcArgs {
  const float* logit_bias;
  const float* sel_bias;
  float* logits_out;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  float* partials;  // [gridDim.x][N] probability sums of each block
  int32_t* cpart;   // [gridDim.x][N] counts of each block
  float* prob_sum;
  int* done;        // finished-block counter for the final sum, zero at launch
  int* status;
  int T, d, N, k, gate_mode;
};

// Epilogue staging, placed over the TMA ring once the accumulator is final.
constexpr int RT_OFF_R = 0;                                            // float [128][257]
constexpr int RT_OFF_L = RT_OFF_R + RT_BM * RT_RSTRIDE * 4;            // u64 [4][128][9]
constexpr int RT_OFF_M = RT_OFF_L + 4 * RT_BM * RT_LSTRIDE * 8;        // float [4][128]
constexpr int RT_OFF_Z = RT_OFF_M + 4 * RT_BM * 4;                     // float [4][128]
static_assert(RT_OFF_Z + 4 * RT_BM * 4 <= RT_STAGES * RT_STAGE_BYTES, "staging fits the ring");

// Named barrier 1 over the epilogue warps only; the and-form returns whether
// every epilogue thread passed true.
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(RT_EPI_THREADS) : "memory");
}
__device__ __forceinline__ bool epi_all(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(RT_EPI_THREADS)
      : "memory");
  return r != 0;
}

struct __align__(8) RtState {
  uint64_t full[RT_STAGES];
  uint64_t empty[RT_STAGES];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(RT_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap map_x,
                     const __grid_constant__ CUtensorMap map_w, const RouterTcArgs a) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ RtState st;
  __shared__ float s_lb[RT_NMAX], s_sb[RT_NMAX];
  __shared__ float s_psum[4][RT_NMAX];  // [TMEM lane group][expert]
  __shared__ int s_cnt[RT_NMAX];

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
  const uint32_t ring = (ptx::smem_addr(dyn_smem) + 1023u) & ~1023u;
  const int KB = (a.d + RT_BK - 1) / RT_BK;
  const int N = a.N;
  const int row0 = blockIdx.x * RT_BM;

  if (threadIdx.x == 0) {
    for (int i = 0; i < RT_STAGES; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&st.acc_full), 1);
    ptx::mbar_init(ptx::smem_addr(&st.drain), 1);
    st.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&map_x);
    ptx::prefetch_tmap(&map_w);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&st.tmem_base), RT_TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = st.tmem_base;
  volatile int* abort_flag = &st.abort;
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < RT_NMAX; e += RT_THREADS) {
    s_lb[e] = (e < N && a.logit_bias) ? a.logit_bias[e] : 0.f;
    s_sb[e] = (e < N && a.sel_bias) ? a.sel_bias[e] : 0.f;
    s_cnt[e] = 0;
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_phase(ptx::smem_addr(&st.empty[stage]), phase ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = ptx::smem_addr(&st.full[stage]);
        const uint32_t dst = ring + stage * RT_STAGE_BYTES;
        ptx::mbar_arrive_expect_tx(fb, RT_STAGE_BYTES);
        ptx::tma_load_2d(dst, &map_x, fb, kb * RT_BK, row0);
        ptx::tma_load_2d(dst + RT_A_BYTES, &map_w, fb, kb * RT_BK, 0);
        ptx::tma_load_2d(dst + RT_A_BYTES + RT_B_HALF, &map_w, fb, kb * RT_BK, 128);
        ++issued;
        if (++stage == RT_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        const long long n = issued < RT_STAGES ? issued : RT_STAGES;
        for (long long i = 1; i <= n; ++i) {
          const long long q = issued - i;
          drain_wait(ptx::smem_addr(&st.full[q % RT_STAGES]), (uint32_t)((q / RT_STAGES) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_phase(ptx::smem_addr(&st.full[stage]), phase, abort_flag, a.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t src = ring + stage * RT_STAGE_BYTES;
        const uint64_t adesc = ptx::sdesc_k128(src);
        const uint64_t bdesc = ptx::sdesc_k128(src + RT_A_BYTES);
#pragma unroll
        for (int k = 0; k < RT_BK / 16; ++k)
          ptx::mma_bf16(tmem_base, adesc + 2 * k, bdesc + 2 * k, RT_IDESC, (kb | k) != 0);
        ptx::mma_commit(ptx::smem_addr(&st.empty[stage]));
        if (++stage == RT_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        ptx::mma_commit(ptx::smem_addr(&st.acc_full));
      } else {
        ptx::mma_commit(ptx::smem_addr(&st.drain));
        drain_wait(ptx::smem_addr(&st.drain), 0);
      }
    }
  } else {
    // ------------------------- epilogue: 64 scores of one token per thread --
    const int g = warp & 3;                 // TMEM lane group (warp rank mod 4)
    const int q = (warp - 2) >> 2;          // column quarter
    const int row = g * 32 + lane;
    const long long t = (long long)row0 + row;
    const bool valid = t < a.T;
    const int col0 = q * RT_QCOLS;
    const int nq = (N + RT_QCOLS - 1) / RT_QCOLS;
    const bool active = q < nq;             // warp-uniform
    uint8_t* stage = dyn_smem + (ring - ptx::smem_addr(dyn_smem));
    float* s_r = reinterpret_cast<float*>(stage + RT_OFF_R);
    uint64_t* s_l = reinterpret_cast<uint64_t*>(stage + RT_OFF_L);
    float* s_m = reinterpret_cast<float*>(stage + RT_OFF_M);
    float* s_z = reinterpret_cast<float*>(stage + RT_OFF_Z);
    const bool ok = epi_all(wait_phase(ptx::smem_addr(&st.acc_full), 0, abort_flag, a.status));
    if (ok) {
      ptx::tc_fence_after();
      float m = -FLT_MAX;
      if (active) {
        uint64_t L[RT_LIST];
#pragma unroll
        for (int s = 0; s < RT_LIST; ++s) L[s] = 0;  // below every packed key
        const uint32_t taddr = tmem_base + ((uint32_t)(g * 32) << 16) + (uint32_t)col0;
#pragma unroll 1
        for (int c = 0; c < RT_QCOLS / 32; ++c) {
          uint32_t u[32];
          ptx::tmem_ld32(taddr + 32 * c, u);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j0 = 0; j0 < 32; j0 += 8) {
            uint64_t cw[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int j = j0 + jj;
              const int e = col0 + 32 * c + j;
              const float r = a.logit_bias ? __fadd_rn(__uint_as_float(u[j]), s_lb[e])
                                           : __uint_as_float(u[j]);
              s_r[row * RT_RSTRIDE + e] = r;
              const bool in = e < N;
              if (in) m = fmaxf(m, r);
              cw[jj] = in ? pack_key(a.sel_bias ? __fadd_rn(r, s_sb[e]) : r, e) : 0ull;
            }
            sort8(cw);
            merge_top8(L, cw);
          }
        }
        uint64_t* lst = s_l + (size_t)(q * RT_BM + row) * RT_LSTRIDE;
#pragma unroll
        for (int s = 0; s < RT_LIST; ++s) lst[s] = L[s];
        s_m[q * RT_BM + row] = m;
      }
      epi_sync();
      // token max over the quarters, then exp and the quarter's partial sum
      float mt = s_m[row];
      for (int i = 1; i < nq; ++i) mt = fmaxf(mt, s_m[i * RT_BM + row]);
      float zq = 0.f;
      float v[RT_QCOLS];
      if (active) {
#pragma unroll
        for (int j = 0; j < RT_QCOLS; ++j) {
          v[j] = (col0 + j < N) ? expf(s_r[row * RT_RSTRIDE + col0 + j] - mt) : 0.f;
          zq += v[j];
        }
        s_z[q * RT_BM + row] = zq;
      }
      epi_sync();
      float z = s_z[row];
      for (int i = 1; i < nq; ++i) z += s_z[i * RT_BM + row];
      if (active) {
        // probabilities summed over the warp's 32 tokens, 32 columns at a time
#pragma unroll
        for (int c = 0; c < RT_QCOLS / 32; ++c) {
          float p[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) p[j] = valid ? v[c * 32 + j] / z : 0.f;
#pragma unroll
          for (int o = 16, W = 32; o > 0; o >>= 1, W >>= 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < W / 2; ++i) {
              const float send = upper ? p[i] : p[i + W / 2];
              const float keep = upper ? p[i + W / 2] : p[i];
              p[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
          }
          s_psum[g][col0 + c * 32 + lane] = p[0];
        }
      } else {
        s_psum[g][col0 + lane] = 0.f;
        s_psum[g][col0 + 32 + lane] = 0.f;
      }
      if (q == 0 && valid) {
        // merge the sorted quarter lists: the k largest words overall
        int h0 = 0, h1 = 0, h2 = 0, h3 = 0;
        int sel[kMaxTopK];
        float rsel[kMaxTopK];
#pragma unroll
        for (int s = 0; s < kMaxTopK; ++s) {
          if (s < a.k) {
            uint64_t best = 0;
            int bq = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int h = i == 0 ? h0 : i == 1 ? h1 : i == 2 ? h2 : h3;
              if (i < nq && h < RT_LIST) {
                const uint64_t w = s_l[(size_t)(i * RT_BM + row) * RT_LSTRIDE + h];
                if (w > best) {
                  best = w;
                  bq = i;
                }
              }
            }
            h0 += bq == 0;
            h1 += bq == 1;
            h2 += bq == 2;
            h3 += bq == 3;
            sel[s] = key_index(best);
            rsel[s] = s_r[row * RT_RSTRIDE + sel[s]];
          }
        }
        float gw[kMaxTopK];
        float zs = 0.f;
        if (a.gate_mode == MOE_GATE_TOPK_SOFTMAX) {
          float mk = rsel[0];
#pragma unroll
          for (int s = 1; s < kMaxTopK; ++s)
            if (s < a.k) mk = fmaxf(mk, rsel[s]);
#pragma unroll
          for (int s = 0; s < kMaxTopK; ++s)
            if (s < a.k) {
              gw[s] = expf(rsel[s] - mk);
              zs += gw[s];
            }
        } else {
#pragma unroll
          for (int s = 0; s < kMaxTopK; ++s)
            if (s < a.k) {
              gw[s] = expf(rsel[s] - mt) / z;
              zs += gw[s];
            }
        }
#pragma unroll
        for (int s = 0; s < kMaxTopK; ++s)
          if (s < a.k) {
            a.topk_idx[t * a.k + s] = sel[s];
            a.topk_w[t * a.k + s] = gw[s] / zs;
            atomicAdd(&s_cnt[sel[s]], 1);
          }
      }
      if (a.logits_out) {  // row-major copy of the staged scores, coalesced
        const int et = threadIdx.x - 64;
        for (int i = et; i < RT_BM * N; i += RT_EPI_THREADS) {
          const int rr = i / N, e = i - rr * N;
          if (row0 + rr < a.T) a.logits_out[(long long)(row0 + rr) * N + e] = s_r[rr * RT_RSTRIDE + e];
        }
      }
    } else {
      s_psum[g][col0 + lane] = 0.f;
      s_psum[g][col0 + 32 + lane] = 0.f;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  // block partial of the probability sums (lane groups in order) and counts
  for (int e = threadIdx.x; e < N; e += RT_THREADS) {
    a.partials[(size_t)blockIdx.x * N + e] = ((s_psum[0][e] + s_psum[1][e]) + s_psum[2][e]) + s_psum[3][e];
    a.cpart[(size_t)blockIdx.x * N + e] = s_cnt[e];
  }
  router_finish<RT_THREADS>(a.partials, a.cpart, N, (int)gridDim.x, a.prob_sum, a.counts, a.done);
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, RT_TMEM_COLS);
  }
}

}  // namespace

bool router_tc_applies(const moe_config& c, const float* logits_in) {
  return logits_in == nullptr && c.dtype == MOE_BF16 && c.n_experts > 32 &&
         c.n_experts <= RT_NMAX;
}

cudaError_t launch_router_tc(const moe_config& c, const void* x, const void* w_router,
                             const float* logit_bias, const float* sel_bias, float* logits_out,
                             int32_t* topk_idx, float* topk_w, int32_t* counts, float* prob_sum,
                             float* partials, int32_t* cpart, int* status, cudaStream_t s) {
  CUtensorMap mx, mw;
  if (!make_map(&mx, x, c.T, c.d_model) || !make_map(&mw, w_router, c.n_experts, c.d_model))
    return cudaErrorInvalidValue;
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)RT_SMEM);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int grid = ceil_div(c.T, RT_BM);
  RouterTcArgs a;
  a.logit_bias = logit_bias;
  a.sel_bias = sel_bias;
  a.logits_out = logits_out;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.counts = counts;
  a.partials = partials;
  a.cpart = cpart;
  a.prob_sum = prob_sum;
  a.done = status + 1;
  a.status = status;
  a.T = c.T;
  a.d = c.d_model;
  a.N = c.n_experts;
  a.k = c.top_k;
  a.gate_mode = c.gate_mode;
  ProfScope p(K_ROUTER, s);
  return launch_pdl(router_tc_kernel, dim3(grid), dim3(RT_THREADS), RT_SMEM, s, 1, mx, mw, a);
}

}  // namespace moe
