// K1 for 8 to 32 experts (bf16) on the tensor cores.
//
// Same computation as router.cu and router_tc.cu ("Mixture of experts and
// speculative decoding", steps 1-3 and "Keeping the experts busy"): scores
// r = x W_r^T (+ logit_bias), top-k on r + sel_bias with ties to the lower
// index, gate weights from the unbiased scores, per-expert counts and
// probability sums.
//
// With few experts the scores are a thin contraction (d_model x 32 per
// token) whose cost is reading x once, so the aim is to stream x at the
// memory rate with as many SMs as there are tokens to feed them. A CTA takes
// 128 tokens and one slice of d_model: a cluster of CS CTAs (1, 2 or 4)
// covers a token tile, each streaming its slice of x and of W_r through a
// 6-stage TMA ring into tcgen05.mma (M = 128 tokens, N = 32 experts, rows
// past N read as zero). The CTAs of ranks 1..CS-1 store their 128 x 32 fp32
// partial scores into the leader's shared memory; after the cluster barrier
// the leader adds them to its own in rank order (a fixed order, so results
// repeat bit for bit) and routes the tile: one epilogue thread per token
// selects the top k of its 32 packed keys with the comparator networks of
// topk_select.cuh, then the softmax, gates and per-expert sums.
#include <float.h>

#include "device_util.cuh"
#include "moe_internal.h"
#include "router_finish.cuh"
#include "sm103_ptx.cuh"
#include "sm103_wait.cuh"
#include "topk_select.cuh"

namespace moe {
namespace {

constexpr int R32_BM = 128;                        // tokens per tile = TMEM lanes
constexpr int R32_BN = 32;                         // experts (MMA N)
constexpr int R32_BK = 64;                         // K block (one 128-byte swizzle row)
constexpr int R32_STAGES = 6;
constexpr int R32_A_BYTES = R32_BM * R32_BK * 2;   // 16 KB of tokens
constexpr int R32_B_BYTES = R32_BN * R32_BK * 2;   // 4 KB of router rows
constexpr int R32_STAGE_BYTES = R32_A_BYTES + R32_B_BYTES;
constexpr int R32_MAX_CLUSTER = 4;
constexpr int R32_PSTRIDE = 36;                    // floats per row of a peer's partial
constexpr int R32_PART_BYTES = (R32_MAX_CLUSTER - 1) * R32_BM * R32_PSTRIDE * 4;
constexpr size_t R32_SMEM = (size_t)R32_STAGES * R32_STAGE_BYTES + R32_PART_BYTES + 1024;
constexpr int R32_THREADS = 192;                   // TMA warp, MMA warp, 4 epilogue warps
constexpr int R32_EPI_THREADS = 128;
constexpr int R32_TMEM_COLS = 32;
constexpr int R32_RSTRIDE = 33;                    // staged scores, floats per row
constexpr uint32_t R32_IDESC = ptx::idesc_bf16_f32(R32_BM, R32_BN);
static_assert(R32_BM * R32_RSTRIDE * 4 <= R32_STAGES * R32_STAGE_BYTES, "staging fits the ring");
static_assert(R32_STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte alignment of the swizzle");

struct Router32Args {
  const float* logit_bias;
  const float* sel_bias;
  float* logits_out;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  float* partials;  // [tiles][N] probability sums of each tile
  int32_t* cpart;   // [tiles][N] counts of each tile
  float* prob_sum;
  int* done;        // finished-tile counter for the final sum, zero at launch
  int* status;
  int T, d, N, k, gate_mode, cs;
};

struct __align__(8) R32State {
  uint64_t full[R32_STAGES];
  uint64_t empty[R32_STAGES];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  uint32_t peer_ok[R32_MAX_CLUSTER];  // leader: 1 when rank r's partial arrived intact
};

// Named barrier 1 over the 4 epilogue warps; returns whether all passed true.
__device__ __forceinline__ bool epi_all(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(R32_EPI_THREADS)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(R32_EPI_THREADS) : "memory");
}

__global__ void __launch_bounds__(R32_THREADS, 1)
    router_tc32_kernel(const __grid_constant__ CUtensorMap map_x,
                       const __grid_constant__ CUtensorMap map_w, const Router32Args a) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ R32State st;
  __shared__ float s_lb[R32_BN], s_sb[R32_BN];
  __shared__ float s_psum[4][R32_BN];  // [TMEM lane group][expert]
  __shared__ int s_cnt[R32_BN];

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
  const uint32_t base = (ptx::smem_addr(dyn_smem) + 1023u) & ~1023u;
  const uint32_t ring = base;
  const uint32_t part = base + R32_STAGES * R32_STAGE_BYTES;  // peers' partials (leader)
  uint8_t* base_ptr = dyn_smem + (base - ptx::smem_addr(dyn_smem));
  const int cs = a.cs;
  const int rank = cs > 1 ? (int)ptx::cluster_ctarank() : 0;
  const int tile = blockIdx.x / cs;
  const int row0 = tile * R32_BM;
  const int N = a.N;
  const int KB = (a.d + R32_BK - 1) / R32_BK;
  const int kb_lo = (int)((long long)KB * rank / cs);
  const int kb_hi = (int)((long long)KB * (rank + 1) / cs);

  if (threadIdx.x == 0) {
    for (int i = 0; i < R32_STAGES; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&st.acc_full), 1);
    ptx::mbar_init(ptx::smem_addr(&st.drain), 1);
    st.abort = 0;
    for (int i = 0; i < R32_MAX_CLUSTER; ++i) st.peer_ok[i] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&map_x);
    ptx::prefetch_tmap(&map_w);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&st.tmem_base), R32_TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = st.tmem_base;
  volatile int* abort_flag = &st.abort;
  // every CTA of the cluster has initialised its shared memory before any
  // peer writes into it
  if (cs > 1) ptx::cluster_sync();
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < R32_BN) {
    const int e = threadIdx.x;
    s_lb[e] = (e < N && a.logit_bias) ? a.logit_bias[e] : 0.f;
    s_sb[e] = (e < N && a.sel_bias) ? a.sel_bias[e] : 0.f;
    s_cnt[e] = 0;
  }
  __syncthreads();

  bool ok = false;  // epilogue warps: the accumulator of this CTA is final
  if (warp == 0) {
    // ------------------------------------------------------- TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool good = true;
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (!wait_phase(ptx::smem_addr(&st.empty[stage]), phase ^ 1u, abort_flag, a.status)) {
          good = false;
          break;
        }
        const uint32_t fb = ptx::smem_addr(&st.full[stage]);
        const uint32_t dst = ring + stage * R32_STAGE_BYTES;
        ptx::mbar_arrive_expect_tx(fb, R32_STAGE_BYTES);
        ptx::tma_load_2d(dst, &map_x, fb, kb * R32_BK, row0);
        ptx::tma_load_2d(dst + R32_A_BYTES, &map_w, fb, kb * R32_BK, 0);
        ++issued;
        if (++stage == R32_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!good) {
        const long long n = issued < R32_STAGES ? issued : R32_STAGES;
        for (long long i = 1; i <= n; ++i) {
          const long long q = issued - i;
          drain_wait(ptx::smem_addr(&st.full[q % R32_STAGES]), (uint32_t)((q / R32_STAGES) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool good = true;
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (!wait_phase(ptx::smem_addr(&st.full[stage]), phase, abort_flag, a.status)) {
          good = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t src = ring + stage * R32_STAGE_BYTES;
        const uint64_t adesc = ptx::sdesc_k128(src);
        const uint64_t bdesc = ptx::sdesc_k128(src + R32_A_BYTES);
#pragma unroll
        for (int k = 0; k < R32_BK / 16; ++k)
          ptx::mma_bf16(tmem_base, adesc + 2 * k, bdesc + 2 * k, R32_IDESC,
                        (kb != kb_lo) || (k != 0));
        ptx::mma_commit(ptx::smem_addr(&st.empty[stage]));
        if (++stage == R32_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (good) {
        ptx::mma_commit(ptx::smem_addr(&st.acc_full));
      } else {
        ptx::mma_commit(ptx::smem_addr(&st.drain));
        drain_wait(ptx::smem_addr(&st.drain), 0);
      }
    }
  }

  // ------------------------------- epilogue: this CTA's 128 x 32 partial --
  const int g = warp & 3;  // TMEM lane group (warp rank mod 4)
  const int row = g * 32 + lane;
  float v[R32_BN];
  if (warp >= 2) {
    ok = epi_all(wait_phase(ptx::smem_addr(&st.acc_full), 0, abort_flag, a.status));
    if (ok) {
      ptx::tc_fence_after();
      uint32_t u[32];
      ptx::tmem_ld32(tmem_base + ((uint32_t)(g * 32) << 16), u);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < R32_BN; ++c) v[c] = __uint_as_float(u[c]);
    }
    if (rank > 0) {  // hand the partial to the leader
      if (ok) {
        const uint32_t dst = ptx::mapa_shared(
            part + (uint32_t)(((rank - 1) * R32_BM + row) * R32_PSTRIDE * 4), 0);
#pragma unroll
        for (int c = 0; c < R32_BN; c += 4)
          ptx::st_cluster_v4(dst + c * 4, v[c], v[c + 1], v[c + 2], v[c + 3]);
      }
      if (threadIdx.x == 64)
        ptx::st_cluster_u32(ptx::mapa_shared(ptx::smem_addr(&st.peer_ok[rank]), 0), ok ? 1u : 2u);
    }
  }
  ptx::tc_fence_before();
  if (cs > 1) ptx::cluster_sync();  // peers' partials are in the leader's shared memory

  if (rank == 0) {
    if (warp >= 2) {
      bool all = ok;
      for (int r = 1; r < cs; ++r) all = all && st.peer_ok[r] == 1u;
      float* s_r = reinterpret_cast<float*>(base_ptr);  // the ring is idle now
      const long long t = (long long)row0 + row;
      const bool valid = t < a.T;
      if (all) {
        // partial scores of ranks 1..cs-1, added in rank order
        for (int r = 1; r < cs; ++r) {
          const float4* pr = reinterpret_cast<const float4*>(
              base_ptr + (part - base) + ((r - 1) * R32_BM + row) * R32_PSTRIDE * 4);
#pragma unroll
          for (int c = 0; c < R32_BN / 4; ++c) {
            const float4 q = pr[c];
            v[4 * c] += q.x;
            v[4 * c + 1] += q.y;
            v[4 * c + 2] += q.z;
            v[4 * c + 3] += q.w;
          }
        }
        float m = -FLT_MAX;
        uint64_t L[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) L[s] = 0;  // below every packed key
#pragma unroll
        for (int c0 = 0; c0 < R32_BN; c0 += 8) {
          uint64_t cw[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int e = c0 + j;
            const float r = a.logit_bias ? __fadd_rn(v[e], s_lb[e]) : v[e];
            v[e] = r;
            s_r[row * R32_RSTRIDE + e] = r;
            const bool in = e < N;
            if (in) m = fmaxf(m, r);
            cw[j] = in ? pack_key(a.sel_bias ? __fadd_rn(r, s_sb[e]) : r, e) : 0ull;
          }
          sort8(cw);
          merge_top8(L, cw);
        }
        float z = 0.f;
#pragma unroll
        for (int e = 0; e < R32_BN; ++e) {
          v[e] = e < N ? expf(v[e] - m) : 0.f;
          z += v[e];
        }
        // probabilities summed over the warp's 32 tokens: lane l ends with expert l
        float p[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) p[e] = valid ? v[e] / z : 0.f;
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
        s_psum[g][lane] = p[0];
        if (valid) {
          int sel[kMaxTopK];
          float rsel[kMaxTopK];
#pragma unroll
          for (int s = 0; s < kMaxTopK; ++s) {
            sel[s] = key_index(L[s]);
            rsel[s] = s < a.k ? s_r[row * R32_RSTRIDE + sel[s]] : 0.f;
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
                gw[s] = expf(rsel[s] - m) / z;
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
      } else {
        s_psum[g][lane] = 0.f;
      }
      if (a.logits_out && __shfl_sync(0xffffffffu, (int)all, 0)) {
        epi_sync();  // every row of s_r is written
        const int et = threadIdx.x - 64;
        for (int i = et; i < R32_BM * N; i += R32_EPI_THREADS) {
          const int rr = i / N, e = i - rr * N;
          if (row0 + rr < a.T)
            a.logits_out[(long long)(row0 + rr) * N + e] = s_r[rr * R32_RSTRIDE + e];
        }
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += R32_THREADS) {
      a.partials[(size_t)tile * N + e] =
          ((s_psum[0][e] + s_psum[1][e]) + s_psum[2][e]) + s_psum[3][e];
      a.cpart[(size_t)tile * N + e] = s_cnt[e];
    }
    router_finish<R32_THREADS>(a.partials, a.cpart, N, (int)gridDim.x / cs, a.prob_sum, a.counts,
                               a.done);
  }
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, R32_TMEM_COLS);
  }
}

}  // namespace

// Cluster size: the largest of 4, 2, 1 that keeps the grid within one CTA
// per SM and gives every CTA at least two K blocks.
int router_tc32_cluster(const moe_config& c) {
  const int tiles = ceil_div(c.T, R32_BM);
  const int KB = ceil_div(c.d_model, R32_BK);
  int cs = R32_MAX_CLUSTER;
  const int sms = num_sms();
  while (cs > 1 && (tiles * cs > sms || KB < 2 * cs)) cs /= 2;
  return cs;
}

cudaError_t launch_router_tc32(const moe_config& c, const void* x, const void* w_router,
                               const float* logit_bias, const float* sel_bias, float* logits_out,
                               int32_t* topk_idx, float* topk_w, int32_t* counts, float* prob_sum,
                               float* partials, int32_t* cpart, int* status, cudaStream_t s) {
  CUtensorMap mx, mw;
  if (!make_map(&mx, x, c.T, c.d_model) || !make_map(&mw, w_router, c.n_experts, c.d_model, R32_BN))
    return cudaErrorInvalidValue;
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(router_tc32_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)R32_SMEM);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  Router32Args a;
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
  a.cs = router_tc32_cluster(c);
  const int grid = ceil_div(c.T, R32_BM) * a.cs;
  ProfScope p(K_ROUTER, s);
  return launch_pdl(router_tc32_kernel, dim3(grid), dim3(R32_THREADS), R32_SMEM, s, a.cs, mx, mw,
                    a);
}

}  // namespace moe
