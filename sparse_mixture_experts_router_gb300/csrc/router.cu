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
// Scores are fp32 sums, in one of these kernels (router_tc.cu has the one
// for bf16 with 32 < N <= 256):
//  - bf16 with up to 32 experts and T >= 256: mma.sync tensor-core tiles of
//    16 tokens (router_mma_kernel, below);
//  - fp32, or bf16 below 256 tokens, with up to 32 experts: the 8 warps of a
//    block split d_model and
//    score a group of 2-8 tokens against all N experts together on the CUDA
//    cores, reading x once from HBM and W_r from L2 with 16-byte loads;
//  - fp32 with more experts, or scores given: a register-tiled block GEMM.
//    A block scores 64 tokens against all N (<= 256) experts; each thread
//    owns a TM x 8 tile (tokens x consecutive experts); 32-wide K slices of
//    x and W_r are staged transposed in shared memory with the next slice
//    prefetched into registers. Bound by fp32 FMA throughput.
//  - decode-sized layers: decode_front_kernel (routing, permutation and
//    gather in one block).
// All hand every token to the same warp-level selection: lane l holds the
// scores of experts l, l+32, ...; k rounds of a (key desc, index asc) warp
// argmax choose the top k (equal keys go to the lower index); the gates and
// the full softmax come from the unbiased scores. Counts use shared-memory
// integer atomics (order-free, exact); the per-expert probability sums are
// added in a fixed order (tokens of a warp, warps of a block, then blocks in
// a separate pass), so the results are bitwise reproducible.
#include <float.h>

#include "device_util.cuh"
#include "moe_internal.h"
#include "router_finish.cuh"
#include "seg_table.cuh"
#include "sm103_ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileTokens = 64;              // tokens per block, tiled kernel
constexpr int kKC = 32;                      // K slice of the tiled kernel
constexpr int kSmallMaxBlocks = 4 * 152;     // few-expert kernel: grid-stride beyond this
constexpr int kSmallTargetWarps = 2 * 152 * kWarps;  // few-expert kernel: warps to keep busy

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
  float* partials;  // [gridDim.x][N] probability sums of each block
  int32_t* cpart;   // [gridDim.x][N] counts of each block
  int* status;
  // The last block to finish sums the partials into prob_sum and counts;
  // `done` counts finished blocks and is zero at launch.
  float* prob_sum;
  int* done;
  int T, d, N, k, gate_mode;
};

// Eight (bf16) or four (fp32) elements of a 16-byte vector as fp32.
template <typename TX> struct V16;
template <> struct V16<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void cvt(const uint4& q, float* f) {
    bf16x2_to_f32(q.x, f[0], f[1]);
    bf16x2_to_f32(q.y, f[2], f[3]);
    bf16x2_to_f32(q.z, f[4], f[5]);
    bf16x2_to_f32(q.w, f[6], f[7]);
  }
};
template <> struct V16<float> {
  static constexpr int n = 4;
  __device__ static void cvt(const uint4& q, float* f) {
    f[0] = __uint_as_float(q.x); f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z); f[3] = __uint_as_float(q.w);
  }
};

// (key, index) order of the top-k: larger key first, then lower index.
__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Selection, gates and statistics of one token, by one full warp. r[j] is
// the unbiased score of expert lane + 32*j (any value where that index is
// >= N). Adds softmax(r) to psum and the kept experts to bcount; lane 0
// writes topk_idx / topk_w.
template <int EJ>
__device__ __forceinline__ void select_token(const float (&r)[EJ], int lane, long long t,
                                             const RouterArgs& a, float (&psum)[EJ],
                                             int* bcount, int* sel_sm = nullptr) {
  const int N = a.N;
  float key[EJ];
#pragma unroll
  for (int j = 0; j < EJ; ++j) {
    const int e = lane + 32 * j;
    key[j] = (e < N && a.sel_bias) ? __fadd_rn(r[j], a.sel_bias[e]) : r[j];
    if (key[j] != key[j]) key[j] = -INFINITY;  // a NaN key ranks below every number
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
  for (int j = 0; j < EJ; ++j) psum[j] += p[j] / z;

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
    float mine = 0.f;
#pragma unroll
    for (int j = 0; j < EJ; ++j)
      if (j == (bi >> 5)) mine = r[j];
    rsel[s] = __shfl_sync(0xffffffffu, mine, bi & 31);
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
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
      a.topk_idx[t * a.k + s] = sel[s];
      a.topk_w[t * a.k + s] = g[s];
      atomicAdd(&bcount[sel[s]], 1);
      if (sel_sm) sel_sm[t * a.k + s] = sel[s];  // also in shared memory (decode_front_kernel)
    }
  }
}

// Per-block probability partial (warps summed in order) and counts, then the
// last block's fixed-order total.
template <int EJ>
__device__ __forceinline__ void finish_block(const float (&psum)[EJ], float* wprob, int* bcount,
                                             const RouterArgs& a) {
  const int NP = 32 * EJ;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
#pragma unroll
  for (int j = 0; j < EJ; ++j) wprob[warp * NP + lane + 32 * j] = psum[j];
  __syncthreads();
  for (int e = threadIdx.x; e < a.N; e += kThreads) {
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += wprob[w * NP + e];
    a.partials[(size_t)blockIdx.x * a.N + e] = s;
    a.cpart[(size_t)blockIdx.x * a.N + e] = bcount[e];
  }
  router_finish<kThreads>(a.partials, a.cpart, a.N, (int)gridDim.x, a.prob_sum, a.counts, a.done);
}

// Reduce-scatter of a warp's NV (16 or 32) partial sums: after the step
// with offset o a lane keeps half of its values (the upper half when
// lane & o), each summed with its partner's; lanes that end up holding the
// same value then add their halves. Afterwards value i (summed over the
// warp) is held by lanes i * 32/NV ... in v[0].
template <int NV>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int lane) {
#pragma unroll
  for (int o = 16, L = NV; o > 0; o >>= 1, L >>= 1) {
    if (L > 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < L / 2; ++i) {
        const float send = upper ? v[i] : v[i + L / 2];
        const float keep = upper ? v[i + L / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
}

// Scores of a group of TPW tokens t0.. after reduce_scatter (value q*NP + e
// is token t0+q's score for expert e): one shuffle hands expert e's score to
// lane e, the logit bias is added (and the score written when asked), and
// the warp selects for each token in turn.
template <int NP, int TPW>
__device__ __forceinline__ void select_group(float v0, int lane, long long t0, const RouterArgs& a,
                                             float (&psum)[1], int* bcount) {
  constexpr int NV = NP * TPW;
  constexpr int SPREAD = 32 / NV;
  const int N = a.N;
#pragma unroll
  for (int q = 0; q < TPW; ++q) {
    const long long t = t0 + q;
    const int src = ((q * NP + (lane < NP ? lane : 0)) % NV) * SPREAD;
    const float sum = __shfl_sync(0xffffffffu, v0, src);
    if (t < a.T) {  // warp-uniform
      float r[1] = {0.f};
      if (lane < N) {
        r[0] = a.logit_bias ? __fadd_rn(sum, a.logit_bias[lane]) : sum;
        if (a.logits_out) a.logits_out[t * N + lane] = r[0];
      }
      select_token<1>(r, lane, t, a, psum, bcount);
    }
  }
}

// ---------------------------------------------------------------------------
// Few experts (N <= 32): a group of TPW tokens is scored by `wsplit` warps
// of one block (1 for large batches, up to 8 when there are few tokens, so
// a decode step still spreads its row over a whole block). A warp takes
// every (32*wsplit)-th 16-byte vector of the group's rows, starting at its
// own 32-vector slice, and keeps NV = NP*TPW partial dot products (NP = N
// rounded up to 8, 16 or 32); x vectors are loaded 32/NP per token at a
// time, all in flight before the first is used, and the router rows come
// through L1 (NP of them per x vector, which is where the larger NP find
// their memory parallelism). A butterfly reduce-scatter then leaves lane
// (i * 32/NV) with value i summed over the warp; the group's warps add
// their sums in warp order through shared memory, one shuffle hands expert
// e's score of token q to lane e of the group's first warp, and that warp
// selects for each of the group's tokens in turn.
template <typename TX, int NP, int TPW>
__global__ void __launch_bounds__(kThreads, 2) router_small_kernel(const RouterArgs a, int wsplit) {
  constexpr int EPV = V16<TX>::n;
  constexpr int NV = NP * TPW;
  static_assert(NV == 16 || NV == 32, "reduce-scatter below assumes 16 or 32 values");
  constexpr int kSmallBatch = 32 / NP;  // x vectors per token in flight: 4, 2 or 1
  __shared__ float wprob[kWarps * 32];
  __shared__ int bcount[32];
  __shared__ float red[kWarps][32];
  const int N = a.N;
  const int vec = a.d / EPV;  // 16-byte vectors per row
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int gpb = kWarps / wsplit;  // token groups per block and round
  const int wi = warp % wsplit;     // this warp's slice of the group's vectors
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < 32) bcount[threadIdx.x] = 0;
  __syncthreads();
  const uint4* x = static_cast<const uint4*>(a.x);
  const uint4* w = static_cast<const uint4*>(a.w);
  float psum[1] = {0.f};
  const long long groups = (a.T + TPW - 1) / TPW;
  const long long rounds = (groups + gpb - 1) / gpb;
  for (long long rd = blockIdx.x; rd < rounds; rd += gridDim.x) {  // block-uniform
    const long long g = rd * gpb + warp / wsplit;
    const long long t0 = g * TPW;
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = 0.f;
    const uint4* xr[TPW];
#pragma unroll
    for (int q = 0; q < TPW; ++q) xr[q] = (t0 + q < a.T) ? x + (t0 + q) * vec : nullptr;
    const int stride = 32 * wsplit;
    for (int vb = 32 * wi + lane; vb < vec; vb += stride * kSmallBatch) {
      uint4 xq[kSmallBatch][TPW];  // a batch of x vectors in flight before any is used
#pragma unroll
      for (int b = 0; b < kSmallBatch; ++b)
#pragma unroll
        for (int q = 0; q < TPW; ++q) {
          const int vv = vb + stride * b;
          xq[b][q] = (xr[q] && vv < vec) ? __ldg(xr[q] + vv) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
      for (int b = 0; b < kSmallBatch; ++b) {
        const int vv = vb + stride * b;
        if (vv >= vec) break;
        float xf[TPW][EPV];
#pragma unroll
        for (int q = 0; q < TPW; ++q) V16<TX>::cvt(xq[b][q], xf[q]);
#pragma unroll
        for (int e = 0; e < NP; ++e) {
          const uint4 wq = (e < N) ? __ldg(w + (size_t)e * vec + vv) : make_uint4(0, 0, 0, 0);
          float wf[EPV];
          V16<TX>::cvt(wq, wf);
#pragma unroll
          for (int q = 0; q < TPW; ++q)
#pragma unroll
            for (int i = 0; i < EPV; ++i) v[q * NP + e] = fmaf(xf[q][i], wf[i], v[q * NP + e]);
        }
      }
    }
    reduce_scatter<NV>(v, lane);
    if (wsplit > 1) {  // the group's warps, added in warp order
      red[warp][lane] = v[0];
      __syncthreads();
      if (wi == 0)
        for (int j = 1; j < wsplit; ++j) v[0] += red[warp + j][lane];
      __syncthreads();
    }
    if (wi == 0) select_group<NP, TPW>(v[0], lane, t0, a, psum, bcount);
  }
  __syncthreads();
  finish_block<1>(psum, wprob, bcount, a);
}

// One m16n8k16 tensor-core MMA, bf16 operands and fp32 accumulation (the
// fragments as mma.sync defines them: lane (g, c) = (lane / 4, lane % 4)
// holds A rows g and g + 8, k = 2c, 2c + 1, 2c + 8, 2c + 9, B column g at
// the same k, and D rows g and g + 8, columns 2c and 2c + 1).
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// Decode-sized batches (bf16, T <= 64, N <= 32): the routing, the
// permutation (with the capacity cut), the grouped GEMM's segment table and
// the row gather in one block, in place of the router, the permutation and
// the gather launches and the status reset (the block clears the call's
// status words itself once the grids before it have finished). At these
// sizes each of those launches was latency rather than work: the router's
// blocks met in a cross-block sum, the permutation and the gather each ran
// on one block. Results are those of the separate kernels' definitions:
// the same selection (select_token), probability sums in a fixed order
// (tokens of a warp, then warps), counts by integer atomics, and each
// expert's pairs ranked in ascending pair order.
constexpr int kFrontThreads = 512;
constexpr int kFrontWarps = kFrontThreads / 32;
constexpr int kFrontMaxT = 16;
constexpr size_t kFrontMaxRouterBytes = 128 * 1024;  // router rows staged in shared memory
constexpr int front_np(int N) { return N <= 8 ? 8 : N <= 16 ? 16 : 32; }
constexpr int kFrontMaxPairs = kFrontMaxT * kMaxTopK;

struct FrontArgs {
  RouterArgs r;
  int capacity, n_shared, tile_m;
  int32_t* offsets;
  int32_t* sorted_pair;
  int32_t* inv_pos;
  int32_t* seg;
  uint4* x_perm;  // null: the caller gathers
};

template <int NP>
__global__ void __launch_bounds__(kFrontThreads, 1) decode_front_kernel(const FrontArgs f) {
  extern __shared__ uint4 w_sm[];            // [NP][vec] router rows, rows past N zero
  __shared__ float sc[kFrontMaxT][32];       // scores
  __shared__ float part[kFrontWarps][16][NP + 1];  // warp partial score tiles
  __shared__ float wprob[kFrontWarps][32];   // per-warp probability sums
  __shared__ int bcount[32];
  __shared__ int sidx[kFrontMaxPairs];       // expert of each pair
  __shared__ int srow[kFrontMaxPairs];       // pair of each row
  __shared__ int soff[33];
  __shared__ int sscr[32 + kMaxShared + 1];
  const RouterArgs& a = f.r;
  const int N = a.N, k = a.k, T = a.T, P = T * k;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int vec = a.d / 8;
  {  // the router rows into shared memory, all copies in flight at once; they
     // are inputs of the call, not results of the grid before it, so the
     // copies start before the wait on that grid
    const uint4* w = static_cast<const uint4*>(a.w);
    const int nw = N * vec;
    for (int i = threadIdx.x; i < NP * vec; i += kFrontThreads) {
      const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(w_sm + i));
      const uint4* src = w + (i < nw ? i : 0);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                   "r"(i < nw ? 16 : 0)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < 3) a.status[threadIdx.x] = 0;
  if (threadIdx.x < 32) bcount[threadIdx.x] = 0;
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  const uint4* x = static_cast<const uint4*>(a.x);
  // 1. scores on the tensor cores: the T <= 16 tokens are one m16 tile (rows
  // past T zero); the warps split d_model into 32-element chunks, lane
  // (g, c) feeding elements 8c .. 8c + 7 of a chunk of x rows g and g + 8 and
  // of router row g of each 8-expert group to two MMAs (both operands see the
  // same permutation of the chunk's k); the warps' partial tiles meet in
  // warp order
  {
    constexpr int NT = NP / 8;
    constexpr int U = 4;
    const int g = lane / 4, c = lane % 4;
    const int chunks = (vec + 3) / 4;
    const int per_warp = (chunks + kFrontWarps - 1) / kFrontWarps;
    const int ch_end = min(chunks, (warp + 1) * per_warp);
    const uint4 zero = make_uint4(0, 0, 0, 0);
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[j][q] = 0.f;
    for (int ch0 = warp * per_warp; ch0 < ch_end; ch0 += U) {
      uint4 xa[U], xb[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vi = (ch0 + u) * 4 + c;
        const bool in = ch0 + u < ch_end && vi < vec;
        xa[u] = (in && g < T) ? __ldg(x + (size_t)g * vec + vi) : zero;
        xb[u] = (in && g + 8 < T) ? __ldg(x + (size_t)(g + 8) * vec + vi) : zero;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vi = (ch0 + u) * 4 + c;
        const bool in = ch0 + u < ch_end && vi < vec;
#pragma unroll
        for (int j = 0; j < NT; ++j) {  // router rows past N are zero in w_sm
          const uint4 wv = in ? w_sm[(8 * j + g) * vec + vi] : zero;
          mma_16816_bf16(acc[j], xa[u].x, xb[u].x, xa[u].y, xb[u].y, wv.x, wv.y);
          mma_16816_bf16(acc[j], xa[u].z, xb[u].z, xa[u].w, xb[u].w, wv.z, wv.w);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      part[warp][g][8 * j + 2 * c] = acc[j][0];
      part[warp][g][8 * j + 2 * c + 1] = acc[j][1];
      part[warp][g + 8][8 * j + 2 * c] = acc[j][2];
      part[warp][g + 8][8 * j + 2 * c + 1] = acc[j][3];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < T * N; i += kFrontThreads) {
      const int r = i / N, e = i - r * N;
      float sum = 0.f;
      for (int ww = 0; ww < kFrontWarps; ++ww) sum += part[ww][r][e];
      sc[r][e] = a.logit_bias ? __fadd_rn(sum, a.logit_bias[e]) : sum;
    }
    __syncthreads();
  }

  // 2. selection, gates and statistics: a warp per token
  float psum[1] = {0.f};
  for (int t = warp; t < T; t += kFrontWarps) {
    float r[1] = {lane < N ? sc[t][lane] : 0.f};
    if (a.logits_out && lane < N) a.logits_out[(size_t)t * N + lane] = r[0];
    select_token<1>(r, lane, t, a, psum, bcount, sidx);
  }
  wprob[warp][lane] = psum[0];
  __syncthreads();
  if (threadIdx.x < N) {
    float s = 0.f;
    for (int j = 0; j < kFrontWarps; ++j) s += wprob[j][threadIdx.x];
    a.prob_sum[threadIdx.x] = s;
    a.counts[threadIdx.x] = bcount[threadIdx.x];
  }
  // 3. permutation: kept rows per expert, their offsets, each pair's rank
  if (warp == 0) {
    const int kept = lane < N ? (f.capacity > 0 ? min(bcount[lane], f.capacity) : bcount[lane]) : 0;
    if (lane < N) soff[lane] = kept;
    __syncwarp();
    const int total = warp_exclusive_scan(soff, N, lane);
    if (lane == 0) soff[N] = total;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += kFrontThreads) {
    const int e = sidx[p];
    int pos = -1;
    if (e >= 0) {
      int rank = 0;
      for (int q = 0; q < p; ++q) rank += sidx[q] == e;
      if (f.capacity == 0 || rank < f.capacity) pos = soff[e] + rank;
    }
    f.inv_pos[p] = pos;
    if (pos >= 0) {
      f.sorted_pair[pos] = p;
      srow[pos] = p;
    }
  }
  for (int e = threadIdx.x; e <= N; e += kFrontThreads) f.offsets[e] = soff[e];
  __syncthreads();
  if (f.seg != nullptr) write_seg_table(soff, N, f.n_shared, T, P, f.tile_m, f.seg, sscr);
  // 4. the gather: row r of x_perm is x[srow[r] / k]
  if (f.x_perm != nullptr) {  // (x is in L2 from the scores) 8 loads a thread in flight
    constexpr int kGB = 8;
    const int total = soff[N] * vec;
    for (int i0 = threadIdx.x; i0 < total; i0 += kFrontThreads * kGB) {
      uint4 v[kGB];
#pragma unroll
      for (int b = 0; b < kGB; ++b) {
        const int i = i0 + b * kFrontThreads;
        if (i < total) {
          const int row = i / vec, c = i - row * vec;
          v[b] = __ldg(x + (size_t)(srow[row] / k) * vec + c);
        }
      }
#pragma unroll
      for (int b = 0; b < kGB; ++b) {
        const int i = i0 + b * kFrontThreads;
        if (i < total) f.x_perm[i] = v[b];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Few experts with bf16 tokens (N <= 32): the scores on the tensor cores,
// with mma.sync m16n8k16 (bf16 operands, fp32 accumulation). On the CUDA
// cores each bf16 product also costs a conversion of the router weight,
// which kept the streaming kernel issue-bound at about a fifth of HBM; here
// one instruction covers 16 tokens x 8 experts x 16 elements of d_model.
//
// A block scores a tile of 16 tokens; its 8 warps split d_model into
// 32-element chunks (warp w takes the w-th eighth of them). In a chunk, lane
// (g, c) = (lane / 4, lane % 4) loads one 16-byte vector, elements
// 8c .. 8c + 7, of x rows g and g + 8 and of router row g of each
// 8-expert group, and feeds it to two MMAs: elements 0-3 as the fragment's
// k = 2c, 2c + 1, 2c + 8, 2c + 9 of the first, elements 4-7 as those of the
// second. Both operands see the same permutation of the chunk's 32 k, so the
// products summed are exactly the dot product's. The warps' 16 x NP partial
// tiles meet in shared memory in warp order; each warp then selects for two
// of the tile's tokens (select_token), and the blocks' statistics meet as in
// the other kernels. Blocks walk the token tiles grid-stride.
// Measured on one GB300 (kernel time, L2 flushed): 21 us for the Mixtral
// prefill shape (T = 4096, N = 8, d = 4096) against 27 us for the CUDA-core
// streaming kernel this replaced, 25 against 101 us at N = 32, 23 against
// 35 us at N = 16, d = 7168. A variant that staged each thread's loads in a
// private cp.async ring (about 170 KB in flight per SM, no registers held)
// was slower (23, 35 and 21 us): the cost is the per-tile selection and the
// tiles' latency, not the bytes in flight.

constexpr int kMmaTile = 16;  // tokens a block tile

template <int NP>
__global__ void __launch_bounds__(kThreads, 2) router_mma_kernel(const RouterArgs a) {
  constexpr int NT = NP / 8;             // 8-expert column tiles
  constexpr int U = NT == 1 ? 8 : NT == 2 ? 4 : 2;  // chunks whose loads are in flight together
  __shared__ float part[kWarps][kMmaTile][NP + 1];  // warp partial tiles
  __shared__ float sc[kMmaTile][32];                // the tile's scores
  __shared__ float wprob[kWarps * 32];
  __shared__ int bcount[32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, c = lane % 4;
  const int N = a.N;
  const int vec = a.d / 8;               // 16-byte vectors a row
  const int chunks = (vec + 3) / 4;      // 32-element chunks
  // the warp's chunks are consecutive, so its U loads of a row cover
  // 64 U contiguous bytes
  const int per_warp = (chunks + kWarps - 1) / kWarps;
  const int ch_begin = warp * per_warp, ch_end = min(chunks, ch_begin + per_warp);
  const uint4* x = static_cast<const uint4*>(a.x);
  const uint4* w = static_cast<const uint4*>(a.w);
  const uint4 zero = make_uint4(0, 0, 0, 0);
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < 32) bcount[threadIdx.x] = 0;
  float psum[1] = {0.f};
  const long long tiles = (a.T + kMmaTile - 1) / kMmaTile;
  for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {  // block-uniform
    const long long t0 = tile * kMmaTile;
    const long long r0 = t0 + g, r1 = t0 + g + 8;
    const bool in0 = r0 < a.T, in1 = r1 < a.T;
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[j][q] = 0.f;
    for (int ch0 = ch_begin; ch0 < ch_end; ch0 += U) {
      uint4 xa[U], xb[U], wv[U][NT];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vi = (ch0 + u) * 4 + c;  // this lane's vector of the chunk
        const bool in = ch0 + u < ch_end && vi < vec;
        xa[u] = (in && in0) ? __ldg(x + r0 * vec + vi) : zero;
        xb[u] = (in && in1) ? __ldg(x + r1 * vec + vi) : zero;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int e = 8 * j + g;
          wv[u][j] = (in && e < N) ? __ldg(w + (size_t)e * vec + vi) : zero;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          mma_16816_bf16(acc[j], xa[u].x, xb[u].x, xa[u].y, xb[u].y, wv[u][j].x, wv[u][j].y);
          mma_16816_bf16(acc[j], xa[u].z, xb[u].z, xa[u].w, xb[u].w, wv[u][j].z, wv[u][j].w);
        }
    }
    // accumulator (row g or g + 8, expert 8j + 2c + {0, 1})
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      part[warp][g][8 * j + 2 * c] = acc[j][0];
      part[warp][g][8 * j + 2 * c + 1] = acc[j][1];
      part[warp][g + 8][8 * j + 2 * c] = acc[j][2];
      part[warp][g + 8][8 * j + 2 * c + 1] = acc[j][3];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kMmaTile * N; i += kThreads) {
      const int r = i / N, e = i - r * N;
      float sum = 0.f;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) sum += part[ww][r][e];
      sc[r][e] = a.logit_bias ? __fadd_rn(sum, a.logit_bias[e]) : sum;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kMmaTile / kWarps; ++q) {
      const int tl = warp * (kMmaTile / kWarps) + q;
      const long long t = t0 + tl;
      if (t < a.T) {  // warp-uniform
        float r[1] = {lane < N ? sc[tl][lane] : 0.f};
        if (a.logits_out && lane < N) a.logits_out[t * N + lane] = r[0];
        select_token<1>(r, lane, t, a, psum, bcount);
      }
    }
    __syncthreads();  // part and sc are rewritten by the next tile
  }
  finish_block<1>(psum, wprob, bcount, a);
}

// ---------------------------------------------------------------------------
// Many experts: 64 tokens x (32*EJ) experts per block, register tiles.
template <typename TX, int EJ>
__global__ void __launch_bounds__(kThreads) router_tiled_kernel(const RouterArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int BN = 32 * EJ;            // padded experts
  constexpr int BM = kTileTokens;        // 64 tokens
  constexpr int NEG = BN / 8;            // expert groups of 8
  constexpr int TM = BN / 32;            // tokens per thread (BM = 256/NEG * TM)
  constexpr int XV = (BM * kKC) / (8 * kThreads);   // 8-element vectors of x per thread (1)
  constexpr int WVEC = BN * kKC / 8;                  // 8-element vectors of a W slice
  constexpr int WV = (WVEC + kThreads - 1) / kThreads;
  constexpr int REGION = (BM * BN > kKC * (BM + BN)) ? BM * BN : kKC * (BM + BN);
  static_assert(BM == (kThreads / NEG) * TM, "tile shape");
  static_assert(XV == 1, "x slice: one 8-element vector per thread");

  float* xs = reinterpret_cast<float*>(smem_raw);          // [kKC][BM]
  float* wsm = xs + kKC * BM;                              // [kKC][BN]
  float* lt = reinterpret_cast<float*>(smem_raw);          // [BM][BN], reuses xs/wsm
  float* wprob = lt + REGION;                              // [kWarps][BN]
  int* bcount = reinterpret_cast<int*>(wprob + kWarps * BN);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int eg = tid % NEG, tg = tid / NEG;
  const long long t0 = (long long)blockIdx.x * BM;
  const int N = a.N;
  pdl_wait();
  pdl_trigger();
  for (int e = tid; e < BN; e += kThreads) bcount[e] = 0;

  if (a.logits_in == nullptr) {
    const TX* x = static_cast<const TX*>(a.x);
    const TX* w = static_cast<const TX*>(a.w);
    // global -> register mapping of one K slice
    const int xt = tid % BM, xk = (tid / BM) * 8;
    int we[WV], wk[WV];
    bool wact[WV];
#pragma unroll
    for (int i = 0; i < WV; ++i) {
      const int idx = tid + kThreads * i;
      wact[i] = idx < WVEC;
      we[i] = idx % BN;
      wk[i] = (idx / BN) * 8;
    }
    float xr[8], wr[WV][8];
    auto load_slice = [&](int k0) {
      const long long t = t0 + xt;
      float f[8];
      if (t < a.T && k0 + xk < a.d) {
        if (sizeof(TX) == 2) {
          V16<TX>::cvt(__ldg(reinterpret_cast<const uint4*>(x + t * a.d + k0 + xk)), f);
        } else {
          V16<TX>::cvt(__ldg(reinterpret_cast<const uint4*>(x + t * a.d + k0 + xk)), f);
          V16<TX>::cvt(__ldg(reinterpret_cast<const uint4*>(x + t * a.d + k0 + xk + 4)), f + 4);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) f[q] = 0.f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) xr[q] = f[q];
#pragma unroll
      for (int i = 0; i < WV; ++i) {
        if (wact[i] && we[i] < N && k0 + wk[i] < a.d) {
          const TX* src = w + (size_t)we[i] * a.d + k0 + wk[i];
          if (sizeof(TX) == 2) {
            V16<TX>::cvt(__ldg(reinterpret_cast<const uint4*>(src)), wr[i]);
          } else {
            V16<TX>::cvt(__ldg(reinterpret_cast<const uint4*>(src)), wr[i]);
            V16<TX>::cvt(__ldg(reinterpret_cast<const uint4*>(src + 4)), wr[i] + 4);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) wr[i][q] = 0.f;
        }
      }
    };
    float acc[TM][8];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    load_slice(0);
    for (int k0 = 0; k0 < a.d; k0 += kKC) {
#pragma unroll
      for (int q = 0; q < 8; ++q) xs[(xk + q) * BM + xt] = xr[q];
#pragma unroll
      for (int i = 0; i < WV; ++i)
        if (wact[i])
#pragma unroll
          for (int q = 0; q < 8; ++q) wsm[(wk[i] + q) * BN + we[i]] = wr[i][q];
      __syncthreads();
      if (k0 + kKC < a.d) load_slice(k0 + kKC);
#pragma unroll 4
      for (int kk = 0; kk < kKC; ++kk) {
        float av[TM], bv[8];
        if (TM >= 4) {
#pragma unroll
          for (int i = 0; i < TM; i += 4) {
            const float4 q4 = *reinterpret_cast<const float4*>(xs + kk * BM + tg * TM + i);
            av[i] = q4.x; av[i + 1] = q4.y; av[i + 2] = q4.z; av[i + 3] = q4.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < TM; ++i) av[i] = xs[kk * BM + tg * TM + i];
        }
        const float4 b0 = *reinterpret_cast<const float4*>(wsm + kk * BN + eg * 8);
        const float4 b1 = *reinterpret_cast<const float4*>(wsm + kk * BN + eg * 8 + 4);
        bv[0] = b0.x; bv[1] = b0.y; bv[2] = b0.z; bv[3] = b0.w;
        bv[4] = b1.x; bv[5] = b1.y; bv[6] = b1.z; bv[7] = b1.w;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      __syncthreads();
    }
    // scores (+ logit bias) into the [BM][BN] tile
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      float o[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = eg * 8 + j;
        o[j] = (e < N && a.logit_bias) ? __fadd_rn(acc[i][j], a.logit_bias[e]) : acc[i][j];
      }
      float* dst = lt + (size_t)(tg * TM + i) * BN + eg * 8;
      *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(o[4], o[5], o[6], o[7]);
    }
  } else {
    for (int i = tid; i < BM * BN; i += kThreads) {
      const int r = i / BN, e = i % BN;
      const long long t = t0 + r;
      lt[i] = (t < a.T && e < N) ? a.logits_in[t * N + e] : 0.f;
    }
  }
  __syncthreads();

  if (a.logits_out) {
    for (int i = tid; i < BM * N; i += kThreads) {
      const int r = i / N, e = i % N;
      if (t0 + r < a.T) a.logits_out[(t0 + r) * N + e] = lt[r * BN + e];
    }
  }

  float psum[EJ];
#pragma unroll
  for (int j = 0; j < EJ; ++j) psum[j] = 0.f;
  constexpr int TPW_SEL = BM / kWarps;  // 8 tokens per warp
  for (int i = 0; i < TPW_SEL; ++i) {
    const int tl = warp * TPW_SEL + i;
    const long long t = t0 + tl;
    if (t >= a.T) break;  // warp-uniform
    float r[EJ];
#pragma unroll
    for (int j = 0; j < EJ; ++j) r[j] = lt[tl * BN + lane + 32 * j];
    select_token<EJ>(r, lane, t, a, psum, bcount);
  }
  __syncthreads();  // lt is read above; wprob does not alias it, bcount does not either
  finish_block<EJ>(psum, wprob, bcount, a);
}


template <typename K>
cudaError_t launch_k(K kernel, const RouterArgs& a, int grid, size_t smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ProfScope p(K_ROUTER, s);
  return launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, s, 1, a);
}

bool use_small(const moe_config& c, const float* logits_in) {
  return logits_in == nullptr && c.n_experts <= 32;
}

// Blocks of the router launch; router_partials_bytes() sizes the partials
// buffer for the larger of the two choices.
// Few-expert kernel: warps per token group (2 tokens for N <= 8, else 1),
// so that about kSmallTargetWarps warps have work.
int router_small_wsplit(const moe_config& c) {
  const int tpw = c.n_experts <= 8 ? 2 : 1;
  const long long groups = ceil_div(c.T, tpw);
  int ws = 1;
  while (ws < kWarps && groups * ws * 2 <= kSmallTargetWarps) ws *= 2;
  return ws;
}

// bf16 scores of up to 32 experts for prefill-sized batches: the mma.sync
// kernel. Below kMmaMinTokens its 16-token tiles leave most SMs idle and
// the warp kernel, which spreads each token's row over a block, is faster
// (15 against 17 us at T = 32 and 64, N = 8, d = 4096).
constexpr int kMmaMinTokens = 256;
bool use_mma(const moe_config& c, const float* logits_in) {
  return logits_in == nullptr && c.dtype == MOE_BF16 && c.n_experts <= 32 &&
         c.d_model % 8 == 0 && c.T >= kMmaMinTokens;
}

int router_grid(const moe_config& c, const float* logits_in) {
  if (use_mma(c, logits_in)) {
    const int tiles = ceil_div(c.T, kMmaTile);
    return tiles < kSmallMaxBlocks ? tiles : kSmallMaxBlocks;
  }
  if (use_small(c, logits_in)) {
    // one round of kWarps / wsplit token groups per block, at most 4 blocks per SM
    const int tpw = c.n_experts <= 8 ? 2 : 1;
    const int gpb = kWarps / router_small_wsplit(c);
    const int blocks = ceil_div(ceil_div(c.T, tpw), gpb);
    return blocks < kSmallMaxBlocks ? blocks : kSmallMaxBlocks;
  }
  return ceil_div(c.T, kTileTokens);
}

template <typename TX>
cudaError_t launch_dtype(const moe_config& c, const RouterArgs& a, int grid, cudaStream_t s) {
  if (use_mma(c, a.logits_in)) {
    ProfScope p(K_ROUTER, s);
    if (c.n_experts <= 8)
      return launch_pdl(router_mma_kernel<8>, dim3(grid), dim3(kThreads), 0, s, 1, a);
    if (c.n_experts <= 16)
      return launch_pdl(router_mma_kernel<16>, dim3(grid), dim3(kThreads), 0, s, 1, a);
    return launch_pdl(router_mma_kernel<32>, dim3(grid), dim3(kThreads), 0, s, 1, a);
  }
  if (use_small(c, a.logits_in)) {
    const int ws = router_small_wsplit(c);
    ProfScope p(K_ROUTER, s);
    if (c.n_experts <= 8)
      return launch_pdl(router_small_kernel<TX, 8, 2>, dim3(grid), dim3(kThreads), 0, s, 1, a, ws);
    if (c.n_experts <= 16)
      return launch_pdl(router_small_kernel<TX, 16, 1>, dim3(grid), dim3(kThreads), 0, s, 1, a, ws);
    return launch_pdl(router_small_kernel<TX, 32, 1>, dim3(grid), dim3(kThreads), 0, s, 1, a, ws);
  }
  auto smem = [](int BN) {  // must match the layout in router_tiled_kernel
    const size_t tile = sizeof(float) * (size_t)kTileTokens * BN;
    const size_t slices = sizeof(float) * (size_t)kKC * (kTileTokens + BN);
    return (tile > slices ? tile : slices) + sizeof(float) * kWarps * BN + sizeof(int) * BN;
  };
  if (c.n_experts <= 32) return launch_k(router_tiled_kernel<TX, 1>, a, grid, smem(32), s);
  if (c.n_experts <= 64) return launch_k(router_tiled_kernel<TX, 2>, a, grid, smem(64), s);
  if (c.n_experts <= 128) return launch_k(router_tiled_kernel<TX, 4>, a, grid, smem(128), s);
  return launch_k(router_tiled_kernel<TX, 8>, a, grid, smem(256), s);
}

}  // namespace

bool decode_front_applies(const moe_config& c) {
  return c.dtype == MOE_BF16 && c.T >= 1 && c.T <= kFrontMaxT && c.n_experts <= 32 &&
         c.d_model % 8 == 0 && !reroutes(c) &&
         (size_t)front_np(c.n_experts) * c.d_model * 2 <= kFrontMaxRouterBytes;
}

cudaError_t launch_decode_front(const moe_config& c, const void* x, const void* w_router,
                                const float* logit_bias, const float* sel_bias, int32_t* topk_idx,
                                float* topk_w, int32_t* counts, float* prob_sum, int32_t* offsets,
                                int32_t* sorted_pair, int32_t* inv_pos, void* x_perm, int32_t* seg,
                                int tile_m, int* status, cudaStream_t s) {
  FrontArgs f{};
  RouterArgs& a = f.r;
  a.x = x; a.w = w_router; a.logit_bias = logit_bias; a.sel_bias = sel_bias;
  a.logits_in = nullptr; a.logits_out = nullptr; a.topk_idx = topk_idx; a.topk_w = topk_w;
  a.counts = counts; a.partials = nullptr; a.cpart = nullptr; a.status = status;
  a.prob_sum = prob_sum; a.done = nullptr;
  a.T = c.T; a.d = c.d_model; a.N = c.n_experts; a.k = c.top_k; a.gate_mode = c.gate_mode;
  f.capacity = c.capacity;
  f.n_shared = c.n_shared;
  f.tile_m = tile_m;
  f.offsets = offsets;
  f.sorted_pair = sorted_pair;
  f.inv_pos = inv_pos;
  f.seg = seg;
  f.x_perm = static_cast<uint4*>(x_perm);
  const size_t smem = (size_t)front_np(c.n_experts) * c.d_model * 2;
  void (*kernel)(FrontArgs) = c.n_experts <= 8    ? decode_front_kernel<8>
                              : c.n_experts <= 16 ? decode_front_kernel<16>
                                                  : decode_front_kernel<32>;
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    for (auto kfn : {decode_front_kernel<8>, decode_front_kernel<16>, decode_front_kernel<32>})
      if ((e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kFrontMaxRouterBytes)) != cudaSuccess)
        return e;
    configured_device = dev;
  }
  ProfScope p(K_DECODE_FRONT, s);
  return launch_pdl(kernel, dim3(1), dim3(kFrontThreads), smem, s, 1, f);
}

// The most blocks any router kernel for this configuration launches: the
// tiled kernel (given scores, or N > 32 in fp32) takes one per 64 tokens,
// the tensor-core kernel one per 128, and for up to 32 experts the warp
// kernel at most min(T, kSmallMaxBlocks).
int router_partial_blocks(const moe_config& c) {
  const int tiled = ceil_div(c.T, kTileTokens);
  if (c.n_experts > 32) return tiled;
  const int warp_blocks = c.T < kSmallMaxBlocks ? c.T : kSmallMaxBlocks;
  return warp_blocks > tiled ? warp_blocks : tiled;
}

size_t router_partials_bytes(const moe_config& c) {
  // probability sums (float) then counts (int32), [blocks][N] each
  return 2 * sizeof(float) * (size_t)router_partial_blocks(c) * (size_t)c.n_experts;
}

cudaError_t launch_router(const moe_config& c, const void* x, const void* w_router,
                          const float* logit_bias, const float* sel_bias,
                          const float* logits_in, float* logits_out, int32_t* topk_idx,
                          float* topk_w, int32_t* counts, float* prob_sum, float* partials,
                          int* status, cudaStream_t s) {
  // status[1] counts finished router blocks for the final sum in the last
  // block; the caller zeroes status[0..1] before each call.
  if (c.T == 0) {
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.n_experts, s);
    if (e != cudaSuccess) return e;
    return cudaMemsetAsync(prob_sum, 0, sizeof(float) * c.n_experts, s);
  }
  int32_t* cpart = reinterpret_cast<int32_t*>(partials) +
                   (size_t)router_partial_blocks(c) * (size_t)c.n_experts;
  if (router_tc_applies(c, logits_in))
    return launch_router_tc(c, x, w_router, logit_bias, sel_bias, logits_out, topk_idx, topk_w,
                            counts, prob_sum, partials, cpart, status, s);
  RouterArgs a;
  a.x = x; a.w = w_router; a.logit_bias = logit_bias; a.sel_bias = sel_bias;
  a.logits_in = logits_in; a.logits_out = logits_out; a.topk_idx = topk_idx;
  a.topk_w = topk_w; a.counts = counts; a.partials = partials; a.cpart = cpart;
  a.status = status; a.prob_sum = prob_sum; a.done = status + 1;
  a.T = c.T; a.d = c.d_model; a.N = c.n_experts; a.k = c.top_k; a.gate_mode = c.gate_mode;
  const int grid = router_grid(c, logits_in);
  return (c.dtype == MOE_BF16) ? launch_dtype<__nv_bfloat16>(c, a, grid, s)
                               : launch_dtype<float>(c, a, grid, s);
}

}  // namespace moe
