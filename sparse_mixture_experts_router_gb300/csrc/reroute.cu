// Capacity overflow rerouted instead of dropped ("Mixture of experts and
// speculative decoding", "Keeping the experts busy": the pairs over an
// expert's capacity are dropped or rerouted; the page gives no order).
//
// The reading computed here works in rounds:
//  round 0  the capacity cut: each expert keeps the first C of its (token,
//           slot) pairs in ascending pair order; the rest are pending, and
//           room[e] = C - kept at e.
//  round r  every pending pair, in slot order within its token, proposes
//           the expert with the highest selection key fp32(r + sel_bias)
//           (ties to the lower index, NaN below every number) that has room
//           at the start of the round, that the token does not hold (its k
//           routed experts and those it was rerouted to) and that no lower
//           slot of the token proposed to in this round; a pair with no such
//           expert is dropped. Each expert accepts the round's proposals in
//           ascending pair id up to its room; the others stay pending.
// The rounds end when one has no proposal. A round that rejects a proposal
// fills an expert, so there are at most N + 1 rounds after the cut. The
// result is unique: it does not depend on the grid or on timing.
//
// One cooperative kernel runs all rounds. Block b owns a contiguous range of
// tokens and each of its warps a contiguous sub-range, so (block, warp,
// token, slot) order is ascending pair order. Per round:
//  1. propose - each warp walks its tokens; a token's pending slots take, in
//               slot order, its best eligible experts (a warp argmax over the
//               token's N keys, one per slot). Each proposal is given its
//               rank among the warp's proposals to that expert (a per-warp
//               shared-memory counter; the warp takes its tokens in order).
//  2. publish - the block's proposal count per expert goes to global memory,
//               in one of two buffers by round parity; the warp counts become
//               warp bases inside the block. One grid barrier.
//  3. accept  - every block sums the published counts of the blocks before it
//               (its base per expert) and of all blocks (the round's totals).
//               A proposal is accepted iff block base + warp base + its rank
//               < room. Every block then takes the totals off its own copy of
//               room, so all copies agree without a second barrier.
// A round's buffer is rewritten two rounds later, after the barrier between,
// which every block passes only once all blocks have finished reading it.
#include <limits.h>
#include <math.h>

#include "device_util.cuh"
#include "moe_internal.h"
#include "sm103_wait.cuh"

namespace moe {
namespace {

constexpr int kRrThreads = 512;
constexpr int kRrWarps = kRrThreads / 32;
constexpr int kRrMaxBlocks = 512;              // bound of the published-count buffers
constexpr int kMaxWords = kMaxExperts / 32;    // held-set words per token
constexpr int32_t kPending = -2;
constexpr int kNone = INT_MAX;                 // "no candidate" in the argmax
constexpr int kBatch = 8;                      // published counts loaded at once a thread

struct RerouteArgs {
  const float* logits;      // [T][N] router scores
  const float* sel_bias;    // [N] or null
  const int32_t* topk_idx;  // [T][k]
  int32_t* assign;          // [T][k] out
  int32_t* rounds_out;      // [1] out or null
  uint32_t* held;           // [T][W] experts a token holds, one bit each
  int32_t* prop;            // [T*k] expert proposed this round
  int32_t* prank;           // [T*k] rank among the warp's proposals to it
  int32_t* pub;             // [2][G][N] published counts per block and expert
  int* status;              // status word; status[2] is the barrier counter
  int T, N, k, W, capacity, tokens_per_warp;
  unsigned long long limit_ns;
};

// Bounded grid barrier: the block's writes are made visible, then thread 0
// waits until `target` blocks have arrived. False if the wait ran out (the
// status word then says MOE_ERR_TIMEOUT).
__device__ bool rr_grid_barrier(int* counter, int* status, int target, uint64_t limit_ns) {
  __shared__ int ok;
  __syncthreads();
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

// (key, expert) b beats a: a real candidate over none, a larger key, or an
// equal key with a lower index.
__device__ __forceinline__ bool beats(float kb, int eb, float ka, int ea) {
  return eb != kNone && (ea == kNone || kb > ka || (kb == ka && eb < ea));
}

__global__ void __launch_bounds__(kRrThreads, 1) reroute_kernel(RerouteArgs a) {
  extern __shared__ int sh[];
  const int N = a.N, k = a.k, W = a.W;
  int* s_cnt = sh;                       // [kRrWarps][N] counts, then bases
  int* s_room = sh + kRrWarps * N;       // [N]
  int* s_tot = s_room + N;               // [N]
  int* s_base = s_tot + N;               // [N]
  __shared__ int s_any;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int gw = blockIdx.x * kRrWarps + warp;
  const int t_lo = min(a.T, gw * a.tokens_per_warp);
  const int t_hi = min(a.T, t_lo + a.tokens_per_warp);
  const int npl = (N + 31) / 32;  // experts per lane in the argmax
  for (int i = threadIdx.x; i < kRrWarps * N; i += kRrThreads) s_cnt[i] = 0;
  for (int e = threadIdx.x; e < N; e += kRrThreads) s_room[e] = a.capacity > 0 ? a.capacity : INT_MAX;
  __syncthreads();
  int* mine = s_cnt + warp * N;

  // round 0: every pair proposes its routed expert; the token holds them all
  for (int t = t_lo; t < t_hi; ++t) {
    const size_t p = (size_t)t * k + lane;
    int e = -1;
    if (lane < k) {
      e = a.topk_idx[p];
      if (e < 0 || e >= N) {
        set_status(a.status, MOE_ERR_DEVICE_CHECK);
        e = -1;
      }
      a.assign[p] = e >= 0 ? kPending : -1;
      a.prop[p] = e;
      if (e >= 0) a.prank[p] = atomicAdd(&mine[e], 1);
    }
    for (int i = 0; i < W; ++i) {
      const uint32_t bit = (e >= 0 && (e >> 5) == i) ? (1u << (e & 31)) : 0u;
      const uint32_t word = __reduce_or_sync(0xffffffffu, bit);
      if (lane == i) a.held[(size_t)t * W + i] = word;
    }
  }

  int round = 0;
  for (;; ++round) {
    if (round > 0) {
      // ---- 1. propose
      for (int t = t_lo; t < t_hi; ++t) {
        const size_t p0 = (size_t)t * k;
        const bool pend = lane < k && a.assign[p0 + lane] == kPending;
        uint32_t pmask = __ballot_sync(0xffffffffu, pend);
        if (pmask == 0) continue;
        float key[kMaxWords];
        uint32_t elig = 0;  // bit i: expert lane + 32 i can take a proposal
#pragma unroll
        for (int i = 0; i < kMaxWords; ++i) {
          key[i] = -INFINITY;
          const int e = lane + 32 * i;
          if (i < npl && e < N) {
            float r = a.logits[(size_t)t * N + e];
            if (a.sel_bias) r = __fadd_rn(r, a.sel_bias[e]);
            key[i] = isnan(r) ? -INFINITY : r;
            const uint32_t h = a.held[(size_t)t * W + i];
            if (!((h >> lane) & 1u) && s_room[e] > 0) elig |= 1u << i;
          }
        }
        while (pmask) {
          const int s = __ffs(pmask) - 1;
          pmask &= pmask - 1;
          float bk = -INFINITY;
          int be = kNone;
#pragma unroll
          for (int i = 0; i < kMaxWords; ++i)
            if ((elig >> i) & 1u) {
              if (beats(key[i], lane + 32 * i, bk, be)) {
                bk = key[i];
                be = lane + 32 * i;
              }
            }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ok_ = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (beats(ok_, oe, bk, be)) {
              bk = ok_;
              be = oe;
            }
          }
          if (lane == s) {
            if (be == kNone) {
              a.assign[p0 + s] = -1;  // no expert left for it: dropped
            } else {
              a.prop[p0 + s] = be;
              a.prank[p0 + s] = mine[be]++;
            }
          }
          if (be != kNone && (be & 31) == lane) elig &= ~(1u << (be >> 5));
          __syncwarp();
        }
      }
    }
    __syncthreads();
    // ---- 2. publish the block's counts; warp counts become warp bases
    int32_t* pub = a.pub + (size_t)(round & 1) * gridDim.x * N;
    for (int e = threadIdx.x; e < N; e += kRrThreads) {
      int acc = 0;
      for (int w = 0; w < kRrWarps; ++w) {
        const int v = s_cnt[w * N + e];
        s_cnt[w * N + e] = acc;
        acc += v;
      }
      pub[(size_t)blockIdx.x * N + e] = acc;
    }
    for (int e = threadIdx.x; e < N; e += kRrThreads) {
      s_base[e] = 0;
      s_tot[e] = 0;
    }
    if (threadIdx.x == 0) s_any = 0;
    if (!rr_grid_barrier(a.status + 2, a.status, (round + 1) * (int)gridDim.x, a.limit_ns)) return;
    // ---- 3. the block's base and the round's total per expert: the G x N
    // published counts are read by all threads at once (kBatch independent
    // loads in flight each) and summed with shared-memory atomics (integer
    // sums: the order does not change them)
    const int total = (int)gridDim.x * N;
    for (int q0 = threadIdx.x; q0 < total; q0 += kRrThreads * kBatch) {
      int v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int q = q0 + j * kRrThreads;
        v[j] = q < total ? __ldcg(pub + q) : 0;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (v[j] != 0) {
          const int q = q0 + j * kRrThreads;
          const int b = q / N, e = q - b * N;
          atomicAdd(&s_tot[e], v[j]);
          if (b < (int)blockIdx.x) atomicAdd(&s_base[e], v[j]);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += kRrThreads) {
      const int base = s_base[e];
      for (int w = 0; w < kRrWarps; ++w) s_cnt[w * N + e] += base;
      if (s_tot[e] != 0) s_any = 1;
    }
    __syncthreads();
    if (!s_any) break;  // no proposal in this round: every pair is settled
    for (int t = t_lo; t < t_hi; ++t) {
      const size_t p = (size_t)t * k + lane;
      if (lane < k && a.assign[p] == kPending) {
        const int e = a.prop[p];
        if (e >= 0 && mine[e] + a.prank[p] < s_room[e]) {
          a.assign[p] = e;
          atomicOr(&a.held[(size_t)t * W + (e >> 5)], 1u << (e & 31));
        }
      }
      __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += kRrThreads) {
      s_room[e] -= min(s_room[e], s_tot[e]);
      for (int w = 0; w < kRrWarps; ++w) s_cnt[w * N + e] = 0;
    }
    __syncthreads();
    if (round > N + 1) {  // cannot happen (see above); stop rather than loop
      set_status(a.status, MOE_ERR_DEVICE_CHECK);
      return;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.rounds_out) *a.rounds_out = round - 1;
}

}  // namespace

size_t reroute_scratch_bytes(const moe_config& c, size_t* held, size_t* per_pair, size_t* pub) {
  const size_t T = (size_t)c.T, P = T * c.top_k, W = (size_t)(c.n_experts + 31) / 32;
  const size_t h = align_up(sizeof(uint32_t) * T * W, 256);
  const size_t pp = align_up(sizeof(int32_t) * P, 256);
  const size_t pb = align_up(sizeof(int32_t) * 2 * kRrMaxBlocks * (size_t)c.n_experts, 256);
  if (held) *held = h;
  if (per_pair) *per_pair = pp;
  if (pub) *pub = pb;
  return h + 2 * pp + pb;
}

cudaError_t launch_reroute(const moe_config& c, const float* logits, const float* sel_bias,
                           const int32_t* topk_idx, int32_t* assign, int32_t* rounds,
                           void* scratch, int* status, cudaStream_t s) {
  if (c.T == 0) return rounds ? cudaMemsetAsync(rounds, 0, sizeof(int32_t), s) : cudaSuccess;
  size_t hb = 0, ppb = 0, pbb = 0;
  reroute_scratch_bytes(c, &hb, &ppb, &pbb);
  char* base = static_cast<char*>(scratch);
  RerouteArgs a;
  a.logits = logits;
  a.sel_bias = sel_bias;
  a.topk_idx = topk_idx;
  a.assign = assign;
  a.rounds_out = rounds;
  a.held = reinterpret_cast<uint32_t*>(base);
  a.prop = reinterpret_cast<int32_t*>(base + hb);
  a.prank = reinterpret_cast<int32_t*>(base + hb + ppb);
  a.pub = reinterpret_cast<int32_t*>(base + hb + 2 * ppb);
  a.status = status;
  a.T = c.T;
  a.N = c.n_experts;
  a.k = c.top_k;
  a.W = (c.n_experts + 31) / 32;
  a.capacity = c.capacity;
  a.limit_ns = kWaitLimitNs;
  const size_t smem = sizeof(int) * ((size_t)kRrWarps * c.n_experts + 3 * c.n_experts);
  // one block an SM at most (a cooperative grid must be resident at once),
  // and no more blocks than it takes to give every warp a token
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reroute_kernel,
                                                                kRrThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int grid = num_sms();
  grid = grid < kRrMaxBlocks ? grid : kRrMaxBlocks;
  const int need = ceil_div(c.T, kRrWarps);
  grid = grid < need ? grid : need;
  a.tokens_per_warp = ceil_div(c.T, grid * kRrWarps);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRrThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfScope p(K_REROUTE, s);
  return cudaLaunchKernelEx(&cfg, reroute_kernel, a);
}

}  // namespace moe
