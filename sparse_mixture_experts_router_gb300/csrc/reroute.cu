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
// token, slot) order is ascending pair order. Round 0's proposals are the
// routed experts. Then, per round r:
//  1. publish - the block's count of round-r proposals per expert goes to
//               global memory, in one of two buffers by round parity; the
//               per-warp counts become warp bases inside the block. One grid
//               barrier.
//  2. totals  - every block sums the published counts of the blocks before it
//               (its base per expert) and of all blocks (the round's totals),
//               all threads reading at once. From the totals every block
//               derives the room left for round r + 1 itself, so all copies
//               agree without a second barrier. A round without proposals
//               ends the kernel.
//  3. walk    - each warp takes its tokens in order, once: a round-r proposal
//               is accepted iff block base + warp base + its rank among the
//               warp's proposals to that expert < room; then the token's
//               still-pending slots take, in slot order, its best eligible
//               experts for round r + 1 (a warp argmax over the token's N
//               keys, one per slot), each ranked by a per-warp shared-memory
//               counter. A token's state, scores and held set are loaded
//               together, and the next token's loads are issued before the
//               current one is processed, so a round costs about one memory
//               round trip per warp plus the barrier.
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

// A selection key as an unsigned integer with the same order: the sign bit
// flipped for positive keys, all bits for negative ones (-0 is made +0 first,
// as the two compare equal). 0 is below every key, -inf included, and marks
// "no candidate" in the warp argmax.
__device__ __forceinline__ uint32_t key_order(float v) {
  if (v == 0.0f) v = 0.0f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The next token a warp walks after t: among its first 32 tokens only those
// still live, after them every token.
__device__ __forceinline__ int next_walked(int t, int t_lo, int t_hi, uint32_t live) {
  const int j = t + 1 - t_lo;
  if (j < 32) {
    const uint32_t m = live & (0xffffffffu << j);
    if (m) return t_lo + __ffs(m) - 1;
    return min(t_hi, t_lo + 32);
  }
  return min(t_hi, t + 1);
}

// One token's loads for a round's walk: its pairs' state, proposal and
// rank (lanes < k), its selection keys (expert lane + 32 i in key[i]) and
// its held-set words (the same in every lane).
template <int NW>
struct TokLoad {
  int st, pr, rk;
  uint32_t key[NW];  // key_order of the selection keys
  uint32_t hw[NW];
};

template <int NW>
__device__ __forceinline__ void load_token(const RerouteArgs& a, int t, int lane, TokLoad<NW>& L) {
  const size_t p = (size_t)t * a.k + lane;
  L.st = lane < a.k ? a.assign[p] : -1;
  L.pr = lane < a.k ? a.prop[p] : -1;
  L.rk = lane < a.k ? a.prank[p] : 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const int e = lane + 32 * i;
    float r = -INFINITY;
    if (e < a.N) {
      r = a.logits[(size_t)t * a.N + e];
      if (a.sel_bias) r = __fadd_rn(r, a.sel_bias[e]);
      if (isnan(r)) r = -INFINITY;
    }
    L.key[i] = key_order(r);
    L.hw[i] = i < a.W ? a.held[(size_t)t * a.W + i] : 0u;
  }
}

template <int NW>
__global__ void __launch_bounds__(kRrThreads, 1) reroute_kernel(RerouteArgs a) {
  extern __shared__ int sh[];
  const int N = a.N, k = a.k, W = a.W;
  int* s_cnt = sh;                       // [kRrWarps][N] counts of the proposals being made
  int* s_wbase = sh + kRrWarps * N;      // [kRrWarps][N] bases of the last round's proposals
  int* s_room = s_wbase + kRrWarps * N;  // [N] room the last round's proposals saw
  int* s_next = s_room + N;              // [N] room for the proposals being made
  int* s_tot = s_next + N;               // [N]
  int* s_base = s_tot + N;               // [N]
  __shared__ int s_any;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int gw = blockIdx.x * kRrWarps + warp;
  const int t_lo = min(a.T, gw * a.tokens_per_warp);
  const int t_hi = min(a.T, t_lo + a.tokens_per_warp);
  for (int i = threadIdx.x; i < kRrWarps * N; i += kRrThreads) s_cnt[i] = 0;
  for (int e = threadIdx.x; e < N; e += kRrThreads) s_room[e] = a.capacity > 0 ? a.capacity : INT_MAX;
  __syncthreads();
  int* mine = s_cnt + warp * N;
  const int* my_base = s_wbase + warp * N;

  // round 0: every pair proposes its routed expert; the token holds them all
  {
    int e_next = (t_lo < t_hi && lane < k) ? a.topk_idx[(size_t)t_lo * k + lane] : -1;
    for (int t = t_lo; t < t_hi; ++t) {
      int e = e_next;
      if (t + 1 < t_hi && lane < k) e_next = a.topk_idx[(size_t)(t + 1) * k + lane];
      const size_t p = (size_t)t * k + lane;
      if (lane < k) {
        if (e < 0 || e >= N) {
          set_status(a.status, MOE_ERR_DEVICE_CHECK);
          e = -1;
        }
        a.assign[p] = e >= 0 ? kPending : -1;
        a.prop[p] = e;
        if (e >= 0) a.prank[p] = atomicAdd(&mine[e], 1);
      } else {
        e = -1;
      }
      for (int i = 0; i < W; ++i) {
        const uint32_t bit = (e >= 0 && (e >> 5) == i) ? (1u << (e & 31)) : 0u;
        const uint32_t word = __reduce_or_sync(0xffffffffu, bit);
        if (lane == i) a.held[(size_t)t * W + i] = word;
      }
    }
  }

  // the warp's first 32 tokens that still have a pending pair (bit j: token
  // t_lo + j); tokens past them are walked every round
  uint32_t live = t_hi - t_lo >= 32 ? 0xffffffffu : (1u << (t_hi - t_lo)) - 1u;
  int round = 0;
  for (;; ++round) {
    __syncthreads();
    // ---- 1. publish this round's counts; warp counts become warp bases
    int32_t* pub = a.pub + (size_t)(round & 1) * gridDim.x * N;
    for (int e = threadIdx.x; e < N; e += kRrThreads) {
      int acc = 0;
      for (int w = 0; w < kRrWarps; ++w) {
        const int v = s_cnt[w * N + e];
        s_wbase[w * N + e] = acc;
        s_cnt[w * N + e] = 0;
        acc += v;
      }
      pub[(size_t)blockIdx.x * N + e] = acc;
      s_base[e] = 0;
      s_tot[e] = 0;
    }
    if (threadIdx.x == 0) s_any = 0;
    if (!rr_grid_barrier(a.status + 2, a.status, (round + 1) * (int)gridDim.x, a.limit_ns)) return;
    // ---- 2. the block's base and the round's total per expert: the G x N
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
      const int base = s_base[e], tot = s_tot[e];
      for (int w = 0; w < kRrWarps; ++w) s_wbase[w * N + e] += base;
      s_next[e] = s_room[e] - min(s_room[e], tot);
      if (tot != 0) s_any = 1;
    }
    __syncthreads();
    if (!s_any) break;  // no proposal in this round: every pair is settled
    if (round > N + 1) {  // cannot happen (a rejecting round fills an expert)
      set_status(a.status, MOE_ERR_DEVICE_CHECK);
      return;
    }
    // ---- 3. walk: accept this round's proposals, make the next round's
    TokLoad<NW> cur, nxt;
    int t = next_walked(t_lo - 1, t_lo, t_hi, live);
    if (t < t_hi) load_token<NW>(a, t, lane, cur);
    while (t < t_hi) {
      const int tn = next_walked(t, t_lo, t_hi, live);
      if (tn < t_hi) load_token<NW>(a, tn, lane, nxt);
      const size_t p = (size_t)t * k + lane;
      int st = cur.st;
      const bool was_pending = lane < k && st == kPending;
      bool accepted = false;
      if (was_pending && cur.pr >= 0 && my_base[cur.pr] + cur.rk < s_room[cur.pr]) {
        st = cur.pr;
        accepted = true;
      }
      // the held set gains the accepted experts (every lane keeps the words);
      // round 0's are the routed experts, which it holds already
      uint32_t amask = round > 0 ? __ballot_sync(0xffffffffu, accepted) : 0u;
      bool held_changed = amask != 0;
      while (amask) {
        const int s = __ffs(amask) - 1;
        amask &= amask - 1;
        const int ea = __shfl_sync(0xffffffffu, st, s);
#pragma unroll
        for (int i = 0; i < NW; ++i)
          if ((ea >> 5) == i) cur.hw[i] |= 1u << (ea & 31);
      }
      // the slots still pending propose for the next round
      uint32_t pmask = __ballot_sync(0xffffffffu, lane < k && st == kPending);
      int new_pr = -1, new_rk = 0;
      if (pmask) {
        uint32_t elig = 0;  // bit i: expert lane + 32 i can take a proposal
#pragma unroll
        for (int i = 0; i < NW; ++i) {
          const int e = lane + 32 * i;
          if (e < N && !((cur.hw[i] >> lane) & 1u) && s_next[e] > 0) elig |= 1u << i;
        }
        while (pmask) {
          const int s = __ffs(pmask) - 1;
          pmask &= pmask - 1;
          // the lane's best eligible key (its experts ascend with i, so the
          // first of equal keys is the lower index), then the warp's largest
          // key and the lowest expert that holds it
          uint32_t bk = 0;
          int be = kNone;
#pragma unroll
          for (int i = 0; i < NW; ++i)
            if (((elig >> i) & 1u) && cur.key[i] > bk) {
              bk = cur.key[i];
              be = lane + 32 * i;
            }
          const uint32_t top = __reduce_max_sync(0xffffffffu, bk);
          be = (int)__reduce_min_sync(0xffffffffu,
                                      (top != 0 && bk == top) ? (uint32_t)be : (uint32_t)kNone);
          if (lane == s) {
            if (be == kNone) {
              st = -1;  // no expert left for it: dropped
            } else {
              new_pr = be;
              new_rk = mine[be]++;
            }
          }
          if (be != kNone && (be & 31) == lane) elig &= ~(1u << (be >> 5));
          __syncwarp();
        }
      }
      if (lane < k) {
        if (st != cur.st) a.assign[p] = st;
        if (st == kPending) {
          a.prop[p] = new_pr;
          a.prank[p] = new_rk;
        }
      }
      if (held_changed && lane < W) {
#pragma unroll
        for (int i = 0; i < NW; ++i)
          if (i == lane) a.held[(size_t)t * W + i] = cur.hw[i];
      }
      // a token without a pending pair is done for the remaining rounds
      if (t - t_lo < 32 && !__any_sync(0xffffffffu, lane < k && st == kPending))
        live &= ~(1u << (t - t_lo));
      cur = nxt;
      t = tn;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += kRrThreads) s_room[e] = s_next[e];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.rounds_out)
    *a.rounds_out = round > 0 ? round - 1 : 0;
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
  const size_t smem = sizeof(int) * ((size_t)2 * kRrWarps * c.n_experts + 4 * c.n_experts);
  // keys and held words per lane: one per 32 experts, rounded up to a power of 2
  void (*kernel)(RerouteArgs) = a.W <= 1   ? reroute_kernel<1>
                                : a.W <= 2 ? reroute_kernel<2>
                                : a.W <= 4 ? reroute_kernel<4>
                                           : reroute_kernel<8>;
  // one block an SM at most (a cooperative grid must be resident at once),
  // and no more blocks than it takes to give every warp a token
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kRrThreads,
                                                                smem);
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
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace moe
