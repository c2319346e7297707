// K2: grouping of the (token, slot) pairs by expert, and the row gather.
//
// The batched form of the per-expert dispatch loop of the pages' toy layers
// ("Mixture of experts and speculative decoding", "A toy MoE layer in
// PyTorch"; "Mixture of Experts and Guided Decoding", sparse MoE code):
// every pair that chose expert e lands in e's contiguous row segment, in
// ascending pair order, so the result is unique and bit-exact.
//
// Launch shapes, by the number of pairs P = T*k:
//  P <= 2048          - one block does everything but the row gather
//                       (permute_small_kernel), then the gather.
//  P <= 65536         - one launch per expert group (permute_group_kernel),
//                       then the gather: each block owns a group of experts,
//                       takes the per-expert totals (the router's counts, or
//                       its own histogram), scans them into offsets, and
//                       ranks its experts' pairs in two ordered passes.
//  larger             - four launches:
//    hist   - one block per chunk of 2048 pairs counts pairs per expert with
//             warp-aggregated shared-memory atomics (one atomic per distinct
//             expert in a warp, found with __match_any_sync).
//    scan   - one block: per expert, exclusive scan of the chunk counts; then
//             the exclusive scan over experts gives expert_offsets; the chunk
//             table becomes each chunk's first row per expert.
//    rank   - one block per chunk: per-warp counts, a scan over the 8 warps,
//             then each warp walks its 256 pairs in order, 32 at a time; a
//             pair's row is its warp base + the number of lower lanes with
//             the same expert (__match_any_sync + popc of the lane mask).
//  gather     - one warp per token reads its row once with 16-byte loads
//               and stores it to the rows of each of its kept pairs.
// The segment table of the grouped GEMM comes with the first two shapes and
// from seg_table_kernel after the third.
#include "device_util.cuh"
#include "moe_internal.h"
#include "seg_table.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = kPermuteChunk;            // 2048 pairs
constexpr int kPerWarp = kChunk / kWarps;        // 256 pairs
constexpr int kRounds = kPerWarp / 32;           // 8
// An expert index of -1 marks a pair with no expert (capacity rerouting
// dropped it): it gets no row and inv_pos -1, and is not an error.
constexpr int32_t kNoExpert = -1;
constexpr int32_t kOutside = -3;  // past the last pair


__global__ void __launch_bounds__(kThreads) permute_hist_kernel(const int32_t* __restrict__ idx,
                                                                int P, int N, int32_t* hist,
                                                                int* status) {
  extern __shared__ int sh[];
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < N; e += kThreads) sh[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int base = blockIdx.x * kChunk + warp * kPerWarp;
  for (int r = 0; r < kRounds; ++r) {
    const int p = base + r * 32 + lane;
    int e = -1;
    if (p < P) {
      e = idx[p];
      if (e < 0 || e >= N) {
        if (e != kNoExpert) set_status(status, MOE_ERR_DEVICE_CHECK);
        e = -1;
      }
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&sh[e], __popc(peers));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += kThreads) hist[(size_t)blockIdx.x * N + e] = sh[e];
}

// Per expert, the chunk counts become each chunk's first rank inside the
// expert (exclusive scan over chunks); the experts' kept rows (count, or
// min(count, capacity)) scanned over experts give expert_offsets.
__global__ void __launch_bounds__(kThreads) permute_scan_kernel(int32_t* hist, int nchunks, int N,
                                                                int capacity, int32_t* offsets) {
  extern __shared__ int tot[];  // [N + 1]
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < N; e += kThreads) {
    int run = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int v = hist[(size_t)c * N + e];
      hist[(size_t)c * N + e] = run;
      run += v;
    }
    tot[e] = (capacity > 0 && run > capacity) ? capacity : run;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int total = warp_exclusive_scan(tot, N, threadIdx.x);
    if (threadIdx.x == 0) tot[N] = total;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= N; e += kThreads) offsets[e] = tot[e];
}

__global__ void __launch_bounds__(kThreads) permute_rank_kernel(const int32_t* __restrict__ idx,
                                                                int P, int N, int capacity,
                                                                const int32_t* __restrict__ chunk_base,
                                                                const int32_t* __restrict__ offsets,
                                                                int32_t* sorted_pair,
                                                                int32_t* inv_pos) {
  extern __shared__ int wh[];  // [kWarps][N]
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < kWarps * N; i += kThreads) wh[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int base = blockIdx.x * kChunk + warp * kPerWarp;
  int* mine = wh + warp * N;

  int ev[kRounds];
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int p = base + r * 32 + lane;
    int e = (p < P) ? idx[p] : kOutside;
    if (e == kNoExpert) inv_pos[p] = -1;  // a pair with no expert: no row
    if (e < 0 || e >= N) e = -1;
    ev[r] = e;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += kThreads) {
    int acc = chunk_base[(size_t)blockIdx.x * N + e];
    for (int w = 0; w < kWarps; ++w) {
      const int v = wh[w * N + e];
      wh[w * N + e] = acc;
      acc += v;
    }
  }
  __syncthreads();
  const uint32_t lt = lanemask_lt();
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int p = base + r * 32 + lane;
    const int e = ev[r];
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int rank = mine[e] + __popc(peers & lt);  // among expert e's pairs
      if (capacity == 0 || rank < capacity) {
        const int pos = offsets[e] + rank;
        sorted_pair[pos] = p;
        inv_pos[p] = pos;
      } else {
        inv_pos[p] = -1;  // dropped by the capacity
      }
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
}

// One warp per token: x_perm[inv_pos[t*k + slot]] = x[t] for every kept
// slot. The token's row is read from HBM once and written to all of its
// rows; a row-by-row gather reads a token's row k times, and with x_perm
// streaming through L2 those repeated reads went back to HBM (DeepSeek-V3
// shape: about twice the unique bytes). A row is written only when
// sorted_pair confirms that it holds the pair: a pair dropped by the
// capacity (-1), or one whose expert index was out of range (reported in the
// status word; its inv_pos entry is not written), writes nothing.
__global__ void __launch_bounds__(kThreads) permute_gather_kernel(const uint4* __restrict__ x,
                                                                  const int32_t* __restrict__ inv_pos,
                                                                  const int32_t* __restrict__ sorted_pair,
                                                                  int T, int P, int k,
                                                                  int vec_per_row,
                                                                  uint4* __restrict__ x_perm) {
  const int t = blockIdx.x * kWarps + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  pdl_wait();
  pdl_trigger();
  if (t >= T) return;
  const int pair = t * k + lane;
  int my = lane < k ? __ldg(inv_pos + pair) : -1;
  if (my < 0 || my >= P || __ldg(sorted_pair + my) != pair) my = -1;
  int rows[kMaxTopK];
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) rows[s] = __shfl_sync(0xffffffffu, my, s);
  const uint4* src = x + (size_t)t * vec_per_row;
#pragma unroll 4
  for (int i = lane; i < vec_per_row; i += 32) {
    const uint4 v = __ldg(src + i);
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (s < k && rows[s] >= 0) x_perm[(size_t)rows[s] * vec_per_row + i] = v;
  }
}

// The counting, scans and stable ranks of the permutation (and optionally
// the grouped GEMM's segment table) in one block when the T*k pairs fit one
// chunk (decode-sized batches): two launches (this and the row gather)
// instead of five. Same results as the multi-block path.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;
__global__ void __launch_bounds__(kSmallThreads) permute_small_kernel(
    const int32_t* __restrict__ idx, int P, int N, int capacity, int32_t* offsets,
    int32_t* sorted_pair, int32_t* inv_pos, int* status, int32_t* seg, int n_shared, int T,
    int tile_m) {
  extern __shared__ int sh[];
  int* wh = sh;                        // [kSmallWarps][N] counts, then rank bases
  int* soff = sh + kSmallWarps * N;    // [N+1] offsets
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < kSmallWarps * N; i += kSmallThreads) wh[i] = 0;
  __syncthreads();
  const int per_warp = (P + kSmallWarps - 1) / kSmallWarps;
  const int p0 = warp * per_warp, p1 = min(P, p0 + per_warp);
  int* mine = wh + warp * N;
  for (int b = p0; b < p1; b += 32) {
    const int p = b + lane;
    int e = -1;
    if (p < p1) {
      e = idx[p];
      if (e == kNoExpert) inv_pos[p] = -1;  // a pair with no expert: no row
      if (e < 0 || e >= N) {
        if (e != kNoExpert) set_status(status, MOE_ERR_DEVICE_CHECK);
        e = -1;
      }
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += kSmallThreads) {
    int tot = 0;
    for (int w = 0; w < kSmallWarps; ++w) tot += wh[w * N + e];
    soff[e] = (capacity > 0 && tot > capacity) ? capacity : tot;  // rows kept
  }
  __syncthreads();
  if (warp == 0) {
    const int total = warp_exclusive_scan(soff, N, lane);
    if (lane == 0) soff[N] = total;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= N; e += kSmallThreads) offsets[e] = soff[e];
  for (int e = threadIdx.x; e < N; e += kSmallThreads) {
    int base = 0;
    for (int w = 0; w < kSmallWarps; ++w) {
      const int v = wh[w * N + e];
      wh[w * N + e] = base;
      base += v;
    }
  }
  __syncthreads();
  const uint32_t lt = lanemask_lt();
  for (int b = p0; b < p1; b += 32) {
    const int p = b + lane;
    int e = (p < p1) ? idx[p] : -1;
    if (e < 0 || e >= N) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int rank = mine[e] + __popc(peers & lt);  // among expert e's pairs
      if (capacity == 0 || rank < capacity) {
        const int pos = soff[e] + rank;
        sorted_pair[pos] = p;
        inv_pos[p] = pos;
      } else {
        inv_pos[p] = -1;  // dropped by the capacity
      }
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  if (seg != nullptr) {  // segment table of the grouped GEMM
    __syncthreads();
    write_seg_table(soff, N, n_shared, T, P, tile_m, seg, wh);  // wh is free again
  }
}

// Mid-sized batches: block g owns experts [g*epb, min(N, (g+1)*epb)).
// Every block forms all N offsets (from `counts` when given, else from its
// own histogram of the pairs) so no block waits for another; block 0 writes
// expert_offsets and the segment table. Each of the 32 warps covers one
// contiguous range of pairs: a first pass counts the block's experts per
// warp, a scan over the warps turns the counts into row bases, and a second
// pass assigns rows in pair order (lower lanes with the same expert first).
constexpr int kGroupThreads = 1024;
constexpr int kGroupWarps = kGroupThreads / 32;
constexpr int kGroupMaxPairs = 1 << 16;  // above this the chunked path is faster
constexpr int kGroupBlocks = 16;
constexpr int kGroupBatch = 8;  // rounds of 32 pairs loaded ahead
__global__ void __launch_bounds__(kGroupThreads) permute_group_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ counts, int P, int N, int epb,
    int capacity, int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos, int* status,
    int32_t* seg,
    int n_shared, int T, int tile_m) {
  extern __shared__ int sh[];
  int* s_off = sh;                      // [N + 1] totals, then offsets
  int* s_wc = sh + N + 1;               // [kGroupWarps][epb] counts, then row bases
  int* s_seg = s_wc + kGroupWarps * epb;  // [N + n_shared + 1] (block 0)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e_lo = blockIdx.x * epb, e_hi = min(N, e_lo + epb);
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < N; e += kGroupThreads) s_off[e] = counts ? counts[e] : 0;
  for (int i = threadIdx.x; i < kGroupWarps * epb; i += kGroupThreads) s_wc[i] = 0;
  __syncthreads();
  const int per_warp = ((P + kGroupWarps - 1) / kGroupWarps + 31) / 32 * 32;
  const int p0 = warp * per_warp, p1 = min(P, p0 + per_warp);
  // The passes below walk the warp's range kGroupBatch rounds at a time,
  // loading a batch's expert indices before using any of them.
  if (counts == nullptr) {
    for (int b0 = p0; b0 < p1; b0 += 32 * kGroupBatch) {
      int ev[kGroupBatch];
#pragma unroll
      for (int r = 0; r < kGroupBatch; ++r) {
        const int p = b0 + 32 * r + lane;
        ev[r] = p < p1 ? idx[p] : -1;
      }
#pragma unroll
      for (int r = 0; r < kGroupBatch; ++r) {
        const int p = b0 + 32 * r + lane;
        int e = ev[r];
        if (p < p1 && (e < 0 || e >= N)) {
          if (e != kNoExpert) set_status(status, MOE_ERR_DEVICE_CHECK);
          e = -1;
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_off[e], __popc(peers));
      }
    }
    __syncthreads();
  }
  if (warp == 0) {
    // the routed pairs must add up to T*k; then each expert keeps at most
    // `capacity` rows
    int routed = 0;
    for (int e = lane; e < N; e += 32) {
      routed += s_off[e];
      if (capacity > 0 && s_off[e] > capacity) s_off[e] = capacity;
    }
    for (int o = 16; o > 0; o >>= 1) routed += __shfl_xor_sync(0xffffffffu, routed, o);
    __syncwarp();
    const int total = warp_exclusive_scan(s_off, N, lane);
    if (lane == 0) {
      s_off[N] = total;
      if (counts != nullptr && routed != P) set_status(status, MOE_ERR_DEVICE_CHECK);
    }
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e <= N; e += kGroupThreads) offsets[e] = s_off[e];
    if (seg != nullptr) write_seg_table(s_off, N, n_shared, T, P, tile_m, seg, s_seg);
  }
  // pass 1: per-warp counts of this block's experts
  int* mine = s_wc + warp * epb;  // mine[e - e_lo] for e in [e_lo, e_hi)
  for (int b0 = p0; b0 < p1; b0 += 32 * kGroupBatch) {
    int ev[kGroupBatch];
#pragma unroll
    for (int r = 0; r < kGroupBatch; ++r) {
      const int p = b0 + 32 * r + lane;
      ev[r] = p < p1 ? idx[p] : -1;
    }
#pragma unroll
    for (int r = 0; r < kGroupBatch; ++r) {
      const int e = ev[r];
      const bool own = e >= e_lo && e < e_hi;
      const uint32_t peers = __match_any_sync(0xffffffffu, own ? e : -1);
      if (own && lane == __ffs(peers) - 1) mine[e - e_lo] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < e_hi - e_lo; j += kGroupThreads) {
    int acc = 0;  // rank bases inside the expert
    for (int w = 0; w < kGroupWarps; ++w) {
      const int v = s_wc[w * epb + j];
      s_wc[w * epb + j] = acc;
      acc += v;
    }
  }
  __syncthreads();
  // pass 2: rows in pair order
  const uint32_t lt = lanemask_lt();
  for (int b0 = p0; b0 < p1; b0 += 32 * kGroupBatch) {
    int ev[kGroupBatch];
#pragma unroll
    for (int r = 0; r < kGroupBatch; ++r) {
      const int p = b0 + 32 * r + lane;
      ev[r] = p < p1 ? idx[p] : -1;
    }
#pragma unroll
    for (int r = 0; r < kGroupBatch; ++r) {
      const int p = b0 + 32 * r + lane;
      const int e = ev[r];
      if (blockIdx.x == 0 && p < p1 && e == kNoExpert) inv_pos[p] = -1;  // no expert: no row
      const bool own = e >= e_lo && e < e_hi;
      const uint32_t peers = __match_any_sync(0xffffffffu, own ? e : -1);
      if (own) {
        const int rank = mine[e - e_lo] + __popc(peers & lt);  // among expert e's pairs
        if (capacity == 0 || rank < capacity) {
          const int pos = s_off[e] + rank;
          sorted_pair[pos] = p;
          inv_pos[p] = pos;
        } else {
          inv_pos[p] = -1;  // dropped by the capacity
        }
      }
      __syncwarp();
      if (own && lane == __ffs(peers) - 1) mine[e - e_lo] += __popc(peers);
      __syncwarp();
    }
  }
}

// Segment table of the grouped GEMM from the expert offsets (one block).
// The offsets come from the caller when moe_grouped_swiglu is called on its
// own, so they are checked first: they must start at 0, never decrease and
// end at most at T*k. Otherwise the status word gets MOE_ERR_DEVICE_CHECK
// and the table holds zero tiles, so the GEMMs do no work.
constexpr int kSegThreads = 256;
__global__ void __launch_bounds__(kSegThreads) seg_table_kernel(
    const int32_t* __restrict__ offsets, int N, int n_shared, int T, int P, int tile_m,
    int32_t* seg, int* status) {
  extern __shared__ int sh[];
  int* off = sh;             // [N + 1]
  int* scratch = sh + N + 1; // [N + n_shared + 1]
  pdl_wait();
  pdl_trigger();
  int good = 1;
  for (int e = threadIdx.x; e <= N; e += kSegThreads) {
    off[e] = offsets[e];
    if (e == 0 && off[0] != 0) good = 0;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += kSegThreads)
    if (off[e + 1] < off[e]) good = 0;
  if (threadIdx.x == 0 && off[N] > P) good = 0;
  const bool ok = __syncthreads_and(good) != 0;
  if (!ok) {
    if (threadIdx.x == 0) set_status(status, MOE_ERR_DEVICE_CHECK);
    for (int e = threadIdx.x; e <= N; e += kSegThreads) off[e] = 0;  // no routed rows
    __syncthreads();
  }
  write_seg_table(off, N, n_shared, ok ? T : 0, P, tile_m, seg, scratch);
}

}  // namespace

size_t permute_scratch_bytes(const moe_config& c) {
  const long long P = (long long)c.T * c.top_k;
  return sizeof(int32_t) * (size_t)ceil_div(P, kChunk) * (size_t)c.n_experts;
}

cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* topk_idx,
                           const int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                           int32_t* inv_pos, void* x_perm, int32_t* chunk_hist, int* status,
                           int32_t* seg, int tile_m, cudaStream_t s) {
  const int N = c.n_experts;
  const int P = c.T * c.top_k;
  const int cap = c.capacity;
  if (P == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (N + 1), s);
  const int vec = (int)(c.d_model * elem_bytes(c.dtype) / 16);
  auto gather = [&]() {
    if (x_perm == nullptr) return cudaSuccess;  // the caller gathers (FP8 layer: with quantization)
    ProfScope p(K_PERMUTE_GATHER, s);
    return launch_pdl(permute_gather_kernel, dim3(ceil_div(c.T, kWarps)), dim3(kThreads), 0, s, 1,
                      static_cast<const uint4*>(x), (const int32_t*)inv_pos,
                      (const int32_t*)sorted_pair, c.T, P, c.top_k, vec,
                      static_cast<uint4*>(x_perm));
  };
  if (P <= kChunk) {
    const size_t smem = sizeof(int) * ((size_t)kSmallWarps * N + N + 1);
    {
      ProfScope p(K_PERMUTE_SMALL, s);
      cudaError_t e = launch_pdl(permute_small_kernel, dim3(1), dim3(kSmallThreads), smem, s, 1,
                                 topk_idx, P, N, cap, offsets, sorted_pair, inv_pos, status, seg,
                                 c.n_shared, c.T, tile_m);
      if (e != cudaSuccess) return e;
    }
    return gather();
  }
  if (P <= kGroupMaxPairs) {
    const int groups = N < kGroupBlocks ? N : kGroupBlocks;
    const int epb = ceil_div(N, groups);
    const size_t smem =
        sizeof(int) * ((size_t)N + 1 + (size_t)kGroupWarps * epb + N + c.n_shared + 1);
    {
      ProfScope p(K_PERMUTE_GROUP, s);
      cudaError_t e = launch_pdl(permute_group_kernel, dim3(ceil_div(N, epb)), dim3(kGroupThreads),
                                 smem, s, 1, topk_idx, counts, P, N, epb, cap, offsets, sorted_pair,
                                 inv_pos, status, seg, c.n_shared, c.T, tile_m);
      if (e != cudaSuccess) return e;
    }
    return gather();
  }
  const int nch = ceil_div(P, kChunk);
  cudaError_t e;
  {
    ProfScope p(K_PERMUTE_HIST, s);
    e = launch_pdl(permute_hist_kernel, dim3(nch), dim3(kThreads), sizeof(int) * N, s, 1, topk_idx,
                   P, N, chunk_hist, status);
    if (e != cudaSuccess) return e;
  }
  {
    ProfScope p(K_PERMUTE_SCAN, s);
    e = launch_pdl(permute_scan_kernel, dim3(1), dim3(kThreads), sizeof(int) * (N + 1), s, 1,
                   chunk_hist, nch, N, cap, offsets);
    if (e != cudaSuccess) return e;
  }
  {
    ProfScope p(K_PERMUTE_RANK, s);
    e = launch_pdl(permute_rank_kernel, dim3(nch), dim3(kThreads), sizeof(int) * kWarps * N, s, 1,
                   topk_idx, P, N, cap, (const int32_t*)chunk_hist, (const int32_t*)offsets,
                   sorted_pair, inv_pos);
    if (e != cudaSuccess) return e;
  }
  e = gather();
  if (e != cudaSuccess || seg == nullptr) return e;
  return launch_seg_table(c, offsets, seg, tile_m, status, s);
}

cudaError_t launch_seg_table(const moe_config& c, const int32_t* offsets, int32_t* seg,
                             int tile_m, int* status, cudaStream_t s) {
  ProfScope p(K_SEG_TABLE, s);
  const size_t smem = sizeof(int) * ((size_t)2 * c.n_experts + c.n_shared + 2);
  return launch_pdl(seg_table_kernel, dim3(1), dim3(kSegThreads), smem, s, 1, offsets, c.n_experts,
                    c.n_shared, c.T, c.T * c.top_k, tile_m, seg, status);
}

}  // namespace moe
