// K2: grouping of the (token, slot) pairs by expert, and the row gather.
//
// The batched form of the per-expert dispatch loop of the pages' toy layers
// ("Mixture of experts and speculative decoding", "A toy MoE layer in
// PyTorch"; "Mixture of Experts and Guided Decoding", sparse MoE code):
// every pair that chose expert e lands in e's contiguous row segment, in
// ascending pair order, so the result is unique and bit-exact.
//
// Four launches (one single-block kernel when all pairs fit one chunk):
//  hist   - one block per chunk of 2048 pairs counts pairs per expert with
//           warp-aggregated shared-memory atomics (one atomic per distinct
//           expert in a warp, found with __match_any_sync).
//  scan   - one block: per expert, exclusive scan of the chunk counts; then
//           the exclusive scan over experts gives expert_offsets; the chunk
//           table becomes each chunk's first row per expert.
//  rank   - one block per chunk: per-warp counts, a scan over the 8 warps,
//           then each warp walks its 256 pairs in order, 32 at a time; a
//           pair's row is its warp base + the number of lower lanes with the
//           same expert (__match_any_sync + popc of the lane mask).
//  gather - one warp per output row copies the token row with 16-byte loads
//           and stores.
#include "device_util.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = kPermuteChunk;            // 2048 pairs
constexpr int kPerWarp = kChunk / kWarps;        // 256 pairs
constexpr int kRounds = kPerWarp / 32;           // 8

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
        set_status(status, MOE_ERR_DEVICE_CHECK);
        e = -1;
      }
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&sh[e], __popc(peers));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += kThreads) hist[(size_t)blockIdx.x * N + e] = sh[e];
}

__global__ void __launch_bounds__(kThreads) permute_scan_kernel(int32_t* hist, int nchunks, int N,
                                                                int32_t* offsets) {
  extern __shared__ int tot[];
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < N; e += kThreads) {
    int run = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int v = hist[(size_t)c * N + e];
      hist[(size_t)c * N + e] = run;
      run += v;
    }
    tot[e] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < N; ++e) {
      const int v = tot[e];
      tot[e] = run;
      offsets[e] = run;
      run += v;
    }
    offsets[N] = run;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += kThreads)
    for (int c = 0; c < nchunks; ++c) hist[(size_t)c * N + e] += tot[e];
}

__global__ void __launch_bounds__(kThreads) permute_rank_kernel(const int32_t* __restrict__ idx,
                                                                int P, int N,
                                                                const int32_t* __restrict__ chunk_base,
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
    int e = (p < P) ? idx[p] : -1;
    if (e >= N) e = -1;
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
      const int pos = mine[e] + __popc(peers & lt);
      sorted_pair[pos] = p;
      inv_pos[p] = pos;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
}

// One warp per output row: x_perm[row] = x[sorted_pair[row] / k].
__global__ void __launch_bounds__(kThreads) permute_gather_kernel(const uint4* __restrict__ x,
                                                                  const int32_t* __restrict__ sorted_pair,
                                                                  int P, int k, int vec_per_row,
                                                                  uint4* __restrict__ x_perm) {
  const int row = blockIdx.x * kWarps + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  pdl_wait();
  pdl_trigger();
  if (row >= P) return;
  // Rows past the last valid pair stay unwritten when some expert index was
  // out of range (already reported in the status word); never read through
  // such a row.
  const int pair = sorted_pair[row];
  if (pair < 0 || pair >= P) return;
  const int t = pair / k;
  const uint4* src = x + (size_t)t * vec_per_row;
  uint4* dst = x_perm + (size_t)row * vec_per_row;
#pragma unroll 4
  for (int i = lane; i < vec_per_row; i += 32) dst[i] = __ldg(src + i);
}

// The counting, scans and stable ranks of the permutation (and optionally
// the grouped GEMM's segment table) in one block when the T*k pairs fit one
// chunk (decode-sized batches): two launches (this and the row gather)
// instead of five. Same results as the multi-block path.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;
__global__ void __launch_bounds__(kSmallThreads) permute_small_kernel(
    const int32_t* __restrict__ idx, int P, int N, int k, const uint4* __restrict__ x,
    int vec_per_row, uint4* __restrict__ x_perm, int32_t* offsets, int32_t* sorted_pair,
    int32_t* inv_pos, int* status, int32_t* seg, int n_shared, int T, int tile_m) {
  (void)x; (void)vec_per_row; (void)x_perm; (void)k;
  extern __shared__ int sh[];
  int* wh = sh;                        // [kSmallWarps][N] counts, then row bases
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
      if (e < 0 || e >= N) {
        set_status(status, MOE_ERR_DEVICE_CHECK);
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
    soff[e] = tot;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < N; ++e) {
      const int v = soff[e];
      soff[e] = run;
      offsets[e] = run;
      run += v;
    }
    soff[N] = run;
    offsets[N] = run;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += kSmallThreads) {
    int base = soff[e];
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
    if (e >= N) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int pos = mine[e] + __popc(peers & lt);
      sorted_pair[pos] = p;
      inv_pos[p] = pos;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  if (seg != nullptr) {  // segment table of the grouped GEMM (as seg_table_kernel)
    const int E = N + n_shared;
    int32_t* mt_start = seg + 2;
    int32_t* rows = seg + 3 + E;
    int32_t* a_row0 = seg + 3 + 2 * E;
    int32_t* out_row0 = seg + 3 + 3 * E;
    for (int e = threadIdx.x; e < E; e += kSmallThreads) {
      rows[e] = e < N ? soff[e + 1] - soff[e] : T;
      a_row0[e] = e < N ? soff[e] : 0;
      out_row0[e] = e < N ? soff[e] : P + (e - N) * T;
    }
    if (threadIdx.x == 0) {
      int run = 0;
      for (int e = 0; e < E; ++e) {
        mt_start[e] = run;
        const int r = e < N ? soff[e + 1] - soff[e] : T;
        run += (r + tile_m - 1) / tile_m;
      }
      mt_start[E] = run;
      seg[0] = E;
      seg[1] = run;
    }
  }
}

// Segment table of the grouped GEMM from the expert offsets (one block).
// The offsets come from the caller when moe_grouped_swiglu is called on its
// own, so they are checked first: they must start at 0, never decrease and
// end at most at T*k. Otherwise the status word gets MOE_ERR_DEVICE_CHECK
// and the table holds zero tiles, so the GEMMs do no work.
__global__ void seg_table_kernel(const int32_t* __restrict__ offsets, int N, int n_shared, int T,
                                 int P, int tile_m, int32_t* seg, int* status) {
  __shared__ int ok;
  const int E = N + n_shared;
  pdl_wait();
  pdl_trigger();
  int32_t* mt_start = seg + 2;
  int32_t* rows = seg + 3 + E;
  int32_t* a_row0 = seg + 3 + 2 * E;
  int32_t* out_row0 = seg + 3 + 3 * E;
  if (threadIdx.x == 0) {
    int good = offsets[0] == 0 && offsets[N] <= P;
    for (int e = 0; e < N && good; ++e) good = offsets[e + 1] >= offsets[e];
    ok = good;
    if (!good) set_status(status, MOE_ERR_DEVICE_CHECK);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    if (e < N) {
      rows[e] = ok ? offsets[e + 1] - offsets[e] : 0;
      a_row0[e] = ok ? offsets[e] : 0;
      out_row0[e] = ok ? offsets[e] : 0;
    } else {
      rows[e] = ok ? T : 0;
      a_row0[e] = 0;
      out_row0[e] = P + (e - N) * T;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      mt_start[e] = run;
      run += (rows[e] + tile_m - 1) / tile_m;
    }
    mt_start[E] = run;
    seg[0] = E;
    seg[1] = run;
  }
}

}  // namespace

size_t permute_scratch_bytes(const moe_config& c) {
  const long long P = (long long)c.T * c.top_k;
  return sizeof(int32_t) * (size_t)ceil_div(P, kChunk) * (size_t)c.n_experts;
}

cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* topk_idx,
                           int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos,
                           void* x_perm, int32_t* chunk_hist, int* status, int32_t* seg,
                           int tile_m, cudaStream_t s) {
  const int N = c.n_experts;
  const int P = c.T * c.top_k;
  if (P == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (N + 1), s);
  if (P <= kChunk) {
    const int vec = (int)(c.d_model * elem_bytes(c.dtype) / 16);
    const size_t smem = sizeof(int) * ((size_t)kSmallWarps * N + N + 1);
    {
      ProfScope p(K_PERMUTE_SMALL, s);
      cudaError_t e = launch_pdl(permute_small_kernel, dim3(1), dim3(kSmallThreads), smem, s, 1,
                                 topk_idx, P, N, c.top_k, static_cast<const uint4*>(x), vec,
                                 static_cast<uint4*>(x_perm), offsets, sorted_pair, inv_pos, status,
                                 seg, c.n_shared, c.T, tile_m);
      if (e != cudaSuccess) return e;
    }
    ProfScope p(K_PERMUTE_GATHER, s);
    return launch_pdl(permute_gather_kernel, dim3(ceil_div(P, kWarps)), dim3(kThreads), 0, s, 1,
                      static_cast<const uint4*>(x), sorted_pair, P, c.top_k, vec,
                      static_cast<uint4*>(x_perm));
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
    e = launch_pdl(permute_scan_kernel, dim3(1), dim3(kThreads), sizeof(int) * N, s, 1, chunk_hist,
                   nch, N, offsets);
    if (e != cudaSuccess) return e;
  }
  {
    ProfScope p(K_PERMUTE_RANK, s);
    e = launch_pdl(permute_rank_kernel, dim3(nch), dim3(kThreads), sizeof(int) * kWarps * N, s, 1,
                   topk_idx, P, N, (const int32_t*)chunk_hist, sorted_pair, inv_pos);
    if (e != cudaSuccess) return e;
  }
  {
    const int vec = (int)(c.d_model * elem_bytes(c.dtype) / 16);
    ProfScope p(K_PERMUTE_GATHER, s);
    e = launch_pdl(permute_gather_kernel, dim3(ceil_div(P, kWarps)), dim3(kThreads), 0, s, 1,
                   static_cast<const uint4*>(x), (const int32_t*)sorted_pair, P, c.top_k, vec,
                   static_cast<uint4*>(x_perm));
  }
  if (e != cudaSuccess || seg == nullptr) return e;
  return launch_seg_table(c, offsets, seg, tile_m, status, s);
}

cudaError_t launch_seg_table(const moe_config& c, const int32_t* offsets, int32_t* seg,
                             int tile_m, int* status, cudaStream_t s) {
  ProfScope p(K_SEG_TABLE, s);
  return launch_pdl(seg_table_kernel, dim3(1), dim3(256), 0, s, 1, offsets, c.n_experts, c.n_shared,
                    c.T, c.T * c.top_k, tile_m, seg, status);
}

}  // namespace moe
