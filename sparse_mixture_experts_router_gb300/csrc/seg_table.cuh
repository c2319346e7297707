// The grouped GEMM's segment table, written by the kernels that know the
// experts' row offsets (the permutation kernels and the decode-sized
// routing kernel), and the warp scan it is built with.
#pragma once

#include <stdint.h>

namespace moe {

// Exclusive scan of v[0..n) in place by one warp (32 at a time, carrying the
// running total); returns the total to every lane.
__device__ __forceinline__ int warp_exclusive_scan(int* v, int n, int lane) {
  int run = 0;
  for (int b = 0; b < n; b += 32) {
    const int x = (b + lane < n) ? v[b + lane] : 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (b + lane < n) v[b + lane] = run + incl - x;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  return run;
}

// Segment table of the grouped GEMM, [E, total tiles, mt_start[E+1],
// rows[E], a_row0[E], out_row0[E]], from the routed experts' offsets
// off[0..N] (shared experts take T rows of x each). Called by a whole block;
// `scratch` holds E + 1 ints of shared memory.
__device__ __forceinline__ void write_seg_table(const int* off, int N, int n_shared, int T, int P, int tile_m,
                                int32_t* seg, int* scratch) {
  const int E = N + n_shared;
  int32_t* mt_start = seg + 2;
  int32_t* rows = seg + 3 + E;
  int32_t* a_row0 = seg + 3 + 2 * E;
  int32_t* out_row0 = seg + 3 + 3 * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int r = e < N ? off[e + 1] - off[e] : T;
    rows[e] = r;
    a_row0[e] = e < N ? off[e] : 0;
    out_row0[e] = e < N ? off[e] : P + (e - N) * T;
    scratch[e] = (r + tile_m - 1) / tile_m;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int total = warp_exclusive_scan(scratch, E, threadIdx.x);
    if (threadIdx.x == 0) {
      scratch[E] = total;
      seg[0] = E;
      seg[1] = total;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) mt_start[e] = scratch[e];
}

}  // namespace moe
