// The end of every router kernel: each block leaves its per-expert
// probability sums and counts in a [blocks][N] scratch, and the last block
// to finish adds them up into prob_sum and counts. Blocks are summed in a
// fixed order (thread j of an expert's group adds blocks j, j + G, j + 2G,
// ... in turn, then the group's G sums meet in a fixed xor butterfly), so
// the result does not depend on which block finished last, and no other
// launch or memset is needed.
#pragma once

#include <stdint.h>

#include "device_util.cuh"

namespace moe {

// Call from all NT threads of each of the nblk blocks that hold partials,
// after the block has written its row b of partials[nblk][N] and
// cpart[nblk][N]. `done` counts finished blocks and must be zero at launch.
template <int NT>
__device__ __forceinline__ void router_finish(const float* partials, const int32_t* cpart, int N,
                                              int nblk, float* prob_sum, int32_t* counts,
                                              int* done) {
  static_assert(NT % 32 == 0, "whole warps");
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(done, 1) == nblk - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // G threads per expert: a power of two up to 32 with G * N <= NT when possible
  int G = 1;
  while (G < 32 && 2 * G * N <= NT) G *= 2;
  const int per_pass = NT / G;
  const int j = threadIdx.x % G, gi = threadIdx.x / G;
  for (int e0 = 0; e0 < N; e0 += per_pass) {
    const int e = e0 + gi;
    float s = 0.f;
    int c = 0;
    if (e < N)
      for (int b = j; b < nblk; b += G) {
        s += __ldcg(partials + (size_t)b * N + e);
        c += __ldcg(cpart + (size_t)b * N + e);
      }
    for (int o = G / 2; o > 0; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    if (j == 0 && e < N) {
      prob_sum[e] = s;
      counts[e] = c;
    }
  }
}

}  // namespace moe
