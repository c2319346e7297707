// Top-k selection on packed 64-bit keys for the tensor-core router: a key and its expert index become one word that orders by key
// and then by lower index, so a plain unsigned comparison decides both, and
// small comparator networks keep the 8 largest words of a thread's scores.
#pragma once

#include <math.h>
#include <stdint.h>

namespace moe {

constexpr int kKeyIndexBase = 255;  // index stored as kKeyIndexBase - e (e <= 255)

// Selection key -> 64-bit word: larger word = larger key, then lower index.
// NaN ranks as -inf and -0 as +0, as the comparisons of the keys would have it.
__device__ __forceinline__ uint64_t pack_key(float key, int e) {
  if (key != key) key = -INFINITY;
  if (key == 0.f) key = 0.f;
  const uint32_t b = __float_as_uint(key);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)ord << 32) | (uint32_t)(kKeyIndexBase - e);
}

// Compare-exchange putting the larger word first.
__device__ __forceinline__ void cex(uint64_t& a, uint64_t& b) {
  const bool sw = b > a;
  const uint64_t hi = sw ? b : a;
  b = sw ? a : b;
  a = hi;
}
// Sorts 8 words into descending order: 19 comparators in 6 layers (a
// standard minimal network, checked on all 0/1 inputs).
__device__ __forceinline__ void sort8(uint64_t (&c)[8]) {
  cex(c[0], c[2]); cex(c[1], c[3]); cex(c[4], c[6]); cex(c[5], c[7]);
  cex(c[0], c[4]); cex(c[1], c[5]); cex(c[2], c[6]); cex(c[3], c[7]);
  cex(c[0], c[1]); cex(c[2], c[3]); cex(c[4], c[5]); cex(c[6], c[7]);
  cex(c[2], c[4]); cex(c[3], c[5]);
  cex(c[1], c[4]); cex(c[3], c[6]);
  cex(c[1], c[2]); cex(c[3], c[4]); cex(c[5], c[6]);
}
// L (sorted descending) <- the 8 largest of L and c (c sorted descending):
// max(L[i], c[7-i]) holds exactly those 8 as a bitonic sequence, which three
// half-cleaner layers sort.
__device__ __forceinline__ void merge_top8(uint64_t (&L)[8], const uint64_t (&c)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) L[i] = c[7 - i] > L[i] ? c[7 - i] : L[i];
  cex(L[0], L[4]); cex(L[1], L[5]); cex(L[2], L[6]); cex(L[3], L[7]);
  cex(L[0], L[2]); cex(L[1], L[3]); cex(L[4], L[6]); cex(L[5], L[7]);
  cex(L[0], L[1]); cex(L[2], L[3]); cex(L[4], L[5]); cex(L[6], L[7]);
}

// Expert index of a packed word.
__device__ __forceinline__ int key_index(uint64_t w) { return kKeyIndexBase - (int)(uint32_t)w; }

}  // namespace moe
