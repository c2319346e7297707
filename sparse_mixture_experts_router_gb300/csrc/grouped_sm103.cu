// K3/K4: grouped SwiGLU expert GEMMs on the 5th-generation tensor cores.
//
// Every expert of the layer is an ordinary SwiGLU FFN ("MoE inference: the
// call centre with 256 specialists and 8 taking each call", "The bare
// mechanism"; read as down(SiLU(gate(x)) * up(x))). After the permutation,
// expert e owns a contiguous, ragged segment of rows, so all experts run as
// one grouped GEMM per projection:
//
//   gate/up  H[row]  = SiLU(A[row] Wg[e]^T) * (A[row] Wu[e]^T)     (bf16 out)
//   down     Yp[row] = w_row * (H[row] Wd[e]^T)                    (bf16 out)
//
// with A = x_perm for routed experts and A = x for shared experts, w_row the
// row's gate weight (1 for shared rows). This is the layer's main dense
// contraction ("Mixture of experts and speculative decoding": an expert
// costs about 2 flops per parameter); the router's score contraction for
// many experts is the only other one (router_tc.cu).
//
// Design (sm_103a, one CTA per SM, persistent):
//  - Tiles: 128 rows of one segment x 256 accumulator columns. For gate/up
//    the B tile stacks 128 gate rows over the matching 128 up rows, so one
//    128x256x16 tcgen05.mma computes both projections into one TMEM
//    accumulator; the epilogue pairs column j with column 128+j. For down the
//    256 columns are 256 output features.
//  - Tile list: segment-major, then N tile, then M tile (fastest), so the
//    CTAs running at the same time share weight tiles through L2. CTA b takes
//    tiles b, b+grid, ...; the list length and segment table live on the
//    device (no host synchronisation on the routing). Rows of a tile past its
//    segment's end are computed on whatever rows follow and never stored.
//  - Warp roles (320 threads): warp 0 issues TMA loads (128-byte swizzle,
//    64-wide K blocks) into a 4-stage shared-memory ring; warp 1 allocates
//    512 TMEM columns (two 256-column accumulators) and issues tcgen05.mma
//    from one thread, releasing ring slots and publishing finished
//    accumulators with tcgen05.commit; warps 2-9 drain an accumulator with
//    tcgen05.ld (each warp owns the 32 TMEM lanes its index allows, two
//    warps per lane quarter, each taking half the columns), apply the SwiGLU
//    or gate-weight epilogue and store bf16 rows, while the MMA warp fills
//    the other accumulator.
//  - NVFP4 operands (OP_NVF4, 1-CTA tiles, 448 threads): stages also carry
//    the E4M3 block scales of their A and B rows; four more warps, one per
//    TMEM lane quarter, write them into Tensor Memory with tcgen05.st, where
//    the block-scaled MMA (kind::mxf4nvf4) reads them. The scales take 128
//    TMEM columns, so two 256-column accumulators do not fit: consecutive
//    tiles alternate between columns [0, 256) and [128, 384), the epilogue
//    drains the shared middle 128 columns first and frees them as soon as
//    its tcgen05.ld has landed, and the next tile's MMAs start then.
//  - Every wait is bounded (2 s of %globaltimer). A wait that runs out
//    records MOE_ERR_TIMEOUT in the status word and sets a shared abort flag
//    that ends the other roles' loops; the producer then waits (bounded) for
//    its own TMA copies in flight, the MMA thread for its own MMAs, and TMEM
//    is freed before the CTA exits.
#include <cuda.h>

#include <algorithm>
#include <type_traits>
#include <mutex>

#include "device_util.cuh"
#include "moe_internal.h"
#include "sm103_ptx.cuh"
#include "sm103_wait.cuh"

namespace moe {
namespace {

constexpr int BM = kTileM;       // 128 rows
constexpr int BK = 64;           // 64 bf16 = one 128-byte swizzle row
constexpr int BN = 256;          // accumulator columns per tile
constexpr int UMMA_K = 16;       // K of one tcgen05.mma kind::f16
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;           // 16 KB
constexpr int B_HALF_BYTES = 128 * BK * 2;     // 16 KB
constexpr int B_BYTES = BN * BK * 2;           // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES; // 48 KB
constexpr int NUM_ACC = 2;
constexpr int TMEM_COLS = BN * NUM_ACC;        // 512
constexpr int THREADS = 192;      // decode kernel: producer, MMA, 4 epilogue warps
constexpr int EPI_THREADS = 128;
// Grouped and pair kernels: two epilogue warps per TMEM lane quarter, each
// draining half of the accumulator's columns, so the epilogue keeps up with
// the MMA at the E4M3 rate.
constexpr int EPI_WARPS = 8;
constexpr int G_EPI_THREADS = 32 * EPI_WARPS;  // 256
constexpr int G_THREADS = 64 + G_EPI_THREADS;  // 320

// Epilogues. The forward's two, and the backward's (1-CTA kernel only):
//  EPI_SWIGLU_SAVE  gate/up as EPI_SWIGLU, also storing the pre-activations
//                   a | b (bf16) in aux [rows][2 * n_out];
//  EPI_SWIGLU_BWD   dH = dO W_d (B MN-major) and, per element, the SwiGLU
//                   backward: da = dH * b * SiLU'(a), db = dH * SiLU(a) from
//                   aux, stored as da | db in out [rows][2 * n_out];
//  EPI_DGRAD        dA = [da | db] [W_g ; W_u] (B MN-major, K = 2 d_ff,
//                   W_g rows for the first kb_split K blocks), stored plain.
enum { EPI_SWIGLU = 0, EPI_DOWN = 1, EPI_SWIGLU_SAVE = 2, EPI_SWIGLU_BWD = 3, EPI_DGRAD = 4 };
// gate/up layout: B stacks 128 gate rows over 128 up rows; 128 output columns
__host__ __device__ constexpr bool gu_like(int EPI) {
  return EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_SAVE;
}
// B stored MN-major (K rows of an expert's weight, N columns contiguous)
__host__ __device__ constexpr bool b_mn(int EPI) {
  return EPI == EPI_SWIGLU_BWD || EPI == EPI_DGRAD;
}
constexpr int B_MN_BOX_BYTES = 64 * 128;  // one TMA box: 64 K rows x 64 bf16 columns

// Operand types. A stage row is 128 bytes in every case: 64 bf16, 128 E4M3
// or 256 packed E2M1 (NVFP4) elements of K, and one MMA takes 32 bytes of K
// (16 bf16 with kind::f16, 32 E4M3 with kind::f8f6f4, 64 E2M1 with
// kind::mxf4nvf4), so rings, descriptors and K steps are shared; the K
// extent of a block, the instruction and the epilogue scales (E4M3 and
// NVFP4: one fp32 scale per A row and per weight output channel) differ.
// NVFP4 stages also carry the E4M3 block scales of their 256 K elements
// (16 a row: 2 KB for A, 4 KB for B), which the MMA reads from Tensor
// Memory; they take 128 TMEM columns, so the NVFP4 kernel's consecutive
// accumulators share columns (the regions below; 1-CTA tiles only).
enum { OP_BF16 = 0, OP_E4M3 = 1, OP_NVF4 = 2 };
template <int OP>
struct Op {
  static constexpr int EPK = OP == OP_BF16 ? 64 : OP == OP_E4M3 ? 128 : 256;  // K per block
  static constexpr int KC = OP == OP_BF16 ? 64 : 128;  // TMA inner coordinate step per block
  static constexpr bool scaled = OP != OP_BF16;        // row and channel scales in the epilogue
  static constexpr int SF_A = OP == OP_NVF4 ? BM * 16 : 0;
  static constexpr int SF_B = OP == OP_NVF4 ? BN * 16 : 0;
  static constexpr int STAGE = STAGE_BYTES + SF_A + SF_B;  // 48 KB, or 54 KB for NVFP4
  // NVFP4: one accumulator-full phase a unit; where its accumulator lies
  // rotates through the TMEM regions below
  static constexpr int NACC = OP == OP_NVF4 ? 1 : NUM_ACC;
  static constexpr size_t SMEM = (size_t)STAGES * STAGE + 1024;  // + 1 KB alignment slack
  // NVFP4 adds four warps (the last), one per TMEM lane quarter, that write
  // each stage's block scales into Tensor Memory
  static constexpr int THREADS = G_THREADS + (OP == OP_NVF4 ? 128 : 0);
};
// TMEM columns of the NVFP4 block scales: two buffers (alternate K blocks)
// of 64 columns after the accumulator regions, A's 16 then B's 32 (4 and 8
// a MMA).
// NVFP4 accumulators: three 128-column regions R0-R2 = columns [0, 384);
// the scale buffers follow. Even work units of a CTA accumulate in R0-R1
// (columns 0-255), odd ones in R1-R2 (128-383). The epilogue drains R1
// first and frees each region once its tcgen05.ld has landed, so a unit's
// MMAs wait only for that first load of the previous unit (the other
// region was freed a unit earlier).
constexpr int NVF4_REGION_COLS = 128;
constexpr int SF_TMEM_COL = 3 * NVF4_REGION_COLS;
constexpr int SF_TMEM_BUF = 64;
static_assert(SF_TMEM_COL + 2 * SF_TMEM_BUF == TMEM_COLS, "TMEM columns");
template <int OP>
__host__ __device__ constexpr uint32_t idesc_op(int M, int N) {
  return OP == OP_BF16 ? ptx::idesc_bf16_f32(M, N)
         : OP == OP_E4M3 ? ptx::idesc_e4m3_f32(M, N)
                         : ptx::idesc_nvf4_f32(M, N);
}
template <int OP>
__device__ __forceinline__ void mma_op(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  if constexpr (OP == OP_BF16)
    ptx::mma_bf16(d, a, b, idesc, accumulate);
  else
    ptx::mma_e4m3(d, a, b, idesc, accumulate);
}
template <int OP>
__device__ __forceinline__ void mma_op_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  if constexpr (OP == OP_BF16)
    ptx::mma_bf16_pair(d, a, b, idesc, accumulate);
  else
    ptx::mma_e4m3_pair(d, a, b, idesc, accumulate);
}

struct GemmArgs {
  const int32_t* seg;          // segment table (moe_internal.h)
  const int32_t* sorted_pair;  // down: row -> pair id (may be null when topk_w is null)
  const float* topk_w;         // down: pair -> gate weight, or null
  void* out;                   // bf16 [rows][ldo]
  int* status;
  long long ldo;
  int n_routed;
  int n_pairs;                 // T*k, bound for sorted_pair values
  int K;                       // reduction length
  int n_out;                   // valid output columns
  int NT;                      // N tiles per segment
  int b_rows;                  // rows of one expert's weight matrix
  // split-K (few tiles, e.g. decode): fp32 partial rows of every split
  float* partial;              // [s_max][R][pc] fp32, or null when s_max == 1
  int s_max;                   // largest split factor the partial buffer holds
  int pc;                      // partial columns (2*d_ff for gate/up, d for down)
  long long R;                 // output rows
  // E4M3 operands only (null otherwise): the fp32 scale of every A row
  // (routed rows; the shared experts' token rows), of every weight output
  // channel [E][b_rows] (gate or down; up), and, for gate/up, the running
  // max |H| of every output row (fp32 bits, for the H quantization).
  const float* a_scale;
  const float* a_scale_shared;
  const float* b_scale0;
  const float* b_scale1;
  unsigned* h_amax;
  // Backward epilogues: bf16 [rows][2 * n_out] pre-activations a | b
  // (written by EPI_SWIGLU_SAVE, read by EPI_SWIGLU_BWD), and for MN-major B
  // the K blocks taken from map_b0 before map_b1 (EPI_DGRAD: d_ff / 64).
  __nv_bfloat16* aux;
  long long ld_aux;
  int kb_split;
  // Gate/up with the row gather fused (weight-stationary pairs, bf16): the
  // tokens x [T][K] and top-k; the B rows come from x through sorted_pair.
  const __nv_bfloat16* gx;
  int gk;
  int gT;
};

struct __align__(8) SharedState {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t sf_ready[STAGES];  // NVFP4: the stage's block scales are in Tensor Memory
  uint64_t acc_full[NUM_ACC];
  uint64_t acc_empty[NUM_ACC];
  uint64_t slot_empty[3];  // NVFP4: accumulator regions R0-R2 are free
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct Tile {
  int s, m, n;
};

// Segment-major, N tile, then M tile fastest (see file comment).
__device__ __forceinline__ Tile decode_tile(const int32_t* __restrict__ seg, int E, int NT,
                                            int tile) {
  const int32_t* mts = seg + 2;
  int lo = 0, hi = E;  // invariant: mts[lo]*NT <= tile < mts[hi]*NT
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(mts + mid) * NT <= tile) lo = mid;
    else hi = mid;
  }
  const int m0 = __ldg(mts + lo);
  const int mt = __ldg(mts + lo + 1) - m0;
  const int local = tile - m0 * NT;
  return Tile{lo, local % mt, local / mt};
}

// SiLU(g) = g * sigmoid(g). The quotient is the fast reciprocal-multiply
// (a few ulp in fp32, far below the bf16 rounding of the result); as g goes
// to -inf the divisor overflows to inf and the result goes to -0, the limit.
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }
__device__ __forceinline__ float sigmoid(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }

// Eight consecutive channel scales times a row scale, from two warp-uniform
// 16-byte loads (p 16-byte aligned); zeros when the group is past the output.
__device__ __forceinline__ void load_scales8(const float* p, bool in, float row, float (&s)[8]) {
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
  if (in) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  s[0] = row * a.x;
  s[1] = row * a.y;
  s[2] = row * a.z;
  s[3] = row * a.w;
  s[4] = row * b.x;
  s[5] = row * b.y;
  s[6] = row * b.z;
  s[7] = row * b.w;
}

// The same from this warp's staged copy of the tile's channel scales in
// shared memory (zeros past the output already in place).
__device__ __forceinline__ void staged_scales8(const float* p, float row, float (&s)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  s[0] = row * a.x;
  s[1] = row * a.y;
  s[2] = row * a.z;
  s[3] = row * a.w;
  s[4] = row * b.x;
  s[5] = row * b.y;
  s[6] = row * b.z;
  s[7] = row * b.w;
}

// Split factor of every tile when there are fewer tiles than two waves of
// CTAs: among S in [1, s_max] with at least kMinKbPerSplit K blocks per
// split, the largest whose wave efficiency (units / whole waves of the grid)
// is within 3% of the best; more, shorter units keep more weight bytes in
// flight per SM, which is what decode-sized GEMMs are bound by. Every CTA
// computes the same value.
constexpr int kMinKbPerSplit = 8;
__device__ __forceinline__ int choose_splits(int tiles, int grid, int KB, int s_max) {
  if (s_max <= 1 || tiles <= 0 || tiles >= 2 * grid) return 1;
  // tiles < 2 * grid here, so tiles * S stays far inside 32 bits; each split
  // factor's wave efficiency once (candidates: S <= s_max with at least
  // kMinKbPerSplit K blocks a split, a condition that holds for a prefix of S)
  float eff[kMaxSplitK + 1];
  float best = 0.f;
#pragma unroll
  for (int S = 1; S <= kMaxSplitK; ++S) {
    eff[S] = -1.f;
    if (S == 1 || (S <= s_max && KB / S >= kMinKbPerSplit)) {
      const int units = tiles * S;
      eff[S] = (float)units / (float)((units + grid - 1) / grid * grid);
      best = fmaxf(best, eff[S]);
    }
  }
  int pick = 1;
#pragma unroll
  for (int S = 2; S <= kMaxSplitK; ++S)
    if (eff[S] >= 0.f && eff[S] >= best - 0.03f) pick = S;
  return pick;
}
__device__ __forceinline__ int kb_begin(int split, int S, int KB) {
  return (int)(((long long)split * KB) / S);
}

// Gate weight of an output row of the down projection (1 for shared rows
// and when no weights are given; 0 for a pair id out of range).
__device__ __forceinline__ float row_scale(const GemmArgs& a, int seg_id, long long orow) {
  if (seg_id >= a.n_routed || !a.topk_w) return 1.0f;
  const int pair = __ldg(a.sorted_pair + orow);
  return (pair >= 0 && pair < a.n_pairs) ? __ldg(a.topk_w + pair) : 0.0f;
}

// The fused epilogue of one 128-row accumulator: each thread drains its
// TMEM lane (row) 32 columns at a time and stores bf16 (SwiGLU of the paired
// gate/up columns, or the gate-weighted down projection). Two warps share a
// lane quarter; `half` picks which half of the columns this one drains. Rows
// past the segment's end (valid = false) are loaded but not stored. gw is
// the row's gate weight (down projection). E4M3 and NVFP4: sa is the row's
// A scale and sb0/sb1 point at the tile's first weight channel scale (gate,
// up; or down), or, when `ss` is given, the 128 channel scales of this
// warp's columns are staged there (gate/up: 64 gate then 64 up; down: 128);
// gate/up also records the row's max |H|.
template <int EPI, int OP>
__device__ __forceinline__ void epilogue_fused(const GemmArgs& args, uint32_t tbase, const Tile& t,
                                               int half, bool valid, long long orow,
                                               __nv_bfloat16* out, float sa, const float* sb0,
                                               const float* sb1, float gw,
                                               const float* ss = nullptr) {
  if constexpr (gu_like(EPI)) {
    float hmax = 0.f;
#pragma unroll 1
    for (int c = 2 * half; c < 2 * half + 2; ++c) {
      uint32_t g[32], u[32];
      ptx::tmem_ld32(tbase + c * 32, g);
      ptx::tmem_ld32(tbase + 128 + c * 32, u);
      const int col0 = t.n * 128 + c * 32;
      ptx::tmem_ld_wait();
      uint32_t pk[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // E4M3: the 8 gate and 8 up channel scales of this column group, one
        // warp-uniform 16-byte load each (n_out is a multiple of 16, so a
        // group is wholly inside or wholly past it)
        float sg[8], su[8];
        if constexpr (Op<OP>::scaled) {
          if (ss) {
            staged_scales8(ss + (c - 2 * half) * 32 + q * 8, sa, sg);
            staged_scales8(ss + 64 + (c - 2 * half) * 32 + q * 8, sa, su);
          } else {
            const bool in = col0 + q * 8 < args.n_out;
            load_scales8(sb0 + c * 32 + q * 8, in, sa, sg);
            load_scales8(sb1 + c * 32 + q * 8, in, sa, su);
          }
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * q + jj;
          float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
          float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
          if constexpr (Op<OP>::scaled) {
            g0 *= sg[2 * jj];
            g1 *= sg[2 * jj + 1];
            u0 *= su[2 * jj];
            u1 *= su[2 * jj + 1];
          }
          pk[j] = f32x2_to_bf16x2(silu(g0) * u0, silu(g1) * u1);
          if constexpr (Op<OP>::scaled) {
            float h0, h1;
            bf16x2_to_f32(pk[j], h0, h1);
            hmax = fmaxf(hmax, fmaxf(fabsf(h0), fabsf(h1)));
          }
        }
      }
      if (valid) {
        __nv_bfloat16* dst = out + orow * args.ldo + col0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (col0 + q * 8 < args.n_out)
            *reinterpret_cast<uint4*>(dst + q * 8) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        if constexpr (EPI == EPI_SWIGLU_SAVE) {  // the pre-activations a | b, bf16
          __nv_bfloat16* pa = args.aux + orow * args.ld_aux + col0;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (col0 + q * 8 >= args.n_out) continue;
            uint32_t wa[4], wb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = 8 * q + 2 * i;
              wa[i] = f32x2_to_bf16x2(__uint_as_float(g[j]), __uint_as_float(g[j + 1]));
              wb[i] = f32x2_to_bf16x2(__uint_as_float(u[j]), __uint_as_float(u[j + 1]));
            }
            *reinterpret_cast<uint4*>(pa + q * 8) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
            *reinterpret_cast<uint4*>(pa + args.n_out + q * 8) =
                make_uint4(wb[0], wb[1], wb[2], wb[3]);
          }
        }
      }
    }
    if constexpr (Op<OP>::scaled)
      if (valid && hmax > 0.f) atomicMax(args.h_amax + orow, __float_as_uint(hmax));
  } else if constexpr (EPI == EPI_SWIGLU_BWD) {
#pragma unroll 1
    for (int c = 4 * half; c < 4 * half + 4; ++c) {
      uint32_t v[32];
      ptx::tmem_ld32(tbase + c * 32, v);
      const int col0 = t.n * 256 + c * 32;
      const bool in = valid && col0 < args.n_out;  // n_out is a multiple of 64
      uint4 av[4], bv[4];
      if (in) {
        const __nv_bfloat16* pa = args.aux + orow * args.ld_aux + col0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          av[q] = __ldg(reinterpret_cast<const uint4*>(pa) + q);
          bv[q] = __ldg(reinterpret_cast<const uint4*>(pa + args.n_out) + q);
        }
      }
      ptx::tmem_ld_wait();
      if (in) {
        uint32_t pda[16], pdb[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t aw[4] = {av[q].x, av[q].y, av[q].z, av[q].w};
          const uint32_t bw[4] = {bv[q].x, bv[q].y, bv[q].z, bv[q].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a0, a1, b0, b1;
            bf16x2_to_f32(aw[i], a0, a1);
            bf16x2_to_f32(bw[i], b0, b1);
            const float dh0 = __uint_as_float(v[8 * q + 2 * i]);
            const float dh1 = __uint_as_float(v[8 * q + 2 * i + 1]);
            const float s0 = sigmoid(a0), s1 = sigmoid(a1);
            pda[4 * q + i] = f32x2_to_bf16x2(dh0 * b0 * s0 * (1.f + a0 * (1.f - s0)),
                                             dh1 * b1 * s1 * (1.f + a1 * (1.f - s1)));
            pdb[4 * q + i] = f32x2_to_bf16x2(dh0 * a0 * s0, dh1 * a1 * s1);
          }
        }
        __nv_bfloat16* dst = out + orow * args.ldo + col0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          *reinterpret_cast<uint4*>(dst + q * 8) =
              make_uint4(pda[4 * q], pda[4 * q + 1], pda[4 * q + 2], pda[4 * q + 3]);
          *reinterpret_cast<uint4*>(dst + args.n_out + q * 8) =
              make_uint4(pdb[4 * q], pdb[4 * q + 1], pdb[4 * q + 2], pdb[4 * q + 3]);
        }
      }
    }
  } else {
    const float scale = valid ? gw * sa : 0.0f;
#pragma unroll 1
    for (int c = 4 * half; c < 4 * half + 4; ++c) {
      uint32_t v[32];
      ptx::tmem_ld32(tbase + c * 32, v);
      const int col0 = t.n * 256 + c * 32;
      ptx::tmem_ld_wait();
      uint32_t pk[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float sd[8];
        if constexpr (Op<OP>::scaled) {
          if (ss)
            staged_scales8(ss + (c - 4 * half) * 32 + q * 8, scale, sd);
          else
            load_scales8(sb0 + c * 32 + q * 8, col0 + q * 8 < args.n_out, scale, sd);
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * q + jj;
          float y0 = __uint_as_float(v[2 * j]), y1 = __uint_as_float(v[2 * j + 1]);
          if constexpr (Op<OP>::scaled) {
            y0 *= sd[2 * jj];
            y1 *= sd[2 * jj + 1];
          } else {
            y0 *= scale;
            y1 *= scale;
          }
          pk[j] = f32x2_to_bf16x2(y0, y1);
        }
      }
      if (valid) {
        __nv_bfloat16* dst = out + orow * args.ldo + col0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (col0 + q * 8 < args.n_out)
            *reinterpret_cast<uint4*>(dst + q * 8) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
  }
}

// NVFP4 epilogue of one work unit, whose accumulator's N halves (B rows
// 0-127 and 128-255 of the stages) lie in regions r0 and r0+1 (r0 = 0 for
// an even unit of the CTA, 1 for an odd one). The warp drains the half in
// R1 first and frees R1 (one arrival a thread) as soon as that load has
// landed, so the next unit's MMAs can start; the other region is freed
// after its last load. It scales, applies the SwiGLU or the gate weight and
// stores bf16, or, for a split-K unit (prow given), stores the scaled fp32
// partials. Gate/up: N half 0 holds the tile's 128 gate columns and half 1
// its up columns; the warp takes columns 64*half..64*half+63 of both, keeps
// the R1 half (up for an even unit, gate for an odd one) in registers and
// streams the other in 16 columns at a time. Down: N half i holds output
// columns 128i..128i+127; the warp takes 64 from 64*half. ss: the warp's
// 128 staged channel scales (gate/up: its 64 gate then 64 up columns; down:
// its 64 columns of half 0 then of half 1).
template <int EPI>
__device__ __forceinline__ void epilogue_nvf4(const GemmArgs& args, uint32_t tq, int r0,
                                              uint64_t* slot_empty, const Tile& t, int half,
                                              bool valid, long long orow, __nv_bfloat16* out,
                                              float sa, const float* sb0, const float* sb1,
                                              float gw, const float* ss, float* prow) {
  const int lane = threadIdx.x % 32;
  if constexpr (gu_like(EPI)) {
    const int second = r0 == 0 ? 0 : 2;  // the region of the half not in R1
    const uint32_t tk = tq + (uint32_t)NVF4_REGION_COLS + 64 * half;
    const uint32_t tw = tq + (uint32_t)(second * NVF4_REGION_COLS) + 64 * half;
    const int cw = 64 * half;  // the warp's first column of the tile
    const int col0 = t.n * 128 + cw;
    auto run = [&](auto up_first) {
      constexpr bool UF = decltype(up_first)::value;  // the kept half holds the up columns
      const float* sk = UF ? sb1 : sb0;
      const float* sw = UF ? sb0 : sb1;
      uint32_t k[2][32];
      ptx::tmem_ld32(tk, k[0]);
      ptx::tmem_ld32(tk + 32, k[1]);
      if (prow) {
        // split-K: lane l fetches the scales of column l of each 32
        float myk[2] = {0.f, 0.f}, myw[2] = {0.f, 0.f};
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
          if (col0 + 32 * cc + lane < args.n_out) {
            myk[cc] = __ldg(sk + cw + 32 * cc + lane);
            myw[cc] = __ldg(sw + cw + 32 * cc + lane);
          }
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_addr(&slot_empty[1]));
        float* pk_row = prow + (UF ? args.n_out : 0);
        float* pw_row = prow + (UF ? 0 : args.n_out);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t w[32];
          ptx::tmem_ld32(tw + 32 * cc, w);
          ptx::tmem_ld_wait();
          if (cc == 1) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_addr(&slot_empty[second]));
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float a[8], b[8];  // every lane takes part in the shuffles
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              a[e] = __uint_as_float(k[cc][8 * q + e]) * sa *
                     __shfl_sync(0xffffffffu, myk[cc], 8 * q + e);
              b[e] = __uint_as_float(w[8 * q + e]) * sa *
                     __shfl_sync(0xffffffffu, myw[cc], 8 * q + e);
            }
            const int c = col0 + 32 * cc + 8 * q;
            if (!valid || c >= args.n_out) continue;
            float4* dk = reinterpret_cast<float4*>(pk_row + c);
            float4* dw = reinterpret_cast<float4*>(pw_row + c);
            dk[0] = make_float4(a[0], a[1], a[2], a[3]);
            dk[1] = make_float4(a[4], a[5], a[6], a[7]);
            dw[0] = make_float4(b[0], b[1], b[2], b[3]);
            dw[1] = make_float4(b[4], b[5], b[6], b[7]);
          }
        }
        return;
      }
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_addr(&slot_empty[1]));
      // scale the kept half in place
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float s8[8];
          staged_scales8(ss + (UF ? 64 : 0) + 32 * cc + 8 * q, sa, s8);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            k[cc][8 * q + e] = __float_as_uint(__uint_as_float(k[cc][8 * q + e]) * s8[e]);
        }
      float hmax = 0.f;
#pragma unroll
      for (int p = 0; p < 4; ++p) {  // 16 columns of the streamed half at a time
        uint32_t w[16];
        ptx::tmem_ld16(tw + 16 * p, w);
        ptx::tmem_ld_wait();
        if (p == 3) {
          ptx::tc_fence_before();
          ptx::mbar_arrive(ptx::smem_addr(&slot_empty[second]));
        }
        uint32_t pk[8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float s8[8];
          staged_scales8(ss + (UF ? 0 : 64) + 16 * p + 8 * h, sa, s8);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int j = 8 * h + e;  // column 16p + j of the warp's 64
            const float w0 = __uint_as_float(w[j]) * s8[e];
            const float w1 = __uint_as_float(w[j + 1]) * s8[e + 1];
            const float k0 = __uint_as_float(k[p >> 1][16 * (p & 1) + j]);
            const float k1 = __uint_as_float(k[p >> 1][16 * (p & 1) + j + 1]);
            const float g0 = UF ? w0 : k0, g1 = UF ? w1 : k1;
            const float u0 = UF ? k0 : w0, u1 = UF ? k1 : w1;
            pk[j / 2] = f32x2_to_bf16x2(silu(g0) * u0, silu(g1) * u1);
            float h0, h1;
            bf16x2_to_f32(pk[j / 2], h0, h1);
            hmax = fmaxf(hmax, fmaxf(fabsf(h0), fabsf(h1)));
          }
        }
        if (valid) {
          __nv_bfloat16* dst = out + orow * args.ldo + col0 + 16 * p;
#pragma unroll
          for (int q = 0; q < 2; ++q)
            if (col0 + 16 * p + 8 * q < args.n_out)
              *reinterpret_cast<uint4*>(dst + 8 * q) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      if (valid && hmax > 0.f) atomicMax(args.h_amax + orow, __float_as_uint(hmax));
    };
    if (r0 == 0)
      run(std::true_type{});
    else
      run(std::false_type{});
  } else {
    const float scale = valid ? gw * sa : 0.0f;
#pragma unroll 1
    for (int step = 0; step < 2; ++step) {
      const int i = step ^ r0 ^ 1;  // the N half in R1 first
      const int region = r0 + i;
      const uint32_t tb = tq + (uint32_t)(region * NVF4_REGION_COLS) + 64 * half;
      uint32_t v[2][32];
      ptx::tmem_ld32(tb, v[0]);
      ptx::tmem_ld32(tb + 32, v[1]);
      float my[2] = {0.f, 0.f};  // split-K: lane l fetches column l's scale
      if (prow) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int cw = 128 * i + 64 * half + 32 * cc;
          if (t.n * 256 + cw + lane < args.n_out) my[cc] = __ldg(sb0 + cw + lane);
        }
      }
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_addr(&slot_empty[region]));
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = t.n * 256 + 128 * i + 64 * half + 32 * cc;
        if (prow) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float y[8];  // every lane takes part in the shuffles
#pragma unroll
            for (int e = 0; e < 8; ++e)
              y[e] = __uint_as_float(v[cc][8 * q + e]) * sa *
                     __shfl_sync(0xffffffffu, my[cc], 8 * q + e);
            if (!valid || col0 + q * 8 >= args.n_out) continue;
            float4* d0 = reinterpret_cast<float4*>(prow + col0 + q * 8);
            d0[0] = make_float4(y[0], y[1], y[2], y[3]);
            d0[1] = make_float4(y[4], y[5], y[6], y[7]);
          }
          continue;
        }
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float sd[8];
          staged_scales8(ss + 64 * i + 32 * cc + q * 8, scale, sd);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = 4 * q + jj;
            pk[j] = f32x2_to_bf16x2(__uint_as_float(v[cc][2 * j]) * sd[2 * jj],
                                    __uint_as_float(v[cc][2 * j + 1]) * sd[2 * jj + 1]);
          }
        }
        if (!valid) continue;
        __nv_bfloat16* dst = out + orow * args.ldo + col0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (col0 + q * 8 < args.n_out)
            *reinterpret_cast<uint4*>(dst + q * 8) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
  }
}

// E4M3 epilogue scales of one accumulator row: the row's A scale (x_perm row
// or token for gate/up, H row for down) and the tile's first weight-channel
// scales (gate, up; or down). bf16: 1 and null.
template <int EPI, int OP>
__device__ __forceinline__ void row_scales(const GemmArgs& args, const int32_t* seg, int E,
                                           const Tile& t, int r, bool valid, long long orow,
                                           float& sa, const float*& sb0, const float*& sb1) {
  sa = 1.f;
  sb0 = sb1 = nullptr;
  if constexpr (Op<OP>::scaled) {
    const long long wbase = (long long)t.s * args.b_rows + t.n * (gu_like(EPI) ? 128 : 256);
    sb0 = args.b_scale0 + wbase;
    if (gu_like(EPI)) {
      sb1 = args.b_scale1 + wbase;
      const long long arow = __ldg(seg + 3 + 2 * E + t.s) + r;
      if (valid) sa = __ldg((t.s >= args.n_routed ? args.a_scale_shared : args.a_scale) + arow);
    } else if (valid) {
      sa = __ldg(args.a_scale + orow);
    }
  }
}

// NVFP4 block-scale maps (E4M3 bytes [rows][stride], boxes of 128 rows x
// 16 bytes = the scales of one 256-element K block): A rows, the shared
// experts' A rows, and the weight rows of B's two halves. Unused otherwise.
struct SfMaps {
  CUtensorMap a, a_shared, b0, b1;
};

// NVFP4: one lane quarter's copy of a stage's block scales in Tensor
// Memory. The stage holds them as TMA left them: row r of A (128 rows) at
// sf + r*16 and row r of B (256 rows) at sf + 2048 + r*16, the four 32-bit
// words of a row being the scales of the block's four MMAs (four
// 16-element groups each). The block-scaled MMA reads row m's word from
// column m/32 of the lanes congruent to m mod 32 -- in every lane quarter
// -- so lane l of the quarter gets, for MMA j, the words of rows l + 32c:
// A at column sfa + 4j + c (c < 4), B at column sfa + 16 + 8j + c (c < 8).
// Executed by a full warp; the lane field of sfa_t is the warp's quarter.
__device__ __forceinline__ void sf_store_quarter(uint32_t sf, uint32_t sfa_t, int lane) {
  uint32_t va[16], vb[32];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 w = ptx::ld_shared_v4(sf + (uint32_t)(lane + 32 * c) * 16u);
    va[c] = w.x;
    va[4 + c] = w.y;
    va[8 + c] = w.z;
    va[12 + c] = w.w;
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 w = ptx::ld_shared_v4(sf + 2048u + (uint32_t)(lane + 32 * c) * 16u);
    vb[c] = w.x;
    vb[8 + c] = w.y;
    vb[16 + c] = w.z;
    vb[24 + c] = w.w;
  }
  uint32_t lo[16], hi[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    lo[i] = vb[i];
    hi[i] = vb[16 + i];
  }
  ptx::tmem_st16(sfa_t, va);
  ptx::tmem_st16(sfa_t + 16, lo);
  ptx::tmem_st16(sfa_t + 32, hi);
}

template <int EPI, int OP>
__global__ void __launch_bounds__(Op<OP>::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_a_shared,
                        const __grid_constant__ CUtensorMap map_b0,
                        const __grid_constant__ CUtensorMap map_b1, const GemmArgs args,
                        const __grid_constant__ SfMaps sf) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ SharedState st;

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
  const uint32_t ring = (ptx::smem_addr(dyn_smem) + 1023u) & ~1023u;

  const int32_t* seg = args.seg;
  const int KB = (args.K + Op<OP>::EPK - 1) / Op<OP>::EPK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.empty[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.sf_ready[i]), OP == OP_NVF4 ? 4 : 1);
    }
    for (int i = 0; i < NUM_ACC; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.acc_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.acc_empty[i]), G_EPI_THREADS);
    }
    for (int i = 0; i < 3; ++i) ptx::mbar_init(ptx::smem_addr(&st.slot_empty[i]), G_EPI_THREADS);
    ptx::mbar_init(ptx::smem_addr(&st.drain), 1);
    st.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&map_a);
    ptx::prefetch_tmap(&map_a_shared);
    ptx::prefetch_tmap(&map_b0);
    ptx::prefetch_tmap(&map_b1);
    if constexpr (OP == OP_NVF4) {
      ptx::prefetch_tmap(&sf.a);
      ptx::prefetch_tmap(&sf.a_shared);
      ptx::prefetch_tmap(&sf.b0);
      ptx::prefetch_tmap(&sf.b1);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&st.tmem_base), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = st.tmem_base;
  volatile int* abort_flag = &st.abort;
  pdl_wait();  // the segment table and the operands come from earlier kernels
  pdl_trigger();
  const int E = __ldg(seg);
  const int tiles = __ldg(seg + 1) * args.NT;
  const int S = choose_splits(tiles, gridDim.x, KB, args.s_max);
  const int total = tiles * S;  // work units: (tile, split), splits of a tile adjacent

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < total && ok; unit += gridDim.x) {
        const int split = unit % S;
        const Tile t = decode_tile(seg, E, args.NT, unit / S);
        const CUtensorMap* am = &map_a;
        int a_row;
        if (gu_like(EPI)) {
          a_row = __ldg(seg + 3 + 2 * E + t.s) + t.m * BM;
          if (t.s >= args.n_routed) am = &map_a_shared;
        } else {
          a_row = __ldg(seg + 3 + 3 * E + t.s) + t.m * BM;
        }
        const int b_row = t.s * args.b_rows + t.n * (gu_like(EPI) ? 128 : 256);
        const int kb1 = kb_begin(split + 1, S, KB);
        for (int kb = kb_begin(split, S, KB); kb < kb1; ++kb) {
          if (!wait_phase(ptx::smem_addr(&st.empty[stage]), phase ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_addr(&st.full[stage]);
          const uint32_t a_dst = ring + stage * Op<OP>::STAGE;
          const uint32_t b_dst = a_dst + A_BYTES;
          ptx::mbar_arrive_expect_tx(fb, Op<OP>::STAGE);
          ptx::tma_load_2d(a_dst, am, fb, kb * Op<OP>::KC, a_row);
          if constexpr (OP == OP_NVF4) {
            // block scales: A's 128 rows, then B's two 128-row halves
            const uint32_t sf_dst = a_dst + STAGE_BYTES;
            const bool sh = gu_like(EPI) && t.s >= args.n_routed;
            ptx::tma_load_2d(sf_dst, sh ? &sf.a_shared : &sf.a, fb, kb * 16, a_row);
            ptx::tma_load_2d(sf_dst + 2048, &sf.b0, fb, kb * 16, b_row);
            if (gu_like(EPI))
              ptx::tma_load_2d(sf_dst + 4096, &sf.b1, fb, kb * 16, b_row);
            else
              ptx::tma_load_2d(sf_dst + 4096, &sf.b0, fb, kb * 16, b_row + 128);
          }
          if constexpr (b_mn(EPI)) {
            // K rows kb*64.. of this expert's B (from map_b1 past kb_split),
            // as 4 boxes of 64 N columns
            const bool second = kb >= args.kb_split;
            const CUtensorMap* bm = second ? &map_b1 : &map_b0;
            const int krow = t.s * args.b_rows + (second ? kb - args.kb_split : kb) * BK;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              ptx::tma_load_2d(b_dst + q * B_MN_BOX_BYTES, bm, fb, t.n * 256 + q * 64, krow);
          } else if (gu_like(EPI)) {
            ptx::tma_load_2d(b_dst, &map_b0, fb, kb * Op<OP>::KC, b_row);
            ptx::tma_load_2d(b_dst + B_HALF_BYTES, &map_b1, fb, kb * Op<OP>::KC, b_row);
          } else {
            ptx::tma_load_2d(b_dst, &map_b0, fb, kb * Op<OP>::KC, b_row);
            ptx::tma_load_2d(b_dst + B_HALF_BYTES, &map_b0, fb, kb * Op<OP>::KC, b_row + 128);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA can exit.
        const long long n = issued < STAGES ? issued : STAGES;
        for (long long i = 1; i <= n; ++i) {
          const long long q = issued - i;
          drain_wait(ptx::smem_addr(&st.full[q % STAGES]), (uint32_t)((q / STAGES) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if constexpr (OP == OP_NVF4) {
      // Lane 0 waits until a stage's operands have landed and its block
      // scales are in TMEM (the last four warps, below), then issues the
      // block-scaled MMAs (N = 256). A unit accumulates in regions R0-R1 or
      // R1-R2 (even and odd units) and first waits until both are free.
      // The scales of consecutive K blocks alternate between two TMEM
      // buffers.
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0, kcount = 0;
        uint32_t region_phase = 0;  // bit i: parity of region i's next release
        int r0 = 0;                 // the unit's first region: 0 or 1
        bool ok = true;
        for (int unit = blockIdx.x; unit < total && ok; unit += gridDim.x) {
          if (!wait_phase(ptx::smem_addr(&st.slot_empty[r0]), ((region_phase >> r0) & 1u) ^ 1u,
                          abort_flag, args.status) ||
              !wait_phase(ptx::smem_addr(&st.slot_empty[r0 + 1]),
                          ((region_phase >> (r0 + 1)) & 1u) ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          region_phase ^= 3u << r0;
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(r0 * NVF4_REGION_COLS);
          const int split = unit % S;
          const int kb0 = kb_begin(split, S, KB), kb1 = kb_begin(split + 1, S, KB);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!wait_phase(ptx::smem_addr(&st.full[stage]), phase, abort_flag, args.status) ||
                !wait_phase(ptx::smem_addr(&st.sf_ready[stage]), phase, abort_flag,
                            args.status)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t a_src = ring + stage * Op<OP>::STAGE;
            const uint32_t sfa_t = tmem_base + SF_TMEM_COL + (kcount & 1u) * SF_TMEM_BUF;
            const uint32_t sfb_t = sfa_t + 16;
            const uint64_t adesc = ptx::sdesc_k128(a_src);
            const uint64_t bdesc = ptx::sdesc_k128(a_src + A_BYTES);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // +32 bytes (64 E2M1) of K per step
              ptx::mma_nvf4(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_op<OP>(BM, BN),
                            sfa_t + 4 * k, sfb_t + 8 * k, (kb > kb0 || k > 0) ? 1u : 0u);
            ptx::mma_commit(ptx::smem_addr(&st.empty[stage]));
            ++kcount;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          ptx::mma_commit(ptx::smem_addr(&st.acc_full[0]));
          r0 ^= 1;
        }
        if (!ok) {
          ptx::mma_commit(ptx::smem_addr(&st.drain));
          drain_wait(ptx::smem_addr(&st.drain), 0);
        }
      }
    } else if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < total && ok; unit += gridDim.x) {
        if (!wait_phase(ptx::smem_addr(&st.acc_empty[acc]), acc_phase ^ 1u, abort_flag,
                        args.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const int split = unit % S;
        const int kb0 = kb_begin(split, S, KB), kb1 = kb_begin(split + 1, S, KB);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_phase(ptx::smem_addr(&st.full[stage]), phase, abort_flag, args.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_src = ring + stage * Op<OP>::STAGE;
          const uint64_t adesc = ptx::sdesc_k128(a_src);
          if constexpr (b_mn(EPI)) {
            const uint64_t bdesc = ptx::sdesc_mn128(a_src + A_BYTES, B_MN_BOX_BYTES);
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k)  // B: +2048 bytes (two 8-row K groups) a step
              ptx::mma_bf16(d_tmem, adesc + 2 * k, bdesc + 128 * k,
                            ptx::idesc_bf16_f32_mn(BM, BN, false), (kb > kb0 || k > 0) ? 1u : 0u);
          } else {
            const uint64_t bdesc = ptx::sdesc_k128(a_src + A_BYTES);
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
              // +32 bytes of K per step = +2 in the descriptor's address field
              mma_op<OP>(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_op<OP>(BM, BN),
                         (kb > kb0 || k > 0) ? 1u : 0u);
            }
          }
          ptx::mma_commit(ptx::smem_addr(&st.empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_addr(&st.acc_full[acc]));
        if (++acc == NUM_ACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        ptx::mma_commit(ptx::smem_addr(&st.drain));
        drain_wait(ptx::smem_addr(&st.drain), 0);
      }
    }
  } else if (OP == OP_NVF4 && warp >= G_THREADS / 32) {
    // ------------------------------------------ NVFP4 block-scale warps --
    // One warp per TMEM lane quarter writes each stage's block scales into
    // its quarter of the stage's scale buffer (sf_store_quarter) and hands
    // the stage to the MMA thread (sf_ready, four arrivals), so the tensor
    // pipe only runs MMAs. A buffer is rewritten only after the MMAs of the
    // K block that last used it -- two blocks back -- have completed (that
    // block's empty barrier).
    const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
    int stage = 0;
    uint32_t phase = 0, kcount = 0;
    bool ok = true;
    for (int unit = blockIdx.x; unit < total && ok; unit += gridDim.x) {
      const int split = unit % S;
      const int kb1 = kb_begin(split + 1, S, KB);
      for (int kb = kb_begin(split, S, KB); kb < kb1; ++kb) {
        ok = wait_phase(ptx::smem_addr(&st.full[stage]), phase, abort_flag, args.status);
        if (ok && kcount >= 2) {
          const uint32_t k2 = kcount - 2;
          ok = wait_phase(ptx::smem_addr(&st.empty[k2 % STAGES]), (k2 / STAGES) & 1u, abort_flag,
                          args.status);
        }
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        sf_store_quarter(ring + stage * Op<OP>::STAGE + STAGE_BYTES,
                         tmem_base + lanes + SF_TMEM_COL + (kcount & 1u) * SF_TMEM_BUF, lane);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&st.sf_ready[stage]));
        ++kcount;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    const int sub = warp & 3;  // TMEM lanes [32*sub, 32*sub+32) are this warp's
    const int half = (warp - 2) >> 2;  // which half of the columns
    const int row_in_tile = sub * 32 + lane;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
    // E4M3 / NVFP4: each epilogue warp's copy of the channel scales of its
    // columns of the current tile
    __shared__ __align__(16) float ch_scales[EPI_WARPS][128];
    int acc = 0;
    uint32_t acc_phase = 0;
    int r0 = 0;  // NVFP4: the unit's first accumulator region (unit parity)
    for (int unit = blockIdx.x; unit < total; unit += gridDim.x) {
      const int split = unit % S;
      const Tile t = decode_tile(seg, E, args.NT, unit / S);
      // Everything that does not depend on the accumulator is fetched while
      // the MMAs of this tile still run: the row's place, its scales and
      // gate weight, and the tile's channel scales.
      const int rows = __ldg(seg + 3 + E + t.s);
      const int row0 = __ldg(seg + 3 + 3 * E + t.s);
      const int r = t.m * BM + row_in_tile;
      const bool valid = r < rows;
      const long long orow = (long long)row0 + r;
      const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * BN);
      float sa;
      const float* sb0;
      const float* sb1;
      row_scales<EPI, OP>(args, seg, E, t, r, valid, orow, sa, sb0, sb1);
      const float gw = (EPI == EPI_DOWN && valid) ? row_scale(args, t.s, orow) : 1.0f;
      const float* ss = nullptr;
      if constexpr (Op<OP>::scaled) {
        if (S == 1) {
          float* mine = ch_scales[warp - 2];
          __syncwarp();  // the previous tile's reads of `mine` are done
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = lane + 32 * i;
            // the tile column of the warp's j-th gate (then up) or down
            // column; NVFP4 down takes 64 from each N half
            int cw;
            if (gu_like(EPI))
              cw = 64 * half + (j & 63);
            else
              cw = OP == OP_NVF4 ? 128 * (j >> 6) + 64 * half + (j & 63) : 128 * half + j;
            const int col = t.n * (gu_like(EPI) ? 128 : 256) + cw;
            const float* src = (gu_like(EPI) && j >= 64 ? sb1 : sb0) + cw;
            mine[j] = col < args.n_out ? __ldg(src) : 0.0f;
          }
          __syncwarp();
          ss = mine;
        }
      }
      bool ok = wait_phase(ptx::smem_addr(&st.acc_full[acc]), acc_phase, abort_flag, args.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      if constexpr (OP == OP_NVF4) {
        float* prow =
            S == 1 ? nullptr : args.partial + ((long long)split * args.R + orow) * args.pc;
        epilogue_nvf4<EPI>(args, tmem_base + ((uint32_t)(sub * 32) << 16), r0, st.slot_empty, t,
                           half, valid, orow, out, sa, sb0, sb1, gw, ss, prow);
        r0 ^= 1;
      } else if (S == 1) {
        epilogue_fused<EPI, OP>(args, tbase, t, half, valid, orow, out, sa, sb0, sb1, gw, ss);
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_addr(&st.acc_empty[acc]));
      } else {
        // Split-K unit: this split's fp32 partial rows; splitk_reduce_kernel
        // sums the splits in order and applies the epilogue.
        float* prow = args.partial + ((long long)split * args.R + orow) * args.pc;
        constexpr int HALF_CHUNKS = gu_like(EPI) ? 2 : 4;
#pragma unroll 1
        for (int c = half * HALF_CHUNKS; c < (half + 1) * HALF_CHUNKS; ++c) {
          uint32_t v[32], u[32];
          ptx::tmem_ld32(tbase + c * 32, v);
          if (EPI == EPI_SWIGLU) ptx::tmem_ld32(tbase + 128 + c * 32, u);
          const int col0 = t.n * (EPI == EPI_SWIGLU ? 128 : 256) + c * 32;
          float my0 = 0.f, my1 = 0.f;  // E4M3: lane l fetches column l's scales
          if constexpr (Op<OP>::scaled)
            if (col0 + (threadIdx.x % 32) < args.n_out) {
              my0 = __ldg(sb0 + c * 32 + threadIdx.x % 32);
              if (EPI == EPI_SWIGLU) my1 = __ldg(sb1 + c * 32 + threadIdx.x % 32);
            }
          ptx::tmem_ld_wait();
          if constexpr (Op<OP>::scaled) {  // partials carry their scales (sums are linear)
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              v[jj] = __float_as_uint(__uint_as_float(v[jj]) * sa * __shfl_sync(0xffffffffu, my0, jj));
              if (EPI == EPI_SWIGLU)
                u[jj] = __float_as_uint(__uint_as_float(u[jj]) * sa * __shfl_sync(0xffffffffu, my1, jj));
            }
          }
          if (valid) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (col0 + q * 8 >= args.n_out) continue;
              float4* d0 = reinterpret_cast<float4*>(prow + col0 + q * 8);
              d0[0] = make_float4(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1]),
                                  __uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
              d0[1] = make_float4(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]),
                                  __uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
              if (EPI == EPI_SWIGLU) {
                float4* d1 = reinterpret_cast<float4*>(prow + args.n_out + col0 + q * 8);
                d1[0] = make_float4(__uint_as_float(u[8 * q]), __uint_as_float(u[8 * q + 1]),
                                    __uint_as_float(u[8 * q + 2]), __uint_as_float(u[8 * q + 3]));
                d1[1] = make_float4(__uint_as_float(u[8 * q + 4]), __uint_as_float(u[8 * q + 5]),
                                    __uint_as_float(u[8 * q + 6]), __uint_as_float(u[8 * q + 7]));
              }
            }
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_addr(&st.acc_empty[acc]));
      }
      if (++acc == Op<OP>::NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // ------------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// The same grouped GEMM on CTA pairs (clusters of 2, tcgen05 cta_group::2):
// a pair computes a 256-row x 256-column tile with one 256x256x16 MMA per K
// step, issued by the even CTA. Each CTA stages its own 128 A rows and half
// of B (the gate rows in the even CTA and the up rows in the odd one, or
// output features 0-127 / 128-255 for down) and holds its 128 accumulator
// rows in its own TMEM. Per SM this halves the B bytes per MMA cycle and
// leaves room for a 6-stage ring (32 KB a stage). Used for large segments
// only: a 256-row tile wastes up to 255 rows at a segment's end.
constexpr int PSTAGES = 6;
constexpr int P_STAGE_BYTES = A_BYTES + B_HALF_BYTES;               // 32 KB per CTA
constexpr size_t DYN_SMEM_PAIR = (size_t)PSTAGES * P_STAGE_BYTES + 1024;
constexpr int PAIR_TILE_M = 2 * BM;

struct __align__(8) PairState {
  uint64_t full[PSTAGES];
  uint64_t empty[PSTAGES];
  uint64_t acc_full[NUM_ACC];
  uint64_t acc_empty[NUM_ACC];  // in the even CTA: arrivals of both CTAs' epilogues
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int EPI, int OP>
__global__ void __launch_bounds__(G_THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a,
                             const __grid_constant__ CUtensorMap map_a_shared,
                             const __grid_constant__ CUtensorMap map_b0,
                             const __grid_constant__ CUtensorMap map_b1, const GemmArgs args) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ PairState st;

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t ring = (ptx::smem_addr(dyn_smem) + 1023u) & ~1023u;

  const int32_t* seg = args.seg;  // built with 256-row tiles
  const int KB = (args.K + Op<OP>::EPK - 1) / Op<OP>::EPK;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < PSTAGES; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.empty[i]), 1);
    }
    for (int i = 0; i < NUM_ACC; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.acc_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.acc_empty[i]), 2 * G_EPI_THREADS);
    }
    ptx::mbar_init(ptx::smem_addr(&st.drain), 1);
    st.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&map_a);
    ptx::prefetch_tmap(&map_a_shared);
    ptx::prefetch_tmap(&map_b0);
    ptx::prefetch_tmap(&map_b1);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(&st.tmem_base), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers initialised before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem_base = st.tmem_base;
  volatile int* abort_flag = &st.abort;
  pdl_wait();  // the segment table and the operands come from earlier kernels
  pdl_trigger();
  const int E = __ldg(seg);
  const int tiles = __ldg(seg + 1) * args.NT;

  if (warp == 0) {
    // ----------------------------------------------- TMA producer (both CTAs) --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = cluster; tile < tiles && ok; tile += nclusters) {
        const Tile t = decode_tile(seg, E, args.NT, tile);
        const CUtensorMap* am = &map_a;
        const CUtensorMap* bm = &map_b0;
        int a_row, b_row;
        if (EPI == EPI_SWIGLU) {
          a_row = __ldg(seg + 3 + 2 * E + t.s) + t.m * PAIR_TILE_M + (int)rank * BM;
          if (t.s >= args.n_routed) am = &map_a_shared;
          if (rank == 1) bm = &map_b1;  // up rows in the odd CTA
          b_row = t.s * args.b_rows + t.n * 128;
        } else {
          a_row = __ldg(seg + 3 + 3 * E + t.s) + t.m * PAIR_TILE_M + (int)rank * BM;
          b_row = t.s * args.b_rows + t.n * 256 + (int)rank * 128;
        }
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_phase(ptx::smem_addr(&st.empty[stage]), phase ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const uint32_t full_local = ptx::smem_addr(&st.full[stage]);
          const uint32_t full_leader = ptx::mapa_shared(full_local, 0);
          const uint32_t a_dst = ring + stage * P_STAGE_BYTES;
          if (leader) ptx::mbar_arrive_expect_tx(full_local, 2 * P_STAGE_BYTES);
          ptx::tma_load_2d_pair(a_dst, am, full_leader, kb * Op<OP>::EPK, a_row);
          ptx::tma_load_2d_pair(a_dst + A_BYTES, bm, full_leader, kb * Op<OP>::EPK, b_row);
          ++issued;
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        const long long n = issued < PSTAGES ? issued : PSTAGES;
        for (long long i = 1; i <= n; ++i) {
          const long long q = issued - i;
          drain_wait(ptx::smem_addr(&st.full[q % PSTAGES]), (uint32_t)((q / PSTAGES) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer (even CTA only) --
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = cluster; tile < tiles && ok; tile += nclusters) {
        if (!wait_phase(ptx::smem_addr(&st.acc_empty[acc]), acc_phase ^ 1u, abort_flag,
                        args.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_phase(ptx::smem_addr(&st.full[stage]), phase, abort_flag, args.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_src = ring + stage * P_STAGE_BYTES;
          const uint64_t adesc = ptx::sdesc_k128(a_src);
          const uint64_t bdesc = ptx::sdesc_k128(a_src + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            mma_op_pair<OP>(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_op<OP>(2 * BM, BN),
                            (kb | k) != 0);
          ptx::mma_commit_pair(ptx::smem_addr(&st.empty[stage]), 0x3);
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair(ptx::smem_addr(&st.acc_full[acc]), 0x3);
        if (++acc == NUM_ACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        ptx::mma_commit_pair(ptx::smem_addr(&st.drain), 0x1);
        drain_wait(ptx::smem_addr(&st.drain), 0);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (both CTAs) --
    const int sub = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_in_tile = sub * 32 + lane;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
    static_assert(NUM_ACC == 2, "two accumulators");
    const uint32_t acc_empty_leader0 = ptx::mapa_shared(ptx::smem_addr(&st.acc_empty[0]), 0);
    const uint32_t acc_empty_leader1 = ptx::mapa_shared(ptx::smem_addr(&st.acc_empty[1]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = cluster; tile < tiles; tile += nclusters) {
      const Tile t = decode_tile(seg, E, args.NT, tile);
      bool ok = wait_phase(ptx::smem_addr(&st.acc_full[acc]), acc_phase, abort_flag, args.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      const int rows = __ldg(seg + 3 + E + t.s);
      const int r = t.m * PAIR_TILE_M + (int)rank * BM + row_in_tile;
      const bool valid = r < rows;
      const long long orow = (long long)__ldg(seg + 3 + 3 * E + t.s) + r;
      const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * BN);
      float sa;
      const float* sb0;
      const float* sb1;
      row_scales<EPI, OP>(args, seg, E, t, r, valid, orow, sa, sb0, sb1);
      const float gw = (EPI == EPI_DOWN && valid) ? row_scale(args, t.s, orow) : 1.0f;
      epilogue_fused<EPI, OP>(args, tbase, t, half, valid, orow, out, sa, sb0, sb1, gw);
      ptx::tc_fence_before();
      ptx::mbar_arrive_cluster(acc ? acc_empty_leader1 : acc_empty_leader0);
      if (++acc == NUM_ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // ------------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // no CTA leaves while its peer may still use its smem
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Weight-stationary CTA pairs ("swap AB") for segments of a few hundred rows
// (e.g. 256 experts of ~256 rows each): a 256-row token tile would waste up
// to half its rows at a segment's end, a 128-row 1-CTA tile up to 127 and
// moves 1.5x the operand bytes per MMA cycle of a pair. Here the MMA's M side
// is the weights -- 256 output features of one expert, 128 in each CTA -- and
// its N side the segment's token rows: a segment of R rows is cut into
// ceil(R / 256) token tiles of equal height h (rounded up to 16) and the MMA
// takes N = the tile's rows rounded up to 32, each CTA staging N/2 of them,
// so a tile computes at most 31 rows that are not stored.
//  - gate/up: two MMAs a K step (gate, then up rows of the same 128 features
//    of each CTA) into TMEM columns [0, N) and [256, 256 + N), so the
//    epilogue thread of a feature holds both of its products. That fills
//    the 512 columns: one accumulator, whose epilogue the next tile's MMAs
//    wait for. Per CTA a 64-wide K block stages 32 KB of weights and N/2
//    token rows (<= 16 KB): 4 stages.
//  - down: one MMA a K step (128 output features a CTA); two accumulators;
//    a stage is 16 KB of W_d and N/2 rows of H: 6 stages.
//  - The epilogue thread of TMEM lane j of CTA r owns feature
//    256 n + 128 r + j for every token (column) of the tile; a warp stores
//    32 consecutive features (64 bytes) of each token row.
// Tile order, warp roles, barriers, the bounded waits and teardown are those
// of grouped_gemm_pair_kernel.
// A CTA stages its N/2 token rows with a single TMA box: one tensor map per
// box height 16, 32, ..., 128 (N a multiple of 32). A tile's loads as a sum
// of power-of-two boxes (N a multiple of 16) were measured up to 1.4x slower
// in the down projection: one box a stage is what keeps the MMAs fed.
constexpr int SW_TOK_BOXES = 8;
struct TokMaps {
  CUtensorMap box[SW_TOK_BOXES];  // box i: 16 (i + 1) rows
};
template <int EPI>
struct Sw {
  static constexpr int W_BYTES = (EPI == EPI_SWIGLU ? 2 : 1) * A_BYTES;  // per CTA a stage
  static constexpr int TOK_MAX_BYTES = 128 * 128;  // 128 token rows (N/2 <= 128) of 128 bytes
  static constexpr int STAGE = W_BYTES + TOK_MAX_BYTES;
  static constexpr int STAGES = EPI == EPI_SWIGLU ? 4 : 6;
  static constexpr int NACC = EPI == EPI_SWIGLU ? 1 : 2;
  static constexpr size_t SMEM = (size_t)STAGES * STAGE + 1024;
};
constexpr int SW_MAX_STAGES = 6;

struct __align__(8) SwapState {
  uint64_t full[SW_MAX_STAGES];
  uint64_t empty[SW_MAX_STAGES];
  uint64_t gfull[SW_MAX_STAGES];  // fused gather: this CTA's token copies of a stage landed
  uint64_t acc_full[NUM_ACC];
  uint64_t acc_empty[NUM_ACC];  // in the even CTA: arrivals of both CTAs' epilogues
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
// Warps of the fused gather: one issues the copies, one publishes stages.
constexpr int SW_GATHER_THREADS = 64;

// Token tile m of a segment of `rows` rows (the segment table counts
// ceil(rows / 256) tiles): its first row r0, its rows nr (> 0), and the
// MMA's N: the tile height rounded up to 32 (<= 256), N/2 rows in each CTA.
// Every tile of a segment takes the same N, the last one included (its
// columns past nr are computed and not stored): tiles of one weight slab
// then take the same time, run side by side on neighbouring CTA pairs and
// share the slab through L2. With N sized to each tile's own rows the
// Mixtral-shaped gate/up read 3.27 GB from DRAM a launch (1.68x its weight
// bytes), with one N 2.16 GB, in the same time.
__device__ __forceinline__ void swap_tile_rows(int rows, int m, int& r0, int& nr, int& n_mma) {
  const int ntt = (rows + PAIR_TILE_M - 1) / PAIR_TILE_M;
  const int h = (((rows + ntt - 1) / ntt) + 15) & ~15;  // <= 256
  r0 = m * h;
  nr = min(h, rows - r0);
  n_mma = (h + 31) & ~31;
}

template <int EPI, int OP, bool GATHER>
__global__ void __launch_bounds__(GATHER ? G_THREADS + SW_GATHER_THREADS : G_THREADS, 1)
    grouped_swap_pair_kernel(const __grid_constant__ CUtensorMap map_w0,
                             const __grid_constant__ CUtensorMap map_w1,
                             const __grid_constant__ TokMaps tok,
                             const __grid_constant__ TokMaps tok_sh, const GemmArgs args) {
  using C = Sw<EPI>;
  constexpr bool GU = EPI == EPI_SWIGLU;
  static_assert(!GATHER || (GU && OP == OP_BF16), "the fused gather is built for bf16 gate/up");
  extern __shared__ uint8_t dyn_smem[];
  __shared__ SwapState st;

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t ring = (ptx::smem_addr(dyn_smem) + 1023u) & ~1023u;

  const int32_t* seg = args.seg;  // built with 256-row tiles
  const int KB = (args.K + Op<OP>::EPK - 1) / Op<OP>::EPK;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      // the even CTA's full barrier: the producer's expect-tx arrival, and
      // with the fused gather one arrival from each CTA's gather warp
      ptx::mbar_init(ptx::smem_addr(&st.full[i]), GATHER ? 3 : 1);
      ptx::mbar_init(ptx::smem_addr(&st.empty[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.gfull[i]), 32);
    }
    for (int i = 0; i < NUM_ACC; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.acc_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.acc_empty[i]), 2 * G_EPI_THREADS);
    }
    ptx::mbar_init(ptx::smem_addr(&st.drain), 1);
    st.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&map_w0);
    ptx::prefetch_tmap(&map_w1);
    if (!GATHER) {
      for (int i = 0; i < SW_TOK_BOXES; ++i) {
        ptx::prefetch_tmap(&tok.box[i]);
        ptx::prefetch_tmap(&tok_sh.box[i]);
      }
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(&st.tmem_base), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers initialised before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem_base = st.tmem_base;
  volatile int* abort_flag = &st.abort;
  pdl_wait();  // the segment table and the operands come from earlier kernels
  pdl_trigger();
  const int E = __ldg(seg);
  const int tiles = __ldg(seg + 1) * args.NT;

  if (warp == 0) {
    // ----------------------------------------------- TMA producer (both CTAs) --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = cluster; tile < tiles && ok; tile += nclusters) {
        const Tile t = decode_tile(seg, E, args.NT, tile);
        int r0, nr;
        int nmma;
        swap_tile_rows(__ldg(seg + 3 + E + t.s), t.m, r0, nr, nmma);
        const int half = nmma >> 1;  // token rows this CTA stages (multiple of 16)
        const TokMaps* tm = (GU && t.s >= args.n_routed) ? &tok_sh : &tok;
        const int tok_row = __ldg(seg + 3 + (GU ? 2 : 3) * E + t.s) + r0 + (int)rank * half;
        const int w_row = t.s * args.b_rows + t.n * 256 + (int)rank * 128;
        const uint32_t bytes = (uint32_t)(C::W_BYTES + (GATHER ? 0 : half * 128));
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_phase(ptx::smem_addr(&st.empty[stage]), phase ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const uint32_t full_local = ptx::smem_addr(&st.full[stage]);
          const uint32_t full_leader = ptx::mapa_shared(full_local, 0);
          const uint32_t w_dst = ring + stage * C::STAGE;
          if (leader) ptx::mbar_arrive_expect_tx(full_local, 2 * bytes);
          const int kc = kb * Op<OP>::KC;
          ptx::tma_load_2d_pair(w_dst, &map_w0, full_leader, kc, w_row);
          if (GU) ptx::tma_load_2d_pair(w_dst + A_BYTES, &map_w1, full_leader, kc, w_row);
          if (!GATHER)
            ptx::tma_load_2d_pair(w_dst + C::W_BYTES, &tm->box[(half >> 4) - 1], full_leader, kc,
                                  tok_row);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        const long long n = issued < C::STAGES ? issued : C::STAGES;
        for (long long i = 1; i <= n; ++i) {
          const long long q = issued - i;
          drain_wait(ptx::smem_addr(&st.full[q % C::STAGES]), (uint32_t)((q / C::STAGES) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer (even CTA only) --
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = cluster; tile < tiles && ok; tile += nclusters) {
        const Tile t = decode_tile(seg, E, args.NT, tile);
        int r0, nr;
        int nmma;
        swap_tile_rows(__ldg(seg + 3 + E + t.s), t.m, r0, nr, nmma);
        const uint32_t idesc = idesc_op<OP>(2 * BM, nmma);
        if (!wait_phase(ptx::smem_addr(&st.acc_empty[acc]), acc_phase ^ 1u, abort_flag,
                        args.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_phase(ptx::smem_addr(&st.full[stage]), phase, abort_flag, args.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t w_src = ring + stage * C::STAGE;
          const uint64_t wdesc0 = ptx::sdesc_k128(w_src);
          const uint64_t wdesc1 = ptx::sdesc_k128(w_src + A_BYTES);
          const uint64_t tdesc = ptx::sdesc_k128(w_src + C::W_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint32_t accum = (kb | k) != 0;
            mma_op_pair<OP>(d_tmem, wdesc0 + 2 * k, tdesc + 2 * k, idesc, accum);
            if (GU) mma_op_pair<OP>(d_tmem + BN, wdesc1 + 2 * k, tdesc + 2 * k, idesc, accum);
          }
          ptx::mma_commit_pair(ptx::smem_addr(&st.empty[stage]), 0x3);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair(ptx::smem_addr(&st.acc_full[acc]), 0x3);
        if (++acc == C::NACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        ptx::mma_commit_pair(ptx::smem_addr(&st.drain), 0x1);
        drain_wait(ptx::smem_addr(&st.drain), 0);
      }
    }
  } else if (GATHER && warp == G_THREADS / 32) {
    // ------------------------------------------ fused row gather (both CTAs) --
    // The B operand's token rows come straight from x: lane l copies piece
    // l % 8 (16 bytes) of rows l / 8 + 4 q, q < 32, with cp.async (eight
    // lanes a 128-byte row, so a warp instruction reads four whole rows)
    // into the 128-byte-swizzled slot (piece j of row r at j ^ (r % 8)). K
    // past d_model reads as zero. Each lane keeps its 32 rows' offsets in x
    // for the whole tile, so a stage is 32 independent copies a lane. The
    // stage's gfull barrier gets one arrival from each lane when its copies
    // have landed; the next warp publishes the stage.
    const __nv_bfloat16* gx = args.gx;
    const int d = args.K;
    const int pc = lane & 7;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = cluster; tile < tiles && ok; tile += nclusters) {
      const Tile t = decode_tile(seg, E, args.NT, tile);
      const int rows = __ldg(seg + 3 + E + t.s);
      int r0, nr;
      int nmma;
      swap_tile_rows(rows, t.m, r0, nr, nmma);
      const int half = nmma >> 1;
      const int a_row0 = __ldg(seg + 3 + 2 * E + t.s);
      // element offset in x of each of this lane's rows, -1 for none
      long long eoff[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int row = (lane >> 3) + 4 * q;
        const int r = r0 + (int)rank * half + row;  // row within the segment
        int tk = -1;
        if (row < half && r < rows) {
          if (t.s >= args.n_routed) {
            tk = r;  // shared experts read x row by row
          } else {
            const int pair = __ldg(args.sorted_pair + a_row0 + r);
            if (pair >= 0 && pair < args.n_pairs) tk = pair / args.gk;
          }
        }
        eoff[q] = tk < 0 ? -1LL : (long long)tk * d;
      }
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_phase(ptx::smem_addr(&st.empty[stage]), phase ^ 1u, abort_flag, args.status)) {
          ok = false;
          break;
        }
        const uint32_t b_dst = ring + stage * C::STAGE + C::W_BYTES;
        const int kel = kb * 64 + pc * 8;
        const uint32_t nbytes = kel < d ? 16u : 0u;  // d_model is a multiple of 8
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          if (eoff[q] < 0) continue;
          const int row = (lane >> 3) + 4 * q;
          ptx::cp_async16(b_dst + (uint32_t)(row * 128 + ((pc ^ (row & 7)) << 4)),
                          nbytes ? (const void*)(gx + eoff[q] + kel) : (const void*)gx, nbytes);
        }
        ptx::cp_async_mbar_arrive(ptx::smem_addr(&st.gfull[stage]));
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    ptx::cp_async_wait_all();  // no copy is left in flight when the CTA exits
  } else if (GATHER && warp == G_THREADS / 32 + 1) {
    // ------------------------------------- fused gather: publishing a stage --
    // Waits, stage by stage, until the gather warp's copies have landed,
    // makes them visible to the tensor cores (a proxy fence; this warp has no
    // copies of its own in flight, so the fence does not wait for later
    // stages' copies) and arrives on the even CTA's full barrier.
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = cluster; tile < tiles && ok; tile += nclusters) {
      for (int kb = 0; kb < KB; ++kb) {
        const bool landed =
            wait_phase(ptx::smem_addr(&st.gfull[stage]), phase, abort_flag, args.status);
        if (!__all_sync(0xffffffffu, landed)) {
          ok = false;
          break;
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
          ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_addr(&st.full[stage]), 0));
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------ epilogue (both CTAs) --
    // Warps 2-9: the two warps of a TMEM lane quarter take alternate 32-token
    // chunks of the tile.
    const int sub = warp & 3;
    const int hf = (warp - 2) >> 2;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
    // per epilogue warp: a 32-token x 32-feature bf16 block, so that each
    // token row's 64 bytes leave as four 16-byte stores
    __shared__ __align__(16) __nv_bfloat16 stage_out[EPI_WARPS][32 * 32];
    __nv_bfloat16* stg = stage_out[warp - 2];
    const uint32_t acc_empty_leader0 = ptx::mapa_shared(ptx::smem_addr(&st.acc_empty[0]), 0);
    const uint32_t acc_empty_leader1 = ptx::mapa_shared(ptx::smem_addr(&st.acc_empty[1]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = cluster; tile < tiles; tile += nclusters) {
      const Tile t = decode_tile(seg, E, args.NT, tile);
      int r0, nr;
      int nmma;
      swap_tile_rows(__ldg(seg + 3 + E + t.s), t.m, r0, nr, nmma);
      const long long orow0 = (long long)__ldg(seg + 3 + 3 * E + t.s) + r0;
      const int fw0 = t.n * 256 + (int)rank * 128 + sub * 32;  // the warp's first feature
      const int f = fw0 + lane;                                 // this thread's feature
      const bool fvalid = f < args.n_out;
      // E4M3: the feature's weight-channel scales, and the tokens' row scales
      float sw0 = 1.f, sw1 = 1.f;
      const float* tok_scale = nullptr;
      long long tok_row0 = orow0;
      if constexpr (Op<OP>::scaled) {
        const long long wrow = (long long)t.s * args.b_rows + f;
        sw0 = fvalid ? __ldg(args.b_scale0 + wrow) : 0.f;
        if (GU) {
          sw1 = fvalid ? __ldg(args.b_scale1 + wrow) : 0.f;
          tok_row0 = (long long)__ldg(seg + 3 + 2 * E + t.s) + r0;
          tok_scale = t.s >= args.n_routed ? args.a_scale_shared : args.a_scale;
        } else {
          tok_scale = args.a_scale;
        }
      }
      // Lane l fetches the row factor of token c0 + l of each of the warp's
      // (at most 4) chunks -- for down its gate weight, for E4M3 its A row
      // scale -- before waiting for the accumulator, so the dependent loads
      // overlap the tile's MMAs.
      float rfs[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tkn = hf * 32 + 64 * j + lane;
        float rf = 1.f;
        if (tkn < nr) {
          if (!GU) rf = row_scale(args, t.s, orow0 + tkn);
          if constexpr (Op<OP>::scaled) rf *= __ldg(tok_scale + tok_row0 + tkn);
        }
        rfs[j] = rf;
      }
      bool ok = wait_phase(ptx::smem_addr(&st.acc_full[acc]), acc_phase, abort_flag, args.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c0 = hf * 32 + 64 * j;
        if (c0 >= nr) break;  // warp-uniform
        uint32_t a[32], b[32];
        ptx::tmem_ld32(tbase + c0, a);
        if (GU) ptx::tmem_ld32(tbase + BN + c0, b);
        const float rf = rfs[j];
        ptx::tmem_ld_wait();
        const int cn = min(32, nr - c0);  // warp-uniform
        // bf16 results into this warp's 32 x 32 staging block, transposed:
        // row c (token) holds the warp's 32 features
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float hv;
          if constexpr (GU) {
            float g = __uint_as_float(a[c]), u = __uint_as_float(b[c]);
            if constexpr (Op<OP>::scaled) {
              const float r = __shfl_sync(0xffffffffu, rf, c);
              g *= sw0 * r;
              u *= sw1 * r;
            }
            hv = silu(g) * u;
          } else {
            hv = __uint_as_float(a[c]) * __shfl_sync(0xffffffffu, rf, c);
            if constexpr (Op<OP>::scaled) hv *= sw0;
          }
          stg[c * 32 + lane] = __float2bfloat16_rn(hv);
        }
        __syncwarp();
        // 16-byte row pieces: lane l stores piece l % 4 of token rows
        // l / 4 + 8 i, masked to the tile's rows and the output's columns
        const int piece = lane & 3;
        const bool cvalid = fw0 + piece * 8 < args.n_out;  // n_out is a multiple of 8
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = (lane >> 2) + 8 * i;
          const uint4 v = *reinterpret_cast<const uint4*>(stg + row * 32 + piece * 8);
          const long long orow = orow0 + c0 + row;
          if (row < cn && cvalid)
            *reinterpret_cast<uint4*>(out + orow * args.ldo + fw0 + piece * 8) = v;
          if constexpr (Op<OP>::scaled && GU) {
            // the H row's max |H| over this warp's 32 features, one atomic
            float h0, h1, h2, h3, h4, h5, h6, h7;
            bf16x2_to_f32(v.x, h0, h1);
            bf16x2_to_f32(v.y, h2, h3);
            bf16x2_to_f32(v.z, h4, h5);
            bf16x2_to_f32(v.w, h6, h7);
            float m = cvalid ? fmaxf(fmaxf(fmaxf(fabsf(h0), fabsf(h1)), fmaxf(fabsf(h2), fabsf(h3))),
                                     fmaxf(fmaxf(fabsf(h4), fabsf(h5)), fmaxf(fabsf(h6), fabsf(h7))))
                             : 0.f;
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            if (piece == 0 && row < cn && m > 0.f) atomicMax(args.h_amax + orow, __float_as_uint(m));
          }
        }
        __syncwarp();  // the block is read before the next chunk rewrites it
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive_cluster(acc ? acc_empty_leader1 : acc_empty_leader0);
      if (++acc == C::NACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // ------------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // no CTA leaves while its peer may still use its smem
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Decode-sized batches (T <= 64, so every expert segment has at most 64
// rows): swap A and B. The expert weights are the MMA's M side (128 output
// features of one expert per tile) and the segment's few token rows the N
// side (16-64), so a stage holds only bytes the product needs: for gate/up
// a 128x64 tile of W_gate and of W_up and Ntok x 64 of the tokens, for down
// a 128x64 tile of W_down and Ntok x 64 of H. Gate and up accumulate in two
// TMEM column ranges of one 256-column buffer; the epilogue thread of TMEM
// lane j owns output feature j of the tile for every token of the segment.
// The ring has as many stages as fit in shared memory (5 for gate/up, 8+
// for down), so more weight bytes are in flight per SM than with 128-row
// token tiles. Tiles, splits and the partial-row layout are those of
// grouped_gemm_kernel, so splitk_reduce_kernel finishes split tiles.
constexpr int kDecodeMaxRows = 64;
constexpr int TOK_BOX = 16;                       // token rows per TMA box
constexpr int TOK_BOX_BYTES = TOK_BOX * BK * 2;   // 2 KB
constexpr size_t DYN_SMEM_DECODE = 200 * 1024 + 1024;
constexpr int kDecodeMaxStages = 16;

struct __align__(8) DecodeState {
  uint64_t full[kDecodeMaxStages];
  uint64_t empty[kDecodeMaxStages];
  uint64_t acc_full[NUM_ACC];
  uint64_t acc_empty[NUM_ACC];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct DecodeShape {
  int stages;       // ring depth
  int stage_bytes;  // multiple of 1024
  int a_bytes;      // weight bytes a stage (16 or 32 KB)
};

template <int EPI, int OP>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_decode_kernel(const __grid_constant__ CUtensorMap map_w0,
                          const __grid_constant__ CUtensorMap map_w1,
                          const __grid_constant__ CUtensorMap map_tok,
                          const __grid_constant__ CUtensorMap map_tok_shared, const GemmArgs args,
                          const DecodeShape shape) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ DecodeState st;

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
  const uint32_t ring = (ptx::smem_addr(dyn_smem) + 1023u) & ~1023u;
  const int STG = shape.stages;

  const int32_t* seg = args.seg;
  const int KB = (args.K + Op<OP>::EPK - 1) / Op<OP>::EPK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STG; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.empty[i]), 1);
    }
    for (int i = 0; i < NUM_ACC; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.acc_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.acc_empty[i]), EPI_THREADS);
    }
    ptx::mbar_init(ptx::smem_addr(&st.drain), 1);
    st.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&map_w0);
    ptx::prefetch_tmap(&map_w1);
    ptx::prefetch_tmap(&map_tok);
    ptx::prefetch_tmap(&map_tok_shared);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&st.tmem_base), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = st.tmem_base;
  volatile int* abort_flag = &st.abort;
  pdl_wait();  // the segment table and the operands come from earlier kernels
  pdl_trigger();
  const int E = __ldg(seg);
  const int tiles = __ldg(seg + 1) * args.NT;
  const int S = choose_splits(tiles, gridDim.x, KB, args.s_max);
  const int total = tiles * S;

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < total && ok; unit += gridDim.x) {
        const int split = unit % S;
        const Tile t = decode_tile(seg, E, args.NT, unit / S);
        const int rows = __ldg(seg + 3 + E + t.s);
        const int nbox = (rows + TOK_BOX - 1) / TOK_BOX;
        const int w_row = t.s * args.b_rows + t.n * BM;
        int tok_row;
        const CUtensorMap* tm = &map_tok;
        if (EPI == EPI_SWIGLU) {
          tok_row = __ldg(seg + 3 + 2 * E + t.s);
          if (t.s >= args.n_routed) tm = &map_tok_shared;
        } else {
          tok_row = __ldg(seg + 3 + 3 * E + t.s);
        }
        const uint32_t tx = (uint32_t)shape.a_bytes + (uint32_t)(nbox * TOK_BOX_BYTES);
        const int kb1 = kb_begin(split + 1, S, KB);
        for (int kb = kb_begin(split, S, KB); kb < kb1; ++kb) {
          if (!wait_phase(ptx::smem_addr(&st.empty[stage]), phase ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_addr(&st.full[stage]);
          const uint32_t dst = ring + stage * shape.stage_bytes;
          ptx::mbar_arrive_expect_tx(fb, tx);
          ptx::tma_load_2d(dst, &map_w0, fb, kb * Op<OP>::EPK, w_row);
          if (EPI == EPI_SWIGLU) ptx::tma_load_2d(dst + A_BYTES, &map_w1, fb, kb * Op<OP>::EPK, w_row);
          for (int b = 0; b < nbox; ++b)
            ptx::tma_load_2d(dst + shape.a_bytes + b * TOK_BOX_BYTES, tm, fb, kb * Op<OP>::EPK,
                             tok_row + b * TOK_BOX);
          ++issued;
          if (++stage == STG) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        const long long n = issued < STG ? issued : STG;
        for (long long i = 1; i <= n; ++i) {
          const long long q = issued - i;
          drain_wait(ptx::smem_addr(&st.full[q % STG]), (uint32_t)((q / STG) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < total && ok; unit += gridDim.x) {
        const Tile t = decode_tile(seg, E, args.NT, unit / S);
        const int rows = __ldg(seg + 3 + E + t.s);
        const int ntok = ((rows + TOK_BOX - 1) / TOK_BOX) * TOK_BOX;
        const uint32_t idesc = idesc_op<OP>(BM, ntok);
        if (!wait_phase(ptx::smem_addr(&st.acc_empty[acc]), acc_phase ^ 1u, abort_flag,
                        args.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const int split = unit % S;
        const int kb0 = kb_begin(split, S, KB), kb1 = kb_begin(split + 1, S, KB);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_phase(ptx::smem_addr(&st.full[stage]), phase, abort_flag, args.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t src = ring + stage * shape.stage_bytes;
          const uint64_t w0 = ptx::sdesc_k128(src);
          const uint64_t w1 = ptx::sdesc_k128(src + A_BYTES);
          const uint64_t tk = ptx::sdesc_k128(src + shape.a_bytes);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
            mma_op<OP>(d_tmem, w0 + 2 * k, tk + 2 * k, idesc, accum);
            if (EPI == EPI_SWIGLU) mma_op<OP>(d_tmem + 128, w1 + 2 * k, tk + 2 * k, idesc, accum);
          }
          ptx::mma_commit(ptx::smem_addr(&st.empty[stage]));
          if (++stage == STG) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_addr(&st.acc_full[acc]));
        if (++acc == NUM_ACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        ptx::mma_commit(ptx::smem_addr(&st.drain));
        drain_wait(ptx::smem_addr(&st.drain), 0);
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    const int sub = warp & 3;
    const int j = sub * 32 + lane;  // TMEM lane = output feature within the tile
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int unit = blockIdx.x; unit < total; unit += gridDim.x) {
      const int split = unit % S;
      const Tile t = decode_tile(seg, E, args.NT, unit / S);
      bool ok = wait_phase(ptx::smem_addr(&st.acc_full[acc]), acc_phase, abort_flag, args.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      const int rows = __ldg(seg + 3 + E + t.s);
      const long long row0 = __ldg(seg + 3 + 3 * E + t.s);
      const int f = t.n * BM + j;
      const bool fvalid = f < args.n_out;
      const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * BN);
      // E4M3: the feature's weight-channel scales and the tokens' row scales
      float sw0 = 1.f, sw1 = 1.f;
      const float* tok_scale = nullptr;
      long long tok_row0 = 0;
      if constexpr (Op<OP>::scaled) {
        const long long wrow = (long long)t.s * args.b_rows + f;
        sw0 = fvalid ? __ldg(args.b_scale0 + wrow) : 0.f;
        if (EPI == EPI_SWIGLU) {
          sw1 = fvalid ? __ldg(args.b_scale1 + wrow) : 0.f;
          tok_row0 = __ldg(seg + 3 + 2 * E + t.s);
          tok_scale = t.s >= args.n_routed ? args.a_scale_shared : args.a_scale;
        } else {
          tok_row0 = row0;
          tok_scale = args.a_scale;
        }
      }
      for (int c0 = 0; c0 < rows; c0 += 32) {
        uint32_t a[32], b[32];
        ptx::tmem_ld32(tbase + c0, a);
        if (EPI == EPI_SWIGLU) ptx::tmem_ld32(tbase + 128 + c0, b);
        ptx::tmem_ld_wait();
        const int cn = min(32, rows - c0);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c >= cn) break;  // cn is the same for the whole warp
          const long long orow = row0 + c0 + c;
          float av = __uint_as_float(a[c]);
          float bv = EPI == EPI_SWIGLU ? __uint_as_float(b[c]) : 0.f;
          if constexpr (Op<OP>::scaled) {
            const float st = __ldg(tok_scale + tok_row0 + c0 + c);
            av *= sw0 * st;
            bv *= sw1 * st;
          }
          if (S == 1) {
            __nv_bfloat16 hb;
            if (EPI == EPI_SWIGLU) hb = __float2bfloat16_rn(silu(av) * bv);
            else hb = __float2bfloat16_rn(row_scale(args, t.s, orow) * av);
            if (fvalid) out[orow * args.ldo + f] = hb;
            if constexpr (Op<OP>::scaled && EPI == EPI_SWIGLU) {
              // the H row's max |H| over this warp's 32 features, one atomic
              float m = fvalid ? fabsf(__bfloat162float(hb)) : 0.f;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
              if (lane == 0 && m > 0.f) atomicMax(args.h_amax + orow, __float_as_uint(m));
            }
          } else if (fvalid) {
            float* prow = args.partial + ((long long)split * args.R + orow) * args.pc;
            prow[f] = av;
            if (EPI == EPI_SWIGLU) prow[args.n_out + f] = bv;
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_addr(&st.acc_empty[acc]));
      if (++acc == NUM_ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // ------------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Split-K epilogue: every output element from the partials of all S splits,
// summed in split order, then the same epilogue as the fused path. One
// thread per 4 output columns of one row; its (up to kMaxSplitK) partial
// loads are issued together before any is summed. E4M3 partials already
// carry their scales; for gate/up the rows' max |H| is gathered per block in
// shared memory (a block spans at most 256 rows) and sent with one atomic
// per row.
template <int EPI, int OP>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const GemmArgs a, int gemm_grid) {
  __shared__ unsigned s_max[256];
  __shared__ int s_splits;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0)  // once a block: the choice loops over the split factors
    s_splits = choose_splits(__ldg(a.seg + 1) * a.NT, gemm_grid,
                             (a.K + Op<OP>::EPK - 1) / Op<OP>::EPK, a.s_max);
  __syncthreads();
  const int S = s_splits;
  if (S == 1) return;  // the GEMM finished its tiles itself
  const int groups = a.n_out / 4;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long first_row = ((long long)blockIdx.x * blockDim.x) / groups;
  constexpr bool kAmax = Op<OP>::scaled && EPI == EPI_SWIGLU;
  if (kAmax) {
    s_max[threadIdx.x] = 0u;
    __syncthreads();
  }
  if (i < a.R * groups) {
    const long long orow = i / groups;
    const int col = (int)(i % groups) * 4;
    float4 pv[kMaxSplitK], pu[kMaxSplitK];
#pragma unroll
    for (int sp = 0; sp < kMaxSplitK; ++sp) {
      if (sp < S) {
        const float* src = a.partial + ((long long)sp * a.R + orow) * a.pc + col;
        pv[sp] = __ldcg(reinterpret_cast<const float4*>(src));
        if (EPI == EPI_SWIGLU) pu[sp] = __ldcg(reinterpret_cast<const float4*>(src + a.n_out));
      }
    }
    float v[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int sp = 0; sp < kMaxSplitK; ++sp) {
      if (sp < S) {
        v[0] += pv[sp].x; v[1] += pv[sp].y; v[2] += pv[sp].z; v[3] += pv[sp].w;
        if (EPI == EPI_SWIGLU) {
          u[0] += pu[sp].x; u[1] += pu[sp].y; u[2] += pu[sp].z; u[3] += pu[sp].w;
        }
      }
    }
    float h[4];
    if (EPI == EPI_SWIGLU) {
#pragma unroll
      for (int q = 0; q < 4; ++q) h[q] = silu(v[q]) * u[q];
    } else {
      // the row's segment: routed rows are [0, n_pairs), shared rows follow
      const float sc = (orow < a.n_pairs) ? row_scale(a, 0, orow) : 1.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) h[q] = sc * v[q];
    }
    const uint32_t p0 = f32x2_to_bf16x2(h[0], h[1]), p1 = f32x2_to_bf16x2(h[2], h[3]);
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + orow * a.ldo + col;
    *reinterpret_cast<uint2*>(dst) = make_uint2(p0, p1);
    if (kAmax) {
      float r0, r1, r2, r3;
      bf16x2_to_f32(p0, r0, r1);
      bf16x2_to_f32(p1, r2, r3);
      const float m = fmaxf(fmaxf(fabsf(r0), fabsf(r1)), fmaxf(fabsf(r2), fabsf(r3)));
      atomicMax(&s_max[orow - first_row], __float_as_uint(m));
    }
  }
  if (kAmax) {
    __syncthreads();
    const long long row = first_row + threadIdx.x;
    if (s_max[threadIdx.x] != 0u && row < a.R) atomicMax(a.h_amax + row, s_max[threadIdx.x]);
  }
}

// The down projection's split-K partials reduced straight into y, in place
// of splitk_reduce_kernel<EPI_DOWN> followed by the combine: for token t,
//   y[t] = sum over its kept slots, then its shared experts, of
//          bf16(g * sum over splits of partial[split][row])
// -- the values the reduction would have written to y_perm, summed in fp32
// in the combine's order -- so the bits are those of the two kernels. When
// the GEMM ran unsplit (S = 1, decided on the device as it does) the rows
// are read from y_perm instead. One thread per token and four output
// columns; a term's S partial loads are issued together before any is
// added, as in splitk_reduce_kernel.
constexpr int kCombineThreads = 128;  // small blocks: a decode step's few rows reach more SMs
template <int NT>
__global__ void __launch_bounds__(kCombineThreads) splitk_combine_kernel(
    const GemmArgs a, int gemm_grid, const int32_t* __restrict__ inv_pos,
    const float* __restrict__ topk_w, __nv_bfloat16* __restrict__ y, int T, int k, int n_shared) {
  __shared__ int s_splits;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0)  // once a block: the choice loops over the split factors
    s_splits = choose_splits(__ldg(a.seg + 1) * a.NT, gemm_grid, (a.K + 63) / 64, a.s_max);
  const int d = a.n_out;
  const int groups = d / 4;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const bool in = i < (long long)T * groups;
  const long long t = in ? i / groups : 0;
  const int c = in ? (int)(i - t * groups) * 4 : 0;
  const long long P = (long long)T * k;
  // the terms' rows (-1: dropped) and gate weights, loaded while the split
  // count is being chosen
  long long row[NT];
  float g[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    row[j] = -1;
    g[j] = 1.0f;
    if (in && j < k + n_shared) {
      if (j < k) {
        const int pos = __ldg(inv_pos + t * k + j);
        g[j] = __ldg(topk_w + t * k + j);
        if (pos >= 0 && pos < P) row[j] = pos;
      } else {
        row[j] = P + (long long)(j - k) * T + t;
      }
    }
  }
  __syncthreads();
  if (!in) return;
  const int S = s_splits;
  const __nv_bfloat16* yp = static_cast<const __nv_bfloat16*>(a.out);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    if (row[j] < 0) continue;  // dropped (or past the terms): contributes nothing
    float v[4];
    if (S == 1) {
      const uint2 q = __ldg(reinterpret_cast<const uint2*>(yp + row[j] * a.ldo + c));
      bf16x2_to_f32(q.x, v[0], v[1]);
      bf16x2_to_f32(q.y, v[2], v[3]);
    } else {
      float4 pv[kMaxSplitK];
#pragma unroll
      for (int sp = 0; sp < kMaxSplitK; ++sp)
        if (sp < S)
          pv[sp] = __ldcg(reinterpret_cast<const float4*>(
              a.partial + ((long long)sp * a.R + row[j]) * a.pc + c));
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int sp = 0; sp < kMaxSplitK; ++sp) {
        if (sp < S) {
          s4[0] += pv[sp].x;
          s4[1] += pv[sp].y;
          s4[2] += pv[sp].z;
          s4[3] += pv[sp].w;
        }
      }
      const uint32_t p0 = f32x2_to_bf16x2(g[j] * s4[0], g[j] * s4[1]);
      const uint32_t p1 = f32x2_to_bf16x2(g[j] * s4[2], g[j] * s4[3]);
      bf16x2_to_f32(p0, v[0], v[1]);
      bf16x2_to_f32(p1, v[2], v[3]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = fmaf(1.0f, v[q], acc[q]);
  }
  *reinterpret_cast<uint2*>(y + t * d + c) =
      make_uint2(f32x2_to_bf16x2(acc[0], acc[1]), f32x2_to_bf16x2(acc[2], acc[3]));
}

// ---------------------------------------------------------------- host side --
template <int EPI, int OP>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& a_sh, const CUtensorMap& b0,
                        const CUtensorMap& b1, const GemmArgs& args, int max_tiles,
                        cudaStream_t s, const SfMaps* sf = nullptr, bool skip_reduce = false) {
  static const SfMaps no_sf{};  // never read by the bf16 and E4M3 kernels
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI, OP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Op<OP>::SMEM);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  // With split-K possible every SM takes part; otherwise no more CTAs than tiles.
  const int grid = (args.s_max > 1 || max_tiles >= num_sms()) ? num_sms() : max_tiles;
  if (grid <= 0) return cudaSuccess;
  cudaError_t e;
  {
    ProfScope p(gu_like(EPI)              ? K_GATE_UP
                : EPI == EPI_SWIGLU_BWD ? K_BWD_DH
                : EPI == EPI_DGRAD      ? K_BWD_DA
                                        : K_DOWN,
                s);
    e = launch_pdl(grouped_gemm_kernel<EPI, OP>, dim3(grid), dim3(Op<OP>::THREADS), Op<OP>::SMEM, s, 1, a,
                   a_sh, b0, b1, args, sf ? *sf : no_sf);
  }
  if (e != cudaSuccess || args.s_max <= 1 || skip_reduce) return e;
  const long long n = args.R * (args.n_out / 4);
  ProfScope p(K_SPLITK_REDUCE, s);
  return launch_pdl(splitk_reduce_kernel<EPI, OP>, dim3((unsigned)((n + 255) / 256)), dim3(256), 0,
                    s, 1, args, grid);
}

template <int EPI, int OP>
cudaError_t launch_decode(const CUtensorMap& w0, const CUtensorMap& w1, const CUtensorMap& tok,
                          const CUtensorMap& tok_sh, const GemmArgs& args, int max_rows,
                          cudaStream_t s, bool skip_reduce = false) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(grouped_decode_kernel<EPI, OP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)DYN_SMEM_DECODE);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  DecodeShape sh;
  sh.a_bytes = (EPI == EPI_SWIGLU) ? 2 * A_BYTES : A_BYTES;
  const int tok_bytes = ((max_rows + TOK_BOX - 1) / TOK_BOX) * TOK_BOX_BYTES;
  sh.stage_bytes = (sh.a_bytes + tok_bytes + 1023) / 1024 * 1024;
  sh.stages = std::min(kDecodeMaxStages, (int)((DYN_SMEM_DECODE - 1024) / sh.stage_bytes));
  const int grid = num_sms();
  cudaError_t e;
  {
    ProfScope p(EPI == EPI_SWIGLU ? K_GATE_UP : K_DOWN, s);
    e = launch_pdl(grouped_decode_kernel<EPI, OP>, dim3(grid), dim3(THREADS), DYN_SMEM_DECODE, s, 1,
                   w0, w1, tok, tok_sh, args, sh);
  }
  if (e != cudaSuccess || args.s_max <= 1 || skip_reduce) return e;
  const long long n = args.R * (args.n_out / 4);
  ProfScope p(K_SPLITK_REDUCE, s);
  return launch_pdl(splitk_reduce_kernel<EPI, OP>, dim3((unsigned)((n + 255) / 256)), dim3(256), 0,
                    s, 1, args, grid);
}

long long mt_bound_of(const moe_config& c, int tile_m) {
  // Upper bound of M tiles: every segment may end in a partial tile.
  const long long P = (long long)c.T * c.top_k;
  return (P + tile_m - 1) / tile_m + c.n_experts +
         (long long)c.n_shared * ((c.T + tile_m - 1) / tile_m);
}

cudaError_t configure_pair_kernels() {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device == dev) return cudaSuccess;
  const void* kernels[4] = {(const void*)grouped_gemm_pair_kernel<EPI_SWIGLU, OP_BF16>,
                            (const void*)grouped_gemm_pair_kernel<EPI_DOWN, OP_BF16>,
                            (const void*)grouped_gemm_pair_kernel<EPI_SWIGLU, OP_E4M3>,
                            (const void*)grouped_gemm_pair_kernel<EPI_DOWN, OP_E4M3>};
  cudaError_t e = cudaSuccess;
  for (const void* k : kernels)
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DYN_SMEM_PAIR);
  if (e == cudaSuccess) configured_device = dev;
  return e;
}

// Clusters of 2 that can be resident at once with one CTA per SM (0 if the
// pair kernels cannot be configured on this device).
int max_pair_clusters() {
  static thread_local int cached_dev = -1, cached = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (cached_dev == dev) return cached;
  if (configure_pair_kernels() != cudaSuccess) {
    cudaGetLastError();
    cached_dev = dev;
    cached = 0;
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (num_sms() / 2));
  cfg.blockDim = dim3(G_THREADS);
  cfg.dynamicSmemBytes = DYN_SMEM_PAIR;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<EPI_SWIGLU, OP_BF16>, &cfg) !=
      cudaSuccess)
    n = 0;
  cudaGetLastError();  // clear a failed query
  cached_dev = dev;
  cached = n;
  return n;
}

template <int EPI, int OP>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& a_sh, const CUtensorMap& b0,
                        const CUtensorMap& b1, const GemmArgs& args, int max_tiles,
                        cudaStream_t s) {
  const int clusters = std::min(max_tiles, max_pair_clusters());
  if (clusters <= 0) return cudaSuccess;
  ProfScope p(EPI == EPI_SWIGLU ? K_GATE_UP : K_DOWN, s);
  return launch_pdl(grouped_gemm_pair_kernel<EPI, OP>, dim3(2 * clusters), dim3(G_THREADS),
                    DYN_SMEM_PAIR, s, 2, a, a_sh, b0, b1, args);
}

cudaError_t launch_splitk_combine(const moe_config& c, const GemmArgs& d, int gemm_grid,
                                  const int32_t* inv_pos, const float* topk_w, void* y,
                                  cudaStream_t s) {
  const int terms = c.top_k + c.n_shared;
  const dim3 grid((unsigned)ceil_div((long long)c.T * (c.d_model / 4), kCombineThreads));
  __nv_bfloat16* yo = static_cast<__nv_bfloat16*>(y);
  ProfScope p(K_COMBINE, s);
  if (terms <= 2)
    return launch_pdl(splitk_combine_kernel<2>, grid, dim3(kCombineThreads), 0, s, 1, d, gemm_grid, inv_pos,
                      topk_w, yo, c.T, c.top_k, c.n_shared);
  if (terms <= 4)
    return launch_pdl(splitk_combine_kernel<4>, grid, dim3(kCombineThreads), 0, s, 1, d, gemm_grid, inv_pos,
                      topk_w, yo, c.T, c.top_k, c.n_shared);
  if (terms <= 8)
    return launch_pdl(splitk_combine_kernel<8>, grid, dim3(kCombineThreads), 0, s, 1, d, gemm_grid, inv_pos,
                      topk_w, yo, c.T, c.top_k, c.n_shared);
  return launch_pdl(splitk_combine_kernel<kMaxTopK + kMaxShared>, grid, dim3(kCombineThreads), 0, s, 1, d,
                    gemm_grid, inv_pos, topk_w, yo, c.T, c.top_k, c.n_shared);
}

cudaError_t configure_swap_kernels() {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device == dev) return cudaSuccess;
  const void* kernels[5] = {(const void*)grouped_swap_pair_kernel<EPI_SWIGLU, OP_BF16, false>,
                            (const void*)grouped_swap_pair_kernel<EPI_DOWN, OP_BF16, false>,
                            (const void*)grouped_swap_pair_kernel<EPI_SWIGLU, OP_E4M3, false>,
                            (const void*)grouped_swap_pair_kernel<EPI_DOWN, OP_E4M3, false>,
                            (const void*)grouped_swap_pair_kernel<EPI_SWIGLU, OP_BF16, true>};
  const size_t smem[5] = {Sw<EPI_SWIGLU>::SMEM, Sw<EPI_DOWN>::SMEM, Sw<EPI_SWIGLU>::SMEM,
                          Sw<EPI_DOWN>::SMEM, Sw<EPI_SWIGLU>::SMEM};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 5 && e == cudaSuccess; ++i)
    e = cudaFuncSetAttribute(kernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem[i]);
  if (e == cudaSuccess) configured_device = dev;
  return e;
}

// Token maps of the weight-stationary pair kernel: one per box height.
bool make_tok_maps(TokMaps* m, const void* base, long long rows, long long cols, bool u8) {
  for (int i = 0; i < SW_TOK_BOXES; ++i) {
    const unsigned h = 16u * (unsigned)(i + 1);
    if (!(u8 ? make_map_u8(&m->box[i], base, rows, cols, h) : make_map(&m->box[i], base, rows, cols, h)))
      return false;
  }
  return true;
}

template <int EPI, int OP, bool GATHER = false>
cudaError_t launch_swap_pair(const CUtensorMap& w0, const CUtensorMap& w1, const TokMaps& tok,
                             const TokMaps& tok_sh, const GemmArgs& args, int max_tiles,
                             cudaStream_t s) {
  static_assert(Sw<EPI>::SMEM <= DYN_SMEM_PAIR, "resident like the pair kernel");
  cudaError_t e = configure_swap_kernels();
  if (e != cudaSuccess) return e;
  const int clusters = std::min(max_tiles, max_pair_clusters());
  if (clusters <= 0) return cudaSuccess;
  ProfScope p(EPI == EPI_SWIGLU ? K_GATE_UP : K_DOWN, s);
  return launch_pdl(grouped_swap_pair_kernel<EPI, OP, GATHER>, dim3(2 * clusters),
                    dim3(GATHER ? G_THREADS + SW_GATHER_THREADS : G_THREADS), Sw<EPI>::SMEM, s, 2,
                    w0, w1, tok,
                    tok_sh, args);
}

}  // namespace

int gemm_tiles(const moe_config& c) {
  if (c.dtype != MOE_BF16 || c.n_experts <= 0) return MOE_TILES_CTA;
  const bool pairs_ok = max_pair_clusters() > 0;
  if (c.tiles == MOE_TILES_CTA) return MOE_TILES_CTA;
  if (c.tiles == MOE_TILES_PAIR || c.tiles == MOE_TILES_WEIGHT_PAIR)
    return pairs_ok ? c.tiles : MOE_TILES_CTA;
  // Chosen here: a projection that may be split along K (few rows) runs
  // 1-CTA tiles (or swap-AB decode tiles); every larger batch runs the
  // weight-stationary pairs, which were as fast as or faster than 256-row
  // pair tiles on every measured layer (equal on 128 Zipf-skewed experts,
  // 4% faster on 8 experts of ~1024 rows, 12% faster on 256 experts of
  // ~256 rows, where 256-row tiles are a third padding).
  const SplitKPlan plan = splitk_plan(c);
  if (plan.s_max_gu > 1 || plan.s_max_dn > 1 || !pairs_ok) return MOE_TILES_CTA;
  return MOE_TILES_WEIGHT_PAIR;
}

bool gather_fused(const moe_config& c) {
  if (c.dtype != MOE_BF16 || gemm_tiles(c) != MOE_TILES_WEIGHT_PAIR) return false;
  return c.gather == MOE_GATHER_FUSED;
}

bool use_pair_tiles(const moe_config& c) { return gemm_tiles(c) != MOE_TILES_CTA; }

int seg_tile_m(const moe_config& c) { return use_pair_tiles(c) ? PAIR_TILE_M : BM; }

SplitKPlan splitk_plan(const moe_config& c) {
  SplitKPlan p{1, 1, 0};
  if (c.dtype != MOE_BF16) return p;
  const long long R = (long long)c.T * (c.top_k + c.n_shared);
  if (R == 0) return p;
  const size_t per_gu = (size_t)R * 2 * c.d_ff * sizeof(float);
  const size_t per_dn = (size_t)R * c.d_model * sizeof(float);
  auto smax = [](size_t per) {
    const size_t s = kSplitKBudget / per;
    return s >= 2 ? (int)(s < (size_t)kMaxSplitK ? s : (size_t)kMaxSplitK) : 1;
  };
  p.s_max_gu = smax(per_gu);
  p.s_max_dn = smax(per_dn);
  const size_t b_gu = p.s_max_gu > 1 ? p.s_max_gu * per_gu : 0;
  const size_t b_dn = p.s_max_dn > 1 ? p.s_max_dn * per_dn : 0;
  p.partial_bytes = b_gu > b_dn ? b_gu : b_dn;
  return p;
}

cudaError_t launch_grouped_bf16(const moe_config& c, const void* x_perm, const void* x,
                                const int32_t* seg, const int32_t* sorted_pair,
                                const float* topk_w, const void* w_gate, const void* w_up,
                                const void* w_down, void* h, void* y_perm, float* partial,
                                long long xp_rows, long long h_rows, int* status, cudaStream_t s,
                                const int32_t* inv_pos, void* y, bool* combined) {
  if (combined) *combined = false;
  const long long P = (long long)c.T * c.top_k;
  const int E = c.n_experts + c.n_shared;
  const long long R = P + (long long)c.n_shared * c.T;  // rows of H and y_perm
  if (R == 0) return cudaSuccess;
  const int tiles = gemm_tiles(c);
  const bool pair = tiles != MOE_TILES_CTA;
  const bool decode = !pair && c.T <= kDecodeMaxRows;  // every segment has <= 64 rows
  const long long mt_bound = mt_bound_of(c, pair ? PAIR_TILE_M : BM);
  const SplitKPlan plan = splitk_plan(c);
  if (pair) {
    cudaError_t e = configure_pair_kernels();
    if (e != cudaSuccess) return e;
  }

  // x_perm is null when the gate/up kernel gathers the rows itself; its maps
  // then point at x and are not used
  const bool has_xp = P > 0 && x_perm != nullptr;
  const void* xp = has_xp ? x_perm : x;
  const long long xp_n = has_xp ? std::max(P, xp_rows) : c.T;
  CUtensorMap m_xp, m_x, m_wg, m_wu, m_h, m_wd;
  const bool ok =
      make_map(&m_xp, xp, xp_n, c.d_model) &&
      make_map(&m_x, c.n_shared > 0 ? x : xp, c.n_shared > 0 ? c.T : (has_xp ? P : c.T),
               c.d_model) &&
      make_map(&m_wg, w_gate, (long long)E * c.d_ff, c.d_model) &&
      make_map(&m_wu, w_up, (long long)E * c.d_ff, c.d_model) &&
      make_map(&m_h, h, std::max(R, h_rows), c.d_ff) &&
      make_map(&m_wd, w_down, (long long)E * c.d_model, c.d_ff);
  if (!ok) return cudaErrorInvalidValue;

  GemmArgs g{};
  g.seg = seg;
  g.sorted_pair = sorted_pair;
  g.topk_w = nullptr;
  g.out = h;
  g.status = status;
  g.ldo = c.d_ff;
  g.n_routed = c.n_experts;
  g.n_pairs = (int)P;
  g.K = c.d_model;
  g.n_out = c.d_ff;
  g.NT = (c.d_ff + 127) / 128;
  g.b_rows = c.d_ff;
  g.partial = partial;
  g.s_max = plan.s_max_gu;
  g.pc = 2 * c.d_ff;
  g.R = R;
  g.a_scale = g.a_scale_shared = g.b_scale0 = g.b_scale1 = nullptr;
  g.h_amax = nullptr;
  if (decode) {
    // token tiles of 16 rows over x_perm / x (gate/up) and H (down)
    CUtensorMap t_xp, t_x, t_h;
    const bool ok2 = make_map(&t_xp, xp, xp_n, c.d_model, TOK_BOX) &&
                     make_map(&t_x, c.n_shared > 0 ? x : xp,
                              c.n_shared > 0 ? c.T : (has_xp ? P : c.T), c.d_model, TOK_BOX) &&
                     make_map(&t_h, h, std::max(R, h_rows), c.d_ff, TOK_BOX);
    if (!ok2) return cudaErrorInvalidValue;
    const int max_rows = c.T;  // a segment holds at most T rows
    cudaError_t e = launch_decode<EPI_SWIGLU, OP_BF16>(m_wg, m_wu, t_xp, t_x, g, max_rows, s);
    if (e != cudaSuccess) return e;
    GemmArgs d = g;
    d.topk_w = topk_w;
    d.out = y_perm;
    d.ldo = c.d_model;
    d.K = c.d_ff;
    d.n_out = c.d_model;
    d.NT = (c.d_model + BM - 1) / BM;
    d.b_rows = c.d_model;
    d.s_max = plan.s_max_dn;
    d.pc = c.d_model;
    // with y given, a split down projection is reduced straight into y
    const bool fuse = y != nullptr && inv_pos != nullptr && topk_w != nullptr && d.s_max > 1;
    e = launch_decode<EPI_DOWN, OP_BF16>(m_wd, m_wd, t_h, t_h, d, max_rows, s, fuse);
    if (e != cudaSuccess || !fuse) return e;
    *combined = true;
    return launch_splitk_combine(c, d, num_sms(), inv_pos, topk_w, y, s);
  }

  GemmArgs d = g;
  d.topk_w = topk_w;
  d.out = y_perm;
  d.ldo = c.d_model;
  d.K = c.d_ff;
  d.n_out = c.d_model;
  d.NT = (c.d_model + 255) / 256;
  d.b_rows = c.d_model;
  d.s_max = plan.s_max_dn;
  d.pc = c.d_model;
  if (tiles == MOE_TILES_WEIGHT_PAIR) {
    // weights on the MMA's M side, 256 features a pair tile; token boxes
    // of 128..8 rows over x_perm / x (gate/up) and H (down)
    TokMaps t_xp, t_x, t_h;
    if (!make_tok_maps(&t_xp, xp, xp_n, c.d_model, false) ||
        !make_tok_maps(&t_x, c.n_shared > 0 ? x : xp, c.n_shared > 0 ? c.T : (has_xp ? P : c.T),
                       c.d_model, false) ||
        !make_tok_maps(&t_h, h, std::max(R, h_rows), c.d_ff, false))
      return cudaErrorInvalidValue;
    g.NT = (c.d_ff + 255) / 256;
    g.s_max = d.s_max = 1;
    cudaError_t e;
    if (!has_xp && P > 0) {  // the row gather runs inside the gate/up kernel
      g.gx = static_cast<const __nv_bfloat16*>(x);
      g.gk = c.top_k;
      g.gT = c.T;
      e = launch_swap_pair<EPI_SWIGLU, OP_BF16, true>(m_wg, m_wu, t_xp, t_x, g,
                                                      (int)(mt_bound * g.NT), s);
    } else {
      e = launch_swap_pair<EPI_SWIGLU, OP_BF16>(m_wg, m_wu, t_xp, t_x, g, (int)(mt_bound * g.NT),
                                                s);
    }
    if (e != cudaSuccess) return e;
    return launch_swap_pair<EPI_DOWN, OP_BF16>(m_wd, m_wd, t_h, t_h, d, (int)(mt_bound * d.NT), s);
  }
  cudaError_t e = pair ? launch_pair<EPI_SWIGLU, OP_BF16>(m_xp, m_x, m_wg, m_wu, g,
                                                         (int)(mt_bound * g.NT), s)
                       : launch_gemm<EPI_SWIGLU, OP_BF16>(m_xp, m_x, m_wg, m_wu, g,
                                                          (int)(mt_bound * g.NT), s);
  if (e != cudaSuccess) return e;
  if (pair)
    return launch_pair<EPI_DOWN, OP_BF16>(m_h, m_h, m_wd, m_wd, d, (int)(mt_bound * d.NT), s);
  const bool fuse = y != nullptr && inv_pos != nullptr && topk_w != nullptr && d.s_max > 1;
  e = launch_gemm<EPI_DOWN, OP_BF16>(m_h, m_h, m_wd, m_wd, d, (int)(mt_bound * d.NT), s, nullptr,
                                     fuse);
  if (e != cudaSuccess || !fuse) return e;
  *combined = true;
  return launch_splitk_combine(c, d, num_sms(), inv_pos, topk_w, y, s);
}

cudaError_t launch_grouped_e4m3(const moe_config& c, const uint8_t* xq_perm,
                                const float* xp_scale, const uint8_t* xq, const float* x_scale,
                                const int32_t* seg, const int32_t* sorted_pair,
                                const float* topk_w, const uint8_t* wg_q, const float* wg_s,
                                const uint8_t* wu_q, const float* wu_s, const uint8_t* wd_q,
                                const float* wd_s, void* h, unsigned* h_amax, uint8_t* hq,
                                float* h_scale, void* y_perm, float* partial, long long xp_rows,
                                long long h_rows, int* status, cudaStream_t s) {
  const long long P = (long long)c.T * c.top_k;
  const int E = c.n_experts + c.n_shared;
  const long long R = P + (long long)c.n_shared * c.T;
  if (R == 0) return cudaSuccess;
  const int tiles = gemm_tiles(c);
  const bool pair = tiles != MOE_TILES_CTA;
  const bool decode = !pair && c.T <= kDecodeMaxRows;
  const long long mt_bound = mt_bound_of(c, pair ? PAIR_TILE_M : BM);
  const SplitKPlan plan = splitk_plan(c);
  if (pair) {
    cudaError_t e = configure_pair_kernels();
    if (e != cudaSuccess) return e;
  }
  // A tensors: routed token rows (x_perm) and, for shared experts, x itself
  const void* a_r = P > 0 ? (const void*)xq_perm : (const void*)xq;
  const long long a_r_rows = P > 0 ? std::max(P, xp_rows) : c.T;
  const void* a_s = c.n_shared > 0 ? (const void*)xq : a_r;
  const long long a_s_rows = c.n_shared > 0 ? padded_rows(c.T) : a_r_rows;  // x_q is padded

  GemmArgs g{};
  g.seg = seg;
  g.sorted_pair = sorted_pair;
  g.topk_w = nullptr;
  g.out = h;
  g.status = status;
  g.ldo = c.d_ff;
  g.n_routed = c.n_experts;
  g.n_pairs = (int)P;
  g.K = c.d_model;
  g.n_out = c.d_ff;
  g.NT = (c.d_ff + 127) / 128;
  g.b_rows = c.d_ff;
  g.partial = partial;
  g.s_max = plan.s_max_gu;
  g.pc = 2 * c.d_ff;
  g.R = R;
  g.a_scale = xp_scale;
  g.a_scale_shared = x_scale;
  g.b_scale0 = wg_s;
  g.b_scale1 = wu_s;
  g.h_amax = h_amax;
  GemmArgs d = g;
  d.topk_w = topk_w;
  d.out = y_perm;
  d.ldo = c.d_model;
  d.K = c.d_ff;
  d.n_out = c.d_model;
  d.b_rows = c.d_model;
  d.s_max = plan.s_max_dn;
  d.pc = c.d_model;
  d.a_scale = h_scale;
  d.a_scale_shared = h_scale;
  d.b_scale0 = wd_s;
  d.b_scale1 = wd_s;
  d.h_amax = nullptr;
  // H (bf16, with its rows' max |H|) -> E4M3 codes and row scales
  QuantArgs qh{};
  qh.src = static_cast<const __nv_bfloat16*>(h);
  qh.rows = R;
  qh.cols = c.d_ff;
  qh.amax_in = h_amax;
  qh.q = hq;
  qh.scale = h_scale;

  CUtensorMap m_wg, m_wu, m_wd;
  if (!make_map_u8(&m_wg, wg_q, (long long)E * c.d_ff, c.d_model) ||
      !make_map_u8(&m_wu, wu_q, (long long)E * c.d_ff, c.d_model) ||
      !make_map_u8(&m_wd, wd_q, (long long)E * c.d_model, c.d_ff))
    return cudaErrorInvalidValue;
  const unsigned box = decode ? TOK_BOX : (unsigned)BM;
  CUtensorMap m_xp, m_x, m_h;
  if (!make_map_u8(&m_xp, a_r, a_r_rows, c.d_model, box) ||
      !make_map_u8(&m_x, a_s, a_s_rows, c.d_model, box) ||
      !make_map_u8(&m_h, hq, std::max(R, h_rows), c.d_ff, box))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (decode) {
    const int max_rows = c.T;  // a segment holds at most T rows
    e = launch_decode<EPI_SWIGLU, OP_E4M3>(m_wg, m_wu, m_xp, m_x, g, max_rows, s);
    if (e == cudaSuccess) e = launch_quantize_rows(qh, s);
    if (e != cudaSuccess) return e;
    d.NT = (c.d_model + BM - 1) / BM;
    return launch_decode<EPI_DOWN, OP_E4M3>(m_wd, m_wd, m_h, m_h, d, max_rows, s);
  }
  d.NT = (c.d_model + 255) / 256;
  if (tiles == MOE_TILES_WEIGHT_PAIR) {
    TokMaps t_xp, t_x, t_h;
    if (!make_tok_maps(&t_xp, a_r, a_r_rows, c.d_model, true) ||
        !make_tok_maps(&t_x, a_s, a_s_rows, c.d_model, true) ||
        !make_tok_maps(&t_h, hq, std::max(R, h_rows), c.d_ff, true))
      return cudaErrorInvalidValue;
    g.NT = (c.d_ff + 255) / 256;
    g.s_max = d.s_max = 1;
    e = launch_swap_pair<EPI_SWIGLU, OP_E4M3>(m_wg, m_wu, t_xp, t_x, g, (int)(mt_bound * g.NT), s);
    if (e == cudaSuccess) e = launch_quantize_rows(qh, s);
    if (e != cudaSuccess) return e;
    return launch_swap_pair<EPI_DOWN, OP_E4M3>(m_wd, m_wd, t_h, t_h, d, (int)(mt_bound * d.NT), s);
  }
  e = pair ? launch_pair<EPI_SWIGLU, OP_E4M3>(m_xp, m_x, m_wg, m_wu, g, (int)(mt_bound * g.NT), s)
           : launch_gemm<EPI_SWIGLU, OP_E4M3>(m_xp, m_x, m_wg, m_wu, g, (int)(mt_bound * g.NT), s);
  if (e == cudaSuccess) e = launch_quantize_rows(qh, s);
  if (e != cudaSuccess) return e;
  return pair ? launch_pair<EPI_DOWN, OP_E4M3>(m_h, m_h, m_wd, m_wd, d, (int)(mt_bound * d.NT), s)
              : launch_gemm<EPI_DOWN, OP_E4M3>(m_h, m_h, m_wd, m_wd, d, (int)(mt_bound * d.NT), s);
}

cudaError_t launch_grouped_nvf4(const moe_config& c, Nvf4Matrix xp, Nvf4Matrix xs,
                                const int32_t* seg, const int32_t* sorted_pair,
                                const float* topk_w, Nvf4Matrix wg, Nvf4Matrix wu, Nvf4Matrix wd,
                                void* h, unsigned* h_amax, uint8_t* hq, uint8_t* h_sf,
                                float* h_scale, void* y_perm, float* partial, long long xp_rows,
                                long long xs_rows, long long h_rows, int* status, cudaStream_t s) {
  const long long P = (long long)c.T * c.top_k;
  const int E = c.n_experts + c.n_shared;
  const long long R = P + (long long)c.n_shared * c.T;
  if (R == 0) return cudaSuccess;
  const long long mt_bound = mt_bound_of(c, BM);
  const SplitKPlan plan = splitk_plan(c);
  // the shared experts' A rows (x); without shared experts the map is unused
  const Nvf4Matrix as = c.n_shared > 0 ? xs : xp;
  const long long as_rows = c.n_shared > 0 ? xs_rows : xp_rows;
  const long long sfd = nvf4_sf_stride(c.d_model), sff = nvf4_sf_stride(c.d_ff);

  GemmArgs g{};
  g.seg = seg;
  g.sorted_pair = sorted_pair;
  g.topk_w = nullptr;
  g.out = h;
  g.status = status;
  g.ldo = c.d_ff;
  g.n_routed = c.n_experts;
  g.n_pairs = (int)P;
  g.K = c.d_model;
  g.n_out = c.d_ff;
  g.NT = (c.d_ff + 127) / 128;
  g.b_rows = c.d_ff;
  g.partial = partial;
  g.s_max = plan.s_max_gu;
  g.pc = 2 * c.d_ff;
  g.R = R;
  g.a_scale = xp.scale;
  g.a_scale_shared = as.scale;
  g.b_scale0 = wg.scale;
  g.b_scale1 = wu.scale;
  g.h_amax = h_amax;
  GemmArgs d = g;
  d.topk_w = topk_w;
  d.out = y_perm;
  d.ldo = c.d_model;
  d.K = c.d_ff;
  d.n_out = c.d_model;
  d.NT = (c.d_model + 255) / 256;
  d.b_rows = c.d_model;
  d.s_max = plan.s_max_dn;
  d.pc = c.d_model;
  d.a_scale = h_scale;
  d.a_scale_shared = h_scale;
  d.b_scale0 = wd.scale;
  d.b_scale1 = wd.scale;
  d.h_amax = nullptr;
  // H (bf16, with its rows' max |H|) -> NVFP4
  QuantArgs qh{};
  qh.src = static_cast<const __nv_bfloat16*>(h);
  qh.rows = R;
  qh.cols = c.d_ff;
  qh.amax_in = h_amax;
  qh.q = hq;
  qh.sf = h_sf;
  qh.ld_sf = (int)sff;
  qh.scale = h_scale;

  // codes: bytes [rows][K / 2]; block scales: bytes [rows][stride]
  CUtensorMap m_xp, m_x, m_wg, m_wu, m_h, m_wd;
  SfMaps sg, sd;
  const long long wrows_ff = (long long)E * c.d_ff, wrows_d = (long long)E * c.d_model;
  if (!make_map_u8(&m_xp, xp.q, xp_rows, c.d_model / 2) ||
      !make_map_u8(&m_x, as.q, as_rows, c.d_model / 2) ||
      !make_map_u8(&m_wg, wg.q, wrows_ff, c.d_model / 2) ||
      !make_map_u8(&m_wu, wu.q, wrows_ff, c.d_model / 2) ||
      !make_map_u8(&m_h, hq, h_rows, c.d_ff / 2) ||
      !make_map_u8(&m_wd, wd.q, wrows_d, c.d_ff / 2) ||
      !make_map_sf(&sg.a, xp.sf, xp_rows, sfd) || !make_map_sf(&sg.a_shared, as.sf, as_rows, sfd) ||
      !make_map_sf(&sg.b0, wg.sf, wrows_ff, sfd) || !make_map_sf(&sg.b1, wu.sf, wrows_ff, sfd) ||
      !make_map_sf(&sd.a, h_sf, h_rows, sff) || !make_map_sf(&sd.b0, wd.sf, wrows_d, sff))
    return cudaErrorInvalidValue;
  sd.a_shared = sd.a;
  sd.b1 = sd.b0;
  cudaError_t e = launch_gemm<EPI_SWIGLU, OP_NVF4>(m_xp, m_x, m_wg, m_wu, g,
                                                   (int)(mt_bound * g.NT), s, &sg);
  if (e == cudaSuccess) e = launch_quantize_rows_nvf4(qh, s);
  if (e != cudaSuccess) return e;
  return launch_gemm<EPI_DOWN, OP_NVF4>(m_h, m_h, m_wd, m_wd, d, (int)(mt_bound * d.NT), s, &sd);
}

// ---- backward -----------------------------------------------------------------

namespace {
GemmArgs bwd_args(const moe_config& c, const int32_t* seg, int* status, long long R) {
  GemmArgs g{};
  g.seg = seg;
  g.status = status;
  g.n_routed = c.n_experts;
  g.n_pairs = (int)((long long)c.T * c.top_k);
  g.s_max = 1;
  g.R = R;
  return g;
}
}  // namespace

cudaError_t launch_bwd_recompute(const moe_config& c, const void* x_perm, const void* x,
                                 const int32_t* seg, const void* w_gate, const void* w_up,
                                 const void* w_down, void* h, void* ab, void* o, long long xp_rows,
                                 long long r_rows, int* status, cudaStream_t s) {
  const long long P = (long long)c.T * c.top_k;
  const int E = c.n_experts + c.n_shared;
  const long long R = P + (long long)c.n_shared * c.T;
  if (R == 0) return cudaSuccess;
  CUtensorMap m_xp, m_x, m_wg, m_wu, m_h, m_wd;
  const bool ok = make_map(&m_xp, x_perm, std::max(P, xp_rows), c.d_model) &&
                  make_map(&m_x, c.n_shared > 0 ? x : x_perm, c.n_shared > 0 ? c.T : P,
                           c.d_model) &&
                  make_map(&m_wg, w_gate, (long long)E * c.d_ff, c.d_model) &&
                  make_map(&m_wu, w_up, (long long)E * c.d_ff, c.d_model) &&
                  make_map(&m_h, h, std::max(R, r_rows), c.d_ff) &&
                  make_map(&m_wd, w_down, (long long)E * c.d_model, c.d_ff);
  if (!ok) return cudaErrorInvalidValue;
  const long long mt = mt_bound_of(c, BM);
  GemmArgs g = bwd_args(c, seg, status, R);
  g.out = h;
  g.ldo = c.d_ff;
  g.K = c.d_model;
  g.n_out = c.d_ff;
  g.NT = (c.d_ff + 127) / 128;
  g.b_rows = c.d_ff;
  g.pc = 2 * c.d_ff;
  g.aux = static_cast<__nv_bfloat16*>(ab);
  g.ld_aux = 2LL * c.d_ff;
  cudaError_t e = launch_gemm<EPI_SWIGLU_SAVE, OP_BF16>(m_xp, m_x, m_wg, m_wu, g, (int)(mt * g.NT), s);
  if (e != cudaSuccess) return e;
  GemmArgs d = bwd_args(c, seg, status, R);  // unweighted: topk_w null
  d.out = o;
  d.ldo = c.d_model;
  d.K = c.d_ff;
  d.n_out = c.d_model;
  d.NT = (c.d_model + 255) / 256;
  d.b_rows = c.d_model;
  d.pc = c.d_model;
  return launch_gemm<EPI_DOWN, OP_BF16>(m_h, m_h, m_wd, m_wd, d, (int)(mt * d.NT), s);
}

cudaError_t launch_bwd_dgrad(const moe_config& c, const int32_t* seg, const void* dO,
                             const void* ab, const void* w_gate, const void* w_up,
                             const void* w_down, void* dab, void* dA, long long r_rows,
                             int* status, cudaStream_t s) {
  const long long P = (long long)c.T * c.top_k;
  const int E = c.n_experts + c.n_shared;
  const long long R = P + (long long)c.n_shared * c.T;
  if (R == 0) return cudaSuccess;
  const long long rows = std::max(R, r_rows);
  // A operands K-major (128-row boxes); B MN-major (64 x 64 boxes of the
  // weights viewed as [E * K][N])
  CUtensorMap m_do, m_dab, m_wd, m_wg, m_wu;
  const bool ok = make_map(&m_do, dO, rows, c.d_model) &&
                  make_map(&m_dab, dab, rows, 2LL * c.d_ff) &&
                  make_map(&m_wd, w_down, (long long)E * c.d_model, c.d_ff, 64) &&
                  make_map(&m_wg, w_gate, (long long)E * c.d_ff, c.d_model, 64) &&
                  make_map(&m_wu, w_up, (long long)E * c.d_ff, c.d_model, 64);
  if (!ok) return cudaErrorInvalidValue;
  const long long mt = mt_bound_of(c, BM);
  // dH = dO W_d, K = d_model; SwiGLU backward into dab
  GemmArgs g = bwd_args(c, seg, status, R);
  g.out = dab;
  g.ldo = 2LL * c.d_ff;
  g.K = c.d_model;
  g.n_out = c.d_ff;
  g.NT = (c.d_ff + 255) / 256;
  g.b_rows = c.d_model;
  g.kb_split = (c.d_model + BK - 1) / BK;
  g.aux = static_cast<__nv_bfloat16*>(const_cast<void*>(ab));
  g.ld_aux = 2LL * c.d_ff;
  cudaError_t e =
      launch_gemm<EPI_SWIGLU_BWD, OP_BF16>(m_do, m_do, m_wd, m_wd, g, (int)(mt * g.NT), s);
  if (e != cudaSuccess) return e;
  // dA = da W_g + db W_u, K = 2 d_ff (W_g rows for the first d_ff / 64 blocks)
  GemmArgs d = bwd_args(c, seg, status, R);
  d.out = dA;
  d.ldo = c.d_model;
  d.K = 2 * c.d_ff;
  d.n_out = c.d_model;
  d.NT = (c.d_model + 255) / 256;
  d.b_rows = c.d_ff;
  d.kb_split = c.d_ff / BK;
  return launch_gemm<EPI_DGRAD, OP_BF16>(m_dab, m_dab, m_wg, m_wu, d, (int)(mt * d.NT), s);
}

}  // namespace moe
