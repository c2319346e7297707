// Weight gradients of the grouped expert GEMMs on the 5th-generation tensor
// cores:
//
//   dW[e] (M x N, fp32) = A_e^T B_e,   K = the rows of expert e's segment,
//
// with A_e and B_e the segment's row slices of two bf16 matrices: for the
// gate and up projections A = da or db (columns of da | db) and B = the
// expert's input rows (x_perm, or x for a shared expert); for the down
// projection A = dO and B = H. This is the gradient of every expert's
// linear maps in "MoE inference: the call centre with 256 specialists and 8
// taking each call", "The bare mechanism" (SwiGLU experts), by the chain
// rule, summed over the tokens the expert took.
//
// Both operands are read as they lie in memory, rows along K: TMA boxes of
// 64 rows x 64 columns with the 128-byte swizzle give the MN-major layout
// tcgen05 reads directly (no transpose pass). Tiles are 128 x 256 outputs of
// one expert, persistent CTAs, warp-specialised like the forward GEMM:
// warp 0 loads (4-stage ring of 48 KB), warp 1 issues tcgen05.mma from one
// thread into one of two 256-column TMEM accumulators, warps 2-9 drain them
// (two warps per TMEM lane quarter, half the columns each): 32 x 32 fp32
// blocks go through a swizzled shared-memory buffer (one per warp) to TMA
// tensor stores, so the output leaves in whole 128-byte lines. (Measured
// alternatives, slower on these shapes: a 3-stage ring with two buffers a
// warp; CTA pairs with 256 x 256 tiles; plain coalesced stores after a
// shared-memory transpose.) The same
// kernel with one segment of K rows (no segment table) computes the router's
// two gradient products.
// A segment's last K block may run past its end into the next segment's
// rows: warp 1 zeroes those rows of both operands in shared memory (whole
// 128-byte lines, so the swizzle does not matter) and fences them to the
// async proxy before the MMAs read the stage. Experts that took no rows get
// a zero gradient written without touching the tensor cores. Waits are
// bounded as in the forward kernels.
#include <cuda.h>

#include <algorithm>

#include "device_util.cuh"
#include "moe_internal.h"
#include "sm103_ptx.cuh"
#include "sm103_wait.cuh"

namespace moe {
namespace {

constexpr int WM = 128, WN = 256, WKB = 64;
constexpr int BOX_BYTES = 64 * 128;            // 64 K rows x 64 bf16
constexpr int WA_BYTES = 2 * BOX_BYTES;        // M = 128: two boxes
constexpr int WB_BYTES = 4 * BOX_BYTES;        // N = 256: four boxes
constexpr int W_STAGE_BYTES = WA_BYTES + WB_BYTES;  // 48 KB
constexpr int W_STAGES = 4;
constexpr int W_ACC = 2;
constexpr int W_TMEM_COLS = WN * W_ACC;        // 512
constexpr int W_EPI_THREADS = 256;
constexpr int W_THREADS = 64 + W_EPI_THREADS;  // 320
constexpr int STG_BYTES = 32 * 128;              // one 32 x 32 fp32 block
constexpr int W_STG_BYTES = 8 * STG_BYTES;         // one block per epilogue warp
constexpr size_t W_DYN_SMEM = (size_t)W_STAGES * W_STAGE_BYTES + W_STG_BYTES + 1024;

struct WgradArgs {
  const int32_t* seg;  // segment table (moe_internal.h), or null: one segment
  int rows1;           // of rows1 rows from row 0 of A and B
  int* status;
  int M, N;            // one expert's gradient
  int MT, NT;          // its tiles
  int a_col0;          // first column of A taken (the up half of da | db: d_ff)
  int b_in_rows;       // 1: B rows are input rows (x_perm; x for shared experts)
  int n_routed;
};

struct __align__(8) WState {
  uint64_t full[W_STAGES];
  uint64_t empty[W_STAGES];
  uint64_t acc_full[W_ACC];
  uint64_t acc_empty[W_ACC];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct WTile {
  int e, m, n, rows, a_row, b_row;
};

// Expert-major, then N tile, then M tile.
__device__ __forceinline__ WTile wtile(const WgradArgs& a, int E, int tile) {
  const int per = a.MT * a.NT;
  WTile w;
  w.e = tile / per;
  const int r = tile - w.e * per;
  w.n = r / a.MT;
  w.m = r - w.n * a.MT;
  if (!a.seg) {
    w.rows = a.rows1;
    w.a_row = w.b_row = 0;
    return w;
  }
  w.rows = __ldg(a.seg + 3 + E + w.e);
  w.a_row = __ldg(a.seg + 3 + 3 * E + w.e);
  w.b_row = a.b_in_rows ? __ldg(a.seg + 3 + 2 * E + w.e) : w.a_row;
  return w;
}

__global__ void __launch_bounds__(W_THREADS, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                 const __grid_constant__ CUtensorMap map_b_shared,
                 const __grid_constant__ CUtensorMap map_out, const WgradArgs args) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ WState st;
  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
  const uint32_t ring = (ptx::smem_addr(dyn_smem) + 1023u) & ~1023u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < W_STAGES; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.empty[i]), 1);
    }
    for (int i = 0; i < W_ACC; ++i) {
      ptx::mbar_init(ptx::smem_addr(&st.acc_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&st.acc_empty[i]), W_EPI_THREADS);
    }
    ptx::mbar_init(ptx::smem_addr(&st.drain), 1);
    st.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&map_a);
    ptx::prefetch_tmap(&map_b);
    ptx::prefetch_tmap(&map_b_shared);
    ptx::prefetch_tmap(&map_out);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&st.tmem_base), W_TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = st.tmem_base;
  volatile int* abort_flag = &st.abort;
  pdl_wait();
  pdl_trigger();
  const int E = args.seg ? __ldg(args.seg) : 1;
  const int tiles = E * args.MT * args.NT;

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        const WTile w = wtile(args, E, tile);
        const CUtensorMap* bm = w.e >= args.n_routed ? &map_b_shared : &map_b;
        const int KB = (w.rows + WKB - 1) / WKB;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_phase(ptx::smem_addr(&st.empty[stage]), phase ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_addr(&st.full[stage]);
          const uint32_t a_dst = ring + stage * W_STAGE_BYTES;
          const uint32_t b_dst = a_dst + WA_BYTES;
          ptx::mbar_arrive_expect_tx(fb, W_STAGE_BYTES);
#pragma unroll
          for (int i = 0; i < 2; ++i)
            ptx::tma_load_2d(a_dst + i * BOX_BYTES, &map_a, fb, args.a_col0 + w.m * WM + 64 * i,
                             w.a_row + kb * WKB);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ptx::tma_load_2d(b_dst + q * BOX_BYTES, bm, fb, w.n * WN + 64 * q, w.b_row + kb * WKB);
          ++issued;
          if (++stage == W_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        const long long n = issued < W_STAGES ? issued : W_STAGES;
        for (long long i = 1; i <= n; ++i) {
          const long long q = issued - i;
          drain_wait(ptx::smem_addr(&st.full[q % W_STAGES]), (uint32_t)((q / W_STAGES) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------ MMA issuer (lane 0) and row masking --
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32_mn(WM, WN, true);
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      const WTile w = wtile(args, E, tile);
      const int KB = (w.rows + WKB - 1) / WKB;
      if (KB == 0) continue;  // no rows: the epilogue writes zeros
      bool got = true;
      if (lane == 0)
        got = wait_phase(ptx::smem_addr(&st.acc_empty[acc]), acc_phase ^ 1u, abort_flag,
                         args.status);
      if (!__shfl_sync(0xffffffffu, got, 0)) {
        ok = false;
        break;
      }
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * WN);
      for (int kb = 0; kb < KB; ++kb) {
        got = wait_phase(ptx::smem_addr(&st.full[stage]), phase, abort_flag, args.status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint32_t a_src = ring + stage * W_STAGE_BYTES;
        const int valid = w.rows - kb * WKB;
        if (valid < WKB) {
          // rows [valid, 64) of the block belong to the next segment (or lie
          // past the tensor): zero them in all six boxes
          const int lines = WKB - valid;
          for (int i = lane; i < 6 * lines * 8; i += 32) {
            const int box = i / (lines * 8), rem = i - box * lines * 8;
            const int line = valid + rem / 8, chunk = rem % 8;
            ptx::st_shared_zero16(a_src + box * BOX_BYTES + line * 128 + chunk * 16);
          }
          ptx::fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          ptx::tc_fence_after();
          const uint64_t adesc = ptx::sdesc_mn128(a_src, BOX_BYTES);
          const uint64_t bdesc = ptx::sdesc_mn128(a_src + WA_BYTES, BOX_BYTES);
#pragma unroll
          for (int k = 0; k < WKB / 16; ++k)  // K = 16 a step: +2048 bytes, +128 in the field
            ptx::mma_bf16(d_tmem, adesc + 128 * k, bdesc + 128 * k, IDESC, (kb | k) != 0);
          ptx::mma_commit(ptx::smem_addr(&st.empty[stage]));
        }
        __syncwarp();
        if (++stage == W_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) ptx::mma_commit(ptx::smem_addr(&st.acc_full[acc]));
      if (++acc == W_ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && lane == 0) {
      ptx::mma_commit(ptx::smem_addr(&st.drain));
      drain_wait(ptx::smem_addr(&st.drain), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int sub = warp & 3;          // TMEM lanes [32 sub, 32 sub + 32)
    const int half = (warp - 2) >> 2;  // columns [128 half, 128 half + 128)
    const uint32_t stg = ring + W_STAGES * W_STAGE_BYTES + (warp - 2) * STG_BYTES;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
      const WTile w = wtile(args, E, tile);
      const bool zero = w.rows == 0;  // no rows: a zero gradient, no MMA
      uint32_t tbase = 0;
      if (!zero) {
        const bool ok =
            wait_phase(ptx::smem_addr(&st.acc_full[acc]), acc_phase, abort_flag, args.status);
        if (!__all_sync(0xffffffffu, ok)) break;
        ptx::tc_fence_after();
        tbase = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * WN);
      }
#pragma unroll 1
      for (int c = 4 * half; c < 4 * half + 4; ++c) {
        uint32_t v[32];
        if (!zero) {
          ptx::tmem_ld32(tbase + c * 32, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        // the previous block's store has read the buffer
        const uint32_t buf = stg;
        if (lane == 0) ptx::bulk_wait_read<0>();
        __syncwarp();
        if (!zero) ptx::tmem_ld_wait();
        // row `lane` of the 32 x 32 block, 16-byte chunk q at q ^ (row % 8)
#pragma unroll
        for (int q = 0; q < 8; ++q)
          ptx::st_shared_v4(buf + lane * 128 + ((q ^ (lane & 7)) << 4), v[4 * q], v[4 * q + 1],
                            v[4 * q + 2], v[4 * q + 3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_3d(&map_out, buf, w.n * WN + c * 32, w.m * WM + sub * 32, w.e);
          ptx::bulk_commit();
        }
      }
      if (!zero) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_addr(&st.acc_empty[acc]));
        if (++acc == W_ACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
    }
    if (lane == 0) ptx::bulk_wait_all();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, W_TMEM_COLS);
  }
}

cudaError_t launch_wgrad(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b_sh,
                         const CUtensorMap& out, const WgradArgs& args, int E, int prof_id,
                         cudaStream_t s) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)W_DYN_SMEM);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const long long tiles = (long long)E * args.MT * args.NT;
  if (tiles == 0) return cudaSuccess;
  const int grid = (int)std::min<long long>(tiles, num_sms());
  ProfScope p(prof_id, s);
  return launch_pdl(wgrad_kernel, dim3(grid), dim3(W_THREADS), W_DYN_SMEM, s, 1, a, b, b_sh, out,
                    args);
}

}  // namespace

cudaError_t launch_bwd_wgrad(const moe_config& c, const int32_t* seg, const void* x_perm,
                             const void* x, const void* dab, const void* dO, const void* h,
                             float* dw_gate, float* dw_up, float* dw_down, long long xp_rows,
                             long long r_rows, int* status, cudaStream_t s) {
  const long long P = (long long)c.T * c.top_k;
  const long long R = P + (long long)c.n_shared * c.T;
  const int E = c.n_experts + c.n_shared;
  const long long rows = std::max(R, r_rows);
  CUtensorMap m_dab, m_do, m_h, m_xp, m_x, o_g, o_u, o_d;
  const bool ok = make_map_out3d(&o_g, dw_gate, E, c.d_ff, c.d_model) &&
                  make_map_out3d(&o_u, dw_up, E, c.d_ff, c.d_model) &&
                  make_map_out3d(&o_d, dw_down, E, c.d_model, c.d_ff) &&
                  make_map(&m_dab, dab, rows, 2LL * c.d_ff, 64) &&
                  make_map(&m_do, dO, rows, c.d_model, 64) &&
                  make_map(&m_h, h, rows, c.d_ff, 64) &&
                  make_map(&m_xp, x_perm, std::max(P, xp_rows), c.d_model, 64) &&
                  make_map(&m_x, c.n_shared > 0 ? x : x_perm, c.n_shared > 0 ? c.T : P,
                           c.d_model, 64);
  if (!ok) return cudaErrorInvalidValue;
  WgradArgs a{};
  a.seg = seg;
  a.status = status;
  a.n_routed = c.n_experts;
  // dW_g, dW_u [E][d_ff][d]: A = da or db columns, B = the expert's input rows
  a.M = c.d_ff;
  a.N = c.d_model;
  a.MT = ceil_div(c.d_ff, WM);
  a.NT = ceil_div(c.d_model, WN);
  a.b_in_rows = 1;
  a.a_col0 = 0;
  cudaError_t e = launch_wgrad(m_dab, m_xp, m_x, o_g, a, E, K_WGRAD, s);
  if (e != cudaSuccess) return e;
  a.a_col0 = c.d_ff;
  e = launch_wgrad(m_dab, m_xp, m_x, o_u, a, E, K_WGRAD, s);
  if (e != cudaSuccess) return e;
  // dW_d [E][d][d_ff]: A = dO, B = H (both in the output-row space)
  a.M = c.d_model;
  a.N = c.d_ff;
  a.MT = ceil_div(c.d_model, WM);
  a.NT = ceil_div(c.d_ff, WN);
  a.b_in_rows = 0;
  a.a_col0 = 0;
  return launch_wgrad(m_do, m_h, m_h, o_d, a, E, K_WGRAD, s);
}

cudaError_t launch_bwd_router_grads(const moe_config& c, const void* dr_bf, const void* drT_bf,
                                    int n_pad, int t_pad, const void* x, const void* w_router,
                                    float* dx, float* dw_router, int* status, cudaStream_t s) {
  CUtensorMap m_dr, m_drt, m_x, m_wr, o_dx, o_wr;
  const bool ok = make_map(&m_dr, dr_bf, std::max(c.T, 1), n_pad, 64) &&
                  make_map(&m_drt, drT_bf, n_pad, t_pad, 64) &&
                  make_map(&m_x, x, std::max(c.T, 1), c.d_model, 64) &&
                  make_map(&m_wr, w_router, c.n_experts, c.d_model, 64) &&
                  make_map_out3d(&o_dx, dx, 1, std::max(c.T, 1), c.d_model) &&
                  make_map_out3d(&o_wr, dw_router, 1, c.n_experts, c.d_model);
  if (!ok) return cudaErrorInvalidValue;
  WgradArgs a{};
  a.status = status;
  a.n_routed = 1;
  a.N = c.d_model;
  a.NT = ceil_div(c.d_model, WN);
  // dx = dr W_r: K = the N experts, A = dr^T [N][T], B = W_r [N][d]
  cudaError_t e = cudaSuccess;
  if (c.T > 0) {
    a.rows1 = c.n_experts;
    a.M = c.T;
    a.MT = ceil_div(c.T, WM);
    e = launch_wgrad(m_drt, m_wr, m_wr, o_dx, a, 1, K_BWD_ROUTER, s);
    if (e != cudaSuccess) return e;
  }
  // dW_r = dr^T x: K = the T tokens, A = dr [T][N], B = x [T][d]
  a.rows1 = c.T;
  a.M = c.n_experts;
  a.MT = ceil_div(c.n_experts, WM);
  return launch_wgrad(m_dr, m_x, m_x, o_wr, a, 1, K_BWD_ROUTER, s);
}

}  // namespace moe
