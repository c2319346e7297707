// Internal declarations shared by the CUDA translation units of libmoe.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// Limits of this build (checked on the host before any launch).
constexpr int kMaxExperts = 256;     // router keeps a [tokens x N] score tile in smem
constexpr int kMaxTopK = 8;
constexpr int kMaxShared = 4;

// Permutation chunk: pairs handled by one block (8 warps x 8 rounds x 32).
constexpr int kPermuteChunk = 2048;

// Grouped GEMM tiling (bf16, tcgen05). A tile is 128 rows of one expert
// segment times 128 SwiGLU columns (gate and up side by side in one
// 128x256 accumulator) or times 256 output columns of the down projection.
constexpr int kTileM = 128;
constexpr int kSwigluTileN = 128;
constexpr int kDownTileN = 256;

// Device status word codes (stored as the negative status values).
__host__ __device__ constexpr int status_timeout() { return MOE_ERR_TIMEOUT; }
__host__ __device__ constexpr int status_check() { return MOE_ERR_DEVICE_CHECK; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }
inline size_t elem_bytes(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }

// Segment table of the grouped GEMM, in device memory (int32 words):
//   [0] E = number of segments (N routed + n_shared)
//   [1] total M tiles
//   [2 .. 2+E]        mt_start[e]: first M tile of segment e (E+1 entries)
//   [3+E  .. 3+2E)    rows[e]
//   [3+2E .. 3+3E)    a_row0[e]: first input row (x_perm row, or 0 in x)
//   [3+3E .. 3+4E)    out_row0[e]: first output row in H / y_perm
inline size_t seg_table_words(int E) { return 3 + 4 * (size_t)E + 1; }

// ---- launchers (enqueue only; return cudaError_t of the launch) -----------
cudaError_t launch_router(const moe_config& c, const void* x, const void* w_router,
                          const float* logit_bias, const float* sel_bias,
                          const float* logits_in, float* logits_out,
                          int32_t* topk_idx, float* topk_w, int32_t* counts,
                          float* prob_sum, float* partials, int* status,
                          cudaStream_t s);
size_t router_partials_bytes(const moe_config& c);
// Tensor-core router (router_tc.cu): bf16, 32 < N <= 256, scores computed
// (not given). Its grid never exceeds router_partial_blocks(c).
bool router_tc_applies(const moe_config& c, const float* logits_in);
cudaError_t launch_router_tc(const moe_config& c, const void* x, const void* w_router,
                             const float* logit_bias, const float* sel_bias, float* logits_out,
                             int32_t* topk_idx, float* topk_w, int32_t* counts, float* prob_sum,
                             float* partials, int32_t* cpart, int* status, cudaStream_t s);
// Row-wise E4M3 quantization (fp8.cu): output row r of q/scale comes from
// source row r, or from token gather[r] / k; rows at or past *rows_dev are
// skipped; amax_in, when set, gives each row's max |v| (fp32 bits); clear,
// when set, zeroes clear[clear_base + i * clear_stride + r] for i < clear_n.
struct QuantArgs {
  const __nv_bfloat16* src;
  long long rows;
  int cols;                  // multiple of 8
  const int32_t* gather;
  int k;
  long long src_rows;
  const int32_t* rows_dev;
  const unsigned* amax_in;
  uint8_t* q;
  float* scale;
  unsigned* clear;
  long long clear_base, clear_stride;
  int clear_n;
  // NVFP4 only (nvfp4.cu): q holds packed E2M1 codes [rows][cols / 2] and
  // sf the E4M3 block scales [rows][ld_sf]; cols a multiple of 64.
  uint8_t* sf;
  int ld_sf;
};
cudaError_t launch_quantize_rows(const QuantArgs& a, cudaStream_t s);
// Row-wise NVFP4 quantization (nvfp4.cu): per row one fp32 scale
// amax / 2688, per 16 elements one E4M3 block scale, per element one E2M1
// code; other fields as launch_quantize_rows.
cudaError_t launch_quantize_rows_nvf4(const QuantArgs& a, cudaStream_t s);
// Bytes of one row of NVFP4 block scales: cols / 16, rounded up to 16.
inline int nvf4_sf_stride(int cols) { return (cols / 16 + 15) / 16 * 16; }

// An NVFP4 matrix: codes [rows][cols / 2], block scales [rows][stride] and
// fp32 row scales [rows].
struct Nvf4Matrix {
  const uint8_t* q;
  const uint8_t* sf;
  const float* scale;
};
// The grouped SwiGLU GEMMs with NVFP4 operands (1-CTA tiles; the segment
// table built with kTileM rows a tile; split-K partials for few tiles):
// gate/up from xp (routed rows) / xs (the shared experts' token rows)
// writes H in bf16 and each H row's max |H|; H is quantized into hq (its
// buffers written, so non-const); down reads hq.
cudaError_t launch_grouped_nvf4(const moe_config& c, Nvf4Matrix xp, Nvf4Matrix xs,
                                const int32_t* seg, const int32_t* sorted_pair,
                                const float* topk_w, Nvf4Matrix wg, Nvf4Matrix wu, Nvf4Matrix wd,
                                void* h, unsigned* h_amax, uint8_t* hq, uint8_t* h_sf,
                                float* h_scale, void* y_perm, float* partial, long long xp_rows,
                                long long xs_rows, long long h_rows, int* status, cudaStream_t s);

// The grouped SwiGLU GEMMs with E4M3 operands (CTA-pair, 1-CTA or swap-AB
// decode tiles, chosen as for bf16): gate/up from xq_perm / xq (shared experts)
// writes H in bf16 and each H row's max |H|; H is quantized into hq; down
// reads hq. Row scales as QuantArgs writes them; weight scales per output
// channel [E][rows of one expert's matrix]. The segment table must be built
// with seg_tile_m(c) rows a tile.
cudaError_t launch_grouped_e4m3(const moe_config& c, const uint8_t* xq_perm,
                                const float* xp_scale, const uint8_t* xq, const float* x_scale,
                                const int32_t* seg, const int32_t* sorted_pair,
                                const float* topk_w, const uint8_t* wg_q, const float* wg_s,
                                const uint8_t* wu_q, const float* wu_s, const uint8_t* wd_q,
                                const float* wd_s, void* h, unsigned* h_amax, uint8_t* hq,
                                float* h_scale, void* y_perm, float* partial, long long xp_rows,
                                long long h_rows, int* status, cudaStream_t s);
// Row-major uint8 matrix [rows][cols] read in boxes of box_rows rows x 128
// bytes with the 128-byte swizzle (the E4M3 operands).
// NVFP4 block scales [rows][stride] bytes, boxes of box_rows rows x 16 bytes.
bool make_map_sf(CUtensorMap* m, const void* base, long long rows, long long stride,
                 unsigned box_rows = 128u);
bool make_map_u8(CUtensorMap* m, const void* base, long long rows, long long cols,
                 unsigned box_rows = 128u);

// Zeroes the status word, the router's block counter and the decode kernel's
// grid-barrier counter (a kernel, so it keeps the chain of programmatic
// dependent launches).
cudaError_t launch_reset_status(int* status, cudaStream_t s);
// Blocks the router's per-block partials are sized for.
int router_partial_blocks(const moe_config& c);
// SMs of the current device.
int num_sms();

// With seg != null it also builds the grouped GEMM's segment table (tile
// height tile_m) from the offsets it computes; with x_perm == null it skips
// the row gather. `counts` (pairs per expert,
// as the router left them) may be null; when given, mid-sized batches take
// their offsets from it instead of counting the pairs again.
cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* topk_idx,
                           const int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                           int32_t* inv_pos, void* x_perm, int32_t* chunk_hist, int* status,
                           int32_t* seg, int tile_m, cudaStream_t s);
size_t permute_scratch_bytes(const moe_config& c);

cudaError_t launch_seg_table(const moe_config& c, const int32_t* offsets, int32_t* seg,
                             int tile_m, int* status, cudaStream_t s);

// Capacity overflow rerouted in rounds (reroute.cu): assign[p] is the
// expert pair p runs on, -1 if dropped; *rounds (may be null) the rounds
// after the capacity cut. One cooperative launch; status[2] must be zero at
// launch (launch_reset_status). scratch: reroute_scratch_bytes(c) bytes,
// 256-byte aligned; the optional outputs give its parts' sizes.
size_t reroute_scratch_bytes(const moe_config& c, size_t* held = nullptr,
                             size_t* per_pair = nullptr, size_t* pub = nullptr);
cudaError_t launch_reroute(const moe_config& c, const float* logits, const float* sel_bias,
                           const int32_t* topk_idx, int32_t* assign, int32_t* rounds,
                           void* scratch, int* status, cudaStream_t s);
// Decode-sized layers (bf16, T <= 64, N <= 32, no reroute): routing,
// permutation with the capacity cut, segment table (tile height tile_m) and
// row gather (skipped when x_perm is null) in one single-block launch
// (router.cu). It also clears status[0..2], so no reset launch precedes it.
bool decode_front_applies(const moe_config& c);
cudaError_t launch_decode_front(const moe_config& c, const void* x, const void* w_router,
                                const float* logit_bias, const float* sel_bias, int32_t* topk_idx,
                                float* topk_w, int32_t* counts, float* prob_sum, int32_t* offsets,
                                int32_t* sorted_pair, int32_t* inv_pos, void* x_perm, int32_t* seg,
                                int tile_m, int* status, cudaStream_t s);
// Whether a layer reroutes its capacity overflow (cfg.overflow with a cap).
inline bool reroutes(const moe_config& c) {
  return c.overflow == MOE_OVERFLOW_REROUTE && c.capacity > 0;
}
// Tiling of the bf16 and E4M3 grouped GEMMs (a MOE_TILES_* value other than
// AUTO): cfg.tiles when it names one that can run, else the library's choice
// (grouped_sm103.cu). Both CTA-pair tilings cut segments into tiles of at
// most 256 rows, so the segment table must then be built with that height.
int gemm_tiles(const moe_config& c);
// Whether moe_layer_forward fuses the row gather into the gate/up GEMM
// (bf16, weight-stationary pairs; cfg.gather or the library's choice).
bool gather_fused(const moe_config& c);
bool use_pair_tiles(const moe_config& c);
int seg_tile_m(const moe_config& c);

// bf16 tcgen05 path: gate/up (SwiGLU epilogue into h) then down (gate
// weight epilogue into y_perm). When a GEMM has fewer tiles than two waves
// of the grid (small batches), each tile may be split along K; the splits
// write fp32 partial rows into `partial` and a reduce kernel sums them in
// split order and applies the epilogue.
constexpr size_t kSplitKBudget = 64ull << 20;  // bytes of partial rows at most
constexpr int kMaxSplitK = 16;
struct SplitKPlan {
  int s_max_gu, s_max_dn;  // largest split factor per GEMM (1: never split)
  size_t partial_bytes;    // fp32 partial rows buffer
};
SplitKPlan splitk_plan(const moe_config& c);
// With y and inv_pos given (the layer forward), a down projection that may
// be split along K is reduced straight into y (the combine fused with the
// split-K reduction); *combined then says the combine is done.
cudaError_t launch_grouped_bf16(const moe_config& c, const void* x_perm, const void* x,
                                const int32_t* seg, const int32_t* sorted_pair,
                                const float* topk_w, const void* w_gate, const void* w_up,
                                const void* w_down, void* h, void* y_perm, float* partial,
                                long long xp_rows, long long h_rows, int* status,
                                cudaStream_t s, const int32_t* inv_pos = nullptr,
                                void* y = nullptr, bool* combined = nullptr);
// Rows allocated for library-owned x_perm / H: at least one 128-row tile, so
// that a small batch's tiles read allocated (masked) rows rather than the
// tensor map's out-of-bounds fill.
inline long long padded_rows(long long rows) { return rows < kTileM ? kTileM : rows; }
// fp32 CUDA-core path.
cudaError_t launch_grouped_f32(const moe_config& c, const void* x_perm, const void* x,
                               const int32_t* seg, const int32_t* sorted_pair,
                               const float* topk_w, const void* w_gate, const void* w_up,
                               const void* w_down, void* h, void* y_perm, int* status,
                               cudaStream_t s);

cudaError_t launch_combine(const moe_config& c, const void* y_perm, const int32_t* inv_pos,
                           const float* topk_w, void* y, cudaStream_t s);

cudaError_t launch_balance_stats(int N, int T, int k, const int32_t* counts,
                                 const float* prob_sum, float alpha, float* f, float* P,
                                 float* aux, cudaStream_t s);

// 2-D TMA tensor map of a row-major bf16 matrix [rows][cols], boxes of
// box_rows x 64 columns with the 128-byte swizzle (tma_maps.cu).
bool make_map(CUtensorMap* m, const void* base, long long rows, long long cols,
              unsigned box_rows = 128u);
// 3-D TMA map of an fp32 output [E][M][N] stored in 32 x 32 boxes.
bool make_map_out3d(CUtensorMap* m, void* base, long long E, long long M, long long N);

// ---- decode-sized layers in one kernel (decode_fused.cu) -------------------
constexpr int kDecodeFusedMaxT = 1;
// bf16, 1 <= T <= kDecodeFusedMaxT, N <= 32, d_model a multiple of 256,
// d_ff of 256, x of all tokens (fp32) within the kernel's shared memory.
bool decode_fused_applies(const moe_config& c);
// Its workspace: the gate/up pre-activation halves and the down
// projection's partial sums (0 when it does not apply).
size_t decode_fused_ws_bytes(const moe_config& c);
// The whole layer forward (routing, both projections, the gated sum) as one
// cooperative launch; ws: decode_fused_ws_bytes(c) bytes, 256-byte aligned;
// status[2] must be zero at launch (launch_reset_status).
cudaError_t launch_decode_fused(const moe_config& c, const void* x, const void* w_router,
                                const float* logit_bias, const float* sel_bias,
                                const void* w_gate, const void* w_up, const void* w_down,
                                void* y, int32_t* topk_idx, float* topk_w, int32_t* counts,
                                float* prob_sum, void* ws, int* status, cudaStream_t s);

// ---- backward (bwd.cu, wgrad_sm103.cu, grouped_sm103.cu) -------------------
// dL/dg of every pair (0 for a dropped one) and dO = g * dy per expert row
// (dy for shared-expert rows), from the unweighted expert outputs o.
cudaError_t launch_bwd_gate(const moe_config& c, const void* dy, const void* o,
                            const int32_t* inv_pos, const float* topk_w, float* dg, void* dO,
                            cudaStream_t s);
// dL/dr: softmax backward of the gates plus the balance term, in bf16 as
// dr [T][n_pad] and its transpose drT [n_pad][t_pad] (the operands of the
// two router gradient products; n_pad, t_pad multiples of 8).
cudaError_t launch_bwd_score(const moe_config& c, const float* logits, const int32_t* topk_idx,
                             const float* topk_w, const float* dg, const int32_t* counts,
                             float alpha, float aux_grad, void* dr_bf, void* drT_bf, int n_pad,
                             int t_pad, cudaStream_t s);
// dx [T][d] fp32 += the token's dA rows (kept slots, then shared experts).
cudaError_t launch_bwd_dx(const moe_config& c, const void* dA, const int32_t* inv_pos, float* dx,
                          cudaStream_t s);
// dx = dr W_r and dW_r = dr^T x on the tensor cores (wgrad kernel, one segment).
cudaError_t launch_bwd_router_grads(const moe_config& c, const void* dr_bf, const void* drT_bf,
                                    int n_pad, int t_pad, const void* x, const void* w_router,
                                    float* dx, float* dw_router, int* status, cudaStream_t s);
// Forward recompute for the backward (1-CTA tiles; seg built with kTileM):
// h, the pre-activations ab = a | b [rows][2 d_ff], and the unweighted
// expert outputs o [rows][d], all bf16.
cudaError_t launch_bwd_recompute(const moe_config& c, const void* x_perm, const void* x,
                                 const int32_t* seg, const void* w_gate, const void* w_up,
                                 const void* w_down, void* h, void* ab, void* o, long long xp_rows,
                                 long long r_rows, int* status, cudaStream_t s);
// Activation gradients through the experts: dab = da | db [rows][2 d_ff]
// from dO and ab, then dA [rows][d] = dab [W_g ; W_u]. d_ff % 64 == 0.
cudaError_t launch_bwd_dgrad(const moe_config& c, const int32_t* seg, const void* dO,
                             const void* ab, const void* w_gate, const void* w_up,
                             const void* w_down, void* dab, void* dA, long long r_rows,
                             int* status, cudaStream_t s);
// Weight gradients (fp32): dW_g[e] = da_e^T A_e, dW_u[e] = db_e^T A_e,
// dW_d[e] = dO_e^T h_e, A = x_perm rows (x for shared experts).
cudaError_t launch_bwd_wgrad(const moe_config& c, const int32_t* seg, const void* x_perm,
                             const void* x, const void* dab, const void* dO, const void* h,
                             float* dw_gate, float* dw_up, float* dw_down, long long xp_rows,
                             long long r_rows, int* status, cudaStream_t s);

// ---- profiling hooks (abi.cu) ----------------------------------------------
enum KernelId {
  K_RESET = 0,
  K_ROUTER,
  K_PERMUTE_HIST,
  K_PERMUTE_SCAN,
  K_PERMUTE_RANK,
  K_PERMUTE_GATHER,
  K_PERMUTE_SMALL,
  K_PERMUTE_GROUP,
  K_SEG_TABLE,
  K_GATE_UP,
  K_DOWN,
  K_SPLITK_REDUCE,
  K_COMBINE,
  K_BALANCE,
  K_QUANTIZE,
  K_BWD_GATE,
  K_BWD_SCORE,
  K_BWD_DH,
  K_BWD_DA,
  K_BWD_DX,
  K_BWD_ROUTER,
  K_WGRAD,
  K_DECODE_FUSED,
  K_REROUTE,
  K_DECODE_FRONT,
  K_NUM
};
void prof_begin(int id, cudaStream_t s);
void prof_end(int id, cudaStream_t s);
void count_launch();

// Launch with programmatic stream serialization (see pdl_wait() in
// device_util.cuh); an optional cluster width for CTA-pair kernels.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct ProfScope {
  int id;
  cudaStream_t s;
  ProfScope(int i, cudaStream_t st) : id(i), s(st) { prof_begin(id, s); }
  ~ProfScope() { prof_end(id, s); count_launch(); }
};

}  // namespace moe
