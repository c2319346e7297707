// The C ABI of libmoe.so (include/moe.h): argument checks, workspace
// layout, the call sequence of the layer, device status, and the optional
// per-kernel event profiler. Every computation runs in the kernels of the
// other translation units; nothing here touches tensor data on the host.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "device_util.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<uint64_t> g_launches{0};

int fail_cuda(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return MOE_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Carves 256-byte-aligned regions out of a workspace; with base == nullptr
// it only measures.
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t bytes) {
    off = align_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += bytes;
    return p;
  }
};

long long pairs(const moe_config& c) { return (long long)c.T * c.top_k; }
long long rows_total(const moe_config& c) { return pairs(c) + (long long)c.n_shared * c.T; }

struct RouterWs {
  int* status;
  float* partials;
};
RouterWs carve_router(Carver& cv, const moe_config& c) {
  RouterWs w;
  w.status = cv.take<int>(256);
  w.partials = cv.take<float>(router_partials_bytes(c));
  return w;
}
struct PermuteWs {
  int* status;
  int32_t* hist;
};
PermuteWs carve_permute(Carver& cv, const moe_config& c) {
  PermuteWs w;
  w.status = cv.take<int>(256);
  w.hist = cv.take<int32_t>(permute_scratch_bytes(c));
  return w;
}
struct GroupedWs {
  int* status;
  int32_t* seg;
  void* h;
  float* partial;
};
GroupedWs carve_grouped(Carver& cv, const moe_config& c) {
  GroupedWs w;
  const SplitKPlan plan = splitk_plan(c);
  w.status = cv.take<int>(256);
  w.seg = cv.take<int32_t>(sizeof(int32_t) * seg_table_words(c.n_experts + c.n_shared));
  w.h = cv.take<void>((size_t)padded_rows(rows_total(c)) * c.d_ff * elem_bytes(c.dtype));
  w.partial = cv.take<float>(plan.partial_bytes);
  return w;
}
struct LayerWs {
  int* status;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  float* prob_sum;
  int32_t* offsets;
  int32_t* sorted_pair;
  int32_t* inv_pos;
  void* x_perm;
  void* y_perm;
  float* partials;
  int32_t* hist;
  int32_t* seg;
  void* h;
  float* partial;
  float* dpart;  // the one-kernel decode path's workspace
  // capacity rerouting only (empty otherwise): the router's scores, the
  // pairs' experts after the reroute, and the reroute kernel's scratch
  float* logits;
  int32_t* assign;
  void* rr;
};
LayerWs carve_layer(Carver& cv, const moe_config& c) {
  LayerWs w;
  const size_t P = (size_t)pairs(c), N = (size_t)c.n_experts, eb = elem_bytes(c.dtype);
  w.status = cv.take<int>(256);
  w.topk_idx = cv.take<int32_t>(sizeof(int32_t) * P);
  w.topk_w = cv.take<float>(sizeof(float) * P);
  w.counts = cv.take<int32_t>(sizeof(int32_t) * N);
  w.prob_sum = cv.take<float>(sizeof(float) * N);
  w.offsets = cv.take<int32_t>(sizeof(int32_t) * (N + 1));
  w.sorted_pair = cv.take<int32_t>(sizeof(int32_t) * P);
  w.inv_pos = cv.take<int32_t>(sizeof(int32_t) * P);
  w.x_perm = cv.take<void>((size_t)padded_rows((long long)P) * c.d_model * eb);
  w.y_perm = cv.take<void>((size_t)rows_total(c) * c.d_model * eb);
  w.partials = cv.take<float>(router_partials_bytes(c));
  w.hist = cv.take<int32_t>(permute_scratch_bytes(c));
  w.seg = cv.take<int32_t>(sizeof(int32_t) * seg_table_words(c.n_experts + c.n_shared));
  w.h = cv.take<void>((size_t)padded_rows(rows_total(c)) * c.d_ff * eb);
  const SplitKPlan plan = splitk_plan(c);
  w.partial = cv.take<float>(plan.partial_bytes);
  w.dpart = cv.take<float>(decode_fused_ws_bytes(c));
  // null unless the layer reroutes: the router then writes no scores
  const bool rr = reroutes(c);
  w.logits = rr ? cv.take<float>(sizeof(float) * (size_t)c.T * N) : nullptr;
  w.assign = rr ? cv.take<int32_t>(sizeof(int32_t) * P) : nullptr;
  w.rr = rr ? cv.take<void>(reroute_scratch_bytes(c)) : nullptr;
  return w;
}

// Capacity rerouting without a layer around it.
struct RerouteWs {
  int* status;
  void* rr;
};
RerouteWs carve_reroute(Carver& cv, const moe_config& c) {
  RerouteWs w;
  w.status = cv.take<int>(256);
  w.rr = cv.take<void>(reroute_scratch_bytes(c));
  return w;
}

// The pairs' experts the permutation groups: the router's choice, or with
// rerouting on, the reroute kernel's assignment (launched here). Then the
// cut is already applied and the router's counts no longer hold, so the
// permutation runs without a cap (*pc) and counts its own pairs.
struct PermuteIn {
  const int32_t* idx;
  const int32_t* counts;
  moe_config pc;
};
cudaError_t overflow_stage(const moe_config& c, const float* sel_bias, const int32_t* idx,
                           const int32_t* counts, const float* logits, int32_t* assign, void* rr,
                           int* status, cudaStream_t s, PermuteIn* out) {
  out->idx = idx;
  out->counts = counts;
  out->pc = c;
  if (!reroutes(c) || c.T == 0) return cudaSuccess;
  out->idx = assign;
  out->counts = nullptr;
  out->pc.capacity = 0;
  return launch_reroute(c, logits, sel_bias, idx, assign, nullptr, rr, status, s);
}

// The quantized layers' routing and permutation (no row gather: their
// quantizers gather the rows): the single-block decode launch, or the status
// reset, the router, the overflow stage and the permutation. *rc gets a
// host-side status; the return value is the CUDA error.
cudaError_t route_and_permute(const moe_config& c, const void* x, const void* w_router,
                              const float* logit_bias, const float* sel_bias, int32_t* idx,
                              float* tw, int32_t* cnt, float* ps, const LayerWs& w, int tile_m,
                              cudaStream_t s, int* rc) {
  *rc = MOE_OK;
  if (decode_front_applies(c))
    return launch_decode_front(c, x, w_router, logit_bias, sel_bias, idx, tw, cnt, ps, w.offsets,
                               w.sorted_pair, w.inv_pos, nullptr, w.seg, tile_m, w.status, s);
  cudaError_t e = launch_reset_status(w.status, s);
  if (e != cudaSuccess) return e;
  e = launch_router(c, x, w_router, logit_bias, sel_bias, nullptr, w.logits, idx, tw, cnt, ps,
                    w.partials, w.status, s);
  if (e != cudaSuccess || c.T == 0) return e;
  PermuteIn pin;
  if ((e = overflow_stage(c, sel_bias, idx, cnt, w.logits, w.assign, w.rr, w.status, s, &pin)) !=
      cudaSuccess)
    return e;
  return launch_permute(pin.pc, x, pin.idx, pin.counts, w.offsets, w.sorted_pair, w.inv_pos,
                        nullptr, w.hist, w.status, w.seg, tile_m, s);
}

// The FP8 layer: the bf16 layer's routing and output buffers, E4M3 copies
// of the routed rows and of x (shared experts), H in bf16 with its rows' max
// |H|, and H in E4M3, each with fp32 row scales.
struct LayerFp8Ws {
  LayerWs base;  // x_perm unused
  uint8_t* xq_perm;
  float* xp_scale;
  uint8_t* xq;
  float* x_scale;
  unsigned* h_amax;
  uint8_t* hq;
  float* h_scale;
};
LayerFp8Ws carve_layer_fp8(Carver& cv, const moe_config& c) {
  LayerFp8Ws w;
  moe_config b = c;
  b.dtype = MOE_BF16;
  w.base = carve_layer(cv, b);
  const size_t P = (size_t)pairs(c), R = (size_t)rows_total(c);
  w.xq_perm = cv.take<uint8_t>((size_t)padded_rows((long long)P) * c.d_model);
  w.xp_scale = cv.take<float>(sizeof(float) * P);
  w.xq = cv.take<uint8_t>((size_t)padded_rows(c.T) * c.d_model);
  w.x_scale = cv.take<float>(sizeof(float) * (size_t)c.T);
  w.h_amax = cv.take<unsigned>(sizeof(unsigned) * R);
  w.hq = cv.take<uint8_t>((size_t)padded_rows((long long)R) * c.d_ff);
  w.h_scale = cv.take<float>(sizeof(float) * R);
  return w;
}

// The NVFP4 layer: the bf16 layer's routing and output buffers, NVFP4 copies
// (codes, block scales, row scales) of the routed rows and of x (shared
// experts), H in bf16 with its rows' max |H|, and H in NVFP4.
struct LayerNvf4Ws {
  LayerWs base;  // x_perm unused
  uint8_t *xq_perm, *xp_sf;
  float* xp_scale;
  uint8_t *xq, *x_sf;
  float* x_scale;
  unsigned* h_amax;
  uint8_t *hq, *h_sf;
  float* h_scale;
};
LayerNvf4Ws carve_layer_nvf4(Carver& cv, const moe_config& c) {
  LayerNvf4Ws w;
  moe_config b = c;
  b.dtype = MOE_BF16;
  w.base = carve_layer(cv, b);
  const size_t P = (size_t)pairs(c), R = (size_t)rows_total(c);
  const size_t Pp = (size_t)padded_rows((long long)P), Tp = (size_t)padded_rows(c.T),
               Rp = (size_t)padded_rows((long long)R);
  const size_t sfd = (size_t)nvf4_sf_stride(c.d_model), sff = (size_t)nvf4_sf_stride(c.d_ff);
  w.xq_perm = cv.take<uint8_t>(Pp * c.d_model / 2);
  w.xp_sf = cv.take<uint8_t>(Pp * sfd);
  w.xp_scale = cv.take<float>(sizeof(float) * P);
  w.xq = cv.take<uint8_t>(Tp * c.d_model / 2);
  w.x_sf = cv.take<uint8_t>(Tp * sfd);
  w.x_scale = cv.take<float>(sizeof(float) * (size_t)c.T);
  w.h_amax = cv.take<unsigned>(sizeof(unsigned) * R);
  w.hq = cv.take<uint8_t>(Rp * c.d_ff / 2);
  w.h_sf = cv.take<uint8_t>(Rp * sff);
  w.h_scale = cv.take<float>(sizeof(float) * R);
  return w;
}

int check_ws(const moe_config& c, void* ws, size_t ws_bytes, size_t need) {
  (void)c;
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return MOE_ERR_MISALIGNED;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// All non-null device pointers 16-byte aligned.
bool all_aligned(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p && !aligned(p, 16)) return false;
  return true;
}

int reset_status(int* status, cudaStream_t s) {
  cudaError_t e = launch_reset_status(status, s);
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

// The bf16 path is built for sm_103a only.
int check_device(const moe_config& c) {
  if (c.dtype != MOE_BF16) return MOE_OK;
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return fail_cuda(e);
  return (major == 10 && minor == 3) ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

int seg_tile(const moe_config& c) { return c.dtype == MOE_BF16 ? seg_tile_m(c) : kTileM; }

// seg_ready: the segment table was already built (by the permutation).
int grouped_impl(const moe_config& c, const void* x_perm, long long xp_rows, const void* x,
                 const int32_t* offsets, const int32_t* sorted_pair, const float* topk_w,
                 const void* wg, const void* wu, const void* wd, void* y_perm, int32_t* seg,
                 bool seg_ready, void* h, float* partial, int* status, cudaStream_t s,
                 const int32_t* inv_pos = nullptr, void* y = nullptr, bool* combined = nullptr) {
  if (rows_total(c) == 0) return MOE_OK;
  cudaError_t e = cudaSuccess;
  if (!seg_ready) {
    e = launch_seg_table(c, offsets, seg, seg_tile(c), status, s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  e = (c.dtype == MOE_BF16)
          ? launch_grouped_bf16(c, x_perm, x, seg, sorted_pair, topk_w, wg, wu, wd, h, y_perm, partial,
                                xp_rows, padded_rows(rows_total(c)), status, s, inv_pos, y,
                                combined)
          : launch_grouped_f32(c, x_perm, x, seg, sorted_pair, topk_w, wg, wu, wd, h, y_perm, status, s);
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

// ---- profiler ---------------------------------------------------------------
const char* kKernelNames[K_NUM] = {"reset_status",  "router_topk",    "permute_hist",
                                   "permute_scan",  "permute_rank",   "permute_gather",
                                   "permute_small", "permute_group",  "seg_table",
                                   "gate_up",       "down",           "splitk_reduce",
                                   "combine",       "balance_stats",  "quantize",
                                   "bwd_gate",      "bwd_score",      "bwd_dh_swiglu",
                                   "bwd_da",        "bwd_dx",         "bwd_router",
                                   "bwd_wgrad",     "decode_fused",   "reroute",
                                   "decode_front"};
struct Prof {
  std::mutex mu;
  uint32_t mask = 0;
  std::vector<cudaEvent_t> pool;
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> done;
  cudaEvent_t open[K_NUM] = {};
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};
Prof& prof() {
  static Prof* p = new Prof();  // never destroyed: events may outlive static teardown order
  return *p;
}

}  // namespace

// Zeroes the workspace header words, [0] device status and [1] the router's
// finished-block counter, after the previous grid on the stream has
// finished (so a late error of the previous call is not wiped out). A
// kernel rather than a memset: it stays in the chain of programmatic
// dependent launches, where a memset node breaks it.
namespace {
__global__ void reset_status_kernel(int* status) {
  pdl_wait();
  if (threadIdx.x < 3) status[threadIdx.x] = 0;
  __syncwarp();
  pdl_trigger();
}
}  // namespace

cudaError_t launch_reset_status(int* status, cudaStream_t s) {
  ProfScope p(K_RESET, s);
  return launch_pdl(reset_status_kernel, dim3(1), dim3(32), 0, s, 1, status);
}


void prof_begin(int id, cudaStream_t s) {
  Prof& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  if (!((p.mask >> id) & 1u)) return;
  cudaEvent_t e = p.get();
  cudaEventRecord(e, s);
  p.open[id] = e;
}
void prof_end(int id, cudaStream_t s) {
  Prof& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  if (!((p.mask >> id) & 1u) || !p.open[id]) return;
  cudaEvent_t e = p.get();
  cudaEventRecord(e, s);
  p.done.push_back({id, {p.open[id], e}});
  p.open[id] = nullptr;
}
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return 100; }

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, bad shape or bad enum)";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error (see moe_last_cuda_error)";
    case MOE_ERR_TIMEOUT: return "a bounded device wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side input check failed";
    default: return "unknown status";
  }
}

int moe_last_cuda_error(void) { return g_last_cuda_error; }

int moe_check_config(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d_model < 1 || c->n_experts < 1 || c->top_k < 1 || c->n_shared < 0 ||
      c->d_ff < 1)
    return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->gate_mode != MOE_GATE_TOPK_SOFTMAX && c->gate_mode != MOE_GATE_ALL_SOFTMAX_RENORM)
    return MOE_ERR_INVALID_ARG;
  if (c->top_k > c->n_experts || c->capacity < 0) return MOE_ERR_INVALID_ARG;
  if (c->tiles < MOE_TILES_AUTO || c->tiles > MOE_TILES_WEIGHT_PAIR) return MOE_ERR_INVALID_ARG;
  if (c->gather < MOE_GATHER_AUTO || c->gather > MOE_GATHER_FUSED) return MOE_ERR_INVALID_ARG;
  if (c->overflow != MOE_OVERFLOW_DROP && c->overflow != MOE_OVERFLOW_REROUTE)
    return MOE_ERR_INVALID_ARG;
  if (c->n_experts > kMaxExperts || c->top_k > kMaxTopK || c->n_shared > kMaxShared)
    return MOE_ERR_UNSUPPORTED;
  if (c->d_model % 8 != 0 || c->d_ff % 8 != 0) return MOE_ERR_UNSUPPORTED;
  // Row indices, TMA coordinates and pair ids are 32-bit.
  const long long R = (long long)c->T * (c->top_k + c->n_shared);
  if (R >= (1LL << 30) || (long long)(c->n_experts + c->n_shared) * (c->d_ff > c->d_model ? c->d_ff : c->d_model) >= (1LL << 31))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

size_t moe_router_workspace_size(const moe_config* c) {
  if (moe_check_config(c) != MOE_OK) return 0;
  Carver cv(nullptr);
  carve_router(cv, *c);
  return align_up(cv.off, 256);
}
size_t moe_permute_workspace_size(const moe_config* c) {
  if (moe_check_config(c) != MOE_OK) return 0;
  Carver cv(nullptr);
  carve_permute(cv, *c);
  return align_up(cv.off, 256);
}
size_t moe_grouped_workspace_size(const moe_config* c) {
  if (moe_check_config(c) != MOE_OK) return 0;
  Carver cv(nullptr);
  carve_grouped(cv, *c);
  return align_up(cv.off, 256);
}
size_t moe_workspace_size(const moe_config* c) {
  if (moe_check_config(c) != MOE_OK) return 0;
  Carver cv(nullptr);
  carve_layer(cv, *c);
  return align_up(cv.off, 256);
}

int moe_router_topk(const moe_config* cfg, const void* x, const void* w_router,
                    const float* logit_bias, const float* sel_bias, const float* logits_in,
                    float* logits_out, int32_t* topk_idx, float* topk_w, int32_t* counts,
                    float* prob_sum, void* ws, size_t ws_bytes, moe_stream_t stream) {
  int rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe_config& c = *cfg;
  if (!counts || !prob_sum) return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && (!topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && !logits_in && (!x || !w_router)) return MOE_ERR_INVALID_ARG;
  if (logits_in && logit_bias) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({x, w_router, logit_bias, sel_bias, logits_in, logits_out, topk_idx, topk_w,
                    counts, prob_sum}))
    return MOE_ERR_MISALIGNED;
  if ((rc = check_ws(c, ws, ws_bytes, moe_router_workspace_size(cfg))) != MOE_OK) return rc;
  Carver cv(ws);
  RouterWs w = carve_router(cv, c);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = reset_status(w.status, s)) != MOE_OK) return rc;
  cudaError_t e = launch_router(c, x, w_router, logit_bias, sel_bias, logits_in, logits_out,
                                topk_idx, topk_w, counts, prob_sum, w.partials, w.status, s);
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

int moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                int32_t* expert_offsets, int32_t* sorted_pair, int32_t* inv_pos, void* x_perm,
                void* ws, size_t ws_bytes, moe_stream_t stream) {
  int rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe_config& c = *cfg;
  if (!expert_offsets) return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && (!x || !topk_idx || !sorted_pair || !inv_pos || !x_perm))
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned({x, topk_idx, expert_offsets, sorted_pair, inv_pos, x_perm}))
    return MOE_ERR_MISALIGNED;
  if ((rc = check_ws(c, ws, ws_bytes, moe_permute_workspace_size(cfg))) != MOE_OK) return rc;
  Carver cv(ws);
  PermuteWs w = carve_permute(cv, c);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = reset_status(w.status, s)) != MOE_OK) return rc;
  cudaError_t e = launch_permute(c, x, topk_idx, nullptr, expert_offsets, sorted_pair, inv_pos,
                                 x_perm, w.hist, w.status, nullptr, 0, s);
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

int moe_grouped_swiglu(const moe_config* cfg, const void* x_perm, const void* x,
                       const int32_t* expert_offsets, const int32_t* sorted_pair,
                       const float* topk_w, const void* w_gate, const void* w_up,
                       const void* w_down, void* y_perm, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  int rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe_config& c = *cfg;
  if (rows_total(c) > 0) {
    if (!expert_offsets || !w_gate || !w_up || !w_down || !y_perm) return MOE_ERR_INVALID_ARG;
    if (pairs(c) > 0 && !x_perm) return MOE_ERR_INVALID_ARG;
    if (c.n_shared > 0 && !x) return MOE_ERR_INVALID_ARG;
    if (topk_w && !sorted_pair) return MOE_ERR_INVALID_ARG;
  }
  if (!all_aligned({x_perm, x, expert_offsets, sorted_pair, topk_w, w_gate, w_up, w_down, y_perm}))
    return MOE_ERR_MISALIGNED;
  if ((rc = check_ws(c, ws, ws_bytes, moe_grouped_workspace_size(cfg))) != MOE_OK) return rc;
  if ((rc = check_device(c)) != MOE_OK) return rc;
  Carver cv(ws);
  GroupedWs w = carve_grouped(cv, c);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = reset_status(w.status, s)) != MOE_OK) return rc;
  return grouped_impl(c, x_perm, pairs(c), x, expert_offsets, sorted_pair, topk_w, w_gate, w_up,
                      w_down, y_perm, w.seg, false, w.h, w.partial, w.status, s);
}

int moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* inv_pos,
                const float* topk_w, void* y, moe_stream_t stream) {
  int rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe_config& c = *cfg;
  if (c.T > 0 && (!y_perm || !inv_pos || !y)) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({y_perm, inv_pos, topk_w, y})) return MOE_ERR_MISALIGNED;
  cudaError_t e = launch_combine(c, y_perm, inv_pos, topk_w, y, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

size_t moe_reroute_workspace_size(const moe_config* c) {
  if (moe_check_config(c) != MOE_OK) return 0;
  Carver cv(nullptr);
  carve_reroute(cv, *c);
  return align_up(cv.off, 256);
}

int moe_reroute(const moe_config* cfg, const float* logits, const float* sel_bias,
                const int32_t* topk_idx, int32_t* assign, int32_t* rounds, void* ws,
                size_t ws_bytes, moe_stream_t stream) {
  int rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe_config& c = *cfg;
  if (c.T > 0 && (!logits || !topk_idx || !assign)) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({logits, sel_bias, topk_idx, assign, rounds})) return MOE_ERR_MISALIGNED;
  if ((rc = check_ws(c, ws, ws_bytes, moe_reroute_workspace_size(cfg))) != MOE_OK) return rc;
  Carver cv(ws);
  RerouteWs w = carve_reroute(cv, c);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = reset_status(w.status, s)) != MOE_OK) return rc;
  cudaError_t e = launch_reroute(c, logits, sel_bias, topk_idx, assign, rounds, w.rr, w.status, s);
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

int moe_layer_forward(const moe_config* cfg, const void* x, const void* w_router,
                      const float* logit_bias, const float* sel_bias, const void* w_gate,
                      const void* w_up, const void* w_down, void* y, int32_t* topk_idx,
                      float* topk_w, int32_t* counts, float* prob_sum, void* ws, size_t ws_bytes,
                      moe_stream_t stream) {
  int rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe_config& c = *cfg;
  if (c.T > 0 && (!x || !w_router || !w_gate || !w_up || !w_down || !y)) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({x, w_router, logit_bias, sel_bias, w_gate, w_up, w_down, y, topk_idx, topk_w,
                    counts, prob_sum}))
    return MOE_ERR_MISALIGNED;
  if ((rc = check_ws(c, ws, ws_bytes, moe_workspace_size(cfg))) != MOE_OK) return rc;
  if ((rc = check_device(c)) != MOE_OK) return rc;
  Carver cv(ws);
  LayerWs w = carve_layer(cv, c);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* idx = topk_idx ? topk_idx : w.topk_idx;
  float* tw = topk_w ? topk_w : w.topk_w;
  int32_t* cnt = counts ? counts : w.counts;
  float* ps = prob_sum ? prob_sum : w.prob_sum;
  if (decode_fused_applies(c) && !reroutes(c)) {
    // a single token: the whole layer in one kernel
    if ((rc = reset_status(w.status, s)) != MOE_OK) return rc;
    cudaError_t e = launch_decode_fused(c, x, w_router, logit_bias, sel_bias, w_gate, w_up, w_down,
                                        y, idx, tw, cnt, ps, w.dpart, w.status, s);
    return e == cudaSuccess ? MOE_OK : fail_cuda(e);
  }
  // with the gather fused into the gate/up GEMM, x_perm is neither written
  // nor read
  void* x_perm = gather_fused(c) ? nullptr : w.x_perm;
  cudaError_t e;
  if (decode_front_applies(c)) {
    // a decode-sized batch: routing, permutation and gather in one launch
    // (which also clears the status words)
    e = launch_decode_front(c, x, w_router, logit_bias, sel_bias, idx, tw, cnt, ps, w.offsets,
                            w.sorted_pair, w.inv_pos, x_perm, w.seg, seg_tile(c), w.status, s);
    if (e != cudaSuccess) return fail_cuda(e);
  } else {
    if ((rc = reset_status(w.status, s)) != MOE_OK) return rc;
    e = launch_router(c, x, w_router, logit_bias, sel_bias, nullptr, w.logits, idx, tw, cnt, ps,
                      w.partials, w.status, s);
    if (e != cudaSuccess) return fail_cuda(e);
    if (c.T == 0) return MOE_OK;
    PermuteIn pin;
    if ((e = overflow_stage(c, sel_bias, idx, cnt, w.logits, w.assign, w.rr, w.status, s, &pin)) !=
        cudaSuccess)
      return fail_cuda(e);
    e = launch_permute(pin.pc, x, pin.idx, pin.counts, w.offsets, w.sorted_pair, w.inv_pos,
                       x_perm, w.hist, w.status, w.seg, seg_tile(c), s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  bool combined = false;
  rc = grouped_impl(c, x_perm, padded_rows(pairs(c)), x, w.offsets, w.sorted_pair, tw, w_gate,
                    w_up, w_down, w.y_perm, w.seg, true, w.h, w.partial, w.status, s, w.inv_pos, y,
                    &combined);
  if (rc != MOE_OK || combined) return rc;
  e = launch_combine(c, w.y_perm, w.inv_pos, nullptr, y, s);
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

// ---- backward -----------------------------------------------------------------
// Workspace of moe_layer_backward: the forward's routing and permutation,
// the recomputed rows (x_perm, H, a | b, o), and the gradients' rows (dL/dg,
// dO, dL/dr, da | db, dA). o and dA share one buffer: o is read only by the
// gate-gradient kernel, before dA is written.
struct BwdWs {
  int* status;
  float* logits;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  float* prob_sum;
  int32_t* offsets;
  int32_t* sorted_pair;
  int32_t* inv_pos;
  void* x_perm;
  float* partials;
  int32_t* hist;
  int32_t* seg;
  void* h;
  void* ab;
  void* o_dA;
  float* dg;
  void* dO;
  void* dr_bf;   // [T][n_pad] bf16
  void* drT_bf;  // [n_pad][t_pad] bf16
  void* dab;
  int32_t* assign;  // capacity rerouting only
  void* rr;
};
int bwd_n_pad(const moe_config& c) { return (c.n_experts + 7) / 8 * 8; }
int bwd_t_pad(const moe_config& c) { return (c.T + 7) / 8 * 8; }
BwdWs carve_bwd(Carver& cv, const moe_config& c) {
  BwdWs w;
  const size_t P = (size_t)pairs(c), N = (size_t)c.n_experts, T = (size_t)c.T;
  const size_t R = (size_t)padded_rows(rows_total(c)), d = c.d_model, f = c.d_ff;
  w.status = cv.take<int>(256);
  w.logits = cv.take<float>(sizeof(float) * T * N);
  w.topk_idx = cv.take<int32_t>(sizeof(int32_t) * P);
  w.topk_w = cv.take<float>(sizeof(float) * P);
  w.counts = cv.take<int32_t>(sizeof(int32_t) * N);
  w.prob_sum = cv.take<float>(sizeof(float) * N);
  w.offsets = cv.take<int32_t>(sizeof(int32_t) * (N + 1));
  w.sorted_pair = cv.take<int32_t>(sizeof(int32_t) * P);
  w.inv_pos = cv.take<int32_t>(sizeof(int32_t) * P);
  w.x_perm = cv.take<void>((size_t)padded_rows((long long)P) * d * 2);
  w.partials = cv.take<float>(router_partials_bytes(c));
  w.hist = cv.take<int32_t>(permute_scratch_bytes(c));
  w.seg = cv.take<int32_t>(sizeof(int32_t) * seg_table_words(c.n_experts + c.n_shared));
  w.h = cv.take<void>(R * f * 2);
  w.ab = cv.take<void>(R * 2 * f * 2);
  w.o_dA = cv.take<void>(R * d * 2);
  w.dg = cv.take<float>(sizeof(float) * P);
  w.dO = cv.take<void>(R * d * 2);
  const size_t np = (size_t)bwd_n_pad(c), tp = (size_t)bwd_t_pad(c);
  w.dr_bf = cv.take<void>(std::max<size_t>(T, 1) * np * 2);
  w.drT_bf = cv.take<void>(np * std::max<size_t>(tp, 8) * 2);
  w.dab = cv.take<void>(R * 2 * f * 2);
  const bool rr = reroutes(c);
  w.assign = rr ? cv.take<int32_t>(sizeof(int32_t) * P) : nullptr;
  w.rr = rr ? cv.take<void>(reroute_scratch_bytes(c)) : nullptr;
  return w;
}

size_t moe_workspace_size_backward(const moe_config* c) {
  if (moe_check_config(c) != MOE_OK || c->dtype != MOE_BF16 || c->d_ff % 64 != 0) return 0;
  Carver cv(nullptr);
  carve_bwd(cv, *c);
  return align_up(cv.off, 256);
}

int moe_layer_backward(const moe_config* cfg, const void* x, const void* w_router,
                       const float* logit_bias, const float* sel_bias, const void* w_gate,
                       const void* w_up, const void* w_down, const void* dy, float alpha,
                       float aux_grad, float* dx, float* dw_router, float* dw_gate,
                       float* dw_up, float* dw_down, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  int rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe_config& c = *cfg;
  if (c.dtype != MOE_BF16 || c.d_ff % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (!x || !w_router || !w_gate || !w_up || !w_down || !dy || !dx || !dw_router || !dw_gate ||
      !dw_up || !dw_down)
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned({x, w_router, logit_bias, sel_bias, w_gate, w_up, w_down, dy, dx, dw_router,
                    dw_gate, dw_up, dw_down}))
    return MOE_ERR_MISALIGNED;
  if ((rc = check_ws(c, ws, ws_bytes, moe_workspace_size_backward(cfg))) != MOE_OK) return rc;
  if ((rc = check_device(c)) != MOE_OK) return rc;
  Carver cv(ws);
  BwdWs w = carve_bwd(cv, c);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = reset_status(w.status, s)) != MOE_OK) return rc;
  // forward recompute: routing (with the scores), permutation, H, a | b, o
  cudaError_t e = launch_router(c, x, w_router, logit_bias, sel_bias, nullptr, w.logits,
                                w.topk_idx, w.topk_w, w.counts, w.prob_sum, w.partials, w.status,
                                s);
  if (e != cudaSuccess) return fail_cuda(e);
  const long long xp_rows = padded_rows(pairs(c)), r_rows = padded_rows(rows_total(c));
  if (c.T > 0) {
    PermuteIn pin;
    if ((e = overflow_stage(c, sel_bias, w.topk_idx, w.counts, w.logits, w.assign, w.rr, w.status,
                            s, &pin)) != cudaSuccess)
      return fail_cuda(e);
    e = launch_permute(pin.pc, x, pin.idx, pin.counts, w.offsets, w.sorted_pair, w.inv_pos,
                       w.x_perm, w.hist, w.status, w.seg, kTileM, s);
    if (e != cudaSuccess) return fail_cuda(e);
    e = launch_bwd_recompute(c, w.x_perm, x, w.seg, w_gate, w_up, w_down, w.h, w.ab, w.o_dA,
                             xp_rows, r_rows, w.status, s);
    if (e != cudaSuccess) return fail_cuda(e);
    // dL/dg and dO, then dL/dr
    e = launch_bwd_gate(c, dy, w.o_dA, w.inv_pos, w.topk_w, w.dg, w.dO, s);
    if (e != cudaSuccess) return fail_cuda(e);
    e = launch_bwd_score(c, w.logits, w.topk_idx, w.topk_w, w.dg, w.counts, alpha, aux_grad,
                         w.dr_bf, w.drT_bf, bwd_n_pad(c), bwd_t_pad(c), s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  // dx = dr W_r and dW_r = dr^T x (dW_r = 0 when T = 0)
  e = launch_bwd_router_grads(c, w.dr_bf, w.drT_bf, bwd_n_pad(c), bwd_t_pad(c), x, w_router, dx,
                              dw_router, w.status, s);
  if (e != cudaSuccess) return fail_cuda(e);
  if (c.T > 0) {
    // through the experts: da | db, dA; then dx += dA rows
    e = launch_bwd_dgrad(c, w.seg, w.dO, w.ab, w_gate, w_up, w_down, w.dab, w.o_dA, r_rows,
                         w.status, s);
    if (e != cudaSuccess) return fail_cuda(e);
    e = launch_bwd_dx(c, w.o_dA, w.inv_pos, dx, s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  // expert weight gradients (zero for experts that took no rows, and for T = 0)
  if (c.T == 0) {
    const size_t E = (size_t)c.n_experts + c.n_shared;
    const size_t wbytes = E * c.d_ff * c.d_model * sizeof(float);
    for (float* p : {dw_gate, dw_up, dw_down})
      if ((e = cudaMemsetAsync(p, 0, wbytes, s)) != cudaSuccess) return fail_cuda(e);
    return MOE_OK;
  }
  e = launch_bwd_wgrad(c, w.seg, w.x_perm, x, w.dab, w.dO, w.h, dw_gate, dw_up, dw_down, xp_rows,
                       r_rows, w.status, s);
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

size_t moe_workspace_size_fp8(const moe_config* c) {
  if (moe_check_config(c) != MOE_OK || c->dtype != MOE_BF16) return 0;
  if (c->d_model % 16 != 0 || c->d_ff % 16 != 0) return 0;
  Carver cv(nullptr);
  carve_layer_fp8(cv, *c);
  return align_up(cv.off, 256);
}

int moe_quantize_fp8(int64_t rows, int32_t cols, const void* src, uint8_t* q, float* scale,
                     moe_stream_t stream) {
  if (rows < 0 || cols < 8 || cols % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!src || !q || !scale) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({src, q, scale})) return MOE_ERR_MISALIGNED;
  QuantArgs a{};
  a.src = static_cast<const __nv_bfloat16*>(src);
  a.rows = rows;
  a.cols = cols;
  a.q = q;
  a.scale = scale;
  cudaError_t e = launch_quantize_rows(a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

int moe_layer_forward_fp8(const moe_config* cfg, const void* x, const void* w_router,
                          const float* logit_bias, const float* sel_bias, const uint8_t* wg_q,
                          const float* wg_scale, const uint8_t* wu_q, const float* wu_scale,
                          const uint8_t* wd_q, const float* wd_scale, void* y, int32_t* topk_idx,
                          float* topk_w, int32_t* counts, float* prob_sum, void* ws,
                          size_t ws_bytes, moe_stream_t stream) {
  int rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe_config& c = *cfg;
  if (c.dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;  // bf16 tokens, E4M3 experts
  // E4M3 rows are read by TMA, whose row pitch must be a multiple of 16 bytes
  if (c.d_model % 16 != 0 || c.d_ff % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if (c.T > 0 && (!x || !w_router || !wg_q || !wg_scale || !wu_q || !wu_scale || !wd_q ||
                  !wd_scale || !y))
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned({x, w_router, logit_bias, sel_bias, wg_q, wg_scale, wu_q, wu_scale, wd_q,
                    wd_scale, y, topk_idx, topk_w, counts, prob_sum}))
    return MOE_ERR_MISALIGNED;
  if ((rc = check_ws(c, ws, ws_bytes, moe_workspace_size_fp8(cfg))) != MOE_OK) return rc;
  if ((rc = check_device(c)) != MOE_OK) return rc;
  Carver cv(ws);
  LayerFp8Ws w8 = carve_layer_fp8(cv, c);
  LayerWs& w = w8.base;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* idx = topk_idx ? topk_idx : w.topk_idx;
  float* tw = topk_w ? topk_w : w.topk_w;
  int32_t* cnt = counts ? counts : w.counts;
  float* ps = prob_sum ? prob_sum : w.prob_sum;
  const long long P = pairs(c);
  cudaError_t e = route_and_permute(c, x, w_router, logit_bias, sel_bias, idx, tw, cnt, ps, w,
                                    seg_tile_m(c), s, &rc);
  if (e != cudaSuccess) return fail_cuda(e);
  if (rc != MOE_OK || c.T == 0) return rc;
  // routed rows: gathered and quantized in one pass; their H maxima cleared
  QuantArgs qa{};
  qa.src = static_cast<const __nv_bfloat16*>(x);
  qa.rows = P;
  qa.cols = c.d_model;
  qa.gather = w.sorted_pair;
  qa.k = c.top_k;
  qa.src_rows = c.T;
  qa.rows_dev = w.offsets + c.n_experts;
  qa.q = w8.xq_perm;
  qa.scale = w8.xp_scale;
  qa.clear = w8.h_amax;
  qa.clear_n = 1;
  e = launch_quantize_rows(qa, s);
  if (e == cudaSuccess && c.n_shared > 0) {  // x for the shared experts
    QuantArgs qs{};
    qs.src = static_cast<const __nv_bfloat16*>(x);
    qs.rows = c.T;
    qs.cols = c.d_model;
    qs.q = w8.xq;
    qs.scale = w8.x_scale;
    qs.clear = w8.h_amax;
    qs.clear_base = P;
    qs.clear_stride = c.T;
    qs.clear_n = c.n_shared;
    e = launch_quantize_rows(qs, s);
  }
  if (e == cudaSuccess)
    e = launch_grouped_e4m3(c, w8.xq_perm, w8.xp_scale, w8.xq, w8.x_scale, w.seg, w.sorted_pair, tw,
                            wg_q, wg_scale, wu_q, wu_scale, wd_q, wd_scale, w.h, w8.h_amax, w8.hq,
                            w8.h_scale, w.y_perm, w.partial, padded_rows(P),
                            padded_rows(rows_total(c)), w.status, s);
  if (e == cudaSuccess) e = launch_combine(c, w.y_perm, w.inv_pos, nullptr, y, s);
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

int32_t moe_nvfp4_scale_stride(int32_t cols) { return cols > 0 ? nvf4_sf_stride(cols) : 0; }

namespace {
// NVFP4 expert GEMMs read each operand row in 128-byte TMA boxes of codes
// (256 elements) and step K by 64 per MMA.
bool nvf4_shape_ok(const moe_config& c) {
  return c.d_model % 64 == 0 && c.d_ff % 64 == 0 && c.d_model >= 256 && c.d_ff >= 256;
}
}  // namespace

size_t moe_workspace_size_nvfp4(const moe_config* c) {
  if (moe_check_config(c) != MOE_OK || c->dtype != MOE_BF16 || !nvf4_shape_ok(*c)) return 0;
  Carver cv(nullptr);
  carve_layer_nvf4(cv, *c);
  return align_up(cv.off, 256);
}

int moe_quantize_nvfp4(int64_t rows, int32_t cols, const void* src, uint8_t* q, uint8_t* sf,
                       float* scale, moe_stream_t stream) {
  if (rows < 0 || cols < 16 || cols % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!src || !q || !sf || !scale) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({src, q, sf, scale})) return MOE_ERR_MISALIGNED;
  QuantArgs a{};
  a.src = static_cast<const __nv_bfloat16*>(src);
  a.rows = rows;
  a.cols = cols;
  a.q = q;
  a.sf = sf;
  a.ld_sf = nvf4_sf_stride(cols);
  a.scale = scale;
  cudaError_t e = launch_quantize_rows_nvf4(a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

int moe_layer_forward_nvfp4(const moe_config* cfg, const void* x, const void* w_router,
                            const float* logit_bias, const float* sel_bias, const uint8_t* wg_q,
                            const uint8_t* wg_sf, const float* wg_scale, const uint8_t* wu_q,
                            const uint8_t* wu_sf, const float* wu_scale, const uint8_t* wd_q,
                            const uint8_t* wd_sf, const float* wd_scale, void* y,
                            int32_t* topk_idx, float* topk_w, int32_t* counts, float* prob_sum,
                            void* ws, size_t ws_bytes, moe_stream_t stream) {
  int rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe_config& c = *cfg;
  if (c.dtype != MOE_BF16 || !nvf4_shape_ok(c)) return MOE_ERR_UNSUPPORTED;
  if (c.T > 0 && (!x || !w_router || !wg_q || !wg_sf || !wg_scale || !wu_q || !wu_sf ||
                  !wu_scale || !wd_q || !wd_sf || !wd_scale || !y))
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned({x, w_router, logit_bias, sel_bias, wg_q, wg_sf, wg_scale, wu_q, wu_sf,
                    wu_scale, wd_q, wd_sf, wd_scale, y, topk_idx, topk_w, counts, prob_sum}))
    return MOE_ERR_MISALIGNED;
  if ((rc = check_ws(c, ws, ws_bytes, moe_workspace_size_nvfp4(cfg))) != MOE_OK) return rc;
  if ((rc = check_device(c)) != MOE_OK) return rc;
  Carver cv(ws);
  LayerNvf4Ws w4 = carve_layer_nvf4(cv, c);
  LayerWs& w = w4.base;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* idx = topk_idx ? topk_idx : w.topk_idx;
  float* tw = topk_w ? topk_w : w.topk_w;
  int32_t* cnt = counts ? counts : w.counts;
  float* ps = prob_sum ? prob_sum : w.prob_sum;
  const long long P = pairs(c);
  // the NVFP4 GEMMs run 128-row tiles
  cudaError_t e = route_and_permute(c, x, w_router, logit_bias, sel_bias, idx, tw, cnt, ps, w,
                                    kTileM, s, &rc);
  if (e != cudaSuccess) return fail_cuda(e);
  if (rc != MOE_OK || c.T == 0) return rc;
  const int sfd = nvf4_sf_stride(c.d_model);
  // routed rows: gathered and quantized in one pass; their H maxima cleared
  QuantArgs qa{};
  qa.src = static_cast<const __nv_bfloat16*>(x);
  qa.rows = P;
  qa.cols = c.d_model;
  qa.gather = w.sorted_pair;
  qa.k = c.top_k;
  qa.src_rows = c.T;
  qa.rows_dev = w.offsets + c.n_experts;
  qa.q = w4.xq_perm;
  qa.sf = w4.xp_sf;
  qa.ld_sf = sfd;
  qa.scale = w4.xp_scale;
  qa.clear = w4.h_amax;
  qa.clear_n = 1;
  e = launch_quantize_rows_nvf4(qa, s);
  if (e == cudaSuccess && c.n_shared > 0) {  // x for the shared experts
    QuantArgs qs{};
    qs.src = static_cast<const __nv_bfloat16*>(x);
    qs.rows = c.T;
    qs.cols = c.d_model;
    qs.q = w4.xq;
    qs.sf = w4.x_sf;
    qs.ld_sf = sfd;
    qs.scale = w4.x_scale;
    qs.clear = w4.h_amax;
    qs.clear_base = P;
    qs.clear_stride = c.T;
    qs.clear_n = c.n_shared;
    e = launch_quantize_rows_nvf4(qs, s);
  }
  if (e == cudaSuccess)
    e = launch_grouped_nvf4(c, Nvf4Matrix{w4.xq_perm, w4.xp_sf, w4.xp_scale},
                            Nvf4Matrix{w4.xq, w4.x_sf, w4.x_scale}, w.seg, w.sorted_pair, tw,
                            Nvf4Matrix{wg_q, wg_sf, wg_scale}, Nvf4Matrix{wu_q, wu_sf, wu_scale},
                            Nvf4Matrix{wd_q, wd_sf, wd_scale}, w.h, w4.h_amax, w4.hq, w4.h_sf,
                            w4.h_scale, w.y_perm, w.partial, padded_rows(P), padded_rows(c.T),
                            padded_rows(rows_total(c)), w.status, s);
  if (e == cudaSuccess) e = launch_combine(c, w.y_perm, w.inv_pos, nullptr, y, s);
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

int moe_balance_stats(int32_t n_experts, int32_t T, int32_t top_k, const int32_t* counts,
                      const float* prob_sum, float alpha, float* f, float* P, float* aux,
                      moe_stream_t stream) {
  if (n_experts < 1 || n_experts > kMaxExperts || T < 0 || top_k < 1 || top_k > n_experts)
    return MOE_ERR_INVALID_ARG;
  if (!counts || !prob_sum || !f || !P || !aux) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({counts, prob_sum, f, P}) || ((uintptr_t)aux % 4)) return MOE_ERR_MISALIGNED;
  cudaError_t e = launch_balance_stats(n_experts, T, top_k, counts, prob_sum, alpha, f, P, aux,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : fail_cuda(e);
}

int moe_stream_status(const void* ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return MOE_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  int st = 0;
  e = cudaMemcpy(&st, ws, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  return st;
}

void moe_profile_enable(int mask) {
  Prof& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  p.mask = (uint32_t)mask;
  for (int i = 0; i < K_NUM; ++i)  // a kind switched off mid-launch leaves no open event
    if (!((p.mask >> i) & 1u)) p.open[i] = nullptr;
}

int moe_profile_collect(float* total_ms, int32_t* launches, int max_kernels) {
  Prof& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  std::vector<double> ms(K_NUM, 0.0);
  std::vector<int> n(K_NUM, 0);
  if (!p.done.empty()) cudaEventSynchronize(p.done.back().second.second);
  for (auto& d : p.done) {
    float t = 0.f;
    cudaEventSynchronize(d.second.second);
    if (cudaEventElapsedTime(&t, d.second.first, d.second.second) == cudaSuccess) {
      ms[d.first] += t;
      n[d.first] += 1;
    }
    p.pool.push_back(d.second.first);
    p.pool.push_back(d.second.second);
  }
  p.done.clear();
  for (int i = 0; i < K_NUM && i < max_kernels; ++i) {
    if (total_ms) total_ms[i] = (float)ms[i];
    if (launches) launches[i] = n[i];
  }
  return K_NUM;
}

const char* moe_profile_kernel_name(int id) {
  return (id >= 0 && id < K_NUM) ? kKernelNames[id] : "";
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
