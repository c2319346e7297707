// moe_router_topk_noalloc: the router entry point for callers that cannot
// allocate device memory and cannot hand the library a workspace.
//
// Some callers own every byte of device memory up front: an inference
// runtime whose memory planner assigns all buffers before the first step,
// or a plugin interface that gives an operator only its inputs and outputs
// and has no workspace slot. They can neither call cudaMalloc nor pass the
// scratch that moe_router_topk takes. This entry point runs the same router
// kernels, with their scratch (one status word and the per-block
// probability sums and counts) in a fixed array of this library's own device
// memory instead of a caller workspace.
//
// Limits and rules (also stated in include/moe.h):
//  - The array is kNoallocScratchBytes (1 MiB) per GPU that loads the
//    library, held until the process exits. A call needs 256 + 8 * B * N
//    bytes of it (a float sum and an int count per block and expert), with
//    B = ceil(T / 64), or max(ceil(T / 64), min(T, 608)) when N <= 32 (the
//    most blocks a router kernel runs); a larger call returns
//    MOE_ERR_WORKSPACE and launches nothing.
//  - The array's device address is looked up once per CUDA context, by the
//    first call made while that context is current; make that first call
//    before any stream capture. The lookup is keyed on the context's
//    process-unique id, so a context created after cudaDeviceReset (or a
//    second context on the same device) gets its own lookup.
//  - Errors the kernels find while they run (a bounded wait that ran out)
//    go to a status word at the start of the array; the caller reads it
//    with moe_router_topk_noalloc_status, which synchronises the stream.
//  - Every call shares the one array and it keeps the last call's contents.
//    The status word and the router's finished-block counter are cleared at
//    the start of every call; the per-block sums and counts are fully
//    rewritten before they are read. Calls whose work overlaps on the
//    GPU (different streams, or different host threads without ordering)
//    race on the array and give undefined results.
//  - Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda.h>

#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr size_t kNoallocScratchBytes = 1u << 20;  // 1 MiB
constexpr size_t kStatusBytes = 256;
constexpr int kMaxContexts = 64;

static __device__ __align__(256) unsigned char g_router_scratch[kNoallocScratchBytes];

// Driver entry points for the current context and its id, looked up through
// the runtime (the library does not link the driver library).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CtxFns {
  CtxGetCurrentFn current = nullptr;
  CtxGetIdFn id = nullptr;
};

const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return f;
}

// Process-unique id of the current CUDA context, creating the device's
// primary context first if the runtime has not done so yet (cudaSetDevice on
// the current device does that and allocates nothing).
cudaError_t current_context_id(unsigned long long* id) {
  const CtxFns& f = ctx_fns();
  if (!f.current || !f.id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (f.current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  if (!ctx) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (f.current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorUnknown;
  }
  return f.id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

std::mutex g_setup_mu;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
ScratchEntry g_scratch[kMaxContexts] = {};
int g_scratch_n = 0;

// Device address of g_router_scratch in the current context (looked up once
// per context). Returns a cudaError_t.
cudaError_t scratch_for_current_context(void** out) {
  unsigned long long id = 0;
  cudaError_t e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(g_setup_mu);
  for (int i = 0; i < g_scratch_n; ++i)
    if (g_scratch[i].ctx_id == id) {
      *out = g_scratch[i].addr;
      return cudaSuccess;
    }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_router_scratch);
  if (e != cudaSuccess) return e;
  // A full table drops its oldest entry (a context that no longer exists is
  // never looked up again).
  if (g_scratch_n == kMaxContexts) {
    for (int i = 1; i < kMaxContexts; ++i) g_scratch[i - 1] = g_scratch[i];
    --g_scratch_n;
  }
  g_scratch[g_scratch_n++] = ScratchEntry{id, p};
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_router_topk_noalloc(const moe_config* cfg, const void* x, const void* w_router,
                                       const float* logit_bias, const float* sel_bias,
                                       const float* logits_in, float* logits_out,
                                       int32_t* topk_idx, float* topk_w, int32_t* counts,
                                       float* prob_sum, moe_stream_t stream) {
  int rc = moe_check_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe_config& c = *cfg;
  if (!counts || !prob_sum) return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && (!topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && !logits_in && (!x || !w_router)) return MOE_ERR_INVALID_ARG;
  if (logits_in && logit_bias) return MOE_ERR_INVALID_ARG;
  for (const void* p : {x, w_router, (const void*)logit_bias, (const void*)sel_bias,
                        (const void*)logits_in, (const void*)logits_out, (const void*)topk_idx,
                        (const void*)topk_w, (const void*)counts, (const void*)prob_sum})
    if (p && ((uintptr_t)p % 16)) return MOE_ERR_MISALIGNED;
  if (kStatusBytes + router_partials_bytes(c) > kNoallocScratchBytes) return MOE_ERR_WORKSPACE;

  void* scratch = nullptr;
  cudaError_t e = scratch_for_current_context(&scratch);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  int* status = static_cast<int*>(scratch);
  float* partials = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + kStatusBytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  e = launch_reset_status(status, s);  // status, router block counter
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_router(c, x, w_router, logit_bias, sel_bias, logits_in, logits_out, topk_idx, topk_w,
                    counts, prob_sum, partials, status, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_router_topk_noalloc_status(moe_stream_t stream) {
  void* scratch = nullptr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = scratch_for_current_context(&scratch);
  int st = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&st, scratch, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? st : MOE_ERR_CUDA;
}
