// moe_permute_noalloc: the histogram + permutation step with its scratch
// memory in a fixed device array owned by this library, for callers that
// cannot allocate device memory themselves.
//
// Who needs it: code that runs where cudaMalloc is not allowed or not wanted
// -- inside a CUDA stream capture that is being recorded into a graph, inside
// a serving runtime whose device memory is planned once at start-up, or in a
// plugin whose host framework owns every allocation and hands it only the
// input and output tensors.  Such a caller cannot size and pass the workspace
// that moe_permute needs, so this variant keeps the per-block counts and bases
// in `g_permute_scratch` below instead.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library is loaded holds kNoAllocScratchBytes of it until the process
// exits.  Host code may not use the symbol itself as a device pointer (on the
// host it names a shadow object, not GPU memory), so its device address is
// looked up with cudaGetSymbolAddress in the CUDA context that is current at
// the call.  The lookup is cheap and is repeated on every call made outside a
// stream capture, so a context that was destroyed and re-created (for example
// after cudaDeviceReset) never reaches a stale address.  A call made while its
// stream is being captured cannot look anything up; it uses the address found
// by the last call outside capture in the same context, so make one call in
// each context (device) before any stream capture starts.
//
// All calls share the one array, and it keeps whatever the previous call left
// in it.  The kernels overwrite every count and base they read, and the call
// clears the status word it owns before launching.  Two calls that run on the
// GPU at the same time (different streams, no ordering between them) race on
// the array and give wrong results: order them on one stream or with events.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <unordered_map>

#include "../../include/moe_layer.h"
#include "moe_internal.h"

namespace moe {
namespace {

// Per-block counts and bases, E x ceil(T/64) int32 each: 262144 entries cover
// E = 256 experts with up to 65536 tokens.  Plus one 256-byte status word.
constexpr int64_t kNoAllocMaxEntries = 262144;
constexpr size_t kNoAllocStatusBytes = 256;
constexpr size_t kNoAllocScratchBytes =
    kNoAllocStatusBytes + 2 * size_t(kNoAllocMaxEntries) * sizeof(int32_t);

static __device__ __align__(256) uint8_t g_permute_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
std::unordered_map<CUcontext, uint8_t*> g_scratch_addr;  // by CUDA context

moe_status_t report(moe_status_t s, const char* msg) {
  set_last_error_text(msg);
  return s;
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The calling thread's current CUDA context (null if it cannot be read).
CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// Device address of g_permute_scratch in the current context: looked up afresh
// outside stream capture, taken from the last lookup in this context during one.
moe_status_t scratch_address(cudaStream_t st, uint8_t** out) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t qe = cudaStreamIsCapturing(st, &cs);
  if (qe != cudaSuccess) (void)cudaGetLastError();  // the query's own error is not the caller's
  const bool capturing = qe != cudaSuccess || cs != cudaStreamCaptureStatusNone;
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> g(g_mu);
  if (!capturing) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess || !p) {
      char buf[256];
      snprintf(buf, sizeof buf, "moe_permute_noalloc: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      return report(MOE_ERR_CUDA, buf);
    }
    g_scratch_addr[ctx] = static_cast<uint8_t*>(p);
  }
  auto it = g_scratch_addr.find(ctx);
  if (it == g_scratch_addr.end())
    return report(MOE_ERR_INVALID_ARG,
                  "moe_permute_noalloc: first call in this context made during a stream capture; "
                  "call it once before capturing");
  *out = it->second;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status_t moe_permute_noalloc(
    const moe_config_t* cfg, const int32_t* topk_ids, const float* topk_w, const void* x,
    int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm_token, int32_t* inv_row,
    float* row_weight, void* x_perm, float* x_perm_scales, uint32_t* device_status,
    moe_stream_t stream) {
  moe_status_t s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (cfg->wtype == MOE_DTYPE_NVFP4)
    return report(MOE_ERR_UNSUPPORTED, "NVFP4 layers run through moe_forward / moe_forward_stack");
  const int64_t nblk = (cfg->T + kPermTok - 1) / kPermTok;
  if (nblk * cfg->E > kNoAllocMaxEntries) {
    char buf[256];
    snprintf(buf, sizeof buf,
             "moe_permute_noalloc: E * ceil(T/64) = %lld exceeds the fixed scratch of %lld "
             "entries (e.g. T <= 65536 at E = 256); use moe_permute with a workspace",
             static_cast<long long>(nblk * cfg->E), static_cast<long long>(kNoAllocMaxEntries));
    return report(MOE_ERR_UNSUPPORTED, buf);
  }
  if ((s = check_ptr4(expert_counts, "expert_counts")) != MOE_OK) return s;
  if ((s = check_ptr4(expert_offsets, "expert_offsets")) != MOE_OK) return s;
  if (device_status && (s = check_ptr4(device_status, "device_status")) != MOE_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cfg->T == 0) {
    cudaError_t e = cudaMemsetAsync(expert_counts, 0, size_t(cfg->E) * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(expert_offsets, 0, size_t(cfg->E + 1) * 4, st);
    return e == cudaSuccess ? MOE_OK : report(MOE_ERR_CUDA, cudaGetErrorString(e));
  }
  if ((s = check_ptr4(topk_ids, "topk_ids")) != MOE_OK) return s;
  if ((s = check_ptr4(perm_token, "perm_token")) != MOE_OK) return s;
  if ((s = check_ptr4(inv_row, "inv_row")) != MOE_OK) return s;
  if (row_weight) {
    if ((s = check_ptr4(row_weight, "row_weight")) != MOE_OK) return s;
    if (!topk_w) return report(MOE_ERR_INVALID_ARG, "row_weight needs topk_w");
    if ((s = check_ptr4(topk_w, "topk_w")) != MOE_OK) return s;
  }
  if (x_perm) {
    if ((s = check_ptr(x, "x")) != MOE_OK) return s;
    if ((s = check_ptr(x_perm, "x_perm")) != MOE_OK) return s;
    if (cfg->wtype == MOE_DTYPE_FP8_E4M3 && (s = check_ptr4(x_perm_scales, "x_perm_scales")) != MOE_OK)
      return s;
  }

  uint8_t* base = nullptr;
  if ((s = scratch_address(st, &base)) != MOE_OK) return s;
  uint32_t* own_status = reinterpret_cast<uint32_t*>(base);
  int32_t* blk_counts = reinterpret_cast<int32_t*>(base + kNoAllocStatusBytes);
  int32_t* blk_base = blk_counts + kNoAllocMaxEntries;
  uint32_t* err = device_status ? device_status : own_status;

  // The scratch status word starts every call at zero; counts and bases are
  // fully rewritten by the kernels before they are read.
  cudaError_t e = cudaMemsetAsync(own_status, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = launch_hist(topk_ids, cfg->T, cfg->k, cfg->E, blk_counts, err, st);
  if (e == cudaSuccess)
    e = launch_scan(blk_counts, static_cast<int>(nblk), cfg->E, blk_base, expert_counts,
                    expert_offsets, st);
  if (e == cudaSuccess)
    e = launch_scatter(topk_ids, topk_w, x, cfg->T, cfg->k, cfg->E, cfg->H,
                       cfg->wtype == MOE_DTYPE_FP8_E4M3, blk_base, expert_offsets, perm_token,
                       inv_row, row_weight, x_perm, x_perm_scales, err, st);
  if (e != cudaSuccess) return report(MOE_ERR_CUDA, cudaGetErrorString(e));
  return MOE_OK;
}
