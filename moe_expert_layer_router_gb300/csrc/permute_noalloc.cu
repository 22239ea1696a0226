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
// looked up with cudaGetSymbolAddress once per device, on the first call made
// while that device is current.  Make that first call before any stream
// capture starts.
//
// All calls share the one array, and it keeps whatever the previous call left
// in it.  The kernels overwrite every count and base they read, and the call
// clears the status word it owns before launching.  Two calls that run on the
// GPU at the same time (different streams, no ordering between them) race on
// the array and give wrong results: order them on one stream or with events.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

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

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint8_t* g_scratch_addr[kMaxDevices] = {};

moe_status_t report(moe_status_t s, const char* msg) {
  set_last_error_text(msg);
  return s;
}

// Device address of g_permute_scratch on the current device (looked up once).
moe_status_t scratch_address(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report(MOE_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return report(MOE_ERR_UNSUPPORTED, "moe_permute_noalloc: device index above 63");
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess || !p) {
      char buf[256];
      snprintf(buf, sizeof buf, "moe_permute_noalloc: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      return report(MOE_ERR_CUDA, buf);
    }
    g_scratch_addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool ok4(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3) == 0; }
bool ok16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status_t moe_permute_noalloc(
    const moe_config_t* cfg, const int32_t* topk_ids, const float* topk_w, const void* x,
    int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm_token, int32_t* inv_row,
    float* row_weight, void* x_perm, float* x_perm_scales, uint32_t* device_status,
    moe_stream_t stream) {
  if (!cfg) return report(MOE_ERR_INVALID_ARG, "moe_permute_noalloc: cfg is NULL");
  if (cfg->T < 0 || cfg->E < 1 || cfg->E > kMaxExperts || cfg->k < 1 || cfg->k > cfg->E ||
      cfg->k > 16 || cfg->H < 128 || cfg->H % 128 ||
      (cfg->wtype != MOE_DTYPE_BF16 && cfg->wtype != MOE_DTYPE_FP8_E4M3) ||
      cfg->T * int64_t(cfg->k) >= (int64_t(1) << 31))
    return report(MOE_ERR_INVALID_ARG, "moe_permute_noalloc: invalid layer configuration");
  const int64_t nblk = (cfg->T + kPermTok - 1) / kPermTok;
  if (nblk * cfg->E > kNoAllocMaxEntries) {
    char buf[256];
    snprintf(buf, sizeof buf,
             "moe_permute_noalloc: E * ceil(T/64) = %lld exceeds the fixed scratch of %lld "
             "entries (e.g. T <= 65536 at E = 256); use moe_permute with a workspace",
             static_cast<long long>(nblk * cfg->E), static_cast<long long>(kNoAllocMaxEntries));
    return report(MOE_ERR_UNSUPPORTED, buf);
  }
  if (!ok4(expert_counts) || !ok4(expert_offsets))
    return report(MOE_ERR_INVALID_ARG, "moe_permute_noalloc: counts/offsets NULL or misaligned");
  if (device_status && !ok4(device_status))
    return report(MOE_ERR_INVALID_ARG, "moe_permute_noalloc: device_status misaligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cfg->T == 0) {
    cudaError_t e = cudaMemsetAsync(expert_counts, 0, size_t(cfg->E) * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(expert_offsets, 0, size_t(cfg->E + 1) * 4, st);
    return e == cudaSuccess ? MOE_OK : report(MOE_ERR_CUDA, cudaGetErrorString(e));
  }
  if (!ok4(topk_ids) || !ok4(perm_token) || !ok4(inv_row))
    return report(MOE_ERR_INVALID_ARG, "moe_permute_noalloc: ids/perm/inv NULL or misaligned");
  if (row_weight && (!ok4(row_weight) || !ok4(topk_w)))
    return report(MOE_ERR_INVALID_ARG, "moe_permute_noalloc: row_weight needs aligned topk_w");
  if (x_perm && (!ok16(x) || !ok16(x_perm)))
    return report(MOE_ERR_INVALID_ARG, "moe_permute_noalloc: x / x_perm NULL or misaligned");
  if (x_perm && cfg->wtype == MOE_DTYPE_FP8_E4M3 && !ok4(x_perm_scales))
    return report(MOE_ERR_INVALID_ARG, "moe_permute_noalloc: fp8 needs x_perm_scales");

  uint8_t* base = nullptr;
  moe_status_t s = scratch_address(&base);
  if (s != MOE_OK) return s;
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
