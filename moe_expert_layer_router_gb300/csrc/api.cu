// Host side of the C ABI declared in include/moe_layer.h: argument validation,
// workspace layout, TMA descriptor encoding and the launch sequence of each
// step.  Everything here runs on the host; every step of the layer runs in
// the kernels of router.cu, permute.cu, grouped_gemm.cu and combine.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/moe_layer.h"
#include "moe_internal.h"

namespace moe {

// ------------------------------------------------------------------ errors
static thread_local std::string g_last_error;

static moe_status_t fail(moe_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

// Lets other translation units report host-side failures through
// moe_last_error_message().
void set_last_error_text(const char* msg) { g_last_error = msg ? msg : ""; }

static moe_status_t cuda_fail(cudaError_t e, const char* where) {
  return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define MOE_CUDA(call)                                   \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);  \
  } while (0)

// ------------------------------------------------------------------ device info
static int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

static int sm_count() {
  static std::mutex mu;
  static std::unordered_map<int, int> cache;
  const int d = current_device();
  std::lock_guard<std::mutex> g(mu);
  auto it = cache.find(d);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 1;
  cache[d] = n;
  return n;
}

static int gemm_grid() {
  static std::mutex mu;
  static std::unordered_map<int, int> cache;
  const int n = sm_count();
  const int d = current_device();
  std::lock_guard<std::mutex> g(mu);
  auto it = cache.find(d);
  if (it != cache.end()) return it->second;
  const int grid = grouped_gemm_grid(n);
  cache[d] = grid;
  return grid;
}

cudaError_t ensure_smem_attr(const void* func, int bytes) {
  static std::mutex mu;
  static std::unordered_map<const void*, uint64_t> done;  // device bitmask per kernel
  const int d = current_device();
  const uint64_t bit = d < 64 ? (uint64_t(1) << d) : 0;
  {
    std::lock_guard<std::mutex> g(mu);
    if (bit && (done[func] & bit)) return cudaSuccess;
  }
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(mu);
  done[func] |= bit;
  return cudaSuccess;
}

// ------------------------------------------------------------------ failure-path test
static thread_local int32_t g_gemm1_stalls = 0;

bool take_gemm1_stall() {
  if (g_gemm1_stalls <= 0) return false;
  --g_gemm1_stalls;
  return true;
}

// ------------------------------------------------------------------ tracing
static thread_local moe_trace_t* g_trace = nullptr;

void trace_mark(cudaStream_t stream, int id) {
  moe_trace_t* t = g_trace;
  if (!t || t->count >= t->capacity) return;
  if (t->kernel_mask != 0u && (id < 0 || ((t->kernel_mask >> id) & 1u) == 0u)) return;
  if (cudaEventRecord(static_cast<cudaEvent_t>(t->events[t->count]), stream) != cudaSuccess) return;
  t->kernel_ids[t->count] = id;
  t->count += 1;
}

// ------------------------------------------------------------------ TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Row-major [rows, inner] matrix, 128-byte swizzled boxes of box_rows x box_inner.
static moe_status_t encode_2d(CUtensorMap* m, bool bf16, const void* base, uint64_t inner,
                              uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const uint64_t esz = bf16 ? 2 : 1;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * esz};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a [%llu, %llu] matrix",
                static_cast<int>(r), static_cast<unsigned long long>(rows),
                static_cast<unsigned long long>(inner));
  return MOE_OK;
}

// ------------------------------------------------------------------ validation
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

moe_status_t check_config(const moe_config_t* c) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cfg is NULL");
  if (c->T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %lld is negative", (long long)c->T);
  if (c->E < 1 || c->E > kMaxExperts)
    return fail(MOE_ERR_UNSUPPORTED, "E = %d outside 1..%d", c->E, kMaxExperts);
  if (c->k < 1 || c->k > c->E || c->k > 16)
    return fail(MOE_ERR_INVALID_ARG, "k = %d outside 1..min(E, 16)", c->k);
  if (c->H < 128 || c->H % 128)
    return fail(MOE_ERR_UNSUPPORTED, "H = %d is not a positive multiple of 128", c->H);
  if (c->I < 128 || c->I % 128)
    return fail(MOE_ERR_UNSUPPORTED, "I = %d is not a positive multiple of 128", c->I);
  if (c->I_shared < 0 || c->I_shared % 128)
    return fail(MOE_ERR_UNSUPPORTED, "I_shared = %d is not 0 or a multiple of 128", c->I_shared);
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID)
    return fail(MOE_ERR_INVALID_ARG, "score = %d is not a moe_score_t", c->score);
  if (c->renormalize != 0 && c->renormalize != 1)
    return fail(MOE_ERR_INVALID_ARG, "renormalize = %d is not 0 or 1", c->renormalize);
  if (!std::isfinite(c->route_scale) || c->route_scale <= 0.0f)
    return fail(MOE_ERR_INVALID_ARG, "route_scale must be finite and > 0");
  if (c->wtype != MOE_DTYPE_BF16 && c->wtype != MOE_DTYPE_FP8_E4M3 && c->wtype != MOE_DTYPE_NVFP4)
    return fail(MOE_ERR_INVALID_ARG, "wtype = %d is not a moe_dtype_t", c->wtype);
  if (c->wtype == MOE_DTYPE_NVFP4 && (c->H % 256 || c->I % 256 || c->I_shared % 256))
    return fail(MOE_ERR_UNSUPPORTED, "NVFP4 layers need H, I and I_shared multiples of 256");
  if (c->T * int64_t(c->k) >= (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "T*k = %lld does not fit int32 row indices",
                (long long)(c->T * c->k));
  return MOE_OK;
}

moe_status_t check_ptr(const void* p, const char* name, bool needs16) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);
  if (needs16 && !aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return MOE_OK;
}

moe_status_t check_ptr4(const void* p, const char* name) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(p) & 3) return fail(MOE_ERR_INVALID_ARG, "%s is not 4-byte aligned", name);
  return MOE_OK;
}

#define MOE_TRY(expr)                     \
  do {                                    \
    moe_status_t s_ = (expr);             \
    if (s_ != MOE_OK) return s_;          \
  } while (0)

// ------------------------------------------------------------------ workspace layout
constexpr size_t kHeaderBytes = 256;

static size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

struct Layout {
  size_t blk_counts = 0, blk_base = 0;        // permute
  size_t amap = 0;                            // bf16 grouped ffn: cut A tensor maps
  size_t sched1 = 0, sched2 = 0, h = 0, hs = 0;  // grouped ffn
  size_t h_sc = 0, hs_sc = 0;                 // fp8: scales of h and of the shared h
  size_t ids = 0, w = 0, counts = 0, offsets = 0, perm_token = 0, inv_row = 0, row_weight = 0,
         x_perm = 0, y_perm = 0, shared_out = 0;  // forward
  size_t x_perm_sc = 0, xq = 0, xq_sc = 0;    // forward, fp8: x_perm scales, quantised x
  size_t pad_offsets = 0;                     // NVFP4: offsets of the 128-row-padded segments
  size_t total = 0;
};

// NVFP4 keeps every expert's rows in whole 128-row blocks: at most R + 127 E rows.
static int64_t nvfp4_rows(const moe_config_t& c) {
  const int64_t r = c.T * c.k + int64_t(c.E) * (kNvfp4Rows - 1);
  return (r + kNvfp4Rows - 1) / kNvfp4Rows * kNvfp4Rows;
}
static int64_t nvfp4_tokens(const moe_config_t& c) {
  return (c.T + kNvfp4Rows - 1) / kNvfp4Rows * kNvfp4Rows;
}

static Layout layout(const moe_config_t& c, int op) {
  Layout L;
  size_t at = kHeaderBytes;
  auto take = [&](size_t bytes) {
    const size_t o = at;
    at += up256(bytes);
    return o;
  };
  const int64_t T = c.T, R = c.T * c.k;
  const int nblk = static_cast<int>((T + kPermTok - 1) / kPermTok);
  const int G = c.E + (c.I_shared > 0 ? 1 : 0);
  const bool perm = op == MOE_OP_PERMUTE || op == MOE_OP_FORWARD;
  const bool ffn = op == MOE_OP_GROUPED_FFN || op == MOE_OP_FORWARD;
  if (perm) {
    L.blk_counts = take(size_t(nblk) * c.E * 4);
    L.blk_base = take(size_t(nblk) * c.E * 4);
  }
  const bool fp8 = c.wtype == MOE_DTYPE_FP8_E4M3;
  const bool fp4 = c.wtype == MOE_DTYPE_NVFP4;
  const size_t esz = fp8 ? 1 : 2;  // bytes per element of x_perm and h
  if (fp4) {
    // codes (half a byte per element) and MMA-layout scales (1/16 byte) over
    // the padded rows; the expert outputs as fp16 + scales in fp32-sized regions
    const size_t Rp = size_t(nvfp4_rows(c)), Tp = size_t(nvfp4_tokens(c));
    if (ffn) {
      L.sched1 = take(size_t(sched_ints(G)) * 4);
      L.sched2 = take(size_t(sched_ints(G)) * 4);
      L.h = take(Rp * c.I / 2);
      L.hs = take(Tp * c.I_shared / 2);
      L.h_sc = take(Rp * c.I / 16);
      L.hs_sc = take(Tp * c.I_shared / 16);
    }
    if (op == MOE_OP_GROUPED_FFN) {
      // the expert outputs as fp16 + power-of-two scales per 32 columns, widened
      // into the caller's fp32 rows by the last kernel of the call
      L.y_perm = take(size_t(R) * c.H * 2 + size_t(R) * (c.H / 32) * 4);
      L.shared_out = take(size_t(T) * c.H * 2 + size_t(T) * (c.H / 32) * 4);
    }
    if (op == MOE_OP_FORWARD) {
      L.ids = take(size_t(R) * 4);
      L.w = take(size_t(R) * 4);
      L.counts = take(size_t(c.E) * 4);
      L.offsets = take(size_t(c.E + 1) * 4);
      L.pad_offsets = take(size_t(c.E + 1) * 4);
      L.perm_token = take(size_t(R) * 4);
      L.inv_row = take(size_t(R) * 4);
      L.row_weight = take(size_t(R) * 4);
      L.x_perm = take(Rp * c.H / 2);
      L.x_perm_sc = take(Rp * c.H / 16);
      L.xq = take(Tp * c.H / 2);
      L.xq_sc = take(Tp * c.H / 16);
      L.y_perm = take(size_t(R) * c.H * 4);
      L.shared_out = take(size_t(T) * c.H * 4);
    }
    L.total = at;
    return L;
  }
  if (ffn) {
    L.sched1 = take(size_t(sched_ints(G)) * 4);
    L.sched2 = take(size_t(sched_ints(G)) * 4);
    L.h = take(size_t(R) * c.I * esz);
    L.hs = take(size_t(T) * c.I_shared * esz);
    if (!fp8) L.amap = take(size_t(2) * c.E * 128);
    if (fp8) {
      L.h_sc = take(size_t(R) * (c.I / 128) * 4);
      L.hs_sc = take(size_t(T) * (c.I_shared / 128) * 4);
    }
  }
  if (op == MOE_OP_FORWARD) {
    L.ids = take(size_t(R) * 4);
    L.w = take(size_t(R) * 4);
    L.counts = take(size_t(c.E) * 4);
    L.offsets = take(size_t(c.E + 1) * 4);
    L.perm_token = take(size_t(R) * 4);
    L.inv_row = take(size_t(R) * 4);
    L.row_weight = take(size_t(R) * 4);
    L.x_perm = take(size_t(R) * c.H * esz);
    if (fp8) {
      L.x_perm_sc = take(size_t(R) * (c.H / 128) * 4);
      L.xq = take(size_t(T) * c.H);
      L.xq_sc = take(size_t(T) * (c.H / 128) * 4);
    }
    L.y_perm = take(size_t(R) * c.H * 4);
    L.shared_out = take(size_t(T) * c.H * 4);
  }
  L.total = at;
  return L;
}

static moe_status_t check_ws(const moe_config_t& c, int op, const void* ws, size_t bytes) {
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) & 255)
    return fail(MOE_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  const size_t need = layout(c, op).total;
  if (bytes < need)
    return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", bytes, need);
  return MOE_OK;
}

template <typename P>
static P at(void* ws, size_t off) {
  return reinterpret_cast<P>(static_cast<uint8_t*>(ws) + off);
}

static uint32_t* err_word(void* ws) { return static_cast<uint32_t*>(ws); }

}  // namespace moe

// ======================================================================== weights
struct moe_weights {
  moe_config_t cfg;
  int device;
  void* table;          // device: CUtensorMap maps1[2G], maps2[G] (+ fp8: scale pointers)
  CUtensorMap* maps1;
  CUtensorMap* maps2;
  const float** scales1;  // fp8: gate of group g at 2g, up at 2g+1 (NVFP4: scale bytes)
  const float** scales2;  // fp8: down of group g at g
  const float** gs1;      // NVFP4: tensor-scale pointers, indexed like scales1
  const float** gs2;
  float* act;             // NVFP4: device [2] = g_x, g_h
};

// Descriptor tables one call reads: a single layer's, or a layer stack's
// (layer 0's entries plus a device layer index and the per-layer stride).
struct moe_stack {
  moe_config_t cfg;
  int device;
  int32_t num_layers;
  int32_t G;
  void* table;              // device: maps [L][3G] | router maps [L] | bias [L] | fp8 scales [L][3G]
                            //   | NVFP4: tensor scales [L][3G] | activation scales [L][2]
  CUtensorMap* maps;
  CUtensorMap* router;
  const float** bias;
  const float** scales;
  const float** gs;
  float* act;
};

namespace moe {
struct WeightView {
  const CUtensorMap* maps1;
  const CUtensorMap* maps2;
  const float* const* scales1;
  const float* const* scales2;
  const int32_t* layer;
  int32_t stride;
  int32_t num_layers;
  const float* const* gs1 = nullptr;  // NVFP4 tensor scales
  const float* const* gs2 = nullptr;
  const float* act = nullptr;         // NVFP4 [num_layers][2]
};
static WeightView view_of(const moe_weights* W) {
  WeightView v{W->maps1, W->maps2, W->scales1, W->scales2, nullptr, 0, 1};
  v.gs1 = W->gs1;
  v.gs2 = W->gs2;
  v.act = W->act;
  return v;
}
static WeightView view_of(const moe_stack* S, const int32_t* layer) {
  const bool scaled = S->cfg.wtype != MOE_DTYPE_BF16;
  WeightView v{S->maps, S->maps + 2 * S->G, scaled ? S->scales : nullptr,
               scaled ? S->scales + 2 * S->G : nullptr, layer, 3 * S->G, S->num_layers};
  if (S->cfg.wtype == MOE_DTYPE_NVFP4) {
    v.gs1 = S->gs;
    v.gs2 = S->gs + 2 * S->G;
    v.act = S->act;
  }
  return v;
}
}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

moe_status_t moe_test_stall_gemm1(int32_t count) {
  if (count < 0) return fail(MOE_ERR_INVALID_ARG, "count = %d is negative", count);
  g_gemm1_stalls = count;
  return MOE_OK;
}

moe_status_t moe_set_trace(moe_trace_t* trace) {
  if (trace && (!trace->events || !trace->kernel_ids || trace->capacity < 0 || trace->count < 0))
    return fail(MOE_ERR_INVALID_ARG, "trace needs events, kernel_ids and a capacity");
  g_trace = trace;
  return MOE_OK;
}

const char* moe_last_error_message(void) { return g_last_error.c_str(); }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MOE_ERR_BOUNDS: return "device index out of bounds";
  }
  return "unknown status";
}

moe_status_t moe_workspace_size(const moe_config_t* cfg, int32_t op, size_t* bytes) {
  MOE_TRY(check_config(cfg));
  if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
  if (op < MOE_OP_ROUTE || op > MOE_OP_FORWARD) return fail(MOE_ERR_INVALID_ARG, "op = %d", op);
  *bytes = layout(*cfg, op).total;
  return MOE_OK;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || ws_bytes < kHeaderBytes) return fail(MOE_ERR_WORKSPACE, "workspace NULL or too small");
  if (reinterpret_cast<uintptr_t>(ws) & 255)
    return fail(MOE_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  MOE_CUDA(cudaMemsetAsync(ws, 0, kHeaderBytes, reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status_t moe_get_device_error(void* ws, moe_stream_t stream, int32_t* device_bits) {
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t w = 0;
  MOE_CUDA(cudaMemcpyAsync(&w, ws, 4, cudaMemcpyDeviceToHost, st));
  MOE_CUDA(cudaMemsetAsync(ws, 0, 4, st));
  MOE_CUDA(cudaStreamSynchronize(st));
  if (device_bits) *device_bits = static_cast<int32_t>(w);
  if (w & kErrTimeout) return fail(MOE_ERR_DEVICE_TIMEOUT, "a kernel wait timed out (bits 0x%x)", w);
  if (w & kErrDupIds)
    return fail(MOE_ERR_BOUNDS, "a token listed the same expert twice among its k ids (bits 0x%x)", w);
  if (w & (kErrBounds | kErrNoSelect))
    return fail(MOE_ERR_BOUNDS, "a kernel met an out-of-range index (bits 0x%x)", w);
  return MOE_OK;
}

// Validates one layer's weight list and encodes its 3G TMA descriptors
// (GEMM1: gate / up of group g at 2g / 2g+1; GEMM2: down of group g at 2G+g)
// and, for fp8, the matching scale pointers, into maps[3G] / scales[3G].
static moe_status_t encode_layer_nvfp4(const moe_config_t* cfg, const moe_weight_list_t* wl,
                                       CUtensorMap* maps, const float** scales, const float** gs,
                                       float* act, bool encode);

static moe_status_t encode_layer(const moe_config_t* cfg, const moe_weight_list_t* wl,
                                 CUtensorMap* maps, const float** scales, bool encode = true,
                                 const float** gs = nullptr, float* act = nullptr) {
  if (cfg->wtype == MOE_DTYPE_NVFP4) return encode_layer_nvfp4(cfg, wl, maps, scales, gs, act, encode);
  const bool fp8 = cfg->wtype == MOE_DTYPE_FP8_E4M3;
  if (!wl->gate || !wl->up || !wl->down)
    return fail(MOE_ERR_INVALID_ARG, "gate/up/down pointer arrays must not be NULL");
  if (fp8 && (!wl->gate_scales || !wl->up_scales || !wl->down_scales))
    return fail(MOE_ERR_INVALID_ARG, "fp8 weights need gate/up/down scale pointer arrays");
  const int E = cfg->E;
  for (int e = 0; e < E; ++e) {
    char nm[64];
    snprintf(nm, sizeof nm, "gate[%d]", e);
    MOE_TRY(check_ptr(wl->gate[e], nm));
    snprintf(nm, sizeof nm, "up[%d]", e);
    MOE_TRY(check_ptr(wl->up[e], nm));
    snprintf(nm, sizeof nm, "down[%d]", e);
    MOE_TRY(check_ptr(wl->down[e], nm));
    if (fp8) {
      snprintf(nm, sizeof nm, "gate_scales[%d]", e);
      MOE_TRY(check_ptr4(wl->gate_scales[e], nm));
      snprintf(nm, sizeof nm, "up_scales[%d]", e);
      MOE_TRY(check_ptr4(wl->up_scales[e], nm));
      snprintf(nm, sizeof nm, "down_scales[%d]", e);
      MOE_TRY(check_ptr4(wl->down_scales[e], nm));
    }
  }
  const bool shared = cfg->I_shared > 0;
  if (shared) {
    MOE_TRY(check_ptr(wl->shared_gate, "shared_gate"));
    MOE_TRY(check_ptr(wl->shared_up, "shared_up"));
    MOE_TRY(check_ptr(wl->shared_down, "shared_down"));
    if (fp8) {
      MOE_TRY(check_ptr4(wl->shared_gate_scales, "shared_gate_scales"));
      MOE_TRY(check_ptr4(wl->shared_up_scales, "shared_up_scales"));
      MOE_TRY(check_ptr4(wl->shared_down_scales, "shared_down_scales"));
    }
  }
  if (!encode) return MOE_OK;  // checks only
  const int G = E + (shared ? 1 : 0);
  CUtensorMap* m1 = maps;
  CUtensorMap* m2 = maps + 2 * G;
  const uint64_t H = cfg->H, I = cfg->I, Is = cfg->I_shared;
  for (int g = 0; g < G; ++g) {
    const bool sh = g == E;
    const uint64_t inter = sh ? Is : I;
    const void* wg = sh ? wl->shared_gate : wl->gate[g];
    const void* wu = sh ? wl->shared_up : wl->up[g];
    const void* wd = sh ? wl->shared_down : wl->down[g];
    if (!fp8) {
      // bf16 pair tiles: each CTA loads 64 gate + 64 up rows, or 128 down rows
      MOE_TRY(encode_2d(&m1[2 * g], true, wg, H, inter, kTileK, kGemmBRows / 2));
      MOE_TRY(encode_2d(&m1[2 * g + 1], true, wu, H, inter, kTileK, kGemmBRows / 2));
      MOE_TRY(encode_2d(&m2[g], true, wd, inter, H, kTileK, kGemmBRows));
    } else {
      // fp8: 128 weight rows x 128 K bytes per box
      MOE_TRY(encode_2d(&m1[2 * g], false, wg, H, inter, 128, kFp8WRows));
      MOE_TRY(encode_2d(&m1[2 * g + 1], false, wu, H, inter, 128, kFp8WRows));
      MOE_TRY(encode_2d(&m2[g], false, wd, inter, H, 128, kFp8WRows));
      scales[2 * g] = sh ? wl->shared_gate_scales : wl->gate_scales[g];
      scales[2 * g + 1] = sh ? wl->shared_up_scales : wl->up_scales[g];
      scales[2 * G + g] = sh ? wl->shared_down_scales : wl->down_scales[g];
    }
  }

  return MOE_OK;
}

// NVFP4: GEMM1 descriptor of group g at 2g (the stacked gate/up codes, 2I x H/2
// bytes; 2g+1 repeats it), GEMM2 at 2G+g (down codes, H x I/2 bytes); boxes of
// 256 rows x 128 bytes.  scales[] hold the MMA-layout scale bytes, gs[] the
// tensor-scale pointers (same indexing); act[0..1] = g_x, g_h.
static moe_status_t encode_layer_nvfp4(const moe_config_t* cfg, const moe_weight_list_t* wl,
                                       CUtensorMap* maps, const float** scales, const float** gs,
                                       float* act, bool encode) {
  if (!wl->gate || !wl->down || !wl->gate_sf || !wl->down_sf || !wl->gate_tscale ||
      !wl->down_tscale)
    return fail(MOE_ERR_INVALID_ARG,
                "NVFP4 weights need gate, down, gate_sf, down_sf, gate_tscale and down_tscale arrays");
  if (!std::isfinite(wl->input_scale) || wl->input_scale <= 0.0f ||
      !std::isfinite(wl->hidden_scale) || wl->hidden_scale <= 0.0f)
    return fail(MOE_ERR_INVALID_ARG, "NVFP4 input_scale and hidden_scale must be finite and > 0");
  const int E = cfg->E;
  char nm[64];
  for (int e = 0; e < E; ++e) {
    snprintf(nm, sizeof nm, "gate[%d]", e);
    MOE_TRY(check_ptr(wl->gate[e], nm));
    snprintf(nm, sizeof nm, "down[%d]", e);
    MOE_TRY(check_ptr(wl->down[e], nm));
    snprintf(nm, sizeof nm, "gate_sf[%d]", e);
    MOE_TRY(check_ptr(wl->gate_sf[e], nm));
    snprintf(nm, sizeof nm, "down_sf[%d]", e);
    MOE_TRY(check_ptr(wl->down_sf[e], nm));
    snprintf(nm, sizeof nm, "gate_tscale[%d]", e);
    MOE_TRY(check_ptr4(wl->gate_tscale[e], nm));
    snprintf(nm, sizeof nm, "down_tscale[%d]", e);
    MOE_TRY(check_ptr4(wl->down_tscale[e], nm));
  }
  const bool shared = cfg->I_shared > 0;
  if (shared) {
    MOE_TRY(check_ptr(wl->shared_gate, "shared_gate"));
    MOE_TRY(check_ptr(wl->shared_down, "shared_down"));
    MOE_TRY(check_ptr(wl->shared_gate_sf, "shared_gate_sf"));
    MOE_TRY(check_ptr(wl->shared_down_sf, "shared_down_sf"));
    MOE_TRY(check_ptr4(wl->shared_gate_tscale, "shared_gate_tscale"));
    MOE_TRY(check_ptr4(wl->shared_down_tscale, "shared_down_tscale"));
  }
  if (!encode) return MOE_OK;
  const int G = E + (shared ? 1 : 0);
  CUtensorMap* m1 = maps;
  CUtensorMap* m2 = maps + 2 * G;
  const uint64_t H = cfg->H, I = cfg->I, Is = cfg->I_shared;
  for (int g = 0; g < G; ++g) {
    const bool sh = g == E;
    const uint64_t inter = sh ? Is : I;
    const void* wgu = sh ? wl->shared_gate : wl->gate[g];
    const void* wd = sh ? wl->shared_down : wl->down[g];
    MOE_TRY(encode_2d(&m1[2 * g], false, wgu, H / 2, 2 * inter, 128, 2 * kNvfp4Rows));
    m1[2 * g + 1] = m1[2 * g];
    MOE_TRY(encode_2d(&m2[g], false, wd, inter / 2, H, 128, 2 * kNvfp4Rows));
    scales[2 * g] = static_cast<const float*>(sh ? wl->shared_gate_sf : wl->gate_sf[g]);
    scales[2 * g + 1] = scales[2 * g];
    scales[2 * G + g] = static_cast<const float*>(sh ? wl->shared_down_sf : wl->down_sf[g]);
    gs[2 * g] = sh ? wl->shared_gate_tscale : wl->gate_tscale[g];
    gs[2 * g + 1] = gs[2 * g];
    gs[2 * G + g] = sh ? wl->shared_down_tscale : wl->down_tscale[g];
  }
  act[0] = wl->input_scale;
  act[1] = wl->hidden_scale;
  return MOE_OK;
}

moe_status_t moe_weights_create(const moe_config_t* cfg, const moe_weight_list_t* wl,
                                moe_weights_t* out) {
  MOE_TRY(check_config(cfg));
  if (!wl || !out) return fail(MOE_ERR_INVALID_ARG, "weights or out is NULL");
  *out = nullptr;
  const bool fp8 = cfg->wtype == MOE_DTYPE_FP8_E4M3;
  if (fp8 && (cfg->H / 128 > kFp8MaxKBlocks || cfg->I / 128 > kFp8MaxKBlocks ||
              cfg->I_shared / 128 > kFp8MaxKBlocks))
    return fail(MOE_ERR_UNSUPPORTED, "fp8 layers need H, I and I_shared <= %d",
                128 * kFp8MaxKBlocks);
  const bool fp4 = cfg->wtype == MOE_DTYPE_NVFP4;
  const int G = cfg->E + (cfg->I_shared > 0 ? 1 : 0);
  std::vector<CUtensorMap> maps(3 * G);
  std::vector<const float*> scales((fp8 || fp4) ? 3 * G : 0);
  std::vector<const float*> gs(fp4 ? 3 * G : 0);
  float act[2] = {0.0f, 0.0f};
  MOE_TRY(encode_layer(cfg, wl, maps.data(), scales.data(), true, gs.data(), act));
  // device table: maps [3G] | scale pointers [3G] | NVFP4: tensor-scale pointers [3G] | g_x, g_h
  void* table = nullptr;
  const size_t map_bytes = maps.size() * sizeof(CUtensorMap);
  const size_t sc_bytes = scales.size() * sizeof(const float*);
  const size_t gs_bytes = gs.size() * sizeof(const float*);
  const size_t act_bytes = fp4 ? sizeof(act) : 0;
  MOE_CUDA(cudaMalloc(&table, map_bytes + sc_bytes + gs_bytes + act_bytes));
  uint8_t* tb = static_cast<uint8_t*>(table);
  cudaError_t e = cudaMemcpy(tb, maps.data(), map_bytes, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && sc_bytes)
    e = cudaMemcpy(tb + map_bytes, scales.data(), sc_bytes, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && gs_bytes)
    e = cudaMemcpy(tb + map_bytes + sc_bytes, gs.data(), gs_bytes, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && act_bytes)
    e = cudaMemcpy(tb + map_bytes + sc_bytes + gs_bytes, act, act_bytes, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(table);
    return cuda_fail(e, "cudaMemcpy(weight table)");
  }
  moe_weights* w = new moe_weights;
  w->cfg = *cfg;
  w->device = current_device();
  w->table = table;
  w->maps1 = static_cast<CUtensorMap*>(table);
  w->maps2 = static_cast<CUtensorMap*>(table) + 2 * G;
  const float** sp = reinterpret_cast<const float**>(tb + map_bytes);
  w->scales1 = (fp8 || fp4) ? sp : nullptr;
  w->scales2 = (fp8 || fp4) ? sp + 2 * G : nullptr;
  const float** gp = reinterpret_cast<const float**>(tb + map_bytes + sc_bytes);
  w->gs1 = fp4 ? gp : nullptr;
  w->gs2 = fp4 ? gp + 2 * G : nullptr;
  w->act = fp4 ? reinterpret_cast<float*>(tb + map_bytes + sc_bytes + gs_bytes) : nullptr;
  *out = w;
  return MOE_OK;
}

moe_status_t moe_stack_create(const moe_config_t* cfg, int32_t num_layers,
                              const moe_weight_list_t* layers, const void* const* w_router,
                              const float* const* logit_bias, moe_stack_t* out) {
  MOE_TRY(check_config(cfg));
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (num_layers < 1) return fail(MOE_ERR_INVALID_ARG, "num_layers = %d", num_layers);
  if (!layers || !w_router) return fail(MOE_ERR_INVALID_ARG, "layers or w_router is NULL");
  const bool fp8 = cfg->wtype == MOE_DTYPE_FP8_E4M3;
  if (fp8 && (cfg->H / 128 > kFp8MaxKBlocks || cfg->I / 128 > kFp8MaxKBlocks ||
              cfg->I_shared / 128 > kFp8MaxKBlocks))
    return fail(MOE_ERR_UNSUPPORTED, "fp8 layers need H, I and I_shared <= %d",
                128 * kFp8MaxKBlocks);
  const int L = num_layers;
  const int G = cfg->E + (cfg->I_shared > 0 ? 1 : 0);
  const int E_pad = (cfg->E + 15) / 16 * 16;
  std::vector<CUtensorMap> maps(size_t(L) * 3 * G), router(L);
  std::vector<const float*> bias(L, nullptr);
  const bool fp4 = cfg->wtype == MOE_DTYPE_NVFP4;
  std::vector<const float*> scales((fp8 || fp4) ? size_t(L) * 3 * G : 0);
  std::vector<const float*> gs(fp4 ? size_t(L) * 3 * G : 0);
  std::vector<float> act(fp4 ? size_t(L) * 2 : 0);
  // every layer's arguments are checked before anything is encoded
  for (int l = 0; l < L; ++l) {
    MOE_TRY(encode_layer(cfg, &layers[l], nullptr, nullptr, false));
    char nm[48];
    snprintf(nm, sizeof nm, "w_router[%d]", l);
    MOE_TRY(check_ptr(w_router[l], nm));
    if (logit_bias && logit_bias[l]) {
      snprintf(nm, sizeof nm, "logit_bias[%d]", l);
      MOE_TRY(check_ptr4(logit_bias[l], nm));
      bias[l] = logit_bias[l];
    }
  }
  for (int l = 0; l < L; ++l) {
    MOE_TRY(encode_layer(cfg, &layers[l], maps.data() + size_t(l) * 3 * G,
                         (fp8 || fp4) ? scales.data() + size_t(l) * 3 * G : nullptr, true,
                         fp4 ? gs.data() + size_t(l) * 3 * G : nullptr,
                         fp4 ? act.data() + size_t(l) * 2 : nullptr));
    // boxes of E_pad / 2 router rows (the router kernel loads one or two per stage)
    MOE_TRY(encode_2d(&router[l], true, w_router[l], cfg->H, cfg->E, kTileK, E_pad / 2));
  }
  // device table: maps [L][3G] | router maps [L] | bias [L] | fp8 scales [L][3G]
  const size_t maps_b = maps.size() * sizeof(CUtensorMap);
  const size_t router_b = router.size() * sizeof(CUtensorMap);
  const size_t bias_b = bias.size() * sizeof(const float*);
  const size_t scales_b = scales.size() * sizeof(const float*);
  const size_t gs_b = gs.size() * sizeof(const float*);
  const size_t act_b = act.size() * sizeof(float);
  void* table = nullptr;
  MOE_CUDA(cudaMalloc(&table, maps_b + router_b + bias_b + scales_b + gs_b + act_b));
  uint8_t* tb = static_cast<uint8_t*>(table);
  cudaError_t e = cudaMemcpy(tb, maps.data(), maps_b, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(tb + maps_b, router.data(), router_b, cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(tb + maps_b + router_b, bias.data(), bias_b, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && scales_b)
    e = cudaMemcpy(tb + maps_b + router_b + bias_b, scales.data(), scales_b, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && gs_b)
    e = cudaMemcpy(tb + maps_b + router_b + bias_b + scales_b, gs.data(), gs_b,
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess && act_b)
    e = cudaMemcpy(tb + maps_b + router_b + bias_b + scales_b + gs_b, act.data(), act_b,
                   cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(table);
    return cuda_fail(e, "cudaMemcpy(stack table)");
  }
  moe_stack* st = new moe_stack;
  st->cfg = *cfg;
  st->device = current_device();
  st->num_layers = L;
  st->G = G;
  st->table = table;
  st->maps = reinterpret_cast<CUtensorMap*>(tb);
  st->router = reinterpret_cast<CUtensorMap*>(tb + maps_b);
  st->bias = reinterpret_cast<const float**>(tb + maps_b + router_b);
  st->scales = (fp8 || fp4) ? reinterpret_cast<const float**>(tb + maps_b + router_b + bias_b)
                            : nullptr;
  st->gs = fp4 ? reinterpret_cast<const float**>(tb + maps_b + router_b + bias_b + scales_b)
               : nullptr;
  st->act = fp4 ? reinterpret_cast<float*>(tb + maps_b + router_b + bias_b + scales_b + gs_b)
                : nullptr;
  *out = st;
  return MOE_OK;
}

void moe_stack_destroy(moe_stack_t st) {
  if (!st) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(st->device);
  cudaDeviceSynchronize();
  cudaFree(st->table);
  cudaSetDevice(prev);
  delete st;
}

void moe_weights_destroy(moe_weights_t w) {
  if (!w) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(w->device);
  cudaDeviceSynchronize();
  cudaFree(w->table);
  cudaSetDevice(prev);
  delete w;
}

}  // extern "C"

// ======================================================================== steps
namespace moe {

static moe_status_t run_route(const moe_config_t& c, const void* x, const void* w_router,
                              const float* bias, int32_t* ids, float* w, float* logits,
                              uint32_t* err, cudaStream_t st, const RouterTable* table = nullptr) {
  const int E_pad = (c.E + 15) / 16 * 16;
  CUtensorMap mx, mw;
  MOE_TRY(encode_2d(&mx, true, x, c.H, c.T, kTileK, kTileM));
  if (table) mw = mx;  // unused: the kernel reads the layer's descriptor from the table
  // boxes of E_pad / 2 router rows (the router kernel loads one or two per stage)
  else MOE_TRY(encode_2d(&mw, true, w_router, c.H, c.E, kTileK, E_pad / 2));
  trace_mark(st, MOE_K_ROUTER);
  MOE_CUDA(launch_router(mx, mw, c.T, c.H, c.E, E_pad, c.k, c.score, c.renormalize, c.route_scale,
                         bias, ids, w, logits, err, sm_count(), st, table));
  return MOE_OK;
}

static moe_status_t run_permute(const moe_config_t& c, const Layout& L, void* ws, const int32_t* ids,
                                const float* topk_w, const void* x, int32_t* counts,
                                int32_t* offsets, int32_t* perm_token, int32_t* inv_row,
                                float* row_weight, void* x_perm, float* x_perm_scales,
                                cudaStream_t st) {
  uint32_t* err = err_word(ws);
  const int nblk = static_cast<int>((c.T + kPermTok - 1) / kPermTok);
  int32_t* blk_counts = at<int32_t*>(ws, L.blk_counts);
  int32_t* blk_base = at<int32_t*>(ws, L.blk_base);
  trace_mark(st, MOE_K_HIST);
  MOE_CUDA(launch_hist(ids, c.T, c.k, c.E, blk_counts, err, st));
  trace_mark(st, MOE_K_SCAN);
  MOE_CUDA(launch_scan(blk_counts, nblk, c.E, blk_base, counts, offsets, st));
  trace_mark(st, MOE_K_SCATTER);
  MOE_CUDA(launch_scatter(ids, topk_w, x, c.T, c.k, c.E, c.H, c.wtype == MOE_DTYPE_FP8_E4M3,
                          blk_base, offsets, perm_token, inv_row, row_weight, x_perm,
                          x_perm_scales, err, st));
  return MOE_OK;
}

// bf16 grouped FFN.  GEMM1's routed rows come from x_perm (tile loads) or,
// when gather_rows (row -> token) is given, straight from the unpermuted
// tokens x_perm = x by TMA row gathers (the permuted copy is never written).
static moe_status_t run_ffn(const moe_config_t& c, const WeightView& W, const Layout& L, void* ws,
                            const void* x_perm, const int32_t* offsets, const float* row_weight,
                            const void* x_shared, void* y_perm, void* shared_out,
                            cudaStream_t st, const int32_t* gather_rows = nullptr,
                            float* y_scales = nullptr, float* shared_scales = nullptr) {
  uint32_t* err = err_word(ws);
  const bool shared = c.I_shared > 0 && x_shared != nullptr;
  const int64_t R = c.T * c.k;
  int32_t* s1 = at<int32_t*>(ws, L.sched1);
  int32_t* s2 = at<int32_t*>(ws, L.sched2);
  __nv_bfloat16* h = at<__nv_bfloat16*>(ws, L.h);
  __nv_bfloat16* hs = at<__nv_bfloat16*>(ws, L.hs);
  const int n1r = c.I / kGemm1TileN, n1s = c.I_shared / kGemm1TileN;
  const int n2 = (c.H + kGemm2TileN - 1) / kGemm2TileN;
  CUtensorMap a0, a1, b0, b1;
  if (gather_rows) MOE_TRY(encode_2d(&a0, true, x_perm, c.H, c.T, kTileK, 1));
  else MOE_TRY(encode_2d(&a0, true, x_perm, c.H, R, kTileK, kTileM));
  if (shared) MOE_TRY(encode_2d(&a1, true, x_shared, c.H, c.T, kTileK, kTileM));
  else a1 = a0;
  MOE_TRY(encode_2d(&b0, true, h, c.I, R, kTileK, kTileM));
  if (shared) MOE_TRY(encode_2d(&b1, true, hs, c.I_shared, c.T, kTileK, kTileM));
  else b1 = b0;
  // the plan kernel also writes each expert's A maps of both GEMMs with the row
  // extent cut at the end of its rows (zeros past it; GemmArgs::amap); not on
  // the fused-dispatch path, whose GEMM1 gathers rows from x
  uint8_t* cut = (L.amap && !gather_rows) ? at<uint8_t*>(ws, L.amap) : nullptr;
  trace_mark(st, MOE_K_PLAN);
  MOE_CUDA(launch_plan(offsets, c.E, shared ? 1 : 0, c.T, n1r, n1s, n2, n2, s1, s2, kGemmTileRows,
                       kGemmTileRows, st, &a0, &b0, cut, R));

  GemmArgs g1{};
  g1.b_maps = W.maps1;
  g1.layer = W.layer;
  g1.layer_stride = W.stride;
  g1.num_layers = W.num_layers;
  g1.offsets = offsets;
  g1.sched = s1;
  g1.out0 = h;
  g1.out1 = hs;
  g1.row_weight = nullptr;
  g1.gather_rows = gather_rows;
  g1.err = err;
  g1.R = static_cast<int32_t>(R);
  g1.E = c.E;
  g1.has_shared = shared ? 1 : 0;
  g1.T = static_cast<int32_t>(c.T);
  g1.K_routed = c.H;
  g1.K_shared = c.H;
  g1.N_routed = c.I;
  g1.N_shared = c.I_shared;
  g1.stall_test = take_gemm1_stall() ? 1 : 0;
  g1.amap = cut;
  const int grid = gemm_grid();
  trace_mark(st, MOE_K_GEMM1);
  MOE_CUDA(launch_grouped_gemm(true, a0, a1, g1, grid, st));

  GemmArgs g2 = g1;
  g2.amap = cut ? cut + size_t(c.E) * 128 : nullptr;
  g2.stall_test = 0;
  g2.gather_rows = nullptr;
  g2.b_maps = W.maps2;
  g2.sched = s2;
  g2.out0 = y_perm;
  g2.out1 = shared_out;
  g2.out_scales0 = y_scales;  // non-null: fp16 y with power-of-two scales
  g2.out_scales1 = shared_scales;
  g2.row_weight = row_weight;
  g2.K_routed = c.I;
  g2.K_shared = c.I_shared;
  g2.N_routed = c.H;
  g2.N_shared = c.H;
  trace_mark(st, MOE_K_GEMM2);
  MOE_CUDA(launch_grouped_gemm(false, b0, b1, g2, grid, st));
  return MOE_OK;
}

// fp8: e4m3 rows (x_perm, x_shared) with 1x128 scales -> GEMM1 (e4m3 h + scales
// in the workspace) -> GEMM2 (fp32 y_perm / shared_out).
static moe_status_t run_ffn_fp8(const moe_config_t& c, const WeightView& W, const Layout& L,
                                void* ws, const void* x_perm, const float* x_perm_scales,
                                const int32_t* offsets, const float* row_weight,
                                const void* x_shared, const float* x_shared_scales, void* y_perm,
                                void* shared_out, cudaStream_t st) {
  uint32_t* err = err_word(ws);
  const bool shared = c.I_shared > 0 && x_shared != nullptr;
  const int64_t R = c.T * c.k;
  int32_t* s1 = at<int32_t*>(ws, L.sched1);
  int32_t* s2 = at<int32_t*>(ws, L.sched2);
  uint8_t* h = at<uint8_t*>(ws, L.h);
  uint8_t* hs = at<uint8_t*>(ws, L.hs);
  float* h_sc = at<float*>(ws, L.h_sc);
  float* hs_sc = at<float*>(ws, L.hs_sc);
  // GEMM1 tiles: 128 intermediate columns (gate + up); GEMM2 tiles: 256 output columns
  const int n1r = c.I / kFp8WRows, n1s = c.I_shared / kFp8WRows;
  const int n2 = (c.H + 2 * kFp8WRows - 1) / (2 * kFp8WRows);
  trace_mark(st, MOE_K_PLAN);
  MOE_CUDA(launch_plan(offsets, c.E, shared ? 1 : 0, c.T, n1r, n1s, n2, n2, s1, s2,
                       kFp8Tile1Tokens, kFp8Tile2Tokens, st));
  const int grid = sm_count();
  // token rows: 32 rows x 128 bytes per box
  CUtensorMap t0, t1;
  MOE_TRY(encode_2d(&t0, false, x_perm, c.H, R, 128, 32));
  if (shared) MOE_TRY(encode_2d(&t1, false, x_shared, c.H, c.T, 128, 32));
  else t1 = t0;
  Fp8GemmArgs g1{};
  g1.w_maps = W.maps1;
  g1.w_scales = W.scales1;
  g1.layer = W.layer;
  g1.layer_stride = W.stride;
  g1.num_layers = W.num_layers;
  g1.offsets = offsets;
  g1.sched = s1;
  g1.tok_scales0 = x_perm_scales;
  g1.tok_scales1 = shared ? x_shared_scales : x_perm_scales;
  g1.out0 = h;
  g1.out1 = hs;
  g1.out_scales0 = h_sc;
  g1.out_scales1 = hs_sc;
  g1.row_weight = nullptr;
  g1.err = err;
  g1.E = c.E;
  g1.has_shared = shared ? 1 : 0;
  g1.T = static_cast<int32_t>(c.T);
  g1.K_routed = c.H;
  g1.K_shared = c.H;
  g1.N_routed = c.I;
  g1.N_shared = c.I_shared;
  trace_mark(st, MOE_K_GEMM1);
  MOE_CUDA(launch_grouped_gemm_fp8(true, t0, t1, g1, grid, st));

  CUtensorMap u0, u1;
  MOE_TRY(encode_2d(&u0, false, h, c.I, R, 128, 32));
  if (shared) MOE_TRY(encode_2d(&u1, false, hs, c.I_shared, c.T, 128, 32));
  else u1 = u0;
  Fp8GemmArgs g2 = g1;
  g2.w_maps = W.maps2;
  g2.w_scales = W.scales2;
  g2.sched = s2;
  g2.tok_scales0 = h_sc;
  g2.tok_scales1 = shared ? hs_sc : h_sc;
  g2.out0 = y_perm;
  g2.out1 = shared_out;
  g2.out_scales0 = nullptr;
  g2.out_scales1 = nullptr;
  g2.row_weight = row_weight;
  g2.K_routed = c.I;
  g2.K_shared = c.I_shared;
  g2.N_routed = c.H;
  g2.N_shared = c.H;
  trace_mark(st, MOE_K_GEMM2);
  MOE_CUDA(launch_grouped_gemm_fp8(false, u0, u1, g2, grid, st));
  return MOE_OK;
}

// NVFP4 permuted activations: the 128-row-padded expert segments and the
// token-order copy for the shared expert (codes + MMA-layout scales each).
struct Nvfp4Acts {
  int32_t* pad_offsets;  // [E+1]
  uint8_t* x;            // [Rp, H/2]
  uint8_t* x_sf;         // Rp * H/16 bytes
  uint8_t* xs;           // [Tp, H/2] or null
  uint8_t* xs_sf;
};

// NVFP4 permutation: histogram, scan (with the 128-row padded offsets) and the
// quantising scatter.
static moe_status_t run_permute_nvfp4(const moe_config_t& c, const WeightView& W,
                                      int32_t* blk_counts, int32_t* blk_base, uint32_t* err,
                                      const void* x, const int32_t* ids, const float* topk_w,
                                      int32_t* counts, int32_t* offsets, int32_t* perm_token,
                                      int32_t* inv_row, float* row_weight, const Nvfp4Acts& A,
                                      cudaStream_t st) {
  const int nblk = static_cast<int>((c.T + kPermTok - 1) / kPermTok);
  trace_mark(st, MOE_K_HIST);
  MOE_CUDA(launch_hist(ids, c.T, c.k, c.E, blk_counts, err, st));
  trace_mark(st, MOE_K_SCAN);
  MOE_CUDA(launch_scan(blk_counts, nblk, c.E, blk_base, counts, offsets, st, A.pad_offsets));
  Nvfp4Scatter q{};
  q.pad_offsets = A.pad_offsets;
  q.act_scales = W.act;
  q.layer = W.layer;
  q.num_layers = W.num_layers;
  q.rows_pad = nvfp4_rows(c);
  q.x_codes = A.x;
  q.x_sf = A.x_sf;
  q.xs_codes = A.xs;
  q.xs_sf = A.xs_sf;
  trace_mark(st, MOE_K_SCATTER);
  MOE_CUDA(launch_scatter_nvfp4(ids, topk_w, x, c.T, c.k, c.E, c.H, blk_base, offsets, perm_token,
                                inv_row, row_weight, q, err, st));
  return MOE_OK;
}

// NVFP4 expert FFN: the tile plan, GEMM1 (NVFP4 h + scales in the workspace)
// and GEMM2 (fp16 y with power-of-two scales per 32 columns, unpadded rows).
// A.xs null: no shared-expert group.
static moe_status_t run_ffn_nvfp4(const moe_config_t& c, const WeightView& W, const Layout& L,
                                  void* ws, const int32_t* offsets, const Nvfp4Acts& A,
                                  const float* row_weight, void* y, float* y_sc, void* shared_out,
                                  float* sh_sc, cudaStream_t st) {
  uint32_t* err = err_word(ws);
  const bool shared = c.I_shared > 0 && A.xs != nullptr;
  const int64_t R = c.T * c.k;
  const int64_t Rp = nvfp4_rows(c), Tp = nvfp4_tokens(c);
  int32_t* s1 = at<int32_t*>(ws, L.sched1);
  int32_t* s2 = at<int32_t*>(ws, L.sched2);
  uint8_t* h = at<uint8_t*>(ws, L.h);
  uint8_t* hs = at<uint8_t*>(ws, L.hs);
  uint8_t* h_sf = at<uint8_t*>(ws, L.h_sc);
  uint8_t* hs_sf = at<uint8_t*>(ws, L.hs_sc);
  // GEMM1 tiles: 128 h columns (256 stacked gate/up rows); GEMM2 tiles: 256 y columns
  const int n1r = c.I / 128, n1s = c.I_shared / 128, n2 = c.H / 256;
  trace_mark(st, MOE_K_PLAN);
  MOE_CUDA(launch_plan(offsets, c.E, shared ? 1 : 0, c.T, n1r, n1s, n2, n2, s1, s2, kNvfp4Rows,
                       kNvfp4Rows, st));
  const int grid = sm_count();
  CUtensorMap a0, a1;
  MOE_TRY(encode_2d(&a0, false, A.x, c.H / 2, Rp, 128, kNvfp4Rows));
  if (shared) MOE_TRY(encode_2d(&a1, false, A.xs, c.H / 2, Tp, 128, kNvfp4Rows));
  else a1 = a0;
  Nvfp4GemmArgs g1{};
  g1.w_maps = W.maps1;
  g1.w_sf = reinterpret_cast<const uint8_t* const*>(W.scales1);
  g1.w_gs = W.gs1;
  g1.act_scales = W.act;
  g1.layer = W.layer;
  g1.layer_stride = W.stride;
  g1.num_layers = W.num_layers;
  g1.offsets = offsets;
  g1.pad_offsets = A.pad_offsets;
  g1.sched = s1;
  g1.a_sf0 = A.x_sf;
  g1.a_sf1 = shared ? A.xs_sf : A.x_sf;
  g1.out0 = h;
  g1.out1 = hs;
  g1.out_sf0 = h_sf;
  g1.out_sf1 = hs_sf;
  g1.err = err;
  g1.E = c.E;
  g1.has_shared = shared ? 1 : 0;
  g1.T = static_cast<int32_t>(c.T);
  g1.K_routed = c.H;
  g1.K_shared = c.H;
  g1.N_routed = c.I;
  g1.N_shared = c.I_shared;
  trace_mark(st, MOE_K_GEMM1);
  MOE_CUDA(launch_grouped_gemm_nvfp4(true, a0, a1, a0, a1, g1, grid, st));  // no y maps

  CUtensorMap b0, b1;
  MOE_TRY(encode_2d(&b0, false, h, c.I / 2, Rp, 128, kNvfp4Rows));
  if (shared) MOE_TRY(encode_2d(&b1, false, hs, c.I_shared / 2, Tp, 128, kNvfp4Rows));
  else b1 = b0;
  Nvfp4GemmArgs g2 = g1;
  g2.w_maps = W.maps2;
  g2.w_sf = reinterpret_cast<const uint8_t* const*>(W.scales2);
  g2.w_gs = W.gs2;
  g2.sched = s2;
  g2.a_sf0 = h_sf;
  g2.a_sf1 = shared ? hs_sf : h_sf;
  g2.out0 = y;
  g2.out1 = shared_out;
  g2.out_sf0 = nullptr;
  g2.out_sf1 = nullptr;
  g2.out_scales0 = y_sc;
  g2.out_scales1 = sh_sc;
  g2.row_weight = row_weight;
  g2.K_routed = c.I;
  g2.K_shared = c.I_shared;
  g2.N_routed = c.H;
  g2.N_shared = c.H;
  // fp16 y and shared output for GEMM2's TMA stores: 32-row x 64-column boxes
  // (the 2-byte element type only sets the element size; the bits are copied)
  CUtensorMap y0, y1;
  MOE_TRY(encode_2d(&y0, true, y, c.H, R, 64, 32));
  if (shared) MOE_TRY(encode_2d(&y1, true, shared_out, c.H, c.T, 64, 32));
  else y1 = y0;
  trace_mark(st, MOE_K_GEMM2);
  MOE_CUDA(launch_grouped_gemm_nvfp4(false, b0, b1, y0, y1, g2, grid, st));
  return MOE_OK;
}

// The whole NVFP4 permutation + expert FFN of the layer forward, in the workspace.
static moe_status_t run_nvfp4(const moe_config_t& c, const WeightView& W, const Layout& L, void* ws,
                              const void* x, const int32_t* ids, const float* topk_w,
                              int32_t* counts, int32_t* offsets, int32_t* perm_token,
                              int32_t* inv_row, float* row_weight, void* y, float* y_sc,
                              void* shared_out, float* sh_sc, cudaStream_t st) {
  const bool shared = c.I_shared > 0;
  Nvfp4Acts A;
  A.pad_offsets = at<int32_t*>(ws, L.pad_offsets);
  A.x = at<uint8_t*>(ws, L.x_perm);
  A.x_sf = at<uint8_t*>(ws, L.x_perm_sc);
  A.xs = shared ? at<uint8_t*>(ws, L.xq) : nullptr;
  A.xs_sf = shared ? at<uint8_t*>(ws, L.xq_sc) : nullptr;
  MOE_TRY(run_permute_nvfp4(c, W, at<int32_t*>(ws, L.blk_counts), at<int32_t*>(ws, L.blk_base),
                            err_word(ws), x, ids, topk_w, counts, offsets, perm_token, inv_row,
                            row_weight, A, st));
  return run_ffn_nvfp4(c, W, L, ws, offsets, A, row_weight, y, y_sc, shared_out, sh_sc, st);
}

static bool same_shape(const moe_config_t& a, const moe_config_t& b) {
  return a.H == b.H && a.E == b.E && a.I == b.I && a.I_shared == b.I_shared && a.wtype == b.wtype;
}

// The layer forward after validation: route (one router matrix, or a stack's
// router table), permute, grouped FFN over the view's descriptors, combine.
static moe_status_t forward_impl(const moe_config_t* cfg, const WeightView& W, const void* x,
                                 const void* w_router, const float* logit_bias,
                                 const RouterTable* rt, void* out, int32_t* topk_ids_out,
                                 float* topk_w_out, uint32_t flags, void* ws,
                                 moe_stream_t stream) {
  const bool fp8 = cfg->wtype == MOE_DTYPE_FP8_E4M3;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Layout L = layout(*cfg, MOE_OP_FORWARD);
  uint32_t* err = err_word(ws);
  int32_t* ids = topk_ids_out ? topk_ids_out : at<int32_t*>(ws, L.ids);
  float* w = topk_w_out ? topk_w_out : at<float*>(ws, L.w);
  int32_t* counts = at<int32_t*>(ws, L.counts);
  int32_t* offsets = at<int32_t*>(ws, L.offsets);
  int32_t* perm_token = at<int32_t*>(ws, L.perm_token);
  int32_t* inv_row = at<int32_t*>(ws, L.inv_row);
  float* row_weight = at<float*>(ws, L.row_weight);
  const bool fused = (flags & MOE_FORWARD_FUSED_DISPATCH) && !fp8;
  void* x_perm = at<void*>(ws, L.x_perm);
  void* y_perm = at<void*>(ws, L.y_perm);
  void* shared_out = cfg->I_shared > 0 ? at<void*>(ws, L.shared_out) : nullptr;

  MOE_TRY(run_route(*cfg, x, w_router, logit_bias, ids, w, nullptr, err, st, rt));
  const int64_t R = cfg->T * cfg->k;
  if (cfg->wtype == MOE_DTYPE_NVFP4) {
    // expert and shared outputs as fp16 + power-of-two scales, as for bf16 layers
    float* y_sc = reinterpret_cast<float*>(static_cast<uint8_t*>(y_perm) + size_t(R) * cfg->H * 2);
    float* sh_sc = shared_out ? reinterpret_cast<float*>(static_cast<uint8_t*>(shared_out) +
                                                         size_t(cfg->T) * cfg->H * 2)
                              : nullptr;
    MOE_TRY(run_nvfp4(*cfg, W, L, ws, x, ids, w, counts, offsets, perm_token, inv_row, row_weight,
                      y_perm, y_sc, shared_out, sh_sc, st));
    trace_mark(st, MOE_K_COMBINE);
    MOE_CUDA(launch_combine_half(y_perm, y_sc, inv_row, shared_out, sh_sc, out, cfg->T, cfg->k,
                                 cfg->H, R, err, st));
    trace_mark(st, -1);
    return MOE_OK;
  }
  float* x_perm_sc = fp8 ? at<float*>(ws, L.x_perm_sc) : nullptr;
  MOE_TRY(run_permute(*cfg, L, ws, ids, w, x, counts, offsets, perm_token, inv_row, row_weight,
                      fused ? nullptr : x_perm, x_perm_sc, st));
  // bf16 layers keep y and the shared output as fp16 with a power-of-two
  // scale per 32 columns, inside the fp32-sized workspace regions: the
  // scales follow the fp16 rows
  float* y_sc = fp8 ? nullptr : reinterpret_cast<float*>(static_cast<uint8_t*>(y_perm) +
                                                         size_t(R) * cfg->H * 2);
  float* sh_sc = (fp8 || !shared_out) ? nullptr
                                      : reinterpret_cast<float*>(static_cast<uint8_t*>(shared_out) +
                                                                 size_t(cfg->T) * cfg->H * 2);
  if (fused) {
    // fused dispatch: GEMM1 gathers each expert's rows from x by token index
    MOE_TRY(run_ffn(*cfg, W, L, ws, x, offsets, row_weight, x, y_perm, shared_out, st,
                    perm_token, y_sc, sh_sc));
  } else if (!fp8) {
    MOE_TRY(run_ffn(*cfg, W, L, ws, x_perm, offsets, row_weight, x, y_perm, shared_out, st,
                    nullptr, y_sc, sh_sc));
  } else {
    // the shared expert reads every token: quantise x once more, unpermuted
    uint8_t* xq = cfg->I_shared > 0 ? at<uint8_t*>(ws, L.xq) : nullptr;
    float* xq_sc = cfg->I_shared > 0 ? at<float*>(ws, L.xq_sc) : nullptr;
    if (xq) {
      trace_mark(st, MOE_K_QUANT);
      MOE_CUDA(launch_quant_act_fp8(x, cfg->T, cfg->H, xq, xq_sc, st));
    }
    MOE_TRY(run_ffn_fp8(*cfg, W, L, ws, x_perm, x_perm_sc, offsets, row_weight, xq, xq_sc,
                        y_perm, shared_out, st));
  }
  trace_mark(st, MOE_K_COMBINE);
  if (fp8)
    MOE_CUDA(launch_combine(y_perm, inv_row, shared_out, out, cfg->T, cfg->k, cfg->H, R, err, st));
  else
    MOE_CUDA(launch_combine_half(y_perm, y_sc, inv_row, shared_out, sh_sc, out, cfg->T, cfg->k,
                                 cfg->H, R, err, st));
  trace_mark(st, -1);
  return MOE_OK;
}


}  // namespace moe

extern "C" {

moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* w_router,
                       const float* logit_bias, int32_t* topk_ids, float* topk_w,
                       float* logits_out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  MOE_TRY(check_ws(*cfg, MOE_OP_ROUTE, ws, ws_bytes));
  if (cfg->T == 0) return MOE_OK;
  MOE_TRY(check_ptr(x, "x"));
  MOE_TRY(check_ptr(w_router, "w_router"));
  MOE_TRY(check_ptr4(topk_ids, "topk_ids"));
  MOE_TRY(check_ptr4(topk_w, "topk_w"));
  if (logit_bias) MOE_TRY(check_ptr4(logit_bias, "logit_bias"));
  if (logits_out) MOE_TRY(check_ptr(logits_out, "logits_out"));
  if (logits_out && cfg->E % 4)
    return fail(MOE_ERR_UNSUPPORTED, "logits_out needs E to be a multiple of 4");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const moe_status_t s = run_route(*cfg, x, w_router, logit_bias, topk_ids, topk_w, logits_out,
                                   err_word(ws), st);
  trace_mark(st, -1);
  return s;
}

moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_ids, const float* topk_w,
                         const void* x, int32_t* expert_counts, int32_t* expert_offsets,
                         int32_t* perm_token, int32_t* inv_row, float* row_weight, void* x_perm,
                         float* x_perm_scales, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->wtype == MOE_DTYPE_NVFP4)
    return fail(MOE_ERR_UNSUPPORTED, "NVFP4 layers permute through moe_permute_nvfp4");
  MOE_TRY(check_ws(*cfg, MOE_OP_PERMUTE, ws, ws_bytes));
  MOE_TRY(check_ptr4(expert_counts, "expert_counts"));
  MOE_TRY(check_ptr4(expert_offsets, "expert_offsets"));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cfg->T == 0) {
    MOE_CUDA(cudaMemsetAsync(expert_counts, 0, size_t(cfg->E) * 4, st));
    MOE_CUDA(cudaMemsetAsync(expert_offsets, 0, size_t(cfg->E + 1) * 4, st));
    return MOE_OK;
  }
  MOE_TRY(check_ptr4(topk_ids, "topk_ids"));
  MOE_TRY(check_ptr4(perm_token, "perm_token"));
  MOE_TRY(check_ptr4(inv_row, "inv_row"));
  if (row_weight) {
    MOE_TRY(check_ptr4(row_weight, "row_weight"));
    if (!topk_w) return fail(MOE_ERR_INVALID_ARG, "row_weight needs topk_w");
    MOE_TRY(check_ptr4(topk_w, "topk_w"));
  }
  if (x_perm) {
    MOE_TRY(check_ptr(x, "x"));
    MOE_TRY(check_ptr(x_perm, "x_perm"));
    if (cfg->wtype == MOE_DTYPE_FP8_E4M3) MOE_TRY(check_ptr4(x_perm_scales, "x_perm_scales"));
  }
  Layout L = layout(*cfg, MOE_OP_PERMUTE);
  const moe_status_t s = run_permute(*cfg, L, ws, topk_ids, topk_w, x, expert_counts,
                                     expert_offsets, perm_token, inv_row, row_weight, x_perm,
                                     x_perm_scales, st);
  trace_mark(st, -1);
  return s;
}

moe_status_t moe_grouped_ffn(const moe_config_t* cfg, moe_weights_t weights, const void* x_perm,
                             const float* x_perm_scales, const int32_t* expert_offsets,
                             const float* row_weight, const void* x_shared,
                             const float* x_shared_scales, void* y_perm, void* shared_out,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->wtype == MOE_DTYPE_NVFP4)
    return fail(MOE_ERR_UNSUPPORTED, "NVFP4 layers run their experts through moe_grouped_ffn_nvfp4");
  MOE_TRY(check_ws(*cfg, MOE_OP_GROUPED_FFN, ws, ws_bytes));
  if (!weights) return fail(MOE_ERR_INVALID_ARG, "weights is NULL");
  if (!same_shape(weights->cfg, *cfg))
    return fail(MOE_ERR_INVALID_ARG, "weights were created for a different layer shape");
  const bool fp8 = cfg->wtype == MOE_DTYPE_FP8_E4M3;
  if (cfg->T == 0) return MOE_OK;
  if (fp8) {
    MOE_TRY(check_ptr4(x_perm_scales, "x_perm_scales"));
    if (x_shared && cfg->I_shared > 0) MOE_TRY(check_ptr4(x_shared_scales, "x_shared_scales"));
  }
  MOE_TRY(check_ptr(x_perm, "x_perm"));
  MOE_TRY(check_ptr4(expert_offsets, "expert_offsets"));
  MOE_TRY(check_ptr(y_perm, "y_perm"));
  if (row_weight) MOE_TRY(check_ptr4(row_weight, "row_weight"));
  if (x_shared && cfg->I_shared > 0) {
    MOE_TRY(check_ptr(x_shared, "x_shared"));
    MOE_TRY(check_ptr(shared_out, "shared_out"));
  }
  Layout L = layout(*cfg, MOE_OP_GROUPED_FFN);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const void* xs = cfg->I_shared > 0 ? x_shared : nullptr;
  const moe_status_t s =
      fp8 ? run_ffn_fp8(*cfg, view_of(weights), L, ws, x_perm, x_perm_scales, expert_offsets, row_weight,
                        xs, x_shared_scales, y_perm, shared_out, st)
          : run_ffn(*cfg, view_of(weights), L, ws, x_perm, expert_offsets, row_weight, xs, y_perm,
                    shared_out, st);
  trace_mark(st, -1);
  return s;
}

moe_status_t moe_nvfp4_rows(const moe_config_t* cfg, int64_t* padded_rows, int64_t* padded_tokens) {
  MOE_TRY(check_config(cfg));
  if (cfg->wtype != MOE_DTYPE_NVFP4) return fail(MOE_ERR_INVALID_ARG, "not an NVFP4 layer");
  if (padded_rows) *padded_rows = nvfp4_rows(*cfg);
  if (padded_tokens) *padded_tokens = nvfp4_tokens(*cfg);
  return MOE_OK;
}

moe_status_t moe_permute_nvfp4(const moe_config_t* cfg, moe_weights_t weights,
                               const int32_t* topk_ids, const float* topk_w, const void* x,
                               int32_t* expert_counts, int32_t* expert_offsets,
                               int32_t* pad_offsets, int32_t* perm_token, int32_t* inv_row,
                               float* row_weight, uint8_t* x_perm, uint8_t* x_perm_sf,
                               uint8_t* x_tok, uint8_t* x_tok_sf, void* ws, size_t ws_bytes,
                               moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->wtype != MOE_DTYPE_NVFP4)
    return fail(MOE_ERR_INVALID_ARG, "moe_permute_nvfp4 takes NVFP4 layers only");
  MOE_TRY(check_ws(*cfg, MOE_OP_PERMUTE, ws, ws_bytes));
  if (!weights) return fail(MOE_ERR_INVALID_ARG, "weights is NULL");
  if (!same_shape(weights->cfg, *cfg))
    return fail(MOE_ERR_INVALID_ARG, "weights were created for a different layer shape");
  MOE_TRY(check_ptr4(expert_counts, "expert_counts"));
  MOE_TRY(check_ptr4(expert_offsets, "expert_offsets"));
  MOE_TRY(check_ptr4(pad_offsets, "pad_offsets"));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cfg->T == 0) {
    MOE_CUDA(cudaMemsetAsync(expert_counts, 0, size_t(cfg->E) * 4, st));
    MOE_CUDA(cudaMemsetAsync(expert_offsets, 0, size_t(cfg->E + 1) * 4, st));
    MOE_CUDA(cudaMemsetAsync(pad_offsets, 0, size_t(cfg->E + 1) * 4, st));
    return MOE_OK;
  }
  MOE_TRY(check_ptr4(topk_ids, "topk_ids"));
  MOE_TRY(check_ptr(x, "x"));
  MOE_TRY(check_ptr4(perm_token, "perm_token"));
  MOE_TRY(check_ptr4(inv_row, "inv_row"));
  if (row_weight) {
    MOE_TRY(check_ptr4(row_weight, "row_weight"));
    if (!topk_w) return fail(MOE_ERR_INVALID_ARG, "row_weight needs topk_w");
    MOE_TRY(check_ptr4(topk_w, "topk_w"));
  }
  MOE_TRY(check_ptr(x_perm, "x_perm"));
  MOE_TRY(check_ptr(x_perm_sf, "x_perm_sf"));
  if (x_tok) MOE_TRY(check_ptr(x_tok_sf, "x_tok_sf"));
  if (x_tok) MOE_TRY(check_ptr(x_tok, "x_tok"));
  const Layout L = layout(*cfg, MOE_OP_PERMUTE);
  Nvfp4Acts A{pad_offsets, x_perm, x_perm_sf, x_tok, x_tok ? x_tok_sf : nullptr};
  const moe_status_t s = run_permute_nvfp4(
      *cfg, view_of(weights), at<int32_t*>(ws, L.blk_counts), at<int32_t*>(ws, L.blk_base),
      err_word(ws), x, topk_ids, topk_w, expert_counts, expert_offsets, perm_token, inv_row,
      row_weight, A, st);
  trace_mark(st, -1);
  return s;
}

moe_status_t moe_grouped_ffn_nvfp4(const moe_config_t* cfg, moe_weights_t weights,
                                   const uint8_t* x_perm, const uint8_t* x_perm_sf,
                                   const int32_t* expert_offsets, const int32_t* pad_offsets,
                                   const float* row_weight, const uint8_t* x_tok,
                                   const uint8_t* x_tok_sf, float* y_perm, float* shared_out,
                                   void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->wtype != MOE_DTYPE_NVFP4)
    return fail(MOE_ERR_INVALID_ARG, "moe_grouped_ffn_nvfp4 takes NVFP4 layers only");
  MOE_TRY(check_ws(*cfg, MOE_OP_GROUPED_FFN, ws, ws_bytes));
  if (!weights) return fail(MOE_ERR_INVALID_ARG, "weights is NULL");
  if (!same_shape(weights->cfg, *cfg))
    return fail(MOE_ERR_INVALID_ARG, "weights were created for a different layer shape");
  if (cfg->T == 0) return MOE_OK;
  MOE_TRY(check_ptr(x_perm, "x_perm"));
  MOE_TRY(check_ptr(x_perm_sf, "x_perm_sf"));
  MOE_TRY(check_ptr4(expert_offsets, "expert_offsets"));
  MOE_TRY(check_ptr4(pad_offsets, "pad_offsets"));
  MOE_TRY(check_ptr(y_perm, "y_perm"));
  if (row_weight) MOE_TRY(check_ptr4(row_weight, "row_weight"));
  const bool shared = cfg->I_shared > 0 && shared_out != nullptr;
  if (shared) {
    MOE_TRY(check_ptr(shared_out, "shared_out"));
    MOE_TRY(check_ptr(x_tok, "x_tok"));
    MOE_TRY(check_ptr(x_tok_sf, "x_tok_sf"));
  }
  const Layout L = layout(*cfg, MOE_OP_GROUPED_FFN);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t R = cfg->T * cfg->k;
  // GEMM2 writes fp16 rows + power-of-two scales into the workspace; they are
  // widened exactly into the caller's fp32 rows
  void* y16 = at<void*>(ws, L.y_perm);
  float* y_sc = reinterpret_cast<float*>(static_cast<uint8_t*>(y16) + size_t(R) * cfg->H * 2);
  void* s16 = shared ? at<void*>(ws, L.shared_out) : nullptr;
  float* s_sc = shared ? reinterpret_cast<float*>(static_cast<uint8_t*>(s16) +
                                                  size_t(cfg->T) * cfg->H * 2)
                       : nullptr;
  Nvfp4Acts A{const_cast<int32_t*>(pad_offsets), const_cast<uint8_t*>(x_perm),
              const_cast<uint8_t*>(x_perm_sf), shared ? const_cast<uint8_t*>(x_tok) : nullptr,
              shared ? const_cast<uint8_t*>(x_tok_sf) : nullptr};
  MOE_TRY(run_ffn_nvfp4(*cfg, view_of(weights), L, ws, expert_offsets, A, row_weight, y16, y_sc,
                        s16, s_sc, st));
  MOE_CUDA(launch_widen_half(y16, y_sc, y_perm, R, cfg->H, st));
  if (shared) MOE_CUDA(launch_widen_half(s16, s_sc, shared_out, cfg->T, cfg->H, st));
  trace_mark(st, -1);
  return MOE_OK;
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* y_perm, const int32_t* inv_row,
                         const void* shared_out, void* out, void* ws, size_t ws_bytes,
                         moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  MOE_TRY(check_ws(*cfg, MOE_OP_COMBINE, ws, ws_bytes));
  if (cfg->T == 0) return MOE_OK;
  MOE_TRY(check_ptr(y_perm, "y_perm"));
  MOE_TRY(check_ptr4(inv_row, "inv_row"));
  MOE_TRY(check_ptr(out, "out"));
  if (shared_out) MOE_TRY(check_ptr(shared_out, "shared_out"));
  if (out == y_perm) return fail(MOE_ERR_INVALID_ARG, "out must not alias y_perm");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  trace_mark(st, MOE_K_COMBINE);
  MOE_CUDA(launch_combine(y_perm, inv_row, shared_out, out, cfg->T, cfg->k, cfg->H,
                          cfg->T * cfg->k, err_word(ws), st));
  trace_mark(st, -1);
  return MOE_OK;
}

moe_status_t moe_forward(const moe_config_t* cfg, moe_weights_t weights, const void* x,
                         const void* w_router, const float* logit_bias, void* out,
                         int32_t* topk_ids_out, float* topk_w_out, void* ws, size_t ws_bytes,
                         moe_stream_t stream) {
  return moe_forward_ex(cfg, weights, x, w_router, logit_bias, out, topk_ids_out, topk_w_out, 0,
                        ws, ws_bytes, stream);
}

moe_status_t moe_forward_ex(const moe_config_t* cfg, moe_weights_t weights, const void* x,
                            const void* w_router, const float* logit_bias, void* out,
                            int32_t* topk_ids_out, float* topk_w_out, uint32_t flags, void* ws,
                            size_t ws_bytes, moe_stream_t stream) {
  if (flags & ~uint32_t(MOE_FORWARD_FUSED_DISPATCH))
    return fail(MOE_ERR_INVALID_ARG, "unknown forward flags 0x%x", flags);
  MOE_TRY(check_config(cfg));
  MOE_TRY(check_ws(*cfg, MOE_OP_FORWARD, ws, ws_bytes));
  if (!weights) return fail(MOE_ERR_INVALID_ARG, "weights is NULL");
  if (!same_shape(weights->cfg, *cfg))
    return fail(MOE_ERR_INVALID_ARG, "weights were created for a different layer shape");
  if (cfg->T == 0) return MOE_OK;
  MOE_TRY(check_ptr(x, "x"));
  MOE_TRY(check_ptr(w_router, "w_router"));
  MOE_TRY(check_ptr(out, "out"));
  if (logit_bias) MOE_TRY(check_ptr4(logit_bias, "logit_bias"));
  if (topk_ids_out) MOE_TRY(check_ptr4(topk_ids_out, "topk_ids_out"));
  if (topk_w_out) MOE_TRY(check_ptr4(topk_w_out, "topk_w_out"));
  return forward_impl(cfg, view_of(weights), x, w_router, logit_bias, nullptr, out, topk_ids_out,
                      topk_w_out, flags, ws, stream);
}

moe_status_t moe_forward_stack(const moe_config_t* cfg, moe_stack_t stack, const int32_t* layer,
                               const void* x, void* out, int32_t* topk_ids_out, float* topk_w_out,
                               void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  MOE_TRY(check_ws(*cfg, MOE_OP_FORWARD, ws, ws_bytes));
  if (!stack) return fail(MOE_ERR_INVALID_ARG, "stack is NULL");
  if (!same_shape(stack->cfg, *cfg))
    return fail(MOE_ERR_INVALID_ARG, "the stack was created for a different layer shape");
  MOE_TRY(check_ptr4(layer, "layer"));
  if (cfg->T == 0) return MOE_OK;
  MOE_TRY(check_ptr(x, "x"));
  MOE_TRY(check_ptr(out, "out"));
  if (topk_ids_out) MOE_TRY(check_ptr4(topk_ids_out, "topk_ids_out"));
  if (topk_w_out) MOE_TRY(check_ptr4(topk_w_out, "topk_w_out"));
  const RouterTable rt{stack->router, stack->bias, layer, stack->num_layers};
  return forward_impl(cfg, view_of(stack, layer), x, nullptr, nullptr, &rt, out, topk_ids_out,
                      topk_w_out, 0u, ws, stream);
}

moe_status_t moe_quantize_weight_fp8(const float* w, int64_t N, int64_t K, uint8_t* q,
                                     float* scales, moe_stream_t stream) {
  if (N <= 0 || K <= 0 || N % 128 || K % 128)
    return fail(MOE_ERR_INVALID_ARG, "N and K must be positive multiples of 128");
  MOE_TRY(check_ptr4(w, "w"));
  MOE_TRY(check_ptr(q, "q", false));
  MOE_TRY(check_ptr4(scales, "scales"));
  if (K / 128 > 65535 || N / 128 > 65535) return fail(MOE_ERR_UNSUPPORTED, "matrix too large");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  trace_mark(st, MOE_K_QUANT);
  MOE_CUDA(launch_quant_weight_fp8(w, N, K, q, scales, st));
  trace_mark(st, -1);
  return MOE_OK;
}

moe_status_t moe_quantize_act_fp8(const void* x, int64_t M, int64_t K, uint8_t* q, float* scales,
                                  moe_stream_t stream) {
  if (M < 0 || K <= 0 || K % 128)
    return fail(MOE_ERR_INVALID_ARG, "M >= 0 and K a positive multiple of 128 required");
  if (M == 0) return MOE_OK;
  MOE_TRY(check_ptr(x, "x"));
  MOE_TRY(check_ptr(q, "q", false));
  if (reinterpret_cast<uintptr_t>(q) & 7) return fail(MOE_ERR_INVALID_ARG, "q is not 8-byte aligned");
  MOE_TRY(check_ptr4(scales, "scales"));
  if (M * (K / 128) * 16 / 256 >= (int64_t(1) << 31))
    return fail(MOE_ERR_UNSUPPORTED, "matrix too large");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  trace_mark(st, MOE_K_QUANT);
  MOE_CUDA(launch_quant_act_fp8(x, M, K, q, scales, st));
  trace_mark(st, -1);
  return MOE_OK;
}

moe_status_t moe_quantize_weight_nvfp4(const void* w, const void* w2, int64_t N, int64_t K,
                                       uint8_t* codes, uint8_t* sf, float* tensor_scale,
                                       moe_stream_t stream) {
  if (N <= 0 || K <= 0 || K % 64 || N % 128)
    return fail(MOE_ERR_INVALID_ARG,
                "NVFP4 weights need K a positive multiple of 64 and N of 128");
  MOE_TRY(check_ptr(w, "w"));
  if (w2) MOE_TRY(check_ptr(w2, "w2"));
  MOE_TRY(check_ptr(codes, "codes"));
  MOE_TRY(check_ptr(sf, "sf"));
  MOE_TRY(check_ptr4(tensor_scale, "tensor_scale"));
  if ((w2 ? 2 * N : N) * (K / 16) >= (int64_t(1) << 39)) return fail(MOE_ERR_UNSUPPORTED, "matrix too large");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  trace_mark(st, MOE_K_QUANT);
  MOE_CUDA(launch_quant_weight_nvfp4(w, w2, N, K, codes, sf, tensor_scale, st));
  trace_mark(st, -1);
  return MOE_OK;
}

moe_status_t moe_quantize_act_nvfp4(const void* x, int64_t M, int64_t K, float g, uint8_t* codes,
                                    uint8_t* sf, moe_stream_t stream) {
  if (M < 0 || K <= 0 || K % 16)
    return fail(MOE_ERR_INVALID_ARG, "M >= 0 and K a positive multiple of 16 required");
  if (!std::isfinite(g) || g <= 0.0f) return fail(MOE_ERR_INVALID_ARG, "g must be finite and > 0");
  if (M == 0) return MOE_OK;
  MOE_TRY(check_ptr(x, "x"));
  if (!codes || (reinterpret_cast<uintptr_t>(codes) & 7))
    return fail(MOE_ERR_INVALID_ARG, "codes is NULL or not 8-byte aligned");
  if (!sf) return fail(MOE_ERR_INVALID_ARG, "sf is NULL");
  if (M * (K / 16) >= (int64_t(1) << 39)) return fail(MOE_ERR_UNSUPPORTED, "matrix too large");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  trace_mark(st, MOE_K_QUANT);
  MOE_CUDA(launch_quant_act_nvfp4(x, M, K, g, codes, sf, st));
  trace_mark(st, -1);
  return MOE_OK;
}

}  // extern "C"
