// Internal interface between the C-ABI host code (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

// Bits of the sticky status word at the start of every workspace.
constexpr uint32_t kErrBounds = 1u;    // an index outside its range was skipped
constexpr uint32_t kErrTimeout = 2u;   // a bounded wait expired
constexpr uint32_t kErrNoSelect = 4u;  // a token had fewer than k selectable logits (NaN)
constexpr uint32_t kErrDupIds = 8u;    // a token listed one expert in two of its k slots

// A wait that takes longer than this is treated as a hang: the waiting role
// records kErrTimeout, raises the CTA's abort flag and leaves its loop.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Tile shapes shared by the host (tensor-map boxes, schedules) and kernels.
constexpr int kTileM = 128;        // rows of one accumulator tile (UMMA M)
constexpr int kTileK = 64;         // bf16 K per stage = one 128-byte swizzle row
constexpr int kGemm1TileN = 128;   // h columns per GEMM1 tile (gate 128 + up 128 = UMMA N 256)
constexpr int kGemm2TileN = 256;   // y columns per GEMM2 tile
constexpr int kMaxExperts = 256;
constexpr int kMaxGroups = kMaxExperts + 1;  // routed experts + the shared expert
constexpr int kPermTok = 64;       // tokens per histogram / scatter block
constexpr int kGemmTileRows = 256; // rows of one grouped-GEMM work tile (a CTA pair)
constexpr int kGemmBRows = 128;    // weight rows one CTA of the pair loads per stage (TMA box)
constexpr int kFp8Tile1Tokens = 64; // tokens per fp8 GEMM1 tile (the MMA's N side)
constexpr int kFp8Tile2Tokens = 32; // tokens per fp8 GEMM2 tile
constexpr int kFp8WRows = 128;     // weight rows per fp8 tile (the MMA's M side)
constexpr int kFp8MaxKBlocks = 64; // fp8: at most 64 K blocks of 128 (H, I <= 8192)

// Tile schedule of one grouped GEMM, in device memory (int32):
//   [0]            number of tiles
//   [1 .. G+1]     first tile of each processing slot (exclusive prefix, [G+1] = total)
//   [G+2 .. 2G+1]  group processed in each slot (heaviest first)
__host__ __device__ inline int sched_ints(int G) { return 2 * G + 2; }

// Layer of a layer-stack call: *layer when given (read at kernel time; an
// index outside [0, n) sets kErrBounds and selects layer 0), else 0.
__device__ __forceinline__ int resolve_layer(const int32_t* layer, int n, uint32_t* err) {
  if (layer == nullptr) return 0;
  const int l = *reinterpret_cast<const volatile int32_t*>(layer);
  if (l < 0 || l >= n) {
    if (threadIdx.x == 0) atomicOr(err, kErrBounds);
    return 0;
  }
  return l;
}

struct GemmArgs {
  const CUtensorMap* b_maps;   // GEMM1: gate of group g at 2g, up at 2g+1; GEMM2: down at g
                               // (layer 0's, in a layer stack)
  const int32_t* layer;        // layer stack: device layer index, else null
  int32_t layer_stride;        // descriptors per layer in the stack table
  int32_t num_layers;
  const int32_t* offsets;      // [E+1] routed row offsets
  const int32_t* sched;        // tile schedule (see above)
  void* out0;                  // routed output rows (GEMM1: bf16 h, GEMM2: fp32 y or fp16 y)
  void* out1;                  // shared-expert output rows (same types)
  float* out_scales0;          // GEMM2: null for fp32 y; else y is fp16 and these are its
  float* out_scales1;          //   power-of-two scales, [rows][N/32] (routed / shared)
  const float* row_weight;     // GEMM2: per routed row scale, or null
  const int32_t* gather_rows;  // GEMM1: row -> token map; routed A rows are gathered from the
                               // unpermuted tokens (map_a0 has one-row boxes), or null
  uint32_t* err;               // sticky status word
  int32_t R;                   // routed rows (T*k)
  int32_t E;
  int32_t has_shared;
  int32_t T;                   // rows of the shared group
  int32_t K_routed, K_shared;  // reduction sizes
  int32_t N_routed, N_shared;  // output columns
  int32_t stall_test;          // failure-path test: pair 0 waits on a barrier nothing ends
  const uint8_t* amap;         // [E] 128-byte A tensor maps, expert e's with its row extent
                               // cut at offsets[e + 1] (written by the plan kernel), or null
};

// Failure-path test hook (moe_test_stall_gemm1): whether the next bf16 GEMM1
// launch of the calling thread should stall its first CTA pair (consumes one).
bool take_gemm1_stall();

// fp8 grouped GEMM (weights on the MMA's M side, tokens on N).
struct Fp8GemmArgs {
  const CUtensorMap* w_maps;      // GEMM1: gate of group g at 2g, up at 2g+1; GEMM2: down at g
  const float* const* w_scales;   // same indexing; each [rows/128, K/128] fp32
  const int32_t* layer;           // layer stack: device layer index (both tables advance
  int32_t layer_stride;           //   by layer_stride entries per layer), else null
  int32_t num_layers;
  const int32_t* offsets;         // [E+1] routed row offsets
  const int32_t* sched;           // tile schedule (64-token tiles)
  const float* tok_scales0;       // routed token scales [T*k, K/128]
  const float* tok_scales1;       // shared-expert token scales [T, K/128]
  void* out0;                     // routed out: GEMM1 e4m3 h [T*k, I], GEMM2 fp32 y [T*k, H]
  void* out1;                     // shared out: GEMM1 e4m3 h [T, I_s], GEMM2 fp32 [T, H]
  float* out_scales0;             // GEMM1: h scales [T*k, I/128]
  float* out_scales1;             // GEMM1: shared h scales [T, I_s/128]
  const float* row_weight;        // GEMM2: per routed row scale, or null
  uint32_t* err;
  int32_t E, has_shared, T;
  int32_t K_routed, K_shared;     // reduction sizes
  int32_t N_routed, N_shared;     // output columns (GEMM1: I, I_s; GEMM2: H, H)
};

// NVFP4 grouped GEMM (tokens on the MMA's M side, 128-row blocks of each
// expert's rows padded to a multiple of 128).
constexpr int kNvfp4Rows = 128;     // token rows per tile = padding granule of the permuted rows
struct Nvfp4GemmArgs {
  const CUtensorMap* w_maps;      // GEMM1: stacked gate/up of group g at 2g; GEMM2: down at g
  const uint8_t* const* w_sf;     // same indexing: the matrix's scales in the MMA layout
  const float* const* w_gs;       // same indexing: the matrix's fp32 tensor scale (device)
  const float* act_scales;        // [num_layers][2] static tensor scales g_x, g_h (device)
  const int32_t* layer;           // layer stack: device layer index (tables advance by
  int32_t layer_stride;           //   layer_stride entries per layer), else null
  int32_t num_layers;
  const int32_t* offsets;         // [E+1] routed row offsets
  const int32_t* pad_offsets;     // [E+1] offsets of each expert's 128-row-padded segment
  const int32_t* sched;           // tile schedule (128-row tiles)
  const uint8_t* a_sf0;           // routed A scales (MMA layout over the padded rows)
  const uint8_t* a_sf1;           // shared-expert A scales (MMA layout over token rows)
  void* out0;                     // GEMM1: h codes [padded rows, I/2]; GEMM2: fp16 y [T*k, H]
  void* out1;                     // GEMM1: shared h codes [T pad, I_s/2]; GEMM2: fp16 [T, H]
  uint8_t* out_sf0;               // GEMM1: h scales (MMA layout)
  uint8_t* out_sf1;               // GEMM1: shared h scales (MMA layout)
  float* out_scales0;             // GEMM2: y power-of-two scales [T*k, H/32]
  float* out_scales1;             // GEMM2: shared [T, H/32]
  const float* row_weight;        // GEMM2: per routed row (unpadded order), or null
  uint32_t* err;
  int32_t E, has_shared, T;
  int32_t K_routed, K_shared;     // reduction sizes (multiples of 256)
  int32_t N_routed, N_shared;     // GEMM1: I, I_shared (h columns); GEMM2: H, H
};

// --------------------------------------------------------------- launchers
// Router of one layer, or (w_table non-null) of layer *layer of a stack whose
// router descriptors and bias pointers are device tables [num_layers].
struct RouterTable {
  const CUtensorMap* w_table;
  const float* const* bias_table;
  const int32_t* layer;
  int32_t num_layers;
};
cudaError_t launch_router(const CUtensorMap& map_x, const CUtensorMap& map_w, int64_t T, int H,
                          int E, int E_pad, int k, int score, int renormalize, float route_scale,
                          const float* bias, int32_t* topk_ids, float* topk_w, float* logits_out,
                          uint32_t* err, int sm_count, cudaStream_t stream,
                          const RouterTable* table = nullptr);

cudaError_t launch_hist(const int32_t* ids, int64_t T, int k, int E, int32_t* blk_counts,
                        uint32_t* err, cudaStream_t stream);

// pad_offsets (optional, [E+1]): exclusive scan of the counts rounded up to
// multiples of 128 (the NVFP4 layout of the permuted rows).
cudaError_t launch_scan(const int32_t* blk_counts, int nblk, int E, int32_t* blk_base,
                        int32_t* counts, int32_t* offsets, cudaStream_t stream,
                        int32_t* pad_offsets = nullptr);

cudaError_t launch_scatter(const int32_t* ids, const float* topk_w, const void* x, int64_t T,
                           int k, int E, int H, int fp8, const int32_t* blk_base,
                           const int32_t* offsets, int32_t* perm_token, int32_t* inv_row,
                           float* row_weight, void* x_perm, float* x_perm_scales, uint32_t* err,
                           cudaStream_t stream);

// NVFP4 scatter: the maps as launch_scatter; each token quantised once with the
// static tensor scale *g_x (g_x = act_scales + 2 * layer), its codes written to
// its k padded rows (pad_offsets) with MMA-layout scales, and (xs_codes non-null)
// to its own row of the token-order copy for the shared expert.  The scales of
// every padding row are set to zero.
struct Nvfp4Scatter {
  const int32_t* pad_offsets;
  const float* act_scales;
  const int32_t* layer;
  int32_t num_layers;
  int64_t rows_pad;     // rows of x_perm (bounds check)
  uint8_t* x_codes;     // [rows_pad, H/2]
  uint8_t* x_sf;        // MMA layout over rows_pad rows
  uint8_t* xs_codes;    // [T pad, H/2] or null
  uint8_t* xs_sf;
};
cudaError_t launch_scatter_nvfp4(const int32_t* ids, const float* topk_w, const void* x,
                                 int64_t T, int k, int E, int H, const int32_t* blk_base,
                                 const int32_t* offsets, int32_t* perm_token, int32_t* inv_row,
                                 float* row_weight, const Nvfp4Scatter& q, uint32_t* err,
                                 cudaStream_t stream);

// Grid (a multiple of 2) of the grouped GEMMs: as many CTA pairs as the
// device can hold at once.
int grouped_gemm_grid(int sm_count);

// With cut (bf16 layers: 2 E x 128 bytes, 128-byte aligned) the plan kernel also
// writes each expert's copies of cut_a1 (GEMM1's A map) and cut_a2 (GEMM2's) with
// the row extent cut at the end of the expert's rows (GemmArgs::amap), never past
// cut_rows (both templates' row extent).
cudaError_t launch_plan(const int32_t* offsets, int E, int has_shared, int64_t T, int n1_routed,
                        int n1_shared, int n2_routed, int n2_shared, int32_t* sched1,
                        int32_t* sched2, int tile_rows1, int tile_rows2, cudaStream_t stream,
                        const CUtensorMap* cut_a1 = nullptr, const CUtensorMap* cut_a2 = nullptr,
                        uint8_t* cut = nullptr, int64_t cut_rows = 0);

cudaError_t launch_grouped_gemm_fp8(bool gate_up, const CUtensorMap& tok_map0,
                                    const CUtensorMap& tok_map1, const Fp8GemmArgs& args, int grid,
                                    cudaStream_t stream);

// map_y0 / map_y1: GEMM2's fp16 outputs (routed rows, shared-expert rows) as
// 2-byte tensors with 32-row x 64-column boxes, 128-byte swizzle; unused by GEMM1.
cudaError_t launch_grouped_gemm_nvfp4(bool gemm1, const CUtensorMap& map_a0,
                                      const CUtensorMap& map_a1, const CUtensorMap& map_y0,
                                      const CUtensorMap& map_y1, const Nvfp4GemmArgs& args,
                                      int grid, cudaStream_t stream);

cudaError_t launch_grouped_gemm(bool swiglu, const CUtensorMap& map_a0, const CUtensorMap& map_a1,
                                const GemmArgs& args, int grid, cudaStream_t stream);

cudaError_t launch_combine(const void* y_perm, const int32_t* inv_row, const void* shared_out,
                           void* out, int64_t T, int k, int H, int64_t R, uint32_t* err,
                           cudaStream_t stream);

// Combine of fp16 expert rows with one power-of-two scale per 32 columns
// ([rows][H/32] fp32), as written by the grouped GEMM2 with out_scales set.
cudaError_t launch_combine_half(const void* y, const float* y_scales, const int32_t* inv_row,
                                const void* shared, const float* shared_scales, void* out,
                                int64_t T, int k, int H, int64_t R, uint32_t* err,
                                cudaStream_t stream);

// fp16 rows with one power-of-two scale per 32 columns ([rows][H/32] fp32)
// widened to fp32 rows: out[r][c] = float(y[r][c]) * scales[r][c / 32] (exact).
cudaError_t launch_widen_half(const void* y, const float* scales, float* out, int64_t rows, int H,
                              cudaStream_t stream);

cudaError_t launch_quant_weight_fp8(const float* w, int64_t N, int64_t K, uint8_t* q,
                                    float* scales, cudaStream_t stream);

cudaError_t launch_quant_act_fp8(const void* x, int64_t M, int64_t K, uint8_t* q, float* scales,
                                 cudaStream_t stream);

// NVFP4 weights: bf16 [N, K] (w2 null) or the stacked gate/up pair (w, w2 both
// [N, K]; output rows interleaved in 128-row blocks [w 128 | w2 128]); codes
// [rows, K/2], MMA-layout scales, tensor scale amax / 2688 into *tensor_scale.
cudaError_t launch_quant_weight_nvfp4(const void* w, const void* w2, int64_t N, int64_t K,
                                      uint8_t* codes, uint8_t* sf, float* tensor_scale,
                                      cudaStream_t stream);

// NVFP4 activations with a static tensor scale: codes [M, K/2], row-major
// scales [M, K/16] (e4m3 codes).
cudaError_t launch_quant_act_nvfp4(const void* x, int64_t M, int64_t K, float g, uint8_t* codes,
                                   uint8_t* sf, cudaStream_t stream);

}  // namespace moe

#include "../../include/moe_layer.h"

namespace moe {
// Host-side argument checks shared by every entry point (api.cu): the layer
// configuration, and a pointer that must be non-null and 16-byte (check_ptr)
// or 4-byte (check_ptr4) aligned.  A failure sets moe_last_error_message().
moe_status_t check_config(const moe_config_t* c);
moe_status_t check_ptr(const void* p, const char* name, bool needs16 = true);
moe_status_t check_ptr4(const void* p, const char* name);

// Raises a kernel's dynamic shared-memory limit on the current device (once per device).
cudaError_t ensure_smem_attr(const void* func, int bytes);

// Sets the text returned by moe_last_error_message() on the calling thread.
void set_last_error_text(const char* msg);

// Kernel tracing (see moe_set_trace): records an event before kernel `id` on
// `stream` (id = -1: after the last kernel of a call).  No-op without a trace.
void trace_mark(cudaStream_t stream, int id);
}  // namespace moe
