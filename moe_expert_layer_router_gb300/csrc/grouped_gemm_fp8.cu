// fp8 e4m3 grouped GEMMs with 128x128 weight block scales and per-token 1x128
// activation scales, for the small-batch (memory-bound) regime: the expert
// weights are streamed once from HBM and every expert sees only a few tokens
// (fp8 expert GEMMs as in "Memory-Compute Disaggregation for Large-Model
// Inference: AFD Architecture Analysis and Performance Validation", section
// 1; grouped matrix multiplication over per-expert weights as in "ASAP: A
// DiSaggregated and Asynchronous Inference System for MoE Prefill", section
// 3.4.2, and "DWDP: Distributed Weight Data Parallelism for
// High-Performance LLM Inference on NVL72", section 4.2).
//
// Swapped operands: the MMA's M side is 128 weight rows of one expert, its N
// side the expert's tokens (up to 64 per tile), so D^T[weight row, token]
// lands in TMEM with one weight row per lane.  Each 128-wide K block is a
// separate tcgen05 kind::f8f6f4 product (4 MMAs of K = 32) into its own TMEM
// partial; the epilogue warps add it into fp32 registers scaled by
//   s_w[row block, k block] * s_x[token, k block]
// (the weight scale is one value per tile and K block).  A tile walks its K
// blocks starting at block (tile index mod K blocks): at any moment the CTAs
// then read different 128-byte columns of their weight slabs, which spreads
// the weight stream over the HBM channels when the row pitch is a power of
// two (W_down: 2 KB).  Partials rotate
// through 4 (GEMM1) or 8 (GEMM2) TMEM buffers so the MMAs run ahead.
//
//   GEMM1 (kGateUp): 128 W_gate rows and the same 128 W_up rows of expert e;
//     h = silu(g) * u for 128 consecutive intermediate columns -- exactly one
//     1x128 quantisation group per token -- quantised in the epilogue:
//     s_h = amax/448, q = rn_satfinite(h / s_h) (fp32), e4m3 codes + scales out.
//   GEMM2: 128 W_down rows; y[token, row] = row_weight * sum, fp32 out.
// Warp roles: warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer,
// warps 2..5 epilogue (one weight row per thread).  Persistent CTAs, tiles
// from the device-built schedule (heaviest experts first).
#include <cuda_fp8.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int kKB = 128;                    // K elements (bytes) per block = one scale block
constexpr int kWRows = 128;                 // weight rows per tile (UMMA M)
constexpr int kWBytes = kWRows * kKB;       // 16 KB per weight box
constexpr int kTokBox = 32;                 // token rows per TMA box
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxKB = kFp8MaxKBlocks;      // K blocks per row (H or I up to 8192)

// Every tile holds two 128-row weight blocks: GEMM1 the gate and the up rows
// of 128 intermediate columns, GEMM2 two consecutive 128-row blocks of W_down
// (256 output columns).  A stage is both blocks' 128-byte K slice plus the
// tokens'.  GEMM1: 64-token tiles, 5 stages of 40 KB.  GEMM2: 32-token tiles,
// 4 stages of 36 KB: GEMM2 streamed W_down faster with fewer loads in flight
// (DeepSeek-V3 at 512 tokens: 6 stages 0.683 ms, 5 0.666, 4 and 3 0.630, 2
// 0.707); GEMM1 on 4 stages was slightly slower than on 5.
template <bool kGateUp>
struct Cfg {
  static constexpr int kTok = kGateUp ? kFp8Tile1Tokens : kFp8Tile2Tokens;  // tokens per tile
  static constexpr int kTokBytes = kTok * kKB;                               // token region per stage
  static constexpr int kStages = kGateUp ? 5 : 4;
  static constexpr int kStageBytes = 2 * kWBytes + kTokBytes;
  static constexpr int kBufCols = 128;                      // TMEM columns per partial
  static constexpr int kBufs = kTmemCols / kBufCols;        // 4
};
constexpr int kBlk1Col = 64;  // TMEM column of the second block's partial

template <bool kGateUp>
struct __align__(8) SmemCtl {
  uint64_t full[Cfg<kGateUp>::kStages];
  uint64_t empty[Cfg<kGateUp>::kStages];
  uint64_t pfull[Cfg<kGateUp>::kBufs];
  uint64_t pempty[Cfg<kGateUp>::kBufs];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float tok_scale[Cfg<kGateUp>::kTok * kMaxKB];  // s_x of the tile's tokens, [token][k block]
  float red[4][Cfg<kGateUp>::kTok];              // per-warp amax of h (GEMM1)
};

template <bool kGateUp>
constexpr size_t smem_bytes() {
  return 1024 + size_t(Cfg<kGateUp>::kStages) * Cfg<kGateUp>::kStageBytes +
         sizeof(SmemCtl<kGateUp>);
}

struct Tile {
  int g, tok_blk, w_blk, rows, row0, K;
};

__device__ __forceinline__ Tile decode_tile(int t, const Fp8GemmArgs& a, int G, int tok) {
  const int32_t* ts = a.sched + 1;
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(ts + mid) <= t) lo = mid; else hi = mid - 1;
  }
  Tile x;
  x.g = __ldg(a.sched + G + 2 + lo);
  const int local = t - __ldg(ts + lo);
  const bool routed = x.g < a.E;
  x.rows = routed ? __ldg(a.offsets + x.g + 1) - __ldg(a.offsets + x.g) : a.T;
  x.row0 = routed ? __ldg(a.offsets + x.g) : 0;
  x.K = routed ? a.K_routed : a.K_shared;
  const int mt = (x.rows + tok - 1) / tok;
  x.w_blk = local / mt;
  x.tok_blk = local - x.w_blk * mt;
  return x;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kWaitTimeoutNs) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

// Barriers among the 4 epilogue warps only (named barrier 1, 128 threads).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Barrier that also ORs `v` over the 128 epilogue threads, so that a decision
// to stop (a wait that gave up) is taken by all of them together.
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

template <bool kGateUp>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap map_b0,
                            const __grid_constant__ CUtensorMap map_b1, const Fp8GemmArgs args) {
  using C = Cfg<kGateUp>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SmemCtl<kGateUp>& c = *reinterpret_cast<SmemCtl<kGateUp>*>(smem + C::kStages * C::kStageBytes);
  auto stage_w = [&](int s, int which) { return smem + s * C::kStageBytes + which * kWBytes; };
  auto stage_t = [&](int s) { return smem + s * C::kStageBytes + 2 * kWBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = args.E + args.has_shared;
  // weight descriptors and scales of this call's layer (layer stacks)
  const int layer = resolve_layer(args.layer, args.num_layers, args.err);
  const CUtensorMap* wmaps = args.w_maps + layer * args.layer_stride;
  const float* const* wscales = args.w_scales + layer * args.layer_stride;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&c.full[s], 1);
      ptx::mbar_init(&c.empty[s], 1);
    }
    for (int b = 0; b < C::kBufs; ++b) {
      ptx::mbar_init(&c.pfull[b], 1);
      ptx::mbar_init(&c.pempty[b], 4);
    }
    ptx::mbar_init(&c.drain, 1);
    c.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&c.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  const int num_tiles = __ldg(args.sched);
  volatile int* abort = &c.abort;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- TMA producer
      uint32_t it = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort; t += gridDim.x) {
        const Tile x = decode_tile(t, args, G, C::kTok);
        const bool routed = x.g < args.E;
        const void* map_t = routed ? static_cast<const void*>(&map_b0)
                                   : static_cast<const void*>(&map_b1);
        const int left = x.rows - x.tok_blk * C::kTok;
        const int n_tok = left < C::kTok ? left : C::kTok;
        const int n_box = (n_tok + kTokBox - 1) / kTokBox;
        const int tok_row = x.row0 + x.tok_blk * C::kTok;
        // the two weight blocks: gate and up rows of the same 128 columns
        // (GEMM1), or W_down rows [256 w, +128) and [256 w + 128, +128) (GEMM2;
        // past H the second box is zero-filled)
        const CUtensorMap* mw0 = kGateUp ? wmaps + 2 * x.g : wmaps + x.g;
        const CUtensorMap* mw1 = kGateUp ? mw0 + 1 : mw0;
        const int w_row0 = x.w_blk * (kGateUp ? kWRows : 2 * kWRows);
        const int w_row1 = kGateUp ? w_row0 : w_row0 + kWRows;
        const uint32_t bytes = 2 * kWBytes + n_box * kTokBox * kKB;
        const int kb_n = x.K / kKB;
        bool ok = true;
        const int rot = t % kb_n;
        for (int kb = 0; kb < kb_n; ++kb, ++it) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          const int kbe = kb + rot < kb_n ? kb + rot : kb + rot - kb_n;
          if (!ptx::mbar_wait(&c.empty[s], ph ^ 1, abort, args.err)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&c.full[s], bytes);
          ptx::tma_load_2d(stage_w(s, 0), mw0, &c.full[s], kbe * kKB, w_row0);
          ptx::tma_load_2d(stage_w(s, 1), mw1, &c.full[s], kbe * kKB, w_row1);
          for (int bx = 0; bx < n_box; ++bx)
            ptx::tma_load_2d(stage_t(s) + bx * kTokBox * kKB, map_t, &c.full[s], kbe * kKB,
                             tok_row + bx * kTokBox);
        }
        if (!ok) break;
      }
      if (*abort) {
        const uint32_t first = it > uint32_t(C::kStages) ? it - C::kStages : 0;
        for (uint32_t j = first; j < it; ++j)
          drain_wait(&c.full[j % C::kStages], (j / C::kStages) & 1, args.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------- MMA issuer
      uint32_t it = 0, pb = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        const Tile x = decode_tile(t, args, G, C::kTok);
        const int left = x.rows - x.tok_blk * C::kTok;
        const int n_tok = left < C::kTok ? left : C::kTok;
        const int n_mma = ((n_tok + kTokBox - 1) / kTokBox) * kTokBox;  // 32 or 64
        const uint32_t idesc = ptx::idesc_e4m3(kWRows, n_mma);
        const int kb_n = x.K / kKB;
        bool ok = true;
        for (int kb = 0; kb < kb_n; ++kb, ++it, ++pb) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          const int b = pb % C::kBufs;
          const uint32_t bph = (pb / C::kBufs) & 1;
          if (!ptx::mbar_wait(&c.pempty[b], bph ^ 1, abort, args.err)) { ok = false; break; }
          if (!ptx::mbar_wait(&c.full[s], ph, abort, args.err)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint64_t dt = ptx::sw128_desc(ptx::smem_u32(stage_t(s)));
          const uint32_t d0 = tmem_base + b * C::kBufCols;
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            const uint64_t dw = ptx::sw128_desc(ptx::smem_u32(stage_w(s, w)));
#pragma unroll
            for (int k = 0; k < kKB / 32; ++k)
              ptx::mma_f8(d0 + w * kBlk1Col, dw + 2 * k, dt + 2 * k, idesc, k != 0);
          }
          ptx::mma_commit(&c.empty[s]);
          ptx::mma_commit(&c.pfull[b]);
        }
        if (!ok) break;
      }
      ptx::mma_commit(&c.drain);
      drain_wait(&c.drain, 0, args.err);
    }
  } else {
    // ------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;
    const int r = q * 32 + lane;                 // weight row within the tile
    const int et = threadIdx.x - 64;             // 0..127 among the epilogue threads
    uint32_t pb = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const Tile x = decode_tile(t, args, G, C::kTok);
      const bool routed = x.g < args.E;
      const int left = x.rows - x.tok_blk * C::kTok;
      const int n_tok = left < C::kTok ? left : C::kTok;
      const int kb_n = x.K / kKB;
      const int tok_row = x.row0 + x.tok_blk * C::kTok;
      // stage the tile's token scales [token][k block] in shared memory
      const float* ts = routed ? args.tok_scales0 : args.tok_scales1;
      epi_sync();
      for (int i = et; i < n_tok * kb_n; i += 128) {
        const int j = i / kb_n, kb = i - j * kb_n;
        c.tok_scale[j * kMaxKB + kb] = __ldg(ts + int64_t(tok_row + j) * kb_n + kb);
      }
      epi_sync();
      // block scales of the tile's two weight blocks (GEMM2: row blocks 2w and
      // 2w+1 of W_down; the second exists only while 256 w + 128 < H)
      const bool blk1 = kGateUp || (2 * x.w_blk + 1) * kWRows < args.N_routed;
      const float* ws0 = wscales[kGateUp ? 2 * x.g : x.g] +
                         int64_t(kGateUp ? x.w_blk : 2 * x.w_blk) * kb_n;
      const float* ws1 = kGateUp ? wscales[2 * x.g + 1] + int64_t(x.w_blk) * kb_n
                                 : (blk1 ? ws0 + kb_n : ws0);
      float acc0[C::kTok], acc1[C::kTok];
#pragma unroll
      for (int j = 0; j < C::kTok; ++j) {
        acc0[j] = 0.0f;
        acc1[j] = 0.0f;
      }
      bool ok = true;
      const int rot = t % kb_n;
      for (int kb = 0; kb < kb_n; ++kb, ++pb) {
        const int kbe = kb + rot < kb_n ? kb + rot : kb + rot - kb_n;
        const int b = pb % C::kBufs;
        const uint32_t bph = (pb / C::kBufs) & 1;
        if (!ptx::mbar_wait(&c.pfull[b], bph, abort, args.err)) { ok = false; break; }
        ptx::tc_fence_after();
        const float sw0 = __ldg(ws0 + kbe);
        const float sw1 = __ldg(ws1 + kbe);
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * C::kBufCols;
#pragma unroll
        for (int half = 0; half < C::kTok / 32; ++half) {
          if (half * 32 < n_tok) {  // warp-uniform
            uint32_t p0[32], p1[32];
            ptx::tmem_ld32(taddr + half * 32, p0);
            ptx::tmem_ld32(taddr + kBlk1Col + half * 32, p1);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float sx = c.tok_scale[(half * 32 + j) * kMaxKB + kbe];
              acc0[half * 32 + j] += __uint_as_float(p0[j]) * (sw0 * sx);
              acc1[half * 32 + j] += __uint_as_float(p1[j]) * (sw1 * sx);
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&c.pempty[b]);
      }
      if (epi_any(!ok || *abort)) break;  // uniform over the epilogue warps
      if constexpr (kGateUp) {
        // h for this weight row (intermediate column) and each token; one
        // 128-wide quantisation group per token = the 128 threads.
        uint8_t* hq = static_cast<uint8_t*>(routed ? args.out0 : args.out1);
        float* hs = routed ? args.out_scales0 : args.out_scales1;
        const int n_i = routed ? args.N_routed : args.N_shared;  // I or I_shared
        const int col = x.w_blk * kWRows + r;
#pragma unroll
        for (int j = 0; j < C::kTok; ++j) {
          acc0[j] = silu_f(acc0[j]) * acc1[j];
          float a = fabsf(acc0[j]);
#pragma unroll
          for (int d = 16; d >= 1; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));
          if (lane == 0) c.red[q][j] = a;
        }
        epi_sync();
#pragma unroll
        for (int j = 0; j < C::kTok; ++j) {
          if (j < n_tok) {
            const float amax = fmaxf(fmaxf(c.red[0][j], c.red[1][j]), fmaxf(c.red[2][j], c.red[3][j]));
            const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
            const int64_t row = tok_row + j;
            hq[row * n_i + col] = static_cast<uint8_t>(
                __nv_cvt_float_to_fp8(__fdiv_rn(acc0[j], s), __NV_SATFINITE, __NV_E4M3));
            if (r == 0) hs[row * (n_i / kKB) + x.w_blk] = s;
          }
        }
      } else {
        float* y = static_cast<float*>(routed ? args.out0 : args.out1);
        const int n_o = args.N_routed;  // H for both groups
        const int col = x.w_blk * 2 * kWRows + r;  // block 0; block 1 is 128 columns on
#pragma unroll
        for (int j = 0; j < C::kTok; ++j) {
          if (j < n_tok) {
            const int64_t row = tok_row + j;
            const float w = (routed && args.row_weight) ? __ldg(args.row_weight + row) : 1.0f;
            y[row * n_o + col] = w * acc0[j];
            if (blk1) y[row * n_o + col + kWRows] = w * acc1[j];
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool kGateUp>
cudaError_t launch_impl(const CUtensorMap& b0, const CUtensorMap& b1, const Fp8GemmArgs& args,
                        int grid, cudaStream_t stream) {
  constexpr size_t smem = smem_bytes<kGateUp>();
  static_assert(smem <= 232448, "shared memory budget");
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(grouped_gemm_fp8_kernel<kGateUp>),
                                   static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  grouped_gemm_fp8_kernel<kGateUp><<<grid, kThreads, smem, stream>>>(b0, b1, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm_fp8(bool gate_up, const CUtensorMap& tok_map0,
                                    const CUtensorMap& tok_map1, const Fp8GemmArgs& args, int grid,
                                    cudaStream_t stream) {
  return gate_up ? launch_impl<true>(tok_map0, tok_map1, args, grid, stream)
                 : launch_impl<false>(tok_map0, tok_map1, args, grid, stream);
}

}  // namespace moe
