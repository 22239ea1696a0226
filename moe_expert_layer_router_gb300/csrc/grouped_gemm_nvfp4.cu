// NVFP4 grouped GEMMs: E2M1 tokens x E2M1 expert weights, one UE4M3 scale per
// 16 elements along K on both sides, on the tcgen05 block-scaled tensor cores
// (kind::mxf4nvf4, scale_vec::4X).  MoE weights in NVFP4 as in the DWDP
// write-up's experimental setup (section A4); grouped matrix multiplication
// over per-expert weight buffers as in "ASAP: A DiSaggregated and Asynchronous
// Inference System for MoE Prefill", section 3.4.2, and "DWDP: Distributed
// Weight Data Parallelism for High-Performance LLM Inference on NVL72",
// section 4.2.
//
// A tile is 128 token rows (UMMA M) x 128 W weight rows (UMMA N = 128 W), K in
// stages of 256 elements (128 bytes per row).  Each expert's rows are padded to
// a multiple of 128 in the permuted buffers, so a tile is one aligned row block
// and its scales are whole 512-byte atoms (see nvfp4.cuh, sf_offset).
//   stage = A 16 KB | B 16 W KB | A scales 2 KB | B scales 2 W KB (W = 2: 54 KB)
// A block-scaled MMA of M = 128 costs the same ~135 cycles for N = 128 and
// N = 256, so both GEMMs use W = 2: one MMA per K = 64 covers 256 weight rows,
// into a single 256-column accumulator (TMEM cannot hold two next to the scale
// slots).  Eight epilogue warps, given 192 registers each by setmaxnreg, read
// all of it with one wait and release it at once.
// A and B arrive by TMA (128-byte swizzle), the scale atoms by 1-D bulk copies
// on their own barrier, issued first.  Four scale warps, one per TMEM lane
// quarter, move each stage's scales into that stage's TMEM scale slot with
// tcgen05.st, in the layout the MMA reads for 128 rows: lane j (of every
// quarter), column c + i holds the four K-block scales of row 32i + j (A: 4
// columns per MMA, B: 4 W).  They then arrive on the stage's sf_ready barrier,
// on which the MMA lane waits before issuing the stage's 4 MMAs of K = 64.
// (Issued from the MMA lane, tcgen05.cp of the same atoms blocked it for about
// 60 cycles each.)  A slot is rewritten only once the stage's smem was
// refilled, i.e. after the MMAs that read the slot completed.
// TMEM: accumulators in columns [0, 256), scale slots from column 256.
//
//   GEMM1 (kGemm1): B = 256 rows of the expert's stacked gate/up matrix, whose
//     rows are interleaved in 128-row blocks [gate 128 | up 128]: tile n holds
//     the gate and up rows of h columns [128 n, 128 n + 128).  h = silu(g) * u
//     with g, u = accumulator * g_x * g_w, quantised to NVFP4 with the static
//     scale g_h: packed codes and MMA-layout scales of every row of the block.
//   GEMM2: y = accumulator * g_h * g_w * row weight,
//     B = 256 rows of W_down; written as fp16 with a power-of-two scale per 32
//     columns (only the block's real rows, at their unpadded row index).  Each
//     epilogue warp puts its 32 rows x 64 columns into a 4 KB shared-memory box
//     (128-byte swizzle) that one lane writes out with a TMA store; a warp with
//     fewer than 32 real rows (the segment's end) stages them through 512 bytes
//     of that buffer instead, 4 rows x 128 bytes per store instruction.  GEMM2
//     runs 3 stages, GEMM1 4.
// Warp roles, by warpgroup: 0 = TMA producer (warp 0), TMEM allocator + MMA
// issuer (warp 1) and two idle warps; 1 and 2 = the epilogue (one row per
// thread, two warps per TMEM lane quarter, one per 128-column half); 3 = the
// scale warps.  Persistent CTAs over the device-built tile schedule (heaviest
// experts first, tiles of one weight block adjacent), which every CTA first
// copies into shared memory together with the row offsets and the weight
// tensor scales.
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRows = 128;                  // token rows per tile
constexpr int kRowBytes = 128;              // K bytes per stage and row (256 elements)
constexpr int kABytes = kRows * kRowBytes;  // 16 KB
constexpr int kSfaBytes = 2048;             // 4 atoms of 512 bytes (4 MMAs of K = 64)
constexpr uint32_t kTmemCols = 512;
constexpr int kSfCol = 256;                 // first scale slot
constexpr int kStageOutBytes = 4096;        // GEMM2, per epilogue warp: 32 rows x 128 B of fp16 y

template <bool kGemm1>
struct Cfg {
  static constexpr int W = 2;                        // 128-row weight blocks per tile
  static constexpr int kCols = 128 * W;              // UMMA N
  static constexpr int kBBytes = kCols * kRowBytes;
  static constexpr int kSfbBytes = 2048 * W;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  // GEMM2 runs 3 stages: with its fp16 stores it is faster than with 4
  // (1.42 vs 1.49 ms on DeepSeek-V3), and the freed shared memory stages y
  static constexpr int kStages = kGemm1 ? 4 : 3;
  static constexpr int kAccBufs = W == 2 ? 1 : 2;
  static constexpr int kAccCols = kCols;
  // warpgroups (4 warps each): 0 = producer, MMA lane, two idle warps;
  // 1, 2 = the epilogue; 3 = the scale warps
  static constexpr int kEpiWarp0 = 4;
  static constexpr int kEpiWarps = 8;
  static constexpr int kSfWarp0 = kEpiWarp0 + kEpiWarps;  // first scale warp
  static constexpr int kThreads = 32 * (kSfWarp0 + 4);     // 512
  // register split (setmaxnreg): launched with 128 per thread, the producer
  // group and the scale group drop to 64 and the epilogue groups rise to 192:
  // 2 x 128 x 64 + 2 x 128 x 192 = 65536 = 512 x 128
  static constexpr int kLaunchRegs = 128;
  static constexpr int kLowRegs = 64;
  static constexpr int kHighRegs = 192;
  static_assert(2 * 128 * kLowRegs + 2 * 128 * kHighRegs == kThreads * kLaunchRegs,
                "register split must add up to the launch's registers");
  static constexpr int kSlotCols = 16 + 16 * W;      // A scales 16, B scales 16 W
  static constexpr int kOutBytes = kGemm1 ? 0 : kEpiWarps * kStageOutBytes;
  static constexpr uint32_t kIdesc = ptx::idesc_nvf4(kRows, kCols);
  static_assert(kAccBufs * kAccCols <= kSfCol, "accumulators below the scale slots");
  static_assert(kSfCol + kSlotCols * kStages <= int(kTmemCols), "TMEM budget");
};

template <bool kGemm1>
struct __align__(8) SmemCtl {
  static constexpr int S = Cfg<kGemm1>::kStages;
  uint64_t full[S];     // A and B of the stage landed
  uint64_t sf_full[S];  // the stage's scale atoms landed (loaded first)
  uint64_t empty[S];
  uint64_t sf_ready[S];
  uint64_t afull[2];
  uint64_t aempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int32_t sched[2 * kMaxGroups + 2];  // copy of the tile schedule
  int32_t off[kMaxExperts + 1];       // copies of the row offsets and the padded offsets
  int32_t pad[kMaxExperts + 1];
  float gw[kMaxGroups];               // each group's weight tensor scale
};

static_assert(kStageOutBytes % 1024 == 0, "y staging buffers keep the 128-byte swizzle alignment");

template <bool kGemm1>
constexpr size_t smem_bytes() {
  using C = Cfg<kGemm1>;
  return 1024 + size_t(C::kStages) * C::kStageBytes + C::kOutBytes + sizeof(SmemCtl<kGemm1>);
}

struct Tile {
  int g, rb, nb, rows, K;
};

__device__ __forceinline__ Tile decode_tile(int t, const Nvfp4GemmArgs& a, const int32_t* sched,
                                            const int32_t* off, int G) {
  const int32_t* ts = sched + 1;
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ts[mid] <= t) lo = mid; else hi = mid - 1;
  }
  Tile x;
  x.g = sched[G + 2 + lo];
  const int local = t - ts[lo];
  const bool routed = x.g < a.E;
  x.rows = routed ? off[x.g + 1] - off[x.g] : a.T;
  x.K = routed ? a.K_routed : a.K_shared;
  const int mt = (x.rows + kRows - 1) / kRows;
  x.nb = local / mt;
  x.rb = local - x.nb * mt;
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

// Barrier over the epilogue warps that also ORs `v` over them, so that a
// decision to stop is taken by all of them together.
template <int kEpiThreads>
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kEpiThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

template <bool kGemm1>
__global__ void __launch_bounds__(Cfg<kGemm1>::kThreads, 1)
    grouped_gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap map_a0,
                              const __grid_constant__ CUtensorMap map_a1,
                              const __grid_constant__ CUtensorMap map_y0,
                              const __grid_constant__ CUtensorMap map_y1,
                              const Nvfp4GemmArgs args) {
  using C = Cfg<kGemm1>;
  constexpr int kStages = C::kStages;
  constexpr int kStageBytes = C::kStageBytes;
  constexpr int kThreads = C::kThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + kStages * kStageBytes;
  SmemCtl<kGemm1>& c = *reinterpret_cast<SmemCtl<kGemm1>*>(out_stage + C::kOutBytes);
  auto stage_a = [&](int s) { return smem + s * kStageBytes; };
  auto stage_b = [&](int s) { return smem + s * kStageBytes + kABytes; };
  auto stage_sfa = [&](int s) { return smem + s * kStageBytes + kABytes + C::kBBytes; };
  auto stage_sfb = [&](int s) {
    return smem + s * kStageBytes + kABytes + C::kBBytes + kSfaBytes;
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = args.E + args.has_shared;
  const int layer = resolve_layer(args.layer, args.num_layers, args.err);
  const int tab = layer * args.layer_stride;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&c.full[s], 1);
      ptx::mbar_init(&c.sf_full[s], 1);
      ptx::mbar_init(&c.empty[s], 1);
      ptx::mbar_init(&c.sf_ready[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&c.afull[b], 1);
      ptx::mbar_init(&c.aempty[b], C::kEpiWarps);
    }
    ptx::mbar_init(&c.drain, 1);
    c.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&c.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  for (int i = threadIdx.x; i < 2 * G + 2; i += kThreads) c.sched[i] = __ldg(args.sched + i);
  for (int i = threadIdx.x; i <= args.E; i += kThreads) {
    c.off[i] = __ldg(args.offsets + i);
    c.pad[i] = __ldg(args.pad_offsets + i);
  }
  for (int g = threadIdx.x; g < G; g += kThreads) c.gw[g] = *args.w_gs[tab + (kGemm1 ? 2 * g : g)];
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  const int num_tiles = c.sched[0];
  volatile int* abort = &c.abort;
  // each warpgroup changes its register count at the top of its own branch,
  // every warp of the group executing the same setmaxnreg
  const int wgrp = warp >> 2;
  if (wgrp == 0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(C::kLowRegs) : "memory");
  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- TMA producer
      uint32_t it = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort; t += gridDim.x) {
        const Tile x = decode_tile(t, args, c.sched, c.off, G);
        const bool routed = x.g < args.E;
        const int prow0 = (routed ? c.pad[x.g] : 0) + x.rb * kRows;
        const void* map_a = routed ? static_cast<const void*>(&map_a0)
                                   : static_cast<const void*>(&map_a1);
        const int widx = kGemm1 ? 2 * x.g : x.g;
        const CUtensorMap* map_b = args.w_maps + tab + widx;
        const int atoms = x.K / 64;  // scale atoms per 128-row block
        const uint8_t* asf = (routed ? args.a_sf0 : args.a_sf1) + int64_t(prow0 / kRows) * atoms * 512;
        const uint8_t* bsf = args.w_sf[tab + widx] + int64_t(C::W * x.nb) * atoms * 512;
        const int ks_n = x.K / 256;
        bool ok = true;
        for (int ks = 0; ks < ks_n; ++ks, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!ptx::mbar_wait(&c.empty[s], ph ^ 1, abort, args.err)) { ok = false; break; }
          // the scale atoms first, on their own barrier: the scale warps move
          // them into TMEM while A and B are still in flight
          ptx::mbar_arrive_expect_tx(&c.sf_full[s], kSfaBytes + C::kSfbBytes);
          ptx::bulk_load(stage_sfa(s), asf + ks * kSfaBytes, kSfaBytes, &c.sf_full[s]);
#pragma unroll
          for (int h = 0; h < C::W; ++h)  // the tile's 128-row weight blocks
            ptx::bulk_load(stage_sfb(s) + h * 2048, bsf + (int64_t(h) * atoms + 4 * ks) * 512, 2048,
                           &c.sf_full[s]);
          ptx::mbar_arrive_expect_tx(&c.full[s], kABytes + C::kBBytes);
          ptx::tma_load_2d(stage_a(s), map_a, &c.full[s], ks * kRowBytes, prow0);
          ptx::tma_load_2d(stage_b(s), map_b, &c.full[s], ks * kRowBytes, x.nb * C::kCols);
        }
        if (!ok) break;
      }
      if (*abort) {
        const uint32_t first = it > uint32_t(kStages) ? it - kStages : 0;
        for (uint32_t j = first; j < it; ++j) {
          drain_wait(&c.sf_full[j % kStages], (j / kStages) & 1, args.err);
          drain_wait(&c.full[j % kStages], (j / kStages) & 1, args.err);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------- MMA issuer
      uint32_t it = 0, tc = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tc) {
        const Tile x = decode_tile(t, args, c.sched, c.off, G);
        const int buf = tc % C::kAccBufs;
        const uint32_t bph = (tc / C::kAccBufs) & 1;
        if (!ptx::mbar_wait(&c.aempty[buf], bph ^ 1, abort, args.err)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + buf * C::kAccCols;
        const int ks_n = x.K / 256;
        bool ok = true;
        for (int ks = 0; ks < ks_n; ++ks, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          // data in smem, scales in TMEM
          if (!ptx::mbar_wait(&c.full[s], ph, abort, args.err)) { ok = false; break; }
          if (!ptx::mbar_wait(&c.sf_ready[s], ph, abort, args.err)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t slot = tmem_base + kSfCol + C::kSlotCols * s;
          const uint64_t da = ptx::sw128_desc(ptx::smem_u32(stage_a(s)));
          const uint64_t db = ptx::sw128_desc(ptx::smem_u32(stage_b(s)));
#pragma unroll
          for (int m = 0; m < 4; ++m)
            ptx::mma_nvf4(d, da + 2 * m, db + 2 * m, C::kIdesc, slot + 4 * m,
                          slot + 16 + 4 * C::W * m, (ks | m) != 0);
          ptx::mma_commit(&c.empty[s]);
        }
        if (!ok) break;
        ptx::mma_commit(&c.afull[buf]);
      }
      ptx::mma_commit(&c.drain);
      drain_wait(&c.drain, 0, args.err);
    }
  }  // warps 2 and 3 have no role
  } else if (wgrp == 3) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(C::kLowRegs) : "memory");
    // ------------------------------------------------------ scale warps
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const uint32_t lane_q = static_cast<uint32_t>(q * 32) << 16;
    uint32_t it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const Tile x = decode_tile(t, args, c.sched, c.off, G);
      const int ks_n = x.K / 256;
      bool ok = true;
      for (int ks = 0; ks < ks_n; ++ks, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!ptx::mbar_wait(&c.sf_full[s], ph, abort, args.err)) { ok = false; break; }
        const uint32_t slot = tmem_base + kSfCol + C::kSlotCols * s;
        // every lane quarter gets the whole atom layout: lane j, column
        // 4 (W) m + i holds the scales of row 32i + j for MMA m (A at +0, B at +16)
        {
          const uint8_t* src = stage_sfa(s) + lane * 16;
          uint32_t v[16];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint4 w = *reinterpret_cast<const uint4*>(src + 512 * m);
            v[4 * m] = w.x;
            v[4 * m + 1] = w.y;
            v[4 * m + 2] = w.z;
            v[4 * m + 3] = w.w;
          }
          ptx::tmem_st16(slot + lane_q, v);
        }
#pragma unroll
        for (int h = 0; h < C::W; ++h) {
          // B rows 128 h + 32 i + j of MMA m -> column 16 + 4 W m + 4 h + i
          const uint8_t* src = stage_sfb(s) + h * 2048 + lane * 16;
          uint32_t v[16];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint4 w = *reinterpret_cast<const uint4*>(src + 512 * m);
            v[4 * m] = w.x;
            v[4 * m + 1] = w.y;
            v[4 * m + 2] = w.z;
            v[4 * m + 3] = w.w;
          }
          if constexpr (C::W == 1) {
            ptx::tmem_st16(slot + lane_q + 16, v);
          } else {
#pragma unroll
            for (int m = 0; m < 4; ++m)
              ptx::tmem_st4(slot + lane_q + 16 + 8 * m + 4 * h, v[4 * m], v[4 * m + 1],
                            v[4 * m + 2], v[4 * m + 3]);
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&c.sf_ready[s]);
      }
      if (!ok) break;
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(C::kHighRegs) : "memory");
    // ------------------------------------------------------ epilogue warps
    const int q = warp & 3;
    const int r = q * 32 + lane;  // row of the tile (TMEM lane)
    const int half = (warp - C::kEpiWarp0) / 4;  // which 128 (GEMM1: 64) of the tile's columns
    const float gx = __ldg(args.act_scales + 2 * layer);
    const float gh = __ldg(args.act_scales + 2 * layer + 1);
    uint32_t tc = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tc) {
      const Tile x = decode_tile(t, args, c.sched, c.off, G);
      const bool routed = x.g < args.E;
      const int buf = tc % C::kAccBufs;
      const uint32_t bph = (tc / C::kAccBufs) & 1;
      // this tile's scale and (GEMM2) row weight, loaded before the wait
      const float gw = c.gw[x.g];
      const int valid_rows = x.rows - x.rb * kRows;
      const int64_t wrow0 = (routed ? int64_t(c.off[x.g]) : 0) + int64_t(x.rb) * kRows + q * 32;
      const int valid_w = valid_rows - q * 32;
      const bool valid = lane < valid_w;
      const float rw = (!kGemm1 && valid && routed && args.row_weight)
                           ? __ldg(args.row_weight + wrow0 + lane) : 1.0f;
      const bool ok = ptx::mbar_wait(&c.afull[buf], bph, abort, args.err);
      if (epi_any<32 * C::kEpiWarps>(!ok || *abort)) break;  // uniform over the epilogue warps
      ptx::tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::kAccCols;
      if constexpr (kGemm1) {
        // accumulator columns [0,128) gate, [128,256) up of h columns
        // [128 nb, 128 nb + 128); this warp: h columns 64 half + [0, 64), in
        // two chunks of 32, the single accumulator released once both are read
        float h[2][32];
        {
          uint32_t g0[32], u0[32], g1[32], u1[32];
          ptx::tmem_ld32(taddr + 64 * half, g0);
          ptx::tmem_ld32(taddr + 128 + 64 * half, u0);
          ptx::tmem_ld32(taddr + 64 * half + 32, g1);
          ptx::tmem_ld32(taddr + 128 + 64 * half + 32, u1);
          ptx::tmem_ld_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&c.aempty[buf]);  // accumulator free
          const float alpha = __fmul_rn(gx, gw);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            h[0][i] = silu_f(__uint_as_float(g0[i]) * alpha) * (__uint_as_float(u0[i]) * alpha);
            h[1][i] = silu_f(__uint_as_float(g1[i]) * alpha) * (__uint_as_float(u1[i]) * alpha);
          }
        }
        const int n_h = routed ? args.N_routed : args.N_shared;  // I or I_shared
        const int64_t p = (routed ? c.pad[x.g] : 0) + int64_t(x.rb) * kRows + r;
        uint8_t* codes = static_cast<uint8_t*>(routed ? args.out0 : args.out1) + p * (n_h / 2) +
                         x.nb * 64 + half * 32;
        uint8_t* sf = routed ? args.out_sf0 : args.out_sf1;
        uint32_t scw = 0;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float b0[16], b1[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            b0[i] = h[hh][i];
            b1[i] = h[hh][16 + i];
          }
          uint2 q0, q1;
          const uint32_t s0 = nvfp4::quantize16(b0, gh, q0);
          const uint32_t s1 = nvfp4::quantize16(b1, gh, q1);
          *reinterpret_cast<uint4*>(codes + hh * 16) = make_uint4(q0.x, q0.y, q1.x, q1.y);
          scw |= (s0 | (s1 << 8)) << (16 * hh);
        }
        // the 4 scales of h blocks 8 nb + 4 half + [0, 4): one word of the atom
        *reinterpret_cast<uint32_t*>(sf + nvfp4::sf_offset(p, 8 * x.nb + 4 * half, n_h)) = scw;
      } else {
        // y columns 256 nb + 128 half + [0, 128) of this warp's 32 rows, as fp16
        // with a power-of-two scale s = 2^(floor(log2 amax) - 14) per 32 columns
        // (|y| / s < 2^15); packed right after each TMEM load so that the single
        // accumulator is released after the fourth
        const float alpha = __fmul_rn(gh, gw);
        const int n_out = args.N_routed;  // H
        const float wa = rw * alpha;
        uint32_t pk[4][16];
        float scl[4];
        uint32_t a128[4][32];
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) ptx::tmem_ld32(taddr + 128 * half + 32 * cb, a128[cb]);
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&c.aempty[buf]);  // accumulator free
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          const uint32_t* a32 = a128[cb];
          float amax = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(wa * __uint_as_float(a32[j])));
          int sb = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 14;
          sb = sb < 1 ? 1 : sb;
          scl[cb] = __uint_as_float(static_cast<uint32_t>(sb) << 23);
          const float inv = __uint_as_float(static_cast<uint32_t>(254 - sb) << 23);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __half2 hh = __floats2half2_rn(wa * __uint_as_float(a32[2 * e]) * inv,
                                                 wa * __uint_as_float(a32[2 * e + 1]) * inv);
            pk[cb][e] = *reinterpret_cast<const uint32_t*>(&hh);
          }
        }
        const int col0 = x.nb * C::kCols + 128 * half;
        __half* y = static_cast<__half*>(routed ? args.out0 : args.out1) + col0;
        float* ys = (routed ? args.out_scales0 : args.out_scales1) + col0 / 32;
        // the row's 4 scales are contiguous: one 16-byte store
        if (valid)
          __stcs(reinterpret_cast<float4*>(ys + (wrow0 + lane) * (n_out / 32)),
                 make_float4(scl[0], scl[1], scl[2], scl[3]));
        uint8_t* stg = out_stage + (warp - C::kEpiWarp0) * kStageOutBytes;
        // the buffer is rewritten only once the previous TMA stores have read it
        if (lane == 0) ptx::bulk_wait_read_all();
        __syncwarp();
        if (valid_w >= 32) {
          // all 32 rows are the segment's own: TMA stores of the 32-row x
          // 64-column boxes, row `lane` written in the 128-byte swizzle
          const void* ymap = routed ? static_cast<const void*>(&map_y0)
                                    : static_cast<const void*>(&map_y1);
#pragma unroll
          for (int c64 = 0; c64 < 2; ++c64) {
            if (c64 == 1) {
              if (lane == 0) ptx::bulk_wait_read_all();
              __syncwarp();
            }
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16) {
              const uint32_t* v = &pk[2 * c64 + (c16 >> 2)][4 * (c16 & 3)];
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((c16 ^ (lane & 7)) << 4)) =
                  make_uint4(v[0], v[1], v[2], v[3]);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_2d(ymap, stg, col0 + 64 * c64, static_cast<int32_t>(wrow0));
              ptx::bulk_commit();
            }
          }
        } else {
          // the segment's last rows: staged stores, 64 columns (128 bytes of a
          // row) at a time, 4 rows per round through 512 bytes of the buffer,
          // so that each store instruction writes 4 whole 128-byte lines
          uint4* st4 = reinterpret_cast<uint4*>(stg);
#pragma unroll
          for (int c64 = 0; c64 < 2; ++c64) {
#pragma unroll
            for (int r4 = 0; r4 < 8; ++r4) {
              if ((lane >> 2) == r4) {
                const int l = lane & 3;
#pragma unroll
                for (int c16 = 0; c16 < 8; ++c16) {
                  const uint32_t* v = &pk[2 * c64 + (c16 >> 2)][4 * (c16 & 3)];
                  st4[l * 8 + (c16 ^ l)] = make_uint4(v[0], v[1], v[2], v[3]);
                }
              }
              __syncwarp();
              const int i = lane >> 3, cc = lane & 7;
              const uint4 val = st4[i * 8 + (cc ^ i)];
              const int row = 4 * r4 + i;
              if (row < valid_w)  // streaming: y is read once, by the combine
                __stcs(reinterpret_cast<uint4*>(y + (wrow0 + row) * n_out + 64 * c64 + cc * 8),
                       val);
              __syncwarp();
            }
          }
        }
      }
    }
    if (!kGemm1 && lane == 0) ptx::bulk_wait_all();  // every TMA store of y has completed
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool kGemm1>
cudaError_t launch_impl(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& y0,
                        const CUtensorMap& y1, const Nvfp4GemmArgs& args, int grid,
                        cudaStream_t stream) {
  constexpr size_t smem = smem_bytes<kGemm1>();
  static_assert(smem <= 232448, "shared memory budget");
  const void* fn = reinterpret_cast<const void*>(grouped_gemm_nvfp4_kernel<kGemm1>);
  cudaError_t e = ensure_smem_attr(fn, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // the register split assumes the block is launched with kLaunchRegs per
  // thread; with fewer, the epilogue's setmaxnreg.inc could never be served
  cudaFuncAttributes fa{};
  e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != Cfg<kGemm1>::kLaunchRegs) {
    set_last_error_text("NVFP4 GEMM kernel built with an unexpected register count");
    return cudaErrorInvalidConfiguration;
  }
  grouped_gemm_nvfp4_kernel<kGemm1><<<grid, Cfg<kGemm1>::kThreads, smem, stream>>>(a0, a1, y0, y1,
                                                                                    args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm_nvfp4(bool gemm1, const CUtensorMap& map_a0,
                                      const CUtensorMap& map_a1, const CUtensorMap& map_y0,
                                      const CUtensorMap& map_y1, const Nvfp4GemmArgs& args,
                                      int grid, cudaStream_t stream) {
  return gemm1 ? launch_impl<true>(map_a0, map_a1, map_y0, map_y1, args, grid, stream)
               : launch_impl<false>(map_a0, map_a1, map_y0, map_y1, args, grid, stream);
}

}  // namespace moe
