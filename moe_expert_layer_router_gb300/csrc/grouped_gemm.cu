// Persistent grouped GEMM on the sm_103a tensor cores: CTA pairs (tcgen05
// cta_group::2), TMEM accumulators, TMA loads.
//
// One launch covers every expert of a layer: the hidden-state rows of expert
// e (its segment of the permuted activations) times that expert's weight
// matrix, read from its own allocation through a per-expert TMA descriptor
// (the grouped matrix multiplication of "ASAP: A DiSaggregated and
// Asynchronous Inference System for MoE Prefill", section 3.4.2, with the
// per-expert weight list of "DWDP: Distributed Weight Data Parallelism for
// High-Performance LLM Inference on NVL72", section 4.2).  The shared expert
// is one more group whose rows are the unpermuted tokens.
//
//   GEMM1 (kSwiGLU):  h = silu(A W_gate^T) * (A W_up^T)   bf16 out
//   GEMM2:            y = row_weight * (A W_down^T)       fp32 out, or fp16 with
//                     a power-of-two scale per 32 columns (the layer forward)
// (y is never rounded to bf16: the k expert rows of a token are rounded to bf16
// only once, after the combine has summed them.  Scaled fp16 keeps 11
// significant bits of every value at half the bytes of fp32.)
//
// Work unit: a 256-row x 256-column pair tile computed by the two CTAs of a
// cluster with one 256x256x16 MMA per 16-wide K step.  Each CTA loads its own
// 128 rows of A and one half of B, so a stage is 32 KB per CTA (instead of 48
// KB for a single-CTA 128x256 tile) and the ring holds 5 stages (6 were
// slower under the power cap: GEMM1 6.34 vs 6.07 ms, GEMM2 3.38 vs 3.26 ms on
// DeepSeek-V3; 4 were slower still).  B halves:
//   GEMM1: CTA r loads W_gate and W_up rows [128 n + 64 r, +64) (64 + 64 rows),
//          so TMEM columns are [gate | up] of output columns 128 n + 64 r + [0,64)
//   GEMM2: CTA r loads W_down rows [256 n + 128 r, +128)
// An expert's last tile, when at most 128 rows are left, is a half tile: an
// M=128 pair MMA (64 rows per CTA, half the time of M=256).  Its TMEM layout
// (measured): CTA r holds rows 64 r + [0,64); lanes 0-63 carry the first 128
// output columns of the pair and lanes 64-127 the same rows' other 128, both in
// TMEM columns 0-127.  Either way every epilogue thread owns one output row and
// holds both the gate and the up value of each of its columns.
// Rows of an A box past the tile's expert segment are loaded as zeros, through
// the expert's copy of the A tensor map whose row extent the plan kernel cut
// at the segment's end: the kernels run into the GPU's power cap, and products
// with zeros draw less power than products with the next expert's rows.
//
// Warp roles per CTA (192 threads, one CTA per SM):
//   warp 0      TMA producer (one lane), completing on the even CTA's barriers
//   warp 1      pair-collective TMEM allocation; in the even CTA one lane
//               issues the pair MMAs and multicasts their completion
//   warps 2..5  epilogue: TMEM -> registers -> SwiGLU / row scale -> HBM
// TMEM holds two 256-column fp32 accumulators, so the epilogue of tile i
// overlaps the MMAs of tile i+1.  Tiles come from a device-built schedule
// (heaviest group first) and are dealt to the persistent pairs round robin.
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// Ring depth of each GEMM (stages of 32 KB per CTA).
constexpr int kStagesG1 = 5;
constexpr int kStagesG2 = 5;
constexpr int kStages = kStagesG1 > kStagesG2 ? kStagesG1 : kStagesG2;  // barrier arrays
constexpr int kThreads = 192;
constexpr int kPairRows = kGemmTileRows;      // 256 rows per pair tile (128 per CTA)
static_assert(kPairRows == 2 * kTileM, "a pair tile is two CTA tiles");
static_assert(2 * kGemmBRows == 256 && kGemm1TileN == kGemmBRows && kGemm2TileN == 2 * kGemmBRows,
              "each CTA loads one 128-row half of the 256-row B operand");
constexpr int kABytes = kTileM * kTileK * 2;  // 16 KB: this CTA's 128 rows
constexpr int kBBytes = kGemmBRows * kTileK * 2;  // 16 KB: this CTA's half of B (TMA box)
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kTileN = 256;                   // UMMA N (both CTAs' B halves)
constexpr uint32_t kIdescFull = ptx::idesc_bf16(kPairRows, kTileN);
constexpr uint32_t kIdescHalf = ptx::idesc_bf16(kTileM, kTileN);
constexpr uint32_t kTmemCols = 512;           // two 256-column fp32 accumulators
constexpr uint16_t kBothCtas = 0x3;

struct __align__(8) SmemCtl {
  uint64_t full[kStages];    // even CTA: both CTAs' loads of a stage landed
  uint64_t empty[kStages];   // both CTAs: the pair MMAs of a stage are done
  uint64_t tfull[2];         // both CTAs: an accumulator is complete
  uint64_t tempty[2];        // even CTA: both epilogues drained an accumulator
  uint64_t drain;
  uint64_t stall;            // failure-path test only: never arrived on
  uint32_t tmem_base;
  int abort;
  int32_t sched[2 * kMaxGroups + 2];
  int32_t offsets[kMaxExperts + 1];
};

// Epilogue staging: each epilogue warp transposes its 32 rows x 32 columns
// through shared memory so global stores cover whole lines of a few rows.
constexpr int kStageOutBytes = 4096;  // per epilogue warp (32 rows x 128 B)
template <bool kSwiGLU>
constexpr int stages_of() { return kSwiGLU ? kStagesG1 : kStagesG2; }
template <bool kSwiGLU>
constexpr size_t smem_bytes() {
  return 1024 + size_t(stages_of<kSwiGLU>()) * kStageBytes + 4 * kStageOutBytes + sizeof(SmemCtl);
}

// A group's tiles run in chunks of kChunkM m-tiles: all n-blocks of one chunk
// (m-tiles of one n-block consecutive) before the next chunk.  A group with
// many rows (the shared expert, whose rows are all T tokens, or a hot expert)
// then keeps a few m-tiles of A in L2 while every n-block reads them, instead
// of streaming all its rows once per n-block; groups of at most kChunkM m-tiles
// run n-block by n-block as before.
constexpr int kChunkM = 8;

struct Tile {
  int g, m_blk, n_blk, rows, row0, K, N;
  bool half;  // at most 128 rows left: M=128 pair MMA, 64 rows per CTA
};

__device__ __forceinline__ Tile decode_tile(int t, const SmemCtl& c, const GemmArgs& a, int G,
                                            int tile_n) {
  const int32_t* ts = c.sched + 1;
  int lo = 0, hi = G - 1;
  while (lo < hi) {  // last slot whose first tile is <= t
    const int mid = (lo + hi + 1) >> 1;
    if (ts[mid] <= t) lo = mid; else hi = mid - 1;
  }
  Tile x;
  x.g = c.sched[G + 2 + lo];
  const int local = t - ts[lo];
  const bool routed = x.g < a.E;
  x.rows = routed ? c.offsets[x.g + 1] - c.offsets[x.g] : a.T;
  x.row0 = routed ? c.offsets[x.g] : 0;
  x.K = routed ? a.K_routed : a.K_shared;
  x.N = routed ? a.N_routed : a.N_shared;
  const int mt = (x.rows + kPairRows - 1) / kPairRows;
  const int nt = (x.N + tile_n - 1) / tile_n;
  const int full_chunks = mt / kChunkM;
  int chunk = local / (kChunkM * nt), cm = kChunkM;
  if (chunk >= full_chunks) {  // the last, partial chunk (the only one when mt < kChunkM)
    chunk = full_chunks;
    cm = mt - full_chunks * kChunkM;
  }
  const int r = local - chunk * kChunkM * nt;
  x.n_blk = r / cm;
  x.m_blk = chunk * kChunkM + (r - x.n_blk * cm);
  x.half = x.rows - x.m_blk * kPairRows <= kTileM;
  return x;
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Bounded wait without the abort short-cut, used only while draining work
// that is certain to complete before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kWaitTimeoutNs) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

// B operand of this CTA for a tile: GEMM1 -- gate and up rows [128 n + 64 r,
// +64) (two boxes); GEMM2 -- W_down rows [256 n + 128 r, +128).
template <bool kSwiGLU>
__device__ __forceinline__ void b_operand(const Tile& x, uint32_t rank, const CUtensorMap* bmaps,
                                          const CUtensorMap*& mb, int& b_row) {
  if (kSwiGLU) {
    mb = bmaps + 2 * x.g;
    b_row = x.n_blk * kGemm1TileN + int(rank) * (kGemmBRows / 2);
  } else {
    mb = bmaps + x.g;
    b_row = x.n_blk * kGemm2TileN + int(rank) * kGemmBRows;
  }
}

template <bool kSwiGLU>
__device__ __forceinline__ void load_b_impl(uint8_t* bs, const CUtensorMap* mb, uint32_t fb,
                                            int kb, int b_row) {
  if (kSwiGLU) {
    ptx::tma_load_2d_pair(bs, mb, fb, kb * kTileK, b_row);
    ptx::tma_load_2d_pair(bs + kBBytes / 2, mb + 1, fb, kb * kTileK, b_row);
  } else {
    ptx::tma_load_2d_pair(bs, mb, fb, kb * kTileK, b_row);
  }
}

template <bool kSwiGLU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_bf16_kernel(const __grid_constant__ CUtensorMap map_a0,
                             const __grid_constant__ CUtensorMap map_a1, const GemmArgs args) {
  constexpr int kStages = stages_of<kSwiGLU>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_tiles = smem;
  uint8_t* b_tiles = smem + kStages * kABytes;
  uint8_t* out_stage = smem + kStages * kStageBytes;
  SmemCtl& c = *reinterpret_cast<SmemCtl*>(out_stage + 4 * kStageOutBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0: issues the pair MMAs
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  const int G = args.E + args.has_shared;
  constexpr int kTileNOut = kSwiGLU ? kGemm1TileN : kGemm2TileN;  // output columns per tile
  // weight descriptors of this call's layer (layer stacks index their table)
  const CUtensorMap* bmaps =
      args.b_maps + resolve_layer(args.layer, args.num_layers, args.err) * args.layer_stride;

  for (int i = threadIdx.x; i < sched_ints(G); i += kThreads) c.sched[i] = args.sched[i];
  for (int i = threadIdx.x; i <= args.E; i += kThreads) c.offsets[i] = args.offsets[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&c.full[s], 1);
      ptx::mbar_init(&c.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&c.tfull[s], 1);
      ptx::mbar_init(&c.tempty[s], 8);  // 4 epilogue warps in each CTA
    }
    ptx::mbar_init(&c.drain, 1);
    ptx::mbar_init(&c.stall, 1);
    c.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&c.tmem_base, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  if (threadIdx.x == 0) {
    ptx::prefetch_tmap(&map_a0);
    ptx::prefetch_tmap(&map_a1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before anyone signals them
  ptx::tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  const int num_tiles = c.sched[0];
  volatile int* abort = &c.abort;

  if (warp == 0) {
    // -------------------------------------------------- TMA producer (both CTAs)
    const uint32_t full0 = ptx::mapa(ptx::smem_u32(&c.full[0]), 0);
    uint32_t it = 0;
    if (args.gather_rows == nullptr) {
      // tile loads: one lane issues everything
      if (lane == 0) {
        for (int t = pair; t < num_tiles && !*abort; t += num_pairs) {
          const Tile x = decode_tile(t, c, args, G, kTileNOut);
          const void* map_a = x.g < args.E ? static_cast<const void*>(&map_a0)
                                           : static_cast<const void*>(&map_a1);
          const CUtensorMap* mb;
          int b_row;
          b_operand<kSwiGLU>(x, rank, bmaps, mb, b_row);
          // A rows of this CTA: 128 (full tile) or 64 (half tile; the box still
          // brings 128 rows, the MMA reads the first 64)
          const int a_row = x.row0 + x.m_blk * kPairRows +
                            int(rank) * (x.half ? kTileM / 2 : kTileM);
          // A box rows past the end of the expert's rows (the MMA computes them,
          // the epilogue discards them) come through the expert's copy of the A
          // map whose row extent ends there (written by the plan kernel), so the
          // TMA fills them with zeros: a product with zeros draws less power
          // than one with the next expert's rows.
          if (args.amap != nullptr && x.g < args.E && a_row + kTileM > x.row0 + x.rows) {
            const uint8_t* cut = args.amap + size_t(x.g) * 128;
            ptx::fence_tensormap_acquire(cut);
            map_a = cut;
          }
          const int kb_n = x.K / kTileK;
          bool ok = true;
          for (int kb = 0; kb < kb_n; ++kb, ++it) {
            const int s = it % kStages;
            const uint32_t ph = (it / kStages) & 1;
            if (!ptx::mbar_wait(&c.empty[s], ph ^ 1, abort, args.err)) { ok = false; break; }
            if (leader) ptx::mbar_arrive_expect_tx(&c.full[s], 2 * kStageBytes);
            const uint32_t fb = full0 + s * 8;
            ptx::tma_load_2d_pair(a_tiles + s * kABytes, map_a, fb, kb * kTileK, a_row);
            load_b_impl<kSwiGLU>(b_tiles + s * kBBytes, mb, fb, kb, b_row);
          }
          if (!ok) break;
        }
      }
    } else {
      // GEMM1 fed straight from the unpermuted tokens: each lane gathers 4 of
      // this CTA's routed A rows per stage by token index.  Lane 0 takes every
      // barrier decision and broadcasts it, so the warp never diverges.
      bool stop = false;
      for (int t = pair; t < num_tiles && !stop; t += num_pairs) {
        const Tile x = decode_tile(t, c, args, G, kTileNOut);
        const bool routed = x.g < args.E;
        const int cta_rows = x.half ? kTileM / 2 : kTileM;
        const void* map_a = routed ? static_cast<const void*>(&map_a0)
                                   : static_cast<const void*>(&map_a1);
        const CUtensorMap* mb;
        int b_row;
        b_operand<kSwiGLU>(x, rank, bmaps, mb, b_row);
        const int a_row = x.row0 + x.m_blk * kPairRows + int(rank) * cta_rows;
        // gathers bring exactly the rows used; tile loads (shared expert) 128
        const uint32_t a_bytes = routed ? uint32_t(cta_rows) * 128u : uint32_t(kABytes);
        int tok[4] = {0, 0, 0, 0};
        const bool g_lane = routed && lane < cta_rows / 4;
        if (g_lane) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int pr = a_row + 4 * lane + j;  // permuted row; past the segment: any token
            tok[j] = pr < args.R ? __ldg(args.gather_rows + pr) : 0;
          }
        }
        const int kb_n = x.K / kTileK;
        for (int kb = 0; kb < kb_n; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          int ok = 1;
          if (lane == 0) ok = ptx::mbar_wait(&c.empty[s], ph ^ 1, abort, args.err) ? 1 : 0;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            stop = true;
            break;
          }
          const uint32_t fb = full0 + s * 8;
          if (lane == 0 && leader) ptx::mbar_arrive_expect_tx(&c.full[s], 2 * (a_bytes + kBBytes));
          if (routed) {
            if (g_lane)
              ptx::tma_gather4_pair(a_tiles + s * kABytes + lane * 512, map_a, fb, kb * kTileK,
                                    tok[0], tok[1], tok[2], tok[3]);
          } else if (lane == 0) {
            ptx::tma_load_2d_pair(a_tiles + s * kABytes, map_a, fb, kb * kTileK, a_row);
          }
          if (lane == 0) load_b_impl<kSwiGLU>(b_tiles + s * kBBytes, mb, fb, kb, b_row);
        }
        if (__shfl_sync(0xffffffffu, *abort ? 1 : 0, 0)) stop = true;
      }
    }
    if (lane == 0 && *abort && leader) {
      // Both CTAs' loads of a stage complete on the even CTA's barrier: wait
      // for the stages issued last so no copy is in flight at exit.
      const uint32_t first = it > kStages ? it - kStages : 0;
      for (uint32_t j = first; j < it; ++j)
        drain_wait(&c.full[j % kStages], (j / kStages) & 1, args.err);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------ pair MMA issuer
      uint32_t it = 0;
      int local = 0;
      for (int t = pair; t < num_tiles; t += num_pairs, ++local) {
        const Tile x = decode_tile(t, c, args, G, kTileNOut);
        const int acc = local & 1;
        const uint32_t acc_ph = (local >> 1) & 1;
        if (!ptx::mbar_wait(&c.tempty[acc], acc_ph ^ 1, abort, args.err)) break;
        // failure-path test: before its first tile, pair 0 waits on a barrier
        // that nothing arrives on; the bounded wait gives up, sets the timeout
        // bit and the abort flag, and the pair abandons its tiles (every load
        // already issued still lands and is drained below)
        if (args.stall_test && pair == 0 && local == 0 &&
            !ptx::mbar_wait(&c.stall, 0, abort, args.err))
          break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kTileN;
        const uint32_t idesc = x.half ? kIdescHalf : kIdescFull;
        const int kb_n = x.K / kTileK;
        bool ok = true;
        for (int kb = 0; kb < kb_n; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!ptx::mbar_wait(&c.full[s], ph, abort, args.err)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint64_t da = ptx::sw128_desc(ptx::smem_u32(a_tiles + s * kABytes));
          const uint64_t db = ptx::sw128_desc(ptx::smem_u32(b_tiles + s * kBBytes));
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k)
            ptx::mma_f16_pair(d_tmem, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);
          ptx::mma_commit_pair_mc(&c.empty[s], kBothCtas);
        }
        if (!ok) break;
        ptx::mma_commit_pair_mc(&c.tfull[acc], kBothCtas);
      }
      // Every pair MMA issued by this thread has finished once `drain` flips.
      ptx::mma_commit_pair_mc(&c.drain, 0x1);
      drain_wait(&c.drain, 0, args.err);
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    const uint32_t tempty0 = ptx::mapa(ptx::smem_u32(&c.tempty[0]), 0);
    int local = 0;
    for (int t = pair; t < num_tiles; t += num_pairs, ++local) {
      const Tile x = decode_tile(t, c, args, G, kTileNOut);
      const int acc = local & 1;
      const uint32_t acc_ph = (local >> 1) & 1;
      if (!ptx::mbar_wait(&c.tfull[acc], acc_ph, abort, args.err)) break;
      ptx::tc_fence_after();
      // Row of this thread and, for half tiles, which 128-column half of the
      // pair's N it holds (warp-uniform: lane quarters 0-1 vs 2-3).  Rows of
      // this warp are m_base + 0..31.
      const int hs = x.half ? (r >> 6) : 0;
      const int m_base = x.m_blk * kPairRows +
                         (x.half ? int(rank) * (kTileM / 2) + ((q * 32) & 63) : int(rank) * kTileM + q * 32);
      const int m = m_base + lane;
      const bool valid = m < x.rows;
      const bool routed = x.g < args.E;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kTileN;
      if (m_base >= x.rows) {
        // all 32 rows of this warp lie past the tile's rows: nothing to read or
        // write (skipping the TMEM loads and the math saves power)
      } else if (kSwiGLU) {
        // full tile: TMEM columns [g | u] of output columns 128 n + [0,64), then
        // [g | u] of 128 n + [64,128); half tile: one [g | u] block, the one of
        // CTA-half hs.  Each 32-column chunk: 32 rows x 64 B staged, then written
        // 8 rows x 64 B per store instruction.
        uint4* st16 = reinterpret_cast<uint4*>(out_stage + (warp - 2) * kStageOutBytes);
        __nv_bfloat16* base = routed ? static_cast<__nv_bfloat16*>(args.out0) +
                                           int64_t(x.row0) * x.N
                                     : static_cast<__nv_bfloat16*>(args.out1);
        const int nblocks = x.half ? 1 : 2;
#pragma unroll 1
        for (int blk = 0; blk < nblocks; ++blk) {
          const int out_col = x.n_blk * kGemm1TileN + (x.half ? hs : blk) * 64;
#pragma unroll 1
          for (int cb = 0; cb < 2; ++cb) {
            uint32_t gr[32], ur[32];
            ptx::tmem_ld32(taddr + blk * 128 + cb * 32, gr);
            ptx::tmem_ld32(taddr + blk * 128 + 64 + cb * 32, ur);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t p[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = v * 8 + e * 2;
                const float h0 = silu_f(__uint_as_float(gr[i])) * __uint_as_float(ur[i]);
                const float h1 = silu_f(__uint_as_float(gr[i + 1])) * __uint_as_float(ur[i + 1]);
                p[e] = pack_bf16(h0, h1);
              }
              st16[lane * 4 + (v ^ ((lane >> 1) & 3))] = make_uint4(p[0], p[1], p[2], p[3]);
            }
            __syncwarp();
#pragma unroll
            for (int it = 0; it < 4; ++it) {
              const int i = it * 8 + (lane >> 2), vv = lane & 3;
              const uint4 val = st16[i * 4 + (vv ^ ((i >> 1) & 3))];
              if (m_base + i < x.rows)
                *reinterpret_cast<uint4*>(base + int64_t(m_base + i) * x.N + out_col + cb * 32 +
                                          vv * 8) = val;
            }
            __syncwarp();
          }
        }
      } else if (args.out_scales0 != nullptr) {
        // fp16 y: each 32-column chunk of a row is scaled by a power of two
        // s = 2^(floor(log2 amax) - 14), so that |y| / s < 2^15 fits fp16 with
        // its full 11-bit precision; s goes to out_scales[row][column / 32].
        // Staged and stored like h: 8 rows x 64 B per store instruction.
        uint4* st16 = reinterpret_cast<uint4*>(out_stage + (warp - 2) * kStageOutBytes);
        __half* base = routed ? static_cast<__half*>(args.out0) + int64_t(x.row0) * x.N
                              : static_cast<__half*>(args.out1);
        const int nsc = x.N / 32;
        float* sbase = routed ? args.out_scales0 + int64_t(x.row0) * nsc : args.out_scales1;
        const float w = (valid && routed && args.row_weight) ? args.row_weight[x.row0 + m] : 1.0f;
        const int col0 = x.n_blk * kGemm2TileN + hs * 128;
        const int ncb = (x.half ? 128 : kGemm2TileN) / 32;
#pragma unroll 1
        for (int cb = 0; cb < ncb; ++cb) {
          if (col0 + cb * 32 >= x.N) break;  // warp-uniform
          uint32_t yr[32];
          ptx::tmem_ld32(taddr + cb * 32, yr);
          ptx::tmem_ld_wait();
          float amax = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(w * __uint_as_float(yr[j])));
          // biased exponent of the scale, kept a normal float (amax = 0 gives the
          // smallest normal; every value is then 0)
          int sb = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 14;
          sb = sb < 1 ? 1 : sb;
          const float scale = __uint_as_float(static_cast<uint32_t>(sb) << 23);
          const float inv = __uint_as_float(static_cast<uint32_t>(254 - sb) << 23);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = v * 8 + e * 2;
              const __half2 hh = __floats2half2_rn(w * __uint_as_float(yr[i]) * inv,
                                                   w * __uint_as_float(yr[i + 1]) * inv);
              p[e] = *reinterpret_cast<const uint32_t*>(&hh);
            }
            st16[lane * 4 + (v ^ ((lane >> 1) & 3))] = make_uint4(p[0], p[1], p[2], p[3]);
          }
          if (valid) sbase[int64_t(m) * nsc + (col0 >> 5) + cb] = scale;
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int i = it * 8 + (lane >> 2), vv = lane & 3;
            const uint4 val = st16[i * 4 + (vv ^ ((i >> 1) & 3))];
            if (m_base + i < x.rows)
              *reinterpret_cast<uint4*>(base + int64_t(m_base + i) * x.N + col0 + cb * 32 +
                                        vv * 8) = val;
          }
          __syncwarp();
        }
      } else {
        // full tile: 256 TMEM columns = output columns 256 n + [0,256);
        // half tile: 128 TMEM columns = output columns 256 n + 128 hs + [0,128).
        // Each 32-column chunk: 32 rows x 128 B staged, then written 4 rows x
        // 128 B per store instruction.
        float4* st4 = reinterpret_cast<float4*>(out_stage + (warp - 2) * kStageOutBytes);
        float* base = routed ? static_cast<float*>(args.out0) + int64_t(x.row0) * x.N
                             : static_cast<float*>(args.out1);
        const float w = (valid && routed && args.row_weight) ? args.row_weight[x.row0 + m] : 1.0f;
        const int col0 = x.n_blk * kGemm2TileN + hs * 128;
        const int ncb = (x.half ? 128 : kGemm2TileN) / 32;
#pragma unroll 1
        for (int cb = 0; cb < ncb; ++cb) {
          if (col0 + cb * 32 >= x.N) break;  // warp-uniform
          uint32_t yr[32];
          ptx::tmem_ld32(taddr + cb * 32, yr);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int v = 0; v < 8; ++v)
            st4[lane * 8 + (v ^ (lane & 7))] =
                make_float4(w * __uint_as_float(yr[4 * v]), w * __uint_as_float(yr[4 * v + 1]),
                            w * __uint_as_float(yr[4 * v + 2]), w * __uint_as_float(yr[4 * v + 3]));
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int i = it * 4 + (lane >> 3), vv = lane & 7;
            const float4 val = st4[i * 8 + (vv ^ (i & 7))];
            if (m_base + i < x.rows)
              *reinterpret_cast<float4*>(base + int64_t(m_base + i) * x.N + col0 + cb * 32 +
                                         vv * 4) = val;
          }
          __syncwarp();
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(tempty0 + acc * 8);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the pair's MMAs, copies and remote arrivals are over
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <bool kSwiGLU>
cudaError_t launch_impl(const CUtensorMap& a0, const CUtensorMap& a1, const GemmArgs& args, int grid,
                        cudaStream_t stream) {
  constexpr size_t kSmem = smem_bytes<kSwiGLU>();
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(grouped_gemm_bf16_kernel<kSwiGLU>),
                                   static_cast<int>(kSmem));
  if (e != cudaSuccess) return e;
  grouped_gemm_bf16_kernel<kSwiGLU><<<grid, kThreads, kSmem, stream>>>(a0, a1, args);
  return cudaGetLastError();
}

template <bool kSwiGLU>
int max_pairs() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<kSwiGLU>();
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_bf16_kernel<kSwiGLU>, &cfg) != cudaSuccess)
    return 0;
  return n;
}

}  // namespace

int grouped_gemm_grid(int sm_count) {
  // One CTA pair for every pair of SMs that can hold one at the same time.
  ensure_smem_attr(reinterpret_cast<const void*>(grouped_gemm_bf16_kernel<true>),
                   static_cast<int>(smem_bytes<true>()));
  ensure_smem_attr(reinterpret_cast<const void*>(grouped_gemm_bf16_kernel<false>),
                   static_cast<int>(smem_bytes<false>()));
  int pairs = max_pairs<true>();
  const int p2 = max_pairs<false>();
  if (p2 > 0 && (pairs <= 0 || p2 < pairs)) pairs = p2;
  if (pairs <= 0 || pairs > sm_count / 2) pairs = sm_count / 2;
  return 2 * (pairs > 0 ? pairs : 1);
}

cudaError_t launch_grouped_gemm(bool swiglu, const CUtensorMap& map_a0, const CUtensorMap& map_a1,
                                const GemmArgs& args, int grid, cudaStream_t stream) {
  return swiglu ? launch_impl<true>(map_a0, map_a1, args, grid, stream)
                : launch_impl<false>(map_a0, map_a1, args, grid, stream);
}

}  // namespace moe
