// Persistent grouped GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
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
//   GEMM1 (kSwiGLU):  h = silu(A W_gate^T) * (A W_up^T)      tile 128 x (128 gate + 128 up), bf16 out
//   GEMM2:            y = row_weight * (A W_down^T)          tile 128 x 256, fp32 out
// (y stays fp32 so that the k expert rows of a token are rounded to bf16 only
// once, after the combine has summed them.)
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer (one lane): A tile + B tile(s) per 64-wide K step
//   warp 1      TMEM allocator; one lane issues tcgen05.mma (128 x 256 x 16)
//   warps 2..5  epilogue: TMEM -> registers -> SwiGLU (bf16) / row scale (fp32) -> HBM
// Shared memory holds a 4-stage ring of 48 KB stages; TMEM holds two 128x256
// fp32 accumulators so the epilogue of tile i overlaps the MMAs of tile i+1.
// Tiles come from a device-built schedule (heaviest group first) and are
// dealt to the persistent CTAs round robin.
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kABytes = kTileM * kTileK * 2;  // 16 KB
constexpr int kBRows = 256;                   // UMMA N
constexpr int kBBytes = kBRows * kTileK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr uint32_t kIdesc = ptx::idesc_bf16(kTileM, kBRows);
constexpr uint32_t kTmemCols = 512;  // two 256-column fp32 accumulators

struct __align__(8) SmemCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int32_t sched[2 * kMaxGroups + 2];
  int32_t offsets[kMaxExperts + 1];
};

constexpr size_t kSmemBytes = 1024 + size_t(kStages) * kStageBytes + sizeof(SmemCtl);

struct Tile {
  int g, m_blk, n_blk, rows, row0, K, N;
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
  const int mt = (x.rows + kTileM - 1) / kTileM;
  x.n_blk = local / mt;
  x.m_blk = local - x.n_blk * mt;
  (void)tile_n;
  return x;
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Bounded wait without the abort short-cut: used only while draining copies
// that are certain to complete, before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kWaitTimeoutNs) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

template <bool kSwiGLU>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_bf16_kernel(const __grid_constant__ CUtensorMap map_a0,
                             const __grid_constant__ CUtensorMap map_a1, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_tiles = smem;
  uint8_t* b_tiles = smem + kStages * kABytes;
  SmemCtl& c = *reinterpret_cast<SmemCtl*>(smem + kStages * kStageBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = args.E + args.has_shared;
  const int tile_n = kSwiGLU ? kGemm1TileN : kGemm2TileN;

  for (int i = threadIdx.x; i < sched_ints(G); i += kThreads) c.sched[i] = args.sched[i];
  for (int i = threadIdx.x; i <= args.E; i += kThreads) c.offsets[i] = args.offsets[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&c.full[s], 1);
      ptx::mbar_init(&c.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&c.tfull[s], 1);
      ptx::mbar_init(&c.tempty[s], 4);
    }
    ptx::mbar_init(&c.drain, 1);
    c.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&c.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    ptx::prefetch_tmap(&map_a0);
    ptx::prefetch_tmap(&map_a1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  const int num_tiles = c.sched[0];
  volatile int* abort = &c.abort;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      uint32_t it = 0;
      for (int t = blockIdx.x; t < num_tiles && !*abort; t += gridDim.x) {
        const Tile x = decode_tile(t, c, args, G, tile_n);
        const void* map_a = x.g < args.E ? static_cast<const void*>(&map_a0)
                                         : static_cast<const void*>(&map_a1);
        const CUtensorMap* mb = kSwiGLU ? args.b_maps + 2 * x.g : args.b_maps + x.g;
        const int a_row = x.row0 + x.m_blk * kTileM;
        const int kb_n = x.K / kTileK;
        bool ok = true;
        for (int kb = 0; kb < kb_n; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!ptx::mbar_wait(&c.empty[s], ph ^ 1, abort, args.err)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&c.full[s], kStageBytes);
          ptx::tma_load_2d(a_tiles + s * kABytes, map_a, &c.full[s], kb * kTileK, a_row);
          uint8_t* bs = b_tiles + s * kBBytes;
          if (kSwiGLU) {
            ptx::tma_load_2d(bs, mb, &c.full[s], kb * kTileK, x.n_blk * kGemm1TileN);
            ptx::tma_load_2d(bs + kBBytes / 2, mb + 1, &c.full[s], kb * kTileK,
                             x.n_blk * kGemm1TileN);
          } else {
            ptx::tma_load_2d(bs, mb, &c.full[s], kb * kTileK, x.n_blk * kGemm2TileN);
          }
        }
        if (!ok) break;
      }
      if (*abort) {
        // Let every load already issued land before the CTA leaves.
        const uint32_t first = it > kStages ? it - kStages : 0;
        for (uint32_t j = first; j < it; ++j)
          drain_wait(&c.full[j % kStages], (j / kStages) & 1, args.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      uint32_t it = 0;
      int local = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
        const Tile x = decode_tile(t, c, args, G, tile_n);
        const int acc = local & 1;
        const uint32_t acc_ph = (local >> 1) & 1;
        if (!ptx::mbar_wait(&c.tempty[acc], acc_ph ^ 1, abort, args.err)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBRows;
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
            ptx::mma_f16(d_tmem, da + 2 * k, db + 2 * k, kIdesc, (kb | k) != 0);
          ptx::mma_commit(&c.empty[s]);
        }
        if (!ok) break;
        ptx::mma_commit(&c.tfull[acc]);
      }
      // Every MMA issued by this thread has finished once `drain` flips.
      ptx::mma_commit(&c.drain);
      drain_wait(&c.drain, 0, args.err);
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    int local = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
      const Tile x = decode_tile(t, c, args, G, tile_n);
      const int acc = local & 1;
      const uint32_t acc_ph = (local >> 1) & 1;
      if (!ptx::mbar_wait(&c.tfull[acc], acc_ph, abort, args.err)) break;
      ptx::tc_fence_after();
      const int m = x.m_blk * kTileM + r;
      const bool valid = m < x.rows;
      const bool routed = x.g < args.E;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBRows;
      if (kSwiGLU) {
        __nv_bfloat16* dst = nullptr;
        if (valid)
          dst = (routed ? static_cast<__nv_bfloat16*>(args.out0) + int64_t(x.row0 + m) * x.N
                        : static_cast<__nv_bfloat16*>(args.out1) + int64_t(m) * x.N) +
                x.n_blk * kGemm1TileN;
#pragma unroll 1
        for (int cb = 0; cb < kGemm1TileN / 32; ++cb) {
          uint32_t gr[32], ur[32];
          ptx::tmem_ld32(taddr + cb * 32, gr);
          ptx::tmem_ld32(taddr + kGemm1TileN + cb * 32, ur);
          ptx::tmem_ld_wait();
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + cb * 32);
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
              d4[v] = make_uint4(p[0], p[1], p[2], p[3]);
            }
          }
        }
      } else {
        float w = 1.0f;
        float* dst = nullptr;
        if (valid) {
          if (routed && args.row_weight) w = args.row_weight[x.row0 + m];
          dst = (routed ? static_cast<float*>(args.out0) + int64_t(x.row0 + m) * x.N
                        : static_cast<float*>(args.out1) + int64_t(m) * x.N) +
                x.n_blk * kGemm2TileN;
        }
#pragma unroll 1
        for (int cb = 0; cb < kGemm2TileN / 32; ++cb) {
          if (x.n_blk * kGemm2TileN + cb * 32 >= x.N) break;  // warp-uniform
          uint32_t yr[32];
          ptx::tmem_ld32(taddr + cb * 32, yr);
          ptx::tmem_ld_wait();
          if (valid) {
            float4* d4 = reinterpret_cast<float4*>(dst + cb * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              d4[v] = make_float4(w * __uint_as_float(yr[4 * v]), w * __uint_as_float(yr[4 * v + 1]),
                                  w * __uint_as_float(yr[4 * v + 2]), w * __uint_as_float(yr[4 * v + 3]));
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&c.tempty[acc]);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool kSwiGLU>
cudaError_t launch_impl(const CUtensorMap& a0, const CUtensorMap& a1, const GemmArgs& args, int grid,
                        cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(grouped_gemm_bf16_kernel<kSwiGLU>),
                                   static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  grouped_gemm_bf16_kernel<kSwiGLU><<<grid, kThreads, kSmemBytes, stream>>>(a0, a1, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm(bool swiglu, const CUtensorMap& map_a0, const CUtensorMap& map_a1,
                                const GemmArgs& args, int grid, cudaStream_t stream) {
  return swiglu ? launch_impl<true>(map_a0, map_a1, args, grid, stream)
                : launch_impl<false>(map_a0, map_a1, args, grid, stream);
}

}  // namespace moe
