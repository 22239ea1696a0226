// Token-to-expert histogram and permutation (the per-expert token counts of
// the dispatch metadata, "ASAP: A DiSaggregated and Asynchronous Inference
// System for MoE Prefill", table 2), plus the tile planner of the grouped GEMMs.
//
// Deterministic and atomic-free across blocks:
//   hist     block b (64 tokens) counts its (token, slot) entries per expert
//            into shared memory -> blk_counts[e][b]
//   scan     one warp per expert scans blk_counts[e][*] (exclusive) ->
//            blk_base[e][b] and counts[e]; a block scan of counts -> offsets
//   scatter  block b sets bit t of word mask[e] for each token t of the
//            block that chose e; the rank of (t, e) inside the block is the
//            popcount of the bits below t, so
//              row(t, j) = offsets[e] + blk_base[e][b] + rank
//            orders every expert's rows by ascending token index.  The same
//            block then reads each of its tokens' hidden state once and
//            writes it to the token's k rows (16-byte vector accesses), so x
//            crosses HBM once on the way in.  For small batches a second grid
//            dimension splits the columns (in multiples of 128) over more
//            blocks; each recomputes the ranks, the first writes the maps.
#include <cuda_fp8.h>

#include <cstring>

#include "moe_internal.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kHistThreads = 256;
constexpr int kScanThreads = 1024;
constexpr int kScatterThreads = 256;
constexpr int kMaxK = 16;

__global__ void __launch_bounds__(kHistThreads)
    hist_kernel(const int32_t* __restrict__ ids, int64_t T, int k, int E, int nblk,
                int32_t* __restrict__ blk_counts, uint32_t* err) {
  __shared__ int cnt[kMaxExperts];
  __shared__ int32_t sid[kPermTok * kMaxK];
  for (int e = threadIdx.x; e < E; e += kHistThreads) cnt[e] = 0;
  const int64_t t0 = int64_t(blockIdx.x) * kPermTok;
  const int n = static_cast<int>(T - t0 < kPermTok ? T - t0 : kPermTok) * k;
  const int32_t* src = ids + t0 * k;
  for (int i = threadIdx.x; i < n; i += kHistThreads) sid[i] = src[i];
  __syncthreads();
  bool dup = false;
  for (int i = threadIdx.x; i < n; i += kHistThreads) {
    const int e = sid[i];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&cnt[e], 1);
    else atomicOr(err, kErrBounds);
    // a token must list k distinct experts: compare with its earlier slots
    for (int j = i - i % k; j < i; ++j) dup |= sid[j] == e;
  }
  if (dup) atomicOr(err, kErrDupIds);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kHistThreads) blk_counts[int64_t(e) * nblk + blockIdx.x] = cnt[e];
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += u;
  }
  return v;
}

__global__ void __launch_bounds__(kScanThreads)
    scan_kernel(const int32_t* __restrict__ blk_counts, int nblk, int E,
                int32_t* __restrict__ blk_base, int32_t* __restrict__ counts,
                int32_t* __restrict__ offsets, int32_t* __restrict__ pad_offsets) {
  __shared__ int tot[kMaxExperts];
  __shared__ int wsum[32];
  __shared__ int psum[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Each warp scans its experts' columns in batches of 256 blocks: the batch's
  // 8 loads per lane are issued together, and the next expert's first batch is
  // loaded while the current one is scanned, so the warp waits on one memory
  // latency per batch instead of one per 32 blocks.
  constexpr int kB = 8;  // 32-block chunks per batch
  auto load = [&](int e, int b0, int (&v)[kB]) {
    const int32_t* src = blk_counts + int64_t(e) * nblk;
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int b = b0 + j * 32 + lane;
      v[j] = b < nblk ? src[b] : 0;
    }
  };
  int nxt[kB];
  if (warp < E) load(warp, 0, nxt);
  for (int e = warp; e < E; e += kScanThreads / 32) {
    int32_t* dst = blk_base + int64_t(e) * nblk;
    int carry = 0;
    for (int b0 = 0; b0 < nblk; b0 += 32 * kB) {
      int v[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) v[j] = nxt[j];
      // prefetch: this expert's next batch, else the next expert's first
      if (b0 + 32 * kB < nblk) load(e, b0 + 32 * kB, nxt);
      else if (e + kScanThreads / 32 < E) load(e + kScanThreads / 32, 0, nxt);
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        if (b0 + j * 32 >= nblk) break;  // warp-uniform: chunks past the last block
        const int b = b0 + j * 32 + lane;
        const int inc = warp_incl_scan(v[j], lane);
        if (b < nblk) dst[b] = carry + inc - v[j];
        carry += __shfl_sync(0xffffffffu, inc, 31);
      }
    }
    if (lane == 0) tot[e] = carry;
  }
  __syncthreads();
  // exclusive scan of the E totals (E <= 256 < blockDim)
  const int v = threadIdx.x < E ? tot[threadIdx.x] : 0;
  const int inc = warp_incl_scan(v, lane);
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int s = wsum[lane];
    const int si = warp_incl_scan(s, lane);
    wsum[lane] = si - s;
  }
  __syncthreads();
  if (threadIdx.x < E) {
    counts[threadIdx.x] = v;
    offsets[threadIdx.x] = wsum[warp] + inc - v;
    if (threadIdx.x == E - 1) offsets[E] = wsum[warp] + inc;
  }
  if (pad_offsets == nullptr) return;
  // the same scan over the counts rounded up to whole 128-row blocks
  const int pv = (v + kNvfp4Rows - 1) / kNvfp4Rows * kNvfp4Rows;
  const int pinc = warp_incl_scan(pv, lane);
  if (lane == 31) psum[warp] = pinc;
  __syncthreads();
  if (warp == 0) {
    const int s = psum[lane];
    const int si = warp_incl_scan(s, lane);
    psum[lane] = si - s;
  }
  __syncthreads();
  if (threadIdx.x < E) {
    pad_offsets[threadIdx.x] = psum[warp] + pinc - pv;
    if (threadIdx.x == E - 1) pad_offsets[E] = psum[warp] + pinc;
  }
}

__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kScatterThreads)
    scatter_kernel(const int32_t* __restrict__ ids, const float* __restrict__ topk_w,
                   const __nv_bfloat16* __restrict__ x, int64_t T, int k, int E, int H, int nblk,
                   int fp8, const int32_t* __restrict__ blk_base,
                   const int32_t* __restrict__ offsets, int32_t* __restrict__ perm_token,
                   int32_t* __restrict__ inv_row, float* __restrict__ row_weight,
                   void* __restrict__ x_perm, float* __restrict__ x_perm_scales, uint32_t* err) {
  __shared__ uint32_t mask[kMaxExperts][kPermTok / 32];
  __shared__ int32_t rows_s[kPermTok * kMaxK];
  for (int i = threadIdx.x; i < E * (kPermTok / 32); i += kScatterThreads)
    (&mask[0][0])[i] = 0u;
  __syncthreads();
  const int64_t t0 = int64_t(blockIdx.x) * kPermTok;
  const int nt = static_cast<int>(T - t0 < kPermTok ? T - t0 : kPermTok);
  const int n = nt * k;
  const int32_t* src = ids + t0 * k;
  for (int i = threadIdx.x; i < n; i += kScatterThreads) {
    const int tl = i / k;
    const int e = src[i];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicOr(&mask[e][tl >> 5], 1u << (tl & 31));
  }
  __syncthreads();
  const int64_t R = T * k;
  const bool write_maps = blockIdx.y == 0;
  for (int i = threadIdx.x; i < n; i += kScatterThreads) {
    const int tl = i / k;
    const int e = src[i];
    int32_t row = -1;
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
      const int wd = tl >> 5;
      int rank = __popc(mask[e][wd] & ((1u << (tl & 31)) - 1u));
      for (int w = 0; w < wd; ++w) rank += __popc(mask[e][w]);
      const int64_t r = int64_t(offsets[e]) + blk_base[int64_t(e) * nblk + blockIdx.x] + rank;
      if (r >= 0 && r < R) row = static_cast<int32_t>(r);
      else if (write_maps) atomicOr(err, kErrBounds);
    } else if (write_maps) {
      atomicOr(err, kErrBounds);
    }
    rows_s[i] = row;
    if (write_maps) {
      inv_row[t0 * k + i] = row;
      if (row >= 0) {
        perm_token[row] = static_cast<int32_t>(t0 + tl);
        if (row_weight) row_weight[row] = topk_w[t0 * k + i];
      }
    }
  }
  __syncthreads();
  if (!x_perm) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = kScatterThreads / 32;
  const int nch = H / 8;  // 8-element chunks per row (16 B of bf16 in, 16 or 8 B out)
  // this block's column slice, in whole 128-column groups: chunks [c_lo, c_hi)
  const int groups = H / 128;
  const int g_lo = static_cast<int>(int64_t(groups) * blockIdx.y / gridDim.y);
  const int g_hi = static_cast<int>(int64_t(groups) * (blockIdx.y + 1) / gridDim.y);
  const int c_lo = g_lo * 16, c_hi = g_hi * 16;
  if (!fp8) {
    uint4* dst = static_cast<uint4*>(x_perm);
    for (int tl = warp; tl < nt; tl += nwarps) {
      const uint4* s4 = reinterpret_cast<const uint4*>(x + (t0 + tl) * int64_t(H));
      const int32_t* rr = rows_s + tl * k;
      // 8 x 16 bytes per lane in flight: enough outstanding reads per SM to
      // cover HBM latency with the 8 KB-per-warp write burst behind them
      for (int c0 = c_lo; c0 < c_hi; c0 += 32 * 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int cc = c0 + u * 32 + lane;
          if (cc < c_hi) v[u] = __ldcs(s4 + cc);
        }
        for (int j = 0; j < k; ++j) {
          const int32_t row = rr[j];
          if (row < 0) continue;
          uint4* d4 = dst + int64_t(row) * nch;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int cc = c0 + u * 32 + lane;
            if (cc < c_hi) __stcs(d4 + cc, v[u]);  // streamed: x_perm (1.9 GB) outlives L2
          }
        }
      }
    }
  } else {
    // e4m3 codes, one fp32 scale per 128 features (16 chunks = 16 lanes).
    uint2* dst = static_cast<uint2*>(x_perm);
    const int ng = H / 128;
    for (int tl = warp; tl < nt; tl += nwarps) {
      const uint4* s4 = reinterpret_cast<const uint4*>(x + (t0 + tl) * int64_t(H));
      const int32_t* rr = rows_s + tl * k;
      for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
        const int cc = c0 + lane;  // slices are multiples of 16 chunks: half warps stay whole
        const bool on = cc < c_hi;
        const uint4 v = on ? __ldcs(s4 + cc) : make_uint4(0, 0, 0, 0);
        float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                      bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
        for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
        uint2 q;
        q.x = cvt_e4m3x4(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s), __fdiv_rn(f[2], s), __fdiv_rn(f[3], s));
        q.y = cvt_e4m3x4(__fdiv_rn(f[4], s), __fdiv_rn(f[5], s), __fdiv_rn(f[6], s), __fdiv_rn(f[7], s));
        if (!on) continue;
        for (int j = 0; j < k; ++j) {
          const int32_t row = rr[j];
          if (row < 0) continue;
          dst[int64_t(row) * nch + cc] = q;
          if ((cc & 15) == 0) x_perm_scales[int64_t(row) * ng + (cc >> 4)] = s;
        }
      }
    }
  }
}

// NVFP4 scatter: the ranks and maps as scatter_kernel; each lane quantises one
// 16-element block of a token (nvfp4.cuh) and writes its 8 code bytes to the
// token's k rows at their positions in the 128-row-padded layout
// (pad_offsets[e] + the row's index inside expert e), the scales of 4 adjacent
// blocks as one 32-bit word of the MMA scale layout.  Afterwards every block
// zeroes part of the padding rows' scales, so that padding contributes 0.
__global__ void __launch_bounds__(kScatterThreads)
    scatter_nvfp4_kernel(const int32_t* __restrict__ ids, const float* __restrict__ topk_w,
                         const __nv_bfloat16* __restrict__ x, int64_t T, int k, int E, int H,
                         int nblk, const int32_t* __restrict__ blk_base,
                         const int32_t* __restrict__ offsets, int32_t* __restrict__ perm_token,
                         int32_t* __restrict__ inv_row, float* __restrict__ row_weight,
                         const Nvfp4Scatter qa, uint32_t* err) {
  __shared__ uint32_t mask[kMaxExperts][kPermTok / 32];
  __shared__ int64_t pos_s[kPermTok * kMaxK];
  for (int i = threadIdx.x; i < E * (kPermTok / 32); i += kScatterThreads)
    (&mask[0][0])[i] = 0u;
  __syncthreads();
  const int64_t t0 = int64_t(blockIdx.x) * kPermTok;
  const int nt = static_cast<int>(T - t0 < kPermTok ? T - t0 : kPermTok);
  const int n = nt * k;
  const int32_t* src = ids + t0 * k;
  for (int i = threadIdx.x; i < n; i += kScatterThreads) {
    const int tl = i / k;
    const int e = src[i];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      atomicOr(&mask[e][tl >> 5], 1u << (tl & 31));
  }
  __syncthreads();
  const int64_t R = T * k;
  const bool write_maps = blockIdx.y == 0;
  for (int i = threadIdx.x; i < n; i += kScatterThreads) {
    const int tl = i / k;
    const int e = src[i];
    int32_t row = -1;
    int64_t pos = -1;
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
      const int wd = tl >> 5;
      int rank = __popc(mask[e][wd] & ((1u << (tl & 31)) - 1u));
      for (int w = 0; w < wd; ++w) rank += __popc(mask[e][w]);
      const int64_t local = int64_t(blk_base[int64_t(e) * nblk + blockIdx.x]) + rank;
      const int64_t r = int64_t(offsets[e]) + local;
      const int64_t p = int64_t(qa.pad_offsets[e]) + local;
      if (r >= 0 && r < R && p >= 0 && p < qa.rows_pad) {
        row = static_cast<int32_t>(r);
        pos = p;
      } else if (write_maps) {
        atomicOr(err, kErrBounds);
      }
    } else if (write_maps) {
      atomicOr(err, kErrBounds);
    }
    pos_s[i] = pos;
    if (write_maps) {
      inv_row[t0 * k + i] = row;
      if (row >= 0) {
        perm_token[row] = static_cast<int32_t>(t0 + tl);
        if (row_weight) row_weight[row] = topk_w[t0 * k + i];
      }
    }
  }
  __syncthreads();

  const int layer = resolve_layer(qa.layer, qa.num_layers, err);
  const float g = __ldg(qa.act_scales + 2 * layer);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = kScatterThreads / 32;
  // this block's column slice, in whole 128-column groups (8 blocks each)
  const int groups = H / 128;
  const int b_lo = static_cast<int>(int64_t(groups) * blockIdx.y / gridDim.y) * 8;
  const int b_hi = static_cast<int>(int64_t(groups) * (blockIdx.y + 1) / gridDim.y) * 8;
  for (int tl = warp; tl < nt; tl += nwarps) {
    const __nv_bfloat16* xr = x + (t0 + tl) * int64_t(H);
    const int64_t* pp = pos_s + tl * k;
    for (int b0 = b_lo; b0 < b_hi; b0 += 32) {
      const int b = b0 + lane;
      const bool on = b < b_hi;  // groups of 4 lanes are all on or all off
      float f[16];
      if (on) {
        const uint4 u0 = __ldcs(reinterpret_cast<const uint4*>(xr + b * 16));
        const uint4 u1 = __ldcs(reinterpret_cast<const uint4*>(xr + b * 16 + 8));
        const uint32_t w8[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          f[2 * j] = __uint_as_float(w8[j] << 16);
          f[2 * j + 1] = __uint_as_float(w8[j] & 0xffff0000u);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) f[j] = 0.0f;
      }
      uint2 q;
      const uint32_t sc = nvfp4::quantize16(f, g, q);
      uint32_t w4 = sc << (8 * (lane & 3));
      w4 |= __shfl_xor_sync(0xffffffffu, w4, 1);
      w4 |= __shfl_xor_sync(0xffffffffu, w4, 2);
      if (!on) continue;
      for (int j = 0; j < k; ++j) {
        const int64_t p = pp[j];
        if (p < 0) continue;
        *reinterpret_cast<uint2*>(qa.x_codes + p * (H / 2) + b * 8) = q;
        if ((lane & 3) == 0)
          *reinterpret_cast<uint32_t*>(qa.x_sf + nvfp4::sf_offset(p, b, H)) = w4;
      }
      if (qa.xs_codes) {
        const int64_t t = t0 + tl;
        *reinterpret_cast<uint2*>(qa.xs_codes + t * (H / 2) + b * 8) = q;
        if ((lane & 3) == 0)
          *reinterpret_cast<uint32_t*>(qa.xs_sf + nvfp4::sf_offset(t, b, H)) = w4;
      }
    }
  }

  // padding rows: zero scale words (4 blocks each), spread over the whole grid
  const int wpr = H / 64;
  const int64_t gthreads = int64_t(gridDim.x) * gridDim.y * blockDim.x;
  const int64_t gtid =
      (int64_t(blockIdx.y) * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t routed_words = int64_t(E) * (kNvfp4Rows - 1) * wpr;
  const int64_t t_pad = (T + kNvfp4Rows - 1) / kNvfp4Rows * kNvfp4Rows;
  const int64_t shared_words = qa.xs_sf ? (t_pad - T) * wpr : 0;
  for (int64_t i = gtid; i < routed_words + shared_words; i += gthreads) {
    if (i < routed_words) {
      const int e = static_cast<int>(i / ((kNvfp4Rows - 1) * wpr));
      const int64_t rem = i - int64_t(e) * (kNvfp4Rows - 1) * wpr;
      const int rr = static_cast<int>(rem / wpr), w = static_cast<int>(rem - int64_t(rr) * wpr);
      const int cnt = offsets[e + 1] - offsets[e];
      const int pad = qa.pad_offsets[e + 1] - qa.pad_offsets[e] - cnt;
      if (rr >= pad) continue;
      const int64_t p = int64_t(qa.pad_offsets[e]) + cnt + rr;
      if (p < qa.rows_pad) *reinterpret_cast<uint32_t*>(qa.x_sf + nvfp4::sf_offset(p, 4 * w, H)) = 0u;
    } else {
      const int64_t j = i - routed_words;
      const int64_t t = T + j / wpr;
      const int w = static_cast<int>(j % wpr);
      *reinterpret_cast<uint32_t*>(qa.xs_sf + nvfp4::sf_offset(t, 4 * w, H)) = 0u;
    }
  }
}

// Tile schedules of GEMM1 and GEMM2 from the row offsets: per group
// ceil(rows/tile_rows) x n_tiles tiles; groups ordered by descending tile count
// (ties: lower group first) so the heaviest experts start first.
// With `cut` (bf16 layers), also each expert's copies of the two GEMMs' A
// tensor maps with the row extent cut at the end of its rows, offsets[e + 1]:
// cut[e] from a1 (GEMM1), cut[E + e] from a2 (GEMM2).
__global__ void __launch_bounds__(256)
    plan_kernel(const int32_t* __restrict__ offsets, int E, int has_shared, int64_t T,
                int n1r, int n1s, int n2r, int n2s, int32_t* __restrict__ sched1,
                int32_t* __restrict__ sched2, int tile_rows1, int tile_rows2,
                const __grid_constant__ CUtensorMap a1, const __grid_constant__ CUtensorMap a2,
                uint8_t* __restrict__ cut, int64_t cut_rows) {
  __shared__ int tiles[2][kMaxGroups];
  __shared__ int order[2][kMaxGroups];
  if (cut != nullptr) {
    for (int i = threadIdx.x; i < 2 * E; i += blockDim.x) {
      const int e = i < E ? i : i - E;
      const uint4* src = reinterpret_cast<const uint4*>(i < E ? &a1 : &a2);
      uint4* dst = reinterpret_cast<uint4*>(cut + size_t(i) * 128);
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j] = src[j];
      // within [1, cut_rows], the templates' own extent: the cut never reaches
      // past the buffer, whatever the offsets hold (an expert with no rows has
      // no tiles; its map still gets a nonzero extent)
      const int64_t end = offsets[e + 1];
      const int64_t ext = end < 1 ? 1 : (end > cut_rows ? cut_rows : end);
      ptx::tensormap_set_extent<1>(dst, static_cast<uint32_t>(ext));
    }
    ptx::fence_tensormap_release();
  }
  const int G = E + has_shared;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    const int64_t rows = g < E ? int64_t(offsets[g + 1]) - offsets[g] : T;
    const int mt1 = static_cast<int>((rows + tile_rows1 - 1) / tile_rows1);
    const int mt2 = static_cast<int>((rows + tile_rows2 - 1) / tile_rows2);
    tiles[0][g] = mt1 * (g < E ? n1r : n1s);
    tiles[1][g] = mt2 * (g < E ? n2r : n2s);
  }
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    for (int w = 0; w < 2; ++w) {
      const int tg = tiles[w][g];
      int rank = 0;
      for (int h = 0; h < G; ++h) {
        const int th = tiles[w][h];
        rank += (th > tg) || (th == tg && h < g);
      }
      order[w][rank] = g;
    }
  }
  __syncthreads();
  if (threadIdx.x < 64) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* s = w ? sched2 : sched1;
    int carry = 0;
    for (int b0 = 0; b0 < G; b0 += 32) {
      const int b = b0 + lane;
      const int v = b < G ? tiles[w][order[w][b]] : 0;
      const int inc = warp_incl_scan(v, lane);
      if (b < G) {
        s[1 + b] = carry + inc - v;
        s[G + 2 + b] = order[w][b];
      }
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
      s[0] = carry;
      s[1 + G] = carry;
    }
  }
}

}  // namespace

cudaError_t launch_hist(const int32_t* ids, int64_t T, int k, int E, int32_t* blk_counts,
                        uint32_t* err, cudaStream_t stream) {
  const int nblk = static_cast<int>((T + kPermTok - 1) / kPermTok);
  hist_kernel<<<nblk, kHistThreads, 0, stream>>>(ids, T, k, E, nblk, blk_counts, err);
  return cudaGetLastError();
}

cudaError_t launch_scan(const int32_t* blk_counts, int nblk, int E, int32_t* blk_base,
                        int32_t* counts, int32_t* offsets, cudaStream_t stream,
                        int32_t* pad_offsets) {
  scan_kernel<<<1, kScanThreads, 0, stream>>>(blk_counts, nblk, E, blk_base, counts, offsets,
                                              pad_offsets);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const int32_t* ids, const float* topk_w, const void* x, int64_t T,
                           int k, int E, int H, int fp8, const int32_t* blk_base,
                           const int32_t* offsets, int32_t* perm_token, int32_t* inv_row,
                           float* row_weight, void* x_perm, float* x_perm_scales, uint32_t* err,
                           cudaStream_t stream) {
  const int nblk = static_cast<int>((T + kPermTok - 1) / kPermTok);
  // about 8 blocks per SM (two waves of 4 resident blocks), in whole
  // 128-column slices: the copies are latency-bound with fewer warps per SM
  int sm = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev);
  int ysplit = (8 * sm + nblk - 1) / nblk;
  if (ysplit > H / 128) ysplit = H / 128;
  if (ysplit < 1 || !x_perm) ysplit = 1;
  scatter_kernel<<<dim3(nblk, ysplit), kScatterThreads, 0, stream>>>(
      ids, topk_w, static_cast<const __nv_bfloat16*>(x), T, k, E, H, nblk, fp8, blk_base, offsets,
      perm_token, inv_row, row_weight, x_perm, x_perm_scales, err);
  return cudaGetLastError();
}

cudaError_t launch_scatter_nvfp4(const int32_t* ids, const float* topk_w, const void* x,
                                 int64_t T, int k, int E, int H, const int32_t* blk_base,
                                 const int32_t* offsets, int32_t* perm_token, int32_t* inv_row,
                                 float* row_weight, const Nvfp4Scatter& q, uint32_t* err,
                                 cudaStream_t stream) {
  const int nblk = static_cast<int>((T + kPermTok - 1) / kPermTok);
  // Column slices: about 12 blocks per SM (3 waves of 4 resident blocks; the
  // quantisation is latency-bound at fewer warps), each slice a whole number
  // of 512 columns (one 16-element block per lane and step) unless that leaves
  // less than one wave.  DeepSeek-V3 shapes: T = 16384 0.393 ms with 2 blocks
  // per SM -> 0.277 ms; T = 4096 0.131 -> 0.064 ms with 512-column slices;
  // T = 512 0.052 ms with the finest slices (128 columns).
  int sm = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev);
  if (nblk <= 0) return cudaSuccess;
  const int groups = H / 128;
  const int wide = groups / 4 > 0 ? groups / 4 : 1;  // slices of 512 columns
  int ysplit = (12 * sm + nblk - 1) / nblk;
  if (ysplit <= wide) {
    const int per = (wide + ysplit / 2) / ysplit;  // 512-column units per slice
    ysplit = wide / (per > 0 ? per : 1);
  } else if (int64_t(nblk) * wide >= 4 * int64_t(sm)) {
    ysplit = wide;
  }
  if (ysplit > groups) ysplit = groups;
  if (ysplit < 1) ysplit = 1;
  scatter_nvfp4_kernel<<<dim3(nblk, ysplit), kScatterThreads, 0, stream>>>(
      ids, topk_w, static_cast<const __nv_bfloat16*>(x), T, k, E, H, nblk, blk_base, offsets,
      perm_token, inv_row, row_weight, q, err);
  return cudaGetLastError();
}

cudaError_t launch_plan(const int32_t* offsets, int E, int has_shared, int64_t T, int n1_routed,
                        int n1_shared, int n2_routed, int n2_shared, int32_t* sched1,
                        int32_t* sched2, int tile_rows1, int tile_rows2, cudaStream_t stream,
                        const CUtensorMap* cut_a1, const CUtensorMap* cut_a2, uint8_t* cut,
                        int64_t cut_rows) {
  CUtensorMap none;
  memset(&none, 0, sizeof none);
  const bool with_cut = cut != nullptr && cut_a1 != nullptr && cut_a2 != nullptr && cut_rows > 0;
  plan_kernel<<<1, 256, 0, stream>>>(offsets, E, has_shared, T, n1_routed, n1_shared, n2_routed,
                                     n2_shared, sched1, sched2, tile_rows1, tile_rows2,
                                     with_cut ? *cut_a1 : none, with_cut ? *cut_a2 : none,
                                     with_cut ? cut : nullptr, cut_rows);
  return cudaGetLastError();
}

}  // namespace moe
