// Router: logits = x W_r^T on the tensor cores, with top-k selection and the
// gate weights fused into the epilogue ("gated routing" of "Memory-Compute
// Disaggregation for Large-Model Inference: AFD Architecture Analysis and
// Performance Validation", section 3, Data-Flow Closed Loop step 3; k of E
// experts per token as in "ASAP: A DiSaggregated and Asynchronous Inference
// System for MoE Prefill", section 5.1).
//
// A cluster of S CTAs (S = 1, 2, 4 or 8) owns 128 tokens; CTA c of the
// cluster accumulates the K slice [c H / S, (c + 1) H / S) of the 128 x E_pad
// logit tile in TMEM (the E <= 256 router rows, padded to a multiple of 16,
// form the N side).  S grows while the grid still fits the GPU, so a small
// batch spreads its K loop over many SMs instead of running one CTA per 128
// tokens through all of H.
//
//   S = 1: each epilogue thread holds one token's complete logit row.
//   S > 1: each CTA parks its partial tile in shared memory; after a cluster
//          barrier CTA c finishes tokens [c 128 / S, (c + 1) 128 / S), S
//          threads per token, each summing the S partials of E_pad / S
//          logits over distributed shared memory (in CTA order).  Thread p
//          of a token owns experts 4 S m + 4 p + {0..3}, so the S threads read
//          one contiguous 16 S-byte segment of a peer's row per load.
// A thread scans its logits once, keeping the k largest (strictly greater
// replaces, so among equal logits the lower expert index stays ahead) and a
// running softmax normaliser; the S threads of a token then merge their lists
// and normalisers by shuffles, ordering equal logits by expert index, which
// selects exactly what one scan of the whole row would.
#include <math.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 192;
// Each token tile walks its K slice starting at a tile-dependent k-step (and
// wraps around), so that the CTAs running at once do not all read the same
// router-weight k-block (and the same column offset of their token rows) at
// the same moment.
constexpr bool kRotateK = true;
constexpr int kABytes = kTileM * kTileK * 2;
constexpr int kMaxBBytes = 256 * kTileK * 2;

struct __align__(8) RouterCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float bias[kMaxExperts];
};

constexpr size_t kSmemBytes = 1024 + size_t(kStages) * (kABytes + kMaxBBytes) + sizeof(RouterCtl);
constexpr int kMaxSplit = 8;  // CTAs per cluster (portable cluster size)
// Partial logit tile of one CTA, [128 tokens][E_pad + 4] fp32, in the stage
// area once the main loop is over (the +4 skews rows across banks).
static_assert(kTileM * (256 + 4) * 4 <= kStages * (kABytes + kMaxBBytes), "partial tile fits");

struct RouterArgs {
  int64_t T;
  int H, E, E_pad, k, score, renormalize;
  float route_scale;
  const float* bias;
  int32_t* topk_ids;
  float* topk_w;
  float* logits_out;
  uint32_t* err;
  uint32_t tmem_cols;
  RouterTable table;  // layer stacks: per-layer router descriptors and biases
};

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kWaitTimeoutNs) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

// Insert (v, e) into a descending list of KMAX entries; strict comparison keeps
// an earlier (lower-index) equal value ahead of a later one.  Used while
// scanning experts in increasing index order.
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&tv)[KMAX], int (&ti)[KMAX], float v, int e) {
  if (!(v > tv[KMAX - 1])) return;
#pragma unroll
  for (int i = KMAX - 1; i > 0; --i) {
    const bool shift = v > tv[i - 1];
    const bool here = !shift && v > tv[i];
    tv[i] = shift ? tv[i - 1] : (here ? v : tv[i]);
    ti[i] = shift ? ti[i - 1] : (here ? e : ti[i]);
  }
  if (v > tv[0]) {
    tv[0] = v;
    ti[0] = e;
  }
}

// (v, e) ahead of (w, f) in the selection order: valid before empty (index
// -1), larger logit first, lower expert index among equal logits.
__device__ __forceinline__ bool ahead(float v, int e, float w, int f) {
  return e >= 0 && (f < 0 || v > w || (v == w && e < f));
}

// Top KMAX of two lists sorted by `ahead` (disjoint expert ranges): the
// better of tv[i] and ov[KMAX-1-i] for each i gives the KMAX best as a bitonic
// sequence, which log2(KMAX) rounds of compare-exchanges sort.
template <int KMAX>
__device__ __forceinline__ void topk_merge(float (&tv)[KMAX], int (&ti)[KMAX],
                                           const float (&ov)[KMAX], const int (&oi)[KMAX]) {
#pragma unroll
  for (int i = 0; i < KMAX; ++i) {
    const bool take = ahead(ov[KMAX - 1 - i], oi[KMAX - 1 - i], tv[i], ti[i]);
    tv[i] = take ? ov[KMAX - 1 - i] : tv[i];
    ti[i] = take ? oi[KMAX - 1 - i] : ti[i];
  }
#pragma unroll
  for (int d = KMAX / 2; d >= 1; d >>= 1) {
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      if ((i & d) == 0) {
        const bool swap = ahead(tv[i + d], ti[i + d], tv[i], ti[i]);
        const float v = tv[i];
        const int e = ti[i];
        tv[i] = swap ? tv[i + d] : v;
        ti[i] = swap ? ti[i + d] : e;
        tv[i + d] = swap ? v : tv[i + d];
        ti[i + d] = swap ? e : ti[i + d];
      }
    }
  }
}

// Online softmax normaliser: add the logit v to (run_max, run_sum).
__device__ __forceinline__ void softmax_add(float& run_max, float& run_sum, float v) {
  if (v > run_max) {
    run_sum = run_sum * expf(run_max - v) + 1.0f;
    run_max = v;
  } else {
    run_sum += expf(v - run_max);
  }
}

// Gate weights of one token from its top-k list and softmax normaliser;
// writes ids and weights (k entries).
template <int KMAX>
__device__ __forceinline__ void finish_token(const RouterArgs& a, int64_t t, const float (&tv)[KMAX],
                                             const int (&ti)[KMAX], float run_max, float run_sum) {
  const int k = a.k;
  float w[KMAX];
  float denom = 0.0f;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (j < k) {
      bad |= ti[j] < 0;
      if (a.score == 0) {
        w[j] = a.renormalize ? expf(tv[j] - tv[0]) : expf(tv[j] - run_max) / run_sum;
      } else {
        w[j] = 1.0f / (1.0f + expf(-tv[j]));
      }
      denom += w[j];
    } else {
      w[j] = 0.0f;
    }
  }
  if (bad) atomicOr(a.err, kErrNoSelect);
  const float norm = a.renormalize ? a.route_scale / denom : a.route_scale;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (j < k) {
      a.topk_ids[t * k + j] = ti[j];
      a.topk_w[t * k + j] = w[j] * norm;
    }
  }
}

template <int KMAX>
__global__ void __launch_bounds__(kThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap map_x,
                  const __grid_constant__ CUtensorMap map_w, const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int b_bytes = a.E_pad * kTileK * 2;
  const int stage_bytes = kABytes + b_bytes;
  uint8_t* a_tiles = smem;
  uint8_t* b_tiles = smem + kStages * kABytes;
  RouterCtl& c = *reinterpret_cast<RouterCtl*>(smem + kStages * (kABytes + kMaxBBytes));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = static_cast<int>(ptx::cluster_nctarank());   // K split of this token tile
  const uint32_t crank = ptx::cluster_ctarank();
  const int64_t m0 = int64_t(blockIdx.x / S) * kTileM;
  // this call's router matrix and bias (a layer stack indexes its tables)
  const float* bias = a.bias;
  const void* map_w_ptr = &map_w;
  if (a.table.w_table) {
    const int l = resolve_layer(a.table.layer, a.table.num_layers, a.err);
    map_w_ptr = a.table.w_table + l;
    bias = a.table.bias_table[l];
  }

  for (int i = threadIdx.x; i < a.E; i += kThreads) c.bias[i] = bias ? bias[i] : 0.0f;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&c.full[s], 1);
      ptx::mbar_init(&c.empty[s], 1);
    }
    ptx::mbar_init(&c.tfull, 1);
    ptx::mbar_init(&c.drain, 1);
    c.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&c.tmem_base, a.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  volatile int* abort = &c.abort;
  // the softmax normaliser over all E is needed only for unrenormalised softmax
  const bool need_norm = a.score == 0 && !a.renormalize;
  const int kb_all = a.H / kTileK;
  const int kb0 = static_cast<int>(crank) * kb_all / S;  // this CTA's K slice (S <= kb_all)
  const int kb1 = (static_cast<int>(crank) + 1) * kb_all / S;
  const int kb_n = kb1 - kb0;
  const int rot = kRotateK ? static_cast<int>((blockIdx.x / S) % static_cast<unsigned>(kb_n)) : 0;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      for (int i = 0; i < kb_n; ++i, ++it) {
        const int kb = kb0 + (i + rot) % kb_n;
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!ptx::mbar_wait(&c.empty[s], ph ^ 1, abort, a.err)) break;
        ptx::mbar_arrive_expect_tx(&c.full[s], stage_bytes);
        ptx::tma_load_2d(a_tiles + s * kABytes, &map_x, &c.full[s], kb * kTileK, int32_t(m0));
        ptx::tma_load_2d(b_tiles + s * kMaxBBytes, map_w_ptr, &c.full[s], kb * kTileK, 0);
      }
      if (*abort) {
        const uint32_t first = it > kStages ? it - kStages : 0;
        for (uint32_t j = first; j < it; ++j)
          drain_wait(&c.full[j % kStages], (j / kStages) & 1, a.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16(kTileM, a.E_pad);
      bool ok = true;
      for (int i = 0; i < kb_n; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!ptx::mbar_wait(&c.full[s], ph, abort, a.err)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint64_t da = ptx::sw128_desc(ptx::smem_u32(a_tiles + s * kABytes));
        const uint64_t db = ptx::sw128_desc(ptx::smem_u32(b_tiles + s * kMaxBBytes));
#pragma unroll
        for (int k = 0; k < kTileK / 16; ++k)
          ptx::mma_f16(tmem_base, da + 2 * k, db + 2 * k, idesc, (i != 0) || (k != 0));
        ptx::mma_commit(&c.empty[s]);
      }
      if (ok) ptx::mma_commit(&c.tfull);
      ptx::mma_commit(&c.drain);
      drain_wait(&c.drain, 0, a.err);
    }
  } else if (S > 1) {
    // partial tile -> this CTA's shared memory, row = token
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int stride = a.E_pad + 4;
    float* part = reinterpret_cast<float*>(smem) + r * stride;
    if (ptx::mbar_wait(&c.tfull, 0, abort, a.err)) {
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < a.E_pad; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld32(taddr + c0, v);
        ptx::tmem_ld_wait();
        // E_pad is a multiple of 16: the last chunk may hold only 16 columns
        const int n4 = (a.E_pad - c0 < 32 ? a.E_pad - c0 : 32) / 4;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < n4)
            reinterpret_cast<float4*>(part + c0)[j] =
                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                            __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
      }
    }
  } else {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int64_t t = m0 + r;
    const bool valid = t < a.T;
    if (ptx::mbar_wait(&c.tfull, 0, abort, a.err)) {
      ptx::tc_fence_after();
      float tv[KMAX];
      int ti[KMAX];
#pragma unroll
      for (int i = 0; i < KMAX; ++i) {
        tv[i] = -INFINITY;
        ti[i] = -1;
      }
      float run_max = -INFINITY, run_sum = 0.0f;  // softmax over all E (online)
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      float* lrow = (valid && a.logits_out) ? a.logits_out + t * a.E : nullptr;
#pragma unroll 1
      for (int c0 = 0; c0 < a.E_pad; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld32(taddr + c0, v);
        ptx::tmem_ld_wait();
        float lv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int e = c0 + j;
          lv[j] = e < a.E ? __uint_as_float(v[j]) + c.bias[e] : -INFINITY;
        }
        if (lrow) {
          if (c0 + 32 <= a.E) {
            float4* d = reinterpret_cast<float4*>(lrow + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              d[j] = make_float4(lv[4 * j], lv[4 * j + 1], lv[4 * j + 2], lv[4 * j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c0 + j < a.E) lrow[c0 + j] = lv[j];
          }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (c0 + j < a.E) {
            topk_insert<KMAX>(tv, ti, lv[j], c0 + j);
            if (need_norm) softmax_add(run_max, run_sum, lv[j]);
          }
        }
      }
      if (valid) finish_token<KMAX>(a, t, tv, ti, run_max, run_sum);
    }
  }

  if (S > 1) {
    ptx::cluster_sync();  // every CTA's partial tile is in its shared memory
    if (warp >= 2) {
      // tokens [crank 128 / S, +128 / S) of the tile, S threads per token
      const int et = threadIdx.x - 64;
      const int p = et % S;
      const int tl = static_cast<int>(crank) * (kTileM / S) + et / S;
      const int64_t t = m0 + tl;
      const bool valid = t < a.T;
      const int nchunk = a.E_pad / (4 * S);  // E_pad is a multiple of 4 S
      const uint32_t src = ptx::smem_u32(reinterpret_cast<float*>(smem) + tl * (a.E_pad + 4) + 4 * p);
      uint32_t peer[kMaxSplit];
#pragma unroll
      for (int j = 0; j < kMaxSplit; ++j) peer[j] = j < S ? ptx::mapa(src, j) : 0u;
      float tv[KMAX];
      int ti[KMAX];
#pragma unroll
      for (int i = 0; i < KMAX; ++i) {
        tv[i] = -INFINITY;
        ti[i] = -1;
      }
      float run_max = -INFINITY, run_sum = 0.0f;
      float* lrow = (valid && a.logits_out) ? a.logits_out + t * a.E : nullptr;
      // the S partials of four logits per chunk; chunk m + 1 is loaded before
      // chunk m is scanned, so the remote-load latency overlaps the scan
      float4 nxt[kMaxSplit];
#pragma unroll
      for (int j = 0; j < kMaxSplit; ++j)
        nxt[j] = j < S ? ptx::ld_cluster_f32x4(peer[j]) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
      for (int m = 0; m < nchunk; ++m) {
        float4 pv[kMaxSplit];
#pragma unroll
        for (int j = 0; j < kMaxSplit; ++j) pv[j] = nxt[j];
        if (m + 1 < nchunk) {
          const uint32_t off = 16u * S * (m + 1);
#pragma unroll
          for (int j = 0; j < kMaxSplit; ++j)
            if (j < S) nxt[j] = ptx::ld_cluster_f32x4(peer[j] + off);
        }
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < kMaxSplit; ++j)
          if (j < S) {
            v[0] += pv[j].x;
            v[1] += pv[j].y;
            v[2] += pv[j].z;
            v[3] += pv[j].w;
          }
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int e = 4 * S * m + 4 * p + h;  // increasing in (m, h)
          if (e < a.E) {
            const float lv = v[h] + c.bias[e];
            if (lrow) lrow[e] = lv;
            topk_insert<KMAX>(tv, ti, lv, e);
            if (need_norm) softmax_add(run_max, run_sum, lv);
          }
        }
      }
      // merge the S lists of the token (adjacent lanes)
#pragma unroll
      for (int d = 1; d < kMaxSplit; d <<= 1) {
        if (d < S) {
          float ov[KMAX];
          int oi[KMAX];
#pragma unroll
          for (int i = 0; i < KMAX; ++i) {
            ov[i] = __shfl_xor_sync(0xffffffffu, tv[i], d);
            oi[i] = __shfl_xor_sync(0xffffffffu, ti[i], d);
          }
          topk_merge<KMAX>(tv, ti, ov, oi);
          const float om = __shfl_xor_sync(0xffffffffu, run_max, d);
          const float os = __shfl_xor_sync(0xffffffffu, run_sum, d);
          if (om > run_max) {
            run_sum = run_sum * expf(run_max - om) + os;
            run_max = om;
          } else if (om != -INFINITY) {
            run_sum += os * expf(om - run_max);
          }
        }
      }
      if (valid && p == 0) finish_token<KMAX>(a, t, tv, ti, run_max, run_sum);
    }
    ptx::cluster_sync();  // no CTA leaves while a peer still reads its partial tile
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

template <int KMAX>
cudaLaunchConfig_t cluster_config(int grid, int split, cudaStream_t stream,
                                  cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = static_cast<unsigned>(split);
  attr->val.clusterDim.y = 1;
  attr->val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Largest K split (power of two, <= kMaxSplit) whose clusters can be resident.
template <int KMAX>
int max_split() {
  static int cached = 0;
  if (cached) return cached;
  int split = kMaxSplit;
  for (; split > 1; split >>= 1) {
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = cluster_config<KMAX>(split, split, nullptr, &attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, router_kernel<KMAX>, &cfg) == cudaSuccess && n > 0) break;
    cudaGetLastError();
  }
  cached = split;
  return split;
}

template <int KMAX>
cudaError_t launch_k(const CUtensorMap& mx, const CUtensorMap& mw, const RouterArgs& a, int tiles,
                     int sm_count, cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(router_kernel<KMAX>),
                                   static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  // split K while the grid still fits the GPU, every CTA keeps a K step and
  // E_pad divides into 16-byte chunks per finishing thread
  const int kb_all = a.H / kTileK;
  const int cap = max_split<KMAX>();
  int split = 1;
  while (split < cap && tiles * split * 2 <= sm_count && split * 2 <= kb_all &&
         a.E_pad % (8 * split) == 0)
    split *= 2;
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg = cluster_config<KMAX>(tiles * split, split, stream, &attr);
  e = cudaLaunchKernelEx(&cfg, router_kernel<KMAX>, mx, mw, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const CUtensorMap& map_x, const CUtensorMap& map_w, int64_t T, int H,
                          int E, int E_pad, int k, int score, int renormalize, float route_scale,
                          const float* bias, int32_t* topk_ids, float* topk_w, float* logits_out,
                          uint32_t* err, int sm_count, cudaStream_t stream,
                          const RouterTable* table) {
  RouterArgs a;
  a.T = T;
  a.H = H;
  a.E = E;
  a.E_pad = E_pad;
  a.k = k;
  a.score = score;
  a.renormalize = renormalize;
  a.route_scale = route_scale;
  a.bias = bias;
  a.topk_ids = topk_ids;
  a.topk_w = topk_w;
  a.logits_out = logits_out;
  a.err = err;
  a.table = table ? *table : RouterTable{nullptr, nullptr, nullptr, 0};
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(E_pad)) cols <<= 1;
  a.tmem_cols = cols;
  const int tiles = static_cast<int>((T + kTileM - 1) / kTileM);
  if (k <= 2) return launch_k<2>(map_x, map_w, a, tiles, sm_count, stream);
  if (k <= 4) return launch_k<4>(map_x, map_w, a, tiles, sm_count, stream);
  if (k <= 8) return launch_k<8>(map_x, map_w, a, tiles, sm_count, stream);
  return launch_k<16>(map_x, map_w, a, tiles, sm_count, stream);
}

}  // namespace moe
