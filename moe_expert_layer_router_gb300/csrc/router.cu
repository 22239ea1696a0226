// Router: logits = x W_r^T on the tensor cores, with top-k selection and the
// gate weights fused into the epilogue ("gated routing" of "Memory-Compute
// Disaggregation for Large-Model Inference: AFD Architecture Analysis and
// Performance Validation", section 3, Data-Flow Closed Loop step 3; k of E
// experts per token as in "ASAP: A DiSaggregated and Asynchronous Inference
// System for MoE Prefill", section 5.1).
//
// One CTA per 128 tokens.  The E (<= 256, padded to a multiple of 16) router
// rows form the N side of one 128 x E_pad tcgen05 accumulator, so each
// epilogue thread holds one token's complete logit row: it scans the row
// once, keeping the k largest (strictly greater replaces, so among equal
// logits the lower expert index stays ahead) and a running softmax
// normaliser, then writes ids, weights and optionally the fp32 logits.
#include <math.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 192;
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
// an earlier (lower-index) equal value ahead of a later one.
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
  const int64_t m0 = int64_t(blockIdx.x) * kTileM;

  for (int i = threadIdx.x; i < a.E; i += kThreads) c.bias[i] = a.bias ? a.bias[i] : 0.0f;
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
  const int kb_n = a.H / kTileK;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      for (int kb = 0; kb < kb_n; ++kb, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!ptx::mbar_wait(&c.empty[s], ph ^ 1, abort, a.err)) break;
        ptx::mbar_arrive_expect_tx(&c.full[s], stage_bytes);
        ptx::tma_load_2d(a_tiles + s * kABytes, &map_x, &c.full[s], kb * kTileK, int32_t(m0));
        ptx::tma_load_2d(b_tiles + s * kMaxBBytes, &map_w, &c.full[s], kb * kTileK, 0);
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
      for (int kb = 0; kb < kb_n; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = (kb / kStages) & 1;
        if (!ptx::mbar_wait(&c.full[s], ph, abort, a.err)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint64_t da = ptx::sw128_desc(ptx::smem_u32(a_tiles + s * kABytes));
        const uint64_t db = ptx::sw128_desc(ptx::smem_u32(b_tiles + s * kMaxBBytes));
#pragma unroll
        for (int k = 0; k < kTileK / 16; ++k)
          ptx::mma_f16(tmem_base, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);
        ptx::mma_commit(&c.empty[s]);
      }
      if (ok) ptx::mma_commit(&c.tfull);
      ptx::mma_commit(&c.drain);
      drain_wait(&c.drain, 0, a.err);
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
            if (lv[j] > run_max) {
              run_sum = run_sum * expf(run_max - lv[j]) + 1.0f;
              run_max = lv[j];
            } else {
              run_sum += expf(lv[j] - run_max);
            }
          }
        }
      }
      if (valid) {
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
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

template <int KMAX>
cudaError_t launch_k(const CUtensorMap& mx, const CUtensorMap& mw, const RouterArgs& a, int grid,
                     cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(router_kernel<KMAX>),
                                   static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  router_kernel<KMAX><<<grid, kThreads, kSmemBytes, stream>>>(mx, mw, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const CUtensorMap& map_x, const CUtensorMap& map_w, int64_t T, int H,
                          int E, int E_pad, int k, int score, int renormalize, float route_scale,
                          const float* bias, int32_t* topk_ids, float* topk_w, float* logits_out,
                          uint32_t* err, cudaStream_t stream) {
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
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(E_pad)) cols <<= 1;
  a.tmem_cols = cols;
  const int grid = static_cast<int>((T + kTileM - 1) / kTileM);
  if (k <= 2) return launch_k<2>(map_x, map_w, a, grid, stream);
  if (k <= 4) return launch_k<4>(map_x, map_w, a, grid, stream);
  if (k <= 8) return launch_k<8>(map_x, map_w, a, grid, stream);
  return launch_k<16>(map_x, map_w, a, grid, stream);
}

}  // namespace moe
