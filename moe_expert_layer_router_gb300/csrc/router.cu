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
// After the K loop the logit tile (S > 1: each CTA's partial) goes from TMEM
// to shared memory, and after a cluster barrier CTA c finishes tokens
// [c 128 / S, (c + 1) 128 / S) with Q = 4 S threads per token, 16 warps in
// all.  Thread p of a token owns experts 4 Q m + 4 p + {0..3} and reads each
// as the sum of the S partials (distributed shared memory, in CTA order) plus
// the bias.  The selection takes three passes over a thread's logits: the
// thread's few largest values give a threshold that the token's k-th largest
// logit cannot be below; the logits at or above it are marked in a bitmask;
// only the marked ones are inserted into the thread's top-k list (strictly
// greater replaces, so among equal logits the lower expert index stays
// ahead).  The Q lists and softmax normalisers of a token are then merged by
// shuffles, ordering equal logits by expert index, which selects exactly what
// one scan of the whole row would.
#include <math.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kStages = 4;
// warp 0: TMA producer, warp 1: MMA issuer, warps 2..17: TMEM copy-out and
// the top-k selection
constexpr int kEpiWarps = 16;
constexpr int kThreads = 64 + 32 * kEpiWarps;
// Each token tile walks its K slice starting at a tile-dependent k-step (and
// wraps around), so that the CTAs running at once do not all read the same
// router-weight k-block (and the same column offset of their token rows) at
// the same moment.
constexpr bool kRotateK = true;
constexpr int kABytes = kTileM * kTileK * 2;
constexpr int kMaxBBytes = 256 * kTileK * 2;
// CTA pairs (one cluster of 2 per 256 tokens, K unsplit): each CTA loads its
// 128 token rows and half of the router rows per stage, so a stage is at most
// 32 KB and six fit where a single CTA fits four 48 KB stages.
constexpr int kPairStages = 6;
constexpr int kMaxStages = kPairStages;
template <bool PAIR>
constexpr int stages_of() { return PAIR ? kPairStages : kStages; }
template <bool PAIR>
constexpr int b_slot_bytes() { return PAIR ? kMaxBBytes / 2 : kMaxBBytes; }

struct __align__(16) RouterCtl {
  float bias[kMaxExperts];  // first, so that four experts' biases are one 16-byte load
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = 1024 + size_t(kStages) * (kABytes + kMaxBBytes) + sizeof(RouterCtl);
constexpr int kMaxSplit = 8;  // CTAs per cluster (portable cluster size)
// Partial logit tile of one CTA, [128 tokens][E_pad + 4] fp32, in the stage
// area once the main loop is over (the +4 skews rows across banks).
static_assert(kTileM * (256 + 4) * 4 <= kStages * (kABytes + kMaxBBytes), "partial tile fits");
static_assert(kPairStages * (kABytes + kMaxBBytes / 2) == kStages * (kABytes + kMaxBBytes),
              "both layouts put the control block at the same offset");

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

// Gate weights of one token from its top-k list and softmax normaliser, which
// the Q threads of the token hold alike (Q a power of two; thread p is lane
// p of the token's group).  Thread p computes slots j = p, p + Q, ...; every
// thread then sums all k weights in slot order (the same fp32 sum as one
// thread would form) and writes its own slots.
template <int KMAX>
__device__ __forceinline__ void finish_token(const RouterArgs& a, int64_t t, bool valid, int p,
                                             int Q, const float (&tv)[KMAX], const int (&ti)[KMAX],
                                             float run_max, float run_sum) {
  const int k = a.k;
  const int base = (threadIdx.x & 31) & ~(Q - 1);  // lane of thread 0 of the group
  float w[KMAX];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    float v = 0.0f;
    if (j < k && (j & (Q - 1)) == p) {
      bad |= ti[j] < 0;
      if (a.score == 0) {
        v = a.renormalize ? expf(tv[j] - tv[0]) : expf(tv[j] - run_max) / run_sum;
      } else {
        v = 1.0f / (1.0f + expf(-tv[j]));
      }
    }
    w[j] = __shfl_sync(0xffffffffu, v, base + (j & (Q - 1)));
  }
  float denom = 0.0f;
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (j < k) denom += w[j];
  if (bad && valid) atomicOr(a.err, kErrNoSelect);
  const float norm = a.renormalize ? a.route_scale / denom : a.route_scale;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (valid && j < k && (j & (Q - 1)) == p) {
      a.topk_ids[t * k + j] = ti[j];
      a.topk_w[t * k + j] = w[j] * norm;
    }
  }
}

// PAIR: the cluster is a CTA pair that owns 256 tokens (CTA r: rows 128 r ..
// 128 r + 127) over all of H; one thread of the even CTA issues M = 256 pair
// MMAs whose B (the E_pad router rows) is split between the two CTAs, and each
// CTA's TMEM receives its own 128 x E_pad logit tile.  Otherwise the cluster
// is the K split of one 128-token tile.
template <int KMAX, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap map_x,
                  const __grid_constant__ CUtensorMap map_w, const RouterArgs a) {
  constexpr int kSt = stages_of<PAIR>();
  constexpr int kBSlot = b_slot_bytes<PAIR>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // router rows per TMA box: E_pad / 2 (a pair CTA loads one box, a single CTA two)
  const int b_half_rows = a.E_pad / 2;
  const int b_bytes = (PAIR ? 1 : 2) * b_half_rows * kTileK * 2;  // this CTA's B per stage
  const int stage_bytes = kABytes + b_bytes;
  uint8_t* a_tiles = smem;
  uint8_t* b_tiles = smem + kSt * kABytes;
  RouterCtl& c = *reinterpret_cast<RouterCtl*>(smem + kSt * (kABytes + kBSlot));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = ptx::cluster_ctarank();
  const bool leader = crank == 0;
  // K split of this token tile, and this CTA's slice index in it
  const int S = PAIR ? 1 : static_cast<int>(ptx::cluster_nctarank());
  const int kr = PAIR ? 0 : static_cast<int>(crank);
  const int tile = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x) / S;
  const int64_t m0 = PAIR ? int64_t(tile) * (2 * kTileM) + int64_t(crank) * kTileM
                          : int64_t(tile) * kTileM;
  // this call's router matrix and bias (a layer stack indexes its tables)
  const float* bias = a.bias;
  const void* map_w_ptr = &map_w;
  if (a.table.w_table) {
    const int l = resolve_layer(a.table.layer, a.table.num_layers, a.err);
    map_w_ptr = a.table.w_table + l;
    bias = a.table.bias_table[l];
  }

  for (int i = threadIdx.x; i < a.E_pad; i += kThreads)
    c.bias[i] = bias && i < a.E ? bias[i] : 0.0f;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      ptx::mbar_init(&c.full[s], 1);
      ptx::mbar_init(&c.empty[s], 1);
    }
    ptx::mbar_init(&c.tfull, 1);
    ptx::mbar_init(&c.drain, 1);
    c.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    if (PAIR) {
      ptx::tmem_alloc_pair(&c.tmem_base, a.tmem_cols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&c.tmem_base, a.tmem_cols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();  // both CTAs' barriers exist before either signals them
  ptx::tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  volatile int* abort = &c.abort;
  // the softmax normaliser over all E is needed only for unrenormalised softmax
  const bool need_norm = a.score == 0 && !a.renormalize;
  const int kb_all = a.H / kTileK;
  const int kb0 = kr * kb_all / S;  // this CTA's K slice (S <= kb_all)
  const int kb1 = (kr + 1) * kb_all / S;
  const int kb_n = kb1 - kb0;
  const int rot = kRotateK ? tile % kb_n : 0;  // the same in both CTAs of a pair

  if (warp == 0) {
    if (lane == 0) {
      // PAIR: both CTAs' copies of a stage complete on the even CTA's barrier
      const uint32_t full0 = ptx::mapa(ptx::smem_u32(&c.full[0]), 0);
      uint32_t it = 0;
      for (int i = 0; i < kb_n; ++i, ++it) {
        const int kb = kb0 + (i + rot) % kb_n;
        const int s = it % kSt;
        const uint32_t ph = (it / kSt) & 1;
        if (!ptx::mbar_wait(&c.empty[s], ph ^ 1, abort, a.err)) break;
        if (PAIR) {
          const uint32_t fb = full0 + s * 8;
          if (leader) ptx::mbar_arrive_expect_tx(&c.full[s], 2 * stage_bytes);
          ptx::tma_load_2d_pair(a_tiles + s * kABytes, &map_x, fb, kb * kTileK, int32_t(m0));
          ptx::tma_load_2d_pair(b_tiles + s * kBSlot, map_w_ptr, fb, kb * kTileK,
                                int32_t(crank) * b_half_rows);
        } else {
          ptx::mbar_arrive_expect_tx(&c.full[s], stage_bytes);
          ptx::tma_load_2d(a_tiles + s * kABytes, &map_x, &c.full[s], kb * kTileK, int32_t(m0));
          ptx::tma_load_2d(b_tiles + s * kBSlot, map_w_ptr, &c.full[s], kb * kTileK, 0);
          ptx::tma_load_2d(b_tiles + s * kBSlot + b_half_rows * kTileK * 2, map_w_ptr,
                           &c.full[s], kb * kTileK, b_half_rows);
        }
      }
      // no copy may be in flight at exit (PAIR: the even CTA's barriers see
      // both CTAs' copies; the odd CTA waits at the final cluster barrier)
      if (*abort && (!PAIR || leader)) {
        const uint32_t first = it > kSt ? it - kSt : 0;
        for (uint32_t j = first; j < it; ++j)
          drain_wait(&c.full[j % kSt], (j / kSt) & 1, a.err);
      }
    }
  } else if (warp == 1) {
    if (PAIR && lane == 0 && leader) {
      const uint32_t idesc = ptx::idesc_bf16(2 * kTileM, a.E_pad);
      bool ok = true;
      for (int i = 0; i < kb_n; ++i) {
        const int s = i % kSt;
        const uint32_t ph = (i / kSt) & 1;
        if (!ptx::mbar_wait(&c.full[s], ph, abort, a.err)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint64_t da = ptx::sw128_desc(ptx::smem_u32(a_tiles + s * kABytes));
        const uint64_t db = ptx::sw128_desc(ptx::smem_u32(b_tiles + s * kBSlot));
#pragma unroll
        for (int k = 0; k < kTileK / 16; ++k)
          ptx::mma_f16_pair(tmem_base, da + 2 * k, db + 2 * k, idesc, (i != 0) || (k != 0));
        ptx::mma_commit_pair_mc(&c.empty[s], 0x3);
      }
      if (ok) ptx::mma_commit_pair_mc(&c.tfull, 0x3);
      // every pair MMA issued by this thread has finished once `drain` flips
      ptx::mma_commit_pair_mc(&c.drain, 0x1);
      drain_wait(&c.drain, 0, a.err);
    } else if (!PAIR && lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16(kTileM, a.E_pad);
      bool ok = true;
      for (int i = 0; i < kb_n; ++i) {
        const int s = i % kSt;
        const uint32_t ph = (i / kSt) & 1;
        if (!ptx::mbar_wait(&c.full[s], ph, abort, a.err)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint64_t da = ptx::sw128_desc(ptx::smem_u32(a_tiles + s * kABytes));
        const uint64_t db = ptx::sw128_desc(ptx::smem_u32(b_tiles + s * kBSlot));
#pragma unroll
        for (int k = 0; k < kTileK / 16; ++k)
          ptx::mma_f16(tmem_base, da + 2 * k, db + 2 * k, idesc, (i != 0) || (k != 0));
        ptx::mma_commit(&c.empty[s]);
      }
      if (ok) ptx::mma_commit(&c.tfull);
      ptx::mma_commit(&c.drain);
      drain_wait(&c.drain, 0, a.err);
    }
  } else {
    // Logit tile -> this CTA's shared memory, row = token (S > 1: the partial
    // over this CTA's K slice).  Warp w may read TMEM lane quarter w % 4; the
    // kEpiWarps / 4 warps of a quarter take every (kEpiWarps / 4)-th 32-column
    // chunk.
    const int q = warp & 3;
    const int r = q * 32 + lane;
    float* part = reinterpret_cast<float*>(smem) + r * (a.E_pad + 4);
    if (ptx::mbar_wait(&c.tfull, 0, abort, a.err)) {
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c0 = 32 * ((warp - 2) >> 2); c0 < a.E_pad; c0 += 32 * (kEpiWarps / 4)) {
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
  }

  ptx::cluster_sync();  // every CTA's logit tile is in its shared memory
  if (warp >= 2) {
    // CTA c finishes tokens [c 128 / S, (c + 1) 128 / S) with Q = 4 S adjacent
    // threads per token (Q <= 32 divides the warp).  Thread p of a token owns
    // experts 4 Q m + 4 p + {0..3}, m = 0..nchunk-1 (at most 64 of them), and
    // reads each as the sum of the S partial tiles in CTA order plus the bias.
    const int Q = 4 * S;
    const int et = threadIdx.x - 64;
    const int p = et & (Q - 1);
    const int tl = kr * (kTileM / S) + et / Q;
    const int64_t t = m0 + tl;
    const bool valid = t < a.T;
    const int nchunk = (a.E_pad + 4 * Q - 1) / (4 * Q);
    const int row = tl * (a.E_pad + 4) + 4 * p;  // float index of this thread's first expert
    float* own = reinterpret_cast<float*>(smem) + row;
    uint32_t peer[kMaxSplit];
#pragma unroll
    for (int j = 0; j < kMaxSplit; ++j)
      peer[j] = j < S ? ptx::mapa(ptx::smem_u32(own), j) : 0u;
    // Logits of experts 4 Q m + 4 p + {0..3}: the S partials summed in CTA
    // order (this CTA's own from local shared memory), plus the bias.  Pass 1
    // stores them over this CTA's own partial of those experts, which no other
    // CTA reads (CTA j reads only the rows of the tokens it finishes).
    auto logits4 = [&](int m, float (&v)[4]) {
      float4 acc = *reinterpret_cast<const float4*>(own + 4 * Q * m);
      if (S > 1) {
        acc = kr == 0 ? acc : ptx::ld_cluster_f32x4(peer[0] + 16u * Q * m);
#pragma unroll
        for (int j = 1; j < kMaxSplit; ++j)
          if (j < S) {
            const float4 pv = j == kr ? *reinterpret_cast<const float4*>(own + 4 * Q * m)
                                      : ptx::ld_cluster_f32x4(peer[j] + 16u * Q * m);
            acc.x += pv.x;
            acc.y += pv.y;
            acc.z += pv.z;
            acc.w += pv.w;
          }
      }
      const float4 b = *reinterpret_cast<const float4*>(&c.bias[4 * Q * m + 4 * p]);
      v[0] = acc.x + b.x;
      v[1] = acc.y + b.y;
      v[2] = acc.z + b.z;
      v[3] = acc.w + b.w;
    };

    // Pass 1: logits out, the softmax normaliser, and this thread's kTop
    // largest logits.  With m = ceil(k / Q) <= kTop, the Q threads' m-th
    // largest values are Q m >= k logits of the token, so their minimum theta
    // is at most the token's k-th largest logit: every selected expert has a
    // logit >= theta.
    constexpr int kTop = (KMAX + 3) / 4;
    float top[kTop];
#pragma unroll
    for (int i = 0; i < kTop; ++i) top[i] = -INFINITY;
    float run_max = -INFINITY, run_sum = 0.0f;  // softmax over all E (online)
    float* lrow = (valid && a.logits_out) ? a.logits_out + t * a.E : nullptr;
    // chunks of this thread that hold at least one expert < E
    const int n_m = a.E > 4 * p ? min(nchunk, (a.E - 4 * p + 4 * Q - 1) / (4 * Q)) : 0;
#pragma unroll 2
    for (int m = 0; m < n_m; ++m) {
      const int e0 = 4 * Q * m + 4 * p;
      float v[4];
      logits4(m, v);
      *reinterpret_cast<float4*>(own + 4 * Q * m) = make_float4(v[0], v[1], v[2], v[3]);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if (e0 + h < a.E) {
          if (lrow) lrow[e0 + h] = v[h];
          float x = v[h];
#pragma unroll
          for (int i = 0; i < kTop; ++i) {
            const float hi = fmaxf(top[i], x);
            x = fminf(top[i], x);
            top[i] = hi;
          }
          if (need_norm) softmax_add(run_max, run_sum, v[h]);
        }
      }
    }
    const int mth = ((a.k + Q - 1) / Q < kTop ? (a.k + Q - 1) / Q : kTop) - 1;
    float theta = top[0];
#pragma unroll
    for (int i = 1; i < kTop; ++i)
      if (i == mth) theta = top[i];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1)
      if (d < Q) theta = fminf(theta, __shfl_xor_sync(0xffffffffu, theta, d));

    // Pass 2: the candidates (logit >= theta) as a bitmask of positions 4 m + h.
    uint64_t cand = 0;
#pragma unroll 4
    for (int m = 0; m < n_m; ++m) {
      const int e0 = 4 * Q * m + 4 * p;
      const float4 v = *reinterpret_cast<const float4*>(own + 4 * Q * m);
      const float vh[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int h = 0; h < 4; ++h)
        if (e0 + h < a.E && vh[h] >= theta) cand |= 1ull << (4 * m + h);
    }

    // Pass 3: the candidates in increasing expert order into the top-k list
    // (strictly greater replaces, so the lower index stays ahead among equal
    // logits).  The warp iterates as long as any lane has a candidate left.
    float tv[KMAX];
    int ti[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      tv[i] = -INFINITY;
      ti[i] = -1;
    }
    while (__any_sync(0xffffffffu, cand != 0)) {
      if (cand != 0) {
        const int i = __ffsll(static_cast<long long>(cand)) - 1;
        cand &= cand - 1;
        const int m = i >> 2, h = i & 3;
        topk_insert<KMAX>(tv, ti, own[4 * Q * m + h], 4 * Q * m + 4 * p + h);
      }
    }

    // merge the Q lists of the token (adjacent lanes)
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      if (d < Q) {
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
    finish_token<KMAX>(a, t, valid, p, Q, tv, ti, run_max, run_sum);
  }
  ptx::cluster_sync();  // no CTA leaves while a peer still reads its logit tile

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (PAIR)
      ptx::tmem_dealloc_pair(tmem_base, a.tmem_cols);
    else
      ptx::tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

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
    cudaLaunchConfig_t cfg = cluster_config(split, split, nullptr, &attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, router_kernel<KMAX, false>, &cfg) == cudaSuccess &&
        n > 0)
      break;
    cudaGetLastError();
  }
  cached = split;
  return split;
}

template <int KMAX>
cudaError_t launch_k(const CUtensorMap& mx, const CUtensorMap& mw, const RouterArgs& a, int tiles,
                     int sm_count, cudaStream_t stream) {
  // both kernels may use the full shared memory (the cluster occupancy query
  // below depends on it)
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(router_kernel<KMAX, false>),
                                   static_cast<int>(kSmemBytes));
  if (e == cudaSuccess)
    e = ensure_smem_attr(reinterpret_cast<const void*>(router_kernel<KMAX, true>),
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
  // unsplit tiles: CTA pairs over 256 tokens each (router-row halves of a
  // multiple of 16 rows)
  const bool pair = split == 1 && tiles > 1 && a.E_pad % 32 == 0;
  cudaLaunchAttribute attr;
  if (pair) {
    cudaLaunchConfig_t cfg = cluster_config(2 * ((tiles + 1) / 2), 2, stream, &attr);
    e = cudaLaunchKernelEx(&cfg, router_kernel<KMAX, true>, mx, mw, a);
  } else {
    cudaLaunchConfig_t cfg = cluster_config(tiles * split, split, stream, &attr);
    e = cudaLaunchKernelEx(&cfg, router_kernel<KMAX, false>, mx, mw, a);
  }
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
