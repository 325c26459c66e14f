// route.cu -- router product, softmax gate and top-k selection.
//
// logits[t,e] = sum_h x[t,h] * W_r[e,h] with fp32 accumulation; p = softmax
// over all E in fp32 (not renormalised over the selection); the k largest
// logits in descending order with ties to the lower expert index.  (The
// jina-ocr-v1 decoder sends each token to 6 of its 64 routed experts;
// kg.zhiyong.dev, section "The speed comes from three layers working together".)
//
// Up to 256 tokens (decode sizes) the router runs on CUDA cores, latency-first.
// Up to 128 tokens: one cluster of eight CTAs per one or two tokens, each CTA
// computing an eighth of the tokens' logits, which meet in the leader CTA's
// shared memory; from 129 to 256 tokens: one CTA per token.  In both, each lane
// owns a contiguous 8-element slice of every 256-element block of h (16-byte
// loads of x and W) and the 32 partial sums are combined by a fixed butterfly;
// the summation order is fixed, so results are run-to-run identical and equal
// between the two forms; it differs from a sequential sum only by fp32 rounding
// (far below the router gaps the selection depends on).  One warp per token
// takes the softmax and the k selection rounds.  Above 256 tokens the product
// is a dense contraction on tcgen05 (below).
#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lsv {
namespace {

constexpr int kRouteTcMinTokens = 256;  // above this many tokens the router runs on tensor cores
// Router form by token count (measured at 1..256 tokens): clusters of one token up to
// LSV_ROUTE_TT1_MAX, clusters of two tokens up to LSV_ROUTE_CLUSTER_MAX, then one CTA per token.
#ifndef LSV_ROUTE_TT1_MAX
#define LSV_ROUTE_TT1_MAX 64
#endif
#ifndef LSV_ROUTE_CLUSTER_MAX
#define LSV_ROUTE_CLUSTER_MAX 128
#endif
constexpr int kLoadAhead = 5;  // 16-byte pieces per row and lane in flight together (H = 1280: a whole row)

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// One cluster of kRcCluster CTAs per TT tokens.  CTA r computes the logits of
// experts [r*per, r*per + per) for the cluster's tokens (one warp per expert in
// turn: each lane owns a contiguous 8-element slice of every 256-element block
// of h, kLoadAhead 16-byte pieces of the weight row in flight together, a fixed
// butterfly over the lanes) and stores them into the leader CTA's shared
// memory.  After the cluster barrier the leader's warp i takes token i's
// softmax and top-k, and all its warps place the tokens' rows.  Splitting the
// experts over eight SMs cuts the router weight bytes each SM reads per token
// eightfold; several tokens per cluster cut the weight bytes read in all.
constexpr int kRcCluster = 8;
constexpr int kRcWarps = 8;

// Softmax over the E logits in lg (fp32) and the k largest, descending, ties to the lower
// expert: k rounds of a warp-wide maximum over the experts not yet taken.  Lane r returns
// the r-th choice (expert, probability) in (*e_out, *p_out); lanes >= k return -1.  kPerLane
// experts per lane (E <= 32 kPerLane): one warp's dependent chain, so it is instantiated for
// the smallest count that holds E.
template <int kPerLane>
__device__ __forceinline__ void softmax_topk_warp_n(const float* lg, int E, int k, int* e_out, float* p_out) {
  const int lane = threadIdx.x & 31;
  float v[kPerLane];
  int taken = 0;  // bit j: expert lane + 32j is absent or already chosen
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? lg[e] : -INFINITY;
    if (e < E)
      m = fmaxf(m, v[j]);
    else
      taken |= 1 << j;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.0f;
#pragma unroll
  for (int j = 0; j < kPerLane; ++j)
    if (lane + 32 * j < E) z += expf(v[j] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  int my_e = -1;
  float my_v = 0.0f;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      const int e = lane + 32 * j;
      if (!((taken >> j) & 1) && (v[j] > bv || (v[j] == bv && e < be))) {
        bv = v[j];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be < E && (be & 31) == lane) taken |= 1 << (be >> 5);
    if (lane == r) {
      my_e = be < E ? be : -1;
      my_v = bv;
    }
  }
  *e_out = my_e;
  *p_out = my_e >= 0 ? expf(my_v - m) / z : 0.0f;
}

__device__ __forceinline__ void softmax_topk_warp(const float* lg, int E, int k, int* e_out, float* p_out) {
  if (E <= 64)
    softmax_topk_warp_n<2>(lg, E, k, e_out, p_out);
  else if (E <= 128)
    softmax_topk_warp_n<4>(lg, E, k, e_out, p_out);
  else
    softmax_topk_warp_n<kMaxExperts / 32>(lg, E, k, e_out, p_out);
}

template <int TT>
__global__ void __launch_bounds__(kRcWarps * 32) route_cluster_kernel(const bf16* __restrict__ x,
                                                                      const bf16* __restrict__ wr, int T, int H,
                                                                      int E, int k, int32_t* __restrict__ idx,
                                                                      float* __restrict__ w,
                                                                      float* __restrict__ logits,
                                                                      const RouteSlots sl) {
  __shared__ float lg[TT][kMaxExperts];  // the leader's copy receives every CTA's logits
  __shared__ int sel_row[TT][kMaxTopK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();
  const int t0 = blockIdx.y * TT;
  const int nt = min(TT, T - t0);
  const int n8 = H / 8;  // 16-byte groups per row
  const int per = (E + kRcCluster - 1) / kRcCluster;
  const int e_lo = (int)rank * per, e_hi = min(E, e_lo + per);
  cluster_arrive_relaxed();  // the matching wait below: every CTA of the cluster is running
  pdl_wait();
  pdl_trigger();
  const uint32_t lg_leader = mapa_shared(smem_u32(&lg[0][0]), 0);
  bool waited = false;
  for (int e = e_lo + warp; e < e_hi; e += kRcWarps) {
    float acc[TT];
#pragma unroll
    for (int i = 0; i < TT; ++i) acc[i] = 0.0f;
    for (int c0 = lane; c0 < n8; c0 += 32 * kLoadAhead) {
      uint4 wv[kLoadAhead];
#pragma unroll
      for (int u = 0; u < kLoadAhead; ++u) {
        const int c = c0 + 32 * u;
        wv[u] = c < n8 ? __ldg(reinterpret_cast<const uint4*>(wr + (size_t)e * H) + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < TT; ++i) {
        uint4 xv[kLoadAhead];
#pragma unroll
        for (int u = 0; u < kLoadAhead; ++u) {
          const int c = c0 + 32 * u;
          xv[u] = (c < n8 && i < nt) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + i) * H) + c)
                                     : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kLoadAhead; ++u) {
          float xf[8], wf[8];
          bf16x8_to_f32(xv[u], xf);
          bf16x8_to_f32(wv[u], wf);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i] = fmaf(xf[j], wf[j], acc[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < TT; ++i)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
    if (!waited) {
      cluster_wait();
      waited = true;
    }
    if (lane == 0)
#pragma unroll
      for (int i = 0; i < TT; ++i)
        st_shared_cluster_f32(lg_leader + 4u * (uint32_t)(i * kMaxExperts + e), acc[i]);
  }
  if (!waited) cluster_wait();
  cluster_sync();  // the leader's lg holds all E logits (release by the writers, acquire here)
  if (rank != 0) return;

  const bool slots = sl.xperm != nullptr;
  for (int i = warp; i < nt; i += kRcWarps) {
    const int t = t0 + i;
    if (logits)
      for (int e = lane; e < E; e += 32) logits[(size_t)t * E + e] = lg[i][e];
    int my_e;
    float my_p;
    softmax_topk_warp(lg[i], E, k, &my_e, &my_p);
    if (lane < k && my_e >= 0) {
      idx[(size_t)t * k + lane] = my_e;
      w[(size_t)t * k + lane] = my_p;
      if (slots) {
        // the next free row of expert my_e's region
        const int row = my_e * T + atomicAdd(&sl.slots[my_e], 1);
        sl.inv[(size_t)t * k + lane] = row;
        sel_row[i][lane] = row;
      }
    }
  }
  if (!slots) return;

  // place the tokens' rows at their k rows of the routed row space
  __syncthreads();
  for (int q = warp; q < nt * k; q += kRcWarps) {
    const int i = q / k, r = q - (q / k) * k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(t0 + i) * H);
    uint4* dst = reinterpret_cast<uint4*>(sl.xperm + (size_t)sel_row[i][r] * H);
    for (int c = lane; c < n8; c += 32) dst[c] = __ldg(src + c);
  }
}

// From 129 to 256 tokens: one CTA of 16 warps per token.  Warp w computes experts
// 4w..4w+3 (then 4w+64..) over the whole row, with the same lane layout and
// summation order as the cluster kernel, so both give the same logits bit for
// bit.  Measured faster than the clusters at 192 and 256 tokens (the clusters'
// CTAs outnumber the SMs' slots there).
constexpr int kRouteWarps = 16;
constexpr int kExpPerWarp = 4;

__global__ void __launch_bounds__(kRouteWarps * 32) route_token_kernel(const bf16* __restrict__ x,
                                                                       const bf16* __restrict__ wr, int T, int H,
                                                                       int E, int k, int32_t* __restrict__ idx,
                                                                       float* __restrict__ w,
                                                                       float* __restrict__ logits,
                                                                       const RouteSlots sl) {
  constexpr int TT = 1;
  __shared__ float lg[TT][kMaxExperts];
  __shared__ int sel_row[kMaxTopK];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * TT;
  const int nt = min(TT, T - t0);
  const int n8 = H / 8;  // 16-byte groups per row
  const bool slots = sl.xperm != nullptr;

  // warp w owns experts [4w, 4w+4), [4w+64, 4w+68), ...; each lane loads kLoadAhead 16-byte pieces
  // of each of the four rows (and of x) before it uses any, so that one memory round trip
  // covers a whole row block
  for (int e0 = warp * kExpPerWarp; e0 < E; e0 += kRouteWarps * kExpPerWarp) {
    float acc[kExpPerWarp][TT];
#pragma unroll
    for (int q = 0; q < kExpPerWarp; ++q)
#pragma unroll
      for (int i = 0; i < TT; ++i) acc[q][i] = 0.0f;
    for (int c0 = lane; c0 < n8; c0 += 32 * kLoadAhead) {
      uint4 wv[kExpPerWarp][kLoadAhead];
      uint4 xv[TT][kLoadAhead];
#pragma unroll
      for (int u = 0; u < kLoadAhead; ++u) {
        const int c = c0 + 32 * u;
#pragma unroll
        for (int q = 0; q < kExpPerWarp; ++q)
          wv[q][u] = (c < n8 && e0 + q < E) ? __ldg(reinterpret_cast<const uint4*>(wr + (size_t)(e0 + q) * H) + c)
                                            : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < TT; ++i)
          xv[i][u] = (c < n8 && i < nt) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + i) * H) + c)
                                        : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kLoadAhead; ++u)
#pragma unroll
        for (int i = 0; i < TT; ++i) {
          float xf[8];
          bf16x8_to_f32(xv[i][u], xf);
#pragma unroll
          for (int q = 0; q < kExpPerWarp; ++q) {
            float wf[8];
            bf16x8_to_f32(wv[q][u], wf);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[q][i] = fmaf(xf[j], wf[j], acc[q][i]);
          }
        }
    }
#pragma unroll
    for (int q = 0; q < kExpPerWarp; ++q)
#pragma unroll
      for (int i = 0; i < TT; ++i) {
        float v = acc[q][i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0 && e0 + q < E) lg[i][e0 + q] = v;
      }
  }
  __syncthreads();

  // softmax + top-k of the token by warp 0; lane r < k takes the r-th choice's row
  if (warp == 0) {
    const int t = t0;
    if (logits)
      for (int e = lane; e < E; e += 32) logits[(size_t)t * E + e] = lg[0][e];
    int my_e;
    float my_p;
    softmax_topk_warp(lg[0], E, k, &my_e, &my_p);
    if (lane < k && my_e >= 0) {
      idx[(size_t)t * k + lane] = my_e;
      w[(size_t)t * k + lane] = my_p;
      if (slots) {
        // the next free row of expert my_e's region
        const int row = my_e * T + atomicAdd(&sl.slots[my_e], 1);
        sl.inv[(size_t)t * k + lane] = row;
        sel_row[lane] = row;
      }
    }
  }
  if (!slots) return;

  // place the token's row at its k rows of the routed row space
  __syncthreads();
  if (warp < k) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t0 * H);
    uint4* dst = reinterpret_cast<uint4*>(sl.xperm + (size_t)sel_row[warp] * H);
    for (int c = lane; c < n8; c += 32) dst[c] = __ldg(src + c);
  }
}

// ----------------------------------------------------------------------------- tensor-core router
// For large T the router product is a dense contraction: one CTA per 128-token
// tile computes D[128 tokens x NPAD experts] = x_tile * W_r^T on tcgen05 (bf16
// in, fp32 accumulators in TMEM).  A row of D is one token's E logits and sits
// in one TMEM lane, so the epilogue thread of that lane does the softmax (an
// online max/sum) and the top-k (insertion in increasing expert order, strict
// comparison, so ties keep the lower expert) without talking to other threads.
constexpr int kRtThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kRtStages = 4;

template <int NPAD>
struct RtSmem {
  static constexpr int kA = 128 * 128;            // 128 tokens x 64 bf16
  static constexpr int kB = NPAD * 128;           // NPAD experts x 64 bf16
  static constexpr int kStage = kA + kB;
  static constexpr int kTotal = 1024 + kRtStages * kStage + (2 * kRtStages + 1) * 8 + 16;
};

template <int NPAD>
__global__ void __launch_bounds__(kRtThreads, 1) route_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                 const __grid_constant__ CUtensorMap wmap, int T,
                                                                 int H, int E, int k, int32_t* __restrict__ idx,
                                                                 float* __restrict__ w,
                                                                 float* __restrict__ logits, int* err,
                                                                 uint64_t wait_ns) {
  using SM = RtSmem<NPAD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRtStages * SM::kStage);
  uint64_t* empty = full + kRtStages;
  uint64_t* tfull = empty + kRtStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * 128;
  const int nk = H / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, NPAD);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      for (int kc = 0; kc < nk; ++kc) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, wait_ns)) {
          set_error(err, kErrTimeout);
          break;
        }
        uint8_t* a_s = smem + stage * SM::kStage;
        mbar_arrive_expect_tx(&full[stage], SM::kStage);
        tma_load_2d(a_s, &xmap, &full[stage], kc * 64, t0, pol);
        tma_load_2d(a_s + SM::kA, &wmap, &full[stage], kc * 64, 0, pol);
        if (++stage == kRtStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, NPAD);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kc = 0; kc < nk; ++kc) {
        if (!mbar_wait(&full[stage], phase, wait_ns)) {
          set_error(err, kErrTimeout);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_s = smem_u32(smem + stage * SM::kStage);
        const uint32_t b_s = a_s + SM::kA;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem_base, sdesc_kmajor_sw128(a_s + kk * 32), sdesc_kmajor_sw128(b_s + kk * 32), idesc,
                    (kc | kk) ? 1u : 0u);
        umma_commit(&empty[stage]);
        if (++stage == kRtStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // on a timeout the epilogue still gets its wake-up; every MMA issued has completed by then
      umma_commit(tfull);
      (void)ok;
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int t = t0 + 32 * q + lane;
    const bool got = mbar_wait(tfull, 0, wait_ns);
    if (!got) set_error(err, kErrTimeout);
    tc_fence_after_sync();
    float m = -INFINITY, z = 0.0f;
    float bv[kMaxTopK];
    int be[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      bv[s] = -INFINITY;
      be[s] = 0x7fffffff;
    }
    const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16);
    for (int c0 = 0; c0 < NPAD; c0 += 16) {
      uint32_t r[16];
      tmem_ld_32x32b_x16(t_row + c0, r);
      tmem_ld_wait();
      if (!got || t >= T) continue;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int e = c0 + j;
        if (e < E) {
          const float v = __uint_as_float(r[j]);
          if (logits) logits[(size_t)t * E + e] = v;
          // online softmax
          if (v > m) {
            z = z * expf(m - v) + 1.0f;
            m = v;
          } else {
            z += expf(v - m);
          }
          // insertion into the descending top-k list; strict > keeps the lower expert first on ties
#pragma unroll
          for (int s = kMaxTopK - 1; s >= 0; --s) {
            if (s < k && v > bv[s]) {
              if (s + 1 < kMaxTopK) {
                bv[s + 1] = bv[s];
                be[s + 1] = be[s];
              }
              bv[s] = v;
              be[s] = e;
            }
          }
        }
      }
    }
    if (got && t < T) {
#pragma unroll
      for (int s = 0; s < kMaxTopK; ++s)
        if (s < k) {
          idx[(size_t)t * k + s] = be[s];
          w[(size_t)t * k + s] = expf(bv[s] - m) / z;
        }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, NPAD);
  }
}

template <int NPAD>
cudaError_t run_route_tc(const bf16* x, const bf16* wr, int T, int H, int E, int k, int32_t* idx, float* w,
                         float* logits, int* err, int device, cudaStream_t s) {
  using SM = RtSmem<NPAD>;
  const cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(route_tc_kernel<NPAD>), SM::kTotal, device);
  if (e != cudaSuccess) return e;
  CUtensorMap xmap, wmap;
  if (!make_map(&xmap, x, T, H, 128) || !make_map(&wmap, wr, E, H, NPAD)) return cudaErrorInvalidValue;
  return launch_pdl(route_tc_kernel<NPAD>, dim3((T + 127) / 128), dim3(kRtThreads), SM::kTotal, s, xmap, wmap, T, H,
                    E, k, idx, w, logits, err, wait_limit_ns());
}

}  // namespace

cudaError_t launch_route(const bf16* x, const bf16* wr, int T, int H, int E, int k, int32_t* idx, float* w,
                         float* logits, cudaStream_t s, const RouteSlots* slots) {
  RouteSlots sl = {};
  if (slots) sl = *slots;
  if (T == 0) return cudaSuccess;
  static_assert(kSlotMaxTokens == kRouteTcMinTokens, "slot placement needs the one-token-per-CTA router");
  if (T > kRouteTcMinTokens) {
    if (slots) return cudaErrorInvalidValue;
    DeviceCtx* dc = nullptr;
    const cudaError_t e = device_ctx(&dc);
    if (e != cudaSuccess) return e;
    if (E <= 64) return run_route_tc<64>(x, wr, T, H, E, k, idx, w, logits, dc->err, dc->device, s);
    if (E <= 128) return run_route_tc<128>(x, wr, T, H, E, k, idx, w, logits, dc->err, dc->device, s);
    return run_route_tc<256>(x, wr, T, H, E, k, idx, w, logits, dc->err, dc->device, s);
  }
  if (T > LSV_ROUTE_CLUSTER_MAX)
    return launch_pdl(route_token_kernel, dim3(T), dim3(kRouteWarps * 32), 0, s, x, wr, T, H, E, k, idx, w, logits,
                      sl);
  // one cluster per TT tokens
  const int TT = T <= LSV_ROUTE_TT1_MAX ? 1 : 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kRcCluster, (T + TT - 1) / TT);
  cfg.blockDim = dim3(kRcWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kRcCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (TT == 1) return cudaLaunchKernelEx(&cfg, route_cluster_kernel<1>, x, wr, T, H, E, k, idx, w, logits, sl);
  return cudaLaunchKernelEx(&cfg, route_cluster_kernel<2>, x, wr, T, H, E, k, idx, w, logits, sl);
}

}  // namespace lsv
