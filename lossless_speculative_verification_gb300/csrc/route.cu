// route.cu -- router product, softmax gate and top-k selection.
//
// logits[t,e] = sum_h x[t,h] * W_r[e,h] with fp32 accumulation; p = softmax
// over all E in fp32 (not renormalised over the selection); the k largest
// logits in descending order with ties to the lower expert index.
// (jina-ocr-v1: "64 routed experts ... Top-6 routing", kg.zhiyong.dev, section
// "The speed comes from three layers working together".)
//
// Up to 256 tokens (decode sizes) the router runs on CUDA cores, latency-first:
// one CTA takes TT tokens.  Warp w computes experts 4w..4w+3 (then 4w+64..)
// for all TT tokens; inside a warp each lane owns a contiguous 8-element slice
// of every 256-element block of h (16-byte loads of x and W), and the 32
// partial sums are combined by a fixed butterfly.  The summation order is fixed, so
// results are run-to-run identical; it differs from a sequential sum only by
// fp32 rounding (far below the router gaps the selection depends on).  The
// E logits of each token then go through shared memory to one warp per token
// for the softmax and the k selection rounds.
#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lsv {
namespace {

constexpr int kRouteWarps = 16;
constexpr int kRouteTcMinTokens = 256;  // above this many tokens the router runs on tensor cores
constexpr int kExpPerWarp = 4;
constexpr int kLoadAhead = 5;  // 16-byte pieces per row and lane in flight together (H = 1280: a whole row)

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <int TT>
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(const bf16* __restrict__ x,
                                                                 const bf16* __restrict__ wr, int T, int H,
                                                                 int E, int k, int32_t* __restrict__ idx,
                                                                 float* __restrict__ w,
                                                                 float* __restrict__ logits, const RouteSlots sl) {
  __shared__ float lg[TT][kMaxExperts];
  __shared__ int sel_row[kMaxTopK];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * TT;
  const int nt = min(TT, T - t0);
  const int n8 = H / 8;  // 16-byte groups per row
  const bool slots = TT == 1 && sl.xperm != nullptr;

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

  // softmax + top-k: one warp per token.  The selection is by rank: an expert's
  // rank is the number of experts with a larger logit, or an equal logit and a
  // lower index, so ranks are distinct and ties go to the lower index.
  for (int i = warp; i < nt; i += kRouteWarps) {
    const int t = t0 + i;
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, lg[i][e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.0f;
    for (int e = lane; e < E; e += 32) z += expf(lg[i][e] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (logits)
      for (int e = lane; e < E; e += 32) logits[(size_t)t * E + e] = lg[i][e];
    for (int e = lane; e < E; e += 32) {
      const float v = lg[i][e];
      int r = 0;
      for (int e2 = 0; e2 < E; ++e2) {
        const float v2 = lg[i][e2];
        r += (v2 > v || (v2 == v && e2 < e)) ? 1 : 0;
      }
      if (r < k) {
        idx[(size_t)t * k + r] = e;
        w[(size_t)t * k + r] = expf(v - m) / z;
        if (slots) {
          // the next free row of expert e's region
          const int row = e * T + atomicAdd(&sl.slots[e], 1);
          sl.inv[(size_t)t * k + r] = row;
          sel_row[r] = row;
        }
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
  const dim3 block(kRouteWarps * 32);
  // about one CTA per SM at decode sizes; more tokens per CTA once T is large
  // one CTA per token (at most 256 tokens here; more go to the tensor-core router above)
  return launch_pdl(route_kernel<1>, dim3(T), block, 0, s, x, wr, T, H, E, k, idx, w, logits, sl);
}

}  // namespace lsv
