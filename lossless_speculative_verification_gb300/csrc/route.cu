// route.cu -- router product, softmax gate and top-k selection.
//
// logits[t,e] = sum_h x[t,h] * W_r[e,h] with fp32 accumulation; p = softmax
// over all E in fp32 (not renormalised over the selection); the k largest
// logits in descending order with ties to the lower expert index.
// (jina-ocr-v1: "64 routed experts ... Top-6 routing", kg.zhiyong.dev, section
// "The speed comes from three layers working together".)
//
// One CTA takes TT tokens.  Warp w computes experts 4w..4w+3 (then 4w+64..)
// for all TT tokens; inside a warp each lane owns a contiguous 8-element slice
// of every 256-element block of h (16-byte loads of x and W), and the 32
// partial sums are combined by a fixed butterfly.  The summation order is fixed, so
// results are run-to-run identical; it differs from a sequential sum only by
// fp32 rounding (far below the router gaps the selection depends on).  The
// E logits of each token then go through shared memory to one warp per token
// for the softmax and the k selection rounds.
#include "internal.h"
#include "ptx.cuh"

namespace lsv {
namespace {

constexpr int kRouteWarps = 16;
constexpr int kExpPerWarp = 4;

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
                                                                 float* __restrict__ logits) {
  __shared__ float lg[TT][kMaxExperts];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * TT;
  const int nt = min(TT, T - t0);
  const int n8 = H / 8;  // 16-byte groups per row

  // warp w owns experts [4w, 4w+4), [4w+64, 4w+68), ...: four independent rows in flight per step
  for (int e0 = warp * kExpPerWarp; e0 < E; e0 += kRouteWarps * kExpPerWarp) {
    float acc[kExpPerWarp][TT];
#pragma unroll
    for (int q = 0; q < kExpPerWarp; ++q)
#pragma unroll
      for (int i = 0; i < TT; ++i) acc[q][i] = 0.0f;
#pragma unroll 5
    for (int c = lane; c < n8; c += 32) {
      uint4 wv[kExpPerWarp];
#pragma unroll
      for (int q = 0; q < kExpPerWarp; ++q)
        wv[q] = (e0 + q < E) ? __ldg(reinterpret_cast<const uint4*>(wr + (size_t)(e0 + q) * H) + c)
                             : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < TT; ++i) {
        if (i < nt) {
          float xf[8];
          bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + i) * H) + c), xf);
#pragma unroll
          for (int q = 0; q < kExpPerWarp; ++q) {
            float wf[8];
            bf16x8_to_f32(wv[q], wf);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[q][i] = fmaf(xf[j], wf[j], acc[q][i]);
          }
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

  // softmax + top-k: one warp per token
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
    uint32_t taken = 0;  // bit j: expert lane + 32 j already selected
    for (int s = 0; s < k; ++s) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
      for (int j = 0, e = lane; e < E; ++j, e += 32) {
        const float v = lg[i][e];
        if (!(taken & (1u << j)) && (v > bv || (v == bv && e < be))) {
          bv = v;
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
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == 0) {
        idx[(size_t)t * k + s] = be;
        w[(size_t)t * k + s] = expf(bv - m) / z;
      }
    }
  }
}

}  // namespace

cudaError_t launch_route(const bf16* x, const bf16* wr, int T, int H, int E, int k, int32_t* idx, float* w,
                         float* logits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 block(kRouteWarps * 32);
  // about one CTA per SM at decode sizes; more tokens per CTA once T is large
  if (T <= 256) return launch_pdl(route_kernel<1>, dim3(T), block, 0, s, x, wr, T, H, E, k, idx, w, logits);
  if (T <= 1024)
    return launch_pdl(route_kernel<4>, dim3((T + 3) / 4), block, 0, s, x, wr, T, H, E, k, idx, w, logits);
  return launch_pdl(route_kernel<8>, dim3((T + 7) / 8), block, 0, s, x, wr, T, H, E, k, idx, w, logits);
}

}  // namespace lsv
