// route.cu -- router product, softmax gate and top-k selection (one warp per token).
//
// logits[t,e] = sum_h x[t,h] * W_r[e,h] accumulated in fp32 in increasing h
// (each bf16 x bf16 product is exact in fp32, so an FMA chain in index order
// gives the same bits as a multiply-then-add chain); p = softmax over all E in
// fp32 (not renormalised over the selection); the k largest logits in
// descending order with ties to the lower expert index.
// (jina-ocr-v1: "64 routed experts ... Top-6 routing", kg.zhiyong.dev, section
// "The speed comes from three layers working together".)
//
// The router matrix is tiny (E x H bf16, 160 KB at E=64, H=1280) and is read
// through L1/L2 by every warp; x rows are read once.  The step is latency
// bound, not bandwidth bound.
#include "internal.h"
#include "ptx.cuh"

namespace lsv {
namespace {

constexpr int kRouteWarps = 8;
constexpr int kMaxPerLane = kMaxExperts / 32;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <int PER_LANE>
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(const bf16* __restrict__ x,
                                                                 const bf16* __restrict__ wr, int T, int H,
                                                                 int E, int k, int32_t* __restrict__ idx,
                                                                 float* __restrict__ w,
                                                                 float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  if (t >= T) return;

  float acc[PER_LANE];
#pragma unroll
  for (int j = 0; j < PER_LANE; ++j) acc[j] = 0.0f;

  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  for (int h8 = 0; h8 < H / 8; ++h8) {
    float xf[8];
    bf16x8_to_f32(__ldg(xr + h8), xf);
#pragma unroll
    for (int j = 0; j < PER_LANE; ++j) {
      const int e = lane + 32 * j;
      if (e < E) {
        float wf[8];
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(wr + (size_t)e * H) + h8), wf);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j] = fmaf(xf[i], wf[i], acc[j]);
      }
    }
  }

  // softmax over all E experts
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < PER_LANE; ++j)
    if (lane + 32 * j < E) m = fmaxf(m, acc[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.0f;
#pragma unroll
  for (int j = 0; j < PER_LANE; ++j)
    if (lane + 32 * j < E) z += expf(acc[j] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);

  if (logits) {
#pragma unroll
    for (int j = 0; j < PER_LANE; ++j)
      if (lane + 32 * j < E) logits[(size_t)t * E + lane + 32 * j] = acc[j];
  }

  // top-k: k rounds of a warp-wide (value desc, index asc) maximum
  uint32_t taken = 0;
  for (int s = 0; s < k; ++s) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < PER_LANE; ++j) {
      const int e = lane + 32 * j;
      if (e < E && !(taken & (1u << j)) && (acc[j] > bv || (acc[j] == bv && e < be))) {
        bv = acc[j];
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

}  // namespace

cudaError_t launch_route(const bf16* x, const bf16* wr, int T, int H, int E, int k, int32_t* idx, float* w,
                         float* logits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((T + kRouteWarps - 1) / kRouteWarps), block(kRouteWarps * 32);
  if (E <= 32)
    route_kernel<1><<<grid, block, 0, s>>>(x, wr, T, H, E, k, idx, w, logits);
  else if (E <= 64)
    route_kernel<2><<<grid, block, 0, s>>>(x, wr, T, H, E, k, idx, w, logits);
  else if (E <= 128)
    route_kernel<4><<<grid, block, 0, s>>>(x, wr, T, H, E, k, idx, w, logits);
  else
    route_kernel<kMaxPerLane><<<grid, block, 0, s>>>(x, wr, T, H, E, k, idx, w, logits);
  return cudaGetLastError();
}

}  // namespace lsv
