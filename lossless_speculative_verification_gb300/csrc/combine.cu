// combine.cu -- gate-weighted combine of expert outputs, and the residual +
// RMSNorm update between stacked layers.
//
// combine:  out[t,:] = sum_{s<k} topk_w[t,s] * y_perm[inv[t*k+s],:] + y_shared[t,:]
// (the MoE layer output: gate-weighted routed experts plus the always-on
// shared experts; kg.zhiyong.dev, "The speed comes from three layers working
// together").  A gather, not a scatter: each output element is summed by one
// thread in slot order, so the result is deterministic without atomics.
//
// rmsnorm_residual:  x <- bf16(x + y);  h = bf16(x * rsqrt(mean(x^2) + eps))
#include "internal.h"
#include "ptx.cuh"

namespace lsv {
namespace {

constexpr int kCombThreads = 128;

__global__ void __launch_bounds__(kCombThreads) combine_kernel(const float* __restrict__ y_perm,
                                                               const int32_t* __restrict__ inv,
                                                               const float* __restrict__ topk_w,
                                                               const float* __restrict__ y_sh, int T, int H,
                                                               int k, bf16* __restrict__ out, int* err) {
  const int t = blockIdx.x;
  const int h4 = blockIdx.y * kCombThreads + threadIdx.x;  // group of 4 columns
  __shared__ int rows[kMaxTopK];
  pdl_wait();
  pdl_trigger();
  __shared__ float wts[kMaxTopK];
  if (threadIdx.x < k) {
    int r = inv[(size_t)t * k + threadIdx.x];
    if (r < 0 || r >= T * k) {  // never read outside y_perm
      if (blockIdx.y == 0) set_error(err, kErrDeviceIndex);
      r = -1;
    }
    rows[threadIdx.x] = r;
    wts[threadIdx.x] = topk_w[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  if (h4 * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < k; ++s) {
    if (rows[s] < 0) continue;
    const float4 v = __ldg(reinterpret_cast<const float4*>(y_perm + (size_t)rows[s] * H) + h4);
    const float w = wts[s];
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  if (y_sh) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(y_sh + (size_t)t * H) + h4);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(out + (size_t)t * H)[h4] = pk;
}

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_residual_kernel(bf16* __restrict__ x,
                                                                        const bf16* __restrict__ y,
                                                                        bf16* __restrict__ h, int H,
                                                                        float eps) {
  const int t = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  bf16* xr = x + (size_t)t * H;
  const bf16* yr = y + (size_t)t * H;
  bf16* hr = h + (size_t)t * H;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += kNormThreads) {
    const bf16 v = __float2bfloat16_rn(__bfloat162float(xr[c]) + __bfloat162float(yr[c]));
    xr[c] = v;
    const float f = __bfloat162float(v);
    ss = fmaf(f, f, ss);
  }
  __shared__ float red[kNormThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float scale = rsqrtf(tot / (float)H + eps);
  for (int c = threadIdx.x; c < H; c += kNormThreads) hr[c] = __float2bfloat16_rn(__bfloat162float(xr[c]) * scale);
}

}  // namespace

cudaError_t launch_combine(const float* y_perm, const int32_t* inv, const float* topk_w, const float* y_sh,
                           int T, int H, int k, bf16* out, int* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(T, (H / 4 + kCombThreads - 1) / kCombThreads);
  return launch_pdl(combine_kernel, grid, dim3(kCombThreads), 0, s, y_perm, inv, topk_w, y_sh, T, H, k, out, err);
}

cudaError_t launch_rmsnorm_residual(bf16* x, const bf16* y, bf16* h, int T, int H, float eps, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(rmsnorm_residual_kernel, dim3(T), dim3(kNormThreads), 0, s, x, y, h, H, eps);
}

}  // namespace lsv
