// combine.cu -- gate-weighted combine of expert outputs, and the residual +
// RMSNorm update between stacked layers.
//
// combine:  out[t,:] = sum_{s<k} topk_w[t,s] * y_perm[inv[t*k+s],:] + y_shared[t,:]
// (y in fp32 for the moe_combine entry point, bf16 inside the fused layer)
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

// One CTA per token; thread c owns 8 consecutive columns and issues one 16-byte
// (bf16) or two 16-byte (fp32) loads per source row, all independent, so every
// thread has its k+1 rows in flight at once.
// Raw 16-byte pieces per source row: one for 8 bf16 columns, two for 8 fp32 columns.
template <typename YT>
struct Piece;
template <>
struct Piece<bf16> {
  uint4 a;
  __device__ __forceinline__ void load(const bf16* p) { a = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ void add_to(float (&acc)[8], float w) const {
    const uint32_t q[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = fmaf(w, __uint_as_float(q[i] << 16), acc[2 * i]);
      acc[2 * i + 1] = fmaf(w, __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
    }
  }
};
template <>
struct Piece<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void add_to(float (&acc)[8], float w) const {
    acc[0] = fmaf(w, a.x, acc[0]); acc[1] = fmaf(w, a.y, acc[1]); acc[2] = fmaf(w, a.z, acc[2]);
    acc[3] = fmaf(w, a.w, acc[3]); acc[4] = fmaf(w, b.x, acc[4]); acc[5] = fmaf(w, b.y, acc[5]);
    acc[6] = fmaf(w, b.z, acc[6]); acc[7] = fmaf(w, b.w, acc[7]);
  }
};

template <typename YT>
__global__ void __launch_bounds__(256) combine_kernel(const YT* __restrict__ y_perm, const int32_t* __restrict__ inv,
                                                      const float* __restrict__ topk_w, const YT* __restrict__ y_sh,
                                                      int T, int H, int k, int rows_y, bf16* __restrict__ out,
                                                      int* err, int32_t* __restrict__ clear, int n_clear) {
  const int t = blockIdx.x;
  __shared__ int rows[kMaxTopK];
  __shared__ float wts[kMaxTopK];
  pdl_wait();
  pdl_trigger();
  // the layer's counter block, for the next call (everything that used it has completed)
  if (clear && t == 0)
    for (int i = threadIdx.x; i < n_clear; i += blockDim.x) clear[i] = 0;
  if (threadIdx.x < k) {
    int r = inv[(size_t)t * k + threadIdx.x];
    if (r < 0 || r >= rows_y) {  // never read outside y_perm
      set_error(err, kErrDeviceIndex);
      r = -1;
    }
    rows[threadIdx.x] = r;
    wts[threadIdx.x] = topk_w[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
    Piece<YT> v[kMaxTopK + 1];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (s < k && rows[s] >= 0) v[s].load(y_perm + (size_t)rows[s] * H + c);
    if (y_sh) v[kMaxTopK].load(y_sh + (size_t)t * H + c);
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    // slot order, then the shared term
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (s < k && rows[s] >= 0) v[s].add_to(acc, wts[s]);
    if (y_sh) v[kMaxTopK].add_to(acc, 1.0f);
    uint4 pk;
    __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0], acc[1]), b1 = __floats2bfloat162_rn(acc[2], acc[3]);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[4], acc[5]), b3 = __floats2bfloat162_rn(acc[6], acc[7]);
    pk.x = *reinterpret_cast<uint32_t*>(&b0);
    pk.y = *reinterpret_cast<uint32_t*>(&b1);
    pk.z = *reinterpret_cast<uint32_t*>(&b2);
    pk.w = *reinterpret_cast<uint32_t*>(&b3);
    *reinterpret_cast<uint4*>(out + (size_t)t * H + c) = pk;
  }
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

cudaError_t launch_combine(const void* y_perm, const int32_t* inv, const float* topk_w, const void* y_sh,
                           bool y_bf16, int T, int H, int k, int rows_y, bf16* out, int* err, cudaStream_t s,
                           int32_t* clear, int n_clear) {
  if (T == 0) return cudaSuccess;
  int threads = ((H / 8 + 31) / 32) * 32;
  if (threads > 256) threads = 256;
  if (y_bf16)
    return launch_pdl(combine_kernel<bf16>, dim3(T), dim3(threads), 0, s, static_cast<const bf16*>(y_perm), inv,
                      topk_w, static_cast<const bf16*>(y_sh), T, H, k, rows_y, out, err, clear, n_clear);
  return launch_pdl(combine_kernel<float>, dim3(T), dim3(threads), 0, s, static_cast<const float*>(y_perm), inv,
                    topk_w, static_cast<const float*>(y_sh), T, H, k, rows_y, out, err, clear, n_clear);
}

cudaError_t launch_rmsnorm_residual(bf16* x, const bf16* y, bf16* h, int T, int H, float eps, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(rmsnorm_residual_kernel, dim3(T), dim3(kNormThreads), 0, s, x, y, h, H, eps);
}

}  // namespace lsv
