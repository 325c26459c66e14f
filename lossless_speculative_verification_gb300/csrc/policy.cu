// policy.cu -- choice of the number of drafts K from measured step costs.
//
// The pages decompose the speculative speedup as S = tau / c (evolve.pub
// review, Table 8): tau is the mean number of tokens one verify step commits
// and c the cost of a speculative step relative to a plain greedy step.  With
// conditional acceptances a_i = P(draft i accepted | drafts 1..i-1 accepted)
// the committed count of a step with K drafts is 1 + L, L the accepted prefix,
// so tau(K) = sum_{i=0..K} prod_{j<=i} a_j (the empty product is 1).  Under
// CUDA graphs the pages find K = 1 best (1.17x) although tau keeps growing with
// K (kg.zhiyong.dev, "Start with the result"): the choice follows the measured
// costs, which is what spec_k_policy computes.
//
// The acceptances come from what the verifier reports: accept_histogram_kernel
// counts the accepted lengths L of a batch into a device histogram, and
// spec_cond_accept_from_histogram turns counts into a_i = #(L >= i) / #(L >= i-1).
#include <math.h>

#include "internal.h"
#include "lsv.h"
#include "ptx.cuh"

namespace lsv {
namespace {

__global__ void accept_histogram_kernel(const int32_t* __restrict__ accept_len, int B, int K,
                                        unsigned long long* __restrict__ hist, int* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ unsigned int local[kMaxVerifyRows];
  for (int i = threadIdx.x; i <= K; i += blockDim.x) local[i] = 0;
  __syncthreads();
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
    const int l = accept_len[b];
    if (l < 0 || l > K) {
      set_error(err, kErrDeviceIndex);
      continue;
    }
    atomicAdd(&local[l], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i <= K; i += blockDim.x)
    if (local[i]) atomicAdd(&hist[i], (unsigned long long)local[i]);
}

}  // namespace

cudaError_t launch_accept_histogram(const int32_t* accept_len, int B, int K, int64_t* hist, int* err,
                                    cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const int threads = 256;
  int blocks = (B + threads - 1) / threads;
  if (blocks > 1024) blocks = 1024;
  return launch_pdl(accept_histogram_kernel, dim3(blocks), dim3(threads), 0, s, accept_len, B, K,
                    reinterpret_cast<unsigned long long*>(hist), err);
}

}  // namespace lsv

extern "C" {

lsv_status spec_cond_accept_from_histogram(const int64_t* hist, int32_t K, double* cond) {
  if (K < 0 || K + 1 > lsv::kMaxVerifyRows) return LSV_ERR_UNSUPPORTED;
  if (K == 0) return LSV_OK;
  if (!hist || !cond) return LSV_ERR_INVALID_ARG;
  // reached[i] = #(L >= i); a_i = reached[i] / reached[i-1]
  double reached = 0.0;
  double tail[lsv::kMaxVerifyRows + 1];
  for (int i = K; i >= 0; --i) {
    if (hist[i] < 0) return LSV_ERR_INVALID_ARG;
    reached += (double)hist[i];
    tail[i] = reached;
  }
  for (int i = 1; i <= K; ++i) cond[i - 1] = tail[i - 1] > 0.0 ? tail[i] / tail[i - 1] : 0.0;
  return LSV_OK;
}

lsv_status spec_k_policy(const double* cond_accept, int32_t kmax, const double* step_cost, int32_t* k_best,
                         double* tau_out, double* speedup_out) {
  if (kmax < 0 || kmax + 1 > lsv::kMaxVerifyRows) return LSV_ERR_UNSUPPORTED;
  if ((kmax > 0 && !cond_accept) || !step_cost || !k_best) return LSV_ERR_INVALID_ARG;
  for (int i = 0; i < kmax; ++i)
    if (!(cond_accept[i] >= 0.0 && cond_accept[i] <= 1.0)) return LSV_ERR_INVALID_ARG;
  for (int k = 0; k <= kmax; ++k)
    if (!(step_cost[k] > 0.0) || !isfinite(step_cost[k])) return LSV_ERR_INVALID_ARG;
  double tau = 1.0, reach = 1.0, best = -1.0;
  int kb = 0;
  for (int k = 0; k <= kmax; ++k) {
    if (k > 0) {
      reach *= cond_accept[k - 1];  // P(the first k drafts are all accepted)
      tau += reach;
    }
    const double s = tau * step_cost[0] / step_cost[k];
    if (tau_out) tau_out[k] = tau;
    if (speedup_out) speedup_out[k] = s;
    if (s > best) {  // strict: equal speedups keep the smaller K
      best = s;
      kb = k;
    }
  }
  *k_best = kb;
  return LSV_OK;
}

lsv_status spec_accept_histogram(const int32_t* accept_len, int32_t B, int32_t K, int64_t* hist,
                                 lsv_stream stream) {
  if (B < 0 || K < 0) return LSV_ERR_INVALID_ARG;
  if (K + 1 > lsv::kMaxVerifyRows) return LSV_ERR_UNSUPPORTED;
  if (B == 0) return LSV_OK;
  if (!accept_len || !hist) return LSV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(accept_len) & 3) || (reinterpret_cast<uintptr_t>(hist) & 7))
    return LSV_ERR_MISALIGNED;
  lsv::DeviceCtx* dc = nullptr;
  if (lsv::device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  return lsv::launch_accept_histogram(accept_len, B, K, hist, dc->err, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? LSV_OK
             : LSV_ERR_CUDA;
}

}  // extern "C"
