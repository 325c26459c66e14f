// prefetch.cu -- bulk L2 prefetch of expert weights.
//
// The weights do not depend on the routing, but the routing steps (router,
// permutation) are latency-bound and leave HBM idle.  Issuing bulk L2
// prefetches of the weights the grouped-expert kernel will read first lets
// that idle time stream useful bytes.  The kernel issues
// cp.async.bulk.prefetch.L2 requests (no completion to wait for) and exits;
// the data arrives in L2 while the following kernels run.
#include "internal.h"
#include "ptx.cuh"

namespace lsv {
namespace {

struct PrefetchPlan {
  const uint8_t* base[4];
  uint64_t bytes[4];
  int n;
  uint64_t budget;
};

constexpr uint64_t kPrefetchChunk = 32768;

__global__ void __launch_bounds__(128) l2_prefetch_kernel(const PrefetchPlan plan) {
  // the weights are never written by the preceding kernels: start at once, and
  // only wait for the predecessor at the end, so that this kernel's completion
  // still implies its predecessor's (the next kernel waits on this one)
  pdl_trigger();
  const uint64_t nth = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j * kPrefetchChunk < plan.budget; j += nth) {
    uint64_t off = j * kPrefetchChunk;
    int r = 0;
    while (r < plan.n && off >= plan.bytes[r]) {
      off -= plan.bytes[r];
      ++r;
    }
    if (r >= plan.n) break;
    uint64_t len = plan.bytes[r] - off;
    if (len > kPrefetchChunk) len = kPrefetchChunk;
    const uint64_t left = plan.budget - j * kPrefetchChunk;
    if (len > left) len = left;
    len &= ~uint64_t(15);
    if (len) prefetch_l2_bulk(plan.base[r] + off, (uint32_t)len);
  }
  pdl_wait();
}

}  // namespace

cudaError_t launch_weight_prefetch(const bf16* w_gate_up, const bf16* w_down, const bf16* ws_gate_up,
                                   const bf16* ws_down, int H, int E, int S, int I, uint64_t budget,
                                   const DeviceCtx& dc, cudaStream_t s) {
  PrefetchPlan plan = {};
  auto add = [&](const bf16* p, uint64_t bytes) {
    if (p && bytes) {
      plan.base[plan.n] = reinterpret_cast<const uint8_t*>(p);
      plan.bytes[plan.n] = bytes;
      ++plan.n;
    }
  };
  // the order in which the grouped-expert kernel deals its items
  add(S > 0 ? ws_gate_up : nullptr, (uint64_t)2 * S * I * H * 2);
  add(w_gate_up, (uint64_t)E * 2 * I * H * 2);
  add(S > 0 ? ws_down : nullptr, (uint64_t)H * S * I * 2);
  add(w_down, (uint64_t)E * H * I * 2);
  uint64_t total = 0;
  for (int r = 0; r < plan.n; ++r) total += plan.bytes[r];
  plan.budget = (budget < total ? budget : total) & ~uint64_t(15);
  if (plan.budget == 0) return cudaSuccess;
  return launch_pdl(l2_prefetch_kernel, dim3(dc.num_sms), dim3(128), 0, s, plan);
}

}  // namespace lsv
