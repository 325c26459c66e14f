// cache.cu -- the two data movements of a verify pass around its kernels: the
// embedding rows of the verified tokens, and the append of the verified
// positions' keys and values to each sequence's cache (the verify pass sees
// every sequence's K+1 positions at once and appends them before attending;
// kg.zhiyong.dev, "The speed comes from three layers working together": the
// main decoder verifies the drafts in one pass).
#include "internal.h"
#include "lsv.h"
#include "ptx.cuh"

namespace lsv {
namespace {

constexpr int kCpThreads = 128;

// out[i, :] = table[idx[i], :] (rows of `row16` 16-byte vectors); an index outside [0, n_table)
// writes a zero row and raises LSV_ERR_DEVICE_INDEX.
__global__ void __launch_bounds__(kCpThreads) gather_rows_kernel(const uint4* __restrict__ table,
                                                                 const int32_t* __restrict__ idx, int n_table,
                                                                 int row16, uint4* __restrict__ out, int* err) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const int r = __ldcg(idx + i);
  uint4* o = out + (size_t)i * row16;
  if (r < 0 || r >= n_table) {
    if (threadIdx.x == 0) set_error(err, kErrDeviceIndex);
    for (int c = threadIdx.x; c < row16; c += kCpThreads) o[c] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* s = table + (size_t)r * row16;
  for (int c = threadIdx.x; c < row16; c += kCpThreads) o[c] = s[c];
}

// Row j of sequence b's Q new rows goes to cache position ctx_len[b] - Q + j, for keys and values.
// A length outside [Q, L] raises LSV_ERR_DEVICE_INDEX and writes nothing for that sequence.
__global__ void __launch_bounds__(kCpThreads) cache_append_kernel(const uint4* __restrict__ k_new,
                                                                  const uint4* __restrict__ v_new,
                                                                  uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                                  const int32_t* __restrict__ ctx_len, int Q, int L,
                                                                  int row16, int* err) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x / Q, j = blockIdx.x - (blockIdx.x / Q) * Q;
  const int n = __ldcg(ctx_len + b);
  if (n < Q || n > L) {
    if (threadIdx.x == 0 && j == 0) set_error(err, kErrDeviceIndex);
    return;
  }
  const size_t src = (size_t)blockIdx.x * row16;
  const size_t dst = ((size_t)b * L + (n - Q + j)) * row16;
  for (int c = threadIdx.x; c < row16; c += kCpThreads) {
    k_cache[dst + c] = k_new[src + c];
    v_cache[dst + c] = v_new[src + c];
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace lsv

using namespace lsv;

extern "C" {

lsv_status lsv_gather_rows(const void* table, const int32_t* idx, int32_t n, int32_t n_table, int32_t row_elems,
                           void* out, lsv_stream stream) {
  if (n < 0 || n_table <= 0 || row_elems <= 0) return LSV_ERR_INVALID_ARG;
  if (row_elems % 8 || n > (1 << 30)) return LSV_ERR_UNSUPPORTED;
  if (n == 0) return LSV_OK;
  if (!table || !idx || !out) return LSV_ERR_INVALID_ARG;
  if (!al16(table) || !al16(idx) || !al16(out)) return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  return launch_pdl(gather_rows_kernel, dim3(n), dim3(kCpThreads), 0, reinterpret_cast<cudaStream_t>(stream),
                    static_cast<const uint4*>(table), idx, n_table, row_elems / 8, static_cast<uint4*>(out),
                    dc->err) == cudaSuccess
             ? LSV_OK
             : LSV_ERR_CUDA;
}

lsv_status spec_cache_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int32_t* ctx_len, int32_t B, int32_t Q, int32_t L, int32_t row_elems,
                             lsv_stream stream) {
  if (B < 0 || Q <= 0 || L <= 0 || row_elems <= 0) return LSV_ERR_INVALID_ARG;
  if (row_elems % 8 || Q > L || (long long)B * Q > (1ll << 30)) return LSV_ERR_UNSUPPORTED;
  if (B == 0) return LSV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !ctx_len) return LSV_ERR_INVALID_ARG;
  if (!al16(k_new) || !al16(v_new) || !al16(k_cache) || !al16(v_cache) || !al16(ctx_len)) return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  return launch_pdl(cache_append_kernel, dim3(B * Q), dim3(kCpThreads), 0, reinterpret_cast<cudaStream_t>(stream),
                    static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), static_cast<uint4*>(k_cache),
                    static_cast<uint4*>(v_cache), ctx_len, Q, L, row_elems / 8, dc->err) == cudaSuccess
             ? LSV_OK
             : LSV_ERR_CUDA;
}

}  // extern "C"
