// accept.cu -- vocabulary-wide greedy token and prefix acceptance.
//
// For every verified row (b, j) the greedy token g[b,j] is the smallest index
// attaining the row maximum.  accept_len[b] is the length of the longest
// prefix of drafts that equals g[b,0..]; the committed tokens are that prefix
// followed by g[b, accept_len] -- the correction at the first mismatch, or the
// bonus token when every draft matched.  This makes the committed text
// identical to greedy decoding (kg.zhiyong.dev, "Why FastMTP fits OCR
// particularly well"; evolve.pub review, Section 3.1 / Eq. 2).
//
// Phase 1 streams the logits once: each CTA owns a chunk of one row, streams it
// through a ring of shared-memory buffers filled by 1-D bulk copies (48 KB in
// flight per CTA from a single issuing thread, four CTAs per SM), scans it and writes the
// chunk's (max, first index).  Phase 2 (one CTA per sequence, one warp per
// row) reduces the chunk partials and applies the rule.
// No atomics decide anything, so the result is deterministic.
#include <limits.h>

#include <mutex>

#include "internal.h"
#include "lsv.h"
#include "ptx.cuh"

namespace lsv {
namespace {

constexpr int kAccThreads = 256;
#ifndef LSV_ACC_CTAS_PER_SM
#define LSV_ACC_CTAS_PER_SM 4
#endif
#ifndef LSV_ACC_PIECE
#define LSV_ACC_PIECE 16384
#endif
#ifndef LSV_ACC_RING
#define LSV_ACC_RING 3
#endif
constexpr int kAccCtasPerSm = LSV_ACC_CTAS_PER_SM;  // resident CTAs per SM the chunking plans for (one wave)
constexpr int kPiece = LSV_ACC_PIECE;                // bytes per bulk copy
constexpr int kRingSlots = LSV_ACC_RING;             // bulk copies in flight per CTA
constexpr int kMinChunk = 2048;       // elements
constexpr int kScanVec = 4;           // 16-byte vectors a thread holds per scan step

// (value desc, index asc) maximum
__device__ __forceinline__ void better(float v, int i, float& bv, int& bi) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__device__ __forceinline__ void scan8(const uint4& q, int base, float& bv, int& bi) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16);
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u);
    if (lo > bv) { bv = lo; bi = base + 2 * i; }      // increasing index: strict > keeps the first
    if (hi > bv) { bv = hi; bi = base + 2 * i + 1; }
  }
}

// Block-wide (max, first index) of the per-thread candidates, written by thread 0.
__device__ __forceinline__ void block_reduce_store(float bv, int bi, float* pv, int* pi, size_t at) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    better(ov, oi, bv, bi);
  }
  __shared__ float sv[kAccThreads / 32];
  __shared__ int si[kAccThreads / 32];
  if ((threadIdx.x & 31) == 0) {
    sv[threadIdx.x >> 5] = bv;
    si[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kAccThreads / 32; ++w) better(sv[w], si[w], bv, bi);
    pv[at] = bv;
    pi[at] = bi;
  }
}

// Rows whose start is not 16-byte aligned (V not a multiple of 8): 2-byte loads.
__global__ void __launch_bounds__(kAccThreads) argmax_partial_scalar_kernel(const bf16* __restrict__ logits, int V,
                                                                            int chunk, int nchunk,
                                                                            float* __restrict__ pv,
                                                                            int* __restrict__ pi) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, c = blockIdx.y;
  const bf16* row = logits + (size_t)r * V;
  const int begin = c * chunk;
  const int end = min(V, begin + chunk);
  float bv = -INFINITY;
  int bi = begin;  // a chunk of -inf gives its first index, so a row of -inf gives 0
  for (int e = begin + threadIdx.x; e < end; e += kAccThreads) {
    const float f = __bfloat162float(row[e]);
    if (f > bv) { bv = f; bi = e; }
  }
  block_reduce_store(bv, bi, pv, pi, (size_t)r * nchunk + c);
}

// 16-byte aligned rows: the chunk streams through a ring of kRingSlots shared
// buffers filled by 1-D bulk copies (one thread issues them; kRingSlots x 16 KB
// in flight), and the 256 threads scan each buffer as it lands.
__global__ void __launch_bounds__(kAccThreads) argmax_partial_bulk_kernel(const bf16* __restrict__ logits, int V,
                                                                          int chunk, int nchunk,
                                                                          float* __restrict__ pv,
                                                                          int* __restrict__ pi, int* err,
                                                                          uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __shared__ uint64_t bar[kRingSlots];
  const int r = blockIdx.x, c = blockIdx.y;
  const int begin = c * chunk;                 // a multiple of 8 elements
  const int end = min(V, begin + chunk);
  const uint8_t* src = reinterpret_cast<const uint8_t*>(logits + (size_t)r * V + begin);
  const int bytes = (end - begin) * 2;         // a multiple of 16
  const int npieces = (bytes + kPiece - 1) / kPiece;
  if (threadIdx.x == 0) {
    for (int q = 0; q < kRingSlots; ++q) mbar_init(&bar[q], 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int q = 0; q < kRingSlots && q < npieces; ++q) {
      const int n = min(kPiece, bytes - q * kPiece);
      mbar_arrive_expect_tx(&bar[q], n);
      bulk_load(ring + q * kPiece, src + (size_t)q * kPiece, n, &bar[q]);
    }
  }
  float bv = -INFINITY;
  int bi = begin;  // a chunk of -inf gives its first index, so a row of -inf gives 0
  bool ok = true;
  int q_fail = npieces;
  for (int q = 0; q < npieces; ++q) {
    const int slot = q % kRingSlots;
    if (!mbar_wait(&bar[slot], (q / kRingSlots) & 1, wait_ns)) {
      set_error(err, kErrTimeout);
      ok = false;
    }
    if (__syncthreads_or(!ok)) {
      ok = false;
      q_fail = q;
      break;
    }
    const int n = min(kPiece, bytes - q * kPiece);
    const uint4* v = reinterpret_cast<const uint4*>(ring + slot * kPiece);
    const int e0 = begin + q * (kPiece / 2);
    for (int j0 = threadIdx.x; j0 < n / 16; j0 += kScanVec * kAccThreads) {
      // this thread's vectors of the piece, in increasing index order
      uint4 w[kScanVec];
      __nv_bfloat162 m2 = __float2bfloat162_rn(-INFINITY);
#pragma unroll
      for (int u = 0; u < kScanVec; ++u) {
        const int j = j0 + u * kAccThreads;
        w[u] = j < n / 16 ? v[j] : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);  // -inf pairs
        m2 = __hmax2(m2, *reinterpret_cast<const __nv_bfloat162*>(&w[u].x));
        m2 = __hmax2(m2, *reinterpret_cast<const __nv_bfloat162*>(&w[u].y));
        m2 = __hmax2(m2, *reinterpret_cast<const __nv_bfloat162*>(&w[u].z));
        m2 = __hmax2(m2, *reinterpret_cast<const __nv_bfloat162*>(&w[u].w));
      }
      const float m = fmaxf(__low2float(m2), __high2float(m2));
      if (m > bv) {
        // a new maximum (rare after the first pieces): locate its first occurrence among the
        // values still in registers; equal values seen earlier keep their lower index
        for (int u = 0; u < kScanVec; ++u) {
          const int j = j0 + u * kAccThreads;
          if (j < n / 16) scan8(w[u], e0 + 8 * j, bv, bi);
        }
      }
    }
    __syncthreads();  // the slot is free again
    if (threadIdx.x == 0 && q + kRingSlots < npieces) {
      const int qn = q + kRingSlots;
      const int nn = min(kPiece, bytes - qn * kPiece);
      mbar_arrive_expect_tx(&bar[slot], nn);
      bulk_load(ring + slot * kPiece, src + (size_t)qn * kPiece, nn, &bar[slot]);
    }
  }
  if (!ok && threadIdx.x == 0) {
    // a wait gave up at piece q_fail: let the copies still in flight into this CTA's ring land
    // (again with a limit) before the CTA exits
    for (int q = q_fail; q < npieces && q < q_fail + kRingSlots; ++q)
      mbar_wait(&bar[q % kRingSlots], (q / kRingSlots) & 1, wait_ns);
  }
  block_reduce_store(bv, bi, pv, pi, (size_t)r * nchunk + c);
}

// One CTA per sequence, one warp per verified row: each warp reduces its row's
// chunk partials; then one thread applies the acceptance rule.  argmax rows of
// sequence b start at b * argmax_ld; accept_len and committed may be null.
constexpr int kFinWarps = 32;

__global__ void __launch_bounds__(kFinWarps * 32) accept_finalize_kernel(
    const float* __restrict__ pv, const int* __restrict__ pi, int nchunk, const int32_t* __restrict__ drafts,
    int B, int K, int32_t* __restrict__ argmax, int argmax_ld, int32_t* __restrict__ accept_len,
    int32_t* __restrict__ committed) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  __shared__ int g[kMaxVerifyRows];
  for (int j = threadIdx.x >> 5; j <= K; j += blockDim.x >> 5) {
    const size_t r = (size_t)b * (K + 1) + j;
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int c = lane; c < nchunk; c += 32) better(pv[r * nchunk + c], pi[r * nchunk + c], bv, bi);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      better(ov, oi, bv, bi);
    }
    if (lane == 0) {
      g[j] = bi;
      if (argmax) argmax[(size_t)b * argmax_ld + j] = bi;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && accept_len && committed) {
    int L = 0;
    while (L < K && drafts[(size_t)b * K + L] == g[L]) ++L;
    accept_len[b] = L;
    int32_t* cm = committed + (size_t)b * (K + 1);
    for (int i = 0; i < L; ++i) cm[i] = drafts[(size_t)b * K + i];
    cm[L] = g[L];
    for (int i = L + 1; i <= K; ++i) cm[i] = -1;
  }
}

// Chunks per row and chunk length: one wave of about kAccCtasPerSm CTAs per SM
// in total, at least kMinChunk elements per chunk, chunk lengths a multiple of
// 8 elements (so that every chunk of an aligned row starts on 16 bytes).
void chunk_plan(int R, int V, int num_sms, int* chunk, int* nchunk) {
  const long long target = (long long)num_sms * kAccCtasPerSm;
  long long n = target / (R > 0 ? R : 1);
  const long long max_chunks = ((long long)V + kMinChunk - 1) / kMinChunk;
  if (n > max_chunks) n = max_chunks;
  if (n < 1) n = 1;
  long long per = ((long long)V + n - 1) / n;
  per = (per + 7) / 8 * 8;
  *chunk = (int)per;
  *nchunk = (int)(((long long)V + per - 1) / per);
}

}  // namespace

size_t accept_ws_bytes(int B, int K, int V, int num_sms) {
  const int R = B * (K + 1);
  if (R == 0) return 256;
  int chunk, nchunk;
  chunk_plan(R, V, num_sms, &chunk, &nchunk);
  const size_t one = ((size_t)R * nchunk * 4 + 255) / 256 * 256;
  return 2 * one;
}

cudaError_t launch_accept(const bf16* logits, const int32_t* drafts, int B, int K, int V, int32_t* argmax,
                          int32_t* accept_len, int32_t* committed, void* ws, const DeviceCtx& dc,
                          cudaStream_t s) {
  const int R = B * (K + 1);
  if (R == 0) return cudaSuccess;
  int chunk, nchunk;
  chunk_plan(R, V, dc.num_sms, &chunk, &nchunk);
  const size_t one = ((size_t)R * nchunk * 4 + 255) / 256 * 256;
  float* pv = reinterpret_cast<float*>(ws);
  int* pi = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ws) + one);
  const bool aligned = (V % 8 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  cudaError_t e;
  if (aligned) {
    constexpr int kSmem = kRingSlots * kPiece + 128;
    e = ensure_smem_attr(reinterpret_cast<const void*>(argmax_partial_bulk_kernel), kSmem, dc.device);
    if (e != cudaSuccess) return e;
    e = launch_pdl(argmax_partial_bulk_kernel, dim3(R, nchunk), dim3(kAccThreads), kSmem, s, logits, V, chunk, nchunk,
                   pv, pi, dc.err, wait_limit_ns());
  } else {
    e = launch_pdl(argmax_partial_scalar_kernel, dim3(R, nchunk), dim3(kAccThreads), 0, s, logits, V, chunk, nchunk,
                   pv, pi);
  }
  if (e != cudaSuccess) return e;
  return launch_accept_finalize(pv, pi, nchunk, drafts, B, K, argmax, accept_len, committed, s);
}

cudaError_t launch_accept_finalize(const float* pv, const int* pi, int nchunk, const int32_t* drafts, int B, int K,
                                   int32_t* argmax, int32_t* accept_len, int32_t* committed, cudaStream_t s,
                                   int argmax_ld) {
  if (B == 0) return cudaSuccess;
  return launch_pdl(accept_finalize_kernel, dim3(B), dim3(32 * min(K + 1, kFinWarps)), 0, s, pv, pi, nchunk, drafts,
                    B, K, argmax, argmax_ld > 0 ? argmax_ld : K + 1, accept_len, committed);
}

}  // namespace lsv

// ----------------------------------------------------------------------------- no-allocation variant
// Some callers cannot allocate device memory at the point where they verify
// drafts: a host that runs the library as a plugin and passes only the
// tensors of the call, or a decode loop whose memory is fixed before it
// starts.  For them the chunk partials of the argmax live in this fixed array
// instead of a caller workspace.  It exists once per device that loads the
// library and stays allocated until the process exits.
namespace lsv {
namespace {
constexpr int kNoAllocPartials = 16384;  // (max, index) pairs: 128 KiB in total
static __device__ __align__(256) unsigned char g_noalloc_scratch[2 * kNoAllocPartials * 4];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// Device address of the scratch array for the current device.  The first call
// on a device resolves it (host code may not use the array's name as an
// address); later calls reuse the cached value.
cudaError_t noalloc_scratch(int device, void** out) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[device] = p;
  }
  *out = g_noalloc_addr[device];
  return cudaSuccess;
}
}  // namespace
}  // namespace lsv

extern "C" lsv_status spec_verify_accept_noalloc(const void* logits, const int32_t* drafts, int32_t B, int32_t K,
                                                 int32_t V, int32_t* argmax_opt, int32_t* accept_len,
                                                 int32_t* committed, lsv_stream stream) {
  using namespace lsv;
  if (B < 0 || K < 0 || V <= 0) return LSV_ERR_INVALID_ARG;
  if (K + 1 > kMaxVerifyRows || (long long)B * (K + 1) >= (1ll << 31)) return LSV_ERR_UNSUPPORTED;
  if (B == 0) return LSV_OK;
  if (!logits || !accept_len || !committed || (K > 0 && !drafts)) return LSV_ERR_INVALID_ARG;
  const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!a16(logits) || !a16(drafts) || !a16(argmax_opt) || !a16(accept_len) || !a16(committed))
    return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  // problems whose partials do not fit the fixed array are refused, never truncated
  if (accept_ws_bytes(B, K, V, dc->num_sms) > sizeof(g_noalloc_scratch)) return LSV_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (noalloc_scratch(dc->device, &scratch) != cudaSuccess) return LSV_ERR_CUDA;
  return launch_accept(static_cast<const bf16*>(logits), drafts, B, K, V, argmax_opt, accept_len, committed, scratch,
                       *dc, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LSV_OK
             : LSV_ERR_CUDA;
}
