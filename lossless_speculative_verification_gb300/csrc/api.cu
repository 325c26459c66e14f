// api.cu -- the extern "C" entry points declared in include/lsv.h: argument
// validation (before any launch), workspace layout, the per-device error word
// and the launch sequence of each call.
#include <stdio.h>
#include <string.h>

#include <map>
#include <mutex>

#include "internal.h"
#include "lsv.h"
#include "ptx.cuh"

namespace lsv {

// The device error word: one int per device (a module-scope __device__ variable
// exists once per device the library is used on).
__device__ int g_device_error = 0;

namespace {
std::mutex g_mu;
DeviceCtx g_ctx[64];
uint64_t g_wait_ns = 2000000000ull;

__global__ void wait_selftest_kernel(int* err, const int* never_set, uint64_t limit_ns) {
  if (threadIdx.x == 0) {
    if (!wait_counter_geq(never_set, 1, limit_ns)) set_error(err, kErrTimeout);
  }
}
__device__ int g_never_set = 0;

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
}  // namespace

uint64_t wait_limit_ns() { return g_wait_ns; }

cudaError_t device_ctx(DeviceCtx** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceCtx& c = g_ctx[dev];
  if (c.device != dev) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int l2 = 0;
    e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return e;
    c.l2_bytes = l2;
    c.num_sms = sms;
    c.err = static_cast<int*>(p);
    c.device = dev;
  }
  *out = &c;
  return cudaSuccess;
}

cudaError_t ensure_smem_attr(const void* kernel, int bytes, int device) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;
  std::lock_guard<std::mutex> lk(mu);
  int& have = done[std::make_pair(kernel, device)];
  if (have >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

cudaError_t launch_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t s) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_never_set);
  if (e != cudaSuccess) return e;
  wait_selftest_kernel<<<1, 32, 0, s>>>(err, static_cast<const int*>(p), limit_ns);
  return cudaGetLastError();
}

WsLayout ws_layout(int T, int H, int E, int k, int S, int I) {
  WsLayout L;
  const size_t n = (size_t)T * k;
  const int G = E + (S > 0 ? 1 : 0);
  L.nblk = n == 0 ? 1 : (int)((n + kPermChunk - 1) / kPermChunk);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.counters = take(kCounterBytes);
  L.topk_idx = take(n * 4);
  L.topk_w = take(n * 4);
  L.counts = take((size_t)E * 4);
  L.offsets = take((size_t)(E + 1) * 4);
  L.perm = take(n * 4);
  L.inv = take(n * 4);
  L.blk_counts = take((size_t)L.nblk * E * 4);
  L.table = take((size_t)table_ints(G) * 4);
  const size_t rows = routed_rows(T, k, E);
  L.xperm = take(rows * H * 2);
  L.act = take(rows * I * 2);
  L.act_sh = take((size_t)T * S * I * 2);
  L.y_perm = take(rows * H * 4);
  L.y_sh = take((size_t)T * H * 4);
  L.total = align256(o);
  return L;
}

}  // namespace lsv

using namespace lsv;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

lsv_status check_shape(const lsv_moe_shape* s) {
  if (!s) return LSV_ERR_INVALID_ARG;
  if (s->T < 0 || s->H <= 0 || s->E <= 0 || s->k < 0 || s->S < 0 || s->I <= 0) return LSV_ERR_INVALID_ARG;
  if (s->k > s->E) return LSV_ERR_INVALID_ARG;
  if (s->H % 64 || s->I % 64 || s->H > kMaxHidden || s->E > kMaxExperts || s->k > kMaxTopK ||
      s->S > kMaxShared || (long long)s->S * s->I > kMaxHidden)
    return LSV_ERR_UNSUPPORTED;
  if ((long long)s->T * s->k >= (1ll << 30) || (long long)s->T * s->H >= (1ll << 40)) return LSV_ERR_UNSUPPORTED;
  return LSV_OK;
}

lsv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LSV_OK : LSV_ERR_CUDA; }

// L2 prefetch budget of moe_verify_layer, as a percentage of L2.  Measured on
// GB300 at the decode shape (T=128): 0 % gives a 101.5 us layer, 30/60/80 %
// all give 117.9 us, because the router waits for the prefetch grid to
// complete before it starts.  So the layer does not prefetch by default;
// moe_prefetch_weights stays available for callers that can issue it earlier
// (for instance before the attention block of the same decoder layer).
#ifndef LSV_PREFETCH_L2_PCT
#define LSV_PREFETCH_L2_PCT 0
#endif
uint64_t default_prefetch_bytes(const DeviceCtx& dc, int T, int E, int k, int S, int I, int H) {
  const uint64_t shared = (uint64_t)3 * S * I * H * 2;
  const uint64_t cap = (uint64_t)dc.l2_bytes * LSV_PREFETCH_L2_PCT / 100;
  if ((long long)T * k >= 2ll * E) return cap;
  return shared < cap ? shared : cap;
}

}  // namespace

extern "C" {

const char* lsv_status_string(lsv_status s) {
  switch (s) {
    case LSV_OK: return "ok";
    case LSV_ERR_INVALID_ARG: return "invalid argument";
    case LSV_ERR_UNSUPPORTED: return "unsupported shape";
    case LSV_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case LSV_ERR_WORKSPACE: return "workspace missing or too small";
    case LSV_ERR_CUDA: return "CUDA call failed";
    case LSV_ERR_TIMEOUT: return "device wait timed out";
    case LSV_ERR_DEVICE_INDEX: return "device index out of range";
  }
  return "unknown status";
}

int32_t lsv_version(void) { return 100; }

lsv_status lsv_set_wait_limit_ns(uint64_t ns) {
  if (ns == 0) return LSV_ERR_INVALID_ARG;
  g_wait_ns = ns;
  return LSV_OK;
}

size_t lsv_workspace_size(const lsv_moe_shape* s) {
  if (check_shape(s) != LSV_OK) return 0;
  return ws_layout(s->T, s->H, s->E, s->k, s->S, s->I).total;
}

lsv_status lsv_get_device_error(int32_t* code_out, lsv_stream stream) {
  if (!code_out) return LSV_ERR_INVALID_ARG;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, dc->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return LSV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LSV_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyAsync(dc->err, &zero, sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess) return LSV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return LSV_ERR_CUDA;
  }
  *code_out = v;
  return LSV_OK;
}

lsv_status lsv_selftest_wait_timeout(uint64_t limit_ns, lsv_stream stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return LSV_ERR_INVALID_ARG;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  return from_cuda(launch_wait_selftest(dc->err, limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

lsv_status moe_prefetch_weights(const lsv_moe_weights* wt, const lsv_moe_shape* shape, size_t max_bytes,
                                lsv_stream stream) {
  lsv_status st = check_shape(shape);
  if (st != LSV_OK) return st;
  if (!wt) return LSV_ERR_INVALID_ARG;
  if (max_bytes == 0) return LSV_OK;
  if (!aligned16(wt->w_gate_up) || !aligned16(wt->w_down) || !aligned16(wt->ws_gate_up) || !aligned16(wt->ws_down))
    return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  return from_cuda(launch_weight_prefetch(static_cast<const bf16*>(wt->w_gate_up), static_cast<const bf16*>(wt->w_down),
                                          static_cast<const bf16*>(wt->ws_gate_up), static_cast<const bf16*>(wt->ws_down),
                                          shape->H, shape->E, shape->S, shape->I, max_bytes, *dc,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

lsv_status moe_route(const void* x, const void* w_router, const lsv_moe_shape* shape, int32_t* topk_idx,
                     float* topk_w, float* logits_opt, lsv_stream stream) {
  lsv_status st = check_shape(shape);
  if (st != LSV_OK) return st;
  if (shape->T == 0) return LSV_OK;
  if (!x || !w_router || (shape->k > 0 && (!topk_idx || !topk_w))) return LSV_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(topk_idx) || !aligned16(topk_w) ||
      !aligned16(logits_opt))
    return LSV_ERR_MISALIGNED;
  return from_cuda(launch_route(static_cast<const bf16*>(x), static_cast<const bf16*>(w_router), shape->T,
                                shape->H, shape->E, shape->k, topk_idx, topk_w, logits_opt,
                                reinterpret_cast<cudaStream_t>(stream)));
}

lsv_status moe_permute(const int32_t* topk_idx, const lsv_moe_shape* shape, int32_t* counts, int32_t* offsets,
                       int32_t* perm_src, int32_t* inv, void* ws, size_t ws_bytes, lsv_stream stream) {
  lsv_status st = check_shape(shape);
  if (st != LSV_OK) return st;
  if (!counts || !offsets) return LSV_ERR_INVALID_ARG;
  const size_t n = (size_t)shape->T * shape->k;
  if (n > 0 && (!topk_idx || !perm_src || !inv)) return LSV_ERR_INVALID_ARG;
  if (!aligned16(topk_idx) || !aligned16(counts) || !aligned16(offsets) || !aligned16(perm_src) || !aligned16(inv))
    return LSV_ERR_MISALIGNED;
  const WsLayout L = ws_layout(shape->T, shape->H, shape->E, shape->k, shape->S, shape->I);
  if (!ws || ws_bytes < L.total) return LSV_ERR_WORKSPACE;
  if (!aligned16(ws)) return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  return from_cuda(launch_permute(topk_idx, shape->T, shape->k, shape->E, counts, offsets, perm_src, inv,
                                  reinterpret_cast<int32_t*>(w + L.blk_counts), L.nblk, dc->err,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

lsv_status moe_grouped_ffn(const void* x, const int32_t* perm_src, const int32_t* offsets, const int32_t* counts,
                           const lsv_moe_weights* wt, const lsv_moe_shape* shape, float* y_perm, float* y_shared,
                           void* ws, size_t ws_bytes, lsv_stream stream) {
  lsv_status st = check_shape(shape);
  if (st != LSV_OK) return st;
  if (!wt || !offsets || !counts) return LSV_ERR_INVALID_ARG;
  if (shape->T == 0) return LSV_OK;
  const size_t n = (size_t)shape->T * shape->k;
  if (!x) return LSV_ERR_INVALID_ARG;
  if (n > 0 && (!perm_src || !y_perm || !wt->w_gate_up || !wt->w_down)) return LSV_ERR_INVALID_ARG;
  if (shape->S > 0 && (!y_shared || !wt->ws_gate_up || !wt->ws_down)) return LSV_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(perm_src) || !aligned16(offsets) || !aligned16(counts) || !aligned16(y_perm) ||
      !aligned16(y_shared) || !aligned16(wt->w_gate_up) || !aligned16(wt->w_down) || !aligned16(wt->ws_gate_up) ||
      !aligned16(wt->ws_down))
    return LSV_ERR_MISALIGNED;
  const WsLayout L = ws_layout(shape->T, shape->H, shape->E, shape->k, shape->S, shape->I);
  if (!ws || ws_bytes < L.total) return LSV_ERR_WORKSPACE;
  if (!aligned16(ws)) return LSV_ERR_MISALIGNED;
  if (n == 0 && shape->S == 0) return LSV_OK;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  // with no routed pairs the routed weights are never read; any valid pointer serves their tensor maps
  const void* wgu = wt->w_gate_up ? wt->w_gate_up : wt->ws_gate_up;
  const void* wd = wt->w_down ? wt->w_down : wt->ws_down;
  return from_cuda(launch_ffn(static_cast<const bf16*>(x), perm_src, offsets, nullptr, 0,
                              static_cast<const bf16*>(wgu), static_cast<const bf16*>(wd),
                              static_cast<const bf16*>(wt->ws_gate_up),
                              static_cast<const bf16*>(wt->ws_down), shape->T, shape->H, shape->E, shape->k,
                              shape->S, shape->I, y_perm, y_shared, /*y_bf16=*/false, static_cast<uint8_t*>(ws), L,
                              *dc, reinterpret_cast<cudaStream_t>(stream)));
}

lsv_status moe_combine(const float* y_perm, const int32_t* inv, const float* topk_w, const float* y_shared,
                       const lsv_moe_shape* shape, void* out, lsv_stream stream) {
  lsv_status st = check_shape(shape);
  if (st != LSV_OK) return st;
  if (shape->T == 0) return LSV_OK;
  if (!out || (shape->k > 0 && (!y_perm || !inv || !topk_w)) || (shape->S > 0 && !y_shared))
    return LSV_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(inv) || !aligned16(topk_w) || !aligned16(y_shared) || !aligned16(out))
    return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  return from_cuda(launch_combine(y_perm, inv, topk_w, shape->S > 0 ? y_shared : nullptr, /*y_bf16=*/false,
                                  shape->T, shape->H, shape->k, shape->T * shape->k, static_cast<bf16*>(out), dc->err,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

lsv_status moe_verify_layer(const void* x, const lsv_moe_weights* wt, const lsv_moe_shape* shape, void* out,
                            int32_t* topk_idx_opt, int32_t* counts_opt, void* ws, size_t ws_bytes,
                            lsv_stream stream) {
  lsv_status st = check_shape(shape);
  if (st != LSV_OK) return st;
  if (!wt) return LSV_ERR_INVALID_ARG;
  const int T = shape->T, H = shape->H, E = shape->E, k = shape->k, S = shape->S, I = shape->I;
  if (T == 0) return LSV_OK;
  if (!x || !out || !wt->w_router || !wt->w_gate_up || !wt->w_down) return LSV_ERR_INVALID_ARG;
  if (S > 0 && (!wt->ws_gate_up || !wt->ws_down)) return LSV_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(wt->w_router) || !aligned16(wt->w_gate_up) ||
      !aligned16(wt->w_down) || !aligned16(wt->ws_gate_up) || !aligned16(wt->ws_down) || !aligned16(topk_idx_opt) ||
      !aligned16(counts_opt))
    return LSV_ERR_MISALIGNED;
  const WsLayout L = ws_layout(T, H, E, k, S, I);
  if (!ws || ws_bytes < L.total) return LSV_ERR_WORKSPACE;
  if (!aligned16(ws)) return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* idx = topk_idx_opt ? topk_idx_opt : reinterpret_cast<int32_t*>(w + L.topk_idx);
  float* tw = reinterpret_cast<float*>(w + L.topk_w);
  int32_t* counts = counts_opt ? counts_opt : reinterpret_cast<int32_t*>(w + L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(w + L.perm);
  int32_t* inv = reinterpret_cast<int32_t*>(w + L.inv);
  // inside the layer the expert outputs stay in bf16 (half the bytes between the experts and the combine)
  bf16* y_perm = reinterpret_cast<bf16*>(w + L.y_perm);
  bf16* y_sh = reinterpret_cast<bf16*>(w + L.y_sh);
  const bf16* wgu = static_cast<const bf16*>(wt->w_gate_up);
  const bf16* wdn = static_cast<const bf16*>(wt->w_down);
  const bf16* wsgu = static_cast<const bf16*>(wt->ws_gate_up);
  const bf16* wsdn = static_cast<const bf16*>(wt->ws_down);
  // The counter block is zero on entry (the previous call's expert kernel cleared it), so the
  // expert kernel can begin its routing-independent shared-expert items while the router runs.
  int32_t* table = reinterpret_cast<int32_t*>(w + L.table);
  int32_t* cnt = reinterpret_cast<int32_t*>(w + L.counters);
  cudaError_t e = cudaSuccess;
  const uint64_t pf = default_prefetch_bytes(*dc, T, E, k, S, I, H);
  if (e == cudaSuccess && pf) e = launch_weight_prefetch(wgu, wdn, wsgu, wsdn, H, E, S, I, pf, *dc, s);
  const int BN = ffn_token_tile(T, k, E);
  if (use_slots(T)) {
    // the router places the rows, the expert kernel builds its item table: no permutation launch
    RouteSlots sl;
    sl.xperm = reinterpret_cast<bf16*>(w + L.xperm);
    sl.inv = inv;
    sl.slots = cnt + kCntSlots;
    if (e == cudaSuccess)
      e = launch_route(static_cast<const bf16*>(x), static_cast<const bf16*>(wt->w_router), T, H, E, k, idx, tw,
                       nullptr, s, &sl);
    if (e == cudaSuccess)
      e = launch_ffn(static_cast<const bf16*>(x), nullptr, nullptr, cnt + kCntSlots, T, wgu, wdn, wsgu, wsdn,
                     T, H, E, k, S, I, y_perm, y_sh, /*y_bf16=*/true, w, L, *dc, s, /*with_prep=*/false,
                     /*early=*/true, counts_opt);
  } else {
    if (e == cudaSuccess)
      e = launch_route(static_cast<const bf16*>(x), static_cast<const bf16*>(wt->w_router), T, H, E, k, idx, tw,
                       nullptr, s);
    const bool fused = (long long)T * k <= kPermFusedMax;  // permutation, gather and plan in one launch
    if (e == cudaSuccess) {
      if (fused)
        e = launch_permute_gather(idx, T, k, E, H, S, I, BN, static_cast<const bf16*>(x), counts, offsets, perm,
                                  inv, reinterpret_cast<bf16*>(w + L.xperm), table, dc->err, s);
      else
        e = launch_permute(idx, T, k, E, counts, offsets, perm, inv, reinterpret_cast<int32_t*>(w + L.blk_counts),
                           L.nblk, dc->err, s);
    }
    if (e == cudaSuccess)
      e = launch_ffn(static_cast<const bf16*>(x), perm, offsets, nullptr, 0, wgu, wdn, wsgu, wsdn, T, H, E, k, S, I,
                     y_perm, y_sh, /*y_bf16=*/true, w, L, *dc, s, /*with_prep=*/!fused, /*early=*/true);
  }
  if (e == cudaSuccess)
    e = launch_combine(y_perm, inv, tw, S > 0 ? y_sh : nullptr, /*y_bf16=*/true, T, H, k,
                       use_slots(T) ? E * T : T * k, static_cast<bf16*>(out), dc->err, s, cnt,
                       (int)(kCounterBytes / 4));
  return from_cuda(e);
}

size_t spec_verify_attention_workspace_size(int32_t B, int32_t Q, int32_t L, int32_t nh, int32_t d) {
  if (B < 0 || Q < 1 || Q > kMaxAttnQ || L < Q || L > kAttnMaxL || nh < 1 || (d != 64 && d != 128)) return 0;
  if ((long long)B * L * nh * d >= (1ll << 40) || (long long)B * nh > kAttnMaxPairs || nh > 65535 || B > 65535)
    return 0;
  return attention_ws_bytes(B, Q, L, nh, d);
}

lsv_status spec_verify_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* ctx_len,
                                 int32_t B, int32_t Q, int32_t L, int32_t nh, int32_t d, float scale, void* out,
                                 void* ws, size_t ws_bytes, lsv_stream stream) {
  if (B < 0 || Q < 1 || L < 1 || nh < 1 || d < 1 || !(scale > 0.f) || !std::isfinite(scale))
    return LSV_ERR_INVALID_ARG;
  const size_t need = spec_verify_attention_workspace_size(B, Q, L, nh, d);
  if (need == 0) return LSV_ERR_UNSUPPORTED;
  if (B == 0) return LSV_OK;
  if (!q || !k_cache || !v_cache || !ctx_len || !out) return LSV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(ctx_len) || !aligned16(out))
    return LSV_ERR_MISALIGNED;
  if (!ws || ws_bytes < need) return LSV_ERR_WORKSPACE;
  if (!aligned16(ws)) return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  return from_cuda(launch_attention(static_cast<const bf16*>(q), static_cast<const bf16*>(k_cache),
                                    static_cast<const bf16*>(v_cache), ctx_len, B, Q, L, nh, d, scale,
                                    static_cast<bf16*>(out), ws, *dc, reinterpret_cast<cudaStream_t>(stream)));
}

size_t spec_verify_lmhead_workspace_size(int32_t B, int32_t K, int32_t V, int32_t H) {
  if (B < 0 || K < 0 || K + 1 > kMaxVerifyRows || V <= 0 || H <= 0 || H % 64 || H > kMaxHidden) return 0;
  if ((long long)B * (K + 1) >= (1ll << 31) || (long long)B * (K + 1) * ((V + 127) / 128) >= (1ll << 31)) return 0;
  return lmhead_ws_bytes(B, K, V);
}

lsv_status spec_verify_lmhead(const void* hidden, const void* w_vocab, const int32_t* drafts, int32_t B, int32_t K,
                              int32_t V, int32_t H, int32_t* argmax_opt, int32_t* accept_len, int32_t* committed,
                              void* ws, size_t ws_bytes, lsv_stream stream) {
  if (B < 0 || K < 0 || V <= 0 || H <= 0) return LSV_ERR_INVALID_ARG;
  if (K + 1 > kMaxVerifyRows || H % 64 || H > kMaxHidden) return LSV_ERR_UNSUPPORTED;
  const size_t need = spec_verify_lmhead_workspace_size(B, K, V, H);
  if (need == 0) return LSV_ERR_UNSUPPORTED;
  if (B == 0) return LSV_OK;
  if (!hidden || !w_vocab || !accept_len || !committed || (K > 0 && !drafts)) return LSV_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(w_vocab) || !aligned16(drafts) || !aligned16(argmax_opt) ||
      !aligned16(accept_len) || !aligned16(committed))
    return LSV_ERR_MISALIGNED;
  if (!ws || ws_bytes < need) return LSV_ERR_WORKSPACE;
  if (!aligned16(ws)) return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  return from_cuda(launch_lmhead_accept(static_cast<const bf16*>(hidden), static_cast<const bf16*>(w_vocab), drafts,
                                        B, K, V, H, argmax_opt, accept_len, committed, ws, *dc,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

size_t spec_verify_workspace_size(int32_t B, int32_t K, int32_t V) {
  if (B < 0 || K < 0 || K + 1 > kMaxVerifyRows || V <= 0) return 0;
  if ((long long)B * (K + 1) >= (1ll << 31)) return 0;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return 0;
  return accept_ws_bytes(B, K, V, dc->num_sms);
}

lsv_status spec_verify_accept(const void* logits, const int32_t* drafts, int32_t B, int32_t K, int32_t V,
                              int32_t* argmax_opt, int32_t* accept_len, int32_t* committed, void* ws,
                              size_t ws_bytes, lsv_stream stream) {
  if (B < 0 || K < 0 || V <= 0) return LSV_ERR_INVALID_ARG;
  if (K + 1 > kMaxVerifyRows || (long long)B * (K + 1) >= (1ll << 31)) return LSV_ERR_UNSUPPORTED;
  if (B == 0) return LSV_OK;
  if (!logits || !accept_len || !committed || (K > 0 && !drafts)) return LSV_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(drafts) || !aligned16(argmax_opt) || !aligned16(accept_len) ||
      !aligned16(committed))
    return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  if (!ws || ws_bytes < accept_ws_bytes(B, K, V, dc->num_sms)) return LSV_ERR_WORKSPACE;
  if (!aligned16(ws)) return LSV_ERR_MISALIGNED;
  return from_cuda(launch_accept(static_cast<const bf16*>(logits), drafts, B, K, V, argmax_opt, accept_len,
                                 committed, ws, *dc, reinterpret_cast<cudaStream_t>(stream)));
}

lsv_status rmsnorm_residual(void* x, const void* y, void* h, int32_t T, int32_t H, float eps, lsv_stream stream) {
  if (T < 0 || H <= 0 || !(eps >= 0.0f)) return LSV_ERR_INVALID_ARG;
  if (T == 0) return LSV_OK;
  if (!x || !y || !h) return LSV_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(h)) return LSV_ERR_MISALIGNED;
  return from_cuda(launch_rmsnorm_residual(static_cast<bf16*>(x), static_cast<const bf16*>(y), static_cast<bf16*>(h),
                                           T, H, eps, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
