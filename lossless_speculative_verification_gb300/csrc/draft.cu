// draft.cu -- the recursive FastMTP draft block.
//
// One shared dense draft block, applied K times, proposes the drafts that the
// verify pass then checks (kg.zhiyong.dev, "The speed comes from three layers
// working together"; evolve.pub review, "Scope & Claims").  The pages say no
// more about the block; the reading implemented here is an MTP module of the
// decoder's family.  Step i takes the previous state h and token t (step 1:
// the verifier's last hidden state and the last committed token):
//   u = W_p [RMSNorm(h); RMSNorm(E[t])]
//   a = RMSNorm(u); q, k, v = W_q a, W_k a, W_v a; k and v go into the block's
//   cache of the sequence, and q attends to it (causal, its own entry included)
//   u = u + W_o attn;  f = RMSNorm(u);  u = u + W_down(silu(W_gate f) * W_up f)
//   draft = argmax_v (W_vocab RMSNorm(u))_v,  h_next = u
// Every value passed between kernels is bf16; sums are fp32.
//
// Kernels of this file: the row normalisation that also gathers embedding
// rows, the append of a step's keys and values to the caches, and a dense
// bf16 product y = x W^T on tcgen05 (TMA-fed, TMEM accumulators, bf16 store)
// for products of more than 256 rows.  The rest reuses the library's own
// kernels: the few-row split-K product (skinny.cu) for the projections, with
// the RMSNorms of u folded into the q/k/v and gate/up products and the
// residual adds into the W_o and down epilogues, the verify-attention kernel
// at one query per sequence, and the output layer fused with the greedy
// search, which writes each step's token straight into the drafts.
#include <math.h>

#include "internal.h"
#include "lsv.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lsv {
namespace {

// ----------------------------------------------------------------------------- dense product
constexpr int kDgThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kDgEpiThreads = 128;
constexpr int kDgStages = 8;
constexpr int kDgM = 128;                // rows of x per item (one TMEM lane each)
constexpr int kDgN = 32;                 // rows of w (output columns) per item
constexpr int kDgAChunk = kDgM * 128;    // one 64-wide K chunk of the x tile
constexpr int kDgBChunk = kDgN * 128;    // one 64-wide K chunk of the w tile

struct DgSmem {
  static constexpr int kStage = kDgAChunk + kDgBChunk;
  static constexpr int kRing = kDgStages * kStage;
  static constexpr int kBars = (2 * kDgStages + 5) * 8;
  static constexpr int kTotal = 1024 + kRing + kBars + 16;
};

struct DgParams {
  int M, N, K;
  int ntn;     // output column tiles
  int nitems;  // row tiles x column tiles
  bf16* y;     // [M, ldy]
  int ldy;
  int* err;
  uint64_t wait_ns;
};

// y[m, n] = bf16(sum_k x[m, k] w[n, k]): persistent CTAs over (row tile, column tile) items.
__global__ void __launch_bounds__(kDgThreads, 1) dense_gemm_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                   const __grid_constant__ CUtensorMap wmap,
                                                                   const DgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DgSmem::kRing);
  uint64_t* full = bars;
  uint64_t* empty = bars + kDgStages;
  uint64_t* tfull = bars + 2 * kDgStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* final_bar = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDgStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kDgEpiThreads);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * kDgN);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&wmap);
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();
  pdl_wait();  // x comes from the preceding kernel
  const int nk = p.K / 64;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < p.nitems && ok; it += gridDim.x) {
        const int tm = it / p.ntn, tn = it - tm * p.ntn;
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          uint8_t* a_s = smem + stage * DgSmem::kStage;
          uint8_t* b_s = a_s + kDgAChunk;
          mbar_arrive_expect_tx(&full[stage], kDgAChunk + kDgBChunk);
          tma_load_2d(a_s, &xmap, &full[stage], kc * 64, tm * kDgM, pol_x);
          tma_load_2d(b_s, &wmap, &full[stage], kc * 64, tn * kDgN, pol_w);
          if (++stage == kDgStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        __threadfence_block();
        mbar_arrive(&full[stage]);  // wake the MMA issuer so that it sees the abort
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16_f32(kDgM, kDgN);
      for (int it = blockIdx.x; it < p.nitems && ok; it += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.wait_ns)) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kDgN);
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&full[stage], phase, p.wait_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          if (*abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_s = smem_u32(smem + stage * DgSmem::kStage);
          const uint32_t b_s = a_s + kDgAChunk;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d_tmem, sdesc_kmajor_sw128(a_s + kk * 32), sdesc_kmajor_sw128(b_s + kk * 32), idesc,
                      (kc | kk) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == kDgStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        *abort_flag = 1;
        __threadfence_block();
        mbar_arrive(&tfull[acc]);  // wake the epilogue so that it sees the abort
      }
      umma_commit(final_bar);  // every MMA has completed before TMEM is released
      if (!mbar_wait(final_bar, 0, p.wait_ns)) set_error(p.err, kErrTimeout);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    // Warp w reads TMEM lanes 32*(w%4)..+31: one row of x per thread, kDgN output columns.
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = blockIdx.x; it < p.nitems; it += gridDim.x) {
      const int tm = it / p.ntn, tn = it - tm * p.ntn;
      const bool got = mbar_wait(&tfull[acc], acc_phase, p.wait_ns);
      if (!got) set_error(p.err, kErrTimeout);
      if (named_bar_red_or(1, kDgEpiThreads, !got || *abort_flag)) break;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * kDgN);
      static_assert(kDgN == 32, "two 16-column TMEM loads per row");
      uint32_t r0[16], r1[16];
      tmem_ld_32x32b_x16(t_row, r0);
      tmem_ld_32x32b_x16(t_row + 16, r1);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
      const int row = tm * kDgM + 32 * q + lane;  // rows past M are the zero-filled part of the tile
      const int n0 = tn * kDgN;
      if (row >= p.M) continue;
      bf16* yr = p.y + (size_t)row * p.ldy + n0;
      auto col = [&](int j) { return __uint_as_float(j < 16 ? r0[j & 15] : r1[j & 15]); };
      if (n0 + kDgN <= p.N) {
        uint32_t pk[kDgN / 2];
#pragma unroll
        for (int j = 0; j < kDgN / 2; ++j) {
          const __nv_bfloat162 v = __floats2bfloat162_rn(col(2 * j), col(2 * j + 1));
          pk[j] = *reinterpret_cast<const uint32_t*>(&v);
        }
#pragma unroll
        for (int j = 0; j < kDgN / 8; ++j)
          reinterpret_cast<uint4*>(yr)[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < kDgN; ++j)
          if (n0 + j < p.N) yr[j] = __float2bfloat16_rn(col(j));
      }
    }
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 2 * kDgN);
  }
}

// ----------------------------------------------------------------------------- small kernels
constexpr int kDnThreads = 256;

// Row b of blockIdx.y == 0: y[b, 0:H] = bf16(RMSNorm(a[b, :])).  Of blockIdx.y == 1 (the block's
// input): y[b, H:2H] = bf16(RMSNorm(e[rows[b * rows_ld], :])), an embedding row; a row index
// outside [0, nsrc) writes zeros and raises LSV_ERR_DEVICE_INDEX.
__global__ void __launch_bounds__(kDnThreads) draft_norm_kernel(const bf16* __restrict__ a,
                                                                const bf16* __restrict__ e, const int32_t* rows,
                                                                int rows_ld, int nsrc, bf16* __restrict__ y,
                                                                int ldy, int H, float eps, int* err) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const bf16* xr = a + (size_t)b * H;
  bf16* yr = y + (size_t)b * ldy;
  if (blockIdx.y == 1) {
    yr += H;
    const int src = __ldcg(rows + (size_t)b * rows_ld);
    if (src < 0 || src >= nsrc) {
      if (threadIdx.x == 0) set_error(err, kErrDeviceIndex);
      for (int c = threadIdx.x; c < H; c += kDnThreads) yr[c] = __float2bfloat16_rn(0.f);
      return;
    }
    xr = e + (size_t)src * H;
  }
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += kDnThreads) {
    const float f = __bfloat162float(xr[c]);
    ss = fmaf(f, f, ss);
  }
  __shared__ float red[kDnThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kDnThreads / 32; ++w) tot += red[w];
  const float scale = rsqrtf(tot / (float)H + eps);
  for (int c = threadIdx.x; c < H; c += kDnThreads) yr[c] = __float2bfloat16_rn(__bfloat162float(xr[c]) * scale);
}

// The step's key and value rows of sequence b go to cache position len_in[b] (all heads: one
// row of H values); len_out[b] = len_in[b] + 1.  A full cache raises LSV_ERR_DEVICE_INDEX.
__global__ void __launch_bounds__(128) draft_append_kernel(const bf16* __restrict__ k, const bf16* __restrict__ v,
                                                           bf16* __restrict__ kc, bf16* __restrict__ vc,
                                                           const int32_t* len_in, int32_t* len_out, int L, int H,
                                                           int* err) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int n = __ldcg(len_in + b);
  if (n < 0 || n >= L) {
    if (threadIdx.x == 0) {
      set_error(err, kErrDeviceIndex);
      len_out[b] = n < 0 ? 0 : n;
    }
    return;
  }
  const uint4* ks = reinterpret_cast<const uint4*>(k + (size_t)b * H);
  const uint4* vs = reinterpret_cast<const uint4*>(v + (size_t)b * H);
  uint4* kd = reinterpret_cast<uint4*>(kc + ((size_t)b * L + n) * H);
  uint4* vd = reinterpret_cast<uint4*>(vc + ((size_t)b * L + n) * H);
  for (int c = threadIdx.x; c < H / 8; c += blockDim.x) {
    kd[c] = ks[c];
    vd[c] = vs[c];
  }
  if (threadIdx.x == 0) len_out[b] = n + 1;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }


}  // namespace

cudaError_t launch_dense_gemm(const bf16* x, const bf16* w, bf16* y, int M, int N, int K, const DeviceCtx& dc,
                              cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  const cudaError_t ea = ensure_smem_attr(reinterpret_cast<const void*>(dense_gemm_kernel), DgSmem::kTotal, dc.device);
  if (ea != cudaSuccess) return ea;
  DgParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.ntn = (N + kDgN - 1) / kDgN;
  p.nitems = ((M + kDgM - 1) / kDgM) * p.ntn;
  p.y = y;
  p.ldy = N;
  p.err = dc.err;
  p.wait_ns = wait_limit_ns();
  CUtensorMap xmap, wmap;
  if (!make_map(&xmap, x, M, K, kDgM) || !make_map(&wmap, w, N, K, kDgN)) return cudaErrorInvalidValue;
  const int grid = p.nitems < dc.num_sms ? p.nitems : dc.num_sms;
  return launch_pdl(dense_gemm_kernel, dim3(grid), dim3(kDgThreads), DgSmem::kTotal, s, xmap, wmap, p);
}

// Workspace of the draft loop: activations, the lengths, and the sub-workspaces of the
// kernels it uses (each of which needs zero on first use and leaves its counters zero).
struct DraftWs {
  size_t inp, u, a, q, k, v, attn, y, f, hn, act, z, len0, len1, attn_ws, lm_ws, total;
  size_t attn_bytes, lm_bytes;
};

DraftWs draft_ws_layout(int B, int H, int nh, int I, int V, int L) {
  DraftWs w = {};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += round256(bytes);
    return at;
  };
  const size_t act = (size_t)B * H * 2;
  w.inp = take(2 * act);
  w.u = take(act);
  w.a = take(act);
  w.q = take(act);
  w.k = take(act);
  w.v = take(act);
  w.attn = take(act);
  w.y = take(act);
  w.f = take(act);
  w.hn = take(act);
  w.act = take((size_t)B * I * 2);
  w.z = take(act);
  w.len0 = take((size_t)B * 4);
  w.len1 = take((size_t)B * 4);
  w.attn_bytes = spec_verify_attention_workspace_size(B, 1, L, nh, H / nh);
  w.lm_bytes = spec_verify_lmhead_workspace_size(B, 0, V, H);
  w.attn_ws = take(w.attn_bytes);
  w.lm_ws = take(w.lm_bytes);
  w.total = (w.attn_bytes && w.lm_bytes) ? o : 0;
  return w;
}

}  // namespace lsv

using namespace lsv;

extern "C" {

lsv_status dense_matmul(const void* x, const void* w, void* y, int32_t M, int32_t N, int32_t K, lsv_stream stream) {
  if (M < 0 || N < 0 || K <= 0) return LSV_ERR_INVALID_ARG;
  if (K % 64 || K > kMaxHidden || N % 8) return LSV_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return LSV_OK;
  if (!x || !w || !y) return LSV_ERR_INVALID_ARG;
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!al(x) || !al(w) || !al(y)) return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  const bf16* xb = static_cast<const bf16*>(x);
  const bf16* wb = static_cast<const bf16*>(w);
  bf16* yb = static_cast<bf16*>(y);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // few rows of x: the weights on the MMA's M side, K split over clusters (skinny.cu)
  const cudaError_t e = M <= kSkMaxRows ? launch_skinny(xb, M, K, &wb, &N, &yb, &N, 1, false, *dc, s)
                                        : launch_dense_gemm(xb, wb, yb, M, N, K, *dc, s);
  return e == cudaSuccess ? LSV_OK : LSV_ERR_CUDA;
}

size_t spec_draft_workspace_size(int32_t B, int32_t H, int32_t nh, int32_t I, int32_t V, int32_t L) {
  if (B < 0 || H <= 0 || nh <= 0 || H % nh || I <= 0 || V <= 0 || L <= 0) return 0;
  const int d = H / nh;
  if (H % 64 || H > kMaxHidden || (d != 64 && d != 128) || I % 64 || I > kMaxHidden) return 0;
  if (B > kSkMaxRows) return 0;
  return draft_ws_layout(B < 1 ? 1 : B, H, nh, I, V, L).total;
}

lsv_status spec_draft_loop(const lsv_draft_weights* wt, const void* h0, const int32_t* t0, void* k_cache,
                           void* v_cache, const int32_t* ctx_len, int32_t B, int32_t K, int32_t H, int32_t nh,
                           int32_t I, int32_t V, int32_t L, int32_t* drafts, void* h_out, void* ws, size_t ws_bytes,
                           lsv_stream stream) {
  if (B < 0 || K < 1 || K + 1 > kMaxVerifyRows || !wt) return LSV_ERR_INVALID_ARG;
  const size_t need = spec_draft_workspace_size(B, H, nh, I, V, L);
  if (need == 0) return LSV_ERR_UNSUPPORTED;
  if (B == 0) return LSV_OK;
  const void* ptrs[] = {wt->emb, wt->w_proj, wt->w_q, wt->w_k, wt->w_v, wt->w_o, wt->w_gate_up, wt->w_down,
                        wt->w_vocab, h0, k_cache, v_cache, ws};
  for (const void* p : ptrs) {
    if (!p) return LSV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p) & 15) return LSV_ERR_MISALIGNED;
  }
  if (!t0 || !ctx_len || !drafts) return LSV_ERR_INVALID_ARG;
  if (h_out && (reinterpret_cast<uintptr_t>(h_out) & 15)) return LSV_ERR_MISALIGNED;
  if (ws_bytes < need) return LSV_ERR_WORKSPACE;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const DraftWs L8 = draft_ws_layout(B, H, nh, I, V, L);
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto act = [&](size_t off) { return reinterpret_cast<bf16*>(w + off); };
  auto i32 = [&](size_t off) { return reinterpret_cast<int32_t*>(w + off); };
  auto wgt = [](const void* p) { return static_cast<const bf16*>(p); };
  const bf16* emb = wgt(wt->emb);
  bf16* kc = static_cast<bf16*>(k_cache);
  bf16* vc = static_cast<bf16*>(v_cache);
  const float eps = 1e-6f;
  const int d = H / nh;
  const int nH = H, n2I = 2 * I, ldH = H, ldI = I;
  const int nqkv[3] = {H, H, H}, ldqkv[3] = {H, H, H};
  const bf16* wqkv[3] = {wgt(wt->w_q), wgt(wt->w_k), wgt(wt->w_v)};
  bf16* yqkv[3] = {act(L8.q), act(L8.k), act(L8.v)};
  cudaError_t e = cudaSuccess;
  const int32_t* len_cur = ctx_len;
  for (int i = 0; i < K && e == cudaSuccess; ++i) {
    int32_t* len_next = i32((i & 1) ? L8.len1 : L8.len0);
    const bf16* h_prev = i == 0 ? static_cast<const bf16*>(h0) : act(L8.u);
    // the previous token: t0, then the last step's draft (column i - 1 of drafts)
    const int32_t* t_prev = i == 0 ? t0 : drafts + (i - 1);
    const int t_ld = i == 0 ? 1 : K;
    // the block's input [RMSNorm(h); RMSNorm(E[t])], one launch for both halves
    e = launch_pdl(draft_norm_kernel, dim3(B, 2), dim3(kDnThreads), 0, s, h_prev, emb, t_prev, t_ld, V, act(L8.inp),
                   2 * H, H, eps, dc->err);
    auto sk1 = [&](const bf16* x, int K_, const bf16* wm, int n, bf16* y, int ldy, bool swiglu) {
      return launch_skinny(x, B, K_, &wm, &n, &y, &ldy, 1, swiglu, *dc, s);
    };
    if (e == cudaSuccess) e = sk1(act(L8.inp), 2 * H, wgt(wt->w_proj), nH, act(L8.u), ldH, false);
    // q, k, v of RMSNorm(u): the norm is folded into the products (each output row scaled by its
    // input row's 1/rms), so the normalised rows are never stored
    if (e == cudaSuccess) e = launch_skinny(act(L8.u), B, H, wqkv, nqkv, yqkv, ldqkv, 3, false, *dc, s, eps);
    if (e == cudaSuccess)
      e = launch_pdl(draft_append_kernel, dim3(B), dim3(128), 0, s, (const bf16*)act(L8.k), (const bf16*)act(L8.v), kc,
                     vc, len_cur, len_next, L, H, dc->err);
    if (e == cudaSuccess)
      e = launch_attention(act(L8.q), kc, vc, len_next, B, 1, L, nh, d, 1.0f / sqrtf((float)d), act(L8.attn),
                           w + L8.attn_ws, *dc, s);
    // u += attn W_o^T, the residual added in the product's epilogue (one rounding)
    const bf16* res_u = act(L8.u);
    if (e == cudaSuccess) {
      const bf16* wo = wgt(wt->w_o);
      bf16* yu = act(L8.u);
      e = launch_skinny(act(L8.attn), B, H, &wo, &nH, &yu, &ldH, 1, false, *dc, s, 0.0f, &res_u);
    }
    // the dense SwiGLU FFN of RMSNorm(u) (the norm folded in), then u += act W_down^T
    if (e == cudaSuccess) {
      const bf16* wgu = wgt(wt->w_gate_up);
      bf16* ya = act(L8.act);
      e = launch_skinny(act(L8.u), B, H, &wgu, &n2I, &ya, &ldI, 1, true, *dc, s, eps);
    }
    if (e == cudaSuccess) {
      const bf16* wd = wgt(wt->w_down);
      bf16* yu = act(L8.u);
      e = launch_skinny(act(L8.act), B, I, &wd, &nH, &yu, &ldH, 1, false, *dc, s, 0.0f, &res_u);
    }
    // the draft token: the greedy token of W_vocab RMSNorm(u), which is the greedy token of W_vocab u
    // (the norm scales a row's logits by one positive factor), written to column i of drafts
    if (e == cudaSuccess)
      e = launch_lmhead_accept(act(L8.u), wgt(wt->w_vocab), nullptr, B, 0, V, H, drafts + i, nullptr, nullptr,
                               w + L8.lm_ws, *dc, s, K);
    len_cur = len_next;
  }
  if (e == cudaSuccess && h_out) e = cudaMemcpyAsync(h_out, act(L8.u), (size_t)B * H * 2, cudaMemcpyDeviceToDevice, s);
  return e == cudaSuccess ? LSV_OK : LSV_ERR_CUDA;
}

}  // extern "C"
