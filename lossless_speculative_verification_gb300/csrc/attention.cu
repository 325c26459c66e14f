// attention.cu -- causal attention of the verified positions over the cache.
//
// In the verify pass every sequence presents its K+1 positions (the last
// committed token and the K drafts) at once; each attends to the sequence's
// cache up to and including itself (kg.zhiyong.dev, "Why FastMTP fits OCR
// particularly well": the drafts are verified in one pass; evolve.pub review,
// Section 3.1).  With Q = K+1 query rows and thousands of cached positions the
// work is a stream over the cache, so it runs on CUDA cores:
//
//   split kernel: CTA (split, head, sequence) takes up to kAtChunk cached
//     positions.  Lane = position for the scores (each lane reads its key row
//     with 16-byte loads and forms Q dot products in fp32), then lane = four
//     head dimensions for the values (each lane reads 8 bytes of each value
//     row).  An online softmax keeps, per query, the running maximum, the sum
//     of exponentials and the unnormalised output; the four warps' states are
//     merged and written as the split's partial.
//   combine kernel: per (head, sequence), the splits' partials rescaled to the
//     common maximum and summed; out = sum / normaliser, rounded to bf16.
#include "internal.h"
#include "ptx.cuh"

namespace lsv {
namespace {

constexpr int kAtThreads = 128;
constexpr int kAtWarps = kAtThreads / 32;
#ifndef LSV_ATTN_CHUNK
#define LSV_ATTN_CHUNK 512
#endif
constexpr int kAtChunk = LSV_ATTN_CHUNK;  // cached positions per split (a multiple of 128)
static_assert(kAtChunk % (32 * kAtWarps) == 0, "a split is a whole number of warp blocks");
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
__global__ void __launch_bounds__(kAtThreads) attn_split_kernel(
    const bf16* __restrict__ q, const bf16* __restrict__ kc, const bf16* __restrict__ vc,
    const int32_t* __restrict__ ctx_len, int Q, int L, int nh, float scale, int nsplit, float* __restrict__ o_part,
    float* __restrict__ ml_part, int* err) {
  constexpr int DL = D / 32;  // value dimensions per lane
  __shared__ __align__(16) float q_s[kMaxAttnQ][D];
  __shared__ float p_s[kAtWarps][kMaxAttnQ][32];
  __shared__ float m_s[kAtWarps][kMaxAttnQ], l_s[kAtWarps][kMaxAttnQ];
  __shared__ float o_s[kAtWarps][kMaxAttnQ][D];
  pdl_wait();
  pdl_trigger();
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int n = ctx_len[b];
  if (n < Q || n > L) {
    if (threadIdx.x == 0) set_error(err, kErrDeviceIndex);
    n = 0;  // contributes nothing; the combine writes zeros
  }
  const size_t row_stride = (size_t)nh * D;  // elements between consecutive positions of one sequence
  // queries, pre-scaled so that the softmax can use exp2
  for (int i = threadIdx.x; i < Q * D; i += kAtThreads) {
    const int j = i / D, c = i - j * D;
    q_s[j][c] = __bfloat162float(q[(((size_t)b * Q + j) * nh + h) * D + c]) * (scale * kLog2e);
  }
  __syncthreads();
  const int t_begin = split * kAtChunk;
  const int t_end = min(n, t_begin + kAtChunk);
  const int first_masked = n - Q;  // positions > first_masked + j are hidden from query j
  float m[kMaxAttnQ], l[kMaxAttnQ], o[kMaxAttnQ][DL];
#pragma unroll
  for (int j = 0; j < kMaxAttnQ; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int c = 0; c < DL; ++c) o[j][c] = 0.f;
  }
  const bf16* kb = kc + ((size_t)b * L * nh + h) * D;
  const bf16* vb = vc + ((size_t)b * L * nh + h) * D;
  for (int t0 = t_begin + 32 * warp; t0 < t_end; t0 += 32 * kAtWarps) {
    // scores: lane = position
    const int t = t0 + lane;
    float s[kMaxAttnQ];
#pragma unroll
    for (int j = 0; j < kMaxAttnQ; ++j) s[j] = 0.f;
    if (t < t_end) {
      const uint4* kr = reinterpret_cast<const uint4*>(kb + (size_t)t * row_stride);
#pragma unroll 4
      for (int c8 = 0; c8 < D / 8; ++c8) {
        const uint4 kv = __ldg(kr + c8);
        const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
        float kf[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          kf[2 * i] = __uint_as_float(w[i] << 16);
          kf[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
#pragma unroll
        for (int j = 0; j < kMaxAttnQ; ++j)
          if (j < Q) {
            const float4 qa = *reinterpret_cast<const float4*>(&q_s[j][8 * c8]);
            const float4 qb = *reinterpret_cast<const float4*>(&q_s[j][8 * c8 + 4]);
            s[j] = fmaf(qa.x, kf[0], s[j]);
            s[j] = fmaf(qa.y, kf[1], s[j]);
            s[j] = fmaf(qa.z, kf[2], s[j]);
            s[j] = fmaf(qa.w, kf[3], s[j]);
            s[j] = fmaf(qb.x, kf[4], s[j]);
            s[j] = fmaf(qb.y, kf[5], s[j]);
            s[j] = fmaf(qb.z, kf[6], s[j]);
            s[j] = fmaf(qb.w, kf[7], s[j]);
          }
      }
    }
    // online softmax per query over these 32 positions
#pragma unroll
    for (int j = 0; j < kMaxAttnQ; ++j) {
      if (j >= Q) continue;
      const bool vis = t < t_end && t <= first_masked + j;
      const float sj = vis ? s[j] : -INFINITY;
      float bm = sj;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
      const float mn = fmaxf(m[j], bm);
      const float pj = vis ? exp2f(sj - mn) : 0.f;
      float ps = pj;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      const float corr = (m[j] == -INFINITY) ? 0.f : exp2f(m[j] - mn);
      if (mn != -INFINITY) {
        l[j] = l[j] * corr + ps;
#pragma unroll
        for (int c = 0; c < DL; ++c) o[j][c] *= corr;
        m[j] = mn;
      }
      p_s[warp][j][lane] = pj;
    }
    __syncwarp();
    // values: lane = DL head dimensions
    const int nk = min(32, t_end - t0);
#pragma unroll 8
    for (int kk = 0; kk < nk; ++kk) {
      const bf16* vr = vb + (size_t)(t0 + kk) * row_stride + lane * DL;
      float vf[DL];
      if constexpr (DL == 4) {
        const uint2 vv = __ldg(reinterpret_cast<const uint2*>(vr));
        vf[0] = __uint_as_float(vv.x << 16);
        vf[1] = __uint_as_float(vv.x & 0xFFFF0000u);
        vf[2] = __uint_as_float(vv.y << 16);
        vf[3] = __uint_as_float(vv.y & 0xFFFF0000u);
      } else {
        const uint32_t vv = __ldg(reinterpret_cast<const uint32_t*>(vr));
        vf[0] = __uint_as_float(vv << 16);
        vf[1] = __uint_as_float(vv & 0xFFFF0000u);
      }
#pragma unroll
      for (int j = 0; j < kMaxAttnQ; ++j) {
        if (j >= Q) continue;
        const float pj = p_s[warp][j][kk];
#pragma unroll
        for (int c = 0; c < DL; ++c) o[j][c] = fmaf(pj, vf[c], o[j][c]);
      }
    }
    __syncwarp();
  }
  // merge the warps' states and write this split's partial
#pragma unroll
  for (int j = 0; j < kMaxAttnQ; ++j) {
    if (j >= Q) continue;
    if (lane == 0) {
      m_s[warp][j] = m[j];
      l_s[warp][j] = l[j];
    }
#pragma unroll
    for (int c = 0; c < DL; ++c) o_s[warp][j][lane * DL + c] = o[j][c];
  }
  __syncthreads();
  const size_t part = (((size_t)b * nh + h) * nsplit + split) * Q;
  for (int i = threadIdx.x; i < Q * D; i += kAtThreads) {
    const int j = i / D, c = i - j * D;
    float mm = -INFINITY;
    for (int w = 0; w < kAtWarps; ++w) mm = fmaxf(mm, m_s[w][j]);
    float lsum = 0.f, osum = 0.f;
    if (mm != -INFINITY)
      for (int w = 0; w < kAtWarps; ++w) {
        if (m_s[w][j] == -INFINITY) continue;
        const float f = exp2f(m_s[w][j] - mm);
        lsum += l_s[w][j] * f;
        osum += o_s[w][j][c] * f;
      }
    o_part[(part + j) * D + c] = osum;
    if (c == 0) {
      ml_part[(part + j) * 2] = mm;
      ml_part[(part + j) * 2 + 1] = lsum;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(const float* __restrict__ o_part,
                                                         const float* __restrict__ ml_part, int Q, int nh,
                                                         int nsplit, bf16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  for (int j = 0; j < Q; ++j) {
    float mm = -INFINITY;
    for (int s = 0; s < nsplit; ++s) mm = fmaxf(mm, ml_part[((((size_t)b * nh + h) * nsplit + s) * Q + j) * 2]);
    float lsum = 0.f, osum = 0.f;
    if (mm != -INFINITY)
      for (int s = 0; s < nsplit; ++s) {
        const size_t at = (((size_t)b * nh + h) * nsplit + s) * Q + j;
        const float ms = ml_part[at * 2];
        if (ms == -INFINITY) continue;
        const float f = exp2f(ms - mm);
        lsum += ml_part[at * 2 + 1] * f;
        osum += o_part[at * D + c] * f;
      }
    out[(((size_t)b * Q + j) * nh + h) * D + c] = __float2bfloat16_rn(lsum > 0.f ? osum / lsum : 0.f);
  }
}

}  // namespace

int attention_splits(int L) { return L <= 0 ? 1 : (L + kAtChunk - 1) / kAtChunk; }

size_t attention_ws_bytes(int B, int Q, int L, int nh, int d) {
  const size_t parts = (size_t)B * nh * attention_splits(L) * Q;
  const size_t o = (parts * d * 4 + 255) / 256 * 256;
  const size_t ml = (parts * 2 * 4 + 255) / 256 * 256;
  return o + ml + 256;
}

cudaError_t launch_attention(const bf16* q, const bf16* kc, const bf16* vc, const int32_t* ctx_len, int B, int Q,
                             int L, int nh, int d, float scale, bf16* out, void* ws, const DeviceCtx& dc,
                             cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const int nsplit = attention_splits(L);
  const size_t parts = (size_t)B * nh * nsplit * Q;
  float* o_part = reinterpret_cast<float*>(ws);
  float* ml_part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + (parts * d * 4 + 255) / 256 * 256);
  const dim3 grid(nsplit, nh, B);
  cudaError_t e;
  if (d == 128)
    e = launch_pdl(attn_split_kernel<128>, grid, dim3(kAtThreads), 0, s, q, kc, vc, ctx_len, Q, L, nh, scale, nsplit,
                   o_part, ml_part, dc.err);
  else
    e = launch_pdl(attn_split_kernel<64>, grid, dim3(kAtThreads), 0, s, q, kc, vc, ctx_len, Q, L, nh, scale, nsplit,
                   o_part, ml_part, dc.err);
  if (e != cudaSuccess) return e;
  if (d == 128)
    return launch_pdl(attn_combine_kernel<128>, dim3(nh, B), dim3(128), 0, s, (const float*)o_part,
                      (const float*)ml_part, Q, nh, nsplit, out);
  return launch_pdl(attn_combine_kernel<64>, dim3(nh, B), dim3(64), 0, s, (const float*)o_part,
                    (const float*)ml_part, Q, nh, nsplit, out);
}

}  // namespace lsv
