// attention.cu -- causal attention of the verified positions over the cache.
//
// In the verify pass every sequence presents its K+1 positions (the last
// committed token and the K drafts) at once; each attends to the sequence's
// cache up to and including itself (kg.zhiyong.dev, "Why FastMTP fits OCR
// particularly well": the drafts are verified in one pass; evolve.pub review,
// Section 3.1).  With Q = K+1 <= 8 query rows per head and thousands of cached
// positions, the step is a stream of the cache through the SMs: per cached
// position and head it reads 2*d bf16 values and does 4*Q*d flops.
//
// One CTA takes one (split, head, sequence): up to kAtChunk cached positions.
//   warp 4 (producer): TMA loads of 64-position key and value tiles (the head's
//     d columns of 64 cache rows, 128-byte swizzle) into a kAtStages ring;
//   warps 0-3 (consumers): each takes 16 positions of every tile.  Scores
//     S = q K^T and the weighted values P V run on the tensor cores as
//     m16n8k16 warp MMAs whose 16 rows are the queries (rows >= Q are zero):
//     S stays in registers, the online softmax (running maximum and sum per
//     query, in fp32, exp2 of log2e-scaled scores) turns it into P in the
//     register layout the second MMA takes as its A operand, and the
//     fragments of K (ldmatrix) and V (ldmatrix.trans) come from the swizzled
//     tiles without bank conflicts.
// The four warps' states merge in shared memory into the split's partial
// (running maximum, sum, unnormalised output).  The last CTA of a
// (sequence, head) to finish -- a counter per (sequence, head), which it resets
// -- merges the splits and writes the bf16 output, so one launch does it all.
#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lsv {
namespace {

constexpr int kAtConsumers = 4;
constexpr int kAtThreads = 32 * (kAtConsumers + 1);
constexpr int kAtTile = 64;  // positions per ring stage (16 per consumer warp)
constexpr int kAtStages = 3;
#ifndef LSV_ATTN_CHUNK
#define LSV_ATTN_CHUNK 512
#endif
constexpr int kAtChunk = LSV_ATTN_CHUNK;  // cached positions per CTA
static_assert(kAtChunk % kAtTile == 0, "a split is a whole number of tiles");
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kAtBarMerge = 1;  // named barrier of the consumer warps

template <int D>
struct AtSmem {
  static constexpr int kBox = kAtTile * 128;          // 64 columns x 64 rows of bf16
  static constexpr int kStage = 2 * (D / 64) * kBox;  // key boxes, then value boxes
  static constexpr int kRing = kAtStages * kStage;
  // merge buffers (in the ring once the stream is done)
  static constexpr int kMergeO = kAtConsumers * kMaxAttnQ * D * 4;
  static_assert(kMergeO + 2 * kAtConsumers * kMaxAttnQ * 4 <= kRing, "merge buffers fit in the ring");
  static constexpr int kBars = 2 * kAtStages * 8;
  static constexpr int kTotal = 1024 + kRing + kBars + 16;
};

struct AtParams {
  const bf16* q;           // [B, Q, nh, D]
  const int32_t* ctx_len;  // [B]
  int Q, L, nh, nsplit;
  float qk_scale;  // scale * log2(e)
  float* o_part;   // [B, nh, nsplit, Q, D]
  float* ml_part;  // [B, nh, nsplit, Q, 2]: running maximum (log2 units), sum
  int* cnt;        // [B * nh] splits finished; zero between launches
  bf16* out;       // [B, Q, nh, D]
  int* err;
  uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Offset in a tile of the 16-byte chunk holding columns [8c, 8c+8) of row r
// (128-byte swizzle: chunk c of row r sits at c ^ (r mod 8)).
__device__ __forceinline__ uint32_t sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

template <int D>
__global__ void __launch_bounds__(kAtThreads) attn_split_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                const __grid_constant__ CUtensorMap vmap,
                                                                const AtParams p) {
  using SM = AtSmem<D>;
  constexpr int NB = D / 64;  // boxes per tensor per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kRing);
  uint64_t* empty = full + kAtStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kAtStages);
  volatile int* last_flag = abort_flag + 1;
  volatile int* issued_s = abort_flag + 2;
  int* done_s = const_cast<int*>(abort_flag + 3);
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();  // q, the lengths and the caches may come from the preceding kernel
  pdl_trigger();
  const int n = p.ctx_len[b];
  if (n < p.Q || n > p.L) {
    if (split == 0) {
      if (threadIdx.x == 0) set_error(p.err, kErrDeviceIndex);
      for (int i = threadIdx.x; i < p.Q * D; i += kAtThreads) {
        const int j = i / D, c = i - j * D;
        p.out[(((size_t)b * p.Q + j) * p.nh + h) * D + c] = __float2bfloat16_rn(0.f);
      }
    }
    return;
  }
  const int t_begin = split * kAtChunk;
  if (t_begin >= n) return;  // no cached position of this sequence in the split
  const int t_end = min(n, t_begin + kAtChunk);
  const int ntiles = (t_end - t_begin + kAtTile - 1) / kAtTile;
  const int nactive = (n + kAtChunk - 1) / kAtChunk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kAtConsumers);
    }
    *abort_flag = 0;
    *issued_s = 0;
    *done_s = ntiles;
    fence_barrier_init();
  }
  if (threadIdx.x == 32 * kAtConsumers) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  __syncthreads();

  if (warp == kAtConsumers) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const int row0 = b * p.L + t_begin;
      int i = 0;
      for (; i < ntiles; ++i) {
        const int s = i % kAtStages;
        if (!mbar_wait(&empty[s], ((i / kAtStages) & 1) ^ 1u, p.wait_ns)) {
          set_error(p.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + s * SM::kStage;
        mbar_arrive_expect_tx(&full[s], SM::kStage);
#pragma unroll
        for (int c = 0; c < NB; ++c) {
          tma_load_2d(st + c * SM::kBox, &kmap, &full[s], h * D + 64 * c, row0 + i * kAtTile, pol);
          tma_load_2d(st + (NB + c) * SM::kBox, &vmap, &full[s], h * D + 64 * c, row0 + i * kAtTile, pol);
        }
      }
      *issued_s = i;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    const bool row_ok = g < p.Q;
    // q as the A operand: row g = query g, k-step s covers dims [16s, 16s+16)
    uint32_t qa[D / 16][2];
    {
      const bf16* qr = p.q + (((size_t)b * p.Q + (row_ok ? g : 0)) * p.nh + h) * D;
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        qa[s][0] = row_ok ? *reinterpret_cast<const uint32_t*>(qr + 16 * s + 2 * t) : 0u;
        qa[s][1] = row_ok ? *reinterpret_cast<const uint32_t*>(qr + 16 * s + 2 * t + 8) : 0u;
      }
    }
    const int lim = row_ok ? n - p.Q + g : -1;  // last position query g sees
    float m_run = -INFINITY, l_run = 0.f;
    float o[D / 8][2];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = 0.f;
    // ldmatrix addressing: lane supplies row (lane & 7) of matrix (lane >> 3)
    const int mi = lane >> 3, mr = lane & 7;
    const int k_row = 16 * warp + 8 * (mi >> 1) + mr;  // S: matrices (n-tile, k half) = (mi>>1, mi&1)
    const int k_half = mi & 1;
    const int v_row = 16 * warp + 8 * (mi & 1) + mr;  // PV: matrices (k half, n-tile) = (mi&1, mi>>1)
    const int v_half = mi >> 1;
    int done = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % kAtStages;
      // every lane waits; the warp leaves together if any lane ran out of time
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (i / kAtStages) & 1, p.wait_ns))) {
        if (lane == 0) set_error(p.err, kErrTimeout);
        *abort_flag = 1;
        break;
      }
      const uint32_t kb = smem_u32(smem + s * SM::kStage);
      const uint32_t vb = kb + NB * SM::kBox;
      // scores of this warp's 16 positions: two n-tiles of 8
      float sc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int ch = 2 * ks + k_half;  // 16-byte chunk (8 dims) within the head
        uint32_t r[4];
        ldmatrix_x4(kb + (ch >> 3) * SM::kBox + sw128(k_row, ch & 7), r);
        mma_bf16_m16n8k16_top(sc[0], qa[ks][0], qa[ks][1], r[0], r[1]);
        mma_bf16_m16n8k16_top(sc[1], qa[ks][0], qa[ks][1], r[2], r[3]);
      }
      // online softmax of row g over its columns 2t, 2t+1 of both n-tiles
      const int pos0 = t_begin + i * kAtTile + 16 * warp + 2 * t;  // absolute position of sc[0][0]
      float sv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int pos = pos0 + 8 * (e >> 1) + (e & 1);
        sv[e] = pos <= lim ? sc[e >> 1][e & 1] * p.qk_scale : -INFINITY;
      }
      float bm = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      const float m_new = fmaxf(m_run, bm);
      const float corr = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
      float pr[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pr[e] = sv[e] == -INFINITY ? 0.f : exp2f(sv[e] - m_new);
      l_run = l_run * corr + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
      m_run = m_new;
      if (!__all_sync(0xffffffffu, corr == 1.f)) {
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
          o[nt][0] *= corr;
          o[nt][1] *= corr;
        }
      }
      const uint32_t pa0 = pack_bf16(pr[0], pr[1]);  // P[g][k = 2t, 2t+1]
      const uint32_t pa2 = pack_bf16(pr[2], pr[3]);  // P[g][k = 2t+8, 2t+9]
      // cache rows at or past n may hold anything (even NaN): zero them in the B operand
      const bool tail = pos0 - 2 * t + 15 >= n;
      const uint32_t m_lo = (pos0 < n ? 0xFFFFu : 0u) | (pos0 + 1 < n ? 0xFFFF0000u : 0u);
      const uint32_t m_hi = (pos0 + 8 < n ? 0xFFFFu : 0u) | (pos0 + 9 < n ? 0xFFFF0000u : 0u);
#pragma unroll
      for (int u = 0; u < D / 16; ++u) {
        const int ch = 2 * u + v_half;
        uint32_t r[4];
        ldmatrix_x4_trans(vb + (ch >> 3) * SM::kBox + sw128(v_row, ch & 7), r);
        if (tail) {
          r[0] &= m_lo;
          r[1] &= m_hi;
          r[2] &= m_lo;
          r[3] &= m_hi;
        }
        mma_bf16_m16n8k16_top(o[2 * u], pa0, pa2, r[0], r[1]);
        mma_bf16_m16n8k16_top(o[2 * u + 1], pa0, pa2, r[2], r[3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      done = i + 1;
    }
    if (done < ntiles && lane == 0) atomicMin(done_s, done);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);

    named_bar_sync(kAtBarMerge, 32 * kAtConsumers);  // every consumer is done with the ring
    if (!*abort_flag) {
      float* o_s = reinterpret_cast<float*>(smem);  // [warp][row][D]
      float* m_s = o_s + kAtConsumers * kMaxAttnQ * D;
      float* l_s = m_s + kAtConsumers * kMaxAttnQ;
      if (row_ok) {
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
          o_s[(warp * kMaxAttnQ + g) * D + 8 * nt + 2 * t] = o[nt][0];
          o_s[(warp * kMaxAttnQ + g) * D + 8 * nt + 2 * t + 1] = o[nt][1];
        }
        if (t == 0) {
          m_s[warp * kMaxAttnQ + g] = m_run;
          l_s[warp * kMaxAttnQ + g] = l_run;
        }
      }
      named_bar_sync(kAtBarMerge, 32 * kAtConsumers);
      // the split's state: the warps' states rescaled to their common maximum
      const size_t bh = (size_t)b * p.nh + h;
      const size_t part = (bh * p.nsplit + split) * p.Q;
      for (int e = threadIdx.x; e < p.Q * D; e += 32 * kAtConsumers) {
        const int j = e / D, c = e - j * D;
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAtConsumers; ++w) mm = fmaxf(mm, m_s[w * kMaxAttnQ + j]);
        float ls = 0.f, os = 0.f;
        if (mm != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kAtConsumers; ++w) {
            const float mw = m_s[w * kMaxAttnQ + j];
            if (mw == -INFINITY) continue;
            const float f = exp2f(mw - mm);
            ls += l_s[w * kMaxAttnQ + j] * f;
            os += o_s[(w * kMaxAttnQ + j) * D + c] * f;
          }
        }
        if (nactive == 1) {
          p.out[(((size_t)b * p.Q + j) * p.nh + h) * D + c] = __float2bfloat16_rn(ls > 0.f ? os / ls : 0.f);
        } else {
          p.o_part[(part + j) * D + c] = os;
          if (c == 0) {
            p.ml_part[(part + j) * 2] = mm;
            p.ml_part[(part + j) * 2 + 1] = ls;
          }
        }
      }
      if (nactive > 1) {
        // the last split of (b, h) to finish merges all of them
        __threadfence();
        named_bar_sync(kAtBarMerge, 32 * kAtConsumers);
        if (threadIdx.x == 0) *last_flag = atomicAdd(&p.cnt[bh], 1) == nactive - 1;
        named_bar_sync(kAtBarMerge, 32 * kAtConsumers);
        if (*last_flag) {
          __threadfence();
          const size_t part0 = bh * p.nsplit * p.Q;
          for (int e = threadIdx.x; e < p.Q * D; e += 32 * kAtConsumers) {
            const int j = e / D, c = e - j * D;
            float mm = -INFINITY;
            for (int sp = 0; sp < nactive; ++sp) mm = fmaxf(mm, __ldcg(&p.ml_part[(part0 + sp * p.Q + j) * 2]));
            float ls = 0.f, os = 0.f;
            if (mm != -INFINITY) {
              for (int sp = 0; sp < nactive; ++sp) {
                const size_t at = part0 + sp * p.Q + j;
                const float ms = __ldcg(&p.ml_part[at * 2]);
                if (ms == -INFINITY) continue;
                const float f = exp2f(ms - mm);
                ls += __ldcg(&p.ml_part[at * 2 + 1]) * f;
                os += __ldcg(&p.o_part[at * D + c]) * f;
              }
            }
            p.out[(((size_t)b * p.Q + j) * p.nh + h) * D + c] = __float2bfloat16_rn(ls > 0.f ? os / ls : 0.f);
          }
          if (threadIdx.x == 0) p.cnt[bh] = 0;  // ready for the next launch
        }
      }
    }
  }
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // let the copies already issued land before the CTA's shared memory goes away
    for (int i = *done_s; i < *issued_s; ++i) mbar_wait(&full[i % kAtStages], (i / kAtStages) & 1, p.wait_ns);
  }
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

int attention_splits(int L) { return L <= 0 ? 1 : (L + kAtChunk - 1) / kAtChunk; }

// The split counters sit in a block of fixed size at the start of every workspace, so that
// calls of different shapes sharing one workspace never write partials over another shape's
// counters (each call leaves its own counters zero).
constexpr size_t kAttnCounterBytes = (size_t)kAttnMaxPairs * 4;

size_t attention_ws_bytes(int B, int Q, int L, int nh, int d) {
  const size_t parts = (size_t)B * nh * attention_splits(L) * Q;
  return kAttnCounterBytes + round256(parts * d * 4) + round256(parts * 2 * 4);
}

cudaError_t launch_attention(const bf16* q, const bf16* kc, const bf16* vc, const int32_t* ctx_len, int B, int Q,
                             int L, int nh, int d, float scale, bf16* out, void* ws, const DeviceCtx& dc,
                             cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  static int attr_done[64][2] = {{0}};
  if (dc.device < 0 || dc.device >= 64) return cudaErrorInvalidDevice;
  const int di = d == 128 ? 1 : 0;
  if (!attr_done[dc.device][di]) {
    const cudaError_t e =
        d == 128 ? cudaFuncSetAttribute(attn_split_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        AtSmem<128>::kTotal)
                 : cudaFuncSetAttribute(attn_split_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        AtSmem<64>::kTotal);
    if (e != cudaSuccess) return e;
    attr_done[dc.device][di] = 1;
  }
  AtParams p;
  p.q = q;
  p.ctx_len = ctx_len;
  p.Q = Q;
  p.L = L;
  p.nh = nh;
  p.nsplit = attention_splits(L);
  p.qk_scale = scale * kLog2e;
  const size_t parts = (size_t)B * nh * p.nsplit * Q;
  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  p.cnt = reinterpret_cast<int*>(w);
  p.o_part = reinterpret_cast<float*>(w + kAttnCounterBytes);
  p.ml_part = reinterpret_cast<float*>(w + kAttnCounterBytes + round256(parts * d * 4));
  p.out = out;
  p.err = dc.err;
  p.wait_ns = wait_limit_ns();
  // the caches as [B*L rows, nh*d columns]; a tile is d columns of 64 rows
  CUtensorMap kmap, vmap;
  if (!make_map(&kmap, kc, (uint64_t)B * L, (uint64_t)nh * d, kAtTile) ||
      !make_map(&vmap, vc, (uint64_t)B * L, (uint64_t)nh * d, kAtTile))
    return cudaErrorInvalidValue;
  const dim3 grid(p.nsplit, nh, B);
  if (d == 128)
    return launch_pdl(attn_split_kernel<128>, grid, dim3(kAtThreads), AtSmem<128>::kTotal, s, kmap, vmap, p);
  return launch_pdl(attn_split_kernel<64>, grid, dim3(kAtThreads), AtSmem<64>::kTotal, s, kmap, vmap, p);
}

}  // namespace lsv
