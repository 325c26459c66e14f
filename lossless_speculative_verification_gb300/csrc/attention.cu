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
// attn_split_kernel: persistent CTAs (as many as fit on the GPU) take work
// items (split, sequence, head) -- up to kAtChunk cached positions of one
// head of one sequence -- from an atomic dealer, split-major so that the
// short last splits come last.
//   warp 4 (producer): deals items (one ahead) and streams their 64-position
//     key and value tiles (the head's d columns of 64 cache rows, 128-byte
//     swizzle) by TMA into a kAtStages ring, without a gap between items; the
//     first tile of an item also carries the item's query rows.  A small
//     record per stage tells the consumers what the stage holds.
//   warps 0-3 (consumers): each takes 16 positions of every tile.  Scores
//     S = q K^T and the weighted values P V run on the tensor cores as
//     m16n8k16 warp MMAs whose 16 rows are the queries (rows >= Q are zero):
//     S stays in registers, the online softmax (running maximum and sum per
//     query, in fp32, exp2 of log2e-scaled scores) turns it into P in the
//     register layout the second MMA takes as its A operand, and the
//     fragments of q and K (ldmatrix) and V (ldmatrix.trans) come from the
//     swizzled tiles without bank conflicts.  At the end of an item the four
//     warps put their states (running maximum, sum, unnormalised output) in
//     the freed stage buffer and merge them into the item's one partial state.
// attn_combine_kernel (programmatic dependent launch): per (sequence, head),
// the splits' states rescaled to their common maximum and summed;
// out = sum / normaliser in bf16.  It also rewinds the dealer.
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lsv {
namespace {

constexpr int kAtConsumers = 4;
constexpr int kAtThreads = 32 * (kAtConsumers + 1);
constexpr int kAtTile = 64;  // positions per ring stage (16 per consumer warp)
#ifndef LSV_ATTN_STAGES
#define LSV_ATTN_STAGES 3
#endif
constexpr int kAtStages = LSV_ATTN_STAGES;
#ifndef LSV_ATTN_CHUNK
#define LSV_ATTN_CHUNK 256
#endif
constexpr int kAtChunk = LSV_ATTN_CHUNK;  // cached positions per item
static_assert(kAtChunk % kAtTile == 0, "an item is a whole number of tiles");
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kAttnCtlInts = 64;  // dealer at [0]; the rest reserved

template <int D>
struct AtSmem {
  static constexpr int kBox = kAtTile * 128;       // 64 columns x 64 rows of bf16
  static constexpr int kQBox = kMaxAttnQ * 128;    // 64 columns x 8 query rows
  static constexpr int kKV = 2 * (D / 64) * kBox;  // key boxes, then value boxes
  static constexpr int kStage = kKV + (D / 64) * kQBox;
  static_assert(kAtConsumers * kMaxAttnQ * (D + 2) * 4 <= kStage, "the warps' states fit in a stage");
  static constexpr int kRing = kAtStages * kStage;
  static constexpr int kMeta = kAtStages * 32;
  static constexpr int kBars = (2 * kAtStages + 1) * 8;
  static constexpr int kTotal = 1024 + kRing + kMeta + kBars + 16;
};

struct AtMeta {
  int b, h, split, i, ntiles, n, end, pad;
};

struct AtParams {
  const int32_t* ctx_len;  // [B]
  int B, Q, L, nh, nsplit;
  int total;       // nsplit * B * nh items
  float qk_scale;  // scale * log2(e)
  float* o_part;   // [B*nh, nsplit, Q, D]
  float* ml_part;  // [B*nh, nsplit, Q, 2]: running maximum (log2 units), sum
  int* dealer;     // zero before the launch; the combine rewinds it
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
                                                                const __grid_constant__ CUtensorMap qmap,
                                                                const AtParams p) {
  using SM = AtSmem<D>;
  constexpr int NB = D / 64;  // boxes per tensor per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile AtMeta* meta = reinterpret_cast<volatile AtMeta*>(smem + SM::kRing);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kRing + SM::kMeta);
  uint64_t* empty = full + kAtStages;
  uint64_t* merge_bar = empty + kAtStages;  // the consumer warps meet here at the end of an item
  volatile int* abort_flag = reinterpret_cast<volatile int*>(merge_bar + 1);
  volatile int* issued_s = abort_flag + 1;
  int* done_s = const_cast<int*>(abort_flag + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kAtConsumers);
    }
    mbar_init(merge_bar, kAtConsumers);
    *abort_flag = 0;
    *issued_s = 0;
    *done_s = 1 << 30;
    fence_barrier_init();
  }
  if (threadIdx.x == 32 * kAtConsumers) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&qmap);
  }
  __syncthreads();
  pdl_wait();  // q, the lengths, the caches and the dealer come from earlier work on the stream
  pdl_trigger();

  if (warp == kAtConsumers) {
    // ------------------------------------------------------------ dealer + TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const int per_split = p.B * p.nh;
      int k = 0;  // tiles (and the end record) put in the ring so far
      bool ok = true;
      int item = atomicAdd(p.dealer, 1);
      while (ok && item < p.total) {
        const int cur = item;
        item = atomicAdd(p.dealer, 1);  // dealt one ahead: its latency hides behind this item's tiles
        const int split = cur / per_split;
        const int bh = cur - split * per_split;
        const int b = bh / p.nh, h = bh - b * p.nh;
        const int n = __ldcg(p.ctx_len + b);  // L2: the lengths may be rewritten between launches
        const int t_begin = split * kAtChunk;
        if (n < p.Q || n > p.L || t_begin >= n) continue;  // nothing to stream (the combine reports bad lengths)
        const int ntiles = (min(n, t_begin + kAtChunk) - t_begin + kAtTile - 1) / kAtTile;
        const int row0 = b * p.L + t_begin;
        for (int i = 0; i < ntiles; ++i, ++k) {
          const int s = k % kAtStages;
          if (!mbar_wait(&empty[s], ((k / kAtStages) & 1) ^ 1u, p.wait_ns)) {
            set_error(p.err, kErrTimeout);
            *abort_flag = 1;
            ok = false;
            break;
          }
          meta[s].b = b;
          meta[s].h = h;
          meta[s].split = split;
          meta[s].i = i;
          meta[s].ntiles = ntiles;
          meta[s].n = n;
          meta[s].end = 0;
          uint8_t* st = smem + s * SM::kStage;
          mbar_arrive_expect_tx(&full[s], SM::kKV + (i == 0 ? NB * SM::kQBox : 0));
#pragma unroll
          for (int c = 0; c < NB; ++c) {
            tma_load_2d(st + c * SM::kBox, &kmap, &full[s], h * D + 64 * c, row0 + i * kAtTile, pol);
            tma_load_2d(st + (NB + c) * SM::kBox, &vmap, &full[s], h * D + 64 * c, row0 + i * kAtTile, pol);
            if (i == 0) tma_load_2d(st + SM::kKV + c * SM::kQBox, &qmap, &full[s], h * D + 64 * c, b * p.Q, pol);
          }
        }
      }
      if (ok) {
        // end record
        const int s = k % kAtStages;
        if (mbar_wait(&empty[s], ((k / kAtStages) & 1) ^ 1u, p.wait_ns)) {
          meta[s].end = 1;
          mbar_arrive(&full[s]);
        } else {
          set_error(p.err, kErrTimeout);
          *abort_flag = 1;
        }
      }
      *issued_s = k;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    const bool row_ok = g < p.Q;
    const int mi = lane >> 3, mr = lane & 7;            // ldmatrix: lane gives row mr of matrix mi
    const int k_row = 16 * warp + 8 * (mi >> 1) + mr;  // S: matrices (n-tile, k half) = (mi>>1, mi&1)
    const int k_half = mi & 1;
    const int v_row = 16 * warp + 8 * (mi & 1) + mr;  // PV: matrices (k half, n-tile) = (mi&1, mi>>1)
    const int v_half = mi >> 1;
    uint32_t qa[D / 16][2];
    float o[D / 8][2];
    float m_run = -INFINITY, l_run = 0.f;
    int lim = -1;
    uint32_t merge_phase = 0;
    // the consumer warps meet at the end of an item (bounded; false: timed out)
    auto meet = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(merge_bar);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(merge_bar, merge_phase, p.wait_ns));
      merge_phase ^= 1u;
      return ok;
    };
    for (int k = 0;; ++k) {
      const int s = k % kAtStages;
      // every lane waits; the warp leaves together if any lane ran out of time
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (k / kAtStages) & 1, p.wait_ns))) {
        if (lane == 0) {
          set_error(p.err, kErrTimeout);
          atomicMin(done_s, k);
        }
        *abort_flag = 1;
        break;
      }
      if (meta[s].end) break;
      const int b = meta[s].b, h = meta[s].h, split = meta[s].split, i = meta[s].i, n = meta[s].n;
      const int ntiles = meta[s].ntiles;
      uint8_t* stage = smem + s * SM::kStage;
      const uint32_t kb = smem_u32(stage);
      const uint32_t vb = kb + NB * SM::kBox;
      if (i == 0) {
        // a new item: its queries as the A operand (row g = query g; k-step ks covers dims [16ks, 16ks+16))
        const uint32_t qb = kb + SM::kKV;
#pragma unroll
        for (int ks = 0; ks < D / 16; ks += 2) {
          // matrices (k-step ks + (mi>>1), k half mi&1), rows = queries 0..7
          const int ch = 2 * ks + mi;
          uint32_t r[4];
          ldmatrix_x4(qb + (ch >> 3) * SM::kQBox + sw128(mr, ch & 7), r);
          qa[ks][0] = row_ok ? r[0] : 0u;
          qa[ks][1] = row_ok ? r[1] : 0u;
          qa[ks + 1][0] = row_ok ? r[2] : 0u;
          qa[ks + 1][1] = row_ok ? r[3] : 0u;
        }
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = 0.f;
        m_run = -INFINITY;
        l_run = 0.f;
        lim = row_ok ? n - p.Q + g : -1;  // last position query g sees
      }
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
      const int pos0 = split * kAtChunk + i * kAtTile + 16 * warp + 2 * t;  // position of sc[0][0]
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
      if (i == ntiles - 1) {
        // the item's last tile: merge the four warps' states through the stage buffer, once
        // every warp is done reading the tile, into the item's one partial state
        float* o_s = reinterpret_cast<float*>(stage);  // [warp][row][D]
        float* ml_s = o_s + kAtConsumers * kMaxAttnQ * D;   // [warp][row][2]
        if (!meet()) {
          if (lane == 0) set_error(p.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        float l = l_run + __shfl_xor_sync(0xffffffffu, l_run, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if (row_ok) {
          float* op = o_s + (warp * kMaxAttnQ + g) * D + 2 * t;
#pragma unroll
          for (int nt = 0; nt < D / 8; ++nt) *reinterpret_cast<float2*>(op + 8 * nt) = make_float2(o[nt][0], o[nt][1]);
          if (t == 0) *reinterpret_cast<float2*>(ml_s + (warp * kMaxAttnQ + g) * 2) = make_float2(m_run, l);
        }
        if (!meet()) {
          if (lane == 0) set_error(p.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        const size_t part = (((size_t)b * p.nh + h) * p.nsplit + split) * p.Q;
        for (int e = threadIdx.x; e < p.Q * (D / 4); e += 32 * kAtConsumers) {
          const int j = e / (D / 4), c4 = e - j * (D / 4);
          float mw[kAtConsumers], mm = -INFINITY;
#pragma unroll
          for (int w = 0; w < kAtConsumers; ++w) {
            mw[w] = ml_s[(w * kMaxAttnQ + j) * 2];
            mm = fmaxf(mm, mw[w]);
          }
          float ls = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w = 0; w < kAtConsumers; ++w) {
            const float f = mw[w] == -INFINITY ? 0.f : exp2f(mw[w] - mm);  // a warp that saw no position adds 0
            const float4 v = *reinterpret_cast<const float4*>(o_s + (w * kMaxAttnQ + j) * D + 4 * c4);
            ls += ml_s[(w * kMaxAttnQ + j) * 2 + 1] * f;
            acc.x = fmaf(v.x, f, acc.x);
            acc.y = fmaf(v.y, f, acc.y);
            acc.z = fmaf(v.z, f, acc.z);
            acc.w = fmaf(v.w, f, acc.w);
          }
          *reinterpret_cast<float4*>(p.o_part + (part + j) * D + 4 * c4) = acc;
          if (c4 == 0) *reinterpret_cast<float2*>(p.ml_part + (part + j) * 2) = make_float2(mm, ls);
        }
        fence_proxy_async_shared();  // the states written here come before the next TMA fill of the stage
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // let the copies already issued land before the CTA's shared memory goes away
    for (int kk = *done_s; kk < *issued_s; ++kk) mbar_wait(&full[kk % kAtStages], (kk / kAtStages) & 1, p.wait_ns);
  }
}

// Per (head, sequence): merge the splits' states and write the output.  Each
// thread takes four output columns of one query and reads every split's state
// of them (independent loads, issued together).
constexpr int kAcThreads = 256;
constexpr int kAcUnroll = 8;

template <int D>
__global__ void __launch_bounds__(kAcThreads) attn_combine_kernel(const float* __restrict__ o_part,
                                                                  const float* __restrict__ ml_part,
                                                                  const int32_t* __restrict__ ctx_len, int Q, int L,
                                                                  int nh, int nsplit, bf16* __restrict__ out,
                                                                  int* dealer, int* err) {
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, b = blockIdx.y;
  if (h == 0 && b == 0 && threadIdx.x == 0) *dealer = 0;  // the split kernel is done with it
  const int n = __ldcg(ctx_len + b);
  const bool bad = n < Q || n > L;
  if (bad && h == 0 && threadIdx.x == 0) set_error(err, kErrDeviceIndex);
  const int nparts = bad ? 0 : (n + kAtChunk - 1) / kAtChunk;
  const size_t base = ((size_t)b * nh + h) * nsplit * Q;  // first state row of (b, h)
  const float2* ml = reinterpret_cast<const float2*>(ml_part) + base;
  const float4* o4 = reinterpret_cast<const float4*>(o_part) + base * (D / 4);
  for (int e = threadIdx.x; e < Q * (D / 4); e += kAcThreads) {
    const int j = e / (D / 4), c4 = e - j * (D / 4);
    float mm = -INFINITY, ls = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < nparts; s0 += kAcUnroll) {
      float2 mlv[kAcUnroll];
      float4 v[kAcUnroll];
#pragma unroll
      for (int u = 0; u < kAcUnroll; ++u) {
        const bool in = s0 + u < nparts;
        mlv[u] = in ? ml[(s0 + u) * Q + j] : make_float2(-INFINITY, 0.f);
        v[u] = in ? o4[((s0 + u) * Q + j) * (D / 4) + c4] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // fold this group into the running (maximum, sum, output)
      float gm = mm;
#pragma unroll
      for (int u = 0; u < kAcUnroll; ++u) gm = fmaxf(gm, mlv[u].x);
      if (gm == -INFINITY) continue;
      const float r = mm == -INFINITY ? 0.f : exp2f(mm - gm);
      ls *= r;
      acc.x *= r;
      acc.y *= r;
      acc.z *= r;
      acc.w *= r;
#pragma unroll
      for (int u = 0; u < kAcUnroll; ++u) {
        const float f = mlv[u].x == -INFINITY ? 0.f : exp2f(mlv[u].x - gm);
        ls = fmaf(mlv[u].y, f, ls);
        acc.x = fmaf(v[u].x, f, acc.x);
        acc.y = fmaf(v[u].y, f, acc.y);
        acc.z = fmaf(v[u].z, f, acc.z);
        acc.w = fmaf(v[u].w, f, acc.w);
      }
      mm = gm;
    }
    const float inv = ls > 0.f ? 1.f / ls : 0.f;
    uint2 pk;
    pk.x = pack_bf16(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(out + (((size_t)b * Q + j) * nh + h) * D + 4 * c4) = pk;
  }
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

template <int D>
cudaError_t launch_attention_d(const bf16* q, const bf16* kc, const bf16* vc, const int32_t* ctx_len, int B, int Q,
                               int L, int nh, float scale, bf16* out, void* ws, const DeviceCtx& dc,
                               cudaStream_t s) {
  static int grid_per_sm[64] = {0};
  static std::mutex mu;
  if (dc.device < 0 || dc.device >= 64) return cudaErrorInvalidDevice;
  std::unique_lock<std::mutex> lk(mu);
  if (!grid_per_sm[dc.device]) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, AtSmem<D>::kTotal);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_split_kernel<D>, kAtThreads, AtSmem<D>::kTotal);
    if (e != cudaSuccess) return e;
    grid_per_sm[dc.device] = per_sm > 0 ? per_sm : 1;
  }
  const int per_sm_cached = grid_per_sm[dc.device];
  lk.unlock();
  AtParams p;
  p.ctx_len = ctx_len;
  p.B = B;
  p.Q = Q;
  p.L = L;
  p.nh = nh;
  p.nsplit = attention_splits(L);
  p.total = p.nsplit * B * nh;
  p.qk_scale = scale * kLog2e;
  const size_t parts = (size_t)B * nh * p.nsplit * Q;
  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  p.dealer = reinterpret_cast<int*>(w);
  p.o_part = reinterpret_cast<float*>(w + round256(kAttnCtlInts * 4));
  p.ml_part = reinterpret_cast<float*>(w + round256(kAttnCtlInts * 4) + round256(parts * D * 4));
  p.err = dc.err;
  p.wait_ns = wait_limit_ns();
  // the caches as [B*L rows, nh*d columns] (a tile: d columns of 64 rows), the queries as
  // [B*Q rows, nh*d columns] (a sequence's queries: d columns of 8 rows from its first)
  CUtensorMap kmap, vmap, qmap;
  if (!make_map(&kmap, kc, (uint64_t)B * L, (uint64_t)nh * D, kAtTile) ||
      !make_map(&vmap, vc, (uint64_t)B * L, (uint64_t)nh * D, kAtTile) ||
      !make_map(&qmap, q, (uint64_t)B * Q, (uint64_t)nh * D, kMaxAttnQ))
    return cudaErrorInvalidValue;
  const long long cap = (long long)per_sm_cached * dc.num_sms;
  const int grid = (int)(p.total < cap ? p.total : cap);
  cudaError_t e = launch_pdl(attn_split_kernel<D>, dim3(grid), dim3(kAtThreads), AtSmem<D>::kTotal, s, kmap, vmap,
                             qmap, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_combine_kernel<D>, dim3(nh, B), dim3(kAcThreads), 0, s, (const float*)p.o_part,
                    (const float*)p.ml_part, ctx_len, Q, L, nh, p.nsplit, out, p.dealer, dc.err);
}

}  // namespace

int attention_splits(int L) { return L <= 0 ? 1 : (L + kAtChunk - 1) / kAtChunk; }

size_t attention_ws_bytes(int B, int Q, int L, int nh, int d) {
  const size_t parts = (size_t)B * nh * attention_splits(L) * Q;
  return round256(kAttnCtlInts * 4) + round256(parts * d * 4) + round256(parts * 2 * 4);
}

cudaError_t launch_attention(const bf16* q, const bf16* kc, const bf16* vc, const int32_t* ctx_len, int B, int Q,
                             int L, int nh, int d, float scale, bf16* out, void* ws, const DeviceCtx& dc,
                             cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  if (d == 128) return launch_attention_d<128>(q, kc, vc, ctx_len, B, Q, L, nh, scale, out, ws, dc, s);
  return launch_attention_d<64>(q, kc, vc, ctx_len, B, Q, L, nh, scale, out, ws, dc, s);
}

}  // namespace lsv
