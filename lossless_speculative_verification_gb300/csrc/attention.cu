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
// One persistent kernel (as many CTAs as fit on the GPU) does it all.  Work
// comes from two atomic dealers in the workspace:
//   split items (split, sequence, head): up to kAtChunk cached positions of
//     one head of one sequence, dealt split-major so the short last splits
//     come last;
//   merge items (sequence, head), dealt once the split items run out: the
//     merge of that pair's partial states into the output, started when all
//     of them are published (a counter per pair that every writing lane
//     release-adds to).
//   warp 4 (producer): deals items.  A split item's 64-position key and value
//     tiles (the head's d columns of 64 cache rows, 128-byte swizzle) stream
//     by TMA into a kAtStages ring without a gap between items; the first
//     tile of an item also carries the item's query rows.  A merge item goes
//     into the ring as a record once its states are complete.
//   warps 0-3 (consumers): each takes 16 positions of every tile.  Scores
//     S = q K^T and the weighted values P V run on the tensor cores as
//     m16n8k16 warp MMAs whose 16 rows are the queries (rows >= Q are zero):
//     S stays in registers, the online softmax (running maximum and sum per
//     query, in fp32, exp2 of log2e-scaled scores) turns it into P in the
//     register layout the second MMA takes as its A operand, and the
//     fragments of q and K (ldmatrix) and V (ldmatrix.trans) come from the
//     swizzled tiles without bank conflicts.  At the end of a split item each
//     warp writes its state (running maximum, sum, unnormalised output).  On
//     a merge record they rescale the pair's states to their common maximum,
//     sum them and write out = sum / normaliser in bf16.
// The last CTA to leave rewinds the dealers; each merge clears its counter.
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
constexpr int kAtChunk = LSV_ATTN_CHUNK;  // cached positions per split item
static_assert(kAtChunk % kAtTile == 0, "an item is a whole number of tiles");
constexpr float kLog2e = 1.4426950408889634f;
// Control block at the start of the workspace: [0] split dealer, [1] merge dealer,
// [2] CTAs finished, then one published-state counter per (sequence, head).
constexpr int kAttnCtlInts = 64;
constexpr size_t kAttnCtlBytes = ((size_t)kAttnCtlInts + kAttnMaxPairs) * 4;
enum : int { kRecTile = 0, kRecMerge = 1, kRecEnd = 2 };

template <int D>
struct AtSmem {
  static constexpr int kBox = kAtTile * 128;       // 64 columns x 64 rows of bf16
  static constexpr int kQBox = kMaxAttnQ * 128;    // 64 columns x 8 query rows
  static constexpr int kKV = 2 * (D / 64) * kBox;  // key boxes, then value boxes
  static constexpr int kStage = kKV + (D / 64) * kQBox;
  static constexpr int kRing = kAtStages * kStage;
  static constexpr int kMeta = kAtStages * 32;
  static constexpr int kBars = 2 * kAtStages * 8;
  static constexpr int kTotal = 1024 + kRing + kMeta + kBars + 16;
};

struct AtMeta {
  int type, b, h, split, i, ntiles, n, pad;
};

struct AtParams {
  const int32_t* ctx_len;  // [B]
  bf16* out;               // [B, Q, nh, D]
  int B, Q, L, nh, nsplit;
  int total;       // nsplit * B * nh split items
  float qk_scale;  // scale * log2(e)
  float* o_part;   // [B*nh, nsplit, warps, Q, D]
  float* ml_part;  // [B*nh, nsplit, warps, Q, 2]: running maximum (log2 units), sum
  int* ctl;        // control block; zero before the launch, zero after it
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

__device__ __forceinline__ int splits_of(int n) { return (n + kAtChunk - 1) / kAtChunk; }

template <int D>
__global__ void __launch_bounds__(kAtThreads) attn_kernel(const __grid_constant__ CUtensorMap kmap,
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
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kAtStages);
  volatile int* issued_s = abort_flag + 1;
  int* done_s = const_cast<int*>(abort_flag + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* split_dealer = p.ctl;
  int* merge_dealer = p.ctl + 1;
  int* exit_count = p.ctl + 2;
  int* published = p.ctl + kAttnCtlInts;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kAtConsumers);
    }
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
  pdl_wait();  // q, the lengths, the caches and the control block come from earlier work on the stream
  pdl_trigger();

  if (warp == kAtConsumers) {
    // ------------------------------------------------------------ dealer + TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const int per_split = p.B * p.nh;
      int k = 0;  // records put in the ring so far
      bool ok = true;
      // claim the ring slot of record k (false: timed out)
      auto claim = [&](int kk) {
        if (mbar_wait(&empty[kk % kAtStages], ((kk / kAtStages) & 1) ^ 1u, p.wait_ns)) return true;
        set_error(p.err, kErrTimeout);
        *abort_flag = 1;
        return false;
      };
      int item = atomicAdd(split_dealer, 1);
      while (ok && item < p.total) {
        const int cur = item;
        item = atomicAdd(split_dealer, 1);  // dealt one ahead: its latency hides behind this item's tiles
        const int split = cur / per_split;
        const int bh = cur - split * per_split;
        const int b = bh / p.nh, h = bh - b * p.nh;
        const int n = __ldg(p.ctx_len + b);
        const int t_begin = split * kAtChunk;
        if (n < p.Q || n > p.L || t_begin >= n) continue;  // nothing to stream (the merge reports bad lengths)
        const int ntiles = (min(n, t_begin + kAtChunk) - t_begin + kAtTile - 1) / kAtTile;
        const int row0 = b * p.L + t_begin;
        for (int i = 0; i < ntiles; ++i, ++k) {
          if (!(ok = claim(k))) break;
          const int s = k % kAtStages;
          meta[s].type = kRecTile;
          meta[s].b = b;
          meta[s].h = h;
          meta[s].split = split;
          meta[s].i = i;
          meta[s].ntiles = ntiles;
          meta[s].n = n;
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
      // merges, once every split item has been dealt
      int m = ok ? atomicAdd(merge_dealer, 1) : per_split;
      while (ok && m < per_split) {
        const int cur = m;
        m = atomicAdd(merge_dealer, 1);
        const int b = cur / p.nh, h = cur - b * p.nh;
        const int n = __ldg(p.ctx_len + b);
        const bool bad = n < p.Q || n > p.L;
        if (bad && h == 0) set_error(p.err, kErrDeviceIndex);
        // every writing lane of every warp of every split of the pair publishes once
        const int target = bad ? 0 : splits_of(n) * kAtConsumers * 4 * p.Q;
        if (!wait_counter_geq(published + cur, target, p.wait_ns)) {
          set_error(p.err, kErrTimeout);
          *abort_flag = 1;
          ok = false;
          break;
        }
        published[cur] = 0;  // complete: nothing else adds to it in this launch
        if (!(ok = claim(k))) break;
        const int s = k % kAtStages;
        meta[s].type = kRecMerge;
        meta[s].b = b;
        meta[s].h = h;
        meta[s].n = bad ? 0 : n;
        mbar_arrive(&full[s]);
        ++k;
      }
      if (ok && claim(k)) {
        meta[k % kAtStages].type = kRecEnd;
        mbar_arrive(&full[k % kAtStages]);
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
      const int type = meta[s].type;
      if (type == kRecEnd) break;
      const int b = meta[s].b, h = meta[s].h, n = meta[s].n;
      if (type == kRecMerge) {
        // ---------------------------------------------------- merge of (b, h)
        // Every warp finds each query's common maximum and normaliser itself (no
        // barrier between the warps), then sums its share of the output columns.
        const int nparts = n == 0 ? 0 : splits_of(n) * kAtConsumers;
        const size_t base = ((size_t)b * p.nh + h) * p.nsplit * kAtConsumers * p.Q;  // first state row
        const float2* ml = reinterpret_cast<const float2*>(p.ml_part) + base;
        float mmq[kMaxAttnQ], inv_l[kMaxAttnQ];
#pragma unroll
        for (int j = 0; j < kMaxAttnQ; ++j) {
          mmq[j] = -INFINITY;
          inv_l[j] = 0.f;
          if (j >= p.Q) continue;
          float mm = -INFINITY;
          for (int sp = lane; sp < nparts; sp += 32) mm = fmaxf(mm, __ldcg(&ml[sp * p.Q + j].x));
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
          float ls = 0.f;
          if (mm != -INFINITY)
            for (int sp = lane; sp < nparts; sp += 32) {
              const float2 v = __ldcg(&ml[sp * p.Q + j]);
              if (v.x != -INFINITY) ls += v.y * exp2f(v.x - mm);
            }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
          mmq[j] = mm;
          inv_l[j] = ls > 0.f ? 1.f / ls : 0.f;
        }
        const float4* o4 = reinterpret_cast<const float4*>(p.o_part) + base * (D / 4);
        for (int e = threadIdx.x; e < p.Q * (D / 4); e += 32 * kAtConsumers) {
          const int j = e / (D / 4), c4 = e - j * (D / 4);
          float mm = -INFINITY, il = 0.f;
#pragma unroll
          for (int jj = 0; jj < kMaxAttnQ; ++jj)
            if (jj == j) {
              mm = mmq[jj];
              il = inv_l[jj];
            }
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          if (mm != -INFINITY) {
#pragma unroll 4
            for (int sp = 0; sp < nparts; ++sp) {
              const float ms = __ldcg(&ml[sp * p.Q + j].x);
              const float4 v = __ldcg(&o4[(sp * p.Q + j) * (D / 4) + c4]);
              const float f = ms == -INFINITY ? 0.f : exp2f(ms - mm);  // a state that saw no position adds 0
              acc.x = fmaf(v.x, f, acc.x);
              acc.y = fmaf(v.y, f, acc.y);
              acc.z = fmaf(v.z, f, acc.z);
              acc.w = fmaf(v.w, f, acc.w);
            }
          }
          uint2 pk;
          pk.x = pack_bf16(acc.x * il, acc.y * il);
          pk.y = pack_bf16(acc.z * il, acc.w * il);
          *reinterpret_cast<uint2*>(p.out + (((size_t)b * p.Q + j) * p.nh + h) * D + 4 * c4) = pk;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }
      // ------------------------------------------------------ a tile of a split item
      const int split = meta[s].split, i = meta[s].i, ntiles = meta[s].ntiles;
      const uint32_t kb = smem_u32(smem + s * SM::kStage);
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (i == ntiles - 1) {
        // the item's last tile: write this warp's state and publish it
        float l = l_run + __shfl_xor_sync(0xffffffffu, l_run, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const size_t row = ((((size_t)b * p.nh + h) * p.nsplit + split) * kAtConsumers + warp) * p.Q + g;
        if (row_ok) {
          float* op = p.o_part + row * D + 2 * t;
#pragma unroll
          for (int nt = 0; nt < D / 8; ++nt)
            *reinterpret_cast<float2*>(op + 8 * nt) = make_float2(o[nt][0], o[nt][1]);
          if (t == 0) *reinterpret_cast<float2*>(p.ml_part + row * 2) = make_float2(m_run, l);
          red_release_gpu_add(published + b * p.nh + h, 1);
        }
      }
    }
  }
  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      // let the copies already issued land before the CTA's shared memory goes away
      for (int kk = *done_s; kk < *issued_s; ++kk)
        mbar_wait(&full[kk % kAtStages], (kk / kAtStages) & 1, p.wait_ns);
    }
    return;  // the control block needs zeroing again after an error
  }
  if (threadIdx.x == 0 && atomicAdd(exit_count, 1) == (int)gridDim.x - 1) {
    // every CTA is past its dealing: rewind for the next launch
    *split_dealer = 0;
    *merge_dealer = 0;
    *exit_count = 0;
  }
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

template <int D>
cudaError_t launch_attention_d(const bf16* q, const bf16* kc, const bf16* vc, const int32_t* ctx_len, int B, int Q,
                               int L, int nh, float scale, bf16* out, void* ws, const DeviceCtx& dc,
                               cudaStream_t s) {
  static int grid_per_sm[64] = {0};
  if (dc.device < 0 || dc.device >= 64) return cudaErrorInvalidDevice;
  if (!grid_per_sm[dc.device]) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, AtSmem<D>::kTotal);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_kernel<D>, kAtThreads, AtSmem<D>::kTotal);
    if (e != cudaSuccess) return e;
    grid_per_sm[dc.device] = per_sm > 0 ? per_sm : 1;
  }
  AtParams p;
  p.ctx_len = ctx_len;
  p.out = out;
  p.B = B;
  p.Q = Q;
  p.L = L;
  p.nh = nh;
  p.nsplit = attention_splits(L);
  p.total = p.nsplit * B * nh;
  p.qk_scale = scale * kLog2e;
  const size_t parts = (size_t)B * nh * p.nsplit * kAtConsumers * Q;
  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  p.ctl = reinterpret_cast<int*>(w);
  p.o_part = reinterpret_cast<float*>(w + round256(kAttnCtlBytes));
  p.ml_part = reinterpret_cast<float*>(w + round256(kAttnCtlBytes) + round256(parts * D * 4));
  p.err = dc.err;
  p.wait_ns = wait_limit_ns();
  // the caches as [B*L rows, nh*d columns] (a tile: d columns of 64 rows), the queries as
  // [B*Q rows, nh*d columns] (a sequence's queries: d columns of 8 rows from its first)
  CUtensorMap kmap, vmap, qmap;
  if (!make_map(&kmap, kc, (uint64_t)B * L, (uint64_t)nh * D, kAtTile) ||
      !make_map(&vmap, vc, (uint64_t)B * L, (uint64_t)nh * D, kAtTile) ||
      !make_map(&qmap, q, (uint64_t)B * Q, (uint64_t)nh * D, kMaxAttnQ))
    return cudaErrorInvalidValue;
  // every CTA must be resident at once: a merge waits for split items held by other CTAs
  const long long cap = (long long)grid_per_sm[dc.device] * dc.num_sms;
  const long long want = (long long)p.total + (long long)B * nh;
  const int grid = (int)(want < cap ? want : cap);
  return launch_pdl(attn_kernel<D>, dim3(grid), dim3(kAtThreads), AtSmem<D>::kTotal, s, kmap, vmap, qmap, p);
}

}  // namespace

int attention_splits(int L) { return L <= 0 ? 1 : (L + kAtChunk - 1) / kAtChunk; }

size_t attention_ws_bytes(int B, int Q, int L, int nh, int d) {
  const size_t parts = (size_t)B * nh * attention_splits(L) * kAtConsumers * Q;
  return round256(kAttnCtlBytes) + round256(parts * d * 4) + round256(parts * 2 * 4);
}

cudaError_t launch_attention(const bf16* q, const bf16* kc, const bf16* vc, const int32_t* ctx_len, int B, int Q,
                             int L, int nh, int d, float scale, bf16* out, void* ws, const DeviceCtx& dc,
                             cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  if (d == 128) return launch_attention_d<128>(q, kc, vc, ctx_len, B, Q, L, nh, scale, out, ws, dc, s);
  return launch_attention_d<64>(q, kc, vc, ctx_len, B, Q, L, nh, scale, out, ws, dc, s);
}

}  // namespace lsv
