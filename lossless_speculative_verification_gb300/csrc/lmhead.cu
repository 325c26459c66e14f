// lmhead.cu -- the verifier's output layer fused with the greedy-token search.
//
// The verify logits are the verifier's output layer applied to its last hidden
// state of each verified position: logit[r,v] = sum_h hidden[r,h] * W_v[v,h].
// Greedy verification needs only each row's greedy token g[r] (the first index
// attaining the maximum), so the logits are never written out: every tile of
// the product is reduced to (max, first index) per hidden row as it leaves the
// tensor cores, over all the tiles a CTA takes, and the acceptance rule then
// runs on those per-CTA partials
// (kg.zhiyong.dev, "Why FastMTP fits OCR particularly well"; evolve.pub
// review, Section 3.1 / Eq. 2).
//
// Orientation: the MMA's M side is 128 hidden rows (the verified positions) and
// its N side 176 vocabulary rows, so that one TMEM lane holds one position's
// logits of the tile and its thread finds the tile maximum without talking to
// other threads.  Both operands are K-major with the 128-byte swizzle, loaded
// by TMA; the weights stream from HBM once (evict-first), the hidden rows stay
// in L2 (evict-last).  One persistent CTA per SM takes the (row tile,
// vocabulary tile) items round robin: warp 0 issues TMA, warp 1 allocates TMEM
// and issues tcgen05.mma, warps 2-5 scan the accumulators.  Two accumulators
// let the scan of one tile overlap the MMAs of the next.
#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lsv {
namespace {

#ifndef LSV_LH_FIT_ROWS
#define LSV_LH_FIT_ROWS 1
#endif
constexpr int kLhThreads = 192;          // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kLhEpiThreads = 128;
// Vocabulary rows per tile.  Each stage moves the 128 hidden rows' chunk and the weight rows'
// chunk into shared memory, and the hidden part is re-read for every tile; that fill, not HBM,
// bounds the kernel at 128 rows per tile.  176 rows make the weights 58 % of the fill instead of
// 50 %, and 129,280 rows give 735 tiles, 4.8 per SM (5 on most SMs), a smaller tail than 1,010
// tiles of 128 (6.6 per SM).
#ifndef LSV_LH_N
#define LSV_LH_N 176
#endif
constexpr int kLhTile = 128;              // hidden rows per row tile (the MMA's M)
constexpr int kLhN = LSV_LH_N;            // vocabulary rows per tile (the MMA's N: a multiple of 16, <= 256)
constexpr int kLhChunk = kLhTile * 128;   // bytes of one 64-wide K chunk of the hidden rows
constexpr int kLhWChunk = kLhN * 128;     // the same for the weight rows
constexpr int kLhStages = (192 * 1024) / (kLhChunk + kLhWChunk);
constexpr int kLhAccCols = kLhN <= 128 ? 128 : 256;  // TMEM columns between the two accumulators
constexpr int kLhTmemCols = 2 * kLhAccCols;
static_assert(kLhN % 16 == 0 && kLhN >= 16 && kLhN <= 256, "MMA N");
static_assert(kLhWChunk % 1024 == 0, "128-byte swizzle atoms");

struct LhSmem {
  static constexpr int kStage = kLhChunk + kLhWChunk;
  static constexpr int kRing = kLhStages * kStage;
  static constexpr int kBars = (2 * kLhStages + 5) * 8;
  static constexpr int kTotal = 1024 /*alignment slack*/ + kRing + kBars + 16;
};

struct LhParams {
  int R, H, V;
  int ntv;     // vocabulary tiles
  int nitems;  // row tiles x vocabulary tiles
  int nslot;   // partials per row: min(ntv, grid); vocabulary tile tv goes to slot tv % nslot
  int hbytes;       // bytes of one hidden-row chunk of a full row tile (rows of the box x 128)
  int hbytes_last;  // the same for the last row tile
  int wbytes_last;  // bytes of one weight-row chunk of the last vocabulary tile
  float* pv;   // [R, nslot] maxima over a CTA's vocabulary tiles of the row
  int* pi;     // [R, nslot] their first indices
  int* err;
  uint64_t wait_ns;
};

__global__ void __launch_bounds__(kLhThreads, 1) lmhead_argmax_kernel(const __grid_constant__ CUtensorMap hmap,
                                                                      const __grid_constant__ CUtensorMap hmap_last,
                                                                      const __grid_constant__ CUtensorMap wmap,
                                                                      const __grid_constant__ CUtensorMap wmap_last,
                                                                      const LhParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LhSmem::kRing);
  uint64_t* full = bars;
  uint64_t* empty = bars + kLhStages;
  uint64_t* tfull = bars + 2 * kLhStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* final_bar = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLhStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kLhEpiThreads);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kLhTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&hmap);
    tma_prefetch_desc(&hmap_last);
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&wmap_last);
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();
  pdl_wait();  // the hidden rows may come from the preceding kernel
  const int nk = p.H / 64;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int ntr = p.nitems / p.ntv;
      for (int it = blockIdx.x; it < p.nitems && ok; it += gridDim.x) {
        const int tr = it / p.ntv, tv = it - tr * p.ntv;
        const bool last = tr == ntr - 1, last_v = tv == p.ntv - 1;
        const CUtensorMap* hm = last ? &hmap_last : &hmap;
        const CUtensorMap* wm = last_v ? &wmap_last : &wmap;
        const int hb = last ? p.hbytes_last : p.hbytes;
        const int wb = last_v ? p.wbytes_last : kLhWChunk;
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          uint8_t* a_s = smem + stage * LhSmem::kStage;
          uint8_t* b_s = a_s + kLhChunk;
          mbar_arrive_expect_tx(&full[stage], hb + wb);
          tma_load_2d(a_s, hm, &full[stage], kc * 64, tr * kLhTile, pol_x);
          tma_load_2d(b_s, wm, &full[stage], kc * 64, tv * kLhN, pol_w);
          if (++stage == kLhStages) {
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
      const uint32_t idesc = idesc_bf16_f32(kLhTile, kLhN);
      for (int it = blockIdx.x; it < p.nitems && ok; it += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.wait_ns)) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kLhAccCols);
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
          const uint32_t a_s = smem_u32(smem + stage * LhSmem::kStage);
          const uint32_t b_s = a_s + kLhChunk;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d_tmem, sdesc_kmajor_sw128(a_s + kk * 32), sdesc_kmajor_sw128(b_s + kk * 32), idesc,
                      (kc | kk) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == kLhStages) {
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
    // Warp w reads TMEM lanes 32*(w%4)..+31: one hidden row per thread.  The thread scans the
    // columns in increasing vocabulary index with a strict comparison, across all the
    // vocabulary tiles this CTA takes for the row, so that it keeps the first index of their
    // maximum; it writes one (max, index) per row and CTA.
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    float best = -INFINITY;
    int bi = INT_MAX;
    int cur_tr = -1, cur_tv = 0;
    auto flush = [&]() {
      const int row = cur_tr * kLhTile + 32 * q + lane;
      if (cur_tr >= 0 && row < p.R) {
        const size_t at = (size_t)row * p.nslot + cur_tv % p.nslot;
        p.pv[at] = best;
        p.pi[at] = bi;
      }
    };
    bool ok = true;
    for (int it = blockIdx.x; it < p.nitems; it += gridDim.x) {
      const int tr = it / p.ntv, tv = it - tr * p.ntv;
      const bool got = mbar_wait(&tfull[acc], acc_phase, p.wait_ns);
      if (!got) set_error(p.err, kErrTimeout);
      if (named_bar_red_or(1, kLhEpiThreads, !got || *abort_flag)) {
        ok = false;
        break;
      }
      if (tr != cur_tr) {
        flush();
        best = -INFINITY;
        bi = tv * kLhN;  // a row of -inf keeps the first index this CTA saw (0 over the grid)
        cur_tr = tr;
      }
      cur_tv = tv;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * kLhAccCols);
      const int v0 = tv * kLhN;
      const int vn = min(kLhN, p.V - v0);  // columns past the vocabulary hold zero-filled rows
      for (int c0 = 0; c0 < kLhN; c0 += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(t_row + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float v = __uint_as_float(r[j]);
          if (c0 + j < vn && v > best) {
            best = v;
            bi = v0 + c0 + j;
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (ok) flush();
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kLhTmemCols);
  }
}

}  // namespace

size_t lmhead_ws_bytes(int B, int K, int V) {
  const size_t R = (size_t)B * (K + 1);
  const size_t ntv = ((size_t)V + kLhN - 1) / kLhN;
  const size_t one = (R * ntv * 4 + 255) / 256 * 256;
  return R == 0 ? 256 : 2 * one;
}

cudaError_t launch_lmhead_accept(const bf16* hidden, const bf16* w_vocab, const int32_t* drafts, int B, int K,
                                 int V, int H, int32_t* argmax, int32_t* accept_len, int32_t* committed, void* ws,
                                 const DeviceCtx& dc, cudaStream_t s, int argmax_ld) {
  const int R = B * (K + 1);
  if (R == 0) return cudaSuccess;
  const cudaError_t ea =
      ensure_smem_attr(reinterpret_cast<const void*>(lmhead_argmax_kernel), LhSmem::kTotal, dc.device);
  if (ea != cudaSuccess) return ea;
  LhParams p;
  p.R = R;
  p.H = H;
  p.V = V;
  p.ntv = (V + kLhN - 1) / kLhN;
  p.nitems = ((R + kLhTile - 1) / kLhTile) * p.ntv;
  const size_t one = ((size_t)R * p.ntv * 4 + 255) / 256 * 256;
  p.pv = reinterpret_cast<float*>(ws);
  p.pi = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ws) + one);
  p.err = dc.err;
  p.wait_ns = wait_limit_ns();
  // The last row tile stages only the rows it has, rounded up to 16 (a TMA box reaching far past
  // the tensor's end makes every load of it slow: 92 vs 62 us for the whole call at 32 positions).
  // The MMA still reads 128 rows of the A tile; the rows past them hold whatever an earlier stage
  // left, and their results are never written (rows >= R are skipped).
  const int tail = R - (R - 1) / kLhTile * kLhTile;  // rows of the last row tile, 1..128
  const int hrows_last = LSV_LH_FIT_ROWS ? (tail + 15) / 16 * 16 : kLhTile;
  p.hbytes = kLhTile * 128;
  p.hbytes_last = hrows_last * 128;
  // the same for the last vocabulary tile's weight rows
  const int vtail = V - (p.ntv - 1) * kLhN;
  const int wrows_last = LSV_LH_FIT_ROWS ? (vtail + 15) / 16 * 16 : kLhN;
  p.wbytes_last = wrows_last * 128;
  CUtensorMap hmap, hmap_last, wmap, wmap_last;
  if (!make_map(&hmap, hidden, R, H, kLhTile) || !make_map(&hmap_last, hidden, R, H, (uint32_t)hrows_last) ||
      !make_map(&wmap, w_vocab, V, H, kLhN) || !make_map(&wmap_last, w_vocab, V, H, (uint32_t)wrows_last))
    return cudaErrorInvalidValue;
  const int grid = p.nitems < dc.num_sms ? p.nitems : dc.num_sms;
  // a CTA's vocabulary tiles of one row tile are congruent modulo the grid: one slot per CTA
  p.nslot = p.ntv < grid ? p.ntv : grid;
  cudaError_t e =
      launch_pdl(lmhead_argmax_kernel, dim3(grid), dim3(kLhThreads), LhSmem::kTotal, s, hmap, hmap_last, wmap,
                 wmap_last, p);
  if (e != cudaSuccess) return e;
  return launch_accept_finalize(p.pv, p.pi, p.nslot, drafts, B, K, argmax, accept_len, committed, s, argmax_ld);
}

}  // namespace lsv
