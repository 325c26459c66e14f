// ffn.cu -- grouped SwiGLU experts (routed + shared) on tcgen05 tensor cores.
//
// Expert e:  y = W_down,e ( silu(W_gate,e x) * (W_up,e x) ),  silu(z) = z / (1 + e^-z)
// (DeepSeek-style MoE FFN of the jina-ocr-v1 decoder: 64 routed experts, top-6,
// two shared experts; kg.zhiyong.dev, section "The speed comes from three
// layers working together").
//
// Groups: g < E is routed expert g, fed by its segment of the permuted token
// rows; g == E (when S > 0) is the S shared experts taken together as one
// SwiGLU of intermediate S*I (gate rows and up rows are concatenated in the
// weight layout, and the S down matrices sit side by side), fed by every token.
//
// Orientation ("swap AB"): the MMA's M side is 128 weight rows and its N side
// is up to BN tokens, so one weight tile is streamed from HBM exactly once per
// token tile; at decode sizes (about 12 tokens per expert) every expert's
// weights are read once in total.  Both operands are K-major in shared memory
// with the 128-byte swizzle, loaded by TMA.
//
//   gate/up item (g, token tile, 64 features f0..f0+63):
//     A = [gate rows f0..f0+63 ; up rows f0..f0+63]  (two 64-row TMA boxes)
//     D[128 x n] in TMEM: lanes 0-63 gate, lanes 64-127 up
//     epilogue: act[row, f] = bf16( silu(gate) * up )
//   down item (g, token tile, 128 outputs h0..h0+127):
//     A = W_down rows h0..h0+127, B = act rows;  y[row, h] = D (fp32)
//
// One persistent CTA per SM, warp-specialised: warp 0 issues TMA, warp 1
// allocates TMEM and issues tcgen05.mma (one thread), warps 2-9 drain TMEM.
// A STAGES-deep shared-memory ring (KCH K-chunks per stage, so that the
// neighbouring 128-byte pieces of each weight row are requested together)
// decouples loads from MMAs, and two TMEM accumulators decouple MMAs from the
// epilogue.  Items are dealt dynamically: the producer takes the next index
// from a global counter and passes it to the MMA and epilogue warps through a
// small shared-memory ring.  Every gate/up item precedes every down item in
// the global order, and a down item waits (bounded) on a per-group counter of
// finished gate/up items; the wait always ends, because every gate/up item of
// that group was dealt earlier to a running CTA whose progress on it depends
// on nothing else.
#include "ffn_plan.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lsv {
namespace {

constexpr int kFfnThreads = 320;         // 10 warps
constexpr int kEpiWarps = 8;             // warps 2..9: two per TMEM lane quadrant
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kATileBytes = 128 * 128;   // 128 rows x 64 bf16
constexpr int kXchStride = 9;            // padded 8-value row of the gate/up exchange buffer
constexpr int kXchPair = 2 * 32 * kXchStride;  // floats per (pair, buffer): gate->up and up->gate halves
constexpr int kEpiBarAll = 5;            // named barrier over all epilogue warps (ids 1..4: warp pairs)

// Decode-size pipeline: K chunks (64 wide) per stage and stage count.
#ifndef LSV_FFN_KCH32
#define LSV_FFN_KCH32 2
#endif
#ifndef LSV_FFN_STAGES32
#define LSV_FFN_STAGES32 5
#endif

struct FfnParams {
  int T, H, E, k, S, I, G;
  const int32_t* offsets;  // [E+1]
  const int32_t* table;    // tile table (see internal.h)
  int* done;               // [G]
  bf16* act;               // [T*k, I]
  bf16* act_sh;            // [T, S*I]
  void* y_perm;            // [T*k, H] fp32, or bf16 when y_bf16
  void* y_sh;              // [T, H]   fp32, or bf16 when y_bf16
  int y_bf16;
  int* err;
  uint64_t wait_ns;
  int* counter;            // next item to deal
  int n_static;            // leading gate/up items of the shared group, decodable without the table
};

struct FfnMaps {
  CUtensorMap wgu;     // [E*2I, H]   box 64 x 64
  CUtensorMap wsgu;    // [2SI, H]    box 64 x 64
  CUtensorMap wd;      // [E*H, I]    box 64 x 128
  CUtensorMap wsd;     // [H, SI]     box 64 x 128
  CUtensorMap xperm;   // [T*k, H]    box 64 x BN
  CUtensorMap x;       // [T, H]      box 64 x BN
  CUtensorMap act;     // [T*k, I]    box 64 x BN
  CUtensorMap act_sh;  // [T, SI]     box 64 x BN
};

struct Item {
  int gu;    // 1: gate/up, 0: down
  int slot;  // position of the group in the dealing order
  int g;     // group
  int ft;    // feature tile (64 features for gate/up, 128 outputs for down)
  int row0;  // first token row of the tile in the group's row space
  int cnt;   // valid token rows in the tile (1..BN)
  int nk;    // 64-wide K chunks
  int need;  // gate/up items of group g (for a down item's dependency)
};

template <int BN>
__device__ __forceinline__ Item decode_item(int it, const FfnParams& p) {
  if (it < p.n_static) {
    // the shared group's gate/up items come first and their layout is fixed by T alone
    Item m;
    const int nft = p.S * p.I / 64;
    const int tt = it / nft;
    m.gu = 1;
    m.slot = 0;
    m.g = p.E;
    m.ft = it - tt * nft;
    m.row0 = tt * BN;
    m.cnt = min(BN, p.T - tt * BN);
    m.nk = p.H / 64;
    m.need = p.n_static;
    return m;
  }
  const int* tb = p.table;
  const int G = p.G;
  const int n_gu = tb[0];
  Item m;
  m.gu = it < n_gu;
  const int* starts = m.gu ? tb + 8 : tb + 8 + G + 1;
  const int local_it = m.gu ? it : it - n_gu;
  int lo = 0, hi = G - 1;  // largest g with starts[g] <= local_it
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (starts[mid] <= local_it) lo = mid; else hi = mid - 1;
  }
  m.slot = lo;
  m.g = slot_group(lo, p.E, p.S);
  const bool routed = m.g < p.E;
  const int inter = routed ? p.I : p.S * p.I;
  const int nft = m.gu ? inter / 64 : (p.H + 127) / 128;
  const int local = local_it - starts[m.slot];
  const int tt = local / nft;
  m.ft = local - tt * nft;
  int seg0, segn;
  if (routed) {
    seg0 = p.offsets[m.g];
    segn = p.offsets[m.g + 1] - seg0;
  } else {
    seg0 = 0;
    segn = p.T;
  }
  m.row0 = seg0 + tt * BN;
  m.cnt = min(BN, segn - tt * BN);
  m.nk = m.gu ? p.H / 64 : inter / 64;
  m.need = tb[8 + m.slot + 1] - tb[8 + m.slot];
  return m;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

template <int BN, int STAGES, int KCH>
struct Smem {
  static constexpr int kChunkA = kATileBytes;               // one 64-wide K chunk of A
  static constexpr int kChunkB = BN * 128;                  // one 64-wide K chunk of B
  static constexpr int kStageBytes = KCH * (kChunkA + kChunkB);
  static constexpr int kRing = STAGES * kStageBytes;
  static constexpr int kXch = 4 /*pairs*/ * 2 /*buffers*/ * kXchPair * 4;
  static constexpr int kItemSlots = 4;
  static constexpr int kBars = (2 * STAGES + 5 + 2 * kItemSlots) * 8;
  static constexpr int kTotal = 1024 /*alignment slack*/ + kRing + kXch + kBars + 16 + kItemSlots * 4;
  static constexpr int kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                   : (2 * BN <= 256) ? 256 : 512;
};

template <int BN, int STAGES, int KCH>
__global__ void __launch_bounds__(kFfnThreads, 1) ffn_kernel(const __grid_constant__ FfnMaps maps,
                                                              const FfnParams p) {
  using SM = Smem<BN, STAGES, KCH>;
  constexpr int NS = SM::kItemSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xch = reinterpret_cast<float*>(smem + SM::kRing);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kRing + SM::kXch);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* final_bar = tempty + 2;
  uint64_t* item_full = final_bar + 1;
  uint64_t* item_empty = item_full + NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(item_empty + NS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiThreads);
    }
    for (int q = 0; q < NS; ++q) {
      mbar_init(&item_full[q], 1);
      mbar_init(&item_empty[q], 1 + kEpiThreads);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, SM::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&maps.wgu);
    tma_prefetch_desc(&maps.wd);
    tma_prefetch_desc(&maps.wsgu);
    tma_prefetch_desc(&maps.wsd);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // The prologue above overlaps the previous kernels.  Items below n_static need
  // nothing they produce; every thread waits for them (griddepcontrol.wait)
  // before its first other item.
  pdl_trigger();
  bool waited = false;
  auto wait_inputs = [&](int it) {
    if (!waited && it >= p.n_static) {
      pdl_wait();
      waited = true;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer + item dealer
    if (lane == 0) {
      int n_items = -1;
      int* counter = p.counter;
      // without early items the counters are zeroed by the preceding kernel: wait for it first
      if (p.n_static == 0) wait_inputs(0);
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t slot_phase = 0;
      bool ok = true;
      while (ok) {
        if (!mbar_wait(&item_empty[slot], slot_phase ^ 1u, p.wait_ns)) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        int it = atomicAdd(counter, 1);
        if (it >= p.n_static) {
          wait_inputs(it);
          if (n_items < 0) n_items = p.table[0] + p.table[1];
          if (it >= n_items) it = -1;
        }
        item_slot[slot] = it;
        mbar_arrive(&item_full[slot]);  // release: the slot write is visible to the waiters
        if (++slot == NS) {
          slot = 0;
          slot_phase ^= 1u;
        }
        if (it < 0) break;
        const Item m = decode_item<BN>(it, p);
        const bool routed = m.g < p.E;
        if (!m.gu) {
          if (!wait_counter_geq(&p.done[m.slot], m.need, p.wait_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        const CUtensorMap* amap = m.gu ? (routed ? &maps.wgu : &maps.wsgu) : (routed ? &maps.wd : &maps.wsd);
        const CUtensorMap* bmap = m.gu ? (routed ? &maps.xperm : &maps.x) : (routed ? &maps.act : &maps.act_sh);
        int arow0, arow1 = 0;
        if (m.gu) {
          const int inter = routed ? p.I : p.S * p.I;
          const int gbase = routed ? m.g * 2 * p.I : 0;
          arow0 = gbase + m.ft * 64;
          arow1 = gbase + inter + m.ft * 64;
        } else {
          arow0 = (routed ? m.g * p.H : 0) + m.ft * 128;
        }
        for (int kc0 = 0; kc0 < m.nk; kc0 += KCH) {
          const int nch = min(KCH, m.nk - kc0);
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          uint8_t* a_s = smem + stage * SM::kStageBytes;
          uint8_t* b_s = a_s + KCH * SM::kChunkA;
          mbar_arrive_expect_tx(&full[stage], nch * (SM::kChunkA + SM::kChunkB));
          // all K chunks of one weight row block back to back: neighbouring 128-byte pieces of
          // every row reach the memory system together
          for (int c = 0; c < nch; ++c)
            tma_load_2d(a_s + c * SM::kChunkA, amap, &full[stage], (kc0 + c) * 64, arow0, pol_w);
          if (m.gu)
            for (int c = 0; c < nch; ++c)
              tma_load_2d(a_s + c * SM::kChunkA + kATileBytes / 2, amap, &full[stage], (kc0 + c) * 64, arow1,
                          pol_w);
          for (int c = 0; c < nch; ++c)
            tma_load_2d(b_s + c * SM::kChunkB, bmap, &full[stage], (kc0 + c) * 64, m.row0, pol_x);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        __threadfence_block();
        mbar_arrive(&full[stage]);  // wake the MMA issuer so that it sees the abort
        // and hand out an end marker in case the consumers wait for an item
        item_slot[slot] = -1;
        mbar_arrive(&item_full[slot]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int slot = 0;
      uint32_t slot_phase = 0;
      bool ok = true;
      while (ok) {
        if (!mbar_wait(&item_full[slot], slot_phase, p.wait_ns)) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        const int it = item_slot[slot];
        mbar_arrive(&item_empty[slot]);
        if (++slot == NS) {
          slot = 0;
          slot_phase ^= 1u;
        }
        if (it < 0 || *abort_flag) break;
        wait_inputs(it);
        const Item m = decode_item<BN>(it, p);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.wait_ns)) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int n_mma = max(16, (m.cnt + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(128, n_mma);
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kc0 = 0; kc0 < m.nk; kc0 += KCH) {
          const int nch = min(KCH, m.nk - kc0);
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
          const uint32_t a_s = smem_u32(smem + stage * SM::kStageBytes);
          const uint32_t b_s = a_s + KCH * SM::kChunkA;
          for (int c = 0; c < nch; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(d_tmem, sdesc_kmajor_sw128(a_s + c * SM::kChunkA + kk * 32),
                        sdesc_kmajor_sw128(b_s + c * SM::kChunkB + kk * 32), idesc,
                        ((kc0 + c) | kk) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // tell the epilogue that no more accumulators come (end marker or abort)
      *abort_flag = ok ? *abort_flag : 1;
      __threadfence_block();
      if (!ok) mbar_arrive(&tfull[acc]);
      // every MMA issued by this thread has completed before TMEM is released
      umma_commit(final_bar);
      if (!mbar_wait(final_bar, 0, p.wait_ns)) set_error(p.err, kErrTimeout);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    // Warp w may read TMEM lanes 32*(w%4)..+31.  Two warps per quadrant split the
    // 16-column chunks of an accumulator (half h takes chunks h, h+2, ...).  For
    // gate/up items the warp holding gate rows (quadrant 0/1) and the one holding
    // the matching up rows (quadrant 2/3) swap half of each chunk through shared
    // memory, so that both compute SwiGLU on eight columns.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int pair = (q & 1) + 2 * half;     // gate/up warp pair, named barrier 1 + pair
    const bool is_gate = q < 2;
    float* xpair = xch + pair * 2 * kXchPair;
    int acc = 0;
    uint32_t acc_phase = 0;
    int slot = 0;
    uint32_t slot_phase = 0;
    int nx = 0;  // chunks exchanged so far (selects the buffer)
    while (true) {
      const bool got_item = mbar_wait(&item_full[slot], slot_phase, p.wait_ns);
      if (!got_item) set_error(p.err, kErrTimeout);
      const int it = got_item ? item_slot[slot] : -1;
      mbar_arrive(&item_empty[slot]);
      if (++slot == NS) {
        slot = 0;
        slot_phase ^= 1u;
      }
      // the same decision in all epilogue warps keeps their named barriers matched
      if (named_bar_red_or(kEpiBarAll, kEpiThreads, it < 0)) break;
      wait_inputs(it);
      const Item m = decode_item<BN>(it, p);
      const bool got = mbar_wait(&tfull[acc], acc_phase, p.wait_ns);
      if (!got) set_error(p.err, kErrTimeout);
      if (named_bar_red_or(kEpiBarAll, kEpiThreads, !got || *abort_flag)) break;
      tc_fence_after_sync();
      const bool routed = m.g < p.E;
      const int nrows_out = routed ? p.T * p.k : p.T;
      const int n_mma = max(16, (m.cnt + 15) & ~15);
      const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
      if (m.gu) {
        bf16* out = routed ? p.act : p.act_sh;
        const int ld = routed ? p.I : p.S * p.I;
        const int f = m.ft * 64 + (q & 1) * 32 + lane;
        for (int c0 = 16 * half; c0 < n_mma; c0 += 32) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(t_row + c0, r);
          tmem_ld_wait();
          float* buf = xpair + (nx & 1) * kXchPair;
          float* g2u = buf + lane * kXchStride;                 // gate values of columns 8..15
          float* u2g = buf + (32 + lane) * kXchStride;          // up values of columns 0..7
          if (is_gate) {
#pragma unroll
            for (int j = 0; j < 8; ++j) g2u[j] = __uint_as_float(r[8 + j]);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) u2g[j] = __uint_as_float(r[j]);
          }
          named_bar_sync(1 + pair, 64);
          const int jb = is_gate ? 0 : 8;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int col = c0 + jb + j;
            const float gv = is_gate ? __uint_as_float(r[j]) : g2u[j];
            const float uv = is_gate ? u2g[j] : __uint_as_float(r[8 + j]);
            if (col < m.cnt && m.row0 + col < nrows_out)
              out[(size_t)(m.row0 + col) * ld + f] = __float2bfloat16_rn(silu(gv) * uv);
          }
          ++nx;
        }
      } else {
        void* out = routed ? p.y_perm : p.y_sh;
        const int h = m.ft * 128 + q * 32 + lane;
        for (int c0 = 16 * half; c0 < n_mma; c0 += 32) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(t_row + c0, r);
          tmem_ld_wait();
          if (h < p.H) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = c0 + j;
              if (col < m.cnt && m.row0 + col < nrows_out) {
                const size_t o = (size_t)(m.row0 + col) * p.H + h;
                if (p.y_bf16)
                  static_cast<bf16*>(out)[o] = __float2bfloat16_rn(__uint_as_float(r[j]));
                else
                  static_cast<float*>(out)[o] = __uint_as_float(r[j]);
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&tempty[acc]);
      if (m.gu) {
        // publish this gate/up item to the down items of its group
        named_bar_sync(kEpiBarAll, kEpiThreads);
        if (threadIdx.x == 64) {
          fence_proxy_async_global();
          __threadfence();
          atomicAdd(&p.done[m.slot], 1);
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, SM::kTmemCols);
  }
}

// Gathers the routed token rows into expert order (x_perm[r] = x[perm[r] / k])
// and builds the tile table from the expert offsets.
template <int BN>
__global__ void __launch_bounds__(256) ffn_prep_kernel(const bf16* __restrict__ x, const int32_t* __restrict__ perm,
                                                       const int32_t* __restrict__ offsets, int T, int H, int E,
                                                       int k, int S, int I, bf16* __restrict__ xperm,
                                                       int32_t* __restrict__ table, int* err, bool zero_counters) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int nrows = T * k;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row < nrows) {
    const int src = perm[row];
    if (src < 0 || src >= nrows) {
      set_error(err, kErrDeviceIndex);
    } else {
      const uint4* s = reinterpret_cast<const uint4*>(x + (size_t)(src / k) * H);
      uint4* d = reinterpret_cast<uint4*>(xperm + (size_t)row * H);
      // all loads of a stretch first, then the stores: every lane keeps 8 pieces in flight
      for (int c0 = lane; c0 < H / 8; c0 += 8 * 32) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (c0 + 32 * u < H / 8) v[u] = __ldg(s + c0 + 32 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (c0 + 32 * u < H / 8) d[c0 + 32 * u] = v[u];
      }
    }
  }
  if (blockIdx.x == 0 && threadIdx.x < 32) build_item_table(offsets, T, H, E, k, S, I, BN, table, err, zero_counters);
}

// ----------------------------------------------------------------------------- host side
template <int BN, int STAGES, int KCH>
cudaError_t run_ffn(const bf16* x, const int32_t* perm, const int32_t* offsets, const bf16* w_gate_up,
                    const bf16* w_down, const bf16* ws_gate_up, const bf16* ws_down, int T, int H, int E, int k,
                    int S, int I, void* y_perm, void* y_sh, bool y_bf16, uint8_t* ws, const WsLayout& L,
                    const DeviceCtx& dc, cudaStream_t s, bool with_prep, bool early) {
  using SM = Smem<BN, STAGES, KCH>;
  static_assert(SM::kTotal <= 232448, "shared memory budget");
  static int attr_done[64] = {0};
  if (dc.device >= 0 && dc.device < 64 && !attr_done[dc.device]) {
    cudaError_t e = cudaFuncSetAttribute(ffn_kernel<BN, STAGES, KCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SM::kTotal);
    if (e != cudaSuccess) return e;
    attr_done[dc.device] = 1;
  }
  int32_t* table = reinterpret_cast<int32_t*>(ws + L.table);
  bf16* xperm = reinterpret_cast<bf16*>(ws + L.xperm);
  bf16* act = reinterpret_cast<bf16*>(ws + L.act);
  bf16* act_sh = reinterpret_cast<bf16*>(ws + L.act_sh);
  const int G = E + (S > 0 ? 1 : 0);
  const int nrows = T * k;

  if (with_prep) {
    const int prep_blocks = max(1, (nrows + 7) / 8);
    const cudaError_t e = launch_pdl(ffn_prep_kernel<BN>, dim3(prep_blocks), dim3(256), 0, s, x, perm, offsets, T,
                                     H, E, k, S, I, xperm, table, dc.err, /*zero_counters=*/!early);
    if (e != cudaSuccess) return e;
  }

  FfnMaps maps;
  const int SI = S > 0 ? S * I : 64;
  const bool ok = make_map(&maps.wgu, w_gate_up, (uint64_t)E * 2 * I, H, 64) &&
                  make_map(&maps.wsgu, S > 0 ? ws_gate_up : w_gate_up, S > 0 ? (uint64_t)2 * S * I : 1, H, 64) &&
                  make_map(&maps.wd, w_down, (uint64_t)E * H, I, 128) &&
                  make_map(&maps.wsd, S > 0 ? ws_down : w_down, S > 0 ? (uint64_t)H : 1, S > 0 ? SI : I, 128) &&
                  make_map(&maps.xperm, xperm, nrows, H, BN) && make_map(&maps.x, x, T, H, BN) &&
                  make_map(&maps.act, act, nrows, I, BN) &&
                  make_map(&maps.act_sh, S > 0 ? (const void*)act_sh : (const void*)act, S > 0 ? T : 1,
                           S > 0 ? SI : I, BN);
  if (!ok) return cudaErrorInvalidValue;

  FfnParams p;
  p.T = T; p.H = H; p.E = E; p.k = k; p.S = S; p.I = I; p.G = G;
  p.offsets = offsets;
  p.table = table;
  p.done = table + table_counters(G);
  p.counter = table + table_counters(G) + G;
  p.n_static = (early && S > 0) ? ((T + BN - 1) / BN) * (S * I / 64) : 0;
  p.act = act;
  p.act_sh = act_sh;
  p.y_perm = y_perm;
  p.y_sh = y_sh;
  p.y_bf16 = y_bf16 ? 1 : 0;
  p.err = dc.err;
  p.wait_ns = wait_limit_ns();
  return launch_pdl(ffn_kernel<BN, STAGES, KCH>, dim3(dc.num_sms), dim3(kFfnThreads), SM::kTotal, s, maps, p);
}

}  // namespace

// Token tile: the smallest of 32/64/128/256 that holds the mean rows per expert
// with room for the spread of a multinomial draw.
int ffn_token_tile(int T, int k, int E) {
  const double mean = E > 0 ? (double)T * k / E : 0.0;
  if (mean <= 20.0) return 32;
  if (mean <= 44.0) return 64;
  if (mean <= 96.0) return 128;
  return 256;
}

cudaError_t launch_ffn(const bf16* x, const int32_t* perm, const int32_t* offsets, const bf16* w_gate_up,
                       const bf16* w_down, const bf16* ws_gate_up, const bf16* ws_down, int T, int H, int E,
                       int k, int S, int I, void* y_perm, void* y_sh, bool y_bf16, uint8_t* ws,
                       const WsLayout& L, const DeviceCtx& dc, cudaStream_t s, bool with_prep, bool early) {
  switch (ffn_token_tile(T, k, E)) {
    case 32:
      return run_ffn<32, LSV_FFN_STAGES32, LSV_FFN_KCH32>(x, perm, offsets, w_gate_up, w_down, ws_gate_up, ws_down,
                                                          T, H, E, k, S, I, y_perm, y_sh, y_bf16, ws, L, dc, s, with_prep, early);
    case 64:
      return run_ffn<64, 4, 2>(x, perm, offsets, w_gate_up, w_down, ws_gate_up, ws_down, T, H, E, k, S, I, y_perm,
                               y_sh, y_bf16, ws, L, dc, s, with_prep, early);
    case 128:
      return run_ffn<128, 6, 1>(x, perm, offsets, w_gate_up, w_down, ws_gate_up, ws_down, T, H, E, k, S, I, y_perm,
                                y_sh, y_bf16, ws, L, dc, s, with_prep, early);
    default:
      return run_ffn<256, 4, 1>(x, perm, offsets, w_gate_up, w_down, ws_gate_up, ws_down, T, H, E, k, S, I, y_perm,
                                y_sh, y_bf16, ws, L, dc, s, with_prep, early);
  }
}

}  // namespace lsv
