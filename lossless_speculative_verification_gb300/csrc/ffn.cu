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
//     A = gate row f0, up row f0, gate row f0+1, up row f0+1, ...  (one 3-D TMA box)
//     D[128 x n] in TMEM: lane 2j gate of feature f0+j, lane 2j+1 its up
//     epilogue: act[row, f] = bf16( silu(gate) * up )
//   down item (g, token tile, 128 outputs h0..h0+127):
//     A = W_down rows h0..h0+127, B = act rows;  y[row, h] = D (fp32)
//
// One persistent CTA per SM, warp-specialised: warp 0 issues TMA, warp 1
// allocates TMEM and issues tcgen05.mma (one thread), warps 2-9 drain TMEM,
// warp 10 builds the shared-memory item table once the routing is known.
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
#include <mutex>

#include "ffn_plan.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lsv {
namespace {

constexpr int kFfnThreads = 352;         // 11 warps
constexpr int kEpiWarps = 8;             // warps 2..9: two per TMEM lane quadrant
constexpr int kTabWarp = 10;             // builds the shared-memory item table
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kATileBytes = 128 * 128;   // 128 rows x 64 bf16
constexpr int kEpiBarAll = 1;            // named barrier over all epilogue warps

// Token tiles from which on the producer takes each next item index one item early.
#ifndef LSV_FFN_DEAL_AHEAD_BN
#define LSV_FFN_DEAL_AHEAD_BN 128
#endif

// Pipeline of the CTA-pair kernel (token tiles of 256 rows): stages and K chunks per stage.
#ifndef LSV_FFN_STAGES256P
#define LSV_FFN_STAGES256P 6
#endif
#ifndef LSV_FFN_KCH256P
#define LSV_FFN_KCH256P 1
#endif

// Decode-size pipeline: K chunks (64 wide) per stage and stage count.
#ifndef LSV_FFN_KCH32
#define LSV_FFN_KCH32 2
#endif
#ifndef LSV_FFN_STAGES32
#define LSV_FFN_STAGES32 5
#endif

struct FfnParams {
  int T, H, E, k, S, I, G;
  const int32_t* offsets;  // [E+1] (compact row space)
  const int32_t* seg_counts;  // [E] rows per expert (slot placement), with
  int seg_cap;                // rows reserved per expert (0: compact row space, offsets)
  int rows_routed;            // rows of the routed row space
  int32_t* counts_out;        // slot placement: optional copy of seg_counts
  int BN;                     // token tile (item table)
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
  int* exit_count;         // CTAs finished (with clear_at_end, the last one clears the counters)
  int clear_at_end;
  int32_t* slots_clear;    // slot placement: the per-expert row counters, cleared at the end
  int n_static;            // leading gate/up items of the shared group, decodable without the table
  int deal_ahead;          // take each next item index one item early
};

// Token-row boxes of 16, 32, 64 and 128 rows: an item loads the smallest that holds its rows (at
// most the token tile a CTA stages), so an expert with few rows moves few bytes.
constexpr int kBoxN = 4;
__host__ __device__ constexpr int box_rows(int b) { return 16 << b; }

struct FfnMaps {
  CUtensorMap wgu;             // [E*2I, H]   as {H, 2, E*2I}, box 64 x 2 x 64 (gate/up interleaved)
  CUtensorMap wsgu;            // [2SI, H]    as {H, 2, SI},   box 64 x 2 x 64
  CUtensorMap wd;              // [E*H, I]    box 64 x 128
  CUtensorMap wsd;             // [H, SI]     box 64 x 128
  CUtensorMap xperm[kBoxN];    // [T*k, H]    box 64 x box_rows(b)
  CUtensorMap x[kBoxN];        // [T, H]
  CUtensorMap act[kBoxN];      // [T*k, I]
  CUtensorMap act_sh[kBoxN];   // [T, SI]
};

struct Item {
  int gu;    // 1: gate/up, 0: down
  int slot;  // position of the group in the dealing order
  int g;     // group
  int ft;    // first feature tile (64 features for gate/up, 128 outputs for down); FPI tiles per item
  int nft;   // feature tiles of this kind in the group
  int row0;  // first token row of the tile in the group's row space
  int cnt;   // valid token rows in the tile (1..BN)
  int nk;    // 64-wide K chunks
  int need;  // completions a down item of group g waits for (one per gate/up feature tile)
};

// Shared-memory item table, so that decoding an item costs no global-memory
// round trips: the item table's layout up to its down starts ([0] gate/up
// items, [1] down items, [8, 8+G] gate/up starts per slot, [9+G, 9+2G] down
// starts per slot), then [10+2G, 10+2G+E) first row per expert and
// [10+2G+E, 10+2G+2E) rows per expert.
constexpr int kTabInts = 8 + 2 * (kMaxExperts + 2) + 2 * kMaxExperts;
constexpr int kDealFailed = -2;  // the mailbox wait ran out

// Item `it` of the dealing order.  FPI feature tiles per item (2 for CTA pairs:
// tile ft + rank goes to the CTA of that rank).
template <int BN, int FPI>
__device__ __forceinline__ Item decode_item(int it, const FfnParams& p, const int* tab) {
  if (it < p.n_static) {
    // the shared group's gate/up items come first and their layout is fixed by T alone
    Item m;
    const int nft = p.S * p.I / 64;
    const int nit = (nft + FPI - 1) / FPI;
    const int tt = it / nit;
    m.gu = 1;
    m.slot = 0;
    m.g = p.E;
    m.ft = (it - tt * nit) * FPI;
    m.nft = nft;
    m.row0 = tt * BN;
    m.cnt = min(BN, p.T - tt * BN);
    m.nk = p.H / 64;
    m.need = p.n_static * FPI;
    return m;
  }
  const int G = p.G;
  const int n_gu = tab[0];
  const int* seg_first = tab + 10 + 2 * G;
  const int* seg_rows = seg_first + p.E;
  Item m;
  m.gu = it < n_gu;
  const int* starts = m.gu ? tab + 8 : tab + 9 + G;
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
  m.nft = m.gu ? inter / 64 : (p.H + 127) / 128;
  const int nit = (m.nft + FPI - 1) / FPI;
  const int local = local_it - starts[m.slot];
  const int tt = local / nit;
  m.ft = (local - tt * nit) * FPI;
  int seg0, segn;
  if (routed) {
    seg0 = seg_first[m.g];
    segn = seg_rows[m.g];
  } else {
    seg0 = 0;
    segn = p.T;
  }
  m.row0 = seg0 + tt * BN;
  m.cnt = min(BN, segn - tt * BN);
  m.nk = m.gu ? p.H / 64 : inter / 64;
  m.need = (tab[8 + m.slot + 1] - tab[8 + m.slot]) * FPI;
  return m;
}

// silu(z) = z / (1 + e^-z) with the hardware exponential and the fast divide (the
// result is rounded to bf16; for z below about -88, e^-z overflows and it gives -0).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

template <int BN, int STAGES, int KCH, bool PAIR>
struct Smem {
  static constexpr int kChunkA = kATileBytes;                   // one 64-wide K chunk of A
  static constexpr int kChunkB = (PAIR ? BN / 2 : BN) * 128;    // one 64-wide K chunk of this CTA's B rows
  static constexpr int kStageBytes = KCH * (kChunkA + kChunkB);
  static constexpr int kRing = STAGES * kStageBytes;
  static constexpr int kItemSlots = 4;
  static constexpr int kBars = (2 * STAGES + 6 + 4 * kItemSlots) * 8;
  static constexpr int kTotal = 1024 /*alignment slack*/ + kRing + kBars + 16 + 2 * kItemSlots * 4 +
                                kItemSlots * (int)sizeof(Item) + kTabInts * 4;
  static constexpr int kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                   : (2 * BN <= 256) ? 256 : 512;
};

// PAIR: the kernel runs as clusters of two CTAs.  The even CTA (the leader)
// deals items and passes each index to its peer through a shared-memory
// mailbox; both CTAs stage their own A tile (feature tile ft + rank) and their
// half of the token rows, and count the bytes on the leader's stage barrier.
// The leader issues one M = 256 MMA stream for both (cta_group::2) and its
// commits release the stage and accumulator barriers of both CTAs; each
// CTA's epilogue drains its own TMEM and reports back to the leader.
template <int BN, int STAGES, int KCH, bool PAIR>
__global__ void __launch_bounds__(kFfnThreads, 1) ffn_kernel(const __grid_constant__ FfnMaps maps,
                                                              const FfnParams p) {
  using SM = Smem<BN, STAGES, KCH, PAIR>;
  constexpr int NS = SM::kItemSlots;
  constexpr int FPI = PAIR ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kRing);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* final_bar = tempty + 2;
  uint64_t* item_full = final_bar + 1;
  uint64_t* item_empty = item_full + NS;
  uint64_t* deal_full = item_empty + NS;   // PAIR, peer: an index is in the mailbox
  uint64_t* deal_empty = deal_full + NS;   // PAIR, leader: the peer has taken the index
  uint64_t* tab_ready = deal_empty + NS;   // the table warp has filled `tab`
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tab_ready + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_slot = reinterpret_cast<volatile int*>(tmem_slot + 2);
  volatile int* deal_slot = item_slot + NS;
  Item* item_ring = reinterpret_cast<Item*>(const_cast<int*>(deal_slot + NS));  // decoded items
  int* tab = reinterpret_cast<int*>(item_ring + NS);                             // kTabInts

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], PAIR ? 2 : kEpiThreads);
    }
    for (int q = 0; q < NS; ++q) {
      mbar_init(&item_full[q], 1);
      mbar_init(&item_empty[q], (!PAIR || leader ? 1 : 0) + kEpiThreads);
      mbar_init(&deal_full[q], 1);
      mbar_init(&deal_empty[q], 1);
    }
    mbar_init(final_bar, 1);
    mbar_init(tab_ready, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, SM::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, SM::kTmemCols);
      tmem_relinquish();
    }
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&maps.wgu);
    tma_prefetch_desc(&maps.wd);
    tma_prefetch_desc(&maps.wsgu);
    tma_prefetch_desc(&maps.wsd);
  }
  __syncwarp();
  tc_fence_before_sync();
  if constexpr (PAIR)
    cluster_sync();  // both CTAs' barriers exist before either signals the other
  else
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
      int* counter = p.counter;
      // without early items the preceding kernel (the standalone prep) clears the counters: wait for it
      if (p.n_static == 0) wait_inputs(0);
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      bool have_tab = false;
      int dq = 0;  // mailbox position (PAIR)
      uint32_t dq_phase = 0;
      // An index past the early items needs the routing: wait for the preceding kernels and for
      // the shared-memory item table; -1 past the last item.
      auto resolve = [&](int it) {
        if (it >= p.n_static) {
          wait_inputs(it);
          if (!have_tab) {
            if (!mbar_wait(tab_ready, 0, p.wait_ns)) {
              set_error(p.err, kErrTimeout);
              return -1;
            }
            have_tab = true;
          }
          if (it >= tab[0] + tab[1]) it = -1;
        }
        return it;
      };
      // Next index from the counter; a pair's leader also posts it to the peer's mailbox at once.
      auto deal = [&]() -> int {
        const int raw = atomicAdd(counter, 1);
        if constexpr (PAIR) {
          if (!mbar_wait(&deal_empty[dq], dq_phase ^ 1u, p.wait_ns)) {
            set_error(p.err, kErrTimeout);
            return kDealFailed;
          }
          st_shared_cluster_s32(mapa_shared(smem_u32((const void*)&deal_slot[dq]), 1), raw);
          mbar_arrive_cluster(mapa_shared(smem_u32(&deal_full[dq]), 1));
          if (++dq == NS) {
            dq = 0;
            dq_phase ^= 1u;
          }
        }
        return raw;
      };
      int ahead = -1;  // index taken from the counter one item early (p.deal_ahead)
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
        int it = -1;
        if (!PAIR || leader) {
          const int raw = ahead >= 0 ? ahead : deal();
          ahead = -1;
          if (raw == kDealFailed) {
            ok = false;
            break;
          }
          it = resolve(raw);
        } else if constexpr (PAIR) {
          // the peer takes the leader's indices, in order, from its mailbox
          if (!mbar_wait_cluster(&deal_full[dq], dq_phase, p.wait_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          const int raw = deal_slot[dq];
          mbar_arrive_cluster(mapa_shared(smem_u32(&deal_empty[dq]), 0));
          if (++dq == NS) {
            dq = 0;
            dq_phase ^= 1u;
          }
          it = resolve(raw);
        }
        Item m;
        if (it >= 0) {
          m = decode_item<BN, FPI>(it, p, tab);
          item_ring[slot] = m;
        }
        item_slot[slot] = it;
        mbar_arrive(&item_full[slot]);  // release: the slot writes are visible to the waiters
        if (++slot == NS) {
          slot = 0;
          slot_phase ^= 1u;
        }
        if (it < 0) break;
        // Take the next index now, so that the counter's round trip overlaps this item's loads.
        // A held index never waits on anything (only a gate/up item is held while the current one
        // is a gate/up item, and all gate/up items precede all down items), so every down item's
        // wait still ends.
        if (p.deal_ahead && (!PAIR || leader)) {
          ahead = deal();
          if (ahead == kDealFailed) {
            ok = false;
            break;
          }
        }
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
        // this CTA's feature tile; past the group's last tile (odd count, PAIR) it stages the last
        // one again and its epilogue discards the result
        const int ft = min(m.ft + (int)rank, m.nft - 1);
        // gate/up: the gate rows of 64 features, each staged next to its up row (3-D box);
        // down: 128 output rows
        const int arow0 = m.gu ? (routed ? m.g * 2 * p.I : 0) + ft * 64 : (routed ? m.g * p.H : 0) + ft * 128;
        // PAIR: the MMA takes n/2 token rows from each CTA
        const int n_mma = max(16, (m.cnt + 15) & ~15);
        const int brow0 = m.row0 + (PAIR ? (int)rank * (n_mma / 2) : 0);
        // the smallest token-row box that holds this CTA's rows of the item
        const int rows_cta = PAIR ? n_mma / 2 : n_mma;
        int bx = 0;
        while (bx + 1 < kBoxN && box_rows(bx) < rows_cta && box_rows(bx + 1) <= (PAIR ? BN / 2 : BN)) ++bx;
        const int b_bytes = box_rows(bx) * 128;
        const CUtensorMap* bmap = m.gu ? (routed ? &maps.xperm[bx] : &maps.x[bx])
                                       : (routed ? &maps.act[bx] : &maps.act_sh[bx]);
        for (int kc0 = 0; kc0 < m.nk; kc0 += KCH) {
          const int nch = min(KCH, m.nk - kc0);
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          uint8_t* a_s = smem + stage * SM::kStageBytes;
          uint8_t* b_s = a_s + KCH * SM::kChunkA;
          if constexpr (PAIR) {
            // both CTAs' bytes complete the leader's stage barrier
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * nch * (SM::kChunkA + b_bytes));
            const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
            for (int c = 0; c < nch; ++c) {
              if (m.gu)
                tma_load_3d_pair(a_s + c * SM::kChunkA, amap, fb, (kc0 + c) * 64, 0, arow0, pol_w);
              else
                tma_load_2d_pair(a_s + c * SM::kChunkA, amap, fb, (kc0 + c) * 64, arow0, pol_w);
            }
            for (int c = 0; c < nch; ++c)
              tma_load_2d_pair(b_s + c * SM::kChunkB, bmap, fb, (kc0 + c) * 64, brow0, pol_x);
          } else {
            mbar_arrive_expect_tx(&full[stage], nch * (SM::kChunkA + b_bytes));
            // all K chunks of one weight row block back to back: neighbouring 128-byte pieces of
            // every row reach the memory system together
            for (int c = 0; c < nch; ++c) {
              if (m.gu)
                tma_load_3d(a_s + c * SM::kChunkA, amap, &full[stage], (kc0 + c) * 64, 0, arow0, pol_w);
              else
                tma_load_2d(a_s + c * SM::kChunkA, amap, &full[stage], (kc0 + c) * 64, arow0, pol_w);
            }
            for (int c = 0; c < nch; ++c)
              tma_load_2d(b_s + c * SM::kChunkB, bmap, &full[stage], (kc0 + c) * 64, brow0, pol_x);
          }
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
    // ------------------------------------------------------------ MMA issuer (the leader's, for a pair)
    if (lane == 0 && (!PAIR || leader)) {
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
        const Item m = item_ring[slot];
        mbar_arrive(&item_empty[slot]);
        if (++slot == NS) {
          slot = 0;
          slot_phase ^= 1u;
        }
        if (it < 0 || *abort_flag) break;
        const bool freed = PAIR ? mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, p.wait_ns)
                                : mbar_wait(&tempty[acc], acc_phase ^ 1u, p.wait_ns);
        if (!freed) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int n_mma = max(16, (m.cnt + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(PAIR ? 256 : 128, n_mma);
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
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = sdesc_kmajor_sw128(a_s + c * SM::kChunkA + kk * 32);
              const uint64_t bd = sdesc_kmajor_sw128(b_s + c * SM::kChunkB + kk * 32);
              const uint32_t accum = ((kc0 + c) | kk) ? 1u : 0u;
              if constexpr (PAIR)
                umma_bf16_pair(d_tmem, ad, bd, idesc, accum);
              else
                umma_bf16(d_tmem, ad, bd, idesc, accum);
            }
          }
          if constexpr (PAIR)
            umma_commit_pair_mc(&empty[stage], 0x3);
          else
            umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair_mc(&tfull[acc], 0x3);
        else
          umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // tell the epilogue that no more accumulators come (end marker or abort)
      *abort_flag = ok ? *abort_flag : 1;
      __threadfence_block();
      if (!ok) mbar_arrive(&tfull[acc]);
      // every MMA issued by this thread has completed before TMEM is released
      if constexpr (PAIR)
        umma_commit_pair_mc(final_bar, 0x1);
      else
        umma_commit(final_bar);
      if (!mbar_wait(final_bar, 0, p.wait_ns)) set_error(p.err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp == kTabWarp) {
    // ------------------------------------------------------------ item table
    // As soon as the routing is complete: the shared-memory item table, from the per-expert
    // row counts (slot placement) or from the table and offsets the preceding kernel wrote.
    pdl_wait();
    const int G = p.G;
    int* seg_first = tab + 10 + 2 * G;
    int* seg_rows = seg_first + p.E;
    if (p.seg_cap > 0) {
      build_item_table(nullptr, p.seg_counts, p.T, p.H, p.E, p.k, p.S, p.I, p.BN, tab, p.err, seg_rows);
      __syncwarp();
      for (int e = lane; e < p.E; e += 32) {
        seg_first[e] = e * p.seg_cap;
        if (p.counts_out && blockIdx.x == 0) p.counts_out[e] = seg_rows[e];
      }
    } else {
      if (lane < 2) tab[lane] = p.table[lane];
      for (int i = lane; i <= 2 * G + 1; i += 32) tab[8 + i] = p.table[8 + i];
      for (int e = lane; e < p.E; e += 32) {
        seg_first[e] = p.offsets[e];
        seg_rows[e] = p.offsets[e + 1] - p.offsets[e];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(tab_ready);  // release: the table is visible to the waiter
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    // Warp w may read TMEM lanes 32*(w%4)..+31.  Two warps per quadrant split the
    // accumulator's columns in blocks of EC = 16 (half h takes blocks h, h+2, ...).
    // A gate/up accumulator holds feature j's gate products in lane 2j and its up
    // products in lane 2j+1: the two lanes swap half of each block with one
    // shuffle per column, and each computes SwiGLU on the other half.
    constexpr int EC = 16;
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const bool is_up = lane & 1;
    int acc = 0;
    uint32_t acc_phase = 0;
    int slot = 0;
    uint32_t slot_phase = 0;
    while (true) {
      const bool got_item = mbar_wait(&item_full[slot], slot_phase, p.wait_ns);
      if (!got_item) set_error(p.err, kErrTimeout);
      const int it = got_item ? item_slot[slot] : -1;
      Item m;
      if (it >= 0) m = item_ring[slot];
      mbar_arrive(&item_empty[slot]);
      if (++slot == NS) {
        slot = 0;
        slot_phase ^= 1u;
      }
      // the same decision in all epilogue warps keeps their named barriers matched
      if (named_bar_red_or(kEpiBarAll, kEpiThreads, it < 0)) break;
      wait_inputs(it);
      const bool got = mbar_wait(&tfull[acc], acc_phase, p.wait_ns);
      if (!got) set_error(p.err, kErrTimeout);
      if (named_bar_red_or(kEpiBarAll, kEpiThreads, !got || *abort_flag)) break;
      tc_fence_after_sync();
      const bool routed = m.g < p.E;
      const int nrows_out = routed ? p.rows_routed : p.T;
      const int n_mma = max(16, (m.cnt + 15) & ~15);
      const int ft = m.ft + (int)rank;
      const bool own = ft < m.nft;  // false: the duplicate tile of an odd count (PAIR)
      const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
      if (m.gu) {
        bf16* out = routed ? p.act : p.act_sh;
        const int ld = routed ? p.I : p.S * p.I;
        const int f = ft * 64 + 16 * q + (lane >> 1);
        for (int c0 = EC * half; c0 < n_mma; c0 += 2 * EC) {
          uint32_t r[EC];
          tmem_ld_32x32b_x16(t_row + c0, r);
          tmem_ld_wait();
          // the gate lane takes the block's first EC/2 columns, the up lane the rest
          const int cb = c0 + (is_up ? EC / 2 : 0);
#pragma unroll
          for (int j = 0; j < EC / 2; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, __uint_as_float(is_up ? r[j] : r[EC / 2 + j]), 1);
            const float gv = is_up ? other : __uint_as_float(r[j]);
            const float uv = is_up ? __uint_as_float(r[EC / 2 + j]) : other;
            const int col = cb + j;
            if (own && col < m.cnt && m.row0 + col < nrows_out)
              out[(size_t)(m.row0 + col) * ld + f] = __float2bfloat16_rn(silu(gv) * uv);
          }
        }
      } else {
        void* out = routed ? p.y_perm : p.y_sh;
        const int h = ft * 128 + q * 32 + lane;
        for (int c0 = EC * half; c0 < n_mma; c0 += 2 * EC) {
          uint32_t r[EC];
          tmem_ld_32x32b_x16(t_row + c0, r);
          tmem_ld_wait();
          if (own && h < p.H) {
#pragma unroll
            for (int j = 0; j < EC; ++j) {
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
      if constexpr (PAIR) {
        // one arrival per CTA on the leader's accumulator barrier, after all of this CTA's TMEM reads
        named_bar_sync(kEpiBarAll, kEpiThreads);
        if (threadIdx.x == 64) {
          mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
          if (m.gu) {
            // publish this gate/up tile to the down items of its group
            fence_proxy_async_global();
            __threadfence();
            atomicAdd(&p.done[m.slot], 1);
          }
        }
      } else {
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
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  __syncwarp();
  tc_fence_before_sync();
  if constexpr (PAIR)
    cluster_sync();  // the leader's MMAs into the peer's TMEM and shared memory are complete
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, SM::kTmemCols);
    else
      tmem_dealloc(tmem_base, SM::kTmemCols);
  }
  // Standalone calls: the last CTA to finish sets the counters back to zero for the next call
  // (every other CTA has finished everything that reads or adds to them).  Inside the layer the
  // combine kernel that follows clears them instead, off this kernel's critical path.
  if (p.clear_at_end) {
    __shared__ int s_last;
    if (threadIdx.x == 0) {
      __threadfence();
      s_last = atomicAdd(p.exit_count, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (s_last) {
      for (int g = threadIdx.x; g < p.G; g += blockDim.x) p.done[g] = 0;
      if (p.seg_cap > 0)
        for (int e = threadIdx.x; e < p.E; e += blockDim.x) p.slots_clear[e] = 0;
      if (threadIdx.x == 0) {
        *p.counter = 0;
        *p.exit_count = 0;
      }
    }
  }
}

// Gathers the routed token rows into expert order (x_perm[r] = x[perm[r] / k])
// and builds the tile table from the expert offsets.
template <int BN>
__global__ void __launch_bounds__(256) ffn_prep_kernel(const bf16* __restrict__ x, const int32_t* __restrict__ perm,
                                                       const int32_t* __restrict__ offsets, int T, int H, int E,
                                                       int k, int S, int I, bf16* __restrict__ xperm,
                                                       int32_t* __restrict__ table, int* err,
                                                       int32_t* __restrict__ counters) {
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
  if (blockIdx.x == 0 && threadIdx.x < 32) {
    build_item_table(offsets, nullptr, T, H, E, k, S, I, BN, table, err);
    if (counters) {  // standalone call: clear the expert kernel's counters as well
      const int G = E + (S > 0 ? 1 : 0);
      for (int g = lane; g < G; g += 32) counters[kCntDone + g] = 0;
      if (lane == 0) counters[kCntDeal] = 0;
    }
  }
}

// ----------------------------------------------------------------------------- host side
template <int BN, int STAGES, int KCH, bool PAIR>
cudaError_t run_ffn(const bf16* x, const int32_t* perm, const int32_t* offsets, const int32_t* seg_counts,
                    int seg_cap, const bf16* w_gate_up,
                    const bf16* w_down, const bf16* ws_gate_up, const bf16* ws_down, int T, int H, int E, int k,
                    int S, int I, void* y_perm, void* y_sh, bool y_bf16, uint8_t* ws, const WsLayout& L,
                    const DeviceCtx& dc, cudaStream_t s, bool with_prep, bool early, int32_t* counts_out) {
  using SM = Smem<BN, STAGES, KCH, PAIR>;
  static_assert(SM::kTotal <= 232448, "shared memory budget");
  static_assert(!PAIR || ffn_fpi(BN) == 2, "CTA pairs take two feature tiles per item");
  auto kernel = ffn_kernel<BN, STAGES, KCH, PAIR>;
  static int attr_done[64] = {0};
  static int grid_for[64] = {0};  // PAIR: CTAs of the largest set of co-resident pairs
  static std::mutex mu;
  if (dc.device < 0 || dc.device >= 64) return cudaErrorInvalidDevice;
  std::unique_lock<std::mutex> lk(mu);
  if (!attr_done[dc.device]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kTotal);
    if (e != cudaSuccess) return e;
    grid_for[dc.device] = dc.num_sms;
    if (PAIR) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * ((dc.num_sms + 1) / 2));
      cfg.blockDim = dim3(kFfnThreads);
      cfg.dynamicSmemBytes = SM::kTotal;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
      if (e != cudaSuccess) return e;
      if (clusters < 1) return cudaErrorInvalidConfiguration;
      grid_for[dc.device] = 2 * min(clusters, (dc.num_sms + 1) / 2);
    }
    attr_done[dc.device] = 1;
  }
  const int grid_cached = grid_for[dc.device];
  lk.unlock();
  int32_t* table = reinterpret_cast<int32_t*>(ws + L.table);
  int32_t* counters = reinterpret_cast<int32_t*>(ws + L.counters);
  bf16* xperm = reinterpret_cast<bf16*>(ws + L.xperm);
  bf16* act = reinterpret_cast<bf16*>(ws + L.act);
  bf16* act_sh = reinterpret_cast<bf16*>(ws + L.act_sh);
  const int G = E + (S > 0 ? 1 : 0);
  const int nrows = T * k;
  const int rows_routed = seg_cap > 0 ? E * seg_cap : nrows;

  if (with_prep) {
    const int prep_blocks = max(1, (nrows + 7) / 8);
    const cudaError_t e = launch_pdl(ffn_prep_kernel<BN>, dim3(prep_blocks), dim3(256), 0, s, x, perm, offsets, T,
                                     H, E, k, S, I, xperm, table, dc.err, early ? nullptr : counters);
    if (e != cudaSuccess) return e;
  }

  FfnMaps maps;
  const int SI = S > 0 ? S * I : 64;
  constexpr int BROWS = PAIR ? BN / 2 : BN;  // token rows one CTA stages per K chunk
  const bool ok = make_map_gu(&maps.wgu, w_gate_up, (uint64_t)E * 2 * I, I, H) &&
                  make_map_gu(&maps.wsgu, S > 0 ? ws_gate_up : w_gate_up, S > 0 ? (uint64_t)S * I : 1,
                              S > 0 ? (uint64_t)S * I : 1, H) &&
                  make_map(&maps.wd, w_down, (uint64_t)E * H, I, 128) &&
                  make_map(&maps.wsd, S > 0 ? ws_down : w_down, S > 0 ? (uint64_t)H : 1, S > 0 ? SI : I, 128);
  if (!ok) return cudaErrorInvalidValue;
  for (int b = 0; b < kBoxN; ++b) {
    const uint32_t h = box_rows(b) <= BROWS ? box_rows(b) : BROWS;  // heights past the tile: never chosen
    if (!make_map(&maps.xperm[b], xperm, rows_routed, H, h) || !make_map(&maps.x[b], x, T, H, h) ||
        !make_map(&maps.act[b], act, rows_routed, I, h) ||
        !make_map(&maps.act_sh[b], S > 0 ? (const void*)act_sh : (const void*)act, S > 0 ? T : 1, S > 0 ? SI : I, h))
      return cudaErrorInvalidValue;
  }

  FfnParams p;
  p.T = T; p.H = H; p.E = E; p.k = k; p.S = S; p.I = I; p.G = G;
  p.offsets = offsets;
  p.seg_counts = seg_counts;
  p.seg_cap = seg_cap;
  p.rows_routed = rows_routed;
  p.counts_out = counts_out;
  p.BN = BN;
  p.table = table;
  p.done = counters + kCntDone;
  p.counter = counters + kCntDeal;
  p.exit_count = counters + kCntExit;
  p.clear_at_end = early ? 0 : 1;  // the layer (early items) clears them in its combine
  p.slots_clear = seg_cap > 0 ? const_cast<int32_t*>(seg_counts) : nullptr;
  constexpr int FPI = PAIR ? 2 : 1;
  p.n_static = (early && S > 0) ? ((T + BN - 1) / BN) * ((S * I / 64 + FPI - 1) / FPI) : 0;
  p.act = act;
  p.act_sh = act_sh;
  p.y_perm = y_perm;
  p.y_sh = y_sh;
  p.y_bf16 = y_bf16 ? 1 : 0;
  p.err = dc.err;
  p.wait_ns = wait_limit_ns();
  // With many short items (large token tiles) the counter's round trip at each item boundary
  // would drain the ring; with few long ones, holding an index would lengthen the tail.
  p.deal_ahead = BN >= LSV_FFN_DEAL_AHEAD_BN ? 1 : 0;
  if (!PAIR) return launch_pdl(kernel, dim3(dc.num_sms), dim3(kFfnThreads), SM::kTotal, s, maps, p);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_cached);
  cfg.blockDim = dim3(kFfnThreads);
  cfg.dynamicSmemBytes = SM::kTotal;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, maps, p);
}

}  // namespace

// Token tile: the smallest of 32/64/128/256 that holds the mean rows per expert
// with room for the spread of a multinomial draw.
#ifndef LSV_FFN_MAX_BN
#define LSV_FFN_MAX_BN 256
#endif
#ifndef LSV_FFN_BN32_MAX_MEAN
#define LSV_FFN_BN32_MAX_MEAN 20.0
#endif
#ifndef LSV_FFN_BN64_MAX_MEAN
#define LSV_FFN_BN64_MAX_MEAN 44.0
#endif
#ifndef LSV_FFN_BN128_MAX_MEAN
#define LSV_FFN_BN128_MAX_MEAN 96.0
#endif
int ffn_token_tile(int T, int k, int E) {
  const double mean = E > 0 ? (double)T * k / E : 0.0;
  if (mean <= LSV_FFN_BN32_MAX_MEAN) return 32;
  if (mean <= LSV_FFN_BN64_MAX_MEAN || LSV_FFN_MAX_BN <= 64) return 64;
  if (mean <= LSV_FFN_BN128_MAX_MEAN || LSV_FFN_MAX_BN <= 128) return 128;
  return 256;
}

cudaError_t launch_ffn(const bf16* x, const int32_t* perm, const int32_t* offsets, const int32_t* seg_counts,
                       int seg_cap, const bf16* w_gate_up, const bf16* w_down, const bf16* ws_gate_up,
                       const bf16* ws_down, int T, int H, int E, int k, int S, int I, void* y_perm, void* y_sh,
                       bool y_bf16, uint8_t* ws, const WsLayout& L, const DeviceCtx& dc, cudaStream_t s,
                       bool with_prep, bool early, int32_t* counts_out) {
#define LSV_RUN_FFN(BN_, ST_, KCH_, PAIR_)                                                                     \
  run_ffn<BN_, ST_, KCH_, PAIR_>(x, perm, offsets, seg_counts, seg_cap, w_gate_up, w_down, ws_gate_up, ws_down, \
                                 T, H, E, k, S, I, y_perm, y_sh, y_bf16, ws, L, dc, s, with_prep, early,   \
                                 counts_out)
  switch (ffn_token_tile(T, k, E)) {
    case 32:
      return LSV_RUN_FFN(32, LSV_FFN_STAGES32, LSV_FFN_KCH32, false);
    case 64:
      return LSV_RUN_FFN(64, 4, 2, false);
    case 128:
      return LSV_RUN_FFN(128, 6, 1, false);
    default:
      if constexpr (ffn_fpi(256) == 2)
        return LSV_RUN_FFN(256, LSV_FFN_STAGES256P, LSV_FFN_KCH256P, true);
      else
        return LSV_RUN_FFN(256, 4, 1, false);
  }
#undef LSV_RUN_FFN
}

}  // namespace lsv
