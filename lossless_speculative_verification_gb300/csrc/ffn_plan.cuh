// ffn_plan.cuh -- the work plan of the grouped-expert kernel: the order in
// which expert groups are dealt and the per-group item table, built by one warp
// of whichever kernel finishes the permutation.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace lsv {

// Feature tiles per item.  With token tiles of 256 rows the expert kernel runs
// as CTA pairs (one MMA stream over two SMs, M = 256): an item is then two
// neighbouring feature tiles of one token tile, one per CTA of the pair.
#ifndef LSV_FFN_PAIR
#define LSV_FFN_PAIR 1
#endif
__host__ __device__ constexpr int ffn_fpi(int BN) { return (LSV_FFN_PAIR && BN >= 256) ? 2 : 1; }

// Dealing order of the groups: the shared group (the largest items) first, then
// the routed experts in index order.
__host__ __device__ __forceinline__ int slot_group(int slot, int E, int S) {
  return S > 0 ? (slot == 0 ? E : slot - 1) : slot;
}

// Item table (layout in internal.h), for token tiles of BN rows and
// ffn_fpi(BN) feature tiles per item.  Rows per expert come from the expert
// offsets (compact row space: offsets must partition [0, T*k)) or, when
// `counts` is given, from per-expert row counts of at most T (slot placement).
// Executed by all 32 lanes of one warp.  Inconsistent offsets or counts
// schedule no item and raise LSV_ERR_DEVICE_INDEX.
// rows_out [E] (optional) receives the rows of every routed expert.
__device__ __forceinline__ void build_item_table(const int32_t* offsets, const int32_t* counts, int T, int H, int E,
                                                 int k, int S, int I, int BN, int32_t* table, int* err,
                                                 int32_t* rows_out = nullptr) {
  const int lane = threadIdx.x & 31;
  const int nrows = T * k;
  const int G = E + (S > 0 ? 1 : 0);
  const int fpi = ffn_fpi(BN);
  const int nft_dn = ((H + 127) / 128 + fpi - 1) / fpi;
  const int nft_gu_r = (I / 64 + fpi - 1) / fpi;
  const int nft_gu_s = (S * I / 64 + fpi - 1) / fpi;
  // Slot j*32 + lane is lane's j-th slot.  All rows-per-expert loads are issued first, so that
  // the table costs one round trip to memory.  counts/offsets may live in global or shared
  // memory: plain (generic) loads.
  constexpr int PER = (kMaxExperts + 1 + 31) / 32;  // 9 slots per lane covers G <= 257
  int rows[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int slot = j * 32 + lane;
    const int g = slot < G ? slot_group(slot, E, S) : G;
    rows[j] = 0;
    if (g < E) rows[j] = counts ? counts[g] : offsets[g + 1] - offsets[g];
  }
  if (rows_out) {
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int slot = j * 32 + lane;
      const int g = slot < G ? slot_group(slot, E, S) : G;
      if (g < E) rows_out[g] = rows[j];
    }
  }
  int bad = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int slot = j * 32 + lane;
    const int g = slot < G ? slot_group(slot, E, S) : G;
    if (g < E && (counts ? (rows[j] < 0 || rows[j] > T) : rows[j] < 0)) bad = 1;
  }
  if (!counts && lane == 0 && (offsets[0] != 0 || offsets[E] != nrows)) bad = 1;
  bad = __any_sync(0xffffffffu, bad);
  if (bad && lane == 0) set_error(err, kErrDeviceIndex);
  // items per slot, then exclusive scans in slot order (j-major, lanes within j)
  int gu_carry = 0, dn_carry = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    if (j * 32 > G) break;  // past the end marker (the same for every lane)
    const int slot = j * 32 + lane;
    const int g = slot < G ? slot_group(slot, E, S) : G;
    int ntt = 0, nft_gu = 0;
    if (!bad) {
      if (g < E) {
        ntt = rows[j] > 0 ? (rows[j] + BN - 1) / BN : 0;
        nft_gu = nft_gu_r;
      } else if (g < G) {
        ntt = (T + BN - 1) / BN;
        nft_gu = nft_gu_s;
      }
    }
    const int gu = ntt * nft_gu, dn = ntt * nft_dn;
    int gu_incl = gu, dn_incl = dn;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, gu_incl, o);
      const int b = __shfl_up_sync(0xffffffffu, dn_incl, o);
      if (lane >= o) {
        gu_incl += a;
        dn_incl += b;
      }
    }
    if (slot <= G) {
      table[8 + slot] = gu_carry + gu_incl - gu;
      table[8 + G + 1 + slot] = dn_carry + dn_incl - dn;
    }
    gu_carry += __shfl_sync(0xffffffffu, gu_incl, 31);
    dn_carry += __shfl_sync(0xffffffffu, dn_incl, 31);
  }
  if (lane == 0) {
    table[0] = gu_carry;
    table[1] = dn_carry;
    table[2] = G;
  }
}

}  // namespace lsv
