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
__device__ __forceinline__ void build_item_table(const int32_t* offsets, const int32_t* counts, int T, int H, int E,
                                                 int k, int S, int I, int BN, int32_t* table, int* err) {
  const int lane = threadIdx.x & 31;
  const int nrows = T * k;
  const int G = E + (S > 0 ? 1 : 0);
  const int fpi = ffn_fpi(BN);
  const int nft_dn = ((H + 127) / 128 + fpi - 1) / fpi;
  constexpr int PER = (kMaxExperts + 1 + 31) / 32;  // 9 slots per lane covers G <= 257
  int gu_loc[PER], dn_loc[PER];
  int gu_sum = 0, dn_sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int slot = lane * PER + j;
    const int g = slot < G ? slot_group(slot, E, S) : G;
    int ntt = 0, nft_gu = 0;
    if (g < E) {
      const int c = counts ? counts[g] : offsets[g + 1] - offsets[g];
      ntt = c > 0 ? (c + BN - 1) / BN : 0;
      nft_gu = (I / 64 + fpi - 1) / fpi;
    } else if (g < G) {
      ntt = (T + BN - 1) / BN;
      nft_gu = (S * I / 64 + fpi - 1) / fpi;
    }
    gu_loc[j] = ntt * nft_gu;
    dn_loc[j] = ntt * nft_dn;
    gu_sum += gu_loc[j];
    dn_sum += dn_loc[j];
  }
  int bad = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int g = lane * PER + j;
    if (g < E && (counts ? (counts[g] < 0 || counts[g] > T) : offsets[g] > offsets[g + 1])) bad = 1;
  }
  if (!counts && lane == 0 && (offsets[0] != 0 || offsets[E] != nrows)) bad = 1;
  bad = __any_sync(0xffffffffu, bad);
  if (bad) {
    gu_sum = dn_sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) gu_loc[j] = dn_loc[j] = 0;
    if (lane == 0) set_error(err, kErrDeviceIndex);
  }
  int gu_incl = gu_sum, dn_incl = dn_sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, gu_incl, o);
    const int b = __shfl_up_sync(0xffffffffu, dn_incl, o);
    if (lane >= o) {
      gu_incl += a;
      dn_incl += b;
    }
  }
  int gu_run = gu_incl - gu_sum, dn_run = dn_incl - dn_sum;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int slot = lane * PER + j;
    if (slot <= G) {
      table[8 + slot] = gu_run;
      table[8 + G + 1 + slot] = dn_run;
    }
    gu_run += gu_loc[j];
    dn_run += dn_loc[j];
  }
  if (lane == 31) {
    table[0] = gu_incl;
    table[1] = dn_incl;
    table[2] = G;
  }
}

}  // namespace lsv
