// permute.cu -- expert histogram, exclusive scan and stable permutation of the
// (token, slot) pairs into expert-contiguous order.
//
// Entry i = t*k + s carries expert idx[i].  counts[e] = #entries of e,
// offsets = exclusive scan, and perm_src lists the entries of expert 0, then
// expert 1, ..., each expert's entries in increasing i (= increasing token,
// since a token picks an expert at most once).  Positions are computed from
// ranks, never from the order in which atomics land, so the result is unique
// and run-to-run identical.
//
// Two-level form: blocks own contiguous ranges of kPermChunk entries.  With
// more than one block a count kernel first writes per-block histograms; the
// scatter kernel derives every block's base per expert from them.  Inside a
// block, entries are ranked a round of 1024 at a time: __match_any_sync groups
// equal experts within a warp, and a per-expert scan over the 32 warps orders
// the warps.
#include "ffn_plan.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace lsv {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads) permute_count_kernel(const int32_t* __restrict__ idx, int n, int E,
                                                                 int32_t* __restrict__ blk_counts, int* err) {
  __shared__ int cnt[kMaxExperts];
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += kThreads) cnt[e] = 0;
  __syncthreads();
  const int begin = blockIdx.x * kPermChunk;
  const int end = min(n, begin + kPermChunk);
  for (int i = begin + threadIdx.x; i < end; i += kThreads) {
    const int e = idx[i];
    if (e < 0 || e >= E)
      set_error(err, kErrDeviceIndex);
    else
      atomicAdd(&cnt[e], 1);  // integer counts: the result does not depend on the order
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) blk_counts[(size_t)blockIdx.x * E + e] = cnt[e];
}

// Exclusive scan of v[0..E) into out[0..E] by warp 0 (E <= 256: 8 per lane).
__device__ void warp_exclusive_scan(const int* v, int* out, int E) {
  const int lane = threadIdx.x & 31;
  constexpr int PER = kMaxExperts / 32;
  int loc[PER];
  int sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane * PER + j;
    loc[j] = e < E ? v[e] : 0;
    sum += loc[j];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - sum;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane * PER + j;
    if (e < E) out[e] = run;
    run += loc[j];
  }
  if (lane == 31) out[E] = incl;
}

__global__ void __launch_bounds__(kThreads) permute_scatter_kernel(
    const int32_t* __restrict__ idx, int n, int E, int nblk, const int32_t* __restrict__ blk_counts,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, int* err) {
  __shared__ int tot[kMaxExperts];
  __shared__ int off[kMaxExperts + 1];
  __shared__ int base[kMaxExperts];
  __shared__ int wcnt[kWarps][kMaxExperts];

  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int begin = blockIdx.x * kPermChunk;
  const int end = min(n, begin + kPermChunk);

  // totals per expert and this block's share of earlier blocks
  if (nblk == 1) {
    for (int e = tid; e < E; e += kThreads) tot[e] = 0;
    __syncthreads();
    for (int i = begin + tid; i < end; i += kThreads) {
      const int e = idx[i];
      if (e >= 0 && e < E) atomicAdd(&tot[e], 1);
      else set_error(err, kErrDeviceIndex);
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) base[e] = 0;
  } else {
    for (int e = tid; e < E; e += kThreads) {
      int t = 0, pre = 0;
      for (int b = 0; b < nblk; ++b) {
        const int c = blk_counts[(size_t)b * E + e];
        if (b < blockIdx.x) pre += c;
        t += c;
      }
      tot[e] = t;
      base[e] = pre;
    }
  }
  __syncthreads();
  if (warp == 0) warp_exclusive_scan(tot, off, E);
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = tid; e < E; e += kThreads) {
      counts[e] = tot[e];
      offsets[e] = off[e];
    }
    if (tid == 0) offsets[E] = off[E];
  }
  for (int e = tid; e < E; e += kThreads) base[e] += off[e];
  __syncthreads();

  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r0 = begin; r0 < end; r0 += kThreads) {
    for (int q = tid; q < kWarps * E; q += kThreads) (&wcnt[0][0])[(q / E) * kMaxExperts + q % E] = 0;
    __syncthreads();
    const int i = r0 + tid;
    int e = (i < end) ? idx[i] : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0 && rank == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    for (int ee = tid; ee < E; ee += kThreads) {
      int acc = base[ee];
#pragma unroll 4
      for (int w = 0; w < kWarps; ++w) {
        const int c = wcnt[w][ee];
        wcnt[w][ee] = acc;
        acc += c;
      }
      base[ee] = acc;
    }
    __syncthreads();
    if (e >= 0) {
      const int pos = wcnt[warp][e] + rank;
      perm[pos] = i;
      inv[i] = pos;
    }
    __syncthreads();
  }
}

// Permutation, row gather and item table in one launch, for up to
// kPermFusedMax pairs.  CTA c owns the 32 pairs [32c, 32c+32): it histograms all pairs
// (cheap at these sizes) and, separately, the pairs before its slice, which
// gives every expert's offset and the slice's base inside each expert segment;
// warp 0 ranks the slice with __match_any_sync, and all warps copy the slice's
// token rows into expert order.  CTA 0 also writes counts/offsets and the item
// table of the grouped-expert kernel.
constexpr int kPgThreads = 256;
constexpr int kPgSlice = 32;

__global__ void __launch_bounds__(kPgThreads) permute_gather_kernel(
    const int32_t* __restrict__ idx, int T, int k, int E, int H, int S, int I, int BN, const bf16* __restrict__ x,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, bf16* __restrict__ xperm, int32_t* __restrict__ table, int* err) {
  __shared__ int tot[kMaxExperts];
  __shared__ int pre[kMaxExperts];
  __shared__ int off[kMaxExperts + 1];
  __shared__ int pos_s[kPgSlice];
  // the grouped-expert kernel that follows may start its routing-independent
  // items at once; anything that reads this kernel's results waits for it
  pdl_trigger();
  pdl_wait();
  const int n = T * k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s0 = blockIdx.x * kPgSlice;
  const int s1 = min(n, s0 + kPgSlice);
  for (int e = tid; e < E; e += kPgThreads) {
    tot[e] = 0;
    pre[e] = 0;
  }
  __syncthreads();
  for (int i = tid; i < n; i += kPgThreads) {
    const int e = idx[i];
    if (e < 0 || e >= E) {
      if (blockIdx.x == 0) set_error(err, kErrDeviceIndex);
      continue;
    }
    atomicAdd(&tot[e], 1);  // integer counts: independent of the order
    if (i < s0) atomicAdd(&pre[e], 1);
  }
  __syncthreads();
  if (warp == 0) warp_exclusive_scan(tot, off, E);
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = tid; e < E; e += kPgThreads) {
      counts[e] = tot[e];
      offsets[e] = off[e];
    }
    if (tid == 0) offsets[E] = off[E];
  }
  if (warp == 0) {
    const int i = s0 + lane;
    int e = i < s1 ? idx[i] : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int pos = -1;
    if (e >= 0) {
      pos = off[e] + pre[e] + rank;
      perm[pos] = i;
      inv[i] = pos;
    }
    pos_s[lane] = pos;
  } else if (warp == 1 && blockIdx.x == 0) {
    build_item_table(off, nullptr, T, H, E, k, S, I, BN, table, err);
  }
  __syncthreads();
  for (int j = warp; j < s1 - s0; j += kPgThreads / 32) {
    const int pos = pos_s[j];
    if (pos < 0) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)((s0 + j) / k) * H);
    uint4* dst = reinterpret_cast<uint4*>(xperm + (size_t)pos * H);
    for (int c = lane; c < H / 8; c += 32) dst[c] = __ldg(src + c);
  }
}

}  // namespace

cudaError_t launch_permute_gather(const int32_t* idx, int T, int k, int E, int H, int S, int I, int BN,
                                  const bf16* x, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                  bf16* xperm, int32_t* table, int* err, cudaStream_t s) {
  const int n = T * k;
  const int grid = n == 0 ? 1 : (n + kPgSlice - 1) / kPgSlice;
  return launch_pdl(permute_gather_kernel, dim3(grid), dim3(kPgThreads), 0, s, idx, T, k, E, H, S, I, BN, x,
                    counts, offsets, perm, inv, xperm, table, err);
}

cudaError_t launch_permute(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                           int32_t* perm, int32_t* inv, int32_t* blk_counts, int nblk, int* err,
                           cudaStream_t s) {
  const int n = T * k;
  if (nblk > 1) {
    cudaError_t e = launch_pdl(permute_count_kernel, dim3(nblk), dim3(kThreads), 0, s, idx, n, E, blk_counts, err);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(permute_scatter_kernel, dim3(nblk), dim3(kThreads), 0, s, idx, n, E, nblk,
                    (const int32_t*)blk_counts, counts, offsets, perm, inv, err);
}

}  // namespace lsv
