// skinny.cu -- dense products y = x W^T for few rows of x (M <= 256), the shape
// of every projection of the FastMTP draft block at decode batch sizes.
//
// The bytes are the weights, so the kernel is built to stream them from as
// many SMs as possible: the weight rows sit on the MMA's M side (128 per
// tile), the rows of x on its N side (M rounded up to 16), and the K range of
// a tile is split over the CTAs of a thread-block cluster (1, 2, 4 or 8,
// chosen so that the launch fits one wave).  Cluster rank r owns a slice of
// 128/ns accumulator rows: every CTA sends each slice of its fp32 partial tile
// straight from TMEM to the slice's owner with asynchronous stores into
// distributed shared memory (counted on the owner's mbarrier), and each owner
// sums its slice over the ranks in rank order (so the result is
// deterministic) and stores bf16.  No workspace, no atomics, and no CTA waits
// for another to finish reading.
//
// One launch can carry up to three weight matrices that share x (the block's
// q, k and v projections).  In the SwiGLU form the weight is a gate/up pair
// [2F, K] staged interleaved (gate row f next to up row f, 64 features per
// tile) and the epilogue writes silu(gate) * up.
//
// Warp 0 issues TMA, warp 1 the tcgen05 MMAs (accumulator in TMEM), warps 2..5
// move the accumulator to shared memory.  The weights of the first ring
// stages are requested before the wait for the preceding kernel (they do not
// depend on it), so their stream overlaps that kernel's tail.
#include <math.h>

#include <map>
#include <mutex>

#include "internal.h"
#include "lsv.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lsv {
namespace {

constexpr int kSkThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kSkMaxStages = 8;
constexpr int kSkATile = 128 * 128;  // one 64-wide K chunk of 128 weight rows

struct SkJob {
  bf16* y;         // output [M, ldy]
  const bf16* r;   // optional residual [M, ldy] added before the bf16 store (may be y itself)
  int ldy;
  int n_out;       // output columns of this job
  int tile0;       // first tile of this job
};

struct SkParams {
  int M, nk, n_mma, nsplit, njobs, stages;
  SkJob job[kSkMaxJobs];
  const bf16* x;   // the rows of x (for their mean squares)
  float norm_eps;  // > 0: scale output column m by 1/sqrt(mean_k x[m,k]^2 + eps) (RMSNorm of x folded in)
  int* err;
  uint64_t wait_ns;
};

struct SkMaps {
  CUtensorMap w[kSkMaxJobs];
  CUtensorMap x;
};

__device__ __forceinline__ float sk_silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// 1/sqrt(mean square + eps) of x rows 4c4..4c4+3, from every rank's share in rank order.
__device__ __forceinline__ float4 row_scales(const float* recv_ss, int ns, int n_mma, int c4, int K, float eps) {
  float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = 0; r < ns; ++r) {
    const float4 v = *reinterpret_cast<const float4*>(recv_ss + r * n_mma + 4 * c4);
    t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
  }
  const float inv_k = 1.0f / (float)K;
  return make_float4(rsqrtf(t.x * inv_k + eps), rsqrtf(t.y * inv_k + eps), rsqrtf(t.z * inv_k + eps),
                     rsqrtf(t.w * inv_k + eps));
}

// Grid (nsplit, tiles): blockIdx.y is the weight tile, blockIdx.x its K split and cluster rank.
template <bool kSwiglu>
__global__ void __launch_bounds__(kSkThreads) skinny_gemm_kernel(const __grid_constant__ SkMaps maps,
                                                                 const SkParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = kSkATile + p.n_mma * 128;
  __shared__ uint64_t full[kSkMaxStages], empty[kSkMaxStages], tfull, final_bar, recv_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ns = p.nsplit;
  const int split = blockIdx.x;  // == the CTA's rank in its cluster
  const int tile_g = blockIdx.y;
  int job = 0;
  for (int j = 1; j < p.njobs; ++j)
    if (tile_g >= p.job[j].tile0) job = j;
  const int tile = tile_g - p.job[job].tile0;
  const int c0 = split * p.nk / ns, c1 = (split + 1) * p.nk / ns;  // at least one chunk (ns <= nk)
  uint32_t tcols = 32;
  while (tcols < (uint32_t)p.n_mma) tcols <<= 1;
  // rank r sums accumulator rows [r * slot_rows, (r + 1) * slot_rows) (ns is 1, 2, 4 or 8, so a
  // slice is even and SwiGLU pairs stay together); recv[src] receives rank src's partial of them
  const int slot_rows = 128 / ns;
  float* recv = reinterpret_cast<float*>(smem + p.stages * stage_bytes);  // [ns][slot_rows][n_mma]
  float* recv_ss = recv + ns * slot_rows * p.n_mma;                       // [ns][n_mma] (norm_eps > 0)
  const bool norm = p.norm_eps > 0.0f;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull, 1);
    mbar_init(&final_bar, 1);
    mbar_init(&recv_bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    // the other ranks' partials of this CTA's rows (and of the rows' mean squares)
    if (ns > 1)
      mbar_arrive_expect_tx(&recv_bar, (uint32_t)((ns - 1) * (slot_rows + (p.norm_eps > 0.0f ? 1 : 0)) * p.n_mma * 4));
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, tcols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&maps.w[job]);
    tma_prefetch_desc(&maps.x);
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_slot;
  pdl_trigger();
  cluster_arrive_relaxed();  // matched by one cluster_wait per thread before any store into a peer

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      const CUtensorMap* wm = &maps.w[job];
      auto load_a = [&](int kc, int stage) {
        uint8_t* a_s = smem + stage * stage_bytes;
        if (kSwiglu)
          tma_load_3d(a_s, wm, &full[stage], kc * 64, 0, tile * 64, pol_w);
        else
          tma_load_2d(a_s, wm, &full[stage], kc * 64, tile * 128, pol_w);
      };
      auto load_b = [&](int kc, int stage) {
        tma_load_2d(smem + stage * stage_bytes + kSkATile, &maps.x, &full[stage], kc * 64, 0, pol_x);
      };
      // the first stages: the weights before the wait for the preceding kernel, x after it
      const int npre = min(p.stages, c1 - c0);
      for (int q = 0; q < npre; ++q) {
        mbar_arrive_expect_tx(&full[q], stage_bytes);
        load_a(c0 + q, q);
      }
      pdl_wait();  // x comes from the preceding kernel
      for (int q = 0; q < npre; ++q) load_b(c0 + q, q);
      bool ok = true;
      int q = npre;
      for (; q < c1 - c0; ++q) {
        const int stage = q % p.stages;
        if (!mbar_wait(&empty[stage], ((uint32_t)(q / p.stages) & 1u) ^ 1u, p.wait_ns)) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], stage_bytes);
        load_a(c0 + q, stage);
        load_b(c0 + q, stage);
      }
      if (!ok) {
        abort_flag = 1;
        __threadfence_block();
        mbar_arrive(&full[q % p.stages]);  // wake the MMA issuer so that it sees the abort
      }
    }
    __syncwarp();
    cluster_wait();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, p.n_mma);
      bool ok = true;
      for (int q = 0; q < c1 - c0; ++q) {
        const int stage = q % p.stages;
        if (!mbar_wait(&full[stage], (uint32_t)(q / p.stages) & 1u, p.wait_ns)) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        if (abort_flag) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_s = smem_u32(smem + stage * stage_bytes);
        const uint32_t b_s = a_s + kSkATile;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem_base, sdesc_kmajor_sw128(a_s + kk * 32), sdesc_kmajor_sw128(b_s + kk * 32), idesc,
                    (q | kk) ? 1u : 0u);
        umma_commit(&empty[stage]);
      }
      if (ok) {
        umma_commit(&tfull);
      } else {
        abort_flag = 1;
        __threadfence_block();
        mbar_arrive(&tfull);  // wake the epilogue so that it sees the abort
      }
      umma_commit(&final_bar);  // every MMA has completed before TMEM and the ring are reused
      if (!mbar_wait(&final_bar, 0, p.wait_ns)) set_error(p.err, kErrTimeout);
    }
    __syncwarp();
    cluster_wait();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    if (norm) {
      // While the MMAs run: this split's share of each x row's sum of squares (its K chunks),
      // one warp per row in turn, sent to every rank (its own: a plain shared store).
      pdl_wait();  // x comes from the preceding kernel
      const int we = warp - 2;
      const int q0 = c0 * 8, q1 = c1 * 8;  // 16-byte pieces of the row in this split
      float* ss_own = recv_ss + split * p.n_mma;
      for (int m = we; m < p.n_mma; m += 4) {
        float a = 0.0f;
        if (m < p.M) {
          const uint4* row = reinterpret_cast<const uint4*>(p.x + (size_t)m * p.nk * 64);
          for (int q = q0 + lane; q < q1; q += 32) {
            float f[8];
            const uint4 v = __ldg(row + q);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              f[2 * i] = __uint_as_float(wv[i] << 16);
              f[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) a = fmaf(f[i], f[i], a);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) ss_own[m] = a;
      }
      named_bar_sync(1, 128);  // the epilogue warps' shares are in ss_own
    }
    // Warp w reads TMEM lanes 32*(w%4)..+31 (one weight row per thread) and sends each row to
    // the rank that sums it: into that rank's recv[split] (its own rows: plain shared stores).
    const bool got = mbar_wait(&tfull, 0, p.wait_ns);
    if (!got) set_error(p.err, kErrTimeout);
    tc_fence_after_sync();
    const int qd = warp & 3;
    const int row = 32 * qd + lane;
    const int dst_rank = row / slot_rows;
    const int off = ((split * slot_rows) + row - dst_rank * slot_rows) * p.n_mma;
    float* mine = recv + off;
    cluster_wait();  // every CTA of the cluster runs, with its receive barrier armed
    if (norm) {
      // this split's sums of squares to every other rank's recv_ss[split]
      const int tid = threadIdx.x - 64, q4 = p.n_mma / 4;
      const float* ss_own = recv_ss + split * p.n_mma;
      for (int u = tid; u < (ns - 1) * q4; u += 128) {
        const int d = u / q4 + (u / q4 >= split ? 1 : 0), c = u % q4;
        const float4 v = *reinterpret_cast<const float4*>(ss_own + 4 * c);
        st_async_f4(mapa_shared(smem_u32(ss_own + 4 * c), (uint32_t)d), v,
                    mapa_shared(smem_u32(&recv_bar), (uint32_t)d));
      }
    }
    const uint32_t dst = mapa_shared(smem_u32(recv + off), (uint32_t)dst_rank);
    const uint32_t dst_bar = mapa_shared(smem_u32(&recv_bar), (uint32_t)dst_rank);
    const uint32_t t_row = tmem_base + ((uint32_t)(32 * qd) << 16);
    const bool live = got && !abort_flag;
    for (int cc = 0; cc < p.n_mma; cc += 16) {
      uint32_t r[16];
      if (live) {
        tmem_ld_32x32b_x16(t_row + cc, r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = 0u;  // the owner still counts these bytes
      }
#pragma unroll
      for (int j = 0; j < 16; j += 4) {
        const float4 v = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                                     __uint_as_float(r[j + 3]));
        if (dst_rank == split)
          *reinterpret_cast<float4*>(mine + cc + j) = v;
        else
          st_async_f4(dst + (uint32_t)((cc + j) * 4), v, dst_bar);
      }
    }
    tc_fence_before_sync();
  }
  __syncwarp();
  __syncthreads();  // this CTA's own rows are in recv[split]
  if (ns > 1 && !mbar_wait(&recv_bar, 0, p.wait_ns)) set_error(p.err, kErrTimeout);  // and the others'

  // ------------------------------------------------------------ reduction of this rank's rows
  // Summed over the ranks in rank order; 4 columns per unit.
  {
    const SkJob& jb = p.job[job];
    const int r0 = split * slot_rows;
    const int q4 = p.n_mma / 4;
    const int src_stride = slot_rows * p.n_mma;  // floats between two ranks' partials
    if (kSwiglu) {
      // units: (feature pair, 4 columns)
      const int units = slot_rows / 2 * q4;
      for (int u = threadIdx.x; u < units; u += kSkThreads) {
        const int pl = u / q4, c4 = u % q4;  // pair within the slice
        const float* pg = recv + (2 * pl) * p.n_mma + 4 * c4;
        const float* pu = pg + p.n_mma;
        float4 a[8], b[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < ns) {
            a[r] = *reinterpret_cast<const float4*>(pg + r * src_stride);
            b[r] = *reinterpret_cast<const float4*>(pu + r * src_stride);
          }
        const int pr = r0 / 2 + pl;
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), v = g;
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < ns) {
            g.x += a[r].x; g.y += a[r].y; g.z += a[r].z; g.w += a[r].w;
            v.x += b[r].x; v.y += b[r].y; v.z += b[r].z; v.w += b[r].w;
          }
        if (norm) {
          const float4 sc = row_scales(recv_ss, ns, p.n_mma, c4, p.nk * 64, p.norm_eps);
          g.x *= sc.x; g.y *= sc.y; g.z *= sc.z; g.w *= sc.w;
          v.x *= sc.x; v.y *= sc.y; v.z *= sc.z; v.w *= sc.w;
        }
        const int f = tile * 64 + pr;
        if (f < jb.n_out) {
          bf16* yc = jb.y + (size_t)(4 * c4) * jb.ldy + f;
          const int m = p.M - 4 * c4;
          if (m > 0) yc[0] = __float2bfloat16_rn(sk_silu(g.x) * v.x);
          if (m > 1) yc[jb.ldy] = __float2bfloat16_rn(sk_silu(g.y) * v.y);
          if (m > 2) yc[2 * jb.ldy] = __float2bfloat16_rn(sk_silu(g.z) * v.z);
          if (m > 3) yc[3 * jb.ldy] = __float2bfloat16_rn(sk_silu(g.w) * v.w);
        }
      }
    } else {
      // units: (row, 4 columns), consecutive threads on consecutive rows (coalesced stores)
      const int rows = slot_rows;
      const int units = rows * q4;
      for (int u = threadIdx.x; u < units; u += kSkThreads) {
        const int rl = u % rows, c4 = u / rows;
        const int rr = r0 + rl;
        const float* pa = recv + rl * p.n_mma + 4 * c4;
        float4 a[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < ns) a[r] = *reinterpret_cast<const float4*>(pa + r * src_stride);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < ns) {
            acc.x += a[r].x; acc.y += a[r].y; acc.z += a[r].z; acc.w += a[r].w;
          }
        if (norm) {
          const float4 sc = row_scales(recv_ss, ns, p.n_mma, c4, p.nk * 64, p.norm_eps);
          acc.x *= sc.x; acc.y *= sc.y; acc.z *= sc.z; acc.w *= sc.w;
        }
        const int f = tile * 128 + rr;
        if (f < jb.n_out) {
          const size_t at = (size_t)(4 * c4) * jb.ldy + f;
          bf16* yc = jb.y + at;
          const int m = p.M - 4 * c4;
          if (jb.r) {
            // the residual stream plus this product, rounded once
            const bf16* rc = jb.r + at;
            if (m > 0) acc.x += __bfloat162float(rc[0]);
            if (m > 1) acc.y += __bfloat162float(rc[jb.ldy]);
            if (m > 2) acc.z += __bfloat162float(rc[2 * jb.ldy]);
            if (m > 3) acc.w += __bfloat162float(rc[3 * jb.ldy]);
          }
          if (m > 0) yc[0] = __float2bfloat16_rn(acc.x);
          if (m > 1) yc[jb.ldy] = __float2bfloat16_rn(acc.y);
          if (m > 2) yc[2 * jb.ldy] = __float2bfloat16_rn(acc.z);
          if (m > 3) yc[3 * jb.ldy] = __float2bfloat16_rn(acc.w);
        }
      }
    }
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, tcols);
  }
}

// Ring stages: `base` (four keep two CTAs per SM up to 64 rows of x; eight give a lone CTA per SM
// more bytes in flight), within 200 KB together with the receive slots (at least two).
// Bytes per accumulator column of the receive slots: ns ranks x 128/ns rows x fp32 = 512, plus, with
// the norm folded in, up to 8 ranks' mean-square shares (32).
int sk_recv_per_col(bool norm) { return norm ? 544 : 512; }

int sk_stages(int n_mma, int base, bool norm) {
  const int stage = kSkATile + n_mma * 128;
  int st = base > kSkMaxStages ? kSkMaxStages : base;
  while (st > 2 && st * stage + sk_recv_per_col(norm) * n_mma > 200 * 1024) --st;
  return st;
}

// The ring, then the receive slots.  At n_mma = 256, two stages and the norm's shares that would be
// 233 KB, past the 227 KB a CTA may have, so products with the norm folded in take at most 128 rows
// of x per launch.
int sk_smem(int n_mma, int stages, bool norm) {
  return 1024 + stages * (kSkATile + n_mma * 128) + sk_recv_per_col(norm) * n_mma;
}

// CTAs of clusters of `ns` that the device holds at once for this shared-memory size (cached).
int sk_capacity(bool swiglu, int ns, int smem, const DeviceCtx& dc) {
  static std::mutex mu;
  static std::map<long long, int> cache;
  const long long key = ((long long)dc.device << 40) | ((long long)swiglu << 36) | ((long long)ns << 28) | smem;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int cap = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ns, 64);
  cfg.blockDim = dim3(kSkThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ns;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  cudaError_t e;
  if (swiglu) {
    e = ensure_smem_attr(reinterpret_cast<const void*>(skinny_gemm_kernel<true>), smem, dc.device);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&clusters, skinny_gemm_kernel<true>, &cfg);
  } else {
    e = ensure_smem_attr(reinterpret_cast<const void*>(skinny_gemm_kernel<false>), smem, dc.device);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&clusters, skinny_gemm_kernel<false>, &cfg);
  }
  if (e == cudaSuccess) cap = clusters * ns;
  cache[key] = cap;
  return cap;
}

}  // namespace

cudaError_t launch_skinny(const bf16* x, int M, int K, const bf16* const* w, const int* n_rows, bf16* const* y,
                          const int* ldy, int njobs, bool swiglu, const DeviceCtx& dc, cudaStream_t s,
                          float norm_eps, const bf16* const* res) {
  if (M <= 0 || M > kSkMaxRows || njobs < 1 || njobs > kSkMaxJobs || K <= 0 || K % 64) return cudaErrorInvalidValue;
  if (norm_eps > 0.0f && M > 128) {
    // two launches of at most 128 rows each (the norm is per row, so this is exact)
    bf16* y2[kSkMaxJobs];
    const bf16* r2[kSkMaxJobs];
    for (int j = 0; j < njobs; ++j) {
      y2[j] = y[j] + (size_t)128 * ldy[j];
      r2[j] = res && res[j] ? res[j] + (size_t)128 * ldy[j] : nullptr;
    }
    const cudaError_t e = launch_skinny(x, 128, K, w, n_rows, y, ldy, njobs, swiglu, dc, s, norm_eps, res);
    if (e != cudaSuccess) return e;
    return launch_skinny(x + (size_t)128 * K, M - 128, K, w, n_rows, y2, ldy, njobs, swiglu, dc, s, norm_eps,
                         res ? r2 : nullptr);
  }
  SkParams p = {};
  SkMaps maps;
  p.M = M;
  p.nk = K / 64;
  p.n_mma = ((M + 15) / 16) * 16;
  p.njobs = njobs;
  int tiles = 0;
  for (int j = 0; j < njobs; ++j) {
    SkJob& jb = p.job[j];
    jb.y = y[j];
    jb.r = res ? res[j] : nullptr;
    jb.ldy = ldy[j];
    jb.n_out = swiglu ? n_rows[j] / 2 : n_rows[j];
    jb.tile0 = tiles;
    tiles += (jb.n_out + (swiglu ? 63 : 127)) / (swiglu ? 64 : 128);
    const bool okm = swiglu ? make_map_gu(&maps.w[j], w[j], jb.n_out, jb.n_out, K)
                            : make_map(&maps.w[j], w[j], n_rows[j], K, 128);
    if (!okm) return cudaErrorInvalidValue;
  }
  for (int j = njobs; j < kSkMaxJobs; ++j) maps.w[j] = maps.w[0];
  if (!make_map(&maps.x, x, M, K, p.n_mma)) return cudaErrorInvalidValue;
  if (tiles > 65535) return cudaErrorInvalidValue;
  const bool norm = norm_eps > 0.0f;
  p.stages = sk_stages(p.n_mma, 4, norm);
  int smem = sk_smem(p.n_mma, p.stages, norm);
  // splits per tile: the one of 1, 2, 4, 8 (at most the K chunks) whose launch fits one wave and
  // gives the SMs the smallest share of the weights (the fewer splits on equal shares)
  int ns = 1;
  double best = 1e30;
  for (int c = 1; c <= 8 && c <= p.nk; c *= 2) {
    const int cap = sk_capacity(swiglu, c, smem, dc);
    if (c > 1 && (long long)tiles * c > cap) break;
    const double share = (double)(((long long)tiles * c + dc.num_sms - 1) / dc.num_sms) / c;
    if (share < best - 1e-9) {
      best = share;
      ns = c;
    }
  }
  // at most one CTA per SM: a deeper ring, if the clusters still fit at once
  if ((long long)tiles * ns <= dc.num_sms) {
    const int st = sk_stages(p.n_mma, kSkMaxStages, norm);
    const int sm2 = sk_smem(p.n_mma, st, norm);
    if (st > p.stages && (long long)tiles * ns <= sk_capacity(swiglu, ns, sm2, dc)) {
      p.stages = st;
      smem = sm2;
    }
  }
  p.nsplit = ns;
  p.x = x;
  p.norm_eps = norm_eps;
  p.err = dc.err;
  p.wait_ns = wait_limit_ns();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ns, tiles);
  cfg.blockDim = dim3(kSkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = ns;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e;
  if (swiglu) {
    e = ensure_smem_attr(reinterpret_cast<const void*>(skinny_gemm_kernel<true>), smem, dc.device);
    return e != cudaSuccess ? e : cudaLaunchKernelEx(&cfg, skinny_gemm_kernel<true>, maps, p);
  }
  e = ensure_smem_attr(reinterpret_cast<const void*>(skinny_gemm_kernel<false>), smem, dc.device);
  return e != cudaSuccess ? e : cudaLaunchKernelEx(&cfg, skinny_gemm_kernel<false>, maps, p);
}

}  // namespace lsv

using namespace lsv;

extern "C" {

lsv_status dense_swiglu(const void* x, const void* w_gate_up, void* y, int32_t M, int32_t F, int32_t K,
                        lsv_stream stream) {
  if (M < 0 || F <= 0 || K <= 0) return LSV_ERR_INVALID_ARG;
  if (M > kSkMaxRows || K % 64 || K > kMaxHidden || F % 8 || F > 32768) return LSV_ERR_UNSUPPORTED;
  if (M == 0) return LSV_OK;
  if (!x || !w_gate_up || !y) return LSV_ERR_INVALID_ARG;
  auto al = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  if (!al(x) || !al(w_gate_up) || !al(y)) return LSV_ERR_MISALIGNED;
  DeviceCtx* dc = nullptr;
  if (device_ctx(&dc) != cudaSuccess) return LSV_ERR_CUDA;
  const bf16* wp = static_cast<const bf16*>(w_gate_up);
  bf16* yp = static_cast<bf16*>(y);
  const int n = 2 * F, ld = F;
  return launch_skinny(static_cast<const bf16*>(x), M, K, &wp, &n, &yp, &ld, 1, true, *dc,
                       reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LSV_OK
             : LSV_ERR_CUDA;
}

}  // extern "C"
