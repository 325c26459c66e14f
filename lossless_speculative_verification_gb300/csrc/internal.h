// internal.h -- launchers and shared host-side declarations of the library
// (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace lsv {

typedef __nv_bfloat16 bf16;

// Limits shared by validation and kernels.
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kMaxShared = 8;
constexpr int kMaxHidden = 16384;
constexpr int kMaxVerifyRows = 64;  // K + 1 per sequence
constexpr int kMaxAttnQ = 8;        // verified positions per sequence in the attention
constexpr int kAttnMaxPairs = 1 << 18;  // (sequence, head) pairs per attention call
constexpr int kAttnMaxL = 1 << 16;      // cache capacity per sequence in the attention

// Per-device state: the error word's device address and the SM count.
struct DeviceCtx {
  int device = -1;
  int num_sms = 0;
  int l2_bytes = 0;
  int* err = nullptr;
};
cudaError_t device_ctx(DeviceCtx** out);
uint64_t wait_limit_ns();
// Raise `kernel`'s dynamic shared-memory limit to `bytes` on `device`, once per
// (kernel, device) pair; safe to call from several host threads at once.
cudaError_t ensure_smem_attr(const void* kernel, int bytes, int device);

// ---------------------------------------------------------------- FFN tile table
// int32 table in the workspace, written by the kernel that completes the
// permutation, read by the FFN kernel.
//   [0] gate/up items  [1] down items  [2] groups G
//   [8 .. 8+G]             gate/up item start per group slot (exclusive scan, G+1 entries)
//   [8+G+1 .. 8+2G+1]      down item start per group slot (G+1 entries)
// Group slots are the dealing order: the shared group first (when S > 0),
// then routed experts 0..E-1.
__host__ __device__ inline int table_ints(int G) { return 8 + 2 * (G + 1); }

// ---------------------------------------------------------------- counter block
// The first kCounterBytes of the workspace, at the same place for every shape:
// the counters of one layer call.  They are zero when a call begins -- the
// caller zeroes the block once, and every call clears them when it is done
// with them (the layer in its combine kernel, a standalone expert call in the
// expert kernel's last CTA) -- so no launch has to clear them first.
constexpr int kCntDone = 0;                      // [kMaxExperts + 1] finished gate/up tiles per group slot
constexpr int kCntDeal = kMaxExperts + 1;        // next item to deal
constexpr int kCntExit = kMaxExperts + 2;        // expert-kernel CTAs finished
constexpr int kCntSlots = kMaxExperts + 4;       // [kMaxExperts] rows placed per expert (slot placement)
constexpr size_t kCounterBytes = 4096;
static_assert((kCntSlots + kMaxExperts) * 4 <= (int)kCounterBytes, "counter block");

// Slot placement (token counts up to kSlotMaxTokens, where the router runs on
// CUDA cores): inside moe_verify_layer the router itself places each routed
// row at expert e's next free row of a fixed region [e*T, (e+1)*T) -- an
// atomic per-expert counter, so rows of one expert appear in any order, which
// no result depends on -- and each expert kernel CTA builds the item table from
// the per-expert counts.
constexpr int kSlotMaxTokens = 256;
inline bool use_slots(int T) { return T > 0 && T <= kSlotMaxTokens; }
// Rows of the routed row space (x_perm, act, y_perm) the workspace provides.
inline size_t routed_rows(int T, int k, int E) {
  const size_t compact = (size_t)T * k;
  const size_t slots = use_slots(T) ? (size_t)E * T : 0;
  return compact > slots ? compact : slots;
}

struct FfnGeom {
  int T, H, E, k, S, I, G, BN;
};

// Workspace layout (byte offsets, each region 256-byte aligned).
struct WsLayout {
  size_t counters;  // always 0: the counter block leads the workspace
  size_t topk_idx, topk_w, counts, offsets, perm, inv, blk_counts, table, xperm, act, act_sh, y_perm, y_sh;
  size_t total;
  int nblk;  // permutation blocks
};
WsLayout ws_layout(int T, int H, int E, int k, int S, int I);

constexpr int kPermChunk = 1024;      // (token, slot) entries per block of the two-level permutation
constexpr int kPermFusedMax = 8192;   // up to this many entries: one fused permutation + gather launch

// Launch with programmatic stream serialization: the kernel may start while its
// predecessor in the stream finishes; it must call pdl_wait() before touching
// memory the predecessor writes or reads.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- launchers
// Slot placement by the CUDA-core router (see use_slots): where to place the
// routed rows and what the last router CTA writes.
struct RouteSlots {
  bf16* xperm;     // [E*T, H] routed row space
  int32_t* inv;    // [T*k] row of each (token, rank)
  int32_t* slots;  // [E] rows taken per expert, zeroed before the router
};

cudaError_t launch_route(const bf16* x, const bf16* wr, int T, int H, int E, int k, int32_t* idx, float* w,
                         float* logits, cudaStream_t s, const RouteSlots* slots = nullptr);

cudaError_t launch_permute(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                           int32_t* perm, int32_t* inv, int32_t* blk_counts, int nblk, int* err,
                           cudaStream_t s);

// Permutation + row gather + item table in one launch (T*k <= kPermFusedMax).
cudaError_t launch_permute_gather(const int32_t* idx, int T, int k, int E, int H, int S, int I, int BN,
                                  const bf16* x, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                  bf16* xperm, int32_t* table, int* err, cudaStream_t s);

// Bulk L2 prefetch of the expert weights in the order the grouped-expert kernel
// consumes them (shared gate/up, routed gate/up, shared down, routed down), up
// to `budget` bytes.
cudaError_t launch_weight_prefetch(const bf16* w_gate_up, const bf16* w_down, const bf16* ws_gate_up,
                                   const bf16* ws_down, int H, int E, int S, int I, uint64_t budget,
                                   const DeviceCtx& dc, cudaStream_t s);

int ffn_token_tile(int T, int k, int E);
// Grouped experts.  with_prep: first gather the routed rows and build the item
// table (otherwise launch_permute_gather already did).  early: the table's
// counters were zeroed before the routing began, and the shared group's
// gate/up items (which do not depend on the routing) may start before the
// preceding kernels finish.
// y_perm/y_sh are fp32, or bf16 when y_bf16 (the fused layer keeps them in bf16).
// seg_cap > 0: slot placement (expert e's rows are [e*seg_cap, e*seg_cap +
// seg_counts[e]); every CTA builds the item table from seg_counts; offsets and
// perm unused; counts_out, if given, receives seg_counts).
cudaError_t launch_ffn(const bf16* x, const int32_t* perm, const int32_t* offsets, const int32_t* seg_counts,
                       int seg_cap, const bf16* w_gate_up, const bf16* w_down, const bf16* ws_gate_up,
                       const bf16* ws_down, int T, int H, int E, int k, int S, int I, void* y_perm, void* y_sh,
                       bool y_bf16, uint8_t* ws, const WsLayout& L, const DeviceCtx& dc, cudaStream_t s,
                       bool with_prep = true, bool early = false, int32_t* counts_out = nullptr);

// rows_y: rows of y_perm (inv entries outside [0, rows_y) raise LSV_ERR_DEVICE_INDEX).
// clear: optional int32 region of n_clear entries zeroed once the previous kernels completed.
cudaError_t launch_combine(const void* y_perm, const int32_t* inv, const float* topk_w, const void* y_sh,
                           bool y_bf16, int T, int H, int k, int rows_y, bf16* out, int* err, cudaStream_t s,
                           int32_t* clear = nullptr, int n_clear = 0);

cudaError_t launch_rmsnorm_residual(bf16* x, const bf16* y, bf16* h, int T, int H, float eps, cudaStream_t s);

size_t accept_ws_bytes(int B, int K, int V, int num_sms);
// Reduce per-(row, chunk) (max, first index) partials [B*(K+1), nchunk] to greedy tokens and apply
// the acceptance rule (one CTA per sequence).  argmax rows of sequence b start at b * argmax_ld
// (0: K + 1); accept_len and committed both null: the greedy tokens alone.
cudaError_t launch_accept_finalize(const float* pv, const int* pi, int nchunk, const int32_t* drafts, int B, int K,
                                   int32_t* argmax, int32_t* accept_len, int32_t* committed, cudaStream_t s,
                                   int argmax_ld = 0);
// Causal attention of Q verified positions per sequence over the cache.
int attention_splits(int L);
size_t attention_ws_bytes(int B, int Q, int L, int nh, int d);
cudaError_t launch_attention(const bf16* q, const bf16* kc, const bf16* vc, const int32_t* ctx_len, int B, int Q,
                             int L, int nh, int d, float scale, bf16* out, void* ws, const DeviceCtx& dc,
                             cudaStream_t s);
// Dense products for few rows of x (skinny.cu): y_j = x W_j^T for up to kSkMaxJobs weight matrices
// W_j [n_rows[j], K] sharing x [M, K] (M <= kSkMaxRows), or in the SwiGLU form y = silu(x W_g^T) * (x W_u^T)
// with W = [W_g; W_u] of n_rows = 2F rows.  K split over the CTAs of a cluster, reduced in shared memory.
// norm_eps > 0 folds RMSNorm of x's rows in (output row m scaled by 1/sqrt(mean_k x[m,k]^2 + eps));
// res[j] (optional, [M, ldy[j]], may equal y[j]) is added before the bf16 store.
constexpr int kSkMaxRows = 256;
constexpr int kSkMaxJobs = 3;
cudaError_t launch_skinny(const bf16* x, int M, int K, const bf16* const* w, const int* n_rows, bf16* const* y,
                          const int* ldy, int njobs, bool swiglu, const DeviceCtx& dc, cudaStream_t s,
                          float norm_eps = 0.0f, const bf16* const* res = nullptr);
// y[M, N] = bf16(x[M, K] w[N, K]^T) on tcgen05 (K % 64 == 0, N % 8 == 0).
cudaError_t launch_dense_gemm(const bf16* x, const bf16* w, bf16* y, int M, int N, int K, const DeviceCtx& dc,
                              cudaStream_t s);
// Counts of the accepted lengths of a batch into hist [K+1].
cudaError_t launch_accept_histogram(const int32_t* accept_len, int B, int K, int64_t* hist, int* err,
                                    cudaStream_t s);
// The verifier's output layer fused with the greedy-token search, then acceptance.  argmax_ld: the
// stride between sequences in argmax (0: K + 1); argmax may be null, and accept_len and committed
// may both be null (no rule: the greedy tokens alone).
size_t lmhead_ws_bytes(int B, int K, int V);
cudaError_t launch_lmhead_accept(const bf16* hidden, const bf16* w_vocab, const int32_t* drafts, int B, int K,
                                 int V, int H, int32_t* argmax, int32_t* accept_len, int32_t* committed, void* ws,
                                 const DeviceCtx& dc, cudaStream_t s, int argmax_ld = 0);
cudaError_t launch_accept(const bf16* logits, const int32_t* drafts, int B, int K, int V, int32_t* argmax,
                          int32_t* accept_len, int32_t* committed, void* ws, const DeviceCtx& dc,
                          cudaStream_t s);

cudaError_t launch_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t s);

}  // namespace lsv
