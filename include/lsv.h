/*
 * lsv.h -- C ABI of the GB300 (sm_103a) FastMTP verification step.
 *
 * The method (jina-ocr-v1; kg.zhiyong.dev "Jina AI's jina-ocr-v1 Is Selling
 * Throughput", section "The speed comes from three layers working together";
 * evolve.pub review "Summary", "Scope & Claims" (Section 3.1, Eq. 2)):
 * B sequences each carry K drafted tokens; the decoder verifies all B*(K+1)
 * positions in one pass.  Every decoder layer's FFN is a DeepSeek-style MoE
 * (64 routed experts, top-6 routing, 2 shared experts), and a greedy rule then
 * commits the longest draft prefix that matches the verifier's greedy tokens
 * plus one correction (or, when every draft matches, a bonus) token, so the
 * committed text equals plain greedy decoding.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers (memory the caller allocated on
 *     the current CUDA device), contiguous, row-major, 16-byte aligned unless a
 *     pointer is documented as optional and passed as NULL.
 *   - bf16 tensors are passed as `const void*` / `void*` holding IEEE bfloat16.
 *   - The caller owns all memory.  The library allocates no device memory; it
 *     keeps one device error word per device and the fixed scratch array of
 *     spec_verify_accept_noalloc (128 KiB per device), and nothing else.
 *   - Work is enqueued asynchronously on `stream` (NULL = the legacy default
 *     stream).  Argument errors are returned synchronously BEFORE any launch,
 *     with outputs untouched.  Errors found by kernels (an index out of range,
 *     a bounded wait that ran out) are written to the device error word; read
 *     it with lsv_get_device_error.
 *   - Entry points are thread-compatible: concurrent calls must use distinct
 *     workspaces.
 */
#ifndef LSV_H_
#define LSV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *lsv_stream;

typedef enum {
  LSV_OK = 0,
  LSV_ERR_INVALID_ARG = 1,  /* NULL pointer, negative or inconsistent size */
  LSV_ERR_UNSUPPORTED = 2,  /* shape outside the supported set (see each call) */
  LSV_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned */
  LSV_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than the queried size */
  LSV_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed (launch, attribute, tensor map) */
  LSV_ERR_TIMEOUT = 6,      /* device: a bounded wait ran out (kernel unwound, outputs undefined) */
  LSV_ERR_DEVICE_INDEX = 7  /* device: an index read from memory was out of range (outputs undefined) */
} lsv_status;

/* One MoE FFN layer: T tokens of width H; E routed experts of which each token
 * uses the top k; S shared experts; every expert is a SwiGLU of intermediate I.
 * Supported: T >= 0; H % 64 == 0, 64 <= H <= 16384; I % 64 == 0, 64 <= I;
 * S*I <= 16384; 1 <= E <= 256; 0 <= k <= min(E, 8); 0 <= S <= 8. */
typedef struct {
  int32_t T, H, E, k, S, I;
} lsv_moe_shape;

/* Expert weights (bf16, device).
 *   w_router   [E, H]
 *   w_gate_up  [E, 2I, H]  rows 0..I-1 of expert e: gate projection, rows I..2I-1: up projection
 *   w_down     [E, H, I]
 *   ws_gate_up [2*S*I, H]  rows s*I..s*I+I-1: gate of shared expert s; rows S*I+s*I..: its up
 *   ws_down    [H, S*I]    columns s*I..s*I+I-1: down projection of shared expert s
 * Expert e computes  y = W_down,e (silu(W_gate,e x) * (W_up,e x)),
 * silu(z) = z / (1 + exp(-z)); no biases. */
typedef struct {
  const void *w_router;
  const void *w_gate_up;
  const void *w_down;
  const void *ws_gate_up;
  const void *ws_down;
} lsv_moe_weights;

/* Bytes of workspace moe_verify_layer / moe_grouped_ffn / moe_permute need for
 * `shape` (a multiple of 256).  Returns 0 for an unsupported shape.
 * The first 4 KiB of the workspace are a counter block, at the same place for
 * every shape: they must be zero before the workspace's first use, and every
 * call that raises no device error leaves them zero again, so one workspace
 * serves any sequence of calls and shapes (zero them again after an error). */
size_t lsv_workspace_size(const lsv_moe_shape *shape);

/* Start streaming expert weights into L2, in the order moe_grouped_ffn reads
 * them (shared gate/up, routed gate/up, shared down, routed down), up to
 * max_bytes.  Returns at once; the data arrives while later work on the stream
 * runs.  A hint only: results never depend on it.  Useful when the caller
 * has independent work to overlap with it (for instance the attention block
 * before the MoE FFN); moe_verify_layer does not issue it, because its own
 * next kernel would wait for the prefetch grid to finish. */
lsv_status moe_prefetch_weights(const lsv_moe_weights *weights, const lsv_moe_shape *shape, size_t max_bytes,
                                lsv_stream stream);

/* Router: logits[t,e] = sum_h x[t,h] W_r[e,h] (fp32 accumulation in increasing
 * h); gate p = softmax over all E experts in fp32 (NOT renormalised over the
 * selection); the k experts with the largest logits in descending order, ties
 * to the lower expert index.
 * (kg.zhiyong.dev, "The speed comes from three layers working together":
 *  64 routed experts, top-6 routing.)
 *   x         [T, H] bf16          in
 *   w_router  [E, H] bf16          in
 *   topk_idx  [T, k] int32         out
 *   topk_w    [T, k] fp32          out  p of the selected experts
 *   logits_opt[T, E] fp32 or NULL  out */
lsv_status moe_route(const void *x, const void *w_router, const lsv_moe_shape *shape, int32_t *topk_idx,
                     float *topk_w, float *logits_opt, lsv_stream stream);

/* Expert-contiguous order of the T*k (token, slot) pairs (entry i = t*k + s):
 *   counts [E]     pairs per expert
 *   offsets[E+1]   exclusive prefix sum, offsets[E] = T*k
 *   perm_src[T*k]  entries grouped by expert, each group in increasing token order
 *   inv   [T*k]    inverse: inv[perm_src[r]] = r
 * Deterministic (no atomics decide any position).  An index outside [0,E)
 * sets LSV_ERR_DEVICE_INDEX on the device.  ws: lsv_workspace_size(shape). */
lsv_status moe_permute(const int32_t *topk_idx, const lsv_moe_shape *shape, int32_t *counts, int32_t *offsets,
                       int32_t *perm_src, int32_t *inv, void *ws, size_t ws_bytes, lsv_stream stream);

/* Grouped SwiGLU experts on the permuted pairs plus the shared experts:
 *   y_perm  [T*k, H] fp32  y_perm[r] = E_e(x[perm_src[r] / k]) for r in expert e's segment
 *   y_shared[T, H]   fp32  sum over shared experts s of S_s(x[t])  (ignored when S == 0; may be NULL then)
 * bf16 tensor-core products with fp32 accumulation; the SwiGLU activation is
 * rounded to bf16 before the down projection.  counts/offsets as from
 * moe_permute.  ws: lsv_workspace_size(shape). */
lsv_status moe_grouped_ffn(const void *x, const int32_t *perm_src, const int32_t *offsets, const int32_t *counts,
                           const lsv_moe_weights *weights, const lsv_moe_shape *shape, float *y_perm,
                           float *y_shared, void *ws, size_t ws_bytes, lsv_stream stream);

/* Gate-weighted combine:
 *   out[t,:] = sum_{s<k} topk_w[t,s] * y_perm[inv[t*k+s],:] + y_shared[t,:]   (bf16 out)
 * summed in fp32 in slot order, then the shared term; y_shared may be NULL
 * (no shared experts). */
lsv_status moe_combine(const float *y_perm, const int32_t *inv, const float *topk_w, const float *y_shared,
                       const lsv_moe_shape *shape, void *out, lsv_stream stream);

/* The whole MoE layer: route, permute, grouped experts, combine.
 *   x   [T, H] bf16 in;  out [T, H] bf16 out
 *   topk_idx_opt [T, k] int32 and counts_opt [E] int32: optional copies of the routing.
 * The expert outputs are kept in bf16 between the experts and the combine.
 * Up to 256 tokens the router itself places each routed row (one launch less);
 * the order of rows inside an expert is then decided by atomics, which no
 * output depends on: out is bit-identical from run to run.
 * ws: lsv_workspace_size(shape). */
lsv_status moe_verify_layer(const void *x, const lsv_moe_weights *weights, const lsv_moe_shape *shape, void *out,
                            int32_t *topk_idx_opt, int32_t *counts_opt, void *ws, size_t ws_bytes,
                            lsv_stream stream);

/* Bytes of workspace spec_verify_accept needs (a multiple of 256).  Its
 * contents need no initialisation: every call writes what it reads. */
size_t spec_verify_workspace_size(int32_t B, int32_t K, int32_t V);

/* Greedy verification (kg.zhiyong.dev, "Why FastMTP fits OCR particularly
 * well": bonus token when all drafts match; committed text matches ordinary
 * greedy decoding; evolve.pub review, Section 3.1 / Eq. 2).
 *   logits [B, K+1, V] bf16: row j is the verifier's prediction for the
 *          position after input j (input 0 = last committed token, input j = draft j)
 *   drafts [B, K] int32
 *   g[b,j]        = the smallest index attaining the row maximum; logits are finite or
 *                   -inf (a row of -inf gives 0); with a NaN in a row its g is unspecified
 *   accept_len[b] = largest L <= K with drafts[b,i] == g[b,i] for all i < L
 *   committed[b]  = drafts[b,0..L-1], g[b,L], then -1 (K+1 entries)
 *   argmax_opt [B, K+1] int32 or NULL: g
 * A draft outside [0,V) is a mismatch, not an error.  1 <= K+1 <= 64,
 * 1 <= V < 2^31, B >= 0.  ws: spec_verify_workspace_size(B,K,V). */
lsv_status spec_verify_accept(const void *logits, const int32_t *drafts, int32_t B, int32_t K, int32_t V,
                              int32_t *argmax_opt, int32_t *accept_len, int32_t *committed, void *ws,
                              size_t ws_bytes, lsv_stream stream);

/* Causal attention of the verified positions over their sequences' caches
 * (the verify pass presents every sequence's K+1 positions at once):
 *   q       [B, Q, nh, d] bf16: queries of the Q = K+1 verified positions
 *   k_cache [B, L, nh, d] bf16, v_cache [B, L, nh, d] bf16: per-sequence caches of
 *           capacity L; entries 0..ctx_len[b]-1 are valid and the last Q of them
 *           belong to the verified positions themselves
 *   ctx_len [B] int32 (device): Q <= ctx_len[b] <= L
 *   out     [B, Q, nh, d] bf16:
 *     out[b,j,h] = sum_{t <= p} softmax_t(scale * q[b,j,h].k[b,t,h]) v[b,t,h],
 *     p = ctx_len[b] - Q + j (query j sees the cache up to and including itself)
 * fp32 scores and accumulation.  Supported: d in {64, 128}, 1 <= Q <= 8,
 * L <= 65536, B, nh <= 65535, B*nh <= 262144, scale > 0.  Cache entries at or past
 * ctx_len[b] are never used, whatever they hold.  A ctx_len outside [Q, L] raises
 * LSV_ERR_DEVICE_INDEX (that sequence's output is zero).
 * Device pointers, 16-byte aligned.
 * ws: spec_verify_attention_workspace_size(B,Q,L,nh,d) bytes (0: unsupported).
 * Its first 256 bytes hold a work counter, at the same place for every shape:
 * zero before the first use; every call that raises no device error leaves it
 * zero again, so one workspace serves any later call whose size fits (zero it
 * again after an error).
 * Two launches (the stream over the caches, then the merge of its partial
 * states); a call may start before the previous work on the stream ends
 * (programmatic dependent launch) but reads nothing before that work is done. */
size_t spec_verify_attention_workspace_size(int32_t B, int32_t Q, int32_t L, int32_t nh, int32_t d);
lsv_status spec_verify_attention(const void *q, const void *k_cache, const void *v_cache, const int32_t *ctx_len,
                                 int32_t B, int32_t Q, int32_t L, int32_t nh, int32_t d, float scale, void *out,
                                 void *ws, size_t ws_bytes, lsv_stream stream);

/* The data movements of a verify pass around its kernels (one launch each).
 *
 * lsv_gather_rows: out[i, :] = table[idx[i], :] for i < n, rows of row_elems
 *   bf16 (for example the embedding rows of the verified tokens).
 *   table [n_table, row_elems], idx [n] int32 (device), out [n, row_elems].
 *   row_elems % 8 == 0.  An index outside [0, n_table) writes a zero row and
 *   raises LSV_ERR_DEVICE_INDEX.
 *
 * spec_cache_append: the keys and values of the Q verified positions of every
 *   sequence go to its cache before the verify attention reads it:
 *   k_cache[b, ctx_len[b] - Q + j, :] = k_new[b*Q + j, :] (the same for v),
 *   k_new, v_new [B*Q, row_elems] bf16 (row_elems = heads * head width),
 *   k_cache, v_cache [B, L, row_elems] bf16, ctx_len [B] int32 (device): the
 *   lengths after the append, as spec_verify_attention takes them.
 *   row_elems % 8 == 0, 1 <= Q <= L.  A length outside [Q, L] raises
 *   LSV_ERR_DEVICE_INDEX and leaves that sequence's cache alone.
 * Device pointers, 16-byte aligned. */
lsv_status lsv_gather_rows(const void *table, const int32_t *idx, int32_t n, int32_t n_table, int32_t row_elems,
                           void *out, lsv_stream stream);
lsv_status spec_cache_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             const int32_t *ctx_len, int32_t B, int32_t Q, int32_t L, int32_t row_elems,
                             lsv_stream stream);

/* Greedy verification with the verify logits produced by the verifier's output
 * layer, inside the call (the logits are never written to memory):
 *   hidden  [B*(K+1), H] bf16: the verifier's last hidden state of every verified
 *           position, row b*(K+1)+j for sequence b, input position j (as for the
 *           logit rows of spec_verify_accept)
 *   w_vocab [V, H] bf16: the output layer; logit[r,v] = sum_h hidden[r,h] * w_vocab[v,h]
 * The greedy token is the smallest v attaining the row maximum of the logits
 * computed from the bf16 inputs with fp32 accumulation (tensor cores); the rule,
 * drafts and outputs are those of spec_verify_accept.  Supported: H % 64 == 0,
 * H <= 16384, 1 <= K+1 <= 64, V >= 1, B >= 0.  Device pointers, 16-byte aligned.
 * ws: spec_verify_lmhead_workspace_size(B,K,V,H) bytes (0: unsupported shape). */
size_t spec_verify_lmhead_workspace_size(int32_t B, int32_t K, int32_t V, int32_t H);
lsv_status spec_verify_lmhead(const void *hidden, const void *w_vocab, const int32_t *drafts, int32_t B, int32_t K,
                              int32_t V, int32_t H, int32_t *argmax_opt, int32_t *accept_len, int32_t *committed,
                              void *ws, size_t ws_bytes, lsv_stream stream);

/* Choice of the number of drafts K (the pages' decomposition S = tau / c).
 *   cond_accept [kmax] (host): a_i = P(draft i accepted | drafts 1..i-1 accepted), in [0, 1]
 *   step_cost [kmax+1] (host): cost of one step with K drafts (drafting plus
 *             verification), K = 0 being a plain greedy step; > 0, any unit
 * tau(K) = sum_{i=0..K} prod_{j<=i} a_j is the mean number of tokens a step
 * commits; speedup(K) = tau(K) * step_cost[0] / step_cost[K].  *k_best is the K
 * of the largest speedup (the smaller K on equal values); tau_out and
 * speedup_out (host, kmax+1 entries each) are optional.  Host only, no device
 * work; 0 <= kmax <= 63. */
lsv_status spec_k_policy(const double *cond_accept, int32_t kmax, const double *step_cost, int32_t *k_best,
                         double *tau_out, double *speedup_out);

/* Accumulate the accepted lengths of a batch (accept_len [B] int32, device, as
 * spec_verify_accept writes them) into hist [K+1] int64 (device, 8-byte aligned):
 * hist[L] += #{b : accept_len[b] == L}.  Not cleared by the call.  A length
 * outside [0, K] raises LSV_ERR_DEVICE_INDEX and is not counted.  One launch. */
lsv_status spec_accept_histogram(const int32_t *accept_len, int32_t B, int32_t K, int64_t *hist,
                                 lsv_stream stream);

/* Conditional acceptances from such a histogram (host copy):
 * cond[i-1] = #(L >= i) / #(L >= i-1) for i = 1..K, 0 where nothing reached draft i. */
lsv_status spec_cond_accept_from_histogram(const int64_t *hist, int32_t K, double *cond);

/* Dense product y [M, N] = bf16(x [M, K] w [N, K]^T), bf16 inputs, fp32 accumulation
 * (tcgen05).  Device pointers, 16-byte aligned; K % 64 == 0, K <= 16384,
 * N % 8 == 0.  No workspace.  One launch.  Up to 256 rows of x (the decode
 * shapes), the weight rows take the MMA's M side and each 128-row weight tile's
 * K range is split over a thread-block cluster of up to 8 CTAs whose partial
 * sums are added in shared memory in a fixed order (deterministic); w (not x)
 * may then be read before the work that precedes the call on the stream has
 * finished, so that work must not write w. */
lsv_status dense_matmul(const void *x, const void *w, void *y, int32_t M, int32_t N, int32_t K, lsv_stream stream);

/* The FFN form of the same product for few rows of x:
 *   y [M, F] = bf16(silu(x [M, K] w_gate^T) * (x w_up^T)),  silu(z) = z / (1 + e^-z),
 *   w_gate_up [2F, K]: rows 0..F-1 w_gate, F..2F-1 w_up.
 * bf16 inputs, fp32 sums, deterministic.  1 <= M <= 256 (M = 0: no-op),
 * K % 64 == 0, K <= 16384, F % 8 == 0, F <= 32768.  Device pointers, 16-byte
 * aligned.  No workspace.  One launch. */
lsv_status dense_swiglu(const void *x, const void *w_gate_up, void *y, int32_t M, int32_t F, int32_t K,
                        lsv_stream stream);

/* Weights of the FastMTP draft block (bf16, device, 16-byte aligned):
 *   emb [V, H] (token embedding), w_proj [H, 2H], w_q, w_k, w_v, w_o [H, H],
 *   w_gate_up [2I, H] (rows 0..I-1 gate, I..2I-1 up), w_down [H, I],
 *   w_vocab [V, H] (the output layer, shared with the verifier). */
typedef struct {
  const void *emb;
  const void *w_proj;
  const void *w_q;
  const void *w_k;
  const void *w_v;
  const void *w_o;
  const void *w_gate_up;
  const void *w_down;
  const void *w_vocab;
} lsv_draft_weights;

/* K recursive applications of the shared draft block (one dense block that
 * proposes the drafts the verify pass checks).  Step i takes the previous
 * state h and token t (step 1: h0 [B, H] bf16, the verifier's last hidden
 * state, and t0 [B] int32, the last committed token):
 *   u = W_p [RMSNorm(h); RMSNorm(emb[t])];  a = RMSNorm(u)
 *   q, k, v = W_q a, W_k a, W_v a;  k, v are written to the block's caches
 *     k_cache, v_cache [B, L, nh, H/nh] bf16 at position ctx_len[b] + i - 1, and
 *     q attends to positions 0..ctx_len[b] + i - 1 (scale 1/sqrt(H/nh))
 *   u = u + W_o attn;  f = RMSNorm(u);  u = u + W_down (silu(W_gate f) * W_up f)
 *   t = argmax_v (W_vocab RMSNorm(u))_v (the smallest index of the maximum), h = u
 * RMSNorm: unit weight, eps 1e-6.  Every value stored between kernels is bf16:
 * the block input, u, q, k, v, the attention output, the activation; the
 * RMSNorms of u are folded into the products that read them (each output row
 * scaled by its input row's 1/rms in fp32) and never stored, the residual adds
 * happen in the products' epilogues, and t is taken from W_vocab u (the same
 * greedy token: the norm scales a row's logits by one positive factor).
 * drafts [B, K] int32 (device) receives t of every step; h_out [B, H] bf16
 * (optional) the last u.  ctx_len [B] int32 (device) is read, not written;
 * ctx_len[b] + K <= L.  Supported: 0 <= B <= 256, H % 64 == 0, H <= 16384,
 * H/nh in {64, 128}, I % 64 == 0, I <= 16384, 1 <= K <= 63.  Per step, 11
 * launches and no copies: the block input's norms (step i > 1 reads its token
 * from column i - 1 of drafts), the projections as the few-row products of
 * dense_matmul / dense_swiglu (q, k and v in one launch), the cache append, the
 * attention of spec_verify_attention at one query (two launches), and the
 * output layer fused with the greedy search of spec_verify_lmhead (two
 * launches), which writes the step's token into column i of drafts.
 * ws: spec_draft_workspace_size(B, H, nh, I, V, L) bytes, zero before the first
 * use; calls that raise no device error leave it fit for the next call. */
size_t spec_draft_workspace_size(int32_t B, int32_t H, int32_t nh, int32_t I, int32_t V, int32_t L);
lsv_status spec_draft_loop(const lsv_draft_weights *weights, const void *h0, const int32_t *t0, void *k_cache,
                           void *v_cache, const int32_t *ctx_len, int32_t B, int32_t K, int32_t H, int32_t nh,
                           int32_t I, int32_t V, int32_t L, int32_t *drafts, void *h_out, void *ws, size_t ws_bytes,
                           lsv_stream stream);

/* spec_verify_accept without a workspace, for callers that cannot allocate
 * device memory at the point where they verify: for example a host that runs
 * this library as a plugin and hands it only the tensors of the call (no
 * allocator and no workspace), or a decode loop whose memory is fixed before
 * it starts and may not grow.  The paper has no counterpart; this is a
 * convenience of the library.
 *   Same arguments, rule and outputs as spec_verify_accept, minus ws/ws_bytes.
 *   The argmax partials live in one fixed device array of 128 KiB (16,384
 *   (max, index) pairs), held by every device that loads the library until
 *   the process exits.  A call needs B*(K+1) rows times the chunks per row
 *   (on a 152-SM GB300: 4 chunks per row at 128 rows of 129,280 logits, 1
 *   chunk per row from 305 rows on), so up to 16,384 rows; a larger problem
 *   returns LSV_ERR_UNSUPPORTED before any launch.
 *   The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 *   routine.  The first call on each device looks up the array's device
 *   address (cudaGetSymbolAddress) and caches it.  All calls on a device share
 *   the array and it keeps the previous call's contents; nothing in it needs
 *   to start at zero, since each call writes every partial it reads.  Calls
 *   that overlap on the GPU (different streams, no ordering between them)
 *   race on the array: order them on one stream or with events. */
lsv_status spec_verify_accept_noalloc(const void *logits, const int32_t *drafts, int32_t B, int32_t K, int32_t V,
                                      int32_t *argmax_opt, int32_t *accept_len, int32_t *committed,
                                      lsv_stream stream);

/* Residual update and normalisation between stacked layers:
 *   x[t,:] <- bf16(x[t,:] + y[t,:]);   h[t,:] = bf16(x[t,:] / sqrt(mean(x[t,:]^2) + eps))
 * x [T,H] bf16 in/out, y [T,H] bf16 in, h [T,H] bf16 out; fp32 arithmetic;
 * unit norm weight. */
lsv_status rmsnorm_residual(void *x, const void *y, void *h, int32_t T, int32_t H, float eps,
                            lsv_stream stream);

/* Synchronise `stream`, return the current device's error word in *code_out
 * (an lsv_status value, 0 if none) and clear it. */
lsv_status lsv_get_device_error(int32_t *code_out, lsv_stream stream);

/* Upper bound, in nanoseconds, of every bounded wait inside the kernels
 * (default 2e9).  Process-wide; takes effect for launches after the call. */
lsv_status lsv_set_wait_limit_ns(uint64_t ns);

/* Launch one CTA that waits on a flag nothing ever sets, using the same
 * bounded wait as the kernels; it must end by writing LSV_ERR_TIMEOUT to the
 * error word.  For testing the failure path without faulting the GPU. */
lsv_status lsv_selftest_wait_timeout(uint64_t limit_ns, lsv_stream stream);

const char *lsv_status_string(lsv_status status);

/* 100 * major + minor. */
int32_t lsv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LSV_H_ */
