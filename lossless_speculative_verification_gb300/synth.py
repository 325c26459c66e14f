"""Seeded synthetic inputs for the FastMTP verify step.

This module draws the tensors that both the CUDA path and the CPU oracle
consume.  It holds none of the method's arithmetic: no router product, no
softmax, no selection, no expert FFN, no argmax and no acceptance rule.  What
it does hold is input shaping:

* bf16 rounding of float32 draws (round to nearest even), so that every
  consumer sees the same bf16 bits;
* hidden states drawn as N(0,1) rows rescaled onto the sphere of radius
  sqrt(H) (unit mean square, the distribution of "N(0,1) after RMSNorm");
* verifier logits N(0, std 2) with a *planted* row maximum, so that the
  greedy token of every row is known by construction (a tie with a second
  index is planted in a fraction of the rows);
* draft tokens that agree with the planted greedy token with a given
  probability per position (the pages report conditional acceptances
  0.830 / 0.663 / 0.636 at positions 1/2/3, Table 8 of the jina-ocr-v1
  paper as quoted by the evolve.pub review);
* an optional per-row rejection callback for the hidden states, which the
  tests use to enforce a minimum gap between consecutive router places
  (the callback is supplied by the caller; this module never computes it).

Randomness: numpy PCG64 streams spawned from one SeedSequence per problem,
one stream per tensor, so that adding a tensor never shifts another one.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# Conditional acceptance at draft positions 1/2/3 reported for K=3 on an L4
# (jina-ocr-v1 paper, Table 8, as summarised in the evolve.pub review).
PAGE_ACCEPT = (0.830, 0.663, 0.636)

VOCAB = 129_280          # decoder vocabulary of the DeepSeek-OCR family decoder
SWEEP_B = (1, 4, 8, 16, 32, 64)
SWEEP_K = (0, 1, 2, 3)   # K = 0: the plain greedy step


# --------------------------------------------------------------------------- bf16 bits
def bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_value(u) -> np.ndarray:
    """Widen bf16 bits (uint16) to float32 exactly."""
    u = np.ascontiguousarray(u, dtype=np.uint16)
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_next_up(u: np.ndarray) -> np.ndarray:
    """The next larger bf16 value (finite inputs only)."""
    u = np.asarray(u, dtype=np.uint16)
    neg = (u & np.uint16(0x8000)) != 0
    zero_neg = u == np.uint16(0x8000)
    out = np.where(neg, u - np.uint16(1), u + np.uint16(1)).astype(np.uint16)
    out = np.where(zero_neg, np.uint16(0x0001), out)
    return out.astype(np.uint16)


def streams(seed: int, n: int) -> list[np.random.Generator]:
    ss = np.random.SeedSequence(seed)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(n)]


# --------------------------------------------------------------------------- shapes
@dataclass(frozen=True)
class MoeDims:
    """One MoE FFN layer: T tokens of width H, E routed experts (top-k) of
    SwiGLU intermediate I, and S always-on shared experts of intermediate I."""
    T: int
    H: int
    E: int
    k: int
    S: int
    I: int


@dataclass(frozen=True)
class Workload:
    name: str
    dims: MoeDims
    B: int = 0
    K: int = 0
    V: int = 0
    hidden: str = "sphere"        # "sphere" (unit RMS rows) or "normal" (N(0, 0.02))
    accept: tuple = PAGE_ACCEPT
    layers: int = 1
    zipf_s: float = 0.0


def _verify_dims(B, K, H=1280, E=64, k=6, S=2, I=896):
    return MoeDims(T=B * (K + 1), H=H, E=E, k=k, S=S, I=I)


WORKLOADS = {
    # 4 sequences x (K=3)+1 = 16 tokens, hidden 256, 8 experts top-2, 1 shared,
    # intermediate 128, everything N(0, 0.02); acceptance over a 1024-token vocab
    # with each draft equal to the greedy token with probability 0.8.
    "tiny": Workload("tiny", MoeDims(16, 256, 8, 2, 1, 128), B=4, K=3, V=1024,
                     hidden="normal", accept=(0.8, 0.8, 0.8)),
    # 32 sequences x (K=3)+1 = 128 tokens through the decoder MoE layer shape
    # (64 routed experts top-6 + 2 shared, hidden 1280, intermediate 896),
    # then greedy acceptance over the 129,280-token vocabulary.
    "decode": Workload("decode", _verify_dims(32, 3), B=32, K=3, V=VOCAB),
    # 8 pages x (1,156 visual + 64 prompt tokens) = 9,760 tokens, same layer.
    "prefill": Workload("prefill", MoeDims(9760, 1280, 64, 6, 2, 896)),
    # 11 layers of the decode layer shape at 64 x (K=3)+1 = 256 tokens, router
    # popularity skewed Zipf(1.2) over the experts, then K=3 acceptance.
    "stack": Workload("stack", _verify_dims(64, 3), B=64, K=3, V=VOCAB, layers=11,
                      zipf_s=1.2),
}


def sweep_workload(B: int, K: int) -> Workload:
    """One point of the (batch, K) verify sweep through the decode layer."""
    return Workload(f"sweep_b{B}_k{K}", _verify_dims(B, K), B=B, K=K, V=VOCAB,
                    accept=PAGE_ACCEPT[:K])


def sweep_seed(B: int, K: int) -> int:
    return 1000 * B + K


# --------------------------------------------------------------------------- MoE tensors
@dataclass
class MoeProblem:
    dims: MoeDims
    x: np.ndarray            # [T,H] bf16 bits
    w_router: np.ndarray     # [E,H]
    w_gate_up: np.ndarray    # [E,2I,H]: rows 0..I-1 gate, I..2I-1 up
    w_down: np.ndarray       # [E,H,I]
    ws_gate_up: np.ndarray   # [2*S*I,H]: rows 0..S*I-1 gates of the S shared experts, then their ups
    ws_down: np.ndarray      # [H,S*I]
    resampled: int = 0
    extra: dict = field(default_factory=dict)


def _normal_bf16(rng, shape, std):
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def moe_weights(d: MoeDims, rngs, std=0.02):
    """Router, routed-expert and shared-expert weights, N(0, std) in bf16."""
    r_router, r_gu, r_dn, r_sgu, r_sdn = rngs
    w_router = _normal_bf16(r_router, (d.E, d.H), std)
    w_gate_up = np.empty((d.E, 2 * d.I, d.H), dtype=np.uint16)
    w_down = np.empty((d.E, d.H, d.I), dtype=np.uint16)
    for e in range(d.E):                     # per expert keeps the float32 temporaries small
        w_gate_up[e] = _normal_bf16(r_gu, (2 * d.I, d.H), std)
        w_down[e] = _normal_bf16(r_dn, (d.H, d.I), std)
    ws_gate_up = _normal_bf16(r_sgu, (2 * d.S * d.I, d.H), std)
    ws_down = _normal_bf16(r_sdn, (d.H, d.S * d.I), std)
    return w_router, w_gate_up, w_down, ws_gate_up, ws_down


def hidden_rows(rng, n, H, kind) -> np.ndarray:
    if kind == "normal":
        return _normal_bf16(rng, (n, H), 0.02)
    z = rng.standard_normal((n, H), dtype=np.float32).astype(np.float64)
    z *= math.sqrt(H) / np.sqrt((z * z).sum(axis=1, keepdims=True))
    return bf16_bits(z.astype(np.float32))


def _resample(x, rng, row_ok, draw, max_rounds):
    """Redraw rows of x that the caller's predicate rejects (deterministic in the seed)."""
    total = 0
    for _ in range(max_rounds):
        ok = np.asarray(row_ok(x), dtype=bool)
        bad = np.nonzero(~ok)[0]
        if bad.size == 0:
            return total
        x[bad] = draw(rng, bad.size)
        total += int(bad.size)
    raise RuntimeError("row predicate still failing after %d rounds" % max_rounds)


def moe_problem(w: Workload | MoeDims, seed: int = 0, row_ok=None, hidden: str | None = None,
                max_rounds: int = 200) -> MoeProblem:
    """One MoE layer's weights and hidden states.

    row_ok(x_bits, w_router_bits) -> bool[T] (optional) rejects hidden rows;
    rejected rows are redrawn from the hidden-state stream until all pass.
    """
    d = w.dims if isinstance(w, Workload) else w
    kind = hidden or (w.hidden if isinstance(w, Workload) else "sphere")
    rs = streams(seed, 6)
    w_router, w_gate_up, w_down, ws_gate_up, ws_down = moe_weights(d, rs[:5])
    x = hidden_rows(rs[5], d.T, d.H, kind)
    n = 0
    if row_ok is not None:
        n = _resample(x, rs[5], lambda xx: row_ok(xx, w_router),
                      lambda rng, m: hidden_rows(rng, m, d.H, kind), max_rounds)
    return MoeProblem(d, x, w_router, w_gate_up, w_down, ws_gate_up, ws_down, n)


# --------------------------------------------------------------------------- stack
def zipf_shares(E: int, s: float) -> np.ndarray:
    r = np.arange(1, E + 1, dtype=np.float64)
    z = r ** (-s)
    return z / z.sum()


def stack_problem(w: Workload, seed: int = 0, row_ok=None, max_rounds: int = 200):
    """Per-layer weights for the layer stack plus the residual stream x0 and the
    first layer input h0.

    Popularity skew: every hidden row carries a DC component of 1 (x0 = z + 1),
    and router row e of every layer gets a constant added, chosen so that the
    constant shifts expert e's router score by ln(zipf share of its rank); the
    rank of each expert is a seeded permutation per layer.  This tilts the
    softmax gate towards a Zipf(s) popularity without touching the selection
    rule itself.
    """
    d = w.dims
    rs = streams(seed, 2 + 6 * w.layers)
    r_x, r_perm = rs[0], rs[1]

    def draw(rng, m):
        z = rng.standard_normal((m, d.H), dtype=np.float32).astype(np.float64) + 1.0
        return z

    x0f = draw(r_x, d.T)

    def to_h(xf):
        # rows rescaled to unit mean square (the normalised layer input)
        return bf16_bits((xf * np.sqrt(d.H / (xf * xf).sum(axis=1, keepdims=True))).astype(np.float32))

    shares = zipf_shares(d.E, w.zipf_s)
    beta = np.log(shares)
    layers = []
    for l in range(w.layers):
        w_router, w_gate_up, w_down, ws_gate_up, ws_down = moe_weights(d, rs[2 + 6 * l: 7 + 6 * l])
        layers.append(dict(w_router=w_router, w_gate_up=w_gate_up, w_down=w_down,
                           ws_gate_up=ws_gate_up, ws_down=ws_down))
    h0 = to_h(x0f)
    mean_h = float(bf16_value(h0).astype(np.float64).mean())
    for l in range(w.layers):
        rank = r_perm.permutation(d.E)              # expert e gets zipf rank rank[e]
        shift = beta[rank] / (d.H * mean_h)
        wr = bf16_value(layers[l]["w_router"]).astype(np.float64) + shift[:, None]
        layers[l]["w_router"] = bf16_bits(wr.astype(np.float32))
        layers[l]["zipf_rank"] = rank
    n = 0
    if row_ok is not None:
        wr0 = layers[0]["w_router"]
        for _ in range(max_rounds):
            ok = np.asarray(row_ok(h0, wr0), dtype=bool)
            bad = np.nonzero(~ok)[0]
            if bad.size == 0:
                break
            x0f[bad] = draw(r_x, bad.size)
            h0 = to_h(x0f)
            n += int(bad.size)
        else:
            raise RuntimeError("row predicate still failing")
    x0 = bf16_bits(x0f.astype(np.float32))
    return dict(dims=d, x0=x0, h0=h0, layers=layers, resampled=n)


# --------------------------------------------------------------------------- verify logits
def verify_logits(B: int, K: int, V: int, seed: int, std: float = 2.0, tie_frac: float = 0.25):
    """Verifier logits [B, K+1, V] in bf16 bits with a planted greedy token per row.

    Every row is drawn N(0, std) and rounded to bf16; one uniformly chosen
    index g is then raised to the next bf16 above the row's largest value, so
    g is the unique maximum.  In about tie_frac of the rows a second uniformly
    chosen index h != g is set to the same value; the greedy token with ties
    going to the lower index is then min(g, h).  Returns (logits, planted).
    """
    r_val, r_g, r_tie = streams(seed, 3)
    R = B * (K + 1)
    logits = np.empty((R, V), dtype=np.uint16)
    chunk = max(1, (1 << 24) // max(V, 1))
    for r0 in range(0, R, chunk):
        r1 = min(R, r0 + chunk)
        logits[r0:r1] = _normal_bf16(r_val, (r1 - r0, V), std)
    g = r_g.integers(0, V, size=R)
    top = bf16_bits(bf16_value(logits).max(axis=1))
    logits[np.arange(R), g] = bf16_next_up(top)
    planted = g.copy()
    if V > 1:
        tie = r_tie.random(R) < tie_frac
        h = (g + 1 + r_tie.integers(0, V - 1, size=R)) % V
        rows = np.nonzero(tie)[0]
        logits[rows, h[rows]] = logits[rows, g[rows]]
        planted[rows] = np.minimum(g[rows], h[rows])
    return logits.reshape(B, K + 1, V), planted.reshape(B, K + 1).astype(np.int32)


def draft_tokens(planted: np.ndarray, V: int, probs, seed: int) -> np.ndarray:
    """Drafts [B, K]: draft j equals planted[b, j] with probability probs[j],
    independently per position, else a uniform token among the other V-1."""
    B, K1 = planted.shape
    K = K1 - 1
    (rng,) = streams(seed + 0x5EED, 1)
    p = np.asarray(probs, dtype=np.float64)[:K]
    hit = rng.random((B, K)) < p[None, :]
    other = (planted[:, :K] + 1 + rng.integers(0, max(V - 1, 1), size=(B, K))) % V
    return np.where(hit, planted[:, :K], other).astype(np.int32)


def verify_problem(w: Workload, seed: int = 0):
    """Logits, planted greedy tokens and drafts for w's (B, K, V)."""
    logits, planted = verify_logits(w.B, w.K, w.V, seed)
    drafts = draft_tokens(planted, w.V, w.accept, seed)
    return logits, planted, drafts


# --------------------------------------------------------------------------- verifier output layer
@dataclass
class LmHeadProblem:
    B: int
    K: int
    V: int
    H: int
    hidden: np.ndarray    # [B*(K+1), H] bf16 bits: the verifier's last hidden states
    w_vocab: np.ndarray   # [V, H] bf16 bits
    greedy: np.ndarray    # [B, K+1] greedy tokens as the caller's row check found them
    drafts: np.ndarray    # [B, K] int32
    redrawn: int


def lmhead_problem(B: int, K: int, V: int = VOCAB, H: int = 1280, seed: int = 0, row_check=None,
                   accept=PAGE_ACCEPT, max_rounds: int = 200) -> LmHeadProblem:
    """The verifier's output layer as the source of the verify logits.

    w_vocab ~ N(0, 0.02) and hidden rows = RMSNorm(N(0, 1)), both in bf16.
    row_check(hidden, w_vocab) -> (greedy [R], ok [R]) comes from the caller (this module does
    none of the method's arithmetic): rows it rejects are redrawn, and the drafts are drawn
    from its greedy tokens with the conditional acceptances `accept`, as for the synthetic
    logits.  Without a row check the greedy tokens are unknown and the drafts are uniform.
    """
    rs = streams(seed, 3)
    w_vocab = np.empty((V, H), dtype=np.uint16)
    for v0 in range(0, V, 16384):             # bounded float32 temporaries
        w_vocab[v0:v0 + 16384] = _normal_bf16(rs[0], (min(16384, V - v0), H), 0.02)
    hidden = hidden_rows(rs[1], B * (K + 1), H, "sphere")
    redrawn = 0
    greedy = np.zeros(B * (K + 1), np.int32)
    if row_check is not None:
        for _ in range(max_rounds):
            greedy, ok = row_check(hidden, w_vocab)
            bad = np.nonzero(~np.asarray(ok, bool))[0]
            if bad.size == 0:
                break
            hidden[bad] = hidden_rows(rs[1], bad.size, H, "sphere")
            redrawn += int(bad.size)
        else:
            raise RuntimeError("row predicate still failing after %d rounds" % max_rounds)
    greedy = np.asarray(greedy, np.int32).reshape(B, K + 1)
    probs = list(accept[:K]) + [accept[-1]] * max(0, K - len(accept))
    drafts = draft_tokens(greedy, V, probs, seed + 7)
    return LmHeadProblem(B, K, V, H, hidden, w_vocab, greedy, drafts, redrawn)


# --------------------------------------------------------------------------- verify attention
# Decoder prefix of a page: 256 visual tokens for the 1024x1024 view plus up to nine local
# tiles of 100 tokens (at most 1,156), then the page's text so far (about 1,085 output tokens
# per page); jina-ocr-v1 coverage on kg.zhiyong.dev, "The first layer is the visual input" and
# the throughput paragraph.
VISUAL_BASE, VISUAL_TILE, VISUAL_MAX_TILES = 256, 100, 9
PAGE_TEXT_TOKENS = 1_085
ATTN_HEADS, ATTN_HEAD_DIM = 10, 128   # hidden 1280 = 10 heads x 128


@dataclass
class AttentionProblem:
    B: int
    Q: int
    L: int
    nh: int
    d: int
    q: np.ndarray         # [B, Q, nh, d] bf16 bits
    k_cache: np.ndarray   # [B, L, nh, d] bf16 bits
    v_cache: np.ndarray   # [B, L, nh, d] bf16 bits
    ctx_len: np.ndarray   # [B] int32, Q <= ctx_len <= L


def page_context_lengths(rng, B: int, Q: int) -> np.ndarray:
    """Cache entries per sequence in the verify pass: the visual prefix (256 + 100 x a uniform
    number of tiles in 0..9), a uniform point of the page's ~1,085 text tokens, and the Q
    verified positions themselves."""
    vis = VISUAL_BASE + VISUAL_TILE * rng.integers(0, VISUAL_MAX_TILES + 1, size=B)
    txt = rng.integers(0, PAGE_TEXT_TOKENS + 1, size=B)
    return (vis + txt + Q).astype(np.int32)


def page_cache_capacity(Q: int, align: int = 64) -> int:
    n = VISUAL_BASE + VISUAL_TILE * VISUAL_MAX_TILES + PAGE_TEXT_TOKENS + Q
    return (n + align - 1) // align * align


def attention_problem(B: int, Q: int, nh: int = ATTN_HEADS, d: int = ATTN_HEAD_DIM, L: int | None = None,
                      ctx_len=None, seed: int = 0, qk_std: float = 1.0) -> AttentionProblem:
    """q, k ~ N(0, qk_std) and v ~ N(0, 1) in bf16 (at scale 1/sqrt(d) the scores have a standard
    deviation of about qk_std^2).  The cache past each sequence's length holds the same draws; the
    attention must not read it.
    ctx_len defaults to the page recipe above and L to its capacity."""
    rs = streams(seed, 4)
    if ctx_len is None:
        ctx_len = page_context_lengths(rs[3], B, Q)
    ctx_len = np.asarray(ctx_len, np.int32)
    if L is None:
        L = page_cache_capacity(Q)
    q = _normal_bf16(rs[0], (B, Q, nh, d), qk_std)
    k = _normal_bf16(rs[1], (B, L, nh, d), qk_std)
    v = _normal_bf16(rs[2], (B, L, nh, d), 1.0)
    return AttentionProblem(B, Q, L, nh, d, q, k, v, ctx_len)


# --------------------------------------------------------------------------- FastMTP draft block
DRAFT_FFN = 7_168   # (top-6 + 2 shared) x 896: the width the MoE layer activates per token


@dataclass
class DraftProblem:
    B: int
    K: int
    H: int
    nh: int
    I: int
    V: int
    L: int
    weights: dict        # bf16 bits: emb, w_proj, w_q, w_k, w_v, w_o, w_gate_up, w_down, w_vocab
    h0: np.ndarray       # [B, H] bf16 bits: the verifier's last hidden state of every sequence
    t0: np.ndarray       # [B] int32: the last committed token
    k_cache: np.ndarray  # [B, L, nh, d] bf16 bits: the draft block's own cache
    v_cache: np.ndarray
    ctx_len: np.ndarray  # [B] int32 entries already in the block's cache (room for K more)


def draft_problem(B: int, K: int = 3, H: int = 1280, nh: int = ATTN_HEADS, I: int = DRAFT_FFN, V: int = VOCAB,
                  seed: int = 0, lens=None, std: float = 0.02) -> DraftProblem:
    """Synthetic inputs of the recursive draft block: weights N(0, std) (the embedding N(0, 1)),
    unit-RMS hidden states, uniform last tokens, block caches N(0, 1) with the page recipe's
    lengths (visual prefix + text so far) and room for the K appended entries."""
    rs = streams(seed, 14)
    names = ["w_proj", "w_q", "w_k", "w_v", "w_o", "w_gate_up", "w_down", "w_vocab"]
    shapes = [(H, 2 * H), (H, H), (H, H), (H, H), (H, H), (2 * I, H), (H, I), (V, H)]
    wts = {n: _normal_bf16(r, s, std) for n, s, r in zip(names, shapes, rs[:8])}
    wts["emb"] = _normal_bf16(rs[8], (V, H), 1.0)
    h0 = hidden_rows(rs[9], B, H, "sphere")
    t0 = rs[10].integers(0, V, size=B).astype(np.int32)
    if lens is None:
        lens = page_context_lengths(rs[11], B, 1) - 1
    lens = np.asarray(lens, np.int32)
    L = (int(lens.max()) + K + 63) // 64 * 64
    d = H // nh
    kc = _normal_bf16(rs[12], (B, L, nh, d), 1.0)
    vc = _normal_bf16(rs[13], (B, L, nh, d), 1.0)
    return DraftProblem(B, K, H, nh, I, V, L, wts, h0, t0, kc, vc, lens)


# --------------------------------------------------------------------------- a decoder around the verify step
@dataclass
class DecoderProblem:
    layers: list         # per layer: dict of bf16 bits w_q, w_k, w_v, w_o [H, H] and the MoE weights
    emb: np.ndarray      # [V, H] token embedding (shared with the draft block)
    w_vocab: np.ndarray  # [V, H] output layer (shared with the draft block)
    draft: dict          # the draft block's weights (emb and w_vocab included)
    dims: MoeDims        # the MoE layer's H, E, k, S, I (T unused)
    nh: int
    V: int
    I_draft: int


def decoder_problem(n_layers: int, dims: MoeDims, V: int, nh: int = ATTN_HEADS, I_draft: int = DRAFT_FFN,
                    seed: int = 0, out_scale: float = 1.0, mimic_draft: bool = False,
                    std: float = 0.02) -> DecoderProblem:
    """Synthetic weights of an n_layers decoder (attention block + MoE FFN per layer) and its draft
    block, all N(0, std) in bf16 except the embedding N(0, 1).

    out_scale multiplies the two projections that write into the residual stream (W_o and the
    experts' down projections), so that at out_scale < 1 the stream stays close to the token
    embedding.  mimic_draft sets the draft block to pass the embedding of its input token
    through (W_p = [0 | I], W_o = 0, W_down = 0): it then proposes the greedy token of the
    embedding alone, which the verifier agrees with more often the smaller out_scale is."""
    H = dims.H
    rs = streams(seed, 4 + n_layers * 9 + 8)
    emb = _normal_bf16(rs[0], (V, H), 1.0)
    w_vocab = _normal_bf16(rs[1], (V, H), std)
    layers = []
    for l in range(n_layers):
        r = rs[4 + 9 * l: 13 + 9 * l]
        w_router, w_gate_up, w_down, ws_gate_up, ws_down = moe_weights(dims, r[4:9], std)
        if out_scale != 1.0:
            w_down = bf16_bits(bf16_value(w_down) * np.float32(out_scale))
            ws_down = bf16_bits(bf16_value(ws_down) * np.float32(out_scale))
        layers.append(dict(w_q=_normal_bf16(r[0], (H, H), std), w_k=_normal_bf16(r[1], (H, H), std),
                           w_v=_normal_bf16(r[2], (H, H), std), w_o=_normal_bf16(r[3], (H, H), std * out_scale),
                           w_router=w_router, w_gate_up=w_gate_up, w_down=w_down, ws_gate_up=ws_gate_up,
                           ws_down=ws_down))
    rd = rs[4 + 9 * n_layers:]
    if mimic_draft:
        w_proj = bf16_bits(np.concatenate([np.zeros((H, H), np.float32), np.eye(H, dtype=np.float32)], axis=1))
        w_o_d = np.zeros((H, H), np.uint16)
        w_down_d = np.zeros((H, I_draft), np.uint16)
    else:
        w_proj = _normal_bf16(rd[0], (H, 2 * H), std)
        w_o_d = _normal_bf16(rd[1], (H, H), std)
        w_down_d = _normal_bf16(rd[2], (H, I_draft), std)
    draft = dict(emb=emb, w_proj=w_proj, w_q=_normal_bf16(rd[3], (H, H), std), w_k=_normal_bf16(rd[4], (H, H), std),
                 w_v=_normal_bf16(rd[5], (H, H), std), w_o=w_o_d, w_gate_up=_normal_bf16(rd[6], (2 * I_draft, H), std),
                 w_down=w_down_d, w_vocab=w_vocab)
    return DecoderProblem(layers, emb, w_vocab, draft, dims, nh, V, I_draft)
