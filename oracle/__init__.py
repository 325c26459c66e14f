"""CPU oracle for the FastMTP verification step (TEST INFRASTRUCTURE ONLY).

Plain, slow C loops (oracle.c) behind a ctypes wrapper.  Only the tests, the
smoke check and the benchmark's CPU-baseline leg may import this package; the
CUDA library never links, loads or calls it, and the two share no code.

Pins (checked by tests marked "not gpu"):
  route      -- torch.softmax / torch.topk special cases, planted one-hot
                routing, exact-tie order, brute force on tiny inputs
  route_gaps -- brute-force fp64 sort on tiny inputs
  permute    -- bincount / cumsum, bijection and sort-order invariants
  experts    -- closed form with H = I = 1, identical-expert invariant
                (k = E gives one dense SwiGLU FFN), dense brute force in
                torch fp64 with a different formulation (all experts masked)
  combine    -- closed form on hand-built inputs
  layer      -- the two above composed; shared-only and single-expert cases
  accept     -- exhaustive brute force on tiny vocabularies, planted greedy
                tokens, torch.argmax, greedy-decoding equivalence on a toy
                model, closed form of tokens per step vs the pages' 2.73
  rmsnorm    -- closed form on constant rows, torch rms_norm in fp64
  lmhead     -- pure-Python brute force on tiny inputs, a planted row that is a
                scaled copy of the hidden state, duplicated rows (first index),
                torch fp64 matmul + argmax
  attention  -- pure-Python brute force, one visible key (the output is its
                value), identical keys (the mean of the values), causality
                (later keys change nothing), torch scaled_dot_product_attention
                in fp64 with an explicit mask
  k_policy   -- the pages' tau = 2.73 / 2.74 from their conditional
                acceptances; a Monte Carlo decode loop (Bernoulli draft
                acceptances, per-K step costs) whose measured tokens per unit
                cost and best K match S = tau / c; the acceptance estimate
                recovers the simulated acceptances and tau equals the mean
                committed count
  draft_block -- torch fp64 formulation (rms_norm, linear,
                scaled_dot_product_attention, silu, argmax); with attention
                and FFN switched off it is the (pinned) output-layer oracle;
                zero queries give the mean of the visible values; the K-step
                loop is the chained block; its drafts, verified by the
                acceptance rule against a toy verifier, commit exactly the
                verifier's greedy sequence.  It is the plain definition in
                float64: no value is rounded to bf16 anywhere in it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library next to it (gcc, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i = ctypes.c_int
            sig = {
                "oracle_route": [P, P, i, i, i, i, P, P, P],
                "oracle_route_gaps": [P, P, i, i, i, i, P],
                "oracle_permute": [P, i, i, i, P, P, P, P],
                "oracle_expert_rows": [P, P, P, i, i, i, P, P, i, P],
                "oracle_shared_rows": [P, P, P, i, i, i, P, i, P],
                "oracle_combine": [P, P, P, P, i, i, i, P],
                "oracle_moe_layer": [P, P, P, P, P, P, i, i, i, i, i, i, P, i, P, P, P],
                "oracle_rmsnorm_residual": [P, P, i, i, ctypes.c_double, P, P],
                "oracle_accept": [P, P, i, i, i, P, P, P],
            }
            for name, args in sig.items():
                f = getattr(_lib, name)
                f.argtypes = args
                f.restype = ctypes.c_int
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, name):
    if rc != 0:
        raise ValueError("%s failed with code %d" % (name, rc))


def route(x, w_router, k, return_logits=False):
    """Top-k routing of every token row of x (bf16 bits [T,H]) by w_router ([E,H])."""
    x = _c(x, np.uint16); w = _c(w_router, np.uint16)
    T, H = x.shape
    E = w.shape[0]
    idx = np.zeros((T, k), np.int32)
    p = np.zeros((T, k), np.float64)
    logits = np.zeros((T, E), np.float32) if return_logits else None
    _check(_load().oracle_route(_p(x), _p(w), T, H, E, k, _p(idx), _p(p), _p(logits)), "route")
    return (idx, p, logits) if return_logits else (idx, p)


def route_gaps(x, w_router, k):
    x = _c(x, np.uint16); w = _c(w_router, np.uint16)
    T, H = x.shape
    gap = np.zeros(T, np.float64)
    _check(_load().oracle_route_gaps(_p(x), _p(w), T, H, w.shape[0], k, _p(gap)), "route_gaps")
    return gap


def gap_ok(k, min_gap=1e-3):
    """Row predicate for the input generator: consecutive router places >= min_gap apart."""
    return lambda x, w_router: route_gaps(x, w_router, k) >= min_gap


def permute(topk_idx, E):
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    inv = np.zeros(T * k, np.int32)
    _check(_load().oracle_permute(_p(idx), T, k, E, _p(counts), _p(offsets), _p(perm), _p(inv)), "permute")
    return counts, offsets, perm, inv


def expert_rows(x, w_gate_up, w_down, token, expert):
    x = _c(x, np.uint16); wgu = _c(w_gate_up, np.uint16); wd = _c(w_down, np.uint16)
    token = _c(token, np.int32); expert = _c(expert, np.int32)
    E, I2, H = wgu.shape
    y = np.zeros((token.size, H), np.float64)
    _check(_load().oracle_expert_rows(_p(x), _p(wgu), _p(wd), H, I2 // 2, E, _p(token), _p(expert),
                                      token.size, _p(y)), "expert_rows")
    return y


def shared_rows(x, ws_gate_up, ws_down, S, token=None):
    x = _c(x, np.uint16); wgu = _c(ws_gate_up, np.uint16); wd = _c(ws_down, np.uint16)
    T, H = x.shape
    token = np.arange(T, dtype=np.int32) if token is None else _c(token, np.int32)
    I = wgu.shape[0] // (2 * S) if S > 0 else 1
    y = np.zeros((token.size, H), np.float64)
    _check(_load().oracle_shared_rows(_p(x), _p(wgu), _p(wd), H, I, S, _p(token), token.size, _p(y)),
           "shared_rows")
    return y


def combine(y_perm, inv, topk_w, y_shared, T, k):
    yp = _c(y_perm, np.float32); inv = _c(inv, np.int32); w = _c(topk_w, np.float32)
    ys = None if y_shared is None else _c(y_shared, np.float32)
    H = yp.shape[1]
    out = np.zeros((T, H), np.float64)
    _check(_load().oracle_combine(_p(yp), _p(inv), _p(w), _p(ys), T, k, H, _p(out)), "combine")
    return out


def moe_layer(x, w_router, w_gate_up, w_down, ws_gate_up, ws_down, k, S, tokens=None):
    """MoE layer output (double) for the listed tokens (all when None), plus routing."""
    x = _c(x, np.uint16)
    T, H = x.shape
    E = w_router.shape[0]
    I = w_gate_up.shape[1] // 2
    tok = None if tokens is None else _c(tokens, np.int32)
    n = T if tok is None else tok.size
    out = np.zeros((n, H), np.float64)
    idx = np.zeros((n, k), np.int32)
    w = np.zeros((n, k), np.float64)
    wsg = _c(ws_gate_up, np.uint16) if S > 0 else np.zeros(1, np.uint16)
    wsd = _c(ws_down, np.uint16) if S > 0 else np.zeros(1, np.uint16)
    _check(_load().oracle_moe_layer(_p(x), _p(_c(w_router, np.uint16)), _p(_c(w_gate_up, np.uint16)),
                                    _p(_c(w_down, np.uint16)), _p(wsg), _p(wsd), T, H, E, k, S, I,
                                    _p(tok), n, _p(out), _p(idx), _p(w)), "moe_layer")
    return out, idx, w


def rmsnorm_residual(x, y, eps=1e-6):
    x = _c(x, np.uint16); y = _c(y, np.uint16)
    T, H = x.shape
    xn = np.zeros((T, H), np.float64)
    hn = np.zeros((T, H), np.float64)
    _check(_load().oracle_rmsnorm_residual(_p(x), _p(y), T, H, eps, _p(xn), _p(hn)), "rmsnorm_residual")
    return xn, hn


def accept(logits, drafts):
    """Greedy verification: logits [B,K+1,V] bf16 bits, drafts [B,K] int32."""
    lg = _c(logits, np.uint16); d = _c(drafts, np.int32)
    B, K1, V = lg.shape
    K = K1 - 1
    if d.shape != (B, K):
        raise ValueError("drafts must be [B,K]")
    argmax = np.zeros((B, K1), np.int32)
    alen = np.zeros(B, np.int32)
    committed = np.zeros((B, K1), np.int32)
    _check(_load().oracle_accept(_p(lg), _p(d), B, K, V, _p(argmax), _p(alen), _p(committed)), "accept")
    return argmax, alen, committed


# ----------------------------------------------------------------------------- verifier output layer
def lmhead_argmax(hidden, w_vocab, chunk=8192):
    """Greedy tokens of the verifier's output layer, straight from its definition.

    logit[r, v] = sum_h hidden[r, h] * w_vocab[v, h], evaluated in fp64 from the exact bf16
    inputs (numpy's matmul is the only step taken from a library); g[r] = the first index
    attaining the row maximum; gap[r] = that maximum minus the largest logit of any other
    index (0 when the maximum is attained twice).  hidden [R, H] as bf16 bits (or float64
    values), w_vocab [V, H] as bf16 bits.
    """
    hidden = np.asarray(hidden)
    hf = hidden if hidden.dtype == np.float64 else _bf16_to_f64(_c(hidden, np.uint16))
    wv = _c(w_vocab, np.uint16)
    R, H = hf.shape
    V = wv.shape[0]
    best = np.full(R, -np.inf)
    second = np.full(R, -np.inf)
    g = np.zeros(R, np.int64)
    for v0 in range(0, V, chunk):
        lg = hf @ _bf16_to_f64(wv[v0:v0 + chunk]).T              # [R, n]
        i = np.argmax(lg, axis=1)                                # first occurrence within the chunk
        m = lg[np.arange(R), i]
        lg[np.arange(R), i] = -np.inf
        m2 = lg.max(axis=1)
        # merge with the running (best, second): the earlier chunk wins ties (lower index)
        new = m > best
        second = np.where(new, np.maximum(best, m2), np.maximum(second, m))
        g = np.where(new, v0 + i, g)
        best = np.where(new, m, best)
    return g.astype(np.int32), best - second


def lmhead_row_check(min_gap=1e-3):
    """For the input generator: (greedy tokens, rows whose top-2 logits are >= min_gap apart)."""
    def row_check(hidden, w_vocab):
        g, gap = lmhead_argmax(hidden, w_vocab)
        return g, gap >= min_gap
    return row_check


def _bf16_to_f64(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def accept_from_greedy(greedy, drafts):
    """The acceptance rule of `accept` applied to given greedy tokens greedy [B, K+1]."""
    g = np.asarray(greedy, np.int64)
    d = np.asarray(drafts, np.int64)
    B, K1 = g.shape
    K = K1 - 1
    alen = np.zeros(B, np.int32)
    committed = np.full((B, K1), -1, np.int32)
    for b in range(B):
        L = 0
        while L < K and d[b, L] == g[b, L]:
            L += 1
        alen[b] = L
        committed[b, :L] = d[b, :L]
        committed[b, L] = g[b, L]
    return alen, committed


# ----------------------------------------------------------------------------- verify attention
def verify_attention(q, k_cache, v_cache, ctx_len, scale):
    """Causal attention of the Q verified positions over their sequence's cache, from its
    definition, in fp64 from the exact bf16 inputs.

    q [B, Q, nh, d]; k_cache, v_cache [B, L, nh, d] (bf16 bits); ctx_len [B]: cache entries of
    sequence b, the last Q of which belong to the verified positions.  Query j of sequence b
    sits at position p = ctx_len[b] - Q + j and sees keys 0..p:
        out[b, j, h] = sum_{t <= p} softmax_t(scale * q[b,j,h] . k[b,t,h]) * v[b,t,h]
    Returns out [B, Q, nh, d] float64.
    """
    qf = _bf16_to_f64(_c(q, np.uint16))
    kf = _bf16_to_f64(_c(k_cache, np.uint16))
    vf = _bf16_to_f64(_c(v_cache, np.uint16))
    B, Q, nh, d = qf.shape
    out = np.zeros((B, Q, nh, d), np.float64)
    for b in range(B):
        n = int(ctx_len[b])
        if n < Q or n > kf.shape[1]:
            raise ValueError("ctx_len[%d] = %d outside [Q, L]" % (b, n))
        for j in range(Q):
            p = n - Q + j
            s = np.einsum("hd,thd->ht", qf[b, j], kf[b, :p + 1]) * scale     # [nh, p+1]
            s -= s.max(axis=1, keepdims=True)
            w = np.exp(s)
            w /= w.sum(axis=1, keepdims=True)
            out[b, j] = np.einsum("ht,thd->hd", w, vf[b, :p + 1])
    return out


# ----------------------------------------------------------------------------- K policy
def k_policy(cond_accept, step_cost):
    """The number of drafts K that maximises the speedup S = tau / c (evolve.pub review,
    Table 8 decomposition), from conditional acceptances a_1..a_kmax and the costs c_0..c_kmax
    of a step with K drafts (c_0: a plain greedy step).

    tau(K) = 1 + a_1 + a_1 a_2 + ... + a_1 ... a_K (tokens a step commits on average: the
    accepted prefix plus the correction or bonus token), S(K) = tau(K) c_0 / c_K.
    Returns (k_best, tau [kmax+1], S [kmax+1]); equal speedups keep the smaller K.
    """
    a = [float(x) for x in cond_accept]
    c = [float(x) for x in step_cost]
    assert len(c) == len(a) + 1
    tau = []
    for K in range(len(c)):
        prefix_probs = [float(np.prod(a[:i])) for i in range(K + 1)]   # P(first i drafts accepted)
        tau.append(sum(prefix_probs))
    S = [tau[K] * c[0] / c[K] for K in range(len(c))]
    k_best = 0
    for K in range(1, len(c)):
        if S[K] > S[k_best]:
            k_best = K
    return k_best, np.array(tau), np.array(S)


def cond_accept_from_lengths(lengths, K):
    """a_i = P(draft i accepted | drafts 1..i-1 accepted), counted from accepted lengths L:
    #(L >= i) / #(L >= i-1) for i = 1..K (0 where no step reached draft i)."""
    L = np.asarray(lengths, np.int64)
    out = []
    for i in range(1, K + 1):
        reached = int(np.count_nonzero(L >= i - 1))
        out.append(np.count_nonzero(L >= i) / reached if reached else 0.0)
    return np.array(out)


# ----------------------------------------------------------------------------- FastMTP draft block
def _rms64(x, eps=1e-6):
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)


def _silu64(z):
    return z / (1.0 + np.exp(-z))


def draft_block(h_prev, tok_prev, w, k_cache, v_cache, ctx_len, nh, eps=1e-6):
    """One application of the shared FastMTP draft block to every sequence (kg.zhiyong.dev, "The
    speed comes from three layers working together": one dense draft block proposes the drafts;
    evolve.pub review, "Scope & Claims": one shared block applied recursively).

    The pages fix no more than that; the reading (an MTP module of the decoder's family):
        u  = W_p [RMSNorm(h_prev); RMSNorm(E[tok_prev])]
        a  = RMSNorm(u);  q, k, v = W_q a, W_k a, W_v a       (nh heads of d = H / nh)
        the block's cache of the sequence gets k, v at position ctx_len[b]; q attends to
        positions 0..ctx_len[b] (softmax with scale 1/sqrt(d))
        u  = u + W_o attn
        f  = RMSNorm(u);  u = u + W_down (silu(W_gate f) * (W_up f))
        h_next = u;  draft = argmax_v (W_vocab RMSNorm(u))_v   (the first index of the maximum)
    RMSNorm has unit weight.  Everything is evaluated in float64 from the exact bf16 weights and
    inputs; nothing is rounded on the way (the definition, not any storage format).

    h_prev [B, H] float64 or bf16 bits; tok_prev [B] int; w: dict of bf16-bit arrays emb [V, H],
    w_proj [H, 2H], w_q, w_k, w_v, w_o [H, H], w_gate_up [2I, H] (gate rows, then up rows),
    w_down [H, I], w_vocab [V, H]; k_cache, v_cache [B, L, nh, d] float64 (updated in place at
    position ctx_len[b]); ctx_len [B].
    Returns (h_next [B, H] float64, draft [B] int32, gap [B]: top-two logit difference).
    """
    f64 = lambda u: _bf16_to_f64(w[u]) if w[u].dtype == np.uint16 else np.asarray(w[u], np.float64)
    h = np.asarray(h_prev, np.float64) if np.asarray(h_prev).dtype != np.uint16 else _bf16_to_f64(h_prev)
    B, H = h.shape
    d = H // nh
    E = f64("emb")
    Wp, Wq, Wk, Wv, Wo = f64("w_proj"), f64("w_q"), f64("w_k"), f64("w_v"), f64("w_o")
    Wgu, Wd, Wv_out = f64("w_gate_up"), f64("w_down"), f64("w_vocab")
    I = Wd.shape[1]
    tok = np.asarray(tok_prev, np.int64)
    inp = np.concatenate([_rms64(h, eps), _rms64(E[tok], eps)], axis=1)         # [B, 2H]
    u = inp @ Wp.T
    a = _rms64(u, eps)
    q, k, v = a @ Wq.T, a @ Wk.T, a @ Wv.T
    attn = np.zeros((B, H))
    for b in range(B):
        n = int(ctx_len[b])
        k_cache[b, n] = k[b].reshape(nh, d)
        v_cache[b, n] = v[b].reshape(nh, d)
        qs = q[b].reshape(nh, d)
        s = np.einsum("hd,thd->ht", qs, k_cache[b, :n + 1]) / np.sqrt(d)
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        attn[b] = np.einsum("ht,thd->hd", p, v_cache[b, :n + 1]).reshape(H)
    u = u + attn @ Wo.T
    f = _rms64(u, eps)
    act = _silu64(f @ Wgu[:I].T) * (f @ Wgu[I:].T)
    u = u + act @ Wd.T
    hn = _rms64(u, eps)
    logits = hn @ Wv_out.T
    draft = np.argmax(logits, axis=1).astype(np.int32)
    top2 = np.sort(logits, axis=1)[:, -2:] if logits.shape[1] > 1 else np.concatenate([logits, logits], 1)
    return u, draft, top2[:, 1] - top2[:, 0]


def draft_loop(h0, t0, w, k_cache, v_cache, ctx_len, nh, K, return_state=False):
    """K recursive applications of the draft block: step i takes step i-1's output state and
    draft token (step 1: the verifier's last hidden state and the last committed token), and
    appends to the block's cache at ctx_len + i - 1.  Returns (drafts [B, K], gaps [B, K]),
    plus the last state [B, H] with return_state."""
    h = h0
    t = np.asarray(t0, np.int64)
    n = np.asarray(ctx_len, np.int64).copy()
    B = n.size
    drafts = np.zeros((B, K), np.int32)
    gaps = np.zeros((B, K))
    for i in range(K):
        h, t, g = draft_block(h, t, w, k_cache, v_cache, n, nh)
        drafts[:, i] = t
        gaps[:, i] = g
        n += 1
    return (drafts, gaps, h) if return_state else (drafts, gaps)
