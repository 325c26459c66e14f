"""Pins for the CPU oracle: every check ties it to something other than itself
(page numbers, closed forms, invariants, library special cases, brute force
in a different formulation).  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from lossless_speculative_verification_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(a):
    return synth.bf16_bits(np.asarray(a, dtype=np.float32))


def val64(u):
    return synth.bf16_value(u).astype(np.float64)


def tiny_problem(T=12, H=32, E=8, k=2, S=1, I=16, seed=0, std=0.3):
    """Small layer with bigger weights than the workloads so that outputs are O(1)."""
    rs = synth.streams(seed, 6)
    d = synth.MoeDims(T, H, E, k, S, I)
    w = [bits(r.standard_normal(s) * std) for r, s in zip(
        rs[:5], [(E, H), (E, 2 * I, H), (E, H, I), (2 * S * I, H), (H, S * I)])]
    x = bits(rs[5].standard_normal((T, H)))
    return d, x, w


# ----------------------------------------------------------------------------- router
def test_route_matches_torch_softmax_and_topk():
    d, x, (wr, *_rest) = tiny_problem(T=64, E=16, k=4)
    gaps = oracle.route_gaps(x, wr, d.k)
    keep = gaps >= 1e-3
    idx, p = oracle.route(x, wr, d.k)
    logits = torch.from_numpy(val64(x)) @ torch.from_numpy(val64(wr)).T
    prob = torch.softmax(logits, dim=-1)
    tv, ti = torch.topk(logits, d.k, dim=-1)
    assert keep.sum() > 40
    np.testing.assert_array_equal(idx[keep], ti.numpy()[keep])
    ref_p = torch.gather(prob, 1, torch.from_numpy(idx).long()).numpy()
    np.testing.assert_allclose(p, ref_p, rtol=1e-5, atol=1e-7)


def test_route_planted_one_hot():
    # x = unit vector at column c, so the router score of expert e is W_r[e, c].
    E, H, k, c = 10, 24, 4, 7
    order = np.array([3, 8, 0, 5, 9, 1, 2, 4, 6, 7])          # planted ranking
    wr = np.zeros((E, H), np.float32)
    wr[order, c] = 2.25 - 0.25 * np.arange(E)                  # bf16-exact steps of 0.25
    wr[:, (c + 1) % H] = 5.0                                   # decoy column: a transposed product would see it
    x = np.zeros((1, H), np.float32)
    x[0, c] = 1.0
    idx, p = oracle.route(bits(x), bits(wr), k)
    np.testing.assert_array_equal(idx[0], order[:k])
    s = 2.25 - 0.25 * np.arange(E)
    z = np.exp(s - s.max())
    np.testing.assert_allclose(p[0], (z / z.sum())[:k], rtol=1e-12)


def test_route_ties_go_to_lower_index_and_softmax_sums_to_one():
    E, H = 8, 16
    rs = np.random.default_rng(3)
    row = rs.standard_normal(H)
    wr = np.tile(row, (E, 1))                                  # all experts identical: all scores tie
    x = bits(rs.standard_normal((5, H)))
    idx, p = oracle.route(x, bits(wr), E)
    np.testing.assert_array_equal(idx, np.tile(np.arange(E), (5, 1)))
    np.testing.assert_allclose(p, 1.0 / E, rtol=1e-12)
    # two duplicated rows among distinct ones: the lower index comes first
    wr2 = rs.standard_normal((E, H))
    wr2[6] = wr2[2]
    x1 = np.zeros((1, H)); x1[0] = wr2[2]                      # makes expert 2 (and 6) the largest score
    idx2, p2 = oracle.route(bits(x1), bits(wr2), 3)
    assert list(idx2[0][:2]) == [2, 6]
    assert p2[0][0] == p2[0][1]
    # with k = E the selected probabilities are the whole softmax
    _, xx, (wr3, *_r) = tiny_problem(T=9, E=8, k=8)
    _, p3 = oracle.route(xx, wr3, 8)
    np.testing.assert_allclose(p3.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(p3, axis=1) <= 0)


def test_route_gaps_brute_force():
    d, x, (wr, *_r) = tiny_problem(T=20, E=9, k=3)
    got = oracle.route_gaps(x, wr, d.k)
    for t in range(d.T):
        v = sorted((float(np.dot(val64(x[t]), val64(wr[e]))) for e in range(d.E)), reverse=True)
        want = min(v[p] - v[p + 1] for p in range(d.k))
        assert got[t] == pytest.approx(want, rel=1e-12, abs=1e-15)


# ----------------------------------------------------------------------------- permutation
@pytest.mark.parametrize("T,k,E", [(16, 2, 8), (128, 6, 64), (1, 1, 1), (0, 3, 4), (37, 5, 7)])
def test_permute_invariants(T, k, E):
    rs = np.random.default_rng(T * 31 + k)
    idx = np.array([rs.permutation(E)[:k] for _ in range(T)], dtype=np.int32).reshape(T, k)
    counts, offsets, perm, inv = oracle.permute(idx, E)
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    assert sorted(perm.tolist()) == list(range(T * k))
    np.testing.assert_array_equal(inv[perm], np.arange(T * k))
    # expert-major, then token-ascending: the stable sort of entries by expert
    np.testing.assert_array_equal(perm, np.argsort(flat, kind="stable"))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg // max(k, 1)) > 0)


def test_permute_rejects_out_of_range():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 4]], np.int32), 4)


# ----------------------------------------------------------------------------- experts
SIGMOID_2 = 0.8807970779778823   # 1/(1+e^-2)
SIGMOID_HALF = 0.6224593312018546  # 1/(1+e^-0.5)


def test_expert_closed_form_scalar():
    # H = I = 1: E(x) = d * silu(g*x) * (u*x); gate and up swapped would give a different number
    a, g, u, dd = 1.0, 2.0, 0.5, -1.5
    wgu = bits(np.array([[[g], [u]]]))
    wd = bits(np.array([[[dd]]]))
    y = oracle.expert_rows(bits([[a]]), wgu, wd, [0], [0])
    want = dd * (g * a * SIGMOID_2) * (u * a)
    assert y[0, 0] == pytest.approx(want, rel=1e-15)
    assert want == pytest.approx(-1.3211956169668235, rel=1e-15)
    swapped = dd * (u * a * SIGMOID_HALF) * (g * a)
    assert abs(y[0, 0] - swapped) > 0.1


def dense_ffn(x64, wg, wu, wd):
    """SwiGLU FFN in torch fp64: (silu(x Wg^T) * (x Wu^T)) Wd^T."""
    return (F.silu(x64 @ wg.T) * (x64 @ wu.T)) @ wd.T


def torch_layer(x, wr, wgu, wd, wsgu, wsd, k, S):
    """The layer evaluated densely: every expert on every token, masked by the
    top-k set; a different formulation from the oracle's per-token routing."""
    X = torch.from_numpy(val64(x))
    Wr = torch.from_numpy(val64(wr))
    E = wr.shape[0]
    I = wgu.shape[1] // 2
    logits = X @ Wr.T
    P = torch.softmax(logits, dim=-1)
    mask = torch.zeros_like(P)
    if k > 0:
        mask.scatter_(1, torch.topk(logits, k, dim=-1).indices, 1.0)
    out = torch.zeros_like(X)
    for e in range(E):
        G = torch.from_numpy(val64(wgu[e]))
        Y = dense_ffn(X, G[:I], G[I:], torch.from_numpy(val64(wd[e])))
        out += (mask[:, e] * P[:, e])[:, None] * Y
    if S > 0:
        G = torch.from_numpy(val64(wsgu))
        D = torch.from_numpy(val64(wsd))
        for s in range(S):
            out += dense_ffn(X, G[s * I:(s + 1) * I], G[S * I + s * I:S * I + (s + 1) * I], D[:, s * I:(s + 1) * I])
    return out.numpy()


@pytest.mark.parametrize("shape", [dict(T=12, H=32, E=8, k=2, S=1, I=16),
                                   dict(T=9, H=24, E=6, k=3, S=2, I=8),
                                   dict(T=5, H=16, E=4, k=4, S=0, I=32)])
def test_layer_vs_dense_torch(shape):
    d, x, (wr, wgu, wd, wsgu, wsd) = tiny_problem(**shape, seed=11)
    gaps = oracle.route_gaps(x, wr, d.k)
    out, idx, p = oracle.moe_layer(x, wr, wgu, wd, wsgu, wsd, d.k, d.S)
    ref = torch_layer(x, wr, wgu, wd, wsgu, wsd, d.k, d.S)
    keep = gaps >= 1e-3
    assert keep.sum() >= d.T // 2
    # the oracle's gate uses float router scores (the kernel's precision); torch's are fp64
    np.testing.assert_allclose(out[keep], ref[keep], rtol=1e-5, atol=1e-6)


def test_layer_identical_experts_reduces_to_dense_ffn():
    d, x, (wr, wgu, wd, wsgu, wsd) = tiny_problem(T=10, H=32, E=6, k=6, S=1, I=16, seed=5)
    wgu[:] = wgu[0]
    wd[:] = wd[0]
    X = torch.from_numpy(val64(x))
    G = torch.from_numpy(val64(wgu[0]))
    f = dense_ffn(X, G[:16], G[16:], torch.from_numpy(val64(wd[0]))).numpy()
    sh = oracle.shared_rows(x, wsgu, wsd, 1)
    # k = E: the gate probabilities sum to one, so the routed part is exactly the dense FFN
    out, _, _ = oracle.moe_layer(x, wr, wgu, wd, wsgu, wsd, 6, 1)
    np.testing.assert_allclose(out - sh, f, rtol=1e-9, atol=1e-12)
    # k < E: the routed part is (sum of the selected probabilities) x the dense FFN (no renormalisation)
    out2, _, p2 = oracle.moe_layer(x, wr, wgu, wd, wsgu, wsd, 2, 1)
    np.testing.assert_allclose(out2 - sh, p2.sum(axis=1)[:, None] * f, rtol=1e-9, atol=1e-12)
    assert np.all(p2.sum(axis=1) < 1.0)


def test_layer_special_cases():
    d, x, (wr, wgu, wd, wsgu, wsd) = tiny_problem(T=6, H=16, E=1, k=1, S=2, I=8, seed=9)
    # a single routed expert always has gate probability 1
    out, idx, p = oracle.moe_layer(x, wr, wgu, wd, wsgu, wsd, 1, 2)
    assert np.all(idx == 0) and np.allclose(p, 1.0)
    routed = oracle.expert_rows(x, wgu, wd, np.arange(6), np.zeros(6, np.int32))
    shared = oracle.shared_rows(x, wsgu, wsd, 2)
    np.testing.assert_allclose(out, routed + shared, rtol=1e-12)
    # no routed slot: the layer is its shared experts
    out0, _, _ = oracle.moe_layer(x, wr, wgu, wd, wsgu, wsd, 0, 2)
    np.testing.assert_allclose(out0, shared, rtol=1e-12)
    # two shared experts of intermediate I equal one SwiGLU of intermediate 2I built by concatenation
    X = torch.from_numpy(val64(x))
    G = torch.from_numpy(val64(wsgu))
    D = torch.from_numpy(val64(wsd))
    cat = dense_ffn(X, G[:16], G[16:], D).numpy()
    np.testing.assert_allclose(shared, cat, rtol=1e-9, atol=1e-12)


def test_combine_closed_form():
    T, k, H = 3, 2, 4
    y_perm = np.arange(T * k * H, dtype=np.float32).reshape(T * k, H) / 8
    inv = np.array([5, 0, 3, 1, 4, 2], np.int32)
    w = np.array([[0.5, 0.25], [1.0, 0.0], [0.125, 2.0]], np.float32)
    ysh = np.full((T, H), 10.0, np.float32)
    out = oracle.combine(y_perm, inv, w, ysh, T, k)
    want = np.stack([0.5 * y_perm[5] + 0.25 * y_perm[0] + 10,
                     1.0 * y_perm[3] + 0.0 * y_perm[1] + 10,
                     0.125 * y_perm[4] + 2.0 * y_perm[2] + 10])
    np.testing.assert_array_equal(out, want)


# ----------------------------------------------------------------------------- acceptance
def brute_accept(logits, drafts):
    """Committed tokens as greedy decoding writes them: g_0 .. g_L where L is the
    longest prefix of drafts equal to the greedy tokens (np.argmax: first maximum)."""
    g = np.argmax(synth.bf16_value(logits), axis=-1)
    B, K = drafts.shape
    alen = np.zeros(B, np.int32)
    comm = -np.ones((B, K + 1), np.int32)
    for b in range(B):
        L = next(L for L in range(K, -1, -1) if all(drafts[b, i] == g[b, i] for i in range(L)))
        alen[b] = L
        comm[b, :L + 1] = g[b, :L + 1]
    return g, alen, comm


@pytest.mark.parametrize("K", [0, 1, 2, 3])
def test_accept_exhaustive_tiny_vocab(K):
    V = 4
    rs = np.random.default_rng(K)
    # values from a 3-level grid so that exact ties are common
    lg = bits(rs.integers(-1, 2, size=(1, K + 1, V)).astype(np.float32))
    tuples = list(itertools.product(range(-1, V + 1), repeat=K))      # includes ids outside [0,V)
    drafts = np.array(tuples, np.int32).reshape(len(tuples), K)
    logits = np.repeat(lg, len(tuples), axis=0)
    g, alen, comm = oracle.accept(logits, drafts)
    g2, alen2, comm2 = brute_accept(logits, drafts)
    np.testing.assert_array_equal(g, g2)
    np.testing.assert_array_equal(alen, alen2)
    np.testing.assert_array_equal(comm, comm2)


def test_accept_planted_greedy_tokens_and_torch_argmax():
    for B, K, V, seed in [(4, 3, 1024, 0), (8, 2, 7, 1), (3, 1, 129_280, 2), (16, 3, 2, 3)]:
        logits, planted = synth.verify_logits(B, K, V, seed)
        g, _, _ = oracle.accept(logits, np.zeros((B, K), np.int32))
        np.testing.assert_array_equal(g, planted)
        t = torch.from_numpy(synth.bf16_value(logits).astype(np.float32))
        np.testing.assert_array_equal(g, torch.argmax(t, dim=-1).numpy())


def test_accept_all_match_gives_bonus_and_first_miss_gives_correction():
    B, K, V = 5, 3, 50
    logits, planted = synth.verify_logits(B, K, V, 7)
    g, alen, comm = oracle.accept(logits, planted[:, :K])
    assert np.all(alen == K)
    np.testing.assert_array_equal(comm, planted)                     # K drafts + the bonus token
    bad = planted[:, :K].copy()
    bad[:, 0] = (bad[:, 0] + 1) % V
    g, alen, comm = oracle.accept(logits, bad)
    assert np.all(alen == 0)
    np.testing.assert_array_equal(comm[:, 0], planted[:, 0])          # the correction token
    assert np.all(comm[:, 1:] == -1)


def toy_logits(prev2, prev1, V, table):
    """Deterministic toy language model: logits depend on the last two tokens."""
    return table[(prev2 * 131 + prev1 * 7) % table.shape[0]]


@pytest.mark.parametrize("K", [1, 2, 3])
def test_speculative_loop_equals_greedy_decoding(K):
    """The pages' lossless claim: the committed text equals plain greedy decoding."""
    V, n_tok = 13, 60
    for seed in range(12):
        rs = np.random.default_rng(100 * K + seed)
        table = bits(rs.integers(-2, 3, size=(97, V)).astype(np.float32))    # many exact ties
        # plain greedy decoding (first maximum)
        seq = [1, 2]
        while len(seq) < n_tok + 2:
            row = synth.bf16_value(toy_logits(seq[-2], seq[-1], V, table))
            seq.append(int(np.argmax(row)))
        greedy = seq[2:]
        # speculative: a corrupted greedy drafter proposes K tokens, the verifier scores K+1 positions
        out = [1, 2]
        steps = 0
        while len(out) < n_tok + 2:
            ctx = list(out)
            drafts = []
            for _ in range(K):
                row = synth.bf16_value(toy_logits(ctx[-2], ctx[-1], V, table))
                tok = int(np.argmax(row))
                if rs.random() < 0.3:
                    tok = int(rs.integers(0, V))
                drafts.append(tok)
                ctx.append(tok)
            inputs = out[-2:] + drafts
            lg = np.stack([toy_logits(inputs[j], inputs[j + 1], V, table) for j in range(K + 1)])[None]
            _, alen, comm = oracle.accept(lg, np.array([drafts], np.int32))
            out.extend(int(c) for c in comm[0, :alen[0] + 1])
            steps += 1
        assert out[2:2 + n_tok] == greedy[:n_tok]
        assert steps < n_tok


def test_tokens_per_step_closed_form_matches_pages():
    with open(os.path.join(GOLDEN, "page_numbers.json")) as f:
        pages = json.load(f)
    a = pages["conditional_accept_k3"]["value"]
    tau = 1 + a[0] + a[0] * a[1] + a[0] * a[1] * a[2]
    assert tau == pytest.approx(pages["tau_k3"]["value"], abs=0.005)
    assert (tau - 1) / 3 == pytest.approx(pages["acceptance_rate_k3"]["value"], abs=0.002)
    # Monte Carlo through the oracle with the workload's draft generator
    B, K, V = 200_000, 3, 8
    logits, planted = synth.verify_logits(B, K, V, 1234)
    drafts = synth.draft_tokens(planted, V, a, 1234)
    _, alen, _ = oracle.accept(logits, drafts)
    committed = alen + 1
    sigma = committed.std()
    assert committed.mean() == pytest.approx(tau, abs=4 * sigma / math.sqrt(B))
    # committed-count distribution: P(n) = prod a_{<n-1} (1 - a_{n-1}), P(K+1) = prod a
    pn = [1 - a[0], a[0] * (1 - a[1]), a[0] * a[1] * (1 - a[2]), a[0] * a[1] * a[2]]
    hist = np.bincount(committed, minlength=5)[1:] / B
    np.testing.assert_allclose(hist, pn, atol=0.005)


# ----------------------------------------------------------------------------- rmsnorm
def test_rmsnorm_residual_closed_form_and_torch():
    T, H = 4, 64
    x = bits(np.full((T, H), 1.5))
    y = bits(np.full((T, H), 0.5))
    xn, hn = oracle.rmsnorm_residual(x, y, eps=1e-6)
    assert np.all(xn == 2.0)
    np.testing.assert_allclose(hn, 2.0 / math.sqrt(4.0 + 1e-6), rtol=1e-14)
    rs = np.random.default_rng(0)
    x = bits(rs.standard_normal((T, H)))
    y = bits(rs.standard_normal((T, H)) * 0.1)
    xn, hn = oracle.rmsnorm_residual(x, y, eps=1e-6)
    np.testing.assert_allclose(xn, val64(bits(val64(x) + val64(y))), rtol=0, atol=0)
    ref = F.rms_norm(torch.from_numpy(xn), (H,), eps=1e-6).numpy()
    np.testing.assert_allclose(hn, ref, rtol=1e-12)


# ----------------------------------------------------------------------------- verifier output layer
def _lmhead_brute(hidden, w_vocab):
    """Pure-Python definition: every logit by a plain sum, then a scan in increasing index."""
    hs, wv = val64(hidden), val64(w_vocab)
    g, gap = [], []
    for r in range(hs.shape[0]):
        lg = [sum(float(hs[r, h]) * float(wv[v, h]) for h in range(hs.shape[1])) for v in range(wv.shape[0])]
        best = 0
        for v in range(1, len(lg)):
            if lg[v] > lg[best]:
                best = v
        g.append(best)
        gap.append(lg[best] - max(lg[v] for v in range(len(lg)) if v != best))
    return np.array(g), np.array(gap)


@pytest.mark.parametrize("chunk", [5, 7, 1000])
def test_lmhead_argmax_brute_force(chunk):
    rs = np.random.default_rng(11)
    # small integers: exact products, frequent exact ties between different rows
    hidden = bits(rs.integers(-2, 3, size=(6, 5)))
    w_vocab = bits(rs.integers(-2, 3, size=(37, 5)))
    # a later copy of row 0's winning row: a tie at the maximum, which the first index wins
    w_vocab[36] = w_vocab[_lmhead_brute(hidden, w_vocab)[0][0]]
    g, gap = oracle.lmhead_argmax(hidden, w_vocab, chunk=chunk)
    rg, rgap = _lmhead_brute(hidden, w_vocab)
    np.testing.assert_array_equal(g, rg)
    np.testing.assert_allclose(gap, rgap, rtol=0, atol=1e-12)
    assert gap[0] == 0 and g[0] != 36


def test_lmhead_argmax_planted_and_duplicates():
    rs = np.random.default_rng(12)
    H, V = 64, 300
    hidden = bits(rs.standard_normal((3, H)))
    w_vocab = bits(rs.standard_normal((V, H)) * 0.02)
    # row 17 is twice hidden row 0: by Cauchy-Schwarz it beats every small random row
    w_vocab[17] = bits(2.0 * val64(hidden[0]))
    # rows 40 and 200 are the same large copy of hidden row 1: the lower index wins, gap 0
    w_vocab[40] = bits(3.0 * val64(hidden[1]))
    w_vocab[200] = w_vocab[40]
    g, gap = oracle.lmhead_argmax(hidden, w_vocab, chunk=64)
    assert g[0] == 17 and gap[0] > 0
    assert g[1] == 40 and gap[1] == 0


def test_lmhead_argmax_matches_torch():
    rs = np.random.default_rng(13)
    H, V = 128, 5000
    hidden = bits(rs.standard_normal((8, H)))
    w_vocab = bits(rs.standard_normal((V, H)) * 0.02)
    g, gap = oracle.lmhead_argmax(hidden, w_vocab, chunk=999)
    lg = torch.from_numpy(val64(hidden)) @ torch.from_numpy(val64(w_vocab)).T
    np.testing.assert_array_equal(g, torch.argmax(lg, dim=1).numpy())
    top2 = torch.topk(lg, 2, dim=1).values
    np.testing.assert_allclose(gap, (top2[:, 0] - top2[:, 1]).numpy(), rtol=1e-12, atol=1e-15)


def test_accept_from_greedy_matches_accept():
    # the rule on given greedy tokens equals the C oracle's rule on logits whose greedy tokens they are
    for seed in range(5):
        B, K, V = 50, 3, 16
        logits, planted = synth.verify_logits(B, K, V, seed)
        drafts = synth.draft_tokens(planted, V, [0.7, 0.6, 0.5], seed)
        g, alen, comm = oracle.accept(logits, drafts)
        alen2, comm2 = oracle.accept_from_greedy(g, drafts)
        np.testing.assert_array_equal(alen, alen2)
        np.testing.assert_array_equal(comm, comm2)


# ----------------------------------------------------------------------------- verify attention
def _attn_problem(B=2, Q=3, L=9, nh=2, d=4, seed=0, lens=(9, 5)):
    rs = np.random.default_rng(seed)
    q = bits(rs.standard_normal((B, Q, nh, d)))
    k = bits(rs.standard_normal((B, L, nh, d)))
    v = bits(rs.standard_normal((B, L, nh, d)))
    return q, k, v, np.array(lens[:B], np.int32)


def test_attention_brute_force():
    q, k, v, n = _attn_problem()
    scale = 0.5
    out = oracle.verify_attention(q, k, v, n, scale)
    qf, kf, vf = val64(q), val64(k), val64(v)
    B, Q, nh, d = qf.shape
    for b in range(B):
        for j in range(Q):
            p = int(n[b]) - Q + j
            for h in range(nh):
                s = [scale * sum(float(qf[b, j, h, c]) * float(kf[b, t, h, c]) for c in range(d)) for t in range(p + 1)]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                z = sum(e)
                ref = [sum(e[t] / z * float(vf[b, t, h, c]) for t in range(p + 1)) for c in range(d)]
                np.testing.assert_allclose(out[b, j, h], ref, rtol=1e-12, atol=1e-14)


def test_attention_special_cases():
    # a sequence whose cache holds only its Q positions: query 0 sees key 0 alone (output = v_0);
    # identical keys: uniform weights, the mean of the visible values
    q, k, v, _ = _attn_problem(B=1, Q=3, L=6, lens=(3,))
    out = oracle.verify_attention(q, k, v, np.array([3], np.int32), 0.7)
    np.testing.assert_allclose(out[0, 0], val64(v[0, 0]), rtol=0, atol=0)
    k2 = k.copy()
    k2[0, :, :, :] = k[0, 0]
    out2 = oracle.verify_attention(q, k2, v, np.array([6], np.int32), 0.7)
    for j in range(3):
        np.testing.assert_allclose(out2[0, j], val64(v[0, :4 + j]).mean(axis=0), rtol=1e-12)


def test_attention_is_causal():
    q, k, v, n = _attn_problem(B=1, L=9, lens=(9,))
    out = oracle.verify_attention(q, k, v, n, 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[0, 8] = bits(np.full((2, 4), 9.0))     # the last key: seen only by the last query
    v2[0, 8] = bits(np.full((2, 4), -9.0))
    out2 = oracle.verify_attention(q, k2, v2, n, 0.5)
    np.testing.assert_array_equal(out[0, :2], out2[0, :2])
    assert not np.allclose(out[0, 2], out2[0, 2])


def test_attention_matches_torch_sdpa():
    q, k, v, n = _attn_problem(B=2, Q=4, L=40, nh=3, d=16, seed=3, lens=(40, 17))
    scale = 0.25
    out = oracle.verify_attention(q, k, v, n, scale)
    for b in range(2):
        L = int(n[b])
        qt = torch.from_numpy(val64(q[b])).permute(1, 0, 2)          # [nh, Q, d]
        kt = torch.from_numpy(val64(k[b, :L])).permute(1, 0, 2)      # [nh, L, d]
        vt = torch.from_numpy(val64(v[b, :L])).permute(1, 0, 2)
        pos = torch.arange(L - 4, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos                      # [Q, L]
        ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
        np.testing.assert_allclose(out[b], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------------------- K policy
def test_k_policy_tau_matches_the_pages():
    page = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))
    a = page["conditional_accept_k3"]["value"]
    _, tau, S = oracle.k_policy(a, [1.0, 1.0, 1.0, 1.0])
    assert abs(tau[3] - page["tau_k3"]["value"]) < 0.005
    assert abs(tau[3] - page["tau_k3_graph"]["value"]) < 0.011
    assert tau[0] == 1.0 and abs(tau[1] - (1 + a[0])) < 1e-15
    np.testing.assert_allclose(S, tau)      # equal costs: the speedup is tau itself


def _simulate(a, cost, K, steps, rng):
    """Speculative decoding with Bernoulli conditional acceptances: tokens per unit cost."""
    L = np.zeros(steps, np.int64)
    alive = np.ones(steps, bool)
    for i in range(K):
        alive &= rng.random(steps) < a[i]
        L += alive
    return (L + 1).sum() / (steps * cost[K]), L


def test_k_policy_matches_a_simulated_decode_loop():
    rng = np.random.default_rng(11)
    a = [0.83, 0.663, 0.636]
    for cost in ([1.0, 1.3, 1.6, 1.9], [1.0, 1.05, 1.3, 2.2], [1.0, 1.8, 2.6, 3.4]):
        k_best, tau, S = oracle.k_policy(a, cost)
        greedy = 1.0 / cost[0]
        emp = []
        for K in range(4):
            rate, _ = _simulate(a, cost, K, 200_000, rng)
            emp.append(rate / greedy)
        emp = np.array(emp)
        np.testing.assert_allclose(emp, S, rtol=0.01)
        assert int(np.argmax(emp)) == k_best
    # the graph-mode finding: with dear drafts K = 1 wins although tau grows with K
    k_best, tau, S = oracle.k_policy(a, [1.0, 1.56, 2.2, 2.5])
    assert k_best == 1 and tau[3] > tau[1]


def test_cond_accept_estimate():
    rng = np.random.default_rng(12)
    a = [0.83, 0.663, 0.636]
    _, L = _simulate(a, [1, 1, 1, 1], 3, 400_000, rng)
    est = oracle.cond_accept_from_lengths(L, 3)
    np.testing.assert_allclose(est, a, atol=0.004)
    _, tau, _ = oracle.k_policy(est, [1, 1, 1, 1])
    assert abs(tau[3] - (L + 1).mean()) < 1e-12   # tau of the estimate = the mean committed count
    assert list(oracle.cond_accept_from_lengths(np.zeros(5, int), 2)) == [0.0, 0.0]


# ----------------------------------------------------------------------------- FastMTP draft block
def _draft_weights(H=64, I=96, V=50, seed=0, std=0.1):
    rs = np.random.default_rng(seed)
    g = lambda *s: bits(rs.standard_normal(s) * std)
    return dict(emb=bits(rs.standard_normal((V, H))), w_proj=g(H, 2 * H), w_q=g(H, H), w_k=g(H, H), w_v=g(H, H),
                w_o=g(H, H), w_gate_up=g(2 * I, H), w_down=g(H, I), w_vocab=g(V, H))


def _draft_inputs(B=3, H=64, nh=4, L=12, lens=(3, 7, 0), seed=1):
    rs = np.random.default_rng(seed)
    d = H // nh
    h = val64(bits(rs.standard_normal((B, H))))
    kc = val64(bits(rs.standard_normal((B, L, nh, d))))
    vc = val64(bits(rs.standard_normal((B, L, nh, d))))
    return h, rs.integers(0, 50, size=B), kc, vc, np.array(lens[:B])


def test_draft_block_matches_torch_formulation():
    w = _draft_weights()
    h, t, kc, vc, n = _draft_inputs()
    nh = 4
    h1, draft, _ = oracle.draft_block(h, t, w, kc.copy(), vc.copy(), n, nh)
    T = lambda u: torch.from_numpy(val64(w[u]))
    rms = lambda x: F.rms_norm(x, (x.shape[-1],), eps=1e-6)
    x = torch.cat([rms(torch.from_numpy(h)), rms(T("emb")[torch.from_numpy(t)])], dim=1)
    u = F.linear(x, T("w_proj"))
    a = rms(u)
    q, k, v = F.linear(a, T("w_q")), F.linear(a, T("w_k")), F.linear(a, T("w_v"))
    B, H = u.shape
    d = H // nh
    att = torch.zeros(B, H, dtype=torch.float64)
    for b in range(B):
        m = int(n[b])
        ks = torch.cat([torch.from_numpy(kc[b, :m]), k[b].view(1, nh, d)]).permute(1, 0, 2)   # [nh, m+1, d]
        vs = torch.cat([torch.from_numpy(vc[b, :m]), v[b].view(1, nh, d)]).permute(1, 0, 2)
        att[b] = F.scaled_dot_product_attention(q[b].view(nh, 1, d), ks, vs).reshape(H)
    u = u + F.linear(att, T("w_o"))
    f = rms(u)
    I = w["w_down"].shape[1]
    u = u + F.linear(F.silu(F.linear(f, T("w_gate_up")[:I])) * F.linear(f, T("w_gate_up")[I:]), T("w_down"))
    logits = F.linear(rms(u), T("w_vocab"))
    np.testing.assert_allclose(h1, u.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(draft, torch.argmax(logits, dim=1).numpy())


def test_draft_block_without_attention_and_ffn_is_the_output_layer():
    # W_p = [I | 0], W_o = 0, W_down = 0: the block passes RMSNorm(h) through, so its draft is the
    # output layer's greedy token of RMSNorm(RMSNorm(h)) -- the (separately pinned) lmhead oracle
    H = 64
    w = _draft_weights(H=H)
    w["w_proj"] = bits(np.concatenate([np.eye(H), np.zeros((H, H))], axis=1))
    w["w_o"] = bits(np.zeros((H, H)))
    w["w_down"] = bits(np.zeros((H, 96)))
    h, t, kc, vc, n = _draft_inputs(H=H)
    h1, draft, _ = oracle.draft_block(h, t, w, kc, vc, n, 4)
    # RMSNorm by hand: x / sqrt(mean(x^2) + eps), eps 1e-6
    norm = lambda x: x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(h1, norm(h), rtol=1e-13, atol=1e-15)
    g, _ = oracle.lmhead_argmax(norm(h1), w["w_vocab"])
    np.testing.assert_array_equal(draft, g)


def test_draft_block_attention_with_zero_queries_is_the_mean_value():
    # W_q = 0: every visible cache entry gets the same weight; W_o = I and W_down = 0 expose the
    # attention output as h_next - u
    H, nh = 64, 4
    w = _draft_weights(H=H)
    w["w_q"] = bits(np.zeros((H, H)))
    w["w_o"] = bits(np.eye(H))
    w["w_down"] = bits(np.zeros((H, 96)))
    h, t, kc, vc, n = _draft_inputs(H=H)
    kc2, vc2 = kc.copy(), vc.copy()
    h1, _, _ = oracle.draft_block(h, t, w, kc2, vc2, n, nh)
    x = np.concatenate([oracle._rms64(h), oracle._rms64(val64(w["emb"])[t])], axis=1)
    u = x @ val64(w["w_proj"]).T
    for b in range(3):
        m = int(n[b])
        mean_v = vc2[b, :m + 1].mean(axis=0).reshape(H)     # includes the entry the step appended
        np.testing.assert_allclose(h1[b] - u[b], mean_v, rtol=1e-9, atol=1e-12)


def test_draft_loop_chains_the_block():
    w = _draft_weights()
    h, t, kc, vc, n = _draft_inputs()
    drafts, _ = oracle.draft_loop(h, t, w, kc.copy(), vc.copy(), n, 4, K=3)
    kc2, vc2, hh, tt, nn = kc.copy(), vc.copy(), h, t, n.copy()
    for i in range(3):
        hh, tt, _ = oracle.draft_block(hh, tt, w, kc2, vc2, nn, 4)
        np.testing.assert_array_equal(drafts[:, i], tt)
        nn = nn + 1


def test_draft_problem_shapes_and_oracle_run():
    p = synth.draft_problem(2, K=3, H=128, nh=2, I=256, V=300, seed=4)
    assert p.k_cache.shape == (2, p.L, 2, 64) and p.L >= int(p.ctx_len.max()) + 3
    kc, vc = val64(p.k_cache), val64(p.v_cache)
    drafts, gaps = oracle.draft_loop(p.h0, p.t0, p.weights, kc, vc, p.ctx_len, p.nh, p.K)
    assert drafts.shape == (2, 3) and np.all((drafts >= 0) & (drafts < 300)) and np.all(gaps >= 0)
    # the loop appended K entries per sequence to the block's cache and left the rest alone
    for b in range(2):
        n = int(p.ctx_len[b])
        np.testing.assert_array_equal(kc[b, :n], val64(p.k_cache[b, :n]))
        assert not np.array_equal(kc[b, n:n + 3], val64(p.k_cache[b, n:n + 3]))
        np.testing.assert_array_equal(kc[b, n + 3:], val64(p.k_cache[b, n + 3:]))


def test_speculative_loop_with_the_draft_block_is_greedy():
    # the drafts of the recursive block, checked by the acceptance rule against a verifier's greedy
    # tokens, commit exactly the verifier's greedy sequence (lossless, whatever the drafter proposes)
    V, H, nh, I = 50, 64, 4, 96
    w = _draft_weights(H=H, I=I, V=V, seed=5)
    verifier = lambda ctx: (7 * sum(ctx) + 3 * ctx[-1] + len(ctx)) % V     # a deterministic toy verifier
    ref = [1, 2, 3]
    while len(ref) < 40:
        ref.append(verifier(ref))
    out = [1, 2, 3]
    L = 64
    kc = np.zeros((1, L, nh, H // nh))
    vc = np.zeros((1, L, nh, H // nh))
    n, steps, accepted = 0, 0, 0
    emb = val64(w["emb"])
    while len(out) < len(ref):
        K = 3
        h0 = emb[[out[-1]]]
        drafts, _ = oracle.draft_loop(h0, [out[-1]], w, kc, vc, [n], nh, K)
        greedy = np.array([[verifier(out + list(drafts[0, :j])) for j in range(K + 1)]])
        alen, comm = oracle.accept_from_greedy(greedy, drafts)
        out += [int(c) for c in comm[0, :alen[0] + 1]]
        accepted += int(alen[0])
        n, steps = n + 1, steps + 1
    assert len(out) >= len(ref) and out[:len(ref)] == ref
    assert steps <= len(ref) - 3      # never fewer than one committed token per verify step


def test_k_policy_reads_the_pages_speedups():
    # S = tau / c with the pages' printed figures: eager K = 3 (83.1 vs 42.7 tok/s, tau 2.73) and
    # graphs K = 1 (185.6 vs 158.3 tok/s) give the printed 1.95x and 1.17x; with the relative step
    # cost c(1) they imply, the policy picks K = 1 under graphs whenever the dearer steps keep
    # their speedups below 1.17x
    page = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))
    a = page["conditional_accept_k3"]["value"]
    greedy_e, spec_e = page["eager_tok_s"]["value"]
    greedy_g, spec_g = page["graph_tok_s"]["value"]
    assert round(spec_e / greedy_e, 2) == page["eager_speedup"]["value"]
    assert round(spec_g / greedy_g, 2) == page["graph_speedup_best"]["value"]
    _, tau, _ = oracle.k_policy(a, [1.0] * 4)
    c3_eager = tau[3] / (spec_e / greedy_e)
    c1_graph = tau[1] / (spec_g / greedy_g)
    _, _, S = oracle.k_policy(a, [1.0, 1.0, 1.0, c3_eager])
    assert abs(S[3] - spec_e / greedy_e) < 1e-9 and 1.35 < c3_eager < 1.45
    # graphs: with c(1) from the pages and c(2), c(3) dear enough for S <= 1.17, K = 1 is chosen
    k, _, S = oracle.k_policy(a, [1.0, c1_graph, tau[2] / 1.16, tau[3] / 1.16])
    assert k == 1 and abs(S[1] - spec_g / greedy_g) < 1e-9


def test_attention_single_query_is_plain_decode_attention():
    # Q = 1: the one query sits at the last cache entry and sees all n of them (no mask at all)
    q, k, v, n = _attn_problem(B=2, Q=1, L=20, nh=3, d=8, seed=6, lens=(20, 9))
    out = oracle.verify_attention(q, k, v, n, 0.35)
    for b in range(2):
        m = int(n[b])
        ref = F.scaled_dot_product_attention(torch.from_numpy(val64(q[b])).permute(1, 0, 2),
                                             torch.from_numpy(val64(k[b, :m])).permute(1, 0, 2),
                                             torch.from_numpy(val64(v[b, :m])).permute(1, 0, 2), scale=0.35)
        np.testing.assert_allclose(out[b], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-14)


def test_page_context_lengths_follow_the_recipe():
    rs = synth.streams(3, 1)[0]
    n = synth.page_context_lengths(rs, 20000, 4)
    vis_txt = n - 4
    assert vis_txt.min() >= 256 and vis_txt.max() <= 1156 + 1085
    assert synth.page_cache_capacity(4) >= n.max() and synth.page_cache_capacity(4) % 64 == 0
    # mean: 256 + 100 * 4.5 visual + 542.5 text
    assert abs(vis_txt.mean() - (256 + 450 + 542.5)) < 15
