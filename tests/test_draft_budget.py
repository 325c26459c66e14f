"""The draft block's error budget (tests/draft_budget.py) checked on the CPU, before any GPU run.

A bf16-storage model of the block -- torch float64 arithmetic with a bf16 store (torch's own
rounding) at every point where the GPU path stores a value between kernels -- is compared with
the exact oracle.  Without the stores it must be the oracle; with them, its deviation must sit
at the first-order estimate and inside the bounds the GPU test uses."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from lossless_speculative_verification_gb300 import synth

import draft_budget


def _val64(bits):
    return synth.bf16_value(bits).astype(np.float64)


def storage_model(p, tokens, store=True):
    """K steps of the block with the caller's tokens as each step's input token (teacher forcing),
    storing in bf16 where the GPU path does: the block input, u, RMSNorm(u), q, k, v, the
    attention output, W_o attn, u + W_o attn, f, the SwiGLU activation, the FFN output, the new
    state, and its RMSNorm.  Returns (last state, per-step logits)."""
    R = (lambda x: x.to(torch.float32).to(torch.bfloat16).to(torch.float64)) if store else (lambda x: x)
    W = {n: torch.from_numpy(_val64(v)) for n, v in p.weights.items()}
    rms = lambda x: F.rms_norm(x, (x.shape[-1],), eps=1e-6)
    h = torch.from_numpy(_val64(p.h0))
    t = torch.from_numpy(p.t0.astype(np.int64))
    kc, vc = torch.from_numpy(_val64(p.k_cache)), torch.from_numpy(_val64(p.v_cache))
    n = p.ctx_len.astype(np.int64).copy()
    B, H = h.shape
    nh, d, I = p.nh, H // p.nh, p.I
    logits = []
    for i in range(p.K):
        u = R(R(torch.cat([rms(h), rms(W["emb"][t])], 1)) @ W["w_proj"].T)
        a = R(rms(u))
        q, k, v = R(a @ W["w_q"].T), R(a @ W["w_k"].T), R(a @ W["w_v"].T)
        att = torch.zeros(B, H, dtype=torch.float64)
        for b in range(B):
            m = int(n[b])
            kc[b, m], vc[b, m] = k[b].view(nh, d), v[b].view(nh, d)
            att[b] = F.scaled_dot_product_attention(q[b].view(nh, 1, d), kc[b, :m + 1].permute(1, 0, 2),
                                                    vc[b, :m + 1].permute(1, 0, 2)).reshape(H)
        u = R(u + R(R(att) @ W["w_o"].T))
        f = R(rms(u))
        act = R(F.silu(f @ W["w_gate_up"][:I].T) * (f @ W["w_gate_up"][I:].T))
        u = R(u + R(act @ W["w_down"].T))
        logits.append((R(rms(u)) @ W["w_vocab"].T).numpy())
        h, t, n = u, torch.from_numpy(tokens[:, i].astype(np.int64)), n + 1
    return h.numpy(), logits


def _oracle(p):
    wf = {n: _val64(v) for n, v in p.weights.items()}
    return oracle.draft_loop(p.h0, p.t0, wf, _val64(p.k_cache), _val64(p.v_cache), p.ctx_len, p.nh, p.K,
                             return_state=True)


def test_storage_model_without_stores_is_the_oracle():
    p = synth.draft_problem(3, K=3, H=128, nh=2, I=192, V=300, seed=8, lens=[5, 40, 17])
    drafts, _, h = _oracle(p)
    h_model, _ = storage_model(p, drafts, store=False)
    np.testing.assert_allclose(h_model, h, rtol=1e-10, atol=1e-12)


def test_swiglu_gains_quadrature():
    # the quadrature against a seeded Monte Carlo of the same expectations
    s = 0.716
    rs = np.random.default_rng(0)
    g, v = rs.normal(0, s, 4_000_000), rs.normal(0, s, 4_000_000)
    sig = 1 / (1 + np.exp(-g))
    f_mc = np.sqrt(np.mean((g * sig * v) ** 2))
    j_mc = np.sqrt(np.mean((sig * (1 + g * (1 - sig)) * v) ** 2) + np.mean((g * sig) ** 2))
    f_q, j_q = draft_budget.swiglu_gains(s)
    assert abs(f_q - f_mc) < 2e-3 and abs(j_q - j_mc) < 3e-3


@pytest.mark.parametrize("H,nh,I,V", [(1280, 10, 7168, 2048), (256, 2, 512, 3000)])
def test_bf16_storage_error_is_within_the_budget(H, nh, I, V):
    torch.set_num_threads(min(8, torch.get_num_threads()))
    p = synth.draft_problem(4, K=3, H=H, nh=nh, I=I, V=V, seed=2, lens=[150, 400, 37, 900])
    drafts, _, h = _oracle(p)
    h_model, logits = storage_model(p, drafts)
    h_plain, logits_plain = storage_model(p, drafts, store=False)
    rel = np.linalg.norm(h_model - h) / np.linalg.norm(h)
    est = draft_budget.state_rel_estimate(H, I, p.K)
    # the first-order estimate describes the stores (within 25 %), and both sit inside the bound
    assert 0.75 * est <= rel <= 1.25 * est, (rel, est)
    assert est < draft_budget.STATE_REL
    draft_budget.assert_state_close(h_model, h, "bf16-storage model")
    # logit deviation: one standard deviation of a logit's error at the estimated state error is
    # est * sigma_logit; the gap used for bit-exact drafts is far above it
    sigma_logit = float(np.sqrt((_val64(p.weights["w_vocab"]) ** 2).mean())) * np.sqrt(H)
    dl = logits[-1] - logits_plain[-1]
    assert np.sqrt((dl ** 2).mean()) <= 1.25 * np.hypot(est, draft_budget.EPS_STORE) * sigma_logit
    assert np.abs(dl).max() * 2 < draft_budget.draft_gap(_val64(p.weights["w_vocab"]))
