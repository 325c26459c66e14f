"""A verify pass of an n-layer decoder, composed from the library's entry points.

The FastMTP verify step runs the drafted positions of every sequence through
the main decoder in one pass and keeps the longest prefix that greedy
decoding would have produced (kg.zhiyong.dev, "The speed comes from three
layers working together" and "Why FastMTP fits OCR particularly well").  The
pages give the decoder as an MoE decoder; the plainest reading is a stack of
pre-norm layers, each an attention block and the MoE FFN on the residual
stream x:

    h = RMSNorm(x);  q, k, v = h W_q^T, h W_k^T, h W_v^T   (the Q new keys and values appended)
    x = x + attention(q, caches) W_o^T;  h = RMSNorm(x);  x = x + MoE(h)

followed by the output layer fused with the greedy search and the acceptance
rule on RMSNorm(x).  Every step runs in the library's kernels
(lsv_gather_rows, rmsnorm_residual, dense_matmul, spec_cache_append,
spec_verify_attention, moe_verify_layer, spec_verify_lmhead); this module only
orders the calls and owns the buffers, so that a verify pass (and a draft +
verify step) can be replayed as one CUDA graph.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import api


def _dev(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


class Decoder:
    """Device weights and per-layer key/value caches [B, L, nh, d] of a synthetic decoder
    (synth.DecoderProblem).  verify() runs one verify pass over Q positions per sequence, for the
    first tokens.shape[0] <= B sequences."""

    def __init__(self, prob, B: int, L: int, device="cuda"):
        self.prob, self.B, self.L, self.device = prob, B, L, device
        d = prob.dims
        self.H, self.nh = d.H, prob.nh
        self.hd = d.H // prob.nh
        self.V = prob.V
        self.emb = _dev(prob.emb, device)
        self.w_vocab = _dev(prob.w_vocab, device)
        self.layers = []
        for lw in prob.layers:
            t = {n: _dev(lw[n], device) for n in ("w_q", "w_k", "w_v", "w_o")}
            t["moe"] = api.weights(*[_dev(lw[n], device) for n in ("w_router", "w_gate_up", "w_down", "ws_gate_up",
                                                                    "ws_down")])
            t["kc"] = torch.zeros((B, L, self.nh, self.hd), dtype=torch.bfloat16, device=device)
            t["vc"] = torch.zeros_like(t["kc"])
            self.layers.append(t)
        dw = dict(prob.draft)
        dw["emb"], dw["w_vocab"] = prob.emb, prob.w_vocab
        self.draft_w = {n: (self.emb if n == "emb" else self.w_vocab if n == "w_vocab" else _dev(dw[n], device))
                        for n in api.DRAFT_WEIGHTS}
        self._bufs = {}

    def fill_caches(self, seed: int):
        """N(0, 1) keys and values everywhere (the entries of a prefix that is not replayed)."""
        g = torch.Generator(device=self.device).manual_seed(seed)
        for t in self.layers:
            t["kc"].copy_(torch.randn(t["kc"].shape, generator=g, device=self.device).to(torch.bfloat16))
            t["vc"].copy_(torch.randn(t["vc"].shape, generator=g, device=self.device).to(torch.bfloat16))

    def buffers(self, B: int, Q: int):
        """The activations, workspaces and outputs of a pass over Q positions of B sequences."""
        if (B, Q) not in self._bufs:
            H, dev = self.H, self.device
            T = B * Q
            d = self.prob.dims
            b = {n: torch.zeros((T, H), dtype=torch.bfloat16, device=dev) for n in ("x", "h", "zero", "q", "k", "v",
                                                                                     "a", "o", "y")}
            b["sh"] = api.shape(T, H, d.E, d.k, d.S, d.I)
            b["mws"] = api.workspace(b["sh"], dev)
            b["aws"] = api.spec_verify_attention_workspace(B, Q, self.L, self.nh, self.hd, dev)
            b["lws"] = api.spec_verify_lmhead_workspace(B, Q - 1, self.V, H, dev)
            b["argmax"] = torch.zeros((B, Q), dtype=torch.int32, device=dev)
            b["alen"] = torch.zeros(B, dtype=torch.int32, device=dev)
            b["comm"] = torch.zeros((B, Q), dtype=torch.int32, device=dev)
            self._bufs[(B, Q)] = b
        return self._bufs[(B, Q)]

    def verify(self, tokens, ctx_after, drafts):
        """One verify pass.  tokens [B, Q] int32: input 0 is each sequence's last committed token,
        inputs 1..Q-1 its drafts (drafts [B, Q-1] int32, the same tokens); ctx_after [B] int32: the
        cache lengths once the Q positions are appended.  Returns the pass's buffers: argmax [B, Q]
        (the greedy token after each input), alen [B], comm [B, Q] (the rule's outputs), x [B*Q, H]
        (the last residual stream, the draft block's next input state)."""
        B, Q = tokens.shape
        b = self.buffers(B, Q)
        nh, hd = self.nh, self.hd
        api.gather_rows(self.emb, tokens.reshape(-1), out=b["x"])
        y = b["zero"]
        for t in self.layers:
            api.rmsnorm_residual(b["x"], y, h=b["h"])
            for n in ("q", "k", "v"):
                api.dense_matmul(b["h"], t["w_" + n], out=b[n])
            kc, vc = t["kc"][:B], t["vc"][:B]
            api.spec_cache_append(b["k"].view(B, Q, nh, hd), b["v"].view(B, Q, nh, hd), kc, vc, ctx_after)
            api.spec_verify_attention(b["q"].view(B, Q, nh, hd), kc, vc, ctx_after, b["aws"],
                                      out=b["a"].view(B, Q, nh, hd))
            api.dense_matmul(b["a"], t["w_o"], out=b["o"])
            api.rmsnorm_residual(b["x"], b["o"], h=b["h"])
            api.moe_verify_layer(b["h"], t["moe"], b["sh"], b["mws"], out=b["y"])
            y = b["y"]
        api.rmsnorm_residual(b["x"], y, h=b["h"])
        api.spec_verify_lmhead(b["h"], self.w_vocab, drafts, b["lws"], Q - 1, argmax=b["argmax"],
                               accept_len=b["alen"], committed=b["comm"])
        return b

    def launches_per_verify(self, B: int, Q: int) -> int:
        """Library kernel launches of one verify pass (the MoE layer: 3 up to 256 tokens)."""
        T = B * Q
        moe = 3 if T <= 256 else (4 if T * self.prob.dims.k <= 8192 else 6)
        return 1 + len(self.layers) * (1 + 3 + 1 + 2 + 1 + 1 + moe) + 1 + 2
