"""The FastMTP speculative loop end to end on the GPU, every step in the library's kernels: the
draft block (spec_draft_loop) proposes K tokens from the verifier's last state, the verify pass of
a decoder (decoder.Decoder: attention + MoE layers, then the output layer fused with the greedy
search and the acceptance rule) checks them, and the committed stream must equal plain greedy
decoding through the same kernels, token for token -- "lossless" in the pages' sense: the committed
text matches ordinary greedy decoding (kg.zhiyong.dev, "Why FastMTP fits OCR particularly well").

The decoder is small (2 layers, hidden 256, 8 experts top-2, vocabulary 2048) and synthetic.  With
mimic_draft the draft block proposes the greedy token of the embedding alone, and out_scale sets
how often the layers change it, so that the accepted lengths span 0..K."""
import numpy as np
import pytest
import torch

from lossless_speculative_verification_gb300 import api, synth
from lossless_speculative_verification_gb300.decoder import Decoder

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu

B, P, N_NEW = 4, 6, 40


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    yield
    torch.cuda.synchronize()
    assert api.get_device_error() == 0


def make(seed, out_scale):
    dims = synth.MoeDims(0, 256, 8, 2, 1, 128)
    prob = synth.decoder_problem(2, dims, V=2048, nh=2, I_draft=256, seed=seed, out_scale=out_scale, mimic_draft=True)
    # a sequence that keeps accepting runs ahead of the slowest one: room for (K + 1) tokens a round
    dec = Decoder(prob, B, L=P + 4 * N_NEW + 32)
    prompt = np.random.default_rng(seed + 7).integers(0, prob.V, size=(B, P)).astype(np.int32)
    return dec, torch.from_numpy(prompt).cuda()


def prefill(dec, prompt):
    ctx = torch.full((B,), P, dtype=torch.int32, device="cuda")
    b = dec.verify(prompt, ctx, prompt[:, 1:].contiguous())
    return b


def greedy(dec, prompt):
    b = prefill(dec, prompt)
    t = b["argmax"][:, P - 1].clone()
    out = [t.cpu().numpy()]
    empty = torch.zeros((B, 0), dtype=torch.int32, device="cuda")
    for i in range(N_NEW - 1):
        ctx = torch.full((B,), P + 1 + i, dtype=torch.int32, device="cuda")
        b = dec.verify(t.view(B, 1).contiguous(), ctx, empty)
        t = b["argmax"][:, 0].clone()
        out.append(t.cpu().numpy())
    return np.stack(out, axis=1)                                   # [B, N_NEW]


def speculative(dec, prompt, K):
    H = dec.H
    b = prefill(dec, prompt)
    t_last = b["argmax"][:, P - 1].clone()
    h0 = b["x"].view(B, P, H)[:, P - 1].contiguous()
    ctx = np.full(B, P, np.int64)
    committed = [[int(v)] for v in t_last.cpu().numpy()]
    Ld = P + 4 * N_NEW + 32
    g = torch.Generator(device="cuda").manual_seed(3)
    dk = torch.randn((B, Ld, dec.nh, dec.hd), generator=g, device="cuda").to(torch.bfloat16)
    dv = torch.randn((B, Ld, dec.nh, dec.hd), generator=g, device="cuda").to(torch.bfloat16)
    dws = api.spec_draft_workspace(B, H, dec.nh, dec.prob.I_draft, dec.V, Ld)
    lengths = []
    while min(len(c) for c in committed) < N_NEW:
        dctx = torch.from_numpy(ctx.astype(np.int32)).cuda()
        drafts = api.spec_draft_loop(dec.draft_w, h0, t_last, dk, dv, dctx, K, dws)
        tokens = torch.cat([t_last.view(B, 1), drafts], dim=1).contiguous()
        ctx_after = torch.from_numpy((ctx + K + 1).astype(np.int32)).cuda()
        b = dec.verify(tokens, ctx_after, drafts)
        alen = b["alen"].cpu().numpy()
        comm = b["comm"].cpu().numpy()
        lengths.extend(alen.tolist())
        for s in range(B):
            committed[s].extend(int(c) for c in comm[s, :alen[s] + 1])
        ctx += alen + 1
        idx = torch.from_numpy(alen.astype(np.int64)).cuda()
        t_last = b["comm"].gather(1, idx.view(B, 1).to(torch.int64)).view(B).contiguous()
        h0 = b["x"].view(B, K + 1, H)[torch.arange(B, device="cuda"), idx].contiguous()
    return np.array([c[:N_NEW] for c in committed]), np.array(lengths)


@pytest.mark.parametrize("seed", [0, 1])
def test_speculative_loop_commits_the_greedy_sequence(seed):
    seen = set()
    for out_scale in (0.05, 0.6):
        dec, prompt = make(seed, out_scale)
        ref = greedy(dec, prompt)
        for K in (1, 2, 3):
            got, lengths = speculative(dec, prompt, K)
            np.testing.assert_array_equal(got, ref, err_msg="K=%d, out_scale %g" % (K, out_scale))
            seen |= {(K, int(L)) for L in lengths}
            assert lengths.min() >= 0 and lengths.max() <= K
    # the runs exercise both full acceptances (the bonus token) and early mismatches
    assert (3, 3) in seen and any(L < K for K, L in seen), sorted(seen)
