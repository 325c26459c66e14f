"""The FastMTP draft block on the GPU (spec_draft_loop) and its dense product
(dense_matmul) against the oracle.

The oracle is the block's exact definition in float64; the GPU path stores every value between
its kernels in bf16.  The bounds come from the error budget in draft_budget.py, derived and
checked on the CPU before any GPU run: the last state (and the appended keys and values) within
rel-L2 1e-2 and every element within 6 times that of the RMS; drafts, integers decided by an
argmax, bit for bit wherever the exact top-two logits are at least 6 standard deviations of the
budget's logit error apart at every step (the inputs of sequences that fall short are redrawn).
The rest of the caches must be untouched."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from lossless_speculative_verification_gb300 import api, synth

import draft_budget
from draft_budget import assert_state_close
from gpu_util import bf16_f64, from_dev_bf16, need_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    yield
    torch.cuda.synchronize()
    assert api.get_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(32, 1280, 2560), (1, 8, 64), (130, 1288, 1280), (4, 7168, 1280), (300, 96, 192)])
def test_dense_matmul(M, N, K):
    rs = np.random.default_rng(M + N + K)
    x = synth.bf16_bits(rs.standard_normal((M, K)).astype(np.float32))
    w = synth.bf16_bits((rs.standard_normal((N, K)) * 0.02).astype(np.float32))
    got = bf16_f64(from_dev_bf16(api.dense_matmul(to_dev(x), to_dev(w))))
    torch.cuda.synchronize()
    ref = bf16_f64(x) @ bf16_f64(w).T
    # fp32 sums, one bf16 rounding
    np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=1e-4 * np.sqrt((ref ** 2).mean()))


# Few rows of x (the cluster split-K path): the draft block's projections at decode sizes (W_p, the
# FFN's down projection, W_o at 64 rows), ragged shapes (rows past a tile, a partial last weight
# tile, one chunk of K) and the longest K
SKINNY = [(32, 1280, 2560), (32, 1280, 7168), (1, 8, 64), (7, 96, 192), (256, 136, 16384), (64, 1280, 1280),
          (17, 392, 4096)]


@pytest.mark.parametrize("M,N,K", SKINNY)
def test_dense_matmul_few_rows(M, N, K):
    rs = np.random.default_rng(M * 7 + N + K)
    x = synth.bf16_bits(rs.standard_normal((M, K)).astype(np.float32))
    w = synth.bf16_bits((rs.standard_normal((N, K)) * 0.02).astype(np.float32))
    a = api.dense_matmul(to_dev(x), to_dev(w))
    b = api.dense_matmul(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))   # the splits add in a fixed order
    got = bf16_f64(from_dev_bf16(a))
    ref = bf16_f64(x) @ bf16_f64(w).T
    # fp32 sums, one bf16 rounding
    np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=1e-4 * np.sqrt((ref ** 2).mean()))


@pytest.mark.parametrize("M,F,K", [(32, 7168, 1280), (4, 512, 256), (19, 136, 640), (256, 64, 128), (1, 8, 4096)])
def test_dense_swiglu(M, F, K):
    rs = np.random.default_rng(M + F + K)
    x = synth.bf16_bits(rs.standard_normal((M, K)).astype(np.float32))
    w = synth.bf16_bits((rs.standard_normal((2 * F, K)) * 0.02).astype(np.float32))
    a = api.dense_swiglu(to_dev(x), to_dev(w))
    b = api.dense_swiglu(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    got = bf16_f64(from_dev_bf16(a))
    g = bf16_f64(x) @ bf16_f64(w[:F]).T
    u = bf16_f64(x) @ bf16_f64(w[F:]).T
    ref = g / (1.0 + np.exp(-g)) * u
    np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=1e-4 * np.sqrt((ref ** 2).mean()))


def test_dense_swiglu_rejects_bad_shapes():
    lib = api._ffi.load()
    x = torch.zeros((300, 64), dtype=torch.bfloat16, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    assert lib.dense_swiglu(p(x), p(x), p(x), 300, 8, 64, None) == api._ffi.ERR_UNSUPPORTED    # > 256 rows
    assert lib.dense_swiglu(p(x), p(x), p(x), 4, 8, 96, None) == api._ffi.ERR_UNSUPPORTED      # K % 64
    assert lib.dense_swiglu(p(x), p(x), p(x), 4, 12, 64, None) == api._ffi.ERR_UNSUPPORTED     # F % 8


def gap_checked(B, K, H, nh, I, V, seed, rounds=80):
    """The problem with every sequence's drafts decided by at least the budget's gap in the exact
    oracle, and the oracle's drafts, last states and caches (sequences are independent: only the
    redrawn ones are run again)."""
    p = synth.draft_problem(B, K=K, H=H, nh=nh, I=I, V=V, seed=seed)
    w64 = {n: bf16_f64(v) for n, v in p.weights.items()}        # converted once for every oracle run
    min_gap = draft_budget.draft_gap(w64["w_vocab"])
    rng = np.random.default_rng(seed + 99)
    kc0, vc0 = bf16_f64(p.k_cache), bf16_f64(p.v_cache)
    kc, vc = kc0.copy(), vc0.copy()
    drafts, gaps, h = oracle.draft_loop(p.h0, p.t0, w64, kc, vc, p.ctx_len, nh, K, return_state=True)
    for _ in range(rounds):
        bad = np.nonzero(gaps.min(axis=1) < min_gap)[0]
        if bad.size == 0:
            return p, drafts, h, kc, vc
        p.h0[bad] = synth.hidden_rows(rng, bad.size, H, "sphere")
        p.t0[bad] = rng.integers(0, V, size=bad.size).astype(np.int32)
        kb, vb = kc0[bad].copy(), vc0[bad].copy()
        d2, g2, h2 = oracle.draft_loop(p.h0[bad], p.t0[bad], w64, kb, vb, p.ctx_len[bad], nh, K,
                                       return_state=True)
        drafts[bad], gaps[bad], h[bad], kc[bad], vc[bad] = d2, g2, h2, kb, vb
    raise RuntimeError("gap condition not met")


def run(p, K):
    w = {n: to_dev(p.weights[n]) for n in api.DRAFT_WEIGHTS}
    kc, vc = to_dev(p.k_cache), to_dev(p.v_cache)
    B, H = p.h0.shape
    ws = api.spec_draft_workspace(B, H, p.nh, p.I, p.V, p.L)
    h_out = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    drafts = api.spec_draft_loop(w, to_dev(p.h0), torch.from_numpy(p.t0).cuda(), kc, vc,
                                 torch.from_numpy(p.ctx_len).cuda(), K, ws, h_out=h_out)
    torch.cuda.synchronize()
    return drafts.cpu().numpy(), from_dev_bf16(h_out), from_dev_bf16(kc), from_dev_bf16(vc)


def check(B, K, H, nh, I, V, seed):
    p, ref_drafts, ref_h, ref_kc, ref_vc = gap_checked(B, K, H, nh, I, V, seed)
    drafts, h, kc, vc = run(p, K)
    np.testing.assert_array_equal(drafts, ref_drafts)
    assert_state_close(bf16_f64(h), ref_h, "last state")
    for b in range(B):
        n = int(p.ctx_len[b])
        np.testing.assert_array_equal(kc[b, :n], p.k_cache[b, :n])       # earlier entries untouched
        np.testing.assert_array_equal(vc[b, :n], p.v_cache[b, :n])
        np.testing.assert_array_equal(kc[b, n + K:], p.k_cache[b, n + K:])
        np.testing.assert_array_equal(vc[b, n + K:], p.v_cache[b, n + K:])
    # the appended keys and values are projections of the normalised state: the same budget
    for name, got_c, ref_c in (("keys", kc, ref_kc), ("values", vc, ref_vc)):
        app = np.concatenate([bf16_f64(got_c[b, int(p.ctx_len[b]):int(p.ctx_len[b]) + K]) for b in range(B)])
        ref_app = np.concatenate([ref_c[b, int(p.ctx_len[b]):int(p.ctx_len[b]) + K] for b in range(B)])
        assert_state_close(app, ref_app, "appended " + name)


def test_draft_loop_small():
    check(B=4, K=3, H=256, nh=2, I=512, V=3000, seed=1)


def test_draft_loop_decoder_shape():
    # 32 sequences, K = 3, hidden 1280 (10 heads x 128), FFN 7,168, vocabulary 129,280
    check(B=32, K=3, H=1280, nh=10, I=synth.DRAFT_FFN, V=synth.VOCAB, seed=2)
