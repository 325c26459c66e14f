"""The verifier's output layer fused with greedy verification (spec_verify_lmhead)
against the oracle: greedy tokens, accepted lengths and committed tokens must
match bit for bit.  The generator keeps the top two logits of every row at
least 1e-3 apart, far above the difference between fp32 tensor-core
accumulation and the fp64 oracle, so both sides take the same decision; the
special cases plant exact ties (identical weight rows give identical logits on
both sides)."""
import functools

import numpy as np
import pytest
import torch

import oracle
from lossless_speculative_verification_gb300 import api, synth

from gpu_util import need_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    yield
    torch.cuda.synchronize()
    assert api.get_device_error() == 0


def run(hidden, w_vocab, drafts, K):
    R, H = hidden.shape
    V = w_vocab.shape[0]
    B = R // (K + 1)
    ws = api.spec_verify_lmhead_workspace(B, K, V, H)
    argmax = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    alen, comm = api.spec_verify_lmhead(to_dev(hidden), to_dev(w_vocab), torch.from_numpy(drafts).cuda(), ws, K,
                                        argmax=argmax)
    torch.cuda.synchronize()
    return argmax.cpu().numpy(), alen.cpu().numpy(), comm.cpu().numpy()


def check(p):
    g, alen, comm = run(p.hidden, p.w_vocab, p.drafts, p.K)
    np.testing.assert_array_equal(g, p.greedy)
    ralen, rcomm = oracle.accept_from_greedy(p.greedy, p.drafts)
    np.testing.assert_array_equal(alen, ralen)
    np.testing.assert_array_equal(comm, rcomm)


@functools.lru_cache(maxsize=None)
def problem(B, K, V, H, seed):
    return synth.lmhead_problem(B, K, V=V, H=H, seed=seed, row_check=oracle.lmhead_row_check())


def test_lmhead_decode_shape():
    # 32 sequences x (K=3)+1 positions, the 129,280-token vocabulary, hidden 1280
    check(problem(32, 3, synth.VOCAB, 1280, 0))


@pytest.mark.parametrize("B,K,V,H", [(1, 1, 129_280, 1280), (40, 3, 5000, 256), (3, 0, 1000, 128),
                                     (64, 7, 4099, 192), (32, 0, 129_280, 1280), (17, 7, 3001, 256),
                                     (9, 7, 2000, 128)])
def test_lmhead_shapes(B, K, V, H):
    # one sequence; two row tiles (160 rows); K = 0; ragged vocabulary tiles (V % 128 != 0); the draft
    # block's 32 rows; a last row tile of 8 rows (box of 16); 72 rows in one tile (box of 80)
    check(problem(B, K, V, H, 1000 * B + K))


def test_lmhead_ties_take_the_first_index():
    rs = np.random.default_rng(21)
    B, K, V, H = 4, 1, 1000, 128
    p = problem(B, K, V, H, 77)
    w = p.w_vocab.copy()
    hid = p.hidden
    # row 0: its winner copied to a later index in another vocabulary tile; row 1: to a later
    # index in the same tile; row 2: a new winner (0.01 x its hidden row: about 1.3 against a
    # typical maximum of 0.7, and far below the other rows' maxima) at two places
    w[900] = w[p.greedy[0, 0]]
    g1 = int(p.greedy[0, 1])
    w[min(V - 1, g1 + 1 if (g1 + 1) // 128 == g1 // 128 else g1 - 1)] = w[g1]
    big = synth.bf16_bits(0.01 * synth.bf16_value(hid[2]).astype(np.float32))
    w[130] = big
    w[610] = big
    g, gap = oracle.lmhead_argmax(hid, w)
    assert gap[0] == 0 and gap[1] == 0 and gap[2] == 0 and g[2] == 130
    drafts = synth.draft_tokens(g.reshape(B, K + 1).astype(np.int32), V, [0.5], 3)
    ga, alen, comm = run(hid, w, drafts, K)
    np.testing.assert_array_equal(ga.reshape(-1), g)
    ralen, rcomm = oracle.accept_from_greedy(g.reshape(B, K + 1), drafts)
    np.testing.assert_array_equal(alen, ralen)
    np.testing.assert_array_equal(comm, rcomm)


def test_lmhead_negative_logits_and_last_tile():
    # every logit negative: the zero-filled rows past the vocabulary must never win; the
    # largest logit sits in the last, partial vocabulary tile
    B, K, V, H = 2, 1, 1000, 128
    rs = np.random.default_rng(5)
    hid = synth.bf16_bits(np.abs(rs.standard_normal((B * (K + 1), H))).astype(np.float32) + 0.5)
    w = synth.bf16_bits(-np.abs(rs.standard_normal((V, H))).astype(np.float32) - 1.0)
    w[V - 1] = synth.bf16_bits(np.full(H, -0.01, np.float32))
    g, gap = oracle.lmhead_argmax(hid, w)
    assert np.all(g == V - 1) and np.all(gap > 1e-3)
    drafts = np.full((B, K), V - 1, np.int32)
    ga, alen, comm = run(hid, w, drafts, K)
    np.testing.assert_array_equal(ga.reshape(-1), g)
    np.testing.assert_array_equal(alen, np.full(B, K))


def test_lmhead_is_deterministic():
    p = problem(40, 3, 5000, 256, 40003)
    a = run(p.hidden, p.w_vocab, p.drafts, p.K)
    b = run(p.hidden, p.w_vocab, p.drafts, p.K)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_lmhead_zero_hidden_rows_give_token_zero():
    # a hidden row of zeros makes every logit of its row +0 or -0 (the weights' signs vary), which
    # are equal: the greedy token is 0, the first index, however the CTAs' results combine
    B, K, V, H = 3, 1, 4099, 128
    p = problem(B, K, V, H, 91)
    hid = p.hidden.copy()
    hid[1] = 0
    hid[4] = 0x8000                              # -0 everywhere
    g, _ = oracle.lmhead_argmax(hid, p.w_vocab)
    assert g[1] == 0 and g[4] == 0
    drafts = synth.draft_tokens(g.reshape(B, K + 1).astype(np.int32), V, [0.5], 5)
    ga, alen, comm = run(hid, p.w_vocab, drafts, K)
    np.testing.assert_array_equal(ga.reshape(-1), g)
    ralen, rcomm = oracle.accept_from_greedy(g.reshape(B, K + 1), drafts)
    np.testing.assert_array_equal(alen, ralen)
    np.testing.assert_array_equal(comm, rcomm)


def test_lmhead_workspace_reuse():
    # one workspace across calls of different shapes: whatever a call leaves in it, the next call's
    # results do not depend on it
    ws = api.spec_verify_lmhead_workspace(64, 7, 4099, 192)
    for B, K, V, H, seed in [(64, 7, 4099, 192, 1), (3, 0, 1000, 128, 2), (40, 3, 5000, 256, 3),
                             (64, 7, 4099, 192, 4), (1, 1, 2000, 128, 5)]:
        p = problem(B, K, V, H, seed)
        argmax = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
        alen, comm = api.spec_verify_lmhead(to_dev(p.hidden), to_dev(p.w_vocab), torch.from_numpy(p.drafts).cuda(),
                                            ws, K, argmax=argmax)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(argmax.cpu().numpy(), p.greedy)
        ralen, rcomm = oracle.accept_from_greedy(p.greedy, p.drafts)
        np.testing.assert_array_equal(alen.cpu().numpy(), ralen)
        np.testing.assert_array_equal(comm.cpu().numpy(), rcomm)
