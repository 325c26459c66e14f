"""Causal attention of the verified positions over the cache (spec_verify_attention)
against the oracle's fp64 definition, element by element.  The kernel computes
scores and sums in fp32 and rounds the output to bf16, so the comparison uses
the layer tolerances (rel-L2 1e-2, max-abs 2e-2)."""
import functools

import numpy as np
import pytest
import torch

import oracle
from lossless_speculative_verification_gb300 import api, synth

from gpu_util import assert_layer_close, bf16_f64, from_dev_bf16, need_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    yield
    torch.cuda.synchronize()
    assert api.get_device_error() == 0


def run(p, scale=None, ws=None):
    ws = api.spec_verify_attention_workspace(p.B, p.Q, p.L, p.nh, p.d) if ws is None else ws
    out = api.spec_verify_attention(to_dev(p.q), to_dev(p.k_cache), to_dev(p.v_cache),
                                    torch.from_numpy(p.ctx_len).cuda(), ws, scale=scale)
    torch.cuda.synchronize()
    return from_dev_bf16(out)


def check(p, scale=None, what=""):
    sc = 1.0 / np.sqrt(p.d) if scale is None else scale
    ref = oracle.verify_attention(p.q, p.k_cache, p.v_cache, p.ctx_len, sc)
    got = run(p, scale)
    assert_layer_close(bf16_f64(got), ref, what)
    return got


@functools.lru_cache(maxsize=None)
def problem(B, Q, nh, d, L=None, lens=None, seed=0, qk_std=1.0):
    return synth.attention_problem(B, Q, nh=nh, d=d, L=L, ctx_len=None if lens is None else np.array(lens),
                                   seed=seed, qk_std=qk_std)


def test_attention_page_workload():
    # 32 sequences x 4 verified positions, 10 heads x 128, page-shaped prefixes (visual + text)
    check(problem(32, 4, synth.ATTN_HEADS, synth.ATTN_HEAD_DIM), what="page")


@pytest.mark.parametrize("B,Q,nh,d,L,lens", [
    (3, 4, 2, 128, 1100, (4, 511, 1100)),           # only the verified positions; a split's edge; full
    (2, 1, 3, 128, 1537, (1537, 513)),              # Q = 1 (plain decoding); a ragged last split
    (4, 8, 2, 64, 700, (8, 9, 520, 700)),           # Q at its maximum; d = 64
    (1, 2, 1, 64, 64, (33,)),                       # one partial warp of positions
])
def test_attention_shapes(B, Q, nh, d, L, lens):
    check(problem(B, Q, nh, d, L, lens, seed=B * 100 + Q), what="B%d Q%d d%d" % (B, Q, d))


def test_attention_peaked_scores():
    # larger q/k spread: softmax weights dominated by a few positions per query (scores with a
    # standard deviation of about 9), which stresses the running-maximum rescaling
    check(problem(4, 4, 2, 128, 2048, (2048, 1500, 700, 4), seed=3, qk_std=3.0), what="peaked")


def test_attention_reads_no_masked_entries():
    # the cache past a sequence's length holds NaN (keys) and huge values (values) in one sequence
    # and NaN in both in another: none of it may reach the output
    p = problem(3, 4, 2, 128, 1024, (600, 1024, 77), seed=9)
    k, v = p.k_cache.copy(), p.v_cache.copy()
    nan = np.uint16(0x7FC0)
    k[0, 600:] = nan
    v[0, 600:] = synth.bf16_bits(np.float32(1e4))
    k[2, 77:] = nan
    v[2, 77:] = nan
    p2 = synth.AttentionProblem(p.B, p.Q, p.L, p.nh, p.d, p.q, k, v, p.ctx_len)
    got = check(p2, what="masked")
    ref = run(p)
    np.testing.assert_array_equal(got, ref)


def test_attention_empty_batch_and_determinism():
    ws = api.spec_verify_attention_workspace(1, 4, 256, 2, 128)
    q = torch.empty((0, 4, 2, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.empty((0, 256, 2, 128), dtype=torch.bfloat16, device="cuda")
    out = api.spec_verify_attention(q, kv, kv, torch.empty(0, dtype=torch.int32, device="cuda"), ws)
    assert out.shape == (0, 4, 2, 128)
    p = problem(8, 4, 3, 128, 1300, (1300, 4, 600, 1200, 513, 512, 1024, 77), seed=5)
    a = run(p)
    b = run(p)
    np.testing.assert_array_equal(a, b)


def test_attention_workspace_reuse_across_shapes():
    # one workspace (sized for the largest call) through calls of different shapes: the split
    # counters each call leaves behind must be zero for the next
    big = problem(8, 4, 3, 128, 1300, (1300, 4, 600, 1200, 513, 512, 1024, 77), seed=5)
    small = problem(3, 2, 5, 64, 2100, (2100, 1025, 2), seed=6)
    ws = api.spec_verify_attention_workspace(8, 8, 2100, 5, 128)
    a1 = run(big, ws=ws)
    b1 = run(small, ws=ws)
    a2 = run(big, ws=ws)
    b2 = run(small, ws=ws)
    np.testing.assert_array_equal(a1, a2)
    np.testing.assert_array_equal(b1, b2)
    np.testing.assert_array_equal(a1, run(big))
    assert_layer_close(bf16_f64(b1), oracle.verify_attention(small.q, small.k_cache, small.v_cache, small.ctx_len,
                                                             1 / 8), "small after big")


def test_attention_bad_length_sets_the_error_word():
    p = problem(2, 4, 1, 64, 128, (100, 100), seed=1)
    bad = synth.AttentionProblem(p.B, p.Q, p.L, p.nh, p.d, p.q, p.k_cache, p.v_cache,
                                 np.array([100, 129], np.int32))
    assert api.get_device_error() == 0
    got = run(bad)
    assert api.get_device_error() == 7    # LSV_ERR_DEVICE_INDEX; reading the word clears it
    assert np.all(bf16_f64(got[1]) == 0)
    ref = oracle.verify_attention(p.q[:1], p.k_cache[:1], p.v_cache[:1], p.ctx_len[:1], 1 / 8)
    assert_layer_close(bf16_f64(got[:1]), ref, "good sequence beside a bad one")
