"""The K policy (spec_k_policy, spec_cond_accept_from_histogram: host functions of
the library, no device work) against the oracle, and the device histogram of
accepted lengths (spec_accept_histogram) against np.bincount."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def api():
    from lossless_speculative_verification_gb300 import _build
    _build.build()
    from lossless_speculative_verification_gb300 import api
    return api


COSTS = [[1.0, 1.3, 1.6, 1.9], [1.0, 1.05, 1.3, 2.2], [1.0, 1.56, 2.2, 2.5], [2.0, 2.0, 2.0, 2.0],
         [1.0, 1.0, 10.0, 1.0]]


@pytest.mark.parametrize("cost", COSTS)
def test_k_policy_matches_the_oracle(api, cost):
    a = [0.830, 0.663, 0.636]
    k, tau, S = api.spec_k_policy(a, cost)
    k_ref, tau_ref, S_ref = oracle.k_policy(a, cost)
    assert k == k_ref
    np.testing.assert_allclose(tau, tau_ref, rtol=1e-14)
    np.testing.assert_allclose(S, S_ref, rtol=1e-14)


def test_k_policy_edges(api):
    assert api.spec_k_policy([], [3.0])[0] == 0                  # kmax = 0: greedy only
    assert api.spec_k_policy([1.0, 1.0], [1.0, 2.0, 3.0])[0] == 0  # S = 1 everywhere: the smaller K
    assert api.spec_k_policy([0.0, 0.5], [1.0, 0.5, 0.5])[0] == 1  # free drafts, none accepted: the cheaper step
    with pytest.raises(RuntimeError):
        api.spec_k_policy([1.5], [1.0, 1.0])
    with pytest.raises(RuntimeError):
        api.spec_k_policy([0.5], [1.0, 0.0])


def test_cond_accept_from_histogram_matches_the_oracle(api):
    rng = np.random.default_rng(3)
    for K in (1, 3, 7):
        L = np.minimum(rng.geometric(0.4, size=5000) - 1, K)
        hist = np.bincount(L, minlength=K + 1).astype(np.int64)
        np.testing.assert_allclose(api.spec_cond_accept_from_histogram(hist, K),
                                   oracle.cond_accept_from_lengths(L, K), rtol=1e-15)
    np.testing.assert_array_equal(api.spec_cond_accept_from_histogram(np.array([4, 0, 0], np.int64), 2), [0, 0])


@pytest.mark.gpu
def test_accept_histogram_on_the_gpu(api):
    import torch
    from gpu_util import need_gpu
    need_gpu()
    rng = np.random.default_rng(4)
    K = 3
    hist = None
    ref = np.zeros(K + 1, np.int64)
    for B in (1, 32, 1000, 70_000):
        L = rng.integers(0, K + 1, size=B).astype(np.int32)
        hist = api.spec_accept_histogram(torch.from_numpy(L).cuda(), K, hist)
        ref += np.bincount(L, minlength=K + 1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hist.cpu().numpy(), ref)
    assert api.get_device_error() == 0
    bad = torch.tensor([0, 4, 1], dtype=torch.int32, device="cuda")
    h2 = api.spec_accept_histogram(bad, K)
    torch.cuda.synchronize()
    assert api.get_device_error() == 7
    np.testing.assert_array_equal(h2.cpu().numpy(), [1, 1, 0, 0])
