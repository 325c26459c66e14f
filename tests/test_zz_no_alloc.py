"""spec_verify_accept_noalloc: the acceptance entry point for callers that cannot allocate
device memory where they verify -- a host that runs the library as a plugin and passes only
the call's tensors, or a decode loop whose memory is fixed before it starts.  Its scratch is
a fixed array inside the library that every call shares, so each call must give exactly what
spec_verify_accept gives with a caller workspace (and what the oracle gives), whatever the
previous call left in that array.  This file is collected last: it passes on its own in a
fresh process and after every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from lossless_speculative_verification_gb300 import _ffi, api, synth

from gpu_util import need_gpu, to_dev

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _filled(shape):
    return torch.full(shape, -7, dtype=torch.int32, device="cuda")


def _reference(lg, dr, B, K, V):
    arg = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    alen, comm = api.spec_verify_accept(lg, dr, api.spec_verify_workspace(B, K, V), argmax=arg)
    return arg, alen, comm


def test_noalloc_matches_workspace_entry_point_and_oracle_on_consecutive_calls():
    need_gpu()
    lib = _ffi.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # calls in a row through the C ABI: the first (64 x 4 rows) writes more of the array than the
    # second (one sequence) and the third, so the later calls run over the earlier ones' leftovers
    for B, K, seed in [(64, 3, 0), (1, 3, 1), (32, 2, 2)]:
        w = synth.sweep_workload(B, K)
        logits, _, drafts = synth.verify_problem(w, seed=seed)
        lg = to_dev(logits)
        dr = torch.from_numpy(drafts).cuda()
        ref_arg, ref_len, ref_comm = _reference(lg, dr, B, K, w.V)
        arg, alen, comm = _filled((B, K + 1)), _filled((B,)), _filled((B, K + 1))
        rc = lib.spec_verify_accept_noalloc(_p(lg), _p(dr), B, K, w.V, _p(arg), _p(alen), _p(comm), stream)
        assert rc == _ffi.OK
        torch.cuda.synchronize()
        assert api.get_device_error() == 0
        # integer results: identical, bit for bit, to the workspace entry point and to the oracle
        assert torch.equal(arg, ref_arg) and torch.equal(alen, ref_len) and torch.equal(comm, ref_comm)
        o_arg, o_len, o_comm = oracle.accept(logits, drafts)
        np.testing.assert_array_equal(arg.cpu().numpy(), o_arg)
        np.testing.assert_array_equal(alen.cpu().numpy(), o_len)
        np.testing.assert_array_equal(comm.cpu().numpy(), o_comm)


def test_noalloc_through_the_python_binding():
    need_gpu()
    B, K = 16, 3
    w = synth.sweep_workload(B, K)
    logits, _, drafts = synth.verify_problem(w, seed=7)
    lg, dr = to_dev(logits), torch.from_numpy(drafts).cuda()
    ref_arg, ref_len, ref_comm = _reference(lg, dr, B, K, w.V)
    arg, alen, comm = _filled((B, K + 1)), _filled((B,)), _filled((B, K + 1))
    api.spec_verify_accept_noalloc(lg, dr, argmax=arg, accept_len=alen, committed=comm)
    torch.cuda.synchronize()
    assert torch.equal(arg, ref_arg) and torch.equal(alen, ref_len) and torch.equal(comm, ref_comm)
    with pytest.raises(ValueError):
        api.spec_verify_accept_noalloc(lg, dr[:, :2])                     # drafts must be [B, K]
    with pytest.raises(ValueError):
        api.spec_verify_accept_noalloc(lg, dr, argmax=torch.zeros((B, K + 1), dtype=torch.int64, device="cuda"))


def test_noalloc_at_its_largest_size_and_beyond():
    need_gpu()
    lib = _ffi.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    K, V = 3, 1024
    # the array holds 16,384 partials; a call needs what spec_verify_workspace_size reports for
    # it: the largest batch that fits, then one more
    cap = 2 * 16384 * 4
    B = 1
    while lib.spec_verify_workspace_size(2 * B, K, V) <= cap:
        B *= 2
    lo, hi = B, 2 * B                                     # fits at lo, not at hi
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if lib.spec_verify_workspace_size(mid, K, V) <= cap else (lo, mid)
    B = lo
    assert B * (K + 1) > 15000                            # one chunk per row here: up to 16,384 rows
    logits, planted = synth.verify_logits(B, K, V, seed=11)
    drafts = synth.draft_tokens(planted, V, [0.8, 0.6, 0.5], seed=12)
    lg, dr = to_dev(logits), torch.from_numpy(drafts).cuda()
    arg, alen, comm = _filled((B, K + 1)), _filled((B,)), _filled((B, K + 1))
    assert lib.spec_verify_accept_noalloc(_p(lg), _p(dr), B, K, V, _p(arg), _p(alen), _p(comm), stream) == _ffi.OK
    torch.cuda.synchronize()
    o_arg, o_len, o_comm = oracle.accept(logits, drafts)
    np.testing.assert_array_equal(arg.cpu().numpy(), o_arg)
    np.testing.assert_array_equal(alen.cpu().numpy(), o_len)
    np.testing.assert_array_equal(comm.cpu().numpy(), o_comm)
    # one sequence more does not fit; the call returns before any launch and leaves the outputs alone
    rc = lib.spec_verify_accept_noalloc(_p(lg), _p(dr), B + 1, K, V, _p(arg), _p(alen), _p(comm), stream)
    assert rc == _ffi.ERR_UNSUPPORTED
    t = torch.zeros(64, dtype=torch.int32, device="cuda")
    # 8192 sequences x 4 rows of 129,280 logits: refused before anything is read
    assert lib.spec_verify_accept_noalloc(_p(t), _p(t), 8192, 3, 129_280, None, _p(t), _p(t), None) == \
        _ffi.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert api.get_device_error() == 0
