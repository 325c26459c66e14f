"""spec_verify_accept_noalloc: the acceptance entry point for callers that cannot
allocate device memory when they verify (inside a stream capture, inside a
latency-critical decode loop, or in a host that offers no allocator or
workspace).  Its scratch is a fixed array inside the library, so it must give
exactly what spec_verify_accept gives with a caller workspace, call after call,
whatever the previous call left in that array.  This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

from lossless_speculative_verification_gb300 import _ffi, api, synth

from gpu_util import need_gpu, to_dev

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    need_gpu()
    lib = _ffi.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two calls in a row with different shapes: the second sees the first one's leftovers in the scratch
    for B, K, seed in [(32, 3, 0), (64, 2, 1)]:
        w = synth.sweep_workload(B, K)
        logits, _, drafts = synth.verify_problem(w, seed=seed)
        lg = to_dev(logits)
        dr = torch.from_numpy(drafts).cuda()
        ref_arg = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
        ws = api.spec_verify_workspace(B, K, w.V)
        ref_len, ref_comm = api.spec_verify_accept(lg, dr, ws, argmax=ref_arg)
        arg = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
        alen = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        comm = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
        rc = lib.spec_verify_accept_noalloc(_p(lg), _p(dr), B, K, w.V, _p(arg), _p(alen), _p(comm), stream)
        assert rc == _ffi.OK
        torch.cuda.synchronize()
        assert api.get_device_error() == 0
        # integer results: identical, bit for bit
        assert torch.equal(arg, ref_arg)
        assert torch.equal(alen, ref_len)
        assert torch.equal(comm, ref_comm)


def test_noalloc_refuses_problems_beyond_its_scratch():
    need_gpu()
    lib = _ffi.load()
    t = torch.zeros(64, dtype=torch.int32, device="cuda")
    # 8192 sequences x 4 rows = 32768 rows needs more partials than the fixed array holds;
    # the call returns before any launch, so the small dummy buffers are never read
    rc = lib.spec_verify_accept_noalloc(_p(t), _p(t), 8192, 3, 129_280, None, _p(t), _p(t), None)
    assert rc == _ffi.ERR_UNSUPPORTED
