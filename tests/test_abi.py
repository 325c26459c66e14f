"""The C-ABI library: it builds, loads, exports every symbol include/lsv.h
declares, and rejects bad arguments on the host without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from lossless_speculative_verification_gb300 import _build, _ffi
    _build.build()
    return _ffi.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "lsv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(", src, re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


def test_header_declares_the_boundary():
    names = header_functions()
    for n in ["moe_route", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_verify_layer",
              "spec_verify_accept", "lsv_workspace_size", "lsv_get_device_error", "lsv_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from lossless_speculative_verification_gb300 import _ffi
    for n in header_functions():
        assert hasattr(lib, n), n
        assert n in _ffi.SIGNATURES, "binding lacks " + n
    assert lib.lsv_version() == 100


def test_status_strings(lib):
    assert lib.lsv_status_string(0) == b"ok"
    assert lib.lsv_status_string(6) == b"device wait timed out"
    assert lib.lsv_status_string(99) == b"unknown status"


def test_workspace_size_is_host_only_and_validates(lib):
    from lossless_speculative_verification_gb300._ffi import MoeShape
    ok = MoeShape(128, 1280, 64, 6, 2, 896)
    n = lib.lsv_workspace_size(ctypes.byref(ok))
    assert n > 0 and n % 256 == 0
    # x_perm + act + act_sh + y_perm + y_sh at least
    assert n >= 768 * 1280 * 2 + 768 * 896 * 2 + 128 * 1792 * 2 + 768 * 1280 * 4 + 128 * 1280 * 4
    for bad in [MoeShape(128, 1000, 64, 6, 2, 896),   # H % 64
                MoeShape(128, 1280, 64, 9, 2, 896),   # k > 8
                MoeShape(128, 1280, 4, 6, 2, 896),    # k > E
                MoeShape(-1, 1280, 64, 6, 2, 896),
                MoeShape(128, 1280, 300, 6, 2, 896),  # E > 256
                MoeShape(128, 1280, 64, 6, 2, 900)]:  # I % 64
        assert lib.lsv_workspace_size(ctypes.byref(bad)) == 0
    assert lib.lsv_workspace_size(None) == 0


def test_argument_errors_return_before_any_launch(lib):
    from lossless_speculative_verification_gb300._ffi import MoeShape, MoeWeights
    sh = MoeShape(16, 256, 8, 2, 1, 128)
    bad = MoeShape(16, 250, 8, 2, 1, 128)
    p16 = ctypes.c_void_p(0x10000)
    p_odd = ctypes.c_void_p(0x10008)
    # NULL / unsupported / misaligned: all decided on the host
    assert lib.moe_route(None, p16, ctypes.byref(sh), p16, p16, None, None) == 1
    assert lib.moe_route(p16, p16, ctypes.byref(bad), p16, p16, None, None) == 2
    assert lib.moe_route(p16, p_odd, ctypes.byref(sh), p16, p16, None, None) == 3
    assert lib.moe_combine(p16, p16, p16, None, ctypes.byref(sh), p16, None) == 1   # S > 0 needs y_shared
    w = MoeWeights(p16.value, p16.value, None, p16.value, p16.value)
    assert lib.moe_verify_layer(p16, ctypes.byref(w), ctypes.byref(sh), p16, None, None, p16, 1 << 30, None) == 1
    w = MoeWeights(p16.value, p16.value, p16.value, p16.value, p16.value)
    assert lib.moe_verify_layer(p16, ctypes.byref(w), ctypes.byref(sh), p16, None, None, None, 0, None) == 4
    assert lib.moe_verify_layer(p16, ctypes.byref(w), ctypes.byref(sh), p16, None, None, p16, 16, None) == 4
    assert lib.moe_permute(p16, ctypes.byref(sh), None, p16, p16, p16, p16, 1 << 30, None) == 1
    assert lib.spec_verify_accept(p16, p16, 4, 64, 1024, None, p16, p16, p16, 1 << 20, None) == 2   # K+1 > 64
    assert lib.spec_verify_accept(p16, p16, -1, 3, 1024, None, p16, p16, p16, 1 << 20, None) == 1
    assert lib.spec_verify_accept(None, p16, 4, 3, 1024, None, p16, p16, p16, 1 << 20, None) == 1
    assert lib.spec_verify_accept(p_odd, p16, 4, 3, 1024, None, p16, p16, p16, 1 << 20, None) == 3
    assert lib.rmsnorm_residual(p16, p16, None, 4, 256, 1e-6, None) == 1
    # verifier output layer: unsupported hidden width, missing input, misaligned, empty batch
    assert lib.spec_verify_lmhead_workspace_size(4, 3, 1000, 250) == 0
    assert lib.spec_verify_lmhead(p16, p16, p16, 4, 3, 1000, 250, None, p16, p16, p16, 1 << 20, None) == 2
    assert lib.spec_verify_lmhead(None, p16, p16, 4, 3, 1000, 256, None, p16, p16, p16, 1 << 20, None) == 1
    assert lib.spec_verify_lmhead(p_odd, p16, p16, 4, 3, 1000, 256, None, p16, p16, p16, 1 << 20, None) == 3
    assert lib.spec_verify_lmhead(p16, p16, p16, 4, 3, 1000, 256, None, p16, p16, p16, 16, None) == 4
    assert lib.spec_verify_lmhead(None, None, None, 0, 3, 1000, 256, None, None, None, None, 0, None) == 0
    # attention: d outside {64, 128} and Q above 8 are unsupported; null, misaligned, small workspace
    assert lib.spec_verify_attention_workspace_size(4, 4, 1024, 10, 96) == 0
    assert lib.spec_verify_attention_workspace_size(4, 9, 1024, 10, 128) == 0
    assert lib.spec_verify_attention_workspace_size(4, 4, 3, 10, 128) == 0
    need = lib.spec_verify_attention_workspace_size(4, 4, 1024, 10, 128)
    assert need >= 4 * 10 * 2 * 4 * (128 * 4 + 8)
    att = lambda q, B, Q, d, scale, ws_bytes: lib.spec_verify_attention(q, p16, p16, p16, B, Q, 1024, 10, d, scale,
                                                                        p16, p16, ws_bytes, None)
    assert att(p16, 4, 4, 96, 0.1, need) == 2
    assert att(p16, 4, 4, 128, 0.0, need) == 1
    assert att(None, 4, 4, 128, 0.1, need) == 1
    assert att(p_odd, 4, 4, 128, 0.1, need) == 3
    assert att(p16, 4, 4, 128, 0.1, need - 1) == 4
    assert lib.spec_verify_attention(None, None, None, None, 0, 4, 1024, 10, 128, 0.1, None, None, 0, None) == 0
    # attention limits: cache capacity, (sequence, head) pairs
    assert lib.spec_verify_attention_workspace_size(4, 4, 65537, 10, 128) == 0
    assert lib.spec_verify_attention_workspace_size(30000, 4, 1024, 10, 128) == 0
    assert lib.spec_verify_attention_workspace_size(0, 4, 1024, 10, 128) > 0
    # policy and histogram limits
    cost = (ctypes.c_double * 65)(*([1.0] * 65))
    kb = ctypes.c_int32(0)
    assert lib.spec_k_policy(cost, 64, cost, ctypes.byref(kb), None, None) == 2
    assert lib.spec_k_policy(None, 1, cost, ctypes.byref(kb), None, None) == 1
    assert lib.spec_accept_histogram(p16, 4, 64, p16, None) == 2
    assert lib.spec_accept_histogram(p16, -1, 3, p16, None) == 1
    assert lib.spec_accept_histogram(None, 0, 3, None, None) == 0
    assert lib.spec_cond_accept_from_histogram(None, 3, None) == 1
    # dense product: K % 64, N % 8; null, misaligned
    assert lib.dense_matmul(p16, p16, p16, 4, 8, 100, None) == 2
    assert lib.dense_matmul(p16, p16, p16, 4, 12, 128, None) == 2
    assert lib.dense_matmul(None, p16, p16, 4, 8, 128, None) == 1
    assert lib.dense_matmul(p_odd, p16, p16, 4, 8, 128, None) == 3
    assert lib.dense_matmul(None, None, None, 0, 8, 128, None) == 0
    # draft loop: unsupported head width, workspace sizes, small workspace
    assert lib.spec_draft_workspace_size(4, 1280, 5, 7168, 1000, 2048) == 0       # d = 256
    assert lib.spec_draft_workspace_size(4, 1280, 10, 7100, 1000, 2048) == 0      # I % 64
    assert lib.spec_draft_workspace_size(4, 1280, 10, 7168, 1000, 2048) > 0
    from lossless_speculative_verification_gb300 import _ffi
    dw = _ffi.DraftWeights(*([p16] * 9))
    assert lib.spec_draft_loop(ctypes.byref(dw), p16, p16, p16, p16, p16, 4, 3, 1280, 10, 7168, 1000, 2048, p16,
                               None, p16, 16, None) == 4
    assert lib.spec_draft_loop(ctypes.byref(dw), p16, p16, p16, p16, p16, 4, 0, 1280, 10, 7168, 1000, 2048, p16,
                               None, p16, 1 << 30, None) == 1
    assert lib.lsv_set_wait_limit_ns(0) == 1
    assert lib.lsv_selftest_wait_timeout(0, None) == 1
    # empty work is a no-op that succeeds without a device
    empty = MoeShape(0, 256, 8, 2, 1, 128)
    assert lib.moe_route(None, None, ctypes.byref(empty), None, None, None, None) == 0
    assert lib.spec_verify_accept(None, None, 0, 3, 1024, None, None, None, None, 0, None) == 0


def test_product_path_has_no_oracle_dependency():
    """The package and the CUDA sources never import, link or name the oracle."""
    pkg = os.path.join(ROOT, "lossless_speculative_verification_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "liboracle" not in src and "oracle.c" not in src, f
