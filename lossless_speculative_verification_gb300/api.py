"""Python surface of the C ABI: the same entry points, taking torch CUDA tensors.

Each function checks dtypes/devices, passes data pointers and the current
CUDA stream to liblsv.so, and returns the output tensors.  Every step of the
computation runs in the library's kernels.  Workspaces are passed explicitly
(the library allocates nothing); `workspace(...)` sizes one.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _ffi
from ._ffi import MoeShape, MoeWeights, check


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _need_shape(t, shape, name):
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _verify_outputs(logits, drafts, argmax, accept_len, committed):
    """Check the acceptance call's tensors against logits [B, K+1, V]; allocate missing outputs."""
    _need(logits, torch.bfloat16, "logits"); _need(drafts, torch.int32, "drafts")
    if logits.dim() != 3:
        raise ValueError("logits must be [B, K+1, V]")
    B, K1, V = logits.shape
    _need_shape(drafts, (B, K1 - 1), "drafts")
    for name, t, shp in (("argmax", argmax, (B, K1)), ("accept_len", accept_len, (B,)),
                         ("committed", committed, (B, K1))):
        _need(t, torch.int32, name)
        _need_shape(t, shp, name)
    dev = logits.device
    accept_len = torch.empty(B, dtype=torch.int32, device=dev) if accept_len is None else accept_len
    committed = torch.empty((B, K1), dtype=torch.int32, device=dev) if committed is None else committed
    return B, K1 - 1, V, accept_len, committed


def shape(T, H, E, k, S, I) -> MoeShape:
    return MoeShape(T, H, E, k, S, I)


def weights(w_router, w_gate_up, w_down, ws_gate_up=None, ws_down=None) -> MoeWeights:
    for n, t in (("w_router", w_router), ("w_gate_up", w_gate_up), ("w_down", w_down),
                 ("ws_gate_up", ws_gate_up), ("ws_down", ws_down)):
        _need(t, torch.bfloat16, n)
    w = MoeWeights(*(t.data_ptr() if t is not None else None
                     for t in (w_router, w_gate_up, w_down, ws_gate_up, ws_down)))
    # the struct holds raw pointers: keep the tensors alive as long as the struct
    w._tensors = (w_router, w_gate_up, w_down, ws_gate_up, ws_down)
    return w


def workspace_size(sh: MoeShape) -> int:
    n = _ffi.load().lsv_workspace_size(ctypes.byref(sh))
    if n == 0:
        raise ValueError("unsupported MoE shape")
    return int(n)


def workspace(sh: MoeShape, device=None) -> torch.Tensor:
    """Zero-filled: the layer wants the workspace's counter block zero before the first call."""
    return torch.zeros(workspace_size(sh), dtype=torch.uint8, device=device or "cuda")


def moe_prefetch_weights(w: MoeWeights, sh: MoeShape, max_bytes: int, stream=None) -> None:
    check("moe_prefetch_weights", _ffi.load().moe_prefetch_weights(ctypes.byref(w), ctypes.byref(sh), max_bytes,
                                                                   _stream(stream)))


def moe_route(x, w_router, k, topk_idx=None, topk_w=None, logits=None, stream=None):
    _need(x, torch.bfloat16, "x"); _need(w_router, torch.bfloat16, "w_router")
    T, H = x.shape
    E = w_router.shape[0]
    sh = MoeShape(T, H, E, k, 0, 64)
    topk_idx = torch.empty((T, k), dtype=torch.int32, device=x.device) if topk_idx is None else topk_idx
    topk_w = torch.empty((T, k), dtype=torch.float32, device=x.device) if topk_w is None else topk_w
    check("moe_route", _ffi.load().moe_route(_ptr(x), _ptr(w_router), ctypes.byref(sh), _ptr(topk_idx),
                                             _ptr(topk_w), _ptr(logits), _stream(stream)))
    return topk_idx, topk_w


def moe_permute(topk_idx, E, ws, H=64, S=0, I=64, stream=None):
    _need(topk_idx, torch.int32, "topk_idx")
    T, k = topk_idx.shape
    sh = MoeShape(T, H, E, k, S, I)
    dev = topk_idx.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    check("moe_permute", _ffi.load().moe_permute(_ptr(topk_idx), ctypes.byref(sh), _ptr(counts), _ptr(offsets),
                                                 _ptr(perm), _ptr(inv), _ptr(ws), ws.numel(), _stream(stream)))
    return counts, offsets, perm, inv


def moe_grouped_ffn(x, perm, offsets, counts, w: MoeWeights, sh: MoeShape, ws, y_perm=None, y_shared=None,
                    stream=None):
    _need(x, torch.bfloat16, "x")
    dev = x.device
    if y_perm is None:
        y_perm = torch.empty((sh.T * sh.k, sh.H), dtype=torch.float32, device=dev)
    if y_shared is None and sh.S > 0:
        y_shared = torch.empty((sh.T, sh.H), dtype=torch.float32, device=dev)
    check("moe_grouped_ffn", _ffi.load().moe_grouped_ffn(
        _ptr(x), _ptr(perm), _ptr(offsets), _ptr(counts), ctypes.byref(w), ctypes.byref(sh), _ptr(y_perm),
        _ptr(y_shared), _ptr(ws), ws.numel(), _stream(stream)))
    return y_perm, y_shared


def moe_combine(y_perm, inv, topk_w, y_shared, sh: MoeShape, out=None, stream=None):
    out = torch.empty((sh.T, sh.H), dtype=torch.bfloat16, device=y_perm.device) if out is None else out
    check("moe_combine", _ffi.load().moe_combine(_ptr(y_perm), _ptr(inv), _ptr(topk_w), _ptr(y_shared),
                                                 ctypes.byref(sh), _ptr(out), _stream(stream)))
    return out


def moe_verify_layer(x, w: MoeWeights, sh: MoeShape, ws, out=None, topk_idx=None, counts=None, stream=None):
    _need(x, torch.bfloat16, "x")
    out = torch.empty((sh.T, sh.H), dtype=torch.bfloat16, device=x.device) if out is None else out
    check("moe_verify_layer", _ffi.load().moe_verify_layer(
        _ptr(x), ctypes.byref(w), ctypes.byref(sh), _ptr(out), _ptr(topk_idx), _ptr(counts), _ptr(ws),
        ws.numel(), _stream(stream)))
    return out


def spec_verify_workspace(B, K, V, device=None) -> torch.Tensor:
    n = _ffi.load().spec_verify_workspace_size(B, K, V)
    if n == 0:
        raise ValueError("unsupported verify shape")
    return torch.empty(int(n), dtype=torch.uint8, device=device or "cuda")


def spec_verify_accept(logits, drafts, ws, argmax=None, accept_len=None, committed=None, stream=None):
    B, K, V, accept_len, committed = _verify_outputs(logits, drafts, argmax, accept_len, committed)
    check("spec_verify_accept", _ffi.load().spec_verify_accept(
        _ptr(logits), _ptr(drafts), B, K, V, _ptr(argmax), _ptr(accept_len), _ptr(committed), _ptr(ws),
        ws.numel(), _stream(stream)))
    return accept_len, committed


def spec_verify_attention_workspace(B, Q, L, nh, d, device=None) -> torch.Tensor:
    """Workspace of spec_verify_attention, zeroed (its counters must start at zero; every call
    leaves them zero)."""
    n = _ffi.load().spec_verify_attention_workspace_size(B, Q, L, nh, d)
    if n == 0:
        raise ValueError("unsupported attention shape")
    return torch.zeros(int(n), dtype=torch.uint8, device=device or "cuda")


def spec_verify_attention(q, k_cache, v_cache, ctx_len, ws, scale=None, out=None, stream=None):
    """Causal attention of the verified positions q [B, Q, nh, d] over the caches [B, L, nh, d]."""
    _need(q, torch.bfloat16, "q"); _need(k_cache, torch.bfloat16, "k_cache"); _need(v_cache, torch.bfloat16, "v_cache")
    _need(ctx_len, torch.int32, "ctx_len")
    B, Q, nh, d = q.shape
    L = k_cache.shape[1]
    if tuple(k_cache.shape) != (B, L, nh, d) or tuple(v_cache.shape) != (B, L, nh, d):
        raise ValueError("k_cache and v_cache must be [B, L, nh, d] = [%d, L, %d, %d]" % (B, nh, d))
    if tuple(ctx_len.shape) != (B,):
        raise ValueError("ctx_len must be [B]")
    for t, name in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    if tuple(out.shape) != (B, Q, nh, d) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 [B, Q, nh, d] tensor")
    check("spec_verify_attention", _ffi.load().spec_verify_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(ctx_len), B, Q, L, nh, d, scale, _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream)))
    return out


def dense_matmul(x, w, out=None, stream=None):
    """out [M, N] = bf16(x [M, K] w [N, K]^T) on the tensor cores."""
    _need(x, torch.bfloat16, "x"); _need(w, torch.bfloat16, "w")
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or not x.is_contiguous() or not w.is_contiguous():
        raise ValueError("x [M, K] and w [N, K] must be contiguous with the same K")
    out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device) if out is None else out
    check("dense_matmul", _ffi.load().dense_matmul(_ptr(x), _ptr(w), _ptr(out), M, N, K, _stream(stream)))
    return out


def gather_rows(table, idx, out=None, stream=None):
    """out[i] = table[idx[i]] (bf16 rows; e.g. the embedding rows of the verified tokens)."""
    _need(table, torch.bfloat16, "table"); _need(idx, torch.int32, "idx")
    n_table, row = table.shape
    n = idx.numel()
    out = torch.empty((n, row), dtype=torch.bfloat16, device=table.device) if out is None else out
    _need(out, torch.bfloat16, "out")
    _need_shape(out, (n, row), "out")
    check("lsv_gather_rows", _ffi.load().lsv_gather_rows(_ptr(table), _ptr(idx), n, n_table, row, _ptr(out),
                                                         _stream(stream)))
    return out


def spec_cache_append(k_new, v_new, k_cache, v_cache, ctx_len, stream=None):
    """Keys and values of the Q verified positions [B, Q, ...] into the caches [B, L, ...] at
    ctx_len[b] - Q + j (ctx_len: the lengths after the append)."""
    for n, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, torch.bfloat16, n)
    _need(ctx_len, torch.int32, "ctx_len")
    B, Q = k_new.shape[:2]
    L = k_cache.shape[1]
    row = k_new[0, 0].numel()
    if k_cache.shape[0] != B or k_cache[0, 0].numel() != row or v_new.shape != k_new.shape or \
            v_cache.shape != k_cache.shape:
        raise ValueError("k_new/v_new [B, Q, ...] and caches [B, L, ...] with the same row width")
    check("spec_cache_append", _ffi.load().spec_cache_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                                             _ptr(ctx_len), B, Q, L, row, _stream(stream)))


def dense_swiglu(x, w_gate_up, out=None, stream=None):
    """out [M, F] = bf16(silu(x w_gate^T) * (x w_up^T)) with w_gate_up = [w_gate; w_up] [2F, K],
    for few rows of x (M <= 256)."""
    _need(x, torch.bfloat16, "x"); _need(w_gate_up, torch.bfloat16, "w_gate_up")
    M, K = x.shape
    if w_gate_up.shape[1] != K or w_gate_up.shape[0] % 2:
        raise ValueError("x [M, K] and w_gate_up [2F, K] must have the same K")
    F = w_gate_up.shape[0] // 2
    out = torch.empty((M, F), dtype=torch.bfloat16, device=x.device) if out is None else out
    _need(out, torch.bfloat16, "out")
    _need_shape(out, (M, F), "out")
    check("dense_swiglu", _ffi.load().dense_swiglu(_ptr(x), _ptr(w_gate_up), _ptr(out), M, F, K, _stream(stream)))
    return out


DRAFT_WEIGHTS = ("emb", "w_proj", "w_q", "w_k", "w_v", "w_o", "w_gate_up", "w_down", "w_vocab")


def spec_draft_workspace(B, H, nh, I, V, L, device=None) -> torch.Tensor:
    """Workspace of spec_draft_loop, zeroed (its sub-workspaces need zero on first use)."""
    n = _ffi.load().spec_draft_workspace_size(B, H, nh, I, V, L)
    if n == 0:
        raise ValueError("unsupported draft-block shape")
    return torch.zeros(int(n), dtype=torch.uint8, device=device or "cuda")


def spec_draft_loop(weights, h0, t0, k_cache, v_cache, ctx_len, K, ws, h_out=None, out=None, stream=None):
    """K recursive draft-block steps; returns drafts [B, K] int32 (the caches get the K new entries)."""
    for n in DRAFT_WEIGHTS:
        _need(weights[n], torch.bfloat16, n)
    _need(h0, torch.bfloat16, "h0"); _need(t0, torch.int32, "t0"); _need(ctx_len, torch.int32, "ctx_len")
    _need(k_cache, torch.bfloat16, "k_cache"); _need(v_cache, torch.bfloat16, "v_cache")
    B, H = h0.shape
    _, L, nh, d = k_cache.shape
    V = weights["w_vocab"].shape[0]
    I = weights["w_down"].shape[1]
    if tuple(v_cache.shape) != tuple(k_cache.shape) or nh * d != H or k_cache.shape[0] != B:
        raise ValueError("caches must be [B, L, nh, H/nh]")
    w = _ffi.DraftWeights(*[_ptr(weights[n]) for n in DRAFT_WEIGHTS])
    drafts = torch.empty((B, K), dtype=torch.int32, device=h0.device) if out is None else out
    _need(drafts, torch.int32, "out")
    _need_shape(drafts, (B, K), "out")
    check("spec_draft_loop", _ffi.load().spec_draft_loop(
        ctypes.byref(w), _ptr(h0), _ptr(t0), _ptr(k_cache), _ptr(v_cache), _ptr(ctx_len), B, K, H, nh, I, V, L,
        _ptr(drafts), _ptr(h_out), _ptr(ws), ws.numel(), _stream(stream)))
    return drafts


def spec_k_policy(cond_accept, step_cost):
    """(k_best, tau [kmax+1], speedup [kmax+1]) from conditional acceptances and step costs."""
    import numpy as np
    a = np.ascontiguousarray(cond_accept, dtype=np.float64)
    c = np.ascontiguousarray(step_cost, dtype=np.float64)
    kmax = a.size
    if c.size != kmax + 1:
        raise ValueError("step_cost needs one entry per K = 0..kmax")
    k = ctypes.c_int32(0)
    tau = np.zeros(kmax + 1, np.float64)
    sp = np.zeros(kmax + 1, np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    check("spec_k_policy", _ffi.load().spec_k_policy(
        a.ctypes.data_as(dp) if kmax else None, kmax, c.ctypes.data_as(dp), ctypes.byref(k),
        tau.ctypes.data_as(dp), sp.ctypes.data_as(dp)))
    return int(k.value), tau, sp


def spec_accept_histogram(accept_len, K, hist=None, stream=None):
    """Add the batch's accepted lengths to hist [K+1] int64 (device; created zeroed if None)."""
    _need(accept_len, torch.int32, "accept_len")
    if hist is None:
        hist = torch.zeros(K + 1, dtype=torch.int64, device=accept_len.device)
    check("spec_accept_histogram", _ffi.load().spec_accept_histogram(
        _ptr(accept_len), accept_len.numel(), K, _ptr(hist), _stream(stream)))
    return hist


def spec_cond_accept_from_histogram(hist, K):
    import numpy as np
    h = np.ascontiguousarray(hist.cpu().numpy() if isinstance(hist, torch.Tensor) else hist, dtype=np.int64)
    cond = np.zeros(max(K, 1), np.float64)
    check("spec_cond_accept_from_histogram", _ffi.load().spec_cond_accept_from_histogram(
        h.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), K, cond.ctypes.data_as(ctypes.POINTER(ctypes.c_double))))
    return cond[:K]


def spec_verify_lmhead_workspace(B, K, V, H, device=None) -> torch.Tensor:
    n = _ffi.load().spec_verify_lmhead_workspace_size(B, K, V, H)
    if n == 0:
        raise ValueError("unsupported verify shape")
    return torch.empty(int(n), dtype=torch.uint8, device=device or "cuda")


def spec_verify_lmhead(hidden, w_vocab, drafts, ws, K, argmax=None, accept_len=None, committed=None, stream=None):
    """Greedy verification with the logits produced by the output layer w_vocab [V, H] from
    hidden [B*(K+1), H] inside the call."""
    _need(hidden, torch.bfloat16, "hidden"); _need(w_vocab, torch.bfloat16, "w_vocab"); _need(drafts, torch.int32, "drafts")
    R, H = hidden.shape
    V = w_vocab.shape[0]
    if R % (K + 1):
        raise ValueError("hidden rows must be B*(K+1)")
    B = R // (K + 1)
    dev = hidden.device
    accept_len = torch.empty(B, dtype=torch.int32, device=dev) if accept_len is None else accept_len
    committed = torch.empty((B, K + 1), dtype=torch.int32, device=dev) if committed is None else committed
    check("spec_verify_lmhead", _ffi.load().spec_verify_lmhead(
        _ptr(hidden), _ptr(w_vocab), _ptr(drafts), B, K, V, H, _ptr(argmax), _ptr(accept_len), _ptr(committed),
        _ptr(ws), ws.numel(), _stream(stream)))
    return accept_len, committed


def spec_verify_accept_noalloc(logits, drafts, argmax=None, accept_len=None, committed=None, stream=None):
    """spec_verify_accept without a workspace, for callers that cannot allocate device memory
    where they verify (a plugin host that passes only the call's tensors, a decode loop whose
    memory is fixed in advance): its scratch is a fixed array inside the library.  The outputs
    it is not given are allocated here, by torch, so a caller that may not allocate passes them."""
    B, K, V, accept_len, committed = _verify_outputs(logits, drafts, argmax, accept_len, committed)
    check("spec_verify_accept_noalloc", _ffi.load().spec_verify_accept_noalloc(
        _ptr(logits), _ptr(drafts), B, K, V, _ptr(argmax), _ptr(accept_len), _ptr(committed),
        _stream(stream)))
    return accept_len, committed


def rmsnorm_residual(x, y, h=None, eps=1e-6, stream=None):
    _need(x, torch.bfloat16, "x"); _need(y, torch.bfloat16, "y")
    T, H = x.shape
    h = torch.empty_like(x) if h is None else h
    check("rmsnorm_residual", _ffi.load().rmsnorm_residual(_ptr(x), _ptr(y), _ptr(h), T, H, eps, _stream(stream)))
    return h


def get_device_error(stream=None) -> int:
    v = ctypes.c_int32(0)
    check("lsv_get_device_error", _ffi.load().lsv_get_device_error(ctypes.byref(v), _stream(stream)))
    return int(v.value)


def set_wait_limit_ns(ns: int) -> None:
    check("lsv_set_wait_limit_ns", _ffi.load().lsv_set_wait_limit_ns(ns))


def selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    check("lsv_selftest_wait_timeout", _ffi.load().lsv_selftest_wait_timeout(limit_ns, _stream(stream)))
