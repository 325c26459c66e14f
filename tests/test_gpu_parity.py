"""GPU path vs the CPU oracle, call by call through the C ABI, on the same
seeded inputs.  Integer results (routing, permutation, counts, greedy tokens,
acceptance) must match bit for bit; floating-point layer outputs within
rel-L2 <= 1e-2 and max-abs <= 2e-2 (bf16 tensor-core products against the
fp64 oracle)."""
import functools

import numpy as np
import pytest
import torch

import oracle
from lossless_speculative_verification_gb300 import api, synth

from gpu_util import (DevProblem, assert_layer_close, bf16_f64, dev_problem, from_dev_bf16, need_gpu,
                      sample_rows, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    yield
    torch.cuda.synchronize()
    assert api.get_device_error() == 0


# ----------------------------------------------------------------------------- router
@pytest.mark.parametrize("name", ["tiny", "decode", "prefill"])
def test_route_parity(name):
    P = dev_problem(name)
    d = P.d
    logits = torch.empty((d.T, d.E), dtype=torch.float32, device="cuda")
    idx, w = api.moe_route(P.x, P.w_router, d.k, logits=logits)
    torch.cuda.synchronize()
    ref = P.oracle_route()
    np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"])
    # both sides accumulate exact bf16 products in fp32, in different orders
    np.testing.assert_allclose(logits.cpu().numpy(), ref["logits"], rtol=0, atol=2e-5)
    np.testing.assert_allclose(w.cpu().numpy(), ref["p"], rtol=1e-5, atol=1e-9)


@pytest.mark.parametrize("T,H,E,k", [(300, 256, 8, 2), (257, 1280, 64, 6), (513, 512, 128, 8),
                                     (1000, 256, 256, 6), (640, 1280, 64, 1)])
def test_route_parity_tensor_core_path(T, H, E, k):
    """Above 256 tokens the router runs on tcgen05 (one lane per token); every padded width."""
    d = synth.MoeDims(T, H, E, k, 0, 64)
    prob = synth.moe_problem(d, seed=T + E, hidden="sphere", row_ok=oracle.gap_ok(k))
    x, wr = to_dev(prob.x), to_dev(prob.w_router)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    idx, w = api.moe_route(x, wr, k, logits=logits)
    torch.cuda.synchronize()
    ridx, rp, rlog = oracle.route(prob.x, prob.w_router, k, return_logits=True)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(logits.cpu().numpy(), rlog, rtol=0, atol=2e-5 * np.sqrt(H / 256))
    np.testing.assert_allclose(w.cpu().numpy(), rp, rtol=1e-5, atol=1e-9)


@pytest.mark.parametrize("T,H,E,k", [(1, 1280, 64, 6), (37, 2048, 128, 4), (97, 1280, 64, 6), (128, 512, 256, 8),
                                     (129, 1280, 64, 6), (193, 512, 256, 8), (256, 256, 8, 2), (255, 1280, 64, 1)])
def test_route_parity_cuda_core_paths(T, H, E, k):
    """Up to 128 tokens the router runs as clusters of eight CTAs over one or two tokens (ragged last
    cluster included), each CTA an eighth of the experts; from 129 to 256 tokens as one CTA per token.
    H past one 1,280-wide pass of the lanes."""
    d = synth.MoeDims(T, H, E, k, 0, 64)
    prob = synth.moe_problem(d, seed=3 * T + E, hidden="sphere", row_ok=oracle.gap_ok(k))
    x, wr = to_dev(prob.x), to_dev(prob.w_router)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    idx, w = api.moe_route(x, wr, k, logits=logits)
    torch.cuda.synchronize()
    ridx, rp, rlog = oracle.route(prob.x, prob.w_router, k, return_logits=True)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(logits.cpu().numpy(), rlog, rtol=0, atol=2e-5 * np.sqrt(H / 256))
    np.testing.assert_allclose(w.cpu().numpy(), rp, rtol=1e-5, atol=1e-9)


# ----------------------------------------------------------------------------- permutation
def random_routing(T, k, E, seed):
    rs = np.random.default_rng(seed)
    return np.argsort(rs.random((T, E)), axis=1)[:, :k].astype(np.int32)


@pytest.mark.parametrize("T,k,E", [(16, 2, 8), (128, 6, 64), (1, 1, 1), (9760, 6, 64), (20000, 8, 256),
                                   (1365, 6, 64), (0, 6, 64)])
def test_permute_parity(T, k, E):
    idx = random_routing(T, k, E, T + k)
    sh = api.shape(T, 64, E, k, 0, 64)
    ws = api.workspace(sh)
    counts, offsets, perm, inv = api.moe_permute(torch.from_numpy(idx).cuda().reshape(T, k), E, ws)
    torch.cuda.synchronize()
    rc, ro, rp, ri = oracle.permute(idx, E)
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(perm.cpu().numpy(), rp)
    np.testing.assert_array_equal(inv.cpu().numpy(), ri)


def test_permute_reports_out_of_range_index():
    idx = random_routing(64, 2, 8, 3)
    idx[5, 1] = 8
    sh = api.shape(64, 64, 8, 2, 0, 64)
    ws = api.workspace(sh)
    api.moe_permute(torch.from_numpy(idx).cuda(), 8, ws)
    torch.cuda.synchronize()
    assert api.get_device_error() == 7
    assert api.get_device_error() == 0


# ----------------------------------------------------------------------------- grouped experts
@pytest.mark.parametrize("name,nsample", [("tiny", 10**9), ("decode", 10**9), ("prefill", 160)])
def test_grouped_ffn_parity(name, nsample):
    P = dev_problem(name)
    d, prob = P.d, P.prob
    r = P.oracle_route()
    dev = lambda a: torch.from_numpy(a).cuda()
    y_perm, y_sh = api.moe_grouped_ffn(P.x, dev(r["perm"]), dev(r["offsets"]), dev(r["counts"]), P.wts, P.sh, P.ws)
    torch.cuda.synchronize()
    rows = sample_rows(d.T * d.k, nsample, 1)
    # also every row of the least- and most-loaded experts (ragged token tiles)
    for e in (int(np.argmin(r["counts"])), int(np.argmax(r["counts"]))):
        rows = np.union1d(rows, np.arange(r["offsets"][e], r["offsets"][e + 1]))
    expert = np.searchsorted(r["offsets"], rows, side="right") - 1
    token = r["perm"][rows] // d.k
    ref = oracle.expert_rows(prob.x, prob.w_gate_up, prob.w_down, token, expert)
    assert_layer_close(y_perm.cpu().numpy()[rows], ref, "routed")
    toks = sample_rows(d.T, min(nsample, d.T), 2)
    ref_sh = oracle.shared_rows(prob.x, prob.ws_gate_up, prob.ws_down, d.S, toks)
    assert_layer_close(y_sh.cpu().numpy()[toks], ref_sh, "shared")


# Token tiles of 256 rows run as CTA pairs, each item two feature tiles (one per CTA).  These shapes
# give odd feature-tile counts (the second CTA of the last item has no tile of its own), a partial
# last down tile (H % 128 == 64) and ragged token tiles, through the standalone and the fused paths.
PAIR_SHAPES = [(1100, 1344, 16, 2, 1, 960), (1500, 1280, 8, 1, 2, 896), (2100, 1280, 64, 6, 2, 896)]


@functools.lru_cache(maxsize=None)
def pair_problem(T, H, E, k, S, I):
    d = synth.MoeDims(T, H, E, k, S, I)
    return DevProblem(synth.moe_problem(d, seed=5, row_ok=oracle.gap_ok(k)))


@pytest.mark.parametrize("T,H,E,k,S,I", PAIR_SHAPES)
def test_grouped_ffn_pairs(T, H, E, k, S, I):
    P = pair_problem(T, H, E, k, S, I)
    d, prob = P.d, P.prob
    r = P.oracle_route()
    dev = lambda a: torch.from_numpy(a).cuda()
    y_perm, y_sh = api.moe_grouped_ffn(P.x, dev(r["perm"]), dev(r["offsets"]), dev(r["counts"]), P.wts, P.sh, P.ws)
    torch.cuda.synchronize()
    rows = sample_rows(d.T * d.k, 128, 11)
    for e in (int(np.argmin(r["counts"])), int(np.argmax(r["counts"]))):
        rows = np.union1d(rows, np.arange(r["offsets"][e], r["offsets"][e + 1])[-40:])
    expert = np.searchsorted(r["offsets"], rows, side="right") - 1
    token = r["perm"][rows] // d.k
    ref = oracle.expert_rows(prob.x, prob.w_gate_up, prob.w_down, token, expert)
    assert_layer_close(y_perm.cpu().numpy()[rows], ref, "routed")
    toks = sample_rows(d.T, 96, 12)
    ref_sh = oracle.shared_rows(prob.x, prob.ws_gate_up, prob.ws_down, d.S, toks)
    assert_layer_close(y_sh.cpu().numpy()[toks], ref_sh, "shared")


@pytest.mark.parametrize("T,H,E,k,S,I", PAIR_SHAPES)
def test_layer_pairs(T, H, E, k, S, I):
    P = pair_problem(T, H, E, k, S, I)
    d, prob = P.d, P.prob
    idx = torch.empty((d.T, d.k), dtype=torch.int32, device="cuda")
    out = api.moe_verify_layer(P.x, P.wts, P.sh, P.ws, topk_idx=idx)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), P.oracle_route()["idx"])
    toks = sample_rows(d.T, 96, 13)
    ref, _, _ = oracle.moe_layer(prob.x, prob.w_router, prob.w_gate_up, prob.w_down, prob.ws_gate_up,
                                 prob.ws_down, d.k, d.S, tokens=toks)
    assert_layer_close(bf16_f64(from_dev_bf16(out))[toks], ref, "pairs")


# Token tiles of 64 and 128 rows: the tile follows the mean rows per expert (T k / E), 24 at
# T = 256 (BN = 64, the router places the rows) and 60 at T = 640 (BN = 128, the fused
# permutation + gather places them).
TILE_SHAPES = [(256, 1280, 64, 6, 2, 896, 10**9), (640, 1280, 64, 6, 2, 896, 200)]


@pytest.mark.parametrize("T,H,E,k,S,I,nsample", TILE_SHAPES)
def test_grouped_ffn_token_tiles(T, H, E, k, S, I, nsample):
    P = pair_problem(T, H, E, k, S, I)
    d, prob = P.d, P.prob
    r = P.oracle_route()
    dev = lambda a: torch.from_numpy(a).cuda()
    y_perm, y_sh = api.moe_grouped_ffn(P.x, dev(r["perm"]), dev(r["offsets"]), dev(r["counts"]), P.wts, P.sh, P.ws)
    torch.cuda.synchronize()
    rows = sample_rows(d.T * d.k, nsample, 21)
    for e in (int(np.argmin(r["counts"])), int(np.argmax(r["counts"]))):
        rows = np.union1d(rows, np.arange(r["offsets"][e], r["offsets"][e + 1]))
    expert = np.searchsorted(r["offsets"], rows, side="right") - 1
    token = r["perm"][rows] // d.k
    ref = oracle.expert_rows(prob.x, prob.w_gate_up, prob.w_down, token, expert)
    assert_layer_close(y_perm.cpu().numpy()[rows], ref, "routed T=%d" % T)
    toks = sample_rows(d.T, min(nsample, d.T), 22)
    ref_sh = oracle.shared_rows(prob.x, prob.ws_gate_up, prob.ws_down, d.S, toks)
    assert_layer_close(y_sh.cpu().numpy()[toks], ref_sh, "shared T=%d" % T)


@pytest.mark.parametrize("T,H,E,k,S,I,nsample", TILE_SHAPES)
def test_layer_token_tiles(T, H, E, k, S, I, nsample):
    P = pair_problem(T, H, E, k, S, I)
    d, prob = P.d, P.prob
    idx = torch.empty((d.T, d.k), dtype=torch.int32, device="cuda")
    out = api.moe_verify_layer(P.x, P.wts, P.sh, P.ws, topk_idx=idx)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), P.oracle_route()["idx"])
    toks = sample_rows(d.T, nsample, 23)
    ref, _, _ = oracle.moe_layer(prob.x, prob.w_router, prob.w_gate_up, prob.w_down, prob.ws_gate_up,
                                 prob.ws_down, d.k, d.S, tokens=toks)
    assert_layer_close(bf16_f64(from_dev_bf16(out))[toks], ref, "T=%d" % T)


def test_weight_prefetch_leaves_the_layer_bit_identical():
    # the L2 hint changes where the weights are read from, never the result
    P = dev_problem("decode")
    a = api.moe_verify_layer(P.x, P.wts, P.sh, P.ws)
    torch.cuda.synchronize()
    for budget in (0, 48 << 20, 1 << 40):
        api.moe_prefetch_weights(P.wts, P.sh, budget)
        b = api.moe_verify_layer(P.x, P.wts, P.sh, P.ws)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), budget
    assert api.get_device_error() == 0


# ----------------------------------------------------------------------------- combine
def test_combine_parity():
    T, k, H = 128, 6, 1280
    rs = np.random.default_rng(0)
    y_perm = rs.standard_normal((T * k, H)).astype(np.float32)
    inv = rs.permutation(T * k).astype(np.int32)
    w = rs.random((T, k)).astype(np.float32)
    ysh = rs.standard_normal((T, H)).astype(np.float32)
    sh = api.shape(T, H, 64, k, 2, 896)
    dev = lambda a: torch.from_numpy(a).cuda()
    out = api.moe_combine(dev(y_perm), dev(inv), dev(w), dev(ysh), sh)
    torch.cuda.synchronize()
    ref = oracle.combine(y_perm, inv, w, ysh, T, k)
    got = bf16_f64(from_dev_bf16(out))
    # fp32 sum then one bf16 rounding: within half a bf16 ulp plus the fp32 sum error
    np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=1e-6)


# ----------------------------------------------------------------------------- whole layer
@pytest.mark.parametrize("name,nsample", [("tiny", 10**9), ("decode", 10**9), ("prefill", 96)])
def test_layer_parity(name, nsample):
    P = dev_problem(name)
    d, prob = P.d, P.prob
    idx = torch.empty((d.T, d.k), dtype=torch.int32, device="cuda")
    counts = torch.empty(d.E, dtype=torch.int32, device="cuda")
    out = api.moe_verify_layer(P.x, P.wts, P.sh, P.ws, topk_idx=idx, counts=counts)
    torch.cuda.synchronize()
    r = P.oracle_route()
    np.testing.assert_array_equal(idx.cpu().numpy(), r["idx"])
    np.testing.assert_array_equal(counts.cpu().numpy(), r["counts"])
    toks = sample_rows(d.T, nsample, 3)
    ref, ref_idx, _ = oracle.moe_layer(prob.x, prob.w_router, prob.w_gate_up, prob.w_down, prob.ws_gate_up,
                                       prob.ws_down, d.k, d.S, tokens=toks)
    np.testing.assert_array_equal(ref_idx, r["idx"][toks])
    assert_layer_close(bf16_f64(from_dev_bf16(out))[toks], ref, name)


@pytest.mark.parametrize("B,K", [(1, 0), (4, 0), (1, 1)])
def test_layer_parity_smallest_batches(B, K):
    # the plain greedy step (K = 0) of the sweep: one to four tokens through the decode layer
    w = synth.sweep_workload(B, K)
    d = w.dims
    prob = synth.moe_problem(w, seed=synth.sweep_seed(B, K), row_ok=oracle.gap_ok(d.k))
    P = DevProblem(prob)
    idx = torch.empty((d.T, d.k), dtype=torch.int32, device="cuda")
    out = api.moe_verify_layer(P.x, P.wts, P.sh, P.ws, topk_idx=idx)
    torch.cuda.synchronize()
    ref, ref_idx, _ = oracle.moe_layer(prob.x, prob.w_router, prob.w_gate_up, prob.w_down, prob.ws_gate_up,
                                       prob.ws_down, d.k, d.S)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    assert_layer_close(bf16_f64(from_dev_bf16(out)), ref, "T=%d" % d.T)


@pytest.mark.parametrize("extra,H,E,k,S,I", [(0, 1280, 64, 6, 2, 896), (1, 1280, 64, 6, 2, 896),
                                              (-115, 512, 256, 8, 1, 128)])
def test_layer_routing_selection_and_counts(extra, H, E, k, S, I):
    # the layer's selection for every token and its per-expert row counts, at one token per SM, one
    # more (both the per-token router) and 37 tokens over 256 experts (the cluster router)
    T = torch.cuda.get_device_properties(0).multi_processor_count + extra
    d = synth.MoeDims(T, H, E, k, S, I)
    prob = synth.moe_problem(d, seed=T + E, hidden="sphere", row_ok=oracle.gap_ok(k))
    P = DevProblem(prob)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    out = api.moe_verify_layer(P.x, P.wts, P.sh, P.ws, topk_idx=idx, counts=counts)
    torch.cuda.synchronize()
    ridx, _ = oracle.route(prob.x, prob.w_router, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_array_equal(counts.cpu().numpy(), np.bincount(ridx.reshape(-1), minlength=E))
    toks = sample_rows(T, 24, 3)
    ref, _, _ = oracle.moe_layer(prob.x, prob.w_router, prob.w_gate_up, prob.w_down, prob.ws_gate_up,
                                 prob.ws_down, k, S, tokens=toks)
    assert_layer_close(bf16_f64(from_dev_bf16(out))[toks], ref, "T=%d E=%d" % (T, E))


def test_layer_workspace_reuse_across_shapes():
    # one workspace for calls of different shapes and paths: every call must leave the counter
    # block at zero for the next one
    probs = [dev_problem("decode"), pair_problem(*PAIR_SHAPES[0]), dev_problem("tiny"), dev_problem("decode")]
    n = max(api.workspace_size(P.sh) for P in probs)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    for P in probs:
        d, prob = P.d, P.prob
        out = api.moe_verify_layer(P.x, P.wts, P.sh, ws)
        torch.cuda.synchronize()
        toks = sample_rows(d.T, 32, 7)
        ref, _, _ = oracle.moe_layer(prob.x, prob.w_router, prob.w_gate_up, prob.w_down, prob.ws_gate_up,
                                     prob.ws_down, d.k, d.S, tokens=toks)
        assert_layer_close(bf16_f64(from_dev_bf16(out))[toks], ref, "reuse T=%d" % d.T)
    assert not ws[:4096].any()


def test_layer_is_deterministic():
    P = dev_problem("decode")
    a = api.moe_verify_layer(P.x, P.wts, P.sh, P.ws)
    b = api.moe_verify_layer(P.x, P.wts, P.sh, P.ws)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_layer_shared_only_and_no_shared():
    # k = 0: the output is the shared experts alone; S = 0: routed experts alone
    base = synth.WORKLOADS["tiny"].dims
    for d in (synth.MoeDims(base.T, base.H, base.E, 0, 1, base.I), synth.MoeDims(base.T, base.H, base.E, 2, 0, base.I)):
        prob = synth.moe_problem(d, seed=4, hidden="normal", row_ok=oracle.gap_ok(max(d.k, 1)))
        x = to_dev(prob.x)
        sh = api.shape(d.T, d.H, d.E, d.k, d.S, d.I)
        wts = api.weights(to_dev(prob.w_router), to_dev(prob.w_gate_up), to_dev(prob.w_down),
                          to_dev(prob.ws_gate_up) if d.S else None, to_dev(prob.ws_down) if d.S else None)
        out = api.moe_verify_layer(x, wts, sh, api.workspace(sh))
        torch.cuda.synchronize()
        ref, _, _ = oracle.moe_layer(prob.x, prob.w_router, prob.w_gate_up, prob.w_down, prob.ws_gate_up,
                                     prob.ws_down, d.k, d.S)
        assert_layer_close(bf16_f64(from_dev_bf16(out)), ref, "k=%d S=%d" % (d.k, d.S))


# ----------------------------------------------------------------------------- acceptance
def run_accept(logits, drafts):
    B, K1, V = logits.shape
    ws = api.spec_verify_workspace(B, K1 - 1, V)
    argmax = torch.empty((B, K1), dtype=torch.int32, device="cuda")
    alen, comm = api.spec_verify_accept(to_dev(logits), torch.from_numpy(drafts).cuda(), ws, argmax=argmax)
    torch.cuda.synchronize()
    return argmax.cpu().numpy(), alen.cpu().numpy(), comm.cpu().numpy()


@pytest.mark.parametrize("B", synth.SWEEP_B)
@pytest.mark.parametrize("K", synth.SWEEP_K)
def test_accept_parity_sweep(B, K):
    w = synth.sweep_workload(B, K)
    logits, planted, drafts = synth.verify_problem(w, seed=synth.sweep_seed(B, K))
    g, alen, comm = run_accept(logits, drafts)
    rg, ralen, rcomm = oracle.accept(logits, drafts)
    np.testing.assert_array_equal(g, rg)
    np.testing.assert_array_equal(g, planted)
    np.testing.assert_array_equal(alen, ralen)
    np.testing.assert_array_equal(comm, rcomm)


@pytest.mark.parametrize("B,K,V", [(4, 3, 1024), (3, 2, 1023), (5, 1, 7), (2, 0, 100), (1, 7, 129_281),
                                   (2, 63, 64), (600, 3, 4096), (4100, 1, 1024),
                                   (4096, 0, 1001), (4096, 2, 2048)])
def test_accept_edge_shapes(B, K, V):
    logits, planted = synth.verify_logits(B, K, V, seed=V + K)
    drafts = synth.draft_tokens(planted, V, [0.9] * K, seed=B)
    if K > 0:
        drafts[0, 0] = V + 5        # outside the vocabulary: a mismatch
        drafts[-1, -1] = -3
    g, alen, comm = run_accept(logits, drafts)
    rg, ralen, rcomm = oracle.accept(logits, drafts)
    np.testing.assert_array_equal(g, rg)
    np.testing.assert_array_equal(alen, ralen)
    np.testing.assert_array_equal(comm, rcomm)


@pytest.mark.parametrize("V", [129_280, 1001])
def test_accept_rows_of_minus_infinity(V):
    # a row that is -inf everywhere (a fully masked vocabulary) has greedy token 0, the first index
    # of its maximum; rows -inf except at one place, and rows with +inf, follow the same rule
    B, K = 6, 3
    logits, planted = synth.verify_logits(B, K, V, seed=21)
    ninf, pinf = np.uint16(0xFF80), np.uint16(0x7F80)
    logits[0, :, :] = ninf                       # every row of sequence 0
    logits[1, 2, :] = ninf
    logits[2, 1, :] = ninf
    logits[2, 1, V - 1] = synth.bf16_bits(np.float32([-3.0]))[0]   # the only finite value: the last index
    logits[3, 0, V // 2] = pinf
    logits[3, 0, V // 3] = pinf                  # two +inf: the lower index wins
    drafts = synth.draft_tokens(planted, V, [0.9] * K, seed=3)
    drafts[0] = 0                                # drafts that equal the -inf rows' greedy token 0
    g, alen, comm = run_accept(logits, drafts)
    rg, ralen, rcomm = oracle.accept(logits, drafts)
    assert rg[0].tolist() == [0] * (K + 1) and rg[2, 1] == V - 1 and rg[3, 0] == V // 3
    np.testing.assert_array_equal(g, rg)
    np.testing.assert_array_equal(alen, ralen)
    np.testing.assert_array_equal(comm, rcomm)


def test_accept_natural_ties():
    # plain N(0,2) bf16 rows: near the top many values collide, so ties at the maximum occur naturally
    rs = np.random.default_rng(5)
    B, K, V = 64, 3, 129_280
    logits = synth.bf16_bits(rs.standard_normal((B, K + 1, V)).astype(np.float32) * 2)
    lg = synth.bf16_value(logits)
    ties = (lg == lg.max(axis=-1, keepdims=True)).sum(axis=-1) > 1
    assert ties.any()
    drafts = np.argmax(lg, axis=-1)[:, :K].astype(np.int32)
    g, alen, comm = run_accept(logits, drafts)
    rg, ralen, rcomm = oracle.accept(logits, drafts)
    np.testing.assert_array_equal(g, rg)
    np.testing.assert_array_equal(alen, ralen)
    assert np.all(alen == K)
    np.testing.assert_array_equal(comm, rcomm)


def test_speculative_loop_on_gpu_equals_greedy():
    V, n_tok, K = 4099, 40, 3
    rs = np.random.default_rng(9)
    table = synth.bf16_bits(rs.integers(-3, 4, size=(61, V)).astype(np.float32))

    def row(a, b):
        return table[(a * 131 + b * 7) % table.shape[0]]

    seq = [1, 2]
    while len(seq) < n_tok + 2:
        seq.append(int(np.argmax(synth.bf16_value(row(seq[-2], seq[-1])))))
    out = [1, 2]
    while len(out) < n_tok + 2:
        ctx = list(out)
        drafts = []
        for _ in range(K):
            tok = int(np.argmax(synth.bf16_value(row(ctx[-2], ctx[-1]))))
            if rs.random() < 0.3:
                tok = int(rs.integers(0, V))
            drafts.append(tok)
            ctx.append(tok)
        inputs = out[-2:] + drafts
        lg = np.stack([row(inputs[j], inputs[j + 1]) for j in range(K + 1)])[None]
        _, alen, comm = run_accept(lg, np.array([drafts], np.int32))
        out.extend(int(c) for c in comm[0, :alen[0] + 1])
    assert out[2:2 + n_tok] == seq[2:2 + n_tok]


def test_accept_workspace_reuse():
    # one workspace across calls of different shapes: each call must leave its counters at zero
    ws = api.spec_verify_workspace(64, 7, 129_280)
    for B, K, V, seed in [(32, 3, 129_280, 1), (64, 7, 129_280, 2), (3, 1, 4096, 3), (32, 3, 129_280, 4)]:
        logits, planted = synth.verify_logits(B, K, V, seed=seed)
        drafts = synth.draft_tokens(planted, V, [0.8] * K, seed=seed)
        argmax = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
        alen, comm = api.spec_verify_accept(to_dev(logits), torch.from_numpy(drafts).cuda(), ws, argmax=argmax)
        torch.cuda.synchronize()
        rg, ralen, rcomm = oracle.accept(logits, drafts)
        np.testing.assert_array_equal(argmax.cpu().numpy(), rg)
        np.testing.assert_array_equal(alen.cpu().numpy(), ralen)
        np.testing.assert_array_equal(comm.cpu().numpy(), rcomm)


def test_accept_is_deterministic():
    w = synth.sweep_workload(64, 3)
    logits, planted, drafts = synth.verify_problem(w, seed=1)
    a = run_accept(logits, drafts)
    b = run_accept(logits, drafts)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


# ----------------------------------------------------------------------------- rmsnorm + residual
def test_rmsnorm_residual_parity():
    rs = np.random.default_rng(2)
    T, H = 256, 1280
    x = synth.bf16_bits(rs.standard_normal((T, H)).astype(np.float32))
    y = synth.bf16_bits(rs.standard_normal((T, H)).astype(np.float32) * 0.3)
    xd, yd = to_dev(x), to_dev(y)
    h = api.rmsnorm_residual(xd, yd, eps=1e-6)
    torch.cuda.synchronize()
    rx, rh = oracle.rmsnorm_residual(x, y, eps=1e-6)
    np.testing.assert_array_equal(bf16_f64(from_dev_bf16(xd)), rx)
    np.testing.assert_allclose(bf16_f64(from_dev_bf16(h)), rh, rtol=2 ** -8, atol=1e-6)


# ----------------------------------------------------------------------------- failure path
def test_bounded_wait_reports_timeout():
    assert api.get_device_error() == 0
    api.selftest_wait_timeout(2_000_000)     # 2 ms on a flag that nothing sets
    torch.cuda.synchronize()
    assert api.get_device_error() == 6
    assert api.get_device_error() == 0
    # the context is still usable afterwards
    P = dev_problem("tiny")
    api.moe_verify_layer(P.x, P.wts, P.sh, P.ws)
    torch.cuda.synchronize()
    assert api.get_device_error() == 0
