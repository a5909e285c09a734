"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test fixes one oracle function to something independent of it: the
hand-worked format tables in ``tests/golden``, the pages' printed byte
figures, float64 library routines (torch/numpy), closed forms, invariants,
and brute force on tiny inputs.  A dropped term, a wrong sign, a transposed
operand or a swapped nibble in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synthgen
from conftest import read_golden

torch.set_default_dtype(torch.float64)


# ---------------------------------------------------------------- formats

def _e2m1_golden():
    return {int(a): float(b) for a, b in (r.split() for r in read_golden("e2m1_values.txt"))}


def _e4m3_golden():
    return {int(a, 16): float(b) for a, b in (r.split() for r in read_golden("e4m3_values.txt"))}


def test_e2m1_matches_hand_worked_table():
    g = _e2m1_golden()
    assert len(g) == 16
    for c, v in g.items():
        o = oracle.e2m1(c)
        assert o == v and math.copysign(1, o) == math.copysign(1, v), (c, o, v)


def test_e4m3_matches_hand_worked_spots():
    for c, v in _e4m3_golden().items():
        o = oracle.e4m3(c)
        if math.isnan(v):
            assert math.isnan(o), c
        else:
            assert o == v and math.copysign(1, o) == math.copysign(1, v), (hex(c), o, v)


def test_e4m3_structure_all_codes():
    vals = [oracle.e4m3(c) for c in range(256)]
    pos = vals[:0x7F]
    # strictly increasing over the finite positive codes, sign symmetric,
    # NaN exactly at S.1111.111, no infinities
    assert all(b > a for a, b in zip(pos, pos[1:]))
    for c in range(0x7F):
        assert vals[c | 0x80] == -vals[c] or (c == 0 and vals[0x80] == 0.0)
    assert [c for c in range(256) if math.isnan(vals[c])] == [0x7F, 0xFF]
    assert not any(math.isinf(v) for v in vals)
    # within each binade the 8 mantissa steps are evenly spaced; subnormal
    # spacing equals the first normal binade's spacing (2^-9)
    for e in range(16):
        row = pos[8 * e: 8 * e + 8]
        d = np.diff(row)
        assert np.all(d == d[0])
    assert pos[8] - pos[7] == pos[1] - pos[0] == 2.0 ** -9


def test_e4m3_roundtrip_through_generator_encoder():
    # the generator quantises drawn scales to E4M3 with its own encoder;
    # encoding a representable value must give back its code
    for c in range(1, 0x7F):
        v = oracle.e4m3(c)
        out = synthgen.scales(0, 0, 99, 0, 1, lo=v, hi=v)
        assert out[0] == c, (hex(c), v, out[0])


def test_generator_scale_codes_in_declared_range():
    s = synthgen.scales(5, 3, synthgen.T_GATE_S, 0, 200000)
    vals = np.array([oracle.e4m3(int(c)) for c in range(256)])[s]
    assert s.min() == 0x02 and s.max() == 0x18
    assert vals.min() >= 2.0 ** -8 and vals.max() <= 2.0 ** -4


def test_bf16_rounding_matches_library_on_float_inputs():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [1.0, -2.5, 3.0e38, 1e-40, 0.0]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_bf16(float(a)) for a in v], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_hand_worked_midpoints():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even (1.0)
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 lies halfway between 1+2^-7 (odd) and 1+2^-6 (even)
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # slightly above the midpoint rounds up; double rounding through float
    # would lose the 2^-40 and round down
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.round_bf16(-1.0) == 0xBF80
    for b in (0x0001, 0x3F80, 0x7F7F, 0x8001, 0xC2F7):
        assert oracle.round_bf16(oracle.bf16_value(b)) == b


# ---------------------------------------------------------------- NVFP4 decode / byte model

def _decode_with_table(p, e, rows, cols):
    """Independent dequantisation from the golden tables (not the oracle)."""
    t2 = np.array([v for _, v in sorted(_e2m1_golden().items())])
    t8 = np.array([oracle.e4m3(c) for c in range(256)])  # pinned above
    c = p.codes[e].astype(np.int64)
    nib = np.empty((rows, cols), np.int64)
    nib[:, 0::2] = c & 15
    nib[:, 1::2] = c >> 4
    sc = np.repeat(t8[p.scales[e]], 16, axis=1)
    return t2[nib] * sc * float(p.tscale[e])


def test_nvfp4_matrix_layout_against_table_decode():
    w = synthgen.WORKLOADS["tiny"]
    L = synthgen.make_layer(w, 0)
    L.gate.tscale[:] = np.linspace(0.5, 2.0, w.E, dtype=np.float32)
    for e in (0, 7, 15):
        got = oracle.nvfp4_matrix(L.gate, e, w.I, w.H)
        assert np.array_equal(got, _decode_with_table(L.gate, e, w.I, w.H))
        got = oracle.nvfp4_matrix(L.down, e, w.H, w.I)
        assert np.array_equal(got, _decode_with_table(L.down, e, w.H, w.I))


def test_nvfp4_nibble_order_single_element():
    # one nonzero element at an odd column must land in the high nibble
    p = synthgen.Proj(np.zeros((1, 1, 8), np.uint8), np.full((1, 1, 1), 0x38, np.uint8), np.ones(1, np.float32))
    p.codes[0, 0, 2] = 0x70  # column 5 = code 7 (6.0), column 4 = code 0
    m = oracle.nvfp4_matrix(p, 0, 1, 16)
    expect = np.zeros((1, 16))
    expect[0, 5] = 6.0
    assert np.array_equal(m, expect)


def test_byte_model_matches_page_figures():
    figs = {r.split()[0]: (float(r.split()[1]), float(r.split()[2])) for r in read_golden("page_byte_figures.txt")}
    proj = synthgen.nvfp4_bytes(512, 2048) - 4  # the pages' figure has no tensor scale
    assert proj == 589_824
    k2 = 2 * 8 * 3 * proj * 39
    k1 = 1 * 8 * 3 * proj * 39
    tiles = 16 * proj
    assert k2 == 1_104_150_528
    for name, got in (("routed_bytes_k2", k2), ("routed_bytes_k1", k1), ("layer_16_tiles", tiles)):
        v, tol = figs[name]
        assert abs(got - v) / v <= tol, (name, got, v)


# ---------------------------------------------------------------- router

def _bf(x):
    return torch.from_numpy(synthgen.bf16_to_f32(x).astype(np.float64))


@pytest.fixture(scope="module")
def k2layer():
    w = synthgen.WORKLOADS["k2_layer"]
    L = synthgen.make_layer(w, 0)
    return w, L, oracle.OracleLayer.from_workload(w, L)


def test_router_logits_f64_match_library_matmul(k2layer):
    w, L, ol = k2layer
    x = synthgen.make_x(w, 0)
    ref = (_bf(x) @ _bf(L.router_w).T).numpy()
    got = oracle.router_logits_f64(ol, x)
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_router_logits_f32_within_float_error_bound(k2layer):
    w, L, ol = k2layer
    x = synthgen.make_x(w, 1)
    ref = (_bf(x) @ _bf(L.router_w).T).numpy()
    bound = (_bf(x).abs() @ _bf(L.router_w).abs().T).numpy() * (w.H + 5) * 2.0 ** -24
    got = oracle.router_logits_f32(ol, x).astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound)
    # and it is not the double result rounded: the fixed order leaves
    # float rounding visible
    assert np.any(got != ref.astype(np.float32))


def test_router_fixed_order_hand_worked():
    # H=256: lane l holds k = 8l..8l+7.  x = 2^24 at k=0 (lane 0), 1 at k=8
    # (lane 1) and 1 at k=24 (lane 3), w = 1 there.  The pairwise rounds add
    # lanes 1 and 3 first (distance 2): 1 + 1 = 2, then lane 0 + lane 1
    # (distance 1): 2^24 + 2, exact.  A left-to-right sum would lose both
    # ones (2^24 + 1 rounds to 2^24 under ties-to-even).
    H = 256
    one = 0x3F80
    x = np.zeros((1, H), np.uint16)
    W = np.zeros((1, H), np.uint16)
    for k, xv in ((0, 0x4B80), (8, one), (24, one)):
        x[0, k] = xv
        W[0, k] = one
    lay = synthgen.Layer(router_w=W, router_b=None, gate=None, up=None, down=None)
    ol = oracle.OracleLayer(lay, H, 1, 1, 16, 0)
    assert oracle.router_logits_f32(ol, x)[0, 0] == 2.0 ** 24 + 2
    # the same three terms inside one lane (k = 0, 1, 2) lose the ones
    x2 = np.zeros((1, H), np.uint16)
    W2 = np.zeros((1, H), np.uint16)
    for k, xv in ((0, 0x4B80), (1, one), (2, one)):
        x2[0, k] = xv
        W2[0, k] = one
    lay2 = synthgen.Layer(router_w=W2, router_b=None, gate=None, up=None, down=None)
    ol2 = oracle.OracleLayer(lay2, H, 1, 1, 16, 0)
    assert oracle.router_logits_f32(ol2, x2)[0, 0] == 2.0 ** 24


def test_topk_against_library_and_invariants(k2layer):
    w, L, ol = k2layer
    x = synthgen.make_x(w, 2, K=16)
    l32 = oracle.router_logits_f32(ol, x)
    idx, wt = oracle.topk(l32, w.top_k)
    l64 = torch.from_numpy(l32.astype(np.float64))
    ref_vals, ref_idx = torch.topk(l64, w.top_k, dim=1)
    assert np.array_equal(idx, ref_idx.numpy())  # no exact ties in this draw
    p = torch.softmax(l64, dim=1)
    sel = torch.gather(p, 1, ref_idx)
    ref_w = (sel / sel.sum(1, keepdim=True)).numpy()
    assert np.allclose(wt, ref_w, rtol=1e-6, atol=0)
    assert np.allclose(wt.astype(np.float64).sum(1), 1.0, atol=1e-6)
    for r in range(x.shape[0]):
        assert len(set(idx[r])) == w.top_k
        unsel = np.setdiff1d(np.arange(w.E), idx[r])
        assert l32[r, idx[r]].min() >= l32[r, unsel].max()
        assert np.all(np.diff(l32[r, idx[r]]) <= 0)


@pytest.fixture(scope="module")
def zipf_layer():
    # the skewed-routing workload: router bias b[e] = -1.1 ln(e + 1) (a Zipf
    # log-prior over the experts, added to the logits before the softmax)
    w = synthgen.WORKLOADS["k16_zipf_stack40"]
    L = synthgen.make_layer(w, 0, experts=[])
    return w, L, oracle.OracleLayer.from_workload(w, L)


def test_zipf_bias_is_the_log_prior(zipf_layer):
    w, L, _ = zipf_layer
    e = np.arange(w.E, dtype=np.float64)
    assert np.allclose(L.router_b, -1.1 * np.log(e + 1.0), rtol=0, atol=1e-6)
    assert L.router_b[0] == 0.0 and np.all(np.diff(L.router_b) < 0)


def test_router_logits_with_bias_match_library(zipf_layer):
    w, L, ol = zipf_layer
    x = synthgen.make_x(w, 3)
    ref = (_bf(x) @ _bf(L.router_w).T + torch.from_numpy(L.router_b.astype(np.float64))).numpy()
    assert np.allclose(oracle.router_logits_f64(ol, x), ref, rtol=0, atol=1e-12)
    # FP32 fixed order: the dot product's error bound, plus the rounding of
    # the final bias add (half an ulp of the result)
    got = oracle.router_logits_f32(ol, x).astype(np.float64)
    bound = (_bf(x).abs() @ _bf(L.router_w).abs().T).numpy() * (w.H + 5) * 2.0 ** -24 + np.abs(ref) * 2.0 ** -24
    assert np.all(np.abs(got - ref) <= bound)


def test_topk_with_bias_against_library(zipf_layer):
    w, L, ol = zipf_layer
    x = synthgen.make_x(w, 4)
    l32 = oracle.router_logits_f32(ol, x)
    idx, wt = oracle.topk(l32, w.top_k)
    l64 = torch.from_numpy(l32.astype(np.float64))
    _, ref_idx = torch.topk(l64, w.top_k, dim=1)
    assert np.array_equal(idx, ref_idx.numpy())
    p = torch.softmax(l64, dim=1)
    sel = torch.gather(p, 1, ref_idx)
    assert np.allclose(wt, (sel / sel.sum(1, keepdim=True)).numpy(), rtol=1e-6, atol=0)
    # the prior shows: low expert ids are chosen far more often than without it
    unb = oracle.topk(l32 - L.router_b[None, :], w.top_k)[0]
    assert (idx < 16).sum() > 3 * (unb < 16).sum()


def test_router_bias_flips_selection_hand_worked():
    # H = 256, x = e_0 (1.0 at k = 0), router column 0 = (1.0, 0.5, 0, 0):
    # unbiased logits (1.0, 0.5, 0, 0).  Bias (0, 0.75, 0, -1) added before
    # the softmax gives (1.0, 1.25, 0, -1): top-1 is expert 1 (it would be 0
    # without the bias, or with the bias subtracted), and the top-2 weights
    # are the softmax of (1.25, 1.0) over the pair: 1 / (1 + e^-0.25) and
    # 1 / (1 + e^0.25).  A bias added after the softmax, or used for the
    # selection only, would weight expert 1 by e^0.5 / (e^1 + e^0.5) instead.
    H, E = 256, 4
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80
    W = np.zeros((E, H), np.uint16)
    W[0, 0], W[1, 0] = 0x3F80, 0x3F00
    b = np.array([0.0, 0.75, 0.0, -1.0], np.float32)
    lay = synthgen.Layer(router_w=W, router_b=b, gate=None, up=None, down=None)
    ol = oracle.OracleLayer(lay, H, E, 2, 16, 0)
    l32 = oracle.router_logits_f32(ol, x)
    assert l32.tolist() == [[1.0, 1.25, 0.0, -1.0]]
    idx, wt = oracle.topk(l32, 1)
    assert idx.tolist() == [[1]] and wt.tolist() == [[1.0]]
    idx, wt = oracle.topk(l32, 2)
    assert idx.tolist() == [[1, 0]]
    assert abs(wt[0, 0] - 1 / (1 + math.exp(-0.25))) < 1e-7
    assert abs(wt[0, 1] - 1 / (1 + math.exp(0.25))) < 1e-7


def test_topk_exact_ties_go_to_lower_index():
    logits = np.array([[1.0, 3.0, 3.0, 0.5, 3.0, 2.0]], np.float32)
    idx, w = oracle.topk(logits, 3)
    assert idx.tolist() == [[1, 2, 4]]
    assert np.allclose(w, 1 / 3)
    idx, _ = oracle.topk(logits, 6)
    assert idx.tolist() == [[1, 2, 4, 5, 0, 3]]


def test_softmax_closed_form_two_experts():
    # w_0 = 1 / (1 + e^{l1 - l0}) for top-2 of 2
    logits = np.array([[0.75, -0.5]], np.float32)
    _, w = oracle.topk(logits, 2)
    assert abs(w[0, 0] - 1 / (1 + math.exp(-1.25))) < 1e-7


# ---------------------------------------------------------------- sigmoid scoring (Laguna router tail)

def test_sigmoid_f32_against_exact_values():
    # within a few FP32 ulps of the exact logistic function over the range
    # routing logits take, exact at 0, clamped beyond |l| = 80
    xs = np.concatenate([np.linspace(-30, 30, 60001), [-79.9, -50.0, 50.0, 79.9]])
    got = np.array([oracle.sigmoid_f32(v) for v in np.float32(xs)], np.float64)
    ex = 1.0 / (1.0 + np.exp(-np.float32(xs).astype(np.float64)))
    ulp = np.spacing(np.float32(ex)).astype(np.float64)
    assert np.max(np.abs(got - ex) / ulp) <= 4.0
    assert oracle.sigmoid_f32(0.0) == 0.5
    assert oracle.sigmoid_f32(100.0) == oracle.sigmoid_f32(80.0) == 1.0
    assert oracle.sigmoid_f32(-100.0) == oracle.sigmoid_f32(-80.0) > 0.0
    # monotone (non-decreasing) and symmetric to FP32 accuracy
    assert np.all(np.diff(got[:60001]) >= 0)
    sym = np.array([oracle.sigmoid_f32(v) + oracle.sigmoid_f32(-v) for v in np.float32(xs[::97])])
    assert np.max(np.abs(sym - 1.0)) <= 2.0 ** -22


def test_topk_sigmoid_selection_bias_hand_worked():
    # logits (2, 0, -1): scores sigma = (0.8808, 0.5, 0.2689).  Selection bias
    # (0, 0.9, 0) makes the keys (0.8808, 1.4, 0.2689): expert 1 ranks first
    # (expert 0 without the bias or with it subtracted), yet the weights are
    # the unbiased scores renormalised over the selection: top-2 weights
    # 0.5 / 1.3808 and 0.8808 / 1.3808 -- expert 1, selected first, weighs
    # less (weights from the keys would give 1.4 / 2.2808 instead).
    logits = np.array([[2.0, 0.0, -1.0]], np.float32)
    bias = np.array([0.0, 0.9, 0.0], np.float32)
    s = [1 / (1 + math.exp(-2.0)), 0.5]
    idx, w = oracle.topk_sigmoid(logits, bias, 1)
    assert idx.tolist() == [[1]] and w.tolist() == [[1.0]]
    idx, w = oracle.topk_sigmoid(logits, bias, 2)
    assert idx.tolist() == [[1, 0]]
    assert abs(w[0, 0] - s[1] / (s[0] + s[1])) < 1e-6 and abs(w[0, 1] - s[0] / (s[0] + s[1])) < 1e-6
    idx, _ = oracle.topk_sigmoid(logits, None, 2)
    assert idx.tolist() == [[0, 1]]


def test_topk_sigmoid_against_library(zipf_layer):
    w, L, ol = zipf_layer
    x = synthgen.make_x(w, 5)
    nob = oracle.OracleLayer(synthgen.Layer(router_w=L.router_w, router_b=None, gate=None, up=None, down=None),
                             w.H, w.E, w.top_k, w.I, 0)
    l32 = oracle.router_logits_f32(nob, x)
    bias = (np.arange(w.E) % 7 - 3).astype(np.float32) * 0.05
    idx, wt = oracle.topk_sigmoid(l32, bias, w.top_k)
    s64 = torch.sigmoid(torch.from_numpy(l32.astype(np.float64)))
    keys = s64 + torch.from_numpy(bias.astype(np.float64))
    _, ref_idx = torch.topk(keys, w.top_k, dim=1)
    assert np.array_equal(idx, ref_idx.numpy())
    sel = torch.gather(s64, 1, ref_idx)
    assert np.allclose(wt, (sel / sel.sum(1, keepdim=True)).numpy(), rtol=1e-6, atol=0)


# ---------------------------------------------------------------- grouping

def _group_brute(idx, E):
    K, k = idx.shape
    G = min(E, K * k)
    experts = sorted(set(idx.ravel().tolist()))
    pairs, offs = [], []
    for e in experts:
        offs.append(len(pairs))
        pairs += [r * k + s for r in range(K) for s in range(k) if idx[r, s] == e]
    n = len(experts)
    out = [n] + experts + [-1] * (G - n) + offs + [K * k] * (G + 1 - n) + pairs
    return np.array(out, np.int32)


@pytest.mark.parametrize("seed", range(6))
def test_group_brute_force(seed):
    rng = np.random.default_rng(seed)
    K, E, k = [(1, 16, 2), (2, 256, 8), (16, 256, 8), (4, 8, 8), (16, 8, 3), (3, 5, 5)][seed]
    idx = np.stack([rng.permutation(E)[:k] for _ in range(K)]).astype(np.int32)
    g = oracle.group(idx, E)
    assert np.array_equal(g, _group_brute(idx, E))
    n = g[0]
    assert n <= min(E, K * k)
    assert sorted(g[2 + 2 * min(E, K * k):].tolist()) == list(range(K * k))


def test_group_degenerate_cases():
    # K=1 gives n = k; identical rows give n = k; k = E gives n = E
    idx = np.array([[3, 1]], np.int32)
    assert oracle.group(idx, 16)[0] == 2
    idx = np.tile(np.array([[5, 2, 9]], np.int32), (4, 1))
    g = oracle.group(idx, 16)
    assert g[0] == 3 and g[1:4].tolist() == [2, 5, 9]
    idx = np.array([[2, 0, 1], [1, 2, 0]], np.int32)
    assert oracle.group(idx, 3)[0] == 3


# ---------------------------------------------------------------- experts and the layer

def _bf16_round_t(t):
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)


def _dense_expert_torch(L, e, x64, shared=False):
    gp, up, dp = (L.sh_gate, L.sh_up, L.sh_down) if shared else (L.gate, L.up, L.down)
    H = x64.shape[1]
    I = gp.codes.shape[1]
    G = torch.from_numpy(_decode_with_table(gp, e, I, H))
    U = torch.from_numpy(_decode_with_table(up, e, I, H))
    D = torch.from_numpy(_decode_with_table(dp, e, H, I))
    h = _bf16_round_t(torch.nn.functional.silu(x64 @ G.T) * (x64 @ U.T))
    return h @ D.T


def test_expert_equals_dense_swiglu_mlp():
    # E = k = 1 reduces the layer to a dense SwiGLU MLP
    w = synthgen.Workload("e1", K=3, H=256, E=1, top_k=1, I=128, Is=0, layers=1, seed=11)
    L = synthgen.make_layer(w, 0)
    x = synthgen.make_x(w, 0)
    ol = oracle.OracleLayer.from_workload(w, L)
    r = oracle.moe_layer(ol, x)
    ref = _dense_expert_torch(L, 0, _bf(x)).numpy()
    assert np.all(r["idx"] == 0) and np.allclose(r["w"], 1.0)
    assert np.allclose(r["y_f64"], ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())


@pytest.mark.parametrize("with_shared", [False, True])
def test_layer_against_brute_force_dense(with_shared):
    w = synthgen.Workload("bf", K=5, H=256, E=16, top_k=4, I=128, Is=128 if with_shared else 0,
                          layers=1, seed=12, routed_scale=2.5)
    L = synthgen.make_layer(w, 0)
    x = synthgen.make_x(w, 0)
    res = synthgen.make_x(w, 7)
    ol = oracle.OracleLayer.from_workload(w, L)
    r = oracle.moe_layer(ol, x, residual=res)
    x64 = _bf(x)
    # every expert on every row, then the routing mask
    dense = torch.stack([_dense_expert_torch(L, e, x64) for e in range(w.E)])  # [E, K, H]
    l64 = x64 @ _bf(L.router_w).T
    p = torch.softmax(l64, 1)
    mask = torch.zeros(w.K, w.E)
    for rr in range(w.K):
        top = torch.topk(l64[rr], w.top_k).indices
        mask[rr, top] = p[rr, top] / p[rr, top].sum()
        assert sorted(top.tolist()) == sorted(r["idx"][rr].tolist())
    y = 2.5 * torch.einsum("ke,ekh->kh", mask, dense)
    if with_shared:
        y = y + _dense_expert_torch(L, 0, x64, shared=True)
    y = y + _bf(res)
    assert np.allclose(r["y_f64"], y.numpy(), rtol=0, atol=1e-6 * float(y.abs().max()))
    yb = synthgen.bf16_to_f32(r["y"]).astype(np.float64)
    assert np.allclose(yb, y.numpy(), rtol=2.0 ** -8, atol=1e-6)


def test_sigmoid_layer_against_brute_force_dense():
    # the Laguna variant end to end: sigmoid scores, selection-only bias,
    # renormalised scores, routed scale 2.5, shared expert, residual
    w = synthgen.Workload("sg", K=4, H=256, E=16, top_k=4, I=128, Is=128, layers=1, seed=14, routed_scale=2.5)
    L = synthgen.make_layer(w, 0)
    L.router_b = (np.arange(w.E, dtype=np.float32) % 5 - 2) * 0.04
    x = synthgen.make_x(w, 0)
    res = synthgen.make_x(w, 9)
    r = oracle.moe_layer(oracle.OracleLayer.from_workload(w, L, scoring=oracle.SCORE_SIGMOID), x, residual=res)
    x64 = _bf(x)
    dense = torch.stack([_dense_expert_torch(L, e, x64) for e in range(w.E)])
    s64 = torch.sigmoid(x64 @ _bf(L.router_w).T)
    keys = s64 + torch.from_numpy(L.router_b.astype(np.float64))
    mask = torch.zeros(w.K, w.E)
    for rr in range(w.K):
        top = torch.topk(keys[rr], w.top_k).indices
        mask[rr, top] = s64[rr, top] / s64[rr, top].sum()
        assert r["idx"][rr].tolist() == top.tolist()
    y = 2.5 * torch.einsum("ke,ekh->kh", mask, dense) + _dense_expert_torch(L, 0, x64, shared=True) + _bf(res)
    assert np.allclose(r["y_f64"], y.numpy(), rtol=0, atol=1e-6 * float(y.abs().max()))


def test_combine_linearity_routed_scale_and_residual():
    w = synthgen.Workload("lin", K=2, H=256, E=16, top_k=2, I=128, Is=128, layers=1, seed=13)
    L = synthgen.make_layer(w, 0)
    L.sh_gate.codes[:] = 0  # zero shared weights isolate the routed part
    x = synthgen.make_x(w, 0)
    res = synthgen.make_x(w, 3)
    a = oracle.moe_layer(oracle.OracleLayer.from_workload(w, L, routed_scale=1.0), x)["y_f64"]
    b = oracle.moe_layer(oracle.OracleLayer.from_workload(w, L, routed_scale=2.5), x)["y_f64"]
    c = oracle.moe_layer(oracle.OracleLayer.from_workload(w, L, routed_scale=1.0), x, residual=res)["y_f64"]
    assert np.array_equal(b, 2.5 * a)
    assert np.allclose(c - a, synthgen.bf16_to_f32(res), rtol=0, atol=1e-12 * np.abs(c).max())
    assert np.abs(a).max() > 0


# ---------------------------------------------------------------- rmsnorm, attention, lm_head, accept

def test_rmsnorm_against_library():
    x = synthgen.normal_bf16(1, 0, 5, 0, 4 * 2048, 0.3, 2.0).reshape(4, 2048)
    got = synthgen.bf16_to_f32(oracle.rmsnorm(x)).astype(np.float64)
    x64 = _bf(x)
    ref = (x64 * torch.rsqrt(x64.pow(2).mean(1, keepdim=True) + 1e-6)).numpy()
    assert np.allclose(got, ref, rtol=2.0 ** -8, atol=0)
    assert np.allclose(np.sqrt((got ** 2).mean(1)), 1.0, atol=1e-2)


def test_rmsnorm_fp32_steps_hand_worked():
    # H = 256, two nonzero entries: x[10] = 1.9375, x[77] = 3.34375.
    #   ss   = 1.9375^2 + 3.34375^2 = 14.9345703125       (exact in FP32)
    #   mean = ss / 256 = 0.058338165283203125             (exact)
    #   mean + eps -> 0.058339164 (FP32), sqrt -> 0.24153501 (FP32),
    #   inv = 1 / 0.24153501 -> 4.140187 (FP32)
    #   x[77] * inv -> 13.84375 exactly, the midpoint of the bf16 neighbours
    #   13.8125 (0x415D) and 13.875 (0x415E): ties to even give 0x415E;
    #   x[10] * inv -> 8.021612 -> bf16 8.0 (0x4100).
    # A single rounding of 1/sqrt(mean + eps) gives inv = 4.1401863, one
    # FP32 ulp lower, and x[77] -> 0x415D; evaluating in double also gives
    # 0x415D: the oracle's two correctly rounded FP32 steps are what this pins.
    x = np.zeros((1, 256), np.uint16)
    x[0, 10], x[0, 77] = 0x3FF8, 0x4056
    out = oracle.rmsnorm(x)
    expect = np.zeros((1, 256), np.uint16)
    expect[0, 10], expect[0, 77] = 0x4100, 0x415E
    assert np.array_equal(out, expect), (hex(out[0, 10]), hex(out[0, 77]))
    f32 = np.float32
    inv_single = f32(1.0 / np.sqrt(np.float64(f32(14.9345703125 / 256)) + np.float64(f32(1e-6))))
    assert inv_single == f32(4.1401863) and f32(3.34375) * inv_single < f32(13.84375)


def _att_inputs(K, H, nq, nkv, hd, C, seed):
    g = lambda t, n, s: synthgen.normal_bf16(seed, 0, t, 0, n, 0.0, s)
    Wq = g(30, nq * hd * H, 0.05).reshape(nq * hd, H)
    Wk = g(31, nkv * hd * H, 0.05).reshape(nkv * hd, H)
    Wv = g(32, nkv * hd * H, 0.05).reshape(nkv * hd, H)
    Wo = g(33, H * nq * hd, 0.05).reshape(H, nq * hd)
    kc = g(34, nkv * C * hd, 1.0).reshape(nkv, C, hd)
    vc = g(35, nkv * C * hd, 1.0).reshape(nkv, C, hd)
    x = g(36, K * H, 1.0).reshape(K, H)
    return x, Wq, Wk, Wv, Wo, kc, vc


def test_attention_against_library_sdpa():
    K, H, nq, nkv, hd, C = 3, 256, 4, 2, 32, 37
    x, Wq, Wk, Wv, Wo, kc, vc = _att_inputs(K, H, nq, nkv, hd, C, 21)
    got = synthgen.bf16_to_f32(oracle.attention(x, Wq, Wk, Wv, Wo, kc, vc, nq, nkv, hd)).astype(np.float64)
    xn = _bf(oracle.rmsnorm(x))
    q = _bf16_round_t(xn @ _bf(Wq).T).view(K, nq, hd).transpose(0, 1)
    kn = _bf16_round_t(xn @ _bf(Wk).T).view(K, nkv, hd).transpose(0, 1)
    vn = _bf16_round_t(xn @ _bf(Wv).T).view(K, nkv, hd).transpose(0, 1)
    kk = torch.cat([_bf(kc.reshape(-1, hd)).view(nkv, C, hd), kn], 1).repeat_interleave(nq // nkv, 0)
    vv = torch.cat([_bf(vc.reshape(-1, hd)).view(nkv, C, hd), vn], 1).repeat_interleave(nq // nkv, 0)
    mask = torch.ones(K, C + K, dtype=torch.bool)
    for r in range(K):
        mask[r, C + r + 1:] = False
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask)
    o = _bf16_round_t(o.transpose(0, 1).reshape(K, nq * hd))
    ref = _bf(x) + o @ _bf(Wo).T
    assert np.allclose(got, ref.numpy(), rtol=2.0 ** -7, atol=1e-3)


def test_attention_single_key_returns_value():
    # no cache, one row: the only visible key is the row's own -> o = v
    K, H, nq, nkv, hd = 1, 256, 2, 1, 32
    x, Wq, Wk, Wv, Wo, kc, vc = _att_inputs(K, H, nq, nkv, hd, 0, 22)
    kc = np.zeros((nkv, 0, hd), np.uint16)
    vc = np.zeros((nkv, 0, hd), np.uint16)
    got = synthgen.bf16_to_f32(oracle.attention(x, Wq, Wk, Wv, Wo, kc, vc, nq, nkv, hd)).astype(np.float64)
    xn = oracle.rmsnorm(x)
    v = _bf(oracle.linear_bf16(xn, Wv))  # [1, hd]
    o = torch.cat([v, v], 1)  # both q heads share kv head 0
    ref = _bf(x) + o @ _bf(Wo).T
    assert np.allclose(got, ref.numpy(), rtol=2.0 ** -7, atol=1e-3)


def test_attention_uniform_scores_average_values():
    # Wq = 0 -> all scores 0 -> o = mean of the visible values
    K, H, nq, nkv, hd, C = 2, 256, 2, 1, 32, 5
    x, Wq, Wk, Wv, Wo, kc, vc = _att_inputs(K, H, nq, nkv, hd, C, 23)
    Wq = np.zeros_like(Wq)
    got = synthgen.bf16_to_f32(oracle.attention(x, Wq, Wk, Wv, Wo, kc, vc, nq, nkv, hd)).astype(np.float64)
    vn = _bf(oracle.linear_bf16(oracle.rmsnorm(x), Wv))
    vall = torch.cat([_bf(vc.reshape(C, hd)), vn], 0)
    for r in range(K):
        o = _bf16_round_t(vall[: C + r + 1].mean(0))
        ref = _bf(x[r:r + 1]) + torch.cat([o, o])[None] @ _bf(Wo).T
        assert np.allclose(got[r], ref.numpy()[0], rtol=2.0 ** -7, atol=1e-3)


def test_lm_argmax_against_library():
    K, H, V = 4, 512, 3001
    x = synthgen.normal_bf16(2, 0, 50, 0, K * H).reshape(K, H)
    W = synthgen.normal_bf16(2, 0, 51, 0, V * H, 0.0, 0.02).reshape(V, H)
    tok, best = oracle.lm_argmax(x, W)
    l64 = _bf(x) @ _bf(W).T
    top2 = torch.topk(l64, 2, dim=1)
    for r in range(K):
        margin = float(top2.values[r, 0] - top2.values[r, 1])
        if margin > 1e-4:
            assert tok[r] == int(top2.indices[r, 0])
        assert abs(best[r] - float(l64[r, tok[r]])) < 1e-4


def test_lm_argmax_exact_tie_lowest_index():
    K, H, V = 1, 256, 10
    x = synthgen.normal_bf16(3, 0, 52, 0, H).reshape(K, H)
    W = synthgen.normal_bf16(3, 0, 53, 0, V * H, 0.0, 0.02).reshape(V, H)
    l64 = (_bf(x) @ _bf(W).T)[0]
    b = int(torch.argmax(l64))
    W[7] = W[b]
    W[2] = W[b]
    tok, _ = oracle.lm_argmax(x, W)
    assert tok[0] == min(2, b)


def test_accept_prefix_golden_and_brute_force():
    for row in read_golden("accept_cases.txt"):
        d, t, n = row.split("|")
        assert oracle.accept_prefix(np.array(d.split(), np.int32), np.array(t.split(), np.int32)) == int(n)
    for K in range(1, 9):
        for pattern in range(1 << K):
            eq = np.array([(pattern >> i) & 1 for i in range(K)], bool)
            t = np.arange(K, dtype=np.int32) + 100
            d = np.where(eq, t, t + 1).astype(np.int32)
            assert oracle.accept_prefix(d, t) == int(np.cumprod(eq).sum())


# ---------------------------------------------------------------- multi-round verify loop

def _tiny_loop_model(K, R, ctx0=20, layers=2):
    import dataclasses
    w = synthgen.Workload("loop_pin", K=K, H=256, E=8, top_k=2, I=128, Is=128, layers=layers, seed=17,
                          attention=True, n_q_heads=2, n_kv_heads=1, vocab=512)
    w = dataclasses.replace(w, ctx=ctx0 + R * K + 16)
    atts, moes = [], []
    for l in range(layers):
        a = synthgen.make_attention(w, l)
        a["kc"][:, ctx0:] = 0
        a["vc"][:, ctx0:] = 0
        atts.append(a)
        moes.append(synthgen.make_layer(w, l))
    return w, atts, moes, synthgen.make_lm_head(w)


def test_synthetic_drafts_rule():
    t = np.array([0, 5, 511, 7], np.int32)
    coin = np.array([1, 0, 0, 1], np.uint8)
    alt = np.array([3, 0, 510, 100], np.int32)
    d = oracle.synthetic_drafts(t, coin, alt, 512)
    assert d.tolist() == [0, 6, 510, 7]  # (511 + 1 + 510) mod 512 = 510
    # never the target where the coin is off, whatever alt (< vocab - 1)
    alts = np.arange(511, dtype=np.int32)
    assert np.all(oracle.synthetic_drafts(np.full(511, 9, np.int32), np.zeros(511, np.uint8), alts, 512) != 9)


def test_verify_rounds_commit_length():
    # all drafts right: every round commits all K rows; all wrong: one row
    K, R, ctx0 = 2, 3, 20
    w, atts, moes, lm = _tiny_loop_model(K, R, ctx0)
    x = np.stack([synthgen.make_x(w, 500 + t) for t in range(R)])
    alt = np.zeros((R, K), np.int32)
    full = oracle.verify_rounds(w, lambda l: (atts[l], moes[l]), lm, x, np.ones((R, K), np.uint8), alt, ctx0)
    assert full["n"].tolist() == [K] * R and full["len"] == ctx0 + R * K
    none = oracle.verify_rounds(w, lambda l: (atts[l], moes[l]), lm, x, np.zeros((R, K), np.uint8), alt, ctx0)
    assert none["n"].tolist() == [0] * R and none["len"] == ctx0 + R
    # the first round sees the same cache either way
    assert np.array_equal(full["targets"][0], none["targets"][0])


def test_verify_rounds_causal_consistency():
    # Two fully accepted rounds of K rows each must give the rows of round 2
    # exactly the greedy tokens they get as rows K..2K-1 of one round of 2K
    # rows: block-causal attention over an in-place cache is attention over
    # the concatenated sequence.  Pins where and in what order the commit
    # appends (a wrong position, a reversed row order or a missing row
    # changes the second round's tokens).
    K, R, ctx0 = 2, 2, 20
    w, atts, moes, lm = _tiny_loop_model(K, R, ctx0)
    x = np.stack([synthgen.make_x(w, 600 + t) for t in range(R)])
    two = oracle.verify_rounds(w, lambda l: (atts[l], moes[l]), lm, x, np.ones((R, K), np.uint8),
                               np.zeros((R, K), np.int32), ctx0)
    import dataclasses
    w2 = dataclasses.replace(w, K=2 * K)
    one = oracle.verify_rounds(w2, lambda l: (atts[l], moes[l]), lm, x.reshape(1, 2 * K, w.H),
                               np.ones((1, 2 * K), np.uint8), np.zeros((1, 2 * K), np.int32), ctx0)
    assert np.array_equal(two["targets"].reshape(-1), one["targets"].reshape(-1))
    for l in range(w.layers):
        assert np.array_equal(two["kc"][l], one["kc"][l]) and np.array_equal(two["vc"][l], one["vc"][l])


# ---------------------------------------------------------------- Laguna layer schedule: RoPE / YaRN, window, dense MLP

def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(3)
    rd, hd = 64, 128
    f = oracle.rope_freqs(rd, 10000.0)
    q, k = rng.standard_normal(hd), rng.standard_normal(hd)
    assert np.array_equal(oracle.rope_vec(q, rd, f, 0), q)  # position 0 rotates by nothing
    r = oracle.rope_vec(q, rd, f, 12345)
    assert np.array_equal(r[rd:], q[rd:])  # dims past the rotary ones untouched
    pn = lambda v: v[: rd // 2] ** 2 + v[rd // 2: rd] ** 2
    assert np.allclose(pn(r), pn(q), rtol=1e-12)  # each pair keeps its length
    # q_m . k_n depends only on m - n
    d1 = oracle.rope_vec(q, rd, f, 700) @ oracle.rope_vec(k, rd, f, 650)
    d2 = oracle.rope_vec(q, rd, f, 16400) @ oracle.rope_vec(k, rd, f, 16350)
    assert abs(d1 - d2) <= 1e-9 * (abs(d1) + 1.0)
    # rotate-half pairing: pair 0 is (dim 0, dim rd/2), angle = position * 1
    e = np.zeros(hd)
    e[0] = 1.0
    v = oracle.rope_vec(e, rd, f, 1.0)
    assert abs(v[0] - math.cos(1.0)) < 1e-15 and abs(v[rd // 2] - math.sin(1.0)) < 1e-15


def test_yarn_frequencies_closed_form():
    rd, s, L0 = 64, 4.0, 4096
    base = 10000.0 ** (-2.0 * np.arange(rd // 2) / rd)
    assert np.allclose(oracle.rope_freqs(rd, 10000.0, 1.0, L0), base, rtol=1e-15, atol=0)
    f = oracle.rope_freqs(rd, 10000.0, s, L0)
    r = L0 * base / (2 * math.pi)
    g = np.clip((r - 1.0) / 31.0, 0.0, 1.0)
    assert np.allclose(f, (1 - g) * base / s + g * base, rtol=1e-15)
    assert abs(f[0] - base[0]) < 1e-15 and abs(f[-1] - base[-1] / s) < 1e-18  # fast pairs kept, slow ones interpolated
    assert np.all(f <= base * (1 + 1e-15)) and np.all(f >= base / s * (1 - 1e-15))


def _att_case(K, H, nq, nkv, C, seed):
    hd = 128
    g = lambda t, n, sd: synthgen.normal_bf16(seed, 0, t, 0, n, 0.0, sd)
    return (g(36, K * H, 1.0).reshape(K, H), g(30, nq * hd * H, 0.05).reshape(nq * hd, H),
            g(31, nkv * hd * H, 0.05).reshape(nkv * hd, H), g(32, nkv * hd * H, 0.05).reshape(nkv * hd, H),
            g(33, H * nq * hd, 0.05).reshape(H, nq * hd), g(34, nkv * C * hd, 1.0).reshape(nkv, C, hd),
            g(35, nkv * C * hd, 1.0).reshape(nkv, C, hd))


def _torch_rope(x, rd, f, pos):  # independent restatement: rotate-half pairs, double
    x = x.clone()
    ang = torch.tensor(pos, dtype=torch.float64)[:, None] * torch.from_numpy(f)[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    a, b = x[..., : rd // 2].clone(), x[..., rd // 2: rd].clone()
    x[..., : rd // 2] = a * c[:, None, :] - b * s[:, None, :]
    x[..., rd // 2: rd] = b * c[:, None, :] + a * s[:, None, :]
    return x


@pytest.mark.parametrize("window,rd,yarn", [(0, 0, 1.0), (24, 128, 1.0), (40, 64, 4.0)])
def test_attention_ex_against_library_sdpa(window, rd, yarn):
    K, H, nq, nkv, C, hd = 3, 256, 4, 2, 37, 128
    x, Wq, Wk, Wv, Wo, kc, vc = _att_case(K, H, nq, nkv, C, 31)
    got = oracle.attention_ex(x, Wq, Wk, Wv, Wo, kc, vc, nq, nkv, hd, window=window, rotary_dim=rd,
                              yarn_factor=yarn, yarn_orig=16)
    xn = _bf(oracle.rmsnorm(x))
    q = _bf16_round_t(xn @ _bf(Wq).T).view(K, nq, hd)
    kn = _bf16_round_t(xn @ _bf(Wk).T).view(K, nkv, hd)
    vn = _bf16_round_t(xn @ _bf(Wv).T).view(K, nkv, hd)
    temp = 1.0
    if rd:
        base = 10000.0 ** (-2.0 * np.arange(rd // 2) / rd)
        if yarn > 1:
            g = np.clip((16 * base / (2 * math.pi) - 1.0) / 31.0, 0.0, 1.0)
            base = (1 - g) * base / yarn + g * base
            temp = (0.1 * math.log(yarn) + 1.0) ** 2
        pos = [C + r for r in range(K)]
        q = _bf16_round_t(_torch_rope(q, rd, base, pos))
        kn = _bf16_round_t(_torch_rope(kn, rd, base, pos))
    assert np.array_equal(got["k_new"], kn.reshape(K, -1).to(torch.float32).to(torch.bfloat16).view(torch.int16)
                          .numpy().view(np.uint16))
    kk = torch.cat([_bf(kc.reshape(-1, hd)).view(nkv, C, hd), kn.transpose(0, 1)], 1).repeat_interleave(nq // nkv, 0)
    vv = torch.cat([_bf(vc.reshape(-1, hd)).view(nkv, C, hd), vn.transpose(0, 1)], 1).repeat_interleave(nq // nkv, 0)
    mask = torch.zeros(K, C + K, dtype=torch.bool)
    for r in range(K):
        lo = max(0, C + r - window + 1) if window else 0
        mask[r, lo: C + r + 1] = True
    o = torch.nn.functional.scaled_dot_product_attention(q.transpose(0, 1), kk, vv, attn_mask=mask,
                                                         scale=temp / math.sqrt(hd))
    o = _bf16_round_t(o.transpose(0, 1).reshape(K, nq * hd))
    assert np.allclose(synthgen.bf16_to_f32(got["o"]), o.numpy(), rtol=2.0 ** -7, atol=2e-3)
    ref = _bf(x) + o @ _bf(Wo).T
    assert np.allclose(synthgen.bf16_to_f32(got["x"]), ref.numpy(), rtol=2.0 ** -7, atol=2e-3)
    if window == 0 and rd == 0:  # the plain block is the original attention function
        assert np.array_equal(got["x"], oracle.attention(x, Wq, Wk, Wv, Wo, kc, vc, nq, nkv, hd))


def test_dense_mlp_against_library():
    K, H, I = 3, 256, 512
    g = lambda t, n, sd: synthgen.normal_bf16(32, 0, t, 0, n, 0.0, sd)
    xn = oracle.rmsnorm(g(1, K * H, 1.0).reshape(K, H))
    res = g(2, K * H, 1.0).reshape(K, H)
    Wg, Wu, Wd = g(3, I * H, 0.05).reshape(I, H), g(4, I * H, 0.05).reshape(I, H), g(5, H * I, 0.05).reshape(H, I)
    y = oracle.dense_mlp(xn, res, Wg, Wu, Wd)
    x64 = _bf(xn)
    h = _bf16_round_t(torch.nn.functional.silu(x64 @ _bf(Wg).T) * (x64 @ _bf(Wu).T))
    ref = _bf(res) + h @ _bf(Wd).T
    assert np.allclose(synthgen.bf16_to_f32(y), ref.numpy(), rtol=2.0 ** -8, atol=1e-6)
