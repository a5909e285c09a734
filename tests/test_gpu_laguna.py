"""GPU parity of the Laguna router/combine variant (PR #844, "4. What I
ported", router-tail and combine rows; "5. Numerical safety"): sigmoid scores,
a bias that steers the selection only, the selected scores renormalised, the
routed sum scaled by 2.5, the shared expert and the residual added.

Selection (indices, grouping) must match the oracle bit for bit -- both sides
evaluate the same FP32 sigmoid sequence -- the weights within FP32 rounding,
y within rel-L2 <= 5e-3 and max-abs <= 3e-2 * max|ref|.

The combine is also checked bit for bit against its documented FP32
expression, evaluated here from the kernel's own down partials (read back
from the workspace) and routing weights: each product and sum rounded on its
own, no fused multiply-add -- the contraction question the pages raise about
routed * 2.5 + shared (an FMA skips the product's rounding)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthgen
from helpers import assert_parity, bf16_bits, to_dev_bf16, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M(cuda_ok):
    import moe_nvfp4_block_gb300 as M
    return M


def _bias(E, seed):
    # a selection bias of the size a trained correction bias has next to
    # scores in (0, 1): 0.05 N(0, 1) per expert
    return (synthgen.bf16_to_f32(synthgen.normal_bf16(seed, 0, synthgen.T_ROUTER_B, 0, E)) * 0.05).astype(np.float32)


def _run(M, dl, x, res, ws):
    K = x.shape[0]
    xd, rd = to_dev_bf16(x), (None if res is None else to_dev_bf16(res))
    y = torch.empty_like(xd)
    idx = torch.empty((K, dl.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((K, dl.top_k), dtype=torch.float32, device="cuda")
    grp = torch.empty(M.moe_group_ints(K, dl.n_experts, dl.top_k), dtype=torch.int32, device="cuda")
    M.moe_verify_layer(dl, xd, rd, y, ws, idx, w, grp)
    torch.cuda.synchronize()
    assert M.moe_workspace_error(ws) == 0
    return bf16_bits(y), idx.cpu().numpy(), w.cpu().numpy(), grp.cpu().numpy()


def _bf16_rne(v32):
    u = v32.view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF).astype(np.uint16)


def _combine_bits(M, dl, ws, K, w, res):
    """y recomputed from the workspace's down partials with the documented
    FP32 expression; also the variant with routed_scale * acc + shared
    contracted into one rounding (for the report)."""
    off = M.lib.moe_debug_partials_offset(ctypes.byref(dl.c()), K)
    k, H = dl.top_k, dl.hidden
    words = ws[off: off + 8 * K * (k + 1) * H].view(torch.int64).cpu().numpy().astype(np.uint64)
    part = (words & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32).reshape(K, k + 1, H)
    f32 = np.float32
    acc = np.zeros((K, H), f32)
    for s in range(k):
        acc = (acc + (w[:, s:s + 1].astype(f32) * part[:, s, :]).astype(f32)).astype(f32)
    scale = f32(dl.routed_scale)
    v = (scale * acc).astype(f32)
    if dl.shared_inter:
        v = (v + part[:, k, :]).astype(f32)
    fused = (scale.astype(np.float64) * acc.astype(np.float64) +
             (part[:, k, :].astype(np.float64) if dl.shared_inter else 0.0)).astype(f32)
    if res is not None:
        r = synthgen.bf16_to_f32(res)
        v = (v + r).astype(f32)
        fused = (fused + r).astype(f32)
    return _bf16_rne(v), int(np.count_nonzero(v.view(np.uint32) != fused.view(np.uint32)))


@pytest.mark.parametrize("K", [1, 2, 8, 16])
def test_sigmoid_scoring_layer(M, K):
    w = synthgen.WORKLOADS["k2_layer"]
    L = synthgen.make_layer(w, 5)
    L.router_b = _bias(w.E, 31)
    dl = upload(L, w, routed_scale=2.5, scoring=M.MOE_SCORE_SIGMOID)
    x = synthgen.make_x(w, 60 + K, K=K)
    res = synthgen.make_x(w, 70 + K, K=K)
    ws = M.workspace(dl, K)
    y, idx, wt, grp = _run(M, dl, x, res, ws)
    ol = oracle.OracleLayer.from_workload(w, L, routed_scale=2.5, scoring=oracle.SCORE_SIGMOID)
    ref = oracle.moe_layer(ol, x, residual=res)
    np.testing.assert_array_equal(idx, ref["idx"], err_msg="routing indices")
    np.testing.assert_array_equal(grp, ref["group"], err_msg="grouping")
    np.testing.assert_allclose(wt, ref["w"], rtol=4e-6, atol=1e-7, err_msg="routing weights")
    assert_parity(y, ref["y"], f"sigmoid-scored layer K={K}")
    # the bias steers the selection: without it the experts differ
    nob = oracle.topk_sigmoid(oracle.router_logits_f32(
        oracle.OracleLayer(synthgen.Layer(router_w=L.router_w, router_b=None, gate=None, up=None, down=None),
                           w.H, w.E, w.top_k, w.I, 0), x), None, w.top_k)[0]
    assert not np.array_equal(np.sort(nob, 1), np.sort(idx, 1))
    # the combine, bit for bit from the kernel's own partials and weights
    yc, n_fused_diff = _combine_bits(M, dl, ws, K, wt, res)
    np.testing.assert_array_equal(y, yc, err_msg="combine expression")


def test_sigmoid_scoring_general_topk(M):
    # E > 256 and k > 8 take the general top-k path
    w = synthgen.Workload("sg_big", K=4, H=512, E=384, top_k=12, I=128, Is=128, layers=1, seed=15)
    L = synthgen.make_layer(w, 0)
    L.router_b = _bias(w.E, 32)
    dl = upload(L, w, routed_scale=2.5, scoring=M.MOE_SCORE_SIGMOID)
    x = synthgen.make_x(w, 1)
    ws = M.workspace(dl, w.K)
    y, idx, wt, grp = _run(M, dl, x, None, ws)
    ref = oracle.moe_layer(oracle.OracleLayer.from_workload(w, L, routed_scale=2.5, scoring=oracle.SCORE_SIGMOID), x)
    np.testing.assert_array_equal(idx, ref["idx"])
    np.testing.assert_array_equal(grp, ref["group"])
    np.testing.assert_allclose(wt, ref["w"], rtol=4e-6, atol=1e-7)
    assert_parity(y, ref["y"], "sigmoid-scored layer, general top-k")


def test_sigmoid_router_topk_standalone(M):
    w = synthgen.WORKLOADS["k2_layer"]
    L = synthgen.make_layer(w, 6, experts=[])
    L.router_b = _bias(w.E, 33)
    dl = upload(L, w, scoring=M.MOE_SCORE_SIGMOID)
    K = 8
    x = synthgen.make_x(w, 3, K=K)
    idx = torch.empty((K, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((K, w.top_k), dtype=torch.float32, device="cuda")
    grp = torch.empty(M.moe_group_ints(K, w.E, w.top_k), dtype=torch.int32, device="cuda")
    M.moe_router_topk(dl, to_dev_bf16(x), idx, wt, grp, M.workspace(dl, K))
    torch.cuda.synchronize()
    nob = oracle.OracleLayer(synthgen.Layer(router_w=L.router_w, router_b=None, gate=None, up=None, down=None),
                             w.H, w.E, w.top_k, w.I, 0)
    ri, rw = oracle.topk_sigmoid(oracle.router_logits_f32(nob, x), L.router_b, w.top_k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ri)
    np.testing.assert_allclose(wt.cpu().numpy(), rw, rtol=4e-6, atol=1e-7)
    np.testing.assert_array_equal(grp.cpu().numpy(), oracle.group(ri, w.E))


@pytest.mark.parametrize("scoring", [0, 1])
def test_combine_expression_bit_exact(M, scoring):
    """Both scorings share the combine: bit for bit the documented FP32
    expression over the kernel's own partials, at the full k2_layer shape
    with the Laguna routed scale."""
    w = synthgen.WORKLOADS["k2_layer"]
    L = synthgen.make_layer(w, 7)
    dl = upload(L, w, routed_scale=2.5, scoring=scoring)
    x = synthgen.make_x(w, 8)
    res = synthgen.make_x(w, 9)
    ws = M.workspace(dl, w.K)
    y, idx, wt, grp = _run(M, dl, x, res, ws)
    yc, n_fused_diff = _combine_bits(M, dl, ws, w.K, wt, res)
    np.testing.assert_array_equal(y, yc)
    # (the contracted form differs from the rounded one on some outputs
    # before the final bf16 rounding; reported, not asserted)
    print(f"scoring {scoring}: {n_fused_diff} of {y.size} FP32 values differ under contraction")
