"""GPU parity of the verify step around the MoE layers: RMSNorm and lm_head
argmax (bit-exact: both use the fixed FP32 order), and stacks of MoE decoder
blocks teacher-forced on the oracle's own per-layer inputs (routing exact,
outputs within rel-L2 <= 5e-3 and max-abs <= 3e-2 * max|ref|)."""
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


@pytest.mark.parametrize("K,H,scale", [(1, 256, 1.0), (2, 2048, 1.0), (8, 2048, 37.0), (16, 2048, 1e-3),
                                       (5, 768, 1e4), (16, 4096, 1.0)])
def test_rmsnorm_bit_exact(M, K, H, scale):
    x = synthgen.normal_bf16(K, H, 60, 0, K * H, 0.1, scale).reshape(K, H)
    out = torch.empty(K, H, dtype=torch.bfloat16, device="cuda")
    M.moe_rmsnorm(to_dev_bf16(x), out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_bits(out), oracle.rmsnorm(x))


@pytest.mark.parametrize("K,H,V", [(1, 256, 1000), (4, 2048, 151936), (16, 2048, 20011), (3, 512, 77)])
def test_lm_head_argmax_exact(M, K, H, V):
    x = oracle.rmsnorm(synthgen.normal_bf16(V, K, 61, 0, K * H).reshape(K, H))
    W = synthgen.normal_bf16(V, K, 62, 0, V * H, 0.0, 0.02).reshape(V, H)
    tok = torch.empty(K, dtype=torch.int32, device="cuda")
    best = torch.empty(K, dtype=torch.float32, device="cuda")
    ws = M.lm_head_workspace(K)
    Wd = to_dev_bf16(W)
    M.moe_lm_head_argmax(to_dev_bf16(x), Wd, tok, ws, best)
    torch.cuda.synchronize()
    rt, rb = oracle.lm_argmax(x, W)
    np.testing.assert_array_equal(tok.cpu().numpy(), rt)
    np.testing.assert_array_equal(best.cpu().numpy(), rb)
    # again on the same workspace (ticket reset)
    M.moe_lm_head_argmax(to_dev_bf16(x), Wd, tok, ws, best)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tok.cpu().numpy(), rt)


def test_lm_head_exact_ties_lowest_index(M):
    K, H, V = 2, 512, 4099
    x = oracle.rmsnorm(synthgen.normal_bf16(1, 0, 63, 0, K * H).reshape(K, H))
    W = synthgen.normal_bf16(1, 0, 64, 0, V * H, 0.0, 0.02).reshape(V, H)
    rt, _ = oracle.lm_argmax(x, W)
    for r in range(K):  # copies of the winning row, earlier and later
        W[(rt[r] + 1700) % V] = W[rt[r]]
        W[(rt[r] + 2900) % V] = W[rt[r]]
    rt2, _ = oracle.lm_argmax(x, W)
    tok = torch.empty(K, dtype=torch.int32, device="cuda")
    M.moe_lm_head_argmax(to_dev_bf16(x), to_dev_bf16(W), tok, M.lm_head_workspace(K))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tok.cpu().numpy(), rt2)
    for r in range(K):
        assert rt2[r] == min(rt[r], (rt[r] + 1700) % V, (rt[r] + 2900) % V)


def _stack_case(M, name, n_layers):
    w = synthgen.WORKLOADS[name]
    hl = [synthgen.make_layer(w, l) for l in range(n_layers)]
    dls = [upload(L, w) for L in hl]
    x0 = synthgen.make_x(w, 77)
    xf, xs = oracle.moe_stack(w, lambda l: hl[l], x0, n_layers=n_layers, collect=True)
    return w, hl, dls, x0, xf, xs


@pytest.mark.parametrize("name,n_layers", [("k8_stack40", 6), ("k16_zipf_stack40", 6)])
def test_stack_teacher_forced(M, name, n_layers):
    """Each layer is fed the oracle's input x_l (teacher forcing from the
    oracle): GPU rmsnorm must match bit for bit, routing exactly, and the
    block output within tolerance of the oracle's x_{l+1}."""
    w, hl, dls, x0, xf, xs = _stack_case(M, name, n_layers)
    ws = M.workspace(dls[0], w.K)
    xn = torch.empty(w.K, w.H, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((w.K, w.top_k), dtype=torch.int32, device="cuda")
    for l in range(n_layers):
        xd = to_dev_bf16(xs[l])
        M.moe_rmsnorm(xd, xn)
        y = torch.empty_like(xd)
        M.moe_verify_layer(dls[l], xn, xd, y, ws, idx_out=idx)
        torch.cuda.synchronize()
        ref_xn = oracle.rmsnorm(xs[l])
        np.testing.assert_array_equal(bf16_bits(xn), ref_xn, err_msg=f"layer {l} rmsnorm")
        ref = oracle.moe_layer(oracle.OracleLayer.from_workload(w, hl[l]), ref_xn, residual=xs[l])
        np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"], err_msg=f"layer {l} routing")
        nxt = xs[l + 1] if l + 1 < n_layers else xf
        assert_parity(bf16_bits(y), nxt, f"{name} layer {l}")


def test_native_stack_equals_layer_sequence(M):
    """moe_verify_stack (the launch configuration the benchmark's stack
    sweep times) runs the same kernels as rmsnorm + moe_verify_layer per
    layer: bit-identical result; and free-running it stays close to the
    oracle's free-running stack over a few layers."""
    w = synthgen.WORKLOADS["k8_stack40"]
    n = 4
    hl = [synthgen.make_layer(w, l) for l in range(n)]
    dls = [upload(L, w) for L in hl]
    x0 = synthgen.make_x(w, 78)
    c = M.layer_array(dls)
    ws = M.stack_workspace(c, w.K)
    xa = to_dev_bf16(x0)
    M.moe_verify_stack(c, xa, ws)
    wsl = M.workspace(dls[0], w.K)
    xb = to_dev_bf16(x0)
    xn = torch.empty_like(xb)
    for l in range(n):
        M.moe_rmsnorm(xb, xn)
        M.moe_verify_layer(dls[l], xn, xb, xb, wsl)
    torch.cuda.synchronize()
    assert M.moe_workspace_error(ws) == 0
    np.testing.assert_array_equal(bf16_bits(xa), bf16_bits(xb))
    ref = oracle.moe_stack(w, lambda l: hl[l], x0, n_layers=n)
    assert_parity(bf16_bits(xa), ref, "free-running 4-layer stack")
