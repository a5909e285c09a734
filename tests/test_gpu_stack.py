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


@pytest.mark.parametrize("name", ["k8_stack40", "k16_zipf_stack40"])
def test_stack_teacher_forced_all_layers(M, name):
    """Every one of the 40 layers is fed the oracle's own input x_l (teacher
    forcing from the free-running oracle stack).  Per layer: the GPU RMSNorm
    matches bit for bit, the routing exactly, the block output is within
    tolerance of the oracle's x_{l+1}; and the kernel the stack runs (the
    RMSNorm applied inside the layer kernel, two n-blocks at K = 16) gives
    bit for bit the result of RMSNorm + layer call on the same x_l."""
    w = synthgen.WORKLOADS[name]
    x = synthgen.make_x(w, 77)
    ws = M.workspace(upload(synthgen.make_layer(w, 0, experts=[]), w), w.K)
    xn = torch.empty(w.K, w.H, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((w.K, w.top_k), dtype=torch.int32, device="cuda")
    for l in range(w.layers):
        L = synthgen.make_layer(w, l)
        dl = upload(L, w)
        ref_xn = oracle.rmsnorm(x)
        ref = oracle.moe_layer(oracle.OracleLayer.from_workload(w, L), ref_xn, residual=x)
        xd = to_dev_bf16(x)
        M.moe_rmsnorm(xd, xn)
        y = torch.empty_like(xd)
        M.moe_verify_layer(dl, xn, xd, y, ws, idx_out=idx)
        c = M.layer_array([dl])
        sws = M.stack_workspace(c, w.K)
        xs = xd.clone()
        M.moe_verify_stack(c, xs, sws)
        torch.cuda.synchronize()
        assert M.moe_workspace_error(ws) == 0 and M.moe_workspace_error(sws) == 0
        np.testing.assert_array_equal(bf16_bits(xn), ref_xn, err_msg=f"layer {l} rmsnorm")
        np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"], err_msg=f"layer {l} routing")
        assert_parity(bf16_bits(y), ref["y"], f"{name} layer {l}")
        np.testing.assert_array_equal(bf16_bits(xs), bf16_bits(y), err_msg=f"layer {l}: fused-norm stack kernel")
        x = ref["y"]
        del dl, L


@pytest.mark.parametrize("name,K", [("k8_stack40", 8), ("k8_stack40", 16), ("k16_zipf_stack40", 16)])
def test_native_stack_equals_layer_sequence(M, name, K):
    """moe_verify_stack (the launch configuration the benchmark's stack
    sweep times: the RMSNorm inside the layer kernel, programmatic overlap
    between layers; at K = 16 the two-n-block kernel) gives bit for bit the
    result of rmsnorm + moe_verify_layer per layer; and free-running it stays
    close to the oracle's free-running stack over a few layers."""
    w = synthgen.WORKLOADS[name]
    n = 4
    hl = [synthgen.make_layer(w, l) for l in range(n)]
    dls = [upload(L, w) for L in hl]
    x0 = synthgen.make_x(w, 78, K=K)
    c = M.layer_array(dls)
    ws = M.stack_workspace(c, K)
    xa = to_dev_bf16(x0)
    M.moe_verify_stack(c, xa, ws)
    wsl = M.workspace(dls[0], K)
    xb = to_dev_bf16(x0)
    xn = torch.empty_like(xb)
    for l in range(n):
        M.moe_rmsnorm(xb, xn)
        M.moe_verify_layer(dls[l], xn, xb, xb, wsl)
    torch.cuda.synchronize()
    assert M.moe_workspace_error(ws) == 0
    np.testing.assert_array_equal(bf16_bits(xa), bf16_bits(xb))
    import dataclasses
    ref = oracle.moe_stack(dataclasses.replace(w, K=K), lambda l: hl[l], x0, n_layers=n)
    assert_parity(bf16_bits(xa), ref, f"free-running 4-layer stack, {name} K={K}")
