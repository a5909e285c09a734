"""GPU parity of the MoE verify layer against the CPU oracle, through the C ABI.

Routing indices, weights' order and the grouping table must match the oracle
bit for bit; the layer output y must meet rel-L2 <= 5e-3 and
max-abs <= 3e-2 * max|ref|; router weights are FP32 values and are compared
within FP32 rounding.  Sizes span the verify workloads (K = 1..16, hidden
2048, 256 experts, top-8, intermediate 512) plus small shapes with ragged K,
degenerate routing and extreme activations.
"""
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


def run_layer(M, dl, x, residual=None, ws=None):
    K = x.shape[0]
    ws = M.workspace(dl, K) if ws is None else ws
    xd = to_dev_bf16(x)
    rd = None if residual is None else to_dev_bf16(residual)
    y = torch.empty_like(xd)
    idx = torch.full((K, dl.top_k), -7, dtype=torch.int32, device="cuda")
    w = torch.empty((K, dl.top_k), dtype=torch.float32, device="cuda")
    grp = torch.full((M.moe_group_ints(K, dl.n_experts, dl.top_k),), -7, dtype=torch.int32, device="cuda")
    M.moe_verify_layer(dl, xd, rd, y, ws, idx, w, grp)
    torch.cuda.synchronize()
    assert M.moe_workspace_error(ws) == 0
    return bf16_bits(y), idx.cpu().numpy(), w.cpu().numpy(), grp.cpu().numpy()


def check(w, L, x, res, got, routed_scale=None, what=""):
    ol = oracle.OracleLayer.from_workload(w, L, routed_scale=routed_scale)
    ref = oracle.moe_layer(ol, x, residual=res)
    y, idx, wt, grp = got
    np.testing.assert_array_equal(idx, ref["idx"], err_msg=f"{what} routing indices")
    np.testing.assert_array_equal(grp, ref["group"], err_msg=f"{what} grouping")
    np.testing.assert_allclose(wt, ref["w"], rtol=4e-6, atol=1e-7, err_msg=f"{what} routing weights")
    return assert_parity(y, ref["y"], what)


def _case(w, layer=0, x_inst=0, res_inst=None, **mods):
    L = synthgen.make_layer(w, layer)
    x = synthgen.make_x(w, x_inst)
    res = None if res_inst is None else synthgen.make_x(w, res_inst)
    return L, x, res


@pytest.mark.parametrize("name", ["tiny", "k2_layer"])
def test_workload_layers(M, name):
    w = synthgen.WORKLOADS[name]
    L, x, _ = _case(w)
    dl = upload(L, w)
    check(w, L, x, None, run_layer(M, dl, x), what=name)


@pytest.mark.parametrize("name", ["k8_stack40", "k16_zipf_stack40"])
def test_stack_shaped_layer_full_size(M, name):
    # one layer of the 40-layer stacks at full size, residual included
    w = synthgen.WORKLOADS[name]
    L, x, res = _case(w, layer=3, x_inst=5, res_inst=6)
    dl = upload(L, w)
    check(w, L, x, res, run_layer(M, dl, x, res), what=name)


SMALL = dict(H=512, E=32, top_k=4, I=256, Is=256)


@pytest.mark.parametrize("K", [1, 2, 3, 5, 7, 8, 9, 13, 16])
def test_ragged_rows(M, K):
    w = synthgen.Workload(f"r{K}", K=K, layers=1, seed=100 + K, **SMALL)
    L, x, res = _case(w, res_inst=9)
    dl = upload(L, w)
    check(w, L, x, res, run_layer(M, dl, x, res), what=f"K={K}")


def test_identical_rows_dedup_to_k_experts(M):
    w = synthgen.Workload("same", K=16, layers=1, seed=7, **SMALL)
    L, x, _ = _case(w)
    x = np.tile(x[:1], (16, 1))
    got = run_layer(M, upload(L, w), x)
    assert got[3][0] == w.top_k
    check(w, L, x, None, got, what="identical rows")


def test_top_k_equals_experts(M):
    w = synthgen.Workload("kE", K=16, H=256, E=8, top_k=8, I=128, Is=128, layers=1, seed=8)
    L, x, res = _case(w, res_inst=2)
    got = run_layer(M, upload(L, w), x, res)
    assert got[3][0] == 8
    check(w, L, x, res, got, what="top_k = E")


@pytest.mark.parametrize("K,E,top_k", [(3, 1024, 8), (2, 300, 16), (16, 1024, 32)])
def test_general_topk_path(M, K, E, top_k):
    # more than 256 experts or more than 8 selections take the general top-k
    # (k rounds of a warp arg-max over up to 32 logits per lane); the last
    # case is the largest expert count and selection the library accepts
    w = synthgen.Workload(f"g{E}k{top_k}", K=K, H=256, E=E, top_k=top_k, I=128, Is=128, layers=1,
                          seed=500 + top_k, zipf_s=1.1)
    L, x, res = _case(w, res_inst=4)
    got = run_layer(M, upload(L, w), x, res)
    check(w, L, x, res, got, what=f"E={E}, top-{top_k}")


def test_routed_scale_and_no_shared(M):
    w = synthgen.Workload("rs", K=4, H=1024, E=64, top_k=6, I=128, Is=0, layers=1, seed=9, routed_scale=2.5)
    L, x, res = _case(w, res_inst=3)
    check(w, L, x, res, run_layer(M, upload(L, w), x, res), what="routed scale 2.5, no shared")


def test_tensor_scales_and_zipf_bias(M):
    w = synthgen.Workload("ts", K=6, H=768, E=48, top_k=8, I=256, Is=256, layers=1, seed=10, zipf_s=1.1)
    L, x, _ = _case(w)
    rng = np.random.default_rng(1)
    for p in (L.gate, L.up, L.down, L.sh_gate, L.sh_up, L.sh_down):
        p.tscale[:] = rng.uniform(0.25, 4.0, p.tscale.shape).astype(np.float32)
    check(w, L, x, None, run_layer(M, upload(L, w), x), what="tensor scales + bias")


def test_extreme_activation_range(M):
    # bf16 rows far outside FP16 range: the per-row power-of-two rescaling
    # must keep the tensor-core inputs exact
    w = synthgen.Workload("big", K=3, H=512, E=16, top_k=4, I=128, Is=128, layers=1, seed=11)
    L, x, _ = _case(w)
    xf = synthgen.bf16_to_f32(x)
    xf[0] *= 2.0 ** 40
    xf[1] *= 2.0 ** -40
    x = (xf.view(np.uint32) >> 16).astype(np.uint16)
    got = run_layer(M, upload(L, w), x)
    check(w, L, x, None, got, what="extreme range")
    ref = oracle.moe_layer(oracle.OracleLayer.from_workload(w, L), x)["y"]
    for r in range(w.K):  # each row on its own scale
        assert_parity(got[0][r:r + 1], ref[r:r + 1], f"extreme range row {r}")


def test_deterministic_and_workspace_reuse(M):
    w = synthgen.WORKLOADS["k2_layer"]
    L, x, res = _case(w, res_inst=1)
    dl = upload(L, w)
    ws = M.workspace(dl, w.K)
    a = run_layer(M, dl, x, res, ws=ws)
    b = run_layer(M, dl, x, res, ws=ws)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


@pytest.mark.parametrize("name", ["k2_layer", "k16_zipf_stack40"])
def test_host_activations_match_device_activations(M, name):
    # x, the residual and y in pinned host memory (x staged into the
    # workspace by one CTA -- 64 KB at K = 16, the most it takes -- the
    # residual read and y written across the host link) give the
    # device-buffer call's routing and output bit for bit
    w = synthgen.WORKLOADS[name]
    L, x, res = _case(w, res_inst=1)
    dl = upload(L, w)
    ws = M.workspace(dl, w.K)
    want = run_layer(M, dl, x, res, ws=ws)
    hx = torch.from_numpy(x).view(torch.bfloat16).pin_memory()
    hr = torch.from_numpy(res).view(torch.bfloat16).pin_memory()
    hy = torch.zeros_like(hx).pin_memory()
    idx = torch.full((w.K, dl.top_k), -7, dtype=torch.int32, device="cuda")
    wt = torch.empty((w.K, dl.top_k), dtype=torch.float32, device="cuda")
    grp = torch.full((M.moe_group_ints(w.K, dl.n_experts, dl.top_k),), -7, dtype=torch.int32, device="cuda")
    M.moe_verify_layer(dl, hx, hr, hy, ws, idx, wt, grp)
    torch.cuda.synchronize()
    assert M.moe_workspace_error(ws) == 0
    got = (hy.view(torch.int16).numpy().view(np.uint16), idx.cpu().numpy(), wt.cpu().numpy(), grp.cpu().numpy())
    for u, v in zip(want, got):
        assert np.array_equal(u, v)
    with pytest.raises(ValueError):
        M.moe_verify_layer(dl, torch.from_numpy(x).view(torch.bfloat16), None, hy, ws)  # not pinned
    # the C ABI itself refuses pageable activations before launching anything
    import ctypes
    xp = np.ascontiguousarray(x)
    c = dl.c()
    rc = M.lib.moe_verify_layer(ctypes.byref(c), ctypes.c_void_p(xp.ctypes.data), w.K, None,
                                ctypes.c_void_p(hy.data_ptr()), None, None, None, ctypes.c_void_p(ws.data_ptr()),
                                ws.numel(), None)
    assert rc == M.MOE_ERR_INVALID_ARG


def test_one_workspace_across_shapes(M):
    # The workspace's counters sit at fixed offsets and the words the CTAs
    # exchange carry the call's tag, so one zero-filled workspace serves calls
    # of any K and layer that fit in it: every call matches the oracle even
    # right after calls whose layouts put other data where its words lie.
    cases = []
    for K, E in ((16, 32), (3, 32), (9, 64), (1, 32), (16, 64), (5, 32)):
        w = synthgen.Workload(f"s{K}e{E}", K=K, layers=1, seed=400 + K + E, **dict(SMALL, E=E))
        L, x, res = _case(w, res_inst=3)
        cases.append((w, L, x, res, upload(L, w)))
    n = max(M.moe_verify_layer_workspace_size(dl, w.K) for w, _, _, _, dl in cases)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for w, L, x, res, dl in cases:
            check(w, L, x, res, run_layer(M, dl, x, res, ws=ws), what=f"shared workspace {w.name}, pass {rep}")


def test_router_topk_entry_matches_layer_routing(M):
    w = synthgen.WORKLOADS["k16_zipf_stack40"]
    L, x, _ = _case(w, layer=1, x_inst=2)
    dl = upload(L, w)
    ws = M.workspace(dl, w.K)
    xd = to_dev_bf16(x)
    idx = torch.empty((w.K, w.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((w.K, w.top_k), dtype=torch.float32, device="cuda")
    grp = torch.empty((M.moe_group_ints(w.K, w.E, w.top_k),), dtype=torch.int32, device="cuda")
    M.moe_router_topk(dl, xd, idx, wt, grp, ws)
    torch.cuda.synchronize()
    ol = oracle.OracleLayer.from_workload(w, L)
    ridx, rw = oracle.topk(oracle.router_logits_f32(ol, x), w.top_k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(wt.cpu().numpy(), rw, rtol=4e-6, atol=1e-7)
    np.testing.assert_array_equal(grp.cpu().numpy(), oracle.group(ridx, w.E))


def test_accept_prefix_against_oracle(M):
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(3)
    for K in list(range(0, 10)) + [16, 33, 100, 4096]:
        for trial in range(4):
            t = rng.integers(0, 151936, K).astype(np.int32)
            d = t.copy()
            if K and trial:
                j = int(rng.integers(0, K))
                d[j] += 1
            dd, tt = torch.from_numpy(d).cuda(), torch.from_numpy(t).cuda()
            M.verify_accept_prefix(dd, tt, out)
            torch.cuda.synchronize()
            assert int(out.item()) == oracle.accept_prefix(d, t), (K, trial)


def test_wait_timeout_reports_error_and_recovers(M):
    # a zero wait limit makes every device-side wait give up at once; the
    # kernels must return, report MOE_ERR_DEVICE_TIMEOUT and leave the
    # context usable
    w = synthgen.WORKLOADS["k2_layer"]
    L, x, _ = _case(w)
    dl = upload(L, w)
    ws = M.workspace(dl, w.K)
    xd = to_dev_bf16(x)
    y = torch.empty_like(xd)
    try:
        M.moe_debug_set_wait_limit_ns(0)
        M.moe_verify_layer(dl, xd, None, y, ws)
        torch.cuda.synchronize()
    finally:
        M.moe_debug_set_wait_limit_ns(2_000_000_000)
    assert M.moe_workspace_error(ws) == M.MOE_ERR_DEVICE_TIMEOUT
    ws.zero_()
    check(w, L, x, None, run_layer(M, dl, x, ws=ws), what="after timeout")
