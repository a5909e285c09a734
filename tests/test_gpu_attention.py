"""GPU parity of the GQA attention block of the full verify step against the
oracle (rel-L2 <= 5e-3, max-abs <= 3e-2 * max|ref|).  Checked on the
attention output o itself (before the o-projection), on the new keys and
values, and on the block output x + o.Wo^T.  The block output alone would not
do: at the full-step shape the attention term is only ~1.5% of |x + attn|,
so a large error in o would still leave the block output within tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synthgen
from helpers import assert_parity, bf16_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M(cuda_ok):
    import moe_nvfp4_block_gb300 as M
    return M


def make(K, H, nq, nkv, C, seed, wsig=0.02):
    hd = 128
    g = lambda t, n, s: synthgen.normal_bf16(seed, 0, t, 0, n, 0.0, s)
    x = g(synthgen.T_X, K * H, 1.0).reshape(K, H)
    Wq = g(synthgen.T_ATT_Q, nq * hd * H, wsig).reshape(nq * hd, H)
    Wk = g(synthgen.T_ATT_K, nkv * hd * H, wsig).reshape(nkv * hd, H)
    Wv = g(synthgen.T_ATT_V, nkv * hd * H, wsig).reshape(nkv * hd, H)
    Wo = g(synthgen.T_ATT_O, H * nq * hd, wsig).reshape(H, nq * hd)
    kc = g(synthgen.T_KCACHE, nkv * C * hd, 1.0).reshape(nkv, C, hd)
    vc = g(synthgen.T_VCACHE, nkv * C * hd, 1.0).reshape(nkv, C, hd)
    return x, Wq, Wk, Wv, Wo, kc, vc


def run(M, K, H, nq, nkv, C, seed, wsig=0.02):
    x, Wq, Wk, Wv, Wo, kc, vc = make(K, H, nq, nkv, C, seed, wsig)
    d = [to_dev_bf16(a) for a in (x, Wq, Wk, Wv, Wo, kc, vc)]
    out = torch.empty_like(d[0])
    kn = torch.empty(K, nkv * 128, dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    o = torch.empty(K, nq * 128, dtype=torch.bfloat16, device="cuda")
    ws = M.attention_workspace(K, H, nq, nkv)
    M.moe_attention_block(d[0], *d[1:5], d[5], d[6], out, ws, nq, nkv, k_new=kn, v_new=vn, o_out=o)
    torch.cuda.synchronize()
    ref, ref_o = oracle.attention(x, Wq, Wk, Wv, Wo, kc, vc, nq, nkv, 128, with_o=True)
    xn = oracle.rmsnorm(x)
    return dict(y=bf16_bits(out), ref=ref, o=bf16_bits(o), ref_o=ref_o, kn=bf16_bits(kn),
                rk=oracle.linear_bf16(xn, Wk), vn=bf16_bits(vn), rv=oracle.linear_bf16(xn, Wv), x=x)


def _check_all(r, what, term_tol=None):
    assert_parity(r["kn"], r["rk"], f"{what}: k_new")
    assert_parity(r["vn"], r["rv"], f"{what}: v_new")
    assert_parity(r["o"], r["ref_o"], f"{what}: attention output o")
    assert_parity(r["y"], r["ref"], f"{what}: block output")
    if term_tol is None:
        return
    # the o-projection's contribution y - x (where it is large enough next to
    # x that the final bf16 rounding of y does not swamp it)
    xf = synthgen.bf16_to_f32(r["x"]).astype(np.float64)
    dy = synthgen.bf16_to_f32(r["y"]) - xf
    dr = synthgen.bf16_to_f32(r["ref"]) - xf
    rel = np.linalg.norm(dy - dr) / np.linalg.norm(dr)
    assert rel <= term_tol, f"{what}: attention term rel-L2 {rel:.3e}"


@pytest.mark.parametrize("K,H,nq,nkv,C", [(1, 256, 2, 1, 16), (3, 512, 4, 2, 160), (4, 1024, 8, 2, 1024),
                                          (2, 512, 16, 2, 48), (4, 256, 4, 4, 0), (16, 256, 2, 2, 64)])
def test_attention_block_small(M, K, H, nq, nkv, C):
    _check_all(run(M, K, H, nq, nkv, C, seed=K * 7 + C, wsig=0.05), f"attention K={K} C={C}", term_tol=3e-2)


@pytest.mark.parametrize("K,nq,nkv,C", [(16, 32, 8, 304), (8, 16, 4, 1008), (1, 48, 8, 144), (2, 64, 8, 1024),
                                        (2, 32, 8, 0)])
def test_attention_block_streamed_shapes(M, K, nq, nkv, C):
    # H = 2048: the streamed projection (x fragments of rows 8..15 when K > 8;
    # o-projections 2048 .. 8192 wide), several 16-row query tiles per KV head,
    # caches ending inside a 128-position chunk, and an empty cache
    _check_all(run(M, K, 2048, nq, nkv, C, seed=K * 11 + C, wsig=0.02), f"attention K={K} nq={nq} C={C}")


def test_attention_block_full_step_shape(M):
    # the full verify step's attention: K=4, 32 q heads, 8 kv heads, 16,384 cached positions
    _check_all(run(M, 4, 2048, 32, 8, 16384, seed=4), "attention full-step shape")


def test_streamed_kernels_wait_timeout_reports_error_and_recovers(M):
    # a zero wait limit makes every ring wait of the streamed projection,
    # split attention and lm_head give up at once: the calls return, report
    # MOE_ERR_DEVICE_TIMEOUT, drain their own copies, and the next calls (at
    # the default limit) are correct
    K, H, nq, nkv, C, V = 4, 2048, 32, 8, 1024, 4096
    x, Wq, Wk, Wv, Wo, kc, vc = make(K, H, nq, nkv, C, seed=77)
    d = [to_dev_bf16(a) for a in (x, Wq, Wk, Wv, Wo, kc, vc)]
    ws = M.attention_workspace(K, H, nq, nkv)
    lm = synthgen.normal_bf16(77, 0, synthgen.T_LM_HEAD, 0, V * H, 0.0, 0.02).reshape(V, H)
    xn = oracle.rmsnorm(x)
    lmd, xnd = to_dev_bf16(lm), to_dev_bf16(xn)
    tok = torch.empty(K, dtype=torch.int32, device="cuda")
    lws = M.lm_head_workspace(K)
    out = torch.empty_like(d[0])
    try:
        M.moe_debug_set_wait_limit_ns(0)
        M.moe_attention_block(d[0], *d[1:5], d[5], d[6], out, ws, nq, nkv)
        M.moe_lm_head_argmax(xnd, lmd, tok, lws)
        torch.cuda.synchronize()
    finally:
        M.moe_debug_set_wait_limit_ns(2_000_000_000)
    assert M.moe_workspace_error(ws) == M.MOE_ERR_DEVICE_TIMEOUT
    assert M.moe_workspace_error(lws) == M.MOE_ERR_DEVICE_TIMEOUT
    M.moe_attention_block(d[0], *d[1:5], d[5], d[6], out, ws, nq, nkv)
    M.moe_lm_head_argmax(xnd, lmd, tok, lws)
    torch.cuda.synchronize()
    assert M.moe_workspace_error(ws) == 0 and M.moe_workspace_error(lws) == 0
    ref = oracle.attention(x, Wq, Wk, Wv, Wo, kc, vc, nq, nkv, 128)
    assert_parity(bf16_bits(out), ref, "attention block after the timeout")
    ref_tok, _ = oracle.lm_argmax(xn, lm)
    np.testing.assert_array_equal(tok.cpu().numpy(), ref_tok)
