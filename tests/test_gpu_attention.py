"""GPU parity of the GQA attention block of the full verify step against the
oracle (rel-L2 <= 5e-3, max-abs <= 3e-2 * max|ref| on the block output; the
new keys/values are bf16 GEMV outputs compared the same way)."""
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
    ws = M.attention_workspace(K, H, nq, nkv)
    M.moe_attention_block(d[0], *d[1:5], d[5], d[6], out, ws, nq, nkv, k_new=kn, v_new=vn)
    torch.cuda.synchronize()
    ref = oracle.attention(x, Wq, Wk, Wv, Wo, kc, vc, nq, nkv, 128)
    xn = oracle.rmsnorm(x)
    return bf16_bits(out), ref, bf16_bits(kn), oracle.linear_bf16(xn, Wk), bf16_bits(vn), oracle.linear_bf16(xn, Wv)


@pytest.mark.parametrize("K,H,nq,nkv,C", [(1, 256, 2, 1, 16), (3, 512, 4, 2, 160), (4, 1024, 8, 2, 1024),
                                          (2, 512, 16, 2, 48), (4, 256, 4, 4, 0), (16, 256, 2, 2, 64)])
def test_attention_block_small(M, K, H, nq, nkv, C):
    y, ref, kn, rk, vn, rv = run(M, K, H, nq, nkv, C, seed=K * 7 + C, wsig=0.05)
    assert_parity(kn, rk, "k_new")
    assert_parity(vn, rv, "v_new")
    assert_parity(y, ref, f"attention K={K} C={C}")
    # the attention contribution itself (y - x) must be accurate, not only y
    x = make(K, H, nq, nkv, C, K * 7 + C, 0.05)[0]
    xf = synthgen.bf16_to_f32(x).astype(np.float64)
    dy = synthgen.bf16_to_f32(y) - xf
    dr = synthgen.bf16_to_f32(ref) - xf
    assert np.linalg.norm(dy - dr) / np.linalg.norm(dr) < 3e-2


def test_attention_block_full_step_shape(M):
    # the full verify step's attention: K=4, 32 q heads, 8 kv heads, 16,384 cached positions
    y, ref, kn, rk, vn, rv = run(M, 4, 2048, 32, 8, 16384, seed=4)
    assert_parity(kn, rk, "k_new")
    assert_parity(y, ref, "attention full-step shape")
