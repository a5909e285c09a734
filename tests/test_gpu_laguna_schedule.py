"""GPU parity of the Laguna layer schedule (README, "Why this challenge
exists"): sliding-window attention (512 positions, 64 q heads, RoPE theta
10000), full attention (48 q heads, YaRN rotary on half the head dims), the
dense SwiGLU MLP of layer 0, and a verify step over a short stack in that
schedule.  Against the oracle: the attention output o, the rotated new keys
and the block outputs within rel-L2 <= 5e-3 and max-abs <= 3e-2 * max|ref|;
the appended cache rows; the greedy tokens exactly (teacher-forced).  The
free-running step must equal the same blocks chained one call at a time on
the GPU bit for bit."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synthgen
from helpers import assert_parity, bf16_bits, to_dev_bf16, upload

pytestmark = pytest.mark.gpu


def _att(K, H, nq, nkv, C, seed):
    hd = 128
    g = lambda t, n, sd: synthgen.normal_bf16(seed, 0, t, 0, n, 0.0, sd)
    return dict(x=g(synthgen.T_X, K * H, 1.0).reshape(K, H), Wq=g(synthgen.T_ATT_Q, nq * hd * H, 0.02).reshape(nq * hd, H),
                Wk=g(synthgen.T_ATT_K, nkv * hd * H, 0.02).reshape(nkv * hd, H),
                Wv=g(synthgen.T_ATT_V, nkv * hd * H, 0.02).reshape(nkv * hd, H),
                Wo=g(synthgen.T_ATT_O, H * nq * hd, 0.02).reshape(H, nq * hd),
                kc=g(synthgen.T_KCACHE, nkv * C * hd, 1.0).reshape(nkv, C, hd),
                vc=g(synthgen.T_VCACHE, nkv * C * hd, 1.0).reshape(nkv, C, hd))


@pytest.mark.parametrize("layer", [0, 3])  # a sliding-window layer and a full-attention (YaRN) layer
@pytest.mark.parametrize("K,C", [(4, 1024), (2, 528)])
def test_laguna_attention(cuda_ok, layer, K, C):
    import moe_nvfp4_block_gb300 as M
    cfg = synthgen.laguna_layer_kind(layer)
    H, nq, nkv = 2048, cfg["n_q_heads"], 8
    a = _att(K, H, nq, nkv, C, 40 + layer + K)
    ref = oracle.attention_ex(a["x"], a["Wq"], a["Wk"], a["Wv"], a["Wo"], a["kc"], a["vc"], nq, nkv, 128,
                              window=cfg["window"], rotary_dim=cfg["rotary_dim"], theta=cfg["rope_theta"],
                              yarn_factor=cfg["yarn_factor"], yarn_orig=cfg["yarn_orig"])
    d = {k: to_dev_bf16(v) for k, v in a.items()}
    out = torch.empty_like(d["x"])
    kn = torch.empty(K, nkv * 128, dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    o = torch.empty(K, nq * 128, dtype=torch.bfloat16, device="cuda")
    ws = M.attention_workspace(K, H, nq, nkv)
    pos = M.attn_pos(cfg["window"], cfg["rotary_dim"], cfg["rope_theta"], cfg["yarn_factor"], cfg["yarn_orig"])
    M.moe_attention_block(d["x"], d["Wq"], d["Wk"], d["Wv"], d["Wo"], d["kc"], d["vc"], out, ws, nq, nkv,
                          k_new=kn, v_new=vn, o_out=o, pos=pos)
    torch.cuda.synchronize()
    assert M.moe_workspace_error(ws) == 0
    assert_parity(bf16_bits(kn), ref["k_new"], "rotated new keys")
    assert_parity(bf16_bits(vn), ref["v_new"], "new values")
    assert_parity(bf16_bits(o), ref["o"], "attention output o")
    assert_parity(bf16_bits(out), ref["x"], "block output")


@pytest.mark.parametrize("K,nq,rd,window,C", [(3, 16, 8, 0, 256), (16, 32, 128, 0, 272), (16, 32, 32, 96, 400),
                                               (8, 64, 128, 512, 1040)])
def test_rotary_paths(cuda_ok, K, nq, rd, window, C):
    # the rotary embedding in the projection's epilogue (rotary widths that
    # are multiples of 16; K = 16: x fragments of two 8-row halves) and in a
    # kernel of its own (width 8), against the oracle
    import moe_nvfp4_block_gb300 as M
    H, nkv = 2048, 8
    a = _att(K, H, nq, nkv, C, 70 + K + rd)
    ref = oracle.attention_ex(a["x"], a["Wq"], a["Wk"], a["Wv"], a["Wo"], a["kc"], a["vc"], nq, nkv, 128,
                              window=window, rotary_dim=rd, theta=10000.0)
    d = {k: to_dev_bf16(v) for k, v in a.items()}
    out = torch.empty_like(d["x"])
    kn = torch.empty(K, nkv * 128, dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    o = torch.empty(K, nq * 128, dtype=torch.bfloat16, device="cuda")
    ws = M.attention_workspace(K, H, nq, nkv)
    M.moe_attention_block(d["x"], d["Wq"], d["Wk"], d["Wv"], d["Wo"], d["kc"], d["vc"], out, ws, nq, nkv,
                          k_new=kn, v_new=vn, o_out=o, pos=M.attn_pos(window, rd, 10000.0))
    torch.cuda.synchronize()
    assert M.moe_workspace_error(ws) == 0
    assert_parity(bf16_bits(kn), ref["k_new"], f"rotated new keys (rd {rd}, K {K})")
    assert_parity(bf16_bits(o), ref["o"], f"attention output o (rd {rd}, K {K})")
    assert_parity(bf16_bits(out), ref["x"], f"block output (rd {rd}, K {K})")


def test_laguna_attention_inplace_append(cuda_ok):
    # the sliding layer with a device length: the rotated keys and the values
    # go into the caches at positions len .. len + K - 1
    import moe_nvfp4_block_gb300 as M
    cfg = synthgen.laguna_layer_kind(1)
    K, H, nq, nkv, C0, cap = 2, 2048, cfg["n_q_heads"], 8, 600, 640
    a = _att(K, H, nq, nkv, cap, 51)
    a["kc"][:, C0:] = 0
    a["vc"][:, C0:] = 0
    ref = oracle.attention_ex(a["x"], a["Wq"], a["Wk"], a["Wv"], a["Wo"], a["kc"][:, :C0], a["vc"][:, :C0], nq, nkv,
                              128, window=cfg["window"], rotary_dim=cfg["rotary_dim"], theta=cfg["rope_theta"])
    d = {k: to_dev_bf16(v) for k, v in a.items()}
    out = torch.empty_like(d["x"])
    kv_len = torch.tensor([C0], dtype=torch.int32, device="cuda")
    ws = M.attention_workspace(K, H, nq, nkv)
    pos = M.attn_pos(cfg["window"], cfg["rotary_dim"], cfg["rope_theta"])
    M.moe_attention_block(d["x"], d["Wq"], d["Wk"], d["Wv"], d["Wo"], d["kc"], d["vc"], out, ws, nq, nkv,
                          kv_len=kv_len, pos=pos)
    torch.cuda.synchronize()
    assert M.moe_workspace_error(ws) == 0
    assert_parity(bf16_bits(out), ref["x"], "block output")
    kc = bf16_bits(d["kc"])
    np.testing.assert_array_equal(kc[:, :C0], a["kc"][:, :C0])
    assert_parity(kc[:, C0:C0 + K].transpose(1, 0, 2).reshape(K, -1), ref["k_new"], "appended rotated keys")
    assert_parity(bf16_bits(d["vc"])[:, C0:C0 + K].transpose(1, 0, 2).reshape(K, -1), ref["v_new"], "appended values")
    assert not np.any(kc[:, C0 + K:])


@pytest.mark.parametrize("K,inter", [(4, 8192), (16, 2048), (1, 256), (12, 8192)])
def test_dense_mlp_block(cuda_ok, K, inter):
    # gate/up in the streamed projection with the SwiGLU in its epilogue
    # (K = 4 at intermediate 8192: 14 row groups per CTA; K = 16: two m-halves;
    # K = 1 at 256), and the row kernels where it does not fit (K = 12 at 8192)
    import moe_nvfp4_block_gb300 as M
    w = dataclasses.replace(synthgen.WORKLOADS["k4_full_step"], K=K)
    mlp = synthgen.make_dense_mlp(w, 0, inter)
    x = synthgen.make_x(w, 12)
    ref = oracle.dense_mlp(oracle.rmsnorm(x), x, mlp["Wg"], mlp["Wu"], mlp["Wd"])
    xd = to_dev_bf16(x)
    out = torch.empty_like(xd)
    M.moe_dense_mlp_block(xd, to_dev_bf16(mlp["Wg"]), to_dev_bf16(mlp["Wu"]), to_dev_bf16(mlp["Wd"]), out,
                          M.dense_mlp_workspace(w.K, w.H, mlp["Wg"].shape[0]))
    torch.cuda.synchronize()
    assert_parity(bf16_bits(out), ref, "dense MLP block")


def _laguna_model(n_layers, K, ctx, vocab):
    base = dataclasses.replace(synthgen.WORKLOADS["k4_full_step"], K=K, ctx=ctx, vocab=vocab, layers=n_layers,
                               E=64, top_k=4, seed=21)
    atts, cfgs, mlps = [], [], []
    for l in range(n_layers):
        cfg = synthgen.laguna_layer_kind(l)
        wl = dataclasses.replace(base, n_q_heads=cfg["n_q_heads"])
        atts.append(synthgen.make_attention(wl, l))
        cfgs.append(cfg)
        mlps.append(synthgen.make_dense_mlp(base, l) if cfg["dense"] else synthgen.make_layer(base, l))
    return base, atts, cfgs, mlps, synthgen.make_lm_head(base)


def test_laguna_schedule_step(cuda_ok):
    import moe_nvfp4_block_gb300 as M
    n_layers, K = 5, 4
    w, atts, cfgs, mlps, lm = _laguna_model(n_layers, K, ctx=640, vocab=4096)
    x0 = synthgen.make_x(w, 13)
    ref = oracle.laguna_step(w, lambda l: (atts[l], cfgs[l], mlps[l]), lm, x0)
    d = lambda a: to_dev_bf16(a)
    layers = []
    for a, cfg, m in zip(atts, cfgs, mlps):
        pos = M.attn_pos(cfg["window"], cfg["rotary_dim"], cfg["rope_theta"], cfg["yarn_factor"], cfg["yarn_orig"])
        if cfg["dense"]:
            layers.append(M.DecoderLayer(d(a["Wq"]), d(a["Wk"]), d(a["Wv"]), d(a["Wo"]), d(a["kc"]), d(a["vc"]), None,
                                         cfg["n_q_heads"], pos, (d(m["Wg"]), d(m["Wu"]), d(m["Wd"]))))
        else:
            layers.append(M.DecoderLayer(d(a["Wq"]), d(a["Wk"]), d(a["Wv"]), d(a["Wo"]), d(a["kc"]), d(a["vc"]),
                                         upload(m, w), cfg["n_q_heads"], pos))
    model = M.VerifyModel(layers, d(lm), w.n_q_heads, w.n_kv_heads)
    # teacher-forced blocks
    for l, (cfg, dl) in enumerate(zip(cfgs, layers)):
        nq = cfg["n_q_heads"]
        xa = d(ref["att_in"][l])
        o = torch.empty(K, nq * 128, dtype=torch.bfloat16, device="cuda")
        M.moe_attention_block(xa, dl.Wq, dl.Wk, dl.Wv, dl.Wo, dl.kcache, dl.vcache, xa,
                              M.attention_workspace(K, w.H, nq, w.n_kv_heads), nq, w.n_kv_heads, o_out=o, pos=dl.pos)
        xm = d(ref["mlp_in"][l])
        if cfg["dense"]:
            ym = torch.empty_like(xm)
            M.moe_dense_mlp_block(xm, *dl.mlp, ym, M.dense_mlp_workspace(K, w.H, dl.mlp[0].shape[0]))
        else:
            xn = torch.empty_like(xm)
            M.moe_rmsnorm(xm, xn)
            ym = torch.empty_like(xm)
            M.moe_verify_layer(dl.moe, xn, xm, ym, M.workspace(dl.moe, K))
        torch.cuda.synchronize()
        assert_parity(bf16_bits(o), ref["att_o"][l], f"layer {l} attention output o")
        assert_parity(bf16_bits(xa), ref["mlp_in"][l], f"layer {l} attention block")
        nxt = ref["att_in"][l + 1] if l + 1 < n_layers else ref["x"]
        assert_parity(bf16_bits(ym), nxt, f"layer {l} {'dense MLP' if cfg['dense'] else 'MoE'} block")
    # greedy tokens, teacher-forced: exact
    tok = torch.empty(K, dtype=torch.int32, device="cuda")
    M.moe_lm_head_argmax(d(oracle.rmsnorm(ref["x"])), model.lm_head, tok, M.lm_head_workspace(K))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tok.cpu().numpy(), ref["target"])
    # the native step, free-running, against the same blocks chained one call
    # at a time on the GPU: bit for bit
    xc = d(x0)
    for cfg, dl in zip(cfgs, layers):
        nq = cfg["n_q_heads"]
        M.moe_attention_block(xc, dl.Wq, dl.Wk, dl.Wv, dl.Wo, dl.kcache, dl.vcache, xc,
                              M.attention_workspace(K, w.H, nq, w.n_kv_heads), nq, w.n_kv_heads, pos=dl.pos)
        if cfg["dense"]:
            M.moe_dense_mlp_block(xc, *dl.mlp, xc, M.dense_mlp_workspace(K, w.H, dl.mlp[0].shape[0]))
        else:
            xn = torch.empty_like(xc)
            M.moe_rmsnorm(xc, xn)
            M.moe_verify_layer(dl.moe, xn, xc, xc, M.workspace(dl.moe, K))
    xn = torch.empty_like(xc)
    M.moe_rmsnorm(xc, xn)
    tok_c = torch.empty(K, dtype=torch.int32, device="cuda")
    M.moe_lm_head_argmax(xn, model.lm_head, tok_c, M.lm_head_workspace(K))
    x = d(x0)
    tgt = torch.empty(K, dtype=torch.int32, device="cuda")
    n = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = model.workspace(K)
    M.moe_verify_step(model, x, torch.from_numpy(ref["target"]).cuda(), tgt, n, ws)
    torch.cuda.synchronize()
    assert M.moe_workspace_error(ws) == 0
    np.testing.assert_array_equal(bf16_bits(x), bf16_bits(xc), err_msg="step vs chained blocks: x")
    np.testing.assert_array_equal(tgt.cpu().numpy(), tok_c.cpu().numpy(), err_msg="step vs chained blocks: tokens")
