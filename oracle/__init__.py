"""CPU oracle for the DFlash MoE verify layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``moe_nvfp4_block_gb300``) never imports, links or executes it.

The arithmetic lives in ``moe_oracle.c`` (plain C11, fp64, compiled with
``-ffp-contract=off`` so that the fixed-order FP32 logits are evaluated exactly
as written).  This module only builds it and marshals numpy arrays.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against values and identities that do not come from the oracle itself
(hand-worked format tables, closed forms, float64 library routines, brute
force on tiny shapes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False, extra_flags=(), out: str | None = None) -> str:
    """Compile the oracle with gcc; ``extra_flags``/``out`` build variants."""
    out = out or _LIB
    if force or extra_flags or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                *extra_flags, _SRC, "-o", out + ".tmp", "-lm"]
        try:
            subprocess.run(base[:3] + ["-fopenmp"] + base[3:], check=True, capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base, check=True)
        os.replace(out + ".tmp", out)
    return out


class Proj(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("tscale", ctypes.c_void_p)]


class LayerC(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("E", ctypes.c_int), ("top_k", ctypes.c_int), ("I", ctypes.c_int),
                ("Is", ctypes.c_int), ("routed_scale", ctypes.c_double),
                ("router_w", ctypes.c_void_p), ("router_b", ctypes.c_void_p),
                ("gate", Proj), ("up", Proj), ("down", Proj),
                ("sh_gate", Proj), ("sh_up", Proj), ("sh_down", Proj), ("scoring", ctypes.c_int)]


SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1

_lib = None


def _bind(L):
    vp, ci, cd = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    L.orc_e2m1.restype = cd
    L.orc_e2m1.argtypes = [ci]
    L.orc_e4m3.restype = cd
    L.orc_e4m3.argtypes = [ci]
    L.orc_bf16.restype = cd
    L.orc_bf16.argtypes = [ctypes.c_uint16]
    L.orc_round_bf16.restype = ctypes.c_uint16
    L.orc_round_bf16.argtypes = [cd]
    L.orc_nvfp4_matrix.argtypes = [vp, ci, ci, ci, vp]
    L.orc_router_logits_f32.argtypes = [vp, vp, ci, vp]
    L.orc_router_logits_f64.argtypes = [vp, vp, ci, vp]
    L.orc_topk.argtypes = [vp, ci, ci, ci, vp, vp]
    L.orc_sigmoid_f32.restype = ctypes.c_float
    L.orc_sigmoid_f32.argtypes = [ctypes.c_float]
    L.orc_topk_sigmoid.argtypes = [vp, vp, ci, ci, ci, vp, vp]
    L.orc_group.argtypes = [vp, ci, ci, ci, vp]
    L.orc_expert.argtypes = [vp, vp, vp, ci, ci, ci, vp, vp, vp]
    L.orc_moe_layer.argtypes = [vp, vp, ci, vp, vp, vp, vp, vp, vp]
    L.orc_rmsnorm.argtypes = [vp, ci, ci, cd, vp]
    L.orc_linear_bf16.argtypes = [vp, vp, ci, ci, ci, vp]
    L.orc_attention.argtypes = [vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp, cd, vp, vp]
    L.orc_lm_argmax.argtypes = [vp, vp, ci, ci, ci, vp, vp]
    L.orc_rope_freqs.argtypes = [ci, cd, cd, ci, vp]
    L.orc_rope_vec.argtypes = [vp, ci, vp, cd]
    L.orc_attention_ex.argtypes = [vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp, cd, ci, ci, cd, cd, ci, vp, vp,
                                   vp, vp]
    L.orc_dense_mlp.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, vp]
    L.orc_accept_prefix.restype = ci
    L.orc_accept_prefix.argtypes = [vp, vp, ci]
    return L


def lib(path: str | None = None):
    """The oracle library (built on first use); ``path`` loads a variant."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


RMS_EPS = 1e-6


class OracleLayer:
    """Keeps numpy arrays alive and exposes the C struct."""

    def __init__(self, layer, H, E, top_k, I, Is, routed_scale=1.0, scoring=SCORE_SOFTMAX):
        self.keep = []

        def arr(a, dt):
            a = _c(a, dt)
            self.keep.append(a)
            return a

        def proj(p):
            if p is None:
                return Proj(None, None, None)
            return Proj(_p(arr(p.codes, np.uint8)), _p(arr(p.scales, np.uint8)), _p(arr(p.tscale, np.float32)))

        rb = None if layer.router_b is None else arr(layer.router_b, np.float32)
        self.c = LayerC(H, E, top_k, I, Is, routed_scale, _p(arr(layer.router_w, np.uint16)), _p(rb),
                        proj(layer.gate), proj(layer.up), proj(layer.down),
                        proj(layer.sh_gate), proj(layer.sh_up), proj(layer.sh_down), scoring)
        self.H, self.E, self.k, self.I, self.Is = H, E, top_k, I, Is

    @classmethod
    def from_workload(cls, w, layer, routed_scale=None, scoring=None):
        return cls(layer, w.H, w.E, w.top_k, w.I, w.Is, w.routed_scale if routed_scale is None else routed_scale,
                   getattr(w, "scoring", SCORE_SOFTMAX) if scoring is None else scoring)

    @property
    def ref(self):
        return ctypes.byref(self.c)


def e2m1(code: int, L=None) -> float:
    return (L or lib()).orc_e2m1(code)


def e4m3(code: int, L=None) -> float:
    return (L or lib()).orc_e4m3(code)


def bf16_value(b: int, L=None) -> float:
    return (L or lib()).orc_bf16(b)


def round_bf16(v: float, L=None) -> int:
    return int((L or lib()).orc_round_bf16(v))


def nvfp4_matrix(p, e, rows, cols, L=None) -> np.ndarray:
    """Dequantised expert e of a projection, float64 [rows, cols]."""
    codes, scales, ts = _c(p.codes, np.uint8), _c(p.scales, np.uint8), _c(p.tscale, np.float32)
    pr = Proj(_p(codes), _p(scales), _p(ts))
    out = np.empty((rows, cols), np.float64)
    (L or lib()).orc_nvfp4_matrix(ctypes.byref(pr), e, rows, cols, _p(out))
    return out


def router_logits_f32(ol: OracleLayer, x, L=None) -> np.ndarray:
    x = _c(x, np.uint16)
    out = np.empty((x.shape[0], ol.E), np.float32)
    (L or lib()).orc_router_logits_f32(ol.ref, _p(x), x.shape[0], _p(out))
    return out


def router_logits_f64(ol: OracleLayer, x, L=None) -> np.ndarray:
    x = _c(x, np.uint16)
    out = np.empty((x.shape[0], ol.E), np.float64)
    (L or lib()).orc_router_logits_f64(ol.ref, _p(x), x.shape[0], _p(out))
    return out


def topk(logits, k, L=None):
    logits = _c(logits, np.float32)
    K, E = logits.shape
    idx = np.empty((K, k), np.int32)
    w = np.empty((K, k), np.float32)
    (L or lib()).orc_topk(_p(logits), K, E, k, _p(idx), _p(w))
    return idx, w


def sigmoid_f32(v: float, L=None) -> float:
    """The FP32 sigmoid of the sigmoid-scored router (a fixed sequence of
    correctly rounded FP32 operations)."""
    return float((L or lib()).orc_sigmoid_f32(float(v)))


def topk_sigmoid(logits, bias, k, L=None):
    """Sigmoid scoring with a selection-only bias: (idx, w) per row."""
    logits = _c(logits, np.float32)
    K, E = logits.shape
    b = None if bias is None else _c(bias, np.float32)
    idx = np.empty((K, k), np.int32)
    w = np.empty((K, k), np.float32)
    (L or lib()).orc_topk_sigmoid(_p(logits), _p(b), K, E, k, _p(idx), _p(w))
    return idx, w


def group_size(K, E, k):
    G = min(E, K * k)
    return 2 + 2 * G + K * k


def group(idx, E, L=None) -> np.ndarray:
    idx = _c(idx, np.int32)
    K, k = idx.shape
    g = np.empty(group_size(K, E, k), np.int32)
    (L or lib()).orc_group(_p(idx), K, E, k, _p(g))
    return g


def expert(gate, up, down, e, H, I, x_row, L=None):
    """One expert on one bf16 row: (d[H] float64, h[I] float64)."""
    keep = [(_c(p.codes, np.uint8), _c(p.scales, np.uint8), _c(p.tscale, np.float32)) for p in (gate, up, down)]
    prs = [Proj(_p(a), _p(b), _p(c)) for a, b, c in keep]
    x_row = _c(x_row, np.uint16)
    d = np.empty(H, np.float64)
    h = np.empty(I, np.float64)
    (L or lib()).orc_expert(ctypes.byref(prs[0]), ctypes.byref(prs[1]), ctypes.byref(prs[2]), e, H, I,
                            _p(x_row), _p(d), _p(h))
    return d, h


def moe_layer(ol: OracleLayer, x_norm, residual=None, L=None):
    """Returns dict(y=bf16 uint16 [K,H], y_f64, idx, w, group)."""
    x_norm = _c(x_norm, np.uint16)
    K = x_norm.shape[0]
    res = None if residual is None else _c(residual, np.uint16)
    y = np.empty((K, ol.H), np.uint16)
    yf = np.empty((K, ol.H), np.float64)
    idx = np.empty((K, ol.k), np.int32)
    w = np.empty((K, ol.k), np.float32)
    g = np.empty(group_size(K, ol.E, ol.k), np.int32)
    (L or lib()).orc_moe_layer(ol.ref, _p(x_norm), K, _p(res), _p(y), _p(idx), _p(w), _p(g), _p(yf))
    return dict(y=y, y_f64=yf, idx=idx, w=w, group=g)


def rmsnorm(x, eps=RMS_EPS, L=None):
    x = _c(x, np.uint16)
    out = np.empty_like(x)
    (L or lib()).orc_rmsnorm(_p(x), x.shape[0], x.shape[1], eps, _p(out))
    return out


def linear_bf16(x, W, L=None):
    x, W = _c(x, np.uint16), _c(W, np.uint16)
    out = np.empty((x.shape[0], W.shape[0]), np.uint16)
    (L or lib()).orc_linear_bf16(_p(x), _p(W), x.shape[0], x.shape[1], W.shape[0], _p(out))
    return out


def attention(x, Wq, Wk, Wv, Wo, kc, vc, nq, nkv, hd, eps=RMS_EPS, L=None, with_o=False):
    """The block output x + o.Wo^T (bf16 [K, H]); with ``with_o`` also the
    attention output o itself (bf16 [K, nq*hd])."""
    x = _c(x, np.uint16)
    K, H = x.shape
    C = kc.shape[1]
    arrs = [_c(a, np.uint16) for a in (Wq, Wk, Wv, Wo, kc, vc)]
    out = np.empty_like(x)
    o = np.empty((K, nq * hd), np.uint16) if with_o else None
    (L or lib()).orc_attention(_p(x), K, H, nq, nkv, hd, C, *[_p(a) for a in arrs], eps, _p(out), _p(o))
    return (out, o) if with_o else out


def rope_freqs(rd, theta=10000.0, yarn_factor=1.0, yarn_orig=0, L=None):
    """Per rotary pair i < rd/2 the angle per position (YaRN-scaled when
    yarn_factor > 1)."""
    f = np.empty(rd // 2, np.float64)
    (L or lib()).orc_rope_freqs(rd, theta, yarn_factor, yarn_orig, _p(f))
    return f


def rope_vec(v, rd, freqs, pos, L=None):
    """One head vector (float64) rotated at position pos (no rounding)."""
    v = np.array(v, np.float64)
    f = _c(freqs, np.float64)
    (L or lib()).orc_rope_vec(_p(v), rd, _p(f), float(pos))
    return v


def attention_ex(x, Wq, Wk, Wv, Wo, kc, vc, nq, nkv, hd, window=0, rotary_dim=0, theta=10000.0, yarn_factor=1.0,
                 yarn_orig=0, eps=RMS_EPS, L=None):
    """A Laguna attention block (RoPE / YaRN, sliding window); returns dict
    (x=block output, k_new, v_new (the rotated new keys and the values), o)."""
    x = _c(x, np.uint16)
    K, H = x.shape
    C = kc.shape[1]
    arrs = [_c(a, np.uint16) for a in (Wq, Wk, Wv, Wo, kc, vc)]
    out = np.empty_like(x)
    kn = np.empty((K, nkv * hd), np.uint16)
    vn = np.empty((K, nkv * hd), np.uint16)
    o = np.empty((K, nq * hd), np.uint16)
    (L or lib()).orc_attention_ex(_p(x), K, H, nq, nkv, hd, C, *[_p(a) for a in arrs], eps, window, rotary_dim,
                                  theta, yarn_factor, yarn_orig, _p(out), _p(kn), _p(vn), _p(o))
    return dict(x=out, k_new=kn, v_new=vn, o=o)


def dense_mlp(x_norm, residual, Wg, Wu, Wd, L=None):
    """Laguna's layer-0 dense SwiGLU MLP: bf16 [K][H]."""
    x_norm = _c(x_norm, np.uint16)
    K, H = x_norm.shape
    I = Wg.shape[0]
    res = None if residual is None else _c(residual, np.uint16)
    y = np.empty_like(x_norm)
    (L or lib()).orc_dense_mlp(_p(x_norm), _p(res), _p(_c(Wg, np.uint16)), _p(_c(Wu, np.uint16)),
                               _p(_c(Wd, np.uint16)), K, H, I, _p(y))
    return y


def lm_argmax(x_norm, W, L=None):
    x_norm, W = _c(x_norm, np.uint16), _c(W, np.uint16)
    K, H = x_norm.shape
    tok = np.empty(K, np.int32)
    best = np.empty(K, np.float32)
    (L or lib()).orc_lm_argmax(_p(x_norm), _p(W), K, H, W.shape[0], _p(tok), _p(best))
    return tok, best


def accept_prefix(draft, target, L=None) -> int:
    d, t = _c(draft, np.int32), _c(target, np.int32)
    return int((L or lib()).orc_accept_prefix(_p(d), _p(t), d.shape[0]))


def moe_stack(w, layers, x0, n_layers=None, L=None, collect=False):
    """Free-running stack of MoE layers: x_{l+1} = moe_l(rmsnorm(x_l)) + x_l.
    ``layers`` is a callable l -> synthgen.Layer.  Returns the final x and,
    with ``collect``, the list of per-layer inputs x_l."""
    x = _c(x0, np.uint16)
    xs = []
    for l in range(n_layers or w.layers):
        if collect:
            xs.append(x.copy())
        ol = OracleLayer.from_workload(w, layers(l))
        x = moe_layer(ol, rmsnorm(x, L=L), residual=x, L=L)["y"]
    return (x, xs) if collect else x


def verify_step(w, layers, lm_head, x0, n_layers=None, L=None):
    """The full verify step: per layer the attention block, then the MoE block
    (x <- x + MoE(rmsnorm(x))), then the lm_head argmax of every row.
    ``layers(l)`` returns (attention dict with Wq, Wk, Wv, Wo, kc, vc; MoE
    synthgen.Layer).  Returns dict(x, target, best, att_in, att_o, moe_in, idx,
    xn): att_o[l] is layer l's attention output o (before the o-projection)."""
    x = _c(x0, np.uint16)
    att_in, moe_in, idx, att_o = [], [], [], []
    for l in range(n_layers or w.layers):
        att, moe = layers(l)
        att_in.append(x.copy())
        x, o = attention(x, att["Wq"], att["Wk"], att["Wv"], att["Wo"], att["kc"], att["vc"], w.n_q_heads,
                         w.n_kv_heads, w.head_dim, L=L, with_o=True)
        att_o.append(o)
        moe_in.append(x.copy())
        r = moe_layer(OracleLayer.from_workload(w, moe), rmsnorm(x, L=L), residual=x, L=L)
        idx.append(r["idx"])
        x = r["y"]
    xn = rmsnorm(x, L=L)
    tok, best = lm_argmax(xn, lm_head, L=L)
    return dict(x=x, target=tok, best=best, att_in=att_in, att_o=att_o, moe_in=moe_in, idx=idx, xn=xn)


def synthetic_drafts(target, coin, alt, vocab):
    """The controlled-acceptance drafter: the target's token where coin is
    set, else (target + 1 + alt) mod vocab (never the target's token)."""
    t = np.asarray(target, np.int64)
    return np.where(np.asarray(coin) != 0, t, (t + 1 + np.asarray(alt, np.int64)) % vocab).astype(np.int32)


def verify_rounds(w, layers, lm_head, x_rounds, coin, alt, ctx0, n_layers=None, L=None):
    """The multi-round verify loop with an in-place KV cache (PR #844, "8. What
    I looked at and did NOT ship", items 1 and 2; "10. Next step"): round t
    runs the K rows x_rounds[t] through every layer -- attention over the
    committed cache positions 0 .. len-1 plus the round's own rows, then the
    MoE block -- takes the greedy token of every row, forms the synthetic
    drafts, counts the accepted prefix n, and commits the first
    c = min(n + 1, K) rows' keys and values of every layer to the cache
    (len += c); the other rows are dropped.
    ``layers(l)`` returns (attention dict with Wq, Wk, Wv, Wo and caches kc, vc
    [nkv][cap][hd] whose first ctx0 positions are valid; MoE synthgen.Layer).
    Returns dict(targets [R][K], drafts [R][K], n [R], len, kc, vc: per layer
    the caches' first len positions)."""
    nl = n_layers or w.layers
    R, K = x_rounds.shape[0], x_rounds.shape[1]
    hd, nq, nkv = w.head_dim, w.n_q_heads, w.n_kv_heads
    kcs, vcs = [], []
    for l in range(nl):
        att, _ = layers(l)
        kcs.append(_c(att["kc"][:, :ctx0], np.uint16))
        vcs.append(_c(att["vc"][:, :ctx0], np.uint16))
    targets = np.zeros((R, K), np.int32)
    drafts = np.zeros((R, K), np.int32)
    ns = np.zeros(R, np.int32)
    for t in range(R):
        x = _c(x_rounds[t], np.uint16)
        knew, vnew = [], []
        for l in range(nl):
            att, moe = layers(l)
            xn = rmsnorm(x, L=L)
            knew.append(linear_bf16(xn, att["Wk"], L=L).reshape(K, nkv, hd))
            vnew.append(linear_bf16(xn, att["Wv"], L=L).reshape(K, nkv, hd))
            x = attention(x, att["Wq"], att["Wk"], att["Wv"], att["Wo"], kcs[l], vcs[l], nq, nkv, hd, L=L)
            x = moe_layer(OracleLayer.from_workload(w, moe), rmsnorm(x, L=L), residual=x, L=L)["y"]
        tok, _ = lm_argmax(rmsnorm(x, L=L), lm_head, L=L)
        d = synthetic_drafts(tok, coin[t], alt[t], lm_head.shape[0])
        n = accept_prefix(d, tok, L=L)
        c = min(n + 1, K)
        for l in range(nl):
            kcs[l] = np.ascontiguousarray(np.concatenate([kcs[l], knew[l][:c].transpose(1, 0, 2)], axis=1))
            vcs[l] = np.ascontiguousarray(np.concatenate([vcs[l], vnew[l][:c].transpose(1, 0, 2)], axis=1))
        targets[t], drafts[t], ns[t] = tok, d, n
    return dict(targets=targets, drafts=drafts, n=ns, len=kcs[0].shape[1], kc=kcs, vc=vcs)


def laguna_step(w, layers, lm_head, x0, n_layers=None, L=None):
    """The verify step of the Laguna layer schedule: per layer the attention
    block with its window / rotary embedding, then its dense MLP (layer 0) or
    MoE block, then the lm_head argmax of every row.  ``layers(l)`` returns
    (attention dict with Wq, Wk, Wv, Wo, kc, vc; configuration dict of
    synthgen.laguna_layer_kind; MLP dict (dense) or MoE synthgen.Layer).
    Returns dict(x, target, att_in, mlp_in, att_o)."""
    x = _c(x0, np.uint16)
    att_in, mlp_in, att_o = [], [], []
    for l in range(n_layers or w.layers):
        att, cfg, mlp = layers(l)
        att_in.append(x.copy())
        r = attention_ex(x, att["Wq"], att["Wk"], att["Wv"], att["Wo"], att["kc"], att["vc"], cfg["n_q_heads"],
                         w.n_kv_heads, w.head_dim, window=cfg["window"], rotary_dim=cfg["rotary_dim"],
                         theta=cfg["rope_theta"], yarn_factor=cfg["yarn_factor"], yarn_orig=cfg["yarn_orig"], L=L)
        x = r["x"]
        att_o.append(r["o"])
        mlp_in.append(x.copy())
        if cfg["dense"]:
            x = dense_mlp(rmsnorm(x, L=L), x, mlp["Wg"], mlp["Wu"], mlp["Wd"], L=L)
        else:
            x = moe_layer(OracleLayer.from_workload(w, mlp), rmsnorm(x, L=L), residual=x, L=L)["y"]
    tok, best = lm_argmax(rmsnorm(x, L=L), lm_head, L=L)
    return dict(x=x, target=tok, best=best, att_in=att_in, mlp_in=mlp_in, att_o=att_o)
