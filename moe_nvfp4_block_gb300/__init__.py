"""Python binding of the GB300 MoE verify-layer library (``include/moe_verify.h``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (torch supplies device memory and
the current stream); bf16 tensors may be passed as ``torch.bfloat16`` or as
their 16-bit patterns (``torch.int16``/``torch.uint16``).  The library must
be built (``__graft_entry__.build()`` or ``python moe_nvfp4_block_gb300/build.py``);
importing this package without it raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_verify.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_WORKSPACE_TOO_SMALL = -3
MOE_ERR_MISALIGNED = -4
MOE_ERR_CUDA = -5
MOE_ERR_DEVICE_TIMEOUT = -6
MOE_ERR_CAPACITY = -7
MOE_MAX_ROWS = 16

# Every symbol the header declares (checked by the tests).
EXPORTS = ("moe_verify_layer_workspace_size", "moe_router_topk", "moe_group_ints", "moe_verify_layer",
           "moe_verify_layer_profiled", "verify_accept_prefix", "moe_rmsnorm", "moe_lm_head_workspace_size",
           "moe_lm_head_argmax", "moe_verify_stack_workspace_size", "moe_verify_stack",
           "moe_attention_workspace_size", "moe_attention_block", "moe_verify_layer_static",
           "moe_verify_step_workspace_size", "moe_verify_step", "moe_workspace_error", "moe_status_string", "moe_host_pointer",
           "moe_debug_set_wait_limit_ns", "moe_debug_set_trace", "moe_debug_partials_offset", "moe_kv_commit",
           "moe_synthetic_drafts", "moe_verify_rounds", "moe_dense_mlp_workspace_size", "moe_dense_mlp_block")


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class moe_nvfp4(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p)]


class moe_layer(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("inter", ctypes.c_int), ("shared_inter", ctypes.c_int), ("routed_scale", ctypes.c_float),
                ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("gate", moe_nvfp4), ("up", moe_nvfp4), ("down", moe_nvfp4),
                ("sh_gate", moe_nvfp4), ("sh_up", moe_nvfp4), ("sh_down", moe_nvfp4), ("scoring", ctypes.c_int)]


MOE_SCORE_SOFTMAX = 0
MOE_SCORE_SIGMOID = 1


class moe_attn_pos(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int), ("rotary_dim", ctypes.c_int), ("rope_theta", ctypes.c_float),
                ("yarn_factor", ctypes.c_float), ("yarn_orig_ctx", ctypes.c_int)]


class moe_decoder_layer(ctypes.Structure):
    _fields_ = [("Wq", ctypes.c_void_p), ("Wk", ctypes.c_void_p), ("Wv", ctypes.c_void_p), ("Wo", ctypes.c_void_p),
                ("kcache", ctypes.c_void_p), ("vcache", ctypes.c_void_p), ("moe", moe_layer),
                ("n_q_heads", ctypes.c_int), ("pos", moe_attn_pos), ("mlp_gate", ctypes.c_void_p),
                ("mlp_up", ctypes.c_void_p), ("mlp_down", ctypes.c_void_p), ("mlp_inter", ctypes.c_int)]


class moe_verify_model(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ctx", ctypes.c_int),
                ("vocab", ctypes.c_int), ("eps", ctypes.c_float), ("layers", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p), ("kv_len", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lp = ctypes.POINTER(moe_layer)
    L.moe_verify_layer_workspace_size.restype = sz
    L.moe_verify_layer_workspace_size.argtypes = [lp, ci]
    L.moe_group_ints.restype = sz
    L.moe_group_ints.argtypes = [ci, ci, ci]
    L.moe_router_topk.restype = ci
    L.moe_router_topk.argtypes = [lp, vp, ci, vp, vp, vp, vp, sz, vp]
    L.moe_verify_layer.restype = ci
    L.moe_verify_layer.argtypes = [lp, vp, ci, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_verify_layer_static.restype = ci
    L.moe_verify_layer_static.argtypes = [lp, vp, ci, vp, vp, vp, vp, vp, vp]
    L.moe_verify_layer_profiled.restype = ci
    L.moe_verify_layer_profiled.argtypes = [lp, vp, ci, vp, vp, vp, sz, vp, vp]
    L.verify_accept_prefix.restype = ci
    L.verify_accept_prefix.argtypes = [vp, vp, ci, vp, vp]
    L.moe_verify_stack_workspace_size.restype = sz
    L.moe_verify_stack_workspace_size.argtypes = [lp, ci, ci]
    L.moe_verify_stack.restype = ci
    L.moe_verify_stack.argtypes = [lp, ci, vp, ci, ctypes.c_float, vp, sz, vp]
    L.moe_attention_workspace_size.restype = sz
    L.moe_attention_workspace_size.argtypes = [ci, ci, ci, ci, ci]
    L.moe_attention_block.restype = ci
    L.moe_attention_block.argtypes = [vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                      vp, vp, vp, vp, vp, sz, vp]
    L.moe_dense_mlp_workspace_size.restype = sz
    L.moe_dense_mlp_workspace_size.argtypes = [ci, ci, ci]
    L.moe_dense_mlp_block.restype = ci
    L.moe_dense_mlp_block.argtypes = [vp, ci, ci, ci, vp, vp, vp, ctypes.c_float, vp, vp, sz, vp]
    mp = ctypes.POINTER(moe_verify_model)
    L.moe_verify_step_workspace_size.restype = sz
    L.moe_verify_step_workspace_size.argtypes = [mp, ci]
    L.moe_verify_step.restype = ci
    L.moe_verify_step.argtypes = [mp, vp, ci, vp, vp, vp, vp, sz, vp]
    L.moe_kv_commit.restype = ci
    L.moe_kv_commit.argtypes = [vp, vp, ci, ci, vp]
    L.moe_synthetic_drafts.restype = ci
    L.moe_synthetic_drafts.argtypes = [vp, vp, vp, ci, ci, vp, vp]
    L.moe_verify_rounds.restype = ci
    L.moe_verify_rounds.argtypes = [mp, vp, ci, ci, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_rmsnorm.restype = ci
    L.moe_rmsnorm.argtypes = [vp, ci, ci, ctypes.c_float, vp, vp]
    L.moe_lm_head_workspace_size.restype = sz
    L.moe_lm_head_workspace_size.argtypes = [ci]
    L.moe_lm_head_argmax.restype = ci
    L.moe_lm_head_argmax.argtypes = [vp, ci, ci, vp, ci, vp, vp, vp, sz, vp]
    L.moe_workspace_error.restype = ci
    L.moe_workspace_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int), vp]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_status_string.argtypes = [ci]
    L.moe_host_pointer.restype = ci
    L.moe_host_pointer.argtypes = [vp, ctypes.POINTER(vp)]
    L.moe_debug_set_wait_limit_ns.restype = None
    L.moe_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.moe_debug_set_trace.restype = None
    L.moe_debug_set_trace.argtypes = [vp]
    L.moe_debug_partials_offset.restype = sz
    L.moe_debug_partials_offset.argtypes = [lp, ci]
    return L


lib = _load()


def status_string(s: int) -> str:
    return lib.moe_status_string(int(s)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def host_pointer(t) -> int:
    """The device address of a pinned host tensor (moe_host_pointer)."""
    d = ctypes.c_void_p()
    _check(lib.moe_host_pointer(ctypes.c_void_p(t.data_ptr()), ctypes.byref(d)), "moe_host_pointer")
    return d.value


def _act_ptr(t):
    """A layer call's activation: a CUDA tensor, or a pinned host tensor
    that the kernel reads or writes across the host link."""
    if t is None or t.is_cuda:
        return _ptr(t)
    d = ctypes.c_void_p()  # moe_host_pointer refuses memory that is not pinned
    if lib.moe_host_pointer(ctypes.c_void_p(t.data_ptr()), ctypes.byref(d)) != MOE_OK:
        raise ValueError("a host activation must be pinned memory")
    return d


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, what):
    if status != MOE_OK:
        raise MoeError(status, what)


@dataclass
class Proj:
    """Device tensors of one NVFP4 projection stack [n_exp][rows][cols]."""
    codes: torch.Tensor   # uint8 [n_exp, rows, cols//2]
    scales: torch.Tensor  # uint8 [n_exp, rows, cols//16]
    tscale: torch.Tensor  # float32 [n_exp]

    def c(self):
        return moe_nvfp4(self.codes.data_ptr(), self.scales.data_ptr(), self.tscale.data_ptr())


@dataclass
class Layer:
    """Device tensors of one MoE layer; ``c()`` gives the ``moe_layer`` struct."""
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int
    routed_scale: float
    router_w: torch.Tensor          # bf16 [E, H]
    router_bias: torch.Tensor | None
    gate: Proj
    up: Proj
    down: Proj
    sh_gate: Proj | None = None
    sh_up: Proj | None = None
    sh_down: Proj | None = None
    scoring: int = MOE_SCORE_SOFTMAX

    def c(self) -> moe_layer:
        z = moe_nvfp4(None, None, None)
        sh = self.shared_inter > 0
        return moe_layer(self.hidden, self.n_experts, self.top_k, self.inter, self.shared_inter,
                         self.routed_scale, self.router_w.data_ptr(),
                         None if self.router_bias is None else self.router_bias.data_ptr(),
                         self.gate.c(), self.up.c(), self.down.c(),
                         self.sh_gate.c() if sh else z, self.sh_up.c() if sh else z,
                         self.sh_down.c() if sh else z, self.scoring)


def moe_group_ints(K: int, n_experts: int, top_k: int) -> int:
    return int(lib.moe_group_ints(K, n_experts, top_k))


def moe_verify_layer_workspace_size(layer: Layer, K: int) -> int:
    c = layer.c()
    return int(lib.moe_verify_layer_workspace_size(ctypes.byref(c), K))


def workspace(layer: Layer, K: int, device=None) -> torch.Tensor:
    """A zero-filled workspace for ``layer`` at K rows (uint8 device tensor)."""
    n = moe_verify_layer_workspace_size(layer, K)
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device or layer.router_w.device)


def moe_router_topk(layer: Layer, x_norm, idx, w, group, ws, stream=None):
    c = layer.c()
    _check(lib.moe_router_topk(ctypes.byref(c), _ptr(x_norm), x_norm.shape[0], _ptr(idx), _ptr(w), _ptr(group),
                               _ptr(ws), ws.numel(), _stream(stream)), "moe_router_topk")


def moe_verify_layer(layer: Layer, x_norm, residual, y, ws, idx_out=None, w_out=None, group_out=None,
                     stream=None, c_layer: moe_layer | None = None):
    c = layer.c() if c_layer is None else c_layer
    _check(lib.moe_verify_layer(ctypes.byref(c), _act_ptr(x_norm), x_norm.shape[0], _act_ptr(residual), _act_ptr(y),
                                _ptr(idx_out), _ptr(w_out), _ptr(group_out), _ptr(ws), ws.numel(),
                                _stream(stream)), "moe_verify_layer")


def moe_verify_layer_static(layer: Layer, x_norm, residual, y, idx_out=None, w_out=None, group_out=None,
                            stream=None):
    """moe_verify_layer with the library's built-in scratch array (no workspace
    argument, no allocation); see include/moe_verify.h for its limits."""
    c = layer.c()
    _check(lib.moe_verify_layer_static(ctypes.byref(c), _ptr(x_norm), x_norm.shape[0], _ptr(residual), _ptr(y),
                                       _ptr(idx_out), _ptr(w_out), _ptr(group_out), _stream(stream)),
           "moe_verify_layer_static")


def moe_verify_layer_profiled(layer: Layer, x_norm, residual, y, ws, events=None, stream=None,
                              c_layer: moe_layer | None = None):
    """``events``: four torch.cuda.Event(enable_timing=True) or None."""
    c = layer.c() if c_layer is None else c_layer
    ev = None
    if events is not None:
        for e in events:
            if not e.cuda_event:  # torch creates the handle on first record
                e.record(stream if stream is not None else torch.cuda.current_stream())
        arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
        ev = ctypes.cast(arr, ctypes.c_void_p)
    _check(lib.moe_verify_layer_profiled(ctypes.byref(c), _ptr(x_norm), x_norm.shape[0], _ptr(residual), _ptr(y),
                                         _ptr(ws), ws.numel(), _stream(stream), ev), "moe_verify_layer_profiled")


def verify_accept_prefix(draft, target, n_accepted, stream=None):
    _check(lib.verify_accept_prefix(_ptr(draft), _ptr(target), draft.shape[0], _ptr(n_accepted),
                                    _stream(stream)), "verify_accept_prefix")


def layer_array(layers) -> ctypes.Array:
    """A C array of ``moe_layer`` structs (keep it alive while in use)."""
    return (moe_layer * len(layers))(*[l.c() for l in layers])


def moe_verify_stack_workspace_size(c_layers, K: int) -> int:
    return int(lib.moe_verify_stack_workspace_size(c_layers, len(c_layers), K))


def stack_workspace(c_layers, K: int, device="cuda") -> torch.Tensor:
    n = moe_verify_stack_workspace_size(c_layers, K)
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "stack workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def moe_verify_stack(c_layers, x, ws, eps=1e-6, stream=None):
    _check(lib.moe_verify_stack(c_layers, len(c_layers), _ptr(x), x.shape[0], float(eps), _ptr(ws), ws.numel(),
                                _stream(stream)), "moe_verify_stack")


def attention_workspace(K, H, nq, nkv, head_dim=128, device="cuda") -> torch.Tensor:
    n = int(lib.moe_attention_workspace_size(K, H, nq, nkv, head_dim))
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "attention workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def attn_pos(window=0, rotary_dim=0, rope_theta=10000.0, yarn_factor=1.0, yarn_orig_ctx=0) -> moe_attn_pos:
    return moe_attn_pos(window, rotary_dim, rope_theta, yarn_factor, yarn_orig_ctx)


def moe_attention_block(x, Wq, Wk, Wv, Wo, kcache, vcache, x_out, ws, nq, nkv, eps=1e-6, k_new=None, v_new=None,
                        stream=None, o_out=None, kv_len=None, pos: moe_attn_pos | None = None):
    K, H = x.shape
    C = kcache.shape[1]
    _check(lib.moe_attention_block(_ptr(x), K, H, nq, nkv, 128, C, _ptr(Wq), _ptr(Wk), _ptr(Wv), _ptr(Wo),
                                   _ptr(kcache) if C else None, _ptr(vcache) if C else None, _ptr(kv_len),
                                   None if pos is None else ctypes.byref(pos), float(eps),
                                   _ptr(x_out), _ptr(k_new), _ptr(v_new), _ptr(o_out), _ptr(ws), ws.numel(),
                                   _stream(stream)),
           "moe_attention_block")


def dense_mlp_workspace(K, H, I, device="cuda") -> torch.Tensor:
    n = int(lib.moe_dense_mlp_workspace_size(K, H, I))
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "dense MLP workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def moe_dense_mlp_block(x, Wg, Wu, Wd, x_out, ws, eps=1e-6, stream=None):
    K, H = x.shape
    _check(lib.moe_dense_mlp_block(_ptr(x), K, H, Wg.shape[0], _ptr(Wg), _ptr(Wu), _ptr(Wd), float(eps), _ptr(x_out),
                                   _ptr(ws), ws.numel(), _stream(stream)), "moe_dense_mlp_block")


@dataclass
class DecoderLayer:
    """Device tensors of one decoder layer: attention weights, KV cache, and
    the MoE block -- or, with ``mlp`` = (Wg, Wu, Wd), a dense SwiGLU MLP.
    ``n_q_heads`` 0 takes the model's; ``pos`` (moe_attn_pos) the window and
    rotary embedding of the attention."""
    Wq: torch.Tensor
    Wk: torch.Tensor
    Wv: torch.Tensor
    Wo: torch.Tensor
    kcache: torch.Tensor
    vcache: torch.Tensor
    moe: Layer | None
    n_q_heads: int = 0
    pos: moe_attn_pos | None = None
    mlp: tuple | None = None


class VerifyModel:
    """Holds the C description (``moe_verify_model``) of a stack of decoder
    layers plus the lm_head; keeps the ctypes arrays alive."""

    def __init__(self, layers, lm_head, n_q_heads, n_kv_heads, eps=1e-6, kv_len=None):
        """``kv_len``: None (caches read only, all positions valid) or a device
        int32 tensor [1] -- the caches' second dimension is then their
        capacity and every step appends its rows in place."""
        self.layers = layers
        self.lm_head = lm_head
        self.kv_len = kv_len
        p = lambda t: t.data_ptr()

        def c_layer(d):
            mg, mu, md = (p(d.mlp[0]), p(d.mlp[1]), p(d.mlp[2])) if d.mlp else (None, None, None)
            return moe_decoder_layer(p(d.Wq), p(d.Wk), p(d.Wv), p(d.Wo), p(d.kcache), p(d.vcache),
                                     d.moe.c() if d.moe is not None else moe_layer(), d.n_q_heads,
                                     d.pos if d.pos is not None else moe_attn_pos(), mg, mu, md,
                                     d.mlp[0].shape[0] if d.mlp else 0)

        self.c_layers = (moe_decoder_layer * len(layers))(*[c_layer(d) for d in layers])
        d0 = layers[0]
        self.c = moe_verify_model(len(layers), d0.Wq.shape[1], n_q_heads, n_kv_heads, 128, d0.kcache.shape[1],
                                  lm_head.shape[0], eps, ctypes.cast(self.c_layers, ctypes.c_void_p),
                                  lm_head.data_ptr(), None if kv_len is None else kv_len.data_ptr())

    def workspace(self, K, device=None):
        n = int(lib.moe_verify_step_workspace_size(ctypes.byref(self.c), K))
        if n == 0:
            raise MoeError(MOE_ERR_INVALID_ARG, "verify step workspace size")
        return torch.zeros(n, dtype=torch.uint8, device=device or self.lm_head.device)


def moe_verify_step(model: VerifyModel, x, draft, target, n_accepted, ws, stream=None):
    _check(lib.moe_verify_step(ctypes.byref(model.c), _ptr(x), x.shape[0], _ptr(draft), _ptr(target),
                               _ptr(n_accepted), _ptr(ws), ws.numel(), _stream(stream)), "moe_verify_step")


def moe_kv_commit(kv_len, n_accepted, K, capacity, stream=None):
    _check(lib.moe_kv_commit(_ptr(kv_len), _ptr(n_accepted), K, capacity, _stream(stream)), "moe_kv_commit")


def moe_synthetic_drafts(target, coin, alt, vocab, draft, stream=None):
    _check(lib.moe_synthetic_drafts(_ptr(target), _ptr(coin), _ptr(alt), target.shape[0], vocab, _ptr(draft),
                                    _stream(stream)), "moe_synthetic_drafts")


def moe_verify_rounds(model: "VerifyModel", x_rounds, coin, alt, x_work, targets, drafts, n_accepted, ws, stream=None):
    """x_rounds bf16 [R, K, H]; coin uint8 [R, K]; alt int32 [R, K]; outputs
    targets, drafts int32 [R, K] and n_accepted int32 [R]."""
    R, K = x_rounds.shape[0], x_rounds.shape[1]
    _check(lib.moe_verify_rounds(ctypes.byref(model.c), _ptr(x_rounds), R, K, _ptr(coin), _ptr(alt), _ptr(x_work),
                                 _ptr(targets), _ptr(drafts), _ptr(n_accepted), _ptr(ws), ws.numel(),
                                 _stream(stream)), "moe_verify_rounds")


def moe_rmsnorm(x, out, eps=1e-6, stream=None):
    _check(lib.moe_rmsnorm(_ptr(x), x.shape[0], x.shape[1], float(eps), _ptr(out), _stream(stream)), "moe_rmsnorm")


def moe_lm_head_workspace_size(K: int) -> int:
    return int(lib.moe_lm_head_workspace_size(K))


def lm_head_workspace(K: int, device="cuda") -> torch.Tensor:
    return torch.zeros(moe_lm_head_workspace_size(K), dtype=torch.uint8, device=device)


def moe_lm_head_argmax(x_norm, W, tok, ws, best_logit=None, stream=None):
    _check(lib.moe_lm_head_argmax(_ptr(x_norm), x_norm.shape[0], x_norm.shape[1], _ptr(W), W.shape[0], _ptr(tok),
                                  _ptr(best_logit), _ptr(ws), ws.numel(), _stream(stream)), "moe_lm_head_argmax")


def moe_workspace_error(ws, stream=None) -> int:
    code = ctypes.c_int(0)
    _check(lib.moe_workspace_error(_ptr(ws), ctypes.byref(code), _stream(stream)), "moe_workspace_error")
    return code.value


def moe_debug_set_wait_limit_ns(ns: int):
    lib.moe_debug_set_wait_limit_ns(int(ns))


def moe_debug_set_trace(buf):
    """Device uint64 tensor [n_sms, 80] for milestone stamps, or None."""
    lib.moe_debug_set_trace(None if buf is None else ctypes.c_void_p(buf.data_ptr()))


def _dev(a, device, dtype=None):
    t = torch.from_numpy(a.copy() if not a.flags.c_contiguous else a)
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device, non_blocking=False)


def layer_from_arrays(router_w, router_bias, gate, up, down, sh=None, top_k=8, routed_scale=1.0,
                      device="cuda", scoring=MOE_SCORE_SOFTMAX) -> Layer:
    """Uploads host arrays to a device ``Layer``.  ``gate``/``up``/``down`` (and
    the optional ``sh`` triple) are (codes uint8, scales uint8, tscale float32)
    numpy arrays shaped [n_exp, rows, cols//2], [n_exp, rows, cols//16], [n_exp];
    ``router_w`` is uint16 bf16 bits [E, H]."""
    def proj(p):
        c, s, t = p
        return Proj(_dev(c, device), _dev(s, device), _dev(t, device))

    E, H = router_w.shape
    I = gate[0].shape[1]
    return Layer(hidden=H, n_experts=E, top_k=top_k, inter=I, shared_inter=0 if sh is None else sh[0][0].shape[1],
                 routed_scale=routed_scale, router_w=_dev(router_w, device, torch.bfloat16),
                 router_bias=None if router_bias is None else _dev(router_bias, device),
                 gate=proj(gate), up=proj(up), down=proj(down),
                 sh_gate=None if sh is None else proj(sh[0]), sh_up=None if sh is None else proj(sh[1]),
                 sh_down=None if sh is None else proj(sh[2]), scoring=scoring)
