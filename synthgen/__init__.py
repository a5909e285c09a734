"""Seeded synthetic inputs for the MoE verify layer (shared by the CUDA path's
tests/benchmark and by the CPU oracle).

This package draws random numbers and stores them in the workload's formats;
it holds none of the layer's arithmetic.  The C core (``synthgen.c``) is a
counter-based SplitMix64 stream, so any expert's weights can be regenerated on
their own (the oracle regenerates only the experts a row routes to).

Workloads (all shapes from the DFlash verify setting the pages describe: 256
routed experts, top-8, a shared expert, expert intermediate 512, hidden 2048,
NVFP4 group-16 expert weights, bf16 router; "Why this challenge exists" on the
mlxfast Laguna XS 2.1 (DFlash) README):

* ``tiny``            K=1, H=256, E=16, top-2, I=128, no shared expert, 1 layer
* ``k2_layer``        K=2, H=2048, E=256, top-8, I=512, shared I=512, 1 layer
* ``k8_stack40``      as k2_layer, K=8, 40 layers, residual + RMSNorm between
* ``k16_zipf_stack40`` as k8_stack40, K=16, router bias -1.1*ln(e+1)
* ``k4_full_step``    K=4, 40 x (GQA attention + MoE) + lm_head argmax

Value recipe: 4-bit codes uniform over all 16 codes; E4M3 block scales
uniform in [2^-8, 2^-4] rounded to E4M3; FP32 tensor scales 1.0; router
weights bf16 N(0, 0.02); activations bf16 N(0, 1); seed = workload index.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synthgen.c")
_LIB = os.path.join(_HERE, "libsynthgen.so")

# Tensor ids: each tensor of each layer draws from its own stream.
T_ROUTER_W, T_ROUTER_B = 1, 2
T_GATE_C, T_GATE_S, T_UP_C, T_UP_S, T_DOWN_C, T_DOWN_S = 3, 4, 5, 6, 7, 8
T_SGATE_C, T_SGATE_S, T_SUP_C, T_SUP_S, T_SDOWN_C, T_SDOWN_S = 9, 10, 11, 12, 13, 14
T_X = 20
T_ATT_Q, T_ATT_K, T_ATT_V, T_ATT_O, T_KCACHE, T_VCACHE = 30, 31, 32, 33, 34, 35
T_LM_HEAD, T_DRAFT_J, T_DRAFT_TOK = 40, 41, 42
T_COIN, T_ALT = 43, 44
T_MLP_G, T_MLP_U, T_MLP_D = 45, 46, 47

SCALE_LO, SCALE_HI = 2.0 ** -8, 2.0 ** -4
ROUTER_SIGMA = 0.02


def build(force: bool = False) -> str:
    """Compile the C core with gcc (OpenMP when available)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
        try:
            subprocess.run(base[:4] + ["-fopenmp"] + base[4:], check=True, capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u64, u32, i64 = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64
        vp, dbl = ctypes.c_void_p, ctypes.c_double
        L.sg_key.restype = u64
        L.sg_key.argtypes = [u64, u32, u32]
        L.sg_u64.restype = u64
        L.sg_u64.argtypes = [u64, u64]
        L.sg_fill_codes.argtypes = [u64, u64, u64, vp]
        L.sg_fill_scales.argtypes = [u64, u64, u64, dbl, dbl, vp]
        L.sg_fill_normal_bf16.argtypes = [u64, u64, u64, dbl, dbl, vp]
        L.sg_fill_uniform_int.argtypes = [u64, u64, u64, u64, vp]
        L.sg_zipf_log_prior.argtypes = [dbl, ctypes.c_int, vp]
        _lib = L
    return _lib


def key(seed: int, layer: int, tensor: int) -> int:
    return int(lib().sg_key(seed, layer, tensor))


def codes(seed, layer, tensor, byte_off, n, out=None):
    out = np.empty(n, np.uint8) if out is None else out
    assert byte_off % 8 == 0 and out.nbytes >= n and out.flags.c_contiguous
    lib().sg_fill_codes(key(seed, layer, tensor), byte_off, n, out.ctypes.data)
    return out


def scales(seed, layer, tensor, off, n, out=None, lo=SCALE_LO, hi=SCALE_HI):
    out = np.empty(n, np.uint8) if out is None else out
    assert out.flags.c_contiguous
    lib().sg_fill_scales(key(seed, layer, tensor), off, n, lo, hi, out.ctypes.data)
    return out


def normal_bf16(seed, layer, tensor, off, n, mu=0.0, sigma=1.0, out=None):
    """bf16 bit patterns (uint16) of mu + sigma*N(0,1)."""
    out = np.empty(n, np.uint16) if out is None else out
    assert out.flags.c_contiguous
    lib().sg_fill_normal_bf16(key(seed, layer, tensor), off, n, mu, sigma, out.ctypes.data)
    return out


def uniform_int(seed, layer, tensor, off, n, bound):
    out = np.empty(n, np.int32)
    lib().sg_fill_uniform_int(key(seed, layer, tensor), off, n, bound, out.ctypes.data)
    return out


def zipf_log_prior(s, n):
    out = np.empty(n, np.float32)
    lib().sg_zipf_log_prior(s, n, out.ctypes.data)
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Workload:
    name: str
    K: int
    H: int
    E: int
    top_k: int
    I: int
    Is: int
    layers: int
    seed: int
    zipf_s: float = 0.0
    attention: bool = False
    n_q_heads: int = 32
    n_kv_heads: int = 8
    head_dim: int = 128
    ctx: int = 16384
    vocab: int = 151936
    routed_scale: float = 1.0

    @property
    def G(self) -> int:
        """Most distinct experts one call can select."""
        return min(self.E, self.K * self.top_k)


WORKLOADS = {
    "tiny": Workload("tiny", K=1, H=256, E=16, top_k=2, I=128, Is=0, layers=1, seed=0),
    "k2_layer": Workload("k2_layer", K=2, H=2048, E=256, top_k=8, I=512, Is=512, layers=1, seed=1),
    "k8_stack40": Workload("k8_stack40", K=8, H=2048, E=256, top_k=8, I=512, Is=512, layers=40, seed=2),
    "k16_zipf_stack40": Workload("k16_zipf_stack40", K=16, H=2048, E=256, top_k=8, I=512, Is=512,
                                 layers=40, seed=3, zipf_s=1.1),
    "k4_full_step": Workload("k4_full_step", K=4, H=2048, E=256, top_k=8, I=512, Is=512, layers=40,
                             seed=4, attention=True),
}


def nvfp4_bytes(rows: int, cols: int) -> int:
    """Bytes of one NVFP4 projection: codes + E4M3 scales + FP32 tensor scale."""
    return rows * cols // 2 + rows * cols // 16 + 4


@dataclass
class Proj:
    """One NVFP4 projection stack [n_exp][rows][cols] in host memory."""
    codes: np.ndarray   # uint8 [n_exp, rows, cols//2]; low nibble = even column
    scales: np.ndarray  # uint8 [n_exp, rows, cols//16]; E4M3 per 16 consecutive columns
    tscale: np.ndarray  # float32 [n_exp]


def make_proj(seed, layer, t_codes, t_scales, n_exp, rows, cols, experts=None) -> Proj:
    """Generate a projection stack; with ``experts`` only those experts are drawn
    (the others stay zero), using the same per-expert stream offsets."""
    cb, sb = rows * cols // 2, rows * cols // 16
    c = np.zeros((n_exp, rows, cols // 2), np.uint8)
    s = np.zeros((n_exp, rows, cols // 16), np.uint8)
    ids = range(n_exp) if experts is None else experts
    if experts is None:
        codes(seed, layer, t_codes, 0, n_exp * cb, c.reshape(-1))
        scales(seed, layer, t_scales, 0, n_exp * sb, s.reshape(-1))
    else:
        for e in ids:
            codes(seed, layer, t_codes, e * cb, cb, c[e].reshape(-1))
            scales(seed, layer, t_scales, e * sb, sb, s[e].reshape(-1))
    return Proj(c, s, np.ones(n_exp, np.float32))


@dataclass
class Layer:
    router_w: np.ndarray   # uint16 bf16 [E, H]
    router_b: np.ndarray   # float32 [E]
    gate: Proj
    up: Proj
    down: Proj
    sh_gate: Proj | None = None
    sh_up: Proj | None = None
    sh_down: Proj | None = None
    extra: dict = field(default_factory=dict)


def make_layer(w: Workload, layer: int, experts=None) -> Layer:
    s = w.seed
    rw = normal_bf16(s, layer, T_ROUTER_W, 0, w.E * w.H, 0.0, ROUTER_SIGMA).reshape(w.E, w.H)
    rb = zipf_log_prior(w.zipf_s, w.E) if w.zipf_s else np.zeros(w.E, np.float32)
    L = Layer(
        router_w=rw, router_b=rb,
        gate=make_proj(s, layer, T_GATE_C, T_GATE_S, w.E, w.I, w.H, experts),
        up=make_proj(s, layer, T_UP_C, T_UP_S, w.E, w.I, w.H, experts),
        down=make_proj(s, layer, T_DOWN_C, T_DOWN_S, w.E, w.H, w.I, experts),
    )
    if w.Is:
        L.sh_gate = make_proj(s, layer, T_SGATE_C, T_SGATE_S, 1, w.Is, w.H)
        L.sh_up = make_proj(s, layer, T_SUP_C, T_SUP_S, 1, w.Is, w.H)
        L.sh_down = make_proj(s, layer, T_SDOWN_C, T_SDOWN_S, 1, w.H, w.Is)
    return L


def make_x(w: Workload, instance: int = 0, K: int | None = None) -> np.ndarray:
    """Activation rows, bf16 N(0,1), [K, H]; ``instance`` selects a fresh draw."""
    K = w.K if K is None else K
    return normal_bf16(w.seed, instance, T_X, 0, K * w.H).reshape(K, w.H)


def make_attention(w: Workload, layer: int) -> dict:
    """bf16 attention weights N(0, 0.02) and a bf16 N(0,1) KV cache of w.ctx
    positions for one layer (no positional encoding)."""
    s, H, hd = w.seed, w.H, w.head_dim
    nq, nkv, C = w.n_q_heads, w.n_kv_heads, w.ctx
    return dict(
        Wq=normal_bf16(s, layer, T_ATT_Q, 0, nq * hd * H, 0.0, ROUTER_SIGMA).reshape(nq * hd, H),
        Wk=normal_bf16(s, layer, T_ATT_K, 0, nkv * hd * H, 0.0, ROUTER_SIGMA).reshape(nkv * hd, H),
        Wv=normal_bf16(s, layer, T_ATT_V, 0, nkv * hd * H, 0.0, ROUTER_SIGMA).reshape(nkv * hd, H),
        Wo=normal_bf16(s, layer, T_ATT_O, 0, H * nq * hd, 0.0, ROUTER_SIGMA).reshape(H, nq * hd),
        kc=normal_bf16(s, layer, T_KCACHE, 0, nkv * C * hd).reshape(nkv, C, hd),
        vc=normal_bf16(s, layer, T_VCACHE, 0, nkv * C * hd).reshape(nkv, C, hd),
    )


def make_lm_head(w: Workload) -> np.ndarray:
    return normal_bf16(w.seed, 0, T_LM_HEAD, 0, w.vocab * w.H, 0.0, ROUTER_SIGMA).reshape(w.vocab, w.H)


def make_drafts(w: Workload, target: np.ndarray, instance: int = 0):
    """Drafted tokens for a verify step: the target's token for the first j
    rows (j uniform in 0..K) and a different token afterwards, so the
    accepted prefix is exactly j.  Returns (draft int32 [K], j)."""
    K = target.shape[0]
    j = int(uniform_int(w.seed, instance, T_DRAFT_J, 0, 1, K + 1)[0])
    other = uniform_int(w.seed, instance, T_DRAFT_TOK, 0, K, w.vocab - 1)
    draft = np.where(np.arange(K) < j, target, (target.astype(np.int64) + 1 + other) % w.vocab).astype(np.int32)
    return draft, j


def make_coins(w: Workload, rounds: int, accept_pct: int = 75, instance: int = 0):
    """Per round and row: whether the synthetic drafter's token is the
    target's (probability accept_pct %), and the offset of its other token
    (uniform in 0 .. vocab-2).  Returns (coin uint8 [R][K], alt int32 [R][K])."""
    n = rounds * w.K
    coin = (uniform_int(w.seed, instance, T_COIN, 0, n, 100) < accept_pct).astype(np.uint8).reshape(rounds, w.K)
    alt = uniform_int(w.seed, instance, T_ALT, 0, n, w.vocab - 1).reshape(rounds, w.K)
    return coin, alt


# The Laguna layer schedule (README, "Why this challenge exists"): blocks of
# four layers, three sliding-window (512 positions, 64 q heads, RoPE theta
# 10000) then one full-attention (48 q heads, YaRN rotary on half the head
# dims); layer 0 a dense bf16 SwiGLU MLP of intermediate 8192, every other
# layer the MoE block.  YaRN factor and original context are readings:
# factor 4 over an original 4,096 positions (the workloads' 16,384-position
# context is four times that).
LAGUNA_WINDOW, LAGUNA_THETA = 512, 10000.0
LAGUNA_SLIDING_HEADS, LAGUNA_FULL_HEADS = 64, 48
LAGUNA_YARN_FACTOR, LAGUNA_YARN_ORIG = 4.0, 4096
LAGUNA_DENSE_INTER = 8192


def laguna_layer_kind(layer: int) -> dict:
    """Attention configuration of layer `layer`: n_q_heads, window,
    rotary_dim, rope_theta, yarn_factor, yarn_orig; and whether its MLP is
    the dense one."""
    full = layer % 4 == 3
    return dict(n_q_heads=LAGUNA_FULL_HEADS if full else LAGUNA_SLIDING_HEADS,
                window=0 if full else LAGUNA_WINDOW, rotary_dim=64 if full else 128, rope_theta=LAGUNA_THETA,
                yarn_factor=LAGUNA_YARN_FACTOR if full else 1.0, yarn_orig=LAGUNA_YARN_ORIG if full else 0,
                dense=layer == 0)


def make_dense_mlp(w: Workload, layer: int, inter: int = LAGUNA_DENSE_INTER) -> dict:
    s, H = w.seed, w.H
    return dict(Wg=normal_bf16(s, layer, T_MLP_G, 0, inter * H, 0.0, ROUTER_SIGMA).reshape(inter, H),
                Wu=normal_bf16(s, layer, T_MLP_U, 0, inter * H, 0.0, ROUTER_SIGMA).reshape(inter, H),
                Wd=normal_bf16(s, layer, T_MLP_D, 0, H * inter, 0.0, ROUTER_SIGMA).reshape(H, inter))
