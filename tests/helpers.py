"""Test helpers: upload generated layers, parity metrics (tolerances of the
verify-layer contract: rel-L2 <= 5e-3 and max-abs <= 3e-2 * max|ref|)."""
import numpy as np

import synthgen

REL_L2 = 5e-3
MAX_ABS_FRAC = 3e-2


def upload(L: "synthgen.Layer", w: "synthgen.Workload", device="cuda", routed_scale=None, scoring=0):
    import moe_nvfp4_block_gb300 as M
    t = lambda p: (p.codes, p.scales, p.tscale)
    sh = None if L.sh_gate is None else (t(L.sh_gate), t(L.sh_up), t(L.sh_down))
    zero_bias = L.router_b is None or not np.any(L.router_b)
    return M.layer_from_arrays(L.router_w, None if zero_bias else L.router_b, t(L.gate), t(L.up), t(L.down), sh,
                               top_k=w.top_k, routed_scale=w.routed_scale if routed_scale is None else routed_scale,
                               device=device, scoring=scoring)


def bf16_bits(t):
    """torch bf16/int16 device tensor -> numpy uint16 bits."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_dev_bf16(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(device)


def parity(got_bits, ref_bits):
    g = synthgen.bf16_to_f32(got_bits).astype(np.float64)
    r = synthgen.bf16_to_f32(ref_bits).astype(np.float64)
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)
    mab = np.abs(g - r).max()
    return rel, mab, np.abs(r).max()


def assert_parity(got_bits, ref_bits, what=""):
    rel, mab, mref = parity(got_bits, ref_bits)
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    assert mab <= MAX_ABS_FRAC * mref, f"{what}: max-abs {mab:.3e} > {MAX_ABS_FRAC} * {mref:.3e}"
    return rel, mab
