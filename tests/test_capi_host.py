"""The C-ABI library on the host (no GPU needed): it builds for sm_103a,
loads, exports every entry point include/moe_verify.h declares, and rejects
bad arguments before enqueuing anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def M():
    import __graft_entry__
    __graft_entry__.build()
    import moe_nvfp4_block_gb300 as M
    return M


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                                    src, flags=re.M))
    return names


def test_exports_every_declared_symbol(M):
    declared = _declared()
    assert {"moe_verify_layer", "moe_router_topk", "verify_accept_prefix"} <= declared
    lib = ctypes.CDLL(M.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert set(M.EXPORTS) == declared


def _layer(M, **kw):
    z = M.moe_nvfp4(16, 16, 16)
    base = dict(hidden=2048, n_experts=256, top_k=8, inter=512, shared_inter=512, routed_scale=1.0,
                router_w=16, router_bias=None, gate=z, up=z, down=z, sh_gate=z, sh_up=z, sh_down=z)
    base.update(kw)
    return M.moe_layer(**base)


def test_workspace_size_and_group_ints(M):
    L = _layer(M)
    lib = M.lib
    for K in (1, 2, 8, 16):
        n = lib.moe_verify_layer_workspace_size(ctypes.byref(L), K)
        assert n > 0 and n % 256 == 0
    assert lib.moe_verify_layer_workspace_size(ctypes.byref(L), 0) == 0
    assert lib.moe_verify_layer_workspace_size(ctypes.byref(L), 17) == 0
    assert M.moe_group_ints(2, 256, 8) == 2 + 2 * 16 + 16
    assert M.moe_group_ints(16, 8, 8) == 2 + 2 * 8 + 128


@pytest.mark.parametrize("kw,status", [
    (dict(hidden=1000), -2), (dict(hidden=4096), -2), (dict(inter=384), -2), (dict(shared_inter=256), -2),
    (dict(top_k=33), -2), (dict(top_k=0), -1), (dict(n_experts=2000), -2), (dict(router_w=None), -1),
    (dict(router_w=8), -4),
])
def test_bad_layers_rejected_on_host(M, kw, status):
    L = _layer(M, **kw)
    r = M.lib.moe_verify_layer(ctypes.byref(L), 16, 2, None, 16, None, None, None, 16, 1 << 30, None)
    assert r == status, (kw, r)


def test_bad_call_arguments_rejected_on_host(M):
    L = _layer(M)
    f = M.lib.moe_verify_layer
    assert f(ctypes.byref(L), 16, 0, None, 16, None, None, None, 16, 1 << 30, None) == -1   # K = 0
    assert f(ctypes.byref(L), 16, 17, None, 16, None, None, None, 16, 1 << 30, None) == -1  # K > 16
    assert f(ctypes.byref(L), None, 2, None, 16, None, None, None, 16, 1 << 30, None) == -1  # no input
    assert f(ctypes.byref(L), 24, 2, None, 16, None, None, None, 16, 1 << 30, None) == -4   # misaligned
    assert f(ctypes.byref(L), 16, 2, None, 16, None, None, None, 16, 100, None) == -3       # workspace
    assert M.lib.verify_accept_prefix(None, 16, 2, 16, None) == -1
    assert M.lib.verify_accept_prefix(16, 16, 2, None, None) == -1
    assert M.lib.verify_accept_prefix(16, 16, -1, 16, None) == -1
    # attention envelope: one query head (o-projection shorter than 256) is refused
    assert M.lib.moe_attention_workspace_size(16, 256, 1, 1, 128) == 0
    assert M.lib.moe_attention_workspace_size(4, 2048, 32, 8, 128) > 0
    for s in range(-6, 1):
        assert M.status_string(s) not in ("", "unknown status")


def test_host_pointer_refuses_unpinned_memory(M):
    # ordinary (pageable) host memory is not mapped into the device's
    # address space: refused with MOE_ERR_INVALID_ARG, the output untouched
    buf = ctypes.create_string_buffer(4096)
    dev = ctypes.c_void_p(12345)
    rc = M.lib.moe_host_pointer(ctypes.cast(buf, ctypes.c_void_p), ctypes.byref(dev))
    assert rc == M.MOE_ERR_INVALID_ARG
    assert dev.value == 12345
    assert M.lib.moe_host_pointer(None, ctypes.byref(dev)) == M.MOE_ERR_INVALID_ARG
