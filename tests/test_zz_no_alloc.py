"""The allocation-free entry point moe_verify_layer_static.

Some callers cannot allocate device memory (an engine whose allocator owns
the GPU, a decode loop that cannot afford cudaMalloc's implicit
synchronisation); for them the layer keeps its scratch in a fixed array
inside the library.  This checks, through the C ABI, that two calls in a row
give the same routing and outputs as moe_verify_layer with a caller-owned
workspace (within the layer's parity tolerance), and that a layer needing
more scratch than the array holds is refused.  This file is collected last
on purpose and does not depend on the other tests having run."""
import ctypes

import numpy as np
import pytest
import torch

import synthgen
from helpers import assert_parity, bf16_bits, to_dev_bf16, upload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["k2_layer", "k16_zipf_stack40"])
def test_static_scratch_matches_caller_workspace(cuda_ok, name):
    import moe_nvfp4_block_gb300 as M
    w = synthgen.WORKLOADS[name]
    dl = upload(synthgen.make_layer(w, 2), w)
    c = dl.c()
    stream = torch.cuda.current_stream()
    for call in range(2):
        x = to_dev_bf16(synthgen.make_x(w, 40 + call))
        res = to_dev_bf16(synthgen.make_x(w, 50 + call))
        outs = []
        for static in (True, False):
            y = torch.empty_like(x)
            idx = torch.empty((w.K, w.top_k), dtype=torch.int32, device="cuda")
            wt = torch.empty((w.K, w.top_k), dtype=torch.float32, device="cuda")
            grp = torch.empty(M.moe_group_ints(w.K, w.E, w.top_k), dtype=torch.int32, device="cuda")
            if static:
                st = M.lib.moe_verify_layer_static(ctypes.byref(c), x.data_ptr(), w.K, res.data_ptr(),
                                                   y.data_ptr(), idx.data_ptr(), wt.data_ptr(), grp.data_ptr(),
                                                   ctypes.c_void_p(stream.cuda_stream))
                assert st == M.MOE_OK, M.status_string(st)
            else:
                ws = M.workspace(dl, w.K)
                M.moe_verify_layer(dl, x, res, y, ws, idx, wt, grp)
            torch.cuda.synchronize()
            outs.append((bf16_bits(y), idx.cpu().numpy(), wt.cpu().numpy(), grp.cpu().numpy()))
        (ys, idxs, ws_, gs), (yr, idxr, wr, gr) = outs
        np.testing.assert_array_equal(idxs, idxr)
        np.testing.assert_array_equal(gs, gr)
        np.testing.assert_allclose(ws_, wr, rtol=4e-6, atol=1e-7)
        assert_parity(ys, yr, f"{name} static scratch, call {call}")


def test_static_scratch_refuses_oversized_layer(cuda_ok):
    import moe_nvfp4_block_gb300 as M
    # 1024 experts, top-32, K=16, hidden 2048, intermediate 512: more than 8 MiB of scratch
    L = M.moe_layer(2048, 1024, 32, 512, 512, 1.0, 16, None, *([M.moe_nvfp4(16, 16, 16)] * 6))
    assert M.lib.moe_verify_layer_workspace_size(ctypes.byref(L), 16) > (8 << 20)
    st = M.lib.moe_verify_layer_static(ctypes.byref(L), 16, 16, None, 16, None, None, None, None)
    assert st == M.MOE_ERR_WORKSPACE_TOO_SMALL
