"""The allocation-free entry point moe_verify_layer_static.

Some callers cannot allocate device memory (an engine whose allocator owns
the GPU, a decode loop that cannot afford cudaMalloc's implicit
synchronisation); for them the layer keeps its scratch in a fixed array
inside the library.  Through the C ABI, two calls in a row must give exactly
the routing and outputs of moe_verify_layer with a caller-owned workspace:
both run the same deterministic kernel, so the results are compared bit for
bit (a race on the shared array would show up here).  The calls run on a
side stream (torch's pool streams do not wait for the legacy default
stream), so the one-time zero fill of the array must be ordered on the
caller's stream.  A layer needing more scratch than the array holds is
refused.  This file is collected last on purpose and does not depend on the
other tests having run."""
import ctypes

import numpy as np
import pytest
import torch

import synthgen
from helpers import bf16_bits, to_dev_bf16, upload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["k2_layer", "k16_zipf_stack40"])
def test_static_scratch_matches_caller_workspace(cuda_ok, name):
    import moe_nvfp4_block_gb300 as M
    w = synthgen.WORKLOADS[name]
    dl = upload(synthgen.make_layer(w, 2), w)
    c = dl.c()
    side = torch.cuda.Stream()
    ws = M.workspace(dl, w.K)
    for call in range(2):
        x = to_dev_bf16(synthgen.make_x(w, 40 + call))
        res = to_dev_bf16(synthgen.make_x(w, 50 + call))
        torch.cuda.synchronize()
        outs = []
        for static in (True, False):
            with torch.cuda.stream(side):
                y = torch.empty_like(x)
                idx = torch.empty((w.K, w.top_k), dtype=torch.int32, device="cuda")
                wt = torch.empty((w.K, w.top_k), dtype=torch.float32, device="cuda")
                grp = torch.empty(M.moe_group_ints(w.K, w.E, w.top_k), dtype=torch.int32, device="cuda")
                if static:
                    st = M.lib.moe_verify_layer_static(ctypes.byref(c), x.data_ptr(), w.K, res.data_ptr(),
                                                       y.data_ptr(), idx.data_ptr(), wt.data_ptr(),
                                                       grp.data_ptr(), ctypes.c_void_p(side.cuda_stream))
                    assert st == M.MOE_OK, M.status_string(st)
                else:
                    M.moe_verify_layer(dl, x, res, y, ws, idx, wt, grp, stream=side)
            side.synchronize()
            outs.append((bf16_bits(y), idx.cpu().numpy(), wt.cpu().numpy(), grp.cpu().numpy()))
        (ys, idxs, ws_, gs), (yr, idxr, wr, gr) = outs
        np.testing.assert_array_equal(idxs, idxr, err_msg=f"{name} call {call}: routing")
        np.testing.assert_array_equal(gs, gr, err_msg=f"{name} call {call}: grouping")
        np.testing.assert_array_equal(ws_.view(np.uint32), wr.view(np.uint32), err_msg=f"{name} call {call}: weights")
        np.testing.assert_array_equal(ys, yr, err_msg=f"{name} call {call}: y")
    assert M.moe_workspace_error(ws) == 0


def test_static_scratch_refuses_oversized_layer(cuda_ok):
    import moe_nvfp4_block_gb300 as M
    # 1024 experts, top-32, K=16, hidden 2048, intermediate 512: more than 8 MiB of scratch
    L = M.moe_layer(2048, 1024, 32, 512, 512, 1.0, 16, None, *([M.moe_nvfp4(16, 16, 16)] * 6))
    assert M.lib.moe_verify_layer_workspace_size(ctypes.byref(L), 16) > (8 << 20)
    st = M.lib.moe_verify_layer_static(ctypes.byref(L), 16, 16, None, 16, None, None, None, None)
    assert st == M.MOE_ERR_WORKSPACE_TOO_SMALL
