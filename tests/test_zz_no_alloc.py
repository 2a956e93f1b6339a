"""The allocation-free permutation index entry point.

Some callers of this library cannot allocate device memory (a plugin whose
host framework owns every allocation, a serving loop that forbids cudaMalloc
after start-up).  moe_permute_index_noalloc serves them: it keeps its only
scratch in a static device array inside the library.  This file checks,
through the C ABI, that it produces exactly what the workspace-based
moe_permute produces, on two calls in a row (the second one after the array
holds the first call's contents), and that sizes beyond the array are
refused before any work.  It is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from sparse_moe_expert_02_gb300 import MoELayer, synth
from sparse_moe_expert_02_gb300 import _lib as L


def _workspace_reference(shape, seed):
    """Route and permute through the workspace entry points."""
    inp = synth.make_inputs(shape, seed=seed, device="cuda")
    layer = MoELayer.from_shape(shape, inp)
    layer.init_ws()
    layer.route(inp["x"])
    layer.permute(inp["x"])
    return layer, layer.views(shape.T)


def _noalloc(idx, T, E, k):
    out = {
        "counts": torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
        "offsets": torch.full((E + 2,), -7, dtype=torch.int32, device="cuda"),
        "tiles": torch.full((E + 2,), -7, dtype=torch.int32, device="cuda"),
        "inv": torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
        "src_tok": torch.full((T * k + T,), -7, dtype=torch.int32, device="cuda"),
    }
    st = L.moe_permute_index_noalloc(idx.contiguous(), T, E, k, out["counts"], out["offsets"], out["tiles"],
                                     out["inv"], out["src_tok"])
    assert st == L.MOE_OK, L.lib().moe_status_str(st)
    return out


@pytest.mark.gpu
def test_noalloc_matches_workspace_path_two_calls_in_a_row():
    # Calls in a row on one array: a large skewed problem (80 chunks of 1024
    # pairs x 512 experts of histograms), then a smaller chunked one (20
    # chunks x 64 experts) whose scan runs over the entries the first call
    # left behind, then one small enough for the single-block kernel.
    cases = [
        (synth.LayerShape("noalloc_T8192_E512_k10", 8192, 128, 512, 128, 10, "bf16", 1.2), 1),
        (synth.LayerShape("noalloc_T2000_E64_k10", 2000, 128, 64, 128, 10, "bf16", 1.0), 2),
        (synth.LayerShape("noalloc_T300_E32_k4", 300, 128, 32, 128, 4, "bf16", 1.2), 3),
    ]
    for shape, seed in cases:
        layer, v = _workspace_reference(shape, seed)
        T, E, k = shape.T, shape.E, shape.top_k
        out = _noalloc(v["blob"][0], T, E, k)
        torch.cuda.synchronize()
        for name in ("counts", "offsets", "tiles", "inv", "src_tok"):
            assert torch.equal(out[name], v[name]), (shape.name, name)
        layer.check()


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_scratch():
    T, E, k = 60000, 1024, 10      # 586 chunks x 1024 experts > 262144 entries
    idx = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    dummy = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = L.moe_permute_index_noalloc(idx, T, E, k, dummy, dummy, dummy, dummy, dummy)
    assert st == L.MOE_ERR_UNSUPPORTED
    st = L.moe_permute_index_noalloc(idx, 0, E, k, dummy, dummy, dummy, dummy, dummy)
    assert st == L.MOE_ERR_INVALID_ARG
