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
    # a large skewed problem first (many chunks), then a small one: the second
    # call runs over the array as the first one left it
    cases = [(synth.PREFILL_BF16, 1), (synth.SMALL_BF16, 2)]
    for shape, seed in cases:
        small = synth.LayerShape(shape.name, shape.T, 128 if shape.D > 512 else shape.D, shape.E,
                                 128, shape.top_k, "bf16", shape.zipf_s)
        layer, v = _workspace_reference(small, seed)
        T, E, k = small.T, small.E, small.top_k
        out = _noalloc(v["blob"][0], T, E, k)
        torch.cuda.synchronize()
        for name in ("counts", "offsets", "tiles", "inv", "src_tok"):
            assert torch.equal(out[name], v[name]), name
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
