"""The expert-parallel layer's local expert step on the GPU.

The exchange of rows between ranks is tested on CPU ranks (test_expert_parallel.py).
Here two ranks' shares of the experts run one after the other on the one GPU, each
through library_local_experts (moe_ffn_forward_routed on that rank's slice of the
expert weights, one expert per row, weight 1, fp32 output); the rows they return,
put back in slot order and combined with the routing weights, must equal the
single-GPU layer's fp32 output to within fp32 rounding and the oracle to the layer
tolerance.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_util import TOL_RMS, cfg_for, check_y, moe_lib, need_gpu, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SPECS = [
    mi.small_spec("qwen", 256, 16, 4, 64, 0, 37, bias=("normal", 0.5)),
    mi.small_spec("gptoss", 256, 8, 2, 128, 0, 29, bias=("normal", 0.1)),
]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
@pytest.mark.parametrize("world", [2, 4])
def test_local_experts_of_each_rank_recombine_to_the_layer(spec, world):
    need_gpu()
    moe = moe_lib()
    from sparse_moe_ffn_route_gb300 import expert_parallel as ep
    lay = mi.make_layer(spec)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec, y_fp32=1)
    T, k, E, d = spec.tokens, spec.top_k, spec.n_experts, spec.d_model
    ids, w, _, _ = moe.moe_route(c, x, router, shared)
    y_layer = moe.moe_ffn_forward(c, x, router, experts, shared)
    owner = ep.owner_of(ids, E, world).reshape(-1)
    epr = E // world
    Y_slots = torch.full((T * k, d), float("nan"), dtype=torch.float32, device="cuda")
    for r in range(world):
        sel = (owner == r).nonzero().flatten()
        rows = x.index_select(0, torch.div(sel, k, rounding_mode="floor"))
        local_ids = (ids.reshape(-1)[sel].to(torch.int64) - r * epr).to(torch.int32)
        Y = ep.library_local_experts(c, experts, r, world)(rows, local_ids)
        assert Y.shape == (sel.numel(), d)
        Y_slots[sel] = Y
    torch.cuda.synchronize()
    assert torch.isfinite(Y_slots).all()
    y = ep.combine(Y_slots, w).cpu().numpy().astype(np.float64)
    ref_gpu = y_layer.cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref_gpu ** 2)))
    assert np.max(np.abs(y - ref_gpu)) <= 1e-4 * rms
    ref = oracle.forward(oracle.gating_for(spec), lay)
    tie = oracle.near_tie_tokens(ref.logits, ref.ids)
    assert np.array_equal(ids.cpu().numpy()[~tie], ref.ids[~tie])
    check_y(y[~tie], ref.y[~tie], f"{spec.name} world {world}")
    assert TOL_RMS == 2e-2
