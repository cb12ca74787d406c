"""The benchmark's host-side accounting (CPU only): the launch counts it claims per
kernel plan, the algorithmic bytes and FLOPs of a step, and the roofline's choice of
bound.  The launch lists are the ones `tests/test_gpu_launches.py` records on the GPU.
"""
import sys
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_inputs as mi  # noqa: E402


@pytest.mark.parametrize("plan,mxfp4,slots,tokens,experts,want", [
    (5, False, 12 * 5, 12, 16, 4),        # router, select + grouping, fused experts, combine
    (5, False, 64 * 9, 64, 256, 5),       # router, select, grouping, fused experts, combine
    (2, False, 8 * 5, 8, 32, 5),          # router, select + grouping, two ring launches, combine
    (2, True, 23 * 2, 23, 16, 5),
    (1, False, 200 * 5, 200, 16, 6),      # router, select, grouping, gate_up, down, combine
    (3, False, 300 * 5, 300, 16, 6),      # router GEMM, select, grouping, two GEMMs, combine or finish
    (4, True, 600 * 2, 600, 4, 9),        # + scale prep, gather, h fix-up
])
def test_launches_per_step_match_the_recorded_lists(plan, mxfp4, slots, tokens, experts, want):
    assert bench.launches_per_step(plan, mxfp4, slots, tokens, experts) == want


def test_step_bytes_and_flops_of_the_headline_routing():
    """Qwen3.5-mini decode, T=64: gate_up and down bytes are the distinct routed experts'
    weights plus the shared expert's, x, h and Y; the one-launch record adds the two."""
    spec = mi.WORKLOADS["qwen35_mini_moe_decode_t64"]
    rng = np.random.default_rng(0)
    ids = np.stack([rng.choice(spec.n_experts, spec.top_k, replace=False) for _ in range(spec.tokens)])
    by, fl, distinct, per_unit = bench.work(spec, ids)
    d, ff, E, T, k = spec.d_model, spec.expert_ff, spec.n_experts, spec.tokens, spec.top_k
    assert distinct == len(np.unique(ids))
    gu_w = 2 * ff * d * 2
    dn_w = d * ff * 2
    assert per_unit == {"gate_up": gu_w, "down": dn_w}
    S = T * (k + 1)
    h = (T * k * ff + T * spec.shared_ff) * 2
    assert by["gate_up"] == distinct * gu_w + 2 * spec.shared_ff * d * 2 + T * d * 2 + h
    assert by["down"] == distinct * dn_w + d * spec.shared_ff * 2 + h + S * d * 4
    assert fl["gate_up"] == 2 * T * k * 2 * ff * d + 2 * T * 2 * spec.shared_ff * d
    assert fl["down"] == 2 * T * k * ff * d + 2 * T * spec.shared_ff * d


def test_roofline_takes_the_bound_of_the_ridge():
    hbm, tf = 6784.0, 1957.0
    mem = bench.kernel_roofline("k", 1e9, 1e10, 0.2, hbm, tf)          # 10 FLOP/B: below the ridge
    assert mem["bound"] == "hbm" and mem["peak"] == hbm
    assert mem["frac"] == pytest.approx(1e9 / 0.2e-3 / 1e9 / hbm)
    cmp_ = bench.kernel_roofline("k", 1e9, 1e12, 1.0, hbm, tf)        # 1000 FLOP/B: above it
    assert cmp_["bound"] == "tensor" and cmp_["peak"] == tf
    assert cmp_["frac"] == pytest.approx(1e12 / 1e-3 / 1e12 / tf)
