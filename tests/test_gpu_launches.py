"""Which of the library's kernels one moe_ffn_forward launches, per kernel plan.

Parity alone cannot see a dispatch slip in which a fallback kernel recomputes what
another kernel already wrote (the results stay right, the time doubles), nor a silent
switch to another kernel family.  The CUDA kernels a call launches are recorded with
the PyTorch profiler and compared, as an ordered list of kernel names, with what the
plan prescribes.  Skipped when the profiler records no CUDA kernels on this machine.
"""
import re

import pytest
import torch

import moe_inputs as mi
from gpu_util import cfg_for, moe_lib, need_gpu, upload

pytestmark = pytest.mark.gpu

# (spec, cfg.path, plan, kernels of one call in launch order)
CASES = [
    (mi.small_spec("qwen", 96, 16, 4, 64, 64, 12, bias=("normal", 0.5)), 1, "DECODE_FUSED",
     ["router_logits_kernel", "select_permute_kernel", "experts_decode_fused_kernel", "combine_kernel"]),
    # more than 32 tokens: the select kernel, then the one-CTA grouping
    (mi.small_spec("qwen", 96, 64, 4, 64, 64, 40, bias=("normal", 0.5)), 1, "DECODE_FUSED",
     ["router_logits_kernel", "router_select_kernel", "permute_one_cta_kernel", "experts_decode_fused_kernel",
      "combine_kernel"]),
    (mi.small_spec("qwen", 128, 32, 4, 64, 64, 8, bias=("normal", 0.5)), 1, "DECODE_RING",
     ["router_logits_kernel", "select_permute_kernel", "ring_stream_kernel", "ring_stream_kernel",
      "combine_kernel"]),
    (mi.small_spec("gptoss", 256, 16, 2, 128, 0, 23, bias=("normal", 0.1)), 1, "DECODE_RING",
     ["router_logits_kernel", "select_permute_kernel", "fp4_stream_kernel", "fp4_stream_kernel",
      "combine_kernel"]),
    (mi.small_spec("qwen", 128, 16, 4, 64, 96, 200, bias=("normal", 0.5)), 1, "DECODE_WARP",
     ["router_logits_kernel", "router_select_kernel", "permute_one_cta_kernel", "gateup_decode_kernel",
      "down_decode_kernel", "combine_kernel"]),
    # prefill (cfg.path 2): the router as a dense GEMM past 256 tokens where it applies,
    # then the grouped GEMMs; the fixed-order combine (deterministic) or the finish of
    # the accumulated down projection
    (mi.small_spec("qwen", 256, 16, 4, 128, 128, 300, bias=("normal", 0.5)), 2, "PREFILL_BF16",
     ["grouped_gemm_kernel", "router_select_kernel", "permute_one_cta_kernel", "grouped_gemm_kernel",
      "grouped_gemm_kernel", "combine_kernel"]),
    (mi.small_spec("gptoss", 128, 4, 2, 128, 0, 600, bias=("normal", 0.1)), 2, "PREFILL_F16",
     ["router_logits_kernel", "router_select_kernel", "fp4_prep_kernel", "permute_one_cta_kernel",
      "gather_rows_f16_kernel", "fp4_gemm_kernel", "h_fix_f16_kernel", "fp4_gemm_kernel", "combine_kernel"]),
]
ACCUMULATED = [
    (mi.small_spec("qwen", 256, 16, 4, 128, 128, 300, bias=("normal", 0.5)), "PREFILL_BF16",
     ["grouped_gemm_kernel", "router_select_kernel", "permute_one_cta_kernel", "grouped_gemm_kernel",
      "grouped_gemm_kernel", "finish_kernel"]),
    (mi.small_spec("gptoss", 128, 4, 2, 128, 0, 600, bias=("normal", 0.1)), "PREFILL_F16",
     ["router_logits_kernel", "router_select_kernel", "fp4_prep_kernel", "permute_one_cta_kernel",
      "gather_rows_f16_kernel", "fp4_gemm_kernel", "h_fix_f16_kernel", "fp4_gemm_kernel", "finish_kernel"]),
]


@pytest.fixture(scope="module")
def profiler_ready():
    """One short profiling session first: the first session of a process can miss the
    kernels of its region while the profiler attaches."""
    need_gpu()
    from torch.profiler import ProfilerActivity, profile
    a = torch.ones(1 << 16, device="cuda")
    for _ in range(2):
        with profile(activities=[ProfilerActivity.CUDA]):
            a.mul_(1.0)
            torch.cuda.synchronize()


def _short(name):
    """The kernel's own name from the profiler's (demangled) signature."""
    m = re.search(r"(\w+)(?:<[^()]*>)?\(", name)
    return m.group(1) if m else name


def _launched(moe, c, spec):
    """The ordered kernel names of one moe_ffn_forward (after a first, untimed call)."""
    x, router, experts, shared = upload(mi.make_layer(spec))
    ws = moe.workspace(c, spec.tokens)
    y = torch.empty_like(x)
    moe.moe_ffn_forward(c, x, router, experts, shared, y=y, ws=ws)      # first call: attributes set
    torch.cuda.synchronize()
    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        moe.moe_ffn_forward(c, x, router, experts, shared, y=y, ws=ws)
        torch.cuda.synchronize()
    assert moe.moe_device_status(ws)[0] == 0
    evs = [e for e in prof.events() if getattr(e, "device_type", None) is not None
           and str(e.device_type).endswith("CUDA")]
    if not evs:
        pytest.skip("the profiler recorded no CUDA kernels here")
    evs.sort(key=lambda e: e.time_range.start)
    got = [_short(e.name) for e in evs]
    return [k for k in got if k.endswith("_kernel") and not k.startswith(("vectorized", "elementwise"))], got


@pytest.mark.parametrize("spec,path,plan,want", CASES,
                         ids=["fused-bf16", "fused-bf16-40-tokens", "ring-bf16", "ring-mxfp4", "warp-four-chunks",
                              "prefill-bf16", "prefill-f16"])
def test_kernels_launched_per_plan(spec, path, plan, want, profiler_ready):
    moe = moe_lib()
    c = cfg_for(spec, path=path)
    assert moe.moe_kernel_plan(c, spec.tokens) == getattr(moe, "PLAN_" + plan)
    ours, got = _launched(moe, c, spec)
    assert ours == want, (plan, got)


@pytest.mark.parametrize("spec,plan,want", ACCUMULATED, ids=["prefill-bf16", "prefill-f16"])
def test_kernels_launched_accumulated_prefill(spec, plan, want, profiler_ready):
    """The library default (cfg.deterministic = 0): the down projection accumulates and
    the finish kernel rounds, with no combine."""
    moe = moe_lib()
    c = cfg_for(spec, path=2, deterministic=0)
    assert moe.moe_kernel_plan(c, spec.tokens) == getattr(moe, "PLAN_" + plan)
    ours, got = _launched(moe, c, spec)
    assert ours == want, (plan, got)
