"""C-ABI host checks that need no GPU: the library loads, exports every function the
header declares, and rejects bad arguments before touching the device."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT

torch = pytest.importorskip("torch")
moe = pytest.importorskip("sparse_moe_ffn_route_gb300")


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, re.M):
            names.add(m.group(1))
    return names


def test_every_declared_function_is_exported():
    names = declared_functions()
    assert {"moe_route", "moe_ffn_forward", "moe_workspace_bytes"} <= names
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert names == set(moe.EXPORTED)


def test_workspace_and_path_queries():
    q = moe.qwen_cfg()
    assert moe.moe_workspace_bytes(q, 0) > 0
    assert moe.moe_workspace_bytes(q, 64) > moe.moe_workspace_bytes(q, 8)
    assert moe.moe_select_path(q, 8) == moe.PATH_DECODE
    assert moe.moe_select_path(q, 4096) == moe.PATH_PREFILL
    g = moe.gptoss_cfg()
    assert moe.moe_select_path(g, 32) == moe.PATH_DECODE
    assert moe.moe_select_path(g, 8192) == moe.PATH_PREFILL
    assert moe.moe_select_path(g.replace(path=moe.PATH_DECODE), 8192) == moe.PATH_DECODE


def test_kernel_plan_per_workload():
    """The kernel family each workload runs (a silent fallback to another family keeps
    results correct, so only this check would notice it)."""
    import moe_inputs as mi
    want = {
        "qwen35_mini_moe_decode_t8": moe.PLAN_DECODE_RING,
        "qwen35_mini_moe_decode_t64": moe.PLAN_DECODE_FUSED,
        "qwen35_mini_moe_prefill_t4096": moe.PLAN_PREFILL_BF16,
        "gptoss_20b_moe_decode_t32": moe.PLAN_DECODE_RING,
        "gptoss_20b_moe_prefill_t8192": moe.PLAN_PREFILL_F16,
    }
    assert set(want) == set(mi.WORKLOADS)
    for name, plan in want.items():
        spec = mi.WORKLOADS[name]
        if spec.family == "qwen":
            c = moe.qwen_cfg(spec.d_model, spec.n_experts, spec.top_k, spec.expert_ff, spec.shared_ff)
        else:
            c = moe.gptoss_cfg(spec.d_model, spec.n_experts, spec.top_k, spec.expert_ff)
        assert moe.moe_kernel_plan(c, spec.tokens) == plan, name


def test_kernel_plan_forms():
    g = moe.gptoss_cfg()
    # forced paths
    assert moe.moe_kernel_plan(g.replace(path=moe.PATH_PREFILL), 32) == moe.PLAN_PREFILL_F16
    assert moe.moe_kernel_plan(g.replace(path=moe.PATH_DECODE_REGISTERS), 32) == moe.PLAN_DECODE_WARP
    assert moe.moe_kernel_plan(g.replace(path=moe.PATH_DECODE), 8192) == moe.PLAN_DECODE_WARP  # 4-chunk items
    # a clamp limit too wide for an f16 h keeps the bf16-dequant GEMMs
    assert moe.moe_kernel_plan(g.replace(glu_limit=300.0), 8192) == moe.PLAN_PREFILL_BF16
    # shapes the tcgen05 tiles do not take fall back to the decode kernels
    q = moe.qwen_cfg(d_model=96, n_experts=8, top_k=2, expert_ff=32, shared_ff=0)
    assert moe.moe_kernel_plan(q, 4096) == moe.PLAN_DECODE_WARP
    # bf16 decode: the ring takes the separate gate / up layout with d, ff, sff
    # multiples of 64; otherwise (or when asked) the register-stream kernels, which
    # bf16 one-chunk items run as one launch
    assert moe.moe_kernel_plan(q, 4) == moe.PLAN_DECODE_FUSED                      # d = 96
    b = moe.qwen_cfg()
    assert moe.moe_kernel_plan(b, 8) == moe.PLAN_DECODE_RING
    assert moe.moe_kernel_plan(b, 64) == moe.PLAN_DECODE_FUSED      # many units: register stream
    assert moe.moe_kernel_plan(b.replace(path=moe.PATH_DECODE_REGISTERS), 8) == moe.PLAN_DECODE_FUSED
    assert moe.moe_kernel_plan(b.replace(interleaved_gate_up=1, shared_ff=0), 8) == moe.PLAN_DECODE_FUSED
    assert moe.moe_kernel_plan(b.replace(shared_ff=96), 8) == moe.PLAN_DECODE_FUSED
    # four-chunk items and MXFP4 keep two launches; so does the test hook
    assert moe.moe_kernel_plan(b.replace(path=moe.PATH_DECODE), 4096) == moe.PLAN_DECODE_WARP
    moe.moe_test_set_decode_fusion(False)
    try:
        assert moe.moe_kernel_plan(b, 64) == moe.PLAN_DECODE_WARP
    finally:
        moe.moe_test_set_decode_fusion(True)
    assert moe._lib.moe_test_set_decode_fusion(2) == -1
    assert moe._lib.moe_kernel_plan(ctypes.byref(moe.qwen_cfg()), -1) == -1


BAD_CFGS = [
    dict(top_k=0), dict(top_k=300), dict(n_experts=0), dict(n_experts=2000), dict(d_model=-1),
    dict(gating=2), dict(act=5), dict(wfmt=3), dict(path=7), dict(expert_weights_scale=float("nan")),
    dict(rms_norm=2), dict(residual=-1), dict(rms_eps=float("nan")), dict(rms_eps=-1e-6),
]


@pytest.mark.parametrize("kw", BAD_CFGS)
def test_invalid_cfg_rejected(kw):
    c = moe.qwen_cfg().replace(**kw)
    assert moe.moe_workspace_bytes(c, 8) == 0
    lib = moe._lib
    fake = ctypes.c_void_p(1 << 20)
    st = lib.moe_ffn_forward(ctypes.byref(c), fake, 8, None, None, None, fake, None, None, fake,
                             1 << 30, None)
    assert st == -1


def test_unsupported_shapes():
    def path(c):
        return moe._lib.moe_select_path(ctypes.byref(c), 8)
    assert path(moe.qwen_cfg(d_model=100)) == -2                    # d % 32
    assert path(moe.gptoss_cfg().replace(interleaved_gate_up=0)) == -2
    assert path(moe.gptoss_cfg().replace(shared_ff=32)) == -2
    assert path(moe.qwen_cfg().replace(reserved=(ctypes.c_int32 * 2)(1, 0))) == -1
    assert path(moe.qwen_cfg().replace(deterministic=2)) == -1
    with pytest.raises(moe.MoeError):
        moe.moe_select_path(moe.qwen_cfg(d_model=100), 8)


def _args(cfg, T, ws_bytes, x=1 << 20, y=2 << 20, ws=3 << 20):
    lib = moe._lib
    P = ctypes.c_void_p
    r = moe._Router(P(4 << 20).value, None)
    e = moe._Experts(gate=5 << 20, up=6 << 20, down=7 << 20)
    s = moe._Shared(8 << 20, 9 << 20, 10 << 20, 11 << 20)
    return lib, (ctypes.byref(cfg), P(x), T, ctypes.byref(r), ctypes.byref(e), ctypes.byref(s),
                 P(y), None, None, P(ws), ws_bytes, None)


def test_argument_errors_before_any_launch():
    c = moe.qwen_cfg()
    need = moe.moe_workspace_bytes(c, 64)
    lib, a = _args(c, 64, need - 1)
    assert lib.moe_ffn_forward(*a) == -3                   # workspace too small
    lib, a = _args(c, 64, need, x=(1 << 20) + 8)
    assert lib.moe_ffn_forward(*a) == -4                   # misaligned x
    lib, a = _args(c, 64, need, ws=(3 << 20) + 4)
    assert lib.moe_ffn_forward(*a) == -4                   # misaligned workspace
    lib, a = _args(c, -1, need)
    assert lib.moe_ffn_forward(*a) == -1                   # negative T
    lib, a = _args(c, 0, need)
    assert lib.moe_ffn_forward(*a) == 0                    # T == 0: no work, no launch
    assert lib.moe_ffn_forward(a[0], None, 0, None, None, None, None, None, None, None, 0,
                               None) == 0                  # ... even with NULL pointers
    lib, a = _args(c, 64, need)
    a = list(a)
    a[5] = None                                            # shared expert missing
    assert lib.moe_ffn_forward(*a) == -1
    assert lib.moe_ffn_forward(*_args(c.replace(y_fp32=2), 64, need)[1]) == -1
    assert lib.moe_topk_from_logits(ctypes.byref(c), None, 4, None, None, None) == -1
    assert lib.moe_mxfp4_to_bf16(ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), 4, 48,
                                 ctypes.c_void_p(3 << 20), None) == -2
    assert lib.moe_device_status(None, None, None) == -1


def test_status_strings():
    for st in range(-7, 1):
        assert moe.moe_status_string(st) != "unknown status"
    assert moe.moe_status_string(-99) == "unknown status"


def test_rms_norm_needs_the_norm_weight_and_a_router():
    """cfg.rms_norm without router.norm_w is an invalid argument; the routed entry point,
    which takes no router, does not support it (both checked before any launch)."""
    c = moe.qwen_cfg(64, 8, 2, 32, 32).replace(rms_norm=1, rms_eps=1e-6)
    fake = ctypes.c_void_p(1 << 20)
    r = moe._Router(fake, None, None)
    sh = moe._Shared(fake, fake, fake, fake)
    ex = moe._Experts(gate=fake, up=fake, down=fake)
    st = moe._lib.moe_ffn_forward(ctypes.byref(c), fake, 8, ctypes.byref(r), ctypes.byref(ex),
                                  ctypes.byref(sh), fake, None, None, fake, 1 << 30, None)
    assert st == -1
    st = moe._lib.moe_ffn_forward_routed(ctypes.byref(c), fake, 8, fake, fake, fake,
                                         ctypes.byref(ex), ctypes.byref(sh), fake, fake, 1 << 30, None)
    assert st == -2
    # the norm's input copy makes the workspace larger
    assert moe.moe_workspace_bytes(c, 64) > moe.moe_workspace_bytes(c.replace(rms_norm=0), 64)


def test_wait_limit_hook_rejects_bad_arguments():
    """The test hook for the bounded waits checks its arguments before any CUDA call."""
    assert moe._lib.moe_test_set_wait_limit(0, 0) == -1
    assert moe._lib.moe_test_set_wait_limit(1 << 20, 2) == -1
