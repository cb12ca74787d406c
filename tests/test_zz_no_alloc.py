"""moe_ffn_forward_noalloc: the layer without a caller workspace.

Callers that are handed only input and output buffers (a plug-in inside a host
program whose memory pool owns the device, or a loop that must not call anything
that may synchronise the device) cannot allocate the workspace moe_ffn_forward
needs; this entry point uses an 8 MiB device array held by the library instead.
The GPU test calls it through the C ABI twice in a row, compares both results with
moe_ffn_forward's on the same inputs within the layer tolerance, and reads the
device status word of each call through moe_noalloc_device_status.  This file is
collected last on purpose.
"""
import numpy as np
import pytest

import moe_inputs as mi
from gpu_util import TOL_RMS, cfg_for, moe_lib, need_gpu, upload

torch = pytest.importorskip("torch")

SPECS = [
    mi.small_spec("qwen", 256, 16, 4, 64, 64, 19, bias=("normal", 0.5)),
    mi.small_spec("gptoss", 256, 8, 2, 128, 0, 23, bias=("normal", 0.1)),
]


def test_noalloc_size_and_token_limits():
    """The array's size comes from the library, and the batch limits the header states
    (79 Qwen3.5-mini tokens, 76 gpt-oss-20b; 76 and 72 with the RMSNorm) are the last
    T whose workspace fits it."""
    moe = moe_lib()
    assert moe.NOALLOC_WORKSPACE_BYTES == moe.moe_noalloc_workspace_bytes() == 8 << 20
    for cfg, rms_norm, last in ((moe.qwen_cfg(), 0, 79), (moe.gptoss_cfg(), 0, 76),
                                (moe.qwen_cfg(), 1, 76), (moe.gptoss_cfg(), 1, 72)):
        c = cfg.replace(rms_norm=rms_norm, rms_eps=1e-6)
        assert moe.moe_workspace_bytes(c, last) <= moe.NOALLOC_WORKSPACE_BYTES
        assert moe.moe_workspace_bytes(c, last + 1) > moe.NOALLOC_WORKSPACE_BYTES


@pytest.mark.gpu
@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_noalloc_matches_forward_twice(spec):
    need_gpu()
    moe = moe_lib()
    lay = mi.make_layer(spec)
    x, router, experts, shared = upload(lay)
    for y_fp32 in (1, 0):
        c = cfg_for(spec, y_fp32=y_fp32)
        ref = moe.moe_ffn_forward(c, x, router, experts, shared).float().cpu().numpy()
        rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
        for _ in range(2):
            ids = torch.empty((spec.tokens, spec.top_k), dtype=torch.int32, device="cuda")
            y = moe.moe_ffn_forward_noalloc(c, x, router, experts, shared, topk_ids=ids)
            st, bits = moe.moe_noalloc_device_status()
            assert st == 0 and bits == 0, (st, bits)
            got = y.float().cpu().numpy()
            assert np.max(np.abs(got - ref)) <= TOL_RMS * rms
            assert ids.min().item() >= 0 and ids.max().item() < spec.n_experts


@pytest.mark.gpu
def test_noalloc_rejects_too_many_tokens():
    need_gpu()
    moe = moe_lib()
    spec = SPECS[1]
    c = cfg_for(spec)
    T = 1
    while moe.moe_workspace_bytes(c, T) <= moe.NOALLOC_WORKSPACE_BYTES:
        T *= 2
    lay = mi.make_layer(spec, T=T)
    x, router, experts, shared = upload(lay)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_ffn_forward_noalloc(c, x, router, experts, shared)
    assert e.value.status == -3
