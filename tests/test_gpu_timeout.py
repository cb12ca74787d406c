"""The give-up path of the bounded device waits.

Every mbarrier wait of the TMA-fed kernels polls a bounded number of times; on
give-up the CTA sets MOE_ERR_TIMEOUT in the device status word, drains the copies
and MMAs it has in flight, frees its TMEM and returns.  The test hook
moe_test_set_wait_limit shortens the poll limit and makes the producer of the CTA
that owns the first unit of work skip its first load, so that the wait for that load
runs out: in the prefill grouped GEMM (tcgen05, TMEM accumulators) and in the MXFP4
decode ring.  In the one-launch bf16 decode the first gate_up unit withholds its
item's count instead, so that the down units of that item wait in vain.  The call
must report MOE_ERR_TIMEOUT through moe_device_status, and the next, normal call on
the same context must run and match the oracle: TMEM was freed, the counters were
zeroed again and nothing was left waiting.  No GPU fault is involved: the skipped load
or count is simply never issued.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_util import cfg_for, check_outputs, moe_lib, need_gpu, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

STATUS_TIMEOUT = 1 << 8
SHORT_POLLS = 1 << 14

CASES = [
    # Qwen-style bf16 layer on the prefill path (router on warp MMAs: T <= 256)
    (mi.small_spec("qwen", 256, 16, 4, 128, 128, 200, bias=("normal", 0.5)), 2, "PREFILL_BF16"),
    # gpt-oss-style MXFP4 layer on the decode ring
    (mi.small_spec("gptoss", 256, 16, 2, 128, 0, 23, bias=("normal", 0.1)), 1, "DECODE_RING"),
    # Qwen-style bf16 layer on the one-launch decode (down units wait on item counts)
    (mi.small_spec("qwen", 96, 16, 4, 64, 64, 12, bias=("normal", 0.5)), 1, "DECODE_FUSED"),
]


@pytest.mark.parametrize("spec,path,plan", CASES, ids=lambda v: v if isinstance(v, str) else "")
def test_wait_gives_up_reports_timeout_and_recovers(spec, path, plan):
    need_gpu()
    moe = moe_lib()
    lay = mi.make_layer(spec)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec, path=path)
    T = spec.tokens
    assert moe.moe_kernel_plan(c, T) == getattr(moe, "PLAN_" + plan)
    ws = moe.workspace(c, T)
    try:
        moe.moe_test_set_wait_limit(SHORT_POLLS, True)
        moe.moe_ffn_forward(c, x, router, experts, shared, ws=ws)
        st, bits = moe.moe_device_status(ws)
    finally:
        moe.moe_test_set_wait_limit(moe.DEFAULT_WAIT_POLLS, False)
    assert st == -7, (st, bits)                       # MOE_ERR_TIMEOUT
    assert bits & STATUS_TIMEOUT
    # the same context afterwards: a normal call runs to the end and is right
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    y16 = moe.moe_ffn_forward(c, x, router, experts, shared, topk_ids=ids, ws=ws)
    y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), x, router, experts, shared, ws=ws)
    assert moe.moe_device_status(ws)[0] == 0
    ids_g = ids.cpu().numpy()
    diff = np.any(ids_g != ref.ids, axis=1)
    assert not np.any(diff & ~oracle.near_tie_tokens(ref.logits, ref.ids))
    if np.any(diff):
        ref = oracle.forward(g, lay, forced_ids=np.where(diff[:, None], ids_g, ref.ids))
    check_outputs(y32, y16, ref.y, f"after the timeout ({plan})")
