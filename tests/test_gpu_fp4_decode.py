"""MXFP4 decode kernels vs the fp64 oracle: scale ranges and token magnitudes (GPU only).

One-chunk MXFP4 decode items run with an f16 token operand: each staged token row
is scaled by a power of two.  The default kernels stream the weights through a
TMA-fed shared-memory ring and apply each block's E8M0 scale in fp32; the
register-stream kernels (MOE_PATH_DECODE_REGISTERS) decode a k group whose scales
all lie in [113, 140] with f16 arithmetic and any other group with the exact bf16
decode against a bf16 (hi, lo) split of the f16 tokens.  These cases put both kinds
of group in one layer, drive the per-token scaling to both ends, and run the
many-token (unstaged) kernels on the same scale ranges.
Source: "Phase 19: MoE - gpt-oss-20b", section 3 (MXFP4: E2M1 codes, one E8M0
scale per 32 inputs).
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_util import check_outputs, cfg_for, moe_lib, need_gpu, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()


def _run(spec, lay, path=1):
    """Forward through the decode path (path 1) and compare with the oracle."""
    moe = moe_lib()
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec, path=path)
    T, k = spec.tokens, spec.top_k
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ws = moe.workspace(c, T)
    y16 = moe.moe_ffn_forward(c, x, router, experts, shared, topk_ids=ids, ws=ws)
    y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), x, router, experts, shared, ws=ws)
    st, bits = moe.moe_device_status(ws)
    assert st == 0, bits
    ids_g = ids.cpu().numpy()
    diff = np.any(ids_g != ref.ids, axis=1)
    assert not np.any(diff & ~oracle.near_tie_tokens(ref.logits, ref.ids))
    if np.any(diff):
        ref = oracle.forward(g, lay, forced_ids=np.where(diff[:, None], ids_g, ref.ids))
    check_outputs(y32, y16, ref.y, spec.name)


# (spec, note): few tokens per expert -> one-chunk items with staged f16 token rows
STAGED_SPECS = [
    (mi.small_spec("gptoss", 96, 12, 4, 96, 0, 5, bias=("normal", 0.1), scale_lo=100,
                   scale_hi=150), "3 blocks per row: ragged k group, both group kinds"),
    (mi.small_spec("gptoss", 256, 8, 2, 192, 0, 7, scale_lo=110, scale_hi=134),
     "mostly fast groups, a few split ones"),
    (mi.small_spec("gptoss", 128, 16, 4, 64, 0, 3, bias=("normal", 0.1), scale_lo=129,
                   scale_hi=160), "all split groups, all two-multiply scales"),
    (mi.small_spec("gptoss", 320, 8, 4, 160, 0, 6, bias=("normal", 0.1), scale_lo=113,
                   scale_hi=140), "the fast range's two ends"),
    (mi.small_spec("gptoss", 640, 8, 4, 576, 0, 6, bias=("normal", 0.1), scale_lo=110,
                   scale_hi=140), "rows over 256 bytes: a last ring stage of one box"),
]


# path 1: one-chunk MXFP4 items stream their weights through the TMA-fed shared-memory
# ring; path 3 keeps every weight load in registers (the kernels above)
KERNELS = pytest.mark.parametrize("path", [1, 3], ids=["ring", "registers"])


@KERNELS
@pytest.mark.parametrize("spec,note", STAGED_SPECS, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_staged_scale_ranges(spec, note, path):
    assert 4 * spec.tokens * spec.top_k <= 16 * spec.n_experts     # one-chunk items
    _run(spec, mi.make_layer(spec), path)


@KERNELS
@pytest.mark.parametrize("shift", [-40, -14, 0, 17, 40])
def test_staged_token_magnitudes(shift, path):
    """x scaled by 2^shift (exact in bf16): the per-token f16 scaling must absorb it.

    The expert biases are zero, so that h (and y) follow x's magnitude down to
    2^-40 and the down kernel's token scaling is driven as far as the gate_up one's.
    """
    spec = mi.small_spec("gptoss", 128, 8, 2, 128, 0, 6, scale_lo=116, scale_hi=126)
    lay = mi.make_layer(spec)
    lay.gu_bias = np.zeros_like(lay.gu_bias)
    lay.dn_bias = np.zeros_like(lay.dn_bias)
    x = mi.bf16_to_f32(lay.x).astype(np.float64) * 2.0 ** shift
    x[1] = 0.0                                   # an all-zero token row
    x[2, 5] *= 2.0 ** 20                         # one large value among ordinary ones
    lay.x = mi.f64_to_bf16(x)
    _run(spec, lay, path)


@pytest.mark.parametrize("scale_lo,scale_hi", [(100, 150), (127, 140), (105, 128), (60, 130)])
def test_unstaged_scale_ranges(scale_lo, scale_hi):
    """Many tokens per expert (4 chunks of 8, token rows read from global memory)."""
    spec = mi.small_spec("gptoss", 128, 4, 2, 128, 0, 40, bias=("normal", 0.1),
                         scale_lo=scale_lo, scale_hi=scale_hi)
    assert 4 * spec.tokens * spec.top_k > 16 * spec.n_experts       # four-chunk items
    _run(spec, mi.make_layer(spec))


def test_decode_many_items_and_ragged_row_tiles():
    """Several items per expert and a ragged last 128-row tile of the down projection
    (d = 320)."""
    spec = mi.small_spec("gptoss", 320, 4, 2, 192, 0, 90, bias=("normal", 0.1))
    _run(spec, mi.make_layer(spec), 1)
