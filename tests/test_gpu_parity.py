"""CUDA path vs the fp64 oracle, element by element, through the C ABI (GPU only)."""
import dataclasses

import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_util import (check_outputs, check_routing, check_y, cfg_for, is_exact, moe_lib, need_gpu,
                      same_bf16,
                      sample_tokens, upload, y_numpy)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()


# ----------------------------------------------------------------------------- MXFP4 decode
@pytest.mark.parametrize("scale", [0, 1, 100, 118, 122, 126, 127, 128, 129, 200, 254, 255])
def test_mxfp4_decode_bit_exact(scale):
    moe = moe_lib()
    rows, n_in = 6, 96
    blocks = mi.random_bytes(77 + scale, 0, (rows, n_in // 32, 16))
    blocks[0, 0, :] = np.arange(16, dtype=np.uint8) * 0x11      # every code, both nibbles
    scales = np.full((rows, n_in // 32), scale, np.uint8)
    scales[1, :] = [scale, 127, 1]
    ref = mi.f64_to_bf16(oracle.mxfp4_decode(blocks, scales))
    out = moe.moe_mxfp4_to_bf16(torch.from_numpy(blocks).cuda(), torch.from_numpy(scales).cuda())
    from sparse_moe_ffn_route_gb300.hostio import to_numpy_bf16
    got = to_numpy_bf16(out)
    nan = np.isnan(mi.bf16_to_f32(ref))
    assert np.array_equal(np.isnan(mi.bf16_to_f32(got)), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ----------------------------------------------------------------------------- top-k
def _logit_sets():
    rng = np.random.default_rng(11)
    yield "normal", rng.standard_normal((300, 256)).astype(np.float32)
    yield "ties", rng.choice(np.float32([-1, -0.0, 0, 0.5, 1]), size=(300, 256))
    yield "coarse", (np.round(rng.standard_normal((300, 32)) * 4) / 4).astype(np.float32)
    yield "wide", rng.standard_normal((64, 1024)).astype(np.float32) * 30
    yield "narrow", rng.standard_normal((70, 5)).astype(np.float32)


@pytest.mark.parametrize("gating,norm,scale", [(0, 1, 1.0), (0, 1, 2.5), (0, 0, 1.0), (1, 1, 1.0)])
def test_topk_from_logits_exact(gating, norm, scale):
    moe = moe_lib()
    for name, L in _logit_sets():
        T, E = L.shape
        for k in sorted({1, min(4, E), min(8, E), E if E <= 32 else 32}):
            c = moe.qwen_cfg(d_model=32, n_experts=E, top_k=k, expert_ff=32, shared_ff=0,
                             expert_weights_scale=scale, norm_topk_prob=norm).replace(gating=gating)
            ids, w = moe.moe_topk_from_logits(c, torch.from_numpy(L).cuda())
            g = oracle.Gating(32, E, k, 32, gating=gating, norm_topk_prob=norm, scale=scale)
            ids_o, w_o = oracle.route_from_logits(g, L.astype(np.float64))
            assert np.array_equal(ids.cpu().numpy(), ids_o), (name, k)
            assert np.allclose(w.cpu().numpy(), w_o, rtol=1e-5, atol=1e-7), (name, k)


# ----------------------------------------------------------------------------- router
ROUTE_SPECS = [
    mi.small_spec("qwen", 64, 8, 2, 32, 32, 33, bias=None),
    mi.small_spec("qwen", 128, 40, 6, 32, 64, 17, bias=("normal", 0.5)),
    mi.small_spec("gptoss", 96, 12, 3, 64, 0, 31, bias=("normal", 0.1)),
    # more than 256 tokens: the tensor-core logits GEMM, its k range cut into parts
    # (4 and 3 here) that the select kernel adds; with and without the shared gate
    mi.small_spec("qwen", 256, 32, 4, 32, 64, 300, bias=("normal", 0.5)),
    mi.small_spec("gptoss", 192, 16, 4, 64, 0, 520, bias=("normal", 0.1)),
    # enough m tiles for every SM: one part, still through the scratch
    mi.small_spec("qwen", 128, 16, 2, 32, 32, 19500, bias=("normal", 0.5)),
    # few tokens and experts: the warp-MMA logits kernel with d cut into parts (4 and
    # 5 here) that the select kernel adds, the shared-gate column included
    mi.small_spec("qwen", 2048, 64, 8, 32, 32, 8, bias=("normal", 0.5)),
    mi.small_spec("gptoss", 2880, 32, 4, 64, 0, 32, bias=("normal", 0.1)),
]


@pytest.mark.parametrize("spec", ROUTE_SPECS, ids=lambda s: s.name)
def test_route_matches_oracle(spec):
    moe = moe_lib()
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    ref = oracle.route(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec)
    T, E = spec.tokens, spec.n_experts
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    sgate = torch.empty(T, dtype=torch.float32, device="cuda") if spec.shared_ff else None
    ids, w, sg, lg = moe.moe_route(c, x, router, shared, sgate=sgate, logits=logits)
    L = lg.cpu().numpy()
    assert np.allclose(L, ref.logits, rtol=1e-5, atol=2e-5)
    check_routing(g, ids.cpu().numpy(), w.cpu().numpy(), L, ref, spec.name)
    if spec.shared_ff:
        assert np.allclose(sg.cpu().numpy(), ref.sgate, rtol=1e-5, atol=1e-6)


# ----------------------------------------------------------------------------- whole layer, small
def _interleaved_bf16(spec):
    """A bf16 layer in the interleaved gate_up layout with clamped GLU and biases."""
    lay = mi.make_layer(spec)
    E, ff, d = spec.n_experts, spec.expert_ff, spec.d_model
    gu = np.empty((E, 2 * ff, d), np.uint16)
    gu[:, 0::2], gu[:, 1::2] = lay.gate, lay.up
    lay.gate_up = gu
    lay.gate = lay.up = None
    rng = np.random.default_rng(5)
    lay.gu_bias = mi.f64_to_bf16(rng.standard_normal((E, 2 * ff)) * 0.5)
    lay.dn_bias = mi.f64_to_bf16(rng.standard_normal((E, d)) * 0.1)
    return lay


LAYER_SPECS = [
    mi.small_spec("qwen", 64, 8, 2, 32, 32, 1),
    mi.small_spec("qwen", 64, 8, 2, 32, 32, 3),
    mi.small_spec("qwen", 128, 16, 4, 64, 96, 33, bias=("normal", 0.5)),
    mi.small_spec("qwen", 96, 6, 6, 32, 0, 31),                                   # E == k
    mi.small_spec("qwen", 64, 8, 3, 32, 32, 40, expert_weights_scale=2.5),
    mi.small_spec("qwen", 64, 8, 3, 32, 32, 9, norm_topk_prob=0),
    mi.small_spec("gptoss", 64, 8, 2, 64, 0, 1, bias=("normal", 0.1)),
    mi.small_spec("gptoss", 96, 12, 4, 96, 0, 37, bias=("normal", 0.1)),
    mi.small_spec("gptoss", 160, 8, 2, 224, 0, 70, bias=("zipf", 1.1)),          # > 32 tokens/expert
    mi.small_spec("gptoss", 64, 4, 4, 32, 0, 19, bias=None, scale_lo=118, scale_hi=120),
]


@pytest.mark.parametrize("spec", LAYER_SPECS, ids=lambda s: s.name)
def test_layer_matches_oracle(spec):
    moe = moe_lib()
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec)
    T, k = spec.tokens, spec.top_k
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = moe.workspace(c, T)
    y16 = moe.moe_ffn_forward(c, x, router, experts, shared, topk_ids=ids, topk_w=w, ws=ws)
    y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), x, router, experts, shared, ws=ws)
    assert moe.moe_device_status(ws)[0] == 0
    ids_g = ids.cpu().numpy()
    diff = np.any(ids_g != ref.ids, axis=1)
    tie = oracle.near_tie_tokens(ref.logits, ref.ids)
    assert not np.any(diff & ~tie)
    if np.any(diff):
        ref = oracle.forward(g, lay, forced_ids=np.where(diff[:, None], ids_g, ref.ids))
    check_outputs(y32, y16, ref.y, spec.name)


# bf16 decode with few tokens per expert: the weights stream through the TMA-fed
# shared-memory ring (separate gate / up, d, ff, sff multiples of 64).  Cases: the
# shared expert with as many units as the routed ones, none, and fewer (ff 192, sff
# 128: the shared expert skips a unit); d = 192 leaves a half unit of down rows.
RING_SPECS = [
    mi.small_spec("qwen", 128, 32, 4, 64, 64, 8, bias=("normal", 0.5)),
    mi.small_spec("qwen", 256, 16, 2, 128, 0, 5),
    mi.small_spec("qwen", 192, 24, 3, 192, 128, 7, bias=("normal", 0.5)),
    mi.small_spec("qwen", 64, 64, 8, 64, 64, 11, bias=("normal", 0.5), expert_weights_scale=2.5),
]


@pytest.mark.parametrize("spec", RING_SPECS, ids=lambda s: s.name)
@pytest.mark.parametrize("path,fused", [(1, True), (3, True), (3, False)],
                         ids=["ring", "registers-one-launch", "registers-two-launches"])
def test_bf16_decode_ring(spec, path, fused):
    """The ring, and the register-stream kernels both as the fused launch (gate_up and
    down units in one grid, down waiting on per-item counters) and as two launches."""
    moe = moe_lib()
    T, k = spec.tokens, spec.top_k
    assert 4 * T * k <= 16 * spec.n_experts                      # one-chunk items
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec, path=path)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ws = moe.workspace(c, T)
    moe.moe_test_set_decode_fusion(fused)
    try:
        want = moe.PLAN_DECODE_RING if path == 1 else (moe.PLAN_DECODE_FUSED if fused else moe.PLAN_DECODE_WARP)
        assert moe.moe_kernel_plan(c, T) == want
        y16 = moe.moe_ffn_forward(c, x, router, experts, shared, topk_ids=ids, ws=ws)
        y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), x, router, experts, shared, ws=ws)
    finally:
        moe.moe_test_set_decode_fusion(True)
    assert moe.moe_device_status(ws)[0] == 0
    ids_g = ids.cpu().numpy()
    diff = np.any(ids_g != ref.ids, axis=1)
    assert not np.any(diff & ~oracle.near_tie_tokens(ref.logits, ref.ids))
    if np.any(diff):
        ref = oracle.forward(g, lay, forced_ids=np.where(diff[:, None], ids_g, ref.ids))
    check_outputs(y32, y16, ref.y, spec.name)


def test_interleaved_bf16_clamped_layer():
    moe = moe_lib()
    spec = mi.small_spec("qwen", 96, 8, 3, 64, 0, 29, bias=("normal", 0.3))
    lay = _interleaved_bf16(spec)
    g = oracle.Gating(96, 8, 3, 64, 0, gating=1, act=1, wfmt=0, interleaved=1)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = moe.qwen_cfg(96, 8, 3, 64, 0).replace(gating=1, act=1, interleaved_gate_up=1)
    ids = torch.empty((29, 3), dtype=torch.int32, device="cuda")
    y16 = moe.moe_ffn_forward(c, x, router, experts, None, topk_ids=ids)
    y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), x, router, experts, None)
    assert np.array_equal(ids.cpu().numpy(), ref.ids)
    check_outputs(y32, y16, ref.y, "interleaved bf16")


@pytest.mark.parametrize("family", ["qwen", "gptoss"])
def test_forced_routing_hot_expert_and_duplicates(family):
    """Every token sends all k slots to experts {3, 3, 1, ...}: one expert gets 2T rows."""
    moe = moe_lib()
    spec = (mi.small_spec("qwen", 64, 8, 3, 32, 32, 45) if family == "qwen"
            else mi.small_spec("gptoss", 64, 8, 3, 64, 0, 45, bias=("normal", 0.1)))
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    T = spec.tokens
    forced = np.tile(np.array([3, 3, 1], np.int32), (T, 1))
    forced[::5, 2] = 7
    ref = oracle.forward(g, lay, forced_ids=forced)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec)
    sg = torch.from_numpy(ref.sgate.astype(np.float32)).cuda() if spec.shared_ff else None
    ids_d = torch.from_numpy(forced).cuda()
    w_d = torch.from_numpy(ref.w.astype(np.float32)).cuda()
    y16 = moe.moe_ffn_forward_routed(c, x, ids_d, w_d, experts, shared, sgate=sg)
    y32 = moe.moe_ffn_forward_routed(c.replace(y_fp32=1), x, ids_d, w_d, experts, shared, sgate=sg)
    check_outputs(y32, y16, ref.y, family)


# The one-launch bf16 decode (gate_up and down units in one grid, down waiting on its
# item's count) at its edges: one token; a shared expert wider than the routed ones
# (the routed items' extra gate_up units do no work but still count); d over one
# 128-row tile with no shared expert (the last down tile ragged).
FUSED_EDGE = [
    mi.small_spec("qwen", 96, 16, 4, 64, 64, 1, bias=("normal", 0.5)),
    mi.small_spec("qwen", 96, 16, 4, 64, 160, 9, bias=("normal", 0.5)),
    mi.small_spec("qwen", 160, 64, 4, 96, 0, 16, bias=("normal", 0.5)),
]


@pytest.mark.parametrize("spec", FUSED_EDGE, ids=lambda s: s.name)
def test_one_launch_decode_edges(spec):
    moe = moe_lib()
    T, k = spec.tokens, spec.top_k
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec)
    assert moe.moe_kernel_plan(c, T) == moe.PLAN_DECODE_FUSED
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ws = moe.workspace(c, T)
    y16 = moe.moe_ffn_forward(c, x, router, experts, shared, topk_ids=ids, ws=ws)
    y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), x, router, experts, shared, ws=ws)
    assert moe.moe_device_status(ws)[0] == 0
    ids_g = ids.cpu().numpy()
    diff = np.any(ids_g != ref.ids, axis=1)
    assert not np.any(diff & ~oracle.near_tie_tokens(ref.logits, ref.ids))
    if np.any(diff):
        ref = oracle.forward(g, lay, forced_ids=np.where(diff[:, None], ids_g, ref.ids))
    check_outputs(y32, y16, ref.y, spec.name)


def test_one_launch_decode_hot_expert_and_duplicates():
    """Every token sends two slots to expert 3 (32 rows: four items of one expert) and
    one each to experts 1 and 5 or 9, through the one-launch decode."""
    moe = moe_lib()
    spec = mi.small_spec("qwen", 96, 64, 4, 64, 64, 16)
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    T = spec.tokens
    forced = np.tile(np.array([3, 3, 1, 5], np.int32), (T, 1))
    forced[::3, 3] = 9
    ref = oracle.forward(g, lay, forced_ids=forced)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec)
    assert moe.moe_kernel_plan(c, T) == moe.PLAN_DECODE_FUSED
    sg = torch.from_numpy(ref.sgate.astype(np.float32)).cuda()
    ids_d = torch.from_numpy(forced).cuda()
    w_d = torch.from_numpy(ref.w.astype(np.float32)).cuda()
    ws = moe.workspace(c, T)
    y16 = moe.moe_ffn_forward_routed(c, x, ids_d, w_d, experts, shared, sgate=sg, ws=ws)
    y32 = moe.moe_ffn_forward_routed(c.replace(y_fp32=1), x, ids_d, w_d, experts, shared, sgate=sg, ws=ws)
    assert moe.moe_device_status(ws)[0] == 0
    check_outputs(y32, y16, ref.y, "one launch, hot expert")


def test_bad_ids_are_flagged_not_faulting():
    moe = moe_lib()
    spec = mi.small_spec("qwen", 64, 8, 2, 32, 32, 6)
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec)
    ids = ref.ids.copy()
    ids[2, 1] = 99
    ids[4, 0] = -3
    ws = moe.workspace(c, 6)
    y = moe.moe_ffn_forward_routed(c.replace(y_fp32=1), x, torch.from_numpy(ids).cuda(),
                                   torch.from_numpy(ref.w.astype(np.float32)).cuda(), experts,
                                   shared, sgate=torch.from_numpy(ref.sgate.astype(np.float32)).cuda(),
                                   ws=ws)
    st, bits = moe.moe_device_status(ws)
    assert st == -6 and bits & 1
    good = [0, 1, 3, 5]
    check_y(y.cpu().numpy().astype(np.float64)[good], ref.y[good], "unaffected tokens")
    assert moe.moe_device_status(ws)[0] == 0            # cleared by the read


def test_deterministic_and_stream_ordered():
    moe = moe_lib()
    spec = mi.small_spec("gptoss", 128, 16, 4, 128, 0, 200, bias=("zipf", 1.1))
    lay = mi.make_layer(spec)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ws = moe.workspace(c, 200)
        ys = [moe.moe_ffn_forward(c, x, router, experts, shared, ws=ws).clone() for _ in range(4)]
    s.synchronize()
    for yy in ys[1:]:
        assert torch.equal(yy.view(torch.int16), ys[0].view(torch.int16))


def test_zero_tokens():
    moe = moe_lib()
    c = moe.qwen_cfg(64, 8, 2, 32, 32)
    spec = mi.small_spec("qwen", 64, 8, 2, 32, 32, 0)
    lay = mi.make_layer(spec)
    x, router, experts, shared = upload(lay)
    y = moe.moe_ffn_forward(c, x, router, experts, shared)
    assert y.shape == (0, 64)


# ----------------------------------------------------------------------------- full-size workloads
@pytest.fixture(scope="module")
def full_layers():
    cache = {}

    def get(name):
        if name not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            spec = mi.WORKLOADS[name]
            lay = mi.make_layer(spec)
            cache[name] = (spec, lay, upload(lay))
        return cache[name]
    return get


def item_rows(slot_expert: np.ndarray, E1: int, rows_per_item: int):
    """The grouping the library uses, from the slots' experts alone: the permute is
    stable, so expert v's rows are its slots in increasing slot order, cut into work
    items of rows_per_item.  Returns {(v, item): slots of that item}."""
    items = {}
    for v in range(E1):
        sl = np.nonzero(slot_expert == v)[0]
        for i in range(0, len(sl), rows_per_item):
            items[(v, i // rows_per_item)] = sl[i:i + rows_per_item]
    return items


def full_sample(name, spec, ids_g, c):
    """Tokens whose outputs are checked against the oracle at full size: every token of
    the Qwen3.5-mini prefill batch (about 6 s of oracle time on 16 cores) and of the
    decode batches; for gpt-oss-20b prefill, the last row of every (expert, work item)
    -- the ragged end of each cold expert's items included -- plus a few others."""
    moe = moe_lib()
    T, k = spec.tokens, spec.top_k
    if spec.family == "qwen" or T <= 64:
        return np.arange(T, dtype=np.int32)
    plan = moe.moe_kernel_plan(c, T)
    rows = {moe.PLAN_PREFILL_F16: 256, moe.PLAN_PREFILL_BF16: 128}.get(plan, 8)
    items = item_rows(ids_g.reshape(-1), spec.n_experts, rows)
    tok = {int(sl[-1]) // k for sl in items.values()}
    tok |= set(sample_tokens(T, 24).tolist())
    return np.array(sorted(tok), dtype=np.int32)


def test_headline_decode_one_launch_equals_two(full_layers):
    """The Qwen3.5-mini T=64 decode batch (221 routed experts, the shared expert's 8
    items): gate_up and down as one launch give the bits of the two-launch form, and
    repeated calls (each zeroing the launch's counters in its grouping) give them again."""
    moe = moe_lib()
    spec, lay, (x, router, experts, shared) = full_layers("qwen35_mini_moe_decode_t64")
    c = cfg_for(spec).replace(y_fp32=1)
    T = spec.tokens
    ws = moe.workspace(c, T)
    assert moe.moe_kernel_plan(c, T) == moe.PLAN_DECODE_FUSED
    y1 = moe.moe_ffn_forward(c, x, router, experts, shared, ws=ws)
    moe.moe_test_set_decode_fusion(False)
    try:
        assert moe.moe_kernel_plan(c, T) == moe.PLAN_DECODE_WARP
        y2 = moe.moe_ffn_forward(c, x, router, experts, shared, ws=ws)
    finally:
        moe.moe_test_set_decode_fusion(True)
    assert moe.moe_device_status(ws)[0] == 0
    assert torch.equal(y1, y2)
    for _ in range(3):
        assert torch.equal(moe.moe_ffn_forward(c, x, router, experts, shared, ws=ws), y1)
    assert moe.moe_device_status(ws)[0] == 0


@pytest.mark.parametrize("name", mi.WORKLOAD_ORDER)
def test_full_workload(name, full_layers):
    """Every workload at full size in the benchmark's configuration (the library's
    defaults: the accumulated prefill)."""
    moe = moe_lib()
    spec, lay, (x, router, experts, shared) = full_layers(name)
    g = oracle.gating_for(spec)
    c = cfg_for(spec, deterministic=0)
    T, k = spec.tokens, spec.top_k
    exact = is_exact(c, T)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = moe.workspace(c, T)
    y = moe.moe_ffn_forward(c, x, router, experts, shared, topk_ids=ids, topk_w=w, ws=ws)
    y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), x, router, experts, shared, ws=ws)
    assert moe.moe_device_status(ws)[0] == 0
    # routing of every token
    logits = torch.empty((T, spec.n_experts), dtype=torch.float32, device="cuda")
    ids2, w2, _, _ = moe.moe_route(c, x, router, shared, logits=logits)
    assert torch.equal(ids2, ids) and torch.equal(w2, w)
    ref_r = oracle.route(g, lay)
    tie, diff = check_routing(g, ids.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy(), ref_r,
                              name)
    # outputs against the oracle (near-tie tokens re-scored with the GPU's selection)
    tok = full_sample(name, spec, ids.cpu().numpy(), c)
    ids_g = ids.cpu().numpy()[tok]
    ref = oracle.forward(g, lay, tokens=tok, forced_ids=ids_g)
    sel = torch.from_numpy(tok).long().cuda()
    err, rms = check_outputs(y32[sel], y[sel], ref.y, name, exact=exact)
    # the bf16 output the benchmark times, against the bar as written
    err16, _ = check_y(y_numpy(y)[tok], ref.y, name + " (bf16 output)")
    print(f"{name}: {len(tok)} of {T} tokens checked, max|dy| fp32 {err / rms:.2e} rms, "
          f"bf16 {err16 / rms:.2e} rms, near-ties {int(tie.sum())}")
    # the host-buffer entry point gives the same result: pageable y (device buffer and
    # a copy) and page-locked y (written by the last kernel across the host link)
    xh = x.cpu().pin_memory()
    yh = moe.moe_ffn_forward_host(c, xh, router, experts, shared, ws=ws)
    same_bf16(yh, y, exact, "pageable y")
    yp = torch.full_like(yh, float("nan")).pin_memory()
    moe.moe_ffn_forward_host(c, xh, router, experts, shared, y_host=yp, ws=ws)
    same_bf16(yp, y, exact, "page-locked y")
    yp32 = torch.full((T, spec.d_model), float("nan"), dtype=torch.float32).pin_memory()
    moe.moe_ffn_forward_host(c.replace(y_fp32=1), xh, router, experts, shared, y_host=yp32, ws=ws)
    if exact:
        assert torch.equal(yp32, y32.cpu())
    else:
        assert float((yp32 - y32.cpu()).abs().max()) <= 2e-5 * rms
    # page-locked but not 16-byte aligned: the staged copy
    buf = torch.full((T * spec.d_model + 1,), float("nan"), dtype=torch.bfloat16).pin_memory()
    yu = buf[1:].view(T, spec.d_model)
    moe.moe_ffn_forward_host(c, xh, router, experts, shared, y_host=yu, ws=ws)
    same_bf16(yu, y, exact, "unaligned y")
    # the bound call: the same step, x_host's contents read at each call
    yb = torch.full((T, spec.d_model), float("nan"), dtype=torch.bfloat16).pin_memory()
    step = moe.BoundForwardHost(c, xh, router, experts, shared, y_host=yb, ws=ws)
    assert step() is yb
    same_bf16(yb, y, exact, "bound call")
    x0 = xh.clone()
    xh.zero_()
    step()
    same_bf16(yb, moe.moe_ffn_forward_host(c, xh, router, experts, shared, ws=ws), exact, "bound call, x = 0")
    xh.copy_(x0)


def test_host_entry_graph_cache():
    """Page-locked host buffers: the host entry replays a cached graph per argument set.
    Six sets (more than the four graphs kept) called in turn, twice, with new x each time,
    give what the device-resident forward gives for the same x."""
    moe = moe_lib()
    spec = mi.small_spec("qwen", 256, 16, 4, 64, 64, 24, bias=("normal", 0.5))
    lay = mi.make_layer(spec)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec)
    T, d = spec.tokens, spec.d_model
    ws = moe.workspace(c, T)
    xh = torch.empty((T, d), dtype=torch.bfloat16).pin_memory()
    ys = [torch.empty((T, d), dtype=torch.bfloat16).pin_memory() for _ in range(6)]
    for rep in range(2):
        for i, yh in enumerate(ys):
            xs = mi.make_x(dataclasses.replace(spec, seed=spec.seed + 31 * i + 7 * rep), T)
            xh.copy_(torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16))
            moe.moe_ffn_forward_host(c, xh, router, experts, shared, y_host=yh, ws=ws)
            want = moe.moe_ffn_forward(c, xh.cuda(), router, experts, shared, ws=ws)
            assert torch.equal(yh.view(torch.int16), want.cpu().view(torch.int16)), (rep, i)


# ----------------------------------------------------------------------------- prefill (tcgen05) path
PREFILL_SPECS = [
    mi.small_spec("qwen", 128, 8, 2, 64, 64, 200),
    mi.small_spec("qwen", 256, 16, 4, 128, 128, 300, bias=("normal", 0.5)),
    mi.small_spec("qwen", 512, 8, 3, 256, 0, 333, expert_weights_scale=1.5),
    mi.small_spec("qwen", 192, 4, 4, 320, 64, 129),                            # E == k, N 192
    mi.small_spec("gptoss", 128, 8, 2, 128, 0, 200, bias=("zipf", 1.1)),
    mi.small_spec("gptoss", 320, 4, 2, 192, 0, 150, bias=("normal", 0.1)),      # N 192 / 160
    mi.small_spec("gptoss", 256, 16, 4, 256, 0, 300, bias=("normal", 0.1), scale_lo=118,
                  scale_hi=120),
]


# (path, deterministic): decode; prefill with the fixed-order combine; prefill with the
# down projection accumulating into per-token sums
PATH_MODES = [(1, 1), (2, 1), (2, 0)]
PATH_MODE_IDS = ["decode", "prefill", "prefill-accumulated"]


@pytest.mark.parametrize("spec", PREFILL_SPECS, ids=lambda s: s.name)
@pytest.mark.parametrize("path,det", PATH_MODES, ids=PATH_MODE_IDS)
def test_layer_paths_match_oracle(spec, path, det):
    moe = moe_lib()
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec, path=path, deterministic=det)
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
    check_outputs(y32, y16, ref.y, f"{spec.name} path {path}", exact=is_exact(c, T))


@pytest.mark.parametrize("spec", PREFILL_SPECS[:2] + PREFILL_SPECS[4:6], ids=lambda s: s.name)
def test_accumulated_prefill_agrees_with_fixed_order(spec):
    """The down projection's atomic per-token sums and the fixed-order gather add the
    same fp32 terms: their fp32 outputs differ only by the rounding of the order."""
    moe = moe_lib()
    lay = mi.make_layer(spec)
    x, router, experts, shared = upload(lay)
    T = spec.tokens
    outs = []
    for det in (1, 0, 0):
        c = cfg_for(spec, path=moe.PATH_PREFILL, deterministic=det, y_fp32=1)
        ws = moe.workspace(c, T)
        ws.fill_(0xFF)                 # scratch starts as garbage: nothing may rely on zeros
        outs.append(moe.moe_ffn_forward(c, x, router, experts, shared, ws=ws).cpu().numpy())
        assert moe.moe_device_status(ws)[0] == 0
    ref = outs[0].astype(np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    for o in outs[1:]:
        assert np.all(np.isfinite(o))
        assert np.max(np.abs(o - ref)) <= 2e-5 * rms


def test_prefill_interleaved_bf16_clamped():
    moe = moe_lib()
    spec = mi.small_spec("qwen", 128, 8, 2, 192, 0, 150, bias=("normal", 0.3))
    lay = _interleaved_bf16(spec)
    g = oracle.Gating(128, 8, 2, 192, 0, gating=1, act=1, wfmt=0, interleaved=1)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = moe.qwen_cfg(128, 8, 2, 192, 0).replace(gating=1, act=1, interleaved_gate_up=1,
                                                 path=moe.PATH_PREFILL)
    ids = torch.empty((150, 2), dtype=torch.int32, device="cuda")
    y16 = moe.moe_ffn_forward(c, x, router, experts, None, topk_ids=ids)
    y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), x, router, experts, None)
    ids_g = ids.cpu().numpy()
    diff = np.any(ids_g != ref.ids, axis=1)
    assert not np.any(diff & ~oracle.near_tie_tokens(ref.logits, ref.ids))
    if np.any(diff):
        ref = oracle.forward(g, lay, forced_ids=np.where(diff[:, None], ids_g, ref.ids))
    check_outputs(y32, y16, ref.y, "prefill interleaved bf16")


@pytest.mark.parametrize("det", [1, 0], ids=["fixed-order", "accumulated"])
def test_prefill_hot_expert_many_tiles(det):
    """Forced routing: every token's two slots go to experts 5 and 2 (> 2 m tiles each)."""
    moe = moe_lib()
    spec = mi.small_spec("qwen", 128, 8, 2, 64, 64, 300)
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    forced = np.tile(np.array([5, 2], np.int32), (300, 1))
    forced[::7] = [2, 7]
    ref = oracle.forward(g, lay, forced_ids=forced)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec, path=moe.PATH_PREFILL, deterministic=det)
    ids_d = torch.from_numpy(forced).cuda()
    w_d = torch.from_numpy(ref.w.astype(np.float32)).cuda()
    sg = torch.from_numpy(ref.sgate.astype(np.float32)).cuda()
    y16 = moe.moe_ffn_forward_routed(c, x, ids_d, w_d, experts, shared, sgate=sg)
    y32 = moe.moe_ffn_forward_routed(c.replace(y_fp32=1), x, ids_d, w_d, experts, shared, sgate=sg)
    check_outputs(y32, y16, ref.y, "hot expert", exact=is_exact(c, 300))


# ----------------------------------------------------------------------------- MXFP4 prefill forms
FP4_PREFILL_SPECS = [
    # about 300 rows per expert: work items of 256 rows (two m tiles) and a ragged one
    mi.small_spec("gptoss", 128, 4, 2, 128, 0, 600, bias=("normal", 0.1)),
    # E == k: every expert takes all 333 tokens; gate_up N 128, down N 192
    mi.small_spec("gptoss", 192, 3, 3, 64, 0, 333),
    # scale bytes spread over 70..130: blocks far below their row's largest scale
    mi.small_spec("gptoss", 256, 8, 2, 192, 0, 700, bias=("zipf", 1.1), scale_lo=70, scale_hi=130),
]


@pytest.mark.parametrize("spec", FP4_PREFILL_SPECS, ids=lambda s: s.name)
@pytest.mark.parametrize("det", [1, 0], ids=["fixed-order", "accumulated"])
def test_mxfp4_prefill_f16_operands(spec, det):
    """The f16-operand MXFP4 grouped GEMMs (two m tiles per decoded weight tile)."""
    moe = moe_lib()
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec, path=moe.PATH_PREFILL, deterministic=det)
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
    check_outputs(y32, y16, ref.y, spec.name, exact=is_exact(c, T))


@pytest.mark.parametrize("path,det", PATH_MODES, ids=PATH_MODE_IDS)
def test_mxfp4_unbounded_glu_limit(path, det):
    """A clamp limit too wide for an f16 h takes the bf16-dequant grouped GEMMs."""
    moe = moe_lib()
    spec = mi.small_spec("gptoss", 128, 8, 2, 128, 0, 300, bias=("normal", 0.1), scale_lo=112,
                         scale_hi=118)
    lay = mi.make_layer(spec)
    g = dataclasses.replace(oracle.gating_for(spec), limit=300.0)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec, path=path, deterministic=det).replace(glu_limit=300.0)
    ids = torch.empty((300, 2), dtype=torch.int32, device="cuda")
    ws = moe.workspace(c, 300)
    y16 = moe.moe_ffn_forward(c, x, router, experts, shared, topk_ids=ids, ws=ws)
    y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), x, router, experts, shared, ws=ws)
    assert moe.moe_device_status(ws)[0] == 0
    ids_g = ids.cpu().numpy()
    diff = np.any(ids_g != ref.ids, axis=1)
    assert not np.any(diff & ~oracle.near_tie_tokens(ref.logits, ref.ids))
    if np.any(diff):
        ref = oracle.forward(g, lay, forced_ids=np.where(diff[:, None], ids_g, ref.ids))
    check_outputs(y32, y16, ref.y, "limit 300", exact=is_exact(c, 300))


@pytest.mark.parametrize("shift", [-40, -14, 0, 30])
@pytest.mark.parametrize("det", [1, 0], ids=["fixed-order", "accumulated"])
def test_mxfp4_prefill_token_magnitudes(shift, det):
    """x scaled by 2^shift (exact in bf16) with zero expert biases, so that h and y
    follow x's magnitude: the per-row f16 staging of x and of h must absorb it."""
    moe = moe_lib()
    spec = mi.small_spec("gptoss", 128, 4, 2, 128, 0, 300, scale_lo=116, scale_hi=126)
    lay = mi.make_layer(spec)
    lay.gu_bias = np.zeros_like(lay.gu_bias)
    lay.dn_bias = np.zeros_like(lay.dn_bias)
    x = mi.bf16_to_f32(lay.x).astype(np.float64) * 2.0 ** shift
    x[1] = 0.0                                   # an all-zero token row
    x[2, 5] *= 2.0 ** 20                         # one large value among ordinary ones
    lay.x = mi.f64_to_bf16(x)
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    xd, router, experts, shared = upload(lay)
    c = cfg_for(spec, path=moe.PATH_PREFILL, deterministic=det)
    ids = torch.empty((300, 2), dtype=torch.int32, device="cuda")
    ws = moe.workspace(c, 300)
    y16 = moe.moe_ffn_forward(c, xd, router, experts, shared, topk_ids=ids, ws=ws)
    y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), xd, router, experts, shared, ws=ws)
    assert moe.moe_device_status(ws)[0] == 0
    ids_g = ids.cpu().numpy()
    diff = np.any(ids_g != ref.ids, axis=1)
    assert not np.any(diff & ~oracle.near_tie_tokens(ref.logits, ref.ids))
    if np.any(diff):
        ref = oracle.forward(g, lay, forced_ids=np.where(diff[:, None], ids_g, ref.ids))
    check_outputs(y32, y16, ref.y, f"shift {shift}", exact=is_exact(c, 300))


# ----------------------------------------------------------------------------- RMSNorm + residual
NORM_CASES = [
    (mi.small_spec("qwen", 128, 16, 4, 64, 96, 33, bias=("normal", 0.5)), 1, 1),       # decode, warp
    (mi.small_spec("qwen", 96, 16, 4, 64, 64, 12, bias=("normal", 0.5)), 1, 1),        # decode, one launch
    (mi.small_spec("qwen", 256, 16, 4, 128, 128, 300, bias=("normal", 0.5)), 2, 1),    # prefill bf16
    (mi.small_spec("qwen", 256, 16, 4, 128, 128, 300, bias=("normal", 0.5)), 2, 0),    # ... accumulated
    (mi.small_spec("gptoss", 96, 12, 4, 96, 0, 7, bias=("normal", 0.1)), 1, 1),        # decode ring
    (mi.small_spec("gptoss", 128, 4, 2, 128, 0, 600, bias=("normal", 0.1)), 2, 1),     # prefill f16
    (mi.small_spec("gptoss", 128, 4, 2, 128, 0, 600, bias=("normal", 0.1)), 2, 0),     # ... accumulated
]


def _eps(spec):
    return 1e-6 if spec.family == "qwen" else 1e-5


@pytest.mark.parametrize("spec,path,det", NORM_CASES, ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_rmsnorm_and_residual_match_oracle(spec, path, det):
    """y = x + MoE(RMSNorm(x)) through every kernel plan, against the oracle."""
    moe = moe_lib()
    lay = mi.make_layer(spec)
    lay.norm_w = mi.make_norm_w(spec)
    g = dataclasses.replace(oracle.gating_for(spec), rms_norm=1, residual=1, rms_eps=_eps(spec))
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec, path=path, deterministic=det).replace(rms_norm=1, residual=1, rms_eps=_eps(spec))
    T, k = spec.tokens, spec.top_k
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ws = moe.workspace(c, T)
    y16 = moe.moe_ffn_forward(c, x, router, experts, shared, topk_ids=ids, ws=ws)
    y32 = moe.moe_ffn_forward(c.replace(y_fp32=1), x, router, experts, shared, ws=ws)
    assert moe.moe_device_status(ws)[0] == 0
    ids_g = ids.cpu().numpy()
    diff = np.any(ids_g != ref.ids, axis=1)
    assert not np.any(diff & ~oracle.near_tie_tokens(ref.logits, ref.ids))
    if np.any(diff):
        ref = oracle.forward(g, lay, forced_ids=np.where(diff[:, None], ids_g, ref.ids))
    check_outputs(y32, y16, ref.y, f"{spec.name} path {path}", exact=is_exact(c, T))
    # the router alone applies the same norm: its ids and logits agree with the layer's
    logits = torch.empty((T, spec.n_experts), dtype=torch.float32, device="cuda")
    ids2, _, _, _ = moe.moe_route(c, x, router, shared, logits=logits, ws=ws)
    assert torch.equal(ids2, ids)
    # (a normalised element may round to the other neighbouring bf16 value in fp32)
    assert np.allclose(logits.cpu().numpy(), ref.logits, rtol=1e-3, atol=2e-3)


def test_residual_with_caller_routing():
    """The routed entry point adds the residual; with rms_norm it refuses (no router)."""
    moe = moe_lib()
    spec = mi.small_spec("qwen", 64, 8, 3, 32, 32, 45)
    lay = mi.make_layer(spec)
    g = dataclasses.replace(oracle.gating_for(spec), residual=1)
    ref = oracle.forward(g, lay)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec).replace(residual=1)
    ids_d = torch.from_numpy(ref.ids).cuda()
    w_d = torch.from_numpy(ref.w.astype(np.float32)).cuda()
    sg = torch.from_numpy(ref.sgate.astype(np.float32)).cuda()
    y16 = moe.moe_ffn_forward_routed(c, x, ids_d, w_d, experts, shared, sgate=sg)
    y32 = moe.moe_ffn_forward_routed(c.replace(y_fp32=1), x, ids_d, w_d, experts, shared, sgate=sg)
    check_outputs(y32, y16, ref.y, "routed residual")
    with pytest.raises(moe.MoeError):
        moe.moe_ffn_forward_routed(c.replace(rms_norm=1, rms_eps=1e-6), x, ids_d, w_d, experts, shared,
                                   sgate=sg)


# ----------------------------------------------------------------------------- CUDA graphs
GRAPH_CASES = [
    (mi.small_spec("qwen", 128, 16, 4, 64, 96, 33, bias=("normal", 0.5)), 1),          # decode
    (mi.small_spec("gptoss", 96, 12, 4, 96, 0, 7, bias=("normal", 0.1)), 1),           # decode ring
    (mi.small_spec("qwen", 128, 32, 4, 64, 64, 8, bias=("normal", 0.5)), 1),            # bf16 decode ring
    (mi.small_spec("gptoss", 128, 4, 2, 128, 0, 600, bias=("normal", 0.1)), 1),        # prefill f16
    (mi.small_spec("qwen", 256, 16, 4, 128, 128, 300, bias=("normal", 0.5)), 1),       # prefill bf16
    (mi.small_spec("gptoss", 128, 4, 2, 128, 0, 600, bias=("normal", 0.1)), 0),        # ... accumulated
    (mi.small_spec("qwen", 256, 16, 4, 128, 128, 300, bias=("normal", 0.5)), 0),       # ... accumulated
]


@pytest.mark.parametrize("spec,det", GRAPH_CASES, ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_forward_captured_in_a_cuda_graph(spec, det):
    """moe_ffn_forward captured once and replayed on new inputs gives, bit for bit, what
    eager calls give (no host synchronisation, no allocation, no state kept between
    calls).  The first, eager call sets the kernels' launch attributes."""
    moe = moe_lib()
    lay = mi.make_layer(spec)
    x, router, experts, shared = upload(lay)
    c = cfg_for(spec, deterministic=det)
    T = spec.tokens
    ws = moe.workspace(c, T)
    y = torch.empty_like(x)
    moe.moe_ffn_forward(c, x, router, experts, shared, y=y, ws=ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            moe.moe_ffn_forward(c, x, router, experts, shared, y=y, ws=ws, stream=s)
    for rep in range(3):
        xs = mi.make_x(dataclasses.replace(spec, seed=spec.seed + 17 * rep), T)
        x.copy_(torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).cuda())
        graph.replay()
        torch.cuda.synchronize()
        want = moe.moe_ffn_forward(c, x, router, experts, shared, ws=moe.workspace(c, T))
        torch.cuda.synchronize()
        same_bf16(y, want, is_exact(c, T), rep)
