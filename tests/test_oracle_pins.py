"""Pins of the fp64 oracle to facts fixed outside it (CPU only).

Each test ties one oracle function to something other than its own code: the
E2M1 table of the MX specification and the nibble-order worked cases from the
gpt-oss page (golden fixtures), library routines (math.ldexp, Python's stable
sort, scipy's softmax/expit) on special cases, closed forms (x = 0, one-hot x,
designed weights), and invariants (identical experts, permutation
equivariance, duplicated tokens, E = k).  Each is chosen so that a plausible
slip in the oracle -- a swapped gate/up, a dropped +1, a one-sided clamp made
two-sided, a transposed down matrix, a wrong nibble or tie order -- fails one.
"""
import math

import numpy as np
import pytest
from scipy.special import expit, softmax

import moe_inputs as mi
import oracle
from conftest import read_golden

BF = mi.f64_to_bf16


def e2m1_table():
    return {int(c): float(v) for c, v in read_golden("e2m1_values.txt")}


def encode_mxfp4(values: np.ndarray, scale: int = 127):
    """Pack E2M1-representable values [rows, n_in] (times 2^(scale-127)) into blocks/scales."""
    tab = e2m1_table()
    inv = {}
    for c in range(16):
        inv.setdefault(tab[c], c)        # +0 -> code 0
    rows, n_in = values.shape
    f = 2.0 ** (scale - 127)
    codes = np.vectorize(lambda v: inv[v / f])(values).astype(np.uint8)
    blocks = (codes[:, 0::2] | (codes[:, 1::2] << 4)).reshape(rows, n_in // 32, 16)
    scales = np.full((rows, n_in // 32), scale, np.uint8)
    return np.ascontiguousarray(blocks), scales


# ----------------------------------------------------------------------------- formats
def test_e2m1_matches_mx_table():
    tab = e2m1_table()
    for c in range(16):
        v = oracle.e2m1(c)
        assert v == tab[c] and math.copysign(1, v) == math.copysign(1, tab[c]), c


def test_e8m0_is_power_of_two():
    for s in range(255):
        assert oracle.e8m0(s) == math.ldexp(1.0, s - 127)
    assert math.isnan(oracle.e8m0(255))


def test_mxfp4_nibble_order_worked_cases():
    for b_idx, byte, scale, v_even, v_odd in read_golden("mxfp4_nibble_order.txt"):
        b_idx, byte, scale = int(b_idx), int(byte, 16), int(scale)
        blocks = np.zeros((1, 1, 16), np.uint8)
        blocks[0, 0, b_idx] = byte
        out = oracle.mxfp4_decode(blocks, np.array([[scale]], np.uint8))[0]
        assert out[2 * b_idx] == float(v_even) and out[2 * b_idx + 1] == float(v_odd)
        assert math.copysign(1, out[2 * b_idx + 1]) == math.copysign(1, float(v_odd))
        rest = np.delete(out, [2 * b_idx, 2 * b_idx + 1])
        assert np.all(rest == 0.0)


@pytest.mark.parametrize("scale", [1, 118, 126, 127, 254])
def test_mxfp4_every_code_every_position(scale):
    tab = e2m1_table()
    codes = np.arange(64) % 16                     # 64 inputs = 2 blocks, codes cycle
    rng = np.random.default_rng(1)
    codes = rng.permutation(codes)
    blocks = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8).reshape(1, 2, 16)
    out = oracle.mxfp4_decode(blocks, np.array([[scale, scale]], np.uint8))[0]
    want = np.array([tab[int(c)] for c in codes]) * math.ldexp(1.0, scale - 127)
    assert np.array_equal(out, want)


def test_mxfp4_scale_applies_per_block():
    blocks = np.full((2, 2, 16), 0x22, np.uint8)   # every element 1.0
    scales = np.array([[120, 130], [127, 1]], np.uint8)
    out = oracle.mxfp4_decode(blocks, scales)
    for r in range(2):
        for b in range(2):
            assert np.all(out[r, 32 * b:32 * b + 32] == math.ldexp(1.0, int(scales[r, b]) - 127))


# ----------------------------------------------------------------------------- top-k
def brute_topk(key, k):
    return sorted(range(len(key)), key=lambda e: (-key[e], e))[:k]


@pytest.mark.parametrize("seed", range(40))
def test_topk_matches_stable_sort(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 11))
    k = int(rng.integers(1, E + 1))
    if seed % 2:
        key = rng.choice([-1.0, -0.0, 0.0, 1.0, 2.0], size=E)   # many ties, signed zeros
    else:
        key = rng.standard_normal(E)
    assert list(oracle.select_topk(key, k)) == brute_topk(list(key), k)


def test_topk_first_seen_on_full_tie():
    assert list(oracle.select_topk(np.zeros(9), 9)) == list(range(9))
    assert list(oracle.select_topk(np.array([0.0, -0.0, 0.0, -0.0]), 4)) == [0, 1, 2, 3]


# ----------------------------------------------------------------------------- gating weights
@pytest.mark.parametrize("scale", [1.0, 2.5])
def test_qwen_renorm_weights(scale):
    rng = np.random.default_rng(7)
    g = oracle.Gating(d_model=32, n_experts=256, top_k=8, expert_ff=32, gating=0, scale=scale)
    logits = rng.standard_normal((50, 256)) * 2
    ids, w = oracle.route_from_logits(g, logits)
    assert np.allclose(w.sum(1), scale, rtol=0, atol=1e-12)
    sel = np.take_along_axis(logits, ids.astype(np.int64), 1)
    # renormalised softmax: ratios depend only on logit differences (denominator cancels)
    assert np.allclose(w / w[:, :1], np.exp(sel - sel[:, :1]), rtol=1e-12)
    for t in range(50):
        assert list(ids[t]) == brute_topk(list(logits[t]), 8)


def test_qwen_weights_without_renorm():
    rng = np.random.default_rng(8)
    g = oracle.Gating(d_model=32, n_experts=64, top_k=4, expert_ff=32, gating=0,
                      norm_topk_prob=0, scale=1.5)
    logits = rng.standard_normal((20, 64))
    ids, w = oracle.route_from_logits(g, logits)
    p = softmax(logits, axis=1)
    assert np.allclose(w, 1.5 * np.take_along_axis(p, ids.astype(np.int64), 1), rtol=1e-12)


def test_gptoss_topk_then_softmax():
    rng = np.random.default_rng(9)
    g = oracle.Gating(d_model=32, n_experts=32, top_k=4, expert_ff=32, gating=1)
    logits = rng.standard_normal((30, 32))
    ids, w = oracle.route_from_logits(g, logits)
    for t in range(30):
        assert list(ids[t]) == brute_topk(list(logits[t]), 4)
        assert np.allclose(w[t], softmax(logits[t, ids[t]]), rtol=1e-13)
    assert np.allclose(w.sum(1), 1.0, atol=1e-13)


# ----------------------------------------------------------------------------- layer closed forms
def small_qwen(E=8, k=3, d=64, ff=32, sff=32, T=5, bias=None, **kw):
    spec = mi.small_spec("qwen", d, E, k, ff, sff, T, bias=bias, **kw)
    return spec, mi.make_layer(spec)


def small_oss(E=8, k=2, d=64, ff=64, T=5, bias=("normal", 0.1)):
    spec = mi.small_spec("gptoss", d, E, k, ff, 0, T, bias=bias)
    return spec, mi.make_layer(spec)


def test_router_and_shared_gate_on_one_hot_x():
    spec, lay = small_qwen(bias=("normal", 0.5))
    g = oracle.gating_for(spec)
    d = spec.d_model
    x = np.zeros((d, d), np.uint16)
    c = BF(1.5)[()]
    for i in range(d):
        x[i, i] = c
    r = oracle.forward(g, lay, x=x)
    Wr = mi.bf16_to_f32(lay.router_w).astype(np.float64)
    b = mi.bf16_to_f32(lay.router_b).astype(np.float64)
    assert np.array_equal(r.logits, 1.5 * Wr.T + b[None, :])     # row i = 1.5 * column i + b
    wsh = mi.bf16_to_f32(lay.sh_gate_inp).astype(np.float64)
    assert np.allclose(r.sgate, expit(1.5 * wsh), rtol=1e-14)


def test_qwen_zero_input_closed_form():
    spec, lay = small_qwen(E=16, k=8)
    g = oracle.gating_for(spec)
    r = oracle.forward(g, lay, x=np.zeros((3, spec.d_model), np.uint16))
    assert np.array_equal(r.ids, np.tile(np.arange(8), (3, 1)))
    assert np.all(r.w == 1.0 / 8) and np.all(r.sgate == 0.5) and np.all(r.y == 0.0)


def test_zero_input_with_bias_routes_by_bias():
    for spec, lay in (small_qwen(E=16, k=4, bias=("normal", 0.5)), small_oss(E=16, k=4)):
        g = oracle.gating_for(spec)
        r = oracle.forward(g, lay, x=np.zeros((2, spec.d_model), np.uint16))
        b = mi.bf16_to_f32(lay.router_b).astype(np.float64)
        assert list(r.ids[0]) == brute_topk(list(b), 4) and list(r.ids[1]) == list(r.ids[0])


def test_swiglu_designed_weights():
    """One expert, ff = 2, gate/up rows pick single inputs: y = D @ [silu(x0) x1, silu(x2) x3]."""
    d, ff = 32, 2
    spec = mi.small_spec("qwen", d, 1, 1, ff, 0, 1)
    lay = mi.make_layer(spec)
    lay.gate[:] = 0
    lay.up[:] = 0
    lay.gate[0, 0, 0] = BF(1.0)[()]
    lay.up[0, 0, 1] = BF(1.0)[()]
    lay.gate[0, 1, 2] = BF(1.0)[()]
    lay.up[0, 1, 3] = BF(1.0)[()]
    rng = np.random.default_rng(3)
    D = BF(rng.standard_normal((d, ff)))
    lay.down[0] = D
    xv = np.zeros(d)
    xv[:4] = [1.0, 2.0, -0.5, 3.0]
    r = oracle.forward(oracle.gating_for(spec), lay, x=BF(xv)[None, :])
    h = np.array([1.0 * expit(1.0) * 2.0, -0.5 * expit(-0.5) * 3.0])
    want = mi.bf16_to_f32(D).astype(np.float64) @ h
    assert np.allclose(r.y[0], want, rtol=1e-14, atol=0)


def test_clamped_glu_designed_weights():
    """One MXFP4 expert; gate_f and up_f are set through single weights and biases.

    down = identity, so y_f = h_f + b_down_f exposes each activation value.
    """
    d = ff = 32
    spec = mi.small_spec("gptoss", d, 1, 1, ff, 0, 1, bias=None)
    lay = mi.make_layer(spec)
    # (gate, up) pairs: zero gate, clamp gate at 7 (gate 12), negative gates left alone
    # (-6 and -9 stay: the gate clamp is one-sided), up = -1 kills h, up clamps at +-7.
    cases = [(0.0, 3.0), (12.0, 0.0), (-6.0, 2.0), (2.0, -1.0), (1.5, 12.0), (3.0, -12.0),
             (6.0, 4.0), (-0.5, -0.5), (-9.0, 1.0)]
    gu = np.zeros((2 * ff, d))
    gbias = np.zeros(2 * ff)

    def split(v):          # v = weight * 1 + bias, weight E2M1-representable, bias bf16-exact
        w = 0.0 if abs(v) < 6 else math.copysign(6.0, v)
        return w, v - w

    for f, (gv, uv) in enumerate(cases):
        gu[2 * f, 0], gbias[2 * f] = split(gv)          # gate = even row, reads input 0
        gu[2 * f + 1, 1], gbias[2 * f + 1] = split(uv)  # up = odd row, reads input 1
    blocks, scales = encode_mxfp4(gu)
    lay.gu_blocks[0], lay.gu_scales[0] = blocks, scales
    lay.gu_bias[0] = BF(gbias)
    dn = np.eye(d, ff)
    lay.dn_blocks[0], lay.dn_scales[0] = encode_mxfp4(dn)
    dbias = BF(np.linspace(-0.25, 0.25, d))
    lay.dn_bias[0] = dbias
    xv = np.zeros(d)
    xv[0] = xv[1] = 1.0
    r = oracle.forward(oracle.gating_for(spec), lay, x=BF(xv)[None, :])
    assert r.ids[0, 0] == 0 and r.w[0, 0] == 1.0
    for f, (gv, uv) in enumerate(cases):
        gate = min(gv, 7.0)
        up = min(max(uv, -7.0), 7.0)
        h = (up + 1.0) * gate * expit(1.702 * gate)
        assert r.y[0, f] == pytest.approx(h + float(mi.bf16_to_f32(dbias[f])), rel=1e-14, abs=1e-15)
    assert r.y[0, 3] == pytest.approx(float(mi.bf16_to_f32(dbias[3])), abs=0)   # up = -1 -> h = 0


# ----------------------------------------------------------------------------- invariants
def _identical_experts(lay, spec):
    if spec.family == "qwen":
        for a in (lay.gate, lay.up, lay.down):
            a[:] = a[0]
    else:
        for a in (lay.gu_blocks, lay.gu_scales, lay.gu_bias, lay.dn_blocks, lay.dn_scales,
                  lay.dn_bias):
            a[:] = a[0]


@pytest.mark.parametrize("family", ["qwen", "gptoss"])
def test_identical_experts_make_routing_irrelevant(family):
    spec, lay = small_qwen(E=8, k=3) if family == "qwen" else small_oss(E=8, k=3)
    spec = mi.small_spec(family, spec.d_model, 8, 3, spec.expert_ff, spec.shared_ff, 6,
                         bias=("normal", 0.5), expert_weights_scale=1.25 if family == "qwen" else 1.0)
    lay = mi.make_layer(spec)
    _identical_experts(lay, spec)
    r = oracle.forward(oracle.gating_for(spec), lay)
    # the same layer with a single expert and top-1: softmax weight 1 times the scale
    one = mi.small_spec(family, spec.d_model, 1, 1, spec.expert_ff, spec.shared_ff, 6, bias=None,
                        expert_weights_scale=spec.expert_weights_scale)
    lay1 = mi.make_layer(one)
    for name in ("gate", "up", "down", "gu_blocks", "gu_scales", "gu_bias", "dn_blocks",
                 "dn_scales", "dn_bias"):
        a = getattr(lay, name)
        if a is not None:
            setattr(lay1, name, np.ascontiguousarray(a[:1]))
    for name in ("sh_gate", "sh_up", "sh_down", "sh_gate_inp", "x"):
        setattr(lay1, name, getattr(lay, name))
    r1 = oracle.forward(oracle.gating_for(one), lay1)
    assert np.allclose(r.y, r1.y, rtol=1e-12, atol=1e-12 * np.abs(r1.y).max())
    assert len({tuple(i) for i in r.ids}) > 1                    # routing did vary


def test_shared_expert_combine():
    """Routed experts zeroed: y = sgate * shared(x), shared(x) from a shared-only twin layer."""
    spec, lay = small_qwen(E=8, k=2, T=4)
    lay.down[:] = 0
    r = oracle.forward(oracle.gating_for(spec), lay)
    twin_spec = mi.small_spec("qwen", spec.d_model, 1, 1, spec.expert_ff, 0, 4)
    twin = mi.make_layer(twin_spec)
    twin.gate[0], twin.up[0], twin.down[0] = lay.sh_gate, lay.sh_up, lay.sh_down
    twin.x = lay.x
    r_sh = oracle.forward(oracle.gating_for(twin_spec), twin)
    assert np.allclose(r.y, r.sgate[:, None] * r_sh.y, rtol=1e-13, atol=1e-15)
    assert np.all((r.sgate > 0) & (r.sgate < 1))


@pytest.mark.parametrize("family", ["qwen", "gptoss"])
def test_permutation_equivariance_and_duplicates(family):
    spec, lay = small_qwen(T=6) if family == "qwen" else small_oss(T=6)
    g = oracle.gating_for(spec)
    r = oracle.forward(g, lay)
    perm = np.array([3, 0, 5, 5, 1, 2, 4, 0])
    rp = oracle.forward(g, lay, x=np.ascontiguousarray(lay.x[perm]))
    assert np.array_equal(rp.y, r.y[perm]) and np.array_equal(rp.ids, r.ids[perm])
    assert np.array_equal(rp.w, r.w[perm]) and np.array_equal(rp.sgate, r.sgate[perm])
    tok = oracle.forward(g, lay, tokens=np.array([4, 1]))
    assert np.array_equal(tok.y, r.y[[4, 1]])


def test_all_experts_selected_when_k_equals_E():
    spec, lay = small_qwen(E=6, k=6)
    r = oracle.forward(oracle.gating_for(spec), lay)
    for t in range(r.ids.shape[0]):
        assert sorted(r.ids[t]) == list(range(6))
        assert list(r.ids[t]) == brute_topk(list(r.logits[t]), 6)


def test_forced_routing_keeps_gating_rule():
    spec, lay = small_oss(E=8, k=2, T=3)
    g = oracle.gating_for(spec)
    r = oracle.forward(g, lay)
    same = oracle.forward(g, lay, forced_ids=r.ids)
    assert np.array_equal(same.y, r.y)
    forced = np.array([[7, 6], [0, 1], [3, 2]], np.int32)
    f = oracle.forward(g, lay, forced_ids=forced)
    assert np.array_equal(f.ids, forced)
    for t in range(3):
        assert np.allclose(f.w[t], softmax(f.logits[t, forced[t]]), rtol=1e-13)


def test_near_tie_detector():
    lg = np.array([[3.0, 1.0, 1.0 + 5e-6, 0.0], [3.0, 2.0, 1.0, 0.0]])
    ids = np.array([[0, 2], [0, 1]])
    assert list(oracle.near_tie_tokens(lg, ids)) == [True, False]


def test_route_only_matches_forward():
    for spec, lay in (small_qwen(E=16, k=4, bias=("normal", 0.5), T=7), small_oss(E=8, k=2, T=7)):
        g = oracle.gating_for(spec)
        f = oracle.forward(g, lay)
        r = oracle.route(g, lay, tokens=np.arange(7)[::-1].copy())
        assert np.array_equal(r.ids, f.ids[::-1]) and np.array_equal(r.w, f.w[::-1])
        assert np.array_equal(r.sgate, f.sgate[::-1]) and np.array_equal(r.logits, f.logits[::-1])


# ----------------------------------------------------------------------------- RMSNorm and residual
def _with_norm(spec, lay):
    lay.norm_w = mi.make_norm_w(spec)
    return lay


def test_rmsnorm_one_hot_closed_form():
    """x = c e_i: mean(x^2) = c^2 / d, so with eps = 0 the MoE input is sqrt(d) sign(c) w_i e_i
    and the logits are sqrt(d) sign(c) w_i W_r[:, i] + b."""
    spec, lay = small_qwen(bias=("normal", 0.5))
    _with_norm(spec, lay)
    g = oracle.gating_for(spec)
    g.rms_norm, g.rms_eps = 1, 0.0
    d = spec.d_model
    x = np.zeros((d, d), np.uint16)
    for i in range(d):
        x[i, i] = BF(-1.5 if i % 2 else 2.25)[()]
    r = oracle.forward(g, lay, x=x)
    Wr = mi.bf16_to_f32(lay.router_w).astype(np.float64)
    b = mi.bf16_to_f32(lay.router_b).astype(np.float64)
    w = mi.bf16_to_f32(lay.norm_w).astype(np.float64)
    sgn = np.where(np.arange(d) % 2, -1.0, 1.0)
    want = math.sqrt(d) * (sgn * w)[:, None] * Wr.T + b[None, :]
    assert np.allclose(r.logits, want, rtol=1e-13, atol=1e-13)


def test_rmsnorm_per_token_scale_invariance():
    """With eps = 0 the normalised input does not depend on each token's scale: tokens
    scaled by different powers of two (exact in bf16) give the same outputs."""
    for spec, lay in (small_qwen(), small_oss()):
        _with_norm(spec, lay)
        g = oracle.gating_for(spec)
        g.rms_norm, g.rms_eps = 1, 0.0
        x = mi.bf16_to_f32(lay.x).astype(np.float64)
        f = 2.0 ** (np.arange(x.shape[0]) % 5 * 3 - 6)
        r0 = oracle.forward(g, lay)
        r1 = oracle.forward(g, lay, x=BF(x * f[:, None]))
        assert np.array_equal(r0.ids, r1.ids)
        assert np.allclose(r0.y, r1.y, rtol=1e-12, atol=1e-12 * np.abs(r0.y).max())


def test_rmsnorm_eps_keeps_zero_rows_finite():
    """A zero token normalises to zero (0 / sqrt(eps)), giving the zero-input closed form."""
    spec, lay = small_qwen(E=16, k=8)
    _with_norm(spec, lay)
    g = oracle.gating_for(spec)
    g.rms_norm = 1
    r = oracle.forward(g, lay, x=np.zeros((2, spec.d_model), np.uint16))
    assert np.array_equal(r.ids, np.tile(np.arange(8), (2, 1)))
    assert np.all(r.y == 0.0) and np.all(r.sgate == 0.5)


@pytest.mark.parametrize("family", ["qwen", "gptoss"])
def test_residual_adds_the_unnormalised_input(family):
    """y(residual) - y(no residual) = x exactly, and with every down projection zero y = x."""
    spec, lay = small_qwen() if family == "qwen" else small_oss()
    _with_norm(spec, lay)
    g = oracle.gating_for(spec)
    g.rms_norm = 1
    x = mi.bf16_to_f32(lay.x).astype(np.float64)
    g.residual = 0
    y0 = oracle.forward(g, lay).y
    g.residual = 1
    y1 = oracle.forward(g, lay).y
    assert np.allclose(y1 - y0, x, rtol=0, atol=1e-12 * max(1.0, np.abs(y0).max()))
    if family == "qwen":
        lay.down[:] = 0
        lay.sh_down[:] = 0
    else:
        lay.dn_blocks[:] = 0
        lay.dn_bias[:] = 0
    assert np.array_equal(oracle.forward(g, lay).y, x)


def test_rmsnorm_eps_inside_the_root():
    """A constant row x = 0.125 with eps = 0.046875: mean(x^2) + eps = 0.0625 whose root is
    0.25, so the MoE input is exactly 0.5 w, and the logits are 0.5 w . W_r^T + b."""
    spec, lay = small_qwen(bias=("normal", 0.5))
    _with_norm(spec, lay)
    g = oracle.gating_for(spec)
    g.rms_norm, g.rms_eps = 1, 0.046875
    x = np.full((2, spec.d_model), BF(0.125)[()], np.uint16)
    r = oracle.forward(g, lay, x=x)
    Wr = mi.bf16_to_f32(lay.router_w).astype(np.float64)
    b = mi.bf16_to_f32(lay.router_b).astype(np.float64)
    w = mi.bf16_to_f32(lay.norm_w).astype(np.float64)
    want = (0.5 * w) @ Wr.T + b
    assert np.allclose(r.logits, np.tile(want, (2, 1)), rtol=1e-13, atol=1e-13)


def test_rmsnorm_output_is_bf16_rounded():
    """The normalised input is a bf16 activation: x = 3 e_0 + (1 + 2^-7) e_2, w = 1,
    eps = 0.  Router rows that pick inputs 0 and 2 expose the two normalised values,
    which must equal the exact quotients rounded to the nearest bf16 (the input
    generator's independent conversion)."""
    spec, lay = small_qwen(E=8, k=1, bias=None)
    _with_norm(spec, lay)
    lay.norm_w[:] = BF(1.0)[()]
    lay.router_w[:] = 0
    lay.router_w[0, 0] = BF(1.0)[()]            # logit 0 = xn[0]
    lay.router_w[1, 2] = BF(1.0)[()]            # logit 1 = xn[2]
    g = oracle.gating_for(spec)
    g.rms_norm, g.rms_eps = 1, 0.0
    d = spec.d_model
    x = np.zeros((1, d), np.float64)
    x[0, 0] = 3.0
    x[0, 2] = 1.0 + 2.0 ** -7                   # exact in bf16 (8 significant bits)
    r = oracle.forward(g, lay, x=BF(x))
    inv = 1.0 / math.sqrt((9.0 + (1.0 + 2.0 ** -7) ** 2) / d)
    exact0, exact2 = 3.0 * inv, (1.0 + 2.0 ** -7) * inv
    b0 = float(mi.bf16_to_f32(BF(exact0))[()])
    b2 = float(mi.bf16_to_f32(BF(exact2))[()])
    assert r.logits[0, 0] == b0 and r.logits[0, 1] == b2
    assert b0 != exact0                          # the case does exercise the rounding
