"""Design readings that rest on arithmetic, checked on the CPU with the oracle.

Native block-scaled FP4 tensor-core MMA (tcgen05 kind::mxf8f6f4 / kind::mxf4) takes
both operands in 8-, 6- or 4-bit element formats with one E8M0 scale per 32
elements: the token operand would have to be quantised to MXFP8 (E4M3 elements) at
best.  The layer's contract bounds the output error by 2e-2 * rms(y) against the
exact result on the given bf16 / MXFP4 inputs.  Quantising only the activations x
of the gpt-oss layer to MXFP8 (the weights stay exact, h stays exact) already
moves y by a third of its rms, far past that bound.  Two MXFP8 terms (x = hi + lo,
lo the MXFP8 rounding of x - hi) keep about eight significant bits and stay within
the bound, but cost two MMAs per block.

MXFP8 per the OCP Microscaling Formats (MX) v1.0 definition: per block of 32, the
shared scale is 2^(floor(log2(amax)) - 8) (8 = the largest exponent of E4M3), and
each element is x / scale rounded to E4M3 (1 sign, 4 exponent bits with bias 7, 3
mantissa bits, largest 448, subnormal step 2^-9), to nearest even, saturating.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle

TOL_RMS = 2e-2


def e4m3(v: np.ndarray) -> np.ndarray:
    """v rounded to E4M3 (round to nearest even, saturating at 448)."""
    a = np.abs(v)
    e = np.maximum(np.floor(np.log2(np.maximum(a, 1e-300))), -6.0)   # subnormals share 2^-6's step
    step = 2.0 ** (e - 3)
    q = np.minimum(np.round(a / step) * step, 448.0)                 # np.round: half to even
    return np.sign(v) * q


def mxfp8(x: np.ndarray) -> np.ndarray:
    """x [T, d] quantised to MXFP8 (E4M3 elements, one power-of-two scale per 32)."""
    T, d = x.shape
    xb = x.reshape(T, d // 32, 32)
    amax = np.abs(xb).max(axis=2, keepdims=True)
    scale = 2.0 ** np.where(amax > 0, np.floor(np.log2(np.maximum(amax, 1e-300))) - 8.0, 0.0)
    return (e4m3(xb / scale) * scale).reshape(T, d)


def test_e4m3_rounding_points():
    # exact values, the largest, a subnormal, a halfway case to even, saturation
    v = np.array([1.0, -1.125, 448.0, 2.0 ** -9, 1.0625, 1.1875, 500.0, 0.0])
    assert e4m3(v).tolist() == [1.0, -1.125, 448.0, 2.0 ** -9, 1.0, 1.25, 448.0, 0.0]


def test_mxfp8_activations_exceed_the_layer_tolerance():
    spec = mi.small_spec("gptoss", 256, 8, 2, 256, 0, 64, bias=("normal", 0.1))
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    x = mi.bf16_to_f32(lay.x).astype(np.float64)
    xq = mxfp8(x)
    # an E4M3 value times a power of two is exact in bf16: the oracle sees xq itself
    xb = mi.f64_to_bf16(xq)
    assert np.array_equal(mi.bf16_to_f32(xb).astype(np.float64), xq)
    rel = np.sqrt(np.mean((xq - x) ** 2)) / np.sqrt(np.mean(x ** 2))
    assert 0.01 < rel < 0.05                      # about 3% per element
    q = oracle.forward(g, lay, x=xb, forced_ids=ref.ids)
    rms = float(np.sqrt(np.mean(ref.y ** 2)))
    err = float(np.max(np.abs(q.y - ref.y)))
    assert err > 5 * TOL_RMS * rms, err / rms     # measured: about 0.34 rms


def test_two_mxfp8_terms_stay_within_the_layer_tolerance():
    spec = mi.small_spec("gptoss", 256, 8, 2, 256, 0, 64, bias=("normal", 0.1))
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    ref = oracle.forward(g, lay)
    x = mi.bf16_to_f32(lay.x).astype(np.float64)
    hi = mxfp8(x)
    xq = hi + mxfp8(x - hi)
    xb = mi.f64_to_bf16(xq)
    assert np.array_equal(mi.bf16_to_f32(xb).astype(np.float64), xq)   # hi + lo is a bf16 value
    rel = np.sqrt(np.mean((xq - x) ** 2)) / np.sqrt(np.mean(x ** 2))
    assert rel < 1e-3                             # about 2^-11 per element
    q = oracle.forward(g, lay, x=xb, forced_ids=ref.ids)
    rms = float(np.sqrt(np.mean(ref.y ** 2)))
    err = float(np.max(np.abs(q.y - ref.y)))
    assert err < TOL_RMS * rms, err / rms         # measured: about 0.015 rms
