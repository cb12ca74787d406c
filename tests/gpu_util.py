"""Helpers shared by the GPU parity tests (no test functions here)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle

TOL_RMS = 2e-2      # layer outputs: max |y_gpu - y_ref| <= 2e-2 * rms(y_ref)
NEAR_TIE = 1e-5     # logit gap under which a selection may legitimately differ


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def moe_lib():
    import sparse_moe_ffn_route_gb300 as moe
    return moe


def cfg_for(spec, **kw):
    """The layer's moe_cfg_t.  Tests take the fixed-order combine (deterministic = 1)
    unless they ask for the accumulated prefill (deterministic = 0, the library's
    default and the benchmark's configuration)."""
    moe = moe_lib()
    if spec.family == "qwen":
        c = moe.qwen_cfg(spec.d_model, spec.n_experts, spec.top_k, spec.expert_ff, spec.shared_ff,
                         expert_weights_scale=spec.expert_weights_scale,
                         norm_topk_prob=spec.norm_topk_prob)
    else:
        c = moe.gptoss_cfg(spec.d_model, spec.n_experts, spec.top_k, spec.expert_ff)
    kw.setdefault("deterministic", 1)
    return c.replace(**kw)


def is_exact(cfg, T):
    """Whether two calls give the same bits: always, except on the prefill path with the
    accumulated down projection (cfg.deterministic = 0), whose atomic adds may run in
    another order and change the last bits of the fp32 sums."""
    moe = moe_lib()
    return bool(cfg.deterministic) or moe.moe_kernel_plan(cfg, T) in (moe.PLAN_DECODE_WARP,
                                                                       moe.PLAN_DECODE_RING,
                                                                       moe.PLAN_DECODE_FUSED)


def bf16_ulps(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """|a - b| in units in the last place of bf16 (bit patterns as uint16; +0 == -0)."""
    def ordered(b):
        b = b.astype(np.int32)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(ordered(a_bits) - ordered(b_bits))


ORDER_TOL = 1e-5    # two accumulated runs: |difference| allowed next to rms(y), beyond one ulp


def bf16_close(a_bits: np.ndarray, b_bits: np.ndarray) -> bool:
    """Two bf16 results of fp32 sums taken in different orders: each pair within one
    unit in the last place, or within ORDER_TOL * rms (near-zero sums, where the fp32
    rounding of the order is many bf16 units of the small result)."""
    if a_bits.size == 0:
        return True
    a = mi.bf16_to_f32(a_bits).astype(np.float64)
    b = mi.bf16_to_f32(b_bits).astype(np.float64)
    rms = float(np.sqrt(np.mean(b ** 2)))
    ok = (bf16_ulps(a_bits, b_bits) <= 1) | (np.abs(a - b) <= ORDER_TOL * rms)
    return bool(np.all(ok))


def same_bf16(a: "torch.Tensor", b: "torch.Tensor", exact: bool, what=""):
    """Two bf16 outputs of the layer: equal bits, or (not exact: the accumulated
    prefill) equal up to the order of the fp32 sums (bf16_close)."""
    ab = a.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    bb = b.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    if exact:
        assert np.array_equal(ab, bb), what
    else:
        assert bf16_close(ab, bb), what


def upload(layer):
    from sparse_moe_ffn_route_gb300 import hostio
    return hostio.upload(layer)


def y_numpy(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def check_outputs(y32: "torch.Tensor", y16: "torch.Tensor", y_ref: np.ndarray, what="", exact=True):
    """Layer output parity.

    The computation is checked on the fp32 output (cfg.y_fp32 = 1) against the
    2e-2 * rms(y_ref) bar; the bf16 output must then be exactly that fp32 result
    rounded to nearest even (bf16 keeps 8 significant bits, so its own rounding
    alone can reach 2^-8 |y|, above the bar wherever |y| > 5.12 rms).  With the
    accumulated prefill (exact = False) the two outputs come from two calls whose
    atomic adds may have run in different orders: the bf16 output then equals
    RNE(fp32 output) up to the order of the sums (bf16_close).
    """
    y32n = y32.cpu().numpy()
    err = check_y(y32n.astype(np.float64), y_ref, what)
    bits = y16.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    rne = mi.f64_to_bf16(y32n)
    if exact:
        assert np.array_equal(bits, rne), f"{what}: bf16 output is not RNE(fp32 output)"
    else:
        assert bf16_close(bits, rne), f"{what}: bf16 output is not RNE(fp32 output) up to the sum order"
    return err


def check_y(y_gpu: np.ndarray, y_ref: np.ndarray, what=""):
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    err = float(np.max(np.abs(y_gpu - y_ref))) if y_ref.size else 0.0
    assert np.all(np.isfinite(y_gpu)), what
    assert err <= TOL_RMS * rms + 1e-30, f"{what}: max err {err:.3e} > {TOL_RMS} * rms {rms:.3e}"
    return err, rms


def check_routing(g, ids_gpu, w_gpu, logits_gpu_f32, ref, what=""):
    """GPU routing vs the oracle.

    (1) On the GPU's own fp32 logits the oracle's selection must equal the GPU's
        bit for bit, and the weights agree to 1e-5 relative.
    (2) Against the oracle's fp64 logits, ids agree except on near-tie tokens,
        which are returned.
    """
    ids_o, w_o = oracle.route_from_logits(g, logits_gpu_f32.astype(np.float64))
    assert np.array_equal(ids_o, ids_gpu), f"{what}: selection differs on the same fp32 logits"
    assert np.allclose(w_gpu, w_o, rtol=1e-5, atol=1e-7), what
    tie = oracle.near_tie_tokens(ref.logits, ref.ids, NEAR_TIE)
    diff = np.any(ids_gpu != ref.ids, axis=1)
    assert not np.any(diff & ~tie), f"{what}: ids differ on tokens {np.nonzero(diff & ~tie)[0]}"
    return tie, diff


def sample_tokens(T, n=48, seed=0):
    if T <= 64:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(8, T - 8), size=n - 16, replace=False)
    return np.sort(np.concatenate([np.arange(8), mid, np.arange(T - 8, T)])).astype(np.int32)
