"""fp64 CPU oracle for the sparse MoE FFN layer forward pass -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package.  The product library never calls it, and it shares no code with
the CUDA path: the arithmetic lives in ``moe_oracle.c`` (plain fp64 loops, OpenMP over
tokens) and this file only marshals numpy arrays through ctypes.

Functions and the passages they follow (page title, section):
  * ``e2m1``, ``e8m0``, ``mxfp4_decode``: "Phase 19: MoE - gpt-oss-20b", section 3
    (MXFP4 dequantisation) and the tensor-layout listing of section 2.
  * ``select_topk``: "qwen35moe CPU-reference golden vectors", Kernel 4 (selection
    sort, first-seen tie-break).
  * ``route_from_logits`` / ``forward``: Kernel 4 above for the softmax/renorm
    gating, "qwen35moe - Forward-Pass Design", section "Shared-expert MoE FFN", and
    "Phase 19", section 2 (Router, Experts) for the gpt-oss gating and experts.
  * ``Gating.rms_norm`` / ``Gating.residual`` (the steps either side of the MoE):
    "qwen35moe - Forward-Pass Design", "Block scaffold" (post_attention_norm, the
    residual adds the un-normalised input); "qwen35moe CPU-reference golden vectors",
    Kernel 3 (RMS = 1 / sqrt(mean(x^2) + eps), times the weight); "Phase 19",
    section 2 (RMSNorm, Decoder layer: out = h + moe(post_norm(h))).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lib = None
_lock = threading.Lock()


class OracleCfg(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("expert_ff", ctypes.c_int32),
                ("shared_ff", ctypes.c_int32), ("gating", ctypes.c_int32),
                ("act", ctypes.c_int32), ("wfmt", ctypes.c_int32),
                ("norm_topk_prob", ctypes.c_int32), ("interleaved", ctypes.c_int32),
                ("scale", ctypes.c_double), ("limit", ctypes.c_double),
                ("alpha", ctypes.c_double), ("rms_norm", ctypes.c_int32),
                ("residual", ctypes.c_int32), ("rms_eps", ctypes.c_double)]


class OracleWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router_w", "router_b", "gate", "up", "gate_up", "down", "gu_blocks", "gu_scales",
        "dn_blocks", "dn_scales", "gu_bias", "dn_bias", "sh_gate", "sh_up", "sh_down",
        "sh_gate_inp", "norm_w")]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c (gcc -O2, OpenMP, no FP contraction) into a shared library."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                           "-std=c11", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _get_lib():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I = ctypes.c_void_p, ctypes.c_int
            lib.oracle_bf16.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16.restype = ctypes.c_double
            lib.oracle_e2m1.argtypes = [I]
            lib.oracle_e2m1.restype = ctypes.c_double
            lib.oracle_e8m0.argtypes = [I]
            lib.oracle_e8m0.restype = ctypes.c_double
            lib.oracle_mxfp4_decode.argtypes = [P, P, ctypes.c_int64, I, P]
            lib.oracle_mxfp4_decode.restype = None
            lib.oracle_select_topk.argtypes = [P, I, I, P]
            lib.oracle_select_topk.restype = None
            lib.oracle_route_from_logits.argtypes = [ctypes.POINTER(OracleCfg), P, I, P, P]
            lib.oracle_route_from_logits.restype = None
            lib.oracle_forward.argtypes = [ctypes.POINTER(OracleCfg),
                                           ctypes.POINTER(OracleWeights), P, I, P, I, P, P, P, P,
                                           P, P]
            lib.oracle_forward.restype = I
            lib.oracle_route.argtypes = [ctypes.POINTER(OracleCfg), ctypes.POINTER(OracleWeights),
                                         P, I, P, I, P, P, P, P]
            lib.oracle_route.restype = I
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = I
            _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


# ----------------------------------------------------------------------------- formats
def bf16(b: int) -> float:
    return _get_lib().oracle_bf16(int(b))


def e2m1(code: int) -> float:
    return _get_lib().oracle_e2m1(int(code))


def e8m0(s: int) -> float:
    return _get_lib().oracle_e8m0(int(s))


def mxfp4_decode(blocks: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """blocks u8 [..., n_in/32, 16], scales u8 [..., n_in/32] -> fp64 [..., n_in]."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    nb = blocks.shape[-2]
    assert blocks.shape[-1] == 16 and scales.shape == blocks.shape[:-1]
    rows = int(np.prod(blocks.shape[:-2]))
    out = np.empty(blocks.shape[:-2] + (nb * 32,), np.float64)
    _get_lib().oracle_mxfp4_decode(_p(blocks), _p(scales), rows, nb * 32, _p(out))
    return out


# ----------------------------------------------------------------------------- routing
def select_topk(keys, k: int) -> np.ndarray:
    keys = np.ascontiguousarray(keys, dtype=np.float64)
    ids = np.empty(k, np.int32)
    _get_lib().oracle_select_topk(_p(keys), keys.shape[0], k, _p(ids))
    return ids


@dataclasses.dataclass
class Gating:
    """The oracle's view of the layer configuration."""
    d_model: int
    n_experts: int
    top_k: int
    expert_ff: int
    shared_ff: int = 0
    gating: int = 0          # 0 softmax->top-k->renorm, 1 top-k->softmax
    act: int = 0             # 0 SwiGLU, 1 clamped GLU
    wfmt: int = 0            # 0 bf16, 1 MXFP4
    norm_topk_prob: int = 1
    interleaved: int = 0
    scale: float = 1.0
    limit: float = 7.0
    alpha: float = 1.702
    rms_norm: int = 0        # 1: the MoE runs on RMSNorm(x) (needs layer.norm_w)
    residual: int = 0        # 1: y = x + MoE(...)
    rms_eps: float = 1e-6

    def c(self) -> OracleCfg:
        return OracleCfg(**dataclasses.asdict(self))


def gating_for(spec) -> Gating:
    """Oracle configuration for a moe_inputs.LayerSpec."""
    if spec.family == "qwen":
        return Gating(spec.d_model, spec.n_experts, spec.top_k, spec.expert_ff, spec.shared_ff,
                      gating=0, act=0, wfmt=0, norm_topk_prob=spec.norm_topk_prob, interleaved=0,
                      scale=spec.expert_weights_scale)
    return Gating(spec.d_model, spec.n_experts, spec.top_k, spec.expert_ff, spec.shared_ff,
                  gating=1, act=1, wfmt=1, norm_topk_prob=1, interleaved=1,
                  scale=spec.expert_weights_scale)


def route_from_logits(g: Gating, logits: np.ndarray):
    """Routing of caller-given logits [T, E] (fp64 holding any values, e.g. fp32 ones)."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    T = logits.shape[0]
    ids = np.empty((T, g.top_k), np.int32)
    w = np.empty((T, g.top_k), np.float64)
    c = g.c()
    _get_lib().oracle_route_from_logits(ctypes.byref(c), _p(logits), T, _p(ids), _p(w))
    return ids, w


# ----------------------------------------------------------------------------- forward
@dataclasses.dataclass
class OracleResult:
    tokens: np.ndarray   # [n] token indices evaluated
    y: np.ndarray        # [n, d] fp64
    ids: np.ndarray      # [n, k] int32, selection order
    w: np.ndarray        # [n, k] fp64 routing weights
    sgate: np.ndarray    # [n] fp64 (0 without shared expert)
    logits: np.ndarray   # [n, E] fp64
    n_nan: int


def weights_of(layer) -> tuple:
    """OracleWeights for a moe_inputs.Layer (returns the struct and the arrays it points to)."""
    keep = []

    def p(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        keep.append(a)
        return a.ctypes.data

    W = OracleWeights(router_w=p(layer.router_w), router_b=p(layer.router_b), gate=p(layer.gate),
                      up=p(layer.up), gate_up=p(getattr(layer, "gate_up", None)), down=p(layer.down),
                      gu_blocks=p(layer.gu_blocks), gu_scales=p(layer.gu_scales),
                      dn_blocks=p(layer.dn_blocks), dn_scales=p(layer.dn_scales),
                      gu_bias=p(layer.gu_bias), dn_bias=p(layer.dn_bias), sh_gate=p(layer.sh_gate),
                      sh_up=p(layer.sh_up), sh_down=p(layer.sh_down),
                      sh_gate_inp=p(layer.sh_gate_inp), norm_w=p(getattr(layer, "norm_w", None)))
    return W, keep


def forward(g: Gating, layer, tokens=None, forced_ids=None, x: Optional[np.ndarray] = None
            ) -> OracleResult:
    """Evaluate the layer for `tokens` (default: all rows of x)."""
    x = np.ascontiguousarray(layer.x if x is None else x, dtype=np.uint16)
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(
        tokens, dtype=np.int32)
    n = tokens.shape[0]
    assert n == 0 or (tokens.min() >= 0 and tokens.max() < T)
    if forced_ids is not None:
        forced_ids = np.ascontiguousarray(forced_ids, dtype=np.int32)
        assert forced_ids.shape == (n, g.top_k)
    y = np.zeros((n, g.d_model), np.float64)
    ids = np.zeros((n, g.top_k), np.int32)
    w = np.zeros((n, g.top_k), np.float64)
    sg = np.zeros(n, np.float64)
    lg = np.zeros((n, g.n_experts), np.float64)
    W, keep = weights_of(layer)
    c = g.c()
    nn = _get_lib().oracle_forward(ctypes.byref(c), ctypes.byref(W), _p(x), T, _p(tokens), n,
                                   _p(forced_ids), _p(y), _p(ids), _p(w), _p(sg), _p(lg))
    del keep
    return OracleResult(tokens, y, ids, w, sg, lg, nn)


def route(g: Gating, layer, tokens=None, x: Optional[np.ndarray] = None) -> OracleResult:
    """Routing only (logits, ids, weights, shared gate) for `tokens`; y is left empty."""
    x = np.ascontiguousarray(layer.x if x is None else x, dtype=np.uint16)
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(
        tokens, dtype=np.int32)
    n = tokens.shape[0]
    ids = np.zeros((n, g.top_k), np.int32)
    w = np.zeros((n, g.top_k), np.float64)
    sg = np.zeros(n, np.float64)
    lg = np.zeros((n, g.n_experts), np.float64)
    W, keep = weights_of(layer)
    c = g.c()
    nn = _get_lib().oracle_route(ctypes.byref(c), ctypes.byref(W), _p(x), T, _p(tokens), n,
                                 _p(ids), _p(w), _p(sg), _p(lg))
    del keep
    return OracleResult(tokens, np.zeros((n, 0)), ids, w, sg, lg, nn)


def num_threads() -> int:
    return _get_lib().oracle_num_threads()


def near_tie_tokens(logits: np.ndarray, ids: np.ndarray, eps: float = 1e-5) -> np.ndarray:
    """Boolean [n]: the token's selection is within `eps` of a tie.

    True when the gap between the k-th and (k+1)-th largest logit, or between two
    adjacent selected logits, is below eps (selection or order may then legitimately
    differ between fp32 and fp64 logits).
    """
    n, k = ids.shape
    s = -np.sort(-logits, axis=1)
    gap_k = s[:, k - 1] - s[:, k] if logits.shape[1] > k else np.full(n, np.inf)
    sel = np.take_along_axis(logits, ids.astype(np.int64), axis=1)
    gap_adj = np.min(np.abs(np.diff(sel, axis=1)), axis=1) if k > 1 else np.full(n, np.inf)
    return (gap_k < eps) | (gap_adj < eps)
