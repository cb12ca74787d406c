"""Seeded synthetic inputs for the sparse MoE FFN layer (shared by oracle and CUDA tests).

This module holds no arithmetic of the MoE method: it only produces the layer's
input tensors (activations, router, expert weights) from a counter-based
generator written in ``gen.c`` (splitmix64 + Box-Muller, definition in that
file's header).  Both the fp64 oracle and the CUDA path consume the same bytes.

Workloads follow the layer shapes on the pages:
  * Qwen3.5-MoE "mini" layer: d_model 2048, 256 experts, top-8, expert/shared
    FF 512, bf16 SwiGLU experts plus a sigmoid-gated shared expert
    (qwen35moe Forward-Pass Design, "Config (mini)" table and "Shared-expert
    MoE FFN" section).
  * gpt-oss-20b layer: d_model 2880, 32 experts, top-4, expert FF 2880, MXFP4
    expert weights with E8M0 scales per 32 inputs (Phase 19: MoE gpt-oss-20b,
    section 1 "architecture" and the tensor-layout listing in section 2).

Tensor layouts are row = output, column = input (y = x W^T), with per-expert
tensors stacked on a leading expert axis.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading
from typing import Optional

import numpy as np

SEED = 0x9E3779B9          # the golden-vector seed of the qwen35moe golden README
LAYER_STREAM = 1_000_000   # stream offset for layer-level tensors (router, x, shared)

# tensor slots inside the layer-level stream
SLOT_ROUTER_W, SLOT_SHARED_GATE_INP, SLOT_ROUTER_BIAS, SLOT_X = 0, 1, 2, 3
SLOT_SH_GATE, SLOT_SH_UP, SLOT_SH_DOWN = 4, 5, 6
SLOT_NORM_W = 7
# tensor slots inside an expert's stream (bf16 experts)
SLOT_E_GATE, SLOT_E_UP, SLOT_E_DOWN = 0, 1, 2
# tensor slots inside an expert's stream (MXFP4 experts)
SLOT_E_GU_BLOCKS, SLOT_E_GU_SCALES, SLOT_E_GU_BIAS = 0, 1, 2
SLOT_E_DN_BLOCKS, SLOT_E_DN_SCALES, SLOT_E_DN_BIAS = 3, 4, 5

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmoegen.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile gen.c into a shared library (gcc, OpenMP, no FP contraction)."""
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
            u64, u32, dbl, ptr = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_double, ctypes.c_void_p
            lib.gen_normal_bf16.argtypes = [u64, u32, u64, u64, dbl, ptr]
            lib.gen_normal_f64.argtypes = [u64, u32, u64, u64, ptr]
            lib.gen_uniform_f64.argtypes = [u64, u32, u64, u64, ptr]
            lib.gen_bytes.argtypes = [u64, u32, u64, ptr]
            lib.gen_int_range_u8.argtypes = [u64, u32, u64, u32, u32, ptr]
            lib.gen_draw.argtypes = [u64, u32, u64]
            lib.gen_draw.restype = u64
            for f in (lib.gen_normal_bf16, lib.gen_normal_f64, lib.gen_uniform_f64, lib.gen_bytes,
                      lib.gen_int_range_u8):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------------------- primitives
def normal_bf16(key: int, slot: int, shape, std: float, first: int = 0,
                out: Optional[np.ndarray] = None) -> np.ndarray:
    n = int(np.prod(shape))
    a = np.empty(shape, dtype=np.uint16) if out is None else out
    _get_lib().gen_normal_bf16(key & (2**64 - 1), slot, first, n, float(std), _ptr(a))
    return a


def normal_f64(key: int, slot: int, n: int, first: int = 0) -> np.ndarray:
    a = np.empty(n, dtype=np.float64)
    _get_lib().gen_normal_f64(key & (2**64 - 1), slot, first, n, _ptr(a))
    return a


def uniform_f64(key: int, slot: int, n: int, first: int = 0) -> np.ndarray:
    a = np.empty(n, dtype=np.float64)
    _get_lib().gen_uniform_f64(key & (2**64 - 1), slot, first, n, _ptr(a))
    return a


def random_bytes(key: int, slot: int, shape, out: Optional[np.ndarray] = None) -> np.ndarray:
    a = np.empty(shape, dtype=np.uint8) if out is None else out
    _get_lib().gen_bytes(key & (2**64 - 1), slot, int(np.prod(shape)), _ptr(a))
    return a


def int_range_u8(key: int, slot: int, shape, lo: int, hi: int,
                 out: Optional[np.ndarray] = None) -> np.ndarray:
    assert 0 <= lo <= hi <= 255
    a = np.empty(shape, dtype=np.uint8) if out is None else out
    _get_lib().gen_int_range_u8(key & (2**64 - 1), slot, int(np.prod(shape)), lo, hi, _ptr(a))
    return a


def f64_to_bf16(v) -> np.ndarray:
    """Round fp64 values to bf16 bit patterns: first to fp32 (RNE), then RNE to 16 bits."""
    with np.errstate(over="ignore"):          # beyond the fp32 range: +-inf, as in bf16
        f = np.asarray(v, dtype=np.float64).astype(np.float32)
    shape = f.shape
    u = np.ascontiguousarray(f.reshape(-1)).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r.reshape(shape)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------- workloads
@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """Shape and value recipe of one synthetic MoE layer workload."""
    name: str
    family: str                  # "qwen" (softmax/renorm, SwiGLU, shared) | "gptoss" (bias, MXFP4)
    d_model: int
    n_experts: int
    top_k: int
    expert_ff: int
    shared_ff: int               # 0: no shared expert
    tokens: int
    bias: Optional[tuple] = None  # None | ("normal", std) | ("zipf", s)
    scale_lo: int = 118          # E8M0 scale range for MXFP4 weights
    scale_hi: int = 126
    expert_weights_scale: float = 1.0
    norm_topk_prob: int = 1
    seed: int = SEED

    @property
    def mxfp4(self) -> bool:
        return self.family == "gptoss"

    def with_tokens(self, T: int) -> "LayerSpec":
        return dataclasses.replace(self, tokens=T)


QWEN_MINI = dict(family="qwen", d_model=2048, n_experts=256, top_k=8, expert_ff=512, shared_ff=512)
GPTOSS_20B = dict(family="gptoss", d_model=2880, n_experts=32, top_k=4, expert_ff=2880, shared_ff=0)

# The five workloads, smallest first.
WORKLOADS = {
    "qwen35_mini_moe_decode_t8": LayerSpec("qwen35_mini_moe_decode_t8", tokens=8, **QWEN_MINI),
    "qwen35_mini_moe_decode_t64": LayerSpec("qwen35_mini_moe_decode_t64", tokens=64, **QWEN_MINI),
    "qwen35_mini_moe_prefill_t4096": LayerSpec("qwen35_mini_moe_prefill_t4096", tokens=4096,
                                               bias=("normal", 0.5), **QWEN_MINI),
    "gptoss_20b_moe_decode_t32": LayerSpec("gptoss_20b_moe_decode_t32", tokens=32,
                                           bias=("normal", 0.1), **GPTOSS_20B),
    "gptoss_20b_moe_prefill_t8192": LayerSpec("gptoss_20b_moe_prefill_t8192", tokens=8192,
                                              bias=("zipf", 1.1), **GPTOSS_20B),
}
WORKLOAD_ORDER = list(WORKLOADS)


@dataclasses.dataclass
class Layer:
    """Host copies of every input tensor of one layer (bf16 as uint16 bit patterns)."""
    spec: LayerSpec
    x: np.ndarray                     # [T, d] bf16
    router_w: np.ndarray              # [E, d] bf16
    router_b: Optional[np.ndarray]    # [E] bf16 or None
    # bf16 experts (qwen)
    gate: Optional[np.ndarray] = None   # [E, ff, d]
    up: Optional[np.ndarray] = None     # [E, ff, d]
    down: Optional[np.ndarray] = None   # [E, d, ff]
    gate_up: Optional[np.ndarray] = None  # [E, 2ff, d] bf16, interleaved rows (gate even, up odd)
    # MXFP4 experts (gpt-oss): gate_up rows interleave gate (even) / up (odd)
    gu_blocks: Optional[np.ndarray] = None   # [E, 2ff, d/32, 16] u8
    gu_scales: Optional[np.ndarray] = None   # [E, 2ff, d/32] u8
    gu_bias: Optional[np.ndarray] = None     # [E, 2ff] bf16
    dn_blocks: Optional[np.ndarray] = None   # [E, d, ff/32, 16] u8
    dn_scales: Optional[np.ndarray] = None   # [E, d, ff/32] u8
    dn_bias: Optional[np.ndarray] = None     # [E, d] bf16
    # shared expert (qwen)
    sh_gate: Optional[np.ndarray] = None     # [sff, d]
    sh_up: Optional[np.ndarray] = None       # [sff, d]
    sh_down: Optional[np.ndarray] = None     # [d, sff]
    sh_gate_inp: Optional[np.ndarray] = None  # [d]
    # RMSNorm weight before the MoE (layers run with the norm / residual steps)
    norm_w: Optional[np.ndarray] = None      # [d] bf16

    @property
    def T(self) -> int:
        return self.x.shape[0]


def make_x(spec: LayerSpec, T: Optional[int] = None) -> np.ndarray:
    """x ~ N(0,1) bf16 [T, d]; token t of any T is the same row (prefix property)."""
    T = spec.tokens if T is None else T
    return normal_bf16(spec.seed + LAYER_STREAM, SLOT_X, (T, spec.d_model), 1.0)


def make_router_bias(spec: LayerSpec) -> Optional[np.ndarray]:
    if spec.bias is None:
        return None
    kind, param = spec.bias
    key = spec.seed + LAYER_STREAM
    if kind == "normal":
        return normal_bf16(key, SLOT_ROUTER_BIAS, (spec.n_experts,), param)
    if kind == "zipf":
        # Zipf(s) expert popularity: expert e gets logit bias -s*ln(rank_e) (the log of an
        # unnormalised Zipf weight rank^-s); ranks are a seeded permutation of 1..E.
        u = uniform_f64(key, SLOT_ROUTER_BIAS, spec.n_experts)
        rank = np.empty(spec.n_experts, dtype=np.int64)
        rank[np.argsort(u, kind="stable")] = np.arange(1, spec.n_experts + 1)
        return f64_to_bf16(-param * np.log(rank.astype(np.float64)))
    raise ValueError(kind)


def make_layer(spec: LayerSpec, T: Optional[int] = None, experts: Optional[list] = None,
               zero_x: bool = False) -> Layer:
    """Generate every input tensor of `spec` (T tokens; default spec.tokens).

    `experts`, if given, restricts which experts' weights are generated (the others stay
    zero) -- only for tests that know the routing in advance.
    """
    T = spec.tokens if T is None else T
    d, E, ff, sff = spec.d_model, spec.n_experts, spec.expert_ff, spec.shared_ff
    key = spec.seed + LAYER_STREAM
    x = np.zeros((T, d), np.uint16) if zero_x else make_x(spec, T)
    lay = Layer(spec=spec, x=x,
                router_w=normal_bf16(key, SLOT_ROUTER_W, (E, d), 1.0 / math.sqrt(d)),
                router_b=make_router_bias(spec))
    which = range(E) if experts is None else experts
    if spec.family == "qwen":
        lay.gate = np.zeros((E, ff, d), np.uint16)
        lay.up = np.zeros((E, ff, d), np.uint16)
        lay.down = np.zeros((E, d, ff), np.uint16)
        for e in which:
            ke = spec.seed + e
            normal_bf16(ke, SLOT_E_GATE, (ff, d), 1.0 / math.sqrt(d), out=lay.gate[e])
            normal_bf16(ke, SLOT_E_UP, (ff, d), 1.0 / math.sqrt(d), out=lay.up[e])
            normal_bf16(ke, SLOT_E_DOWN, (d, ff), 1.0 / math.sqrt(ff), out=lay.down[e])
    else:
        assert d % 32 == 0 and ff % 32 == 0
        lay.gu_blocks = np.zeros((E, 2 * ff, d // 32, 16), np.uint8)
        lay.gu_scales = np.zeros((E, 2 * ff, d // 32), np.uint8)
        lay.gu_bias = np.zeros((E, 2 * ff), np.uint16)
        lay.dn_blocks = np.zeros((E, d, ff // 32, 16), np.uint8)
        lay.dn_scales = np.zeros((E, d, ff // 32), np.uint8)
        lay.dn_bias = np.zeros((E, d), np.uint16)
        for e in which:
            ke = spec.seed + e
            random_bytes(ke, SLOT_E_GU_BLOCKS, lay.gu_blocks[e].shape, out=lay.gu_blocks[e])
            int_range_u8(ke, SLOT_E_GU_SCALES, lay.gu_scales[e].shape, spec.scale_lo,
                         spec.scale_hi, out=lay.gu_scales[e])
            normal_bf16(ke, SLOT_E_GU_BIAS, (2 * ff,), 0.02, out=lay.gu_bias[e])
            random_bytes(ke, SLOT_E_DN_BLOCKS, lay.dn_blocks[e].shape, out=lay.dn_blocks[e])
            int_range_u8(ke, SLOT_E_DN_SCALES, lay.dn_scales[e].shape, spec.scale_lo,
                         spec.scale_hi, out=lay.dn_scales[e])
            normal_bf16(ke, SLOT_E_DN_BIAS, (d,), 0.02, out=lay.dn_bias[e])
    if sff > 0:
        lay.sh_gate_inp = normal_bf16(key, SLOT_SHARED_GATE_INP, (d,), 1.0 / math.sqrt(d))
        lay.sh_gate = normal_bf16(key, SLOT_SH_GATE, (sff, d), 1.0 / math.sqrt(d))
        lay.sh_up = normal_bf16(key, SLOT_SH_UP, (sff, d), 1.0 / math.sqrt(d))
        lay.sh_down = normal_bf16(key, SLOT_SH_DOWN, (d, sff), 1.0 / math.sqrt(sff))
    return lay


def make_norm_w(spec: LayerSpec) -> np.ndarray:
    """RMSNorm weight bf16 [d] ~ 1 + N(0, 0.1): a norm weight near 1, as the pages
    describe the model's (QK-norm weights of about 1 +- 0.1)."""
    z = normal_f64(spec.seed + LAYER_STREAM, SLOT_NORM_W, spec.d_model)
    return f64_to_bf16(1.0 + 0.1 * z)


def small_spec(family: str, d: int, E: int, k: int, ff: int, sff: int, T: int,
               bias=None, **kw) -> LayerSpec:
    """A reduced-size layer with the same value distributions (for tests)."""
    return LayerSpec(f"{family}_d{d}_e{E}_k{k}_ff{ff}_t{T}", family=family, d_model=d,
                     n_experts=E, top_k=k, expert_ff=ff, shared_ff=sff, tokens=T, bias=bias, **kw)
