"""GB300 (sm_103a) sparse Mixture-of-Experts FFN forward pass -- Python binding.

A thin ctypes layer over ``libmoe.so`` whose functions carry the C ABI's names
(``include/moe.h``): it checks tensor placement, passes device pointers and the
current CUDA stream, and raises ``MoeError`` on a non-zero status.  All of the
layer's arithmetic runs in the library's CUDA kernels; PyTorch only provides device
memory and streams.  There is no fallback: if the library is missing, importing
this package fails.

Two gating conventions:
  * Qwen3.5-MoE ("qwen35moe - Forward-Pass Design", section "Shared-expert MoE FFN";
    "qwen35moe CPU-reference golden vectors", Kernel 4): ``qwen_cfg``.
  * gpt-oss ("Phase 19: MoE - gpt-oss-20b", sections 2 and 3): ``gptoss_cfg``.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

from . import build as _build

LIB_PATH = _build.LIB

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED",
                -3: "MOE_ERR_WORKSPACE", -4: "MOE_ERR_ALIGNMENT", -5: "MOE_ERR_CUDA",
                -6: "MOE_ERR_DEVICE_CHECK", -7: "MOE_ERR_TIMEOUT"}
GATING_SOFTMAX_TOPK_RENORM, GATING_TOPK_SOFTMAX = 0, 1
ACT_SWIGLU, ACT_CLAMPED_GLU = 0, 1
WFMT_BF16, WFMT_MXFP4 = 0, 1
PATH_AUTO, PATH_DECODE, PATH_PREFILL, PATH_DECODE_REGISTERS = 0, 1, 2, 3


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({_lib.moe_status_string(status).decode()})")


class MoeCfg(ctypes.Structure):
    """moe_cfg_t."""
    _fields_ = [("d_model", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("expert_ff", ctypes.c_int32),
                ("shared_ff", ctypes.c_int32), ("gating", ctypes.c_int32),
                ("act", ctypes.c_int32), ("wfmt", ctypes.c_int32),
                ("interleaved_gate_up", ctypes.c_int32), ("norm_topk_prob", ctypes.c_int32),
                ("expert_weights_scale", ctypes.c_float), ("glu_limit", ctypes.c_float),
                ("glu_alpha", ctypes.c_float), ("path", ctypes.c_int32),
                ("y_fp32", ctypes.c_int32), ("rms_norm", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("residual", ctypes.c_int32),
                ("deterministic", ctypes.c_int32), ("reserved", ctypes.c_int32 * 2)]

    def replace(self, **kw) -> "MoeCfg":
        c = MoeCfg()
        ctypes.memmove(ctypes.byref(c), ctypes.byref(self), ctypes.sizeof(MoeCfg))
        for k, v in kw.items():
            setattr(c, k, v)
        return c


class _Router(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("norm_w", ctypes.c_void_p)]


class _Experts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate", "up", "gate_up", "gate_up_scales",
                                                "gate_up_bias", "down", "down_scales",
                                                "down_bias")]


class _Shared(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate", "up", "down", "gate_inp")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, C = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(MoeCfg)
    lib.moe_workspace_bytes.argtypes = [C, ctypes.c_int32]
    lib.moe_workspace_bytes.restype = ctypes.c_size_t
    lib.moe_select_path.argtypes = [C, ctypes.c_int32]
    lib.moe_kernel_plan.restype = I
    lib.moe_kernel_plan.argtypes = [C, ctypes.c_int32]
    lib.moe_select_path.restype = I
    lib.moe_route.argtypes = [C, P, ctypes.c_int32, ctypes.POINTER(_Router),
                              ctypes.POINTER(_Shared), P, P, P, P, P, ctypes.c_size_t, P]
    lib.moe_route.restype = I
    lib.moe_topk_from_logits.argtypes = [C, P, ctypes.c_int32, P, P, P]
    lib.moe_topk_from_logits.restype = I
    lib.moe_group_by_expert.argtypes = [C, P, ctypes.c_int32, P, P, P, P, ctypes.c_size_t, P]
    lib.moe_group_by_expert.restype = I
    lib.moe_ffn_forward.argtypes = [C, P, ctypes.c_int32, ctypes.POINTER(_Router),
                                    ctypes.POINTER(_Experts), ctypes.POINTER(_Shared), P, P, P, P,
                                    ctypes.c_size_t, P]
    lib.moe_ffn_forward.restype = I
    lib.moe_ffn_forward_routed.argtypes = [C, P, ctypes.c_int32, P, P, P,
                                           ctypes.POINTER(_Experts), ctypes.POINTER(_Shared), P, P,
                                           ctypes.c_size_t, P]
    lib.moe_ffn_forward_routed.restype = I
    lib.moe_ffn_forward_host.argtypes = [C, P, ctypes.c_int32, ctypes.POINTER(_Router),
                                         ctypes.POINTER(_Experts), ctypes.POINTER(_Shared), P, P,
                                         ctypes.c_size_t, P]
    lib.moe_ffn_forward_host.restype = I
    lib.moe_ffn_forward_noalloc.argtypes = [C, P, ctypes.c_int32, ctypes.POINTER(_Router),
                                            ctypes.POINTER(_Experts), ctypes.POINTER(_Shared), P,
                                            P, P, P]
    lib.moe_ffn_forward_noalloc.restype = I
    lib.moe_noalloc_workspace_bytes.argtypes = []
    lib.moe_noalloc_workspace_bytes.restype = ctypes.c_size_t
    lib.moe_noalloc_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.moe_noalloc_device_status.restype = I
    lib.moe_mxfp4_to_bf16.argtypes = [P, P, ctypes.c_int64, ctypes.c_int32, P, P]
    lib.moe_mxfp4_to_bf16.restype = I
    lib.moe_set_phase_events.argtypes = [P, ctypes.c_int32]
    lib.moe_set_phase_events.restype = I
    lib.moe_test_set_wait_limit.argtypes = [ctypes.c_uint32, ctypes.c_int32]
    lib.moe_test_set_wait_limit.restype = I
    lib.moe_test_set_decode_fusion.argtypes = [ctypes.c_int32]
    lib.moe_test_set_decode_fusion.restype = I
    lib.moe_device_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
    lib.moe_device_status.restype = I
    lib.moe_status_string.argtypes = [I]
    lib.moe_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()
EXPORTED = ("moe_workspace_bytes", "moe_select_path", "moe_kernel_plan", "moe_route", "moe_topk_from_logits",
            "moe_group_by_expert", "moe_ffn_forward", "moe_ffn_forward_routed", "moe_ffn_forward_host",
            "moe_ffn_forward_noalloc", "moe_noalloc_workspace_bytes", "moe_noalloc_device_status",
            "moe_mxfp4_to_bf16", "moe_set_phase_events", "moe_test_set_wait_limit", "moe_test_set_decode_fusion",
            "moe_device_status",
            "moe_status_string")
PHASES = ("router_logits", "router_select", "permute", "gate_up", "down", "combine")


# ----------------------------------------------------------------------------- configs
def qwen_cfg(d_model=2048, n_experts=256, top_k=8, expert_ff=512, shared_ff=512,
             expert_weights_scale=1.0, norm_topk_prob=1, path=PATH_AUTO) -> MoeCfg:
    """Softmax -> top-k -> renorm x scale gating, bf16 SwiGLU experts, shared expert."""
    return MoeCfg(d_model=d_model, n_experts=n_experts, top_k=top_k, expert_ff=expert_ff,
                  shared_ff=shared_ff, gating=GATING_SOFTMAX_TOPK_RENORM, act=ACT_SWIGLU,
                  wfmt=WFMT_BF16, interleaved_gate_up=0, norm_topk_prob=norm_topk_prob,
                  expert_weights_scale=expert_weights_scale, glu_limit=7.0, glu_alpha=1.702,
                  path=path)


def gptoss_cfg(d_model=2880, n_experts=32, top_k=4, expert_ff=2880, glu_limit=7.0,
               glu_alpha=1.702, path=PATH_AUTO) -> MoeCfg:
    """Biased top-k -> softmax gating, MXFP4 interleaved gate_up, clamped GLU, biases."""
    return MoeCfg(d_model=d_model, n_experts=n_experts, top_k=top_k, expert_ff=expert_ff,
                  shared_ff=0, gating=GATING_TOPK_SOFTMAX, act=ACT_CLAMPED_GLU, wfmt=WFMT_MXFP4,
                  interleaved_gate_up=1, norm_topk_prob=1, expert_weights_scale=1.0,
                  glu_limit=glu_limit, glu_alpha=glu_alpha, path=path)


# ----------------------------------------------------------------------------- weights
@dataclasses.dataclass
class Router:
    w: torch.Tensor                       # bf16 [E, d]
    bias: Optional[torch.Tensor] = None   # bf16 [E]
    norm_w: Optional[torch.Tensor] = None  # bf16 [d]: RMSNorm weight (cfg.rms_norm)


@dataclasses.dataclass
class Experts:
    gate: Optional[torch.Tensor] = None            # bf16 [E, ff, d]
    up: Optional[torch.Tensor] = None              # bf16 [E, ff, d]
    gate_up: Optional[torch.Tensor] = None         # bf16 [E, 2ff, d] | u8 [E, 2ff, d/32, 16]
    gate_up_scales: Optional[torch.Tensor] = None  # u8 [E, 2ff, d/32]
    gate_up_bias: Optional[torch.Tensor] = None    # bf16 [E, 2ff]
    down: Optional[torch.Tensor] = None            # bf16 [E, d, ff] | u8 [E, d, ff/32, 16]
    down_scales: Optional[torch.Tensor] = None     # u8 [E, d, ff/32]
    down_bias: Optional[torch.Tensor] = None       # bf16 [E, d]


@dataclasses.dataclass
class Shared:
    gate: torch.Tensor       # bf16 [sff, d]
    up: torch.Tensor         # bf16 [sff, d]
    down: torch.Tensor       # bf16 [d, sff]
    gate_inp: torch.Tensor   # bf16 [d]


def _ptr(t: Optional[torch.Tensor], name: str = "tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _router(r: Router) -> _Router:
    return _Router(_ptr(r.w, "router.w"), _ptr(r.bias, "router.bias"),
                   _ptr(r.norm_w, "router.norm_w"))


def _experts(e: Experts) -> _Experts:
    return _Experts(**{f.name: _ptr(getattr(e, f.name), f"experts.{f.name}")
                       for f in dataclasses.fields(Experts)})


def _shared(s: Optional[Shared]):
    if s is None:
        return None
    return ctypes.byref(_Shared(_ptr(s.gate, "shared.gate"), _ptr(s.up, "shared.up"),
                                _ptr(s.down, "shared.down"), _ptr(s.gate_inp, "shared.gate_inp")))


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


# ----------------------------------------------------------------------------- entry points
def moe_workspace_bytes(cfg: MoeCfg, T: int) -> int:
    return int(_lib.moe_workspace_bytes(ctypes.byref(cfg), T))


def moe_select_path(cfg: MoeCfg, T: int) -> int:
    st = _lib.moe_select_path(ctypes.byref(cfg), T)
    if st < 0:
        raise MoeError(st, "moe_select_path")
    return st


PLAN_DECODE_WARP, PLAN_DECODE_RING, PLAN_PREFILL_BF16, PLAN_PREFILL_F16, PLAN_DECODE_FUSED = 1, 2, 3, 4, 5
PLAN_NAMES = {1: "decode: warp MMAs, register-held weight loads",
              2: "decode: warp MMAs, TMA-fed weight ring",
              3: "prefill: tcgen05 grouped GEMMs, bf16 operands",
              4: "prefill: tcgen05 grouped GEMMs, f16 operands (MXFP4, two m tiles per weight tile)",
              5: "decode: warp MMAs, register-held weight loads, gate_up and down in one launch"}


def moe_kernel_plan(cfg: MoeCfg, T: int) -> int:
    st = _lib.moe_kernel_plan(ctypes.byref(cfg), T)
    if st < 0:
        raise MoeError(st, "moe_kernel_plan")
    return st


def workspace(cfg: MoeCfg, T: int, device=None) -> torch.Tensor:
    """A device byte buffer of moe_workspace_bytes(cfg, T) (torch-allocated)."""
    n = moe_workspace_bytes(cfg, T)
    if n == 0:
        raise MoeError(-1, "moe_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def moe_route(cfg: MoeCfg, x: torch.Tensor, router: Router, shared: Optional[Shared] = None,
              topk_ids=None, topk_w=None, sgate=None, logits=None, ws=None, stream=None):
    """Router only.  Returns (topk_ids int32 [T,k], topk_w fp32 [T,k], sgate | None, logits | None)."""
    T = x.shape[0]
    dev = x.device
    topk_ids = torch.empty((T, cfg.top_k), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    topk_w = torch.empty((T, cfg.top_k), dtype=torch.float32, device=dev) if topk_w is None else topk_w
    ws = workspace(cfg, T, dev) if ws is None else ws
    _check(_lib.moe_route(ctypes.byref(cfg), _ptr(x, "x"), T, ctypes.byref(_router(router)),
                          _shared(shared), _ptr(topk_ids), _ptr(topk_w), _ptr(sgate), _ptr(logits),
                          _ptr(ws), ws.numel(), _stream(stream)), "moe_route")
    return topk_ids, topk_w, sgate, logits


def moe_topk_from_logits(cfg: MoeCfg, logits: torch.Tensor, topk_ids=None, topk_w=None,
                         stream=None):
    T = logits.shape[0]
    dev = logits.device
    topk_ids = torch.empty((T, cfg.top_k), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    topk_w = torch.empty((T, cfg.top_k), dtype=torch.float32, device=dev) if topk_w is None else topk_w
    _check(_lib.moe_topk_from_logits(ctypes.byref(cfg), _ptr(logits, "logits"), T, _ptr(topk_ids),
                                     _ptr(topk_w), _stream(stream)), "moe_topk_from_logits")
    return topk_ids, topk_w


def moe_group_by_expert(cfg: MoeCfg, topk_ids: torch.Tensor, counts=None, offsets=None, perm=None,
                        ws=None, stream=None):
    """Stable grouping of the slots t*k + j by expert: (counts [E], offsets [E+1], perm [T*k])."""
    T = topk_ids.shape[0]
    dev = topk_ids.device
    E = cfg.n_experts
    counts = torch.empty(E, dtype=torch.int32, device=dev) if counts is None else counts
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if offsets is None else offsets
    perm = torch.empty(max(T * cfg.top_k, 1), dtype=torch.int32, device=dev) if perm is None else perm
    ws = workspace(cfg, T, dev) if ws is None else ws
    _check(_lib.moe_group_by_expert(ctypes.byref(cfg), _ptr(topk_ids, "topk_ids"), T, _ptr(counts, "counts"),
                                    _ptr(offsets, "offsets"), _ptr(perm, "perm"), _ptr(ws), ws.numel(),
                                    _stream(stream)), "moe_group_by_expert")
    return counts, offsets, perm


def moe_ffn_forward(cfg: MoeCfg, x: torch.Tensor, router: Router, experts: Experts,
                    shared: Optional[Shared] = None, y=None, topk_ids=None, topk_w=None, ws=None,
                    stream=None) -> torch.Tensor:
    """The whole layer; returns y [T, d] (bf16, or fp32 when cfg.y_fp32)."""
    T = x.shape[0]
    if y is None:
        y = torch.empty(x.shape, dtype=torch.float32 if cfg.y_fp32 else torch.bfloat16,
                        device=x.device)
    ws = workspace(cfg, T, x.device) if ws is None else ws
    _check(_lib.moe_ffn_forward(ctypes.byref(cfg), _ptr(x, "x"), T, ctypes.byref(_router(router)),
                                ctypes.byref(_experts(experts)), _shared(shared), _ptr(y, "y"),
                                _ptr(topk_ids), _ptr(topk_w), _ptr(ws), ws.numel(),
                                _stream(stream)), "moe_ffn_forward")
    return y


def moe_noalloc_workspace_bytes() -> int:
    """Size of the library's own device array that moe_ffn_forward_noalloc works in."""
    return int(_lib.moe_noalloc_workspace_bytes())


NOALLOC_WORKSPACE_BYTES = moe_noalloc_workspace_bytes()


def moe_ffn_forward_noalloc(cfg: MoeCfg, x: torch.Tensor, router: Router, experts: Experts,
                            shared: Optional[Shared] = None, y=None, topk_ids=None, topk_w=None,
                            stream=None) -> torch.Tensor:
    """moe_ffn_forward for callers that cannot allocate device memory: the library's own
    device array (NOALLOC_WORKSPACE_BYTES) serves as workspace (see include/moe.h).  Only
    `y` is allocated here when it is not passed in."""
    T = x.shape[0]
    if y is None:
        y = torch.empty(x.shape, dtype=torch.float32 if cfg.y_fp32 else torch.bfloat16,
                        device=x.device)
    _check(_lib.moe_ffn_forward_noalloc(ctypes.byref(cfg), _ptr(x, "x"), T,
                                        ctypes.byref(_router(router)),
                                        ctypes.byref(_experts(experts)), _shared(shared),
                                        _ptr(y, "y"), _ptr(topk_ids), _ptr(topk_w),
                                        _stream(stream)), "moe_ffn_forward_noalloc")
    return y


def moe_ffn_forward_routed(cfg: MoeCfg, x: torch.Tensor, topk_ids: torch.Tensor,
                           topk_w: torch.Tensor, experts: Experts, shared: Optional[Shared] = None,
                           sgate=None, y=None, ws=None, stream=None) -> torch.Tensor:
    T = x.shape[0]
    if y is None:
        y = torch.empty(x.shape, dtype=torch.float32 if cfg.y_fp32 else torch.bfloat16,
                        device=x.device)
    ws = workspace(cfg, T, x.device) if ws is None else ws
    _check(_lib.moe_ffn_forward_routed(ctypes.byref(cfg), _ptr(x, "x"), T, _ptr(topk_ids),
                                       _ptr(topk_w), _ptr(sgate), ctypes.byref(_experts(experts)),
                                       _shared(shared), _ptr(y, "y"), _ptr(ws), ws.numel(),
                                       _stream(stream)), "moe_ffn_forward_routed")
    return y


def moe_ffn_forward_host(cfg: MoeCfg, x_host: torch.Tensor, router: Router, experts: Experts,
                         shared: Optional[Shared] = None, y_host=None, ws=None,
                         stream=None) -> torch.Tensor:
    """Host x in, host y out (pinned CPU tensors give full copy speed); synchronous."""
    if x_host.is_cuda:
        raise ValueError("x_host must be a CPU tensor")
    T = x_host.shape[0]
    if y_host is None:
        y_host = torch.empty(x_host.shape, dtype=torch.float32 if cfg.y_fp32 else torch.bfloat16)
    ws = workspace(cfg, T) if ws is None else ws
    _check(_lib.moe_ffn_forward_host(ctypes.byref(cfg), x_host.data_ptr(), T,
                                     ctypes.byref(_router(router)), ctypes.byref(_experts(experts)),
                                     _shared(shared), y_host.data_ptr(), _ptr(ws), ws.numel(),
                                     _stream(stream)), "moe_ffn_forward_host")
    return y_host


class BoundForwardHost:
    """moe_ffn_forward_host with its arguments marshalled once, for repeated steps.

    Each call runs one synchronous step exactly as moe_ffn_forward_host does (x_host's
    current contents are copied in, y_host receives the layer's output) but skips the
    per-call argument checks and ctypes marshalling.  The tensors given here must stay
    alive and keep their storage while the object is used.
    """

    def __init__(self, cfg: MoeCfg, x_host: torch.Tensor, router: Router, experts: Experts,
                 shared: Optional[Shared] = None, y_host=None, ws=None, stream=None):
        if x_host.is_cuda:
            raise ValueError("x_host must be a CPU tensor")
        T = x_host.shape[0]
        if y_host is None:
            y_host = torch.empty(x_host.shape, dtype=torch.float32 if cfg.y_fp32 else torch.bfloat16)
        self.ws = workspace(cfg, T) if ws is None else ws
        self.cfg, self.x_host, self.y_host = cfg, x_host, y_host
        self._keep = (router, experts, shared, _router(router), _experts(experts))
        self._args = (ctypes.byref(cfg), x_host.data_ptr(), T, ctypes.byref(self._keep[3]),
                      ctypes.byref(self._keep[4]), _shared(shared), y_host.data_ptr(), _ptr(self.ws),
                      self.ws.numel(), _stream(stream))
        self._fn = _lib.moe_ffn_forward_host

    def __call__(self) -> torch.Tensor:
        st = self._fn(*self._args)
        if st != MOE_OK:
            raise MoeError(st, "moe_ffn_forward_host")
        return self.y_host


def moe_mxfp4_to_bf16(blocks: torch.Tensor, scales: torch.Tensor, out=None,
                      stream=None) -> torch.Tensor:
    """blocks u8 [..., n_in/32, 16], scales u8 [..., n_in/32] -> bf16 [..., n_in]."""
    nb = blocks.shape[-2]
    rows = blocks.numel() // (nb * 16)
    out = torch.empty(tuple(blocks.shape[:-2]) + (nb * 32,), dtype=torch.bfloat16,
                      device=blocks.device) if out is None else out
    _check(_lib.moe_mxfp4_to_bf16(_ptr(blocks, "blocks"), _ptr(scales, "scales"), rows, nb * 32,
                                  _ptr(out, "out"), _stream(stream)), "moe_mxfp4_to_bf16")
    return out


_phase_keepalive = None


def moe_set_phase_events(events) -> None:
    """Record torch.cuda.Event objects (7 for every phase boundary, or 2 for start and
    end only; timing enabled) during later forward calls from this thread; None
    disables.  Each event is recorded once here first so that its CUDA handle exists."""
    global _phase_keepalive
    if events is None:
        _check(_lib.moe_set_phase_events(None, 0), "moe_set_phase_events")
        _phase_keepalive = None
        return
    for e in events:
        e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(_lib.moe_set_phase_events(arr, len(events)), "moe_set_phase_events")
    _phase_keepalive = (arr, events)


DEFAULT_WAIT_POLLS = 1 << 20


def moe_test_set_wait_limit(max_polls: int = DEFAULT_WAIT_POLLS, withhold_first_load: bool = False) -> None:
    """Test hook: the poll limit of the bounded device waits, and whether CTA 0's producer
    of the TMA-fed kernels skips its first load (see include/moe.h).  Synchronises."""
    _check(_lib.moe_test_set_wait_limit(max_polls, int(withhold_first_load)), "moe_test_set_wait_limit")


def moe_test_set_decode_fusion(enable: bool) -> None:
    """Test hook: whether bf16 decode with one-chunk items runs gate_up and down as one
    launch (the default) or as two (see include/moe.h).  Host-side only."""
    _check(_lib.moe_test_set_decode_fusion(int(bool(enable))), "moe_test_set_decode_fusion")


def moe_device_status(ws: torch.Tensor, stream=None):
    """(status, raw bits) of the device check word; synchronises the stream and clears it."""
    bits = ctypes.c_uint32(0)
    st = _lib.moe_device_status(_ptr(ws), _stream(stream), ctypes.byref(bits))
    return st, bits.value


def moe_noalloc_device_status(stream=None):
    """(status, raw bits) of the device check word of the last moe_ffn_forward_noalloc
    call in the current context; synchronises the stream and clears it."""
    bits = ctypes.c_uint32(0)
    st = _lib.moe_noalloc_device_status(_stream(stream), ctypes.byref(bits))
    return st, bits.value


def moe_status_string(status: int) -> str:
    return _lib.moe_status_string(status).decode()
