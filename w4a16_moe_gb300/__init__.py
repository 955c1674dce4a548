"""GB300 (sm_103a) fused W4A16 mixture-of-experts layer.

A thin Python binding over the C ABI of ``libb4moe.so`` (``include/b4moe.h``):
argument marshalling only -- every step of the layer runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (torch serves as the device
allocator and stream provider); their data pointers are handed to the C
entry points as plain addresses.

The library must be built first (``python w4a16_moe_gb300/build.py`` or
``__graft_entry__.build()``); importing this package without it raises.
"""

from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libb4moe.so")

B4_OK = 0
B4_ERR_INVALID_ARGUMENT = 1
B4_ERR_UNSUPPORTED_DEVICE = 2
B4_ERR_WORKSPACE_TOO_SMALL = 3
B4_ERR_CUDA = 4
B4_ERR_TIMEOUT = 5

NVFP4 = 0
MXFP4 = 1
SILU = 0
RELU2 = 1
SWIGLU_OAI = 2
PATH_AUTO = 0
PATH_DECODE = 1
PATH_GROUPED = 2
DECODE_MAX_M = 64
NOALLOC_SCRATCH_BYTES = 64 << 20
FORMATS = {"nvfp4_e4m3_k16": NVFP4, "mxfp4_e8m0_k32": MXFP4}
ACTIVATIONS = {"silu": SILU, "relu2": RELU2, "swiglu_oai": SWIGLU_OAI}
# the gpt-oss models' clamped-swiglu parameters (alpha, beta, limit)
SWIGLU_OAI_DEFAULTS = (1.702, 1.0, 7.0)


class B4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


class _Config(ctypes.Structure):
    _fields_ = [
        ("m", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("num_global_experts", ctypes.c_int32),
        ("num_local_experts", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("inter", ctypes.c_int32),
        ("format", ctypes.c_int32),
        ("path", ctypes.c_int32),
        ("expert_map", ctypes.c_void_p),
        ("swiglu_alpha", ctypes.c_float),
        ("swiglu_beta", ctypes.c_float),
        ("swiglu_limit", ctypes.c_float),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python w4a16_moe_gb300/build.py` "
            "(there is no CPU or Python fallback for this layer)"
        )
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    S = ctypes.c_size_t
    I32 = ctypes.c_int32
    CP = ctypes.POINTER(_Config)
    sigs = {
        "b4_route_capacity_tokens": (I32, [I32]),
        "b4_workspace_bytes": (S, [CP, I32]),
        "b4_prepared_sizes": (I32, [CP, I32, I32, ctypes.POINTER(S), ctypes.POINTER(S)]),
        "b4_prepare_weights": (I32, [CP, I32, I32, P, P, P, P, P]),
        "b4_route_pack": (I32, [CP, P, P, P, P, P]),
        "b4_fused_moe": (I32, [CP, P, P, P, P, P, P, P, P, P, I32, P, P, S, P]),
        "b4_fused_moe_noalloc": (I32, [CP, P, P, P, P, P, P, P, P, P, I32, P, P, P]),
        "b4_linear_workspace_bytes": (S, [CP]),
        "b4_linear": (I32, [CP, P, P, P, P, P, P, S, P]),
        "b4_check_status": (I32, [P, P]),
        "b4_wait_self_test": (I32, [P, S, ctypes.c_uint32, P]),
        "b4_set_timing_events": (I32, [ctypes.POINTER(P), I32]),
        "b4_set_trace": (I32, [P, S]),
        "b4_status_string": (ctypes.c_char_p, [I32]),
        "b4_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
EXPORTED = (
    "b4_route_capacity_tokens",
    "b4_workspace_bytes",
    "b4_prepared_sizes",
    "b4_prepare_weights",
    "b4_route_pack",
    "b4_fused_moe",
    "b4_fused_moe_noalloc",
    "b4_linear_workspace_bytes",
    "b4_linear",
    "b4_check_status",
    "b4_wait_self_test",
    "b4_set_timing_events",
    "b4_set_trace",
    "b4_status_string",
    "b4_last_error",
)


def status_string(status: int) -> str:
    return _lib.b4_status_string(int(status)).decode()


def last_error() -> str:
    return _lib.b4_last_error().decode()


def _check(status: int):
    if status != B4_OK:
        raise B4Error(status, last_error())


@dataclasses.dataclass
class MoEConfig:
    """Shape of one fused MoE call (mirrors ``b4_moe_config``)."""

    m: int
    top_k: int
    num_global_experts: int
    num_local_experts: int
    hidden: int
    inter: int
    format: int = NVFP4
    path: int = PATH_AUTO
    expert_map: torch.Tensor | None = None  # int32 CUDA tensor [E_g] or None
    # read for the SWIGLU_OAI activation only
    swiglu_alpha: float = SWIGLU_OAI_DEFAULTS[0]
    swiglu_beta: float = SWIGLU_OAI_DEFAULTS[1]
    swiglu_limit: float = SWIGLU_OAI_DEFAULTS[2]

    def _c(self) -> _Config:
        em = 0
        if self.expert_map is not None:
            _need(self.expert_map, torch.int32, "expert_map")
            em = self.expert_map.data_ptr()
        return _Config(self.m, self.top_k, self.num_global_experts, self.num_local_experts,
                       self.hidden, self.inter, self.format, self.path, em,
                       self.swiglu_alpha, self.swiglu_beta, self.swiglu_limit)


def _need(t, dtype, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def route_capacity_tokens(m: int) -> int:
    return int(_lib.b4_route_capacity_tokens(int(m)))


def workspace_bytes(cfg: MoEConfig, activation: int) -> int:
    c = cfg._c()
    n = _lib.b4_workspace_bytes(ctypes.byref(c), int(activation))
    if n == 0:
        raise B4Error(B4_ERR_INVALID_ARGUMENT, last_error())
    return int(n)


def prepared_sizes(cfg: MoEConfig, which: int, activation: int):
    c = cfg._c()
    cb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(_lib.b4_prepared_sizes(ctypes.byref(c), int(which), int(activation), ctypes.byref(cb), ctypes.byref(sb)))
    return int(cb.value), int(sb.value)


def prepare_weights(cfg: MoEConfig, which: int, activation: int, src_codes, src_scales, dst_codes=None,
                    dst_scales=None, stream=None):
    """Checkpoint layout -> serving layout.  Allocates the outputs with torch when not given."""
    _need(src_codes, torch.uint8, "src_codes")
    _need(src_scales, torch.uint8, "src_scales")
    cb, sb = prepared_sizes(cfg, which, activation)
    dev = src_codes.device
    if dst_codes is None:
        dst_codes = torch.empty(cb, dtype=torch.uint8, device=dev)
    if dst_scales is None:
        dst_scales = torch.empty(sb, dtype=torch.uint8, device=dev)
    c = cfg._c()
    _check(_lib.b4_prepare_weights(ctypes.byref(c), int(which), int(activation), _ptr(src_codes), _ptr(src_scales),
                                   _ptr(dst_codes), _ptr(dst_scales), _stream(stream)))
    return dst_codes, dst_scales


def route_pack(cfg: MoEConfig, topk_ids, counts, offsets, sorted_routes, stream=None):
    _need(topk_ids, torch.int32, "topk_ids")
    for t, n in ((counts, "counts"), (offsets, "offsets"), (sorted_routes, "sorted_routes")):
        _need(t, torch.int32, n)
    c = cfg._c()
    _check(_lib.b4_route_pack(ctypes.byref(c), _ptr(topk_ids), _ptr(counts), _ptr(offsets), _ptr(sorted_routes),
                              _stream(stream)))


def fused_moe(cfg: MoEConfig, x, w13, s13, gs13, w2, s2, gs2, topk_ids, topk_weights, activation, out, workspace,
              stream=None):
    """Enqueue the fused layer; ``out`` [m, H] bf16 is written in full."""
    _need(x, torch.bfloat16, "x")
    _need(out, torch.bfloat16, "out")
    _need(topk_ids, torch.int32, "topk_ids")
    _need(topk_weights, torch.float32, "topk_weights")
    _need(workspace, torch.uint8, "workspace")
    for t, n in ((w13, "w13"), (s13, "s13"), (w2, "w2"), (s2, "s2")):
        _need(t, torch.uint8, n)
    for t, n in ((gs13, "gs13"), (gs2, "gs2")):
        if t is not None:
            _need(t, torch.float32, n)
    c = cfg._c()
    _check(_lib.b4_fused_moe(ctypes.byref(c), _ptr(x), _ptr(w13), _ptr(s13), _ptr(gs13), _ptr(w2), _ptr(s2),
                             _ptr(gs2), _ptr(topk_ids), _ptr(topk_weights), int(activation), _ptr(out),
                             _ptr(workspace), workspace.numel(), _stream(stream)))


def fused_moe_noalloc(cfg: MoEConfig, x, w13, s13, gs13, w2, s2, gs2, topk_ids, topk_weights, activation, out,
                      device_status=None, stream=None):
    """``fused_moe`` for callers that cannot allocate: the scratch is the library's
    static device array of ``NOALLOC_SCRATCH_BYTES``; larger shapes are refused.
    ``device_status`` (optional int32 CUDA tensor of 2) receives the call's
    device status word.  Calls that overlap on the GPU race on the shared array."""
    _need(x, torch.bfloat16, "x")
    _need(out, torch.bfloat16, "out")
    _need(topk_ids, torch.int32, "topk_ids")
    _need(topk_weights, torch.float32, "topk_weights")
    for t, n in ((w13, "w13"), (s13, "s13"), (w2, "w2"), (s2, "s2")):
        _need(t, torch.uint8, n)
    for t, n in ((gs13, "gs13"), (gs2, "gs2")):
        if t is not None:
            _need(t, torch.float32, n)
    if device_status is not None:
        _need(device_status, torch.int32, "device_status")
        if device_status.numel() < 2:
            raise ValueError("device_status needs 2 elements")
    c = cfg._c()
    _check(_lib.b4_fused_moe_noalloc(ctypes.byref(c), _ptr(x), _ptr(w13), _ptr(s13), _ptr(gs13), _ptr(w2), _ptr(s2),
                                     _ptr(gs2), _ptr(topk_ids), _ptr(topk_weights), int(activation), _ptr(out),
                                     _ptr(device_status), _stream(stream)))


def linear_config(m: int, n: int, k: int, format: int = NVFP4, path: int = PATH_AUTO) -> MoEConfig:
    """Shape of a dense W4A16 linear call: out [m, n] = x [m, k] . W[n, k]^T
    (one expert, top-1, inter = n, hidden = k; ``b4_linear`` in b4moe.h)."""
    return MoEConfig(m=m, top_k=1, num_global_experts=1, num_local_experts=1, hidden=k, inter=n, format=format,
                     path=path)


def linear_workspace_bytes(cfg: MoEConfig) -> int:
    c = cfg._c()
    n = _lib.b4_linear_workspace_bytes(ctypes.byref(c))
    if n == 0:
        raise B4Error(B4_ERR_INVALID_ARGUMENT, last_error())
    return int(n)


def prepare_linear_weights(cfg: MoEConfig, src_codes, src_scales, stream=None):
    """W [n, k] (codes [n, k/2], scales [n, k/g]; a leading expert axis of 1 is
    optional) -> the serving layout ``linear`` reads (the non-gated FC1 layout)."""
    return prepare_weights(cfg, 0, RELU2, src_codes, src_scales, stream=stream)


def linear(cfg: MoEConfig, x, w, s, gs, out, workspace, stream=None):
    """Enqueue the dense W4A16 linear layer; ``out`` [m, n] bf16 is written in full."""
    _need(x, torch.bfloat16, "x")
    _need(out, torch.bfloat16, "out")
    _need(workspace, torch.uint8, "workspace")
    _need(w, torch.uint8, "w")
    _need(s, torch.uint8, "s")
    if gs is not None:
        _need(gs, torch.float32, "gs")
    c = cfg._c()
    _check(_lib.b4_linear(ctypes.byref(c), _ptr(x), _ptr(w), _ptr(s), _ptr(gs), _ptr(out), _ptr(workspace),
                          workspace.numel(), _stream(stream)))


def fused_moe_raw(cfg: MoEConfig, ptrs: dict, activation: int, workspace_ptr: int, workspace_bytes_: int,
                  stream_handle: int) -> int:
    """The C call with raw addresses (host code that manages its own pointers); returns the status."""
    c = cfg._c()
    return int(_lib.b4_fused_moe(ctypes.byref(c), ptrs["x"], ptrs["w13"], ptrs["s13"], ptrs.get("gs13"), ptrs["w2"],
                                 ptrs["s2"], ptrs.get("gs2"), ptrs["topk_ids"], ptrs["topk_weights"], int(activation),
                                 ptrs["out"], workspace_ptr, workspace_bytes_, stream_handle))


_timing_keepalive = None


def set_timing_events(events):
    """Per-kernel timing: a list of torch.cuda.Event(enable_timing=True), or None to stop."""
    global _timing_keepalive
    if events is None:
        _timing_keepalive = None
        _check(_lib.b4_set_timing_events(None, 0))
        return
    for e in events:  # torch creates the CUDA event at its first record
        if not e.cuda_event:
            e.record(torch.cuda.current_stream())
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _timing_keepalive = arr
    _check(_lib.b4_set_timing_events(arr, len(events)))


def set_trace(buffer):
    """Kernel timeline (see b4_set_trace): an int64 CUDA tensor of >= 32768 entries, or None."""
    if buffer is None:
        _check(_lib.b4_set_trace(None, 0))
    else:
        _need(buffer, torch.int64, "trace buffer")
        _check(_lib.b4_set_trace(buffer.data_ptr(), buffer.numel() * 8))


def check_status(workspace, stream=None):
    _check(_lib.b4_check_status(_ptr(workspace), _stream(stream)))


def wait_self_test(workspace, limit_us, stream=None):
    """Enqueue the bounded-wait diagnostic (b4_wait_self_test): a wait that no
    arrival completes runs out after limit_us and leaves B4_ERR_TIMEOUT in the
    workspace's status word (read it with check_status)."""
    _need(workspace, torch.uint8, "workspace")
    _check(_lib.b4_wait_self_test(_ptr(workspace), workspace.numel(), int(limit_us), _stream(stream)))


def raw_lib():
    """The loaded ctypes library (for tests of the C ABI itself)."""
    return _lib
