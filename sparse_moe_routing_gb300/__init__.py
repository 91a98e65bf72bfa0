"""Python binding of libmoe_route (the sparse MoE layer forward, GB300).

Argument marshalling only: every step of the layer runs in the CUDA kernels
of libmoe_route.so, called through its C ABI (include/moe_route.h). torch
supplies device memory and the current stream. There is no CPU fallback: if
the shared library is missing, importing the binding's functions raises.

Build the library with `python -m sparse_moe_routing_gb300.build`.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

__all__ = [
    "MoEConfig", "MoEError", "lib", "lib_path", "abi_version", "status_string",
    "workspace_bytes", "alloc_workspace", "route", "bucket", "experts_forward",
    "layer_forward", "read_device_status", "SOFTMAX_TOPK", "SIGMOID_GROUP_TOPK",
    "F32", "BF16", "Q4_AFFINE_G64", "PATH_AUTO", "PATH_GEMV", "PATH_TC", "PATH_FUSED",
    "inject_stall",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_PKG, "libmoe_route.so")

SOFTMAX_TOPK, SIGMOID_GROUP_TOPK = 0, 1
F32, BF16, Q4_AFFINE_G64 = 0, 1, 2
PATH_AUTO, PATH_GEMV, PATH_TC, PATH_FUSED = 0, 1, 2, 3
_STATUS = ["MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_WORKSPACE",
           "MOE_ERR_CUDA", "MOE_ERR_DEVICE_TIMEOUT", "MOE_ERR_DEVICE_CHECK"]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = "%s: %s" % (where, status_string(status))
        if status == 4:
            try:
                msg += " (%s)" % lib().moe_last_cuda_error().decode()
            except Exception:
                pass
        super().__init__(msg)


class _Cfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("d_ff", ctypes.c_int32), ("d_ff_shared", ctypes.c_int32),
                ("router", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("routed_scaling", ctypes.c_float),
                ("renorm_clamp", ctypes.c_float), ("act_dtype", ctypes.c_int32),
                ("expert_dtype", ctypes.c_int32), ("path", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class _Bank(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("minv", ctypes.c_void_p)]


_P = ctypes.c_void_p
_SIGS = {
    "moe_abi_version": (ctypes.c_int, []),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(_Cfg)]),
    "moe_workspace_init": (ctypes.c_int, [ctypes.POINTER(_Cfg), _P]),
    "moe_read_device_status": (ctypes.c_int, [ctypes.POINTER(_Cfg), _P,
                                              ctypes.POINTER(ctypes.c_uint32)]),
    "moe_route": (ctypes.c_int, [_P, _P, _P, _P, ctypes.POINTER(_Cfg), _P, _P, _P, _P]),
    "moe_bucket": (ctypes.c_int, [_P, ctypes.POINTER(_Cfg), _P, _P, _P, _P, _P, _P, _P]),
    "moe_experts_forward": (ctypes.c_int, [_P, _P, _P, _P, _P, _Bank, _Bank, _Bank, _P, _P, _P,
                                           _P, ctypes.POINTER(_Cfg), _P, _P]),
    "moe_layer_forward": (ctypes.c_int, [_P, _P, _P, _P, _Bank, _Bank, _Bank, _P, _P, _P, _P,
                                         ctypes.POINTER(_Cfg), _P, _P, _P, _P]),
    "moe_launch_count": (ctypes.c_uint64, []),
    "moe_last_cuda_error": (ctypes.c_char_p, []),
    "moe_trace_kernel": (ctypes.c_int, [ctypes.c_int, _P, _P, ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_int)]),
    "moe_inject_stall": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint32]),
}

# kernel families (moe_kernel_t)
KERNELS = {"router_logits": 1, "router_topk": 2, "shared_gate": 3, "bucket": 4,
           "gemv_gateup": 5, "gemv_down": 6, "combine": 7, "tc_gateup": 8, "tc_down": 9,
           "gather": 10, "tc_router": 11, "decode_fused": 12}

_lib = None


def lib():
    """The loaded libmoe_route.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(lib_path):
            raise RuntimeError("libmoe_route.so is not built (%s); run "
                               "`python -m sparse_moe_routing_gb300.build`" % lib_path)
        L = ctypes.CDLL(lib_path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def abi_version() -> int:
    return lib().moe_abi_version()


def status_string(status: int) -> str:
    try:
        return lib().moe_status_string(int(status)).decode()
    except RuntimeError:
        return _STATUS[status] if 0 <= status < len(_STATUS) else "unknown status %d" % status


@dataclass
class MoEConfig:
    """Layer configuration (moe_cfg_t without the workspace fields)."""
    T: int
    d_model: int
    n_experts: int
    top_k: int
    d_ff: int
    d_ff_shared: int = 0
    router: int = SOFTMAX_TOPK
    n_group: int = 1
    topk_group: int = 1
    routed_scaling: float = 1.0
    renorm_clamp: float = 2.0 ** -14
    act_dtype: int = BF16
    expert_dtype: int = BF16
    path: int = PATH_AUTO

    def _c(self, workspace=None) -> _Cfg:
        c = _Cfg(self.T, self.d_model, self.n_experts, self.top_k, self.d_ff, self.d_ff_shared,
                 self.router, self.n_group, self.topk_group, self.routed_scaling,
                 self.renorm_clamp, self.act_dtype, self.expert_dtype, self.path, None, 0)
        if workspace is not None:
            c.workspace = workspace.data_ptr()
            c.workspace_bytes = workspace.numel() * workspace.element_size()
        return c


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _bank(b):
    """A bank is a tensor (f32/bf16) or a (codes, scale, min) tuple (q4)."""
    if isinstance(b, (tuple, list)):
        return _Bank(_ptr(b[0]), _ptr(b[1]), _ptr(b[2]))
    return _Bank(_ptr(b), None, None)


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise MoEError(status, where)


def workspace_bytes(cfg: MoEConfig) -> int:
    n = lib().moe_workspace_bytes(ctypes.byref(cfg._c()))
    if n == 0:
        raise MoEError(1, "moe_workspace_bytes")
    return n


def alloc_workspace(cfg: MoEConfig, device=None, stream=None):
    """Allocates (with torch) and initialises a workspace for cfg."""
    import torch
    n = workspace_bytes(cfg)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    _check(lib().moe_workspace_init(ctypes.byref(cfg._c(ws)), _stream(stream)),
           "moe_workspace_init")
    return ws


def read_device_status(cfg: MoEConfig, workspace, stream=None):
    """Synchronises, returns (status, raw word) and clears the word."""
    info = ctypes.c_uint32(0)
    st = lib().moe_read_device_status(ctypes.byref(cfg._c(workspace)), _stream(stream),
                                      ctypes.byref(info))
    return st, info.value


def route(cfg, workspace, x, W_router, topk_ids, weights, expert_bias=None, w_shared=None,
          s_shared=None, stream=None):
    _check(lib().moe_route(_ptr(x), _ptr(W_router), _ptr(expert_bias), _ptr(w_shared),
                           ctypes.byref(cfg._c(workspace)), _ptr(topk_ids), _ptr(weights),
                           _ptr(s_shared), _stream(stream)), "moe_route")


def bucket(cfg, workspace, topk_ids, counts, offsets, active, n_active, perm, pos, stream=None):
    _check(lib().moe_bucket(_ptr(topk_ids), ctypes.byref(cfg._c(workspace)), _ptr(counts),
                            _ptr(offsets), _ptr(active), _ptr(n_active), _ptr(perm), _ptr(pos),
                            _stream(stream)), "moe_bucket")


def experts_forward(cfg, workspace, x, r_attn, topk_ids, weights, W_gate, W_up, W_down, out,
                    s_shared=None, Ws_gate=None, Ws_up=None, Ws_down=None, w_shared=None,
                    stream=None):
    _check(lib().moe_experts_forward(
        _ptr(x), _ptr(r_attn), _ptr(topk_ids), _ptr(weights), _ptr(s_shared), _bank(W_gate),
        _bank(W_up), _bank(W_down), _ptr(Ws_gate), _ptr(Ws_up), _ptr(Ws_down), _ptr(w_shared),
        ctypes.byref(cfg._c(workspace)), _ptr(out), _stream(stream)), "moe_experts_forward")


def layer_forward(cfg, workspace, x, r_attn, W_router, W_gate, W_up, W_down, out, topk_ids,
                  weights, expert_bias=None, Ws_gate=None, Ws_up=None, Ws_down=None,
                  w_shared=None, stream=None):
    _check(lib().moe_layer_forward(
        _ptr(x), _ptr(r_attn), _ptr(W_router), _ptr(expert_bias), _bank(W_gate), _bank(W_up),
        _bank(W_down), _ptr(Ws_gate), _ptr(Ws_up), _ptr(Ws_down), _ptr(w_shared),
        ctypes.byref(cfg._c(workspace)), _ptr(out), _ptr(topk_ids), _ptr(weights),
        _stream(stream)), "moe_layer_forward")


def inject_stall(kernel: str, wait_us: int):
    """Failure self-test (moe_inject_stall): the next launch of `kernel`
    ("tc_gateup", "tc_down" or "decode_fused") waits on a flag nothing sets
    and gives up after wait_us; None disarms."""
    _check(lib().moe_inject_stall(0 if kernel is None else KERNELS[kernel], int(wait_us)),
           "moe_inject_stall")


def launch_count() -> int:
    """Kernel launches this library has enqueued in this process."""
    return int(lib().moe_launch_count())


class KernelTrace:
    """Brackets every launch of one kernel family with CUDA events recorded on
    the stream it is launched on (moe_trace_kernel). Use as a context manager;
    `durations_ms()` returns one duration per traced launch (up to n)."""

    def __init__(self, kernel: str, n: int):
        import torch
        self.kernel = KERNELS[kernel]
        self.n = n
        self.starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        self.stops = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        self._count = ctypes.c_int(0)
        # torch creates the CUDA event lazily: record once to materialise it
        for e in self.starts + self.stops:
            e.record()
        self._sa = (ctypes.c_void_p * n)(*[e.cuda_event for e in self.starts])
        self._so = (ctypes.c_void_p * n)(*[e.cuda_event for e in self.stops])

    def __enter__(self):
        _check(lib().moe_trace_kernel(self.kernel, self._sa, self._so, self.n,
                                      ctypes.byref(self._count)), "moe_trace_kernel")
        return self

    def __exit__(self, *exc):
        lib().moe_trace_kernel(0, None, None, 0, None)
        return False

    @property
    def count(self) -> int:
        return self._count.value

    def durations_ms(self):
        import torch
        torch.cuda.synchronize()
        m = min(self.count, self.n)
        return [self.starts[i].elapsed_time(self.stops[i]) for i in range(m)]


class MoELayer:
    """One MoE layer's device weights plus its workspace: `forward` is the
    call a user makes (x, r_attn device tensors in, out/ids/weights out).

    weights: dict of device tensors named as in include/moe_route.h
    (W_router, expert_bias, W_gate, W_up, W_down or (codes, scale, min)
    tuples for 4-bit banks, Ws_gate, Ws_up, Ws_down, w_shared)."""

    def __init__(self, cfg: MoEConfig, weights: dict, device=None):
        import torch
        self.cfg = cfg
        self.w = weights
        self.device = device or torch.device("cuda", torch.cuda.current_device())
        self.ws = alloc_workspace(cfg, self.device)
        T, k, d = cfg.T, cfg.top_k, cfg.d_model
        self.out = torch.empty((T, d), dtype=torch.float32, device=self.device)
        self.ids = torch.empty((T, k), dtype=torch.int32, device=self.device)
        self.weights = torch.empty((T, k), dtype=torch.float32, device=self.device)

    def forward(self, x, r_attn, out=None, stream=None):
        w = self.w
        out = self.out if out is None else out
        def bank(name):  # a tensor, or the (codes, scale, min) of a 4-bit bank
            return w[name] if name in w else (w[name + "_q"], w[name + "_scale"], w[name + "_min"])

        layer_forward(self.cfg, self.ws, x, r_attn, w["W_router"], bank("W_gate"), bank("W_up"),
                      bank("W_down"), out, self.ids, self.weights,
                      expert_bias=w.get("expert_bias"), Ws_gate=w.get("Ws_gate"),
                      Ws_up=w.get("Ws_up"), Ws_down=w.get("Ws_down"),
                      w_shared=w.get("w_shared"), stream=stream)
        return out, self.ids, self.weights

    def device_status(self, stream=None):
        return read_device_status(self.cfg, self.ws, stream)
