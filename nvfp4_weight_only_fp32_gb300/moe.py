"""ctypes binding of the C ABI in include/moe_nvfp4.h.

Argument marshalling only: every step of the decode layer runs in the CUDA
library (libmoe_nvfp4.so).  PyTorch supplies device memory and the current
stream.  If the library has not been built this module raises on first use;
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmoe_nvfp4.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_OOM = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_DEVICE = -6

EXPORTED = [
    "moe_init", "moe_destroy", "moe_decode_forward", "moe_decode_forward_host",
    "moe_stage_route", "moe_stage_gate_up", "moe_stage_down",
    "moe_check", "moe_debug_dequant", "moe_get_info", "moe_last_error",
    "moe_route_topk_static", "moe_trace_attach", "moe_debug_inject", "moe_quant_fos",
]

MOE_INJECT_WAIT_STALL = 1


class moe_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("num_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("inter", ctypes.c_int), ("num_shared", ctypes.c_int), ("shared_inter", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("normalize_topk", ctypes.c_int),
                ("routed_scale", ctypes.c_float), ("grouped_min_tokens", ctypes.c_int),
                ("fused", ctypes.c_int), ("score_func", ctypes.c_int),
                ("expert_format", ctypes.c_int), ("shared_format", ctypes.c_int), ("w4a4", ctypes.c_int)]

SCORE_FUNCS = {"sigmoid": 0, "softmax": 1}
# expert weight formats (MOE_FMT_* of the header)
FORMATS = {"nvfp4": 0, "mxfp4": 1, "fp8_block": 2, "mxfp8": 3}


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router_w", "router_b", "w13", "w13_sf", "w13_gs", "w2", "w2_sf", "w2_gs",
        "sw13", "sw13_sf", "sw13_gs", "sw2", "sw2_sf", "sw2_gs")]


class moe_layer_info(ctypes.Structure):
    _fields_ = [("weight_bytes", ctypes.c_size_t), ("workspace_bytes", ctypes.c_size_t),
                ("expert_bytes", ctypes.c_size_t), ("shared_bytes", ctypes.c_size_t),
                ("max_slots", ctypes.c_int), ("sm_count", ctypes.c_int),
                ("single_launch_max_tokens", ctypes.c_int)]


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"moe status {status}: {msg}")
        self.status = status


_lock = threading.Lock()
_lib = None


def lib(path: str | None = None):
    """Load the CUDA library (raises if it is missing).  MOE_LIBRARY may name
    another build of it (e.g. the traced build)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or os.environ.get("MOE_LIBRARY") or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is missing: build it with nvfp4_weight_only_fp32_gb300.build.build()")
            L = ctypes.CDLL(p)
            vp, i, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
            L.moe_init.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(moe_weights), vp,
                                   ctypes.POINTER(vp)]
            L.moe_init.restype = st
            L.moe_destroy.argtypes = [vp]
            L.moe_destroy.restype = None
            L.moe_decode_forward.argtypes = [vp, vp, i, vp, vp, vp, vp]
            L.moe_decode_forward.restype = st
            L.moe_decode_forward_host.argtypes = [vp, vp, i, vp, vp, vp, vp]
            L.moe_decode_forward_host.restype = st
            L.moe_stage_route.argtypes = [vp, vp, i, vp, vp, vp]
            L.moe_stage_route.restype = st
            L.moe_stage_gate_up.argtypes = [vp, vp, i, vp]
            L.moe_stage_gate_up.restype = st
            L.moe_stage_down.argtypes = [vp, i, vp, vp]
            L.moe_stage_down.restype = st
            L.moe_check.argtypes = [vp, vp]
            L.moe_check.restype = st
            L.moe_debug_dequant.argtypes = [vp, i, i, vp, vp]
            L.moe_debug_dequant.restype = st
            L.moe_get_info.argtypes = [vp, ctypes.POINTER(moe_layer_info)]
            L.moe_get_info.restype = st
            L.moe_route_topk_static.argtypes = [vp, vp, i, i, i, i, ctypes.c_float, vp, i, vp, vp, vp]
            L.moe_route_topk_static.restype = st
            L.moe_trace_attach.argtypes = [vp, vp, i]
            L.moe_trace_attach.restype = st
            L.moe_debug_inject.argtypes = [vp, i, i]
            L.moe_debug_inject.restype = st
            L.moe_quant_fos.argtypes = [vp, i, i, vp, vp, vp]
            L.moe_quant_fos.restype = st
            L.moe_last_error.argtypes = []
            L.moe_last_error.restype = ctypes.c_char_p
            _lib = L
    return _lib


def last_error() -> str:
    return lib().moe_last_error().decode()


def _check(status: int):
    if status != MOE_OK:
        raise MoEError(status, last_error())


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# --- C-ABI entry points, same names -----------------------------------------

def moe_init(cfg: moe_config, w: moe_weights, stream=None) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().moe_init(ctypes.byref(cfg), ctypes.byref(w), ctypes.c_void_p(_stream(stream)),
                          ctypes.byref(h)))
    return h


def moe_destroy(h) -> None:
    lib().moe_destroy(h)


def moe_decode_forward(h, x, T, out, topk_ids=None, topk_w=None, stream=None) -> None:
    _check(lib().moe_decode_forward(h, _p(x), int(T), _p(out), _p(topk_ids), _p(topk_w),
                                    ctypes.c_void_p(_stream(stream))))


def moe_decode_forward_host(h, x_host, T, out_host, ids_host=None, w_host=None, stream=None) -> None:
    _check(lib().moe_decode_forward_host(h, _p(x_host), int(T), _p(out_host), _p(ids_host),
                                         _p(w_host), ctypes.c_void_p(_stream(stream))))


def moe_stage_route(h, x, T, topk_ids=None, topk_w=None, stream=None) -> None:
    _check(lib().moe_stage_route(h, _p(x), int(T), _p(topk_ids), _p(topk_w),
                                 ctypes.c_void_p(_stream(stream))))


def moe_stage_gate_up(h, x, T, stream=None) -> None:
    _check(lib().moe_stage_gate_up(h, _p(x), int(T), ctypes.c_void_p(_stream(stream))))


def moe_stage_down(h, T, out, stream=None) -> None:
    _check(lib().moe_stage_down(h, int(T), _p(out), ctypes.c_void_p(_stream(stream))))


def moe_check(h, stream=None) -> int:
    return int(lib().moe_check(h, ctypes.c_void_p(_stream(stream))))


def moe_debug_dequant(h, which, expert, dst, stream=None) -> None:
    _check(lib().moe_debug_dequant(h, int(which), int(expert), _p(dst),
                                   ctypes.c_void_p(_stream(stream))))


def moe_get_info(h) -> moe_layer_info:
    info = moe_layer_info()
    _check(lib().moe_get_info(h, ctypes.byref(info)))
    return info


def moe_debug_inject(h, what, value) -> None:
    _check(lib().moe_debug_inject(h, int(what), int(value)))


def moe_trace_attach(h, buf, blocks_per_kernel) -> None:
    _check(lib().moe_trace_attach(h, _p(buf), int(blocks_per_kernel)))


def moe_route_topk_static(router_w, router_b, num_experts, hidden, top_k, normalize_topk,
                          routed_scale, x, T, topk_ids, topk_w, stream=None) -> None:
    """Routing without any device allocation (scratch in a static device
    array inside the library); see include/moe_nvfp4.h."""
    _check(lib().moe_route_topk_static(_p(router_w), _p(router_b), int(num_experts), int(hidden),
                                       int(top_k), int(normalize_topk), float(routed_scale), _p(x),
                                       int(T), _p(topk_ids), _p(topk_w),
                                       ctypes.c_void_p(_stream(stream))))


def moe_quant_fos(x, rows, n, deq, gs, stream=None) -> None:
    _check(lib().moe_quant_fos(_p(x), int(rows), int(n), _p(deq), _p(gs), ctypes.c_void_p(_stream(stream))))


# --- convenience wrapper ------------------------------------------------------

_NAMES = ("router_w", "router_b", "w13", "w13_sf", "w13_gs", "w2", "w2_sf", "w2_gs",
          "sw13", "sw13_sf", "sw13_gs", "sw2", "sw2_sf", "sw2_gs")


def to_device(layer: dict, device="cuda") -> dict:
    """Canonical numpy/torch tensors -> contiguous CUDA tensors (uint8 codes
    and scales -- FP32 for block-scaled FP8 -- float32 router and tensor
    scales)."""
    out = {}
    for n in _NAMES:
        a = layer.get(n)
        if a is None:
            out[n] = None
            continue
        t = a if isinstance(a, torch.Tensor) else torch.from_numpy(a)
        out[n] = t.to(device).contiguous()
    return out


def make_config(c: dict, max_tokens: int | None = None, grouped_min_tokens: int = 0,
                fused: int = 0) -> moe_config:
    return moe_config(hidden=c["H"], num_experts=c["E"], top_k=c["k"], inter=c["I"],
                      num_shared=c["S"], shared_inter=c["Is"],
                      max_tokens=int(max_tokens if max_tokens else c["T"]),
                      normalize_topk=int(c.get("normalize", 1)),
                      routed_scale=float(c.get("routed_scale", 1.0)),
                      grouped_min_tokens=int(grouped_min_tokens), fused=int(fused),
                      score_func=SCORE_FUNCS[c.get("score_func", "sigmoid")],
                      expert_format=FORMATS[c.get("efmt", "nvfp4")],
                      shared_format=FORMATS[c.get("sfmt", "nvfp4")],
                      w4a4=int(bool(c.get("w4a4", 0))))


class MoELayer:
    """One decode layer on the current CUDA device.

    `layer` is a dict of canonical tensors (numpy or torch) plus "cfg" with the
    sizes H, E, k, I, S, Is and, optionally, "normalize" (1), "routed_scale"
    (1.0), "score_func" ("sigmoid" or "softmax") and the expert formats
    "efmt" / "sfmt" ("nvfp4", "mxfp4", "fp8_block" or "mxfp8") and "w4a4" (0/1);
    the weights are repacked into library memory, so the inputs may be freed
    afterwards."""

    def __init__(self, layer: dict, max_tokens: int | None = None, grouped_min_tokens: int = 0,
                 stream=None, fused: int = 0):
        c = layer["cfg"]
        self.cfg = dict(c)
        self.max_tokens = int(max_tokens if max_tokens else c["T"])
        dev = to_device(layer)
        w = moe_weights(**{n: (None if t is None else t.data_ptr()) for n, t in dev.items()})
        self._cfg = make_config(c, self.max_tokens, grouped_min_tokens, fused)
        self.h = moe_init(self._cfg, w, stream)
        del dev

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x: torch.Tensor, out=None, ids=None, w=None, stream=None):
        T = x.shape[0]
        H, k = self.cfg["H"], self.cfg["k"]
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device) if out is None else out
        ids = torch.empty((T, k), dtype=torch.int32, device=x.device) if ids is None else ids
        w = torch.empty((T, k), dtype=torch.float32, device=x.device) if w is None else w
        moe_decode_forward(self.h, x, T, out, ids, w, stream)
        return out, ids, w

    def dequant(self, which: int, expert: int) -> torch.Tensor:
        c = self.cfg
        I = c["I"] if which in (0, 1) else c["Is"]
        shape = (2 * I, c["H"]) if which in (0, 2) else (c["H"], I)
        dst = torch.empty(shape, dtype=torch.float32, device="cuda")
        moe_debug_dequant(self.h, which, expert, dst)
        return dst

    def info(self) -> moe_layer_info:
        return moe_get_info(self.h)
