"""CPU oracle for the NVFP4 W4A16 sigmoid-top-k MoE decode layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports, links or
runs anything here, and this package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain scalar C, FP64); this module only
builds it with gcc, loads it with ctypes and marshals numpy arrays.  Every
function of ``oracle.c`` cites the page passage it follows.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, plant: int = 0) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP); with
    `plant` > 0 a separate library with that deliberate mistake compiled in
    (tests of the pins only)."""
    out = _LIB if plant == 0 else os.path.join(os.path.dirname(_LIB), f"liboracle_plant{int(plant)}.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp", "-std=c99",
           "-D_DEFAULT_SOURCE", f"-DORC_PLANT={int(plant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class _Layer(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
        ("I", ctypes.c_int), ("S", ctypes.c_int), ("Is", ctypes.c_int),
        ("normalize", ctypes.c_int), ("routed_scale", ctypes.c_double),
        ("router_w", ctypes.c_void_p), ("router_b", ctypes.c_void_p),
        ("w13", ctypes.c_void_p), ("w13_sf", ctypes.c_void_p), ("w13_gs", ctypes.c_void_p),
        ("w2", ctypes.c_void_p), ("w2_sf", ctypes.c_void_p), ("w2_gs", ctypes.c_void_p),
        ("sw13", ctypes.c_void_p), ("sw13_sf", ctypes.c_void_p), ("sw13_gs", ctypes.c_void_p),
        ("sw2", ctypes.c_void_p), ("sw2_sf", ctypes.c_void_p), ("sw2_gs", ctypes.c_void_p),
        ("score_func", ctypes.c_int),
        ("efmt", ctypes.c_int), ("sfmt", ctypes.c_int),
        ("w4a4", ctypes.c_int),
    ]


# Expert weight formats (see oracle.c): name -> code.
FORMATS = {"nvfp4": 0, "mxfp4": 1, "fp8_block": 2, "mxfp8": 3}


def format_code(name: str) -> int:
    if name not in FORMATS:
        raise ValueError(f"unknown expert format {name!r}")
    return FORMATS[name]


def _load(path):
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(build())
    return _lib


@contextlib.contextmanager
def planted(plant: int):
    """Run the oracle with deliberate mistake `plant` compiled in (see the
    ORC_PLANT list in oracle.c) inside the block; the regular library after."""
    global _lib
    regular = lib()
    mutant = _load(build(plant=plant))
    with _lock:
        _lib = mutant
    try:
        yield
    finally:
        with _lock:
            _lib = regular


def _declare(L):
    d, i, vp = ctypes.c_double, ctypes.c_int, ctypes.c_void_p
    L.orc_e2m1.restype = d
    L.orc_e2m1.argtypes = [i]
    L.orc_e4m3.restype = d
    L.orc_e4m3.argtypes = [i]
    L.orc_bf16_round.restype = d
    L.orc_bf16_round.argtypes = [d]
    L.orc_double_to_bf16.restype = ctypes.c_uint16
    L.orc_double_to_bf16.argtypes = [d]
    L.orc_bf16_to_double.restype = d
    L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.orc_dequant.restype = None
    L.orc_dequant.argtypes = [vp, vp, ctypes.c_float, i, i, vp]
    L.orc_dequant_fmt.restype = None
    L.orc_dequant_fmt.argtypes = [i, vp, vp, ctypes.c_float, i, i, vp]
    L.orc_e8m0.restype = d
    L.orc_e8m0.argtypes = [i]
    L.orc_quant_fos.restype = ctypes.c_float
    L.orc_quant_fos.argtypes = [vp, i, vp, vp, vp, vp]
    L.orc_e4m3_from_f32.restype = i
    L.orc_e4m3_from_f32.argtypes = [ctypes.c_float]
    L.orc_e2m1_from_f32.restype = i
    L.orc_e2m1_from_f32.argtypes = [ctypes.c_float]
    L.orc_route.restype = i
    L.orc_route.argtypes = [ctypes.POINTER(_Layer), vp, i, vp, vp, vp, vp]
    L.orc_forward.restype = i
    L.orc_forward.argtypes = [ctypes.POINTER(_Layer), vp, i, vp, vp, vp, vp, i]
    L.orc_max_threads.restype = i
    L.orc_max_threads.argtypes = []


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


class _Bound:
    """Keeps the contiguous arrays alive while the C struct points at them."""

    def __init__(self, layer: dict):
        self.arrs = {}
        c = layer["cfg"]
        efmt = format_code(c.get("efmt", "nvfp4"))
        sfmt = format_code(c.get("sfmt", "nvfp4"))
        # FP8 block scales are FP32; every other scale is one byte per block
        esf = np.float32 if efmt == FORMATS["fp8_block"] else np.uint8
        ssf = np.float32 if sfmt == FORMATS["fp8_block"] else np.uint8
        for name, dt in [("router_w", np.float32), ("router_b", np.float32),
                         ("w13", np.uint8), ("w13_sf", esf), ("w13_gs", np.float32),
                         ("w2", np.uint8), ("w2_sf", esf), ("w2_gs", np.float32),
                         ("sw13", np.uint8), ("sw13_sf", ssf), ("sw13_gs", np.float32),
                         ("sw2", np.uint8), ("sw2_sf", ssf), ("sw2_gs", np.float32)]:
            self.arrs[name] = _c(layer.get(name), dt)
        self.s = _Layer(H=c["H"], E=c["E"], k=c["k"], I=c["I"], S=c["S"], Is=c["Is"],
                        normalize=int(c.get("normalize", 1)),
                        routed_scale=float(c.get("routed_scale", 1.0)),
                        score_func=score_func_code(c), efmt=efmt, sfmt=sfmt,
                        w4a4=int(bool(c.get("w4a4", 0))),
                        **{n: _ptr(a) for n, a in self.arrs.items()})


def score_func_code(c: dict) -> int:
    """The layer's routing score: "sigmoid" (default) -> 0, "softmax" -> 1."""
    f = c.get("score_func", "sigmoid")
    if f not in ("sigmoid", "softmax"):
        raise ValueError(f"unknown score_func {f!r}")
    return 1 if f == "softmax" else 0


def e2m1(code: int) -> float:
    return lib().orc_e2m1(int(code))


def e4m3(code: int) -> float:
    return lib().orc_e4m3(int(code))


def e8m0(code: int) -> float:
    return lib().orc_e8m0(int(code))


def bf16_round(v: float) -> float:
    return lib().orc_bf16_round(float(v))


def to_bf16_bits(v: float) -> int:
    return int(lib().orc_double_to_bf16(float(v)))


def bf16_bits_to_float(b: int) -> float:
    return lib().orc_bf16_to_double(int(b))


def dequant(codes: np.ndarray, sf: np.ndarray, gs: float) -> np.ndarray:
    """[rows, cols/2] codes + [rows, cols/16] scales -> [rows, cols] FP32."""
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    rows, half = codes.shape
    cols = half * 2
    assert sf.shape == (rows, cols // 16)
    out = np.empty((rows, cols), dtype=np.float32)
    lib().orc_dequant(_ptr(codes), _ptr(sf), ctypes.c_float(gs), rows, cols, _ptr(out))
    return out


def dequant_fmt(fmt: str, codes: np.ndarray, sf: np.ndarray, gs: float, rows: int, cols: int) -> np.ndarray:
    """One [rows, cols] matrix of any expert format -> FP32 (gs: NVFP4 only).
    codes: [rows, cols/2] (FP4) or [rows, cols] (FP8) bytes; sf: [rows,
    cols/16] E4M3 (NVFP4), [rows, cols/32] E8M0 (MX), or FP32 [ceil(rows/128),
    ceil(cols/128)] (FP8 block)."""
    f = format_code(fmt)
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.float32 if fmt == "fp8_block" else np.uint8)
    out = np.empty((rows, cols), dtype=np.float32)
    lib().orc_dequant_fmt(f, _ptr(codes), _ptr(sf), ctypes.c_float(gs), rows, cols, _ptr(out))
    return out


def quant_fos(row_bits: np.ndarray):
    """Four-Over-Six NVFP4 quantisation of one BF16 row (length a multiple of
    16) -> (codes [n] uint8 (one code per element), block scale codes [n/16],
    choices [n/16] (4 or 6), global scale, dequantised [n] f64)."""
    row = _c(row_bits, np.uint16)
    n = row.shape[0]
    codes = np.empty(n, np.uint8)
    sf = np.empty(n // 16, np.uint8)
    ch = np.empty(n // 16, np.uint8)
    deq = np.empty(n, np.float64)
    gs = lib().orc_quant_fos(_ptr(row), n, _ptr(codes), _ptr(sf), _ptr(ch), _ptr(deq))
    return codes, sf, ch, float(gs), deq


def e4m3_from_f32(v: float) -> int:
    return int(lib().orc_e4m3_from_f32(float(v)))


def e2m1_from_f32(v: float) -> int:
    return int(lib().orc_e2m1_from_f32(float(v)))


def route(layer: dict, x_bits: np.ndarray):
    """Routing for T tokens -> (ids [T,k] int32, w [T,k] f64, scores [T,E] f64,
    logits [T,E] f64)."""
    b = _Bound(layer)
    x = _c(x_bits, np.uint16)
    T = x.shape[0]
    c = layer["cfg"]
    ids = np.empty((T, c["k"]), dtype=np.int32)
    w = np.empty((T, c["k"]), dtype=np.float64)
    s = np.empty((T, c["E"]), dtype=np.float64)
    z = np.empty((T, c["E"]), dtype=np.float64)
    rc = lib().orc_route(ctypes.byref(b.s), _ptr(x), T, _ptr(ids), _ptr(w), _ptr(s), _ptr(z))
    if rc != 0:
        raise MemoryError("oracle routing failed")
    return ids, w, s, z


def forward(layer: dict, x_bits: np.ndarray, nthreads: int | None = None):
    """Full layer -> (out_bits [T,H] uint16, out_pre [T,H] f64, ids, w)."""
    b = _Bound(layer)
    x = _c(x_bits, np.uint16)
    T = x.shape[0]
    c = layer["cfg"]
    out = np.empty((T, c["H"]), dtype=np.uint16)
    pre = np.empty((T, c["H"]), dtype=np.float64)
    ids = np.empty((T, c["k"]), dtype=np.int32)
    w = np.empty((T, c["k"]), dtype=np.float64)
    nt = nthreads if nthreads else max_threads()
    rc = lib().orc_forward(ctypes.byref(b.s), _ptr(x), T, _ptr(out), _ptr(pre),
                           _ptr(ids), _ptr(w), int(nt))
    if rc != 0:
        raise MemoryError("oracle forward failed")
    return out, pre, ids, w


def max_threads() -> int:
    return int(lib().orc_max_threads())
