"""CPU oracle for the true 1-bit (sign + fp16 group-128 scale) linear layer.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` are the only callers.  The product
(the CUDA library and its Python binding) never imports this package, and this
package imports nothing from the product.

The arithmetic lives in ``bit1_oracle.c`` (plain scalar C, fp64, one bit at a
time); this module compiles it with gcc and wraps it with ctypes.  Every
function cites the page passage it follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bit1_oracle.c")
_LIB = os.path.join(_HERE, "libbit1_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ESHAPE, ERANGE, ECUDA, ENAN = 0, 1, 2, 3, 4, 5
F32, BF16, F16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle into ``libbit1_oracle.so`` (scalar code: no
    auto-vectorisation, so the timed CPU baseline is the plain loop)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fno-tree-vectorize", "-std=c11", "-D_GNU_SOURCE",
               "-shared", "-fPIC", "-pthread", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def configure(lib):
    """Declare the C signatures on a loaded copy of the oracle library."""
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_half_to_double.restype = ctypes.c_double
    lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_double.restype = ctypes.c_double
    lib.orc_double_to_half.argtypes = [ctypes.c_double]
    lib.orc_double_to_half.restype = ctypes.c_uint16
    lib.orc_double_to_bf16.argtypes = [ctypes.c_double]
    lib.orc_double_to_bf16.restype = ctypes.c_uint16
    lib.orc_footprint_bytes.argtypes = [i64, i64]
    lib.orc_footprint_bytes.restype = i64
    lib.orc_gemv.argtypes = [p, p, p, i64, i64, i64, p]
    lib.orc_gemv.restype = ctypes.c_int
    lib.orc_gemv_select.argtypes = [p, p, p, i64, i64, i64, p, i64, p]
    lib.orc_gemv_select.restype = ctypes.c_int
    lib.orc_gemv_swiglu.argtypes = [p, p, p, i64, i64, i64, p]
    lib.orc_gemv_swiglu.restype = ctypes.c_int
    lib.orc_gemv_swiglu_select.argtypes = [p, p, p, i64, i64, i64, p, i64, p]
    lib.orc_gemv_swiglu_select.restype = ctypes.c_int
    lib.orc_gemv_ternary.argtypes = [p, p, p, p, i64, i64, i64, p]
    lib.orc_gemv_ternary.restype = ctypes.c_int
    lib.orc_gemv_ternary_swiglu.argtypes = [p, p, p, p, i64, i64, i64, p]
    lib.orc_gemv_ternary_swiglu.restype = ctypes.c_int
    lib.orc_gemv_ternary_select.argtypes = [p, p, p, p, i64, i64, i64, p, i64, p]
    lib.orc_gemv_ternary_select.restype = ctypes.c_int
    lib.orc_ternary_planes.argtypes = [p, i64, i64, p, p]
    lib.orc_ternary_planes.restype = ctypes.c_int
    lib.orc_ternary_footprint_bytes.argtypes = [i64, i64]
    lib.orc_ternary_footprint_bytes.restype = i64
    lib.orc_t5_pack.argtypes = [p, i64, i64, p]
    lib.orc_t5_pack.restype = ctypes.c_int
    lib.orc_t5_unpack.argtypes = [p, i64, i64, p]
    lib.orc_t5_unpack.restype = ctypes.c_int
    lib.orc_gemv_t5.argtypes = [p, p, p, i64, i64, i64, p]
    lib.orc_gemv_t5.restype = ctypes.c_int
    lib.orc_t5_footprint_bytes.argtypes = [i64, i64]
    lib.orc_t5_footprint_bytes.restype = i64
    lib.orc_gemv_threads.argtypes = [p, p, p, i64, i64, i64, p, ctypes.c_int]
    lib.orc_gemv_threads.restype = ctypes.c_int
    lib.orc_xor_patch.argtypes = [p, i64, i64, p, i64]
    lib.orc_xor_patch.restype = ctypes.c_int
    lib.orc_pack.argtypes = [p, ctypes.c_int, i64, i64, p, p]
    lib.orc_g128x_repack.argtypes = [p, i64, i64, p]
    lib.orc_g128x_repack.restype = ctypes.c_int
    lib.orc_g128x_unpack.argtypes = [p, i64, i64, p]
    lib.orc_g128x_unpack.restype = ctypes.c_int
    lib.orc_pack.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = configure(ctypes.CDLL(_LIB))
    return _lib


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"oracle {what}: status {status}")
        self.status = status


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    """Accept numpy uint16/float16 arrays or torch fp16/bf16/int16 tensors and
    return a C-contiguous uint16 view of the raw bit patterns."""
    if hasattr(a, "detach"):  # torch tensor
        import torch
        t = a.detach().cpu().contiguous()
        if t.dtype in (torch.float16, torch.bfloat16, torch.int16):
            t = t.view(torch.int16)
        a = t.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16 or a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected 16-bit patterns, got {a.dtype}")
    return a


def _u8(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"expected uint8 bits, got {a.dtype}")
    return a


# ---- scalar helpers ----------------------------------------------------

def half_to_double(h: int) -> float:
    return _load().orc_half_to_double(int(h) & 0xFFFF)


def bf16_to_double(b: int) -> float:
    return _load().orc_bf16_to_double(int(b) & 0xFFFF)


def double_to_half(v: float) -> int:
    return int(_load().orc_double_to_half(float(v)))


def double_to_bf16(v: float) -> int:
    return int(_load().orc_double_to_bf16(float(v)))


def footprint_bytes(N: int, K: int) -> int:
    return int(_load().orc_footprint_bytes(int(N), int(K)))


# ---- array entry points ------------------------------------------------

def gemv(bits, scales, x, B: int, N: int, K: int) -> np.ndarray:
    """y[B, N] in fp64: the exact dequantised product (scalar loop)."""
    bits, scales, x = _u8(bits), _u16(scales), _u16(x)
    y = np.zeros((B, N), dtype=np.float64)
    st = _load().orc_gemv(_ptr(bits), _ptr(scales), _ptr(x), B, N, K, _ptr(y))
    if st != OK:
        raise OracleError(st, "gemv")
    return y


def gemv_select(bits, scales, x, B: int, N: int, K: int, rows) -> np.ndarray:
    """y[B, len(rows)] for the listed rows only (sampled checks at full size)."""
    bits, scales, x = _u8(bits), _u16(scales), _u16(x)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    y = np.zeros((B, rows.size), dtype=np.float64)
    st = _load().orc_gemv_select(_ptr(bits), _ptr(scales), _ptr(x), B, N, K,
                                 _ptr(rows), rows.size, _ptr(y))
    if st != OK:
        raise OracleError(st, "gemv_select")
    return y


def gemv_swiglu(bits, scales, x, B: int, N2: int, K: int) -> np.ndarray:
    """Interleaved gate/up rows (2n gate, 2n+1 up) -> silu(gate) * up, [B, N2/2]."""
    bits, scales, x = _u8(bits), _u16(scales), _u16(x)
    h = np.zeros((B, N2 // 2), dtype=np.float64)
    st = _load().orc_gemv_swiglu(_ptr(bits), _ptr(scales), _ptr(x), B, N2, K, _ptr(h))
    if st != OK:
        raise OracleError(st, "gemv_swiglu")
    return h


def gemv_swiglu_select(bits, scales, x, B: int, N2: int, K: int, units) -> np.ndarray:
    """h[B, len(units)] for the listed hidden units only (sampled checks)."""
    bits, scales, x = _u8(bits), _u16(scales), _u16(x)
    units = np.ascontiguousarray(np.asarray(units, dtype=np.int64))
    h = np.zeros((B, units.size), dtype=np.float64)
    st = _load().orc_gemv_swiglu_select(_ptr(bits), _ptr(scales), _ptr(x), B, N2, K,
                                        _ptr(units), units.size, _ptr(h))
    if st != OK:
        raise OracleError(st, "gemv_swiglu_select")
    return h


def gemv_ternary(a, b, scales, x, B: int, N: int, K: int) -> np.ndarray:
    """Ternary product from the two sign planes a, b (t = (a + b) / 2), [B, N]."""
    a, b, scales, x = _u8(a), _u8(b), _u16(scales), _u16(x)
    y = np.zeros((B, N), dtype=np.float64)
    st = _load().orc_gemv_ternary(_ptr(a), _ptr(b), _ptr(scales), _ptr(x), B, N, K, _ptr(y))
    if st != OK:
        raise OracleError(st, "gemv_ternary")
    return y


def gemv_ternary_swiglu(a, b, scales, x, B: int, N2: int, K: int) -> np.ndarray:
    """Ternary interleaved gate/up rows -> silu(gate) * up, [B, N2/2]."""
    a, b, scales, x = _u8(a), _u8(b), _u16(scales), _u16(x)
    h = np.zeros((B, N2 // 2), dtype=np.float64)
    st = _load().orc_gemv_ternary_swiglu(_ptr(a), _ptr(b), _ptr(scales), _ptr(x), B, N2, K, _ptr(h))
    if st != OK:
        raise OracleError(st, "gemv_ternary_swiglu")
    return h


def gemv_ternary_select(a, b, scales, x, B: int, N: int, K: int, rows) -> np.ndarray:
    a, b, scales, x = _u8(a), _u8(b), _u16(scales), _u16(x)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    y = np.zeros((B, rows.size), dtype=np.float64)
    st = _load().orc_gemv_ternary_select(_ptr(a), _ptr(b), _ptr(scales), _ptr(x), B, N, K,
                                         _ptr(rows), rows.size, _ptr(y))
    if st != OK:
        raise OracleError(st, "gemv_ternary_select")
    return y


def ternary_planes(t, N: int, K: int):
    """Codes [N, K] (int8 in {-1, 0, 1}) -> (a, b) planes [N, K/8] each."""
    t = np.ascontiguousarray(np.asarray(t, dtype=np.int8)).reshape(-1)
    a = np.zeros(N * K // 8, dtype=np.uint8)
    b = np.zeros(N * K // 8, dtype=np.uint8)
    st = _load().orc_ternary_planes(_ptr(t), N, K, _ptr(a), _ptr(b))
    if st != OK:
        raise OracleError(st, "ternary_planes")
    return a.reshape(N, K // 8), b.reshape(N, K // 8)


def ternary_footprint_bytes(N: int, K: int) -> int:
    return int(_load().orc_ternary_footprint_bytes(N, K))


def t5_pack(t, N: int, K: int) -> np.ndarray:
    """Codes [N, K] (int8 in {-1, 0, 1}) -> five-per-byte packing [N, K/128*26]."""
    t = np.ascontiguousarray(np.asarray(t, dtype=np.int8)).reshape(-1)
    out = np.zeros(N * (K // 128) * 26, dtype=np.uint8)
    st = _load().orc_t5_pack(_ptr(t), N, K, _ptr(out))
    if st != OK:
        raise OracleError(st, "t5_pack")
    return out.reshape(N, (K // 128) * 26)


def t5_unpack(p, N: int, K: int) -> np.ndarray:
    p = _u8(p)
    t = np.zeros(N * K, dtype=np.int8)
    st = _load().orc_t5_unpack(_ptr(p), N, K, _ptr(t))
    if st != OK:
        raise OracleError(st, "t5_unpack")
    return t.reshape(N, K)


def gemv_t5(p, scales, x, B: int, N: int, K: int) -> np.ndarray:
    """Ternary product straight from the five-per-byte packing, [B, N]."""
    p, scales, x = _u8(p), _u16(scales), _u16(x)
    y = np.zeros((B, N), dtype=np.float64)
    st = _load().orc_gemv_t5(_ptr(p), _ptr(scales), _ptr(x), B, N, K, _ptr(y))
    if st != OK:
        raise OracleError(st, "gemv_t5")
    return y


def t5_footprint_bytes(N: int, K: int) -> int:
    return int(_load().orc_t5_footprint_bytes(N, K))


def gemv_threads(bits, scales, x, B: int, N: int, K: int, nthreads: int) -> np.ndarray:
    """Same scalar loop, rows dispatched over POSIX threads (CPU baseline)."""
    bits, scales, x = _u8(bits), _u16(scales), _u16(x)
    y = np.zeros((B, N), dtype=np.float64)
    st = _load().orc_gemv_threads(_ptr(bits), _ptr(scales), _ptr(x), B, N, K,
                                  _ptr(y), int(nthreads))
    if st != OK:
        raise OracleError(st, "gemv_threads")
    return y


def xor_patch(bits, N: int, K: int, rows) -> np.ndarray:
    """Return a patched copy of ``bits`` (byte-per-row XOR with 0xFF)."""
    out = _u8(bits).copy()
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    st = _load().orc_xor_patch(_ptr(out), N, K, _ptr(rows), rows.size)
    if st != OK:
        raise OracleError(st, "xor_patch")
    return out


def xor_patch_status(bits, N: int, K: int, rows) -> int:
    out = _u8(bits).copy()
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    return int(_load().orc_xor_patch(_ptr(out), N, K, _ptr(rows), rows.size))


def g128x_repack(bits, N: int, K: int) -> np.ndarray:
    """Canonical sign bits [N, K/8] -> the library's g128x storage layout
    (a per-group bit permutation; see the C source for its definition)."""
    src = _u8(bits)
    out = np.zeros_like(src)
    st = _load().orc_g128x_repack(_ptr(src), N, K, _ptr(out))
    if st != OK:
        raise OracleError(st, "g128x_repack")
    return out


def g128x_unpack(bits, N: int, K: int) -> np.ndarray:
    """The inverse of g128x_repack."""
    src = _u8(bits)
    out = np.zeros_like(src)
    st = _load().orc_g128x_unpack(_ptr(src), N, K, _ptr(out))
    if st != OK:
        raise OracleError(st, "g128x_unpack")
    return out


def pack(w, dtype: int, N: int, K: int):
    """(status, bits[N, K/8] uint8, scales[N, K/128] uint16).  ``w`` holds raw
    fp32 (float32 array) or 16-bit patterns (uint16 array) per ``dtype``."""
    if hasattr(w, "detach"):
        import torch
        t = w.detach().cpu().contiguous()
        if t.dtype in (torch.float16, torch.bfloat16):
            t = t.view(torch.int16)
        w = t.numpy()
    w = np.ascontiguousarray(w)
    if dtype == F32:
        if w.dtype != np.float32:
            raise TypeError("fp32 weights expected")
    else:
        w = _u16(w)
    bits = np.zeros((N, K // 8), dtype=np.uint8)
    scales = np.zeros((N, K // 128), dtype=np.uint16)
    st = _load().orc_pack(_ptr(w), int(dtype), N, K, _ptr(bits), _ptr(scales))
    return int(st), bits, scales


def round_fp32(y: np.ndarray) -> np.ndarray:
    """fp64 -> fp32, round to nearest even (C conversion semantics)."""
    return np.asarray(y, dtype=np.float64).astype(np.float32)


def round_bf16_bits(y: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns, directly (one rounding), element by element."""
    f = np.vectorize(double_to_bf16, otypes=[np.uint16])
    return f(np.asarray(y, dtype=np.float64))
