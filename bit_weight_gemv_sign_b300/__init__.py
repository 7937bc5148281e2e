"""Python binding of the bit1 C ABI (include/bit1.h): true 1-bit weights
(sign bit + one fp16 scale per 128 inputs) on NVIDIA B300.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libbit1.so``.  PyTorch provides device memory and streams.  If the
library has not been built (``python -m bit_weight_gemv_sign_b300.build``)
every call raises; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "Bit1Error", "OK", "EINVAL", "ESHAPE", "ERANGE", "ECUDA", "ENAN",
    "F32", "BF16", "F16", "AUTO", "SIMPLE", "LUT", "SPLITK", "TC", "LUT6", "STREAM", "MMA", "FLAG_PDL",
    "FLAG_SWIGLU", "EPI_NONE", "EPI_SWIGLU",
    "bit1_pack", "bit1_pack_flags_status", "bit1_gemv", "bit1_gemv_ex",
    "bit1_gemv_workspace_bytes", "bit1_gemv_pick", "bit1_gemv_launches",
    "bit1_xor_patch", "bit1_status_str", "bit1_version", "bit1_device_wait_timeouts",
    "bit1_group_plan_bytes", "bit1_group_plan", "bit1_gemv_group", "GroupPlan",
    "bit1_group_tc_plan_bytes", "bit1_group_tc_workspace_bytes", "bit1_group_plan_tc",
    "library_path", "load", "bit1_gemv_tc_noalloc",
    "LAYOUT_CANONICAL", "LAYOUT_G128X", "bit1_repack_g128x", "bit1_unpack_g128x",
    "bit1_ternary_planes", "bit1_gemv_ternary", "bit1_gemv_ternary_workspace_bytes",
    "bit1_gemv_ternary_launches", "bit1_ternary_combine",
    "bit1_t5_pack", "bit1_t5_to_planes", "bit1_gemv_t5", "bit1_gemv_t5_launches",
    "bit1_selftest_wait_timeout",
]

OK, EINVAL, ESHAPE, ERANGE, ECUDA, ENAN = 0, 1, 2, 3, 4, 5
F32, BF16, F16 = 0, 1, 2
AUTO, SIMPLE, LUT, SPLITK, TC, LUT6, STREAM, MMA = 0, 1, 2, 3, 4, 5, 6, 7
FLAG_PDL = 1
FLAG_SWIGLU = 2
EPI_NONE, EPI_SWIGLU = 0, 1
LAYOUT_CANONICAL, LAYOUT_G128X = 0, 1

class _Problem(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("y_dtype", ctypes.c_int), ("epilogue", ctypes.c_int)]


_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libbit1.so")
_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _LIB_PATH


class Bit1Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {bit1_status_str(status)} (status {status})")


def load():
    """Load libbit1.so (raises if it is missing: the CUDA path is the only path)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"bit1 CUDA library not found at {_LIB_PATH}; build it with "
                "`python -m bit_weight_gemv_sign_b300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(_LIB_PATH)
        p, i64, i32, u32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_size_t
        lib.bit1_pack.argtypes = [p, i32, i64, i64, p, p, p, p]
        lib.bit1_pack.restype = i32
        lib.bit1_pack_flags_status.argtypes = [u32]
        lib.bit1_pack_flags_status.restype = i32
        lib.bit1_gemv.argtypes = [p, p, p, i64, i64, i64, p, i32, p, sz, p]
        lib.bit1_gemv.restype = i32
        lib.bit1_gemv_ex.argtypes = [p, p, p, i64, i64, i64, p, i32, p, sz, i32, ctypes.c_uint, p]
        lib.bit1_gemv_ex.restype = i32
        lib.bit1_gemv_workspace_bytes.argtypes = [i64, i64, i64]
        lib.bit1_gemv_workspace_bytes.restype = sz
        lib.bit1_gemv_pick.argtypes = [i64, i64, i64, sz]
        lib.bit1_gemv_pick.restype = i32
        lib.bit1_gemv_launches.argtypes = [i64, i64, i64, i32]
        lib.bit1_gemv_launches.restype = i32
        lib.bit1_xor_patch.argtypes = [p, i64, i64, p, i64, p]
        lib.bit1_xor_patch.restype = i32
        lib.bit1_status_str.argtypes = [i32]
        lib.bit1_status_str.restype = ctypes.c_char_p
        lib.bit1_version.argtypes = []
        lib.bit1_version.restype = ctypes.c_char_p
        lib.bit1_device_wait_timeouts.argtypes = []
        lib.bit1_device_wait_timeouts.restype = ctypes.c_uint
        lib.bit1_selftest_wait_timeout.argtypes = [p, p]
        lib.bit1_selftest_wait_timeout.restype = i32
        lib.bit1_group_plan_bytes.argtypes = [i32]
        lib.bit1_group_plan_bytes.restype = sz
        lib.bit1_group_plan.argtypes = [ctypes.POINTER(_Problem), i32, p, sz]
        lib.bit1_group_plan.restype = i32
        lib.bit1_group_plan_batched.argtypes = [ctypes.POINTER(_Problem), i32, i32, p, sz]
        lib.bit1_group_plan_batched.restype = i32
        lib.bit1_group_plan_ex.argtypes = [ctypes.POINTER(_Problem), i32, i32, i32, p, sz]
        lib.bit1_group_plan_ex.restype = i32
        lib.bit1_group_plan_mma.argtypes = [ctypes.POINTER(_Problem), i32, i32, p, sz]
        lib.bit1_group_plan_mma.restype = i32
        lib.bit1_repack_g128x.argtypes = [p, i64, i64, p, p]
        lib.bit1_repack_g128x.restype = i32
        lib.bit1_unpack_g128x.argtypes = [p, i64, i64, p, p]
        lib.bit1_unpack_g128x.restype = i32
        lib.bit1_gemv_group.argtypes = [p, p, ctypes.c_uint, p]
        lib.bit1_gemv_group.restype = i32
        lib.bit1_group_tc_plan_bytes.argtypes = [i32]
        lib.bit1_group_tc_plan_bytes.restype = sz
        lib.bit1_group_tc_workspace_bytes.argtypes = [ctypes.POINTER(_Problem), i32, i32]
        lib.bit1_group_tc_workspace_bytes.restype = sz
        lib.bit1_group_plan_tc.argtypes = [ctypes.POINTER(_Problem), i32, i32, p, sz, p, sz]
        lib.bit1_group_plan_tc.restype = i32
        lib.bit1_gemv_tc_noalloc.argtypes = [p, p, p, i64, i64, i64, p, i32, ctypes.c_uint, p]
        lib.bit1_gemv_tc_noalloc.restype = i32
        lib.bit1_ternary_planes.argtypes = [p, i64, i64, p, p, p, p]
        lib.bit1_ternary_planes.restype = i32
        lib.bit1_gemv_ternary_workspace_bytes.argtypes = [i64, i64, i64]
        lib.bit1_gemv_ternary_workspace_bytes.restype = sz
        lib.bit1_gemv_ternary.argtypes = [p, p, p, p, i64, i64, i64, p, i32, p, sz, i32, ctypes.c_uint, p]
        lib.bit1_gemv_ternary.restype = i32
        lib.bit1_gemv_ternary_launches.argtypes = [i64, i64, i64, i32]
        lib.bit1_gemv_ternary_launches.restype = i32
        lib.bit1_ternary_combine.argtypes = [p, p, i64, p, i32, p]
        lib.bit1_ternary_combine.restype = i32
        lib.bit1_t5_pack.argtypes = [p, i64, i64, p, p, p]
        lib.bit1_t5_pack.restype = i32
        lib.bit1_t5_to_planes.argtypes = [p, i64, i64, p, p, p, p]
        lib.bit1_t5_to_planes.restype = i32
        lib.bit1_gemv_t5.argtypes = [p, p, p, i64, i64, i64, p, i32, p]
        lib.bit1_gemv_t5.restype = i32
        lib.bit1_gemv_t5_launches.argtypes = [i64, i64, i64]
        lib.bit1_gemv_t5_launches.restype = i32
        _lib = lib
        return lib


def bit1_status_str(status: int) -> str:
    return load().bit1_status_str(int(status)).decode()


def bit1_version() -> str:
    return load().bit1_version().decode()


def bit1_device_wait_timeouts() -> int:
    return int(load().bit1_device_wait_timeouts())


def bit1_selftest_wait_timeout(done, stream=None) -> None:
    """Run the bounded-wait self-test kernel (``done``: int32 [1] CUDA tensor,
    set to 1 when the kernel exits)."""
    import torch
    st = load().bit1_selftest_wait_timeout(_dptr(done, "done", (torch.int32,)), _stream(stream))
    _check(st, "bit1_selftest_wait_timeout")


# ---------------------------------------------------------------- helpers

def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dptr(t, name: str, dtype=None) -> int:
    import torch
    if t is None:
        return 0
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if dtype is not None and t.dtype not in dtype:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtype}")
    return t.data_ptr()


def _check(st: int, where: str):
    if st != OK:
        raise Bit1Error(st, where)


_DT = {"float32": F32, "bfloat16": BF16, "float16": F16}


# ---------------------------------------------------------------- entry points

def bit1_pack(w, bits=None, scales=None, flags=None, stream=None):
    """Pack fp32/bf16/fp16 weights [N, K] (CUDA tensor) into (bits uint8 [N, K/8],
    scales int16 [N, K/128] holding fp16 patterns).  ``flags`` (int32 [1] CUDA
    tensor) receives the NaN / range flag word; read it with
    ``bit1_pack_flags_status(int(flags.item()))`` after synchronising."""
    import torch
    N, K = w.shape
    if bits is None:
        bits = torch.empty((N, K // 8), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((N, max(K // 128, 1)), dtype=torch.int16, device=w.device)
    dt = _DT.get(str(w.dtype).replace("torch.", ""))
    if dt is None:
        raise TypeError(f"unsupported weight dtype {w.dtype}")
    st = load().bit1_pack(_dptr(w, "w"), dt, N, K, _dptr(bits, "bits"), _dptr(scales, "scales"),
                          _dptr(flags, "flags"), _stream(stream))
    _check(st, "bit1_pack")
    return bits, scales


def bit1_pack_flags_status(flags: int) -> int:
    return int(load().bit1_pack_flags_status(int(flags) & 0xFFFFFFFF))


def bit1_gemv_ex(bits, scales, x, y=None, y_dtype=None, workspace=None, variant=AUTO, flags=0,
                 stream=None, N=None, K=None):
    """y[B, N] = x[B, K] (bf16) times the packed 1-bit matrix (bits [N, K/8],
    scales [N, K/128] fp16 patterns).  Returns y (fp32 unless y_dtype/BF16).
    With FLAG_SWIGLU in ``flags`` the rows are (gate, up) pairs and y is
    h = silu(gate) * up, [B, N/2]."""
    import torch
    B = x.shape[0] if x.dim() == 2 else 1
    K = x.shape[-1] if K is None else K
    N = bits.shape[0] if N is None else N
    if y is None:
        yt = torch.bfloat16 if y_dtype == BF16 else torch.float32
        y = torch.empty((B, N // 2 if int(flags) & FLAG_SWIGLU else N), dtype=yt, device=x.device)
    ydt = BF16 if y.dtype == torch.bfloat16 else F32
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("y must be float32 or bfloat16")
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dptr(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = load().bit1_gemv_ex(_dptr(bits, "bits"), _dptr(scales, "scales"), _dptr(x, "x"),
                             B, N, K, _dptr(y, "y"), ydt, ws_ptr, ws_bytes, int(variant),
                             int(flags), _stream(stream))
    _check(st, "bit1_gemv")
    return y


def bit1_gemv(bits, scales, x, y=None, y_dtype=None, workspace=None, stream=None):
    return bit1_gemv_ex(bits, scales, x, y=y, y_dtype=y_dtype, workspace=workspace,
                        variant=AUTO, flags=0, stream=stream)


def bit1_gemv_tc_noalloc(bits, scales, x, y=None, y_dtype=None, flags=0, stream=None, N=None, K=None):
    """The tensor-core product without a workspace: its scratch is a static
    device array shared by every call on the device (calls must not overlap
    on the GPU; the first call on a device must precede any stream capture)."""
    import torch
    B = x.shape[0] if x.dim() == 2 else 1
    K = x.shape[-1] if K is None else K
    N = bits.shape[0] if N is None else N
    if y is None:
        yt = torch.bfloat16 if y_dtype == BF16 else torch.float32
        y = torch.empty((B, N // 2 if int(flags) & FLAG_SWIGLU else N), dtype=yt, device=x.device)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("y must be float32 or bfloat16")
    ydt = BF16 if y.dtype == torch.bfloat16 else F32
    st = load().bit1_gemv_tc_noalloc(_dptr(bits, "bits"), _dptr(scales, "scales"), _dptr(x, "x"),
                                     B, N, K, _dptr(y, "y"), ydt, int(flags), _stream(stream))
    _check(st, "bit1_gemv_tc_noalloc")
    return y


def bit1_gemv_workspace_bytes(B: int, N: int, K: int) -> int:
    return int(load().bit1_gemv_workspace_bytes(B, N, K))


def bit1_gemv_pick(B: int, N: int, K: int, ws_bytes: int = 0) -> int:
    return int(load().bit1_gemv_pick(B, N, K, ws_bytes))


def bit1_gemv_launches(B: int, N: int, K: int, variant: int = AUTO) -> int:
    return int(load().bit1_gemv_launches(B, N, K, variant))


def bit1_xor_patch(bits, rows, N=None, K=None, stream=None):
    """Flip every sign bit of the listed rows of ``bits`` in place (rows: a
    host sequence of ints).  Applying the same list again removes the patch."""
    import numpy as np
    N = bits.shape[0] if N is None else N
    K = bits.shape[1] * 8 if K is None else K
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1))
    st = load().bit1_xor_patch(_dptr(bits, "bits"), N, K, r.ctypes.data if r.size else None,
                               r.size, _stream(stream))
    _check(st, "bit1_xor_patch")
    return bits


# ---------------------------------------------------------------- grouped GEMV

def bit1_group_plan_bytes(count: int) -> int:
    return int(load().bit1_group_plan_bytes(int(count)))


def _problem_array(problems):
    import torch
    arr = (_Problem * len(problems))()
    for i, pr in enumerate(problems):
        bits, scales, x, y = pr[:4]
        epi = int(pr[4]) if len(pr) > 4 else EPI_NONE
        if y.dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("y must be float32 or bfloat16")
        arr[i] = _Problem(_dptr(bits, "bits"), _dptr(scales, "scales"), _dptr(x, "x"), _dptr(y, "y"),
                          bits.shape[0], x.shape[-1], BF16 if y.dtype == torch.bfloat16 else F32, epi)
    return arr


def bit1_group_tc_plan_bytes(count: int) -> int:
    return int(load().bit1_group_tc_plan_bytes(int(count)))


def bit1_group_tc_workspace_bytes(problems, B: int) -> int:
    """Workspace bytes of a tensor-core grouped plan (0 on invalid arguments)."""
    return int(load().bit1_group_tc_workspace_bytes(_problem_array(problems), len(problems), int(B)))


def bit1_group_plan_tc(problems, B: int, workspace, host_plan_ptr: int, plan_bytes: int) -> None:
    """Encode a tensor-core grouped plan (problems as for bit1_group_plan, x
    [B, K] for every problem) using ``workspace`` (uint8 CUDA tensor of at
    least bit1_group_tc_workspace_bytes bytes)."""
    st = load().bit1_group_plan_tc(_problem_array(problems), len(problems), int(B), _dptr(workspace, "workspace"),
                                   workspace.numel() * workspace.element_size(), host_plan_ptr, plan_bytes)
    _check(st, "bit1_group_plan_tc")


def bit1_group_plan(problems, host_plan_ptr: int, plan_bytes: int, B: int = 1,
                    layout: int = LAYOUT_CANONICAL, mma: bool = False) -> None:
    """problems: sequence of (bits, scales, x, y) or (bits, scales, x, y,
    epilogue) CUDA tensors; x is [B, K] (or [K] at B = 1) bf16 and y [B, N]
    ([B, N/2] with EPI_SWIGLU, the rows then interleaved gate/up pairs).
    B > 1 calls bit1_group_plan_batched; a non-canonical ``layout`` (every
    problem's bits converted with bit1_repack_g128x) bit1_group_plan_ex;
    ``mma`` bit1_group_plan_mma (register-sourced MMAs, B <= 16)."""
    arr = _problem_array(problems)
    if mma:
        if layout != LAYOUT_CANONICAL:
            raise ValueError("the MMA engine takes the canonical layout")
        st = load().bit1_group_plan_mma(arr, len(problems), int(B), host_plan_ptr, plan_bytes)
    elif layout != LAYOUT_CANONICAL:
        st = load().bit1_group_plan_ex(arr, len(problems), int(B), int(layout), host_plan_ptr, plan_bytes)
    elif B == 1:
        st = load().bit1_group_plan(arr, len(problems), host_plan_ptr, plan_bytes)
    else:
        st = load().bit1_group_plan_batched(arr, len(problems), int(B), host_plan_ptr, plan_bytes)
    _check(st, "bit1_group_plan")


def bit1_repack_g128x(bits, out=None, stream=None, N=None, K=None):
    """Sign bits uint8 [N, K/8] (CUDA, canonical layout) -> the g128x layout
    (``out`` may be ``bits`` itself: converted in place).  Returns out."""
    import torch
    N = bits.shape[0] if N is None else N
    K = bits.shape[-1] * 8 if K is None else K
    if out is None:
        out = torch.empty_like(bits)
    _check(load().bit1_repack_g128x(_dptr(bits, "bits"), N, K, _dptr(out, "out"), _stream(stream)),
           "bit1_repack_g128x")
    return out


def bit1_unpack_g128x(bits, out=None, stream=None, N=None, K=None):
    """The inverse of bit1_repack_g128x."""
    import torch
    N = bits.shape[0] if N is None else N
    K = bits.shape[-1] * 8 if K is None else K
    if out is None:
        out = torch.empty_like(bits)
    _check(load().bit1_unpack_g128x(_dptr(bits, "bits"), N, K, _dptr(out, "out"), _stream(stream)),
           "bit1_unpack_g128x")
    return out


def bit1_gemv_group(device_plan_ptr: int, host_plan_ptr: int, flags: int = 0, stream=None) -> None:
    st = load().bit1_gemv_group(device_plan_ptr, host_plan_ptr, int(flags), _stream(stream))
    _check(st, "bit1_gemv_group")


class GroupPlan:
    """A grouped-GEMV plan: the encoded host copy and its device copy (both
    128-byte aligned).  The tensors named in ``problems`` must stay alive and
    in place while the plan is used.  ``tensor_cores``: the tcgen05 grouped
    kernel (B <= 64, canonical layout; the plan owns its workspace); ``mma``:
    the grouped kernel's register-sourced MMA engine (B <= 16)."""

    def __init__(self, problems, device="cuda", B: int = 1, layout: int = LAYOUT_CANONICAL,
                 tensor_cores: bool = False, mma: bool = False):
        import numpy as np
        import torch
        self.problems = list(problems)
        self.B = int(B)
        self.tensor_cores = bool(tensor_cores)
        self.layout = int(layout)
        if self.tensor_cores:
            if self.layout != LAYOUT_CANONICAL:
                raise ValueError("the tensor-core grouped kernel takes the canonical layout")
            self.nbytes = bit1_group_tc_plan_bytes(len(self.problems))
            nws = bit1_group_tc_workspace_bytes(self.problems, self.B)
            if nws == 0:
                raise Bit1Error(ESHAPE, "bit1_group_tc_workspace_bytes")
            self.workspace = torch.empty(nws, dtype=torch.uint8, device=device)
        else:
            self.nbytes = bit1_group_plan_bytes(len(self.problems))
        self._host_raw = np.zeros(self.nbytes + 128, dtype=np.uint8)
        off = (-self._host_raw.ctypes.data) % 128
        self.host = self._host_raw[off: off + self.nbytes]
        if self.tensor_cores:
            bit1_group_plan_tc(self.problems, self.B, self.workspace, self.host.ctypes.data, self.nbytes)
        else:
            bit1_group_plan(self.problems, self.host.ctypes.data, self.nbytes, self.B, self.layout, mma=mma)
        self._dev_raw = torch.empty(self.nbytes + 128, dtype=torch.uint8, device=device)
        doff = (-self._dev_raw.data_ptr()) % 128
        self.dev = self._dev_raw[doff: doff + self.nbytes]
        self.dev.copy_(torch.from_numpy(self.host))

    def run(self, flags: int = 0, stream=None) -> None:
        bit1_gemv_group(self.dev.data_ptr(), self.host.ctypes.data, flags, stream)


# ---------------------------------------------------------------- ternary (2-bit slots)

def bit1_ternary_planes(codes, a=None, b=None, flags=None, stream=None):
    """Ternary codes int8 [N, K] (CUDA, each -1/0/+1) -> sign planes (a, b),
    uint8 [N, K/8] each, with t = (a + b) / 2.  ``flags`` (int32 [1] CUDA
    tensor) receives the code-range flag (``bit1_pack_flags_status``)."""
    import torch
    N, K = codes.shape
    if a is None:
        a = torch.empty((N, K // 8), dtype=torch.uint8, device=codes.device)
    if b is None:
        b = torch.empty((N, K // 8), dtype=torch.uint8, device=codes.device)
    st = load().bit1_ternary_planes(_dptr(codes, "codes", (torch.int8,)), N, K, _dptr(a, "a"),
                                    _dptr(b, "b"), _dptr(flags, "flags"), _stream(stream))
    _check(st, "bit1_ternary_planes")
    return a, b


def bit1_gemv_ternary_workspace_bytes(B: int, N: int, K: int) -> int:
    return int(load().bit1_gemv_ternary_workspace_bytes(B, N, K))


def bit1_gemv_ternary_launches(B: int, N: int, K: int, variant: int = AUTO) -> int:
    return int(load().bit1_gemv_ternary_launches(B, N, K, int(variant)))


def bit1_gemv_ternary(a, b, scales, x, y=None, y_dtype=None, workspace=None, variant=AUTO, flags=0,
                      stream=None, N=None, K=None):
    """y[B, N] = x[B, K] (bf16) times the ternary matrix given by its planes
    a, b (uint8 [N, K/8]) and scales [N, K/128].  ``workspace`` defaults to
    a fresh buffer of bit1_gemv_ternary_workspace_bytes bytes.  With
    FLAG_SWIGLU the rows are gate/up pairs and y is [B, N/2]."""
    import torch
    B = x.shape[0] if x.dim() == 2 else 1
    K = x.shape[-1] if K is None else K
    N = a.shape[0] if N is None else N
    if y is None:
        yt = torch.bfloat16 if y_dtype == BF16 else torch.float32
        y = torch.empty((B, N // 2 if int(flags) & FLAG_SWIGLU else N), dtype=yt, device=x.device)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("y must be float32 or bfloat16")
    ydt = BF16 if y.dtype == torch.bfloat16 else F32
    if workspace is None:
        workspace = torch.empty(max(bit1_gemv_ternary_workspace_bytes(B, N, K), 256),
                                dtype=torch.uint8, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = load().bit1_gemv_ternary(_dptr(a, "a"), _dptr(b, "b"), _dptr(scales, "scales"), _dptr(x, "x"),
                                  B, N, K, _dptr(y, "y"), ydt, _dptr(workspace, "workspace"), ws_bytes,
                                  int(variant), int(flags), _stream(stream))
    _check(st, "bit1_gemv_ternary")
    return y


def bit1_ternary_combine(ya, yb, y, stream=None) -> None:
    """y = (ya + yb) / 2 elementwise; ya, yb fp32, y fp32 or bf16, same length."""
    import torch
    n = ya.numel()
    if yb.numel() != n or y.numel() != n:
        raise ValueError("ya, yb and y must have the same number of elements")
    ydt = BF16 if y.dtype == torch.bfloat16 else F32
    st = load().bit1_ternary_combine(_dptr(ya, "ya", (torch.float32,)), _dptr(yb, "yb", (torch.float32,)),
                                     n, _dptr(y, "y", (torch.float32, torch.bfloat16)), ydt, _stream(stream))
    _check(st, "bit1_ternary_combine")


# ---------------------------------------------------------------- ternary (five codes per byte)

def bit1_t5_pack(codes, packed=None, flags=None, stream=None):
    """Codes int8 [N, K] (CUDA) -> packed uint8 [N, K/128*26]."""
    import torch
    N, K = codes.shape
    if packed is None:
        packed = torch.empty((N, (K // 128) * 26), dtype=torch.uint8, device=codes.device)
    st = load().bit1_t5_pack(_dptr(codes, "codes", (torch.int8,)), N, K, _dptr(packed, "packed"),
                             _dptr(flags, "flags"), _stream(stream))
    _check(st, "bit1_t5_pack")
    return packed


def bit1_t5_to_planes(packed, K, a=None, b=None, flags=None, stream=None):
    """Packed bytes [N, K/128*26] -> the 2-bit-slot planes (a, b), uint8 [N, K/8] each."""
    import torch
    N = packed.shape[0]
    if a is None:
        a = torch.empty((N, K // 8), dtype=torch.uint8, device=packed.device)
    if b is None:
        b = torch.empty((N, K // 8), dtype=torch.uint8, device=packed.device)
    st = load().bit1_t5_to_planes(_dptr(packed, "packed"), N, K, _dptr(a, "a"), _dptr(b, "b"),
                                  _dptr(flags, "flags"), _stream(stream))
    _check(st, "bit1_t5_to_planes")
    return a, b


def bit1_gemv_t5_launches(B: int, N: int, K: int) -> int:
    return int(load().bit1_gemv_t5_launches(B, N, K))


def bit1_gemv_t5(packed, scales, x, y=None, y_dtype=None, stream=None, N=None, K=None):
    """y[B, N] = x[B, K] (bf16) times the ternary matrix packed five codes per byte."""
    import torch
    B = x.shape[0] if x.dim() == 2 else 1
    K = x.shape[-1] if K is None else K
    N = packed.shape[0] if N is None else N
    if y is None:
        yt = torch.bfloat16 if y_dtype == BF16 else torch.float32
        y = torch.empty((B, N), dtype=yt, device=x.device)
    if y.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("y must be float32 or bfloat16")
    ydt = BF16 if y.dtype == torch.bfloat16 else F32
    st = load().bit1_gemv_t5(_dptr(packed, "packed"), _dptr(scales, "scales"), _dptr(x, "x"), B, N, K,
                             _dptr(y, "y"), ydt, _stream(stream))
    _check(st, "bit1_gemv_t5")
    return y
