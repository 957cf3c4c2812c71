"""few_row_packed_gb300 -- Python binding of liblbv, the few-row low-bit
verify matmul for GB300 (sm_103a).

Argument marshalling only: every step of the verify path runs in the CUDA
kernels of liblbv.so, called through its C ABI (include/lbv.h).  PyTorch is
used only for device memory and streams.  There is no fallback: if the
library is not built, ``lib()`` raises.

    Y[M,N] = X[M,K] . dequant(Wp)[K,N],   1 <= M <= 8
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

FMT_SIGN1_G128 = 0
FMT_AFFINE2 = 1
FMT_Q4_0 = 2
F16 = 0
BF16 = 1
PLAN_MEASURE = 0x1
PLAN_FORCE_FEWROW = 0x2
PLAN_FORCE_GEMV = 0x4
PLAN_PDL = 0x8
PLAN_TCGEN05 = 0x10
PLAN_TEST_WAIT_LIMIT = 0x20
PLAN_TC_E4M3 = 0x40
KERNEL_FEWROW = 1
KERNEL_GEMV = 2
KERNEL_FEWROW_TC = 3
KERNEL_FEWROW_TC8 = 4
FUSED_ROTATE = 0x1
FUSED_ARGMAX = 0x2

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_TIMEOUT, ERR_BOUNDS = range(7)

_HERE = os.path.dirname(os.path.abspath(__file__))
# LBV_LIBRARY=checked selects liblbv_checked.so, the build whose kernels check
# their copy and buffer ranges; the default is the release liblbv.so
CHECKED = os.environ.get("LBV_LIBRARY", "") == "checked"
LIB_PATH = os.path.join(_HERE, "liblbv_checked.so" if CHECKED else "liblbv.so")
_lib = None

FMT_BY_NAME = {"sign1_g128": FMT_SIGN1_G128, "affine2": FMT_AFFINE2, "q4_0": FMT_Q4_0}
DTYPE_BY_NAME = {"f16": F16, "bf16": BF16}


class Problem(ctypes.Structure):
    """One problem of a grouped call (lbv_problem)."""
    _fields_ = [("X", ctypes.c_void_p), ("M", ctypes.c_int), ("ldx", ctypes.c_int),
                ("Wp", ctypes.c_void_p), ("Y", ctypes.c_void_p), ("ldy", ctypes.c_int)]


class LbvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"lbv status {status}: {msg}")
        self.status = status


def build(force: bool = False) -> str:
    """Compile the library LIB_PATH names in-tree for sm_103a (nvcc); returns its path."""
    from . import buildlib
    return buildlib.build(force=force, checked=CHECKED)


def lib():
    """The loaded liblbv.so.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "few_row_packed_gb300.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, U, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
        st = ctypes.c_int
        sig = {
            "lbv_packed_bytes": (S, [I, I, I, I]),
            "lbv_pack_sign_g128": (st, [P, P, I, I, P, S]),
            "lbv_pack_affine2": (st, [P, P, P, I, I, I, P, S]),
            "lbv_pack_q4_0": (st, [P, I, I, P, S]),
            "lbv_plan_packed_bytes": (S, [P]),
            "lbv_plan_pack": (st, [P, P, P, P, P, S]),
            "lbv_plan_create": (st, [I, I, I, I, I, U, ctypes.POINTER(P)]),
            "lbv_plan_destroy": (st, [P]),
            "lbv_plan_query": (st, [P, I, ctypes.POINTER(I), ctypes.POINTER(I),
                                    ctypes.POINTER(S)]),
            "lbv_plan_shape": (st, [P] + [ctypes.POINTER(I)] * 4),
            "lbv_plan_set_shape": (st, [P, I, I, I, I]),
            "lbv_plan_measured": (st, [P, I, ctypes.POINTER(ctypes.c_float),
                                       ctypes.POINTER(ctypes.c_float), ctypes.POINTER(I)]),
            "lbv_plan_device_status": (st, [P]),
            "lbv_plan_rows_histogram": (st, [P, P]),
            "lbv_plan_rows_reset": (st, [P]),
            "lbv_group_rows_histogram": (st, [P, P]),
            "lbv_group_rows_reset": (st, [P]),
            "lbv_rows_histogram": (st, [P]),
            "lbv_verify_gemm": (st, [P, P, I, I, P, P, I, P, S, P]),
            "lbv_fwht128": (st, [P, P, I, I, I, P, P]),
            "lbv_fused_workspace_bytes": (S, []),
            "lbv_group_create": (st, [I, I, I, I, P, P, U, ctypes.POINTER(P)]),
            "lbv_group_destroy": (st, [P]),
            "lbv_group_shape": (st, [P, I] + [ctypes.POINTER(I)] * 3),
            "lbv_group_launches": (I, [P]),
            "lbv_group_problem_launch": (I, [P, I]),
            "lbv_group_set_shape": (st, [P, I, I, I]),
            "lbv_group_device_status": (st, [P]),
            "lbv_verify_grouped": (st, [P, P, P]),
            "lbv_fused_rotation": (st, [P, P, I, I, I, P, P]),
            "lbv_verify_fused_noalloc": (st, [P, P, I, I, P, U, P, P, I, P, P, P]),
            "lbv_verify_fused": (st, [P, P, I, I, P, U, P, P, I, P, P, P, S, P]),
            "lbv_dequant_fp16": (st, [P, P, P, P]),
            "lbv_last_error": (ctypes.c_char_p, []),
            "lbv_version": (ctypes.c_char_p, []),
            "lbv_checked_build": (I, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def last_error() -> str:
    return lib().lbv_last_error().decode()


def _check(status: int):
    if status != OK:
        raise LbvError(status, last_error())


def _ptr(t):
    """Device or host address of a torch tensor / numpy array / int / None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# --- packing (host) -------------------------------------------------------------

def packed_bytes(fmt: int, K: int, N: int, group: int = 128) -> int:
    return int(lib().lbv_packed_bytes(fmt, K, N, group))


def _out(fmt, K, N, group):
    n = packed_bytes(fmt, K, N, group)
    if n == 0:
        raise LbvError(ERR_INVALID_ARG, f"invalid shape K={K} N={N} group={group}")
    return np.zeros(n, np.uint8)


def pack_sign_g128(bits, scales, K: int, N: int) -> np.ndarray:
    bits = np.ascontiguousarray(bits, np.uint32)
    scales = np.ascontiguousarray(scales, np.uint16)
    if bits.size != N * (K // 32) or scales.size != N * (K // 128):
        raise LbvError(ERR_INVALID_ARG, "bits/scales size mismatch")
    out = _out(FMT_SIGN1_G128, K, N, 128)
    _check(lib().lbv_pack_sign_g128(_ptr(bits), _ptr(scales), K, N, _ptr(out), out.size))
    return out


def pack_affine2(codes, scales, biases, K: int, N: int, group: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint32)
    scales = np.ascontiguousarray(scales, np.uint16)
    biases = np.ascontiguousarray(biases, np.uint16)
    if codes.size != N * (K // 16) or scales.size != N * (K // group) or biases.size != scales.size:
        raise LbvError(ERR_INVALID_ARG, "codes/scales/biases size mismatch")
    out = _out(FMT_AFFINE2, K, N, group)
    _check(lib().lbv_pack_affine2(_ptr(codes), _ptr(scales), _ptr(biases), K, N, group,
                                  _ptr(out), out.size))
    return out


def pack_q4_0(blocks, K: int, N: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, np.uint8)
    if blocks.size != N * (K // 32) * 18:
        raise LbvError(ERR_INVALID_ARG, "blocks size mismatch")
    out = _out(FMT_Q4_0, K, N, 32)
    _check(lib().lbv_pack_q4_0(_ptr(blocks), K, N, _ptr(out), out.size))
    return out


def pack(fmt: int, parts, K: int, N: int, group: int = 128, plan=None) -> np.ndarray:
    """Canonical arrays (as produced for the format) -> device-layout bytes: the
    default layout, or the layout `plan` reads (needed for PLAN_TCGEN05 and PLAN_TC_E4M3 plans)."""
    if plan is not None:
        return plan.pack(parts)
    if fmt == FMT_SIGN1_G128:
        return pack_sign_g128(parts[0], parts[1], K, N)
    if fmt == FMT_AFFINE2:
        return pack_affine2(parts[0], parts[1], parts[2], K, N, group)
    return pack_q4_0(parts[0], K, N)


# --- plans -----------------------------------------------------------------------

class Plan:
    """A verify plan for one (format, K, N, group, activation dtype)."""

    def __init__(self, fmt: int, K: int, N: int, group: int = 128, xdtype: int = F16,
                 flags: int = 0):
        h = ctypes.c_void_p()
        _check(lib().lbv_plan_create(fmt, K, N, group, xdtype, flags, ctypes.byref(h)))
        self.handle = h
        self.fmt, self.K, self.N, self.group, self.xdtype, self.flags = fmt, K, N, group, xdtype, flags

    def close(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.lbv_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def packed_bytes(self) -> int:
        """Bytes of the device layout this plan's kernels read."""
        return int(lib().lbv_plan_packed_bytes(self.handle))

    def pack(self, parts) -> np.ndarray:
        """Canonical arrays of the plan's format -> this plan's device layout."""
        arrs = [np.ascontiguousarray(a) for a in parts]
        ptrs = [a.ctypes.data for a in arrs] + [None] * (3 - len(arrs))
        out = np.zeros(self.packed_bytes, np.uint8)
        _check(lib().lbv_plan_pack(self.handle, *ptrs[:3], out.ctypes.data, out.size))
        return out

    def query(self, M: int):
        k, s, w = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
        _check(lib().lbv_plan_query(self.handle, M, ctypes.byref(k), ctypes.byref(s),
                                    ctypes.byref(w)))
        return k.value, s.value, w.value

    def shape(self):
        v = [ctypes.c_int() for _ in range(4)]
        _check(lib().lbv_plan_shape(self.handle, *[ctypes.byref(x) for x in v]))
        return tuple(x.value for x in v)

    def set_shape(self, warps: int, tiles_per_warp: int, splits: int, ctas_n: int = 0):
        _check(lib().lbv_plan_set_shape(self.handle, warps, tiles_per_warp, splits, ctas_n))

    def device_status(self):
        """Raises LbvError(ERR_TIMEOUT) if a kernel of this plan gave up a
        bounded wait since the last check (synchronises the device)."""
        _check(lib().lbv_plan_device_status(self.handle))

    def measured(self, M: int):
        f, g, c = ctypes.c_float(), ctypes.c_float(), ctypes.c_int()
        _check(lib().lbv_plan_measured(self.handle, M, ctypes.byref(f), ctypes.byref(g),
                                       ctypes.byref(c)))
        return f.value, g.value, c.value

    def rows_histogram(self):
        """{M: calls} over the plan's successful verify calls since creation or reset."""
        return _rows(lambda c: lib().lbv_plan_rows_histogram(self.handle, c))

    def rows_reset(self):
        _check(lib().lbv_plan_rows_reset(self.handle))


class Group:
    """A grouped-verify plan: problems of shapes K[i] x N[i], one format."""

    def __init__(self, fmt: int, group: int, xdtype: int, shapes, flags: int = 0):
        shapes = list(shapes)
        self.count = len(shapes)
        self.K = (ctypes.c_int * self.count)(*[int(k) for k, _ in shapes])
        self.N = (ctypes.c_int * self.count)(*[int(n) for _, n in shapes])
        h = ctypes.c_void_p()
        _check(lib().lbv_group_create(fmt, group, xdtype, self.count, self.K, self.N, flags,
                                      ctypes.byref(h)))
        self.handle = h
        self.fmt, self.group, self.xdtype, self.flags = fmt, group, xdtype, flags
        self.shapes = shapes

    def close(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.lbv_group_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def launches(self) -> int:
        return int(lib().lbv_group_launches(self.handle))

    def problem_launch(self, i: int) -> int:
        return int(lib().lbv_group_problem_launch(self.handle, i))

    def shape(self, launch: int = 0):
        """(tiles per unit, K split, cluster rows) of launch class `launch`."""
        v = [ctypes.c_int() for _ in range(3)]
        _check(lib().lbv_group_shape(self.handle, launch, *[ctypes.byref(x) for x in v]))
        return tuple(x.value for x in v)

    def set_shape(self, tpw: int, splits: int, rows: int):
        _check(lib().lbv_group_set_shape(self.handle, tpw, splits, rows))

    def device_status(self):
        _check(lib().lbv_group_device_status(self.handle))

    def rows_histogram(self):
        """{M: active problems} over the group's successful calls since creation or reset."""
        return _rows(lambda c: lib().lbv_group_rows_histogram(self.handle, c))

    def rows_reset(self):
        _check(lib().lbv_group_rows_reset(self.handle))


def _rows(call):
    c = (ctypes.c_uint64 * 8)()
    _check(call(c))
    return {m: int(c[m - 1]) for m in range(1, 9)}


def rows_histogram():
    """{M: calls} over every plan and group of the process since the library loaded."""
    return _rows(lambda c: lib().lbv_rows_histogram(c))


def verify_grouped(group: Group, problems, stream=None):
    """problems: one (X, M, Wp, Y) or (X, M, Wp, Y, ldx, ldy) per shape of the
    group (device tensors; M = 0 skips the problem)."""
    arr = (Problem * group.count)()
    for i, pr in enumerate(problems):
        X, M, Wp, Y = pr[:4]
        K, N = group.shapes[i]
        ldx = pr[4] if len(pr) > 4 else K
        ldy = pr[5] if len(pr) > 5 else N
        arr[i] = Problem(_ptr(X), int(M), int(ldx), _ptr(Wp), _ptr(Y), int(ldy))
    _check(lib().lbv_verify_grouped(group.handle, arr, _stream(stream)))


# --- device calls ------------------------------------------------------------------

def verify_gemm(plan: Plan, X, M: int, Wp, Y, ldx: int | None = None, ldy: int | None = None,
                stream=None):
    """Y[:M, :N] = X[:M, :K] . W (device tensors; X fp16/bf16 bits, Y fp32)."""
    ldx = plan.K if ldx is None else ldx
    ldy = plan.N if ldy is None else ldy
    _check(lib().lbv_verify_gemm(plan.handle, _ptr(X), M, ldx, _ptr(Wp), _ptr(Y), ldy, None, 0,
                                 _stream(stream)))


def verify_gemm_host(plan: Plan, x_host, M: int, Wp, y_host, x_dev, y_dev, stream=None):
    """End-to-end call with host buffers: copies X (pinned host) to the device,
    runs the verify, copies Y back and waits.  x_dev / y_dev are caller-owned
    device staging tensors; Wp stays resident on the device."""
    x_dev[:M].copy_(x_host[:M], non_blocking=True)
    verify_gemm(plan, x_dev, M, Wp, y_dev, stream=stream)
    y_host[:M].copy_(y_dev[:M], non_blocking=True)


def fused_workspace_bytes() -> int:
    return int(lib().lbv_fused_workspace_bytes())


def verify_fused(plan: Plan, X, M: int, Wp, ops: int, Y=None, idx=None, val=None,
                 workspace=None, signs=None, ldx: int | None = None, ldy: int | None = None,
                 stream=None):
    """Fused head: Y = rot(X) . W with FUSED_ROTATE, and with FUSED_ARGMAX the
    per-row argmax column (idx, int32 [M]) and logit (val, fp32 [M] or None);
    Y may be None then.  workspace: device bytes, zeroed once by the caller."""
    ldx = plan.K if ldx is None else ldx
    ldy = plan.N if ldy is None else ldy
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().lbv_verify_fused(plan.handle, _ptr(X), M, ldx, _ptr(Wp), ops, _ptr(signs),
                                  _ptr(Y), ldy, _ptr(idx), _ptr(val), _ptr(workspace), ws,
                                  _stream(stream)))


def verify_fused_noalloc(plan: Plan, X, M: int, Wp, ops: int, Y=None, idx=None, val=None,
                         signs=None, ldx: int | None = None, ldy: int | None = None, stream=None):
    """verify_fused with the argmax scratch in the library's own device memory."""
    ldx = plan.K if ldx is None else ldx
    ldy = plan.N if ldy is None else ldy
    _check(lib().lbv_verify_fused_noalloc(plan.handle, _ptr(X), M, ldx, _ptr(Wp), ops,
                                          _ptr(signs), _ptr(Y), ldy, _ptr(idx), _ptr(val),
                                          _stream(stream)))


def fused_rotation(X, Xr, M: int, K: int, dtype: int = F16, signs=None, stream=None):
    """Test export: the rotation exactly as the fused head computes it."""
    _check(lib().lbv_fused_rotation(_ptr(X), _ptr(Xr), M, K, dtype, _ptr(signs),
                                    _stream(stream)))


def fwht128(X, Xr, M: int, K: int, dtype: int = F16, signs=None, stream=None):
    """Blockwise normalized Walsh-Hadamard rotation of M rows of length K."""
    _check(lib().lbv_fwht128(_ptr(X), _ptr(Xr), M, K, dtype, _ptr(signs), _stream(stream)))


def dequant_fp16(plan: Plan, Wp, W, stream=None):
    """Test export: dense fp16 W[K][N] (device) from the packed device layout."""
    _check(lib().lbv_dequant_fp16(plan.handle, _ptr(Wp), _ptr(W), _stream(stream)))


def version() -> str:
    return lib().lbv_version().decode()
