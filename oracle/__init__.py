"""CPU oracle for dense transposed convolution (ConvTranspose).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` import this package.  The product library (``transposed_convolution_gb300``)
never imports, links or calls it, and the two share no code.

The arithmetic lives in ``ctr_oracle.c``: the plain scatter form
``y[b, oc, i*s - p + t] += x[b, ic, i] * w[ic, oc, t]`` summed in double, started from the
bias, following the gather condition and the un-flipped weight layout of "[ExecuTorch][WebGPU]
Add optimized conv2d op" (Implementation) and the bias-first accumulation of "[WebGPU]
optimizations for audio models" (ConvTranspose commits).  This module only marshals numpy
arrays into that library and adds the element-wise helpers the tests need (rounding to the
I/O precision (fp32, bf16, fp16), LeakyReLU, the rel_l2 metric).

Every function here is pinned by ``tests/test_oracle_pins.py`` against something other than
itself: torch's float64 CPU ConvTranspose, the adjoint of a forward convolution built
element by element, hand-computed fixtures, a plain matmul, the polyphase identity and the
closed-form iSTFT of a sinusoid.  ``leaky_relu`` and the stage order of the vocoder stack are
a reading of "LeakyReLU(0.1) between stages": parity unpinned by the pages for that
placement (the pages print no stack output).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ctr_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libctr_oracle.so")
_lock = threading.Lock()
_lib = None

_I64P = ctypes.POINTER(ctypes.c_int64)
_F64P = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ``ctr_oracle.c`` with gcc and OpenMP into ``_build/libctr_oracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.ctr_oracle_output_size.restype = ctypes.c_int64
            lib.ctr_oracle_output_size.argtypes = [ctypes.c_int64] * 5
            lib.ctr_oracle_output_size_ex.restype = ctypes.c_int64
            lib.ctr_oracle_output_size_ex.argtypes = [ctypes.c_int64] * 7
            lib.ctr_oracle_max_threads.restype = ctypes.c_int
            lib.ctr_oracle_set_threads.restype = None
            lib.ctr_oracle_set_threads.argtypes = [ctypes.c_int]
            lib.ctr_oracle_landed_pairs.restype = ctypes.c_int64
            lib.ctr_oracle_landed_pairs.argtypes = [ctypes.c_int] + [_I64P] * 5
            lib.ctr_oracle_conv_transpose.restype = ctypes.c_int
            lib.ctr_oracle_conv_transpose.argtypes = (
                [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
                + [_I64P] * 5 + [_F64P] * 4)
            lib.ctr_oracle_conv_transpose_groups.restype = ctypes.c_int
            lib.ctr_oracle_conv_transpose_groups.argtypes = (
                [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
                + [_I64P] * 5 + [_F64P] * 4)
            lib.ctr_oracle_conv_transpose_ex.restype = ctypes.c_int
            lib.ctr_oracle_conv_transpose_ex.argtypes = (
                [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
                + [_I64P] * 7 + [_F64P] * 4)
            _lib = lib
    return _lib


def _i64(vals):
    arr = (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])
    return arr


def _tuple(v, ndim):
    if isinstance(v, (int, np.integer)):
        return (int(v),) * ndim
    v = tuple(int(a) for a in v)
    assert len(v) == ndim
    return v


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().ctr_oracle_max_threads())


def set_threads(n: int) -> None:
    """Run the oracle on n threads (n <= 0: the OpenMP default).  The result does not depend
    on the thread count; only the CPU-baseline timing uses this."""
    _load().ctr_oracle_set_threads(int(n))


def output_size(L_in: int, k: int, s: int, p: int, op: int = 0, d: int = 1,
                p_end=None) -> int:
    """L_out = (L_in - 1)*s + (k - 1)*d + 1 + op - p - p_end for one spatial dimension
    (p_end defaults to p: then (L_in - 1)*s - 2p + k + op without dilation)."""
    if d == 1 and p_end is None:
        return int(_load().ctr_oracle_output_size(L_in, k, s, p, op))
    return int(_load().ctr_oracle_output_size_ex(L_in, k, s, d, p, p if p_end is None else p_end,
                                                 op))


def landed_pairs(in_sp, kernel, stride, padding, output_padding=0) -> int:
    """(input position, tap) pairs that land inside the output, per (C_in, C_out) pair."""
    ndim = len(in_sp)
    k = _tuple(kernel, ndim)
    s = _tuple(stride, ndim)
    p = _tuple(padding, ndim)
    op = _tuple(output_padding, ndim)
    return int(_load().ctr_oracle_landed_pairs(ndim, _i64(in_sp), _i64(k), _i64(s),
                                               _i64(p), _i64(op)))


def conv_transpose(x, w, bias=None, stride=1, padding=0, output_padding=0,
                   groups=1, dilation=1, padding_end=None) -> np.ndarray:
    """ConvTranspose in double.

    x: [B, C_in, L] or [B, C_in, H, W]; w: [C_in, C_out/groups, k] or [C_in, C_out/groups,
    kH, kW] (un-flipped torch layout); bias: [C_out] or None; groups divides C_in and C_out
    (groups = C_in = C_out is the depthwise case).  ``padding`` is the front pad of each
    spatial dimension and ``padding_end`` the back pad (default: the front pad, torch's
    symmetric padding); ``dilation`` spaces the taps.  Inputs are converted to float64
    exactly (fp32 and bf16 values are representable).  Returns float64
    [B, C_out, L_out] / [B, C_out, H_out, W_out].
    """
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
    ndim = x.ndim - 2
    assert ndim in (1, 2) and w.ndim == x.ndim
    B, C_in = x.shape[:2]
    assert w.shape[0] == C_in
    G = int(groups)
    C_out = w.shape[1] * G
    in_sp = x.shape[2:]
    k = w.shape[2:]
    s = _tuple(stride, ndim)
    p = _tuple(padding, ndim)
    pe = p if padding_end is None else _tuple(padding_end, ndim)
    d = _tuple(dilation, ndim)
    op = _tuple(output_padding, ndim)
    out_sp = tuple(output_size(in_sp[i], k[i], s[i], p[i], op[i], d[i], pe[i])
                   for i in range(ndim))
    if min(out_sp) <= 0:
        raise ValueError("empty output for this geometry")
    y = np.empty((B, C_out) + out_sp, dtype=np.float64)
    bptr = None
    if bias is not None:
        bias = np.ascontiguousarray(np.asarray(bias, dtype=np.float64))
        assert bias.shape == (C_out,)
        bptr = bias.ctypes.data_as(_F64P)
    lib = _load()
    if d == (1,) * ndim and pe == p:
        rc = lib.ctr_oracle_conv_transpose_groups(
            ndim, B, C_in, C_out, G, _i64(in_sp), _i64(k), _i64(s), _i64(p), _i64(op),
            x.ctypes.data_as(_F64P), w.ctypes.data_as(_F64P), bptr, y.ctypes.data_as(_F64P))
    else:
        rc = lib.ctr_oracle_conv_transpose_ex(
            ndim, B, C_in, C_out, G, _i64(in_sp), _i64(k), _i64(s), _i64(d), _i64(p), _i64(pe),
            _i64(op), x.ctypes.data_as(_F64P), w.ctypes.data_as(_F64P), bptr,
            y.ctypes.data_as(_F64P))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (rc=%d)" % rc)
    return y


def leaky_relu(y, negative_slope: float) -> np.ndarray:
    """max(y, 0) + slope * min(y, 0), element-wise, in double."""
    y = np.asarray(y, dtype=np.float64)
    return np.where(y >= 0.0, y, y * float(negative_slope))


def round_f32(a) -> np.ndarray:
    """Round to the nearest fp32 (ties to even); returned as float64."""
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(a) -> np.ndarray:
    """Round a double straight to the nearest bfloat16 (ties to even); returned as float64.

    bfloat16 keeps 8 significant bits and fp32's exponent range.  For |x| in
    [2**(e-1), 2**e) the spacing is 2**(e-8); below the smallest normal (2**-126) it stays
    2**-133.  Values past the largest finite bfloat16 after rounding become +-inf; NaN and
    inf pass through.
    """
    x = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)
        e = np.maximum(e, -125)
        q = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
        q = np.where(np.abs(q) > _BF16_MAX, np.copysign(np.inf, x), q)
    return np.where(np.isfinite(x), q, x)


_F16_MAX = 65504.0


def round_f16(a) -> np.ndarray:
    """Round a double straight to the nearest IEEE binary16 value (ties to even); returned as
    float64.

    binary16 keeps 11 significant bits and exponents -14 .. 15: for |x| in [2**(e-1), 2**e)
    the spacing is 2**(e-11); below the smallest normal (2**-14) it stays 2**-24.  Values
    past the largest finite value (65504) after rounding become +-inf; NaN and inf pass
    through.
    """
    x = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)
        e = np.maximum(e, -13)
        q = np.ldexp(np.rint(np.ldexp(x, 11 - e)), e - 11)
        q = np.where(np.abs(q) > _F16_MAX, np.copysign(np.inf, x), q)
    return np.where(np.isfinite(x), q, x)


def rel_l2(y, ref) -> float:
    """||y - ref||_2 / ||ref||_2 over all elements, in double."""
    y = np.asarray(y, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    den = float(np.sqrt(np.dot(ref, ref)))
    num = float(np.sqrt(np.dot(y - ref, y - ref)))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
