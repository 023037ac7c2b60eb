"""GB300 (sm_103a) dense transposed convolution: Python binding of the C ABI in ``include/ctr.h``.

The binding only marshals arguments: every step of the computation runs in the CUDA kernels
of ``_build/libctr.so``.  PyTorch provides device memory and streams.  There is no CPU or
PyTorch fallback: if the library has not been built the first call raises ImportError, and
any non-OK status from the library raises ``CtrError``.

Low level (same names as the C ABI): ``ctr_plan_create``, ``ctr_plan_set_activation``,
``ctr_plan_set_path``, ``ctr_plan_set_groups``, ``ctr_plan_set_dilation``, ``ctr_plan_set_pads``,
``ctr_plan_set_auto_pad``, ``ctr_plan_set_layout``, ``ctr_plan_set_streaming``, ``ctr_plan_stream_reset``,
``ctr_plan_set_tile``, ``ctr_plan_set_phase_origin``, ``ctr_plan_chain``, ``ctr_plan_get_path``, ``ctr_plan_output_shape``,
``ctr_packed_weight_bytes``, ``ctr_workspace_bytes``, ``ctr_plan_bind_workspace``,
``ctr_prepack_weight``, ``ctr_forward``, ``ctr_forward_noalloc``, ``ctr_forward_fused``,
``ctr_plan_fusable``, ``ctr_plan_check``,
``ctr_plan_set_wait_limit_ns``,
``ctr_plan_set_timing_events``, ``ctr_plan_describe``, ``ctr_plan_destroy``,
``ctr_status_string``, ``ctr_launch_count``.

Inverse STFT (same names as the C ABI): ``ctr_istft_create``, ``ctr_istft_output_length``,
``ctr_istft_workspace_bytes``, ``ctr_istft_bind_workspace``, ``ctr_istft_set_window``,
``ctr_istft_forward``, ``ctr_istft_describe``, ``ctr_istft_set_timing_events``,
``ctr_istft_destroy``.

High level: ``Plan`` (a plan with its packed weight and workspace held as torch tensors),
``Istft`` (an inverse-STFT plan with its workspace), and
``conv_transpose(x, w, bias, stride, padding, output_padding, negative_slope, groups)``.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB as _LIB_PATH

CTR_OK = 0
CTR_ERR_INVALID_ARG = 1
CTR_ERR_UNSUPPORTED = 2
CTR_ERR_MISALIGNED = 3
CTR_ERR_NO_WORKSPACE = 4
CTR_ERR_CUDA = 5
CTR_ERR_DEVICE_TIMEOUT = 6
CTR_ERR_NOT_PREPARED = 7

CTR_F32 = 0
CTR_BF16 = 1
CTR_F16 = 2
CTR_ACT_NONE = 0
CTR_ACT_LEAKY_RELU = 1
CTR_PATH_AUTO = 0
CTR_PATH_POLYPHASE = 1
CTR_PATH_COL2IM = 2
CTR_PATH_GATHER = 3
CTR_PATH_DEPTHWISE = 4
CTR_LAYOUT_NCHW = 0
CTR_LAYOUT_NHWC = 1
CTR_AUTO_PAD_NOTSET = 0
CTR_AUTO_PAD_SAME_UPPER = 1
CTR_AUTO_PAD_SAME_LOWER = 2
CTR_AUTO_PAD_VALID = 3
CTR_PHASE_AUTO = 0
CTR_PHASE_UNPADDED = 1
CTR_PHASE_OUTPUT = 2
PATH_NAMES = {CTR_PATH_POLYPHASE: "polyphase", CTR_PATH_COL2IM: "col2im", CTR_PATH_GATHER: "gather",
              CTR_PATH_DEPTHWISE: "depthwise"}

# Every symbol include/ctr.h declares, with (restype, argtypes).
_vp = ctypes.c_void_p
_i64p = ctypes.POINTER(ctypes.c_int64)
SIGNATURES = {
    "ctr_plan_create": (ctypes.c_int, [ctypes.POINTER(_vp), ctypes.c_int, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int64, _i64p, _i64p, _i64p, _i64p,
                                       _i64p, ctypes.c_int]),
    "ctr_plan_set_activation": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_float]),
    "ctr_plan_set_path": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int]),
    "ctr_plan_set_groups": (ctypes.c_int, [_vp, ctypes.c_int64]),
    "ctr_plan_set_dilation": (ctypes.c_int, [_vp, _i64p]),
    "ctr_plan_set_pads": (ctypes.c_int, [_vp, _i64p, _i64p]),
    "ctr_plan_set_auto_pad": (ctypes.c_int, [_vp, ctypes.c_int, _i64p]),
    "ctr_plan_set_layout": (ctypes.c_int, [_vp, ctypes.c_int]),
    "ctr_plan_set_streaming": (ctypes.c_int, [_vp, ctypes.c_int]),
    "ctr_plan_stream_reset": (ctypes.c_int, [_vp, _vp]),
    "ctr_plan_set_tile": (ctypes.c_int, [_vp, ctypes.c_int]),
    "ctr_plan_set_phase_origin": (ctypes.c_int, [_vp, ctypes.c_int]),
    "ctr_plan_chain": (ctypes.c_int, [_vp, _vp]),
    "ctr_plan_get_path": (ctypes.c_int, [_vp]),
    "ctr_plan_output_shape": (ctypes.c_int, [_vp, _i64p]),
    "ctr_packed_weight_bytes": (ctypes.c_size_t, [_vp]),
    "ctr_workspace_bytes": (ctypes.c_size_t, [_vp]),
    "ctr_plan_bind_workspace": (ctypes.c_int, [_vp, _vp, ctypes.c_size_t]),
    "ctr_prepack_weight": (ctypes.c_int, [_vp, _vp, _vp, _vp]),
    "ctr_forward": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "ctr_forward_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "ctr_forward_fused": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ctr_plan_fusable": (ctypes.c_int, [_vp]),
    "ctr_plan_check": (ctypes.c_int, [_vp, _vp]),
    "ctr_plan_set_wait_limit_ns": (ctypes.c_int, [_vp, ctypes.c_uint64]),
    "ctr_plan_set_timing_events": (ctypes.c_int, [_vp, _vp, _vp]),
    "ctr_plan_describe": (ctypes.c_int, [_vp, ctypes.c_char_p, ctypes.c_size_t]),
    "ctr_plan_destroy": (None, [_vp]),
    "ctr_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ctr_launch_count": (ctypes.c_uint64, []),
    "ctr_istft_create": (ctypes.c_int, [ctypes.POINTER(_vp), ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int]),
    "ctr_istft_output_length": (ctypes.c_int, [_vp, _i64p]),
    "ctr_istft_workspace_bytes": (ctypes.c_size_t, [_vp]),
    "ctr_istft_bind_workspace": (ctypes.c_int, [_vp, _vp, ctypes.c_size_t]),
    "ctr_istft_set_window": (ctypes.c_int, [_vp, _vp, _vp]),
    "ctr_istft_forward": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp]),
    "ctr_istft_describe": (ctypes.c_int, [_vp, ctypes.c_char_p, ctypes.c_size_t]),
    "ctr_istft_set_timing_events": (ctypes.c_int, [_vp, _vp, _vp]),
    "ctr_istft_destroy": (None, [_vp]),
}


class CtrError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where or "ctr", status_string(status), status))


_lib = None
LIB_PATH = _LIB_PATH


def load_library():
    """Load ``_build/libctr.so`` once.  Raises ImportError when it has not been built: there
    is no fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                "transposed_convolution_gb300: %s is missing; build it first with "
                "`python -m transposed_convolution_gb300.build` (nvcc, sm_103a)" % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class _LazyLib:
    def __getattr__(self, name):
        return getattr(load_library(), name)


lib = _LazyLib()


def status_string(status: int) -> str:
    return lib.ctr_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != CTR_OK:
        raise CtrError(status, where)


def _arr(vals):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


# ------------------------------------------------------------------ C-ABI names

ctr_status_string = status_string


def ctr_launch_count() -> int:
    return int(lib.ctr_launch_count())


def ctr_plan_create(ndim, N, C_in, C_out, in_spatial, kernel, stride, padding,
                    output_padding=None, dtype=CTR_F32):
    """Returns a plan handle (int).  Raises CtrError on a non-OK status."""
    h = _vp()
    op = _arr(output_padding) if output_padding is not None else None
    st = lib.ctr_plan_create(ctypes.byref(h), int(ndim), int(N), int(C_in), int(C_out),
                             _arr(in_spatial), _arr(kernel), _arr(stride), _arr(padding), op,
                             int(dtype))
    _check(st, "ctr_plan_create")
    return h.value


def ctr_plan_set_activation(plan, act, negative_slope=0.0):
    _check(lib.ctr_plan_set_activation(plan, int(act), float(negative_slope)),
           "ctr_plan_set_activation")


def ctr_plan_set_path(plan, path, split_k=0):
    _check(lib.ctr_plan_set_path(plan, int(path), int(split_k)), "ctr_plan_set_path")


def ctr_plan_set_groups(plan, groups):
    _check(lib.ctr_plan_set_groups(plan, int(groups)), "ctr_plan_set_groups")


def ctr_plan_set_dilation(plan, dilation):
    _check(lib.ctr_plan_set_dilation(plan, _arr(dilation)), "ctr_plan_set_dilation")


def ctr_plan_set_pads(plan, pads_begin, pads_end):
    _check(lib.ctr_plan_set_pads(plan, _arr(pads_begin), _arr(pads_end)), "ctr_plan_set_pads")


def ctr_plan_set_layout(plan, layout):
    _check(lib.ctr_plan_set_layout(plan, layout), "ctr_plan_set_layout")


def ctr_plan_set_auto_pad(plan, auto_pad, output_shape=None):
    _check(lib.ctr_plan_set_auto_pad(plan, auto_pad, None if output_shape is None
                                     else _arr(output_shape)), "ctr_plan_set_auto_pad")


def ctr_plan_set_streaming(plan, enable):
    _check(lib.ctr_plan_set_streaming(plan, int(enable)), "ctr_plan_set_streaming")


def ctr_plan_stream_reset(plan, stream):
    _check(lib.ctr_plan_stream_reset(plan, stream), "ctr_plan_stream_reset")


def ctr_plan_set_tile(plan, block_n):
    _check(lib.ctr_plan_set_tile(plan, int(block_n)), "ctr_plan_set_tile")


def ctr_plan_set_phase_origin(plan, origin):
    _check(lib.ctr_plan_set_phase_origin(plan, origin), "ctr_plan_set_phase_origin")


def ctr_plan_chain(plan, next_plan):
    _check(lib.ctr_plan_chain(plan, next_plan), "ctr_plan_chain")


def ctr_plan_get_path(plan) -> int:
    return int(lib.ctr_plan_get_path(plan))


def ctr_plan_output_shape(plan, ndim):
    out = (ctypes.c_int64 * ndim)()
    _check(lib.ctr_plan_output_shape(plan, out), "ctr_plan_output_shape")
    return tuple(int(v) for v in out)


def ctr_packed_weight_bytes(plan) -> int:
    return int(lib.ctr_packed_weight_bytes(plan))


def ctr_workspace_bytes(plan) -> int:
    return int(lib.ctr_workspace_bytes(plan))


def ctr_plan_bind_workspace(plan, ptr, nbytes):
    _check(lib.ctr_plan_bind_workspace(plan, ptr, int(nbytes)), "ctr_plan_bind_workspace")


def ctr_prepack_weight(plan, w_ptr, w_packed_ptr, stream):
    _check(lib.ctr_prepack_weight(plan, w_ptr, w_packed_ptr, stream), "ctr_prepack_weight")


def ctr_forward(plan, x_ptr, w_packed_ptr, bias_ptr, y_ptr, stream):
    _check(lib.ctr_forward(plan, x_ptr, w_packed_ptr, bias_ptr, y_ptr, stream), "ctr_forward")


def ctr_forward_noalloc(plan, x_ptr, w_ptr, bias_ptr, y_ptr, stream):
    """The allocation-free forward: scratch in the library's static device array, weight
    passed in its torch layout and packed on every call (see include/ctr.h)."""
    _check(lib.ctr_forward_noalloc(plan, x_ptr, w_ptr, bias_ptr, y_ptr, stream),
           "ctr_forward_noalloc")


def ctr_forward_fused(plan, x_ptr, w_packed_ptr, bias_ptr, next_w_packed_ptr, next_bias_ptr,
                      y_ptr, stream):
    _check(lib.ctr_forward_fused(plan, x_ptr, w_packed_ptr, bias_ptr, next_w_packed_ptr,
                                 next_bias_ptr, y_ptr, stream), "ctr_forward_fused")


def ctr_plan_fusable(plan) -> bool:
    return bool(lib.ctr_plan_fusable(plan))


def ctr_plan_check(plan, stream):
    _check(lib.ctr_plan_check(plan, stream), "ctr_plan_check")


def ctr_plan_set_wait_limit_ns(plan, limit_ns):
    _check(lib.ctr_plan_set_wait_limit_ns(plan, int(limit_ns)), "ctr_plan_set_wait_limit_ns")


def ctr_plan_set_timing_events(plan, before, after):
    """before/after: cudaEvent_t handles (ints) or None."""
    _check(lib.ctr_plan_set_timing_events(plan, before, after), "ctr_plan_set_timing_events")


def ctr_plan_describe(plan) -> str:
    buf = ctypes.create_string_buffer(512)
    _check(lib.ctr_plan_describe(plan, buf, 512), "ctr_plan_describe")
    return buf.value.decode()


def ctr_plan_destroy(plan):
    lib.ctr_plan_destroy(plan)


def ctr_istft_create(N, n_fft, hop, frames, padding=0, output_padding=0, dtype=CTR_F32):
    """Returns an inverse-STFT plan handle (int).  Raises CtrError on a non-OK status."""
    h = _vp()
    _check(lib.ctr_istft_create(ctypes.byref(h), int(N), int(n_fft), int(hop), int(frames),
                                int(padding), int(output_padding), int(dtype)),
           "ctr_istft_create")
    return h.value


def ctr_istft_output_length(plan) -> int:
    v = ctypes.c_int64()
    _check(lib.ctr_istft_output_length(plan, ctypes.byref(v)), "ctr_istft_output_length")
    return int(v.value)


def ctr_istft_workspace_bytes(plan) -> int:
    return int(lib.ctr_istft_workspace_bytes(plan))


def ctr_istft_bind_workspace(plan, ptr, nbytes):
    _check(lib.ctr_istft_bind_workspace(plan, ptr, int(nbytes)), "ctr_istft_bind_workspace")


def ctr_istft_set_window(plan, window_ptr, stream):
    _check(lib.ctr_istft_set_window(plan, window_ptr, stream), "ctr_istft_set_window")


def ctr_istft_forward(plan, spec_ptr, bias_ptr, y_ptr, stream):
    _check(lib.ctr_istft_forward(plan, spec_ptr, bias_ptr, y_ptr, stream), "ctr_istft_forward")


def ctr_istft_describe(plan) -> str:
    buf = ctypes.create_string_buffer(256)
    _check(lib.ctr_istft_describe(plan, buf, 256), "ctr_istft_describe")
    return buf.value.decode()


def ctr_istft_set_timing_events(plan, before, after):
    _check(lib.ctr_istft_set_timing_events(plan, before, after), "ctr_istft_set_timing_events")


def ctr_istft_destroy(plan):
    lib.ctr_istft_destroy(plan)


# ------------------------------------------------------------------ torch-level helpers

def _torch():
    import torch
    return torch


def _dtype_code(dt):
    torch = _torch()
    if dt == torch.float32:
        return CTR_F32
    if dt == torch.bfloat16:
        return CTR_BF16
    if dt == torch.float16:
        return CTR_F16
    raise TypeError("transposed_convolution_gb300 supports float32, bfloat16 and float16, got %s"
                    % dt)


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _tuple(v, n):
    if isinstance(v, int):
        return (v,) * n
    v = tuple(int(a) for a in v)
    if len(v) != n:
        raise ValueError("expected %d values, got %d" % (n, len(v)))
    return v


class Plan:
    """A ConvTranspose plan with its packed weight and workspace as device tensors."""

    def __init__(self, N, C_in, C_out, in_spatial, kernel, stride=1, padding=0,
                 output_padding=0, dtype=None, negative_slope=None, path=CTR_PATH_AUTO,
                 split_k=0, device=None, block_n=0, groups=1, dilation=1, padding_end=None,
                 streaming=False, phase_origin=CTR_PHASE_AUTO, auto_pad=CTR_AUTO_PAD_NOTSET,
                 output_shape=None, layout="nchw"):
        torch = _torch()
        self.ndim = len(in_spatial)
        self.dtype = dtype if dtype is not None else torch.float32
        self.device = torch.device(device if device is not None else "cuda")
        self.N, self.C_in, self.C_out = int(N), int(C_in), int(C_out)
        self.in_spatial = tuple(int(v) for v in in_spatial)
        self.kernel = _tuple(kernel, self.ndim)
        self.stride = _tuple(stride, self.ndim)
        self.padding = _tuple(padding, self.ndim)
        self.output_padding = _tuple(output_padding, self.ndim)
        self.groups = int(groups)
        self.dilation = _tuple(dilation, self.ndim)
        self.padding_end = self.padding if padding_end is None else _tuple(padding_end, self.ndim)
        if layout not in ("nchw", "nhwc"):
            raise ValueError("layout must be 'nchw' or 'nhwc'")
        self.nhwc = layout == "nhwc"
        # With separate back pads or dilation the plan is created unpadded and given its pads
        # afterwards: the symmetric front padding alone may leave no output.
        separate = self.padding_end != self.padding or self.dilation != (1,) * self.ndim
        self.handle = ctr_plan_create(self.ndim, self.N, self.C_in, self.C_out, self.in_spatial,
                                      self.kernel, self.stride,
                                      (0,) * self.ndim if separate else self.padding,
                                      self.output_padding, _dtype_code(self.dtype))
        try:
            if self.nhwc:
                ctr_plan_set_layout(self.handle, CTR_LAYOUT_NHWC)
            if negative_slope is not None:
                ctr_plan_set_activation(self.handle, CTR_ACT_LEAKY_RELU, negative_slope)
            if self.groups != 1:
                ctr_plan_set_groups(self.handle, self.groups)
            if self.dilation != (1,) * self.ndim:
                ctr_plan_set_dilation(self.handle, self.dilation)
            if separate:
                ctr_plan_set_pads(self.handle, self.padding, self.padding_end)
            if auto_pad != CTR_AUTO_PAD_NOTSET or output_shape is not None:
                ctr_plan_set_auto_pad(self.handle, auto_pad, output_shape)
            self.streaming = bool(streaming)
            if self.streaming:
                ctr_plan_set_streaming(self.handle, 1)
            if path != CTR_PATH_AUTO or split_k:
                ctr_plan_set_path(self.handle, path, split_k)
            if block_n:
                ctr_plan_set_tile(self.handle, block_n)
            if phase_origin != CTR_PHASE_AUTO:
                ctr_plan_set_phase_origin(self.handle, phase_origin)
            self.out_spatial = ctr_plan_output_shape(self.handle, self.ndim)
            self.path = ctr_plan_get_path(self.handle)
            self.packed_bytes = ctr_packed_weight_bytes(self.handle)
            self.workspace_bytes = ctr_workspace_bytes(self.handle)
            self.workspace = None
            if self.workspace_bytes:
                self.workspace = torch.empty(self.workspace_bytes, dtype=torch.uint8,
                                             device=self.device)
                ctr_plan_bind_workspace(self.handle, _ptr(self.workspace), self.workspace_bytes)
            if self.streaming:
                ctr_plan_stream_reset(self.handle, _stream_ptr(None))
        except Exception:
            ctr_plan_destroy(self.handle)
            self.handle = None
            raise
        self.w_packed = None
        self.next_plan = None     # chained: this plan's output feeds next_plan's input
        self.prev_plan = None

    @property
    def in_shape(self):
        if self.nhwc:
            return (self.N,) + self.in_spatial + (self.C_in,)
        return (self.N, self.C_in) + self.in_spatial

    @property
    def out_shape(self):
        if self.nhwc:
            return (self.N,) + tuple(self.out_spatial) + (self.C_out,)
        return (self.N, self.C_out) + tuple(self.out_spatial)

    def describe(self) -> str:
        return ctr_plan_describe(self.handle)

    def prepack(self, w, stream=None):
        """Pack the weight [C_in, C_out/groups, k...] (device, plan dtype) into self.w_packed."""
        torch = _torch()
        w = self._checked(w, (self.C_in, self.C_out // self.groups) + self.kernel, "w")
        self.w_packed = torch.empty(max(self.packed_bytes, 16), dtype=torch.uint8,
                                    device=self.device)
        ctr_prepack_weight(self.handle, _ptr(w), _ptr(self.w_packed), _stream_ptr(stream))
        return self.w_packed

    def chain(self, next_plan):
        """Feed this plan's output straight into next_plan's staged input (ctr_plan_chain):
        afterwards forward() writes no y and returns None, and next_plan.forward(None, ...)
        takes its input from there.  chain(None) unchains."""
        ctr_plan_chain(self.handle, next_plan.handle if next_plan is not None else None)
        if self.next_plan is not None:
            self.next_plan.prev_plan = None
        self.next_plan = next_plan
        if next_plan is not None:
            next_plan.prev_plan = self

    def forward(self, x, bias=None, y=None, stream=None):
        torch = _torch()
        if self.w_packed is None:
            raise RuntimeError("Plan.forward before Plan.prepack")
        if x is not None or self.prev_plan is None:
            x = self._checked(x, self.in_shape, "x")
        if bias is not None:
            bias = self._checked(bias, (self.C_out,), "bias")
        if self.next_plan is not None:
            if y is not None:
                raise ValueError("a chained plan writes no y")
        elif y is None:
            y = torch.empty(self.out_shape, dtype=self.dtype, device=self.device)
        else:
            y = self._checked(y, self.out_shape, "y")
        ctr_forward(self.handle, _ptr(x), _ptr(self.w_packed), _ptr(bias), _ptr(y),
                    _stream_ptr(stream))
        return y

    @property
    def fusable(self):
        """Whether forward_fused can run this plan and the plan it is chained to."""
        return ctr_plan_fusable(self.handle)

    def forward_fused(self, x, bias=None, next_bias=None, y=None, stream=None):
        """This plan and the chained next plan in one kernel (ctr_forward_fused): the same
        result as forward(x, bias) then next_plan.forward(None, next_bias, y)."""
        torch = _torch()
        nxt = self.next_plan
        if nxt is None:
            raise ValueError("forward_fused needs a chained next plan")
        if self.w_packed is None or nxt.w_packed is None:
            raise RuntimeError("forward_fused before prepack")
        if x is not None or self.prev_plan is None:
            x = self._checked(x, self.in_shape, "x")
        if bias is not None:
            bias = self._checked(bias, (self.C_out,), "bias")
        if next_bias is not None:
            next_bias = nxt._checked(next_bias, (nxt.C_out,), "next_bias")
        if y is None:
            y = torch.empty(nxt.out_shape, dtype=nxt.dtype, device=nxt.device)
        else:
            y = nxt._checked(y, nxt.out_shape, "y")
        ctr_forward_fused(self.handle, _ptr(x), _ptr(self.w_packed), _ptr(bias),
                          _ptr(nxt.w_packed), _ptr(next_bias), _ptr(y), _stream_ptr(stream))
        return y

    def stream_reset(self, stream=None):
        """Start a new stream: zero the carried input frames (streaming plans)."""
        ctr_plan_stream_reset(self.handle, _stream_ptr(stream))

    def check(self, stream=None):
        ctr_plan_check(self.handle, _stream_ptr(stream))

    def set_timing_events(self, before, after):
        ctr_plan_set_timing_events(self.handle, before, after)

    def set_wait_limit_ns(self, ns):
        ctr_plan_set_wait_limit_ns(self.handle, ns)

    def _checked(self, t, shape, name):
        if tuple(t.shape) != tuple(shape):
            raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
        if t.dtype != self.dtype:
            raise TypeError("%s has dtype %s, expected %s" % (name, t.dtype, self.dtype))
        if t.device.type != "cuda":
            raise ValueError("%s must be a CUDA tensor" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
        return t

    def close(self):
        if getattr(self, "handle", None):
            ctr_plan_destroy(self.handle)     # also unchains on the library side
            self.handle = None
        nxt, prv = getattr(self, "next_plan", None), getattr(self, "prev_plan", None)
        if nxt is not None:
            nxt.prev_plan = None
        if prv is not None:
            prv.next_plan = None
        self.next_plan = self.prev_plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Istft:
    """An inverse-STFT plan (ctr_istft_*) with its workspace held as a torch tensor: the
    ConvTranspose1d with the windowed inverse real-DFT basis, computed by inverse real FFTs.
    spec [N, n_fft + 2, frames] (real parts of bins 0..n_fft/2, then imaginary parts) ->
    y [N, 1, L_out], float32."""

    def __init__(self, N, n_fft, hop, frames, padding=0, output_padding=0, device=None):
        torch = _torch()
        self.N, self.n_fft, self.hop, self.frames = int(N), int(n_fft), int(hop), int(frames)
        self.device = torch.device(device if device is not None else "cuda")
        self.dtype = torch.float32
        self.handle = ctr_istft_create(N, n_fft, hop, frames, padding, output_padding, CTR_F32)
        try:
            self.L_out = ctr_istft_output_length(self.handle)
            self.workspace_bytes = ctr_istft_workspace_bytes(self.handle)
            self.workspace = torch.empty(max(self.workspace_bytes, 16), dtype=torch.uint8,
                                         device=self.device)
            ctr_istft_bind_workspace(self.handle, _ptr(self.workspace), self.workspace_bytes)
        except Exception:
            ctr_istft_destroy(self.handle)
            self.handle = None
            raise
        self.out_shape = (self.N, 1, self.L_out)
        self.window = None
        # Plan-like attributes, so a caller can hold Istft and Plan objects in one list.
        self.path = -1
        self.packed_bytes = 0
        self.next_plan = self.prev_plan = None

    def set_window(self, window, stream=None):
        """The synthesis window [n_fft] (float32, device); kept referenced by the plan."""
        self.window = Plan._checked(self, window, (self.n_fft,), "window")
        ctr_istft_set_window(self.handle, _ptr(self.window), _stream_ptr(stream))

    prepack = set_window

    def set_timing_events(self, before, after):
        ctr_istft_set_timing_events(self.handle, before, after)

    def check(self, stream=None):
        """No device status: the inverse-STFT kernels have no waits that can time out."""

    def forward(self, spec, bias=None, y=None, stream=None):
        torch = _torch()
        if self.window is None:
            raise RuntimeError("Istft.forward before Istft.set_window")
        spec = Plan._checked(self, spec, (self.N, self.n_fft + 2, self.frames), "spec")
        if bias is not None:
            bias = Plan._checked(self, bias, (1,), "bias")
        if y is None:
            y = torch.empty(self.out_shape, dtype=self.dtype, device=self.device)
        else:
            y = Plan._checked(self, y, self.out_shape, "y")
        ctr_istft_forward(self.handle, _ptr(spec), _ptr(bias), _ptr(y), _stream_ptr(stream))
        return y

    def describe(self) -> str:
        return ctr_istft_describe(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            ctr_istft_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_plan_cache = {}


def conv_transpose(x, w, bias=None, stride=1, padding=0, output_padding=0, negative_slope=None,
                   path=CTR_PATH_AUTO, split_k=0, groups=1, dilation=1, padding_end=None):
    """ConvTranspose1d/2d of torch CUDA tensors (float32 or bfloat16), like
    torch.nn.functional.conv_transpose{1,2}d (groups, dilation), plus separate back pads
    (``padding_end``, ONNX-style; default: ``padding``) and an optional fused LeakyReLU.
    Plans and packed weights are cached per (shapes, weight)."""
    ndim = x.dim() - 2
    key = (tuple(x.shape), tuple(w.shape), x.dtype, str(x.device), w.data_ptr(), w._version,
           _tuple(stride, ndim), _tuple(padding, ndim), _tuple(output_padding, ndim),
           negative_slope, path, split_k, groups, _tuple(dilation, ndim),
           None if padding_end is None else _tuple(padding_end, ndim))
    plan = _plan_cache.get(key)
    if plan is None:
        if len(_plan_cache) > 64:
            _plan_cache.clear()
        plan = Plan(x.shape[0], x.shape[1], w.shape[1] * groups, tuple(x.shape[2:]),
                    tuple(w.shape[2:]), stride, padding, output_padding, dtype=x.dtype,
                    negative_slope=negative_slope, path=path, split_k=split_k, device=x.device,
                    groups=groups, dilation=dilation, padding_end=padding_end)
        plan.prepack(w.contiguous())
        _plan_cache[key] = plan
    return plan.forward(x.contiguous(), None if bias is None else bias.contiguous())
