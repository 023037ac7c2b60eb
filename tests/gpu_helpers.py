"""Helpers of the GPU tests: run the library through the C ABI on torch CUDA tensors, with
NaN guard bands around the output, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import transposed_convolution_gb300 as ctr

GUARD = 64  # elements of NaN before and after y (keeps 16-byte alignment for fp32 and bf16)


def tdtype(dtype: str):
    return {"bf16": torch.bfloat16, "f16": torch.float16}.get(dtype, torch.float32)


def to_dev(a, dtype: str):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float32))).to(
        "cuda").to(tdtype(dtype)).contiguous()


def run_plan(x, w, bias, stride, padding, output_padding, dtype="f32", slope=None,
             path=ctr.CTR_PATH_AUTO, split_k=0, check_guards=True, expect_path=None, block_n=0,
             groups=1, dilation=1, padding_end=None, phase_origin=ctr.CTR_PHASE_AUTO,
             layout="nchw"):
    """Run one ConvTranspose through the library.  x, w, bias: numpy arrays holding values of
    the I/O dtype, x in NCHW order (transposed to channels last on the way in, and y back,
    when layout is "nhwc").  Returns (y as float64 numpy in NCHW order, plan description)."""
    x = np.asarray(x)
    ndim = x.ndim - 2
    plan = ctr.Plan(x.shape[0], x.shape[1], w.shape[1] * groups, tuple(x.shape[2:]),
                    tuple(w.shape[2:]), stride, padding, output_padding, dtype=tdtype(dtype),
                    negative_slope=slope, path=path, split_k=split_k, block_n=block_n,
                    groups=groups, dilation=dilation, padding_end=padding_end,
                    phase_origin=phase_origin, layout=layout)
    to_last = (0,) + tuple(range(2, 2 + ndim)) + (1,)
    to_first = (0, 1 + ndim) + tuple(range(1, 1 + ndim))
    if layout == "nhwc":
        x = np.ascontiguousarray(np.transpose(x, to_last))
    try:
        if expect_path is not None:
            assert plan.path == expect_path, plan.describe()
        plan.prepack(to_dev(w, dtype))
        n = int(np.prod(plan.out_shape))
        buf = torch.full((n + 2 * GUARD,), float("nan"), dtype=tdtype(dtype), device="cuda")
        y = buf[GUARD:GUARD + n].view(plan.out_shape)
        plan.forward(to_dev(x, dtype), to_dev(bias, dtype), y=y)
        plan.check()
        if check_guards:
            g = torch.cat([buf[:GUARD], buf[GUARD + n:]]).float().cpu().numpy()
            assert np.all(np.isnan(g)), "library wrote outside y"
        out = y.float().cpu().numpy().astype(np.float64)
        if layout == "nhwc":
            out = np.ascontiguousarray(np.transpose(out, to_first))
        return out, plan.describe()
    finally:
        plan.close()


def reference(x, w, bias, stride, padding, output_padding, dtype="f32", slope=None, groups=1,
              dilation=1, padding_end=None):
    """Oracle result rounded like the library's output: double sum + bias, then LeakyReLU,
    then one rounding to the I/O dtype."""
    y = oracle.conv_transpose(x, w, bias, stride, padding, output_padding, groups=groups,
                              dilation=dilation, padding_end=padding_end)
    if slope is not None:
        y = oracle.leaky_relu(y, slope)
    if dtype == "bf16":
        return oracle.round_bf16(y)
    if dtype == "f16":
        return oracle.round_f16(y)
    return oracle.round_f32(y)


# rel_l2 bounds: fp32 I/O 1e-5 and bf16 I/O 1e-2 (the stated targets); fp16 I/O 1e-3, from
# one rounding of each output to 11 significant bits (unit roundoff 2**-11 ~ 4.9e-4) on fp32
# sums whose own error is far smaller.
TOL = {"f32": 1e-5, "bf16": 1e-2, "f16": 1e-3}
