"""Channels-last (NHWC) x and y (ctr_plan_set_layout) against the oracle.

The oracle computes in NCHW; the tests transpose x to channels last before the call and y
back after it (a relabelling of memory, none of the method's arithmetic).  Small-integer
inputs make every sum exact, so each path must match bit for bit: the polyphase path with
channel counts that keep 16-byte rows (the vectorised channels-last output stage) and ones
that do not (the element-wise stage), split-K (the reduce writes NHWC), col2im, gather,
grouped plans (gather), an empty input, and a chain from an NHWC input to an NHWC output.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import transposed_convolution_gb300 as ctr  # noqa: E402
from gpu_helpers import reference, run_plan, tdtype, to_dev  # noqa: E402

PATHS = {"gather": ctr.CTR_PATH_GATHER, "polyphase": ctr.CTR_PATH_POLYPHASE,
         "col2im": ctr.CTR_PATH_COL2IM}
CASES = [  # (x shape NCHW, C_out, kernel, stride, padding, output_padding)
    ((2, 64, 40), 32, 4, 2, 1, 0),                   # C_out rows of 16-byte vectors
    ((1, 48, 37), 33, 16, 8, 4, 3),                  # C_out = 33: element-wise stage
    ((1, 20, 9, 11), 24, (4, 4), (2, 2), (1, 1), (0, 1)),
    ((1, 40, 6, 7), 17, (3, 3), (2, 2), (1, 0), (1, 1)),
    ((2, 64, 30), 64, 3, 2, 1, 1),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_nhwc_integer_bit_exact(path, dtype):
    rng = np.random.default_rng(101)
    for n, (xs, co, k, s, p, op) in enumerate(CASES):
        nd = len(xs) - 2
        k = k if isinstance(k, tuple) else (k,)
        x = rng.integers(-2, 3, xs).astype(np.float32)
        w = rng.integers(-2, 3, (xs[1], co) + k).astype(np.float32)
        b = rng.integers(-2, 3, co).astype(np.float32)
        slope = 0.25 if n % 2 else None
        y, desc = run_plan(x, w, b, s, p, op, dtype, slope=slope, path=PATHS[path], layout="nhwc")
        assert "nhwc" in desc, desc
        np.testing.assert_array_equal(y, reference(x, w, b, s, p, op, dtype, slope=slope),
                                      err_msg="%s %s" % (xs, desc))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nhwc_split_k_and_tiles_bit_exact(dtype):
    rng = np.random.default_rng(103)
    for (B, ci, co, L, k, s, p, op) in [(2, 150, 40, 300, 8, 4, 2, 0), (1, 64, 33, 257, 16, 8, 4, 3)]:
        x = rng.integers(-1, 2, (B, ci, L)).astype(np.float32)
        w = rng.integers(-1, 2, (ci, co, k)).astype(np.float32)
        b = rng.integers(-1, 2, co).astype(np.float32)
        for split_k in (1, 3):
            y, desc = run_plan(x, w, b, s, p, op, dtype, path=ctr.CTR_PATH_POLYPHASE,
                               split_k=split_k, layout="nhwc")
            np.testing.assert_array_equal(y, reference(x, w, b, s, p, op, dtype), err_msg=desc)


def test_nhwc_grouped_and_empty():
    rng = np.random.default_rng(105)
    x = rng.integers(-2, 3, (1, 16, 9, 12)).astype(np.float32)
    w = rng.integers(-2, 3, (16, 1, 4, 4)).astype(np.float32)
    b = rng.integers(-2, 3, 16).astype(np.float32)
    y, desc = run_plan(x, w, b, (2, 2), (1, 1), 0, "bf16", groups=16, layout="nhwc",
                       expect_path=ctr.CTR_PATH_GATHER)
    np.testing.assert_array_equal(y, reference(x, w, b, (2, 2), (1, 1), 0, "bf16", groups=16),
                                  err_msg=desc)
    x = np.zeros((2, 32, 0), np.float32)
    w = rng.integers(-2, 3, (32, 24, 3)).astype(np.float32)
    b = rng.integers(-2, 3, 24).astype(np.float32)
    y, desc = run_plan(x, w, b, 2, 0, 1, "f32", path=ctr.CTR_PATH_COL2IM, layout="nhwc",
                       check_guards=True)
    np.testing.assert_array_equal(y, reference(x, w, b, 2, 0, 1, "f32"), err_msg=desc)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nhwc_chain_bit_exact(dtype):
    """The first plan stages an NHWC input, the chained second one writes an NHWC output."""
    rng = np.random.default_rng(107)
    p1 = ctr.Plan(1, 64, 64, (80,), (4,), 2, 1, 0, dtype=tdtype(dtype), negative_slope=0.25,
                  layout="nhwc")
    p2 = ctr.Plan(1, 64, 32, p1.out_spatial, (4,), 2, 1, 0, dtype=tdtype(dtype), layout="nhwc")
    try:
        p1.chain(p2)
        x = rng.integers(-1, 2, (1, 64, 80)).astype(np.float32)
        w1 = rng.integers(-1, 2, (64, 64, 4)).astype(np.float32)
        w2 = rng.integers(-1, 2, (64, 32, 4)).astype(np.float32)
        b1 = rng.integers(-1, 2, 64).astype(np.float32)
        b2 = rng.integers(-1, 2, 32).astype(np.float32)
        p1.prepack(to_dev(w1, dtype))
        p2.prepack(to_dev(w2, dtype))
        y = torch.full(p2.out_shape, float("nan"), dtype=tdtype(dtype), device="cuda")
        p1.forward(to_dev(np.ascontiguousarray(x.transpose(0, 2, 1)), dtype), to_dev(b1, dtype))
        p2.forward(None, to_dev(b2, dtype), y=y)
        p1.check()
        p2.check()
        got = y.float().cpu().numpy().transpose(0, 2, 1)
        h = reference(x, w1, b1, 2, 1, 0, dtype, slope=0.25)
        np.testing.assert_array_equal(got, reference(h, w2, b2, 2, 1, 0, dtype),
                                      err_msg="%s | %s" % (p1.describe(), p2.describe()))
    finally:
        p1.close()
        p2.close()
