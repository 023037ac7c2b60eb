"""GPU parity of dilated ConvTranspose and of separate front and back pads against the oracle.

Dilation spaces the taps: tap t of input i lands at o = i*s - p_front + t*d ("[ExecuTorch]
[WebGPU] Add optimized conv2d op", Implementation: the gather condition with dH).  Front and
back pads are the ONNX ConvTranspose `pads`, which "[WebGPU] optimizations for audio models"
tests together with dilations and output_padding; the output is the padding slice of the
unpadded result.  Checks, every output between NaN guard bands:

* small-integer inputs, where every product and sum is exact, equal the oracle bit for bit
  on every path a plan takes (col2im, gather, forced polyphase over the zero-inserted
  kernel, depthwise, and the automatic polyphase path under separate pads);
* random inputs within rel_l2 1e-5 (fp32) / 1e-2 (bf16);
* the paths agree with one another bit for bit on integer inputs, and a dilation or pads
  equal to the defaults give the undilated symmetric plan's output bit for bit.
"""
import zlib

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import transposed_convolution_gb300 as ctr  # noqa: E402
from gpu_helpers import TOL, reference, run_plan  # noqa: E402

P_AUTO, P_POLY, P_COL, P_GATHER, P_DW = (ctr.CTR_PATH_AUTO, ctr.CTR_PATH_POLYPHASE,
                                         ctr.CTR_PATH_COL2IM, ctr.CTR_PATH_GATHER,
                                         ctr.CTR_PATH_DEPTHWISE)

# (name, B, C_in, C_out, groups, in, k, s, dilation, pad_front, pad_back, op, dtype,
#  forced path, expected path)
CASES = [
    ("col2im_1d", 2, 32, 48, 1, (70,), (3,), (2,), (2,), (1,), (1,), (1,), "f32", P_AUTO, P_COL),
    ("col2im_2d", 1, 32, 24, 1, (13, 17), (3, 3), (2, 2), (2, 3), (1, 2), (2, 0), (1, 0), "bf16",
     P_AUTO, P_COL),
    ("col2im_d4_s3", 1, 24, 32, 1, (41,), (5,), (3,), (4,), (3,), (0,), (2,), "f32", P_AUTO, P_COL),
    ("gather_1d", 1, 4, 3, 1, (33,), (3,), (3,), (2,), (2,), (0,), (1,), "f32", P_AUTO, P_GATHER),
    ("gather_2d", 2, 3, 5, 1, (9, 7), (3, 2), (2, 3), (2, 3), (1, 0), (0, 2), (1, 2), "bf16",
     P_AUTO, P_GATHER),
    ("gather_grouped", 1, 8, 8, 2, (20,), (3,), (2,), (2,), (1,), (2,), (1,), "f32", P_AUTO,
     P_GATHER),
    ("gather_depthwise_dilated", 1, 16, 16, 16, (40,), (4,), (2,), (2,), (1,), (1,), (0,), "bf16",
     P_AUTO, P_GATHER),
    ("polyphase_forced_1d", 1, 32, 32, 1, (60,), (2,), (2,), (3,), (1,), (1,), (1,), "f32",
     P_POLY, P_POLY),
    ("polyphase_forced_2d", 1, 16, 32, 1, (10, 12), (2, 2), (2, 2), (2, 2), (0, 1), (1, 0),
     (0, 1), "bf16", P_POLY, P_POLY),
    ("polyphase_pads_1d", 2, 64, 32, 1, (100,), (4,), (2,), (1,), (2,), (0,), (1,), "f32",
     P_AUTO, P_POLY),
    ("polyphase_pads_2d", 1, 32, 16, 1, (20, 24), (4, 4), (2, 2), (1, 1), (0, 2), (2, 1), (1, 0),
     "f32", P_AUTO, P_POLY),
    ("polyphase_pads_bf16", 1, 128, 64, 1, (300,), (4,), (2,), (1,), (1,), (2,), (0,), "bf16",
     P_AUTO, P_POLY),
    ("polyphase_pads_s8", 1, 64, 32, 1, (50,), (16,), (8,), (1,), (7,), (0,), (3,), "bf16",
     P_AUTO, P_POLY),
    ("col2im_pads", 1, 32, 32, 1, (45,), (3,), (2,), (1,), (2,), (0,), (1,), "f32", P_AUTO, P_COL),
    ("depthwise_pads_1d", 1, 16, 16, 16, (40,), (4,), (2,), (1,), (0,), (2,), (0,), "bf16",
     P_AUTO, P_DW),
    ("depthwise_pads_2d", 2, 8, 8, 8, (17, 23), (4, 4), (2, 2), (1, 1), (2, 0), (0, 1), (0, 1),
     "f32", P_AUTO, P_DW),
]


def _inputs(rng, case, integer):
    _, B, C_in, C_out, G, sp, k, *_rest = case
    if integer:
        x = rng.integers(-3, 4, (B, C_in) + sp).astype(np.float32)
        w = rng.integers(-3, 4, (C_in, C_out // G) + k).astype(np.float32)
        b = rng.integers(-3, 4, (C_out,)).astype(np.float32)
    else:
        x = rng.standard_normal((B, C_in) + sp).astype(np.float32)
        w = rng.uniform(-0.5, 0.5, (C_in, C_out // G) + k).astype(np.float32)
        b = rng.standard_normal(C_out).astype(np.float32)
    return x, w, b


def _run(case, x, w, b, path=None):
    _, B, C_in, C_out, G, sp, k, s, d, pb, pe, op, dtype, forced, expect = case
    return run_plan(x, w, b, s, pb, op, dtype=dtype, groups=G, dilation=d, padding_end=pe,
                    path=forced if path is None else path,
                    expect_path=expect if path is None else path)


def _ref(case, x, w, b):
    _, B, C_in, C_out, G, sp, k, s, d, pb, pe, op, dtype, *_ = case
    return reference(x, w, b, s, pb, op, dtype=dtype, groups=G, dilation=d, padding_end=pe)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_integer_exact(case):
    rng = np.random.default_rng(zlib.crc32(case[0].encode()))
    x, w, b = _inputs(rng, case, integer=True)
    y, desc = _run(case, x, w, b)
    ref = _ref(case, x, w, b)
    assert y.shape == ref.shape, (y.shape, ref.shape, desc)
    np.testing.assert_array_equal(y, ref, err_msg=desc)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_random_within_tolerance(case):
    rng = np.random.default_rng(1 + zlib.crc32(case[0].encode()))
    x, w, b = _inputs(rng, case, integer=False)
    dtype = case[12]
    if dtype == "bf16":   # inputs hold bf16 values; the oracle takes the same values
        x, w, b = (oracle.round_bf16(a).astype(np.float32) for a in (x, w, b))
    y, desc = _run(case, x, w, b)
    err = oracle.rel_l2(y, _ref(case, x, w, b))
    assert err <= TOL[dtype], (err, desc)


@pytest.mark.parametrize("name", ["col2im_1d", "polyphase_forced_1d", "col2im_2d",
                                  "polyphase_pads_1d", "col2im_pads"])
def test_paths_agree(name):
    """Every path the geometry allows gives the same bits on integer inputs."""
    case = next(c for c in CASES if c[0] == name)
    rng = np.random.default_rng(7)
    x, w, b = _inputs(rng, case, integer=True)
    outs = [_run(case, x, w, b, path=p)[0] for p in (P_POLY, P_COL, P_GATHER)]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_default_dilation_and_pads_match_plain_plan():
    """dilation 1 and back pads equal to the front pads are the plain plan, bit for bit."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((1, 64, 80)).astype(np.float32)
    w = rng.uniform(-0.1, 0.1, (64, 32, 4)).astype(np.float32)
    b = rng.standard_normal(32).astype(np.float32)
    plain, _ = run_plan(x, w, b, (2,), (1,), (0,))
    # A plan that was dilated and padded asymmetrically, then set back to the defaults.
    plan = ctr.Plan(1, 64, 32, (80,), (4,), 2, 1, 0, dilation=2, padding_end=(3,))
    try:
        ctr.ctr_plan_set_dilation(plan.handle, [1])
        ctr.ctr_plan_set_pads(plan.handle, [1], [1])
        assert ctr.ctr_plan_output_shape(plan.handle, 1) == plain.shape[2:]
    finally:
        plan.close()
    same, _ = run_plan(x, w, b, (2,), (1,), (0,), dilation=(1,), padding_end=(1,))
    np.testing.assert_array_equal(same, plain)
