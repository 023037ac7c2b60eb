"""GPU parity of grouped and depthwise ConvTranspose against the oracle.

A layer with groups = C_in (C_out = M * C_in; M = 1 is the depthwise upsampler of
"[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to space",
DecomposeDepthwiseConvTransposePass commit) runs on the depthwise kernel; other groups run on
the gather kernel.  Checks:

* small-integer inputs, where every product and sum is exact, equal the oracle bit for bit;
* random inputs within rel_l2 1e-5 (fp32) / 1e-2 (bf16), and the depthwise kernel equal to
  the gather kernel bit for bit (both add the same taps in the same order in fp32);
* ragged rows (width not a multiple of the 8-output chunk), every padding phase of the
  compiled x strides, k = s (one tap per output), k mod s != 0, 2-D with a run-time row
  kernel, channel multipliers, no bias, LeakyReLU, empty input, and the no-allocation entry.
Every output buffer sits between NaN guard bands that must survive the call.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import transposed_convolution_gb300 as ctr  # noqa: E402
import workloads  # noqa: E402
from gpu_helpers import TOL, reference, run_plan, tdtype, to_dev  # noqa: E402

# (B, C_in, C_out, groups, in_spatial, kernel, stride, padding, output_padding)
DEPTHWISE = [
    (2, 16, 16, 16, (300,), (4,), (2,), (1,), (0,)),            # the 4/2 upsampler, ragged row
    (1, 8, 8, 8, (64,), (2,), (2,), (0,), (0,)),                # k = s: one tap per output
    (1, 8, 8, 8, (61,), (2,), (2,), (1,), (1,)),                # k = s, odd padding phase
    (2, 8, 8, 8, (97,), (3,), (2,), (1,), (1,)),                # k mod s != 0
    (1, 8, 8, 8, (50,), (8,), (4,), (2,), (0,)),                # 8/4, phase 2
    (1, 4, 4, 4, (33,), (8,), (4,), (3,), (1,)),                # 8/4, phase 3
    (1, 8, 8, 8, (40,), (16,), (8,), (4,), (0,)),               # 16/8 (codec upsampler shape)
    (1, 4, 4, 4, (37,), (16,), (8,), (5,), (3,)),               # 16/8, phase 5
    (1, 4, 4, 4, (25,), (8,), (8,), (0,), (0,)),                # k = s = 8
    (1, 6, 12, 6, (70,), (4,), (2,), (1,), (0,)),               # channel multiplier 2
    (2, 8, 8, 8, (17, 23), (4, 4), (2, 2), (1, 1), (0, 1)),     # 2-D 4x4/2 (MI-GAN filter)
    (1, 3, 3, 3, (8, 8), (2, 2), (2, 2), (0, 0), (0, 0)),       # 2-D k = s
    (1, 4, 8, 4, (7, 13), (3, 3), (2, 2), (1, 1), (1, 0)),      # 2-D 3x3/2, multiplier 2
    (1, 4, 4, 4, (6, 9), (4, 4), (4, 4), (0, 2), (0, 3)),       # 2-D k = s = 4, x phase 2
    (2, 4, 4, 4, (40, 3), (4, 4), (2, 2), (1, 1), (0, 0)),      # tall: runs of phase rows
]
GROUPED = [
    (2, 8, 12, 4, (50,), (4,), (2,), (1,), (0,)),
    (1, 6, 4, 2, (30,), (5,), (3,), (2,), (1,)),
    (1, 8, 8, 2, (9, 11), (4, 4), (2, 2), (1, 1), (0, 0)),
    (1, 8, 8, 8, (40,), (5,), (2,), (1,), (0,)),                # depthwise, no compiled kernel
    (1, 4, 4, 4, (9, 30), (5, 4), (3, 2), (2, 1), (1, 0)),      # depthwise 2-D, not square
]


def _ids(c):
    return "B%d-%dto%d-g%d-%s-k%s-s%s-p%s-op%s" % (c[0], c[1], c[2], c[3], "x".join(map(str, c[4])),
                                                   c[5], c[6], c[7], c[8])


def _inputs(rng, case, integer, with_bias=True):
    B, C_in, C_out, G, sp, k, s, p, op = case
    if integer:
        x = rng.integers(-3, 4, (B, C_in) + sp).astype(np.float32)
        w = rng.integers(-3, 4, (C_in, C_out // G) + k).astype(np.float32)
        b = rng.integers(-3, 4, (C_out,)).astype(np.float32)
    else:
        x = rng.standard_normal((B, C_in) + sp).astype(np.float32)
        w = rng.uniform(-0.5, 0.5, (C_in, C_out // G) + k).astype(np.float32)
        b = rng.standard_normal(C_out).astype(np.float32)
    if not with_bias:
        b = None
    return x, w, b


def _expect(case):
    return ctr.CTR_PATH_DEPTHWISE if case in DEPTHWISE else ctr.CTR_PATH_GATHER


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", DEPTHWISE + GROUPED, ids=_ids)
def test_integer_exact(case, dtype):
    x, w, b = _inputs(np.random.default_rng(61), case, integer=True)
    _, _, _, G, _, _, s, p, op = case
    y, desc = run_plan(x, w, b, s, p, op, dtype, groups=G, expect_path=_expect(case))
    np.testing.assert_array_equal(y, reference(x, w, b, s, p, op, dtype, groups=G), err_msg=desc)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", DEPTHWISE + GROUPED, ids=_ids)
def test_random_within_tolerance(case, dtype):
    rng = np.random.default_rng(62)
    x, w, b = _inputs(rng, case, integer=False)
    x = oracle.round_bf16(x) if dtype == "bf16" else x
    w = oracle.round_bf16(w) if dtype == "bf16" else w
    b = oracle.round_bf16(b) if dtype == "bf16" else b
    _, _, _, G, _, _, s, p, op = case
    y, desc = run_plan(x, w, b, s, p, op, dtype, slope=0.1, groups=G, expect_path=_expect(case))
    err = oracle.rel_l2(y, reference(x, w, b, s, p, op, dtype, slope=0.1, groups=G))
    assert err <= TOL[dtype], "rel_l2 %.3g %s" % (err, desc)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", DEPTHWISE, ids=_ids)
def test_depthwise_equals_gather(case, dtype):
    rng = np.random.default_rng(63)
    x, w, b = _inputs(rng, case, integer=False, with_bias=case[0] == 1)
    _, _, _, G, _, _, s, p, op = case
    y_dw, _ = run_plan(x, w, b, s, p, op, dtype, groups=G, expect_path=ctr.CTR_PATH_DEPTHWISE)
    y_g, _ = run_plan(x, w, b, s, p, op, dtype, groups=G, path=ctr.CTR_PATH_GATHER,
                      expect_path=ctr.CTR_PATH_GATHER)
    np.testing.assert_array_equal(y_dw, y_g)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_depthwise_full_size_sampled(dtype):
    """The 2-D depthwise upsampler workload the benchmark times (4 x 256 channels, 128x128 ->
    256x256), with its own inputs (bf16 values, also exact in fp32): sampled outputs against
    the oracle computed one by one, and the whole output against the gather kernel."""
    li = workloads.make_workload("depthwise_2d_bf16")[0]
    B, C, H, W = li.x.shape
    x, w, b = li.x, li.w, li.bias
    rng = np.random.default_rng(64)
    y, desc = run_plan(x, w, b, 2, 1, 0, dtype, slope=0.2, groups=C,
                       expect_path=ctr.CTR_PATH_DEPTHWISE)
    y_g, _ = run_plan(x, w, b, 2, 1, 0, dtype, slope=0.2, groups=C, path=ctr.CTR_PATH_GATHER)
    np.testing.assert_array_equal(y, y_g)
    for i in range(64):
        bb, c = int(rng.integers(B)), int(rng.integers(C))
        oy, ox = int(rng.integers(2 * H)), int(rng.integers(2 * W))
        # The output at (oy, ox) depends on input rows/cols within two of (oy + 1) / 2.
        y0, x0 = max(0, (oy + 1) // 2 - 2), max(0, (ox + 1) // 2 - 2)
        y1, x1 = min(H, y0 + 5), min(W, x0 + 5)
        sub = x[bb:bb + 1, c:c + 1, y0:y1, x0:x1]
        ref = oracle.conv_transpose(sub, w[c:c + 1], b[c:c + 1], 2, 1, 0)
        ref = oracle.leaky_relu(ref, 0.2)
        ry, rx = oy - 2 * y0, ox - 2 * x0    # the cropped input shifts the output by 2*y0
        val = ref[0, 0, ry, rx]
        val = oracle.round_bf16(val) if dtype == "bf16" else oracle.round_f32(val)
        tol = 1e-2 * (1 + abs(val)) if dtype == "bf16" else 1e-5 * (1 + abs(val))
        assert abs(y[bb, c, oy, ox] - val) <= tol, (bb, c, oy, ox, y[bb, c, oy, ox], val, desc)


def test_empty_input_and_no_bias():
    # In length 0: the output is bias (or zero) everywhere, on both kernels.
    for path in (ctr.CTR_PATH_DEPTHWISE, ctr.CTR_PATH_GATHER):
        x = np.zeros((1, 4, 0), np.float32)
        w = np.ones((4, 1, 4), np.float32)
        b = np.arange(4, dtype=np.float32)
        y, desc = run_plan(x, w, b, 2, 0, 0, "f32", groups=4, path=path, expect_path=path)
        assert y.shape == (1, 4, 2)
        np.testing.assert_array_equal(y, np.repeat(b[None, :, None], 2, axis=2), err_msg=desc)
        y, _ = run_plan(x, w, None, 2, 0, 0, "f32", groups=4, path=path)
        np.testing.assert_array_equal(y, np.zeros((1, 4, 2)))


def test_noalloc_depthwise():
    rng = np.random.default_rng(65)
    case = DEPTHWISE[0]
    x, w, b = _inputs(rng, case, integer=True)
    B, C_in, C_out, G, sp, k, s, p, op = case
    plan = ctr.Plan(B, C_in, C_out, sp, k, s, p, op, dtype=torch.float32, groups=G)
    try:
        assert plan.path == ctr.CTR_PATH_DEPTHWISE
        y = torch.full(plan.out_shape, float("nan"), device="cuda")
        xd, wd, bd = to_dev(x, "f32"), to_dev(w, "f32"), to_dev(b, "f32")   # held for the call
        st = ctr.lib.ctr_forward_noalloc(plan.handle, xd.data_ptr(), wd.data_ptr(), bd.data_ptr(),
                                         y.data_ptr(), None)
        assert st == ctr.CTR_OK
        torch.cuda.synchronize()
        np.testing.assert_array_equal(y.cpu().numpy().astype(np.float64),
                                      reference(x, w, b, s, p, op, "f32", groups=G))
    finally:
        plan.close()


def test_conv_transpose_groups_matches_torch():
    """The high-level call with groups, against torch's own grouped ConvTranspose on the GPU
    (a library routine, independent of both the kernels and the oracle)."""
    rng = np.random.default_rng(66)
    x = torch.from_numpy(rng.standard_normal((2, 32, 64)).astype(np.float32)).cuda()
    for G, cout in ((32, 32), (32, 64), (4, 16)):
        w = torch.from_numpy(rng.uniform(-0.5, 0.5, (32, cout // G, 4)).astype(np.float32)).cuda()
        b = torch.from_numpy(rng.standard_normal(cout).astype(np.float32)).cuda()
        y = ctr.conv_transpose(x, w, b, stride=2, padding=1, groups=G)
        ref = torch.nn.functional.conv_transpose1d(x.double(), w.double(), b.double(), stride=2,
                                                   padding=1, groups=G)
        assert torch.allclose(y.double(), ref, rtol=1e-5, atol=1e-5)
