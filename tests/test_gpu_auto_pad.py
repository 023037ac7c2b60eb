"""ONNX auto_pad / output_shape (ctr_plan_set_auto_pad) on the GPU, against the oracle.

"[WebGPU] optimizations for audio models" runs the ONNX ConvTranspose tests, whose operator
takes the padding as auto_pad (SAME_UPPER, SAME_LOWER, VALID) or an explicit output_shape
instead of pads.  The test resolves each case into front and back pads from the ONNX
definition on its own (total = unpadded length - target length; SAME_UPPER puts the odd
sample at the end, the others in front), runs the library plan made from the attributes on
every path, and compares it with the oracle's ConvTranspose with those pads: bit for bit on
small-integer inputs.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import transposed_convolution_gb300 as ctr  # noqa: E402
from gpu_helpers import reference, tdtype, to_dev  # noqa: E402

PATHS = {"auto": ctr.CTR_PATH_AUTO, "polyphase": ctr.CTR_PATH_POLYPHASE,
         "col2im": ctr.CTR_PATH_COL2IM, "gather": ctr.CTR_PATH_GATHER}


def onnx_pads(L, k, s, d, op, mode, out_len):
    """(front, back, output length) of one dimension from the ONNX attributes."""
    full = (L - 1) * s + (k - 1) * d + 1 + op
    if out_len is not None:
        total = full - out_len
    elif mode in ("SAME_UPPER", "SAME_LOWER"):
        total = full - L * s
    else:
        total = 0
    half = total // 2
    if mode == "SAME_UPPER":
        front, back = half, total - half
    else:
        front, back = total - half, half
    return front, back, full - total


MODES = {"SAME_UPPER": ctr.CTR_AUTO_PAD_SAME_UPPER, "SAME_LOWER": ctr.CTR_AUTO_PAD_SAME_LOWER,
         "VALID": ctr.CTR_AUTO_PAD_VALID, "NOTSET": ctr.CTR_AUTO_PAD_NOTSET}

CASES = [  # (spatial L, k, s, d, op, mode, output_shape)
    ((37,), (4,), (2,), (1,), (0,), "SAME_UPPER", None),
    ((37,), (3,), (2,), (1,), (0,), "SAME_UPPER", None),     # odd total: extra at the end
    ((37,), (3,), (2,), (1,), (0,), "SAME_LOWER", None),     # odd total: extra in front
    ((30,), (16,), (8,), (1,), (0,), "SAME_LOWER", None),
    ((21,), (5,), (3,), (2,), (1,), "VALID", None),
    ((40,), (4,), (2,), (1,), (1,), "NOTSET", (77,)),        # explicit output_shape
    ((9, 13), (4, 3), (2, 2), (1, 2), (0, 1), "SAME_UPPER", None),
    ((9, 13), (4, 4), (2, 2), (1, 1), (0, 0), "NOTSET", (17, 25)),
    ((6, 7), (3, 5), (3, 2), (1, 1), (2, 1), "SAME_LOWER", None),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_auto_pad_against_oracle(dtype, path):
    rng = np.random.default_rng(503)
    mag = 2 if dtype == "f32" else 1
    ran = 0
    for n, (L, k, s, d, op, mode, out_shape) in enumerate(CASES):
        ci, co = (40, 24) if n % 2 == 0 else (20, 33)
        x = rng.integers(-mag, mag + 1, (2, ci) + L).astype(np.float32)
        w = rng.integers(-mag, mag + 1, (ci, co) + k).astype(np.float32)
        b = rng.integers(-mag, mag + 1, (co,)).astype(np.float32)
        res = [onnx_pads(L[i], k[i], s[i], d[i], op[i], mode,
                         None if out_shape is None else out_shape[i]) for i in range(len(L))]
        front = tuple(r[0] for r in res)
        back = tuple(r[1] for r in res)
        expect_out = tuple(r[2] for r in res)
        try:
            plan = ctr.Plan(2, ci, co, L, k, s, 0, op, dtype=tdtype(dtype), dilation=d,
                            auto_pad=MODES[mode], output_shape=out_shape, path=PATHS[path])
        except ctr.CtrError as ex:
            # a forced path the geometry cannot take (polyphase with dilation, say)
            assert ex.status == ctr.CTR_ERR_UNSUPPORTED and path != "auto", (ex, path)
            continue
        try:
            assert tuple(plan.out_spatial) == expect_out, (plan.describe(), expect_out)
            plan.prepack(to_dev(w, dtype))
            y = plan.forward(to_dev(x, dtype), to_dev(b, dtype))
            plan.check()
            got = y.float().cpu().numpy().astype(np.float64)
            desc = plan.describe()
        finally:
            plan.close()
        ref = reference(x, w, b, s, front, op, dtype, dilation=d, padding_end=back)
        np.testing.assert_array_equal(got, ref, err_msg="%s %s %s" % (mode, (L, k, s, d, op), desc))
        ran += 1
    assert ran >= 3


def test_onnx_pads_restatement():
    """The test's own resolution against torch's ConvTranspose with an explicit
    output_padding-free padding: SAME with an even total is torch padding total/2."""
    torch_f = torch.nn.functional
    x = torch.randn(1, 3, 11, dtype=torch.float64)
    w = torch.randn(3, 2, 4, dtype=torch.float64)
    front, back, out = onnx_pads(11, 4, 2, 1, 0, "SAME_UPPER", None)
    assert front == back == 1 and out == 22
    ref = torch_f.conv_transpose1d(x, w, stride=2, padding=1).numpy()
    mine = oracle.conv_transpose(x.numpy(), w.numpy(), None, 2, front, 0, padding_end=back)
    np.testing.assert_allclose(mine, ref, rtol=0, atol=1e-12)
