"""The paired output stage for stride-2 columns at odd offsets, against the oracle.

With the unpadded phase origin a position's two outputs of a row start at the odd column
2 qx - px when px is odd ("[XNNPACK] Lower dense transposed convs as one polyphase conv +
depth to space", Summary: the padding is sliced off at the store), so the library stores
each lane's second output together with its right neighbour's first, and the outputs no
pair covers (row starts, row ends, the last lane of a warp, positions past the output)
alone.  Small-integer inputs make every product and sum exact, so the result must equal
the oracle bit for bit: 1-D and 2-D, px = 1 and 3, several position tiles with a ragged
tail, channel counts that leave a partial chunk, batches, LeakyReLU, and the odd output
widths for which the library keeps the per-element stage.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transposed_convolution_gb300 as ctr  # noqa: E402
from gpu_helpers import reference, run_plan  # noqa: E402

CASES_1D = [  # (B, C_in, C_out, L, k, p, op): stride 2
    (1, 64, 32, 300, 4, 1, 0),    # even output width: pairs
    (2, 40, 19, 257, 4, 1, 0),    # ragged channels, batch 2
    (1, 32, 8, 131, 8, 3, 0),     # px = 3: the first pair column of a row is past x = 0
    (1, 48, 16, 100, 6, 1, 0),
    (1, 32, 16, 90, 4, 1, 1),     # odd output width: per-element stage
]
CASES_2D = [  # (B, C_in, C_out, H, W, k, p, op)
    (1, 32, 16, 20, 70, 4, 1, 0),   # row pitch 72: warps span rows and the row-end positions
    (2, 24, 9, 13, 33, 4, 1, 0),
    (1, 16, 8, 9, 40, 8, 3, 0),
    (1, 16, 8, 10, 21, 4, 1, (0, 1)),   # odd output width
]


def _ints(rng, shape, mag):
    return rng.integers(-mag, mag + 1, shape).astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_pairs_1d_bit_exact(dtype):
    rng = np.random.default_rng(401)
    mag = 2 if dtype == "f32" else 1
    for n, (B, ci, co, L, k, p, op) in enumerate(CASES_1D):
        x = _ints(rng, (B, ci, L), mag)
        w = _ints(rng, (ci, co, k), mag)
        b = _ints(rng, (co,), mag)
        slope = 0.25 if n % 2 == 0 else None
        y, desc = run_plan(x, w, b, 2, p, op, dtype, slope=slope, path=ctr.CTR_PATH_POLYPHASE,
                           phase_origin=ctr.CTR_PHASE_UNPADDED)
        wout = (L - 1) * 2 - 2 * p + k + op
        assert ("pairs" in desc) == (wout % 2 == 0), desc
        ref = reference(x, w, b, 2, p, op, dtype, slope=slope)
        np.testing.assert_array_equal(y, ref, err_msg=desc)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_pairs_2d_bit_exact(dtype):
    rng = np.random.default_rng(402)
    mag = 2 if dtype == "f32" else 1
    for n, (B, ci, co, H, W, k, p, op) in enumerate(CASES_2D):
        op2 = op if isinstance(op, tuple) else (op, op)
        x = _ints(rng, (B, ci, H, W), mag)
        w = _ints(rng, (ci, co, k, k), mag)
        b = _ints(rng, (co,), mag)
        slope = 0.5 if n % 2 == 1 else None
        y, desc = run_plan(x, w, b, (2, 2), (p, p), op2, dtype, slope=slope,
                           path=ctr.CTR_PATH_POLYPHASE, phase_origin=ctr.CTR_PHASE_UNPADDED)
        wout = (W - 1) * 2 - 2 * p + k + op2[1]
        assert ("pairs" in desc) == (wout % 2 == 0), desc
        ref = reference(x, w, b, (2, 2), (p, p), op2, dtype, slope=slope)
        np.testing.assert_array_equal(y, ref, err_msg=desc)


def test_decoder_shape_uses_pairs():
    """The 2-D decoder layer (128 -> 64 channels, 4x4 kernel, stride 2, padding 1) keeps the
    unpadded origin (output phases would add taps) and takes the paired stores."""
    plan = ctr.Plan(1, 128, 64, (128, 128), (4, 4), (2, 2), (1, 1), 0, dtype=torch.float32)
    try:
        desc = plan.describe()
        assert "out-phases" not in desc and "pairs" in desc, desc
    finally:
        plan.close()
