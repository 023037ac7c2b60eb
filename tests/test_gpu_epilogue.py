"""The GEMM's fused output stage (bias, LeakyReLU, phase interleave, padding slice) against the
oracle, bit for bit, for every whole-phase-set variant (1-D with 1, 2, 4 and 8 phases, 2-D
2x2 and 4x4) and both I/O types, on shapes that hit its edges: odd padding (runs that
start left of the output and unaligned stores), ragged row ends, chunks whose channels run
past C_out, warps whose positions wrap to the next row or batch item, LeakyReLU.
"""
import numpy as np
import pytest

from gpu_helpers import reference, run_plan

import transposed_convolution_gb300 as ctr

# (x shape, w shape, stride, padding, output_padding, dtype, slope); slopes are powers of
# two so that the oracle's double product and the kernel's fp32 product round alike.
CASES = [
    ((2, 40, 100), (40, 37, 4), 2, 1, 0, "bf16", 0.125),        # S2, 16 channels per chunk
    ((1, 48, 96), (48, 70, 3), 1, 1, 0, "bf16", None),          # S1 (stride 1)
    ((2, 24, 64), (24, 33, 8), 4, 2, 0, "bf16", None),          # S4
    ((1, 32, 50), (32, 20, 16), 8, 3, 2, "f32", 0.25),          # S8, fp32, odd padding
    ((2, 40, 30, 40), (40, 20, 4, 4), (2, 2), (1, 1), (0, 0), "f32", None),    # S2x2, wraps
    ((1, 24, 12, 10), (24, 9, 8, 8), (4, 4), (2, 2), (0, 0), "bf16", 0.125),  # S4x4
]


def _ints(rng, shape, mag=2):
    return rng.integers(-mag, mag + 1, shape).astype(np.float32)


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-%dd-k%s" % (c[5], len(c[0]) - 2, c[1][2:]))
def test_output_stage_bit_exact(case):
    xs, ws, s, p, op, dtype, slope = case
    rng = np.random.default_rng(23)
    mag = 1 if dtype == "bf16" else 2
    x, w, b = _ints(rng, xs, mag), _ints(rng, ws, mag), _ints(rng, (ws[1],))
    y, desc = run_plan(x, w, b, s, p, op, dtype, slope=slope, path=ctr.CTR_PATH_POLYPHASE)
    np.testing.assert_array_equal(y, reference(x, w, b, s, p, op, dtype, slope=slope), err_msg=desc)
