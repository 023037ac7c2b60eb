"""The polyphase path with each phase origin (ctr_plan_set_phase_origin), against the oracle.

CTR_PHASE_UNPADDED computes the phases of the unpadded output and slices the padding off
at the store ("[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to
space", Summary); CTR_PHASE_OUTPUT re-indexes the phases by the output itself, folding
p mod s into the packed taps (one more tap when it is not zero), so that every run of s
phases starts at an aligned output offset.  Both add the same products, so on small-integer
inputs (every product and partial sum exact) both must equal the oracle bit for bit: over
the 1-D and 2-D geometry grids, every tile width, split-K (whose reduce runs the same output
mapping), fused LeakyReLU and chained plans.  Random inputs stay within the tolerances.
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

ORIGINS = {"unpadded": ctr.CTR_PHASE_UNPADDED, "output": ctr.CTR_PHASE_OUTPUT}

GRID_1D = [  # (L, k, s, p, op): p mod s = 0 and != 0, op above and below p, m = 1..4
    (1, 4, 2, 1, 0), (5, 4, 2, 1, 1), (37, 16, 8, 4, 0), (37, 16, 8, 4, 3), (9, 3, 2, 1, 1),
    (7, 7, 3, 2, 2), (11, 8, 4, 0, 0), (13, 6, 3, 0, 2), (4, 12, 4, 6, 1), (20, 2, 2, 0, 0),
    (3, 10, 5, 2, 4), (12, 8, 2, 3, 1), (9, 6, 2, 5, 0), (10, 4, 2, 2, 0), (6, 9, 3, 7, 2),
]
GRID_2D = [  # (H, W, ky, kx, sy, sx, py, px, opy, opx)
    (5, 7, 4, 4, 2, 2, 1, 1, 0, 0), (6, 3, 3, 3, 2, 2, 1, 0, 1, 1), (4, 5, 4, 6, 2, 3, 1, 2, 1, 0),
    (9, 2, 6, 2, 3, 1, 2, 0, 2, 0), (7, 6, 4, 4, 2, 2, 3, 2, 1, 0),
]


def _int_inputs(rng, shape_x, shape_w, C_out, mag, with_bias=True):
    x = rng.integers(-mag, mag + 1, shape_x).astype(np.float32)
    w = rng.integers(-mag, mag + 1, shape_w).astype(np.float32)
    b = rng.integers(-mag, mag + 1, (C_out,)).astype(np.float32) if with_bias else None
    return x, w, b


@pytest.mark.parametrize("origin", sorted(ORIGINS))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_integer_grid_bit_exact(dtype, origin):
    rng = np.random.default_rng(21)
    mag = 2 if dtype == "f32" else 1
    n = 0
    for (L, k, s, p, op) in GRID_1D:
        for (ci, co) in [(3, 32), (40, 17)]:
            n += 1
            x, w, b = _int_inputs(rng, (2, ci, L), (ci, co, k), co, mag, with_bias=n % 2 == 0)
            slope = 0.25 if n % 3 == 0 else None
            y, desc = run_plan(x, w, b, s, p, op, dtype, path=ctr.CTR_PATH_POLYPHASE,
                               phase_origin=ORIGINS[origin], slope=slope)
            assert ("out-phases" in desc) == (origin == "output"), desc
            ref = reference(x, w, b, s, p, op, dtype, slope=slope)
            np.testing.assert_array_equal(y, ref, err_msg="%s %s" % ((L, k, s, p, op, ci, co), desc))
    for (H, W, ky, kx, sy, sx, py, px, opy, opx) in GRID_2D:
        x, w, b = _int_inputs(rng, (1, 20, H, W), (20, 9, ky, kx), 9, mag)
        y, desc = run_plan(x, w, b, (sy, sx), (py, px), (opy, opx), dtype,
                           path=ctr.CTR_PATH_POLYPHASE, phase_origin=ORIGINS[origin])
        ref = reference(x, w, b, (sy, sx), (py, px), (opy, opx), dtype)
        np.testing.assert_array_equal(y, ref, err_msg=desc)


@pytest.mark.parametrize("block_n", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_output_phases_tiles_and_split_k_bit_exact(dtype, block_n):
    """Output phases at every tile width, several position tiles with a ragged tail, and
    split-K (the reduce applies the same output mapping)."""
    rng = np.random.default_rng(31 + block_n)
    mag = 2 if dtype == "f32" else 1
    cases = [(2, 100, 70, 300, 4, 2, 1, 0), (1, 96, 33, 131, 16, 8, 4, 3),
             (1, 64, 40, 257, 4, 2, 1, 1)]
    for (B, ci, co, L, k, s, p, op) in cases:
        x, w, b = _int_inputs(rng, (B, ci, L), (ci, co, k), co, mag)
        ref = reference(x, w, b, s, p, op, dtype)
        for split_k in (1, 3):
            y, desc = run_plan(x, w, b, s, p, op, dtype, path=ctr.CTR_PATH_POLYPHASE,
                               split_k=split_k, block_n=block_n,
                               phase_origin=ctr.CTR_PHASE_OUTPUT)
            assert "BN %d," % block_n in desc and "out-phases" in desc, desc
            np.testing.assert_array_equal(y, ref, err_msg=desc)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_output_phases_random_within_tolerance(dtype):
    rng = np.random.default_rng(41)
    cases = [((2, 96, 130), (96, 48, 8), 4, 2, 1), ((1, 128, 600), (128, 64, 4), 2, 1, 0),
             ((1, 64, 30, 20), (64, 24, 4, 4), (2, 2), (1, 1), (1, 0))]
    for (xs, ws, s, p, op) in cases:
        x = workloads._cast(rng.standard_normal(xs), dtype)
        w = workloads._cast(rng.uniform(-0.1, 0.1, ws), dtype)
        b = workloads._cast(rng.normal(0, 0.1, ws[1]), dtype)
        y, desc = run_plan(x, w, b, s, p, op, dtype, path=ctr.CTR_PATH_POLYPHASE,
                           phase_origin=ctr.CTR_PHASE_OUTPUT)
        err = oracle.rel_l2(y, reference(x, w, b, s, p, op, dtype))
        assert err <= TOL[dtype], "rel_l2 %.3g %s" % (err, desc)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chain_into_output_phase_plan_bit_exact(dtype):
    """A chained producer writes the next plan's staged input at that plan's front halo,
    which the output phases change; producer and consumer each in either origin."""
    rng = np.random.default_rng(51)
    C0, C1, C2, L = 32, 32, 32, 40
    for o1 in ORIGINS.values():
        for o2 in ORIGINS.values():
            p1 = ctr.Plan(1, C0, C1, (L,), (4,), 2, 1, 0, dtype=tdtype(dtype),
                          negative_slope=0.25, phase_origin=o1)
            p2 = ctr.Plan(1, C1, C2, p1.out_spatial, (4,), 2, 1, 0, dtype=tdtype(dtype),
                          phase_origin=o2)
            try:
                p1.chain(p2)
                x, w1, b1 = _int_inputs(rng, (1, C0, L), (C0, C1, 4), C1, 2)
                _, w2, b2 = _int_inputs(rng, (1, 1, 1), (C1, C2, 4), C2, 2)
                p1.prepack(to_dev(w1, dtype))
                p2.prepack(to_dev(w2, dtype))
                y = torch.full(p2.out_shape, float("nan"), dtype=tdtype(dtype), device="cuda")
                p1.forward(to_dev(x, dtype), to_dev(b1, dtype))
                p2.forward(None, to_dev(b2, dtype), y=y)
                p1.check()
                p2.check()
                h = reference(x, w1, b1, 2, 1, 0, dtype, slope=0.25)
                ref = reference(h, w2, b2, 2, 1, 0, dtype)
                np.testing.assert_array_equal(y.float().cpu().numpy(), ref,
                                              err_msg="%s | %s" % (p1.describe(), p2.describe()))
            finally:
                p1.close()
                p2.close()
