"""fp16 I/O (CTR_F16) against the oracle.

fp16 operands on the tensor cores (kind::f16 with the fp16 format), fp32 accumulation and
intermediates, one rounding of each output to fp16 ("[WebGPU] optimizations for audio
models", review commits: for float16 the packed weight and the K-padded input stay in the
I/O type while sums and column buffers are f32; and the float16 regression of cancelling
ConvTranspose taps).  The oracle rounds its double result once to fp16.

* small-integer inputs: every product and partial sum is exact, so every path equals the
  oracle bit for bit, over the 1-D and 2-D grids, split-K, both phase origins and fused
  LeakyReLU;
* random inputs within rel_l2 <= 1e-3 (one fp16 rounding: unit roundoff 2**-11);
* cancelling taps: pairs of large taps that cancel exactly leave the small ones intact;
* a chained pair, and grouped fp16 plans (the gather kernel; the depthwise kernel is
  compiled for fp32 and bf16 only).
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

PATHS = {"gather": ctr.CTR_PATH_GATHER, "polyphase": ctr.CTR_PATH_POLYPHASE,
         "col2im": ctr.CTR_PATH_COL2IM}
GRID_1D = [(1, 4, 2, 1, 0), (5, 4, 2, 1, 1), (37, 16, 8, 4, 0), (37, 16, 8, 4, 3), (9, 3, 2, 1, 1),
           (7, 7, 3, 2, 2), (11, 8, 4, 0, 0), (13, 6, 3, 0, 2), (20, 2, 2, 0, 0), (3, 10, 5, 2, 4)]
GRID_2D = [(5, 7, 4, 4, 2, 2, 1, 1, 0, 0), (6, 3, 3, 3, 2, 2, 1, 0, 1, 1), (4, 5, 4, 6, 2, 3, 1, 2, 1, 0)]


def _ints(rng, shape, mag=2):
    return rng.integers(-mag, mag + 1, shape).astype(np.float32)


@pytest.mark.parametrize("path", sorted(PATHS))
def test_f16_integer_grid_bit_exact(path):
    rng = np.random.default_rng(81)
    n = 0
    for (L, k, s, p, op) in GRID_1D:
        for (ci, co) in [(3, 2), (20, 33), (70, 40)]:
            n += 1
            x, w, b = _ints(rng, (2, ci, L)), _ints(rng, (ci, co, k)), _ints(rng, co)
            slope = 0.25 if n % 3 == 0 else None
            y, desc = run_plan(x, w, b if n % 2 else None, s, p, op, "f16", slope=slope,
                               path=PATHS[path], expect_path=PATHS[path])
            ref = reference(x, w, b if n % 2 else None, s, p, op, "f16", slope=slope)
            np.testing.assert_array_equal(y, ref, err_msg="%s %s" % ((L, k, s, p, op, ci, co), desc))
    for (H, W, ky, kx, sy, sx, py, px, opy, opx) in GRID_2D:
        x, w, b = _ints(rng, (1, 20, H, W)), _ints(rng, (20, 24, ky, kx)), _ints(rng, 24)
        y, desc = run_plan(x, w, b, (sy, sx), (py, px), (opy, opx), "f16", path=PATHS[path])
        np.testing.assert_array_equal(y, reference(x, w, b, (sy, sx), (py, px), (opy, opx), "f16"),
                                      err_msg=desc)


@pytest.mark.parametrize("origin", [ctr.CTR_PHASE_UNPADDED, ctr.CTR_PHASE_OUTPUT])
@pytest.mark.parametrize("split_k", [1, 3])
def test_f16_polyphase_tiles_split_and_origins_bit_exact(split_k, origin):
    rng = np.random.default_rng(83 + split_k)
    for (B, ci, co, L, k, s, p, op) in [(2, 100, 70, 300, 4, 2, 1, 0), (1, 96, 33, 131, 16, 8, 4, 3),
                                        (1, 64, 32, 700, 4, 2, 1, 0)]:
        x, w, b = _ints(rng, (B, ci, L), 1), _ints(rng, (ci, co, k), 1), _ints(rng, co, 1)
        y, desc = run_plan(x, w, b, s, p, op, "f16", path=ctr.CTR_PATH_POLYPHASE, split_k=split_k,
                           phase_origin=origin)
        np.testing.assert_array_equal(y, reference(x, w, b, s, p, op, "f16"), err_msg=desc)


@pytest.mark.parametrize("path", sorted(PATHS))
def test_f16_random_within_tolerance(path):
    rng = np.random.default_rng(85)
    cases = [((2, 96, 130), (96, 48, 8), 4, 2, 1), ((1, 33, 77), (33, 70, 3), 2, 1, 1),
             ((1, 64, 30, 20), (64, 24, 4, 4), (2, 2), (1, 1), (1, 0)),
             ((1, 512, 400), (512, 256, 16), 8, 4, 0)]
    for (xs, ws, s, p, op) in cases:
        x = workloads._cast(rng.standard_normal(xs), "f16")
        w = workloads._cast(rng.uniform(-0.1, 0.1, ws), "f16")
        b = workloads._cast(rng.normal(0, 0.1, ws[1]), "f16")
        y, desc = run_plan(x, w, b, s, p, op, "f16", path=PATHS[path])
        err = oracle.rel_l2(y, reference(x, w, b, s, p, op, "f16"))
        assert err <= TOL["f16"], "rel_l2 %.3g %s" % (err, desc)


@pytest.mark.parametrize("path", sorted(PATHS))
def test_f16_cancelling_taps(path):
    """Within one tap, the input channels run big, small, -big, small, ... (big in [300, 600),
    |small| in [0.005, 0.01], all fp16 values; x = 1), so every partial sum passes through
    a large value before the next channel cancels it.  Rounded to fp16 (spacing 0.25 to 0.5
    there) a partial sum would lose each small term; fp32 sums lose at most ~3e-5 per group,
    so every output stays within 2e-3 of the oracle."""
    C_in, C_out, L, k, s = 32, 64, 40, 4, 2
    rng = np.random.default_rng(87)
    x = np.ones((1, C_in, L), np.float32)
    w = np.zeros((C_in, C_out, k), np.float32)
    big = workloads._cast(rng.uniform(300, 600, (C_in // 4, C_out)), "f16")
    small = workloads._cast(rng.uniform(0.005, 0.01, (C_in // 2, C_out))
                            * rng.choice([-1.0, 1.0], (C_in // 2, C_out)), "f16")
    w[0::4, :, 0] = big
    w[2::4, :, 0] = -big
    w[1::2, :, 0] = small
    y, desc = run_plan(x, w, None, s, 1, 0, "f16", path=PATHS[path])
    ref = reference(x, w, None, s, 1, 0, "f16")
    assert np.max(np.abs(y - ref)) <= 2e-3, desc
    # the small terms survive: the outputs they reach are far from zero
    assert np.max(np.abs(y)) >= 0.01, desc


def test_f16_chained_pair_bit_exact():
    rng = np.random.default_rng(89)
    p1 = ctr.Plan(1, 64, 64, (300,), (16,), 8, 4, 0, dtype=torch.float16, negative_slope=0.25)
    p2 = ctr.Plan(1, 64, 32, p1.out_spatial, (4,), 2, 1, 0, dtype=torch.float16)
    try:
        p1.chain(p2)
        x, w1, w2 = _ints(rng, (1, 64, 300), 1), _ints(rng, (64, 64, 16), 1), _ints(rng, (64, 32, 4), 1)
        b1, b2 = _ints(rng, 64, 1), _ints(rng, 32, 1)
        p1.prepack(to_dev(w1, "f16"))
        p2.prepack(to_dev(w2, "f16"))
        y = torch.full(p2.out_shape, float("nan"), dtype=tdtype("f16"), device="cuda")
        p1.forward(to_dev(x, "f16"), to_dev(b1, "f16"))
        p2.forward(None, to_dev(b2, "f16"), y=y)
        p1.check()
        p2.check()
        h = reference(x, w1, b1, 8, 4, 0, "f16", slope=0.25)
        np.testing.assert_array_equal(y.float().cpu().numpy(), reference(h, w2, b2, 2, 1, 0, "f16"),
                                      err_msg="%s | %s" % (p1.describe(), p2.describe()))
    finally:
        p1.close()
        p2.close()


def test_f16_grouped_runs_gather_bit_exact():
    rng = np.random.default_rng(91)
    for (ci, co, G, sp, k, s, p) in [(16, 16, 16, (9, 12), (4, 4), (2, 2), (1, 1)),
                                     (32, 64, 8, (50,), (4,), (2,), (1,))]:
        x = _ints(rng, (1, ci) + sp)
        w = _ints(rng, (ci, co // G) + k)
        b = _ints(rng, co)
        y, desc = run_plan(x, w, b, s, p, 0, "f16", groups=G, expect_path=ctr.CTR_PATH_GATHER)
        ref = reference(x, w, b, s, p, 0, "f16", groups=G)
        np.testing.assert_array_equal(y, ref, err_msg=desc)
