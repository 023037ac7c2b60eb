"""The GEMM's shared-memory pipeline modes against the oracle.

For 16-bit 1-D polyphase plans with several taps, one X box per channel slice (128
positions plus the taps' row shifts) serves every tap through a descriptor that starts
further down the box ("shared-x"), and a weight tile that fits stays resident in shared
memory for the whole kernel ("resident-w").  Each case states which pipeline its plan
describes, so every mode runs: shared X with a resident weight, shared X with per-stage
weight slices (several row tiles), and the default ring.  Small-integer inputs make every
sum exact, so the results must equal the oracle bit for bit, over ragged position tails,
several channel slices, both phase origins, a fused activation and a chained pair.
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
from gpu_helpers import reference, run_plan, tdtype, to_dev  # noqa: E402

# (B, C_in, C_out, L, k, s, p, op, phase origin, expected pipeline text), run with split-K 1
# (the shared-X modes need one K split).
CASES = [
    (1, 64, 32, 1000, 4, 2, 1, 0, ctr.CTR_PHASE_AUTO, "shared-x resident-w"),
    (1, 64, 32, 500, 16, 2, 7, 1, ctr.CTR_PHASE_AUTO, "shared-x resident-w"),   # 8 taps
    (2, 128, 64, 333, 4, 2, 1, 1, ctr.CTR_PHASE_AUTO, "shared-x"),              # 2 row tiles
    (1, 128, 64, 257, 4, 2, 1, 0, ctr.CTR_PHASE_UNPADDED, "shared-x"),
    (1, 200, 32, 150, 6, 2, 2, 0, ctr.CTR_PHASE_AUTO, "shared-x"),              # 4 slices, ragged C_in
    (1, 64, 256, 300, 4, 2, 1, 0, ctr.CTR_PHASE_AUTO, "shared-x"),              # 8 row tiles
    (1, 64, 64, 300, 8, 8, 0, 0, ctr.CTR_PHASE_AUTO, "stages=4"),               # one tap: default
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%dx%d-k%ds%dp%d-%s" % (c[1], c[2], c[4], c[5], c[6], c[9].replace(" ", "_")))
def test_pipeline_modes_bit_exact(case):
    B, ci, co, L, k, s, p, op, origin, mode = case
    rng = np.random.default_rng(ci * 7 + co)
    x = rng.integers(-1, 2, (B, ci, L)).astype(np.float32)
    w = rng.integers(-1, 2, (ci, co, k)).astype(np.float32)
    b = rng.integers(-1, 2, co).astype(np.float32)
    for slope in (None, 0.25):
        y, desc = run_plan(x, w, b, s, p, op, "bf16", slope=slope, path=ctr.CTR_PATH_POLYPHASE,
                           split_k=1, phase_origin=origin)
        assert mode in desc and ("shared-x" in mode) == ("shared-x" in desc), desc
        np.testing.assert_array_equal(y, reference(x, w, b, s, p, op, "bf16", slope=slope),
                                      err_msg=desc)


def test_pipeline_modes_random_within_tolerance():
    rng = np.random.default_rng(71)
    for (B, ci, co, L, k, s, p, op, origin, mode) in CASES:
        x = workloads._cast(rng.standard_normal((B, ci, L)), "bf16")
        w = workloads._cast(rng.uniform(-0.1, 0.1, (ci, co, k)), "bf16")
        b = workloads._cast(rng.normal(0, 0.1, co), "bf16")
        y, desc = run_plan(x, w, b, s, p, op, "bf16", path=ctr.CTR_PATH_POLYPHASE, split_k=1,
                           phase_origin=origin)
        err = oracle.rel_l2(y, reference(x, w, b, s, p, op, "bf16"))
        assert err <= 1e-2, "rel_l2 %.3g %s" % (err, desc)


def test_chained_shared_x_pair_bit_exact():
    """A chained producer and its consumer, both on shared X with resident weights: the
    consumer reads the producer's output from its staged input."""
    rng = np.random.default_rng(73)
    p1 = ctr.Plan(1, 128, 64, (700,), (4,), 2, 1, 0, dtype=torch.bfloat16, negative_slope=0.25)
    p2 = ctr.Plan(1, 64, 32, p1.out_spatial, (4,), 2, 1, 0, dtype=torch.bfloat16)
    try:
        p1.chain(p2)
        assert "shared-x" in p1.describe() and "shared-x" in p2.describe()
        x = rng.integers(-1, 2, (1, 128, 700)).astype(np.float32)
        w1 = rng.integers(-1, 2, (128, 64, 4)).astype(np.float32)
        w2 = rng.integers(-1, 2, (64, 32, 4)).astype(np.float32)
        b1 = rng.integers(-1, 2, 64).astype(np.float32)
        b2 = rng.integers(-1, 2, 32).astype(np.float32)
        p1.prepack(to_dev(w1, "bf16"))
        p2.prepack(to_dev(w2, "bf16"))
        for it in range(2):
            y = torch.full(p2.out_shape, float("nan"), dtype=tdtype("bf16"), device="cuda")
            p1.forward(to_dev(x, "bf16"), to_dev(b1, "bf16"))
            p2.forward(None, to_dev(b2, "bf16"), y=y)
            p1.check()
            p2.check()
            h = reference(x, w1, b1, 2, 1, 0, "bf16", slope=0.25)
            np.testing.assert_array_equal(y.float().cpu().numpy(),
                                          reference(h, w2, b2, 2, 1, 0, "bf16"),
                                          err_msg="call %d" % it)
    finally:
        p1.close()
        p2.close()
