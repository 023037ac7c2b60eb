"""ctr_forward_fused: two chained 1-D layers in one kernel, the first layer's output kept in
shared memory as the second layer's operand.

The result must equal the two chained launches bit for bit (the same products in the same
order, one rounding of the first layer's outputs) and the oracle run stage by stage with
the first layer's output rounded to the I/O type: bit for bit on small-integer inputs,
within the I/O tolerance on random ones, at full size on the vocoder stack's last two
layers (128 -> 64 -> 32 channels, 65536 -> 262144 samples), with the input staged by a
preceding chained plan, and through the bounded-wait timeout path.
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
from gpu_helpers import TOL, reference, tdtype, to_dev  # noqa: E402


def _pair(dtype, B, C0, L, C2, kA=4, sA=2, pA=1, kB=4, sB=2, pB=1, slope=0.25, originB=0):
    a = ctr.Plan(B, C0, 64, (L,), (kA,), sA, pA, 0, dtype=tdtype(dtype), negative_slope=slope)
    b = ctr.Plan(B, 64, C2, a.out_spatial, (kB,), sB, pB, 0, dtype=tdtype(dtype),
                 phase_origin=originB)
    a.chain(b)
    return a, b


def _run_both(a, b, x, wa, ba, wb, bb, dtype):
    """(fused output, chained two-launch output) as float64 numpy."""
    a.prepack(to_dev(wa, dtype))
    b.prepack(to_dev(wb, dtype))
    xd, bad, bbd = to_dev(x, dtype), to_dev(ba, dtype), to_dev(bb, dtype)
    y1 = torch.full(b.out_shape, float("nan"), dtype=tdtype(dtype), device="cuda")
    a.forward_fused(xd, bad, bbd, y=y1)
    a.check()
    y2 = torch.full(b.out_shape, float("nan"), dtype=tdtype(dtype), device="cuda")
    a.forward(xd, bad)
    b.forward(None, bbd, y=y2)
    a.check()
    b.check()
    return (y1.float().cpu().numpy().astype(np.float64), y2.float().cpu().numpy().astype(np.float64))


CASES = [  # (B, C0, L, C2, kA, sA, pA, kB, sB, pB, B's phase origin)
    (1, 128, 1000, 32, 4, 2, 1, 4, 2, 1, ctr.CTR_PHASE_AUTO),
    (2, 128, 257, 32, 4, 2, 1, 4, 2, 1, ctr.CTR_PHASE_AUTO),
    (1, 96, 130, 64, 4, 2, 1, 4, 2, 1, ctr.CTR_PHASE_UNPADDED),
    (2, 96, 700, 32, 4, 2, 1, 4, 2, 1, ctr.CTR_PHASE_UNPADDED),  # paired stores
    # long rows: two MMA groups per tile, several tiles per CTA, tiles ending inside a row,
    # paired stores
    (2, 96, 20000, 32, 4, 2, 1, 4, 2, 1, ctr.CTR_PHASE_UNPADDED),
    (1, 64, 300, 32, 6, 2, 2, 6, 2, 2, ctr.CTR_PHASE_AUTO),
    (1, 128, 77, 32, 4, 2, 0, 4, 2, 0, ctr.CTR_PHASE_AUTO),
    (1, 60, 161, 32, 8, 2, 3, 8, 2, 3, ctr.CTR_PHASE_AUTO),     # 4 and 5 taps, ragged C0
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d-%d-L%d-%d" % c[:4])
def test_fused_integer_bit_exact(case, dtype):
    B, C0, L, C2, kA, sA, pA, kB, sB, pB, origin = case
    rng = np.random.default_rng(C0 + L)
    a, b = _pair(dtype, B, C0, L, C2, kA, sA, pA, kB, sB, pB, 0.25, origin)
    try:
        assert a.fusable, a.describe()
        x = rng.integers(-1, 2, (B, C0, L)).astype(np.float32)
        wa = rng.integers(-1, 2, (C0, 64, kA)).astype(np.float32)
        wb = rng.integers(-1, 2, (64, C2, kB)).astype(np.float32)
        ba = rng.integers(-1, 2, 64).astype(np.float32)
        bb = rng.integers(-1, 2, C2).astype(np.float32)
        fused, chained = _run_both(a, b, x, wa, ba, wb, bb, dtype)
        np.testing.assert_array_equal(fused, chained, err_msg=a.describe())
        h = reference(x, wa, ba, sA, pA, 0, dtype, slope=0.25)
        np.testing.assert_array_equal(fused, reference(h, wb, bb, sB, pB, 0, dtype))
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_fused_random_matches_chain_and_oracle(dtype):
    rng = np.random.default_rng(111)
    a, b = _pair(dtype, 1, 128, 2000, 32, slope=0.1)
    try:
        x = workloads._cast(rng.standard_normal((1, 128, 2000)), dtype)
        wa = workloads._cast(rng.uniform(-0.1, 0.1, (128, 64, 4)), dtype)
        wb = workloads._cast(rng.uniform(-0.1, 0.1, (64, 32, 4)), dtype)
        ba = workloads._cast(rng.normal(0, 0.1, 64), dtype)
        bb = workloads._cast(rng.normal(0, 0.1, 32), dtype)
        fused, chained = _run_both(a, b, x, wa, ba, wb, bb, dtype)
        np.testing.assert_array_equal(fused, chained)
        h = reference(x, wa, ba, 2, 1, 0, dtype, slope=0.1)
        assert oracle.rel_l2(fused, reference(h, wb, bb, 2, 1, 0, dtype)) <= TOL[dtype]
    finally:
        a.close()
        b.close()


def test_fused_vocoder_last_two_layers_full_size():
    """Layers 3 and 4 of the vocoder stack at full size, their input staged by layer 2
    (chained), against the chained launches (bit for bit) and the oracle (within 1e-2)."""
    stages = workloads.make_workload("vocoder_stack_bf16")
    L2, L3, L4 = (li.layer for li in stages[1:])
    rng = np.random.default_rng(113)
    x2 = workloads._cast(rng.standard_normal((1, L2.C_in) + L2.in_sp), "bf16")
    plans = [ctr.Plan(L.B, L.C_in, L.C_out, L.in_sp, L.kernel, L.stride, L.padding,
                      L.output_padding, dtype=torch.bfloat16, negative_slope=L.act_slope)
             for L in (L2, L3, L4)]
    try:
        plans[0].chain(plans[1])
        plans[1].chain(plans[2])
        assert plans[1].fusable, plans[1].describe()
        for p, li in zip(plans, stages[1:]):
            p.prepack(to_dev(li.w, "bf16"))
        bs = [to_dev(li.bias, "bf16") for li in stages[1:]]
        y1 = torch.full(plans[2].out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        plans[0].forward(to_dev(x2, "bf16"), bs[0])
        plans[1].forward_fused(None, bs[1], bs[2], y=y1)
        y2 = torch.full(plans[2].out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        plans[0].forward(to_dev(x2, "bf16"), bs[0])
        plans[1].forward(None, bs[1])
        plans[2].forward(None, bs[2], y=y2)
        for p in plans:
            p.check()
        got = y1.float().cpu().numpy().astype(np.float64)
        np.testing.assert_array_equal(got, y2.float().cpu().numpy().astype(np.float64))
        h = x2.astype(np.float64)
        for li in stages[1:]:
            L = li.layer
            h = reference(h, li.w, li.bias, L.stride, L.padding, L.output_padding, "bf16",
                          slope=L.act_slope)
        err = oracle.rel_l2(got, h)
        print("fused layers 3+4 rel_l2 %.3g" % err)
        assert err <= TOL["bf16"]
    finally:
        for p in plans:
            p.close()


def test_fused_timeout_reports_and_recovers():
    """A 0 ns wait limit makes the fused kernel's bounded waits give up on a healthy run:
    ctr_plan_check reports CTR_ERR_DEVICE_TIMEOUT, and with the normal limit the next call
    is correct."""
    rng = np.random.default_rng(115)
    a, b = _pair("bf16", 1, 128, 600, 32)
    try:
        x = rng.integers(-1, 2, (1, 128, 600)).astype(np.float32)
        wa = rng.integers(-1, 2, (128, 64, 4)).astype(np.float32)
        wb = rng.integers(-1, 2, (64, 32, 4)).astype(np.float32)
        ba = rng.integers(-1, 2, 64).astype(np.float32)
        bb = rng.integers(-1, 2, 32).astype(np.float32)
        a.prepack(to_dev(wa, "bf16"))
        b.prepack(to_dev(wb, "bf16"))
        a.set_wait_limit_ns(0)
        a.forward_fused(to_dev(x, "bf16"), to_dev(ba, "bf16"), to_dev(bb, "bf16"))
        with pytest.raises(ctr.CtrError) as e:
            a.check()
        assert e.value.status == ctr.CTR_ERR_DEVICE_TIMEOUT
        a.set_wait_limit_ns(4_000_000_000)
        y = a.forward_fused(to_dev(x, "bf16"), to_dev(ba, "bf16"), to_dev(bb, "bf16"))
        a.check()
        h = reference(x, wa, ba, 2, 1, 0, "bf16", slope=0.25)
        np.testing.assert_array_equal(y.float().cpu().numpy(), reference(h, wb, bb, 2, 1, 0, "bf16"))
    finally:
        a.close()
        b.close()
