"""Chained plans (ctr_plan_chain): a plan's output stage writes straight into the next plan's
staged input, and the next plan runs without staging.

* The chained results must equal the unchained calls bit for bit (the staged values are the
  same: bf16 rounding, or the tf32 and bf16-pair split of the fp32 output), on repeated calls too
  (the staged halos stay zero).
* Against the oracle, run stage by stage with the output of each stage rounded to the I/O
  type (the value the next stage reads): within rel_l2 <= 1e-5 (fp32 I/O) or <= 1e-2 (bf16)
  on random inputs, bit for bit on small-integer inputs (every product and partial sum is
  then exact), and at full size on the vocoder stack the benchmark runs chained.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, reference, tdtype, to_dev

import oracle
import transposed_convolution_gb300 as ctr
import workloads

pytestmark = pytest.mark.gpu

# Each chain: dtype, batch, input channels and spatial size, then per layer
# (C_out, kernel, stride, padding, output_padding, LeakyReLU slope or None).
CHAINS = [
    ("bf16", 1, 64, (300,), [(64, 16, 8, 4, 0, 0.1), (32, 16, 8, 4, 0, 0.1)]),       # S8 -> S8
    ("bf16", 2, 48, (256,), [(40, 4, 2, 1, 0, 0.1), (40, 4, 2, 1, 1, None)]),        # S2, padded C_in
    ("f32", 1, 64, (200,), [(48, 8, 4, 2, 0, 0.2), (64, 4, 2, 1, 0, None)]),         # S4 -> S2
    ("f32", 2, 32, (20, 17), [(40, (4, 4), (2, 2), (1, 1), (0, 1), 0.1),
                              (32, (4, 4), (2, 2), (1, 1), (0, 0), None)]),          # 2-D
    ("bf16", 1, 32, (100,), [(64, 4, 2, 1, 0, 0.1), (32, 3, 2, 1, 1, None)]),        # col2im next
    ("bf16", 1, 128, (128,), [(64, 16, 8, 4, 0, 0.1), (64, 4, 2, 1, 0, 0.1),
                              (32, 4, 2, 1, 0, None)]),                              # three plans
]


def _make(dtype, B, C_in, sp, layers, rng, chained, integer=False, host=None):
    """Plans for the layers (chained before the weights are packed, when asked), their biases
    and the weights drawn from rng (small integers when `integer`); the host copies (weight,
    bias as numpy values of the I/O type) are appended to `host` when given."""
    plans, bs, ws = [], [], []
    c, s = C_in, tuple(sp)
    for (co, k, st, p, op, slope) in layers:
        pl = ctr.Plan(B, c, co, s, k if isinstance(k, tuple) else (k,) * len(s), st, p, op,
                      dtype=tdtype(dtype), negative_slope=slope)
        if integer:
            w = rng.integers(-2, 3, (c, co) + tuple(pl.kernel)).astype(np.float32)
            b = rng.integers(-2, 3, co).astype(np.float32)
        else:
            w = workloads._cast(rng.uniform(-0.2, 0.2, (c, co) + tuple(pl.kernel)), dtype)
            b = workloads._cast(rng.standard_normal(co), dtype)
        ws.append(w)
        bs.append(to_dev(b, dtype))
        if host is not None:
            host.append((w, b))
        plans.append(pl)
        c, s = co, pl.out_spatial
    if chained:
        for a, nxt in zip(plans[:-1], plans[1:]):
            a.chain(nxt)
    for pl, w in zip(plans, ws):
        pl.prepack(to_dev(w, dtype))
    return plans, bs


def _run_chain(plans, bs, x, dtype):
    """One chained forward pass: only the first layer stages an input, only the last writes
    a y (NaN-filled beforehand, so an unwritten output shows)."""
    y = torch.full(plans[-1].out_shape, float("nan"), dtype=tdtype(dtype), device="cuda")
    assert plans[0].forward(x, bs[0]) is None
    for pl, b in zip(plans[1:-1], bs[1:-1]):
        assert pl.forward(None, b) is None
    plans[-1].forward(None, bs[-1], y=y)
    torch.cuda.synchronize()
    for pl in plans:
        pl.check()
    return y.float().cpu().numpy().astype(np.float64)


def _oracle_chain(x, layers, host, dtype):
    """The oracle stage by stage: each stage's double result plus bias, LeakyReLU, rounded to
    the I/O type, is the next stage's input."""
    h = np.asarray(x, dtype=np.float64)
    for (co, k, st, p, op, slope), (w, b) in zip(layers, host):
        h = reference(h, w, b, st, p, op, dtype, slope=slope)
    return h


@pytest.mark.parametrize("case", CHAINS, ids=lambda c: "%s-%dd-%dlayers" % (c[0], len(c[3]), len(c[4])))
def test_chained_equals_unchained(case):
    dtype, B, C_in, sp, layers = case
    plans0, bs0 = _make(dtype, B, C_in, sp, layers, np.random.default_rng(41), chained=False)
    plans, bs = _make(dtype, B, C_in, sp, layers, np.random.default_rng(41), chained=True)
    try:
        x = torch.from_numpy(np.random.default_rng(42).standard_normal((B, C_in) + tuple(sp))
                             .astype(np.float32)).cuda().to(tdtype(dtype))
        # Unchained: every layer through the torch layout.
        h = x
        for pl, b in zip(plans0, bs0):
            h = pl.forward(h, b)
        ref = h.float().cpu().numpy()
        assert plans[0].path == ctr.CTR_PATH_POLYPHASE
        # Chained: only the first layer stages an input, only the last writes a y.
        for it in range(2):
            y = torch.full(plans[-1].out_shape, float("nan"), dtype=tdtype(dtype), device="cuda")
            assert plans[0].forward(x, bs[0]) is None
            for pl, b in zip(plans[1:-1], bs[1:-1]):
                assert pl.forward(None, b) is None
            plans[-1].forward(None, bs[-1], y=y)
            torch.cuda.synchronize()
            for pl in plans:
                pl.check()
            np.testing.assert_array_equal(y.float().cpu().numpy(), ref, err_msg="call %d" % it)
    finally:
        for pl in plans + plans0:
            pl.close()


def test_chain_errors_on_device():
    """A chained producer refuses a y and cannot be re-chained once packed; a plan fed by a
    chain still accepts an explicit x; a producer whose chain partner is gone refuses to run."""
    rng = np.random.default_rng(43)
    layers = [(64, 4, 2, 1, 0, None), (32, 4, 2, 1, 0, None)]
    plans, bs = _make("bf16", 1, 64, (128,), layers, rng, chained=True)
    try:
        x = torch.randn(1, 64, 128, device="cuda").to(torch.bfloat16)
        with pytest.raises(ValueError):
            plans[0].forward(x, bs[0], y=torch.empty(plans[0].out_shape, dtype=torch.bfloat16,
                                                   device="cuda"))
        st = ctr.lib.ctr_forward(plans[0].handle, x.data_ptr(), plans[0].w_packed.data_ptr(),
                                 None, x.data_ptr(), None)
        assert st == ctr.CTR_ERR_INVALID_ARG
        with pytest.raises(ctr.CtrError):
            plans[0].chain(None)                      # packed for the chained output
        # plans[1] with its own x: staged normally, same as an unchained plan
        x1 = torch.randn((1, 64) + plans[0].out_spatial, device="cuda").to(torch.bfloat16)
        y_a = plans[1].forward(x1, bs[1])
        p1, b1 = _make("bf16", 1, 64, (128,), layers, np.random.default_rng(43), chained=False)
        y_b = p1[1].forward(x1, b1[1])
        torch.cuda.synchronize()
        assert torch.equal(y_a, y_b)
        for pl in p1:
            pl.close()
        # the consumer destroyed: the producer's phase-major weight has no chain to feed
        plans[1].close()
        st = ctr.lib.ctr_forward(plans[0].handle, x.data_ptr(), plans[0].w_packed.data_ptr(),
                                 None, None, None)
        assert st == ctr.CTR_ERR_INVALID_ARG
    finally:
        for pl in plans:
            pl.close()


@pytest.mark.parametrize("case", CHAINS, ids=lambda c: "%s-%dd-%dlayers" % (c[0], len(c[3]), len(c[4])))
def test_chained_matches_oracle(case):
    """Random inputs: the chain's last output against the oracle run stage by stage."""
    dtype, B, C_in, sp, layers = case
    host = []
    plans, bs = _make(dtype, B, C_in, sp, layers, np.random.default_rng(51), chained=True,
                      host=host)
    try:
        x = workloads._cast(np.random.default_rng(52).standard_normal((B, C_in) + tuple(sp)), dtype)
        got = _run_chain(plans, bs, to_dev(x, dtype), dtype)
        ref = _oracle_chain(x, layers, host, dtype)
        assert not np.isnan(got).any()
        err = oracle.rel_l2(got, ref)
        assert err <= TOL[dtype], "rel_l2 %.3g" % err
    finally:
        for pl in plans:
            pl.close()


# Small-integer chains: |x|, |w|, |bias| <= 2 and LeakyReLU slopes that are powers of two, so
# every product and partial sum of every stage is exact and both sides round the same values.
INT_CHAINS = [
    ("bf16", 1, 32, (70,), [(32, 4, 2, 1, 0, 0.25), (32, 4, 2, 1, 0, None)]),        # odd pads
    ("bf16", 2, 16, (40,), [(24, 16, 8, 4, 0, 0.5), (32, 4, 2, 1, 1, 0.25),
                            (32, 4, 2, 0, 0, None)]),                                # S8, S2, op
    ("f32", 1, 32, (50,), [(32, 8, 4, 2, 0, 0.25), (32, 4, 2, 1, 0, None)]),
    ("f32", 1, 16, (9, 13), [(16, (4, 4), (2, 2), (1, 1), (0, 0), 0.5),
                             (16, (4, 4), (2, 2), (1, 1), (1, 0), None)]),           # 2-D
    ("bf16", 1, 32, (30,), [(64, 4, 2, 1, 0, 0.25), (32, 3, 2, 1, 1, None)]),        # col2im next
]


@pytest.mark.parametrize("case", INT_CHAINS,
                         ids=lambda c: "%s-%dd-%dlayers" % (c[0], len(c[3]), len(c[4])))
def test_integer_chain_bit_exact(case):
    dtype, B, C_in, sp, layers = case
    host = []
    rng = np.random.default_rng(61)
    plans, bs = _make(dtype, B, C_in, sp, layers, rng, chained=True, integer=True, host=host)
    try:
        x = rng.integers(-2, 3, (B, C_in) + tuple(sp)).astype(np.float32)
        for it in range(2):
            got = _run_chain(plans, bs, to_dev(x, dtype), dtype)
            np.testing.assert_array_equal(got, _oracle_chain(x, layers, host, dtype),
                                          err_msg="call %d" % it)
    finally:
        for pl in plans:
            pl.close()


def test_chained_split_k_ragged_channels_bit_exact():
    """A chained producer with split-K and a channel count that leaves the last phase-major
    row tile partly empty (40 channels in tiles of 16): the reduce must visit every packed
    row, since the last tile's channels are spread over its whole width."""
    rng = np.random.default_rng(67)
    for dtype in ("f32", "bf16"):
        p1 = ctr.Plan(2, 150, 40, (300,), (8,), 4, 2, 0, dtype=tdtype(dtype), split_k=3,
                      path=ctr.CTR_PATH_POLYPHASE)
        p2 = ctr.Plan(2, 40, 64, p1.out_spatial, (4,), 2, 1, 0, dtype=tdtype(dtype))
        try:
            p1.chain(p2)
            x = rng.integers(-1, 2, (2, 150, 300)).astype(np.float32)
            w1 = rng.integers(-1, 2, (150, 40, 8)).astype(np.float32)
            w2 = rng.integers(-1, 2, (40, 64, 4)).astype(np.float32)
            b1 = rng.integers(-1, 2, 40).astype(np.float32)
            b2 = rng.integers(-1, 2, 64).astype(np.float32)
            p1.prepack(to_dev(w1, dtype))
            p2.prepack(to_dev(w2, dtype))
            y = torch.full(p2.out_shape, float("nan"), dtype=tdtype(dtype), device="cuda")
            p1.forward(to_dev(x, dtype), to_dev(b1, dtype))
            p2.forward(None, to_dev(b2, dtype), y=y)
            p1.check()
            p2.check()
            h = reference(x, w1, b1, 4, 2, 0, dtype)
            np.testing.assert_array_equal(y.float().cpu().numpy(), reference(h, w2, b2, 2, 1, 0, dtype),
                                          err_msg="%s | %s" % (p1.describe(), p2.describe()))
        finally:
            p1.close()
            p2.close()


def test_vocoder_stack_chained_full_size():
    """The four bf16 upsamplers of the vocoder stack (512 -> 32 channels, 1024 -> 262144
    samples, LeakyReLU(0.1) after the first three), chained as the benchmark runs them,
    against the oracle run stage by stage with bf16 rounding between stages."""
    stages = workloads.make_workload("vocoder_stack_bf16")
    plans, bs = [], []
    try:
        for li in stages:
            L = li.layer
            plans.append(ctr.Plan(L.B, L.C_in, L.C_out, L.in_sp, L.kernel, L.stride, L.padding,
                                  L.output_padding, dtype=torch.bfloat16,
                                  negative_slope=L.act_slope))
            bs.append(to_dev(li.bias, "bf16"))
        for a, nxt in zip(plans[:-1], plans[1:]):
            a.chain(nxt)
        for pl, li in zip(plans, stages):
            pl.prepack(to_dev(li.w, "bf16"))
        got = _run_chain(plans, bs, to_dev(stages[0].x, "bf16"), "bf16")
        h = stages[0].x.astype(np.float64)
        for li in stages:
            L = li.layer
            h = reference(h, li.w, li.bias, L.stride, L.padding, L.output_padding, "bf16",
                          slope=L.act_slope)
        err = oracle.rel_l2(got, h)
        print("chained vocoder stack rel_l2 %.3g | %s" % (err, " | ".join(p.describe() for p in plans)))
        assert err <= TOL["bf16"]
    finally:
        for pl in plans:
            pl.close()
