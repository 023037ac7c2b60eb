"""Chained plans (ctr_plan_chain): a plan's output stage writes straight into the next plan's
staged input, and the next plan runs without staging.  The chained results must equal the
unchained calls bit for bit (the staged values are the same: bf16 rounding, or the tf32
hi/lo split of the fp32 output), on repeated calls too (the staged halos stay zero)."""
import numpy as np
import pytest
import torch

from gpu_helpers import tdtype

import transposed_convolution_gb300 as ctr

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


def _make(dtype, B, C_in, sp, layers, rng, chained):
    """Plans for the layers (chained before the weights are packed, when asked), their biases
    and the weights drawn from rng."""
    plans, bs, ws = [], [], []
    c, s = C_in, tuple(sp)
    for (co, k, st, p, op, slope) in layers:
        pl = ctr.Plan(B, c, co, s, k if isinstance(k, tuple) else (k,) * len(s), st, p, op,
                      dtype=tdtype(dtype), negative_slope=slope)
        ws.append(rng.uniform(-0.2, 0.2, (c, co) + tuple(pl.kernel)).astype(np.float32))
        bs.append(torch.from_numpy(rng.standard_normal(co).astype(np.float32)).cuda().to(tdtype(dtype)))
        plans.append(pl)
        c, s = co, pl.out_spatial
    if chained:
        for a, nxt in zip(plans[:-1], plans[1:]):
            a.chain(nxt)
    for pl, w in zip(plans, ws):
        pl.prepack(torch.from_numpy(w).cuda().to(tdtype(dtype)))
    return plans, bs


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
