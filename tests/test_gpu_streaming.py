"""GPU parity of streaming ConvTranspose1d (ctr_plan_set_streaming) against the oracle.

A streaming decoder feeds its upsampler consecutive chunks of frames and overlap-adds the
results ("[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to space",
Test plan: the overlap-add of a streaming decoder). Each call emits the s * L samples its
frames complete, and the plan carries the last m - 1 input frames to the next call. So the
concatenated outputs of a stream must equal the unpadded ConvTranspose of the concatenated
input, up to its last k - s samples. Zero chunks at the end flush those out.

Checks, every output between NaN guard bands:
- small-integer inputs equal the oracle bit for bit;
- random inputs stay within rel_l2 1e-5 (fp32) / 1e-2 (bf16), and equal one plain plan run
  over the whole concatenated input bit for bit;
- chunks shorter than the carried frames; a kernel that is not a multiple of the stride;
  LeakyReLU; split-K plans; ctr_plan_stream_reset starting a new stream; forward before the
  reset refused.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import transposed_convolution_gb300 as ctr  # noqa: E402
from gpu_helpers import GUARD, TOL, tdtype, to_dev  # noqa: E402

# (name, B, C_in, C_out, k, s, chunk frames, data chunks, dtype, slope).  The LeakyReLU
# slopes are powers of two, so that slope * (an exact integer sum) is exact in fp32 and in
# double alike and the integer cases stay bit-exact.
CASES = [
    ("codec_k16_s8", 2, 64, 32, 16, 8, 37, 4, "bf16", None),
    ("k4_s2_f32", 1, 32, 64, 4, 2, 13, 5, "f32", None),
    ("k6_s2_short_chunks", 1, 48, 32, 6, 2, 1, 7, "f32", 0.25),
    ("k5_s2_zero_padded", 2, 32, 32, 5, 2, 7, 3, "bf16", None),
    ("k8_s4_one_frame", 1, 64, 64, 8, 4, 1, 5, "bf16", 0.25),
]


def _flush_chunks(k, s, L):
    m = -(-k // s)
    return -(-(m - 1) // L) if m > 1 else 0


def _run_stream(case, chunks, b, w, split_k=0, block_n=0, expect_mode=None):
    """Feed the chunks through one streaming plan; returns the concatenated output (float64)."""
    name, B, C_in, C_out, k, s, L, _, dtype, slope = case
    plan = ctr.Plan(B, C_in, C_out, (L,), (k,), s, 0, 0, dtype=tdtype(dtype),
                    negative_slope=slope, streaming=True, split_k=split_k, block_n=block_n)
    try:
        assert plan.path == ctr.CTR_PATH_POLYPHASE, plan.describe()
        if expect_mode is not None:
            assert expect_mode in plan.describe(), plan.describe()
        assert plan.out_shape == (B, C_out, s * L)
        plan.prepack(to_dev(w, dtype))
        outs = []
        n = B * C_out * s * L
        for xc in chunks:
            buf = torch.full((n + 2 * GUARD,), float("nan"), dtype=tdtype(dtype), device="cuda")
            y = buf[GUARD:GUARD + n].view(plan.out_shape)
            plan.forward(to_dev(xc, dtype), to_dev(b, dtype), y=y)
            g = torch.cat([buf[:GUARD], buf[GUARD + n:]]).float().cpu().numpy()
            assert np.all(np.isnan(g)), "library wrote outside y"
            outs.append(y.float().cpu().numpy().astype(np.float64))
        plan.check()
        return np.concatenate(outs, axis=2)
    finally:
        plan.close()


def _inputs(case, integer, seed):
    name, B, C_in, C_out, k, s, L, nchunks, dtype, slope = case
    rng = np.random.default_rng(seed)
    if integer:
        xs = [rng.integers(-3, 4, (B, C_in, L)).astype(np.float32) for _ in range(nchunks)]
        w = rng.integers(-3, 4, (C_in, C_out, k)).astype(np.float32)
        b = rng.integers(-3, 4, (C_out,)).astype(np.float32)
    else:
        xs = [rng.standard_normal((B, C_in, L)).astype(np.float32) for _ in range(nchunks)]
        w = rng.uniform(-0.3, 0.3, (C_in, C_out, k)).astype(np.float32)
        b = rng.standard_normal(C_out).astype(np.float32)
        if dtype == "bf16":
            xs = [oracle.round_bf16(a).astype(np.float32) for a in xs]
            w, b = oracle.round_bf16(w).astype(np.float32), oracle.round_bf16(b).astype(np.float32)
    xs += [np.zeros((B, C_in, L), np.float32)] * _flush_chunks(k, s, L)
    return xs, w, b


def _reference(case, xs, w, b):
    name, B, C_in, C_out, k, s, L, nchunks, dtype, slope = case
    x_all = np.concatenate(xs, axis=2)
    y = oracle.conv_transpose(x_all, w, b, s, 0, 0)[:, :, :s * x_all.shape[2]]
    if slope is not None:
        y = oracle.leaky_relu(y, slope)
    return oracle.round_bf16(y) if dtype == "bf16" else oracle.round_f32(y)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_stream_integer_exact(case):
    xs, w, b = _inputs(case, True, 3)
    y = _run_stream(case, xs, b, w)
    ref = _reference(case, xs, w, b)
    assert y.shape == ref.shape
    np.testing.assert_array_equal(y, ref)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_stream_random_matches_oracle_and_whole_input(case):
    name, B, C_in, C_out, k, s, L, nchunks, dtype, slope = case
    xs, w, b = _inputs(case, False, 5)
    # No split-K on either side: one fixed summation order per output.
    y = _run_stream(case, xs, b, w, split_k=1)
    err = oracle.rel_l2(y, _reference(case, xs, w, b))
    assert err <= TOL[dtype], err
    # One plain polyphase plan over the whole input: the same sums, the same bits.
    x_all = np.concatenate(xs, axis=2)
    whole = ctr.Plan(B, C_in, C_out, (x_all.shape[2],), (k,), s, 0, 0, dtype=tdtype(dtype),
                     negative_slope=slope, path=ctr.CTR_PATH_POLYPHASE, split_k=1)
    try:
        whole.prepack(to_dev(w, dtype))
        yw = whole.forward(to_dev(x_all, dtype), to_dev(b, dtype))
        yw = yw.float().cpu().numpy().astype(np.float64)[:, :, :s * x_all.shape[2]]
    finally:
        whole.close()
    np.testing.assert_array_equal(y, yw)


def test_stream_fp32_xring_integer_exact():
    """An fp32 stream on 256-row tiles with four taps: the GEMM runs in X-ring mode (the taps
    share one box of the staged input, whose leading halo holds the carried frames)."""
    case = ("k16_s4_f32_xring", 1, 64, 64, 16, 4, 29, 4, "f32", None)
    xs, w, b = _inputs(case, True, 13)
    y = _run_stream(case, xs, b, w, block_n=256, expect_mode=" x-ring")
    np.testing.assert_array_equal(y, _reference(case, xs, w, b))


def test_stream_reset_starts_a_new_stream():
    case = CASES[1]
    name, B, C_in, C_out, k, s, L, nchunks, dtype, slope = case
    xs, w, b = _inputs(case, True, 9)
    plan = ctr.Plan(B, C_in, C_out, (L,), (k,), s, 0, 0, dtype=tdtype(dtype), streaming=True)
    try:
        plan.prepack(to_dev(w, dtype))
        first = [plan.forward(to_dev(xc, dtype), to_dev(b, dtype)).float().cpu().numpy()
                 for xc in xs[:2]]
        plan.stream_reset()
        again = [plan.forward(to_dev(xc, dtype), to_dev(b, dtype)).float().cpu().numpy()
                 for xc in xs[:2]]
        plan.check()
        for a, c in zip(first, again):
            np.testing.assert_array_equal(a, c)
        # A freshly bound workspace must be reset before the next call.
        ctr.ctr_plan_bind_workspace(plan.handle, ctr._ptr(plan.workspace), plan.workspace_bytes)
        y = torch.empty(plan.out_shape, dtype=tdtype(dtype), device="cuda")
        st = ctr.lib.ctr_forward(plan.handle, ctr._ptr(to_dev(xs[0], dtype)),
                                 ctr._ptr(plan.w_packed), None, ctr._ptr(y), None)
        assert st == ctr.CTR_ERR_NOT_PREPARED
        st = ctr.lib.ctr_forward_noalloc(plan.handle, ctr._ptr(to_dev(xs[0], dtype)),
                                         ctr._ptr(to_dev(w, dtype)), None, ctr._ptr(y), None)
        assert st == ctr.CTR_ERR_UNSUPPORTED
    finally:
        plan.close()
