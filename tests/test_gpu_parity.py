"""GPU parity: the CUDA library, through its C ABI, against the CPU oracle.

* integer-exact grids: small-integer inputs make every product and partial sum exact in
  fp32, tf32 and bf16, so every path must equal the oracle bit for bit;
* tile, split-K and ragged-edge shapes, bit-exact the same way;
* random inputs within rel_l2 <= 1e-5 (fp32 I/O, tf32 + bf16 split) or <= 1e-2 (bf16 I/O);
* the five workloads at full size, in the configuration the benchmark times;
* the iSTFT of a sinusoid at full size, against its closed form;
* edge cases of the pages: empty input, one input step, m = 1 and 3, k = 2s at s = 2, 4, 5,
  6 with and without bias, output_padding > padding, asymmetric 2-D padding, cancelling
  taps in bf16, stacked layers with an activation between them;
* error statuses and the bounded-wait timeout path.
Every output buffer sits between NaN guard bands that must survive the call.
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
from gpu_helpers import TOL, reference, run_plan, to_dev  # noqa: E402

PATHS = {"gather": ctr.CTR_PATH_GATHER, "polyphase": ctr.CTR_PATH_POLYPHASE,
         "col2im": ctr.CTR_PATH_COL2IM}


def _int_inputs(rng, shape_x, shape_w, C_out, mag, with_bias=True):
    x = rng.integers(-mag, mag + 1, shape_x).astype(np.float32)
    w = rng.integers(-mag, mag + 1, shape_w).astype(np.float32)
    b = rng.integers(-mag, mag + 1, (C_out,)).astype(np.float32) if with_bias else None
    return x, w, b


GRID_1D = [  # (L, k, s, p, op)
    (1, 4, 2, 1, 0), (5, 4, 2, 1, 1), (37, 16, 8, 4, 0), (37, 16, 8, 4, 3), (9, 3, 2, 1, 1),
    (7, 7, 3, 2, 2), (6, 5, 1, 2, 0), (11, 8, 4, 0, 0), (13, 6, 3, 0, 2), (4, 12, 4, 6, 1),
    (20, 2, 2, 0, 0), (3, 10, 5, 2, 4), (8, 1, 1, 0, 0),
]
GRID_2D = [  # (H, W, ky, kx, sy, sx, py, px, opy, opx)
    (5, 7, 4, 4, 2, 2, 1, 1, 0, 0), (6, 3, 3, 3, 2, 2, 1, 0, 1, 1), (4, 5, 4, 6, 2, 3, 1, 2, 1, 0),
    (3, 3, 2, 2, 1, 1, 0, 0, 0, 0), (9, 2, 6, 2, 3, 1, 2, 0, 2, 0),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_integer_exact_grid(path, dtype):
    rng = np.random.default_rng(11)
    mag = 2 if dtype == "f32" else 1
    chans = [(3, 2), (20, 9), (70, 33)] if dtype == "f32" else [(3, 2), (20, 9), (40, 17)]
    n = 0
    for (L, k, s, p, op) in GRID_1D:
        for (ci, co) in chans:
            n += 1
            x, w, b = _int_inputs(rng, (2, ci, L), (ci, co, k), co, mag, with_bias=n % 2 == 0)
            y, desc = run_plan(x, w, b, s, p, op, dtype, path=PATHS[path],
                               expect_path=PATHS[path])
            ref = reference(x, w, b, s, p, op, dtype)
            np.testing.assert_array_equal(y, ref, err_msg="%s %s" % ((L, k, s, p, op, ci, co), desc))
    for (H, W, ky, kx, sy, sx, py, px, opy, opx) in GRID_2D:
        for (ci, co) in chans[:2]:
            x, w, b = _int_inputs(rng, (1, ci, H, W), (ci, co, ky, kx), co, mag)
            y, desc = run_plan(x, w, b, (sy, sx), (py, px), (opy, opx), dtype, path=PATHS[path])
            ref = reference(x, w, b, (sy, sx), (py, px), (opy, opx), dtype)
            np.testing.assert_array_equal(y, ref, err_msg=desc)


@pytest.mark.parametrize("split_k", [1, 2, 3, 5])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tiles_and_split_k_bit_exact(dtype, split_k):
    """M over two row tiles with a ragged end, N over several column tiles with a ragged tail,
    K over several slices and taps, forced split-K."""
    rng = np.random.default_rng(5 + split_k)
    mag = 2 if dtype == "f32" else 1
    cases_1d = [(2, 150, 37, 300, 8, 4, 2, 0), (1, 64, 40, 257, 16, 8, 4, 3)]
    for (B, ci, co, L, k, s, p, op) in cases_1d:
        if dtype == "bf16":
            ci = min(ci, 60)
        x, w, b = _int_inputs(rng, (B, ci, L), (ci, co, k), co, mag)
        y, desc = run_plan(x, w, b, s, p, op, dtype, path=ctr.CTR_PATH_POLYPHASE, split_k=split_k)
        np.testing.assert_array_equal(y, reference(x, w, b, s, p, op, dtype), err_msg=desc)
    x, w, b = _int_inputs(rng, (2, 40, 19, 23), (40, 20, 4, 4), 20, mag)
    y, desc = run_plan(x, w, b, (2, 2), (1, 1), (0, 1), dtype, path=ctr.CTR_PATH_POLYPHASE,
                       split_k=split_k)
    np.testing.assert_array_equal(y, reference(x, w, b, (2, 2), (1, 1), (0, 1), dtype), err_msg=desc)
    x, w, b = _int_inputs(rng, (2, 48, 70), (48, 30, 7), 30, mag)
    y, desc = run_plan(x, w, b, 3, 2, 1, dtype, path=ctr.CTR_PATH_COL2IM, split_k=split_k)
    np.testing.assert_array_equal(y, reference(x, w, b, 3, 2, 1, dtype), err_msg=desc)


@pytest.mark.parametrize("block_n", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_every_tile_width_bit_exact(dtype, block_n):
    """Each phase-row tile width of the GEMM (its own kernel instantiation: slice width,
    stage count, TMEM accumulators, and at 256 columns in fp32 the TMEM-resident group
    sums) with enough K for several accumulation groups, with and without split-K."""
    rng = np.random.default_rng(11 + block_n)
    mag = 2 if dtype == "f32" else 1
    # K = 2 taps x 300 channels: 20 fp32 slices of 128 bytes (three groups) or 10 bf16 ones.
    cases = [(2, 300, 70, 150, 8, 4, 2, 0), (1, 96, 33, 131, 16, 8, 4, 3)]
    for (B, ci, co, L, k, s, p, op) in cases:
        if dtype == "bf16":
            ci = min(ci, 120)
        x, w, b = _int_inputs(rng, (B, ci, L), (ci, co, k), co, mag)
        ref = reference(x, w, b, s, p, op, dtype)
        for split_k in (1, 2):
            y, desc = run_plan(x, w, b, s, p, op, dtype, path=ctr.CTR_PATH_POLYPHASE,
                               split_k=split_k, block_n=block_n)
            assert "BN %d," % block_n in desc, desc
            np.testing.assert_array_equal(y, ref, err_msg=desc)
    x, w, b = _int_inputs(rng, (1, 64, 21, 18), (64, 40, 4, 4), 40, mag)
    y, desc = run_plan(x, w, b, (2, 2), (1, 1), (1, 0), dtype, path=ctr.CTR_PATH_POLYPHASE,
                       block_n=block_n)
    np.testing.assert_array_equal(y, reference(x, w, b, (2, 2), (1, 1), (1, 0), dtype), err_msg=desc)


@pytest.mark.parametrize("block_n", [64, 128, 256])
def test_all_positive_long_k_within_tolerance(block_n):
    """The worst case for the tensor core's truncating fp32 accumulation: same-sign products
    over K = 4096 (2 taps x 2048 channels), where the drift is systematic instead of
    averaging out.  The grouped accumulation keeps fp32 I/O within rel_l2 1e-5 at every
    tile width (register sums at 64, TMEM sums at 128 and 256)."""
    rng = np.random.default_rng(47)
    x = rng.uniform(0.0, 1.0, (1, 2048, 300)).astype(np.float32)
    w = rng.uniform(0.0, 1.0, (2048, 64, 16)).astype(np.float32)
    b = rng.uniform(0.0, 1.0, 64).astype(np.float32)
    y, desc = run_plan(x, w, b, 8, 4, 0, "f32", path=ctr.CTR_PATH_POLYPHASE, block_n=block_n)
    err = oracle.rel_l2(y, reference(x, w, b, 8, 4, 0, "f32"))
    assert err <= TOL["f32"], "rel_l2 %.3g %s" % (err, desc)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_random_within_tolerance(path, dtype):
    rng = np.random.default_rng(3)
    cases = [((2, 96, 130), (96, 48, 8), 4, 2, 1), ((1, 33, 77), (33, 70, 3), 2, 1, 1),
             ((1, 64, 30, 20), (64, 24, 4, 4), (2, 2), (1, 1), (1, 0))]
    for (xs, ws, s, p, op) in cases:
        x = workloads._cast(rng.standard_normal(xs), dtype)
        w = workloads._cast(rng.uniform(-0.1, 0.1, ws), dtype)
        b = workloads._cast(rng.normal(0, 0.1, ws[1]), dtype)
        y, desc = run_plan(x, w, b, s, p, op, dtype, path=PATHS[path])
        ref = reference(x, w, b, s, p, op, dtype)
        err = oracle.rel_l2(y, ref)
        assert err <= TOL[dtype], "rel_l2 %.3g %s" % (err, desc)


def _layer_args(layer):
    return layer.stride, layer.padding, layer.output_padding


@pytest.mark.parametrize("name", ["tiny_1d_f32", "codec_upsampler_f32", "istft_f32", "decoder_2d_f32"])
def test_workload_full_size(name):
    (li,) = workloads.make_workload(name)
    layer = li.layer
    s, p, op = _layer_args(layer)
    y, desc = run_plan(li.x, li.w, li.bias, s, p, op, layer.dtype)
    ref = oracle.conv_transpose(li.x, li.w, li.bias, s, p, op)
    err = oracle.rel_l2(y, ref)
    print("%s rel_l2 %.3g %s" % (name, err, desc))
    assert err <= TOL[layer.dtype], "rel_l2 %.3g %s" % (err, desc)


def test_vocoder_stack_full_size():
    """Per stage with the same bf16 input on both sides, and the whole chain."""
    stages = workloads.make_workload("vocoder_stack_bf16")
    x_gpu = stages[0].x
    x_ref = stages[0].x.astype(np.float64)
    for i, li in enumerate(stages):
        layer = li.layer
        s, p, op = _layer_args(layer)
        y, desc = run_plan(x_gpu, li.w, li.bias, s, p, op, "bf16", slope=layer.act_slope)
        ref_same_input = reference(x_gpu, li.w, li.bias, s, p, op, "bf16", slope=layer.act_slope)
        err = oracle.rel_l2(y, ref_same_input)
        assert err <= TOL["bf16"], "stage %d rel_l2 %.3g %s" % (i, err, desc)
        x_ref = reference(x_ref, li.w, li.bias, s, p, op, "bf16", slope=layer.act_slope)
        x_gpu = y.astype(np.float32)
    err = oracle.rel_l2(x_gpu, x_ref)
    print("stack rel_l2 %.3g" % err)
    assert err <= TOL["bf16"]


def test_istft_sinusoid_full_size():
    """ConvTranspose with the Hann-windowed inverse real-DFT basis (N = 4096, hop 1024,
    343 frames, batch 4) on the closed-form spectra of a sinusoid returns 2 * the sinusoid
    where four frames overlap."""
    N, hop, frames, batch, f0 = 4096, 1024, 343, 4, 37
    X = workloads.istft_sinusoid_frames(N, hop, frames, batch, f0, 0.5, 0.25).astype(np.float32)
    w = workloads.istft_basis(N).astype(np.float32)
    y, desc = run_plan(X, w, None, hop, 0, 0, "f32")
    sig = workloads.istft_sinusoid_signal(N, y.shape[-1], batch, f0, 0.5, 0.25)
    lo, hi = 3 * hop, frames * hop
    err = oracle.rel_l2(y[:, 0, lo:hi], 2.0 * sig[:, lo:hi])
    print("istft sinusoid rel_l2 %.3g %s" % (err, desc))
    assert err <= 1e-5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_edge_cases(path, dtype):
    rng = np.random.default_rng(9)
    mag = 1
    cases = [
        ((1, 20, 0), (20, 40, 4), 2, 0, 0),       # empty input: bias only
        ((2, 20, 0), (20, 40, 3), 2, 0, 1),       # empty input, kernel not a multiple of s
        ((1, 20, 1), (20, 40, 4), 2, 1, 0),       # one input step
        ((1, 20, 9), (20, 40, 2), 2, 0, 0),       # m = 1
        ((1, 20, 9), (20, 40, 6), 2, 1, 1),       # m = 3, op = p
        ((1, 20, 9), (20, 40, 4), 2, 0, 1),       # op > p
        ((1, 20, 6), (20, 40, 20), 5, 3, 4),      # op > p, s = 5
    ]
    for s in (2, 4, 5, 6):
        cases.append(((1, 20, 10), (20, 40, 2 * s), s, s // 2, 0))
    for n, (xs, ws, s, p, op) in enumerate(cases):
        x, w, b = _int_inputs(rng, xs, ws, ws[1], mag, with_bias=n % 2 == 0)
        y, desc = run_plan(x, w, b, s, p, op, dtype, path=PATHS[path])
        np.testing.assert_array_equal(y, reference(x, w, b, s, p, op, dtype), err_msg=desc)
    # 2-D: pH != pW and p = 0, unequal strides
    for (xs, ws, s, p, op) in [((1, 20, 5, 6), (20, 24, 4, 4), (2, 2), (1, 0), (0, 1)),
                               ((1, 20, 5, 6), (20, 24, 4, 4), (2, 2), (0, 0), (0, 0)),
                               ((1, 20, 4, 5), (20, 24, 4, 6), (2, 3), (1, 2), (1, 2))]:
        x, w, b = _int_inputs(rng, xs, ws, ws[1], mag)
        y, desc = run_plan(x, w, b, s, p, op, dtype, path=PATHS[path])
        np.testing.assert_array_equal(y, reference(x, w, b, s, p, op, dtype), err_msg=desc)


@pytest.mark.parametrize("path", sorted(PATHS))
def test_cancelling_taps_bf16(path):
    """Pairs of taps that cancel exactly: partial sums must not be rounded to bf16 before
    the later tap cancels them ("[WebGPU] optimizations for audio models", review commit:
    the float16 regression for cancelling ConvTranspose taps)."""
    C_in, C_out, L, k, s = 32, 64, 40, 4, 2
    rng = np.random.default_rng(4)
    x = np.ones((1, C_in, L), np.float32)
    w = np.zeros((C_in, C_out, k), np.float32)
    big = workloads.to_bf16_values(rng.uniform(100, 200, (C_in // 2, C_out)).astype(np.float32))
    w[0::2, :, 0] = big
    w[1::2, :, 0] = -big
    w[:, :, 1] = workloads.to_bf16_values(rng.uniform(-0.01, 0.01, (C_in, C_out)).astype(np.float32))
    y, desc = run_plan(x, w, None, s, 1, 0, "bf16", path=PATHS[path])
    ref = reference(x, w, None, s, 1, 0, "bf16")
    assert oracle.rel_l2(y, ref) <= 1e-2, desc
    assert np.max(np.abs(y - ref)) <= 2e-3


def test_leaky_relu_fused_bit_exact():
    rng = np.random.default_rng(8)
    x, w, b = _int_inputs(rng, (1, 64, 50), (64, 32, 16), 32, 2)
    for dtype in ("f32", "bf16"):
        xx, ww, bb = (x, w, b) if dtype == "f32" else (np.sign(x), np.sign(w), np.sign(b))
        y, desc = run_plan(xx, ww, bb, 8, 4, 0, dtype, slope=0.125)
        np.testing.assert_array_equal(y, reference(xx, ww, bb, 8, 4, 0, dtype, slope=0.125),
                                      err_msg=desc)


def test_deterministic_repeat():
    li = workloads.make_workload("codec_upsampler_f32")[0]
    a, _ = run_plan(li.x, li.w, li.bias, 8, 4, 0, "f32", split_k=3)
    b2, _ = run_plan(li.x, li.w, li.bias, 8, 4, 0, "f32", split_k=3)
    np.testing.assert_array_equal(a, b2)


def test_error_statuses():
    h = ctr.ctr_plan_create(1, 1, 64, 64, [100], [4], [2], [1], [0], ctr.CTR_F32)
    try:
        x = torch.randn(1, 64, 100, device="cuda")
        w = torch.randn(64, 64, 4, device="cuda")
        wp = torch.empty(ctr.ctr_packed_weight_bytes(h), dtype=torch.uint8, device="cuda")
        y = torch.empty(1, 64, 200, device="cuda")
        buf = torch.empty(64 * 200 + 1, device="cuda")
        y_mis = buf[1:].view(1, 64, 200)
        st = ctr._stream_ptr(None)
        with pytest.raises(ctr.CtrError) as e:
            ctr.ctr_forward(h, ctr._ptr(x), ctr._ptr(wp), None, ctr._ptr(y), st)
        assert e.value.status == ctr.CTR_ERR_NOT_PREPARED
        ctr.ctr_prepack_weight(h, ctr._ptr(w), ctr._ptr(wp), st)
        with pytest.raises(ctr.CtrError) as e:
            ctr.ctr_forward(h, ctr._ptr(x), ctr._ptr(wp), None, ctr._ptr(y), st)
        assert e.value.status == ctr.CTR_ERR_NO_WORKSPACE
        ws = torch.empty(ctr.ctr_workspace_bytes(h), dtype=torch.uint8, device="cuda")
        ctr.ctr_plan_bind_workspace(h, ctr._ptr(ws), ws.numel())
        with pytest.raises(ctr.CtrError) as e:
            ctr.ctr_forward(h, ctr._ptr(x), ctr._ptr(wp), None, ctr._ptr(y_mis), st)
        assert e.value.status == ctr.CTR_ERR_MISALIGNED
        ctr.ctr_forward(h, ctr._ptr(x), ctr._ptr(wp), None, ctr._ptr(y), st)
        ctr.ctr_plan_check(h, st)
        ref = oracle.conv_transpose(x.cpu().numpy(), w.cpu().numpy(), None, 2, 1, 0)
        assert oracle.rel_l2(y.cpu().numpy(), ref) <= 1e-5
    finally:
        torch.cuda.synchronize()
        ctr.ctr_plan_destroy(h)


def test_bounded_wait_timeout_reports_and_recovers():
    """A 0 ns wait limit makes the tensor-core kernel's waits give up on a healthy run: the
    kernel records the timeout, drains its copies and MMAs, frees TMEM and returns;
    ctr_plan_check reports CTR_ERR_DEVICE_TIMEOUT and the context stays usable."""
    li = workloads.make_workload("codec_upsampler_f32")[0]
    plan = ctr.Plan(1, 512, 256, (2000,), (16,), 8, 4, 0)
    try:
        plan.prepack(to_dev(li.w, "f32"))
        x = to_dev(li.x, "f32")
        b = to_dev(li.bias, "f32")
        plan.set_wait_limit_ns(0)
        plan.forward(x, b)
        with pytest.raises(ctr.CtrError) as e:
            plan.check()
        assert e.value.status == ctr.CTR_ERR_DEVICE_TIMEOUT
        plan.set_wait_limit_ns(4_000_000_000)
        y = plan.forward(x, b)
        plan.check()
        ref = oracle.conv_transpose(li.x, li.w, li.bias, 8, 4, 0)
        assert oracle.rel_l2(y.cpu().numpy(), ref) <= 1e-5
    finally:
        plan.close()


def test_launches_are_counted():
    before = ctr.ctr_launch_count()
    li = workloads.make_workload("tiny_1d_f32")[0]
    run_plan(li.x, li.w, li.bias, 2, 1, 0, "f32")
    assert ctr.ctr_launch_count() >= before + 2   # weight copy + gather
