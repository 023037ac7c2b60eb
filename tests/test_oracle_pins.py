"""The CPU oracle against its pins (no GPU).

Runs every check of ``tests/pins.py`` on the oracle, then plants plausible mistakes in copies
of the oracle's C source (a dropped bias, a wrong padding sign, a transposed weight operand,
flipped taps, a dropped tap term, a dropped partial sum, a dropped dilation, an off-by-one tap
bound, a back pad taken as the front pad) and shows that each one fails at
least one pin.  The planted copies are compiled into a temporary directory; the committed
oracle is never modified.
"""
import contextlib
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import pins
import workloads


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.conv_transpose)


def test_torch_grid_1d_full():
    """The full 1-D grid: s 1..4, k 1..7, p 0..k-1, op 0..s-1, L_in 1..5."""
    pins.pin_torch_f64_1d(oracle.conv_transpose, full=True)


def test_output_size_clean_upscale():
    """(H - 1)s - 2p + k + op == sH for the clean-upscale geometries of the depthwise
    decomposition ("[XNNPACK] Lower dense transposed convs as one polyphase conv + depth to
    space", DecomposeDepthwiseConvTransposePass commit): k = 2s with p = s/2, and k = s."""
    for H in (1, 7, 128):
        for s in (2, 4, 8):
            assert oracle.output_size(H, 2 * s, s, s // 2, 0) == s * H
            assert oracle.output_size(H, s, s, 0, 0) == s * H
        assert oracle.output_size(H, 3, 2, 1, 1) == 2 * H


def test_output_size_matches_torch_shapes():
    import torch
    import torch.nn.functional as F
    for (L, k, s, p, op) in pins.grid_1d(full=True):
        y = F.conv_transpose1d(torch.zeros(1, 1, L, dtype=torch.float64),
                               torch.zeros(1, 1, k, dtype=torch.float64),
                               stride=s, padding=p, output_padding=op)
        assert y.shape[-1] == oracle.output_size(L, k, s, p, op)


def test_output_size_dilated_matches_torch_shapes():
    """(L_in - 1)s + (k - 1)d + 1 + op - 2p against torch's output shapes with dilation, and
    the front/back form against the symmetric one."""
    import torch
    import torch.nn.functional as F
    for (L, k, s, d, p, op) in pins.grid_dilated_1d():
        y = F.conv_transpose1d(torch.zeros(1, 1, L, dtype=torch.float64),
                               torch.zeros(1, 1, k, dtype=torch.float64),
                               stride=s, padding=p, output_padding=op, dilation=d)
        assert y.shape[-1] == oracle.output_size(L, k, s, p, op, d)
        assert oracle.output_size(L, k, s, p, op, d, p) == oracle.output_size(L, k, s, p, op, d)
    assert oracle.output_size(2, 3, 2, 1, 1, 2, 0) == 7
    assert oracle.output_size(2, 3, 2, 0, 0, 2, 3) == 4


def test_streaming_chunks_with_carried_frames_equal_whole_input():
    """The streaming reading: with the last m - 1 frames of the previous chunk (zeros at the
    start) put in front of each chunk, the s*L samples at s*(m - 1) .. s*(m - 1 + L) of that
    extended chunk's unpadded ConvTranspose are exactly samples s*c*L .. s*(c + 1)*L of the
    whole input's.  Chunks shorter than m - 1 take older frames along."""
    rng = np.random.default_rng(17)
    for (C_in, C_out, k, s, L, nchunks) in ((3, 2, 16, 8, 5, 4), (2, 3, 6, 2, 1, 6),
                                            (2, 2, 5, 2, 3, 3), (1, 2, 4, 4, 2, 3)):
        m = -(-k // s)
        x = rng.standard_normal((2, C_in, L * nchunks))
        w = rng.standard_normal((C_in, C_out, k))
        b = rng.standard_normal(C_out)
        whole = oracle.conv_transpose(x, w, b, s, 0, 0)
        carried = np.zeros((2, C_in, m - 1))
        for c in range(nchunks):
            chunk = x[:, :, c * L:(c + 1) * L]
            ext = np.concatenate([carried, chunk], axis=2)
            y = oracle.conv_transpose(ext, w, b, s, 0, 0)[:, :, s * (m - 1):s * (m - 1 + L)]
            np.testing.assert_allclose(y, whole[:, :, s * c * L:s * (c + 1) * L], rtol=1e-12,
                                       atol=1e-12)
            carried = ext[:, :, ext.shape[2] - (m - 1):]


def test_landed_count_long_input():
    """"[WebGPU] optimizations for audio models", review of the chunked col2im: X =
    [1, 16, 262144], W = [16, 1, 4096], stride 1 has about 1e9 contributions after the GEMM
    contracts C_in: every one of the 262144 * 4096 (input step, tap) pairs lands."""
    n = oracle.landed_pairs((262144,), 4096, 1, 0, 0)
    assert n == 262144 * 4096
    assert abs(n - 1.0e9) / 1.0e9 < 0.08
    # With padding some taps fall outside the output and do not count.
    assert oracle.landed_pairs((4,), 4, 2, 1, 0) == 4 * 4 - 2


def test_empty_input_gives_bias():
    w = np.ones((2, 3, 4))
    b = np.array([1.5, -2.0, 0.0])
    y = oracle.conv_transpose(np.zeros((2, 2, 0)), w, b, 2, 0, 0)
    assert y.shape == (2, 3, 2)
    np.testing.assert_array_equal(y, np.broadcast_to(b[None, :, None], y.shape))
    y0 = oracle.conv_transpose(np.zeros((1, 2, 0)), w, None, 2, 0, 1)
    np.testing.assert_array_equal(y0, np.zeros((1, 3, 3)))


def test_invalid_geometry_rejected():
    with pytest.raises(ValueError):
        oracle.conv_transpose(np.zeros((1, 1, 1)), np.zeros((1, 1, 2)), None, 1, 1, 0)


def test_round_bf16_against_torch():
    import torch
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [0.0, -0.0, 1.0, 3.0e38, -3.4e38, 1e-40]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(v.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    # Ties go to even: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7.
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    # Rounding straight from double: just above a tie goes up.
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 1.0 + 2.0 ** -7


def test_generator_bf16_matches_torch():
    import torch
    v = np.random.default_rng(7).standard_normal(10000).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(workloads.to_bf16_values(v), ref)


def test_leaky_relu_and_rel_l2():
    y = np.array([-2.0, -0.5, 0.0, 3.0])
    np.testing.assert_array_equal(oracle.leaky_relu(y, 0.1), [-0.2, -0.05, 0.0, 3.0])
    assert oracle.rel_l2([3.0, 4.0], [3.0, 4.0]) == 0.0
    assert abs(oracle.rel_l2([3.0, 4.0 + 0.5], [3.0, 4.0]) - 0.1) < 1e-15


def test_workload_shapes():
    """Output sizes, useful-MAC counts and compulsory bytes of the workloads."""
    L = workloads.WORKLOADS
    assert L["tiny_1d_f32"][0].out_sp == (128,)
    assert L["codec_upsampler_f32"][0].out_sp == (16000,)
    assert L["istft_f32"][0].out_sp == (354304,)
    assert L["decoder_2d_f32"][0].out_sp == (256, 256)
    assert [l.out_sp for l in L["vocoder_stack_bf16"]] == [(8192,), (65536,), (131072,), (262144,)]
    assert 2 * L["codec_upsampler_f32"][0].useful_macs == 8388608000
    assert 2 * L["istft_f32"][0].useful_macs == 46059159552
    dw = L["depthwise_2d_bf16"][0]
    assert dw.out_sp == (256, 256)
    assert 2 * dw.useful_macs == 2 * 4 * 256 * 16 * 128 * 128     # one channel per group
    assert dw.compulsory_bytes == 2 * (4 * 256 * 128 * 128 + 256 * 16 + 256 + 4 * 256 * 256 * 256)
    assert workloads.make_layer_inputs(dw, 1).w.shape == (256, 1, 4, 4)


# ---------------------------------------------------------------- planted mistakes

MUTANTS = {
    "dropped_bias": ("const double bv = bias ? bias[oc] : 0.0;", "const double bv = 0.0;"),
    "padding_sign": ("const int64_t ox0 = ix * sw - pw;", "const int64_t ox0 = ix * sw + pw;"),
    "transposed_weight": ("const double *wp = w + (ic * cout_g + ocl) * ntap;",
                          "const double *wp = w + (ocl * C_in + ic) * ntap;"),
    "group_input_channels": ("for (int64_t ic = g * cin_g; ic < (g + 1) * cin_g; ++ic) {",
                             "for (int64_t ic = 0; ic < cin_g; ++ic) {"),
    "flipped_taps": ("arow[ox0 + tx * dw] += xv * wrow[tx];",
                     "arow[ox0 + tx * dw] += xv * wrow[kw - 1 - tx];"),
    "dropped_tap_term_y": ("const int64_t oy = iy * sh - ph + ty * dh;",
                           "const int64_t oy = iy * sh - ph;"),
    "dropped_dilation_y": ("const int64_t oy = iy * sh - ph + ty * dh;",
                           "const int64_t oy = iy * sh - ph + ty;"),
    "tap_bound_floor_x": ("int64_t tx_hi = ox0 < Wo ? (Wo - ox0 + dw - 1) / dw : 0;",
                          "int64_t tx_hi = ox0 < Wo ? (Wo - ox0) / dw : 0;"),
    "back_pad_as_front_pad": ("return (L_in - 1) * s + (k - 1) * d + 1 + op - pb - pe;",
                              "return (L_in - 1) * s + (k - 1) * d + 1 + op - 2 * pb;"),
    "undilated_output_size": ("return (L_in - 1) * s + (k - 1) * d + 1 + op - pb - pe;",
                              "return (L_in - 1) * s + k + op - pb - pe;"),
    "dropped_partial_sum": ("for (int64_t c = 0; c < nchunk; ++c) {",
                            "for (int64_t c = 0; c + 1 < nchunk || c == 0; ++c) {"),
}


@contextlib.contextmanager
def _oracle_lib(path):
    lib = ctypes.CDLL(path)
    real = oracle._load()
    for name in ("ctr_oracle_conv_transpose", "ctr_oracle_conv_transpose_groups",
                 "ctr_oracle_conv_transpose_ex", "ctr_oracle_output_size",
                 "ctr_oracle_output_size_ex", "ctr_oracle_landed_pairs"):
        getattr(lib, name).restype = getattr(real, name).restype
        getattr(lib, name).argtypes = getattr(real, name).argtypes
    saved = oracle._lib
    oracle._lib = lib
    try:
        yield
    finally:
        oracle._lib = saved


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(mutant):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) == 1, "mutation anchor not found: " + old
    tmp = tempfile.mkdtemp()
    try:
        cpath = os.path.join(tmp, "m.c")
        lpath = os.path.join(tmp, "libm.so")
        with open(cpath, "w") as f:
            f.write(src.replace(old, new))
        subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", cpath, "-o", lpath],
                       check=True)
        failed = []
        with _oracle_lib(lpath):
            for pin in pins.ALL_PINS:
                try:
                    pin(oracle.conv_transpose)
                except (AssertionError, ValueError):
                    failed.append(pin.__name__)
        assert failed, "planted mistake %s passed every pin" % mutant
    finally:
        shutil.rmtree(tmp)


def test_round_f16_hand_cases():
    """Round-to-nearest-even into binary16 at the places a plausible mistake shows: ties at
    1 (even mantissa stays, odd rounds up), the overflow threshold (65520 is the tie between
    65504 and 2**16, whose mantissa is even, so it overflows to inf), the subnormal spacing
    2**-24 and its ties, signs, and values that pass through."""
    cases = [
        (1.0 + 2.0 ** -11, 1.0),                      # tie, 1.0 has an even mantissa
        (1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -9),      # tie, 1 + 2**-10 is odd: round up
        (1.0 + 2.0 ** -11 + 2.0 ** -40, 1.0 + 2.0 ** -10),   # just above the tie
        (2048.0 + 1.0, 2048.0), (2048.0 + 3.0, 2052.0),      # spacing 2 above 2048
        (65504.0, 65504.0), (65519.99, 65504.0), (65520.0, np.inf), (-65520.0, -np.inf),
        (2.0 ** -24, 2.0 ** -24), (2.0 ** -25, 0.0), (3 * 2.0 ** -25, 2.0 ** -23),
        (2.0 ** -14 - 2.0 ** -25, 2.0 ** -14),              # top subnormal tie rounds to normal
        (-0.1, -0.0999755859375), (np.inf, np.inf), (-3.0, -3.0),
    ]
    for x, want in cases:
        got = float(oracle.round_f16(x))
        assert got == want, (x, got, want)
    assert np.isnan(oracle.round_f16(np.nan))


def test_round_f16_matches_numpy_conversion():
    """numpy's float64 -> float16 conversion is an independent, correctly rounded
    implementation; the two agree on doubles over the whole binary16 range."""
    rng = np.random.default_rng(23)
    x = rng.standard_normal(200000) * np.exp2(rng.integers(-30, 17, 200000).astype(np.float64))
    got = oracle.round_f16(x)
    ref = x.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(got, ref)
