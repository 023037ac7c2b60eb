"""Seeded random geometries on every path the library chooses, against the oracle.

Each case draws a 1-D or 2-D ConvTranspose (channels, lengths, kernel, stride, padding,
output padding below the stride, sometimes separate back pads or dilation), an I/O type
(fp32, bf16, fp16), a memory layout (NCHW or channels-last), a fused LeakyReLU or none, a
bias or none, and small-integer inputs, for which every product and partial sum is exact:
whatever path and tiling the library picks, the result must equal the oracle's
ConvTranspose rounded once to the I/O type, bit for bit.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transposed_convolution_gb300 as ctr  # noqa: E402
from gpu_helpers import reference, run_plan  # noqa: E402


def _case(rng, large=False):
    ndim = 1 if rng.random() < 0.6 else 2
    s = [int(rng.integers(1, 5)) for _ in range(ndim)]
    k = [int(rng.integers(1, 9 if ndim == 1 or not large else 6)) for _ in range(ndim)]
    d = [1] * ndim
    if rng.random() < 0.15:
        d = [int(rng.integers(1, 3)) for _ in range(ndim)]
    p = [int(rng.integers(0, k[i])) for i in range(ndim)]
    pe = list(p)
    if rng.random() < 0.2:
        pe = [int(rng.integers(0, k[i])) for i in range(ndim)]
    op = [int(rng.integers(0, s[i])) for i in range(ndim)]
    if large:   # several position tiles and row tiles, ragged
        L = [int(rng.integers(100, 700 if ndim == 1 else 26)) if ndim == 1 else
             int(rng.integers(8, 26)) for _ in range(ndim)]
    else:
        L = [int(rng.integers(1, 90 if ndim == 1 else 14)) for _ in range(ndim)]
    # keep the output non-empty
    for i in range(ndim):
        while (L[i] - 1) * s[i] + (k[i] - 1) * d[i] + 1 + op[i] - p[i] - pe[i] < 1:
            L[i] += 1
    ci = int(rng.choice([1, 3, 16, 24, 40, 64, 96] + ([130, 160] if large else [])))
    co = int(rng.choice([1, 5, 8, 17, 32, 64, 70] + ([100, 150] if large else [])))
    B = int(rng.integers(1, 3))
    dtype = str(rng.choice(["f32", "bf16", "f16"]))
    layout = "nhwc" if rng.random() < 0.2 else "nchw"
    slope = float(rng.choice([0.25, 0.5])) if rng.random() < 0.3 else None
    with_bias = rng.random() < 0.8
    return ndim, B, ci, co, L, k, s, p, pe, op, d, dtype, layout, slope, with_bias


@pytest.mark.parametrize("seed", range(16))
def test_random_geometries_bit_exact(seed):
    rng = np.random.default_rng(9000 + seed)
    ran = 0
    for _ in range(30):
        (ndim, B, ci, co, L, k, s, p, pe, op, d, dtype, layout, slope,
         with_bias) = _case(rng)
        mag = 2 if dtype == "f32" else 1
        x = rng.integers(-mag, mag + 1, (B, ci) + tuple(L)).astype(np.float32)
        w = rng.integers(-mag, mag + 1, (ci, co) + tuple(k)).astype(np.float32)
        b = rng.integers(-mag, mag + 1, (co,)).astype(np.float32) if with_bias else None
        try:
            y, desc = run_plan(x, w, b, tuple(s), tuple(p), tuple(op), dtype, slope=slope,
                               dilation=tuple(d), padding_end=tuple(pe), layout=layout)
        except ctr.CtrError as ex:
            # a combination the library documents as unsupported (a layout or type that a
            # chosen kernel does not take) must say so, not compute something else
            assert ex.status == ctr.CTR_ERR_UNSUPPORTED, ex
            continue
        ref = reference(x, w, b, tuple(s), tuple(p), tuple(op), dtype, slope=slope,
                        dilation=tuple(d), padding_end=tuple(pe))
        np.testing.assert_array_equal(
            y, ref, err_msg="%s %s" % ((ndim, B, ci, co, L, k, s, p, pe, op, d, dtype,
                                        layout, slope, with_bias), desc))
        ran += 1
    assert ran >= 20


@pytest.mark.parametrize("seed", range(8))
def test_random_forced_paths_bit_exact(seed):
    """The same random geometries forced onto each tensor-core path and the gather path,
    with random split-K factors, tile widths and phase origins: every combination the
    library accepts must equal the oracle bit for bit; one it refuses must say
    CTR_ERR_UNSUPPORTED."""
    rng = np.random.default_rng(9500 + seed)
    paths = [ctr.CTR_PATH_POLYPHASE, ctr.CTR_PATH_COL2IM, ctr.CTR_PATH_GATHER]
    origins = [ctr.CTR_PHASE_AUTO, ctr.CTR_PHASE_UNPADDED, ctr.CTR_PHASE_OUTPUT]
    ran = 0
    for _ in range(30):
        (ndim, B, ci, co, L, k, s, p, pe, op, d, dtype, layout, slope,
         with_bias) = _case(rng)
        path = paths[int(rng.integers(0, 3))]
        split = int(rng.choice([0, 1, 2, 3]))
        block_n = int(rng.choice([0, 64, 128, 256]))
        origin = origins[int(rng.integers(0, 3))]
        mag = 2 if dtype == "f32" else 1
        x = rng.integers(-mag, mag + 1, (B, ci) + tuple(L)).astype(np.float32)
        w = rng.integers(-mag, mag + 1, (ci, co) + tuple(k)).astype(np.float32)
        b = rng.integers(-mag, mag + 1, (co,)).astype(np.float32) if with_bias else None
        try:
            y, desc = run_plan(x, w, b, tuple(s), tuple(p), tuple(op), dtype, slope=slope,
                               dilation=tuple(d), padding_end=tuple(pe), layout=layout,
                               path=path, split_k=split if path != ctr.CTR_PATH_GATHER else 0,
                               block_n=block_n if path != ctr.CTR_PATH_GATHER else 0,
                               phase_origin=origin if path == ctr.CTR_PATH_POLYPHASE
                               else ctr.CTR_PHASE_AUTO)
        except ctr.CtrError as ex:
            assert ex.status == ctr.CTR_ERR_UNSUPPORTED, (ex, path, split, block_n, origin)
            continue
        ref = reference(x, w, b, tuple(s), tuple(p), tuple(op), dtype, slope=slope,
                        dilation=tuple(d), padding_end=tuple(pe))
        np.testing.assert_array_equal(
            y, ref, err_msg="%s %s" % ((ndim, B, ci, co, L, k, s, p, pe, op, d, dtype, layout,
                                        slope, with_bias, path, split, block_n, origin), desc))
        ran += 1
    assert ran >= 15


@pytest.mark.parametrize("seed", range(4))
def test_random_large_geometries_bit_exact(seed):
    """Longer inputs and more channels: several position and row tiles with ragged tails,
    split-K and the wider tiles, on whatever path the library picks."""
    rng = np.random.default_rng(9800 + seed)
    ran = 0
    for _ in range(12):
        (ndim, B, ci, co, L, k, s, p, pe, op, d, dtype, layout, slope,
         with_bias) = _case(rng, large=True)
        mag = 2 if dtype == "f32" else 1
        x = rng.integers(-mag, mag + 1, (B, ci) + tuple(L)).astype(np.float32)
        w = rng.integers(-mag, mag + 1, (ci, co) + tuple(k)).astype(np.float32)
        b = rng.integers(-mag, mag + 1, (co,)).astype(np.float32) if with_bias else None
        try:
            y, desc = run_plan(x, w, b, tuple(s), tuple(p), tuple(op), dtype, slope=slope,
                               dilation=tuple(d), padding_end=tuple(pe), layout=layout)
        except ctr.CtrError as ex:
            assert ex.status == ctr.CTR_ERR_UNSUPPORTED, ex
            continue
        ref = reference(x, w, b, tuple(s), tuple(p), tuple(op), dtype, slope=slope,
                        dilation=tuple(d), padding_end=tuple(pe))
        np.testing.assert_array_equal(
            y, ref, err_msg="%s %s" % ((ndim, B, ci, co, L, k, s, p, pe, op, d, dtype,
                                        layout, slope, with_bias), desc))
        ran += 1
    assert ran >= 8
