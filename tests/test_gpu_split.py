"""fp32 I/O on the tensor cores: the accuracy of the operand split, output by output.

The library takes every fp32 product x*w as hi_x*hi_w in tf32 (hi = v rounded to tf32)
plus the two cross products hi_x*lo_w + lo_x*hi_w in bf16 (lo = v - hi), and drops
lo_x*lo_w.  Each rounded or dropped term is below about 2^-17 of |x*w|: bf16 keeps 8
significant bits of cross terms below 2^-11 of the product, and lo_x*lo_w is below 2^-22.
With 8 nonzero K elements per output (k = s, or k = 2s with half the channels) the fp32
accumulation adds little more.  So every output must lie within 2^-16 * sum |x*w| of the
exact sum.  A dropped or mispaired cross product leaves an error near 2^-12 of that sum,
and so does a single tf32 product: the test shows that such products would fail.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import transposed_convolution_gb300 as ctr  # noqa: E402
from gpu_helpers import run_plan  # noqa: E402

BOUND = 2.0 ** -16

# (B, C_in, C_out, spatial L, k, s): 8 nonzero K elements per output in each case.
CASES = [
    (2, 8, 64, (700,), (4,), (4,)),          # one tap, 8 channels
    (1, 4, 48, (900,), (8,), (4,)),          # two taps, 4 channels
    (2, 8, 40, (30, 37), (2, 2), (2, 2)),    # 2-D, one tap per phase
]


def _tf32(a):
    """fp32 -> tf32, to nearest with ties away from zero (10 explicit mantissa bits)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x1000) & 0xFFFFE000) & 0xFFFFFFFF
    return u.astype(np.uint32).view(np.float32)


def _case_inputs(rng, B, ci, co, L, k):
    x = rng.uniform(-1.0, 1.0, (B, ci) + L).astype(np.float32)
    w = rng.uniform(-1.0, 1.0, (ci, co) + k).astype(np.float32)
    return x, w


@pytest.mark.parametrize("block_n", [64, 128, 256])
@pytest.mark.parametrize("path", ["polyphase", "col2im"])
def test_split_products_within_bound(path, block_n):
    rng = np.random.default_rng(77 + block_n)
    forced = {"polyphase": ctr.CTR_PATH_POLYPHASE, "col2im": ctr.CTR_PATH_COL2IM}[path]
    for (B, ci, co, L, k, s) in CASES:
        if path == "col2im" and len(L) > 1 and block_n == 256:
            continue   # same kernel as the 1-D cases; keeps the test short
        x, w = _case_inputs(rng, B, ci, co, L, k)
        y, desc = run_plan(x, w, None, s, 0, 0, "f32", path=forced, block_n=block_n)
        exact = oracle.conv_transpose(x.astype(np.float64), w.astype(np.float64), None, s, 0, 0)
        mag = oracle.conv_transpose(np.abs(x).astype(np.float64), np.abs(w).astype(np.float64),
                                    None, s, 0, 0)
        ratio = np.abs(y - exact) / np.maximum(mag, 1e-30)
        assert ratio.max() <= BOUND, (ratio.max(), (B, ci, co, L, k, s), desc)


def test_bound_rejects_single_tf32_products():
    """The bound is tight enough to tell: the same sums with every product taken as one tf32
    product (in float64, so nothing else rounds) exceed it."""
    rng = np.random.default_rng(5)
    B, ci, co, L, k, s = CASES[0]
    x, w = _case_inputs(rng, B, ci, co, L, k)
    exact = oracle.conv_transpose(x.astype(np.float64), w.astype(np.float64), None, s, 0, 0)
    mag = oracle.conv_transpose(np.abs(x).astype(np.float64), np.abs(w).astype(np.float64),
                                None, s, 0, 0)
    one = oracle.conv_transpose(_tf32(x).astype(np.float64), _tf32(w).astype(np.float64),
                                None, s, 0, 0)
    assert (np.abs(one - exact) / mag).max() > 4 * BOUND
