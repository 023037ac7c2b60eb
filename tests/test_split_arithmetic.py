"""The arithmetic of the fp32 split products, checked on the CPU.

For fp32 I/O the library takes a product x*w as hi_x*hi_w (hi = v rounded to tf32, to
nearest with ties away from zero) plus the cross products bf16(hi_x)*bf16(lo_w) +
bf16(lo_x)*bf16(hi_w) (lo = v - hi, bf16 rounding to nearest even), and drops lo_x*lo_w.
The GPU tests bound each output's error by 2^-16 * sum |x*w|; that rests on every single
product being within about 2^-17 of |x*w|, which is checked here with exact float64
arithmetic over random values, values at the edges of a binade and values whose lo part is
at its largest. Dropping either cross product (or both) breaks the bound.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def tf32_rna(a):
    """fp32 -> tf32 (10 explicit mantissa bits), to nearest with ties away from zero."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x1000) & 0xFFFFE000) & 0xFFFFFFFF
    return u.astype(np.uint32).view(np.float32)


def bf16_rn(a):
    """fp32 -> bf16 -> float64, to nearest even (torch's conversion)."""
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def split_product(x, w, cross=(True, True)):
    x = np.asarray(x, np.float32)
    w = np.asarray(w, np.float32)
    hx, hw = tf32_rna(x), tf32_rna(w)
    lx = (x.astype(np.float64) - hx).astype(np.float32)   # exact in fp32
    lw = (w.astype(np.float64) - hw).astype(np.float32)
    assert np.all(lx.astype(np.float64) == x.astype(np.float64) - hx)
    p = hx.astype(np.float64) * hw.astype(np.float64)
    if cross[0]:
        p = p + bf16_rn(hx) * bf16_rn(lw)
    if cross[1]:
        p = p + bf16_rn(lx) * bf16_rn(hw)
    return p


def _values(rng, n):
    mant = rng.integers(0, 1 << 23, n)
    expo = rng.integers(-20, 20, n)
    sign = rng.choice([-1.0, 1.0], n)
    v = sign * (1.0 + mant / float(1 << 23)) * np.exp2(expo)
    # edges: binade bottoms and tops, lo at its largest (a tie in the tf32 rounding)
    edges = np.array([1.0, 1.0 - 2.0**-24, 1.0 + 2.0**-23, 1.0 + 2.0**-11, 1.0 + 2.0**-11 - 2.0**-23,
                      1.5 + 2.0**-12, 1.999999, -1.0 - 3 * 2.0**-12], dtype=np.float64)
    return np.concatenate([v, edges]).astype(np.float32)


def test_split_product_error_bound():
    rng = np.random.default_rng(1234)
    x = _values(rng, 200000)
    w = rng.permutation(_values(rng, 200000))
    exact = x.astype(np.float64) * w.astype(np.float64)
    err = np.abs(split_product(x, w) - exact) / np.abs(exact)
    assert err.max() <= 2.0**-17, err.max()
    # the typical error is far below the worst case
    assert np.sqrt(np.mean(err**2)) < 2.0**-19


@pytest.mark.parametrize("cross", [(False, True), (True, False), (False, False)])
def test_dropping_a_cross_product_breaks_the_bound(cross):
    rng = np.random.default_rng(99)
    x = _values(rng, 20000)
    w = rng.permutation(_values(rng, 20000))
    exact = x.astype(np.float64) * w.astype(np.float64)
    err = np.abs(split_product(x, w, cross) - exact) / np.abs(exact)
    assert err.max() > 2.0**-13, err.max()


def test_tf32_rounding_reference_points():
    # ties go away from zero; 10 explicit bits survive
    assert tf32_rna(np.float32(1.0 + 2.0**-11))[()] == np.float32(1.0 + 2.0**-10)
    assert tf32_rna(np.float32(-(1.0 + 2.0**-11)))[()] == np.float32(-(1.0 + 2.0**-10))
    assert tf32_rna(np.float32(1.0 + 2.0**-11 - 2.0**-23))[()] == np.float32(1.0)
    assert tf32_rna(np.float32(1.0 + 2.0**-10))[()] == np.float32(1.0 + 2.0**-10)
