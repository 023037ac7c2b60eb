"""GPU parity of the inverse STFT computed by inverse real FFTs (ctr_istft_*) against the
oracle: the dense ConvTranspose1d with the windowed inverse real-DFT basis
("[WebGPU] optimizations for audio models", the source-separation model's inverse STFT as a
ConvTranspose1d).

* random onesided spectra, every frame length from 4 to 8192 (both parities of log2(n_fft/2),
  the radix-2 stage), hops below, at and above n_fft / 4, padding, output padding, bias,
  Hann and random windows, one to three batch items, one frame and a ragged frame count,
  within rel_l2 1e-5 (fp32 I/O);
* the closed-form iSTFT of a sinusoid at full size (n_fft 4096, hop 1024, 343 frames, batch 4);
* the iSTFT workload at full size: against the tensor-core ConvTranspose path on the same
  inputs, and sampled outputs against the oracle computed on the frames that reach them;
* no frames (y = bias), determinism, and the error statuses.
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
from gpu_helpers import GUARD, run_plan  # noqa: E402


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float32))).cuda()


def run_istft(spec, window, hop, padding=0, output_padding=0, bias=None, repeat=1):
    """spec [B, n_fft + 2, T] (float32 values), window [n_fft].  Returns y (float64 numpy)."""
    B, C, T = spec.shape
    n_fft = C - 2
    plan = ctr.Istft(B, n_fft, hop, T, padding, output_padding)
    try:
        plan.set_window(_dev(window))
        n = int(np.prod(plan.out_shape))
        buf = torch.full((n + 2 * GUARD,), float("nan"), device="cuda")
        y = buf[GUARD:GUARD + n].view(plan.out_shape)
        spec_d = _dev(spec)
        bias_d = None if bias is None else _dev(np.asarray([bias], np.float32))
        outs = []
        for _ in range(repeat):
            plan.forward(spec_d, bias_d, y=y)
            torch.cuda.synchronize()
            outs.append(y.cpu().numpy().astype(np.float64))
        g = torch.cat([buf[:GUARD], buf[GUARD + n:]]).cpu().numpy()
        assert np.all(np.isnan(g)), "library wrote outside y"
        return outs if repeat > 1 else outs[0]
    finally:
        plan.close()


def reference(spec, window, hop, padding=0, output_padding=0, bias=None):
    n_fft = spec.shape[1] - 2
    w = workloads.istft_basis(n_fft, window)
    b = None if bias is None else np.asarray([bias], np.float64)
    return oracle.conv_transpose(spec, w, b, hop, padding, output_padding)


CASES = [  # (B, n_fft, hop, frames, padding, output_padding, bias, window)
    (1, 4, 1, 5, 0, 0, None, "hann"),
    (2, 8, 2, 7, 0, 1, 0.5, "random"),
    (1, 16, 4, 1, 0, 0, None, "hann"),
    (3, 32, 8, 9, 4, 0, -0.25, "random"),
    (1, 64, 16, 13, 0, 3, None, "hann"),
    (2, 128, 100, 6, 10, 0, None, "random"),        # hop not dividing n_fft
    (1, 256, 64, 33, 128, 0, 1.0, "hann"),          # centre-style padding n_fft / 2
    (1, 512, 512, 4, 0, 0, None, "random"),         # hop = n_fft: no overlap
    (2, 1024, 256, 5, 0, 0, None, "hann"),
    (1, 2048, 700, 3, 0, 5, None, "random"),
    (2, 4096, 1024, 11, 0, 0, None, "hann"),        # the workload's frame
    (1, 8192, 2048, 3, 4096, 0, None, "random"),    # largest frame (one frame a block)
]


def _window(kind, n_fft, rng):
    return workloads.hann_window(n_fft) if kind == "hann" else rng.uniform(0.1, 1.0, n_fft)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d-n%d-hop%d-T%d-p%d-op%d" % c[:6])
def test_random_spectra_within_tolerance(case):
    B, n_fft, hop, T, p, op, bias, wkind = case
    rng = np.random.default_rng(71 + n_fft)
    spec = rng.standard_normal((B, n_fft + 2, T)).astype(np.float32)
    win = _window(wkind, n_fft, rng).astype(np.float32)
    y = run_istft(spec, win, hop, p, op, bias)
    ref = reference(spec, win, hop, p, op, bias)
    assert y.shape == ref.shape
    err = oracle.rel_l2(y, ref)
    assert err <= 1e-5, "rel_l2 %.3g" % err
    # element by element too: no single output far off
    scale = np.abs(ref).max() + 1e-30
    assert np.abs(y - ref).max() <= 1e-5 * scale


def test_sinusoid_full_size():
    """The iSTFT of a sinusoid's closed-form spectra (rectangular analysis frames, hop N/4,
    Hann synthesis window) is 2 * the sinusoid where four frames overlap."""
    N, hop, frames, batch, f0 = 4096, 1024, 343, 4, 37
    X = workloads.istft_sinusoid_frames(N, hop, frames, batch, f0, 0.5, 0.25).astype(np.float32)
    y = run_istft(X, workloads.hann_window(N).astype(np.float32), hop)
    sig = workloads.istft_sinusoid_signal(N, y.shape[-1], batch, f0, 0.5, 0.25)
    lo, hi = 3 * hop, frames * hop
    err = oracle.rel_l2(y[:, 0, lo:hi], 2.0 * sig[:, lo:hi])
    assert err <= 1e-6, err


def test_workload_full_size():
    """The iSTFT workload (batch 4, 343 frames of 4096, hop 1024): the FFT path against the
    tensor-core ConvTranspose path on the same inputs, and sampled outputs against the oracle
    on the frames that reach them."""
    li = workloads.make_workload("istft_irfft_f32")[0]
    L = li.layer
    spec, win = li.x, li.w
    y = run_istft(spec, win, L.stride[0])
    basis = workloads.istft_basis(L.kernel[0], win).astype(np.float32)
    y_tc, desc = run_plan(spec, basis, None, L.stride[0], 0, 0, "f32")
    assert oracle.rel_l2(y, y_tc) <= 1e-5, desc
    rng = np.random.default_rng(72)
    N, hop, T = L.kernel[0], L.stride[0], L.in_sp[0]
    for _ in range(24):
        b, n = int(rng.integers(L.B)), int(rng.integers(y.shape[-1]))
        k0, k1 = max(0, (n - N) // hop + 1), min(T - 1, n // hop)
        sub = spec[b:b + 1, :, k0:k1 + 1]
        ref = oracle.conv_transpose(sub, basis.astype(np.float64), None, hop, 0, 0)
        val = ref[0, 0, n - k0 * hop]
        assert abs(y[b, 0, n] - val) <= 1e-5 * (np.abs(ref).max() + 1e-30), (b, n)


def test_no_frames_and_determinism():
    rng = np.random.default_rng(73)
    win = workloads.hann_window(16).astype(np.float32)
    y = run_istft(np.zeros((2, 18, 0), np.float32), win, 4, 0, 0, bias=0.75)
    assert y.shape == (2, 1, 12)
    np.testing.assert_array_equal(y, np.full((2, 1, 12), 0.75))
    spec = rng.standard_normal((2, 1026, 40)).astype(np.float32)
    outs = run_istft(spec, workloads.hann_window(1024).astype(np.float32), 256, repeat=3)
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_errors():
    plan = ctr.Istft(1, 64, 16, 4)
    try:
        spec = torch.zeros((1, 66, 4), device="cuda")
        y = torch.empty(plan.out_shape, device="cuda")
        st = ctr.lib.ctr_istft_forward(plan.handle, spec.data_ptr(), None, y.data_ptr(), None)
        assert st == ctr.CTR_ERR_NOT_PREPARED
        win = torch.ones(64, device="cuda")
        plan.set_window(win)
        st = ctr.lib.ctr_istft_forward(plan.handle, spec.data_ptr() + 4, None, y.data_ptr(), None)
        assert st == ctr.CTR_ERR_MISALIGNED
        with pytest.raises(ValueError):
            plan.forward(torch.zeros((1, 66, 5), device="cuda"))
    finally:
        plan.close()
    with pytest.raises(ctr.CtrError) as e:
        ctr.ctr_istft_create(1, 64, 16, 4, 0, 0, ctr.CTR_BF16)
    assert e.value.status == ctr.CTR_ERR_UNSUPPORTED
