"""Checks that pin the CPU oracle to facts outside itself.

Each ``pin_*`` function takes the ConvTranspose callable under test (normally
``oracle.conv_transpose``) and raises ``AssertionError`` when the callable disagrees with:

* ``pin_torch_f64_1d`` / ``pin_torch_f64_2d`` -- torch's own float64 CPU ConvTranspose, a
  library routine written independently of this repository;
* ``pin_adjoint`` -- the transpose of a forward strided convolution whose dense matrix is
  built element by element from the forward definition (itself checked against torch's
  conv1d / conv2d);
* ``pin_hand_cases`` -- cases worked out by hand (``tests/golden/hand_cases.json``);
* ``pin_matmul`` -- kernel = stride, no padding: a reshape of the plain matmul
  X^T[L_in, C_in] . W[C_in, C_out*k];
* ``pin_polyphase`` -- the polyphase identity of "[XNNPACK] Lower dense transposed convs as
  one polyphase conv + depth to space" (Summary): one stride-1 convolution with m taps and
  padding m - 1 computing every phase, then the phase interleave and the padding slice;
* ``pin_output_phases`` -- the same polyphase sum re-indexed by the output's own phases:
  with p = s*pq + pm, phase J of output position Q takes the taps s*(m-1-v) + J + pm of the
  kernel over m (+1 when pm > 0) input positions Q + pq - (m-1) + v, with no slice;
* ``pin_istft_sinusoid`` -- the closed-form iSTFT of a sinusoid framed without a window and
  overlap-added with a periodic Hann window at hop N/4, which sums to exactly 2;
* ``pin_torch_f64_groups`` -- torch's float64 ConvTranspose with groups (2, and depthwise);
* ``pin_depthwise_k_equals_s`` -- depthwise with kernel = stride and no padding: every input
  sample times the channel's kernel, laid end to end (an outer product);
* ``pin_adjoint_groups`` -- the transpose of a grouped forward strided convolution whose
  dense matrix is built element by element (itself checked against torch's grouped conv1d);
* ``pin_torch_f64_dilation`` -- torch's float64 ConvTranspose with dilation (1-D grid, 2-D
  with unequal dilations, grouped);
* ``pin_pad_slice`` -- separate front and back pads: the unpadded result (torch float64,
  padding 0) with output_padding positions of bias appended, sliced by the two pads;
* ``pin_adjoint_dilated`` -- the transpose of a dilated forward strided convolution with
  separate front and back pads, its dense matrix built element by element (itself checked
  against torch's conv1d on an explicitly padded input).

``tests/test_oracle_pins.py`` runs them on the oracle and, with mistakes planted in copies
of the oracle source, shows that each planted mistake fails at least one of them.
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np
import torch
import torch.nn.functional as F

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_rng = np.random.default_rng(20260917)


def _close(a, b, rtol=1e-12, atol=1e-12):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= atol + rtol * scale, "max abs err %.3g (scale %.3g)" % (err, scale)


def _torch_ct(x, w, b, s, p, op, groups=1, dilation=1):
    xt = torch.from_numpy(np.asarray(x, dtype=np.float64))
    wt = torch.from_numpy(np.asarray(w, dtype=np.float64))
    bt = None if b is None else torch.from_numpy(np.asarray(b, dtype=np.float64))
    fn = F.conv_transpose1d if xt.dim() == 3 else F.conv_transpose2d
    return fn(xt, wt, bt, stride=s, padding=p, output_padding=op, groups=groups,
              dilation=dilation).numpy()


def grid_1d(full=False):
    """(L_in, k, s, p, op) with L_out > 0: s in 1..4, k in 1..7, p in 0..k-1, op in 0..s-1."""
    Ls = range(1, 6) if full else (1, 2, 5)
    for s in range(1, 5):
        for k in range(1, 8):
            for p in range(0, k):
                for op in range(0, s):
                    for L in Ls:
                        if (L - 1) * s - 2 * p + k + op > 0:
                            yield L, k, s, p, op


def pin_torch_f64_1d(ct, full=False):
    chans = [(1, 1), (2, 3), (3, 2)]
    for n, (L, k, s, p, op) in enumerate(grid_1d(full)):
        C_in, C_out = chans[n % len(chans)]
        B = 1 + n % 2
        x = _rng.standard_normal((B, C_in, L))
        w = _rng.standard_normal((C_in, C_out, k))
        b = _rng.standard_normal(C_out) if n % 3 else None
        _close(ct(x, w, b, s, p, op), _torch_ct(x, w, b, s, p, op))


def pin_torch_f64_2d(ct):
    cases = []
    for (sy, sx) in [(1, 1), (2, 2), (2, 3), (3, 1)]:
        for (ky, kx) in [(1, 1), (2, 3), (4, 4), (3, 2)]:
            for (py, px) in [(0, 0), (1, 0), (0, 1)]:
                if py >= ky or px >= kx:
                    continue
                for (opy, opx) in [(0, 0), (sy - 1, sx - 1)]:
                    for (H, W) in [(1, 1), (2, 3), (4, 2)]:
                        Ho = (H - 1) * sy - 2 * py + ky + opy
                        Wo = (W - 1) * sx - 2 * px + kx + opx
                        if Ho > 0 and Wo > 0:
                            cases.append((H, W, ky, kx, sy, sx, py, px, opy, opx))
    for n, (H, W, ky, kx, sy, sx, py, px, opy, opx) in enumerate(cases):
        C_in, C_out = (2, 3) if n % 2 else (3, 1)
        x = _rng.standard_normal((1, C_in, H, W))
        w = _rng.standard_normal((C_in, C_out, ky, kx))
        b = _rng.standard_normal(C_out)
        _close(ct(x, w, b, (sy, sx), (py, px), (opy, opx)),
               _torch_ct(x, w, b, (sy, sx), (py, px), (opy, opx)))


def forward_conv_matrix_1d(w, L_in, L_out, s, p):
    """Dense matrix A of the forward strided convolution, element by element:
    Conv(y)[ic, i] = sum_{oc, t} w[ic, oc, t] * y[oc, i*s - p + t]  (y = 0 outside [0, L_out)).
    Rows index (ic, i), columns (oc, o)."""
    C_in, C_out, k = w.shape
    A = np.zeros((C_in * L_in, C_out * L_out))
    for ic in range(C_in):
        for i in range(L_in):
            for oc in range(C_out):
                for t in range(k):
                    o = i * s - p + t
                    if 0 <= o < L_out:
                        A[ic * L_in + i, oc * L_out + o] += w[ic, oc, t]
    return A


def pin_adjoint(ct):
    """ConvT is the adjoint of the forward strided conv: <ConvT(x), y> = <x, Conv(y)> for
    every x, y, i.e. the matrix of ConvT equals A^T."""
    n = 0
    for (L, k, s, p, op) in grid_1d(full=False):
        n += 1
        if n % 3:
            continue
        C_in, C_out = (2, 3) if n % 2 else (3, 2)
        w = _rng.standard_normal((C_in, C_out, k))
        L_out = (L - 1) * s - 2 * p + k + op
        A = forward_conv_matrix_1d(w, L, L_out, s, p)
        # The forward definition itself against torch's conv1d (weight [out=C_in, in=C_out, k]).
        yv = _rng.standard_normal((1, C_out, L_out))
        ref = F.conv1d(torch.from_numpy(yv), torch.from_numpy(w), stride=s, padding=p).numpy()
        _close((A @ yv.reshape(-1)).reshape(1, C_in, -1), ref[:, :, :L])
        # The oracle's matrix, column by column from unit inputs.
        M = np.zeros((C_out * L_out, C_in * L))
        for j in range(C_in * L):
            e = np.zeros(C_in * L)
            e[j] = 1.0
            M[:, j] = ct(e.reshape(1, C_in, L), w, None, s, p, op).reshape(-1)
        _close(M, A.T)
        # And the inner-product form on random vectors.
        xv = _rng.standard_normal((1, C_in, L))
        lhs = float(np.sum(ct(xv, w, None, s, p, op) * yv))
        rhs = float(np.dot(xv.reshape(-1), A @ yv.reshape(-1)))
        assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs)), (lhs, rhs)


def pin_hand_cases(ct):
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        data = json.load(f)
    for case in data["cases"]:
        if "x_shape" in case:
            x = np.zeros(case["x_shape"])
        else:
            x = np.array(case["x"], dtype=np.float64)
        w = np.array(case["w"], dtype=np.float64)
        b = None if case["bias"] is None else np.array(case["bias"], dtype=np.float64)
        extra = {k: tuple(case[k]) for k in ("dilation", "padding_end") if k in case}
        y = ct(x, w, b, tuple(case["stride"]), tuple(case["padding"]),
               tuple(case["output_padding"]), **extra)
        np.testing.assert_array_equal(y, np.array(case["y"], dtype=np.float64),
                                      err_msg=case["name"])


def pin_matmul(ct):
    """k = s, p = op = 0: y[b, oc, s*i + t] = sum_ic x[b, ic, i] w[ic, oc, t], a reshape of
    X^T[L_in, C_in] @ W[C_in, C_out*k]; in 2-D with kH = sH, kW = sW likewise."""
    for (B, C_in, C_out, L, s) in [(1, 3, 2, 5, 2), (2, 4, 3, 7, 3), (1, 5, 1, 4, 4), (1, 2, 2, 3, 1)]:
        x = _rng.standard_normal((B, C_in, L))
        w = _rng.standard_normal((C_in, C_out, s))
        y = ct(x, w, None, s, 0, 0)
        for b in range(B):
            G = x[b].T @ w.reshape(C_in, C_out * s)                  # [L, C_out*s]
            ref = G.reshape(L, C_out, s).transpose(1, 0, 2).reshape(C_out, L * s)
            _close(y[b], ref)
    for (C_in, C_out, H, W, sy, sx) in [(3, 2, 3, 4, 2, 2), (2, 3, 2, 2, 3, 1)]:
        x = _rng.standard_normal((1, C_in, H, W))
        w = _rng.standard_normal((C_in, C_out, sy, sx))
        y = ct(x, w, None, (sy, sx), (0, 0), (0, 0))
        G = x[0].reshape(C_in, H * W).T @ w.reshape(C_in, C_out * sy * sx)   # [H*W, C_out*sy*sx]
        ref = (G.reshape(H, W, C_out, sy, sx).transpose(2, 0, 3, 1, 4)
               .reshape(C_out, H * sy, W * sx))
        _close(y[0], ref)


def polyphase_restatement(x, w, b, s, p, op):
    """1-D polyphase form, in double.  One stride-1 conv with m = k/s taps over x padded by
    m - 1 zeros on each side computes every phase,
        D[oc, j, q] = sum_{u<m} sum_ic x[ic, q + u - (m - 1)] * w[ic, oc, s*(m - 1 - u) + j],
    then the phases interleave, y_full[oc, s*q + j] = D[oc, j, q], and the padding slice
    keeps y[oc, o] = y_full[oc, o + p].  One extra zero column covers output_padding > p."""
    B, C_in, L = x.shape
    _, C_out, k = w.shape
    assert k % s == 0
    m = k // s
    Q = L + m - 1
    L_out = (L - 1) * s - 2 * p + k + op
    xp = np.zeros((B, C_in, L + 2 * (m - 1) + 1))
    xp[:, :, m - 1:m - 1 + L] = x
    D = np.zeros((B, C_out, s, Q + 1))
    for u in range(m):
        for j in range(s):
            wt = w[:, :, s * (m - 1 - u) + j]                 # [C_in, C_out]
            D[:, :, j, :] += np.einsum("bcq,co->boq", xp[:, :, u:u + Q + 1], wt)
    y_full = D.transpose(0, 1, 3, 2).reshape(B, C_out, (Q + 1) * s)
    y = y_full[:, :, p:p + L_out]
    assert y.shape[2] == L_out
    if b is not None:
        y = y + b[None, :, None]
    return y


def pin_polyphase(ct):
    for (L, k, s, p, op) in grid_1d(full=False):
        if s == 1:
            continue
        kk = -(-k // s) * s   # zero-pad the kernel to the next multiple of s
        C_in, C_out = 2, 3
        x = _rng.standard_normal((2, C_in, L))
        w = _rng.standard_normal((C_in, C_out, k))
        b = _rng.standard_normal(C_out)
        wpad = np.zeros((C_in, C_out, kk))
        wpad[:, :, :k] = w
        ref = polyphase_restatement(x, wpad, b, s, p, op)[:, :, :(L - 1) * s - 2 * p + k + op]
        _close(ct(x, w, b, s, p, op), ref)


def output_phase_restatement(x, w, b, s, p, op):
    """1-D polyphase form over the output's own phases, in double.  With m = ceil(k/s) and
    p = s*pq + pm (0 <= pm < s), output position Q's phase J is
        y[oc, s*Q + J] = sum_{v < m'} sum_ic x[ic, Q + pq - (m - 1) + v] * w[ic, oc, s*(m - 1 - v) + J + pm]
    with m' = m + (1 if pm > 0 else 0) taps, w = 0 outside [0, k) and x = 0 outside [0, L).
    The output needs no padding slice: its phases start at output 0."""
    B, C_in, L = x.shape
    _, C_out, k = w.shape
    m = -(-k // s)
    pq, pm = divmod(p, s)
    taps = m + (1 if pm else 0)
    L_out = (L - 1) * s - 2 * p + k + op
    Qv = -(-L_out // s)
    y = np.zeros((B, C_out, Qv * s))
    for Q in range(Qv):
        for J in range(s):
            for v in range(taps):
                i = Q + pq - (m - 1) + v
                t = s * (m - 1 - v) + J + pm
                if 0 <= i < L and 0 <= t < k:
                    y[:, :, s * Q + J] += np.einsum("bc,co->bo", x[:, :, i], w[:, :, t])
    y = y[:, :, :L_out]
    if b is not None:
        y = y + b[None, :, None]
    return y


def pin_output_phases(ct):
    for (L, k, s, p, op) in grid_1d(full=False):
        C_in, C_out = 2, 3
        x = _rng.standard_normal((2, C_in, L))
        w = _rng.standard_normal((C_in, C_out, k))
        b = _rng.standard_normal(C_out)
        _close(ct(x, w, b, s, p, op), output_phase_restatement(x, w, b, s, p, op))


def pin_istft_sinusoid(ct, n_fft=64, frames=12, batch=2, bin_f0=5):
    """The onesided spectra of a sinusoid's frames (rectangular window, hop N/4) fed through
    ConvTranspose1d with the Hann-windowed inverse real-DFT basis give 2 * the sinusoid on
    [3*hop, frames*hop), where four frames overlap."""
    hop = n_fft // 4
    w = workloads.istft_basis(n_fft)
    X = workloads.istft_sinusoid_frames(n_fft, hop, frames, batch, bin_f0, 0.7, 0.3)
    y = ct(X, w, None, hop, 0, 0)
    L_out = (frames - 1) * hop + n_fft
    assert y.shape == (batch, 1, L_out)
    sig = workloads.istft_sinusoid_signal(n_fft, L_out, batch, bin_f0, 0.7, 0.3)
    lo, hi = 3 * hop, frames * hop
    _close(y[:, 0, lo:hi], 2.0 * sig[:, lo:hi], rtol=1e-12, atol=1e-12)


def pin_torch_f64_groups(ct):
    """Grouped and depthwise ConvTranspose against torch float64, 1-D grid subset and 2-D."""
    n = 0
    for (L, k, s, p, op) in grid_1d(full=False):
        n += 1
        if n % 2:
            continue
        for (C_in, C_out, G) in ((4, 6, 2), (4, 4, 4), (3, 3, 3)):
            x = _rng.standard_normal((2, C_in, L))
            w = _rng.standard_normal((C_in, C_out // G, k))
            b = _rng.standard_normal(C_out)
            _close(ct(x, w, b, s, p, op, groups=G), _torch_ct(x, w, b, s, p, op, groups=G))
    for (H, W, ky, kx, sy, sx, py, px, G) in ((3, 4, 3, 2, 2, 1, 1, 0, 2), (2, 3, 4, 4, 2, 2, 1, 1, 6)):
        C = 6
        x = _rng.standard_normal((1, C, H, W))
        w = _rng.standard_normal((C, C // G, ky, kx))
        b = _rng.standard_normal(C)
        _close(ct(x, w, b, (sy, sx), (py, px), (0, 0), groups=G),
               _torch_ct(x, w, b, (sy, sx), (py, px), (0, 0), groups=G))


def pin_depthwise_k_equals_s(ct):
    """Depthwise, kernel = stride, no padding: y[b, c, s*i + t] = x[b, c, i] * w[c, 0, t] +
    bias[c] -- each input sample scales the channel's kernel, the copies laid end to end
    (and the 2-D analogue per dimension)."""
    for (B, C, L, s) in ((2, 3, 5, 2), (1, 4, 3, 4), (1, 2, 6, 1)):
        x = _rng.standard_normal((B, C, L))
        w = _rng.standard_normal((C, 1, s))
        b = _rng.standard_normal(C)
        ref = (x[:, :, :, None] * w[None, :, 0, None, :]).reshape(B, C, L * s) + b[None, :, None]
        _close(ct(x, w, b, s, 0, 0, groups=C), ref)
    B, C, H, W, sy, sx = 1, 3, 2, 3, 2, 3
    x = _rng.standard_normal((B, C, H, W))
    w = _rng.standard_normal((C, 1, sy, sx))
    ref = (x[:, :, :, None, :, None] * w[None, :, 0][:, :, None, :, None, :]).reshape(B, C, H * sy, W * sx)
    _close(ct(x, w, None, (sy, sx), (0, 0), (0, 0), groups=C), ref)


def forward_conv_matrix_groups_1d(w, L_in, L_out, s, p, G):
    """Dense matrix of the grouped forward strided convolution, element by element:
    Conv(y)[ic, i] = sum over the C_out/G channels oc of ic's group and taps t of
    w[ic, oc - g*C_out/G, t] * y[oc, i*s - p + t].  Rows (ic, i), columns (oc, o)."""
    C_in, cout_g, k = w.shape
    cin_g = C_in // G
    A = np.zeros((C_in * L_in, cout_g * G * L_out))
    for ic in range(C_in):
        g = ic // cin_g
        for i in range(L_in):
            for ocl in range(cout_g):
                oc = g * cout_g + ocl
                for t in range(k):
                    o = i * s - p + t
                    if 0 <= o < L_out:
                        A[ic * L_in + i, oc * L_out + o] += w[ic, ocl, t]
    return A


def pin_adjoint_groups(ct):
    """Grouped ConvT is the adjoint of the grouped forward strided conv."""
    for (L, k, s, p, op, C_in, C_out, G) in ((4, 3, 2, 1, 1, 4, 2, 2), (3, 4, 2, 1, 0, 3, 3, 3),
                                             (5, 5, 3, 2, 2, 2, 4, 2)):
        w = _rng.standard_normal((C_in, C_out // G, k))
        L_out = (L - 1) * s - 2 * p + k + op
        A = forward_conv_matrix_groups_1d(w, L, L_out, s, p, G)
        yv = _rng.standard_normal((1, C_out, L_out))
        ref = F.conv1d(torch.from_numpy(yv), torch.from_numpy(w), stride=s, padding=p,
                       groups=G).numpy()
        _close((A @ yv.reshape(-1)).reshape(1, C_in, -1), ref[:, :, :L])
        M = np.zeros((C_out * L_out, C_in * L))
        for j in range(C_in * L):
            e = np.zeros(C_in * L)
            e[j] = 1.0
            M[:, j] = ct(e.reshape(1, C_in, L), w, None, s, p, op, groups=G).reshape(-1)
        _close(M, A.T)


def grid_dilated_1d():
    """(L_in, k, s, d, p, op) with d in 2..3, s in 1..3, k in 1..4, p in 0..(k-1)d,
    op < max(s, d) (torch's limit) and L_out > 0."""
    for d in (2, 3):
        for s in range(1, 4):
            for k in range(1, 5):
                for p in range(0, (k - 1) * d + 1):
                    for op in range(0, max(s, d)):
                        for L in (1, 2, 4):
                            if (L - 1) * s + (k - 1) * d + 1 + op - 2 * p > 0:
                                yield L, k, s, d, p, op


def pin_torch_f64_dilation(ct):
    for n, (L, k, s, d, p, op) in enumerate(grid_dilated_1d()):
        C_in, C_out = ((1, 1), (2, 3), (3, 2))[n % 3]
        x = _rng.standard_normal((1 + n % 2, C_in, L))
        w = _rng.standard_normal((C_in, C_out, k))
        b = _rng.standard_normal(C_out) if n % 3 else None
        _close(ct(x, w, b, s, p, op, dilation=d), _torch_ct(x, w, b, s, p, op, dilation=d))
    for (H, W, ky, kx, sy, sx, dy, dx, py, px, opy, opx, G) in (
            (3, 4, 3, 2, 2, 1, 2, 3, 1, 0, 1, 2, 1), (2, 3, 2, 3, 1, 2, 3, 1, 2, 1, 0, 1, 1),
            (4, 2, 2, 2, 2, 2, 2, 2, 1, 1, 1, 0, 2), (2, 2, 3, 3, 3, 2, 1, 2, 0, 2, 2, 1, 3)):
        C = 6
        x = _rng.standard_normal((1, C, H, W))
        w = _rng.standard_normal((C, C // G, ky, kx))
        b = _rng.standard_normal(C)
        args = ((sy, sx), (py, px), (opy, opx))
        _close(ct(x, w, b, *args, groups=G, dilation=(dy, dx)),
               _torch_ct(x, w, b, *args, groups=G, dilation=(dy, dx)))


def _pad_slice_ref(x, w, b, s, d, pb, pe, op):
    """The padding slice: torch's unpadded result (padding 0, no output_padding), op more
    positions of bias (or zeros) at the back of every spatial dimension, then pb positions
    cut at the front and pe at the back."""
    full = _torch_ct(x, w, b, s, 0, 0, dilation=d)
    nd = x.ndim - 2
    bias_v = np.zeros(full.shape[1]) if b is None else np.asarray(b, dtype=np.float64)
    grown = np.empty(full.shape[:2] + tuple(full.shape[2 + i] + op[i] for i in range(nd)))
    grown[...] = bias_v.reshape((1, -1) + (1,) * nd)
    grown[(slice(None), slice(None)) + tuple(slice(0, full.shape[2 + i]) for i in range(nd))] = full
    return grown[(slice(None), slice(None)) +
                 tuple(slice(pb[i], grown.shape[2 + i] - pe[i]) for i in range(nd))]


def pin_pad_slice(ct):
    n = 0
    for (L, k, s, d) in itertools.product((1, 3, 4), (1, 2, 4), (1, 2, 3), (1, 2)):
        full = (L - 1) * s + (k - 1) * d + 1
        for pb in range(0, 3):
            for pe in range(0, 3):
                for op in range(0, max(s, d)):
                    if full + op - pb - pe <= 0:
                        continue
                    n += 1
                    C_in, C_out = ((1, 2), (3, 1), (2, 2))[n % 3]
                    x = _rng.standard_normal((1, C_in, L))
                    w = _rng.standard_normal((C_in, C_out, k))
                    b = _rng.standard_normal(C_out) if n % 2 else None
                    _close(ct(x, w, b, s, pb, op, dilation=d, padding_end=pe),
                           _pad_slice_ref(x, w, b, (s,), (d,), (pb,), (pe,), (op,)))
    for (H, W, ky, kx, sy, sx, dy, dx, pb, pe, op) in (
            (3, 2, 2, 3, 2, 1, 1, 2, (0, 2), (1, 0), (1, 0)),
            (2, 4, 3, 2, 1, 2, 2, 1, (2, 0), (0, 1), (0, 1)),
            (4, 4, 4, 4, 2, 2, 1, 1, (1, 2), (2, 1), (1, 1))):
        x = _rng.standard_normal((1, 2, H, W))
        w = _rng.standard_normal((2, 3, ky, kx))
        b = _rng.standard_normal(3)
        _close(ct(x, w, b, (sy, sx), pb, op, dilation=(dy, dx), padding_end=pe),
               _pad_slice_ref(x, w, b, (sy, sx), (dy, dx), pb, pe, op))


def forward_conv_matrix_dilated_1d(w, L_in, L_out, s, d, pb):
    """Dense matrix of the forward strided convolution with dilation d and front pad pb,
    element by element: Conv(y)[ic, i] = sum_{oc, t} w[ic, oc, t] * y[oc, i*s - pb + t*d]
    (y = 0 outside [0, L_out)).  Rows (ic, i), columns (oc, o)."""
    C_in, C_out, k = w.shape
    A = np.zeros((C_in * L_in, C_out * L_out))
    for ic in range(C_in):
        for i in range(L_in):
            for oc in range(C_out):
                for t in range(k):
                    o = i * s - pb + t * d
                    if 0 <= o < L_out:
                        A[ic * L_in + i, oc * L_out + o] += w[ic, oc, t]
    return A


def pin_adjoint_dilated(ct):
    """ConvT with dilation and front/back pads is the adjoint of the dilated forward conv;
    the output length is (L_in - 1)s + (k - 1)d + 1 + op - pb - pe."""
    for (L, k, s, d, pb, pe, op) in ((4, 3, 2, 2, 1, 0, 1), (3, 2, 3, 2, 0, 2, 0),
                                     (5, 3, 1, 3, 2, 1, 2), (2, 4, 2, 1, 2, 0, 1),
                                     (3, 3, 2, 3, 0, 3, 2)):
        C_in, C_out = 2, 3
        w = _rng.standard_normal((C_in, C_out, k))
        L_out = (L - 1) * s + (k - 1) * d + 1 + op - pb - pe
        A = forward_conv_matrix_dilated_1d(w, L, L_out, s, d, pb)
        yv = _rng.standard_normal((1, C_out, L_out))
        # The forward definition against torch's conv1d on y padded by pb zeros in front and
        # enough at the back for L outputs.
        back = max(0, (L - 1) * s + (k - 1) * d + 1 - pb - L_out)
        ypad = np.pad(yv, ((0, 0), (0, 0), (pb, back)))
        ref = F.conv1d(torch.from_numpy(ypad), torch.from_numpy(w), stride=s, dilation=d).numpy()
        _close((A @ yv.reshape(-1)).reshape(1, C_in, -1), ref[:, :, :L])
        M = np.zeros((C_out * L_out, C_in * L))
        for j in range(C_in * L):
            e = np.zeros(C_in * L)
            e[j] = 1.0
            out = ct(e.reshape(1, C_in, L), w, None, s, pb, op, dilation=d, padding_end=pe)
            assert out.shape == (1, C_out, L_out), out.shape
            M[:, j] = out.reshape(-1)
        _close(M, A.T)


ALL_PINS = [pin_torch_f64_dilation, pin_pad_slice, pin_adjoint_dilated, pin_torch_f64_groups, pin_depthwise_k_equals_s, pin_adjoint_groups,
            pin_torch_f64_1d, pin_torch_f64_2d, pin_adjoint, pin_hand_cases, pin_matmul,
            pin_polyphase, pin_output_phases, pin_istft_sinusoid]
