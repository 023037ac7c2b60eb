"""Seeded synthetic workloads for the ConvTranspose library, its tests and its benchmark.

This module only draws inputs and describes shapes.  It holds none of the convolution's
arithmetic, and both the CPU oracle and the CUDA path take their inputs from here.

The first five workloads stand in for the audio decoders the source pages measure (codec
and vocoder upsamplers with kernel = 2*stride and the iSTFT overlap-add of a
source-separation model, "[XNNPACK] Lower dense transposed convs as one polyphase conv +
depth to space", Summary; "[WebGPU] optimizations for audio models", ConvTranspose commit).
The sixth is the depthwise 4x4 / stride-2 upsampling filter of the image-inpainting network
the XNNPACK page profiles (DecomposeDepthwiseConvTransposePass commit), at a feature-map
size chosen to be bound by HBM.  The seventh is the iSTFT workload again, computed by
inverse real FFTs (its weight input is the Hann window; the basis is implied).  Trained weights, audio and images are not available, so
every tensor is drawn from a seeded generator:

* x ~ N(0, 1); w ~ U(-1/sqrt(fan_in), +1/sqrt(fan_in)) with fan_in = (C_in / groups) *
  prod(k); bias ~ N(0, 0.1) (0.1 read as the standard deviation);
* values are drawn in double and rounded to the I/O precision (fp32, or bf16 with ties to
  even), so both sides see the same exact values;
* the iSTFT weight is the periodic-Hann-windowed inverse real-DFT basis (N = 4096), with the
  2049 real parts in channels 0..2048 and the 2049 imaginary parts in channels 2049..4097.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Tuple

import numpy as np

SEED_BASE = 0x7C0DE5EED


@dataclasses.dataclass(frozen=True)
class Layer:
    """One ConvTranspose call: shapes, geometry, I/O dtype, bias and fused activation."""
    ndim: int
    B: int
    C_in: int
    C_out: int
    in_sp: Tuple[int, ...]
    kernel: Tuple[int, ...]
    stride: Tuple[int, ...]
    padding: Tuple[int, ...]
    output_padding: Tuple[int, ...]
    dtype: str = "f32"              # "f32", "bf16" or "f16"
    bias: bool = True
    act_slope: Optional[float] = None   # LeakyReLU negative slope, None = no activation
    weight: str = "uniform"          # "uniform" or "istft"
    groups: int = 1                  # groups = C_in = C_out: depthwise
    kind: str = "conv"               # "conv", or "istft": the same ConvTranspose with the
                                     # windowed inverse real-DFT basis, computed by FFTs; its
                                     # weight input is then the window [n_fft]

    @property
    def out_sp(self) -> Tuple[int, ...]:
        return tuple((self.in_sp[d] - 1) * self.stride[d] - 2 * self.padding[d]
                     + self.kernel[d] + self.output_padding[d] for d in range(self.ndim))

    @property
    def useful_macs(self) -> int:
        """B * C_in * (C_out / groups) * prod(L_in * k): the GEMM count of the X[M, C_in] x
        W[C_in, k*C_out] formulation, per group."""
        n = self.B * self.C_in * (self.C_out // self.groups)
        for d in range(self.ndim):
            n *= self.in_sp[d] * self.kernel[d]
        return n

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def compulsory_bytes(self) -> int:
        """x + w + bias + y, each once, in the I/O dtype."""
        e = self.elem_bytes
        nx = self.B * self.C_in * int(np.prod(self.in_sp))
        nw = self.C_in * (self.C_out // self.groups) * int(np.prod(self.kernel))
        if self.kind == "istft":
            nw = self.kernel[0]        # the window; the basis is never materialised
        nb = self.C_out if self.bias else 0
        ny = self.B * self.C_out * int(np.prod(self.out_sp))
        return e * (nx + nw + nb + ny)

    @property
    def in_bytes(self) -> int:
        """x in the I/O dtype."""
        return self.elem_bytes * self.B * self.C_in * int(np.prod(self.in_sp))

    @property
    def out_bytes(self) -> int:
        """y in the I/O dtype."""
        return self.elem_bytes * self.B * self.C_out * int(np.prod(self.out_sp))

    def describe(self) -> str:
        dims = "x".join(str(v) for v in self.in_sp)
        ks = "x".join(str(v) for v in self.kernel)
        ss = "x".join(str(v) for v in self.stride)
        ps = "x".join(str(v) for v in self.padding)
        g = f" groups{self.groups}" if self.groups != 1 else ""
        return (f"{self.ndim}d B{self.B} {self.C_in}->{self.C_out}{g} L{dims} k{ks} s{ss} p{ps} "
                f"{self.dtype}")


def _l1(B, C_in, C_out, L, k, s, p, op=0, **kw) -> Layer:
    return Layer(1, B, C_in, C_out, (L,), (k,), (s,), (p,), (op,), **kw)


def _stack() -> List[Layer]:
    chans = [512, 256, 128, 64, 32]
    strides = [8, 8, 2, 2]
    kernels = [16, 16, 4, 4]
    L = 1024
    layers = []
    for i in range(4):
        k, s = kernels[i], strides[i]
        p = (k - s) // 2
        layers.append(_l1(1, chans[i], chans[i + 1], L, k, s, p, dtype="bf16",
                          act_slope=0.1 if i < 3 else None))
        L = (L - 1) * s - 2 * p + k
    return layers


# The workloads, in order.  Index 0 is the tiny case, index 1 the codec upsampler the
# benchmark times at one GPU by default.
WORKLOADS = {
    "tiny_1d_f32": [_l1(1, 16, 8, 64, 4, 2, 1)],
    "codec_upsampler_f32": [_l1(1, 512, 256, 2000, 16, 8, 4)],
    "istft_f32": [_l1(4, 4098, 1, 343, 4096, 1024, 0, bias=False, weight="istft")],
    "decoder_2d_f32": [Layer(2, 1, 128, 64, (128, 128), (4, 4), (2, 2), (1, 1), (0, 0))],
    "vocoder_stack_bf16": _stack(),
    "depthwise_2d_bf16": [Layer(2, 4, 256, 256, (128, 128), (4, 4), (2, 2), (1, 1), (0, 0),
                                dtype="bf16", groups=256)],
    "istft_irfft_f32": [_l1(4, 4098, 1, 343, 4096, 1024, 0, bias=False, weight="istft",
                           kind="istft")],
}
WORKLOAD_ORDER = list(WORKLOADS)


def seed_of(name: str) -> int:
    return SEED_BASE + WORKLOAD_ORDER.index(name)


def to_bf16_values(a: np.ndarray) -> np.ndarray:
    """fp32 array whose values are rounded to bfloat16 (ties to even)."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32)
    return r.view(np.float32)


def _cast(a: np.ndarray, dtype: str) -> np.ndarray:
    """Values drawn in double, rounded to fp32, then (bf16, f16) to the 16-bit I/O type, ties
    to even; returned as float32 holding those values."""
    a32 = np.asarray(a, dtype=np.float64).astype(np.float32)
    if dtype == "bf16":
        return to_bf16_values(a32)
    if dtype == "f16":
        with np.errstate(over="ignore"):
            return a32.astype(np.float16).astype(np.float32)
    return a32


def hann_window(n_fft: int) -> np.ndarray:
    """Periodic Hann window win[t] = 0.5 - 0.5 cos(2 pi t / N), float64."""
    t = np.arange(n_fft, dtype=np.int64)
    return 0.5 - 0.5 * np.cos(2.0 * np.pi * t / n_fft)


def istft_basis(n_fft: int = 4096, window: Optional[np.ndarray] = None) -> np.ndarray:
    """Windowed inverse real-DFT basis as a ConvTranspose1d weight [n_fft + 2, 1, n_fft]
    (float64); the window defaults to the periodic Hann window.

    Channel f (0 <= f <= n_fft/2) carries c_f * win[t] * cos(2 pi f t / N) / N and channel
    n_fft/2 + 1 + f carries -c_f * win[t] * sin(2 pi f t / N) / N, with c_0 = c_{N/2} = 1,
    other c_f = 2.  Feeding the real and imaginary parts of a onesided spectrum into these
    channels gives the windowed inverse real DFT of each frame; a stride of the hop length
    overlap-adds the frames.
    """
    N = n_fft
    nb = N // 2 + 1
    t = np.arange(N, dtype=np.int64)
    win = hann_window(N) if window is None else np.asarray(window, dtype=np.float64)
    w = np.empty((2 * nb, 1, N), dtype=np.float64)
    for f in range(nb):
        c = 1.0 if f in (0, N // 2) else 2.0
        ang = 2.0 * np.pi * ((f * t) % N) / N
        w[f, 0, :] = c * win * np.cos(ang) / N
        w[nb + f, 0, :] = -c * win * np.sin(ang) / N
    return w


def istft_sinusoid_frames(n_fft: int, hop: int, frames: int, batch: int, bin_f0: int,
                          amp: float, phase: float) -> np.ndarray:
    """Onesided spectra [batch, n_fft + 2, frames] of a sinusoid framed with a rectangular
    window, in closed form (no DFT).

    For x[n] = amp * cos(2 pi f0 n / N + phase) and frame k = x[k*hop : k*hop + N], the DFT
    is (amp*N/2) e^{i theta_k} at bin f0 and zero at every other onesided bin, with
    theta_k = phase + 2 pi f0 k hop / N (f0 an integer, 1 <= f0 <= N/2 - 1).  Batch item b
    uses phase + b.
    """
    nb = n_fft // 2 + 1
    X = np.zeros((batch, 2 * nb, frames), dtype=np.float64)
    k = np.arange(frames, dtype=np.float64)
    for b in range(batch):
        theta = phase + b + 2.0 * np.pi * ((bin_f0 * hop * k) % n_fft) / n_fft
        X[b, bin_f0, :] = amp * n_fft / 2.0 * np.cos(theta)
        X[b, nb + bin_f0, :] = amp * n_fft / 2.0 * np.sin(theta)
    return X


def istft_sinusoid_signal(n_fft: int, length: int, batch: int, bin_f0: int, amp: float,
                          phase: float) -> np.ndarray:
    """The sinusoid itself, [batch, length] float64 (batch item b uses phase + b)."""
    n = np.arange(length, dtype=np.int64)
    out = np.empty((batch, length), dtype=np.float64)
    for b in range(batch):
        out[b] = amp * np.cos(2.0 * np.pi * ((bin_f0 * n) % n_fft) / n_fft + phase + b)
    return out


@dataclasses.dataclass
class LayerInputs:
    layer: Layer
    x: Optional[np.ndarray]     # float32 holding I/O-dtype values (None for stack stages > 0)
    w: np.ndarray               # float32 holding I/O-dtype values, [C_in, C_out, k...]
    bias: Optional[np.ndarray]  # float32 [C_out] or None


def make_layer_inputs(layer: Layer, seed: int, with_x: bool = True) -> LayerInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    x = None
    if with_x:
        x = _cast(rng.standard_normal((layer.B, layer.C_in) + tuple(layer.in_sp)), layer.dtype)
    if layer.kind == "istft":
        w = _cast(hann_window(layer.kernel[0]), layer.dtype)
    elif layer.weight == "istft":
        assert layer.ndim == 1 and layer.C_out == 1 and layer.C_in == layer.kernel[0] + 2
        w = _cast(istft_basis(layer.kernel[0]), layer.dtype)
    else:
        cin_g, cout_g = layer.C_in // layer.groups, layer.C_out // layer.groups
        a = 1.0 / math.sqrt(cin_g * int(np.prod(layer.kernel)))
        w = _cast(rng.uniform(-a, a, (layer.C_in, cout_g) + tuple(layer.kernel)), layer.dtype)
    bias = None
    if layer.bias:
        bias = _cast(rng.normal(0.0, 0.1, (layer.C_out,)), layer.dtype)
    return LayerInputs(layer, x, w, bias)


def make_workload(name: str) -> List[LayerInputs]:
    """Inputs of every layer of a workload.  Stack stages after the first take their x from
    the previous stage's output, so only stage 0 carries an x."""
    base = seed_of(name)
    out = []
    for i, layer in enumerate(WORKLOADS[name]):
        out.append(make_layer_inputs(layer, base + 1000 * i, with_x=(i == 0)))
    return out


def integer_inputs(layer: Layer, seed: int, mag: int = 4):
    """Small-integer x, w, bias (|v| <= mag) for bit-exact tests: with C_in * prod(k) * mag^2
    well below 2^8 every product and partial sum is exact in fp32, bf16 and tf32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.integers(-mag, mag + 1, (layer.B, layer.C_in) + tuple(layer.in_sp)).astype(np.float32)
    w = rng.integers(-mag, mag + 1, (layer.C_in, layer.C_out) + tuple(layer.kernel)).astype(np.float32)
    bias = rng.integers(-mag, mag + 1, (layer.C_out,)).astype(np.float32) if layer.bias else None
    return x, w, bias
