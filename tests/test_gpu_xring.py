"""fp32 256-row GEMM tiles in X-ring mode, against the oracle.

With four or more taps along x, an fp32 plan on 256-row tiles shares one staged-input box
per (channel slice, tap row) among that row's taps: each tap reads it through a
descriptor that starts one row further down per tap. Split-K units then take whole channel
slices. These cases force that mode at several tap counts, split-K factors, ragged channel
counts and positions spanning several tiles. On small-integer inputs every product and
partial sum is exact, so the results must equal the oracle bit for bit.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import transposed_convolution_gb300 as ctr  # noqa: E402
from gpu_helpers import reference, run_plan  # noqa: E402

CASES = [  # (B, C_in, C_out, L, k, s, p, op)
    (1, 64, 40, (300,), (16,), (4,), (2,), (1,)),     # 4 taps
    (2, 40, 33, (200,), (20,), (4,), (0,), (3,)),     # 5 taps, ragged channels
    (1, 96, 17, (260,), (8,), (1,), (3,), (0,)),      # 8 taps at stride 1
    (2, 24, 70, (9, 150), (2, 8), (2, 2), (0, 1), (1, 0)),   # 2-D, 4 taps along x per tap row
]


@pytest.mark.parametrize("split", [1, 2, 5])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_xring_bit_exact(case, split):
    B, ci, co, L, k, s, p, op = CASES[case]
    rng = np.random.default_rng(600 + 10 * case + split)
    x = rng.integers(-2, 3, (B, ci) + L).astype(np.float32)
    w = rng.integers(-2, 3, (ci, co) + k).astype(np.float32)
    b = rng.integers(-2, 3, (co,)).astype(np.float32)
    y, desc = run_plan(x, w, b, s, p, op, "f32", path=ctr.CTR_PATH_POLYPHASE, split_k=split,
                       block_n=256)
    kb_per_tap = -(-ci // 32)
    if split <= kb_per_tap:
        assert "x-ring" in desc, desc
    ref = reference(x, w, b, s, p, op, "f32")
    np.testing.assert_array_equal(y, ref, err_msg=desc)
