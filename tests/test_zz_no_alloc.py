"""ctr_forward_noalloc, the forward pass for callers that cannot allocate device memory.

It takes its scratch from the library's static device array and packs the weight on every
call.  The GPU test runs it twice in a row through the C ABI on each tensor-core path
(fused polyphase, split-K, col2im) and on the gather path, and compares every result with
ctr_forward on the same plan and inputs.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import transposed_convolution_gb300 as ctr


def _ensure_lib():
    from transposed_convolution_gb300 import build
    build.build()
    ctr.load_library()


def test_noalloc_rejects_plans_beyond_the_scratch_size():
    """The 4-frame iSTFT plan needs ~210 MB of scratch: refused before any CUDA call."""
    _ensure_lib()
    h = ctr.ctr_plan_create(1, 4, 4098, 1, [343], [4096], [1024], [0], [0], ctr.CTR_F32)
    try:
        p = ctypes.c_void_p(1 << 20)
        st = ctr.lib.ctr_forward_noalloc(h, p, p, None, p, None)
        assert st == ctr.CTR_ERR_NO_WORKSPACE
    finally:
        ctr.ctr_plan_destroy(h)


CASES = [
    # (x shape, w shape, stride, padding, output_padding, dtype, path, split_k)
    # split-K 1: the automatic choice (split 2) needs more scratch than the array holds
    ((1, 512, 1000), (512, 256, 16), 8, 4, 0, "f32", ctr.CTR_PATH_POLYPHASE, 1),
    ((1, 256, 1024), (256, 128, 16), 8, 4, 0, "bf16", ctr.CTR_PATH_POLYPHASE, 0),
    ((2, 96, 300), (96, 40, 8), 4, 2, 1, "f32", ctr.CTR_PATH_POLYPHASE, 3),
    ((1, 64, 33, 29), (64, 32, 4, 4), (2, 2), (1, 1), (0, 1), "f32", ctr.CTR_PATH_POLYPHASE, 0),
    ((2, 48, 70), (48, 30, 7), 3, 2, 1, "bf16", ctr.CTR_PATH_COL2IM, 0),
    ((1, 16, 64), (16, 8, 4), 2, 1, 0, "f32", ctr.CTR_PATH_GATHER, 0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-%s-%d" % (ctr.PATH_NAMES[c[6]], c[5], c[7]))
def test_noalloc_matches_forward_twice(case):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import oracle
    import workloads
    _ensure_lib()
    xs, ws, s, p, op, dtype, path, split_k = case
    rng = np.random.default_rng(42)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dev = lambda a: torch.from_numpy(a).cuda().to(tdt).contiguous()  # noqa: E731
    x = dev(workloads._cast(rng.standard_normal(xs), dtype))
    w = dev(workloads._cast(rng.uniform(-0.1, 0.1, ws), dtype))
    b = dev(workloads._cast(rng.normal(0.0, 0.1, ws[1]), dtype))
    plan = ctr.Plan(xs[0], xs[1], ws[1], xs[2:], ws[2:], s, p, op, dtype=tdt, path=path,
                    split_k=split_k)
    try:
        plan.prepack(w)
        y_ref = plan.forward(x, b)
        plan.check()
        stream = ctr._stream_ptr(None)
        for call in range(2):
            y = torch.full(plan.out_shape, float("nan"), dtype=tdt, device="cuda")
            ctr.ctr_forward_noalloc(plan.handle, ctr._ptr(x), ctr._ptr(w), ctr._ptr(b),
                                    ctr._ptr(y), stream)
            torch.cuda.synchronize()
            got = y.float().cpu().numpy()
            ref = y_ref.float().cpu().numpy()
            assert not np.isnan(got).any(), "call %d left outputs unwritten" % call
            tol = 1e-2 if dtype == "bf16" else 1e-5
            assert oracle.rel_l2(got, ref) <= tol
            # Same kernels on the same data: the results agree exactly.
            np.testing.assert_array_equal(got, ref)
    finally:
        plan.close()
