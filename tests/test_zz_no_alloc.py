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


def _polyphase_case(rng):
    """A small fp32 polyphase plan with its device inputs (split-K 1, so the GEMM's fused
    output stage writes y)."""
    import torch
    import workloads
    x = torch.from_numpy(workloads._cast(rng.standard_normal((1, 64, 300)), "f32")).cuda()
    w = torch.from_numpy(workloads._cast(rng.uniform(-0.1, 0.1, (64, 32, 16)), "f32")).cuda()
    b = torch.from_numpy(workloads._cast(rng.normal(0.0, 0.1, 32), "f32")).cuda()
    plan = ctr.Plan(1, 64, 32, (300,), (16,), 8, 4, 0, path=ctr.CTR_PATH_POLYPHASE, split_k=1)
    return plan, x, w, b


@pytest.mark.gpu
def test_noalloc_leaves_free_device_memory_unchanged():
    """After a first call (which looks up the scratch array's address), further calls change
    the device's free memory by nothing: they allocate no device memory."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _ensure_lib()
    plan, x, w, b = _polyphase_case(np.random.default_rng(7))
    try:
        y = torch.empty(plan.out_shape, dtype=torch.float32, device="cuda")
        stream = ctr._stream_ptr(None)
        args = (plan.handle, ctr._ptr(x), ctr._ptr(w), ctr._ptr(b), ctr._ptr(y), stream)
        ctr.ctr_forward_noalloc(*args)
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        for _ in range(5):
            ctr.ctr_forward_noalloc(*args)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0
    finally:
        plan.close()


@pytest.mark.gpu
def test_noalloc_timeout_is_reported_by_plan_check():
    """A 0 ns wait limit makes the GEMM's bounded waits give up on a healthy run: the
    allocation-free call records the timeout in its scratch status word and ctr_plan_check
    reports it; with the normal limit the next call is correct and the check is clean."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import oracle
    _ensure_lib()
    plan, x, w, b = _polyphase_case(np.random.default_rng(8))
    try:
        y = torch.empty(plan.out_shape, dtype=torch.float32, device="cuda")
        stream = ctr._stream_ptr(None)
        args = (plan.handle, ctr._ptr(x), ctr._ptr(w), ctr._ptr(b), ctr._ptr(y), stream)
        plan.set_wait_limit_ns(0)
        ctr.ctr_forward_noalloc(*args)
        assert ctr.lib.ctr_plan_check(plan.handle, stream) == ctr.CTR_ERR_DEVICE_TIMEOUT
        plan.set_wait_limit_ns(4_000_000_000)
        ctr.ctr_forward_noalloc(*args)
        assert ctr.lib.ctr_plan_check(plan.handle, stream) == ctr.CTR_OK
        ref = oracle.conv_transpose(x.cpu().numpy(), w.cpu().numpy(), b.cpu().numpy(), 8, 4, 0)
        assert oracle.rel_l2(y.cpu().numpy(), ref) <= 1e-5
    finally:
        plan.close()
