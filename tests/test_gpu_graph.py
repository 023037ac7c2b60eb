"""ctr_forward under CUDA-graph capture (the way the benchmark times steps): replays of a
captured forward follow new input data written into the captured buffers, match the oracle
bit for bit on integer-valued inputs, and record the plan's timing events every replay."""
import numpy as np
import pytest

from gpu_helpers import reference, to_dev, tdtype

import transposed_convolution_gb300 as ctr

CASES = [
    # (x shape, w shape, stride, padding, output_padding, dtype, split_k)
    ((1, 64, 200), (64, 32, 16), 8, 4, 0, "f32", 0),
    ((2, 96, 150), (96, 70, 8), 4, 2, 1, "f32", 2),      # split-K: GEMM + reduce kernel
    ((1, 128, 300), (128, 64, 4), 2, 1, 0, "bf16", 0),
    ((1, 40, 19, 23), (40, 20, 4, 4), (2, 2), (1, 1), (0, 1), "f32", 0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-%dd-split%d" % (c[5], len(c[0]) - 2, c[6]))
def test_graph_replay_follows_inputs(case):
    import torch
    xs, ws, s, p, op, dtype, split_k = case
    rng = np.random.default_rng(17)
    w = rng.integers(-2, 3, ws).astype(np.float32)
    b = rng.integers(-2, 3, (ws[1],)).astype(np.float32)
    plan = ctr.Plan(xs[0], xs[1], ws[1], xs[2:], ws[2:], s, p, op, dtype=tdtype(dtype),
                    split_k=split_k)
    try:
        plan.prepack(to_dev(w, dtype))
        x_dev = to_dev(np.zeros(xs, np.float32), dtype)
        b_dev = to_dev(b, dtype)
        y_dev = torch.empty(plan.out_shape, dtype=tdtype(dtype), device="cuda")
        plan.forward(x_dev, b_dev, y=y_dev)          # warm-up outside capture
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        e1.record()
        g = torch.cuda.CUDAGraph()
        ctr.ctr_plan_set_timing_events(plan.handle, e0.cuda_event, e1.cuda_event)
        with torch.cuda.graph(g):
            plan.forward(x_dev, b_dev, y=y_dev)
        ctr.ctr_plan_set_timing_events(plan.handle, None, None)
        for it in range(3):
            x = rng.integers(-2, 3, xs).astype(np.float32)
            x_dev.copy_(to_dev(x, dtype))
            y_dev.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            plan.check()
            np.testing.assert_array_equal(y_dev.float().cpu().numpy().astype(np.float64),
                                          reference(x, w, b, s, p, op, dtype),
                                          err_msg="replay %d" % it)
            assert e0.elapsed_time(e1) > 0.0
    finally:
        plan.close()


@pytest.mark.gpu
def test_timing_events_outside_capture():
    """The measurement hook on plain (uncaptured) calls: both events record and bracket the
    main kernel."""
    import torch
    plan = ctr.Plan(1, 64, 32, (200,), (16,), 8, 4, 0, dtype=torch.float32)
    try:
        plan.prepack(torch.randn(64, 32, 16, device="cuda"))
        x = torch.randn(1, 64, 200, device="cuda")
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        e1.record()
        ctr.ctr_plan_set_timing_events(plan.handle, e0.cuda_event, e1.cuda_event)
        plan.forward(x)
        ctr.ctr_plan_set_timing_events(plan.handle, None, None)
        torch.cuda.synchronize()
        plan.check()
        assert e0.elapsed_time(e1) > 0.0
    finally:
        plan.close()
