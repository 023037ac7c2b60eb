"""The C ABI's host half, without a GPU: the library builds, loads and exports every symbol
include/ctr.h declares; plan validation, output shapes, path choice and workspace sizing.
No call here launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ctr():
    from transposed_convolution_gb300 import build
    build.build()
    import transposed_convolution_gb300 as t
    t.load_library()
    return t


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ctr.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ctr_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ctr_plan_create", "ctr_prepack_weight", "ctr_forward", "ctr_plan_destroy",
                     "ctr_packed_weight_bytes", "ctr_workspace_bytes", "ctr_plan_bind_workspace",
                     "ctr_plan_output_shape", "ctr_plan_check", "ctr_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(ctr):
    raw = ctypes.CDLL(ctr.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), "missing export " + name
        assert name in ctr.SIGNATURES, "binding lacks " + name


def _plan(ctr, *args, **kw):
    return ctr.ctr_plan_create(*args, **kw)


def test_output_shapes_and_paths_of_the_workloads(ctr):
    import workloads
    expect_path = {"tiny_1d_f32": ctr.CTR_PATH_GATHER, "depthwise_2d_bf16": ctr.CTR_PATH_DEPTHWISE}
    for name, layers in workloads.WORKLOADS.items():
        for layer in layers:
            h = _plan(ctr, layer.ndim, layer.B, layer.C_in, layer.C_out, layer.in_sp, layer.kernel,
                      layer.stride, layer.padding, layer.output_padding,
                      ctr.CTR_BF16 if layer.dtype == "bf16" else ctr.CTR_F32)
            try:
                if layer.groups != 1:
                    ctr.ctr_plan_set_groups(h, layer.groups)
                assert ctr.ctr_plan_output_shape(h, layer.ndim) == layer.out_sp
                assert ctr.ctr_plan_get_path(h) == expect_path.get(name, ctr.CTR_PATH_POLYPHASE)
                if ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE:
                    assert ctr.ctr_workspace_bytes(h) > 0
                    assert ctr.ctr_packed_weight_bytes(h) > 0
                assert "path=" in ctr.ctr_plan_describe(h)
            finally:
                ctr.ctr_plan_destroy(h)


def test_col2im_chosen_when_kernel_not_multiple_of_stride(ctr):
    h = _plan(ctr, 1, 2, 32, 32, [50], [3], [2], [1], [1], ctr.CTR_F32)
    assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_COL2IM
    ctr.ctr_plan_destroy(h)
    h = _plan(ctr, 1, 2, 8, 16, [50], [3], [2], [1], [1], ctr.CTR_F32)   # C_in < 16
    assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_GATHER
    ctr.ctr_plan_destroy(h)


@pytest.mark.parametrize("args", [
    (3, 1, 4, 4, [8], [2], [2], [0], [0]),        # ndim
    (1, -1, 4, 4, [8], [2], [2], [0], [0]),       # N < 0
    (1, 1, 0, 4, [8], [2], [2], [0], [0]),        # C_in = 0
    (1, 1, 4, 0, [8], [2], [2], [0], [0]),        # C_out = 0
    (1, 1, 4, 4, [-1], [2], [2], [0], [0]),       # L_in < 0
    (1, 1, 4, 4, [8], [0], [2], [0], [0]),        # k = 0
    (1, 1, 4, 4, [8], [2], [0], [0], [0]),        # s = 0
    (1, 1, 4, 4, [8], [2], [2], [-1], [0]),       # p < 0
    (1, 1, 4, 4, [8], [2], [2], [0], [2]),        # op >= s
    (1, 1, 4, 4, [1], [2], [2], [1], [0]),        # L_out = 0
    (2, 1, 4, 4, [8, 8], [2, 2], [2, 2], [0, 0], [0, -1]),
])
def test_invalid_arguments_rejected(ctr, args):
    with pytest.raises(ctr.CtrError) as e:
        _plan(ctr, *args, dtype=ctr.CTR_F32)
    assert e.value.status == ctr.CTR_ERR_INVALID_ARG


def test_empty_input_is_a_valid_plan(ctr):
    h = _plan(ctr, 1, 1, 4, 4, [0], [4], [2], [0], [0], ctr.CTR_F32)
    assert ctr.ctr_plan_output_shape(h, 1) == (2,)
    ctr.ctr_plan_destroy(h)


def test_host_side_errors_without_gpu(ctr):
    h = _plan(ctr, 1, 1, 64, 64, [100], [4], [2], [1], [0], ctr.CTR_F32)
    try:
        # forward before prepack: rejected before any CUDA call
        st = ctr.lib.ctr_forward(h, ctypes.c_void_p(256), ctypes.c_void_p(256), None,
                                 ctypes.c_void_p(256), None)
        assert st == ctr.CTR_ERR_NOT_PREPARED
        assert ctr.lib.ctr_plan_bind_workspace(h, ctypes.c_void_p(4096 + 16), 1 << 30) == \
            ctr.CTR_ERR_MISALIGNED
        assert ctr.lib.ctr_plan_bind_workspace(h, ctypes.c_void_p(4096), 16) == \
            ctr.CTR_ERR_NO_WORKSPACE
        assert ctr.lib.ctr_plan_set_path(h, 9, 0) == ctr.CTR_ERR_INVALID_ARG
        assert ctr.lib.ctr_plan_set_activation(h, 7, 0.1) == ctr.CTR_ERR_INVALID_ARG
        # forcing each path re-plans
        for p in (ctr.CTR_PATH_GATHER, ctr.CTR_PATH_COL2IM, ctr.CTR_PATH_POLYPHASE):
            ctr.ctr_plan_set_path(h, p, 0)
            assert ctr.ctr_plan_get_path(h) == p
        ctr.ctr_plan_set_path(h, ctr.CTR_PATH_POLYPHASE, 3)
        assert "splits=3" in ctr.ctr_plan_describe(h)
        # forcing the phase-row tile re-plans; other widths are rejected
        for bn in (64, 128, 256):
            ctr.ctr_plan_set_tile(h, bn)
            assert "BN %d," % bn in ctr.ctr_plan_describe(h)
        for bad in (32, 96, 512, -1):
            assert ctr.lib.ctr_plan_set_tile(h, bad) == ctr.CTR_ERR_INVALID_ARG
        ctr.ctr_plan_set_tile(h, 0)
    finally:
        ctr.ctr_plan_destroy(h)
    for s in range(8):
        assert ctr.ctr_status_string(s)
    ctr.ctr_plan_destroy(None)


def test_null_plan_queries(ctr):
    assert ctr.lib.ctr_packed_weight_bytes(None) == 0
    assert ctr.lib.ctr_workspace_bytes(None) == 0
    assert ctr.lib.ctr_plan_get_path(None) == -1
    assert ctr.lib.ctr_plan_create(None, 1, 1, 1, 1, None, None, None, None, None, 0) == \
        ctr.CTR_ERR_INVALID_ARG


def test_no_kernel_launched_by_host_calls(ctr):
    assert ctr.ctr_launch_count() == 0


def test_chain_validation_without_gpu(ctr):
    """ctr_plan_chain: compatible plans chain and unchain; mismatched channels, sizes, dtype
    or path are rejected; destroying either side unchains the other."""
    bf = ctr.CTR_BF16
    a = _plan(ctr, 1, 1, 64, 32, [100], [4], [2], [1], [0], bf)      # out 200 x 32 ch
    b = _plan(ctr, 1, 1, 32, 64, [200], [4], [2], [1], [0], bf)      # in 200 x 32 ch
    c = _plan(ctr, 1, 1, 16, 64, [200], [4], [2], [1], [0], bf)      # wrong channels
    d = _plan(ctr, 1, 1, 32, 64, [201], [4], [2], [1], [0], bf)      # wrong length
    e = _plan(ctr, 1, 1, 32, 64, [200], [4], [2], [1], [0], ctr.CTR_F32)
    try:
        ctr.ctr_plan_chain(a, b)
        for bad in (c, d, e):
            assert ctr.lib.ctr_plan_chain(a, bad) == ctr.CTR_ERR_INVALID_ARG
        assert ctr.lib.ctr_plan_chain(a, a) == ctr.CTR_ERR_INVALID_ARG
        # a chained producer writes no y; without workspaces nothing runs
        st = ctr.lib.ctr_forward(a, ctypes.c_void_p(256), ctypes.c_void_p(256), None,
                                 ctypes.c_void_p(256), None)
        assert st in (ctr.CTR_ERR_NOT_PREPARED, ctr.CTR_ERR_INVALID_ARG)
        ctr.ctr_plan_chain(a, None)
        ctr.ctr_plan_chain(a, b)
    finally:
        ctr.ctr_plan_destroy(b)          # unchains a
        for h in (a, c, d, e):
            ctr.ctr_plan_destroy(h)


def test_groups_routing_without_gpu(ctr):
    """ctr_plan_set_groups: groups must divide both channel counts; groups = C_in runs on the
    depthwise kernel where its x kernel/stride is compiled, other groups on the gather kernel;
    the tensor-core paths and the depthwise kernel refuse plans they cannot run, leaving the
    plan as it was; the packed weight is the grouped torch weight."""
    bf = ctr.CTR_BF16
    h = _plan(ctr, 1, 1, 64, 64, [100], [4], [2], [1], [0], bf)
    try:
        for bad in (0, -1, 3, 128):
            assert ctr.lib.ctr_plan_set_groups(h, bad) == ctr.CTR_ERR_INVALID_ARG
        assert ctr.lib.ctr_plan_set_path(h, ctr.CTR_PATH_DEPTHWISE, 0) == ctr.CTR_ERR_UNSUPPORTED
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
        ctr.ctr_plan_set_groups(h, 64)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_DEPTHWISE
        assert ctr.ctr_packed_weight_bytes(h) == 64 * 1 * 4 * 2
        assert ctr.ctr_workspace_bytes(h) == 0
        assert "path=depthwise" in ctr.ctr_plan_describe(h)
        assert "groups=64" in ctr.ctr_plan_describe(h)
        for p in (ctr.CTR_PATH_POLYPHASE, ctr.CTR_PATH_COL2IM):
            assert ctr.lib.ctr_plan_set_path(h, p, 0) == ctr.CTR_ERR_UNSUPPORTED
            assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_DEPTHWISE
        ctr.ctr_plan_set_path(h, ctr.CTR_PATH_GATHER, 0)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_GATHER
        # a forced gather path stays when the groups change; back to one group re-plans
        ctr.ctr_plan_set_groups(h, 8)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_GATHER
        assert ctr.ctr_packed_weight_bytes(h) == 64 * 8 * 4 * 2
        ctr.ctr_plan_set_path(h, ctr.CTR_PATH_AUTO, 0)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_GATHER
        ctr.ctr_plan_set_groups(h, 1)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
        # a forced tensor-core path refuses groups
        ctr.ctr_plan_set_path(h, ctr.CTR_PATH_POLYPHASE, 0)
        assert ctr.lib.ctr_plan_set_groups(h, 64) == ctr.CTR_ERR_UNSUPPORTED
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
        assert ctr.ctr_packed_weight_bytes(h) > 64 * 64 * 4 * 2 // 2
    finally:
        ctr.ctr_plan_destroy(h)
    cases = [  # (ndim, C_in, C_out, groups, in, k, s, p, op, path)
        (1, 32, 64, 32, [50], [4], [2], [1], [0], ctr.CTR_PATH_DEPTHWISE),     # multiplier 2
        (2, 16, 16, 16, [20, 20], [4, 4], [2, 2], [1, 1], [0, 0], ctr.CTR_PATH_DEPTHWISE),
        (2, 16, 16, 16, [20, 20], [3, 3], [2, 2], [1, 1], [1, 1], ctr.CTR_PATH_DEPTHWISE),
        (2, 16, 16, 16, [20, 20], [5, 16], [3, 8], [2, 4], [0, 0], ctr.CTR_PATH_GATHER),
        (2, 16, 16, 16, [20, 20], [8, 8], [4, 4], [2, 2], [0, 0], ctr.CTR_PATH_GATHER),
        (1, 16, 16, 16, [50], [5], [2], [1], [0], ctr.CTR_PATH_GATHER),        # x kernel 5
        (1, 16, 16, 16, [50], [3], [1], [1], [0], ctr.CTR_PATH_GATHER),        # x stride 1
        (1, 16, 32, 8, [50], [4], [2], [1], [0], ctr.CTR_PATH_GATHER),         # 2 ch per group
    ]
    for nd, ci, co, g, sp, k, s, p, op, path in cases:
        h = _plan(ctr, nd, 2, ci, co, sp, k, s, p, op, ctr.CTR_F32)
        try:
            ctr.ctr_plan_set_groups(h, g)
            assert ctr.ctr_plan_get_path(h) == path, (nd, ci, co, g, k, s)
            taps = int(np.prod(k))
            assert ctr.ctr_packed_weight_bytes(h) == ci * (co // g) * taps * 4
        finally:
            ctr.ctr_plan_destroy(h)
    # chained plans keep one group; a grouped plan does not chain
    a = _plan(ctr, 1, 1, 64, 32, [100], [4], [2], [1], [0], bf)
    b = _plan(ctr, 1, 1, 32, 64, [200], [4], [2], [1], [0], bf)
    c = _plan(ctr, 1, 1, 32, 32, [200], [4], [2], [1], [0], bf)
    try:
        ctr.ctr_plan_chain(a, b)
        assert ctr.lib.ctr_plan_set_groups(a, 2) == ctr.CTR_ERR_INVALID_ARG
        assert ctr.lib.ctr_plan_set_groups(b, 2) == ctr.CTR_ERR_INVALID_ARG
        ctr.ctr_plan_chain(a, None)
        ctr.ctr_plan_set_groups(c, 32)
        assert ctr.lib.ctr_plan_chain(a, c) == ctr.CTR_ERR_INVALID_ARG
    finally:
        for x in (a, b, c):
            ctr.ctr_plan_destroy(x)


def test_dilation_and_pads_without_gpu(ctr):
    """ctr_plan_set_dilation / ctr_plan_set_pads: output lengths (L_in - 1)s + (k - 1)d + 1 +
    op - p_front - p_back as the oracle's, routing of dilated plans (col2im or gather; forced
    polyphase packs the zero-inserted kernel; the depthwise kernel refuses), and invalid
    values or forced paths that cannot take them leave the plan unchanged."""
    import oracle
    f32 = ctr.CTR_F32
    arr = ctr._arr
    h = _plan(ctr, 1, 1, 32, 32, [50], [3], [2], [1], [1], f32)
    try:
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_COL2IM
        ctr.ctr_plan_set_dilation(h, [2])
        assert ctr.ctr_plan_output_shape(h, 1) == (oracle.output_size(50, 3, 2, 1, 1, 2),) == (102,)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_COL2IM
        assert "dil=1x2" in ctr.ctr_plan_describe(h)
        ctr.ctr_plan_set_pads(h, [0], [3])
        assert ctr.ctr_plan_output_shape(h, 1) == (oracle.output_size(50, 3, 2, 0, 1, 2, 3),)
        assert "pads=0x0/0x3" in ctr.ctr_plan_describe(h)
        before = ctr.ctr_plan_output_shape(h, 1)
        for bad in ([0], [-1]):
            assert ctr.lib.ctr_plan_set_dilation(h, arr(bad)) == ctr.CTR_ERR_INVALID_ARG
        assert ctr.lib.ctr_plan_set_pads(h, arr([-1]), arr([0])) == ctr.CTR_ERR_INVALID_ARG
        assert ctr.lib.ctr_plan_set_pads(h, arr([60]), arr([60])) == ctr.CTR_ERR_INVALID_ARG
        assert ctr.ctr_plan_output_shape(h, 1) == before
        # forced polyphase packs (k - 1)d + 1 = 5 dilated taps: m = 3 per phase
        col2im_packed = ctr.ctr_packed_weight_bytes(h)
        ctr.ctr_plan_set_path(h, ctr.CTR_PATH_POLYPHASE, 0)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
        assert "taps=1x3" in ctr.ctr_plan_describe(h)
        assert ctr.ctr_packed_weight_bytes(h) != col2im_packed
        ctr.ctr_plan_set_dilation(h, [1])
        assert "taps=1x2" in ctr.ctr_plan_describe(h)
    finally:
        ctr.ctr_plan_destroy(h)
    # small channel counts: gather; 2-D with unequal dilations
    h = _plan(ctr, 2, 2, 4, 3, [9, 7], [3, 2], [2, 3], [1, 0], [1, 2], f32)
    try:
        ctr.ctr_plan_set_dilation(h, [2, 3])
        ctr.ctr_plan_set_pads(h, [1, 0], [0, 2])
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_GATHER
        assert ctr.ctr_plan_output_shape(h, 2) == (oracle.output_size(9, 3, 2, 1, 1, 2, 0),
                                                   oracle.output_size(7, 2, 3, 0, 2, 3, 2))
    finally:
        ctr.ctr_plan_destroy(h)
    # undilated plans keep their path under any pads
    h = _plan(ctr, 1, 1, 64, 64, [100], [4], [2], [1], [0], ctr.CTR_BF16)
    try:
        ctr.ctr_plan_set_pads(h, [2], [0])
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
        assert ctr.ctr_plan_output_shape(h, 1) == (oracle.output_size(100, 4, 2, 2, 0, 1, 0),)
        # depthwise: dilation reroutes an automatic plan to gather, refuses a forced one
        ctr.ctr_plan_set_groups(h, 64)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_DEPTHWISE
        ctr.ctr_plan_set_path(h, ctr.CTR_PATH_DEPTHWISE, 0)
        assert ctr.lib.ctr_plan_set_dilation(h, arr([2])) == ctr.CTR_ERR_UNSUPPORTED
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_DEPTHWISE
        assert ctr.ctr_plan_output_shape(h, 1) == (oracle.output_size(100, 4, 2, 2, 0, 1, 0),)
        ctr.ctr_plan_set_path(h, ctr.CTR_PATH_AUTO, 0)
        ctr.ctr_plan_set_dilation(h, [2])
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_GATHER
    finally:
        ctr.ctr_plan_destroy(h)
    # chained plans keep their geometry
    a = _plan(ctr, 1, 1, 64, 32, [100], [4], [2], [1], [0], ctr.CTR_BF16)
    b = _plan(ctr, 1, 1, 32, 64, [200], [4], [2], [1], [0], ctr.CTR_BF16)
    try:
        ctr.ctr_plan_chain(a, b)
        assert ctr.lib.ctr_plan_set_dilation(a, arr([2])) == ctr.CTR_ERR_INVALID_ARG
        assert ctr.lib.ctr_plan_set_pads(b, arr([1]), arr([2])) == ctr.CTR_ERR_INVALID_ARG
    finally:
        ctr.ctr_plan_chain(a, None)
        ctr.ctr_plan_destroy(a)
        ctr.ctr_plan_destroy(b)


def test_streaming_plan_without_gpu(ctr):
    """ctr_plan_set_streaming: 1-D polyphase plans without padding emit s*L_in samples a call,
    carry B*(m - 1) staged frames in the workspace, and refuse what they cannot stream."""
    f32, bf = ctr.CTR_F32, ctr.CTR_BF16
    h = _plan(ctr, 1, 2, 64, 32, [50], [16], [8], [0], [0], bf)
    try:
        ws0 = ctr.ctr_workspace_bytes(h)
        ctr.ctr_plan_set_streaming(h, 1)
        assert ctr.ctr_plan_output_shape(h, 1) == (8 * 50,)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
        assert ctr.ctr_workspace_bytes(h) >= ws0 + 2 * 1 * 64 * 2   # B * (m - 1) rows
        for bad in (lambda: ctr.lib.ctr_plan_set_groups(h, 2),
                    lambda: ctr.lib.ctr_plan_set_dilation(h, ctr._arr([2])),
                    lambda: ctr.lib.ctr_plan_set_pads(h, ctr._arr([1]), ctr._arr([1]))):
            assert bad() == ctr.CTR_ERR_INVALID_ARG
        assert ctr.lib.ctr_plan_set_path(h, ctr.CTR_PATH_GATHER, 0) == ctr.CTR_ERR_UNSUPPORTED
        assert ctr.lib.ctr_plan_set_streaming(h, 2) == ctr.CTR_ERR_INVALID_ARG
        ctr.ctr_plan_set_streaming(h, 0)
        assert ctr.ctr_plan_output_shape(h, 1) == (49 * 8 + 16,)
        assert ctr.lib.ctr_plan_stream_reset(h, None) == ctr.CTR_ERR_INVALID_ARG
    finally:
        ctr.ctr_plan_destroy(h)
    # k mod s != 0 and tiny channels: forced onto the zero-padded polyphase path
    h = _plan(ctr, 1, 1, 32, 32, [40], [5], [2], [0], [0], f32)
    try:
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_COL2IM
        ctr.ctr_plan_set_streaming(h, 1)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
        assert ctr.ctr_plan_output_shape(h, 1) == (80,)
    finally:
        ctr.ctr_plan_destroy(h)
    for args in ([2, 1, 64, 32, [8, 8], [4, 4], [2, 2], [0, 0], [0, 0], f32],   # 2-D
                 [1, 1, 64, 32, [50], [4], [2], [1], [0], f32],                  # padding
                 [1, 1, 64, 32, [50], [4], [2], [0], [1], f32],                  # output_padding
                 [1, 1, 64, 32, [50], [2], [4], [0], [0], f32],                  # k < s
                 [1, 1, 64, 32, [50], [40], [2], [0], [0], f32]):                # m - 1 > 16
        h = _plan(ctr, *args)
        try:
            out = ctr.ctr_plan_output_shape(h, args[0])
            assert ctr.lib.ctr_plan_set_streaming(h, 1) == ctr.CTR_ERR_UNSUPPORTED
            assert ctr.ctr_plan_output_shape(h, args[0]) == out
        finally:
            ctr.ctr_plan_destroy(h)
    # A path forced before streaming comes back when streaming is turned off.
    h = _plan(ctr, 1, 1, 64, 32, [50], [4], [2], [0], [0], f32)
    try:
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
        ctr.ctr_plan_set_path(h, ctr.CTR_PATH_GATHER, 0)
        ctr.ctr_plan_set_streaming(h, 1)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
        ctr.ctr_plan_set_streaming(h, 0)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_GATHER
        ctr.ctr_plan_set_path(h, ctr.CTR_PATH_AUTO, 0)
        ctr.ctr_plan_set_streaming(h, 1)
        ctr.ctr_plan_set_streaming(h, 0)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
    finally:
        ctr.ctr_plan_destroy(h)
    a = _plan(ctr, 1, 1, 64, 32, [100], [4], [2], [0], [0], bf)
    b = _plan(ctr, 1, 1, 32, 64, [202], [4], [2], [0], [0], bf)
    try:
        ctr.ctr_plan_set_streaming(a, 1)
        assert ctr.lib.ctr_plan_chain(a, b) == ctr.CTR_ERR_INVALID_ARG
        ctr.ctr_plan_set_streaming(a, 0)
        ctr.ctr_plan_chain(a, b)
        assert ctr.lib.ctr_plan_set_streaming(a, 1) == ctr.CTR_ERR_INVALID_ARG
        assert ctr.lib.ctr_plan_set_streaming(b, 1) == ctr.CTR_ERR_INVALID_ARG
    finally:
        ctr.ctr_plan_chain(a, None)
        ctr.ctr_plan_destroy(a)
        ctr.ctr_plan_destroy(b)


def test_f16_plans_without_gpu(ctr):
    """CTR_F16 plans: the tensor-core paths pack one 16-bit plane like bf16; grouped fp16
    plans run the gather kernel (no depthwise kernel for fp16); the iSTFT plan refuses fp16;
    an unknown dtype code is invalid."""
    f16, bf = ctr.CTR_F16, ctr.CTR_BF16
    a = _plan(ctr, 1, 1, 512, 256, [2000], [16], [8], [4], [0], f16)
    b = _plan(ctr, 1, 1, 512, 256, [2000], [16], [8], [4], [0], bf)
    try:
        assert ctr.ctr_plan_get_path(a) == ctr.CTR_PATH_POLYPHASE
        assert "prec=f16" in ctr.ctr_plan_describe(a)
        assert ctr.ctr_packed_weight_bytes(a) == ctr.ctr_packed_weight_bytes(b)
        assert ctr.ctr_workspace_bytes(a) == ctr.ctr_workspace_bytes(b)
    finally:
        ctr.ctr_plan_destroy(a)
        ctr.ctr_plan_destroy(b)
    h = _plan(ctr, 2, 1, 16, 16, [9, 12], [4, 4], [2, 2], [1, 1], [0, 0], f16)
    try:
        ctr.ctr_plan_set_groups(h, 16)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_GATHER
        assert ctr.lib.ctr_plan_set_path(h, ctr.CTR_PATH_DEPTHWISE, 0) == ctr.CTR_ERR_UNSUPPORTED
    finally:
        ctr.ctr_plan_destroy(h)
    ist = ctypes.c_void_p()
    assert ctr.lib.ctr_istft_create(ctypes.byref(ist), 1, 64, 16, 9, 0, 0, f16) == ctr.CTR_ERR_UNSUPPORTED
    out = ctypes.c_void_p()
    args = [ctypes.byref(out), 1, 1, 16, 8, ctr._arr([64]), ctr._arr([4]), ctr._arr([2]),
            ctr._arr([1]), None, 3]
    assert ctr.lib.ctr_plan_create(*args) == ctr.CTR_ERR_INVALID_ARG


def test_layout_without_gpu(ctr):
    """ctr_plan_set_layout: NHWC keeps the path and sizes of the tensor-core and gather paths;
    a grouped depthwise geometry goes to gather; streaming and a forced depthwise path refuse
    it and stay as they were; an unknown value is invalid."""
    f32, bf = ctr.CTR_F32, ctr.CTR_BF16
    h = _plan(ctr, 1, 1, 512, 256, [2000], [16], [8], [4], [0], f32)
    try:
        ws = ctr.ctr_workspace_bytes(h)
        ctr.ctr_plan_set_layout(h, ctr.CTR_LAYOUT_NHWC)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_POLYPHASE
        assert ctr.ctr_workspace_bytes(h) == ws and " nhwc" in ctr.ctr_plan_describe(h)
        assert ctr.lib.ctr_plan_set_layout(h, 2) == ctr.CTR_ERR_INVALID_ARG
        ctr.ctr_plan_set_layout(h, ctr.CTR_LAYOUT_NCHW)
        assert " nhwc" not in ctr.ctr_plan_describe(h)
    finally:
        ctr.ctr_plan_destroy(h)
    h = _plan(ctr, 2, 1, 16, 16, [9, 12], [4, 4], [2, 2], [1, 1], [0, 0], bf)
    try:
        ctr.ctr_plan_set_groups(h, 16)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_DEPTHWISE
        ctr.ctr_plan_set_layout(h, ctr.CTR_LAYOUT_NHWC)
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_GATHER
        ctr.ctr_plan_set_layout(h, ctr.CTR_LAYOUT_NCHW)
        ctr.ctr_plan_set_path(h, ctr.CTR_PATH_DEPTHWISE, 0)
        assert ctr.lib.ctr_plan_set_layout(h, ctr.CTR_LAYOUT_NHWC) == ctr.CTR_ERR_UNSUPPORTED
        assert ctr.ctr_plan_get_path(h) == ctr.CTR_PATH_DEPTHWISE
    finally:
        ctr.ctr_plan_destroy(h)
    h = _plan(ctr, 1, 1, 64, 32, [50], [16], [8], [0], [0], bf)
    try:
        ctr.ctr_plan_set_streaming(h, 1)
        assert ctr.lib.ctr_plan_set_layout(h, ctr.CTR_LAYOUT_NHWC) == ctr.CTR_ERR_UNSUPPORTED
        ctr.ctr_plan_set_streaming(h, 0)
        ctr.ctr_plan_set_layout(h, ctr.CTR_LAYOUT_NHWC)
        assert ctr.lib.ctr_plan_set_streaming(h, 1) == ctr.CTR_ERR_UNSUPPORTED
    finally:
        ctr.ctr_plan_destroy(h)


def test_fusable_pairs_without_gpu(ctr):
    """ctr_plan_fusable: a chained bf16/fp16 pair 128 -> 64 -> 32 with stride 2 qualifies;
    fp32, a middle width other than 64, an unchained plan or a further chain do not; the
    fused call refuses what does not qualify before launching anything."""
    def pair(dt, c1=64, c2=32, k=4, s=2):
        a = _plan(ctr, 1, 1, 128, c1, [500], [k], [s], [1], [0], dt)
        b = _plan(ctr, 1, 1, c1, c2, [ctr.ctr_plan_output_shape(a, 1)[0]], [4], [2], [1], [0], dt)
        ctr.ctr_plan_chain(a, b)
        return a, b
    for dt, want in ((ctr.CTR_BF16, 1), (ctr.CTR_F16, 1), (ctr.CTR_F32, 0)):
        a, b = pair(dt)
        try:
            assert ctr.lib.ctr_plan_fusable(a) == want, ctr.ctr_plan_describe(a)
            assert ctr.lib.ctr_plan_fusable(b) == 0
        finally:
            ctr.ctr_plan_destroy(a)
            ctr.ctr_plan_destroy(b)
    a, b = pair(ctr.CTR_BF16, c1=32)
    try:
        assert ctr.lib.ctr_plan_fusable(a) == 0
    finally:
        ctr.ctr_plan_destroy(a)
        ctr.ctr_plan_destroy(b)
    a, b = pair(ctr.CTR_BF16)
    c = _plan(ctr, 1, 1, 32, 64, [ctr.ctr_plan_output_shape(b, 1)[0]], [4], [2], [1], [0], ctr.CTR_BF16)
    try:
        ctr.ctr_plan_chain(b, c)
        assert ctr.lib.ctr_plan_fusable(a) == 0      # the second plan feeds a third
        p = ctypes.c_void_p(1 << 20)
        assert ctr.lib.ctr_forward_fused(a, p, p, None, p, None, p, None) == ctr.CTR_ERR_NOT_PREPARED
        ctr.ctr_plan_chain(a, None)
        assert ctr.lib.ctr_forward_fused(a, p, p, None, p, None, p, None) == ctr.CTR_ERR_INVALID_ARG
    finally:
        ctr.ctr_plan_chain(b, None)
        for h in (a, b, c):
            ctr.ctr_plan_destroy(h)


def test_auto_pad_without_gpu(ctr):
    """ONNX auto_pad / output_shape resolve into front and back pads: SAME_* give
    L_in * stride outputs with an odd total padding's extra sample at the end (UPPER) or in
    front (LOWER); an explicit output_shape sets the total; VALID pads nothing; a longer
    output than the unpadded result is refused and leaves the plan as it was."""
    f32 = ctr.CTR_F32
    # 1-D, k = 3, s = 2, L = 5: unpadded length (5 - 1)*2 + 3 = 11, SAME target 10 (total 1)
    for mode, front, back in ((ctr.CTR_AUTO_PAD_SAME_UPPER, 0, 1),
                              (ctr.CTR_AUTO_PAD_SAME_LOWER, 1, 0)):
        h = _plan(ctr, 1, 1, 32, 64, [5], [3], [2], [0], [0], f32)
        try:
            ctr.ctr_plan_set_auto_pad(h, mode)
            assert ctr.ctr_plan_output_shape(h, 1) == (10,)
            d = ctr.ctr_plan_describe(h)
            assert "pads=0x%d/0x%d" % (front, back) in d, d
        finally:
            ctr.ctr_plan_destroy(h)
    # 2-D with dilation 2 in x: unpadded (4-1)*2 + (3-1)*2 + 1 = 11 along x, 4x4/s2 along y
    h = _plan(ctr, 2, 1, 32, 64, [4, 4], [4, 3], [2, 2], [0, 0], [0, 1], f32)
    try:
        ctr.ctr_plan_set_dilation(h, ctr._arr([1, 2]))
        ctr.ctr_plan_set_auto_pad(h, ctr.CTR_AUTO_PAD_SAME_UPPER)
        assert ctr.ctr_plan_output_shape(h, 2) == (8, 8)       # totals 2 and 4 (op 1 included)
        assert "pads=1x2/1x2" in ctr.ctr_plan_describe(h)
        ctr.ctr_plan_set_auto_pad(h, ctr.CTR_AUTO_PAD_NOTSET, [9, 7])   # totals 1 and 5
        assert ctr.ctr_plan_output_shape(h, 2) == (9, 7)
        assert "pads=1x3/0x2" in ctr.ctr_plan_describe(h)
        ctr.ctr_plan_set_auto_pad(h, ctr.CTR_AUTO_PAD_VALID)
        assert ctr.ctr_plan_output_shape(h, 2) == (10, 12)
        # longer than the unpadded result: refused, plan unchanged
        assert ctr.lib.ctr_plan_set_auto_pad(h, 0, ctr._arr([11, 12])) == ctr.CTR_ERR_UNSUPPORTED
        assert ctr.ctr_plan_output_shape(h, 2) == (10, 12)
        assert ctr.lib.ctr_plan_set_auto_pad(h, 4, None) == ctr.CTR_ERR_INVALID_ARG
        assert ctr.lib.ctr_plan_set_auto_pad(h, 0, ctr._arr([0, 5])) == ctr.CTR_ERR_INVALID_ARG
    finally:
        ctr.ctr_plan_destroy(h)


def test_istft_plan_without_gpu(ctr):
    """ctr_istft_*: argument checks, output length, workspace size; no window -> not prepared."""
    h = ctr.ctr_istft_create(4, 4096, 1024, 343)
    try:
        assert ctr.ctr_istft_output_length(h) == 354304
        ws = ctr.ctr_istft_workspace_bytes(h)
        assert ws >= 4 * 343 * 4096 * 4 + 4096 * 12
        assert "n_fft=4096" in ctr.ctr_istft_describe(h)
        assert ctr.lib.ctr_istft_bind_workspace(h, ctypes.c_void_p(4096 + 8), ws) == \
            ctr.CTR_ERR_MISALIGNED
        assert ctr.lib.ctr_istft_bind_workspace(h, ctypes.c_void_p(4096), ws - 1) == \
            ctr.CTR_ERR_NO_WORKSPACE
        st = ctr.lib.ctr_istft_forward(h, ctypes.c_void_p(256), None, ctypes.c_void_p(256), None)
        assert st == ctr.CTR_ERR_NO_WORKSPACE
        ctr.ctr_istft_bind_workspace(h, ctypes.c_void_p(4096), ws)
        st = ctr.lib.ctr_istft_forward(h, ctypes.c_void_p(256), None, ctypes.c_void_p(256), None)
        assert st == ctr.CTR_ERR_NOT_PREPARED
        assert ctr.lib.ctr_istft_set_timing_events(h, ctypes.c_void_p(16), None) == \
            ctr.CTR_ERR_INVALID_ARG
    finally:
        ctr.ctr_istft_destroy(h)
    assert ctr.ctr_istft_output_length(ctr.ctr_istft_create(1, 8, 2, 0)) == 6   # (0-1)*2 + 8
    for bad in [(1, 6, 2, 3, 0, 0), (1, 2, 1, 3, 0, 0), (1, 16384, 4, 3, 0, 0), (1, 16, 0, 3, 0, 0),
                (1, 16, 4, 3, 0, 4), (1, 16, 4, -1, 0, 0), (-1, 16, 4, 3, 0, 0),
                (1, 16, 4, 1, 8, 0)]:
        with pytest.raises(ctr.CtrError) as e:
            ctr.ctr_istft_create(*bad)
        assert e.value.status == ctr.CTR_ERR_INVALID_ARG, bad
    with pytest.raises(ctr.CtrError) as e:
        ctr.ctr_istft_create(1, 16, 4, 3, 0, 0, ctr.CTR_BF16)
    assert e.value.status == ctr.CTR_ERR_UNSUPPORTED
    assert ctr.lib.ctr_istft_workspace_bytes(None) == 0
    ctr.ctr_istft_destroy(None)


def test_tile_model_choices_without_gpu(ctr):
    """The tile model's (BN, split-K) for the fp32 shapes its constants were fitted to: for
    each, the fastest of the BN 64/128/256 x split-K grid in forced-tile timings on GB300
    with inputs and weights cold in HBM (the benchmark's regime)."""
    cases = [  # (ndim, B, C_in, C_out, L, k, s, p) -> (BN, splits)
        ((1, 1, 512, 256, [2000], [16], [8], [4]), (256, 1)),           # codec upsampler
        ((2, 1, 128, 64, [128, 128], [4, 4], [2, 2], [1, 1]), (256, 1)),  # 2-D decoder
        ((1, 4, 4098, 1, [343], [4096], [1024], [0]), (256, 3)),        # iSTFT
        ((1, 2, 256, 128, [1500], [8], [4], [2]), (128, 1)),
        ((1, 1, 1024, 64, [4000], [4], [2], [1]), (128, 4)),
    ]
    for (nd, B, ci, co, L, k, s, p), (bn, sp) in cases:
        h = _plan(ctr, nd, B, ci, co, L, k, s, p, [0] * nd, ctr.CTR_F32)
        try:
            d = ctr.ctr_plan_describe(h)
            if "sms=152 " not in d:
                pytest.skip("the model's choices are pinned for 152 SMs: " + d)
            assert "BN %d," % bn in d and "splits=%d " % sp in d, d
        finally:
            ctr.ctr_plan_destroy(h)


def test_xring_mode_selection_without_gpu(ctr):
    """fp32 polyphase plans on 256-row tiles with four or more taps along x run the GEMM in
    X-ring mode, while a split-K factor leaves every unit at least one channel slice; two-tap
    layers, 16-bit I/O and other tile widths keep the default stage ring."""
    def desc(args, dtype=None, bn=256, split=0):
        nd = len(args[3])
        h = _plan(ctr, nd, *args, [0] * nd, ctr.CTR_F32 if dtype is None else dtype)
        try:
            ctr.ctr_plan_set_path(h, ctr.CTR_PATH_POLYPHASE, split)
            ctr.ctr_plan_set_tile(h, bn)
            return ctr.ctr_plan_describe(h)
        finally:
            ctr.ctr_plan_destroy(h)
    four_taps = (1, 64, 40, [300], [16], [4], [0])      # C_in 64: two channel slices
    assert " x-ring" in desc(four_taps)
    assert " x-ring" in desc(four_taps, split=2)
    assert " x-ring" not in desc(four_taps, split=3)    # a unit would get no channel slice
    assert " x-ring" not in desc(four_taps, bn=128)
    assert " x-ring" not in desc(four_taps, dtype=ctr.CTR_BF16)
    assert " x-ring" not in desc((1, 64, 40, [300], [8], [4], [0]))   # two taps
    assert " x-ring" in desc((4, 4098, 1, [343], [4096], [1024], [0]), bn=0)   # the iSTFT, auto
