"""Full-size rounds through moe_round (the launch configuration the benchmark times).

The 35B-A3B-shaped 40-layer stack serves the 1-, 4- and 16-row workloads (same layer
shape and seed; only the rows differ); the 512-expert 48-layer stack serves the
3-row workload.  |U| of every layer is compared with the oracle's union; outputs of
sampled layers are compared with the oracle element by element.
"""
import numpy as np
import pytest
import torch

import oracle
import spec_verify_layer_gb300 as mv
import syngen
from gpu_helpers import Stack, assert_close, stream_of

pytestmark = pytest.mark.gpu


def round_case(stack, cfg, n_rows, sigma, use_graph, check_layers, tail=0):
    dev = stack.device
    L = len(stack.layers)
    H = cfg.hidden
    xs = np.stack([syngen.rows(cfg, l, n_rows, sigma) for l in range(L)])
    x = torch.from_numpy(xs.view(np.int16)).to(dev)
    out = torch.full((L, n_rows, H), float("nan"), device=dev)
    stats = torch.full((L,), -1, dtype=torch.int32, device=dev)
    ws = stack.ws(n_rows)
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        mv.moe_round(stack.handle, [ly.w for ly in stack.layers], x.data_ptr(), n_rows, out.data_ptr(),
                     stats.data_ptr(), ws.data_ptr(), ws.numel(), use_graph, s.cuda_stream)
        if use_graph:  # replay once more: same ingress buffers, same result
            first = out.clone()
            mv.moe_round(stack.handle, [ly.w for ly in stack.layers], x.data_ptr(), n_rows,
                         out.data_ptr(), stats.data_ptr(), ws.data_ptr(), ws.numel(), True, s.cuda_stream)
    assert mv.moe_last_device_status(stack.handle, s.cuda_stream) == mv.MOE_OK
    assert mv.moe_last_launch_count(stack.handle) == 1  # one fused round kernel
    if use_graph:
        assert torch.equal(first, out)
    st = stats.cpu().numpy()
    got = out.cpu().numpy()
    for l in range(L):
        rt = oracle.route(syngen.router(cfg, l), xs[l], cfg.top_k, tail)
        assert st[l] == rt.union.size, f"layer {l}: |U| {st[l]} vs {rt.union.size}"
    for l in check_layers:
        router = syngen.router(cfg, l)
        rt = oracle.route(router, xs[l], cfg.top_k, tail)
        ref = oracle.layer(router, xs[l], cfg.top_k, rt.union, syngen.experts_stacked(cfg, l, rt.union),
                           tail)
        assert_close(got[l], ref, f"{cfg.name} R={n_rows} layer {l}")
    return got, st


@pytest.fixture(scope="module")
def a3b_stack():
    cfg = syngen.CONFIGS["a3b_r1"]
    s = Stack(cfg, n_layers=cfg.layers)
    yield s
    s.close()


@pytest.mark.parametrize("name", ["a3b_r1", "a3b_r4", "a3b_r16"])
def test_a3b_round(a3b_stack, name):
    cfg = syngen.CONFIGS[name]
    round_case(a3b_stack, cfg, cfg.rows, cfg.row_sigma, True, check_layers=(0, 17, 39))


def test_graph_equals_eager(a3b_stack):
    cfg = syngen.CONFIGS["a3b_r4"]
    g, sg = round_case(a3b_stack, cfg, cfg.rows, cfg.row_sigma, True, check_layers=())
    e, se = round_case(a3b_stack, cfg, cfg.rows, cfg.row_sigma, False, check_layers=())
    np.testing.assert_array_equal(g, e)
    np.testing.assert_array_equal(sg, se)


def test_tiny_round_all_layers():
    cfg = syngen.CONFIGS["tiny"]
    s = Stack(cfg, n_layers=4)
    try:
        round_case(s, cfg, 3, 0.5, True, check_layers=range(4))
    finally:
        s.close()


def test_e512_round():
    cfg = syngen.CONFIGS["e512_r3"]
    s = Stack(cfg, n_layers=cfg.layers)
    try:
        round_case(s, cfg, cfg.rows, cfg.row_sigma, True, check_layers=(0, 23, 47))
    finally:
        s.close()


def test_a3b_round_tail_skip(a3b_stack):
    """The 4-row round with the page's tail skip (rank 7): |U| per layer as the oracle's
    mirror of the rule, sampled layers within tolerance; switching the skip off again
    re-captures the round graph (the setting is part of its key)."""
    cfg = syngen.CONFIGS["a3b_r4"]
    _, plain = round_case(a3b_stack, cfg, cfg.rows, cfg.row_sigma, True, check_layers=())
    try:
        mv.moe_set_tail_skip(a3b_stack.handle, 7)
        _, skipped = round_case(a3b_stack, cfg, cfg.rows, cfg.row_sigma, True, check_layers=(0, 39),
                                tail=7)
    finally:
        mv.moe_set_tail_skip(a3b_stack.handle, 0)
    assert (skipped <= plain).all() and skipped.sum() < plain.sum()
    _, again = round_case(a3b_stack, cfg, cfg.rows, cfg.row_sigma, True, check_layers=())
    np.testing.assert_array_equal(again, plain)


def test_host_buffer_round_equals_device_round(a3b_stack):
    """moe_round_host (rows copied in from host memory, outputs copied back to host memory,
    on the caller's stream around the round) gives moe_round's outputs bitwise: from
    page-locked buffers with the graph and eagerly, and from pageable numpy buffers with
    the work only enqueued (sync = 0).  Wrong arguments are rejected with nothing enqueued."""
    cfg = syngen.CONFIGS["a3b_r4"]
    R, H, L = cfg.rows, cfg.hidden, len(a3b_stack.layers)
    want, want_stats = round_case(a3b_stack, cfg, R, cfg.row_sigma, True, check_layers=())
    xs = np.stack([syngen.rows(cfg, l, R, cfg.row_sigma) for l in range(L)])
    dev = a3b_stack.device
    x_dev = torch.empty((L, R, H), dtype=torch.int16, device=dev)
    out_dev = torch.full((L, R, H), float("nan"), device=dev)
    stats = torch.full((L,), -1, dtype=torch.int32, device=dev)
    ws = a3b_stack.ws(R)
    wl = [ly.w for ly in a3b_stack.layers]
    s = torch.cuda.Stream(dev)

    def call(x_host, out_host, rows=R, layers=wl, use_graph=True, sync=True):
        mv.moe_round_host(a3b_stack.handle, a3b_stack.dims, layers, x_host, rows, out_host, x_dev.data_ptr(),
                          out_dev.data_ptr(), stats.data_ptr(), ws.data_ptr(), ws.numel(), use_graph, sync,
                          s.cuda_stream)

    xh = torch.from_numpy(xs.view(np.int16)).pin_memory()
    oh = torch.empty((L, R, H), dtype=torch.float32).pin_memory()
    for use_graph in (True, True, False):  # capture, replay, eager
        oh.fill_(float("nan"))
        call(xh.data_ptr(), oh.data_ptr(), use_graph=use_graph)
        np.testing.assert_array_equal(oh.numpy(), want)
    np.testing.assert_array_equal(stats.cpu().numpy(), want_stats)

    xp = np.ascontiguousarray(xs.view(np.uint16))
    op = np.full((L, R, H), np.nan, dtype=np.float32)
    call(xp.ctypes.data, op.ctypes.data, sync=False)
    s.synchronize()
    np.testing.assert_array_equal(op, want)
    assert mv.moe_last_device_status(a3b_stack.handle, s.cuda_stream) == mv.MOE_OK

    out_dev.fill_(float("nan"))
    torch.cuda.synchronize(dev)
    for kw in (dict(rows=0), dict(rows=a3b_stack.dims.max_rows + 1), dict(layers=[])):
        with pytest.raises(mv.MoeError) as ei:
            call(xh.data_ptr(), oh.data_ptr(), **kw)
        assert ei.value.code == mv.MOE_EINVAL
    with pytest.raises(mv.MoeError) as ei:
        call(None, oh.data_ptr())
    assert ei.value.code == mv.MOE_EINVAL
    s.synchronize()
    assert torch.isnan(out_dev).all()  # no round ran
