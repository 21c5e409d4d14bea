"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Routing (top-k ids in rank order, the union) must be bit-exact; weights within 1e-6;
layer outputs within max-abs 2e-3 and relative-L2 1e-3 of the oracle's fp64 result.
"""
import numpy as np
import pytest
import torch

import oracle
import spec_verify_layer_gb300 as mv
import syngen
from gpu_helpers import TOL_W, Stack, assert_close, compare, stream_of

pytestmark = pytest.mark.gpu

SHAPES = ["tiny", "a3b_r1", "e512_r3"]   # distinct layer shapes (a3b_r4 / a3b_r16 share a3b_r1's)
# Row counts on both kernels: up to 12 rows the split kernel (CUDA cores), from 13 the
# tensor-core kernel; 5 and 7 rows are the counts just above and below the old staging
# limit, 12 and 13 the two sides of the kernel switch.
ROWS = {"tiny": [(1, 0.0), (3, 0.5), (4, 0.5)],
        "a3b_r1": [(1, 0.0), (4, 0.5), (5, 0.5), (6, 0.5), (7, 0.5), (12, 0.5), (13, 0.5), (16, 0.1)],
        "e512_r3": [(1, 0.0), (1, 1.0), (3, 0.5)]}


@pytest.fixture(scope="module", params=SHAPES)
def stack(request):
    cfg = syngen.CONFIGS[request.param]
    s = Stack(cfg, n_layers=2)
    yield s
    s.close()


def run_route(s, layer, xb):
    dev = s.device
    R, k, E = xb.shape[0], s.cfg.top_k, s.cfg.experts
    x = s.x_dev(xb)
    ids = torch.full((R, k), -1, dtype=torch.int32, device=dev)
    w = torch.zeros((R, k), dtype=torch.float32, device=dev)
    uni = torch.full((E,), -1, dtype=torch.int32, device=dev)
    nu = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = s.ws(R)
    st = stream_of(dev)
    mv.moe_route(s.handle, s.layers[layer].w, x.data_ptr(), R, ids.data_ptr(), w.data_ptr(),
                 uni.data_ptr(), nu.data_ptr(), ws.data_ptr(), ws.numel(), st)
    assert mv.moe_last_device_status(s.handle, st) == mv.MOE_OK
    n = int(nu.item())
    return ids.cpu().numpy(), w.cpu().numpy(), uni.cpu().numpy()[:n]


def run_layer(s, layer, xb):
    dev = s.device
    R = xb.shape[0]
    x = s.x_dev(xb)
    out = torch.full((R, s.cfg.hidden), float("nan"), dtype=torch.float32, device=dev)
    ws = s.ws(R)
    st = stream_of(dev)
    mv.moe_decode_layer(s.handle, s.layers[layer].w, x.data_ptr(), R, out.data_ptr(), ws.data_ptr(),
                        ws.numel(), st)
    assert mv.moe_last_device_status(s.handle, st) == mv.MOE_OK
    assert mv.moe_last_launch_count(s.handle) == 1
    return out.cpu().numpy()


def test_route_bit_exact(stack):
    cfg = stack.cfg
    for layer in range(2):
        router = syngen.router(cfg, layer)
        for R, sigma in ROWS[cfg.name]:
            xb = stack.rows(layer, R, sigma)
            ids, w, uni = run_route(stack, layer, xb)
            rt = oracle.route(router, xb, cfg.top_k)
            np.testing.assert_array_equal(ids, rt.ids)
            np.testing.assert_array_equal(uni, rt.union)
            assert np.abs(w - rt.w).max() <= TOL_W
            assert np.abs(w.astype(np.float64).sum(axis=1) - 1).max() <= 1e-6


def test_layer_matches_oracle(stack):
    cfg = stack.cfg
    for layer in range(2):
        router = syngen.router(cfg, layer)
        for R, sigma in ROWS[cfg.name]:
            xb = stack.rows(layer, R, sigma)
            got = run_layer(stack, layer, xb)
            rt = oracle.route(router, xb, cfg.top_k)
            ref = oracle.layer(router, xb, cfg.top_k, rt.union, syngen.experts_stacked(cfg, layer, rt.union))
            assert_close(got, ref, f"{cfg.name} layer {layer} R={R}")


def test_rows_are_independent_bitwise(stack):
    """A row's output is bit-identical alone, inside a batch, and at any position."""
    cfg = stack.cfg
    R = 4
    xb = stack.rows(0, R, 0.5)
    full = run_layer(stack, 0, xb)
    perm = np.array([2, 0, 3, 1])
    rot = run_layer(stack, 0, xb[perm].copy())
    np.testing.assert_array_equal(rot, full[perm])
    for r in range(R):
        alone = run_layer(stack, 0, xb[r:r + 1].copy())
        np.testing.assert_array_equal(alone[0], full[r])


def test_repeat_runs_are_bitwise_equal(stack):
    xb = stack.rows(1, 3, 0.5)
    a = run_layer(stack, 1, xb)
    b = run_layer(stack, 1, xb)
    np.testing.assert_array_equal(a, b)


# ---- edge cases on the tiny shape -----------------------------------------------

def _tiny_stack(**kw):
    cfg = syngen.CONFIGS["tiny"].with_(**kw)
    return Stack(cfg, n_layers=1)


@pytest.mark.parametrize("inter", [1024, 1536])
def test_intermediate_sizes_in_several_k_chunks(inter):
    """I / 32 not a multiple of 24: the tensor-core down pass stages each group's h' in
    two K chunks (one copy per position, exact adds per chunk); 13 and 16 rows on that
    kernel and 4 rows on the split kernel against the oracle, two layers."""
    s = Stack(syngen.CONFIGS["tiny"].with_(inter=inter, top_k=4), n_layers=2)
    try:
        for layer in range(2):
            router = syngen.router(s.cfg, layer)
            for R, sigma in ((4, 0.5), (13, 0.5), (16, 0.1)):
                xb = s.rows(layer, R, sigma)
                got = run_layer(s, layer, xb)
                rt = oracle.route(router, xb, s.cfg.top_k)
                ref = oracle.layer(router, xb, s.cfg.top_k, rt.union, syngen.experts_stacked(s.cfg, layer, rt.union))
                assert_close(got, ref, f"I={inter} layer {layer} R={R}")
    finally:
        s.close()


def test_single_expert_union():
    s = _tiny_stack(top_k=1)
    try:
        xb = s.rows(0, 5, 0.0)  # 5 identical rows, k = 1 -> |U| = 1
        ids, w, uni = run_route(s, 0, xb)
        assert uni.size == 1 and (ids == uni[0]).all() and (w == 1.0).all()
        got = run_layer(s, 0, xb)
        rt = oracle.route(syngen.router(s.cfg, 0), xb, 1)
        ref = oracle.layer(syngen.router(s.cfg, 0), xb, 1, rt.union, syngen.experts_stacked(s.cfg, 0, rt.union))
        assert_close(got, ref, "U=1")
        assert (got == got[0]).all()
    finally:
        s.close()


def test_k_equals_e_all_experts():
    s = _tiny_stack(top_k=8)
    try:
        xb = s.rows(0, 3, 0.5)
        ids, w, uni = run_route(s, 0, xb)
        assert uni.tolist() == list(range(8))
        got = run_layer(s, 0, xb)
        ref = oracle.layer(syngen.router(s.cfg, 0), xb, 8, np.arange(8), syngen.experts_stacked(s.cfg, 0, range(8)))
        assert_close(got, ref, "k=E")
    finally:
        s.close()


def test_max_rows_and_ragged_counts():
    s = _tiny_stack()
    try:
        router = syngen.router(s.cfg, 0)
        ew = syngen.experts_stacked(s.cfg, 0, range(8))
        for R in (1, 2, 5, 7, 16, 31, 32):
            xb = s.rows(0, R, 0.7)
            got = run_layer(s, 0, xb)
            ref = oracle.layer(router, xb, s.cfg.top_k, np.arange(8), ew)
            assert_close(got, ref, f"R={R}")
            ids, _, uni = run_route(s, 0, xb)
            rt = oracle.route(router, xb, s.cfg.top_k)
            np.testing.assert_array_equal(ids, rt.ids)
            np.testing.assert_array_equal(uni, rt.union)
    finally:
        s.close()


def test_forced_router_ties_pick_lower_id():
    cfg = syngen.CONFIGS["tiny"]
    s = _tiny_stack()
    try:
        router = syngen.router(cfg, 0).copy()
        router[6] = router[1]     # experts 1 and 6 tie for every row
        router[3] = router[5]     # experts 3 and 5 tie for every row
        s.layers[0].router.copy_(torch.from_numpy(router))
        xb = s.rows(0, 8, 1.0)
        ids, w, uni = run_route(s, 0, xb)
        rt = oracle.route(router, xb, cfg.top_k)
        np.testing.assert_array_equal(ids, rt.ids)
        np.testing.assert_array_equal(uni, rt.union)
        got = run_layer(s, 0, xb)
        ref = oracle.layer(router, xb, cfg.top_k, np.arange(8), syngen.experts_stacked(cfg, 0, range(8)))
        assert_close(got, ref, "ties")
    finally:
        s.close()


def test_one_row_counting_path_ties_pick_lower_id():
    """One-row rounds rank the experts by counting (E a power of two >= 32): three
    experts with identical router rows tie at the top for the row and must come out in
    id order, the same as the oracle, and the row's output must equal the same row's
    inside a three-row round (which takes the selection-rounds path) bit for bit."""
    cfg = syngen.CONFIGS["tiny"].with_(experts=64, top_k=4)
    s = Stack(cfg, n_layers=1)
    try:
        xb = s.rows(0, 3, 0.5)
        x0 = np.array([oracle.bf16_to_float(int(v)) for v in xb[0]], dtype=np.float32)
        router = syngen.router(cfg, 0).copy()
        router[40] = 0.05 * x0      # far above every other logit of row 0
        router[3] = router[40]
        router[10] = router[40]
        router[50] = router[20]     # a tie lower down
        s.layers[0].router.copy_(torch.from_numpy(router))
        ids, w, uni = run_route(s, 0, xb[:1].copy())
        rt = oracle.route(router, xb[:1], cfg.top_k)
        np.testing.assert_array_equal(ids, rt.ids)
        np.testing.assert_array_equal(uni, rt.union)
        assert list(ids[0][:3]) == [3, 10, 40]
        assert np.abs(w - rt.w).max() <= TOL_W
        alone = run_layer(s, 0, xb[:1].copy())
        full = run_layer(s, 0, xb)
        np.testing.assert_array_equal(alone[0], full[0])
        ref = oracle.layer(router, xb[:1], cfg.top_k, rt.union, syngen.experts_stacked(cfg, 0, rt.union))
        assert_close(alone, ref, "one-row ties")
    finally:
        s.close()


def test_zero_and_subnormal_scales():
    """Blocks with zero scale contribute nothing; subnormal fp16 scales are honoured."""
    cfg = syngen.CONFIGS["tiny"]
    from spec_verify_layer_gb300.weights import upload_layer
    dims = mv.make_dims(cfg.hidden, cfg.experts, cfg.top_k, cfg.inter, 4)

    def ew_fn(e):
        w = syngen.expert(cfg, 0, e)
        w.sg[::3] = 0                    # zero scales
        w.su[1::5] = 0x0001              # smallest subnormal
        w.sd[:, ::2] = 0x03FF            # largest subnormal
        return w
    dev = torch.device("cuda")
    layer = upload_layer(dims, syngen.router(cfg, 0), ew_fn, dev)
    h = mv.moe_create(dims, 0)
    try:
        xb = syngen.rows(cfg, 0, 4, 0.5)
        x = torch.from_numpy(xb.view(np.int16)).to(dev)
        out = torch.empty(4, cfg.hidden, device=dev)
        from spec_verify_layer_gb300.weights import workspace
        ws = workspace(dims, 4, dev)
        st = stream_of(dev)
        mv.moe_decode_layer(h, layer.w, x.data_ptr(), 4, out.data_ptr(), ws.data_ptr(), ws.numel(), st)
        assert mv.moe_last_device_status(h, st) == mv.MOE_OK
        ews = [ew_fn(e) for e in range(8)]
        stacked = syngen.ExpertW(*(np.ascontiguousarray(np.stack([getattr(w, f) for w in ews]))
                                   for f in ("qg", "sg", "qu", "su", "qd", "sd")))
        ref = oracle.layer(syngen.router(cfg, 0), xb, cfg.top_k, np.arange(8), stacked)
        assert_close(out.cpu().numpy(), ref, "scales")
    finally:
        mv.moe_destroy(h)


# ---- boundary errors on a device ---------------------------------------------------

def test_argument_errors_on_device():
    s = _tiny_stack()
    try:
        dev = s.device
        xb = s.rows(0, 2, 0.5)
        x = s.x_dev(xb)
        out = torch.empty(2, s.cfg.hidden, device=dev)
        ws = s.ws(2)
        st = stream_of(dev)
        lib = mv.lib()
        import ctypes
        w = s.layers[0].w
        rc = lib.moe_decode_layer(s.handle, ctypes.byref(w), x.data_ptr(), 2, out.data_ptr(),
                                  ws.data_ptr(), 100, st)
        assert rc == mv.MOE_EWORKSPACE
        rc = lib.moe_decode_layer(s.handle, ctypes.byref(w), x.data_ptr() + 2, 2, out.data_ptr(),
                                  ws.data_ptr(), ws.numel(), st)
        assert rc == mv.MOE_EINVAL
        rc = lib.moe_decode_layer(s.handle, ctypes.byref(w), x.data_ptr(), 0, out.data_ptr(),
                                  ws.data_ptr(), ws.numel(), st)
        assert rc == mv.MOE_EINVAL
        rc = lib.moe_decode_layer(s.handle, ctypes.byref(w), x.data_ptr(), 33, out.data_ptr(),
                                  ws.data_ptr(), ws.numel(), st)
        assert rc == mv.MOE_EINVAL
        bad = mv.make_layer_w(w.router, w.gateup_nib + 8, w.gateup_scale, w.down_nib, w.down_scale)
        rc = lib.moe_decode_layer(s.handle, ctypes.byref(bad), x.data_ptr(), 2, out.data_ptr(),
                                  ws.data_ptr(), ws.numel(), st)
        assert rc == mv.MOE_EINVAL
        arr = (mv.moe_layer_w * 1)(w)
        rc = lib.moe_round(s.handle, arr, 1, x.data_ptr(), 2, out.data_ptr(), None, ws.data_ptr(),
                           ws.numel(), 1, None)
        assert rc == mv.MOE_EINVAL  # graph capture needs a non-default stream
        assert mv.moe_last_device_status(s.handle, st) == mv.MOE_OK
    finally:
        s.close()


def test_bounded_wait_reports_timeout_without_hanging():
    """A 1 ns bound makes the staging wait give up at once; the kernel drains its copies
    under the default bound, flags MOE_ETIMEOUT and returns.  The next call is clean."""
    s = _tiny_stack()
    try:
        dev = s.device
        xb = s.rows(0, 2, 0.5)
        x = s.x_dev(xb)
        out = torch.empty(2, s.cfg.hidden, device=dev)
        ws = s.ws(2)
        st = stream_of(dev)
        mv.moe_set_wait_limit_ns(s.handle, 1)
        mv.moe_decode_layer(s.handle, s.layers[0].w, x.data_ptr(), 2, out.data_ptr(), ws.data_ptr(),
                            ws.numel(), st)
        assert mv.moe_last_device_status(s.handle, st) == mv.MOE_ETIMEOUT
        mv.moe_set_wait_limit_ns(s.handle, 0)
        got = run_layer(s, 0, xb)
        ref = oracle.layer(syngen.router(s.cfg, 0), xb, s.cfg.top_k, np.arange(8),
                           syngen.experts_stacked(s.cfg, 0, range(8)))
        assert_close(got, ref, "after timeout")
    finally:
        s.close()


def test_calls_with_fewer_rows_than_the_handle_allows():
    """A handle sized for 16 rows serves 1-row and 16-row calls (each call takes the
    kernel and the shared-memory plan of its own row count)."""
    cfg = syngen.CONFIGS["a3b_r1"]
    s = Stack(cfg, n_layers=1, max_rows=16)
    try:
        router = syngen.router(cfg, 0)
        for R, sigma in ((1, 0.0), (16, 0.1)):
            xb = s.rows(0, R, sigma)
            got = run_layer(s, 0, xb)
            rt = oracle.route(router, xb, cfg.top_k)
            ref = oracle.layer(router, xb, cfg.top_k, rt.union, syngen.experts_stacked(cfg, 0, rt.union))
            assert_close(got, ref, f"max_rows 16, R={R}")
        dev = s.device
        xs = np.stack([s.rows(0, 1, 0.0)])
        x = torch.from_numpy(xs.view(np.int16)).to(dev)
        out = torch.empty((1, 1, cfg.hidden), device=dev)
        ws = s.ws(1)
        st = torch.cuda.Stream(dev)
        mv.moe_round(s.handle, [s.layers[0].w], x.data_ptr(), 1, out.data_ptr(), None, ws.data_ptr(), ws.numel(),
                     True, st.cuda_stream)
        assert mv.moe_last_device_status(s.handle, st.cuda_stream) == mv.MOE_OK
        np.testing.assert_array_equal(out.cpu().numpy()[0], run_layer(s, 0, xs[0]))
    finally:
        s.close()


# ---- routing tail skip ----------------------------------------------------------------

TAIL_CASES = {"tiny": [(3, 0.5)], "a3b_r1": [(4, 0.5), (16, 0.1)], "e512_r3": [(3, 0.5)]}


def test_tail_skip_matches_oracle(stack):
    """With the tail skip on, the union (after the skip) is bit-exact and the outputs
    match the oracle's mirror of the rule; rank 1 drops everything, rank k+1 nothing."""
    cfg = stack.cfg
    k = cfg.top_k
    ranks = sorted({1, max(1, k - 1), min(7, k), k + 1})
    try:
        for tail in ranks:
            mv.moe_set_tail_skip(stack.handle, tail)
            for R, sigma in TAIL_CASES[cfg.name]:
                xb = stack.rows(1, R, sigma)
                router = syngen.router(cfg, 1)
                rt = oracle.route(router, xb, k, tail)
                ids, w, uni = run_route(stack, 1, xb)
                np.testing.assert_array_equal(ids, rt.ids)
                np.testing.assert_array_equal(uni, rt.union)
                got = run_layer(stack, 1, xb)
                if rt.union.size == 0:
                    assert not got.any(), "every expert skipped: the output must be zero"
                    continue
                ref = oracle.layer(router, xb, k, rt.union, syngen.experts_stacked(cfg, 1, rt.union), tail)
                assert_close(got, ref, f"{cfg.name} R={R} tail {tail}")
    finally:
        mv.moe_set_tail_skip(stack.handle, 0)


def test_tail_skip_setter_rejects_negative_rank(stack):
    with pytest.raises(mv.MoeError):
        mv.moe_set_tail_skip(stack.handle, -1)


def test_a_later_handle_with_a_smaller_plan_keeps_earlier_handles_working(stack):
    """The kernel's dynamic shared-memory limit is shared by all handles; creating a
    handle for a small shape must not lower it below what a bigger handle launches."""
    small = syngen.CONFIGS["tiny"]
    h2 = mv.moe_create(mv.make_dims(small.hidden, small.experts, small.top_k, small.inter, 1), 0)
    try:
        xb = stack.rows(0, 1, 0.0)
        got = run_layer(stack, 0, xb)
        router = syngen.router(stack.cfg, 0)
        rt = oracle.route(router, xb, stack.cfg.top_k)
        ref = oracle.layer(router, xb, stack.cfg.top_k, rt.union,
                           syngen.experts_stacked(stack.cfg, 0, rt.union))
        assert_close(got, ref, f"{stack.cfg.name} after a second handle")
    finally:
        mv.moe_destroy(h2)


def test_wide_rounds_rows_are_independent_bitwise(stack):
    """Rounds of >= 13 rows run on the tensor cores; there too a row's output is
    bit-identical at any position and whatever other rows share the round."""
    cfg = stack.cfg
    xa = stack.rows(0, 16, 0.5)
    full = run_layer(stack, 0, xa)
    perm = np.roll(np.arange(16), 5)
    rot = run_layer(stack, 0, xa[perm].copy())
    np.testing.assert_array_equal(rot, full[perm])
    other = syngen.rows(cfg, 1, 16, 0.5)
    mixed = np.concatenate([xa[:8], other[8:]])
    got = run_layer(stack, 0, mixed)
    np.testing.assert_array_equal(got[:8], full[:8])
