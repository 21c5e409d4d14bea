"""The allocation-free entry point (for callers that may not allocate device memory):
its output must equal moe_decode_layer's bit for bit (the same kernel on the same
arguments) and match the oracle, on two calls in a row sharing the static scratch.
Collected last on purpose (file name), so a stop-at-first-failure run has already run
every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import spec_verify_layer_gb300 as mv
import syngen
from gpu_helpers import Stack, assert_close, stream_of

pytestmark = pytest.mark.gpu


def _reference(stack, xb):
    dev = stack.device
    R = xb.shape[0]
    x = stack.x_dev(xb)
    out = torch.empty((R, stack.cfg.hidden), dtype=torch.float32, device=dev)
    ws = stack.ws(R)
    st = stream_of(dev)
    mv.moe_decode_layer(stack.handle, stack.layers[0].w, x.data_ptr(), R, out.data_ptr(), ws.data_ptr(),
                        ws.numel(), st)
    assert mv.moe_last_device_status(stack.handle, st) == mv.MOE_OK
    return out.cpu().numpy()


@pytest.mark.parametrize("name,rows,sigma", [("tiny", 3, 0.5), ("a3b_r1", 1, 0.0), ("a3b_r4", 4, 0.5)])
def test_noalloc_matches_decode_layer_twice(name, rows, sigma):
    cfg = syngen.CONFIGS[name]
    stack = Stack(cfg, n_layers=1, max_rows=rows)
    try:
        dev = stack.device
        torch.cuda.set_device(dev.index if dev.index is not None else 0)
        xb = stack.rows(0, rows, sigma)
        ref = _reference(stack, xb)
        router = syngen.router(cfg, 0)
        rt = oracle.route(router, xb, cfg.top_k)
        want = oracle.layer(router, xb, cfg.top_k, rt.union, syngen.experts_stacked(cfg, 0, rt.union))
        x = stack.x_dev(xb)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        st = stream_of(dev)
        for call in range(2):
            out = torch.full((rows, cfg.hidden), float("nan"), dtype=torch.float32, device=dev)
            mv.moe_decode_layer_noalloc(stack.dims, stack.layers[0].w, x.data_ptr(), rows, out.data_ptr(),
                                        status.data_ptr(), st)
            torch.cuda.synchronize(dev)
            assert int(status.item()) == 0
            got = out.cpu().numpy()
            np.testing.assert_array_equal(got, ref, err_msg=f"{name} call {call}")
            assert_close(got, want, f"{name} call {call} against the oracle")
    finally:
        stack.close()


def test_noalloc_reports_a_slot_outside_the_bank_in_the_status_word():
    """An expert table entry outside the bank is not read: the status word the caller
    passes receives bit 2, and the next call with a good table is clean."""
    cfg = syngen.CONFIGS["tiny"]
    stack = Stack(cfg, n_layers=1, max_rows=2)
    try:
        dev = stack.device
        torch.cuda.set_device(dev.index if dev.index is not None else 0)
        ly = stack.layers[0]
        table = torch.arange(cfg.experts, dtype=torch.int32, device=dev)
        table[1] = cfg.experts  # one past the bank
        w_bad = mv.make_layer_w(ly.router.data_ptr(), ly.gu_nib.data_ptr(), ly.gu_sc.data_ptr(),
                                ly.dn_nib.data_ptr(), ly.dn_sc.data_ptr(), table.data_ptr(), cfg.experts)
        xb = stack.rows(0, 2, 0.5)
        x = stack.x_dev(xb)
        out = torch.empty((2, cfg.hidden), dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        st = stream_of(dev)
        mv.moe_decode_layer_noalloc(stack.dims, w_bad, x.data_ptr(), 2, out.data_ptr(), status.data_ptr(), st)
        torch.cuda.synchronize(dev)
        assert int(status.item()) & 2
        status.zero_()
        mv.moe_decode_layer_noalloc(stack.dims, ly.w, x.data_ptr(), 2, out.data_ptr(), status.data_ptr(), st)
        torch.cuda.synchronize(dev)
        assert int(status.item()) == 0
        np.testing.assert_array_equal(out.cpu().numpy(), _reference(stack, xb))
    finally:
        stack.close()


def test_noalloc_argument_errors_launch_nothing():
    """A missing status word and a layer too big for the scratch are refused before any
    launch (every pointer here is a real, small device allocation)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    p = buf.data_ptr()
    w = mv.make_layer_w(p, p, p, p, p)
    lib = mv.lib()
    # without a status word the kernel's findings would be lost: refused
    small = mv.make_dims(256, 8, 2, 256, 1)
    assert lib.moe_decode_layer_noalloc(ctypes.byref(small), ctypes.byref(w), p, 1, p, None, None) == mv.MOE_EINVAL
    # 32 rows x top-32 x intermediate 2048: 8 MiB of exchanged activations alone
    dims = mv.make_dims(2048, 64, 32, 2048, 32)
    assert mv.moe_workspace_bytes(dims, 32) > mv.MOE_NOALLOC_SCRATCH_BYTES
    rc = lib.moe_decode_layer_noalloc(ctypes.byref(dims), ctypes.byref(w), p, 32, p, status.data_ptr(), None)
    assert rc == mv.MOE_EWORKSPACE
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0 and not buf.any()
    # every workload shape of this layer fits
    for name in ("tiny", "a3b_r1", "a3b_r4", "a3b_r16", "e512_r3"):
        cfg = syngen.CONFIGS[name]
        d = mv.make_dims(cfg.hidden, cfg.experts, cfg.top_k, cfg.inter, cfg.rows)
        assert mv.moe_workspace_bytes(d, cfg.rows) <= mv.MOE_NOALLOC_SCRATCH_BYTES
