"""The allocation-free entry point (for callers that may not allocate device memory):
its output must match moe_decode_layer's, on two calls in a row sharing the static
scratch.  Collected last on purpose (file name), so a stop-at-first-failure run has
already run every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

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
        x = stack.x_dev(xb)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        st = stream_of(dev)
        for call in range(2):
            out = torch.full((rows, cfg.hidden), float("nan"), dtype=torch.float32, device=dev)
            mv.moe_decode_layer_noalloc(stack.dims, stack.layers[0].w, x.data_ptr(), rows, out.data_ptr(),
                                        status.data_ptr(), st)
            torch.cuda.synchronize(dev)
            assert int(status.item()) == 0
            assert_close(out.cpu().numpy(), ref.astype(np.float64), f"{name} call {call}")
    finally:
        stack.close()


def test_noalloc_rejects_layers_beyond_its_scratch():
    # 32 rows x top-32 x intermediate 2048 needs 8 MiB of exchanged activations
    dims = mv.make_dims(2048, 64, 32, 2048, 32)
    need = 256 + mv.moe_workspace_bytes(dims, 32)
    assert need > mv.MOE_NOALLOC_SCRATCH_BYTES
    w = mv.make_layer_w(256, 256, 256, 256, 256)  # never dereferenced: rejected first
    rc = mv.lib().moe_decode_layer_noalloc(ctypes.byref(dims), ctypes.byref(w), 256, 32, 256, None, None)
    assert rc == mv.MOE_EWORKSPACE
    # every workload shape of this layer fits
    for name in ("tiny", "a3b_r1", "a3b_r4", "a3b_r16", "e512_r3"):
        cfg = syngen.CONFIGS[name]
        d = mv.make_dims(cfg.hidden, cfg.experts, cfg.top_k, cfg.inter, cfg.rows)
        assert 256 + mv.moe_workspace_bytes(d, cfg.rows) <= mv.MOE_NOALLOC_SCRATCH_BYTES
