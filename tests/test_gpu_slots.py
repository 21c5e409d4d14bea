"""Expert -> slot indirection (a shared slot bank across layers, "which expert lives
where" as ingress data; AlphaInfer docs, sections 2 and 5.1), through the C ABI.

Two layers' experts live, shuffled, in one bank of 2E slots; each layer carries a device
table from expert id to slot.  The round must equal the oracle per layer, equal bitwise
the same round on per-layer weights, follow new table contents on graph replay without
a rebuild, and report (not fault on) a slot outside the bank.
"""
import numpy as np
import pytest
import torch

import oracle
import spec_verify_layer_gb300 as mv
import syngen
from gpu_helpers import Stack, assert_close

pytestmark = pytest.mark.gpu

KEYS = ("gu_nib", "gu_sc", "dn_nib", "dn_sc")


def _as_bytes(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.uint8)


@pytest.fixture(scope="module")
def banked():
    cfg = syngen.CONFIGS["tiny"]
    s = Stack(cfg, n_layers=2, max_rows=4)
    E = cfg.experts
    rng = np.random.default_rng(5)
    slots = rng.permutation(2 * E).astype(np.int32)        # slot of (layer l, expert e)
    table = [slots[:E].copy(), slots[E:].copy()]
    per = {k: _as_bytes(getattr(s.layers[0], k)).numel() // E for k in KEYS}
    bank = {k: torch.empty(2 * E * per[k], dtype=torch.uint8, device=s.device) for k in KEYS}
    for l in range(2):
        for k in KEYS:
            src = _as_bytes(getattr(s.layers[l], k)).view(E, per[k])
            bank[k].view(2 * E, per[k])[torch.from_numpy(table[l]).long().to(s.device)] = src
    tdev = [torch.from_numpy(t).to(s.device) for t in table]
    yield s, bank, tdev, per
    s.close()


def _w(s, bank, tdev, l):
    return mv.make_layer_w(s.layers[l].router.data_ptr(), bank["gu_nib"].data_ptr(), bank["gu_sc"].data_ptr(),
                           bank["dn_nib"].data_ptr(), bank["dn_sc"].data_ptr(), tdev[l].data_ptr(),
                           2 * s.cfg.experts)


def _round(s, wl, xs, use_graph, stream, out=None, stats=None):
    L, R, H = xs.shape[0], xs.shape[1], s.cfg.hidden
    x = torch.from_numpy(xs.view(np.int16)).to(s.device)
    if out is None:
        out = torch.full((L, R, H), float("nan"), device=s.device)
        stats = torch.full((L,), -1, dtype=torch.int32, device=s.device)
    ws = s.ws(R)
    with torch.cuda.stream(stream):
        mv.moe_round(s.handle, wl, x.data_ptr(), R, out.data_ptr(), stats.data_ptr(), ws.data_ptr(), ws.numel(),
                     use_graph, stream.cuda_stream)
    return out, stats, x, ws


def test_bank_round_matches_oracle_and_per_layer_weights(banked):
    s, bank, tdev, _ = banked
    cfg = s.cfg
    xs = np.stack([syngen.rows(cfg, l, 3, 0.5) for l in range(2)])
    st = torch.cuda.Stream(s.device)
    out_b, stats_b, _, _ = _round(s, [_w(s, bank, tdev, l) for l in range(2)], xs, False, st)
    assert mv.moe_last_device_status(s.handle, st.cuda_stream) == mv.MOE_OK
    out_p, stats_p, _, _ = _round(s, [ly.w for ly in s.layers], xs, False, st)
    assert mv.moe_last_device_status(s.handle, st.cuda_stream) == mv.MOE_OK
    np.testing.assert_array_equal(out_b.cpu().numpy(), out_p.cpu().numpy())
    np.testing.assert_array_equal(stats_b.cpu().numpy(), stats_p.cpu().numpy())
    got = out_b.cpu().numpy()
    for l in range(2):
        router = syngen.router(cfg, l)
        rt = oracle.route(router, xs[l], cfg.top_k)
        ref = oracle.layer(router, xs[l], cfg.top_k, rt.union, syngen.experts_stacked(cfg, l, rt.union))
        assert_close(got[l], ref, f"banked layer {l}")


def test_table_is_ingress_for_a_captured_round(banked):
    """Move two experts of layer 0 to each other's slots (bank contents and table entries
    swapped in place): the replayed graph reads the new table and gives the same result."""
    s, bank, tdev, per = banked
    cfg = s.cfg
    xs = np.stack([syngen.rows(cfg, l, 2, 0.5) for l in range(2)])
    st = torch.cuda.Stream(s.device)
    wl = [_w(s, bank, tdev, l) for l in range(2)]
    out, stats, x, ws = _round(s, wl, xs, True, st)
    first = out.clone()
    t0 = tdev[0].cpu().numpy()
    a, b = int(t0[0]), int(t0[1])
    for k in KEYS:
        v = bank[k].view(-1, per[k])
        tmp = v[a].clone()
        v[a] = v[b]
        v[b] = tmp
    tdev[0][0], tdev[0][1] = b, a
    torch.cuda.synchronize(s.device)
    with torch.cuda.stream(st):
        mv.moe_round(s.handle, wl, x.data_ptr(), 2, out.data_ptr(), stats.data_ptr(), ws.data_ptr(), ws.numel(),
                     True, st.cuda_stream)
    assert mv.moe_last_device_status(s.handle, st.cuda_stream) == mv.MOE_OK
    assert mv.moe_last_launch_count(s.handle) == 1
    assert torch.equal(first, out)


def test_slot_outside_the_bank_is_reported(banked):
    s, bank, tdev, _ = banked
    cfg = s.cfg
    bad = tdev[1].clone()
    bad[3] = 2 * cfg.experts  # one past the bank
    w = mv.make_layer_w(s.layers[1].router.data_ptr(), bank["gu_nib"].data_ptr(), bank["gu_sc"].data_ptr(),
                        bank["dn_nib"].data_ptr(), bank["dn_sc"].data_ptr(), bad.data_ptr(), 2 * cfg.experts)
    xb = syngen.rows(cfg, 1, 1, 0.0)
    x = s.x_dev(xb)
    out = torch.empty((1, cfg.hidden), device=s.device)
    ws = s.ws(1)
    st = torch.cuda.current_stream(s.device).cuda_stream
    mv.moe_decode_layer(s.handle, w, x.data_ptr(), 1, out.data_ptr(), ws.data_ptr(), ws.numel(), st)
    assert mv.moe_last_device_status(s.handle, st) == mv.MOE_EINVAL
    # the handle stays usable
    mv.moe_decode_layer(s.handle, _w(s, bank, tdev, 1), x.data_ptr(), 1, out.data_ptr(), ws.data_ptr(),
                        ws.numel(), st)
    assert mv.moe_last_device_status(s.handle, st) == mv.MOE_OK


def test_table_needs_a_bank_size(banked):
    s, bank, tdev, _ = banked
    w = mv.make_layer_w(s.layers[0].router.data_ptr(), bank["gu_nib"].data_ptr(), bank["gu_sc"].data_ptr(),
                        bank["dn_nib"].data_ptr(), bank["dn_sc"].data_ptr(), tdev[0].data_ptr(), 0)
    xb = syngen.rows(s.cfg, 0, 1, 0.0)
    x = s.x_dev(xb)
    out = torch.empty((1, s.cfg.hidden), device=s.device)
    ws = s.ws(1)
    with pytest.raises(mv.MoeError):
        mv.moe_decode_layer(s.handle, w, x.data_ptr(), 1, out.data_ptr(), ws.data_ptr(), ws.numel(),
                            torch.cuda.current_stream(s.device).cuda_stream)
