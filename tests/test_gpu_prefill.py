"""Prefill-width MoE layer (many token rows per call; infero README, "Beyond plain text
decode", MoE: a counting sort by expert, then per-expert GEMMs) through the C ABI.

The output definition is the decode layer's, so the oracle is the same `oracle.layer`
over all tokens (or over sampled tokens: a token's output does not depend on the other
tokens of the call).  Counts per expert are exact integers; outputs within the layer
tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import spec_verify_layer_gb300 as mv
import syngen
from gpu_helpers import Stack, assert_close

pytestmark = pytest.mark.gpu


def _prefill(s: Stack, layer: int, xb: np.ndarray, w=None, counts=True, ws=None):
    T = xb.shape[0]
    dev = s.device
    x = s.x_dev(xb)
    out = torch.full((T, s.cfg.hidden), float("nan"), dtype=torch.float32, device=dev)
    cnt = torch.full((s.cfg.experts,), -1, dtype=torch.int32, device=dev) if counts else None
    nbytes = mv.moe_prefill_workspace_bytes(s.dims, T)
    assert nbytes > 0
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev).cuda_stream
    mv.moe_prefill_layer(s.handle, w if w is not None else s.layers[layer].w, x.data_ptr(), T, out.data_ptr(),
                         cnt.data_ptr() if counts else 0, ws.data_ptr(), ws.numel(), st)
    assert mv.moe_last_device_status(s.handle, st) == mv.MOE_OK
    assert mv.moe_last_launch_count(s.handle) == 7
    return out.cpu().numpy(), (cnt.cpu().numpy() if counts else None)


def _oracle(cfg, layer, xb):
    router = syngen.router(cfg, layer)
    rt = oracle.route(router, xb, cfg.top_k)
    ref = oracle.layer(router, xb, cfg.top_k, rt.union, syngen.experts_stacked(cfg, layer, rt.union))
    hist = np.bincount(rt.ids.reshape(-1), minlength=cfg.experts)
    return ref, hist


@pytest.fixture(scope="module")
def tiny():
    s = Stack(syngen.CONFIGS["tiny"], n_layers=2, max_rows=4)
    yield s
    s.close()


@pytest.fixture(scope="module")
def a3b():
    s = Stack(syngen.CONFIGS["a3b_r1"], n_layers=1, max_rows=16)
    yield s
    s.close()


@pytest.mark.parametrize("T", [1, 2, 3, 31, 64, 65, 200])
def test_tiny_matches_oracle_and_counts(tiny, T):
    xb = syngen.rows(tiny.cfg, 1, T, 1.0)
    got, cnt = _prefill(tiny, 1, xb)
    ref, hist = _oracle(tiny.cfg, 1, xb)
    np.testing.assert_array_equal(cnt, hist)
    assert_close(got, ref, f"tiny prefill T={T}")


def test_a3b_shape_matches_oracle(a3b):
    """48 tokens of the 35B-A3B-shaped layer, spread over many experts (runs of 1 to a
    few tokens per expert: every tile ragged)."""
    cfg = a3b.cfg
    xb = syngen.rows(cfg, 0, 48, 1.0)
    got, cnt = _prefill(a3b, 0, xb)
    ref, hist = _oracle(cfg, 0, xb)
    np.testing.assert_array_equal(cnt, hist)
    assert_close(got, ref, "a3b prefill T=48")


def test_a3b_full_width_full_and_ragged_tiles(a3b):
    """2048 tokens (runs of about 128 tokens per expert).  Every token routed to the
    busiest expert (its runs fill whole 64-token gate/up and 32-token down tiles) and
    every token routed to an expert whose run ends in a ragged tile is compared with the
    oracle element by element; all tokens' counts are exact."""
    cfg = a3b.cfg
    T = 2048
    xb = syngen.rows(cfg, 0, T, 1.0)
    got, cnt = _prefill(a3b, 0, xb)
    router = syngen.router(cfg, 0)
    rt = oracle.route(router, xb, cfg.top_k)
    np.testing.assert_array_equal(cnt, np.bincount(rt.ids.reshape(-1), minlength=cfg.experts))
    assert np.isfinite(got).all()
    full = int(np.argmax(cnt))
    assert cnt[full] >= 128  # two or more full gate/up tiles
    ragged_cands = [e for e in range(cfg.experts) if cnt[e] % 64 not in (0,) and cnt[e] % 32 != 0 and e != full]
    ragged = max(ragged_cands, key=lambda e: cnt[e] % 64)
    picked = np.unique(np.concatenate([np.nonzero((rt.ids == full).any(axis=1))[0],
                                       np.nonzero((rt.ids == ragged).any(axis=1))[0], [0, T - 1]]))
    assert picked.size >= cnt[full]
    xs = xb[picked]
    rs = oracle.route(router, xs, cfg.top_k)
    ref = oracle.layer(router, xs, cfg.top_k, rs.union, syngen.experts_stacked(cfg, 0, rs.union))
    assert_close(got[picked], ref, f"a3b prefill T=2048: {picked.size} tokens of experts {full} "
                                   f"({cnt[full]} picks) and {ragged} ({cnt[ragged]} picks)")


def test_tokens_are_independent_bitwise(tiny):
    """A token's output is the same bits alone and inside a batch of 130."""
    xb = syngen.rows(tiny.cfg, 0, 130, 1.0)
    got, _ = _prefill(tiny, 0, xb, counts=False)
    for t in (0, 64, 129):
        alone, _ = _prefill(tiny, 0, xb[t:t + 1], counts=False)
        np.testing.assert_array_equal(alone[0], got[t])


def test_repeat_calls_are_bitwise_equal(tiny):
    xb = syngen.rows(tiny.cfg, 1, 77, 1.0)
    a, _ = _prefill(tiny, 1, xb)
    b, _ = _prefill(tiny, 1, xb)
    np.testing.assert_array_equal(a, b)


def test_slot_table_matches_per_layer_weights(tiny):
    """The layer's experts, shuffled into a bank of 2E slots and addressed by a device
    table, give bitwise the per-layer result."""
    cfg = tiny.cfg
    E = cfg.experts
    keys = ("gu_nib", "gu_sc", "dn_nib", "dn_sc")
    ly = tiny.layers[0]
    per = {k: getattr(ly, k).view(torch.uint8).numel() // E for k in keys}
    slots = np.random.default_rng(3).permutation(2 * E)[:E].astype(np.int32)
    bank = {k: torch.zeros(2 * E * per[k], dtype=torch.uint8, device=tiny.device) for k in keys}
    idx = torch.from_numpy(slots).long().to(tiny.device)
    for k in keys:
        bank[k].view(2 * E, per[k])[idx] = getattr(ly, k).view(torch.uint8).view(E, per[k])
    table = torch.from_numpy(slots).to(tiny.device)
    w = mv.make_layer_w(ly.router.data_ptr(), bank["gu_nib"].data_ptr(), bank["gu_sc"].data_ptr(),
                        bank["dn_nib"].data_ptr(), bank["dn_sc"].data_ptr(), table.data_ptr(), 2 * E)
    xb = syngen.rows(cfg, 0, 70, 1.0)
    got, _ = _prefill(tiny, 0, xb, w=w)
    ref, _ = _prefill(tiny, 0, xb)
    np.testing.assert_array_equal(got, ref)


def test_argument_errors(tiny):
    dev = tiny.device
    xb = syngen.rows(tiny.cfg, 0, 4, 1.0)
    x = tiny.x_dev(xb)
    out = torch.empty((4, tiny.cfg.hidden), dtype=torch.float32, device=dev)
    nbytes = mv.moe_prefill_workspace_bytes(tiny.dims, 4)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev).cuda_stream
    w = tiny.layers[0].w
    assert mv.moe_prefill_workspace_bytes(tiny.dims, 0) == 0
    with pytest.raises(mv.MoeError):  # no tokens
        mv.moe_prefill_layer(tiny.handle, w, x.data_ptr(), 0, out.data_ptr(), 0, ws.data_ptr(), nbytes, st)
    with pytest.raises(mv.MoeError):  # short workspace
        mv.moe_prefill_layer(tiny.handle, w, x.data_ptr(), 4, out.data_ptr(), 0, ws.data_ptr(), nbytes - 1, st)
    with pytest.raises(mv.MoeError):  # misaligned rows
        mv.moe_prefill_layer(tiny.handle, w, x.data_ptr() + 2, 4, out.data_ptr(), 0, ws.data_ptr(), nbytes, st)
    # the handle stays usable
    got, _ = _prefill(tiny, 0, xb)
    ref, _ = _oracle(tiny.cfg, 0, xb)
    assert_close(got, ref, "after errors")
