"""Host-side tests of the C ABI: symbols, sizes, validation, the int4 block packer.

None of these launch GPU work; they run on any host that can load the library.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import spec_verify_layer_gb300 as mv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe_verify.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_0-9]+)\s*\(", src, re.M)))


def test_library_exports_every_declared_function():
    names = header_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(mv.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe_verify.h but not exported"
    assert set(names) == set(mv.ABI_SYMBOLS)


def test_strerror():
    for code in (0, -1, -2, -3, -4, -5):
        assert len(mv.moe_strerror(code)) >= 2
    assert "unknown" in mv.moe_strerror(-99)


A3B = dict(hidden=2048, n_experts=128, top_k=8, inter=768, max_rows=16)


def dims(**kw):
    d = dict(A3B)
    d.update(kw)
    return mv.make_dims(d["hidden"], d["n_experts"], d["top_k"], d["inter"], d["max_rows"])


def test_packed_sizes():
    d = dims()
    H, I = 2048, 768
    assert mv.moe_packed_bytes(d, mv.MOE_GATEUP, 0) == 2 * H * I // 2
    assert mv.moe_packed_bytes(d, mv.MOE_GATEUP, 1) == 2 * I * (H // 32) * 2
    assert mv.moe_packed_bytes(d, mv.MOE_DOWN, 0) == H * I // 2
    assert mv.moe_packed_bytes(d, mv.MOE_DOWN, 1) == H * (I // 32) * 2
    per_expert = sum(mv.moe_packed_bytes(d, w, p) for w in (0, 1) for p in (0, 1))
    assert per_expert == 3 * H * I * 18 // 32  # 18 bytes per 32 codes
    assert mv.moe_packed_bytes(d, 7, 0) == 0 and mv.moe_packed_bytes(d, 0, 2) == 0


def test_workspace_sizes():
    d = dims()
    w1, w16 = mv.moe_workspace_bytes(d, 1), mv.moe_workspace_bytes(d, 16)
    assert 0 < w1 < w16
    # dominated by the exchanged SwiGLU outputs: rows * k * I fp32
    assert w16 >= 16 * 8 * 768 * 4
    assert mv.moe_workspace_bytes(d, 0) == 0 and mv.moe_workspace_bytes(d, 17) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(hidden=2000), mv.MOE_EINVAL), (dict(inter=100), mv.MOE_EINVAL), (dict(inter=96), mv.MOE_EUNSUPPORTED),
    (dict(top_k=200), mv.MOE_EINVAL), (dict(top_k=0), mv.MOE_EINVAL),
    (dict(max_rows=0), mv.MOE_EINVAL), (dict(hidden=4096), mv.MOE_EUNSUPPORTED),
    (dict(hidden=384), mv.MOE_EUNSUPPORTED), (dict(max_rows=33), mv.MOE_EUNSUPPORTED),
    (dict(n_experts=2048, top_k=8), mv.MOE_EUNSUPPORTED), (dict(top_k=33, n_experts=64), mv.MOE_EUNSUPPORTED),
])
def test_dims_validation(kw, code):
    d = dims(**kw)
    assert mv.moe_workspace_bytes(d, 1) == 0
    h = ctypes.c_void_p()
    rc = mv.lib().moe_create(ctypes.byref(d), 0, ctypes.byref(h))
    assert rc == code and not h.value


def test_create_without_device_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    with pytest.raises(mv.MoeError) as ei:
        mv.moe_create(dims(), 0)
    assert ei.value.code == mv.MOE_ECUDA


def test_null_handle_calls_are_rejected():
    lib = mv.lib()
    w = mv.make_layer_w(256, 256, 256, 256, 256)
    assert lib.moe_decode_layer(None, ctypes.byref(w), 256, 1, 256, 256, 1 << 20, None) == mv.MOE_EINVAL
    assert lib.moe_route(None, ctypes.byref(w), 256, 1, None, None, None, None, 256, 1 << 20, None) == mv.MOE_EINVAL
    assert lib.moe_last_device_status(None, None) == mv.MOE_EINVAL
    # the host-buffer round checks its handle before it reads anything else or copies
    xh, oh = np.zeros(256, np.uint16), np.zeros(256, np.float32)
    ws_list = (mv.moe_layer_w * 1)(w)
    assert lib.moe_round_host(None, ctypes.byref(dims()), ws_list, 1, xh.ctypes.data, 1, oh.ctypes.data, None,
                              None, None, None, 0, 0, 1, None) == mv.MOE_EINVAL
    assert lib.moe_last_launch_count(None) == 0


# ---- packer: decode the documented layout independently and compare ---------------------

def _decode_blocks(by):
    lo = (by & 15).astype(np.int8) - 8
    hi = (by >> 4).astype(np.int8) - 8
    return np.stack([lo, hi], axis=-1)


def _unswizzle(arr, rows, nb):
    # logical block b of a row with key k is stored at position b ^ (k & 7)
    pos = np.arange(nb)[None, :] ^ (np.asarray(rows)[:, None] & 7)
    return np.take_along_axis(arr, pos.reshape(pos.shape + (1,) * (arr.ndim - 2)), axis=1)


def _decode_gateup(nib, sc, E, H, I):
    # codes [E][I][2: gate, up][H/32][16 B], scales [E][I][2][H/32]; key of row (i, m) = i
    NB = H // 32
    rows = np.arange(2 * I) // 2
    by = nib.reshape(E, 2 * I, NB, 16)
    s = sc.reshape(E, 2 * I, NB)
    by = np.stack([_unswizzle(by[e], rows, NB) for e in range(E)])
    s = np.stack([_unswizzle(s[e], rows, NB) for e in range(E)])
    codes = _decode_blocks(by).reshape(E, I, 2, H)
    s = s.reshape(E, I, 2, NB)
    return codes[:, :, 0], codes[:, :, 1], s[:, :, 0], s[:, :, 1]


def _decode_down(nib, sc, E, H, I):
    # codes [E][I/32][H][16 B], scales [E][I/32][H]: block b of output row o at b * H + o
    NBI = I // 32
    by = nib.reshape(E, NBI, H, 16).transpose(0, 2, 1, 3)
    s = sc.reshape(E, NBI, H).transpose(0, 2, 1)
    codes = _decode_blocks(np.ascontiguousarray(by)).reshape(E, H, I)
    return codes, np.ascontiguousarray(s)


@pytest.mark.parametrize("H,I,E", [(256, 256, 1), (512, 256, 3), (2048, 512, 2)])
def test_packer_layout_roundtrip(H, I, E):
    rng = np.random.default_rng(H + I + E)
    d = mv.make_dims(H, max(E, 2), 1, I, 1)
    qg = rng.integers(-8, 8, (E, I, H), dtype=np.int8)
    qu = rng.integers(-8, 8, (E, I, H), dtype=np.int8)
    qd = rng.integers(-8, 8, (E, H, I), dtype=np.int8)
    sg = rng.integers(0, 65535, (E, I, H // 32), dtype=np.uint16)
    su = rng.integers(0, 65535, (E, I, H // 32), dtype=np.uint16)
    sd = rng.integers(0, 65535, (E, H, I // 32), dtype=np.uint16)
    gu_nib = np.zeros(E * mv.moe_packed_bytes(d, 0, 0), np.uint8)
    gu_sc = np.zeros(E * mv.moe_packed_bytes(d, 0, 1) // 2, np.uint16)
    dn_nib = np.zeros(E * mv.moe_packed_bytes(d, 1, 0), np.uint8)
    dn_sc = np.zeros(E * mv.moe_packed_bytes(d, 1, 1) // 2, np.uint16)
    mv.moe_pack_q4(d, mv.MOE_GATEUP, E, qg.ctypes.data, sg.ctypes.data, qu.ctypes.data, su.ctypes.data,
                   gu_nib.ctypes.data, gu_sc.ctypes.data)
    mv.moe_pack_q4(d, mv.MOE_DOWN, E, qd.ctypes.data, sd.ctypes.data, None, None,
                   dn_nib.ctypes.data, dn_sc.ctypes.data)
    g2, u2, sg2, su2 = _decode_gateup(gu_nib, gu_sc, E, H, I)
    np.testing.assert_array_equal(g2, qg)
    np.testing.assert_array_equal(u2, qu)
    np.testing.assert_array_equal(sg2, sg)
    np.testing.assert_array_equal(su2, su)
    d2, sd2 = _decode_down(dn_nib, dn_sc, E, H, I)
    np.testing.assert_array_equal(d2, qd)
    np.testing.assert_array_equal(sd2, sd)


def test_packer_one_hot_nibble_order():
    # element 2t -> low nibble of byte t, element 2t+1 -> high nibble, stored as q + 8
    H, I = 256, 256
    d = mv.make_dims(H, 2, 1, I, 1)
    qd = np.zeros((1, H, I), np.int8)
    qd[0, 5, 35] = 7   # o = 5, i = 35: block 1 of row 5 (stored at block-major position 1 * H + 5), byte 1, high nibble
    sd = np.zeros((1, H, I // 32), np.uint16)
    nib = np.zeros(mv.moe_packed_bytes(d, 1, 0), np.uint8)
    sc = np.zeros(mv.moe_packed_bytes(d, 1, 1) // 2, np.uint16)
    mv.moe_pack_q4(d, mv.MOE_DOWN, 1, qd.ctypes.data, sd.ctypes.data, None, None, nib.ctypes.data, sc.ctypes.data)
    off = (1 * H + 5) * 16
    blk = nib[off:off + 16]
    assert blk[1] == (8 | (15 << 4))
    assert all(b == 0x88 for i, b in enumerate(blk) if i != 1)
    assert (np.delete(nib, np.arange(off, off + 16)) == 0x88).all()


def test_packer_rejects_out_of_range_codes():
    H, I = 256, 256
    d = mv.make_dims(H, 2, 1, I, 1)
    qd = np.zeros((1, H, I), np.int8)
    qd[0, 0, 0] = 8
    sd = np.zeros((1, H, I // 32), np.uint16)
    nib = np.zeros(mv.moe_packed_bytes(d, 1, 0), np.uint8)
    sc = np.zeros(mv.moe_packed_bytes(d, 1, 1) // 2, np.uint16)
    with pytest.raises(mv.MoeError) as ei:
        mv.moe_pack_q4(d, mv.MOE_DOWN, 1, qd.ctypes.data, sd.ctypes.data, None, None, nib.ctypes.data, sc.ctypes.data)
    assert ei.value.code == mv.MOE_EINVAL
