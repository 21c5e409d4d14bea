"""CPU oracle for the MoE verify-round layer -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and its
binding) never loads it, and it never loads the product path.

The arithmetic lives in ``oracle.cpp`` (plain single-threaded C++); this module
only compiles it on demand and marshals numpy arrays.  See that file's header for
the definition it follows and the readings it takes.

Parity status: every function here is pinned by tests/test_oracle_pins.py
(closed forms, brute force, invariants and hand-worked fixtures in tests/golden/).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared"]


def build() -> str:
    if os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", *CXXFLAGS, _SRC, "-o", tmp])
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i32, vp = ctypes.c_int32, ctypes.c_void_p
        L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_half_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_float.restype = ctypes.c_float
        L.oracle_canonical_logit.argtypes = [vp, vp, i32]
        L.oracle_canonical_logit.restype = ctypes.c_float
        L.oracle_route.argtypes = [i32] * 4 + [vp] * 8
        L.oracle_route.restype = i32
        L.oracle_layer.argtypes = [i32] * 5 + [vp, vp, i32] + [vp] * 8
        L.oracle_layer.restype = i32
        L.oracle_layer_dense.argtypes = [i32] * 5 + [vp] * 9
        L.oracle_layer_dense.restype = i32
        L.oracle_route_tail.argtypes = [i32] * 5 + [vp] * 9
        L.oracle_route_tail.restype = i32
        L.oracle_layer_tail.argtypes = [i32] * 6 + [vp, vp, i32] + [vp] * 8
        L.oracle_layer_tail.restype = i32
        L.oracle_layer_dense_tail.argtypes = [i32] * 6 + [vp] * 9
        L.oracle_layer_dense_tail.restype = i32
        L.oracle_expert_ffn.argtypes = [i32, i32] + [vp] * 8
        L.oracle_expert_ffn.restype = i32
        L.oracle_unique_expert_bytes.argtypes = [i32, i32, i32]
        L.oracle_unique_expert_bytes.restype = ctypes.c_int64
        _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "arrays passed to the oracle must be C-contiguous"
    return a.ctypes.data


def half_to_double(bits: int) -> float:
    return float(lib().oracle_half_to_double(int(bits)))


def bf16_to_float(bits: int) -> float:
    return float(lib().oracle_bf16_to_float(int(bits)))


def canonical_logit(w: np.ndarray, x: np.ndarray) -> np.float32:
    w = np.ascontiguousarray(w, np.float32)
    x = np.ascontiguousarray(x, np.float32)
    return np.float32(lib().oracle_canonical_logit(_p(w), _p(x), w.size))


@dataclass
class Route:
    logits: np.ndarray   # [R][E] fp32 (canonical order)
    ids: np.ndarray      # [R][k] int32, rank order
    w: np.ndarray        # [R][k] fp64
    union: np.ndarray    # [U] int32 ascending (after the tail skip, if any)
    gap64: np.ndarray    # [R] fp64 gap between k-th and (k+1)-th exact logit
    keep: np.ndarray = None  # [R][k] bool: the pick's expert is evaluated


def route(router: np.ndarray, x_bf16: np.ndarray, k: int, tail_rank: int = 0) -> Route:
    """Routing of one layer; ``tail_rank`` > 0 drops union experts that every row
    picking them has at 1-based rank >= tail_rank (no renormalisation)."""
    router = np.ascontiguousarray(router, np.float32)
    x_bf16 = np.ascontiguousarray(x_bf16, np.uint16)
    E, H = router.shape
    R = x_bf16.shape[0]
    logits = np.empty((R, E), np.float32)
    ids = np.empty((R, k), np.int32)
    w = np.empty((R, k), np.float64)
    keep = np.empty((R, k), np.uint8)
    uni = np.empty(E, np.int32)
    nu = np.zeros(1, np.int32)
    gap = np.empty(R, np.float64)
    rc = lib().oracle_route_tail(H, E, k, R, int(tail_rank), _p(router), _p(x_bf16), _p(logits),
                                 _p(ids), _p(w), _p(keep), _p(uni), _p(nu), _p(gap))
    if rc != 0:
        raise ValueError(f"oracle_route rejected the dimensions (rc={rc})")
    return Route(logits, ids, w, uni[: nu[0]].copy(), gap, keep.astype(bool))


def layer(router, x_bf16, k: int, prov_ids, ew, tail_rank: int = 0) -> np.ndarray:
    """Output rows [R][H] (fp64).  ``ew`` holds the stacked weights of the experts
    ``prov_ids`` (an object with qg, sg, qu, su, qd, sd arrays, leading axis P)."""
    router = np.ascontiguousarray(router, np.float32)
    x_bf16 = np.ascontiguousarray(x_bf16, np.uint16)
    E, H = router.shape
    R = x_bf16.shape[0]
    I = ew.qg.shape[1]
    prov = np.ascontiguousarray(prov_ids, np.int32)
    out = np.empty((R, H), np.float64)
    rc = lib().oracle_layer_tail(H, E, k, I, R, int(tail_rank), _p(router), _p(x_bf16), prov.size,
                                 _p(prov), _p(ew.qg), _p(ew.sg), _p(ew.qu), _p(ew.su), _p(ew.qd),
                                 _p(ew.sd), _p(out))
    if rc == -2:
        raise KeyError("a routed expert's weights were not provided to the oracle")
    if rc != 0:
        raise ValueError(f"oracle_layer rejected the dimensions (rc={rc})")
    return out


def layer_dense(router, x_bf16, k: int, ew, tail_rank: int = 0) -> np.ndarray:
    """Brute force: all E experts evaluated for every row (ew holds all E experts)."""
    router = np.ascontiguousarray(router, np.float32)
    x_bf16 = np.ascontiguousarray(x_bf16, np.uint16)
    E, H = router.shape
    R = x_bf16.shape[0]
    I = ew.qg.shape[1]
    assert ew.qg.shape[0] == E
    out = np.empty((R, H), np.float64)
    rc = lib().oracle_layer_dense_tail(H, E, k, I, R, int(tail_rank), _p(router), _p(x_bf16),
                                       _p(ew.qg), _p(ew.sg), _p(ew.qu), _p(ew.su), _p(ew.qd),
                                       _p(ew.sd), _p(out))
    if rc != 0:
        raise ValueError(f"oracle_layer_dense rejected the dimensions (rc={rc})")
    return out


def expert_ffn(x_row_bf16: np.ndarray, ew, p: int = 0) -> np.ndarray:
    """y[H] (fp64) of one expert (index p of the stacked weights ``ew``) for one row."""
    x = np.ascontiguousarray(x_row_bf16, np.uint16)
    I, H = ew.qg.shape[1], ew.qg.shape[2]
    y = np.empty(H, np.float64)
    sl = [np.ascontiguousarray(getattr(ew, f)[p]) for f in ("qg", "sg", "qu", "su", "qd", "sd")]
    rc = lib().oracle_expert_ffn(H, I, _p(x), *(_p(a) for a in sl), _p(y))
    if rc != 0:
        raise ValueError(f"oracle_expert_ffn rejected the dimensions (rc={rc})")
    return y


def unique_expert_bytes(H: int, I: int, n_union: int) -> int:
    return int(lib().oracle_unique_expert_bytes(H, I, n_union))


def layer_from_generator(cfg, layer_idx: int, x_bf16=None, tail_rank: int = 0):
    """Route one generated layer, generate only the union experts, evaluate it.

    Returns (Route, out[R][H] fp64).  Inputs come from the shared seeded generator.
    """
    import syngen
    router = syngen.router(cfg, layer_idx)
    x = syngen.rows(cfg, layer_idx) if x_bf16 is None else x_bf16
    rt = route(router, x, cfg.top_k, tail_rank)
    ew = syngen.experts_stacked(cfg, layer_idx, rt.union)
    out = layer(router, x, cfg.top_k, rt.union, ew, tail_rank)
    return rt, out
