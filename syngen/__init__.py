"""Seeded synthetic inputs for the MoE verify-round layer (shared by oracle and GPU tests).

Holds no arithmetic of the layer itself: it draws int4 codes, fp16 scales, fp32
router weights and bf16 activation rows from a counter-based generator
(splitmix64; see syngen.c for the exact definition), and defines the workload
shapes.  Both the CPU oracle and the CUDA path are fed from here; neither
imports the other.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "syngen.c")
_LIB = os.path.join(_HERE, "libsyngen.so")

# tensor ids of the generator streams
T_ROUTER, T_GATE_Q, T_GATE_S, T_UP_Q, T_UP_S, T_DOWN_Q, T_DOWN_S, T_X0, T_XNOISE = range(1, 10)

ROUTER_SIGMA = 0.02
SCALE_SIGMA = 0.02


@dataclass(frozen=True)
class LayerCfg:
    """Shape and input recipe of one workload.

    hidden H, experts E, top-k k, expert intermediate I, verify rows R, layers L,
    row noise sigma (row r = bf16(x0 + sigma * n_r)), seed.
    """
    name: str
    hidden: int
    experts: int
    top_k: int
    inter: int
    rows: int
    layers: int
    row_sigma: float
    seed: int = 0

    def with_(self, **kw) -> "LayerCfg":
        return replace(self, **kw)

    @property
    def expert_bytes(self) -> int:
        """Packed bytes of one expert: 3 matrices of H*I int4 codes, 18 B per 32."""
        return 3 * self.hidden * self.inter * 18 // 32

    @property
    def router_bytes(self) -> int:
        return self.experts * self.hidden * 4


# The five workloads: tiny; 35B-A3B-shaped 1 row; same with 4 MTP rows;
# 512-expert sparse with 3 rows; 16 near-duplicate lookup-copy rows.
CONFIGS = {
    "tiny": LayerCfg("tiny", 512, 8, 2, 256, 1, 1, 0.0),
    "a3b_r1": LayerCfg("a3b_r1", 2048, 128, 8, 768, 1, 40, 0.0),
    "a3b_r4": LayerCfg("a3b_r4", 2048, 128, 8, 768, 4, 40, 0.5),
    "e512_r3": LayerCfg("e512_r3", 2048, 512, 10, 512, 3, 48, 0.5),
    "a3b_r16": LayerCfg("a3b_r16", 2048, 128, 8, 768, 16, 40, 0.1),
}


def _build_if_needed() -> None:
    if os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)


def build() -> str:
    _build_if_needed()
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _build_if_needed()
        L = ctypes.CDLL(_LIB)
        u64, u32, i32, dbl = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_double
        vp = ctypes.c_void_p
        L.sg_q4.argtypes = [u64, u32, u32, u64, u64, vp]
        L.sg_normal_f32.argtypes = [u64, u32, u32, u64, u64, dbl, vp]
        L.sg_absnormal_f16.argtypes = [u64, u32, u32, u64, u64, dbl, vp]
        L.sg_rows_bf16.argtypes = [u64, u32, u32, u32, i32, i32, dbl, vp]
        L.sg_f32_to_bf16.argtypes = [ctypes.c_float]
        L.sg_f32_to_bf16.restype = ctypes.c_uint16
        L.sg_f64_to_f16.argtypes = [dbl]
        L.sg_f64_to_f16.restype = ctypes.c_uint16
        L.sg_stream_key.argtypes = [u64, u32, u32]
        L.sg_stream_key.restype = u64
        L.sg_draw.argtypes = [u64, u64]
        L.sg_draw.restype = u64
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---- raw draws -------------------------------------------------------------

def q4(seed: int, layer: int, tensor: int, start: int, count: int, out=None) -> np.ndarray:
    out = np.empty(count, np.int8) if out is None else out
    lib().sg_q4(seed, layer, tensor, start, count, _ptr(out))
    return out


def normal_f32(seed, layer, tensor, start, count, sigma, out=None) -> np.ndarray:
    out = np.empty(count, np.float32) if out is None else out
    lib().sg_normal_f32(seed, layer, tensor, start, count, float(sigma), _ptr(out))
    return out


def absnormal_f16(seed, layer, tensor, start, count, sigma, out=None) -> np.ndarray:
    out = np.empty(count, np.uint16) if out is None else out
    lib().sg_absnormal_f16(seed, layer, tensor, start, count, float(sigma), _ptr(out))
    return out


def f32_to_bf16(x: float) -> int:
    return int(lib().sg_f32_to_bf16(float(x)))


def f64_to_f16(x: float) -> int:
    return int(lib().sg_f64_to_f16(float(x)))


# ---- layer tensors -----------------------------------------------------------

def router(cfg: LayerCfg, layer: int) -> np.ndarray:
    """Router weights [E][H] fp32 ~ N(0, 0.02)."""
    E, H = cfg.experts, cfg.hidden
    return normal_f32(cfg.seed, layer, T_ROUTER, 0, E * H, ROUTER_SIGMA).reshape(E, H)


def rows(cfg: LayerCfg, layer: int, n_rows: int | None = None, sigma: float | None = None) -> np.ndarray:
    """Activation rows [R][H] as bf16 bit patterns (uint16)."""
    R = cfg.rows if n_rows is None else n_rows
    s = cfg.row_sigma if sigma is None else sigma
    out = np.empty((R, cfg.hidden), np.uint16)
    lib().sg_rows_bf16(cfg.seed, layer, T_X0, T_XNOISE, R, cfg.hidden, float(s), _ptr(out))
    return out


@dataclass
class ExpertW:
    """Unpacked weights of one expert.

    qg, qu: [I][H] int8 codes in [-8, 7]; sg, su: [I][H/32] fp16 bits (gate/up)
    qd: [H][I] int8; sd: [H][I/32] fp16 bits (down).  Weight = fp16(scale) * q.
    """
    qg: np.ndarray
    sg: np.ndarray
    qu: np.ndarray
    su: np.ndarray
    qd: np.ndarray
    sd: np.ndarray


def expert(cfg: LayerCfg, layer: int, e: int) -> ExpertW:
    H, I, s = cfg.hidden, cfg.inter, cfg.seed
    n = H * I
    qg = q4(s, layer, T_GATE_Q, e * n, n).reshape(I, H)
    sg = absnormal_f16(s, layer, T_GATE_S, e * n // 32, n // 32, SCALE_SIGMA).reshape(I, H // 32)
    qu = q4(s, layer, T_UP_Q, e * n, n).reshape(I, H)
    su = absnormal_f16(s, layer, T_UP_S, e * n // 32, n // 32, SCALE_SIGMA).reshape(I, H // 32)
    qd = q4(s, layer, T_DOWN_Q, e * n, n).reshape(H, I)
    sd = absnormal_f16(s, layer, T_DOWN_S, e * n // 32, n // 32, SCALE_SIGMA).reshape(H, I // 32)
    return ExpertW(qg, sg, qu, su, qd, sd)


def experts_stacked(cfg: LayerCfg, layer: int, ids, threads: int = 0) -> ExpertW:
    """Weights of the listed experts stacked along a leading axis [P]."""
    ids = [int(i) for i in ids]
    threads = threads or min(len(ids), os.cpu_count() or 1) or 1
    if threads > 1:
        with ThreadPoolExecutor(threads) as ex:
            ws = list(ex.map(lambda e: expert(cfg, layer, e), ids))
    else:
        ws = [expert(cfg, layer, e) for e in ids]
    return ExpertW(*(np.ascontiguousarray(np.stack([getattr(w, f) for w in ws]))
                     for f in ("qg", "sg", "qu", "su", "qd", "sd")))
