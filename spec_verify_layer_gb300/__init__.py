"""Python binding of the GB300 verify-round MoE library (libmoeverify.so).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  The functions carry the C names (moe_create, moe_route, ...); device
buffers are passed as integer addresses (e.g. ``tensor.data_ptr()``), streams as
``torch.cuda.Stream().cuda_stream`` integers.  A nonzero return code raises
``MoeError``.  If the compiled library is missing this module fails to import --
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoeverify.so")

MOE_OK, MOE_EINVAL, MOE_ECUDA, MOE_EWORKSPACE, MOE_ETIMEOUT, MOE_EUNSUPPORTED = 0, -1, -2, -3, -4, -5
MOE_GATEUP, MOE_DOWN = 0, 1

# exported symbols declared in include/moe_verify.h
ABI_SYMBOLS = (
    "moe_create", "moe_destroy", "moe_workspace_bytes", "moe_packed_bytes", "moe_pack_q4",
    "moe_route", "moe_decode_layer", "moe_round", "moe_round_host", "moe_last_device_status",
    "moe_last_launch_count", "moe_set_wait_limit_ns", "moe_set_tail_skip", "moe_profile",
    "moe_profile_read",
    "moe_profile_phases", "moe_decode_layer_noalloc", "moe_prefill_workspace_bytes",
    "moe_prefill_layer", "moe_strerror",
)
MOE_NOALLOC_SCRATCH_BYTES = 8 << 20
KIND_ROUND = 0
MMA_ROWS = 13  # rounds of at least this many rows run on the tensor cores
# phase intervals of a profiled moe_round, by the kernel that ran it (the library returns
# how many it wrote): the split kernel (rows below 8) and the tensor-core kernel
PHASES_SPLIT = ("router", "barrier1", "routing", "issue", "first_data", "units_before_last",
                "last_gateup", "last_swiglu_down_wait", "last_down", "barrier3")
PHASES_WIDE = ("router", "barrier1", "routing", "first_data", "gateup_stream", "gateup_tail",
               "barrier2", "h_wait", "down", "down_tail", "out_write", "barrier3")


class moe_dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("max_rows", ctypes.c_int32)]


class moe_layer_w(ctypes.Structure):
    _fields_ = [("router", ctypes.c_void_p), ("gateup_nib", ctypes.c_void_p),
                ("gateup_scale", ctypes.c_void_p), ("down_nib", ctypes.c_void_p),
                ("down_scale", ctypes.c_void_p), ("slot_of_expert", ctypes.c_void_p),
                ("n_slots", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {moe_strerror(code)} ({code})")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")

_lib = ctypes.CDLL(LIB_PATH)
_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_lib.moe_create.argtypes = [ctypes.POINTER(moe_dims), ctypes.c_int, ctypes.POINTER(_vp)]
_lib.moe_create.restype = ctypes.c_int
_lib.moe_destroy.argtypes = [_vp]
_lib.moe_destroy.restype = None
_lib.moe_workspace_bytes.argtypes = [ctypes.POINTER(moe_dims), _i32]
_lib.moe_workspace_bytes.restype = _sz
_lib.moe_packed_bytes.argtypes = [ctypes.POINTER(moe_dims), ctypes.c_int, ctypes.c_int]
_lib.moe_packed_bytes.restype = _sz
_lib.moe_pack_q4.argtypes = [ctypes.POINTER(moe_dims), ctypes.c_int, _i32] + [_vp] * 6
_lib.moe_pack_q4.restype = ctypes.c_int
_lib.moe_route.argtypes = [_vp, ctypes.POINTER(moe_layer_w), _vp, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.moe_route.restype = ctypes.c_int
_lib.moe_decode_layer.argtypes = [_vp, ctypes.POINTER(moe_layer_w), _vp, _i32, _vp, _vp, _sz, _vp]
_lib.moe_decode_layer.restype = ctypes.c_int
_lib.moe_round.argtypes = [_vp, ctypes.POINTER(moe_layer_w), _i32, _vp, _i32, _vp, _vp, _vp, _sz,
                           ctypes.c_int, _vp]
_lib.moe_round.restype = ctypes.c_int
_lib.moe_round_host.argtypes = [_vp, ctypes.POINTER(moe_dims), ctypes.POINTER(moe_layer_w), _i32, _vp, _i32, _vp,
                                _vp, _vp, _vp, _vp, _sz, ctypes.c_int, ctypes.c_int, _vp]
_lib.moe_round_host.restype = ctypes.c_int
_lib.moe_last_device_status.argtypes = [_vp, _vp]
_lib.moe_last_device_status.restype = ctypes.c_int
_lib.moe_last_launch_count.argtypes = [_vp]
_lib.moe_last_launch_count.restype = _i32
_lib.moe_set_wait_limit_ns.argtypes = [_vp, ctypes.c_uint64]
_lib.moe_set_wait_limit_ns.restype = ctypes.c_int
_lib.moe_set_tail_skip.argtypes = [_vp, ctypes.c_int32]
_lib.moe_set_tail_skip.restype = ctypes.c_int
_lib.moe_profile.argtypes = [_vp, ctypes.c_int]
_lib.moe_profile.restype = ctypes.c_int
_lib.moe_profile_read.argtypes = [_vp, ctypes.c_int, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_i32)]
_lib.moe_profile_read.restype = ctypes.c_int
_lib.moe_profile_phases.argtypes = [_vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), _i32]
_lib.moe_profile_phases.restype = ctypes.c_int
_lib.moe_decode_layer_noalloc.argtypes = [ctypes.POINTER(moe_dims), ctypes.POINTER(moe_layer_w), _vp, _i32,
                                          _vp, _vp, _vp]
_lib.moe_decode_layer_noalloc.restype = ctypes.c_int
_lib.moe_prefill_workspace_bytes.argtypes = [ctypes.POINTER(moe_dims), _i32]
_lib.moe_prefill_workspace_bytes.restype = _sz
_lib.moe_prefill_layer.argtypes = [_vp, ctypes.POINTER(moe_layer_w), _vp, _i32, _vp, _vp, _vp, _sz, _vp]
_lib.moe_prefill_layer.restype = ctypes.c_int
_lib.moe_strerror.argtypes = [ctypes.c_int]
_lib.moe_strerror.restype = ctypes.c_char_p


def lib() -> ctypes.CDLL:
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, what)


def make_dims(hidden: int, n_experts: int, top_k: int, inter: int, max_rows: int) -> moe_dims:
    return moe_dims(hidden, n_experts, top_k, inter, max_rows)


def make_layer_w(router: int, gateup_nib: int, gateup_scale: int, down_nib: int, down_scale: int,
                 slot_of_expert: int = 0, n_slots: int = 0) -> moe_layer_w:
    """Device pointers of one layer; slot_of_expert (device int32 [E], or 0) maps each
    expert to an entry of a bank of n_slots packed experts that the four weight pointers
    address."""
    return moe_layer_w(router, gateup_nib, gateup_scale, down_nib, down_scale, slot_of_expert or None,
                       int(n_slots))


def moe_strerror(code: int) -> str:
    return _lib.moe_strerror(int(code)).decode()


def moe_create(dims: moe_dims, device: int = 0) -> int:
    h = _vp()
    _check(_lib.moe_create(ctypes.byref(dims), int(device), ctypes.byref(h)), "moe_create")
    return h.value


def moe_destroy(handle: int) -> None:
    _lib.moe_destroy(handle)


def moe_workspace_bytes(dims: moe_dims, rows: int) -> int:
    return int(_lib.moe_workspace_bytes(ctypes.byref(dims), int(rows)))


def moe_packed_bytes(dims: moe_dims, which: int, part: int) -> int:
    return int(_lib.moe_packed_bytes(ctypes.byref(dims), int(which), int(part)))


def moe_pack_q4(dims: moe_dims, which: int, n_experts: int, q_a: int, s_a: int, q_b: int, s_b: int,
                nib_out: int, scale_out: int) -> None:
    """Host packer; all pointers are HOST addresses (e.g. ndarray.ctypes.data)."""
    _check(_lib.moe_pack_q4(ctypes.byref(dims), int(which), int(n_experts), q_a, s_a, q_b, s_b,
                            nib_out, scale_out), "moe_pack_q4")


def moe_route(handle: int, w: moe_layer_w, x_bf16: int, rows: int, topk_ids: int, topk_w: int,
              union_ids: int, n_union: int, ws: int, ws_bytes: int, stream: int) -> None:
    _check(_lib.moe_route(handle, ctypes.byref(w), x_bf16, int(rows), topk_ids, topk_w, union_ids,
                          n_union, ws, int(ws_bytes), stream), "moe_route")


def moe_decode_layer(handle: int, w: moe_layer_w, x_bf16: int, rows: int, out: int, ws: int,
                     ws_bytes: int, stream: int) -> None:
    _check(_lib.moe_decode_layer(handle, ctypes.byref(w), x_bf16, int(rows), out, ws, int(ws_bytes),
                                 stream), "moe_decode_layer")


def moe_prefill_workspace_bytes(dims: moe_dims, tokens: int) -> int:
    return int(_lib.moe_prefill_workspace_bytes(ctypes.byref(dims), int(tokens)))


def moe_prefill_layer(handle: int, w: moe_layer_w, x_bf16: int, tokens: int, out: int, expert_counts: int,
                      ws: int, ws_bytes: int, stream: int) -> None:
    _check(_lib.moe_prefill_layer(handle, ctypes.byref(w), x_bf16, int(tokens), out, expert_counts, ws,
                                  int(ws_bytes), stream), "moe_prefill_layer")


def moe_round(handle: int, layers, x_bf16: int, rows: int, out: int, stats: int, ws: int,
              ws_bytes: int, use_graph: bool, stream: int) -> None:
    arr = (moe_layer_w * len(layers))(*layers)
    _check(_lib.moe_round(handle, arr, len(layers), x_bf16, int(rows), out, stats, ws, int(ws_bytes),
                          1 if use_graph else 0, stream), "moe_round")


def moe_round_host(handle: int, dims: moe_dims, layers, x_host: int, rows: int, out_host: int, x_dev: int,
                   out_dev: int, stats: int, ws: int, ws_bytes: int, use_graph: bool, sync: bool,
                   stream: int) -> None:
    """moe_round with the rows read from host memory and the outputs written to host memory
    (x_host, out_host: host addresses; x_dev, out_dev: the device staging buffers)."""
    arr = (moe_layer_w * len(layers))(*layers)
    _check(_lib.moe_round_host(handle, ctypes.byref(dims), arr, len(layers), x_host, int(rows), out_host, x_dev,
                               out_dev, stats, ws, int(ws_bytes), 1 if use_graph else 0, 1 if sync else 0, stream),
           "moe_round_host")


def moe_last_device_status(handle: int, stream: int) -> int:
    return int(_lib.moe_last_device_status(handle, stream))


def moe_last_launch_count(handle: int) -> int:
    return int(_lib.moe_last_launch_count(handle))


def moe_set_wait_limit_ns(handle: int, ns: int) -> None:
    _check(_lib.moe_set_wait_limit_ns(handle, int(ns)), "moe_set_wait_limit_ns")


def moe_set_tail_skip(handle: int, rank: int) -> None:
    """Routing tail skip threshold (1-based rank; 0 = off); see the header."""
    _check(_lib.moe_set_tail_skip(handle, int(rank)), "moe_set_tail_skip")


def moe_profile(handle: int, enable: bool) -> None:
    _check(_lib.moe_profile(handle, 1 if enable else 0), "moe_profile")


def moe_profile_read(handle: int, kind: int):
    """Returns (total_ms, launches) of one kernel kind recorded since moe_profile(h, True)."""
    t = ctypes.c_double()
    n = _i32()
    _check(_lib.moe_profile_read(handle, int(kind), ctypes.byref(t), ctypes.byref(n)), "moe_profile_read")
    return t.value, n.value


def moe_profile_phases(handle: int):
    """Per-phase device time of the last profiled eager moe_round: {phase: (mean_us, max_us)}."""
    n = len(PHASES_WIDE)
    mean = (ctypes.c_double * n)()
    mx = (ctypes.c_double * n)()
    got = int(_lib.moe_profile_phases(handle, mean, mx, n))
    if got < 0:
        _check(got, "moe_profile_phases")
    names = PHASES_SPLIT if got == len(PHASES_SPLIT) else PHASES_WIDE
    return {p: (mean[i], mx[i]) for i, p in enumerate(names[:got])}


def moe_decode_layer_noalloc(dims: moe_dims, w: moe_layer_w, x_bf16: int, rows: int, out: int,
                             dev_status: int, stream: int) -> None:
    """Allocation-free moe_decode_layer on the current device (static device scratch)."""
    _check(_lib.moe_decode_layer_noalloc(ctypes.byref(dims), ctypes.byref(w), x_bf16, int(rows), out,
                                         dev_status, stream), "moe_decode_layer_noalloc")
