"""Packing and upload of layer weights into device memory (torch tensors).

The packer itself is the library's host routine ``moe_pack_q4``; this module only
parallelises it over experts (ctypes releases the GIL), stages the packed bytes in
pinned host memory and copies them to the device.  Callers supply the unpacked
codes and scales through ``expert_fn(e)``.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

from . import (MOE_DOWN, MOE_GATEUP, make_layer_w, moe_dims, moe_pack_q4, moe_packed_bytes,
               moe_workspace_bytes)


@dataclass
class DeviceLayer:
    router: torch.Tensor      # fp32 [E][H]
    gu_nib: torch.Tensor      # uint8
    gu_sc: torch.Tensor       # int16 (fp16 bits)
    dn_nib: torch.Tensor      # uint8
    dn_sc: torch.Tensor       # int16 (fp16 bits)

    @property
    def w(self):
        return make_layer_w(self.router.data_ptr(), self.gu_nib.data_ptr(), self.gu_sc.data_ptr(),
                            self.dn_nib.data_ptr(), self.dn_sc.data_ptr())

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.router, self.gu_nib, self.gu_sc,
                                                          self.dn_nib, self.dn_sc))


class Packer:
    """Reusable pinned staging for packing one layer at a time."""

    def __init__(self, dims: moe_dims):
        self.dims = dims
        E = dims.n_experts
        self.sizes = {
            "gu_nib": moe_packed_bytes(dims, MOE_GATEUP, 0), "gu_sc": moe_packed_bytes(dims, MOE_GATEUP, 1),
            "dn_nib": moe_packed_bytes(dims, MOE_DOWN, 0), "dn_sc": moe_packed_bytes(dims, MOE_DOWN, 1)}
        self.host = {k: torch.empty(E * v, dtype=torch.uint8, pin_memory=torch.cuda.is_available())
                     for k, v in self.sizes.items()}
        self.np = {k: t.numpy() for k, t in self.host.items()}

    def pack_expert(self, e: int, ew) -> None:
        d, s, n = self.dims, self.sizes, self.np
        moe_pack_q4(d, MOE_GATEUP, 1, ew.qg.ctypes.data, ew.sg.ctypes.data, ew.qu.ctypes.data,
                    ew.su.ctypes.data, n["gu_nib"][e * s["gu_nib"]:].ctypes.data,
                    n["gu_sc"][e * s["gu_sc"]:].ctypes.data)
        moe_pack_q4(d, MOE_DOWN, 1, ew.qd.ctypes.data, ew.sd.ctypes.data, None, None,
                    n["dn_nib"][e * s["dn_nib"]:].ctypes.data, n["dn_sc"][e * s["dn_sc"]:].ctypes.data)

    def pack_all(self, expert_fn, threads: int = 0) -> None:
        E = self.dims.n_experts
        threads = threads or min(E, os.cpu_count() or 1)

        def one(e):
            self.pack_expert(e, expert_fn(e))
        if threads > 1:
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(one, range(E)))
        else:
            for e in range(E):
                one(e)

    def upload(self, router: np.ndarray, device, stream=None) -> DeviceLayer:
        dev = torch.device(device)
        r = torch.from_numpy(np.ascontiguousarray(router, np.float32)).to(dev, non_blocking=False)
        out = {k: torch.empty_like(v, device=dev) for k, v in self.host.items()}
        for k in out:
            out[k].copy_(self.host[k], non_blocking=True)
        torch.cuda.synchronize(dev)  # staging is reused by the next layer
        return DeviceLayer(r, out["gu_nib"], out["gu_sc"].view(torch.int16), out["dn_nib"],
                           out["dn_sc"].view(torch.int16))


def upload_layer(dims: moe_dims, router: np.ndarray, expert_fn, device="cuda", packer: Packer | None = None,
                 threads: int = 0) -> DeviceLayer:
    p = packer or Packer(dims)
    p.pack_all(expert_fn, threads)
    return p.upload(router, device)


def workspace(dims: moe_dims, rows: int, device="cuda") -> torch.Tensor:
    n = moe_workspace_bytes(dims, rows)
    if n == 0:
        raise ValueError("invalid dims or rows for a workspace")
    return torch.empty(n, dtype=torch.uint8, device=device)
