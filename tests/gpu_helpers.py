"""Shared set-up for GPU tests: generated layers packed and uploaded to the device."""
from __future__ import annotations

import numpy as np
import torch

import spec_verify_layer_gb300 as mv
import syngen
from spec_verify_layer_gb300.weights import Packer, workspace

TOL_MAX_ABS = 2e-3
TOL_REL_L2 = 1e-3
TOL_W = 1e-6


def dims_of(cfg, max_rows=None):
    return mv.make_dims(cfg.hidden, cfg.experts, cfg.top_k, cfg.inter, max_rows or max(cfg.rows, 1))


class Stack:
    """L generated layers of one shape on the device (weights shared by row counts)."""

    def __init__(self, cfg, n_layers, device="cuda", max_rows=32):
        self.cfg = cfg
        self.dims = dims_of(cfg, max_rows)
        self.device = torch.device(device)
        p = Packer(self.dims)
        self.layers = []
        for l in range(n_layers):
            p.pack_all(lambda e, l=l: syngen.expert(cfg, l, e))
            self.layers.append(p.upload(syngen.router(cfg, l), self.device))
        self.handle = mv.moe_create(self.dims, self.device.index or 0)

    def rows(self, layer, n_rows, sigma):
        return syngen.rows(self.cfg, layer, n_rows, sigma)

    def x_dev(self, xb: np.ndarray) -> torch.Tensor:
        return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(self.device)

    def ws(self, rows):
        return workspace(self.dims, rows, self.device)

    def close(self):
        if self.handle:
            mv.moe_destroy(self.handle)
            self.handle = None


def stream_of(dev) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def compare(got: np.ndarray, ref: np.ndarray):
    got = got.astype(np.float64)
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    return err, rel


def assert_close(got, ref, what=""):
    err, rel = compare(got, ref)
    assert err <= TOL_MAX_ABS and rel <= TOL_REL_L2, f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}"
    return err, rel
