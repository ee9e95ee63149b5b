"""Helpers for the GPU tests: device buffers for blobs, workspaces and BF16
bit patterns (kept as int16 tensors so no value conversion ever happens)."""
from __future__ import annotations

import numpy as np
import torch

import lossless_bf16_weight_gb300 as uw
import workloads as wl

TOL = 4 * 2.0 ** -8       # per-element bound: |y - y_ref| <= TOL * sum_k |x_k w_k|


def dev_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def empty_bits(*shape) -> torch.Tensor:
    return torch.empty(*shape, dtype=torch.int16, device="cuda")


def workspace(nbytes: int) -> torch.Tensor:
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    uw.workspace_init(ws)
    return ws


class Compressed:
    """A matrix compressed by the library, with its blob on the device."""

    def __init__(self, w: np.ndarray, blob: np.ndarray | None = None):
        self.w = w
        self.blob = uw.compress(w) if blob is None else blob
        self.desc = uw.blob_info(self.blob)
        self.blob_dev = torch.from_numpy(self.blob).cuda()

    def ws(self, batch: int = 0, plan=None) -> torch.Tensor:
        return workspace(uw.workspace_size(self.desc, batch, plan))

    def decompress(self) -> np.ndarray:
        out = empty_bits(self.desc.rows, self.desc.cols)
        ws = self.ws()
        uw.decompress(self.desc, self.blob_dev, out, ws)
        assert uw.check_status(ws) == 0
        return host_bits(out)

    def matmul(self, x_dev: torch.Tensor, plan=None, ws=None) -> np.ndarray:
        y = empty_bits(x_dev.shape[0], self.desc.rows)
        ws = self.ws(x_dev.shape[0], plan) if ws is None else ws
        uw.matmul(self.desc, self.blob_dev, x_dev, y, ws, plan)
        assert uw.check_status(ws) == 0
        return host_bits(y)


def matmul_bf16(w_dev: torch.Tensor, x_dev: torch.Tensor, variant: int = -1) -> np.ndarray:
    rows, cols = w_dev.shape
    ws = workspace(uw.workspace_size_bf16(rows, cols, x_dev.shape[0], variant))
    y = empty_bits(x_dev.shape[0], rows)
    uw.matmul_bf16(w_dev, x_dev, y, ws, variant)
    torch.cuda.synchronize()
    return host_bits(y)


def assert_within_bound(y_bits: np.ndarray, y_ref: np.ndarray, absum: np.ndarray):
    y = wl.bf16_to_f32(y_bits).astype(np.float64)
    err = np.abs(y - y_ref)
    bound = TOL * absum
    bad = ~(err <= bound)
    assert not bad.any(), "max err/bound %.3g at %s (of %d bad)" % (
        float(np.max(err / np.maximum(bound, 1e-300))), np.argwhere(bad)[:3].tolist(), int(bad.sum()))
