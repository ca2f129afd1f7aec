"""Helpers of the GPU tests: device copies of the seeded inputs, tolerance
checks against the oracle, and a zero-copy view of the staging buffer."""

import numpy as np
import torch

from tensor_comm_gemm_gb300 import synth
from tensor_comm_gemm_gb300 import tpoverlap as t

# Tolerances of the parity bar: relative Frobenius error and per-element bound
# |err| <= c * (|ref| + 1), c = 1e-2 for bf16 inputs, 3e-2 for e4m3 inputs.
FROB_TOL = 5e-3
ELEM_TOL = {"bf16": 1e-2, "e4m3": 3e-2}
SAMPLE_TILES = 4096
SAMPLE_TILE = 16


def dev(a: np.ndarray) -> torch.Tensor:
    """Device copy of a uint16 (bf16 bits) or uint8 (e4m3 codes) array."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_f64(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().double().numpy()


def host_bits(y: torch.Tensor) -> np.ndarray:
    return y.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str = "bf16"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), "non-finite outputs"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    bound = ELEM_TOL[dtype] * (np.abs(ref) + 1.0)
    bad = np.abs(got - ref) > bound
    assert rel <= FROB_TOL, "relative Frobenius error %.3e" % rel
    assert not bad.any(), "%d elements outside tolerance, worst %.3e" % (bad.sum(), (np.abs(got - ref) - bound).max())
    return rel


def gather_tiles(y: np.ndarray, tiles: np.ndarray, tile: int = SAMPLE_TILE) -> np.ndarray:
    return np.stack([y[r:r + tile, c:c + tile] for r, c in tiles])


def staging_view(ctx, nbytes: int) -> torch.Tensor:
    """uint8 view of the context's staging buffer (no copy)."""
    class _Arr:
        __cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                    "data": (t.tpo_staging_ptr(ctx), False), "version": 3}
    return torch.as_tensor(_Arr(), device="cuda")


class AgRun:
    """Device buffers and a context for one AG workload."""

    def __init__(self, wl: synth.Workload):
        self.wl = wl
        self.fp8 = wl.dtype == "e4m3"
        self.xs = [dev(x) for x in wl.x]
        self.w = dev(wl.w[0])
        self.y = torch.empty((wl.n, wl.m), dtype=torch.bfloat16, device="cuda")
        self.sx = torch.tensor([wl.scale_inv_x], dtype=torch.float32, device="cuda") if self.fp8 else None
        self.sw = torch.tensor([wl.scale_inv_w], dtype=torch.float32, device="cuda") if self.fp8 else None
        self.ctx = t.tpo_ctx_create(wl.tp, wl.n, wl.k, wl.m, t.TPO_FP8_E4M3 if self.fp8 else t.TPO_BF16)

    def run(self, y=None, sync=True):
        t.tpo_ag_gemm(self.ctx, self.xs, self.w, self.y if y is None else y, self.sx, self.sw)
        if sync:
            st = t.tpo_sync_status(self.ctx)
            assert st == 0, t.tpo_last_error()

    def close(self):
        t.tpo_ctx_destroy(self.ctx)


class KsplitRun:
    def __init__(self, wl: synth.Workload):
        self.wl = wl
        self.xs = [dev(x) for x in wl.x]
        self.ws = [dev(x) for x in wl.w]
        tp, n, m = wl.tp, wl.n, wl.m
        self.y = torch.empty((n, m), dtype=torch.bfloat16, device="cuda")
        self.yb = [torch.empty((n // tp, m), dtype=torch.bfloat16, device="cuda") for _ in range(tp)]
        self.fp8 = wl.dtype == "e4m3"
        self.ctx = t.tpo_ctx_create(tp, n, wl.k, m, t.TPO_FP8_E4M3 if self.fp8 else t.TPO_BF16)
        if self.fp8:
            self.sx = torch.tensor([wl.scale_inv_x], dtype=torch.float32, device="cuda")
            self.sw = torch.tensor([wl.scale_inv_w], dtype=torch.float32, device="cuda")
            t.tpo_set_fp8_scales(self.ctx, self.sx, self.sw)

    def rs(self, sync=True):
        t.tpo_gemm_rs(self.ctx, self.xs, self.ws, self.yb)
        if sync:
            assert t.tpo_sync_status(self.ctx) == 0, t.tpo_last_error()

    def ar(self, chunks, sync=True):
        t.tpo_gemm_ar(self.ctx, self.xs, self.ws, self.y, chunks)
        if sync:
            assert t.tpo_sync_status(self.ctx) == 0, t.tpo_last_error()

    def close(self):
        t.tpo_ctx_destroy(self.ctx)
