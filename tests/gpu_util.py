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


# ---------------------------------------------------------------- bf16 ring (wire) reduction

def decode(a: np.ndarray) -> np.ndarray:
    """Values of bf16 bit patterns (uint16) or e4m3 codes (uint8) as float64."""
    if a.dtype == np.uint16:
        return synth.bf16_bits_to_f32(a).astype(np.float64)
    return synth.e4m3_bits_to_f32(a).astype(np.float64)


def row_owners(op: str, n: int, tp: int, chunks: int) -> np.ndarray:
    """Rank each output row's ring sum ends at: its row block (reduce-scatter)
    or its ring-order part of a row chunk (all-reduce)."""
    i = np.arange(n)
    if op == "rs":
        return i // (n // tp)
    rows_chunk = n // chunks
    return (i % rows_chunk) // (rows_chunk // tp)


def near_bf16_boundary(p: np.ndarray, eps: np.ndarray) -> np.ndarray:
    """True where a value within eps of p could round to a different bf16
    value than p: a rounding midpoint or a power of two (where the spacing
    changes) lies within eps."""
    a = np.abs(p)
    tiny = 2.0 ** -140
    e = np.floor(np.log2(np.maximum(a, tiny)))
    h = 2.0 ** np.maximum(e - 7, -133)            # bf16 spacing in a's binade
    frac = a / h - np.floor(a / h)
    near_mid = np.abs(frac - 0.5) * h <= eps
    near_edge = np.floor(np.log2(np.maximum(a - eps, tiny))) != np.floor(np.log2(np.maximum(a + eps, tiny)))
    return (near_mid | near_edge) & (eps > 0)


def wire_expectation(wl, op: str, chunks: int):
    """What the bf16-ring mode (option reduce=2) must produce, from the oracle.

    Returns (ref, risky, bound): the oracle's ring sum; per element, whether
    any rank's exact partial P_r lies within eps_r of a bf16 rounding
    boundary; and a bound on |result - ref|.  The kernel's partials are fp32
    tensor-core sums, |P~_r - P_r| <= eps_r = (kr + 2) 2^-22 scale
    sum_q |x_q w_q| (four times the first-order bound of a recursive fp32 sum
    of kr products, plus the fp32 scale multiplies).  Where no partial is at
    risk, every rounded partial equals the oracle's and the same fp32 hops on
    the same values give the same bits.  Elsewhere a rounded partial can be
    off by the partial's own fp32 error plus one bf16 spacing at its computed
    magnitude, eps_r + u(|P_r| + eps_r), and each rounded running sum by one
    spacing at its computed magnitude, u(|S_r| + E_r), E_r the error carried
    into it; later hops carry every difference.  So |result - ref| <= E, E
    accumulated hop by hop in the row's ring order from these terms, S_r the
    exact running sums and u(v) = 2^-6 |v| + 2^-133 (one spacing at |v| and in
    the binade above).  The fp32 error matters where the partial nearly
    cancels: it can then exceed a spacing of the exact value."""
    import oracle

    tp, n = wl.tp, wl.n
    sx = wl.scale_inv_x if wl.dtype == "e4m3" else 1.0
    sw = wl.scale_inv_w if wl.dtype == "e4m3" else 1.0
    scale = sx * sw
    ref = oracle.ksplit_wire_bf16(wl.x, wl.w, op=op, n_chunks=chunks, sx=sx, sw=sw)
    parts = [oracle.ksplit([wl.x[r]], [wl.w[r]], sx=sx, sw=sw) for r in range(tp)]
    kr = wl.x[0].shape[1]
    eps = [(kr + 2) * 2.0 ** -22 * scale * (np.abs(decode(wl.x[r])) @ np.abs(decode(wl.w[r])).T)
           for r in range(tp)]
    owners = row_owners(op, n, tp, chunks)
    risky = np.zeros(ref.shape, dtype=bool)
    bound = np.zeros(ref.shape)
    for b in range(tp):
        rows = owners == b
        run = np.zeros((int(rows.sum()), ref.shape[1]))
        err = np.zeros_like(run)   # E: what the result may differ by after this hop
        for j in range(tp):
            r = (b + 1 + j) % tp
            p, e = parts[r][rows], eps[r][rows]
            run = run + p
            risky[rows] |= near_bf16_boundary(p, e)
            err = err + e + 2.0 ** -6 * (np.abs(p) + e) + 2.0 ** -133   # the rounded partial
            err = err + 2.0 ** -6 * (np.abs(run) + err) + 2.0 ** -133   # the rounded running sum
        bound[rows] = err
    return ref, risky, bound


def check_wire(got, wire_ref, risky, bound, dtype):
    """bf16-ring mode against the oracle's ring sum: bit-equal wherever no
    rank's partial is within its fp32 error of a bf16 rounding boundary (bf16
    inputs), within the rounding bound everywhere, and bit-equal on at least
    WIRE_EXACT_FRAC of all elements (a wrong ring order or a dropped rounding
    changes far more)."""
    assert np.all(np.isfinite(got)), "non-finite outputs"
    diff = np.abs(got - wire_ref)
    if dtype == "bf16":
        safe = ~risky
        assert np.array_equal(got[safe], wire_ref[safe]), "%d of %d elements with no partial near a rounding " \
            "boundary differ" % ((got[safe] != wire_ref[safe]).sum(), safe.sum())
    assert np.all(diff <= bound), "worst excess %.3e" % (diff - bound).max()
    if got.size >= 1000:   # a share is only meaningful over many elements
        frac = float(np.mean(got == wire_ref))
        assert frac >= WIRE_EXACT_FRAC[dtype], "only %.4f of the elements equal the oracle's ring sum" % frac


# Share of elements that must match the oracle's bf16 ring sum bit for bit.  A
# mismatch needs a partial within the kernel's fp32 error of a rounding
# boundary: measured 0.99988-0.99999 of the elements match on the test cases
# (bf16 and e4m3, tp 2 to 8); the kernel's arithmetic simulated on the CPU
# with the ring starting at the owner, or with fp32 running sums, matches
# 0.43-0.78 of them on the tp >= 3 cases.
WIRE_EXACT_FRAC = {"bf16": 0.99, "e4m3": 0.99}
