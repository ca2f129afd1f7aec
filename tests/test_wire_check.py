"""The GPU tests' check of the bf16-wire reduction (option reduce=2), run on
the CPU against a simulation of the kernel's arithmetic.

The kernel forms each rank's partial as an fp32 tensor-core sum, rounds it
(times the e4m3 scales) to bf16, adds it in fp32 to the bf16 running sum
received from the previous hop and rounds that to bf16, the ranks of a row in
the ring order that ends at the row's owner.  The simulation does the same
with fp32 sums taken left to right.  The check must accept it, and must
reject the plausible mistakes: the ring starting at the owner, running sums
kept in fp32, partials not rounded.  One case is built so that a partial
nearly cancels: there the fp32 sum is off by more than a bf16 spacing of the
exact value, which the check's bound has to allow for.
"""

import types

import numpy as np
import pytest

from tensor_comm_gemm_gb300 import synth
from gpu_util import check_wire, decode, row_owners, wire_expectation


def round_bf16(a: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bf16 value, ties to even (finite inputs)."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def fp32_partial(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """X . W^T summed in fp32 over K, left to right (each product of two bf16 or
    e4m3 values is exact in fp32)."""
    xd, wd = decode(x).astype(np.float32), decode(w).astype(np.float32)
    acc = np.zeros((xd.shape[0], wd.shape[0]), dtype=np.float32)
    for q in range(xd.shape[1]):
        acc = (acc + np.outer(xd[:, q], wd[:, q]).astype(np.float32)).astype(np.float32)
    return acc


def simulate(wl, op, chunks, start=1, round_sums=True, round_parts=True):
    """The kernel's bf16-ring arithmetic; `start` = 1 begins each row's ring
    after its owner (the kernel's order), 0 at the owner."""
    tp = wl.tp
    scale = np.float32(wl.scale_inv_x * wl.scale_inv_w) if wl.dtype == "e4m3" else np.float32(1.0)
    parts = [(fp32_partial(wl.x[r], wl.w[r]) * scale).astype(np.float32) for r in range(tp)]
    owners = row_owners(op, wl.n, tp, chunks)
    out = np.zeros(parts[0].shape, dtype=np.float32)
    for b in range(tp):
        rows = owners == b
        s = None
        for j in range(tp):
            r = (b + start + j) % tp
            p = round_bf16(parts[r][rows]) if round_parts else parts[r][rows]
            if s is None:
                s = p
            else:
                s = (s + p).astype(np.float32)
                if round_sums:
                    s = round_bf16(s)
        out[rows] = round_bf16(s)
    return out.astype(np.float64)


CASES = [("rs", 3, 192, 96, 48, 1, "bf16"), ("rs", 4, 256, 128, 40, 1, "bf16"), ("ar", 2, 256, 64, 64, 2, "bf16"),
         ("rs", 4, 128, 128, 32, 1, "e4m3"), ("rs", 1, 96, 64, 40, 1, "bf16")]


@pytest.mark.parametrize("op,tp,n,k,m,chunks,dtype", CASES)
def test_check_accepts_the_kernels_arithmetic(op, tp, n, k, m, chunks, dtype):
    wl = synth.make_ksplit(op, tp, n, k, m, seed=40 + tp, n_row_chunks=chunks, dtype=dtype,
                           sigma=(k ** -0.25) if dtype == "bf16" else 1.0)
    ref, risky, bound = wire_expectation(wl, op, chunks)
    check_wire(simulate(wl, op, chunks), ref, risky, bound, dtype)


MISTAKES = {"ring starts at the owner": {"start": 0}, "running sums kept in fp32": {"round_sums": False},
            "partials not rounded": {"round_parts": False}}


@pytest.mark.parametrize("mistake", sorted(MISTAKES))
@pytest.mark.parametrize("op,tp,n,k,m,chunks,dtype", [c for c in CASES if c[1] >= 3])
def test_check_rejects_each_mistake(op, tp, n, k, m, chunks, dtype, mistake):
    wl = synth.make_ksplit(op, tp, n, k, m, seed=40 + tp, n_row_chunks=chunks, dtype=dtype,
                           sigma=(k ** -0.25) if dtype == "bf16" else 1.0)
    ref, risky, bound = wire_expectation(wl, op, chunks)
    with pytest.raises(AssertionError):
        check_wire(simulate(wl, op, chunks, **MISTAKES[mistake]), ref, risky, bound, dtype)


def bf16_bits(v) -> np.ndarray:
    return (np.asarray(v, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def test_bound_covers_a_nearly_cancelling_partial():
    """One rank (the reduce-scatter of tp = 1): the result is the rounded
    partial.  Row 0's terms are 1, 2^-30, -1: the exact partial is 2^-30, the
    fp32 sum taken left to right gives 0, so the rounded results differ by
    2^-30, far more than one bf16 spacing of the exact value."""
    x = bf16_bits([[1.0, 2.0 ** -30, -1.0], [0.5, 0.25, 0.125]])
    w = bf16_bits([[1.0, 1.0, 1.0], [1.0, -1.0, 0.5], [0.75, 0.5, 0.25], [2.0, 1.0, -1.0]])
    wl = types.SimpleNamespace(tp=1, n=2, x=[x], w=[w], dtype="bf16", scale_inv_x=1.0, scale_inv_w=1.0)
    got = simulate(wl, "rs", 1)
    ref, risky, bound = wire_expectation(wl, "rs", 1)
    assert ref[0, 0] == 2.0 ** -30 and got[0, 0] == 0.0
    assert abs(got[0, 0] - ref[0, 0]) > 2.0 ** -5 * abs(ref[0, 0])   # beyond a spacing of the exact value
    check_wire(got, ref, risky, bound, "bf16")
