"""Sizes that are not whole tiles: partial row tiles (per slot, block or part),
partial column tiles and partial K blocks, on the GPU against the oracle.

Every output sits inside a larger buffer whose guard elements before and after
it hold a sentinel: the clipped stores must leave them untouched.
"""

import numpy as np
import pytest
import torch

import oracle
from tensor_comm_gemm_gb300 import synth
from tensor_comm_gemm_gb300 import tpoverlap as t
from gpu_util import AgRun, KsplitRun, assert_close, host_bits, host_f64, staging_view

pytestmark = pytest.mark.gpu

GUARD = 64          # bf16 elements on each side of an output (128 bytes)
SENTINEL = 0x7F7F   # bf16 bits of a large finite value no result takes


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()


class Guarded:
    """An [rows, cols] bf16 output with sentinel guards around it."""

    def __init__(self, rows, cols):
        self.buf = torch.empty(rows * cols + 2 * GUARD, dtype=torch.bfloat16, device="cuda")
        self.buf.view(torch.int16).fill_(SENTINEL)
        self.y = self.buf[GUARD:GUARD + rows * cols].view(rows, cols)

    def poison(self):
        self.y.fill_(float("nan"))

    def guards_intact(self):
        bits = self.buf.view(torch.int16).cpu().numpy().view(np.uint16)
        return bool(np.all(bits[:GUARD] == SENTINEL) and np.all(bits[-GUARD:] == SENTINEL))


# (tp, n, k, m, dtype): rows per slot not a multiple of 128, m not a multiple of
# 256 (nor of 32), k not a whole 128-byte block; the smallest legal sizes
AG_RAGGED = [(3, 600, 200, 264, "bf16"), (2, 1000, 48, 520, "e4m3"), (5, 5, 8, 8, "bf16"),
             (4, 1200, 1000, 1000, "bf16"), (1, 130, 24, 40, "bf16"), (16, 16 * 70, 80, 136, "e4m3"),
             (2, 2 * 640, 264, 776, "bf16"),
             # whole 256-row slots (CTA pairs) with partial column and K tiles
             (2, 1024, 200, 520, "bf16"), (4, 2048, 144, 264, "e4m3")]


@pytest.mark.parametrize("tp,n,k,m,dtype", AG_RAGGED)
def test_ag_ragged_parity_every_observer(tp, n, k, m, dtype):
    wl = synth.make_ag(tp, n, k, m, seed=70 + tp, dist="uniform", dtype=dtype)
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0], wl.scale_inv_x, wl.scale_inv_w)
    run = AgRun(wl)
    out = Guarded(n, m)
    try:
        t.tpo_set_opt(run.ctx, "tail_split", 0)   # whole tiles: modes 0, 1 and 4 give the same bits
        first = None
        for self_rank in sorted({0, tp - 1}):
            t.tpo_set_opt(run.ctx, "self_rank", self_rank)
            for mode in (0, 1, 4):
                t.tpo_set_opt(run.ctx, "mode", mode)
                out.poison()
                run.run(y=out.y)
                assert out.guards_intact(), ("store outside the output", self_rank, mode)
                if first is None:
                    assert_close(host_f64(out.y), ref, dtype)
                    first = host_bits(out.y)
                assert np.array_equal(host_bits(out.y), first), (self_rank, mode)
    finally:
        run.close()


def test_ag_ragged_staging_is_exact_gather():
    wl = synth.make_ag(3, 600, 200, 264, seed=9, dist="uniform")
    run = AgRun(wl)
    try:
        view = staging_view(run.ctx, wl.n * wl.k * 2)
        view.fill_(0xAB)
        torch.cuda.synchronize()
        run.run()
        got = view.cpu().numpy().view(np.uint16).reshape(wl.n, wl.k)
        assert np.array_equal(got, oracle.gather(wl.x))
    finally:
        run.close()


def test_ag_noalloc_ragged_matches_context_path():
    wl = synth.make_ag(3, 600, 200, 264, seed=12, dist="uniform")
    run = AgRun(wl)
    out = Guarded(wl.n, wl.m)
    try:
        t.tpo_set_opt(run.ctx, "tail_split", 0)   # the no-alloc entry point computes whole tiles
        run.run()
        want = host_bits(run.y)
        out.poison()
        t.tpo_ag_gemm_noalloc(wl.tp, wl.n, wl.k, wl.m, t.TPO_BF16, run.xs, run.w, out.y)
        assert out.guards_intact()
        assert np.array_equal(host_bits(out.y), want)
    finally:
        run.close()


# (op, tp, n, k, m, chunks, dtype)
KSPLIT_RAGGED = [("rs", 3, 390, 48, 24, 1, "bf16"), ("rs", 2, 1030, 96, 776, 1, "bf16"),
                 ("rs", 4, 4 * 300, 4 * 208, 520, 1, "e4m3"), ("ar", 2, 600, 32, 40, 3, "bf16"),
                 ("ar", 4, 2056, 64, 272, 2, "bf16"), ("ar", 3, 3 * 2 * 90, 3 * 48, 264, 2, "e4m3"),
                 ("ar", 2, 2 * 700, 2 * 136, 1000, 1, "bf16"),
                 # CTA pairs with partial column and K tiles
                 ("rs", 2, 1024, 2 * 104, 520, 1, "bf16"), ("ar", 2, 2048, 2 * 72, 264, 2, "bf16")]


@pytest.mark.parametrize("op,tp,n,k,m,chunks,dtype", KSPLIT_RAGGED)
def test_ksplit_ragged_parity(op, tp, n, k, m, chunks, dtype):
    wl = synth.make_ksplit(op, tp, n, k, m, seed=80 + tp, n_row_chunks=chunks, dtype=dtype,
                           sigma=(k ** -0.25) if dtype == "bf16" else 1.0)
    ref = oracle.ksplit(wl.x, wl.w, sx=wl.scale_inv_x, sw=wl.scale_inv_w)
    run = KsplitRun(wl)
    try:
        if op == "rs":
            outs = [Guarded(n // tp, m) for _ in range(tp)]
            for o in outs:
                o.poison()
            t.tpo_gemm_rs(run.ctx, run.xs, run.ws, [o.y for o in outs])
            assert t.tpo_sync_status(run.ctx) == 0, t.tpo_last_error()
            assert all(o.guards_intact() for o in outs)
            got = np.concatenate([host_f64(o.y) for o in outs], 0)
            bits = [host_bits(o.y) for o in outs]
            # the per-rank-partial epilogue reduction in fp32 meets the same bar
            t.tpo_set_opt(run.ctx, "reduce", 1)
            for o in outs:
                o.poison()
            t.tpo_gemm_rs(run.ctx, run.xs, run.ws, [o.y for o in outs])
            assert t.tpo_sync_status(run.ctx) == 0, t.tpo_last_error()
            assert all(o.guards_intact() for o in outs)
            assert_close(np.concatenate([host_f64(o.y) for o in outs], 0), ref, dtype)
            t.tpo_set_opt(run.ctx, "reduce", 0)
            t.tpo_gemm_rs(run.ctx, run.xs, run.ws, [o.y for o in outs])
            assert t.tpo_sync_status(run.ctx) == 0
            assert all(np.array_equal(host_bits(o.y), b) for o, b in zip(outs, bits))
        else:
            out = Guarded(n, m)
            out.poison()
            t.tpo_gemm_ar(run.ctx, run.xs, run.ws, out.y, chunks)
            assert t.tpo_sync_status(run.ctx) == 0, t.tpo_last_error()
            assert out.guards_intact()
            got = host_f64(out.y)
            ptr, target = t.tpo_done_counters(run.ctx)
            cnt = torch.as_tensor(_Words(ptr, chunks), device="cuda").cpu().numpy()
            assert target > 0 and np.all(cnt == target), (cnt, target)
        assert_close(got, ref, dtype)
    finally:
        run.close()


class _Words:
    def __init__(self, ptr, count):
        self.__cuda_array_interface__ = {"shape": (count,), "typestr": "<u4", "data": (ptr, False), "version": 3}


def test_ar_ragged_one_chunk_equals_rs_bitwise():
    """With one row chunk AR part b and RS block b sum in the same ring order,
    also when the parts are not whole tiles."""
    wl = synth.make_ksplit("ar", 3, 3 * 150, 3 * 64, 136, seed=5, n_row_chunks=1, sigma=192 ** -0.25)
    run = KsplitRun(wl)
    try:
        run.ar(1)
        ar = host_bits(run.y)
        run.rs()
        rs = np.concatenate([host_bits(y) for y in run.yb], 0)
        assert np.array_equal(ar, rs)
    finally:
        run.close()


@pytest.mark.parametrize("tp,n,k,m,dtype", [(3, 600, 200, 264, "bf16"), (2, 1000, 48, 520, "e4m3"),
                                            (4, 1200, 1000, 1000, "bf16")])
@pytest.mark.parametrize("gemm_ctas", [2, 5])
def test_ag_ragged_several_tiles_per_cta_every_launch(tp, n, k, m, dtype, gemm_ctas):
    """Few GEMM CTAs, so that each stores several ragged tiles one after the
    other, and repeated launches: an output box past the edge must not give
    up a staging buffer that a store in flight still reads."""
    wl = synth.make_ag(tp, n, k, m, seed=60 + tp, dist="uniform", dtype=dtype)
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0], wl.scale_inv_x, wl.scale_inv_w)
    run = AgRun(wl)
    out = Guarded(n, m)
    try:
        t.tpo_set_opt(run.ctx, "gemm_ctas", gemm_ctas)
        t.tpo_set_opt(run.ctx, "tail_split", 0)
        first = None
        for _ in range(6):
            out.poison()
            run.run(y=out.y)
            assert out.guards_intact()
            if first is None:
                assert_close(host_f64(out.y), ref, dtype)
                first = host_bits(out.y)
            assert np.array_equal(host_bits(out.y), first)
    finally:
        run.close()


@pytest.mark.parametrize("op,tp,n,k,m,chunks,dtype", [("rs", 3, 390, 48, 24, 1, "bf16"),
                                                       ("ar", 2, 600, 32, 40, 3, "bf16"),
                                                       ("rs", 2, 1030, 96, 776, 1, "bf16")])
def test_ksplit_ragged_several_tiles_per_cta_every_launch(op, tp, n, k, m, chunks, dtype):
    wl = synth.make_ksplit(op, tp, n, k, m, seed=85 + tp, n_row_chunks=chunks, dtype=dtype, sigma=k ** -0.25)
    ref = oracle.ksplit(wl.x, wl.w, sx=wl.scale_inv_x, sw=wl.scale_inv_w)
    run = KsplitRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "gemm_ctas", 2)
        first = None
        for _ in range(6):
            if op == "rs":
                for y in run.yb:
                    y.fill_(float("nan"))
                t.tpo_gemm_rs(run.ctx, run.xs, run.ws, run.yb)
                assert t.tpo_sync_status(run.ctx) == 0, t.tpo_last_error()
                got = np.concatenate([host_f64(y) for y in run.yb], 0)
                bits = np.concatenate([host_bits(y) for y in run.yb], 0)
            else:
                run.y.fill_(float("nan"))
                t.tpo_gemm_ar(run.ctx, run.xs, run.ws, run.y, chunks)
                assert t.tpo_sync_status(run.ctx) == 0, t.tpo_last_error()
                got, bits = host_f64(run.y), host_bits(run.y)
            if first is None:
                assert_close(got, ref, dtype)
                first = bits
            assert np.array_equal(bits, first)
    finally:
        run.close()
