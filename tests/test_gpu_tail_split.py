"""The AG tail split on the GPU: tail tiles are divided along K among the CTA
groups (tail_split=1: the leftover tiles first, among the GEMM CTAs;
tail_split=2: the last tiles, shared with the producer CTAs once their copy
is done), later parts travel as fp32 partials through the workspace and are
added in K order by the tile's finisher.  Checked against the oracle, across
the modes that share the plan (bitwise), for repeatability, and for the
bounded wait on a partial."""

import numpy as np
import pytest
import torch

import oracle
from tensor_comm_gemm_gb300 import synth
from tensor_comm_gemm_gb300 import tpoverlap as t
from gpu_util import AgRun, assert_close, gather_tiles, host_bits, host_f64, SAMPLE_TILES

pytestmark = pytest.mark.gpu

GUARD = 64
SENTINEL = 0x7F7F


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()


def cdiv(a, b):
    return -(-a // b)


def leftover(ctx, tp, n, m):
    """Tiles mod GEMM CTA groups of the latest launch."""
    cg = t.tpo_get_opt(ctx, "last_cta_group")
    groups = t.tpo_get_opt(ctx, "last_gemm_ctas") // cg
    tiles = tp * cdiv(n // tp, 128 * cg) * cdiv(m, 256)
    return tiles % groups


# (tp, n, k, m, dtype, cta_group, gemm_ctas of schedule 1, gemm_ctas of schedule 2): schedule 1 leaves
# a partial round; schedule 2 (8 producer CTAs) runs two GEMM groups long enough for the producers to join
CASES = [
    (4, 2048, 512, 768, "bf16", 2, 10, 4),     # 24 pair tiles on 5 pairs, 4 K units a tile
    (2, 512, 448, 512, "bf16", 1, 5, 2),       # 7 K blocks: a tile in three parts
    (3, 600, 200, 264, "bf16", 0, 5, 2),       # ragged rows, columns and K
    (2, 1024, 1024, 1024, "e4m3", 2, 6, 4),    # e4m3, one leftover tile in two parts
    (1, 1024, 512, 1280, "bf16", 2, 6, 4),     # tp = 1
    (5, 1280, 320, 512, "bf16", 1, 7, 2),      # odd group count
]


class Guarded:
    def __init__(self, rows, cols):
        self.buf = torch.empty(rows * cols + 2 * GUARD, dtype=torch.bfloat16, device="cuda")
        self.buf.view(torch.int16).fill_(SENTINEL)
        self.y = self.buf[GUARD:GUARD + rows * cols].view(rows, cols)

    def intact(self):
        bits = self.buf.view(torch.int16).cpu().numpy().view(np.uint16)
        return bool(np.all(bits[:GUARD] == SENTINEL) and np.all(bits[-GUARD:] == SENTINEL))


@pytest.mark.parametrize("tp,n,k,m,dtype,cg,gemm1,gemm2", CASES)
@pytest.mark.parametrize("schedule", [1, 2, 3])
def test_split_parity_and_same_bits_in_modes_0_1_2(tp, n, k, m, dtype, cg, gemm1, gemm2, schedule):
    wl = synth.make_ag(tp, n, k, m, seed=90 + tp, dist="normal", sigma=k ** -0.25, dtype=dtype)
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0], wl.scale_inv_x, wl.scale_inv_w)
    run = AgRun(wl)
    out = Guarded(n, m)
    try:
        t.tpo_set_opt(run.ctx, "cta_group", cg)
        t.tpo_set_opt(run.ctx, "gemm_ctas", gemm1 if schedule != 2 else gemm2)
        t.tpo_set_opt(run.ctx, "producer_sms", 0 if schedule != 2 else 8)
        t.tpo_set_opt(run.ctx, "tail_split", schedule)
        out.y.fill_(float("nan"))
        run.run(y=out.y)
        split = t.tpo_get_opt(run.ctx, "last_split_tiles")
        late = t.tpo_get_opt(run.ctx, "last_late_groups")
        assert split > 0
        if schedule != 2:
            assert late == 0 and split == leftover(run.ctx, tp, n, m)
        else:
            assert late > 0
        assert out.intact()
        assert_close(host_f64(out.y), ref, dtype)
        first = host_bits(out.y)
        for mode in (1, 2, 0, 0):
            t.tpo_set_opt(run.ctx, "mode", mode)
            out.y.fill_(float("nan"))
            run.run(y=out.y)
            assert t.tpo_get_opt(run.ctx, "last_split_tiles") == split, mode
            assert t.tpo_get_opt(run.ctx, "last_late_groups") == late, mode
            assert np.array_equal(host_bits(out.y), first), ("split result differs", mode)
        # whole tiles only: the same bar, nothing split
        t.tpo_set_opt(run.ctx, "tail_split", 0)
        t.tpo_set_opt(run.ctx, "mode", 0)
        out.y.fill_(float("nan"))
        run.run(y=out.y)
        assert t.tpo_get_opt(run.ctx, "last_split_tiles") == 0
        assert out.intact()
        assert_close(host_f64(out.y), ref, dtype)
    finally:
        run.close()


@pytest.mark.parametrize("schedule", [1, 2, 3])
def test_split_every_observer_meets_the_bar(schedule):
    tp, n, k, m = 4, 2048, 512, 768
    wl = synth.make_ag(tp, n, k, m, seed=7, dist="uniform")
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0])
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "gemm_ctas", 10 if schedule != 2 else 4)
        t.tpo_set_opt(run.ctx, "producer_sms", 0 if schedule != 2 else 8)
        t.tpo_set_opt(run.ctx, "tail_split", schedule)
        for self_rank in range(tp):
            t.tpo_set_opt(run.ctx, "self_rank", self_rank)
            run.y.fill_(float("nan"))
            run.run()
            assert t.tpo_get_opt(run.ctx, "last_split_tiles") > 0
            assert (t.tpo_get_opt(run.ctx, "last_late_groups") > 0) == (schedule == 2)
            assert_close(host_f64(run.y), ref)
    finally:
        run.close()


def test_split_join_schedule_large_shape():
    """The join schedule on a large shape (24 producer CTAs, so that their copy
    ends early enough to join): sampled parity, modes 0 and 1 agree bitwise."""
    tp, n, k, m = 4, 4096, 1024, 4096
    wl = synth.make_ag(tp, n, k, m, seed=11, dist="normal", sigma=k ** -0.25)
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "tail_split", 2)
        t.tpo_set_opt(run.ctx, "producer_sms", 24)
        run.run()
        assert t.tpo_get_opt(run.ctx, "last_split_tiles") > 0 and t.tpo_get_opt(run.ctx, "last_late_groups") > 0
        bits = host_bits(run.y)
        tiles = synth.sample_tiles(n, m, 16, SAMPLE_TILES, seed=2011)
        ref = oracle.ag(oracle.gather(wl.x), wl.w[0], tiles=tiles)
        assert_close(gather_tiles(host_f64(run.y), tiles), ref)
        t.tpo_set_opt(run.ctx, "mode", 1)
        run.y.fill_(0)
        run.run()
        assert np.array_equal(host_bits(run.y), bits)
    finally:
        run.close()


def test_split_mode_4_matches_whole_tiles():
    """Mode 4 never splits: it agrees bitwise with the unsplit schedule."""
    wl = synth.make_ag(4, 2048, 512, 768, seed=12, dist="uniform")
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "gemm_ctas", 10)
        t.tpo_set_opt(run.ctx, "tail_split", 0)
        run.run()
        whole = host_bits(run.y)
        t.tpo_set_opt(run.ctx, "tail_split", 1)
        t.tpo_set_opt(run.ctx, "mode", 4)
        run.y.fill_(float("nan"))
        run.run()
        assert t.tpo_get_opt(run.ctx, "last_split_tiles") == 0
        assert np.array_equal(host_bits(run.y), whole)
    finally:
        run.close()


def test_missing_partial_times_out_and_context_recovers():
    """A writer that never publishes its partial: the finisher's bounded wait
    ends with a timeout at the partial site; the next call is correct."""
    wl = synth.make_ag(4, 2048, 512, 768, seed=13, dist="uniform")
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0])
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "tail_split", 1)
        t.tpo_set_opt(run.ctx, "gemm_ctas", 10)          # 5 pairs: group 1 (CTAs 2, 3) writes a partial
        t.tpo_set_opt(run.ctx, "wait_timeout_ms", 50)
        t.tpo_set_opt(run.ctx, "debug_skip_partial", 2)
        t.tpo_ag_gemm(run.ctx, run.xs, run.w, run.y)
        assert t.tpo_sync_status(run.ctx) == 4
        code, site, _, _ = t.tpo_last_device_error(run.ctx)
        assert code == 1 and site == 8
        t.tpo_set_opt(run.ctx, "debug_skip_partial", -1)
        t.tpo_set_opt(run.ctx, "wait_timeout_ms", 2000)
        for _ in range(2):
            run.y.fill_(float("nan"))
            run.run()
            assert_close(host_f64(run.y), ref)
    finally:
        run.close()


def test_join_schedule_with_slow_producer_keeps_bits():
    """Schedule 2 with a producer that spins before every publish: the producer
    CTAs join late, the finishers wait longer for their partials, and the
    result is still the bits of the sequential run (same plan)."""
    wl = synth.make_ag(4, 2048, 512, 768, seed=14, dist="uniform")
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "tail_split", 2)
        t.tpo_set_opt(run.ctx, "gemm_ctas", 4)
        t.tpo_set_opt(run.ctx, "producer_sms", 8)
        t.tpo_set_opt(run.ctx, "mode", 1)
        run.run()
        assert t.tpo_get_opt(run.ctx, "last_late_groups") > 0
        want = host_bits(run.y)
        t.tpo_set_opt(run.ctx, "mode", 0)
        t.tpo_set_opt(run.ctx, "debug_delay_ns", 200000)
        for _ in range(2):
            run.y.fill_(float("nan"))
            run.run()
            assert np.array_equal(host_bits(run.y), want)
    finally:
        run.close()


def test_join_schedule_skipped_chunk_times_out_and_recovers():
    """Schedule 2 with a chunk the producer never publishes: the waits on it
    (GEMM and joined producer CTAs alike) end with a timeout; the context then
    gives correct results."""
    wl = synth.make_ag(4, 2048, 512, 768, seed=15, dist="uniform")
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0])
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "tail_split", 2)
        t.tpo_set_opt(run.ctx, "gemm_ctas", 4)
        t.tpo_set_opt(run.ctx, "producer_sms", 8)
        t.tpo_set_opt(run.ctx, "wait_timeout_ms", 50)
        t.tpo_set_opt(run.ctx, "debug_skip_chunk", 2)
        t.tpo_ag_gemm(run.ctx, run.xs, run.w, run.y)
        assert t.tpo_sync_status(run.ctx) == 4
        code, site, _, _ = t.tpo_last_device_error(run.ctx)
        assert code == 1 and site in (1, 2, 3, 4, 5, 8)
        t.tpo_set_opt(run.ctx, "debug_skip_chunk", -1)
        t.tpo_set_opt(run.ctx, "wait_timeout_ms", 2000)
        run.y.fill_(float("nan"))
        run.run()
        assert t.tpo_get_opt(run.ctx, "last_late_groups") > 0
        assert_close(host_f64(run.y), ref)
    finally:
        run.close()
