"""Dynamic tiles (option sched): CTA groups claim their tiles from a
launch-wide counter instead of taking a fixed round robin.  Every tile is
computed the same way whichever group takes it, so the results are bitwise
those of the round robin, in every operation, mode and reduction mode, over
repeated calls (the counter keeps running from launch to launch), and the
automatic choice takes dynamic tiles exactly for launches of at least 8
rounds.  A device timeout with dynamic tiles leaves the context usable."""

import numpy as np
import pytest
import torch

import oracle
from tensor_comm_gemm_gb300 import synth
from tensor_comm_gemm_gb300 import tpoverlap as t
from gpu_util import AgRun, KsplitRun, assert_close, host_bits, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()


def _ag_bits(run, sched, gemm_ctas, mode=0):
    t.tpo_set_opt(run.ctx, "sched", sched)
    t.tpo_set_opt(run.ctx, "gemm_ctas", gemm_ctas)
    t.tpo_set_opt(run.ctx, "mode", mode)
    run.y.fill_(float("nan"))
    run.run()
    assert t.tpo_get_opt(run.ctx, "last_sched") == (2 if sched == 2 else 1)
    return host_bits(run.y)


# (tp, n, k, m, dtype): many tiles on few GEMM CTAs, ragged sizes, both MMA variants
AG_CASES = [(4, 2048, 512, 1024, "bf16"), (3, 600, 200, 264, "bf16"), (2, 1024, 384, 776, "e4m3"),
            (1, 256, 64, 2048, "bf16")]


@pytest.mark.parametrize("tp,n,k,m,dtype", AG_CASES)
def test_ag_dynamic_tiles_bit_identical(tp, n, k, m, dtype):
    if dtype == "bf16":
        wl = synth.make_ag(tp, n, k, m, seed=80 + tp, dist="normal", sigma=k ** -0.25)
    else:
        wl = synth.make_ag(tp, n, k, m, seed=80 + tp, dtype="e4m3")
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0], wl.scale_inv_x, wl.scale_inv_w)
    run = AgRun(wl)
    try:
        first = _ag_bits(run, 1, 0)
        assert_close(host_f64(run.y), ref, dtype)
        for mode in (0, 1, 2, 4):
            for gemm_ctas in (2, 4, 6, 0):
                for rep in range(2):  # repeated calls: the claim counter runs on
                    bits = _ag_bits(run, 2, gemm_ctas, mode)
                    assert np.array_equal(bits, first), (mode, gemm_ctas, rep)
    finally:
        run.close()


@pytest.mark.parametrize("op,tp,n,k,m,chunks,dtype", [("rs", 4, 1024, 1280, 768, 1, "bf16"),
                                                      ("ar", 2, 2048, 512, 520, 2, "bf16"),
                                                      ("rs", 3, 390, 48, 24, 1, "bf16"),
                                                      ("ar", 3, 2304, 384, 1024, 3, "e4m3")])
def test_ksplit_dynamic_tiles_bit_identical_with_done_counters(op, tp, n, k, m, chunks, dtype):
    if dtype == "bf16":
        wl = synth.make_ksplit(op, tp, n, k, m, seed=90 + tp, dist="normal", sigma=k ** -0.25, n_row_chunks=chunks)
    else:
        wl = synth.make_ksplit(op, tp, n, k, m, seed=90 + tp, dtype="e4m3", n_row_chunks=chunks)
    groups = tp if op == "rs" else chunks
    run = KsplitRun(wl)
    try:
        for reduce in (0, 1, 2):
            t.tpo_set_opt(run.ctx, "reduce", reduce)
            first = None
            for sched, gemm_ctas in ((1, 0), (2, 2), (2, 4), (2, 0), (2, 2)):
                t.tpo_set_opt(run.ctx, "sched", sched)
                t.tpo_set_opt(run.ctx, "gemm_ctas", gemm_ctas)
                if op == "rs":
                    run.rs()
                    y = torch.cat(run.yb, 0)
                else:
                    run.ar(chunks)
                    y = run.y
                assert t.tpo_get_opt(run.ctx, "last_sched") == (2 if sched == 2 else 1)
                bits = host_bits(y)
                if first is None:
                    if reduce < 2:
                        ref = oracle.ksplit(wl.x, wl.w, sx=wl.scale_inv_x, sw=wl.scale_inv_w)
                        assert_close(host_f64(y), ref, dtype)
                    first = bits
                assert np.array_equal(bits, first), (reduce, sched, gemm_ctas)
                ptr, target = t.tpo_done_counters(run.ctx)
                torch.cuda.synchronize()

                class _Arr:
                    __cuda_array_interface__ = {"shape": (groups,), "typestr": "<u4", "data": (ptr, False),
                                                "version": 3}
                cnt = torch.as_tensor(_Arr(), device="cuda").cpu().numpy()
                assert np.all(cnt == target), (cnt, target, sched)
    finally:
        run.close()


def test_automatic_choice_follows_the_round_count():
    """Launches of at least 8 rounds take dynamic tiles; fewer keep the round robin."""
    wl = synth.make_ksplit("rs", 2, 2048, 256, 2048, seed=95, dist="normal", sigma=0.25)
    run = KsplitRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "gemm_ctas", 0)
        run.rs()   # 8 x 8 pair tiles over 76 pairs: one round
        assert t.tpo_get_opt(run.ctx, "last_sched") == 1
        t.tpo_set_opt(run.ctx, "gemm_ctas", 4)
        run.rs()   # 64 tiles on 2 pairs: 32 rounds
        assert t.tpo_get_opt(run.ctx, "last_sched") == 2
        t.tpo_set_opt(run.ctx, "sched", 1)
        run.rs()
        assert t.tpo_get_opt(run.ctx, "last_sched") == 1
    finally:
        run.close()


def test_timeout_with_dynamic_tiles_leaves_the_context_usable():
    wl = synth.make_ag(4, 2048, 256, 1024, seed=97, dist="normal", sigma=0.25)
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0])
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "sched", 2)
        t.tpo_set_opt(run.ctx, "gemm_ctas", 4)
        t.tpo_set_opt(run.ctx, "wait_timeout_ms", 100)
        t.tpo_set_opt(run.ctx, "debug_skip_chunk", 2)   # slot 2 is never published: its tiles time out
        t.tpo_ag_gemm(run.ctx, run.xs, run.w, run.y)
        assert t.tpo_sync_status(run.ctx) == 4                # TPO_ERR_TIMEOUT
        t.tpo_set_opt(run.ctx, "debug_skip_chunk", -1)
        t.tpo_set_opt(run.ctx, "wait_timeout_ms", 2000)
        for _ in range(2):
            run.y.fill_(float("nan"))
            run.run()
            assert_close(host_f64(run.y), ref)
    finally:
        run.close()
