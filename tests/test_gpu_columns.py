"""Column plans on the GPU (option col_split): groups whose 32-column strips are
split into more, narrower tiles (down to one strip) give the same bits as
whole 256-column tiles in every mode, stay within the oracle's bar and keep
the done counters' common target.  The automatic plan (the default) is the
one the host model restated in test_schedule picks."""

import numpy as np
import pytest
import torch

import oracle
from tensor_comm_gemm_gb300 import synth
from tensor_comm_gemm_gb300 import tpoverlap as t
from gpu_util import AgRun, KsplitRun, assert_close, host_bits, host_f64
from test_schedule import auto_columns, auto_groups, choose_cg, packed, plan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()


def explicit_plans(groups):
    """col_split values: the fewest tiles (-1), the automatic plan (0, the
    default) and packed extras (4 bits per group) from one extra tile to 15."""
    return [-1, 0, packed([1] * groups), packed([(3 * g + 1) % 16 for g in range(groups)]), packed([15] * groups)]


def expected_auto_plan(op, tp, n, k, m, chunks=1):
    """last_col_plan of the automatic plan, from the host model's restatement."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cg = choose_cg(op, tp, n, chunks)
    pl = plan(op, tp, n, k, m, 2, chunks, cg)
    auto_columns(pl, m, auto_groups(op, cg, num_sms=sms, max_pairs=sms // 2))
    return packed([c - pl["base_cols"] for c in pl["group_cols"]])


@pytest.mark.parametrize("tp,n,k,m", [(4, 2048, 512, 1024), (3, 768, 192, 264), (2, 512, 256, 520),
                                      (1, 256, 64, 2048)])
def test_ag_column_plans_bit_identical(tp, n, k, m):
    wl = synth.make_ag(tp, n, k, m, seed=50 + tp, dist="normal", sigma=k ** -0.25)
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0])
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "tail_split", 0)
        first = None
        for cs in explicit_plans(tp):
            t.tpo_set_opt(run.ctx, "col_split", cs)
            for mode in (0, 2):
                t.tpo_set_opt(run.ctx, "mode", mode)
                run.y.fill_(float("nan"))
                run.run()
                bits = host_bits(run.y)
                if first is None:
                    assert_close(host_f64(run.y), ref)
                    first = bits
                assert np.array_equal(bits, first), (cs, mode, t.tpo_get_opt(run.ctx, "last_col_plan"))
                if cs > 0:
                    assert t.tpo_get_opt(run.ctx, "last_col_plan") != 0
                if cs < 0:
                    assert t.tpo_get_opt(run.ctx, "last_col_plan") == 0
                if cs == 0:
                    assert t.tpo_get_opt(run.ctx, "last_col_plan") == expected_auto_plan("ag", tp, n, k, m)
    finally:
        run.close()


def test_ag_e4m3_column_plans_bit_identical():
    wl = synth.make_ag(4, 2048, 384, 768, seed=57, dtype="e4m3")
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0], wl.scale_inv_x, wl.scale_inv_w)
    run = AgRun(wl)
    try:
        first = None
        for cs in explicit_plans(4):
            t.tpo_set_opt(run.ctx, "col_split", cs)
            run.run()
            bits = host_bits(run.y)
            if first is None:
                assert_close(host_f64(run.y), ref, "e4m3")
                first = bits
            assert np.array_equal(bits, first), cs
    finally:
        run.close()


@pytest.mark.parametrize("op,tp,n,k,m,chunks", [("rs", 4, 1024, 1280, 768, 1), ("ar", 2, 2048, 512, 520, 2),
                                                ("ar", 3, 2304, 384, 1024, 3)])
def test_ksplit_column_plans_bit_identical_with_done_counters(op, tp, n, k, m, chunks):
    wl = synth.make_ksplit(op, tp, n, k, m, seed=60 + tp, dist="normal", sigma=k ** -0.25, n_row_chunks=chunks)
    ref = oracle.ksplit(wl.x, wl.w)
    groups = tp if op == "rs" else chunks
    run = KsplitRun(wl)
    try:
        for mode in (0, 1, 2):
            t.tpo_set_opt(run.ctx, "reduce", mode)
            first = None
            for cs in explicit_plans(groups):
                t.tpo_set_opt(run.ctx, "col_split", cs)
                if op == "rs":
                    run.rs()
                    y = torch.cat(run.yb, 0)
                else:
                    run.ar(chunks)
                    y = run.y
                bits = host_bits(y)
                if first is None:
                    if mode < 2:
                        assert_close(host_f64(y), ref)
                    first = bits
                assert np.array_equal(bits, first), (mode, cs)
                ptr, target = t.tpo_done_counters(run.ctx)
                torch.cuda.synchronize()

                class _Arr:
                    __cuda_array_interface__ = {"shape": (groups,), "typestr": "<u4", "data": (ptr, False),
                                                "version": 3}
                cnt = torch.as_tensor(_Arr(), device="cuda").cpu().numpy()
                assert np.all(cnt == target), (cnt, target, cs)
    finally:
        run.close()
