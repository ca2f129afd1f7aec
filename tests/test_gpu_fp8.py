"""FP8 (e4m3) AG+GEMM on the GPU through the C ABI."""

import numpy as np
import pytest

import oracle
from tensor_comm_gemm_gb300 import synth
from tensor_comm_gemm_gb300 import tpoverlap as t
from gpu_util import AgRun, assert_close, gather_tiles, host_bits, host_f64, SAMPLE_TILES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("tp,n,k,m", [(2, 256, 256, 512), (8, 2048, 384, 768), (3, 768, 128, 256),
                                     (4, 1024, 512, 512)])
def test_fp8_ag_full_parity(tp, n, k, m):
    wl = synth.make_ag(tp, n, k, m, seed=50 + tp, dtype="e4m3")
    ref = oracle.ag(oracle.gather(wl.x), wl.w[0], wl.scale_inv_x, wl.scale_inv_w)
    run = AgRun(wl)
    try:
        run.run()
        assert_close(host_f64(run.y), ref, "e4m3")
        bits = host_bits(run.y)
        t.tpo_set_opt(run.ctx, "mode", 1)
        run.y.fill_(0)
        run.run()
        assert np.array_equal(host_bits(run.y), bits)
    finally:
        run.close()


def test_fp8_staging_is_exact_gather():
    from gpu_util import staging_view
    wl = synth.make_ag(4, 1024, 256, 256, seed=3, dtype="e4m3")
    run = AgRun(wl)
    try:
        run.run()
        got = staging_view(run.ctx, wl.n * wl.k).cpu().numpy().reshape(wl.n, wl.k)
        assert np.array_equal(got, oracle.gather(wl.x))
    finally:
        run.close()


@pytest.mark.slow
def test_workload_fp8_ag_tp8_sampled_parity():
    wl = synth.workload(4)
    run = AgRun(wl)
    try:
        run.run()
        tiles = synth.sample_tiles(wl.n, wl.m, 16, SAMPLE_TILES, seed=1000 + wl.seed)
        ref = oracle.ag(oracle.gather(wl.x), wl.w[0], wl.scale_inv_x, wl.scale_inv_w, tiles=tiles)
        assert_close(gather_tiles(host_f64(run.y), tiles), ref, "e4m3")
    finally:
        run.close()
