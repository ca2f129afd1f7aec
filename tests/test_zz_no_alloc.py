"""tpo_ag_gemm_noalloc: the AG+GEMM entry point that allocates no device memory.

Callers that cannot call cudaMalloc when they run the layer use it: a serving
process that reserved all device memory for its own pool at start-up, or a
runtime whose allocator forbids raw device allocations after initialisation so
that its memory use stays fixed.  They cannot hold a context (creating one
allocates the staging buffer and the counters), so this entry point keeps its
scratch in a static device array of the library instead.

The checks compare it with the context entry point, tpo_ag_gemm, over
consecutive calls: every call reuses the same array, so counters or staging
rows left behind by the previous call would show up as a wrong result or a
timeout.  The file name sorts last, so a run that stops at the first failure
has run every other test before this one; it also passes on its own in a fresh
process.
"""

import numpy as np
import pytest
import torch

import oracle
from tensor_comm_gemm_gb300 import synth
from tensor_comm_gemm_gb300 import tpoverlap as t
from gpu_util import AgRun, SAMPLE_TILE, SAMPLE_TILES, assert_close, gather_tiles, host_bits, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()


def _noalloc(run: AgRun, y):
    wl = run.wl
    dt = t.TPO_FP8_E4M3 if run.fp8 else t.TPO_BF16
    t.tpo_ag_gemm_noalloc(wl.tp, wl.n, wl.k, wl.m, dt, run.xs, run.w, y, run.sx, run.sw)


@pytest.mark.parametrize("cases", [
    [(4, 1024, 512, 768, "bf16", 61), (2, 512, 256, 512, "bf16", 62)],   # different shapes back to back
    [(4, 4096, 4096, 4096, "bf16", 1), (4, 4096, 4096, 4096, "bf16", 1)],  # the 32 MiB limit, twice
    [(8, 2048, 384, 768, "e4m3", 63), (3, 768, 128, 256, "e4m3", 64)],
    [(4, 2048, 1024, 20480, "bf16", 65)],   # 640 pair tiles: at least 8 rounds, dynamic tiles in both entry points
])
def test_noalloc_matches_context_entry_point_on_consecutive_calls(cases):
    for tp, n, k, m, dtype, seed in cases:
        if dtype == "bf16":
            wl = synth.make_ag(tp, n, k, m, seed=seed, dist="normal", sigma=k ** -0.25)
        else:
            wl = synth.make_ag(tp, n, k, m, seed=seed, dtype="e4m3")
        run = AgRun(wl)
        try:
            t.tpo_set_opt(run.ctx, "tail_split", 0)     # the no-alloc entry point computes whole tiles
            run.run()                                   # existing entry point, through a context
            if m >= 16384:                              # many rounds: the context took dynamic tiles
                assert t.tpo_get_opt(run.ctx, "last_sched") == 2
            ref = host_f64(run.y)
            y = torch.full_like(run.y, float("nan"))
            _noalloc(run, y)                            # returns once the GPU work is done
            assert_close(host_f64(y), ref, wl.dtype)    # the tolerance of every parity test
            assert np.array_equal(host_bits(y), host_bits(run.y))  # same kernel, same tile arithmetic
            if n * m > 1 << 22:   # large outputs: sampled tiles against the oracle itself as well
                tiles = synth.sample_tiles(n, m, SAMPLE_TILE, SAMPLE_TILES, seed=1000 + seed)
                want = oracle.ag(oracle.gather(wl.x), wl.w[0], wl.scale_inv_x, wl.scale_inv_w, tiles=tiles)
                assert_close(gather_tiles(host_f64(y), tiles), want, wl.dtype)
            t.tpo_set_opt(run.ctx, "tail_split", 2)     # the split schedule meets the same bar
            run.run()
            assert_close(host_f64(run.y), host_f64(y), wl.dtype)
        finally:
            run.close()


def test_noalloc_rejects_sizes_beyond_the_static_array():
    tp, n, k, m = 2, 4096, 4160, 256                    # n*k*2 bytes just over 32 MiB
    x = [torch.zeros((n // tp, k), dtype=torch.bfloat16, device="cuda") for _ in range(tp)]
    w = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((n, m), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(t.TpoError) as e:
        t.tpo_ag_gemm_noalloc(tp, n, k, m, t.TPO_BF16, x, w, y)
    assert e.value.status == 1
    assert str(t.TPO_NOALLOC_MAX_STAGING_BYTES) in str(e.value)
