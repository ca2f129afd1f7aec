"""AG+GEMM on the GPU through the C ABI, against the CPU oracle."""

import numpy as np
import pytest
import torch

import oracle
from tensor_comm_gemm_gb300 import synth
from tensor_comm_gemm_gb300 import tpoverlap as t
from gpu_util import AgRun, assert_close, gather_tiles, host_bits, host_f64, staging_view, SAMPLE_TILES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()


def ref_ag(wl):
    return oracle.ag(oracle.gather(wl.x), wl.w[0], wl.scale_inv_x, wl.scale_inv_w)


# (tp, n, k, m): several tiles per slot, ragged K (not a multiple of 256), tp=1 and tp=16
SHAPES = [(2, 256, 256, 256), (3, 768, 192, 768), (1, 128, 64, 256), (5, 1280, 320, 512), (16, 2048, 64, 256),
          (4, 1024, 1088, 1024), (16, 4096, 128, 256), (2, 512, 64, 2048)]


@pytest.mark.parametrize("tp,n,k,m", SHAPES)
def test_ag_full_parity_every_observer(tp, n, k, m):
    wl = synth.make_ag(tp, n, k, m, seed=10 + tp, dist="uniform")
    ref = ref_ag(wl)
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "tail_split", 0)   # whole tiles: every mode and grid gives the same bits
        first = None
        for self_rank in sorted({0, tp - 1, tp // 2}):
            t.tpo_set_opt(run.ctx, "self_rank", self_rank)
            for mode in (0, 1, 4):      # overlapped, sequential, split
                t.tpo_set_opt(run.ctx, "mode", mode)
                run.y.fill_(float("nan"))
                run.run()
                if mode == 0:
                    assert_close(host_f64(run.y), ref)
                bits = host_bits(run.y)
                if first is None:
                    first = bits
                assert np.array_equal(bits, first), ("result depends on the observer rank or mode", self_rank, mode)
    finally:
        run.close()


def test_workload_ag_tp2_full_parity():
    wl = synth.workload(0)
    run = AgRun(wl)
    try:
        run.run()
        assert_close(host_f64(run.y), ref_ag(wl))
    finally:
        run.close()


@pytest.mark.parametrize("tp,n,k,m", [(2, 256, 256, 256), (4, 1024, 192, 512)])
def test_staging_bit_exact_after_every_ring_step(tp, n, k, m):
    wl = synth.make_ag(tp, n, k, m, seed=3, dist="uniform")
    run = AgRun(wl)
    nbytes = n * k * 2
    try:
        view = staging_view(run.ctx, nbytes)
        t.tpo_set_opt(run.ctx, "mode", 3)          # producer only
        for self_rank in range(tp):
            t.tpo_set_opt(run.ctx, "self_rank", self_rank)
            for step in range(tp):
                view.fill_(0xAB)
                torch.cuda.synchronize()
                t.tpo_set_opt(run.ctx, "debug_last_step", step)
                run.run()
                got = view.cpu().numpy().view(np.uint16).reshape(n, k)
                want = oracle.staging_after_step(wl.x, self_rank, step, 0xAB)
                assert np.array_equal(got, want), (self_rank, step)
        # a full overlapped call leaves exactly the rank-order gather
        t.tpo_set_opt(run.ctx, "mode", 0)
        t.tpo_set_opt(run.ctx, "debug_last_step", -1)
        view.fill_(0xAB)
        run.run()
        got = view.cpu().numpy().view(np.uint16).reshape(n, k)
        assert np.array_equal(got, oracle.gather(wl.x))
    finally:
        run.close()


@pytest.mark.parametrize("tp,n,k,m", [(2, 256, 256, 256), (4, 2048, 512, 768)])
def test_overlapped_bit_identical_to_sequential(tp, n, k, m):
    wl = synth.make_ag(tp, n, k, m, seed=4, dist="normal", sigma=k ** -0.25)
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "tail_split", 0)   # whole tiles: the same bits for every producer count
        outs = {}
        for mode, psms in [(0, 8), (1, 8), (2, 8), (0, 1), (0, 20), (4, 8), (4, 0), (0, 0)]:
            t.tpo_set_opt(run.ctx, "mode", mode)
            t.tpo_set_opt(run.ctx, "producer_sms", psms)
            run.y.fill_(float("nan"))
            run.run()
            outs[(mode, psms)] = host_bits(run.y)
            if mode == 4:   # split mode leaves the full gather in the staging buffer too
                got = staging_view(run.ctx, wl.n * wl.k * 2).cpu().numpy().view(np.uint16).reshape(wl.n, wl.k)
                assert np.array_equal(got, oracle.gather(wl.x))
        base = outs[(1, 8)]
        for key, v in outs.items():
            assert np.array_equal(v, base), key
        assert_close(synth.bf16_bits_to_f32(base).astype(np.float64), ref_ag(wl))
    finally:
        run.close()


def test_producer_delay_keeps_result_identical():
    """A slow producer (spin before every publish) widens the window in which a
    GEMM load could run ahead of its chunk; the result must not change."""
    wl = synth.make_ag(4, 1024, 256, 512, seed=5, dist="uniform")
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "mode", 1)
        run.run()
        base = host_bits(run.y)
        staging = staging_view(run.ctx, wl.n * wl.k * 2)
        t.tpo_set_opt(run.ctx, "mode", 0)
        t.tpo_set_opt(run.ctx, "debug_delay_ns", 200000)
        for _ in range(3):
            staging.fill_(0xFF)          # NaN pattern: a premature read shows up in Y
            run.y.fill_(0)
            run.run()
            assert np.array_equal(host_bits(run.y), base)
    finally:
        run.close()


def test_identity_and_one_hot_weights_are_exact():
    tp, n, k = 2, 512, 256
    wl = synth.make_ag(tp, n, k, k, seed=6, dist="normal")
    g = oracle.gather(wl.x)
    rng = np.random.default_rng(0)
    perm = rng.permutation(k)
    onehot = np.zeros((2 * k, k), dtype=np.float32)       # m = 2k columns, two one-hots each
    onehot[np.arange(k), perm] = 1.0
    onehot[k + np.arange(k), np.arange(k)] = 1.0
    for w, want in [(np.eye(k, dtype=np.float32), g), (onehot, np.concatenate([g[:, perm], g], 1))]:
        wl2 = synth.Workload("onehot", "ag", "bf16", tp, n, k, w.shape[0], wl.x, [synth.f32_to_bf16_bits(w)])
        run = AgRun(wl2)
        try:
            run.run()
            assert np.array_equal(host_bits(run.y), want)
        finally:
            run.close()


def test_trace_orders_publish_before_acquire():
    wl = synth.make_ag(4, 4096, 1024, 1024, seed=8, dist="uniform")
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "trace", 1)
        t.tpo_set_opt(run.ctx, "self_rank", 1)
        run.run()
        tr = t.tpo_read_trace(run.ctx)
        order = oracle.ring_order(4, 1)
        pubs = [tr[t.TPO_TRACE_PUBLISH + s] for s in order]
        assert all(p > 0 for p in pubs)
        assert pubs[1] <= pubs[2] <= pubs[3]            # ring steps published in arrival order
        for s in order[1:]:                              # a gated slot is read only after its publish
            acq = tr[t.TPO_TRACE_ACQUIRE + s]
            if acq != 2 ** 64 - 1:
                assert acq >= tr[t.TPO_TRACE_PUBLISH + s] - 2000  # timer samples of different SMs
        assert tr[t.TPO_TRACE_START] <= tr[t.TPO_TRACE_END]
    finally:
        run.close()


def test_skipped_chunk_times_out_and_context_recovers():
    wl = synth.make_ag(4, 1024, 256, 512, seed=9, dist="uniform")
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "wait_timeout_ms", 50)
        t.tpo_set_opt(run.ctx, "debug_skip_chunk", 2)     # never published: the GEMM must give up
        t.tpo_ag_gemm(run.ctx, run.xs, run.w, run.y)
        assert t.tpo_sync_status(run.ctx) == 4
        code, site, _, extra = t.tpo_last_device_error(run.ctx)
        assert code == 1 and site in (1, 2, 3, 4, 5, 8)
        t.tpo_set_opt(run.ctx, "debug_skip_chunk", -1)
        t.tpo_set_opt(run.ctx, "wait_timeout_ms", 2000)
        run.run()
        assert_close(host_f64(run.y), ref_ag(wl))
    finally:
        run.close()


def test_call_argument_errors():
    wl = synth.make_ag(2, 256, 256, 256, seed=1, dist="uniform")
    run = AgRun(wl)
    try:
        base = run.y.view(torch.uint8).reshape(-1)
        with pytest.raises(t.TpoError) as e:
            t.tpo_ag_gemm(run.ctx, run.xs, run.w, base[8:].data_ptr())
        assert e.value.status == 1
        with pytest.raises(t.TpoError) as e:
            t.tpo_ag_gemm(run.ctx, [run.xs[0], 0], run.w, run.y)
        assert e.value.status == 1
        sx = torch.ones(1, device="cuda")
        with pytest.raises(t.TpoError) as e:
            t.tpo_ag_gemm(run.ctx, run.xs, run.w, run.y, sx, sx)
        assert e.value.status == 1
        with pytest.raises(t.TpoError):
            t.tpo_set_opt(run.ctx, "self_rank", 2)
        with pytest.raises(t.TpoError):
            t.tpo_set_opt(run.ctx, "no_such_option", 1)
        for bad in (0, 3):   # one or two K blocks per pipeline stage
            with pytest.raises(t.TpoError):
                t.tpo_set_opt(run.ctx, "stage_kblocks", bad)
        assert t.tpo_get_opt(run.ctx, "stage_kblocks") == 1
        with pytest.raises(t.TpoError) as e:
            t.tpo_gemm_ar(run.ctx, [x.data_ptr() for x in run.xs], [run.w.data_ptr()] * 2, run.y,
                          3)   # n % (3*tp) != 0: unequal ring-order parts
        assert e.value.status == 2
    finally:
        run.close()


@pytest.mark.slow
def test_workload_ag_tp4_4096_sampled_parity():
    wl = synth.workload(1)
    run = AgRun(wl)
    try:
        run.run()
        y = host_f64(run.y)
        bits = host_bits(run.y)
        tiles = synth.sample_tiles(wl.n, wl.m, 16, SAMPLE_TILES, seed=1000 + wl.seed)
        ref = oracle.ag(oracle.gather(wl.x), wl.w[0], tiles=tiles)
        assert_close(gather_tiles(y, tiles), ref)
        t.tpo_set_opt(run.ctx, "mode", 1)
        run.y.fill_(0)
        run.run()
        assert np.array_equal(host_bits(run.y), bits)
    finally:
        run.close()


@pytest.mark.parametrize("tp,n,k,m", [(4, 2048, 512, 768), (3, 768, 192, 768), (2, 1024, 4096, 512)])
def test_pair_and_single_sm_variants_agree(tp, n, k, m):
    """The 2-SM (CTA pair) MMA and the single-SM MMA compute every output
    element with the same K order; so do the pairs' one- and two-block
    pipeline stages.  All meet the oracle bar and agree bitwise."""
    wl = synth.make_ag(tp, n, k, m, seed=70 + tp, dist="normal", sigma=k ** -0.25)
    ref = ref_ag(wl)
    run = AgRun(wl)
    try:
        bits = {}
        t.tpo_set_opt(run.ctx, "tail_split", 0)   # whole tiles, so that both variants share the K order
        for cg in (1, 2):
            t.tpo_set_opt(run.ctx, "cta_group", cg)
            for kb in ((1,) if cg == 1 else (1, 2)):
                t.tpo_set_opt(run.ctx, "stage_kblocks", kb)
                for mode in (0, 1):
                    t.tpo_set_opt(run.ctx, "mode", mode)
                    run.y.fill_(float("nan"))
                    run.run()
                    assert_close(host_f64(run.y), ref)
                    bits[(cg, kb, mode)] = host_bits(run.y)
                    even = (k // 64) % 2 == 0   # 64 bf16 elements per K block
                    assert t.tpo_get_opt(run.ctx, "last_stage_kblocks") == (2 if kb == 2 and even else 1)
        for key, b in bits.items():
            assert np.array_equal(b, bits[(1, 1, 0)]), key
    finally:
        run.close()


def test_binding_rejects_mismatched_tensors():
    """The binding refuses tensors whose layout the library would misread."""
    wl = synth.make_ag(2, 256, 256, 256, seed=1, dist="uniform")
    run = AgRun(wl)
    try:
        cases = [
            ([run.xs[0]], run.w, run.y),                                # too few chunks
            ([run.xs[0].t(), run.xs[1]], run.w, run.y),                 # transposed (strided) chunk
            (run.xs, run.w.float(), run.y),                             # 4-byte weight elements
            (run.xs, run.w[:128], run.y),                               # short weight
            (run.xs, run.w, run.y.cpu()),                               # host output
        ]
        for xs, w, y in cases:
            with pytest.raises(t.TpoError) as e:
                t.tpo_ag_gemm(run.ctx, xs, w, y)
            assert e.value.status == t.TPO_ERR_INVALID_ARG
        assert t.tpo_get_opt(run.ctx, "tp") == 2 and t.tpo_get_opt(run.ctx, "m") == 256
        run.run()                                                       # the context is unharmed
        assert_close(host_f64(run.y), ref_ag(wl))
    finally:
        run.close()


def test_pair_variant_rejected_for_128_row_slots():
    wl = synth.make_ag(2, 256, 256, 256, seed=1, dist="uniform")
    run = AgRun(wl)
    try:
        t.tpo_set_opt(run.ctx, "cta_group", 2)
        with pytest.raises(t.TpoError) as e:
            t.tpo_ag_gemm(run.ctx, run.xs, run.w, run.y)
        assert e.value.status == 2
        t.tpo_set_opt(run.ctx, "cta_group", 0)          # auto picks the single-SM variant
        run.run()
        assert_close(host_f64(run.y), ref_ag(wl))
    finally:
        run.close()


@pytest.mark.parametrize("tp,n,k,m,dtype", [(4, 4096, 4096, 4096, "bf16"), (8, 16384, 8192, 28672, "e4m3")])
def test_default_producer_count_follows_the_schedule_model(tp, n, k, m, dtype):
    """The library's default producer count for the C2 and C5 shapes is the
    one the host schedule model (restated in test_schedule) picks."""
    from test_schedule import producer_choice
    fp8 = dtype == "e4m3"
    el = torch.uint8 if fp8 else torch.bfloat16
    xs = [torch.zeros((n // tp, k), dtype=el, device="cuda") for _ in range(tp)]
    w = torch.zeros((m, k), dtype=el, device="cuda")
    y = torch.empty((n, m), dtype=torch.bfloat16, device="cuda")
    sx = torch.ones(1, device="cuda") if fp8 else None
    ctx = t.tpo_ctx_create(tp, n, k, m, t.TPO_FP8_E4M3 if fp8 else t.TPO_BF16)
    try:
        t.tpo_ag_gemm(ctx, xs, w, y, sx, sx)
        assert t.tpo_sync_status(ctx) == 0, t.tpo_last_error()
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        P = producer_choice(tp, n // tp, k, m, elem=1 if fp8 else 2, cg=2, num_sms=sms)
        assert t.tpo_get_opt(ctx, "last_producer_ctas") == P
        assert t.tpo_get_opt(ctx, "last_col_plan") == 0        # whole tiles by default
        assert not torch.isnan(y).any()
    finally:
        t.tpo_ctx_destroy(ctx)


def test_two_contexts_on_two_streams():
    """An AG context and a GEMM+RS context enqueued on two side streams at the
    same time: both results meet the oracle bar (the overlapped AG launch is
    cooperative, so its producer and GEMM CTAs are placed together whatever
    the other stream runs)."""
    from gpu_util import KsplitRun
    wl_ag = synth.make_ag(4, 2048, 512, 768, seed=21, dist="uniform")
    wl_rs = synth.make_ksplit("rs", 4, 2048, 1024, 512, seed=22, sigma=1024 ** -0.25)
    ref_a = ref_ag(wl_ag)
    ref_r = oracle.ksplit(wl_rs.x, wl_rs.w)
    ag, rs = AgRun(wl_ag), KsplitRun(wl_rs)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    try:
        torch.cuda.synchronize()
        for _ in range(3):
            ag.y.fill_(float("nan"))
            for y in rs.yb:
                y.fill_(float("nan"))
            torch.cuda.synchronize()
            t.tpo_ag_gemm(ag.ctx, ag.xs, ag.w, ag.y, stream=s1)
            t.tpo_gemm_rs(rs.ctx, rs.xs, rs.ws, rs.yb, stream=s2)
            t.tpo_ag_gemm(ag.ctx, ag.xs, ag.w, ag.y, stream=s1)
            assert t.tpo_sync_status(ag.ctx) == 0 and t.tpo_sync_status(rs.ctx) == 0
            torch.cuda.synchronize()
            assert_close(host_f64(ag.y), ref_a)
            assert_close(np.concatenate([host_f64(y) for y in rs.yb], 0), ref_r)
    finally:
        ag.close()
        rs.close()


def test_chained_calls_respect_the_launch_before():
    """Back-to-back launches on one stream (with and without programmatic
    dependent launch): the second AG call gathers the first call's output rows, with a
    torch kernel between them, and no synchronisation until the end; its
    result must be the oracle's on the first result."""
    tp, n, k, m = 2, 512, 256, 256
    wl1 = synth.make_ag(tp, n, k, m, seed=71, dist="normal", sigma=k ** -0.25)
    r1 = AgRun(wl1)
    w2_host = synth.make_ag(tp, n, m, m, seed=72, dist="normal", sigma=m ** -0.25).w[0]
    w2 = torch.from_numpy(w2_host.view(np.int16)).view(torch.bfloat16).cuda()
    y2 = torch.empty((n, m), dtype=torch.bfloat16, device="cuda")
    ctx2 = t.tpo_ctx_create(tp, n, m, m, t.TPO_BF16)
    try:
      for pdl in (1, 0):
        t.tpo_set_opt(r1.ctx, "pdl", pdl)
        t.tpo_set_opt(ctx2, "pdl", pdl)
        for rep in range(3):
            r1.y.fill_(float("nan"))
            y2.fill_(float("nan"))
            torch.cuda.synchronize()
            r1.run(sync=False)
            y1 = r1.y * 1.0                        # a torch kernel in between
            t.tpo_ag_gemm(ctx2, [y1[: n // tp], y1[n // tp:]], w2, y2)
            assert t.tpo_sync_status(ctx2) == 0 and t.tpo_sync_status(r1.ctx) == 0
            y1_bits = host_bits(y1)
            assert_close(host_f64(y1), ref_ag(wl1))
            ref2 = oracle.ag(oracle.gather([y1_bits[: n // tp], y1_bits[n // tp:]]), w2_host)
            assert_close(host_f64(y2), ref2)
    finally:
        t.tpo_ctx_destroy(ctx2)
        r1.close()
