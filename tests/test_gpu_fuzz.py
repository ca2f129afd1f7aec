"""Seeded random shapes and options on the GPU, each call against the oracle.

Every case draws an operation (AG, RS, AR), a dtype, sizes that are ragged in
rows, columns and K where the ABI allows it, and launch options (observer
rank, schedule mode, CTA-pair or single-SM tiles, GEMM grid, producer count,
tail split, epilogue-reduction mode, row chunks, column plan, launch kind).  Outputs sit between
sentinel guards; every launch of a case is compared with the oracle, and a
second launch of the same case must give the same bits.
"""

import numpy as np
import pytest
import torch

import oracle
from tensor_comm_gemm_gb300 import synth
from tensor_comm_gemm_gb300 import tpoverlap as t
from gpu_util import AgRun, KsplitRun, assert_close, check_wire, host_bits, host_f64, wire_expectation

pytestmark = pytest.mark.gpu

GUARD = 64
SENTINEL = 0x7F7F
CASES = 48


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()


class Guarded:
    def __init__(self, rows, cols):
        self.buf = torch.empty(rows * cols + 2 * GUARD, dtype=torch.bfloat16, device="cuda")
        self.buf.view(torch.int16).fill_(SENTINEL)
        self.y = self.buf[GUARD:GUARD + rows * cols].view(rows, cols)

    def poison(self):
        self.y.fill_(float("nan"))

    def intact(self):
        bits = self.buf.view(torch.int16).cpu().numpy().view(np.uint16)
        return bool(np.all(bits[:GUARD] == SENTINEL) and np.all(bits[-GUARD:] == SENTINEL))


def draw(seed):
    """One case: (op, dtype, tp, n, k, m, options)."""
    rng = np.random.default_rng(seed)
    op = ["ag", "ag", "rs", "ar"][rng.integers(4)]
    dtype = "e4m3" if rng.random() < 0.3 else "bf16"
    kq = 16 if dtype == "e4m3" else 8                    # 16-byte rows
    tp = int(rng.choice([1, 2, 3, 4, 5, 8]))
    m = int(8 * rng.integers(1, 81))                      # up to 640 columns, 16-byte rows
    opts = {"gemm_ctas": int(rng.choice([0, 0, 2, 3, 5, 8])), "cta_group": int(rng.choice([0, 0, 1])),
            "col_split": int(rng.choice([0, 0, 0, int(rng.integers(1, 1 << 16))])),
            "pdl": int(rng.choice([1, 1, 0])), "cooperative": int(rng.choice([0, 0, 1]))}
    if op == "ag":
        rows = int(rng.choice([int(rng.integers(1, 300)), 256, 512]))
        n, k = tp * rows, int(kq * rng.integers(1, 48))
        opts["self_rank"] = int(rng.integers(tp))
        opts["mode"] = int(rng.choice([0, 0, 1, 2, 4]))
        opts["producer_sms"] = int(rng.choice([0, 0, 1, 4, 9]))
        opts["tail_split"] = int(rng.choice([0, 0, 1, 2])) if opts["mode"] != 4 else 0
    else:
        kr = int(kq * rng.integers(1, 24))
        k = tp * kr
        opts["reduce"] = int(rng.choice([0, 0, 1, 2]))
        if op == "rs":
            n = tp * int(rng.choice([int(rng.integers(1, 300)), 256]))
        else:
            chunks = int(rng.integers(1, 4))
            n = chunks * tp * int(rng.choice([int(rng.integers(1, 200)), 256]))
            opts["chunks"] = chunks
    # tile claiming (drawn apart so that the draws above stay as they were)
    opts["sched"] = int(np.random.default_rng(seed + 7919).choice([0, 1, 2, 2]))
    return op, dtype, tp, n, k, m, opts


@pytest.mark.parametrize("seed", range(CASES))
def test_random_case_matches_oracle(seed):
    op, dtype, tp, n, k, m, opts = draw(1000 + seed)
    chunks = opts.pop("chunks", 1)
    if op == "ag":
        wl = synth.make_ag(tp, n, k, m, seed=seed, dist="uniform", dtype=dtype)
        ref = oracle.ag(oracle.gather(wl.x), wl.w[0], wl.scale_inv_x, wl.scale_inv_w)
        run = AgRun(wl)
        outs = [Guarded(n, m)]
    else:
        wl = synth.make_ksplit(op, tp, n, k, m, seed=seed, n_row_chunks=chunks, dtype=dtype,
                               sigma=(k ** -0.25) if dtype == "bf16" else 1.0)
        ref = oracle.ksplit(wl.x, wl.w, sx=wl.scale_inv_x, sw=wl.scale_inv_w)
        run = KsplitRun(wl)
        outs = [Guarded(n // tp, m) for _ in range(tp)] if op == "rs" else [Guarded(n, m)]
    try:
        pairs = (n // tp) % 256 == 0 if op in ("ag", "rs") else (n // (chunks * tp)) % 256 == 0
        if opts["cta_group"] == 2 and not pairs:
            opts["cta_group"] = 0
        for key, value in opts.items():
            t.tpo_set_opt(run.ctx, key, value)
        if op == "ag" and opts["mode"] == 2:  # GEMM only reads chunks an earlier call published
            t.tpo_set_opt(run.ctx, "mode", 1)
            run.run(y=outs[0].y)
            t.tpo_set_opt(run.ctx, "mode", 2)
        first = None
        for _ in range(2):
            for o in outs:
                o.poison()
            if op == "ag":
                run.run(y=outs[0].y)
            elif op == "rs":
                t.tpo_gemm_rs(run.ctx, run.xs, run.ws, [o.y for o in outs])
                assert t.tpo_sync_status(run.ctx) == 0, t.tpo_last_error()
            else:
                t.tpo_gemm_ar(run.ctx, run.xs, run.ws, outs[0].y, chunks)
                assert t.tpo_sync_status(run.ctx) == 0, t.tpo_last_error()
            assert all(o.intact() for o in outs), ("store outside the output", op, dtype, tp, n, k, m, opts)
            got = np.concatenate([host_f64(o.y) for o in outs], 0)
            bits = np.concatenate([host_bits(o.y) for o in outs], 0)
            if first is None:
                if opts.get("reduce", 0) == 2:   # bf16 ring: the oracle's ring sum
                    wire_ref, risky, bound = wire_expectation(wl, op, chunks)
                    check_wire(got, wire_ref, risky, bound, dtype)
                else:
                    assert_close(got, ref, dtype)
                first = bits
            assert np.array_equal(bits, first), ("second launch differs", op, dtype, tp, n, k, m, opts)
    finally:
        run.close()
