"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself (hand-worked golden values, closed forms, library routines,
brute-force simulation), so that a dropped term, a wrong sign, a wrong index
or a transposed operand fails at least one of them."""

import numpy as np
import pytest
import torch

import oracle
from tensor_comm_gemm_gb300 import synth
from conftest import golden_lines


def bf16(a):
    """bf16 bit patterns of small integers (exact in bf16)."""
    return synth.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


# ---------------------------------------------------------------- ring order

def test_ring_order_golden():
    for ln in golden_lines("ring_order.txt"):
        head, tail = ln.split(":")
        tp, me = map(int, head.split())
        assert oracle.ring_order(tp, me) == list(map(int, tail.split())), ln


def _simulate_ring(tp):
    """Message-passing simulation: at step 0 each rank holds its own chunk; at
    every later step each rank sends the chunk it got last to rank+1 and keeps
    what rank-1 sends it."""
    held = [[r] for r in range(tp)]
    for _ in range(1, tp):
        last = [h[-1] for h in held]
        for r in range(tp):
            held[r].append(last[(r - 1) % tp])
    return held


@pytest.mark.parametrize("tp", [1, 2, 3, 4, 5, 8, 16])
def test_ring_order_matches_simulation(tp):
    sim = _simulate_ring(tp)
    for me in range(tp):
        order = oracle.ring_order(tp, me)
        assert order == sim[me]
        assert sorted(order) == list(range(tp))


# ---------------------------------------------------------------- gather

def _read_blocks(name):
    blocks, cur = {}, None
    for ln in golden_lines(name):
        if ln.startswith("rank") or ln == "gathered":
            cur = ln
            blocks[cur] = []
        else:
            blocks[cur].append([int(v) for v in ln.split()])
    return {k: np.array(v, dtype=np.int16) for k, v in blocks.items()}


def test_gather_golden():
    b = _read_blocks("gather_tp2.txt")
    got = oracle.gather([b["rank 0"], b["rank 1"]])
    assert np.array_equal(got, b["gathered"])


@pytest.mark.parametrize("tp", [2, 3, 4])
def test_staging_after_step_prefix(tp):
    rows, cols = 3, 5
    xs = [np.full((rows, cols), 10 + r, dtype=np.uint16) for r in range(tp)]
    full = oracle.gather(xs)
    for me in range(tp):
        order = oracle.ring_order(tp, me)
        assert np.array_equal(oracle.staging_after_step(xs, me, tp - 1, 0xAB), full)
        for step in range(-1, tp):
            s = oracle.staging_after_step(xs, me, step, 0xAB).reshape(tp, rows, cols)
            for slot in range(tp):
                if slot in order[:step + 1]:
                    assert np.all(s[slot] == 10 + slot)
                else:
                    assert np.all(s[slot] == 0xABAB)


# ---------------------------------------------------------------- AG product

def test_ag_golden_tiny():
    d = {}
    for ln in golden_lines("ag_tp2_tiny.txt"):
        key, *vals = ln.split()
        d.setdefault(key, []).append([int(v) for v in vals])
    g = oracle.gather([bf16(d["x0"]), bf16(d["x1"])])
    y = oracle.ag(g, bf16(d["w"]))
    assert np.array_equal(y, np.array(d["y"], dtype=np.float64))


@pytest.mark.parametrize("tp,rows,k,m", [(2, 2, 3, 5), (2, 3, 7, 4), (3, 4, 6, 9), (4, 1, 16, 3)])
def test_ag_brute_force_integers(tp, rows, k, m):
    """Small-integer inputs make every product and sum exact: the oracle must
    equal a library matmul of the gathered rows against W transposed."""
    rng = np.random.default_rng(tp * 100 + k)
    xs_i = [rng.integers(-8, 9, size=(rows, k)) for _ in range(tp)]
    w_i = rng.integers(-8, 9, size=(m, k))
    y = oracle.ag(oracle.gather([bf16(x) for x in xs_i]), bf16(w_i))
    ref = np.concatenate(xs_i, 0).astype(np.float64) @ w_i.astype(np.float64).T
    assert y.shape == (tp * rows, m)
    assert np.array_equal(y, ref)


def test_ag_identity_and_one_hot():
    rng = np.random.default_rng(7)
    tp, rows, k = 2, 4, 8
    xs = [synth.f32_to_bf16_bits(rng.standard_normal((rows, k)).astype(np.float32)) for _ in range(tp)]
    g = oracle.gather(xs)
    gv = synth.bf16_bits_to_f32(g).astype(np.float64)
    eye = bf16(np.eye(k))
    assert np.array_equal(oracle.ag(g, eye), gv)
    perm = rng.permutation(k)[:5]                 # W[c, perm[c]] = 1, m = 5
    onehot = np.zeros((5, k))
    onehot[np.arange(5), perm] = 1
    assert np.array_equal(oracle.ag(g, bf16(onehot)), gv[:, perm])


def test_ag_tiles_match_full():
    rng = np.random.default_rng(3)
    g = bf16(rng.integers(-4, 5, size=(64, 40)))
    w = bf16(rng.integers(-4, 5, size=(48, 40)))
    full = oracle.ag(g, w)
    tiles = synth.sample_tiles(64, 48, 16, 5, seed=11)
    got = oracle.ag(g, w, tiles=tiles)
    for t, (r0, c0) in enumerate(tiles):
        assert np.array_equal(got[t], full[r0:r0 + 16, c0:c0 + 16])


# ---------------------------------------------------------------- K-split sum / RS

def test_rs_golden_tiny():
    d = {}
    for ln in golden_lines("rs_tp2_tiny.txt"):
        key, *vals = ln.split()
        d.setdefault(key, []).append([int(v) for v in vals])
    xs = [bf16(d["x0"]), bf16(d["x1"])]
    ws = [bf16(d["w0"]), bf16(d["w1"])]
    blocks = oracle.rs_blocks(oracle.ksplit(xs, ws), 2)
    assert np.array_equal(blocks[0], np.array(d["block0"], dtype=np.float64))
    assert np.array_equal(blocks[1], np.array(d["block1"], dtype=np.float64))


@pytest.mark.parametrize("tp,n,kr,m", [(2, 4, 3, 2), (3, 6, 5, 7), (4, 8, 2, 3)])
def test_ksplit_is_block_product(tp, n, kr, m):
    """sum_r X_r W_r^T == [X_0|...|X_tp-1] . [W_0|...|W_tp-1]^T exactly on
    integers, and equals a library matmul; RS hands rank b row block b."""
    rng = np.random.default_rng(n * 10 + m)
    xs_i = [rng.integers(-8, 9, size=(n, kr)) for _ in range(tp)]
    ws_i = [rng.integers(-8, 9, size=(m, kr)) for _ in range(tp)]
    y = oracle.ksplit([bf16(x) for x in xs_i], [bf16(w) for w in ws_i])
    cat = oracle.ag(bf16(np.concatenate(xs_i, 1)), bf16(np.concatenate(ws_i, 1)))
    assert np.array_equal(y, cat)
    ref = sum(x.astype(np.float64) @ w.astype(np.float64).T for x, w in zip(xs_i, ws_i))
    assert np.array_equal(y, ref)
    blocks = oracle.rs_blocks(y, tp)
    for b in range(tp):
        assert np.array_equal(blocks[b], ref[b * n // tp:(b + 1) * n // tp])


def test_ksplit_tiles_match_full():
    rng = np.random.default_rng(5)
    xs = [bf16(rng.integers(-3, 4, size=(32, 8))) for _ in range(3)]
    ws = [bf16(rng.integers(-3, 4, size=(48, 8))) for _ in range(3)]
    full = oracle.ksplit(xs, ws)
    tiles = synth.sample_tiles(32, 48, 16, 4, seed=2)
    got = oracle.ksplit(xs, ws, tiles=tiles)
    for t, (r0, c0) in enumerate(tiles):
        assert np.array_equal(got[t], full[r0:r0 + 16, c0:c0 + 16])


# ---------------------------------------------------------------- decoding / FP8

def test_decode_bf16_exhaustive_vs_torch():
    codes = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode_bf16(int(c)) for c in codes])
    assert np.array_equal(got, ref, equal_nan=True)


def test_decode_e4m3_golden_and_structure():
    for ln in golden_lines("e4m3_codes.txt"):
        code, val = ln.split()
        got = oracle.decode_e4m3(int(code, 16))
        assert got == float(val) and np.signbit(got) == val.startswith("-"), ln
    assert np.isnan(oracle.decode_e4m3(0x7F)) and np.isnan(oracle.decode_e4m3(0xFF))
    pos = [oracle.decode_e4m3(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))          # 127 increasing finite values
    for c in range(0x7F):
        assert oracle.decode_e4m3(c | 0x80) == -pos[c]
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    assert np.array_equal(np.array([oracle.decode_e4m3(c) for c in range(256)]), ref.numpy(), equal_nan=True)


def test_ag_fp8_scales():
    """With e4m3 inputs the product carries sx * sw (the gathered input's
    scale_inv times the weight's)."""
    rng = np.random.default_rng(9)
    vals = np.array([0, 1, -1, 2, -2, 0.5, -0.5, 3, 4, -4, 0.25], dtype=np.float32)
    xs_f = [rng.choice(vals, size=(3, 16)) for _ in range(2)]
    w_f = rng.choice(vals, size=(5, 16))
    enc = synth.f32_to_e4m3_bits
    y = oracle.ag(oracle.gather([enc(x) for x in xs_f]), enc(w_f), sx=0.5, sw=0.25)
    ref = np.concatenate(xs_f, 0).astype(np.float64) @ w_f.astype(np.float64).T * 0.125
    assert np.array_equal(y, ref)


def test_ksplit_fp8_scales():
    """e4m3 K-slices carry one scale_inv for all X_r and one for all W_r: the
    sum over ranks is multiplied by sx * sw."""
    rng = np.random.default_rng(11)
    vals = np.array([0, 1, -1, 2, -2, 0.5, 3, -4, 0.25], dtype=np.float32)
    xs_f = [rng.choice(vals, size=(4, 16)) for _ in range(3)]
    ws_f = [rng.choice(vals, size=(5, 16)) for _ in range(3)]
    enc = synth.f32_to_e4m3_bits
    y = oracle.ksplit([enc(x) for x in xs_f], [enc(w) for w in ws_f], sx=0.5, sw=0.25)
    ref = sum(x.astype(np.float64) @ w.astype(np.float64).T for x, w in zip(xs_f, ws_f)) * 0.125
    assert np.array_equal(y, ref)
    # bf16 inputs ignore the scale arguments
    yb = oracle.ksplit([bf16(x) for x in xs_f], [bf16(w) for w in ws_f], sx=0.5, sw=0.25)
    assert np.array_equal(yb, ref / 0.125)


# ---------------------------------------------------------------- bf16 ring (wire) reduction

def _bf16_table():
    """Every finite bf16 value (sorted) and its 16-bit code."""
    codes = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        vals = (codes << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    ok = np.isfinite(vals) & ~((vals == 0) & (codes >= 0x8000))     # one zero (+0)
    order = np.argsort(vals[ok], kind="stable")
    return vals[ok][order], codes[ok][order]


def _nearest_even_by_search(v, table):
    """Brute force: the nearest finite bf16 value, on a tie the one with an even
    code; past the largest finite value by half a spacing or more, infinity."""
    vals, codes = table
    i = int(np.searchsorted(vals, v))
    if i >= len(vals):
        hi_gap = vals[-1] - vals[-2]
        return np.inf if v - vals[-1] >= hi_gap / 2 else vals[-1]
    if vals[i] == v:
        return v
    if i == 0:
        lo_gap = vals[1] - vals[0]
        return -np.inf if vals[0] - v >= lo_gap / 2 else vals[0]
    lo, hi = vals[i - 1], vals[i]
    if v - lo < hi - v:
        return lo
    if hi - v < v - lo:
        return hi
    return lo if codes[i - 1] % 2 == 0 else hi


def test_round_bf16_matches_nearest_even_search():
    table = _bf16_table()
    vals = table[0]
    rng = np.random.default_rng(12)
    probes = [0.0, 1.0, -1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2.0 ** -133, 2.0 ** -134,
              3 * 2.0 ** -135, 2.0 ** -126 * (1 - 2 ** -9), 3.3895313892515355e38, 3.3961775292304e38,
              3.4e38, -3.4e38]
    pos = vals[vals > 0]
    picks = rng.integers(0, len(pos) - 1, 4000)
    mids = (pos[picks] + pos[picks + 1]) / 2                      # ties, every binade
    probes += list(mids) + list(-mids)
    probes += list(np.nextafter(mids, np.inf)) + list(np.nextafter(mids, -np.inf))
    probes += list(rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000))
    for v in probes:
        assert oracle.round_bf16(v) == _nearest_even_by_search(v, table), v


def _wire_golden():
    d = {}
    for ln in golden_lines("wire_bf16_tp3.txt"):
        key, *v = ln.split()
        d.setdefault(key, []).append([float(x) for x in v])
    return d


def _wire_inputs(d, rows, enc=None):
    enc = enc or (lambda a: synth.f32_to_bf16_bits(np.asarray(a, dtype=np.float32)))
    xs = [enc(np.repeat(np.array(d["x%d" % r]), rows, 0)) for r in range(3)]
    ws = [enc(np.array(d["w%d" % r])) for r in range(3)]
    return xs, ws


def test_wire_bf16_golden_rs_and_ar():
    d = _wire_golden()
    xs, ws = _wire_inputs(d, 3)
    want = np.array([d["rs%d" % b][0] for b in range(3)])
    assert np.array_equal(oracle.ksplit_wire_bf16(xs, ws, op="rs"), want)
    xs6, ws6 = _wire_inputs(d, 6)
    want = np.array([d["ar%d" % i][0] for i in range(6)])
    assert np.array_equal(oracle.ksplit_wire_bf16(xs6, ws6, op="ar", n_chunks=2), want)
    # the golden rows differ from a single rounding of the exact sum
    exact = oracle.ksplit(xs, ws)
    single = np.vectorize(oracle.round_bf16)(exact)
    assert not np.array_equal(single, oracle.ksplit_wire_bf16(xs, ws, op="rs"))


@pytest.mark.parametrize("plant", [1, 2, 3])
def test_wire_bf16_golden_catches_each_planted_mistake(plant, tmp_path):
    """Oracle copies built with one deliberate mistake (partials not rounded,
    running sums not rounded, ring starting at the owner) disagree with the
    hand-worked golden rows."""
    d = _wire_golden()
    xs, ws = _wire_inputs(d, 3)
    want = np.array([d["rs%d" % b][0] for b in range(3)])
    bad = oracle.planted_variant(plant, str(tmp_path))
    assert not np.array_equal(bad.ksplit_wire_bf16(xs, ws, op="rs"), want)


def test_wire_bf16_golden_with_e4m3_scales():
    """e4m3 inputs: the partials carry sx * sw before they are rounded; with a
    power-of-two scale product the golden rows scale exactly."""
    d = _wire_golden()
    xs, ws = _wire_inputs(d, 3, enc=lambda a: synth.f32_to_e4m3_bits(np.asarray(a, dtype=np.float32)))
    want = np.array([d["rs%d" % b][0] for b in range(3)]) * 0.125
    assert np.array_equal(oracle.ksplit_wire_bf16(xs, ws, op="rs", sx=0.5, sw=0.25), want)


@pytest.mark.parametrize("op,tp,n,kr,m,chunks", [("rs", 2, 4, 3, 5, 1), ("rs", 4, 8, 2, 3, 1),
                                                 ("ar", 3, 12, 4, 6, 2), ("ar", 2, 8, 5, 4, 4)])
def test_wire_bf16_exact_when_nothing_rounds(op, tp, n, kr, m, chunks):
    """Small integers keep every partial and every running sum below 256 in
    magnitude, all exact in bf16: the ring sum is then the exact sum."""
    rng = np.random.default_rng(n * 7 + kr)
    xs_i = [rng.integers(-3, 4, size=(n, kr)) for _ in range(tp)]
    ws_i = [rng.integers(-3, 4, size=(m, kr)) for _ in range(tp)]
    ref = sum(x.astype(np.float64) @ w.astype(np.float64).T for x, w in zip(xs_i, ws_i))
    got = oracle.ksplit_wire_bf16([bf16(x) for x in xs_i], [bf16(w) for w in ws_i], op=op, n_chunks=chunks)
    assert np.array_equal(got, ref)


def test_wire_bf16_single_rank_is_the_rounded_product():
    """tp = 1: no hop, so the result is the product rounded to bf16 once."""
    rng = np.random.default_rng(4)
    x = synth.f32_to_bf16_bits(rng.standard_normal((16, 24)).astype(np.float32))
    w = synth.f32_to_bf16_bits(rng.standard_normal((8, 24)).astype(np.float32))
    exact = oracle.ksplit([x], [w])
    got = oracle.ksplit_wire_bf16([x], [w], op="rs")
    table = _bf16_table()
    assert np.array_equal(got, np.vectorize(lambda v: _nearest_even_by_search(v, table))(exact))


def test_wire_bf16_tiles_match_full():
    rng = np.random.default_rng(8)
    xs = [synth.f32_to_bf16_bits(rng.standard_normal((32, 8)).astype(np.float32)) for _ in range(4)]
    ws = [synth.f32_to_bf16_bits(rng.standard_normal((48, 8)).astype(np.float32)) for _ in range(4)]
    for op, ch in (("rs", 1), ("ar", 2)):
        full = oracle.ksplit_wire_bf16(xs, ws, op=op, n_chunks=ch)
        tiles = synth.sample_tiles(32, 48, 16, 4, seed=3)
        got = oracle.ksplit_wire_bf16(xs, ws, op=op, n_chunks=ch, tiles=tiles)
        for t, (r0, c0) in enumerate(tiles):
            assert np.array_equal(got[t], full[r0:r0 + 16, c0:c0 + 16])
