"""The seeded input generator: published splitmix64 vectors, the numpy
definition against the threaded C implementation, and the rounding rules."""

import numpy as np
import pytest
import torch

import oracle
from tensor_comm_gemm_gb300 import synth
from conftest import golden_lines


def test_splitmix64_reference_vectors():
    want = [int(v, 16) for v in golden_lines("splitmix64.txt")]
    assert [int(v) for v in synth.draws(0, 0, len(want))] == want


def test_c_generator_matches_numpy_definition():
    key = synth.stream_key(5, 3)
    u = synth.uniform_pm1(key, 50000)
    assert np.array_equal(synth.fast_uniform_bf16(key, 50000), synth.f32_to_bf16_bits(u))
    assert u.min() >= -1.0 and u.max() < 1.0
    z = synth.normal(key, 50000, 0.5)
    assert np.array_equal(synth.fast_normal_f32(key, 50000, 0.5), z)
    assert np.array_equal(synth.fast_normal_bf16(key, 50000, 0.5), synth.f32_to_bf16_bits(z))
    assert abs(z.mean()) < 0.02 and abs(z.std() - 0.5) < 0.02
    q = synth.fast_quant_e4m3(z * 300, 1.0)
    assert np.array_equal(q, synth.f32_to_e4m3_bits((z * 300).astype(np.float32)))


def test_bf16_rounding_vs_torch():
    x = np.random.default_rng(0).standard_normal(200000).astype(np.float32) * 1e3
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f32_to_bf16_bits(x), ref)


def test_e4m3_encoder_round_trip_ties_and_saturation():
    for c in range(256):
        v = oracle.decode_e4m3(c)
        if not np.isnan(v):
            assert int(synth.f32_to_e4m3_bits(np.float32(v))) == c
    enc = lambda v: oracle.decode_e4m3(int(synth.f32_to_e4m3_bits(np.float32(v))))
    assert enc(1.0625) == 1.0          # tie between 1 (even) and 1.125
    assert enc(1.1875) == 1.25         # tie between 1.125 and 1.25 (even)
    assert enc(500.0) == 448.0 and enc(-1e9) == -448.0
    assert enc(2.0 ** -10) == 0.0      # half of the smallest subnormal: tie to 0
    x = np.clip(np.random.default_rng(1).standard_normal(200000).astype(np.float32) * 100, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(synth.f32_to_e4m3_bits(x), ref)


def test_sample_tiles_distinct_and_in_range():
    t = synth.sample_tiles(4096, 4096, 16, 4096, seed=1001)
    assert t.shape == (4096, 2)
    assert len({(int(a), int(b)) for a, b in t}) == 4096
    assert t.min() >= 0 and t[:, 0].max() <= 4096 - 16 and t[:, 1].max() <= 4096 - 16
    assert np.all(t % 16 == 0)
    assert np.array_equal(t, synth.sample_tiles(4096, 4096, 16, 4096, seed=1001))
    small = synth.sample_tiles(32, 48, 16, 100, seed=1)
    assert len(small) == 6


def test_small_workload_shapes():
    w = synth.workload(0)
    assert w.op == "ag" and w.tp == 2 and len(w.x) == 2 and w.x[0].shape == (128, 256)
    assert w.w[0].shape == (256, 256) and w.x[0].dtype == np.uint16
    v = synth.bf16_bits_to_f32(w.x[0])
    assert v.min() >= -1 and v.max() <= 1    # bf16 rounding may carry 1 - 2**-24 up to 1
