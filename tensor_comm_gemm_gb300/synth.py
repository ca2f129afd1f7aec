"""Seeded synthetic inputs for the tensor-parallel overlap GEMMs.

This module is the one place that both the CUDA path's callers (tests,
``bench.py``) and the CPU oracle draw their inputs from.  It holds no part of
the method's arithmetic: it only draws random numbers, rounds them to the
input storage types (bf16, OCP e4m3) and lays the per-rank buffers out.

Definitions (all counter-based, so any element can be regenerated alone):

* ``mix64`` is the splitmix64 output function; the i-th draw of a stream with
  key ``key`` is ``mix64(key + (i + 1) * 0x9E3779B97F4A7C15 mod 2**64)``.
* The key of tensor ``tid`` of a workload seeded ``seed`` is
  ``mix64(mix64(seed) ^ tid)``.
* Uniform[-1, 1): ``u = (draw >> 40) * 2**-24`` (exact in fp32), ``x = 2u - 1``.
* Normal(0, sigma): element i uses draws 2i and 2i+1,
  ``u1 = ((d0 >> 11) + 1) * 2**-53``, ``u2 = (d1 >> 11) * 2**-53``,
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)`` in double, then ``fp32(z * sigma)``.
* bf16: round-to-nearest-even of the fp32 value.
* e4m3 (OCP FP8 E4M3, bias 7, max 448, no infinities): round-to-nearest-even
  with saturation to +-448 (the ``satfinite`` convention).
* FP8 per-tensor scaling: ``scale = fp32(448 / amax)``, ``q = e4m3(fp32(x*scale))``,
  ``scale_inv = fp32(1 / scale)``; one scale for all ranks' X together (the
  gathered tensor carries a single ``scale_inv`` in TransformerEngine's
  atomic_gemm_overlap_ag, where the gathered input keeps ``B.scale_inv()``),
  one for W.

The "N(0, 1/sqrt(K))" of the workload descriptions is read as a variance, so
``sigma = K ** -0.25`` and every output element has unit variance.
"""

from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading
from typing import List, Optional

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 22  # elements generated per numpy pass (bounds host memory)

E4M3_MAX = 448.0


def mix64(z):
    """splitmix64 output function on uint64 scalars or arrays (wrapping)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z ^ (z >> np.uint64(30))
        z = z * _M1
        z = z ^ (z >> np.uint64(27))
        z = z * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def stream_key(seed: int, tid: int) -> np.uint64:
    return np.uint64(mix64(np.uint64(mix64(np.uint64(seed))) ^ np.uint64(tid)))


def draws(key, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the splitmix64 stream with key ``key``."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(key) + idx * GOLDEN_GAMMA
    return mix64(state)


def uniform_pm1(key, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    for s in range(0, count, _BLOCK):
        c = min(_BLOCK, count - s)
        d = draws(key, s, c)
        u = (d >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
        out[s:s + c] = np.float32(2.0) * u - np.float32(1.0)
    return out


def normal(key, count: int, sigma: float) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    for s in range(0, count, _BLOCK):
        c = min(_BLOCK, count - s)
        d = draws(key, 2 * s, 2 * c)
        d0, d1 = d[0::2], d[1::2]
        u1 = ((d0 >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)
        u2 = (d1 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
        out[s:s + c] = (z * sigma).astype(np.float32)
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """OCP E4M3 encoding with round-to-nearest-even and saturation to +-448."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    sign = (np.signbit(x)).astype(np.uint8) << np.uint8(7)
    # binade exponent of a (a = f * 2**e, f in [1, 2)); subnormals share e = -6
    _, e2 = np.frexp(a)
    e = np.maximum(e2.astype(np.int64) - 1, -6)
    quantum = np.ldexp(1.0, (e - 3).astype(np.int64))
    v = np.rint(a / quantum) * quantum            # np.rint rounds half to even
    v = np.minimum(v, E4M3_MAX)
    # encode the (now representable) magnitude
    _, ev = np.frexp(v)
    ev = ev.astype(np.int64) - 1
    sub = (v < 2.0 ** -6)
    mant_sub = np.rint(v / 2.0 ** -9).astype(np.int64)          # 0..7
    ev_n = np.maximum(ev, -6)
    mant_n = np.rint(v / np.ldexp(1.0, ev_n - 3)).astype(np.int64) - 8
    code = np.where(sub, mant_sub, ((ev_n + 7) << 3) | np.clip(mant_n, 0, 7))
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_bits_to_f32(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    mnt = c & 7
    v = np.where(e == 0, mnt * 2.0 ** -9, (8 + mnt) * np.ldexp(1.0, e - 10))
    v = np.where((c & 0x7F) == 0x7F, np.nan, v)
    return (s * v).astype(np.float32)


def sample_tiles(rows: int, cols: int, tile: int, count: int, seed: int):
    """``count`` distinct (row0, col0) tile origins of a rows x cols output, drawn
    without replacement from a splitmix64 stream; all tiles if count covers them."""
    tr, tc = rows // tile, cols // tile
    total = tr * tc
    if count >= total:
        idx = np.arange(total, dtype=np.int64)
    else:
        key = stream_key(seed, 0)
        chosen, seen, pos = [], set(), 0
        while len(chosen) < count:
            d = draws(key, pos, 2 * count)
            pos += 2 * count
            for v in (d % np.uint64(total)).astype(np.int64).tolist():
                if v not in seen:
                    seen.add(v)
                    chosen.append(v)
                    if len(chosen) == count:
                        break
        idx = np.array(sorted(chosen), dtype=np.int64)
    return np.stack([(idx // tc) * tile, (idx % tc) * tile], axis=1)


# ----------------------------------------------------------------------------
# threaded C implementation of the same draws (gen/tpo_synth.c)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SYNTH_SRC = os.path.join(_HERE, "gen", "tpo_synth.c")
_SYNTH_SO = os.path.join(_HERE, "gen", "libtpo_synth.so")
_lib_lock = threading.Lock()
_lib_handle = None


def build_synth(force: bool = False) -> str:
    """Compile the C generator (plain gcc, no GPU); returns the .so path."""
    if force or not os.path.exists(_SYNTH_SO) or os.path.getmtime(_SYNTH_SO) < os.path.getmtime(_SYNTH_SRC):
        tmp = _SYNTH_SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
                               "-o", tmp, _SYNTH_SRC, "-lm"])
        os.replace(tmp, _SYNTH_SO)
    return _SYNTH_SO


def _lib():
    global _lib_handle
    with _lib_lock:
        if _lib_handle is None:
            lib = ctypes.CDLL(build_synth())
            i64, u64, p = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
            lib.tpo_synth_uniform_bf16.argtypes = [u64, i64, p, ctypes.c_int]
            lib.tpo_synth_normal_bf16.argtypes = [u64, i64, ctypes.c_double, p, ctypes.c_int]
            lib.tpo_synth_normal_f32.argtypes = [u64, i64, ctypes.c_double, p, ctypes.c_int]
            lib.tpo_synth_quant_e4m3.argtypes = [p, i64, ctypes.c_float, p, ctypes.c_int]
            _lib_handle = lib
    return _lib_handle


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def fast_uniform_bf16(key, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    _lib().tpo_synth_uniform_bf16(int(key), count, out.ctypes.data, _threads())
    return out


def fast_normal_bf16(key, count: int, sigma: float) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    _lib().tpo_synth_normal_bf16(int(key), count, float(sigma), out.ctypes.data, _threads())
    return out


def fast_normal_f32(key, count: int, sigma: float) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    _lib().tpo_synth_normal_f32(int(key), count, float(sigma), out.ctypes.data, _threads())
    return out


def fast_quant_e4m3(x: np.ndarray, scale: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _lib().tpo_synth_quant_e4m3(x.ctypes.data, x.size, float(np.float32(scale)), out.ctypes.data, _threads())
    return out


# ----------------------------------------------------------------------------
# workloads

@dataclasses.dataclass
class Workload:
    """Inputs of one call.  ``op`` is 'ag', 'rs' or 'ar'; bf16 tensors are
    uint16 bit arrays, e4m3 tensors uint8 code arrays, all row-major."""
    name: str
    op: str
    dtype: str            # 'bf16' | 'e4m3'
    tp: int
    n: int                # rows of Y (tokens)
    k: int                # global contraction length
    m: int                # columns of Y (features)
    x: List[np.ndarray]   # AG: tp x [n/tp, k]; RS/AR: tp x [n, k/tp]
    w: List[np.ndarray]   # AG: [W] of [m, k]; RS/AR: tp x [m, k/tp]
    scale_inv_x: float = 1.0
    scale_inv_w: float = 1.0
    n_row_chunks: int = 1
    seed: int = 0


def _bf16_tensor(seed, tid, shape, dist, sigma=1.0):
    cnt = int(np.prod(shape))
    key = stream_key(seed, tid)
    v = fast_uniform_bf16(key, cnt) if dist == "uniform" else fast_normal_bf16(key, cnt, sigma)
    return v.reshape(shape)


def _quantize_e4m3(vals: List[np.ndarray]):
    amax = np.float32(max(float(np.max(np.abs(v))) for v in vals))
    scale = np.float32(np.float32(E4M3_MAX) / amax)
    out = [fast_quant_e4m3(v, scale) for v in vals]
    return out, float(np.float32(np.float32(1.0) / scale))


def make_ag(tp, n, k, m, seed, dist="uniform", sigma=1.0, dtype="bf16", name="ag") -> Workload:
    rows = n // tp
    if dtype == "bf16":
        x = [_bf16_tensor(seed, r, (rows, k), dist, sigma) for r in range(tp)]
        w = [_bf16_tensor(seed, 100, (m, k), dist, sigma)]
        return Workload(name, "ag", "bf16", tp, n, k, m, x, w, seed=seed)
    xs = [fast_normal_f32(stream_key(seed, r), rows * k, 1.0).reshape(rows, k) for r in range(tp)]
    xq, sx = _quantize_e4m3(xs)
    del xs
    wf = fast_normal_f32(stream_key(seed, 100), m * k, 1.0).reshape(m, k)
    wq, sw = _quantize_e4m3([wf])
    del wf
    return Workload(name, "ag", "e4m3", tp, n, k, m, xq, wq, sx, sw, seed=seed)


def make_ksplit(op, tp, n, k, m, seed, dist="normal", sigma=1.0, n_row_chunks=1, name=None,
                dtype="bf16") -> Workload:
    kr = k // tp
    if dtype == "bf16":
        x = [_bf16_tensor(seed, r, (n, kr), dist, sigma) for r in range(tp)]
        w = [_bf16_tensor(seed, 100 + r, (m, kr), dist, sigma) for r in range(tp)]
        return Workload(name or op, op, "bf16", tp, n, k, m, x, w, n_row_chunks=n_row_chunks, seed=seed)
    # e4m3: N(0,1) values, one amax-derived scale for all X_r and one for all W_r
    xs = [fast_normal_f32(stream_key(seed, r), n * kr, 1.0).reshape(n, kr) for r in range(tp)]
    xq, sx = _quantize_e4m3(xs)
    del xs
    ws = [fast_normal_f32(stream_key(seed, 100 + r), m * kr, 1.0).reshape(m, kr) for r in range(tp)]
    wq, sw = _quantize_e4m3(ws)
    del ws
    return Workload(name or op, op, "e4m3", tp, n, k, m, xq, wq, sx, sw, n_row_chunks=n_row_chunks, seed=seed)


def workload(idx: int) -> Workload:
    """The five reference workloads (see the module docstring for the recipe)."""
    if idx == 0:   # AG+GEMM tp=2, X_r [128,256], W [256,256], uniform[-1,1)
        return make_ag(2, 256, 256, 256, seed=0, dist="uniform", name="ag_tp2_256")
    if idx == 1:   # AG+GEMM tp=4, M=K=N=4096
        return make_ag(4, 4096, 4096, 4096, seed=1, dist="normal", sigma=4096 ** -0.25,
                       name="ag_tp4_4096")
    if idx == 2:   # row-parallel linear + allreduce, tp=2, 4 row chunks
        return make_ksplit("ar", 2, 8192, 8192, 8192, seed=2, sigma=8192 ** -0.25,
                           n_row_chunks=4, name="ar_tp2_8192")
    if idx == 3:   # GEMM+RS tp=8, MLP down-projection
        return make_ksplit("rs", 8, 16384, 28672, 8192, seed=3, sigma=28672 ** -0.25,
                           name="rs_tp8_16384x8192x28672")
    if idx == 4:   # FP8 AG+GEMM tp=8
        return make_ag(8, 16384, 8192, 28672, seed=4, dtype="e4m3", name="ag_fp8_tp8_16384x28672x8192")
    raise ValueError(idx)


WORKLOAD_SHAPES = {
    # idx: (op, dtype, tp, n, k, m, n_row_chunks)
    0: ("ag", "bf16", 2, 256, 256, 256, 1),
    1: ("ag", "bf16", 4, 4096, 4096, 4096, 1),
    2: ("ar", "bf16", 2, 8192, 8192, 8192, 4),
    3: ("rs", "bf16", 8, 16384, 28672, 8192, 1),
    4: ("ag", "e4m3", 8, 16384, 8192, 28672, 1),
}


def flops(idx: int) -> float:
    _, _, _, n, k, m, _ = WORKLOAD_SHAPES[idx]
    return 2.0 * n * k * m
