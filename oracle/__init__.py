"""CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never links, loads or
calls it.  The arithmetic lives in ``oracle.c`` (plain FP64 loops over the
rounded inputs); this module compiles it with gcc and marshals numpy arrays.

Functions and the passages they follow:

* ``ring_order`` -- TransformerEngine issue "curious about
  atomic_gemm_overlap_ag", listing of CommOverlapP2PBase::atomic_gemm_overlap_ag:
  each step sends to the next rank and receives from the previous one.
* ``gather`` / ``staging_after_step`` -- same listing: the all-gather output
  is contiguous in rank order on every rank after the ring exchanges.
* ``ag`` -- same listing: one TN GEMM of the gathered rows against the weight
  (m output features, n gathered rows); FP8 inputs carry per-tensor scale_inv.
* ``ksplit`` / ``rs_blocks`` -- nvFuser PR "Reference implementation for
  Linear+Allreduce with overlapping" (matmul of the input chunk with the
  transposed weight shard, then all-reduce SUM) and TransformerEngine PR
  "Comm+GEMM overlap API updated to support cuBlasMp backend" (GEMM then
  reduce-scatter): the sum over ranks of X_r . W_r^T, row block b to rank b.
* ``round_bf16`` / ``ksplit_wire_bf16`` -- the same K-split sum as a bf16
  ring computes it (the nvFuser PR's nsys trace: NCCL's bf16 ring all-reduce
  kernel): each rank's partial rounded to bf16, each hop's fp32 sum rounded
  to bf16, ranks in the ring order that ends at the row's owner.

Parity status: every function here is pinned by ``tests/test_oracle.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_handle = None

DT_BF16, DT_E4M3 = 0, 1


_CFLAGS = ["-O2", "-fPIC", "-shared", "-ffp-contract=off", "-pthread"]


def build(force: bool = False) -> str:
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc"] + _CFLAGS + ["-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _declare(lib):
    p, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_bf16.restype = dbl
    lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_decode_e4m3.restype = dbl
    lib.oracle_round_bf16.argtypes = [dbl]
    lib.oracle_round_bf16.restype = dbl
    lib.oracle_ring_order.argtypes = [i32, i32, p]
    lib.oracle_gather.argtypes = [i32, i64, i64, p, p]
    lib.oracle_staging_after_step.argtypes = [i32, i32, i32, i64, i64, p, ctypes.c_uint8, p]
    lib.oracle_ag_tiles.argtypes = [i32, i64, i64, p, p, dbl, dbl, i64, p, p, i64, i64, p, i32]
    lib.oracle_ksplit_tiles.argtypes = [i32, i32, i64, i64, p, p, dbl, dbl, i64, p, p, i64, i64, p, i32]
    lib.oracle_ksplit_wire_bf16_tiles.argtypes = [i32, i32, i64, i64, i64, i32, i32, p, p, dbl, dbl,
                                                  i64, p, p, i64, i64, p, i32]
    return lib


def planted_variant(plant: int, out_dir: str):
    """A copy of the oracle compiled with one deliberate mistake in the bf16
    ring arithmetic (ORACLE_WIRE_PLANT: 1 partials not rounded, 2 running
    sums not rounded, 3 ring starting at the owner), for the pin tests that
    show each mistake fails a golden case.  Returns a module-like object with
    ``ksplit_wire_bf16``."""
    so = os.path.join(out_dir, "liboracle_plant%d.so" % plant)
    subprocess.check_call(["gcc"] + _CFLAGS + ["-DORACLE_WIRE_PLANT=%d" % plant, "-o", so, _SRC, "-lm"])
    lib = _declare(ctypes.CDLL(so))

    class _Variant:
        @staticmethod
        def ksplit_wire_bf16(*a, **kw):
            return _wire(lib, *a, **kw)
    return _Variant


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            _handle = _declare(ctypes.CDLL(build()))
    return _handle


def threads() -> int:
    return max(1, os.cpu_count() or 1)


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return DT_BF16
    if a.dtype == np.uint8:
        return DT_E4M3
    raise TypeError("inputs are bf16 bit patterns (uint16) or e4m3 codes (uint8)")


def _ptrs(arrs):
    arr = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return arr


def decode_bf16(b: int) -> float:
    return _lib().oracle_decode_bf16(int(b))


def decode_e4m3(c: int) -> float:
    return _lib().oracle_decode_e4m3(int(c))


def round_bf16(v: float) -> float:
    """Nearest bf16 value of a double, ties to even."""
    return _lib().oracle_round_bf16(float(v))


def ring_order(tp: int, self_rank: int):
    out = (ctypes.c_int * tp)()
    if _lib().oracle_ring_order(tp, self_rank, out):
        raise ValueError("bad tp/self")
    return list(out)


def gather(xs) -> np.ndarray:
    xs = [np.ascontiguousarray(x) for x in xs]
    rows, cols = xs[0].shape
    out = np.empty((rows * len(xs), cols), dtype=xs[0].dtype)
    _lib().oracle_gather(len(xs), rows, cols * xs[0].itemsize, _ptrs(xs), out.ctypes.data)
    return out


def staging_after_step(xs, self_rank: int, step: int, sentinel: int) -> np.ndarray:
    xs = [np.ascontiguousarray(x) for x in xs]
    rows, cols = xs[0].shape
    out = np.empty((rows * len(xs), cols), dtype=xs[0].dtype)
    rc = _lib().oracle_staging_after_step(len(xs), self_rank, step, rows, cols * xs[0].itemsize,
                                          _ptrs(xs), sentinel, out.ctypes.data)
    if rc:
        raise ValueError("bad arguments")
    return out


def _tiles(tiles, th, tw):
    tiles = np.ascontiguousarray(np.asarray(tiles, dtype=np.int64).reshape(-1, 2))
    return tiles, np.ascontiguousarray(tiles[:, 0]), np.ascontiguousarray(tiles[:, 1])


def ag(g: np.ndarray, w: np.ndarray, sx: float = 1.0, sw: float = 1.0, tiles=None, tile=16,
       nthreads=None) -> np.ndarray:
    """Reference Y = scale * G . W^T (double).  With ``tiles`` (an (T,2) array
    of tile origins) returns a (T, tile, tile) array of those output tiles."""
    g, w = np.ascontiguousarray(g), np.ascontiguousarray(w)
    n, k = g.shape
    m = w.shape[0]
    assert w.shape[1] == k and g.dtype == w.dtype
    if tiles is None:
        tiles, th, tw = np.zeros((1, 2), dtype=np.int64), n, m
    else:
        th = tw = tile
    tiles, r0, c0 = _tiles(tiles, th, tw)
    out = np.empty((len(tiles), th, tw), dtype=np.float64)
    rc = _lib().oracle_ag_tiles(_dt(g), k, m, g.ctypes.data, w.ctypes.data, float(sx), float(sw), len(tiles),
                                r0.ctypes.data, c0.ctypes.data, th, tw, out.ctypes.data, nthreads or threads())
    if rc:
        raise ValueError("bad arguments")
    return out[0] if th == n and tw == m and len(tiles) == 1 else out


def ksplit(xs, ws, tiles=None, tile=16, nthreads=None, sx: float = 1.0, sw: float = 1.0) -> np.ndarray:
    """Reference Y = sum_r X_r . W_r^T (double), times sx * sw for e4m3 inputs;
    tiles as in ``ag``."""
    xs = [np.ascontiguousarray(x) for x in xs]
    ws = [np.ascontiguousarray(x) for x in ws]
    n, kr = xs[0].shape
    m = ws[0].shape[0]
    assert len(xs) == len(ws) and all(x.shape == (n, kr) for x in xs) and all(x.shape == (m, kr) for x in ws)
    if tiles is None:
        tiles, th, tw = np.zeros((1, 2), dtype=np.int64), n, m
    else:
        th = tw = tile
    tiles, r0, c0 = _tiles(tiles, th, tw)
    out = np.empty((len(tiles), th, tw), dtype=np.float64)
    rc = _lib().oracle_ksplit_tiles(_dt(xs[0]), len(xs), kr, m, _ptrs(xs), _ptrs(ws), float(sx), float(sw), len(tiles),
                                    r0.ctypes.data, c0.ctypes.data, th, tw, out.ctypes.data,
                                    nthreads or threads())
    if rc:
        raise ValueError("bad arguments")
    return out[0] if th == n and tw == m and len(tiles) == 1 else out


def _wire(lib, xs, ws, op="rs", n_chunks=1, tiles=None, tile=16, nthreads=None, sx: float = 1.0,
          sw: float = 1.0) -> np.ndarray:
    xs = [np.ascontiguousarray(x) for x in xs]
    ws = [np.ascontiguousarray(x) for x in ws]
    n, kr = xs[0].shape
    m = ws[0].shape[0]
    assert op in ("rs", "ar")
    assert len(xs) == len(ws) and all(x.shape == (n, kr) for x in xs) and all(x.shape == (m, kr) for x in ws)
    if tiles is None:
        tiles, th, tw = np.zeros((1, 2), dtype=np.int64), n, m
    else:
        th = tw = tile
    tiles, r0, c0 = _tiles(tiles, th, tw)
    out = np.empty((len(tiles), th, tw), dtype=np.float64)
    rc = lib.oracle_ksplit_wire_bf16_tiles(_dt(xs[0]), len(xs), kr, m, n, 1 if op == "ar" else 0, int(n_chunks),
                                           _ptrs(xs), _ptrs(ws), float(sx), float(sw), len(tiles), r0.ctypes.data,
                                           c0.ctypes.data, th, tw, out.ctypes.data, nthreads or threads())
    if rc:
        raise ValueError("bad arguments")
    return out[0] if th == n and tw == m and len(tiles) == 1 else out


def ksplit_wire_bf16(xs, ws, op="rs", n_chunks=1, tiles=None, tile=16, nthreads=None, sx: float = 1.0,
                     sw: float = 1.0) -> np.ndarray:
    """The K-split sum as a bf16 ring computes it (double array of bf16
    values): every rank's partial X_r . W_r^T (times sx * sw for e4m3) rounded
    to bf16, every hop's fp32 sum rounded to bf16, ranks in the ring order
    ending at the row's owner (op "rs": row block of n/tp rows; op "ar":
    ring-order part of one of n_chunks row chunks).  Tiles as in ``ag``."""
    return _wire(_lib(), xs, ws, op, n_chunks, tiles, tile, nthreads, sx, sw)


def rs_blocks(y_full: np.ndarray, tp: int):
    """Reduce-scatter hand-out: rank b receives rows [b*n/tp, (b+1)*n/tp)."""
    n = y_full.shape[0]
    assert n % tp == 0
    rows = n // tp
    return [y_full[b * rows:(b + 1) * rows] for b in range(tp)]
