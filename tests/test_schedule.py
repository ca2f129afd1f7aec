"""CPU mirror of the fused kernel's tile schedule and producer split.

The kernel's index arithmetic (tile order, TMA coordinates, producer pieces)
is restated here and checked, for every workload shape and some edge shapes,
to cover each output element exactly once, to keep every tensor-map access in
bounds and 16-byte aligned, and to follow the ring orders of the pages.
"""

import pytest

from tensor_comm_gemm_gb300 import synth

BM, BN, BK_BYTES, COPY_PIECE, EPI_COLS = 128, 256, 128, 16384, 32


def tile_at(op, tp, self_rank, rows_per_group, row_tiles, col_tiles, t, tile_m=BM):
    per = row_tiles * col_tiles
    grp, rem = divmod(t, per)
    c, r = divmod(rem, row_tiles)
    col = c * BN
    if op == "ag":
        slot = (self_rank - grp) % tp
        a_map = 1 if grp == 0 else 0
        a_row = r * tile_m if grp == 0 else slot * rows_per_group + r * tile_m
        gate = -1 if grp == 0 else slot
        return dict(a_map=a_map, a_row=a_row, gate=gate, y_map=0, y_row=slot * rows_per_group + r * tile_m,
                    col=col, seg0=0, group=grp)
    if op == "rs":
        return dict(a_map=-1, a_row=grp * rows_per_group + r * tile_m, gate=-1, y_map=grp, y_row=r * tile_m,
                    col=col, seg0=(grp + 1) % tp, group=grp)
    local = r * tile_m
    owner = (local * tp) // rows_per_group
    return dict(a_map=-1, a_row=grp * rows_per_group + local, gate=-1, y_map=0,
                y_row=grp * rows_per_group + local, col=col, seg0=(owner + 1) % tp, group=grp)


def choose_cg(op, tp, n, chunks):
    """The host's variant choice: CTA pairs when every 256-row tile lies in one
    group (and, for AR, in one ring-order part of its chunk)."""
    groups = tp if op in ("ag", "rs") else chunks
    rows = n // groups
    part = rows // tp if op == "ar" else rows
    return 2 if rows % (2 * BM) == 0 and part % (2 * BM) == 0 else 1


def plan(op, tp, n, k, m, elem=2, chunks=1, cg=1):
    tile_m = BM * cg
    if op == "ag":
        rows = n // tp
        return dict(rows_per_group=rows, row_tiles=rows // tile_m, col_tiles=m // BN, groups=tp,
                    kb=k * elem // BK_BYTES, segs=1, tile_m=tile_m)
    groups = tp if op == "rs" else chunks
    rows = n // groups
    return dict(rows_per_group=rows, row_tiles=rows // tile_m, col_tiles=m // BN, groups=groups,
                kb=(k // tp) * elem // BK_BYTES, segs=tp, tile_m=tile_m)


SHAPES = [("ag", 2, 256, 256, 256, 2, 1), ("ag", 4, 4096, 4096, 4096, 2, 1), ("ag", 8, 16384, 8192, 28672, 1, 1),
          ("ag", 3, 768, 192, 768, 2, 1), ("ag", 1, 128, 64, 256, 2, 1),
          ("ar", 2, 8192, 8192, 8192, 2, 4), ("ar", 3, 2304, 384, 512, 2, 2),
          ("rs", 8, 16384, 28672, 8192, 2, 1), ("rs", 3, 768, 192, 512, 2, 1), ("rs", 1, 256, 64, 256, 2, 1)]


@pytest.mark.parametrize("op,tp,n,k,m,elem,chunks", SHAPES)
@pytest.mark.parametrize("cg", [1, 2])
def test_tiles_cover_output_once_in_bounds(op, tp, n, k, m, elem, chunks, cg):
    if cg == 2 and choose_cg(op, tp, n, chunks) != 2:
        pytest.skip("shape served by the single-SM variant")
    pl = plan(op, tp, n, k, m, elem, chunks, cg)
    tile_m = pl["tile_m"]
    total = pl["groups"] * pl["row_tiles"] * pl["col_tiles"]
    kel = BK_BYTES // elem
    kcols = k if op == "ag" else k // tp
    b_rows = BN // cg
    for self_rank in sorted({0, tp - 1, tp // 2}):
        seen = set()
        gated_order = []
        for t in range(total):
            T = tile_at(op, tp, self_rank, pl["rows_per_group"], pl["row_tiles"], pl["col_tiles"], t, tile_m)
            if op != "ag":
                # the CTAs of a pair share one K-segment order: one owner for all tile rows
                rows_part = pl["rows_per_group"] // tp
                if op == "ar":
                    assert (T["a_row"] % pl["rows_per_group"]) // rows_part == \
                        (T["a_row"] % pl["rows_per_group"] + tile_m - 1) // rows_part
            for rank in range(cg):
                off = BM * rank
                if op == "rs":
                    assert 0 <= T["y_row"] + off and T["y_row"] + off + BM <= n // tp
                    key = (T["y_map"] * (n // tp) + T["y_row"] + off, T["col"])
                else:
                    assert 0 <= T["y_row"] + off and T["y_row"] + off + BM <= n
                    key = (T["y_row"] + off, T["col"])
                assert key not in seen
                seen.add(key)
                a_rows = (n // tp) if (op == "ag" and T["a_map"] == 1) else n
                assert 0 <= T["a_row"] + off and T["a_row"] + off + BM <= a_rows
                # B rows this CTA loads: its share of the tile's columns
                assert T["col"] + b_rows * rank + b_rows <= m
                if op == "ag":
                    src_row = T["a_row"] if T["a_map"] == 0 else self_rank * (n // tp) + T["a_row"]
                    assert src_row == T["y_row"]
            assert T["col"] + BN <= m and (T["col"] * 2) % 16 == 0
            if op == "ag":
                if T["gate"] >= 0 and T["gate"] not in gated_order:
                    gated_order.append(T["gate"])
            else:
                order = [(T["seg0"] + s) % tp for s in range(tp)]
                assert sorted(order) == list(range(tp))
                if op == "rs":
                    assert order[-1] == T["group"]
            for i in range(pl["kb"]):
                x = i * kel
                assert x + kel <= kcols and (x * elem) % 16 == 0
            for c in range(BN // EPI_COLS):
                assert ((T["col"] + c * EPI_COLS) * 2) % 16 == 0
        assert len(seen) == (n // BM) * (m // BN)
        if op == "ag":
            assert gated_order == [(self_rank - s) % tp for s in range(1, tp)]


@pytest.mark.parametrize("chunk_bytes,P", [(128 * 256 * 2, 8), (1024 * 4096 * 2, 8), (2048 * 8192, 8),
                                           (128 * 64 * 2, 8), (384 * 192 * 2, 3), (1024 * 4096 * 2, 152)])
def test_producer_pieces_partition_chunk(chunk_bytes, P):
    pieces = (chunk_bytes + COPY_PIECE - 1) // COPY_PIECE
    covered = 0
    for pid in range(P):
        lo, hi = pieces * pid // P, pieces * (pid + 1) // P
        for i in range(lo, hi):
            nbytes = min(COPY_PIECE, chunk_bytes - i * COPY_PIECE)
            assert 0 < nbytes <= COPY_PIECE and nbytes % 16 == 0
            assert i * COPY_PIECE == covered
            covered += nbytes
    assert covered == chunk_bytes


def test_workload_shapes_fit_the_tiling():
    for idx, (op, dt, tp, n, k, m, chunks) in synth.WORKLOAD_SHAPES.items():
        assert n % (tp * BM) == 0 and m % BN == 0
        if op == "ag":
            assert k % (64 if dt == "bf16" else 128) == 0
        else:
            assert k % tp == 0 and (k // tp) % 64 == 0
            assert n % (chunks * tp * BM) == 0
