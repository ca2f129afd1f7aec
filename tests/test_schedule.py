"""CPU mirror of the fused kernel's tile schedule and producer split.

The kernel's index arithmetic (tile order, TMA coordinates, producer pieces)
is restated here and checked, for every workload shape and for ragged shapes
(partial row, column and K tiles), to cover each output element exactly once
with stores that start inside the output, to load the rows each tile stores,
to keep every TMA inner coordinate 16-byte aligned, and to follow the ring
orders of the pages.
"""

import pytest

from tensor_comm_gemm_gb300 import synth

BM, BN, BK_BYTES, COPY_PIECE, EPI_COLS = 128, 256, 128, 16384, 32


def cdiv(a, b):
    return -(-a // b)


def tile_at(op, tp, self_rank, pl, t):
    """The kernel's tile_at: A and output coordinates are (row, slot) pairs of
    the 3-D [inner, rows, slot] tensor maps."""
    row_tiles, col_tiles, tile_m, rpg = pl["row_tiles"], pl["col_tiles"], pl["tile_m"], pl["rows_per_group"]
    per = row_tiles * col_tiles
    grp, rem = divmod(t, per)
    rb = 2048 // tile_m                    # row tiles per block swept column by column
    full = row_tiles // rb
    if rem < full * rb * col_tiles:
        b, w = divmod(rem, rb * col_tiles)
        c, rr0 = divmod(w, rb)
        r = b * rb + rr0
    else:
        h = row_tiles - full * rb
        c, rr0 = divmod(rem - full * rb * col_tiles, h)
        r = full * rb + rr0
    col = c * BN
    if op == "ag":
        slot = (self_rank - grp) % tp
        return dict(a_map=1 if grp == 0 else 0, a_row=r * tile_m, a_z=0 if grp == 0 else slot,
                    gate=-1 if grp == 0 else slot, y_map=0, y_row=r * tile_m, y_z=slot, col=col, seg0=0, group=grp)
    if op == "rs":
        return dict(a_map=-1, a_row=grp * rpg + r * tile_m, a_z=0, gate=-1, y_map=grp, y_row=r * tile_m, y_z=0,
                    col=col, seg0=(grp + 1) % tp, group=grp)
    part, rr = divmod(r, pl["tiles_per_part"])
    return dict(a_map=-1, a_row=grp * rpg + part * pl["part_rows"] + rr * tile_m, a_z=0, gate=-1, y_map=0,
                y_row=rr * tile_m, y_z=grp * tp + part, col=col, seg0=(part + 1) % tp, group=grp)


def choose_cg(op, tp, n, chunks):
    """The host's variant choice: CTA pairs when every 256-row tile lies in one
    group (and, for AR, in one ring-order part of its chunk)."""
    groups = tp if op in ("ag", "rs") else chunks
    rows = n // groups
    part = rows // tp if op == "ar" else rows
    return 2 if rows % (2 * BM) == 0 and part % (2 * BM) == 0 else 1


def plan(op, tp, n, k, m, elem=2, chunks=1, cg=1):
    tile_m = BM * cg
    groups = tp if op in ("ag", "rs") else chunks
    rows = n // groups
    part_rows = rows // tp if op == "ar" else rows
    tpp = cdiv(part_rows, tile_m)
    kseg = k if op == "ag" else k // tp
    return dict(rows_per_group=rows, part_rows=part_rows, tiles_per_part=tpp,
                row_tiles=tp * tpp if op == "ar" else tpp, col_tiles=cdiv(m, BN), groups=groups,
                kb=cdiv(kseg * elem, BK_BYTES), tile_m=tile_m, y_rows=part_rows)


SHAPES = [("ag", 2, 256, 256, 256, 2, 1), ("ag", 4, 4096, 4096, 4096, 2, 1), ("ag", 8, 16384, 8192, 28672, 1, 1),
          ("ag", 3, 768, 192, 768, 2, 1), ("ag", 1, 128, 64, 256, 2, 1),
          ("ar", 2, 8192, 8192, 8192, 2, 4), ("ar", 3, 2304, 384, 512, 2, 2),
          ("rs", 8, 16384, 28672, 8192, 2, 1), ("rs", 3, 768, 192, 512, 2, 1), ("rs", 1, 256, 64, 256, 2, 1),
          # ragged: partial row tiles, partial column tiles, partial K blocks
          ("ag", 3, 600, 200, 264, 2, 1), ("ag", 2, 1000, 48, 520, 1, 1), ("ag", 5, 5, 8, 8, 2, 1),
          ("rs", 3, 390, 48, 24, 2, 1), ("rs", 2, 1030, 96, 776, 1, 1),
          ("ar", 2, 600, 32, 40, 2, 3), ("ar", 4, 2056, 64, 272, 2, 2),
          # groups of more than 2048 rows: several swept blocks, the last one shorter
          ("ag", 1, 8192, 128, 512, 2, 1), ("ag", 2, 2 * 5000, 64, 264, 2, 1), ("rs", 2, 2 * 2304, 64, 512, 2, 1),
          ("ar", 1, 5000, 64, 264, 2, 1)]


@pytest.mark.parametrize("op,tp,n,k,m,elem,chunks", SHAPES)
@pytest.mark.parametrize("cg", [1, 2])
def test_tiles_cover_output_once_in_bounds(op, tp, n, k, m, elem, chunks, cg):
    if cg == 2 and choose_cg(op, tp, n, chunks) != 2:
        pytest.skip("shape served by the single-SM variant")
    pl = plan(op, tp, n, k, m, elem, chunks, cg)
    total = pl["groups"] * pl["row_tiles"] * pl["col_tiles"]
    kel = BK_BYTES // elem
    kcols = k if op == "ag" else k // tp
    assert (kcols * elem) % 16 == 0 and (m * 2) % 16 == 0  # 16-byte row pitches
    b_rows = BN // cg
    y_rows = pl["y_rows"]
    for self_rank in sorted({0, tp - 1, tp // 2}):
        boxes = set()
        covered = 0
        gated_order = []
        for t in range(total):
            T = tile_at(op, tp, self_rank, pl, t)
            for rank in range(cg):
                off = BM * rank
                # the rows a CTA loads are the rows it stores (same slot, same offset)
                if op == "ag":
                    assert T["a_row"] == T["y_row"] and (T["a_map"] == 1 or T["a_z"] == T["y_z"])
                    if T["a_map"] == 1:
                        assert T["y_z"] == self_rank
                elif op == "rs":
                    assert T["a_row"] == T["y_map"] * pl["rows_per_group"] + T["y_row"]
                else:
                    assert T["a_row"] == T["y_z"] * pl["part_rows"] + T["y_row"]
                assert T["a_row"] + off >= 0 and T["col"] + b_rows * rank >= 0
                for q in range(4):
                    for c in range(BN // EPI_COLS):
                        ox, oy = T["col"] + c * EPI_COLS, T["y_row"] + off + 32 * q
                        assert (ox * 2) % 16 == 0 and oy >= 0   # stores never start at a negative coordinate
                        if ox >= m or oy >= y_rows:
                            continue                            # skipped by the epilogue
                        key = (T["y_map"], T["y_z"], oy, ox)
                        assert key not in boxes
                        boxes.add(key)
                        covered += (min(oy + 32, y_rows) - oy) * (min(ox + EPI_COLS, m) - ox)
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
                assert x < kcols and (x * elem) % 16 == 0
        assert covered == n * m
        if op == "ag":
            assert gated_order == [(self_rank - s) % tp for s in range(1, tp)]


@pytest.mark.parametrize("chunk_bytes,P", [(128 * 256 * 2, 8), (1024 * 4096 * 2, 8), (2048 * 8192, 8),
                                           (128 * 64 * 2, 8), (384 * 192 * 2, 3), (1024 * 4096 * 2, 152),
                                           (200 * 200 * 2, 8), (1 * 8 * 2, 8), (500 * 48, 24)])
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
    """The benchmark workloads are whole tiles (no partial tile anywhere)."""
    for idx, (op, dt, tp, n, k, m, chunks) in synth.WORKLOAD_SHAPES.items():
        assert n % (tp * BM) == 0 and m % BN == 0
        if op == "ag":
            assert k % (64 if dt == "bf16" else 128) == 0
        else:
            assert k % tp == 0 and (k // tp) % 64 == 0
            assert n % (chunks * tp * BM) == 0
