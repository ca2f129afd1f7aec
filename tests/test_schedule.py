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
STRIP, MAX_TILE_STRIPS, MIN_TILE_STRIPS = 32, 8, 4


def cdiv(a, b):
    return -(-a // b)


def set_columns(pl, m, extra=None):
    """The host's set_columns: 32-column strips across m, each group's column
    tiles (the fewest of at most 8 strips, plus extra[g]), group start tiles."""
    pl["strips"] = cdiv(m, STRIP)
    base = cdiv(pl["strips"], MAX_TILE_STRIPS)
    pl["base_cols"] = base
    pl["group_cols"] = [base + (extra[g] if extra else 0) for g in range(pl["groups"])]
    pl["group_base"] = [0]
    for cols in pl["group_cols"]:
        pl["group_base"].append(pl["group_base"][-1] + pl["row_tiles"] * cols)
    pl["total"] = pl["group_base"][-1]
    return pl


def tile_index(pl, t):
    """tile_index: (group, column tile, row tile) of tile t."""
    row_tiles, tile_m = pl["row_tiles"], pl["tile_m"]
    grp = max(g for g in range(pl["groups"]) if pl["group_base"][g] <= t)
    rem, cols = t - pl["group_base"][grp], pl["group_cols"][grp]
    rb = 2048 // tile_m                    # row tiles per block swept column by column
    full = row_tiles // rb
    if rem < full * rb * cols:
        b, w = divmod(rem, rb * cols)
        c, rr0 = divmod(w, rb)
        r = b * rb + rr0
    else:
        h = row_tiles - full * rb
        c, rr0 = divmod(rem - full * rb * cols, h)
        r = full * rb + rr0
    return grp, c, r


def tile_strips(pl, grp, c):
    """First strip and strip count of column tile c of group grp (even split)."""
    cols = pl["group_cols"][grp]
    s0, s1 = c * pl["strips"] // cols, (c + 1) * pl["strips"] // cols
    return s0, s1 - s0


def tile_at(op, tp, self_rank, pl, t):
    """The kernel's tile_at: A and output coordinates are (row, slot) pairs of
    the 3-D [inner, rows, slot] tensor maps; col and ncols the tile's columns."""
    tile_m, rpg = pl["tile_m"], pl["rows_per_group"]
    grp, c, r = tile_index(pl, t)
    s0, w = tile_strips(pl, grp, c)
    col, ncols = s0 * STRIP, w * STRIP
    if op == "ag":
        slot = (self_rank - grp) % tp
        return dict(a_map=1 if grp == 0 else 0, a_row=r * tile_m, a_z=0 if grp == 0 else slot,
                    gate=-1 if grp == 0 else slot, y_map=0, y_row=r * tile_m, y_z=slot, col=col, ncols=ncols,
                    seg0=0, group=grp)
    if op == "rs":
        return dict(a_map=-1, a_row=grp * rpg + r * tile_m, a_z=0, gate=-1, y_map=grp, y_row=r * tile_m, y_z=0,
                    col=col, ncols=ncols, seg0=(grp + 1) % tp, group=grp)
    part, rr = divmod(r, pl["tiles_per_part"])
    return dict(a_map=-1, a_row=grp * rpg + part * pl["part_rows"] + rr * tile_m, a_z=0, gate=-1, y_map=0,
                y_row=rr * tile_m, y_z=grp * tp + part, col=col, ncols=ncols, seg0=(part + 1) % tp, group=grp)


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
    pl = dict(rows_per_group=rows, part_rows=part_rows, tiles_per_part=tpp,
              row_tiles=tp * tpp if op == "ar" else tpp, groups=groups,
              kb=cdiv(kseg * elem, BK_BYTES), tile_m=tile_m, y_rows=part_rows)
    return set_columns(pl, m)


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


def column_plans(pl, m):
    """Column plans to check: the fewest tiles everywhere, the most every group
    may take, and seeded random extras in between."""
    import random
    base, strips = pl["base_cols"], pl["strips"]
    top = min(strips - base, 15)
    plans = [None, [top] * pl["groups"]]
    rnd = random.Random(pl["groups"] * 1000 + m)
    plans += [[rnd.randint(0, top) for _ in range(pl["groups"])] for _ in range(2)]
    return plans


@pytest.mark.parametrize("op,tp,n,k,m,elem,chunks", SHAPES)
@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("cplan", range(4))
def test_tiles_cover_output_once_in_bounds(op, tp, n, k, m, elem, chunks, cg, cplan):
    if cg == 2 and choose_cg(op, tp, n, chunks) != 2:
        pytest.skip("shape served by the single-SM variant")
    pl = plan(op, tp, n, k, m, elem, chunks, cg)
    set_columns(pl, m, column_plans(pl, m)[cplan])
    total = pl["total"]
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
                # the tile's width: whole strips, at most BN; each CTA of a pair
                # loads half of its B rows, which its B box covers
                assert T["ncols"] % STRIP == 0 and STRIP <= T["ncols"] <= BN and T["col"] < m
                b0 = T["col"] + (T["ncols"] // 2) * rank if cg == 2 else T["col"]
                assert b0 >= 0 and T["ncols"] // cg <= b_rows
                assert T["a_row"] + off >= 0
                for q in range(4):
                    for c in range(T["ncols"] // EPI_COLS):
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


TAIL_SPLIT = 2


def plan_split(T, G, L, kbu, kps=2, tp=4, chunk_bytes=1 << 23, cg=2, last=False):
    """The host's plan: (tail_first, full, ga, wa, gb, wb) or None (no split)."""
    if L > 0:
        P = L * cg
        t_copy = tp * chunk_bytes / (P * 31e9) + 3e-6
        late = 1.2 * t_copy / (kps * 0.36e-6)
        E = (T * kbu + L * late) / (G + L)
        if E > late + 1.0:
            full = min(int(E / kbu), T // G)
            wt = (T - full * G) * kbu
            sm = max(int(E - full * kbu), 0)
            if sm * G > wt:
                sm = wt // G
            if wt - sm * G > 0:
                return (0, full, G, sm * G, L, wt - sm * G)
    full, R = divmod(T, G)
    if R == 0:
        return None
    return (0 if last else 1, full, min(G, TAIL_SPLIT * R), R * kbu, 0, 0)


def segments(g, G, T, nkb, kps, plan):
    """The kernel's SegIter for group g (GEMM groups 0..G-1, late groups after):
    (tile, K-block range, kind, writer groups) in order.  Kinds: whole, finish
    (first part of a split tile), write (a later part)."""
    kbu = nkb // kps
    out = []
    if plan is None:
        if g < G:
            for t in range(g, T, G):
                out.append((t, 0, nkb, "whole", []))
        return out
    first, full, ga, wa, gb, wb = plan

    def start_of(w):
        if w <= ga:
            return wa * w // ga if ga else 0
        return wa + wb * (w - ga) // gb

    nfull = full if g < G else 0
    if first:
        whole_base, slot, tail_base = T - full * G, (g - ga + G) % G, 0
    else:
        whole_base, slot, tail_base = 0, g, full * G
    pos, end = (start_of(g), start_of(g + 1)) if g < ga + gb else (0, 0)
    tail = []
    while pos < end:
        tt, lo = divmod(pos, kbu)
        hi = min(kbu, lo + (end - pos))
        kind = "whole" if (lo == 0 and hi == kbu) else ("finish" if lo == 0 else "write")
        writers = []
        if kind == "finish":
            w = g + 1
            while w < ga + gb and start_of(w) < (tt + 1) * kbu:
                writers.append(w)
                w += 1
        tail.append((tail_base + tt, lo * kps, hi * kps, kind, writers))
        pos += hi - lo
    whole = [(whole_base + slot + s * G, 0, kbu * kps, "whole", []) for s in range(nfull)]
    return tail + whole if first else whole + tail


# (T tiles, G GEMM groups, L late groups, K blocks, kps)
SPLIT_CASES = [(256, 64, 0, 64, 2), (256, 68, 0, 64, 2), (256, 70, 0, 64, 2), (256, 76, 0, 64, 2),
               (7168, 72, 0, 64, 2), (7168, 75, 0, 64, 2), (3, 70, 0, 4, 1), (1, 152, 0, 1, 1), (5, 4, 0, 3, 1),
               (9, 4, 0, 7, 1), (130, 64, 0, 2, 2), (100, 152, 0, 32, 1), (64, 2, 0, 1, 1), (17, 16, 0, 5, 1),
               (33, 16, 0, 64, 2), (1, 2, 0, 8, 2), (2, 3, 0, 1, 1),
               (256, 64, 12, 64, 2), (256, 68, 8, 64, 2), (7168, 72, 4, 64, 2), (7168, 64, 12, 64, 2),
               (24, 5, 2, 8, 2), (16, 3, 1, 8, 2), (12, 5, 3, 4, 1), (20, 7, 2, 5, 1), (256, 60, 16, 16, 1)]


def all_groups(G, L, plan):
    return G + (L if plan is not None and not plan[0] else 0)


@pytest.mark.parametrize("T,G,L,nkb,kps", SPLIT_CASES)
@pytest.mark.parametrize("split", [0, 1, 3])
def test_segments_cover_every_k_block_once(T, G, L, nkb, kps, split):
    plan = plan_split(T, G, L if split == 1 else 0, nkb // kps, kps, last=split == 3) if split else None
    seen = {}
    for g in range(all_groups(G, L, plan)):
        for t, lo, hi, kind, _ in segments(g, G, T, nkb, kps, plan):
            assert 0 <= t < T and 0 <= lo < hi <= nkb and lo % kps == 0 and hi % kps == 0
            for kb in range(lo, hi):
                assert (t, kb) not in seen
                seen[(t, kb)] = g
    assert len(seen) == T * nkb


@pytest.mark.parametrize("T,G,L,nkb,kps", SPLIT_CASES)
def test_no_split_keeps_round_robin(T, G, L, nkb, kps):
    for g in range(G):
        assert [s[0] for s in segments(g, G, T, nkb, kps, None)] == list(range(g, T, G))
    if T % G == 0 and L == 0:  # whole rounds: nothing to split
        assert plan_split(T, G, L, nkb // kps, kps) is None


@pytest.mark.parametrize("T,G,L,nkb,kps", SPLIT_CASES)
@pytest.mark.parametrize("last", [False, True])
def test_split_parts_and_dependencies(T, G, L, nkb, kps, last):
    """Each group writes at most one partial, as its first tail segment (after
    which it waits for nothing a lower group holds), and finishes at most one
    split tile, as its last tail segment; a finisher's writer list is exactly
    the higher groups holding the tile's later parts, in K order."""
    plan = plan_split(T, G, 0 if last else L, nkb // kps, kps, last=last)
    if plan is None:
        return
    parts, finish = {}, {}
    for g in range(all_groups(G, L, plan)):
        seg = segments(g, G, T, nkb, kps, plan)
        kinds = [x[3] for x in seg]
        assert kinds.count("write") <= 1 and kinds.count("finish") <= 1
        if "write" in kinds:
            i = kinds.index("write")
            assert all(k == "whole" for k in kinds[:i])       # only whole tiles (no waits) before it
        if "finish" in kinds:
            i = kinds.index("finish")
            assert all(w > g for w in seg[i][4])
            if not plan[0]:
                assert i == len(seg) - 1                       # tail last: the finish is the last segment
            finish[seg[i][0]] = (g, seg[i][4])
        for t, lo, hi, kind, _ in seg:
            if kind != "whole":
                parts.setdefault(t, []).append((lo, hi, g, kind))
    for t, ps in parts.items():
        ps.sort()
        assert len(ps) >= 2
        assert ps[0][3] == "finish" and all(p[3] == "write" for p in ps[1:])
        assert [p[2] for p in ps] == sorted(p[2] for p in ps)  # later K, higher group
        assert finish[t] == (ps[0][2], [p[2] for p in ps[1:]])
        if plan[0]:
            assert len(ps) <= 3


@pytest.mark.parametrize("T,G,L,nkb,kps", [c for c in SPLIT_CASES if c[2] == 0])
def test_split_balances_work(T, G, L, nkb, kps):
    """Tail first: no group holds more than a whole round plus one share of
    the leftover tiles."""
    kbu = nkb // kps
    plan = plan_split(T, G, 0, kbu, kps)
    load = [sum(hi - lo for _, lo, hi, _, _ in segments(g, G, T, nkb, kps, plan)) // kps for g in range(G)]
    R = T % G
    share = cdiv(R * kbu, min(G, TAIL_SPLIT * R)) if R else 0
    assert max(load) <= (T // G) * kbu + share
    if R and kbu >= 2 * cdiv(R, G):  # a tile's K units can be spread: shorter than whole rounds
        assert max(load) < cdiv(T, G) * kbu


def test_late_groups_plan_for_the_headline_shape():
    """AG tp=4, 4096^3 with 24 producer CTAs (12 pairs) and 64 GEMM pairs: the
    GEMM pairs keep three whole rounds, the producer pairs take the rest of the
    last chunk's tiles after their copy, and no GEMM pair does a fourth tile."""
    T, G, L, kbu = 256, 64, 12, 32
    plan = plan_split(T, G, L, kbu)
    assert plan is not None and plan[0] == 0 and plan[1] == 3
    loads = [sum(hi - lo for _, lo, hi, _, _ in segments(g, G, T, 64, 2, plan)) // 2 for g in range(G + L)]
    assert max(loads[:G]) < 4 * kbu and min(loads[G:]) > 0


def gemm_grid(cg, want, P, tiles, max_pairs=76):
    """The host's GEMM grid: single CTAs up to the tile count, or pairs up to
    the co-resident pairs left next to the producers."""
    if cg == 1:
        return max(1, min(want, tiles))
    return 2 * max(1, min(want // 2, max_pairs - P // 2, tiles))


KB_US = 0.33


def tiles_end(pl, G, ready, nkb):
    """The host's schedule model: G CTA groups take tiles round robin in the
    kernel's order; a tile of group g starts no earlier than ready[g]; a tile
    of w strips costs nkb K blocks of KB_US x (0.91 + 0.09 w / 8) microseconds
    (measured: a K block of a 128- to 256-column tile pair costs 559 to 585 SM
    cycles, so the width hardly matters)."""
    ends = [0.0] * G
    for t in range(pl["total"]):
        grp, c, _ = tile_index(pl, t)
        w = tile_strips(pl, grp, c)[1]
        q = t % G
        ends[q] = max(ends[q], ready[grp] if ready else 0.0) + nkb * KB_US * (0.91 + 0.09 * w / MAX_TILE_STRIPS)
    return max(ends)


def gemm_grid(cg, want, P, tiles, max_pairs=76):
    """The host's GEMM grid: single CTAs up to the tile count, or pairs up to
    the co-resident pairs left next to the producers."""
    if cg == 1:
        return max(1, min(want, tiles))
    return 2 * max(1, min(want // 2, max_pairs - P // 2, tiles))


def producer_choice(tp, rows, k, m, elem=2, cg=2, num_sms=152):
    """The host's producer count of an overlapped AG launch (fewest column
    tiles): the fewest producers whose modelled end is within 0.5 % of the
    best, the end being the later of the GEMM's and the copy of all chunks."""
    pl = plan("ag", tp, tp * rows, k, m, elem, 1, cg)
    tiles, nkb = pl["total"], pl["kb"]
    chunk = rows * k * elem
    ends = {}
    for P in range(cg, 33, cg):
        if P > num_sms - 2 * cg:
            break
        G = gemm_grid(cg, num_sms - P, P, tiles, num_sms // 2) // cg
        rate = min(37e9, 705e9 / P) / 1.25
        tau = chunk / (P * rate) * 1e6
        ends[P] = max(tp * tau, tiles_end(pl, G, [g * tau for g in range(tp)], nkb))
    best = min(ends.values())
    return min(q for q, e in ends.items() if e <= best * 1.005)


def packed(extra):
    """The col_split option's encoding: 4 bits of extra column tiles per group."""
    return sum(min(15, e) << (4 * g) for g, e in enumerate(extra[:16]))


def test_producer_model_choices():
    """C2 (4096^3, 4 chunks of 8 MiB): the fewest producers whose copy keeps
    ahead of 4 rounds; C5 (e4m3, 8 chunks of 16 MiB, 7168 tiles): a handful,
    since the first gathered chunk is needed only after ~12 rounds."""
    assert producer_choice(4, 1024, 4096, 4096) == 14
    assert producer_choice(8, 2048, 8192, 28672, elem=1) == 4


def test_explicit_column_plans_keep_tiles_between_one_and_eight_strips():
    """Any col_split value: every group's strips are split evenly into its
    column tiles, each 1 to 8 strips wide, adding up to the group's strips."""
    for m in (256, 264, 520, 1000, 4096):
        pl = plan("ag", 4, 4096, 512, m, 2, 1, 2)
        base = pl["base_cols"]
        top = min(pl["strips"], base + 15) - base
        for extra in ([0] * 4, [top] * 4, [1, 0, top, 2]):
            set_columns(pl, m, extra)
            for g in range(4):
                widths = [tile_strips(pl, g, c)[1] for c in range(pl["group_cols"][g])]
                assert sum(widths) == pl["strips"] and 1 <= min(widths) and max(widths) <= MAX_TILE_STRIPS
                assert max(widths) - min(widths) <= 1


def test_producer_model_properties():
    # a group never starts a tile before its chunk could have landed
    pl = plan("ag", 2, 2 * 256, 64, 256, 2, 1, 2)
    ready = [0.0, 1e6]
    assert tiles_end(pl, 1, ready, 1) >= 1e6
    # more column tiles never lose work: the tiles' strips add up to the group's
    for extra in ([0, 0], [1, 3], [2, 0]):
        set_columns(pl, 256, extra)
        for g in range(2):
            assert sum(tile_strips(pl, g, c)[1] for c in range(pl["group_cols"][g])) == pl["strips"]


AUTO_COLS_PRODUCERS = 32


def auto_columns(pl, m, gemm_groups):
    """The host's automatic column plan (col_split 0): the fewest column tiles,
    unless the launch has at most half as many tiles as GEMM CTA groups; then
    every group gets min(strips, groups // (groups x row tiles)) column tiles."""
    set_columns(pl, m)
    per_col = pl["groups"] * pl["row_tiles"]
    if per_col <= 0 or 2 * pl["total"] > gemm_groups:
        return pl
    cols = min(pl["strips"], gemm_groups // per_col)
    if cols <= pl["base_cols"]:
        return pl
    return set_columns(pl, m, [cols - pl["base_cols"]] * pl["groups"])


def auto_groups(op, cg, num_sms=152, max_pairs=76):
    g = (num_sms - AUTO_COLS_PRODUCERS if op == "ag" else num_sms) // cg
    return min(g, max_pairs) if cg == 2 else g


def test_auto_column_plan():
    """Launches of many tiles keep the fewest (C2, C5, the long-K RS); small
    launches split their columns into more, narrower tiles that still fit in
    one round: C1 (tp=2, 256^3, single-SM tiles) from 2 tiles of 8 strips to
    16 tiles of one strip."""
    for op, tp, n, k, m, elem, chunks, cg in [("ag", 4, 4096, 4096, 4096, 2, 1, 2), ("ag", 8, 16384, 8192, 28672, 1, 1, 2),
                                              ("rs", 8, 16384, 28672, 8192, 2, 1, 2), ("ar", 2, 8192, 8192, 8192, 2, 4, 2)]:
        pl = plan(op, tp, n, k, m, elem, chunks, cg)
        fewest = list(pl["group_cols"])
        assert auto_columns(pl, m, auto_groups(op, cg))["group_cols"] == fewest
    pl = auto_columns(plan("ag", 2, 256, 256, 256, 2, 1, 1), 256, auto_groups("ag", 1))
    assert pl["group_cols"] == [8, 8] and pl["total"] == 16
    for op, tp, n, k, m, elem, chunks in SHAPES:
        for cg in (1, 2):
            pl = plan(op, tp, n, k, m, elem, chunks, cg)
            fewest_total, G = pl["total"], auto_groups(op, cg)
            auto_columns(pl, m, G)
            if pl["total"] != fewest_total:          # split only launches of at most half a round
                assert 2 * fewest_total <= G and pl["total"] <= G
            for g in range(pl["groups"]):            # every tile 1..8 strips, the strips covered once
                widths = [tile_strips(pl, g, c)[1] for c in range(pl["group_cols"][g])]
                assert sum(widths) == pl["strips"] and 1 <= min(widths) and max(widths) <= MAX_TILE_STRIPS


def simulate_dynamic_claims(T, G, speeds, base=0):
    """The dynamic tile protocol on the host: each group claims its first tile,
    then, whenever it starts a tile, claims the one after it (the claim goes
    out one tile ahead); a claim at or past T ends the group.  Claims are
    served in time order from one counter starting at `base`.  Returns the
    tiles each group computed and the counter's final value."""
    import heapq
    counter = base
    tiles = [[] for _ in range(G)]
    events = [(0.0, g) for g in range(G)]   # (time the group asks for its next claim, group)
    heapq.heapify(events)
    pending = [None] * G                     # the claim a group holds for its next tile
    while events:
        now, g = heapq.heappop(events)
        if pending[g] is None:               # first claim
            pending[g] = counter - base
            counter += 1
        t = pending[g]
        if t >= T:
            continue                         # the group's one claim past the end
        tiles[g].append(t)
        pending[g] = counter - base          # the next claim, issued as this tile starts
        counter += 1
        heapq.heappush(events, (now + speeds[g], g))
    return tiles, counter


def test_dynamic_claims_cover_every_tile_once():
    """Every tile is claimed by exactly one group, each group makes exactly one
    claim past the end, so a launch advances the counter by tiles + groups
    (what the host adds to the next launch's base), whatever the groups'
    speeds; with equal speeds the claims follow the tile order."""
    import random
    rnd = random.Random(7)
    for T, G in [(1, 1), (5, 8), (64, 2), (256, 69), (2048, 76), (100, 100)]:
        speeds = [1.0 + 0.2 * rnd.random() for _ in range(G)]
        base = rnd.randrange(1 << 32)
        tiles, counter = simulate_dynamic_claims(T, G, speeds, base)
        assert sorted(t for ts in tiles for t in ts) == list(range(T))
        assert counter - base == T + G
        for ts in tiles:
            assert ts == sorted(ts)          # a group's tiles come in claim order
