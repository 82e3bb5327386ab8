"""Host-side check of the tcgen05 kernel's work split and buffer indexing.

A Python mirror of the kernel's stream-K arithmetic (cta_begin, cta_of, slot_of,
segment walk) and of its global-memory address ranges, run over the shapes the
tests and the benchmark launch: every (tile, chunk) is processed exactly once,
every bulk copy and partial-slot access stays inside its buffer, and the
split-K reducer reads exactly the slots the contributors wrote.
"""
import re
import os

import numpy as np
import pytest

from weight_only_int4_02_gb300 import inputs

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "weight_only_int4_02_gb300", "csrc")
MAX_GRID = 1024
SMS = 152


def ceil_div(a, b):
    return -(-a // b)


def tile_m_for(M):
    for t in (16, 32, 64, 128):
        if M <= t:
            return t
    return 256


# weight formats: 4-bit (also per-group zero-points and BF16 activations, same stages),
# 8-bit codes, 2:4 sparse 4-bit codes
FORMATS = ("int4", "w8", "sparse")


GEMV_MAX_M = 4


def gemv_plan(M, N, K, G, sms=SMS):
    """Mirror of make_gemv_plan: the CUDA-core kernel for one to four rows of X,
    one CTA per block of cw output columns over the whole of K."""
    mr = 1 if M <= 1 else 2 if M <= 2 else 4
    cw = 32 if ceil_div(N, 32) >= sms else 16
    blocks = ceil_div(N, cw)
    KC = ceil_div(ceil_div(K, 64), 4) * 4
    return dict(path=1, tm=mr, mr=mr, cw=cw, blocks=blocks, grid=blocks, KC=KC, ng=ceil_div(K, G),
                n_tiles=ceil_div(N, 128), rows=ceil_div(K, 32), tile_rows=2 * KC)


DECODE_MAX_M = 16
DECODE_AUTO_MAX_M = 8
DEC_STAGE_ROWS = 16
DEC_MAX_RING = 16
DEC_SMEM_BUDGET = 104 * 1024


def dec_words_in_flight(cb):
    return 24 * 1024 if cb == 16 else 80 * 1024 if cb == 80 else 64 * 1024


def decode_block_cols(N, mr, sms=SMS):
    """Mirror of decode_block_cols: with eight rows of X, the narrowest block width that
    gives more CTAs than SMs and at most two per SM; else 128, 64 or 16."""
    if mr == 8:
        for cb in (16, 32, 48, 64, 80, 128):
            if sms < ceil_div(N, cb) <= 2 * sms:
                return cb
    return 128 if ceil_div(N, 128) >= 2 * sms else 64 if ceil_div(N, 64) >= sms else 16


def decode_plan(M, N, K, G, sms=SMS):
    """Mirror of make_decode_plan and of the launch's ring sizing: the decode kernel
    for one to sixteen rows of X, one CTA per block of cb output columns over the whole
    of K."""
    mr = 8 if M <= 8 else 16
    cb = decode_block_cols(N, mr, sms)
    blocks = ceil_div(N, cb)
    KC = ceil_div(ceil_div(K, 64), 4) * 4
    rows = K // 32
    slot = DEC_STAGE_ROWS * (cb * 16 + cb * 2 + M * 64)
    ring = min(dec_words_in_flight(cb) // (DEC_STAGE_ROWS * cb * 16), DEC_SMEM_BUDGET // slot, DEC_MAX_RING)
    sh = group_shift(G)
    return dict(path=3, tm=mr, mr=mr, cb=cb, blocks=blocks, grid=blocks, KC=KC, ng=ceil_div(K, G),
                n_tiles=ceil_div(N, 128), rows=rows, tile_rows=2 * KC, stages=ceil_div(rows, DEC_STAGE_ROWS),
                slot=slot, ring=ring, smem=ring * slot + 3 * DEC_MAX_RING * 8 + 16 + 128, g_shift=sh,
                scale_rows=(DEC_STAGE_ROWS * 32 // G) if (G & (G - 1)) == 0 and G <= DEC_STAGE_ROWS * 32 else 1)


def group_shift(G):
    if G & (G - 1):
        return 30
    return G.bit_length() - 1


def dispatch(M, N, K, G, sms=SMS, fmt="int4", force=0):
    """Mirror of device_plan for the 4-bit FP16 format: path 3 (decode kernel) when
    forced or, by itself, for up to eight rows of X, where K is a multiple of 32;
    path 1 (CUDA-core kernel) only when forced; else the tensor-core plan."""
    if fmt == "int4" and M <= DECODE_MAX_M and K % 32 == 0:
        if force == 3 or (force == 0 and (M <= DECODE_AUTO_MAX_M or (N <= 4096 and K <= 4096 and N >= 16 * sms))):
            return decode_plan(M, N, K, G, sms)
    if fmt == "int4" and M <= GEMV_MAX_M and force == 1:
        return gemv_plan(M, N, K, G, sms)
    return plan(M, N, K, G, sms, fmt)


def check_decode_shape(M, N, K, G, sms=SMS):
    """Mirror of the decode kernel's indexing. In a column block every (column, row of
    32 k, word) is unpacked by exactly one lane of one warp (the stage's team for blocks
    of 16 to 80 columns; with 128 columns both teams take every stage, each its own 64),
    and the shared-memory word it reads (the kernel's own offset arithmetic: one TMA box
    per 64 columns, or per 16 for blocks of 48 and 80, which can straddle two tiles) is
    the global word of layout v2 that holds that column's codes, and the scale it reads
    that column's group scale; the X it reads lies inside X; each box stays inside one
    tile of the packed words and scales; every Y element is written once; with teams
    taking stages in turn, a slot's consecutive stages go to the same team; the ring,
    the reduction and the shared memory fit."""
    P = decode_plan(M, N, K, G, sms)
    cb, mr, rows = P["cb"], P["mr"], P["rows"]
    col_teams = cb == 128
    narrow = cb in (48, 80)
    warp_cols = 64 if col_teams else cb
    box_cols = 16 if narrow else min(cb, 64)
    box_words = DEC_STAGE_ROWS * box_cols * 4
    assert K % 32 == 0 and M <= DECODE_MAX_M
    assert 2 <= P["ring"] <= DEC_MAX_RING
    assert 8 * mr * warp_cols * 4 <= P["ring"] * DEC_STAGE_ROWS * cb * 16    # warps' sums fit the weight ring
    assert 2 * (P["smem"] + 1024) <= 228 * 1024                              # two CTAs per SM
    assert cb % box_cols == 0 and box_cols * 4 <= 256                        # TMA boxes of at most 256 words
    assert mr == 8 or not narrow
    if not col_teams:
        check_alternating_teams(P["ring"], P["stages"])

    def sb_words(sb):   # the kernel's byte offset of sub-block sb, in words
        return ((16 * sb // box_cols) * box_words * 4 + (16 * sb % box_cols) * 16) // 4

    def sb_scales(sb):
        return sb * DEC_STAGE_ROWS * 16 if narrow else 16 * sb

    # blocks 0 .. 3 and the last, every lane's reads
    for b in sorted({0, 1, 2, 3, P["blocks"] - 1} & set(range(P["blocks"]))):
        check_decode_block(P, M, N, K, b, cb, mr, rows, col_teams, narrow, warp_cols, box_cols, box_words,
                           sb_words, sb_scales)
    # every block: each box inside one tile, Y written once
    cols = set()
    for b in range(P["blocks"]):
        n0 = b * cb
        for bx in range(cb // box_cols):
            col = n0 + bx * box_cols
            assert (col & 127) + box_cols <= 128 and ((col & 127) * 4) % 4 == 0
        for c in range(cb):
            if n0 + c < N:
                assert n0 + c not in cols
                cols.add(n0 + c)
    assert len(cols) == N
    return P


def check_alternating_teams(S, stages):
    """Mirror of the consumers' slot and parity tracking with two teams taking the
    stages in turn: each team's (slot, parity) is the stage's; and a wait on a slot's
    full barrier never runs two phases ahead of the slot's earlier stage, because with
    an odd ring (where the earlier stage belongs to the other team) the team first
    waits for that stage's consumption."""
    for team in (0, 1):
        s, ph = team, 0
        for st in range(team, stages, 2):
            assert (s, ph) == (st % S, (st // S) & 1)
            if st >= S and (st - S) % 2 != team:
                assert S % 2 == 1   # only an odd ring hands a slot to the other team, and it waits
            s += 2
            if s >= S:
                s -= S
                ph ^= 1


def check_decode_block(P, M, N, K, b, cb, mr, rows, col_teams, narrow, warp_cols, box_cols, box_words, sb_words,
                       sb_scales):
    n0 = b * cb
    seen = set()
    for st in range(P["stages"]):
        teams = (0, 1) if col_teams else (st % 2,)
        g0 = min((st * DEC_STAGE_ROWS * 32) >> P["g_shift"], P["ng"] - 1)
        for team in teams:
            cbase = 64 * team if col_teams else 0
            for wl in range(4):
                for rr in range(4):
                    rl = 4 * wl + rr
                    row = st * DEC_STAGE_ROWS + rl
                    if row >= rows:
                        continue
                    gl = min((row * 32) >> P["g_shift"], P["ng"] - 1) - g0
                    assert 0 <= gl < P["scale_rows"]
                    for lane in range(32):
                        g, t = lane >> 2, lane & 3
                        for h in range(mr // 8):
                            m = min(8 * h + g, M - 1)
                            assert 0 <= m < M and row * 32 + 8 * t + 7 < K
                        # the kernel's word offset: the warp's box, its row and lane, then the sub-block
                        woff = ((cbase // box_cols) * box_words + (4 * wl * box_cols + cbase % box_cols + g) * 4 + t
                                + rr * box_cols * 4)
                        sc0 = (gl * 16 if narrow else gl * cb + cbase) + g
                        for sb in range(warp_cols // 16):
                            for off in (0, 8):
                                smem_word = woff + sb_words(sb) + off * 4
                                assert smem_word < DEC_STAGE_ROWS * cb * 4
                                nl = cbase + 16 * sb + g + off          # the column this lane stands for
                                key = (nl, row, t)
                                assert key not in seen
                                seen.add(key)
                                # box bx holds [16 rows][box_cols][4 words] from map row
                                # (col >> 7) * tile_rows + st * 16, word (col & 127) * 4 on
                                bx, within = divmod(smem_word, box_words)
                                box_row, box_word = divmod(within, box_cols * 4)
                                col = n0 + bx * box_cols
                                gcol = (col >> 7) * 128 + (col & 127) + box_word // 4
                                assert gcol == n0 + nl and box_word % 4 == t
                                map_row = st * DEC_STAGE_ROWS + box_row              # within the tile
                                assert map_row == row
                                kc, jj = divmod(map_row, 2)
                                # layout v2: word (kc, jj, n_in, wd) holds k = 64 kc + 32 jj + 8 wd .. +7
                                assert 64 * kc + 32 * jj + 8 * t == row * 32 + 8 * t
                                # the scale: [scale_rows][cb] or, with 16-column boxes,
                                # [cb / 16][16 rows][16] from scale row (col >> 7) * ng + g0
                                si = sc0 + sb_scales(sb) + off
                                assert si < DEC_STAGE_ROWS * cb
                                if narrow:
                                    sbx, sw = divmod(si, DEC_STAGE_ROWS * 16)
                                    srow, scol = divmod(sw, 16)
                                    assert n0 + sbx * 16 + scol == n0 + nl and srow == gl
                                else:
                                    srow, scol = divmod(si, cb)
                                    assert scol == nl and srow == gl
    assert len(seen) == cb * rows * 4


def check_gemv_shape(M, N, K, G, sms=SMS):
    """Every (output column, row of 32 k) is read by exactly one thread of one CTA,
    every packed unit and scale it reads lies inside its buffer and holds that
    column's codes, and no two threads write the same Y element."""
    P = gemv_plan(M, N, K, G, sms)
    cw = P["cw"]
    cpt = cw // 8
    units = P["n_tiles"] * P["tile_rows"] * 128
    scales = P["n_tiles"] * P["ng"] * 128
    seen = set()
    writes = set()
    assert 128 % cw == 0                     # a block never straddles a tile
    for b in range(P["blocks"]):             # one CTA per block (grid = blocks)
        for warp in range(8):
            for lane in range(32):
                n0 = b * cw + (lane & 7)
                nt, n_in0 = n0 >> 7, n0 & 127
                r = warp * 4 + (lane >> 3)
                while r < P["rows"]:
                    g = min((r * 32) // G, P["ng"] - 1)
                    for j in range(cpt):
                        n, n_in = n0 + 8 * j, n_in0 + 8 * j
                        assert n >> 7 == nt
                        u = (nt * P["tile_rows"] + r) * 128 + n_in
                        assert 0 <= u < units
                        assert 0 <= (nt * P["ng"] + g) * 128 + n_in < scales
                        # the unit holds k = 32r .. 32r+31 of column n (layout v2: kc = r // 2, j = r % 2)
                        kc, jj = divmod(r, 2)
                        assert u * 4 == (((nt * P["KC"] + kc) * 2 + jj) * 128 + n_in) * 4
                        if n < N:
                            assert (n, r) not in seen
                            seen.add((n, r))
                    r += 32
        for t in range(min(256, P["mr"] * cw)):
            m, c = divmod(t, cw)
            if m < M and b * cw + c < N:
                assert (m, b * cw + c) not in writes
                writes.add((m, b * cw + c))
    assert len(seen) == N * P["rows"]
    assert len(writes) == M * N
    return P


def plan(M, N, K, G, sms=SMS, fmt="int4"):
    tm = tile_m_for(M)
    if fmt == "sparse":
        tm = min(tm, 128)
    ksub = 2 if fmt in ("w8", "sparse") else (4 if tm <= 64 else 2)
    xblocks = 4 if fmt == "sparse" else ksub
    m_tiles, n_tiles, ng = ceil_div(M, tm), ceil_div(N, 128), ceil_div(K, G)
    KC = ceil_div(ceil_div(K, 64), 4) * 4
    iters = KC // xblocks
    total = n_tiles * m_tiles * iters
    units = min(sms, MAX_GRID)           # one work unit per CTA; every CTA loads its own X
    work_tiles = n_tiles * m_tiles
    if work_tiles < units:
        # tile-aligned split: s parts per tile, chosen by the measured cost model
        ring, pre_us, str_us, fix_us, row_us = ((8.0, 0.15, 0.40, 1.4, 0.006) if tm <= 32 else
                                                (0.0, 0.525, 0.525, 2.6, 0.008) if tm == 64 else
                                                (0.0, 0.375, 0.375, 2.9, 0.006) if tm == 128 else
                                                (0.0, 0.70, 0.70, 3.0, 0.0043))
        rows = M if m_tiles == 1 else tm
        best_s, best = 1, 0.0
        s = 1
        while s <= units // work_tiles and s <= iters:
            n = float((iters + s - 1) // s)
            pre = n if n < ring else ring
            cost = pre * pre_us + (n - pre) * str_us + ((fix_us + row_us * rows * float(s - 1)) if s > 1 else 0.0)
            if s == 1 or cost < best:
                best, best_s = cost, s
            s += 1
        units = work_tiles * best_s
        sk_tiles = work_tiles
    else:
        min_iters = max(4, iters // 2 if tm >= 64 else (iters // 4 if tm == 32 else 0))
        units = max(1, min(units, -(-total // min_iters)))
        sk_tiles = work_tiles % units    # tiles past the last whole wave: split, run first
        if 0 < sk_tiles and 2 * sk_tiles < units:
            sk_tiles += units            # at least half a wave: about two contributors a tile
        if fmt == "sparse" and tm >= 128:
            sk_tiles = work_tiles        # 2:4 sparse codes on 128-row tiles: stream-K over every tile
    units = max(1, units)
    return dict(path=2, tm=tm, ksub=ksub, xblocks=xblocks, fmt=fmt, m_tiles=m_tiles, n_tiles=n_tiles,
                KC=KC, iters=iters, ng=ng, total=total, sk_tiles=sk_tiles, sk_iters=sk_tiles * iters, grid=units)


def cta_begin(P, c):
    return c * P["sk_iters"] // P["grid"]


def cta_of(P, i):
    c = (i * P["grid"]) // P["sk_iters"]
    while c + 1 < P["grid"] and cta_begin(P, c + 1) <= i:
        c += 1
    while c > 0 and cta_begin(P, c) > i:
        c -= 1
    return c


def slot_of(P, c, t):
    return 2 * c if cta_begin(P, c) >= t * P["iters"] else 2 * c + 1


def segments(P, c):
    """Mirror of work_begin / work_next: the CTA's range of the split region, then its
    whole tiles sk_tiles + c, + grid, ..."""
    i, end = cta_begin(P, c), cta_begin(P, c + 1)
    while i < end:
        t = i // P["iters"]
        kb = i - t * P["iters"]
        ke = min(P["iters"], kb + (end - i))
        yield t, kb, ke
        i += ke - kb
    t = P["sk_tiles"] + c
    while t < P["n_tiles"] * P["m_tiles"]:
        yield t, 0, P["iters"]
        t += P["grid"]


def check_shape(M, N, K, G, sms=SMS, fmt="int4"):
    """Every (weight tile, stage) is computed once; every global access of the
    producers, the partial slots and the counters stays inside its buffer; the
    reducer of a split tile reads exactly the slots its contributors wrote."""
    P = plan(M, N, K, G, sms, fmt)
    KC, ng, tm, ks, iters = P["KC"], P["ng"], P["tm"], P["ksub"], P["iters"]
    # packed words per (tile, sub-chunk) and sub-chunks per column, per format
    chunk_words = {"int4": 1024, "w8": 2048, "sparse": 1536}[fmt]
    sub_k = 128 if fmt == "sparse" else 64
    KCp = KC * 64 // sub_k
    packed_words = P["n_tiles"] * KCp * chunk_words
    scales_elems = P["n_tiles"] * ng * 128
    partial_floats = 2 * P["grid"] * tm * 128
    assert P["grid"] <= MAX_GRID
    covered = {}
    writers = {}
    for c in range(P["grid"]):
        for (t, kb, ke) in segments(P, c):
            assert 0 <= t < P["n_tiles"] * P["m_tiles"] and 0 <= kb < ke <= iters
            nt, mt = divmod(t, P["m_tiles"])
            for st in range(kb, ke):
                k0 = st * ks * sub_k
                key = (nt, mt, st)
                assert key not in covered
                covered[key] = c
                w0 = (nt * KCp + st * ks) * chunk_words    # one bulk copy of ks sub-chunks
                assert 0 <= w0 and w0 + ks * chunk_words <= packed_words
                assert (w0 * 4) % 16 == 0                  # bulk-copy source alignment
                g0 = min(k0 // G, ng - 1)
                g1 = min((k0 + ks * sub_k - 1) // G, ng - 1)
                assert 1 <= g1 - g0 + 1 <= ks * sub_k // 32  # fits the scale slot
                e0 = (nt * ng + g0) * 128
                assert e0 >= 0 and e0 + (g1 - g0 + 1) * 128 <= scales_elems
                for j in range(P["xblocks"]):
                    assert ((k0 + j * 64) * 2) % 16 == 0    # TMA inner coordinate, 16-byte aligned
                assert mt * tm < M
            split = kb != 0 or ke != iters
            if split:
                slot = slot_of(P, c, t)
                assert 0 <= slot < 2 * P["grid"]
                assert (slot + 1) * tm * 128 <= partial_floats
                writers.setdefault(t, []).append((c, slot))
    assert len(covered) == P["n_tiles"] * P["m_tiles"] * iters
    counter_ids = set()
    for t, ws in writers.items():
        c_lo, c_hi = cta_of(P, t * iters), cta_of(P, t * iters + iters - 1)
        counter = c_lo
        assert counter < P["grid"] and counter not in counter_ids
        counter_ids.add(counter)
        read = [(cc, slot_of(P, cc, t)) for cc in range(c_lo, c_hi + 1)]
        assert sorted(read) == sorted(ws), (t, read, ws)
        assert len(set(s for _, s in ws)) == len(ws)
    # a slot is written by one tile only
    all_slots = [s for ws in writers.values() for _, s in ws]
    assert len(all_slots) == len(set(all_slots))
    return P


SHAPES = sorted(set(
    [(m, n, k, 128) for (m, k, n) in inputs.WORKLOADS["llama2_7b_decode_sweep"]["cases"]]
    + [(m, n, k, 128) for (m, k, n) in inputs.WORKLOADS["llama2_13b_prefill"]["cases"]]
    + [(m, n, k, 128) for (m, k, n) in inputs.WORKLOADS["large_layer_18432x73728"]["cases"]]
    + [(16, 4096, 4096, 128)]
    + [(m, 4096, 4096, g) for m in inputs.EDGE_M for g in (32, 4096)]
    + [(m, 256, 16384, 128) for m in inputs.EDGE_M]
    + [(m, 4096, k, 128) for m in inputs.EDGE_M for k in (4000, 4040)]
    + [(1, 8, 8, 8), (1, 128, 64, 64), (3, 136, 200, 200), (300, 264, 136, 32), (1, 8, 4040, 4040)]
    # a few tiles past the last whole wave, with too few stages for every CTA
    + [(1, 20008, 2048, 64), (1, 19464, 512, 128), (40, 19592, 1024, 32)]))


@pytest.mark.parametrize("M,N,K,G", SHAPES)
def test_schedule_covers_once_and_stays_in_bounds(M, N, K, G):
    check_shape(M, N, K, G)


GEMV_SHAPES = sorted(set((m, n, k, g) for (m, n, k, g) in SHAPES if m <= GEMV_MAX_M and n * k <= 12288 * 4096)
                     | {(2, 8192, 4096, 128), (4, 4096, 11008, 128), (3, 1032, 4040, 32), (2, 8, 8, 8)})


@pytest.mark.parametrize("M,N,K,G", GEMV_SHAPES)
def test_gemv_schedule_covers_once_and_stays_in_bounds(M, N, K, G):
    check_gemv_shape(M, N, K, G)


def test_gemv_column_block_widths():
    """Blocks of 32 columns when that still gives one block per SM, else 16: 16
    for the 4096-wide layers, 32 for 8192 and wider."""
    assert gemv_plan(1, 4096, 4096, 128)["cw"] == 16
    assert gemv_plan(1, 4864, 4096, 128)["cw"] == 32
    assert gemv_plan(1, 8192, 4096, 128)["cw"] == 32
    assert gemv_plan(1, 12288, 4096, 128)["cw"] == 32
    assert gemv_plan(4, 22016, 4096, 128)["cw"] == 32
    assert gemv_plan(3, 4096, 4096, 128)["mr"] == 4 and gemv_plan(2, 4096, 4096, 128)["mr"] == 2
    assert dispatch(4, 12288, 4096, 128, force=1)["path"] == 1
    assert dispatch(5, 4096, 4096, 128, force=1)["path"] == 2


DECODE_SHAPES = sorted(set((m, n, k, g) for (m, n, k, g) in SHAPES if m <= DECODE_MAX_M and k % 32 == 0
                           and n * k <= 22016 * 4096)
                       | {(1, 73728, 18432, 128), (8, 73728, 18432, 128), (16, 73728, 18432, 128), (16, 12288, 4096, 128),
                          (9, 1024, 2048, 64), (2, 264, 544, 32), (13, 4104, 1024, 128), (1, 4096, 4000, 4000),
                          (1, 20008, 2048, 64), (8, 19464, 1024, 128), (3, 12296, 1024, 32), (5, 24320, 512, 512),
                          (2, 7304, 2048, 128)})


@pytest.mark.parametrize("M,N,K,G", DECODE_SHAPES)
def test_decode_schedule_covers_once_and_stays_in_bounds(M, N, K, G):
    check_decode_shape(M, N, K, G)


def random_decode_shapes(n, seed):
    """Seeded random shapes of the decode kernel: 1..16 rows of X, N a multiple of 8,
    K a multiple of 32, groups of 32, 64, 128 or K (the block width, the ring depth and
    its parity follow from them)."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.integers(1, 17))
        N = 8 * int(rng.integers(1, 3500))
        K = 32 * int(rng.integers(1, 200))
        G = int(rng.choice([32, 64, 128, K]))
        out.append((M, N, K, G))
    return out


@pytest.mark.parametrize("M,N,K,G", random_decode_shapes(60, 2026))
def test_decode_schedule_random_shapes(M, N, K, G):
    check_decode_shape(M, N, K, G)



def test_dispatch_rule():
    """The automatic choice for the 4-bit FP16 format: the decode kernel (path 3) for
    up to eight rows of X where K is a multiple of 32 (sixteen on layers of at most
    4096 x 4096 with a 16-column block per SM), the tensor-core kernel otherwise; blocks
    of 128 columns for the 73728-wide layer (576 blocks, two per SM and more), 48 for
    the 12288-wide one, 80 for the 22016-wide one, 16 for the 4096-wide ones
    (measured on GB300)."""
    width = {4096: 16, 12288: 48, 22016: 80, 73728: 128}
    for (N, K) in [(4096, 4096), (12288, 4096), (22016, 4096), (4096, 11008), (73728, 18432)]:
        for M in (1, 2, 4, 8):
            P = dispatch(M, N, K, 128)
            assert P["path"] == 3 and P["tm"] == 8
            assert P["cb"] == width[N]
        # nine to sixteen rows: the decode kernel on the 4096 x 4096 layer, the tensor-core kernel elsewhere
        assert dispatch(9, N, K, 128)["path"] == (3 if (N, K) == (4096, 4096) else 2)
        assert dispatch(16, N, K, 128)["path"] == (3 if (N, K) == (4096, 4096) else 2)
        assert dispatch(16, N, K, 128, force=3)["path"] == 3 and dispatch(16, N, K, 128, force=3)["tm"] == 16
        assert dispatch(17, N, K, 128, force=3)["path"] == 2
        assert dispatch(1, N, K, 128, force=2)["path"] == 2
    assert dispatch(1, 4096, 4040, 128)["path"] == 2          # K not a multiple of 32
    assert dispatch(16, 2048, 4096, 128)["path"] == 2          # fewer 16-column blocks than SMs
    assert dispatch(17, 4096, 4096, 128)["path"] == 2
    assert dispatch(4, 4096, 4096, 128, fmt="w8")["tm"] == 16
    assert dispatch(1, 4096, 4096, 128, force=2)["tm"] == 16
    # ring depth: about 64 KB of packed words in flight, fewer where shared memory says so
    assert decode_plan(1, 4096, 4096, 128)["ring"] == 6 and decode_plan(1, 73728, 18432, 128)["ring"] == 2
    assert decode_plan(1, 22016, 4096, 128)["ring"] == 4 and decode_plan(8, 22016, 4096, 128)["ring"] == 3
    assert decode_plan(1, 12288, 4096, 128)["ring"] == 5 and decode_plan(16, 22016, 4096, 128)["ring"] == 3


@pytest.mark.parametrize("fmt", ["w8", "sparse"])
@pytest.mark.parametrize("M,N,K,G", [s for s in SHAPES if s[0] <= 1024])
def test_schedule_of_other_weight_formats(M, N, K, G, fmt):
    check_shape(M, N, K, G, fmt=fmt)


@pytest.mark.parametrize("sms", [1, 7, 148, 160])
def test_schedule_other_sm_counts(sms):
    for shp in [(16, 4096, 4096, 128), (1, 256, 16384, 128), (4096, 5120, 13824, 128), (3, 136, 200, 200)]:
        check_shape(*shp, sms=sms)


def _constexpr(src, name):
    m = re.search(r"constexpr int %s = ([^;]+);" % name, src)
    return m.group(1)


def tc_cfg(tm, ks, fmt):
    """Mirror of TcCfg<TM, KSUB, FMT> (fmt: int4, zp, bf16, w8, sparse)."""
    sp, w8, zp = fmt == "sparse", fmt == "w8", fmt == "zp"
    sub_k = 128 if sp else 64
    stage_k = ks * sub_k
    xblocks = stage_k // 64
    xblock = tm * 128
    xbytes = xblocks * xblock
    pk = ks * (8192 if w8 else 6144 if sp else 4096)
    sc = (stage_k // 32) * 256
    zpb = (stage_k // 32) * 64 if zp else 0
    SW = (4 if tm >= 128 else 8) if (w8 or sp) else (2 if tm == 256 else 8 if (tm <= 32 or ks == 2) else 6)
    SX = min(8, (220 * 1024 - SW * (pk + sc + zpb)) // xbytes)
    dbufs = 2 if tm <= 128 else 1
    slot = ks * 32 + (ks * 4 * 8 if sp else 0)
    A = 4 if (512 - dbufs * tm) // slot >= 4 else 2
    off_pk = SX * xbytes
    off_sc = off_pk + SW * pk
    off_zp = off_sc + SW * sc
    off_bar = off_zp + SW * zpb
    nbars = 2 * SW + 2 * SX + 2 * A + 4 + 1
    smem = off_bar + nbars * 8 + 64 + 1024
    return dict(SW=SW, SX=SX, A=A, slot=slot, dbufs=dbufs, xblock=xblock, off_pk=off_pk, off_sc=off_sc,
                off_zp=off_zp, off_bar=off_bar, smem=smem, dcol=A * slot, threads=32 * (4 + 4 * ks + 3))


CONFIGS = ([(tm, ks, f) for (tm, ks) in ((16, 4), (32, 4), (64, 4), (128, 2), (256, 2)) for f in ("int4", "zp", "bf16")]
           + [(tm, 2, "w8") for tm in (16, 32, 64, 128, 256)] + [(tm, 2, "sparse") for tm in (16, 32, 64, 128)])


@pytest.mark.parametrize("tm,ks,fmt", CONFIGS)
def test_shared_memory_and_tmem_layout_fits(tm, ks, fmt):
    """Mirror of TcCfg for every instantiated kernel: stage rings, barriers,
    alignment, TMEM columns, threads."""
    src = open(os.path.join(CSRC, "gemm_tc.cuh")).read()
    assert _constexpr(src, "kChunkBytes") == "4096" and _constexpr(src, "kKPad") == "4"
    c = tc_cfg(tm, ks, fmt)
    assert c["SW"] % 2 == 0 and c["A"] % 2 == 0                     # rings shared by two teams in turn
    assert c["SW"] >= 2 and c["SX"] >= 2 and c["A"] >= 2, c
    assert c["smem"] <= 227 * 1024, c
    assert c["xblock"] % 1024 == 0                                  # 128-byte swizzle atoms
    assert c["off_pk"] % 16 == 0 and c["off_sc"] % 16 == 0 and c["off_zp"] % 16 == 0 and c["off_bar"] % 8 == 0
    assert c["dcol"] + c["dbufs"] * tm <= 512
    assert c["threads"] <= 1024


def test_layout_mirror_matches_the_compiled_sizes():
    """Shared-memory bytes of a few configurations as the compiled TcCfg reports them."""
    assert tc_cfg(16, 4, "int4")["smem"] == 214408
    assert tc_cfg(64, 4, "int4")["smem"] == 210200
    assert tc_cfg(128, 2, "int4")["smem"] == 206184
    assert tc_cfg(256, 2, "int4")["smem"] == 216312
    assert tc_cfg(16, 2, "w8")["smem"] == 173480
    assert tc_cfg(256, 2, "w8")["smem"] == 201992
    assert tc_cfg(16, 2, "sparse")["smem"] == 181640
    assert tc_cfg(128, 2, "sparse")["smem"] == 189672


def test_small_layer_splits_are_tile_aligned():
    """With fewer tiles than SMs, every tile has the same number of contributors
    and unit boundaries fall on tile boundaries; the cost model's splits of the
    decode layers (measured against the alternatives on GB300): quarters for
    4096x4096 and 4096x11008 from M = 1 to 128, whole tiles for 12288x4096; for
    the 256-row prefill tiles at M = 256, whole tiles of the 15360-wide layer and
    thirds of the 5120-wide ones (36.5 -> 23.4 us on 256x5120x5120)."""
    expect = {(1, 4096, 4096): 4, (8, 4096, 4096): 4, (16, 4096, 4096): 4, (32, 4096, 4096): 4,
              (1, 12288, 4096): 1, (16, 12288, 4096): 1, (1, 4096, 11008): 4, (16, 4096, 11008): 4,
              (32, 4096, 11008): 4, (64, 4096, 4096): 4, (64, 12288, 4096): 1, (64, 4096, 11008): 4,
              (128, 4096, 4096): 4, (128, 12288, 4096): 1, (128, 4096, 11008): 4,
              (256, 15360, 5120): 1, (256, 5120, 5120): 3, (256, 5120, 13824): 3, (512, 5120, 5120): 1}
    for (M, N, K), s in expect.items():
        P = plan(M, N, K, 128)
        work_tiles = P["n_tiles"] * P["m_tiles"]
        assert P["grid"] == work_tiles * s, (M, N, K, P["grid"])
        for t in range(work_tiles):
            assert cta_begin(P, t * s) == t * P["iters"]


def test_no_alloc_scratch_admission():
    """The fixed 8 MiB scratch of the no-allocation entry point holds the error word,
    the counters and two FP32 partial slots per CTA of the plan: on 152 SMs every
    decode layer fits up to M = 32; at M = 64 only the 12288-wide layer (whole tiles,
    no split); at M = 128 none (the rejected shapes return a workspace error)."""
    limit, partials_off = 8 << 20, 256 + 4 * MAX_GRID

    def need(M, N, K):
        P = plan(M, N, K, 128)
        return partials_off + 2 * P["grid"] * P["tm"] * 128 * 4

    layers = sorted(set((n, k) for (_, k, n) in inputs.WORKLOADS["llama2_7b_decode_sweep"]["cases"]))
    for M in (1, 16, 32, 64, 128):
        for (N, K) in layers:
            fits = need(M, N, K) <= limit
            assert fits == (M <= 32 or (M == 64 and N == 12288)), (M, N, K, need(M, N, K))
    assert need(64, 4096, 4096) == limit + partials_off
    assert need(128, 22016, 4096) > limit and need(16, 4096, 4096) <= limit


def test_split_region_runs_first_and_whole_tiles_close_every_cta():
    """With at least as many tiles as CTAs, the tiles past the last whole wave form the
    split region: every CTA takes an equal share of its stages first, then the same
    number of whole tiles, round-robin, so that the launch ends on whole tiles (direct
    stores) and every partial and fix-up comes before a CTA's whole tiles."""
    for (M, N, K) in [(16, 22016, 4096), (128, 22016, 4096), (16, 73728, 18432), (128, 73728, 18432),
                      (1024, 15360, 5120), (4096, 27648, 5120), (256, 19456, 4096)]:
        P = plan(M, N, K, 128)
        T = P["n_tiles"] * P["m_tiles"]
        assert T >= P["grid"]
        rest = T % P["grid"]
        assert P["sk_tiles"] == (rest + P["grid"] if 0 < 2 * rest < P["grid"] else rest)
        assert P["sk_tiles"] == 0 or P["sk_iters"] >= P["grid"] * P["iters"] // 2   # about two contributors a tile
        whole = (T - P["sk_tiles"]) // P["grid"]
        for c in range(P["grid"]):
            segs = list(segments(P, c))
            full = [s for s in segs if s[1] == 0 and s[2] == P["iters"] and s[0] >= P["sk_tiles"]]
            assert len(full) == whole
            assert segs[len(segs) - len(full):] == full          # whole tiles last
            assert all(t < P["sk_tiles"] for (t, kb, ke) in segs[:len(segs) - len(full)])


def random_tc_shapes(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.choice([1, 3, 16, 17, 40, 64, 100, 128, 200, 256, 300, 1024]))
        N = int(rng.integers(1, 400)) * 8 * int(rng.choice([1, 8, 16]))
        K = int(rng.integers(1, 200)) * 8 * int(rng.choice([1, 4, 16]))
        G = int(rng.choice([32, 64, 128, -1]))
        out.append((M, N, K, K if G == -1 else G))
    return out


@pytest.mark.parametrize("M,N,K,G", random_tc_shapes(80, 7))
def test_schedule_random_shapes(M, N, K, G):
    """Random shapes through the tensor-core kernel's schedule mirror: covered once,
    in bounds, every split tile's reducer reading exactly its writers' slots."""
    if K % G or K < 8 or N < 8:
        pytest.skip("shape outside the entry points' rules")
    check_shape(M, N, K, G)
