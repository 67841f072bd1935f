"""The two-pass prefill's index arithmetic, restated and checked on the CPU.

``gla_chunk_split.cu`` stages the state tile of every chunk c >= 1 inside that
chunk's own output rows (the state pass writes it, the output pass reads it
back before it overwrites those rows), walks (sequence, head, chunk, value
slice) tiles over persistent CTAs, and aligns chunks to the end of each
sequence.  This file restates those formulas -- chunk geometry, staging row
block and column, the output rows of a tile, the tile walk for dense and
packed batches in each of the three launch modes -- and checks, for dense and
packed batches with empty and short sequences, every head size, bf16 and fp32
outputs and the reversed output order:

* the bytes the output pass loads for a tile's state tile are exactly the
  bytes the state pass wrote for that chunk, slice by slice;
* those bytes lie inside the tile's own output bytes (so the output overwrites
  them, and no other tile's output touches them);
* every output element is written by exactly one tile;
* the tile walk hands out every tile exactly once over the CTAs;
* the block-floating-point encoding of a tile row round-trips within its
  stated bound, and its exponent survives in the mantissas' low bits.
"""
import numpy as np
import pytest

C = 128


def geometry(length):
    nch = (length + C - 1) // C
    return nch, length - C * nch  # chunk count, offset of chunk 0 (<= 0)


def block_row(start, length, off, c, reversed_):
    t0 = off + c * C
    return start + length - C - t0 if reversed_ else start + t0


def stage_col(j, dvs, osz):
    return (osz // 2) * dvs * (j // dvs) + (j % dvs)


def tile_walk(B, H, T, cu, nsl, mode, grid):
    """Yield, per CTA, its tiles (s, c, h, sl) in order -- the kernel's walk."""
    per = H * nsl

    def crange(nch):
        c0 = 1 if mode == 2 else 0
        c1 = min(nch, 1) if mode == 1 else nch
        return c0, max(c1, c0)

    out = {}
    for cta in range(grid):
        tiles = []
        idx = cta
        seq, base = 0, 0
        while True:
            if cu is None:
                nch, _ = geometry(T)
                c0, c1 = crange(nch)
                per_c = per * B
                if idx >= per_c * (c1 - c0):
                    break
                c = c0 + idx // per_c
                rem = idx % per_c
                tiles.append((rem // per, c, (rem // nsl) % H, rem % nsl))
            else:
                found = False
                while seq < B:
                    a, b = cu[seq], cu[seq + 1]
                    nch, _ = geometry(b - a)
                    c0, c1 = crange(nch)
                    n = per * (c1 - c0)
                    if idx < base + n:
                        local = idx - base
                        tiles.append((seq, c0 + local // per, (local // nsl) % H, local % nsl))
                        found = True
                        break
                    base += n
                    seq += 1
                if not found:
                    break
            idx += grid
        out[cta] = tiles
    return out


def check_layout(lengths, H, dk, dv, osz, reversed_, packed):
    B = len(lengths)
    if packed:
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(int)
        T = int(cu[-1])
        starts = cu[:-1]
    else:
        assert len(set(lengths)) == 1
        T = lengths[0]
        cu = None
        starts = [s * T for s in range(B)]
    rows = T if packed else B * T
    dvs = 128 if dv == 128 else 64
    nsl = dv // dvs
    seg = dv * osz  # bytes of one (row, head) segment
    # state pass: the bytes written per (s, h, c >= 1)
    staged = {}
    for s in range(B):
        length = lengths[s]
        nch, off = geometry(length)
        for h in range(H):
            for sl_s in range(dv // 64):
                col0 = stage_col(64 * sl_s, dvs, osz)
                for c in range(nch - 1):
                    brow = block_row(starts[s], length, off, c + 1, reversed_)
                    for i in range(dk):
                        row = brow + i
                        assert 0 <= row < rows
                        lo = (row * H + h) * seg + 2 * col0
                        staged.setdefault((s, h, c + 1, sl_s * 64 // dvs), set()).update(
                            range(lo, lo + 128))
    written = np.zeros(rows * H * seg, dtype=np.int32)
    grid = 7
    walks = {m: tile_walk(B, H, T, None if cu is None else list(cu), nsl, m, grid)
             for m in (0, 1, 2)}
    all_tiles = [t for tl in walks[0].values() for t in tl]
    assert len(all_tiles) == len(set(all_tiles))
    expect = {(s, c, h, sl) for s in range(B) for c in range(geometry(lengths[s])[0])
              for h in range(H) for sl in range(nsl)}
    assert set(all_tiles) == expect
    m12 = [t for m in (1, 2) for tl in walks[m].values() for t in tl]
    assert sorted(m12) == sorted(all_tiles)
    assert all(t[1] == 0 for tl in walks[1].values() for t in tl)
    for (s, c, h, sl) in all_tiles:
        length = lengths[s]
        nch, off = geometry(length)
        pad = -off if c == 0 else 0
        out_bytes = set()
        for r in range(pad, C):
            tok = off + c * C + r
            assert 0 <= tok < length
            row = starts[s] + (length - 1 - tok if reversed_ else tok)
            lo = (row * H + h) * seg + sl * dvs * osz
            written[lo:lo + dvs * osz] += 1
            out_bytes.update(range(lo, lo + dvs * osz))
        if c >= 1:
            # the output pass's loads of the staged tile
            brow = block_row(starts[s], length, off, c, reversed_)
            x0 = (osz // 2) * dvs * sl
            loads = set()
            for pn in range(dvs // 64):
                for i in range(dk):
                    lo = ((brow + i) * H + h) * seg + 2 * (x0 + 64 * pn)
                    loads.update(range(lo, lo + 128))
            assert loads == staged[(s, h, c, sl)]
            assert loads <= out_bytes
    # every output element written exactly once (the bf16 / fp32 element bytes)
    assert np.all(written == 1)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (96, 192), (128, 64), (64, 128)])
@pytest.mark.parametrize("osz", [2, 4])
@pytest.mark.parametrize("reversed_", [False, True])
def test_dense_layout(dk, dv, osz, reversed_):
    for T in (1, 127, 128, 129, 300):
        check_layout([T, T], 2, dk, dv, osz, reversed_, packed=False)


@pytest.mark.parametrize("dk,dv", [(128, 128), (96, 192)])
@pytest.mark.parametrize("osz", [2, 4])
@pytest.mark.parametrize("reversed_", [False, True])
def test_packed_layout(dk, dv, osz, reversed_):
    check_layout([300, 0, 1, 129, 128, 5, 513], 2, dk, dv, osz, reversed_, packed=True)


def encode_row(x):
    """Block floating point of one 64-value tile row, as the state pass writes it."""
    x = np.asarray(x, np.float32)
    mx = np.float32(np.max(np.abs(x)))
    field = (mx.view(np.uint32) >> 23) & 0xFF
    E = int(min(max(int(field) - 126, -100), 127))
    up = np.float32(2.0 ** (14 - E))
    m = np.rint(x * up).astype(np.int64)
    assert np.all(np.abs(m) <= 1 << 14)
    bits = ((E + 128) >> np.arange(8)) & 1
    m[:8] = (m[:8] & ~1) | bits
    return m.astype(np.int16), E


def decode_row(m):
    m = m.astype(np.int64)
    E = int(np.sum((m[:8] & 1) << np.arange(8))) - 128
    return (m * 2.0 ** (E - 14)).astype(np.float32), E


def test_block_floating_point_round_trip():
    rng = np.random.default_rng(0)
    for scale in (1e-30, 1e-5, 1.0, 3e4, 1e20):
        for _ in range(50):
            x = (rng.standard_normal(64) * scale).astype(np.float32)
            m, E = encode_row(x)
            y, E2 = decode_row(m)
            assert E2 == E
            mx = float(np.max(np.abs(x)))
            assert mx < 2.0 ** E
            # rounding (half a unit) plus the replaced low bit (one unit)
            assert np.max(np.abs(y - x)) <= 1.5 * 2.0 ** (E - 14) * (1 + 1e-6)
            assert np.max(np.abs(y - x)) <= 2.0 ** -13 * mx * 2 + 1e-38
    # a zero row takes the smallest exponent; the exponent's bits in the low
    # mantissa bits then decode to at most one unit, 2^-114
    x = np.zeros(64, np.float32)
    y, E = decode_row(encode_row(x)[0])
    assert E == -100 and np.max(np.abs(y)) <= 2.0 ** -114
