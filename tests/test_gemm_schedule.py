"""The prefill GEMM's split-region schedule, on the CPU: the invariants its
split-tile hand-off relies on, checked over the layer shapes and the GPU
tests' shapes on a 152-SM grid (and on smaller grids).

The host picks the schedule (whole tiles in full waves, the rest cut by K into
one contiguous chunk range per CTA); each CTA walks its range's items in
order.  The hand-off needs:
  - a split tile's first part (chunk 0 on) is the final item of its CTA, so
    that CTA can keep it in tensor memory and sum the tile after its roles;
  - every other part starts its CTA's range (it goes to that CTA's one
    workspace slot), and belongs to a CTA of higher index than the tile's
    owner, so the owners' waits form no cycle;
  - a CTA owns at most one split tile;
  - the parts of a tile cover its chunks exactly once, in CTA order.
The formulas restate the kernel's chunk ranges (start of CTA b's range =
b * chunks / CTAs, rounded down) and the host's choice of split region.
"""
import pytest

SMS = 152


def token_tile(M):
    tiles = (M + 255) // 256
    per = (M + tiles - 1) // tiles
    return (per + 15) // 16 * 16


def schedule(M, N, K, variant, sms=SMS):
    """(tiles, dp_tiles, nch, usk, grid) as the host chooses them."""
    nt = token_tile(M)
    tiles = ((M + nt - 1) // nt) * ((N + 127) // 128)
    kr = 256 if variant == 0 else 512
    nch = K // kr
    min_chunks = 1024 // kr
    dp, usk, grid = tiles, 0, min(tiles, sms)
    if tiles % sms != 0 and nch >= 2:
        if tiles > sms:
            dp = (tiles // sms - 1) * sms
            usk = (tiles - dp) * nch
            grid = sms
        else:
            g = min(sms, tiles * nch // min_chunks)
            if g > tiles:
                dp, usk, grid = 0, tiles * nch, g
    return tiles, dp, nch, usk, grid


def items(b, tiles, dp, nch, usk, grid):
    """CTA b's items in order: (tile, first chunk, end chunk)."""
    out = [(t, 0, nch) for t in range(b, dp, grid)]
    if usk:
        u, uend = b * usk // grid, (b + 1) * usk // grid
        while u < uend:
            tr, cb = divmod(u, nch)
            ce = min(nch, cb + (uend - u))
            out.append((dp + tr, cb, ce))
            u += ce - cb
    return out


SHAPES = [(M, N, K, 0) for M in (512, 4096, 23552)
          for N, K in ((7168, 5120), (5120, 6144), (34816, 5120), (5120, 17408))]
SHAPES += [(16, 128, 8192, 0), (33, 250, 17408, 0), (20, 256, 16384, 1), (600, 520, 4096, 0),
           (300, 4096, 1024, 0), (40, 128, 4096, 1), (64, 384, 2048, 0), (24, 40, 512, 0),
           (4096, 5120, 6144, 1), (1000, 1000, 2048, 1)]


@pytest.mark.parametrize("sms", [SMS, 7, 1])
@pytest.mark.parametrize("M,N,K,variant", SHAPES)
def test_split_region_hand_off_invariants(M, N, K, variant, sms):
    tiles, dp, nch, usk, grid = schedule(M, N, K, variant, sms)
    per_cta = [items(b, tiles, dp, nch, usk, grid) for b in range(grid)]
    parts = {}  # tile -> [(cta, cb, ce, is_final, starts_range)]
    for b, its in enumerate(per_cta):
        owned = 0
        for i, (t, cb, ce) in enumerate(its):
            whole = cb == 0 and ce == nch
            if t < dp:
                assert whole
            if whole:
                continue
            final = i == len(its) - 1
            starts = (t - dp) * nch + cb == b * usk // grid  # first chunk = the start of b's range
            parts.setdefault(t, []).append((b, cb, ce, final, starts))
            if cb == 0:
                owned += 1
        assert owned <= 1, f"CTA {b} owns {owned} split tiles"
    # every tile is computed exactly once: whole by one CTA, or by its parts
    whole_count = {}
    for b, its in enumerate(per_cta):
        for t, cb, ce in its:
            if cb == 0 and ce == nch:
                whole_count[t] = whole_count.get(t, 0) + 1
    for t in range(tiles):
        assert (t in whole_count) != (t in parts), t
        if t in whole_count:
            assert whole_count[t] == 1
    for t, ps in parts.items():
        ps.sort(key=lambda p: p[1])
        assert len(ps) >= 2
        assert ps[0][1] == 0 and ps[-1][2] == nch
        for a, c in zip(ps, ps[1:]):
            assert a[2] == c[1], "parts are contiguous"
            assert c[0] > a[0], "later chunks belong to CTAs of higher index"
        owner = ps[0]
        assert owner[3], f"tile {t}: its first part is not its CTA's final item"
        for p in ps[1:]:
            assert p[4], f"tile {t}: part of CTA {p[0]} does not start that CTA's range"
        # the CTAs are consecutive, as the workspace indexing (bfirst + k) assumes
        assert [p[0] for p in ps] == list(range(owner[0], owner[0] + len(ps)))


def test_split_region_is_used_where_the_tiles_do_not_fill_waves():
    # M = 512: three of the four layer shapes have fewer tiles than SMs
    for N, K in ((7168, 5120), (5120, 6144), (5120, 17408)):
        tiles, dp, nch, usk, grid = schedule(512, N, K, 0)
        assert tiles < SMS and dp == 0 and usk == tiles * nch and grid == SMS
    # full waves only: no split
    tiles, dp, nch, usk, grid = schedule(4096, 4864, 1024, 0)
    assert tiles == 4 * SMS and usk == 0 and dp == tiles
    # a partial last wave: one wave and a half split
    tiles, dp, nch, usk, grid = schedule(4096, 34816, 5120, 0)
    assert tiles == 4352 and dp == (4352 // SMS - 1) * SMS and usk == (tiles - dp) * nch
