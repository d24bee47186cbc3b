"""The decode launch planner (pkv_plan_decode), host arithmetic behind every
decode launch, checked on the CPU: the plans measured best on GB300 for each
batch, the limits every plan keeps, and argument checks."""

import pytest

import paged_kv_cache_210_gb300 as pkv
from paged_kv_cache_210_gb300 import build as lib_build

T, N, WD = pkv.PKV_SHAPE_TICKET, pkv.PKV_SHAPE_NARROW, pkv.PKV_SHAPE_WIDE


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return pkv.load()


def gb300(**kw):
    """A GB300's figures with a default handle: 152 SMs, 4 ticket / 3 narrow /
    4 wide blocks per SM, 16-block clusters, 64 splits, 2048 tokens."""
    f = dict(num_sms=152, ticket_blocks_per_sm=4, narrow_blocks_per_sm=3, wide_blocks_per_sm=4,
             max_cluster=16, max_splits=64, max_seq_len=2048)
    f.update(kw)
    return pkv.DeviceFigures(**f)


def plan(lib, batch, num_splits=0, **kw):
    return pkv.pkv_plan_decode(gb300(**kw), batch, num_splits, lib=lib)


@pytest.mark.parametrize("batch,shape,splits", [
    (1, N, 16), (2, N, 12), (3, WD, 8), (4, WD, 8),
    (5, WD, 8), (8, WD, 8), (9, WD, 4), (16, WD, 4), (17, WD, 2), (32, WD, 2),
])
def test_cluster_plans_by_batch(lib, batch, shape, splits):
    p = plan(lib, batch)
    assert (p.shape, p.cluster, p.num_splits, p.chunk_pages) == (shape, splits, splits, 0)
    assert p.grid_splits == splits and p.longest_first == 0


@pytest.mark.parametrize("batch", [33, 34, 35, 64, 100, 128, 152])
def test_ticket_plans_by_batch(lib, batch):
    p = plan(lib, batch)
    # ranges of at least 16 pages, sized in the launch from the batch's pages
    assert (p.shape, p.cluster, p.num_splits, p.chunk_pages, p.grid_splits) == (T, 0, 0, 16, 8)
    assert p.longest_first == 1
    # 608 resident ticket blocks x 3 / 40: ranges of about 1.65 x the pages per slot
    assert p.range_div == 46 and p.grid_units == batch + 46


@pytest.mark.parametrize("batch", [153, 256, 1000])
def test_ticket_plans_unsplit_past_two_waves(lib, batch):
    """Batches whose sequences alone fill two waves of ticket blocks run each
    sequence whole, longest first, with no spare units."""
    p = plan(lib, batch)
    assert (p.shape, p.chunk_pages, p.grid_splits, p.range_div, p.grid_units) == (
        T, 128, 1, 0, batch)
    assert p.longest_first == 1


def units_of(lens, least, range_div, max_pages=128):
    """The (sequence, range) units a longest-first launch enumerates, in order."""
    pages = [min(max((n + 15) // 16, 0), max_pages) for n in lens]
    r = max(least, min(128, -(-sum(pages) // range_div))) if range_div else least
    order = sorted(range(len(lens)), key=lambda s: (pages[s] == 0, -pages[s], s))
    return r, [(s, k) for s in order for k in range(max(1, -(-pages[s] // r)))]


def test_units_fit_the_grid():
    """Fewer units than batch + range_div for any lengths (the grid's units):
    random mixes, lengths just past a multiple of the range, and invalid
    lengths; every sequence's ranges cover its pages once."""
    import random
    rnd = random.Random(7)
    cases = [[rnd.choice([0, 1, 17, 33, 257, 2048, 2049, rnd.randint(1, 2048)])
              for _ in range(rnd.randint(1, 300))] for _ in range(300)]
    cases += [[16 * 17 + 1] * 35 + [1] * 5, [2048] + [1] * 63, [16 * 16 + 1] * 40]
    for lens in cases:
        for rd, mp, least in ((1, 128, 16), (5, 128, 16), (38, 128, 16), (76, 128, 16),
                              (38, 16, 16), (0, 128, 128), (0, 16, 16)):
            r, units = units_of(lens, least, rd, mp)
            assert len(units) < len(lens) + max(rd, 1)
            for s, n in enumerate(lens):
                p = min(max((n + 15) // 16, 0), mp)
                ks = [k for (t, k) in units if t == s]
                assert ks == list(range(max(1, -(-p // r))))
                assert p == 0 or (len(ks) - 1) * r < p <= len(ks) * r


def test_every_library_plan_keeps_its_limits(lib):
    for sms in (20, 76, 132, 152):
        for max_cluster in (0, 2, 8, 16):
            for max_splits in (1, 4, 16, 64, 128):
                for batch in list(range(1, 70)) + [100, 255, 256, 1000, 4096]:
                    p = plan(lib, batch, num_sms=sms, max_cluster=max_cluster,
                             max_splits=max_splits)
                    if p.cluster:
                        s = p.cluster
                        assert p.shape in (N, WD) and s in (2, 4, 8, 12, 16)
                        if s in (12, 16):   # two launches' blocks resident at once
                            assert p.shape == N and 2 * batch * 8 * s <= 3 * sms
                        assert s <= max_cluster and s <= max_splits
                        per_sm = 3 if p.shape == N else 4
                        # the whole launch is one wave of its shape's blocks
                        assert batch * 8 * s <= per_sm * sms
                        assert p.longest_first == 0
                        assert p.range_div == 0 and p.grid_units == 0
                    else:
                        assert p.shape == T and p.num_splits == 0
                        least = max(16, -(-128 // max_splits))
                        waves = batch * 8 * -(-128 // least) > 4 * sms
                        assert p.longest_first == int(waves)
                        if waves and batch * 8 > 2 * 4 * sms:      # unsplit
                            assert (p.chunk_pages, p.grid_splits, p.range_div) == (128, 1, 0)
                            assert p.grid_units == batch
                        elif waves:
                            assert p.chunk_pages == least
                            assert p.grid_splits == -(-128 // least) <= max_splits
                            assert p.range_div == max((4 * sms * 3 + 20) // 40, 1)
                            assert p.grid_units == batch + p.range_div
                        else:
                            assert p.chunk_pages == least
                            assert p.grid_splits == -(-128 // least) <= max_splits
                            assert p.range_div == 0 and p.grid_units == 0


def test_chosen_split_counts(lib):
    p = plan(lib, 2, num_splits=4)
    assert (p.shape, p.cluster, p.grid_splits) == (N, 4, 4)
    p = plan(lib, 4, num_splits=16)          # 512 blocks: more than one narrow wave
    assert (p.shape, p.cluster) == (WD, 16)
    p = plan(lib, 2, num_splits=3)           # any size up to the cluster limit
    assert (p.shape, p.cluster, p.grid_splits) == (N, 3, 3)
    p = plan(lib, 2, num_splits=32)          # beyond the cluster limit: ticket
    assert (p.shape, p.cluster, p.num_splits, p.grid_splits) == (T, 0, 32, 32)
    p = plan(lib, 300, num_splits=1)
    assert (p.shape, p.cluster, p.num_splits, p.grid_splits, p.longest_first) == (T, 0, 1, 1, 0)
    p = plan(lib, 2, num_splits=8, max_cluster=0)   # no clusters on the device
    assert (p.shape, p.cluster) == (T, 0)


def test_shorter_context_caps_ranges(lib):
    p = plan(lib, 2, max_seq_len=64)          # 4 pages: S = 16 or 8 would leave empty blocks
    assert p.cluster <= 4 and p.grid_splits == p.cluster
    p = plan(lib, 1000, max_seq_len=256)      # 16 pages: one range of all of them
    assert (p.shape, p.chunk_pages, p.grid_splits) == (T, 16, 1)


def test_invalid_arguments(lib):
    bad = [dict(num_sms=0), dict(ticket_blocks_per_sm=0), dict(wide_blocks_per_sm=0),
           dict(max_cluster=17), dict(max_cluster=-1), dict(max_splits=0),
           dict(max_splits=129), dict(max_seq_len=100), dict(max_seq_len=4096)]
    for kw in bad:
        with pytest.raises(pkv.PkvError):
            plan(lib, 2, **kw)
    for batch, splits in ((0, 0), (-1, 0), (2, -1), (2, 65)):
        with pytest.raises(pkv.PkvError):
            plan(lib, batch, splits)


def test_ranges_per_sequence_by_float_reciprocal():
    """The launch counts a p-page sequence's ranges, ceil(p / r), as
    trunc(float32(p + r - 1) * rcp(r) + 1/256) and a unit's rank k = off / n
    as trunc(off / n) corrected by one step, with float32 arithmetic instead
    of integer division. Checked here for every p, r <= 128 and the offsets a
    grid can hold, with the product and the add rounded separately and as one
    fused multiply-add (the compiler may contract them), and with the rank's
    quotient off by up to 3 ulp (the fast division)."""
    import numpy as np
    f32 = np.float32
    for r in range(1, 129):
        inv = f32(1.0) / f32(r)                      # correctly rounded reciprocal
        p = np.arange(1, 129, dtype=np.int64)
        x = (p + r - 1).astype(f32)
        sep = (x * inv + f32(1.0 / 256.0)).astype(f32)
        fused = (x.astype(np.float64) * np.float64(inv) + 1.0 / 256.0).astype(f32)
        want = -(-p // r)
        assert np.array_equal(sep.astype(np.int64), want)
        assert np.array_equal(fused.astype(np.int64), want)
    off = np.arange(0, 65536 + 256, dtype=np.int64)
    for n in range(2, 9):
        q = off.astype(f32) / f32(n)
        for ulps in (-3, 0, 3):
            qq = q
            for _ in range(abs(ulps)):
                qq = np.nextafter(qq, f32(np.inf) if ulps > 0 else f32(-np.inf)).astype(f32)
            k = qq.astype(np.int64)
            k = np.where(k * n > off, k - 1, k)
            k = np.where((k + 1) * n <= off, k + 1, k)
            assert np.array_equal(k, off // n)


def device_unit_of(u, lens, least, range_div, max_pages=128):
    """The decode launch's unit lookup restated step by step (one block, one
    unit): the page-count histogram, lane l of warp 0 owning the buckets
    128 - 4l - e, the range size from the page total, the units per bucket,
    the inclusive scan over lanes, the bucket holding unit u with the rank
    and range index inside it (float32 quotient corrected by one step), then
    the k-th sequence by index with that page count. Returns (sequence,
    range index) or None past the last unit."""
    import numpy as np
    f32 = np.float32
    pc = [min(max((n + 15) // 16, 0), max_pages) for n in lens]
    hist = [0] * 129
    for p in pc:
        hist[p] += 1
    whole = range_div == 0 and least >= max_pages
    rng = least
    if not whole and range_div > 0:
        total_pages = sum(hist[p] * p for p in range(1, 129))
        rng = max(least, min(128, -(-total_pages // range_div)))
    inv = f32(1.0) / f32(rng)

    def ranges_of(p):
        if whole:
            return 1
        return int(f32(f32(p + rng - 1) * inv) + f32(1.0 / 256.0))
    lane_units = []
    for lane in range(32):
        lane_units.append([hist[128 - 4 * lane - e] * ranges_of(128 - 4 * lane - e)
                           for e in range(4)])
    incl = list(np.cumsum([sum(x) for x in lane_units]))
    pick = None
    for lane in range(32):
        excl = incl[lane] - sum(lane_units[lane])
        for e in range(4):
            if excl <= u < excl + lane_units[lane][e]:
                p = 128 - 4 * lane - e
                per = ranges_of(p)
                off = u - excl
                k = off if per == 1 else int(f32(off) / f32(per))
                if k * per > off:
                    k -= 1
                if (k + 1) * per <= off:
                    k += 1
                pick = (p, k, off - k * per)
            excl += lane_units[lane][e]
    total = incl[-1]
    if u >= total:
        pick = (0, u - total, 0)
    p, k, split = pick
    if p == 0 and k >= hist[0]:
        return None
    same = [s for s in range(len(lens)) if pc[s] == p]
    return same[k], split


def test_device_unit_lookup_matches_the_order():
    """Every unit of the grid maps, by the device's lookup, to the unit at
    that place in the plain order (page count descending, index, range),
    and the units past the last map to nothing: random and adversarial
    batches, split and whole-sequence launches."""
    import random
    rnd = random.Random(11)
    cases = [[rnd.choice([0, 1, 16, 17, 300, 2048, rnd.randint(1, 2048)])
              for _ in range(rnd.randint(1, 120))] for _ in range(40)]
    cases += [[16 * 17] * 43 + [16], [2048] + [1] * 63, [16 * 24 + 1] * 44]
    for lens in cases:
        for rd, least in ((46, 16), (0, 128), (5, 16)):
            r, units = units_of(lens, least, rd)
            grid = len(lens) + max(rd, 0)
            for u in range(grid):
                got = device_unit_of(u, lens, least, rd)
                want = units[u] if u < len(units) else None
                assert got == want, (lens, rd, u, got, want)
